/*
 * dfl.h -- C ABI of the block-diffusion draft-step library (libdfl.so), sm_103a.
 *
 * The library computes one single-pass block-diffusion draft step: per draft
 * layer a softmax mix of target hidden states followed by RMSNorm, separate
 * K/V projections for target-context and draft features with queries from the
 * draft features only, block attention in which every block query sees every
 * context key and attends bidirectionally inside the block, the shared LM head
 * with argmax, greedy acceptance, and optional K-draft sampling with
 * streak-score self-selection.
 *
 * Sources (page title, section):
 *   DFlare post   "DFlare: Scaling Up Draft Capacity for Block Diffusion
 *                 Speculative Decoding" (iplexlaw blog)
 *   DFlash article "DFlash: Block Diffusion for Flash Speculative Decoding"
 *                 (Qiita)
 *   SpecDiff-2 notes "SpecDiff-2 -- Scaling Diffusion Drafter Alignment For
 *                 Faster Speculative Decoding" (MLSys 2026 talk notes)
 *
 * Conventions for every entry point
 *   Ownership  All tensor pointers are caller-owned DEVICE memory (for
 *              example a torch tensor's data_ptr()).  The library never
 *              allocates or frees device memory.  Scratch space comes from the
 *              caller as (ws, ws_bytes); dfl_workspace_size() gives the size.
 *              Host pointers appear only where stated (parameter structs).
 *   Launch     Calls are asynchronous on the given stream (a cudaStream_t
 *              passed as void*, NULL = legacy default stream).  They do not
 *              synchronise and may be captured into a CUDA graph.  Kernels
 *              are launched with programmatic dependent launch: a kernel may
 *              start while the previous kernel in the stream finishes and
 *              waits for it before touching global memory (results are the
 *              same either way); DFL_PDL=0 in the environment, read once per
 *              process, launches plainly.
 *   Layout     Row-major, contiguous.  Weights are [out][in] (in contiguous).
 *              bf16 tensors hold raw bf16 bits (2 bytes per element).
 *              The block residual stream Xb is always fp32.
 *   Alignment  Every tensor pointer must be 16-byte aligned and d, hd,
 *              Hq*hd a multiple of 8, else DFL_ERR_MISALIGNED (checked for
 *              every pointer a 16-byte or TMA access reads or writes).
 *   Sizes      Row counts (N*C context rows, N*B block rows) stay below 2^31:
 *              TMA coordinates and GEMM extents are 32-bit, so larger ones
 *              return DFL_ERR_UNSUPPORTED_SHAPE.
 *   Errors     Argument checks run on the host before any launch and return
 *              a non-zero dfl_status with nothing launched.  A launch failure
 *              returns DFL_ERR_CUDA.  Kernels never trap: a bounded wait that
 *              runs out records DFL_ERR_TIMEOUT in a per-device error word,
 *              read (and cleared) by dfl_get_device_error().
 */
#ifndef DFL_H
#define DFL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dfl_status {
    DFL_OK = 0,
    DFL_ERR_INVALID_ARG = 1,       /* null pointer, non-positive size, bad enum */
    DFL_ERR_UNSUPPORTED_SHAPE = 2, /* a shape this build has no kernel for */
    DFL_ERR_MISALIGNED = 3,        /* pointer or size breaks the 16-byte rule */
    DFL_ERR_WORKSPACE = 4,         /* ws_bytes smaller than dfl_workspace_size() */
    DFL_ERR_CUDA = 5,              /* a CUDA runtime call or launch failed */
    DFL_ERR_TIMEOUT = 6,           /* a device-side bounded wait ran out */
    DFL_ERR_NO_DEVICE = 7,         /* no sm_103a device is current */
    DFL_ERR_BOUNDS = 8             /* (bounds-checked build, -DDFL_CHECK) a kernel computed an
                                      index outside the extent its shape gives; the access was
                                      skipped and the code recorded in the device error word */
} dfl_status;

typedef enum dfl_dtype { DFL_F32 = 0, DFL_BF16 = 1 } dfl_dtype;

typedef void* dfl_stream;          /* a cudaStream_t */

/* Host-side parameters of K-draft sampling. */
typedef struct dfl_sample_params {
    int32_t K;        /* drafts per sequence, 1..64 */
    float T;          /* temperature, > 0 */
    uint64_t seed;    /* Philox4x32-10 key (low word, high word) */
} dfl_sample_params;

/* Shape descriptor for dfl_workspace_size(). Unused fields may be 0. */
typedef struct dfl_shape {
    int32_t N, C, B, d, Hq, Hkv, hd, D, L, V, K, G, row0;
    int32_t dtype;    /* a dfl_dtype */
    int32_t F;        /* FFN width (DFL_OP_BLOCK_FFN, DFL_OP_DRAFT_STEP) */
    int32_t R;        /* new context rows per sequence (DFL_OP_DRAFT_STEP_CACHED,
                         where C is the cache capacity) */
    int32_t fc;       /* 1: the step's context features come from the DFlash
                         fusion (dfl_fc_fuse) instead of per-layer mixtures */
} dfl_shape;

typedef enum dfl_op {
    DFL_OP_DUAL_KV_PROJ = 1,
    DFL_OP_BLOCK_ATTN = 2,
    DFL_OP_LM_HEAD = 3,
    DFL_OP_SELF_SELECT = 4,
    DFL_OP_DRAFT_STEP = 5,
    DFL_OP_TV_ACCEPTANCE = 6,
    DFL_OP_SPEC_ACCEPT = 7,
    DFL_OP_BLOCK_FFN = 8,
    DFL_OP_DRAFT_STEP_CACHED = 9,
    DFL_OP_DRAFT_STEP_HOST = 10,
    DFL_OP_FC_FUSE = 11,           /* rows = N*C, d */
    DFL_OP_SAMPLED_GREEDY = 12     /* N, G, V */
} dfl_op;

/* Library version string (static storage). */
const char* dfl_version(void);

/* Message for a status code (static storage); "unknown status" for a code
 * outside dfl_status. */
const char* dfl_status_string(dfl_status s);

/* Bytes of scratch the operation needs for this shape; 0 if it needs none or
 * the shape is invalid. */
size_t dfl_workspace_size(dfl_op op, const dfl_shape* shape);

/*
 * dfl_rope_table -- rotary cos/sin table for positions 0..P-1.
 *   Reading (the pages give no position scheme): without positions every
 *   [MASK] row of the block is identical; rotary embedding (rotate-half pairs
 *   i, i+hd/2, angle p * theta^(-2i/hd)) is used, context at 0..C-1 and the
 *   block at C..C+B-1.
 *   table  out, device fp32 [P][hd/2][2] = (cos, sin), computed in fp64 and
 *          rounded to fp32.
 *   Errors: INVALID_ARG if P <= 0, hd <= 0 or hd odd, theta <= 0.
 */
dfl_status dfl_rope_table(float* table, int32_t P, int32_t hd, double theta,
                          dfl_stream stream);

/*
 * dfl_layer_mix_rmsnorm -- per-draft-layer mixture of target hidden states.
 *   DFlare post, "Per-draft-layer mixing of different information": each
 *   draft layer learns mixing ratios over L target hidden states, softmax-
 *   normalised, and applies RMSNorm: Xc_l = RMSNorm(sum_i softmax(mix_l)_i H_i).
 *   D draft layers are produced from ONE read of H.
 *   H           in, dt [L] slabs of [rows][d]; slab i starts at element
 *               i * layer_stride.
 *   mix_logits  in, device fp32 [D][L].
 *   gain        in, device fp32 [D][d] RMSNorm gains.
 *   Xc          out, dt [D] slabs of [rows][d] at element l * xc_layer_stride.
 *   Accumulation fp32; bf16 outputs rounded to nearest even.
 *   Errors: INVALID_ARG (null, L/D outside 1..32, rows/d <= 0, strides too
 *   small), MISALIGNED.
 */
dfl_status dfl_layer_mix_rmsnorm(const void* H, int64_t layer_stride, int32_t L,
                                 int64_t rows, int32_t d, dfl_dtype dt, int32_t D,
                                 const float* mix_logits, const float* gain, float eps,
                                 void* Xc, int64_t xc_layer_stride, dfl_stream stream);

/*
 * dfl_fc_fuse -- DFlash's shared context representation: one fully connected
 *   layer over the concatenated hidden states of L target layers.
 *   DFlash article, "Writing a whole block in one forward pass": features
 *   taken from several target layers are fused by a light projection and
 *   injected into the K/V of every draft layer; the DFlare post ("Per-draft-
 *   layer mixing of different information") names this fully connected
 *   fusion as the baseline its per-layer mixtures replace.  Reading: no bias,
 *   and an RMSNorm with its own gain follows (as after DFlare's mixture):
 *     Xc = RMSNorm([H_1 | H_2 | ... | H_L] W_fc^T; gain)
 *   One representation serves all draft layers (dfl_step_args.W_fc).
 *   H           in, dt [L] slabs of [rows][d]; slab i starts at element
 *               i * layer_stride (>= rows*d when L > 1)
 *   W_fc        in, dt [d][L*d]: column block i multiplies slab i
 *   gain        in, device fp32 [d]
 *   Xc          out, dt [rows][d]
 *   ws          dfl_workspace_size(DFL_OP_FC_FUSE) bytes (fp32 [rows][d]
 *               pre-norm features; shape fields N*C = rows, d)
 *   bf16: one tcgen05 GEMM with K = L*d whose A tiles are read slab by slab
 *   (d a multiple of 64); fp32: CUDA-core GEMMs.  d <= 6144.
 *   Errors: INVALID_ARG (null pointer, L outside 1..64, rows or d <= 0, slab
 *   stride too small), MISALIGNED (pointers, d % 8, slab stride bytes % 16),
 *   UNSUPPORTED_SHAPE (bf16 d % 64, d > 6144), WORKSPACE.
 */
dfl_status dfl_fc_fuse(const void* H, int64_t layer_stride, int32_t L, int64_t rows, int32_t d,
                       dfl_dtype dt, const void* W_fc, const float* gain, float eps, void* Xc,
                       void* ws, size_t ws_bytes, dfl_stream stream);

/*
 * dfl_dual_kv_proj -- dual-source projections of one draft layer.
 *   DFlare post, "Separate KV projections by information source": target
 *   context features and draft (anchor + [MASK]) features get separate
 *   key/value projections; queries come from the draft features only.
 *     Kc = Xc Wkc^T, Vc = Xc Wvc^T                    (context rows)
 *     Xn = RMSNorm(Xb; blk_gain)  (reading: pre-norm block input)
 *     Q = Xn Wq^T, Kb = Xn Wkb^T, Vb = Xn Wvb^T      (block rows)
 *   then rotary embedding on Q, Kb (positions C..C+B-1) and Kc (0..C-1).
 *   Xc   in, dt [N*C][d] (rows ordered sequence-major)
 *   Xb   in, fp32 [N*B][d] block residual stream
 *   Wq [Hq*hd][d], Wkc/Wvc/Wkb/Wvb [Hkv*hd][d]: in, dt
 *   rope in, fp32 [C+B][hd/2][2] from dfl_rope_table, or NULL (no rotary)
 *   Q out dt [N*B][Hq][hd]; Kc, Vc out dt [N*C][Hkv][hd]; Kb, Vb out dt [N*B][Hkv][hd]
 *   ws   scratch of dfl_workspace_size(DFL_OP_DUAL_KV_PROJ) bytes
 *   bf16: tcgen05 tensor-core GEMMs, fp32 accumulation.  fp32: CUDA-core GEMMs.
 *   Errors: INVALID_ARG, UNSUPPORTED_SHAPE (bf16 needs hd in {64,128},
 *   Hq % Hkv == 0, d % 8 == 0), MISALIGNED, WORKSPACE.
 */
dfl_status dfl_dual_kv_proj(const void* Xc, const float* Xb, int32_t N, int32_t C,
                            int32_t B, int32_t d, dfl_dtype dt, const float* blk_gain,
                            float eps, const void* Wq, const void* Wkc, const void* Wvc,
                            const void* Wkb, const void* Wvb, int32_t Hq, int32_t Hkv,
                            int32_t hd, const float* rope, void* Q, void* Kc, void* Vc,
                            void* Kb, void* Vb, void* ws, size_t ws_bytes,
                            dfl_stream stream);

/*
 * dfl_block_attn -- block attention, output projection and residual add.
 *   DFlare post, "Generating candidates in parallel, the target decides
 *   acceptance": one forward predicts all mask positions with bidirectional
 *   attention inside the block; DFlash article, "Writing a whole block in one
 *   forward pass": target features enter the K/V of every draft layer.
 *     O = softmax(Q [Kc;Kb]^T / sqrt(hd)) [Vc;Vb]   (no mask; query head h
 *         reads K/V head h / (Hq/Hkv))
 *     Xb <- Xb + O Wo^T                              (reading: output
 *         projection with residual, as in the drafter's transformer layers)
 *   Q, Kc, Vc, Kb, Vb  in, dt, layouts as produced by dfl_dual_kv_proj
 *   Wo   in, dt [d][Hq*hd]
 *   Xb   in/out, fp32 [N*B][d]
 *   ws   scratch of dfl_workspace_size(DFL_OP_BLOCK_ATTN) bytes (split-KV
 *        partial results, then fp32 partials of the output projection split
 *        along K; a buffer without room for the latter is accepted down to
 *        the size without them, and the projection then runs unsplit)
 *   Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, WORKSPACE.
 */
dfl_status dfl_block_attn(const void* Q, const void* Kc, const void* Vc, const void* Kb,
                          const void* Vb, int32_t N, int32_t C, int32_t B, int32_t Hq,
                          int32_t Hkv, int32_t hd, dfl_dtype dt, const void* Wo, int32_t d,
                          float* Xb, void* ws, size_t ws_bytes, dfl_stream stream);

/*
 * dfl_lm_head_argmax -- shared frozen LM head, argmax, optional K-draft sampling.
 *   DFlare post, "Stabilise the front, weight the back": the embedding and LM
 *   head are frozen and shared with the target.  Reading: a final RMSNorm
 *   precedes the head.  For rows r = row0..B-1 of each sequence:
 *     z = RMSNorm(Xb_r; final_gain) W_lm^T,  draft = argmax_v z_v
 *   (lowest index on equal fp32 maxima).
 *   SpecDiff-2 notes, "Parallel drafting with diffusion LMs" / "Self-Selection
 *   Acceptance": with sp != NULL, K independent draws from softmax(z/T) per
 *   row by inverting the CDF at u = ((x0 >> 8) + 1/2) 2^-24, x0 word 0 of
 *   Philox4x32-10(counter (n, r-row0, k, 0), key (seed lo, seed hi)).
 *   Xb          in, fp32 [N][B][d]
 *   W_lm        in, dt [V][d]
 *   argmax_out  out, int32 [N][B-row0]
 *   logits_out  out (nullable), fp32 [N*(B-row0)][V]; required when sp != NULL
 *   sp          in, HOST pointer (nullable)
 *   samples_out out, int32 [N][K][B-row0] (required when sp != NULL)
 *   Errors: INVALID_ARG (row0 outside 0..B-1, V <= 0, K outside 1..64,
 *   T <= 0), UNSUPPORTED_SHAPE, MISALIGNED, WORKSPACE.
 */
dfl_status dfl_lm_head_argmax(const float* Xb, int32_t N, int32_t B, int32_t row0,
                              int32_t d, dfl_dtype dt, const float* final_gain, float eps,
                              const void* W_lm, int32_t V, int32_t* argmax_out,
                              float* logits_out, const dfl_sample_params* sp,
                              int32_t* samples_out, void* ws, size_t ws_bytes,
                              dfl_stream stream);

/*
 * dfl_greedy_accept -- greedy acceptance of one block per sequence.
 *   DFlare post, "Generating candidates in parallel, the target decides
 *   acceptance": under greedy decoding the prefix up to the first mismatch is
 *   accepted and the target supplies the next token.
 *   draft   in, int32 [N][n]     window positions 1..n
 *   target  in, int32 [N][n+1]   target argmax t_1..t_{n+1}
 *   accept_len out, int32 [N]    a = number of leading j with draft_j == t_j
 *   bonus      out, int32 [N]    t_{a+1}
 *   Errors: INVALID_ARG (null, N <= 0, n < 0 or n > 1024).
 */
dfl_status dfl_greedy_accept(const int32_t* draft, const int32_t* target, int32_t N,
                             int32_t n, int32_t* accept_len, int32_t* bonus,
                             dfl_stream stream);

/*
 * dfl_self_select -- streak-score self-selection and greedy acceptance.
 *   SpecDiff-2 notes, "Streak-Distillation" (streak equation) and
 *   "Self-Selection Acceptance": each of K drafts is scored with
 *     S_k = sum_{m=1}^{G} prod_{j<=m} p_j(x_j^k),
 *     p_j(x) = softmax(vlog[n][k][j-1])_x,
 *   the argmax draft k* (lowest k on ties) is selected and greedy acceptance
 *   is applied to it against the argmax of its own verifier rows, reusing the
 *   cached verifier logits (draft probabilities are not used).
 *   vlog    in, dt [N][K][G+1][V]; row G serves the bonus token
 *   drafts  in, int32 [N][K][G]
 *   scores  out, fp32 [N][K]; selected, accept_len, bonus out, int32 [N]
 *   ws      scratch of dfl_workspace_size(DFL_OP_SELF_SELECT) bytes
 *   Errors: INVALID_ARG (K outside 1..64, G outside 1..1024), MISALIGNED,
 *   WORKSPACE.
 */
dfl_status dfl_self_select(const void* vlog, dfl_dtype dt, const int32_t* drafts,
                           int32_t N, int32_t K, int32_t G, int32_t V, float* scores,
                           int32_t* selected, int32_t* accept_len, int32_t* bonus,
                           void* ws, size_t ws_bytes, dfl_stream stream);

/*
 * dfl_self_select_noalloc -- dfl_self_select without a caller workspace.
 *   The pages have no counterpart to this call; it exists for callers that
 *   cannot provide device scratch memory, such as a plugin inside a serving
 *   engine that owns all device memory through its own pool, or a host loop
 *   that must not call cudaMalloc while serving.  It computes exactly what
 *   dfl_self_select computes, with the same arguments minus (ws, ws_bytes).
 *   Scratch: a fixed 768 KiB array inside the library's device image, held
 *   on every GPU that loads the library until the process exits; it fits
 *   N*K*(G+1) <= 65536 verifier rows, larger calls return DFL_ERR_WORKSPACE
 *   with nothing launched.  The library allocates nothing for this call.
 *   The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) and caches it; make that first call before any
 *   stream capture on that device.  The address belongs to the device's
 *   current CUDA context: when another context becomes current there (after
 *   cudaDeviceReset, for example) the next call looks it up again.  All calls on a device share the array
 *   and it keeps the last call's contents (no call relies on them); calls
 *   whose kernels overlap on the GPU race on it and must be serialised.
 *   Errors: as dfl_self_select, plus DFL_ERR_WORKSPACE for the size limit.
 */
dfl_status dfl_self_select_noalloc(const void* vlog, dfl_dtype dt, const int32_t* drafts,
                                   int32_t N, int32_t K, int32_t G, int32_t V, float* scores,
                                   int32_t* selected, int32_t* accept_len, int32_t* bonus,
                                   dfl_stream stream);

/*
 * dfl_tv_acceptance -- per-position acceptance proxy of K drafts.
 *   SpecDiff-2 notes, "Streak-Distillation": alpha = 1 - 1/2 sum_x |P(x) -
 *   Q(x)| with Q = softmax(z_j / T) the drafter's marginal at window position
 *   j and P = softmax(vlog[n][k][j]) the verifier's distribution there given
 *   draft k's prefix; the expected accepted length of draft k under the
 *   streak equation is sum_m prod_{j<=m} alpha_j.
 *   logits  in, fp32 [N*G][V] (the drafter's rows, as from dfl_lm_head_argmax)
 *   vlog    in, dt [N][K][G+1][V]
 *   alpha   out, fp32 [N][K][G]; tokens_per_draft out (nullable) fp32 [N][K]
 *   ws      dfl_workspace_size(DFL_OP_TV_ACCEPTANCE) bytes (row log-sum-exps)
 *   Errors: INVALID_ARG (K outside 1..64, G outside 1..1024, T <= 0),
 *   MISALIGNED (logits, vlog or ws), WORKSPACE.
 */
dfl_status dfl_tv_acceptance(const float* logits, float T, const void* vlog, dfl_dtype dt,
                             int32_t N, int32_t K, int32_t G, int32_t V, float* alpha,
                             float* tokens_per_draft, void* ws, size_t ws_bytes,
                             dfl_stream stream);

/*
 * dfl_spec_accept -- lossless stochastic acceptance of one draft per sequence.
 *   DFlare post, "Generating candidates in parallel, the target decides
 *   acceptance": stochastic decoding needs an acceptance rule that keeps the
 *   target's distribution.  For j = 1..G: accept x_j when u_j Q(x_j) <
 *   P(x_j) (probability min(1, P/Q)), Q = softmax(z_j / T), P =
 *   softmax(v_j); at the first rejection the next token is drawn from the
 *   normalised residual max(0, P - Q); after G acceptances the bonus token is
 *   drawn from P_{G+1}.  Uniforms: u = ((x0 >> 8) + 1/2) 2^-24 from
 *   Philox4x32-10 at counter (n, j, 0, 1) for the tests and (n, j, 0, 2) for
 *   the draw, key (seed lo, seed hi).
 *   logits  in, fp32 [N*G][V]; vlog in, dt [N][K][G+1][V]
 *   drafts  in, int32 [N][K][G]; sel in, int32 [N] draft to verify (nullable:
 *           draft 0; an index outside 0..K-1 is read as draft 0 and records
 *           DFL_ERR_INVALID_ARG in the device error word); a token outside
 *           [0, V) is rejected
 *   accept_len out, int32 [N] (accepted drafts, 0..G); next_token out, int32 [N]
 *   ws      dfl_workspace_size(DFL_OP_SPEC_ACCEPT) bytes (N, G and V of the shape)
 *   Errors: INVALID_ARG, MISALIGNED (logits, vlog or ws), WORKSPACE.
 */
dfl_status dfl_spec_accept(const float* logits, float T, const void* vlog, dfl_dtype dt,
                           const int32_t* drafts, const int32_t* sel, int32_t N, int32_t K,
                           int32_t G, int32_t V, uint64_t seed, int32_t* accept_len,
                           int32_t* next_token, void* ws, size_t ws_bytes, dfl_stream stream);

/*
 * dfl_sampled_greedy_accept -- greedy acceptance against the verifier's own
 *   samples (SpecDiff-2 notes, "Self-Selection Acceptance" and "Streak-
 *   Distillation", read at temperature above zero).  For j = 1..G the
 *   verifier draws y_j from P_j = softmax(v_j) by inverse CDF; x_j is accepted
 *   while x_j == y_j.  The committed token is the verifier's sample at the
 *   first mismatch, or y_{G+1} (row G) after G acceptances.  Draft
 *   probabilities are not used; the expected number accepted is the streak
 *   sum of P_j(x_j), the quantity self-selection maximises.  Uniforms: u =
 *   ((x0 >> 8) + 1/2) 2^-24 of Philox4x32-10 at counter (n, j, 0, 3), key
 *   (seed lo, seed hi).
 *   vlog    in, dt [N][K][G+1][V]; drafts in, int32 [N][K][G]
 *   sel     in, int32 [N] draft to verify (nullable: draft 0; an index
 *           outside 0..K-1 is read as draft 0 and records DFL_ERR_INVALID_ARG
 *           in the device error word)
 *   accept_len out, int32 [N] (0..G); next_token out, int32 [N]
 *   ws      dfl_workspace_size(DFL_OP_SAMPLED_GREEDY) bytes (N, G, V)
 *   Errors: INVALID_ARG (K outside 1..64, G outside 1..1024), MISALIGNED
 *   (vlog or ws), WORKSPACE, UNSUPPORTED_SHAPE (V above 536,862,720).
 */
dfl_status dfl_sampled_greedy_accept(const void* vlog, dfl_dtype dt, const int32_t* drafts,
                                     const int32_t* sel, int32_t N, int32_t K, int32_t G,
                                     int32_t V, uint64_t seed, int32_t* accept_len,
                                     int32_t* next_token, void* ws, size_t ws_bytes,
                                     dfl_stream stream);

/*
 * dfl_philox4x32_10 -- the library's device Philox4x32-10 (Salmon, Moraes,
 *   Dror & Shaw, SC'11), the generator behind every uniform the sampling and
 *   acceptance calls draw, for checks against the published known-answer
 *   vectors.  in: device uint32 [n][6] = counter words 0..3, key words 0..1;
 *   out: device uint32 [n][4] output words.  Errors: INVALID_ARG.
 */
dfl_status dfl_philox4x32_10(const uint32_t* in, int32_t n, uint32_t* out, dfl_stream stream);

/*
 * dfl_block_ffn -- residual SwiGLU feed-forward block of a full draft layer.
 *   Reading (the pages give no width or form; the DFlash article's drafter
 *   layers are decoder layers of the target family): Qwen-style gate/up/down
 *     Xn = RMSNorm(Xb; ffn_gain),  Xb <- Xb + (silu(Xn W1^T) * (Xn W3^T)) W2^T
 *   Xb   in/out, fp32 [N*B][d]
 *   W1, W3 in, dt [F][d]; W2 in, dt [d][F]; ffn_gain in, fp32 [d]
 *   ws   dfl_workspace_size(DFL_OP_BLOCK_FFN) bytes (normalised rows, the
 *        [N*B][F] hidden activations, then, bf16, fp32 partials of the down
 *        projection split along K; a buffer without room for the partials
 *        is accepted and the projection then runs unsplit)
 *   bf16: one tensor-core GEMM for gate and up with the SwiGLU in its
 *   epilogue (needs F % 64 == 0), then the down projection with a residual
 *   epilogue.  fp32: CUDA-core GEMMs.
 *   Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, WORKSPACE.
 */
dfl_status dfl_block_ffn(float* Xb, int32_t N, int32_t B, int32_t d, dfl_dtype dt,
                         const float* ffn_gain, float eps, const void* W1, const void* W3,
                         const void* W2, int32_t F, void* ws, size_t ws_bytes, dfl_stream stream);

/* One draft layer's weights (device pointers, dtype of the step). */
typedef struct dfl_layer_weights {
    const void* Wq;   /* [Hq*hd][d] */
    const void* Wkc;  /* [Hkv*hd][d] */
    const void* Wvc;  /* [Hkv*hd][d] */
    const void* Wkb;  /* [Hkv*hd][d] */
    const void* Wvb;  /* [Hkv*hd][d] */
    const void* Wo;   /* [d][Hq*hd] */
    const void* W1;   /* [F][d] FFN gate, or NULL when the step's F == 0 */
    const void* W3;   /* [F][d] FFN up */
    const void* W2;   /* [d][F] FFN down */
} dfl_layer_weights;

/* Arguments of a whole draft step.  Host struct; tensors are device memory. */
typedef struct dfl_step_args {
    int32_t N, C, B, d, Hq, Hkv, hd, D, L, V;
    int32_t dtype;                 /* a dfl_dtype */
    float eps;
    const void* H;                 /* in [L][N*C][d] */
    int64_t h_layer_stride;        /* elements between target-layer slabs */
    const float* mix_logits;       /* in [D][L] */
    const float* mix_gain;         /* in [D][d] */
    const float* blk_gain;         /* in [D][d] */
    const float* final_gain;       /* in [d] */
    const float* rope;             /* in [C+B][hd/2][2] or NULL */
    const dfl_layer_weights* layers;  /* HOST array [D] */
    const void* W_lm;              /* in [V][d]; NULL when V == 0 */
    const float* Xb0;              /* in [N][B][d] anchor + [MASK] features */
    float* Xb;                     /* out [N][B][d] residual stream after D layers */
    int32_t* draft;                /* out [N][B-1] argmax drafts (V > 0) */
    float* logits;                 /* out, nullable: [N*(B-1)][V] */
    const int32_t* target;         /* in, nullable: [N][B] target argmax tokens */
    int32_t* accept_len;           /* out [N] when target != NULL */
    int32_t* bonus;                /* out [N] when target != NULL */
    const dfl_sample_params* sample;  /* HOST, nullable: K-draft sampling */
    int32_t* samples;              /* out [N][K][B-1] when sample != NULL */
    const void* vlog;              /* in, nullable: [N][K][B][V] verifier logits */
    float* scores;                 /* out [N][K] when vlog != NULL */
    int32_t* selected;             /* out [N] when vlog != NULL */
    /* Optional epilogues after self-selection (vlog != NULL): */
    float* tv_alpha;               /* out, nullable: [N][K][B-1] TV acceptance proxy */
    float* tv_tokens;              /* out, nullable: [N][K] streak sum of tv_alpha */
    int32_t accept_rule;           /* 0: greedy on the selected draft; 1: lossless
                                      stochastic acceptance (dfl_spec_accept); 2:
                                      sampled-greedy acceptance
                                      (dfl_sampled_greedy_accept); the accepted
                                      length and next token of rules 1 and 2
                                      replace accept_len / bonus */
    uint64_t accept_seed;          /* Philox key of rules 1 and 2 */
    int32_t F;                     /* FFN width; 0: layers without a feed-forward block */
    const float* ffn_gain;         /* in [D][d] when F > 0 */
    const void* W_fc;              /* in, nullable: [d][L*d] DFlash fusion (dfl_fc_fuse);
                                      when set, one fused representation is every
                                      layer's context features and mix_logits /
                                      mix_gain are unused */
    const float* fc_gain;          /* in [d] when W_fc != NULL */
} dfl_step_args;

/*
 * dfl_draft_step -- the whole single-pass draft step on one stream.
 *   DFlare post / DFlash article: one block forward through D draft layers
 *   (dfl_layer_mix_rmsnorm once for all layers, then per layer
 *   dfl_dual_kv_proj and dfl_block_attn), the LM head (dfl_lm_head_argmax on
 *   the B-1 mask rows) and the acceptance epilogue: dfl_greedy_accept against
 *   `target`, or, with `sample` and `vlog`, sampling plus dfl_self_select
 *   (whose results replace accept_len/bonus).  V == 0 stops after the layers.
 *   ws: dfl_workspace_size(DFL_OP_DRAFT_STEP) bytes holding the mixed context
 *   features of all D layers and each layer's Q/K/V.
 *   Errors: those of the calls it makes.  Null pointers, sizes, the 16-byte
 *   rule of every pointer and the shape rules that hold for both dtypes are
 *   checked before anything is launched.  A shape that one kernel does not
 *   take (UNSUPPORTED_SHAPE, e.g. a bf16 width outside a tile rule) can be
 *   found after earlier calls of the step were queued; the outputs are then
 *   undefined.
 */
dfl_status dfl_draft_step(const dfl_step_args* args, void* ws, size_t ws_bytes,
                          dfl_stream stream);

/*
 * dfl_draft_step_host -- dfl_draft_step with the target hidden states in host
 *   memory: the same results, bit for bit, as dfl_draft_step on a device copy
 *   of args->H.  The copy is issued here, in `chunks` groups of whole
 *   sequences on a copy stream the library owns (created on the first call),
 *   and each group's mix and context K/V projections of all D layers run as
 *   soon as its rows have landed, so they overlap the copy of the next group;
 *   with greedy drafts (no `sample`) the group's block rows, LM head and
 *   acceptance follow at once too (sequences are independent), otherwise
 *   they run for all sequences after the last group.  bf16 only.
 *   args->H   in, HOST [L][N*C][d] bf16 with args->h_layer_stride (pinned
 *             memory, or the copies are not asynchronous)
 *   H_dev     device buffer of the same layout, overwritten (the copy stream
 *             first waits for the work already queued on `stream`)
 *   chunks    number of groups, >= 1 (above min(N, 16) it is taken as that)
 *   ws        dfl_workspace_size(DFL_OP_DRAFT_STEP_HOST) bytes: the step's
 *             workspace plus the context K/V of every layer
 *   Calls on one device from several host threads are issued one at a time
 *   (they share the copy stream and its events); their work still runs on
 *   their own streams.
 *   Errors: as dfl_draft_step; UNSUPPORTED_SHAPE for fp32 or shapes the bf16
 *   tensor-core path does not take.
 */
dfl_status dfl_draft_step_host(const dfl_step_args* args, void* H_dev, int32_t chunks, void* ws, size_t ws_bytes,
                               dfl_stream stream);

/* Per-layer context K/V cache of a batch of sequences.  Host struct; the
 * tensors are device memory owned by the caller. */
typedef struct dfl_ctx_cache {
    void* K;                 /* in/out [D][N][C][Hkv][hd] (C = args->C, the capacity) */
    void* V;                 /* in/out, same layout as K */
    int64_t layer_stride;    /* elements between the draft layers' slabs, >= N*C*Hkv*hd */
    int32_t R;               /* rows per sequence of args->H this step, >= 1 */
    int32_t* ctx_len;        /* in/out device [N]: positions already cached */
    const int32_t* n_new;    /* in device [N]: valid new rows of each sequence, <= R */
    int32_t advance;         /* nonzero: ctx_len[n] += n_new[n] during the step */
} dfl_ctx_cache;

/*
 * dfl_draft_step_cached -- the draft step with an incremental context K/V
 * cache.  SpecDiff-2 notes, "Future work and limitations" (hardware
 * optimisation): the drafter lacks KV-cache support for its gamma-length
 * drafts.  A context key/value is a row-wise function of that position's
 * target hidden states and of its position, so the keys/values of positions
 * seen in earlier steps are kept and only the positions that arrive with this
 * step are mixed and projected.
 *   For sequence n with c0 = ctx_len[n] and m = n_new[n], rows 0..m-1 of its
 *   R-row slot of H (args->H is [L][N*R][d]; rows m..R-1 are ignored) are the
 *   target hidden states of positions c0..c0+m-1.  Every draft layer
 *   appends their rotated keys and their values at rows c0..c0+m-1 of its
 *   cache, then runs the block over the c0+m cached positions with the
 *   block at positions c0+m..c0+m+B-1; the rest is dfl_draft_step.
 *   args: as dfl_draft_step, with C the cache capacity per sequence and
 *   args->rope holding C+B positions.  bf16 only.
 *   ws: dfl_workspace_size(DFL_OP_DRAFT_STEP_CACHED) bytes, the shape's C the
 *   capacity and R the rows per sequence.
 *   Errors: host-side as dfl_draft_step, UNSUPPORTED_SHAPE for fp32.  A
 *   sequence whose lengths are out of range on the device (c0 < 0, m < 0,
 *   m > R or c0 + m > C) records DFL_ERR_INVALID_ARG in the device error
 *   word and appends nothing; its block runs over min(max(c0, 0), C) cached
 *   positions.
 */
dfl_status dfl_draft_step_cached(const dfl_step_args* args, const dfl_ctx_cache* cache,
                                 void* ws, size_t ws_bytes, dfl_stream stream);

/* Synchronise `stream`, then read and clear this device's error word (DFL_OK
 * if no kernel recorded an error). */
dfl_status dfl_get_device_error(dfl_stream stream, int32_t* code);

/* Upper bound, in nanoseconds, on any single device-side wait (mbarrier or
 * flag) in subsequently launched kernels.  Default 2e9 (2 s); process-wide.
 * Errors: INVALID_ARG for 0. */
dfl_status dfl_set_wait_limit_ns(uint64_t ns);

/* Self-test of the bounded wait: launches one block that waits on an
 * mbarrier no thread arrives at, for at most limit_ns; the kernel records
 * DFL_ERR_TIMEOUT in *status_out (device int32) and returns.  Used by tests
 * to show that a wait which runs out leaves the context usable.
 * Errors: INVALID_ARG (status_out NULL, limit_ns 0 or above 1e10),
 * NO_DEVICE, CUDA. */
dfl_status dfl_selftest_bounded_wait(uint64_t limit_ns, int32_t* status_out,
                                     dfl_stream stream);

/*
 * Kernel tracing.  While enabled, every kernel the library launches is
 * bracketed by a pair of CUDA events recorded on its stream (events come from
 * a pool the library owns; no device memory is allocated).
 * dfl_profile_enable(1) clears earlier records; dfl_profile_enable(0) stops
 * recording.  dfl_profile_report() waits for the recorded events, writes
 * {"kernel": [launches, total_ms], ...} as JSON into buf (truncated to
 * buf_len, NUL-terminated), stores the number of launches in *launches
 * (nullable) and clears the records.
 * Errors: INVALID_ARG (buf NULL or buf_len 0), CUDA.
 */
dfl_status dfl_profile_enable(int32_t on);
dfl_status dfl_profile_report(char* buf, size_t buf_len, int32_t* launches);

#ifdef __cplusplus
}
#endif
#endif /* DFL_H */
