// Host launchers of the draft step's smaller kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dfl.h"

namespace dfl {

struct DevErr;

dfl_status rope_table(float* table, int P, int hd, double theta, cudaStream_t st);
// out[m] = RMSNorm(in[(m / per) * stride + off + m % per]) * gain; bf16 or fp32 out.
// copy (nullable): each input row is also written, unchanged, to the same row of copy.
dfl_status rmsnorm_rows(const float* in, int d, int64_t M, int per, int stride, int off, const float* gain,
                        float eps, void* out, bool bf16, cudaStream_t st, float* copy = nullptr);
// Row plan of a cached draft step: per-row positions and cache rows of the
// new context rows, block positions and the attended context lengths.
dfl_status cache_plan(int N, int R, int B, int C, int32_t* ctx_len, const int32_t* n_new, int advance,
                      int32_t* pos_ctx, int32_t* dst_ctx, int32_t* pos_blk, int32_t* len_new, DevErr err,
                      cudaStream_t st);
dfl_status greedy_accept(const int32_t* draft, const int32_t* target, int N, int n, int32_t* accept_len,
                         int32_t* bonus, cudaStream_t st);
dfl_status argmax_combine(const float* pmax, const int* pidx, int64_t M, int tiles, int32_t* out,
                          cudaStream_t st);
dfl_status sample_rows(const float* logits, int64_t ld, const float* pmax, const double* psum, int64_t M, int per,
                       int tiles, int bn, int V, int K, float T, uint64_t seed, int32_t* samples, cudaStream_t st);
dfl_status tile_partials(const float* logits, int64_t ld, int64_t M, int V, int bn, int tiles, float inv_T,
                         float* pmax, int* pidx, double* psum, cudaStream_t st);
dfl_status rope_inplace_f32(float* x, int64_t rows, int heads, int hd, int per, int pos_off, const float* rope,
                            cudaStream_t st);
dfl_status attn_f32(const float* Q, const float* Kc, const float* Vc, const float* Kb, const float* Vb, int N, int C,
                    int B, int Hq, int Hkv, int hd, float* O, cudaStream_t st);
dfl_status selftest_wait(int* status, uint64_t limit_ns, cudaStream_t st);
dfl_status swiglu_f32(const float* gate, const float* up, float* h, int64_t n, cudaStream_t st);

// bf16 block attention (tensor cores); writes O bf16 [N*B][Hq*hd].  ws holds
// split-KV partials when more than one split is used.
int attn_splits(int N, int C, int B, int Hkv);
// Scratch of attn_bf16; `ragged`: per-sequence context lengths (C the capacity).
size_t attn_ws_bytes(int N, int C, int B, int Hq, int Hkv, int hd, bool ragged = false);
// tcgen05 attention (block_attn_tc.cu): shapes it serves, its scratch, launch.
bool attn_tc_supported(int B, int Hq, int Hkv, int hd);
int attn_tc_kps(int units, int C, int B, bool ragged);   // units: (sequence, K/V head, head subset)
size_t attn_tc_ws_bytes(int N, int C, int B, int Hq, int Hkv, int hd, bool ragged);
dfl_status attn_tc(const void* Q, const void* Kc, const void* Vc, const void* Kb, const void* Vb, int N, int C,
                   int B, int Hq, int Hkv, int hd, void* O, void* ws, cudaStream_t st, const int32_t* ctx_len,
                   int C_stride, int policy_N = 0);
// ctx_len (nullable, device [N]): per-sequence context keys, with C the
// maximum (C_stride context rows per sequence in Kc / Vc).
dfl_status attn_bf16(const void* Q, const void* Kc, const void* Vc, const void* Kb, const void* Vb, int N, int C,
                     int B, int Hq, int Hkv, int hd, void* O, void* ws, cudaStream_t st,
                     const int32_t* ctx_len = nullptr, int C_stride = 0, int policy_N = 0);
// policy_N (0: N): the batch size that decides how keys are split over work
// items, so that a call on a group of sequences splits them as a call on the
// whole batch of policy_N sequences would (same arithmetic, same bits).

// TV acceptance diagnostic and stochastic acceptance (workspace bytes)
size_t tv_ws_bytes(int N, int K, int G);
size_t spec_ws_bytes(int N, int G, int V);
size_t spec_scratch_bytes(int N, int V);
dfl_status lse_rows_f32(const float* logits, int rows, int V, float inv_T, float* lse, cudaStream_t st);
dfl_status tv_run(const float* logits, float inv_T, const void* vlog, bool bf, int N, int K, int G, int V,
                  float* alpha, float* tpd, const float* lse_z, const float* lse_v_all, cudaStream_t st);
dfl_status spec_run(const float* logits, float inv_T, const void* vlog, bool bf, const int32_t* drafts,
                    const int32_t* sel, int N, int K, int G, int V, uint64_t seed, int32_t* accept_len,
                    int32_t* next_token, const float* lse_z, const float* lse_v, bool lse_all, void* scratch,
                    cudaStream_t st);

// sampled-greedy acceptance: scratch of sg_run, workspace of the entry point
size_t sg_scratch_bytes(int N, int G, int V);
size_t sg_ws_bytes(int N, int G, int V);
dfl_status sg_run(const void* vlog, bool bf, const int32_t* drafts, const int32_t* sel, int N, int K, int G, int V,
                  uint64_t seed, int32_t* accept_len, int32_t* next_token, const float* lse_v, bool lse_all,
                  void* scratch, cudaStream_t st);
// Philox4x32-10 of n (counter, key) sextuples (device [n][6] -> [n][4])
dfl_status philox_block(const uint32_t* in, int n, uint32_t* out, cudaStream_t st);

// self-selection
size_t select_ws_bytes(int N, int K, int G);
dfl_status self_select_run(const void* vlog, bool bf16, const int32_t* drafts, int N, int K, int G, int V,
                           float* scores, int32_t* selected, int32_t* accept_len, int32_t* bonus, void* ws,
                           cudaStream_t st);

}  // namespace dfl
