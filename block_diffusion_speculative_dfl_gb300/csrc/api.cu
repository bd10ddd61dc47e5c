// C-ABI entry points of libdfl: argument checks, workspace layout and the
// order of kernel launches for each operation of the draft step.
#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <initializer_list>
#include <mutex>
#include <string>
#include <vector>

#include "internal.h"
#include "small_kernels.h"

// Per-device error word: the first kernel that records an error wins.
__device__ int g_dfl_error_word;

namespace dfl {

namespace {
std::atomic<uint64_t> g_wait_ns{2000000000ull};
constexpr int kMaxDevices = 64;
DeviceCtx g_ctx[kMaxDevices];
std::atomic<bool> g_ready[kMaxDevices];
std::mutex g_mu;

inline size_t al256(size_t b) { return (b + 255) & ~size_t(255); }
inline size_t esz(int dt) { return dt == DFL_BF16 ? 2 : 4; }
inline uint8_t* carve(uint8_t*& p, size_t bytes) {
    uint8_t* r = p;
    p += al256(bytes);
    return r;
}
}  // namespace

// Unique id of the CUDA context current on this thread (0 if none or unknown),
// through the driver's cuCtxGetCurrent / cuCtxGetId.
uint64_t current_context_id() {
    using GetCurrentFn = CUresult (*)(CUcontext*);
    using GetIdFn = CUresult (*)(CUcontext, unsigned long long*);
    static GetCurrentFn get_current = nullptr;
    static GetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrentFn>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetIdFn>(p);
    });
    CUcontext c = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&c) != CUDA_SUCCESS || !c || get_id(c, &id) != CUDA_SUCCESS) return 0;
    return id;
}

DeviceCtx* current_ctx() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    const uint64_t cid = current_context_id();
    if (g_ready[dev].load(std::memory_order_acquire) && cid != 0 && g_ctx[dev].ctx_id.load() == cid)
        return &g_ctx[dev];
    std::lock_guard<std::mutex> lk(g_mu);
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return nullptr;
    if (major != 10 || minor != 3) return nullptr;   // kernels are built for sm_103a only
    DeviceCtx& c = g_ctx[dev];
    // Looking the symbol up binds the runtime's context, so its id is read after.
    int* word = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&word), g_dfl_error_word) != cudaSuccess) return nullptr;
    const uint64_t now = current_context_id();
    if (g_ready[dev].load(std::memory_order_relaxed) && c.ctx_id.load() == now) return &c;
    // First use on this device, or another context than the one the entry was
    // set up in: what belonged to the old context (function attributes, the
    // copy stream and its events) is dropped, not destroyed -- it went with
    // its context.
    {
        std::lock_guard<std::mutex> hk(c.host_mu);
        c.copy_st = nullptr;
        for (cudaEvent_t& e : c.copy_ev) e = nullptr;
    }
    for (auto& f : c.gemm_attr_set) f = false;
    for (auto& f : c.attn_attr_set) f = false;
    c.mix_attr_set = false;
    c.err_word = word;
    c.device = dev;
    c.sm_count = sms;
    c.ctx_id.store(now);
    g_ready[dev].store(true, std::memory_order_release);
    return &c;
}

DevErr dev_err(DeviceCtx* ctx) { return DevErr{ctx->err_word, g_wait_ns.load()}; }

bool pdl_on() {
    static const bool on = [] {
        const char* e = std::getenv("DFL_PDL");
        return !(e && e[0] == '0');
    }();
    return on;
}
uint64_t wait_limit_ns() { return g_wait_ns.load(); }

// ------------------------------------------------------------ workspaces

size_t ws_dual_kv_proj(int N, int B, int d, int dt) { return al256((size_t)N * B * d * esz(dt)); }

// fp32 partials of the output projection's K-split (up to 8 splits of
// [rows][d]); 0 when d is not given.
size_t ws_oproj_split(int64_t rows, int d) { return d > 0 ? al256((size_t)8 * rows * d * 4) : 0; }

// The attention output and scratch, then (optional: used when the caller's
// workspace holds it) room for the output projection's K-split partials.
size_t ws_block_attn(int N, int C, int B, int Hq, int Hkv, int hd, int dt, bool ragged = false, int d = 0) {
    size_t b = al256((size_t)N * B * Hq * hd * esz(dt));
    if (dt == DFL_BF16) b += al256(attn_ws_bytes(N, C, B, Hq, Hkv, hd, ragged)) + ws_oproj_split((int64_t)N * B, d);
    return b;
}

// fp32 pre-norm features of the DFlash fusion, [rows][d]
size_t ws_fc_fuse(int64_t rows, int d) { return al256((size_t)rows * d * 4); }

// Normalised rows and hidden activations, then (bf16, with_split: used when
// the caller's workspace holds it) room for the down projection's K-split
// partials.
size_t ws_block_ffn(int N, int B, int d, int F, int dt, bool with_split = false) {
    const size_t M = (size_t)N * B;
    if (dt == DFL_BF16) return al256(M * d * 2) + al256(M * F * 2) + (with_split ? ws_oproj_split((int64_t)M, d) : 0);
    return al256(M * d * 4) + 3 * al256(M * F * 4);
}

size_t ws_lm_head(int N, int B, int row0, int d, int V, int dt, bool logits_missing) {
    const size_t M = (size_t)N * (B - row0);
    const size_t tiles = (size_t)(V + 255) / 256;
    size_t b = al256(M * d * esz(dt)) + al256(M * tiles * 4) * 2 + al256(M * tiles * 8);
    if (logits_missing) b += al256(M * (size_t)V * 4);
    return b;
}

// Workspace of a whole draft step: the mixed context features of all D
// layers, Q / (Kc, Vc) / Kb / Vb, the cached step's row plan, samples and
// drafts, then scratch shared by the calls in turn.  The cached step mixes
// and projects R rows per sequence, keeps K/V in the caller's cache (C is its
// capacity) and, when sampling, lends the feature area to the logits.
size_t step_ws_bytes(const dfl_shape& s, bool cached);

// Host-input step: the plain step's workspace, then the context K/V of layers
// 1..D-1 (layer 0's are the plain step's Kc / Vc).
size_t kv_layer_bytes(const dfl_shape& s) { return al256((size_t)s.N * s.C * s.Hkv * s.hd * 2); }
size_t step_host_ws_bytes(const dfl_shape& s) {
    if (s.dtype != DFL_BF16 || s.D < 1) return 0;
    return step_ws_bytes(s, false) + (size_t)(s.D - 1) * 2 * kv_layer_bytes(s);
}

size_t step_ws_bytes(const dfl_shape& s, bool cached) {
    if (cached && (s.dtype != DFL_BF16 || s.R < 1)) return 0;
    const size_t e = esz(s.dtype);
    const int64_t rows = (int64_t)s.N * (cached ? s.R : s.C);   // context rows mixed this step
    // per-layer mixtures of all D layers, or one fused representation and its
    // fp32 pre-norm features (DFlash fusion)
    size_t xc = s.fc ? al256((size_t)rows * s.d * e) + ws_fc_fuse(rows, s.d) : (size_t)s.D * rows * s.d * e;
    if (cached && s.V > 0 && s.K > 0) xc = std::max(xc, (size_t)s.N * (s.B - 1) * s.V * 4);
    size_t b = al256(xc);
    b += al256((size_t)s.N * s.B * s.Hq * s.hd * e);                         // Q
    if (!cached) b += 2 * al256((size_t)s.N * s.C * s.Hkv * s.hd * e);       // Kc, Vc
    b += 2 * al256((size_t)s.N * s.B * s.Hkv * s.hd * e);                    // Kb, Vb
    if (cached) b += 2 * al256((size_t)rows * 4) + al256((size_t)s.N * s.B * 4) + al256((size_t)s.N * 4);
    size_t sub = ws_dual_kv_proj(s.N, s.B, s.d, s.dtype);
    sub = std::max(sub, ws_block_attn(s.N, s.C, s.B, s.Hq, s.Hkv, s.hd, s.dtype, cached, s.d));
    if (s.F > 0) sub = std::max(sub, ws_block_ffn(s.N, s.B, s.d, s.F, s.dtype, true));
    if (s.V > 0) {
        sub = std::max(sub, ws_lm_head(s.N, s.B, 1, s.d, s.V, s.dtype, true));
        if (s.K > 0) {
            // self-selection scratch (its verifier-row LSEs are reused), drafter-row LSEs,
            // stochastic-acceptance scratch
            sub = std::max(sub, al256(select_ws_bytes(s.N, s.K, s.B - 1)) + al256((size_t)s.N * (s.B - 1) * 4) +
                                    std::max(spec_scratch_bytes(s.N, s.V), sg_scratch_bytes(s.N, s.B - 1, s.V)));
            b += al256((size_t)s.N * s.K * (s.B - 1) * 4);                   // samples
        }
        b += al256((size_t)s.N * (s.B - 1) * 4);                             // drafts
    }
    return b + sub;
}

}  // namespace dfl

using namespace dfl;

// ------------------------------------------------------------------ misc

extern "C" const char* dfl_version(void) { return "dfl 0.1.0 (sm_103a)"; }

extern "C" const char* dfl_status_string(dfl_status s) {
    switch (s) {
        case DFL_OK: return "ok";
        case DFL_ERR_INVALID_ARG: return "invalid argument";
        case DFL_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case DFL_ERR_MISALIGNED: return "pointer or size not 16-byte aligned";
        case DFL_ERR_WORKSPACE: return "workspace too small";
        case DFL_ERR_CUDA: return "CUDA call or launch failed";
        case DFL_ERR_TIMEOUT: return "device-side wait timed out";
        case DFL_ERR_NO_DEVICE: return "no sm_103a device is current";
        case DFL_ERR_BOUNDS: return "a kernel index fell outside its buffer (bounds-checked build); access skipped";
    }
    return "unknown status";
}

extern "C" size_t dfl_workspace_size(dfl_op op, const dfl_shape* s) {
    if (!s || (s->dtype != DFL_F32 && s->dtype != DFL_BF16)) return 0;
    // every size is a count: a negative one makes the shape invalid
    for (int32_t v : {s->N, s->C, s->B, s->d, s->Hq, s->Hkv, s->hd, s->D, s->L, s->V, s->K, s->G, s->row0, s->F, s->R,
                      s->fc})
        if (v < 0) return 0;
    switch (op) {
        case DFL_OP_DUAL_KV_PROJ: return ws_dual_kv_proj(s->N, s->B, s->d, s->dtype);
        case DFL_OP_BLOCK_ATTN: return ws_block_attn(s->N, s->C, s->B, s->Hq, s->Hkv, s->hd, s->dtype, false, s->d);
        case DFL_OP_LM_HEAD:
            if (s->row0 < 0 || s->row0 >= s->B || s->V <= 0) return 0;
            return ws_lm_head(s->N, s->B, s->row0, s->d, s->V, s->dtype, s->dtype == DFL_F32);
        case DFL_OP_SELF_SELECT: return al256(select_ws_bytes(s->N, s->K, s->G));
        case DFL_OP_TV_ACCEPTANCE: return tv_ws_bytes(s->N, s->K, s->G);
        case DFL_OP_SPEC_ACCEPT: return spec_ws_bytes(s->N, s->G, s->V);
        case DFL_OP_BLOCK_FFN: return s->F > 0 ? ws_block_ffn(s->N, s->B, s->d, s->F, s->dtype, true) : 0;
        case DFL_OP_DRAFT_STEP: return step_ws_bytes(*s, false);
        case DFL_OP_DRAFT_STEP_CACHED: return step_ws_bytes(*s, true);
        case DFL_OP_DRAFT_STEP_HOST: return step_host_ws_bytes(*s);
        case DFL_OP_FC_FUSE: return ws_fc_fuse((int64_t)s->N * s->C, s->d);
        case DFL_OP_SAMPLED_GREEDY: return sg_ws_bytes(s->N, s->G, s->V);
    }
    return 0;
}

extern "C" dfl_status dfl_get_device_error(dfl_stream stream, int32_t* code) {
    if (!code) return DFL_ERR_INVALID_ARG;
    DeviceCtx* ctx = current_ctx();
    if (!ctx) return DFL_ERR_NO_DEVICE;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return DFL_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_dfl_error_word, sizeof(int)) != cudaSuccess) return DFL_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_dfl_error_word, &zero, sizeof(int)) != cudaSuccess) return DFL_ERR_CUDA;
    *code = v;
    return DFL_OK;
}

extern "C" dfl_status dfl_set_wait_limit_ns(uint64_t ns) {
    if (ns == 0) return DFL_ERR_INVALID_ARG;
    g_wait_ns.store(ns);
    return DFL_OK;
}

extern "C" dfl_status dfl_selftest_bounded_wait(uint64_t limit_ns, int32_t* status_out, dfl_stream stream) {
    if (!status_out || limit_ns == 0 || limit_ns > 10000000000ull) return DFL_ERR_INVALID_ARG;
    if (!current_ctx()) return DFL_ERR_NO_DEVICE;
    return selftest_wait(status_out, limit_ns, static_cast<cudaStream_t>(stream));
}

extern "C" dfl_status dfl_rope_table(float* table, int32_t P, int32_t hd, double theta, dfl_stream stream) {
    const dfl::ApiRange nvtx_range("dfl_rope_table");
    if (!table || P <= 0 || hd <= 0 || (hd & 1) || !(theta > 0.0)) return DFL_ERR_INVALID_ARG;
    if (!current_ctx()) return DFL_ERR_NO_DEVICE;
    return rope_table(table, P, hd, theta, static_cast<cudaStream_t>(stream));
}

extern "C" dfl_status dfl_greedy_accept(const int32_t* draft, const int32_t* target, int32_t N, int32_t n,
                                        int32_t* accept_len, int32_t* bonus, dfl_stream stream) {
    const dfl::ApiRange nvtx_range("dfl_greedy_accept");
    if (!target || !accept_len || !bonus || N <= 0 || n < 0 || n > 1024 || (n > 0 && !draft))
        return DFL_ERR_INVALID_ARG;
    if (!current_ctx()) return DFL_ERR_NO_DEVICE;
    return greedy_accept(draft, target, N, n, accept_len, bonus, static_cast<cudaStream_t>(stream));
}

extern "C" dfl_status dfl_philox4x32_10(const uint32_t* in, int32_t n, uint32_t* out, dfl_stream stream) {
    const dfl::ApiRange nvtx_range("dfl_philox4x32_10");
    if (!in || !out || n <= 0) return DFL_ERR_INVALID_ARG;
    if (!current_ctx()) return DFL_ERR_NO_DEVICE;
    return philox_block(in, n, out, static_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------- DFlash fusion

namespace dfl {
namespace {
// Xc = RMSNorm([H_1 .. H_L] W_fc^T; gain): bf16 as one tensor-core GEMM over
// K = L*d whose A tiles come from the L slabs in turn (a 3-D tensor map),
// fp32 as L accumulating CUDA-core GEMMs; the fp32 pre-norm features F then
// go through the row RMSNorm.
dfl_status fc_fuse_impl(DeviceCtx* ctx, const void* H, int64_t layer_stride, int L, int64_t rows, int d, int dt,
                        const void* W_fc, const float* gain, float eps, void* Xc, float* F, cudaStream_t st) {
    dfl_status rc;
    if (dt == DFL_F32) {
        const float* h = static_cast<const float*>(H);
        const float* w = static_cast<const float*>(W_fc);
        for (int i = 0; i < L; ++i)
            if ((rc = gemm_f32_ld(h + (size_t)i * layer_stride, d, w + (size_t)i * d, (int64_t)L * d, F, (int)rows,
                                  d, d, d, i > 0, st)) != DFL_OK)
                return rc;
    } else {
        GemmArgs g{};
        g.A = H; g.M = (int)rows; g.K = L * d;
        g.a_slabs = L; g.a_slab_stride = L > 1 ? layer_stride : (int64_t)rows * d;
        g.B[0] = W_fc; g.b_rows[0] = d; g.b_begin[0] = 0; g.nb = 1; g.N = d;
        g.bn = 0;
        g.m_inner = 0;   // N-tiles innermost: the L slabs of an A row block are read from HBM once
        g.epi = EPI_RESID;
        g.ep.resid = F; g.ep.ld_resid = d; g.ep.resid_store = 1;
        g.tag = "gemm_fc_fuse";
        if ((rc = gemm_tc(ctx, g, st)) != DFL_OK) return rc;
    }
    return rmsnorm_rows(F, d, rows, 1, 1, 0, gain, eps, Xc, dt == DFL_BF16, st);
}

// Host-side checks shared by the entry point and the steps.
dfl_status fc_fuse_check(const void* H, int64_t layer_stride, int L, int64_t rows, int d, int dt, const void* W_fc,
                         const float* gain, const void* Xc) {
    if (!H || !W_fc || !gain || !Xc || L < 1 || L > 64 || rows <= 0 || d <= 0) return DFL_ERR_INVALID_ARG;
    if (dt != DFL_F32 && dt != DFL_BF16) return DFL_ERR_INVALID_ARG;
    if (L > 1 && layer_stride < rows * d) return DFL_ERR_INVALID_ARG;
    if (!rows_fit(rows) || (int64_t)L * d >= ((int64_t)1 << 31)) return DFL_ERR_UNSUPPORTED_SHAPE;
    const void* ptrs[] = {H, W_fc, gain, Xc};
    for (const void* p : ptrs) if (!aligned16(p)) return DFL_ERR_MISALIGNED;
    if (d % 8 != 0 || (layer_stride * (int64_t)esz(dt)) % 16 != 0) return DFL_ERR_MISALIGNED;
    if (dt == DFL_BF16 && d % 64 != 0) return DFL_ERR_UNSUPPORTED_SHAPE;
    if (d > 6144) return DFL_ERR_UNSUPPORTED_SHAPE;   // the row RMSNorm keeps a row in registers
    return DFL_OK;
}
}  // namespace
}  // namespace dfl

extern "C" dfl_status dfl_fc_fuse(const void* H, int64_t layer_stride, int32_t L, int64_t rows, int32_t d,
                                  dfl_dtype dt, const void* W_fc, const float* gain, float eps, void* Xc, void* ws,
                                  size_t ws_bytes, dfl_stream stream) {
    const dfl::ApiRange nvtx_range("dfl_fc_fuse");
    dfl_status rc = fc_fuse_check(H, layer_stride, L, rows, d, dt, W_fc, gain, Xc);
    if (rc != DFL_OK) return rc;
    if (!ws) return DFL_ERR_INVALID_ARG;
    if (!aligned16(ws)) return DFL_ERR_MISALIGNED;
    if (ws_bytes < ws_fc_fuse(rows, d)) return DFL_ERR_WORKSPACE;
    DeviceCtx* ctx = current_ctx();
    if (!ctx) return DFL_ERR_NO_DEVICE;
    return fc_fuse_impl(ctx, H, layer_stride, L, rows, d, dt, W_fc, gain, eps, Xc, static_cast<float*>(ws),
                        static_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------- dual projection

namespace dfl {
namespace {
// Row plan of the cached step: positions and cache rows of the new context
// rows, positions of the block rows (device arrays).
struct KvRowPlan {
    const int32_t* ctx_pos;
    const int32_t* ctx_dst;
    const int32_t* blk_pos;
    int64_t dst_rows;   // rows of the cache layer the context rows are scattered to
};

// bf16 projections of one draft layer: context rows [Kc | Vc] = Xc [Wkc ; Wvc]^T
// (ctx_M rows, ctx_per rows per sequence), block rows [Q | Kb | Vb] =
// RMSNorm(Xb) [Wq ; Wkb ; Wvb]^T, rotary embedding in the GEMM epilogues.
// Without a plan, context row r sits at position r % ctx_per and block row r
// at ctx_per + r % B; with one, the plan gives positions and context rows go
// to plan->ctx_dst (rows < 0 dropped).
// Context rows: [Kc | Vc] = Xc [Wkc ; Wvc]^T with rotary on Kc; row r of the
// call sits at position r % ctx_per (or at plan->ctx_pos[r]).
GemmArgs ctx_kv_args(const void* Xc, int64_t ctx_M, int ctx_per, int d, const void* Wkc, const void* Wvc, int Hkv,
                     int hd, const float* rope, void* Kc, void* Vc, const KvRowPlan* plan) {
    const int kv = Hkv * hd;
    GemmArgs gc{};
    gc.A = Xc; gc.M = (int)ctx_M; gc.K = d;
    gc.B[0] = Wkc; gc.B[1] = Wvc; gc.b_rows[0] = kv; gc.b_rows[1] = kv;
    gc.b_begin[0] = 0; gc.b_begin[1] = kv; gc.nb = 2; gc.N = 2 * kv;
    gc.bn = 0;   // chosen per shape (the grouped launch picks one width for both problems)
    gc.m_inner = 0;
    gc.epi = EPI_STORE;
    const int64_t out_rows = plan ? plan->dst_rows : ctx_M;
    gc.ep.seg[0] = GemmSeg{Kc, 0, kv, rope != nullptr, out_rows};
    gc.ep.seg[1] = GemmSeg{Vc, kv, kv, 0, out_rows};
    gc.ep.nseg = 2;
    gc.ep.rope = rope; gc.ep.hd = hd; gc.ep.rows_per_seq = ctx_per; gc.ep.pos_off = 0;
    if (plan) { gc.ep.row_pos = plan->ctx_pos; gc.ep.row_dst = plan->ctx_dst; }
    gc.tag = plan ? "gemm_ctx_kv_append" : "gemm_ctx_kv";
    return gc;
}

dfl_status dual_kv_proj_bf16(DeviceCtx* ctx, const void* Xc, int64_t ctx_M, int ctx_per, const float* Xb, int N,
                             int B, int d, const float* blk_gain, float eps, const void* Wq, const void* Wkc,
                             const void* Wvc, const void* Wkb, const void* Wvb, int Hq, int Hkv, int hd,
                             const float* rope, void* Q, void* Kc, void* Vc, void* Kb, void* Vb, void* ws,
                             const KvRowPlan* plan, cudaStream_t st, const float* Xb_init = nullptr) {
    const int kv = Hkv * hd, qd = Hq * hd;
    dfl_status rc;
    void* Xn = ws;
    // With Xb_init the block's initial features are normalised from there and
    // copied into the residual stream Xb by the same kernel (a step's first layer).
    if ((rc = rmsnorm_rows(Xb_init ? Xb_init : Xb, d, (int64_t)N * B, 1, 1, 0, blk_gain, eps, Xn, true, st,
                           Xb_init ? const_cast<float*>(Xb) : nullptr)) != DFL_OK)
        return rc;

    // block rows: [Q | Kb | Vb] = Xn [Wq ; Wkb ; Wvb]^T
    GemmArgs gb{};
    gb.A = Xn; gb.M = N * B; gb.K = d;
    gb.B[0] = Wq; gb.B[1] = Wkb; gb.B[2] = Wvb;
    gb.b_rows[0] = qd; gb.b_rows[1] = kv; gb.b_rows[2] = kv;
    gb.b_begin[0] = 0; gb.b_begin[1] = qd; gb.b_begin[2] = qd + kv; gb.nb = 3; gb.N = qd + 2 * kv;
    gb.bn = 0;   // chosen per shape
    gb.m_inner = 1;
    gb.epi = EPI_STORE;
    gb.ep.seg[0] = GemmSeg{Q, 0, qd, rope != nullptr, (int64_t)N * B};
    gb.ep.seg[1] = GemmSeg{Kb, qd, kv, rope != nullptr, (int64_t)N * B};
    gb.ep.seg[2] = GemmSeg{Vb, qd + kv, kv, 0, (int64_t)N * B};
    gb.ep.nseg = 3;
    gb.ep.rope = rope; gb.ep.hd = hd; gb.ep.rows_per_seq = B; gb.ep.pos_off = ctx_per;
    if (plan) gb.ep.row_pos = plan->blk_pos;
    gb.tag = "gemm_block_qkv";
    if (ctx_M <= 0) return gemm_tc(ctx, gb, st);

    const GemmArgs gc = ctx_kv_args(Xc, ctx_M, ctx_per, d, Wkc, Wvc, Hkv, hd, rope, Kc, Vc, plan);
    // One launch for both: the block projection's weights stream from HBM on a
    // few SMs while the others work on context tiles (block tiles first).
    return gemm_tc2(ctx, gb, gc, plan ? "gemm_kv_qkv_append" : "gemm_kv_qkv", st);
}

// bf16 block attention and output projection, Xb += Attn(Q, [Kc;Kb], [Vc;Vb]) Wo^T.
// ctx_len (nullable, device [N]): context keys of each sequence, C the maximum
// and C_stride the context rows per sequence of Kc / Vc.
dfl_status block_attn_bf16(DeviceCtx* ctx, const void* Q, const void* Kc, const void* Vc, const void* Kb,
                           const void* Vb, int N, int C, int B, int Hq, int Hkv, int hd, const void* Wo, int d,
                           float* Xb, void* ws, size_t ws_bytes, const int32_t* ctx_len, int C_stride,
                           cudaStream_t st, int policy_N = 0) {
    const int qd = Hq * hd;
    dfl_status rc;
    uint8_t* p = static_cast<uint8_t*>(ws);
    void* O = carve(p, (size_t)N * B * qd * 2);
    if ((rc = attn_bf16(Q, Kc, Vc, Kb, Vb, N, C, B, Hq, Hkv, hd, O, p, st, ctx_len, C_stride, policy_N)) != DFL_OK)
        return rc;
    GemmArgs g{};   // Xb += O Wo^T
    g.A = O; g.M = N * B; g.K = qd;
    g.B[0] = Wo; g.b_rows[0] = d; g.b_begin[0] = 0; g.nb = 1; g.N = d;
    g.bn = 0;   // chosen per shape
    g.m_inner = 1;
    g.epi = EPI_RESID;
    g.ep.resid = Xb; g.ep.ld_resid = d;
    g.tag = "gemm_o_proj";
    // The projection's few output tiles stream Wo through a few CTAs: when
    // the workspace has room, it is split along K (partials after the
    // attention's scratch) and summed in a fixed order.
    const size_t base = ws_block_attn(N, C, B, Hq, Hkv, hd, DFL_BF16, ctx_len != nullptr);
    const size_t room = ws_oproj_split((int64_t)N * B, d);
    if (room > 0 && ws_bytes >= base + room) {
        g.split_part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + base);
        g.split_part_bytes = room;
    }
    return gemm_tc(ctx, g, st);
}

}  // namespace
}  // namespace dfl


extern "C" dfl_status dfl_dual_kv_proj(const void* Xc, const float* Xb, int32_t N, int32_t C, int32_t B, int32_t d,
                                       dfl_dtype dt, const float* blk_gain, float eps, const void* Wq,
                                       const void* Wkc, const void* Wvc, const void* Wkb, const void* Wvb,
                                       int32_t Hq, int32_t Hkv, int32_t hd, const float* rope, void* Q, void* Kc,
                                       void* Vc, void* Kb, void* Vb, void* ws, size_t ws_bytes,
                                       dfl_stream stream) {
    const dfl::ApiRange nvtx_range("dfl_dual_kv_proj");
    if (N <= 0 || C < 0 || B <= 0 || d <= 0 || Hq <= 0 || Hkv <= 0 || hd <= 0 || Hq % Hkv != 0)
        return DFL_ERR_INVALID_ARG;
    if (dt != DFL_F32 && dt != DFL_BF16) return DFL_ERR_INVALID_ARG;
    if (!rows_fit((int64_t)N * C) || !rows_fit((int64_t)N * B)) return DFL_ERR_UNSUPPORTED_SHAPE;
    if (!Xb || !blk_gain || !Wq || !Wkb || !Wvb || !Q || !Kb || !Vb || !ws) return DFL_ERR_INVALID_ARG;
    if (C > 0 && (!Xc || !Wkc || !Wvc || !Kc || !Vc)) return DFL_ERR_INVALID_ARG;
    if (rope && (hd & 1)) return DFL_ERR_INVALID_ARG;
    const void* ptrs[] = {Xb, blk_gain, Wq, Wkb, Wvb, Q, Kb, Vb, ws, rope ? rope : Xb};
    for (const void* p : ptrs) if (!aligned16(p)) return DFL_ERR_MISALIGNED;
    if (C > 0) {
        const void* cp[] = {Xc, Wkc, Wvc, Kc, Vc};
        for (const void* p : cp) if (!aligned16(p)) return DFL_ERR_MISALIGNED;
    }
    if (d % 8 != 0 || hd % 8 != 0) return DFL_ERR_MISALIGNED;
    if (ws_bytes < ws_dual_kv_proj(N, B, d, dt)) return DFL_ERR_WORKSPACE;
    DeviceCtx* ctx = current_ctx();
    if (!ctx) return DFL_ERR_NO_DEVICE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int kv = Hkv * hd, qd = Hq * hd;
    dfl_status rc;

    if (dt == DFL_F32) {
        float* Xn = static_cast<float*>(ws);
        if ((rc = rmsnorm_rows(Xb, d, (int64_t)N * B, 1, 1, 0, blk_gain, eps, Xn, false, st)) != DFL_OK) return rc;
        const float* w[3] = {static_cast<const float*>(Wq), static_cast<const float*>(Wkb),
                             static_cast<const float*>(Wvb)};
        float* o[3] = {static_cast<float*>(Q), static_cast<float*>(Kb), static_cast<float*>(Vb)};
        const int nout[3] = {qd, kv, kv};
        for (int j = 0; j < 3; ++j)
            if ((rc = gemm_f32(Xn, w[j], o[j], N * B, nout[j], d, nout[j], 0, st)) != DFL_OK) return rc;
        if (C > 0) {
            const float* xc = static_cast<const float*>(Xc);
            if ((rc = gemm_f32(xc, static_cast<const float*>(Wkc), static_cast<float*>(Kc), N * C, kv, d, kv, 0,
                               st)) != DFL_OK)
                return rc;
            if ((rc = gemm_f32(xc, static_cast<const float*>(Wvc), static_cast<float*>(Vc), N * C, kv, d, kv, 0,
                               st)) != DFL_OK)
                return rc;
        }
        if (rope) {
            if ((rc = rope_inplace_f32(static_cast<float*>(Q), (int64_t)N * B, Hq, hd, B, C, rope, st)) != DFL_OK)
                return rc;
            if ((rc = rope_inplace_f32(static_cast<float*>(Kb), (int64_t)N * B, Hkv, hd, B, C, rope, st)) != DFL_OK)
                return rc;
            if (C > 0 &&
                (rc = rope_inplace_f32(static_cast<float*>(Kc), (int64_t)N * C, Hkv, hd, C, 0, rope, st)) != DFL_OK)
                return rc;
        }
        return DFL_OK;
    }

    // bf16: tensor-core GEMMs with the rotary embedding in the epilogue
    if (hd != 64 && hd != 128) return DFL_ERR_UNSUPPORTED_SHAPE;
    if (kv % 128 != 0 || qd % 128 != 0) return DFL_ERR_UNSUPPORTED_SHAPE;
    return dual_kv_proj_bf16(ctx, Xc, (int64_t)N * C, C, Xb, N, B, d, blk_gain, eps, Wq, Wkc, Wvc, Wkb, Wvb, Hq, Hkv,
                             hd, rope, Q, Kc, Vc, Kb, Vb, ws, nullptr, st);
}

// -------------------------------------------------------- block attention

extern "C" dfl_status dfl_block_attn(const void* Q, const void* Kc, const void* Vc, const void* Kb, const void* Vb,
                                     int32_t N, int32_t C, int32_t B, int32_t Hq, int32_t Hkv, int32_t hd,
                                     dfl_dtype dt, const void* Wo, int32_t d, float* Xb, void* ws, size_t ws_bytes,
                                     dfl_stream stream) {
    const dfl::ApiRange nvtx_range("dfl_block_attn");
    if (N <= 0 || C < 0 || B <= 0 || d <= 0 || Hq <= 0 || Hkv <= 0 || hd <= 0 || Hq % Hkv != 0)
        return DFL_ERR_INVALID_ARG;
    if (dt != DFL_F32 && dt != DFL_BF16) return DFL_ERR_INVALID_ARG;
    if (!rows_fit((int64_t)N * C) || !rows_fit((int64_t)N * B)) return DFL_ERR_UNSUPPORTED_SHAPE;
    if (!Q || !Kb || !Vb || !Wo || !Xb || !ws || (C > 0 && (!Kc || !Vc))) return DFL_ERR_INVALID_ARG;
    const void* ptrs[] = {Q, Kb, Vb, Wo, Xb, ws, C > 0 ? Kc : Q, C > 0 ? Vc : Q};
    for (const void* p : ptrs) if (!aligned16(p)) return DFL_ERR_MISALIGNED;
    if (d % 8 != 0 || hd % 8 != 0) return DFL_ERR_MISALIGNED;
    if (ws_bytes < ws_block_attn(N, C, B, Hq, Hkv, hd, dt)) return DFL_ERR_WORKSPACE;
    DeviceCtx* ctx = current_ctx();
    if (!ctx) return DFL_ERR_NO_DEVICE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int qd = Hq * hd;
    dfl_status rc;
    uint8_t* p = static_cast<uint8_t*>(ws);
    void* O = carve(p, (size_t)N * B * qd * esz(dt));
    if (dt == DFL_F32) {
        if (hd > 128) return DFL_ERR_UNSUPPORTED_SHAPE;
        if ((rc = attn_f32(static_cast<const float*>(Q), static_cast<const float*>(Kc), static_cast<const float*>(Vc),
                           static_cast<const float*>(Kb), static_cast<const float*>(Vb), N, C, B, Hq, Hkv, hd,
                           static_cast<float*>(O), st)) != DFL_OK)
            return rc;
        return gemm_f32(static_cast<const float*>(O), static_cast<const float*>(Wo), Xb, N * B, d, qd, d, 1, st);
    }
    if (hd != 64 && hd != 128) return DFL_ERR_UNSUPPORTED_SHAPE;
    if (d % 32 != 0) return DFL_ERR_UNSUPPORTED_SHAPE;
    return block_attn_bf16(ctx, Q, Kc, Vc, Kb, Vb, N, C, B, Hq, Hkv, hd, Wo, d, Xb, ws, ws_bytes, nullptr, C, st);
}

// ------------------------------------------------------- feed-forward

extern "C" dfl_status dfl_block_ffn(float* Xb, int32_t N, int32_t B, int32_t d, dfl_dtype dt, const float* ffn_gain,
                                    float eps, const void* W1, const void* W3, const void* W2, int32_t F, void* ws,
                                    size_t ws_bytes, dfl_stream stream) {
    const dfl::ApiRange nvtx_range("dfl_block_ffn");
    if (!Xb || !ffn_gain || !W1 || !W3 || !W2 || !ws || N <= 0 || B <= 0 || d <= 0 || F <= 0)
        return DFL_ERR_INVALID_ARG;
    if (dt != DFL_F32 && dt != DFL_BF16) return DFL_ERR_INVALID_ARG;
    if (!rows_fit((int64_t)N * B)) return DFL_ERR_UNSUPPORTED_SHAPE;
    const void* ptrs[] = {Xb, ffn_gain, W1, W3, W2, ws};
    for (const void* p : ptrs) if (!aligned16(p)) return DFL_ERR_MISALIGNED;
    if (d % 8 != 0 || F % 8 != 0) return DFL_ERR_MISALIGNED;
    if (ws_bytes < ws_block_ffn(N, B, d, F, dt)) return DFL_ERR_WORKSPACE;
    DeviceCtx* ctx = current_ctx();
    if (!ctx) return DFL_ERR_NO_DEVICE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t M = (int64_t)N * B;
    uint8_t* p = static_cast<uint8_t*>(ws);
    dfl_status rc;
    if (dt == DFL_F32) {
        float* Xn = reinterpret_cast<float*>(carve(p, (size_t)M * d * 4));
        float* gate = reinterpret_cast<float*>(carve(p, (size_t)M * F * 4));
        float* up = reinterpret_cast<float*>(carve(p, (size_t)M * F * 4));
        float* h = reinterpret_cast<float*>(carve(p, (size_t)M * F * 4));
        if ((rc = rmsnorm_rows(Xb, d, M, 1, 1, 0, ffn_gain, eps, Xn, false, st)) != DFL_OK) return rc;
        if ((rc = gemm_f32(Xn, static_cast<const float*>(W1), gate, (int)M, F, d, F, 0, st)) != DFL_OK) return rc;
        if ((rc = gemm_f32(Xn, static_cast<const float*>(W3), up, (int)M, F, d, F, 0, st)) != DFL_OK) return rc;
        if ((rc = swiglu_f32(gate, up, h, M * F, st)) != DFL_OK) return rc;
        return gemm_f32(h, static_cast<const float*>(W2), Xb, (int)M, d, F, d, 1, st);
    }
    if (F % 64 != 0 || d % 32 != 0) return DFL_ERR_UNSUPPORTED_SHAPE;
    void* Xn = carve(p, (size_t)M * d * 2);
    void* h = carve(p, (size_t)M * F * 2);
    if ((rc = rmsnorm_rows(Xb, d, M, 1, 1, 0, ffn_gain, eps, Xn, true, st)) != DFL_OK) return rc;
    {   // h = silu(Xn W1^T) * (Xn W3^T): tiles hold gate and up of the same features
        GemmArgs g{};
        g.A = Xn; g.M = (int)M; g.K = d;
        g.B[0] = W1; g.B[1] = W3; g.b_rows[0] = F; g.b_rows[1] = F; g.nb = 2; g.N = 2 * F;
        g.split_b = 1;
        g.bn = 0;
        g.m_inner = 1;
        g.epi = EPI_SWIGLU;
        g.ep.seg[0] = GemmSeg{h, 0, F, 0, M};
        g.ep.nseg = 1;
        g.tag = "gemm_ffn_gate_up";
        if ((rc = gemm_tc(ctx, g, st)) != DFL_OK) return rc;
    }
    GemmArgs g{};   // Xb += h W2^T
    g.A = h; g.M = (int)M; g.K = F;
    g.B[0] = W2; g.b_rows[0] = d; g.b_begin[0] = 0; g.nb = 1; g.N = d;
    g.bn = 0;
    g.m_inner = 1;
    g.epi = EPI_RESID;
    g.ep.resid = Xb; g.ep.ld_resid = d;
    g.tag = "gemm_ffn_down";
    // A long K (F) over few output tiles: split along K when the workspace
    // has room for the partials (after the activations), summed in a fixed order.
    const size_t base = ws_block_ffn(N, B, d, F, dt);
    const size_t room = ws_oproj_split(M, d);
    if (ws_bytes >= base + room) {
        g.split_part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + base);
        g.split_part_bytes = room;
    }
    return gemm_tc(ctx, g, st);
}

// ---------------------------------------------------------------- LM head

extern "C" dfl_status dfl_lm_head_argmax(const float* Xb, int32_t N, int32_t B, int32_t row0, int32_t d,
                                         dfl_dtype dt, const float* final_gain, float eps, const void* W_lm,
                                         int32_t V, int32_t* argmax_out, float* logits_out,
                                         const dfl_sample_params* sp, int32_t* samples_out, void* ws,
                                         size_t ws_bytes, dfl_stream stream) {
    const dfl::ApiRange nvtx_range("dfl_lm_head_argmax");
    if (N <= 0 || B <= 0 || row0 < 0 || row0 >= B || d <= 0 || V <= 0) return DFL_ERR_INVALID_ARG;
    if (dt != DFL_F32 && dt != DFL_BF16) return DFL_ERR_INVALID_ARG;
    if (!rows_fit((int64_t)N * B)) return DFL_ERR_UNSUPPORTED_SHAPE;
    if (!Xb || !final_gain || !W_lm || !argmax_out || !ws) return DFL_ERR_INVALID_ARG;
    if (sp && (sp->K < 1 || sp->K > 64 || !(sp->T > 0.f) || !samples_out)) return DFL_ERR_INVALID_ARG;
    if (sp && dt == DFL_BF16 && !logits_out) return DFL_ERR_INVALID_ARG;
    const void* ptrs[] = {Xb, final_gain, W_lm, ws, logits_out ? logits_out : Xb};
    for (const void* p : ptrs) if (!aligned16(p)) return DFL_ERR_MISALIGNED;
    if (d % 8 != 0) return DFL_ERR_MISALIGNED;
    const bool logits_missing = (dt == DFL_F32) && !logits_out;
    if (ws_bytes < ws_lm_head(N, B, row0, d, V, dt, logits_missing)) return DFL_ERR_WORKSPACE;
    DeviceCtx* ctx = current_ctx();
    if (!ctx) return DFL_ERR_NO_DEVICE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int nr = B - row0;
    const int64_t M = (int64_t)N * nr;
    const int tiles = (V + 255) / 256;
    uint8_t* p = static_cast<uint8_t*>(ws);
    void* Xn = carve(p, (size_t)M * d * esz(dt));
    float* pmax = reinterpret_cast<float*>(carve(p, (size_t)M * tiles * 4));
    int* pidx = reinterpret_cast<int*>(carve(p, (size_t)M * tiles * 4));
    double* psum = reinterpret_cast<double*>(carve(p, (size_t)M * tiles * 8));
    const float inv_T = sp ? 1.0f / sp->T : 1.0f;
    dfl_status rc;
    if ((rc = rmsnorm_rows(Xb, d, M, nr, B, row0, final_gain, eps, Xn, dt == DFL_BF16, st)) != DFL_OK) return rc;
    if (dt == DFL_F32) {
        float* lg = logits_out ? logits_out : reinterpret_cast<float*>(carve(p, (size_t)M * V * 4));
        if ((rc = gemm_f32(static_cast<const float*>(Xn), static_cast<const float*>(W_lm), lg, (int)M, V, d, V, 0,
                           st)) != DFL_OK)
            return rc;
        if ((rc = tile_partials(lg, V, M, V, 256, tiles, inv_T, pmax, pidx, sp ? psum : nullptr, st)) != DFL_OK)
            return rc;
        if ((rc = argmax_combine(pmax, pidx, M, tiles, argmax_out, st)) != DFL_OK) return rc;
        if (sp) return sample_rows(lg, V, pmax, psum, M, nr, tiles, 256, V, sp->K, sp->T, sp->seed, samples_out, st);
        return DFL_OK;
    }
    GemmArgs g{};
    g.A = Xn; g.M = (int)M; g.K = d;
    g.B[0] = W_lm; g.b_rows[0] = V; g.b_begin[0] = 0; g.nb = 1; g.N = V;
    // Partials are 256 columns wide: 256-wide tiles, or (pair tiles, no logits
    // or sampling sums to store) 512-wide tiles writing two partials each, whose
    // single accumulator exposes its drain once per tile: worth it over a K of
    // 4,096 (Qwen shape 0.389 -> 0.357 ms), not over 2,880 (GPT-OSS shape 0.207
    // -> 0.222 ms), where 256-wide tiles hide their drain behind two accumulators.
    g.bn = (M > GEMM_BM && d >= 4096 && !logits_out && !sp) ? 512 : 256;
    g.m_inner = 1;
    g.epi = EPI_ARGMAX;
    g.ep.part_max = pmax; g.ep.part_idx = pidx; g.ep.part_sum = sp ? psum : nullptr;
    g.ep.inv_T = inv_T;
    g.ep.logits = logits_out; g.ep.ld_logits = V;
    g.tag = "gemm_lm_head";
    if ((rc = gemm_tc(ctx, g, st)) != DFL_OK) return rc;
    if ((rc = argmax_combine(pmax, pidx, M, tiles, argmax_out, st)) != DFL_OK) return rc;
    if (sp) return sample_rows(logits_out, V, pmax, psum, M, nr, tiles, 256, V, sp->K, sp->T, sp->seed, samples_out, st);
    return DFL_OK;
}

// --------------------------------------------------------- self-selection

extern "C" dfl_status dfl_self_select(const void* vlog, dfl_dtype dt, const int32_t* drafts, int32_t N, int32_t K,
                                      int32_t G, int32_t V, float* scores, int32_t* selected, int32_t* accept_len,
                                      int32_t* bonus, void* ws, size_t ws_bytes, dfl_stream stream) {
    const dfl::ApiRange nvtx_range("dfl_self_select");
    if (N <= 0 || K < 1 || K > 64 || G < 1 || G > 1024 || V <= 0) return DFL_ERR_INVALID_ARG;
    if (dt != DFL_F32 && dt != DFL_BF16) return DFL_ERR_INVALID_ARG;
    if (!vlog || !drafts || !scores || !selected || !accept_len || !bonus || !ws) return DFL_ERR_INVALID_ARG;
    if (!aligned16(vlog) || !aligned16(ws)) return DFL_ERR_MISALIGNED;
    if (ws_bytes < al256(select_ws_bytes(N, K, G))) return DFL_ERR_WORKSPACE;
    if (!current_ctx()) return DFL_ERR_NO_DEVICE;
    return self_select_run(vlog, dt == DFL_BF16, drafts, N, K, G, V, scores, selected, accept_len, bonus, ws,
                           static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------- whole step

namespace dfl {
namespace {

// Shapes the bf16 tensor-core path of a step takes (TMA strides, tile widths).
dfl_status step_bf16_shape(const dfl_step_args* a) {
    if (a->Hq <= 0 || a->Hkv <= 0 || a->Hq % a->Hkv != 0 || (a->hd != 64 && a->hd != 128))
        return DFL_ERR_UNSUPPORTED_SHAPE;
    if ((a->Hkv * a->hd) % 128 != 0 || (a->Hq * a->hd) % 128 != 0 || a->d % 32 != 0)
        return DFL_ERR_UNSUPPORTED_SHAPE;
    if (a->rope && !aligned16(a->rope)) return DFL_ERR_MISALIGNED;
    return DFL_OK;
}

// Shape rules of the DFlash fusion in a step.
dfl_status rc_fc_shape(const dfl_step_args* a) {
    if ((int64_t)a->L * a->d >= ((int64_t)1 << 31) || a->d > 6144) return DFL_ERR_UNSUPPORTED_SHAPE;
    if (a->dtype == DFL_BF16 && a->d % 64 != 0) return DFL_ERR_UNSUPPORTED_SHAPE;
    return DFL_OK;
}

// Host-side checks of a step's arguments (no launch).
dfl_status step_check(const dfl_step_args* a, const dfl_ctx_cache* cache, const void* ws) {
    if (!a || !ws) return DFL_ERR_INVALID_ARG;
    const int dt = a->dtype;
    if (dt != DFL_F32 && dt != DFL_BF16) return DFL_ERR_INVALID_ARG;
    if (a->N <= 0 || a->C <= 0 || a->B < 2 || a->d <= 0 || a->D < 1 || a->D > 8 || a->L < 1 || a->V < 0)
        return DFL_ERR_INVALID_ARG;
    if (!a->H || !a->blk_gain || !a->layers || !a->Xb0 || !a->Xb) return DFL_ERR_INVALID_ARG;
    if (a->W_fc ? !a->fc_gain : (!a->mix_logits || !a->mix_gain)) return DFL_ERR_INVALID_ARG;
    if (a->V > 0 && (!a->W_lm || !a->final_gain || !a->draft)) return DFL_ERR_INVALID_ARG;
    if (a->target && (!a->accept_len || !a->bonus)) return DFL_ERR_INVALID_ARG;
    if (a->sample && (!a->samples || a->V == 0)) return DFL_ERR_INVALID_ARG;
    if (a->vlog && (!a->sample || !a->scores || !a->selected || !a->accept_len || !a->bonus))
        return DFL_ERR_INVALID_ARG;
    if ((a->tv_alpha || a->tv_tokens || a->accept_rule != 0) && !a->vlog) return DFL_ERR_INVALID_ARG;
    if (a->tv_tokens && !a->tv_alpha) return DFL_ERR_INVALID_ARG;
    if (a->accept_rule < 0 || a->accept_rule > 2) return DFL_ERR_INVALID_ARG;
    if (a->F < 0 || (a->F > 0 && !a->ffn_gain)) return DFL_ERR_INVALID_ARG;
    for (int l = 0; l < a->D; ++l) {
        const dfl_layer_weights& w = a->layers[l];
        if (!w.Wq || !w.Wkc || !w.Wvc || !w.Wkb || !w.Wvb || !w.Wo) return DFL_ERR_INVALID_ARG;
        if (a->F > 0 && (!w.W1 || !w.W3 || !w.W2)) return DFL_ERR_INVALID_ARG;
    }
    // Shape rules of the calls the step makes that hold for every dtype (each
    // with the status that call returns), checked before the first launch.
    if (a->L > 16 || a->Hq <= 0 || a->Hkv <= 0 || a->hd <= 0 || a->Hq % a->Hkv != 0) return DFL_ERR_INVALID_ARG;
    const int64_t h_rows = (int64_t)a->N * (cache ? cache->R : a->C);
    if (!rows_fit(h_rows) || !rows_fit((int64_t)a->N * a->C) || !rows_fit((int64_t)a->N * a->B))
        return DFL_ERR_UNSUPPORTED_SHAPE;
    if (a->L > 1 && a->h_layer_stride < h_rows * a->d) return DFL_ERR_INVALID_ARG;
    if (a->W_fc && (rc_fc_shape(a) != DFL_OK)) return rc_fc_shape(a);
    if (a->d % 8 != 0 || a->hd % 8 != 0 || a->F % 8 != 0 || a->h_layer_stride % 8 != 0)
        return DFL_ERR_MISALIGNED;
    // The 16-byte rule of every kernel the step launches, likewise.
    const void* al[] = {ws, a->Xb, a->mix_gain, a->blk_gain, a->final_gain, a->W_lm, a->rope, a->ffn_gain,
                        a->logits, a->vlog, a->W_fc, a->fc_gain};
    for (const void* q : al)
        if (q && !aligned16(q)) return DFL_ERR_MISALIGNED;
    for (int l = 0; l < a->D; ++l) {
        const dfl_layer_weights& w = a->layers[l];
        const void* wl[] = {w.Wq, w.Wkc, w.Wvc, w.Wkb, w.Wvb, w.Wo, w.W1, w.W3, w.W2};
        for (const void* q : wl)
            if (q && !aligned16(q)) return DFL_ERR_MISALIGNED;
    }
    if (cache) {
        if (dt != DFL_BF16) return DFL_ERR_UNSUPPORTED_SHAPE;
        if (!cache->K || !cache->V || !cache->ctx_len || !cache->n_new || cache->R < 1) return DFL_ERR_INVALID_ARG;
        if (cache->layer_stride < (int64_t)a->N * a->C * a->Hkv * a->hd) return DFL_ERR_INVALID_ARG;
        if ((int64_t)a->N * a->C >= (int64_t)1 << 31) return DFL_ERR_UNSUPPORTED_SHAPE;
        if (!aligned16(cache->K) || !aligned16(cache->V) || (cache->layer_stride * 2) % 16 != 0)
            return DFL_ERR_MISALIGNED;
        return step_bf16_shape(a);
    }
    return DFL_OK;
}

dfl_shape step_shape(const dfl_step_args* a, const dfl_ctx_cache* cache) {
    dfl_shape s{};
    s.N = a->N; s.C = a->C; s.B = a->B; s.d = a->d; s.Hq = a->Hq; s.Hkv = a->Hkv; s.hd = a->hd; s.D = a->D;
    s.L = a->L; s.V = a->V; s.K = a->sample ? a->sample->K : 0; s.G = a->B - 1; s.row0 = 1; s.dtype = a->dtype;
    s.F = a->F; s.R = cache ? cache->R : 0;
    s.fc = a->W_fc ? 1 : 0;
    return s;
}

dfl_status step_tail(const dfl_step_args* a, const dfl_shape& s, uint8_t* Xc, size_t xc_bytes, int32_t* samples,
                     uint8_t* sub, size_t sub_bytes, dfl_stream stream);

// The whole draft step; with `cache`, the incremental form over the caller's
// context K/V cache (args->C its capacity, args->H the R new rows per sequence).
dfl_status draft_step_impl(const dfl_step_args* a, const dfl_ctx_cache* cache, void* ws, size_t ws_bytes,
                           dfl_stream stream) {
    dfl_status rc = step_check(a, cache, ws);
    if (rc != DFL_OK) return rc;
    if (!aligned16(a->H)) return DFL_ERR_MISALIGNED;   // read by the mix's bulk copies
    const int dt = a->dtype;
    const dfl_shape s = step_shape(a, cache);
    if (ws_bytes < step_ws_bytes(s, cache != nullptr)) return DFL_ERR_WORKSPACE;
    if (!aligned16(ws)) return DFL_ERR_MISALIGNED;
    DeviceCtx* dctx = current_ctx();
    if (!dctx) return DFL_ERR_NO_DEVICE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const dfl_dtype ddt = static_cast<dfl_dtype>(dt);
    const size_t e = esz(dt);
    const int N = a->N, C = a->C, B = a->B, d = a->d;
    const int R = cache ? cache->R : C;
    const int64_t ctx_rows = (int64_t)N * R;   // context rows mixed and projected this step
    uint8_t* p = static_cast<uint8_t*>(ws);
    const bool fc = a->W_fc != nullptr;
    size_t xc_bytes = fc ? al256((size_t)ctx_rows * d * e) + ws_fc_fuse(ctx_rows, d) : (size_t)a->D * ctx_rows * d * e;
    if (cache && a->V > 0 && s.K > 0) xc_bytes = std::max(xc_bytes, (size_t)N * (B - 1) * a->V * 4);
    uint8_t* Xc = carve(p, xc_bytes);
    float* F_fc = fc ? reinterpret_cast<float*>(Xc + al256((size_t)ctx_rows * d * e)) : nullptr;
    void* Q = carve(p, (size_t)N * B * a->Hq * a->hd * e);
    void* Kc = cache ? nullptr : carve(p, (size_t)ctx_rows * a->Hkv * a->hd * e);
    void* Vc = cache ? nullptr : carve(p, (size_t)ctx_rows * a->Hkv * a->hd * e);
    void* Kb = carve(p, (size_t)N * B * a->Hkv * a->hd * e);
    void* Vb = carve(p, (size_t)N * B * a->Hkv * a->hd * e);
    KvRowPlan plan{};
    int32_t* len_new = nullptr;
    if (cache) {
        plan.ctx_pos = reinterpret_cast<int32_t*>(carve(p, (size_t)ctx_rows * 4));
        plan.ctx_dst = reinterpret_cast<int32_t*>(carve(p, (size_t)ctx_rows * 4));
        plan.blk_pos = reinterpret_cast<int32_t*>(carve(p, (size_t)N * B * 4));
        plan.dst_rows = (int64_t)N * C;
        len_new = reinterpret_cast<int32_t*>(carve(p, (size_t)N * 4));
    }
    int32_t* samples = a->samples;
    if (a->V > 0 && s.K > 0) {
        int32_t* own = reinterpret_cast<int32_t*>(carve(p, (size_t)N * s.K * (B - 1) * 4));
        if (!samples) samples = own;
    }
    if (a->V > 0) carve(p, (size_t)N * (B - 1) * 4);
    uint8_t* sub = p;
    const size_t sub_bytes = ws_bytes - (size_t)(sub - static_cast<uint8_t*>(ws));

    // bf16: the first layer's block RMSNorm reads Xb0 and copies it into the
    // residual stream Xb; fp32: a device copy first.
    const bool bf = dt == DFL_BF16;
    if (bf && (rc = step_bf16_shape(a)) != DFL_OK) return rc;
    if (!bf) {
        ProfScope ps("copy_block_init", st);
        if (cudaMemcpyAsync(a->Xb, a->Xb0, (size_t)N * B * d * sizeof(float), cudaMemcpyDeviceToDevice, st) !=
            cudaSuccess)
            return DFL_ERR_CUDA;
    }
    if (cache &&
        (rc = cache_plan(N, R, B, C, cache->ctx_len, cache->n_new, cache->advance, const_cast<int32_t*>(plan.ctx_pos),
                         const_cast<int32_t*>(plan.ctx_dst), const_cast<int32_t*>(plan.blk_pos), len_new,
                         dev_err(dctx), st)) != DFL_OK)
        return rc;
    if (fc) {
        if ((rc = fc_fuse_check(a->H, a->h_layer_stride, a->L, ctx_rows, d, dt, a->W_fc, a->fc_gain, Xc)) != DFL_OK)
            return rc;
        if ((rc = fc_fuse_impl(dctx, a->H, a->h_layer_stride, a->L, ctx_rows, d, dt, a->W_fc, a->fc_gain, a->eps, Xc,
                               F_fc, st)) != DFL_OK)
            return rc;
    } else if ((rc = dfl_layer_mix_rmsnorm(a->H, a->h_layer_stride, a->L, ctx_rows, d, ddt, a->D, a->mix_logits,
                                           a->mix_gain, a->eps, Xc, ctx_rows * d, stream)) != DFL_OK) {
        return rc;
    }
    for (int l = 0; l < a->D; ++l) {
        const dfl_layer_weights& w = a->layers[l];
        const void* xc_l = Xc + (fc ? 0 : (size_t)l * ctx_rows * d * e);   // the fusion serves every layer
        if (cache) {
            void* Kl = static_cast<uint8_t*>(cache->K) + (size_t)l * cache->layer_stride * 2;
            void* Vl = static_cast<uint8_t*>(cache->V) + (size_t)l * cache->layer_stride * 2;
            if ((rc = dual_kv_proj_bf16(dctx, xc_l, ctx_rows, R, a->Xb, N, B, d, a->blk_gain + (size_t)l * d, a->eps,
                                        w.Wq, w.Wkc, w.Wvc, w.Wkb, w.Wvb, a->Hq, a->Hkv, a->hd, a->rope, Q, Kl, Vl,
                                        Kb, Vb, sub, &plan, st, l == 0 ? a->Xb0 : nullptr)) != DFL_OK)
                return rc;
            if ((rc = block_attn_bf16(dctx, Q, Kl, Vl, Kb, Vb, N, C, B, a->Hq, a->Hkv, a->hd, w.Wo, d, a->Xb, sub,
                                      sub_bytes, len_new, C, st)) != DFL_OK)
                return rc;
        } else {
            if (bf) {
                if ((rc = dual_kv_proj_bf16(dctx, xc_l, (int64_t)N * C, C, a->Xb, N, B, d, a->blk_gain + (size_t)l * d,
                                            a->eps, w.Wq, w.Wkc, w.Wvc, w.Wkb, w.Wvb, a->Hq, a->Hkv, a->hd, a->rope, Q,
                                            Kc, Vc, Kb, Vb, sub, nullptr, st, l == 0 ? a->Xb0 : nullptr)) != DFL_OK)
                    return rc;
            } else if ((rc = dfl_dual_kv_proj(xc_l, a->Xb, N, C, B, d, ddt, a->blk_gain + (size_t)l * d, a->eps, w.Wq,
                                              w.Wkc, w.Wvc, w.Wkb, w.Wvb, a->Hq, a->Hkv, a->hd, a->rope, Q, Kc, Vc, Kb,
                                              Vb, sub, sub_bytes, stream)) != DFL_OK) {
                return rc;
            }
            if ((rc = dfl_block_attn(Q, Kc, Vc, Kb, Vb, N, C, B, a->Hq, a->Hkv, a->hd, ddt, w.Wo, d, a->Xb, sub,
                                     sub_bytes, stream)) != DFL_OK)
                return rc;
        }
        if (a->F > 0 && (rc = dfl_block_ffn(a->Xb, N, B, d, ddt, a->ffn_gain + (size_t)l * d, a->eps, w.W1, w.W3,
                                            w.W2, a->F, sub, sub_bytes, stream)) != DFL_OK)
            return rc;
    }
    return step_tail(a, s, Xc, xc_bytes, samples, sub, sub_bytes, stream);
}

// LM head and acceptance epilogue of a step (a7 onwards), on the final Xb.
dfl_status step_tail(const dfl_step_args* a, const dfl_shape& s, uint8_t* Xc, size_t xc_bytes, int32_t* samples,
                     uint8_t* sub, size_t sub_bytes, dfl_stream stream) {
    const int dt = a->dtype;
    const dfl_dtype ddt = static_cast<dfl_dtype>(dt);
    const int N = a->N, B = a->B, d = a->d;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    dfl_status rc;
    if (a->V == 0) return DFL_OK;
    float* logits = a->logits;
    if (!logits && a->sample) {   // sampling walks the logits; borrow the Xc area (no longer needed)
        if ((size_t)N * (B - 1) * a->V * 4 > xc_bytes) return DFL_ERR_WORKSPACE;
        logits = reinterpret_cast<float*>(Xc);
    }
    if ((rc = dfl_lm_head_argmax(a->Xb, N, B, 1, d, ddt, a->final_gain, a->eps, a->W_lm, a->V, a->draft, logits,
                                 a->sample, samples, sub, sub_bytes, stream)) != DFL_OK)
        return rc;
    if (a->vlog) {
        const int K = a->sample->K, G = B - 1;
        if ((rc = dfl_self_select(a->vlog, ddt, samples, N, K, G, a->V, a->scores, a->selected, a->accept_len,
                                  a->bonus, sub, sub_bytes, stream)) != DFL_OK)
            return rc;
        if (!a->tv_alpha && a->accept_rule == 0) return DFL_OK;
        // Reuse self-selection's LSEs of every verifier row (at the start of its
        // scratch); the drafter rows' LSEs are formed once for both epilogues.
        const float* lse_v = reinterpret_cast<const float*>(sub);
        uint8_t* q = sub + al256(select_ws_bytes(N, K, G));
        float* lse_z = reinterpret_cast<float*>(q);
        q += al256((size_t)N * G * 4);
        const float inv_T = 1.0f / a->sample->T;
        if (a->tv_alpha || a->accept_rule == 1)
            if ((rc = lse_rows_f32(logits, N * G, a->V, inv_T, lse_z, st)) != DFL_OK) return rc;
        if (a->tv_alpha && (rc = tv_run(logits, inv_T, a->vlog, dt == DFL_BF16, N, K, G, a->V, a->tv_alpha,
                                        a->tv_tokens, lse_z, lse_v, st)) != DFL_OK)
            return rc;
        if (a->accept_rule == 1)
            return spec_run(logits, inv_T, a->vlog, dt == DFL_BF16, samples, a->selected, N, K, G, a->V,
                            a->accept_seed, a->accept_len, a->bonus, lse_z, lse_v, true, q, st);
        if (a->accept_rule == 2)
            return sg_run(a->vlog, dt == DFL_BF16, samples, a->selected, N, K, G, a->V, a->accept_seed,
                          a->accept_len, a->bonus, lse_v, true, q, st);
        return DFL_OK;
    }
    if (a->target) return dfl_greedy_accept(a->draft, a->target, N, B - 1, a->accept_len, a->bonus, stream);
    return DFL_OK;
}

// dfl_draft_step_host: the copy of H in groups of whole sequences on the
// device's copy stream, each group's mix and context projections (all
// layers) as soon as it has landed, then the block path and the tail.
dfl_status draft_step_host_impl(const dfl_step_args* a, void* H_dev, int chunks, void* ws, size_t ws_bytes,
                                dfl_stream stream) {
    dfl_status rc = step_check(a, nullptr, ws);
    if (rc != DFL_OK) return rc;
    if (!H_dev || chunks < 1) return DFL_ERR_INVALID_ARG;
    if (a->dtype != DFL_BF16) return DFL_ERR_UNSUPPORTED_SHAPE;
    if ((rc = step_bf16_shape(a)) != DFL_OK) return rc;
    if (!aligned16(H_dev) || (a->h_layer_stride * 2) % 16 != 0 || a->d % 8 != 0) return DFL_ERR_MISALIGNED;
    if (a->h_layer_stride < (int64_t)a->N * a->C * a->d) return DFL_ERR_INVALID_ARG;
    const dfl_shape s = step_shape(a, nullptr);
    const size_t plain_bytes = step_ws_bytes(s, false);
    if (ws_bytes < step_host_ws_bytes(s)) return DFL_ERR_WORKSPACE;
    DeviceCtx* dctx = current_ctx();
    if (!dctx) return DFL_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> lk(dctx->host_mu);
    if (!dctx->copy_st) {   // all or nothing: a failed creation leaves nothing half made
        cudaStream_t cs = nullptr;
        cudaEvent_t ev[DeviceCtx::MAX_H_CHUNKS + 1] = {};
        bool ok = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) == cudaSuccess;
        for (cudaEvent_t& e : ev) ok = ok && cudaEventCreateWithFlags(&e, cudaEventDisableTiming) == cudaSuccess;
        if (!ok) {
            for (cudaEvent_t e : ev)
                if (e) cudaEventDestroy(e);
            if (cs) cudaStreamDestroy(cs);
            return DFL_ERR_CUDA;
        }
        for (int i = 0; i <= DeviceCtx::MAX_H_CHUNKS; ++i) dctx->copy_ev[i] = ev[i];
        dctx->copy_st = cs;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int N = a->N, C = a->C, B = a->B, d = a->d, L = a->L, D = a->D;
    const int kv = a->Hkv * a->hd;
    const int64_t ctx_rows = (int64_t)N * C;
    // the plain step's carve, then layers 1..D-1's context K/V past its end
    uint8_t* p = static_cast<uint8_t*>(ws);
    const bool fc = a->W_fc != nullptr;
    const size_t xc_bytes = fc ? al256((size_t)ctx_rows * d * 2) + ws_fc_fuse(ctx_rows, d) : (size_t)D * ctx_rows * d * 2;
    uint8_t* Xc = carve(p, xc_bytes);
    float* F_fc = fc ? reinterpret_cast<float*>(Xc + al256((size_t)ctx_rows * d * 2)) : nullptr;
    if (fc && (rc = fc_fuse_check(H_dev, a->h_layer_stride, L, ctx_rows, d, DFL_BF16, a->W_fc, a->fc_gain, Xc)) !=
                  DFL_OK)
        return rc;
    void* Q = carve(p, (size_t)N * B * a->Hq * a->hd * 2);
    uint8_t* Kc0 = carve(p, (size_t)ctx_rows * kv * 2);
    uint8_t* Vc0 = carve(p, (size_t)ctx_rows * kv * 2);
    void* Kb = carve(p, (size_t)N * B * kv * 2);
    void* Vb = carve(p, (size_t)N * B * kv * 2);
    int32_t* samples = a->samples;
    if (a->V > 0 && s.K > 0) {
        int32_t* own = reinterpret_cast<int32_t*>(carve(p, (size_t)N * s.K * (B - 1) * 4));
        if (!samples) samples = own;
    }
    if (a->V > 0) carve(p, (size_t)N * (B - 1) * 4);
    uint8_t* sub = p;
    const size_t sub_bytes = plain_bytes - (size_t)(sub - static_cast<uint8_t*>(ws));
    uint8_t* extra = static_cast<uint8_t*>(ws) + plain_bytes;
    auto kc_of = [&](int l) { return l == 0 ? Kc0 : extra + (size_t)(l - 1) * 2 * kv_layer_bytes(s); };
    auto vc_of = [&](int l) { return l == 0 ? Vc0 : kc_of(l) + kv_layer_bytes(s); };

    {
    ProfScope ps("copy_block_init", st);
    if (cudaMemcpyAsync(a->Xb, a->Xb0, (size_t)N * B * d * sizeof(float), cudaMemcpyDeviceToDevice, st) !=
        cudaSuccess)
        return DFL_ERR_CUDA;
    }
    // H_dev may still be read by work queued earlier on `stream`
    cudaEvent_t* ev = dctx->copy_ev;
    if (cudaEventRecord(ev[DeviceCtx::MAX_H_CHUNKS], st) != cudaSuccess ||
        cudaStreamWaitEvent(dctx->copy_st, ev[DeviceCtx::MAX_H_CHUNKS], 0) != cudaSuccess)
        return DFL_ERR_CUDA;
    // Sequences are independent: with greedy drafts (no sampling epilogue) each
    // group also runs its block path, LM head and acceptance as soon as its
    // context is projected (the attention splits keys as for the whole batch,
    // so every group's arithmetic is the whole-batch step's).
    const bool group_tail = !a->sample && !a->vlog && (!a->logits || ((size_t)(a->B - 1) * a->V) % 4 == 0);
    const int nch = std::min(std::min(chunks, N), DeviceCtx::MAX_H_CHUNKS);
    const int per = (N + nch - 1) / nch;
    const uint8_t* Hh = static_cast<const uint8_t*>(a->H);
    uint8_t* Hd = static_cast<uint8_t*>(H_dev);
    const size_t lstride = (size_t)a->h_layer_stride * 2;
    for (int c = 0; c * per < N; ++c) {
        const int n0 = c * per, n1 = std::min(N, n0 + per);
        const int64_t r0 = (int64_t)n0 * C, rows = (int64_t)(n1 - n0) * C;
        const size_t off = (size_t)r0 * d * 2, bytes = (size_t)rows * d * 2;
        for (int i = 0; i < L; ++i)
            if (cudaMemcpyAsync(Hd + i * lstride + off, Hh + i * lstride + off, bytes, cudaMemcpyHostToDevice,
                                dctx->copy_st) != cudaSuccess)
                return DFL_ERR_CUDA;
        if (cudaEventRecord(ev[c], dctx->copy_st) != cudaSuccess || cudaStreamWaitEvent(st, ev[c], 0) != cudaSuccess)
            return DFL_ERR_CUDA;
        if (fc) {   // the group's rows of the one fused representation
            if ((rc = fc_fuse_impl(dctx, Hd + off, a->h_layer_stride, L, rows, d, DFL_BF16, a->W_fc, a->fc_gain,
                                   a->eps, Xc + off, F_fc + (size_t)r0 * d, st)) != DFL_OK)
                return rc;
        } else if ((rc = dfl_layer_mix_rmsnorm(Hd + off, a->h_layer_stride, L, rows, d, DFL_BF16, D, a->mix_logits,
                                               a->mix_gain, a->eps, Xc + off, ctx_rows * d, stream)) != DFL_OK) {
            return rc;
        }
        for (int l = 0; l < D; ++l) {   // context rows start at a sequence: position = row % C
            const dfl_layer_weights& w = a->layers[l];
            const GemmArgs gc = ctx_kv_args(Xc + (fc ? 0 : (size_t)l * ctx_rows * d * 2) + off, rows, C, d, w.Wkc, w.Wvc,
                                            a->Hkv, a->hd, a->rope, kc_of(l) + (size_t)r0 * kv * 2,
                                            vc_of(l) + (size_t)r0 * kv * 2, nullptr);
            if ((rc = gemm_tc(dctx, gc, st)) != DFL_OK) return rc;
        }
        if (!group_tail) continue;
        const int Nc = n1 - n0;
        float* Xb_c = a->Xb + (size_t)n0 * B * d;
        for (int l = 0; l < D; ++l) {
            const dfl_layer_weights& w = a->layers[l];
            if ((rc = dual_kv_proj_bf16(dctx, nullptr, 0, C, Xb_c, Nc, B, d, a->blk_gain + (size_t)l * d, a->eps,
                                        w.Wq, w.Wkc, w.Wvc, w.Wkb, w.Wvb, a->Hq, a->Hkv, a->hd, a->rope, Q, nullptr,
                                        nullptr, Kb, Vb, sub, nullptr, st)) != DFL_OK)
                return rc;
            if ((rc = block_attn_bf16(dctx, Q, kc_of(l) + (size_t)r0 * kv * 2, vc_of(l) + (size_t)r0 * kv * 2, Kb, Vb,
                                      Nc, C, B, a->Hq, a->Hkv, a->hd, w.Wo, d, Xb_c, sub, sub_bytes, nullptr, C, st,
                                      N)) != DFL_OK)
                return rc;
            if (a->F > 0 && (rc = dfl_block_ffn(Xb_c, Nc, B, d, DFL_BF16, a->ffn_gain + (size_t)l * d, a->eps, w.W1,
                                                w.W3, w.W2, a->F, sub, sub_bytes, stream)) != DFL_OK)
                return rc;
        }
        if (a->V == 0) continue;
        const size_t G = (size_t)(B - 1);
        if ((rc = dfl_lm_head_argmax(Xb_c, Nc, B, 1, d, DFL_BF16, a->final_gain, a->eps, a->W_lm, a->V,
                                     a->draft + (size_t)n0 * G, a->logits ? a->logits + (size_t)n0 * G * a->V : nullptr,
                                     nullptr, nullptr, sub, sub_bytes, stream)) != DFL_OK)
            return rc;
        if (a->target && (rc = dfl_greedy_accept(a->draft + (size_t)n0 * G, a->target + (size_t)n0 * B, Nc, B - 1,
                                                 a->accept_len + n0, a->bonus + n0, stream)) != DFL_OK)
            return rc;
    }
    if (group_tail) return DFL_OK;
    for (int l = 0; l < D; ++l) {
        const dfl_layer_weights& w = a->layers[l];
        if ((rc = dual_kv_proj_bf16(dctx, nullptr, 0, C, a->Xb, N, B, d, a->blk_gain + (size_t)l * d, a->eps, w.Wq,
                                    w.Wkc, w.Wvc, w.Wkb, w.Wvb, a->Hq, a->Hkv, a->hd, a->rope, Q, nullptr, nullptr, Kb,
                                    Vb, sub, nullptr, st)) != DFL_OK)
            return rc;
        if ((rc = block_attn_bf16(dctx, Q, kc_of(l), vc_of(l), Kb, Vb, N, C, B, a->Hq, a->Hkv, a->hd, w.Wo, d, a->Xb,
                                  sub, sub_bytes, nullptr, C, st)) != DFL_OK)
            return rc;
        if (a->F > 0 && (rc = dfl_block_ffn(a->Xb, N, B, d, DFL_BF16, a->ffn_gain + (size_t)l * d, a->eps, w.W1,
                                            w.W3, w.W2, a->F, sub, sub_bytes, stream)) != DFL_OK)
            return rc;
    }
    return step_tail(a, s, Xc, xc_bytes, samples, sub, sub_bytes, stream);
}

}  // namespace
}  // namespace dfl

extern "C" dfl_status dfl_draft_step(const dfl_step_args* a, void* ws, size_t ws_bytes, dfl_stream stream) {
    const dfl::ApiRange nvtx_range("dfl_draft_step");
    return draft_step_impl(a, nullptr, ws, ws_bytes, stream);
}

extern "C" dfl_status dfl_draft_step_host(const dfl_step_args* a, void* H_dev, int32_t chunks, void* ws,
                                          size_t ws_bytes, dfl_stream stream) {
    const dfl::ApiRange nvtx_range("dfl_draft_step_host");
    return draft_step_host_impl(a, H_dev, chunks, ws, ws_bytes, stream);
}

extern "C" dfl_status dfl_draft_step_cached(const dfl_step_args* a, const dfl_ctx_cache* cache, void* ws,
                                            size_t ws_bytes, dfl_stream stream) {
    const dfl::ApiRange nvtx_range("dfl_draft_step_cached");
    if (!cache) return DFL_ERR_INVALID_ARG;
    return draft_step_impl(a, cache, ws, ws_bytes, stream);
}

// ---------------------------------------------------------------- tracing

namespace dfl {
namespace {
struct ProfRec {
    const char* name;
    cudaEvent_t beg, end;
};
std::mutex g_prof_mu;
std::atomic<bool> g_prof_on{false};
std::vector<ProfRec> g_prof_recs;     // recorded pairs (events owned by the pool)
std::vector<std::pair<cudaEvent_t, cudaEvent_t>> g_prof_pool;
size_t g_prof_used = 0;
}  // namespace

ProfScope::ProfScope(const char* name, cudaStream_t st) : st_(st) {
    if (!g_prof_on.load(std::memory_order_relaxed)) return;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (g_prof_used == g_prof_pool.size()) {
        cudaEvent_t a, b;
        if (cudaEventCreate(&a) != cudaSuccess) return;
        if (cudaEventCreate(&b) != cudaSuccess) { cudaEventDestroy(a); return; }
        g_prof_pool.emplace_back(a, b);
    }
    const auto& ev = g_prof_pool[g_prof_used];
    if (cudaEventRecord(ev.first, st) != cudaSuccess) return;
    slot_ = (int)g_prof_recs.size();
    g_prof_recs.push_back(ProfRec{name, ev.first, ev.second});
    ++g_prof_used;
}

ProfScope::~ProfScope() {
    if (slot_ < 0) return;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    cudaEventRecord(g_prof_recs[slot_].end, st_);
}

}  // namespace dfl

extern "C" dfl_status dfl_profile_enable(int32_t on) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (on) {
        g_prof_recs.clear();
        g_prof_used = 0;
    }
    g_prof_on.store(on != 0);
    return DFL_OK;
}

extern "C" dfl_status dfl_profile_report(char* buf, size_t buf_len, int32_t* launches) {
    if (!buf || buf_len == 0) return DFL_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    std::vector<std::string> names;
    std::vector<std::pair<int, double>> agg;
    for (const ProfRec& r : g_prof_recs) {
        if (cudaEventSynchronize(r.end) != cudaSuccess) return DFL_ERR_CUDA;
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, r.beg, r.end) != cudaSuccess) return DFL_ERR_CUDA;
        size_t i = 0;
        while (i < names.size() && names[i] != r.name) ++i;
        if (i == names.size()) { names.emplace_back(r.name); agg.emplace_back(0, 0.0); }
        agg[i].first += 1;
        agg[i].second += ms;
    }
    std::string out = "{";
    for (size_t i = 0; i < names.size(); ++i) {
        char tmp[256];
        snprintf(tmp, sizeof(tmp), "%s\"%s\": [%d, %.6f]", i ? ", " : "", names[i].c_str(), agg[i].first,
                 agg[i].second);
        out += tmp;
    }
    out += "}";
    const size_t n = out.size() < buf_len - 1 ? out.size() : buf_len - 1;
    memcpy(buf, out.data(), n);
    buf[n] = '\0';
    if (launches) *launches = (int32_t)g_prof_recs.size();
    g_prof_recs.clear();
    g_prof_used = 0;
    return DFL_OK;
}
