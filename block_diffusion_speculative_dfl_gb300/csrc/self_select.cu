// Streak-score self-selection of K drafts and greedy acceptance.
//
// SpecDiff-2 notes, "Streak-Distillation": expected accepted tokens per draft
// = sum_{m=1}^{gamma} prod_{j<=m} alpha_j.  "Self-Selection Acceptance": K
// drafts sampled from one denoising step are scored with the verifier's
// per-token posteriors, the best draft is kept, and greedy acceptance runs
// on it reusing the cached verifier probabilities (draft probabilities are
// not used).
//
// Pass 1 (HBM-bound, one read of the verifier logits): per verifier row its
// log-sum-exp, argmax (lowest index on ties) and the logit at the draft
// token.  Pass 2 (one warp per sequence): log p_j = z[x_j] - LSE_j,
// S_k = sum_m exp(sum_{j<=m} log p_j) in fp64, k* = argmax_k S_k (lowest k on
// ties), then the prefix of x^{k*} matching the argmax of its verifier rows
// and the bonus token.
#include <mutex>

#include "internal.h"
#include "small_kernels.h"

namespace dfl {

namespace {

constexpr int RS_THREADS = 256;
constexpr float kLog2e = 1.4426950408889634f;

struct RowStat {
    float m;    // running max
    float s;    // sum exp(x - m)
    int idx;    // lowest index of the max
};

__device__ __forceinline__ RowStat rs_combine(RowStat a, RowStat b) {
    RowStat r;
    r.m = fmaxf(a.m, b.m);
    r.idx = (b.m > a.m || (b.m == a.m && b.idx < a.idx)) ? b.idx : a.idx;
    const float sa = a.m == -INFINITY ? 0.f : a.s * expf(a.m - r.m);
    const float sb = b.m == -INFINITY ? 0.f : b.s * expf(b.m - r.m);
    r.s = sa + sb;
    return r;
}

__device__ __forceinline__ void rs_push8(RowStat& st, const float (&x)[8], int base) {
    float vm = x[0];
    #pragma unroll
    for (int j = 1; j < 8; ++j) vm = fmaxf(vm, x[j]);
    if (vm > st.m) {
        st.s = st.m == -INFINITY ? 0.f : st.s * expf(st.m - vm);
        st.m = vm;
        int f = 7;
        #pragma unroll
        for (int j = 7; j >= 0; --j) if (x[j] == vm) f = j;
        st.idx = base + f;
    }
    float acc = 0.f;
    #pragma unroll
    for (int j = 0; j < 8; ++j) acc += expf(x[j] - st.m);
    st.s += acc;
}

template <bool BF16>
__device__ __forceinline__ float load1(const void* row, int64_t i) {
    if constexpr (BF16) {
        const uint16_t u = static_cast<const uint16_t*>(row)[i];
        return __uint_as_float((uint32_t)u << 16);
    } else {
        return static_cast<const float*>(row)[i];
    }
}

template <bool BF16>
__global__ void __launch_bounds__(RS_THREADS) verifier_row_stats_kernel(const void* vlog, int K, int G, int V,
                                                                        const int32_t* drafts, float* lse, int* amax,
                                                                        float* zx) {
    grid_dep_begin();
    const int64_t rr = blockIdx.x;
    const int G1 = G + 1;
    const size_t esz = BF16 ? 2 : 4;
    const uint8_t* row = static_cast<const uint8_t*>(vlog) + rr * (int64_t)V * esz;
    RowStat st{-INFINITY, 0.f, 0x7FFFFFFF};
    const bool vec = (V % 8) == 0;
    if (vec) {
        const int chunks = V / 8;
        int c = threadIdx.x;
        if constexpr (BF16) {
            // Four 16-byte loads in flight per thread: chunks c, c + T, c + 2T, c + 3T
            // (increasing indices, so the first maximum found is the lowest).
            for (; c + 3 * RS_THREADS < chunks; c += 4 * RS_THREADS) {
                uint4 u[4];
                #pragma unroll
                for (int q = 0; q < 4; ++q) u[q] = __ldg(reinterpret_cast<const uint4*>(row) + c + q * RS_THREADS);
                float x[4][8];
                #pragma unroll
                for (int q = 0; q < 4; ++q) {
                    x[q][0] = bf16lo(u[q].x); x[q][1] = bf16hi(u[q].x); x[q][2] = bf16lo(u[q].y); x[q][3] = bf16hi(u[q].y);
                    x[q][4] = bf16lo(u[q].z); x[q][5] = bf16hi(u[q].z); x[q][6] = bf16lo(u[q].w); x[q][7] = bf16hi(u[q].w);
                }
                float vm = x[0][0];
                #pragma unroll
                for (int q = 0; q < 4; ++q)
                    #pragma unroll
                    for (int j = 0; j < 8; ++j) vm = fmaxf(vm, x[q][j]);
                if (vm > st.m) {
                    st.s = st.m == -INFINITY ? 0.f : st.s * ex2_ftz((st.m - vm) * kLog2e);
                    st.m = vm;
                    int f = -1;
                    #pragma unroll
                    for (int q = 3; q >= 0; --q)
                        #pragma unroll
                        for (int j = 7; j >= 0; --j)
                            if (x[q][j] == vm) f = (c + q * RS_THREADS) * 8 + j;
                    st.idx = f;
                }
                // exp(x - m) = 2^(x log2(e) - m log2(e)): one FMA and one SFU op per element
                const float nml = -st.m * kLog2e;
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
                #pragma unroll
                for (int q = 0; q < 4; ++q)
                    #pragma unroll
                    for (int j = 0; j < 8; ++j) acc[q] += ex2_ftz(fmaf(x[q][j], kLog2e, nml));
                st.s += (acc[0] + acc[1]) + (acc[2] + acc[3]);
            }
        }
        for (; c < chunks; c += RS_THREADS) {
            float x[8];
            if constexpr (BF16) {
                const uint4 u = reinterpret_cast<const uint4*>(row)[c];
                x[0] = bf16lo(u.x); x[1] = bf16hi(u.x); x[2] = bf16lo(u.y); x[3] = bf16hi(u.y);
                x[4] = bf16lo(u.z); x[5] = bf16hi(u.z); x[6] = bf16lo(u.w); x[7] = bf16hi(u.w);
            } else {
                const float4 u0 = reinterpret_cast<const float4*>(row)[2 * c];
                const float4 u1 = reinterpret_cast<const float4*>(row)[2 * c + 1];
                x[0] = u0.x; x[1] = u0.y; x[2] = u0.z; x[3] = u0.w;
                x[4] = u1.x; x[5] = u1.y; x[6] = u1.z; x[7] = u1.w;
            }
            rs_push8(st, x, c * 8);
        }
    } else {
        for (int i = threadIdx.x; i < V; i += RS_THREADS) {
            const float x = load1<BF16>(row, i);
            if (x > st.m) {
                st.s = st.m == -INFINITY ? 0.f : st.s * expf(st.m - x);
                st.m = x;
                st.idx = i;
            }
            st.s += expf(x - st.m);
        }
    }
    #pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        RowStat b;
        b.m = __shfl_xor_sync(0xFFFFFFFFu, st.m, o);
        b.s = __shfl_xor_sync(0xFFFFFFFFu, st.s, o);
        b.idx = __shfl_xor_sync(0xFFFFFFFFu, st.idx, o);
        st = rs_combine(st, b);
    }
    __shared__ RowStat red[RS_THREADS / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = st;
    __syncthreads();
    if (threadIdx.x == 0) {
        RowStat t = red[0];
        for (int w = 1; w < RS_THREADS / 32; ++w) t = rs_combine(t, red[w]);
        lse[rr] = t.m + logf(t.s);
        amax[rr] = t.idx;
        const int j = (int)(rr % G1);
        if (j < G) {
            const int64_t nk = rr / G1;   // n * K + k
            const int32_t x = drafts[nk * G + j];
            zx[rr] = (x >= 0 && x < V) ? load1<BF16>(row, x) : -INFINITY;
        }
    }
}

__global__ void streak_select_kernel(const int32_t* drafts, int N, int K, int G, const float* lse, const int* amax,
                                     const float* zx, float* scores, int32_t* selected, int32_t* accept_len,
                                     int32_t* bonus) {
    grid_dep_begin();
    const int n = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (n >= N) return;
    const int G1 = G + 1;
    double best = -1.0;
    int bk = 0x7FFFFFFF;
    for (int k = lane; k < K; k += 32) {
        const int64_t r0 = ((int64_t)n * K + k) * G1;
        double c = 0.0, S = 0.0;
        for (int j = 0; j < G; ++j) {
            c += (double)zx[r0 + j] - (double)lse[r0 + j];
            S += exp(c);
        }
        scores[(int64_t)n * K + k] = (float)S;
        if (S > best) { best = S; bk = k; }
    }
    #pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const double v = __shfl_xor_sync(0xFFFFFFFFu, best, o);
        const int i = __shfl_xor_sync(0xFFFFFFFFu, bk, o);
        if (v > best || (v == best && i < bk)) { best = v; bk = i; }
    }
    if (bk >= K) bk = 0;   // no score compared greater (all NaN): draft 0, never an index past the drafts
    const int64_t r0 = ((int64_t)n * K + bk) * G1;
    const int32_t* x = drafts + ((int64_t)n * K + bk) * G;
    int a = G;
    for (int j0 = 0; j0 < G; j0 += 32) {
        const int j = j0 + lane;
        const unsigned mism = __ballot_sync(0xFFFFFFFFu, j < G && x[j] != amax[r0 + j]);
        if (mism) { a = j0 + __ffs(mism) - 1; break; }
    }
    if (lane == 0) {
        selected[n] = bk;
        accept_len[n] = a;
        bonus[n] = amax[r0 + a];
    }
}

}  // namespace

size_t select_ws_bytes(int N, int K, int G) {
    const size_t rows = (size_t)N * K * (G + 1);
    return 3 * ((rows * 4 + 255) & ~size_t(255));
}

dfl_status self_select_run(const void* vlog, bool bf16, const int32_t* drafts, int N, int K, int G, int V,
                           float* scores, int32_t* selected, int32_t* accept_len, int32_t* bonus, void* ws,
                           cudaStream_t st) {
    const size_t rows = (size_t)N * K * (G + 1);
    const size_t slot = (rows * 4 + 255) & ~size_t(255);
    float* lse = static_cast<float*>(ws);
    int* amax = reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + slot);
    float* zx = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + 2 * slot);
    dfl_status rc;
    {
    ProfScope ps("verifier_row_stats", st);
    if (bf16)
        launch_pdl(verifier_row_stats_kernel<true>, (unsigned)rows, RS_THREADS, 0, st, vlog, K, G, V, drafts, lse,
                   amax, zx);
    else
        launch_pdl(verifier_row_stats_kernel<false>, (unsigned)rows, RS_THREADS, 0, st, vlog, K, G, V, drafts, lse,
                   amax, zx);
    rc = last_launch();
    }
    if (rc != DFL_OK) return rc;
    ProfScope ps("streak_select", st);
    launch_pdl(streak_select_kernel, (N + 3) / 4, 128, 0, st, drafts, N, K, G, lse, amax, zx, scores, selected,
               accept_len, bonus);
    return last_launch();
}

}  // namespace dfl

// --------------------------------------------------- no-allocation variant
//
// Some callers cannot hand the library a workspace: a plugin inside a serving
// engine that owns all device memory through its own pool and gives plugins
// no way to borrow from it, or a latency-critical host loop that must never
// call cudaMalloc (which can synchronise the device or fail under memory
// pressure in the middle of serving).  For them, dfl_self_select_noalloc runs
// the same two kernels as dfl_self_select with their scratch in a fixed array
// that lives in the library's own device image.
//
// Limits and sharing: the array is 768 KiB, enough for N*K*(G+1) <= 65536
// verifier rows; every GPU that loads the library holds it until the process
// exits.  All calls on a device share it and it keeps the previous call's
// contents; nothing needs clearing because each call writes every entry it
// later reads.  Calls whose kernels overlap on the GPU (different streams, or
// several host threads) race on the array and must be serialised by the
// caller.

namespace dfl {
namespace {

constexpr size_t kNoAllocRows = 65536;
constexpr size_t kNoAllocSlot = kNoAllocRows * 4;   // one fp32/int32 per row, per array

static __device__ __align__(256) uint8_t g_select_scratch[3 * kNoAllocSlot];

std::mutex g_noalloc_mu;
struct NoAllocAddr {
    uint64_t ctx_id;   // the CUDA context the address belongs to
    void* ptr;
};
NoAllocAddr g_noalloc[64] = {};

// Device address of the array on the current device.  Host code cannot use
// the symbol itself (it names a host-side stand-in), so the address is looked
// up with that device current, once per device and CUDA context, then
// cached.  A new context on the device (after cudaDeviceReset, for one) loads
// the library's device image again, possibly elsewhere, so the cached address
// is only used while the context it was looked up in is current.
dfl_status noalloc_scratch(const DeviceCtx* ctx, void** out) {
    const int dev = ctx->device;
    if (dev < 0 || dev >= 64) return DFL_ERR_NO_DEVICE;
    const uint64_t cid = ctx->ctx_id.load();
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc[dev].ptr || g_noalloc[dev].ctx_id != cid) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_select_scratch) != cudaSuccess || !p) return DFL_ERR_CUDA;
        g_noalloc[dev] = NoAllocAddr{cid, p};
    }
    *out = g_noalloc[dev].ptr;
    return DFL_OK;
}

}  // namespace

}  // namespace dfl

extern "C" dfl_status dfl_self_select_noalloc(const void* vlog, dfl_dtype dt, const int32_t* drafts, int32_t N,
                                              int32_t K, int32_t G, int32_t V, float* scores, int32_t* selected,
                                              int32_t* accept_len, int32_t* bonus, dfl_stream stream) {
    const dfl::ApiRange nvtx_range("dfl_self_select_noalloc");
    using namespace dfl;
    if (N <= 0 || K < 1 || K > 64 || G < 1 || G > 1024 || V <= 0) return DFL_ERR_INVALID_ARG;
    if (dt != DFL_F32 && dt != DFL_BF16) return DFL_ERR_INVALID_ARG;
    if (!vlog || !drafts || !scores || !selected || !accept_len || !bonus) return DFL_ERR_INVALID_ARG;
    if (!aligned16(vlog)) return DFL_ERR_MISALIGNED;
    if ((size_t)N * K * (G + 1) > kNoAllocRows) return DFL_ERR_WORKSPACE;   // beyond the fixed array
    const DeviceCtx* ctx = current_ctx();
    if (!ctx) return DFL_ERR_NO_DEVICE;
    void* scratch = nullptr;
    const dfl_status rc = noalloc_scratch(ctx, &scratch);
    if (rc != DFL_OK) return rc;
    return self_select_run(vlog, dt == DFL_BF16, drafts, N, K, G, V, scores, selected, accept_len, bonus, scratch,
                           static_cast<cudaStream_t>(stream));
}

