// Per-position TV acceptance diagnostic and lossless stochastic acceptance.
//
// SpecDiff-2 notes, "Streak-Distillation": the acceptance probability of a
// position is proxied by alpha = 1 - 1/2 sum_x |P(x) - Q(x)| (P the verifier's
// distribution, Q the drafter's marginal), and the expected accepted length
// of a draft by the streak sum of its alphas.  DFlare post, "Generating
// candidates in parallel, the target decides acceptance": stochastic
// decoding needs an acceptance procedure that keeps the target's
// distribution -- accept x_j with probability min(1, P/Q), on the first
// rejection draw from the normalised residual max(0, P - Q), after a fully
// accepted window draw the bonus token from the next verifier row.
//
// Both start from per-row log-sum-exps (one HBM pass over each row), then
// a second pass forms probabilities from them.
#include <mutex>

#include "internal.h"
#include "philox.cuh"
#include "small_kernels.h"

namespace dfl {

namespace {

constexpr int XT = 256;   // threads per CTA

// Element i of a row stored as fp32 or bf16.
template <bool BF16>
__device__ __forceinline__ float elem(const void* row, int64_t i) {
    if constexpr (BF16) return __uint_as_float((uint32_t)static_cast<const uint16_t*>(row)[i] << 16);
    else return static_cast<const float*>(row)[i];
}

// Row address: row r of `rows` rows of length V; sequence-major layouts with
// an optional selected draft: r = (n, j) -> base + ((n*K + sel[n])*J + j)*V.
struct RowMap {
    const void* base;
    int K, J;             // drafts per sequence, rows per draft
    const int32_t* sel;   // nullable: draft 0
    int* err;             // nullable: error word for a selection outside 0..K-1
};

// Selected draft of sequence n; one outside 0..K-1 reads draft 0 and records
// DFL_ERR_INVALID_ARG in the error word.
__device__ __forceinline__ int64_t sel_of(const RowMap& m, int64_t n) {
    if (!m.sel) return 0;
    const int32_t k = m.sel[n];
    if (k >= 0 && k < m.K) return k;
    if (m.err) atomicCAS(m.err, 0, DFL_ERR_INVALID_ARG);
    return 0;
}

template <bool BF16>
__device__ __forceinline__ const void* row_ptr(const RowMap& m, int64_t r, int V) {
    const int64_t n = r / m.J, j = r % m.J;
    const int64_t k = sel_of(m, n);
    const int64_t off = ((n * m.K + k) * m.J + j) * (int64_t)V;
    return static_cast<const uint8_t*>(m.base) + off * (BF16 ? 2 : 4);
}

// 8 consecutive elements of a row (16-byte loads; row 16-byte aligned).
template <bool BF16>
__device__ __forceinline__ void load8(const void* row, int c, float (&x)[8]) {
    if constexpr (BF16) {
        const uint4 u = reinterpret_cast<const uint4*>(row)[c];
        x[0] = bf16lo(u.x); x[1] = bf16hi(u.x); x[2] = bf16lo(u.y); x[3] = bf16hi(u.y);
        x[4] = bf16lo(u.z); x[5] = bf16hi(u.z); x[6] = bf16lo(u.w); x[7] = bf16hi(u.w);
    } else {
        const float4 a = reinterpret_cast<const float4*>(row)[2 * c], b = reinterpret_cast<const float4*>(row)[2 * c + 1];
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    }
}

__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
    const float M = fmaxf(m, m2);
    s = (m == -INFINITY ? 0.f : s * expf(m - M)) + (m2 == -INFINITY ? 0.f : s2 * expf(m2 - M));
    m = M;
}

// lse[r] = log sum_x exp(scale * row[x]); one CTA per row, online rescaling,
// 16-byte loads when V is a multiple of 8.
template <bool BF16>
__global__ void __launch_bounds__(XT) row_lse_kernel(RowMap m, int V, float scale, float* lse) {
    grid_dep_begin();
    const int64_t r = blockIdx.x;
    const void* row = row_ptr<BF16>(m, r, V);
    float mx = -INFINITY, s = 0.f;
    if ((V & 7) == 0) {
        for (int c = threadIdx.x; c < V / 8; c += XT) {
            float x[8];
            load8<BF16>(row, c, x);
            float cm = x[0] * scale;
            #pragma unroll
            for (int q = 1; q < 8; ++q) cm = fmaxf(cm, x[q] * scale);
            if (cm > mx) { s = (mx == -INFINITY ? 0.f : s * expf(mx - cm)); mx = cm; }
            float a = 0.f;
            #pragma unroll
            for (int q = 0; q < 8; ++q) a += expf(x[q] * scale - mx);
            s += a;
        }
    } else {
        for (int i = threadIdx.x; i < V; i += XT) {
            const float x = elem<BF16>(row, i) * scale;
            if (x > mx) { s = (mx == -INFINITY ? 0.f : s * expf(mx - x)); mx = x; }
            s += expf(x - mx);
        }
    }
    #pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        lse_merge(mx, s, __shfl_xor_sync(0xFFFFFFFFu, mx, o), __shfl_xor_sync(0xFFFFFFFFu, s, o));
    __shared__ float sm[XT / 32], ss[XT / 32];
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) { sm[w] = mx; ss[w] = s; }
    __syncthreads();
    if (threadIdx.x == 0) {
        float M = sm[0], S = ss[0];
        for (int i = 1; i < XT / 32; ++i) lse_merge(M, S, sm[i], ss[i]);
        lse[r] = M + logf(S);
    }
}

// alpha[n][k][j] = 1 - 1/2 sum_x |exp(v - lse_v) - exp(z / T - lse_z)|.
// One CTA per window row (n, j): the drafter's row is read once for all K
// verifier rows of that position, in chunks of 8 drafts.
template <bool BF16>
__global__ void __launch_bounds__(XT) tv_alpha_kernel(const float* logits, const float* lse_z, float inv_T,
                                                      const void* vlog, const float* lse_v, int K, int G, int V,
                                                      float* alpha) {
    grid_dep_begin();
    const int64_t nj = blockIdx.x;   // n * G + j
    const int64_t n = nj / G, j = nj % G;
    const float* z = logits + nj * V;
    const float lz = lse_z[nj];
    __shared__ float red[XT / 32][8];
    for (int k0 = 0; k0 < K; k0 += 8) {
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        const void* vr[8];
        float lv[8];
        #pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int k = k0 + q < K ? k0 + q : k0;
            const int64_t row = (n * K + k) * (G + 1) + j;
            vr[q] = static_cast<const uint8_t*>(vlog) + row * (int64_t)V * (BF16 ? 2 : 4);
            lv[q] = lse_v[row];
        }
        if ((V & 7) == 0) {
            // exp(a - b) = 2^(a log2(e) - b log2(e)): one FMA and one SFU op per element
            constexpr float L2E = 1.4426950408889634f;
            const float zs = inv_T * L2E, zo = -lz * L2E;
            float vo[8];
            #pragma unroll
            for (int q = 0; q < 8; ++q) vo[q] = -lv[q] * L2E;
            for (int c = threadIdx.x; c < V / 8; c += XT) {
                float zz[8], qx[8];
                load8<false>(z, c, zz);
                #pragma unroll
                for (int e = 0; e < 8; ++e) qx[e] = ex2_ftz(fmaf(zz[e], zs, zo));
                #pragma unroll
                for (int q = 0; q < 8; ++q) {
                    float vv[8];
                    load8<BF16>(vr[q], c, vv);
                    #pragma unroll
                    for (int e = 0; e < 8; ++e) acc[q] += fabsf(ex2_ftz(fmaf(vv[e], L2E, vo[q])) - qx[e]);
                }
            }
        } else {
            for (int i = threadIdx.x; i < V; i += XT) {
                const float qx = expf(z[i] * inv_T - lz);
                #pragma unroll
                for (int q = 0; q < 8; ++q) acc[q] += fabsf(expf(elem<BF16>(vr[q], i) - lv[q]) - qx);
            }
        }
        const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
        #pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float t = warp_sum(acc[q]);
            if (l == 0) red[w][q] = t;
        }
        __syncthreads();
        if (threadIdx.x < 8 && k0 + (int)threadIdx.x < K) {
            float t = 0.f;
            for (int i = 0; i < XT / 32; ++i) t += red[i][threadIdx.x];
            alpha[(n * K + k0 + threadIdx.x) * G + j] = 1.f - 0.5f * t;
        }
        __syncthreads();
    }
}

// tokens_per_draft[n][k] = sum_m prod_{j<=m} alpha[n][k][j] (fp64).
__global__ void tv_streak_kernel(const float* alpha, int64_t NK, int G, float* tpd) {
    grid_dep_begin();
    const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (i >= NK) return;
    double prod = 1.0, tot = 0.0;
    for (int j = 0; j < G; ++j) {
        prod *= (double)alpha[i * G + j];
        tot += prod;
    }
    tpd[i] = (float)tot;
}

// Lossless stochastic acceptance, in three kernels so that the
// vocabulary-wide work of the correction draw spreads over the whole GPU.
//  1. spec_test_kernel: per sequence, the acceptance tests u Q(x_j) < P(x_j)
//     in order; stop[n] = first rejected position (G if none).
//  2. residual_group_kernel: for every (sequence, group of RG consecutive
//     tokens) the sum of the draw's weights -- max(0, P - Q) of the rejected
//     position, or P of the bonus row -- lanes adding strided elements
//     (coalesced) in fp32, the group total in fp64.
//  3. residual_pick_kernel: per sequence, an exclusive scan of the group
//     sums, the group holding u * total, and an index-ordered fp64 walk of that
//     group; a target that the walk does not reach (rounding at the group's
//     end) takes the group's last token.
constexpr int RG = 1024;

struct SpecArgs {
    const float* logits;
    const float* lse_z;
    float inv_T;
    RowMap vm;
    const float* lse_v;   // [N][G+1] rows of the verified draft, or [N][K][G+1] when lse_all
    int lse_all;
    const int32_t* drafts;
    int G, V;
    uint32_t key0, key1;
    int* stop;        // [N]
    double* gsum;     // [N][ngroups]
    int ngroups;
};

__device__ __forceinline__ float lse_row(const SpecArgs& a, int64_t n, int j) {
    if (!a.lse_all) return a.lse_v[n * (a.G + 1) + j];
    const int64_t k = sel_of(a.vm, n);
    return a.lse_v[(n * a.vm.K + k) * (a.G + 1) + j];
}

template <bool BF16>
__device__ __forceinline__ float draw_weight(const SpecArgs& a, int64_t n, int j, int i) {
    const bool bonus = (j == a.G);
    const void* vr = row_ptr<BF16>(a.vm, n * (a.G + 1) + j, a.V);
    const float p = expf(elem<BF16>(vr, i) - lse_row(a, n, j));
    if (bonus) return p;
    const float q = expf(a.logits[(n * a.G + j) * (int64_t)a.V + i] * a.inv_T - a.lse_z[n * a.G + j]);
    return p > q ? p - q : 0.f;
}

template <bool BF16>
__global__ void spec_test_kernel(const SpecArgs a, int N) {
    grid_dep_begin();
    const int64_t n = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (n >= N) return;
    const int64_t kd = sel_of(a.vm, n);
    const int32_t* x = a.drafts + (n * a.vm.K + kd) * a.G;
    int j = 0;
    for (; j < a.G; ++j) {
        const int32_t xj = x[j];
        if (xj < 0 || xj >= a.V) break;   // not a token: rejected
        const float* z = a.logits + (n * a.G + j) * (int64_t)a.V;
        const void* vr = row_ptr<BF16>(a.vm, n * (a.G + 1) + j, a.V);
        const double q = exp((double)(z[xj] * a.inv_T - a.lse_z[n * a.G + j]));
        const double p = exp((double)(elem<BF16>(vr, xj) - lse_row(a, n, j)));
        const double u = philox_uniform24((uint32_t)n, (uint32_t)j, 0u, 1u, a.key0, a.key1);
        if (!(u * q < p)) break;
    }
    a.stop[n] = j;
}

template <bool BF16>
__global__ void residual_group_kernel(const SpecArgs a) {
    grid_dep_begin();
    const int64_t n = blockIdx.y;
    const int g = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (g >= a.ngroups) return;
    const int j = a.stop[n];
    const int b = g * RG;
    float acc = 0.f;
    for (int i = b + lane; i < b + RG && i < a.V; i += 32) acc += draw_weight<BF16>(a, n, j, i);
    double t = (double)acc;
    #pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, o);
    if (lane == 0) a.gsum[n * a.ngroups + g] = t;
}

template <bool BF16>
__global__ void residual_pick_kernel(const SpecArgs a, int32_t* accept_len, int32_t* next_token) {
    grid_dep_begin();
    const int64_t n = blockIdx.x;
    const int lane = threadIdx.x;
    const int j = a.stop[n];
    const double* gs = a.gsum + n * a.ngroups;
    // total and the group holding the target (lane 0, in group order)
    __shared__ int gsel;
    __shared__ double excl_s;
    if (lane == 0) {
        double total = 0.0;
        for (int g = 0; g < a.ngroups; ++g) total += gs[g];
        const double u = philox_uniform24((uint32_t)n, (uint32_t)j, 0u, 2u, a.key0, a.key1);
        const double target = u * total;
        double run = 0.0;
        int g = 0;
        for (; g < a.ngroups - 1; ++g) {
            if (run + gs[g] > target) break;
            run += gs[g];
        }
        gsel = g;
        excl_s = target - run;   // target relative to the group's start
    }
    __syncwarp();
    const int g = gsel;
    const double rel = excl_s;
    const int b0 = g * RG, b1 = min(a.V, b0 + RG);
    double run = 0.0;
    int pick = b1 - 1;
    for (int b = b0; b < b1; b += 32) {
        double x = (b + lane < b1) ? (double)draw_weight<BF16>(a, n, j, b + lane) : 0.0;
        #pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(0xFFFFFFFFu, x, o);
            if (lane >= o) x += y;
        }
        const unsigned hit = __ballot_sync(0xFFFFFFFFu, b + lane < b1 && run + x > rel);
        if (hit) { pick = b + __ffs(hit) - 1; break; }
        run += __shfl_sync(0xFFFFFFFFu, x, 31);
    }
    if (lane == 0) {
        accept_len[n] = j;
        next_token[n] = pick;
    }
}

// Sampled-greedy acceptance (SpecDiff-2 notes, "Self-Selection Acceptance"
// and "Streak-Distillation", read at temperature above zero): at every
// window position j the verifier draws its own token y_j from P_j =
// softmax(v_j) by inverse CDF at the Philox uniform of counter (n, j, 0, 3);
// draft token x_j is accepted while it equals y_j, and the verifier's sample
// at the first mismatch (y_G after a fully accepted window) is the committed
// token.  All G+1 draws of a sequence are made in parallel:
//  1. vdraw_group_kernel: per (row, group of RG tokens) the sum of the row's
//     weights exp(v - lse), lanes adding 8 consecutive elements per 16-byte
//     load in fp32, the group total in fp64;
//  2. vdraw_pick_kernel: per row, the group holding u * total (exclusive scan
//     of the group sums) and an index-ordered fp64 walk of that group;
//  3. sg_accept_kernel: per sequence, the first mismatch by warp ballot.
struct SgArgs {
    RowMap vm;            // verifier rows of the verified draft: r = n * (G+1) + j
    const float* lse_v;   // [N][G+1], or [N][K][G+1] when lse_all
    int lse_all;
    int G, V;
    uint32_t key0, key1;
    double* gsum;         // [N*(G+1)][ngroups]
    int32_t* y;           // [N*(G+1)] the verifier's samples
    int ngroups;
};

__device__ __forceinline__ float sg_lse(const SgArgs& a, int64_t r) {
    if (!a.lse_all) return a.lse_v[r];
    const int64_t n = r / (a.G + 1), j = r % (a.G + 1);
    const int64_t k = sel_of(a.vm, n);
    return a.lse_v[(n * a.vm.K + k) * (a.G + 1) + j];
}

template <bool BF16>
__global__ void vdraw_group_kernel(const SgArgs a) {
    grid_dep_begin();
    const int64_t r = blockIdx.x;
    const int g = blockIdx.y * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (g >= a.ngroups) return;
    const void* vr = row_ptr<BF16>(a.vm, r, a.V);
    const float lse = sg_lse(a, r);
    const int b = g * RG, e = min(a.V, b + RG);
    float acc = 0.f;
    if ((a.V & 7) == 0) {   // group bounds are multiples of 8
        for (int c = b / 8 + lane; c < e / 8; c += 32) {
            float x[8];
            load8<BF16>(vr, c, x);
            #pragma unroll
            for (int q = 0; q < 8; ++q) acc += expf(x[q] - lse);
        }
    } else {
        for (int i = b + lane; i < e; i += 32) acc += expf(elem<BF16>(vr, i) - lse);
    }
    double t = (double)acc;
    #pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, o);
    if (lane == 0) a.gsum[r * a.ngroups + g] = t;
}

template <bool BF16>
__global__ void vdraw_pick_kernel(const SgArgs a) {
    grid_dep_begin();
    const int64_t r = blockIdx.x;
    const int lane = threadIdx.x;
    const int64_t n = r / (a.G + 1);
    const int j = (int)(r % (a.G + 1));
    const double* gs = a.gsum + r * a.ngroups;
    // The row's total (lane-strided partial sums, a fixed tree to lane 0, then
    // broadcast so that every lane holds the same value) and the group holding
    // u * total: an exclusive scan of the group sums 32 groups at a time,
    // the last group taking a target that rounding puts past the others.
    double part = 0.0;
    for (int gg = lane; gg < a.ngroups; gg += 32) part += gs[gg];
    #pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_down_sync(0xFFFFFFFFu, part, o);
    const double total = __shfl_sync(0xFFFFFFFFu, part, 0);
    const double target = philox_uniform24((uint32_t)n, (uint32_t)j, 0u, 3u, a.key0, a.key1) * total;
    int g = a.ngroups - 1;
    double before = 0.0;   // sum of the groups before the chunk
    bool found = false;
    for (int base = 0; base < a.ngroups - 1 && !found; base += 32) {
        const int gg = base + lane;
        double x = gg < a.ngroups - 1 ? gs[gg] : 0.0;
        #pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(0xFFFFFFFFu, x, o);
            if (lane >= o) x += y;
        }
        const unsigned hit = __ballot_sync(0xFFFFFFFFu, gg < a.ngroups - 1 && before + x > target);
        const double excl = __shfl_up_sync(0xFFFFFFFFu, x, 1);   // lane l: groups base .. base + l - 1
        if (hit) {
            const int l = __ffs(hit) - 1;
            const double e = __shfl_sync(0xFFFFFFFFu, excl, l);
            g = base + l;
            before += l ? e : 0.0;
            found = true;
        } else {
            before += __shfl_sync(0xFFFFFFFFu, x, 31);
        }
    }
    const double rel = target - before;
    const void* vr = row_ptr<BF16>(a.vm, r, a.V);
    const float lse = sg_lse(a, r);
    const int b0 = g * RG, b1 = min(a.V, b0 + RG);
    double run = 0.0;
    int pick = b1 - 1;   // a target the walk does not reach (rounding at the group's end)
    for (int b = b0; b < b1; b += 32) {
        double x = (b + lane < b1) ? (double)expf(elem<BF16>(vr, b + lane) - lse) : 0.0;
        #pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double t = __shfl_up_sync(0xFFFFFFFFu, x, o);
            if (lane >= o) x += t;
        }
        const unsigned hit = __ballot_sync(0xFFFFFFFFu, b + lane < b1 && run + x > rel);
        if (hit) { pick = b + __ffs(hit) - 1; break; }
        run += __shfl_sync(0xFFFFFFFFu, x, 31);
    }
    if (lane == 0) a.y[r] = pick;
}

__global__ void sg_accept_kernel(const SgArgs a, const int32_t* drafts, int N, int32_t* accept_len,
                                 int32_t* next_token) {
    grid_dep_begin();
    const int64_t n = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (n >= N) return;
    const int64_t k = sel_of(a.vm, n);
    const int32_t* x = drafts + (n * a.vm.K + k) * a.G;
    const int32_t* y = a.y + n * (a.G + 1);
    int acc = a.G;
    for (int j0 = 0; j0 < a.G; j0 += 32) {
        const int j = j0 + lane;
        const unsigned miss = __ballot_sync(0xFFFFFFFFu, j < a.G && x[j] != y[j]);
        if (miss) { acc = j0 + __ffs(miss) - 1; break; }
    }
    if (lane == 0) {
        accept_len[n] = acc;
        next_token[n] = y[acc];
    }
}

inline size_t al256(size_t b) { return (b + 255) & ~size_t(255); }

// The current device's error word (nullptr if none is current).
inline int* err_word() {
    DeviceCtx* c = current_ctx();
    return c ? c->err_word : nullptr;
}

}  // namespace

size_t tv_ws_bytes(int N, int K, int G) { return al256((size_t)N * G * 4) + al256((size_t)N * K * (G + 1) * 4); }
size_t spec_ws_bytes(int N, int G, int V) {
    const size_t ng = (size_t)(V + RG - 1) / RG;
    return al256((size_t)N * G * 4) + al256((size_t)N * (G + 1) * 4) + al256((size_t)N * 4) + al256((size_t)N * ng * 8);
}

// Internal runners with precomputed log-sum-exps (used by the draft step,
// which already has the verifier rows' LSEs from self-selection).
dfl_status lse_rows_f32(const float* logits, int rows, int V, float inv_T, float* lse, cudaStream_t st) {
    ProfScope ps("row_lse", st);
    launch_pdl(row_lse_kernel<false>, (unsigned)rows, XT, 0, st, RowMap{logits, 1, 1, nullptr}, V, inv_T, lse);
    return last_launch();
}

dfl_status tv_run(const float* logits, float inv_T, const void* vlog, bool bf, int N, int K, int G, int V,
                  float* alpha, float* tpd, const float* lse_z, const float* lse_v_all, cudaStream_t st) {
    {
        ProfScope ps("tv_alpha", st);
        if (bf) launch_pdl(tv_alpha_kernel<true>, (unsigned)(N * G), XT, 0, st, logits, lse_z, inv_T, vlog, lse_v_all,
                           K, G, V, alpha);
        else launch_pdl(tv_alpha_kernel<false>, (unsigned)(N * G), XT, 0, st, logits, lse_z, inv_T, vlog, lse_v_all,
                        K, G, V, alpha);
    }
    dfl_status rc = last_launch();
    if (rc != DFL_OK || !tpd) return rc;
    ProfScope ps("tv_streak", st);
    launch_pdl(tv_streak_kernel, (unsigned)((N * K + 127) / 128), 128, 0, st, alpha, (int64_t)N * K, G, tpd);
    return last_launch();
}

size_t spec_scratch_bytes(int N, int V) {
    return al256((size_t)N * 4) + al256((size_t)N * ((V + RG - 1) / RG) * 8);
}

dfl_status spec_run(const float* logits, float inv_T, const void* vlog, bool bf, const int32_t* drafts,
                    const int32_t* sel, int N, int K, int G, int V, uint64_t seed, int32_t* accept_len,
                    int32_t* next_token, const float* lse_z, const float* lse_v, bool lse_all, void* scratch,
                    cudaStream_t st) {
    ProfScope ps("spec_accept", st);
    SpecArgs sa{logits, lse_z, inv_T, RowMap{vlog, K, G + 1, sel, err_word()}, lse_v, lse_all ? 1 : 0, drafts, G, V,
                (uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32), nullptr, nullptr, (V + RG - 1) / RG};
    uint8_t* p = static_cast<uint8_t*>(scratch);
    sa.stop = reinterpret_cast<int*>(p);
    sa.gsum = reinterpret_cast<double*>(p + al256((size_t)N * 4));
    const dim3 ggrid((sa.ngroups + 7) / 8, N);
    if (bf) {
        launch_pdl(spec_test_kernel<true>, (N + 127) / 128, 128, 0, st, sa, N);
        launch_pdl(residual_group_kernel<true>, ggrid, 256, 0, st, sa);
        launch_pdl(residual_pick_kernel<true>, N, 32, 0, st, sa, accept_len, next_token);
    } else {
        launch_pdl(spec_test_kernel<false>, (N + 127) / 128, 128, 0, st, sa, N);
        launch_pdl(residual_group_kernel<false>, ggrid, 256, 0, st, sa);
        launch_pdl(residual_pick_kernel<false>, N, 32, 0, st, sa, accept_len, next_token);
    }
    return last_launch();
}

size_t sg_scratch_bytes(int N, int G, int V) {
    const size_t rows = (size_t)N * (G + 1);
    return al256(rows * 4) + al256(rows * ((V + RG - 1) / RG) * 8);
}

size_t sg_ws_bytes(int N, int G, int V) { return al256((size_t)N * (G + 1) * 4) + sg_scratch_bytes(N, G, V); }

dfl_status sg_run(const void* vlog, bool bf, const int32_t* drafts, const int32_t* sel, int N, int K, int G, int V,
                  uint64_t seed, int32_t* accept_len, int32_t* next_token, const float* lse_v, bool lse_all,
                  void* scratch, cudaStream_t st) {
    if ((int64_t)V > (int64_t)65535 * 8 * RG) return DFL_ERR_UNSUPPORTED_SHAPE;   // groups of a row: grid.y
    ProfScope ps("sampled_greedy", st);
    SgArgs sa{RowMap{vlog, K, G + 1, sel, err_word()}, lse_v, lse_all ? 1 : 0, G, V, (uint32_t)(seed & 0xFFFFFFFFu),
              (uint32_t)(seed >> 32), nullptr, nullptr, (V + RG - 1) / RG};
    uint8_t* p = static_cast<uint8_t*>(scratch);
    const int64_t rows = (int64_t)N * (G + 1);
    sa.y = reinterpret_cast<int32_t*>(p);
    sa.gsum = reinterpret_cast<double*>(p + al256((size_t)rows * 4));
    const dim3 ggrid((unsigned)rows, (sa.ngroups + 7) / 8);
    if (bf) {
        launch_pdl(vdraw_group_kernel<true>, ggrid, 256, 0, st, sa);
        launch_pdl(vdraw_pick_kernel<true>, (unsigned)rows, 32, 0, st, sa);
    } else {
        launch_pdl(vdraw_group_kernel<false>, ggrid, 256, 0, st, sa);
        launch_pdl(vdraw_pick_kernel<false>, (unsigned)rows, 32, 0, st, sa);
    }
    launch_pdl(sg_accept_kernel, (N + 3) / 4, 128, 0, st, sa, drafts, N, accept_len, next_token);
    return last_launch();
}

}  // namespace dfl

using namespace dfl;

extern "C" dfl_status dfl_tv_acceptance(const float* logits, float T, const void* vlog, dfl_dtype dt, int32_t N,
                                        int32_t K, int32_t G, int32_t V, float* alpha, float* tokens_per_draft,
                                        void* ws, size_t ws_bytes, dfl_stream stream) {
    const dfl::ApiRange nvtx_range("dfl_tv_acceptance");
    if (!logits || !vlog || !alpha || !ws || N <= 0 || K < 1 || K > 64 || G < 1 || G > 1024 || V <= 0 ||
        !(T > 0.f))
        return DFL_ERR_INVALID_ARG;
    if (dt != DFL_F32 && dt != DFL_BF16) return DFL_ERR_INVALID_ARG;
    // rows are read with 16-byte loads when V % 8 == 0
    if (!aligned16(logits) || !aligned16(vlog) || !aligned16(ws)) return DFL_ERR_MISALIGNED;
    if (ws_bytes < tv_ws_bytes(N, K, G)) return DFL_ERR_WORKSPACE;
    if (!current_ctx()) return DFL_ERR_NO_DEVICE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    float* lse_z = static_cast<float*>(ws);
    float* lse_v = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + al256((size_t)N * G * 4));
    const float inv_T = 1.0f / T;
    const bool bf = dt == DFL_BF16;
    {
        ProfScope ps("row_lse", st);
        launch_pdl(row_lse_kernel<false>, (unsigned)(N * G), XT, 0, st, RowMap{logits, 1, G, nullptr}, V, inv_T, lse_z);
        // every verifier row of every draft, [N*K][G+1]
        const RowMap all{vlog, 1, G + 1, nullptr};
        if (bf) launch_pdl(row_lse_kernel<true>, (unsigned)(N * K * (G + 1)), XT, 0, st, all, V, 1.f, lse_v);
        else launch_pdl(row_lse_kernel<false>, (unsigned)(N * K * (G + 1)), XT, 0, st, all, V, 1.f, lse_v);
    }
    dfl_status rc = last_launch();
    if (rc != DFL_OK) return rc;
    return tv_run(logits, inv_T, vlog, bf, N, K, G, V, alpha, tokens_per_draft, lse_z, lse_v, st);
}

extern "C" dfl_status dfl_spec_accept(const float* logits, float T, const void* vlog, dfl_dtype dt,
                                      const int32_t* drafts, const int32_t* sel, int32_t N, int32_t K, int32_t G,
                                      int32_t V, uint64_t seed, int32_t* accept_len, int32_t* next_token, void* ws,
                                      size_t ws_bytes, dfl_stream stream) {
    const dfl::ApiRange nvtx_range("dfl_spec_accept");
    if (!logits || !vlog || !drafts || !accept_len || !next_token || !ws || N <= 0 || K < 1 || K > 64 || G < 1 ||
        G > 1024 || V <= 0 || !(T > 0.f))
        return DFL_ERR_INVALID_ARG;
    if (dt != DFL_F32 && dt != DFL_BF16) return DFL_ERR_INVALID_ARG;
    if (!aligned16(logits) || !aligned16(vlog) || !aligned16(ws)) return DFL_ERR_MISALIGNED;
    if (ws_bytes < spec_ws_bytes(N, G, V)) return DFL_ERR_WORKSPACE;
    if (!current_ctx()) return DFL_ERR_NO_DEVICE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    float* lse_z = static_cast<float*>(ws);
    float* lse_v = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + al256((size_t)N * G * 4));
    const float inv_T = 1.0f / T;
    const bool bf = dt == DFL_BF16;
    const RowMap vm{vlog, K, G + 1, sel, err_word()};
    {
        ProfScope ps("row_lse", st);
        launch_pdl(row_lse_kernel<false>, (unsigned)(N * G), XT, 0, st, RowMap{logits, 1, G, nullptr}, V, inv_T, lse_z);
        if (bf) launch_pdl(row_lse_kernel<true>, (unsigned)(N * (G + 1)), XT, 0, st, vm, V, 1.f, lse_v);
        else launch_pdl(row_lse_kernel<false>, (unsigned)(N * (G + 1)), XT, 0, st, vm, V, 1.f, lse_v);
    }
    dfl_status rc = last_launch();
    if (rc != DFL_OK) return rc;
    return spec_run(logits, inv_T, vlog, bf, drafts, sel, N, K, G, V, seed, accept_len, next_token, lse_z, lse_v,
                    false, static_cast<uint8_t*>(ws) + al256((size_t)N * G * 4) + al256((size_t)N * (G + 1) * 4), st);
}

extern "C" dfl_status dfl_sampled_greedy_accept(const void* vlog, dfl_dtype dt, const int32_t* drafts,
                                                const int32_t* sel, int32_t N, int32_t K, int32_t G, int32_t V,
                                                uint64_t seed, int32_t* accept_len, int32_t* next_token, void* ws,
                                                size_t ws_bytes, dfl_stream stream) {
    const dfl::ApiRange nvtx_range("dfl_sampled_greedy_accept");
    if (!vlog || !drafts || !accept_len || !next_token || !ws || N <= 0 || K < 1 || K > 64 || G < 1 || G > 1024 ||
        V <= 0)
        return DFL_ERR_INVALID_ARG;
    if (dt != DFL_F32 && dt != DFL_BF16) return DFL_ERR_INVALID_ARG;
    if (!aligned16(vlog) || !aligned16(ws)) return DFL_ERR_MISALIGNED;
    if (ws_bytes < sg_ws_bytes(N, G, V)) return DFL_ERR_WORKSPACE;
    if (!current_ctx()) return DFL_ERR_NO_DEVICE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    float* lse_v = static_cast<float*>(ws);
    const bool bf = dt == DFL_BF16;
    {
        ProfScope ps("row_lse", st);
        const RowMap vm{vlog, K, G + 1, sel, err_word()};
        if (bf) launch_pdl(row_lse_kernel<true>, (unsigned)(N * (G + 1)), XT, 0, st, vm, V, 1.f, lse_v);
        else launch_pdl(row_lse_kernel<false>, (unsigned)(N * (G + 1)), XT, 0, st, vm, V, 1.f, lse_v);
    }
    dfl_status rc = last_launch();
    if (rc != DFL_OK) return rc;
    return sg_run(vlog, bf, drafts, sel, N, K, G, V, seed, accept_len, next_token, lse_v, false,
                  static_cast<uint8_t*>(ws) + al256((size_t)N * (G + 1) * 4), st);
}
