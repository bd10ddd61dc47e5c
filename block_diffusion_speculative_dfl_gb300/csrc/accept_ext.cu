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
#include "small_kernels.h"

namespace dfl {

namespace {

constexpr int XT = 256;   // threads per CTA

// Philox4x32-10 word 0 (Salmon, Moraes, Dror & Shaw, SC'11); the sampling
// kernel carries its own copy so that this file stands alone.
__device__ __forceinline__ uint32_t philox0(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0,
                                            uint32_t k1) {
    #pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
        const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
        const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c0;
}

__device__ __forceinline__ double uniform24(uint32_t x0) { return ((double)(x0 >> 8) + 0.5) * (1.0 / 16777216.0); }

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
};

template <bool BF16>
__device__ __forceinline__ const void* row_ptr(const RowMap& m, int64_t r, int V) {
    const int64_t n = r / m.J, j = r % m.J;
    const int64_t k = m.sel ? m.sel[n] : 0;
    const int64_t off = ((n * m.K + k) * m.J + j) * (int64_t)V;
    return static_cast<const uint8_t*>(m.base) + off * (BF16 ? 2 : 4);
}

// lse[r] = log sum_x exp(scale * row[x]); one CTA per row, online rescaling.
template <bool BF16>
__global__ void __launch_bounds__(XT) row_lse_kernel(RowMap m, int V, float scale, float* lse) {
    const int64_t r = blockIdx.x;
    const void* row = row_ptr<BF16>(m, r, V);
    float mx = -INFINITY, s = 0.f;
    for (int i = threadIdx.x; i < V; i += XT) {
        const float x = elem<BF16>(row, i) * scale;
        if (x > mx) { s = (mx == -INFINITY ? 0.f : s * expf(mx - x)); mx = x; }
        s += expf(x - mx);
    }
    #pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xFFFFFFFFu, mx, o), s2 = __shfl_xor_sync(0xFFFFFFFFu, s, o);
        const float M = fmaxf(mx, m2);
        s = (mx == -INFINITY ? 0.f : s * expf(mx - M)) + (m2 == -INFINITY ? 0.f : s2 * expf(m2 - M));
        mx = M;
    }
    __shared__ float sm[XT / 32], ss[XT / 32];
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) { sm[w] = mx; ss[w] = s; }
    __syncthreads();
    if (threadIdx.x == 0) {
        float M = sm[0], S = ss[0];
        for (int i = 1; i < XT / 32; ++i) {
            const float M2 = fmaxf(M, sm[i]);
            S = (M == -INFINITY ? 0.f : S * expf(M - M2)) + (sm[i] == -INFINITY ? 0.f : ss[i] * expf(sm[i] - M2));
            M = M2;
        }
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
        for (int i = threadIdx.x; i < V; i += XT) {
            const float qx = expf(z[i] * inv_T - lz);
            #pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] += fabsf(expf(elem<BF16>(vr[q], i) - lv[q]) - qx);
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
    const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (i >= NK) return;
    double prod = 1.0, tot = 0.0;
    for (int j = 0; j < G; ++j) {
        prod *= (double)alpha[i * G + j];
        tot += prod;
    }
    tpd[i] = (float)tot;
}

// Lossless stochastic acceptance of one draft per sequence; one CTA per
// sequence.  Thread 0 runs the acceptance tests; all threads then draw the
// correction (or bonus) token by inverting the CDF of the residual, each
// thread owning a contiguous chunk of the vocabulary: chunk sums in fp64, an
// exclusive scan, and a sequential re-walk of the chunk that holds the target
// with the same arithmetic.
template <bool BF16>
__global__ void __launch_bounds__(XT) spec_accept_kernel(const float* logits, const float* lse_z, float inv_T,
                                                         RowMap vm, const float* lse_v, const int32_t* drafts,
                                                         int G, int V, uint32_t key0, uint32_t key1,
                                                         int32_t* accept_len, int32_t* next_token) {
    const int64_t n = blockIdx.x;
    const int64_t kd = vm.sel ? vm.sel[n] : 0;
    const int32_t* x = drafts + (n * vm.K + kd) * G;
    __shared__ int stop;
    __shared__ double chunk[XT];
    __shared__ double total_s;
    if (threadIdx.x == 0) {
        int j = 0;
        for (; j < G; ++j) {
            const int32_t xj = x[j];
            if (xj < 0 || xj >= V) break;   // not a token: rejected
            const float* z = logits + (n * G + j) * (int64_t)V;
            const void* vr = row_ptr<BF16>(vm, n * (G + 1) + j, V);
            const double q = exp((double)(z[xj] * inv_T - lse_z[n * G + j]));
            const double p = exp((double)(elem<BF16>(vr, xj) - lse_v[n * (G + 1) + j]));
            const double u = uniform24(philox0((uint32_t)n, (uint32_t)j, 0u, 1u, key0, key1));
            if (!(u * q < p)) break;
        }
        stop = j;
    }
    __syncthreads();
    const int j = stop;
    const bool bonus = (j == G);
    const float* z = logits + (n * G + (bonus ? 0 : j)) * (int64_t)V;
    const float lz = bonus ? 0.f : lse_z[n * G + j];
    const void* vr = row_ptr<BF16>(vm, n * (G + 1) + j, V);
    const float lv = lse_v[n * (G + 1) + j];
    const int per = (V + XT - 1) / XT;
    const int c0 = threadIdx.x * per, c1 = min(V, c0 + per);
    auto weight = [&](int i) -> double {
        const float p = expf(elem<BF16>(vr, i) - lv);
        if (bonus) return (double)p;
        const float q = expf(z[i] * inv_T - lz);
        return p > q ? (double)p - (double)q : 0.0;
    };
    double s = 0.0;
    for (int i = c0; i < c1; ++i) s += weight(i);
    chunk[threadIdx.x] = s;
    __syncthreads();
    if (threadIdx.x == 0) {   // exclusive scan of the chunk sums (256 entries)
        double run = 0.0;
        for (int t = 0; t < XT; ++t) { const double c = chunk[t]; chunk[t] = run; run += c; }
        total_s = run;
    }
    __syncthreads();
    const double total = total_s;
    const double u = uniform24(philox0((uint32_t)n, (uint32_t)j, 0u, 2u, key0, key1));
    const double target = u * total;
    const double excl = chunk[threadIdx.x];
    const double next = threadIdx.x + 1 < XT ? chunk[threadIdx.x + 1] : total;
    // The chunk whose [excl, next) holds the target walks itself again, adding
    // from zero in the same order as its chunk sum; the last non-empty chunk
    // also takes a target at or beyond the total (rounding).
    const bool last = c1 == V;
    if (c0 < c1 && target >= excl && (target < next || last)) {
        const double rel = target - excl;
        double run = 0.0;
        int pick = c1 - 1;
        for (int i = c0; i < c1; ++i) {
            run += weight(i);
            if (run > rel) { pick = i; break; }
        }
        accept_len[n] = j;
        next_token[n] = pick;
    }
}

inline size_t al256(size_t b) { return (b + 255) & ~size_t(255); }

}  // namespace

size_t tv_ws_bytes(int N, int K, int G) { return al256((size_t)N * G * 4) + al256((size_t)N * K * (G + 1) * 4); }
size_t spec_ws_bytes(int N, int G) { return al256((size_t)N * G * 4) + al256((size_t)N * (G + 1) * 4); }

}  // namespace dfl

using namespace dfl;

extern "C" dfl_status dfl_tv_acceptance(const float* logits, float T, const void* vlog, dfl_dtype dt, int32_t N,
                                        int32_t K, int32_t G, int32_t V, float* alpha, float* tokens_per_draft,
                                        void* ws, size_t ws_bytes, dfl_stream stream) {
    if (!logits || !vlog || !alpha || !ws || N <= 0 || K < 1 || K > 64 || G < 1 || G > 1024 || V <= 0 ||
        !(T > 0.f))
        return DFL_ERR_INVALID_ARG;
    if (dt != DFL_F32 && dt != DFL_BF16) return DFL_ERR_INVALID_ARG;
    if (ws_bytes < tv_ws_bytes(N, K, G)) return DFL_ERR_WORKSPACE;
    if (!current_ctx()) return DFL_ERR_NO_DEVICE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    float* lse_z = static_cast<float*>(ws);
    float* lse_v = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + al256((size_t)N * G * 4));
    const float inv_T = 1.0f / T;
    const bool bf = dt == DFL_BF16;
    {
        ProfScope ps("row_lse", st);
        row_lse_kernel<false><<<(unsigned)(N * G), XT, 0, st>>>(RowMap{logits, 1, G, nullptr}, V, inv_T, lse_z);
        // every verifier row of every draft, [N*K][G+1]
        const RowMap all{vlog, 1, G + 1, nullptr};
        if (bf) row_lse_kernel<true><<<(unsigned)(N * K * (G + 1)), XT, 0, st>>>(all, V, 1.f, lse_v);
        else row_lse_kernel<false><<<(unsigned)(N * K * (G + 1)), XT, 0, st>>>(all, V, 1.f, lse_v);
    }
    dfl_status rc = last_launch();
    if (rc != DFL_OK) return rc;
    {
        ProfScope ps("tv_alpha", st);
        if (bf) tv_alpha_kernel<true><<<(unsigned)(N * G), XT, 0, st>>>(logits, lse_z, inv_T, vlog, lse_v, K, G, V, alpha);
        else tv_alpha_kernel<false><<<(unsigned)(N * G), XT, 0, st>>>(logits, lse_z, inv_T, vlog, lse_v, K, G, V, alpha);
    }
    if ((rc = last_launch()) != DFL_OK || !tokens_per_draft) return rc;
    ProfScope ps("tv_streak", st);
    tv_streak_kernel<<<(unsigned)((N * K + 127) / 128), 128, 0, st>>>(alpha, (int64_t)N * K, G, tokens_per_draft);
    return last_launch();
}

extern "C" dfl_status dfl_spec_accept(const float* logits, float T, const void* vlog, dfl_dtype dt,
                                      const int32_t* drafts, const int32_t* sel, int32_t N, int32_t K, int32_t G,
                                      int32_t V, uint64_t seed, int32_t* accept_len, int32_t* next_token, void* ws,
                                      size_t ws_bytes, dfl_stream stream) {
    if (!logits || !vlog || !drafts || !accept_len || !next_token || !ws || N <= 0 || K < 1 || K > 64 || G < 1 ||
        G > 1024 || V <= 0 || !(T > 0.f))
        return DFL_ERR_INVALID_ARG;
    if (dt != DFL_F32 && dt != DFL_BF16) return DFL_ERR_INVALID_ARG;
    if (ws_bytes < spec_ws_bytes(N, G)) return DFL_ERR_WORKSPACE;
    if (!current_ctx()) return DFL_ERR_NO_DEVICE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    float* lse_z = static_cast<float*>(ws);
    float* lse_v = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + al256((size_t)N * G * 4));
    const float inv_T = 1.0f / T;
    const bool bf = dt == DFL_BF16;
    const RowMap vm{vlog, K, G + 1, sel};
    {
        ProfScope ps("row_lse", st);
        row_lse_kernel<false><<<(unsigned)(N * G), XT, 0, st>>>(RowMap{logits, 1, G, nullptr}, V, inv_T, lse_z);
        if (bf) row_lse_kernel<true><<<(unsigned)(N * (G + 1)), XT, 0, st>>>(vm, V, 1.f, lse_v);
        else row_lse_kernel<false><<<(unsigned)(N * (G + 1)), XT, 0, st>>>(vm, V, 1.f, lse_v);
    }
    dfl_status rc = last_launch();
    if (rc != DFL_OK) return rc;
    ProfScope ps("spec_accept", st);
    const uint32_t k0 = (uint32_t)(seed & 0xFFFFFFFFu), k1 = (uint32_t)(seed >> 32);
    if (bf)
        spec_accept_kernel<true><<<(unsigned)N, XT, 0, st>>>(logits, lse_z, inv_T, vm, lse_v, drafts, G, V, k0, k1,
                                                             accept_len, next_token);
    else
        spec_accept_kernel<false><<<(unsigned)N, XT, 0, st>>>(logits, lse_z, inv_T, vm, lse_v, drafts, G, V, k0, k1,
                                                              accept_len, next_token);
    return last_launch();
}
