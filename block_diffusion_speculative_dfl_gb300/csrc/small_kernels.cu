// Small kernels of the draft step: rotary table, row RMSNorm, greedy
// acceptance, argmax combine, K-draft sampling, and the fp32 CUDA-core path
// (GEMM, in-place rotary, attention, per-tile partials).
#include "internal.h"
#include "philox.cuh"
#include "small_kernels.h"

namespace dfl {

// ------------------------------------------------------------ rotary table

__global__ void rope_table_kernel(float* table, int P, int hd, double theta) {
    grid_dep_begin();
    const int half = hd / 2;
    const int64_t n = (int64_t)P * half;
    for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < n; t += (int64_t)gridDim.x * blockDim.x) {
        const int p = (int)(t / half), i = (int)(t % half);
        const double inv_freq = pow(theta, -2.0 * (double)i / (double)hd);
        const double ang = (double)p * inv_freq;
        table[2 * t] = (float)cos(ang);
        table[2 * t + 1] = (float)sin(ang);
    }
}

dfl_status rope_table(float* table, int P, int hd, double theta, cudaStream_t st) {
    const int64_t n = (int64_t)P * (hd / 2);
    const int grid = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
    ProfScope ps("rope_table", st);
    return launch_pdl(rope_table_kernel, grid, 256, 0, st, table, P, hd, theta);
}

// ------------------------------------------------------------ row RMSNorm

// out[m] = RMSNorm(in[src_row(m)]) * gain, src_row(m) = (m / per) * stride + off + m % per.
// One 128-thread CTA per row; the row stays in registers between the sum of
// squares and the scaled store (d <= 128 * 4 * RN_MAXV).  OutT = bf16 or float.
constexpr int RN_THREADS = 128;
constexpr int RN_MAXV = 12;   // float4 per thread -> d <= 6144

template <typename OutT>
__global__ void __launch_bounds__(RN_THREADS) rmsnorm_rows_kernel(const float* in, int d, int64_t M, int per,
                                                                  int stride, int off, const float* gain, float eps,
                                                                  OutT* out, float* copy) {
    grid_dep_begin();
    const int64_t m = blockIdx.x;
    const int tid = threadIdx.x;
    const int64_t src = (m / per) * stride + off + m % per;
    const float4* x = reinterpret_cast<const float4*>(in + src * d);
    const int nv = d / 4;
    float4 v[RN_MAXV];
    float ss = 0.f;
    #pragma unroll
    for (int j = 0; j < RN_MAXV; ++j) {
        const int e = tid + j * RN_THREADS;
        v[j] = e < nv ? x[e] : make_float4(0.f, 0.f, 0.f, 0.f);
        ss += v[j].x * v[j].x + v[j].y * v[j].y + v[j].z * v[j].z + v[j].w * v[j].w;
    }
    if (copy) {   // the input row, unchanged, to the same row of `copy`
        float4* c4 = reinterpret_cast<float4*>(copy + src * d);
        #pragma unroll
        for (int j = 0; j < RN_MAXV; ++j)
            if (tid + j * RN_THREADS < nv) c4[tid + j * RN_THREADS] = v[j];
    }
    __shared__ float red[RN_THREADS / 32];
    ss = warp_sum(ss);
    if ((tid & 31) == 0) red[tid >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
    #pragma unroll
    for (int w = 0; w < RN_THREADS / 32; ++w) tot += red[w];
    const float rs = rsqrtf(tot / (float)d + eps);
    OutT* o = out + m * d;
    const float4* g4 = reinterpret_cast<const float4*>(gain);
    #pragma unroll
    for (int j = 0; j < RN_MAXV; ++j) {
        const int e = tid + j * RN_THREADS;
        if (e < nv) {
            const float4 g = __ldg(g4 + e);
            const float y0 = v[j].x * rs * g.x, y1 = v[j].y * rs * g.y, y2 = v[j].z * rs * g.z,
                        y3 = v[j].w * rs * g.w;
            if constexpr (sizeof(OutT) == 2) {
                uint2 u;
                u.x = pack_bf16(y0, y1);
                u.y = pack_bf16(y2, y3);
                *reinterpret_cast<uint2*>(o + 4 * e) = u;
            } else {
                *reinterpret_cast<float4*>(o + 4 * e) = make_float4(y0, y1, y2, y3);
            }
        }
    }
}

dfl_status rmsnorm_rows(const float* in, int d, int64_t M, int per, int stride, int off, const float* gain,
                        float eps, void* out, bool bf16, cudaStream_t st, float* copy) {
    if (d > RN_THREADS * 4 * RN_MAXV || d % 4 != 0) return DFL_ERR_UNSUPPORTED_SHAPE;
    if (M > 0x7FFFFFFF) return DFL_ERR_UNSUPPORTED_SHAPE;
    ProfScope ps("rmsnorm_rows", st);
    if (bf16)
        return launch_pdl(rmsnorm_rows_kernel<__nv_bfloat16>, (unsigned)M, RN_THREADS, 0, st, in, d, M, per, stride,
                          off, gain, eps, static_cast<__nv_bfloat16*>(out), copy);
    return launch_pdl(rmsnorm_rows_kernel<float>, (unsigned)M, RN_THREADS, 0, st, in, d, M, per, stride, off, gain,
                      eps, static_cast<float*>(out), copy);
}

// --------------------------------------------------------- greedy accept

// DFlare post, "Generating candidates in parallel, the target decides
// acceptance": accept the prefix up to the first mismatch, then the target's
// token.  One warp per sequence.
__global__ void greedy_accept_kernel(const int32_t* draft, const int32_t* target, int N, int n,
                                     int32_t* accept_len, int32_t* bonus) {
    grid_dep_begin();
    const int s = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (s >= N) return;
    const int32_t* d = draft + (int64_t)s * n;
    const int32_t* t = target + (int64_t)s * (n + 1);
    int a = n;
    for (int j0 = 0; j0 < n; j0 += 32) {
        const int j = j0 + lane;
        const unsigned mism = __ballot_sync(0xFFFFFFFFu, j < n && d[j] != t[j]);
        if (mism) { a = j0 + __ffs(mism) - 1; break; }
    }
    if (lane == 0) {
        accept_len[s] = a;
        bonus[s] = t[a];
    }
}

dfl_status greedy_accept(const int32_t* draft, const int32_t* target, int N, int n, int32_t* accept_len,
                         int32_t* bonus, cudaStream_t st) {
    ProfScope ps("greedy_accept", st);
    return launch_pdl(greedy_accept_kernel, (N + 7) / 8, 256, 0, st, draft, target, N, n, accept_len, bonus);
}

// ------------------------------------------------------ context-cache plan

// Row plan of a cached draft step (SpecDiff-2 notes, "Future work and
// limitations": KV-cache support for the drafter).  Sequence n with c0 cached
// positions and m new rows: new row i < m sits at position c0 + i and goes to
// cache row n*C + c0 + i; rows i >= m are dropped (-1); the block sits at
// c0 + m .. c0 + m + B - 1 and attends to c0 + m cached positions.  Lengths
// out of range record DFL_ERR_INVALID_ARG and append nothing.  One CTA per
// sequence.
__global__ void cache_plan_kernel(int N, int R, int B, int C, int32_t* ctx_len, const int32_t* n_new, int advance,
                                  int32_t* pos_ctx, int32_t* dst_ctx, int32_t* pos_blk, int32_t* len_new,
                                  DevErr err) {
    grid_dep_begin();
    const int n = blockIdx.x;
    __shared__ int s_c0, s_m;
    if (threadIdx.x == 0) {
        int c0 = ctx_len[n], m = n_new[n];
        const bool ok = c0 >= 0 && c0 <= C && m >= 0 && m <= R && m <= C - c0;
        if (!ok) {
            record_error(err, DFL_ERR_INVALID_ARG);
            c0 = min(max(c0, 0), C);
            m = 0;
        }
        s_c0 = c0;
        s_m = m;
        len_new[n] = c0 + m;
        if (advance && ok) ctx_len[n] = c0 + m;
    }
    __syncthreads();
    const int c0 = s_c0, m = s_m;
    for (int i = threadIdx.x; i < R; i += blockDim.x) {
        pos_ctx[(int64_t)n * R + i] = i < m ? c0 + i : 0;
        dst_ctx[(int64_t)n * R + i] = i < m ? n * C + c0 + i : -1;
    }
    for (int b = threadIdx.x; b < B; b += blockDim.x) pos_blk[(int64_t)n * B + b] = c0 + m + b;
}

dfl_status cache_plan(int N, int R, int B, int C, int32_t* ctx_len, const int32_t* n_new, int advance,
                      int32_t* pos_ctx, int32_t* dst_ctx, int32_t* pos_blk, int32_t* len_new, DevErr err,
                      cudaStream_t st) {
    ProfScope ps("cache_plan", st);
    return launch_pdl(cache_plan_kernel, N, 128, 0, st, N, R, B, C, ctx_len, n_new, advance, pos_ctx, dst_ctx,
                      pos_blk, len_new, err);
}

// --------------------------------------------------------- argmax combine

// argmax over per-tile partials; equal maxima resolve to the lower column
// (tiles are disjoint and ordered, and each partial already holds its tile's
// lowest maximal column).  One warp per row.
__global__ void argmax_combine_kernel(const float* pmax, const int* pidx, int64_t M, int tiles, int32_t* out) {
    grid_dep_begin();
    const int64_t m = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (m >= M) return;
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
    for (int t = lane; t < tiles; t += 32) {
        const float v = pmax[m * tiles + t];
        const int i = pidx[m * tiles + t];
        if (v > bv || (v == bv && i < bi)) { bv = v; bi = i; }
    }
    #pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float v = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
        const int i = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
        if (v > bv || (v == bv && i < bi)) { bv = v; bi = i; }
    }
    if (lane == 0) out[m] = bi;
}

dfl_status argmax_combine(const float* pmax, const int* pidx, int64_t M, int tiles, int32_t* out,
                          cudaStream_t st) {
    ProfScope ps("argmax_combine", st);
    return launch_pdl(argmax_combine_kernel, (unsigned)((M + 7) / 8), 256, 0, st, pmax, pidx, M, tiles, out);
}

// ------------------------------------------------------------- sampling

// SpecDiff-2 notes, "Parallel drafting with diffusion LMs" / "Self-Selection
// Acceptance": K independent draws per window row from softmax(z / T), by
// inverting the CDF at u = ((x0 >> 8) + 1/2) 2^-24.
// Inputs per row: fp32 logits and per-tile partials (tile max m_t, fp64 sum
// s_t of expf((z - m_t) * inv_T) in column order).  Tile weights
// W_t = s_t * exp((m_t - M) / T) are prefix-summed in fp64; the draw walks
// its tile in the same column order with the same expf terms, so the
// within-tile search is consistent with W_t.  One warp per row.
__global__ void sample_kernel(const float* logits, int64_t ld, const float* pmax, const double* psum, int64_t M,
                              int per, int tiles, int bn, int V, int K, float inv_T, uint32_t key0, uint32_t key1,
                              int32_t* samples) {
    grid_dep_begin();
    extern __shared__ double pref[];   // [warps][tiles + 1]
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t m = blockIdx.x * (int64_t)(blockDim.x >> 5) + w;
    if (m >= M) return;
    double* P = pref + (int64_t)w * (tiles + 1);
    const float* pm = pmax + m * tiles;
    const double* ps = psum + m * tiles;
    float Mx = -INFINITY;
    for (int t = lane; t < tiles; t += 32) Mx = fmaxf(Mx, pm[t]);
    Mx = warp_max(Mx);
    // prefix sums: lane owns a contiguous chunk of tiles; each tile weight (an
    // fp64 exp, slow on this part) is computed once, kept in P[t] and turned
    // into the prefix in place
    const int chunk = (tiles + 31) / 32;
    const int t0 = lane * chunk, t1 = min(tiles, t0 + chunk);
    double loc = 0.0;
    for (int t = t0; t < t1; ++t) {
        const double wt = ps[t] * exp((double)(pm[t] - Mx) * (double)inv_T);
        P[t] = wt;
        loc += wt;
    }
    double excl = loc;
    #pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xFFFFFFFFu, excl, o);
        if (lane >= o) excl += y;
    }
    excl -= loc;
    double run = excl;
    for (int t = t0; t < t1; ++t) {
        const double wt = P[t];
        P[t] = run;
        run += wt;
    }
    if (lane == 31) P[tiles] = run;
    __syncwarp();
    const double S = P[tiles];
    const int n_seq = (int)(m / per), j = (int)(m % per);
    for (int k = lane; k < K; k += 32) {
        const double u = philox_uniform24((uint32_t)n_seq, (uint32_t)j, (uint32_t)k, 0u, key0, key1);
        const double target = u * S;
        // first tile whose inclusive prefix exceeds the target
        int lo = 0, hi = tiles - 1;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (P[mid + 1] > target) hi = mid; else lo = mid + 1;
        }
        const int t = lo;
        const double f = exp((double)(pm[t] - Mx) * (double)inv_T);
        const float mt = pm[t];
        const float* z = logits + m * ld + (int64_t)t * bn;
        const int vmax = min(bn, V - t * bn);
        double cum = 0.0;
        int pick = t * bn + vmax - 1;
        for (int v = 0; v < vmax; ++v) {
            cum += (double)expf((z[v] - mt) * inv_T);
            if (P[t] + f * cum > target) { pick = t * bn + v; break; }
        }
        samples[((int64_t)n_seq * K + k) * per + j] = pick;
    }
}

dfl_status sample_rows(const float* logits, int64_t ld, const float* pmax, const double* psum, int64_t M, int per,
                       int tiles, int bn, int V, int K, float T, uint64_t seed, int32_t* samples, cudaStream_t st) {
    const int warps = 4;
    const size_t smem = (size_t)warps * (tiles + 1) * sizeof(double);
    if (smem > 200 * 1024) return DFL_ERR_UNSUPPORTED_SHAPE;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return DFL_ERR_CUDA;
    ProfScope ps("sample_inverse_cdf", st);
    return launch_pdl(sample_kernel, (unsigned)((M + warps - 1) / warps), warps * 32, smem, st, logits, ld, pmax,
                      psum, M, per, tiles, bn, V, K, 1.0f / T, (uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32),
                      samples);
}

// Per-tile partials from materialised fp32 logits (the fp32 path): max,
// lowest argmax and sum of expf((z - max) * inv_T) in column order (groups
// of four in fp32, groups in fp64), exactly as the tensor-core GEMM epilogue
// forms them.  Thread per (row, tile).
__global__ void tile_partials_kernel(const float* logits, int64_t ld, int64_t M, int V, int bn, int tiles,
                                     float inv_T, float* pmax, int* pidx, double* psum) {
    grid_dep_begin();
    const int64_t id = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (id >= M * tiles) return;
    const int64_t m = id / tiles;
    const int t = (int)(id % tiles);
    const float* z = logits + m * ld + (int64_t)t * bn;
    const int vmax = min(bn, V - t * bn);
    float best = -INFINITY;
    int bi = t * bn;
    for (int v = 0; v < vmax; ++v)
        if (z[v] > best) { best = z[v]; bi = t * bn + v; }
    double s = 0.0;
    for (int v = 0; v < vmax; v += 4) {   // groups of four added pairwise in fp32, as the GEMM epilogue does
        float e[4];
        for (int q = 0; q < 4; ++q) e[q] = v + q < vmax ? expf((z[v + q] - best) * inv_T) : 0.f;
        s += (double)((e[0] + e[1]) + (e[2] + e[3]));
    }
    pmax[id] = best;
    pidx[id] = bi;
    if (psum) psum[id] = s;
}

dfl_status tile_partials(const float* logits, int64_t ld, int64_t M, int V, int bn, int tiles, float inv_T,
                         float* pmax, int* pidx, double* psum, cudaStream_t st) {
    const int64_t n = M * tiles;
    ProfScope ps("tile_partials", st);
    return launch_pdl(tile_partials_kernel, (unsigned)((n + 127) / 128), 128, 0, st, logits, ld, M, V, bn, tiles,
                      inv_T, pmax, pidx, psum);
}

// ------------------------------------------------------------ fp32 GEMM

// C[M][N] (=|+=) A[M][K] * B[N][K]^T on CUDA cores, 64x64 tiles.
__global__ void gemm_f32_kernel(const float* A, int64_t lda, const float* B, int64_t ldb, float* C, int M, int N,
                                int K, int ldc, int acc) {
    grid_dep_begin();
    __shared__ float As[16][64 + 1];
    __shared__ float Bs[16][64 + 1];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
    float r[4][4] = {};
    for (int k0 = 0; k0 < K; k0 += 16) {
        for (int i = threadIdx.x; i < 64 * 16; i += 256) {
            const int row = i / 16, kk = i % 16;
            As[kk][row] = (m0 + row < M && k0 + kk < K) ? A[(int64_t)(m0 + row) * lda + k0 + kk] : 0.f;
            Bs[kk][row] = (n0 + row < N && k0 + kk < K) ? B[(int64_t)(n0 + row) * ldb + k0 + kk] : 0.f;
        }
        __syncthreads();
        #pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            float a[4], b[4];
            #pragma unroll
            for (int i = 0; i < 4; ++i) { a[i] = As[kk][ty * 4 + i]; b[i] = Bs[kk][tx + 16 * i]; }
            #pragma unroll
            for (int i = 0; i < 4; ++i)
                #pragma unroll
                for (int j = 0; j < 4; ++j) r[i][j] = fmaf(a[i], b[j], r[i][j]);
        }
        __syncthreads();
    }
    #pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = m0 + ty * 4 + i;
        if (row >= M) continue;
        #pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int col = n0 + tx + 16 * j;
            if (col >= N) continue;
            float* c = C + (int64_t)row * ldc + col;
            *c = acc ? *c + r[i][j] : r[i][j];
        }
    }
}

dfl_status gemm_f32_ld(const float* A, int64_t lda, const float* B, int64_t ldb, float* C, int M, int N, int K,
                       int ldc, int accumulate, cudaStream_t st) {
    dim3 grid((N + 63) / 64, (M + 63) / 64);
    ProfScope ps("gemm_f32", st);
    return launch_pdl(gemm_f32_kernel, grid, 256, 0, st, A, lda, B, ldb, C, M, N, K, ldc, accumulate);
}

dfl_status gemm_f32(const float* A, const float* B, float* C, int M, int N, int K, int ldc, int accumulate,
                    cudaStream_t st) {
    return gemm_f32_ld(A, K, B, K, C, M, N, K, ldc, accumulate, st);
}

// In-place rotate-half rotary on x[rows][heads][hd] (fp32); row r at position
// pos_off + r % per.
__global__ void rope_inplace_f32_kernel(float* x, int64_t rows, int heads, int hd, int per, int pos_off,
                                        const float* rope) {
    grid_dep_begin();
    const int half = hd / 2;
    const int64_t n = rows * heads * half;
    for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < n; t += (int64_t)gridDim.x * blockDim.x) {
        const int i = (int)(t % half);
        const int64_t rh = t / half;
        const int64_t r = rh / heads;
        const int p = pos_off + (int)(r % per);
        const float c = rope[((int64_t)p * half + i) * 2], s = rope[((int64_t)p * half + i) * 2 + 1];
        float* v = x + rh * hd;
        const float a = v[i], b = v[i + half];
        v[i] = a * c - b * s;
        v[i + half] = b * c + a * s;
    }
}

dfl_status rope_inplace_f32(float* x, int64_t rows, int heads, int hd, int per, int pos_off, const float* rope,
                            cudaStream_t st) {
    const int64_t n = rows * heads * (hd / 2);
    const int grid = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
    ProfScope ps("rope_f32", st);
    return launch_pdl(rope_inplace_f32_kernel, grid, 256, 0, st, x, rows, heads, hd, per, pos_off, rope);
}

// h[i] = silu(gate[i]) * up[i] (fp32 path of the feed-forward block).
__global__ void swiglu_f32_kernel(const float* gate, const float* up, float* h, int64_t n) {
    grid_dep_begin();
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const float g = gate[i];
        h[i] = g / (1.f + expf(-g)) * up[i];
    }
}

dfl_status swiglu_f32(const float* gate, const float* up, float* h, int64_t n, cudaStream_t st) {
    ProfScope ps("swiglu_f32", st);
    const int64_t blocks = (n + 255) / 256;
    return launch_pdl(swiglu_f32_kernel, (unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, st, gate, up, h, n);
}

// fp32 block attention: one CTA per (sequence, query head), one warp per
// query row at a time, online softmax over [context ; block] keys, no mask.
__global__ void attn_f32_kernel(const float* Q, const float* Kc, const float* Vc, const float* Kb, const float* Vb,
                                int N, int C, int B, int Hq, int Hkv, int hd, float* O) {
    grid_dep_begin();
    const int n = blockIdx.x / Hq, h = blockIdx.x % Hq;
    const int g = h / (Hq / Hkv);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float scale = rsqrtf((float)hd);
    for (int b = warp; b < B; b += blockDim.x >> 5) {
        const float* q = Q + ((int64_t)(n * B + b) * Hq + h) * hd;
        float qv[4], o[4] = {0.f, 0.f, 0.f, 0.f};
        for (int j = 0; j < 4; ++j) qv[j] = (lane + 32 * j < hd) ? q[lane + 32 * j] : 0.f;
        float mx = -INFINITY, l = 0.f;
        for (int key = 0; key < C + B; ++key) {
            const float* k = key < C ? Kc + ((int64_t)(n * C + key) * Hkv + g) * hd
                                     : Kb + ((int64_t)(n * B + key - C) * Hkv + g) * hd;
            const float* v = key < C ? Vc + ((int64_t)(n * C + key) * Hkv + g) * hd
                                     : Vb + ((int64_t)(n * B + key - C) * Hkv + g) * hd;
            float s = 0.f;
            for (int j = 0; j < 4; ++j) if (lane + 32 * j < hd) s += qv[j] * k[lane + 32 * j];
            s = warp_sum(s) * scale;
            const float mn = fmaxf(mx, s);
            const float al = expf(mx - mn), p = expf(s - mn);
            l = l * al + p;
            for (int j = 0; j < 4; ++j) if (lane + 32 * j < hd) o[j] = o[j] * al + p * v[lane + 32 * j];
            mx = mn;
        }
        float* out = O + ((int64_t)(n * B + b) * Hq + h) * hd;
        for (int j = 0; j < 4; ++j) if (lane + 32 * j < hd) out[lane + 32 * j] = o[j] / l;
    }
}

dfl_status attn_f32(const float* Q, const float* Kc, const float* Vc, const float* Kb, const float* Vb, int N, int C,
                    int B, int Hq, int Hkv, int hd, float* O, cudaStream_t st) {
    ProfScope ps("attn_f32", st);
    return launch_pdl(attn_f32_kernel, N * Hq, 128, 0, st, Q, Kc, Vc, Kb, Vb, N, C, B, Hq, Hkv, hd, O);
}

// ------------------------------------------------------- wait self-test

__global__ void selftest_wait_kernel(int* status, uint64_t limit_ns) {
    grid_dep_begin();
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        *status = 0;
        mbar_init(&bar, 1);
        fence_barrier_init();
        DevErr e{status, limit_ns};
        mbar_wait(&bar, 0, e);   // nothing arrives: runs out, records DFL_ERR_TIMEOUT
    }
}

dfl_status selftest_wait(int* status, uint64_t limit_ns, cudaStream_t st) {
    ProfScope ps("selftest_wait", st);
    return launch_pdl(selftest_wait_kernel, 1, 32, 0, st, status, limit_ns);
}

// ----------------------------------------------------- Philox known answers

// out[i] = Philox4x32-10(counter in[i][0..3], key in[i][4..5]): the device
// generator's four output words, for checks against published vectors.
__global__ void philox_block_kernel(const uint32_t* in, int n, uint32_t* out) {
    grid_dep_begin();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const uint32_t* c = in + (int64_t)i * 6;
    const uint4 x = philox4x32_10(c[0], c[1], c[2], c[3], c[4], c[5]);
    uint32_t* o = out + (int64_t)i * 4;
    o[0] = x.x; o[1] = x.y; o[2] = x.z; o[3] = x.w;
}

dfl_status philox_block(const uint32_t* in, int n, uint32_t* out, cudaStream_t st) {
    ProfScope ps("philox_block", st);
    return launch_pdl(philox_block_kernel, (n + 127) / 128, 128, 0, st, in, n, out);
}

}  // namespace dfl
