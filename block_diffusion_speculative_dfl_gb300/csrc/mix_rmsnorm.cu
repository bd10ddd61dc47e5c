// Per-draft-layer mixture of target hidden states followed by RMSNorm.
//
// DFlare post, "Per-draft-layer mixing of different information": each draft
// layer l mixes the L target hidden states with softmax-normalised ratios
// and applies RMSNorm:  Xc_l[r] = g_l * x / sqrt(mean(x^2) + eps),
// x = sum_i softmax(mix_l)_i H_i[r].  All D draft layers come from one read of
// H, so the stack is streamed from HBM once per draft step.
//
// bf16 kernel: per row, TMA bulk copies stage the L slices H_i[r] in shared
// memory (two rows in flight when they fit), and the D normalised rows are
// staged in shared memory and written back with one bulk copy each.  The L -> D mixing is a tiny matrix product per
// group of positions, run on the tensor cores with mma.sync m16n8k16: A holds
// the mixing weights (rows 0..7 the bf16-rounded weight of draft layer
// 0..7, rows 8..15 the bf16 remainder, so hi + lo carries the fp32 weight
// to ~2^-16), B holds the bf16 hidden states (exact), accumulation is fp32.
// The products of bf16 values are exact in fp32, so the result equals the
// fp32 mixture up to accumulation rounding.
//
// fp32 kernel: plain FFMA mixture, one CTA per row.
#include "internal.h"

namespace dfl {

namespace {

constexpr int MIX_WARPS = 16;
constexpr int MIX_THREADS = MIX_WARPS * 32;
constexpr int MIX_MAXG = 20;            // 16-position groups per warp -> d <= 5120
constexpr int MIX_GCOLS = 4 * MIX_MAXG;  // TMEM columns of gains per thread
constexpr int MIX_TMEM_COLS = 512;       // 4 column blocks of MIX_GCOLS, rounded to a power of two

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                              uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// softmax(mix_logits[l]) [i] in fp32
__device__ float mix_weight(const float* logits, int L, int l, int i) {
    const float* z = logits + l * L;
    float m = z[0];
    for (int j = 1; j < L; ++j) m = fmaxf(m, z[j]);
    float s = 0.f;
    for (int j = 0; j < L; ++j) s += expf(z[j] - m);
    return expf(z[i] - m) / s;
}

__device__ __forceinline__ void split_bf16(float a, uint16_t& hi, uint16_t& lo) {
    const __nv_bfloat16 h = __float2bfloat16_rn(a);
    const __nv_bfloat16 l = __float2bfloat16_rn(a - __bfloat162float(h));
    hi = *reinterpret_cast<const uint16_t*>(&h);
    lo = *reinterpret_cast<const uint16_t*>(&l);
}

struct MixArgs {
    const __nv_bfloat16* H;
    int64_t layer_stride;
    int L;
    int64_t rows;
    int d;
    int D;
    const float* mix_logits;
    const float* gain;
    float eps;
    __nv_bfloat16* Xc;
    int64_t xc_stride;
};

// Shared-memory plan of the bf16 kernel: `nstage` input stages of L padded
// slabs, one output stage of D padded slabs, the zero row, the reduction
// array and the barriers.  Slabs are padded by 16 bytes so that the rows of
// one ldmatrix (8 layers) and the bf16x2 writes of one warp (8 draft layers)
// fall on distinct banks.
struct MixSmem {
    int slab, stage_bytes, out_bytes, nstage, total;
};

__host__ __device__ inline MixSmem mix_smem_plan(int L, int D, int d, int nstage) {
    MixSmem m;
    m.slab = d * 2 + 16;
    m.stage_bytes = ((L * m.slab + 127) / 128) * 128;
    m.out_bytes = ((D * m.slab + 127) / 128) * 128;
    m.nstage = nstage;
    m.total = 128 + nstage * m.stage_bytes + m.out_bytes + 128 + MIX_WARPS * 8 * 4 + 2 * 8 + 16;
    return m;
}

__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 :: "l"(dst), "r"(smem_u32(src)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__global__ void __launch_bounds__(MIX_THREADS, 1) mix_rmsnorm_bf16_kernel(const MixArgs a, const int nstage,
                                                                         const DevErr err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const MixSmem P = mix_smem_plan(a.L, a.D, a.d, nstage);
    uint8_t* in0 = smem;                                   // stage s at in0 + s * stage_bytes
    uint8_t* out = smem + nstage * P.stage_bytes;          // D padded output slabs
    uint8_t* zero_row = out + P.out_bytes;                 // 16 zero bytes
    float* red = reinterpret_cast<float*>(zero_row + 128); // [MIX_WARPS][8]
    uint64_t* full = reinterpret_cast<uint64_t*>(red + MIX_WARPS * 8);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(full + 2);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t tx_bytes = (uint32_t)a.L * (uint32_t)a.d * 2u;
    const uint32_t row_bytes = (uint32_t)a.d * 2u;

    if (tid == 0) {
        for (int q = 0; q < nstage; ++q) mbar_init(&full[q], 1);
        fence_barrier_init();
    }
    if (tid < 4) reinterpret_cast<uint32_t*>(zero_row)[tid] = 0u;
    // The RMSNorm gains do not change from row to row: each thread keeps the
    // 4 * MIX_MAXG gains of the positions it writes in its own TMEM lane
    // (quadrant warp % 4, column block warp / 4) instead of re-reading them
    // from L2 for every row.
    if (warp == 0) { tmem_alloc(tmem_holder, MIX_TMEM_COLS); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tgain = *tmem_holder + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)((warp >> 2) * MIX_GCOLS);

    uint32_t fills0 = 0u, fills1 = 0u;   // copies issued per stage (thread 0 only)
    auto issue = [&](int64_t row, int s) {
        if (s) ++fills1; else ++fills0;
        uint8_t* dst = in0 + s * P.stage_bytes;
        mbar_arrive_expect_tx(&full[s], tx_bytes);
        for (int i = 0; i < a.L; ++i)
            bulk_g2s(dst + i * P.slab, a.H + i * a.layer_stride + row * a.d, row_bytes, &full[s]);
    };
    if (tid == 0)
        for (int q = 0; q < nstage; ++q)
            if (blockIdx.x + (int64_t)q * gridDim.x < a.rows) issue(blockIdx.x + (int64_t)q * gridDim.x, q);

    // A fragments: mixing weights of draft layer l = lane/4 (hi rows 0..7, lo rows 8..15).
    uint32_t afrag[4];
    {
        const int l = lane >> 2;
        const int k0 = 2 * (lane & 3);
        uint16_t hi[4], lo[4];
        const int ks[4] = {k0, k0 + 1, k0 + 8, k0 + 9};
        #pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float w = (l < a.D && ks[j] < a.L) ? mix_weight(a.mix_logits, a.L, l, ks[j]) : 0.f;
            split_bf16(w, hi[j], lo[j]);
        }
        afrag[0] = (uint32_t)hi[0] | ((uint32_t)hi[1] << 16);   // row l,   k0..k0+1
        afrag[1] = (uint32_t)lo[0] | ((uint32_t)lo[1] << 16);   // row l+8, k0..k0+1
        afrag[2] = (uint32_t)hi[2] | ((uint32_t)hi[3] << 16);   // row l,   k0+8..k0+9
        afrag[3] = (uint32_t)lo[2] | ((uint32_t)lo[3] << 16);   // row l+8, k0+8..k0+9
    }

    // ldmatrix row owned by this thread: matrix lane/8 -> (k half, position half)
    const int my_k = ((lane >> 3) & 1) * 8 + (lane & 7);
    const int my_off = (lane >> 4) * 8;
    const int groups = a.d / 16;
    const int l_out = lane >> 2;
    const bool writes = l_out < a.D;
    const float* gain_l = a.gain + (int64_t)(writes ? l_out : 0) * a.d;
    uint8_t* out_l = out + l_out * P.slab;
    const uint32_t zero_addr = smem_u32(zero_row);
    {
        const int n = 2 * (lane & 3);
        #pragma unroll
        for (int c = 0; c < MIX_MAXG / 4; ++c) {
            uint32_t gv[16];
            #pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int g = warp + (4 * c + q) * MIX_WARPS;
                float2 g0 = make_float2(0.f, 0.f), g1 = make_float2(0.f, 0.f);
                if (writes && g < groups) {
                    g0 = __ldg(reinterpret_cast<const float2*>(gain_l + g * 16 + n));
                    g1 = __ldg(reinterpret_cast<const float2*>(gain_l + g * 16 + n + 8));
                }
                gv[4 * q + 0] = __float_as_uint(g0.x);
                gv[4 * q + 1] = __float_as_uint(g0.y);
                gv[4 * q + 2] = __float_as_uint(g1.x);
                gv[4 * q + 3] = __float_as_uint(g1.y);
            }
            tmem_st16(tgain + 16 * c, gv);
        }
        tmem_st_wait();
    }

    int it = 0;
    for (int64_t row = blockIdx.x; row < a.rows; row += gridDim.x, ++it) {
        const int s = (nstage == 2) ? (it & 1) : 0;
        const uint32_t par = (nstage == 2) ? ((it >> 1) & 1) : (it & 1);
        const bool ok = mbar_wait(&full[s], par, err);
        if (!__syncthreads_and(ok)) {
            // A bounded wait ran out (error recorded): let issued copies land, then leave.
            if (tid == 0) {
                if (fills0) mbar_wait(&full[0], (fills0 - 1) & 1, err);
                if (fills1) mbar_wait(&full[1], (fills1 - 1) & 1, err);
            }
            break;
        }
        const uint32_t stage_addr = smem_u32(in0) + (uint32_t)(s * P.stage_bytes);
        const uint32_t base = my_k < a.L ? stage_addr + (uint32_t)(my_k * P.slab) : zero_addr;
        const uint32_t step = my_k < a.L ? 2u : 0u;
        float v[MIX_MAXG][4];
        float ss = 0.f;
        #pragma unroll
        for (int j = 0; j < MIX_MAXG; ++j) {
            const int g = warp + j * MIX_WARPS;
            v[j][0] = v[j][1] = v[j][2] = v[j][3] = 0.f;
            if (g < groups) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4_trans(base + step * (uint32_t)(g * 16 + my_off), b0, b1, b2, b3);
                float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
                mma_16816(c0, afrag, b0, b1);
                mma_16816(c1, afrag, b2, b3);
                v[j][0] = c0[0] + c0[2];
                v[j][1] = c0[1] + c0[3];
                v[j][2] = c1[0] + c1[2];
                v[j][3] = c1[1] + c1[3];
                ss += v[j][0] * v[j][0] + v[j][1] * v[j][1] + v[j][2] * v[j][2] + v[j][3] * v[j][3];
            }
        }
        ss += __shfl_xor_sync(0xFFFFFFFFu, ss, 1);
        ss += __shfl_xor_sync(0xFFFFFFFFu, ss, 2);
        if ((lane & 3) == 0) red[warp * 8 + l_out] = ss;
        if (tid == 0) bulk_wait_read0();   // previous row's output stage has been read out
        __syncthreads();                    // stage s consumed; partial sums visible; output stage free
        if (tid == 0 && row + (int64_t)nstage * gridDim.x < a.rows) issue(row + (int64_t)nstage * gridDim.x, s);
        float tot = 0.f;
        #pragma unroll
        for (int w = 0; w < MIX_WARPS; ++w) tot += red[w * 8 + l_out];
        const float rs = rsqrtf(tot / (float)a.d + a.eps);
        {
            const int n = 2 * (lane & 3);
            #pragma unroll
            for (int c = 0; c < MIX_MAXG / 4; ++c) {
                if (warp + 4 * c * MIX_WARPS >= groups) break;   // warp-uniform
                float gv[16];
                tmem_ld16(tgain + 16 * c, gv);
                if (writes) {
                    #pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int j = 4 * c + q;
                        const int g = warp + j * MIX_WARPS;
                        if (g < groups) {
                            const int p = g * 16 + n;
                            *reinterpret_cast<uint32_t*>(out_l + p * 2) =
                                pack_bf16(v[j][0] * rs * gv[4 * q], v[j][1] * rs * gv[4 * q + 1]);
                            *reinterpret_cast<uint32_t*>(out_l + (p + 8) * 2) =
                                pack_bf16(v[j][2] * rs * gv[4 * q + 2], v[j][3] * rs * gv[4 * q + 3]);
                        }
                    }
                }
            }
        }
        fence_proxy_async_smem();   // make the output stage visible to the bulk copies
        __syncthreads();
        if (tid == 0) {
            for (int l = 0; l < a.D; ++l)
                bulk_s2g(a.Xc + l * a.xc_stride + row * a.d, out + l * P.slab, row_bytes);
            bulk_commit();
        }
    }
    if (tid == 0) bulk_wait0();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(*tmem_holder, MIX_TMEM_COLS);
    }
}

// fp32: one CTA per row; mixtures kept in shared memory until the row's norm is known.
__global__ void mix_rmsnorm_f32_kernel(const float* H, int64_t layer_stride, int L, int64_t rows, int d, int D,
                                       const float* mix_logits, const float* gain, float eps, float* Xc,
                                       int64_t xc_stride) {
    extern __shared__ float fsm[];
    float* w = fsm;              // [D][L]
    float* red = w + D * L;      // [D][32]
    float* buf = red + D * 32;   // [D][d]
    const int tid = threadIdx.x;
    if (tid < D) {
        for (int i = 0; i < L; ++i) w[tid * L + i] = mix_weight(mix_logits, L, tid, i);
    }
    __syncthreads();
    const int64_t row = blockIdx.x;
    float ss[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int e = tid; e < d; e += blockDim.x) {
        float h[32];
        for (int i = 0; i < L; ++i) h[i] = H[i * layer_stride + row * d + e];
        for (int l = 0; l < D; ++l) {
            float x = 0.f;
            for (int i = 0; i < L; ++i) x = fmaf(w[l * L + i], h[i], x);
            buf[l * d + e] = x;
            ss[l] += x * x;
        }
    }
    const int warp = tid >> 5, lane = tid & 31;
    for (int l = 0; l < D; ++l) {
        const float s = warp_sum(ss[l]);
        if (lane == 0) red[l * 32 + warp] = s;
    }
    __syncthreads();
    for (int l = 0; l < D; ++l) {
        float tot = 0.f;
        for (int j = 0; j < (int)(blockDim.x >> 5); ++j) tot += red[l * 32 + j];
        const float rs = rsqrtf(tot / (float)d + eps);
        for (int e = tid; e < d; e += blockDim.x)
            Xc[l * xc_stride + row * d + e] = buf[l * d + e] * rs * gain[(int64_t)l * d + e];
    }
}

}  // namespace

}  // namespace dfl

using namespace dfl;

extern "C" dfl_status dfl_layer_mix_rmsnorm(const void* H, int64_t layer_stride, int32_t L, int64_t rows,
                                            int32_t d, dfl_dtype dt, int32_t D, const float* mix_logits,
                                            const float* gain, float eps, void* Xc, int64_t xc_layer_stride,
                                            dfl_stream stream) {
    if (!H || !mix_logits || !gain || !Xc) return DFL_ERR_INVALID_ARG;
    if (L < 1 || L > 16 || D < 1 || D > 8 || rows <= 0 || d <= 0) return DFL_ERR_INVALID_ARG;
    if (layer_stride < rows * d && L > 1) return DFL_ERR_INVALID_ARG;
    if (xc_layer_stride < rows * d && D > 1) return DFL_ERR_INVALID_ARG;
    if (dt != DFL_F32 && dt != DFL_BF16) return DFL_ERR_INVALID_ARG;
    if (!aligned16(H) || !aligned16(Xc) || !aligned16(gain) || d % 8 != 0 || layer_stride % 8 != 0 ||
        xc_layer_stride % 8 != 0)
        return DFL_ERR_MISALIGNED;
    DeviceCtx* ctx = current_ctx();
    if (!ctx) return DFL_ERR_NO_DEVICE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dt == DFL_BF16) {
        if (d % 16 != 0 || d > 16 * MIX_WARPS * MIX_MAXG) return DFL_ERR_UNSUPPORTED_SHAPE;
        int nstage = 2;
        if (mix_smem_plan(L, D, d, 2).total > 227 * 1024) nstage = 1;
        const int smem = mix_smem_plan(L, D, d, nstage).total;
        if (smem > 227 * 1024) return DFL_ERR_UNSUPPORTED_SHAPE;
        if (!ctx->mix_attr_set) {
            if (cudaFuncSetAttribute(mix_rmsnorm_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     227 * 1024) != cudaSuccess)
                return DFL_ERR_CUDA;
            ctx->mix_attr_set = true;
        }
        MixArgs a{static_cast<const __nv_bfloat16*>(H), layer_stride, L, rows, d, D, mix_logits, gain, eps,
                  static_cast<__nv_bfloat16*>(Xc), xc_layer_stride};
        const int64_t grid = rows < ctx->sm_count ? rows : ctx->sm_count;
        ProfScope ps("mix_rmsnorm_bf16", st);
        mix_rmsnorm_bf16_kernel<<<(unsigned)grid, MIX_THREADS, smem, st>>>(a, nstage, dev_err(ctx));
        return last_launch();
    }
    const size_t smem = (size_t)(D * L + D * 32 + (size_t)D * d) * sizeof(float);
    if (smem > 200 * 1024) return DFL_ERR_UNSUPPORTED_SHAPE;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(mix_rmsnorm_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
        return DFL_ERR_CUDA;
    if (rows > 0x7FFFFFFF) return DFL_ERR_UNSUPPORTED_SHAPE;
    ProfScope ps("mix_rmsnorm_f32", st);
    mix_rmsnorm_f32_kernel<<<(unsigned)rows, 256, smem, st>>>(static_cast<const float*>(H), layer_stride, L, rows,
                                                             d, D, mix_logits, gain, eps, static_cast<float*>(Xc),
                                                             xc_layer_stride);
    return last_launch();
}
