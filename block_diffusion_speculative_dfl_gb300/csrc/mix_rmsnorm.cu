// Per-draft-layer mixture of target hidden states followed by RMSNorm.
//
// DFlare post, "Per-draft-layer mixing of different information": each draft
// layer l mixes the L target hidden states with softmax-normalised ratios
// and applies RMSNorm:  Xc_l[r] = g_l * x / sqrt(mean(x^2) + eps),
// x = sum_i softmax(mix_l)_i H_i[r].  All D draft layers come from one read of
// H, so the stack is streamed from HBM once per draft step.
//
// bf16 kernel: per row, TMA bulk copies stage the L slices H_i[r] in shared
// memory (two rows in flight).  The L -> D mixing is a tiny matrix product per
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

__global__ void __launch_bounds__(MIX_THREADS, 1) mix_rmsnorm_bf16_kernel(const MixArgs a, const DevErr err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const int slab = a.d * 2 + 16;                       // padded: rows of 8 layers hit distinct banks
    const int stage_bytes = ((a.L * slab + 127) / 128) * 128;
    uint8_t* stage[2] = {smem, smem + stage_bytes};
    uint8_t* zero_row = smem + 2 * stage_bytes;          // 16 zero bytes
    float* red = reinterpret_cast<float*>(zero_row + 128);   // [MIX_WARPS][8]
    uint64_t* full = reinterpret_cast<uint64_t*>(red + MIX_WARPS * 8);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t tx_bytes = (uint32_t)a.L * (uint32_t)a.d * 2u;

    if (tid == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        fence_barrier_init();
    }
    if (tid < 4) reinterpret_cast<uint32_t*>(zero_row)[tid] = 0u;
    __syncthreads();

    uint32_t fills[2] = {0u, 0u};   // copies issued per stage (thread 0 only)
    auto issue = [&](int64_t row, int s) {
        ++fills[s];
        mbar_arrive_expect_tx(&full[s], tx_bytes);
        for (int i = 0; i < a.L; ++i)
            bulk_g2s(stage[s] + i * slab, a.H + i * a.layer_stride + row * a.d, (uint32_t)a.d * 2u, &full[s]);
    };
    if (tid == 0) {
        if (blockIdx.x < a.rows) issue(blockIdx.x, 0);
        if (blockIdx.x + gridDim.x < a.rows) issue(blockIdx.x + gridDim.x, 1);
    }

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
    const float* gain_l = a.gain + (int64_t)(l_out < a.D ? l_out : 0) * a.d;

    int it = 0;
    for (int64_t row = blockIdx.x; row < a.rows; row += gridDim.x, ++it) {
        const int s = it & 1;
        const uint32_t par = (it >> 1) & 1;
        const bool ok = mbar_wait(&full[s], par, err);
        if (!__syncthreads_and(ok)) {
            // A bounded wait ran out (error recorded): let issued copies land, then leave.
            if (tid == 0)
                for (int q = 0; q < 2; ++q)
                    if (fills[q]) mbar_wait(&full[q], (fills[q] - 1) & 1, err);
            return;
        }

        const uint32_t base = smem_u32(my_k < a.L ? stage[s] + my_k * slab : zero_row);
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
        __syncthreads();   // stage s fully read; partial sums visible
        if (tid == 0 && row + 2 * (int64_t)gridDim.x < a.rows) issue(row + 2 * (int64_t)gridDim.x, s);
        float tot = 0.f;
        #pragma unroll
        for (int w = 0; w < MIX_WARPS; ++w) tot += red[w * 8 + l_out];
        const float rs = rsqrtf(tot / (float)a.d + a.eps);
        if (l_out < a.D) {
            __nv_bfloat16* out = a.Xc + l_out * a.xc_stride + row * a.d;
            const int n = 2 * (lane & 3);
            #pragma unroll
            for (int j = 0; j < MIX_MAXG; ++j) {
                const int g = warp + j * MIX_WARPS;
                if (g < groups) {
                    const int p = g * 16 + n;
                    const float2 g0 = *reinterpret_cast<const float2*>(gain_l + p);
                    const float2 g1 = *reinterpret_cast<const float2*>(gain_l + p + 8);
                    *reinterpret_cast<uint32_t*>(out + p) = pack_bf16(v[j][0] * rs * g0.x, v[j][1] * rs * g0.y);
                    *reinterpret_cast<uint32_t*>(out + p + 8) = pack_bf16(v[j][2] * rs * g1.x, v[j][3] * rs * g1.y);
                }
            }
        }
        __syncthreads();   // red[] reads done before the next row writes it
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

int mix_bf16_smem_bytes(int L, int d) {
    const int slab = d * 2 + 16;
    const int stage_bytes = ((L * slab + 127) / 128) * 128;
    return 128 + 2 * stage_bytes + 128 + MIX_WARPS * 8 * 4 + 16 + 64;
}

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
        const int smem = mix_bf16_smem_bytes(L, d);
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
        mix_rmsnorm_bf16_kernel<<<(unsigned)grid, MIX_THREADS, smem, st>>>(a, dev_err(ctx));
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
