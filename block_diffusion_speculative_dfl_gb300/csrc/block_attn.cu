// Block attention of one draft layer, bf16 tensor-core kernel.
//
// DFlare post, "Generating candidates in parallel, the target decides
// acceptance": the block is predicted in one forward with bidirectional
// attention inside the block; DFlash article, "Writing a whole block in one
// forward pass": target context features enter every draft layer's K/V.
// So every block query attends to all C context keys and all B block keys:
//   O = softmax(Q [Kc;Kb]^T / sqrt(hd)) [Vc;Vb],  no mask,
// query head h reading K/V head h / (Hq/Hkv).
//
// One CTA per (sequence, K/V head, key split).  Its B*(Hq/Hkv) query rows are
// split over warps, 16 rows each.  64-key K/V tiles are staged in shared
// memory with cp.async (two tiles in flight, 16-byte chunks XOR-swizzled by
// row so ldmatrix is conflict-free); QK^T and PV run on mma.sync m16n8k16
// (bf16 in, fp32 accumulate) with an online softmax in registers.  With more
// than one split, each split writes normalised fp32 partials and its
// log-sum-exp, and a combine kernel merges them.
#include "internal.h"
#include "small_kernels.h"

namespace dfl {

namespace {

constexpr int KT = 64;             // keys per tile
constexpr int ATT_MAX_WARPS = 12;  // 16 query rows per warp; more rows -> more CTAs

struct AttnArgs {
    const __nv_bfloat16 *Q, *Kc, *Vc, *Kb, *Vb;
    int N, C, B, Hq, Hkv, G, R;
    const int32_t* ctx_len;   // nullable [N]: context keys of each sequence (else C)
    int C_stride;             // context rows per sequence in Kc / Vc
    int S, keys_per_split;
    __nv_bfloat16* O;   // written directly when S == 1
    float* Opart;       // [S][N*B*Hq][HD]
    float* lse;         // [S][N*B*Hq], log2 units
    float scale_log2;   // log2(e) / sqrt(hd)
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ST: K/V stages in the ring (ST - 1 tiles in flight while one is used).
template <int HD, int ST>
__global__ void __launch_bounds__(ATT_MAX_WARPS * 32) attn_bf16_kernel(const AttnArgs a) {
    grid_dep_begin();
    constexpr int CH = HD / 8;        // 16-byte chunks per row
    constexpr int ROWB = HD * 2;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const int NW = blockDim.x >> 5;
    const int nthr = blockDim.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sQ = smem_u32(sm);
    const uint32_t sK0 = sQ + NW * 16 * ROWB;
    const uint32_t tileB = KT * ROWB;
    // stage s: K at sK0 + s * 2 * tileB, V right after
    auto swz = [](int row, int chunk) -> uint32_t {
        return (uint32_t)(row * ROWB + ((chunk ^ (row & 7)) << 4));
    };

    const int n = blockIdx.x / a.Hkv, g = blockIdx.x % a.Hkv;
    const int split = blockIdx.y;
    const int r0 = blockIdx.z * NW * 16;   // first query row of this CTA
    const int Cn = a.ctx_len ? a.ctx_len[n] : a.C;   // this sequence's context keys
    const int k_begin = split * a.keys_per_split;
    const int k_end = min(Cn + a.B, k_begin + a.keys_per_split);
    const int ntiles = k_end > k_begin ? (k_end - k_begin + KT - 1) / KT : 0;
    const int64_t NQ = (int64_t)a.N * a.B * a.Hq;
    if (ntiles == 0) {   // split past this sequence's keys: an empty partial (weight 0 in the combine)
        if (a.S > 1) {
            for (int i = threadIdx.x; i < NW * 16; i += nthr) {
                const int row = r0 + i;
                if (row >= a.R) continue;
                const int64_t qrow = (int64_t)(n * a.B + row / a.G) * a.Hq + g * a.G + row % a.G;
                a.lse[(int64_t)split * NQ + qrow] = -INFINITY;
                float* out = a.Opart + ((int64_t)split * NQ + qrow) * HD;
                for (int e = 0; e < HD; ++e) out[e] = 0.f;
            }
        }
        return;
    }

    // Q rows of this CTA: r -> (block row b = r / G, head g*G + r % G)
    for (int i = tid; i < NW * 16 * CH; i += nthr) {
        const int r = i / CH, c = i % CH;
        const int rq = r0 + r;
        const bool ok = rq < a.R;
        const __nv_bfloat16* src = a.Q;
        if (ok) src = a.Q + ((int64_t)(n * a.B + rq / a.G) * a.Hq + g * a.G + rq % a.G) * HD + c * 8;
        cp_async16(sQ + swz(r, c), src, ok ? 16 : 0);
    }
    auto load_tile = [&](int t, int s) {
        const int key0 = k_begin + t * KT;
        const uint32_t dK = sK0 + s * 2 * tileB, dV = dK + tileB;
        for (int i = tid; i < KT * CH; i += nthr) {
            const int kr = i / CH, c = i % CH;
            const int key = key0 + kr;
            const bool ok = key < k_end;
            const __nv_bfloat16 *ks = a.Q, *vs = a.Q;
            if (ok) {
                if (key < Cn) {
                    const int64_t off = (((int64_t)n * a.C_stride + key) * a.Hkv + g) * HD + c * 8;
                    ks = a.Kc + off; vs = a.Vc + off;
                } else {
                    const int64_t off = ((int64_t)(n * a.B + key - Cn) * a.Hkv + g) * HD + c * 8;
                    ks = a.Kb + off; vs = a.Vb + off;
                }
            }
            cp_async16(dK + swz(kr, c), ks, ok ? 16 : 0);
            cp_async16(dV + swz(kr, c), vs, ok ? 16 : 0);
        }
    };
    load_tile(0, 0);
    cp_commit();
    if (ST == 3) {
        if (ntiles > 1) load_tile(1, 1);
        cp_commit();
    }

    uint32_t qf[HD / 16][4];
    float o[HD / 8][4];
    #pragma unroll
    for (int j = 0; j < HD / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};

    for (int t = 0; t < ntiles; ++t) {
        const int s = t % ST;
        if (t + ST - 1 < ntiles) load_tile(t + ST - 1, (t + ST - 1) % ST);
        cp_commit();
        cp_wait<ST - 1>();
        __syncthreads();
        if (t == 0) {
            #pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk) {
                const int r = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                ldsm_x4(sQ + swz(r, 2 * kk + (lane >> 4)), qf[kk]);
            }
        }
        const uint32_t dK = sK0 + s * 2 * tileB, dV = dK + tileB;
        float sc[8][4];
        #pragma unroll
        for (int j = 0; j < 8; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
        #pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
            #pragma unroll
            for (int p = 0; p < 4; ++p) {
                uint32_t b[4];
                ldsm_x4(dK + swz(p * 16 + (lane >> 4) * 8 + (lane & 7), 2 * kk + ((lane >> 3) & 1)), b);
                mma16816(sc[2 * p], qf[kk], b[0], b[1]);
                mma16816(sc[2 * p + 1], qf[kk], b[2], b[3]);
            }
        }
        const int key0 = k_begin + t * KT;
        if (key0 + KT > k_end) {
            #pragma unroll
            for (int j = 0; j < 8; ++j)
                #pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (key0 + j * 8 + 2 * (lane & 3) + (e & 1) >= k_end) sc[j][e] = -INFINITY;
        }
        #pragma unroll
        for (int r = 0; r < 2; ++r) {
            float mx = -INFINITY;
            #pragma unroll
            for (int j = 0; j < 8; ++j) mx = fmaxf(mx, fmaxf(sc[j][2 * r], sc[j][2 * r + 1]));
            mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
            const float mn = fmaxf(mrow[r], mx * a.scale_log2);
            const float alpha = exp2f(mrow[r] - mn);
            float sum = 0.f;
            #pragma unroll
            for (int j = 0; j < 8; ++j) {
                #pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float p = exp2f(sc[j][2 * r + e] * a.scale_log2 - mn);
                    sc[j][2 * r + e] = p;
                    sum += p;
                }
            }
            sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);
            sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 2);
            lrow[r] = lrow[r] * alpha + sum;
            mrow[r] = mn;
            #pragma unroll
            for (int j = 0; j < HD / 8; ++j) { o[j][2 * r] *= alpha; o[j][2 * r + 1] *= alpha; }
        }
        #pragma unroll
        for (int kk = 0; kk < KT / 16; ++kk) {
            uint32_t pa[4];
            pa[0] = pack_bf16(sc[2 * kk][0], sc[2 * kk][1]);
            pa[1] = pack_bf16(sc[2 * kk][2], sc[2 * kk][3]);
            pa[2] = pack_bf16(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
            pa[3] = pack_bf16(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
            #pragma unroll
            for (int p = 0; p < HD / 16; ++p) {
                uint32_t b[4];
                ldsm_x4_t(dV + swz(kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, 2 * p + (lane >> 4)), b);
                mma16816(o[2 * p], pa, b[0], b[1]);
                mma16816(o[2 * p + 1], pa, b[2], b[3]);
            }
        }
        __syncthreads();
    }

    #pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int row = r0 + warp * 16 + (lane >> 2) + 8 * r;
        if (row >= a.R) continue;
        const int64_t qrow = (int64_t)(n * a.B + row / a.G) * a.Hq + g * a.G + row % a.G;
        const float inv = 1.f / lrow[r];
        if (a.S == 1) {
            __nv_bfloat16* out = a.O + qrow * HD + 2 * (lane & 3);
            #pragma unroll
            for (int j = 0; j < HD / 8; ++j)
                *reinterpret_cast<uint32_t*>(out + j * 8) = pack_bf16(o[j][2 * r] * inv, o[j][2 * r + 1] * inv);
        } else {
            float* out = a.Opart + ((int64_t)split * NQ + qrow) * HD + 2 * (lane & 3);
            #pragma unroll
            for (int j = 0; j < HD / 8; ++j)
                *reinterpret_cast<float2*>(out + j * 8) = make_float2(o[j][2 * r] * inv, o[j][2 * r + 1] * inv);
            if ((lane & 3) == 0) a.lse[(int64_t)split * NQ + qrow] = mrow[r] + log2f(lrow[r]);
        }
    }
}

// O[q] = sum_s 2^(lse_s - max) O_s / sum_s 2^(lse_s - max).  One warp per
// query row; lane i owns HD/32 consecutive elements; split weights are formed
// once per row (S <= 64).
template <int HD>
__global__ void attn_combine_kernel(const float* Opart, const float* lse, int S, int64_t NQ, __nv_bfloat16* O) {
    grid_dep_begin();
    constexpr int PER = HD / 32;
    const int64_t q = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (q >= NQ) return;
    float l0 = lane < S ? lse[lane * NQ + q] : -INFINITY;
    float l1 = lane + 32 < S ? lse[(lane + 32) * NQ + q] : -INFINITY;
    const float mx = warp_max(fmaxf(l0, l1));
    const float w0 = lane < S ? exp2f(l0 - mx) : 0.f;
    const float w1 = lane + 32 < S ? exp2f(l1 - mx) : 0.f;
    const float inv = 1.f / warp_sum(w0 + w1);
    float acc[PER];
    #pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.f;
    for (int sp = 0; sp < S; ++sp) {
        const float wgt = __shfl_sync(0xFFFFFFFFu, sp < 32 ? w0 : w1, sp & 31);
        const float* src = Opart + (sp * NQ + q) * HD + lane * PER;
        if constexpr (PER == 4) {
            const float4 t = *reinterpret_cast<const float4*>(src);
            acc[0] += wgt * t.x; acc[1] += wgt * t.y; acc[2] += wgt * t.z; acc[3] += wgt * t.w;
        } else {
            const float2 t = *reinterpret_cast<const float2*>(src);
            acc[0] += wgt * t.x; acc[1] += wgt * t.y;
        }
    }
    __nv_bfloat16* dst = O + q * HD + lane * PER;
    if constexpr (PER == 4) {
        uint2 u;
        u.x = pack_bf16(acc[0] * inv, acc[1] * inv);
        u.y = pack_bf16(acc[2] * inv, acc[3] * inv);
        *reinterpret_cast<uint2*>(dst) = u;
    } else {
        *reinterpret_cast<uint32_t*>(dst) = pack_bf16(acc[0] * inv, acc[1] * inv);
    }
}

int attn_smem(int NW, int hd, int st) { return 128 + NW * 16 * hd * 2 + st * 2 * KT * hd * 2; }

}  // namespace

// Splits of the key range.  Model of the makespan on a 152-SM GB300 with two
// CTAs per SM: (rounds of CTAs over the 304 slots) x (64-key tiles per split
// + ~1.5 tiles of fixed per-CTA cost: Q load, pipeline fill, partial
// write-out, combine); the smallest S at the minimum wins.  At most 64 splits
// (the combine keeps two split weights per lane).  Depends on the shape only,
// so workspace sizes do not depend on the device.
int attn_splits(int N, int C, int B, int Hkv) {
    const int units = N * Hkv;
    const int tiles = (C + B + KT - 1) / KT;
    const int slots = 304;
    int best_s = 1;
    double best = 1e30;
    for (int S = 1; S <= 64 && S <= tiles; ++S) {
        const int per = (tiles + S - 1) / S;
        const int s_eff = (tiles + per - 1) / per;
        if (s_eff != S) continue;
        const double rounds = (double)((units * S + slots - 1) / slots);
        const double cost = rounds * (per + 1.5);
        if (cost < best - 1e-9) { best = cost; best_s = S; }
    }
    return best_s;
}

size_t attn_ws_bytes(int N, int C, int B, int Hq, int Hkv, int hd, bool ragged) {
    if (attn_tc_supported(B, Hq, Hkv, hd)) return attn_tc_ws_bytes(N, C, B, Hq, Hkv, hd, ragged);
    const int S = attn_splits(N, C, B, Hkv);
    if (S == 1) return 0;
    const size_t NQ = (size_t)N * B * Hq;
    return ((S * NQ * hd * sizeof(float) + 255) & ~size_t(255)) + ((S * NQ * sizeof(float) + 255) & ~size_t(255));
}

dfl_status attn_bf16(const void* Q, const void* Kc, const void* Vc, const void* Kb, const void* Vb, int N, int C,
                     int B, int Hq, int Hkv, int hd, void* O, void* ws, cudaStream_t st, const int32_t* ctx_len,
                     int C_stride, int policy_N) {
    if (attn_tc_supported(B, Hq, Hkv, hd)) return attn_tc(Q, Kc, Vc, Kb, Vb, N, C, B, Hq, Hkv, hd, O, ws, st, ctx_len,
                                                          C_stride, policy_N);
    AttnArgs a{};
    a.ctx_len = ctx_len;
    a.C_stride = ctx_len ? C_stride : C;
    a.Q = static_cast<const __nv_bfloat16*>(Q);
    a.Kc = static_cast<const __nv_bfloat16*>(Kc);
    a.Vc = static_cast<const __nv_bfloat16*>(Vc);
    a.Kb = static_cast<const __nv_bfloat16*>(Kb);
    a.Vb = static_cast<const __nv_bfloat16*>(Vb);
    a.N = N; a.C = C; a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.G = Hq / Hkv; a.R = B * a.G;
    a.S = attn_splits(policy_N > 0 ? policy_N : N, C, B, Hkv);
    const int tiles = (C + B + KT - 1) / KT;
    a.keys_per_split = ((tiles + a.S - 1) / a.S) * KT;
    a.O = static_cast<__nv_bfloat16*>(O);
    const size_t NQ = (size_t)N * B * Hq;
    if (a.S > 1) {
        a.Opart = static_cast<float*>(ws);
        a.lse = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) +
                                         ((a.S * NQ * hd * sizeof(float) + 255) & ~size_t(255)));
    }
    a.scale_log2 = 1.4426950408889634f / sqrtf((float)hd);
    int NW = (a.R + 15) / 16;
    const int zblocks = (NW + ATT_MAX_WARPS - 1) / ATT_MAX_WARPS;
    NW = (NW + zblocks - 1) / zblocks;
    // three stages if two CTAs still fit on an SM, else two
    const int stages = 2 * (attn_smem(NW, hd, 3) + 1024) <= 228 * 1024 ? 3 : 2;
    const int smem = attn_smem(NW, hd, stages);
    dim3 grid(N * Hkv, a.S, zblocks);
    dfl_status rc;
    {
    ProfScope ps("attn_bf16", st);
    auto run = [&](auto kern) -> bool {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return false;
        launch_pdl(kern, grid, NW * 32, smem, st, a);
        return true;
    };
    bool ok;
    if (hd == 128) ok = stages == 3 ? run(attn_bf16_kernel<128, 3>) : run(attn_bf16_kernel<128, 2>);
    else if (hd == 64) ok = stages == 3 ? run(attn_bf16_kernel<64, 3>) : run(attn_bf16_kernel<64, 2>);
    else return DFL_ERR_UNSUPPORTED_SHAPE;
    if (!ok) return DFL_ERR_CUDA;
    rc = last_launch();
    }
    if (rc != DFL_OK || a.S == 1) return rc;
    ProfScope ps("attn_combine", st);
    const unsigned cgrid = (unsigned)((NQ + 7) / 8);
    if (hd == 128)
        launch_pdl(attn_combine_kernel<128>, cgrid, 256, 0, st, a.Opart, a.lse, a.S, (int64_t)NQ, a.O);
    else
        launch_pdl(attn_combine_kernel<64>, cgrid, 256, 0, st, a.Opart, a.lse, a.S, (int64_t)NQ, a.O);
    return last_launch();
}

}  // namespace dfl
