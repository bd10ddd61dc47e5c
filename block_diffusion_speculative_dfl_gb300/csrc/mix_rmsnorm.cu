// Per-draft-layer mixture of target hidden states followed by RMSNorm.
//
// DFlare post, "Per-draft-layer mixing of different information": each draft
// layer l mixes the L target hidden states with softmax-normalised ratios
// and applies RMSNorm:  Xc_l[r] = g_l * x / sqrt(mean(x^2) + eps),
// x = sum_i softmax(mix_l)_i H_i[r].  All D draft layers come from one read of
// H, so the stack is streamed from HBM once per draft step.
//
// bf16 kernel: a persistent CTA per SM streams rows through a ring of up to
// four shared-memory stages (one TMA bulk copy per target layer slice), and
// two teams of 16 warps work on alternate rows, so one team's arithmetic
// overlaps the other's waits.  Per row each warp mixes its span of positions
// twice: once for the sum of squares, then (after the team's barrier) with
// the weights scaled by the row's rsqrt factor, writing the bf16 result over
// its consumed input in place and copying it out with 16-byte stores.  The
// L -> D mixing is a tiny matrix product per group of 16 positions, run on
// the tensor cores with mma.sync m16n8k16: A holds the mixing weights (rows
// 0..7 the bf16-rounded weight of draft layer 0..7, rows 8..15 the bf16
// remainder, so hi + lo carries the fp32 weight to ~2^-16), B holds the bf16
// hidden states (exact), accumulation is fp32.  The products of bf16 values
// are exact in fp32, so the result equals the fp32 mixture up to
// accumulation rounding.
//
// fp32 kernel: plain FFMA mixture, one CTA per row.
#include "internal.h"

namespace dfl {

namespace {

constexpr int MIX_TEAMS = 2;               // teams of warps working on alternate rows
constexpr int MIX_TEAM_WARPS = 16;
constexpr int MIX_THREADS = MIX_TEAMS * MIX_TEAM_WARPS * 32;
constexpr int MIX_MAXG = 20;               // 16-position groups per warp -> d <= 5120
constexpr int MIX_GCOLS = 4 * MIX_MAXG;    // TMEM columns of gains per thread
constexpr int MIX_TMEM_COLS = 512;         // 4 column blocks of MIX_GCOLS, rounded to a power of two
constexpr int MIX_MAXSTAGE = 4;            // rows staged at most
constexpr int MIX_ZERO_BYTES = 128 + MIX_MAXG * 32;   // zero rows read in place of target layers >= L

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

// Barrier over the `count` threads of named barrier `id` that also returns
// whether `pred` holds in every one of them.
__device__ __forceinline__ bool team_sync_and(int id, int count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
        "barrier.cta.red.and.pred p, %2, %3, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r) : "r"((uint32_t)pred), "r"(id), "r"(count) : "memory");
    return r != 0;
}

__device__ __forceinline__ void team_sync(int id, int count) {
    asm volatile("barrier.cta.sync %0, %1;" :: "r"(id), "r"(count) : "memory");
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

// Shared-memory plan of the bf16 kernel: `nstage` row stages of max(L, D)
// padded slabs (the L input slabs, overwritten in place by the D output
// slabs), the zero row, the per-team reduction arrays and the barriers.
// Slabs are padded by 16 bytes so that the rows of one ldmatrix (8 layers)
// and the bf16x2 writes of one warp (8 draft layers) fall on distinct banks.
struct MixSmem {
    int slab, stage_bytes, nstage, total;
};

__host__ __device__ inline MixSmem mix_smem_plan(int L, int D, int d, int nstage) {
    MixSmem m;
    m.slab = d * 2 + 16;
    m.stage_bytes = (((L > D ? L : D) * m.slab + 127) / 128) * 128;
    m.nstage = nstage;
    m.total = 128 + nstage * m.stage_bytes + MIX_ZERO_BYTES + MIX_TEAMS * MIX_TEAM_WARPS * 8 * 4 +
              MIX_MAXSTAGE * 2 * 8 + 16;
    return m;
}


// One persistent CTA per SM, two teams of 16 warps.  The CTA's rows are
// numbered k = 0, 1, ...; row k sits in stage k % nstage and is processed by
// team k % 2, so one team's arithmetic overlaps the other's waits.  Per row,
// each warp owns a contiguous span of at most GPW 16-position groups:
//   pass 1  mix its span on the tensor cores, sum of squares per draft layer;
//   team barrier (partial sums of every warp);
//   pass 2  mix again with the weights scaled by rsqrt(mean + eps) (the
//           product comes out normalised), apply the gain and write the bf16
//           result over the consumed input slabs of its span (draft layer l
//           into slab l), then copy its span of the D output rows to global
//           memory with 16-byte stores;
//   team barrier, after which the stage is refilled with row k + nstage.
// Recomputing the mixture (pass 2) costs a few tensor-core instructions and
// keeps nothing live across the barrier, which leaves room for two teams.
// GPW is a compile-time bound so that both passes unroll completely.
template <int GPW>
__global__ void __launch_bounds__(MIX_THREADS, 1) mix_rmsnorm_bf16_kernel(const MixArgs a, const int nstage,
                                                                         const DevErr err) {
    static_assert(GPW % 4 == 0 && GPW <= MIX_MAXG, "group bound");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const MixSmem P = mix_smem_plan(a.L, a.D, a.d, nstage);
    uint8_t* in0 = smem;                                       // stage s at in0 + s * stage_bytes
    uint8_t* zero_rows = smem + nstage * P.stage_bytes;        // MIX_ZERO_BYTES of zeros
    float* red = reinterpret_cast<float*>(zero_rows + MIX_ZERO_BYTES);   // [team][warp][8]
    uint64_t* full = reinterpret_cast<uint64_t*>(red + MIX_TEAMS * MIX_TEAM_WARPS * 8);
    int* fills = reinterpret_cast<int*>(full + MIX_MAXSTAGE);   // copies issued per stage
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(fills + 2 * MIX_MAXSTAGE);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int team = warp / MIX_TEAM_WARPS, tw = warp % MIX_TEAM_WARPS;
    const int bar_id = 1 + team, bar_n = MIX_TEAM_WARPS * 32;
    const uint32_t tx_bytes = (uint32_t)a.L * (uint32_t)a.d * 2u;
    const uint32_t row_bytes = (uint32_t)a.d * 2u;

    if (tid == 0) {
        for (int q = 0; q < nstage; ++q) { mbar_init(&full[q], 1); fills[q] = 0; }
        fence_barrier_init();
    }
    for (int i = tid; i < MIX_ZERO_BYTES / 4; i += MIX_THREADS) reinterpret_cast<uint32_t*>(zero_rows)[i] = 0u;
    // The RMSNorm gains do not change from row to row: warp tw of either team
    // finds the 4 * GPW gains of the positions it writes in TMEM lane quadrant
    // tw % 4, column block tw / 4 (written once, by team 0).
    if (warp == 0) { tmem_alloc(tmem_holder, MIX_TMEM_COLS); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    grid_dep_begin();   // global memory only from here on
    const uint32_t tgain = *tmem_holder + ((uint32_t)(32 * (tw & 3)) << 16) + (uint32_t)((tw >> 2) * MIX_GCOLS);

    // Row k of this CTA.
    auto row_of = [&](int k) -> int64_t { return blockIdx.x + (int64_t)k * gridDim.x; };
    // One warp stages row k's L slices, a slice per lane (L <= 16): issued
    // from one thread, each bulk copy held that thread ~80 ns, and the whole
    // team waited for the issuing warp at its next barrier.
    auto issue = [&](int k) {
        const int s = k % nstage;
        const int64_t row = row_of(k);
        uint8_t* dst = in0 + s * P.stage_bytes;
        if (lane == 0) {
            ++fills[s];
            mbar_arrive_expect_tx(&full[s], tx_bytes);
        }
        __syncwarp();
        if (lane < a.L)
            bulk_g2s(dst + lane * P.slab, a.H + lane * a.layer_stride + row * a.d, row_bytes, &full[s]);
    };
    if (warp == 0)
        for (int q = 0; q < nstage; ++q)
            if (row_of(q) < a.rows) issue(q);

    // A fragments: mixing weights of draft layer l = lane/4 (hi rows 0..7, lo
    // rows 8..15) for target layers k0, k0+1, k0+8, k0+9.
    float wts[4];
    {
        const int l = lane >> 2;
        const int k0 = 2 * (lane & 3);
        const int ks[4] = {k0, k0 + 1, k0 + 8, k0 + 9};
        #pragma unroll
        for (int j = 0; j < 4; ++j) wts[j] = (l < a.D && ks[j] < a.L) ? mix_weight(a.mix_logits, a.L, l, ks[j]) : 0.f;
    }
    auto make_frag = [&](float scale, uint32_t (&f)[4]) {
        uint16_t hi[4], lo[4];
        #pragma unroll
        for (int j = 0; j < 4; ++j) split_bf16(wts[j] * scale, hi[j], lo[j]);
        f[0] = (uint32_t)hi[0] | ((uint32_t)hi[1] << 16);   // row l,   k0..k0+1
        f[1] = (uint32_t)lo[0] | ((uint32_t)lo[1] << 16);   // row l+8, k0..k0+1
        f[2] = (uint32_t)hi[2] | ((uint32_t)hi[3] << 16);   // row l,   k0+8..k0+9
        f[3] = (uint32_t)lo[2] | ((uint32_t)lo[3] << 16);   // row l+8, k0+8..k0+9
    };
    uint32_t afrag[4];
    make_frag(1.f, afrag);

    const int groups = a.d / 16;
    // Warp tw owns the contiguous groups [g0, g0 + ng) (16 positions each).
    const int gpw = (groups + MIX_TEAM_WARPS - 1) / MIX_TEAM_WARPS;
    const int g0 = min(tw * gpw, groups);
    const int ng = min(gpw, groups - g0);
    const int l_out = lane >> 2;
    const int n = 2 * (lane & 3);
    const bool writes = l_out < a.D;
    // ldmatrix row of this thread (matrix lane/8 -> k half, position half): target
    // layer my_k of the stage, or the zero rows, at byte offset j * 32 for group g0 + j.
    const int my_k = ((lane >> 3) & 1) * 8 + (lane & 7);
    const int my_off = (lane >> 4) * 8;
    const bool k_real = my_k < a.L;
    const uint32_t zero_addr = smem_u32(zero_rows);
    const uint32_t ld_rel = (uint32_t)(my_k * P.slab + (g0 * 16 + my_off) * 2);
    // write position of this thread in its span: draft layer l_out, positions n, n+1 (+8) of each group
    const uint32_t st_rel = (uint32_t)(l_out * P.slab + (g0 * 16 + n) * 2);
    if (MIX_TEAMS > 1 && team == 0) {
        const float* gain_l = a.gain + (int64_t)(writes ? l_out : 0) * a.d;
        #pragma unroll 1
        for (int c = 0; c < GPW / 4; ++c) {
            uint32_t gv[16];
            #pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int j = 4 * c + q;
                float2 ga = make_float2(0.f, 0.f), gb = make_float2(0.f, 0.f);
                if (writes && j < ng) {
                    ga = __ldg(reinterpret_cast<const float2*>(gain_l + (g0 + j) * 16 + n));
                    gb = __ldg(reinterpret_cast<const float2*>(gain_l + (g0 + j) * 16 + n + 8));
                }
                gv[4 * q + 0] = __float_as_uint(ga.x);
                gv[4 * q + 1] = __float_as_uint(ga.y);
                gv[4 * q + 2] = __float_as_uint(gb.x);
                gv[4 * q + 3] = __float_as_uint(gb.y);
            }
            tmem_st16(tgain + 16 * c, gv);
        }
        tmem_st_wait();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // mixture of group j of the span: v = (pos n, n+1, n+8, n+9) of draft layer l_out
    auto mix_group = [&](const uint32_t (&af)[4], uint32_t addr, float (&v)[4]) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_trans(addr, b0, b1, b2, b3);
        float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
        mma_16816(c0, af, b0, b1);
        mma_16816(c1, af, b2, b3);
        v[0] = c0[0] + c0[2];   // hi + lo weight rows
        v[1] = c0[1] + c0[3];
        v[2] = c1[0] + c1[2];
        v[3] = c1[1] + c1[3];
    };

    // With a single stage (very wide rows) only team 0 works.
    const int tstep = nstage >= 2 ? MIX_TEAMS : 1;
    const bool full_span = ng == GPW;   // warp-uniform; false only for the last warps of ragged widths
    bool ok = true;
    int s = team % nstage;
    uint32_t par = (uint32_t)(team / nstage) & 1u;
    for (int k = team; team < tstep && row_of(k) < a.rows; k += tstep) {
        const int64_t row = row_of(k);
        ok = mbar_wait(&full[s], par, err);
        uint8_t* stage = in0 + s * P.stage_bytes;
        const uint32_t stage_addr = smem_u32(stage);
        // ldmatrix address of group 0 of the span; group j is 32 bytes further.
        // A zero row sits in the same bank slot (address mod 128) as the real
        // row it replaces, so the 8 rows of every 8x8 matrix hit distinct banks.
        const uint32_t ld0 = k_real ? stage_addr + ld_rel : zero_addr + (ld_rel & 127u);
        // ---- pass 1: sum of squares of this warp's span, per draft layer
        float ss = 0.f;
        if (ok) {
            if (full_span) {
                #pragma unroll 1
                for (int c = 0; c < GPW / 4; ++c) {
                    const uint32_t ldc = ld0 + 128u * c;
                    #pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        float v[4];
                        mix_group(afrag, ldc + 32u * q, v);
                        ss += v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3];
                    }
                }
            } else {
                #pragma unroll 1
                for (int j = 0; j < ng; ++j) {
                    float v[4];
                    mix_group(afrag, ld0 + 32u * j, v);
                    ss += v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3];
                }
            }
        }
        ss += __shfl_xor_sync(0xFFFFFFFFu, ss, 1);
        ss += __shfl_xor_sync(0xFFFFFFFFu, ss, 2);
        if ((lane & 3) == 0) red[(team * MIX_TEAM_WARPS + tw) * 8 + l_out] = ss;
        // The first chunk's gains for pass 2 are fetched across the team's
        // barrier (a tensor-memory round trip costs ~1 us under the mix's load).
        uint32_t gpre[16];
        tmem_ld16_issue(tgain, gpre);
        if (!team_sync_and(bar_id, bar_n, ok)) { tmem_ld16_wait(gpre); break; }   // a bounded wait ran out
        float tot = 0.f;
        #pragma unroll
        for (int w = 0; w < MIX_TEAM_WARPS; ++w) tot += red[(team * MIX_TEAM_WARPS + w) * 8 + l_out];
        const float rs = rsqrtf(tot / (float)a.d + a.eps);
        uint32_t afrag_n[4];
        make_frag(rs, afrag_n);
        // ---- pass 2: normalised bf16 output over the consumed input of the span.
        // The collective mma.sync consumes every lane's ldmatrix result, so a
        // group's input has been read in full before any lane overwrites it.
        auto pass2_chunk = [&](int c, const float (&gv)[16]) {
            const uint32_t ldc = ld0 + 128u * c;
            uint8_t* outc = stage + st_rel + 128 * c;
            #pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (full_span || 4 * c + q < ng) {
                    float v[4];
                    mix_group(afrag_n, ldc + 32u * q, v);
                    if (writes) {
                        *reinterpret_cast<uint32_t*>(outc + 32 * q) = pack_bf16(v[0] * gv[4 * q], v[1] * gv[4 * q + 1]);
                        *reinterpret_cast<uint32_t*>(outc + 32 * q + 16) =
                            pack_bf16(v[2] * gv[4 * q + 2], v[3] * gv[4 * q + 3]);
                    }
                }
            }
        };
        {
            tmem_ld16_wait(gpre);
            float gv[16];
            #pragma unroll
            for (int i = 0; i < 16; ++i) gv[i] = __uint_as_float(gpre[i]);
            pass2_chunk(0, gv);
        }
        #pragma unroll 1
        for (int c = 1; 4 * c < ng; ++c) {
            float gv[16];
            tmem_ld16(tgain + 16 * c, gv);
            pass2_chunk(c, gv);
        }
        // Copy the span's D output rows out: 16 bytes per lane, ng * 32 contiguous bytes per row.
        __syncwarp();
        {
            const uint8_t* src = stage + g0 * 32;
            __nv_bfloat16* dst = a.Xc + row * a.d + g0 * 16;
            // the span's last element of the last layer lies inside the D output slabs
            const bool in = DFL_IN_BOUNDS(err.word, (a.D - 1) * a.xc_stride + row * a.d + (g0 + ng) * 16 - 1,
                                          (a.D - 1) * a.xc_stride + a.rows * a.d);
            for (int l = 0; l < a.D && in; ++l) {
                for (int c = lane; c < 2 * ng; c += 32)
                    *reinterpret_cast<uint4*>(dst + c * 8) = *reinterpret_cast<const uint4*>(src + c * 16);
                src += P.slab;
                dst += a.xc_stride;
            }
        }
        // The stage's next contents come from TMA (the async proxy): order this
        // warp's shared-memory accesses before that write, then refill once
        // every warp is done with the stage.
        fence_proxy_async_smem();
        team_sync(bar_id, bar_n);
        if (tw == 0 && row_of(k + nstage) < a.rows) issue(k + nstage);
        s += tstep;
        if (s >= nstage) { s -= nstage; par ^= 1u; }
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
        // After a wait ran out: let every issued copy land before the CTA exits
        // (the latest fill of stage q completes phase fills[q] - 1).
        for (int q = 0; q < nstage; ++q)
            if (fills[q]) mbar_wait(&full[q], (uint32_t)(fills[q] - 1) & 1u, err);
    }
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(*tmem_holder, MIX_TMEM_COLS);
    }
}

// fp32: one CTA per row; mixtures kept in shared memory until the row's norm is known.
__global__ void mix_rmsnorm_f32_kernel(const float* H, int64_t layer_stride, int L, int64_t rows, int d, int D,
                                       const float* mix_logits, const float* gain, float eps, float* Xc,
                                       int64_t xc_stride) {
    grid_dep_begin();
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
    const dfl::ApiRange nvtx_range("dfl_layer_mix_rmsnorm");
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
        if (d % 16 != 0 || d > 16 * MIX_TEAM_WARPS * MIX_MAXG) return DFL_ERR_UNSUPPORTED_SHAPE;
        int nstage = MIX_MAXSTAGE;   // as many rows in flight as shared memory holds
        while (nstage > 1 && mix_smem_plan(L, D, d, nstage).total > 227 * 1024) --nstage;
        const int smem = mix_smem_plan(L, D, d, nstage).total;
        if (smem > 227 * 1024) return DFL_ERR_UNSUPPORTED_SHAPE;
        const int gpw = (d / 16 + MIX_TEAM_WARPS - 1) / MIX_TEAM_WARPS;
        const int gi = gpw <= 4 ? 0 : gpw <= 8 ? 1 : gpw <= 12 ? 2 : gpw <= 16 ? 3 : 4;
        using KernFn = void (*)(const MixArgs, const int, const DevErr);
        static const KernFn kerns[5] = {mix_rmsnorm_bf16_kernel<4>, mix_rmsnorm_bf16_kernel<8>,
                                        mix_rmsnorm_bf16_kernel<12>, mix_rmsnorm_bf16_kernel<16>,
                                        mix_rmsnorm_bf16_kernel<20>};
        const KernFn kern = kerns[gi];
        if (!ctx->mix_attr_set) {
            for (int i = 0; i < 5; ++i)
                if (cudaFuncSetAttribute(kerns[i], cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) !=
                    cudaSuccess)
                    return DFL_ERR_CUDA;
            ctx->mix_attr_set = true;
        }
        MixArgs a{static_cast<const __nv_bfloat16*>(H), layer_stride, L, rows, d, D, mix_logits, gain, eps,
                  static_cast<__nv_bfloat16*>(Xc), xc_layer_stride};
        const int64_t grid = rows < ctx->sm_count ? rows : ctx->sm_count;
        ProfScope ps("mix_rmsnorm_bf16", st);
        launch_pdl(kern, (unsigned)grid, MIX_THREADS, smem, st, a, nstage, dev_err(ctx));
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
    launch_pdl(mix_rmsnorm_f32_kernel, (unsigned)rows, 256, smem, st, static_cast<const float*>(H), layer_stride, L,
               rows, d, D, mix_logits, gain, eps, static_cast<float*>(Xc), xc_layer_stride);
    return last_launch();
}
