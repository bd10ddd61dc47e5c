// Block attention of one draft layer on the 5th-generation tensor cores.
//
// DFlare post, "Generating candidates in parallel, the target decides
// acceptance": the block is predicted in one forward with bidirectional
// attention inside the block; DFlash article, "Writing a whole block in one
// forward pass": target context features enter every draft layer's K/V.  So
// the R = B * (Hq/Hkv) query rows that share K/V head g of sequence n attend
// to all of that sequence's context keys and all B block keys, no mask:
//   O = softmax(Q [Kc;Kb]^T / sqrt(hd)) [Vc;Vb].
//
// Work item = (split s, sequence n, K/V head g, head subset h): one range of
// at most `kps` keys of the sequence's Cn + B keys, for the Gq = G / hs query
// heads h*Gq .. h*Gq + Gq - 1 of the group (hs = 1 unless B * G exceeds the
// 128 MMA rows; the subsets of one group are consecutive items, so their K/V
// tiles are read from HBM once and from L2 by the others).  A persistent kernel (one CTA per SM)
// takes items from a global counter; empty items (past a shorter sequence's
// keys) are skipped by the scheduler.  Per CTA, two pipelines of 8 warps:
//   warp 0  scheduler + TMA producer of the item's Q rows (3-D box: head dim x
//           G heads x B block rows, zero rows up to 128) and its 64-key K
//           tiles (context cache, then one tile of the block's own keys);
//   warp 7  TMA producer of the matching V tiles.  K and V have rings of
//           their own, so a K slot is refilled as soon as S has read it while
//           its V waits for the P V product;
//   warp 1  issues S = Q K^T (M = 64 or 128 padded query rows, N = 64 keys,
//           K = hd) into one of NSB TMEM buffers as soon as the K tile has
//           landed and the buffer is free;
//   warp 6  issues O += P V (K = 64 keys, N = hd; P read from TMEM, V read
//           MN-major straight from its TMA tile) into a TMEM accumulator as
//           soon as P is written and V has landed;
//   warps 2-5  masked online softmax in base 2 with lazy rescaling (O is
//           rescaled in TMEM only when a row maximum grows by more than 2^8),
//           P written as bf16 over the first half of the tile's own S columns
//           (the A operand of P V), and the item's epilogue (bf16 output, or
//           fp32 partial + log-sum-exp when the sequence's keys span several
//           items).  At M = 128 each thread owns one row (its TMEM lane); at
//           M = 64 the 16 rows of a warp's quadrant are split over its 32
//           threads, each with half of a row's keys and of O.
// When an item has at most 64 query rows the products run with M = 64: the
// Q buffer halves, so the shared memory saved goes to deeper K/V rings.
// A combine kernel merges the partials of multi-item sequences.
#include "internal.h"
#include "small_kernels.h"

namespace dfl {

namespace {

constexpr int AT_KT = 64;           // keys per tile
constexpr int AT_M = 128;           // MMA rows (query rows, zero-padded)
constexpr float AT_LAZY = 8.f;      // rescale O only when a row max grows by more than this (log2 units)
constexpr int AT_IRING = 4;         // scheduled items in flight between the warps
// Warps per pipeline, one role each: 0 scheduler + Q/K producer, 1 S issuer,
// 2..5 softmax, 6 P V issuer, 7 V producer.  A role that blocks on barriers
// has a warp of its own: lanes of one warp waiting on different barriers hold
// one another up.
constexpr int AT_WPP = 8;
static_assert((AT_IRING & (AT_IRING - 1)) == 0, "ring positions are masked");

struct AtArgs {
    int N, B, Hq, Hkv, G, R;
    int hs, Gq;               // head subsets per K/V head, query heads per item (R = B * Gq)
    int C;                    // context keys per sequence (the maximum when ctx_len is given)
    int C_stride;             // context rows per sequence in Kc / Vc
    const int32_t* ctx_len;   // nullable [N]
    int kps;                  // keys per item (multiple of 64)
    int S;                    // items per (sequence, K/V head, head subset)
    int items;                // S * N * Hkv * hs
    int* counter;             // zeroed before the launch
    __nv_bfloat16* O;         // [N*B*Hq][hd]
    float* Opart;             // [S][N*B*Hq][hd]
    float* lse;               // [S][N*B*Hq], log2 units
    float scale_log2;         // log2(e) / sqrt(hd)
};

// MM: rows of the MMAs (64 when an item has at most 64 query rows, else 128).
// An M = 64 product puts row m in TMEM lane 32 (m / 16) + m % 16: the first
// 16 lanes of each warp's quadrant (the same for P read back as its A operand).
template <int HD, int MM>
struct AtCfg {
    static constexpr int NP = 2;                       // independent pipelines per CTA (two items in flight)
    static constexpr int KB = HD / 64;                 // 64-element K-blocks of a head row
    static constexpr int Q_BYTES = MM * HD * 2;        // one Q buffer
    static constexpr int QKB_BYTES = MM * 128;         // one K-block of Q (MM rows x 128 B)
    static constexpr int T_BYTES = AT_KT * HD * 2;     // one K or V tile
    static constexpr int TKB_BYTES = AT_KT * 128;      // one K-block of a K/V tile
    static constexpr int NQB = 1;                      // Q buffers per pipeline
    // S (and P) buffers in TMEM per pipeline: a third one, where the columns
    // allow it, lets S run a tile further ahead of the softmax
    static constexpr int NSB = HD == 64 ? 3 : 2;
    static constexpr int Q_TOTAL = NP * Q_BYTES;
    // K and V tiles have rings of their own: a K slot is free again once S has
    // read it, a V slot only after the P V product
    static constexpr int KST = HD == 128 ? (MM == 64 ? 3 : 2) : 6;    // K slots per pipeline
    static constexpr int VST = KST;                                     // V slots per pipeline
    static_assert(KST >= NSB && VST >= NSB, "completion barriers are shared by the K / V slots and S buffers");
    static constexpr int RING_BYTES = (KST + VST) * T_BYTES;
    static constexpr int O_COL = NSB * AT_KT;          // per pipeline: S buffers from column 0, O after them
    static constexpr int PIPE_COLS = 256;              // TMEM columns per pipeline
    static_assert(O_COL + HD <= PIPE_COLS, "TMEM columns");
    static constexpr int TMEM_COLS = NP * PIPE_COLS;
    static constexpr int THREADS = NP * AT_WPP * 32;
    static constexpr int BAR_BYTES = 512;              // barriers and scheduler slots per pipeline
    static constexpr int SMEM = 1024 + Q_TOTAL + NP * (RING_BYTES + BAR_BYTES);
    static_assert(SMEM <= 227 * 1024, "shared memory");
};

// One work item, decoded identically by every warp.
struct AtItem {
    int n, g, h, s;
    int Cn;          // context keys of the sequence
    int lo, hi;      // key range [lo, hi) of the Cn + B keys
    int nctx;        // context tiles (64 keys from lo, valid below min(hi, Cn))
    int blk;         // 1 if the range reaches into the block keys
    int direct;      // the whole sequence fits one item: write O directly
};

__device__ __forceinline__ bool at_decode(const AtArgs& a, int it, AtItem& x) {
    const int units = a.N * a.Hkv * a.hs;
    x.s = it / units;
    int u = it - x.s * units;
    x.h = u % a.hs;
    u /= a.hs;
    x.n = u / a.Hkv;
    x.g = u - x.n * a.Hkv;
    x.Cn = a.ctx_len ? a.ctx_len[x.n] : a.C;
    const int kn = x.Cn + a.B;
    x.lo = x.s * a.kps;
    if (x.lo >= kn) return false;
    x.hi = min(kn, x.lo + a.kps);
    const int ce = min(x.hi, x.Cn);
    x.nctx = ce > x.lo ? (ce - x.lo + AT_KT - 1) / AT_KT : 0;
    x.blk = x.hi > x.Cn ? 1 : 0;
    x.direct = kn <= a.kps ? 1 : 0;
    return true;
}

// Tile t of an item: context tile (t < nctx) or the block tile; the valid
// keys of its 64 rows are [v0, v1).
__device__ __forceinline__ void at_tile_range(const AtItem& x, int t, int& v0, int& v1) {
    if (t < x.nctx) {
        const int k0 = x.lo + t * AT_KT;
        v0 = 0;
        v1 = min(AT_KT, min(x.hi, x.Cn) - k0);
    } else {
        v0 = max(x.lo, x.Cn) - x.Cn;
        v1 = x.hi - x.Cn;
    }
}

// Barriers and scheduler slots of one pipeline.
template <int KST, int VST, int NQB, int NSB>
struct AtBars {
    // One completion barrier per product and slot: s_done[t % KST] completes when
    // S of tile t is done (its K slot is free, its S is ready for the softmax);
    // pv_done[t % VST] when P V of tile t is done (its V slot and S buffer are
    // free, O holds it).  A waiter for tile t's phase always knows that the
    // slot's previous phase (tile t - ring size) has completed, so the parity
    // test cannot mistake it.
    uint64_t k_full[KST], s_done[KST];
    uint64_t v_full[VST], pv_done[VST];
    uint64_t q_full[NQB], q_empty[NQB];
    uint64_t p_full[NSB];                 // P of the buffer written by all 128 softmax threads
    uint64_t o_full, o_empty;
    uint64_t i_full[AT_IRING], i_empty[AT_IRING];
    uint64_t drain, drain2;               // abort: the S / P V issuer's MMAs are done
    int i_ring[AT_IRING];
    int abort_flag;
};

// Position in a ring of N slots and the phase parity of its current use.
template <int N>
struct AtRing {
    uint32_t i = 0, ph = 0;
    __device__ __forceinline__ void step() {
        if (++i == N) { i = 0; ph ^= 1u; }
    }
};

template <int HD, int MM>
__global__ void __launch_bounds__(AtCfg<HD, MM>::THREADS, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmKc,
               const __grid_constant__ CUtensorMap tmVc, const __grid_constant__ CUtensorMap tmKb,
               const __grid_constant__ CUtensorMap tmVb, const AtArgs a, const DevErr err) {
    using Cfg = AtCfg<HD, MM>;
    constexpr int KST = Cfg::KST, VST = Cfg::VST, NQB = Cfg::NQB, NSB = Cfg::NSB;
    using Bars = AtBars<KST, VST, NQB, NSB>;
    static_assert(sizeof(Bars) + 8 <= Cfg::BAR_BYTES, "barrier area");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* bar_base = sm + Cfg::Q_TOTAL + Cfg::NP * Cfg::RING_BYTES;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bar_base + Cfg::NP * Cfg::BAR_BYTES - 8);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pp = warp / AT_WPP;     // this warp's pipeline
    const int role = warp % AT_WPP;   // see AT_WPP
    uint8_t* sQ = sm + pp * Cfg::Q_BYTES;                                // this pipeline's Q buffer
    uint8_t* sK = sm + Cfg::Q_TOTAL + pp * Cfg::RING_BYTES;              // [KST] K tiles
    uint8_t* sV = sK + KST * Cfg::T_BYTES;                               // [VST] V tiles
    Bars& bb = *reinterpret_cast<Bars*>(bar_base + pp * Cfg::BAR_BYTES);
    volatile int* abort_flag = &bb.abort_flag;

    if ((threadIdx.x % (AT_WPP * 32)) == 0) {
        for (int s = 0; s < KST; ++s) { mbar_init(&bb.k_full[s], 1); mbar_init(&bb.s_done[s], 1); }
        for (int s = 0; s < VST; ++s) { mbar_init(&bb.v_full[s], 1); mbar_init(&bb.pv_done[s], 1); }
        for (int b = 0; b < NQB; ++b) { mbar_init(&bb.q_full[b], 1); mbar_init(&bb.q_empty[b], 1); }
        for (int b = 0; b < NSB; ++b) mbar_init(&bb.p_full[b], 128);
        mbar_init(&bb.o_full, 1); mbar_init(&bb.o_empty, 128);
        for (int r = 0; r < AT_IRING; ++r) { mbar_init(&bb.i_full[r], 1); mbar_init(&bb.i_empty[r], 1 + 2 + 4); }   // V producer, two MMA issuers, four softmax warps
        mbar_init(&bb.drain, 1);
        mbar_init(&bb.drain2, 1);
        bb.abort_flag = 0;
        fence_barrier_init();
    }
    // Zero the Q buffers: MMA rows without a query row stay zero (TMA writes only the R real rows).
    for (int i = threadIdx.x; i < Cfg::Q_TOTAL / 16; i += Cfg::THREADS)
        *reinterpret_cast<uint4*>(sm + i * 16) = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmQ); prefetch_tensormap(&tmKc); prefetch_tensormap(&tmVc);
        prefetch_tensormap(&tmKb); prefetch_tensormap(&tmVb);
    }
    if (warp == 1) { tmem_alloc(tmem_holder, Cfg::TMEM_COLS); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder + pp * Cfg::PIPE_COLS;
    grid_dep_begin();   // global memory only from here on

    if (role == 0 || role == 7) {
        if (role == 0 && lane == 0) {
            // ---------------------------------------- scheduler + TMA producer of Q and K
            int icount = 0, tcount = 0;
            uint32_t k_fills = 0;
            bool aborted = false;
            while (true) {
                int it = -1;
                AtItem x;
                while (true) {   // next non-empty item
                    const int c = atomicAdd(a.counter, 1);
                    if (c >= a.items) break;
                    if (at_decode(a, c, x)) { it = c; break; }
                }
                const int r = icount % AT_IRING;
                if (*abort_flag || !mbar_wait(&bb.i_empty[r], ((icount / AT_IRING) & 1) ^ 1, err)) { aborted = true; break; }
                bb.i_ring[r] = it;
                mbar_arrive(&bb.i_full[r]);
                if (it < 0) break;
                const int qb = icount % NQB;
                if (*abort_flag || !mbar_wait(&bb.q_empty[qb], ((icount / NQB) & 1) ^ 1, err)) { aborted = true; break; }
                mbar_arrive_expect_tx(&bb.q_full[qb], a.R * HD * 2);
                #pragma unroll
                for (int kb = 0; kb < Cfg::KB; ++kb)
                    tma_load_3d(sQ + qb * Cfg::Q_BYTES + kb * Cfg::QKB_BYTES, &tmQ, kb * 64,
                                x.g * a.G + x.h * a.Gq, x.n * a.B, &bb.q_full[qb]);
                const int nt = x.nctx + x.blk;
                for (int t = 0; t < nt && !aborted; ++t) {
                    const int s = tcount % KST;
                    if (*abort_flag || !mbar_wait(&bb.s_done[s], ((tcount / KST) & 1) ^ 1, err)) { aborted = true; break; }
                    mbar_arrive_expect_tx(&bb.k_full[s], Cfg::T_BYTES);
                    const bool ctx = t < x.nctx;
                    const int row = ctx ? x.n * a.C_stride + x.lo + t * AT_KT : x.n * a.B;
                    #pragma unroll
                    for (int kb = 0; kb < Cfg::KB; ++kb)
                        tma_load_2d(sK + s * Cfg::T_BYTES + kb * Cfg::TKB_BYTES, ctx ? &tmKc : &tmKb, x.g * HD + kb * 64,
                                    row, &bb.k_full[s]);
                    k_fills |= 1u << s;
                    ++tcount;
                }
                if (aborted) break;
                ++icount;
            }
            if (aborted) {
                *abort_flag = 1;
                // let issued copies land before the CTA exits: the latest fill of
                // each slot has the parity of its fill count
                for (int s = 0; s < KST; ++s) {
                    if (!(k_fills & (1u << s))) continue;
                    const int last = tcount - 1 - ((tcount - 1 - s) % KST + KST) % KST;   // latest tile using slot s
                    mbar_wait(&bb.k_full[s], (last / KST) & 1, err);
                }
                // the Q load of the item being filled (icount) has been issued
                for (int b = 0; b < NQB; ++b) {
                    const int last = icount - ((icount - b) % NQB + NQB) % NQB;
                    if (last >= 0) mbar_wait(&bb.q_full[b], (last / NQB) & 1, err);
                }
            }
        } else if (role == 7 && lane == 0) {
            // ------------------------------------------------- TMA producer of V
            // follows the scheduled items like the consumers, as far ahead as the V ring allows
            int icount = 0, tcount = 0;
            uint32_t v_fills = 0;
            bool aborted = false;
            while (true) {
                const int r = icount % AT_IRING;
                if (*abort_flag || !mbar_wait(&bb.i_full[r], (icount / AT_IRING) & 1, err)) { aborted = true; break; }
                const int it = bb.i_ring[r];
                mbar_arrive(&bb.i_empty[r]);
                if (it < 0) break;
                AtItem x;
                at_decode(a, it, x);
                const int nt = x.nctx + x.blk;
                for (int t = 0; t < nt && !aborted; ++t) {
                    const int s = tcount % VST;
                    if (*abort_flag || !mbar_wait(&bb.pv_done[s], ((tcount / VST) & 1) ^ 1, err)) { aborted = true; break; }
                    mbar_arrive_expect_tx(&bb.v_full[s], Cfg::T_BYTES);
                    const bool ctx = t < x.nctx;
                    const int row = ctx ? x.n * a.C_stride + x.lo + t * AT_KT : x.n * a.B;
                    #pragma unroll
                    for (int kb = 0; kb < Cfg::KB; ++kb)
                        tma_load_2d(sV + s * Cfg::T_BYTES + kb * Cfg::TKB_BYTES, ctx ? &tmVc : &tmVb, x.g * HD + kb * 64,
                                    row, &bb.v_full[s]);
                    v_fills |= 1u << s;
                    ++tcount;
                }
                if (aborted) break;
                ++icount;
            }
            if (aborted) {
                *abort_flag = 1;
                for (int s = 0; s < VST; ++s) {
                    if (!(v_fills & (1u << s))) continue;
                    const int last = tcount - 1 - ((tcount - 1 - s) % VST + VST) % VST;
                    mbar_wait(&bb.v_full[s], (last / VST) & 1, err);
                }
            }
        }
    } else if (role == 1 || role == 6) {
        // Two MMA issuers, each a plain sequence of waits: warp 1 issues S = Q K^T of
        // every tile as soon as its K has landed and its S buffer is free (up to NSB
        // tiles ahead of the softmax); warp 6 issues O += P V of every tile as soon as
        // its P is written and its V has landed.  Each follows the scheduled items.
        constexpr uint32_t idesc_s = idesc_bf16(MM, AT_KT);
        constexpr uint32_t idesc_o = idesc_bf16_bmn(MM, HD);
        static_assert(NQB == 1, "one Q buffer per pipeline");
        if (role == 1 && lane == 0) {
            // ------------------------------------------------------ S issuer
            AtRing<KST> ks;                       // K slot of tile tcount
            AtRing<NSB> sb;                       // S buffer of tile tcount
            AtRing<VST> pe;                       // V slot of tile tcount - NSB (whose P V frees sb)
            const uint32_t sK32 = smem_u32(sK), qaddr = smem_u32(sQ);
            int icount = 0, tcount = 0;
            bool aborted = false, issued = false;
            while (!aborted) {
                const int r = icount & (AT_IRING - 1);
                if (*abort_flag || !mbar_wait(&bb.i_full[r], (icount / AT_IRING) & 1, err)) { aborted = true; break; }
                const int it = bb.i_ring[r];
                mbar_arrive(&bb.i_empty[r]);
                if (it < 0) break;
                AtItem x;
                at_decode(a, it, x);
                const int nt = x.nctx + x.blk;
                if (!mbar_wait(&bb.q_full[0], icount & 1, err)) { aborted = true; break; }
                for (int t = 0; t < nt; ++t) {
                    // S buffer sb is free once P V of tile tcount - NSB is done; this
                    // thread waited for P V of tile tcount - NSB - VST before issuing
                    // S of tile tcount - VST, so the V slot's previous phase is done
                    if (*abort_flag || !mbar_wait(&bb.k_full[ks.i], ks.ph, err) ||
                        (tcount >= NSB && !mbar_wait(&bb.pv_done[pe.i], pe.ph, err))) { aborted = true; break; }
                    tc_fence_after();
                    const uint32_t kaddr = sK32 + ks.i * Cfg::T_BYTES;
                    #pragma unroll
                    for (int j = 0; j < HD / 16; ++j)
                        mma_bf16(tmem_base + sb.i * AT_KT, sw128_desc(qaddr + (j >> 2) * Cfg::QKB_BYTES + (j & 3) * 32),
                                 sw128_desc(kaddr + (j >> 2) * Cfg::TKB_BYTES + (j & 3) * 32), idesc_s, j > 0);
                    issued = true;
                    mma_commit(&bb.s_done[ks.i]);
                    if (t == nt - 1) mma_commit(&bb.q_empty[0]);
                    if (tcount >= NSB) pe.step();
                    ks.step();
                    sb.step();
                    ++tcount;
                }
                ++icount;
            }
            if (aborted) {
                *abort_flag = 1;
                if (issued) {   // let issued MMAs finish before TMEM is released
                    mma_commit(&bb.drain);
                    mbar_wait(&bb.drain, 0, err);
                }
            }
        } else if (role == 6 && lane == 0) {
            // ------------------------------------------------------ P V issuer
            AtRing<NSB> pb;                       // S / P buffer of tile tcount
            AtRing<VST> vs;                       // V slot of tile tcount
            const uint32_t sV32 = smem_u32(sV);
            int icount = 0;
            bool aborted = false, issued = false;
            while (!aborted) {
                const int r = icount & (AT_IRING - 1);
                if (*abort_flag || !mbar_wait(&bb.i_full[r], (icount / AT_IRING) & 1, err)) { aborted = true; break; }
                const int it = bb.i_ring[r];
                mbar_arrive(&bb.i_empty[r]);
                if (it < 0) break;
                AtItem x;
                at_decode(a, it, x);
                const int nt = x.nctx + x.blk;
                // O is free once the previous item's epilogue has read it
                if (!mbar_wait(&bb.o_empty, (icount & 1) ^ 1, err)) { aborted = true; break; }
                for (int t = 0; t < nt; ++t) {
                    if (*abort_flag || !mbar_wait(&bb.p_full[pb.i], pb.ph, err) || !mbar_wait(&bb.v_full[vs.i], vs.ph, err)) {
                        aborted = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t vaddr = sV32 + vs.i * Cfg::T_BYTES;
                    // P (bf16, 2 per column) sits in the first 32 columns of S buffer pb:
                    // 16 keys per MMA = 8 columns
                    #pragma unroll
                    for (int j = 0; j < AT_KT / 16; ++j)
                        mma_bf16_ts(tmem_base + Cfg::O_COL, tmem_base + pb.i * AT_KT + 8 * j,
                                    sw128_desc_mn(vaddr + j * 16 * 128, Cfg::TKB_BYTES, 1024), idesc_o,
                                    (t == 0 && j == 0) ? 0 : 1);
                    issued = true;
                    mma_commit(&bb.pv_done[vs.i]);
                    if (t == nt - 1) mma_commit(&bb.o_full);
                    pb.step();
                    vs.step();
                }
                ++icount;
            }
            if (aborted) {
                *abort_flag = 1;
                if (issued) {
                    mma_commit(&bb.drain2);
                    mbar_wait(&bb.drain2, 0, err);
                }
            }
        }
    } else {
        // ---------------------------------------------------- softmax + epilogue
        // M = 128: one query row per thread (its TMEM lane) with all 64 keys of a
        // tile and all of O's columns.  M = 64: the 16 rows of the warp's quadrant
        // are shared by its 32 threads (half-split TMEM accesses): thread t holds
        // row 16 q + t % 16, keys [32 (t / 16), + 32) of each tile and half of O's
        // columns; the two halves of a row meet by one shuffle.
        constexpr bool HALF = MM == 64;
        constexpr int KPT = HALF ? AT_KT / 2 : AT_KT;   // keys per thread and tile
        constexpr int OPT = HALF ? HD / 2 : HD;         // O columns per thread
        const int q4 = warp & 3;
        const int hh = HALF ? lane >> 4 : 0;            // this thread's half of the keys and of O
        // query row of the item held by this thread (R of them; the others are padding)
        const int row = HALF ? 16 * q4 + (lane & 15) : 32 * q4 + lane;
        const bool pad = (HALF ? 16 : 32) * q4 >= a.R;  // warp-uniform: padding rows only
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        const int stid = threadIdx.x - pp * AT_WPP * 32 - 64;        // 0..127 within the pipeline's softmax warps
        int icount = 0, tcount = 0;
        bool ok = true;
        while (ok) {
            const int r = icount % AT_IRING;
            ok = mbar_wait(&bb.i_full[r], (icount / AT_IRING) & 1, err);
            if (!__all_sync(0xFFFFFFFFu, ok) || __any_sync(0xFFFFFFFFu, *abort_flag != 0)) { ok = false; break; }
            const int it = bb.i_ring[r];
            __syncwarp();
            if (lane == 0) mbar_arrive(&bb.i_empty[r]);
            if (it < 0) break;
            AtItem x;
            at_decode(a, it, x);
            const int nt = x.nctx + x.blk;
            float m_run = -INFINITY, l_run = 0.f;
            for (int t = 0; t < nt; ++t) {
                const int b = tcount % NSB;
                ok = mbar_wait(&bb.s_done[tcount % KST], (tcount / KST) & 1, err);
                if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; break; }   // also reconverges the warp
                tc_fence_after();
                int v0, v1;
                at_tile_range(x, t, v0, v1);
                if (!pad) {   // padding rows: nothing to compute; their P columns may hold anything
                uint32_t pk[KPT / 2];
                float s[KPT];
                if constexpr (HALF) tmem_ld32_hx2<AT_KT / 2>(tmem_base + lane_off + b * AT_KT, s);
                else tmem_ld64(tmem_base + lane_off + b * AT_KT, s);
                const int k0 = hh * KPT;      // this thread's first key of the tile
                if (v0 > 0 || v1 < AT_KT) {   // edge tile (warp-uniform): keys outside [v0, v1) do not exist
                    #pragma unroll
                    for (int j = 0; j < KPT; ++j)
                        if (k0 + j < v0 || k0 + j >= v1) s[j] = -INFINITY;
                }
                // row maximum of the raw scores (scale > 0 commutes with max), four partial chains
                float m4[4] = {s[0], s[1], s[2], s[3]};
                #pragma unroll
                for (int j = 4; j < KPT; j += 4) {
                    m4[0] = fmaxf(m4[0], s[j]); m4[1] = fmaxf(m4[1], s[j + 1]);
                    m4[2] = fmaxf(m4[2], s[j + 2]); m4[3] = fmaxf(m4[3], s[j + 3]);
                }
                float mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * a.scale_log2;
                if constexpr (HALF) mt = fmaxf(mt, __shfl_xor_sync(0xFFFFFFFFu, mt, 16));
                if (t == 0) {
                    m_run = mt;
                } else {
                    const bool need = mt > m_run + AT_LAZY;
                    if (__any_sync(0xFFFFFFFFu, need)) {
                        // O of this item holds the P V products up to the previous tile: wait for the last one
                        const int tp = tcount - 1;
                        ok = mbar_wait(&bb.pv_done[tp % VST], (tp / VST) & 1, err);
                        if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; break; }
                        tc_fence_after();
                        const float m_new = need ? mt : m_run;
                        const float alpha = exp2f(m_run - m_new);
                        #pragma unroll 1
                        for (int c = 0; c < OPT; c += 32) {
                            float o[32];
                            if constexpr (HALF) tmem_ld32_hx2<HD / 2>(tmem_base + lane_off + Cfg::O_COL + c, o);
                            else tmem_ld32(tmem_base + lane_off + Cfg::O_COL + c, o);
                            #pragma unroll
                            for (int j = 0; j < 32; ++j) o[j] *= alpha;
                            if constexpr (HALF) tmem_st32_hx2<HD / 2>(tmem_base + lane_off + Cfg::O_COL + c, o);
                            else tmem_st32(tmem_base + lane_off + Cfg::O_COL + c, o);
                        }
                        tmem_st_wait();
                        tc_fence_before();
                        l_run *= alpha;
                        m_run = m_new;
                    }
                }
                // p = 2^(s * scale - m): one FMA and one SFU op per score; four partial sums
                float l4[4] = {0.f, 0.f, 0.f, 0.f};
                const float neg_m = -m_run;
                #pragma unroll
                for (int j = 0; j < KPT; j += 2) {
                    const float p0 = ex2_ftz(fmaf(s[j], a.scale_log2, neg_m));
                    const float p1 = ex2_ftz(fmaf(s[j + 1], a.scale_log2, neg_m));
                    l4[(j >> 1) & 3] += p0 + p1;
                    pk[j / 2] = pack_bf16(p0, p1);
                }
                l_run += (l4[0] + l4[1]) + (l4[2] + l4[3]);
                // P over the first half of this tile's S columns (this thread's own lane, whose
                // S it has already read): the A operand of the P V product; key k of a row
                // in column k / 2
                if constexpr (HALF) tmem_st16u_hx2<AT_KT / 4>(tmem_base + lane_off + b * AT_KT, pk);
                else tmem_st32u(tmem_base + lane_off + b * AT_KT, pk);
                tmem_st_wait();
                }
                // Rows of the V tile outside [v0, v1) may hold anything (cache rows past
                // the sequence's length): zero them, so that 0 * V adds exactly nothing.
                if (v0 > 0 || v1 < AT_KT) {
                    // the V tile has landed; its slot is not refilled before this
                    // tile's P V product, which waits for these writes
                    ok = mbar_wait(&bb.v_full[tcount % VST], (tcount / VST) & 1, err);
                    if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; break; }
                    uint8_t* vt = sV + (tcount % VST) * Cfg::T_BYTES;
                    for (int i = stid; i < AT_KT * Cfg::KB * 8; i += 128) {
                        const int kr = (i >> 3) % AT_KT;
                        if (kr >= v0 && kr < v1) continue;
                        *reinterpret_cast<uint4*>(vt + (i >> 3) / AT_KT * Cfg::TKB_BYTES + kr * 128 + (i & 7) * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();   // visible to the P V product's operand reads
                }
                tc_fence_before();
                mbar_arrive(&bb.p_full[b]);
                ++tcount;
            }
            if (!ok) break;
            // ---- epilogue of the item
            ok = mbar_wait(&bb.o_full, icount & 1, err);
            if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; break; }
            tc_fence_after();
            const bool real = row < a.R;   // other MMA rows are padding
            const int64_t NQ = (int64_t)a.N * a.B * a.Hq;
            const int64_t qrow =
                real ? (int64_t)(x.n * a.B + row / a.Gq) * a.Hq + x.g * a.G + x.h * a.Gq + row % a.Gq : 0;
            float l_tot = l_run;   // the row's sum over all keys
            if constexpr (HALF) l_tot += __shfl_xor_sync(0xFFFFFFFFu, l_run, 16);
            const float inv = 1.f / l_tot;
            #pragma unroll 1
            for (int c0 = 0; c0 < OPT && !pad; c0 += 32) {
                float o[32];
                __syncwarp();
                if constexpr (HALF) tmem_ld32_hx2<HD / 2>(tmem_base + lane_off + Cfg::O_COL + c0, o);
                else tmem_ld32(tmem_base + lane_off + Cfg::O_COL + c0, o);
                if (!real) continue;
                const int c = hh * OPT + c0;   // O column of o[0]
                if (!DFL_IN_BOUNDS(err.word, (x.direct ? qrow : (int64_t)x.s * NQ + qrow) * HD + c + 31,
                                   (x.direct ? (int64_t)1 : (int64_t)a.S) * NQ * HD))
                    continue;
                if (x.direct) {
                    uint4* dst = reinterpret_cast<uint4*>(a.O + qrow * HD + c);
                    #pragma unroll
                    for (int j = 0; j < 4; ++j)
                        dst[j] = make_uint4(pack_bf16(o[8 * j] * inv, o[8 * j + 1] * inv),
                                            pack_bf16(o[8 * j + 2] * inv, o[8 * j + 3] * inv),
                                            pack_bf16(o[8 * j + 4] * inv, o[8 * j + 5] * inv),
                                            pack_bf16(o[8 * j + 6] * inv, o[8 * j + 7] * inv));
                } else {
                    float4* dst = reinterpret_cast<float4*>(a.Opart + ((int64_t)x.s * NQ + qrow) * HD + c);
                    #pragma unroll
                    for (int j = 0; j < 8; ++j)
                        dst[j] = make_float4(o[4 * j] * inv, o[4 * j + 1] * inv, o[4 * j + 2] * inv,
                                             o[4 * j + 3] * inv);
                }
            }
            __syncwarp();
            tc_fence_before();
            mbar_arrive(&bb.o_empty);
            if (real && !pad && !x.direct && hh == 0 &&
                DFL_IN_BOUNDS(err.word, (int64_t)x.s * NQ + qrow, (int64_t)a.S * NQ))
                a.lse[(int64_t)x.s * NQ + qrow] = m_run + log2f(l_tot);
            ++icount;
        }
        if (!ok) *abort_flag = 1;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(*tmem_holder, Cfg::TMEM_COLS);
    }
}

// O[q] = sum_s 2^(lse_s - max) O_s / sum_s 2^(lse_s - max) over the items of
// q's sequence, for sequences whose keys span more than one item.  One warp
// per query row; lane i owns HD/32 consecutive elements.
template <int HD>
__global__ void attn_tc_combine_kernel(const float* Opart, const float* lse, int64_t NQ, int rows_per_seq, int B,
                                       int C, const int32_t* ctx_len, int kps, int S_max, int* err,
                                       __nv_bfloat16* O) {
    grid_dep_begin();
    constexpr int PER = HD / 32;
    const int64_t q = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (q >= NQ) return;
    const int n = (int)(q / rows_per_seq);
    int S = ((ctx_len ? ctx_len[n] : C) + B + kps - 1) / kps;
    if (S > S_max) {   // a context length beyond the capacity: never read past the partials
        if (err && lane == 0) atomicCAS(err, 0, DFL_ERR_INVALID_ARG);
        S = S_max;
    }
    if (S <= 1) return;   // written by the attention kernel
    const float l0 = lane < S ? lse[lane * NQ + q] : -INFINITY;
    const float l1 = lane + 32 < S ? lse[(lane + 32) * NQ + q] : -INFINITY;
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

// bf16 [rows][cols] row-major, box = box_rows x 64 columns, 128-byte swizzle.
bool at_map_2d(CUtensorMap* m, const void* base, int64_t rows, int cols, int box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Q [N*B][Hq][hd] as (hd, Hq, N*B); box = 64 x G (query heads of one item) x B block rows.
bool at_map_q(CUtensorMap* m, const void* base, int NB, int Hq, int hd, int G, int B) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)hd, (cuuint64_t)Hq, (cuuint64_t)NB};
    cuuint64_t strides[2] = {(cuuint64_t)hd * 2, (cuuint64_t)Hq * hd * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)B};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int AT_SLOTS = 152;   // one persistent CTA per SM of a GB300

}  // namespace

// Head subsets per K/V head: the fewest that give at most 128 query rows per item.
int at_head_subsets(int B, int G) {
    for (int hs = 1; hs <= G; ++hs)
        if (G % hs == 0 && B * (G / hs) <= AT_M) return hs;
    return 0;
}

bool attn_tc_supported(int B, int Hq, int Hkv, int hd) {
    if (hd != 64 && hd != 128) return false;
    if (Hkv <= 0 || Hq % Hkv != 0) return false;
    const int G = Hq / Hkv;
    return B >= 1 && B <= AT_KT && G <= 256 && at_head_subsets(B, G) > 0;
}

// Keys per item.  Makespan model over 152 persistent CTAs, in units of one
// 64-key tile: with fixed lengths, (rounds of items) x (tiles per item + the
// item's fixed cost: Q load and pipeline turn-around, plus the partial
// write-out and combine when a sequence spans several items); with per-
// sequence lengths (`ragged`, C the capacity), lengths are taken spread evenly
// over [0, C] and items are handed out dynamically: total work / 152 + half an
// item.  Depends on the shape only, so workspace sizes do not depend on the
// device.
int attn_tc_kps(int units, int C, int B, bool ragged) {
    const int ktiles = (C + B + AT_KT - 1) / AT_KT;
    int best_kps = ktiles * AT_KT;
    double best = 1e30;
    for (int S = 1; S <= 64 && S <= ktiles; ++S) {
        const int per = (ktiles + S - 1) / S;
        const int kps = per * AT_KT;
        const int s_eff = (C + B + kps - 1) / kps;
        if (s_eff != S) continue;
        const double ovh = 0.5 + (S > 1 ? 1.0 : 0.0);
        double cost;
        if (!ragged) {
            cost = (double)((units * S + AT_SLOTS - 1) / AT_SLOTS) * (per + 1 + ovh);
        } else {
            double total = 0.0;
            const int samples = 16;
            for (int i = 0; i < samples; ++i) {
                const int cn = (int)((double)C * (i + 0.5) / samples);
                const int kn = cn + B;
                for (int s = 0; s * kps < kn; ++s) {
                    const int lo = s * kps, hi = std::min(kn, lo + kps), ce = std::min(hi, cn);
                    const int t = (ce > lo ? (ce - lo + AT_KT - 1) / AT_KT : 0) + (hi > cn ? 1 : 0);
                    total += t + ovh;
                }
            }
            total *= (double)units / samples;
            cost = std::max((double)per + 1 + ovh, total / AT_SLOTS + 0.5 * (per + 1 + ovh));
        }
        if (cost < best - 1e-9) { best = cost; best_kps = kps; }
    }
    return best_kps;
}

size_t attn_tc_ws_bytes(int N, int C, int B, int Hq, int Hkv, int hd, bool ragged) {
    const int kps = attn_tc_kps(N * Hkv * at_head_subsets(B, Hq / Hkv), C, B, ragged);
    const int S = (C + B + kps - 1) / kps;
    const size_t NQ = (size_t)N * B * Hq;
    size_t b = 256;   // item counter
    if (S > 1) b += ((S * NQ * hd * sizeof(float) + 255) & ~size_t(255)) + ((S * NQ * sizeof(float) + 255) & ~size_t(255));
    return b;
}

dfl_status attn_tc(const void* Q, const void* Kc, const void* Vc, const void* Kb, const void* Vb, int N, int C,
                   int B, int Hq, int Hkv, int hd, void* O, void* ws, cudaStream_t st, const int32_t* ctx_len,
                   int C_stride, int policy_N) {
    DeviceCtx* ctx = current_ctx();
    if (!ctx) return DFL_ERR_NO_DEVICE;
    const bool ragged = ctx_len != nullptr;
    AtArgs a{};
    a.N = N; a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.G = Hq / Hkv;
    a.hs = at_head_subsets(B, a.G); a.Gq = a.G / a.hs; a.R = B * a.Gq;
    a.C = C; a.C_stride = ragged ? C_stride : C; a.ctx_len = ctx_len;
    a.kps = attn_tc_kps((policy_N > 0 ? policy_N : N) * Hkv * a.hs, C, B, ragged);
    a.S = (C + B + a.kps - 1) / a.kps;
    a.items = a.S * N * Hkv * a.hs;
    const size_t NQ = (size_t)N * B * Hq;
    uint8_t* p = static_cast<uint8_t*>(ws);
    a.counter = reinterpret_cast<int*>(p);
    p += 256;
    if (a.S > 1) {
        a.Opart = reinterpret_cast<float*>(p);
        p += (a.S * NQ * hd * sizeof(float) + 255) & ~size_t(255);
        a.lse = reinterpret_cast<float*>(p);
    }
    a.O = static_cast<__nv_bfloat16*>(O);
    a.scale_log2 = 1.4426950408889634f / sqrtf((float)hd);
    CUtensorMap mq, mkc, mvc, mkb, mvb;
    const int kv = Hkv * hd;
    const int64_t ctx_rows = (int64_t)N * a.C_stride;
    const void* kc = C > 0 ? Kc : Kb;   // an empty context is never read; any valid map serves
    const void* vc = C > 0 ? Vc : Vb;
    if (!at_map_q(&mq, Q, N * B, Hq, hd, a.Gq, B) ||
        !at_map_2d(&mkc, kc, C > 0 ? ctx_rows : (int64_t)N * B, kv, AT_KT) ||
        !at_map_2d(&mvc, vc, C > 0 ? ctx_rows : (int64_t)N * B, kv, AT_KT) ||
        !at_map_2d(&mkb, Kb, (int64_t)N * B, kv, AT_KT) || !at_map_2d(&mvb, Vb, (int64_t)N * B, kv, AT_KT))
        return DFL_ERR_CUDA;
    dfl_status rc;
    {
        ProfScope ps("attn_tc", st);
        if (cudaMemsetAsync(a.counter, 0, sizeof(int), st) != cudaSuccess) return DFL_ERR_CUDA;
        const int grid = std::min(ctx->sm_count, a.items);
        const DevErr err = dev_err(ctx);
        auto run = [&](auto kern, int smem, int threads, int slot) -> dfl_status {
            if (!ctx->attn_attr_set[slot]) {
                if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
                    return DFL_ERR_CUDA;
                ctx->attn_attr_set[slot] = true;
            }
            launch_pdl(kern, grid, threads, smem, st, mq, mkc, mvc, mkb, mvb, a, err);
            return last_launch();
        };
        // M = 64 products when each item has at most 64 query rows
        const bool m64 = a.R <= 64;
        if (hd == 128)
            rc = m64 ? run(attn_tc_kernel<128, 64>, AtCfg<128, 64>::SMEM, AtCfg<128, 64>::THREADS, 3)
                     : run(attn_tc_kernel<128, 128>, AtCfg<128, 128>::SMEM, AtCfg<128, 128>::THREADS, 1);
        else
            rc = m64 ? run(attn_tc_kernel<64, 64>, AtCfg<64, 64>::SMEM, AtCfg<64, 64>::THREADS, 2)
                     : run(attn_tc_kernel<64, 128>, AtCfg<64, 128>::SMEM, AtCfg<64, 128>::THREADS, 0);
    }
    if (rc != DFL_OK || a.S == 1) return rc;
    ProfScope ps("attn_combine", st);
    const unsigned cgrid = (unsigned)((NQ + 7) / 8);
    if (hd == 128)
        launch_pdl(attn_tc_combine_kernel<128>, cgrid, 256, 0, st, a.Opart, a.lse, (int64_t)NQ, B * Hq, B, C, ctx_len,
                   a.kps, a.S, ctx->err_word, a.O);
    else
        launch_pdl(attn_tc_combine_kernel<64>, cgrid, 256, 0, st, a.Opart, a.lse, (int64_t)NQ, B * Hq, B, C, ctx_len,
                   a.kps, a.S, ctx->err_word, a.O);
    return last_launch();
}

}  // namespace dfl
