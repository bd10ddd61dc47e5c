// tcgen05 tensor-core GEMM for sm_103a: C[M][N] = A[M][K] * B[N][K]^T.
//
// A and B are bf16, K-major (row-major with K contiguous), loaded by TMA with
// 128-byte swizzling into a shared-memory ring; one elected thread issues
// tcgen05.mma (128 x BN x 16 on one SM, or 256 x BN x 16 over an SM pair; a
// 512-wide pair tile as two 256-wide products per step) into a TMEM
// accumulator, double-buffered up to 256 columns (a 512-wide tile's single
// accumulator fills tensor memory); four epilogue warps (eight for 512-wide
// tiles, two per lane quadrant) read TMEM with tcgen05.ld and apply one of
// four epilogues:
//   EPI_STORE  bf16 store into up to three column segments, rotary embedding
//              on segments that ask for it (stores staged per warp in shared
//              memory, so that each instruction writes whole row segments);
//   EPI_RESID  fp32 residual accumulate (out += C), or plain fp32 store;
//   EPI_ARGMAX per-row max / argmax over the tile's columns (lowest column on
//              ties), optional fp32 logits store and optional per-tile
//              sum of exp((z - tile max) / T) in fp64 for sampling;
//   EPI_SWIGLU the B tile is [gate rows of W1 ; up rows of W3] for the same
//              BN/2 features; stores silu(gate) * up as bf16.
// The grid is persistent (one CTA per SM); tiles are walked in an order that
// keeps the shared operand of consecutive tiles in L2.
#pragma once

#include "common.cuh"

namespace dfl {

enum EpiKind { EPI_STORE = 0, EPI_RESID = 1, EPI_ARGMAX = 2, EPI_SWIGLU = 3 };

struct GemmSeg {
    void* out;        // bf16 [rows][ld] (EPI_STORE)
    int n_begin;      // first global column of the segment
    int ld;           // row stride, elements
    int rope;         // apply rotate-half rotary embedding
    int64_t rows;     // rows of the output buffer (bounds-checked build)
};

struct GemmEpi {
    GemmSeg seg[3];
    int nseg;
    // rotary: row r sits at position pos_off + (r % rows_per_seq), or at
    // row_pos[r] when row_pos is given (per-sequence context lengths)
    const float* rope;   // [P][hd/2][2] (cos, sin)
    int hd;
    int rows_per_seq;
    int pos_off;
    const int32_t* row_pos;   // nullable [M]
    const int32_t* row_dst;   // nullable [M]: output row of GEMM row r (scatter), < 0 skips the row
    // residual
    float* resid;        // fp32 [M][ld_resid]
    int ld_resid;
    int resid_store;     // EPI_RESID: store C instead of adding it (out = C)
    // argmax / sampling partials, [M][tiles_n]
    float* part_max;
    int* part_idx;
    double* part_sum;    // nullable: sum exp((z - tile max) * inv_T)
    float inv_T;
    float* logits;       // nullable fp32 [M][ld_logits]
    int64_t ld_logits;
};

struct GemmShape {
    int M, N, K;
    int tiles_m, tiles_n, num_kb;
    int m_inner;         // 1: consecutive tiles walk M (share B); 0: walk N (share A)
    int b_begin[3];      // first column served by B tensor map 1, 2, 3
    int nb;              // number of B tensor maps
    int split_b;         // B tile = [BN/2 rows of map 0 ; BN/2 rows of map 1] at rows tn * BN/2
    int a_kb_per_slab;   // > 0: A is a 3-D map [slabs][M][K / slabs]; k-block kb reads slab kb / a_kb_per_slab
    // split K (EPI_RESID only): output tile (tmc, tn) is computed by ksplit
    // consecutive tiles of the sequence, split s over k-blocks
    // [s * kb_split, min(num_kb, (s + 1) * kb_split)), each storing its fp32
    // partial at resid + s * part_stride (a fixed-order reduction follows)
    int ksplit;
    int kb_split;
    int64_t part_stride;
};

// One GEMM of a launch: its tensor maps (A, up to three B segments), shape and
// epilogue.  A launch runs one or two problems with the same tile width,
// epilogue kind and cluster shape as one persistent tile sequence (problem 0's
// tiles first), so that a small problem streams its weights while other SMs
// work on a large one.
struct GemmProb {
    CUtensorMap a;
    CUtensorMap b[3];
    GemmShape sh;
    GemmEpi ep;
};

constexpr int GEMM_BM = 128;
constexpr int GEMM_BK = 64;

// Tile width BN (128, 256, or 512 over a CTA pair only) and cluster shape CM.
// CM = 2: each CTA of the pair holds half of the B tile (BN / 2 rows) per
// stage.  BN = 512: each k-step issues two N = 256 pair products (columns
// 0..255 and 256..511 of the tile), whose B halves interleave: CTA r holds
// tile rows r*128.. and 256 + r*128.. (two 128-row copies); the accumulator
// is the whole of tensor memory (one buffer), drained by eight epilogue
// warps (two per lane quadrant, a column half each).
template <int BN, int CM>
struct GemmCfg {
    static_assert(BN != 512 || CM == 2, "512-wide tiles are pair tiles");
    static constexpr int EW = (BN == 512) ? 8 : 4;                 // epilogue warps
    static constexpr int THREADS = 64 + 32 * EW;                   // producer warp, MMA warp, epilogue warps
    static constexpr int NACC = (BN == 512) ? 1 : 2;               // accumulator buffers
    static constexpr int MMA_N = (BN > 256) ? 256 : BN;            // N of one product
    static constexpr int B_BOX = (BN == 512) ? 128 : BN / CM;      // rows of one B copy
    static constexpr int A_BYTES = GEMM_BM * GEMM_BK * 2;
    static constexpr int B_BYTES = BN / CM * GEMM_BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = (200 * 1024 / STAGE_BYTES) < 8 ? (200 * 1024 / STAGE_BYTES) : 8;
    static constexpr int TMEM_COLS = NACC * BN;
    static constexpr int BAR_BYTES = 256;
    static constexpr int STG_BYTES = 32 * 80;                      // bf16 store staging per epilogue warp
    static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + BAR_BYTES + EW * STG_BYTES;
};

// Tile t of a (tiles_mc x tiles_n) grid of cluster tiles (x ksplit K-splits,
// the splits of one output tile consecutive), in walking order.
__device__ __forceinline__ void tile_coords(const GemmShape& sh, int tiles_mc, int t, int& tmc, int& tn, int& ks) {
    ks = t % sh.ksplit;
    t /= sh.ksplit;
    if (sh.m_inner) { tmc = t % tiles_mc; tn = t / tiles_mc; }
    else            { tn = t % sh.tiles_n; tmc = t / sh.tiles_n; }
}

// k-blocks [kb0, kb1) of split ks
__device__ __forceinline__ void split_range(const GemmShape& sh, int ks, int& kb0, int& kb1) {
    kb0 = ks * sh.kb_split;
    kb1 = kb0 + sh.kb_split < sh.num_kb ? kb0 + sh.kb_split : sh.num_kb;
}

// Stores 64 bytes of each lane's row (lane r: q to dst, when ok) through the
// warp's 2,560-byte staging buffer: rows are written to shared memory one per
// lane (80-byte pitch: each quarter-warp's 16-byte writes hit distinct banks),
// then each store instruction covers 8 rows x 64 contiguous bytes (lane l:
// row l / 4 + 8 i, 16-byte chunk l % 4) instead of 32 rows x 16 bytes, a
// quarter of the L2 write requests.  Every lane of the warp calls it.
__device__ __forceinline__ void store_rows_64B(uint8_t* stg, const uint4 (&q)[4], void* dst, bool ok) {
    const int lane = threadIdx.x & 31;
    uint4* srow = reinterpret_cast<uint4*>(stg + lane * 80);
    #pragma unroll
    for (int k = 0; k < 4; ++k) srow[k] = q[k];
    __syncwarp();
    const int c = lane & 3;
    #pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = (lane >> 2) + 8 * i;
        const unsigned long long p = __shfl_sync(0xFFFFFFFFu, reinterpret_cast<unsigned long long>(dst), r);
        const bool rok = __shfl_sync(0xFFFFFFFFu, ok, r);
        const uint4 val = *reinterpret_cast<const uint4*>(stg + r * 80 + c * 16);
        if (rok) reinterpret_cast<uint4*>(p)[c] = val;
    }
    __syncwarp();   // the buffer is written again by the next call
}

// The four rows whose 16-byte chunks a lane stores in store_rows_64B (rows
// l / 4 + 8 i of the warp's 32): their addresses at the tile's first column,
// 0 for a row that is not stored, gathered once per tile instead of by every
// call.
struct StagedRows {
    unsigned long long p[4];
};

__device__ __forceinline__ StagedRows staged_rows(const void* row_base, bool ok) {
    const int lane = threadIdx.x & 31;
    const unsigned long long mine = ok ? reinterpret_cast<unsigned long long>(row_base) : 0ull;
    StagedRows sr;
    #pragma unroll
    for (int i = 0; i < 4; ++i) sr.p[i] = __shfl_sync(0xFFFFFFFFu, mine, (lane >> 2) + 8 * i);
    return sr;
}

// store_rows_64B with the rows gathered beforehand: each lane's 64 bytes go
// `off` bytes past its row's address.
__device__ __forceinline__ void store_rows_64B_at(uint8_t* stg, const uint4 (&q)[4], const StagedRows& sr,
                                                  uint32_t off) {
    const int lane = threadIdx.x & 31;
    uint4* srow = reinterpret_cast<uint4*>(stg + lane * 80);
    #pragma unroll
    for (int k = 0; k < 4; ++k) srow[k] = q[k];
    __syncwarp();
    const int c = lane & 3;
    #pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = (lane >> 2) + 8 * i;
        const uint4 val = *reinterpret_cast<const uint4*>(stg + r * 80 + c * 16);
        if (sr.p[i]) reinterpret_cast<uint4*>(sr.p[i] + off)[c] = val;
    }
    __syncwarp();   // the buffer is written again by the next call
}

// 32 bf16 values of the lane's row, `col` columns past the row's tile start.
__device__ __forceinline__ void store_rows_bf16x32_at(uint8_t* stg, const float (&v)[32], const StagedRows& sr,
                                                      int col) {
    uint4 q[4];
    #pragma unroll
    for (int k = 0; k < 4; ++k)
        q[k] = make_uint4(pack_bf16(v[8 * k + 0], v[8 * k + 1]), pack_bf16(v[8 * k + 2], v[8 * k + 3]),
                          pack_bf16(v[8 * k + 4], v[8 * k + 5]), pack_bf16(v[8 * k + 6], v[8 * k + 7]));
    store_rows_64B_at(stg, q, sr, (uint32_t)col * 2u);
}

// 32 bf16 values of the lane's row.
__device__ __forceinline__ void store_rows_bf16x32(uint8_t* stg, const float (&v)[32], __nv_bfloat16* dst,
                                                   bool ok) {
    uint4 q[4];
    #pragma unroll
    for (int k = 0; k < 4; ++k)
        q[k] = make_uint4(pack_bf16(v[8 * k + 0], v[8 * k + 1]), pack_bf16(v[8 * k + 2], v[8 * k + 3]),
                          pack_bf16(v[8 * k + 4], v[8 * k + 5]), pack_bf16(v[8 * k + 6], v[8 * k + 7]));
    store_rows_64B(stg, q, dst, ok);
}

// 16 fp32 values of the lane's row, from v[0..16).
__device__ __forceinline__ void store_rows_f32x16(uint8_t* stg, const float* v, float* dst, bool ok) {
    uint4 q[4];
    #pragma unroll
    for (int k = 0; k < 4; ++k)
        q[k] = make_uint4(__float_as_uint(v[4 * k]), __float_as_uint(v[4 * k + 1]), __float_as_uint(v[4 * k + 2]),
                          __float_as_uint(v[4 * k + 3]));
    store_rows_64B(stg, q, dst, ok);
}

// ---------------------------------------------------------------- epilogues

// Where one lane's row of a store-epilogue tile goes: output row, whether it
// is stored, and for a rotary segment the (cos, sin) pairs of its position.
struct StoreRow {
    __nv_bfloat16* out;   // the row's first element of the tile's columns
    const float4* cs;     // rotary segments: (cos, sin) pairs of the row's position
    int hd;               // rotary head dimension (0: no rotary)
    bool ok;
};

template <int BN>
__device__ __forceinline__ StoreRow store_row(const GemmShape& sh, const GemmEpi& ep, int row, int n0, int* ew) {
    int s = 0;
    #pragma unroll
    for (int j = 1; j < 3; ++j)
        if (j < ep.nseg && n0 >= ep.seg[j].n_begin) s = j;
    const GemmSeg sg = ep.seg[s];
    const int64_t orow = (row < sh.M) ? (ep.row_dst ? (int64_t)ep.row_dst[row] : (int64_t)row) : -1;
    StoreRow r;
    r.ok = orow >= 0 && DFL_IN_BOUNDS(ew, orow, sg.rows) && DFL_IN_BOUNDS(ew, n0 - sg.n_begin + BN - 1, sg.ld);
    r.out = reinterpret_cast<__nv_bfloat16*>(sg.out) + (r.ok ? orow : 0) * sg.ld + (n0 - sg.n_begin);
    r.hd = sg.rope ? ep.hd : 0;
    const int pos = !(r.ok && sg.rope) ? 0 : (ep.row_pos ? ep.row_pos[row] : ep.pos_off + row % ep.rows_per_seq);
    r.cs = sg.rope ? reinterpret_cast<const float4*>(ep.rope + (int64_t)pos * ep.hd) : nullptr;
    return r;
}

// (cos, sin) of rotation pairs [c, c + 32) of the row: 256 contiguous bytes.
__device__ __forceinline__ void load_rope32(const StoreRow& r, int c, float4 (&t)[16]) {
    #pragma unroll
    for (int j = 0; j < 16; ++j) t[j] = r.ok ? __ldg(r.cs + c / 2 + j) : make_float4(1.f, 0.f, 1.f, 0.f);
}

// bf16 store of the tile's BN columns of the row, with rotary where the
// segment has it.  t: (cos, sin) of pairs [0, 32), already loaded (the
// kernel loads them before the tile's products finish).
template <int BN>
__device__ __forceinline__ void epi_store(const StoreRow& r, uint32_t tbase, uint8_t* stg, float4 (&t)[16]) {
    const StagedRows sr = staged_rows(r.out, r.ok);
    if (r.hd == 0) {
        #pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
            float v[32];
            tmem_ld32(tbase + c * 32, v);
            store_rows_bf16x32_at(stg, v, sr, c * 32);
        }
        return;
    }
    const int hd = r.hd;
    const int half = hd >> 1;
    // One chunk of 32 rotation pairs at a time: its cos/sin serve every head
    // of the tile.
    #pragma unroll 1
    for (int c = 0; c < half; c += 32) {
        if (c > 0) load_rope32(r, c, t);
        #pragma unroll 1
        for (int h0 = 0; h0 < BN; h0 += hd) {
            float x[32], y[32];
            tmem_ld32(tbase + h0 + c, x);
            tmem_ld32(tbase + h0 + c + half, y);
            #pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float a0 = x[2 * j], b0 = y[2 * j], a1 = x[2 * j + 1], b1 = y[2 * j + 1];
                x[2 * j] = a0 * t[j].x - b0 * t[j].y;
                y[2 * j] = b0 * t[j].x + a0 * t[j].y;
                x[2 * j + 1] = a1 * t[j].z - b1 * t[j].w;
                y[2 * j + 1] = b1 * t[j].z + a1 * t[j].w;
            }
            store_rows_bf16x32_at(stg, x, sr, h0 + c);
            store_rows_bf16x32_at(stg, y, sr, h0 + c + half);
        }
    }
}

// First rotation pair of the chunk that the part-p warp of a 512-wide tile
// works on (see epi_store512).
__device__ __forceinline__ int store512_first_pair(int hd, int part) {
    const int nc = hd / 64;   // chunks of 32 pairs per head
    return nc >= 2 ? part * (nc / 2) * 32 : 0;
}

// bf16 store of a 512-wide tile's row with eight epilogue warps, two per
// lane quadrant.  With rotary heads of 64 or more pairs, the part-p warp
// takes pairs [32 p nc/2, 32 (p + 1) nc/2) of every head in the tile (nc =
// chunks per head), so each warp needs only its own chunks of the row's
// cos/sin, the first of them loaded (in t) before the tile's products end;
// with 32-pair heads, or without rotary, it takes its half of the columns.
// tb: the row's lane quadrant at column 0 of the tile.
__device__ __forceinline__ void epi_store512(const StoreRow& r, uint32_t tb, int part, uint8_t* stg,
                                             float4 (&t)[16]) {
    const StagedRows sr = staged_rows(r.out, r.ok);
    if (r.hd == 0) {
        #pragma unroll 1
        for (int c = 0; c < 8; ++c) {
            float v[32];
            tmem_ld32(tb + part * 256 + c * 32, v);
            store_rows_bf16x32_at(stg, v, sr, part * 256 + c * 32);
        }
        return;
    }
    const int hd = r.hd;
    const int half = hd >> 1;
    const int nc = half / 32;
    auto rotate_store = [&](int h0, int c) {
        float x[32], y[32];
        tmem_ld32(tb + h0 + c, x);
        tmem_ld32(tb + h0 + c + half, y);
        #pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float a0 = x[2 * j], b0 = y[2 * j], a1 = x[2 * j + 1], b1 = y[2 * j + 1];
            x[2 * j] = a0 * t[j].x - b0 * t[j].y;
            y[2 * j] = b0 * t[j].x + a0 * t[j].y;
            x[2 * j + 1] = a1 * t[j].z - b1 * t[j].w;
            y[2 * j + 1] = b1 * t[j].z + a1 * t[j].w;
        }
        store_rows_bf16x32_at(stg, x, sr, h0 + c);
        store_rows_bf16x32_at(stg, y, sr, h0 + c + half);
    };
    if (nc >= 2) {
        #pragma unroll 1
        for (int ci = 0; ci < nc / 2; ++ci) {
            const int c = store512_first_pair(hd, part) + ci * 32;
            if (ci > 0) load_rope32(r, c, t);
            #pragma unroll 1
            for (int h0 = 0; h0 < 512; h0 += hd) rotate_store(h0, c);
        }
    } else {
        #pragma unroll 1
        for (int h0 = part * 256; h0 < part * 256 + 256; h0 += hd) rotate_store(h0, 0);
    }
}

template <int BN>
__device__ __forceinline__ void epi_resid(const GemmShape& sh, const GemmEpi& ep, uint32_t tbase,
                                          int row, int n0, int* ew, int ks, uint8_t* stg) {
    const bool ok = row < sh.M && DFL_IN_BOUNDS(ew, (n0 + BN < sh.N ? n0 + BN : sh.N) - 1, ep.ld_resid);
    const bool rd = !ep.resid_store;
    float* out = ep.resid + ks * sh.part_stride + (int64_t)(ok ? row : 0) * ep.ld_resid + n0;
    #pragma unroll 1
    for (int c = 0; c < BN / 32; c += 2) {
        const bool in0 = ok && n0 + c * 32 < sh.N, in1 = ok && n0 + c * 32 + 32 < sh.N;
        float4* p = reinterpret_cast<float4*>(out + c * 32);
        float4 r[16];
        #pragma unroll
        for (int q = 0; q < 8; ++q) {
            r[q] = (in0 && rd) ? p[q] : make_float4(0.f, 0.f, 0.f, 0.f);
            r[8 + q] = (in1 && rd) ? p[8 + q] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float v[32], w[32];
        tmem_ld32(tbase + c * 32, v);
        tmem_ld32(tbase + c * 32 + 32, w);
        #pragma unroll
        for (int q = 0; q < 8; ++q) {
            r[q].x += v[4 * q + 0]; r[q].y += v[4 * q + 1]; r[q].z += v[4 * q + 2]; r[q].w += v[4 * q + 3];
            r[8 + q].x += w[4 * q + 0]; r[8 + q].y += w[4 * q + 1];
            r[8 + q].z += w[4 * q + 2]; r[8 + q].w += w[4 * q + 3];
        }
        if (!rd) {   // a plain store (split partials, fp32 outputs): staged, 16 columns per call
            const bool u0 = n0 + c * 32 < sh.N, u1 = n0 + c * 32 + 32 < sh.N;   // warp-uniform
            const float* rf = reinterpret_cast<const float*>(r);
            if (u0) {
                store_rows_f32x16(stg, rf, out + c * 32, ok);
                store_rows_f32x16(stg, rf + 16, out + c * 32 + 16, ok);
            }
            if (u1) {
                store_rows_f32x16(stg, rf + 32, out + c * 32 + 32, ok);
                store_rows_f32x16(stg, rf + 48, out + c * 32 + 48, ok);
            }
            continue;
        }
        #pragma unroll
        for (int q = 0; q < 8; ++q) {
            if (in0) p[q] = r[q];
            if (in1) p[8 + q] = r[8 + q];
        }
    }
}

// Partials of BN columns from n0: partial tile pt of npt per row (a 512-wide
// tile writes two, one per epilogue warp of a lane quadrant, so the partials
// are 256 columns wide either way).
template <int BN>
__device__ __forceinline__ void epi_argmax(const GemmShape& sh, const GemmEpi& ep, uint32_t tbase,
                                           int row, int n0, int pt, int npt, int* ew, uint8_t* stg) {
    const bool ok = row < sh.M && n0 < sh.N && DFL_IN_BOUNDS(ew, pt, npt) &&
                    (!ep.logits || DFL_IN_BOUNDS(ew, (n0 + BN < sh.N ? n0 + BN : sh.N) - 1, ep.ld_logits));
    float best = -INFINITY;
    int bidx = n0;
    float* lg = ep.logits ? ep.logits + (int64_t)(ok ? row : 0) * ep.ld_logits : nullptr;
    #pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
        float v[32];
        tmem_ld32(tbase + c * 32, v);
        const int cb = n0 + c * 32;
        #pragma unroll
        for (int j = 0; j < 32; ++j)
            if (cb + j < sh.N && v[j] > best) { best = v[j]; bidx = cb + j; }
        if (lg) {
            if (cb + 32 <= sh.N && (ep.ld_logits & 3) == 0) {   // warp-uniform: staged, 16 columns per call
                store_rows_f32x16(stg, v, lg + cb, ok);
                store_rows_f32x16(stg, v + 16, lg + cb + 16, ok);
            } else if (ok) {
                #pragma unroll
                for (int j = 0; j < 32; ++j) if (cb + j < sh.N) lg[cb + j] = v[j];
            }
        }
    }
    // Sum of exp((z - max) / T) over the tile: each group of four terms is
    // added pairwise in fp32, the groups in fp64 (a quarter of the slow fp64
    // additions; the sum stays within ~1e-7 relative of a term-by-term fp64 one).
    double s = 0.0;
    if (ep.part_sum) {
        #pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
            float v[32];
            tmem_ld32(tbase + c * 32, v);
            const int cb = n0 + c * 32;
            #pragma unroll
            for (int j = 0; j < 32; j += 4) {
                float e[4];
                #pragma unroll
                for (int q = 0; q < 4; ++q) e[q] = cb + j + q < sh.N ? expf((v[j + q] - best) * ep.inv_T) : 0.f;
                s += (double)((e[0] + e[1]) + (e[2] + e[3]));
            }
        }
    }
    if (ok) {
        const int64_t o = (int64_t)row * npt + pt;
        ep.part_max[o] = best;
        ep.part_idx[o] = bidx;
        if (ep.part_sum) ep.part_sum[o] = s;
    }
}

template <int BN>
__device__ __forceinline__ void epi_swiglu(const GemmShape& sh, const GemmEpi& ep, uint32_t tbase, int row, int tn,
                                           int* ew, uint8_t* stg) {
    const bool ok = row < sh.M && DFL_IN_BOUNDS(ew, row, ep.seg[0].rows) &&
                    DFL_IN_BOUNDS(ew, (tn + 1) * (BN / 2) - 1, ep.seg[0].ld);
    const GemmSeg sg = ep.seg[0];
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(sg.out) + (int64_t)(ok ? row : 0) * sg.ld + tn * (BN / 2);
    #pragma unroll 1
    for (int c = 0; c < BN / 64; ++c) {
        float g[32], u[32];
        tmem_ld32(tbase + c * 32, g);
        tmem_ld32(tbase + BN / 2 + c * 32, u);
        #pragma unroll
        for (int j = 0; j < 32; ++j) g[j] = g[j] / (1.f + expf(-g[j])) * u[j];
        store_rows_bf16x32(stg, g, out + c * 32, ok);
    }
}

// ------------------------------------------------------------------- kernel
//
// CM = 1: one CTA per 128-row output tile, cta_group::1 products.
// CM = 2: a cluster of two CTAs owns a 256-row tile (rows of M-tiles 2*tmc
// and 2*tmc + 1) of one N-tile.  One thread of the even CTA issues tcgen05
// cta_group::2 products, which read A's two 128-row halves and B's two
// BN/2-row halves from the two CTAs' shared memory; each SM so loads half of
// the B tile, and receives its own 128 rows of the accumulator in its tensor
// memory.  Both CTAs' copies of a stage complete on the even CTA's `full`
// barrier; the products' completion is committed to both CTAs' `empty` and
// `tfull` barriers; the four epilogue warps of each CTA report a drained
// accumulator on the even CTA's `tempty` barrier.

template <int BN, int EPI, int CM>
__global__ void __launch_bounds__(GemmCfg<BN, CM>::THREADS, 1)
gemm_tc_kernel(const __grid_constant__ GemmProb p0, const __grid_constant__ GemmProb p1, const int nprob,
               const DevErr err) {
    using Cfg = GemmCfg<BN, CM>;
    constexpr int STAGES = Cfg::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * Cfg::A_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(sB + STAGES * Cfg::B_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    uint8_t* stg_base = reinterpret_cast<uint8_t*>(full) + Cfg::BAR_BYTES;   // EW store staging buffers

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    static_assert(EPI != EPI_SWIGLU || Cfg::EW == 4, "this epilogue takes whole tiles");
    static_assert(EPI != EPI_ARGMAX || Cfg::EW == 4 || BN == 512, "argmax partials are 256 columns wide");

    const uint32_t crank = (CM > 1) ? cluster_ctarank() : 0u;
    const bool leader = crank == 0;   // the CTA that issues the products
    const int cid = blockIdx.x / CM, nclusters = gridDim.x / CM;
    // cluster tiles of each problem; tile t of the launch belongs to problem 0 if t < T0
    const int tmc0 = (p0.sh.tiles_m + CM - 1) / CM, tmc1 = (p1.sh.tiles_m + CM - 1) / CM;
    const int T0 = tmc0 * p0.sh.tiles_n * p0.sh.ksplit;
    const int total = T0 + (nprob > 1 ? tmc1 * p1.sh.tiles_n * p1.sh.ksplit : 0);
    auto locate = [&](int t, const GemmProb*& P, int& tmc, int& tn, int& ks) {
        const bool second = t >= T0;
        P = second ? &p1 : &p0;
        tile_coords(P->sh, second ? tmc1 : tmc0, second ? t - T0 : t, tmc, tn, ks);
    };
    // shared::cluster address of barrier `b` of this CTA in CTA `rank`
    auto at = [](const uint64_t* b, uint32_t rank) { return mapa_shared(smem_u32(b), rank); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        for (int a = 0; a < 2; ++a) { mbar_init(&tfull[a], 1); mbar_init(&tempty[a], Cfg::EW * CM); }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        for (int q = 0; q < nprob; ++q) {
            const GemmProb& P = q ? p1 : p0;
            prefetch_tensormap(&P.a);
            for (int j = 0; j < P.sh.nb; ++j) prefetch_tensormap(&P.b[j]);
        }
    }
    if (warp == 1) {
        if (CM > 1) { tmem_alloc_pair(tmem_holder, Cfg::TMEM_COLS); tmem_relinquish_pair(); }
        else { tmem_alloc(tmem_holder, Cfg::TMEM_COLS); tmem_relinquish(); }
    }
    tc_fence_before();
    if (CM > 1) cluster_sync(); else __syncthreads();   // the pair's barriers are initialised before any use
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    grid_dep_begin();   // global memory only from here on

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (each CTA loads its own halves)
            int stage = 0;
            uint32_t phase = 0;
            uint32_t fills = 0;   // bit s: stage s has been filled at least once
            bool aborted = false;
            for (int t = cid; t < total && !aborted; t += nclusters) {
                const GemmProb* P;
                int tmc, tn, ks, kb0, kb1;
                locate(t, P, tmc, tn, ks);
                const GemmShape& sh = P->sh;
                split_range(sh, ks, kb0, kb1);
                const int m0 = (tmc * CM + (int)crank) * GEMM_BM, n0 = tn * BN;
                const CUtensorMap* mb = &P->b[0];
                int nb0 = n0;
                if (sh.nb > 2 && n0 >= sh.b_begin[2]) { mb = &P->b[2]; nb0 = n0 - sh.b_begin[2]; }
                else if (sh.nb > 1 && n0 >= sh.b_begin[1]) { mb = &P->b[1]; nb0 = n0 - sh.b_begin[1]; }
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (*abort_flag || !mbar_wait(&empty[stage], phase ^ 1, err)) { aborted = true; break; }
                    const int ax = (sh.a_kb_per_slab ? kb % sh.a_kb_per_slab : kb) * GEMM_BK;
                    const int az = sh.a_kb_per_slab ? kb / sh.a_kb_per_slab : 0;   // A slab (3-D map)
                    uint8_t* dA = sA + stage * Cfg::A_BYTES;
                    uint8_t* dB = sB + stage * Cfg::B_BYTES;
                    if (CM == 1) {
                        mbar_arrive_expect_tx(&full[stage], Cfg::A_BYTES + Cfg::B_BYTES);
                        if (sh.a_kb_per_slab) tma_load_3d(dA, &P->a, ax, m0, az, &full[stage]);
                        else tma_load_2d(dA, &P->a, ax, m0, &full[stage]);
                        if (sh.split_b) {   // [gate half (map 0) ; up half (map 1)] of the same features
                            const int fr = tn * (BN / 2);
                            tma_load_2d(dB, &P->b[0], kb * GEMM_BK, fr, &full[stage]);
                            tma_load_2d(dB + Cfg::B_BYTES / 2, &P->b[1], kb * GEMM_BK, fr, &full[stage]);
                        } else {
                            tma_load_2d(dB, mb, kb * GEMM_BK, nb0, &full[stage]);
                        }
                    } else {
                        // both CTAs' bytes complete on the leader's barrier
                        const uint32_t fb = at(&full[stage], 0);
                        if (leader) mbar_arrive_expect_tx(&full[stage], 2 * (Cfg::A_BYTES + Cfg::B_BYTES));
                        if (sh.a_kb_per_slab) tma_load_3d_pair(dA, &P->a, ax, m0, az, fb);
                        else tma_load_2d_pair(dA, &P->a, ax, m0, fb);
                        if (sh.split_b) {   // this CTA's half: the gate rows (CTA 0) or the up rows (CTA 1)
                            tma_load_2d_pair(dB, crank ? &P->b[1] : &P->b[0], kb * GEMM_BK, tn * (BN / 2), fb);
                        } else if (BN == 512) {   // this CTA's halves of the two products' B tiles
                            tma_load_2d_pair(dB, mb, kb * GEMM_BK, nb0 + (int)crank * 128, fb);
                            tma_load_2d_pair(dB + Cfg::B_BYTES / 2, mb, kb * GEMM_BK, nb0 + 256 + (int)crank * 128, fb);
                        } else {
                            tma_load_2d_pair(dB, mb, kb * GEMM_BK, nb0 + (int)crank * (BN / 2), fb);
                        }
                    }
                    fills |= 1u << stage;
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
            if (aborted) {
                *abort_flag = 1;
                // Let every copy already issued land before the CTA exits.  The
                // latest fill of stage s has parity phase(s) computed from the
                // position of the ring at exit.  (In a pair the copies complete
                // on the leader's barriers, which count both CTAs' bytes.)
                if (leader) {
                    for (int s = 0; s < STAGES; ++s) {
                        if (!(fills & (1u << s))) continue;
                        const uint32_t par = (s < stage) ? phase : (phase ^ 1);
                        mbar_wait(&full[s], par, err);
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ---------------- MMA issuer
            constexpr uint32_t idesc = idesc_bf16(GEMM_BM * CM, Cfg::MMA_N);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool aborted = false;
            bool issued = false;
            for (int t = cid; t < total && !aborted; t += nclusters) {
                const GemmShape& shp = (t >= T0 ? p1 : p0).sh;
                int kb0, kb1;
                split_range(shp, (t >= T0 ? t - T0 : t) % shp.ksplit, kb0, kb1);
                if (*abort_flag || !mbar_wait(&tempty[acc], acc_phase ^ 1, err)) { aborted = true; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (*abort_flag || !mbar_wait(&full[stage], phase, err)) { aborted = true; break; }
                    tc_fence_after();
                    const uint64_t ad = sw128_desc(smem_u32(sA + stage * Cfg::A_BYTES));
                    const uint64_t bd = sw128_desc(smem_u32(sB + stage * Cfg::B_BYTES));
                    #pragma unroll
                    for (int k = 0; k < GEMM_BK / 16; ++k) {
                        const uint32_t accum = (kb != kb0 || k != 0);
                        if (CM == 1) {
                            mma_bf16(d_tmem, ad + 2 * k, bd + 2 * k, idesc, accum);
                        } else {
                            mma_bf16_pair(d_tmem, ad + 2 * k, bd + 2 * k, idesc, accum);
                            if (BN == 512)   // columns 256..511 from the second B halves (16 KB further)
                                mma_bf16_pair(d_tmem + 256, ad + 2 * k, bd + ((Cfg::B_BYTES / 2) >> 4) + 2 * k, idesc,
                                              accum);
                        }
                    }
                    issued = true;
                    if (CM == 1) {
                        mma_commit(&empty[stage]);
                    } else {   // the stage is free in both CTAs
                        mma_commit_pair_both(&empty[stage]);
                    }
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (aborted) break;
                if (CM == 1) {
                    mma_commit(&tfull[acc]);
                } else {
                    mma_commit_pair_both(&tfull[acc]);
                }
                if (++acc == Cfg::NACC) { acc = 0; acc_phase ^= 1; }
            }
            if (aborted) {
                *abort_flag = 1;
                if (issued) {   // let issued MMAs finish before TMEM is released
                    if (CM == 1) mma_commit(drain);
                    else mma_commit_pair(at(drain, 0));
                    mbar_wait(drain, 0, err);
                }
            }
        }
    } else {
        // ---------------- epilogue warps 2..: TMEM lane quadrant = warp % 4,
        // column part (warp - 2) / 4 of COLS columns
        constexpr int COLS = BN * 4 / Cfg::EW;
        const int q = warp & 3;
        const int part = (warp - 2) >> 2;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = cid; t < total; t += nclusters) {
            if (__any_sync(0xFFFFFFFFu, *abort_flag != 0)) break;
            const GemmProb* P;
            int tmc, tn, ks;
            locate(t, P, tmc, tn, ks);
            const int row = (tmc * CM + (int)crank) * GEMM_BM + q * 32 + lane;
            // Store epilogue: place the row and start loading the first rotary
            // chunk while the tile's products are still running (an L2 round
            // trip under the other SMs' operand traffic).
            StoreRow srow{};
            float4 rope0[16];
            if constexpr (EPI == EPI_STORE && BN == 512) {
                srow = store_row<512>(P->sh, P->ep, row, tn * BN, err.word);
                if (srow.hd) load_rope32(srow, store512_first_pair(srow.hd, part), rope0);
            } else if constexpr (EPI == EPI_STORE) {
                srow = store_row<COLS>(P->sh, P->ep, row, tn * BN + part * COLS, err.word);
                if (srow.hd) load_rope32(srow, 0, rope0);
            }
            const bool ready = mbar_wait(&tfull[acc], acc_phase, err);
            if (!__all_sync(0xFFFFFFFFu, ready)) { *abort_flag = 1; break; }
            tc_fence_after();
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN + part * COLS;
            const int n0 = tn * BN + part * COLS;
            uint8_t* stg = stg_base + (warp - 2) * Cfg::STG_BYTES;
            if constexpr (EPI == EPI_STORE && BN == 512)
                epi_store512(srow, tmem_base + ((uint32_t)(q * 32) << 16), part, stg, rope0);
            else if (EPI == EPI_STORE) epi_store<COLS>(srow, tbase, stg, rope0);
            else if (EPI == EPI_RESID) epi_resid<COLS>(P->sh, P->ep, tbase, row, n0, err.word, ks, stg);
            else if (EPI == EPI_SWIGLU) epi_swiglu<BN>(P->sh, P->ep, tbase, row, tn, err.word, stg);   // one part
            else if (BN == 512)
                epi_argmax<COLS>(P->sh, P->ep, tbase, row, n0, 2 * tn + part, (P->sh.N + 255) / 256, err.word,
                                 stg);
            else epi_argmax<BN>(P->sh, P->ep, tbase, row, tn * BN, tn, P->sh.tiles_n, err.word, stg);
            // every lane's tensor-memory reads are complete before the warp reports
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (CM == 1) mbar_arrive(&tempty[acc]);
                else mbar_arrive_cluster(at(&tempty[acc], 0));
            }
            if (++acc == Cfg::NACC) { acc = 0; acc_phase ^= 1; }
        }
    }
    __syncthreads();
    if (CM > 1) cluster_sync();   // neither CTA's tensor memory is read or written any more
    if (warp == 1) {
        tc_fence_after();
        if (CM > 1) tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
        else tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
    if (CM > 1) cluster_sync();   // no CTA leaves while a peer may still arrive on its barriers
}

}  // namespace dfl
