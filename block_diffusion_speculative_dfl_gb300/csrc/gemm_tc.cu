// Host launcher of the tcgen05 GEMM: TMA descriptors, tile grid, launch.
#include <mutex>

#include "gemm_tc.cuh"
#include "internal.h"

namespace dfl {

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

namespace {

// bf16 [rows][K] row-major, box = box_rows x 64 elements, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int rows, int K, int box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {(cuuint32_t)GEMM_BK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 [slabs][rows][w] with slab stride `sstride` elements, box = box_rows x 64
// elements of one slab, 128-byte swizzle (the same shared-memory tile as the
// 2-D map's).
bool make_map_3d(CUtensorMap* m, const void* base, int rows, int w, int slabs, int64_t sstride, int box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)w, (cuuint64_t)rows, (cuuint64_t)slabs};
    cuuint64_t strides[2] = {(cuuint64_t)w * 2, (cuuint64_t)sstride * 2};
    cuuint32_t box[3] = {(cuuint32_t)GEMM_BK, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, int EPI, int CM>
dfl_status launch(DeviceCtx* ctx, const GemmProb& p0, const GemmProb& p1, int nprob, const char* tag,
                  cudaStream_t st, int slot) {
    auto kern = gemm_tc_kernel<BN, EPI, CM>;
    if (!ctx->gemm_attr_set[slot]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, GemmCfg<BN, CM>::SMEM) !=
            cudaSuccess)
            return DFL_ERR_CUDA;
        if (CM > 1 && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 0) != cudaSuccess)
            return DFL_ERR_CUDA;
        ctx->gemm_attr_set[slot] = true;
    }
    int tiles = ((p0.sh.tiles_m + CM - 1) / CM) * p0.sh.tiles_n * p0.sh.ksplit;
    if (nprob > 1) tiles += ((p1.sh.tiles_m + CM - 1) / CM) * p1.sh.tiles_n * p1.sh.ksplit;
    const int max_clusters = ctx->sm_count / CM;
    const int grid = (tiles < max_clusters ? tiles : max_clusters) * CM;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(GemmCfg<BN, CM>::THREADS);
    cfg.dynamicSmemBytes = GemmCfg<BN, CM>::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CM;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // waits in grid_dep_begin
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_on() ? 2 : 1;
    const DevErr err = dev_err(ctx);
    ProfScope ps(tag ? tag : "gemm_tc", st);
    if (cudaLaunchKernelEx(&cfg, kern, p0, p1, nprob, err) != cudaSuccess) return DFL_ERR_CUDA;
    return last_launch();
}

template <int BN, int EPI>
dfl_status launch_cm(DeviceCtx* ctx, const GemmProb& p0, const GemmProb& p1, int nprob, const char* tag,
                     cudaStream_t st, int slot, int cm) {
    if (cm == 2) return launch<BN, EPI, 2>(ctx, p0, p1, nprob, tag, st, slot + 8);
    return launch<BN, EPI, 1>(ctx, p0, p1, nprob, tag, st, slot);
}

// Relative time of one tile of width bn with clusters of cm: its products
// take ~bn units of tensor time and it reads (128 cm + bn) rows of operands
// from L2 per k-block; at ~12 TB/s of L2-to-SM reads a 256-row pair tile of
// width 256 is held to ~0.81 of the tensor rate, so the L2 term weighs 0.62.
double tile_cost(int bn, int cm) {
    const double l2 = 0.62 * (GEMM_BM * cm + bn);
    return bn > l2 ? bn : l2;
}

// Tile widths a problem takes: 512 only as pair tiles with the rotary-store
// or residual epilogue, or with the argmax epilogue when it stores neither
// logits nor sampling sums (the drain a 512-wide tile exposes stays short);
// every B segment must start on a tile boundary; a width the caller fixed is
// the only one.
bool width_ok(const GemmArgs& g, int bn, int cm) {
    const bool light_argmax = g.epi == EPI_ARGMAX && !g.ep.logits && !g.ep.part_sum;
    if (bn == 512 && (cm != 2 || (g.epi != EPI_STORE && g.epi != EPI_RESID && !light_argmax) || g.split_b))
        return false;
    if (g.bn != 0) return g.bn == bn;
    if (g.split_b) return (g.N / 2) % (bn / 2) == 0;
    for (int j = 0; j < g.nb; ++j) if (g.b_begin[j] % bn != 0) return false;
    return true;
}

}  // namespace

// Tile width for bn == 0: the one that minimises (rounds of cluster tiles
// over the persistent grid) x (tile width) -- i.e. the time of the busiest
// SM when every tile costs ~its width -- preferring 256 on ties; 256 needs
// every B segment to start on a 256-column boundary.
static int pick_bn(const GemmArgs& g, int sm_count) {
    if (g.split_b) return (g.N / 2) % 128 == 0 ? 256 : 128;
    const int tiles_m = (g.M + GEMM_BM - 1) / GEMM_BM;
    const int cm = tiles_m >= 2 ? 2 : 1;
    const int tiles_mc = (tiles_m + cm - 1) / cm;
    const int clusters = sm_count / cm;
    // the busiest cluster's rounds of tiles times the cost of one tile
    auto cost = [&](int bn) {
        const int tiles = tiles_mc * ((g.N + bn - 1) / bn);
        return (double)((tiles + clusters - 1) / clusters) * tile_cost(bn, cm);
    };
    int best = 128;
    for (int bn : {256, 512})
        if (width_ok(g, bn, cm) && cost(bn) <= cost(best)) best = bn;
    return best;
}

// Validated problem of one GEMM for tile width bn and cluster size cm.
static dfl_status build_prob(const GemmArgs& g, int cm, GemmProb& P) {
    if (g.M <= 0 || g.N <= 0 || g.K <= 0) return DFL_ERR_INVALID_ARG;
    if (g.K % 8 != 0 || !aligned16(g.A)) return DFL_ERR_MISALIGNED;
    if (g.bn != 128 && g.bn != 256 && g.bn != 512) return DFL_ERR_UNSUPPORTED_SHAPE;
    if (g.bn == 512 && !width_ok(g, 512, cm)) return DFL_ERR_UNSUPPORTED_SHAPE;
    if (g.nb < 1 || g.nb > 3) return DFL_ERR_INVALID_ARG;
    GemmShape& sh = P.sh;
    sh = GemmShape{};
    sh.M = g.M; sh.N = g.N; sh.K = g.K;
    sh.tiles_m = (g.M + GEMM_BM - 1) / GEMM_BM;
    sh.tiles_n = (g.N + g.bn - 1) / g.bn;
    sh.num_kb = (g.K + GEMM_BK - 1) / GEMM_BK;
    sh.m_inner = g.m_inner;
    sh.nb = g.nb;
    sh.split_b = g.split_b;
    sh.ksplit = 1;
    sh.kb_split = sh.num_kb;
    sh.part_stride = 0;
    if (g.split_b && (g.nb != 2 || (g.N / 2) % (g.bn / 2) != 0)) return DFL_ERR_UNSUPPORTED_SHAPE;
    if (g.a_slabs > 0) {
        const int w = g.K / g.a_slabs;
        if (g.K % g.a_slabs != 0 || w % GEMM_BK != 0) return DFL_ERR_UNSUPPORTED_SHAPE;
        if ((g.a_slab_stride * 2) % 16 != 0 || g.a_slab_stride < (int64_t)g.M * w) return DFL_ERR_MISALIGNED;
        if (!make_map_3d(&P.a, g.A, g.M, w, g.a_slabs, g.a_slab_stride, GEMM_BM)) return DFL_ERR_CUDA;
        sh.a_kb_per_slab = w / GEMM_BK;
    } else if (!make_map(&P.a, g.A, g.M, g.K, GEMM_BM)) {
        return DFL_ERR_CUDA;
    }
    for (int j = 0; j < 3; ++j) {
        const int jj = j < g.nb ? j : 0;
        if (!aligned16(g.B[jj])) return DFL_ERR_MISALIGNED;
        // every tile of BN columns must come from one B map
        if (j < g.nb && !g.split_b && (g.b_begin[j] % g.bn != 0)) return DFL_ERR_UNSUPPORTED_SHAPE;
            const int box = g.split_b ? g.bn / 2 : (g.bn == 512 ? 128 : g.bn / cm);   // rows of one B copy
        if (!make_map(&P.b[j], g.B[jj], g.b_rows[jj], g.K, box)) return DFL_ERR_CUDA;
        sh.b_begin[j] = g.b_begin[jj];
    }
    P.ep = g.ep;
    return DFL_OK;
}

static dfl_status launch_probs(DeviceCtx* ctx, const GemmProb& p0, const GemmProb& p1, int nprob, int bn, int epi,
                               int cm, const char* tag, cudaStream_t st) {
    if (bn == 512) {   // pair tiles only (checked when the problem was built)
        if (epi == EPI_STORE) return launch<512, EPI_STORE, 2>(ctx, p0, p1, nprob, tag, st, 16);
        if (epi == EPI_ARGMAX) return launch<512, EPI_ARGMAX, 2>(ctx, p0, p1, nprob, tag, st, 18);
        return launch<512, EPI_RESID, 2>(ctx, p0, p1, nprob, tag, st, 17);
    }
    const int slot = (bn == 256 ? 0 : 4) + epi;
    if (bn == 256) {
        if (epi == EPI_STORE) return launch_cm<256, EPI_STORE>(ctx, p0, p1, nprob, tag, st, slot, cm);
        if (epi == EPI_RESID) return launch_cm<256, EPI_RESID>(ctx, p0, p1, nprob, tag, st, slot, cm);
        if (epi == EPI_SWIGLU) return launch_cm<256, EPI_SWIGLU>(ctx, p0, p1, nprob, tag, st, slot, cm);
        return launch_cm<256, EPI_ARGMAX>(ctx, p0, p1, nprob, tag, st, slot, cm);
    }
    if (epi == EPI_STORE) return launch_cm<128, EPI_STORE>(ctx, p0, p1, nprob, tag, st, slot, cm);
    if (epi == EPI_RESID) return launch_cm<128, EPI_RESID>(ctx, p0, p1, nprob, tag, st, slot, cm);
    if (epi == EPI_SWIGLU) return launch_cm<128, EPI_SWIGLU>(ctx, p0, p1, nprob, tag, st, slot, cm);
    return launch_cm<128, EPI_ARGMAX>(ctx, p0, p1, nprob, tag, st, slot, cm);
}

// out[m][n] += sum over s of part[s][m][n], s in order (one thread per four
// columns; N a multiple of 4).
__global__ void splitk_reduce_kernel(const float* part, int S, int64_t stride, int M, int N, float* out,
                                     int64_t ld) {
    grid_dep_begin();
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;   // float4 index over M x N
    const int64_t per_row = N / 4;
    if (i >= (int64_t)M * per_row) return;
    const int64_t m = i / per_row, c = (i % per_row) * 4;
    float4 acc = *reinterpret_cast<const float4*>(part + m * N + c);
    for (int s = 1; s < S; ++s) {
        const float4 v = *reinterpret_cast<const float4*>(part + s * stride + m * N + c);
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    float4* o = reinterpret_cast<float4*>(out + m * ld + c);
    float4 r = *o;
    r.x += acc.x; r.y += acc.y; r.z += acc.z; r.w += acc.w;
    *o = r;
}

// K-splits of a residual GEMM that leaves SMs idle (few output tiles, each
// streaming a long K): enough splits to spread the tiles' CTAs over the SMs,
// at least eight k-blocks each; 1 when the GEMM does not qualify or the
// partials do not fit the caller's buffer.
static int pick_ksplit(const GemmArgs& g, int sm_count) {
    if (g.epi != EPI_RESID || !g.split_part || g.ep.resid_store || g.N % 4 != 0) return 1;
    const int tm = (g.M + GEMM_BM - 1) / GEMM_BM;
    const int cm = tm >= 2 ? 2 : 1;
    const int tiles = ((tm + cm - 1) / cm) * ((g.N + g.bn - 1) / g.bn) * cm;   // CTAs of the unsplit GEMM
    const int num_kb = (g.K + GEMM_BK - 1) / GEMM_BK;
    int s = sm_count / tiles;
    s = s < 8 ? s : 8;
    s = s < num_kb / 8 ? s : num_kb / 8;
    while (s > 1 && (size_t)s * g.M * g.N * sizeof(float) > g.split_part_bytes) --s;
    return s > 1 ? s : 1;
}

dfl_status gemm_tc(DeviceCtx* ctx, const GemmArgs& g_in, cudaStream_t st) {
    GemmArgs g = g_in;
    if (g.bn == 0) g.bn = pick_bn(g, ctx->sm_count);
    // Pair the M-tiles of each N-tile over two SMs (a 256-row tile of
    // cta_group::2 products) when there is more than one M-tile.
    const int cm = (g.M + GEMM_BM - 1) / GEMM_BM >= 2 ? 2 : 1;
    // A residual GEMM whose partials have room splits K over pair tiles 256
    // wide (measured: the Qwen and GPT-OSS output projections, 37 -> 27 and
    // 36 -> 20 us plus an 8-10 us reduction).
    if (g.epi == EPI_RESID && g.split_part && cm == 2 && g.N % 256 == 0 && g_in.bn == 0) g.bn = 256;
    const int ksplit = pick_ksplit(g, ctx->sm_count);
    GemmArgs gk = g;
    if (ksplit > 1) {   // each split stores its fp32 partial; a fixed-order sum then adds them to the output
        gk.ep.resid = g.split_part;
        gk.ep.ld_resid = g.N;
        gk.ep.resid_store = 1;
    }
    GemmProb P;
    dfl_status rc = build_prob(gk, cm, P);
    if (rc != DFL_OK) return rc;
    if (ksplit > 1) {
        P.sh.ksplit = ksplit;
        P.sh.kb_split = (P.sh.num_kb + ksplit - 1) / ksplit;
        P.sh.part_stride = (int64_t)g.M * g.N;
    }
    if ((rc = launch_probs(ctx, P, P, 1, g.bn, g.epi, cm, g.tag, st)) != DFL_OK || ksplit == 1) return rc;
    ProfScope ps("splitk_reduce", st);
    const int64_t n4 = (int64_t)g.M * (g.N / 4);
    launch_pdl(splitk_reduce_kernel, (unsigned)((n4 + 255) / 256), 256, 0, st, g.split_part, ksplit,
               (int64_t)g.M * g.N, g.M, g.N, g.ep.resid, g.ep.ld_resid);
    return last_launch();
}

// Two independent GEMMs in one launch (same epilogue kind; problem 0's tiles
// first), with a tile width and cluster shape both accept; two launches when
// there is none.
dfl_status gemm_tc2(DeviceCtx* ctx, const GemmArgs& g0_in, const GemmArgs& g1_in, const char* tag, cudaStream_t st) {
    GemmArgs g0 = g0_in, g1 = g1_in;
    // Pair tiles even when a problem has a single M-tile (the block projection
    // of a small batch): the odd CTA of its tiles holds no rows (zero-filled
    // A, nothing stored), but each SM then streams half of the B tile
    // (measured at batch 1: 39.2 -> 37.2 us; batch 2: 65.3 -> 57.8 us).
    const int cm = 2;
    // One tile width for both: of the widths both take, the one with the
    // smallest (rounds of the joint tile sequence) x (cost of a tile).
    const int clusters = ctx->sm_count / cm;
    auto tiles_of = [&](const GemmArgs& g, int bn) {
        return ((g.M + GEMM_BM - 1) / GEMM_BM + cm - 1) / cm * ((g.N + bn - 1) / bn);
    };
    int bn = 0;
    double best = 0.0;
    for (int w : {128, 256, 512}) {
        if (!width_ok(g0, w, cm) || !width_ok(g1, w, cm)) continue;
        const int tiles = tiles_of(g0, w) + tiles_of(g1, w);
        const double c = (double)((tiles + clusters - 1) / clusters) * tile_cost(w, cm);
        if (bn == 0 || c <= best) { bn = w; best = c; }
    }
    if (bn == 0 || g0.epi != g1.epi) {
        dfl_status rc = gemm_tc(ctx, g0, st);
        return rc != DFL_OK ? rc : gemm_tc(ctx, g1, st);
    }
    g0.bn = g1.bn = bn;
    GemmProb P0, P1;
    dfl_status rc = build_prob(g0, cm, P0);
    if (rc == DFL_OK) rc = build_prob(g1, cm, P1);
    if (rc != DFL_OK) return rc;
    return launch_probs(ctx, P0, P1, 2, bn, g0.epi, cm, tag, st);
}

}  // namespace dfl
