// Host-side internals shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "../../include/dfl.h"
#include "gemm_tc.cuh"

namespace dfl {

// Per-device context: error-word address, SM count, cached attributes.
// Everything here belongs to one CUDA context of the device (its id in
// ctx_id); when another context becomes current on the device (after
// cudaDeviceReset, or a context of the caller's own), the entry is set up
// again for it before any use.
struct DeviceCtx {
    int device = -1;
    int sm_count = 0;
    std::atomic<uint64_t> ctx_id{0};   // unique id of the CUDA context this entry was set up in
    int* err_word = nullptr;       // device address of this device's error word
    // max-dynamic-smem attribute set (atomic: calls may come from several
    // host threads; setting it twice is harmless)
    std::atomic<bool> gemm_attr_set[19] = {};   // gemm instantiations
    std::atomic<bool> mix_attr_set{false};
    std::atomic<bool> attn_attr_set[4] = {};    // tcgen05 attention: head dim 64 / 128, M = 64 / 128 products
    // Host-input draft step: a copy stream and events, created on first use.
    // host_mu is held while a call issues its work: the events are shared, and
    // a wait must see the record its own call made.
    static constexpr int MAX_H_CHUNKS = 16;
    std::mutex host_mu;
    cudaStream_t copy_st = nullptr;
    cudaEvent_t copy_ev[MAX_H_CHUNKS + 1] = {};
};

// Context of the current device (initialised on first use); nullptr if no
// usable device.
DeviceCtx* current_ctx();
DevErr dev_err(DeviceCtx* ctx);
uint64_t wait_limit_ns();

inline dfl_status cuda_status(cudaError_t e) { return e == cudaSuccess ? DFL_OK : DFL_ERR_CUDA; }
inline dfl_status last_launch() { return cuda_status(cudaGetLastError()); }

// Every kernel launch of the library goes through launch_pdl: programmatic
// stream serialisation lets the grid start while the previous grid in the
// stream finishes (each kernel waits for it in grid_dep_begin before touching
// global memory).  DFL_PDL=0 in the environment launches plainly instead.
bool pdl_on();

template <typename... P, typename... A>
inline dfl_status launch_pdl(void (*kern)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             A&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl_on() ? 1 : 0;
    return cuda_status(cudaLaunchKernelEx(&cfg, kern, static_cast<A&&>(args)...));
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// Row counts index TMA coordinates and GEMM extents, which are 32-bit.
inline bool rows_fit(int64_t rows) { return rows < ((int64_t)1 << 31); }

// --------------------------------------------------------------- tracing --

// NVTX range around one C-ABI call: the calls show as named ranges in Nsight
// timelines and ncu can select kernels by the call that launched them
// (--nvtx --nvtx-include).  A few nanoseconds when no tool is attached.
class ApiRange {
public:
    explicit ApiRange(const char* name) { nvtxRangePushA(name); }
    ~ApiRange() { nvtxRangePop(); }
    ApiRange(const ApiRange&) = delete;
    ApiRange& operator=(const ApiRange&) = delete;
};


// Records a CUDA event pair around the launches in its scope when tracing is
// on (dfl_profile_enable); a no-op otherwise.
class ProfScope {
public:
    ProfScope(const char* name, cudaStream_t st);
    ~ProfScope();
    ProfScope(const ProfScope&) = delete;
    ProfScope& operator=(const ProfScope&) = delete;
private:
    int slot_ = -1;
    cudaStream_t st_;
};

// ---------------------------------------------------------------- GEMM --

struct GemmArgs {
    const void* A;          // bf16 [M][K]
    int M, K;
    const void* B[3];       // bf16 [n_b][K] each; B[j] serves columns from b_begin[j]
    int b_rows[3];
    int b_begin[3];
    int nb;
    int N;                  // total columns
    int m_inner;
    int bn;                 // 128, 256 or 512 (pair tiles; store, residual or light argmax epilogue); 0: chosen
    int epi;                // EpiKind
    GemmEpi ep;
    const char* tag;        // name in kernel traces
    int split_b;            // EPI_SWIGLU: B tile halves from maps 0 (gate) and 1 (up); N = 2F
    // a_slabs > 0: A is a_slabs slabs of [M][K / a_slabs], slab i at element
    // i * a_slab_stride, read as one [M][K] operand (slab i supplies columns
    // i * K / a_slabs ...); K / a_slabs a multiple of 64
    int a_slabs;
    int64_t a_slab_stride;
    // EPI_RESID with a single M-tile: a buffer for fp32 partials of a K-split
    // (nullable: no split)
    float* split_part;
    size_t split_part_bytes;
};

dfl_status gemm_tc(DeviceCtx* ctx, const GemmArgs& g, cudaStream_t st);
// Two independent GEMMs in one persistent launch (problem g0's tiles first),
// traced as `tag`; two launches when no tile width suits both.
dfl_status gemm_tc2(DeviceCtx* ctx, const GemmArgs& g0, const GemmArgs& g1, const char* tag, cudaStream_t st);

// The driver's cuTensorMapEncodeTiled (resolved once; nullptr if unavailable).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn();

// fp32 CUDA-core GEMM: C = A[M][K] * B[N][K]^T; mode 0 store (ldc), 1 accumulate.
dfl_status gemm_f32(const float* A, const float* B, float* C, int M, int N, int K, int ldc, int accumulate,
                    cudaStream_t st);
// Same with row strides lda (A) and ldb (B) in elements.
dfl_status gemm_f32_ld(const float* A, int64_t lda, const float* B, int64_t ldb, float* C, int M, int N, int K,
                       int ldc, int accumulate, cudaStream_t st);

}  // namespace dfl
