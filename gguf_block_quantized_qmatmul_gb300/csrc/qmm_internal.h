// qmm_internal.h -- launchers shared between the translation units of the library.
#pragma once

#include <cuda_runtime.h>

#include "qmm_dmma.cuh"
#include "qmm_gemv.cuh"
#include "qmm_tc.cuh"
#include "qmm_tcx.cuh"
#include "qmm_stream.cuh"

namespace qmm {

cudaError_t launch_quantize(int type, const float* x, long long rows, long long K, void* out, cudaStream_t s);
cudaError_t launch_dequantize(int type, const void* q, long long rows, long long K, float* out, cudaStream_t s);
cudaError_t launch_splitk_reduce(const float* partial, long long n, int ks, float* y, cudaStream_t s);
cudaError_t launch_stream_q8_0(int am, int epi, const StreamPlan& plan, int smem_max, cudaStream_t s);
cudaError_t launch_stream_q4_k(int am, int epi, const StreamPlan& plan, int smem_max, cudaStream_t s);
cudaError_t launch_stream_q4_0(int am, int epi, const StreamPlan& plan, int smem_max, cudaStream_t s);
cudaError_t launch_stream_q5_0(int am, int epi, const StreamPlan& plan, int smem_max, cudaStream_t s);
cudaError_t launch_stream_q6_k(int am, int epi, const StreamPlan& plan, int smem_max, cudaStream_t s);
cudaError_t launch_gemv_q8_0(int epi, const GemvPlan& plan, int smem_max, cudaStream_t s);
cudaError_t launch_gemv_q4_k(int epi, const GemvPlan& plan, int smem_max, cudaStream_t s);
cudaError_t launch_dmma(int wt, int am, int epi, const DmmaPlan& plan, int smem_max, cudaStream_t s);
cudaError_t launch_dmma_x_0(int wt, int am, int epi, const DmmaPlan& plan, int smem_max, cudaStream_t s);
cudaError_t launch_dmma_q6_k(int am, int epi, const DmmaPlan& plan, int smem_max, cudaStream_t s);
cudaError_t launch_dmma_prep(int wt, int am, const DmmaPlan& plan, void* ext, cudaStream_t s);
cudaError_t launch_tc(int wt, const TcPlan& plan, const void* wq, const float* x, void* ws, float* y, int smem_max,
                      cudaStream_t s);
cudaError_t launch_tcx(int wt, const TcxPlan& plan, const void* wq, const float* x, void* ws, float* y, int smem_max, cudaStream_t s);
cudaError_t launch_tcx_f32(int wt, const TcxPlan& plan, const void* wq, const float* x, void* ws, float* y, int smem_max,
                           cudaStream_t s);
// A 2-D tensor map (rows of `inner` elements, `row_bytes` apart) with a box
// of box_inner x box_outer elements; false when the driver refuses it.
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, unsigned long long inner, unsigned long long outer,
              unsigned long long row_bytes, unsigned box_inner, unsigned box_outer, CUtensorMapSwizzle swz);

// largest activation batch served by the per-thread dp4a GEMV (int8_act,
// Q8_0 weights only); larger decode batches, Q4_K weights and every f32_act
// decode batch up to 8 use the 16-row-tile tensor-core kernel
constexpr int kGemvMaxM = 1;
constexpr int kDecodeMaxM = 8;

// Raise a kernel's dynamic shared-memory limit once per device.
template <typename F>
inline cudaError_t ensure_smem(F* kernel, int smem_max, unsigned long long& done_mask) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (done_mask & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max);
    if (e == cudaSuccess) done_mask |= bit;
    return e;
}

// Launch with programmatic stream serialization: the grid may be scheduled
// once the previous grid in the stream has triggered (griddepcontrol
// .launch_dependents) instead of once it has completed.  Every kernel
// launched this way executes griddepcontrol.wait before it reads what an
// earlier grid writes, writes what an earlier grid reads, or starts a
// bounded wait that needs such data; only constant inputs (the weights) are
// read before it.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem, cudaStream_t s,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace qmm

// many independent small matmuls in one launch (uses ensure_smem above)
#include "qmm_batch.cuh"
