// qmm_tcx.cu -- host side of the exact tcgen05 prefill GEMM (the CPU form):
// activation operand preparation, tensor maps, launches.
#include "qmm_internal.h"

namespace qmm {

namespace {
unsigned long long g_tcx_smem_done;
}

cudaError_t launch_tcx(const TcxPlan& pl, const void* wq, const float* x, void* ws, float* y, int smem_max, cudaStream_t s) {
    const TcxParams& p0 = pl.p;
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    __half* codes = reinterpret_cast<__half*>(wsb + pl.ws_codes);
    float* scales = reinterpret_cast<float*>(wsb + pl.ws_scales);
    // 1. the activation operand: f16 codes [M][K], f(d_a) block-major [K / 32][mp]
    const long long items = (long long)p0.M * (p0.K / 32);
    tcx_act_kernel<T_Q8_0><<<(unsigned)((items + 255) / 256), 256, 0, s>>>(x, p0.M, p0.K, pl.mp, codes, scales);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // 2. tensor maps: raw weight rows as uint16 (128 rows x 272 B); activation codes,
    //    32 K x 128 rows, 64-byte swizzle; activation scales, 128 rows x 8 blocks
    CUtensorMap tw, ta, ts;
    const unsigned long long rb = (unsigned long long)p0.K / 32 * 34;
    if (!make_map(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT16, wq, rb / 2, p0.N, rb, kTxRaw / 2, kTxW, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, codes, p0.K, p0.M, (unsigned long long)p0.K * 2, 32, kTxX,
                  CU_TENSOR_MAP_SWIZZLE_64B) ||
        !make_map(&ts, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, scales, pl.mp, p0.K / 32, (unsigned long long)pl.mp * 4, kTxX, 8,
                  CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    TcxParams p = p0;
    p.y = y;
    // 3. the GEMM, a programmatic dependent of the preparation
    auto* k = qmm_tcx_kernel<T_Q8_0>;
    e = ensure_smem(k, smem_max, g_tcx_smem_done);
    if (e != cudaSuccess) return e;
    return launch_pdl(k, (unsigned)pl.grid, kTxThreads, pl.smem, s, tw, ta, ts, p);
}

}  // namespace qmm
