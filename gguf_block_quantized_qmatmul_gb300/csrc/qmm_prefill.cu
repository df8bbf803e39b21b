// qmm_prefill.cu -- host side of the CPU form's prefill GEMM (Q8_0): the
// activation operand, tensor maps, launches.
#include "qmm_internal.h"

namespace qmm {
namespace {
unsigned long long g_pf_smem_done;
}  // namespace

cudaError_t launch_prefill(const PrefillPlan& pl, const void* wq, const float* x, void* ws, float* y, int smem_max,
                           cudaStream_t s) {
    const PrefillParams& p = pl.p;
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    __half* a = reinterpret_cast<__half*>(wsb + pl.ws_a);
    float* sc = reinterpret_cast<float*>(wsb + pl.ws_s);
    // 1. the activation operand: f16 codes and f32 block scales
    const long long n = (long long)p.M * (p.K / 32);
    prefill_act_kernel<T_Q8_0><<<(unsigned)((n + 255) / 256), 256, 0, s>>>(x, p.M, p.K, a, sc);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // 2. tensor maps: raw weight rows as uint16, the f16 codes (128B swizzle), the scales
    CUtensorMap tw, ta, ts;
    const unsigned long long rb = (unsigned long long)p.K / 32 * 34;
    if (!make_map(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT16, wq, rb / 2, p.N, rb, kPfWRow / 2, kPfBN, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a, p.K, p.M, (unsigned long long)p.K * 2, 64, p.bm,
                  CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&ts, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, sc, p.K / 32, p.M, (unsigned long long)p.K / 8, 8, p.bm,
                  CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    PrefillParams pp = p;
    pp.y = y;
    // 3. the GEMM
    e = ensure_smem(qmm_prefill_kernel<T_Q8_0>, smem_max, g_pf_smem_done);
    if (e != cudaSuccess) return e;
    qmm_prefill_kernel<T_Q8_0><<<pl.grid, (kPfWarps + 1) * 32, pl.smem, s>>>(tw, ta, ts, pp);
    return cudaGetLastError();
}

}  // namespace qmm
