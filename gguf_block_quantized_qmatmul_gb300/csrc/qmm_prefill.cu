// qmm_prefill.cu -- host side of the prefill GEMM: tensor maps, launches.
#include <cudaTypedefs.h>

#include "qmm_internal.h"

namespace qmm {
namespace {

unsigned long long g_smem_done[2];

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

bool make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, unsigned long long inner, unsigned long long outer,
              unsigned long long row_bytes, unsigned box_inner, unsigned box_outer, CUtensorMapSwizzle swz) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_prefill(int am, const PrefillPlan& pl, const void* wq, const float* x, void* ws, int smem_max,
                           cudaStream_t s) {
    const PrefillParams& p = pl.p;
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    __half* a = reinterpret_cast<__half*>(wsb + pl.ws_a);
    __half* a2 = reinterpret_cast<__half*>(wsb + pl.ws_a2);
    float* sc = reinterpret_cast<float*>(wsb + pl.ws_s);
    // 1. the activation operand
    if (am == A_INT8) {
        const long long n = (long long)p.M * (p.K / 32);
        prefill_act_kernel<A_INT8><<<(unsigned)((n + 255) / 256), 256, 0, s>>>(x, p.M, p.K, a, a2, sc);
    } else {
        prefill_act_kernel<A_F32><<<p.M, 256, 0, s>>>(x, p.M, p.K, a, a2, sc);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // 2. tensor maps: raw weight rows as uint16, f16 activation planes (128B swizzle), f32 scales
    CUtensorMap tw, ta, ta2, ts;
    const unsigned long long rb = (unsigned long long)p.K / 32 * 34;
    if (!make_map(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT16, wq, rb / 2, p.N, rb, kPfWRow / 2, kPfBN, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a, p.K, p.M, (unsigned long long)p.K * 2, 64, p.bm,
                  CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    if (am == A_F32) {
        if (!make_map(&ta2, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a2, p.K, p.M, (unsigned long long)p.K * 2, 64, p.bm,
                      CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
        ts = ta;
    } else {
        if (!make_map(&ts, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, sc, p.K / 32, p.M, (unsigned long long)p.K / 8, 8, p.bm,
                      CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
        ta2 = ta;
    }
    PrefillParams pp = p;
    pp.rs = sc;
    // 3. the GEMM
    if (am == A_INT8) {
        e = ensure_smem(qmm_prefill_kernel<A_INT8>, smem_max, g_smem_done[0]);
        if (e != cudaSuccess) return e;
        qmm_prefill_kernel<A_INT8><<<pl.grid, (kPfWarps + 1) * 32, pl.smem, s>>>(tw, ta, ta2, ts, pp);
    } else {
        e = ensure_smem(qmm_prefill_kernel<A_F32>, smem_max, g_smem_done[1]);
        if (e != cudaSuccess) return e;
        qmm_prefill_kernel<A_F32><<<pl.grid, (kPfWarps + 1) * 32, pl.smem, s>>>(tw, ta, ta2, ts, pp);
    }
    return cudaGetLastError();
}

}  // namespace qmm
