// qmm_tc.cu -- host side of the tcgen05 prefill GEMM (the Metal form): tensor
// maps, launches; and the 2-D tensor-map helper both prefill GEMMs use.
#include <cudaTypedefs.h>

#include "qmm_internal.h"

namespace qmm {
namespace {

unsigned long long g_tc_smem_done[5];

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

template <int WT>
cudaError_t tc_go(const TcPlan& pl, const void* wq, const float* x, void* ws, float* y, int smem_max, cudaStream_t s) {
    const TcParams& p0 = pl.p;
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    __half* ahi = reinterpret_cast<__half*>(wsb + pl.ws_ahi);
    __half* alo = reinterpret_cast<__half*>(wsb + pl.ws_alo);
    float* ais = reinterpret_cast<float*>(wsb + pl.ws_ais);
    float* wis = reinterpret_cast<float*>(wsb + pl.ws_wis);
    float* part = p0.ks > 1 ? reinterpret_cast<float*>(wsb + pl.ws_part) : nullptr;
    unsigned* cnt = p0.ks > 1 ? reinterpret_cast<unsigned*>(wsb + pl.ws_cnt) : nullptr;
    uint8_t* w6 = WT == T_Q6_K ? wsb + pl.ws_w6 : nullptr;  // Q6_K super-blocks in 240-byte slots
    // 1. operand preparation: activation pieces, row scales of both operands, split-K counters
    const unsigned pblocks = (unsigned)(p0.M + (p0.N + kTcPrepThreads / 32 - 1) / (kTcPrepThreads / 32));
    tc_prep_kernel<WT><<<pblocks, kTcPrepThreads, 0, s>>>(x, static_cast<const uint8_t*>(wq), p0.M, p0.N, p0.K, ahi,
                                                              alo, ais, wis, cnt, p0.ks > 1 ? p0.tiles : 0, w6);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // 2. tensor maps: raw weight rows as uint16; activation pieces, 64 K x bx rows, 128-byte swizzle
    CUtensorMap tw, tah, tal;
    const unsigned long long rb = WT == T_Q4_K   ? (unsigned long long)p0.K / 256 * 144
                                  : WT == T_Q6_K ? (unsigned long long)p0.K / 256 * kTcQ6Slot
                                                 : (unsigned long long)p0.K / 32 * (WT == T_Q8_0 ? 34 : WT == T_Q5_0 ? 22 : 18);
    const void* wsrc = WT == T_Q6_K ? static_cast<const void*>(w6) : wq;
    if (!make_map(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT16, wsrc, rb / 2, p0.N, rb, p0.raw_row / 2, kTcBW, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&tah, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, ahi, p0.K, p0.M, (unsigned long long)p0.K * 2, kTcBK, p0.bx,
                  CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&tal, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, alo, p0.K, p0.M, (unsigned long long)p0.K * 2, kTcBK, p0.bx,
                  CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    TcParams p = p0;
    p.y = y;
    p.part = part;
    p.cnt = cnt;
    p.ais = ais;
    p.wis = wis;
    // 3. the GEMM, a programmatic dependent of the preparation
    auto* k = qmm_tc_kernel<WT>;
    e = ensure_smem(k, smem_max, g_tc_smem_done[WT == T_Q8_0 ? 0 : WT == T_Q4_K ? 1 : WT == T_Q4_0 ? 2 : WT == T_Q5_0 ? 3 : 4]);
    if (e != cudaSuccess) return e;
    return launch_pdl(k, (unsigned)pl.grid, kTcThreads, pl.smem, s, tw, tah, tal, p);
}

}  // namespace

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

cudaError_t launch_tc(int wt, const TcPlan& plan, const void* wq, const float* x, void* ws, float* y, int smem_max,
                      cudaStream_t s) {
    switch (wt) {
        case T_Q8_0: return tc_go<T_Q8_0>(plan, wq, x, ws, y, smem_max, s);
        case T_Q4_0: return tc_go<T_Q4_0>(plan, wq, x, ws, y, smem_max, s);
        case T_Q5_0: return tc_go<T_Q5_0>(plan, wq, x, ws, y, smem_max, s);
        case T_Q6_K: return tc_go<T_Q6_K>(plan, wq, x, ws, y, smem_max, s);
        default: return tc_go<T_Q4_K>(plan, wq, x, ws, y, smem_max, s);
    }
}

}  // namespace qmm
