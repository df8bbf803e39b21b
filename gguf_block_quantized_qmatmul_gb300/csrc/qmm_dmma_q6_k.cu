// qmm_dmma_q6_k.cu -- instantiations of the decode MMA kernel (16-row weight
// tiles) for Q6_K weights, and their launcher: one k16 MMA per group of 16
// values (s8 codes for int8_act, f16 codes for f32_act); activations are
// prepared as for Q4_K, without its sums.
#include "qmm_internal.h"

namespace qmm {
namespace {
unsigned long long g_smem_done[2][4][2];  // [form][column sets 1, 2, 4][epilogue]

template <int WT, int AM, int NB, int EPI>
cudaError_t go(const DmmaPlan& pl, int smem_max, cudaStream_t s) {
    auto* k = qmm_dmma_kernel<WT, AM, NB, EPI>;
    cudaError_t e = ensure_smem(k, smem_max, g_smem_done[AM][NB == 4 ? 2 : NB - 1][EPI]);
    if (e != cudaSuccess) return e;
    if (!pl.p.ext) {
        k<<<pl.grid, kDmmaThreads, pl.smem, s>>>(pl.p);
        return cudaGetLastError();
    }
    // after the preparing kernel: programmatic dependent launch
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl.grid);
    cfg.blockDim = dim3(kDmmaThreads);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, pl.p);
}

template <int WT>
cudaError_t go_type(int am, int epi, const DmmaPlan& pl, int smem_max, cudaStream_t s) {
    if (am == A_F32) {
        if (epi != E_Y) return cudaErrorInvalidValue;
        return pl.nb == 4   ? go<WT, A_F32, 4, E_Y>(pl, smem_max, s)
               : pl.nb == 2 ? go<WT, A_F32, 2, E_Y>(pl, smem_max, s)
                            : go<WT, A_F32, 1, E_Y>(pl, smem_max, s);
    }
    if (pl.nb == 2)
        return epi == E_Y ? go<WT, A_INT8, 2, E_Y>(pl, smem_max, s) : go<WT, A_INT8, 2, E_SUMS>(pl, smem_max, s);
    return epi == E_Y ? go<WT, A_INT8, 1, E_Y>(pl, smem_max, s) : go<WT, A_INT8, 1, E_SUMS>(pl, smem_max, s);
}
}  // namespace

cudaError_t launch_dmma_q6_k(int am, int epi, const DmmaPlan& pl, int smem_max, cudaStream_t s) {
    return go_type<T_Q6_K>(am, epi, pl, smem_max, s);
}

}  // namespace qmm
