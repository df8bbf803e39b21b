// qmm_dmma.cu -- instantiations of the decode MMA kernel (8-row weight tiles)
// and its launcher.
#include "qmm_internal.h"

namespace qmm {
namespace {
unsigned long long g_smem_done[2][2][2];

template <int WT, int AM, int EPI>
cudaError_t go(const DmmaPlan& pl, int smem_max, cudaStream_t s) {
    auto* k = qmm_dmma_kernel<WT, AM, EPI>;
    cudaError_t e = ensure_smem(k, smem_max, g_smem_done[WT == T_Q8_0 ? 0 : 1][AM][EPI]);
    if (e != cudaSuccess) return e;
    k<<<pl.grid, (kDmmaWarps + 1) * 32, pl.smem, s>>>(pl.p);
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_dmma(int wt, int am, int epi, const DmmaPlan& pl, int smem_max, cudaStream_t s) {
    if (wt == T_Q8_0) {
        if (am == A_F32) return epi == E_Y ? go<T_Q8_0, A_F32, E_Y>(pl, smem_max, s) : cudaErrorInvalidValue;
        return epi == E_Y ? go<T_Q8_0, A_INT8, E_Y>(pl, smem_max, s) : go<T_Q8_0, A_INT8, E_SUMS>(pl, smem_max, s);
    }
    if (am == A_F32) return epi == E_Y ? go<T_Q4_K, A_F32, E_Y>(pl, smem_max, s) : cudaErrorInvalidValue;
    return epi == E_Y ? go<T_Q4_K, A_INT8, E_Y>(pl, smem_max, s) : go<T_Q4_K, A_INT8, E_SUMS>(pl, smem_max, s);
}

}  // namespace qmm
