// qmm_dmma.cu -- instantiations of the decode MMA kernel (16-row weight tiles)
// and its launcher.
#include "qmm_internal.h"

namespace qmm {
namespace {
unsigned long long g_smem_done[2][2][2][2];

template <int WT, int AM, int NB, int EPI>
cudaError_t go(const DmmaPlan& pl, int smem_max, cudaStream_t s) {
    auto* k = qmm_dmma_kernel<WT, AM, NB, EPI>;
    cudaError_t e = ensure_smem(k, smem_max, g_smem_done[WT == T_Q8_0 ? 0 : 1][AM][NB - 1][EPI]);
    if (e != cudaSuccess) return e;
    k<<<pl.grid, (kDmmaWarps + 1) * 32, pl.smem, s>>>(pl.p);
    return cudaGetLastError();
}

template <int WT>
cudaError_t go_type(int am, int epi, const DmmaPlan& pl, int smem_max, cudaStream_t s) {
    if (am == A_F32) {
        if (epi != E_Y) return cudaErrorInvalidValue;
        return pl.nb == 2 ? go<WT, A_F32, 2, E_Y>(pl, smem_max, s) : go<WT, A_F32, 1, E_Y>(pl, smem_max, s);
    }
    return epi == E_Y ? go<WT, A_INT8, 1, E_Y>(pl, smem_max, s) : go<WT, A_INT8, 1, E_SUMS>(pl, smem_max, s);
}
}  // namespace

cudaError_t launch_dmma(int wt, int am, int epi, const DmmaPlan& pl, int smem_max, cudaStream_t s) {
    return wt == T_Q8_0 ? go_type<T_Q8_0>(am, epi, pl, smem_max, s) : go_type<T_Q4_K>(am, epi, pl, smem_max, s);
}

}  // namespace qmm
