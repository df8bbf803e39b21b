// qmm_dmma_x_0.cu -- instantiations of the decode MMA kernel (16-row weight
// tiles) for Q4_0 and Q5_0 weights, and their launcher.  The kernel unpacks
// their nibbles (and Q5_0's fifth bits) into the same signed-code fragments
// as Q8_0; activations are prepared as for Q8_0.
#include "qmm_internal.h"

namespace qmm {
namespace {
unsigned long long g_smem_done[2][2][4][2];  // [Q4_0, Q5_0][form][column sets 1, 2, 4][epilogue]

template <int WT, int AM, int NB, int EPI>
cudaError_t go(const DmmaPlan& pl, int smem_max, cudaStream_t s) {
    auto* k = qmm_dmma_kernel<WT, AM, NB, EPI>;
    cudaError_t e = ensure_smem(k, smem_max, g_smem_done[WT == T_Q4_0 ? 0 : 1][AM][NB == 4 ? 2 : NB - 1][EPI]);
    if (e != cudaSuccess) return e;
    // programmatic dependent launch: the first weight stages stream while the
    // previous grid (the preparing kernel, or the last call) finishes
    return launch_pdl(k, (unsigned)pl.grid, kDmmaThreads, pl.smem, s, pl.p);
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

cudaError_t launch_dmma_x_0(int wt, int am, int epi, const DmmaPlan& pl, int smem_max, cudaStream_t s) {
    return wt == T_Q4_0 ? go_type<T_Q4_0>(am, epi, pl, smem_max, s) : go_type<T_Q5_0>(am, epi, pl, smem_max, s);
}

}  // namespace qmm
