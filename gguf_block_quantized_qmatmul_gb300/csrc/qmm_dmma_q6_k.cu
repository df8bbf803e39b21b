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

cudaError_t launch_dmma_q6_k(int am, int epi, const DmmaPlan& pl, int smem_max, cudaStream_t s) {
    return go_type<T_Q6_K>(am, epi, pl, smem_max, s);
}

}  // namespace qmm
