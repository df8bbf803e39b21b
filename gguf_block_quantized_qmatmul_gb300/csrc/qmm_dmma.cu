// qmm_dmma.cu -- instantiations of the decode MMA kernel (16-row weight tiles)
// and its launcher.
#include "qmm_internal.h"

namespace qmm {
namespace {
unsigned long long g_smem_done[2][2][4][2];  // [Q8_0, Q4_K][form][column sets 1, 2, 4][epilogue]

template <int WT, int AM, int NB, int EPI>
cudaError_t go(const DmmaPlan& pl, int smem_max, cudaStream_t s) {
    auto* k = qmm_dmma_kernel<WT, AM, NB, EPI>;
    cudaError_t e = ensure_smem(k, smem_max, g_smem_done[WT == T_Q8_0 ? 0 : 1][AM][NB == 4 ? 2 : NB - 1][EPI]);
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
template <int WT, int AM>
cudaError_t prep(const DmmaPlan& pl, void* ext, cudaStream_t s) {
    const DmmaParams& p = pl.p;
    long long blocks;
    constexpr int warps = kPrepThreads / 32;
    if (AM == A_F32 && WT == T_Q8_0) blocks = ((long long)p.M * ((p.units + 7) / 8) + warps - 1) / warps;  // a warp per 8 blocks
    else if (WT == T_Q8_0) blocks = ((long long)p.M * p.units + kPrepThreads - 1) / kPrepThreads;        // a thread per 32-block
    else blocks = ((long long)p.M * p.units + warps - 1) / warps;                                         // a warp per super-block
    if (blocks > 1024) blocks = 1024;
    // programmatic dependent launch: scheduled while the previous grid in the
    // stream (normally the last call's decode grid) still runs; the kernel
    // waits for that grid before it reads x or writes ext
    return launch_pdl(dmma_prep_kernel<WT, AM>, (unsigned)blocks, kPrepThreads, 0, s, p, static_cast<uint8_t*>(ext));
}
}  // namespace

cudaError_t launch_dmma_prep(int wt, int am, const DmmaPlan& pl, void* ext, cudaStream_t s) {
    // Q4_0 and Q5_0 weights take Q8_0 activations: the same preparation as Q8_0
    if (is_b32(wt)) return am == A_F32 ? prep<T_Q8_0, A_F32>(pl, ext, s) : prep<T_Q8_0, A_INT8>(pl, ext, s);
    if (wt == T_Q6_K) return am == A_F32 ? prep<T_Q6_K, A_F32>(pl, ext, s) : prep<T_Q6_K, A_INT8>(pl, ext, s);
    return am == A_F32 ? prep<T_Q4_K, A_F32>(pl, ext, s) : prep<T_Q4_K, A_INT8>(pl, ext, s);
}

cudaError_t launch_dmma(int wt, int am, int epi, const DmmaPlan& pl, int smem_max, cudaStream_t s) {
    if (wt == T_Q4_0 || wt == T_Q5_0) return launch_dmma_x_0(wt, am, epi, pl, smem_max, s);
    if (wt == T_Q6_K) return launch_dmma_q6_k(am, epi, pl, smem_max, s);
    return wt == T_Q8_0 ? go_type<T_Q8_0>(am, epi, pl, smem_max, s) : go_type<T_Q4_K>(am, epi, pl, smem_max, s);
}

}  // namespace qmm
