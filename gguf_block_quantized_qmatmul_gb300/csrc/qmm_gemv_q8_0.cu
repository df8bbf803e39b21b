// qmm_gemv_q8_0.cu -- instantiations of the decode GEMV kernel for Q8_0
// weights (M = 1, 2, 4, 8 activation rows; matmul and block-sum epilogues).
#include "qmm_internal.h"

namespace qmm {
namespace {
unsigned long long g_smem_done[2][4];

template <int MT, int EPI>
cudaError_t go(const GemvPlan& pl, int smem_max, cudaStream_t s, unsigned long long& done) {
    auto* k = qmm_gemv_kernel<T_Q8_0, MT, EPI>;
    cudaError_t e = ensure_smem(k, smem_max, done);
    if (e != cudaSuccess) return e;
    return launch_pdl(k, (unsigned)pl.grid, (kGemvWarps + 1) * 32, pl.smem, s, pl.p);
}

template <int EPI>
cudaError_t by_mt(const GemvPlan& pl, int smem_max, cudaStream_t s) {
    unsigned long long* d = g_smem_done[EPI];
    switch (pl.mt) {
        case 1: return go<1, EPI>(pl, smem_max, s, d[0]);
        case 2: return go<2, EPI>(pl, smem_max, s, d[1]);
        case 4: return go<4, EPI>(pl, smem_max, s, d[2]);
        case 8: return go<8, EPI>(pl, smem_max, s, d[3]);
        default: return cudaErrorInvalidValue;
    }
}
}  // namespace

cudaError_t launch_gemv_q8_0(int epi, const GemvPlan& pl, int smem_max, cudaStream_t s) {
    return epi == E_SUMS ? by_mt<E_SUMS>(pl, smem_max, s) : by_mt<E_Y>(pl, smem_max, s);
}

}  // namespace qmm
