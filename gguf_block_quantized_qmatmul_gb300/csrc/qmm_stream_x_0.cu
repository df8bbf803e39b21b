// qmm_stream_x_0.cu -- instantiations of the streaming kernel for Q4_0 and
// Q5_0 weights (32-value blocks paired with Q8_0 activations), and their
// launchers.
#include "qmm_internal.h"

namespace qmm {
namespace {
unsigned long long g_smem_done[2][2][2][4];  // [Q4_0, Q5_0][AM][EPI][nt]

template <int WT, int AM, int NT, int EPI>
cudaError_t go(const StreamPlan& pl, int smem_max, cudaStream_t s, unsigned long long& done) {
    auto* k = qmm_stream_kernel<WT, AM, NT, EPI>;
    cudaError_t e = ensure_smem(k, smem_max, done);
    if (e != cudaSuccess) return e;
    constexpr int threads = (consumer_warps(WT, AM, NT) + 1) * 32;
    k<<<pl.grid, threads, pl.smem, s>>>(pl.p);
    return cudaGetLastError();
}

template <int WT, int AM, int EPI>
cudaError_t by_nt(const StreamPlan& pl, int smem_max, cudaStream_t s) {
    unsigned long long* d = g_smem_done[WT == T_Q5_0 ? 1 : 0][AM][EPI];
    switch (pl.nt) {
        case 1: return go<WT, AM, 1, EPI>(pl, smem_max, s, d[0]);
        case 2: return go<WT, AM, 2, EPI>(pl, smem_max, s, d[1]);
        case 4: return go<WT, AM, 4, EPI>(pl, smem_max, s, d[2]);
        case 8: return go<WT, AM, 8, EPI>(pl, smem_max, s, d[3]);
        default: return cudaErrorInvalidValue;
    }
}

template <int WT>
cudaError_t launch(int am, int epi, const StreamPlan& pl, int smem_max, cudaStream_t s) {
    if (am == A_INT8 && epi == E_Y) return by_nt<WT, A_INT8, E_Y>(pl, smem_max, s);
    if (am == A_INT8 && epi == E_SUMS) return by_nt<WT, A_INT8, E_SUMS>(pl, smem_max, s);
    if (am == A_F32 && epi == E_Y) return by_nt<WT, A_F32, E_Y>(pl, smem_max, s);
    return cudaErrorInvalidValue;
}
}  // namespace

cudaError_t launch_stream_q4_0(int am, int epi, const StreamPlan& pl, int smem_max, cudaStream_t s) {
    return launch<T_Q4_0>(am, epi, pl, smem_max, s);
}

cudaError_t launch_stream_q5_0(int am, int epi, const StreamPlan& pl, int smem_max, cudaStream_t s) {
    return launch<T_Q5_0>(am, epi, pl, smem_max, s);
}

}  // namespace qmm
