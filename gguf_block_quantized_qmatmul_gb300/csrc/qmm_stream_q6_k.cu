// qmm_stream_q6_k.cu -- instantiations of the streaming kernel for
// Q6_K weights (warp MMA tiles, one k16 MMA per group of 16), and their
// launcher.  Every Q6_K matmul (decode and prefill) and its block sums run
// here.
#include "qmm_internal.h"

namespace qmm {
namespace {
unsigned long long g_smem_done[2][2][4];

template <int AM, int NT, int EPI>
cudaError_t go(const StreamPlan& pl, int smem_max, cudaStream_t s, unsigned long long& done) {
    auto* k = qmm_stream_kernel<T_Q6_K, AM, NT, EPI>;
    cudaError_t e = ensure_smem(k, smem_max, done);
    if (e != cudaSuccess) return e;
    constexpr int threads = (consumer_warps(T_Q6_K, AM, NT) + 1) * 32;
    k<<<pl.grid, threads, pl.smem, s>>>(pl.p);
    return cudaGetLastError();
}

template <int AM, int EPI>
cudaError_t by_nt(const StreamPlan& pl, int smem_max, cudaStream_t s) {
    unsigned long long* d = g_smem_done[AM][EPI];
    switch (pl.nt) {
        case 1: return go<AM, 1, EPI>(pl, smem_max, s, d[0]);
        case 2: return go<AM, 2, EPI>(pl, smem_max, s, d[1]);
        case 4: return go<AM, 4, EPI>(pl, smem_max, s, d[2]);
        case 8: return go<AM, 8, EPI>(pl, smem_max, s, d[3]);
        default: return cudaErrorInvalidValue;
    }
}
}  // namespace

cudaError_t launch_stream_q6_k(int am, int epi, const StreamPlan& pl, int smem_max, cudaStream_t s) {
    if (am == A_INT8 && epi == E_Y) return by_nt<A_INT8, E_Y>(pl, smem_max, s);
    if (am == A_INT8 && epi == E_SUMS) return by_nt<A_INT8, E_SUMS>(pl, smem_max, s);
    if (am == A_F32 && epi == E_Y) return by_nt<A_F32, E_Y>(pl, smem_max, s);
    return cudaErrorInvalidValue;
}

}  // namespace qmm
