// qmm_tcx_f32.cu -- host side of the exact-code tcgen05 GEMM in the Metal
// form (f32_act, Q8_0 / Q4_K / Q6_K up to 64 rows): the activation pieces,
// Q6_K's repacked weights, tensor maps, the launch.
#include "qmm_internal.h"

namespace qmm {

namespace {
unsigned long long g_tcx_f32_smem_done[6];

// the f32_act form: pieces of the activations, (Q6_K) repacked weights, then the GEMM
template <int WT, int NX>
cudaError_t tcx_go_f32(const TcxPlan& pl, const void* wq, const float* x, void* ws, float* y, int smem_max, cudaStream_t s) {
    using R = TxRaw<WT, A_F32>;
    const TcxParams& p0 = pl.p;
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    __half* hi = reinterpret_cast<__half*>(wsb + pl.ws_codes);
    __half* lo = reinterpret_cast<__half*>(wsb + pl.ws_scales);
    __half* bsums = reinterpret_cast<__half*>(wsb + pl.ws_bsums);
    float* ais = reinterpret_cast<float*>(wsb + pl.ws_ais);
    uint8_t* w6 = wsb + pl.ws_w6;
    unsigned* cnt = reinterpret_cast<unsigned*>(wsb + pl.ws_cnt);
    tcx_act_f32_kernel<WT><<<(unsigned)p0.M, 256, 0, s>>>(x, p0.M, p0.K, hi, lo, bsums, ais, cnt, p0.ks > 1 ? p0.tiles : 0);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (WT == T_Q6_K) {
        tcx_q6_repack_kernel<T_Q6_K><<<(unsigned)(((long long)p0.N * 32 + 255) / 256), 256, 0, s>>>(static_cast<const uint8_t*>(wq),
                                                                                        p0.N, p0.K, w6);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    // tensor maps: raw weight rows; hi and lo pieces, 64 K x NX rows, 128-byte swizzle; (Q4_K)
    // the sums of 16 (hi, then lo, along each row), 16 x NX rows, 32-byte swizzle
    CUtensorMap tw, ta, ts, tb;
    const unsigned long long rb = (unsigned long long)p0.K / 256 * R::row;
    const void* wsrc = WT == T_Q6_K ? static_cast<const void*>(w6) : wq;
    bool ok = make_map(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT16, wsrc, rb / 2, p0.N, rb, R::row / 2, kTxW, CU_TENSOR_MAP_SWIZZLE_NONE) &&
              make_map(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, hi, p0.K, p0.M, (unsigned long long)p0.K * 2, 64, NX,
                       CU_TENSOR_MAP_SWIZZLE_128B) &&
              make_map(&ts, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, lo, p0.K, p0.M, (unsigned long long)p0.K * 2, 64, NX,
                       CU_TENSOR_MAP_SWIZZLE_128B);
    if (WT == T_Q4_K)
        ok = ok && make_map(&tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, bsums, p0.K / 8, p0.M, (unsigned long long)p0.K / 4, 16, NX,
                            CU_TENSOR_MAP_SWIZZLE_32B);
    else
        tb = ta;  // unused
    if (!ok) return cudaErrorInvalidValue;
    TcxParams p = p0;
    p.y = y;
    p.ais = ais;
    p.part = reinterpret_cast<float*>(wsb + pl.ws_part);
    p.cnt = cnt;
    auto* k = qmm_tcx_kernel<WT, NX, A_F32>;
    e = ensure_smem(k, smem_max, g_tcx_f32_smem_done[2 * (WT == T_Q8_0 ? 0 : WT == T_Q4_K ? 1 : 2) + (NX == 64 ? 1 : 0)]);
    if (e != cudaSuccess) return e;
    return launch_pdl(k, (unsigned)pl.grid, kTxThreads, pl.smem, s, tw, ta, ts, tb, p);
}

}  // namespace

cudaError_t launch_tcx_f32(int wt, const TcxPlan& pl, const void* wq, const float* x, void* ws, float* y, int smem_max,
                           cudaStream_t s) {
    const bool n64 = pl.nx == 64;
    switch (wt) {
        case T_Q8_0: return n64 ? tcx_go_f32<T_Q8_0, 64>(pl, wq, x, ws, y, smem_max, s) : tcx_go_f32<T_Q8_0, 128>(pl, wq, x, ws, y, smem_max, s);
        case T_Q4_K: return n64 ? tcx_go_f32<T_Q4_K, 64>(pl, wq, x, ws, y, smem_max, s) : tcx_go_f32<T_Q4_K, 128>(pl, wq, x, ws, y, smem_max, s);
        default: return n64 ? tcx_go_f32<T_Q6_K, 64>(pl, wq, x, ws, y, smem_max, s) : tcx_go_f32<T_Q6_K, 128>(pl, wq, x, ws, y, smem_max, s);
    }
}

}  // namespace qmm
