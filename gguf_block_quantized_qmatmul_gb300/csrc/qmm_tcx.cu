// qmm_tcx.cu -- host side of the exact tcgen05 prefill GEMM (the CPU form):
// activation operand preparation, tensor maps, launches.  The Metal form's
// launches of the same kernel are in qmm_tcx_f32.cu.
#include "qmm_internal.h"

namespace qmm {

namespace {
unsigned long long g_tcx_smem_done[10];

// the index of a (type, tile width) instance in g_tcx_smem_done
constexpr int tcx_instance(int wt, int nx) {
    return 2 * (wt == T_Q8_0 ? 0 : wt == T_Q4_K ? 1 : wt == T_Q6_K ? 2 : wt == T_Q4_0 ? 3 : 4) + (nx == 64 ? 1 : 0);
}

template <int WT, int NX>
cudaError_t tcx_go(const TcxPlan& pl, const void* wq, const float* x, void* ws, float* y, int smem_max, cudaStream_t s) {
    using R = TxRaw<WT>;
    const TcxParams& p0 = pl.p;
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    __half* codes = reinterpret_cast<__half*>(wsb + pl.ws_codes);
    float* scales = reinterpret_cast<float*>(wsb + pl.ws_scales);
    __half* bsums = reinterpret_cast<__half*>(wsb + pl.ws_bsums);
    uint8_t* w6 = wsb + pl.ws_w6;  // Q6_K: super-blocks in 240-byte slots
    unsigned* cnt = reinterpret_cast<unsigned*>(wsb + pl.ws_cnt);
    // 1. the activation operand: f16 codes [M][K], scales block-major, (Q4_K) sums of 16 codes;
    //    the split-K arrival counters zeroed
    constexpr bool b32 = R::b32;
    const long long items = b32 ? (long long)p0.M * (p0.K / 32) : (long long)p0.M * (p0.K / 256) * 32;
    tcx_act_kernel<WT><<<(unsigned)((items + 255) / 256), 256, 0, s>>>(x, p0.M, p0.K, pl.mp, codes, scales, bsums, cnt,
                                                                      p0.ks > 1 ? p0.tiles : 0);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (WT == T_Q6_K) {
        tcx_q6_repack_kernel<T_Q6_K><<<(unsigned)(((long long)p0.N * 32 + 255) / 256), 256, 0, s>>>(static_cast<const uint8_t*>(wq),
                                                                                        p0.N, p0.K, w6);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    // 2. tensor maps: raw weight rows as uint16 (128 rows x 256 K); activation codes, 64 K x
    //    NX rows, 128-byte swizzle; activation scales; (Q4_K) the sums of 16 codes, 16 x NX
    //    rows, 32-byte swizzle
    CUtensorMap tw, ta, ts, tb;
    const unsigned long long rb = (unsigned long long)p0.K / 256 * R::row;
    const unsigned long long nsc = b32 ? p0.K / 32 : p0.K / 256;
    const void* wsrc = WT == T_Q6_K ? static_cast<const void*>(w6) : wq;
    bool ok = make_map(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT16, wsrc, rb / 2, p0.N, rb, R::row / 2, kTxW, CU_TENSOR_MAP_SWIZZLE_NONE) &&
              make_map(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, codes, p0.K, p0.M, (unsigned long long)p0.K * 2, 64, NX,
                       CU_TENSOR_MAP_SWIZZLE_128B) &&
              make_map(&ts, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, scales, pl.mp, nsc, (unsigned long long)pl.mp * 4, NX,
                       b32 ? 8 : 1, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (WT == T_Q4_K)
        ok = ok && make_map(&tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, bsums, p0.K / 16, p0.M, (unsigned long long)p0.K / 8, 16,
                            NX, CU_TENSOR_MAP_SWIZZLE_32B);
    else
        tb = ts;  // unused
    if (!ok) return cudaErrorInvalidValue;
    TcxParams p = p0;
    p.y = y;
    p.part = reinterpret_cast<float*>(wsb + pl.ws_part);
    p.cnt = cnt;
    // 3. the GEMM, a programmatic dependent of the preparation
    auto* k = qmm_tcx_kernel<WT, NX, A_INT8>;
    e = ensure_smem(k, smem_max, g_tcx_smem_done[tcx_instance(WT, NX)]);
    if (e != cudaSuccess) return e;
    return launch_pdl(k, (unsigned)pl.grid, kTxThreads, pl.smem, s, tw, ta, ts, tb, p);
}
}  // namespace

cudaError_t launch_tcx(int wt, const TcxPlan& pl, const void* wq, const float* x, void* ws, float* y, int smem_max,
                       cudaStream_t s) {
    const bool n64 = pl.nx == 64;
    if (pl.am == A_F32) return launch_tcx_f32(wt, pl, wq, x, ws, y, smem_max, s);
    switch (wt) {
        case T_Q8_0: return n64 ? tcx_go<T_Q8_0, 64>(pl, wq, x, ws, y, smem_max, s) : tcx_go<T_Q8_0, 128>(pl, wq, x, ws, y, smem_max, s);
        case T_Q4_K: return n64 ? tcx_go<T_Q4_K, 64>(pl, wq, x, ws, y, smem_max, s) : tcx_go<T_Q4_K, 128>(pl, wq, x, ws, y, smem_max, s);
        case T_Q4_0: return n64 ? tcx_go<T_Q4_0, 64>(pl, wq, x, ws, y, smem_max, s) : tcx_go<T_Q4_0, 128>(pl, wq, x, ws, y, smem_max, s);
        case T_Q5_0: return n64 ? tcx_go<T_Q5_0, 64>(pl, wq, x, ws, y, smem_max, s) : tcx_go<T_Q5_0, 128>(pl, wq, x, ws, y, smem_max, s);
        default: return n64 ? tcx_go<T_Q6_K, 64>(pl, wq, x, ws, y, smem_max, s) : tcx_go<T_Q6_K, 128>(pl, wq, x, ws, y, smem_max, s);
    }
}

}  // namespace qmm
