// qmm_tc.cuh -- prefill GEMM (M > 8 activation rows) on the 5th-generation
// tensor cores: tcgen05.mma with the accumulator in tensor memory.
//
// Both QMatMul forms ("同一个 GGUF，CPU 和 Metal 生成的文字不一样" section 出处)
// are the exact sum y = sum_k a_k w_k of dequantized operands:
//   int8_act: a = f(d_a) q_a, the row-quantized activations (Q8_0 or Q8K);
//             sum_k a_k w_k equals the CPU form's sum_b f(d_w) f(d_a) isum_b
//             (both are the same real number; only rounding order differs);
//   f32_act:  a = x.
//   w = f(d) q (Q8_0) or (f(d) sc) q - f(dmin) m (Q4_K), one f32 rounding.
// tcgen05 has no integer kind on sm_103a and its f16 kind carries 11 bits per
// operand, so every operand is scaled by a power of two per row (activation
// rows and weight rows separately, into [2^14, 2^15) at the row maximum) and
// split into two f16 pieces, v = hi + lo (exact for the 18-19 significant
// bits of f(d) q, 2^-22 relative otherwise); the product takes three MMAs,
// hi.hi + hi.lo + lo.hi (the dropped lo.lo is below 2^-22 relative), all into
// one f32 accumulator, and the epilogue multiplies by 2^-(s_row + s_col).
//
// One persistent CTA per SM, 128 x 128 output tiles (128 weight rows x 128
// activation rows), 14 warps:
//   producer  TMA: raw weight rows (2-D box, 128 rows x 272 B = 8 Q8_0 blocks,
//             or 144 B = 1 Q4_K super-block, per 256 K) and the activation
//             pieces (128 rows x 64 f16, 128-byte swizzle, per 64 K);
//   converter 8 warps dequantize the raw weight bytes of each 64-K stage into
//             the two f16 pieces and write them straight into tensor memory
//             (tcgen05.st): the weights are the MMA's A operand, read from
//             TMEM, so the three passes re-read only the activation pieces
//             from shared memory (shared-memory bandwidth, which the operand
//             reads and the converters' traffic share, bounded an earlier
//             layout with both operands in shared memory);
//   MMA       one thread issues tcgen05.mma (M 128 weight rows, N 128
//             activation rows, K 16; 12 per 64 K) into one of two TMEM
//             accumulators, commits to mbarriers that free the stage or hand
//             the tile to the epilogue;
//   epilogue  4 warps, one TMEM lane quarter (32 weight rows) each:
//             tcgen05.ld, scale, y stores coalesced along N.
// TMEM: 2 accumulators x 128 columns + 4 stages x 64 columns of weight pieces.
#pragma once

#include <cuda.h>

#include "qmm_device.cuh"
#include "qmm_prefill.cuh"

namespace qmm {

constexpr int kTcBM = 128;   // activation rows per tile (MMA M)
constexpr int kTcBN = 128;   // weight rows per tile (MMA N)
constexpr int kTcBK = 64;    // K per MMA stage
constexpr int kTcRK = 256;   // K per raw weight stage
constexpr int kTcMS = 4;     // MMA stages
constexpr int kTcRS = 2;     // raw weight stages
constexpr int kTcConvWarps = 8;
constexpr int kTcEpiWarps = 4;
constexpr int kTcThreads = (2 + kTcEpiWarps + kTcConvWarps) * 32;
constexpr int kTcPiece = kTcBM * kTcBK * 2;      // one activation piece of a stage: 16 KB
constexpr int kTcStageBytes = 2 * kTcPiece;      // activation hi, lo: 32 KB
constexpr int kTcTmemCols = 512;                 // 2 x 128 accumulator columns + 4 x 64 weight-piece columns
constexpr int kTcWCol0 = 2 * kTcBN;              // first TMEM column of the weight pieces
constexpr int kTcWCols = kTcBK;                  // columns per stage: hi (32) + lo (32), two f16 per column

struct TcParams {
    float* y;
    const float* ais;   // 2^-s per activation row
    const float* wis;   // 2^-s per weight row
    unsigned* err;
    int M, N, K;
    int mtiles, ntiles, tiles;
    int raw_row;        // raw bytes per weight row per raw stage (272 Q8_0, 144 Q4_K)
    int raw_stage;      // bytes per raw stage (128 rows, rounded to 1 KB)
    int off_raw, off_bar;
};

// shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row atoms 1 KB apart
__device__ __forceinline__ uint64_t tc_sdesc(uint32_t addr) {
    return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) |
           ((uint64_t)2 << 61);
}
// instruction descriptor: f32 accumulator, f16 A and B, both K-major, N = 128, M = 128
constexpr uint32_t kTcIdesc = (1u << 4) | ((uint32_t)(kTcBN >> 3) << 17) | ((uint32_t)(kTcBM >> 4) << 24);

// D (TMEM) += A (TMEM, 128 lanes x 16 f16) x B (shared memory)^T
__device__ __forceinline__ void tc_mma(uint32_t tmem, uint32_t ta, uint64_t db, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem),
        "r"(ta), "l"(db), "r"(kTcIdesc), "r"(accumulate)
        : "memory");
}
// 16 32-bit columns of this warp's TMEM lane quarter from registers
__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t v[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

// 32 f32 columns of this warp's TMEM lane quarter
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float v[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// byte offset of the 16-byte chunk c (8 halves) of row r in a [128][64] f16 tile, 128-byte swizzle
__device__ __forceinline__ int tc_chunk(int r, int c) { return r * 128 + (((c ^ r) & 7) << 4); }

// ---------------------------------------------------------------------------
// weight conversion: one thread, the 32 values of one weight row that one
// Q8_0 block or one Q4_K sub-block holds, scaled by 2^s, as 16 words of hi
// and 16 words of lo f16 pairs (k order natural)
// ---------------------------------------------------------------------------

// Q8_0 block at blk (2-byte aligned): w = ds q with ds = f(d) 2^s as f16
// (exact while it is a normal f16); hi = f16(ds q) by one hmul2, lo = ds q - hi
// by one hfma2 (exact: at most 8 significant bits remain)
__device__ __forceinline__ void tc_conv_q8_0(const uint8_t* blk, float wsc, uint32_t h[16], uint32_t l[16]) {
    const float ds = h2f(*reinterpret_cast<const uint16_t*>(blk)) * wsc;
    const __half2 ds2 = __half2half2(__float2half_rn(ds));
    const uintptr_t a = reinterpret_cast<uintptr_t>(blk + 2);
    const uint32_t* w = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
    const uint32_t sh = (uint32_t)(a & 3u) * 8u;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t word = __funnelshift_r(w[i], w[i + 1], sh) ^ 0x80808080u;  // codes 4i..4i+3, biased by 128
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            uint32_t qb = __byte_perm(word, 0x64646464u, p ? 0x4342u : 0x4140u);  // bytes (2p, 2p+1) under 0x64: 1152 + q
            const __half2 q = __hsub2(*reinterpret_cast<__half2*>(&qb), __half2half2(__ushort_as_half(0x6480)));
            const __half2 hi = __hmul2(q, ds2);
            const __half2 lo = __hfma2(q, ds2, __hneg2(hi));
            h[2 * i + p] = *reinterpret_cast<const uint32_t*>(&hi);
            l[2 * i + p] = *reinterpret_cast<const uint32_t*>(&lo);
        }
    }
}

// Q4_K sub-block 2 sub + j of the super-block at sbk (16-byte aligned): w 2^s =
// fma(e 2^s, q, -o 2^s) in f32 (one rounding, as the dequantization contract),
// split as f16(v) + f16(v - f16(v))
__device__ __forceinline__ void tc_conv_q4_k(const uint8_t* sbk, int sub, int j, float wsc, uint32_t h[16], uint32_t l[16]) {
    const uint4 hd = *reinterpret_cast<const uint4*>(sbk);
    const int jj = 2 * sub + j;
    const float es = h2f(hd.x) * (float)q4k_sc(hd.y, hd.w, jj) * wsc;
    const float os = h2f(hd.x >> 16) * (float)q4k_mn(hd.z, hd.w, jj) * wsc;
    const uint4 q0 = *reinterpret_cast<const uint4*>(sbk + 16 + 32 * sub);
    const uint4 q1 = *reinterpret_cast<const uint4*>(sbk + 16 + 32 * sub + 16);
    const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t nb = (qw[i] >> (4 * j)) & 0x0F0F0F0Fu;  // values 4i..4i+3 of the sub-block
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            const float v0 = fmaf(es, (float)((nb >> (16 * p)) & 0xFu), -os);
            const float v1 = fmaf(es, (float)((nb >> (16 * p + 8)) & 0xFu), -os);
            const __half2 hi = __floats2half2_rn(v0, v1);
            const float2 hf = __half22float2(hi);
            const __half2 lo = __floats2half2_rn(v0 - hf.x, v1 - hf.y);
            h[2 * i + p] = *reinterpret_cast<const uint32_t*>(&hi);
            l[2 * i + p] = *reinterpret_cast<const uint32_t*>(&lo);
        }
    }
}

// ---------------------------------------------------------------------------
// the GEMM
// ---------------------------------------------------------------------------
template <int WT>
__global__ void __launch_bounds__(kTcThreads, 1)
    qmm_tc_kernel(const __grid_constant__ CUtensorMap tw, const __grid_constant__ CUtensorMap tah,
                  const __grid_constant__ CUtensorMap tal, const TcParams p) {
    extern __shared__ __align__(1024) uint8_t smraw[];
    uint8_t* sm = smraw + ((1024 - (smem_u32(smraw) & 1023)) & 1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + p.off_bar);
    uint64_t* x_full = bars;                            // [kTcMS] activation pieces landed (TMA)
    uint64_t* w_full = bars + kTcMS;                    // [kTcMS] weight pieces in TMEM (converter warps)
    uint64_t* m_empty = bars + 2 * kTcMS;               // [kTcMS] stage consumed by the MMAs (commit)
    uint64_t* r_full = bars + 3 * kTcMS;                // [kTcRS] raw weight rows landed (TMA)
    uint64_t* r_empty = bars + 3 * kTcMS + kTcRS;       // [kTcRS] raw stage converted
    uint64_t* acc_full = bars + 3 * kTcMS + 2 * kTcRS;  // [2] accumulator complete (commit)
    uint64_t* acc_empty = acc_full + 2;                 // [2] accumulator read (epilogue)
    static_assert((3 * kTcMS + 2 * kTcRS + 4) * 8 <= 256, "mbarriers overlap the TMEM slot");
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + p.off_bar + 256);
    volatile int* flags = reinterpret_cast<volatile int*>(sm + p.off_bar + 320);
    const int kt_n = p.K / kTcBK;
    if (tid == 0) {
        for (int i = 0; i < kTcMS; ++i) {
            mbar_init(smem_u32(&x_full[i]), 1);
            mbar_init(smem_u32(&w_full[i]), kTcConvWarps);
            mbar_init(smem_u32(&m_empty[i]), 1);
        }
        for (int i = 0; i < kTcRS; ++i) {
            mbar_init(smem_u32(&r_full[i]), 1);
            mbar_init(smem_u32(&r_empty[i]), kTcConvWarps);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&acc_full[i]), 1);
            mbar_init(smem_u32(&acc_empty[i]), kTcEpiWarps * 32);
        }
        flags[0] = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                     "n"(kTcTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    grid_dep_wait();  // the operand-preparing grid has completed

    auto stage = [&](int s) { return sm + s * kTcStageBytes; };  // activation hi | lo, 16 KB each
    auto raw = [&](int s) { return sm + p.off_raw + s * p.raw_stage; };
    // tile t: weight rows (t / mtiles) * 128.., activation rows (t % mtiles) * 128..

    if (warp == 0) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            long long g = 0, rg = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < p.tiles && ok; tile += gridDim.x) {
                const int m0 = (tile % p.mtiles) * kTcBN, n0 = (tile / p.mtiles) * kTcBM;
                for (int kt = 0; kt < kt_n && ok; ++kt, ++g) {
                    if ((kt & 3) == 0) {
                        const int rs = (int)(rg % kTcRS);
                        if (rg >= kTcRS) ok = mbar_wait(smem_u32(&r_empty[rs]), (uint32_t)(((rg / kTcRS) - 1) & 1), flags, p.err);
                        if (!ok) break;
                        mbar_arrive_tx(smem_u32(&r_full[rs]), (uint32_t)(kTcBM * p.raw_row));
                        tma_2d(smem_u32(raw(rs)), &tw, (kt >> 2) * (p.raw_row / 2), n0, smem_u32(&r_full[rs]));
                        ++rg;
                    }
                    const int s = (int)(g % kTcMS);
                    if (g >= kTcMS) ok = mbar_wait(smem_u32(&m_empty[s]), (uint32_t)(((g / kTcMS) - 1) & 1), flags, p.err);
                    if (!ok) break;
                    mbar_arrive_tx(smem_u32(&x_full[s]), (uint32_t)kTcStageBytes);
                    tma_2d(smem_u32(stage(s)), &tah, kt * kTcBK, m0, smem_u32(&x_full[s]));
                    tma_2d(smem_u32(stage(s) + kTcPiece), &tal, kt * kTcBK, m0, smem_u32(&x_full[s]));
                }
            }
            // let every copy this thread issued land before the CTA can exit
            for (long long q = (g > kTcMS ? g - kTcMS : 0); q < g; ++q)
                mbar_wait(smem_u32(&x_full[q % kTcMS]), (uint32_t)((q / kTcMS) & 1), flags, p.err);
            for (long long q = (rg > kTcRS ? rg - kTcRS : 0); q < rg; ++q)
                mbar_wait(smem_u32(&r_full[q % kTcRS]), (uint32_t)((q / kTcRS) & 1), flags, p.err);
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issuer ------------------------------
        if (lane == 0) {
            long long g = 0;
            int tc = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < p.tiles && ok; tile += gridDim.x, ++tc) {
                const int ab = tc & 1;
                if (tc >= 2) ok = mbar_wait(smem_u32(&acc_empty[ab]), (uint32_t)(((tc >> 1) - 1) & 1), flags, p.err);
                if (!ok) break;
                tc_fence_after();
                const uint32_t dt = tmem + (uint32_t)(ab * kTcBN);
                for (int kt = 0; kt < kt_n; ++kt, ++g) {
                    const int s = (int)(g % kTcMS);
                    const uint32_t ph = (uint32_t)((g / kTcMS) & 1);
                    ok = mbar_wait(smem_u32(&x_full[s]), ph, flags, p.err) && mbar_wait(smem_u32(&w_full[s]), ph, flags, p.err);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t xhi = smem_u32(stage(s)), xlo = xhi + kTcPiece;
                    const uint32_t whi = tmem + (uint32_t)(kTcWCol0 + s * kTcWCols), wlo = whi + kTcBK / 2;
#pragma unroll
                    for (int pass = 0; pass < 3; ++pass) {
                        // w_hi x_hi, w_hi x_lo, w_lo x_hi
                        const uint32_t wa = pass == 2 ? wlo : whi, xb = pass == 1 ? xlo : xhi;
#pragma unroll
                        for (int kk = 0; kk < kTcBK / 16; ++kk)
                            tc_mma(dt, wa + 8 * kk, tc_sdesc(xb + 32 * kk), (kt | pass | kk) != 0 ? 1u : 0u);
                    }
                    tc_commit(smem_u32(&m_empty[s]));
                }
                if (!ok) break;
                tc_commit(smem_u32(&acc_full[ab]));
            }
            // the last commits must land before TMEM is released
            if (g > 0) mbar_wait(smem_u32(&m_empty[(g - 1) % kTcMS]), (uint32_t)(((g - 1) / kTcMS) & 1), flags, p.err);
        }
    } else if (warp < 2 + kTcEpiWarps) {
        // ------------------------------ epilogue ------------------------------
        const int q = warp & 3;  // TMEM lane quarter: weight rows 32q..32q+31 of the tile
        int tc = 0;
        for (int tile = blockIdx.x; tile < p.tiles; tile += gridDim.x, ++tc) {
            const int ab = tc & 1;
            if (!mbar_wait(smem_u32(&acc_full[ab]), (uint32_t)((tc >> 1) & 1), flags, p.err)) break;
            tc_fence_after();
            const int m0 = (tile % p.mtiles) * kTcBN, n0 = (tile / p.mtiles) * kTcBM;
            const int n = n0 + 32 * q + lane;
            const float wsn = n < p.N ? __ldg(p.wis + n) : 0.0f;
#pragma unroll 1
            for (int c = 0; c < kTcBN / 32; ++c) {
                float v[32];
                tc_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(ab * kTcBN + 32 * c), v);
                const int mb = m0 + 32 * c;
                if (n < p.N && !flags[0]) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int m = mb + i;
                        if (m < p.M) p.y[(long long)m * p.N + n] = v[i] * wsn * __ldg(p.ais + m);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&acc_empty[ab]));
        }
    } else {
        // ------------------------------ converters ------------------------------
        // warp cw: TMEM lane quarter cw & 3 (weight rows 32 (cw & 3) + lane), values
        // 32 j..32 j+31 of each 64-K stage with j = cw >> 2
        const int cw = warp - (2 + kTcEpiWarps);
        const int q = warp & 3, j = cw >> 2;
        const int n = 32 * q + lane;
        long long g = 0, rg = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < p.tiles && ok; tile += gridDim.x) {
            const int n0 = (tile / p.mtiles) * kTcBM;
            const float wsc = n0 + n < p.N ? __frcp_rn(__ldg(p.wis + n0 + n)) : 1.0f;  // 2^s (exact)
            for (int kt = 0; kt < kt_n && ok; ++kt, ++g) {
                const int sub = kt & 3;
                const int rs = (int)(rg % kTcRS);
                if (sub == 0) ok = mbar_wait(smem_u32(&r_full[rs]), (uint32_t)((rg / kTcRS) & 1), flags, p.err);
                const int s = (int)(g % kTcMS);
                if (ok && g >= kTcMS) ok = mbar_wait(smem_u32(&m_empty[s]), (uint32_t)(((g / kTcMS) - 1) & 1), flags, p.err);
                if (!ok) break;
                tc_fence_after();
                const uint8_t* rrow = raw(rs) + n * p.raw_row;
                uint32_t h[16], l[16];
                if (WT == T_Q8_0) tc_conv_q8_0(rrow + (2 * sub + j) * 34, wsc, h, l);
                else tc_conv_q4_k(rrow, sub, j, wsc, h, l);
                const uint32_t col = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(kTcWCol0 + s * kTcWCols + 16 * j);
                tc_st16(col, h);
                tc_st16(col + kTcBK / 2, l);
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&w_full[s]));  // one arrival per converter warp
                if (sub == 3) {
                    if (lane == 0) mbar_arrive(smem_u32(&r_empty[rs]));
                    ++rg;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTcTmemCols) : "memory");
    }
}

// ---------------------------------------------------------------------------
// operand preparation (one launch before the GEMM): activation pieces and
// per-row scales of both operands
// ---------------------------------------------------------------------------
constexpr int kTcPrepThreads = 256;

// 2^-s for a row whose largest magnitude is amax: amax 2^s in [2^14, 2^15)
__device__ __forceinline__ float tc_row_iscale(float amax) {
    int s = 0;
    if (amax > 0.0f) {
        const int e = (int)((__float_as_uint(amax) >> 23) & 0xff) - 127;
        s = 14 - e;
        s = s > 120 ? 120 : (s < -120 ? -120 : s);
    }
    return ldexpf(1.0f, -s);
}

__device__ __forceinline__ void tc_split_store(float v0, float v1, __half* hi, __half* lo) {
    const __half2 h = __floats2half2_rn(v0, v1);
    const float2 hf = __half22float2(h);
    *reinterpret_cast<__half2*>(hi) = h;
    *reinterpret_cast<__half2*>(lo) = __floats2half2_rn(v0 - hf.x, v1 - hf.y);
}

// blocks [0, M): activation rows; blocks [M, M + ceil(N / 8)): 8 weight rows each (a warp per row)
template <int WT, int AM>
__global__ void __launch_bounds__(kTcPrepThreads) tc_prep_kernel(const float* __restrict__ x, const uint8_t* __restrict__ wq,
                                                                 int M, int N, int K, __half* ahi, __half* alo,
                                                                 float* ais, float* wis) {
    grid_dep_launch();
    __shared__ float red[kTcPrepThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if ((int)blockIdx.x < M) {
        const int m = blockIdx.x;
        const float* xr = x + (long long)m * K;
        float amax = 0.0f;
        for (int i = tid; i < K / 4; i += kTcPrepThreads) {
            const float4 v = __ldg(reinterpret_cast<const float4*>(xr) + i);
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if (lane == 0) red[warp] = amax;
        __syncthreads();
        amax = red[0];
#pragma unroll
        for (int i = 1; i < kTcPrepThreads / 32; ++i) amax = fmaxf(amax, red[i]);
        // int8: |f(d_a) q| <= amax (1 + 2^-11), still below 2^15 after scaling
        const float is = tc_row_iscale(amax);
        const float sc = __frcp_rn(is);
        if (tid == 0) ais[m] = is;
        __half* hr = ahi + (long long)m * K;
        __half* lr = alo + (long long)m * K;
        if (AM == A_F32) {
            for (int i = tid; i < K / 2; i += kTcPrepThreads) {
                const float2 v = __ldg(reinterpret_cast<const float2*>(xr) + i);
                tc_split_store(__fmul_rn(v.x, sc), __fmul_rn(v.y, sc), hr + 2 * i, lr + 2 * i);
            }
        } else if (WT == T_Q8_0) {
            for (int b = tid; b < K / 32; b += kTcPrepThreads) {
                uint32_t c[8];
                float d;
                quant_q8_0_32(xr + b * 32, c, d);
                const float ds = h2f(f2h(d)) * sc;  // f(d_a) 2^s: exact
#pragma unroll
                for (int i = 0; i < 8; ++i)
#pragma unroll
                    for (int e = 0; e < 4; e += 2) {
                        const float q0 = (float)(int8_t)(c[i] >> (8 * e)), q1 = (float)(int8_t)(c[i] >> (8 * e + 8));
                        tc_split_store(ds * q0, ds * q1, hr + b * 32 + 4 * i + e, lr + b * 32 + 4 * i + e);
                    }
            }
        } else {
            // Q8K: a warp per super-block, lane l values 8l..8l+7
            for (int sb = warp; sb < K / 256; sb += kTcPrepThreads / 32) {
                const float* src = xr + sb * 256 + 8 * lane;
                const float4 v0 = __ldg(reinterpret_cast<const float4*>(src));
                const float4 v1 = __ldg(reinterpret_cast<const float4*>(src) + 1);
                float bm = fmaxf(fmaxf(fmaxf(fabsf(v0.x), fabsf(v0.y)), fmaxf(fabsf(v0.z), fabsf(v0.w))),
                                 fmaxf(fmaxf(fabsf(v1.x), fabsf(v1.y)), fmaxf(fabsf(v1.z), fabsf(v1.w))));
#pragma unroll
                for (int o = 16; o; o >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o));
                float d, id;
                q8_scale(bm, d, id);
                const float vv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
                const long long k = (long long)sb * 256 + 8 * lane;
#pragma unroll
                for (int e = 0; e < 8; e += 2)
                    tc_split_store(__fmul_rn(d * (float)q8_code(vv[e], id), sc), __fmul_rn(d * (float)q8_code(vv[e + 1], id), sc),
                                   hr + k + e, lr + k + e);
            }
        }
    } else {
        // weight row scales: a bound on |w| per row from the block scales
        const long long n = (long long)(blockIdx.x - M) * (kTcPrepThreads / 32) + warp;
        if (n >= N) return;
        float bmax = 0.0f;
        if (WT == T_Q8_0) {
            const uint8_t* row = wq + n * (long long)(K / 32) * 34;
            for (int b = lane; b < K / 32; b += 32) bmax = fmaxf(bmax, fabsf(h2f(*reinterpret_cast<const uint16_t*>(row + b * 34))) * 127.0f);
        } else {
            const uint8_t* row = wq + n * (long long)(K / 256) * 144;
            for (int b = lane; b < K / 256; b += 32) {
                const uint32_t dd = *reinterpret_cast<const uint32_t*>(row + b * 144);
                bmax = fmaxf(bmax, fabsf(h2f(dd)) * 945.0f + fabsf(h2f(dd >> 16)) * 63.0f);
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, o));
        if (lane == 0) wis[n] = tc_row_iscale(bmax);
    }
}

// ---------------------------------------------------------------------------
// host-side plan
// ---------------------------------------------------------------------------
struct TcPlan {
    TcParams p;
    int grid;
    size_t smem;
    size_t ws_ahi, ws_alo, ws_ais, ws_wis, workspace;
};

inline bool plan_tc(int wt, int am, long long M, long long N, long long K, int sm_count, int smem_max, TcPlan& out) {
    if (K % kTcRK != 0 || M < 9 || K > (1 << 26)) return false;
    TcPlan pl{};
    TcParams& p = pl.p;
    p.M = (int)M;
    p.N = (int)N;
    p.K = (int)K;
    p.mtiles = (int)((M + kTcBM - 1) / kTcBM);
    p.ntiles = (int)((N + kTcBN - 1) / kTcBN);
    p.tiles = p.mtiles * p.ntiles;
    p.raw_row = wt == T_Q8_0 ? kTcRK / 32 * 34 : 144;
    p.raw_stage = round_up(kTcBN * p.raw_row + 64, 1024);  // Q8_0 word loads reach 4 bytes past a row
    p.off_raw = kTcMS * kTcStageBytes;  // activation pieces; weight pieces live in TMEM
    p.off_bar = p.off_raw + kTcRS * p.raw_stage;
    pl.smem = (size_t)p.off_bar + 512 + 1024;  // barriers, TMEM slot, flags; alignment slack
    if ((long long)pl.smem > smem_max) return false;
    pl.grid = p.tiles < sm_count ? p.tiles : sm_count;
    auto r256 = [](size_t v) { return (v + 255) / 256 * 256; };
    pl.ws_ahi = 0;
    pl.ws_alo = r256((size_t)M * K * 2);
    pl.ws_ais = pl.ws_alo + r256((size_t)M * K * 2);
    pl.ws_wis = pl.ws_ais + r256((size_t)M * 4);
    pl.workspace = pl.ws_wis + r256((size_t)N * 4);
    (void)am;
    out = pl;
    return true;
}

}  // namespace qmm
