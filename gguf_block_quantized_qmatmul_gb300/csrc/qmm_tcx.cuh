// qmm_tcx.cuh -- the CPU form's prefill GEMM (int8_act, M > 16 activation
// rows) on the 5th-generation tensor cores with exact per-block sums.
//
// "同一个 GGUF，CPU 和 Metal 生成的文字不一样" section 出处: the CPU form
// quantizes every activation row to Q8_0 and multiplies it block by block as
// an integer dot product,
//   y = sum_b f(d_w) f(d_a) isum_b,   isum_b = sum over the block's 32 values
//   of the weight code times the activation code.
// Its parity bound is taken over the block terms, so every isum_b must be
// formed exactly.  sm_103a's tcgen05 has no integer kind, but every code
// (|q| <= 127) is exact in f16 and every sum of at most 32 products of two
// codes (< 2^19) is exact in the f32 accumulator: an MMA group of one block
// with a restarted accumulator yields isum_b exactly.  The fold, y += isum_b
// f(d_w) f(d_a), is then one scale product and one FMA per output element
// per block, in packed f32x2 arithmetic on the drained accumulator.
//
// One persistent CTA per SM over work units: an output tile of 128 weight
// rows (MMA M, the TMEM lanes) x 128 activation rows (MMA N), all of K.
// 22 warps:
//   producer   TMA: raw weight rows (2-D box of 128 rows x 272 B = 8 Q8_0
//              blocks) with the 8 blocks' activation scales ([8][128] f32,
//              prepared block-major) into a raw ring; per block the
//              activation codes (128 rows x 32 f16, 64-byte swizzle);
//   MMA        one thread: per block two tcgen05.mma (K 16) from shared
//              memory into one of four TMEM accumulators, restarted;
//   epilogue   16 warps, a TMEM lane quarter (32 weight rows) and 32 of the
//              128 accumulator columns each: drain the block's sums, fold
//              them with f(d_w) (read from the raw stage) and f(d_a), keep
//              the tile's running sums in registers, store y at the end;
//   converter  4 warps, one weight row per thread: the block's 32 codes to
//              exact f16, written to shared memory in the MMA's 64-byte
//              swizzled K-major layout.
// A raw stage is released when its blocks are converted and folded.
#pragma once

#include "qmm_tc.cuh"

namespace qmm {

constexpr int kTxW = 128;         // weight rows per tile (MMA M)
constexpr int kTxX = 128;         // activation rows per tile (MMA N)
constexpr int kTxS = 4;           // block stages: weight codes + activation codes in shared memory
constexpr int kTxAcc = 4;         // TMEM accumulators of kTxX columns
constexpr int kTxTmemCols = kTxAcc * kTxX;
constexpr int kTxRaw = 272;       // raw bytes per weight row per raw stage (8 Q8_0 blocks)
constexpr int kTxRawMax = 6;
constexpr int kTxEpiWarps = 16;
constexpr int kTxConvWarps = 4;
constexpr int kTxThreads = (2 + kTxEpiWarps + kTxConvWarps) * 32;
constexpr int kTxStage = 2 * kTxW * 64;                 // A (weights) then B (activations): 8 KB each
constexpr int kTxScaleOff = kTxW * kTxRaw;              // activation scales inside a raw slot
constexpr int kTxRawSlot = (kTxScaleOff + 8 * kTxX * 4 + 1023) / 1024 * 1024;

struct TcxParams {
    float* y;
    unsigned* err;
    int M, N, K;
    int mtiles, ntiles, units;
    int nrs;       // raw stages in K (K / 256)
    int nraw;      // raw slots in shared memory
    int off_raw, off_bar;
};

// D (TMEM) += A (shared memory) x B (shared memory)^T
__device__ __forceinline__ void tcx_mma(uint32_t tmem, uint64_t da, uint64_t db, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
        "l"(da), "l"(db), "r"(idesc), "r"(accumulate)
        : "memory");
}

// signed codes of a word (4 bytes) as two exact f16 pairs: bytes 0, 1 and 2, 3
__device__ __forceinline__ void tcx_codes(uint32_t word, uint32_t& p01, uint32_t& p23) {
    const uint32_t u = word ^ 0x80808080u;  // code + 128
    uint32_t a = __byte_perm(u, 0x64646464u, 0x5140u), b = __byte_perm(u, 0x64646464u, 0x5342u);  // f16 1024 + (code + 128)
    const __half2 off = __half2half2(__ushort_as_half(0x6480));                                    // 1152
    const __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), off), hb = __hsub2(*reinterpret_cast<__half2*>(&b), off);
    p01 = *reinterpret_cast<const uint32_t*>(&ha);
    p23 = *reinterpret_cast<const uint32_t*>(&hb);
}

// Q8_0 block J (0..7) of a 272-byte raw row (16-byte aligned) as 16 words of
// exact f16 code pairs (values 2i, 2i + 1 in word i)
template <int J>
__device__ __forceinline__ void tcx_conv_q8_0(const uint8_t* row, uint32_t h[16]) {
    constexpr int A = (34 * J) & ~15;  // first 16-byte chunk
    constexpr int O = 34 * J - A;      // byte offset of d in the chunk
    const uint4 c0 = *reinterpret_cast<const uint4*>(row + A);
    const uint4 c1 = *reinterpret_cast<const uint4*>(row + A + 16);
    const uint4 c2 = *reinterpret_cast<const uint4*>(row + A + 32);
    const uint32_t w[12] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w, c2.x, c2.y, c2.z, c2.w};
    constexpr int QW = (O + 2) / 4, QS = 8 * ((O + 2) % 4);  // codes: word QW onward, shifted by QS bits
    static_assert(QW + 8 + (QS != 0 ? 1 : 0) <= 12, "the three chunks hold the block");
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t word;
        if constexpr (QS != 0) word = __funnelshift_r(w[QW + i], w[QW + i + 1], QS);
        else word = w[QW + i];
        tcx_codes(word, h[2 * i], h[2 * i + 1]);
    }
}

// f(d) of Q8_0 block j of the raw row at `row` (2-byte aligned)
__device__ __forceinline__ float tcx_block_scale(const uint8_t* row, int j) {
    return h2f(*reinterpret_cast<const uint16_t*>(row + 34 * j));
}

template <int WT>  // T_Q8_0
__global__ void __launch_bounds__(kTxThreads, 1)
    qmm_tcx_kernel(const __grid_constant__ CUtensorMap tw, const __grid_constant__ CUtensorMap ta,
                   const __grid_constant__ CUtensorMap ts, const TcxParams p) {
    extern __shared__ __align__(1024) uint8_t smraw[];
    uint8_t* sm = smraw + ((1024 - (smem_u32(smraw) & 1023)) & 1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + p.off_bar);
    uint64_t* full = bars;                       // [kTxS] activation codes landed and weight codes converted
    uint64_t* empty = full + kTxS;               // [kTxS] stage consumed by the MMAs (commit)
    uint64_t* r_full = empty + kTxS;             // [kTxRawMax] raw weight rows and scales landed (TMA)
    uint64_t* r_empty = r_full + kTxRawMax;      // [kTxRawMax] raw stage converted and folded
    uint64_t* acc_full = r_empty + kTxRawMax;    // [kTxAcc] block sums complete (commit)
    uint64_t* acc_empty = acc_full + kTxAcc;     // [kTxAcc] block sums drained (epilogue)
    static_assert((2 * kTxS + 2 * kTxRawMax + 2 * kTxAcc) * 8 <= 448, "mbarriers overlap the TMEM slot");
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + p.off_bar + 448);
    volatile int* flags = reinterpret_cast<volatile int*>(sm + p.off_bar + 480);  // [0] abort
    if (tid == 0) {
        for (int i = 0; i < kTxS; ++i) {
            mbar_init(smem_u32(&full[i]), 1 + kTxConvWarps);
            mbar_init(smem_u32(&empty[i]), 1);
        }
        for (int i = 0; i < kTxRawMax; ++i) {
            mbar_init(smem_u32(&r_full[i]), 1);
            mbar_init(smem_u32(&r_empty[i]), kTxConvWarps + kTxEpiWarps);
        }
        for (int i = 0; i < kTxAcc; ++i) {
            mbar_init(smem_u32(&acc_full[i]), 1);
            mbar_init(smem_u32(&acc_empty[i]), kTxEpiWarps);
        }
        flags[0] = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                     "n"(kTxTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    grid_dep_wait();  // the activation-preparing grid has completed

    auto wstage = [&](int s) { return sm + s * kTxStage; };               // A: weight codes
    auto xstage = [&](int s) { return sm + s * kTxStage + kTxW * 64; };   // B: activation codes
    auto raw = [&](int s) { return sm + p.off_raw + s * kTxRawSlot; };
    const int nb = p.nrs * 8;  // blocks per unit
    // unit u: weight tile u / mtiles (rows n0..n0+127), activation tile u % mtiles (rows m0..m0+127)

    if (warp == 0) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            long long g = 0, ri = 0, rc = 0;  // blocks issued; raw stages issued; raw stages whose blocks are issued
            int iu = blockIdx.x, ir = 0;      // raw-issue cursor: unit, raw stage
            bool ok = true;
            for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
                const int m0 = (u % p.mtiles) * kTxX;
                for (int r = 0; r < p.nrs && ok; ++r, ++rc) {
                    // raw stages up to nraw - 2 ahead, across units: the slot a new stage
                    // reuses is then two stages old, one the epilogue has finished folding
                    // (waiting on a younger one would hold back this stage's activations)
                    while (ok && iu < p.units && ri <= rc + p.nraw - 2) {
                        const int rs = (int)(ri % p.nraw);
                        if (ri >= p.nraw) ok = mbar_wait(smem_u32(&r_empty[rs]), (uint32_t)(((ri / p.nraw) - 1) & 1), flags, p.err);
                        if (!ok) break;
                        const int in0 = (iu / p.mtiles) * kTxW, im0 = (iu % p.mtiles) * kTxX;
                        mbar_arrive_tx(smem_u32(&r_full[rs]), (uint32_t)(kTxW * kTxRaw + 8 * kTxX * 4));
                        tma_2d(smem_u32(raw(rs)), &tw, ir * (kTxRaw / 2), in0, smem_u32(&r_full[rs]));
                        tma_2d(smem_u32(raw(rs) + kTxScaleOff), &ts, im0, 8 * ir, smem_u32(&r_full[rs]));
                        ++ri;
                        if (++ir >= p.nrs) ir = 0, iu += gridDim.x;
                    }
                    for (int j = 0; j < 8 && ok; ++j, ++g) {
                        const int s = (int)(g % kTxS);
                        if (g >= kTxS) ok = mbar_wait(smem_u32(&empty[s]), (uint32_t)(((g / kTxS) - 1) & 1), flags, p.err);
                        if (!ok) break;
                        mbar_arrive_tx(smem_u32(&full[s]), (uint32_t)(kTxX * 64));
                        tma_2d(smem_u32(xstage(s)), &ta, (r * 8 + j) * 32, m0, smem_u32(&full[s]));
                    }
                }
            }
            // let every copy this thread issued land before the CTA can exit
            for (long long q = (g > kTxS ? g - kTxS : 0); q < g; ++q)
                mbar_drain(smem_u32(&full[q % kTxS]), (uint32_t)((q / kTxS) & 1), flags, p.err);
            for (long long q = (ri > p.nraw ? ri - p.nraw : 0); q < ri; ++q)
                mbar_drain(smem_u32(&r_full[q % p.nraw]), (uint32_t)((q / p.nraw) & 1), flags, p.err);
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issuer ------------------------------
        if (lane == 0) {
            const uint32_t idesc = tc_idesc(kTxX);
            long long g = 0;
            bool ok = true;
            uint32_t ready = 0;  // the next stage's barrier, tested ahead
            for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
                for (int b = 0; b < nb && ok; ++b, ++g) {
                    const int s = (int)(g % kTxS), ab = (int)(g % kTxAcc);
                    if (g >= kTxAcc) ok = mbar_wait(smem_u32(&acc_empty[ab]), (uint32_t)(((g / kTxAcc) - 1) & 1), flags, p.err);
                    if (!ok) break;
                    const uint32_t nxt = mbar_test(smem_u32(&full[(g + 1) % kTxS]), (uint32_t)(((g + 1) / kTxS) & 1));
                    if (!ready) ok = mbar_wait(smem_u32(&full[s]), (uint32_t)((g / kTxS) & 1), flags, p.err);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t wa = smem_u32(wstage(s)), xb = smem_u32(xstage(s));
                    const uint32_t dt = tmem + (uint32_t)(ab * kTxX);
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk) tcx_mma(dt, tc_sdesc(wa + 32 * kk), tc_sdesc(xb + 32 * kk), idesc, kk);
                    tc_commit(smem_u32(&empty[s]));
                    tc_commit(smem_u32(&acc_full[ab]));
                    ready = nxt;
                }
            }
            // the last commits must land before TMEM is released
            if (g > 0) mbar_drain(smem_u32(&empty[(g - 1) % kTxS]), (uint32_t)(((g - 1) / kTxS) & 1), flags, p.err);
        }
    } else if (warp < 2 + kTxEpiWarps) {
        // ------------------------------ epilogue ------------------------------
        const int ew = warp - 2;
        const int q = warp & 3;   // TMEM lane quarter: weight rows 32q..32q+31 of the tile
        const int cq = ew >> 2;   // accumulator columns 32cq..32cq+31: activation rows of the tile
        const uint32_t tq = (uint32_t)(32 * q) << 16;
        const int nl = 32 * q + lane;  // this thread's weight row in the tile
        long long g = 0, rg = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
            const int m0 = (u % p.mtiles) * kTxX, n0 = (u / p.mtiles) * kTxW;
            unsigned long long acc[16];  // running sums of activation rows 32cq + 2i, 2i + 1
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[i] = 0ull;
            for (int r = 0; r < p.nrs && ok; ++r, ++rg) {
                const int rs = (int)(rg % p.nraw);
                const uint8_t* wrow = raw(rs) + nl * kTxRaw;
                const float* asc = reinterpret_cast<const float*>(raw(rs) + kTxScaleOff) + 32 * cq;
                for (int j = 0; j < 8; ++j, ++g) {
                    const int ab = (int)(g % kTxAcc);
                    if (!(ok = mbar_wait(smem_u32(&acc_full[ab]), (uint32_t)((g / kTxAcc) & 1), flags, p.err))) break;
                    tc_fence_after();
                    __syncwarp();
                    const uint32_t acol = tmem + tq + (uint32_t)(ab * kTxX + 32 * cq);
                    uint32_t v0[16], v1[16];
                    tc_ld16(acol, v0);
                    tc_ld16(acol + 16, v1);
                    tc_wait_ld();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&acc_empty[ab]));
                    // fold: y += isum f(d_w) f(d_a)
                    const float dw = tcx_block_scale(wrow, j);
                    const unsigned long long dw2 = f2pack(dw, dw);
                    const float* aj = asc + j * kTxX;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const float4 a4 = *reinterpret_cast<const float4*>(aj + 4 * c);
                        const uint32_t* v = c < 4 ? v0 + 4 * c : v1 + 4 * (c - 4);
                        const unsigned long long s01 = mul2(f2pack(a4.x, a4.y), dw2), s23 = mul2(f2pack(a4.z, a4.w), dw2);
                        acc[2 * c] = fma2(f2pack(__uint_as_float(v[0]), __uint_as_float(v[1])), s01, acc[2 * c]);
                        acc[2 * c + 1] = fma2(f2pack(__uint_as_float(v[2]), __uint_as_float(v[3])), s23, acc[2 * c + 1]);
                    }
                }
                if (!ok) break;
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&r_empty[rs]));  // this warp no longer reads the raw stage
            }
            if (!ok || flags[0]) break;
            const int n = n0 + nl;
            if (n < p.N) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int m = m0 + 32 * cq + 2 * i;
                    if (m < p.M) p.y[(size_t)m * p.N + n] = f2lo(acc[i]);
                    if (m + 1 < p.M) p.y[(size_t)(m + 1) * p.N + n] = f2hi(acc[i]);
                }
            }
        }
    } else {
        // ------------------------------ converters ------------------------------
        const int r = 32 * (warp - 2 - kTxEpiWarps) + lane;  // weight row of the tile
        // this row's four 16-byte chunks in the 64-byte swizzled K-major layout
        const int rbase = (r >> 3) * 512 + (r & 7) * 64, sw = (r >> 1) & 3;
        long long g = 0, rg = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
            for (int rr = 0; rr < p.nrs && ok; ++rr, ++rg) {
                const int rs = (int)(rg % p.nraw);
                if (!(ok = mbar_wait(smem_u32(&r_full[rs]), (uint32_t)((rg / p.nraw) & 1), flags, p.err))) break;
                const uint8_t* wrow = raw(rs) + r * kTxRaw;
#pragma unroll
                for (int j = 0; j < 8; ++j, ++g) {
                    const int s = (int)(g % kTxS);
                    if (g >= kTxS && !(ok = mbar_wait(smem_u32(&empty[s]), (uint32_t)(((g / kTxS) - 1) & 1), flags, p.err))) break;
                    uint32_t h[16];
                    if (j == 0) tcx_conv_q8_0<0>(wrow, h);
                    else if (j == 1) tcx_conv_q8_0<1>(wrow, h);
                    else if (j == 2) tcx_conv_q8_0<2>(wrow, h);
                    else if (j == 3) tcx_conv_q8_0<3>(wrow, h);
                    else if (j == 4) tcx_conv_q8_0<4>(wrow, h);
                    else if (j == 5) tcx_conv_q8_0<5>(wrow, h);
                    else if (j == 6) tcx_conv_q8_0<6>(wrow, h);
                    else tcx_conv_q8_0<7>(wrow, h);
                    uint8_t* a = wstage(s) + rbase;
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        *reinterpret_cast<uint4*>(a + ((c ^ sw) << 4)) = make_uint4(h[4 * c], h[4 * c + 1], h[4 * c + 2], h[4 * c + 3]);
                    fence_proxy_async();  // the generic-proxy stores, before the tensor core reads them
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&full[s]));
                }
                if (!ok) break;
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&r_empty[rs]));
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTxTmemCols) : "memory");
    }
}

// The activation operand, written once per call: one thread per (row m,
// 32-block b) quantizes the block to Q8_0 and writes its codes as f16 to
// codes[m][K] and the f16-rounded scale f(d_a) block-major to scales[b][mp].
template <int WT>  // T_Q8_0
__global__ void tcx_act_kernel(const float* __restrict__ x, int M, int K, int mp, __half* __restrict__ codes,
                               float* __restrict__ scales) {
    grid_dep_launch();
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const int nb = K / 32;
    if (i >= (long long)M * nb) return;
    const int m = (int)(i / nb), b = (int)(i - (long long)m * nb);
    uint32_t c[8];
    float d;
    quant_q8_0_32(x + (long long)m * K + 32 * b, c, d);
    uint32_t h[16];
#pragma unroll
    for (int k = 0; k < 8; ++k) tcx_codes(c[k], h[2 * k], h[2 * k + 1]);
    uint4* o = reinterpret_cast<uint4*>(codes + (long long)m * K + 32 * b);
#pragma unroll
    for (int k = 0; k < 4; ++k) o[k] = make_uint4(h[4 * k], h[4 * k + 1], h[4 * k + 2], h[4 * k + 3]);
    scales[(long long)b * mp + m] = h2f(f2h(d));
}

// ---------------------------------------------------------------------------
// host-side plan
// ---------------------------------------------------------------------------
struct TcxPlan {
    TcxParams p;
    int grid;
    size_t smem;
    int mp;  // activation scale rows: M rounded up to 4 (16-byte rows for the tensor map)
    size_t ws_codes, ws_scales, workspace;
};

inline bool plan_tcx(int wt, long long M, long long N, long long K, int sm_count, int smem_max, TcxPlan& out) {
    if (wt != T_Q8_0 || K % 256 != 0 || M < 17 || K > (1 << 26) || M > (1 << 24) || N > (1 << 24)) return false;
    TcxPlan pl{};
    TcxParams& p = pl.p;
    p.M = (int)M;
    p.N = (int)N;
    p.K = (int)K;
    p.mtiles = (int)((M + kTxX - 1) / kTxX);
    p.ntiles = (int)((N + kTxW - 1) / kTxW);
    p.units = p.mtiles * p.ntiles;
    p.nrs = (int)(K / 256);
    p.off_raw = kTxS * kTxStage;
    const int fixed = 512 + 1024;  // barriers, TMEM slot, flags; alignment slack
    p.nraw = (smem_max - p.off_raw - fixed) / kTxRawSlot;
    if (p.nraw > kTxRawMax) p.nraw = kTxRawMax;
    if (p.nraw < 3) return false;  // the epilogue holds a raw stage while the converters fill the next
    p.off_bar = p.off_raw + p.nraw * kTxRawSlot;
    pl.smem = (size_t)p.off_bar + fixed;
    pl.grid = p.units < sm_count ? p.units : sm_count;
    pl.mp = (int)((M + 3) / 4 * 4);
    auto r256 = [](size_t v) { return (v + 255) / 256 * 256; };
    pl.ws_codes = 0;
    pl.ws_scales = r256((size_t)M * K * 2);
    pl.workspace = pl.ws_scales + r256((size_t)(K / 32) * pl.mp * 4);
    out = pl;
    return true;
}

}  // namespace qmm
