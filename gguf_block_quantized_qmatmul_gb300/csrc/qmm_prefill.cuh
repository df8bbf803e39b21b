// qmm_prefill.cuh -- the CPU form's prefill GEMM (int8_act, M > 16 activation
// rows) for Q8_0 weights, with exact integer block sums.
//
// "同一个 GGUF，CPU 和 Metal 生成的文字不一样" section 出处: the CPU form
// quantizes each activation row to Q8_0 and takes integer block dot products,
//   y = sum_b f(d_w) f(d_a) isum_b, isum_b the exact integer dot of the 32
//   weight codes and the row's activation codes.
// Its parity bound is taken over the block terms f(d_w) f(d_a) isum_b, which
// can cancel far more than the element products do; a sum of element
// products in f32 (the tcgen05 GEMM's form) then misses it, so this kernel
// forms every isum_b exactly and folds it with its two scales.
//
// GB300 mapping.  tcgen05 has no integer kind on sm_103a, and a per-block
// fold of a tcgen05 accumulator (one FMA per output element per 32 K) would
// cost as much issue as the MMAs themselves; warp-level MMAs keep their
// accumulators in registers, where the fold is cheap.  The warp-level f16 MMA
// runs at ~4x the rate of the warp-level int8 MMA (about 605 vs 152 TFLOP/s
// measured), and every code (|q| <= 127) is exact in f16, as is every
// per-block sum (< 2^24 in the f32 accumulator), so the block sums are taken
// with mma.m16n8k16.f16 on integer-valued operands: still exact.  A small
// prologue kernel writes the activation operand once per call into the
// workspace: f16 codes [M][K] and f32 scales f(d_a) [M][K/32].
// The GEMM CTA owns a 128 x 128 output tile; a producer warp fetches per K
// chunk of 256 one 2-D TMA box of raw weight bytes (128 rows x 272 bytes = 8
// Q8_0 blocks per row), 128B-swizzled boxes of the f16 activation codes and a
// box of their scales; 8 consumer warps convert the weight codes to f16 in
// registers (exact), run the MMAs of one 32-value block with a zero
// accumulator and fold the block sum into the f32 result with f(d_w) f(d_a).
// (Packed f32x2 arithmetic and a 2x unroll of the block loop were measured
// slower on this kernel and are not used.)
#pragma once

#include "qmm_device.cuh"

namespace qmm {

constexpr int kPfWarps = 8;            // consumer warps (+1 producer)
constexpr int kPfBN = 128;             // weight rows per tile
constexpr int kPfKC = 256;             // K values per stage (8 Q8_0 blocks)
constexpr int kPfWRow = kPfKC / 32 * 34;  // raw bytes per weight row per stage (272)

struct PrefillParams {
    float* y;
    unsigned* err;
    int M, N, K;
    int bm;           // activation rows per tile (128)
    int n_mt, n_nt, ntiles;
    int kchunks;
    int stages;
    int stage_bytes;
    int off_w, off_a, off_s;  // offsets inside a stage
};

// byte offset of (row, half index h) in a [rows][64 halves] 128B-swizzled box
__device__ __forceinline__ int swz128(int row, int h) { return row * 128 + ((((h >> 3) ^ row) & 7) << 4); }

template <int WT>  // T_Q8_0
__global__ void __launch_bounds__((kPfWarps + 1) * 32, 1)
    qmm_prefill_kernel(const __grid_constant__ CUtensorMap tw, const __grid_constant__ CUtensorMap ta,
                       const __grid_constant__ CUtensorMap ts, const PrefillParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte alignment for the swizzled boxes
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = p.stages;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);  // full[S], empty[S]
    volatile int* flags = reinterpret_cast<volatile int*>(smem + 256);
    uint8_t* stage0 = smem + 1024;
    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(smem_u32(&bars[i]), 1);
            mbar_init(smem_u32(&bars[S + i]), kPfWarps);
        }
        flags[0] = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const int BM = p.bm;

    if (warp == kPfWarps) {
        // ------------------------------ producer ------------------------------
        if (lane != 0) return;
        long long g = 0;
        const uint32_t a_box = (uint32_t)BM * 128;  // bytes of one [BM][64 halves] box
        const uint32_t tx = (uint32_t)kPfBN * kPfWRow + a_box * 4 + (uint32_t)BM * 32;
        for (int t = blockIdx.x; t < p.ntiles; t += gridDim.x) {
            const int m0 = (t % p.n_mt) * BM, n0 = (t / p.n_mt) * kPfBN;
            bool ok = true;
            for (int kc = 0; kc < p.kchunks; ++kc, ++g) {
                const int slot = (int)(g % S);
                if (g >= S && !mbar_wait(smem_u32(&bars[S + slot]), (uint32_t)(((g / S) - 1) & 1), flags, p.err)) {
                    ok = false;
                    break;
                }
                uint8_t* st = stage0 + (long long)slot * p.stage_bytes;
                const uint32_t fb = smem_u32(&bars[slot]);
                mbar_arrive_tx(fb, tx);
                tma_2d(smem_u32(st + p.off_w), &tw, kc * (kPfWRow / 2), n0, fb);
                for (int s = 0; s < 4; ++s) tma_2d(smem_u32(st + p.off_a + s * a_box), &ta, kc * kPfKC + s * 64, m0, fb);
                tma_2d(smem_u32(st + p.off_s), &ts, kc * 8, m0, fb);
            }
            if (!ok) break;
        }
        const long long first = g > S ? g - S : 0;
        for (long long q = first; q < g; ++q) mbar_drain(smem_u32(&bars[q % S]), (uint32_t)((q / S) & 1), flags, p.err);
        return;
    }

    // ------------------------------ consumers ------------------------------
    // warps 2 (M) x 4 (N), warp tile 64 x 32 (4 m16 x 4 n8)
    constexpr int MI = 4;
    const int wm = warp >> 2, wn = warp & 3;
    const int g8 = lane >> 2, t4 = lane & 3;
    const int rp = ((g8 & 1) << 2) | (g8 >> 1);  // tile row of MMA row g (a permutation of 0..7)
    long long g = 0;
    for (int t = blockIdx.x; t < p.ntiles; t += gridDim.x) {
        const int m0 = (t % p.n_mt) * BM, n0 = (t / p.n_mt) * kPfBN;
        // acc[i][j][0] = (row g, cols 2t, 2t+1), acc[i][j][1] = (row g+8, ...): packed f32 pairs
        unsigned long long acc[MI][4][2];
#pragma unroll
        for (int i = 0; i < MI; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j][0] = acc[i][j][1] = 0ull;
        for (int kc = 0; kc < p.kchunks; ++kc, ++g) {
            const int slot = (int)(g % S);
            const bool ok = mbar_wait(smem_u32(&bars[slot]), (uint32_t)((g / S) & 1), flags, p.err);
            if (ok) {
                const uint8_t* st = stage0 + (long long)slot * p.stage_bytes;
                const uint8_t* W = st + p.off_w;
                const uint8_t* A = st + p.off_a;
                const float* SC = reinterpret_cast<const float*>(st + p.off_s);
#pragma unroll 1
                for (int b = 0; b < 8; ++b) {
                    // weight (B) fragments and scales of the warp's 4 n8 tiles
                    uint32_t bf[4][4];
                    unsigned long long dw[4];  // (f(d_w) of col 2t, of col 2t+1)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int nr = wn * 32 + 8 * j;
                        uint32_t w0, w1;
                        lds8_unaligned(W + (nr + g8) * kPfWRow + 34 * b + 2 + 8 * t4, w0, w1);
                        bf[j][0] = s8x2_to_h2(w0, SEL01);
                        bf[j][1] = s8x2_to_h2(w0, SEL23);
                        bf[j][2] = s8x2_to_h2(w1, SEL01);
                        bf[j][3] = s8x2_to_h2(w1, SEL23);
                        dw[j] = f2pack(h2f(*reinterpret_cast<const uint16_t*>(W + (nr + 2 * t4) * kPfWRow + 34 * b)),
                                       h2f(*reinterpret_cast<const uint16_t*>(W + (nr + 2 * t4 + 1) * kPfWRow + 34 * b)));
                    }
                    // activation (A) fragments: 8 halves at K offset 32b + 8t of rows g, g+8
                    const int hk = b * 32 + 8 * t4;        // half index inside the 256-value chunk
                    const int box = (hk >> 6) * BM * 128;  // which 64-half box
#pragma unroll
                    for (int i = 0; i < MI; ++i) {
                        // MMA row g holds tile row rperm(g): the rows a quarter-warp reads are 4 apart,
                        // so their 128B-swizzled chunks do not share banks
                        const int r0 = wm * (MI * 16) + 16 * i + rp, r1 = r0 + 8;
                        const uint4 x0 = ld128(A + box + swz128(r0, hk & 63));
                        const uint4 x1 = ld128(A + box + swz128(r1, hk & 63));
                        const float da0 = SC[r0 * 8 + b], da1 = SC[r1 * 8 + b];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            float d[4] = {0.f, 0.f, 0.f, 0.f};  // the block's exact integer sums
                            mma_f16(d, x0.x, x1.x, x0.y, x1.y, bf[j][0], bf[j][1]);
                            mma_f16(d, x0.z, x1.z, x0.w, x1.w, bf[j][2], bf[j][3]);
                            const float w0 = f2lo(dw[j]), w1 = f2hi(dw[j]);
                            acc[i][j][0] = f2pack(fmaf(d[0], da0 * w0, f2lo(acc[i][j][0])), fmaf(d[1], da0 * w1, f2hi(acc[i][j][0])));
                            acc[i][j][1] = f2pack(fmaf(d[2], da1 * w0, f2lo(acc[i][j][1])), fmaf(d[3], da1 * w1, f2hi(acc[i][j][1])));
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars[S + slot]));
        }
        if (flags[0]) continue;
        // store: thread owns (row g, cols 2t, 2t+1) and (row g+8, ...) of each m16 x n8 tile
#pragma unroll
        for (int i = 0; i < MI; ++i) {
            const int ra = m0 + wm * (MI * 16) + 16 * i + rp, rb = ra + 8;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int c = n0 + wn * 32 + 8 * j + 2 * t4;
                if (ra < p.M) {
                    if (c < p.N) p.y[(long long)ra * p.N + c] = f2lo(acc[i][j][0]);
                    if (c + 1 < p.N) p.y[(long long)ra * p.N + c + 1] = f2hi(acc[i][j][0]);
                }
                if (rb < p.M) {
                    if (c < p.N) p.y[(long long)rb * p.N + c] = f2lo(acc[i][j][1]);
                    if (c + 1 < p.N) p.y[(long long)rb * p.N + c + 1] = f2hi(acc[i][j][1]);
                }
            }
        }
    }
}

// activation prologue: the A operand of the prefill GEMM, written to the
// workspace; one thread per (row, 32-block): Q8_0 codes as f16, scale f(d)
template <int WT>  // T_Q8_0
__global__ void prefill_act_kernel(const float* __restrict__ x, int M, int K, __half* __restrict__ a,
                                   float* __restrict__ sc) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long nb = K / 32;
    if (i >= (long long)M * nb) return;
    const long long r = i / nb, b = i - r * nb;
    uint32_t c[8];
    float d;
    quant_q8_0_32(x + r * K + b * 32, c, d);
    uint32_t h[16];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        h[2 * k] = s8x2_to_h2(c[k], SEL01);
        h[2 * k + 1] = s8x2_to_h2(c[k], SEL23);
    }
    uint4* dst = reinterpret_cast<uint4*>(a + r * K + b * 32);
#pragma unroll
    for (int k = 0; k < 4; ++k) dst[k] = make_uint4(h[4 * k], h[4 * k + 1], h[4 * k + 2], h[4 * k + 3]);
    sc[r * nb + b] = h2f(f2h(d));
}

// ---------------------------------------------------------------------------
// host-side planning
// ---------------------------------------------------------------------------

struct PrefillPlan {
    PrefillParams p;
    int grid;
    size_t smem;
    size_t workspace;  // bytes of the activation operand
    size_t ws_a, ws_s;  // offsets in the workspace
};

inline bool plan_prefill(int wt, long long M, long long N, long long K, int sm_count, int smem_max, PrefillPlan& out) {
    if (wt != T_Q8_0 || K % kPfKC != 0 || M < 9 || K > (1 << 26) || M > (1 << 24) || N > (1 << 24)) return false;
    PrefillPlan pl{};
    PrefillParams& p = pl.p;
    p.M = (int)M;
    p.N = (int)N;
    p.K = (int)K;
    p.bm = 128;
    p.n_mt = (int)((M + p.bm - 1) / p.bm);
    p.n_nt = (int)((N + kPfBN - 1) / kPfBN);
    p.ntiles = p.n_mt * p.n_nt;
    p.kchunks = (int)(K / kPfKC);
    const int a_box = p.bm * 128;
    p.off_w = 0;
    p.off_a = round_up(kPfBN * kPfWRow, 1024);
    p.off_s = p.off_a + 4 * a_box;
    p.stage_bytes = round_up(p.off_s + p.bm * 32, 1024);
    const int base = 1024 + 1024;  // alignment slack + barriers
    const int stages = (smem_max - base) / p.stage_bytes;
    if (stages < 2) return false;
    p.stages = stages > 4 ? 4 : stages;
    pl.smem = (size_t)base + (size_t)p.stages * p.stage_bytes;
    pl.grid = p.ntiles < sm_count ? p.ntiles : sm_count;
    // workspace: activation planes (16-byte aligned pieces)
    pl.ws_a = 0;
    pl.ws_s = (size_t)M * K * 2;
    pl.workspace = pl.ws_s + (size_t)M * (K / 32) * 4;
    pl.workspace = (pl.workspace + 255) / 256 * 256;
    out = pl;
    return true;
}

}  // namespace qmm
