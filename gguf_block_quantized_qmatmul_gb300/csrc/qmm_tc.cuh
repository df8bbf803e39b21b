// qmm_tc.cuh -- the Metal form's prefill GEMM (f32_act, M > 16 activation
// rows) on the 5th-generation tensor cores: tcgen05.mma with the accumulator
// in tensor memory.
//
// "同一个 GGUF，CPU 和 Metal 生成的文字不一样" section 出处: the Metal form
// multiplies f32 activations by weights dequantized in the kernel,
//   y = sum_k x_k w_k, w = f(d) q (Q8_0), (f(d) sc) q - f(dmin) m (Q4_K),
//   f(d) (code - off) (Q4_0, Q5_0) or (f(d) sc) code (Q6_K).
// Its parity bound is taken over the element products x_k w_k, which an f32
// accumulation meets.  (The CPU form's bound is taken over block terms, which
// can cancel far more; it runs on kernels that form exact integer block
// sums.)  tcgen05 has no integer kind on sm_103a and its f16 kind carries 11
// bits per operand, so every operand is scaled by a power of two per row
// (activation rows and weight rows separately, into [2^14, 2^15) at the row
// maximum) and split into two f16 pieces, v = hi + lo (2^-22 relative); the
// product takes three MMAs, hi.hi + hi.lo + lo.hi (the dropped lo.lo is below
// 2^-22 relative), into an f32 accumulator restarted every kchunk raw stages
// (see kTcChunk1), and the epilogue multiplies by 2^-(s_row + s_col) and adds
// the chunks.
//
// One persistent CTA per SM over work units: an output tile of 128 weight
// rows x bx activation rows (bx <= 256, a multiple of 16, the MMA's N) and
// one of ks slices of K.  18 warps:
//   producer  TMA: raw weight rows (2-D box of 128 rows per 256 K: 272 B = 8
//             Q8_0 blocks, 144 B = 1 Q4_K super-block or 8 Q4_0 blocks, 176 B
//             = 8 Q5_0 blocks, or a 240-byte slot holding 1 Q6_K super-block;
//             up to six stages in flight) and the activation pieces (bx rows
//             x 64 f16, 128-byte swizzle, hi and lo, per 64 K: two 32-value
//             blocks per stage, so each handoff between roles covers two);
//   MMA       one thread: per 64-K stage twelve tcgen05.mma (M 128, N bx, K 16:
//             hi.hi, hi.lo, lo.hi, four K steps each) with the weights as the A
//             operand in tensor memory and the activation piece from shared
//             memory; it tests the next stage's barrier before issuing the
//             current one, so a ready stage costs no stall;
//   epilogue  8 warps, a TMEM lane quarter (32 weight rows) and half of the
//             accumulator columns each: tcgen05.ld, scale, y stores coalesced
//             along N (later chunks of the unit: added into y); with
//             K split, unscaled partial tiles in the workspace, and the unit
//             that completes a tile sums its ks partials in slice order
//             (deterministic) and writes y;
//   converter 8 warps in two groups (even and odd stages): each thread one
//             weight row's 64 values of a stage, read from the raw stage with
//             conflict-free 16-byte loads, dequantized, split into hi and lo,
//             written straight into tensor memory (tcgen05.st).
// TMEM: accumulators (two of 128 columns when bx <= 128, else one of 256) and
// two stages x 64 columns of weight pieces at column 256.
#pragma once

#include "qmm_device.cuh"

namespace qmm {

constexpr int kTcBW = 128;      // weight rows per tile (MMA M, the TMEM lanes)
constexpr int kTcBXMax = 256;   // activation rows per tile, at most (MMA N)
constexpr int kTcBK = 64;       // K per stage: two 32-value blocks, 128-byte swizzled activation rows
constexpr int kTcRK = 256;      // K per raw weight stage
constexpr int kTcSub = kTcRK / kTcBK;  // stages per raw stage
constexpr int kTcS = 2;         // stages: activation pieces in shared memory, weight pieces in TMEM
constexpr int kTcRSMax = 6;     // raw weight stages, at most
constexpr int kTcConvWarps = 8;
constexpr int kTcEpiWarps = 8;
constexpr int kTcThreads = (2 + kTcEpiWarps + kTcConvWarps) * 32;
constexpr int kTcTmemCols = 512;
constexpr int kTcWCol0 = 256;   // weight pieces: stage s at 256 + 64 s (hi 32 columns, lo 32 columns)
constexpr int kTcMaxSplit = 16;
// Accumulation chunks.  The tensor core's f32 accumulation truncates: its
// error grows with the number of MMAs chained into one accumulator and leans
// toward zero (measured: at 14336 x 4096, M = 1024, 768 chained MMAs put the
// worst output at 0.23 of the bound, 0.07 when the chains were eight times
// shorter).  A unit restarts its accumulator every `kchunk` raw stages and
// the epilogue adds the chunks' results into y in f32 with round-to-nearest.
// With two accumulators (bx <= 128) the epilogue drains one chunk while the
// MMAs fill the other: 1024 K.  With one, the MMAs wait for each drain: 4096 K.
// (Tiles of at most 192 rows, which would leave room for two accumulators,
// measured 35 % slower at M = 1024.)
constexpr int kTcChunk2 = 4, kTcChunk1 = 16;

struct TcParams {
    float* y;
    float* part;        // partial tiles [ks][M][N] when K is split
    unsigned* cnt;      // per-tile arrival counters when K is split (zeroed by the preparation launch)
    const float* ais;   // 2^-s per activation row
    const float* wis;   // 2^-s per weight row
    unsigned* err;
    int M, N, K;
    int bx;             // activation rows per tile (MMA N)
    int nacc;           // accumulators: 2 when bx <= 128
    int kchunk;         // raw stages per accumulation chunk
    int mtiles, ntiles, tiles;
    int ks, units;      // K slices; work units = tiles x ks
    int nrs;            // raw stages in K
    int raw_row;        // raw bytes per weight row per raw stage (272 Q8_0, 144 Q4_K)
    int raw_stage;      // bytes per raw stage (128 rows, rounded to 1 KB)
    int nraw;           // raw stages in shared memory
    int piece;          // bytes of one activation piece (bx rows x 64 B)
    int off_raw, off_bar;
};

// shared-memory matrix descriptor: K-major, 128-byte swizzle (rows of 64 f16), 8-row atoms 1 KB apart
__device__ __forceinline__ uint64_t tc_sdesc128(uint32_t addr) {
    return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) |
           ((uint64_t)2 << 61);
}
// instruction descriptor: f32 accumulator, f16 A and B, both K-major, M = 128, N = bx
__device__ __forceinline__ uint32_t tc_idesc(int bx) {
    return (1u << 4) | ((uint32_t)(bx >> 3) << 17) | ((uint32_t)(kTcBW >> 4) << 24);
}

// D (TMEM) += A (TMEM, 128 lanes x 16 f16) x B (shared memory)^T
__device__ __forceinline__ void tc_mma(uint32_t tmem, uint32_t ta, uint64_t db, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem),
        "r"(ta), "l"(db), "r"(idesc), "r"(accumulate)
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
// non-blocking test of an mbarrier phase; the result is consumed later
__device__ __forceinline__ uint32_t mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok;
}

// 16 f32 columns of this warp's TMEM lane quarter (the wait is separate)
__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t r[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------------------
// weight conversion: one thread, the 32 values of one weight row that one
// Q8_0 block or one Q4_K sub-block holds, scaled by 2^s, as 16 words of hi
// and 16 words of lo f16 pairs (k order natural)
// ---------------------------------------------------------------------------

// hi = f16(ds q) by one hmul2, lo = ds q - hi by one hfma2 (exact: at most 8
// significant bits remain), for the byte pair (2p, 2p+1) of a word of codes
__device__ __forceinline__ void tc_q8_pair(uint32_t word, int p, __half2 ds2, uint32_t& h, uint32_t& l) {
    uint32_t qb = __byte_perm(word, 0x64646464u, p ? 0x4342u : 0x4140u);  // bytes under 0x64: 1152 + q
    const __half2 q = __hsub2(*reinterpret_cast<__half2*>(&qb), __half2half2(__ushort_as_half(0x6480)));
    const __half2 hi = __hmul2(q, ds2);
    const __half2 lo = __hfma2(q, ds2, __hneg2(hi));
    h = *reinterpret_cast<const uint32_t*>(&hi);
    l = *reinterpret_cast<const uint32_t*>(&lo);
}

// Q8_0 block J (0..7) of a 272-byte raw row at row (16-byte aligned): w 2^s =
// ds q with ds = f(d) 2^s as f16 (exact while it is a normal f16).  The block
// sits at byte 34 J; three 16-byte loads cover it (rows 272 B apart make a
// quarter warp's 16-byte loads hit 32 distinct banks).
template <int J>
__device__ __forceinline__ void tc_conv_q8_0(const uint8_t* row, float wsc, uint32_t h[16], uint32_t l[16]) {
    constexpr int A = (34 * J) & ~15;  // first 16-byte chunk
    constexpr int O = 34 * J - A;      // byte offset of d in the chunk (even, < 16)
    const uint4 c0 = *reinterpret_cast<const uint4*>(row + A);
    const uint4 c1 = *reinterpret_cast<const uint4*>(row + A + 16);
    const uint4 c2 = *reinterpret_cast<const uint4*>(row + A + 32);
    const uint32_t w[12] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w, c2.x, c2.y, c2.z, c2.w};
    const uint32_t dbits = (w[O / 4] >> (8 * (O % 4))) & 0xFFFFu;
    const __half2 ds2 = __half2half2(__float2half_rn(h2f(dbits) * wsc));
    constexpr int QW = (O + 2) / 4, QS = 8 * ((O + 2) % 4);  // codes: word QW onward, shifted by QS bits
    static_assert(QW + 8 + (QS != 0 ? 1 : 0) <= 12, "the three chunks hold the block");
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t word;
        if constexpr (QS != 0) word = __funnelshift_r(w[QW + i], w[QW + i + 1], QS);
        else word = w[QW + i];
        word ^= 0x80808080u;  // codes biased by 128
        tc_q8_pair(word, 0, ds2, h[2 * i], l[2 * i]);
        tc_q8_pair(word, 1, ds2, h[2 * i + 1], l[2 * i + 1]);
    }
}

// Q4_K sub-block J (0..7) of the super-block at sbk (16-byte aligned): w 2^s =
// fma(e 2^s, q, -o 2^s) in f32 (one rounding, as the dequantization contract),
// split as f16(v) + f16(v - f16(v))
template <int J>
__device__ __forceinline__ void tc_conv_q4_k(const uint8_t* sbk, float wsc, uint32_t h[16], uint32_t l[16]) {
    constexpr int C = J >> 1, NIB = J & 1;  // byte 32 C + i holds sub-block 2 C (low nibble) and 2 C + 1 (high)
    const uint4 hd = *reinterpret_cast<const uint4*>(sbk);
    const float es = h2f(hd.x) * (float)q4k_sc(hd.y, hd.w, J) * wsc;
    const float os = h2f(hd.x >> 16) * (float)q4k_mn(hd.z, hd.w, J) * wsc;
    const uint4 q0 = *reinterpret_cast<const uint4*>(sbk + 16 + 32 * C);
    const uint4 q1 = *reinterpret_cast<const uint4*>(sbk + 16 + 32 * C + 16);
    const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t nb = (qw[i] >> (4 * NIB)) & 0x0F0F0F0Fu;  // values 4i..4i+3 of the sub-block
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

// Q4_0 / Q5_0 block J (0..7) of a raw row (144 / 176 bytes, 16-byte
// aligned): w 2^s = ds (code - off) with ds = f(d) 2^s as f16; the 4-bit
// fields (code j in the low nibble of byte j, code j + 16 in its high
// nibble) plus, for Q5_0, bit 4 from the block's word of fifth bits, biased
// to code - off + 128 and converted as the Q8_0 codes are.
template <int WT, int J>
__device__ __forceinline__ void tc_conv_x_0(const uint8_t* row, float wsc, uint32_t h[16], uint32_t l[16]) {
    constexpr int BB = WT == T_Q5_0 ? 22 : 18;    // bytes per block
    constexpr int QS = WT == T_Q5_0 ? 6 : 2;      // offset of the 16 nibble bytes
    constexpr int A = (BB * J) & ~15, O = BB * J - A;
    constexpr int NC = (O + BB + 15) / 16;        // 16-byte chunks covering the block
    uint32_t w[12];
#pragma unroll
    for (int c = 0; c < 3; ++c) {
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (c < NC) v = *reinterpret_cast<const uint4*>(row + A + 16 * c);
        w[4 * c] = v.x;
        w[4 * c + 1] = v.y;
        w[4 * c + 2] = v.z;
        w[4 * c + 3] = v.w;
    }
    const uint32_t dbits = (w[O / 4] >> (8 * (O % 4))) & 0xFFFFu;
    const __half2 ds2 = __half2half2(__float2half_rn(h2f(dbits) * wsc));
    constexpr int QW = (O + QS) / 4, QSH = 8 * ((O + QS) % 4);
    static_assert(QW + 4 + (QSH != 0 ? 1 : 0) <= 12, "the chunks hold the block");
    uint32_t q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (QSH != 0) q[i] = __funnelshift_r(w[QW + i], w[QW + i + 1], QSH);
        else q[i] = w[QW + i];
    }
    uint32_t hb = 0;
    if constexpr (WT == T_Q5_0) {
        constexpr int HW = (O + 2) / 4, HSH = 8 * ((O + 2) % 4);
        if constexpr (HSH != 0) hb = __funnelshift_r(w[HW], w[HW + 1], HSH);
        else hb = w[HW];
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        // values 4k..4k+3: low nibbles of word k (k < 4) or high nibbles of word k - 4
        uint32_t word = k < 4 ? (q[k & 3] & 0x0F0F0F0Fu) : ((q[k & 3] >> 4) & 0x0F0F0F0Fu);
        if constexpr (WT == T_Q5_0) {
            // bits 4k..4k+3 of the fifth-bit word to bit 4 of the four bytes (no overlapping copies)
            word |= ((((hb >> (4 * k)) & 0xFu) * 0x00204081u) & 0x01010101u) << 4;
            word += 0x70707070u;  // code - 16 + 128
        } else {
            word += 0x78787878u;  // code - 8 + 128
        }
        tc_q8_pair(word, 0, ds2, h[2 * k], l[2 * k]);
        tc_q8_pair(word, 1, ds2, h[2 * k + 1], l[2 * k + 1]);
    }
}

// Q6_K stage J (0..7) of a super-block repacked into a 240-byte slot at sbk
// (16-byte aligned; the preparation launch copies each 210-byte super-block
// there: ql[128], qh[64], 16 int8 group scales, f16 d).  Value l of the stage
// is value 32 J + l of the super-block: its low four bits are nibble
// (J % 4) / 2 of ql[64 (J / 4) + 32 (J % 2) + l], its high two bits are bits
// 2 (J % 4).. of qh[32 (J / 4) + l], the code is those six bits - 32, and its
// group is 2 J + l / 16.  w 2^s = (f(d) 2^s sc) code, exact in f32 (18 + 6
// bits), split as f16(v) + f16(v - f16(v)).
template <int J>
__device__ __forceinline__ void tc_conv_q6_k(const uint8_t* sbk, float wsc, uint32_t h[16], uint32_t l[16]) {
    constexpr int H = J >> 2, Q = J & 3;
    const uint4 a0 = *reinterpret_cast<const uint4*>(sbk + 64 * H + 32 * (Q & 1));
    const uint4 a1 = *reinterpret_cast<const uint4*>(sbk + 64 * H + 32 * (Q & 1) + 16);
    const uint4 b0 = *reinterpret_cast<const uint4*>(sbk + 128 + 32 * H);
    const uint4 b1 = *reinterpret_cast<const uint4*>(sbk + 128 + 32 * H + 16);
    const uint4 sc = *reinterpret_cast<const uint4*>(sbk + 192);
    const uint4 dd = *reinterpret_cast<const uint4*>(sbk + 208);
    const uint32_t scw = (J < 2 ? sc.x : J < 4 ? sc.y : J < 6 ? sc.z : sc.w) >> (16 * (J & 1));  // sc_2J, sc_2J+1
    const float fd = h2f(dd.x) * wsc;
    const float e0 = fd * (float)(int8_t)(scw & 0xFFu), e1 = fd * (float)(int8_t)((scw >> 8) & 0xFFu);
    const uint32_t qa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const uint32_t qb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t c = ((qa[i] >> (4 * (Q >> 1))) & 0x0F0F0F0Fu) | (((qb[i] >> (2 * Q)) & 0x03030303u) << 4);
        const float e = i < 4 ? e0 : e1;
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            const float v0 = e * (float)((int)((c >> (16 * p)) & 63u) - 32);
            const float v1 = e * (float)((int)((c >> (16 * p + 8)) & 63u) - 32);
            const __half2 hi = __floats2half2_rn(v0, v1);
            const float2 hf = __half22float2(hi);
            const __half2 lo = __floats2half2_rn(v0 - hf.x, v1 - hf.y);
            h[2 * i + p] = *reinterpret_cast<const uint32_t*>(&hi);
            l[2 * i + p] = *reinterpret_cast<const uint32_t*>(&lo);
        }
    }
}

// K slice `split` of ks: raw stages [r0, r1)
__device__ __forceinline__ void tc_slice(const TcParams& p, int split, int& r0, int& r1) {
    r0 = split * p.nrs / p.ks;
    r1 = (split + 1) * p.nrs / p.ks;
}

// one 32-value block J (0..7) of a raw stage: hi and lo pieces
template <int WT, int J>
__device__ __forceinline__ void tc_conv_block(const uint8_t* rrow, float wsc, uint32_t h[16], uint32_t l[16]) {
    if (WT == T_Q8_0) tc_conv_q8_0<J>(rrow, wsc, h, l);
    else if (WT == T_Q4_0 || WT == T_Q5_0) tc_conv_x_0<WT, J>(rrow, wsc, h, l);
    else if (WT == T_Q6_K) tc_conv_q6_k<J>(rrow, wsc, h, l);
    else tc_conv_q4_k<J>(rrow, wsc, h, l);
}

// one converter warp's share of a raw stage: stages G and G + 2 of the four
// it feeds (G = the warp's group; stage j holds blocks 2 j and 2 j + 1, their
// hi pieces in 32 TMEM columns, then their lo pieces); g0 = the global index
// of the raw stage's first stage
template <int WT, int G>
__device__ __forceinline__ bool tc_convert_raw(const uint8_t* rrow, float wsc, long long g0, uint32_t tq, uint32_t tmem,
                                               uint64_t* full, uint64_t* empty, volatile int* flags, unsigned* err,
                                               int lane) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int j = 2 * u + G;
        const long long g = g0 + j;
        const int s = (int)(g % kTcS);
        if (g >= kTcS && !mbar_wait(smem_u32(&empty[s]), (uint32_t)(((g / kTcS) - 1) & 1), flags, err)) return false;
        tc_fence_after();
        const uint32_t col = tmem + tq + (uint32_t)(kTcWCol0 + 64 * s);
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            uint32_t h[16], l[16];
            if (u == 0 && b == 0) tc_conv_block<WT, 2 * G>(rrow, wsc, h, l);
            else if (u == 0) tc_conv_block<WT, 2 * G + 1>(rrow, wsc, h, l);
            else if (b == 0) tc_conv_block<WT, 2 * G + 4>(rrow, wsc, h, l);
            else tc_conv_block<WT, 2 * G + 5>(rrow, wsc, h, l);
            tc_st16(col + 16 * b, h);
            tc_st16(col + 32 + 16 * b, l);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&full[s]));  // one of the group's four converter arrivals
    }
    return true;
}

// split-K fix-up of one tile by the 256 epilogue threads: thread t takes
// columns n0 + (t & 31) + 32 e (e < 4) and rows m0 + (t >> 5) + 8 j; per
// batch of four rows it loads up to four slices' sixteen values at once (64
// independent loads) and adds them in slice order, so the sum is the same
// on every run
__device__ __forceinline__ void tc_fixup(const TcParams& p, int t, int m0, int n0) {
    const int cl = t & 31, rg = t >> 5;
    const size_t slice = (size_t)p.M * p.N;
    float ws4[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int ne = n0 + cl + 32 * e;
        ws4[e] = ne < p.N ? __ldg(p.wis + ne) : 0.0f;
    }
    for (int j0 = 0; j0 < p.bx / 8; j0 += 4) {
        float acc[16];
        uint32_t okm = 0;  // element 4 u + e is in the tile and in y
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int mr = rg + 8 * (j0 + u), m = m0 + mr, ne = n0 + cl + 32 * e;  // rows of this tile only
                if (mr < p.bx && m < p.M && ne < p.N) okm |= 1u << (4 * u + e);
                acc[4 * u + e] = 0.0f;
            }
        const float* base = p.part + (size_t)(m0 + rg + 8 * j0) * p.N + n0 + cl;
        for (int s0 = 0; s0 < p.ks; s0 += 2) {
            float v[2][16];
#pragma unroll
            for (int sp = 0; sp < 2; ++sp)
#pragma unroll
                for (int el = 0; el < 16; ++el)
                    v[sp][el] = s0 + sp < p.ks && ((okm >> el) & 1u)
                                    ? __ldcg(base + (s0 + sp) * slice + (size_t)(8 * (el >> 2)) * p.N + 32 * (el & 3))
                                    : 0.0f;
#pragma unroll
            for (int sp = 0; sp < 2; ++sp)
#pragma unroll
                for (int el = 0; el < 16; ++el) acc[el] += v[sp][el];
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int mr = rg + 8 * (j0 + u), m = m0 + mr;
            if (mr >= p.bx || m >= p.M) continue;
            const float am = __ldg(p.ais + m);
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if ((okm >> (4 * u + e)) & 1u) p.y[(size_t)m * p.N + n0 + cl + 32 * e] = acc[4 * u + e] * ws4[e] * am;
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
    uint64_t* full = bars;                          // [kTcS] activation pieces landed and weight pieces in TMEM
    uint64_t* empty = full + kTcS;                  // [kTcS] stage consumed by the MMAs (commit)
    uint64_t* r_full = empty + kTcS;                // [kTcRSMax] raw weight rows landed (TMA)
    uint64_t* r_empty = r_full + kTcRSMax;          // [kTcRSMax] raw stage converted
    uint64_t* acc_full = r_empty + kTcRSMax;        // [2] accumulator complete (commit)
    uint64_t* acc_empty = acc_full + 2;             // [2] accumulator read (epilogue)
    uint64_t* epi_done = acc_empty + 2;             // partial tile stored (epilogue warps)
    uint64_t* fix_ready = epi_done + 1;             // arrival counted, fixflag set
    static_assert((2 * kTcS + 2 * kTcRSMax + 6) * 8 <= 256, "mbarriers overlap the TMEM slot");
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + p.off_bar + 256);
    volatile int* flags = reinterpret_cast<volatile int*>(sm + p.off_bar + 320);  // [0] abort, [1] fix-up owner
    if (tid == 0) {
        for (int i = 0; i < kTcS; ++i) {
            mbar_init(smem_u32(&full[i]), 1 + kTcConvWarps / 2);
            mbar_init(smem_u32(&empty[i]), 1);
        }
        for (int i = 0; i < kTcRSMax; ++i) {
            mbar_init(smem_u32(&r_full[i]), 1);
            mbar_init(smem_u32(&r_empty[i]), kTcConvWarps);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&acc_full[i]), 1);
            mbar_init(smem_u32(&acc_empty[i]), kTcEpiWarps);
        }
        mbar_init(smem_u32(epi_done), kTcEpiWarps);
        mbar_init(smem_u32(fix_ready), 1);
        flags[0] = 0;
        flags[1] = 0;
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

    auto stage = [&](int s) { return sm + s * 2 * p.piece; };  // activation hi | lo
    auto raw = [&](int s) { return sm + p.off_raw + s * p.raw_stage; };
    // unit u: tile u % tiles (weight rows (tile / mtiles) * 128.., activation
    // rows (tile % mtiles) * bx..), K slice u / tiles

    if (warp == 0) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            long long g = 0;            // stages issued
            long long ri = 0;           // raw stages issued
            int iu = blockIdx.x, ir = 0, ir1 = 0;  // raw-issue cursor: unit, raw stage, end
            if (iu < p.units) tc_slice(p, iu / p.tiles, ir, ir1);
            bool ok = true;
            long long rc = 0;           // raw stages whose activation stages are issued
            for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
                const int tile = u % p.tiles;
                const int m0 = (tile % p.mtiles) * p.bx;
                int r0, r1;
                tc_slice(p, u / p.tiles, r0, r1);
                for (int r = r0; r < r1 && ok; ++r, ++rc) {
                    // raw weight rows up to nraw - 1 raw stages ahead, across units
                    while (ok && iu < p.units && ri <= rc + p.nraw - 1) {
                        const int rs = (int)(ri % p.nraw);
                        if (ri >= p.nraw) ok = mbar_wait(smem_u32(&r_empty[rs]), (uint32_t)(((ri / p.nraw) - 1) & 1), flags, p.err);
                        if (!ok) break;
                        const int n0 = ((iu % p.tiles) / p.mtiles) * kTcBW;
                        mbar_arrive_tx(smem_u32(&r_full[rs]), (uint32_t)(kTcBW * p.raw_row));
                        tma_2d(smem_u32(raw(rs)), &tw, ir * (p.raw_row / 2), n0, smem_u32(&r_full[rs]));
                        ++ri;
                        if (++ir >= ir1) {
                            iu += gridDim.x;
                            if (iu < p.units) tc_slice(p, iu / p.tiles, ir, ir1);
                        }
                    }
                    for (int j = 0; j < kTcSub && ok; ++j, ++g) {
                        const int s = (int)(g % kTcS);
                        if (g >= kTcS) ok = mbar_wait(smem_u32(&empty[s]), (uint32_t)(((g / kTcS) - 1) & 1), flags, p.err);
                        if (!ok) break;
                        const int kx = (r * kTcSub + j) * kTcBK;
                        mbar_arrive_tx(smem_u32(&full[s]), (uint32_t)(2 * p.piece));
                        tma_2d(smem_u32(stage(s)), &tah, kx, m0, smem_u32(&full[s]));
                        tma_2d(smem_u32(stage(s) + p.piece), &tal, kx, m0, smem_u32(&full[s]));
                    }
                }
            }
            // let every copy this thread issued land before the CTA can exit
            for (long long q = (g > kTcS ? g - kTcS : 0); q < g; ++q)
                mbar_drain(smem_u32(&full[q % kTcS]), (uint32_t)((q / kTcS) & 1), flags, p.err);
            for (long long q = (ri > p.nraw ? ri - p.nraw : 0); q < ri; ++q)
                mbar_drain(smem_u32(&r_full[q % p.nraw]), (uint32_t)((q / p.nraw) & 1), flags, p.err);
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issuer ------------------------------
        if (lane == 0) {
            const uint32_t idesc = tc_idesc(p.bx);
            // stage 0's hi-piece descriptor in its 32-bit halves: a stage's and a K step's
            // offsets / 16 add to the start-address field (shared addresses are below 2^18)
            const uint64_t d0 = tc_sdesc128(smem_u32(stage(0)));
            const uint32_t lo0 = (uint32_t)d0, dhi = (uint32_t)(d0 >> 32);
            long long g = 0;
            int cc = 0;  // accumulation chunks issued
            bool ok = true;
            uint32_t ready = 0;  // the next stage's barrier, tested ahead
            for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
              int r0, r1;
              tc_slice(p, u / p.tiles, r0, r1);
              for (int c0 = r0; c0 < r1 && ok; c0 += p.kchunk, ++cc) {
                const int ab = p.nacc == 2 ? (cc & 1) : 0;
                const int use = p.nacc == 2 ? (cc >> 1) : cc;
                if (use > 0) ok = mbar_wait(smem_u32(&acc_empty[ab]), (uint32_t)((use - 1) & 1), flags, p.err);
                if (!ok) break;
                tc_fence_after();
                const uint32_t dt = tmem + (uint32_t)(ab * 128);
                const int nst = ((c0 + p.kchunk < r1 ? c0 + p.kchunk : r1) - c0) * kTcSub;
                for (int i = 0; i < nst; ++i, ++g) {
                    const int s = (int)(g % kTcS);
                    const uint32_t nxt = mbar_test(smem_u32(&full[(g + 1) % kTcS]), (uint32_t)(((g + 1) / kTcS) & 1));
                    if (!ready) ok = mbar_wait(smem_u32(&full[s]), (uint32_t)((g / kTcS) & 1), flags, p.err);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t xhi = lo0 + (uint32_t)((s * 2 * p.piece) >> 4), xlo = xhi + (uint32_t)(p.piece >> 4);
                    const uint32_t whi = tmem + (uint32_t)(kTcWCol0 + 64 * s), wlo = whi + 32;
#pragma unroll
                    for (int pass = 0; pass < 3; ++pass) {
                        // w_hi x_hi, w_hi x_lo, w_lo x_hi
                        const uint32_t wa = pass == 2 ? wlo : whi, xb = pass == 1 ? xlo : xhi;
#pragma unroll
                        for (int kk = 0; kk < kTcBK / 16; ++kk)
                            tc_mma(dt, wa + 8 * kk, ((uint64_t)dhi << 32) | (xb + 2 * kk), idesc, (i | pass | kk) != 0 ? 1u : 0u);
                    }
                    tc_commit(smem_u32(&empty[s]));
                    ready = nxt;
                }
                if (!ok) break;
                tc_commit(smem_u32(&acc_full[ab]));
              }
            }
            // the last commits must land before TMEM is released
            if (g > 0) mbar_drain(smem_u32(&empty[(g - 1) % kTcS]), (uint32_t)(((g - 1) / kTcS) & 1), flags, p.err);
        }
    } else if (warp < 2 + kTcEpiWarps) {
        // ------------------------------ epilogue ------------------------------
        const int ew = warp - 2;
        const int q = warp & 3;        // TMEM lane quarter: weight rows 32q..32q+31 of the tile
        const int half = ew >> 2;      // accumulator columns: 16-column chunks half, half + 2, ...
        const uint32_t tq = (uint32_t)(32 * q) << 16;
        const int nch = p.bx / 16;
        int cc = 0, fix = 0;  // accumulation chunks read; split-K fix-ups
        bool ok = true;
        for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
            const int tile = u % p.tiles, split = u / p.tiles;
            const int m0 = (tile % p.mtiles) * p.bx, n0 = (tile / p.mtiles) * kTcBW;
            const int n = n0 + 32 * q + lane;
            const bool nok = n < p.N;
            // the scales first: their loads complete while the accumulator fills; the
            // warp's activation-row scales (rows 16 c + i, c = half + 2 k) go to its own
            // 128-float area of shared memory
            const float wsn = nok && p.ks == 1 ? __ldg(p.wis + n) : 0.0f;
            float* asc = reinterpret_cast<float*>(sm + p.off_bar + 512) + ew * (kTcBXMax / 2);
            if (p.ks == 1) {
#pragma unroll
                for (int k = 0; k < kTcBXMax / 64; ++k) {
                    const int j = 32 * k + lane;                  // 0..127: chunk half + 2 (j >> 4), row j & 15
                    const int mr = 16 * (half + 2 * (j >> 4)) + (j & 15), m = m0 + mr;
                    asc[j] = mr < p.bx && m < p.M ? __ldg(p.ais + m) : 0.0f;
                }
            }
            float* dst = p.ks == 1 ? p.y : p.part + (size_t)split * p.M * p.N;
            int r0, r1;
            tc_slice(p, split, r0, r1);
            // the unit's accumulation chunks: the first stores its (scaled) result,
            // later ones add theirs to it (this thread wrote those elements itself)
            for (int c0 = r0; c0 < r1; c0 += p.kchunk, ++cc) {
                const bool first = c0 == r0;
                const int ab = p.nacc == 2 ? (cc & 1) : 0;
                const int use = p.nacc == 2 ? (cc >> 1) : cc;
                if (!(ok = mbar_wait(smem_u32(&acc_full[ab]), (uint32_t)(use & 1), flags, p.err))) break;
                tc_fence_after();
                __syncwarp();
                const uint32_t acol = tmem + tq + (uint32_t)(ab * 128);
                uint32_t r[16];
                if (half < nch) tc_ld16(acol + 16 * half, r);
                for (int c = half, k = 0; c < nch; c += 2, ++k) {
                    tc_wait_ld();
                    float v[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
                    if (c + 2 < nch) tc_ld16(acol + 16 * (c + 2), r);  // the next 16 columns' load overlaps the stores
                    const int mb = m0 + 16 * c;
                    if (nok && !flags[0]) {
                        float* yr = dst + (size_t)mb * p.N + n;
                        const float* ak = asc + 16 * k;
#pragma unroll
                        for (int i = 0; i < 16; ++i) v[i] = p.ks == 1 ? v[i] * wsn * ak[i] : v[i];
                        if (first) {
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                if (mb + i < p.M) yr[(size_t)i * p.N] = v[i];
                        } else {  // later chunks add to what this thread stored (four loads in flight:
                                  // 18 warps leave 96 registers a thread)
                            float* yp = yr;
#pragma unroll
                            for (int h = 0; h < 16; h += 4) {
                                float o[4];
#pragma unroll
                                for (int i = 0; i < 4; ++i) o[i] = mb + h + i < p.M ? yp[(size_t)i * p.N] : 0.0f;
#pragma unroll
                                for (int i = 0; i < 4; ++i)
                                    if (mb + h + i < p.M) yp[(size_t)i * p.N] = o[i] + v[h + i];
                                yp += (size_t)4 * p.N;
                            }
                        }
                    }
                }
                __syncwarp();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&acc_empty[ab]));
            }
            if (!ok) break;
            __syncwarp();  // the scale area is rewritten for the next unit
            if (p.ks > 1) {
                // the unit that completes the tile sums its ks partials in slice order
                __threadfence();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(epi_done));
                if (ew == 0 && lane == 0) {
                    int owner = 0;
                    if (mbar_wait(smem_u32(epi_done), (uint32_t)(fix & 1), flags, p.err)) {
                        __threadfence();
                        owner = atomicAdd(p.cnt + tile, 1u) == (unsigned)(p.ks - 1);
                    }
                    flags[1] = owner;
                    mbar_arrive(smem_u32(fix_ready));
                }
                if (!mbar_wait(smem_u32(fix_ready), (uint32_t)(fix & 1), flags, p.err)) break;
                ++fix;
                if (flags[1]) {
                    __threadfence();
                    tc_fixup(p, ew * 32 + lane, m0, n0);
                }
            }
        }
    } else {
        // ------------------------------ converters ------------------------------
        // warp cw: TMEM lane quarter cw & 3 (weight rows 32 (cw & 3) + lane), the
        // stages of parity cw >> 2 of every raw stage
        const int cw = warp - (2 + kTcEpiWarps);
        const int q = warp & 3, grp = cw >> 2;
        const int nrow = 32 * q + lane;
        const uint32_t tq = (uint32_t)(32 * q) << 16;
        long long g0 = 0, rg = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
            const int tile = u % p.tiles;
            const int n0 = (tile / p.mtiles) * kTcBW;
            const float wsc = n0 + nrow < p.N ? __frcp_rn(__ldg(p.wis + n0 + nrow)) : 1.0f;  // 2^s (exact)
            int r0, r1;
            tc_slice(p, u / p.tiles, r0, r1);
            for (int r = r0; r < r1 && ok; ++r, ++rg, g0 += kTcSub) {
                const int rs = (int)(rg % p.nraw);
                ok = mbar_wait(smem_u32(&r_full[rs]), (uint32_t)((rg / p.nraw) & 1), flags, p.err);
                if (!ok) break;
                const uint8_t* rrow = raw(rs) + nrow * p.raw_row;
                ok = grp == 0 ? tc_convert_raw<WT, 0>(rrow, wsc, g0, tq, tmem, full, empty, flags, p.err, lane)
                              : tc_convert_raw<WT, 1>(rrow, wsc, g0, tq, tmem, full, empty, flags, p.err, lane);
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&r_empty[rs]));
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

// blocks [0, M): activation rows; blocks [M, M + ceil(N / 8)): 8 weight rows each (a warp per row)
// Q6_K: every 210-byte super-block is also copied into a 240-byte slot of w6
// (rows of K / 256 slots), which the GEMM's tensor map reads: 210-byte blocks
// cannot start every copy on the 16-byte boundary a TMA copy needs.
constexpr int kTcQ6Slot = 240;
template <int WT>
__global__ void __launch_bounds__(kTcPrepThreads) tc_prep_kernel(const float* __restrict__ x, const uint8_t* __restrict__ wq,
                                                                 int M, int N, int K, __half* ahi, __half* alo,
                                                                 float* ais, float* wis, unsigned* cnt, int ncnt,
                                                                 uint8_t* __restrict__ w6) {
    grid_dep_launch();
    __shared__ float red[kTcPrepThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (blockIdx.x == 0)
        for (int i = tid; i < ncnt; i += kTcPrepThreads) cnt[i] = 0u;  // split-K arrival counters
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
        const float is = tc_row_iscale(amax);
        const float sc = __frcp_rn(is);
        if (tid == 0) ais[m] = is;
        __half* hr = ahi + (long long)m * K;
        __half* lr = alo + (long long)m * K;
        // thread t: values 16 g .. 16 g + 15 with g = t + 256 i (a Q8_0 block is two
        // neighbouring threads, a Q8K block sixteen); 32-byte stores of both pieces
        const int ng = K / 16;
        for (int g0 = 0; g0 < ng; g0 += kTcPrepThreads) {
            const int g = g0 + tid;
            const bool on = g < ng;
            float v[16];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 t = on ? __ldg(reinterpret_cast<const float4*>(xr + 16 * g) + i) : make_float4(0.f, 0.f, 0.f, 0.f);
                v[4 * i] = t.x;
                v[4 * i + 1] = t.y;
                v[4 * i + 2] = t.z;
                v[4 * i + 3] = t.w;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = __fmul_rn(v[i], sc);
            if (on) {
                uint32_t hw[8], lw[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const __half2 h = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
                    const float2 hf = __half22float2(h);
                    const __half2 l = __floats2half2_rn(v[2 * i] - hf.x, v[2 * i + 1] - hf.y);
                    hw[i] = *reinterpret_cast<const uint32_t*>(&h);
                    lw[i] = *reinterpret_cast<const uint32_t*>(&l);
                }
                uint4* ho = reinterpret_cast<uint4*>(hr + 16 * g);
                uint4* lo = reinterpret_cast<uint4*>(lr + 16 * g);
                ho[0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                ho[1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
                lo[0] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                lo[1] = make_uint4(lw[4], lw[5], lw[6], lw[7]);
            }
        }
    } else {
        // weight row scales: a bound on |w| per row from the block scales
        const long long n = (long long)(blockIdx.x - M) * (kTcPrepThreads / 32) + warp;
        if (n >= N) return;
        float bmax = 0.0f;
        if (is_b32(WT)) {
            // |w| <= |f(d)| times the largest |code|: 127 (Q8_0), 8 (Q4_0), 16 (Q5_0)
            constexpr int BB = WT == T_Q8_0 ? 34 : WT == T_Q5_0 ? 22 : 18;
            constexpr float CM = WT == T_Q8_0 ? 127.0f : WT == T_Q5_0 ? 16.0f : 8.0f;
            const uint8_t* row = wq + n * (long long)(K / 32) * BB;
            for (int b = lane; b < K / 32; b += 32) bmax = fmaxf(bmax, fabsf(h2f(*reinterpret_cast<const uint16_t*>(row + b * BB))) * CM);
        } else if (WT == T_Q6_K) {
            // |w| <= |f(d)| max_j |sc_j| 32; the row's super-blocks to their slots (2-byte words)
            const int nsb = K / 256;
            const uint8_t* row = wq + n * (long long)nsb * 210;
            for (int b = lane; b < nsb; b += 32) {
                const uint8_t* sb = row + b * 210;
                int scm = 0;
#pragma unroll
                for (int j = 0; j < 16; ++j) scm = max(scm, abs((int)(int8_t)__ldg(sb + 192 + j)));
                bmax = fmaxf(bmax, fabsf(h2f(__ldg(reinterpret_cast<const unsigned short*>(sb + 208)))) * (float)scm * 32.0f);
            }
            const uint16_t* src = reinterpret_cast<const uint16_t*>(row);
            uint16_t* dst = reinterpret_cast<uint16_t*>(w6 + n * (long long)nsb * kTcQ6Slot);
            for (int i = lane; i < nsb * 105; i += 32) {
                const int b = i / 105, hw = i - 105 * b;
                dst[b * (kTcQ6Slot / 2) + hw] = __ldg(src + i);
            }
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
    size_t ws_ahi, ws_alo, ws_ais, ws_wis, ws_part, ws_cnt, ws_w6, workspace;
};

// Modelled SM cycles of one work unit of `nr` raw stages (fitted to GB300
// timings): a 64-K stage costs twelve M 128 x N bx x K 16 MMAs at ~7 cycles
// per activation row, with a floor of ~800 cycles for the issuing thread at
// small N; a unit adds its accumulator hand-off (the epilogue's drain of a single
// accumulator stalls the MMAs); a split tile's last unit also sums the ks
// partial tiles, at ~24 B a cycle through L2.
inline double tc_unit_cycles(int bx, int nacc, int kchunk, int ks, int nr, bool last) {
    const double stage = bx * 7.0 > 800.0 ? bx * 7.0 : 800.0;
    const int chunks = (nr + kchunk - 1) / kchunk;  // one accumulator: the MMAs wait for each chunk's drain
    double c = nr * kTcSub * stage + (nacc == 1 ? 6000.0 * chunks : 1500.0);
    if (ks > 1 && last) c += ks * bx * (kTcBW * 4.0 / 24.0);
    return c;
}

inline bool plan_tc(int wt, long long M, long long N, long long K, int sm_count, int smem_max, TcPlan& out) {
    if (K % kTcRK != 0 || M < 9 || K > (1 << 26) || M > (1 << 24) || N > (1 << 24)) return false;
    TcPlan pl{};
    TcParams& p = pl.p;
    p.M = (int)M;
    p.N = (int)N;
    p.K = (int)K;
    p.mtiles = (int)((M + kTcBXMax - 1) / kTcBXMax);
    p.bx = round_up((int)((M + p.mtiles - 1) / p.mtiles), 16);
    p.nacc = p.bx <= 128 ? 2 : 1;
    p.kchunk = p.nacc == 2 ? kTcChunk2 : kTcChunk1;
    p.ntiles = (int)((N + kTcBW - 1) / kTcBW);
    p.tiles = p.mtiles * p.ntiles;
    p.nrs = (int)(K / kTcRK);
    p.raw_row = wt == T_Q8_0 ? kTcRK / 32 * 34 : wt == T_Q5_0 ? kTcRK / 32 * 22 : wt == T_Q6_K ? kTcQ6Slot : 144;  // Q4_K, Q4_0: 144
    p.raw_stage = round_up(kTcBW * p.raw_row, 1024);
    p.piece = p.bx * 128;
    p.off_raw = kTcS * 2 * p.piece;  // activation pieces; weight pieces live in TMEM
    const int fixed = 512 + kTcEpiWarps * kTcBXMax / 2 * 4 + 1024;  // barriers, TMEM slot, flags; epilogue scales; alignment slack
    p.nraw = (smem_max - p.off_raw - fixed) / p.raw_stage;
    if (p.nraw > kTcRSMax) p.nraw = kTcRSMax;
    if (p.nraw < 2) return false;
    p.off_bar = p.off_raw + p.nraw * p.raw_stage;
    pl.smem = (size_t)p.off_bar + fixed;
    // K slices: the smallest ks whose modelled makespan (units dealt round-robin
    // to one CTA per SM) is within 2 % of the best
    double best = 0.0;
    int best_ks = 1;
    const int kmax = p.nrs < kTcMaxSplit ? p.nrs : kTcMaxSplit;
    double cost[kTcMaxSplit + 1] = {};
    for (int ks = 1; ks <= kmax; ++ks) {
        const long long units = (long long)p.tiles * ks;
        const int grid = units < sm_count ? (int)units : sm_count;
        double worst = 0.0;
        for (int c = 0; c < grid; ++c) {
            double t = 0.0;
            for (long long u = c; u < units; u += grid) {
                const int split = (int)(u / p.tiles);
                const int nr = (split + 1) * p.nrs / ks - split * p.nrs / ks;
                t += tc_unit_cycles(p.bx, p.nacc, p.kchunk, ks, nr, split == ks - 1);
            }
            if (t > worst) worst = t;
        }
        cost[ks] = worst;
        if (ks == 1 || worst < best) best = worst;
    }
    for (int ks = 1; ks <= kmax; ++ks)
        if (cost[ks] <= best * 1.02) {
            best_ks = ks;
            break;
        }
    p.ks = best_ks;
    p.units = p.tiles * p.ks;
    pl.grid = p.units < sm_count ? p.units : sm_count;
    auto r256 = [](size_t v) { return (v + 255) / 256 * 256; };
    pl.ws_ahi = 0;
    pl.ws_alo = r256((size_t)M * K * 2);
    pl.ws_ais = pl.ws_alo + r256((size_t)M * K * 2);
    pl.ws_wis = pl.ws_ais + r256((size_t)M * 4);
    pl.ws_part = pl.ws_wis + r256((size_t)N * 4);
    pl.ws_cnt = pl.ws_part + (p.ks > 1 ? r256((size_t)p.ks * M * N * 4) : 0);
    pl.ws_w6 = pl.ws_cnt + (p.ks > 1 ? r256((size_t)p.tiles * 4) : 0);
    pl.workspace = pl.ws_w6 + (wt == T_Q6_K ? r256((size_t)N * (K / 256) * kTcQ6Slot) : 0);
    out = pl;
    return true;
}

}  // namespace qmm
