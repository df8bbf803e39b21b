// qmm_tcx.cuh -- the CPU form's prefill GEMM (int8_act, M > 16 activation
// rows; Q8_0, Q4_K and Q6_K weights) on the 5th-generation tensor cores with
// exact per-block sums; the same GEMM of exact weight codes also serves the
// Metal form (f32_act) up to 64 rows, with each activation row split into two
// f16 pieces (see TxRaw).
//
// "同一个 GGUF，CPU 和 Metal 生成的文字不一样" section 出处: the CPU form
// quantizes every activation row (Q8_0, or Q8K for K-quant weights) and
// multiplies it block by block as an integer dot product,
//   Q8_0: y = sum_b f(d_w) f(d_a) isum_b;
//   Q4_K: y = sum_s d_a (f(d) S_sc - f(dmin) S_m);   Q6_K: y = sum_s d_a f(d) S.
// Its parity bound is taken over the block (super-block) terms, so every
// isum_b, S_sc, S_m and S must be formed whole before it is scaled.
// sm_103a's tcgen05 has no integer kind, but integer codes are exact f16
// operands and integer partial sums below 2^24 are exact in the f32
// accumulator, so an MMA group with a restarted accumulator yields them:
//   Q8_0: one group per 32-value block (isum_b < 2^19);
//   Q4_K: one group per super-block on codes sc_j q (<= 945): S_sc (past
//         2^24 only for adversarial blocks, whose rounding stays inside the
//         bound); S_m as one more K 16 MMA of the m_j against the 16 sums of
//         16 activation codes;
//   Q6_K: its int8 group scales times codes reach 4064, not exact in f16, so
//         each scale is split sc_g = 16 a_g + b_g and the super-block takes
//         two groups, S_a on a_g q (|.| <= 256) and S_b on b_g q (<= 480),
//         each exact (< 2^24); S = 16 S_a + S_b.
// The fold, y += (block sum) x scales, is one scale product and one FMA per
// output element per block (Q8_0) or per super-block (Q4_K, Q6_K), in packed
// f32x2 arithmetic on the drained accumulators.
//
// One persistent CTA per SM over work units: an output tile of 128 weight
// rows (MMA M, the TMEM lanes) x NX = 64 or 128 activation rows (MMA N), over
// all of K or, with few tiles, one of ks K slices.  Block stages hold two
// 32-value blocks (64 K: 128-byte swizzled rows), so every handoff between
// roles covers two blocks.  22 warps:
//   producer   TMA: raw weight rows (2-D box of 128 rows x 256 K: 272 B of
//              Q8_0, 144 B of Q4_K, a 240-byte slot of Q6_K) with that
//              stretch's activation scales (prepared block-major) and, for
//              Q4_K, the sums of 16 codes, into a raw ring; per block stage
//              the activation codes (NX rows x 64 f16, 128-byte swizzle);
//   MMA        one thread: per block two (Q6_K: four) tcgen05.mma (K 16)
//              from shared memory into TMEM accumulators (a ring of 512
//              columns), restarted per block or super-block;
//   epilogue   16 warps, a TMEM lane quarter (32 weight rows) and NX / 4
//              accumulator columns each: drain the sums, fold them with the
//              weight scales (read from the raw stage) and the activation
//              scales, keep the tile's running sums in registers, store y
//              (or a partial tile) at the end;
//   converter  4 warps, one weight row per thread: each block's 32 codes to
//              exact f16, written to shared memory in the MMA's 128-byte
//              swizzled K-major layout.
// A raw stage is released when its blocks are converted and folded.
#pragma once

#include "qmm_tc.cuh"

namespace qmm {

constexpr int kTxW = 128;         // weight rows per tile (MMA M)
constexpr int kTxX = 128;         // activation rows per tile (MMA N), at most: 64 or 128
constexpr int kTxSMax = 8;        // block stages (weight codes + activation codes in shared memory), at most
constexpr int kTxTmemCols = 512;  // a ring of 512 / NX accumulators of NX columns
constexpr int kTxAccMax = kTxTmemCols / 64;
constexpr int kTxRawMax = 6;
constexpr int kTxMaxSplit = 16;   // K slices of a tile, at most
constexpr int kTxEpiWarps = 16;
constexpr int kTxConvWarps = 4;
constexpr int kTxThreads = (2 + kTxEpiWarps + kTxConvWarps) * 32;

// A raw stage holds 256 K of the tile's 128 weight rows and what the fold
// needs of the tile's 128 activation rows:
//   Q8_0: rows of 272 B (8 blocks); f(d_a) of the 8 blocks, [8][128] f32;
//   Q4_K: rows of 144 B (1 super-block); d_a, [128] f32; the min term's
//         activation operand (16 sums of 16 codes per row, f16, 32-byte
//         swizzle) and its weight operand (m_j twice each, written by the
//         converters);
//   Q6_K: rows of 240 B (1 super-block repacked into a 16-byte aligned slot);
//         d_a, [128] f32.
// A block stage holds the block's weight codes (Q6_K: two tiles, a_g q and
// b_g q, for the group scales split as sc_g = 16 a_g + b_g) and the 128
// activation rows' codes.
// The f32_act form (AM = A_F32) takes the same weight codes and each
// activation row scaled by a power of two and split into two f16 pieces,
// x 2^s = hi + lo: two MMAs per K step into one accumulator (Q4_K: the min
// term's sums of 16 values in two pieces as well); the fold needs no
// activation scale (2^-s is applied at the store).
template <int WT, int AM = A_INT8>
struct TxRaw {
    static constexpr bool b32 = WT == T_Q8_0 || WT == T_Q4_0 || WT == T_Q5_0;      // 32-value blocks, Q8_0 activations
    static constexpr int bb = WT == T_Q8_0 ? 34 : WT == T_Q5_0 ? 22 : 18;           // bytes per 32-value block
    static constexpr int pieces = AM == A_F32 ? 2 : 1;                             // activation pieces
    static constexpr int row = b32 ? 8 * bb : WT == T_Q4_K ? 144 : 240;
    static constexpr int scales = kTxW * row;                                      // f(d_a) (int8_act)
    static constexpr int bsum = WT == T_Q4_K ? scales + 1024 : 0;                  // Q4_K: pieces x [128][16] f16
    static constexpr int amin = WT == T_Q4_K ? bsum + pieces * kTxX * 32 : 0;     // Q4_K: [128][16] f16
    static constexpr int slot = b32 ? (scales + 8 * kTxX * 4 + 1023) / 1024 * 1024
                                : WT == T_Q4_K ? amin + kTxW * 32
                                               : (scales + kTxX * 4 + 1023) / 1024 * 1024;
    // bytes a raw stage's copies bring, for tiles of nx activation rows
    __host__ __device__ static constexpr int tx(int nx) {
        return AM == A_F32    ? kTxW * row + (WT == T_Q4_K ? pieces * nx * 32 : 0)
               : b32 ? kTxW * row + 8 * nx * 4
               : WT == T_Q4_K ? kTxW * row + nx * 4 + nx * 32
                              : kTxW * row + nx * 4;
    }
    // accumulators (drain units) per raw stage: Q8_0 one per block; Q4_K S_sc
    // and S_m; Q6_K S_a and S_b (S = 16 S_a + S_b)
    static constexpr int drains = b32 ? 8 : 2;
    static constexpr int wtiles = WT == T_Q6_K ? 2 : 1;  // weight-code tiles per block stage
    // 32-value blocks per block stage (2 or 4): every handoff between the
    // roles covers that many blocks.  A stage holds bps / 2 "atoms" of 64 K,
    // each 128-byte swizzled rows: a weight tile of 128 rows and an
    // activation tile of nx rows per atom.
    __host__ __device__ static constexpr int bps(int nx) {
        return AM == A_F32 ? (WT == T_Q4_K && nx == 64 ? 4 : 2) : WT == T_Q4_K || (b32 && nx == 64) ? 4 : 2;
    }
    __host__ __device__ static constexpr int atoms(int nx) { return bps(nx) / 2; }
    __host__ __device__ static constexpr int wtile(int nx) { return atoms(nx) * kTxW * 128; }  // bytes of a weight tile
    // activation tiles: piece p of atom a at p atoms(nx) + a
    __host__ __device__ static constexpr int stage(int nx) { return wtiles * wtile(nx) + pieces * atoms(nx) * nx * 128; }
    // block stages (a multiple of 8 KB each)
    __host__ __device__ static constexpr int stages(int nx) { return AM == A_INT8 && WT == T_Q4_K && bps(nx) == 2 ? 4 : 2; }
};
static_assert(TxRaw<T_Q8_0>::slot % 1024 == 0 && TxRaw<T_Q4_K>::slot % 1024 == 0 && TxRaw<T_Q6_K>::slot % 1024 == 0 &&
                  TxRaw<T_Q8_0, A_F32>::slot % 1024 == 0 && TxRaw<T_Q4_K, A_F32>::slot % 1024 == 0 &&
                  TxRaw<T_Q6_K, A_F32>::slot % 1024 == 0 && TxRaw<T_Q4_0>::slot % 1024 == 0 &&
                  TxRaw<T_Q5_0>::slot % 1024 == 0,
              "1 KB aligned raw slots");

struct TcxParams {
    float* y;
    unsigned* err;
    const float* ais;  // f32_act: 2^-s per activation row
    float* part;    // partial tiles [ks][M][N] when K is split
    unsigned* cnt;  // per-tile arrival counters when K is split (zeroed by the activation launch)
    int M, N, K;
    int mtiles, ntiles, tiles;
    int ks, units;  // K slices; work units = tiles x ks
    int nrs;        // raw stages in K (K / 256)
    int nraw;       // raw slots in shared memory
    int off_raw, off_bar;
};

// work unit u: tile u % tiles (weight rows n0 = (tile / mtiles) 128.., activation
// rows m0 = (tile % mtiles) NX..), K slice u / tiles: raw stages [r0, r1)
__device__ __forceinline__ void tcx_slice(const TcxParams& p, int u, int& tile, int& r0, int& r1) {
    tile = u % p.tiles;
    const int split = u / p.tiles;
    r0 = split * p.nrs / p.ks;
    r1 = (split + 1) * p.nrs / p.ks;
}

// D (TMEM) += A (shared memory) x B (shared memory)^T
__device__ __forceinline__ void tcx_mma(uint32_t tmem, uint64_t da, uint64_t db, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
        "l"(da), "l"(db), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 8 f32 columns of this warp's TMEM lane quarter (the wait is separate)
__device__ __forceinline__ void tcx_ld8(uint32_t taddr, uint32_t r[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}

// shared-memory matrix descriptor: K-major, 32-byte swizzle (rows of 16 f16), 8-row atoms 256 B apart
__device__ __forceinline__ uint64_t tcx_sdesc32(uint32_t addr) {
    return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((uint64_t)(256 >> 4) << 32) | ((uint64_t)1 << 46) |
           ((uint64_t)6 << 61);
}

// codes biased by 128 (4 bytes of code + 128) as two exact f16 pairs: bytes 0, 1 and 2, 3
__device__ __forceinline__ void tcx_codes_biased(uint32_t u, uint32_t& p01, uint32_t& p23) {
    uint32_t a = __byte_perm(u, 0x64646464u, 0x5140u), b = __byte_perm(u, 0x64646464u, 0x5342u);  // f16 1024 + (code + 128)
    const __half2 off = __half2half2(__ushort_as_half(0x6480));                                    // 1152
    const __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), off), hb = __hsub2(*reinterpret_cast<__half2*>(&b), off);
    p01 = *reinterpret_cast<const uint32_t*>(&ha);
    p23 = *reinterpret_cast<const uint32_t*>(&hb);
}

// signed codes of a word (4 bytes) as two exact f16 pairs: bytes 0, 1 and 2, 3
__device__ __forceinline__ void tcx_codes(uint32_t word, uint32_t& p01, uint32_t& p23) {
    tcx_codes_biased(word ^ 0x80808080u, p01, p23);
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

// Q4_K sub-block J (0..7) of the super-block at sbk (16-byte aligned) as 16
// words of exact f16 pairs sc_J q (at most 63 x 15 = 945): its codes are
// nibble J % 2 of bytes 16 + 32 (J / 2) .. + 31
template <int J>
__device__ __forceinline__ void tcx_conv_q4_k(const uint8_t* sbk, uint32_t h[16]) {
    const uint4 hd = *reinterpret_cast<const uint4*>(sbk);
    const float sc = (float)q4k_sc(hd.y, hd.w, J);
    const __half2 sc2 = __half2half2(__float2half_rn(sc));              // exact
    const __half2 nsc = __half2half2(__float2half_rn(-1024.0f * sc));  // exact: 1024 times a 6-bit integer
    const uint4 q0 = *reinterpret_cast<const uint4*>(sbk + 16 + 32 * (J >> 1));
    const uint4 q1 = *reinterpret_cast<const uint4*>(sbk + 32 + 32 * (J >> 1));
    const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t nb = (qw[i] >> (4 * (J & 1))) & 0x0F0F0F0Fu;  // values 4i..4i+3
        uint32_t a = __byte_perm(nb, 0x64646464u, 0x5140u), b = __byte_perm(nb, 0x64646464u, 0x5342u);  // 1024 + q
        // (1024 + q) sc - 1024 sc with one rounding: the exact q sc (at most 945)
        const __half2 ha = __hfma2(*reinterpret_cast<__half2*>(&a), sc2, nsc);
        const __half2 hb = __hfma2(*reinterpret_cast<__half2*>(&b), sc2, nsc);
        h[2 * i] = *reinterpret_cast<const uint32_t*>(&ha);
        h[2 * i + 1] = *reinterpret_cast<const uint32_t*>(&hb);
    }
}

// Q6_K stage J (0..7) of a super-block in its 240-byte slot at sbk (16-byte
// aligned: ql[128], qh[64], 16 int8 group scales, f16 d): values 32 J + l, l <
// 32, in groups 2 J (l < 16) and 2 J + 1.  Value 128 H + 32 Q + l (H = J / 4,
// Q = J % 4) takes its low 4 bits from nibble Q / 2 of ql[64 H + 32 (Q % 2) +
// l] and its high 2 bits from bits 2 Q, 2 Q + 1 of qh[32 H + l]; the code is
// the 6 bits less 32.  With sc_g = 16 a_g + b_g (a_g = sc_g >> 4 in [-8, 7],
// b_g = sc_g & 15), ha holds a_g code (|.| <= 256) and hb b_g code (<= 480),
// both exact f16: (1024 + u) t - 1056 t rounds once, to the exact (u - 32) t.
template <int J>
__device__ __forceinline__ void tcx_conv_q6_k(const uint8_t* sbk, uint32_t ha[16], uint32_t hb[16]) {
    constexpr int H = J >> 2, Q = J & 3;
    const uint4 l0 = *reinterpret_cast<const uint4*>(sbk + 64 * H + 32 * (Q & 1));
    const uint4 l1 = *reinterpret_cast<const uint4*>(sbk + 64 * H + 32 * (Q & 1) + 16);
    const uint4 h0 = *reinterpret_cast<const uint4*>(sbk + 128 + 32 * H);
    const uint4 h1 = *reinterpret_cast<const uint4*>(sbk + 128 + 32 * H + 16);
    const uint32_t scw = *reinterpret_cast<const uint32_t*>(sbk + 192 + 4 * (J >> 1)) >> (16 * (J & 1));  // sc_2J, sc_2J+1
    const uint32_t ql[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
    const uint32_t qh[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
    for (int e = 0; e < 2; ++e) {  // group 2 J + e: words 4 e .. 4 e + 3
        const int sc = (int)(int8_t)((scw >> (8 * e)) & 0xFFu);
        const float a = (float)(sc >> 4), b = (float)(sc & 15);
        const __half2 a2 = __half2half2(__float2half_rn(a)), na = __half2half2(__float2half_rn(-1056.0f * a));
        const __half2 b2 = __half2half2(__float2half_rn(b)), nb = __half2half2(__float2half_rn(-1056.0f * b));
#pragma unroll
        for (int i = 4 * e; i < 4 * e + 4; ++i) {
            const uint32_t u = ((ql[i] >> (4 * (Q >> 1))) & 0x0F0F0F0Fu) | (((qh[i] >> (2 * Q)) & 0x03030303u) << 4);
            uint32_t p = __byte_perm(u, 0x64646464u, 0x5140u), q = __byte_perm(u, 0x64646464u, 0x5342u);  // 1024 + u
            const __half2 xp = *reinterpret_cast<__half2*>(&p), xq = *reinterpret_cast<__half2*>(&q);
            const __half2 pa = __hfma2(xp, a2, na), qa = __hfma2(xq, a2, na);
            const __half2 pb = __hfma2(xp, b2, nb), qb = __hfma2(xq, b2, nb);
            ha[2 * i] = *reinterpret_cast<const uint32_t*>(&pa);
            ha[2 * i + 1] = *reinterpret_cast<const uint32_t*>(&qa);
            hb[2 * i] = *reinterpret_cast<const uint32_t*>(&pb);
            hb[2 * i + 1] = *reinterpret_cast<const uint32_t*>(&qb);
        }
    }
}

// Q4_0 / Q5_0 block J (0..7) of a raw row (144 / 176 bytes, 16-byte aligned)
// as 16 words of exact f16 code pairs, code - 8 (Q4_0) or code - 16 (Q5_0):
// the 4-bit fields (value j in the low nibble of byte j, value j + 16 in its
// high nibble) plus, for Q5_0, bit 4 from the block's word of fifth bits
template <int WT, int J>
__device__ __forceinline__ void tcx_conv_x_0(const uint8_t* row, uint32_t h[16]) {
    constexpr int BB = WT == T_Q5_0 ? 22 : 18;  // bytes per block
    constexpr int QS = WT == T_Q5_0 ? 6 : 2;    // offset of the 16 nibble bytes
    constexpr int A = (BB * J) & ~15, O = BB * J - A;
    constexpr int NC = (O + BB + 15) / 16;      // 16-byte chunks covering the block
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
            word |= ((((hb >> (4 * k)) & 0xFu) * 0x00204081u) & 0x01010101u) << 4;  // bit 4 of each byte
            word += 0x70707070u;  // code - 16 + 128
        } else {
            word += 0x78787878u;  // code - 8 + 128
        }
        tcx_codes_biased(word, h[2 * k], h[2 * k + 1]);
    }
}

// a 32-value block type's block J as exact f16 codes
template <int WT, int J>
__device__ __forceinline__ void tcx_conv_b32(const uint8_t* row, uint32_t h[16]) {
    if constexpr (WT == T_Q8_0) tcx_conv_q8_0<J>(row, h);
    else tcx_conv_x_0<WT, J>(row, h);
}

// f(d) of 32-value block j (BB bytes each, d first) of the raw row at `row`
template <int BB>
__device__ __forceinline__ float tcx_block_scale(const uint8_t* row, int j) {
    return h2f(*reinterpret_cast<const uint16_t*>(row + BB * j));
}

// K split: y of a tile (rows m0.., n0..) as the sum of its ks partial tiles in
// slice order, by the tile's last unit; thread t of the 16 epilogue warps
// takes column n0 + t % 128 and every fourth row from t / 128 (stores
// coalesced along N), four rows' loads of a slice in flight at a time
template <int NX>
__device__ __forceinline__ void tcx_fixup(const float* __restrict__ part, float* __restrict__ y, int M, int N, int ks,
                                          int t, int m0, int n0) {
    const int n = n0 + (t & (kTxW - 1));
    if (n >= N) return;
    const int r0 = t >> 7;
    const size_t slice = (size_t)M * N;
    for (int c = 0; c < NX / 4; c += 4) {
        float sum[4];
        for (int k = 0; k < ks; ++k) {
            const float* src = part + k * slice + n;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int m = m0 + r0 + 4 * (c + i);
                const float v = m < M ? __ldcg(src + (size_t)m * N) : 0.0f;
                sum[i] = k == 0 ? v : sum[i] + v;
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int m = m0 + r0 + 4 * (c + i);
            if (m < M) y[(size_t)m * N + n] = sum[i];
        }
    }
}

// tensor maps: tw raw weight rows; ta activation codes (f32_act: the hi pieces); ts
// int8_act: activation scales, f32_act: the lo pieces; tb Q4_K: sums of 16 codes
// (f32_act: hi sums, then lo sums, along each row)
template <int WT, int NX, int AM>  // T_Q8_0, T_Q4_0, T_Q5_0 (int8_act), T_Q4_K or T_Q6_K; tiles of NX = 64 or 128 rows; A_INT8 or A_F32
__global__ void __launch_bounds__(kTxThreads, 1)
    qmm_tcx_kernel(const __grid_constant__ CUtensorMap tw, const __grid_constant__ CUtensorMap ta,
                   const __grid_constant__ CUtensorMap ts, const __grid_constant__ CUtensorMap tb, const TcxParams p) {
    using R = TxRaw<WT, AM>;
    constexpr bool kF32 = AM == A_F32;
    constexpr bool kB32 = R::b32;  // Q8_0, Q4_0, Q5_0: a fold per 32-value block
    static_assert(NX == 64 || NX == 128, "tile widths");
    constexpr int kAcc = kTxTmemCols / NX;  // TMEM accumulators
    constexpr int CW = NX / 4;              // accumulator columns an epilogue warp drains
    extern __shared__ __align__(1024) uint8_t smraw[];
    uint8_t* sm = smraw + ((1024 - (smem_u32(smraw) & 1023)) & 1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + p.off_bar);
    constexpr int kTxS = R::stages(NX);
    static_assert(kTxS <= kTxSMax, "block stages");
    uint64_t* full = bars;                       // [kTxS] activation codes landed and weight codes converted
    uint64_t* empty = full + kTxS;               // [kTxS] stage consumed by the MMAs (commit)
    uint64_t* r_full = empty + kTxS;             // [kTxRawMax] raw stage landed (TMA)
    uint64_t* r_empty = r_full + kTxRawMax;      // [kTxRawMax] raw stage converted and folded
    uint64_t* min_ready = r_empty + kTxRawMax;   // [kTxRawMax] Q4_K: the min term's weight operand written
    uint64_t* acc_full = min_ready + kTxRawMax;  // [kAcc] accumulator complete (commit)
    uint64_t* acc_empty = acc_full + kAcc;       // [kAcc] accumulator drained (epilogue)
    uint64_t* epi_done = acc_empty + kAcc;       // K split: the unit's partial tile stored (epilogue warps)
    uint64_t* fix_ready = epi_done + 1;          // K split: whether this CTA completes the tile is known
    static_assert((2 * kTxSMax + 3 * kTxRawMax + 2 * kTxAccMax + 2) * 8 <= 448, "mbarriers overlap the TMEM slot");
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + p.off_bar + 448);
    volatile int* flags = reinterpret_cast<volatile int*>(sm + p.off_bar + 480);  // [0] abort, [1] tile owner
    if (tid == 0) {
        for (int i = 0; i < kTxS; ++i) {
            mbar_init(smem_u32(&full[i]), 1 + kTxConvWarps);
            mbar_init(smem_u32(&empty[i]), 1);
        }
        for (int i = 0; i < kTxRawMax; ++i) {
            mbar_init(smem_u32(&r_full[i]), 1);
            mbar_init(smem_u32(&r_empty[i]), kTxConvWarps + kTxEpiWarps);
            mbar_init(smem_u32(&min_ready[i]), kTxConvWarps);
        }
        for (int i = 0; i < kAcc; ++i) {
            mbar_init(smem_u32(&acc_full[i]), 1);
            mbar_init(smem_u32(&acc_empty[i]), kTxEpiWarps);
        }
        mbar_init(smem_u32(epi_done), kTxEpiWarps);
        mbar_init(smem_u32(fix_ready), 1);
        flags[0] = 0;
        flags[1] = 0;
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

    auto wstage = [&](int s) { return sm + s * R::stage(NX); };                            // A: weight codes (Q6_K: a q, then b q)
    auto xstage = [&](int s) { return sm + s * R::stage(NX) + R::wtiles * R::wtile(NX); };  // B: activation codes
    constexpr int kBps = R::bps(NX);        // blocks per block stage
    constexpr int kSpr = 8 / kBps;          // block stages per raw stage
    // Drain groups: accumulators handed from the MMAs to the epilogue with one
    // commit and returned with one release (barriers 0 .. kGrp - 1).  A super-block's
    // two (Q4_K S_sc and S_m, Q6_K S_a and S_b) are one group; so are a block
    // stage's 32-value blocks at 64-row tiles (two or four), whose epilogue loads
    // two of them before each wait; 128-row tiles, with half as many accumulators
    // and twice the columns, hand each 32-value block over alone.
    constexpr int kG = kB32 ? (NX == 128 ? 1 : kBps) : 2;
    constexpr int kL = kB32 && NX == 128 ? 1 : 2;  // 32-value blocks per TMEM load round trip
    constexpr int kGrp = kAcc / kG;
    static_assert(kBps % kG == 0 && kAcc % kG == 0, "accumulator groups");
    auto raw = [&](int s) { return sm + p.off_raw + s * R::slot; };

    if (warp == 0) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            long long g = 0, ri = 0, rc = 0;  // blocks issued; raw stages issued; raw stages whose blocks are issued
            int iu = blockIdx.x, ir = 0, ir1 = 0, itile = 0;  // raw-issue cursor: unit, raw stage, its slice's end, tile
            if (iu < p.units) tcx_slice(p, iu, itile, ir, ir1);
            bool ok = true;
            for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
                int tile, r0, r1;
                tcx_slice(p, u, tile, r0, r1);
                const int m0 = (tile % p.mtiles) * NX;
                for (int r = r0; r < r1 && ok; ++r, ++rc) {
                    // raw stages up to nraw - 2 ahead, across units: the slot a new stage
                    // reuses is then two stages old, one the epilogue has finished folding
                    // (waiting on a younger one would hold back this stage's activations)
                    while (ok && iu < p.units && ri <= rc + p.nraw - 2) {
                        const int rs = (int)(ri % p.nraw);
                        if (ri >= p.nraw) ok = mbar_wait(smem_u32(&r_empty[rs]), (uint32_t)(((ri / p.nraw) - 1) & 1), flags, p.err);
                        if (!ok) break;
                        const int in0 = (itile / p.mtiles) * kTxW, im0 = (itile % p.mtiles) * NX;
                        const uint32_t fb = smem_u32(&r_full[rs]);
                        mbar_arrive_tx(fb, (uint32_t)R::tx(NX));
                        tma_2d(smem_u32(raw(rs)), &tw, ir * (R::row / 2), in0, fb);
                        if (kF32) {
                            if (WT == T_Q4_K) {
                                tma_2d(smem_u32(raw(rs) + R::bsum), &tb, 16 * ir, im0, fb);
                                tma_2d(smem_u32(raw(rs) + R::bsum + kTxX * 32), &tb, p.K / 16 + 16 * ir, im0, fb);
                            }
                        } else if (kB32) {
                            tma_2d(smem_u32(raw(rs) + R::scales), &ts, im0, 8 * ir, fb);
                        } else {
                            tma_2d(smem_u32(raw(rs) + R::scales), &ts, im0, ir, fb);
                            if (WT == T_Q4_K) tma_2d(smem_u32(raw(rs) + R::bsum), &tb, 16 * ir, im0, fb);
                        }
                        ++ri;
                        if (++ir >= ir1) {
                            iu += gridDim.x;
                            if (iu < p.units) tcx_slice(p, iu, itile, ir, ir1);
                        }
                    }
                    for (int j = 0; j < kSpr && ok; ++j, ++g) {  // block stages: blocks kBps j ..
                        const int s = (int)(g % kTxS);
                        if (g >= kTxS) ok = mbar_wait(smem_u32(&empty[s]), (uint32_t)(((g / kTxS) - 1) & 1), flags, p.err);
                        if (!ok) break;
                        mbar_arrive_tx(smem_u32(&full[s]), (uint32_t)(R::pieces * NX * 64 * kBps));
#pragma unroll
                        for (int a = 0; a < kBps / 2; ++a) {  // one box of 64 K per atom (and piece)
                            tma_2d(smem_u32(xstage(s) + a * NX * 128), &ta, (r * 8 + kBps * j + 2 * a) * 32, m0,
                                   smem_u32(&full[s]));
                            if (kF32)
                                tma_2d(smem_u32(xstage(s) + (kBps / 2 + a) * NX * 128), &ts, (r * 8 + kBps * j + 2 * a) * 32, m0,
                                       smem_u32(&full[s]));
                        }
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
            const uint32_t idesc = tc_idesc(NX);
            // shared-memory descriptors of stage 0's weight and activation tiles, split in
            // their 32-bit halves; the high half is the same for every 128-byte-swizzled tile
            const uint64_t d0w = tc_sdesc128(smem_u32(wstage(0))), d0x = tc_sdesc128(smem_u32(xstage(0)));
            const uint32_t wlo0 = (uint32_t)d0w, xlo0 = (uint32_t)d0x, dhi = (uint32_t)(d0w >> 32);
            long long g = 0, rg = 0;  // blocks; raw stages
            uint32_t du = 0;          // drain units (a launch drains far fewer than 2^32)
            bool ok = true;
            uint32_t ready = 0;  // the next stage's barrier, tested ahead
            for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
                int tile, r0, r1;
                tcx_slice(p, u, tile, r0, r1);
                for (int r = r0; r < r1 && ok; ++r, ++rg) {
                    // super-blocks: S_sc and S_m (Q4_K), S_a and S_b (Q6_K), once the epilogue
                    // drained the group's last use
                    const uint32_t dcol = (uint32_t)((du % kAcc) * NX), dcol2 = (uint32_t)(((du + 1) % kAcc) * NX);
                    if (!kB32 && du >= kAcc)
                        ok = mbar_wait(smem_u32(&acc_empty[(du / kG) % kGrp]), (uint32_t)(((du / kAcc) - 1) & 1), flags, p.err);
                    for (int j = 0; j < kSpr && ok; ++j, ++g) {  // block stages: blocks kBps j ..
                        const int s = (int)(g % kTxS);
                        uint32_t dq[kBps];  // Q8_0: the accumulator of each block of the stage
                        const uint32_t d0 = du + kBps * j;  // the stage's first accumulator (a group start)
                        if (kB32) {
#pragma unroll
                            for (int b = 0; b < kBps; b += kG)
                                if (ok && d0 + b >= kAcc)
                                    ok = mbar_wait(smem_u32(&acc_empty[((d0 + b) / kG) % kGrp]),
                                                   (uint32_t)((((d0 + b) / kAcc) - 1) & 1), flags, p.err);
#pragma unroll
                            for (int b = 0; b < kBps; ++b) dq[b] = (uint32_t)(((d0 + b) % kAcc) * NX);
                        }
                        if (!ok) break;
                        const uint32_t nxt = mbar_test(smem_u32(&full[(g + 1) % kTxS]), (uint32_t)(((g + 1) / kTxS) & 1));
                        if (!ready) ok = mbar_wait(smem_u32(&full[s]), (uint32_t)((g / kTxS) & 1), flags, p.err);
                        if (!ok) break;
                        tc_fence_after();
                        // the stage's descriptors: the base's, plus the byte offset / 16 in the
                        // start-address field (no carry: shared addresses are below 2^18)
                        const uint32_t wlo = wlo0 + (uint32_t)s * (R::stage(NX) >> 4), xlo = xlo0 + (uint32_t)s * (R::stage(NX) >> 4);
                        auto desc = [&](uint32_t lo, uint32_t off) { return ((uint64_t)dhi << 32) | (lo + (off >> 4)); };
                        // K = 16 steps ks: atom ks / 4, 32 bytes each along its 128-byte swizzled rows
#pragma unroll
                        for (int ks = 0; ks < 2 * kBps; ++ks) {
                            const uint32_t col = kB32 ? dq[ks >> 1] : dcol;
                            const uint32_t accu = kB32 ? (uint32_t)(ks & 1) : (uint32_t)(j | ks);
                            const uint32_t wk = (ks >> 2) * kTxW * 128 + 32 * (ks & 3);
                            const uint32_t xk = (ks >> 2) * NX * 128 + 32 * (ks & 3);
                            tcx_mma(tmem + col, desc(wlo, wk), desc(xlo, xk), idesc, accu);
                            if (kF32)  // the lo piece into the same accumulator
                                tcx_mma(tmem + col, desc(wlo, wk), desc(xlo, xk + (kBps / 2) * NX * 128), idesc, 1u);
                            if (WT == T_Q6_K) {
                                tcx_mma(tmem + dcol2, desc(wlo, wk + R::wtile(NX)), desc(xlo, xk), idesc, accu);
                                if (kF32)
                                    tcx_mma(tmem + dcol2, desc(wlo, wk + R::wtile(NX)), desc(xlo, xk + (kBps / 2) * NX * 128), idesc, 1u);
                            }
                        }
                        tc_commit(smem_u32(&empty[s]));
                        if (kB32) {
#pragma unroll
                            for (int b = 0; b < kBps; b += kG) tc_commit(smem_u32(&acc_full[((d0 + b) / kG) % kGrp]));
                        }
                        ready = nxt;
                    }
                    if (!ok) break;
                    if (WT == T_Q6_K) tc_commit(smem_u32(&acc_full[(du / kG) % kGrp]));
                    if (WT == T_Q4_K) {
                        // S_m = sum_j m_j bsum_j: one K 16 MMA over the 16 sums of 16 codes
                        const uint32_t mcol = dcol2;
                        const int rs = (int)(rg % p.nraw);
                        if (ok) ok = mbar_wait(smem_u32(&min_ready[rs]), (uint32_t)((rg / p.nraw) & 1), flags, p.err);
                        if (!ok) break;
                        tc_fence_after();
                        tcx_mma(tmem + mcol, tcx_sdesc32(smem_u32(raw(rs) + R::amin)), tcx_sdesc32(smem_u32(raw(rs) + R::bsum)),
                                idesc, 0u);
                        if (kF32)
                            tcx_mma(tmem + mcol, tcx_sdesc32(smem_u32(raw(rs) + R::amin)),
                                    tcx_sdesc32(smem_u32(raw(rs) + R::bsum + kTxX * 32)), idesc, 1u);
                        tc_commit(smem_u32(&acc_full[(du / kG) % kGrp]));
                    }
                    du += R::drains;
                }
            }
            // the last commits must land before TMEM is released
            if (g > 0) mbar_drain(smem_u32(&empty[(g - 1) % kTxS]), (uint32_t)(((g - 1) / kTxS) & 1), flags, p.err);
            if (du > 0)
                mbar_drain(smem_u32(&acc_full[((du - 1) / kG) % kGrp]),
                           (uint32_t)(((du - 1) / kAcc) & 1), flags, p.err);
        }
    } else if (warp < 2 + kTxEpiWarps) {
        // ------------------------------ epilogue ------------------------------
        const int ew = warp - 2;
        const int q = warp & 3;   // TMEM lane quarter: weight rows 32q..32q+31 of the tile
        const int cq = ew >> 2;   // accumulator columns CW cq..CW cq + CW - 1: activation rows of the tile
        const uint32_t tq = (uint32_t)(32 * q) << 16;
        const int nl = 32 * q + lane;  // this thread's weight row in the tile
        // drain units: a launch drains far fewer than 2^32 accumulators
        uint32_t du = 0;
        long long rg = 0;
        bool ok = true;
        // a super-block's group: wait for it, then the columns of its two accumulators
        auto grp_wait = [&](uint32_t d) {
            ok = mbar_wait(smem_u32(&acc_full[(d / kG) % kGrp]), (uint32_t)((d / kAcc) & 1), flags, p.err);
            return tmem + tq + (uint32_t)((d % kAcc) * NX + CW * cq);
        };
        auto grp_release = [&](uint32_t d) {  // after the group's last TMEM load completed
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&acc_empty[(d / kG) % kGrp]));
        };
        // 8-column pieces a super-block's drain loads per TMEM round trip: all of them
        // at 64-row tiles, one at a time at 128 (the running sums hold 2 CW registers)
        constexpr int kH = NX == 64 ? CW / 8 : 1;
        for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
            int r0, r1;
            {
                int tile_;
                tcx_slice(p, u, tile_, r0, r1);
            }
            unsigned long long acc[CW / 2];  // running sums of activation rows CW cq + 2i, 2i + 1
#pragma unroll
            for (int i = 0; i < CW / 2; ++i) acc[i] = 0ull;
            for (int r = r0; r < r1 && ok; ++r, ++rg) {
                const int rs = (int)(rg % p.nraw);
                const uint8_t* wrow = raw(rs) + nl * R::row;
                const float* asc = reinterpret_cast<const float*>(raw(rs) + R::scales) + CW * cq;
                if (kB32) {
                    for (int j = 0; j < 8; j += kG, du += kG) {  // a drain group: blocks j .. j + kG - 1
                        ok = mbar_wait(smem_u32(&acc_full[(du / kG) % kGrp]), (uint32_t)((du / kAcc) & 1), flags, p.err);
                        if (!ok) break;
                        tc_fence_after();
                        __syncwarp();
#pragma unroll
                        for (int l0 = 0; l0 < kG; l0 += kL) {  // kL blocks per TMEM load round trip
                            uint32_t vv[kL][CW];
#pragma unroll
                            for (int b = 0; b < kL; ++b) {
                                const uint32_t acol = tmem + tq + (uint32_t)(((du + l0 + b) % kAcc) * NX + CW * cq);
#pragma unroll
                                for (int h = 0; h < CW / 16; ++h) tc_ld16(acol + 16 * h, vv[b] + 16 * h);
                            }
                            tc_wait_ld();
                            if (l0 + kL >= kG) {
                                tc_fence_before();  // the group's accumulators go back to the MMAs
                                __syncwarp();
                                if (lane == 0) mbar_arrive(smem_u32(&acc_empty[(du / kG) % kGrp]));
                            }
#pragma unroll
                            for (int b = 0; b < kL; ++b) {
                                // fold: y += isum f(d_w) f(d_a)
                                const float dw = tcx_block_scale<R::bb>(wrow, j + l0 + b);
                                const unsigned long long dw2 = f2pack(dw, dw);
                                const float* aj = asc + (j + l0 + b) * NX;
#pragma unroll
                                for (int c = 0; c < CW / 4; ++c) {
                                    const uint32_t* v = vv[b] + 4 * c;
                                    if constexpr (kF32) {  // y 2^s += S f(d_w) (sums of x 2^s)
                                        acc[2 * c] = fma2(f2pack(__uint_as_float(v[0]), __uint_as_float(v[1])), dw2, acc[2 * c]);
                                        acc[2 * c + 1] = fma2(f2pack(__uint_as_float(v[2]), __uint_as_float(v[3])), dw2, acc[2 * c + 1]);
                                    } else {
                                        const float4 a4 = *reinterpret_cast<const float4*>(aj + 4 * c);
                                        const unsigned long long s01 = mul2(f2pack(a4.x, a4.y), dw2), s23 = mul2(f2pack(a4.z, a4.w), dw2);
                                        acc[2 * c] = fma2(f2pack(__uint_as_float(v[0]), __uint_as_float(v[1])), s01, acc[2 * c]);
                                        acc[2 * c + 1] = fma2(f2pack(__uint_as_float(v[2]), __uint_as_float(v[3])), s23, acc[2 * c + 1]);
                                    }
                                }
                            }
                        }
                    }
                } else if (WT == T_Q6_K) {
                    // y += d_a f(d) S with S = 16 S_a + S_b (S_a, S_b exact integers in f32;
                    // 16 S_a exact, the sum rounded once, relative to |S|)
                    const uint32_t ca = grp_wait(du);
                    const uint32_t cb = ca + NX;  // the group's second accumulator (du is even)
                    if (!ok) break;
                    tc_fence_after();
                    __syncwarp();
                    const float fd = h2f(*reinterpret_cast<const uint16_t*>(wrow + 208));
                    const unsigned long long fd2 = f2pack(fd, fd), k16 = f2pack(16.0f, 16.0f);
#pragma unroll
                    for (int h0 = 0; h0 < CW / 8; h0 += kH) {
                        uint32_t vA[kH][8], vB[kH][8];
#pragma unroll
                        for (int hh = 0; hh < kH; ++hh) {
                            tcx_ld8(ca + 8 * (h0 + hh), vA[hh]);
                            tcx_ld8(cb + 8 * (h0 + hh), vB[hh]);
                        }
                        tc_wait_ld();
                        if (h0 + kH >= CW / 8) grp_release(du);
#pragma unroll
                        for (int hh = 0; hh < kH; ++hh)
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            const int h = h0 + hh;
                            const uint32_t* va = vA[hh];
                            const uint32_t* vb = vB[hh];
                            const float4 a4 = kF32 ? make_float4(1.0f, 1.0f, 1.0f, 1.0f)  // f32_act: 2^-s at the store
                                                   : *reinterpret_cast<const float4*>(asc + 8 * h + 4 * c);
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const int i = 4 * c + 2 * e;
                                const unsigned long long t = fma2(f2pack(__uint_as_float(va[i]), __uint_as_float(va[i + 1])), k16,
                                                                  f2pack(__uint_as_float(vb[i]), __uint_as_float(vb[i + 1])));
                                const unsigned long long sc2 = kF32 ? fd2 : mul2(e ? f2pack(a4.z, a4.w) : f2pack(a4.x, a4.y), fd2);
                                acc[4 * h + 2 * c + e] = fma2(t, sc2, acc[4 * h + 2 * c + e]);
                            }
                        }
                    }
                    du += 2;
                } else {
                    // y += d_a (f(d) S_sc - f(dmin) S_m): S_sc and S_m exact integers in f32
                    const uint32_t ca = grp_wait(du);
                    const uint32_t cm = ca + NX;  // the group's second accumulator (du is even)
                    if (!ok) break;
                    tc_fence_after();
                    __syncwarp();
                    const uint32_t dd = *reinterpret_cast<const uint32_t*>(wrow);  // f16 d, f16 dmin
                    // f32_act: the min operand holds the sums of 16 over 16 (they fit f16), so f(dmin) 16
                    const float fm = -h2f(dd >> 16) * (kF32 ? 16.0f : 1.0f);
                    const unsigned long long fd2 = f2pack(h2f(dd), h2f(dd)), fm2 = f2pack(fm, fm);
#pragma unroll
                    for (int h0 = 0; h0 < CW / 8; h0 += kH) {
                        uint32_t vS[kH][8], vM[kH][8];
#pragma unroll
                        for (int hh = 0; hh < kH; ++hh) {
                            tcx_ld8(ca + 8 * (h0 + hh), vS[hh]);
                            tcx_ld8(cm + 8 * (h0 + hh), vM[hh]);
                        }
                        tc_wait_ld();
                        if (h0 + kH >= CW / 8) grp_release(du);
#pragma unroll
                        for (int hh = 0; hh < kH; ++hh)
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            const int h = h0 + hh;
                            const uint32_t* vs = vS[hh];
                            const uint32_t* vm = vM[hh];
                            if constexpr (kF32) {
                                // y 2^s += f(d) S_sc - f(dmin) S_m (sums of x 2^s, 2^-s applied at the store)
#pragma unroll
                                for (int e = 0; e < 2; ++e) {
                                    const int i = 4 * c + 2 * e;
                                    unsigned long long& a = acc[4 * h + 2 * c + e];
                                    a = fma2(f2pack(__uint_as_float(vs[i]), __uint_as_float(vs[i + 1])), fd2, a);
                                    a = fma2(f2pack(__uint_as_float(vm[i]), __uint_as_float(vm[i + 1])), fm2, a);
                                }
                            } else {
                                const float4 a4 = *reinterpret_cast<const float4*>(asc + 8 * h + 4 * c);
#pragma unroll
                                for (int e = 0; e < 2; ++e) {
                                    const int i = 4 * c + 2 * e;
                                    const unsigned long long t =
                                        fma2(f2pack(__uint_as_float(vs[i]), __uint_as_float(vs[i + 1])), fd2,
                                             mul2(f2pack(__uint_as_float(vm[i]), __uint_as_float(vm[i + 1])), fm2));
                                    const unsigned long long a2 = e ? f2pack(a4.z, a4.w) : f2pack(a4.x, a4.y);
                                    acc[4 * h + 2 * c + e] = fma2(t, a2, acc[4 * h + 2 * c + e]);
                                }
                            }
                        }
                    }
                    du += 2;
                }
                if (!ok) break;
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&r_empty[rs]));  // this warp no longer reads the raw stage
            }
            if (!ok || flags[0]) break;
            const int tile = u % p.tiles;
            const int m0 = (tile % p.mtiles) * NX, n0 = (tile / p.mtiles) * kTxW;
            const int n = n0 + nl;
            float* dst = p.ks == 1 ? p.y : p.part + (size_t)(u / p.tiles) * p.M * p.N;
            if (n < p.N) {
#pragma unroll
                for (int i = 0; i < CW / 2; ++i) {
                    const int m = m0 + CW * cq + 2 * i;
                    if (m < p.M) dst[(size_t)m * p.N + n] = kF32 ? f2lo(acc[i]) * __ldg(p.ais + m) : f2lo(acc[i]);
                    if (m + 1 < p.M) dst[(size_t)(m + 1) * p.N + n] = kF32 ? f2hi(acc[i]) * __ldg(p.ais + m + 1) : f2hi(acc[i]);
                }
            }
            if (p.ks > 1) {
                // the unit that completes the tile sums its ks partials in slice order
                const uint32_t fix = (uint32_t)(((u - (int)blockIdx.x) / (int)gridDim.x) & 1);  // this CTA's unit count
                __threadfence();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(epi_done));
                if (ew == 0 && lane == 0) {
                    int owner = 0;
                    if (mbar_wait(smem_u32(epi_done), fix, flags, p.err)) {
                        __threadfence();
                        owner = atomicAdd(p.cnt + tile, 1u) == (unsigned)(p.ks - 1);
                    }
                    flags[1] = owner;
                    mbar_arrive(smem_u32(fix_ready));
                }
                if (!(ok = mbar_wait(smem_u32(fix_ready), fix, flags, p.err))) break;
                if (flags[1]) {
                    __threadfence();
                    tcx_fixup<NX>(p.part, p.y, p.M, p.N, p.ks, ew * 32 + lane, m0, n0);
                }
            }
        }
    } else {
        // ------------------------------ converters ------------------------------
        const int r = 32 * (warp - 2 - kTxEpiWarps) + lane;  // weight row of the tile
        // this row's eight 16-byte chunks (four per block) in the 128-byte swizzled K-major layout
        const int rbase = (r >> 3) * 1024 + (r & 7) * 128, sw = r & 7;
        long long rg = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
            int tile, r0, r1;
            tcx_slice(p, u, tile, r0, r1);
            for (int rr = r0; rr < r1 && ok; ++rr, ++rg) {
                const int rs = (int)(rg % p.nraw);
                if (!(ok = mbar_wait(smem_u32(&r_full[rs]), (uint32_t)((rg / p.nraw) & 1), flags, p.err))) break;
                const uint8_t* wrow = raw(rs) + r * R::row;
                if (WT == T_Q4_K) {
                    // the min term's weight operand: m_j twice each, 16 f16 = two 16-byte
                    // chunks in the 32-byte swizzled K-major layout
                    const uint4 hd = *reinterpret_cast<const uint4*>(wrow);
                    uint32_t mw[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const __half mh = __float2half_rn((float)q4k_mn(hd.z, hd.w, j));  // exact
                        const __half2 m2 = __halves2half2(mh, mh);
                        mw[j] = *reinterpret_cast<const uint32_t*>(&m2);
                    }
                    uint8_t* am = raw(rs) + R::amin + (r >> 3) * 256 + (r & 7) * 32;
                    const int s32 = (r >> 2) & 1;
                    *reinterpret_cast<uint4*>(am + ((0 ^ s32) << 4)) = make_uint4(mw[0], mw[1], mw[2], mw[3]);
                    *reinterpret_cast<uint4*>(am + ((1 ^ s32) << 4)) = make_uint4(mw[4], mw[5], mw[6], mw[7]);
                    fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&min_ready[rs]));
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const long long g = rg * kSpr + j / kBps;  // the block's stage
                    const int s = (int)(g % kTxS);
                    const int b = j % kBps;                       // its place in the stage
                    const int c0 = 4 * (b & 1);                   // its first chunk in the atom's 128-byte row
                    const int ab = (b >> 1) * kTxW * 128;         // its atom
                    if (b == 0 && g >= kTxS &&
                        !(ok = mbar_wait(smem_u32(&empty[s]), (uint32_t)(((g / kTxS) - 1) & 1), flags, p.err)))
                        break;
                    uint32_t h[16];
                    if (WT == T_Q6_K) {
                        uint32_t h2[16];
                        if (j == 0) tcx_conv_q6_k<0>(wrow, h, h2);
                        else if (j == 1) tcx_conv_q6_k<1>(wrow, h, h2);
                        else if (j == 2) tcx_conv_q6_k<2>(wrow, h, h2);
                        else if (j == 3) tcx_conv_q6_k<3>(wrow, h, h2);
                        else if (j == 4) tcx_conv_q6_k<4>(wrow, h, h2);
                        else if (j == 5) tcx_conv_q6_k<5>(wrow, h, h2);
                        else if (j == 6) tcx_conv_q6_k<6>(wrow, h, h2);
                        else tcx_conv_q6_k<7>(wrow, h, h2);
                        uint8_t* a2 = wstage(s) + R::wtile(NX) + ab + rbase;
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            *reinterpret_cast<uint4*>(a2 + (((c0 + c) ^ sw) << 4)) =
                                make_uint4(h2[4 * c], h2[4 * c + 1], h2[4 * c + 2], h2[4 * c + 3]);
                    } else if (kB32) {
                        if (j == 0) tcx_conv_b32<WT, 0>(wrow, h);
                        else if (j == 1) tcx_conv_b32<WT, 1>(wrow, h);
                        else if (j == 2) tcx_conv_b32<WT, 2>(wrow, h);
                        else if (j == 3) tcx_conv_b32<WT, 3>(wrow, h);
                        else if (j == 4) tcx_conv_b32<WT, 4>(wrow, h);
                        else if (j == 5) tcx_conv_b32<WT, 5>(wrow, h);
                        else if (j == 6) tcx_conv_b32<WT, 6>(wrow, h);
                        else tcx_conv_b32<WT, 7>(wrow, h);
                    } else {
                        if (j == 0) tcx_conv_q4_k<0>(wrow, h);
                        else if (j == 1) tcx_conv_q4_k<1>(wrow, h);
                        else if (j == 2) tcx_conv_q4_k<2>(wrow, h);
                        else if (j == 3) tcx_conv_q4_k<3>(wrow, h);
                        else if (j == 4) tcx_conv_q4_k<4>(wrow, h);
                        else if (j == 5) tcx_conv_q4_k<5>(wrow, h);
                        else if (j == 6) tcx_conv_q4_k<6>(wrow, h);
                        else tcx_conv_q4_k<7>(wrow, h);
                    }
                    uint8_t* a = wstage(s) + ab + rbase;
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        *reinterpret_cast<uint4*>(a + (((c0 + c) ^ sw) << 4)) = make_uint4(h[4 * c], h[4 * c + 1], h[4 * c + 2], h[4 * c + 3]);
                    if (b == kBps - 1) {
                        fence_proxy_async();  // the generic-proxy stores, before the tensor core reads them
                        __syncwarp();
                        if (lane == 0) mbar_arrive(smem_u32(&full[s]));
                    }
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

// The activation operand, written once per call.  Q8_0: one thread per
// (row m, 32-block b) quantizes the block to Q8_0, writes its codes as f16 to
// codes[m][K] and the f16-rounded scale f(d_a) block-major to scales[b][mp].
// Q4_K: one warp per (row m, super-block b), lane l taking values 8l..8l+7,
// quantizes it to Q8K (f32 d = amax / 127 over the 256 values), writes the
// codes as f16, d to scales[b][mp] and the 16 sums of 16 codes (at most
// 2032 in magnitude, exact in f16) to bsums[m][K / 16].  It also zeroes the
// GEMM's ncnt split-K arrival counters.
template <int WT>
__global__ void tcx_act_kernel(const float* __restrict__ x, int M, int K, int mp, __half* __restrict__ codes,
                               float* __restrict__ scales, __half* __restrict__ bsums, unsigned* __restrict__ cnt, int ncnt) {
    grid_dep_launch();
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < ncnt; i += (long long)gridDim.x * blockDim.x)
        cnt[i] = 0u;
    if (WT == T_Q8_0 || WT == T_Q4_0 || WT == T_Q5_0) {  // Q8_0 activations
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
    } else {
        const long long w = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
        const int lane = threadIdx.x & 31;
        const int nsb = K / 256;
        if (w >= (long long)M * nsb) return;  // whole warps leave together
        const int m = (int)(w / nsb), b = (int)(w - (long long)m * nsb);
        const float4* src = reinterpret_cast<const float4*>(x + (long long)m * K + 256 * b + 8 * lane);
        const float4 v0 = __ldg(src), v1 = __ldg(src + 1);
        float amax = fmaxf(fmaxf(fmaxf(fabsf(v0.x), fabsf(v0.y)), fmaxf(fabsf(v0.z), fabsf(v0.w))),
                           fmaxf(fmaxf(fabsf(v1.x), fabsf(v1.y)), fmaxf(fabsf(v1.z), fabsf(v1.w))));
#pragma unroll
        for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        float d, id;
        q8_scale(amax, d, id);
        const uint32_t w0 = pack4(q8_code(v0.x, id), q8_code(v0.y, id), q8_code(v0.z, id), q8_code(v0.w, id));
        const uint32_t w1 = pack4(q8_code(v1.x, id), q8_code(v1.y, id), q8_code(v1.z, id), q8_code(v1.w, id));
        uint32_t h[4];
        tcx_codes(w0, h[0], h[1]);
        tcx_codes(w1, h[2], h[3]);
        *reinterpret_cast<uint4*>(codes + (long long)m * K + 256 * b + 8 * lane) = make_uint4(h[0], h[1], h[2], h[3]);
        const int s8 = bsum4(w0) + bsum4(w1);
        const int s16 = s8 + __shfl_xor_sync(0xffffffffu, s8, 1);  // lanes 2i, 2i + 1: codes 16i..16i+15
        if ((lane & 1) == 0) bsums[(long long)m * (K / 16) + 16 * b + (lane >> 1)] = __float2half_rn((float)s16);
        if (lane == 0) scales[(long long)b * mp + m] = d;
    }
}

// The f32_act operand, written once per call: one 256-thread block per
// activation row m finds the row's largest magnitude, takes 2^s with
// max |x| 2^s in [2^14, 2^15) and splits every value exactly into two f16
// pieces, x 2^s = hi + lo (hi[m][K], lo[m][K]); for Q4_K each 16 values' sum
// of x 2^s, over 16 (at most 2^15, so it fits f16), is split the same way into
// bsums[m][K / 16 + j] after the hi sums bsums[m][j]; ais[m] = 2^-s.  It also
// zeroes the GEMM's ncnt split-K arrival counters.
template <int WT>
__global__ void tcx_act_f32_kernel(const float* __restrict__ x, int M, int K, __half* __restrict__ hi, __half* __restrict__ lo,
                                   __half* __restrict__ bsums, float* __restrict__ ais, unsigned* __restrict__ cnt, int ncnt) {
    grid_dep_launch();
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < ncnt; i += (long long)gridDim.x * blockDim.x)
        cnt[i] = 0u;
    __shared__ float red[32];
    const int m = blockIdx.x, tid = threadIdx.x;
    if (m >= M) return;
    const float* xr = x + (long long)m * K;
    float amax = 0.0f;
    for (int k = 4 * tid; k < K; k += 4 * blockDim.x) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(xr + k));
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((tid & 31) == 0) red[tid >> 5] = amax;
    __syncthreads();
    if (tid < 32) {
        float a = tid < (int)(blockDim.x >> 5) ? red[tid] : 0.0f;
#pragma unroll
        for (int o = 16; o; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        if (tid == 0) red[0] = a;
    }
    __syncthreads();
    const float is = tc_row_iscale(red[0]);
    const float sc = __frcp_rn(is);  // 2^s, exact
    if (tid == 0) ais[m] = is;
    __half* hr = hi + (long long)m * K;
    __half* lr = lo + (long long)m * K;
    __half* br = bsums + (long long)m * (K / 8);
    for (int g = tid; g < K / 16; g += blockDim.x) {  // 16 values per thread
        const float4* src = reinterpret_cast<const float4*>(xr + 16 * g);
        uint32_t hw[8], lw[8];
        float sum = 0.0f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 v4 = __ldg(src + q);
            const float v[4] = {v4.x * sc, v4.y * sc, v4.z * sc, v4.w * sc};
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const __half2 h2 = __floats2half2_rn(v[2 * e], v[2 * e + 1]);
                const float2 hf = __half22float2(h2);
                const __half2 l2 = __floats2half2_rn(v[2 * e] - hf.x, v[2 * e + 1] - hf.y);
                hw[2 * q + e] = *reinterpret_cast<const uint32_t*>(&h2);
                lw[2 * q + e] = *reinterpret_cast<const uint32_t*>(&l2);
            }
            sum += v[0];
            sum += v[1];
            sum += v[2];
            sum += v[3];
        }
        uint4* ho = reinterpret_cast<uint4*>(hr + 16 * g);
        uint4* lo4 = reinterpret_cast<uint4*>(lr + 16 * g);
        ho[0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        ho[1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
        lo4[0] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        lo4[1] = make_uint4(lw[4], lw[5], lw[6], lw[7]);
        if (WT == T_Q4_K) {
            const float s16 = sum * 0.0625f;  // exact
            const __half sh = __float2half_rn(s16);
            br[g] = sh;
            br[K / 16 + g] = __float2half_rn(s16 - __half2float(sh));
        }
    }
}

// Q6_K: every 210-byte super-block copied into a 240-byte slot (rows of K / 256
// slots), 16-byte aligned for the GEMM's tensor map; one warp per weight row,
// 2-byte words
template <int WT>  // T_Q6_K
__global__ void tcx_q6_repack_kernel(const uint8_t* __restrict__ wq, int N, int K, uint8_t* __restrict__ w6) {
    grid_dep_launch();
    const long long n = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (n >= N) return;
    const int nsb = K / 256;
    const uint16_t* src = reinterpret_cast<const uint16_t*>(wq + n * (long long)nsb * 210);
    uint16_t* dst = reinterpret_cast<uint16_t*>(w6 + n * (long long)nsb * TxRaw<T_Q6_K>::row);
    for (int i = lane; i < nsb * 105; i += 32) {
        const int b = i / 105, hw = i - 105 * b;
        dst[b * (TxRaw<T_Q6_K>::row / 2) + hw] = __ldg(src + i);
    }
}

// ---------------------------------------------------------------------------
// host-side plan
// ---------------------------------------------------------------------------
struct TcxPlan {
    TcxParams p;
    int am;  // A_INT8 (exact block sums) or A_F32 (two activation pieces)
    int nx;  // activation rows per tile: 64 or 128
    int grid;
    size_t smem;
    int mp;  // activation scale rows: M rounded up to 4 (16-byte rows for the tensor map)
    // workspace: activation codes (f32_act: the hi pieces), int8_act scales or f32_act lo
    // pieces, Q4_K sums of 16, f32_act 2^-s per row, Q6_K repacked weights, split-K partials
    // and counters
    size_t ws_codes, ws_scales, ws_bsums, ws_ais, ws_w6, ws_part, ws_cnt, workspace;
};

template <int AM>
inline int tcx_raw_slot_am(int wt) {
    switch (wt) {
        case T_Q8_0: return TxRaw<T_Q8_0, AM>::slot;
        case T_Q4_0: return TxRaw<T_Q4_0, AM>::slot;
        case T_Q5_0: return TxRaw<T_Q5_0, AM>::slot;
        case T_Q4_K: return TxRaw<T_Q4_K, AM>::slot;
        default: return TxRaw<T_Q6_K, AM>::slot;
    }
}
template <int AM>
inline int tcx_stages_am(int wt, int nx) {
    switch (wt) {
        case T_Q8_0: return TxRaw<T_Q8_0, AM>::stages(nx);
        case T_Q4_0: return TxRaw<T_Q4_0, AM>::stages(nx);
        case T_Q5_0: return TxRaw<T_Q5_0, AM>::stages(nx);
        case T_Q4_K: return TxRaw<T_Q4_K, AM>::stages(nx);
        default: return TxRaw<T_Q6_K, AM>::stages(nx);
    }
}
template <int AM>
inline int tcx_stage_bytes_am(int wt, int nx) {
    switch (wt) {
        case T_Q8_0: return TxRaw<T_Q8_0, AM>::stage(nx);
        case T_Q4_0: return TxRaw<T_Q4_0, AM>::stage(nx);
        case T_Q5_0: return TxRaw<T_Q5_0, AM>::stage(nx);
        case T_Q4_K: return TxRaw<T_Q4_K, AM>::stage(nx);
        default: return TxRaw<T_Q6_K, AM>::stage(nx);
    }
}
inline int tcx_raw_slot(int wt, int am) { return am == A_F32 ? tcx_raw_slot_am<A_F32>(wt) : tcx_raw_slot_am<A_INT8>(wt); }
inline int tcx_stages(int wt, int am, int nx) { return am == A_F32 ? tcx_stages_am<A_F32>(wt, nx) : tcx_stages_am<A_INT8>(wt, nx); }
inline int tcx_stage_bytes(int wt, int am, int nx) {
    return am == A_F32 ? tcx_stage_bytes_am<A_F32>(wt, nx) : tcx_stage_bytes_am<A_INT8>(wt, nx);
}

inline bool plan_tcx(int wt, int am, long long M, long long N, long long K, int sm_count, int smem_max, TcxPlan& out) {
    // int8_act: Q8_0, Q4_0, Q5_0, Q4_K, Q6_K; f32_act: Q8_0, Q4_K, Q6_K
    const bool b32 = wt == T_Q8_0 || wt == T_Q4_0 || wt == T_Q5_0;
    if ((!b32 && wt != T_Q4_K && wt != T_Q6_K) || (am == A_F32 && (wt == T_Q4_0 || wt == T_Q5_0)) || K % 256 != 0 || M < 17 ||
        K > (1 << 26) || M > (1 << 24) || N > (1 << 24))
        return false;
    TcxPlan pl{};
    pl.am = am;
    TcxParams& p = pl.p;
    p.M = (int)M;
    p.N = (int)N;
    p.K = (int)K;
    // 64-row tiles when they hold all activation rows: half the fold and the
    // accumulator drains of a 128-row tile
    pl.nx = M <= 64 ? 64 : kTxX;
    p.mtiles = (int)((M + pl.nx - 1) / pl.nx);
    p.ntiles = (int)((N + kTxW - 1) / kTxW);
    if ((long long)p.mtiles * p.ntiles * kTxMaxSplit > INT32_MAX) return false;
    p.tiles = p.mtiles * p.ntiles;
    p.nrs = (int)(K / 256);
    // K slices: with few tiles, the smallest ks whose busiest CTA (units dealt
    // round-robin, one CTA per SM) carries the fewest raw stages, counting a
    // unit's start as half a stage and a split unit's partial tile, arrival
    // and share of the sum of partials as three (measured: the 112 and 224
    // tiles of 14336 weight rows at M <= 64 and M = 256 run fastest unsplit,
    // the 32 and 64 of 4096 rows fastest in 4 and 2 slices)
    {
        double best = 0.0;
        int best_ks = 1;
        const int kmax = p.nrs < kTxMaxSplit ? p.nrs : kTxMaxSplit;
        for (int ks = 1; ks <= kmax; ++ks) {
            const long long units = (long long)p.tiles * ks;
            const long long grid = units < sm_count ? units : sm_count;
            const long long per = (units + grid - 1) / grid;  // units of the busiest CTA
            const double stages = (double)p.nrs / ks + (ks > 1 ? 3.0 : 0.5);
            const double worst = per * stages;
            if (ks == 1 || worst < best * 0.98) best = worst, best_ks = ks;
        }
        p.ks = best_ks;
    }
    p.units = p.tiles * p.ks;
    p.off_raw = tcx_stages(wt, am, pl.nx) * tcx_stage_bytes(wt, am, pl.nx);
    const int fixed = 512 + 1024;  // barriers, TMEM slot, flags; alignment slack
    p.nraw = (smem_max - p.off_raw - fixed) / tcx_raw_slot(wt, am);
    if (p.nraw > kTxRawMax) p.nraw = kTxRawMax;
    if (p.nraw < 3) return false;  // the epilogue holds a raw stage while the converters fill the next
    p.off_bar = p.off_raw + p.nraw * tcx_raw_slot(wt, am);
    pl.smem = (size_t)p.off_bar + fixed;
    pl.grid = p.units < sm_count ? p.units : sm_count;
    pl.mp = (int)((M + 3) / 4 * 4);
    auto r256 = [](size_t v) { return (v + 255) / 256 * 256; };
    pl.ws_codes = 0;
    pl.ws_scales = r256((size_t)M * K * 2);
    const size_t per = b32 ? 32 : 256;  // values per activation scale
    pl.ws_bsums = pl.ws_scales + (am == A_F32 ? r256((size_t)M * K * 2) : r256((size_t)(K / per) * pl.mp * 4));
    pl.ws_ais = pl.ws_bsums + (wt == T_Q4_K || (wt == T_Q6_K && am == A_INT8) ? r256((size_t)M * (K / 16) * 2 * (am == A_F32 ? 2 : 1)) : 0);
    pl.ws_w6 = pl.ws_ais + (am == A_F32 ? r256((size_t)M * 4) : 0);
    pl.ws_part = pl.ws_w6 + (wt == T_Q6_K ? r256((size_t)N * (K / 256) * TxRaw<T_Q6_K>::row) : 0);
    pl.ws_cnt = pl.ws_part + (p.ks > 1 ? r256((size_t)p.ks * M * N * 4) : 0);
    pl.workspace = pl.ws_cnt + (p.ks > 1 ? r256((size_t)p.tiles * 4) : 0);
    out = pl;
    return true;
}

}  // namespace qmm
