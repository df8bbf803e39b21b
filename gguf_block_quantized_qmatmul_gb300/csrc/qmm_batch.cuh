// qmm_batch.cuh -- many independent small matmuls in one launch: the linears
// of a decode step (q/k/v, o, gate/up, down, the output head), which one at
// a time are bound by launch latency rather than by their weight bytes.
//
// Both QMatMul forms ("同一个 GGUF，CPU 和 Metal 生成的文字不一样" section
// 出处), for every weight type: the 32-value blocks (Q8_0, Q4_0, Q5_0 with
// Q8_0 activations) and the 256-value super-blocks (Q4_K, Q6_K with Q8K
// activations), so that a whole step of a mixed-type file (the Q4_K_M files
// of the "GGUF 文件" page hold Q5_0, Q8_0, Q4_K and Q6_K matrices) is one
// launch:
//   int8_act: per weight unit the exact int32 sums of weight codes times the
//             row-quantized activation codes, then
//             Q8_0/Q4_0/Q5_0: y += f(d_w) f(d_a) isum;
//             Q4_K: y += d_a (f(d) S_sc - f(dmin) S_m), S_sc = sum_j sc_j isum_j,
//                   S_m = sum_j m_j bsum_j (bsum_j: sub-block j's activation codes);
//             Q6_K: y += d_a f(d) S, S = sum_g sc_g isum_g over 16 groups of 16;
//             each super-block's S_sc, S_m and S are whole int32 sums before
//             the one conversion to f32 (its four pieces' lanes add them exactly);
//   f32_act:  y += f32 products of the dequantized weight and x: f(d) sum(q x)
//             per 32-value block, e_j sum(q x) - o_j sum(x) per Q4_K
//             sub-block (e_j = f(d) sc_j, o_j = f(dmin) m_j), f(d) sc_g
//             sum(q x) per Q6_K group.
//
// The rows of all items are one virtual stream, each row weighted by its
// cost (its values times a per-type, per-form cost of 32 values measured at
// saturation); CTA c (one per SM) takes the rows whose first position falls in
// its 1/G share of the total, item by item (a "piece": consecutive rows of one
// item, contiguous bytes).  A producer
// lane streams each piece in stages of whole rows, one 1-D bulk copy per
// stage, into a ring of shared-memory slots (the copy engine pays a fixed cost
// per contiguous segment, so stages are large).  16 consumer warps stage the
// item's activation rows in shared memory when a piece starts (int8_act
// quantizes them, Q8_0 per 32 values or Q8K per 256; f32_act copies them, with
// the Q4_K sub-block sums of x), then take each stage's rows in lane groups:
// lpr lanes per group, up to two rows per group sharing the activation loads,
// lane gl taking units gl, gl + lpr, ... of its rows (a unit: one 32-value
// block or one 64-value piece of a super-block); the group sums its lanes with
// a shuffle tree.
// lpr, the units per lane and the rows per stage are planned per item on the
// host.
#pragma once

#include <algorithm>

#include "qmm_stream.cuh"

namespace qmm {

constexpr int kBatchMax = 256;  // items per launch (the launch parameters carry the table)
constexpr int T_MIX = 7;        // kernel variant whose items carry their own weight type
constexpr int kBatchWarps = 16;            // consumer warps; + 1 producer warp
constexpr int kBatchStagesMax = 6;         // ring slots, fewer when the activations need the room
constexpr int kBatchStageCap = 56 * 1024;  // the most bytes of whole rows a stage is planned to hold

struct BatchItem {
    const uint8_t* wq;
    const float* x;
    float* y;
    long long c0;     // the item's first position in the launch's cost order
    int cpr;          // the cost of one of its rows (batch_row_cost)
    int M, N, K;
    int wt;            // weight type (T_Q8_0, T_Q4_0, T_Q5_0, T_Q4_K, T_Q6_K)
    int lpr, bpl, tr;  // lanes per row, units per lane, rows per stage (set by the launcher)
};
struct BatchParams {
    BatchItem it[kBatchMax];
    long long total;  // the cost of all items
    unsigned* err;    // the device error word (bounded waits)
    int count;
    int act_bytes;    // the most shared-memory bytes one item's staged activations take
    int slot_bytes;   // bytes of one weight stage slot (set by the launcher)
    int stages;       // slots in the ring, 2..16 (set by the launcher)
};

// Shared-memory bytes of one staged activation unit (row m, unit b):
//   Q8_0 codes (int8_act, 32-value types): 32 codes, the f16-rounded scale as f32 at 32;
//   f32 (f32_act, 32-value types): 32 floats (+16 bytes of padding);
//   Q8K (int8_act, super-block types): 8 slots of 48 bytes, each 32 codes; the
//     8 int32 code sums of the 32-value sub-blocks at 384, f32 d at 416;
//   f32 (f32_act, super-block types): 8 slots of 144 bytes, each 32 floats; the
//     8 f32 sums of x of the sub-blocks at 1152.
// A super-block's 32-value quarters go to slots in the order its pieces read
// them: piece c reads slots 2c and 2c + 1 (Q4_K: sub-blocks 2c, 2c + 1, in
// order; Q6_K: quarters p and p + 2 of half hh, c = 2 hh + p).  Slot and unit
// strides are odd numbers of 16-byte granules, so that the eight lanes of a
// quarter-warp (two quads on consecutive super-blocks) read eight distinct
// granules of the 128-byte bank row.
__host__ __device__ constexpr int batch_act_unit(int wt, int am) {
    return is_sb(wt) ? (am == A_INT8 ? 432 : 1200) : (am == A_INT8 ? 48 : 144);
}
// the staged slot of 32-value quarter q (value / 32) of a super-block of type wt
__host__ __device__ constexpr int batch_slot(int wt, int q) {
    return wt == T_Q6_K ? (q & 4) | ((q & 1) << 1) | ((q >> 1) & 1) : q;
}
// weight rows a lane group works on at once (they share the activation loads)
__host__ __device__ constexpr int batch_rows_per_group(int wt, int am, int mt) {
    return is_sb(wt) ? (am == A_INT8 && mt == 1 ? 2 : 1) : (mt == 1 || (am == A_INT8 && mt == 2) ? 2 : 1);
}

cudaError_t launch_batch(int wt, int am, const BatchParams& p, int max_m, int sm_count, int smem_max, cudaStream_t s);
// The cost of one weight row of K values of type wt in form am: the CTAs take
// equal shares of the launch's total cost, so that types that are cheap in
// bytes but dear in unpacking (Q5_0, Q4_0) do not leave the CTAs holding
// bandwidth-bound rows (Q8_0) idle.
int batch_row_cost(int wt, int am, int K);
cudaError_t launch_batch_mix(int am, BatchParams& p, int mt, int grid, int smem_max, cudaStream_t s);
// lpr, bpl and tr for a row of nu units of weight type wt, rb bytes
void plan_batch_item(int wt, int nu, long long rb, int am, int mt, int& lpr, int& bpl, int& tr);

namespace {

// One 32-value weight block at byte offset o (even) of shared memory s: the
// f32 scale and eight words of signed codes (values 4k..4k+3 in word k).  The
// payload is read as aligned words from its rounded-down start and realigned
// with one funnel shift per word; up to 4 bytes past the block are read (the
// slot's slack) and never used.
template <int WT>
__device__ __forceinline__ float load_block(const uint8_t* s, int o, uint32_t c[8]) {
    const uint32_t dword = ld32(s + (o & ~3));
    const float d = h2f((dword >> ((o & 2) << 3)) & 0xFFFFu);
    const int ps = o + 2;  // the payload after the f16 scale
    const uint8_t* a = s + (ps & ~3);
    const uint32_t sh = (uint32_t)(ps & 3) << 3;  // 0 or 16
    if (WT == T_Q8_0) {
        uint32_t w[9];
#pragma unroll
        for (int k = 0; k < 9; ++k) w[k] = ld32(a + 4 * k);
#pragma unroll
        for (int k = 0; k < 8; ++k) c[k] = __funnelshift_r(w[k], w[k + 1], sh);
    } else {
        // (Q5_0) the fifth bits' word, then 16 nibble bytes: code j in the low
        // nibble of byte j, code j + 16 in its high nibble
        constexpr int QW = WT == T_Q5_0 ? 1 : 0;
        uint32_t w[QW + 5];
#pragma unroll
        for (int k = 0; k < QW + 5; ++k) w[k] = ld32(a + 4 * k);
        uint32_t q[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) q[k] = __funnelshift_r(w[QW + k], w[QW + k + 1], sh);
        const uint32_t hb = WT == T_Q5_0 ? __funnelshift_r(w[0], w[1], sh) : 0u;
        constexpr uint32_t OFF = WT == T_Q5_0 ? 0x10101010u : 0x08080808u;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            uint32_t v = k < 4 ? (q[k & 3] & 0x0F0F0F0Fu) : ((q[k & 3] >> 4) & 0x0F0F0F0Fu);
            if (WT == T_Q5_0) v |= ((((hb >> (4 * k)) & 0xFu) * 0x00204081u) & 0x01010101u) << 4;
            c[k] = __vsub4(v, OFF);
        }
    }
    return d;
}

// NW words from shared byte offset o (any alignment): aligned loads from the
// rounded-down start, realigned with one funnel shift per word (reads up to 4
// bytes past the last word).
template <int NW>
__device__ __forceinline__ void ld_words(const uint8_t* s, int o, uint32_t (&w)[NW]) {
    const uint8_t* a = s + (o & ~3);
    const uint32_t sh = (uint32_t)(o & 3) << 3;
    uint32_t r[NW + 1];
#pragma unroll
    for (int k = 0; k <= NW; ++k) r[k] = ld32(a + 4 * k);
#pragma unroll
    for (int k = 0; k < NW; ++k) w[k] = __funnelshift_r(r[k], r[k + 1], sh);
}

__device__ __forceinline__ unsigned long long pack2(uint32_t lo, uint32_t hi) {
    unsigned long long d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo), "r"(hi));
    return d;
}
__device__ __forceinline__ float2 unpack2(unsigned long long v) {
    uint32_t lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(v));
    return make_float2(__uint_as_float(lo), __uint_as_float(hi));
}
__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long ffma2(unsigned long long a, unsigned long long b, unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// sum over NW words of (byte - OFF) * x, the words' bytes unsigned codes and
// x the NW * 4 floats at xs (16-byte aligned): a byte becomes the float
// 2^23 + byte by a byte permute, and 2^23 + OFF is taken off exactly
template <int NW, int OFF>
__device__ __forceinline__ float dot_u8_f32(const uint32_t* w, const uint8_t* xs) {
    const uint32_t nb = __float_as_uint(-(8388608.0f + (float)OFF));
    const unsigned long long neg = pack2(nb, nb);
    unsigned long long s01 = 0, s23 = 0;
#pragma unroll
    for (int k = 0; k < NW; ++k) {
        const uint4 xv = ld128(xs + 16 * k);
        const unsigned long long q01 =
            add2(pack2(__byte_perm(w[k], 0x4B000000u, 0x7440u), __byte_perm(w[k], 0x4B000000u, 0x7441u)), neg);
        const unsigned long long q23 =
            add2(pack2(__byte_perm(w[k], 0x4B000000u, 0x7442u), __byte_perm(w[k], 0x4B000000u, 0x7443u)), neg);
        s01 = ffma2(q01, pack2(xv.x, xv.y), s01);
        s23 = ffma2(q23, pack2(xv.z, xv.w), s23);
    }
    const float2 r = unpack2(add2(s01, s23));
    return r.x + r.y;
}

// out[m] = the same sum for each activation row m < M, x of row m at
// xs + m * astep: each code is converted once and used for every row
template <int NW, int OFF, int MT>
__device__ __forceinline__ void dot_u8_f32_rows(const uint32_t* w, const uint8_t* xs, int astep, int M, float (&out)[MT]) {
    const uint32_t nb = __float_as_uint(-(8388608.0f + (float)OFF));
    const unsigned long long neg = pack2(nb, nb);
    unsigned long long s01[MT], s23[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) s01[m] = 0, s23[m] = 0;
#pragma unroll
    for (int k = 0; k < NW; ++k) {
        const unsigned long long q01 =
            add2(pack2(__byte_perm(w[k], 0x4B000000u, 0x7440u), __byte_perm(w[k], 0x4B000000u, 0x7441u)), neg);
        const unsigned long long q23 =
            add2(pack2(__byte_perm(w[k], 0x4B000000u, 0x7442u), __byte_perm(w[k], 0x4B000000u, 0x7443u)), neg);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m >= M) break;
            const uint4 xv = ld128(xs + m * astep + 16 * k);
            s01[m] = ffma2(q01, pack2(xv.x, xv.y), s01[m]);
            s23[m] = ffma2(q23, pack2(xv.z, xv.w), s23[m]);
        }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        const float2 r = unpack2(add2(s01[m], s23[m]));
        out[m] = r.x + r.y;
    }
}

// acc[h][m] += the contribution of 32-value block b of weight row h (h < R)
// to output row m, where v[h].  wo[h]: the weight blocks' offsets; ao: the
// offset of the activation unit for row 0; astep: the offset between
// activation rows.  The R rows share each activation load.
template <int WT, int AM, int MT, int R>
__device__ __forceinline__ void block_dot(const uint8_t* s, const int (&wo)[R], int ao, int astep, int M,
                                          const bool (&v)[R], float (&acc)[R][MT]) {
    uint32_t c[R][8];
    float dw[R];
#pragma unroll
    for (int h = 0; h < R; ++h) dw[h] = load_block<WT>(s, wo[h], c[h]);
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        if (m >= M) break;
        const uint8_t* a = s + ao + m * astep;
        if (AM == A_INT8) {
            // codes in bytes 0-31, the activation block's scale (f16-rounded, as f32) in bytes 32-35
            const uint4 a0 = ld128(a), a1 = ld128(a + 16);
            const float da = *reinterpret_cast<const float*>(a + 32);
#pragma unroll
            for (int h = 0; h < R; ++h) {
                // two independent chains of four
                int e = dp4a(c[h][0], a0.x, 0), o = dp4a(c[h][1], a0.y, 0);
                e = dp4a(c[h][2], a0.z, e);
                o = dp4a(c[h][3], a0.w, o);
                e = dp4a(c[h][4], a1.x, e);
                o = dp4a(c[h][5], a1.y, o);
                e = dp4a(c[h][6], a1.z, e);
                o = dp4a(c[h][7], a1.w, o);
                const float t = fmaf(dw[h] * da, (float)(e + o), acc[h][m]);
                acc[h][m] = v[h] ? t : acc[h][m];
            }
        } else {
            // signed codes as unsigned bytes (code + 128), less 128 in the conversion
#pragma unroll
            for (int h = 0; h < R; ++h) {
                uint32_t u[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) u[k] = c[h][k] ^ 0x80808080u;
                const float t = fmaf(dw[h], dot_u8_f32<8, 128>(u, a), acc[h][m]);
                acc[h][m] = v[h] ? t : acc[h][m];
            }
        }
    }
}

// Super-block types are taken in 64-value pieces: piece c of a Q4_K
// super-block is sub-blocks 2c, 2c + 1; piece i of a Q6_K super-block is
// quarters p and p + 2 of half hh (i = 2 hh + p), which share their ql and
// qh bytes.  The four pieces of a super-block sit on four consecutive lanes
// (lane groups of a multiple of 4 lanes).  int8_act sums each piece in int32
// and adds the four with two exchanges inside the quad, so that the whole
// super-block sum is converted to f32 once (by the lane of piece 0); f32_act
// adds each piece's f32 terms where it is.

// The int32 sum of the four lanes of a quad (lanes 4k..4k+3), on every lane.
__device__ __forceinline__ int quad_sum(int v) {
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    return v + __shfl_xor_sync(0xffffffffu, v, 2);
}

// acc[h][m] += piece c of the Q4_K super-block of weight row h (144 bytes at
// the 16-byte aligned offset wo[h]: f16 d, f16 dmin, 12 bytes of 6-bit scales
// and mins, 128 bytes of nibbles: sub-block 2c in the low nibbles of bytes
// 32c..32c+31, 2c + 1 in the high nibbles), where v[h].  ao: the offset of the
// activation super-block for row 0.
//   int8_act: S_sc = sum_j sc_j isum_j, S_m = sum_j m_j bsum_j over the whole
//             super-block, y += d_a (f(d) S_sc - f(dmin) S_m);
//   f32_act:  y += e_j sum(q x) - o_j sum(x), e_j = f(d) sc_j, o_j = f(dmin) m_j.
template <int AM, int MT, int R>
__device__ __forceinline__ void q4k_piece_dot(const uint8_t* s, const int (&wo)[R], int c, int ao, int astep, int M,
                                              const bool (&v)[R], float (&acc)[R][MT]) {
    // the 6-bit scale and min of sub-blocks 2c, 2c + 1: j < 4 in the low 6 bits
    // of bytes j (scales) and 4 + j (mins); j >= 4 in the nibbles of byte 8 + j - 4
    // with the high 2 bits in bits 6-7 of bytes j - 4 and j
    const uint32_t sh = 16u * (uint32_t)(c & 1);  // byte (2c) & 3 of the word, times 8
    const bool low = c < 2;
    uint32_t lo[R][8], hi[R][8];
    int sc0[R], sc1[R], mn0[R], mn1[R];
    float fd[R], fm[R];
#pragma unroll
    for (int h = 0; h < R; ++h) {
        const uint4 hw = ld128(s + wo[h]);  // d | dmin, scale bytes 0-3, 4-7, 8-11
        fd[h] = h2f(hw.x);
        fm[h] = h2f(hw.x >> 16);
        const uint32_t a0 = hw.y >> sh, a1 = hw.z >> sh, a2 = hw.w >> sh;
        const int ls0 = (int)(a0 & 63u), ls1 = (int)((a0 >> 8) & 63u);
        const int lm0 = (int)(a1 & 63u), lm1 = (int)((a1 >> 8) & 63u);
        const int hs0 = (int)((a2 & 15u) | ((a0 >> 2) & 48u)), hs1 = (int)(((a2 >> 8) & 15u) | ((a0 >> 10) & 48u));
        const int hm0 = (int)(((a2 >> 4) & 15u) | ((a1 >> 2) & 48u)), hm1 = (int)(((a2 >> 12) & 15u) | ((a1 >> 10) & 48u));
        sc0[h] = low ? ls0 : hs0, sc1[h] = low ? ls1 : hs1;
        mn0[h] = low ? lm0 : hm0, mn1[h] = low ? lm1 : hm1;
        const uint4 qa = ld128(s + wo[h] + 16 + 32 * c), qb = ld128(s + wo[h] + 32 + 32 * c);
        const uint32_t qq[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            lo[h][k] = qq[k] & 0x0F0F0F0Fu;
            hi[h][k] = (qq[k] >> 4) & 0x0F0F0F0Fu;
        }
    }
    if (AM == A_INT8) {
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m >= M) break;
            const uint8_t* a = s + ao + m * astep;
            const uint4 a0 = ld128(a + 96 * c), a1 = ld128(a + 96 * c + 16);        // slot 2c: sub-block 2c
            const uint4 a2 = ld128(a + 96 * c + 48), a3 = ld128(a + 96 * c + 64);   // slot 2c + 1
            const uint2 bs = ld64(a + 384 + 8 * c);
            const float da = *reinterpret_cast<const float*>(a + 416);
#pragma unroll
            for (int h = 0; h < R; ++h) {
                int s0 = dp4a(lo[h][0], a0.x, 0), s1 = dp4a(hi[h][0], a2.x, 0);
                s0 = dp4a(lo[h][1], a0.y, s0), s1 = dp4a(hi[h][1], a2.y, s1);
                s0 = dp4a(lo[h][2], a0.z, s0), s1 = dp4a(hi[h][2], a2.z, s1);
                s0 = dp4a(lo[h][3], a0.w, s0), s1 = dp4a(hi[h][3], a2.w, s1);
                s0 = dp4a(lo[h][4], a1.x, s0), s1 = dp4a(hi[h][4], a3.x, s1);
                s0 = dp4a(lo[h][5], a1.y, s0), s1 = dp4a(hi[h][5], a3.y, s1);
                s0 = dp4a(lo[h][6], a1.z, s0), s1 = dp4a(hi[h][6], a3.z, s1);
                s0 = dp4a(lo[h][7], a1.w, s0), s1 = dp4a(hi[h][7], a3.w, s1);
                const int ssc = quad_sum(sc0[h] * s0 + sc1[h] * s1);
                const int smn = quad_sum(mn0[h] * (int)bs.x + mn1[h] * (int)bs.y);
                const float t = da * (fd[h] * (float)ssc - fm[h] * (float)smn);
                acc[h][m] = v[h] && c == 0 ? acc[h][m] + t : acc[h][m];
            }
        }
    } else {
#pragma unroll
        for (int h = 0; h < R; ++h) {
            // e_j and o_j are exact f32 products (11-bit by 6-bit)
            const float e0 = fd[h] * (float)sc0[h], e1 = fd[h] * (float)sc1[h];
            const float o0 = fm[h] * (float)mn0[h], o1 = fm[h] * (float)mn1[h];
            float sl[MT], sh2[MT];
            dot_u8_f32_rows<8, 0, MT>(lo[h], s + ao + 288 * c, astep, M, sl);         // slot 2c
            dot_u8_f32_rows<8, 0, MT>(hi[h], s + ao + 288 * c + 144, astep, M, sh2);  // slot 2c + 1
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if (m >= M) break;
                const float2 X = *reinterpret_cast<const float2*>(s + ao + m * astep + 1152 + 8 * c);
                const float t = (e0 * sl[m] - o0 * X.x) + (e1 * sh2[m] - o1 * X.y);
                acc[h][m] = v[h] ? acc[h][m] + t : acc[h][m];
            }
        }
    }
}

// acc[h][m] += piece i of the Q6_K super-block of weight row h (210 bytes at
// the even offset wo[h]: ql 0-127, qh 128-191, 16 int8 group scales 192-207,
// f16 d 208), where v[h].  Value 128 hh + 32 q + l takes the low 4 bits from
// nibble q / 2 of ql byte 64 hh + 32 (q % 2) + l and the high 2 bits from bits
// 2q, 2q + 1 of qh byte 32 hh + l; the code is the 6 bits less 32.
//   int8_act: S = sum_g sc_g isum_g over the whole super-block, y += d_a f(d) S;
//   f32_act:  y += f(d) sc_g sum(q x) per group of 16.
template <int AM, int MT, int R>
__device__ __forceinline__ void q6k_piece_dot(const uint8_t* s, const int (&wo)[R], int i, int ao, int astep, int M,
                                              const bool (&v)[R], float (&acc)[R][MT]) {
    const int hh = i >> 1, p = i & 1;
    const int g0 = 8 * hh + 2 * p;  // groups g0, g0 + 1 (quarter p) and g0 + 4, g0 + 5 (quarter p + 2)
    const uint32_t ush = 4u - 2u * (uint32_t)p, dsh = 2u * (uint32_t)p;
    // ca: quarter p, cb: quarter p + 2; the 6-bit fields as unsigned bytes, less 32 for int8_act
    uint32_t ca[R][8], cb[R][8];
    int sc[R][4];
    float fd[R];
#pragma unroll
    for (int h = 0; h < R; ++h) {
        uint32_t ql[8], qh[8];
        ld_words<8>(s, wo[h] + 64 * hh + 32 * p, ql);
        ld_words<8>(s, wo[h] + 128 + 32 * hh, qh);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            ca[h][k] = (ql[k] & 0x0F0F0F0Fu) | ((qh[k] << ush) & 0x30303030u);
            cb[h][k] = ((ql[k] >> 4) & 0x0F0F0F0Fu) | ((qh[k] >> dsh) & 0x30303030u);
            if (AM == A_INT8) ca[h][k] = __vsub4(ca[h][k], 0x20202020u), cb[h][k] = __vsub4(cb[h][k], 0x20202020u);
        }
        // the four group scales: two aligned 16-bit loads
        const uint32_t s01 = *reinterpret_cast<const uint16_t*>(s + wo[h] + 192 + g0);
        const uint32_t s45 = *reinterpret_cast<const uint16_t*>(s + wo[h] + 196 + g0);
        sc[h][0] = (int)(s01 << 24) >> 24, sc[h][1] = (int)(s01 << 16) >> 24;
        sc[h][2] = (int)(s45 << 24) >> 24, sc[h][3] = (int)(s45 << 16) >> 24;
        fd[h] = h2f(*reinterpret_cast<const uint16_t*>(s + wo[h] + 208));
    }
    if (AM == A_INT8) {
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m >= M) break;
            const uint8_t* a = s + ao + m * astep;
            const float da = *reinterpret_cast<const float*>(a + 416);
            a += 96 * i;  // slot 2i: quarter p; slot 2i + 1: quarter p + 2
            const uint4 a0 = ld128(a), a1 = ld128(a + 16), a2 = ld128(a + 48), a3 = ld128(a + 64);
#pragma unroll
            for (int h = 0; h < R; ++h) {
                const uint32_t* qa = ca[h];
                const uint32_t* qb = cb[h];
                int i0 = dp4a(qa[0], a0.x, 0), i1 = dp4a(qa[4], a1.x, 0);
                int i2 = dp4a(qb[0], a2.x, 0), i3 = dp4a(qb[4], a3.x, 0);
                i0 = dp4a(qa[1], a0.y, i0), i1 = dp4a(qa[5], a1.y, i1), i2 = dp4a(qb[1], a2.y, i2), i3 = dp4a(qb[5], a3.y, i3);
                i0 = dp4a(qa[2], a0.z, i0), i1 = dp4a(qa[6], a1.z, i1), i2 = dp4a(qb[2], a2.z, i2), i3 = dp4a(qb[6], a3.z, i3);
                i0 = dp4a(qa[3], a0.w, i0), i1 = dp4a(qa[7], a1.w, i1), i2 = dp4a(qb[3], a2.w, i2), i3 = dp4a(qb[7], a3.w, i3);
                const int S = quad_sum(sc[h][0] * i0 + sc[h][1] * i1 + sc[h][2] * i2 + sc[h][3] * i3);
                const float t = da * fd[h] * (float)S;
                acc[h][m] = v[h] && i == 0 ? acc[h][m] + t : acc[h][m];
            }
        }
    } else {
        const uint8_t* xa = s + ao + 288 * i;  // slot 2i: quarter p; slot 2i + 1: quarter p + 2
#pragma unroll
        for (int h = 0; h < R; ++h) {
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                // group g of the piece: 16 values; f(d) sc_g is an exact f32 product (11-bit by 7-bit)
                float sq[MT];
                dot_u8_f32_rows<4, 32, MT>((g < 2 ? ca[h] : cb[h]) + 4 * (g & 1), xa + 144 * (g >> 1) + 64 * (g & 1),
                                           astep, M, sq);
                const float e = fd[h] * (float)sc[h][g];
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    if (m >= M) break;
                    acc[h][m] = v[h] ? fmaf(e, sq[m], acc[h][m]) : acc[h][m];
                }
            }
        }
    }
}

// Weight units per row: 32-value blocks, or 64-value pieces of super-blocks.
__host__ __device__ constexpr int batch_units(int wt, int K) { return is_sb(wt) ? K / 64 : K / 32; }

// The contribution of unit b (b < nb) of the R rows at wrow[h] to acc.
template <int WT, int AM, int MT, int R>
__device__ __forceinline__ void unit_dot(const uint8_t* s, const int (&wrow)[R], int b, int acts, int astep, int M,
                                         const bool (&v)[R], float (&acc)[R][MT]) {
    constexpr int BB = unit_bytes(WT), ES = batch_act_unit(WT, AM);
    int wo[R];
    if (is_sb(WT)) {
#pragma unroll
        for (int h = 0; h < R; ++h) wo[h] = wrow[h] + (b >> 2) * BB;
        if (WT == T_Q4_K) q4k_piece_dot<AM, MT, R>(s, wo, b & 3, acts + (b >> 2) * ES, astep, M, v, acc);
        else q6k_piece_dot<AM, MT, R>(s, wo, b & 3, acts + (b >> 2) * ES, astep, M, v, acc);
    } else {
#pragma unroll
        for (int h = 0; h < R; ++h) wo[h] = wrow[h] + b * BB;
        block_dot<WT, AM, MT, R>(s, wo, acts + b * ES, astep, M, v, acc);
    }
}

// The first item whose cost reaches past lo (items are in cost order).
__device__ __forceinline__ int batch_first_item(const BatchParams& p, long long lo) {
    int a = 0, b = p.count;  // invariant: items before a end at or before lo
    while (a < b) {
        const int m = (a + b) >> 1;
        const long long end = m + 1 < p.count ? p.it[m + 1].c0 : p.total;
        if (end <= lo) a = m + 1;
        else b = m;
    }
    return a;
}

// The rows of item it whose first cost position lies in [lo, hi): [r0, r1).
__device__ __forceinline__ void batch_rows(const BatchItem& it, long long lo, long long hi, long long& r0, long long& r1) {
    const long long c0 = it.c0, rc = it.cpr;
    r0 = lo > c0 ? (lo - c0 + rc - 1) / rc : 0;
    r1 = hi > c0 ? (hi - c0 + rc - 1) / rc : 0;
    if (r1 > it.N) r1 = it.N;
    if (r0 > r1) r0 = r1;
}

__device__ __forceinline__ long long batch_row_bytes(int wt, int K) {
    return (long long)(K / unit_vals(wt)) * unit_bytes(wt);
}

// The item's activation rows into shared memory at o, unit (m, b) at
// (m * nu + b) * batch_act_unit, in the layout of weight type wt (the consumer
// warps; rows are contiguous).
template <int AM>
__device__ __forceinline__ void stage_acts(const BatchItem& it, int wt, uint8_t* o, int tid, int warp, int lane) {
    const int M = it.M;
    if (!is_sb(wt)) {
        if (AM == A_INT8) {
            for (int blk = tid; blk < M * (it.K / 32); blk += kBatchWarps * 32) {
                uint32_t c[8];
                float d;
                quant_q8_0_32(it.x + 32ll * blk, c, d);
                uint8_t* u = o + blk * 48;
                *reinterpret_cast<uint4*>(u) = make_uint4(c[0], c[1], c[2], c[3]);
                *reinterpret_cast<uint4*>(u + 16) = make_uint4(c[4], c[5], c[6], c[7]);
                *reinterpret_cast<float*>(u + 32) = h2f(f2h(d));
            }
        } else {
            const float4* src = reinterpret_cast<const float4*>(it.x);
            for (int idx = tid; idx < M * it.K / 4; idx += kBatchWarps * 32)
                *reinterpret_cast<float4*>(o + (idx >> 3) * 144 + (idx & 7) * 16) = __ldg(src + idx);
        }
        return;
    }
    // super-block types: one warp per 256 values, lane l taking values 8l..8l+7
    // (sub-block l / 4), stored in the slot order of weight type wt
    const int slot = batch_slot(wt, lane >> 2), part = lane & 3;
    for (int u = warp; u < M * (it.K / 256); u += kBatchWarps) {
        const float4* src = reinterpret_cast<const float4*>(it.x + 256ll * u + 8 * lane);
        const float4 v0 = __ldg(src), v1 = __ldg(src + 1);
        uint8_t* dst = o + u * batch_act_unit(T_Q4_K, AM);
        if (AM == A_INT8) {
            // Q8K: d = amax / 127 over the 256 values (f32), codes rounded from x / d
            float amax = fmaxf(fmaxf(fmaxf(fabsf(v0.x), fabsf(v0.y)), fmaxf(fabsf(v0.z), fabsf(v0.w))),
                               fmaxf(fmaxf(fabsf(v1.x), fabsf(v1.y)), fmaxf(fabsf(v1.z), fabsf(v1.w))));
#pragma unroll
            for (int off = 16; off; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
            float d, id;
            q8_scale(amax, d, id);
            const uint32_t w0 = pack4(q8_code(v0.x, id), q8_code(v0.y, id), q8_code(v0.z, id), q8_code(v0.w, id));
            const uint32_t w1 = pack4(q8_code(v1.x, id), q8_code(v1.y, id), q8_code(v1.z, id), q8_code(v1.w, id));
            *reinterpret_cast<uint2*>(dst + 48 * slot + 8 * part) = make_uint2(w0, w1);
            int sum = bsum4(w0) + bsum4(w1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            if (part == 0) *reinterpret_cast<int*>(dst + 384 + lane) = sum;  // sub-block lane / 4
            if (lane == 0) *reinterpret_cast<float*>(dst + 416) = d;
        } else {
            *reinterpret_cast<float4*>(dst + 144 * slot + 32 * part) = v0;
            *reinterpret_cast<float4*>(dst + 144 * slot + 32 * part + 16) = v1;
            float sum = ((v0.x + v0.y) + (v0.z + v0.w)) + ((v1.x + v1.y) + (v1.z + v1.w));
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            if (part == 0) *reinterpret_cast<float*>(dst + 1152 + lane) = sum;
        }
    }
}

// One piece (rows [r0, r1) of item it, weight type WT) through the ring.
template <int WT, int AM, int MT>
__device__ __forceinline__ void batch_piece(const BatchParams& p, const BatchItem& it, long long r0, long long r1,
                                            uint8_t* smem, int acts, uint64_t* bars, volatile int* flags, int& slot,
                                            uint32_t& phase, int warp, int lane) {
    constexpr int ES = batch_act_unit(WT, AM);
    constexpr int R = batch_rows_per_group(WT, AM, MT);
    const int S = p.stages;
    const int nb = batch_units(WT, it.K), M = it.M, rb = (int)batch_row_bytes(WT, it.K);
    // lanes in groups of lpr, R weight rows per group: lane gl of a group takes the
    // rows' units gl, gl + lpr, ... (bpl of them), and the group sums its lanes.
    // A warp holds rpw groups; its rows are j0 + grp + h * rpw.
    const int lpr = it.lpr, bpl = it.bpl, tr = it.tr, rpw = 32 / lpr;
    const int grp = lane / lpr, gl = lane - grp * lpr;
    const int astep = it.K / unit_vals(WT) * ES;
    for (long long r = r0; r < r1; r += tr) {
        const bool ok = mbar_wait(smem_u32(&bars[slot]), phase, flags, p.err);
        const int rows = (int)(r + tr < r1 ? tr : r1 - r);
        const int st = 1024 + slot * p.slot_bytes + (int)((r * rb) & 15);
        for (int j0 = warp * rpw * R; ok && j0 < rows; j0 += kBatchWarps * rpw * R) {
            bool jv[R];
            int wrow[R];
#pragma unroll
            for (int h = 0; h < R; ++h) {
                const int j = j0 + grp + h * rpw;
                jv[h] = grp < rpw && j < rows;
                wrow[h] = st + (jv[h] ? j : j0) * rb;  // lanes without a row read row j0 and discard it
            }
            float acc[R][MT];
#pragma unroll
            for (int h = 0; h < R; ++h)
#pragma unroll
                for (int m = 0; m < MT; ++m) acc[h][m] = 0.0f;
            for (int q = 0; q < bpl; ++q) {
                const int b = gl + q * lpr;
                bool v[R];
#pragma unroll
                for (int h = 0; h < R; ++h) v[h] = jv[h] && b < nb;
                unit_dot<WT, AM, MT, R>(smem, wrow, b < nb ? b : 0, acts, astep, M, v, acc);
            }
            // the group's sums: a tree over offsets below lpr, lanes past the group masked
#pragma unroll
            for (int off = 16; off; off >>= 1) {
                if (off >= lpr) continue;
                const bool in = gl + off < lpr;
#pragma unroll
                for (int h = 0; h < R; ++h)
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        const float o = __shfl_down_sync(0xffffffffu, acc[h][m], off);
                        acc[h][m] = in ? acc[h][m] + o : acc[h][m];
                    }
            }
            if (gl == 0 && !flags[0]) {
#pragma unroll
                for (int h = 0; h < R; ++h) {
                    if (!jv[h]) continue;
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        if (m >= M) break;
                        it.y[(long long)m * it.N + r + j0 + grp + h * rpw] = acc[h][m];
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars[S + slot]));
        if (++slot == S) slot = 0, phase ^= 1;
    }
}

template <int WT, int AM, int MT>
__global__ void __launch_bounds__((kBatchWarps + 1) * 32, 1) qmm_batch_kernel(const BatchParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = p.stages;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);                 // full[S], empty[S]
    volatile int* flags = reinterpret_cast<volatile int*>(smem + 256);  // [0] abort
    constexpr int ring = 1024;                                          // S slots of p.slot_bytes
    const int acts = ring + S * p.slot_bytes;                           // staged activations
    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(smem_u32(&bars[i]), 1);
            mbar_init(smem_u32(&bars[S + i]), kBatchWarps);
        }
        flags[0] = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const long long lo = p.total * blockIdx.x / gridDim.x, hi = p.total * (blockIdx.x + 1) / gridDim.x;

    if (warp == kBatchWarps) {
        // ------------------------------ producer ------------------------------
        if (lane != 0) return;
        long long g = 0;
        int slot = 0, round = 0;
        bool ok = true;
        for (int i = batch_first_item(p, lo); i < p.count && p.it[i].c0 < hi && ok; ++i) {
            const BatchItem& it = p.it[i];
            const long long rb = batch_row_bytes(WT == T_MIX ? it.wt : WT, it.K);
            long long r0, r1;
            batch_rows(it, lo, hi, r0, r1);
            const int tr = it.tr;
            const long long end = (long long)it.N * rb;  // the item's buffer
            for (long long r = r0; r < r1 && ok; r += tr, ++g) {
                if (round > 0 && !(ok = mbar_wait(smem_u32(&bars[S + slot]), (uint32_t)((round - 1) & 1), flags, p.err))) break;
                uint8_t* st = smem + ring + slot * p.slot_bytes;
                const long long s0 = r * rb, e = (r + tr < r1 ? r + tr : r1) * rb;
                const long long a = s0 & ~15ll;
                long long b = (e + 15) & ~15ll;
                if (b > end) {  // the buffer's ragged end: its last bytes by plain loads
                    b = e & ~15ll;
                    for (long long q = b > a ? b : a; q < e; ++q) st[q - a] = it.wq[q];
                    fence_proxy_async();
                }
                const uint32_t fb = smem_u32(&bars[slot]);
                mbar_arrive_tx(fb, (uint32_t)(b > a ? b - a : 0));
                if (b > a) bulk_g2s(smem_u32(st), it.wq + a, (uint32_t)(b - a), fb);
                if (++slot == S) slot = 0, ++round;
            }
        }
        const long long first = g > S ? g - S : 0;
        for (long long q = first; q < g; ++q) mbar_drain(smem_u32(&bars[q % S]), (uint32_t)((q / S) & 1), flags, p.err);
        return;
    }

    // ------------------------------ consumers ------------------------------
    int slot = 0;
    uint32_t phase = 0;
    const float* prep_x = nullptr;  // the activations now in shared memory
    int prep_m = 0, prep_k = 0, prep_layout = -1;
    for (int i = batch_first_item(p, lo); i < p.count && p.it[i].c0 < hi; ++i) {
        const BatchItem& it = p.it[i];
        const int wt = WT == T_MIX ? it.wt : WT;
        long long r0, r1;
        batch_rows(it, lo, hi, r0, r1);
        if (r0 >= r1) continue;
        const int layout = is_sb(wt) ? wt : 0;  // Q8_0 blocks, or Q8K in a type's slot order
        if (it.x != prep_x || it.M != prep_m || it.K != prep_k || layout != prep_layout) {
            consumer_sync<kBatchWarps>();  // the previous activations are no longer read
            stage_acts<AM>(it, wt, smem + acts, tid, warp, lane);
            consumer_sync<kBatchWarps>();
            prep_x = it.x, prep_m = it.M, prep_k = it.K, prep_layout = layout;
        }
        if (WT != T_MIX) {
            batch_piece<WT, AM, MT>(p, it, r0, r1, smem, acts, bars, flags, slot, phase, warp, lane);
        } else {
            switch (wt) {
                case T_Q8_0: batch_piece<T_Q8_0, AM, MT>(p, it, r0, r1, smem, acts, bars, flags, slot, phase, warp, lane); break;
                case T_Q4_0: batch_piece<T_Q4_0, AM, MT>(p, it, r0, r1, smem, acts, bars, flags, slot, phase, warp, lane); break;
                case T_Q5_0: batch_piece<T_Q5_0, AM, MT>(p, it, r0, r1, smem, acts, bars, flags, slot, phase, warp, lane); break;
                case T_Q4_K: batch_piece<T_Q4_K, AM, MT>(p, it, r0, r1, smem, acts, bars, flags, slot, phase, warp, lane); break;
                default: batch_piece<T_Q6_K, AM, MT>(p, it, r0, r1, smem, acts, bars, flags, slot, phase, warp, lane); break;
            }
        }
    }
}

template <int WT, int AM>
cudaError_t batch_go_mt(BatchParams& p, int mt, int grid, int smem_max, cudaStream_t s) {
    const long long acts = ((long long)p.act_bytes + 15) / 16 * 16;
    // as many ring slots as fit beside the activations, up to kBatchStagesMax; two at least
    const long long room = (long long)smem_max - 1024 - acts - 64;
    p.stages = (int)std::min<long long>(kBatchStagesMax, room / p.slot_bytes);
    if (p.stages < 2) return cudaErrorInvalidValue;
    const size_t smem = 1024 + (size_t)p.stages * p.slot_bytes + (size_t)acts + 64;
    static unsigned long long done[4];  // per MT variant: devices whose shared-memory limit is raised
    auto launch = [&](auto* k, unsigned long long& d) {
        cudaError_t e = ensure_smem(k, smem_max, d);
        if (e != cudaSuccess) return e;
        k<<<grid, (kBatchWarps + 1) * 32, smem, s>>>(p);
        return cudaGetLastError();
    };
    switch (mt) {
        case 1: return launch(qmm_batch_kernel<WT, AM, 1>, done[0]);
        case 2: return launch(qmm_batch_kernel<WT, AM, 2>, done[1]);
        case 4: return launch(qmm_batch_kernel<WT, AM, 4>, done[2]);
        default: return launch(qmm_batch_kernel<WT, AM, 8>, done[3]);
    }
}

}  // namespace
}  // namespace qmm
