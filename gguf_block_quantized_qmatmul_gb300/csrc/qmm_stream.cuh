// qmm_stream.cuh -- the streaming kernel behind qmm_matmul and qmm_block_sums.
//
// One persistent CTA per SM.  A producer warp streams the raw GGUF bytes of
// 16-row weight tiles into a ring of shared-memory stages with 1-D bulk
// copies (cp.async.bulk, mbarrier completion); CW consumer warps compute on
// each stage while the next ones are in flight: one warp-level tensor-core
// product per 32-value block (Q8_0, Q4_0, Q5_0), sub-block of 32 (Q4_K) or
// group of 16 (Q6_K, one k16 MMA) of 16 rows against 8
// activation rows (int8: mma.m16n8k32.s8, exact int32 block sums) or 4
// activation rows split into two f16 pieces (f32_act: mma.m16n8k16.f16, f32
// accumulate).  (Decode int8_act with M <= 8 runs in qmm_gemv.cuh instead.)
//
// Block arithmetic ("同一个 GGUF，CPU 和 Metal 生成的文字不一样" section 出处):
//   int8_act (CPU form): per-block exact int32 sums isum of weight codes times
//     the row-quantized activation codes, then
//     Q8_0: y += f(d_w) f(d_a) isum;  Q4_K: S_sc = sum_j sc_j isum_j,
//     S_m = sum_j m_j (sum of sub-block j's activation codes),
//     y += d_a (f(d) S_sc - f(dmin) S_m);  Q6_K: S = sum_j sc_j isum_j over its
//     16 groups of 16 (signed 6-bit codes), y += d_a f(d) S.
//   f32_act (Metal form): each activation row is scaled by a power of two and
//     split into two f16 pieces (x 2^s = hi + lo to 2^-22 relative); weight
//     codes are exact in f16; y += f(d) sum(q x) (Q8_0) or e_j sum(q x) -
//     o_j sum(x) with e_j = f(d) sc_j, o_j = f(dmin) m_j (Q4_K).
// Activations of the CTA's (row chunk, K slice) are prepared in shared memory
// by the consumer warps while the producer already streams the first weight
// stages.  When the K dimension is split across CTAs (to fit the activation
// slice in shared memory), partial sums go to a workspace and the
// last-arriving CTA of a tile adds them in slice order (deterministic).
#pragma once

#include "qmm_device.cuh"

namespace qmm {

template <int WT>
struct Unit;
template <>
struct Unit<T_Q8_0> {
    static constexpr int vals = 32, bytes = 34, per_stage = 32;
};
template <>
struct Unit<T_Q4_K> {
    static constexpr int vals = 256, bytes = 144, per_stage = 8;
};
template <>
struct Unit<T_Q4_0> {
    static constexpr int vals = 32, bytes = 18, per_stage = 32;
};
template <>
struct Unit<T_Q5_0> {
    static constexpr int vals = 32, bytes = 22, per_stage = 32;
};
template <>
struct Unit<T_Q6_K> {
    static constexpr int vals = 256, bytes = 210, per_stage = 8;
};
__host__ __device__ constexpr int unit_vals(int wt) { return wt == T_Q4_K || wt == T_Q6_K ? 256 : 32; }
__host__ __device__ constexpr int unit_bytes(int wt) {
    return wt == T_Q4_K ? 144 : wt == T_Q6_K ? 210 : wt == T_Q4_0 ? 18 : wt == T_Q5_0 ? 22 : 34;
}
// super-block weight types (paired with Q8K activations)
__host__ __device__ constexpr bool is_sb(int wt) { return wt == T_Q4_K || wt == T_Q6_K; }

// Signed codes of values 8t..8t+7 of a 32-value weight block (2-byte
// aligned in shared memory): w0 holds values 8t..8t+3, w1 8t+4..8t+7, one
// byte each.  Q8_0: the int8 codes; Q4_0 / Q5_0: the 4-bit field (low nibble
// of byte j for value j, high nibble for value j + 16) plus, for Q5_0, bit 4
// from the block's 32-bit word of fifth bits, minus the offset 8 / 16.
template <int WT>
__device__ __forceinline__ void b32_codes8(const uint8_t* blk, int t, uint32_t& w0, uint32_t& w1) {
    if (WT == T_Q8_0) {
        lds8_unaligned(blk + 2 + 8 * t, w0, w1);
    } else {
        constexpr int QS = WT == T_Q5_0 ? 6 : 2;
        uint32_t x0, x1;
        lds8_unaligned(blk + QS + 8 * (t & 1), x0, x1);
        const uint32_t sh = 4u * (uint32_t)(t >> 1);
        uint32_t l0 = (x0 >> sh) & 0x0F0F0F0Fu, l1 = (x1 >> sh) & 0x0F0F0F0Fu;
        if (WT == T_Q5_0) {
            const uint16_t* hw = reinterpret_cast<const uint16_t*>(blk + 2);
            const uint32_t hb = (((uint32_t)hw[0] | ((uint32_t)hw[1] << 16)) >> (8 * t)) & 0xFFu;
            // bits 0..3 of hb to bit 4 of bytes 0..3 (the shifted copies do not overlap)
            l0 |= (((hb & 0xFu) * 0x00204081u) & 0x01010101u) << 4;
            l1 |= ((((hb >> 4) & 0xFu) * 0x00204081u) & 0x01010101u) << 4;
            w0 = __vsub4(l0, 0x10101010u);
            w1 = __vsub4(l1, 0x10101010u);
        } else {
            w0 = __vsub4(l0, 0x08080808u);
            w1 = __vsub4(l1, 0x08080808u);
        }
    }
}

// consumer warps per CTA for a kernel variant (host and device agree on it)
__host__ __device__ constexpr int consumer_warps(int wt, int am, int nt) {
    return is_b32(wt) && nt <= 2 ? 16 : 8;
}
// activation rows per CTA chunk
__host__ __device__ constexpr int chunk_rows(int am, int nt) { return am == A_INT8 ? 8 * nt : 4 * nt; }

// ---------------------------------------------------------------------------
// activation preparation (consumer warps)
// ---------------------------------------------------------------------------

template <int WT, int AM, int CW>
__device__ __forceinline__ void prepare_acts(const StreamParams& p, uint8_t* smem, int m0, int k0, int klen, int tid) {
    constexpr int NTH = CW * 32;
    const int MR = p.mr;
    if (AM == A_INT8 && is_b32(WT)) {  // Q8_0 activations
        uint8_t* codes = smem + p.off_codes;
        float* da = reinterpret_cast<float*>(smem + p.off_scale);
        const int nb = p.slice_units;  // blocks of 32 in the (largest) slice
        for (int idx = tid; idx < MR * nb; idx += NTH) {
            const int r = idx / nb, b = idx - r * nb;
            const int m = m0 + r;
            uint32_t c[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            float s = 0.0f;
            if (m < p.M && b * 32 < klen) {
                float d;
                quant_q8_0_32(p.x + (long long)m * p.K + k0 + b * 32, c, d);
                s = h2f(f2h(d));
            }
            uint4* d0 = reinterpret_cast<uint4*>(codes + r * p.code_pitch + b * 32);
            uint4* d1 = d0 + 1;
            *d0 = make_uint4(c[0], c[1], c[2], c[3]);
            *d1 = make_uint4(c[4], c[5], c[6], c[7]);
            da[r * p.scale_pitch + b] = s;
        }
    } else if (AM == A_INT8 && is_sb(WT)) {  // Q8K activations (Q4_K also needs the sums of each 32)
        uint8_t* codes = smem + p.off_codes;
        float* da = reinterpret_cast<float*>(smem + p.off_scale);
        int* bs = reinterpret_cast<int*>(smem + p.off_aux);
        const int nsb = p.slice_units;  // super-blocks of 256
        for (int idx = tid; idx < MR * nsb; idx += NTH) {
            const int r = idx / nsb, sb = idx - r * nsb;
            const int m = m0 + r;
            const bool live = m < p.M && sb * 256 < klen;
            const float* src = p.x + (long long)m * p.K + k0 + sb * 256;
            float d = 0.0f, id = 0.0f;
            if (live) q8_scale(q8k_amax(src), d, id);
            for (int j = 0; j < 8; ++j) {
                uint32_t w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                int sum = 0;
                if (live) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        float4 v = __ldg(reinterpret_cast<const float4*>(src + 32 * j) + i);
                        w[i] = pack4(q8_code(v.x, id), q8_code(v.y, id), q8_code(v.z, id), q8_code(v.w, id));
                        sum += bsum4(w[i]);
                    }
                }
                uint4* d0 = reinterpret_cast<uint4*>(codes + r * p.code_pitch + sb * 256 + 32 * j);
                uint4* d1 = d0 + 1;
                *d0 = make_uint4(w[0], w[1], w[2], w[3]);
                *d1 = make_uint4(w[4], w[5], w[6], w[7]);
                if (WT == T_Q4_K) bs[r * p.aux_pitch + sb * 8 + j] = sum;
            }
            da[r * p.scale_pitch + sb] = d;
        }
    } else {
        // f32_act: per-row power-of-two scale from the slice's max |x|, then
        // two f16 pieces per value; Q4_K also needs the scaled sum of each 32.
        __half* pieces = reinterpret_cast<__half*>(smem + p.off_codes);
        float* rs = reinterpret_cast<float*>(smem + p.off_rs);   // [MR][2]: 2^s, 2^-s
        float* xs = reinterpret_cast<float*>(smem + p.off_aux);  // [MR][slice/32]
        const int warp = tid >> 5, lane = tid & 31;
        for (int r = warp; r < MR; r += CW) {
            const int m = m0 + r;
            float amax = 0.0f;
            if (m < p.M) {
                const float4* src = reinterpret_cast<const float4*>(p.x + (long long)m * p.K + k0);
                for (int i = lane; i < klen / 4; i += 32) {
                    float4 v = __ldg(src + i);
                    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
                }
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            if (lane == 0) {
                int s = 0;
                if (amax > 0.0f) {
                    const int e = (int)((__float_as_uint(amax) >> 23) & 0xff) - 127;  // amax in [2^e, 2^(e+1))
                    s = 14 - e;
                    s = s > 100 ? 100 : (s < -100 ? -100 : s);
                }
                rs[2 * r] = ldexpf(1.0f, s);
                rs[2 * r + 1] = ldexpf(1.0f, -s);
            }
        }
        consumer_sync<CW>();
        const int nch = p.slice_units * Unit<WT>::vals / 32;  // chunks of 32 values
        for (int idx = tid; idx < MR * nch; idx += NTH) {
            const int r = idx / nch, c = idx - r * nch;
            const int m = m0 + r;
            uint32_t hw[16], lw[16];
            float sum = 0.0f;
            if (m < p.M && c * 32 < klen) {
                const float scale = rs[2 * r];
                const float4* src = reinterpret_cast<const float4*>(p.x + (long long)m * p.K + k0 + c * 32);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 v4 = __ldg(src + i);
                    const float v[4] = {__fmul_rn(v4.x, scale), __fmul_rn(v4.y, scale), __fmul_rn(v4.z, scale),
                                        __fmul_rn(v4.w, scale)};
                    uint32_t hb[4], lb[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const __half h = __float2half_rn(v[k]);
                        const __half l = __float2half_rn(__fsub_rn(v[k], __half2float(h)));
                        hb[k] = __half_as_ushort(h);
                        lb[k] = __half_as_ushort(l);
                        sum = __fadd_rn(sum, v[k]);
                    }
                    hw[2 * i] = hb[0] | (hb[1] << 16);
                    hw[2 * i + 1] = hb[2] | (hb[3] << 16);
                    lw[2 * i] = lb[0] | (lb[1] << 16);
                    lw[2 * i + 1] = lb[2] | (lb[3] << 16);
                }
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) hw[i] = lw[i] = 0u;
            }
            uint4* dh = reinterpret_cast<uint4*>(pieces + (long long)(2 * r) * p.code_pitch + c * 32);
            uint4* dl = reinterpret_cast<uint4*>(pieces + (long long)(2 * r + 1) * p.code_pitch + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                dh[i] = make_uint4(hw[4 * i], hw[4 * i + 1], hw[4 * i + 2], hw[4 * i + 3]);
                dl[i] = make_uint4(lw[4 * i], lw[4 * i + 1], lw[4 * i + 2], lw[4 * i + 3]);
            }
            if (WT == T_Q4_K) xs[r * p.aux_pitch + c] = sum;
        }
    }
}

// ---------------------------------------------------------------------------
// warp tensor-core products over 16-row blocks
// ---------------------------------------------------------------------------

// acc layout: int8: acc[nt][0..3] = (row g, col 2t), (g, 2t+1), (g+8, 2t), (g+8, 2t+1)
//             f32 : acc[nt][0..1] = (row g, act row 4nt+t), (g+8, 4nt+t)
template <int WT, int AM, int NT, int EPI, int CW>
__device__ __forceinline__ void stage_mma(const StreamParams& p, const uint8_t* smem, const uint8_t* st, int nunits,
                                          int ur0, int gu0, int off0, int off1, int warp, int lane,
                                          float (&acc)[NT][4], int tile, int m0) {
    const int g = lane >> 2, t = lane & 3;
    const uint8_t* row0 = st + g * p.row_stride + off0;
    const uint8_t* row1 = st + (g + 8) * p.row_stride + off1;
    for (int u = warp; u < nunits; u += CW) {
        const int ur = ur0 + u;  // unit index inside the K slice
        if (is_b32(WT)) {
            const uint8_t* b0 = row0 + u * Unit<WT>::bytes;
            const uint8_t* b1 = row1 + u * Unit<WT>::bytes;
            const float dw0 = h2f(*reinterpret_cast<const uint16_t*>(b0));
            const float dw1 = h2f(*reinterpret_cast<const uint16_t*>(b1));
            uint32_t w0, w1, v0, v1;  // 8 signed codes of rows g and g+8: values 8t..8t+7
            b32_codes8<WT>(b0, t, w0, w1);
            b32_codes8<WT>(b1, t, v0, v1);
            if (AM == A_INT8) {
                const uint8_t* codes = smem + p.off_codes;
                const float* da = reinterpret_cast<const float*>(smem + p.off_scale);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const uint2 bb = ld64(codes + (nt * 8 + g) * p.code_pitch + ur * 32 + 8 * t);
                    int d[4];
                    mma_s8(d, w0, v0, w1, v1, bb.x, bb.y);
                    if (EPI == E_Y) {
                        const float da0 = da[(nt * 8 + 2 * t) * p.scale_pitch + ur];
                        const float da1 = da[(nt * 8 + 2 * t + 1) * p.scale_pitch + ur];
                        acc[nt][0] = fmaf((float)d[0], dw0 * da0, acc[nt][0]);
                        acc[nt][1] = fmaf((float)d[1], dw0 * da1, acc[nt][1]);
                        acc[nt][2] = fmaf((float)d[2], dw1 * da0, acc[nt][2]);
                        acc[nt][3] = fmaf((float)d[3], dw1 * da1, acc[nt][3]);
                    } else {
                        const int n0 = tile * kTileRows + g, n1 = n0 + 8;
                        const int ma = m0 + nt * 8 + 2 * t, mb = ma + 1;
                        const long long nbk = p.units, gb = gu0 + u;
                        if (ma < p.M && n0 < p.N) p.sums[((long long)ma * p.N + n0) * nbk + gb] = d[0];
                        if (mb < p.M && n0 < p.N) p.sums[((long long)mb * p.N + n0) * nbk + gb] = d[1];
                        if (ma < p.M && n1 < p.N) p.sums[((long long)ma * p.N + n1) * nbk + gb] = d[2];
                        if (mb < p.M && n1 < p.N) p.sums[((long long)mb * p.N + n1) * nbk + gb] = d[3];
                    }
                }
            } else {
                const uint8_t* pieces = smem + p.off_codes;
                const uint32_t A1a0 = s8x2_to_h2(w0, SEL01), A1a2 = s8x2_to_h2(w0, SEL23);
                const uint32_t A1a1 = s8x2_to_h2(v0, SEL01), A1a3 = s8x2_to_h2(v0, SEL23);
                const uint32_t A2a0 = s8x2_to_h2(w1, SEL01), A2a2 = s8x2_to_h2(w1, SEL23);
                const uint32_t A2a1 = s8x2_to_h2(v1, SEL01), A2a3 = s8x2_to_h2(v1, SEL23);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int prow = 2 * (nt * 4 + (g >> 1)) + (g & 1);
                    const uint4 bb = ld128(pieces + ((long long)prow * p.code_pitch + ur * 32 + 8 * t) * 2);
                    float d[4] = {0.f, 0.f, 0.f, 0.f};
                    mma_f16(d, A1a0, A1a1, A1a2, A1a3, bb.x, bb.y);
                    mma_f16(d, A2a0, A2a1, A2a2, A2a3, bb.z, bb.w);
                    acc[nt][0] = fmaf(dw0, d[0] + d[1], acc[nt][0]);
                    acc[nt][1] = fmaf(dw1, d[2] + d[3], acc[nt][1]);
                }
            }
        } else if (WT == T_Q6_K) {
            // Q6_K super-block: 16 groups of 16 values, one k16 MMA each.  Group
            // j = 8h + 2q + s holds values 128h + 32q + 16s + l (l < 16); thread t
            // takes l = 4t..4t+3: one ql word (nibble plane q / 2) and one qh
            // word (bit pair q) per row.  Blocks are 2-byte aligned: words are
            // read from the rounded-down start and realigned by a funnel shift.
            const int o0 = (int)(row0 - smem) + u * 210, o1 = (int)(row1 - smem) + u * 210;
            const uint8_t* a0p = smem + (o0 & ~3);
            const uint8_t* a1p = smem + (o1 & ~3);
            const uint32_t sh0 = (uint32_t)(o0 & 2) * 8u, sh1 = (uint32_t)(o1 & 2) * 8u;
            auto w0 = [&](int off) { return __funnelshift_r(ld32(a0p + off), ld32(a0p + off + 4), sh0); };
            auto w1 = [&](int off) { return __funnelshift_r(ld32(a1p + off), ld32(a1p + off + 4), sh1); };
            const float fD0 = h2f(*reinterpret_cast<const uint16_t*>(smem + o0 + 208));
            const float fD1 = h2f(*reinterpret_cast<const uint16_t*>(smem + o1 + 208));
            const int8_t* sc0p = reinterpret_cast<const int8_t*>(smem + o0 + 192);
            const int8_t* sc1p = reinterpret_cast<const int8_t*>(smem + o1 + 192);
            int ssc[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) ssc[nt][i] = 0;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int sg = 0; sg < 2; ++sg) {
                    const int lo = 16 * sg + 4 * t;  // l of this thread's first value
                    const uint32_t L00 = w0(64 * h + lo), L01 = w0(64 * h + 32 + lo), H0 = w0(128 + 32 * h + lo);
                    const uint32_t L10 = w1(64 * h + lo), L11 = w1(64 * h + 32 + lo), H1 = w1(128 + 32 * h + lo);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int j = 8 * h + 2 * q + sg;
                        const int vb = 128 * h + 32 * q + lo;  // value index of this thread's first value
                        const uint32_t n0 = ((q & 1 ? L01 : L00) >> (4 * (q >> 1))) & 0x0F0F0F0Fu;
                        const uint32_t n1 = ((q & 1 ? L11 : L10) >> (4 * (q >> 1))) & 0x0F0F0F0Fu;
                        const uint32_t c0 = __vsub4(n0 | (((H0 >> (2 * q)) & 0x03030303u) << 4), 0x20202020u);
                        const uint32_t c1 = __vsub4(n1 | (((H1 >> (2 * q)) & 0x03030303u) << 4), 0x20202020u);
                        if (AM == A_INT8) {
                            const uint8_t* codes = smem + p.off_codes;
                            const int s0 = sc0p[j], s1 = sc1p[j];
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
                                const uint32_t bb = ld32(codes + (nt * 8 + g) * p.code_pitch + ur * 256 + vb);
                                int d[4];
                                mma_s8_k16(d, c0, c1, bb);
                                ssc[nt][0] += s0 * d[0];
                                ssc[nt][1] += s0 * d[1];
                                ssc[nt][2] += s1 * d[2];
                                ssc[nt][3] += s1 * d[3];
                            }
                        } else {
                            const uint8_t* pieces = smem + p.off_codes;
                            const uint32_t a0 = s8x2_to_h2(c0, SEL01), a2 = s8x2_to_h2(c0, SEL23);
                            const uint32_t a1 = s8x2_to_h2(c1, SEL01), a3 = s8x2_to_h2(c1, SEL23);
                            const float e0 = __fmul_rn(fD0, (float)sc0p[j]), e1 = __fmul_rn(fD1, (float)sc1p[j]);
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
                                const int prow = 2 * (nt * 4 + (g >> 1)) + (g & 1);
                                const uint2 bb = ld64(pieces + ((long long)prow * p.code_pitch + ur * 256 + vb) * 2);
                                float d[4] = {0.f, 0.f, 0.f, 0.f};
                                mma_f16(d, a0, a1, a2, a3, bb.x, bb.y);
                                acc[nt][0] = fmaf(e0, d[0] + d[1], acc[nt][0]);
                                acc[nt][1] = fmaf(e1, d[2] + d[3], acc[nt][1]);
                            }
                        }
                    }
                }
            if (AM == A_INT8) {
                const float* da = reinterpret_cast<const float*>(smem + p.off_scale);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    if (EPI == E_Y) {
                        const float da0 = da[(nt * 8 + 2 * t) * p.scale_pitch + ur];
                        const float da1 = da[(nt * 8 + 2 * t + 1) * p.scale_pitch + ur];
                        acc[nt][0] += da0 * (fD0 * (float)ssc[nt][0]);
                        acc[nt][1] += da1 * (fD0 * (float)ssc[nt][1]);
                        acc[nt][2] += da0 * (fD1 * (float)ssc[nt][2]);
                        acc[nt][3] += da1 * (fD1 * (float)ssc[nt][3]);
                    } else {
                        const int n0 = tile * kTileRows + g, n1 = n0 + 8;
                        const int ma = m0 + nt * 8 + 2 * t, mb = ma + 1;
                        const long long nsb = p.units, gs = gu0 + u;
                        if (ma < p.M && n0 < p.N) p.sums[((long long)ma * p.N + n0) * nsb + gs] = ssc[nt][0];
                        if (mb < p.M && n0 < p.N) p.sums[((long long)mb * p.N + n0) * nsb + gs] = ssc[nt][1];
                        if (ma < p.M && n1 < p.N) p.sums[((long long)ma * p.N + n1) * nsb + gs] = ssc[nt][2];
                        if (mb < p.M && n1 < p.N) p.sums[((long long)mb * p.N + n1) * nsb + gs] = ssc[nt][3];
                    }
                }
            }
        } else {  // Q4_K super-block
            const uint8_t* s0 = row0 + u * 144;
            const uint8_t* s1 = row1 + u * 144;
            const uint4 h0 = ld128(s0), h1 = ld128(s1);
            const uint32_t W00 = h0.y, W01 = h0.z, W02 = h0.w, W10 = h1.y, W11 = h1.z, W12 = h1.w;
            const float fD0 = h2f(h0.x), fDm0 = h2f(h0.x >> 16), fD1 = h2f(h1.x), fDm1 = h2f(h1.x >> 16);
            if (AM == A_INT8) {
                const uint8_t* codes = smem + p.off_codes;
                const float* da = reinterpret_cast<const float*>(smem + p.off_scale);
                const int* bs = reinterpret_cast<const int*>(smem + p.off_aux);
                int ssc[NT][4], smn[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) ssc[nt][i] = smn[nt][i] = 0;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint2 q0 = ld64(s0 + 16 + 32 * c + 8 * t);
                    const uint2 q1 = ld64(s1 + 16 + 32 * c + 8 * t);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int j = 2 * c + h;
                        const uint32_t a0 = (q0.x >> (4 * h)) & 0x0F0F0F0Fu, a2 = (q0.y >> (4 * h)) & 0x0F0F0F0Fu;
                        const uint32_t a1 = (q1.x >> (4 * h)) & 0x0F0F0F0Fu, a3 = (q1.y >> (4 * h)) & 0x0F0F0F0Fu;
                        const int sc0 = q4k_sc(W00, W02, j), mn0 = q4k_mn(W01, W02, j);
                        const int sc1 = q4k_sc(W10, W12, j), mn1 = q4k_mn(W11, W12, j);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const uint2 bb = ld64(codes + (nt * 8 + g) * p.code_pitch + ur * 256 + 32 * j + 8 * t);
                            int d[4];
                            mma_s8(d, a0, a1, a2, a3, bb.x, bb.y);
                            const int bs0 = bs[(nt * 8 + 2 * t) * p.aux_pitch + ur * 8 + j];
                            const int bs1 = bs[(nt * 8 + 2 * t + 1) * p.aux_pitch + ur * 8 + j];
                            ssc[nt][0] += sc0 * d[0];
                            ssc[nt][1] += sc0 * d[1];
                            ssc[nt][2] += sc1 * d[2];
                            ssc[nt][3] += sc1 * d[3];
                            smn[nt][0] += mn0 * bs0;
                            smn[nt][1] += mn0 * bs1;
                            smn[nt][2] += mn1 * bs0;
                            smn[nt][3] += mn1 * bs1;
                        }
                    }
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    if (EPI == E_Y) {
                        const float da0 = da[(nt * 8 + 2 * t) * p.scale_pitch + ur];
                        const float da1 = da[(nt * 8 + 2 * t + 1) * p.scale_pitch + ur];
                        acc[nt][0] += da0 * (fD0 * (float)ssc[nt][0] - fDm0 * (float)smn[nt][0]);
                        acc[nt][1] += da1 * (fD0 * (float)ssc[nt][1] - fDm0 * (float)smn[nt][1]);
                        acc[nt][2] += da0 * (fD1 * (float)ssc[nt][2] - fDm1 * (float)smn[nt][2]);
                        acc[nt][3] += da1 * (fD1 * (float)ssc[nt][3] - fDm1 * (float)smn[nt][3]);
                    } else {
                        const int n0 = tile * kTileRows + g, n1 = n0 + 8;
                        const int ma = m0 + nt * 8 + 2 * t, mb = ma + 1;
                        const long long nsb = p.units, gs = gu0 + u;
                        if (ma < p.M && n0 < p.N) { int* o = p.sums + (((long long)ma * p.N + n0) * nsb + gs) * 2; o[0] = ssc[nt][0]; o[1] = smn[nt][0]; }
                        if (mb < p.M && n0 < p.N) { int* o = p.sums + (((long long)mb * p.N + n0) * nsb + gs) * 2; o[0] = ssc[nt][1]; o[1] = smn[nt][1]; }
                        if (ma < p.M && n1 < p.N) { int* o = p.sums + (((long long)ma * p.N + n1) * nsb + gs) * 2; o[0] = ssc[nt][2]; o[1] = smn[nt][2]; }
                        if (mb < p.M && n1 < p.N) { int* o = p.sums + (((long long)mb * p.N + n1) * nsb + gs) * 2; o[0] = ssc[nt][3]; o[1] = smn[nt][3]; }
                    }
                }
            } else {
                const uint8_t* pieces = smem + p.off_codes;
                const float* xs = reinterpret_cast<const float*>(smem + p.off_aux);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint2 q0 = ld64(s0 + 16 + 32 * c + 8 * t);
                    const uint2 q1 = ld64(s1 + 16 + 32 * c + 8 * t);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int j = 2 * c + h;
                        const uint32_t n0x = (q0.x >> (4 * h)) & 0x0F0F0F0Fu, n0y = (q0.y >> (4 * h)) & 0x0F0F0F0Fu;
                        const uint32_t n1x = (q1.x >> (4 * h)) & 0x0F0F0F0Fu, n1y = (q1.y >> (4 * h)) & 0x0F0F0F0Fu;
                        const uint32_t A1a0 = u4x2_to_h2(n0x, SEL01), A1a2 = u4x2_to_h2(n0x, SEL23);
                        const uint32_t A1a1 = u4x2_to_h2(n1x, SEL01), A1a3 = u4x2_to_h2(n1x, SEL23);
                        const uint32_t A2a0 = u4x2_to_h2(n0y, SEL01), A2a2 = u4x2_to_h2(n0y, SEL23);
                        const uint32_t A2a1 = u4x2_to_h2(n1y, SEL01), A2a3 = u4x2_to_h2(n1y, SEL23);
                        const float e0 = fD0 * (float)q4k_sc(W00, W02, j), o0 = fDm0 * (float)q4k_mn(W01, W02, j);
                        const float e1 = fD1 * (float)q4k_sc(W10, W12, j), o1 = fDm1 * (float)q4k_mn(W11, W12, j);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const int prow = 2 * (nt * 4 + (g >> 1)) + (g & 1);
                            const uint4 bb = ld128(pieces + ((long long)prow * p.code_pitch + ur * 256 + 32 * j + 8 * t) * 2);
                            float d[4] = {0.f, 0.f, 0.f, 0.f};
                            mma_f16(d, A1a0, A1a1, A1a2, A1a3, bb.x, bb.y);
                            mma_f16(d, A2a0, A2a1, A2a2, A2a3, bb.z, bb.w);
                            const float X = xs[(nt * 4 + t) * p.aux_pitch + ur * 8 + j];
                            acc[nt][0] += fmaf(e0, d[0] + d[1], -o0 * X);
                            acc[nt][1] += fmaf(e1, d[2] + d[3], -o1 * X);
                        }
                    }
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------

template <int WT, int AM, int NT, int EPI>
__global__ void __launch_bounds__((consumer_warps(WT, AM, NT) + 1) * 32, 1)
    qmm_stream_kernel(const StreamParams p) {
    constexpr int CW = consumer_warps(WT, AM, NT);
    constexpr int UB = Unit<WT>::bytes;
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = p.stages;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);  // full[S], empty[S]
    volatile int* flags = reinterpret_cast<volatile int*>(smem + p.off_flags);  // [0] abort, [1] last
    const int pair = blockIdx.x % p.pairs;
    const int slice = pair % p.kslices, mc = pair / p.kslices;
    const int tile0 = blockIdx.x / p.pairs;
    const int m0 = mc * p.mr;
    const int su0 = slice * p.slice_units;                 // first unit of the slice
    const int sunits = min(p.slice_units, p.units - su0);  // units in this slice
    const int nchunks = (sunits + p.ups - 1) / p.ups;

    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(smem_u32(&bars[i]), 1);
            mbar_init(smem_u32(&bars[S + i]), CW);
        }
        flags[0] = 0;
        flags[1] = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == CW) {
        // ----------------------------- producer -----------------------------
        // Lane r (< 16) owns weight row r of the tile: it copies the 16-byte
        // aligned superset of the row's chunk with one bulk copy (and the
        // ragged tail at the very end of the buffer with plain loads); lane 0
        // waits for the slot and posts the stage's byte count.
        long long g = 0;
        bool ok = true;
        for (int tile = tile0; tile < p.ntiles && ok; tile += p.per_pair) {
            const long long row = (long long)tile * kTileRows + lane;
            const bool has_row = lane < kTileRows && row < p.N;
            for (int ch = 0; ch < nchunks; ++ch, ++g) {
                const int slot = (int)(g % S);
                if (g >= S) {
                    int okl = 1;
                    if (lane == 0) okl = mbar_wait(smem_u32(&bars[S + slot]), (uint32_t)(((g / S) - 1) & 1), flags, p.err);
                    ok = __shfl_sync(0xffffffffu, okl, 0) != 0;
                    if (!ok) break;
                }
                const int cu0 = su0 + ch * p.ups;
                const int cnu = min(p.ups, su0 + sunits - cu0);
                uint8_t* st = smem + p.off_stage + (long long)slot * kTileRows * p.row_stride;
                uint32_t bytes = 0;
                long long a = 0;
                if (has_row) {
                    const long long s0 = row * p.rb + (long long)cu0 * UB;
                    const long long e = s0 + (long long)cnu * UB;
                    a = s0 & ~15ll;
                    long long b = (e + 15) & ~15ll;
                    if (b > p.total_bytes) {
                        b = e & ~15ll;
                        for (long long q = b; q < e; ++q) st[lane * p.row_stride + (q - a)] = p.wq[q];
                        fence_proxy_async();
                    }
                    if (b > a) bytes = (uint32_t)(b - a);
                }
                const uint32_t tx = __reduce_add_sync(0xffffffffu, bytes);
                const uint32_t fb = smem_u32(&bars[slot]);
                if (lane == 0) mbar_arrive_tx(fb, tx);
                __syncwarp();
                if (bytes) bulk_g2s(smem_u32(st + lane * p.row_stride), p.wq + a, bytes, fb);
            }
        }
        // wait for the copies still in flight into this block's stages
        if (lane == 0) {
            const long long first = g > S ? g - S : 0;
            for (long long q = first; q < g; ++q) mbar_drain(smem_u32(&bars[q % S]), (uint32_t)((q / S) & 1), flags, p.err);
        }
        return;
    }

    // ------------------------------- consumers -------------------------------
    const int k0 = su0 * Unit<WT>::vals;
    const int klen = sunits * Unit<WT>::vals;
    prepare_acts<WT, AM, CW>(p, smem, m0, k0, klen, tid);
    consumer_sync<CW>();

    constexpr int MR = chunk_rows(AM, NT);
    constexpr int NRED = CW;  // partial sums per output in `red`
    float* red = reinterpret_cast<float*>(smem + p.off_red);
    const float* rs = reinterpret_cast<const float*>(smem + p.off_rs);
    const int g8 = lane >> 2, t4 = lane & 3;
    long long g = 0;
    for (int tile = tile0; tile < p.ntiles; tile += p.per_pair) {
        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[nt][i] = 0.0f;
        const long long rowA = (long long)tile * kTileRows + g8, rowB = rowA + 8;
        for (int ch = 0; ch < nchunks; ++ch, ++g) {
            const int slot = (int)(g % S);
            const bool ok = mbar_wait(smem_u32(&bars[slot]), (uint32_t)((g / S) & 1), flags, p.err);
            const int cu0 = su0 + ch * p.ups;
            const int cnu = min(p.ups, su0 + sunits - cu0);
            if (ok) {
                const uint8_t* st = smem + p.off_stage + (long long)slot * kTileRows * p.row_stride;
                const int off0 = (int)((rowA * p.rb + (long long)cu0 * UB) & 15);
                const int off1 = (int)((rowB * p.rb + (long long)cu0 * UB) & 15);
                stage_mma<WT, AM, NT, EPI, CW>(p, smem, st, cnu, cu0 - su0, cu0, off0, off1, warp, lane, acc, tile, m0);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars[S + slot]));
        }
        if (EPI != E_Y) continue;
        // ---- tile epilogue: red[NRED][16][MR], then sum, scale and store
        {
            float* rw = red + warp * kTileRows * MR;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                if (AM == A_INT8) {
                    rw[g8 * MR + nt * 8 + 2 * t4] = acc[nt][0];
                    rw[g8 * MR + nt * 8 + 2 * t4 + 1] = acc[nt][1];
                    rw[(g8 + 8) * MR + nt * 8 + 2 * t4] = acc[nt][2];
                    rw[(g8 + 8) * MR + nt * 8 + 2 * t4 + 1] = acc[nt][3];
                } else {
                    rw[g8 * MR + nt * 4 + t4] = acc[nt][0];
                    rw[(g8 + 8) * MR + nt * 4 + t4] = acc[nt][1];
                }
            }
        }
        consumer_sync<CW>();
        const bool aborted = flags[0] != 0;
        for (int o = tid; o < kTileRows * MR; o += CW * 32) {
            const int r = o / MR, c = o - r * MR;
            float v = 0.0f;
#pragma unroll
            for (int w = 0; w < NRED; ++w) v += red[(w * kTileRows + r) * MR + c];
            if (AM == A_F32) v *= rs[2 * c + 1];
            const long long n = (long long)tile * kTileRows + r;
            const int m = m0 + c;
            if (!aborted && n < p.N && m < p.M) {
                if (p.kslices == 1) p.y[(long long)m * p.N + n] = v;
                else p.partial[((long long)slice * p.M + m) * p.N + n] = v;
            }
        }
        if (p.kslices > 1) {
            __threadfence();
            consumer_sync<CW>();
            if (tid == 0) {
                const unsigned old = atomicAdd(&p.counters[(long long)mc * p.ntiles + tile], 1u);
                flags[1] = (old == (unsigned)(p.kslices - 1)) ? 1 : 0;
            }
            consumer_sync<CW>();
            if (flags[1] && !aborted) {
                __threadfence();
                for (int o = tid; o < kTileRows * MR; o += CW * 32) {
                    const int r = o / MR, c = o - r * MR;
                    const long long n = (long long)tile * kTileRows + r;
                    const int m = m0 + c;
                    if (n < p.N && m < p.M) {
                        float v = 0.0f;
                        for (int s = 0; s < p.kslices; ++s) v += __ldcg(p.partial + ((long long)s * p.M + m) * p.N + n);
                        p.y[(long long)m * p.N + n] = v;
                    }
                }
            }
        }
        consumer_sync<CW>();
    }
}

// ---------------------------------------------------------------------------
// host-side planning (path, shared-memory layout, grid, split of K)
// ---------------------------------------------------------------------------

struct StreamPlan {
    StreamParams p;
    int nt;
    int cw;
    int grid;
    size_t smem;
    size_t workspace;  // bytes of partial sums + counters (0 when K is not split)
};

// Fills the layout for wtype/mode/epilogue and sizes; returns false if no
// layout fits in smem_max.
inline bool plan_stream(int wt, int am, int epi, long long M, long long N, long long K, int sm_count, int smem_max,
                        StreamPlan& out) {
    StreamPlan pl{};
    StreamParams& p = pl.p;
    const int uv = unit_vals(wt), ub = unit_bytes(wt);
    int nt;
    if (am == A_INT8) nt = M <= 8 ? 1 : M <= 16 ? 2 : M <= 32 ? 4 : 8;
    else nt = M <= 4 ? 1 : M <= 8 ? 2 : M <= 16 ? 4 : 8;
    if (is_sb(wt) && am == A_INT8 && nt > 4) nt = 4;  // register budget of the integer super-block sums
    const int cw = consumer_warps(wt, am, nt);
    const int mr = chunk_rows(am, nt);
    p.M = (int)M;
    p.N = (int)N;
    p.K = (int)K;
    p.mr = mr;
    p.mchunks = (int)((M + mr - 1) / mr);
    p.units = (int)(K / uv);
    p.rb = (long long)p.units * ub;
    p.total_bytes = p.rb * N;
    p.ntiles = (int)((N + kTileRows - 1) / kTileRows);
    // Units per stage: a row's chunk is one bulk copy, and the copy engine pays a
    // fixed cost per segment, so chunks are as long as three stages allow.  An
    // unsplit K comes first (a K split adds partial sums and a reduction): the
    // first K split, in increasing order, with a candidate chunk that leaves
    // three stages wins; the largest such chunk is taken.
    const int cand_b32[4] = {128, 96, 64, 32}, cand_sb[3] = {16, 12, 8};
    const int* cand = is_sb(wt) ? cand_sb : cand_b32;
    const int ncand = is_sb(wt) ? 3 : 4;
    const int red_bytes = cw * kTileRows * mr * 4;
    for (int ks = 1; ks <= p.units && p.kslices == 0; ++ks) {
        const int su = (p.units + ks - 1) / ks;
        if ((long long)(ks - 1) * su >= p.units) continue;  // empty last slice
        int prev = 0;
        for (int ci = 0; ci < ncand && p.kslices == 0; ++ci) {
            const int ups = su < cand[ci] ? su : cand[ci];
            if (ups == prev) continue;
            prev = ups;
            // row pitch in a stage: room for the 16-byte superset; the remainder
            // mod 128 spreads the rows of one access over the banks
            const int want = 16;
            int row_stride = round_up(ups * ub + 32, 16);
            row_stride += ((want - row_stride % 128) + 128) % 128;
            const int stage_bytes = kTileRows * row_stride;
            const int kv = su * uv;  // values per slice
            int codes, scale_pitch = 0, aux_pitch = 0, code_pitch;
            if (am == A_INT8) {
                code_pitch = kv + 16;
                codes = mr * code_pitch;
                scale_pitch = su;
                if (wt == T_Q4_K) aux_pitch = su * 8;  // sums of each 32 activation codes (Q6_K needs none)
            } else {
                code_pitch = kv + 8;  // halves
                codes = mr * 2 * code_pitch * 2;
                if (wt == T_Q4_K) aux_pitch = kv / 32;
            }
            int off = round_up(2 * 8 * 8, 128);  // up to 8 stages x 2 barriers
            const int off_flags = off;
            off += 128;
            const int off_codes = off;
            off = round_up(off + codes, 128);
            const int off_scale = off;
            off = round_up(off + mr * scale_pitch * 4, 128);
            const int off_aux = off;
            off = round_up(off + mr * aux_pitch * 4, 128);
            const int off_rs = off;
            off = round_up(off + mr * 2 * 4, 128);
            const int off_red = off;
            off = round_up(off + red_bytes, 128);
            const int off_stage = off;
            int stages = (smem_max - off) / stage_bytes;
            if (stages > 8) stages = 8;
            if (stages < 3 && !(ks == p.units && ci == ncand - 1)) continue;  // a shorter chunk, else a split
            if (stages < 2) return false;
            p.kslices = ks;
            p.slice_units = su;
            p.ups = ups;
            p.row_stride = row_stride;
            p.stages = stages;
            p.code_pitch = code_pitch;
            p.scale_pitch = scale_pitch;
            p.aux_pitch = aux_pitch;
            p.off_flags = off_flags;
            p.off_codes = off_codes;
            p.off_scale = off_scale;
            p.off_aux = off_aux;
            p.off_rs = off_rs;
            p.off_red = off_red;
            p.off_stage = off_stage;
            pl.smem = (size_t)off_stage + (size_t)stages * stage_bytes;
        }
    }
    if (p.kslices == 0) return false;
    p.pairs = p.kslices * p.mchunks;
    int per = sm_count / p.pairs;
    if (per < 1) per = 1;
    if (per > p.ntiles) per = p.ntiles;
    p.per_pair = per;
    pl.grid = p.pairs * per;
    pl.nt = nt;
    pl.cw = cw;
    pl.workspace = (epi == E_Y && p.kslices > 1)
                       ? (size_t)p.kslices * (size_t)M * (size_t)N * 4 + (size_t)p.mchunks * p.ntiles * 4 + 256
                       : 0;
    out = pl;
    return true;
}

}  // namespace qmm
