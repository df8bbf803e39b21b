// qmm_dmma.cuh -- decode matmul (M <= 8 activation rows) on warp tensor cores
// with 16-row weight tiles.
//
// Serves both forms of "同一个 GGUF，CPU 和 Metal 生成的文字不一样" section 出处
// at decode batch sizes: the CPU form (activations quantized per row to Q8_0 /
// Q8K, exact integer block sums) and the Metal form (f32 activations times
// weights dequantized in-kernel).
//
// The MMA's A operand holds 16 weight rows, its B operand the activations:
//   int8_act: B column c = activation row c (M <= 8); mma.m16n8k32.s8 takes
//     the raw Q8_0 codes, or the Q4_K nibbles (0..15), as A with no conversion.
//     Q8_0: y += f(d_w) f(d_a) isum per block.  Q4_K: S_sc accumulates
//     sc_j * isum_j exactly in int32; S_m = sum_j m_j bsum_j comes from one
//     f16 MMA per super-block over the 16 sums of 16 activation codes (every
//     product and partial sum is an integer below 2^24, so it is exact).
//   f32_act: every activation row is scaled by a power of two and split into
//     two exact f16 pieces, x 2^s = hi + lo; B column 2r holds hi of row r and
//     column 2r+1 its lo (a second column set serves rows 4..7).  Weight codes
//     become exact f16: Q8_0 q; Q4_K sc_j * q (<= 945) with the 6-bit factor
//     folded into the conversion, so the 16 MMAs of a super-block chain in
//     one accumulator and are scaled once by f(d).  The min term
//     f(dmin) sum_j m_j X_j (X_j = sum of the sub-block's x) is one
//     mma.m16n8k8 per super-block with X_j / 32 in two f16 pieces.
// The MMA k order is a fixed permutation of each 32-value group: thread t4
// of a quad owns values 4t4..4t4+3 and 16+4t4..16+4t4+3 of the group, read
// as two 4-byte words; the f32 activation planes are stored in the matching
// order.  Weight tiles stream through a shared-memory ring as one bulk copy
// per row and K chunk (~4.3 KB), into rows at a pitch of 16 mod 128 bytes so
// that the word loads of 8 rows x 4 threads hit 32 distinct banks.  K is
// split across CTAs only when the activation rows of the whole K range do not
// fit in shared memory; the slices' partial sums then go to the workspace and
// a second small kernel adds them in slice order.
#pragma once

#include "qmm_device.cuh"
#include "qmm_stream.cuh"

namespace qmm {

constexpr int kDmmaWarps = 16;
constexpr int kDmmaRows = 16;  // weight rows per tile

struct DmmaParams {
    const uint8_t* wq;
    const float* x;
    float* y;
    int32_t* sums;
    float* partial;   // [kslices][M][N] when K is split (summed by splitk_reduce_kernel)
    unsigned* err;
    long long total_bytes;
    long long rb;
    int M, N, K;
    int units;        // weight units per row (32-blocks or super-blocks)
    int kslices, slice_units, per_slice;
    int ups;          // units per stage (K chunk of a tile)
    int ntiles;       // ceil(N / 16)
    int stages;
    int stage_bytes;
    int row_pitch;    // bytes between rows in a stage with one copy per row (0: one contiguous copy)
    int off_flags, off_act, off_scale, off_aux, off_rs, off_red, off_stage;
    int act_pitch;    // int8: bytes per activation row; f32: halves per (row, piece) plane
};

// position p (0..31) of a 32-value group in the MMA k order -> value index
__host__ __device__ constexpr int dmma_kperm(int p) {
    return 4 * (p >> 3) + ((p & 4) ? 16 : 0) + ((p & 3) == 1 ? 2 : (p & 3) == 2 ? 1 : (p & 3));
}

// ---------------------------------------------------------------------------
// activation preparation (consumer warps, once per CTA)
// ---------------------------------------------------------------------------
template <int WT, int AM>
__device__ __forceinline__ void dmma_prepare(const DmmaParams& p, uint8_t* smem, int k0, int klen, int tid) {
    constexpr int NTH = kDmmaWarps * 32;
    const int su = p.slice_units;
    if (AM == A_INT8 && WT == T_Q8_0) {
        uint8_t* codes = smem + p.off_act;
        float* da = reinterpret_cast<float*>(smem + p.off_scale);  // [unit][8 rows]
        for (int idx = tid; idx < p.M * su; idx += NTH) {
            const int r = idx / su, b = idx - r * su;
            uint32_t c[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            float s = 0.0f;
            if (b * 32 < klen) {
                float d;
                quant_q8_0_32(p.x + (long long)r * p.K + k0 + b * 32, c, d);
                s = h2f(f2h(d));
            }
            uint4* d0 = reinterpret_cast<uint4*>(codes + r * p.act_pitch + b * 32);
            d0[0] = make_uint4(c[0], c[1], c[2], c[3]);
            d0[1] = make_uint4(c[4], c[5], c[6], c[7]);
            da[b * 8 + r] = s;
        }
    } else if (AM == A_INT8 && WT == T_Q4_K) {
        uint8_t* codes = smem + p.off_act;
        float* da = reinterpret_cast<float*>(smem + p.off_scale);       // [super-block][8 rows]
        uint32_t* bs = reinterpret_cast<uint32_t*>(smem + p.off_aux);   // [super-block][pair][8 rows] f16x2
        for (int idx = tid; idx < p.M * su; idx += NTH) {
            const int r = idx / su, sb = idx - r * su;
            const bool live = sb * 256 < klen;
            const float* src = p.x + (long long)r * p.K + k0 + sb * 256;
            float d = 0.0f, id = 0.0f;
            if (live) q8_scale(q8k_amax(src), d, id);
            for (int q = 0; q < 8; ++q) {  // 32 values: two sums of 16
                uint32_t w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                int s0 = 0, s1 = 0;
                if (live) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float4 v = __ldg(reinterpret_cast<const float4*>(src + 32 * q) + i);
                        w[i] = pack4(q8_code(v.x, id), q8_code(v.y, id), q8_code(v.z, id), q8_code(v.w, id));
                        if (i < 4) s0 += bsum4(w[i]);
                        else s1 += bsum4(w[i]);
                    }
                }
                uint4* d0 = reinterpret_cast<uint4*>(codes + r * p.act_pitch + sb * 256 + 32 * q);
                d0[0] = make_uint4(w[0], w[1], w[2], w[3]);
                d0[1] = make_uint4(w[4], w[5], w[6], w[7]);
                // |sum of 16 codes| <= 2032: exact in f16
                bs[(sb * 8 + q) * 8 + r] = f2h((float)s0) | (f2h((float)s1) << 16);
            }
            da[sb * 8 + r] = d;
        }
    } else {
        // f32_act: per-row power-of-two scale; planes 2r (hi) and 2r+1 (lo) in MMA k order
        __half* pl = reinterpret_cast<__half*>(smem + p.off_act);
        float* rs = reinterpret_cast<float*>(smem + p.off_rs);               // [8][2]: 2^s, 2^-s
        uint16_t* xs = reinterpret_cast<uint16_t*>(smem + p.off_aux);        // Q4_K: [sb][16 planes][8 sub-blocks]
        const int warp = tid >> 5, lane = tid & 31;
        if (warp < p.M) {
            const int r = warp;
            float amax = 0.0f;
            const float4* src = reinterpret_cast<const float4*>(p.x + (long long)r * p.K + k0);
            for (int i = lane; i < klen / 4; i += 32) {
                const float4 v = __ldg(src + i);
                amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            if (lane == 0) {
                int s = 0;
                if (amax > 0.0f) {
                    const int e = (int)((__float_as_uint(amax) >> 23) & 0xff) - 127;
                    s = 14 - e;
                    s = s > 100 ? 100 : (s < -100 ? -100 : s);
                }
                rs[2 * r] = ldexpf(1.0f, s);
                rs[2 * r + 1] = ldexpf(1.0f, -s);
            }
        }
        consumer_sync<kDmmaWarps>();
        const int nch = su * Unit<WT>::vals / 32;
        for (int idx = tid; idx < p.M * nch; idx += NTH) {
            const int r = idx / nch, c = idx - r * nch;
            float v[32];
            float sum = 0.0f;
            if (c * 32 < klen) {
                const float scale = rs[2 * r];
                const float4* src = reinterpret_cast<const float4*>(p.x + (long long)r * p.K + k0 + c * 32);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 v4 = __ldg(src + i);
                    v[4 * i] = __fmul_rn(v4.x, scale);
                    v[4 * i + 1] = __fmul_rn(v4.y, scale);
                    v[4 * i + 2] = __fmul_rn(v4.z, scale);
                    v[4 * i + 3] = __fmul_rn(v4.w, scale);
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) sum = __fadd_rn(sum, v[i]);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = 0.0f;
            }
            uint32_t hw[16], lw[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                uint32_t hb[2], lb[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float f = v[dmma_kperm(2 * q + e)];
                    const __half h = __float2half_rn(f);
                    hb[e] = __half_as_ushort(h);
                    lb[e] = __half_as_ushort(__float2half_rn(__fsub_rn(f, __half2float(h))));
                }
                hw[q] = hb[0] | (hb[1] << 16);
                lw[q] = lb[0] | (lb[1] << 16);
            }
            uint4* dh = reinterpret_cast<uint4*>(pl + (long long)(2 * r) * p.act_pitch + c * 32);
            uint4* dl = reinterpret_cast<uint4*>(pl + (long long)(2 * r + 1) * p.act_pitch + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                dh[i] = make_uint4(hw[4 * i], hw[4 * i + 1], hw[4 * i + 2], hw[4 * i + 3]);
                dl[i] = make_uint4(lw[4 * i], lw[4 * i + 1], lw[4 * i + 2], lw[4 * i + 3]);
            }
            if (WT == T_Q4_K) {
                // X_j / 32 (|.| < 2^15) in two f16 pieces
                const float xq = __fmul_rn(sum, 0.03125f);
                const __half h = __float2half_rn(xq);
                const __half l = __float2half_rn(__fsub_rn(xq, __half2float(h)));
                const int sb = c >> 3, j = c & 7;
                xs[(sb * 16 + 2 * r) * 8 + j] = __half_as_ushort(h);
                xs[(sb * 16 + 2 * r + 1) * 8 + j] = __half_as_ushort(l);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// weight-side helpers
// ---------------------------------------------------------------------------

// The thread's code words of a Q8_0 block at `blk` (2-byte aligned in shared
// memory): bytes 4t..4t+3 (lo) and 16+4t..16+4t+3 (hi) of the 32 codes, and
// the same one byte further on (lo1, hi1).
__device__ __forceinline__ void q8_0_words(const uint8_t* blk, int t, uint32_t& lo, uint32_t& hi, uint32_t& lo1,
                                           uint32_t& hi1) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(blk + 2);
    const uint32_t* w = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
    const uint32_t sh = (uint32_t)(a & 3u) * 8u;
    const uint32_t w0 = w[t], w1 = w[t + 1], w4 = w[t + 4], w5 = w[t + 5];
    lo = __funnelshift_r(w0, w1, sh);
    hi = __funnelshift_r(w4, w5, sh);
    lo1 = __funnelshift_r(w0, w1, sh + 8);
    hi1 = __funnelshift_r(w4, w5, sh + 8);
}

__device__ __forceinline__ uint32_t h2_sub(uint32_t a, uint32_t b) {
    __half2 r = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
    return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t h2_mul(uint32_t a, uint32_t b) {
    __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
    return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t h2_fma(uint32_t a, uint32_t b, uint32_t c) {
    __half2 r = __hfma2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b), *reinterpret_cast<__half2*>(&c));
    return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t h2_lo2(uint32_t a) { return __byte_perm(a, 0, 0x1010); }
__device__ __forceinline__ uint32_t h2_hi2(uint32_t a) { return __byte_perm(a, 0, 0x3232); }

// signed bytes 0 and 2 of w -> exact f16x2: 0x64 | (b ^ 0x80) is 1152 + b
__device__ __forceinline__ uint32_t s8_02_h2(uint32_t w) { return h2_sub((w & 0x00FF00FFu) ^ 0x64806480u, 0x64806480u); }

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <int WT, int AM, int NB, int EPI>
__global__ void __launch_bounds__((kDmmaWarps + 1) * 32, 1) qmm_dmma_kernel(const DmmaParams p) {
    constexpr int UB = Unit<WT>::bytes;
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = p.stages;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
    volatile int* flags = reinterpret_cast<volatile int*>(smem + p.off_flags);
    const int slice = blockIdx.x % p.kslices;
    const int grp0 = blockIdx.x / p.kslices;
    const int su0 = slice * p.slice_units;
    const int sunits = min(p.slice_units, p.units - su0);
    const bool whole = p.row_pitch == 0;  // short rows: one contiguous copy of the 16 rows per stage
    const int nch = (sunits + p.ups - 1) / p.ups;
    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(smem_u32(&bars[i]), 1);
            mbar_init(smem_u32(&bars[S + i]), kDmmaWarps);
        }
        flags[0] = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kDmmaWarps) {
        // ------------------------------ producer ------------------------------
        long long g = 0;
        bool ok = true;
        for (int grp = grp0; grp < p.ntiles && ok; grp += p.per_slice) {
            for (int ch = 0; ch < nch && ok; ++ch, ++g) {
                const int slot = (int)(g % S);
                if (g >= S) {
                    int okl = 1;
                    if (lane == 0) okl = mbar_wait(smem_u32(&bars[S + slot]), (uint32_t)(((g / S) - 1) & 1), flags, p.err);
                    ok = __shfl_sync(0xffffffffu, okl, 0) != 0;
                    if (!ok) break;
                }
                const int cu0 = su0 + ch * p.ups;
                const int cnu = min(p.ups, su0 + sunits - cu0);
                uint8_t* st = smem + p.off_stage + (long long)slot * p.stage_bytes;
                long long a = 0, b = 0;
                int dst = 0;
                const long long row = (long long)grp * kDmmaRows + lane;
                if (whole ? lane == 0 : (lane < kDmmaRows && row < p.N)) {
                    const long long r0 = (long long)grp * kDmmaRows;
                    const long long s0 = whole ? r0 * p.rb : row * p.rb + (long long)cu0 * UB;
                    const long long e = whole ? min(r0 + kDmmaRows, (long long)p.N) * p.rb : s0 + (long long)cnu * UB;
                    a = s0 & ~15ll;
                    b = (e + 15) & ~15ll;
                    dst = whole ? 0 : lane * p.row_pitch;
                    if (b > p.total_bytes) {
                        b = e & ~15ll;
                        for (long long q = b; q < e; ++q) st[dst + (q - a)] = p.wq[q];
                        fence_proxy_async();
                    }
                }
                const uint32_t bytes = b > a ? (uint32_t)(b - a) : 0u;
                const uint32_t tx = __reduce_add_sync(0xffffffffu, bytes);
                const uint32_t fb = smem_u32(&bars[slot]);
                if (lane == 0) mbar_arrive_tx(fb, tx);
                __syncwarp();
                if (bytes) bulk_g2s(smem_u32(st + dst), p.wq + a, bytes, fb);
            }
        }
        if (lane == 0) {
            const long long first = g > S ? g - S : 0;
            for (long long q = first; q < g; ++q) mbar_wait(smem_u32(&bars[q % S]), (uint32_t)((q / S) & 1), flags, p.err);
        }
        return;
    }

    // ------------------------------ consumers ------------------------------
    const int k0 = su0 * Unit<WT>::vals;
    const int klen = sunits * Unit<WT>::vals;
    dmma_prepare<WT, AM>(p, smem, k0, klen, tid);
    consumer_sync<kDmmaWarps>();

    const int g8 = lane >> 2, t4 = lane & 3;
    const uint8_t* act = smem + p.off_act;
    const float* da = reinterpret_cast<const float*>(smem + p.off_scale);
    const uint32_t* aux = reinterpret_cast<const uint32_t*>(smem + p.off_aux);
    const float* rs = reinterpret_cast<const float*>(smem + p.off_rs);
    float* red = reinterpret_cast<float*>(smem + p.off_red);  // [16 warps][16 weight rows][8 activation rows]
    // B-operand column of this thread: activation row (int8) or (row, piece) plane (f32), per column set
    bool bval[NB];
    const uint8_t* bcol[NB];
#pragma unroll
    for (int s = 0; s < NB; ++s) {
        if (AM == A_INT8) {
            bval[s] = g8 < p.M;
            bcol[s] = act + (bval[s] ? g8 : 0) * p.act_pitch;
        } else {
            const int pl = 8 * s + g8;
            bval[s] = (pl >> 1) < p.M;
            bcol[s] = act + (long long)(bval[s] ? pl : 0) * p.act_pitch * 2;
        }
    }
    // Q4_K min-term A fragments: bytes of the packed 6-bit mins as f16 pairs
    const uint32_t sel_m2 = (uint32_t)((2 * (t4 & 1)) | 0x40 | ((2 * (t4 & 1) + 1) << 8) | 0x4000);  // m_{2t}, m_{2t+1}
    const uint32_t sel_m1 = (uint32_t)(t4 | 0x40 | (t4 << 8) | 0x4000);                                   // m_t, m_t
    long long g = 0;
    for (int grp = grp0; grp < p.ntiles; grp += p.per_slice) {
        float acc[NB][2][2];
#pragma unroll
        for (int s = 0; s < NB; ++s) acc[s][0][0] = acc[s][0][1] = acc[s][1][0] = acc[s][1][1] = 0.0f;
        for (int ch = 0; ch < nch; ++ch, ++g) {
            const int slot = (int)(g % S);
            const bool ok = mbar_wait(smem_u32(&bars[slot]), (uint32_t)((g / S) & 1), flags, p.err);
            const int cu0 = su0 + ch * p.ups;
            const int cnu = min(p.ups, su0 + sunits - cu0);
            if (ok) {
                const uint8_t* st = smem + p.off_stage + (long long)slot * p.stage_bytes;
                auto rowptr = [&](int r) -> const uint8_t* {
                    const long long n = (long long)grp * kDmmaRows + r;
                    if (whole) return st + (int)(((long long)grp * kDmmaRows * p.rb) & 15) + (long long)r * p.rb;
                    return st + r * p.row_pitch + (int)((n * p.rb + (long long)cu0 * UB) & 15);
                };
                const uint8_t* r0p = rowptr(g8);
                const uint8_t* r1p = rowptr(g8 + 8);
                const int ur0 = cu0 - su0;  // first unit of the chunk inside the slice
#pragma unroll 1
                for (int uu = warp; uu < cnu; uu += kDmmaWarps) {
                    const int u = ur0 + uu;  // unit index inside the slice (activation side)
                    if (WT == T_Q8_0) {
                        const uint8_t* b0p = r0p + 34 * uu;
                        const uint8_t* b1p = r1p + 34 * uu;
                        const float dw0 = h2f(*reinterpret_cast<const uint16_t*>(b0p));
                        const float dw1 = h2f(*reinterpret_cast<const uint16_t*>(b1p));
                        uint32_t lo0, hi0, lo0s, hi0s, lo1, hi1, lo1s, hi1s;
                        q8_0_words(b0p, t4, lo0, hi0, lo0s, hi0s);
                        q8_0_words(b1p, t4, lo1, hi1, lo1s, hi1s);
                        if (AM == A_F32) {
                            const uint32_t a0 = s8_02_h2(lo0), a1 = s8_02_h2(lo1), a2 = s8_02_h2(lo0s), a3 = s8_02_h2(lo1s);
                            const uint32_t c0 = s8_02_h2(hi0), c1 = s8_02_h2(hi1), c2 = s8_02_h2(hi0s), c3 = s8_02_h2(hi1s);
#pragma unroll
                            for (int s = 0; s < NB; ++s) {
                                uint4 xv = make_uint4(0u, 0u, 0u, 0u);
                                if (bval[s]) xv = ld128(bcol[s] + (u * 32 + 8 * t4) * 2);
                                float d[4] = {0.f, 0.f, 0.f, 0.f};
                                mma_f16(d, a0, a1, a2, a3, xv.x, xv.y);
                                mma_f16(d, c0, c1, c2, c3, xv.z, xv.w);
                                acc[s][0][0] = fmaf(dw0, d[0] + d[1], acc[s][0][0]);
                                acc[s][1][0] = fmaf(dw1, d[2] + d[3], acc[s][1][0]);
                            }
                        } else {
                            uint32_t b0 = 0u, b1 = 0u;
                            if (bval[0]) {
                                b0 = ld32(bcol[0] + u * 32 + 4 * t4);
                                b1 = ld32(bcol[0] + u * 32 + 16 + 4 * t4);
                            }
                            int d[4];
                            mma_s8(d, lo0, lo1, hi0, hi1, b0, b1);
                            if (EPI == E_Y) {
                                const float2 dap = *reinterpret_cast<const float2*>(da + u * 8 + 2 * t4);
                                acc[0][0][0] = fmaf((float)d[0], dw0 * dap.x, acc[0][0][0]);
                                acc[0][0][1] = fmaf((float)d[1], dw0 * dap.y, acc[0][0][1]);
                                acc[0][1][0] = fmaf((float)d[2], dw1 * dap.x, acc[0][1][0]);
                                acc[0][1][1] = fmaf((float)d[3], dw1 * dap.y, acc[0][1][1]);
                            } else {
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const int m = 2 * t4 + (i & 1);
                                    const long long n = (long long)grp * kDmmaRows + g8 + 8 * (i >> 1);
                                    if (m < p.M && n < p.N) p.sums[((long long)m * p.N + n) * p.units + su0 + u] = d[i];
                                }
                            }
                        }
                    } else {
                        const uint8_t* s0p = r0p + 144 * uu;
                        const uint8_t* s1p = r1p + 144 * uu;
                        const uint4 h0 = ld128(s0p), h1 = ld128(s1p);
                        uint32_t sc03[2], sc47[2], mn03[2], mn47[2];
                        q4k_unpack4(h0.y, h0.z, h0.w, sc03[0], sc47[0], mn03[0], mn47[0]);
                        q4k_unpack4(h1.y, h1.z, h1.w, sc03[1], sc47[1], mn03[1], mn47[1]);
                        if (AM == A_F32) {
                            float d[NB][4];
#pragma unroll
                            for (int s = 0; s < NB; ++s) d[s][0] = d[s][1] = d[s][2] = d[s][3] = 0.0f;
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                // per row: (sc_{2c}, sc_{2c+1}/16) and (-1024 sc_{2c}, -64 sc_{2c+1})
                                const uint32_t sel = (uint32_t)((2 * (c & 1)) | 0x40 | ((2 * (c & 1) + 1) << 8) | 0x5000);
                                uint32_t P[2], Q[2];
#pragma unroll
                                for (int r = 0; r < 2; ++r) {
                                    P[r] = h2_sub(__byte_perm(c < 2 ? sc03[r] : sc47[r], 0x00005464u, sel), 0x54006400u);
                                    Q[r] = h2_mul(P[r], 0xE400E400u);
                                }
                                const uint32_t qa0 = ld32(s0p + 16 + 32 * c + 4 * t4), qb0 = ld32(s0p + 32 + 32 * c + 4 * t4);
                                const uint32_t qa1 = ld32(s1p + 16 + 32 * c + 4 * t4), qb1 = ld32(s1p + 32 + 32 * c + 4 * t4);
                                const uint32_t qa0s = qa0 >> 8, qb0s = qb0 >> 8, qa1s = qa1 >> 8, qb1s = qb1 >> 8;
#pragma unroll
                                for (int h = 0; h < 2; ++h) {
                                    // low nibbles (sub-block 2c): 1024 + n; high nibbles (2c+1): 1024 + 16 n
                                    const uint32_t mk = h ? 0x00F000F0u : 0x000F000Fu;
                                    const uint32_t S0 = h ? h2_hi2(P[0]) : h2_lo2(P[0]), N0 = h ? h2_hi2(Q[0]) : h2_lo2(Q[0]);
                                    const uint32_t S1 = h ? h2_hi2(P[1]) : h2_lo2(P[1]), N1 = h ? h2_hi2(Q[1]) : h2_lo2(Q[1]);
                                    const uint32_t a0 = h2_fma((qa0 & mk) | 0x64006400u, S0, N0);
                                    const uint32_t a1 = h2_fma((qa1 & mk) | 0x64006400u, S1, N1);
                                    const uint32_t a2 = h2_fma((qa0s & mk) | 0x64006400u, S0, N0);
                                    const uint32_t a3 = h2_fma((qa1s & mk) | 0x64006400u, S1, N1);
                                    const uint32_t c0 = h2_fma((qb0 & mk) | 0x64006400u, S0, N0);
                                    const uint32_t c1 = h2_fma((qb1 & mk) | 0x64006400u, S1, N1);
                                    const uint32_t c2 = h2_fma((qb0s & mk) | 0x64006400u, S0, N0);
                                    const uint32_t c3 = h2_fma((qb1s & mk) | 0x64006400u, S1, N1);
                                    const int j = 2 * c + h;
#pragma unroll
                                    for (int s = 0; s < NB; ++s) {
                                        uint4 xv = make_uint4(0u, 0u, 0u, 0u);
                                        if (bval[s]) xv = ld128(bcol[s] + ((u * 8 + j) * 32 + 8 * t4) * 2);
                                        mma_f16(d[s], a0, a1, a2, a3, xv.x, xv.y);
                                        mma_f16(d[s], c0, c1, c2, c3, xv.z, xv.w);
                                    }
                                }
                            }
                            // min term: sum_j m_j X_j / 32 for rows g8, g8+8
                            const uint32_t ma0 = h2_sub(__byte_perm(t4 < 2 ? mn03[0] : mn47[0], 0x64646464u, sel_m2), 0x64006400u);
                            const uint32_t ma1 = h2_sub(__byte_perm(t4 < 2 ? mn03[1] : mn47[1], 0x64646464u, sel_m2), 0x64006400u);
                            const float fD0 = h2f(h0.x), fD1 = h2f(h1.x);
                            const float fM0 = 32.0f * h2f(h0.x >> 16), fM1 = 32.0f * h2f(h1.x >> 16);
#pragma unroll
                            for (int s = 0; s < NB; ++s) {
                                uint32_t xb = 0u;
                                if (bval[s]) xb = aux[(u * 16 + 8 * s + g8) * 4 + t4];
                                float dm[4] = {0.f, 0.f, 0.f, 0.f};
                                mma_f16_k8(dm, ma0, ma1, xb);
                                acc[s][0][0] += fD0 * (d[s][0] + d[s][1]) - fM0 * (dm[0] + dm[1]);
                                acc[s][1][0] += fD1 * (d[s][2] + d[s][3]) - fM1 * (dm[2] + dm[3]);
                            }
                        } else {
                            int ssc[4] = {0, 0, 0, 0};
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                const uint32_t qa0 = ld32(s0p + 16 + 32 * c + 4 * t4), qb0 = ld32(s0p + 32 + 32 * c + 4 * t4);
                                const uint32_t qa1 = ld32(s1p + 16 + 32 * c + 4 * t4), qb1 = ld32(s1p + 32 + 32 * c + 4 * t4);
#pragma unroll
                                for (int h = 0; h < 2; ++h) {
                                    const int j = 2 * c + h;
                                    const uint32_t sh = 4u * h;
                                    uint32_t b0 = 0u, b1 = 0u;
                                    if (bval[0]) {
                                        b0 = ld32(bcol[0] + u * 256 + 32 * j + 4 * t4);
                                        b1 = ld32(bcol[0] + u * 256 + 32 * j + 16 + 4 * t4);
                                    }
                                    int dj[4];
                                    mma_s8(dj, (qa0 >> sh) & 0x0F0F0F0Fu, (qa1 >> sh) & 0x0F0F0F0Fu, (qb0 >> sh) & 0x0F0F0F0Fu,
                                           (qb1 >> sh) & 0x0F0F0F0Fu, b0, b1);
                                    const uint32_t selj = 0x4440u | (uint32_t)(j & 3);
                                    const int sc0 = (int)__byte_perm(j < 4 ? sc03[0] : sc47[0], 0, selj);
                                    const int sc1 = (int)__byte_perm(j < 4 ? sc03[1] : sc47[1], 0, selj);
                                    ssc[0] += sc0 * dj[0];
                                    ssc[1] += sc0 * dj[1];
                                    ssc[2] += sc1 * dj[2];
                                    ssc[3] += sc1 * dj[3];
                                }
                            }
                            // S_m = sum_j m_j (sum of the sub-block's 32 codes), as 16 slots of sums of 16
                            const uint32_t ma0 = h2_sub(__byte_perm(mn03[0], 0x64646464u, sel_m1), 0x64006400u);
                            const uint32_t ma1 = h2_sub(__byte_perm(mn03[1], 0x64646464u, sel_m1), 0x64006400u);
                            const uint32_t ma2 = h2_sub(__byte_perm(mn47[0], 0x64646464u, sel_m1), 0x64006400u);
                            const uint32_t ma3 = h2_sub(__byte_perm(mn47[1], 0x64646464u, sel_m1), 0x64006400u);
                            uint32_t xb0 = 0u, xb1 = 0u;
                            if (bval[0]) {
                                xb0 = aux[(u * 8 + t4) * 8 + g8];
                                xb1 = aux[(u * 8 + t4 + 4) * 8 + g8];
                            }
                            float sm[4] = {0.f, 0.f, 0.f, 0.f};
                            mma_f16(sm, ma0, ma1, ma2, ma3, xb0, xb1);
                            if (EPI == E_Y) {
                                const float2 dap = *reinterpret_cast<const float2*>(da + u * 8 + 2 * t4);
                                const float fD0 = h2f(h0.x), fD1 = h2f(h1.x), fM0 = h2f(h0.x >> 16), fM1 = h2f(h1.x >> 16);
                                acc[0][0][0] = fmaf(dap.x, fD0 * (float)ssc[0] - fM0 * sm[0], acc[0][0][0]);
                                acc[0][0][1] = fmaf(dap.y, fD0 * (float)ssc[1] - fM0 * sm[1], acc[0][0][1]);
                                acc[0][1][0] = fmaf(dap.x, fD1 * (float)ssc[2] - fM1 * sm[2], acc[0][1][0]);
                                acc[0][1][1] = fmaf(dap.y, fD1 * (float)ssc[3] - fM1 * sm[3], acc[0][1][1]);
                            } else {
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const int m = 2 * t4 + (i & 1);
                                    const long long n = (long long)grp * kDmmaRows + g8 + 8 * (i >> 1);
                                    if (m < p.M && n < p.N) {
                                        int* o = p.sums + (((long long)m * p.N + n) * p.units + su0 + u) * 2;
                                        o[0] = ssc[i];
                                        o[1] = (int)sm[i];
                                    }
                                }
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars[S + slot]));
        }
        if (EPI != E_Y) continue;
        // ---- tile epilogue: 16 warp partials of (weight row, activation row)
        if (AM == A_F32) {
#pragma unroll
            for (int s = 0; s < NB; ++s) {
                red[warp * 128 + g8 * 8 + t4 + 4 * s] = acc[s][0][0];
                red[warp * 128 + (g8 + 8) * 8 + t4 + 4 * s] = acc[s][1][0];
            }
        } else {
            *reinterpret_cast<float2*>(red + warp * 128 + g8 * 8 + 2 * t4) = make_float2(acc[0][0][0], acc[0][0][1]);
            *reinterpret_cast<float2*>(red + warp * 128 + (g8 + 8) * 8 + 2 * t4) = make_float2(acc[0][1][0], acc[0][1][1]);
        }
        consumer_sync<kDmmaWarps>();
        if (tid < 128) {
            const int m = tid & 7;
            const long long n = (long long)grp * kDmmaRows + (tid >> 3);
            float v = 0.0f;
#pragma unroll
            for (int w = 0; w < kDmmaWarps; ++w) v += red[w * 128 + tid];
            if (AM == A_F32) v *= rs[2 * m + 1];
            if (!flags[0] && m < p.M && n < p.N) {
                if (p.kslices == 1) p.y[(long long)m * p.N + n] = v;
                else p.partial[((long long)slice * p.M + m) * p.N + n] = v;
            }
        }
        consumer_sync<kDmmaWarps>();
    }
}

// ---------------------------------------------------------------------------
// host-side planning
// ---------------------------------------------------------------------------

struct DmmaPlan {
    DmmaParams p;
    int nb;   // B column sets (2 for f32_act with M > 4)
    int grid;
    size_t smem;
    size_t workspace;
};

// Shared-memory layout for K split in `ks` slices and `ups` units per stage;
// false when fewer than two stages fit.
inline bool dmma_layout(int wt, int am, long long M, int ks, int ups, int smem_max, DmmaPlan& pl) {
    DmmaParams& p = pl.p;
    const int uv = wt == T_Q8_0 ? 32 : 256, ub = wt == T_Q8_0 ? 34 : 144;
    const int su = (p.units + ks - 1) / ks;
    if ((long long)(ks - 1) * su >= p.units) return false;
    if (ups > su) ups = su;
    const int kv = su * uv;
    int act, scale = 0, aux = 0;
    if (am == A_INT8) {
        p.act_pitch = pitch_mod(kv, 16);  // 4-byte B loads of 8 rows x 4 threads: 32 banks
        act = (int)M * p.act_pitch;
        scale = su * 8 * 4;
        if (wt == T_Q4_K) aux = su * 8 * 8 * 4;
    } else {
        p.act_pitch = pitch_mod(2 * kv, 64) / 2;  // 16-byte B loads of 2 planes per quarter-warp
        act = 2 * (int)M * p.act_pitch * 2;
        if (wt == T_Q4_K) aux = su * 16 * 8 * 2;
    }
    int off = 256;
    p.off_flags = off;
    off += 128;
    p.off_act = off;
    off = round_up(off + act, 128);
    p.off_scale = off;
    off = round_up(off + scale, 128);
    p.off_aux = off;
    off = round_up(off + aux, 128);
    p.off_rs = off;
    off = round_up(off + 64, 128);
    p.off_red = off;
    off = round_up(off + kDmmaWarps * 128 * 4, 128);
    p.off_stage = off;
    long long sb;
    if (ks == 1 && ups == su && 16 * p.rb <= 36864) {
        sb = 16 * p.rb + 64;  // short rows: one contiguous copy of the whole tile
        p.row_pitch = 0;
    } else {
        p.row_pitch = pitch_mod(ups * ub + 48, 16);
        sb = 16LL * p.row_pitch;
    }
    sb = (sb + 127) / 128 * 128;
    const long long stages = (smem_max - off) / sb;
    if (stages < 2) return false;
    p.kslices = ks;
    p.slice_units = su;
    p.ups = ups;
    p.stages = stages > 8 ? 8 : (int)stages;
    p.stage_bytes = (int)sb;
    pl.smem = (size_t)off + (size_t)p.stages * sb;
    return true;
}

inline bool plan_dmma(int wt, int am, long long M, long long N, long long K, int sm_count, int smem_max,
                      DmmaPlan& out) {
    if (M < 1 || M > 8) return false;
    DmmaPlan pl{};
    DmmaParams& p = pl.p;
    const int uv = wt == T_Q8_0 ? 32 : 256, ub = wt == T_Q8_0 ? 34 : 144;
    p.M = (int)M;
    p.N = (int)N;
    p.K = (int)K;
    p.units = (int)(K / uv);
    p.rb = (long long)p.units * ub;
    p.total_bytes = p.rb * N;
    p.ntiles = (int)((N + kDmmaRows - 1) / kDmmaRows);
    pl.nb = (am == A_F32 && M > 4) ? 2 : 1;
    // K chunk per stage: ~3.3-4.6 KB per row copy (one SM's bulk-copy rate
    // caps smaller copies); smaller chunks only when nothing else fits
    const int big[3] = {wt == T_Q8_0 ? 128 : 32, wt == T_Q8_0 ? 112 : 28, wt == T_Q8_0 ? 96 : 24};
    bool found = false;
    for (int ks = 1; ks <= 16 && !found; ++ks)
        for (int i = 0; i < 3 && !found; ++i) found = dmma_layout(wt, am, M, ks, big[i], smem_max, pl);
    for (int ks = 1; ks <= 16 && !found; ++ks) found = dmma_layout(wt, am, M, ks, wt == T_Q8_0 ? 32 : 8, smem_max, pl);
    if (!found) return false;
    int per = sm_count / p.kslices;
    if (per < 1) per = 1;
    if (per > p.ntiles) per = p.ntiles;
    p.per_slice = per;
    pl.grid = per * p.kslices;
    pl.workspace = p.kslices > 1 ? (size_t)p.kslices * M * N * 4 : 0;
    out = pl;
    return true;
}

}  // namespace qmm
