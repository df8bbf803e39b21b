// qmm_dmma.cuh -- decode matmul on warp tensor cores with 8-row weight tiles.
//
// Serves the f32_act form (the Metal form of "同一个 GGUF，CPU 和 Metal 生成的文字
// 不一样" section 出处: f32 activations times weights dequantized in-kernel) and
// the int8_act form for 5..8 activation rows, both for M <= 8.
//
// Operands are swapped with respect to a plain GEMM: the MMA's A operand (16
// rows) holds the activations -- for f32_act the 8 activation rows split in
// two exact f16 pieces (x 2^s = hi + lo), for int8_act the 8 rows of codes --
// and the B operand (8 columns) holds 8 weight rows.  A weight tile is
// therefore only 8 rows: a tile is 8 rows x the CTA's K range, streamed in
// stages of 8 row chunks of >= 4 KB each (one bulk copy per row; one copy for
// the whole tile when rows are short).  16 consumer warps split the K range
// of a stage block by block; per block:
//   Q8_0: two mma.m16n8k16.f16 (f32_act) or one mma.m16n8k32.s8 (int8_act),
//         then y += f(d_w) * sum (and f(d_a) for int8_act) in registers;
//   Q4_K: per 32-value sub-block the same, with e_j = f(d) sc_j and
//         o_j = f(dmin) m_j: y += e_j sum(q x) - o_j sum(x) (f32_act), or the
//         exact integer S_sc, S_m of the CPU form (int8_act).
// Warp partials of a tile are summed in shared memory (one named barrier per
// tile).  K is split across CTAs only when the activation rows of the whole K
// range do not fit in shared memory; the slices' partial sums then go to the
// workspace and a second small kernel adds them in slice order.
#pragma once

#include "qmm_device.cuh"
#include "qmm_stream.cuh"

namespace qmm {

constexpr int kDmmaWarps = 16;

struct DmmaParams {
    const uint8_t* wq;
    const float* x;
    float* y;
    int32_t* sums;
    float* partial;   // [kslices][M][N] when K is split (summed by qmm_splitk_reduce_kernel)
    unsigned* err;
    long long total_bytes;
    long long rb;
    int M, N, K;
    int units;        // weight units per row (32-blocks or super-blocks)
    int kslices, slice_units, per_slice;
    int ups;          // units per stage (K chunk of a tile)
    int ngroups;      // ceil(N / 8)
    int stages;
    int stage_bytes;
    int row_pitch;    // bytes between rows in a stage with one copy per row (0: one contiguous copy)
    int off_flags, off_codes, off_scale, off_aux, off_rs, off_red, off_stage;
    int code_pitch;   // int8: bytes per activation row; f32: halves per activation row and piece
};

template <int WT, int AM>
__device__ __forceinline__ void dmma_prepare(const DmmaParams& p, uint8_t* smem, int k0, int klen, int tid) {
    constexpr int NTH = kDmmaWarps * 32;
    const int su = p.slice_units;
    if (AM == A_INT8 && WT == T_Q8_0) {
        uint8_t* codes = smem + p.off_codes;
        float* da = reinterpret_cast<float*>(smem + p.off_scale);
        for (int idx = tid; idx < p.M * su; idx += NTH) {
            const int r = idx / su, b = idx - r * su;
            uint32_t c[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            float s = 0.0f;
            if (r < p.M && b * 32 < klen) {
                float d;
                quant_q8_0_32(p.x + (long long)r * p.K + k0 + b * 32, c, d);
                s = h2f(f2h(d));
            }
            uint4* d0 = reinterpret_cast<uint4*>(codes + r * p.code_pitch + b * 32);
            d0[0] = make_uint4(c[0], c[1], c[2], c[3]);
            d0[1] = make_uint4(c[4], c[5], c[6], c[7]);
            da[r * su + b] = s;
        }
    } else if (AM == A_INT8 && WT == T_Q4_K) {
        uint8_t* codes = smem + p.off_codes;
        float* da = reinterpret_cast<float*>(smem + p.off_scale);
        int* bs = reinterpret_cast<int*>(smem + p.off_aux);
        for (int idx = tid; idx < p.M * su; idx += NTH) {
            const int r = idx / su, sb = idx - r * su;
            const bool live = r < p.M && sb * 256 < klen;
            const float* src = p.x + (long long)r * p.K + k0 + sb * 256;
            float d = 0.0f, id = 0.0f;
            if (live) q8_scale(q8k_amax(src), d, id);
            for (int j = 0; j < 8; ++j) {
                uint32_t w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                int sum = 0;
                if (live) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float4 v = __ldg(reinterpret_cast<const float4*>(src + 32 * j) + i);
                        w[i] = pack4(q8_code(v.x, id), q8_code(v.y, id), q8_code(v.z, id), q8_code(v.w, id));
                        sum += bsum4(w[i]);
                    }
                }
                uint4* d0 = reinterpret_cast<uint4*>(codes + r * p.code_pitch + sb * 256 + 32 * j);
                d0[0] = make_uint4(w[0], w[1], w[2], w[3]);
                d0[1] = make_uint4(w[4], w[5], w[6], w[7]);
                bs[r * su * 8 + sb * 8 + j] = sum;
            }
            da[r * su + sb] = d;
        }
    } else {
        // f32_act: per-row power-of-two scale, two f16 pieces; planes hi[8][..], lo[8][..]
        __half* hi = reinterpret_cast<__half*>(smem + p.off_codes);
        __half* lo = hi + p.M * p.code_pitch;
        float* rs = reinterpret_cast<float*>(smem + p.off_rs);   // [8][2]: 2^s, 2^-s
        float* xs = reinterpret_cast<float*>(smem + p.off_aux);  // [8][slice/32] (Q4_K)
        const int warp = tid >> 5, lane = tid & 31;
        if (warp < p.M) {
            const int r = warp;
            float amax = 0.0f;
            if (r < p.M) {
                const float4* src = reinterpret_cast<const float4*>(p.x + (long long)r * p.K + k0);
                for (int i = lane; i < klen / 4; i += 32) {
                    const float4 v = __ldg(src + i);
                    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
                }
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
            uint32_t hw[16], lw[16];
            float sum = 0.0f;
            if (r < p.M && c * 32 < klen) {
                const float scale = rs[2 * r];
                const float4* src = reinterpret_cast<const float4*>(p.x + (long long)r * p.K + k0 + c * 32);
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
            uint4* dh = reinterpret_cast<uint4*>(hi + (long long)r * p.code_pitch + c * 32);
            uint4* dl = reinterpret_cast<uint4*>(lo + (long long)r * p.code_pitch + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                dh[i] = make_uint4(hw[4 * i], hw[4 * i + 1], hw[4 * i + 2], hw[4 * i + 3]);
                dl[i] = make_uint4(lw[4 * i], lw[4 * i + 1], lw[4 * i + 2], lw[4 * i + 3]);
            }
            if (WT == T_Q4_K) xs[r * su * 8 + c] = sum;
        }
    }
}

// 6-bit scale and min of sub-block j of a Q4_K header (words W0..W2 = scales bytes 0..11)
__device__ __forceinline__ void q4k_scmin(const uint4& h, int j, int& sc, int& mn) {
    sc = q4k_sc(h.y, h.w, j);
    mn = q4k_mn(h.z, h.w, j);
}

template <int WT, int AM, int EPI>
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
    const bool whole = p.row_pitch == 0;  // short rows: one contiguous copy of the 8 rows per stage
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
        for (int grp = grp0; grp < p.ngroups && ok; grp += p.per_slice) {
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
                const long long row = (long long)grp * 8 + lane;
                if (whole ? lane == 0 : (lane < 8 && row < p.N)) {
                    const long long s0 = whole ? (long long)grp * 8 * p.rb : row * p.rb + (long long)cu0 * UB;
                    const long long e = whole ? min((long long)grp * 8 + 8, (long long)p.N) * p.rb : s0 + (long long)cnu * UB;
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
    const uint8_t* codes = smem + p.off_codes;
    const float* da = reinterpret_cast<const float*>(smem + p.off_scale);
    const int* bsum = reinterpret_cast<const int*>(smem + p.off_aux);
    const float* xs = reinterpret_cast<const float*>(smem + p.off_aux);
    const float* rs = reinterpret_cast<const float*>(smem + p.off_rs);
    const __half* hi = reinterpret_cast<const __half*>(smem + p.off_codes);
    const __half* lo = hi + p.M * p.code_pitch;
    // activation row of this thread's A fragment; rows >= M repeat row M-1 (their outputs are dropped)
    const int ga = (lane >> 2) < p.M ? (lane >> 2) : p.M - 1;
    float* red = reinterpret_cast<float*>(smem + p.off_red);  // [2][16 warps][64]
    const int su = p.slice_units;
    long long g = 0;
    int tcount = 0;
    for (int grp = grp0; grp < p.ngroups; grp += p.per_slice, ++tcount) {
        float acc0 = 0.0f, acc1 = 0.0f;  // (activation row g8, weight rows 2t4 and 2t4+1)
        for (int ch = 0; ch < nch; ++ch, ++g) {
            const int slot = (int)(g % S);
            const bool ok = mbar_wait(smem_u32(&bars[slot]), (uint32_t)((g / S) & 1), flags, p.err);
            const int cu0 = su0 + ch * p.ups;
            const int cnu = min(p.ups, su0 + sunits - cu0);
            if (ok) {
                const uint8_t* st = smem + p.off_stage + (long long)slot * p.stage_bytes;
                // rows of this thread in the stage: g8 (B operand), 2t4 and 2t4+1 (scales)
                auto rowptr = [&](int r) -> const uint8_t* {
                    const long long n = (long long)grp * 8 + r;
                    if (whole) return st + (int)(((long long)grp * 8 * p.rb) & 15) + (long long)r * p.rb;
                    return st + r * p.row_pitch + (int)((n * p.rb + (long long)cu0 * UB) & 15);
                };
                const uint8_t* rB = rowptr(g8);
                const uint8_t* rS0 = rowptr(2 * t4);
                const uint8_t* rS1 = rowptr(2 * t4 + 1);
                const int ur0 = cu0 - su0;  // first unit of the chunk inside the slice
                for (int uu = warp; uu < cnu; uu += kDmmaWarps) {
                    const int u = ur0 + uu;  // unit index inside the slice (activation side)
                    if (WT == T_Q8_0) {
                        uint32_t w0, w1;
                        lds8_unaligned(rB + 34 * uu + 2 + 8 * t4, w0, w1);
                        const float dw0 = h2f(*reinterpret_cast<const uint16_t*>(rS0 + 34 * uu));
                        const float dw1 = h2f(*reinterpret_cast<const uint16_t*>(rS1 + 34 * uu));
                        if (AM == A_F32) {
                            const uint4 xh = ld128(reinterpret_cast<const uint8_t*>(hi + ga * p.code_pitch + u * 32 + 8 * t4));
                            const uint4 xl = ld128(reinterpret_cast<const uint8_t*>(lo + ga * p.code_pitch + u * 32 + 8 * t4));
                            float d[4] = {0.f, 0.f, 0.f, 0.f};
                            mma_f16(d, xh.x, xl.x, xh.y, xl.y, s8x2_to_h2(w0, SEL01), s8x2_to_h2(w0, SEL23));
                            mma_f16(d, xh.z, xl.z, xh.w, xl.w, s8x2_to_h2(w1, SEL01), s8x2_to_h2(w1, SEL23));
                            acc0 = fmaf(dw0, d[0] + d[2], acc0);
                            acc1 = fmaf(dw1, d[1] + d[3], acc1);
                        } else {
                            const uint2 xa = ld64(codes + ga * p.code_pitch + u * 32 + 8 * t4);
                            int d[4];
                            mma_s8(d, xa.x, 0u, xa.y, 0u, w0, w1);
                            if (EPI == E_Y) {
                                const float dam = da[ga * su + u];
                                acc0 = fmaf((float)d[0], dam * dw0, acc0);
                                acc1 = fmaf((float)d[1], dam * dw1, acc1);
                            } else {
                                const long long n0 = (long long)grp * 8 + 2 * t4;
                                if (g8 < p.M && n0 < p.N) p.sums[((long long)g8 * p.N + n0) * p.units + su0 + u] = d[0];
                                if (g8 < p.M && n0 + 1 < p.N) p.sums[((long long)g8 * p.N + n0 + 1) * p.units + su0 + u] = d[1];
                            }
                        }
                    } else {
                        const uint8_t* sbB = rB + 144 * uu;
                        const uint4 h0 = ld128(rS0 + 144 * uu), h1 = ld128(rS1 + 144 * uu);
                        const float fD0 = h2f(h0.x), fDm0 = h2f(h0.x >> 16), fD1 = h2f(h1.x), fDm1 = h2f(h1.x >> 16);
                        int ssc0 = 0, smn0 = 0, ssc1 = 0, smn1 = 0;
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const uint2 q = ld64(sbB + 16 + 32 * c + 8 * t4);
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const int j = 2 * c + h;
                                const uint32_t nx = (q.x >> (4 * h)) & 0x0F0F0F0Fu, ny = (q.y >> (4 * h)) & 0x0F0F0F0Fu;
                                int sc0, mn0, sc1, mn1;
                                q4k_scmin(h0, j, sc0, mn0);
                                q4k_scmin(h1, j, sc1, mn1);
                                if (AM == A_F32) {
                                    const int kk = u * 256 + 32 * j + 8 * t4;
                                    const uint4 xh = ld128(reinterpret_cast<const uint8_t*>(hi + ga * p.code_pitch + kk));
                                    const uint4 xl = ld128(reinterpret_cast<const uint8_t*>(lo + ga * p.code_pitch + kk));
                                    float d[4] = {0.f, 0.f, 0.f, 0.f};
                                    mma_f16(d, xh.x, xl.x, xh.y, xl.y, u4x2_to_h2(nx, SEL01), u4x2_to_h2(nx, SEL23));
                                    mma_f16(d, xh.z, xl.z, xh.w, xl.w, u4x2_to_h2(ny, SEL01), u4x2_to_h2(ny, SEL23));
                                    const float X = xs[ga * su * 8 + u * 8 + j];
                                    acc0 += fmaf(fD0 * (float)sc0, d[0] + d[2], -(fDm0 * (float)mn0) * X);
                                    acc1 += fmaf(fD1 * (float)sc1, d[1] + d[3], -(fDm1 * (float)mn1) * X);
                                } else {
                                    const uint2 xa = ld64(codes + ga * p.code_pitch + u * 256 + 32 * j + 8 * t4);
                                    int d[4];
                                    mma_s8(d, xa.x, 0u, xa.y, 0u, nx, ny);
                                    const int bsj = bsum[ga * su * 8 + u * 8 + j];
                                    ssc0 += sc0 * d[0];
                                    ssc1 += sc1 * d[1];
                                    smn0 += mn0 * bsj;
                                    smn1 += mn1 * bsj;
                                }
                            }
                        }
                        if (AM == A_INT8) {
                            if (EPI == E_Y) {
                                const float dam = da[ga * su + u];
                                acc0 += dam * (fD0 * (float)ssc0 - fDm0 * (float)smn0);
                                acc1 += dam * (fD1 * (float)ssc1 - fDm1 * (float)smn1);
                            } else {
                                const long long n0 = (long long)grp * 8 + 2 * t4;
                                if (g8 < p.M && n0 < p.N) { int* o = p.sums + (((long long)g8 * p.N + n0) * p.units + su0 + u) * 2; o[0] = ssc0; o[1] = smn0; }
                                if (g8 < p.M && n0 + 1 < p.N) { int* o = p.sums + (((long long)g8 * p.N + n0 + 1) * p.units + su0 + u) * 2; o[0] = ssc1; o[1] = smn1; }
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars[S + slot]));
        }
        if (EPI != E_Y) continue;
        // ---- tile epilogue: 16 warp partials of (activation row, weight row)
        float* rb2 = red + (tcount & 1) * kDmmaWarps * 64;
        rb2[warp * 64 + g8 * 8 + 2 * t4] = acc0;
        rb2[warp * 64 + g8 * 8 + 2 * t4 + 1] = acc1;
        consumer_sync<kDmmaWarps>();
        if (tid < 64) {
            const int m = tid >> 3;
            const long long n = (long long)grp * 8 + (tid & 7);
            float v = 0.0f;
#pragma unroll
            for (int w = 0; w < kDmmaWarps; ++w) v += rb2[w * 64 + tid];
            if (AM == A_F32) v *= rs[2 * m + 1];
            if (!flags[0] && m < p.M && n < p.N) {
                if (p.kslices == 1) p.y[(long long)m * p.N + n] = v;
                else p.partial[((long long)slice * p.M + m) * p.N + n] = v;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// host-side planning
// ---------------------------------------------------------------------------

struct DmmaPlan {
    DmmaParams p;
    int grid;
    size_t smem;
    size_t workspace;
};

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
    p.ngroups = (int)((N + 7) / 8);
    for (int ks = 1; ks <= 16 && ks <= p.units; ++ks) {
        const int su = (p.units + ks - 1) / ks;
        if ((long long)(ks - 1) * su >= p.units) continue;
        const int kv = su * uv;
        int codes, scale = 0, aux = 0, rsb = 0;
        if (am == A_INT8) {
            p.code_pitch = pitch_mod(kv, 32);  // 8-byte A loads of 4 rows per half-warp: no bank conflict
            codes = (int)M * p.code_pitch;
            scale = (int)M * su * 4;
            if (wt == T_Q4_K) aux = (int)M * su * 8 * 4;
        } else {
            p.code_pitch = pitch_mod(2 * kv, 64) / 2;  // halves; 16-byte A loads of 2 rows per quarter-warp
            codes = 2 * (int)M * p.code_pitch * 2;
            if (wt == T_Q4_K) aux = (int)M * (kv / 32) * 4;
        }
        rsb = 8 * 2 * 4;
        int off = 256;
        p.off_flags = off;
        off += 128;
        p.off_codes = off;
        off = round_up(off + codes, 128);
        p.off_scale = off;
        off = round_up(off + scale, 128);
        p.off_aux = off;
        off = round_up(off + aux, 128);
        p.off_rs = off;
        off = round_up(off + rsb, 128);
        p.off_red = off;
        off = round_up(off + 2 * kDmmaWarps * 64 * 4, 128);
        p.off_stage = off;
        long long sb;
        // K chunk per stage: ~4 KB per row copy (4096 values of Q8_0, 8192 of Q4_K)
        const int ups = su < (wt == T_Q8_0 ? 128 : 32) ? su : (wt == T_Q8_0 ? 128 : 32);
        if (ks == 1 && ups == su && p.rb < 2048) {
            sb = 8 * p.rb + 64;  // short rows: one contiguous copy of the whole tile
            p.row_pitch = 0;
        } else {
            // one copy per row; a pitch of 16 mod 128 bytes keeps the 8 rows of a
            // B fragment load on distinct banks (row bytes are often 0 mod 128)
            p.row_pitch = pitch_mod(ups * ub + 48, 16);
            sb = 8LL * p.row_pitch;
        }
        p.ups = ups;
        sb = (sb + 127) / 128 * 128;
        const int stages = sb > 0 ? (int)((smem_max - off) / sb) : 0;
        if (stages < 2) continue;
        p.kslices = ks;
        p.slice_units = su;
        p.stages = stages > 8 ? 8 : stages;
        p.stage_bytes = (int)sb;
        pl.smem = (size_t)off + (size_t)p.stages * sb;
        break;
    }
    if (p.kslices == 0) return false;
    int per = sm_count / p.kslices;
    if (per < 1) per = 1;
    if (per > p.ngroups) per = p.ngroups;
    p.per_slice = per;
    pl.grid = per * p.kslices;
    pl.workspace = p.kslices > 1 ? (size_t)p.kslices * M * N * 4 : 0;
    out = pl;
    return true;
}

}  // namespace qmm
