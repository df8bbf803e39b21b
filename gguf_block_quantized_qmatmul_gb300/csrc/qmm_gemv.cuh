// qmm_gemv.cuh -- the decode GEMV kernel (int8_act, M <= 8 activation rows).
//
// The CPU form of QMatMul ("同一个 GGUF，CPU 和 Metal 生成的文字不一样" section
// 出处): each activation row is quantized (Q8_0 for Q8_0 weights, Q8K for
// Q4_K weights) and multiplied block by block as integer dot products.
//
// GB300 mapping.  Decode is a pure weight stream, so the kernel is organised
// around moving the raw GGUF bytes with as few, as large copies as possible:
// a stage is a group of TR consecutive weight rows (whole rows are contiguous
// in the GGUF layout), fetched by ONE 1-D bulk copy (cp.async.bulk) of the
// 16-byte aligned superset of the group's bytes, completed on an mbarrier.
// One producer lane keeps up to 8 such stages in flight per SM; 16 consumer
// warps work on the oldest.  Each weight row of a stage is owned by 16/TR
// warps; every thread takes whole blocks (a 34-byte Q8_0 block, or a 64-value
// pair of Q4_K sub-blocks) and forms exact int32 dp4a sums against the
// activation codes, which the consumer warps quantized into shared memory at
// the start (overlapped with the first copies).  Row partials are reduced with
// warp shuffles and one named barrier per stage.
#pragma once

#include "qmm_device.cuh"

namespace qmm {

constexpr int kGemvWarps = 16;  // consumer warps; + 1 producer warp

struct GemvParams {
    const uint8_t* wq;
    const float* x;
    float* y;
    int32_t* sums;
    unsigned* err;
    long long total_bytes;  // N * rb
    long long rb;           // bytes per weight row
    int M, N, K;
    int units;              // blocks (Q8_0) or super-blocks (Q4_K) per row
    int tr;                 // rows per stage (1, 2, 4, 8 or 16)
    int ngroups;            // ceil(N / tr)
    int stages;
    int stage_bytes;        // shared bytes per stage slot
    int off_flags, off_codes, off_scale, off_aux, off_red, off_stage;
    int code_pitch;         // bytes per (activation row, 16-byte plane)
};

template <int WT, int MT>
__device__ __forceinline__ void gemv_prepare(const GemvParams& p, uint8_t* smem, int tid) {
    constexpr int NTH = kGemvWarps * 32;
    uint8_t* codes = smem + p.off_codes;
    float* da = reinterpret_cast<float*>(smem + p.off_scale);
    if (WT == T_Q8_0) {
        const int nb = p.units;
        for (int idx = tid; idx < MT * nb; idx += NTH) {
            const int r = idx / nb, b = idx - r * nb;
            uint32_t c[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            float s = 0.0f;
            if (r < p.M) {
                float d;
                quant_q8_0_32(p.x + (long long)r * p.K + b * 32, c, d);
                s = h2f(f2h(d));
            }
            // two 16-byte halves in separate planes [r][half][block]: the lanes
            // of a row read consecutive blocks without bank conflicts
            *reinterpret_cast<uint4*>(codes + (2 * r) * p.code_pitch + b * 16) = make_uint4(c[0], c[1], c[2], c[3]);
            *reinterpret_cast<uint4*>(codes + (2 * r + 1) * p.code_pitch + b * 16) = make_uint4(c[4], c[5], c[6], c[7]);
            da[r * nb + b] = s;
        }
    } else {
        int* bs = reinterpret_cast<int*>(smem + p.off_aux);
        const int nsb = p.units;
        for (int idx = tid; idx < MT * nsb; idx += NTH) {
            const int r = idx / nsb, sb = idx - r * nsb;
            const bool live = r < p.M;
            const float* src = p.x + (long long)r * p.K + sb * 256;
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
                // 64-value pairs of sub-blocks in four 16-byte planes [r][piece][pair]
                const int pair = sb * 4 + (j >> 1), h = j & 1;
                *reinterpret_cast<uint4*>(codes + (4 * r + 2 * h) * p.code_pitch + pair * 16) = make_uint4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<uint4*>(codes + (4 * r + 2 * h + 1) * p.code_pitch + pair * 16) = make_uint4(w[4], w[5], w[6], w[7]);
                bs[r * nsb * 8 + sb * 8 + j] = sum;
            }
            da[r * nsb + sb] = d;
        }
    }
}

// One 34-byte Q8_0 block (2-byte aligned) -> f32 scale and 8 code words.
__device__ __forceinline__ float q8_0_block_words(const uint8_t* blk, uint32_t c[8]) {
    const uintptr_t addr = reinterpret_cast<uintptr_t>(blk);
    const uint8_t* aw = reinterpret_cast<const uint8_t*>(addr & ~uintptr_t(3));
    const uint32_t sh = (uint32_t)(addr & 2u) * 8u;  // 0 or 16
    uint32_t w[9];
#pragma unroll
    for (int k = 0; k < 9; ++k) w[k] = ld32(aw + 4 * k);
#pragma unroll
    for (int k = 0; k < 8; ++k) c[k] = __funnelshift_rc(w[k], w[k + 1], 16u + sh);
    return h2f(sh ? (w[0] >> 16) : w[0]);
}

template <int WT, int MT, int EPI>
__global__ void __launch_bounds__((kGemvWarps + 1) * 32, 1) qmm_gemv_kernel(const GemvParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = p.stages;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);  // full[S], empty[S]
    volatile int* flags = reinterpret_cast<volatile int*>(smem + p.off_flags);
    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(smem_u32(&bars[i]), 1);
            mbar_init(smem_u32(&bars[S + i]), kGemvWarps);
        }
        flags[0] = 0;
        fence_mbar_init();
    }
    __syncthreads();
    grid_dep_launch();  // the next call's first grid may be scheduled (it waits for this one)

    if (warp == kGemvWarps) {
        // ------------------------------ producer ------------------------------
        if (lane != 0) return;
        long long g = 0;
        for (int grp = blockIdx.x; grp < p.ngroups; grp += gridDim.x, ++g) {
            const int slot = (int)(g % S);
            // launched programmatically, the first stages stream while the
            // previous grid finishes; the bounded waits start after it
            if (g == S) grid_dep_wait();
            if (g >= S && !mbar_wait(smem_u32(&bars[S + slot]), (uint32_t)(((g / S) - 1) & 1), flags, p.err)) break;
            uint8_t* st = smem + p.off_stage + (long long)slot * p.stage_bytes;
            const long long s0 = (long long)grp * p.tr * p.rb;
            const long long e = min((long long)(grp + 1) * p.tr, (long long)p.N) * p.rb;
            const long long a = s0 & ~15ll;
            long long b = (e + 15) & ~15ll;
            if (b > p.total_bytes) {  // ragged end of the buffer: the last bytes by plain loads
                b = e & ~15ll;
                for (long long q = b; q < e; ++q) st[q - a] = p.wq[q];
                fence_proxy_async();
            }
            const uint32_t fb = smem_u32(&bars[slot]);
            mbar_arrive_tx(fb, (uint32_t)(b > a ? b - a : 0));
            if (b > a) bulk_g2s(smem_u32(st), p.wq + a, (uint32_t)(b - a), fb);
        }
        const long long first = g > S ? g - S : 0;
        for (long long q = first; q < g; ++q) mbar_drain(smem_u32(&bars[q % S]), (uint32_t)((q / S) & 1), flags, p.err);
        return;
    }

    // ------------------------------ consumers ------------------------------
    grid_dep_wait();  // x may be the previous grid's output
    gemv_prepare<WT, MT>(p, smem, tid);
    consumer_sync<kGemvWarps>();

    const int W = kGemvWarps / p.tr;         // warps per row
    const int r = warp / W;                   // row of the stage this warp works on
    const int li = (warp % W) * 32 + lane;    // lane index inside the row
    const int LPR = W * 32;                   // lanes per row
    const uint8_t* codes = smem + p.off_codes;
    const float* da = reinterpret_cast<const float*>(smem + p.off_scale);
    const int* bsum = reinterpret_cast<const int*>(smem + p.off_aux);
    float* red = reinterpret_cast<float*>(smem + p.off_red);  // [2][16 warps][MT]
    long long g = 0;
    for (int grp = blockIdx.x; grp < p.ngroups; grp += gridDim.x, ++g) {
        const int slot = (int)(g % S);
        const bool ok = mbar_wait(smem_u32(&bars[slot]), (uint32_t)((g / S) & 1), flags, p.err);
        const long long n = (long long)grp * p.tr + r;
        const bool row_ok = ok && n < p.N;
        float acc[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = 0.0f;
        if (row_ok) {
            const uint8_t* st = smem + p.off_stage + (long long)slot * p.stage_bytes;
            const int off = (int)(((long long)grp * p.tr * p.rb) & 15);
            const uint8_t* row = st + off + (long long)r * p.rb;
            if (WT == T_Q8_0) {
                for (int base = li - lane; base < p.units; base += 2 * LPR) {
                    // two blocks per iteration for independent load streams (warp-uniform trip count)
                    const bool l0 = base + lane < p.units;
                    const int b0 = l0 ? base + lane : p.units - 1;
                    const int b1 = b0 + LPR;
                    const bool l1 = l0 && b1 < p.units;
                    uint32_t c0[8], c1[8];
                    const float dw0 = q8_0_block_words(row + 34 * b0, c0);
                    const float dw1 = q8_0_block_words(row + 34 * (l1 ? b1 : b0), c1);
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        const uint4 x0 = ld128(codes + (2 * m) * p.code_pitch + b0 * 16);
                        const uint4 x1 = ld128(codes + (2 * m + 1) * p.code_pitch + b0 * 16);
                        const int bb = l1 ? b1 : b0;
                        const uint4 y0 = ld128(codes + (2 * m) * p.code_pitch + bb * 16);
                        const uint4 y1 = ld128(codes + (2 * m + 1) * p.code_pitch + bb * 16);
                        int s0 = dp4a(c0[0], x0.x, 0), s1 = dp4a(c1[0], y0.x, 0);
                        s0 = dp4a(c0[1], x0.y, s0); s1 = dp4a(c1[1], y0.y, s1);
                        s0 = dp4a(c0[2], x0.z, s0); s1 = dp4a(c1[2], y0.z, s1);
                        s0 = dp4a(c0[3], x0.w, s0); s1 = dp4a(c1[3], y0.w, s1);
                        s0 = dp4a(c0[4], x1.x, s0); s1 = dp4a(c1[4], y1.x, s1);
                        s0 = dp4a(c0[5], x1.y, s0); s1 = dp4a(c1[5], y1.y, s1);
                        s0 = dp4a(c0[6], x1.z, s0); s1 = dp4a(c1[6], y1.z, s1);
                        s0 = dp4a(c0[7], x1.w, s0); s1 = dp4a(c1[7], y1.w, s1);
                        if (EPI == E_Y) {
                            if (l0) acc[m] = fmaf((float)s0, dw0 * da[m * p.units + b0], acc[m]);
                            if (l1) acc[m] = fmaf((float)s1, dw1 * da[m * p.units + b1], acc[m]);
                        } else if (m < p.M) {
                            if (l0) p.sums[((long long)m * p.N + n) * p.units + b0] = s0;
                            if (l1) p.sums[((long long)m * p.N + n) * p.units + b1] = s1;
                        }
                    }
                }
            } else {
                const int ntask = p.units * 4;  // (super-block, pair of sub-blocks)
                // warp-uniform trip count; the 4 tasks of a super-block sit on 4 consecutive lanes
                for (int base = li - lane; base < ntask; base += LPR) {
                    const int q = base + lane;
                    const bool live = q < ntask;
                    const int qc = live ? q : ntask - 1;
                    const int u = qc >> 2, c = qc & 3;
                    const uint8_t* sb = row + 144 * u;
                    const uint4 hw = ld128(sb);  // d, dmin, packed scales
                    const uint4 qa = ld128(sb + 16 + 32 * c), qb = ld128(sb + 32 + 32 * c);
                    const int j0 = 2 * c, j1 = 2 * c + 1;
                    int sc0, mn0, sc1, mn1;
                    if (c < 2) {
                        sc0 = (int)((hw.y >> (8 * j0)) & 63u);
                        mn0 = (int)((hw.z >> (8 * j0)) & 63u);
                        sc1 = (int)((hw.y >> (8 * j1)) & 63u);
                        mn1 = (int)((hw.z >> (8 * j1)) & 63u);
                    } else {
                        const int k0 = j0 - 4, k1 = j1 - 4;
                        sc0 = (int)(((hw.w >> (8 * k0)) & 15u) | (((hw.y >> (8 * k0 + 6)) & 3u) << 4));
                        mn0 = (int)(((hw.w >> (8 * k0 + 4)) & 15u) | (((hw.z >> (8 * k0 + 6)) & 3u) << 4));
                        sc1 = (int)(((hw.w >> (8 * k1)) & 15u) | (((hw.y >> (8 * k1 + 6)) & 3u) << 4));
                        mn1 = (int)(((hw.w >> (8 * k1 + 4)) & 15u) | (((hw.z >> (8 * k1 + 6)) & 3u) << 4));
                    }
                    const uint32_t qq[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
                    uint32_t lo[8], hi[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        lo[k] = qq[k] & 0x0F0F0F0Fu;
                        hi[k] = (qq[k] >> 4) & 0x0F0F0F0Fu;
                    }
                    const float fD = h2f(hw.x), fDm = h2f(hw.x >> 16);
                    const int pair = u * 4 + c;
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        const uint4 a0 = ld128(codes + (4 * m + 0) * p.code_pitch + pair * 16);
                        const uint4 a1 = ld128(codes + (4 * m + 1) * p.code_pitch + pair * 16);
                        const uint4 a2 = ld128(codes + (4 * m + 2) * p.code_pitch + pair * 16);
                        const uint4 a3 = ld128(codes + (4 * m + 3) * p.code_pitch + pair * 16);
                        int s0 = dp4a(lo[0], a0.x, 0), s1 = dp4a(hi[0], a2.x, 0);
                        s0 = dp4a(lo[1], a0.y, s0); s1 = dp4a(hi[1], a2.y, s1);
                        s0 = dp4a(lo[2], a0.z, s0); s1 = dp4a(hi[2], a2.z, s1);
                        s0 = dp4a(lo[3], a0.w, s0); s1 = dp4a(hi[3], a2.w, s1);
                        s0 = dp4a(lo[4], a1.x, s0); s1 = dp4a(hi[4], a3.x, s1);
                        s0 = dp4a(lo[5], a1.y, s0); s1 = dp4a(hi[5], a3.y, s1);
                        s0 = dp4a(lo[6], a1.z, s0); s1 = dp4a(hi[6], a3.z, s1);
                        s0 = dp4a(lo[7], a1.w, s0); s1 = dp4a(hi[7], a3.w, s1);
                        const int2 b2 = *reinterpret_cast<const int2*>(bsum + m * p.units * 8 + u * 8 + j0);
                        int ssc = live ? sc0 * s0 + sc1 * s1 : 0;
                        int smn = live ? mn0 * b2.x + mn1 * b2.y : 0;
                        if (EPI == E_Y) {
                            acc[m] += da[m * p.units + u] * (fD * (float)ssc - fDm * (float)smn);
                        } else {
                            ssc += __shfl_xor_sync(0xffffffffu, ssc, 1);
                            smn += __shfl_xor_sync(0xffffffffu, smn, 1);
                            ssc += __shfl_xor_sync(0xffffffffu, ssc, 2);
                            smn += __shfl_xor_sync(0xffffffffu, smn, 2);
                            if (live && c == 0 && m < p.M) {
                                int* o = p.sums + (((long long)m * p.N + n) * p.units + u) * 2;
                                o[0] = ssc;
                                o[1] = smn;
                            }
                        }
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars[S + slot]));
        if (EPI != E_Y) continue;
        // row partials: warp shuffles, then the W warps of a row via shared memory
        float* rb2 = red + (int)(g & 1) * kGemvWarps * MT;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            float v = acc[m];
#pragma unroll
            for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0) rb2[warp * MT + m] = v;
        }
        consumer_sync<kGemvWarps>();
        if (tid < p.tr * MT) {
            const int rr = tid / MT, m = tid - rr * MT;
            const long long nn = (long long)grp * p.tr + rr;
            float v = 0.0f;
            for (int w = 0; w < W; ++w) v += rb2[(rr * W + w) * MT + m];
            if (m < p.M && nn < p.N && !flags[0]) p.y[(long long)m * p.N + nn] = v;
        }
    }
}

// ---------------------------------------------------------------------------
// host-side planning
// ---------------------------------------------------------------------------

struct GemvPlan {
    GemvParams p;
    int mt;
    int grid;
    size_t smem;
};

// Returns false when this kernel cannot serve the shape (M > 8, or a row too
// long for a ring of at least three whole-row stages).
inline bool plan_gemv(int wt, long long M, long long N, long long K, int sm_count, int smem_max, GemvPlan& out) {
    if (M < 1 || M > 8) return false;
    GemvPlan pl{};
    GemvParams& p = pl.p;
    const int uv = wt == T_Q8_0 ? 32 : 256, ub = wt == T_Q8_0 ? 34 : 144;
    const int mt = M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8;
    p.M = (int)M;
    p.N = (int)N;
    p.K = (int)K;
    p.units = (int)(K / uv);
    p.rb = (long long)p.units * ub;
    p.total_bytes = p.rb * N;
    const int codes = mt * (int)K;                             // activation codes
    const int scale = mt * p.units * 4;
    const int aux = wt == T_Q4_K ? mt * p.units * 8 * 4 : 0;   // sub-block code sums
    p.code_pitch = wt == T_Q8_0 ? p.units * 16 : p.units * 64;
    int off = 256;                                             // barriers (<= 16 x 8 B)
    p.off_flags = off;
    off += 128;
    p.off_codes = off;
    off = round_up(off + codes, 128);
    p.off_scale = off;
    off = round_up(off + scale, 128);
    p.off_aux = off;
    off = round_up(off + aux, 128);
    p.off_red = off;
    off = round_up(off + 2 * kGemvWarps * mt * 4, 128);
    p.off_stage = off;
    // rows per stage: about 32 KB per bulk copy (whole rows), a power of two <= 16
    int tr = 16;
    while (tr > 1 && (long long)tr * p.rb > 40 * 1024) tr >>= 1;
    const long long sb = round_up((int)((long long)tr * p.rb + 64), 128);
    if (sb > smem_max) return false;
    int stages = (int)((smem_max - off) / sb);
    if (stages > 8) stages = 8;
    if (stages < 3) return false;
    p.tr = tr;
    p.stage_bytes = (int)sb;
    p.stages = stages;
    p.ngroups = (int)((N + tr - 1) / tr);
    pl.mt = mt;
    pl.grid = p.ngroups < sm_count ? p.ngroups : sm_count;
    pl.smem = (size_t)off + (size_t)stages * sb;
    out = pl;
    return true;
}

}  // namespace qmm
