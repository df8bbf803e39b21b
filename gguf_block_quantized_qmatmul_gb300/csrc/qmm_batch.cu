// qmm_batch.cu -- many independent small matmuls in one launch: the linears
// of a decode step (q/k/v, o, gate/up, down, the output head), which one at
// a time are bound by launch latency rather than by their weight bytes.
//
// Both QMatMul forms ("同一个 GGUF，CPU 和 Metal 生成的文字不一样" section
// 出处), for the 32-value block types (Q8_0, Q4_0, Q5_0 weights with Q8_0
// activations):
//   int8_act: y = sum_b f(d_w) f(d_a) isum_b, isum_b the exact int32 dot of
//             the weight codes and the row-quantized activation codes;
//   f32_act:  y = sum_b f(d_w) sum_i code_i x_i (f32 products and sums).
//
// The weight bytes of all items are one virtual stream; CTA c (one per SM)
// takes the rows whose first byte falls in its 1/G share of it, item by item
// (a "piece": consecutive rows of one item, contiguous bytes).  A producer
// lane streams each piece in stages of whole rows, one 1-D bulk copy per
// stage, into a ring of shared-memory slots (the copy engine pays a fixed cost
// per contiguous segment, so stages are large).  16 consumer warps stage the
// item's activation rows in shared memory when a piece starts (int8_act
// quantizes them; f32_act copies them), then take each stage's rows in lane
// groups: lpr lanes per group, two rows per group sharing the activation
// loads, lane gl taking blocks gl, gl + lpr, ...; the group sums its lanes
// with a shuffle tree.  lpr, the blocks per lane and the rows per stage are
// planned per K on the host.
#include <algorithm>

#include "qmm_internal.h"

namespace qmm {
namespace {

constexpr int kBatchWarps = 16;            // consumer warps; + 1 producer warp
constexpr int kBatchStagesMax = 6;         // ring slots, fewer when the activations need the room
constexpr int kBatchStageCap = 56 * 1024;  // the most bytes of whole rows a stage is planned to hold
constexpr int kActInt8 = 48;               // int8_act: bytes per activation block in shared memory
constexpr int kActF32 = 144;               // f32_act: bytes per activation block in shared memory

// weight rows a lane group works on at once (they share the activation loads)
__host__ __device__ constexpr int batch_rows_per_group(int am, int mt) { return mt == 1 || (am == A_INT8 && mt == 2) ? 2 : 1; }

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
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b, unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// acc[h][m] += the contribution of block b of weight row h (h < R) to output
// row m, where v[h].  wo[h]: the weight blocks' offsets; ao: the offset of the
// activation block for row 0; astep: the offset between activation rows.
// The R rows share each activation load.
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
            // f32 products of code and x, summed in f32 pairs; a code becomes a float
            // exactly as the bit pattern of 2^23 + (code + 128) minus 2^23 + 128
            const unsigned long long neg = pack2(__float_as_uint(-8388736.0f), __float_as_uint(-8388736.0f));
            unsigned long long s01[R], s23[R];
#pragma unroll
            for (int h = 0; h < R; ++h) s01[h] = 0, s23[h] = 0;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint4 xv = ld128(a + 16 * k);
                const unsigned long long x01 = pack2(xv.x, xv.y), x23 = pack2(xv.z, xv.w);
#pragma unroll
                for (int h = 0; h < R; ++h) {
                    const uint32_t u = c[h][k] ^ 0x80808080u;
                    const unsigned long long q01 =
                        add2(pack2(__byte_perm(u, 0x4B000000u, 0x7440u), __byte_perm(u, 0x4B000000u, 0x7441u)), neg);
                    const unsigned long long q23 =
                        add2(pack2(__byte_perm(u, 0x4B000000u, 0x7442u), __byte_perm(u, 0x4B000000u, 0x7443u)), neg);
                    s01[h] = fma2(q01, x01, s01[h]);
                    s23[h] = fma2(q23, x23, s23[h]);
                }
            }
#pragma unroll
            for (int h = 0; h < R; ++h) {
                const unsigned long long s2 = add2(s01[h], s23[h]);
                const float2 sv = unpack2(s2);
                const float t = fmaf(dw[h], sv.x + sv.y, acc[h][m]);
                acc[h][m] = v[h] ? t : acc[h][m];
            }
        }
    }
}

// The first item whose weight bytes reach past lo (items are in byte order).
__device__ __forceinline__ int batch_first_item(const BatchParams& p, long long lo) {
    int a = 0, b = p.count;  // invariant: items before a end at or before lo
    while (a < b) {
        const int m = (a + b) >> 1;
        const long long end = m + 1 < p.count ? p.it[m + 1].byte0 : p.total;
        if (end <= lo) a = m + 1;
        else b = m;
    }
    return a;
}

// The rows of item it whose first weight byte lies in [lo, hi): [r0, r1).
__device__ __forceinline__ void batch_rows(const BatchItem& it, long long rb, long long lo, long long hi, long long& r0,
                                           long long& r1) {
    const long long b0 = it.byte0;
    r0 = lo > b0 ? (lo - b0 + rb - 1) / rb : 0;
    r1 = hi > b0 ? (hi - b0 + rb - 1) / rb : 0;
    if (r1 > it.N) r1 = it.N;
    if (r0 > r1) r0 = r1;
}

template <int WT, int AM, int MT>
__global__ void __launch_bounds__((kBatchWarps + 1) * 32, 1) qmm_batch_kernel(const BatchParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int BB = WT == T_Q8_0 ? 34 : WT == T_Q5_0 ? 22 : 18;
    constexpr int ES = AM == A_INT8 ? kActInt8 : kActF32;
    constexpr int R = batch_rows_per_group(AM, MT);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = p.stages;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);                 // full[S], empty[S]
    volatile int* flags = reinterpret_cast<volatile int*>(smem + 256);  // [0] abort
    constexpr int ring = 1024;                                          // S slots of p.slot_bytes
    const int acts = ring + S * p.slot_bytes;  // activation blocks: [M][K/32] of ES bytes
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
        for (int i = batch_first_item(p, lo); i < p.count && p.it[i].byte0 < hi && ok; ++i) {
            const BatchItem& it = p.it[i];
            const long long rb = (long long)(it.K / 32) * BB;
            long long r0, r1;
            batch_rows(it, rb, lo, hi, r0, r1);
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
    int prep_m = 0, prep_k = 0;
    for (int i = batch_first_item(p, lo); i < p.count && p.it[i].byte0 < hi; ++i) {
        const BatchItem& it = p.it[i];
        const int nb = it.K / 32, M = it.M, rb = nb * BB;
        long long r0, r1;
        batch_rows(it, rb, lo, hi, r0, r1);
        if (r0 >= r1) continue;
        if (it.x != prep_x || M != prep_m || it.K != prep_k) {
            // the item's activation rows into shared memory, block (m, b) at (m * nb + b) * ES
            consumer_sync<kBatchWarps>();  // the previous activations are no longer read
            if (AM == A_INT8) {
                for (int blk = tid; blk < M * nb; blk += kBatchWarps * 32) {
                    uint32_t c[8];
                    float d;
                    quant_q8_0_32(it.x + 32ll * blk, c, d);  // rows are contiguous: block blk of [M][K/32]
                    uint8_t* o = smem + acts + blk * ES;
                    *reinterpret_cast<uint4*>(o) = make_uint4(c[0], c[1], c[2], c[3]);
                    *reinterpret_cast<uint4*>(o + 16) = make_uint4(c[4], c[5], c[6], c[7]);
                    *reinterpret_cast<float*>(o + 32) = h2f(f2h(d));
                }
            } else {
                const float4* src = reinterpret_cast<const float4*>(it.x);
                for (int idx = tid; idx < M * it.K / 4; idx += kBatchWarps * 32)
                    *reinterpret_cast<float4*>(smem + acts + (idx >> 3) * ES + (idx & 7) * 16) = __ldg(src + idx);
            }
            consumer_sync<kBatchWarps>();
            prep_x = it.x, prep_m = M, prep_k = it.K;
        }
        // lanes in groups of lpr, R weight rows per group: lane gl of a group takes the
        // rows' blocks gl, gl + lpr, ... (bpl of them), and the group sums its lanes.
        // A warp holds rpw groups; its rows are j0 + grp + h * rpw.
        const int lpr = it.lpr, bpl = it.bpl, tr = it.tr, rpw = 32 / lpr;
        const int grp = lane / lpr, gl = lane - grp * lpr;
        const int astep = nb * ES;
        for (long long r = r0; r < r1; r += tr) {
            const bool ok = mbar_wait(smem_u32(&bars[slot]), phase, flags, p.err);
            const int rows = (int)(r + tr < r1 ? tr : r1 - r);
            const int st = ring + slot * p.slot_bytes + (int)((r * rb) & 15);
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
                    const int cb = b < nb ? b : 0;
                    bool v[R];
                    int wo[R];
#pragma unroll
                    for (int h = 0; h < R; ++h) v[h] = jv[h] && b < nb, wo[h] = wrow[h] + cb * BB;
                    block_dot<WT, AM, MT, R>(smem, wo, acts + cb * ES, astep, M, v, acc);
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
}

template <int WT, int AM>
cudaError_t go_mt(BatchParams& p, int mt, int grid, int smem_max, cudaStream_t s) {
    const long long acts = (long long)p.max_mk / 32 * (AM == A_INT8 ? kActInt8 : kActF32);
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

template <int WT>
cudaError_t go(int am, BatchParams& p, int mt, int grid, int smem_max, cudaStream_t s) {
    return am == A_INT8 ? go_mt<WT, A_INT8>(p, mt, grid, smem_max, s) : go_mt<WT, A_F32>(p, mt, grid, smem_max, s);
}

}  // namespace

void plan_batch_item(int nb, int bb, int am, int mt, int& lpr, int& bpl, int& tr) {
    // Lanes per row (lpr) and blocks per lane (bpl = ceil(nb / lpr)) for a row of
    // nb blocks, and rows per stage (tr).  A warp holds 32 / lpr lane groups of R
    // rows each; a stage is one pass of the 16 consumer warps over its rows, at
    // most kBatchStageCap bytes.  The cost of a pass is about 30 issue slots per
    // block and row a lane takes, 12 per block for the shared activation loads,
    // and the groups' reductions and bookkeeping; the plan with the least cost
    // per row wins.
    const int R = batch_rows_per_group(am, mt);
    const long long rb = (long long)nb * bb;
    const long long cap = std::max<long long>(1, (kBatchStageCap - 32) / rb);
    double best = 1e300;
    lpr = 32, bpl = (nb + 31) / 32, tr = (int)std::min<long long>(kBatchWarps, cap);
    for (int l = 1; l <= 32; ++l) {
        const int b = (nb + l - 1) / l;
        if ((nb + b - 1) / b != l) continue;  // the same bpl with fewer lanes
        const long long t = std::min<long long>((long long)kBatchWarps * (32 / l) * R, cap);
        int levels = 0;
        while ((1 << levels) < l) ++levels;
        const double cost = ((30.0 * R + 12.0) * b + R * (3.0 * levels + 15.0) + 15.0) / (double)t;
        if (cost < best) best = cost, lpr = l, bpl = b, tr = (int)t;
    }
}

cudaError_t launch_batch(int wt, int am, const BatchParams& p0, int max_m, int sm_count, int smem_max, cudaStream_t s) {
    const int mt = max_m <= 1 ? 1 : max_m <= 2 ? 2 : max_m <= 4 ? 4 : 8;
    BatchParams p = p0;
    const int bb = wt == T_Q8_0 ? 34 : wt == T_Q5_0 ? 22 : 18;
    long long stage = 0, rows = 0;
    int last_k = -1, lpr = 0, bpl = 0, tr = 0;  // items of one K share a plan
    for (int i = 0; i < p.count; ++i) {
        BatchItem& it = p.it[i];
        if (it.K != last_k) plan_batch_item(it.K / 32, bb, am, mt, lpr, bpl, tr), last_k = it.K;
        it.lpr = lpr, it.bpl = bpl, it.tr = tr;
        stage = std::max(stage, (long long)it.tr * (it.K / 32) * bb);
        rows += it.N;
    }
    // a slot holds a stage's rows plus the 16-byte alignment slack and the
    // few bytes the block loads read past the last block
    p.slot_bytes = (int)((stage + 32 + 127) / 128 * 128);

    long long grid = sm_count;
    if (grid > rows) grid = rows < 1 ? 1 : rows;
    if (wt == T_Q8_0) return go<T_Q8_0>(am, p, mt, (int)grid, smem_max, s);
    if (wt == T_Q4_0) return go<T_Q4_0>(am, p, mt, (int)grid, smem_max, s);
    return go<T_Q5_0>(am, p, mt, (int)grid, smem_max, s);
}

}  // namespace qmm
