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
// The weight bytes of all items are one virtual stream; CTA c takes the
// rows whose first byte falls in its 1/G share of it.  For every item it
// meets, the CTA quantizes the item's activation rows into shared memory
// (int8_act), then each warp takes two rows at a time: the lanes read whole
// blocks straight from global memory (every byte once, no shared-memory
// staging), form the per-block sums, and a shuffle reduction gives y.
#include "qmm_internal.h"

namespace qmm {
namespace {

constexpr int kBatchWarps = 8;

__device__ __forceinline__ uint32_t ldg32(const uint8_t* p) { return __ldg(reinterpret_cast<const unsigned int*>(p)); }
__device__ __forceinline__ uint32_t ldg16(const uint8_t* p) { return __ldg(reinterpret_cast<const unsigned short*>(p)); }

// One 32-value block at blk (2-byte aligned, global memory): the f32 scale
// and eight words of signed codes (values 4k..4k+3 in word k).  Reads stay
// inside the block's 4-byte-aligned span, never past its last byte's word.
template <int WT>
__device__ __forceinline__ float load_block(const uint8_t* blk, uint32_t c[8]) {
    const uint8_t* a = reinterpret_cast<const uint8_t*>(reinterpret_cast<uintptr_t>(blk) & ~uintptr_t(3));
    const bool odd = a != blk;  // block starts at a + 2
    if (WT == T_Q8_0) {
        // d: bytes 0-1; codes: bytes 2-33
        uint32_t w[9];
#pragma unroll
        for (int k = 0; k < 8; ++k) w[k] = ldg32(a + 4 * k);
        w[8] = odd ? ldg32(a + 32) : ldg16(a + 32);
#pragma unroll
        for (int k = 0; k < 8; ++k) c[k] = odd ? w[k + 1] : __funnelshift_r(w[k], w[k + 1], 16);
        return h2f(odd ? (w[0] >> 16) : (w[0] & 0xFFFFu));
    } else {
        // d: bytes 0-1; (Q5_0) fifth bits: bytes 2-5; 16 nibble bytes after them
        constexpr int QS = WT == T_Q5_0 ? 6 : 2;
        constexpr int NW = (QS + 16 + 2 + 3) / 4;  // words of the aligned span when the block starts at a + 2
        uint32_t w[NW];
#pragma unroll
        for (int k = 0; k < NW; ++k) {
            // the last word of an aligned block holds two bytes past it: read them as 16 bits
            if (k == NW - 1 && !odd && (4 * k + 4 > QS + 16)) w[k] = ldg16(a + 4 * k);
            else if (k == NW - 1 && !odd && 4 * k >= QS + 16) w[k] = 0u;
            else w[k] = ldg32(a + 4 * k);
        }
        auto at = [&](int byte) -> uint32_t {  // the 4 bytes at block offset `byte` (even)
            const int o = byte + (odd ? 2 : 0);
            return (o & 3) ? __funnelshift_r(w[o >> 2], w[(o >> 2) + 1], 16) : w[o >> 2];
        };
        uint32_t q[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) q[k] = at(QS + 4 * k);
        const uint32_t hb = WT == T_Q5_0 ? at(2) : 0u;
        constexpr uint32_t OFF = WT == T_Q5_0 ? 0x10101010u : 0x08080808u;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            // values 4k..4k+3: low nibbles of word k (k < 4) or high nibbles of word k - 4
            uint32_t v = k < 4 ? (q[k & 3] & 0x0F0F0F0Fu) : ((q[k & 3] >> 4) & 0x0F0F0F0Fu);
            if (WT == T_Q5_0) v |= ((((hb >> (4 * k)) & 0xFu) * 0x00204081u) & 0x01010101u) << 4;
            c[k] = __vsub4(v, OFF);
        }
        return h2f(odd ? (w[0] >> 16) : (w[0] & 0xFFFFu));
    }
}

// resident CTAs per SM: more for one activation row (fewer registers a thread)
__host__ __device__ constexpr int batch_ctas_per_sm(int mt) { return mt == 1 ? 3 : 2; }

template <int WT, int AM, int MT>
__global__ void __launch_bounds__(kBatchWarps * 32, batch_ctas_per_sm(MT)) qmm_batch_kernel(const BatchParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    constexpr int BB = WT == T_Q8_0 ? 34 : WT == T_Q5_0 ? 22 : 18;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const long long lo = p.total * blockIdx.x / gridDim.x, hi = p.total * (blockIdx.x + 1) / gridDim.x;
    for (int i = 0; i < p.count; ++i) {
        const BatchItem& it = p.it[i];
        const long long rb = (long long)(it.K / 32) * BB;
        const long long b0 = it.byte0;
        if (b0 + (long long)it.N * rb <= lo || b0 >= hi) continue;
        // rows whose first byte lies in [lo, hi)
        const long long r0 = lo > b0 ? (lo - b0 + rb - 1) / rb : 0;
        long long r1 = (hi - b0 + rb - 1) / rb;
        if (r1 > it.N) r1 = it.N;
        if (r0 >= r1) continue;
        const int nb = it.K / 32, M = it.M;
        uint8_t* codes = smem;                                            // [M][K] int8
        float* da = reinterpret_cast<float*>(smem + (size_t)M * it.K);    // [M][K/32]
        if (AM == A_INT8) {
            __syncthreads();  // the previous item's codes are no longer read
            for (int idx = tid; idx < M * nb; idx += kBatchWarps * 32) {
                const int m = idx / nb, b = idx - m * nb;
                uint32_t c[8];
                float d;
                quant_q8_0_32(it.x + (long long)m * it.K + 32 * b, c, d);
                uint4* o = reinterpret_cast<uint4*>(codes + (size_t)m * it.K + 32 * b);
                o[0] = make_uint4(c[0], c[1], c[2], c[3]);
                o[1] = make_uint4(c[4], c[5], c[6], c[7]);
                da[m * nb + b] = h2f(f2h(d));
            }
            __syncthreads();
        }
        for (long long r = r0 + warp; r < r1; r += 2 * kBatchWarps) {
            const long long rr[2] = {r, r + kBatchWarps};
            const bool live1 = rr[1] < r1;
            float acc[2][MT];
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int m = 0; m < MT; ++m) acc[j][m] = 0.0f;
            for (int b = lane; b < nb; b += 32) {
                uint32_t c[2][8];
                float dw[2];
                dw[0] = load_block<WT>(it.wq + rr[0] * rb + (long long)b * BB, c[0]);
                dw[1] = live1 ? load_block<WT>(it.wq + rr[1] * rb + (long long)b * BB, c[1]) : 0.0f;
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    if (m >= M) break;
                    if (AM == A_INT8) {
                        const uint4* ap = reinterpret_cast<const uint4*>(codes + (size_t)m * it.K + 32 * b);
                        const uint4 a0 = ap[0], a1 = ap[1];
                        const uint32_t av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                        const float s = da[m * nb + b];
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            int isum = 0;
#pragma unroll
                            for (int k = 0; k < 8; ++k) isum = __dp4a((int)c[j][k], (int)av[k], isum);
                            acc[j][m] = fmaf(dw[j] * s, (float)isum, acc[j][m]);
                        }
                    } else {
                        const float4* xp = reinterpret_cast<const float4*>(it.x + (long long)m * it.K + 32 * b);
                        float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const float4 v = __ldg(xp + k);
                            const float xv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                s0 = fmaf((float)(int8_t)(c[0][k] >> (8 * e)), xv[e], s0);
                                s1 = fmaf((float)(int8_t)(c[1][k] >> (8 * e)), xv[e], s1);
                            }
                        }
                        acc[0][m] = fmaf(dw[0], s0, acc[0][m]);
                        acc[1][m] = fmaf(dw[1], s1, acc[1][m]);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int m = 0; m < MT; ++m) {
#pragma unroll
                    for (int o = 16; o; o >>= 1) acc[j][m] += __shfl_xor_sync(0xffffffffu, acc[j][m], o);
                }
            if (lane == 0) {
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    if (m >= M) break;
                    it.y[(long long)m * it.N + rr[0]] = acc[0][m];
                    if (live1) it.y[(long long)m * it.N + rr[1]] = acc[1][m];
                }
            }
        }
    }
}

template <int WT, int AM>
cudaError_t go_mt(const BatchParams& p, int mt, int grid, cudaStream_t s) {
    const size_t smem = AM == A_INT8 ? (size_t)p.max_mk + (size_t)p.max_mk / 32 * 4 : 0;
    switch (mt) {
        case 1: qmm_batch_kernel<WT, AM, 1><<<grid, kBatchWarps * 32, smem, s>>>(p); break;
        case 2: qmm_batch_kernel<WT, AM, 2><<<grid, kBatchWarps * 32, smem, s>>>(p); break;
        case 4: qmm_batch_kernel<WT, AM, 4><<<grid, kBatchWarps * 32, smem, s>>>(p); break;
        default: qmm_batch_kernel<WT, AM, 8><<<grid, kBatchWarps * 32, smem, s>>>(p); break;
    }
    return cudaGetLastError();
}

template <int WT>
cudaError_t go(int am, const BatchParams& p, int mt, int grid, cudaStream_t s) {
    return am == A_INT8 ? go_mt<WT, A_INT8>(p, mt, grid, s) : go_mt<WT, A_F32>(p, mt, grid, s);
}

}  // namespace

cudaError_t launch_batch(int wt, int am, const BatchParams& p, int max_m, int sm_count, cudaStream_t s) {
    const int mt = max_m <= 1 ? 1 : max_m <= 2 ? 2 : max_m <= 4 ? 4 : 8;
    long long rows = 0;
    for (int i = 0; i < p.count; ++i) rows += p.it[i].N;
    long long grid = (long long)sm_count * batch_ctas_per_sm(mt);
    const long long want = (rows + 2 * kBatchWarps - 1) / (2 * kBatchWarps);  // at least one row pair per warp
    if (grid > want) grid = want < 1 ? 1 : want;
    if (wt == T_Q8_0) return go<T_Q8_0>(am, p, mt, (int)grid, s);
    if (wt == T_Q4_0) return go<T_Q4_0>(am, p, mt, (int)grid, s);
    return go<T_Q5_0>(am, p, mt, (int)grid, s);
}

}  // namespace qmm
