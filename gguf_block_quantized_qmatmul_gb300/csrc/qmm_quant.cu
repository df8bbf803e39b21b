// qmm_quant.cu -- quantize (Q8_0, Q4_K, Q4_0, Q5_0, Q6_K weights; Q8_0, Q8_K
// activations) and dequantize kernels.
//
// "自己量化" section 3 (QTensor::quantize) and section 和下载的 Q8_0 逐字节比
// (Q8_0 scale max|x|/127); "同一个 GGUF，CPU 和 Metal 生成的文字不一样" section
// 出处 (activations quantized per row to Q8_0 / Q8K; CANDLE_DEQUANTIZE_ALL).
// These are load-time / export operations: one thread per block, reads as
// 16-byte vectors, plain stores.  Every rounding step is an explicit
// round-to-nearest intrinsic so the codes match the CPU definition bit for bit.
#include "qmm_internal.h"

namespace qmm {
namespace {

__global__ void quant_q8_0_kernel(const float* __restrict__ x, long long nblocks, long long nb_row, long long K,
                                  uint8_t* __restrict__ out) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= nblocks) return;
    const long long r = i / nb_row, b = i - r * nb_row;
    uint32_t c[8];
    float d;
    quant_q8_0_32(x + r * K + b * 32, c, d);
    uint16_t* o = reinterpret_cast<uint16_t*>(out + i * 34);  // 2-byte aligned block
    o[0] = (uint16_t)f2h(d);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        o[1 + 2 * k] = (uint16_t)(c[k] & 0xffffu);
        o[2 + 2 * k] = (uint16_t)(c[k] >> 16);
    }
}

__global__ void quant_q8_k_kernel(const float* __restrict__ x, long long nblocks, long long nb_row, long long K,
                                  uint8_t* __restrict__ out) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= nblocks) return;
    const long long r = i / nb_row, b = i - r * nb_row;
    const float* src = x + r * K + b * 256;
    float d, id;
    q8_scale(q8k_amax(src), d, id);
    uint32_t* o = reinterpret_cast<uint32_t*>(out + i * 292);  // 4-byte aligned block
    o[0] = __float_as_uint(d);
    int sums[16];
    for (int j = 0; j < 16; ++j) {
        int s = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float4 v = __ldg(reinterpret_cast<const float4*>(src + 16 * j) + k);
            uint32_t w = pack4(q8_code(v.x, id), q8_code(v.y, id), q8_code(v.z, id), q8_code(v.w, id));
            o[1 + 4 * j + k] = w;
            s += bsum4(w);
        }
        sums[j] = s;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)
        o[65 + j] = ((uint32_t)sums[2 * j] & 0xffffu) | ((uint32_t)sums[2 * j + 1] << 16);
}

// Closed-form min/max reading of Q4_K: per sub-block step s_j = (hi - lo)/15
// with lo = min(0, min x), hi = max x, offset mu_j = -lo; d = max s_j / 63,
// dmin = max mu_j / 63; sc_j, m_j nearest integers of s_j/d, mu_j/dmin in
// [0, 63]; codes nearest integers of (x + f(dmin) m_j) / (f(d) sc_j) in [0, 15].
__global__ void quant_q4_k_kernel(const float* __restrict__ x, long long nblocks, long long nb_row, long long K,
                                  uint8_t* __restrict__ out) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= nblocks) return;
    const long long r = i / nb_row, b = i - r * nb_row;
    const float* src = x + r * K + b * 256;
    float s[8], mu[8];
    float smax = 0.0f, mumax = 0.0f;
    for (int j = 0; j < 8; ++j) {
        float lo = 0.0f, hi = __ldg(src + 32 * j);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            float4 v = __ldg(reinterpret_cast<const float4*>(src + 32 * j) + k);
            float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (vv[q] < lo) lo = vv[q];
                if (vv[q] > hi) hi = vv[q];
            }
        }
        s[j] = __fdiv_rn(__fsub_rn(hi, lo), 15.0f);
        mu[j] = __fsub_rn(0.0f, lo);
        if (s[j] > smax) smax = s[j];
        if (mu[j] > mumax) mumax = mu[j];
    }
    const float d = __fdiv_rn(smax, 63.0f), dmin = __fdiv_rn(mumax, 63.0f);
    int sc[8], mn[8];
    for (int j = 0; j < 8; ++j) {
        sc[j] = d > 0.0f ? (int)fminf(fmaxf(roundf(__fdiv_rn(s[j], d)), 0.0f), 63.0f) : 0;
        mn[j] = dmin > 0.0f ? (int)fminf(fmaxf(roundf(__fdiv_rn(mu[j], dmin)), 0.0f), 63.0f) : 0;
    }
    const uint32_t D = f2h(d), Dm = f2h(dmin);
    const float fD = h2f(D), fDm = h2f(Dm);
    uint32_t words[36];
    words[0] = D | (Dm << 16);
    uint8_t sb[12];
    for (int j = 0; j < 4; ++j) {
        sb[j] = (uint8_t)((sc[j] & 63) | ((sc[j + 4] >> 4) << 6));
        sb[4 + j] = (uint8_t)((mn[j] & 63) | ((mn[j + 4] >> 4) << 6));
        sb[8 + j] = (uint8_t)((sc[j + 4] & 15) | ((mn[j + 4] & 15) << 4));
    }
    for (int k = 0; k < 3; ++k)
        words[1 + k] = (uint32_t)sb[4 * k] | ((uint32_t)sb[4 * k + 1] << 8) | ((uint32_t)sb[4 * k + 2] << 16) |
                       ((uint32_t)sb[4 * k + 3] << 24);
    for (int c = 0; c < 4; ++c) {
        const float e_lo = __fmul_rn(fD, (float)sc[2 * c]), o_lo = __fmul_rn(fDm, (float)mn[2 * c]);
        const float e_hi = __fmul_rn(fD, (float)sc[2 * c + 1]), o_hi = __fmul_rn(fDm, (float)mn[2 * c + 1]);
        for (int l4 = 0; l4 < 8; ++l4) {
            const float4 vl = __ldg(reinterpret_cast<const float4*>(src + 64 * c) + l4);
            const float4 vh = __ldg(reinterpret_cast<const float4*>(src + 64 * c + 32) + l4);
            const float a[4] = {vl.x, vl.y, vl.z, vl.w}, h[4] = {vh.x, vh.y, vh.z, vh.w};
            uint32_t w = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int ql = e_lo > 0.0f ? (int)fminf(fmaxf(roundf(__fdiv_rn(__fadd_rn(a[q], o_lo), e_lo)), 0.0f), 15.0f) : 0;
                const int qh = e_hi > 0.0f ? (int)fminf(fmaxf(roundf(__fdiv_rn(__fadd_rn(h[q], o_hi), e_hi)), 0.0f), 15.0f) : 0;
                w |= (uint32_t)(ql | (qh << 4)) << (8 * q);
            }
            words[4 + 8 * c + l4] = w;
        }
    }
    uint4* o = reinterpret_cast<uint4*>(out + i * 144);  // 16-byte aligned block
#pragma unroll
    for (int k = 0; k < 9; ++k) o[k] = make_uint4(words[4 * k], words[4 * k + 1], words[4 * k + 2], words[4 * k + 3]);
}

// Q4_0 / Q5_0 (OFF = 8 / 16; weights paired with Q8_0 activations, 18 / 22
// bytes per 32 values): the value m of largest magnitude (the first on ties,
// sign kept) sets d = m / -OFF; codes roundf(x (1/d)) + OFF clamped to
// [0, 2 OFF - 1].  Block: f16 d; (Q5_0) a little-endian word whose bit i is
// bit 4 of code i; 16 bytes, byte j = code j | code j + 16 << 4.
template <int OFF>
__global__ void quant_x_0_kernel(const float* __restrict__ x, long long nblocks, long long nb_row, long long K,
                                 uint8_t* __restrict__ out) {
    constexpr int BYTES = OFF == 16 ? 22 : 18;
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= nblocks) return;
    const long long r = i / nb_row, b = i - r * nb_row;
    const float4* src = reinterpret_cast<const float4*>(x + r * K + b * 32);
    float v[32];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float4 t = __ldg(src + k);
        v[4 * k] = t.x;
        v[4 * k + 1] = t.y;
        v[4 * k + 2] = t.z;
        v[4 * k + 3] = t.w;
    }
    float amax = 0.0f, m = 0.0f;
#pragma unroll
    for (int k = 0; k < 32; ++k) {
        const float a = fabsf(v[k]);
        if (a > amax) {
            amax = a;
            m = v[k];
        }
    }
    const float d = __fdiv_rn(m, (float)(-OFF));
    const float id = d != 0.0f ? __fdiv_rn(1.0f, d) : 0.0f;
    int c[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) {
        float t = roundf(__fmul_rn(v[k], id));
        t = t == t ? t : 0.0f;  // 0 * inf (a zero where 1/d overflows): x / d = 0
        c[k] = (int)fminf(fmaxf(__fadd_rn(t, (float)OFF), 0.0f), (float)(2 * OFF - 1));
    }
    uint16_t* o = reinterpret_cast<uint16_t*>(out + i * BYTES);  // 2-byte aligned block
    o[0] = (uint16_t)f2h(d);
    int q0 = 1;
    if (OFF == 16) {
        uint32_t h = 0;
#pragma unroll
        for (int k = 0; k < 32; ++k) h |= (uint32_t)((c[k] >> 4) & 1) << k;
        o[1] = (uint16_t)(h & 0xffffu);
        o[2] = (uint16_t)(h >> 16);
        q0 = 3;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t b0 = (uint32_t)((c[2 * j] & 15) | ((c[2 * j + 16] & 15) << 4));
        const uint32_t b1 = (uint32_t)((c[2 * j + 1] & 15) | ((c[2 * j + 17] & 15) << 4));
        o[q0 + j] = (uint16_t)(b0 | (b1 << 8));
    }
}

template <int OFF>
__global__ void dequant_x_0_kernel(const uint8_t* __restrict__ q, long long nblocks, float* __restrict__ out) {
    constexpr int BYTES = OFF == 16 ? 22 : 18;
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= nblocks) return;
    const uint16_t* blk = reinterpret_cast<const uint16_t*>(q + i * BYTES);
    const float d = h2f(blk[0]);
    const uint32_t h = OFF == 16 ? (uint32_t)blk[1] | ((uint32_t)blk[2] << 16) : 0u;
    const int q0 = OFF == 16 ? 3 : 1;
    float v[32];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t pair = blk[q0 + j];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int l = 2 * j + e;
            const uint32_t byte = (pair >> (8 * e)) & 0xffu;
            const int lo = (int)((byte & 15u) | (((h >> l) & 1u) << 4)) - OFF;
            const int hi = (int)((byte >> 4) | (((h >> (l + 16)) & 1u) << 4)) - OFF;
            v[l] = d * (float)lo;         // exact: 11 x 5 bits
            v[l + 16] = d * (float)hi;
        }
    }
    float4* o = reinterpret_cast<float4*>(out + i * 32);
#pragma unroll
    for (int k = 0; k < 8; ++k) o[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
}

__global__ void dequant_q8_0_kernel(const uint8_t* __restrict__ q, long long nblocks, float* __restrict__ out) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= nblocks) return;
    const uint16_t* blk = reinterpret_cast<const uint16_t*>(q + i * 34);
    const float d = h2f(blk[0]);
    float4* o = reinterpret_cast<float4*>(out + i * 32);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t w = (uint32_t)blk[1 + 2 * k] | ((uint32_t)blk[2 + 2 * k] << 16);
        o[k] = make_float4(d * (float)(int8_t)(w & 0xff), d * (float)(int8_t)((w >> 8) & 0xff),
                           d * (float)(int8_t)((w >> 16) & 0xff), d * (float)(int8_t)(w >> 24));
    }
}

__global__ void dequant_q8_k_kernel(const uint8_t* __restrict__ q, long long nchunks, float* __restrict__ out) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;  // one 32-value chunk
    if (i >= nchunks) return;
    const long long b = i >> 3, c = i & 7;
    const uint32_t* blk = reinterpret_cast<const uint32_t*>(q + b * 292);
    const float d = __uint_as_float(blk[0]);
    float4* o = reinterpret_cast<float4*>(out + i * 32);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t w = blk[1 + 8 * c + k];
        o[k] = make_float4(__fmul_rn(d, (float)(int8_t)(w & 0xff)), __fmul_rn(d, (float)(int8_t)((w >> 8) & 0xff)),
                           __fmul_rn(d, (float)(int8_t)((w >> 16) & 0xff)), __fmul_rn(d, (float)(int8_t)(w >> 24)));
    }
}

__global__ void dequant_q4_k_kernel(const uint8_t* __restrict__ q, long long nsub, float* __restrict__ out) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;  // one sub-block of 32
    if (i >= nsub) return;
    const long long b = i >> 3;
    const int j = (int)(i & 7);
    const uint32_t* blk = reinterpret_cast<const uint32_t*>(q + b * 144);
    const uint32_t hd = blk[0], W0 = blk[1], W1 = blk[2], W2 = blk[3];
    const float e = __fmul_rn(h2f(hd), (float)q4k_sc(W0, W2, j));
    const float o = __fmul_rn(h2f(hd >> 16), (float)q4k_mn(W1, W2, j));
    const int c = j >> 1, sh = (j & 1) * 4;
    float4* dst = reinterpret_cast<float4*>(out + i * 32);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t w = blk[4 + 8 * c + k];
        float v[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) v[t] = __fsub_rn(__fmul_rn(e, (float)((w >> (8 * t + sh)) & 15u)), o);
        dst[k] = make_float4(v[0], v[1], v[2], v[3]);
    }
}

// Q6_K (paired with Q8K activations; 210 bytes per 256 values): ql[128]
// holds the codes' low 4 bits, qh[64] their high 2 bits, then 16 int8 group
// scales and the f16 d.  Value i: half h = i / 128, w = i % 128, quarter
// q = w / 32, l = w % 32; low bits in nibble q / 2 of ql[64h + 32 (q % 2) + l],
// high bits in bits 2q..2q+1 of qh[32h + l]; stored code = code + 32.
// Quantizer (a reading, the signed-max rule per group of 16): the group's
// value m_j of largest magnitude (the first on ties) gives s_j = m_j / -32;
// d = max |s_j| / 127; sc_j = roundf(s_j / d) in [-127, 127]; with
// e_j = f(D) sc_j, code = roundf(x / e_j) in [-32, 31] (0 where e_j = 0).
__device__ __forceinline__ int q6k_ql_byte(int i) { return 64 * (i >> 7) + 32 * ((i >> 5) & 1) + (i & 31); }
__device__ __forceinline__ int q6k_ql_shift(int i) { return 4 * ((i >> 6) & 1); }
__device__ __forceinline__ int q6k_qh_byte(int i) { return 128 + 32 * (i >> 7) + (i & 31); }
__device__ __forceinline__ int q6k_qh_shift(int i) { return 2 * ((i >> 5) & 3); }

__global__ void quant_q6_k_kernel(const float* __restrict__ x, long long nblocks, long long nb_row, long long K,
                                  uint8_t* __restrict__ out) {
    const long long blk = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (blk >= nblocks) return;
    const long long r = blk / nb_row, b = blk - r * nb_row;
    const float* src = x + r * K + b * 256;
    float s[16];
    float smax = 0.0f;
    for (int j = 0; j < 16; ++j) {
        float amax = 0.0f, m = 0.0f;
        for (int i = 0; i < 16; ++i) {
            const float v = __ldg(src + 16 * j + i);
            if (fabsf(v) > amax) amax = fabsf(v), m = v;
        }
        s[j] = __fdiv_rn(m, -32.0f);
        if (fabsf(s[j]) > smax) smax = fabsf(s[j]);
    }
    const float d = __fdiv_rn(smax, 127.0f);
    const uint32_t D = f2h(d);
    const float fD = h2f(D);
    uint32_t w[53];  // the block as 16-bit pairs: bytes 0..209 (and one pad half)
    for (int k = 0; k < 53; ++k) w[k] = 0u;
    for (int j = 0; j < 16; ++j) {
        const int sc = d > 0.0f ? (int)fminf(fmaxf(roundf(__fdiv_rn(s[j], d)), -127.0f), 127.0f) : 0;
        w[(192 + j) >> 2] |= ((uint32_t)sc & 0xFFu) << (8 * ((192 + j) & 3));
        const float e = __fmul_rn(fD, (float)sc);
        for (int i = 16 * j; i < 16 * j + 16; ++i) {
            const int c = e != 0.0f ? (int)fminf(fmaxf(roundf(__fdiv_rn(__ldg(src + i), e)), -32.0f), 31.0f) : 0;
            const uint32_t u = (uint32_t)(c + 32);
            const int bl = q6k_ql_byte(i), bh = q6k_qh_byte(i);
            w[bl >> 2] |= (u & 15u) << (8 * (bl & 3) + q6k_ql_shift(i));
            w[bh >> 2] |= (u >> 4) << (8 * (bh & 3) + q6k_qh_shift(i));
        }
    }
    w[52] |= D;  // bytes 208, 209
    uint16_t* o = reinterpret_cast<uint16_t*>(out + blk * 210);  // 2-byte aligned block
    for (int k = 0; k < 105; ++k) o[k] = (uint16_t)(w[k >> 1] >> (16 * (k & 1)));
}

// one thread per 32 values (a quarter of a half: one ql nibble plane, one qh bit pair)
__global__ void dequant_q6_k_kernel(const uint8_t* __restrict__ q, long long nchunks, float* __restrict__ out) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= nchunks) return;
    const long long b = i >> 3;
    const int c = (int)(i & 7), h = c >> 2, qq = c & 3;
    const uint8_t* blk = q + b * 210;
    const float fD = h2f((uint32_t)blk[208] | ((uint32_t)blk[209] << 8));
    const float e0 = __fmul_rn(fD, (float)(int8_t)blk[192 + 8 * h + 2 * qq]);
    const float e1 = __fmul_rn(fD, (float)(int8_t)blk[192 + 8 * h + 2 * qq + 1]);
    const uint8_t* ql = blk + 64 * h + 32 * (qq & 1);
    const uint8_t* qh = blk + 128 + 32 * h;
    const int sl = 4 * (qq >> 1), shh = 2 * qq;
    float4* dst = reinterpret_cast<float4*>(out + i * 32);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        float v[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int l = 4 * k + t;
            const int code = (int)(((ql[l] >> sl) & 15) | (((qh[l] >> shh) & 3) << 4)) - 32;
            v[t] = __fmul_rn(l < 16 ? e0 : e1, (float)code);
        }
        dst[k] = make_float4(v[0], v[1], v[2], v[3]);
    }
}

inline unsigned grid_for(long long n, int block) { return (unsigned)((n + block - 1) / block); }

// y[i] = sum over K slices s = 0..ks-1 of partial[s][i], in slice order.
__global__ void splitk_reduce_kernel(const float* __restrict__ partial, long long n, int ks, float* __restrict__ y) {
    grid_dep_launch();  // the next call's preparing grid may be scheduled (it waits for this one)
    grid_dep_wait();    // launched while the split kernel runs: wait for its partial sums
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    float v = 0.0f;
    for (int s = 0; s < ks; ++s) v += partial[(long long)s * n + i];
    y[i] = v;
}

}  // namespace

cudaError_t launch_splitk_reduce(const float* partial, long long n, int ks, float* y, cudaStream_t s) {
    // programmatic dependent launch: scheduled while the split kernel still runs
    return launch_pdl(splitk_reduce_kernel, (unsigned)grid_for(n, 256), 256, 0, s, partial, n, ks, y);
}

cudaError_t launch_quantize(int type, const float* x, long long rows, long long K, void* out, cudaStream_t s) {
    const int bs = 128;
    if (type == T_Q8_0) {
        const long long nb = K / 32, n = rows * nb;
        quant_q8_0_kernel<<<grid_for(n, bs), bs, 0, s>>>(x, n, nb, K, static_cast<uint8_t*>(out));
    } else if (type == T_Q8_K) {
        const long long nb = K / 256, n = rows * nb;
        quant_q8_k_kernel<<<grid_for(n, bs), bs, 0, s>>>(x, n, nb, K, static_cast<uint8_t*>(out));
    } else if (type == T_Q4_K) {
        const long long nb = K / 256, n = rows * nb;
        quant_q4_k_kernel<<<grid_for(n, bs), bs, 0, s>>>(x, n, nb, K, static_cast<uint8_t*>(out));
    } else if (type == T_Q6_K) {
        const long long nb = K / 256, n = rows * nb;
        quant_q6_k_kernel<<<grid_for(n, bs), bs, 0, s>>>(x, n, nb, K, static_cast<uint8_t*>(out));
    } else if (type == T_Q4_0 || type == T_Q5_0) {
        const long long nb = K / 32, n = rows * nb;
        if (type == T_Q4_0) quant_x_0_kernel<8><<<grid_for(n, bs), bs, 0, s>>>(x, n, nb, K, static_cast<uint8_t*>(out));
        else quant_x_0_kernel<16><<<grid_for(n, bs), bs, 0, s>>>(x, n, nb, K, static_cast<uint8_t*>(out));
    } else {
        return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_dequantize(int type, const void* q, long long rows, long long K, float* out, cudaStream_t s) {
    const int bs = 256;
    const uint8_t* qb = static_cast<const uint8_t*>(q);
    const long long n = rows * (K / 32);  // 32-value chunks
    if (type == T_Q8_0) dequant_q8_0_kernel<<<grid_for(n, bs), bs, 0, s>>>(qb, n, out);
    else if (type == T_Q8_K) dequant_q8_k_kernel<<<grid_for(n, bs), bs, 0, s>>>(qb, n, out);
    else if (type == T_Q4_K) dequant_q4_k_kernel<<<grid_for(n, bs), bs, 0, s>>>(qb, n, out);
    else if (type == T_Q6_K) dequant_q6_k_kernel<<<grid_for(n, bs), bs, 0, s>>>(qb, n, out);
    else if (type == T_Q4_0) dequant_x_0_kernel<8><<<grid_for(n, bs), bs, 0, s>>>(qb, n, out);
    else if (type == T_Q5_0) dequant_x_0_kernel<16><<<grid_for(n, bs), bs, 0, s>>>(qb, n, out);
    else return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace qmm
