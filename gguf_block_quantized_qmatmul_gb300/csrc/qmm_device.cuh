// qmm_device.cuh -- device primitives of the GGUF block-quantized matmul.
//
// Block arithmetic follows the candle tutorial pages ("同一个 GGUF，CPU 和
// Metal 生成的文字不一样" section 出处; "自己量化" sections 3 and
// 和下载的 Q8_0 逐字节比).  Every quantization step is written with explicit
// round-to-nearest intrinsics (__fdiv_rn, __fmul_rn, __fadd_rn, __fsub_rn) so
// that no FMA contraction can change a code: the codes and scales are a
// bit-exact contract with an independent CPU implementation.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace qmm {

enum : int { T_F32 = 0, T_Q8_0 = 1, T_Q4_K = 2, T_Q8_K = 3, T_Q4_0 = 4, T_Q5_0 = 5, T_Q6_K = 6 };
// weight types of 32-value blocks with one f16 scale and signed codes (paired with Q8_0 activations)
__host__ __device__ constexpr bool is_b32(int wt) { return wt == T_Q8_0 || wt == T_Q4_0 || wt == T_Q5_0; }
enum : int { A_INT8 = 0, A_F32 = 1 };
enum : int { E_Y = 0, E_SUMS = 1 };

constexpr unsigned ERR_TIMEOUT = 1u;

// ---------------------------------------------------------------------------
// scalar helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ float h2f(uint32_t bits16) {
    return __half2float(__ushort_as_half((unsigned short)(bits16 & 0xffffu)));
}
__device__ __forceinline__ uint32_t f2h(float f) { return (uint32_t)__half_as_ushort(__float2half_rn(f)); }

// Q8 scale rule: d = amax / 127 in f32; codes use the reciprocal 1/d.
__device__ __forceinline__ void q8_scale(float amax, float& d, float& id) {
    d = __fdiv_rn(amax, 127.0f);
    id = d != 0.0f ? __fdiv_rn(1.0f, d) : 0.0f;
}

// nearest integer (ties away from zero) of x * id, clamped to [-127, 127];
// 0 where the product is NaN (0 * inf: a zero in a block so small that the
// f32 reciprocal of its scale overflows; x / d = 0 there)
__device__ __forceinline__ int q8_code(float x, float id) {
    float r = roundf(__fmul_rn(x, id));
    r = r == r ? r : 0.0f;
    r = fminf(fmaxf(r, -127.0f), 127.0f);
    return (int)r;
}

__device__ __forceinline__ uint32_t pack4(int a, int b, int c, int d) {
    return (uint32_t)(a & 0xff) | ((uint32_t)(b & 0xff) << 8) | ((uint32_t)(c & 0xff) << 16) |
           ((uint32_t)(d & 0xff) << 24);
}

// Quantize 32 consecutive floats (16-byte aligned) to a Q8_0 block: 8 code
// words and the f32 scale d (stored by callers as f16).
__device__ __forceinline__ void quant_q8_0_32(const float* __restrict__ src, uint32_t codes[8], float& d) {
    float4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __ldg(reinterpret_cast<const float4*>(src) + i);
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
    float id;
    q8_scale(amax, d, id);
#pragma unroll
    for (int i = 0; i < 8; ++i)
        codes[i] = pack4(q8_code(v[i].x, id), q8_code(v[i].y, id), q8_code(v[i].z, id), q8_code(v[i].w, id));
}

// Sum of the four signed bytes of w.
__device__ __forceinline__ int bsum4(uint32_t w) {
    return (int)(int8_t)(w & 0xff) + (int)(int8_t)((w >> 8) & 0xff) + (int)(int8_t)((w >> 16) & 0xff) +
           (int)(int8_t)(w >> 24);
}

// Quantize 256 floats to Q8_K: codes[64] words, f32 d, sums of each 16.
// (Two passes: the scale needs the whole block's max first.)
__device__ __forceinline__ float q8k_amax(const float* __restrict__ src) {
    float amax = 0.0f;
    for (int i = 0; i < 64; ++i) {
        float4 v = __ldg(reinterpret_cast<const float4*>(src) + i);
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
    return amax;
}

// Q4_K 6-bit unpack: scales bytes 0-3 in W0, 4-7 in W1, 8-11 in W2.
__device__ __forceinline__ int q4k_sc(uint32_t W0, uint32_t W2, int j) {
    return j < 4 ? (int)((W0 >> (8 * j)) & 63u)
                 : (int)(((W2 >> (8 * (j - 4))) & 15u) | (((W0 >> (8 * (j - 4) + 6)) & 3u) << 4));
}
__device__ __forceinline__ int q4k_mn(uint32_t W1, uint32_t W2, int j) {
    return j < 4 ? (int)((W1 >> (8 * j)) & 63u)
                 : (int)(((W2 >> (8 * (j - 4) + 4)) & 15u) | (((W1 >> (8 * (j - 4) + 6)) & 3u) << 4));
}

// ---------------------------------------------------------------------------
// PTX wrappers: mbarrier, 1-D bulk copy (TMA), warp MMA
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t tx) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(tx) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Spin limit of a bounded wait in SM clocks: 2^31 (about a second), unless
// the word after the device error word holds a smaller log2 (a test hook of
// the host library lowers it so that an injected stall ends in milliseconds).
__device__ __forceinline__ long long wait_limit(const unsigned* err) {
    const unsigned lg = *reinterpret_cast<const volatile unsigned*>(err + 1);
    return 1ll << (lg == 0u || lg > 31u ? 31u : lg);
}

// The limit is read from global memory only once a wait has lasted 2^15
// clocks (below every limit the hook allows), so no handoff between a block's
// roles waits for an L2 round trip.
constexpr long long kWaitLimitCheck = 1ll << 15;

// The spinning part of a bounded wait, out of line: inlined at every wait of
// a many-role kernel it made up much of the code those roles' loops fetch.
// `drain` ignores the abort flag.  Gives up after wait_limit() SM clocks (or,
// unless `drain`, at once when another warp of the block already gave up),
// raising the device error word and the block-wide abort flag.
static __device__ __noinline__ bool mbar_spin(uint32_t bar, uint32_t parity, volatile int* abort_flag, unsigned* err,
                                              bool drain) {
    const long long t0 = clock64();
    long long lim = 0;
    while (true) {
        if (mbar_try(bar, parity)) return true;
        if (!drain && *abort_flag) return false;
        const long long dt = clock64() - t0;
        if (dt > kWaitLimitCheck) {
            if (lim == 0) lim = wait_limit(err);
            if (dt > lim) {
                atomicOr(err, ERR_TIMEOUT);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

// Bounded wait on an mbarrier phase: a first test inline, then mbar_spin.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned* err) {
    if (mbar_try(bar, parity)) return true;
    return mbar_spin(bar, parity, abort_flag, err, false);
}

// Bounded wait for a phase whose arrivals were certainly issued (a copy or an
// MMA commit of this block), ignoring the abort flag: a producer calls it for
// each of its copies still in flight before the block exits, so that even on
// the abort path nothing is still writing the block's shared or tensor memory
// when it is released.
__device__ __forceinline__ bool mbar_drain(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           unsigned* err) {
    if (mbar_try(bar, parity)) return true;
    return mbar_spin(bar, parity, abort_flag, err, true);
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// load one TMA box (2-D tensor map) into shared memory, completing on an mbarrier
__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Programmatic dependent launch: a grid launched with programmatic stream
// serialization may start before the previous grid in its stream completes;
// grid_dep_wait() blocks until that grid has completed and its writes are
// visible, grid_dep_launch() lets the next such grid start.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <int CW>
__device__ __forceinline__ void consumer_sync() {  // the CW consumer warps only
    asm volatile("bar.sync 1, %0;" ::"n"(CW * 32) : "memory");
}

// Shared-memory loads through pointers derived from the kernel's __shared__
// array (the compiler keeps them in the shared address space and may schedule
// them freely between the mbarrier waits, which clobber memory).
__device__ __forceinline__ uint32_t ld32(const uint8_t* p) { return *reinterpret_cast<const uint32_t*>(p); }
__device__ __forceinline__ uint2 ld64(const uint8_t* p) { return *reinterpret_cast<const uint2*>(p); }
__device__ __forceinline__ uint4 ld128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ int dp4a(uint32_t a, uint32_t b, int c) { return __dp4a((int)a, (int)b, c); }

// D = A(16x32 s8) * B(32x8 s8), exact int32, C = 0
__device__ __forceinline__ void mma_s8(int d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                       uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};"
        : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "r"(0));
}

// D = A(16x16 s8) * B(16x8 s8), exact int32, C = 0.  Fragments: a0 row g, a1
// row g + 8, k = 4t..4t+3; b0 k = 4t..4t+3, column g (g = lane / 4, t = lane % 4).
__device__ __forceinline__ void mma_s8_k16(int d[4], uint32_t a0, uint32_t a1, uint32_t b0) {
    asm("mma.sync.aligned.m16n8k16.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%7,%7,%7,%7};"
        : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
        : "r"(a0), "r"(a1), "r"(b0), "r"(0));
}

// D = A(16x32 u8) * B(32x8 s8), exact int32, C = 0
__device__ __forceinline__ void mma_u8s8(int d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k32.row.col.s32.u8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};"
        : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "r"(0));
}

// D = A(16x16 f16) * B(16x8 f16), f32, C = 0
__device__ __forceinline__ void mma_f16_z(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

// D += A(16x16 f16) * B(16x8 f16), f32 accumulate
__device__ __forceinline__ void mma_f16(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D = A(16x8 f16) * B(8x8 f16), f32, C = 0
__device__ __forceinline__ void mma_f16_k8(float d[4], uint32_t a0, uint32_t a1, uint32_t b0) {
    asm(
        "mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%7,%7,%7,%7};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(b0), "f"(0.0f));
}

// Packed f32x2 arithmetic (two lanes per instruction).
__device__ __forceinline__ unsigned long long f2pack(float lo, float hi) {
    return (unsigned long long)__float_as_uint(lo) | ((unsigned long long)__float_as_uint(hi) << 32);
}
__device__ __forceinline__ unsigned long long mul2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b, unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ float f2lo(unsigned long long v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float f2hi(unsigned long long v) { return __uint_as_float((uint32_t)(v >> 32)); }

// The 16 six-bit factors of a Q4_K header as packed bytes: sc0..3, sc4..7,
// m0..3, m4..7 (header words W0, W1, W2 = scales bytes 0-3, 4-7, 8-11).
__device__ __forceinline__ void q4k_unpack4(uint32_t W0, uint32_t W1, uint32_t W2, uint32_t& sc03, uint32_t& sc47,
                                            uint32_t& mn03, uint32_t& mn47) {
    sc03 = W0 & 0x3F3F3F3Fu;
    mn03 = W1 & 0x3F3F3F3Fu;
    sc47 = (W2 & 0x0F0F0F0Fu) | ((W0 >> 2) & 0x30303030u);
    mn47 = ((W2 >> 4) & 0x0F0F0F0Fu) | ((W1 >> 2) & 0x30303030u);
}
// byte j (0..3) of w as f16x2 (v, v), exact: (1024 + v) - 1024
__device__ __forceinline__ uint32_t byte_h2(uint32_t w, int j) {
    const uint32_t sel = (uint32_t)(j | 0x40 | (j << 8) | 0x4000);  // bytes j, 0x64, j, 0x64
    uint32_t h = __byte_perm(w, 0x64646464u, sel);
    __half2 r = __hsub2(*reinterpret_cast<__half2*>(&h), __half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400)));
    return *reinterpret_cast<uint32_t*>(&r);
}
// two nibble codes (bytes lo, lo+1 of w, values 0..15) times the f16x2 factor
// sc2 = (sc, sc), exact: (1024 + n) * sc - 1024 * sc with one rounding (n sc <= 945)
__device__ __forceinline__ uint32_t u4x2_scaled(uint32_t w, uint32_t sel, uint32_t sc2, uint32_t negsc2) {
    uint32_t h = __byte_perm(w, 0x64646464u, sel);
    __half2 r = __hfma2(*reinterpret_cast<__half2*>(&h), *reinterpret_cast<__half2*>(&sc2), *reinterpret_cast<__half2*>(&negsc2));
    return *reinterpret_cast<uint32_t*>(&r);
}

// Two signed bytes (byte lanes lo, lo+1 of w) -> exact f16x2 via 1024 + (q + 128) - 1152.
__device__ __forceinline__ uint32_t s8x2_to_h2(uint32_t w, uint32_t sel) {
    uint32_t h = __byte_perm(w ^ 0x80808080u, 0x64646464u, sel);
    __half2 r = __hsub2(*reinterpret_cast<__half2*>(&h), __half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480)));
    return *reinterpret_cast<uint32_t*>(&r);
}
// Two unsigned nibble bytes (0..15) -> exact f16x2 via (1024 + n) - 1024.
__device__ __forceinline__ uint32_t u4x2_to_h2(uint32_t w, uint32_t sel) {
    uint32_t h = __byte_perm(w, 0x64646464u, sel);
    __half2 r = __hsub2(*reinterpret_cast<__half2*>(&h), __half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400)));
    return *reinterpret_cast<uint32_t*>(&r);
}
constexpr uint32_t SEL01 = 0x5140u;  // bytes 0,1 of w into the low bytes of two halves
constexpr uint32_t SEL23 = 0x7362u;  // bytes 2,3

// 8 bytes starting at a 2-byte aligned shared address, as two words.
__device__ __forceinline__ void lds8_unaligned(const uint8_t* p, uint32_t& r0, uint32_t& r1) {
    uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t* w = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
    uint32_t sh = (uint32_t)(a & 3u) * 8u;
    uint32_t w0 = w[0], w1 = w[1], w2 = w[2];
    r0 = __funnelshift_r(w0, w1, sh);
    r1 = __funnelshift_r(w1, w2, sh);
}

// ---------------------------------------------------------------------------
// Streaming block-MMA kernel: plan shared by host and device
// ---------------------------------------------------------------------------

constexpr int kTileRows = 16;  // weight rows per tile (the MMA M dimension)

inline int round_up(int v, int a) { return (v + a - 1) / a * a; }
// smallest pitch >= v (v a multiple of 16) with pitch % 128 == want
inline int pitch_mod(int v, int want) {
    v = round_up(v, 16);
    return v + ((want - v % 128) % 128 + 128) % 128;
}

struct StreamParams {
    const uint8_t* wq;
    const float* x;
    float* y;
    int32_t* sums;
    float* partial;
    unsigned* counters;
    unsigned* err;
    long long total_bytes;  // N * row_bytes
    long long rb;           // bytes per weight row
    int M, N, K;
    int mr;                 // activation rows per chunk
    int mchunks, kslices, pairs, per_pair;
    int units;              // weight units per row (K / unit values)
    int slice_units;        // units per K slice (last slice may be shorter)
    int ups;                // units per stage
    int stages;
    int row_stride;         // bytes per weight row inside a stage
    int ntiles;
    // shared-memory layout (bytes from the dynamic smem base)
    int off_stage, off_codes, off_scale, off_aux, off_rs, off_red, off_flags;
    int code_pitch;         // MMA int8_act: bytes per activation row; f32_act: halves per (row, piece);
                            // DOT: bytes per (row, 16-byte lane piece)
    int scale_pitch;        // entries per activation row in the scale array
    int aux_pitch;          // entries per activation row in the aux array (Q8K sub-block sums, Q4_K x sums)
};

}  // namespace qmm
