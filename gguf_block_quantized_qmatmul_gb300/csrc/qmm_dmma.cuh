// qmm_dmma.cuh -- decode matmul (M <= 16 activation rows) on warp tensor cores
// with 16-row weight tiles.
//
// Serves both forms of "同一个 GGUF，CPU 和 Metal 生成的文字不一样" section 出处
// at decode batch sizes: the CPU form (activations quantized per row to Q8_0 /
// Q8K, exact integer block sums) and the Metal form (f32 activations times
// weights dequantized in-kernel).
//
// The MMA's A operand holds 16 weight rows, its B operand the activations:
//   int8_act: B column c of column set s = activation row 8 s + c; mma.m16n8k32 takes the
//     raw Q8_0 codes, or the Q4_K nibbles (low as 0..15, high as 16 n), as A
//     with no conversion.  Q8_0: y += f(d_w) f(d_a) isum per block.  Q4_K: S_sc
//     accumulates sc_j * isum_j exactly in int32; S_m = sum_j m_j bsum_j is one
//     f16 MMA per super-block over the 16 sums of 16 activation codes (every
//     product and partial sum is an integer below 2^24, so it is exact).
//   f32_act: each weight unit (Q8_0 block, Q4_K super-block) of each
//     activation row is scaled by its own power of two 2^s and split into two
//     exact f16 pieces, x 2^s = hi + lo; B column 2r holds hi of row r and
//     column 2r+1 its lo (further column sets serve rows 4..15).  Weight codes
//     become exact f16: Q8_0 q; Q4_K sc_j * q (<= 945), the 6-bit factor
//     folded into the conversion, so the 16 MMAs of a super-block chain in one
//     accumulator.  The min term f(dmin) sum_j m_j X_j (X_j = the sub-block's
//     sum of x 2^s) is one mma.m16n8k8 per super-block with X_j / 32 in two f16
//     pieces.  2^-s is applied with the unit's weight scale.
// The MMA k order is a fixed permutation of each 32-value group: thread t4
// of a quad owns values 4t4..4t4+3 and 16+4t4..16+4t4+3 of the group, read as
// two 4-byte words; the f32 activation planes are stored in the matching
// order.  Weight tiles stream through a shared-memory ring as one bulk copy
// per row and K chunk (~4 KB: one SM's bulk-copy engine pays a fixed cost per
// contiguous segment), into rows at a pitch of 16 mod 128 bytes so that the
// word loads of 8 rows x 4 threads hit 32 distinct banks.
// Activations are prepared in the layout the MMAs read: inside the kernel
// for small weight matrices (one launch), or once per call by
// dmma_prep_kernel for large ones, whose output every CTA fetches with a few
// bulk copies after its first weight stages are in flight (programmatic
// dependent launch).  Every grid is launched programmatically: it streams its
// first weight stages while the previous grid in the stream finishes, and
// waits for that grid (griddepcontrol.wait) before it touches the activations
// or starts a bounded wait.  K is split across CTAs only when the activation rows of
// the whole K range do not fit in shared memory; the slices' partial sums then
// go to the workspace and a second small kernel adds them in slice order.
#pragma once

#include "qmm_device.cuh"
#include "qmm_stream.cuh"

namespace qmm {

constexpr int kDmmaWarps = 16;
constexpr int kDmmaRows = 16;  // weight rows per tile
constexpr int kDmmaMaxM = 16;  // activation rows: two int8 column sets, four f32 ones

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
    int off_flags, off_act, off_scale, off_aux, off_red, off_stage;
    int act_pitch;    // int8: bytes per activation row; f32: halves per (row, piece) plane
    int sstride;      // activation scales per unit: 8 * column sets (int8; also the rows of the Q4_K sums), 4 * column sets (f32)
    int xplanes;      // f32 Q4_K: activation planes per unit in the sums of 32 (16, or 8 * column sets when more)
    int aux_unit;     // bytes of the Q4_K aux layout per unit
    // Activations prepared once by dmma_prep_kernel (null: every CTA prepares
    // its own slice).  Byte offsets in ext: codes (int8 [M][K]) or f16 planes
    // ([2M][K] in MMA k order), scales [unit][sstride], aux [unit][...].
    const uint8_t* ext;
    long long ext_codes, ext_scale, ext_aux;
    // Failure test hook (0 = off): when s > 0, block 0's producer issues no
    // weight stage from stage s - 1 on, so that the consumers' bounded wait
    // for that stage runs out (QMM_ERR_TIMEOUT) and the block takes its abort
    // path.  Set only by the library's test hook, never by a plan.
    int stall_stage;
};

// position p (0..31) of a 32-value group in the MMA k order -> value index
__host__ __device__ constexpr int dmma_kperm(int p) {
    return 4 * (p >> 3) + ((p & 4) ? 16 : 0) + ((p & 3) == 1 ? 2 : (p & 3) == 2 ? 1 : (p & 3));
}

// ---------------------------------------------------------------------------
// activation preparation: per-unit work items, shared by the in-kernel path
// (shared memory, one K slice) and dmma_prep_kernel (global memory, all K)
// ---------------------------------------------------------------------------
struct ActDst {
    uint8_t* act;     // int8 codes [M][pitch] bytes, or f16 planes [2M][pitch] halves
    long long pitch;
    float* scale;     // [unit][sstride]
    int sstride;
    uint8_t* aux;     // int8 Q4_K: [unit][8 pairs][sstride rows] f16x2 sums of 16 codes; f32 Q4_K: [unit][xplanes][8] X halves
    int xplanes;
};

// int8 Q8_0, one thread: the 32-block b of row r (src: its 32 floats)
__device__ __forceinline__ void prep_i8_q8_0(const float* src, int r, int b, const ActDst& o) {
    uint32_t c[8];
    float d;
    quant_q8_0_32(src, c, d);
    uint4* dst = reinterpret_cast<uint4*>(o.act + r * o.pitch + b * 32);
    dst[0] = make_uint4(c[0], c[1], c[2], c[3]);
    dst[1] = make_uint4(c[4], c[5], c[6], c[7]);
    o.scale[b * o.sstride + r] = h2f(f2h(d));
}

// int8 Q8K, one warp: super-block sb of row r (src: its 256 floats); lane l
// quantizes values 8l..8l+7
template <bool AUX>  // AUX: also the sums of 16 codes (Q4_K's min term; Q6_K has none)
__device__ __forceinline__ void prep_i8_q8k(const float* src, int r, int sb, int lane, const ActDst& o) {
    const float4 v0 = __ldg(reinterpret_cast<const float4*>(src) + 2 * lane);
    const float4 v1 = __ldg(reinterpret_cast<const float4*>(src) + 2 * lane + 1);
    float amax = fmaxf(fmaxf(fmaxf(fabsf(v0.x), fabsf(v0.y)), fmaxf(fabsf(v0.z), fabsf(v0.w))),
                       fmaxf(fmaxf(fabsf(v1.x), fabsf(v1.y)), fmaxf(fabsf(v1.z), fabsf(v1.w))));
#pragma unroll
    for (int m = 16; m; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
    float d, id;
    q8_scale(amax, d, id);
    const uint32_t w0 = pack4(q8_code(v0.x, id), q8_code(v0.y, id), q8_code(v0.z, id), q8_code(v0.w, id));
    const uint32_t w1 = pack4(q8_code(v1.x, id), q8_code(v1.y, id), q8_code(v1.z, id), q8_code(v1.w, id));
    *reinterpret_cast<uint2*>(o.act + r * o.pitch + sb * 256 + 8 * lane) = make_uint2(w0, w1);
    const int s8 = bsum4(w0) + bsum4(w1);
    const int s16 = s8 + __shfl_xor_sync(0xffffffffu, s8, 1);   // sum of 16 codes (lanes 2i, 2i+1)
    const int s16n = __shfl_down_sync(0xffffffffu, s16, 2);      // the next sum of 16
    // |sum of 16 codes| <= 2032: exact in f16
    if (AUX && (lane & 3) == 0)
        reinterpret_cast<uint32_t*>(o.aux)[(sb * 8 + (lane >> 2)) * o.sstride + r] = f2h((float)s16) | (f2h((float)s16n) << 16);
    if (lane == 0) o.scale[sb * o.sstride + r] = d;
}

// f32: one lane's 8 values of a 32-group (positions 8t..8t+7 of the MMA k
// order: values 4t..4t+3 and 16+4t..16+4t+3), scaled by 2^s and split in two
// f16 pieces; returns the sum of the 8 scaled values
__device__ __forceinline__ float prep_f32_lane(const float4 a, const float4 b, float scale, __half* hi, __half* lo) {
    const float v[8] = {__fmul_rn(a.x, scale), __fmul_rn(a.z, scale), __fmul_rn(a.y, scale), __fmul_rn(a.w, scale),
                        __fmul_rn(b.x, scale), __fmul_rn(b.z, scale), __fmul_rn(b.y, scale), __fmul_rn(b.w, scale)};
    uint32_t hw[4], lw[4];
    float sum = 0.0f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t hb[2], lb[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const float f = v[2 * q + e];
            const __half h = __float2half_rn(f);
            hb[e] = __half_as_ushort(h);
            lb[e] = __half_as_ushort(__float2half_rn(__fsub_rn(f, __half2float(h))));
            sum = __fadd_rn(sum, f);
        }
        hw[q] = hb[0] | (hb[1] << 16);
        lw[q] = lb[0] | (lb[1] << 16);
    }
    *reinterpret_cast<uint4*>(hi) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    *reinterpret_cast<uint4*>(lo) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    return sum;
}

// s of the power-of-two scale 2^s for a unit with largest magnitude amax:
// amax 2^s lies in [2^14, 2^15)
__device__ __forceinline__ int unit_shift(float amax) {
    if (!(amax > 0.0f)) return 0;
    const int e = (int)((__float_as_uint(amax) >> 23) & 0xff) - 127;
    const int s = 14 - e;
    return s > 100 ? 100 : (s < -100 ? -100 : s);
}

__device__ __forceinline__ float lane_amax(const float4 a, const float4 b) {
    return fmaxf(fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w))),
                 fmaxf(fmaxf(fabsf(b.x), fabsf(b.y)), fmaxf(fabsf(b.z), fabsf(b.w))));
}

// f32 Q8_0, one warp: the 8 blocks g0..g0+7 of row r (src: row start, block
// index relative to it); lanes 4i..4i+3 take block g0+i
__device__ __forceinline__ void prep_f32_q8_0(const float* src, int r, int g0, int nblocks, int lane, const ActDst& o) {
    const int b = g0 + (lane >> 2), t = lane & 3;
    const bool live = b < nblocks;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f), c = a;
    if (live) {
        a = __ldg(reinterpret_cast<const float4*>(src + b * 32 + 4 * t));
        c = __ldg(reinterpret_cast<const float4*>(src + b * 32 + 16 + 4 * t));
    }
    float amax = lane_amax(a, c);
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const int s = unit_shift(amax);
    if (!live) return;
    __half* pl = reinterpret_cast<__half*>(o.act);
    prep_f32_lane(a, c, ldexpf(1.0f, s), pl + (2 * r) * o.pitch + b * 32 + 8 * t, pl + (2 * r + 1) * o.pitch + b * 32 + 8 * t);
    if (t == 0) o.scale[b * o.sstride + r] = ldexpf(1.0f, -s);
}

// f32 Q4_K, one warp: super-block sb of row r (src: its 256 floats); lanes
// 4c..4c+3 take 32-group c (sub-block c)
template <bool AUX>  // AUX: also the scaled sums of each 32 (Q4_K's min term; Q6_K has none)
__device__ __forceinline__ void prep_f32_q4_k(const float* src, int r, int sb, int lane, const ActDst& o) {
    const int c = lane >> 2, t = lane & 3;
    const float4 a = __ldg(reinterpret_cast<const float4*>(src + c * 32 + 4 * t));
    const float4 b = __ldg(reinterpret_cast<const float4*>(src + c * 32 + 16 + 4 * t));
    float amax = lane_amax(a, b);
#pragma unroll
    for (int m = 16; m; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
    const int s = unit_shift(amax);
    __half* pl = reinterpret_cast<__half*>(o.act);
    const long long k = (long long)sb * 256 + c * 32 + 8 * t;
    float sum = prep_f32_lane(a, b, ldexpf(1.0f, s), pl + (2 * r) * o.pitch + k, pl + (2 * r + 1) * o.pitch + k);
    sum = __fadd_rn(sum, __shfl_xor_sync(0xffffffffu, sum, 1));
    sum = __fadd_rn(sum, __shfl_xor_sync(0xffffffffu, sum, 2));
    if (AUX && t == 0) {
        // X_c / 32 (|.| < 2^15) in two f16 pieces
        const float xq = __fmul_rn(sum, 0.03125f);
        const __half h = __float2half_rn(xq);
        const __half l = __float2half_rn(__fsub_rn(xq, __half2float(h)));
        uint16_t* xs = reinterpret_cast<uint16_t*>(o.aux);
        xs[(sb * o.xplanes + 2 * r) * 8 + c] = __half_as_ushort(h);
        xs[(sb * o.xplanes + 2 * r + 1) * 8 + c] = __half_as_ushort(l);
    }
    if (lane == 0) o.scale[sb * o.sstride + r] = ldexpf(1.0f, -s);
}

// Items are per thread for int8 Q8_0 and per warp otherwise.
template <int WT, int AM>
__host__ __device__ constexpr bool prep_per_warp() { return !(AM == A_INT8 && is_b32(WT)); }

// The work items of rows 0..M-1 over units u0..u0+nu-1 of x, written at unit
// index 0 of `o`; item indices first, first+step, ...
template <int WT, int AM>
__device__ __forceinline__ void prep_items(const float* x, int M, int K, int u0, int nu, const ActDst& o,
                                           long long first, long long step, int lane) {
    constexpr int UV = Unit<WT>::vals;
    const long long k0 = (long long)u0 * UV;
    if (AM == A_INT8 && is_b32(WT)) {  // Q8_0 activations (Q8_0, Q4_0, Q5_0 weights)
        for (long long i = first; i < (long long)M * nu; i += step) {
            const int r = (int)(i / nu), b = (int)(i - (long long)r * nu);
            prep_i8_q8_0(x + (long long)r * K + k0 + b * 32, r, b, o);
        }
    } else if (AM == A_INT8) {
        for (long long i = first; i < (long long)M * nu; i += step) {
            const int r = (int)(i / nu), sb = (int)(i - (long long)r * nu);
            prep_i8_q8k<WT == T_Q4_K>(x + (long long)r * K + k0 + sb * 256, r, sb, lane, o);
        }
    } else if (is_b32(WT)) {
        const int ng = (nu + 7) / 8;
        for (long long i = first; i < (long long)M * ng; i += step) {
            const int r = (int)(i / ng), gi = (int)(i - (long long)r * ng);
            prep_f32_q8_0(x + (long long)r * K + k0, r, 8 * gi, nu, lane, o);
        }
    } else {
        for (long long i = first; i < (long long)M * nu; i += step) {
            const int r = (int)(i / nu), sb = (int)(i - (long long)r * nu);
            prep_f32_q4_k<WT == T_Q4_K>(x + (long long)r * K + k0 + sb * 256, r, sb, lane, o);
        }
    }
}

// Small blocks spread the preparation over many SMs as soon as the previous
// grid's CTAs leave them (measured faster than 1024-thread blocks).
constexpr int kPrepThreads = 128;

// Once per call, for large weight matrices: the whole K range into ext.
template <int WT, int AM>
__global__ void __launch_bounds__(kPrepThreads) dmma_prep_kernel(const DmmaParams p, uint8_t* ext) {
    // The decode grid may launch now and stream its first weight stages; it
    // waits for this grid before it touches the activations.
    grid_dep_launch();
    grid_dep_wait();  // the previous grid in the stream may still be writing x or reading ext
    ActDst o;
    o.act = ext + p.ext_codes;
    o.pitch = p.K;
    o.scale = reinterpret_cast<float*>(ext + p.ext_scale);
    o.sstride = p.sstride;
    o.aux = ext + p.ext_aux;
    o.xplanes = p.xplanes;
    const long long tid = (long long)blockIdx.x * kPrepThreads + threadIdx.x;
    if (prep_per_warp<WT, AM>())
        prep_items<WT, AM>(p.x, p.M, p.K, 0, p.units, o, tid >> 5, (long long)gridDim.x * (kPrepThreads / 32), threadIdx.x & 31);
    else
        prep_items<WT, AM>(p.x, p.M, p.K, 0, p.units, o, tid, (long long)gridDim.x * kPrepThreads, threadIdx.x & 31);
}

// ---------------------------------------------------------------------------
// weight-side helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t h2_sub(uint32_t a, uint32_t b) {
    __half2 r = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
    return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ __half2 u2h(uint32_t v) { return *reinterpret_cast<__half2*>(&v); }
__device__ __forceinline__ uint32_t h2u(__half2 v) { return *reinterpret_cast<uint32_t*>(&v); }

// One lop3 each: (a & b) | c and (a & b) ^ c.  Callers pass b and c in
// registers (see opaque()): with two immediate operands the compiler splits
// the expression into two logic instructions.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t and_xor(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// a constant the compiler keeps in a register instead of folding it
__device__ __forceinline__ uint32_t opaque(uint32_t v) {
    asm volatile("" : "+r"(v));
    return v;
}

// signed bytes 0 and 2 of w -> exact f16x2: 0x64 | (b ^ 0x80) is 1152 + b
__device__ __forceinline__ uint32_t s8_02_h2(uint32_t w, uint32_t m00ff, uint32_t k6480) {
    return h2_sub(and_xor(w, m00ff, k6480), 0x64806480u);
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
// Warps: kDmmaWarps consumers, one producer (bulk copies), one reducer that
// sums the consumers' tile partials (so that consumers never wait for each
// other at the end of a tile).
constexpr int kDmmaThreads = (kDmmaWarps + 2) * 32;

// activation rows a tile's partial sums hold per weight row: 8 per int8 column
// set, 4 per f32 column set (hi and lo pieces of 4 rows), 8 at least
__host__ __device__ constexpr int dmma_red_cols(int am, int nb) {
    return (am == A_INT8 ? 8 * nb : 4 * nb) > 8 ? (am == A_INT8 ? 8 * nb : 4 * nb) : 8;
}

template <int WT, int AM, int NB, int EPI>
__global__ void __launch_bounds__(kDmmaThreads, 1) qmm_dmma_kernel(const DmmaParams p) {
    constexpr int UB = Unit<WT>::bytes;
    constexpr int RW = dmma_red_cols(AM, NB);  // activation rows per weight row in the reduction buffer
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = p.stages;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);  // full[S], empty[S], red full, red empty, activations
    uint64_t* rfull = bars + 2 * S;
    uint64_t* rempty = bars + 2 * S + 1;
    uint64_t* abar = bars + 2 * S + 2;
    volatile int* flags = reinterpret_cast<volatile int*>(smem + p.off_flags);
    const int slice = blockIdx.x % p.kslices;
    const int grp0 = blockIdx.x / p.kslices;
    const int su0 = slice * p.slice_units;
    const int sunits = min(p.slice_units, p.units - su0);
    const bool whole = p.row_pitch == 0;  // short rows: one contiguous copy of the 16 rows per stage
    const int nch = (sunits + p.ups - 1) / p.ups;
    float* red = reinterpret_cast<float*>(smem + p.off_red);  // [16 warps][16 weight rows][8 activation rows]
    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(smem_u32(&bars[i]), 1);
            mbar_init(smem_u32(&bars[S + i]), kDmmaWarps);
        }
        mbar_init(smem_u32(rfull), kDmmaWarps * 32);
        mbar_init(smem_u32(rempty), 32);
        mbar_init(smem_u32(abar), 1);
        flags[0] = 0;
        fence_mbar_init();
    }
    __syncthreads();
    grid_dep_launch();  // the next grid (a K-split reduction, the next call) may be scheduled

    if (warp == kDmmaWarps) {
        // ------------------------------ producer ------------------------------
        // Prepared activations: wait for the preparing grid, then fetch this
        // CTA's K slice with one copy per row (int8) or (row, piece) plane
        // (f32), one for the scales and one for the aux sums.
        auto fetch_act = [&]() {
            grid_dep_wait();
            const int k0 = su0 * Unit<WT>::vals, klen = sunits * Unit<WT>::vals;
            const int nrow = AM == A_INT8 ? p.M : 2 * p.M;  // up to 32
            const int vb = AM == A_INT8 ? 1 : 2;  // bytes per activation value
            // copies: the nrow rows (or row pieces), the scales, the Q4_K aux sums;
            // lane l takes copies l and l + 32
            auto item = [&](int i, long long& src, uint32_t& dst, uint32_t& bytes) {
                src = 0, dst = 0, bytes = 0;
                if (i < nrow) {
                    src = p.ext_codes + ((long long)i * p.K + k0) * vb;
                    dst = p.off_act + i * p.act_pitch * vb;
                    bytes = (uint32_t)(klen * vb);
                } else if (i == nrow) {
                    src = p.ext_scale + (long long)su0 * p.sstride * 4;
                    dst = p.off_scale;
                    bytes = (uint32_t)(sunits * p.sstride * 4);
                } else if (i == nrow + 1 && WT == T_Q4_K) {
                    src = p.ext_aux + (long long)su0 * p.aux_unit;
                    dst = p.off_aux;
                    bytes = (uint32_t)sunits * (uint32_t)p.aux_unit;
                }
            };
            long long src[2];
            uint32_t dst[2], bytes[2];
            item(lane, src[0], dst[0], bytes[0]);
            item(lane + 32, src[1], dst[1], bytes[1]);
            const uint32_t tx = __reduce_add_sync(0xffffffffu, bytes[0] + bytes[1]);
            if (lane == 0) mbar_arrive_tx(smem_u32(abar), tx);
            __syncwarp();
#pragma unroll
            for (int c = 0; c < 2; ++c)
                if (bytes[c]) bulk_g2s(smem_u32(smem + dst[c]), p.ext + src[c], bytes[c], smem_u32(abar));
        };
        bool act_done = p.ext == nullptr;
        long long g = 0;
        bool ok = true;
        for (int grp = grp0; grp < p.ntiles && ok; grp += p.per_slice) {
            for (int ch = 0; ch < nch && ok; ++ch, ++g) {
                const int slot = (int)(g % S);
                if (g == S) {  // the first stages are in flight: wait for the previous grid
                    grid_dep_wait();
                    if (!act_done) {  // and fetch the prepared activations
                        fetch_act();
                        act_done = true;
                    }
                }
                if (g >= S) {
                    int okl = 1;
                    if (lane == 0) okl = mbar_wait(smem_u32(&bars[S + slot]), (uint32_t)(((g / S) - 1) & 1), flags, p.err);
                    ok = __shfl_sync(0xffffffffu, okl, 0) != 0;
                    if (!ok) break;
                }
                if (p.stall_stage > 0 && blockIdx.x == 0 && g == p.stall_stage - 1) {
                    ok = false;  // injected stall: nothing from this stage on is issued
                    break;
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
        if (!act_done) fetch_act();
        if (lane == 0) {
            const long long first = g > S ? g - S : 0;
            for (long long q = first; q < g; ++q) mbar_drain(smem_u32(&bars[q % S]), (uint32_t)((q / S) & 1), flags, p.err);
            if (p.ext) mbar_drain(smem_u32(abar), 0u, flags, p.err);
        }
        return;
    }
    if (warp == kDmmaWarps + 1) {
        // ------------------------------ reducer ------------------------------
        if (EPI != E_Y) return;
        // a programmatically launched grid may be resident long before its
        // activations exist: start the bounded waits only once they can come
        grid_dep_wait();
        int tc = 0;
        for (int grp = grp0; grp < p.ntiles; grp += p.per_slice, ++tc) {
            if (!mbar_wait(smem_u32(rfull), (uint32_t)(tc & 1), flags, p.err)) break;
#pragma unroll
            for (int i = 0; i < kDmmaRows * RW / 32; ++i) {
                const int o = lane + 32 * i;
                const int m = o % RW;
                const long long n = (long long)grp * kDmmaRows + o / RW;
                float v = 0.0f;
#pragma unroll
                for (int w = 0; w < kDmmaWarps; ++w) v += red[w * kDmmaRows * RW + o];
                if (!flags[0] && m < p.M && n < p.N) {
                    if (p.kslices == 1) p.y[(long long)m * p.N + n] = v;
                    else p.partial[((long long)slice * p.M + m) * p.N + n] = v;
                }
            }
            __syncwarp();
            mbar_arrive(smem_u32(rempty));
        }
        return;
    }

    // ------------------------------ consumers ------------------------------
    if (p.ext) {
        grid_dep_wait();  // as the reducer: bounded waits start once the activations can come
        mbar_wait(smem_u32(abar), 0u, flags, p.err);
    } else {
        ActDst o;
        o.act = smem + p.off_act;
        o.pitch = p.act_pitch;
        o.scale = reinterpret_cast<float*>(smem + p.off_scale);
        o.sstride = p.sstride;
        o.aux = smem + p.off_aux;
        o.xplanes = p.xplanes;
        grid_dep_wait();  // x may be the previous grid's output
        if (prep_per_warp<WT, AM>())
            prep_items<WT, AM>(p.x, p.M, p.K, su0, sunits, o, warp, kDmmaWarps, lane);
        else
            prep_items<WT, AM>(p.x, p.M, p.K, su0, sunits, o, tid, kDmmaWarps * 32, lane);
        consumer_sync<kDmmaWarps>();
    }

    const int g8 = lane >> 2, t4 = lane & 3;
    const uint8_t* act = smem + p.off_act;
    const float* asc = reinterpret_cast<const float*>(smem + p.off_scale);
    const uint32_t* aux = reinterpret_cast<const uint32_t*>(smem + p.off_aux);
    // B-operand column of this thread: activation row (int8) or (row, piece)
    // plane (f32), per column set.  Columns past the batch read a valid row;
    // their outputs are never written.
    int bc[NB];
#pragma unroll
    for (int s = 0; s < NB; ++s) {
        if (AM == A_INT8) {
            const int r = 8 * s + g8;
            bc[s] = r < p.M ? r : r % p.M;
        }
        else {
            const int pl = 8 * s + g8;
            bc[s] = (pl >> 1) < p.M ? pl : pl % (2 * p.M);
        }
    }
    // f32: this thread's output activation row of column set s is t4 + 4 s
    // (its scale index); rows past the batch read row 0's
    int ar[NB];
#pragma unroll
    for (int s = 0; s < NB; ++s) ar[s] = t4 + 4 * s < p.M ? t4 + 4 * s : 0;
    // Q4_K min-term A fragments: bytes of the packed 6-bit mins as f16 pairs
    const uint32_t sel_m2 = (uint32_t)((2 * (t4 & 1)) | 0x40 | ((2 * (t4 & 1) + 1) << 8) | 0x4000);  // m_{2t}, m_{2t+1}
    const uint32_t sel_m1 = (uint32_t)(t4 | 0x40 | (t4 << 8) | 0x4000);                                   // m_t, m_t
    const uint32_t kM00FF = opaque(0x00FF00FFu), k6480 = opaque(0x64806480u);
    const uint32_t kM000F = opaque(0x000F000Fu), kM00F0 = opaque(0x00F000F0u), k6400 = opaque(0x64006400u);
    long long g = 0;
    int tc = 0;
    for (int grp = grp0; grp < p.ntiles; grp += p.per_slice, ++tc) {
        float acc[NB][2][2];
#pragma unroll
        for (int s = 0; s < NB; ++s) acc[s][0][0] = acc[s][0][1] = acc[s][1][0] = acc[s][1][1] = 0.0f;
        for (int ch = 0; ch < nch; ++ch, ++g) {
            const int slot = (int)(g % S);
            const bool ok = mbar_wait(smem_u32(&bars[slot]), (uint32_t)((g / S) & 1), flags, p.err);
            const int cu0 = su0 + ch * p.ups;
            const int cnu = min(p.ups, su0 + sunits - cu0);
            if (ok && warp < cnu) {
                const uint8_t* st = smem + p.off_stage + (long long)slot * p.stage_bytes;
                auto rowptr = [&](int r) -> const uint8_t* {
                    const long long n = (long long)grp * kDmmaRows + r;
                    if (whole) return st + (int)(((long long)grp * kDmmaRows * p.rb) & 15) + (long long)r * p.rb;
                    return st + r * p.row_pitch + (int)((n * p.rb + (long long)cu0 * UB) & 15);
                };
                const uint8_t* r0p = rowptr(g8);
                const int dr = (int)(rowptr(g8 + 8) - r0p);  // row g8+8 relative to row g8 (a multiple of 16)
                const int u0 = cu0 - su0 + warp;              // first unit of this warp (slice-relative)
                if (is_b32(WT)) {
                    // The warp's blocks are 16 apart (16 x 34, 18 or 22 bytes, a multiple of
                    // 4): their payload bytes share one 4-byte alignment.
                    constexpr int QOFF = WT == T_Q5_0 ? 6 : 2;  // codes (Q8_0) or nibble bytes after d (and qh)
                    const uint8_t* q0 = r0p + UB * warp;
                    const uintptr_t a = reinterpret_cast<uintptr_t>(q0 + QOFF);
                    const uint32_t sh = (uint32_t)(a & 3u) * 8u;
                    const uint32_t* w0p = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3)) + t4;
                    const uintptr_t ah = reinterpret_cast<uintptr_t>(q0 + 2);  // Q5_0: the word of fifth bits
                    const uint32_t shh = (uint32_t)(ah & 3u) * 8u;
                    const uint32_t* h0p = reinterpret_cast<const uint32_t*>(ah & ~uintptr_t(3));
                    const uint16_t* s0p = reinterpret_cast<const uint16_t*>(q0);
                    const uint8_t* xp[NB];
#pragma unroll
                    for (int s = 0; s < NB; ++s)
                        xp[s] = AM == A_F32 ? act + (long long)bc[s] * p.act_pitch * 2 + (u0 * 32 + 8 * t4) * 2
                                            : act + bc[s] * p.act_pitch + u0 * 32 + 4 * t4;
                    const float* sp = AM == A_F32 ? asc + u0 * p.sstride : asc + u0 * p.sstride + 2 * t4;
                    int u = u0;
#pragma unroll 2
                    for (int uu = warp; uu < cnu; uu += kDmmaWarps, u += kDmmaWarps) {
                        const uint32_t* w1p = reinterpret_cast<const uint32_t*>(reinterpret_cast<const uint8_t*>(w0p) + dr);
                        const float dw0 = h2f(s0p[0]);
                        const float dw1 = h2f(*reinterpret_cast<const uint16_t*>(reinterpret_cast<const uint8_t*>(s0p) + dr));
                        // signed codes of values 4 t4 .. 4 t4 + 3 (lo) and 16 + 4 t4 .. (hi), rows g8 and g8 + 8
                        uint32_t lo0, hi0, lo1, hi1;
                        if (WT == T_Q8_0) {
                            lo0 = __funnelshift_r(w0p[0], w0p[1], sh), hi0 = __funnelshift_r(w0p[4], w0p[5], sh);
                            lo1 = __funnelshift_r(w1p[0], w1p[1], sh), hi1 = __funnelshift_r(w1p[4], w1p[5], sh);
                        } else {
                            // nibble bytes 4 t4 .. 4 t4 + 3 hold both: values 4 t4 + i in the low
                            // nibbles, 16 + 4 t4 + i in the high nibbles
                            const uint32_t n0 = __funnelshift_r(w0p[0], w0p[1], sh), n1 = __funnelshift_r(w1p[0], w1p[1], sh);
                            uint32_t l0 = n0 & 0x0F0F0F0Fu, h0 = (n0 >> 4) & 0x0F0F0F0Fu;
                            uint32_t l1 = n1 & 0x0F0F0F0Fu, h1 = (n1 >> 4) & 0x0F0F0F0Fu;
                            if (WT == T_Q5_0) {
                                const uint32_t* h1p = reinterpret_cast<const uint32_t*>(reinterpret_cast<const uint8_t*>(h0p) + dr);
                                const uint32_t f0 = __funnelshift_r(h0p[0], h0p[1], shh), f1 = __funnelshift_r(h1p[0], h1p[1], shh);
                                // bit i of the word is bit 4 of code i: four bits to bit 4 of four bytes
                                l0 |= ((((f0 >> (4 * t4)) & 0xFu) * 0x00204081u) & 0x01010101u) << 4;
                                h0 |= ((((f0 >> (16 + 4 * t4)) & 0xFu) * 0x00204081u) & 0x01010101u) << 4;
                                l1 |= ((((f1 >> (4 * t4)) & 0xFu) * 0x00204081u) & 0x01010101u) << 4;
                                h1 |= ((((f1 >> (16 + 4 * t4)) & 0xFu) * 0x00204081u) & 0x01010101u) << 4;
                            }
                            constexpr uint32_t OFF = WT == T_Q5_0 ? 0x10101010u : 0x08080808u;
                            lo0 = __vsub4(l0, OFF), hi0 = __vsub4(h0, OFF), lo1 = __vsub4(l1, OFF), hi1 = __vsub4(h1, OFF);
                        }
                        if (AM == A_F32) {
                            const uint32_t lo0s = lo0 >> 8, hi0s = hi0 >> 8;  // codes 1 and 3 in bytes 0 and 2
                            const uint32_t lo1s = lo1 >> 8, hi1s = hi1 >> 8;
                            const uint32_t a0 = s8_02_h2(lo0, kM00FF, k6480), a1 = s8_02_h2(lo1, kM00FF, k6480);
                            const uint32_t a2 = s8_02_h2(lo0s, kM00FF, k6480), a3 = s8_02_h2(lo1s, kM00FF, k6480);
                            const uint32_t c0 = s8_02_h2(hi0, kM00FF, k6480), c1 = s8_02_h2(hi1, kM00FF, k6480);
                            const uint32_t c2 = s8_02_h2(hi0s, kM00FF, k6480), c3 = s8_02_h2(hi1s, kM00FF, k6480);
#pragma unroll
                            for (int s = 0; s < NB; ++s) {
                                const uint4 xv = ld128(xp[s]);
                                const float io = sp[ar[s]];  // 2^-s of (activation row, block)
                                float d[4];
                                mma_f16_z(d, a0, a1, a2, a3, xv.x, xv.y);
                                mma_f16(d, c0, c1, c2, c3, xv.z, xv.w);
                                acc[s][0][0] = fmaf(dw0 * io, d[0] + d[1], acc[s][0][0]);
                                acc[s][1][0] = fmaf(dw1 * io, d[2] + d[3], acc[s][1][0]);
                                xp[s] += kDmmaWarps * 32 * 2;
                            }
                            sp += kDmmaWarps * p.sstride;
                        } else {
#pragma unroll
                            for (int s = 0; s < NB; ++s) {
                            const uint32_t b0 = ld32(xp[s]), b1 = ld32(xp[s] + 16);
                            xp[s] += kDmmaWarps * 32;
                            int d[4];
                            mma_s8(d, lo0, lo1, hi0, hi1, b0, b1);
                            if (EPI == E_Y) {
                                const float2 dv = *reinterpret_cast<const float2*>(sp + 8 * s);
                                acc[s][0][0] = fmaf((float)d[0], dw0 * dv.x, acc[s][0][0]);
                                acc[s][0][1] = fmaf((float)d[1], dw0 * dv.y, acc[s][0][1]);
                                acc[s][1][0] = fmaf((float)d[2], dw1 * dv.x, acc[s][1][0]);
                                acc[s][1][1] = fmaf((float)d[3], dw1 * dv.y, acc[s][1][1]);
                            } else {
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const int m = 8 * s + 2 * t4 + (i & 1);
                                    const long long n = (long long)grp * kDmmaRows + g8 + 8 * (i >> 1);
                                    if (m < p.M && n < p.N) p.sums[((long long)m * p.N + n) * p.units + su0 + u] = d[i];
                                }
                            }
                            }
                            if (EPI == E_Y) sp += kDmmaWarps * p.sstride;
                        }
                        w0p += kDmmaWarps * UB / 4;
                        h0p += kDmmaWarps * UB / 4;
                        s0p += kDmmaWarps * UB / 2;
                    }
                } else if (WT == T_Q6_K) {
                    // Q6_K super-blocks (210 bytes; a warp's blocks are 16 x 210 bytes apart, a
                    // multiple of 4, so they share one alignment): 16 groups of 16 values, one k16
                    // MMA each.  Group j = 8h + 2q + sg holds values 128h + 32q + 16sg + l (l < 16);
                    // thread t4 takes l = 4t4..4t4+3 from one ql word (nibble plane q / 2) and one
                    // qh word (bit pair q) per row, read as aligned words and realigned.
                    const int o0 = (int)(r0p - smem) + 210 * warp;
                    const uint32_t sh = (uint32_t)(o0 & 2) * 8u;
                    const uint8_t* a0p = smem + (o0 & ~3);
                    int u = u0;
#pragma unroll 1
                    for (int uu = warp; uu < cnu; uu += kDmmaWarps, u += kDmmaWarps, a0p += kDmmaWarps * 210) {
                        const uint8_t* a1p = a0p + dr;
                        const uint8_t* b0p = a0p + (sh >> 3);  // the block of row g8; row g8 + 8 at + dr
                        const float fD0 = h2f(*reinterpret_cast<const uint16_t*>(b0p + 208));
                        const float fD1 = h2f(*reinterpret_cast<const uint16_t*>(b0p + dr + 208));
                        const int8_t* sc0p = reinterpret_cast<const int8_t*>(b0p + 192);
                        const int8_t* sc1p = reinterpret_cast<const int8_t*>(b0p + dr + 192);
                        int ssc[NB][4];
                        float tf[NB][2];
#pragma unroll
                        for (int s = 0; s < NB; ++s) {
                            ssc[s][0] = ssc[s][1] = ssc[s][2] = ssc[s][3] = 0;
                            tf[s][0] = tf[s][1] = 0.0f;
                        }
#pragma unroll
                        for (int h = 0; h < 2; ++h)
#pragma unroll
                            for (int sg = 0; sg < 2; ++sg) {
                                const int lo = 16 * sg + 4 * t4;
                                auto w0 = [&](int off) { return __funnelshift_r(ld32(a0p + off), ld32(a0p + off + 4), sh); };
                                auto w1 = [&](int off) { return __funnelshift_r(ld32(a1p + off), ld32(a1p + off + 4), sh); };
                                const uint32_t L00 = w0(64 * h + lo), L01 = w0(64 * h + 32 + lo), H0 = w0(128 + 32 * h + lo);
                                const uint32_t L10 = w1(64 * h + lo), L11 = w1(64 * h + 32 + lo), H1 = w1(128 + 32 * h + lo);
#pragma unroll
                                for (int q = 0; q < 4; ++q) {
                                    const int j = 8 * h + 2 * q + sg;
                                    const uint32_t n0 = ((q & 1 ? L01 : L00) >> (4 * (q >> 1))) & 0x0F0F0F0Fu;
                                    const uint32_t n1 = ((q & 1 ? L11 : L10) >> (4 * (q >> 1))) & 0x0F0F0F0Fu;
                                    const uint32_t c0 = __vsub4(n0 | (((H0 >> (2 * q)) & 0x03030303u) << 4), 0x20202020u);
                                    const uint32_t c1 = __vsub4(n1 | (((H1 >> (2 * q)) & 0x03030303u) << 4), 0x20202020u);
                                    if (AM == A_INT8) {
                                        const int vb = 128 * h + 32 * q + lo;  // this thread's first value
                                        const int s0 = sc0p[j], s1 = sc1p[j];
#pragma unroll
                                        for (int s = 0; s < NB; ++s) {
                                            int d[4];
                                            mma_s8_k16(d, c0, c1, ld32(act + bc[s] * p.act_pitch + u * 256 + vb));
                                            ssc[s][0] += s0 * d[0];
                                            ssc[s][1] += s0 * d[1];
                                            ssc[s][2] += s1 * d[2];
                                            ssc[s][3] += s1 * d[3];
                                        }
                                    } else {
                                        // the planes hold each quad of a 32-group as values 0, 2, 1, 3:
                                        // codes 0 and 2 go with the first pair, 1 and 3 with the second
                                        const uint32_t a0 = s8_02_h2(c0, kM00FF, k6480), a1 = s8_02_h2(c1, kM00FF, k6480);
                                        const uint32_t a2 = s8_02_h2(c0 >> 8, kM00FF, k6480), a3 = s8_02_h2(c1 >> 8, kM00FF, k6480);
                                        const float e0 = __fmul_rn(fD0, (float)sc0p[j]), e1 = __fmul_rn(fD1, (float)sc1p[j]);
#pragma unroll
                                        for (int s = 0; s < NB; ++s) {
                                            const uint2 xv = ld64(act + ((long long)bc[s] * p.act_pitch + u * 256 + 32 * (4 * h + q) +
                                                                         8 * t4 + 4 * sg) * 2);
                                            float d[4];
                                            mma_f16_z(d, a0, a1, a2, a3, xv.x, xv.y);
                                            tf[s][0] = fmaf(e0, d[0] + d[1], tf[s][0]);
                                            tf[s][1] = fmaf(e1, d[2] + d[3], tf[s][1]);
                                        }
                                    }
                                }
                            }
#pragma unroll
                        for (int s = 0; s < NB; ++s) {
                            if (AM == A_F32) {
                                const float io = asc[u * p.sstride + ar[s]];  // 2^-s of (activation row, super-block)
                                acc[s][0][0] = fmaf(io, tf[s][0], acc[s][0][0]);
                                acc[s][1][0] = fmaf(io, tf[s][1], acc[s][1][0]);
                            } else if (EPI == E_Y) {
                                const float2 dv = *reinterpret_cast<const float2*>(asc + u * p.sstride + 8 * s + 2 * t4);
                                acc[s][0][0] = fmaf(dv.x, fD0 * (float)ssc[s][0], acc[s][0][0]);
                                acc[s][0][1] = fmaf(dv.y, fD0 * (float)ssc[s][1], acc[s][0][1]);
                                acc[s][1][0] = fmaf(dv.x, fD1 * (float)ssc[s][2], acc[s][1][0]);
                                acc[s][1][1] = fmaf(dv.y, fD1 * (float)ssc[s][3], acc[s][1][1]);
                            } else {
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const int m = 8 * s + 2 * t4 + (i & 1);
                                    const long long n = (long long)grp * kDmmaRows + g8 + 8 * (i >> 1);
                                    if (m < p.M && n < p.N) p.sums[((long long)m * p.N + n) * p.units + su0 + u] = ssc[s][i];
                                }
                            }
                        }
                    }
                } else {
                    const uint8_t* h0p = r0p + 144 * warp;
                    int u = u0;
#pragma unroll 1
                    for (int uu = warp; uu < cnu; uu += kDmmaWarps, u += kDmmaWarps, h0p += kDmmaWarps * 144) {
                        const uint8_t* h1p = h0p + dr;
                        const uint4 h0 = ld128(h0p), h1 = ld128(h1p);
                        uint32_t sc03[2], sc47[2], mn03[2], mn47[2];
                        q4k_unpack4(h0.y, h0.z, h0.w, sc03[0], sc47[0], mn03[0], mn47[0]);
                        q4k_unpack4(h1.y, h1.z, h1.w, sc03[1], sc47[1], mn03[1], mn47[1]);
                        if (AM == A_F32) {
                            float d[NB][4];
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                // per row: P = (sc_{2c}, sc_{2c+1}/16), Q = (-1024 sc_{2c}, -64 sc_{2c+1})
                                const uint32_t sel = (uint32_t)((2 * (c & 1)) | 0x40 | ((2 * (c & 1) + 1) << 8) | 0x5000);
                                __half2 P[2], Q[2];
#pragma unroll
                                for (int r = 0; r < 2; ++r) {
                                    P[r] = __hsub2(u2h(__byte_perm(c < 2 ? sc03[r] : sc47[r], 0x00005464u, sel)), u2h(0x54006400u));
                                    Q[r] = __hmul2(P[r], u2h(0xE400E400u));
                                }
                                const uint32_t qa0 = ld32(h0p + 16 + 32 * c + 4 * t4), qb0 = ld32(h0p + 32 + 32 * c + 4 * t4);
                                const uint32_t qa1 = ld32(h1p + 16 + 32 * c + 4 * t4), qb1 = ld32(h1p + 32 + 32 * c + 4 * t4);
                                const uint32_t qa0s = qa0 >> 8, qb0s = qb0 >> 8, qa1s = qa1 >> 8, qb1s = qb1 >> 8;
#pragma unroll
                                for (int h = 0; h < 2; ++h) {
                                    // low nibbles (sub-block 2c): 1024 + n; high nibbles (2c+1): 1024 + 16 n
                                    const uint32_t mk = h ? kM00F0 : kM000F;
                                    const __half2 S0 = h ? __high2half2(P[0]) : __low2half2(P[0]);
                                    const __half2 N0 = h ? __high2half2(Q[0]) : __low2half2(Q[0]);
                                    const __half2 S1 = h ? __high2half2(P[1]) : __low2half2(P[1]);
                                    const __half2 N1 = h ? __high2half2(Q[1]) : __low2half2(Q[1]);
                                    const uint32_t a0 = h2u(__hfma2(u2h(and_or(qa0, mk, k6400)), S0, N0));
                                    const uint32_t a1 = h2u(__hfma2(u2h(and_or(qa1, mk, k6400)), S1, N1));
                                    const uint32_t a2 = h2u(__hfma2(u2h(and_or(qa0s, mk, k6400)), S0, N0));
                                    const uint32_t a3 = h2u(__hfma2(u2h(and_or(qa1s, mk, k6400)), S1, N1));
                                    const uint32_t c0 = h2u(__hfma2(u2h(and_or(qb0, mk, k6400)), S0, N0));
                                    const uint32_t c1 = h2u(__hfma2(u2h(and_or(qb1, mk, k6400)), S1, N1));
                                    const uint32_t c2 = h2u(__hfma2(u2h(and_or(qb0s, mk, k6400)), S0, N0));
                                    const uint32_t c3 = h2u(__hfma2(u2h(and_or(qb1s, mk, k6400)), S1, N1));
                                    const int j = 2 * c + h;
#pragma unroll
                                    for (int s = 0; s < NB; ++s) {
                                        const uint4 xv = ld128(act + (long long)bc[s] * p.act_pitch * 2 + ((u * 8 + j) * 32 + 8 * t4) * 2);
                                        if (j == 0) mma_f16_z(d[s], a0, a1, a2, a3, xv.x, xv.y);
                                        else mma_f16(d[s], a0, a1, a2, a3, xv.x, xv.y);
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
                                float dm[4];
                                mma_f16_k8(dm, ma0, ma1, aux[(u * p.xplanes + bc[s]) * 4 + t4]);
                                const float io = asc[u * p.sstride + ar[s]];  // 2^-s of (activation row, super-block)
                                acc[s][0][0] = fmaf(io, fD0 * (d[s][0] + d[s][1]) - fM0 * (dm[0] + dm[1]), acc[s][0][0]);
                                acc[s][1][0] = fmaf(io, fD1 * (d[s][2] + d[s][3]) - fM1 * (dm[2] + dm[3]), acc[s][1][0]);
                            }
                        } else {
                            // S_sc: low nibbles as they are, high nibbles as 16 n (their sums are then
                            // multiples of 16 and are divided back exactly at the end); one set of
                            // sums per column set (8 activation rows each)
                            int sl[NB][4], shi[NB][4];
                            const uint8_t* xb[NB];
#pragma unroll
                            for (int s = 0; s < NB; ++s) {
                                xb[s] = act + bc[s] * p.act_pitch + u * 256 + 4 * t4;
#pragma unroll
                                for (int i = 0; i < 4; ++i) sl[s][i] = shi[s][i] = 0;
                            }
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                const uint32_t qa0 = ld32(h0p + 16 + 32 * c + 4 * t4), qb0 = ld32(h0p + 32 + 32 * c + 4 * t4);
                                const uint32_t qa1 = ld32(h1p + 16 + 32 * c + 4 * t4), qb1 = ld32(h1p + 32 + 32 * c + 4 * t4);
#pragma unroll
                                for (int h = 0; h < 2; ++h) {
                                    const int j = 2 * c + h;
                                    const uint32_t mk = h ? 0xF0F0F0F0u : 0x0F0F0F0Fu;
                                    const uint32_t selj = 0x4440u | (uint32_t)(j & 3);
                                    const int sc0 = (int)__byte_perm(j < 4 ? sc03[0] : sc47[0], 0, selj);
                                    const int sc1 = (int)__byte_perm(j < 4 ? sc03[1] : sc47[1], 0, selj);
#pragma unroll
                                    for (int s = 0; s < NB; ++s) {
                                        int dj[4];
                                        mma_u8s8(dj, qa0 & mk, qa1 & mk, qb0 & mk, qb1 & mk, ld32(xb[s] + 32 * j),
                                                 ld32(xb[s] + 32 * j + 16));
                                        int* t = h ? shi[s] : sl[s];
                                        t[0] += sc0 * dj[0];
                                        t[1] += sc0 * dj[1];
                                        t[2] += sc1 * dj[2];
                                        t[3] += sc1 * dj[3];
                                    }
                                }
                            }
                            // S_m = sum_j m_j (sum of the sub-block's 32 codes), as 16 slots of sums of 16
                            const uint32_t ma0 = h2_sub(__byte_perm(mn03[0], 0x64646464u, sel_m1), 0x64006400u);
                            const uint32_t ma1 = h2_sub(__byte_perm(mn03[1], 0x64646464u, sel_m1), 0x64006400u);
                            const uint32_t ma2 = h2_sub(__byte_perm(mn47[0], 0x64646464u, sel_m1), 0x64006400u);
                            const uint32_t ma3 = h2_sub(__byte_perm(mn47[1], 0x64646464u, sel_m1), 0x64006400u);
#pragma unroll
                            for (int s = 0; s < NB; ++s) {
                                int ssc[4];
#pragma unroll
                                for (int i = 0; i < 4; ++i) ssc[i] = sl[s][i] + (shi[s][i] >> 4);
                                float sm[4];
                                mma_f16_z(sm, ma0, ma1, ma2, ma3, aux[(u * 8 + t4) * p.sstride + bc[s]],
                                          aux[(u * 8 + t4 + 4) * p.sstride + bc[s]]);
                                if (EPI == E_Y) {
                                    const float2 dv = *reinterpret_cast<const float2*>(asc + u * p.sstride + 8 * s + 2 * t4);
                                    const float fD0 = h2f(h0.x), fD1 = h2f(h1.x), fM0 = h2f(h0.x >> 16), fM1 = h2f(h1.x >> 16);
                                    acc[s][0][0] = fmaf(dv.x, fD0 * (float)ssc[0] - fM0 * sm[0], acc[s][0][0]);
                                    acc[s][0][1] = fmaf(dv.y, fD0 * (float)ssc[1] - fM0 * sm[1], acc[s][0][1]);
                                    acc[s][1][0] = fmaf(dv.x, fD1 * (float)ssc[2] - fM1 * sm[2], acc[s][1][0]);
                                    acc[s][1][1] = fmaf(dv.y, fD1 * (float)ssc[3] - fM1 * sm[3], acc[s][1][1]);
                                } else {
#pragma unroll
                                    for (int i = 0; i < 4; ++i) {
                                        const int m = 8 * s + 2 * t4 + (i & 1);
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
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars[S + slot]));
        }
        if (EPI != E_Y) continue;
        // ---- tile partials of (weight row, activation row) to the reducer;
        // its buffer is free once the reducer has read the previous tile
        if (tc >= 1) mbar_wait(smem_u32(rempty), (uint32_t)((tc - 1) & 1), flags, p.err);
        float* rb = red + warp * kDmmaRows * RW;
        if (AM == A_F32) {
#pragma unroll
            for (int s = 0; s < NB; ++s) {
                rb[g8 * RW + t4 + 4 * s] = acc[s][0][0];
                rb[(g8 + 8) * RW + t4 + 4 * s] = acc[s][1][0];
            }
        } else {
#pragma unroll
            for (int s = 0; s < NB; ++s) {
                *reinterpret_cast<float2*>(rb + g8 * RW + 8 * s + 2 * t4) = make_float2(acc[s][0][0], acc[s][0][1]);
                *reinterpret_cast<float2*>(rb + (g8 + 8) * RW + 8 * s + 2 * t4) = make_float2(acc[s][1][0], acc[s][1][1]);
            }
        }
        mbar_arrive(smem_u32(rfull));
    }
}

// ---------------------------------------------------------------------------
// host-side planning
// ---------------------------------------------------------------------------

struct DmmaPlan {
    DmmaParams p;
    int nb;   // B column sets: int8 1 (M <= 8) or 2; f32 1 (M <= 4), 2 (M <= 8) or 4
    int grid;
    size_t smem;
    size_t workspace;  // ext_bytes + split-K partial sums
    size_t ext_bytes;  // prepared activations (0: prepared inside the decode kernel)
};

// Weight matrices at least this large prepare the activations once per call
// (a second, small launch) when the batch has more than a few rows; smaller
// ones, bound by launch latency, prepare them inside the single decode launch.
constexpr long long kDmmaExtMinBytes = 32ll << 20;

// The planner first looks for a chunk size that leaves this many stages.
constexpr int kDmmaPreferStages = 2;

// Shared-memory layout for K split in `ks` slices and `ups` units per stage;
// false when fewer than two stages fit.
inline bool dmma_layout(int wt, int am, long long M, int nb, int ks, int ups, int smem_max, DmmaPlan& pl,
                        int min_stages = 2) {
    DmmaParams& p = pl.p;
    const int uv = is_b32(wt) ? 32 : 256, ub = unit_bytes(wt);
    const int su = (p.units + ks - 1) / ks;
    if ((long long)(ks - 1) * su >= p.units) return false;
    if (ups > su) ups = su;
    const int kv = su * uv;
    int act, aux = 0;
    if (am == A_INT8) {
        p.act_pitch = pitch_mod(kv, 16);  // 4-byte B loads of 8 rows x 4 threads: 32 banks
        act = (int)M * p.act_pitch;
        p.sstride = 8 * nb;
        p.xplanes = 0;
        p.aux_unit = 8 * p.sstride * 4;  // Q4_K: [8 pairs of sums of 16][rows] f16x2
        if (wt == T_Q4_K) aux = su * p.aux_unit;
    } else {
        p.act_pitch = pitch_mod(2 * kv, 64) / 2;  // 16-byte B loads of 2 planes per quarter-warp
        act = 2 * (int)M * p.act_pitch * 2;
        p.sstride = 4 * nb;
        p.xplanes = 8 * nb > 16 ? 8 * nb : 16;
        p.aux_unit = p.xplanes * 8 * 2;  // Q4_K: [planes][8 sums of 32] halves
        if (wt == T_Q4_K) aux = su * p.aux_unit;
    }
    const int scale = su * p.sstride * 4;
    int off = 256;  // mbarriers: 2 per stage (<= 8 stages), 2 for the reducer, 1 for the activations
    p.off_flags = off;
    off += 128;
    p.off_act = off;
    off = round_up(off + act, 128);
    p.off_scale = off;
    off = round_up(off + scale, 128);
    p.off_aux = off;
    off = round_up(off + aux, 128);
    p.off_red = off;
    off = round_up(off + kDmmaWarps * kDmmaRows * dmma_red_cols(am, nb) * 4, 128);
    p.off_stage = off;
    long long sb;
    if (ks == 1 && ups == su && 16 * p.rb <= 36864) {
        sb = 16 * p.rb + 64;  // short rows: one contiguous copy of the whole tile
        p.row_pitch = 0;
    } else {
        // Q8_0 word loads reach 18 bytes past the chunk (2-byte offset
        // rounding and the 9th word); a copy starts up to 15 bytes early
        p.row_pitch = pitch_mod(ups * ub + (is_b32(wt) || wt == T_Q6_K ? 32 : 0), 16);
        sb = 16LL * p.row_pitch;
    }
    sb = (sb + 127) / 128 * 128;
    const long long stages = (smem_max - off) / sb;
    if (stages < min_stages) return false;
    p.kslices = ks;
    p.slice_units = su;
    p.ups = ups;
    p.stages = stages > 8 ? 8 : (int)stages;
    p.stage_bytes = (int)sb;
    pl.smem = (size_t)off + (size_t)p.stages * sb;
    return true;
}

inline bool plan_dmma(int wt, int am, long long M, long long N, long long K, int sm_count, int smem_max,
                      DmmaPlan& out, bool ext_ok = true) {
    if (M < 1 || M > kDmmaMaxM) return false;
    DmmaPlan pl{};
    DmmaParams& p = pl.p;
    const int uv = is_b32(wt) ? 32 : 256, ub = unit_bytes(wt);
    p.M = (int)M;
    p.N = (int)N;
    p.K = (int)K;
    p.units = (int)(K / uv);
    p.rb = (long long)p.units * ub;
    p.total_bytes = p.rb * N;
    p.ntiles = (int)((N + kDmmaRows - 1) / kDmmaRows);
    // B column sets: 8 activation rows each (int8), or 4 rows of two pieces (f32)
    pl.nb = am == A_INT8 ? (M > 8 ? 2 : 1) : (M > 8 ? 4 : M > 4 ? 2 : 1);
    // K chunk per stage.  One SM's bulk-copy engine caps row copies below
    // ~3 KB, so the first tier takes the fewest K slices that fit a chunk of
    // >= 96 Q8_0 blocks (32 super-blocks; a shorter K as one chunk, unsplit),
    // chunks that divide the slice first (the 16 warps of a stage stay busy);
    // the second tier allows smaller chunks, again with the fewest slices.
    // (Q4_0 and Q5_0 blocks are shorter: their chunks hold more blocks for about the same bytes)
    const int cq[5] = {128, 112, 96, 80, 64}, c4[5] = {256, 224, 192, 160, 128}, c5[5] = {256, 192, 128, 96, 64},
              ck[2] = {32, 16};
    const int* cand = wt == T_Q8_0 ? cq : wt == T_Q4_0 ? c4 : wt == T_Q5_0 ? c5 : ck;
    const int nbig = is_b32(wt) ? 3 : 1, ncand = is_b32(wt) ? 5 : 2;
    const int minbig = cand[nbig - 1];
    bool found = false;
    for (int minst = kDmmaPreferStages; minst >= 2 && !found; --minst)
        for (int ks = 1; ks <= 16 && !found; ++ks) {
            const int su = (p.units + ks - 1) / ks;
            if (ks > 1 && 3 * su < 2 * minbig) break;  // slices too short for a full chunk
            for (int pass = 0; pass < 2 && !found; ++pass)
                for (int i = 0; i < nbig && !found; ++i) {
                    const int u = cand[i] < su ? cand[i] : su;
                    if ((su % u == 0) == (pass == 0)) found = dmma_layout(wt, am, M, pl.nb, ks, u, smem_max, pl, minst);
                }
        }
    for (int ks = 1; ks <= 16 && !found; ++ks) {
        const int su = (p.units + ks - 1) / ks;
        for (int i = nbig; i < ncand && !found; ++i) {
            const int u = cand[i] < su ? cand[i] : su;
            if (su % u == 0) found = dmma_layout(wt, am, M, pl.nb, ks, u, smem_max, pl);
        }
    }
    if (!found) return false;
    int per = sm_count / p.kslices;
    if (per < 1) per = 1;
    if (per > p.ntiles) per = p.ntiles;
    p.per_slice = per;
    pl.grid = per * p.kslices;
    pl.ext_bytes = 0;
    // Large weights with more than a few activation rows: prepare the activations once per
    // call in their own launch.  Up to 2 rows (4 for 32-value blocks) every CTA prepares its
    // own slice from x (a few KB, hot in L2): measured faster on 28672 x 8192, since the
    // separate launch would sit between the previous call's grid and this one's consumers.
    if (ext_ok && p.total_bytes >= kDmmaExtMinBytes && M > (is_b32(wt) ? 4 : 2)) {
        auto r256 = [](long long v) { return (v + 255) / 256 * 256; };
        p.ext_codes = 0;
        long long off = r256(am == A_INT8 ? M * K : 2 * M * K * 2);
        p.ext_scale = off;
        off = r256(off + (long long)p.units * p.sstride * 4);
        p.ext_aux = off;
        if (wt == T_Q4_K) off = r256(off + (long long)p.units * p.aux_unit);
        pl.ext_bytes = (size_t)off;
    }
    pl.workspace = pl.ext_bytes + (p.kslices > 1 ? (size_t)p.kslices * M * N * 4 : 0);
    out = pl;
    return true;
}

}  // namespace qmm
