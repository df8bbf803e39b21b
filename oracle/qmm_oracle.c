/*
 * qmm_oracle.c -- plain, slow CPU oracle for GGUF block-quantized matmul.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link,
 * import or execute this file: only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py use it.  It shares no code, no
 * header and no constant table with the CUDA library; the two are written
 * independently from the same definitions and compared on the same inputs.
 *
 * Sources (page titles and sections of the candle tutorial pages):
 *  [p1] "同一个 GGUF，CPU 和 Metal 生成的文字不一样", section 出处: the CPU
 *       quantized matmul first quantizes every activation row to Q8_0 (for
 *       Q8_0/Q4_0/Q5_0 weights) or Q8K (for K-quants) and then takes integer
 *       block dot products; the Metal kernel multiplies f32 activations by
 *       weight blocks dequantized inside the kernel.  CANDLE_DEQUANTIZE_ALL
 *       dequantizes every weight to f32 and uses a plain f32 matmul.
 *  [p3] "自己量化", sections 3 (量化) and 和下载的 Q8_0 逐字节比: a Q8_0 block
 *       holds 32 values and its scale is max|x|/127 with no freedom of choice;
 *       K-quants need the last dimension divisible by 256; blocks run along a
 *       row; activations are quantized row by row in groups of 32 (Q8_0) or
 *       256 (Q8K) (动脑筋答案).  Section 大小和误差 prints the file sizes that
 *       pin the bytes per block (34 B per 32 values for Q8_0, 144 B per 256
 *       for Q4K).
 *  Block field layouts (f16 d / int8 codes; f16 d, f16 dmin, 12 bytes of
 *  6-bit sub-block scales and mins, 128 bytes of 4-bit codes; f32 d, int8
 *  codes, 16 int16 sums of 16 codes) follow the public GGUF layout.
 *
 * Readings where the pages are silent: Q4_0, Q5_0 and Q6_K use the public GGUF block layouts and the
 * signed-max quantizers written below; rounding of codes is round-half-away-from-zero (C roundf); codes of
 * Q8_0/Q8K use the f32 scale d and the reciprocal 1/d; Q8K is symmetric
 * (+-127); Q4_K uses the closed-form min/max quantizer written below; the
 * dequantized Q4_K weight is (f(d)*sc)*q - f(dmin)*m with each product exact
 * in f32 and one rounding in the subtraction.
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp -shared -fPIC (no -ffast-math):
 * every float operation is a single IEEE-754 binary32 operation in program
 * order, on x86-64 and on aarch64 alike.
 *
 * Parity pins: every function here is checked by tests/test_oracle_pins.py
 * against facts fixed by the pages or by mathematics (sizes, scale rule,
 * exhaustive f16 conversion, brute-force integer sums, round-trip bounds,
 * closed forms, row-permutation and batch invariance, the activation-
 * quantization error scale).  The code choices of the Q4_K, Q4_0, Q5_0 and
 * Q6_K quantizers themselves have no external pin ("parity unpinned" beyond
 * the round-trip bounds, closed forms and the oracle-vs-GPU bit-exact
 * comparison): the pages give neither the algorithms nor these layouts.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* type ids used only inside the oracle and its Python wrapper */
enum { ORC_Q8_0 = 1, ORC_Q4_K = 2, ORC_Q8_K = 3, ORC_Q4_0 = 4, ORC_Q5_0 = 5, ORC_Q6_K = 6 };

/* bytes of one block and values per block (page [p3] sizes; GGUF layout) */
#define ORC_Q8_0_VALS 32
#define ORC_Q8_0_BYTES 34
#define ORC_QK_VALS 256
#define ORC_Q4_K_BYTES 144
#define ORC_Q8_K_BYTES 292
#define ORC_Q4_0_BYTES 18   /* page [p3] file sizes: Q4_0 18 B per 32 values */
#define ORC_Q5_0_BYTES 22   /* Q5_0 22 B per 32 values */
#define ORC_Q6_K_BYTES 210  /* the downloaded Q4_K_M file closes with Q6K at 210 B per 256 values */

/* ------------------------------------------------------------------ */
/* IEEE-754 binary16 <-> binary32, written from the format definition  */
/* ------------------------------------------------------------------ */

static uint32_t f2u(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float u2f(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* binary32 -> binary16, round to nearest, ties to even, with subnormals. */
uint16_t orc_f32_to_f16(float f) {
    uint32_t b = f2u(f);
    uint16_t sign = (uint16_t)((b >> 16) & 0x8000u);
    uint32_t a = b & 0x7fffffffu;
    if (a >= 0x7f800000u) {                       /* Inf or NaN */
        if (a == 0x7f800000u) return sign | 0x7c00u;
        return (uint16_t)(sign | 0x7c00u | 0x0200u | ((a >> 13) & 0x03ffu));
    }
    /* 65520 = largest half (65504) + half an ulp (16): ties go to the even
       neighbour, which is 2^16, i.e. overflow to infinity. */
    if (a >= 0x477ff000u) return sign | 0x7c00u;
    int e = (int)(a >> 23) - 127;                 /* unbiased exponent */
    uint32_t mant = a & 0x007fffffu;
    if (e >= -14) {                               /* normal half */
        uint32_t h = ((uint32_t)(e + 15) << 10) | (mant >> 13);
        uint32_t rem = mant & 0x1fffu;
        if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h += 1u; /* carry may bump the exponent: still correct */
        return (uint16_t)(sign | h);
    }
    if (a == 0) return sign;
    /* subnormal half: value = m * 2^(e-23) with m the 24-bit significand
       (or the 23-bit one for a binary32 subnormal input); the half unit is
       2^-24, so the half integer is m * 2^(e+1) = m >> (-(e+1)). */
    uint64_t m;
    int shift;
    if ((a >> 23) == 0) {                          /* binary32 subnormal: mant * 2^-149 */
        m = mant;
        shift = 125;                               /* 2^-149 / 2^-24 */
    } else {
        m = (uint64_t)(mant | 0x00800000u);
        shift = -(e + 1);
    }
    if (shift > 62) return sign;                   /* far below half the smallest subnormal */
    uint64_t q = m >> shift;
    uint64_t rem = m & ((1ull << shift) - 1ull);
    uint64_t half = 1ull << (shift - 1);
    if (rem > half || (rem == half && (q & 1ull))) q += 1ull;  /* may reach 0x400 = min normal: correct */
    return (uint16_t)(sign | (uint16_t)q);
}

/* binary16 -> binary32 (exact). */
float orc_f16_to_f32(uint16_t h) {
    uint32_t sign = ((uint32_t)h & 0x8000u) << 16;
    uint32_t ex = ((uint32_t)h >> 10) & 0x1fu;
    uint32_t mant = (uint32_t)h & 0x03ffu;
    if (ex == 0x1fu) return u2f(sign | 0x7f800000u | (mant << 13));
    if (ex == 0) {
        /* subnormal or zero: mant * 2^-24, computed exactly in float */
        float v = (float)mant * u2f(0x33800000u);  /* 2^-24 */
        return sign ? -v : v;
    }
    return u2f(sign | ((ex - 15u + 127u) << 23) | (mant << 13));
}

void orc_f32_to_f16_array(const float* x, int64_t n, uint16_t* out) {
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_f16(x[i]);
}

void orc_f16_to_f32_array(const uint16_t* h, int64_t n, float* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f16_to_f32(h[i]);
}

/* Exhaustive self-check helper: converts the 2^32 bit patterns from lo to hi
   (exclusive) and compares with the compiler's _Float16 conversion, which is
   an independent implementation.  Returns the number of mismatches (NaN
   payloads are compared as "both NaN"). */
int64_t orc_f16_check_range(uint64_t lo, uint64_t hi) {
    int64_t bad = 0;
    #pragma omp parallel for schedule(static) reduction(+:bad)
    for (int64_t i = (int64_t)lo; i < (int64_t)hi; ++i) {
        float f = u2f((uint32_t)i);
        uint16_t mine = orc_f32_to_f16(f);
        _Float16 ref = (_Float16)f;
        uint16_t rb; memcpy(&rb, &ref, 2);
        int mine_nan = ((mine & 0x7c00u) == 0x7c00u) && (mine & 0x03ffu);
        int ref_nan = ((rb & 0x7c00u) == 0x7c00u) && (rb & 0x03ffu);
        if (mine_nan || ref_nan) { if (mine_nan != ref_nan) ++bad; }
        else if (mine != rb) ++bad;
    }
    return bad;
}

/* ------------------------------------------------------------------ */
/* block sizes                                                          */
/* ------------------------------------------------------------------ */

int64_t orc_block_values(int t) {
    return (t == ORC_Q8_0 || t == ORC_Q4_0 || t == ORC_Q5_0) ? 32
           : (t == ORC_Q4_K || t == ORC_Q8_K || t == ORC_Q6_K) ? ORC_QK_VALS : 0;
}

int64_t orc_block_bytes(int t) {
    switch (t) {
        case ORC_Q8_0: return ORC_Q8_0_BYTES;
        case ORC_Q4_K: return ORC_Q4_K_BYTES;
        case ORC_Q8_K: return ORC_Q8_K_BYTES;
        case ORC_Q4_0: return ORC_Q4_0_BYTES;
        case ORC_Q5_0: return ORC_Q5_0_BYTES;
        case ORC_Q6_K: return ORC_Q6_K_BYTES;
        default: return 0;
    }
}

static void put_u16(uint8_t* p, uint16_t v) { p[0] = (uint8_t)(v & 0xff); p[1] = (uint8_t)(v >> 8); }
static uint16_t get_u16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static void put_f32(uint8_t* p, float f) { uint32_t u = f2u(f); p[0] = u & 0xff; p[1] = (u >> 8) & 0xff; p[2] = (u >> 16) & 0xff; p[3] = u >> 24; }
static float get_f32(const uint8_t* p) { return u2f((uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24)); }

/* ------------------------------------------------------------------ */
/* Q8_0: 32 values, f16 d = max|x|/127, int8 codes  ([p3] section 3)    */
/* ------------------------------------------------------------------ */

static void q8_0_block(const float* x, uint8_t* out) {
    float amax = 0.0f;
    for (int i = 0; i < 32; ++i) { float a = fabsf(x[i]); if (a > amax) amax = a; }
    float d = amax / 127.0f;
    float id = d != 0.0f ? 1.0f / d : 0.0f;
    put_u16(out, orc_f32_to_f16(d));
    for (int i = 0; i < 32; ++i) {
        float v = x[i] * id;
        float r = roundf(v);
        if (r != r) r = 0.0f;  /* 0 * inf: a zero in a block whose reciprocal overflows; x/d = 0 */
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        out[2 + i] = (uint8_t)(int8_t)(int)r;
    }
}

void orc_quantize_q8_0(const float* x, int64_t rows, int64_t K, uint8_t* out) {
    int64_t nb = K / 32;
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb; ++b)
            q8_0_block(x + r * K + b * 32, out + (r * nb + b) * ORC_Q8_0_BYTES);
}

/* ------------------------------------------------------------------ */
/* Q8K: 256 values, f32 d = max|x|/127, int8 codes, 16 int16 sums       */
/* ------------------------------------------------------------------ */

static void q8_k_block(const float* x, uint8_t* out) {
    float amax = 0.0f;
    for (int i = 0; i < 256; ++i) { float a = fabsf(x[i]); if (a > amax) amax = a; }
    float d = amax / 127.0f;
    float id = d != 0.0f ? 1.0f / d : 0.0f;
    put_f32(out, d);
    int8_t q[256];
    for (int i = 0; i < 256; ++i) {
        float r = roundf(x[i] * id);
        if (r != r) r = 0.0f;  /* 0 * inf: a zero in a block whose reciprocal overflows; x/d = 0 */
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        q[i] = (int8_t)(int)r;
        out[4 + i] = (uint8_t)q[i];
    }
    for (int j = 0; j < 16; ++j) {
        int s = 0;
        for (int i = 0; i < 16; ++i) s += q[16 * j + i];
        put_u16(out + 4 + 256 + 2 * j, (uint16_t)(int16_t)s);
    }
}

void orc_quantize_q8_k(const float* x, int64_t rows, int64_t K, uint8_t* out) {
    int64_t nb = K / 256;
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb; ++b)
            q8_k_block(x + r * K + b * 256, out + (r * nb + b) * ORC_Q8_K_BYTES);
}

/* ------------------------------------------------------------------ */
/* Q4_0 / Q5_0: 32 values, f16 d, 4- or 5-bit codes with an offset      */
/* ([p1] 出处: these weights pair with Q8_0 activations; [p3] 大小和误差: */
/* 18 and 22 bytes per 32 values).  The pages give neither the layout   */
/* nor the quantizer.  Layout (public GGUF): bytes 0-1 f16 d; Q5_0 then  */
/* 4 bytes whose little-endian word holds bit 4 of code i at bit i;     */
/* then 16 bytes, byte j = code j (low nibble) | code j + 16 (high).    */
/* Quantizer (a reading): with off = 8 (Q4_0) or 16 (Q5_0), the value  */
/* m of largest magnitude (the first on ties, sign kept) gives          */
/* d = m / -off, so m maps to code 0 and the signed grid -off..off-1 is */
/* used in full; code = roundf(x * (1/d)) + off, clamped to             */
/* [0, 2 off - 1]; the weight is f(d) * (code - off).                   */
/* ------------------------------------------------------------------ */

static void x_0_block(const float* x, int off, uint8_t* out) {
    float amax = 0.0f, m = 0.0f;
    for (int i = 0; i < 32; ++i) {
        float a = fabsf(x[i]);
        if (a > amax) { amax = a; m = x[i]; }
    }
    float d = m / (float)(-off);
    float id = d != 0.0f ? 1.0f / d : 0.0f;
    put_u16(out, orc_f32_to_f16(d));
    int c[32];
    for (int i = 0; i < 32; ++i) {
        float t = roundf(x[i] * id);
        if (t != t) t = 0.0f;  /* 0 * inf: a zero in a block whose reciprocal overflows; x/d = 0 */
        float r = t + (float)off;
        if (r < 0.0f) r = 0.0f;
        if (r > (float)(2 * off - 1)) r = (float)(2 * off - 1);
        c[i] = (int)r;
    }
    uint8_t* qs = out + 2;
    if (off == 16) {
        uint32_t h = 0;
        for (int i = 0; i < 32; ++i) h |= (uint32_t)((c[i] >> 4) & 1) << i;
        out[2] = (uint8_t)(h & 0xff);
        out[3] = (uint8_t)((h >> 8) & 0xff);
        out[4] = (uint8_t)((h >> 16) & 0xff);
        out[5] = (uint8_t)(h >> 24);
        qs = out + 6;
    }
    for (int j = 0; j < 16; ++j) qs[j] = (uint8_t)((c[j] & 15) | ((c[j + 16] & 15) << 4));
}

static void quantize_x_0(const float* x, int64_t rows, int64_t K, int off, int bytes, uint8_t* out) {
    int64_t nb = K / 32;
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb; ++b) x_0_block(x + r * K + b * 32, off, out + (r * nb + b) * bytes);
}

void orc_quantize_q4_0(const float* x, int64_t rows, int64_t K, uint8_t* out) { quantize_x_0(x, rows, K, 8, ORC_Q4_0_BYTES, out); }
void orc_quantize_q5_0(const float* x, int64_t rows, int64_t K, uint8_t* out) { quantize_x_0(x, rows, K, 16, ORC_Q5_0_BYTES, out); }

/* signed codes (code - off) of a Q4_0 / Q5_0 block */
static void x_0_codes(int t, const uint8_t* blk, int c[32]) {
    const int off = t == ORC_Q5_0 ? 16 : 8;
    const uint8_t* qs = blk + (t == ORC_Q5_0 ? 6 : 2);
    uint32_t h = 0;
    if (t == ORC_Q5_0) h = (uint32_t)blk[2] | ((uint32_t)blk[3] << 8) | ((uint32_t)blk[4] << 16) | ((uint32_t)blk[5] << 24);
    for (int j = 0; j < 16; ++j) {
        c[j] = ((qs[j] & 15) | (int)(((h >> j) & 1) << 4)) - off;
        c[j + 16] = ((qs[j] >> 4) | (int)(((h >> (j + 16)) & 1) << 4)) - off;
    }
}

/* signed codes of any 32-value weight block (Q8_0, Q4_0, Q5_0) */
static void b32_codes(int t, const uint8_t* blk, int c[32]) {
    if (t == ORC_Q8_0) {
        for (int i = 0; i < 32; ++i) c[i] = (int8_t)blk[2 + i];
    } else {
        x_0_codes(t, blk, c);
    }
}

/* ------------------------------------------------------------------ */
/* Q4_K: 256 values = 8 sub-blocks of 32.                               */
/*   bytes 0-1 f16 d, 2-3 f16 dmin, 4-15 packed 6-bit (sc, m) x 8,      */
/*   16-143 4-bit codes: byte 16+32c+l = sub-block 2c value l (low       */
/*   nibble) | sub-block 2c+1 value l (high nibble).                     */
/*   6-bit packing: byte j (j<4) low 6 bits = sc_j, top 2 bits = bits    */
/*   4-5 of sc_{j+4}; byte 4+j low 6 bits = m_j, top 2 bits = bits 4-5   */
/*   of m_{j+4}; byte 8+j low nibble = low 4 bits of sc_{j+4}, high      */
/*   nibble = low 4 bits of m_{j+4}.                                     */
/* ------------------------------------------------------------------ */

static void pack_scales(const int sc[8], const int mn[8], uint8_t s[12]) {
    for (int j = 0; j < 4; ++j) {
        s[j] = (uint8_t)((sc[j] & 63) | ((sc[j + 4] >> 4) << 6));
        s[4 + j] = (uint8_t)((mn[j] & 63) | ((mn[j + 4] >> 4) << 6));
        s[8 + j] = (uint8_t)((sc[j + 4] & 15) | ((mn[j + 4] & 15) << 4));
    }
}

static void unpack_scales(const uint8_t s[12], int sc[8], int mn[8]) {
    for (int j = 0; j < 4; ++j) {
        sc[j] = s[j] & 63;
        mn[j] = s[4 + j] & 63;
        sc[j + 4] = (s[8 + j] & 15) | ((s[j] >> 6) << 4);
        mn[j + 4] = (s[8 + j] >> 4) | ((s[4 + j] >> 6) << 4);
    }
}

static float clampf(float v, float lo, float hi) { return v < lo ? lo : (v > hi ? hi : v); }

/* Closed-form min/max reading of the K-quant scheme: each sub-block j gets
   step s_j = (hi_j - lo_j)/15 with lo_j = min(0, min x), hi_j = max x and
   offset mu_j = -lo_j; the super-block scales are d = max s_j / 63 and
   dmin = max mu_j / 63; the 6-bit factors are the nearest integers
   sc_j = s_j/d, m_j = mu_j/dmin; codes are the nearest integers to
   (x + f(dmin) m_j) / (f(d) sc_j), clamped to [0, 15]. */
static void q4_k_block(const float* x, uint8_t* out) {
    float s[8], mu[8];
    for (int j = 0; j < 8; ++j) {
        float lo = 0.0f, hi = x[32 * j];
        for (int i = 0; i < 32; ++i) {
            float v = x[32 * j + i];
            if (v < lo) lo = v;
            if (v > hi) hi = v;
        }
        s[j] = (hi - lo) / 15.0f;   /* sub-block step */
        mu[j] = 0.0f - lo;          /* sub-block offset (>= 0) */
    }
    float smax = 0.0f, mumax = 0.0f;
    for (int j = 0; j < 8; ++j) { if (s[j] > smax) smax = s[j]; if (mu[j] > mumax) mumax = mu[j]; }
    float d = smax / 63.0f, dmin = mumax / 63.0f;
    int sc[8], mn[8];
    for (int j = 0; j < 8; ++j) {
        sc[j] = d > 0.0f ? (int)clampf(roundf(s[j] / d), 0.0f, 63.0f) : 0;
        mn[j] = dmin > 0.0f ? (int)clampf(roundf(mu[j] / dmin), 0.0f, 63.0f) : 0;
    }
    uint16_t D = orc_f32_to_f16(d), Dm = orc_f32_to_f16(dmin);
    put_u16(out, D);
    put_u16(out + 2, Dm);
    pack_scales(sc, mn, out + 4);
    float fD = orc_f16_to_f32(D), fDm = orc_f16_to_f32(Dm);
    uint8_t q[256];
    for (int j = 0; j < 8; ++j) {
        float e = fD * (float)sc[j];
        float o = fDm * (float)mn[j];
        for (int i = 0; i < 32; ++i) {
            float v = e > 0.0f ? clampf(roundf((x[32 * j + i] + o) / e), 0.0f, 15.0f) : 0.0f;
            q[32 * j + i] = (uint8_t)(int)v;
        }
    }
    for (int c = 0; c < 4; ++c)
        for (int l = 0; l < 32; ++l)
            out[16 + 32 * c + l] = (uint8_t)(q[64 * c + l] | (q[64 * c + 32 + l] << 4));
}

void orc_quantize_q4_k(const float* x, int64_t rows, int64_t K, uint8_t* out) {
    int64_t nb = K / 256;
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb; ++b)
            q4_k_block(x + r * K + b * 256, out + (r * nb + b) * ORC_Q4_K_BYTES);
}

/* unpack helper shared by dequantize and the products */
static void q4_k_codes(const uint8_t* blk, uint8_t q[256]) {
    for (int c = 0; c < 4; ++c)
        for (int l = 0; l < 32; ++l) {
            uint8_t b = blk[16 + 32 * c + l];
            q[64 * c + l] = b & 15;
            q[64 * c + 32 + l] = b >> 4;
        }
}


/* ------------------------------------------------------------------ */
/* Q6_K: 256 values = 16 groups of 16, signed 6-bit codes.               */
/*   bytes 0-127 ql (low 4 bits), 128-191 qh (high 2 bits), 192-207 the */
/*   16 int8 group scales, 208-209 f16 d (the public GGUF field order).  */
/*   Value i: half h = i / 128, w = i % 128, quarter q = w / 32,          */
/*   l = w % 32.  Its low 4 bits are nibble q / 2 (0 low, 1 high) of ql  */
/*   byte 64h + 32 (q % 2) + l; its high 2 bits are bits 2q, 2q+1 of qh  */
/*   byte 32h + l; the code is those 6 bits minus 32.  Group j = i / 16  */
/*   has the scale sc_j.  The weight is (f(d) sc_j) code, exact in f32   */
/*   (an 11-bit by 7-bit product times at most 2^5).                     */
/* Quantizer (a reading, the same signed-max rule as Q4_0 / Q5_0 per     */
/* group): m_j, the group's value of largest magnitude (the first on     */
/* ties, sign kept), gives s_j = m_j / -32; d = max_j |s_j| / 127;        */
/* sc_j = roundf(s_j / d) clamped to [-127, 127] (0 when d = 0); with    */
/* e_j = f(D) sc_j, code = roundf(x / e_j) clamped to [-32, 31] (0 when  */
/* e_j = 0).                                                            */
/* ------------------------------------------------------------------ */

static int q6_k_index_ql(int i) { int h = i / 128, w = i % 128; return 64 * h + 32 * ((w / 32) % 2) + w % 32; }
static int q6_k_shift_ql(int i) { return 4 * ((i % 128) / 64); }
static int q6_k_index_qh(int i) { int h = i / 128, w = i % 128; return 128 + 32 * h + w % 32; }
static int q6_k_shift_qh(int i) { return 2 * ((i % 128) / 32); }

static void q6_k_block(const float* x, uint8_t* out) {
    float s[16];
    for (int j = 0; j < 16; ++j) {
        float amax = 0.0f, m = 0.0f;
        for (int i = 0; i < 16; ++i) {
            float a = fabsf(x[16 * j + i]);
            if (a > amax) { amax = a; m = x[16 * j + i]; }
        }
        s[j] = m / -32.0f;
    }
    float smax = 0.0f;
    for (int j = 0; j < 16; ++j) if (fabsf(s[j]) > smax) smax = fabsf(s[j]);
    float d = smax / 127.0f;
    int sc[16];
    for (int j = 0; j < 16; ++j) sc[j] = d > 0.0f ? (int)clampf(roundf(s[j] / d), -127.0f, 127.0f) : 0;
    uint16_t D = orc_f32_to_f16(d);
    float fD = orc_f16_to_f32(D);
    memset(out, 0, ORC_Q6_K_BYTES);
    for (int j = 0; j < 16; ++j) {
        out[192 + j] = (uint8_t)(int8_t)sc[j];
        float e = fD * (float)sc[j];
        for (int i = 16 * j; i < 16 * j + 16; ++i) {
            int c = e != 0.0f ? (int)clampf(roundf(x[i] / e), -32.0f, 31.0f) : 0;
            int u = c + 32;  /* 0..63 */
            out[q6_k_index_ql(i)] |= (uint8_t)((u & 15) << q6_k_shift_ql(i));
            out[q6_k_index_qh(i)] |= (uint8_t)((u >> 4) << q6_k_shift_qh(i));
        }
    }
    put_u16(out + 208, D);
}

void orc_quantize_q6_k(const float* x, int64_t rows, int64_t K, uint8_t* out) {
    int64_t nb = K / 256;
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb; ++b)
            q6_k_block(x + r * K + b * 256, out + (r * nb + b) * ORC_Q6_K_BYTES);
}

/* the 256 signed codes and the 16 group scales of a Q6_K super-block */
static void q6_k_codes(const uint8_t* blk, int c[256], int sc[16]) {
    for (int i = 0; i < 256; ++i) {
        int lo = (blk[q6_k_index_ql(i)] >> q6_k_shift_ql(i)) & 15;
        int hi = (blk[q6_k_index_qh(i)] >> q6_k_shift_qh(i)) & 3;
        c[i] = (lo | (hi << 4)) - 32;
    }
    for (int j = 0; j < 16; ++j) sc[j] = (int8_t)blk[192 + j];
}

/* ------------------------------------------------------------------ */
/* Dequantize ([p1] CANDLE_DEQUANTIZE_ALL form)                          */
/* ------------------------------------------------------------------ */

static void dequant_row(int t, const uint8_t* q, int64_t K, float* out) {
    if (t == ORC_Q8_0) {
        for (int64_t b = 0; b < K / 32; ++b) {
            const uint8_t* blk = q + b * ORC_Q8_0_BYTES;
            float d = orc_f16_to_f32(get_u16(blk));
            for (int i = 0; i < 32; ++i) out[b * 32 + i] = d * (float)(int8_t)blk[2 + i];
        }
    } else if (t == ORC_Q4_0 || t == ORC_Q5_0) {
        const int64_t bytes = orc_block_bytes(t);
        for (int64_t b = 0; b < K / 32; ++b) {
            const uint8_t* blk = q + b * bytes;
            float d = orc_f16_to_f32(get_u16(blk));
            int c[32];
            x_0_codes(t, blk, c);
            for (int i = 0; i < 32; ++i) out[b * 32 + i] = d * (float)c[i];  /* exact: 11 x 5 bits */
        }
    } else if (t == ORC_Q8_K) {
        for (int64_t b = 0; b < K / 256; ++b) {
            const uint8_t* blk = q + b * ORC_Q8_K_BYTES;
            float d = get_f32(blk);
            for (int i = 0; i < 256; ++i) out[b * 256 + i] = d * (float)(int8_t)blk[4 + i];
        }
    } else if (t == ORC_Q6_K) {
        for (int64_t b = 0; b < K / 256; ++b) {
            const uint8_t* blk = q + b * ORC_Q6_K_BYTES;
            float fD = orc_f16_to_f32(get_u16(blk + 208));
            int c[256], sc[16];
            q6_k_codes(blk, c, sc);
            for (int i = 0; i < 256; ++i) {
                float e = fD * (float)sc[i / 16];     /* exact: 11 x 7 bits */
                out[b * 256 + i] = e * (float)c[i];   /* exact: |c| <= 2^5 */
            }
        }
    } else if (t == ORC_Q4_K) {
        for (int64_t b = 0; b < K / 256; ++b) {
            const uint8_t* blk = q + b * ORC_Q4_K_BYTES;
            float fD = orc_f16_to_f32(get_u16(blk)), fDm = orc_f16_to_f32(get_u16(blk + 2));
            int sc[8], mn[8];
            unpack_scales(blk + 4, sc, mn);
            uint8_t c[256];
            q4_k_codes(blk, c);
            for (int j = 0; j < 8; ++j) {
                float e = fD * (float)sc[j];   /* exact: 11 x 6 bits */
                float o = fDm * (float)mn[j];  /* exact */
                for (int i = 0; i < 32; ++i) {
                    float t1 = e * (float)c[32 * j + i];  /* exact: 17 x 4 bits */
                    out[b * 256 + 32 * j + i] = t1 - o;   /* the one rounding */
                }
            }
        }
    }
}

void orc_dequantize(int t, const uint8_t* q, int64_t rows, int64_t K, float* out) {
    int64_t rb = K / orc_block_values(t) * orc_block_bytes(t);
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) dequant_row(t, q + r * rb, K, out + r * K);
}

/* ------------------------------------------------------------------ */
/* Integer block sums ([p1] 出处: integer dot of quantized activation   */
/* and weight blocks)                                                   */
/*   Q8_0 x Q8_0: out[m][n][b] = sum_{i<32} qw*qa  (int32)              */
/*   Q4_K x Q8K : out[m][n][s][0] = S_sc = sum_j sc_j * sum_{i in j} q*a */
/*                out[m][n][s][1] = S_m  = sum_j m_j * (bsum_2j+bsum_2j+1)*/
/* ------------------------------------------------------------------ */

/* any 32-value weight block (Q8_0, Q4_0, Q5_0) against Q8_0 activations */
static void sums_b32(int t, const uint8_t* wrow, const uint8_t* arow, int64_t nb, int32_t* out) {
    const int64_t wb = orc_block_bytes(t);
    for (int64_t b = 0; b < nb; ++b) {
        const uint8_t* a = arow + b * ORC_Q8_0_BYTES;
        int c[32];
        b32_codes(t, wrow + b * wb, c);
        int32_t s = 0;
        for (int i = 0; i < 32; ++i) s += (int32_t)c[i] * (int32_t)(int8_t)a[2 + i];
        out[b] = s;
    }
}

static void sums_q4_k(const uint8_t* wrow, const uint8_t* arow, int64_t nsb, int32_t* out) {
    for (int64_t s = 0; s < nsb; ++s) {
        const uint8_t* w = wrow + s * ORC_Q4_K_BYTES;
        const uint8_t* a = arow + s * ORC_Q8_K_BYTES;
        int sc[8], mn[8];
        unpack_scales(w + 4, sc, mn);
        uint8_t q[256];
        q4_k_codes(w, q);
        int32_t ssc = 0, sm = 0;
        for (int j = 0; j < 8; ++j) {
            int32_t isum = 0;
            for (int i = 0; i < 32; ++i) isum += (int32_t)q[32 * j + i] * (int32_t)(int8_t)a[4 + 32 * j + i];
            int32_t bs = (int16_t)get_u16(a + 260 + 4 * j) + (int16_t)get_u16(a + 260 + 4 * j + 2);
            ssc += sc[j] * isum;
            sm += mn[j] * bs;
        }
        out[2 * s] = ssc;
        out[2 * s + 1] = sm;
    }
}

/* Q6_K x Q8K: S = sum_j sc_j * sum_{i in group j} code_i * a_i (int32) */
static void sums_q6_k(const uint8_t* wrow, const uint8_t* arow, int64_t nsb, int32_t* out) {
    for (int64_t s = 0; s < nsb; ++s) {
        const uint8_t* w = wrow + s * ORC_Q6_K_BYTES;
        const uint8_t* a = arow + s * ORC_Q8_K_BYTES;
        int c[256], sc[16];
        q6_k_codes(w, c, sc);
        int32_t S = 0;
        for (int j = 0; j < 16; ++j) {
            int32_t isum = 0;
            for (int i = 16 * j; i < 16 * j + 16; ++i) isum += (int32_t)c[i] * (int32_t)(int8_t)a[4 + i];
            S += sc[j] * isum;
        }
        out[s] = S;
    }
}

/* wq: N rows of weight blocks; xq: M rows of activation blocks (Q8_0 for
   Q8_0 / Q4_0 / Q5_0 weights, Q8K for Q4_K and Q6_K weights).  out: int32
   [M][N][nb] (32-value blocks), [M][N][nsb][2] (Q4_K) or [M][N][nsb] (Q6_K). */
void orc_block_sums(int wtype, const uint8_t* wq, const uint8_t* xq, int64_t M, int64_t N, int64_t K, int32_t* out) {
    if (wtype != ORC_Q4_K && wtype != ORC_Q6_K) {
        int64_t nb = K / 32, rbw = nb * orc_block_bytes(wtype), rba = nb * ORC_Q8_0_BYTES;
        #pragma omp parallel for schedule(static) collapse(2)
        for (int64_t m = 0; m < M; ++m)
            for (int64_t n = 0; n < N; ++n)
                sums_b32(wtype, wq + n * rbw, xq + m * rba, nb, out + (m * N + n) * nb);
    } else if (wtype == ORC_Q6_K) {
        int64_t nsb = K / 256, rbw = nsb * ORC_Q6_K_BYTES, rba = nsb * ORC_Q8_K_BYTES;
        #pragma omp parallel for schedule(static) collapse(2)
        for (int64_t m = 0; m < M; ++m)
            for (int64_t n = 0; n < N; ++n)
                sums_q6_k(wq + n * rbw, xq + m * rba, nsb, out + (m * N + n) * nsb);
    } else {
        int64_t nsb = K / 256, rbw = nsb * ORC_Q4_K_BYTES, rba = nsb * ORC_Q8_K_BYTES;
        #pragma omp parallel for schedule(static) collapse(2)
        for (int64_t m = 0; m < M; ++m)
            for (int64_t n = 0; n < N; ++n)
                sums_q4_k(wq + n * rbw, xq + m * rba, nsb, out + (m * N + n) * nsb * 2);
    }
}

/* ------------------------------------------------------------------ */
/* The two QMatMul forms ([p1] 出处), evaluated in double.               */
/*   y[m][n] and the tolerance scale T[m][n] = sum of |scaled terms|.    */
/* ------------------------------------------------------------------ */

/* int8_act ("CPU form"): quantize each activation row (Q8_0 or Q8K),
   integer block sums, then y = sum over blocks of scale products x sums. */
void orc_matmul_int8_act(int wtype, const uint8_t* wq, const float* x, int64_t M, int64_t N, int64_t K,
                         double* y, double* T) {
    if (wtype == ORC_Q6_K) {  /* Q6_K weights with Q8K activations */
        int64_t nsb = K / 256, rbw = nsb * ORC_Q6_K_BYTES, rba = nsb * ORC_Q8_K_BYTES;
        uint8_t* xq = (uint8_t*)malloc((size_t)(M * rba));
        orc_quantize_q8_k(x, M, K, xq);
        #pragma omp parallel for schedule(dynamic, 16) collapse(2)
        for (int64_t m = 0; m < M; ++m)
            for (int64_t n = 0; n < N; ++n) {
                double acc = 0.0, t = 0.0;
                for (int64_t s = 0; s < nsb; ++s) {
                    const uint8_t* w = wq + n * rbw + s * ORC_Q6_K_BYTES;
                    const uint8_t* a = xq + m * rba + s * ORC_Q8_K_BYTES;
                    int32_t S;
                    sums_q6_k(w, a, 1, &S);
                    double term = (double)get_f32(a) * (double)orc_f16_to_f32(get_u16(w + 208)) * (double)S;
                    acc += term;
                    t += fabs(term);
                }
                y[m * N + n] = acc;
                T[m * N + n] = t;
            }
        free(xq);
    } else if (wtype != ORC_Q4_K) {  /* Q8_0, Q4_0, Q5_0 weights with Q8_0 activations */
        int64_t nb = K / 32, wb = orc_block_bytes(wtype), rbw = nb * wb, rba = nb * ORC_Q8_0_BYTES;
        uint8_t* xq = (uint8_t*)malloc((size_t)(M * rba));
        orc_quantize_q8_0(x, M, K, xq);
        #pragma omp parallel for schedule(dynamic, 16) collapse(2)
        for (int64_t m = 0; m < M; ++m)
            for (int64_t n = 0; n < N; ++n) {
                const uint8_t* w = wq + n * rbw;
                const uint8_t* a = xq + m * rba;
                double acc = 0.0, t = 0.0;
                for (int64_t b = 0; b < nb; ++b) {
                    int32_t s;
                    sums_b32(wtype, w + b * wb, a + b * ORC_Q8_0_BYTES, 1, &s);
                    double term = (double)orc_f16_to_f32(get_u16(w + b * wb)) *
                                  (double)orc_f16_to_f32(get_u16(a + b * ORC_Q8_0_BYTES)) * (double)s;
                    acc += term;
                    t += fabs(term);
                }
                y[m * N + n] = acc;
                T[m * N + n] = t;
            }
        free(xq);
    } else {
        int64_t nsb = K / 256, rbw = nsb * ORC_Q4_K_BYTES, rba = nsb * ORC_Q8_K_BYTES;
        uint8_t* xq = (uint8_t*)malloc((size_t)(M * rba));
        orc_quantize_q8_k(x, M, K, xq);
        #pragma omp parallel for schedule(dynamic, 16) collapse(2)
        for (int64_t m = 0; m < M; ++m)
            for (int64_t n = 0; n < N; ++n) {
                int32_t ss[2];
                double acc = 0.0, t = 0.0;
                for (int64_t s = 0; s < nsb; ++s) {
                    const uint8_t* w = wq + n * rbw + s * ORC_Q4_K_BYTES;
                    const uint8_t* a = xq + m * rba + s * ORC_Q8_K_BYTES;
                    sums_q4_k(w, a, 1, ss);
                    double da = (double)get_f32(a);
                    double t1 = da * (double)orc_f16_to_f32(get_u16(w)) * (double)ss[0];
                    double t2 = da * (double)orc_f16_to_f32(get_u16(w + 2)) * (double)ss[1];
                    acc += t1 - t2;
                    t += fabs(t1) + fabs(t2);
                }
                y[m * N + n] = acc;
                T[m * N + n] = t;
            }
        free(xq);
    }
}

/* f32_act ("Metal form"): f32 activations times dequantized weights.
   Identical by definition to the dequantize-all form followed by an exact
   matmul; here the sum is taken in double. */
void orc_matmul_f32_act(int wtype, const uint8_t* wq, const float* x, int64_t M, int64_t N, int64_t K,
                        double* y, double* T) {
    int64_t rb = K / orc_block_values(wtype) * orc_block_bytes(wtype);
    #pragma omp parallel
    {
        float* w = (float*)malloc((size_t)K * sizeof(float));
        #pragma omp for schedule(dynamic, 16)
        for (int64_t n = 0; n < N; ++n) {
            dequant_row(wtype, wq + n * rb, K, w);
            for (int64_t m = 0; m < M; ++m) {
                const float* xr = x + m * K;
                double acc = 0.0, t = 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    double term = (double)xr[k] * (double)w[k];
                    acc += term;
                    t += fabs(term);
                }
                y[m * N + n] = acc;
                T[m * N + n] = t;
            }
        }
        free(w);
    }
}

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads used by the parallel loops from now on (n <= 0: all available).
   Each output element's summation order is fixed, so results do not depend
   on it; the benchmark times the single-threaded configurations with 1. */
void orc_set_num_threads(int n) {
#ifdef _OPENMP
    omp_set_num_threads(n > 0 ? n : omp_get_num_procs());
#else
    (void)n;
#endif
}
