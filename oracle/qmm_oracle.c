/*
 * qmm_oracle.c -- the plain, slow, scalar CPU oracle for the block-quantized
 * weight x Q8 activation matmul.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check of the
 * package entry module and the CPU-baseline leg of the benchmark may load or
 * call this library.  The CUDA library never links, includes or calls it, and
 * it shares no code, header, table or helper with the CUDA path.
 *
 * Every routine here follows the pages it cites, in their order and notation,
 * with no blocking, fusion or reordering beyond what they state.  Floating
 * point is IEEE binary32 where the pages fix it (the quantizers and the fp32
 * fold of each block's exact integer sum); the diagnostics are binary64.
 * Build with -O2 -ffp-contract=off and no fast-math, so that no multiply-add
 * is fused and every float operation rounds once, as written.
 *
 * Pages (cited by title and section):
 *   [minfer] "10 . CPU matmul: quantized weights x Q8_0 activations"
 *            (yusiwen.cn/minfer/inference_e2e_walkthrough/10-cpu-matmul-kernels)
 *   [ggml]   "ggml Q4_0 vec_dot Walkthrough" (blog.kkkzoz.top)
 *   [krafla] "Architecture" (jonpark0.github.io/krafla)
 *   [kvad]   "kvad -- the same ideas, at scale" (kvad.eu/docs/internals/engine)
 *
 * Readings taken where the pages are silent or garbled:
 *   - Q8_K activation blocks are 292 B: f32 d, int8 qs[256], int16 bsums[16].
 *   - The Q8_K inverse scale is 127/amax, the same expression as Q8_0.
 *   - Q4_0 codes are min(15, trunc(x*id + 8.5)) with d = m / -8.
 *   - Q4_K 6-bit scale packing, Q2_K code order and the whole Q6_K layout
 *     follow the GGUF byte layouts; the K-quant weight quantizers are plain
 *     min/max (Q4_K, Q2_K) and signed-extreme (Q6_K) schemes.  These are
 *     "parity unpinned" against any external source: they are pinned only by
 *     their encode/decode round trips and the brute-force dot products.
 *   - Q4_1 (20 B), Q5_0 (22 B), Q5_1 (24 B) and Q5_K (176 B) follow the GGUF
 *     byte layouts (the pages give the 22/24/176-B sizes and that Q5_0/Q5_1
 *     add a plane of high bits).  Q4_1/Q5_0/Q5_1 pair with Q8_0 activations
 *     like every 32-value type; their min term uses the exact integer sum of
 *     the activation block's codes.  Their quantizers are the Q4_0 idea on 5
 *     bits (Q5_0) and a plain min/max grid (Q4_1, Q5_1, and Q5_K as Q4_K).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_Q4_0 0
#define ORC_Q8_0 1
#define ORC_Q4_K 2
#define ORC_Q6_K 3
#define ORC_Q2_K 4
#define ORC_Q8_K 5
#define ORC_Q4_1 6
#define ORC_Q5_0 7
#define ORC_Q5_1 8
#define ORC_Q5_K 9

/* ------------------------------------------------------------------------- */
/* Block sizes.  [minfer] s2.3 (block.rs constants: 18, 34, 144, 210);       */
/* [ggml] s1.1 (block_q8_0 = 34 B, block_q4_0 = 18 B), s1.2 (block_q2_K =   */
/* 84 B).  Q8_K is the 292-B f32-d layout (see the readings above).          */
/* [minfer] s1 (the data-flow diagram: 18/22/24/34/144/176/210 B per block)  */
/* and s3.2 (Q5_0/Q5_1 "22/24 B blocks", dot_q5_k_q8_k over 176-B rows).     */
/* Q4_1's 20 B (f16 d, f16 m, 16 B of nibbles) is the GGUF layout.           */
/* ------------------------------------------------------------------------- */
int orc_block_bytes(int type) {
    switch (type) {
    case ORC_Q4_0: return 2 + 16;
    case ORC_Q8_0: return 2 + 32;
    case ORC_Q4_K: return 2 + 2 + 12 + 128;
    case ORC_Q6_K: return 128 + 64 + 16 + 2;
    case ORC_Q2_K: return 16 + 64 + 2 + 2;
    case ORC_Q8_K: return 4 + 256 + 2 * 16;
    case ORC_Q4_1: return 2 + 2 + 16;
    case ORC_Q5_0: return 2 + 4 + 16;
    case ORC_Q5_1: return 2 + 2 + 4 + 16;
    case ORC_Q5_K: return 2 + 2 + 12 + 32 + 128;
    default: return 0;
    }
}

int orc_block_values(int type) {
    switch (type) {
    case ORC_Q4_0: case ORC_Q8_0: case ORC_Q4_1: case ORC_Q5_0: case ORC_Q5_1: return 32;
    case ORC_Q4_K: case ORC_Q6_K: case ORC_Q2_K: case ORC_Q8_K: case ORC_Q5_K: return 256;
    default: return 0;
    }
}

/* The activation format each weight type pairs with: [minfer] s2.4 and s3.2
 * (cpu_quant_matmul_f32): K-quant weights take Q8_K, all others Q8_0. */
int orc_act_type(int wtype) {
    return (wtype == ORC_Q4_K || wtype == ORC_Q6_K || wtype == ORC_Q2_K || wtype == ORC_Q5_K) ? ORC_Q8_K : ORC_Q8_0;
}

/* ------------------------------------------------------------------------- */
/* IEEE binary16 <-> binary32.  The pages store d as "f16(d)" ([minfer]      */
/* s3.2, quantize_avx2) and read it back with fp16_to_f32.  Conversion to    */
/* half rounds to nearest, ties to even, keeps subnormals, and overflows to  */
/* infinity; conversion back is exact.                                       */
/* ------------------------------------------------------------------------- */
uint16_t orc_f32_to_f16(float f) {
    uint32_t x;
    memcpy(&x, &f, 4);
    uint32_t sign = (x >> 16) & 0x8000u;
    uint32_t exp = (x >> 23) & 0xFFu;
    uint32_t man = x & 0x7FFFFFu;
    if (exp == 0xFFu) {                      /* infinity or NaN */
        if (man == 0) return (uint16_t)(sign | 0x7C00u);
        return (uint16_t)(sign | 0x7E00u | (man >> 13));
    }
    if (exp == 0) return (uint16_t)sign;     /* f32 zero/subnormal: below half's range */
    int e = (int)exp - 127 + 15;             /* rebiased half exponent */
    if (e >= 31) return (uint16_t)(sign | 0x7C00u);
    if (e >= 1) {                            /* normal half: drop 13 mantissa bits */
        uint32_t h = ((uint32_t)e << 10) | (man >> 13);
        uint32_t rest = man & 0x1FFFu;
        if (rest > 0x1000u || (rest == 0x1000u && (h & 1u))) h += 1u; /* carry may reach inf: correct */
        return (uint16_t)(sign | h);
    }
    /* subnormal half: value = m * 2^(exp-150); in units of 2^-24 that is m >> (126-exp) */
    uint32_t m = man | 0x800000u;
    int shift = 126 - (int)exp;              /* >= 14 here */
    if (shift > 25) return (uint16_t)sign;   /* below half of the smallest subnormal */
    uint32_t q = m >> shift;
    uint32_t rest = m & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rest > half || (rest == half && (q & 1u))) q += 1u;
    return (uint16_t)(sign | q);
}

float orc_f16_to_f32(uint16_t h) {
    uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
    uint32_t exp = (h >> 10) & 0x1Fu;
    uint32_t man = h & 0x3FFu;
    float out;
    if (exp == 0) {
        out = ldexpf((float)man, -24);       /* zero or subnormal: exact */
        if (sign) out = -out;
        return out;
    }
    uint32_t bits;
    if (exp == 31) bits = sign | 0x7F800000u | (man << 13);
    else bits = sign | ((exp - 15 + 127) << 23) | (man << 13);
    memcpy(&out, &bits, 4);
    return out;
}

static uint16_t rd16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static void wr16(uint8_t* p, uint16_t v) { p[0] = (uint8_t)(v & 0xFF); p[1] = (uint8_t)(v >> 8); }
static float rdf32(const uint8_t* p) { float f; memcpy(&f, p, 4); return f; }
static void wrf32(uint8_t* p, float f) { memcpy(p, &f, 4); }
static int16_t rdi16(const uint8_t* p) { return (int16_t)rd16(p); }

/* round to nearest integer, ties to even (the default IEEE rounding mode); a value
 * beyond the int range saturates and NaN gives 0, so the conversion is defined for
 * every input (only degenerate scales can produce such quotients) */
static int rne(float v) {
    float r = nearbyintf(v);
    if (r != r) return 0;
    if (r >= 2147483648.0f) return 2147483647;
    if (r <= -2147483648.0f) return -2147483647 - 1;
    return (int)r;
}
static int clampi(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }

/* ------------------------------------------------------------------------- */
/* Activation quantizer Q8_0.  [minfer] s3.2 "The activation quantizers":    */
/* per 32 values amax = max|x|, d = amax/127 stored as f16, id = 127/amax    */
/* (0 for an all-zero block: the zero-block guard), each code the nearest    */
/* integer to x*id (ties to even) narrowed with saturation to int8.          */
/* [ggml] s1.1 gives the same block: fp16 d + int8 qs[32], 34 bytes.         */
/* Q8_0 weights are quantized by the same routine.                           */
/* ------------------------------------------------------------------------- */
void orc_quantize_q8_0(const float* x, uint8_t* out, int64_t n) {
    for (int64_t b = 0; b < n / 32; b++) {
        const float* xb = x + b * 32;
        uint8_t* ob = out + b * 34;
        float amax = 0.0f;
        for (int i = 0; i < 32; i++) {
            float a = fabsf(xb[i]);
            if (a > amax) amax = a;
        }
        float d = amax / 127.0f;
        wr16(ob, orc_f32_to_f16(d));
        float id = (amax != 0.0f) ? 127.0f / amax : 0.0f;
        for (int i = 0; i < 32; i++) {
            float v = xb[i] * id;
            ob[2 + i] = (uint8_t)(int8_t)clampi(rne(v), -128, 127);
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Activation quantizer Q8_K.  [minfer] s3.2 (quantize_row_q8_k_buf): per    */
/* 256 values amax, d = amax/127, int8 codes with saturating rounding, and   */
/* bsums[g] = the exact sum of the 16 SATURATED codes of group g.  Layout:   */
/* f32 d @0, qs[256] @4, int16 bsums[16] @260 (292 B).                       */
/* ------------------------------------------------------------------------- */
void orc_quantize_q8_K(const float* x, uint8_t* out, int64_t n) {
    for (int64_t b = 0; b < n / 256; b++) {
        const float* xb = x + b * 256;
        uint8_t* ob = out + b * 292;
        float amax = 0.0f;
        for (int i = 0; i < 256; i++) {
            float a = fabsf(xb[i]);
            if (a > amax) amax = a;
        }
        float d = amax / 127.0f;
        wrf32(ob, d);
        float id = (amax != 0.0f) ? 127.0f / amax : 0.0f;
        for (int g = 0; g < 16; g++) {
            int sum = 0;
            for (int i = 0; i < 16; i++) {
                float v = xb[g * 16 + i] * id;
                int q = clampi(rne(v), -128, 127);
                ob[4 + g * 16 + i] = (uint8_t)(int8_t)q;
                sum += q;
            }
            wr16(ob + 260 + 2 * g, (uint16_t)(int16_t)sum);
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Weight quantizer Q4_0.  [ggml] s1.1 and [kvad] "The scale that wasted a   */
/* code": m is the value of largest magnitude (its sign kept; the first one  */
/* on a tie), d = m / -8 so that m decodes exactly as code -8, and the       */
/* opposite extreme clips to 7/8 of its value.  Codes are stored +8 as       */
/* nibbles; byte j holds element j (low nibble) and j+16 (high nibble).      */
/* ------------------------------------------------------------------------- */
void orc_quantize_q4_0(const float* x, uint8_t* out, int64_t n) {
    for (int64_t b = 0; b < n / 32; b++) {
        const float* xb = x + b * 32;
        uint8_t* ob = out + b * 18;
        float amax = 0.0f, m = 0.0f;
        for (int i = 0; i < 32; i++) {
            if (fabsf(xb[i]) > amax) { amax = fabsf(xb[i]); m = xb[i]; }
        }
        float d = m / -8.0f;
        float id = (d != 0.0f) ? 1.0f / d : 0.0f;
        wr16(ob, orc_f32_to_f16(d));
        uint8_t code[32];
        for (int i = 0; i < 32; i++) {
            float t = xb[i] * id + 8.5f;     /* two roundings, as written: multiply, then add */
            int c = (int)t;                  /* t >= 0 here, so truncation is floor */
            code[i] = (uint8_t)clampi(c, 0, 15);
        }
        for (int j = 0; j < 16; j++) ob[2 + j] = (uint8_t)(code[j] | (code[j + 16] << 4));
    }
}

/* ------------------------------------------------------------------------- */
/* Q4_K: 144 B per 256 values: f16 d @0, f16 dmin @2, 12 B of packed 6-bit   */
/* scales and mins @4, 128 B of nibbles @16 ([minfer] s3.2, the K-quant dot  */
/* and its value formula q*d_s - min_s).  For j = 0..3, byte qs[32j+l]       */
/* holds element 64j+l in its low nibble (sub-block 2j) and 64j+32+l in its  */
/* high nibble (sub-block 2j+1), as that listing pairs them.                 */
/* ------------------------------------------------------------------------- */
void orc_q4_K_unpack_scales(const uint8_t* b, int sc[8], int mn[8]) {
    for (int s = 0; s < 4; s++) {
        sc[s] = b[s] & 63;
        mn[s] = b[s + 4] & 63;
    }
    for (int s = 4; s < 8; s++) {
        sc[s] = (b[s + 4] & 15) | ((b[s - 4] >> 6) << 4);
        mn[s] = (b[s + 4] >> 4) | ((b[s] >> 6) << 4);
    }
}

static void q4_K_pack_scales(const int sc[8], const int mn[8], uint8_t* b) {
    for (int s = 0; s < 4; s++) {
        b[s] = (uint8_t)((sc[s] & 63) | ((sc[s + 4] >> 4) << 6));
        b[s + 4] = (uint8_t)((mn[s] & 63) | ((mn[s + 4] >> 4) << 6));
        b[s + 8] = (uint8_t)((sc[s + 4] & 15) | ((mn[s + 4] & 15) << 4));
    }
}

/* Reading: a plain min/max scheme.  Per sub-block, min_s = max(0, -min x),
 * scale_s = (max x + min_s)/15; d = max scale_s / 63, dmin = max min_s / 63;
 * 6-bit sc_s = RNE(scale_s/d), m_s = RNE(min_s/dmin); then each code is
 * RNE((x + dmin16*m_s) / (d16*sc_s)) in 0..15, using the stored f16 d, dmin. */
void orc_quantize_q4_K(const float* x, uint8_t* out, int64_t n) {
    for (int64_t b = 0; b < n / 256; b++) {
        const float* xb = x + b * 256;
        uint8_t* ob = out + b * 144;
        float scl[8], mns[8];
        float maxscl = 0.0f, maxmin = 0.0f;
        for (int s = 0; s < 8; s++) {
            float lo = xb[32 * s], hi = xb[32 * s];
            for (int i = 1; i < 32; i++) {
                float v = xb[32 * s + i];
                if (v < lo) lo = v;
                if (v > hi) hi = v;
            }
            mns[s] = lo < 0.0f ? -lo : 0.0f;
            scl[s] = (hi + mns[s]) / 15.0f;
            if (scl[s] > maxscl) maxscl = scl[s];
            if (mns[s] > maxmin) maxmin = mns[s];
        }
        float d = maxscl / 63.0f, dmin = maxmin / 63.0f;
        uint16_t dh = orc_f32_to_f16(d), dmh = orc_f32_to_f16(dmin);
        wr16(ob, dh);
        wr16(ob + 2, dmh);
        int sc[8], mn[8];
        for (int s = 0; s < 8; s++) {
            sc[s] = d > 0.0f ? clampi(rne(scl[s] / d), 0, 63) : 0;
            mn[s] = dmin > 0.0f ? clampi(rne(mns[s] / dmin), 0, 63) : 0;
        }
        q4_K_pack_scales(sc, mn, ob + 4);
        float df = orc_f16_to_f32(dh), dmf = orc_f16_to_f32(dmh);
        uint8_t q[256];
        for (int s = 0; s < 8; s++) {
            float ds = df * (float)sc[s];
            float dm = dmf * (float)mn[s];
            for (int i = 0; i < 32; i++) {
                float v = xb[32 * s + i];
                q[32 * s + i] = (uint8_t)(ds > 0.0f ? clampi(rne((v + dm) / ds), 0, 15) : 0);
            }
        }
        for (int j = 0; j < 4; j++)
            for (int l = 0; l < 32; l++)
                ob[16 + 32 * j + l] = (uint8_t)(q[64 * j + l] | (q[64 * j + 32 + l] << 4));
    }
}

/* ------------------------------------------------------------------------- */
/* Q2_K: [ggml] s1.2.  84 B per 256 values: scales[16] @0 (low nibble = the  */
/* group scale sc, high nibble = the group min m), qs[64] @16 (2-bit codes), */
/* f16 d @80, f16 dmin @82.  A weight decodes as d*sc*q - dmin*m over 16     */
/* groups of 16.  Code order (reading, GGUF): for half h, shift s, lane l,   */
/* element 128h + 32s + l is (qs[32h + l] >> 2s) & 3.                        */
/* Quantizer (reading): the Q4_K scheme with 2-bit codes and 4-bit sc, m.    */
/* ------------------------------------------------------------------------- */
void orc_quantize_q2_K(const float* x, uint8_t* out, int64_t n) {
    for (int64_t b = 0; b < n / 256; b++) {
        const float* xb = x + b * 256;
        uint8_t* ob = out + b * 84;
        float scl[16], mns[16];
        float maxscl = 0.0f, maxmin = 0.0f;
        for (int g = 0; g < 16; g++) {
            float lo = xb[16 * g], hi = xb[16 * g];
            for (int i = 1; i < 16; i++) {
                float v = xb[16 * g + i];
                if (v < lo) lo = v;
                if (v > hi) hi = v;
            }
            mns[g] = lo < 0.0f ? -lo : 0.0f;
            scl[g] = (hi + mns[g]) / 3.0f;
            if (scl[g] > maxscl) maxscl = scl[g];
            if (mns[g] > maxmin) maxmin = mns[g];
        }
        float d = maxscl / 15.0f, dmin = maxmin / 15.0f;
        uint16_t dh = orc_f32_to_f16(d), dmh = orc_f32_to_f16(dmin);
        wr16(ob + 80, dh);
        wr16(ob + 82, dmh);
        int sc[16], mn[16];
        for (int g = 0; g < 16; g++) {
            sc[g] = d > 0.0f ? clampi(rne(scl[g] / d), 0, 15) : 0;
            mn[g] = dmin > 0.0f ? clampi(rne(mns[g] / dmin), 0, 15) : 0;
            ob[g] = (uint8_t)(sc[g] | (mn[g] << 4));
        }
        float df = orc_f16_to_f32(dh), dmf = orc_f16_to_f32(dmh);
        uint8_t q[256];
        for (int g = 0; g < 16; g++) {
            float ds = df * (float)sc[g];
            float dm = dmf * (float)mn[g];
            for (int i = 0; i < 16; i++) {
                float v = xb[16 * g + i];
                q[16 * g + i] = (uint8_t)(ds > 0.0f ? clampi(rne((v + dm) / ds), 0, 3) : 0);
            }
        }
        memset(ob + 16, 0, 64);
        for (int h = 0; h < 2; h++)
            for (int s = 0; s < 4; s++)
                for (int l = 0; l < 32; l++)
                    ob[16 + 32 * h + l] |= (uint8_t)(q[128 * h + 32 * s + l] << (2 * s));
    }
}

/* ------------------------------------------------------------------------- */
/* Q6_K: 210 B per 256 values ([minfer] s2.3 gives only the size).  Reading, */
/* GGUF layout: ql[128] @0, qh[64] @128, int8 scales[16] @192, f16 d @208.   */
/* For half n and lane l, elements 128n+l+32k (k = 0..3) take their low 4    */
/* bits from ql[64n+l] (k=0 low, k=2 high nibble) and ql[64n+l+32] (k=1 low, */
/* k=3 high nibble), and their top 2 bits from qh[32n+l] bits 2k..2k+1.      */
/* A weight decodes as d * scales[e/16] * (q - 32).                          */
/* Quantizer (reading): per group of 16, the Q4_0 idea with 6 bits: the      */
/* signed extreme m_g gives s_g = m_g / -32; d = max|s_g| / 127 (f16);       */
/* sc_g = RNE(s_g/d) (int8); codes RNE(x / (d16*sc_g)) in -32..31, +32.      */
/* ------------------------------------------------------------------------- */
void orc_quantize_q6_K(const float* x, uint8_t* out, int64_t n) {
    for (int64_t b = 0; b < n / 256; b++) {
        const float* xb = x + b * 256;
        uint8_t* ob = out + b * 210;
        float sg[16];
        float amax_s = 0.0f;
        for (int g = 0; g < 16; g++) {
            float amax = 0.0f, m = 0.0f;
            for (int i = 0; i < 16; i++) {
                float v = xb[16 * g + i];
                if (fabsf(v) > amax) { amax = fabsf(v); m = v; }
            }
            sg[g] = m / -32.0f;
            if (fabsf(sg[g]) > amax_s) amax_s = fabsf(sg[g]);
        }
        float d = amax_s / 127.0f;
        uint16_t dh = orc_f32_to_f16(d);
        wr16(ob + 208, dh);
        int sc[16];
        for (int g = 0; g < 16; g++) {
            sc[g] = d > 0.0f ? clampi(rne(sg[g] / d), -128, 127) : 0;
            ob[192 + g] = (uint8_t)(int8_t)sc[g];
        }
        float df = orc_f16_to_f32(dh);
        uint8_t c[256];
        for (int g = 0; g < 16; g++) {
            float ds = df * (float)sc[g];
            for (int i = 0; i < 16; i++) {
                float v = xb[16 * g + i];
                int q = ds != 0.0f ? clampi(rne(v / ds), -32, 31) : 0;
                c[16 * g + i] = (uint8_t)(q + 32);
            }
        }
        for (int h = 0; h < 2; h++) {
            for (int l = 0; l < 32; l++) {
                int c0 = c[128 * h + l], c1 = c[128 * h + l + 32];
                int c2 = c[128 * h + l + 64], c3 = c[128 * h + l + 96];
                ob[64 * h + l] = (uint8_t)((c0 & 15) | ((c2 & 15) << 4));
                ob[64 * h + l + 32] = (uint8_t)((c1 & 15) | ((c3 & 15) << 4));
                ob[128 + 32 * h + l] =
                    (uint8_t)((c0 >> 4) | ((c1 >> 4) << 2) | ((c2 >> 4) << 4) | ((c3 >> 4) << 6));
            }
        }
    }
}

/* ------------------------------------------------------------------------- */
/* 32-value formats with a min or a fifth bit ([minfer] s3.2: "Q5_0/Q5_1 add */
/* their high-bit planes (22/24 B blocks)"; layouts are GGUF readings):      */
/*   Q4_1  f16 d @0, f16 m @2, qs[16] @4        value d*q + m,   q in 0..15  */
/*   Q5_0  f16 d @0, qh[4] @2, qs[16] @6        value d*(q-16),  q in 0..31  */
/*   Q5_1  f16 d @0, f16 m @2, qh[4] @4, qs[16] @8   value d*q + m, 0..31    */
/* Nibbles as in Q4_0 (byte j: element j low, j+16 high); bit i of the       */
/* little-endian 32-bit qh is the fifth bit of element i.                    */
/* ------------------------------------------------------------------------- */
static void pack_nibbles(const uint8_t code[32], uint8_t* qs) {
    for (int j = 0; j < 16; j++) qs[j] = (uint8_t)((code[j] & 15) | ((code[j + 16] & 15) << 4));
}

static void pack_high_bits(const uint8_t code[32], uint8_t* qh) {
    uint32_t h = 0;
    for (int i = 0; i < 32; i++) h |= (uint32_t)((code[i] >> 4) & 1) << i;
    for (int k = 0; k < 4; k++) qh[k] = (uint8_t)(h >> (8 * k));
}

/* Reading: a min/max grid.  m = min x, d = (max x - m) / levels, and each code
 * the nearest grid step (x - m)/d rounded half up, clamped to levels; computed
 * with the f32 d and m, stored as f16. */
static void quantize_minmax_32(const float* xb, int levels, float* d_out, float* m_out, uint8_t code[32]) {
    float lo = xb[0], hi = xb[0];
    for (int i = 1; i < 32; i++) {
        if (xb[i] < lo) lo = xb[i];
        if (xb[i] > hi) hi = xb[i];
    }
    float d = (hi - lo) / (float)levels;
    float id = (d != 0.0f) ? 1.0f / d : 0.0f;
    for (int i = 0; i < 32; i++) {
        float t = (xb[i] - lo) * id + 0.5f;  /* >= 0.5, so truncation is floor */
        code[i] = (uint8_t)clampi((int)t, 0, levels);
    }
    *d_out = d;
    *m_out = lo;
}

void orc_quantize_q4_1(const float* x, uint8_t* out, int64_t n) {
    for (int64_t b = 0; b < n / 32; b++) {
        uint8_t* ob = out + b * 20;
        float d, m;
        uint8_t code[32];
        quantize_minmax_32(x + b * 32, 15, &d, &m, code);
        wr16(ob, orc_f32_to_f16(d));
        wr16(ob + 2, orc_f32_to_f16(m));
        pack_nibbles(code, ob + 4);
    }
}

void orc_quantize_q5_1(const float* x, uint8_t* out, int64_t n) {
    for (int64_t b = 0; b < n / 32; b++) {
        uint8_t* ob = out + b * 24;
        float d, m;
        uint8_t code[32];
        quantize_minmax_32(x + b * 32, 31, &d, &m, code);
        wr16(ob, orc_f32_to_f16(d));
        wr16(ob + 2, orc_f32_to_f16(m));
        pack_high_bits(code, ob + 4);
        pack_nibbles(code, ob + 8);
    }
}

/* Reading: the Q4_0 scheme on 5 bits.  m = the value of largest magnitude (the
 * first on a tie), d = m / -16, codes min(31, trunc(x/d + 16.5)). */
void orc_quantize_q5_0(const float* x, uint8_t* out, int64_t n) {
    for (int64_t b = 0; b < n / 32; b++) {
        const float* xb = x + b * 32;
        uint8_t* ob = out + b * 22;
        float amax = 0.0f, m = 0.0f;
        for (int i = 0; i < 32; i++) {
            if (fabsf(xb[i]) > amax) { amax = fabsf(xb[i]); m = xb[i]; }
        }
        float d = m / -16.0f;
        float id = (d != 0.0f) ? 1.0f / d : 0.0f;
        wr16(ob, orc_f32_to_f16(d));
        uint8_t code[32];
        for (int i = 0; i < 32; i++) {
            float t = xb[i] * id + 16.5f;
            code[i] = (uint8_t)clampi((int)t, 0, 31);
        }
        pack_high_bits(code, ob + 2);
        pack_nibbles(code, ob + 6);
    }
}

/* ------------------------------------------------------------------------- */
/* Q5_K: 176 B per 256 values ([minfer] s1 and s3.2 give the size and the    */
/* dot_q5_k_q8_k arm).  Reading, GGUF layout: f16 d @0, f16 dmin @2, the     */
/* Q4_K 12-byte scale/min packing @4, qh[32] @16, qs[128] @48.  For chunk j  */
/* = 0..3 and lane l: element 64j+l has low nibble qs[32j+l] & 15 and fifth  */
/* bit (qh[l] >> 2j) & 1; element 64j+32+l has qs[32j+l] >> 4 and bit 2j+1.  */
/* A weight decodes as d*sc_s*q - dmin*m_s.  Quantizer: the Q4_K scheme with */
/* codes 0..31.                                                              */
/* ------------------------------------------------------------------------- */
void orc_quantize_q5_K(const float* x, uint8_t* out, int64_t n) {
    for (int64_t b = 0; b < n / 256; b++) {
        const float* xb = x + b * 256;
        uint8_t* ob = out + b * 176;
        float scl[8], mns[8];
        float maxscl = 0.0f, maxmin = 0.0f;
        for (int s = 0; s < 8; s++) {
            float lo = xb[32 * s], hi = xb[32 * s];
            for (int i = 1; i < 32; i++) {
                float v = xb[32 * s + i];
                if (v < lo) lo = v;
                if (v > hi) hi = v;
            }
            mns[s] = lo < 0.0f ? -lo : 0.0f;
            scl[s] = (hi + mns[s]) / 31.0f;
            if (scl[s] > maxscl) maxscl = scl[s];
            if (mns[s] > maxmin) maxmin = mns[s];
        }
        float d = maxscl / 63.0f, dmin = maxmin / 63.0f;
        uint16_t dh = orc_f32_to_f16(d), dmh = orc_f32_to_f16(dmin);
        wr16(ob, dh);
        wr16(ob + 2, dmh);
        int sc[8], mn[8];
        for (int s = 0; s < 8; s++) {
            sc[s] = d > 0.0f ? clampi(rne(scl[s] / d), 0, 63) : 0;
            mn[s] = dmin > 0.0f ? clampi(rne(mns[s] / dmin), 0, 63) : 0;
        }
        q4_K_pack_scales(sc, mn, ob + 4);
        float df = orc_f16_to_f32(dh), dmf = orc_f16_to_f32(dmh);
        uint8_t q[256];
        for (int s = 0; s < 8; s++) {
            float ds = df * (float)sc[s];
            float dm = dmf * (float)mn[s];
            for (int i = 0; i < 32; i++) {
                float v = xb[32 * s + i];
                q[32 * s + i] = (uint8_t)(ds > 0.0f ? clampi(rne((v + dm) / ds), 0, 31) : 0);
            }
        }
        memset(ob + 16, 0, 32);
        for (int j = 0; j < 4; j++)
            for (int l = 0; l < 32; l++) {
                int lo = q[64 * j + l], hi = q[64 * j + 32 + l];
                ob[48 + 32 * j + l] = (uint8_t)((lo & 15) | ((hi & 15) << 4));
                ob[16 + l] |= (uint8_t)(((lo >> 4) << (2 * j)) | ((hi >> 4) << (2 * j + 1)));
            }
    }
}

/* ------------------------------------------------------------------------- */
/* Decoding a block to its integer codes (and scale factors).  These are the */
/* per-format decode formulas above, read back out of the bytes.             */
/* ------------------------------------------------------------------------- */

/* Q4_0 element i of a block: low nibble of byte i for i < 16, high nibble of
 * byte i-16 otherwise, minus 8 ([ggml] s2; [minfer] s3.2 scalar kernel). */
static int q4_0_code(const uint8_t* blk, int i) {
    const uint8_t* qs = blk + 2;
    return (i < 16 ? (qs[i] & 0x0F) : (qs[i - 16] >> 4)) - 8;
}

static int q4_K_code(const uint8_t* blk, int e) {   /* 0..15 */
    int j = e / 64, r = e % 64;
    uint8_t byte = blk[16 + 32 * j + (r % 32)];
    return r < 32 ? (byte & 0x0F) : (byte >> 4);
}

static int q2_K_code(const uint8_t* blk, int e) {   /* 0..3 */
    int h = e / 128, s = (e % 128) / 32, l = e % 32;
    return (blk[16 + 32 * h + l] >> (2 * s)) & 3;
}

/* the stored 4-bit code of element i of a 32-value block whose nibbles start at qs */
static int nibble_code(const uint8_t* qs, int i) { return i < 16 ? (qs[i] & 0x0F) : (qs[i - 16] >> 4); }

/* the fifth bit of element i: bit i of the little-endian 32-bit word at qh */
static int fifth_bit(const uint8_t* qh, int i) { return (qh[i / 8] >> (i % 8)) & 1; }

static int q4_1_code(const uint8_t* blk, int i) { return nibble_code(blk + 4, i); }                           /* 0..15 */
static int q5_0_code(const uint8_t* blk, int i) { return nibble_code(blk + 6, i) | (fifth_bit(blk + 2, i) << 4); } /* 0..31 */
static int q5_1_code(const uint8_t* blk, int i) { return nibble_code(blk + 8, i) | (fifth_bit(blk + 4, i) << 4); } /* 0..31 */

static int q5_K_code(const uint8_t* blk, int e) {   /* 0..31 */
    int j = e / 64, r = e % 64, l = r % 32;
    uint8_t byte = blk[48 + 32 * j + l];
    int low = r < 32 ? (byte & 0x0F) : (byte >> 4);
    int high = (blk[16 + l] >> (2 * j + (r >= 32))) & 1;
    return low | (high << 4);
}

static int q6_K_code(const uint8_t* blk, int e) {   /* 0..63 (stored code, before -32) */
    int h = e / 128, k = (e % 128) / 32, l = e % 32;
    const uint8_t* ql = blk;
    const uint8_t* qh = blk + 128;
    int low;
    switch (k) {
    case 0: low = ql[64 * h + l] & 15; break;
    case 1: low = ql[64 * h + l + 32] & 15; break;
    case 2: low = ql[64 * h + l] >> 4; break;
    default: low = ql[64 * h + l + 32] >> 4; break;
    }
    int high = (qh[32 * h + l] >> (2 * k)) & 3;
    return low | (high << 4);
}

/* Exact dequantized values, in binary64 (every product here is exact in
 * double: an 11-bit significand times small integers).  Used for the
 * brute-force dot products and the round-trip pins. */
void orc_dequantize(int type, const uint8_t* in, double* out, int64_t n) {
    int bv = orc_block_values(type), bb = orc_block_bytes(type);
    for (int64_t b = 0; b < n / bv; b++) {
        const uint8_t* blk = in + b * bb;
        double* o = out + b * bv;
        switch (type) {
        case ORC_Q4_0: {
            double d = orc_f16_to_f32(rd16(blk));
            for (int i = 0; i < 32; i++) o[i] = d * q4_0_code(blk, i);
        } break;
        case ORC_Q8_0: {
            double d = orc_f16_to_f32(rd16(blk));
            for (int i = 0; i < 32; i++) o[i] = d * (int8_t)blk[2 + i];
        } break;
        case ORC_Q8_K: {
            double d = rdf32(blk);
            for (int i = 0; i < 256; i++) o[i] = d * (int8_t)blk[4 + i];
        } break;
        case ORC_Q4_K: {
            double d = orc_f16_to_f32(rd16(blk)), dmin = orc_f16_to_f32(rd16(blk + 2));
            int sc[8], mn[8];
            orc_q4_K_unpack_scales(blk + 4, sc, mn);
            for (int e = 0; e < 256; e++) o[e] = d * sc[e / 32] * q4_K_code(blk, e) - dmin * mn[e / 32];
        } break;
        case ORC_Q2_K: {
            double d = orc_f16_to_f32(rd16(blk + 80)), dmin = orc_f16_to_f32(rd16(blk + 82));
            for (int e = 0; e < 256; e++) {
                int g = e / 16;
                o[e] = d * (blk[g] & 15) * q2_K_code(blk, e) - dmin * (blk[g] >> 4);
            }
        } break;
        case ORC_Q6_K: {
            double d = orc_f16_to_f32(rd16(blk + 208));
            for (int e = 0; e < 256; e++)
                o[e] = d * (int8_t)blk[192 + e / 16] * (q6_K_code(blk, e) - 32);
        } break;
        case ORC_Q4_1: {
            double d = orc_f16_to_f32(rd16(blk)), m = orc_f16_to_f32(rd16(blk + 2));
            for (int i = 0; i < 32; i++) o[i] = d * q4_1_code(blk, i) + m;
        } break;
        case ORC_Q5_0: {
            double d = orc_f16_to_f32(rd16(blk));
            for (int i = 0; i < 32; i++) o[i] = d * (q5_0_code(blk, i) - 16);
        } break;
        case ORC_Q5_1: {
            double d = orc_f16_to_f32(rd16(blk)), m = orc_f16_to_f32(rd16(blk + 2));
            for (int i = 0; i < 32; i++) o[i] = d * q5_1_code(blk, i) + m;
        } break;
        case ORC_Q5_K: {
            double d = orc_f16_to_f32(rd16(blk)), dmin = orc_f16_to_f32(rd16(blk + 2));
            int sc[8], mn[8];
            orc_q4_K_unpack_scales(blk + 4, sc, mn);
            for (int e = 0; e < 256; e++) o[e] = d * sc[e / 32] * q5_K_code(blk, e) - dmin * mn[e / 32];
        } break;
        default: break;
        }
    }
}

/* Raw integer codes (test helper): the value each element's code stands for
 * before scaling: Q4_0 q-8, Q8_0/Q8_K q, Q4_K/Q2_K q, Q6_K q-32, Q4_1/Q5_1/Q5_K q
 * (their min is added, or subtracted, separately), Q5_0 q-16. */
void orc_codes(int type, const uint8_t* in, int32_t* out, int64_t n) {
    int bv = orc_block_values(type), bb = orc_block_bytes(type);
    for (int64_t b = 0; b < n / bv; b++) {
        const uint8_t* blk = in + b * bb;
        int32_t* o = out + b * bv;
        for (int e = 0; e < bv; e++) {
            switch (type) {
            case ORC_Q4_0: o[e] = q4_0_code(blk, e); break;
            case ORC_Q8_0: o[e] = (int8_t)blk[2 + e]; break;
            case ORC_Q8_K: o[e] = (int8_t)blk[4 + e]; break;
            case ORC_Q4_K: o[e] = q4_K_code(blk, e); break;
            case ORC_Q2_K: o[e] = q2_K_code(blk, e); break;
            case ORC_Q6_K: o[e] = q6_K_code(blk, e) - 32; break;
            case ORC_Q4_1: o[e] = q4_1_code(blk, e); break;
            case ORC_Q5_0: o[e] = q5_0_code(blk, e) - 16; break;
            case ORC_Q5_1: o[e] = q5_1_code(blk, e); break;
            case ORC_Q5_K: o[e] = q5_K_code(blk, e); break;
            default: o[e] = 0;
            }
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Exact integer block sums.  [ggml] s2 (factorized dot: the codes multiply  */
/* as integers, the scales apply once per block); [minfer] s3.2 scalar       */
/* kernels.  One int32 per 32-value block for Q4_0/Q8_0; two per K-quant     */
/* super-block: (value term, min term).                                      */
/*   Q4_K  value = sum_j s_lo*sc[2j] + s_hi*sc[2j+1],                        */
/*         min   = sum_s m_s*(bsum[2s] + bsum[2s+1])      ([minfer] s3.2)    */
/*   Q2_K  value = sum_g sc_g * sum_{i in g} q_i*a_i,  min = sum_g m_g*bsum_g */
/*   Q6_K  value = sum_g sc_g * sum_{i in g} q_i*a_i (q the stored 0..63),   */
/*         min   = sum_g sc_g * bsum_g; the dot's integer is value - 32*min.  */
/*   Q4_1, Q5_1  isum = sum_i q_i*a_i (q unsigned); the min contributes      */
/*         m * sum_i a_i, the activation block's own code sum               */
/*   Q5_0  isum = sum_i (q_i - 16)*a_i                                       */
/*   Q5_K  value = sum_s sc_s * sum_{i in s} q_i*a_i, min as Q4_K            */
/* ------------------------------------------------------------------------- */
static int32_t act_block_sum(const uint8_t* ab) {
    int32_t s = 0;
    for (int j = 0; j < 32; j++) s += (int8_t)ab[2 + j];
    return s;
}

static int32_t blk32_isum(int wtype, const uint8_t* wb, const uint8_t* ab) {
    int32_t si = 0;
    if (wtype == ORC_Q4_0) {
        /* the scalar kernel of [minfer] s3.2 / [ggml] s2: byte j pairs its low
         * nibble with activation j and its high nibble with activation j+16 */
        for (int j = 0; j < 16; j++) {
            int v0 = (wb[2 + j] & 0x0F) - 8;
            int v1 = (wb[2 + j] >> 4) - 8;
            si += v0 * (int8_t)ab[2 + j];
            si += v1 * (int8_t)ab[2 + j + 16];
        }
    } else if (wtype == ORC_Q8_0) {
        for (int j = 0; j < 32; j++) si += (int8_t)wb[2 + j] * (int8_t)ab[2 + j];
    } else { /* Q4_1, Q5_0, Q5_1: element by element */
        for (int i = 0; i < 32; i++) {
            int c = wtype == ORC_Q4_1 ? q4_1_code(wb, i) : wtype == ORC_Q5_0 ? q5_0_code(wb, i) - 16 : q5_1_code(wb, i);
            si += c * (int8_t)ab[2 + i];
        }
    }
    return si;
}

static void kblk_isums(int wtype, const uint8_t* wb, const uint8_t* ab, int32_t* value, int32_t* minterm) {
    const int8_t* a = (const int8_t*)(ab + 4);
    int bs[16];
    for (int g = 0; g < 16; g++) bs[g] = rdi16(ab + 260 + 2 * g);
    int32_t v = 0, m = 0;
    if (wtype == ORC_Q4_K) {
        int sc[8], mn[8];
        orc_q4_K_unpack_scales(wb + 4, sc, mn);
        for (int s = 0; s < 8; s++) m += mn[s] * (bs[2 * s] + bs[2 * s + 1]);
        int32_t sumi1 = 0, sumi2 = 0;
        for (int j = 0; j < 4; j++) {
            int32_t s_lo = 0, s_hi = 0;
            for (int l = 0; l < 32; l++) {
                s_lo += (wb[16 + 32 * j + l] & 0x0F) * a[64 * j + l];
                s_hi += (wb[16 + 32 * j + l] >> 4) * a[64 * j + 32 + l];
            }
            sumi1 += s_lo * sc[2 * j];
            sumi2 += s_hi * sc[2 * j + 1];
        }
        v = sumi1 + sumi2;
    } else if (wtype == ORC_Q5_K) {
        int sc[8], mn[8];
        orc_q4_K_unpack_scales(wb + 4, sc, mn);
        for (int s = 0; s < 8; s++) {
            int32_t si = 0;
            for (int i = 0; i < 32; i++) si += q5_K_code(wb, 32 * s + i) * a[32 * s + i];
            v += sc[s] * si;
            m += mn[s] * (bs[2 * s] + bs[2 * s + 1]);
        }
    } else if (wtype == ORC_Q2_K) {
        for (int g = 0; g < 16; g++) {
            int32_t s = 0;
            for (int i = 0; i < 16; i++) s += q2_K_code(wb, 16 * g + i) * a[16 * g + i];
            v += (wb[g] & 15) * s;
            m += (wb[g] >> 4) * bs[g];
        }
    } else { /* Q6_K */
        for (int g = 0; g < 16; g++) {
            int sc = (int8_t)wb[192 + g];
            int32_t s = 0;
            for (int i = 0; i < 16; i++) s += q6_K_code(wb, 16 * g + i) * a[16 * g + i];
            v += sc * s;
            m += sc * bs[g];
        }
    }
    *value = v;
    *minterm = m;
}

/* Block sums of one weight row against one activation row: out holds K/32
 * int32 (32-value types) or 2*K/256 int32 (K-quants, value then min). */
void orc_blocksums_row(int wtype, const uint8_t* wrow, const uint8_t* xrow, int64_t K, int32_t* out) {
    int at = orc_act_type(wtype);
    int wb = orc_block_bytes(wtype), ab = orc_block_bytes(at);
    if (at == ORC_Q8_0) {
        for (int64_t b = 0; b < K / 32; b++) out[b] = blk32_isum(wtype, wrow + b * wb, xrow + b * ab);
    } else {
        for (int64_t b = 0; b < K / 256; b++)
            kblk_isums(wtype, wrow + b * wb, xrow + b * ab, &out[2 * b], &out[2 * b + 1]);
    }
}

/* ------------------------------------------------------------------------- */
/* The row dot with its fp32 fold, in the pages' order.                      */
/*  Q4_0/Q8_0: s += (float)isum * dw * dx   ([minfer] s3.2 scalar kernel)    */
/*  Q4_K: d = dw*dx, dmin = dminw*dx; sumf -= dmin*min; sumf += d*value      */
/*        ([minfer] s3.2, the K-quant dot walked)                            */
/*  Q2_K: the same two-term fold with its own (value, min) ([ggml] s1.2)     */
/*  Q6_K: d = dw*dx; sumf += d*(value - 32*min)  (reading)                   */
/*  Q4_1/Q5_1: s += (float)isum*dw*dx; s += (float)asum*mw*dx   (reading)     */
/*  Q5_0: as Q4_0; Q5_K: as Q4_K                                             */
/* ------------------------------------------------------------------------- */
float orc_dot_row(int wtype, const uint8_t* wrow, const uint8_t* xrow, int64_t K) {
    int at = orc_act_type(wtype);
    int wb = orc_block_bytes(wtype), ab = orc_block_bytes(at);
    float s = 0.0f;
    if (at == ORC_Q8_0) {
        for (int64_t b = 0; b < K / 32; b++) {
            const uint8_t* w = wrow + b * wb;
            const uint8_t* a = xrow + b * ab;
            float dx = orc_f16_to_f32(rd16(w));
            float dy = orc_f16_to_f32(rd16(a));
            int32_t si = blk32_isum(wtype, w, a);
            s += (float)si * dx * dy;
            if (wtype == ORC_Q4_1 || wtype == ORC_Q5_1) {
                float mx = orc_f16_to_f32(rd16(w + 2));
                s += (float)act_block_sum(a) * mx * dy;
            }
        }
        return s;
    }
    for (int64_t b = 0; b < K / 256; b++) {
        const uint8_t* w = wrow + b * wb;
        const uint8_t* a = xrow + b * ab;
        float ad = rdf32(a);
        int32_t value, minterm;
        kblk_isums(wtype, w, a, &value, &minterm);
        if (wtype == ORC_Q4_K || wtype == ORC_Q5_K) {
            float d = orc_f16_to_f32(rd16(w)) * ad;
            float dmin = orc_f16_to_f32(rd16(w + 2)) * ad;
            s -= dmin * (float)minterm;
            s += d * (float)value;
        } else if (wtype == ORC_Q2_K) {
            float d = orc_f16_to_f32(rd16(w + 80)) * ad;
            float dmin = orc_f16_to_f32(rd16(w + 82)) * ad;
            s -= dmin * (float)minterm;
            s += d * (float)value;
        } else { /* Q6_K */
            float d = orc_f16_to_f32(rd16(w + 208)) * ad;
            s += d * (float)(value - 32 * minterm);
        }
    }
    return s;
}

/* Diagnostic: the same factorization with every scale product and the sum
 * taken in binary64 (no fp32 rounding at all beyond the stored scales). */
double orc_dot_row_exact(int wtype, const uint8_t* wrow, const uint8_t* xrow, int64_t K) {
    int at = orc_act_type(wtype);
    int wb = orc_block_bytes(wtype), ab = orc_block_bytes(at);
    double s = 0.0;
    if (at == ORC_Q8_0) {
        for (int64_t b = 0; b < K / 32; b++) {
            const uint8_t* w = wrow + b * wb;
            const uint8_t* a = xrow + b * ab;
            s += (double)orc_f16_to_f32(rd16(w)) * (double)orc_f16_to_f32(rd16(a)) *
                 (double)blk32_isum(wtype, w, a);
            if (wtype == ORC_Q4_1 || wtype == ORC_Q5_1)
                s += (double)orc_f16_to_f32(rd16(w + 2)) * (double)orc_f16_to_f32(rd16(a)) *
                     (double)act_block_sum(a);
        }
        return s;
    }
    for (int64_t b = 0; b < K / 256; b++) {
        const uint8_t* w = wrow + b * wb;
        const uint8_t* a = xrow + b * ab;
        double ad = rdf32(a);
        int32_t value, minterm;
        kblk_isums(wtype, w, a, &value, &minterm);
        if (wtype == ORC_Q4_K || wtype == ORC_Q5_K)
            s += ad * ((double)orc_f16_to_f32(rd16(w)) * value - (double)orc_f16_to_f32(rd16(w + 2)) * minterm);
        else if (wtype == ORC_Q2_K)
            s += ad * ((double)orc_f16_to_f32(rd16(w + 80)) * value -
                       (double)orc_f16_to_f32(rd16(w + 82)) * minterm);
        else
            s += ad * (double)orc_f16_to_f32(rd16(w + 208)) * (double)(value - 32 * minterm);
    }
    return s;
}

/* Diagnostic: the unfactorized dot of [ggml] s2 (left version): dequantize
 * every weight and every activation, multiply, add -- in binary64. */
double orc_dot_row_bruteforce(int wtype, const uint8_t* wrow, const uint8_t* xrow, int64_t K) {
    double* w = (double*)malloc(sizeof(double) * (size_t)K);
    double* a = (double*)malloc(sizeof(double) * (size_t)K);
    if (!w || !a) { free(w); free(a); return NAN; }
    orc_dequantize(wtype, wrow, w, K);
    orc_dequantize(orc_act_type(wtype), xrow, a, K);
    double s = 0.0;
    for (int64_t i = 0; i < K; i++) s += w[i] * a[i];
    free(w);
    free(a);
    return s;
}

/* ------------------------------------------------------------------------- */
/* The matmul: out[t][o] = dot(W row o, x row t), token-major output         */
/* ([minfer] s3.2 mm_rows: outer loop over rows o, inner over tokens t).     */
/* Rows are split evenly over nthreads, each row computed by exactly one     */
/* thread ([minfer] s3.2 thread pool, chunk()), so the result is identical   */
/* for any thread count.                                                     */
/* ------------------------------------------------------------------------- */
typedef struct {
    int wtype;
    const uint8_t* W;
    const uint8_t* X;
    float* out;
    int64_t M, N, K, r0, r1;
} orc_job;

static void* orc_rows(void* p) {
    orc_job* j = (orc_job*)p;
    int at = orc_act_type(j->wtype);
    int64_t ws = (j->K / orc_block_values(j->wtype)) * orc_block_bytes(j->wtype);
    int64_t xs = (j->K / orc_block_values(at)) * orc_block_bytes(at);
    for (int64_t o = j->r0; o < j->r1; o++)
        for (int64_t t = 0; t < j->M; t++)
            j->out[t * j->N + o] = orc_dot_row(j->wtype, j->W + o * ws, j->X + t * xs, j->K);
    return NULL;
}

int orc_matmul(int wtype, const uint8_t* W, const uint8_t* X, float* out, int64_t M, int64_t N, int64_t K,
               int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    orc_job jobs[256];
    for (int i = 0; i < nthreads; i++) {
        jobs[i].wtype = wtype; jobs[i].W = W; jobs[i].X = X; jobs[i].out = out;
        jobs[i].M = M; jobs[i].N = N; jobs[i].K = K;
        jobs[i].r0 = N * i / nthreads;
        jobs[i].r1 = N * (i + 1) / nthreads;
    }
    if (nthreads == 1) { orc_rows(&jobs[0]); return 0; }
    int started = 0;
    for (int i = 1; i < nthreads; i++) {
        if (pthread_create(&th[i], NULL, orc_rows, &jobs[i]) != 0) break;
        started = i;
    }
    orc_rows(&jobs[0]);
    for (int i = 1; i <= started; i++) pthread_join(th[i], NULL);
    for (int i = started + 1; i < nthreads; i++) orc_rows(&jobs[i]); /* threads that failed to start */
    return 0;
}

/* Block sums for a whole matmul: out[t][o][b] (b over the per-row count). */
void orc_blocksums(int wtype, const uint8_t* W, const uint8_t* X, int32_t* out, int64_t M, int64_t N, int64_t K) {
    int at = orc_act_type(wtype);
    int64_t ws = (K / orc_block_values(wtype)) * orc_block_bytes(wtype);
    int64_t xs = (K / orc_block_values(at)) * orc_block_bytes(at);
    int64_t per = (at == ORC_Q8_0) ? K / 32 : 2 * (K / 256);
    for (int64_t t = 0; t < M; t++)
        for (int64_t o = 0; o < N; o++) orc_blocksums_row(wtype, W + o * ws, X + t * xs, K, out + (t * N + o) * per);
}

/* Whole-matrix diagnostics: y_exact and the brute force, token-major. */
void orc_matmul_exact(int wtype, const uint8_t* W, const uint8_t* X, double* out, int64_t M, int64_t N, int64_t K,
                      int bruteforce) {
    int at = orc_act_type(wtype);
    int64_t ws = (K / orc_block_values(wtype)) * orc_block_bytes(wtype);
    int64_t xs = (K / orc_block_values(at)) * orc_block_bytes(at);
    for (int64_t t = 0; t < M; t++)
        for (int64_t o = 0; o < N; o++)
            out[t * N + o] = bruteforce ? orc_dot_row_bruteforce(wtype, W + o * ws, X + t * xs, K)
                                        : orc_dot_row_exact(wtype, W + o * ws, X + t * xs, K);
}

/* ------------------------------------------------------------------------- */
/* The Q8 KV cache.  [krafla] "Architecture", Attention ("Q8 cache"): each    */
/* position's K and V are stored per KV head as int8 codes with one float     */
/* scale, quantized by the activations' rule; each query head is quantized   */
/* the same way; the scores are integer dot products, and the V sum widens    */
/* the int8 values to float as it goes (head_dim 64: 68 bytes per head).      */
/* Readings:                                                                  */
/*   - a row is one head vector of hd values: f32 d @0, int8 codes @4         */
/*     (4 + hd bytes); the rule is the Q8_0 one (amax, d = amax/127, codes    */
/*     nearest-even of x*127/amax) over the whole head vector;               */
/*   - the cache holds row (p, kvh) at (p*Hkv + kvh) * (4 + hd): a position's */
/*     heads side by side, positions appended in order;                       */
/*   - query head h reads KV head h / (Hq/Hkv): [krafla] "Architecture",      */
/*     "Data flow for one token" (GQA head h -> kv head h / (n_heads /        */
/*     n_kv_heads)), not a reading;                                           */
/*   - a score is ((dq * dk) * isum) * scale in f32 (isum exact: |isum| <=    */
/*     hd * 128 * 128 < 2^24), scale the caller's factor (1/sqrt(hd) for      */
/*     attention);                                                            */
/*   - the V sum out[h][i] = sum_p w[h][p] * dv[p] * v[p][i] is given here    */
/*     exactly (binary64): the device sums in f32, so it is checked against   */
/*     an error bound, not bit for bit.                                       */
/* ------------------------------------------------------------------------- */
int orc_kv_row_bytes(int hd) { return 4 + hd; }

void orc_kv_quantize(const float* x, uint8_t* out, int64_t rows, int hd) {
    for (int64_t r = 0; r < rows; r++) {
        const float* xr = x + r * hd;
        uint8_t* o = out + r * (4 + hd);
        float amax = 0.0f;
        for (int i = 0; i < hd; i++) {
            float a = fabsf(xr[i]);
            if (a > amax) amax = a;
        }
        wrf32(o, amax / 127.0f);
        float id = (amax != 0.0f) ? 127.0f / amax : 0.0f;
        for (int i = 0; i < hd; i++) o[4 + i] = (uint8_t)(int8_t)clampi(rne(xr[i] * id), -128, 127);
    }
}

void orc_kv_scores(const uint8_t* q, const uint8_t* kc, float* s, int Hq, int Hkv, int64_t P, int hd, float scale) {
    const int G = Hq / Hkv, rb = 4 + hd;
    for (int h = 0; h < Hq; h++) {
        const uint8_t* qr = q + (int64_t)h * rb;
        const int kvh = h / G;
        for (int64_t p = 0; p < P; p++) {
            const uint8_t* kr = kc + (p * Hkv + kvh) * rb;
            int32_t isum = 0;
            for (int i = 0; i < hd; i++) isum += (int8_t)qr[4 + i] * (int8_t)kr[4 + i];
            float dd = rdf32(qr) * rdf32(kr);
            s[(int64_t)h * P + p] = (dd * (float)isum) * scale;
        }
    }
}

void orc_kv_wsum(const float* w, const uint8_t* vc, double* out, int Hq, int Hkv, int64_t P, int hd) {
    const int G = Hq / Hkv, rb = 4 + hd;
    for (int h = 0; h < Hq; h++) {
        const int kvh = h / G;
        for (int i = 0; i < hd; i++) {
            double acc = 0.0;
            for (int64_t p = 0; p < P; p++) {
                const uint8_t* vr = vc + (p * Hkv + kvh) * rb;
                acc += (double)w[(int64_t)h * P + p] * (double)rdf32(vr) * (double)(int8_t)vr[4 + i];
            }
            out[(int64_t)h * hd + i] = acc;
        }
    }
}

/* ------------------------------------------------------------------------- */
/* RMSNorm ahead of the activation quantizer: [krafla] "Architecture",       */
/* "Data flow for one token" (h = rmsnorm(x) ; qa = quantize_q8(h)).  The     */
/* page gives no formula; reading, the usual definition                       */
/*   h_i = (x_i * s) * w_i,  s = 1 / sqrt(ss / K + eps),  ss = sum_i x_i^2.   */
/* ss is the plain sum of squares, left to right, in binary64 (the square of  */
/* an f32 is exact there) and rounded once to f32; every later step is an f32 */
/* operation rounded once.  A model whose norm scales by 1 + w passes that    */
/* vector as w.                                                               */
/* ------------------------------------------------------------------------- */
void orc_rmsnorm(const float* x, const float* w, float eps, float* h, int64_t M, int64_t K) {
    for (int64_t t = 0; t < M; t++) {
        const float* xr = x + t * K;
        double ss = 0.0;
        for (int64_t i = 0; i < K; i++) ss += (double)xr[i] * (double)xr[i];
        const float mean = (float)ss / (float)K;
        const float sc = 1.0f / sqrtf(mean + eps);
        for (int64_t i = 0; i < K; i++) h[t * K + i] = (xr[i] * sc) * w[i];
    }
}
