/*
 * rem_oracle.c -- plain CPU oracle for the row-exact few-row quantized mat-vec.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg load this library.  It shares no code, header, table or
 * helper with the CUDA path under quantized_few_row_gb300/.
 *
 * What it computes (mlx-native 0.18.0 src/ops/row_exact_matvec.rs, module
 * doc "Row-exact few-row mat-vec" and the RowExactWeight enum):
 *     Wf = dequantize(W)                         (exact f32 weights per format)
 *     y[b, j, i] = sum_k (f64)Wf[b*n + i, k] * (f64)x[b, j, k]   (natural k order)
 *     A[b, j, i] = sum_k |(f64)Wf[b*n + i, k] * (f64)x[b, j, k]| (for the tolerance)
 *
 * Block formats.  The page fixes the block sizes (the *_BLOCK_BYTES /
 * *_BLOCK_VALUES constants and RowExactWeight::row_bytes) and names the GGML
 * types (F16, Q8_0, Q4_K, Q6_K, Q5_0).  The byte layout inside a block is the
 * public GGML layout of the same name (reading 1 of the oracle notes):
 *   Q8_0  34 B : d f16 | qs int8[32]                    w = d*q
 *   Q5_0  22 B : d f16 | qh u32 | qs u8[16]             q = nibble | qh_bit<<4, w = d*(q-16)
 *   Q4_K 144 B : d f16 | dmin f16 | scales u8[12] | qs u8[128]
 *                8 sub-blocks of 32, 6-bit (sc, mn) packed in scales,
 *                w = (d*sc)*q - (dmin*mn)
 *   Q6_K 210 B : ql u8[128] | qh u8[64] | sc int8[16] | d f16
 *                16 sub-blocks of 16, w = (d*sc)*(q-32)
 * Every f32 step below is one separately rounded IEEE operation (reading 2):
 * the file must be compiled with -ffp-contract=off and without -ffast-math.
 *
 * Quantizers (test-data generators, reading 3) round x/d with roundf (ties
 * away from zero) against the stored fp16 scale.  Parity only depends on
 * the bytes they produce.
 *
 * Dense weights (the row-independent gemv of nuvec-core 0.6.0 src/gpu.rs,
 * gemv_rows: F32, F16 and BF16 matrices under the same row contract):
 *   F32   4 B : one binary32 per element
 *   BF16  2 B : the upper 16 bits of a binary32 (widening is exact; the
 *               "quantizer" rounds binary32 to nearest even)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { W_F16 = 0, W_Q8_0 = 1, W_Q4_K = 2, W_Q6_K = 3, W_Q5_0 = 4, W_F32 = 5, W_BF16 = 6 };

/* ------------------------------------------------------------------ */
/* Block constants (row_exact_matvec.rs, the *_BLOCK_* constants).     */
/* ------------------------------------------------------------------ */

int rem_oracle_block_values(int wtype) {
    switch (wtype) {
    case W_F16: return 1;
    case W_F32: return 1;
    case W_BF16: return 1;
    case W_Q8_0: return 32;
    case W_Q5_0: return 32;
    case W_Q4_K: return 256;
    case W_Q6_K: return 256;
    default: return 0;
    }
}

int rem_oracle_block_bytes(int wtype) {
    switch (wtype) {
    case W_F16: return 2;
    case W_F32: return 4;
    case W_BF16: return 2;
    case W_Q8_0: return 34;
    case W_Q5_0: return 22;
    case W_Q4_K: return 144;
    case W_Q6_K: return 210;
    default: return 0;
    }
}

/* RowExactWeight::row_bytes: bytes of one weight row of k elements. */
uint64_t rem_oracle_row_bytes(int wtype, uint32_t k) {
    int bv = rem_oracle_block_values(wtype);
    if (bv == 0) return 0;
    return (uint64_t)(k / (uint32_t)bv) * (uint64_t)rem_oracle_block_bytes(wtype);
}

/* ------------------------------------------------------------------ */
/* IEEE binary16 <-> binary32, written from the IEEE 754 definition.   */
/* ------------------------------------------------------------------ */

static float bits_to_f32(uint32_t b) { float f; memcpy(&f, &b, 4); return f; }
static uint32_t f32_to_bits(float f) { uint32_t b; memcpy(&b, &f, 4); return b; }

/* Exact widening of a binary16 bit pattern. */
float rem_oracle_h2f(uint16_t h) {
    uint32_t sign = (uint32_t)(h >> 15);
    uint32_t e = (uint32_t)(h >> 10) & 0x1Fu;
    uint32_t man = (uint32_t)h & 0x3FFu;
    if (e == 0) {
        /* zero or subnormal: man * 2^-24, exact in f32 */
        float v = (float)man * 0x1p-24f;
        return sign ? -v : v;
    }
    if (e == 31) /* inf / NaN: keep the payload */
        return bits_to_f32((sign << 31) | 0x7F800000u | (man << 13));
    return bits_to_f32((sign << 31) | ((e + 112u) << 23) | (man << 13));
}

/* Narrow f32 to binary16.  mode 0: round to nearest, ties to even.
 * mode 1: round toward +infinity. */
static uint16_t f2h_mode(float f, int mode) {
    uint32_t x = f32_to_bits(f);
    uint32_t sign = x >> 31;
    uint32_t ax = x & 0x7FFFFFFFu;
    uint16_t hs = (uint16_t)(sign << 15);
    if (ax > 0x7F800000u) return (uint16_t)(hs | 0x7E00u);      /* NaN */
    if (ax == 0x7F800000u) return (uint16_t)(hs | 0x7C00u);     /* inf */
    if (ax == 0) return hs;                                      /* +-0 */

    /* |f| = sig * 2^ex exactly, sig < 2^24 */
    uint32_t e = ax >> 23;
    uint32_t sig = (e == 0) ? (ax & 0x7FFFFFu) : ((ax & 0x7FFFFFu) | 0x800000u);
    int ex = (e == 0) ? -149 : (int)e - 150;
    /* floor(log2 |f|) */
    int lg = ex;
    { uint32_t s = sig; while (s > 1) { s >>= 1; ++lg; } }
    /* binary16 quantum at this magnitude: 2^(lg-10), never below 2^-24 */
    int qe = lg - 10;
    if (qe < -24) qe = -24;
    int shift = qe - ex; /* bits of sig below the quantum */
    uint64_t q;
    int inexact, above_half, at_half;
    if (shift <= 0) {
        q = (uint64_t)sig << (-shift);
        inexact = 0; above_half = 0; at_half = 0;
    } else if (shift >= 40) {
        q = 0; inexact = 1; above_half = 0; at_half = 0;
    } else {
        uint64_t s64 = sig;
        q = s64 >> shift;
        uint64_t rem = s64 & ((1ull << shift) - 1ull);
        uint64_t half = 1ull << (shift - 1);
        inexact = rem != 0;
        above_half = rem > half;
        at_half = rem == half;
    }
    if (mode == 0) {
        if (above_half || (at_half && (q & 1ull))) q += 1;
    } else {
        /* toward +inf: a positive inexact value rounds up, a negative one
         * truncates toward zero */
        if (inexact && !sign) q += 1;
    }
    /* value = q * 2^qe ; encode */
    if (qe == -24) {
        /* subnormal quantum: q < 1024 is subnormal, q == 1024 is the
         * smallest normal, which the plain encoding q also expresses */
        return (uint16_t)(hs | (uint16_t)q);
    }
    int E = qe + 25; /* biased exponent for q in [1024, 2048) */
    if (q >= 2048) { q >>= 1; E += 1; }
    if (E >= 31) {
        /* overflow: RNE gives inf; toward +inf gives inf for positive and
         * the largest finite magnitude for negative values */
        if (mode == 1 && sign) return (uint16_t)(hs | 0x7BFFu);
        return (uint16_t)(hs | 0x7C00u);
    }
    return (uint16_t)(hs | (uint16_t)(E << 10) | (uint16_t)(q - 1024));
}

uint16_t rem_oracle_f2h_rn(float f) { return f2h_mode(f, 0); }

/* bfloat16: the upper half of a binary32 bit pattern. */
static uint32_t f2u(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    return u;
}
static float u2f(uint32_t u) {
    float f;
    memcpy(&f, &u, 4);
    return f;
}
float rem_oracle_bf2f(uint16_t b) { return u2f((uint32_t)b << 16); }

/* binary32 -> bfloat16, round to nearest, ties to even on the 16 dropped
 * bits; NaN stays NaN (quiet bit set), infinities stay infinite. */
uint16_t rem_oracle_f2bf_rn(float f) {
    uint32_t u = f2u(f);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep = u >> 16, rest = u & 0xFFFFu;
    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) keep += 1u;  /* carries into the exponent */
    return (uint16_t)keep;
}
uint16_t rem_oracle_f2h_ru(float f) { return f2h_mode(f, 1); }

static uint16_t rd16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static uint32_t rd32(const uint8_t* p) {
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}
static void wr16(uint8_t* p, uint16_t v) { p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); }
static void wr32(uint8_t* p, uint32_t v) {
    p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); p[2] = (uint8_t)(v >> 16); p[3] = (uint8_t)(v >> 24);
}

/* ------------------------------------------------------------------ */
/* Dequantizers: one block -> floats, in the oracle's element order.   */
/* ------------------------------------------------------------------ */

static void deq_q8_0(const uint8_t* b, float* out) {
    float d = rem_oracle_h2f(rd16(b));
    for (int e = 0; e < 32; ++e) out[e] = d * (float)(int8_t)b[2 + e];
}

static void deq_q5_0(const uint8_t* b, float* out) {
    float d = rem_oracle_h2f(rd16(b));
    uint32_t qh = rd32(b + 2);
    const uint8_t* qs = b + 6;
    for (int e = 0; e < 32; ++e) {
        int nib = (e < 16) ? (qs[e] & 0x0F) : (qs[e - 16] >> 4);
        int hb = (int)((qh >> e) & 1u);
        int q = nib | (hb << 4);
        out[e] = d * (float)(q - 16);
    }
}

/* 6-bit sub-block scale and min of a Q4_K block. */
static void q4k_scale_min(const uint8_t* sc12, int s, int* sc, int* mn) {
    if (s < 4) {
        *sc = sc12[s] & 63;
        *mn = sc12[s + 4] & 63;
    } else {
        *sc = (sc12[s + 4] & 0x0F) | ((sc12[s - 4] >> 6) << 4);
        *mn = (sc12[s + 4] >> 4) | ((sc12[s] >> 6) << 4);
    }
}

static void deq_q4_k(const uint8_t* b, float* out) {
    float d = rem_oracle_h2f(rd16(b));
    float dmin = rem_oracle_h2f(rd16(b + 2));
    const uint8_t* sc12 = b + 4;
    const uint8_t* qs = b + 16;
    for (int e = 0; e < 256; ++e) {
        int c = e / 64;           /* 64-value chunk, 32 qs bytes each   */
        int hi = (e % 64) >= 32;  /* second half: high nibbles          */
        int l = e % 32;
        int s = 2 * c + hi;       /* sub-block of 32                    */
        int sc, mn;
        q4k_scale_min(sc12, s, &sc, &mn);
        uint8_t byte = qs[32 * c + l];
        int q = hi ? (byte >> 4) : (byte & 0x0F);
        float scale = d * (float)sc;
        float minv = dmin * (float)mn;
        float prod = scale * (float)q;
        out[e] = prod - minv;
    }
}

static void deq_q6_k(const uint8_t* b, float* out) {
    const uint8_t* ql = b;
    const uint8_t* qh = b + 128;
    const int8_t* sc = (const int8_t*)(b + 192);
    float d = rem_oracle_h2f(rd16(b + 208));
    for (int e = 0; e < 256; ++e) {
        int h = e / 128;
        int t = (e % 128) / 32;
        int l = e % 32;
        uint8_t lb = ql[64 * h + l + 32 * (t & 1)];
        int lo = (t < 2) ? (lb & 0x0F) : (lb >> 4);
        int hb = (qh[32 * h + l] >> (2 * t)) & 3;
        int q = lo | (hb << 4);
        int s = 8 * h + 2 * t + l / 16;
        float scale = d * (float)sc[s];
        out[e] = scale * (float)(q - 32);
    }
}

/* Dequantize one row of k elements. */
static void deq_row(int wtype, const uint8_t* row, uint32_t k, float* out) {
    switch (wtype) {
    case W_F16:
        for (uint32_t e = 0; e < k; ++e) out[e] = rem_oracle_h2f(rd16(row + 2 * e));
        break;
    case W_BF16:
        for (uint32_t e = 0; e < k; ++e) out[e] = rem_oracle_bf2f(rd16(row + 2 * e));
        break;
    case W_F32:
        for (uint32_t e = 0; e < k; ++e) {
            const uint8_t* p = row + 4 * e;
            out[e] = u2f((uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24));
        }
        break;
    case W_Q8_0:
        for (uint32_t blk = 0; blk < k / 32; ++blk) deq_q8_0(row + 34 * blk, out + 32 * blk);
        break;
    case W_Q5_0:
        for (uint32_t blk = 0; blk < k / 32; ++blk) deq_q5_0(row + 22 * blk, out + 32 * blk);
        break;
    case W_Q4_K:
        for (uint32_t blk = 0; blk < k / 256; ++blk) deq_q4_k(row + 144 * blk, out + 256 * blk);
        break;
    case W_Q6_K:
        for (uint32_t blk = 0; blk < k / 256; ++blk) deq_q6_k(row + 210 * blk, out + 256 * blk);
        break;
    default:
        break;
    }
}

/* Dequantize `rows` rows of k elements into out[rows][k].  0 on success. */
int rem_oracle_dequantize(const uint8_t* w, int wtype, uint32_t rows, uint32_t k, float* out) {
    uint64_t rb = rem_oracle_row_bytes(wtype, k);
    if (rb == 0) return -1;
    for (uint32_t r = 0; r < rows; ++r) deq_row(wtype, w + (uint64_t)r * rb, k, out + (uint64_t)r * k);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Quantizers (test-data generators).                                  */
/* ------------------------------------------------------------------ */

static int clampi(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }

static void quant_q8_0(const float* v, uint8_t* b) {
    float amax = 0.0f;
    for (int e = 0; e < 32; ++e) { float a = fabsf(v[e]); if (a > amax) amax = a; }
    float dq = amax / 127.0f;
    uint16_t dh = rem_oracle_f2h_rn(dq);
    float d = rem_oracle_h2f(dh);
    wr16(b, dh);
    for (int e = 0; e < 32; ++e) {
        int q = 0;
        if (d != 0.0f) q = clampi((int)roundf(v[e] / d), -127, 127);
        b[2 + e] = (uint8_t)(int8_t)q;
    }
}

static void quant_q5_0(const float* v, uint8_t* b) {
    float amax = 0.0f, vmax = 0.0f;
    for (int e = 0; e < 32; ++e) {
        float a = fabsf(v[e]);
        if (a > amax) { amax = a; vmax = v[e]; }
    }
    float dq = vmax / -16.0f;
    uint16_t dh = rem_oracle_f2h_rn(dq);
    float d = rem_oracle_h2f(dh);
    int q[32];
    for (int e = 0; e < 32; ++e) {
        q[e] = 16;
        if (d != 0.0f) q[e] = clampi((int)roundf(v[e] / d) + 16, 0, 31);
    }
    wr16(b, dh);
    uint32_t qh = 0;
    for (int e = 0; e < 32; ++e) qh |= (uint32_t)((q[e] >> 4) & 1) << e;
    wr32(b + 2, qh);
    for (int i = 0; i < 16; ++i) b[6 + i] = (uint8_t)((q[i] & 0x0F) | ((q[i + 16] & 0x0F) << 4));
}

static void quant_q4_k(const float* v, uint8_t* b) {
    float lo[8], hi[8];
    for (int s = 0; s < 8; ++s) {
        float mnv = 0.0f, mxv = 0.0f; /* range always includes 0 */
        for (int e = 0; e < 32; ++e) {
            float x = v[32 * s + e];
            if (x < mnv) mnv = x;
            if (x > mxv) mxv = x;
        }
        lo[s] = mnv;
        hi[s] = mxv;
    }
    /* 1. dmin covers the most negative sub-block with mn <= 63 */
    float mneg = 0.0f;
    for (int s = 0; s < 8; ++s) if (-lo[s] > mneg) mneg = -lo[s];
    uint16_t dminh = rem_oracle_f2h_ru(mneg / 63.0f);
    float dmin = rem_oracle_h2f(dminh);
    /* 2. per sub-block min multiplier */
    int mn[8];
    for (int s = 0; s < 8; ++s) {
        mn[s] = 0;
        if (dmin > 0.0f) mn[s] = clampi((int)ceilf(-lo[s] / dmin), 0, 63);
    }
    /* 3. d so that 15*d*sc covers hi + dmin*mn with sc <= 63 */
    float range[8], rmax = 0.0f;
    for (int s = 0; s < 8; ++s) {
        float off = dmin * (float)mn[s];
        range[s] = hi[s] + off;
        float r15 = range[s] / 15.0f;
        if (r15 > rmax) rmax = r15;
    }
    uint16_t dh = rem_oracle_f2h_ru(rmax / 63.0f);
    float d = rem_oracle_h2f(dh);
    /* 4. sub-block scales */
    int sc[8];
    for (int s = 0; s < 8; ++s) {
        sc[s] = 0;
        if (d > 0.0f) sc[s] = clampi((int)ceilf(range[s] / 15.0f / d), 1, 63);
    }
    /* 5. codes */
    uint8_t q[256];
    for (int s = 0; s < 8; ++s) {
        float off = dmin * (float)mn[s];
        float den = d * (float)sc[s];
        for (int e = 0; e < 32; ++e) {
            int c = 0;
            if (den > 0.0f) c = clampi((int)roundf((v[32 * s + e] + off) / den), 0, 15);
            q[32 * s + e] = (uint8_t)c;
        }
    }
    /* pack */
    wr16(b, dh);
    wr16(b + 2, dminh);
    uint8_t* s12 = b + 4;
    for (int s = 0; s < 4; ++s) {
        s12[s] = (uint8_t)((sc[s] & 63) | ((sc[s + 4] >> 4) << 6));
        s12[s + 4] = (uint8_t)((mn[s] & 63) | ((mn[s + 4] >> 4) << 6));
        s12[s + 8] = (uint8_t)((sc[s + 4] & 0x0F) | ((mn[s + 4] & 0x0F) << 4));
    }
    uint8_t* qs = b + 16;
    for (int c = 0; c < 4; ++c)
        for (int l = 0; l < 32; ++l)
            qs[32 * c + l] = (uint8_t)(q[64 * c + l] | (q[64 * c + 32 + l] << 4));
}

static void quant_q6_k(const float* v, uint8_t* b) {
    float amax[16], top = 0.0f;
    for (int s = 0; s < 16; ++s) {
        float a = 0.0f;
        for (int e = 0; e < 16; ++e) { float t = fabsf(v[16 * s + e]); if (t > a) a = t; }
        amax[s] = a;
        if (a > top) top = a;
    }
    uint16_t dh = rem_oracle_f2h_ru(top / (31.0f * 127.0f));
    float d = rem_oracle_h2f(dh);
    int sc[16];
    float d31 = 31.0f * d;
    for (int s = 0; s < 16; ++s) {
        sc[s] = 0;
        if (d > 0.0f) sc[s] = clampi((int)ceilf(amax[s] / d31), 0, 127);
    }
    uint8_t q[256];
    for (int s = 0; s < 16; ++s) {
        float den = d * (float)sc[s];
        for (int e = 0; e < 16; ++e) {
            int c = 32;
            if (den > 0.0f) c = clampi((int)roundf(v[16 * s + e] / den) + 32, 0, 63);
            q[16 * s + e] = (uint8_t)c;
        }
    }
    /* pack: the element of (half h, quarter t, lane l) is e = 128h + 32t + l */
    uint8_t* ql = b;
    uint8_t* qh = b + 128;
    memset(ql, 0, 128);
    memset(qh, 0, 64);
    for (int e = 0; e < 256; ++e) {
        int h = e / 128, t = (e % 128) / 32, l = e % 32;
        int lo = q[e] & 0x0F, hb = q[e] >> 4;
        int qi = 64 * h + l + 32 * (t & 1);
        ql[qi] |= (uint8_t)(t < 2 ? lo : (lo << 4));
        qh[32 * h + l] |= (uint8_t)(hb << (2 * t));
    }
    for (int s = 0; s < 16; ++s) b[192 + s] = (uint8_t)(int8_t)sc[s];
    wr16(b + 208, dh);
}

/* Quantize src[rows][k] into `rows` rows of blocks.  F16 rounds to nearest
 * even.  0 on success, -1 on a bad type or a k that is not a multiple of the
 * block. */
int rem_oracle_quantize(const float* src, int wtype, uint32_t rows, uint32_t k, uint8_t* w) {
    int bv = rem_oracle_block_values(wtype);
    if (bv == 0 || k % (uint32_t)bv != 0) return -1;
    uint64_t rb = rem_oracle_row_bytes(wtype, k);
    for (uint32_t r = 0; r < rows; ++r) {
        const float* v = src + (uint64_t)r * k;
        uint8_t* row = w + (uint64_t)r * rb;
        uint32_t nb = k / (uint32_t)bv;
        for (uint32_t blk = 0; blk < nb; ++blk) {
            const float* vb = v + (uint64_t)blk * bv;
            switch (wtype) {
            case W_F16: wr16(row + 2 * blk, rem_oracle_f2h_rn(vb[0])); break;
            case W_BF16: wr16(row + 2 * blk, rem_oracle_f2bf_rn(vb[0])); break;
            case W_F32: {
                uint32_t u = f2u(vb[0]);
                uint8_t* p = row + 4 * blk;
                p[0] = (uint8_t)u; p[1] = (uint8_t)(u >> 8); p[2] = (uint8_t)(u >> 16); p[3] = (uint8_t)(u >> 24);
                break;
            }
            case W_Q8_0: quant_q8_0(vb, row + 34 * blk); break;
            case W_Q5_0: quant_q5_0(vb, row + 22 * blk); break;
            case W_Q4_K: quant_q4_k(vb, row + 144 * blk); break;
            case W_Q6_K: quant_q6_k(vb, row + 210 * blk); break;
            default: return -1;
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* The mat-vec definition in f64.                                      */
/* ------------------------------------------------------------------ */

/*
 * For each listed weight row r (global row = b*n + i, b = r / n, i = r % n)
 * and each input row j < m:
 *     y[c*m + j] = sum_{kk<k} (f64)Wf[r, kk] * (f64)x[b*xbs + j*xrs + kk]
 *     a[c*m + j] = sum_{kk<k} |(f64)Wf[r, kk] * (f64)x[...]|
 * where c indexes the row list.  Summation in natural k order.  Rows are
 * independent, so they run in parallel (OpenMP) without changing results.
 */
int rem_oracle_matvec_rows(const uint8_t* w, int wtype, uint32_t n, uint32_t k,
                           const float* x, uint32_t m, uint64_t xrs, uint64_t xbs,
                           const uint64_t* rows, uint64_t nrows, double* y, double* a) {
    uint64_t rb = rem_oracle_row_bytes(wtype, k);
    if (rb == 0 || n == 0 || m == 0) return -1;
    int err = 0;
#pragma omp parallel
    {
        float* wf = (float*)malloc(sizeof(float) * (size_t)k);
        if (!wf) {
#pragma omp atomic write
            err = -2;
        }
        /* every thread reaches the worksharing loop */
#pragma omp for schedule(dynamic, 16)
        for (int64_t c = 0; c < (int64_t)nrows; ++c) {
            if (!wf) continue;
            uint64_t r = rows[c];
            uint64_t bidx = r / n;
            deq_row(wtype, w + r * rb, k, wf);
            for (uint32_t j = 0; j < m; ++j) {
                const float* xr = x + bidx * xbs + (uint64_t)j * xrs;
                double s = 0.0, sa = 0.0;
                for (uint32_t kk = 0; kk < k; ++kk) {
                    double p = (double)wf[kk] * (double)xr[kk];
                    s += p;
                    sa += fabs(p);
                }
                y[(uint64_t)c * m + j] = s;
                a[(uint64_t)c * m + j] = sa;
            }
        }
        free(wf);
    }
    return err;
}

/* ------------------------------------------------------------------ */
/* Affine quantization (nuvec-core 0.6.0 src/gpu.rs: Quantize /         */
/* Dequantize / QuantizedMatmul in QuantMode::Affine with (group_size,  */
/* bits), and pack_factor: values per packing unit -- 8 for 3 and 5     */
/* bits, 4 for 6 bits, 32/bits for 4 and 8 bits -- so a packing unit is */
/* a whole number of bytes (3, 5, 3, 4, 4).  The pages give no element  */
/* formula or bit order; the reading:                                   */
/*   codes   rows x (k*bits/32) uint32 words, little-endian: a row's    */
/*           codes are one bit stream, byte j holding stream bits       */
/*           8j .. 8j+7 (bit 0 lowest), and code i occupies stream bits */
/*           [bits*i, bits*i + bits), lowest bit first (for 4 and 8     */
/*           bits: word i / (32/bits), bits bits*(i % (32/bits)));      */
/*   scales, biases  rows x (k/group_size) binary16, one per group;     */
/*   w = fl(fl(scale*q) + bias), the product rounded, then the add.     */
/* ------------------------------------------------------------------ */

static int affine_ok(int bits, int gs, uint32_t k) {
    return (bits == 3 || bits == 4 || bits == 5 || bits == 6 || bits == 8) && (gs == 32 || gs == 64 || gs == 128) &&
           k > 0 && k % (uint32_t)gs == 0;
}

/* Code i of a row whose code bytes (k*bits/8 of them) start at cb. */
static uint32_t affine_code(const uint8_t* cb, int bits, uint32_t k, uint32_t i) {
    const uint64_t bit = (uint64_t)bits * i, nbytes = (uint64_t)k * (uint64_t)bits / 8;
    uint32_t v = cb[bit / 8];
    if (bit / 8 + 1 < nbytes) v |= (uint32_t)cb[bit / 8 + 1] << 8;
    return (v >> (bit % 8)) & ((1u << bits) - 1u);
}

static void deq_affine_row(const uint32_t* codes, const uint16_t* sc, const uint16_t* bi, int bits, int gs,
                           uint32_t k, float* out) {
    const uint8_t* cb = (const uint8_t*)codes;
    for (uint32_t i = 0; i < k; ++i) {
        uint32_t q = affine_code(cb, bits, k, i);
        float s = rem_oracle_h2f(sc[i / (uint32_t)gs]), b = rem_oracle_h2f(bi[i / (uint32_t)gs]);
        float p = s * (float)q;
        out[i] = p + b;
    }
}

/* Dequantize `rows` rows of k elements into out[rows][k].  0 on success. */
int rem_oracle_affine_dequantize(const uint32_t* codes, const uint16_t* scales, const uint16_t* biases, int bits,
                                 int gs, uint32_t rows, uint32_t k, float* out) {
    if (!affine_ok(bits, gs, k)) return -1;
    const uint64_t cw = (uint64_t)k * bits / 32, ng = k / (uint32_t)gs;
    for (uint32_t r = 0; r < rows; ++r)
        deq_affine_row(codes + r * cw, scales + r * ng, biases + r * ng, bits, gs, k, out + (uint64_t)r * k);
    return 0;
}

/* Test-data quantizer: per group lo = min, hi = max, scale = fp16_rn((hi -
 * lo) / (2^bits - 1)), bias = fp16_rn(lo), q = clamp(roundf((v - bias) /
 * scale), 0, 2^bits - 1) against the stored scale and bias (q = 0 when the
 * stored scale is 0).  0 on success. */
int rem_oracle_affine_quantize(const float* src, int bits, int gs, uint32_t rows, uint32_t k, uint32_t* codes,
                               uint16_t* scales, uint16_t* biases) {
    if (!affine_ok(bits, gs, k)) return -1;
    const uint32_t qmax = (1u << bits) - 1u;
    const uint64_t cw = (uint64_t)k * bits / 32, ng = k / (uint32_t)gs;
    for (uint32_t r = 0; r < rows; ++r) {
        const float* v = src + (uint64_t)r * k;
        uint32_t* cr = codes + r * cw;
        uint8_t* cb = (uint8_t*)cr;
        for (uint64_t w = 0; w < cw; ++w) cr[w] = 0;
        for (uint64_t g = 0; g < ng; ++g) {
            const float* vg = v + g * gs;
            float lo = vg[0], hi = vg[0];
            for (int e = 1; e < gs; ++e) {
                if (vg[e] < lo) lo = vg[e];
                if (vg[e] > hi) hi = vg[e];
            }
            uint16_t sh = rem_oracle_f2h_rn((hi - lo) / (float)qmax), bh = rem_oracle_f2h_rn(lo);
            scales[r * ng + g] = sh;
            biases[r * ng + g] = bh;
            float sf = rem_oracle_h2f(sh), bf = rem_oracle_h2f(bh);
            for (int e = 0; e < gs; ++e) {
                long q = 0;
                if (sf != 0.0f) {
                    q = (long)roundf((vg[e] - bf) / sf);
                    if (q < 0) q = 0;
                    if (q > (long)qmax) q = (long)qmax;
                }
                /* code i -> stream bits [bits*i, bits*i + bits) */
                uint64_t bit = (g * gs + (uint64_t)e) * (uint64_t)bits;
                uint32_t sh = (uint32_t)q << (bit % 8);
                cb[bit / 8] |= (uint8_t)(sh & 0xFFu);
                if (sh >> 8) cb[bit / 8 + 1] |= (uint8_t)(sh >> 8);
            }
        }
    }
    return 0;
}

/* f64 y and sum|w*x| for selected global rows of an affine weight (as
 * rem_oracle_matvec_rows). */
int rem_oracle_affine_matvec_rows(const uint32_t* codes, const uint16_t* scales, const uint16_t* biases, int bits,
                                  int gs, uint32_t n, uint32_t k, const float* x, uint32_t m, uint64_t xrs,
                                  uint64_t xbs, const uint64_t* rows, uint64_t nrows, double* y, double* a) {
    if (!affine_ok(bits, gs, k) || n == 0 || m == 0) return -1;
    const uint64_t cw = (uint64_t)k * bits / 32, ng = k / (uint32_t)gs;
    int err = 0;
#pragma omp parallel
    {
        float* wf = (float*)malloc(sizeof(float) * (size_t)k);
        if (!wf) {
#pragma omp atomic write
            err = -2;
        }
#pragma omp for schedule(dynamic, 16)
        for (int64_t c = 0; c < (int64_t)nrows; ++c) {
            if (!wf) continue;
            uint64_t r = rows[c], bidx = r / n;
            deq_affine_row(codes + r * cw, scales + r * ng, biases + r * ng, bits, gs, k, wf);
            for (uint32_t j = 0; j < m; ++j) {
                const float* xr = x + bidx * xbs + (uint64_t)j * xrs;
                double sum = 0.0, sa = 0.0;
                for (uint32_t kk = 0; kk < k; ++kk) {
                    double p = (double)wf[kk] * (double)xr[kk];
                    sum += p;
                    sa += fabs(p);
                }
                y[(uint64_t)c * m + j] = sum;
                a[(uint64_t)c * m + j] = sa;
            }
        }
        free(wf);
    }
    return err;
}

/* Threads the parallel region above uses. */
int rem_oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Array helpers for the binding: elementwise conversions. */
void rem_oracle_h2f_array(const uint16_t* h, float* out, uint64_t count) {
    for (uint64_t i = 0; i < count; ++i) out[i] = rem_oracle_h2f(h[i]);
}
void rem_oracle_f2h_array(const float* f, uint16_t* out, uint64_t count, int mode) {
    for (uint64_t i = 0; i < count; ++i) out[i] = f2h_mode(f[i], mode);
}
void rem_oracle_bf2f_array(const uint16_t* b, float* out, uint64_t count) {
    for (uint64_t i = 0; i < count; ++i) out[i] = rem_oracle_bf2f(b[i]);
}
void rem_oracle_f2bf_array(const float* f, uint16_t* out, uint64_t count) {
    for (uint64_t i = 0; i < count; ++i) out[i] = rem_oracle_f2bf_rn(f[i]);
}
