/*
 * oracle.c -- plain, slow CPU oracle for block-32 quantized matmul over tiled weights.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the CPU-baseline leg of the
 * benchmark load this file (as liboracle.so, through oracle/__init__.py).  The product library never
 * links, includes or calls it, and this file includes nothing from the product sources.
 *
 * Sources followed ("Hexagon backend developer details", section "Tiled Weight Formats"):
 *   - "Tile Dimensions and Grid Layout": n_k_tiles = K/32, n_col_tiles = (N+31)/32,
 *     tile_idx = ct*n_k_tiles + kt, tile_offset = tile_idx*tile_size.
 *   - "Block-32 Quantized Formats": the Q4_0 / IQ4_NL 576-byte tile (column pair cp, byte
 *     cp*32+row = (q[row][2cp+1] << 4) | q[row][2cp], FP16 row scales at 512+2*row) and the Q8_0
 *     1088-byte tile (bytes cp*64+2*row+0/1 = q[row][2cp] / q[row][2cp+1], FP16 row scales at
 *     1024+2*row); IQ4_NL dequantizes through a 16-entry non-linear table times the row scale.
 *     The MXFP4 544-byte tile keeps the Q4_0 nibble layout for 4-bit E2M1 codes and stores one E8M0
 *     exponent byte per row at 512+row; it dequantizes as the FP4 value of the code times the
 *     power-of-two fp16 scale whose bits are clamp(e - 112, 0, 30) << 10.  The Q4_1 640-byte tile
 *     keeps the Q4_0 nibble layout and stores the FP16 pair (d, m) of a row at 512+4*row and
 *     514+4*row.
 *
 * Readings where the pages are silent:
 *   - Flat (untiled) rows are GGML blocks: Q4_0 / IQ4_NL = {fp16 d; u8 qs[16]} (18 B), element j in
 *     the low nibble of qs[j] and element j+16 in its high nibble; Q8_0 = {fp16 d; i8 qs[32]} (34 B).
 *   - Rows past N in the last column tile are zero bytes (d = 0, quants 0).
 *   - Activation quantization (Q8_0, per 32 elements): amax = max|x|, d = amax/127, id = d ? 1/d : 0,
 *     q = round-half-away(x*id) clamped to [-127,127] (a NaN product, 0*inf, gives 0), stored d = fp16(d).
 *   - Weight quantizers (test-data generation): Q4_0 takes the signed element of largest magnitude m,
 *     d = m/-8, id = d ? 1/d : 0, q = min(15, trunc(x*id + 8.5)) (0 for a NaN or negative value);
 *     Q8_0 uses the activation rule;
 *     IQ4_NL takes d = m/lut[0], d16 = fp16(d), and for each x the index i minimising
 *     |x - f32(d16)*lut[i]| (lowest index on ties).
 *   - The IQ4_NL table itself is not printed on the pages; the built-in one holds the 16 levels of
 *     GGML's published IQ4_NL format, and callers may pass another table in.
 *   - Q4_1: "m (min)" read as the GGML affine rule, weight = d*q + m; flat block {fp16 d; fp16 m;
 *     u8 qs[16]} (20 B, nibble order as Q4_0).  So a block adds d_a * m_w * sum_j a_q[j] to the
 *     product.  Quantizer (test data): min and max of the block, d = (max - min)/15, id = d ? 1/d : 0,
 *     q = min(15, trunc((x - min)*id + 0.5)) (0 for NaN), d and m = min stored as fp16.
 *   - MXFP4: the flat block is {u8 e; u8 qs[16]} (17 B, nibble order as Q4_0); the FP4 table is the
 *     OCP E2M1 code set {0, 0.5, 1, 1.5, 2, 3, 4, 6} with a sign bit (code = s<<3 | e<<1 | m).
 *     Integer weights are twice the FP4 value (0..12 with sign) and the block scale is half the
 *     fp16 scale, which is the same product.  Quantizer (test data): e = floor(log2 amax) - 2 + 127
 *     (0 for an all-zero block, clamped to 0..254), then the nearest FP4 level under the dequantizing
 *     scale, lowest code on ties.
 *   - Q4_K ("K-Quants Formats": the Q4_1 tile, each 256-k super-block split along K into 8 tiles of 32
 *     k, the row pair being (d * sc, -dmin * m) as FP16).  The flat super-block is GGML's block_q4_K,
 *     which the pages do not print: {fp16 d; fp16 dmin; u8 scales[12]; u8 qs[128]} (144 B per 256
 *     weights).  Sub-block j (0..7) has a 6-bit scale sc_j and min m_j packed in scales[]: for j < 4
 *     the low 6 bits of scales[j] and scales[j+4]; for j >= 4 the low and high nibble of scales[j+4]
 *     plus, as bits 4..5, the top two bits of scales[j-4] and scales[j].  Weight i of sub-block j is
 *     nibble (j & 1) of qs[32*(j/2) + i], worth d*sc_j*q - dmin*m_j.  The tile row pair is
 *     fp16(f32(d)*sc_j) and fp16(-(f32(dmin)*m_j)) (exact fp32 products, rounded to nearest even).
 *     Quantizer (test data): per sub-block mn = min(0, min x), range = max x - mn, scale = range/15,
 *     min = -mn; d = max scale/63, dmin = max min/63 (fp16); sc_j, m_j = trunc(v*(63/max) + 0.5)
 *     clamped to 63; then q = min(15, trunc((x + f32(dmin)*m_j) * (1/(f32(d)*sc_j)) + 0.5)).
 *   - Matmul: Y[m,n] = sum_b f64(d_w[n,b]) * f64(d_a[m,b]) * S_b[m,n], where S_b is the exact integer
 *     dot product of the block's integer weights (q-8, q, lut[q]) and activation quants.  The oracle
 *     also returns B[m,n] = sum_b sum_j |d_w*w_int * d_a*q_a|, the scale of the error bound.
 *
 * Build: gcc -O2 -fno-fast-math -ffp-contract=off -fPIC -shared -o liboracle.so oracle.c -lm
 * All float arithmetic below is IEEE binary32 or binary64 as written; there is no FMA contraction.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

enum { ORC_Q4_0 = 0, ORC_Q8_0 = 1, ORC_IQ4_NL = 2, ORC_MXFP4 = 3, ORC_Q4_1 = 4, ORC_Q4_K = 5 };

/* Types whose tile holds a (d, m) pair per row: weight = d*q + m. */
static int affine_tile(int type) { return type == ORC_Q4_1 || type == ORC_Q4_K; }

/* OCP Microscaling FP4 (E2M1): code = sign<<3 | exponent<<1 | mantissa; value = 0.5 * mantissa for
 * exponent 0, else 2^(exponent-1) * (1 + mantissa/2).  Twice the value, as an integer. */
static int e2m1_twice(int code)
{
    int ex = (code >> 1) & 3, mant = code & 1;
    int v2 = (ex == 0) ? mant : (1 << (ex - 1)) * (2 + mant);   /* 2 * value */
    return (code & 8) ? -v2 : v2;
}

/* The pages' E8M0 -> fp16 conversion: fp16 bits clamp(e - 112, 0, 30) << 10, a power of two
 * (2^(e-127) for 113 <= e <= 142), 0 for e <= 112 and 2^15 from e = 142 on. */
uint16_t orc_e8m0_to_f16_bits(int e)
{
    int f = e - 112;
    if (f < 0) f = 0;
    if (f > 30) f = 30;
    return (uint16_t)(f << 10);
}

/* The oracle's own copy of the 16-entry IQ4_NL table.  The pages name the table
 * (iq4_nl_to_fp16_lut) but print no values.  These are the 16 levels of GGML's published IQ4_NL
 * format (its non-linear value table), so that IQ4_NL weights from GGUF files decode to their own
 * values; ascending, lut[0] = -127 the most negative, and not symmetric (the top level is 113). */
const int8_t orc_iq4nl_table[16] = {-127, -104, -83, -65, -49, -35, -22, -10, 1, 13, 25, 38, 53, 69, 89, 113};

/* ------------------------------------------------------------------------------------------------
 * IEEE 754 binary16 <-> binary32, written from the format definition (1 sign bit, 5 exponent bits
 * with bias 15, 10 fraction bits; subnormals when the exponent field is 0; inf/NaN when it is 31).
 * Conversion to half rounds to nearest, ties to even, and overflows to infinity.
 * ---------------------------------------------------------------------------------------------- */
static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float bits_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

float orc_f16_to_f32(uint16_t h)
{
    uint32_t sign = (uint32_t)(h >> 15) & 1u;
    uint32_t expo = (uint32_t)(h >> 10) & 0x1Fu;
    uint32_t frac = (uint32_t)h & 0x3FFu;
    double mag;
    if (expo == 0) {
        mag = ldexp((double)frac, -24);                 /* subnormal: frac * 2^-24 */
    } else if (expo == 31) {
        if (frac != 0) return bits_f32(0x7FC00000u | (sign << 31));
        return sign ? -INFINITY : INFINITY;
    } else {
        mag = ldexp((double)(frac | 0x400u), (int)expo - 25);  /* 1.frac * 2^(e-15) */
    }
    return (float)(sign ? -mag : mag);                  /* exact: every half is a float */
}

uint16_t orc_f32_to_f16(float f)
{
    uint32_t u = f32_bits(f);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    if (isnan(f)) return (uint16_t)(sign | 0x7E00u);
    double a = fabs((double)f);
    if (isinf(f) || a >= 65520.0) return (uint16_t)(sign | 0x7C00u);  /* >= max half + half ulp */
    if (a == 0.0) return sign;
    /* Find the half-precision quantum for this magnitude: 2^-24 for subnormals, else 2^(e-10). */
    int e;
    frexp(a, &e);                      /* a = m * 2^e with m in [0.5, 1) */
    int unbiased = e - 1;              /* a in [2^unbiased, 2^(unbiased+1)) */
    int qexp = unbiased < -14 ? -24 : unbiased - 10;
    double scaled = ldexp(a, -qexp);   /* exact: a is a float, scaling by a power of two */
    double fl = floor(scaled);
    double rem = scaled - fl;
    double n = fl;
    if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0)) n = fl + 1.0;
    /* n * 2^qexp is the rounded magnitude; re-encode it. */
    double r = ldexp(n, qexp);
    if (r >= 65520.0) return (uint16_t)(sign | 0x7C00u);
    if (r < ldexp(1.0, -14)) {         /* subnormal (or rounded up to the smallest normal) */
        uint32_t m = (uint32_t)ldexp(r, 24);
        if (m >= 0x400u) return (uint16_t)(sign | 0x0400u);
        return (uint16_t)(sign | m);
    }
    int re;
    frexp(r, &re);
    int ub = re - 1;
    uint32_t mant = (uint32_t)(ldexp(r, -ub) * 1024.0) - 1024u;
    return (uint16_t)(sign | (uint16_t)((ub + 15) << 10) | (uint16_t)mant);
}

/* ------------------------------------------------------------------------------------------------
 * Sizes ("Block-32 Quantized Formats"; "Tile Dimensions and Grid Layout").
 * ---------------------------------------------------------------------------------------------- */
int64_t orc_block_bytes(int type)
{
    if (type == ORC_Q4_0 || type == ORC_IQ4_NL) return 18;  /* fp16 d + 16 bytes of nibbles */
    if (type == ORC_Q8_0) return 34;                        /* fp16 d + 32 int8 */
    if (type == ORC_MXFP4) return 17;                       /* E8M0 e + 16 bytes of nibbles */
    if (type == ORC_Q4_1) return 20;                        /* fp16 d + fp16 m + 16 bytes of nibbles */
    if (type == ORC_Q4_K) return 144;                       /* one super-block of 256 weights */
    return 0;
}

/* Bytes of one flat row of K weights. */
int64_t orc_row_bytes(int type, int64_t K)
{
    if (type == ORC_Q4_K) return K / 256 * 144;
    return K / 32 * orc_block_bytes(type);
}

int64_t orc_tile_bytes(int type)
{
    if (type == ORC_Q4_0 || type == ORC_IQ4_NL) return 576;  /* 512 quant bytes + 32 fp16 scales */
    if (type == ORC_Q8_0) return 1088;                       /* 1024 quant bytes + 32 fp16 scales */
    if (type == ORC_MXFP4) return 544;                       /* 512 quant bytes + 32 E8M0 exponents */
    if (type == ORC_Q4_1 || type == ORC_Q4_K) return 640;    /* 512 quant bytes + 32 fp16 (d, m) pairs */
    return 0;
}

int64_t orc_tile_index(int64_t ct, int64_t kt, int64_t n_k_tiles) { return ct * n_k_tiles + kt; }

int64_t orc_tiled_bytes(int type, int64_t K, int64_t N)
{
    int64_t n_k_tiles = K / 32;
    int64_t n_col_tiles = (N + 31) / 32;
    return n_col_tiles * n_k_tiles * orc_tile_bytes(type);
}

/* ------------------------------------------------------------------------------------------------
 * Flat GGML block access (reading of the pages' "flat row-major GGML layouts").
 * Element j (0..31) of a 4-bit block: qs[j] low nibble for j < 16, qs[j-16] high nibble otherwise.
 * ---------------------------------------------------------------------------------------------- */
static uint16_t load_u16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static void store_u16(uint8_t *p, uint16_t v) { p[0] = (uint8_t)(v & 0xFF); p[1] = (uint8_t)(v >> 8); }

/* Bytes before the quants in a flat block: the fp16 scale, or MXFP4's one exponent byte. */
static int flat_head(int type) { return type == ORC_MXFP4 ? 1 : (type == ORC_Q4_1 ? 4 : 2); }

static int flat_code(int type, const uint8_t *blk, int j)
{
    const uint8_t *qs = blk + flat_head(type);
    if (type == ORC_Q8_0) return (int)(int8_t)qs[j];
    if (j < 16) return qs[j] & 0x0F;
    return qs[j - 16] >> 4;
}

static void flat_set_code(int type, uint8_t *blk, int j, int code)
{
    uint8_t *qs = blk + flat_head(type);
    if (type == ORC_Q8_0) { qs[j] = (uint8_t)(int8_t)code; return; }
    if (j < 16) qs[j] = (uint8_t)((qs[j] & 0xF0) | (code & 0x0F));
    else qs[j - 16] = (uint8_t)((qs[j - 16] & 0x0F) | ((code & 0x0F) << 4));
}

/* Integer weight value of a code: Q4_0 q-8, Q8_0 q, IQ4_NL lut[q] (IQ4_NL per "Block-32 Quantized
 * Formats": the index is looked up in the 16-entry table, then scaled by the row scale). */
static int weight_int(int type, int code, const int8_t *lut)
{
    if (type == ORC_Q4_0) return code - 8;
    if (type == ORC_Q8_0) return code;
    if (type == ORC_MXFP4) return e2m1_twice(code & 15);
    if (affine_tile(type)) return code;
    return (int)lut[code & 15];
}

/* Scale of a block's integer weights: the fp16 scale (Q4_1: d), or for MXFP4 half the fp16 power of
 * two made from the exponent byte (the integer weights are twice the FP4 values). */
/* The additive min of a block (Q4_1 only; 0 otherwise). */
static double block_min(int type, const uint8_t *scale_bytes)
{
    if (affine_tile(type)) return (double)orc_f16_to_f32(load_u16(scale_bytes + 2));
    return 0.0;
}

static double block_scale(int type, const uint8_t *scale_bytes)
{
    if (type == ORC_MXFP4) return 0.5 * (double)orc_f16_to_f32(orc_e8m0_to_f16_bits(scale_bytes[0]));
    return (double)orc_f16_to_f32(load_u16(scale_bytes));
}

/* ------------------------------------------------------------------------------------------------
 * Quantization of one 32-element block.
 * ---------------------------------------------------------------------------------------------- */

/* Q8_0 rule, used for activations and Q8_0 weights.  q[] and the fp16 scale are written. */
void orc_quantize_block_q8_0(const float *x, int8_t *q, uint16_t *d16)
{
    float amax = 0.0f;
    for (int j = 0; j < 32; ++j) {
        float a = fabsf(x[j]);
        if (a > amax) amax = a;
    }
    float d = amax / 127.0f;
    float id = (d != 0.0f) ? 1.0f / d : 0.0f;
    for (int j = 0; j < 32; ++j) {
        float v = x[j] * id;
        float r;
        if (isnan(v)) r = 0.0f;              /* 0 * inf when 1/d overflowed */
        else r = roundf(v);                  /* round half away from zero */
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        q[j] = (int8_t)r;
    }
    *d16 = orc_f32_to_f16(d);
}

/* Q4_0 rule: signed max-magnitude element m (first on ties), d = m / -8, q = min(15, trunc(x*id+8.5)). */
static void quantize_block_q4_0(const float *x, uint8_t *codes, uint16_t *d16)
{
    float amax = 0.0f, m = 0.0f;
    for (int j = 0; j < 32; ++j) {
        if (fabsf(x[j]) > amax) { amax = fabsf(x[j]); m = x[j]; }
    }
    float d = m / -8.0f;
    float id = (d != 0.0f) ? 1.0f / d : 0.0f;
    for (int j = 0; j < 32; ++j) {
        float v = x[j] * id + 8.5f;          /* two roundings: product, then sum (no FMA) */
        int c;
        if (!(v >= 0.0f)) c = 0;             /* NaN (0 * inf) or negative */
        else if (v >= 15.0f) c = 15;         /* min(15, .) taken before the conversion */
        else c = (int)v;                     /* truncation toward zero */
        codes[j] = (uint8_t)c;
    }
    *d16 = orc_f32_to_f16(d);
}

/* IQ4_NL rule: d = m / lut[0], then nearest table entry to x under the stored fp16 scale. */
static void quantize_block_iq4_nl(const float *x, const int8_t *lut, uint8_t *codes, uint16_t *d16)
{
    float amax = 0.0f, m = 0.0f;
    for (int j = 0; j < 32; ++j) {
        if (fabsf(x[j]) > amax) { amax = fabsf(x[j]); m = x[j]; }
    }
    float d = m / (float)lut[0];
    *d16 = orc_f32_to_f16(d);
    float ds = orc_f16_to_f32(*d16);
    for (int j = 0; j < 32; ++j) {
        int best = 0;
        float best_err = INFINITY;
        for (int i = 0; i < 16; ++i) {
            float level = ds * (float)lut[i];
            float err = fabsf(x[j] - level);
            if (err < best_err) { best_err = err; best = i; }
        }
        codes[j] = (uint8_t)best;
    }
}

/* Q4_1 rule: d = (max - min)/15, q = min(15, trunc((x - min)*(1/d) + 0.5)), m = min. */
static void quantize_block_q4_1(const float *x, uint8_t *codes, uint16_t *d16, uint16_t *m16)
{
    float mn = INFINITY, mx = -INFINITY;
    for (int j = 0; j < 32; ++j) {
        if (x[j] < mn) mn = x[j];
        if (x[j] > mx) mx = x[j];
    }
    float d = (mx - mn) / 15.0f;
    float id = (d != 0.0f) ? 1.0f / d : 0.0f;
    for (int j = 0; j < 32; ++j) {
        float v = (x[j] - mn) * id + 0.5f;   /* three roundings: difference, product, sum (no FMA) */
        int c;
        if (!(v >= 0.0f)) c = 0;             /* NaN */
        else if (v >= 15.0f) c = 15;
        else c = (int)v;                     /* truncation toward zero */
        codes[j] = (uint8_t)c;
    }
    *d16 = orc_f32_to_f16(d);
    *m16 = orc_f32_to_f16(mn);
}

/* MXFP4 rule: e = floor(log2 amax) - 2 + 127 (so that amax / 2^(e-127) lies in [4, 8)), 0 for an
 * all-zero block, clamped to 0..254; then the code whose level s * fp4(code) is nearest to x, where s
 * is the dequantizing scale (the pages' fp16 power of two), lowest code on ties. */
static void quantize_block_mxfp4(const float *x, uint8_t *codes, uint8_t *e_out)
{
    float amax = 0.0f;
    for (int j = 0; j < 32; ++j)
        if (fabsf(x[j]) > amax) amax = fabsf(x[j]);
    int e = 0;
    if (amax > 0.0f) {
        int ex;
        (void)frexpf(amax, &ex);             /* amax = f * 2^ex, f in [0.5, 1): floor(log2 amax) = ex - 1 */
        e = (ex - 1) - 2 + 127;
        if (e < 0) e = 0;
        if (e > 254) e = 254;
    }
    *e_out = (uint8_t)e;
    const float s = orc_f16_to_f32(orc_e8m0_to_f16_bits(e));
    for (int j = 0; j < 32; ++j) {
        int best = 0;
        float best_err = INFINITY;
        for (int i = 0; i < 16; ++i) {
            float level = s * (0.5f * (float)e2m1_twice(i));
            float err = fabsf(x[j] - level);
            if (err < best_err) { best_err = err; best = i; }
        }
        codes[j] = (uint8_t)best;
    }
}

/* Q4_K super-block access.  scales[] packing of the 6-bit (sc, m) of sub-block j, see the header. */
static void q4k_scale_min(const uint8_t *scales, int j, int *sc, int *m)
{
    if (j < 4) {
        *sc = scales[j] & 63;
        *m = scales[j + 4] & 63;
    } else {
        *sc = (scales[j + 4] & 0x0F) | ((scales[j - 4] >> 6) << 4);
        *m = (scales[j + 4] >> 4) | ((scales[j] >> 6) << 4);
    }
}

static int q4k_code(const uint8_t *sb, int j, int i) { return (sb[16 + 32 * (j / 2) + i] >> (4 * (j & 1))) & 15; }

static int clamp63(float v)   /* trunc(v) for v >= 0, clamped to 0..63 (0 for NaN) */
{
    if (!(v >= 0.0f)) return 0;
    if (v >= 63.0f) return 63;
    return (int)v;
}

static void quantize_superblock_q4_k(const float *x, uint8_t *sb)
{
    float scale[8], mins[8], max_scale = 0.0f, max_min = 0.0f;
    for (int j = 0; j < 8; ++j) {
        const float *xj = x + 32 * j;
        float mn = 0.0f, mx = xj[0];
        for (int i = 0; i < 32; ++i) {
            if (xj[i] < mn) mn = xj[i];
            if (xj[i] > mx) mx = xj[i];
        }
        float range = mx - mn;
        if (!(range > 0.0f)) range = 0.0f;
        scale[j] = range / 15.0f;
        mins[j] = 0.0f - mn;
        if (scale[j] > max_scale) max_scale = scale[j];
        if (mins[j] > max_min) max_min = mins[j];
    }
    const float isc = max_scale > 0.0f ? 63.0f / max_scale : 0.0f;
    const float imn = max_min > 0.0f ? 63.0f / max_min : 0.0f;
    const uint16_t d16 = orc_f32_to_f16(max_scale / 63.0f), dmin16 = orc_f32_to_f16(max_min / 63.0f);
    int sc[8], m[8];
    for (int j = 0; j < 8; ++j) {
        sc[j] = clamp63(scale[j] * isc + 0.5f);
        m[j] = clamp63(mins[j] * imn + 0.5f);
    }
    memset(sb, 0, 144);
    store_u16(sb, d16);
    store_u16(sb + 2, dmin16);
    for (int i = 0; i < 4; ++i) {
        sb[4 + i] = (uint8_t)((sc[i] & 63) | ((sc[i + 4] >> 4) << 6));
        sb[8 + i] = (uint8_t)((m[i] & 63) | ((m[i + 4] >> 4) << 6));
        sb[12 + i] = (uint8_t)((sc[i + 4] & 15) | ((m[i + 4] & 15) << 4));
    }
    const float d = orc_f16_to_f32(d16), dmin = orc_f16_to_f32(dmin16);
    for (int j = 0; j < 8; ++j) {
        const float D = d * (float)sc[j], M = dmin * (float)m[j];   /* exact products */
        const float id = D != 0.0f ? 1.0f / D : 0.0f;
        for (int i = 0; i < 32; ++i) {
            float v = (x[32 * j + i] + M) * id + 0.5f;
            int c;
            if (!(v >= 0.0f)) c = 0;
            else if (v >= 15.0f) c = 15;
            else c = (int)v;
            sb[16 + 32 * (j / 2) + i] |= (uint8_t)(c << (4 * (j & 1)));
        }
    }
}

/* Quantize N rows of K floats (row n at w + n*K) into flat GGML blocks, row after row. */
void orc_quantize_rows(int type, const float *w, int64_t N, int64_t K, const int8_t *lut, uint8_t *flat)
{
    int64_t nb = K / 32, bb = orc_block_bytes(type);
    if (type == ORC_Q4_K) {
        for (int64_t n = 0; n < N; ++n)
            for (int64_t b = 0; b < K / 256; ++b)
                quantize_superblock_q4_k(w + n * K + b * 256, flat + n * orc_row_bytes(type, K) + b * 144);
        return;
    }
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t b = 0; b < nb; ++b) {
            const float *x = w + n * K + b * 32;
            uint8_t *blk = flat + (n * nb + b) * bb;
            memset(blk, 0, (size_t)bb);
            uint16_t d16 = 0;
            if (type == ORC_Q8_0) {
                int8_t q[32];
                orc_quantize_block_q8_0(x, q, &d16);
                for (int j = 0; j < 32; ++j) flat_set_code(type, blk, j, q[j]);
            } else if (type == ORC_Q4_1) {
                uint8_t codes[32];
                uint16_t m16;
                quantize_block_q4_1(x, codes, &d16, &m16);
                for (int j = 0; j < 32; ++j) flat_set_code(type, blk, j, codes[j]);
                store_u16(blk + 2, m16);
            } else if (type == ORC_MXFP4) {
                uint8_t codes[32], e;
                quantize_block_mxfp4(x, codes, &e);
                for (int j = 0; j < 32; ++j) flat_set_code(type, blk, j, codes[j]);
                blk[0] = e;
                continue;
            } else {
                uint8_t codes[32];
                if (type == ORC_Q4_0) quantize_block_q4_0(x, codes, &d16);
                else quantize_block_iq4_nl(x, lut, codes, &d16);
                for (int j = 0; j < 32; ++j) flat_set_code(type, blk, j, codes[j]);
            }
            store_u16(blk, d16);
        }
    }
}

/* Dequantize flat rows to fp64 (used by the pins: a path that never touches the tile layout). */
void orc_dequantize_flat(int type, const uint8_t *flat, int64_t N, int64_t K, const int8_t *lut, double *out)
{
    int64_t nb = K / 32, bb = orc_block_bytes(type);
    if (type == ORC_Q4_K) {   /* d*sc_j*q - dmin*m_j in fp64 */
        for (int64_t n = 0; n < N; ++n)
            for (int64_t b = 0; b < K / 256; ++b) {
                const uint8_t *sb = flat + n * orc_row_bytes(type, K) + b * 144;
                double d = orc_f16_to_f32(load_u16(sb)), dmin = orc_f16_to_f32(load_u16(sb + 2));
                for (int j = 0; j < 8; ++j) {
                    int sc, m;
                    q4k_scale_min(sb + 4, j, &sc, &m);
                    for (int i = 0; i < 32; ++i)
                        out[n * K + b * 256 + 32 * j + i] = d * sc * q4k_code(sb, j, i) - dmin * m;
                }
            }
        return;
    }
    for (int64_t n = 0; n < N; ++n)
        for (int64_t b = 0; b < nb; ++b) {
            const uint8_t *blk = flat + (n * nb + b) * bb;
            double d = block_scale(type, blk), mn = block_min(type, blk);
            for (int j = 0; j < 32; ++j)
                out[n * K + b * 32 + j] = d * (double)weight_int(type, flat_code(type, blk, j), lut) + mn;
        }
}

/* ------------------------------------------------------------------------------------------------
 * Repack / unpack ("Tile Dimensions and Grid Layout" + "Block-32 Quantized Formats").
 * Row n of the weight lives in column tile ct = n/32 at tile row r = n%32; K-block kt is tile kt.
 * ---------------------------------------------------------------------------------------------- */
void orc_repack(int type, const uint8_t *flat, int64_t K, int64_t N, uint8_t *tiled)
{
    int64_t n_k_tiles = K / 32, n_col_tiles = (N + 31) / 32;
    int64_t ts = orc_tile_bytes(type), bb = orc_block_bytes(type);
    int64_t scale_off = (type == ORC_Q8_0) ? 1024 : 512;
    memset(tiled, 0, (size_t)(n_col_tiles * n_k_tiles * ts));   /* padding rows stay zero */
    for (int64_t ct = 0; ct < n_col_tiles; ++ct)
        for (int64_t kt = 0; kt < n_k_tiles; ++kt) {
            uint8_t *tile = tiled + orc_tile_index(ct, kt, n_k_tiles) * ts;
            for (int r = 0; r < 32; ++r) {
                int64_t n = ct * 32 + r;
                if (n >= N) continue;
                if (type == ORC_Q4_K) {   /* tile kt = sub-block kt % 8 of super-block kt / 8 */
                    const uint8_t *sb = flat + n * orc_row_bytes(type, K) + (kt / 8) * 144;
                    int j = (int)(kt % 8), sc, m;
                    q4k_scale_min(sb + 4, j, &sc, &m);
                    for (int cp = 0; cp < 16; ++cp)
                        tile[cp * 32 + r] = (uint8_t)(q4k_code(sb, j, 2 * cp) | (q4k_code(sb, j, 2 * cp + 1) << 4));
                    float d = orc_f16_to_f32(load_u16(sb)), dmin = orc_f16_to_f32(load_u16(sb + 2));
                    store_u16(tile + scale_off + 4 * r, orc_f32_to_f16(d * (float)sc));
                    store_u16(tile + scale_off + 4 * r + 2, orc_f32_to_f16(-(dmin * (float)m)));
                    continue;
                }
                const uint8_t *blk = flat + (n * n_k_tiles + kt) * bb;
                for (int cp = 0; cp < 16; ++cp) {
                    int c0 = flat_code(type, blk, 2 * cp);
                    int c1 = flat_code(type, blk, 2 * cp + 1);
                    if (type == ORC_Q8_0) {
                        tile[cp * 64 + 2 * r + 0] = (uint8_t)(int8_t)c0;
                        tile[cp * 64 + 2 * r + 1] = (uint8_t)(int8_t)c1;
                    } else {
                        tile[cp * 32 + r] = (uint8_t)(((c1 & 0x0F) << 4) | (c0 & 0x0F));
                    }
                }
                if (type == ORC_MXFP4) {
                    tile[scale_off + r] = blk[0];            /* one exponent byte per row */
                } else if (type == ORC_Q4_1) {
                    for (int i = 0; i < 4; ++i) tile[scale_off + 4 * r + i] = blk[i];   /* d, m */
                } else {
                    tile[scale_off + 2 * r + 0] = blk[0];
                    tile[scale_off + 2 * r + 1] = blk[1];
                }
            }
        }
}

/* Inverse of orc_repack for the block-32 types (Q4_K's tile products cannot be split back). */
void orc_unpack(int type, const uint8_t *tiled, int64_t K, int64_t N, uint8_t *flat)
{
    if (type == ORC_Q4_K) return;
    int64_t n_k_tiles = K / 32;
    int64_t ts = orc_tile_bytes(type), bb = orc_block_bytes(type);
    int64_t scale_off = (type == ORC_Q8_0) ? 1024 : 512;
    for (int64_t n = 0; n < N; ++n) {
        int64_t ct = n / 32;
        int r = (int)(n % 32);
        for (int64_t kt = 0; kt < n_k_tiles; ++kt) {
            const uint8_t *tile = tiled + orc_tile_index(ct, kt, n_k_tiles) * ts;
            uint8_t *blk = flat + (n * n_k_tiles + kt) * bb;
            memset(blk, 0, (size_t)bb);
            if (type == ORC_MXFP4) {
                blk[0] = tile[scale_off + r];
            } else if (type == ORC_Q4_1) {
                for (int i = 0; i < 4; ++i) blk[i] = tile[scale_off + 4 * r + i];
            } else {
                blk[0] = tile[scale_off + 2 * r + 0];
                blk[1] = tile[scale_off + 2 * r + 1];
            }
            for (int cp = 0; cp < 16; ++cp) {
                int c0, c1;
                if (type == ORC_Q8_0) {
                    c0 = (int)(int8_t)tile[cp * 64 + 2 * r + 0];
                    c1 = (int)(int8_t)tile[cp * 64 + 2 * r + 1];
                } else {
                    c0 = tile[cp * 32 + r] & 0x0F;
                    c1 = tile[cp * 32 + r] >> 4;
                }
                flat_set_code(type, blk, 2 * cp, c0);
                flat_set_code(type, blk, 2 * cp + 1, c1);
            }
        }
    }
}

/* Integer weight and fp16 row scale of element (n, k), read from the tiled buffer. */
static int tiled_weight(int type, const uint8_t *tiled, int64_t n_k_tiles, int64_t n, int64_t k,
                        const int8_t *lut)
{
    int64_t ct = n / 32, kt = k / 32;
    int r = (int)(n % 32), c = (int)(k % 32), cp = c / 2;
    const uint8_t *tile = tiled + orc_tile_index(ct, kt, n_k_tiles) * orc_tile_bytes(type);
    int code;
    if (type == ORC_Q8_0) code = (int)(int8_t)tile[cp * 64 + 2 * r + (c & 1)];
    else code = (c & 1) ? (tile[cp * 32 + r] >> 4) : (tile[cp * 32 + r] & 0x0F);
    return weight_int(type, code, lut);
}

static double tiled_scale(int type, const uint8_t *tiled, int64_t n_k_tiles, int64_t n, int64_t kt)
{
    int64_t ct = n / 32;
    int r = (int)(n % 32);
    const uint8_t *tile = tiled + orc_tile_index(ct, kt, n_k_tiles) * orc_tile_bytes(type);
    int64_t scale_off = (type == ORC_Q8_0) ? 1024 : 512;
    return block_scale(type, tile + scale_off + (type == ORC_MXFP4 ? r : (affine_tile(type) ? 4 * r : 2 * r)));
}

static double tiled_min(int type, const uint8_t *tiled, int64_t n_k_tiles, int64_t n, int64_t kt)
{
    if (!affine_tile(type)) return 0.0;
    const uint8_t *tile = tiled + orc_tile_index(n / 32, kt, n_k_tiles) * orc_tile_bytes(type);
    return block_min(type, tile + 512 + 4 * (n % 32));
}

/* ------------------------------------------------------------------------------------------------
 * Activation quantization: x is M rows of K floats with row stride ldx; a_q is [M][K] int8 and
 * a_d is [M][K/32] fp16 bits (the per-32 Q8_0 blocks stored as two arrays).
 * ---------------------------------------------------------------------------------------------- */
void orc_quantize_act(const float *x, int64_t M, int64_t K, int64_t ldx, int8_t *a_q, uint16_t *a_d)
{
    int64_t nb = K / 32;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t b = 0; b < nb; ++b)
            orc_quantize_block_q8_0(x + m * ldx + b * 32, a_q + m * K + b * 32, a_d + m * nb + b);
}

/* ------------------------------------------------------------------------------------------------
 * Matmul over the tiled weight.  One output element:
 *   S_b   = sum_{j<32} w_int[n, 32b+j] * a_q[m, 32b+j]          (exact, int64)
 *   Y     = sum_b f64(d_w[n,b]) * f64(d_a[m,b]) * S_b            (fp64)
 *   Bound = sum_b sum_j |f64(d_w) * w_int * f64(d_a) * a_q|      (fp64)
 * ---------------------------------------------------------------------------------------------- */
static void one_output(int type, const uint8_t *tiled, int64_t K, const int8_t *a_q, const uint16_t *a_d,
                       int64_t m, int64_t n, const int8_t *lut, double *y, double *bound)
{
    int64_t n_k_tiles = K / 32;
    double acc = 0.0, bacc = 0.0;
    for (int64_t b = 0; b < n_k_tiles; ++b) {
        int64_t s = 0, sabs = 0, asum = 0;
        double dw = tiled_scale(type, tiled, n_k_tiles, n, b);
        double mw = tiled_min(type, tiled, n_k_tiles, n, b);
        double da = (double)orc_f16_to_f32(a_d[m * n_k_tiles + b]);
        double babs = 0.0;
        for (int j = 0; j < 32; ++j) {
            int64_t k = b * 32 + j;
            int64_t w = tiled_weight(type, tiled, n_k_tiles, n, k, lut);
            int64_t a = a_q[m * K + k];
            s += w * a;
            asum += a;
            sabs += (w * a < 0) ? -(w * a) : (w * a);
            babs += fabs(dw * (double)w + mw) * fabs((double)a);   /* |dequantized weight| * |a_q| */
        }
        /* sum_j (dw*w_j + mw) * da * a_j = da * (dw * S_b + mw * sum_j a_j) */
        acc += dw * da * (double)s + mw * da * (double)asum;
        bacc += affine_tile(type) ? fabs(da) * babs : fabs(dw * da) * (double)sabs;
    }
    *y = acc;
    *bound = bacc;
}

void orc_matmul(int type, const uint8_t *tiled, int64_t K, int64_t N, const int8_t *a_q,
                const uint16_t *a_d, int64_t M, const int8_t *lut, double *y, double *bound)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            one_output(type, tiled, K, a_q, a_d, m, n, lut, y + m * N + n, bound + m * N + n);
}

/* The same, for a list of (m, n) output positions only. */
void orc_matmul_at(int type, const uint8_t *tiled, int64_t K, const int8_t *a_q, const uint16_t *a_d,
                   int64_t count, const int64_t *ms, const int64_t *ns, const int8_t *lut,
                   double *y, double *bound)
{
    for (int64_t i = 0; i < count; ++i)
        one_output(type, tiled, K, a_q, a_d, ms[i], ns[i], lut, y + i, bound + i);
}
