/*
 * CPU oracle for the CSA2 cache write — TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the package's smoke check and the benchmark's CPU-baseline
 * leg may load this code.  The CUDA library never links, includes or calls it,
 * and it shares no code with the CUDA sources.
 *
 * It restates, one plain step at a time, how one cache entry is produced:
 *   compress -> RMSNorm -> RoPE on the 64-d tail -> main-KV FP4 (E2M1 + E4M3/16)
 *   -> index-K projection 512->128 -> index-K MXFP4 (E2M1 + E8M0/32).
 *
 * Sources (web pages about DeepSeek-V4.1-Flash):
 *   [dilfish]  "4. 层维度(下):CSA2 与每 token 890 字节", §4.2 compressor formula,
 *              §4.4 entry formats b(D,G), §4.5 FP4 range.
 *   [zartbot]  "DeepSeek-V4.1 Flash: 把 KV Cache 压缩推到极致", §2.3.1 (index K is
 *              projected from main KV), §2.4.4 (E2M1 + one E4M3 scale per 16
 *              channels, no global scale; quantise after RoPE; RMSNorm before).
 *
 * The pages fix the formats but not every floating-point order.  Because the
 * quantised bytes must be reproduced bit for bit, every binary32 operation
 * here is written out in a fixed order (the readings are listed below); all
 * other arithmetic is binary64.  Compile with -ffp-contract=off and without
 * -ffast-math so that each C operator is one IEEE operation.
 *
 * Readings where the pages are silent:
 *   R1 compressor: c = fmaf(w0, x0, w1*x1) / (w0 + w1), binary32, positions
 *      (2j, 2j+1) in 0-based numbering ((2j-1, 2j) in the page's 1-based one).
 *   R2 RMSNorm (weight 1, eps 1e-6): 32 partial sums, partial i accumulates
 *      channels 16i..16i+15 in order with fmaf; partials combined pairwise
 *      p[i] += p[i+off] for off = 16,8,4,2,1; r = 1/sqrtf(ss/512 + 1e-6f);
 *      y = c*r.
 *   R3 RoPE: interleaved pairs (448+2i, 449+2i), i = 0..31, at the entry's
 *      absolute index; y0' = fmaf(y0,cos,-(y1*sin)), y1' = fmaf(y0,sin,y1*cos);
 *      cos/sin = binary64 cos/sin of p * pow(theta, -(2i)/64.0), rounded to
 *      binary32.
 *   R4 main FP4: per 16 channels s = E4M3_RNE(amax/6) (saturating at 448);
 *      code = E2M1_RNE_sat(y/s) (binary32 division); s == 0 -> all codes +0.
 *      Code of channel 2k in the low nibble of byte k; 256 code bytes then 32
 *      scale bytes.
 *   R5 index K: k[o] = sequential fmaf over channels 0..511 starting at 0, of
 *      the post-RoPE, pre-quantisation binary32 latent times W[o][ch].
 *   R6 MXFP4 (OCP MX rule): X = floor(log2(amax)) - 2 clamped to [-127,127],
 *      scale byte X+127, code = E2M1_RNE_sat(v / 2^X); amax == 0 -> byte 0 and
 *      codes +0.
 *   E2M1/E4M3 rounding is to nearest with ties to the even code; the sign bit
 *   is the sign bit of the binary32 input (so a small negative value gives -0).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define D_LATENT 512
#define D_ROPE 64
#define ROPE_FIRST (D_LATENT - D_ROPE)
#define D_INDEX 128
#define MAIN_GROUP 16
#define MX_GROUP 32
#define MAIN_ENTRY_BYTES (D_LATENT / 2 + D_LATENT / MAIN_GROUP) /* 288 */
#define INDEX_CODE_BYTES (D_INDEX / 2)                          /* 64 */
#define INDEX_SCALE_BYTES (D_INDEX / MX_GROUP)                  /* 4 */

/* ------------------------------------------------------------ small formats */

static float bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* E2M1 magnitudes by code 0..7: exponent 2 bits (bias 1), mantissa 1 bit. */
static const double E2M1_GRID[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double oracle_e2m1_decode(uint8_t code) {
    double v = E2M1_GRID[code & 7];
    return (code & 8) ? -v : v;
}

/* Nearest grid point, ties to the even code, magnitudes >= 6 saturate to 6. */
uint8_t oracle_e2m1_encode(float v) {
    uint8_t sign = signbit(v) ? 8 : 0;
    double a = fabs((double)v);
    if (isnan(v)) return 0;
    if (a >= 6.0) return sign | 7;
    int best = 0;
    for (int c = 1; c < 8; c++) {
        double dc = fabs(a - E2M1_GRID[c]), db = fabs(a - E2M1_GRID[best]);
        if (dc < db || (dc == db && (c % 2) == 0)) best = c;
    }
    return (uint8_t)(sign | best);
}

/* E4M3 (bias 7, no infinities, 0x7F/0xFF = NaN, max 448). */
double oracle_e4m3_decode(uint8_t code) {
    int e = (code >> 3) & 15, m = code & 7;
    double v = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return (code & 0x80) ? -v : v;
}

/* Nearest of the 127 non-negative finite codes, ties to the even code,
 * saturating at 448 (the largest finite value). */
uint8_t oracle_e4m3_encode(float v) {
    uint8_t sign = signbit(v) ? 0x80 : 0;
    double a = fabs((double)v);
    if (isnan(v)) return 0x7F;
    if (a >= 448.0) return sign | 0x7E;
    int best = 0;
    for (int c = 1; c <= 0x7E; c++) {
        double dc = fabs(a - oracle_e4m3_decode((uint8_t)c));
        double db = fabs(a - oracle_e4m3_decode((uint8_t)best));
        if (dc < db || (dc == db && (c % 2) == 0)) best = c;
    }
    return (uint8_t)(sign | best);
}

/* FP8 SWA rows: n binary32 values -> n E4M3 bytes, each on its own (no scale). */
void oracle_e4m3_encode_rows(const float *v, int64_t n, uint8_t *out) {
    for (int64_t i = 0; i < n; i++) out[i] = oracle_e4m3_encode(v[i]);
}

/* ------------------------------------------------------- group quantisers */

/* Main KV group (R4): 16 binary32 values -> 8 code bytes + 1 E4M3 scale. */
void oracle_fp4_group_quantize(const float *y, uint8_t *codes8, uint8_t *scale) {
    float amax = 0.0f;
    for (int i = 0; i < MAIN_GROUP; i++) {
        float a = fabsf(y[i]);
        if (a > amax) amax = a;
    }
    float s_f = amax / 6.0f;
    uint8_t s_code = oracle_e4m3_encode(s_f);
    float s = (float)oracle_e4m3_decode(s_code);
    *scale = s_code;
    for (int k = 0; k < MAIN_GROUP / 2; k++) {
        uint8_t lo = 0, hi = 0;
        if (s != 0.0f) {
            float q0 = y[2 * k] / s;
            float q1 = y[2 * k + 1] / s;
            lo = oracle_e2m1_encode(q0);
            hi = oracle_e2m1_encode(q1);
        }
        codes8[k] = (uint8_t)(lo | (hi << 4));
    }
}

/* MXFP4 block (R6): 32 binary32 values -> 16 code bytes + 1 E8M0 scale. */
void oracle_mxfp4_block_quantize(const float *v, uint8_t *codes16, uint8_t *scale) {
    double amax = 0.0;
    for (int i = 0; i < MX_GROUP; i++) {
        double a = fabs((double)v[i]);
        if (a > amax) amax = a;
    }
    if (amax == 0.0) {
        *scale = 0;
        memset(codes16, 0, MX_GROUP / 2);
        return;
    }
    int e;
    frexp(amax, &e);            /* amax = f * 2^e, f in [0.5,1): floor(log2) = e-1 */
    int X = (e - 1) - 2;        /* 2 = exponent of the largest E2M1 value (6 = 1.5*2^2) */
    if (X < -127) X = -127;
    if (X > 127) X = 127;
    *scale = (uint8_t)(X + 127);
    for (int k = 0; k < MX_GROUP / 2; k++) {
        float q0 = (float)ldexp((double)v[2 * k], -X);     /* exact: power-of-two scaling */
        float q1 = (float)ldexp((double)v[2 * k + 1], -X);
        codes16[k] = (uint8_t)(oracle_e2m1_encode(q0) | (oracle_e2m1_encode(q1) << 4));
    }
}

/* Quantise n rows of 128 binary32 values to MXFP4 (used for index K and for the
 * indexer queries). codes: [n][64], scales: [n][4]. */
void oracle_mxfp4_rows(const float *v, int64_t n, uint8_t *codes, uint8_t *scales) {
    for (int64_t r = 0; r < n; r++)
        for (int b = 0; b < D_INDEX / MX_GROUP; b++)
            oracle_mxfp4_block_quantize(v + r * D_INDEX + b * MX_GROUP,
                                        codes + r * INDEX_CODE_BYTES + b * (MX_GROUP / 2),
                                        scales + r * INDEX_SCALE_BYTES + b);
}

/* ---------------------------------------------------------- entry stages */

/* R1: compress one entry (m = 2) or pass one token through (m = 1). */
void oracle_compress(const uint16_t *x0, const uint16_t *x1, const float *w0,
                     const float *w1, int m, float *c) {
    for (int ch = 0; ch < D_LATENT; ch++) {
        float a = bf16_to_f32(x0[ch]);
        if (m == 1) {
            c[ch] = a;
        } else {
            float b = bf16_to_f32(x1[ch]);
            float num = fmaf(w0[ch], a, w1[ch] * b);
            float den = w0[ch] + w1[ch];
            c[ch] = num / den;
        }
    }
}

/* R2: RMSNorm with weight 1. */
void oracle_rmsnorm(const float *c, float *y) {
    float p[32];
    for (int i = 0; i < 32; i++) {
        p[i] = 0.0f;
        for (int k = 0; k < 16; k++) p[i] = fmaf(c[16 * i + k], c[16 * i + k], p[i]);
    }
    for (int off = 16; off >= 1; off /= 2)
        for (int i = 0; i < off; i++) p[i] = p[i] + p[i + off];
    float ss = p[0];
    float r = 1.0f / sqrtf(ss / 512.0f + 1e-6f);
    for (int ch = 0; ch < D_LATENT; ch++) y[ch] = c[ch] * r;
}

/* R3: cos/sin table for positions [0, P): cs[(p*32 + i)*2 + {0,1}]. */
void oracle_rope_table(int64_t P, double theta, float *cs) {
    for (int i = 0; i < D_ROPE / 2; i++) {
        double inv_freq = pow(theta, -(double)(2 * i) / 64.0);
        for (int64_t p = 0; p < P; p++) {
            double ang = (double)p * inv_freq;
            cs[(p * 32 + i) * 2 + 0] = (float)cos(ang);
            cs[(p * 32 + i) * 2 + 1] = (float)sin(ang);
        }
    }
}

/* R3: rotate the 64-d tail in place with the table row of one position. */
void oracle_rope_apply(float *y, const float *cs_row /* [32][2] */) {
    for (int i = 0; i < D_ROPE / 2; i++) {
        float co = cs_row[2 * i], si = cs_row[2 * i + 1];
        float y0 = y[ROPE_FIRST + 2 * i], y1 = y[ROPE_FIRST + 2 * i + 1];
        y[ROPE_FIRST + 2 * i] = fmaf(y0, co, -(y1 * si));
        y[ROPE_FIRST + 2 * i + 1] = fmaf(y0, si, y1 * co);
    }
}

/* R5: index-K projection k = W y, W bf16 [128][512]. */
void oracle_project(const float *y, const uint16_t *W, float *k) {
    for (int o = 0; o < D_INDEX; o++) {
        float acc = 0.0f;
        for (int ch = 0; ch < D_LATENT; ch++)
            acc = fmaf(y[ch], bf16_to_f32(W[o * D_LATENT + ch]), acc);
        k[o] = acc;
    }
}

/* R4 over a full latent: 288-byte main-KV entry. */
void oracle_main_entry(const float *y, uint8_t *entry) {
    for (int g = 0; g < D_LATENT / MAIN_GROUP; g++)
        oracle_fp4_group_quantize(y + g * MAIN_GROUP, entry + g * (MAIN_GROUP / 2),
                                  entry + D_LATENT / 2 + g);
}

/*
 * Whole cache write for one sequence chunk.
 *   x        bf16 [T][512]; m = 2 needs even T
 *   entry0   absolute index of the first entry written (RoPE position)
 *   cs       table from oracle_rope_table covering entry0 + T/m positions
 *   main_kv  [T/m][288], idx_codes [T/m][64], idx_scales [T/m][4]
 * Entries are independent; the loop is parallel over them when OpenMP is on.
 */
void oracle_compress_quantize(const uint16_t *x, int64_t T, int m, const float *w0,
                              const float *w1, const uint16_t *W, int64_t entry0,
                              const float *cs, uint8_t *main_kv, uint8_t *idx_codes,
                              uint8_t *idx_scales) {
    int64_t n = T / m;
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; j++) {
        float c[D_LATENT], y[D_LATENT], k[D_INDEX];
        const uint16_t *x0 = x + (j * m) * D_LATENT;
        const uint16_t *x1 = (m == 2) ? x + (j * m + 1) * D_LATENT : x0;
        oracle_compress(x0, x1, w0, w1, m, c);
        oracle_rmsnorm(c, y);
        oracle_rope_apply(y, cs + (entry0 + j) * 64);
        oracle_main_entry(y, main_kv + j * MAIN_ENTRY_BYTES);
        oracle_project(y, W, k);
        oracle_mxfp4_rows(k, 1, idx_codes + j * INDEX_CODE_BYTES,
                          idx_scales + j * INDEX_SCALE_BYTES);
    }
}

/* Intermediate binary32 vectors of one entry, for the stage pins. */
void oracle_entry_stages(const uint16_t *x0, const uint16_t *x1, int m, const float *w0,
                         const float *w1, const float *cs_row, const uint16_t *W,
                         float *c, float *y_norm, float *y_rope, float *k) {
    oracle_compress(x0, x1, w0, w1, m, c);
    oracle_rmsnorm(c, y_norm);
    memcpy(y_rope, y_norm, sizeof(float) * D_LATENT);
    oracle_rope_apply(y_rope, cs_row);
    oracle_project(y_rope, W, k);
}
