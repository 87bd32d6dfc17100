/*
 * CPU fp64 oracle for the two-stage quantized MoE expert computation.
 * TEST INFRASTRUCTURE ONLY: see oracle.h for who may use it, the pages it
 * follows and the readings it takes. Plain loops, no blocking or fusion.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------------------
 * Element and scale formats (OCP MX; "fp4x2" and "1x32" e8m0 on the aiter pages,
 * PR 4463 "Three tuner defects" item 2, PR 6259 "Test Result").
 * ------------------------------------------------------------------------- */

/* e2m1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0. */
double orc_e2m1_value(int code) {
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -mag : mag;
}

/* e4m3fn: sign bit 7, exponent bits 6..3 (bias 7), mantissa bits 2..0,
 * S.1111.111 is NaN, no infinities. */
double orc_e4m3_value(int byte) {
    int s = (byte >> 7) & 1, e = (byte >> 3) & 15, m = byte & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) mag = ldexp(m / 8.0, -6);
    else mag = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* e8m0: unsigned exponent with bias 127; 0xFF is NaN. */
double orc_e8m0_value(int byte) {
    if ((byte & 0xFF) == 0xFF) return NAN;
    return ldexp(1.0, (byte & 0xFF) - 127);
}

double orc_bf16_value(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

float orc_f32_from_f64(double v) { return (float)v; }

/* bf16 has 8 significant bits, exponent range of fp32. Round v to that grid
 * (nearest, ties to even) in one step, then read the bits off the exact fp32. */
uint16_t orc_bf16_from_f64(double v) {
    if (isnan(v)) return 0x7FC0;
    if (v == 0.0) return signbit(v) ? 0x8000 : 0x0000;
    double a = fabs(v);
    int e;
    frexp(a, &e);              /* a = f * 2^e, f in [0.5, 1): leading bit 2^(e-1) */
    int lead = e - 1;
    if (lead < -126) lead = -126; /* subnormal quantum 2^-133 */
    double q = ldexp(1.0, lead - 7);
    double r = rint(a / q) * q;
    const double bf16_max = ldexp(255.0 / 128.0, 127);
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    if (r > bf16_max) return sign | 0x7F80;
    float f = (float)r; /* exact: r is on the bf16 grid */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(sign | ((u >> 16) & 0x7FFF));
}

typedef struct {
    int mbits;       /* stored mantissa bits */
    int emin;        /* exponent of the smallest normal (subnormal quantum shares it) */
    int emax_elem;   /* exponent of the largest normal */
    double maxv;     /* largest finite magnitude */
    int ncodes;      /* codes per sign */
} fmt_t;

static fmt_t fmt_of(int fmt) {
    fmt_t f;
    if (fmt == ORC_FMT_E2M1) { f.mbits = 1; f.emin = 0; f.emax_elem = 2; f.maxv = 6.0; f.ncodes = 8; }
    else { f.mbits = 3; f.emin = -6; f.emax_elem = 8; f.maxv = 448.0; f.ncodes = 128; }
    return f;
}

static double code_value(int code, int fmt) {
    return fmt == ORC_FMT_E2M1 ? orc_e2m1_value(code) : orc_e4m3_value(code);
}

double orc_round_to_format(double x, int fmt) {
    fmt_t f = fmt_of(fmt);
    double a = fabs(x);
    if (a == 0.0) return x;
    int e;
    frexp(a, &e);
    int lead = e - 1;
    if (lead < f.emin) lead = f.emin;
    double q = ldexp(1.0, lead - f.mbits);
    double r = rint(a / q) * q; /* a/q is exact: q is a power of two */
    if (r > f.maxv) r = f.maxv;
    return copysign(r, x);
}

int orc_encode(double r, int fmt) {
    fmt_t f = fmt_of(fmt);
    int sign_bit = fmt == ORC_FMT_E2M1 ? 8 : 128;
    double a = fabs(r);
    for (int c = 0; c < f.ncodes; ++c) {
        double v = code_value(c, fmt);
        if (v == a) return signbit(r) ? (c | sign_bit) : c;
    }
    return -1;
}

/* One 1x32 block: scale byte and 32 codes. */
static void quantize_block(const double* v, int fmt, uint8_t* code32, uint8_t* scale) {
    fmt_t f = fmt_of(fmt);
    double amax = 0.0;
    for (int i = 0; i < 32; ++i) amax = fmax(amax, fabs(v[i]));
    if (amax == 0.0) {
        *scale = 127;
        for (int i = 0; i < 32; ++i) code32[i] = 0;
        return;
    }
    int e;
    frexp(amax, &e);
    int E = (e - 1) - f.emax_elem; /* floor(log2 amax) - emax_elem */
    if (E < -127) E = -127;
    if (E > 127) E = 127;
    *scale = (uint8_t)(E + 127);
    for (int i = 0; i < 32; ++i) {
        double r = orc_round_to_format(ldexp(v[i], -E), fmt);
        code32[i] = (uint8_t)orc_encode(r, fmt);
    }
}

static void store_codes(const uint8_t* code32, int fmt, uint8_t* dst) {
    if (fmt == ORC_FMT_E2M1) {
        for (int j = 0; j < 16; ++j) dst[j] = (uint8_t)(code32[2 * j] | (code32[2 * j + 1] << 4));
    } else {
        memcpy(dst, code32, 32);
    }
}

void orc_mx_quantize_f64(const double* v, int64_t nblocks, int fmt, uint8_t* codes, uint8_t* scales) {
    int bytes_per_block = fmt == ORC_FMT_E2M1 ? 16 : 32;
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < nblocks; ++b) {
        uint8_t c32[32];
        quantize_block(v + b * 32, fmt, c32, scales + b);
        store_codes(c32, fmt, codes + b * bytes_per_block);
    }
}

void orc_mx_quantize_f32(const float* v, int64_t nblocks, int fmt, uint8_t* codes, uint8_t* scales) {
    int bytes_per_block = fmt == ORC_FMT_E2M1 ? 16 : 32;
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < nblocks; ++b) {
        double d[32];
        uint8_t c32[32];
        for (int i = 0; i < 32; ++i) d[i] = (double)v[b * 32 + i];
        quantize_block(d, fmt, c32, scales + b);
        store_codes(c32, fmt, codes + b * bytes_per_block);
    }
}

void orc_mx_quantize_bf16(const uint16_t* v, int64_t nblocks, int fmt, uint8_t* codes, uint8_t* scales) {
    int bytes_per_block = fmt == ORC_FMT_E2M1 ? 16 : 32;
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < nblocks; ++b) {
        double d[32];
        uint8_t c32[32];
        for (int i = 0; i < 32; ++i) d[i] = orc_bf16_value(v[b * 32 + i]);
        quantize_block(d, fmt, c32, scales + b);
        store_codes(c32, fmt, codes + b * bytes_per_block);
    }
}

static double element_of(const uint8_t* codes, int64_t i, int fmt) {
    if (fmt == ORC_FMT_E2M1) {
        uint8_t byte = codes[i >> 1];
        return orc_e2m1_value((i & 1) ? (byte >> 4) : (byte & 15));
    }
    return orc_e4m3_value(codes[i]);
}

void orc_mx_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t nblocks, int fmt, double* out) {
    for (int64_t i = 0; i < nblocks * 32; ++i)
        out[i] = element_of(codes, i, fmt) * orc_e8m0_value(scales[i / 32]);
}

/* ---------------------------------------------------------------------------
 * Expert sort with per-expert padding to tile_m (aiter PR 5118, Summary:
 * "moe_sorting pads every expert up to a full block_m").
 * ------------------------------------------------------------------------- */
int64_t orc_sort(const int32_t* ids, int T, int K, int E, int tile_m,
                 int32_t* sorted_ids, int32_t* block_expert, int32_t* num_blocks,
                 int32_t* expert_count, int32_t* expert_offset) {
    int64_t n = (int64_t)T * K, dropped = 0;
    for (int e = 0; e < E; ++e) expert_count[e] = 0;
    for (int64_t p = 0; p < n; ++p) {
        int e = ids[p];
        if (e < 0 || e >= E) ++dropped;
        else ++expert_count[e];
    }
    int64_t off = 0;
    for (int e = 0; e < E; ++e) {
        expert_offset[e] = (int32_t)off;
        int64_t padded = (expert_count[e] + tile_m - 1) / tile_m * tile_m;
        off += padded;
    }
    expert_offset[E] = (int32_t)off;
    *num_blocks = (int32_t)(off / tile_m);
    for (int64_t r = 0; r < off; ++r) sorted_ids[r] = (int32_t)n; /* padding sentinel */
    int32_t* cursor = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
    for (int e = 0; e < E; ++e) cursor[e] = expert_offset[e];
    for (int64_t p = 0; p < n; ++p) { /* ascending p keeps pairs of one expert in order */
        int e = ids[p];
        if (e < 0 || e >= E) continue;
        sorted_ids[cursor[e]++] = (int32_t)p;
    }
    free(cursor);
    for (int e = 0; e < E; ++e)
        for (int32_t b = expert_offset[e] / tile_m; b < expert_offset[e + 1] / tile_m; ++b)
            block_expert[b] = e;
    return dropped;
}

/* ---------------------------------------------------------------------------
 * Activations (aiter PR 6259 Motivation; PR 4471 Motivation).
 * ------------------------------------------------------------------------- */
static double sigmoid(double g) { return 1.0 / (1.0 + exp(-g)); }

double orc_act(int act, double g, double u, double beta, double lbeta) {
    if (act == ORC_ACT_SILU) return g * sigmoid(g) * u;
    double situ = beta * tanh(g / beta) * sigmoid(g);
    double up = lbeta * tanh(u / lbeta);
    return situ * up;
}

/* ---------------------------------------------------------------------------
 * Forward pass pieces.
 * ------------------------------------------------------------------------- */

/* The activation row the stage-1 GEMM sees: bf16 x as is (a16), or x
 * quantised to fp8 / fp4 with 1x32 e8m0 scales along H and dequantised
 * (a8 / a4; aiter PR 4463 "What"). */
void orc_activation_row(const uint16_t* xrow, int H, int a_dtype, double* a) {
    if (a_dtype == ORC_A_BF16) {
        for (int h = 0; h < H; ++h) a[h] = orc_bf16_value(xrow[h]);
        return;
    }
    int fmt = a_dtype == ORC_A_FP8 ? ORC_FMT_E4M3 : ORC_FMT_E2M1;
    int nb = H / 32;
    uint8_t* codes = (uint8_t*)malloc((size_t)H);
    uint8_t* scales = (uint8_t*)malloc((size_t)nb);
    orc_mx_quantize_bf16(xrow, nb, fmt, codes, scales);
    orc_mx_dequantize(codes, scales, nb, fmt, a);
    free(codes);
    free(scales);
}

/* Stage-1 output held in fp32, then requantised: bf16 (a16) or fp8/fp4 1x32
 * along I (a8/a4; aiter PR 6259 Technical Details, PR 4463 item 2). */
void orc_requantize_intermediate(const double* y, int I, int a_dtype, double* yq) {
    if (a_dtype == ORC_A_BF16) {
        for (int i = 0; i < I; ++i) yq[i] = orc_bf16_value(orc_bf16_from_f64((double)(float)y[i]));
        return;
    }
    int fmt = a_dtype == ORC_A_FP8 ? ORC_FMT_E4M3 : ORC_FMT_E2M1;
    int nb = I / 32;
    double* y32 = (double*)malloc(sizeof(double) * (size_t)I);
    uint8_t* codes = (uint8_t*)malloc((size_t)I);
    uint8_t* scales = (uint8_t*)malloc((size_t)nb);
    for (int i = 0; i < I; ++i) y32[i] = (double)(float)y[i];
    orc_mx_quantize_f64(y32, nb, fmt, codes, scales);
    orc_mx_dequantize(codes, scales, nb, fmt, yq);
    free(y32);
    free(codes);
    free(scales);
}

/* Dequantised weight row: codes [len/2] + e8m0 scales [len/32]. */
static void weight_row(const uint8_t* codes, const uint8_t* scales, int len, double* out) {
    for (int i = 0; i < len; ++i) {
        uint8_t byte = codes[i >> 1];
        int c = (i & 1) ? (byte >> 4) : (byte & 15);
        out[i] = orc_e2m1_value(c) * orc_e8m0_value(scales[i / 32]);
    }
}

static int bad_shape(int T, int H, int I, int E, int K) {
    return T < 0 || H <= 0 || I <= 0 || E <= 0 || K <= 0 || H % 32 || I % 32;
}

int64_t orc_moe_forward(const uint16_t* x, const int32_t* ids, const float* w,
                        int T, int H, int I, int E, int K,
                        const uint8_t* w13, const uint8_t* w13s,
                        const uint8_t* w2, const uint8_t* w2s,
                        int act, double beta, double lbeta, int a_dtype, int tile_m,
                        const int32_t* subset, int nsub,
                        double* out_f64, uint16_t* out_bf16, double* inter) {
    if (bad_shape(T, H, I, E, K) || tile_m <= 0) return -1;
    if (!subset) nsub = T;
    int64_t n = (int64_t)T * K;
    /* 1. the sort drives the grouping */
    int64_t cap = n + (int64_t)(E < n ? E : n) * (tile_m - 1) + tile_m;
    int32_t* sorted_ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)(cap > 0 ? cap : 1));
    int32_t* block_expert = (int32_t*)malloc(sizeof(int32_t) * (size_t)(cap / tile_m + 1));
    int32_t* count = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
    int32_t* offset = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E + 1));
    int32_t nblocks = 0;
    int64_t dropped = orc_sort(ids, T, K, E, tile_m, sorted_ids, block_expert, &nblocks, count, offset);

    /* token -> subset slot */
    int32_t* slot = (int32_t*)malloc(sizeof(int32_t) * (size_t)(T > 0 ? T : 1));
    for (int t = 0; t < T; ++t) slot[t] = -1;
    for (int i = 0; i < nsub; ++i) {
        int t = subset ? subset[i] : i;
        if (t < 0 || t >= T) { dropped = -1; goto done_early; }
        slot[t] = i;
    }

    {
        double* a = (double*)malloc(sizeof(double) * (size_t)nsub * H + 1);
        double* yq = (double*)malloc(sizeof(double) * (size_t)nsub * K * I + 1);
        double* z = (double*)malloc(sizeof(double) * (size_t)nsub * K * H + 1);
        char* valid = (char*)calloc((size_t)nsub * K + 1, 1);

#pragma omp parallel for schedule(dynamic)
        for (int i = 0; i < nsub; ++i) {
            int t = subset ? subset[i] : i;
            orc_activation_row(x + (size_t)t * H, H, a_dtype, a + (size_t)i * H);
        }

        /* 2. stage 1 per block of sorted rows (one expert per block) */
#pragma omp parallel for schedule(dynamic)
        for (int32_t b = 0; b < nblocks; ++b) {
            int e = block_expert[b];
            double* wg = (double*)malloc(sizeof(double) * (size_t)H);
            double* wu = (double*)malloc(sizeof(double) * (size_t)H);
            double* y = (double*)malloc(sizeof(double) * (size_t)tile_m * I);
            int rows[4096];
            int nr = 0;
            for (int r = 0; r < tile_m && nr < 4096; ++r) {
                int32_t p = sorted_ids[(int64_t)b * tile_m + r];
                if (p >= n) continue; /* padding */
                int t = p / K;
                if (slot[t] < 0) continue;
                rows[nr++] = slot[t] * K + (p % K);
            }
            if (nr > 0) {
                for (int j = 0; j < I; ++j) {
                    size_t gate = ((size_t)e * 2 * I + j), up = ((size_t)e * 2 * I + I + j);
                    weight_row(w13 + gate * (H / 2), w13s + gate * (H / 32), H, wg);
                    weight_row(w13 + up * (H / 2), w13s + up * (H / 32), H, wu);
                    for (int q = 0; q < nr; ++q) {
                        const double* ar = a + (size_t)(rows[q] / K) * H;
                        double g = 0.0, u = 0.0;
                        for (int h = 0; h < H; ++h) { g += ar[h] * wg[h]; u += ar[h] * wu[h]; }
                        y[(size_t)q * I + j] = orc_act(act, g, u, beta, lbeta);
                    }
                }
                for (int q = 0; q < nr; ++q) {
                    orc_requantize_intermediate(y + (size_t)q * I, I, a_dtype, yq + (size_t)rows[q] * I);
                    valid[rows[q]] = 1;
                }
                /* 3. stage 2 for the same rows */
                double* w2r = wg; /* reuse: needs I <= H doubles */
                double* tmp = NULL;
                if (I > H) { tmp = (double*)malloc(sizeof(double) * (size_t)I); w2r = tmp; }
                for (int h = 0; h < H; ++h) {
                    size_t row = (size_t)e * H + h;
                    weight_row(w2 + row * (I / 2), w2s + row * (I / 32), I, w2r);
                    for (int q = 0; q < nr; ++q) {
                        const double* yr = yq + (size_t)rows[q] * I;
                        double s = 0.0;
                        for (int i = 0; i < I; ++i) s += yr[i] * w2r[i];
                        z[(size_t)rows[q] * H + h] = s;
                    }
                }
                free(tmp);
            }
            free(wg);
            free(wu);
            free(y);
        }

        /* 4. combine: out[t] = sum over valid k of w[t,k] * z[t,k], ascending k */
#pragma omp parallel for schedule(static)
        for (int i = 0; i < nsub; ++i) {
            int t = subset ? subset[i] : i;
            for (int h = 0; h < H; ++h) {
                double s = 0.0;
                for (int k = 0; k < K; ++k) {
                    int row = i * K + k;
                    if (!valid[row]) continue;
                    s += (double)w[(size_t)t * K + k] * z[(size_t)row * H + h];
                }
                out_f64[(size_t)i * H + h] = s;
                if (out_bf16) out_bf16[(size_t)i * H + h] = orc_bf16_from_f64(s);
            }
            if (inter)
                for (int k = 0; k < K; ++k)
                    for (int j = 0; j < I; ++j)
                        inter[((size_t)i * K + k) * I + j] = valid[i * K + k] ? yq[((size_t)i * K + k) * I + j] : NAN;
        }
        free(a);
        free(yq);
        free(z);
        free(valid);
    }
done_early:
    free(slot);
    free(sorted_ids);
    free(block_expert);
    free(count);
    free(offset);
    return dropped;
}

int64_t orc_moe_dense(const uint16_t* x, const int32_t* ids, const float* w,
                      int T, int H, int I, int E, int K,
                      const uint8_t* w13, const uint8_t* w13s,
                      const uint8_t* w2, const uint8_t* w2s,
                      int act, double beta, double lbeta, int a_dtype,
                      double* out_f64, uint16_t* out_bf16) {
    if (bad_shape(T, H, I, E, K)) return -1;
    int64_t dropped = 0;
    for (int t = 0; t < T; ++t)
        for (int k = 0; k < K; ++k)
            if (ids[t * K + k] < 0 || ids[t * K + k] >= E) ++dropped;
#pragma omp parallel for schedule(dynamic)
    for (int t = 0; t < T; ++t) {
        double* a = (double*)malloc(sizeof(double) * (size_t)H);
        double* y = (double*)malloc(sizeof(double) * (size_t)I);
        double* yq = (double*)malloc(sizeof(double) * (size_t)I);
        double* acc = (double*)calloc((size_t)H, sizeof(double));
        orc_activation_row(x + (size_t)t * H, H, a_dtype, a);
        for (int k = 0; k < K; ++k) {
            int e = ids[t * K + k];
            if (e < 0 || e >= E) continue;
            for (int j = 0; j < I; ++j) {
                double g = 0.0, u = 0.0;
                size_t gate = (size_t)e * 2 * I + j, up = gate + I;
                for (int h = 0; h < H; ++h) {
                    uint8_t bg = w13[gate * (H / 2) + h / 2], bu = w13[up * (H / 2) + h / 2];
                    double wg = orc_e2m1_value((h & 1) ? bg >> 4 : bg & 15) * orc_e8m0_value(w13s[gate * (H / 32) + h / 32]);
                    double wu = orc_e2m1_value((h & 1) ? bu >> 4 : bu & 15) * orc_e8m0_value(w13s[up * (H / 32) + h / 32]);
                    g += a[h] * wg;
                    u += a[h] * wu;
                }
                y[j] = orc_act(act, g, u, beta, lbeta);
            }
            orc_requantize_intermediate(y, I, a_dtype, yq);
            for (int h = 0; h < H; ++h) {
                size_t row = (size_t)e * H + h;
                double s = 0.0;
                for (int i = 0; i < I; ++i) {
                    uint8_t bw = w2[row * (I / 2) + i / 2];
                    s += yq[i] * orc_e2m1_value((i & 1) ? bw >> 4 : bw & 15) * orc_e8m0_value(w2s[row * (I / 32) + i / 32]);
                }
                acc[h] += (double)w[t * K + k] * s;
            }
        }
        for (int h = 0; h < H; ++h) {
            out_f64[(size_t)t * H + h] = acc[h];
            if (out_bf16) out_bf16[(size_t)t * H + h] = orc_bf16_from_f64(acc[h]);
        }
        free(a);
        free(y);
        free(yq);
        free(acc);
    }
    return dropped;
}

/* ---------------------------------------------------------------------------
 * Expert parallelism over R ranks ("Add Kimi-K3 A8W4 support to the FlyDSL
 * MegaMoE V2 operator", Motivation and Technical Details: EP8 with 112 experts
 * per rank; each rank computes its experts' share of a token and sends it back
 * over the combine wire, quantised to fp8 blockwise 1x32). Rank r owns global
 * experts [r*El, (r+1)*El). Its share of token t is the top-k-weighted sum of
 * the stage-2 rows of t's pairs routed to it (the grouped forward with every
 * other pair dropped), held in fp32; with wire != 0 it is then quantised to
 * e4m3 with 1x32 e8m0 scales along H and dequantised (the wire), and the
 * shares are added over r (fp64) and rounded once to bf16.
 * ------------------------------------------------------------------------- */
int64_t orc_ep_forward(const uint16_t* x, const int32_t* ids, const float* w,
                       int T, int H, int I, int El, int R, int K,
                       const uint8_t* w13, const uint8_t* w13s,
                       const uint8_t* w2, const uint8_t* w2s,
                       int act, double beta, double lbeta, int a_dtype, int wire,
                       const int32_t* subset, int nsub,
                       double* out_f64, uint16_t* out_bf16) {
    if (bad_shape(T, H, I, El, K) || R <= 0) return -1;
    if (!subset) nsub = T;
    int64_t n = (int64_t)T * K;
    int32_t* ids_r = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
    double* part = (double*)malloc(sizeof(double) * (size_t)nsub * H + 1);
    double* p32 = (double*)malloc(sizeof(double) * (size_t)H);
    double* deq = (double*)malloc(sizeof(double) * (size_t)H);
    uint8_t* codes = (uint8_t*)malloc((size_t)H);
    uint8_t* scales = (uint8_t*)malloc((size_t)(H / 32));
    for (int64_t i = 0; i < (int64_t)nsub * H; ++i) out_f64[i] = 0.0;
    for (int r = 0; r < R; ++r) {
        for (int64_t p = 0; p < n; ++p)
            ids_r[p] = (ids[p] >= r * El && ids[p] < (r + 1) * El) ? ids[p] - r * El : -1;
        const size_t e0 = (size_t)r * El;
        int64_t st = orc_moe_forward(x, ids_r, w, T, H, I, El, K,
                                     w13 + e0 * 2 * I * (H / 2), w13s + e0 * 2 * I * (H / 32),
                                     w2 + e0 * H * (I / 2), w2s + e0 * H * (I / 32),
                                     act, beta, lbeta, a_dtype, 16, subset, nsub, part, NULL, NULL);
        if (st < 0) { nsub = -1; break; }
        for (int i = 0; i < nsub; ++i) {
            const double* pr = part + (size_t)i * H;
            if (wire) {
                for (int h = 0; h < H; ++h) p32[h] = (double)(float)pr[h];  /* the share is held in fp32 */
                orc_mx_quantize_f64(p32, H / 32, ORC_FMT_E4M3, codes, scales);
                orc_mx_dequantize(codes, scales, H / 32, ORC_FMT_E4M3, deq);
                for (int h = 0; h < H; ++h) out_f64[(size_t)i * H + h] += deq[h];
            } else {
                for (int h = 0; h < H; ++h) out_f64[(size_t)i * H + h] += pr[h];
            }
        }
    }
    if (nsub >= 0 && out_bf16)
        for (int64_t i = 0; i < (int64_t)nsub * H; ++i) out_bf16[i] = orc_bf16_from_f64(out_f64[i]);
    free(ids_r); free(part); free(p32); free(deq); free(codes); free(scales);
    return nsub < 0 ? -1 : 0;
}

/* Stage 1 of one expert for a list of token rows (the same steps as the grouped
 * forward: activation operand, g and u against the expert's dequantised gate and
 * up rows, act, fp32 holding, requantisation). */
int64_t orc_expert_stage1(const uint16_t* x, const int32_t* tokens, int nrows, int H, int I,
                          const uint8_t* w13e, const uint8_t* w13se, int act, double beta, double lbeta,
                          int a_dtype, double* y32, double* yq) {
    if (nrows < 0 || H <= 0 || I <= 0 || H % 32 || I % 32) return -1;
    double* W = (double*)malloc(sizeof(double) * (size_t)2 * I * H); /* dequantised gate and up rows */
    for (int j = 0; j < 2 * I; ++j)
        weight_row(w13e + (size_t)j * (H / 2), w13se + (size_t)j * (H / 32), H, W + (size_t)j * H);
#pragma omp parallel for schedule(dynamic)
    for (int r = 0; r < nrows; ++r) {
        double* a = (double*)malloc(sizeof(double) * (size_t)H);
        double* y = (double*)malloc(sizeof(double) * (size_t)I);
        orc_activation_row(x + (size_t)tokens[r] * H, H, a_dtype, a);
        for (int j = 0; j < I; ++j) {
            const double* wg = W + (size_t)j * H;
            const double* wu = W + (size_t)(I + j) * H;
            double g = 0.0, u = 0.0;
            for (int h = 0; h < H; ++h) { g += a[h] * wg[h]; u += a[h] * wu[h]; }
            y[j] = orc_act(act, g, u, beta, lbeta);
            if (y32) y32[(size_t)r * I + j] = (double)(float)y[j];
        }
        orc_requantize_intermediate(y, I, a_dtype, yq + (size_t)r * I);
        free(a);
        free(y);
    }
    free(W);
    return 0;
}

/* ---------------------------------------------------------------------------
 * Top-k softmax router. The pages route every token to its top 16 experts
 * (aiter PR 6259, Motivation: topk=16) but do not spell out the router; this is
 * the plain reading used by the small parity workload: softmax over the E
 * logits of a token, the K experts of largest probability, their probabilities
 * renormalised to sum to one. Softmax is strictly increasing in the logit, so
 * the K largest probabilities are the K largest logits; selecting on the logits
 * keeps ties exact (equal logits: the lower expert id first) even where two
 * probabilities would round to the same double. Selection order: descending
 * logit, then ascending id.
 * ------------------------------------------------------------------------- */
int64_t orc_route(const float* logits, int T, int E, int K, int32_t* ids, double* weights) {
    if (T < 0 || E <= 0 || K <= 0 || K > E) return -1;
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        const float* l = logits + (size_t)t * E;
        double* p = (double*)malloc(sizeof(double) * (size_t)E);
        char* taken = (char*)calloc((size_t)E, 1);
        double m = -INFINITY;
        for (int e = 0; e < E; ++e) m = fmax(m, (double)l[e]);
        double s = 0.0;
        for (int e = 0; e < E; ++e) { p[e] = exp((double)l[e] - m); s += p[e]; }
        for (int e = 0; e < E; ++e) p[e] /= s;                 /* softmax over all E */
        double sel = 0.0;
        for (int k = 0; k < K; ++k) {
            int best = -1;
            for (int e = 0; e < E; ++e)
                if (!taken[e] && (best < 0 || l[e] > l[best])) best = e;  /* strict: lower id wins ties */
            taken[best] = 1;
            ids[(size_t)t * K + k] = best;
            weights[(size_t)t * K + k] = p[best];
            sel += p[best];
        }
        for (int k = 0; k < K; ++k) weights[(size_t)t * K + k] /= sel;  /* renormalise over the K */
        free(p);
        free(taken);
    }
    return 0;
}

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
