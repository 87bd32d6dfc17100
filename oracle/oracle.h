/*
 * CPU fp64 oracle for the two-stage quantized MoE expert computation.
 *
 * TEST INFRASTRUCTURE ONLY. Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference leg of bench.py may load this library. The product
 * (the CUDA path under quantized_moe_expert_sort_gb300/) never includes,
 * links or calls anything here, and this file includes nothing from it.
 *
 * Sources (ROCm/aiter pull-request pages):
 *   - "Add Kimi-K3 A8W4 support to the FlyDSL MegaMoE V2 operator" (aiter PR 6259),
 *     Motivation: SiTUv2 situ(g)=b*tanh(g/b)*sigmoid(g), up=lb*tanh(u/lb), b=4, lb=25;
 *     Technical Details: fp8 1x32 block quantisation.
 *   - "Add an opt-in a4w4 SiTUv2 MoE path and fix three SiTUv2 tuner defects"
 *     (aiter PR 4463), What / Three tuner defects: activation dtypes a16w4 / a8w4 /
 *     a4w4; fp4x2 = two e2m1 codes per byte (low and high nibble).
 *   - "Retune Kimi-K3 a16w4 MoE tile geometry" (aiter PR 5118), Summary:
 *     moe_sorting pads every expert up to a full block_m; stage 2 applies the
 *     top-k weight and scatters rows back to their token ("bf16 atomic scatter").
 *   - "Support SiTUv2 in the packed-int4 MoE stage1 epilogue" (aiter PR 4471),
 *     Motivation: y = silu(g)*u for SiLU; SiTUv2 applied in the stage-1 epilogue.
 *
 * Readings where the pages are silent (the plain reading in each case):
 *   - MX scale rule: OCP MX, E = floor(log2(amax)) - emax_elem, clamped to
 *     [-127,127]; codes = RNE(v / 2^E) saturating; an all-zero block gets scale
 *     byte 127 and +0 codes.
 *   - fp8 is e4m3fn (max 448, no infinities).
 *   - fp4x2 byte j of a row: element 2j in the low nibble, 2j+1 in the high one.
 *   - w13 rows 0..I-1 are the gate projection, rows I..2I-1 the up projection.
 *   - the stage-1 output y is held in fp32 before its requantisation (bf16 for
 *     a16, fp8/fp4 1x32 for a8/a4), the precision the GPU path decides codes in.
 *   - the top-k weight multiplies the stage-2 row in full precision; the
 *     per-token sum is rounded once to bf16 (round to nearest even).
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_FMT_E2M1 = 0, ORC_FMT_E4M3 = 1 };
enum { ORC_ACT_SILU = 0, ORC_ACT_SITUV2 = 1 };
enum { ORC_A_BF16 = 0, ORC_A_FP8 = 1, ORC_A_FP4 = 2 };

/* Decoders of the element and scale formats. */
double orc_e2m1_value(int code);      /* code in [0,16) */
double orc_e4m3_value(int byte);      /* e4m3fn; 0x7F/0xFF decode to NaN */
double orc_e8m0_value(int byte);      /* 2^(byte-127); 0xFF decodes to NaN */
double orc_bf16_value(uint16_t bits);
uint16_t orc_bf16_from_f64(double v); /* round to nearest even, overflow to inf */
float orc_f32_from_f64(double v);     /* C cast (round to nearest even) */

/* Round one finite value to the element format (RNE, saturating); returns the
 * representable value. fmt is ORC_FMT_E2M1 or ORC_FMT_E4M3. */
double orc_round_to_format(double x, int fmt);
/* Code of a representable value (sign taken from signbit). -1 if not representable. */
int orc_encode(double r, int fmt);

/* MX 1x32 block quantisation of nblocks*32 values.
 * e2m1: codes has nblocks*16 bytes (packed, low nibble first); e4m3: nblocks*32.
 * scales has nblocks bytes (e8m0). */
void orc_mx_quantize_f64(const double* v, int64_t nblocks, int fmt, uint8_t* codes, uint8_t* scales);
void orc_mx_quantize_f32(const float* v, int64_t nblocks, int fmt, uint8_t* codes, uint8_t* scales);
void orc_mx_quantize_bf16(const uint16_t* v, int64_t nblocks, int fmt, uint8_t* codes, uint8_t* scales);
/* Dequantise nblocks*32 values back to fp64. */
void orc_mx_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t nblocks, int fmt, double* out);

/* The expert sort ("moe_sorting"): bucket pairs p = t*K+k by expert e = ids[p],
 * ascending p inside an expert, every non-empty expert padded to a multiple of
 * tile_m with the sentinel T*K. Blocks of tile_m rows are listed in ascending
 * expert order. Pairs whose id is outside [0,E) are dropped.
 * sorted_ids needs room for T*K + min(E,T*K)*(tile_m-1) entries, block_expert for
 * that / tile_m, expert_count for E, expert_offset for E+1.
 * Returns the number of dropped pairs. */
int64_t orc_sort(const int32_t* ids, int T, int K, int E, int tile_m,
                 int32_t* sorted_ids, int32_t* block_expert, int32_t* num_blocks,
                 int32_t* expert_count, int32_t* expert_offset);

/* y = act(g, u): SiLU  g*sigmoid(g)*u;
 *               SiTUv2 beta*tanh(g/beta)*sigmoid(g) * lbeta*tanh(u/lbeta). */
double orc_act(int act, double g, double u, double beta, double lbeta);

/* The stage-1 activation operand of one token: bf16 x as is (a16), or x
 * quantised to fp8 / fp4 with 1x32 e8m0 scales along H and dequantised
 * (a8 / a4). a receives H doubles. */
void orc_activation_row(const uint16_t* xrow, int H, int a_dtype, double* a);

/* The stage-1 output of one routed pair, y [I] (act(g, u) in fp64), held in
 * fp32 and requantised: bf16 (a16) or fp8 / fp4 with 1x32 e8m0 scales along I
 * (a8 / a4), dequantised into yq [I]. */
void orc_requantize_intermediate(const double* y, int I, int a_dtype, double* yq);

/* Stage 1 of one expert (w13e [2I, H/2] + w13se [2I, H/32]) for nrows token
 * rows tokens[r] of x (bf16 [*, H]): y32 [nrows, I] (optional) receives the
 * stage-1 output as held in fp32 before its requantisation, yq [nrows, I] the
 * requantised intermediate -- the values orc_moe_forward produces for those
 * pairs. Returns 0, or -1 on a bad argument. */
int64_t orc_expert_stage1(const uint16_t* x, const int32_t* tokens, int nrows, int H, int I,
                          const uint8_t* w13e, const uint8_t* w13se, int act, double beta, double lbeta,
                          int a_dtype, double* y32, double* yq);

/* Expert parallelism over R ranks of El experts each (global ids [0, R*El)):
 * rank r's share of every token (its routed pairs' weighted stage-2 rows, the
 * grouped forward with the other pairs dropped) held in fp32, with wire != 0
 * quantised to e4m3 1x32 (e8m0 scales along H) and dequantised, then summed
 * over the ranks and rounded once to bf16. Weights are the global arrays.
 * Arguments otherwise as orc_moe_forward. Returns 0, or -1 on a bad argument. */
int64_t orc_ep_forward(const uint16_t* x, const int32_t* ids, const float* w,
                       int T, int H, int I, int El, int R, int K,
                       const uint8_t* w13, const uint8_t* w13s,
                       const uint8_t* w2, const uint8_t* w2s,
                       int act, double beta, double lbeta, int a_dtype, int wire,
                       const int32_t* subset, int nsub,
                       double* out_f64, uint16_t* out_bf16);

/* Top-k softmax router over E logits per token (fp32 [T,E], finite or -inf,
 * at least one finite per token): ids [T,K] in descending logit order (equal
 * logits: lower id first), weights [T,K] = the softmax probabilities of those
 * experts renormalised over the K. Returns 0, or -1 on a bad argument. */
int64_t orc_route(const float* logits, int T, int E, int K, int32_t* ids, double* weights);

/* Whole forward pass, grouped by expert through orc_sort.
 * x bf16 [T,H]; ids int32 [T,K]; w fp32 [T,K];
 * w13 [E,2I,H/2] + w13s [E,2I,H/32]; w2 [E,H,I/2] + w2s [E,H,I/32].
 * subset: token indices to evaluate (NULL = all T), nsub entries.
 * out_f64 [nsub,H] (sum before rounding), out_bf16 [nsub,H];
 * inter (optional) [nsub*K, I]: the requantised stage-1 output of pair
 * (subset[i], k) at row i*K+k, NaN for a dropped pair.
 * Returns the number of dropped pairs, or -1 on a bad argument. */
int64_t orc_moe_forward(const uint16_t* x, const int32_t* ids, const float* w,
                        int T, int H, int I, int E, int K,
                        const uint8_t* w13, const uint8_t* w13s,
                        const uint8_t* w2, const uint8_t* w2s,
                        int act, double beta, double lbeta, int a_dtype, int tile_m,
                        const int32_t* subset, int nsub,
                        double* out_f64, uint16_t* out_bf16, double* inter);

/* The same function written as a plain per-token loop over (t,k), no sort:
 * the brute-force check of orc_moe_forward. Same arguments, all tokens. */
int64_t orc_moe_dense(const uint16_t* x, const int32_t* ids, const float* w,
                      int T, int H, int I, int E, int K,
                      const uint8_t* w13, const uint8_t* w13s,
                      const uint8_t* w2, const uint8_t* w2s,
                      int act, double beta, double lbeta, int a_dtype,
                      double* out_f64, uint16_t* out_bf16);

/* Threads the OpenMP parts use (for reporting). */
int orc_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif
