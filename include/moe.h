/*
 * moe.h - C ABI of the GB300 (sm_103a) two-stage quantized MoE expert computation.
 *
 * The operation (from the ROCm/aiter pull-request pages this library follows):
 *   - "Retune Kimi-K3 a16w4 MoE tile geometry" (aiter PR 5118), Summary:
 *     moe_sorting groups the routed (token, k) pairs by expert and pads every
 *     expert to a full tile of rows; stage 2 applies the top-k weight and
 *     scatters each row back to its token.
 *   - "Add an opt-in a4w4 SiTUv2 MoE path and fix three SiTUv2 tuner defects"
 *     (aiter PR 4463), What: the activation dtype is bf16 (a16w4), fp8 (a8w4)
 *     or fp4x2 (a4w4); weights are MXFP4 (e2m1 codes, two per byte, with an
 *     e8m0 scale per 32 elements along K).
 *   - "Add Kimi-K3 A8W4 support to the FlyDSL MegaMoE V2 operator" (aiter PR
 *     6259), Motivation: SiTUv2, situ(g) = beta*tanh(g/beta)*sigmoid(g),
 *     up = lbeta*tanh(u/lbeta), y = situ(g)*up, with beta = 4, lbeta = 25 for
 *     Kimi-K3; Technical Details: SiTUv2 in the stage-1 epilogue, 1x32
 *     blockwise fp8 quantisation.
 *   - "Support SiTUv2 in the packed-int4 MoE stage1 epilogue" (aiter PR 4471),
 *     Motivation: SiLU is y = silu(g)*u; an unsupported activation must be
 *     rejected instead of silently computing SiLU.
 *
 * For each token t and each of its K routed experts e = topk_ids[t,k]:
 *   a      = x[t] (bf16) or x[t] quantised to fp8/fp4 with 1x32 e8m0 scales
 *   g_j    = a . W13[e, j, :],  u_j = a . W13[e, I+j, :]      (j < I)
 *   y_j    = act(g_j, u_j), then requantised: bf16 (a16) or fp8/fp4 1x32 along I
 *   z_h    = y . W2[e, h, :]                                   (h < H)
 *   out[t] = bf16( sum_k topk_weights[t,k] * z )   (fp32 sum, one rounding)
 *
 * Layouts (all row-major, K contiguous; plain, not pre-swizzled):
 *   x            bf16   [T, H]
 *   topk_ids     int32  [T, K]   expert ids; ids outside [0,E) are dropped and
 *                                flagged (moe_get_error); duplicates are legal
 *   topk_weights fp32   [T, K]
 *   w13          uint8  [E, 2I, H/2]  e2m1 codes; rows 0..I-1 gate, I..2I-1 up;
 *                                     byte j of a row = element 2j (low nibble),
 *                                     element 2j+1 (high nibble)
 *   w13_scale    uint8  [E, 2I, H/32] e8m0 scales
 *   w2           uint8  [E, H, I/2]
 *   w2_scale     uint8  [E, H, I/32]
 *   out          bf16   [T, H]   overwritten
 *
 * Ownership: every tensor argument is a caller-owned device pointer (16-byte
 * aligned) unless the function says "host". The context owns its workspace
 * (sort buffers, quantised activations, intermediate, fp32 combine buffer),
 * sized once at moe_create for max_tokens. moe_forward and moe_sort allocate
 * nothing and never synchronise the stream; they only enqueue kernels.
 *
 * Errors: argument checks run on the host before anything is enqueued and
 * return a status; no C++ exception crosses this ABI. A CUDA launch error
 * returns MOE_ERR_CUDA (text in moe_last_error_message()). Conditions found on
 * the device (bad expert ids, a bounded wait that ran out) set bits of a
 * device error word read by moe_get_error.
 *
 * Requirements: a GPU of compute capability 10.3 (GB300); hidden and inter
 * multiples of 128; 1 <= num_experts <= 4096.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct moe_ctx moe_ctx;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size, T > max_tokens, beta <= 0 ... */
  MOE_ERR_UNSUPPORTED = 2,   /* unknown activation or dtype, wrong GPU, shape outside the limits */
  MOE_ERR_CUDA = 3,          /* a CUDA call failed */
  MOE_ERR_OOM = 4,           /* workspace allocation failed in moe_create */
  MOE_ERR_BAD_EXPERT_ID = 5, /* reported by moe_get_error's return: ids outside [0,E) were dropped */
  MOE_ERR_TIMEOUT = 6        /* reported by moe_get_error's return: a device wait ran out */
} moe_status;

typedef enum { MOE_ACT_SILU = 0, MOE_ACT_SITUV2 = 1 } moe_act;
typedef enum { MOE_A_BF16 = 0, MOE_A_FP8 = 1, MOE_A_FP4 = 2 } moe_adtype;

/* Device error word bits (moe_get_error). */
#define MOE_DEVERR_BAD_EXPERT 1
#define MOE_DEVERR_TIMEOUT 2
#define MOE_DEVERR_OVERFLOW 4
#define MOE_DEVERR_LAUNCH 8  /* a kernel got less shared memory than it needs and returned without work */

/* Sort output: device pointers into the context's workspace, valid until the
 * next call on the same context. Sizes are upper bounds; the real counts live
 * on the device in meta = {num_blocks, num_active, num_rows}.
 * ("Retune Kimi-K3 a16w4 MoE tile geometry", Summary: moe_sorting pads every
 * expert up to a full block_m.) */
typedef struct {
  int32_t* sorted_ids;     /* [max_rows]   pair id p = t*K+k per row; padding rows hold T*K */
  int32_t* block_expert;   /* [max_blocks] expert of each tile_m block, ascending */
  int32_t* expert_count;   /* [E]          valid pairs per expert */
  int32_t* expert_offset;  /* [E+1]        first row of each expert; expert_offset[E] = num_rows */
  int32_t* active_experts; /* [E]          experts with a nonzero count, ascending */
  int32_t* meta;           /* [4]          num_blocks, num_active, num_rows, (reserved) */
  int32_t tile_m;
  int64_t max_rows;
  int64_t max_blocks;
} moe_sort_view;

/* Workspace view for inspection (tests, debugging): device pointers owned by ctx.
 * inter_codes rows follow the sorted order of the last moe_forward (sort.tile_m
 * gives its padding: 1 on the few-rows tensor-core path, 128 on the many-rows
 * one); the element format follows its a_dtype: fp8 -> e4m3 bytes, fp4 -> e2m1
 * pairs, bf16 -> layout 2 below (a16_terms e2m1 code terms whose sum carries the bf16
 * intermediate). act_codes / act_scales hold per-token codes only after
 * moe_quantize_activations-style use; the forward writes activations straight
 * into sorted order. */
typedef struct {
  moe_sort_view sort;
  uint8_t* act_codes;      /* [max_tokens, H * bytes/elt] */
  uint8_t* act_scales;     /* [max_tokens, act_scale_stride] (first H/32 bytes of a row used) */
  uint8_t* inter_codes;    /* [max_rows, I * bytes/elt] */
  uint8_t* inter_scales;   /* [max_rows, inter_scale_stride] (first I/32 bytes of a row used) */
  float* acc32;            /* [max_tokens, H] fp32 combine buffer */
  int32_t act_scale_stride;   /* H/32 rounded up to 16 */
  int32_t inter_scale_stride; /* bytes per scale (sub-)row: I/32 rounded up to 16 */
  int32_t inter_scale_layout; /* 0: row-major [rows, inter_scale_stride];
                                 1: per 128-row tile b and 4-block chunk c, 512 bytes at
                                    (b * I/128 + c) * 512, byte 16*(m%32) + 4*(m/32) + kb%4
                                    for tile row m and 32-block kb (many-rows path);
                                 2: a16_terms e2m1 code terms per value, term t of row r
                                    stored as sub-row a16_terms * r + t: codes [a16_terms rows,
                                    I/2] (two codes per byte), scales [a16_terms rows,
                                    inter_scale_stride]; value = sum of the terms */
  /* The stage-1 activation operand the last moe_forward wrote (x quantised per
     32 along H) in the same sorted row order and with the same layout number as
     the intermediate above (H in place of I): codes [rows, H * bytes/elt] (layout
     2: [a16_terms rows, H/2]), scales as inter_scale_layout with
     act_sorted_scale_stride bytes per (sub-)row (layouts 0 and 2). */
  uint8_t* act_sorted_codes;
  uint8_t* act_sorted_scales;
  int32_t act_sorted_scale_stride;
  int32_t a16_terms;          /* e2m1 code terms per bf16 value in layout 2 (each term's scale
                                 by the MX rule on what the earlier terms left over) */
} moe_workspace_view;

/* Create a context on `device` for fixed (hidden, inter, num_experts, topk) and
 * up to max_tokens tokens per call. Allocates the whole workspace once.
 * Returns MOE_ERR_UNSUPPORTED if the device is not compute capability 10.3 or
 * a size is outside the limits above, MOE_ERR_OOM if allocation fails. */
moe_status moe_create(moe_ctx** ctx, int hidden, int inter, int num_experts, int topk, int max_tokens, int device);

/* Free the context and its workspace (synchronises its device). NULL is a no-op. */
moe_status moe_destroy(moe_ctx* ctx);

/* The expert sort alone (S1): bucket the num_tokens*topk pairs of topk_ids
 * (device int32 [T,K]) by expert, ascending pair id inside an expert, each
 * non-empty expert padded to a multiple of tile_m (1..256, a power of two) with
 * the sentinel T*K. Fills *out with pointers into ctx's workspace. Enqueued on
 * `stream` (a cudaStream_t; NULL = legacy default stream). */
moe_status moe_sort(moe_ctx* ctx, const int32_t* topk_ids, int num_tokens, int tile_m, moe_sort_view* out,
                    void* stream);

/* Scratch of moe_sort_noalloc, in ints (a 1 MiB device array per GPU). */
#define MOE_SORT_NOALLOC_SCRATCH_INTS 262144

/* The expert sort of moe_sort, into buffers the caller passes; the call itself
 * allocates no device memory. The aiter pages
 * have no counterpart: it serves callers of this library that cannot call
 * cudaMalloc -- a serving engine whose memory pool owns the GPU's memory, a
 * decode loop that must not risk the device synchronisation an allocation can
 * cause, or a library that routes tokens without holding a moe_ctx.
 * Runs on the calling thread's current device, enqueued on `stream`.
 * Outputs (device, caller-owned; same meaning as moe_sort_view):
 *   sorted_ids     [T*K + min(E, T*K)*(tile_m-1)]   block_expert [that / tile_m]
 *   expert_count   [E]   expert_offset [E+1]   active_experts [E]
 *   meta           [4]   num_blocks, num_active, num_rows, device flag bits
 *                        (MOE_DEVERR_BAD_EXPERT when ids were dropped)
 * Scratch: for T*K > 8192 the histogram rows, ceil(T*K/4096) * E ints, live in
 * a file-scope device array of MOE_SORT_NOALLOC_SCRATCH_INTS ints; larger
 * problems are rejected with MOE_ERR_INVALID_ARG (use moe_sort). Every call
 * shares that array: calls whose kernels overlap on the GPU (different streams
 * without ordering, or several host threads) race and must be serialised by
 * the caller. The first call on a device loads the library's module that holds
 * the array (under lazy module loading this is when its 1 MiB is reserved,
 * which can synchronise the device), looks up the array's device address and
 * sets kernel attributes: make that first call at start-up, before any stream
 * capture. */
moe_status moe_sort_noalloc(const int32_t* topk_ids, int num_tokens, int topk, int num_experts, int tile_m,
                            int32_t* sorted_ids, int32_t* block_expert, int32_t* expert_count,
                            int32_t* expert_offset, int32_t* active_experts, int32_t* meta, void* stream);

/* The whole two-stage forward pass (sort, activation quantisation, stage 1,
 * stage 2, combine) for num_tokens tokens, enqueued on `stream`. act and
 * a_dtype are the moe_act / moe_adtype values; beta and linear_beta are always
 * passed explicitly (no defaults; "Add an opt-in a4w4 SiTUv2 MoE path...",
 * Three tuner defects item 1) and must be finite and > 0; SiLU ignores them.
 * out (bf16 [T,H]) is overwritten. */
moe_status moe_forward(moe_ctx* ctx, const void* x, const int32_t* topk_ids, const float* topk_weights,
                       int num_tokens, const uint8_t* w13, const uint8_t* w13_scale, const uint8_t* w2,
                       const uint8_t* w2_scale, int act, float beta, float linear_beta, int a_dtype, void* out,
                       void* stream);

/* moe_forward with HOST buffers for the per-call data: x_host (bf16 [T,H]),
 * topk_ids_host, topk_weights_host and out_host (bf16 [T,H]) live in host
 * memory; the weights are device pointers. A buffer in page-locked memory that
 * the device can address (cudaHostAlloc / cudaMallocHost memory under unified
 * addressing, e.g. torch's pin_memory) is read or written by the kernels in
 * place, over the host link; any other buffer is copied through ctx-owned
 * device staging. Synchronises `stream` before returning. */
moe_status moe_forward_host(moe_ctx* ctx, const void* x_host, const int32_t* topk_ids_host,
                            const float* topk_weights_host, int num_tokens, const uint8_t* w13,
                            const uint8_t* w13_scale, const uint8_t* w2, const uint8_t* w2_scale, int act,
                            float beta, float linear_beta, int a_dtype, void* out_host, void* stream);

/* Activation block quantisation alone (S2): x bf16 [T,H] (device) -> codes and
 * e8m0 scales per 32 along H, the operand format stage 1 reads. a_dtype
 * MOE_A_FP8: e4m3 codes [T,H]; MOE_A_FP4: e2m1 pairs [T,H/2]. Scale rule
 * (OCP MX): an all-zero block gets scale 127 and +0 codes, else
 * E = floor(log2(amax)) - emax (2 for e2m1, 8 for e4m3), clamped to
 * [-127,127], scale byte E+127, code = RNE(v / 2^E) saturating.
 * MOE_A_BF16: the bf16 values re-encoded as IEEE half [T,H] (2 bytes each)
 * times one power of two per token, E = floor(log2(row amax)) - 15, written
 * into all H/32 scale bytes of the row; exact for every value no more than
 * 2^31 below its row's maximum.
 * Needs no context. */
moe_status moe_quantize_activations(const void* x, int num_tokens, int hidden, int a_dtype, uint8_t* codes,
                                    uint8_t* scales, void* stream);

/* Top-k softmax router (upstream of the expert computation). For each of the
 * num_tokens rows of logits (device fp32 [T,E], finite or -inf, at least one
 * finite per row; NaN is not allowed): softmax over the E logits, the topk
 * experts of largest probability, their probabilities renormalised over the
 * topk. The pages route every token to its top 16 of the global experts ("Add
 * Kimi-K3 A8W4 support to the FlyDSL MegaMoE V2 operator", Motivation); the
 * router arithmetic is the plain reading of that routing. Selection compares
 * the logits exactly (softmax is increasing in the logit), in descending order,
 * equal logits taking the lower expert id first; weights are computed in fp32
 * as exp(l_k - l_max) / sum over the chosen of exp(l_j - l_max).
 * Outputs (device, caller-owned): topk_ids int32 [T,K], topk_weights fp32 [T,K],
 * both in selection order -- the layout moe_forward takes. Limits:
 * 1 <= topk <= min(num_experts, 32), num_experts <= 4096; otherwise
 * MOE_ERR_INVALID_ARG. Needs no context; enqueued on `stream`. */
moe_status moe_route(const float* logits, int num_tokens, int num_experts, int topk, int32_t* topk_ids,
                     float* topk_weights, void* stream);

/* MXFP4 weight quantisation: fp32 w [rows, cols] (device, cols % 32 == 0) ->
 * e2m1 codes [rows, cols/2] + e8m0 scales [rows, cols/32] with the same rule.
 * Needs no context. */
moe_status moe_quantize_mxfp4(const float* w, int64_t rows, int cols, uint8_t* codes, uint8_t* scales,
                              void* stream);

/* Pointers into ctx's workspace (see moe_workspace_view). */
moe_status moe_get_workspace(moe_ctx* ctx, moe_workspace_view* out);

/* Synchronise ctx's device, read and clear the device error word.
 * *device_flags receives MOE_DEVERR_* bits. Returns MOE_OK when no bit was
 * set, else MOE_ERR_CUDA (MOE_DEVERR_LAUNCH), MOE_ERR_TIMEOUT or
 * MOE_ERR_BAD_EXPERT_ID, in that order of precedence. */
moe_status moe_get_error(moe_ctx* ctx, int32_t* device_flags);

/* Benchmark support: when enabled, each moe_forward records a CUDA event on
 * its stream before every kernel launch (group) and after the last one, so
 * that moe_read_profile can report per-kernel device time. Off by default. */
moe_status moe_set_profiling(moe_ctx* ctx, int enable);

/* After a profiled moe_forward: wait for its last event and return, in launch
 * order, the device time in ms (ms[i]) and a static name (names[i]) of each
 * launch group: "sort", "act_quant", "stage1", "stage2", "finalize".
 * *count is the capacity on entry and the number written on return. */
moe_status moe_read_profile(moe_ctx* ctx, float* ms, const char** names, int* count);

/* Expert parallelism emulated on one GPU ("Add Kimi-K3 A8W4 support to the
 * FlyDSL MegaMoE V2 operator": EP8 with 112 experts per rank; tokens dispatched
 * to the ranks owning their experts; each rank's stage-2 result sent back over
 * the combine wire quantised to fp8 blockwise 1x32). `ranks` ranks (<= 16) own
 * equal slices of the global experts: rank r owns [r*El, (r+1)*El), where El =
 * experts_per_rank. moe_ep_forward takes the same arguments as moe_forward, with
 * global expert ids and the global weight arrays [ranks*El, ...], and runs:
 *   dispatch: for each rank, the tokens with a pair routed to it (token order)
 *     copied into the rank's receive buffer (bf16 x, local ids with -1 for the
 *     pairs of other ranks, top-k weights) -- then one stream synchronisation so
 *     that the host knows each rank's token count (moe_ep_counts);
 *   per rank: the forward pass on its received tokens against its slice of the
 *     weights, its fp32 share of each token kept (no bf16 rounding);
 *   combine: each share quantised to e4m3 with an e8m0 scale per 32 along H
 *     (the MX rule), dequantised and summed over ranks in rank order (fp32),
 *     rounded once to bf16 into out (tokens without routed pairs get zeros).
 * Ids outside [0, ranks*El) are dropped and flagged (moe_ep_get_error). All
 * buffers are allocated at moe_ep_create for max_tokens tokens per call. */
typedef struct moe_ep moe_ep;
moe_status moe_ep_create(moe_ep** ep, int hidden, int inter, int experts_per_rank, int ranks, int topk,
                         int max_tokens, int device);
moe_status moe_ep_destroy(moe_ep* ep);
moe_status moe_ep_forward(moe_ep* ep, const void* x, const int32_t* topk_ids, const float* topk_weights,
                          int num_tokens, const uint8_t* w13, const uint8_t* w13_scale, const uint8_t* w2,
                          const uint8_t* w2_scale, int act, float beta, float linear_beta, int a_dtype, void* out,
                          void* stream);
/* Tokens each rank received in the last moe_ep_forward (host int32 [ranks]). */
moe_status moe_ep_counts(moe_ep* ep, int32_t* counts);
/* moe_get_error over the ranks: the union of their device flags, the first non-OK status. */
moe_status moe_ep_get_error(moe_ep* ep, int32_t* device_flags);

/* Prepacked stage-2 weights (an optimisation of the few-rows path; the plain
 * layout stays the contract and is still needed by the many-rows path).
 * moe_prepack_size: bytes of the packed copy (as many as w2 + w2_scale).
 * moe_prepack: enqueues on `stream` a copy of w2 [E,H,I/2] / w2_scale [E,H,I/32]
 * (device) into `packed` (device, caller-owned, 16-byte aligned, size above) as
 * contiguous blocks, one per (expert e, 128-row tile ht of H, 128-element chunk kc
 * of I): codes, 8 KB per block, row r (0..127) at block byte 64 r, holding
 * w2[e, 128 ht + r, 64 kc .. 64 kc + 63] -- for a_dtype bf16 and fp4 with the
 * 16-byte chunk c of row r stored at chunk c ^ ((r / 2) % 4) (the image the
 * kind::mxf4 kernels read), for fp8 in order; then the scales, 512 bytes per
 * block, byte 16*(r%32) + 4*(r/32) + b = w2_scale[e, 128 ht + r, 4 kc + b].
 * It binds the copy to ctx: later moe_forward calls with this same w2 pointer
 * and this a_dtype read it on the few-rows path. The caller keeps `packed`
 * alive and unchanged while bound; packed == NULL unbinds. Redo it if w2
 * changes. */
moe_status moe_prepack_size(moe_ctx* ctx, int64_t* bytes);
moe_status moe_prepack(moe_ctx* ctx, const uint8_t* w2, const uint8_t* w2_scale, int a_dtype, void* packed,
                       void* stream);

/* Failure-detection support (no GPU fault is involved in either).
 * moe_selftest_wait: one warp waits on a shared-memory barrier with the same
 * bounded wait every pipeline stage uses, but with a limit of limit_ns
 * (0 .. 1e10); complete != 0 completes the barrier first. A wait that runs out
 * sets MOE_DEVERR_TIMEOUT in ctx's device error word and the kernel returns,
 * so the next moe_get_error reports MOE_ERR_TIMEOUT and the context stays
 * usable. Enqueued on `stream`.
 * moe_debug_inject(MOE_INJECT_ALLOC_FAIL, n): the next moe_create (on any
 * thread) treats its n-th workspace allocation (0-based) as failed: it frees
 * what it had allocated and returns MOE_ERR_OOM. One-shot; n < 0 disarms. */
#define MOE_INJECT_ALLOC_FAIL 1
moe_status moe_selftest_wait(moe_ctx* ctx, int64_t limit_ns, int complete, void* stream);
moe_status moe_debug_inject(int what, int64_t arg);

/* Static text for a status. */
const char* moe_status_string(moe_status s);

/* Text of the last failing CUDA call or argument check on this thread. */
const char* moe_last_error_message(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
