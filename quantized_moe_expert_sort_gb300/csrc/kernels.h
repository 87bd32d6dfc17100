// Internal interface between the C-ABI host code and the kernel files.
#pragma once

#include <cstdint>
#include <utility>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda.h>

namespace moe {

// Sort output (device pointers). meta[] holds device-side counters.
enum { META_NUM_BLOCKS = 0, META_NUM_ACTIVE = 1, META_NUM_ROWS = 2, META_WORDS = 4 };

struct SortOut {
  int32_t* sorted_ids;      // [cap_rows]   pair id p = t*K+k per sorted row, sentinel T*K on padding
  int32_t* block_expert;    // [cap_blocks] expert of each tile_m block
  int32_t* expert_count;    // [E]          valid pairs per expert
  int32_t* expert_offset;   // [E+1]        first sorted row of each expert (padded prefix sum)
  int32_t* active_experts;  // [E]          experts with count > 0, ascending
  int32_t* meta;            // [META_WORDS] num_blocks, num_active, num_rows
  int32_t* pair_row = nullptr;  // [T*K] (optional) sorted row of each pair, -1 if dropped
  int4* active_info = nullptr;  // [E]   (optional) {expert, count, first row, 0} of each active expert
  int neg_masked = 0;           // 1: negative ids mean "no expert here" (skipped, not flagged)
};

constexpr int SORT_SMALL_MAX_PAIRS = 8192;  // single-CTA sort up to this many pairs
constexpr int SORT_CHUNK = 4096;            // pairs per CTA in the multi-CTA sort
constexpr int SORT_MAX_EXPERTS = 4096;      // shared-memory bound of the sort kernels

// Kernel launch; pdl = programmatic dependent launch: the kernel may start while
// the previous kernel in the stream drains, and waits for it (griddepcontrol.wait)
// before it reads that kernel's results. Every kernel launched with pdl calls
// pdl_wait() before its first dependent read.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                            Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

size_t sort_small_smem(int E);
size_t sort_scatter_smem(int E, long n);  // dynamic shared memory of the fused sort + scatter
// Text returned by moe_last_error_message() on this thread.
void set_last_error_message(const char* msg);
cudaError_t prep_set_smem_limits();
cudaError_t launch_sort(const int32_t* ids, long n, int E, int tile_m, const SortOut& so, int* hist,
                        int hist_cap_chunks, int* err, cudaStream_t st);
cudaError_t launch_act_quant(const void* x, int T, int H, int fmt, uint8_t* xq, uint8_t* xs, int xs_stride,
                             float* acc32, int num_sms, cudaStream_t st);
cudaError_t launch_weight_quant(const float* w, long nblocks, uint8_t* codes, uint8_t* scales, int num_sms,
                                cudaStream_t st);
cudaError_t launch_finalize(const float* acc32, long n, void* out, int num_sms, cudaStream_t st);
// Activation quantisation for the tensor-core paths: each token's row is
// quantised once (four threads per 32-block) and written straight to the sorted
// rows of its routed pairs, codes [rows, row_bytes] and e8m0 scales
// [rows, sstride], both row-major. mode SW_A8: e4m3; SW_A4: e2m1;
// SW_A16: A16_TERMS e2m1 terms whose sum carries the bf16 value, term t of
// sorted row r stored as sub-row r * A16_TERMS + t (codes [sub-rows, H/2],
// scales [sub-rows, sstride]).
// sstride 0 (SW_A8 / SW_A4 only): scales go to the 512-byte tcgen05.cp
// chunks of 128-row tiles instead (byte 16*(m%32) + 4*(m/32) + b%4 of chunk
// (r/128) * H/128 + b/4 for sorted row r, m = r % 128, 32-block b).
struct ScatterOut {
  uint8_t* codes;
  uint8_t* scales;
  int sstride;
  float* acc32;         // fp32 combine buffer [T,H], zeroed (nullptr: untouched)
  const float* topk_w;  // row_tok / row_w (optional): token and top-k weight of every sorted row
  int32_t* row_tok;
  float* row_w;
};
cudaError_t launch_act_scatter(const void* x, int T, int H, int K, int mode, const int32_t* pair_row,
                               const ScatterOut& so, int num_sms, cudaStream_t st);
// The single-CTA sort and the scatter above in one launch (n <= SORT_SMALL_MAX_PAIRS):
// every CTA sorts in shared memory, CTA 0 writes the sort outputs.
cudaError_t launch_sort_scatter(const int32_t* ids, long n, int E, int tile_m, const SortOut& so, int* err,
                                const void* x, int T, int H, int K, int mode, const ScatterOut& sc, int num_sms,
                                cudaStream_t st);

// One warp waits on an mbarrier with a limit of limit_ns (complete != 0: the
// barrier completes first); a wait that runs out sets DEV_ERR_TIMEOUT in *err.
cudaError_t launch_wait_selftest(uint64_t limit_ns, int complete, int* err, cudaStream_t st);

// Stage-2 weights repacked for the few-rows kernels (kernels_pack.cu): codes as 8 KB
// blocks [E][H/128][I/128][128 rows][64 bytes] (swz: each block pre-swizzled as the
// 64-byte-swizzle shared-memory image), scales as 512-byte tcgen05.cp chunks
// [E][H/128][I/128] (byte 16*(r%32) + 4*(r/32) + b for row r, 32-block b).
cudaError_t launch_prepack_w2(const uint8_t* w2, const uint8_t* w2s, int E, int H, int I, int swz, uint8_t* pc,
                              uint8_t* ps, int num_sms, cudaStream_t st);

// Expert-parallel emulation (kernels_ep.cu): ranks of El experts, received rows [R][maxT].
constexpr int EP_MAX_RANKS = 16;
struct EpShares {
  const float* acc[EP_MAX_RANKS];  // each rank's fp32 share [its received rows, H]
};
cudaError_t launch_ep_dispatch(const void* x, const int32_t* ids, const float* w, int T, int H, int K, int El, int R,
                               int maxT, int32_t* recv_tok, int32_t* recv_ids, float* recv_w, int32_t* slot,
                               int32_t* counts, void* recv_x, int* err, int num_sms, cudaStream_t st);
cudaError_t launch_ep_combine(const EpShares& shares, const int32_t* counts, const int32_t* slot, int T, int H, int R,
                              int maxT, uint8_t* codes, uint8_t* scales, void* out, int num_sms, cudaStream_t st);

// Top-k softmax router over E logits per token (kernels_route.cu).
constexpr int ROUTE_MAX_EXPERTS = 4096;
constexpr int ROUTE_MAX_TOPK = 32;
cudaError_t route_set_smem_limits();
cudaError_t launch_route(const float* logits, int T, int E, int K, int32_t* ids, float* weights, int num_sms,
                         cudaStream_t st);

// Parameters of the grouped stage kernels.
struct StageParams {
  // activation operand of this stage: block-scaled codes [rows, Kdim] + e8m0 [rows, Kdim/32]
  const uint8_t* aq;
  const uint8_t* as;
  // weight scales [E, Ndim, Kdim/32]
  const uint8_t* wscale;
  // sort output
  const int32_t* sorted_ids;
  const int32_t* block_expert;
  const int32_t* expert_offset;
  const int32_t* expert_count;
  const int32_t* active_experts;
  const int32_t* meta;
  // stage-1 output (intermediate) or stage-2 combine target
  uint8_t* oq;        // stage 1: [rows, I] codes
  uint8_t* os;        // stage 1: [rows, I/32] scales
  float* acc32;       // stage 2: [T, H]
  const float* topk_w;  // stage 2: [T*K]
  const int32_t* row_tok;  // few-rows path: token of each sorted row
  const float* row_w;      // few-rows path: top-k weight of each sorted row
  const int4* active_info; // few-rows path: {expert, count, first row, 0} per active expert
  int xs_stride;       // bytes per row of the activation-scale array (as)
  int os_stride;       // stage 1: bytes per row of the output-scale array (os)
  int tile_group;      // many-rows stage 2: N tiles per group of the tile order (<= 0: block-major)
  const uint8_t* wpacked;  // few-rows stage 2, prepacked weights: the packed codes (wscale: their scales)

  int T, H, I, E, K;
  int act;
  float beta, lbeta;
  int* err;
};

// Row stride of the workspace's e8m0 scale arrays: kdim/32 bytes rounded up to
// 16, so that every row can be moved with one 16-byte-aligned bulk copy.
__host__ __device__ inline int scale_row_stride(int kdim) { return ((kdim / 32) + 15) & ~15; }

// tcgen05 family (block-scaled tensor-core MMA, 128 x 128 tiles, tile_m = 128)
enum { TC_A8W4 = 0, TC_A4W4 = 1 };
constexpr int TC_TILE_M = 128;
constexpr int TC_MAX_K = 4096;  // reduction length the tensor-core stages accept (weight-scale staging)
using TcParams = StageParams;
cudaError_t tc_set_smem_limits();
cudaError_t launch_tc_stage(int kind, int stage, const TcParams& p, const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                            int grid, cudaStream_t st);

// tcgen05 family for few routed rows per expert (decode): the weight tile is
// the M = 128 operand and the expert's routed rows the N <= 64 operand.
enum { SW_A16 = 0, SW_A8 = 1, SW_A4 = 2 };
constexpr int A16_TERMS = 6;  // e2m1 code terms carrying one bf16 value (few-rows path)
cudaError_t swap_set_smem_limits();
// Shared-memory bytes per operand row (TMA box width) of the few-rows kernels'
// (kind, stage): the tensor maps the host encodes must use this box width.
int swap_row_bytes(int kind, int stage);
// packed (stage 2 only): the weights come prepacked (launch_prepack_w2).
// ks (stage 1 only): 1, or a split of K over clusters of ks = 2 or 3 CTAs (grid a multiple of ks).
// swap_split_max_clusters: how many such clusters of the stage-1 kernel fit on the device at once.
int swap_split_max_clusters(int kind, int ks);
cudaError_t launch_swap_stage(int kind, int stage, bool packed, int ks, const StageParams& p, const CUtensorMap& tm_w,
                              const CUtensorMap& tm_x, int grid, cudaStream_t st);


}  // namespace moe
