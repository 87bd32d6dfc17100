// moe_sort_noalloc: the expert sort into caller-provided buffers, for callers
// that cannot allocate device memory.
//
// Who needs it: code that runs where a device allocation is not allowed or not
// wanted -- a serving engine whose memory pool has already claimed the GPU's
// memory at start-up, a latency-critical decode loop that must not risk the
// implicit device synchronisation a cudaMalloc can cause, or a one-shot routing
// call from another library that has no context object to own a workspace.
// moe_sort needs a moe_ctx (moe_create allocates its workspace); this entry
// point needs none.
//
// The only scratch the multi-CTA sort needs (one histogram row of num_experts
// counters per 4096-pair chunk) lives in the file-scope device array below,
// so the entry point itself never calls cudaMalloc / cudaFree or any routine
// that allocates. Every GPU that loads this library holds the array (1 MiB)
// until the process exits.
#include <cstdio>
#include <mutex>

#include "../../include/moe.h"
#include "common.cuh"
#include "kernels.h"

namespace {

// Histogram scratch of the multi-CTA sort: ceil(T*K / 4096) * E ints at most.
static __device__ __align__(256) int g_sort_noalloc_scratch[MOE_SORT_NOALLOC_SCRATCH_INTS];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
int* g_scratch_addr[kMaxDevices];  // device address of the array, per device
bool g_setup_done[kMaxDevices];

thread_local char g_noalloc_msg[256];

// Reports through moe_last_error_message(), like every other entry point.
moe_status noalloc_fail(moe_status s) {
  moe::set_last_error_message(g_noalloc_msg);
  return s;
}

// Once per device, with that device current: look up the array's device
// address (the host-side symbol is only a stand-in, not a device pointer) and
// raise the sort kernels' shared-memory limits. Allocates nothing.
moe_status setup_device(int dev, int** scratch) {
  if (dev < 0 || dev >= kMaxDevices) {
    snprintf(g_noalloc_msg, sizeof(g_noalloc_msg), "moe_sort_noalloc: device %d outside [0, %d)", dev, kMaxDevices);
    return noalloc_fail(MOE_ERR_UNSUPPORTED);
  }
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_setup_done[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_sort_noalloc_scratch);
    if (e != cudaSuccess) {
      snprintf(g_noalloc_msg, sizeof(g_noalloc_msg), "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
      return noalloc_fail(MOE_ERR_CUDA);
    }
    e = moe::prep_set_smem_limits();
    if (e != cudaSuccess) {
      snprintf(g_noalloc_msg, sizeof(g_noalloc_msg), "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
      return noalloc_fail(MOE_ERR_CUDA);
    }
    g_scratch_addr[dev] = static_cast<int*>(p);
    g_setup_done[dev] = true;
  }
  *scratch = g_scratch_addr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_sort_noalloc(const int32_t* topk_ids, int num_tokens, int topk, int num_experts,
                                       int tile_m, int32_t* sorted_ids, int32_t* block_expert,
                                       int32_t* expert_count, int32_t* expert_offset, int32_t* active_experts,
                                       int32_t* meta, void* stream) {
  if (num_tokens < 0 || topk <= 0 || num_experts <= 0 || num_experts > moe::SORT_MAX_EXPERTS ||
      tile_m < 1 || tile_m > 256 || (tile_m & (tile_m - 1))) {
    snprintf(g_noalloc_msg, sizeof(g_noalloc_msg),
             "moe_sort_noalloc: bad sizes (T=%d K=%d E=%d tile_m=%d; E <= %d, tile_m a power of two <= 256)",
             num_tokens, topk, num_experts, tile_m, moe::SORT_MAX_EXPERTS);
    return noalloc_fail(MOE_ERR_INVALID_ARG);
  }
  const long n = (long)num_tokens * topk;
  if (n > (1L << 30)) {
    snprintf(g_noalloc_msg, sizeof(g_noalloc_msg), "moe_sort_noalloc: T*K = %ld too large", n);
    return noalloc_fail(MOE_ERR_INVALID_ARG);
  }
  if (n > moe::SORT_SMALL_MAX_PAIRS) {
    const long chunks = (n + moe::SORT_CHUNK - 1) / moe::SORT_CHUNK;
    if (chunks * num_experts > MOE_SORT_NOALLOC_SCRATCH_INTS) {
      snprintf(g_noalloc_msg, sizeof(g_noalloc_msg),
               "moe_sort_noalloc: ceil(T*K/%d) * E = %ld exceeds the %d-int scratch; use moe_sort",
               moe::SORT_CHUNK, chunks * num_experts, MOE_SORT_NOALLOC_SCRATCH_INTS);
      return noalloc_fail(MOE_ERR_INVALID_ARG);
    }
  }
  if (!sorted_ids || !block_expert || !expert_count || !expert_offset || !active_experts || !meta ||
      (n > 0 && !topk_ids)) {
    snprintf(g_noalloc_msg, sizeof(g_noalloc_msg), "moe_sort_noalloc: NULL pointer");
    return noalloc_fail(MOE_ERR_INVALID_ARG);
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    snprintf(g_noalloc_msg, sizeof(g_noalloc_msg), "cudaGetDevice: %s", cudaGetErrorString(e));
    return noalloc_fail(MOE_ERR_CUDA);
  }
  int* scratch = nullptr;
  moe_status s = setup_device(dev, &scratch);
  if (s != MOE_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // meta[3] collects the device flags of this call: clear it first.
  e = cudaMemsetAsync(meta + 3, 0, sizeof(int32_t), st);
  if (e != cudaSuccess) {
    snprintf(g_noalloc_msg, sizeof(g_noalloc_msg), "cudaMemsetAsync: %s", cudaGetErrorString(e));
    return noalloc_fail(MOE_ERR_CUDA);
  }
  moe::SortOut so;
  so.sorted_ids = sorted_ids;
  so.block_expert = block_expert;
  so.expert_count = expert_count;
  so.expert_offset = expert_offset;
  so.active_experts = active_experts;
  so.meta = meta;
  const int cap_chunks = MOE_SORT_NOALLOC_SCRATCH_INTS / num_experts;
  e = moe::launch_sort(topk_ids, n, num_experts, tile_m, so, scratch, cap_chunks, meta + 3, st);
  if (e != cudaSuccess) {
    snprintf(g_noalloc_msg, sizeof(g_noalloc_msg), "sort launch: %s", cudaGetErrorString(e));
    return noalloc_fail(MOE_ERR_CUDA);
  }
  return MOE_OK;
}
