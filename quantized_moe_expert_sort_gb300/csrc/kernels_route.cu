// Top-k softmax router: per token, softmax over the E router logits, the K
// experts of largest probability, their probabilities renormalised over the K.
//
// The aiter pages route each token to its top 16 experts ("Add Kimi-K3 A8W4
// support to the FlyDSL MegaMoE V2 operator", Motivation: topk=16); the router
// arithmetic itself is the plain reading used by the small workload. Softmax
// is strictly increasing in the logit, so the K largest probabilities are the K
// largest logits: selection compares the fp32 logits exactly (equal logits: the
// lower expert id first), which makes the ids independent of how exp rounds.
// The renormalised weight of a chosen expert is its softmax probability over
// the chosen K alone (the full-softmax denominator cancels):
//   w_k = exp(l_k - l_max) / sum_j exp(l_j - l_max),  j over the K chosen.
//
// One warp per token: the logits row is staged in shared memory; lane l owns
// elements l, l + 32, ...; each round the warp takes the maximum of the lanes'
// current best (value, then lowest id) with two hardware reductions, the owner
// lane marks it taken and rescans its own elements.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kRouteWarps = 8;

// fp32 -> unsigned key with the same order (non-NaN inputs); -0 and +0 are
// one key, as they compare equal.
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

}  // namespace

__global__ void __launch_bounds__(kRouteWarps * 32) route_topk_kernel(const float* __restrict__ logits, int T, int E,
                                                                      int K, int32_t* __restrict__ ids,
                                                                      float* __restrict__ weights) {
  extern __shared__ __align__(16) float rsm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* row = rsm + (size_t)warp * E;
  const int per = (E + 31) / 32;  // elements per lane (<= MOE_ROUTE_MAX_EXPERTS / 32)
  for (long t = (long)blockIdx.x * kRouteWarps + warp; t < T; t += (long)gridDim.x * kRouteWarps) {
    const float* src = logits + t * E;
    for (int e = lane; e < E; e += 32) row[e] = __ldg(src + e);
    __syncwarp();
    uint32_t taken[4] = {0u, 0u, 0u, 0u};  // bit j: element lane + 32 j already chosen
    auto rescan = [&](uint32_t* key, int* idx) {
      uint32_t bk = 0u;
      int bi = 0x7FFFFFFF;
      for (int j = 0; j < per; ++j) {
        const int e = lane + 32 * j;
        if (e < E && !((taken[j >> 5] >> (j & 31)) & 1u)) {
          const uint32_t k = order_key(row[e]);
          if (bi == 0x7FFFFFFF || k > bk) { bk = k; bi = e; }  // strict: the lower id keeps ties
        }
      }
      *key = bk;
      *idx = bi;
    };
    uint32_t bk;
    int bi;
    rescan(&bk, &bi);
    uint32_t my_key = 0u;
    int my_id = 0;
    for (int k = 0; k < K; ++k) {
      const uint32_t kmax = __reduce_max_sync(0xFFFFFFFFu, bi == 0x7FFFFFFF ? 0u : bk);
      const int win = (int)__reduce_min_sync(0xFFFFFFFFu, (bi != 0x7FFFFFFF && bk == kmax) ? (uint32_t)bi : 0x7FFFFFFFu);
      if (lane == k) { my_key = kmax; my_id = win; }
      if ((win & 31) == lane) {  // the owner marks it and finds its next best
        const int j = win >> 5;
        taken[j >> 5] |= 1u << (j & 31);
        rescan(&bk, &bi);
      }
    }
    const float lmax = key_value(__shfl_sync(0xFFFFFFFFu, my_key, 0));
    float ex = 0.0f;
    if (lane < K) ex = expf(key_value(my_key) - lmax);
    float s = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
    if (lane < K) {
      ids[t * K + lane] = my_id;
      weights[t * K + lane] = ex / s;
    }
    __syncwarp();
  }
}

cudaError_t route_set_smem_limits() {
  return cudaFuncSetAttribute(route_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)(sizeof(float) * kRouteWarps * ROUTE_MAX_EXPERTS));
}

cudaError_t launch_route(const float* logits, int T, int E, int K, int32_t* ids, float* weights, int num_sms,
                         cudaStream_t st) {
  long blocks = ((long)T + kRouteWarps - 1) / kRouteWarps;
  const long cap = (long)num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  route_topk_kernel<<<(unsigned)blocks, kRouteWarps * 32, sizeof(float) * kRouteWarps * E, st>>>(logits, T, E, K, ids,
                                                                                               weights);
  return cudaGetLastError();
}

}  // namespace moe
