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
// One warp per token. Selection is exact in two steps:
//  1. Threshold. With t0 the K-th largest of the 32 lanes' maxima, at least K
//     elements are >= t0 (those K maxima), so the K-th largest logit is >= t0
//     and every element of the top K -- ties at the boundary included -- is
//     among the candidates {e : l_e >= t0}.  For Gaussian logits (E = 896,
//     K = 16) there are about 30 of them.
//  2. Order. The candidates are put in (logit descending, id ascending) order;
//     the first K are the result.
// When more candidates pass the threshold than step 2 takes (128 in the
// register kernel, 512 in the shared-memory one: heavy ties, e.g. a quantised
// logit grid), the warp falls back to K rounds of "take the largest
// remaining": the maximum of the lanes' current best (value, then lowest id)
// with two hardware reductions, the owner lane marking it.
//
// Two kernels. For E <= 1024 (route_reg_kernel) each lane keeps its PER = E/32
// (rounded up to 4, 8, 16 or 32) logits in registers, read with 16-byte loads
// when E % 4 == 0; t0 comes from a bitonic sort of the 32 lane maxima across
// the warp, and up to 32 candidates are ordered by a second bitonic sort (more:
// each candidate's slot is the number of candidates before it). Larger E (up to
// 4096, route_topk_kernel) stages the row in shared memory, lane l owning
// elements l, l + 32, ..., and ranks the candidates.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kRouteWarps = 8;
constexpr int kCandMax = 128;      // candidates above the threshold the rank step takes (E <= 1024)
constexpr int kCandMaxWide = 512;  // the same for the shared-memory kernel (E up to 4096)

struct RouteScratch {  // per warp, after the staged logits rows
  uint32_t ckey[kCandMaxWide];
  int32_t cid[kCandMaxWide];
  uint32_t skey[ROUTE_MAX_TOPK];
  int32_t sid[ROUTE_MAX_TOPK];
};

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

// Candidate list (rank step) and chosen slots of one warp, in shared memory.
struct RouteCand {
  uint32_t ckey[kCandMax];
  int32_t cid[kCandMax];
  uint32_t skey[ROUTE_MAX_TOPK];
  int32_t sid[ROUTE_MAX_TOPK];
};

// Register-resident router for E <= 32 * PER. Lane l holds the logits of
// elements eid(j), j < PER: with VEC (E % 4 == 0, 16-byte aligned rows) the 4
// floats of 16-byte word l + 32 (j / 4), else element l + 32 j. Slots past E
// hold -inf and are excluded by their index. Logits are compared as floats
// (-0 == +0, as in the order-key kernel; NaN is outside the contract), ties by id.
//
// The K-th largest lane maximum comes from a bitonic sort of the 32 maxima
// across the warp; up to 32 candidates are put in (logit desc, id asc) order by
// a second bitonic sort, so lane k holds the k-th expert.
template <int PER, bool VEC>
__global__ void __launch_bounds__(kRouteWarps * 32) route_reg_kernel(const float* __restrict__ logits, int T, int E,
                                                                     int K, int32_t* __restrict__ ids,
                                                                     float* __restrict__ weights) {
  __shared__ RouteCand cand[kRouteWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  RouteCand* rc = cand + warp;
  const float ninf = -__int_as_float(0x7F800000);
  auto eid = [&](int j) { return VEC ? 4 * (lane + 32 * (j >> 2)) + (j & 3) : lane + 32 * j; };
  for (long t = (long)blockIdx.x * kRouteWarps + warp; t < T; t += (long)gridDim.x * kRouteWarps) {
    const float* src = logits + t * E;
    float v[PER];
    if (VEC) {
#pragma unroll
      for (int j4 = 0; j4 < PER / 4; ++j4) {
        const int q = lane + 32 * j4;
        float4 w = make_float4(ninf, ninf, ninf, ninf);
        if (4 * q < E) w = __ldg(reinterpret_cast<const float4*>(src) + q);
        v[4 * j4] = w.x;
        v[4 * j4 + 1] = w.y;
        v[4 * j4 + 2] = w.z;
        v[4 * j4 + 3] = w.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < PER; ++j) {
        const int e = lane + 32 * j;
        v[j] = e < E ? __ldg(src + e) : ninf;
      }
    }
    // 1. threshold: the K-th largest lane maximum (bitonic sort, descending)
    float s = ninf;
#pragma unroll
    for (int j = 0; j < PER; ++j) s = fmaxf(s, v[j]);
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1)
#pragma unroll
      for (int j = k >> 1; j > 0; j >>= 1) {
        const float o = __shfl_xor_sync(0xFFFFFFFFu, s, j);
        s = (((lane & j) == 0) == ((lane & k) == 0)) ? fmaxf(s, o) : fminf(s, o);
      }
    const float t0 = __shfl_sync(0xFFFFFFFFu, s, K - 1);
    // candidates: this lane's count, an exclusive prefix over the lanes
    int cnt = 0;
#pragma unroll
    for (int j = 0; j < PER; ++j) cnt += (v[j] >= t0 && eid(j) < E) ? 1 : 0;
    int pre = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xFFFFFFFFu, pre, o);
      if (lane >= o) pre += x;
    }
    const int C = __shfl_sync(0xFFFFFFFFu, pre, 31);
    float my_v = ninf;
    int my_id = 0;
    if (C <= kCandMax) {
      int pos = pre - cnt;
#pragma unroll
      for (int j = 0; j < PER; ++j)
        if (v[j] >= t0 && eid(j) < E) {
          rc->ckey[pos] = __float_as_uint(v[j]);
          rc->cid[pos] = eid(j);
          ++pos;
        }
      __syncwarp();
      if (C <= 32) {
        // 2. bitonic sort of the candidates by (logit desc, id asc); padding lanes sort last
        float ck = lane < C ? __uint_as_float(rc->ckey[lane]) : ninf;
        int ci = lane < C ? rc->cid[lane] : 0x7FFFFFFF;
#pragma unroll
        for (int k = 2; k <= 32; k <<= 1)
#pragma unroll
          for (int j = k >> 1; j > 0; j >>= 1) {
            const float ok = __shfl_xor_sync(0xFFFFFFFFu, ck, j);
            const int oi = __shfl_xor_sync(0xFFFFFFFFu, ci, j);
            const bool o_first = ok > ck || (ok == ck && oi < ci);  // the partner comes first
            const bool keep_first = ((lane & j) == 0) == ((lane & k) == 0);
            if (keep_first ? o_first : !o_first) { ck = ok; ci = oi; }
          }
        my_v = ck;
        my_id = ci;
      } else {
        // 2. rank the candidates; slot < K is the output position
        for (int c = lane; c < C; c += 32) {
          const float k = __uint_as_float(rc->ckey[c]);
          const int id = rc->cid[c];
          int r = 0;
          for (int d = 0; d < C; ++d) {
            const float kd = __uint_as_float(rc->ckey[d]);
            r += (kd > k) || (kd == k && rc->cid[d] < id);
          }
          if (r < K) { rc->skey[r] = __float_as_uint(k); rc->sid[r] = id; }
        }
        __syncwarp();
        if (lane < K) { my_v = __uint_as_float(rc->skey[lane]); my_id = rc->sid[lane]; }
      }
      __syncwarp();
    } else {
      // K rounds of "take the largest remaining" (bit j of taken: slot j chosen)
      uint32_t taken = 0u;
      for (int k = 0; k < K; ++k) {
        uint32_t bk = 0u;  // order key of the best live slot (0: none)
        int bi = 0x7FFFFFFF;
#pragma unroll
        for (int j = 0; j < PER; ++j) {
          const int e = eid(j);
          const uint32_t kj = order_key(v[j]);
          if (e < E && !((taken >> j) & 1u) && (kj > bk || (kj == bk && e < bi))) { bk = kj; bi = e; }
        }
        const uint32_t kmax = __reduce_max_sync(0xFFFFFFFFu, bk);
        const int win = (int)__reduce_min_sync(0xFFFFFFFFu, bk == kmax ? (uint32_t)bi : 0x7FFFFFFFu);
        if (lane == k) { my_v = key_value(kmax); my_id = win; }
#pragma unroll
        for (int j = 0; j < PER; ++j)
          if (eid(j) == win) taken |= 1u << j;
      }
    }
    const float lmax = __shfl_sync(0xFFFFFFFFu, my_v, 0);
    float ex = 0.0f;
    if (lane < K) ex = expf(my_v - lmax);
    float sum = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
    if (lane < K) {
      ids[t * K + lane] = my_id;
      weights[t * K + lane] = ex / sum;
    }
  }
}

}  // namespace

__global__ void __launch_bounds__(kRouteWarps * 32) route_topk_kernel(const float* __restrict__ logits, int T, int E,
                                                                      int K, int32_t* __restrict__ ids,
                                                                      float* __restrict__ weights) {
  extern __shared__ __align__(16) float rsm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* row = rsm + (size_t)warp * E;
  RouteScratch* rs = reinterpret_cast<RouteScratch*>(rsm + (size_t)kRouteWarps * E) + warp;
  const int per = (E + 31) / 32;  // elements per lane (<= ROUTE_MAX_EXPERTS / 32)
  const uint32_t lt_mask = (1u << lane) - 1u;
  const bool vec = (E & 3) == 0 && (reinterpret_cast<uintptr_t>(logits) & 15) == 0;
  for (long t = (long)blockIdx.x * kRouteWarps + warp; t < T; t += (long)gridDim.x * kRouteWarps) {
    const float* src = logits + t * E;
    if (vec) {
      for (int q = lane; q < E / 4; q += 32)
        reinterpret_cast<float4*>(row)[q] = __ldg(reinterpret_cast<const float4*>(src) + q);
    } else {
      for (int e = lane; e < E; e += 32) row[e] = __ldg(src + e);
    }
    __syncwarp();
    // 1. threshold: the K-th largest lane maximum (lanes without elements hold
    // key 0, below every non-NaN logit's key; K <= E keeps them out of the top K)
    uint32_t lm = 0u;
    for (int j = 0; j < per; ++j) {
      const int e = lane + 32 * j;
      if (e < E) lm = max(lm, order_key(row[e]));
    }
    int lr = 0;  // this lane's maximum ranked among the 32 (key descending, lane ascending)
#pragma unroll 8
    for (int l = 0; l < 32; ++l) {
      const uint32_t o = __shfl_sync(0xFFFFFFFFu, lm, l);
      lr += (o > lm) || (o == lm && l < lane);
    }
    const uint32_t t0 = __reduce_min_sync(0xFFFFFFFFu, lr < K ? lm : 0xFFFFFFFFu);
    int C = 0;
    for (int j = 0; j < per; ++j) {
      const int e = lane + 32 * j;
      const uint32_t k = e < E ? order_key(row[e]) : 0u;
      const bool pass = e < E && k >= t0;
      const uint32_t b = __ballot_sync(0xFFFFFFFFu, pass);
      const int pos = C + __popc(b & lt_mask);
      if (pass && pos < kCandMaxWide) { rs->ckey[pos] = k; rs->cid[pos] = e; }
      C += __popc(b);
    }
    __syncwarp();
    uint32_t my_key = 0u;
    int my_id = 0;
    if (C <= kCandMaxWide) {
      // 2. rank the candidates; slot < K is the output position
      for (int c = lane; c < C; c += 32) {
        const uint32_t k = rs->ckey[c];
        const int id = rs->cid[c];
        int r = 0;
        for (int d = 0; d < C; ++d) {
          const uint32_t kd = rs->ckey[d];
          r += (kd > k) || (kd == k && rs->cid[d] < id);
        }
        if (r < K) { rs->skey[r] = k; rs->sid[r] = id; }
      }
      __syncwarp();
      if (lane < K) { my_key = rs->skey[lane]; my_id = rs->sid[lane]; }
    } else {
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
      for (int k = 0; k < K; ++k) {
        const uint32_t kmax = __reduce_max_sync(0xFFFFFFFFu, bi == 0x7FFFFFFF ? 0u : bk);
        const int win =
            (int)__reduce_min_sync(0xFFFFFFFFu, (bi != 0x7FFFFFFF && bk == kmax) ? (uint32_t)bi : 0x7FFFFFFFu);
        if (lane == k) { my_key = kmax; my_id = win; }
        if ((win & 31) == lane) {  // the owner marks it and finds its next best
          const int j = win >> 5;
          taken[j >> 5] |= 1u << (j & 31);
          rescan(&bk, &bi);
        }
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

static size_t route_smem_bytes(int E) { return sizeof(float) * kRouteWarps * E + sizeof(RouteScratch) * kRouteWarps; }

cudaError_t route_set_smem_limits() {
  return cudaFuncSetAttribute(route_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)route_smem_bytes(ROUTE_MAX_EXPERTS));
}

// Grid of one wave: CTAs resident at once (the kernel's occupancy, looked up once),
// tokens spread so that every warp takes ceil(T / warps) of them.
template <int P, bool V> static unsigned route_grid(int T, int num_sms) {
  static int occ = 0;  // per instantiation
  if (occ == 0 &&
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, route_reg_kernel<P, V>, kRouteWarps * 32, 0) != cudaSuccess)
    occ = 1;
  const long resident = (long)(occ > 0 ? occ : 1) * num_sms;
  const long per_warp = ((long)T + resident * kRouteWarps - 1) / (resident * kRouteWarps);
  const long blocks = ((long)T + per_warp * kRouteWarps - 1) / (per_warp * kRouteWarps);
  return (unsigned)(blocks > 0 ? blocks : 1);
}

cudaError_t launch_route(const float* logits, int T, int E, int K, int32_t* ids, float* weights, int num_sms,
                         cudaStream_t st) {
  long blocks = ((long)T + kRouteWarps - 1) / kRouteWarps;
  const long cap = (long)num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const dim3 b(kRouteWarps * 32);
  const bool vec = E % 4 == 0 && (reinterpret_cast<uintptr_t>(logits) & 15) == 0;
  if (E <= 1024) {
    // PER: the smallest of 4, 8, 16, 32 with 32 * PER >= E. One wave of resident
    // CTAs, each warp taking the same number of tokens (no partial last wave).
#define MOE_ROUTE_REG(P)                                                                                   \
  (vec ? route_reg_kernel<P, true><<<route_grid<P, true>(T, num_sms), b, 0, st>>>(       \
             logits, T, E, K, ids, weights)                                                                 \
       : route_reg_kernel<P, false><<<route_grid<P, false>(T, num_sms), b, 0, st>>>(     \
             logits, T, E, K, ids, weights))
    if (E <= 128) MOE_ROUTE_REG(4);
    else if (E <= 256) MOE_ROUTE_REG(8);
    else if (E <= 512) MOE_ROUTE_REG(16);
    else MOE_ROUTE_REG(32);
#undef MOE_ROUTE_REG
  } else {
    route_topk_kernel<<<dim3((unsigned)blocks), b, route_smem_bytes(E), st>>>(logits, T, E, K, ids, weights);
  }
  return cudaGetLastError();
}

}  // namespace moe
