// Expert parallelism emulated on one GPU: the dispatch and combine steps around
// the per-rank expert computation ("Add Kimi-K3 A8W4 support to the FlyDSL
// MegaMoE V2 operator": EP8, 112 experts per rank, dispatch of each token to
// the ranks that own its experts, fp8 blockwise 1x32 quantisation of the
// stage-2 result on the combine wire). Rank r owns the global experts
// [r * El, (r + 1) * El). The buffers a real EP exchange would send are
// materialised: each rank's received rows (bf16 x, local expert ids, top-k
// weights) and each rank's combine payload (e4m3 codes + e8m0 scales per 32 of
// H); the per-rank expert computation runs on them with the rank's slice of
// the weights, and the combine sums the dequantised payloads per token.
#include "common.cuh"
#include "kernels.h"

namespace moe {

// One CTA per rank r: the tokens with a pair routed to r, in token order (a
// block-wide scan), and each such token's received row: home token, local
// expert ids (-1 for the pairs of other ranks), top-k weights (0 for those).
// slot[t * R + r] = the token's row on rank r, or -1. CTA 0 flags ids outside
// [0, R * El) (dropped: no rank receives them).
__global__ void __launch_bounds__(1024) ep_route_kernel(const int32_t* __restrict__ ids, const float* __restrict__ w,
                                                        int T, int K, int El, int maxT, int32_t* __restrict__ recv_tok,
                                                        int32_t* __restrict__ recv_ids, float* __restrict__ recv_w,
                                                        int32_t* __restrict__ slot, int32_t* __restrict__ counts,
                                                        int* err) {
  __shared__ int scan_smem[32];
  const int r = blockIdx.x, R = gridDim.x;
  const int lo = r * El, hi = lo + El;
  int base = 0;
  for (int t0 = 0; t0 < T; t0 += blockDim.x) {
    const int t = t0 + threadIdx.x;
    int has = 0, bad = 0;
    if (t < T)
      for (int k = 0; k < K; ++k) {
        const int e = ids[(size_t)t * K + k];
        has |= (e >= lo && e < hi);
        bad |= (e < 0 || e >= El * R);
      }
    if (bad && r == 0) set_error(err, DEV_ERR_BAD_EXPERT);
    int total;
    const int pos = base + block_exclusive_scan(has, scan_smem, &total);
    if (t < T) {
      slot[(size_t)t * R + r] = has ? pos : -1;
      if (has) {
        const size_t row = (size_t)r * maxT + pos;
        recv_tok[row] = t;
        for (int k = 0; k < K; ++k) {
          const int e = ids[(size_t)t * K + k];
          const bool mine = e >= lo && e < hi;
          recv_ids[row * K + k] = mine ? e - lo : -1;
          recv_w[row * K + k] = mine ? w[(size_t)t * K + k] : 0.0f;
        }
      }
    }
    base += total;
  }
  if (threadIdx.x == 0) counts[r] = base;
}

// The dispatch payload: x rows (bf16) into each receiving rank's buffer, one warp per (token, rank).
__global__ void __launch_bounds__(256) ep_copy_kernel(const __nv_bfloat16* __restrict__ x, int T, int H, int R, int maxT,
                                                      const int32_t* __restrict__ slot, __nv_bfloat16* __restrict__ recv_x) {
  const int lane = threadIdx.x & 31;
  const long nw = (long)gridDim.x * (blockDim.x / 32);
  for (long i = (long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); i < (long)T * R; i += nw) {
    const long t = i / R;
    const int r = (int)(i % R);
    const int s = slot[t * R + r];
    if (s < 0) continue;
    const uint4* src = reinterpret_cast<const uint4*>(x + t * H);
    uint4* dst = reinterpret_cast<uint4*>(recv_x + ((size_t)r * maxT + s) * H);
    for (int j = lane; j < H / 8; j += 32) dst[j] = __ldg(src + j);
  }
}

// The combine payload: each rank's fp32 share of each received token, quantised
// to e4m3 with an e8m0 scale per 32 along H (the MX rule of the activations),
// one warp per 32-block.
__global__ void __launch_bounds__(256) ep_wire_kernel(EpShares shares, int H, int R, int maxT,
                                                      const int32_t* __restrict__ counts, uint8_t* __restrict__ codes,
                                                      uint8_t* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int nb = H / 32;
  const long nw = (long)gridDim.x * (blockDim.x / 32);
  for (long i = (long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); i < (long)R * maxT * nb; i += nw) {
    const int r = (int)(i / ((long)maxT * nb));
    const long rem = i % ((long)maxT * nb);
    const int s = (int)(rem / nb), b = (int)(rem % nb);
    if (s >= counts[r]) continue;
    const float v = shares.acc[r][(size_t)s * H + 32 * b + lane];
    uint32_t sc;
    const uint32_t code = block_quant_lane(v, FMT_E4M3, &sc);
    const size_t row = (size_t)r * maxT + s;
    codes[row * H + 32 * b + lane] = (uint8_t)code;
    if (lane == 0) scales[row * nb + b] = (uint8_t)sc;
  }
}

// out[t] = bf16(sum over ranks, in rank order, of the dequantised payload of t).
__global__ void __launch_bounds__(256) ep_combine_kernel(const uint8_t* __restrict__ codes,
                                                         const uint8_t* __restrict__ scales, const int32_t* __restrict__ slot,
                                                         int T, int H, int R, int maxT, __nv_bfloat16* __restrict__ out) {
  const long n8 = (long)T * H / 8;
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (long)gridDim.x * blockDim.x) {
    const long t = i / (H / 8);
    const int h0 = (int)(i % (H / 8)) * 8;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int r = 0; r < R; ++r) {
      const int s = slot[t * R + r];
      if (s < 0) continue;
      const size_t row = (size_t)r * maxT + s;
      const float sc = e8m0_to_f32(scales[row * (H / 32) + h0 / 32]);
      const uint2 q = *reinterpret_cast<const uint2*>(codes + row * H + h0);
      const uint32_t wd[2] = {q.x, q.y};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t h2;
        const uint16_t pair = (uint16_t)(wd[j / 2] >> (16 * (j % 2)));
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));
        acc[2 * j] += __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu))) * sc;
        acc[2 * j + 1] += __half2float(__ushort_as_half((unsigned short)(h2 >> 16))) * sc;
      }
    }
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __nv_bfloat162 v = __floats2bfloat162_rn(acc[2 * j], acc[2 * j + 1]);
      o[j] = *reinterpret_cast<const uint32_t*>(&v);
    }
    *reinterpret_cast<uint4*>(out + t * H + h0) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

static long grid_of(long work, int threads, int num_sms) {
  long b = (work + threads - 1) / threads;
  const long cap = (long)num_sms * 8;
  return b < 1 ? 1 : (b > cap ? cap : b);
}

cudaError_t launch_ep_dispatch(const void* x, const int32_t* ids, const float* w, int T, int H, int K, int El, int R,
                               int maxT, int32_t* recv_tok, int32_t* recv_ids, float* recv_w, int32_t* slot,
                               int32_t* counts, void* recv_x, int* err, int num_sms, cudaStream_t st) {
  ep_route_kernel<<<R, 1024, 0, st>>>(ids, w, T, K, El, maxT, recv_tok, recv_ids, recv_w, slot, counts, err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ep_copy_kernel<<<(unsigned)grid_of((long)T * R * 32, 256, num_sms), 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(x), T, H, R, maxT, slot, static_cast<__nv_bfloat16*>(recv_x));
  return cudaGetLastError();
}

cudaError_t launch_ep_combine(const EpShares& shares, const int32_t* counts, const int32_t* slot, int T, int H, int R,
                              int maxT, uint8_t* codes, uint8_t* scales, void* out, int num_sms, cudaStream_t st) {
  ep_wire_kernel<<<(unsigned)grid_of((long)R * maxT * (H / 32) * 32, 256, num_sms), 256, 0, st>>>(shares, H, R, maxT,
                                                                                                   counts, codes, scales);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ep_combine_kernel<<<(unsigned)grid_of((long)T * H / 8, 256, num_sms), 256, 0, st>>>(
      codes, scales, slot, T, H, R, maxT, static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

}  // namespace moe
