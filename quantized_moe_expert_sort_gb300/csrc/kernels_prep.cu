// Expert sort, activation block quantisation, weight quantisation and the
// bf16 finalize of the combine buffer.
//
// The sort follows "Retune Kimi-K3 a16w4 MoE tile geometry" (aiter PR 5118),
// Summary: moe_sorting buckets the routed (token, k) pairs by expert and pads
// every expert up to a full tile of rows. Within an expert, pairs keep
// ascending pair id p = t*K + k; padding rows hold the sentinel T*K; blocks of
// tile_m rows are listed in ascending expert order. It is integer work and is
// bit-exact by construction: histogram -> scan -> placement whose rank inside
// an expert is computed, not raced for.
#include "common.cuh"
#include "kernels.h"

namespace moe {

// ---------------------------------------------------------------------------
// Sort building blocks
// ---------------------------------------------------------------------------

// Scan of padded per-expert counts: writes expert_count, expert_offset,
// active list, meta, block_expert and the padding sentinels.
// cnt[e] (shared) holds counts on entry; on exit cursor[e] = expert_offset[e].
__device__ void sort_scan_and_fill(const int* cnt, int* cursor, int E, int tile_m, int sentinel,
                                   const SortOut& so, int* scan_smem) {
  int per = (E + blockDim.x - 1) / blockDim.x;
  int e0 = threadIdx.x * per, e1 = min(E, e0 + per);
  int rows = 0, act = 0;
  for (int e = e0; e < e1; ++e) {
    int c = cnt[e];
    rows += (c + tile_m - 1) / tile_m * tile_m;
    act += c > 0;
  }
  int total_rows, total_act;
  int row_base = block_exclusive_scan(rows, scan_smem, &total_rows);
  int act_base = block_exclusive_scan(act, scan_smem, &total_act);
  int off = row_base, ai = act_base;
  for (int e = e0; e < e1; ++e) {
    int c = cnt[e];
    int padded = (c + tile_m - 1) / tile_m * tile_m;
    so.expert_count[e] = c;
    so.expert_offset[e] = off;
    cursor[e] = off;
    if (c > 0) {
      if (so.active_info) so.active_info[ai] = make_int4(e, c, off, 0);
      so.active_experts[ai++] = e;
    }
    off += padded;
  }
  if (threadIdx.x == 0) {
    so.expert_offset[E] = total_rows;
    so.meta[META_NUM_BLOCKS] = total_rows / tile_m;
    so.meta[META_NUM_ACTIVE] = total_act;
    so.meta[META_NUM_ROWS] = total_rows;
  }
  __syncthreads();
  // padding sentinels and per-block expert ids
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int c = cnt[e];
    if (c == 0) continue;
    int o = cursor[e];
    int padded = (c + tile_m - 1) / tile_m * tile_m;
    for (int r = o + c; r < o + padded; ++r) so.sorted_ids[r] = sentinel;
    for (int b = o / tile_m; b < (o + padded) / tile_m; ++b) so.block_expert[b] = e;
  }
}

// The padded per-expert offsets alone (cursor[e] = first row of e), in shared memory.
__device__ void sort_scan_offsets(const int* cnt, int* cursor, int E, int tile_m, int* scan_smem) {
  int per = (E + blockDim.x - 1) / blockDim.x;
  int e0 = threadIdx.x * per, e1 = min(E, e0 + per);
  int rows = 0;
  for (int e = e0; e < e1; ++e) rows += (cnt[e] + tile_m - 1) / tile_m * tile_m;
  int total_rows;
  int off = block_exclusive_scan(rows, scan_smem, &total_rows);
  for (int e = e0; e < e1; ++e) {
    cursor[e] = off;
    off += (cnt[e] + tile_m - 1) / tile_m * tile_m;
  }
}

// Stable placement of pairs [p0, p1) given cursor[e] = first free row of e.
// Chunks of blockDim.x pairs in ascending order; inside a chunk the rank of a
// pair among equal experts is (pairs of earlier warps, from a per-expert byte
// table) + (earlier lanes of its warp, from __match_any_sync).
__device__ void sort_place_range(const int32_t* ids, long p0, long p1, int E, int* cursor,
                                 uint8_t* wtab /* [E][32] */, int32_t* sorted_ids, int32_t* pair_row) {
  int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned lt_mask = (1u << lane) - 1u;
  for (long base = p0; base < p1; base += blockDim.x) {
    long p = base + threadIdx.x;
    int e = -1;
    if (p < p1) {
      int v = ids[p];
      if (v >= 0 && v < E) e = v;
    }
    unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
    int rank = __popc(peers & lt_mask);
    int wcount = __popc(peers);
    bool leader = (peers & lt_mask) == 0;
    if (e >= 0 && leader) wtab[e * 32 + warp] = (uint8_t)wcount;
    __syncthreads();
    if (e >= 0) {
      const uint32_t* row = reinterpret_cast<const uint32_t*>(wtab + e * 32);
      int prefix = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        uint32_t word = row[q];
        int lo = q * 4;  // warps lo..lo+3
        if (lo + 4 <= warp) {
          prefix += __dp4a((int)word, 0x01010101, 0);
        } else if (lo < warp) {
          uint32_t keep = 0xFFFFFFFFu >> (8 * (4 - (warp - lo)));
          prefix += __dp4a((int)(word & keep), 0x01010101, 0);
        }
      }
      const int pos = cursor[e] + prefix + rank;
      if (sorted_ids) sorted_ids[pos] = (int32_t)p;
      if (pair_row) pair_row[p] = pos;
    } else if (pair_row && p < p1) {
      pair_row[p] = -1;
    }
    __syncthreads();
    if (e >= 0 && leader) {
      wtab[e * 32 + warp] = 0;
      atomicAdd(&cursor[e], wcount);
    }
    __syncthreads();
  }
}

// Single-CTA sort for small T*K (decode): histogram, scan, placement in one launch.
__global__ void __launch_bounds__(1024) sort_small_kernel(const int32_t* __restrict__ ids, int n, int E, int tile_m,
                                                          SortOut so, int* err) {
  extern __shared__ __align__(16) uint8_t smem[];
  int* cnt = reinterpret_cast<int*>(smem);                // [E]
  int* cursor = cnt + E;                                  // [E]
  int* scan_smem = cursor + E;                            // [32]
  uint8_t* wtab = reinterpret_cast<uint8_t*>(scan_smem + 32);  // [E][32]
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  for (int i = threadIdx.x; i < E * 8; i += blockDim.x) reinterpret_cast<uint32_t*>(wtab)[i] = 0u;
  __syncthreads();
  bool bad = false;
  for (int p = threadIdx.x; p < n; p += blockDim.x) {
    int e = ids[p];
    if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
    else if (!(so.neg_masked && e < 0)) bad = true;
  }
  if (bad) set_error(err, DEV_ERR_BAD_EXPERT);
  __syncthreads();
  sort_scan_and_fill(cnt, cursor, E, tile_m, n, so, scan_smem);
  __syncthreads();
  sort_place_range(ids, 0, n, E, cursor, wtab, so.sorted_ids, so.pair_row);
}

// Multi-CTA sort, pass 1: per-chunk histograms hist[g][e].
__global__ void __launch_bounds__(1024) sort_hist_kernel(const int32_t* __restrict__ ids, long n, int E, int chunk,
                                                         int* __restrict__ hist, int* err, int neg_masked) {
  extern __shared__ __align__(16) uint8_t smem[];
  int* cnt = reinterpret_cast<int*>(smem);
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  long p0 = (long)blockIdx.x * chunk, p1 = min(n, p0 + chunk);
  bool bad = false;
  for (long p = p0 + threadIdx.x; p < p1; p += blockDim.x) {
    int e = ids[p];
    if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
    else if (!(neg_masked && e < 0)) bad = true;
  }
  if (bad) set_error(err, DEV_ERR_BAD_EXPERT);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(long)blockIdx.x * E + e] = cnt[e];
}

// Multi-CTA sort, pass 2 (one CTA): totals, scan, fill; hist[g][e] becomes the
// first row of chunk g's pairs of expert e.
__global__ void __launch_bounds__(1024) sort_scan_kernel(int* __restrict__ hist, int G, int E, int tile_m, int sentinel,
                                                         SortOut so) {
  pdl_wait();
  pdl_launch_dependents();
  extern __shared__ __align__(16) uint8_t smem[];
  int* cnt = reinterpret_cast<int*>(smem);
  int* cursor = cnt + E;
  int* scan_smem = cursor + E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int s = 0;
    for (int g = 0; g < G; ++g) s += hist[(long)g * E + e];
    cnt[e] = s;
  }
  __syncthreads();
  sort_scan_and_fill(cnt, cursor, E, tile_m, sentinel, so, scan_smem);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = cursor[e];
    for (int g = 0; g < G; ++g) {
      int c = hist[(long)g * E + e];
      hist[(long)g * E + e] = run;
      run += c;
    }
  }
}

// Multi-CTA sort, pass 3: stable placement of each chunk.
__global__ void __launch_bounds__(1024) sort_place_kernel(const int32_t* __restrict__ ids, long n, int E, int chunk,
                                                          const int* __restrict__ hist, int32_t* sorted_ids,
                                                          int32_t* pair_row) {
  pdl_wait();
  pdl_launch_dependents();
  extern __shared__ __align__(16) uint8_t smem[];
  int* cursor = reinterpret_cast<int*>(smem);
  uint8_t* wtab = reinterpret_cast<uint8_t*>(cursor + E);
  for (int e = threadIdx.x; e < E; e += blockDim.x) cursor[e] = hist[(long)blockIdx.x * E + e];
  for (int i = threadIdx.x; i < E * 8; i += blockDim.x) reinterpret_cast<uint32_t*>(wtab)[i] = 0u;
  __syncthreads();
  long p0 = (long)blockIdx.x * chunk, p1 = min(n, p0 + chunk);
  sort_place_range(ids, p0, p1, E, cursor, wtab, sorted_ids, pair_row);
}

// ---------------------------------------------------------------------------
// Activation block quantisation (S2): x bf16 [T,H] -> codes + e8m0 scales per
// 32 along H ("Add an opt-in a4w4 SiTUv2 MoE path...", What: a8w4 = fp8,
// a4w4 = fp4x2 activations; 1x32 scales). One warp per (token, 32-block);
// lane l handles element l. Scale rows are xs_stride bytes apart.
// Also zeroes the fp32 combine buffer acc32 [T,H] for the stage-2 scatter.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) act_quant_kernel(const __nv_bfloat16* __restrict__ x, int T, int H, int fmt,
                                                        uint8_t* __restrict__ xq, uint8_t* __restrict__ xs,
                                                        int xs_stride, float* __restrict__ acc32) {
  int lane = threadIdx.x & 31;
  long nwarps = (long)gridDim.x * (blockDim.x >> 5);
  long gw = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  int nb = H / 32;
  int bpb = fmt_bytes_per_32(fmt);
  for (long blk = gw; blk < (long)T * nb; blk += nwarps) {
    long t = blk / nb;
    int b = (int)(blk % nb);
    float v = __bfloat162float(x[t * H + b * 32 + lane]);
    uint32_t s;
    uint32_t code = block_quant_lane(v, fmt, &s);
    block_store_lane(xq + (t * nb + b) * bpb, code, fmt, lane);
    if (lane == 0) xs[t * xs_stride + b] = (uint8_t)s;
  }
  if (acc32) {
    long n4 = (long)T * H / 4;
    float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (long)gridDim.x * blockDim.x)
      reinterpret_cast<float4*>(acc32)[i] = z;
  }
}

// The bf16 activation operand: each token row re-encoded as IEEE half times
// one power-of-two scale per row, E = floor(log2(row amax)) - 15, so that the
// row maximum lands in [2^15, 2^16). Every bf16 value (8 significant bits) no
// more than 2^31 below its row's maximum is represented exactly. The row scale
// is written into every 32-block scale byte of the row, so the operand reads
// like any other block-scaled one. One CTA per token row (H % 8 == 0), 16-byte
// loads and stores; the remaining CTAs zero the fp32 combine buffer.
__global__ void __launch_bounds__(256) act_encode_f16_kernel(const __nv_bfloat16* __restrict__ x, int T, int H,
                                                             uint8_t* __restrict__ xq, uint8_t* __restrict__ xs,
                                                             int xs_stride, float* __restrict__ acc32) {
  __shared__ float red[8];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (long t = blockIdx.x; t < T; t += gridDim.x) {
    const uint4* row = reinterpret_cast<const uint4*>(x + t * H);
    const int n8 = H / 8;
    float amax = 0.0f;
    for (int i = threadIdx.x; i < n8; i += blockDim.x) {
      uint4 v = row[i];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        amax = fmaxf(amax, fabsf(__uint_as_float(w[q] << 16)));
        amax = fmaxf(amax, fabsf(__uint_as_float(w[q] & 0xFFFF0000u)));
      }
    }
    amax = warp_max(amax);
    if (lane == 0) red[warp] = amax;
    __syncthreads();
    amax = 0.0f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) amax = fmaxf(amax, red[w]);
    __syncthreads();
    int E = 0;
    uint32_t sbyte = 127;
    if (amax > 0.0f) {
      E = floor_log2_f32(amax) - 15;
      E = E < -127 ? -127 : (E > 127 ? 127 : E);
      sbyte = (uint32_t)(E + 127);
    }
    const float m = exp2_neg(E);
    uint4* q = reinterpret_cast<uint4*>(xq + t * (long)H * 2);
    for (int i = threadIdx.x; i < n8; i += blockDim.x) {
      uint4 v = row[i];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float lo = __fmul_rn(__uint_as_float(w[k] << 16), m), hi = __fmul_rn(__uint_as_float(w[k] & 0xFFFF0000u), m);
        o[k] = (uint32_t)__half_as_ushort(__float2half_rn(lo)) | ((uint32_t)__half_as_ushort(__float2half_rn(hi)) << 16);
      }
      q[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    for (int b = threadIdx.x; b < H / 32; b += blockDim.x) xs[t * xs_stride + b] = (uint8_t)sbyte;
  }
  if (acc32) {
    long n4 = (long)T * H / 4;
    float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (long)gridDim.x * blockDim.x)
      reinterpret_cast<float4*>(acc32)[i] = z;
  }
}

// Thread-local 1x32 scale: amax -> (e8m0 byte, multiplier 2^-E) with
// E = floor(log2 amax) - emax clamped to [-127, 127]; amax == 0 -> byte 127, 0.
__device__ __forceinline__ uint32_t block_scale_of(float amax, int emax, float* mul) {
  if (!(amax > 0.0f)) {
    *mul = 0.0f;
    return 127u;
  }
  int E = floor_log2_f32(amax) - emax;
  E = E < -127 ? -127 : (E > 127 ? 127 : E);
  *mul = exp2_neg(E);
  return (uint32_t)(E + 127);
}

// Quantise each 32-block of a token (four threads per block) and write it to the
// sorted rows of the token's K routed pairs (see launch_act_scatter). A16: A16_TERMS e2m1
// terms per value, term t quantising (MX rule) what terms 0..t-1 left over (in
// fp32 the residual v - code * 2^E is exact), term t of sorted row r written as
// sub-row r * A16_TERMS + t. Work units (token, 32-block) are taken 8 per warp
// and pass by warps gw0, gw0 + nw, ...; pair_row may live in shared memory.
template <int MODE, bool CHUNK>
__device__ __forceinline__ void scatter_units(const __nv_bfloat16* __restrict__ x, int T, int H, int K,
                                              const int32_t* pair_row, const ScatterOut& so, long gw0, long nw) {
  // Four threads (a quad of lanes) per (token, 32-block): thread q holds elements
  // 8q..8q+7, the block maximum is reduced across the quad, and the quad's threads
  // take the top-k destinations k = q, q + 4, ... (each writes the whole block).
  constexpr int kTerms = MODE == SW_A16 ? A16_TERMS : 1;
  constexpr int kWords = MODE == SW_A8 ? 2 : 1;  // code words per thread and term (8 e4m3 / 8 e2m1)
  const int nb = H / 32;
  const long total = (long)T * nb;
  const long row_bytes = MODE == SW_A8 ? (long)H : H / 2;  // one (sub-)row
  const int lane = threadIdx.x & 31, q = lane & 3, qbase = lane & ~3;
  // warp-uniform loop: 8 blocks per warp and pass, every lane runs every pass
  for (long w0 = gw0 * 8; w0 < total; w0 += nw * 8) {
    const long w = w0 + (lane >> 2);
    const bool valid = w < total;
    const long t = valid ? w / nb : 0;
    const int b = valid ? (int)(w % nb) : 0;
    float v[8];
    {
      const uint4 qd = valid ? __ldg(reinterpret_cast<const uint4*>(x + t * H + 32 * b) + q) : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t wd[4] = {qd.x, qd.y, qd.z, qd.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[2 * j] = __uint_as_float(wd[j] << 16);
        v[2 * j + 1] = __uint_as_float(wd[j] & 0xFFFF0000u);
      }
    }
    uint32_t c[kTerms][kWords];  // this thread's codes per term
    uint32_t sc[kTerms];         // e8m0 scale byte per term (the same in the quad)
#pragma unroll
    for (int tt = 0; tt < kTerms; ++tt) {
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
      float mul;
      if (MODE == SW_A8) {
        sc[tt] = block_scale_of(amax, 8, &mul);
#pragma unroll
        for (int i = 0; i < 2; ++i)
          c[tt][i] = cvt_e4m3x2(__fmul_rn(v[4 * i], mul), __fmul_rn(v[4 * i + 1], mul)) |
                     (cvt_e4m3x2(__fmul_rn(v[4 * i + 2], mul), __fmul_rn(v[4 * i + 3], mul)) << 16);
      } else {
        sc[tt] = block_scale_of(amax, 2, &mul);
        uint32_t acc = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          acc |= cvt_e2m1x2(__fmul_rn(v[2 * k], mul), __fmul_rn(v[2 * k + 1], mul)) << (8 * k);
        c[tt][0] = acc;
        if (tt + 1 < kTerms) {
          // A16: the next term quantises the exact residual of this one
          const float sv = e8m0_to_f32(sc[tt]);
#pragma unroll
          for (int i = 0; i < 8; ++i) v[i] -= e2m1_to_f32((acc >> (4 * i)) & 0xFu) * sv;
        }
      }
    }
    // Scale bytes of blocks 4i..4i+3 of the warp's token packed into one word (quads
    // 0 and 4 of the warp hold the words): when H / 32 % 8 == 0 a warp's 8 units are
    // blocks 8j..8j+7 of one token, and the 4 bytes are adjacent in both scale layouts.
    const bool pack = nb % 8 == 0;
    uint32_t sw[kTerms];
#pragma unroll
    for (int tt = 0; tt < kTerms; ++tt) {
      const uint32_t s1 = __shfl_down_sync(0xFFFFFFFFu, sc[tt], 4);
      const uint32_t s2 = __shfl_down_sync(0xFFFFFFFFu, sc[tt], 8);
      const uint32_t s3 = __shfl_down_sync(0xFFFFFFFFu, sc[tt], 12);
      sw[tt] = sc[tt] | (s1 << 8) | (s2 << 16) | (s3 << 24);
    }
    const bool sw_lane = ((lane >> 2) & 3) == 0;  // quads 0 and 4: blocks b .. b + 3, b % 4 == 0
    // the whole block's codes in every thread of the quad
    uint32_t full[kTerms][4 * kWords];
#pragma unroll
    for (int tt = 0; tt < kTerms; ++tt)
#pragma unroll
      for (int s = 0; s < 4; ++s)
#pragma unroll
        for (int i = 0; i < kWords; ++i) full[tt][kWords * s + i] = __shfl_sync(0xFFFFFFFFu, c[tt][i], qbase + s);
    if (!valid) continue;
    for (int k = q; k < K; k += 4) {
      const int r = pair_row[t * K + k];
      if (r < 0) continue;
      if (so.row_tok && b == 0) {
        so.row_tok[r] = (int32_t)t;
        so.row_w[r] = __ldg(so.topk_w + t * K + k);
      }
      uint8_t* dst = so.codes + (size_t)r * kTerms * row_bytes;
      if (MODE == SW_A8) {
        uint4* d0 = reinterpret_cast<uint4*>(dst + 32 * b);
        d0[0] = make_uint4(full[0][0], full[0][1], full[0][2], full[0][3]);
        d0[1] = make_uint4(full[0][4], full[0][5], full[0][6], full[0][7]);
      } else {
#pragma unroll
        for (int tt = 0; tt < kTerms; ++tt)
          *reinterpret_cast<uint4*>(dst + (size_t)tt * row_bytes + 16 * b) =
              make_uint4(full[tt][0], full[tt][1], full[tt][2], full[tt][3]);
      }
      if (CHUNK) {  // tcgen05.cp chunks of 128-row tiles (many-rows path)
        const int m = r & 127;
        const size_t o = ((size_t)(r >> 7) * (nb / 4) + (b >> 2)) * 512 + 16 * (m & 31) + 4 * (m >> 5);
        if (!pack) so.scales[o + (b & 3)] = (uint8_t)sc[0];
        else if (sw_lane) *reinterpret_cast<uint32_t*>(so.scales + o) = sw[0];
      } else {
#pragma unroll
        for (int tt = 0; tt < kTerms; ++tt) {
          const size_t o = ((size_t)r * kTerms + tt) * so.sstride + b;
          if (!pack) so.scales[o] = (uint8_t)sc[tt];
          else if (sw_lane) *reinterpret_cast<uint32_t*>(so.scales + o) = sw[tt];
        }
      }
    }
  }
}

// Zero the fp32 combine buffer.
__device__ __forceinline__ void scatter_tail(int T, int H, const ScatterOut& so, long tid0, long nthreads) {
  if (so.acc32) {
    const long n4 = (long)T * H / 4;
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    for (long i = tid0; i < n4; i += nthreads) reinterpret_cast<float4*>(so.acc32)[i] = z;
  }
}

template <int MODE, bool CHUNK>
__global__ void __launch_bounds__(128) act_scatter_kernel(const __nv_bfloat16* __restrict__ x, int T, int H, int K,
                                                          const int32_t* __restrict__ pair_row, ScatterOut so) {
  pdl_wait();  // the sort's pair rows
  pdl_launch_dependents();
  scatter_units<MODE, CHUNK>(x, T, H, K, pair_row, so, (long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5),
                             (long)gridDim.x * (blockDim.x / 32));
  scatter_tail(T, H, so, (long)blockIdx.x * blockDim.x + threadIdx.x, (long)gridDim.x * blockDim.x);
}

// L2 prefetch of a contiguous range (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// The sort and the activation scatter in one launch, for up to
// SORT_SMALL_MAX_PAIRS pairs ("Add an opt-in a4w4 SiTUv2 MoE path...", Three
// tuner defects item 2: a separate quant kernel costs a launch at small token
// counts). Every CTA sorts all pairs in shared memory (the same histogram, scan
// and stable placement as sort_small_kernel: identical results in every CTA),
// CTA 0 publishes the sort, and each CTA then quantises its share of the
// (token, 32-block) units straight into the sorted rows, reading each pair's
// row from its own shared-memory copy. Each CTA first pulls its share of x into
// L2, so that load overlaps the sort.
template <int MODE, bool CHUNK>
__global__ void __launch_bounds__(1024) sort_scatter_kernel(const int32_t* __restrict__ ids, int n, int E, int tile_m,
                                                            SortOut so, int* err, const __nv_bfloat16* __restrict__ x,
                                                            int T, int H, int K, ScatterOut sc) {
  extern __shared__ __align__(16) uint8_t smem[];
  int* cnt = reinterpret_cast<int*>(smem);                     // [E]
  int* cursor = cnt + E;                                       // [E]
  int* scan_smem = cursor + E;                                 // [32]
  int32_t* prow = scan_smem + 32;                              // [n]
  uint8_t* wtab = reinterpret_cast<uint8_t*>(prow + ((n + 3) & ~3));  // [E][32]
  const bool lead = blockIdx.x == 0;
  {  // this CTA's share of x, into L2 ahead of the scatter (4 KB pieces)
    const long xb = (long)T * H * 2;
    for (long o = ((long)blockIdx.x * blockDim.x + threadIdx.x) * 4096; o < xb;
         o += (long)gridDim.x * blockDim.x * 4096)
      prefetch_l2(reinterpret_cast<const uint8_t*>(x) + o, (uint32_t)min(4096L, xb - o));
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  if (n >= E) {
    for (int i = threadIdx.x; i < E * 8; i += blockDim.x) reinterpret_cast<uint32_t*>(wtab)[i] = 0u;
  } else {  // few pairs: clear only the table rows of experts that occur
    for (int p = threadIdx.x; p < n; p += blockDim.x) {
      const int e = ids[p];
      if (e >= 0 && e < E) {
        uint4* row = reinterpret_cast<uint4*>(wtab + e * 32);
        row[0] = make_uint4(0u, 0u, 0u, 0u);
        row[1] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }
  __syncthreads();
  bool bad = false;
  for (int p = threadIdx.x; p < n; p += blockDim.x) {
    int e = ids[p];
    if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
    else if (!(so.neg_masked && e < 0)) bad = true;
  }
  if (bad && lead) set_error(err, DEV_ERR_BAD_EXPERT);
  __syncthreads();
  // only CTA 0 writes the sort's global outputs; the others keep offsets in shared memory
  if (lead) {
    sort_scan_and_fill(cnt, cursor, E, tile_m, n, so, scan_smem);
  } else {
    sort_scan_offsets(cnt, cursor, E, tile_m, scan_smem);
  }
  __syncthreads();
  sort_place_range(ids, 0, n, E, cursor, wtab, lead ? so.sorted_ids : nullptr, prow);
  __syncthreads();
  if (lead && so.pair_row)
    for (int p = threadIdx.x; p < n; p += blockDim.x) so.pair_row[p] = prow[p];
  // the dependent kernel may launch now; it waits for this grid's completion
  pdl_launch_dependents();
  scatter_units<MODE, CHUNK>(x, T, H, K, prow, sc, (long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5),
                             (long)gridDim.x * (blockDim.x / 32));
  scatter_tail(T, H, sc, (long)blockIdx.x * blockDim.x + threadIdx.x, (long)gridDim.x * blockDim.x);
}

// MXFP4 weight quantisation: fp32 [rows, cols] -> e2m1 codes [rows, cols/2] +
// e8m0 scales [rows, cols/32], the same 1x32 rule as the activations.
__global__ void __launch_bounds__(256) weight_quant_kernel(const float* __restrict__ w, long nblocks,
                                                           uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  int lane = threadIdx.x & 31;
  long nwarps = (long)gridDim.x * (blockDim.x >> 5);
  for (long blk = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); blk < nblocks; blk += nwarps) {
    float v = w[blk * 32 + lane];
    uint32_t s;
    uint32_t code = block_quant_lane(v, FMT_E2M1, &s);
    block_store_lane(codes + blk * 16, code, FMT_E2M1, lane);
    if (lane == 0) scales[blk] = (uint8_t)s;
  }
}

// out = bf16_RNE(acc32), 4 elements per thread.
__global__ void __launch_bounds__(256) finalize_kernel(const float* __restrict__ acc32, long n4, __nv_bfloat16* __restrict__ out) {
  pdl_wait();  // the combine buffer is complete
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (long)gridDim.x * blockDim.x) {
    float4 v = reinterpret_cast<const float4*>(acc32)[i];
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
    uint2 o;
    o.x = *reinterpret_cast<uint32_t*>(&a);
    o.y = *reinterpret_cast<uint32_t*>(&b);
    reinterpret_cast<uint2*>(out)[i] = o;
  }
}

// Self-test of the bounded wait every pipeline uses: one warp waits on an
// mbarrier that is completed first (complete != 0) or never, with a wall-clock
// limit; a wait that runs out sets DEV_ERR_TIMEOUT and the kernel returns.
__global__ void __launch_bounds__(32) wait_selftest_kernel(uint64_t limit_ns, int complete, int* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0 && complete) mbar_arrive(&bar);
  __syncwarp();
  if (threadIdx.x == 0) mbar_wait_limit(&bar, 0, err, limit_ns);
}

// ---------------------------------------------------------------------------
// Host-side launchers
// ---------------------------------------------------------------------------
cudaError_t launch_wait_selftest(uint64_t limit_ns, int complete, int* err, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(limit_ns, complete, err);
  return cudaGetLastError();
}

size_t sort_small_smem(int E) { return (size_t)E * 8 + 32 * 4 + (size_t)E * 32; }

cudaError_t launch_sort(const int32_t* ids, long n, int E, int tile_m, const SortOut& so, int* hist, int hist_cap_chunks,
                        int* err, cudaStream_t st) {
  if (n <= SORT_SMALL_MAX_PAIRS) {
    sort_small_kernel<<<1, 1024, sort_small_smem(E), st>>>(ids, (int)n, E, tile_m, so, err);
    return cudaGetLastError();
  }
  int chunk = SORT_CHUNK;
  int G = (int)((n + chunk - 1) / chunk);
  if (G > hist_cap_chunks) return cudaErrorInvalidValue;
  sort_hist_kernel<<<G, 1024, (size_t)E * 4, st>>>(ids, n, E, chunk, hist, err, so.neg_masked);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess)
    e = launch_k(sort_scan_kernel, dim3(1), dim3(1024), (size_t)E * 8 + 32 * 4, st, true, hist, G, E, tile_m, (int)n, so);
  if (e == cudaSuccess)
    e = launch_k(sort_place_kernel, dim3(G), dim3(1024), (size_t)E * 4 + (size_t)E * 32, st, true, ids, n, E, chunk,
                 (const int*)hist, so.sorted_ids, so.pair_row);
  return e;
}

template <int M, bool C>
static cudaError_t set_sort_scatter_limit() {
  return cudaFuncSetAttribute(sort_scatter_kernel<M, C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)sort_scatter_smem(SORT_MAX_EXPERTS, SORT_SMALL_MAX_PAIRS));
}

cudaError_t prep_set_smem_limits() {
  cudaError_t e = cudaFuncSetAttribute(sort_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)sort_small_smem(SORT_MAX_EXPERTS));
  if (e != cudaSuccess) return e;
  if ((e = set_sort_scatter_limit<SW_A16, false>()) != cudaSuccess) return e;
  if ((e = set_sort_scatter_limit<SW_A8, false>()) != cudaSuccess) return e;
  if ((e = set_sort_scatter_limit<SW_A8, true>()) != cudaSuccess) return e;
  if ((e = set_sort_scatter_limit<SW_A4, false>()) != cudaSuccess) return e;
  if ((e = set_sort_scatter_limit<SW_A4, true>()) != cudaSuccess) return e;
  e = cudaFuncSetAttribute(sort_place_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)((size_t)SORT_MAX_EXPERTS * 36));
  return e;
}

cudaError_t launch_act_quant(const void* x, int T, int H, int fmt, uint8_t* xq, uint8_t* xs, int xs_stride,
                             float* acc32, int num_sms, cudaStream_t st) {
  const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(x);
  long cap = (long)num_sms * 8;
  if (fmt == FMT_F16) {
    long blocks = (long)T;
    long zb = ((long)T * H / 4 + 255) / 256;
    if (acc32 && zb > blocks) blocks = zb;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    act_encode_f16_kernel<<<(int)blocks, 256, 0, st>>>(xb, T, H, xq, xs, xs_stride, acc32);
    return cudaGetLastError();
  }
  long work = (long)T * (H / 32);
  long blocks = (work + 7) / 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  act_quant_kernel<<<(int)blocks, 256, 0, st>>>(xb, T, H, fmt, xq, xs, xs_stride, acc32);
  return cudaGetLastError();
}

static long scatter_blocks(int T, int H, int threads, int num_sms) {
  const long work = (long)T * (H / 32);  // 32-blocks, four threads each
  long blocks = (work * 4 + threads - 1) / threads;
  const long floor_blocks = ((long)T * H / 4 + threads - 1) / threads;  // enough threads to zero acc32 quickly
  if (blocks < floor_blocks / 4) blocks = floor_blocks / 4;
  const long cap = (long)num_sms * (threads == 128 ? 16 : 1);
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return blocks;
}

cudaError_t launch_act_scatter(const void* x, int T, int H, int K, int mode, const int32_t* pair_row,
                               const ScatterOut& so, int num_sms, cudaStream_t st) {
  const long blocks = scatter_blocks(T, H, 128, num_sms);
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  const bool chunk = so.sstride == 0;
#define MOE_SCATTER(M, C) \
  launch_k(act_scatter_kernel<M, C>, dim3((unsigned)blocks), dim3(128), 0, st, true, xb, T, H, K, pair_row, so)
  cudaError_t e;
  if (mode == SW_A16) e = MOE_SCATTER(SW_A16, false);
  else if (mode == SW_A8 && chunk) e = MOE_SCATTER(SW_A8, true);
  else if (mode == SW_A8) e = MOE_SCATTER(SW_A8, false);
  else if (chunk) e = MOE_SCATTER(SW_A4, true);
  else e = MOE_SCATTER(SW_A4, false);
#undef MOE_SCATTER
  return e;
}

size_t sort_scatter_smem(int E, long n) {
  return (size_t)E * 8 + 32 * 4 + (size_t)((n + 3) & ~3L) * 4 + (size_t)E * 32;
}

cudaError_t launch_sort_scatter(const int32_t* ids, long n, int E, int tile_m, const SortOut& so, int* err,
                                const void* x, int T, int H, int K, int mode, const ScatterOut& sc, int num_sms,
                                cudaStream_t st) {
  if (n > SORT_SMALL_MAX_PAIRS) return cudaErrorInvalidValue;
  // every CTA repeats the sort, so the scatter is spread only as far as its work
  // needs: about 64 (token, 32-block) units per CTA, up to one CTA per SM
  long blocks = ((long)T * (H / 32) + 63) / 64;
  if (blocks > num_sms) blocks = num_sms;
  if (blocks < 1) blocks = 1;
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  const bool chunk = sc.sstride == 0;
  const size_t smem = sort_scatter_smem(E, n);
#define MOE_SORT_SCATTER(M, C)                                                                                \
  launch_k(sort_scatter_kernel<M, C>, dim3((unsigned)blocks), dim3(1024), smem, st, true, ids, (int)n, E, tile_m, \
           so, err, xb, T, H, K, sc)
  cudaError_t e;
  if (mode == SW_A16) e = MOE_SORT_SCATTER(SW_A16, false);
  else if (mode == SW_A8 && chunk) e = MOE_SORT_SCATTER(SW_A8, true);
  else if (mode == SW_A8) e = MOE_SORT_SCATTER(SW_A8, false);
  else if (chunk) e = MOE_SORT_SCATTER(SW_A4, true);
  else e = MOE_SORT_SCATTER(SW_A4, false);
#undef MOE_SORT_SCATTER
  return e;
}

cudaError_t launch_weight_quant(const float* w, long nblocks, uint8_t* codes, uint8_t* scales, int num_sms,
                                cudaStream_t st) {
  long blocks = (nblocks + 7) / 8;
  long cap = (long)num_sms * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  weight_quant_kernel<<<(int)blocks, 256, 0, st>>>(w, nblocks, codes, scales);
  return cudaGetLastError();
}

cudaError_t launch_finalize(const float* acc32, long n, void* out, int num_sms, cudaStream_t st) {
  long n4 = n / 4;
  long blocks = (n4 + 255) / 256;
  long cap = (long)num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_k(finalize_kernel, dim3((unsigned)blocks), dim3(256), 0, st, true, acc32, n4,
                  reinterpret_cast<__nv_bfloat16*>(out));
}

}  // namespace moe
