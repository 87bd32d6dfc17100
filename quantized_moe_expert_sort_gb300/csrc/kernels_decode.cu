// Grouped stage-1 / stage-2 kernels for few routed rows per expert (decode).
//
// Work: "Add an opt-in a4w4 SiTUv2 MoE path..." (aiter PR 4463, Performance)
// notes the small token tiers are weight-bandwidth bound: every active expert's
// MXFP4 weights are streamed once while only a handful of token rows use them.
// These kernels are built for that regime: weights are the wide M side of an
// m16n8 MMA, the expert's sorted token rows the n=8 side.
//
// Per CTA: one producer warp streams weight tiles (64 rows x 128 K-codes,
// 4 KB, SWIZZLE_64B) through a TMA + mbarrier ring; four consumer warps each
// own 16 weight rows, dequantise e2m1 in registers (to f16 for the bf16
// activation path, to 2^-6-scaled e4m3 for the fp8 / fp4 paths) and issue one
// MMA group per 32-element K block with a fresh accumulator, which is then
// scaled by the weight and activation e8m0 scales in fp32.
//
// Stage 1 ("Support SiTUv2 in the packed-int4 MoE stage1 epilogue", Motivation;
// "Add Kimi-K3 A8W4 support...", Technical Details): a CTA item is
// (expert, 32 gate columns j..j+31 and the matching up columns I+j..). Each
// consumer warp holds gate rows in MMA rows 0-7 and the same up rows in 8-15,
// so y = act(g, u) is formed in the thread that holds both, then requantised
// per 32 along I (bf16 -> block-scaled f16, fp8 or fp4) into the intermediate.
// Stage 2 ("Retune Kimi-K3 a16w4 MoE tile geometry", Summary / relevant files:
// down GEMM with top-k weight and an atomic scatter to the token): a CTA item
// is (expert, 64 rows of H); each valid row's result times its top-k weight is
// added into the fp32 combine buffer.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kTileRows = 64;
constexpr int kRowBytes = 64;  // 128 e2m1 codes per row per stage
constexpr int kStageBytes = kTileRows * kRowBytes;

// Exponent added back in the per-block scale: e2m1 -> e4m3 weights hold
// 2^-6 times their value, and so do e2m1 activations converted the same way,
// so the block result is multiplied by 2^+6 (fp8 activations) or 2^+12 (fp4).
template <int FMT> constexpr int scale_exp_fix() { return FMT == FMT_F16 ? 0 : (FMT == FMT_E4M3 ? 6 : 12); }

// Bytes of one 32-element block of activation codes, and of this thread's 8.
template <int FMT> constexpr int blk_bytes() { return FMT == FMT_F16 ? 64 : (FMT == FMT_E4M3 ? 32 : 16); }
template <int FMT> constexpr int frag_words() { return FMT == FMT_F16 ? 4 : (FMT == FMT_E4M3 ? 2 : 1); }

struct SmemLayout {
  uint32_t wbuf, sbuf, sbuf_bytes, ytile, bars, total;
};

__host__ __device__ inline SmemLayout smem_layout(int kdim, bool with_ytile) {
  SmemLayout L;
  L.wbuf = 0;
  L.sbuf = DEC_STAGES * kStageBytes;
  L.sbuf_bytes = (uint32_t)(kTileRows * (kdim / 32) + 15) & ~15u;
  L.ytile = L.sbuf + 2 * L.sbuf_bytes;
  L.bars = L.ytile + (with_ytile ? DEC_TOK * 32 * 4 : 0);
  L.total = L.bars + (2 * DEC_STAGES + 4) * 8 + 1024;  // + slack for 1 KB alignment
  return L;
}

// 2^e as fp32 for an exponent that may leave the normal range.
__device__ __forceinline__ float pow2f(int e) {
  if (e >= -126 && e <= 127) return __uint_as_float((uint32_t)(e + 127) << 23);
  if (e > 127) return __uint_as_float(0x7F800000u);
  if (e < -149) return 0.0f;
  return __uint_as_float(1u << (e + 149));
}

template <int FMT>
__device__ __forceinline__ void load_frag(const uint8_t* rowp, int k, uint32_t* f) {
  // rowp: start of a code row; k: first element (multiple of 8) of this thread's 8.
  if (FMT == FMT_F16) {
    uint4 v = __ldg(reinterpret_cast<const uint4*>(rowp + (size_t)k * 2));
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
  } else if (FMT == FMT_E4M3) {
    uint2 v = __ldg(reinterpret_cast<const uint2*>(rowp + k));
    f[0] = v.x; f[1] = v.y;
  } else {
    f[0] = __ldg(reinterpret_cast<const uint32_t*>(rowp + k / 2));
  }
}

// One 32-block: d = A(16 weight rows, 32 codes) x B(32, 8 tokens), fresh accumulator.
template <int FMT>
__device__ __forceinline__ void block_mma(uint32_t wlo, uint32_t whi, const uint32_t* b, float* d) {
  d[0] = d[1] = d[2] = d[3] = 0.0f;
  if (FMT == FMT_F16) {
    uint32_t ag[4], au[4];
    e2m1x8_to_f16x8(wlo, ag);
    e2m1x8_to_f16x8(whi, au);
    uint32_t a0[4] = {ag[0], au[0], ag[1], au[1]};
    mma_f16_16816(d, a0, b[0], b[1]);
    uint32_t a1[4] = {ag[2], au[2], ag[3], au[3]};
    mma_f16_16816(d, a1, b[2], b[3]);
  } else {
    uint32_t ge, go, ue, uo;
    e2m1x8_to_e4m3(wlo, ge, go);
    e2m1x8_to_e4m3(whi, ue, uo);
    uint32_t a[4] = {ge, ue, go, uo};
    uint32_t b0, b1;
    if (FMT == FMT_E4M3) {
      b0 = __byte_perm(b[0], b[1], 0x6420);
      b1 = __byte_perm(b[0], b[1], 0x7531);
    } else {
      e2m1x8_to_e4m3(b[0], b0, b1);
    }
    mma_e4m3_16832(d, a, b0, b1);
  }
}

}  // namespace

// ---------------------------------------------------------------------------
// Stage 1
// ---------------------------------------------------------------------------
template <int FMT>
__global__ void __launch_bounds__(kThreads) decode_stage1_kernel(StageParams p, const __grid_constant__ CUtensorMap tm_w13) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int H = p.H, I = p.I, K = p.K;
  const SmemLayout L = smem_layout(H, true);
  uint8_t* wbuf = smem + L.wbuf;
  uint8_t* sbuf = smem + L.sbuf;
  float* ytile = reinterpret_cast<float*>(smem + L.ytile);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + DEC_STAGES;
  uint64_t* sfull = empty + DEC_STAGES;
  uint64_t* sempty = sfull + 2;

  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < DEC_STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], kConsumerWarps); }
    for (int s = 0; s < 2; ++s) { mbar_init(&sfull[s], 1); mbar_init(&sempty[s], kConsumerWarps); }
    fence_barrier_init();
  }
  __syncthreads();

  const int n_jt = I / 32;
  const int num_items = p.meta[META_NUM_ACTIVE] * n_jt;
  const int kstages = H / 128;
  const int sb_row = H / 32;  // scale bytes per weight row

  if (warp == kConsumerWarps) {
    // ---------------- producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tm_w13);
      uint32_t stage = 0;
      int li = 0;
      for (int item = blockIdx.x; item < num_items; item += gridDim.x, ++li) {
        const int e = p.active_experts[item / n_jt], jt = item % n_jt;
        const int passes = (p.expert_count[e] + DEC_TOK - 1) / DEC_TOK;
        const int sb = li & 1;
        if (!mbar_wait_or_abort(&sempty[sb], ((li >> 1) & 1) ^ 1, p.err, &abort_flag)) return;
        mbar_arrive_expect_tx(&sfull[sb], 2u * 32u * (uint32_t)sb_row);
        const uint8_t* gs = p.wscale + ((size_t)e * 2 * I + (size_t)jt * 32) * sb_row;
        bulk_g2s(sbuf + sb * L.sbuf_bytes, gs, 32u * sb_row, &sfull[sb]);
        bulk_g2s(sbuf + sb * L.sbuf_bytes + 32 * sb_row, gs + (size_t)I * sb_row, 32u * sb_row, &sfull[sb]);
        for (int pass = 0; pass < passes; ++pass) {
          for (int ks = 0; ks < kstages; ++ks, ++stage) {
            const int slot = stage % DEC_STAGES;
            if (!mbar_wait_or_abort(&empty[slot], ((stage / DEC_STAGES) & 1) ^ 1, p.err, &abort_flag)) return;
            mbar_arrive_expect_tx(&full[slot], kStageBytes);
            tma_load_4d(wbuf + slot * kStageBytes, &tm_w13, ks * kRowBytes, jt * 32, 0, e, &full[slot]);
          }
        }
      }
    }
    return;
  }

  // ---------------- consumers ----------------
  const int g = lane >> 2, c = lane & 3;
  const int rg = 8 * warp + g, ru = 32 + 8 * warp + g;  // gate / up rows of this thread in the tile
  const long TK = (long)p.T * K;
  uint32_t stage = 0;
  int li = 0;
  for (int item = blockIdx.x; item < num_items; item += gridDim.x, ++li) {
    const int e = p.active_experts[item / n_jt], jt = item % n_jt;
    const int m = p.expert_count[e];
    const int passes = (m + DEC_TOK - 1) / DEC_TOK;
    const int sb = li & 1;
    mbar_wait_or_abort(&sfull[sb], (li >> 1) & 1, p.err, &abort_flag);
    const uint8_t* srow_g = sbuf + sb * L.sbuf_bytes + rg * sb_row;
    const uint8_t* srow_u = sbuf + sb * L.sbuf_bytes + ru * sb_row;
    for (int pass = 0; pass < passes; ++pass) {
      const int row0 = p.expert_offset[e] + pass * DEC_TOK;
      // B-operand row: token of group row g
      const uint8_t* brow = nullptr;
      {
        int pid = p.sorted_ids[row0 + g];
        if (pid < TK) brow = p.aq + (size_t)(pid / K) * H * blk_bytes<FMT>() / 32;
      }
      int ctok[2], cval[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        int pid = p.sorted_ids[row0 + 2 * c + q];
        cval[q] = pid < TK;
        ctok[q] = cval[q] ? pid / K : 0;
      }
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      for (int ks = 0; ks < kstages; ++ks, ++stage) {
        // activation fragments and scales of the 4 blocks of this stage
        uint32_t bf[4][frag_words<FMT>()];
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) {
          if (brow) load_frag<FMT>(brow, ks * 128 + kb * 32 + 8 * c, bf[kb]);
          else {
#pragma unroll
            for (int q = 0; q < frag_words<FMT>(); ++q) bf[kb][q] = 0u;
          }
        }
        uint32_t xs4[2];
#pragma unroll
        for (int q = 0; q < 2; ++q)
          xs4[q] = cval[q] ? __ldg(reinterpret_cast<const uint32_t*>(p.as + (size_t)ctok[q] * (H / 32) + ks * 4)) : 0u;
        const uint32_t wsg4 = *reinterpret_cast<const uint32_t*>(srow_g + ks * 4);
        const uint32_t wsu4 = *reinterpret_cast<const uint32_t*>(srow_u + ks * 4);

        const int slot = stage % DEC_STAGES;
        mbar_wait_or_abort(&full[slot], (stage / DEC_STAGES) & 1, p.err, &abort_flag);
        const uint8_t* tile = wbuf + slot * kStageBytes;
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) {
          uint32_t wlo = *reinterpret_cast<const uint32_t*>(tile + swz_offset(rg, kb, kRowBytes) + 4 * c);
          uint32_t whi = *reinterpret_cast<const uint32_t*>(tile + swz_offset(ru, kb, kRowBytes) + 4 * c);
          float d[4];
          block_mma<FMT>(wlo, whi, bf[kb], d);
          int eg = (int)((wsg4 >> (8 * kb)) & 0xFF) - 127 + scale_exp_fix<FMT>();
          int eu = (int)((wsu4 >> (8 * kb)) & 0xFF) - 127 + scale_exp_fix<FMT>();
          int x0 = (int)((xs4[0] >> (8 * kb)) & 0xFF) - 127;
          int x1 = (int)((xs4[1] >> (8 * kb)) & 0xFF) - 127;
          acc[0] = fmaf(d[0], pow2f(eg + x0), acc[0]);
          acc[1] = fmaf(d[1], pow2f(eg + x1), acc[1]);
          acc[2] = fmaf(d[2], pow2f(eu + x0), acc[2]);
          acc[3] = fmaf(d[3], pow2f(eu + x1), acc[3]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
      }
      // epilogue: y = act(gate, up) for columns 2c, 2c+1 at gate column jt*32 + rg
      named_bar_sync(1, kConsumerWarps * 32);
      ytile[(2 * c) * 32 + rg] = act_apply(p.act, acc[0], acc[2], p.beta, p.lbeta);
      ytile[(2 * c + 1) * 32 + rg] = act_apply(p.act, acc[1], acc[3], p.beta, p.lbeta);
      named_bar_sync(1, kConsumerWarps * 32);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int n = 2 * warp + q;
        const int row = row0 + n;
        if (p.sorted_ids[row] >= TK) continue;  // padding row: nothing to store (warp-uniform)
        float v = ytile[n * 32 + lane];
        if (FMT == FMT_F16) v = __bfloat162float(__float2bfloat16_rn(v));  // the a16 intermediate is bf16
        uint32_t s;
        uint32_t code = block_quant_lane(v, FMT, &s);
        block_store_lane(p.oq + (size_t)row * (I / 32) * blk_bytes<FMT>() + (size_t)jt * blk_bytes<FMT>(), code, FMT, lane);
        if (lane == 0) p.os[(size_t)row * (I / 32) + jt] = (uint8_t)s;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sempty[sb]);
  }
}

// ---------------------------------------------------------------------------
// Stage 2
// ---------------------------------------------------------------------------
template <int FMT>
__global__ void __launch_bounds__(kThreads) decode_stage2_kernel(StageParams p, const __grid_constant__ CUtensorMap tm_w2) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int H = p.H, I = p.I, K = p.K;
  const SmemLayout L = smem_layout(I, false);
  uint8_t* wbuf = smem + L.wbuf;
  uint8_t* sbuf = smem + L.sbuf;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + DEC_STAGES;
  uint64_t* sfull = empty + DEC_STAGES;
  uint64_t* sempty = sfull + 2;

  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < DEC_STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], kConsumerWarps); }
    for (int s = 0; s < 2; ++s) { mbar_init(&sfull[s], 1); mbar_init(&sempty[s], kConsumerWarps); }
    fence_barrier_init();
  }
  __syncthreads();

  const int n_ht = H / kTileRows;
  const int num_items = p.meta[META_NUM_ACTIVE] * n_ht;
  const int kstages = I / 128;
  const int sb_row = I / 32;

  if (warp == kConsumerWarps) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_w2);
      uint32_t stage = 0;
      int li = 0;
      for (int item = blockIdx.x; item < num_items; item += gridDim.x, ++li) {
        const int e = p.active_experts[item / n_ht], ht = item % n_ht;
        const int passes = (p.expert_count[e] + DEC_TOK - 1) / DEC_TOK;
        const int sb = li & 1;
        if (!mbar_wait_or_abort(&sempty[sb], ((li >> 1) & 1) ^ 1, p.err, &abort_flag)) return;
        mbar_arrive_expect_tx(&sfull[sb], (uint32_t)kTileRows * sb_row);
        bulk_g2s(sbuf + sb * L.sbuf_bytes, p.wscale + ((size_t)e * H + (size_t)ht * kTileRows) * sb_row,
                 (uint32_t)kTileRows * sb_row, &sfull[sb]);
        for (int pass = 0; pass < passes; ++pass) {
          for (int ks = 0; ks < kstages; ++ks, ++stage) {
            const int slot = stage % DEC_STAGES;
            if (!mbar_wait_or_abort(&empty[slot], ((stage / DEC_STAGES) & 1) ^ 1, p.err, &abort_flag)) return;
            mbar_arrive_expect_tx(&full[slot], kStageBytes);
            tma_load_3d(wbuf + slot * kStageBytes, &tm_w2, ks * kRowBytes, ht * kTileRows, e, &full[slot]);
          }
        }
      }
    }
    return;
  }

  const int g = lane >> 2, c = lane & 3;
  const int r0 = 16 * warp + g, r1 = r0 + 8;
  const long TK = (long)p.T * K;
  const size_t arow_bytes = (size_t)(I / 32) * blk_bytes<FMT>();
  uint32_t stage = 0;
  int li = 0;
  for (int item = blockIdx.x; item < num_items; item += gridDim.x, ++li) {
    const int e = p.active_experts[item / n_ht], ht = item % n_ht;
    const int m = p.expert_count[e];
    const int passes = (m + DEC_TOK - 1) / DEC_TOK;
    const int sb = li & 1;
    mbar_wait_or_abort(&sfull[sb], (li >> 1) & 1, p.err, &abort_flag);
    const uint8_t* srow0 = sbuf + sb * L.sbuf_bytes + r0 * sb_row;
    const uint8_t* srow1 = sbuf + sb * L.sbuf_bytes + r1 * sb_row;
    for (int pass = 0; pass < passes; ++pass) {
      const int row0 = p.expert_offset[e] + pass * DEC_TOK;
      const uint8_t* brow = (p.sorted_ids[row0 + g] < TK) ? p.aq + (size_t)(row0 + g) * arow_bytes : nullptr;
      int cval[2], crow[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        crow[q] = row0 + 2 * c + q;
        cval[q] = p.sorted_ids[crow[q]] < TK;
      }
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      for (int ks = 0; ks < kstages; ++ks, ++stage) {
        uint32_t bf[4][frag_words<FMT>()];
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) {
          if (brow) load_frag<FMT>(brow, ks * 128 + kb * 32 + 8 * c, bf[kb]);
          else {
#pragma unroll
            for (int q = 0; q < frag_words<FMT>(); ++q) bf[kb][q] = 0u;
          }
        }
        uint32_t xs4[2];
#pragma unroll
        for (int q = 0; q < 2; ++q)
          xs4[q] = cval[q] ? __ldg(reinterpret_cast<const uint32_t*>(p.as + (size_t)crow[q] * (I / 32) + ks * 4)) : 0u;
        const uint32_t ws04 = *reinterpret_cast<const uint32_t*>(srow0 + ks * 4);
        const uint32_t ws14 = *reinterpret_cast<const uint32_t*>(srow1 + ks * 4);
        const int slot = stage % DEC_STAGES;
        mbar_wait_or_abort(&full[slot], (stage / DEC_STAGES) & 1, p.err, &abort_flag);
        const uint8_t* tile = wbuf + slot * kStageBytes;
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) {
          uint32_t wlo = *reinterpret_cast<const uint32_t*>(tile + swz_offset(r0, kb, kRowBytes) + 4 * c);
          uint32_t whi = *reinterpret_cast<const uint32_t*>(tile + swz_offset(r1, kb, kRowBytes) + 4 * c);
          float d[4];
          block_mma<FMT>(wlo, whi, bf[kb], d);
          int e0 = (int)((ws04 >> (8 * kb)) & 0xFF) - 127 + scale_exp_fix<FMT>();
          int e1 = (int)((ws14 >> (8 * kb)) & 0xFF) - 127 + scale_exp_fix<FMT>();
          int x0 = (int)((xs4[0] >> (8 * kb)) & 0xFF) - 127;
          int x1 = (int)((xs4[1] >> (8 * kb)) & 0xFF) - 127;
          acc[0] = fmaf(d[0], pow2f(e0 + x0), acc[0]);
          acc[1] = fmaf(d[1], pow2f(e0 + x1), acc[1]);
          acc[2] = fmaf(d[2], pow2f(e1 + x0), acc[2]);
          acc[3] = fmaf(d[3], pow2f(e1 + x1), acc[3]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
      }
      // epilogue: acc32[t, h] += w[p] * z for the valid columns
      const int h0 = ht * kTileRows + r0, h1 = ht * kTileRows + r1;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        if (!cval[q]) continue;
        const int pid = p.sorted_ids[crow[q]];
        const float wt = p.topk_w[pid];
        float* dst = p.acc32 + (size_t)(pid / K) * H;
        atomicAdd(dst + h0, wt * acc[q]);
        atomicAdd(dst + h1, wt * acc[2 + q]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sempty[sb]);
  }
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------
template <int FMT>
static cudaError_t set_limits_fmt() {
  cudaError_t e = cudaFuncSetAttribute(decode_stage1_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem_layout(16384, true).total);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(decode_stage2_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)smem_layout(16384, false).total);
}

cudaError_t decode_set_smem_limits() {
  cudaError_t e = set_limits_fmt<FMT_F16>();
  if (e == cudaSuccess) e = set_limits_fmt<FMT_E4M3>();
  if (e == cudaSuccess) e = set_limits_fmt<FMT_E2M1>();
  return e;
}

template <typename Kern>
static int occupancy(Kern k, size_t smem) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, kThreads, smem) != cudaSuccess) return 1;
  return n < 1 ? 1 : n;
}

int decode_s1_blocks_per_sm(int fmt, int H) {
  size_t s = smem_layout(H, true).total;
  if (fmt == FMT_F16) return occupancy(decode_stage1_kernel<FMT_F16>, s);
  if (fmt == FMT_E4M3) return occupancy(decode_stage1_kernel<FMT_E4M3>, s);
  return occupancy(decode_stage1_kernel<FMT_E2M1>, s);
}

int decode_s2_blocks_per_sm(int fmt, int I) {
  size_t s = smem_layout(I, false).total;
  if (fmt == FMT_F16) return occupancy(decode_stage2_kernel<FMT_F16>, s);
  if (fmt == FMT_E4M3) return occupancy(decode_stage2_kernel<FMT_E4M3>, s);
  return occupancy(decode_stage2_kernel<FMT_E2M1>, s);
}

cudaError_t launch_decode_stage1(int fmt, const StageParams& p, const CUtensorMap& tm, int grid, cudaStream_t st) {
  size_t s = smem_layout(p.H, true).total;
  if (fmt == FMT_F16) decode_stage1_kernel<FMT_F16><<<grid, kThreads, s, st>>>(p, tm);
  else if (fmt == FMT_E4M3) decode_stage1_kernel<FMT_E4M3><<<grid, kThreads, s, st>>>(p, tm);
  else decode_stage1_kernel<FMT_E2M1><<<grid, kThreads, s, st>>>(p, tm);
  return cudaGetLastError();
}

cudaError_t launch_decode_stage2(int fmt, const StageParams& p, const CUtensorMap& tm, int grid, cudaStream_t st) {
  size_t s = smem_layout(p.I, false).total;
  if (fmt == FMT_F16) decode_stage2_kernel<FMT_F16><<<grid, kThreads, s, st>>>(p, tm);
  else if (fmt == FMT_E4M3) decode_stage2_kernel<FMT_E4M3><<<grid, kThreads, s, st>>>(p, tm);
  else decode_stage2_kernel<FMT_E2M1><<<grid, kThreads, s, st>>>(p, tm);
  return cudaGetLastError();
}

}  // namespace moe
