// Grouped stage-1 / stage-2 kernels for few routed rows per expert (decode).
//
// Regime: "Add an opt-in a4w4 SiTUv2 MoE path..." (aiter PR 4463, Performance)
// notes that the small token tiers are weight-bandwidth bound: every active
// expert's MXFP4 weights are streamed once while only a handful of token rows
// use them. Here the weights are the wide M side of an m16n8 MMA and the
// expert's sorted token rows the n = 8 side.
//
// CTA = 4 consumer warps + 1 producer warp. A work unit is (one 8-row block
// of the sort, which belongs to one expert, a 64-row weight tile of that
// expert); the producer reads a unit's routing metadata one unit ahead and
// hands it to the consumers through shared memory. Per unit it copies the
// tile's e8m0 weight scales and the 8 rows' activation scales; per K stage
// (128 codes) it issues one TMA of the 64 x 64-byte weight tile (SWIZZLE_64B)
// and one bulk copy per valid row of that row's 128 activation codes, into a
// padded, bank-conflict-free buffer. Consumers dequantise e2m1 in registers
// (to f16 for the bf16 path, to 2^-6-scaled e4m3 for the fp8/fp4 paths), run
// one MMA group per 32-element K block into a fresh accumulator and add it,
// times the block's scale, into fp32 accumulators.
//
// Stage 1 ("Support SiTUv2 in the packed-int4 MoE stage1 epilogue",
// Motivation; "Add Kimi-K3 A8W4 support...", Technical Details): the tile holds
// gate rows j..j+31 and up rows I+j..I+j+31; warp w owns gate rows 8w..8w+7 as
// MMA rows 0-7 and the same up rows as MMA rows 8-15, so y = act(g, u) is formed
// in the thread holding both, then requantised per 32 along I (bf16 ->
// block-scaled f16, fp8 or fp4) into the sorted intermediate.
// Stage 2 ("Retune Kimi-K3 a16w4 MoE tile geometry", Summary: down GEMM, top-k
// weight, atomic scatter to the token): the tile is 64 rows of H; each valid
// row's result times its top-k weight is added to the fp32 combine buffer.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kTileRows = 64;
constexpr int kRowBytes = 64;                  // 128 e2m1 codes per weight row per stage
constexpr int kStageBytes = kTileRows * kRowBytes;

// B-operand (activation / intermediate) traits per element format.
template <int FMT> struct BFmt;
template <> struct BFmt<FMT_F16> {
  static constexpr int kChunk = 256;   // bytes of 128 elements
  static constexpr int kStride = 320;  // padded row stride in smem: LDS.128 phases conflict-free
  static constexpr int kWords = 4;     // 32-bit words per thread per 32-block
  static constexpr int kBlk = 64;      // bytes per 32-block
  static constexpr int kFix = 0;       // exponent added back after the K loop
};
template <> struct BFmt<FMT_E4M3> {
  static constexpr int kChunk = 128, kStride = 160, kWords = 2, kBlk = 32, kFix = 6;
};
template <> struct BFmt<FMT_E2M1> {
  static constexpr int kChunk = 64, kStride = 144, kWords = 1, kBlk = 16, kFix = 12;
};

template <int FMT> constexpr int num_stages(int stage) {
  return stage == 1 ? (FMT == FMT_F16 ? 5 : 6) : 6;
}

struct Layout {
  uint32_t wbuf, bbuf, sbuf, sbuf_bytes, xsbuf, xs_bytes, ytile, info, bars, total;
};

// kdim: reduction length (H for stage 1, I for stage 2).
template <int FMT, int STAGE>
__host__ __device__ inline Layout make_layout(int kdim) {
  constexpr int NS = num_stages<FMT>(STAGE);
  Layout L;
  L.wbuf = 0;
  L.bbuf = NS * kStageBytes;
  L.sbuf = L.bbuf + NS * DEC_TOK * BFmt<FMT>::kStride;
  L.sbuf_bytes = (uint32_t)(kTileRows * (kdim / 32) + 15) & ~15u;
  L.xsbuf = L.sbuf + 2 * L.sbuf_bytes;
  L.xs_bytes = DEC_TOK * (uint32_t)scale_row_stride(kdim);
  L.ytile = L.xsbuf + 2 * L.xs_bytes;
  L.info = L.ytile + (STAGE == 1 ? DEC_TOK * 32 * 4 : 0);
  L.bars = L.info + 2 * (DEC_TOK + 2) * 4;
  L.total = L.bars + (2 * NS + 4) * 8 + 1024;  // + slack for the 1 KB alignment of the base
  return L;
}

// e8m0 byte kb of a 32-bit word -> 2^(s-127) as fp32. Byte 0 (2^-127) reads
// as 0 and byte 255 (NaN) as infinity; neither occurs in real scales.
__device__ __forceinline__ float e8m0_byte(uint32_t w, int kb) {
  return __uint_as_float(((w >> (8 * kb)) & 0xFFu) << 23);
}

// One 32-block: d = A(16 weight rows x 32 codes) x B(32 x 8 rows), fresh accumulator.
template <int FMT>
__device__ __forceinline__ void block_mma(uint32_t wlo, uint32_t whi, const uint32_t* b, float* d) {
  d[0] = d[1] = d[2] = d[3] = 0.0f;
  if constexpr (FMT == FMT_F16) {
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
    if constexpr (FMT == FMT_E4M3) {
      b0 = __byte_perm(b[0], b[1], 0x6420);
      b1 = __byte_perm(b[0], b[1], 0x7531);
    } else {
      e2m1x8_to_e4m3(b[0], b0, b1);
    }
    mma_e4m3_16832(d, a, b0, b1);
  }
}

template <int FMT>
__device__ __forceinline__ void load_bfrag(const uint8_t* p, uint32_t* b) {
  if constexpr (FMT == FMT_F16) {
    uint4 v = *reinterpret_cast<const uint4*>(p);
    b[0] = v.x; b[1] = v.y; b[2] = v.z; b[3] = v.w;
  } else if constexpr (FMT == FMT_E4M3) {
    uint2 v = *reinterpret_cast<const uint2*>(p);
    b[0] = v.x; b[1] = v.y;
  } else {
    b[0] = *reinterpret_cast<const uint32_t*>(p);
  }
}

}  // namespace

// ---------------------------------------------------------------------------
// The kernel (STAGE 1 or 2)
// ---------------------------------------------------------------------------
template <int FMT, int STAGE>
__global__ void __launch_bounds__(kThreads, 4) decode_stage_kernel(StageParams p, const __grid_constant__ CUtensorMap tmap) {
  constexpr int NS = num_stages<FMT>(STAGE);
  using BF = BFmt<FMT>;
  // bf16 stage-1 activations carry one scale per token (constant along K).
  constexpr bool kRowScale = (STAGE == 1 && FMT == FMT_F16);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int H = p.H, I = p.I, K = p.K;
  const int kdim = STAGE == 1 ? H : I;
  const Layout L = make_layout<FMT, STAGE>(kdim);
  uint8_t* wbuf = smem + L.wbuf;
  uint8_t* bbuf = smem + L.bbuf;
  uint8_t* sbuf = smem + L.sbuf;
  uint8_t* xsbuf = smem + L.xsbuf;
  float* ytile = reinterpret_cast<float*>(smem + L.ytile);
  int* uinfo = reinterpret_cast<int*>(smem + L.info);  // per unit buffer: [expert, tile, 8 pair ids]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + NS;
  uint64_t* ufull = empty + NS;
  uint64_t* uempty = ufull + 2;

  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < NS; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], kConsumerWarps); }
    for (int s = 0; s < 2; ++s) { mbar_init(&ufull[s], 1); mbar_init(&uempty[s], kConsumerWarps); }
    fence_barrier_init();
  }
  __syncthreads();

  const int tiles = STAGE == 1 ? I / 32 : H / kTileRows;   // weight tiles per expert
  const int num_units = p.meta[META_NUM_BLOCKS] * tiles;  // sort blocks are DEC_TOK rows
  const int kstages = kdim / 128;
  const int sb_row = kdim / 32;                               // weight-scale bytes per row
  const int xss = p.xs_stride;                                // activation-scale bytes per row
  const long TK = (long)p.T * K;
  const size_t brow_bytes = (size_t)(kdim / 32) * BF::kBlk;   // one B-operand row

  if (warp == kConsumerWarps) {
    // ------------------------------- producer -------------------------------
    if (lane == 0) tma_prefetch_desc(&tmap);
    uint32_t stage = 0;
    int unit = 0;
    // routing metadata of the next unit, loaded one unit ahead
    int nxt_e = 0, nxt_pid = (int)TK;
    if (blockIdx.x < num_units) {
      const int b = blockIdx.x / tiles;
      nxt_e = p.block_expert[b];
      if (lane < DEC_TOK) nxt_pid = p.sorted_ids[b * DEC_TOK + lane];
    }
    for (int u = blockIdx.x; u < num_units; u += gridDim.x, ++unit) {
      const int b = u / tiles, tile = u % tiles;
      const int e = nxt_e, pid = nxt_pid;
      const int un = u + gridDim.x;
      if (un < num_units) {
        const int bn = un / tiles;
        nxt_e = p.block_expert[bn];
        if (lane < DEC_TOK) nxt_pid = p.sorted_ids[bn * DEC_TOK + lane];
      }
      // source rows of this unit's B operand (stage 1: token rows, stage 2: sorted rows)
      const long src = (lane < DEC_TOK && pid < TK) ? (STAGE == 1 ? (long)(pid / K) : (long)(b * DEC_TOK + lane)) : -1;
      const unsigned valid = __ballot_sync(0xFFFFFFFFu, src >= 0);
      const int nvalid = __popc(valid);
      const int ub = unit & 1;
      if (!mbar_wait_or_abort(&uempty[ub], ((unit >> 1) & 1) ^ 1, p.err, &abort_flag)) return;
      int pids[DEC_TOK];
#pragma unroll
      for (int r = 0; r < DEC_TOK; ++r) pids[r] = __shfl_sync(0xFFFFFFFFu, pid, r);
      if (lane == 0) {
        int* info = uinfo + ub * (DEC_TOK + 2);
        info[0] = e;
        info[1] = tile;
#pragma unroll
        for (int r = 0; r < DEC_TOK; ++r) info[2 + r] = pids[r];
        const uint32_t sbytes = (uint32_t)kTileRows * sb_row;
        mbar_arrive_expect_tx(&ufull[ub], sbytes + (uint32_t)nvalid * xss);  // releases the info writes
        uint8_t* sdst = sbuf + ub * L.sbuf_bytes;
        if (STAGE == 1) {
          const uint8_t* gs = p.wscale + ((size_t)e * 2 * I + (size_t)tile * 32) * sb_row;
          bulk_g2s(sdst, gs, sbytes / 2, &ufull[ub]);
          bulk_g2s(sdst + sbytes / 2, gs + (size_t)I * sb_row, sbytes / 2, &ufull[ub]);
        } else {
          bulk_g2s(sdst, p.wscale + ((size_t)e * H + (size_t)tile * kTileRows) * sb_row, sbytes, &ufull[ub]);
        }
      }
      for (int r = 0; r < DEC_TOK; ++r) {
        const long s = __shfl_sync(0xFFFFFFFFu, src, r);
        if (lane == 0 && s >= 0)
          bulk_g2s(xsbuf + ub * L.xs_bytes + r * xss, p.as + (size_t)s * xss, (uint32_t)xss, &ufull[ub]);
      }
      for (int ks = 0; ks < kstages; ++ks, ++stage) {
        const int slot = stage % NS;
        if (!mbar_wait_or_abort(&empty[slot], ((stage / NS) & 1) ^ 1, p.err, &abort_flag)) return;
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[slot], kStageBytes + (uint32_t)nvalid * BF::kChunk);
          if (STAGE == 1) tma_load_4d(wbuf + slot * kStageBytes, &tmap, ks * kRowBytes, tile * 32, 0, e, &full[slot]);
          else tma_load_3d(wbuf + slot * kStageBytes, &tmap, ks * kRowBytes, tile * kTileRows, e, &full[slot]);
        }
        for (int r = 0; r < DEC_TOK; ++r) {
          const long s = __shfl_sync(0xFFFFFFFFu, src, r);
          if (lane == 0 && s >= 0)
            bulk_g2s(bbuf + (slot * DEC_TOK + r) * BF::kStride, p.aq + (size_t)s * brow_bytes + (size_t)ks * BF::kChunk,
                     BF::kChunk, &full[slot]);
        }
      }
    }
    return;
  }

  // ------------------------------- consumers --------------------------------
  const int g = lane >> 2, c = lane & 3;
  // weight-tile rows of this thread: stage 1 gate/up pair, stage 2 rows r and r+8
  const int r_lo = STAGE == 1 ? 8 * warp + g : 16 * warp + g;
  const int r_hi = STAGE == 1 ? 32 + 8 * warp + g : 16 * warp + g + 8;
  uint32_t off_lo[4], off_hi[4];
#pragma unroll
  for (int kb = 0; kb < 4; ++kb) {
    off_lo[kb] = swz_offset(r_lo, kb, kRowBytes) + 4 * c;
    off_hi[kb] = swz_offset(r_hi, kb, kRowBytes) + 4 * c;
  }
  const uint32_t boff = g * BF::kStride + c * (BF::kBlk / 4);
  uint32_t stage = 0;
  int unit = 0;
  for (int u = blockIdx.x; u < num_units; u += gridDim.x, ++unit) {
    {
      const int b = u / tiles;
      const int row0 = b * DEC_TOK;
      const int ub = unit & 1;
      mbar_wait_or_abort(&ufull[ub], (unit >> 1) & 1, p.err, &abort_flag);
      const int* info = uinfo + ub * (DEC_TOK + 2);
      const int tile = info[1];
      int cpid[2];
      bool cval[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        cpid[q] = info[2 + 2 * c + q];
        cval[q] = cpid[q] < TK;
      }
      int wpid[2];  // pair ids of the two columns this warp stores in the stage-1 epilogue
#pragma unroll
      for (int q = 0; q < 2; ++q) wpid[q] = info[2 + 2 * warp + q];
      const uint8_t* srow_lo = sbuf + ub * L.sbuf_bytes + r_lo * sb_row;
      const uint8_t* srow_hi = sbuf + ub * L.sbuf_bytes + r_hi * sb_row;
      const uint8_t* xrow0 = xsbuf + ub * L.xs_bytes + (2 * c) * xss;
      const uint8_t* xrow1 = xrow0 + xss;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      for (int ks = 0; ks < kstages; ++ks, ++stage) {
        const int slot = stage % NS;
        mbar_wait_or_abort(&full[slot], (stage / NS) & 1, p.err, &abort_flag);
        const uint32_t ws_lo = *reinterpret_cast<const uint32_t*>(srow_lo + ks * 4);
        const uint32_t ws_hi = *reinterpret_cast<const uint32_t*>(srow_hi + ks * 4);
        uint32_t xs0 = 0, xs1 = 0;
        if constexpr (!kRowScale) {
          xs0 = *reinterpret_cast<const uint32_t*>(xrow0 + ks * 4);
          xs1 = *reinterpret_cast<const uint32_t*>(xrow1 + ks * 4);
        }
        const uint8_t* tile_s = wbuf + slot * kStageBytes;
        const uint8_t* btile = bbuf + slot * DEC_TOK * BF::kStride + boff;
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) {
          const uint32_t wlo = *reinterpret_cast<const uint32_t*>(tile_s + off_lo[kb]);
          const uint32_t whi = *reinterpret_cast<const uint32_t*>(tile_s + off_hi[kb]);
          uint32_t b[BF::kWords];
          load_bfrag<FMT>(btile + kb * BF::kBlk, b);
          float d[4];
          block_mma<FMT>(wlo, whi, b, d);
          const float f_lo = e8m0_byte(ws_lo, kb), f_hi = e8m0_byte(ws_hi, kb);
          if constexpr (kRowScale) {
            acc[0] = fmaf(d[0], f_lo, acc[0]);
            acc[1] = fmaf(d[1], f_lo, acc[1]);
            acc[2] = fmaf(d[2], f_hi, acc[2]);
            acc[3] = fmaf(d[3], f_hi, acc[3]);
          } else {
            const float x0 = e8m0_byte(xs0, kb), x1 = e8m0_byte(xs1, kb);
            acc[0] = fmaf(d[0], f_lo * x0, acc[0]);
            acc[1] = fmaf(d[1], f_lo * x1, acc[1]);
            acc[2] = fmaf(d[2], f_hi * x0, acc[2]);
            acc[3] = fmaf(d[3], f_hi * x1, acc[3]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
      }
      // constant factors: the e4m3 re-expression of e2m1 codes, and the per-token scale
      float col_f[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        col_f[q] = __uint_as_float((uint32_t)(127 + BF::kFix) << 23);
        if constexpr (kRowScale) col_f[q] *= e8m0_byte(*(q ? xrow1 : xrow0), 0);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&uempty[ub]);

      if constexpr (STAGE == 1) {
        // y = act(gate, up) for columns 2c, 2c+1 at gate column tile*32 + r_lo
        named_bar_sync(1, kConsumerWarps * 32);
        ytile[(2 * c) * 32 + r_lo] = act_apply(p.act, acc[0] * col_f[0], acc[2] * col_f[0], p.beta, p.lbeta);
        ytile[(2 * c + 1) * 32 + r_lo] = act_apply(p.act, acc[1] * col_f[1], acc[3] * col_f[1], p.beta, p.lbeta);
        named_bar_sync(1, kConsumerWarps * 32);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int n = 2 * warp + q;
          const int row = row0 + n;
          if (wpid[q] >= TK) continue;  // padding row (warp-uniform)
          float v = ytile[n * 32 + lane];
          if (FMT == FMT_F16) v = __bfloat162float(__float2bfloat16_rn(v));  // the a16 intermediate is bf16
          uint32_t s;
          const uint32_t code = block_quant_lane(v, FMT, &s);
          block_store_lane(p.oq + (size_t)row * (I / 32) * BF::kBlk + (size_t)tile * BF::kBlk, code, FMT, lane);
          if (lane == 0) p.os[(size_t)row * p.os_stride + tile] = (uint8_t)s;
        }
      } else {
        // acc32[t, h] += w[p] * z for the valid columns
        const int h_lo = tile * kTileRows + r_lo, h_hi = tile * kTileRows + r_hi;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          if (!cval[q]) continue;
          const float wt = p.topk_w[cpid[q]] * col_f[q];
          float* dst = p.acc32 + (size_t)(cpid[q] / K) * H;
          atomicAdd(dst + h_lo, wt * acc[q]);
          atomicAdd(dst + h_hi, wt * acc[2 + q]);
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------
template <int FMT, int STAGE>
static cudaError_t set_limit() {
  return cudaFuncSetAttribute(decode_stage_kernel<FMT, STAGE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)make_layout<FMT, STAGE>(16384).total);
}

cudaError_t decode_set_smem_limits() {
  cudaError_t e = set_limit<FMT_F16, 1>();
  if (e == cudaSuccess) e = set_limit<FMT_E4M3, 1>();
  if (e == cudaSuccess) e = set_limit<FMT_E2M1, 1>();
  if (e == cudaSuccess) e = set_limit<FMT_F16, 2>();
  if (e == cudaSuccess) e = set_limit<FMT_E4M3, 2>();
  if (e == cudaSuccess) e = set_limit<FMT_E2M1, 2>();
  return e;
}

template <int FMT, int STAGE>
static int occ(int kdim) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_stage_kernel<FMT, STAGE>, kThreads,
                                                    make_layout<FMT, STAGE>(kdim).total) != cudaSuccess)
    return 1;
  return n < 1 ? 1 : n;
}

int decode_s1_blocks_per_sm(int fmt, int H) {
  return fmt == FMT_F16 ? occ<FMT_F16, 1>(H) : (fmt == FMT_E4M3 ? occ<FMT_E4M3, 1>(H) : occ<FMT_E2M1, 1>(H));
}

int decode_s2_blocks_per_sm(int fmt, int I) {
  return fmt == FMT_F16 ? occ<FMT_F16, 2>(I) : (fmt == FMT_E4M3 ? occ<FMT_E4M3, 2>(I) : occ<FMT_E2M1, 2>(I));
}

template <int FMT, int STAGE>
static void launch(const StageParams& p, const CUtensorMap& tm, int grid, cudaStream_t st) {
  const int kdim = STAGE == 1 ? p.H : p.I;
  decode_stage_kernel<FMT, STAGE><<<grid, kThreads, make_layout<FMT, STAGE>(kdim).total, st>>>(p, tm);
}

cudaError_t launch_decode_stage1(int fmt, const StageParams& p, const CUtensorMap& tm, int grid, cudaStream_t st) {
  if (fmt == FMT_F16) launch<FMT_F16, 1>(p, tm, grid, st);
  else if (fmt == FMT_E4M3) launch<FMT_E4M3, 1>(p, tm, grid, st);
  else launch<FMT_E2M1, 1>(p, tm, grid, st);
  return cudaGetLastError();
}

cudaError_t launch_decode_stage2(int fmt, const StageParams& p, const CUtensorMap& tm, int grid, cudaStream_t st) {
  if (fmt == FMT_F16) launch<FMT_F16, 2>(p, tm, grid, st);
  else if (fmt == FMT_E4M3) launch<FMT_E4M3, 2>(p, tm, grid, st);
  else launch<FMT_E2M1, 2>(p, tm, grid, st);
  return cudaGetLastError();
}

}  // namespace moe
