// Grouped stage-1 / stage-2 kernels on the 5th-generation tensor cores
// (tcgen05 block-scaled MMA, TMEM accumulators, TMA operand staging) for many
// routed rows per expert (prefill).
//
// What they compute is the same as the decode kernels ("Add Kimi-K3 A8W4
// support..." Technical Details; "Add an opt-in a4w4 SiTUv2 MoE path...",
// What / Performance: at large token counts the activation traffic and the MMA
// rate matter). Kinds:
//   a8w4: tcgen05.mma kind::mxf8f6f4, A = e4m3 activations, B = e2m1 weights
//         (expanded by TMA to one 16-element group per 16 bytes), 1x32 e8m0
//         scales (scale_vec::1X), K = 32 per MMA, K tile 128.
//   a4w4: kind::mxf4, A and B packed e2m1, scale_vec::2X, K = 64 per MMA, K tile 256.
//
// Tile: M = 128 sorted rows (one sort block of one expert) x N = 128 weight
// rows. Stage 1: N = 64 gate rows + the same 64 up rows, so each epilogue
// thread (one token row) holds g and u for 64 columns j, forms y = act(g, u)
// and requantises y per 32 along I by itself. Stage 2: N = 128 rows of H; each
// thread adds w * z for its row into the fp32 combine buffer (vector red).
//
// Tile order: stage 1 runs block-major (the N tiles of one 128-row block back to
// back, so the block's activations are re-read from L2). Stage 2 adds into the
// fp32 combine buffer; when that buffer is larger than L2 the N tiles are taken
// in groups of p.tile_group (block-major inside a group), so the CTAs in flight
// add into a slice of T x 128 x tile_group fp32 that stays in L2 instead of
// into random rows of the whole buffer.
//
// CTA (one per SM, persistent over tiles): warp 0 issues all loads with TMA /
// bulk copies -- the 128 sorted rows (stage 1 reads activations the quantiser
// wrote in sorted order, stage 2 the intermediate), the weight tile, the rows'
// e8m0 scales (already in tcgen05.cp chunks in global memory) per stage, and the
// tile's weight scales (row-major) once per tile into a staging buffer; warp 1
// transposes the stage's weight scales from staging into the tcgen05.cp chunk
// layout (smem to smem, fence.proxy.async, mbarrier arrive); warp 2 owns TMEM
// and issues tcgen05.cp + tcgen05.mma; warps 4-7 run the epilogue from
// double-buffered accumulators.
// Scale layout in TMEM (M = 128): row m reads lane m, column base + m/32,
// byte = the MMA's scale id; in shared memory byte 16*(m%32) + 4*(m/32) + kb
// of a 512-byte chunk holds the scale of row m for K block kb (4 blocks).
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace moe {
namespace {

constexpr int kThreadsTc = 384;        // warps 0-3 producer / scales / MMA / idle, 4-11 epilogue
constexpr int kEpiWarps = 8;
constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kNS = 4;          // pipeline stages
constexpr int kTileBytes = 128 * 128;  // one 128-row x 128-byte operand tile

template <int KIND> struct Kind;
template <> struct Kind<TC_A8W4> {
  static constexpr int kKTile = 128;   // elements per stage
  static constexpr int kBlocks = 4;    // 32-element scale blocks per stage
  static constexpr int kChunks = 1;    // 512-byte scale chunks per stage and operand
  static constexpr int kFmt = FMT_E4M3;
};
template <> struct Kind<TC_A4W4> {
  static constexpr int kKTile = 256, kBlocks = 8, kChunks = 2, kFmt = FMT_E2M1;
};

// Transaction bytes a weight tile reports to its mbarrier: TMA counts the packed
// global bytes, also for the 16U4_ALIGN16B type that expands each 8-byte group
// of 16 fp4 codes into 16 bytes of shared memory (the 8-byte gaps are left as
// they are, so the B tiles are zeroed once at kernel start).
template <int KIND> constexpr uint32_t weight_tile_tx() { return KIND == TC_A8W4 ? kTileBytes / 2 : kTileBytes; }

// (block, N tile) of a linear tile index: N tiles in groups of G (the last group
// may be smaller), block-major inside a group. G >= ntn is plain block-major.
__device__ __forceinline__ void tile_coords(int tile, int nb, int ntn, int G, int* b, int* nt) {
  const int gsz = nb * G;
  const int g = tile / gsz;
  const int r = tile - g * gsz;
  const int gg = min(G, ntn - g * G);
  *b = r / gg;
  *nt = g * G + r % gg;
}

struct TcLayout {
  static constexpr uint32_t a = 0;                                  // kNS x 16 KB
  static constexpr uint32_t b = a + kNS * kTileBytes;               // kNS x 16 KB
  static constexpr uint32_t sfa = b + kNS * kTileBytes;             // kNS x 2 chunks
  static constexpr uint32_t sfb = sfa + kNS * 1024;
  static constexpr uint32_t ws = sfb + kNS * 1024;                 // 2 x weight-scale staging
  static constexpr uint32_t ws_bytes = 128 * 128;                  // 128 rows x up to 128 scale bytes (K <= 4096)
  static constexpr uint32_t epi = ws + 2 * ws_bytes;               // stage-2 transpose: per epilogue warp 32 x 36 fp32
  static constexpr uint32_t epi_bytes = 32 * 36 * 4;
  static constexpr uint32_t bars = epi + kEpiWarps * epi_bytes;
  static constexpr uint32_t tmem_slot = bars + (2 * kNS + 8) * 8;
  static constexpr uint32_t total = tmem_slot + 16 + 1024;        // + alignment slack
};

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfCol0 = 2 * kBN;  // scale slots after the two accumulators

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* m, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}


__device__ __forceinline__ void red_add_v4(float* dst, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

// Byte offset of (row m, block kb % 4) inside a 512-byte scale chunk.
__device__ __forceinline__ uint32_t sf_off(int m) { return 16u * (m & 31) + 4u * (m >> 5); }

}  // namespace

// ---------------------------------------------------------------------------
template <int KIND, int STAGE>
__global__ void __launch_bounds__(kThreadsTc, 1) tc_stage_kernel(TcParams p, const __grid_constant__ CUtensorMap tm_a,
                                                                 const __grid_constant__ CUtensorMap tm_b) {
  using KD = Kind<KIND>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + TcLayout::bars);  // a stage's copies and scales are ready
  uint64_t* empty = full + kNS;
  uint64_t* tfull = empty + kNS;
  uint64_t* tempty = tfull + 2;
  uint64_t* wsfull = tempty + 2;   // weight scales of a tile landed in staging
  uint64_t* wsempty = wsfull + 2;  // staging buffer free again
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + TcLayout::tmem_slot);
  __shared__ int abort_flag;
  __shared__ __align__(8) uint64_t drain;  // completion of every tcgen05 op of the MMA thread

  if (dynamic_smem_bytes() < TcLayout::total) {  // launched with less shared memory than the layout needs
    if (threadIdx.x == 0) set_error(p.err, DEV_ERR_LAUNCH);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = p.H, I = p.I, K = p.K, T = p.T;
  const long TK = (long)T * K;
  const int kdim = STAGE == 1 ? H : I;
  const int ktiles = (kdim + KD::kKTile - 1) / KD::kKTile;
  const int nblk_k = kdim / 32;                       // valid 32-blocks along K
  const int ntn = STAGE == 1 ? I / 64 : H / kBN;      // N tiles per expert
  const int G = STAGE == 1 || p.tile_group <= 0 ? ntn : p.tile_group;  // N tiles per group (tile order)

  if (threadIdx.x == 0) {
    abort_flag = 0;
    // full: the TMA issuer's expect_tx arrive (and the copies' bytes) + the 32 scale-transpose lanes
    for (int s = 0; s < kNS; ++s) { mbar_init(&full[s], 1 + 32); mbar_init(&empty[s], 1); }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&tfull[s], 1);
      mbar_init(&tempty[s], kEpiWarps);
      mbar_init(&wsfull[s], 1);
      mbar_init(&wsempty[s], 32);
    }
    mbar_init(&drain, 1);
    fence_barrier_init();
  }
  if (KIND == TC_A8W4) {
    // zero the weight tiles: the unpacking TMA never writes their 8-byte gaps
    for (uint32_t i = threadIdx.x; i < kNS * kTileBytes / 16; i += blockDim.x)
      reinterpret_cast<uint4*>(smem + TcLayout::b)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async();
  }
  if (warp == 2) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tbase = *tmem_slot;
  // everything above overlapped the previous kernel's tail; its results are read from here on
  pdl_wait();
  pdl_launch_dependents();
  const int nb = p.meta[META_NUM_BLOCKS];
  const int num_tiles = nb * ntn;

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0) {
      tma_prefetch_desc(&tm_a);
      tma_prefetch_desc(&tm_b);
      const int sb_row = kdim / 32;  // weight-scale bytes per row
      uint32_t stage = 0;
      int lt = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x, ++lt) {
        int b, nt;
        tile_coords(tile, nb, ntn, G, &b, &nt);
        const int e = p.block_expert[b];
        // the tile's weight scales, row-major, into the staging buffer of this tile parity
        const int tp = lt & 1;
        if (!mbar_wait_or_abort(&wsempty[tp], ((lt >> 1) & 1) ^ 1, p.err, &abort_flag)) break;
        uint8_t* wst = smem + TcLayout::ws + tp * TcLayout::ws_bytes;
        mbar_arrive_expect_tx(&wsfull[tp], 128u * sb_row);
        if (STAGE == 1) {
          const uint8_t* g = p.wscale + ((size_t)e * 2 * I + (size_t)nt * 64) * sb_row;
          bulk_g2s(wst, g, 64u * sb_row, &wsfull[tp]);
          bulk_g2s(wst + 64 * sb_row, g + (size_t)I * sb_row, 64u * sb_row, &wsfull[tp]);
        } else {
          bulk_g2s(wst, p.wscale + ((size_t)e * H + (size_t)nt * kBN) * sb_row, 128u * sb_row, &wsfull[tp]);
        }
        for (int ks = 0; ks < ktiles; ++ks, ++stage) {
          const int slot = stage % kNS;
          if (!mbar_wait_or_abort(&empty[slot], ((stage / kNS) & 1) ^ 1, p.err, &abort_flag)) { ok = false; break; }
          uint8_t* sa = smem + TcLayout::a + slot * kTileBytes;
          uint8_t* sb = smem + TcLayout::b + slot * kTileBytes;
          int nchunk = 0;  // row-scale chunks of this stage inside K (the rest are filled by the scale warp)
          for (int c = 0; c < KD::kChunks; ++c) nchunk += (ks * KD::kBlocks + 4 * c) < nblk_k;
          mbar_arrive_expect_tx(&full[slot], kTileBytes + weight_tile_tx<KIND>() + 512u * nchunk);
          // A: 128 sorted rows (stage 1: activations written in sorted order; stage 2: the intermediate)
          tma_load_2d(sa, &tm_a, ks * 128, b * kBM, &full[slot]);
          if (STAGE == 1) {
            tma_load_4d(sb, &tm_b, ks * 128, nt * 64, 0, e, &full[slot]);
            tma_load_4d(sb + 64 * 128, &tm_b, ks * 128, nt * 64, 1, e, &full[slot]);
          } else {
            tma_load_3d(sb, &tm_b, ks * 128, nt * kBN, e, &full[slot]);
          }
          // row scales: stored in tcgen05.cp chunks per 128-row tile already
          for (int c = 0; c < nchunk; ++c)
            bulk_g2s(smem + TcLayout::sfa + slot * 1024 + 512 * c,
                     p.as + ((size_t)b * (nblk_k / 4) + (ks * KD::kBlocks) / 4 + c) * 512, 512u, &full[slot]);
        }
      }
      // Before the CTA may exit, every copy this thread started must have landed
      // (after an abort the consumers no longer wait for them): the last kNS
      // operand stages and the last two scale stagings. In a normal run these
      // phases completed long ago and the waits return at once; after an abort the
      // bounded wait outlasts any copy in flight.
      for (uint32_t g = stage > (uint32_t)kNS ? stage - kNS : 0u; g < stage; ++g)
        mbar_wait(&full[g % kNS], (g / kNS) & 1, p.err);
      for (int l = lt > 2 ? lt - 2 : 0; l < lt; ++l) mbar_wait(&wsfull[l & 1], (l >> 1) & 1, p.err);
    }
  } else if (warp == 1) {
    // ---------------- weight scales: staging (row-major) -> tcgen05.cp chunks ----------------
    const int sb_row = kdim / 32;
    uint32_t stage = 0;
    int lt = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x, ++lt) {
      const int tp = lt & 1;
      if (!mbar_wait_or_abort(&wsfull[tp], (lt >> 1) & 1, p.err, &abort_flag)) break;
      const uint8_t* wst = smem + TcLayout::ws + tp * TcLayout::ws_bytes;
      for (int ks = 0; ks < ktiles; ++ks, ++stage) {
        const int slot = stage % kNS;
        if (!mbar_wait_or_abort(&empty[slot], ((stage / kNS) & 1) ^ 1, p.err, &abort_flag)) { ok = false; break; }
        uint8_t* dA = smem + TcLayout::sfa + slot * 1024;
        uint8_t* dB = smem + TcLayout::sfb + slot * 1024;
        for (int c = 0; c < KD::kChunks; ++c) {
          const int kb0 = ks * KD::kBlocks + 4 * c;  // first 32-block of this chunk
          const bool in = kb0 < nblk_k;              // kdim % 128 == 0: a chunk is all in or all out
          if (!in)  // past the end of K: neutral scales (the operands there are zero)
            *reinterpret_cast<uint4*>(dA + 512 * c + 16 * lane) =
                make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int m = 4 * lane + i;
            *reinterpret_cast<uint32_t*>(dB + 512 * c + sf_off(m)) =
                in ? *reinterpret_cast<const uint32_t*>(wst + m * sb_row + kb0) : 0x7F7F7F7Fu;
          }
        }
        fence_proxy_async();  // generic smem writes -> visible to tcgen05.cp
        mbar_arrive(&full[slot]);
      }
      __syncwarp();
      if (!ok) break;
      mbar_arrive(&wsempty[tp]);
    }
  } else if (warp == 2) {
    // ------------------------------ MMA issuer ------------------------------
    // Descriptors are formed once and advanced by 16-byte-unit offsets (the
    // issuing thread's instruction stream is on the critical path).
    if (lane == 0) {
      const uint64_t dA0 = tc::sdesc(smem_u32(smem + TcLayout::a), 16, 1024, tc::SW_128B);
      const uint64_t dB0 = tc::sdesc(smem_u32(smem + TcLayout::b), 16, 1024, tc::SW_128B);
      const uint64_t dSA = tc::sdesc(smem_u32(smem + TcLayout::sfa), 0, 128, tc::SW_NONE);
      const uint64_t dSB = tc::sdesc(smem_u32(smem + TcLayout::sfb), 0, 128, tc::SW_NONE);
      constexpr uint32_t id0 = KIND == TC_A8W4 ? tc::idesc_bs(kBM, kBN, tc::F8F6F4_E4M3, tc::F8F6F4_E2M1, 0, 0)
                                               : tc::idesc_bs(kBM, kBN, tc::MXF4_E2M1, tc::MXF4_E2M1, 0, 0);
      uint32_t stage = 0;
      int lt = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x, ++lt) {
        const int buf = lt & 1;
        if (!mbar_wait_or_abort(&tempty[buf], ((lt >> 1) & 1) ^ 1, p.err, &abort_flag)) break;
        tc::fence_after();
        const uint32_t d = tbase + buf * kBN;
        for (int ks = 0; ks < ktiles; ++ks, ++stage) {
          const int slot = stage % kNS;
          // an aborted wait leaves the stage unread: no MMA runs on operands that never landed
          if (!mbar_wait_or_abort(&full[slot], (stage / kNS) & 1, p.err, &abort_flag)) {
            ok = false;
            break;
          }
          tc::fence_after();
          const uint32_t sfa = tbase + kSfCol0 + slot * 16;
          const uint32_t sfb = sfa + 8;
#pragma unroll
          for (int c = 0; c < KD::kChunks; ++c) {
            tc::cp_32x128b_warpx4(sfa + 4 * c, dSA + ((slot * 1024 + 512 * c) >> 4));
            tc::cp_32x128b_warpx4(sfb + 4 * c, dSB + ((slot * 1024 + 512 * c) >> 4));
          }
          const uint64_t da = dA0 + ((slot * kTileBytes) >> 4);
          const uint64_t db = dB0 + ((slot * kTileBytes) >> 4);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t acc = (ks > 0 || i > 0) ? 1u : 0u;
            if (KIND == TC_A8W4) {
              tc::mma_mxf8f6f4(d, da + 2 * i, db + 2 * i, id0 | ((uint32_t)i << 4) | ((uint32_t)i << 29), sfa, sfb, acc);
            } else {
              const uint32_t id = id0 | ((2u * (i & 1)) << 4) | ((2u * (i & 1)) << 29);
              tc::mma_mxf4(d, da + 2 * i, db + 2 * i, id, sfa + 4 * (i >> 1), sfb + 4 * (i >> 1), acc);
            }
          }
          tc::commit(&empty[slot]);
        }
        if (!ok) break;  // a partial accumulator is never handed to the epilogue
        tc::commit(&tfull[buf]);
      }
      // every MMA / copy this thread issued has finished before TMEM is released
      tc::commit(&drain);
      mbar_wait(&drain, 0, p.err);
    }
  } else if (warp >= 4) {
    // ------------------------------ epilogue ------------------------------
    const int q = warp & 3;                // TMEM lane quadrant this warp may access
    const int grp = (warp - 4) >> 2;       // column group: 0 -> warps 4-7, 1 -> warps 8-11
    const int m = 32 * q + lane;           // tile row of this thread (= TMEM lane)
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    const ActK ak = act_consts(p.beta, p.lbeta);
    int lt = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++lt) {
      int b, nt;
      tile_coords(tile, nb, ntn, G, &b, &nt);
      const int buf = lt & 1;
      const int row = b * kBM + m;
      const int pid = p.sorted_ids[row];
      const bool valid = pid < TK;
      // a timed-out wait means the accumulator never completed: no store or reduction
      bool ready = true;
      if (lane == 0) ready = mbar_wait_or_abort(&tfull[buf], (lt >> 1) & 1, p.err, &abort_flag);
      ready = __shfl_sync(0xFFFFFFFFu, ready ? 1 : 0, 0) != 0;
      __syncwarp();  // tcgen05.ld is .sync.aligned: the whole warp, converged
      if (!ready) break;
      tc::fence_after();
      const uint32_t d = tbase + lane_off + buf * kBN;
      if (STAGE == 1) {
        {
          const int h = grp;  // the group's 32 intermediate columns
          uint32_t gr[32], ur[32];
          tc::ld_32x32b_x16(d + 32 * h, gr);
          tc::ld_32x32b_x16(d + 32 * h + 16, gr + 16);
          tc::ld_32x32b_x16(d + 64 + 32 * h, ur);
          tc::ld_32x32b_x16(d + 64 + 32 * h + 16, ur + 16);
          tc::ld_wait();
          // the accumulator goes back to the MMA warp before this tile's global stores
          tc::fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty[buf]);
          float y[32];
          float amax = 0.0f;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            y[i] = act_apply<false>(p.act, __uint_as_float(gr[i]), __uint_as_float(ur[i]), p.beta, p.lbeta, ak);
            amax = fmaxf(amax, fabsf(y[i]));
          }
          if (valid) {
            // 1x32 block quantisation of y along I (same rule as the activations)
            const int fmt = KD::kFmt;
            uint32_t sbyte = 127;
            float mul = 1.0f;
            if (amax > 0.0f) {
              int E = floor_log2_f32(amax) - fmt_emax(fmt);
              E = E < -127 ? -127 : (E > 127 ? 127 : E);
              sbyte = (uint32_t)(E + 127);
              mul = exp2_neg(E);
            }
            const int j0 = nt * 64 + 32 * h;  // first intermediate column of this block
            if (fmt == FMT_E4M3) {
              uint32_t w[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const uint32_t lo = amax > 0.0f ? cvt_e4m3x2(__fmul_rn(y[4 * i], mul), __fmul_rn(y[4 * i + 1], mul)) : 0u;
                const uint32_t hi = amax > 0.0f ? cvt_e4m3x2(__fmul_rn(y[4 * i + 2], mul), __fmul_rn(y[4 * i + 3], mul)) : 0u;
                w[i] = lo | (hi << 16);
              }
              uint4* dst = reinterpret_cast<uint4*>(p.oq + (size_t)row * I + j0);
              dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
              dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
            } else {
              uint32_t w[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                uint32_t acc = 0;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const uint32_t byte =
                      amax > 0.0f ? cvt_e2m1x2(__fmul_rn(y[8 * i + 2 * k], mul), __fmul_rn(y[8 * i + 2 * k + 1], mul)) : 0u;
                  acc |= byte << (8 * k);
                }
                w[i] = acc;
              }
              *reinterpret_cast<uint4*>(p.oq + (size_t)row * (I / 2) + j0 / 2) = make_uint4(w[0], w[1], w[2], w[3]);
            }
            // scale byte in the stage-2 chunk layout
            const int kb = j0 / 32;
            p.os[((size_t)b * (I / 128) + kb / 4) * 512 + sf_off(m) + (kb & 3)] = (uint8_t)sbyte;
          }
        }
      } else {
        // Each thread holds row m (one routed pair) x 32 columns of H. The warp
        // transposes them through shared memory so that one vector red covers
        // 4 rows x 128 contiguous bytes instead of 32 rows x 16 bytes.
        const int t = valid ? pid / K : 0;
        const float wt = valid ? p.topk_w[pid] : 0.0f;
        float* tb = reinterpret_cast<float*>(smem + TcLayout::epi + (warp - 4) * TcLayout::epi_bytes);
        const unsigned vmask = __ballot_sync(0xFFFFFFFFu, valid);
        uint32_t rr2[2][32];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          tc::ld_32x32b_x16(d + 32 * (2 * grp + cc), rr2[cc]);
          tc::ld_32x32b_x16(d + 32 * (2 * grp + cc) + 16, rr2[cc] + 16);
        }
        tc::ld_wait();
        // the accumulator goes back to the MMA warp before this tile's reductions
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int c = 2 * grp + cc;
          const uint32_t* r = rr2[cc];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            *reinterpret_cast<float4*>(tb + lane * 36 + 4 * i) =
                make_float4(wt * __uint_as_float(r[4 * i]), wt * __uint_as_float(r[4 * i + 1]),
                            wt * __uint_as_float(r[4 * i + 2]), wt * __uint_as_float(r[4 * i + 3]));
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rr = 4 * i + (lane >> 3);  // row of the warp this lane adds for
            const int tr = __shfl_sync(0xFFFFFFFFu, t, rr);
            if ((vmask >> rr) & 1u) {
              const float4 v = *reinterpret_cast<const float4*>(tb + rr * 36 + 4 * (lane & 7));
              red_add_v4(p.acc32 + (size_t)tr * H + (size_t)nt * kBN + 32 * c + 4 * (lane & 7), v.x, v.y, v.z, v.w);
            }
          }
          __syncwarp();
        }
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 2) {
    __syncwarp();
    tc::fence_after();
    tc::tmem_dealloc(tbase, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
template <int KIND, int STAGE>
static cudaError_t set_limit_tc() {
  return cudaFuncSetAttribute(tc_stage_kernel<KIND, STAGE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)TcLayout::total);
}

cudaError_t tc_set_smem_limits() {
  cudaError_t e = set_limit_tc<TC_A8W4, 1>();
  if (e == cudaSuccess) e = set_limit_tc<TC_A8W4, 2>();
  if (e == cudaSuccess) e = set_limit_tc<TC_A4W4, 1>();
  if (e == cudaSuccess) e = set_limit_tc<TC_A4W4, 2>();
  return e;
}

cudaError_t launch_tc_stage(int kind, int stage, const TcParams& p, const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                            int grid, cudaStream_t st) {
  const size_t smem = TcLayout::total;
  const dim3 g(grid), b(kThreadsTc);
  if (kind == TC_A8W4 && stage == 1) return launch_k(tc_stage_kernel<TC_A8W4, 1>, g, b, smem, st, true, p, tm_a, tm_b);
  if (kind == TC_A8W4) return launch_k(tc_stage_kernel<TC_A8W4, 2>, g, b, smem, st, true, p, tm_a, tm_b);
  if (stage == 1) return launch_k(tc_stage_kernel<TC_A4W4, 1>, g, b, smem, st, true, p, tm_a, tm_b);
  return launch_k(tc_stage_kernel<TC_A4W4, 2>, g, b, smem, st, true, p, tm_a, tm_b);
}

}  // namespace moe
