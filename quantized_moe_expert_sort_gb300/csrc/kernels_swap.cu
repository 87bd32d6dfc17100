// Grouped stage-1 / stage-2 kernels on the 5th-generation tensor cores for
// few routed rows per expert (decode and small batches).
//
// At decode the path streams the fp4 weights of every active expert once and
// each expert sees only a handful of routed rows ("Retune Kimi-K3 a16w4 MoE
// tile geometry", Summary: the 1-token shape is bound by weight traffic). The
// weight tile therefore takes the M = 128 side of the block-scaled MMA and the
// expert's routed rows the N side (16..64 columns), so one MMA instruction
// covers 128 output features of up to 64 rows, and the tensor pipe keeps up
// with HBM while the SMs stay free to stream.
//
// Kinds (A = weights, e2m1 with e8m0 per 32 along K; B = the routed rows):
//   SW_A8 : kind::mxf8f6f4, B = e4m3 1x32-scaled activations ("Add Kimi-K3
//           A8W4 support..." Technical Details), weights expanded by TMA to one
//           16-element group per 16 bytes of shared memory, K tile 128.
//   SW_A4 : kind::mxf4, A and B packed e2m1 ("Add an opt-in a4w4 SiTUv2 MoE
//           path..."), scale_vec::2X, K tile 256.
//   SW_A16: bf16 activations ("Retune Kimi-K3 a16w4 MoE tile geometry"). Each
//           bf16 value is carried as hi + lo, two e4m3 codes with their own
//           1x32 e8m0 scales (hi: the block rounded to e4m3 with emax 7, so no
//           code saturates; lo: the exact residual, rounded the same way); two
//           MMAs accumulate hi and lo into the same accumulator. hi + lo equals
//           the bf16 value exactly for elements within 2^12 of their block's
//           largest magnitude, and within 2^-11 of the block maximum otherwise.
//
// Unit of work: (active expert, 128-row weight tile). Stage 1 loads the gate
// and the up rows of the same 128 intermediate columns j as two A tiles into
// two accumulators, so TMEM lane j holds g and u of column j for every routed
// row; the epilogue forms y = act(g, u) and requantises y per 32 along I
// across the warp's 32 lanes. Stage 2 loads 128 rows of H; lane h adds
// w * z[h] for each routed row into the fp32 combine buffer (one coalesced
// 128-byte red per warp and row). Experts with more than kNMax rows are
// split into several items that stream the weight tile again.
//
// CTA (one per SM, persistent): warp 0 enumerates items, publishes them in a
// ring in shared memory and issues TMA for the weight tiles and the routed
// rows (sorted rows are contiguous per expert: no gather); warp 1 copies the
// e8m0 scales of both operands with cp.async straight into the tcgen05.cp
// chunk layout, two stages ahead of its mbarrier arrivals; warp 2 owns TMEM
// and issues tcgen05.cp + tcgen05.mma; warps 4-7 run the epilogue from
// double-buffered accumulators.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace moe {
namespace {

constexpr int kThreadsSw = 256;
constexpr int kEpiWarpsSw = 4;
constexpr int kTile = 128 * 128;  // one 128-row x 128-byte operand tile
constexpr int kURing = 4;         // items in flight in the shared-memory ring
constexpr int kSfLag = 2;         // stages warp 1 runs ahead of its arrivals

template <int KIND> struct SwKind;
template <> struct SwKind<SW_A16> {
  static constexpr int kKTile = 128, kBlocks = 4, kChunks = 1, kNMax = 32;
  static constexpr bool kHiLo = true, kMxf4 = false;
};
template <> struct SwKind<SW_A8> {
  static constexpr int kKTile = 128, kBlocks = 4, kChunks = 1, kNMax = 64;
  static constexpr bool kHiLo = false, kMxf4 = false;
};
template <> struct SwKind<SW_A4> {
  static constexpr int kKTile = 256, kBlocks = 8, kChunks = 2, kNMax = 64;
  static constexpr bool kHiLo = false, kMxf4 = true;
};

template <int STAGE> constexpr int sw_stages() { return STAGE == 1 ? 4 : 6; }

struct UItem {
  int e, tile, row0, nrows;  // nrows < 0: end of work
  int pid[64];
  float w[64];
};

template <int STAGE> struct SwLayout {
  static constexpr int kNS = sw_stages<STAGE>();
  static constexpr uint32_t a_bytes = (STAGE == 1 ? 2 : 1) * kTile;    // gate + up, or one tile
  static constexpr uint32_t b_bytes = 64 * 128;                        // kNMax rows (x2 for hi / lo at 32)
  static constexpr uint32_t sf_bytes = 4 * 1024;                       // sfa gate, sfa up, sfb, sfb lo
  static constexpr uint32_t a = 0;
  static constexpr uint32_t b = a + kNS * a_bytes;
  static constexpr uint32_t sf = b + kNS * b_bytes;
  static constexpr uint32_t items = sf + kNS * sf_bytes;
  static constexpr uint32_t bars = items + kURing * sizeof(UItem);
  static constexpr uint32_t tmem_slot = bars + (2 * kNS + 4 + 2 * kURing + 1) * 8;
  static constexpr uint32_t total = tmem_slot + 16 + 1024;  // + alignment slack
};

constexpr uint32_t kTmemColsSw = 512;
constexpr uint32_t kSfColSw = 256;  // scale slots: 32 columns per pipeline slot from here

__device__ __forceinline__ void tma_load_2d_sw(void* dst, const CUtensorMap* m, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Byte offset of (row m, block kb % 4) inside a 512-byte scale chunk.
__device__ __forceinline__ uint32_t sf_off_sw(int m) { return 16u * (m & 31) + 4u * (m >> 5); }

// Weight tile bytes one TMA load reports: packed global bytes (see the
// 16U4_ALIGN16B note of the prefill kernels), 16 KB for packed e2m1.
template <int KIND> constexpr uint32_t w_tile_tx() { return SwKind<KIND>::kMxf4 ? kTile : kTile / 2; }

}  // namespace

template <int KIND, int STAGE>
__global__ void __launch_bounds__(kThreadsSw, 1) swap_stage_kernel(StageParams p, const __grid_constant__ CUtensorMap tm_w,
                                                                   const __grid_constant__ CUtensorMap tm_x) {
  using KD = SwKind<KIND>;
  using L = SwLayout<STAGE>;
  constexpr int kNS = L::kNS;
  constexpr int NMAX = KD::kNMax;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::bars);
  uint64_t* empty = full + kNS;
  uint64_t* tfull = empty + kNS;
  uint64_t* tempty = tfull + 2;
  uint64_t* ufull = tempty + 2;
  uint64_t* uempty = ufull + kURing;
  uint64_t* drain = uempty + kURing;
  UItem* items = reinterpret_cast<UItem*>(smem + L::items);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::tmem_slot);
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = p.H, I = p.I, K = p.K;
  const int kdim = STAGE == 1 ? H : I;
  const int ktiles = (kdim + KD::kKTile - 1) / KD::kKTile;
  const int nblk_k = kdim / 32;
  const int ntn = STAGE == 1 ? I / 128 : H / 128;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < kNS; ++s) { mbar_init(&full[s], 1 + 32); mbar_init(&empty[s], 1); }
    for (int s = 0; s < 2; ++s) { mbar_init(&tfull[s], 1); mbar_init(&tempty[s], kEpiWarpsSw); }
    for (int s = 0; s < kURing; ++s) { mbar_init(&ufull[s], 1); mbar_init(&uempty[s], 2 + kEpiWarpsSw); }
    mbar_init(drain, 1);
    fence_barrier_init();
  }
  if (!KD::kMxf4) {
    // zero the weight tiles: the unpacking TMA never writes their 8-byte gaps
    for (uint32_t i = threadIdx.x; i < kNS * L::a_bytes / 16; i += blockDim.x)
      reinterpret_cast<uint4*>(smem + L::a)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async();
  }
  if (warp == 2) {
    tc::tmem_alloc(tmem_slot, kTmemColsSw);
    tc::tmem_relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 0) {
    // ------------------- item enumeration + TMA producer -------------------
    if (lane == 0) {
      tma_prefetch_desc(&tm_w);
      tma_prefetch_desc(&tm_x);
    }
    const int nunits = p.meta[META_NUM_ACTIVE] * ntn;
    uint32_t stage = 0;
    int it = 0;
    int u = blockIdx.x;
    int e_next = u < nunits ? p.active_experts[u / ntn] : -1;
    bool stop = false;
    while (!stop) {
      const bool more = u < nunits;
      const int e = e_next, tile = more ? u % ntn : 0;
      const int cnt = more ? p.expert_count[e] : 0;
      const int off = more ? p.expert_offset[e] : 0;
      u += gridDim.x;
      e_next = u < nunits ? p.active_experts[u / ntn] : -1;
      const int nch = more ? (cnt + NMAX - 1) / NMAX : 1;
      for (int ch = 0; ch < nch; ++ch, ++it) {
        const int us = it % kURing;
        if (!mbar_wait_or_abort(&uempty[us], ((it / kURing) & 1) ^ 1, p.err, &abort_flag)) { stop = true; break; }
        UItem* ui = items + us;
        const int row0 = off + ch * NMAX;
        const int nrows = more ? min(NMAX, cnt - ch * NMAX) : -1;
        if (STAGE == 2 && more) {
          for (int n = lane; n < nrows; n += 32) {
            const int pid = p.sorted_ids[row0 + n];
            ui->pid[n] = pid;
            ui->w[n] = p.topk_w[pid];
          }
        }
        if (lane == 0) { ui->e = e; ui->tile = tile; ui->row0 = row0; ui->nrows = nrows; }
        __syncwarp();
        if (lane == 0) mbar_arrive(&ufull[us]);
        if (!more) { stop = true; break; }
        if (lane == 0) {
          const int nbox = (nrows + 15) / 16;
          const uint32_t btx = (uint32_t)nbox * 16 * 128 * (KD::kHiLo ? 2 : 1);
          for (int ks = 0; ks < ktiles; ++ks, ++stage) {
            const int slot = stage % kNS;
            if (!mbar_wait_or_abort(&empty[slot], ((stage / kNS) & 1) ^ 1, p.err, &abort_flag)) { stop = true; break; }
            uint8_t* sa = smem + L::a + slot * L::a_bytes;
            uint8_t* sb = smem + L::b + slot * L::b_bytes;
            mbar_arrive_expect_tx(&full[slot], (STAGE == 1 ? 2 : 1) * w_tile_tx<KIND>() + btx);
            if (STAGE == 1) {
              tma_load_4d(sa, &tm_w, ks * 128, tile * 128, 0, e, &full[slot]);
              tma_load_4d(sa + kTile, &tm_w, ks * 128, tile * 128, 1, e, &full[slot]);
            } else {
              tma_load_3d(sa, &tm_w, ks * 128, tile * 128, e, &full[slot]);
            }
            // routed rows: contiguous sorted rows [row0, row0 + nrows), 16-row boxes
            // (rows past this expert belong to later experts and only fill unused columns)
            for (int bx = 0; bx < nbox; ++bx) {
              tma_load_2d_sw(sb + bx * 16 * 128, &tm_x, ks * 128, row0 + 16 * bx, &full[slot]);
              if (KD::kHiLo)
                tma_load_2d_sw(sb + (NMAX + bx * 16) * 128, &tm_x, kdim + ks * 128, row0 + 16 * bx, &full[slot]);
            }
          }
        }
        stop = __shfl_sync(0xFFFFFFFFu, stop ? 1 : 0, 0) != 0;
        stage = __shfl_sync(0xFFFFFFFFu, stage, 0);
        if (stop) break;
      }
    }
  } else if (warp == 1) {
    // ---------- e8m0 scales of both operands into tcgen05.cp chunks ----------
    const int sb_w = kdim / 32;  // weight-scale bytes per row
    uint32_t stage = 0, pend = 0;
    int it = 0;
    while (true) {
      const int us = it % kURing;
      if (!mbar_wait_or_abort(&ufull[us], (it / kURing) & 1, p.err, &abort_flag)) break;
      const UItem* ui = items + us;
      const int e = ui->e, tile = ui->tile, row0 = ui->row0, nrows = ui->nrows;
      __syncwarp();
      if (lane == 0) mbar_arrive(&uempty[us]);
      ++it;
      if (nrows < 0) break;
      const uint8_t* wsrc = STAGE == 1 ? p.wscale + ((size_t)e * 2 * I + (size_t)tile * 128) * sb_w
                                       : p.wscale + ((size_t)e * H + (size_t)tile * 128) * sb_w;
      bool ok = true;
      for (int ks = 0; ks < ktiles; ++ks) {
        const int slot = stage % kNS;
        if (!mbar_wait_or_abort(&empty[slot], ((stage / kNS) & 1) ^ 1, p.err, &abort_flag)) { ok = false; break; }
        uint8_t* sf = smem + L::sf + slot * L::sf_bytes;  // [sfa gate | sfa up | sfb | sfb lo], 1 KB each
        for (int c = 0; c < KD::kChunks; ++c) {
          const int kb0 = ks * KD::kBlocks + 4 * c;
          if (kb0 < nblk_k) {  // kdim % 128 == 0: a chunk is all in or all out
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int m = 4 * lane + i;
              cp_async4(sf + 512 * c + sf_off_sw(m), wsrc + (size_t)m * sb_w + kb0);
              if (STAGE == 1) cp_async4(sf + 1024 + 512 * c + sf_off_sw(m), wsrc + ((size_t)I + m) * sb_w + kb0);
            }
            for (int n = lane; n < nrows; n += 32) {
              const uint8_t* src = p.as + (size_t)(row0 + n) * p.xs_stride + kb0;
              cp_async4(sf + 2048 + 512 * c + sf_off_sw(n), src);
              if (KD::kHiLo) cp_async4(sf + 3072 + 512 * c + sf_off_sw(n), src + nblk_k);
            }
          } else {  // past the end of K: neutral scales (the operands there are zero)
            const uint4 n127 = make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
            *reinterpret_cast<uint4*>(sf + 512 * c + 16 * lane) = n127;
            *reinterpret_cast<uint4*>(sf + 1024 + 512 * c + 16 * lane) = n127;
            *reinterpret_cast<uint4*>(sf + 2048 + 512 * c + 16 * lane) = n127;
            *reinterpret_cast<uint4*>(sf + 3072 + 512 * c + 16 * lane) = n127;
          }
        }
        cp_async_commit();
        ++stage;
        ++pend;
        if (pend > kSfLag) {
          cp_async_wait<kSfLag>();
          fence_proxy_async();  // this thread's generic-proxy smem writes -> visible to tcgen05.cp
          mbar_arrive(&full[(stage - pend) % kNS]);
          --pend;
        }
      }
      if (!ok) break;
    }
    cp_async_wait<0>();
    fence_proxy_async();
    while (pend > 0) {
      mbar_arrive(&full[(stage - pend) % kNS]);
      --pend;
    }
  } else if (warp == 2) {
    // ------------------------------ MMA issuer ------------------------------
    if (lane == 0) {
      uint32_t stage = 0;
      int it = 0;
      while (true) {
        const int us = it % kURing;
        if (!mbar_wait_or_abort(&ufull[us], (it / kURing) & 1, p.err, &abort_flag)) break;
        const int nrows = items[us].nrows;
        mbar_arrive(&uempty[us]);
        if (nrows < 0) break;
        const int buf = it & 1;
        ++it;
        if (!mbar_wait_or_abort(&tempty[buf], (((it - 1) >> 1) & 1) ^ 1, p.err, &abort_flag)) break;
        tc::fence_after();
        const int nmma = (nrows + 15) / 16 * 16;
        const uint32_t dg = tbase + buf * 2 * NMAX;
        const uint32_t du = dg + NMAX;
        bool ok = true;
        for (int ks = 0; ks < ktiles; ++ks, ++stage) {
          const int slot = stage % kNS;
          if (!mbar_wait_or_abort(&full[slot], (stage / kNS) & 1, p.err, &abort_flag)) { ok = false; break; }
          tc::fence_after();
          const uint32_t sfc = tbase + kSfColSw + slot * 32;  // sfa gate +0, sfa up +8, sfb +16, sfb lo +24
          const uint32_t sfs = smem_u32(smem + L::sf + slot * L::sf_bytes);
          for (int c = 0; c < KD::kChunks; ++c) {
            tc::cp_32x128b_warpx4(sfc + 4 * c, tc::sdesc(sfs + 512 * c, 0, 128, tc::SW_NONE));
            if (STAGE == 1) tc::cp_32x128b_warpx4(sfc + 8 + 4 * c, tc::sdesc(sfs + 1024 + 512 * c, 0, 128, tc::SW_NONE));
            tc::cp_32x128b_warpx4(sfc + 16 + 4 * c, tc::sdesc(sfs + 2048 + 512 * c, 0, 128, tc::SW_NONE));
            if (KD::kHiLo) tc::cp_32x128b_warpx4(sfc + 24 + 4 * c, tc::sdesc(sfs + 3072 + 512 * c, 0, 128, tc::SW_NONE));
          }
          const uint32_t sa = smem_u32(smem + L::a + slot * L::a_bytes);
          const uint32_t sb = smem_u32(smem + L::b + slot * L::b_bytes);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint64_t db = tc::sdesc(sb + 32 * i, 16, 1024, tc::SW_128B);
            const uint32_t acc = (ks > 0 || i > 0) ? 1u : 0u;
#pragma unroll
            for (int g = 0; g < (STAGE == 1 ? 2 : 1); ++g) {
              const uint64_t da = tc::sdesc(sa + g * kTile + 32 * i, 16, 1024, tc::SW_128B);
              const uint32_t d = g == 0 ? dg : du;
              const uint32_t sfa = sfc + 8 * g;
              if (KD::kMxf4) {
                const uint32_t id = tc::idesc_bs(128, nmma, tc::MXF4_E2M1, tc::MXF4_E2M1, 2 * (i & 1), 2 * (i & 1));
                tc::mma_mxf4(d, da, db, id, sfa + 4 * (i >> 1), sfc + 16 + 4 * (i >> 1), acc);
              } else {
                const uint32_t id = tc::idesc_bs(128, nmma, tc::F8F6F4_E2M1, tc::F8F6F4_E4M3, i, i);
                tc::mma_mxf8f6f4(d, da, db, id, sfa, sfc + 16, acc);
                if (KD::kHiLo) {
                  const uint64_t dbl = tc::sdesc(sb + NMAX * 128 + 32 * i, 16, 1024, tc::SW_128B);
                  tc::mma_mxf8f6f4(d, da, dbl, id, sfa, sfc + 24, 1u);
                }
              }
            }
          }
          tc::commit(&empty[slot]);
        }
        if (!ok) break;
        tc::commit(&tfull[buf]);
      }
      // every MMA / copy this thread issued has finished before TMEM is released
      tc::commit(drain);
      mbar_wait(drain, 0, p.err);
    }
  } else if (warp >= 4) {
    // ------------------------------ epilogue ------------------------------
    const int q = warp & 3;                 // TMEM lane quadrant of this warp
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    int it = 0;
    while (true) {
      const int us = it % kURing;
      if (!mbar_wait_or_abort(&ufull[us], (it / kURing) & 1, p.err, &abort_flag)) break;
      const UItem* ui = items + us;
      const int tile = ui->tile, row0 = ui->row0, nrows = ui->nrows;
      if (nrows < 0) break;
      const int buf = it & 1;
      if (!mbar_wait_or_abort(&tfull[buf], (it >> 1) & 1, p.err, &abort_flag)) break;
      ++it;
      __syncwarp();  // tcgen05.ld is .sync.aligned: the whole warp, converged
      tc::fence_after();
      const uint32_t dg = tbase + lane_off + buf * 2 * NMAX;
      if (STAGE == 1) {
        const int j = tile * 128 + 32 * q + lane;  // intermediate column of this lane
        for (int c0 = 0; c0 < nrows; c0 += 16) {
          uint32_t gr[16], ur[16];
          tc::ld_32x32b_x16(dg + c0, gr);
          tc::ld_32x32b_x16(dg + NMAX + c0, ur);
          tc::ld_wait();
          const int nn = min(16, nrows - c0);
#pragma unroll
          for (int n = 0; n < 16; ++n) {
            if (n < nn) {
              const int row = row0 + c0 + n;
              float y = act_apply(p.act, __uint_as_float(gr[n]), __uint_as_float(ur[n]), p.beta, p.lbeta);
              if (KD::kHiLo) {
                // bf16 intermediate, carried as hi + lo e4m3 (same rule as the activations)
                y = __bfloat162float(__float2bfloat16_rn(y));
                const float amax = warp_max(fabsf(y));
                uint32_t s0 = 127u;
                float mul = 0.0f;
                if (amax > 0.0f) {
                  int E = floor_log2_f32(amax) - 7;
                  E = E < -127 ? -127 : (E > 127 ? 127 : E);
                  s0 = (uint32_t)(E + 127);
                  mul = exp2_neg(E);
                }
                const uint32_t hc = cvt_e4m3x2(__fmul_rn(y, mul), 0.0f) & 0xFFu;
                const float r = y - e4m3_to_f32(hc) * e8m0_to_f32(s0);
                const float rmax = warp_max(fabsf(r));
                uint32_t s1 = 127u;
                float mul1 = 0.0f;
                if (rmax > 0.0f) {
                  int E = floor_log2_f32(rmax) - 7;
                  E = E < -127 ? -127 : (E > 127 ? 127 : E);
                  s1 = (uint32_t)(E + 127);
                  mul1 = exp2_neg(E);
                }
                const uint32_t lc = cvt_e4m3x2(__fmul_rn(r, mul1), 0.0f) & 0xFFu;
                p.oq[(size_t)row * (2 * I) + j] = (uint8_t)hc;
                p.oq[(size_t)row * (2 * I) + I + j] = (uint8_t)lc;
                if (lane == 0) {
                  p.os[(size_t)row * p.os_stride + j / 32] = (uint8_t)s0;
                  p.os[(size_t)row * p.os_stride + I / 32 + j / 32] = (uint8_t)s1;
                }
              } else {
                const int emax = KD::kMxf4 ? 2 : 8;
                const float amax = warp_max(fabsf(y));
                uint32_t sb = 127u;
                float mul = 0.0f;
                if (amax > 0.0f) {
                  int E = floor_log2_f32(amax) - emax;
                  E = E < -127 ? -127 : (E > 127 ? 127 : E);
                  sb = (uint32_t)(E + 127);
                  mul = exp2_neg(E);
                }
                if (KD::kMxf4) {
                  const uint32_t code = cvt_e2m1x2(__fmul_rn(y, mul), 0.0f) & 0xFu;
                  const uint32_t nb = __shfl_down_sync(0xFFFFFFFFu, code, 1);
                  if ((lane & 1) == 0) p.oq[(size_t)row * (I / 2) + j / 2] = (uint8_t)(code | (nb << 4));
                } else {
                  p.oq[(size_t)row * I + j] = (uint8_t)(cvt_e4m3x2(__fmul_rn(y, mul), 0.0f) & 0xFFu);
                }
                if (lane == 0) p.os[(size_t)row * p.os_stride + j / 32] = (uint8_t)sb;
              }
            }
          }
        }
      } else {
        const int h = tile * 128 + 32 * q + lane;
        for (int c0 = 0; c0 < nrows; c0 += 16) {
          uint32_t r[16];
          tc::ld_32x32b_x16(dg + c0, r);
          tc::ld_wait();
          const int nn = min(16, nrows - c0);
#pragma unroll
          for (int n = 0; n < 16; ++n) {
            if (n < nn) {
              const int pid = ui->pid[c0 + n];
              const float w = ui->w[c0 + n];
              atomicAdd(p.acc32 + (size_t)(pid / K) * H + h, w * __uint_as_float(r[n]));
            }
          }
        }
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&tempty[buf]);
        mbar_arrive(&uempty[us]);
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 2) {
    __syncwarp();
    tc::fence_after();
    tc::tmem_dealloc(tbase, kTmemColsSw);
  }
}

// ---------------------------------------------------------------------------
template <int KIND, int STAGE>
static cudaError_t set_limit_sw() {
  return cudaFuncSetAttribute(swap_stage_kernel<KIND, STAGE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)SwLayout<STAGE>::total);
}

cudaError_t swap_set_smem_limits() {
  cudaError_t e = set_limit_sw<SW_A16, 1>();
  if (e == cudaSuccess) e = set_limit_sw<SW_A16, 2>();
  if (e == cudaSuccess) e = set_limit_sw<SW_A8, 1>();
  if (e == cudaSuccess) e = set_limit_sw<SW_A8, 2>();
  if (e == cudaSuccess) e = set_limit_sw<SW_A4, 1>();
  if (e == cudaSuccess) e = set_limit_sw<SW_A4, 2>();
  return e;
}

template <int KIND>
static void launch_sw(int stage, const StageParams& p, const CUtensorMap& tm_w, const CUtensorMap& tm_x, int grid,
                      cudaStream_t st) {
  if (stage == 1)
    swap_stage_kernel<KIND, 1><<<grid, kThreadsSw, SwLayout<1>::total, st>>>(p, tm_w, tm_x);
  else
    swap_stage_kernel<KIND, 2><<<grid, kThreadsSw, SwLayout<2>::total, st>>>(p, tm_w, tm_x);
}

cudaError_t launch_swap_stage(int kind, int stage, const StageParams& p, const CUtensorMap& tm_w, const CUtensorMap& tm_x,
                              int grid, cudaStream_t st) {
  if (kind == SW_A16) launch_sw<SW_A16>(stage, p, tm_w, tm_x, grid, st);
  else if (kind == SW_A8) launch_sw<SW_A8>(stage, p, tm_w, tm_x, grid, st);
  else launch_sw<SW_A4>(stage, p, tm_w, tm_x, grid, st);
  return cudaGetLastError();
}

}  // namespace moe
