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
//   SW_A16: bf16 activations ("Retune Kimi-K3 a16w4 MoE tile geometry"), on
//           kind::mxf4 like SW_A4: each bf16 value is carried as the sum of
//           kTerms = 6 e2m1 codes, each term with its own 1x32 e8m0 scale (term
//           t quantises, by the MX rule, what the earlier terms left over).
//           Each term lowers the block's scale exponent by at least 2 and leaves
//           a residual below twice its own scale, so after n terms every value
//           is within 2^(1-2n) of its 32-block's maximum (2^-11 for six); on
//           N(0,1) data 99.97% of values come out exact. The weights stay
//           packed. The terms of sorted row r are stored as
//           sub-rows r * kTerms + t, so they sit side by side in the N dimension
//           of one MMA (column n * kTerms + t for item row n) and the weights are
//           read once; few rows need few columns.
//
// Unit of work: (active expert, two 128-row weight tiles). Stage 1 loads the
// gate and the up rows of the same 128 intermediate columns j as the two A
// tiles, into two accumulators, so TMEM lane j holds g and u of column j for
// every routed row; the epilogue forms y = act(g, u) and requantises y per 32
// along I across the warp's 32 lanes. Stage 2 loads 256 consecutive rows of H;
// lane h adds w * z[h] for each routed row into the fp32 combine buffer (one
// coalesced 128-byte red per warp and row). Experts with more than kNMax rows
// are split into several items that stream the weight tiles again.
//
// CTA (one per SM, persistent): warp 3 enumerates the items (expert ids,
// counts and offsets fetched 32 units at a time) and publishes them in a ring
// in shared memory (at stage 2 with each item's row tokens and top-k weights,
// copied in by cp.async); warp 0 issues TMA for the weight tiles and the routed
// rows (sorted rows are contiguous per expert: no gather) and prefetches scale
// rows into L2; warp 1 copies the e8m0 scales of both operands with cp.async
// straight into the tcgen05.cp chunk layout, kSfLag stages ahead of its
// mbarrier arrivals; warp 2 owns TMEM and issues tcgen05.cp + tcgen05.mma;
// warps 4-7 (stage 1) or 4-11 (stage 2: two warpgroups on alternate items) run
// the epilogue from double-buffered accumulators.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace moe {
namespace {

// Threads per CTA: 4 role warps + one epilogue warpgroup (stage 1) or two (stage 2).
template <int STAGE> constexpr int threads_sw() { return STAGE == 2 ? 384 : 256; }
constexpr int kEpiWarpsSw = 4;  // warps per epilogue warpgroup; two warpgroups take alternate items

template <int KIND> struct SwKind;
// kNMax: routed rows per item; kTerms: code terms per value (B rows = kTerms x rows);
// kURing: items in flight in the shared-memory ring (each slot also holds the token
// and top-k weight of its rows). SW_A8's 5 unpacked operand stages leave room
// for a shorter item ring.
template <> struct SwKind<SW_A16> {
  // 13 rows x 6 terms = 78 sub-rows: 80 accumulator columns, which leaves TMEM room for
  // the scale slots of nine stage-2 operand stages
  static constexpr int kNMax = 13, kTerms = A16_TERMS, kURing = 32;
  static constexpr bool kMxf4 = true;
};
template <> struct SwKind<SW_A8> {
  static constexpr int kNMax = 64, kTerms = 1, kURing = 16;
  static constexpr bool kMxf4 = false;
};
template <> struct SwKind<SW_A4> {
  static constexpr int kNMax = 64, kTerms = 1, kURing = 32;
  static constexpr bool kMxf4 = true;
};

// Operand pipeline of one (kind, stage).
//   kKTile: K per stage; kRow: shared-memory bytes per operand row (the TMA box
//   width and the swizzle span); kNS: operand stages; kSfRing: scale-chunk slots
//   (a ring of its own, deeper than the operand ring); kSfLag: stages the scale
//   warp's copies run ahead of its arrivals.
// Packed e2m1 (mxf4) streams K in 128-byte rows (K tile 256) at stage 1. At stage
// 2 K = inter is a few hundred (384 for the TP8 shard: 192 bytes per row):
// 128-byte boxes would leave half of every second box outside the matrix, and
// with 42 KB stages only four fit, too few in flight for this short-item,
// latency-bound stream. 64-byte rows (K tile 128, 64-byte swizzle) fit K exactly
// and halve the stage, so nine are in flight (measured: TP8 a16w4 T = 64 stage 2
// 140 -> 115 us).
// kind::mxf8f6f4 takes the weights expanded to one 16-element group per 16 bytes
// (128-byte rows for a K tile of 128), so its tiles take twice the shared memory
// per HBM byte.
// KS > 1 (stage 1 only): the split-K variant, KS CTAs of a cluster per unit, three operand stages.
template <int KIND, int STAGE, int KS = 1> struct SwCfg {
  static constexpr bool kNarrow = SwKind<KIND>::kMxf4 && STAGE == 2;
  static constexpr int kKTile = SwKind<KIND>::kMxf4 && !kNarrow ? 256 : 128;
  static constexpr int kChunks = kKTile / 128;                      // 4-block scale chunks per stage
  static constexpr int kBlocks = kKTile / 32;                       // 32-blocks per stage
  static constexpr int kRow = SwKind<KIND>::kMxf4 ? kKTile / 2 : 128;
  static constexpr int kXStep = SwKind<KIND>::kMxf4 ? kKTile / 2 : kKTile;  // TMA x per stage (bytes / 4-bit elements)
  static constexpr int kKSteps = kRow / 32;                         // MMAs per tile and stage (32 bytes of K each)
  static constexpr int kNS = KS > 1 ? 3 : (kNarrow ? 9 : (SwKind<KIND>::kMxf4 ? 4 : 5));
  static constexpr int kSfRing = kNarrow ? 16 : 8;
  // split-K CTAs run only a few stages each: their scale arrivals may not lag far behind
  static constexpr int kSfLag = KS > 1 ? 1 : (kNarrow ? 8 : 4);
  static constexpr uint32_t kSwz = kRow == 128 ? tc::SW_128B : tc::SW_64B;
  static constexpr int kSfCols = kChunks == 2 ? 32 : 16;            // TMEM columns per scale slot
};

template <int KIND> constexpr int acc_cols() {  // TMEM columns of one accumulator (largest MMA N)
  return (SwKind<KIND>::kTerms * SwKind<KIND>::kNMax + 15) / 16 * 16;
}

struct UItem {
  int e, tile, row0, nrows;  // nrows < 0: end of work
};

template <int KIND, int STAGE, int KS = 1> struct SwLayout {
  using C = SwCfg<KIND, STAGE, KS>;
  static constexpr int kNS = C::kNS;
  static constexpr int kURing = SwKind<KIND>::kURing, kSfRing = C::kSfRing;
  static constexpr uint32_t tile_bytes = 128 * C::kRow;                // one 128-row operand tile
  static constexpr uint32_t a_bytes = 2 * tile_bytes;                  // two weight tiles
  static constexpr uint32_t b_bytes = acc_cols<KIND>() * C::kRow;      // B rows = terms x routed rows
  static constexpr uint32_t sf_op = C::kChunks * 512;                  // one operand's chunks
  static constexpr uint32_t sf_bytes = 3 * sf_op;                      // sfa tile 0, sfa tile 1, sfb
  static constexpr uint32_t a = 0;
  static constexpr uint32_t b = a + kNS * a_bytes;
  static constexpr uint32_t sf = b + kNS * b_bytes;
  static constexpr uint32_t items = sf + kSfRing * sf_bytes;
  static constexpr uint32_t rows = items + kURing * sizeof(UItem);     // per slot: int tok[kNMax], float w[kNMax]
  static constexpr uint32_t row_bytes = 8 * SwKind<KIND>::kNMax;
  // split-K: per partner rank, the g and u partial sums of a 16-row chunk, 128 columns
  static constexpr uint32_t red = rows + kURing * row_bytes;
  static constexpr uint32_t red_bytes = (KS - 1) * 16 * 128 * 8;
  static constexpr uint32_t bars = red + red_bytes;
  static constexpr uint32_t tmem_slot = bars + (2 * kNS + 4 + 3 * kURing + kSfRing + 1 + (KS > 1 ? 8 : 0)) * 8;
  static constexpr uint32_t total = tmem_slot + 16 + 1024;  // + alignment slack
};

constexpr uint32_t kTmemColsSw = 512;
// TMEM: accumulators (2 buffers x 2 tiles) from column 0, then one scale slot per
// operand stage: [sfa tile 0 | sfa tile 1 | sfb], 4 columns per 4-block chunk.
template <int KIND> constexpr uint32_t sf_col0() { return 4 * acc_cols<KIND>(); }

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
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// One arrival on `bar` once every cp.async this thread issued so far has landed
// (the barrier's expected count includes it).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
template <int N> __device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// L2 prefetch of a contiguous range (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Warp-uniform bounded wait: lane 0 polls, the outcome is broadcast, and the
// warp reconverges (memory ordering for the data the barrier guards).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int* err, volatile int* abort) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait_or_abort(bar, parity, err, abort);
  ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
  __syncwarp();
  return ok;
}

// ---- thread-block cluster helpers (split-K stage 1) ----------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of this CTA's shared-memory location `saddr` in the shared memory of CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_v2(uint32_t addr, float a, float b) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(a), "f"(b) : "memory");
}
// Arrive on an mbarrier of another CTA of the cluster, releasing this thread's earlier
// writes (including its st.shared::cluster) at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, "
      "p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
// Warp-uniform bounded wait for a barrier that other CTAs of the cluster arrive on
// (acquire at cluster scope: their shared-memory writes are visible afterwards).
__device__ __forceinline__ bool warp_wait_cluster(uint64_t* bar, uint32_t parity, int* err, volatile int* abort) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) {
    const uint64_t t0 = global_ns();
    ok = false;
    while (true) {
      if (mbar_try_wait_cluster(bar, parity, MOE_SUSPEND_NS)) { ok = true; break; }
      if (*abort) break;
      if (global_ns() - t0 > MOE_WAIT_NS) {
        *abort = 1;
        set_error(err, DEV_ERR_TIMEOUT);
        break;
      }
    }
  }
  ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
  __syncwarp();
  return ok;
}
// All threads of all CTAs of the cluster (memory ordered at cluster scope).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Requantise one intermediate row y (lane = column j) per 32 along I: kTerms = 1
// gives e4m3 (!kMxf4) or e2m1 codes with an e8m0 scale per block (MX rule); kTerms
// > 1 carries the bf16-rounded y as kTerms e2m1 code terms, term t quantising
// what the earlier terms left (exact residuals). Row r's term t is sub-row
// r * kTerms + t of the codes (I / 2 bytes) and of the scales (os_stride bytes).
template <int kTerms, bool kMxf4>
__device__ __noinline__ void requant_row(float y, int row, int j, int lane, int I, uint8_t* oq, uint8_t* os,
                                         int os_stride) {
  if (kTerms > 1) y = __bfloat162float(__float2bfloat16_rn(y));
#pragma unroll 1
  for (int t = 0; t < kTerms; ++t) {
    constexpr int emax = kMxf4 ? 2 : 8;
    const float amax = warp_max(fabsf(y));
    uint32_t sb = 127u;
    float mul = 0.0f;
    if (amax > 0.0f) {
      int E = floor_log2_f32(amax) - emax;
      E = E < -127 ? -127 : (E > 127 ? 127 : E);
      sb = (uint32_t)(E + 127);
      mul = exp2_neg(E);
    }
    if (kMxf4) {
      const uint32_t code = cvt_e2m1x2(__fmul_rn(y, mul), 0.0f) & 0xFu;
      const uint32_t nb = __shfl_down_sync(0xFFFFFFFFu, code, 1);
      if ((lane & 1) == 0) oq[((size_t)row * kTerms + t) * (I / 2) + j / 2] = (uint8_t)(code | (nb << 4));
      if (t + 1 < kTerms) y -= e2m1_to_f32(code) * e8m0_to_f32(sb);  // exact residual
    } else {
      oq[(size_t)row * I + j] = (uint8_t)(cvt_e4m3x2(__fmul_rn(y, mul), 0.0f) & 0xFFu);
    }
    if (lane == 0) os[((size_t)row * kTerms + t) * os_stride + j / 32] = (uint8_t)sb;
  }
}

// Byte offset of (row m, block kb % 4) inside a 512-byte scale chunk.
__device__ __forceinline__ uint32_t sf_off_sw(int m) { return 16u * (m & 31) + 4u * (m >> 5); }

// Weight tile bytes one TMA load reports: packed global bytes (see the
// 16U4_ALIGN16B note of the prefill kernels), 16 KB for packed e2m1.
template <int KIND, int STAGE> constexpr uint32_t w_tile_tx() {
  return SwKind<KIND>::kMxf4 ? SwLayout<KIND, STAGE>::tile_bytes : SwLayout<KIND, STAGE>::tile_bytes / 2;
}

}  // namespace

// PK (stage 2 only): the weights come prepacked (launch_prepack_w2): the weight map
// addresses 128-row x 128-element blocks and p.wscale holds 512-byte scale chunks.
// KS > 1 (stage 1 only): split-K over a cluster of KS CTAs ("Support SiTUv2 in
// the packed-int4 MoE stage1 epilogue", Technical Details: a split-K stage 1 must
// carry the SiTUv2 epilogue past its reduction). The CTAs of a cluster run the same
// items, each over its share of K; ranks 1..KS-1 move their per-row g and u partial
// sums into rank 0's shared memory (DSMEM), and rank 0 adds them and only then applies
// the activation and the requantisation -- the activation never sees a partial sum.
template <int KIND, int STAGE, bool PK, int KS>
__global__ void __launch_bounds__(threads_sw<STAGE>(), 1) swap_stage_kernel(StageParams p, const __grid_constant__ CUtensorMap tm_w,
                                                                   const __grid_constant__ CUtensorMap tm_x) {
  using KD = SwKind<KIND>;
  using L = SwLayout<KIND, STAGE, KS>;
  using C = SwCfg<KIND, STAGE, KS>;
  static_assert(KS == 1 || STAGE == 1, "split-K is a stage-1 variant");
  constexpr int kNS = L::kNS;
  constexpr int NMAX = KD::kNMax;
  constexpr int kAccCols = acc_cols<KIND>();
  constexpr int kURing = KD::kURing, kSfRing = C::kSfRing, kSfLag = C::kSfLag;
  constexpr int kEpiGroups = STAGE == 2 ? 2 : 1;  // epilogue warpgroups (one per accumulator buffer at stage 2)
  static_assert(4 * kAccCols + kNS * C::kSfCols <= (int)kTmemColsSw, "TMEM columns");
  static_assert(kSfRing > kSfLag && L::total <= 232448, "shared memory");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::bars);  // a stage's copies and scale chunks landed
  uint64_t* empty = full + kNS;
  uint64_t* tfull = empty + kNS;
  uint64_t* tempty = tfull + 2;
  uint64_t* ufull = tempty + 2;
  uint64_t* uempty = ufull + kURing;
  uint64_t* rfull = uempty + kURing;    // the slot's row tokens / weights have landed (stage 2)
  uint64_t* sfempty = rfull + kURing;   // scale-ring slot free (MMA commit)
  uint64_t* drain = sfempty + kSfRing;
  uint64_t* red_full = drain + 1;   // split-K, rank 0: the partners' partial sums of a chunk (per quadrant)
  uint64_t* red_empty = red_full + 4;  // split-K, ranks > 0: rank 0 has read this rank's partial sums
  UItem* items = reinterpret_cast<UItem*>(smem + L::items);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::tmem_slot);
  __shared__ int abort_flag;

  if (dynamic_smem_bytes() < L::total) {  // launched with less shared memory than the layout needs
    if (threadIdx.x == 0) set_error(p.err, DEV_ERR_LAUNCH);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = p.H, I = p.I;
  const int kdim = STAGE == 1 ? H : I;
  const int ktiles = (kdim + C::kKTile - 1) / C::kKTile;
  const int nblk_k = kdim / 32;
  const int ntn = STAGE == 1 ? I / 128 : (H + 255) / 256;  // units per expert
  // split-K: units go to clusters (consecutive CTAs); rank r takes K tiles [ks0, ks1)
  const int crank = KS > 1 ? (int)cluster_ctarank() : 0;
  const long cid = KS > 1 ? blockIdx.x / KS : blockIdx.x;
  const long ncl = KS > 1 ? gridDim.x / KS : gridDim.x;
  const int ks0 = (ktiles * crank) / KS, ks1 = (ktiles * (crank + 1)) / KS;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    // full: the TMA issuer's expect_tx arrive (and the copies' bytes) + the scale warp's 32 lanes
    for (int s = 0; s < kNS; ++s) { mbar_init(&full[s], 1 + 32); mbar_init(&empty[s], 1); }
    for (int s = 0; s < 2; ++s) { mbar_init(&tfull[s], 1); mbar_init(&tempty[s], kEpiWarpsSw); }
    // an item is released by the TMA issuer, the scale warp, the MMA issuer and the epilogue warps
    for (int s = 0; s < kURing; ++s) {
      mbar_init(&ufull[s], 1);
      mbar_init(&uempty[s], 3 + kEpiWarpsSw);
      mbar_init(&rfull[s], 32);  // one cp.async-tracking arrival per scheduler lane
    }
    for (int s = 0; s < kSfRing; ++s) mbar_init(&sfempty[s], 1);
    mbar_init(drain, 1);
    if (KS > 1)
      for (int q = 0; q < 4; ++q) {
        mbar_init(&red_full[q], KS - 1);
        mbar_init(&red_empty[q], 1);
      }
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
  if (KS > 1) cluster_sync();  // every CTA's barriers are initialised before any remote arrive
  const uint32_t tbase = *tmem_slot;
  // everything above overlapped the previous kernel's tail; its results are read from here on
  pdl_wait();
  pdl_launch_dependents();

  if (warp == 3) {
    // ------------------------------ item scheduler ------------------------------
    // Units u = blockIdx.x + k * gridDim.x, unit = (active expert u / ntn, tile u % ntn);
    // {expert, count, first row} of 32 units are fetched at once, one batch ahead.
    const int nunits = p.meta[META_NUM_ACTIVE] * ntn;
    int it = 0;
    bool done = false;
    long base = cid;
    long u = base + (long)lane * ncl;
    int4 info = u < nunits ? p.active_info[u / ntn] : make_int4(-1, 0, 0, 0);
    while (!done) {
      const int4 cur = info;
      const long cbase = base;
      base += 32L * ncl;
      u = base + (long)lane * ncl;
      info = u < nunits ? p.active_info[u / ntn] : make_int4(-1, 0, 0, 0);  // next batch, in flight
      for (int l = 0; l < 32 && !done; ++l) {
        const long ul = cbase + (long)l * ncl;
        const int el = __shfl_sync(0xFFFFFFFFu, cur.x, l);
        const int cl = __shfl_sync(0xFFFFFFFFu, cur.y, l);
        const int ol = __shfl_sync(0xFFFFFFFFu, cur.z, l);
        const bool more = ul < nunits;
        const int nch = more ? (cl + NMAX - 1) / NMAX : 1;
        for (int ch = 0; ch < nch; ++ch, ++it) {
          const int us = it % kURing;
          if (!warp_wait(&uempty[us], ((it / kURing) & 1) ^ 1, p.err, &abort_flag)) { done = true; break; }
          if (lane == 0) {
            UItem* ui = items + us;
            ui->e = el;
            ui->tile = more ? (int)(ul % ntn) : 0;
            ui->row0 = ol + ch * NMAX;
            ui->nrows = more ? min(NMAX, cl - ch * NMAX) : -1;
            mbar_arrive(&ufull[us]);
          }
          __syncwarp();
          if (!more) {
            // a second end marker: at stage 2 the two epilogue warpgroups take
            // alternate items and each must meet one
            const int ue = (it + 1) % kURing;
            if (warp_wait(&uempty[ue], (((it + 1) / kURing) & 1) ^ 1, p.err, &abort_flag) && lane == 0) {
              items[ue].nrows = -1;
              mbar_arrive(&ufull[ue]);
            }
            __syncwarp();
            done = true;
            break;
          }
          if (STAGE == 2) {
            // token and top-k weight of the item's rows, copied into the slot while
            // the item waits in the ring (only the epilogue reads them)
            const int r0 = ol + ch * NMAX, nr = min(NMAX, cl - ch * NMAX);
            int* rt = reinterpret_cast<int*>(smem + L::rows + us * L::row_bytes);
            float* rw = reinterpret_cast<float*>(rt + NMAX);
            for (int n = lane; n < nr; n += 32) {
              cp_async4(rt + n, p.row_tok + r0 + n);
              cp_async4(rw + n, p.row_w + r0 + n);
            }
            cp_async_arrive_noinc(&rfull[us]);
          }
        }
      }
    }
    cp_async_wait<0>();  // this warp's row-token copies have landed before the CTA may exit
  } else if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    // At the start of each item the weight-scale rows of the next item are
    // prefetched into L2, ahead of the scale warp's 4-byte copies.
    if (lane == 0) {
      tma_prefetch_desc(&tm_w);
      tma_prefetch_desc(&tm_x);
      const int sb_w = kdim / 32;
      // Scale rows (weights and the item's sub-rows) are prefetched into L2 kPfAhead
      // items ahead, so the scale warp's 4-byte copies do not pay the latency of
      // HBM under the weight stream: one long stage-1 item covers it, short
      // stage-2 items need several.
      constexpr int kPfAhead = STAGE == 2 ? 4 : 1;
      bool pf_end = false;
      auto prefetch_scales = [&](int j) {
        if (pf_end) return;
        const int un = j % kURing;
        if (!mbar_wait_or_abort(&ufull[un], (j / kURing) & 1, p.err, &abort_flag)) { pf_end = true; return; }
        const UItem nx = items[un];
        if (nx.nrows < 0) { pf_end = true; return; }  // no item is published past the end markers
        if (STAGE == 1) {
          const uint8_t* g = p.wscale + ((size_t)nx.e * 2 * I + (size_t)nx.tile * 128) * sb_w;
          bulk_prefetch_l2(g, 128u * sb_w);
          bulk_prefetch_l2(g + (size_t)I * sb_w, 128u * sb_w);
        } else if (PK) {  // the item's chunks: tiles 2 tile, 2 tile + 1, all K chunks, contiguous
          const int ht0 = 2 * nx.tile, nt = min(2, H / 128 - ht0), kcn = I / 128;
          bulk_prefetch_l2(p.wscale + ((size_t)nx.e * (H / 128) + ht0) * kcn * 512, (uint32_t)(nt * kcn * 512));
        } else {
          const int rows = min(256, H - nx.tile * 256);
          bulk_prefetch_l2(p.wscale + ((size_t)nx.e * H + (size_t)nx.tile * 256) * sb_w, (uint32_t)rows * sb_w);
        }
        const int nsub = nx.nrows * KD::kTerms;
        bulk_prefetch_l2(p.as + (size_t)nx.row0 * KD::kTerms * p.xs_stride, (uint32_t)(nsub * p.xs_stride));
      };
      for (int j = 0; j < kPfAhead; ++j) prefetch_scales(j);
      uint32_t stage = 0;
      int it = 0;
      bool ok = true;
      while (ok) {
        const int us = it % kURing;
        if (!mbar_wait_or_abort(&ufull[us], (it / kURing) & 1, p.err, &abort_flag)) break;
        const UItem ui = items[us];
        mbar_arrive_relaxed(&uempty[us]);
        ++it;
        if (ui.nrows < 0) break;
        prefetch_scales(it + kPfAhead - 1);
        const int nsub = ui.nrows * KD::kTerms;  // B rows: the item's sub-rows
        const int nbox = (nsub + 15) / 16;
        const uint32_t btx = (uint32_t)nbox * 16 * C::kRow;
        for (int ks = ks0; ks < ks1; ++ks, ++stage) {
          const int slot = stage % kNS;
          if (!mbar_wait_or_abort(&empty[slot], ((stage / kNS) & 1) ^ 1, p.err, &abort_flag)) { ok = false; break; }
          uint8_t* sa = smem + L::a + slot * L::a_bytes;
          uint8_t* sb = smem + L::b + slot * L::b_bytes;
          const int kx = ks * C::kXStep;
          if (PK) {
            // one contiguous 8 KB block per 128-row tile; a second tile past H (odd H / 128)
            // is not loaded (its rows are never stored). kind::mxf4: the block is stored
            // pre-swizzled, one bulk copy; kind::mxf8f6f4: the unpacking TMA.
            const int ht0 = 2 * ui.tile, kcn = I / 128;
            const bool two = ht0 + 1 < H / 128;
            mbar_arrive_expect_tx(&full[slot], (two ? 2 : 1) * w_tile_tx<KIND, STAGE>() + btx);
            const int y0 = ((ui.e * (H / 128) + ht0) * kcn + ks) * 128;
            if (KD::kMxf4) {
              bulk_g2s(sa, p.wpacked + (size_t)y0 * 64, 8192u, &full[slot]);
              if (two) bulk_g2s(sa + L::tile_bytes, p.wpacked + (size_t)(y0 + kcn * 128) * 64, 8192u, &full[slot]);
            } else {
              tma_load_2d_sw(sa, &tm_w, 0, y0, &full[slot]);
              if (two) tma_load_2d_sw(sa + L::tile_bytes, &tm_w, 0, y0 + kcn * 128, &full[slot]);
            }
          } else {
            mbar_arrive_expect_tx(&full[slot], 2 * w_tile_tx<KIND, STAGE>() + btx);
            if (STAGE == 1) {
              tma_load_4d(sa, &tm_w, kx, ui.tile * 128, 0, ui.e, &full[slot]);
              tma_load_4d(sa + L::tile_bytes, &tm_w, kx, ui.tile * 128, 1, ui.e, &full[slot]);
            } else {  // rows past H (odd H / 128) are filled with zeros
              tma_load_3d(sa, &tm_w, kx, ui.tile * 256, ui.e, &full[slot]);
              tma_load_3d(sa + L::tile_bytes, &tm_w, kx, ui.tile * 256 + 128, ui.e, &full[slot]);
            }
          }
          // routed rows: contiguous sub-rows [row0 * kTerms, (row0 + nrows) * kTerms), 16-row boxes
          // (rows past this expert belong to later experts and only fill unused columns)
          for (int bx = 0; bx < nbox; ++bx)
            tma_load_2d_sw(sb + bx * 16 * C::kRow, &tm_x, kx, ui.row0 * KD::kTerms + 16 * bx, &full[slot]);
        }
      }
      // every copy this thread started has landed before the CTA may exit (after an
      // abort nobody else waits for them): in a normal run these phases completed long
      // ago; after an abort the bounded wait outlasts any copy in flight
      for (uint32_t g = stage > (uint32_t)kNS ? stage - kNS : 0u; g < stage; ++g)
        mbar_wait(&full[g % kNS], (g / kNS) & 1, p.err);
    }
  } else if (warp == 1) {
    // ---------- e8m0 scales of both operands into tcgen05.cp chunks ----------
    // Stage g's chunks go to scale slot g % kSfRing (freed by the MMA of stage
    // g - kSfRing); warp 1 arrives on the operand slot's full barrier kSfLag stages
    // later, once its copies have landed, after checking that the operand slot
    // has been re-armed for that stage.
    const int sb_w = kdim / 32;  // weight-scale bytes per row
    uint32_t stage = 0, pend = 0;
    int it = 0;
    bool ok = true;
    auto arrive_oldest = [&]() {
      const uint32_t g = stage - pend;
      // the operand slot of stage g is in g's phase once the MMA released stage g - kNS
      ok = ok && warp_wait(&empty[g % kNS], ((g / kNS) & 1) ^ 1, p.err, &abort_flag);
      mbar_arrive(&full[g % kNS]);
      --pend;
    };
    while (ok) {
      const int us = it % kURing;
      if (!warp_wait(&ufull[us], (it / kURing) & 1, p.err, &abort_flag)) break;
      const UItem ui = items[us];
      __syncwarp();
      if (lane == 0) mbar_arrive_relaxed(&uempty[us]);
      ++it;
      if (ui.nrows < 0) break;
      const int nsub = ui.nrows * KD::kTerms;
      const size_t sub0 = (size_t)ui.row0 * KD::kTerms;
      // first row of tile 0; tile 1 is I rows further (up rows) in stage 1, 128 rows in stage 2
      const uint8_t* wsrc = STAGE == 1 ? p.wscale + ((size_t)ui.e * 2 * I + (size_t)ui.tile * 128) * sb_w
                                       : p.wscale + ((size_t)ui.e * H + (size_t)ui.tile * 256) * sb_w;
      const size_t w1 = STAGE == 1 ? (size_t)I : 128;
      const bool t1 = STAGE == 1 || ui.tile * 256 + 128 < H;  // second tile inside the matrix
      for (int ks = ks0; ks < ks1 && ok; ++ks) {
        const int fslot = stage % kSfRing;
        if (!warp_wait(&sfempty[fslot], ((stage / kSfRing) & 1) ^ 1, p.err, &abort_flag)) { ok = false; break; }
        uint8_t* sf = smem + L::sf + fslot * L::sf_bytes;  // [sfa tile 0 | sfa tile 1 | sfb], sf_op bytes each
        for (int c = 0; c < C::kChunks; ++c) {
          const int kb0 = ks * C::kBlocks + 4 * c;
          if (kb0 < nblk_k) {  // kdim % 128 == 0: a chunk is all in or all out
            if (PK) {  // the chunk is stored as it lands: 16 bytes per lane
              const uint8_t* pk = p.wscale + ((size_t)ui.e * (H / 128) + 2 * ui.tile) * (I / 128) * 512 +
                                  (size_t)(kb0 / 4) * 512 + 16 * lane;
              cp_async16(sf + 512 * c + 16 * lane, pk);
              if (t1) cp_async16(sf + L::sf_op + 512 * c + 16 * lane, pk + (size_t)(I / 128) * 512);
            } else {
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int m = 4 * lane + i;
                cp_async4(sf + 512 * c + sf_off_sw(m), wsrc + (size_t)m * sb_w + kb0);
                if (t1) cp_async4(sf + L::sf_op + 512 * c + sf_off_sw(m), wsrc + (w1 + m) * sb_w + kb0);
              }
            }
            for (int n = lane; n < nsub; n += 32)
              cp_async4(sf + 2 * L::sf_op + 512 * c + sf_off_sw(n), p.as + (sub0 + n) * p.xs_stride + kb0);
          } else {  // past the end of K: neutral scales (the operands there are zero)
            const uint4 n127 = make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
            *reinterpret_cast<uint4*>(sf + 512 * c + 16 * lane) = n127;
            *reinterpret_cast<uint4*>(sf + L::sf_op + 512 * c + 16 * lane) = n127;
            *reinterpret_cast<uint4*>(sf + 2 * L::sf_op + 512 * c + 16 * lane) = n127;
          }
        }
        cp_async_commit();
        ++stage;
        ++pend;
        if (pend > kSfLag) {
          cp_async_wait<kSfLag>();
          fence_proxy_async();  // this thread's generic-proxy smem writes -> visible to tcgen05.cp
          arrive_oldest();
        }
      }
    }
    cp_async_wait<0>();
    fence_proxy_async();
    while (pend > 0 && ok) arrive_oldest();
  } else if (warp == 2) {
    // ------------------------------ MMA issuer ------------------------------
    // One thread; its instruction stream is on the critical path (a block-scaled
    // MMA takes ~100 cycles), so descriptors are formed once and advanced by adding
    // 16-byte-unit offsets to their start-address field, and the ring positions
    // are counters rather than divisions.
    if (lane == 0) {
      // K-major, swizzled: 8-row groups kRow * 8 bytes apart; a K step advances the
      // start address by 32 bytes inside the swizzle span
      const uint64_t dA0 = tc::sdesc(smem_u32(smem + L::a), 16, 8 * C::kRow, C::kSwz);
      const uint64_t dB0 = tc::sdesc(smem_u32(smem + L::b), 16, 8 * C::kRow, C::kSwz);
      const uint64_t dS0 = tc::sdesc(smem_u32(smem + L::sf), 0, 128, tc::SW_NONE);
      const uint32_t sf0 = tbase + sf_col0<KIND>();
      int slot = 0, fslot = 0;
      uint32_t phase = 0;
      int it = 0;
      while (true) {
        const int us = it % kURing;
        if (!mbar_wait_or_abort(&ufull[us], (it / kURing) & 1, p.err, &abort_flag)) break;
        const int nrows = items[us].nrows;
        mbar_arrive_relaxed(&uempty[us]);
        if (nrows < 0) break;
        const int buf = it & 1;
        ++it;
        if (!mbar_wait_or_abort(&tempty[buf], (((it - 1) >> 1) & 1) ^ 1, p.err, &abort_flag)) break;
        tc::fence_after();
        const int nmma = (nrows * KD::kTerms + 15) / 16 * 16;  // the item's sub-rows
        const uint32_t id0 = KD::kMxf4 ? tc::idesc_bs(128, nmma, tc::MXF4_E2M1, tc::MXF4_E2M1, 0, 0)
                                       : tc::idesc_bs(128, nmma, tc::F8F6F4_E2M1, tc::F8F6F4_E4M3, 0, 0);
        const uint32_t dg = tbase + buf * 2 * kAccCols;
        bool ok = true;
        for (int ks = ks0; ks < ks1; ++ks) {
          if (!mbar_wait_or_abort(&full[slot], phase, p.err, &abort_flag)) {
            ok = false;
            break;
          }
          tc::fence_after();
          constexpr uint32_t kOpCols = 4 * C::kChunks;  // TMEM columns of one operand's scale chunks
          const uint32_t sfc = sf0 + slot * C::kSfCols;  // sfa tile 0, sfa tile 1, sfb: kOpCols apart
          const uint64_t ds = dS0 + (uint64_t)((fslot * L::sf_bytes) >> 4);
          const int kleft = kdim - ks * C::kKTile;  // K of this tile inside the matrix (> 0)
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c) {
            if (c > 0 && 128 * c >= kleft) break;  // a chunk wholly past the end of K is not used
            tc::cp_32x128b_warpx4(sfc + 4 * c, ds + (512 * c >> 4));
            tc::cp_32x128b_warpx4(sfc + kOpCols + 4 * c, ds + ((L::sf_op + 512 * c) >> 4));
            tc::cp_32x128b_warpx4(sfc + 2 * kOpCols + 4 * c, ds + ((2 * L::sf_op + 512 * c) >> 4));
          }
          const uint64_t da = dA0 + (uint64_t)((slot * L::a_bytes) >> 4);
          const uint64_t db = dB0 + (uint64_t)((slot * L::b_bytes) >> 4);
#pragma unroll
          for (int i = 0; i < C::kKSteps; ++i) {
            if (i > 0 && i * (C::kKTile / C::kKSteps) >= kleft) break;  // K steps past the end of K
            const uint32_t acc = (ks > ks0 || i > 0) ? 1u : 0u;
#pragma unroll
            for (int g = 0; g < 2; ++g) {
              const uint64_t dai = da + ((g * L::tile_bytes + 32 * i) >> 4);
              const uint64_t dbi = db + ((32 * i) >> 4);
              if (KD::kMxf4) {  // scale_vec::2X: K block pair 2(i&1), 2(i&1)+1 of chunk i/2
                const uint32_t id = id0 | ((2u * (i & 1)) << 4) | ((2u * (i & 1)) << 29);
                tc::mma_mxf4(dg + g * kAccCols, dai, dbi, id, sfc + kOpCols * g + 4 * (i >> 1),
                             sfc + 2 * kOpCols + 4 * (i >> 1), acc);
              } else {
                const uint32_t id = id0 | ((uint32_t)i << 4) | ((uint32_t)i << 29);
                tc::mma_mxf8f6f4(dg + g * kAccCols, dai, dbi, id, sfc + kOpCols * g, sfc + 2 * kOpCols, acc);
              }
            }
          }
          tc::commit(&empty[slot]);
          tc::commit(&sfempty[fslot]);
          if (++slot == kNS) { slot = 0; phase ^= 1; }
          if (++fslot == kSfRing) fslot = 0;
        }
        if (!ok) break;
        tc::commit(&tfull[buf]);
      }
      // every MMA / copy this thread issued has finished before TMEM is released
      tc::commit(drain);
      mbar_wait(drain, 0, p.err);
    }
  } else if (warp >= 4 && (warp - 4) / kEpiWarpsSw < kEpiGroups) {
    // ------------------------------ epilogue ------------------------------
    // Stage 2: warpgroup wg (warps 4-7, 8-11) takes items wg, wg + 2, ... and so
    // accumulator buffer wg, so one warpgroup's TMEM loads overlap the other's
    // global reductions (its items are short). Stage 1 (long items) runs one
    // warpgroup over both buffers; warps 8-11 stay idle there.
    const int q = warp & 3;  // TMEM lane quadrant of this warp
    const int wg = (warp - 4) / kEpiWarpsSw;
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    int tok_a = 0, tok_b = 0;
    int red_cnt = 0;  // split-K: chunks exchanged so far (barrier phases)
    float w_a = 0.0f, w_b = 0.0f;
    int it = wg;
    while (true) {
      const int us = it % kURing;
      if (!warp_wait(&ufull[us], (it / kURing) & 1, p.err, &abort_flag)) break;
      const UItem ui = items[us];
      if (ui.nrows < 0) break;
      const int nrows = ui.nrows, row0 = ui.row0;
      __syncwarp();
      if (STAGE == 2) {
        // token and top-k weight of the item's rows (lanes n and 32 + n), staged in
        // the slot by the scheduler long before the item reaches the epilogue
        if (!warp_wait(&rfull[us], (it / kURing) & 1, p.err, &abort_flag)) break;
        const int* rt = reinterpret_cast<const int*>(smem + L::rows + us * L::row_bytes);
        const float* rw = reinterpret_cast<const float*>(rt + NMAX);
        tok_a = lane < nrows ? rt[lane] : 0;
        w_a = lane < nrows ? rw[lane] : 0.0f;
        if (NMAX > 32) {
          tok_b = 32 + lane < nrows ? rt[32 + lane] : 0;
          w_b = 32 + lane < nrows ? rw[32 + lane] : 0.0f;
        }
        // (the slot is released after the stores below, which consume these values)
      } else if (lane == 0) {
        mbar_arrive_relaxed(&uempty[us]);  // the item is in registers
      }
      const int buf = it & 1;
      if (!warp_wait(&tfull[buf], (it >> 1) & 1, p.err, &abort_flag)) break;
      it += kEpiGroups;  // (warp_wait reconverged the warp: tcgen05.ld is .sync.aligned)
      tc::fence_after();
      const uint32_t dg = tbase + lane_off + buf * 2 * kAccCols;
      // Values of item rows [c0, c0 + 16) of both accumulators: row n sums columns
      // n * kTerms + t (its code terms, in order of t); only the chunks of 16
      // columns in use are read, both accumulators' chunk under one wait.
      auto load_pair = [&](uint32_t acc0, uint32_t acc1, int c0, float* v0, float* v1) {
        const int nch = (min(16, nrows - c0) * KD::kTerms + 15) / 16;  // warp-uniform
#pragma unroll
        for (int n = 0; n < 16; ++n) { v0[n] = 0.0f; v1[n] = 0.0f; }
#pragma unroll
        for (int ch = 0; ch < KD::kTerms; ++ch) {  // 16 rows x kTerms columns = kTerms chunks of 16
          if (ch < nch) {
            uint32_t r0[16], r1[16];
            tc::ld_32x32b_x16(acc0 + c0 * KD::kTerms + 16 * ch, r0);
            tc::ld_32x32b_x16(acc1 + c0 * KD::kTerms + 16 * ch, r1);
            tc::ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int n = (16 * ch + j) / KD::kTerms;
              v0[n] += __uint_as_float(r0[j]);
              v1[n] += __uint_as_float(r1[j]);
            }
          }
        }
      };
      // after the item's last TMEM load the accumulator goes back to the MMA warp,
      // before this item's global stores (so the release does not wait for them)
      auto release_acc = [&](int c0) {
        if (c0 + 16 >= nrows) {
          tc::fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty[buf]);
        }
      };
      if (STAGE == 1) {
        const int j = ui.tile * 128 + 32 * q + lane;  // intermediate column of this lane
        // y = act(g, u) of item rows [c0, c0 + 16), requantised per 32 along I across the
        // warp (one out-of-line call per row keeps this rarely repeated code small)
        const ActK ak = act_consts(p.beta, p.lbeta);
        auto requant_rows = [&](int c0, const float* gv, const float* uv) {
          const int nn = min(16, nrows - c0);
#pragma unroll
          for (int n = 0; n < 16; ++n)
            if (n < nn)
              requant_row<KD::kTerms, KD::kMxf4>(act_apply<(KD::kTerms > 1)>(p.act, gv[n], uv[n], p.beta, p.lbeta, ak), row0 + c0 + n, j,
                                                 lane, I, p.oq, p.os, p.os_stride);
        };
        bool ok = true;
        for (int c0 = 0; c0 < nrows && ok; c0 += 16) {
          float gv[16], uv[16];
          load_pair(dg, dg + kAccCols, c0, gv, uv);
          release_acc(c0);
          if (KS > 1 && ks0 == ks1) {  // an empty K share (the host avoids it): a zero partial
#pragma unroll
            for (int n = 0; n < 16; ++n) { gv[n] = 0.0f; uv[n] = 0.0f; }
          }
          if (KS > 1) {
            const int nn = min(16, nrows - c0);
            // (n, column 32 q + lane) of rank r's partial sums: float2 at red + ((r-1) * 16 + n) * 1024 + 8 * col
            const uint32_t col8 = 8u * (32 * q + lane);
            if (crank != 0) {
              // the previous chunk's partial sums must have been read before this chunk overwrites them
              if (red_cnt > 0 && !warp_wait_cluster(&red_empty[q], (red_cnt - 1) & 1, p.err, &abort_flag)) {
                ok = false;
                break;
              }
              const uint32_t dst = mapa_shared(smem_u32(smem + L::red) + (uint32_t)(crank - 1) * 16 * 1024 + col8, 0);
#pragma unroll
              for (int n = 0; n < 16; ++n)
                if (n < nn) st_cluster_v2(dst + n * 1024, gv[n], uv[n]);
              __syncwarp();
              if (lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(&red_full[q]), 0));
              ++red_cnt;
              continue;  // rank 0 finishes the chunk
            }
            if (!warp_wait_cluster(&red_full[q], red_cnt & 1, p.err, &abort_flag)) {
              ok = false;
              break;
            }
#pragma unroll
            for (int r = 1; r < KS; ++r)
#pragma unroll
              for (int n = 0; n < 16; ++n)
                if (n < nn) {
                  const float2 v = *reinterpret_cast<const float2*>(smem + L::red + ((r - 1) * 16 + n) * 1024 + col8);
                  gv[n] += v.x;
                  uv[n] += v.y;
                }
            __syncwarp();
            if (lane == 0)
              for (int r = 1; r < KS; ++r) mbar_arrive_remote(mapa_shared(smem_u32(&red_empty[q]), r));
            ++red_cnt;
          }
          requant_rows(c0, gv, uv);
        }
        if (!ok) break;
      } else {
        const int h0 = ui.tile * 256 + 32 * q + lane;  // rows of H of this lane in tiles 0 and 1
        const bool h1ok = h0 + 128 < H;
        for (int c0 = 0; c0 < nrows; c0 += 16) {
          float v0[16], v1[16];
          load_pair(dg, dg + kAccCols, c0, v0, v1);
          release_acc(c0);
          const int nn = min(16, nrows - c0);
#pragma unroll
          for (int n = 0; n < 16; ++n) {
            if (n < nn) {
              const int col = c0 + n;  // warp-uniform
              const int t = __shfl_sync(0xFFFFFFFFu, col < 32 ? tok_a : tok_b, col & 31);
              const float w = __shfl_sync(0xFFFFFFFFu, col < 32 ? w_a : w_b, col & 31);
              float* dst = p.acc32 + (size_t)t * H + h0;
              atomicAdd(dst, w * v0[n]);
              if (h1ok) atomicAdd(dst + 128, w * v1[n]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_relaxed(&uempty[us]);  // the row values have been consumed
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (KS > 1) cluster_sync();  // no CTA leaves while a partner may still touch its shared memory
  if (warp == 2) {
    __syncwarp();
    tc::fence_after();
    tc::tmem_dealloc(tbase, kTmemColsSw);
  }
}

// ---------------------------------------------------------------------------
template <int KIND, int STAGE, bool PK, int KS>
static cudaError_t set_limit_one() {
  return cudaFuncSetAttribute(swap_stage_kernel<KIND, STAGE, PK, KS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)SwLayout<KIND, STAGE, KS>::total);
}

template <int KIND>
static cudaError_t set_limit_sw() {
  cudaError_t e = set_limit_one<KIND, 1, false, 1>();
  if (e == cudaSuccess) e = set_limit_one<KIND, 1, false, 2>();
  if (e == cudaSuccess) e = set_limit_one<KIND, 1, false, 3>();
  if (e == cudaSuccess) e = set_limit_one<KIND, 2, false, 1>();
  if (e == cudaSuccess) e = set_limit_one<KIND, 2, true, 1>();
  return e;
}

int swap_row_bytes(int kind, int stage) {
  if (kind == SW_A16) return stage == 1 ? SwCfg<SW_A16, 1>::kRow : SwCfg<SW_A16, 2>::kRow;
  if (kind == SW_A8) return stage == 1 ? SwCfg<SW_A8, 1>::kRow : SwCfg<SW_A8, 2>::kRow;
  return stage == 1 ? SwCfg<SW_A4, 1>::kRow : SwCfg<SW_A4, 2>::kRow;
}

cudaError_t swap_set_smem_limits() {
  cudaError_t e = set_limit_sw<SW_A16>();
  if (e == cudaSuccess) e = set_limit_sw<SW_A8>();
  if (e == cudaSuccess) e = set_limit_sw<SW_A4>();
  return e;
}

// Split-K launch: clusters of KS consecutive CTAs, with programmatic dependent launch.
template <int KIND, int KS>
static cudaError_t launch_split(const StageParams& p, const CUtensorMap& tm_w, const CUtensorMap& tm_x, int grid,
                                cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads_sw<1>());
  cfg.dynamicSmemBytes = SwLayout<KIND, 1, KS>::total;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = KS;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, swap_stage_kernel<KIND, 1, false, KS>, p, tm_w, tm_x);
}

template <int KIND>
static cudaError_t launch_sw(int stage, bool packed, int ks, const StageParams& p, const CUtensorMap& tm_w,
                             const CUtensorMap& tm_x, int grid, cudaStream_t st) {
  if (stage == 1) {
    if (ks == 3) return launch_split<KIND, 3>(p, tm_w, tm_x, grid, st);
    if (ks == 2) return launch_split<KIND, 2>(p, tm_w, tm_x, grid, st);
    return launch_k(swap_stage_kernel<KIND, 1, false, 1>, dim3(grid), dim3(threads_sw<1>()), SwLayout<KIND, 1>::total,
                    st, true, p, tm_w, tm_x);
  }
  if (packed)
    return launch_k(swap_stage_kernel<KIND, 2, true, 1>, dim3(grid), dim3(threads_sw<2>()), SwLayout<KIND, 2>::total, st,
                    true, p, tm_w, tm_x);
  return launch_k(swap_stage_kernel<KIND, 2, false, 1>, dim3(grid), dim3(threads_sw<2>()), SwLayout<KIND, 2>::total, st,
                  true, p, tm_w, tm_x);
}

template <int KIND, int KS>
static int max_clusters() {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(KS * 64);
  cfg.blockDim = dim3(threads_sw<1>());
  cfg.dynamicSmemBytes = SwLayout<KIND, 1, KS>::total;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = KS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, swap_stage_kernel<KIND, 1, false, KS>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

int swap_split_max_clusters(int kind, int ks) {
  if (kind == SW_A16) return ks == 3 ? max_clusters<SW_A16, 3>() : max_clusters<SW_A16, 2>();
  if (kind == SW_A8) return ks == 3 ? max_clusters<SW_A8, 3>() : max_clusters<SW_A8, 2>();
  return ks == 3 ? max_clusters<SW_A4, 3>() : max_clusters<SW_A4, 2>();
}

cudaError_t launch_swap_stage(int kind, int stage, bool packed, int ks, const StageParams& p, const CUtensorMap& tm_w,
                              const CUtensorMap& tm_x, int grid, cudaStream_t st) {
  if (kind == SW_A16) return launch_sw<SW_A16>(stage, packed, ks, p, tm_w, tm_x, grid, st);
  if (kind == SW_A8) return launch_sw<SW_A8>(stage, packed, ks, p, tm_w, tm_x, grid, st);
  return launch_sw<SW_A4>(stage, packed, ks, p, tm_w, tm_x, grid, st);
}

}  // namespace moe
