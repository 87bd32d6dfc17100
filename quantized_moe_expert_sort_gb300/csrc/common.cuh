// Device helpers shared by the MoE kernels (sm_103a).
//
// Formats follow the OCP MX definitions used on the aiter pages ("Add an opt-in
// a4w4 SiTUv2 MoE path...", Three tuner defects item 2: fp4x2 packs two e2m1
// codes per byte; "Add Kimi-K3 A8W4 support...", Technical Details: fp8 1x32
// block scales). Quantised activations are "block-scaled codes": a code array
// plus one e8m0 scale per 32 elements along K, with codes in one of the formats:
//   FMT_E4M3 : fp8 e4m3fn (a8 path)
//   FMT_E2M1 : fp4 e2m1, two per byte, element 2j in the low nibble (a4 path;
//              also the code terms that carry bf16 values on the a16 path)
//   FMT_F16  : IEEE half times one power of two per token: the bf16 mode of the
//              stand-alone activation quantiser (moe_quantize_activations) only;
//              the forward pass does not use it
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda.h>

namespace moe {

enum ActFmt : int { FMT_F16 = 0, FMT_E4M3 = 1, FMT_E2M1 = 2 };
enum Act : int { ACT_SILU = 0, ACT_SITUV2 = 1 };

// Device error word bits (read back by moe_get_error).
enum : int {
  DEV_ERR_BAD_EXPERT = 1,   // a routed expert id was outside [0, E); the pair was dropped
  DEV_ERR_TIMEOUT = 2,      // a bounded wait ran out; the kernel returned early
  DEV_ERR_OVERFLOW = 4,     // sorted rows would exceed the workspace; extra rows dropped
  DEV_ERR_LAUNCH = 8,       // a kernel got less shared memory than its layout needs; it returned at once
};

// Programmatic dependent launch: wait for the previous kernel in the stream (a
// no-op when launched without the attribute), and let the next one start.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void set_error(int* err, int bit) {
  if (err) atomicOr(err, bit);
}

// ---------------------------------------------------------------------------
// Scale and element formats
// ---------------------------------------------------------------------------

// e8m0 byte -> 2^(s-127) as fp32 (s = 0 is the fp32 subnormal 2^-127).
__device__ __forceinline__ float e8m0_to_f32(uint32_t s) {
  uint32_t bits = (s == 0u) ? 0x00400000u : (s == 255u ? 0x7FC00000u : (s << 23));
  return __uint_as_float(bits);
}

// floor(log2(a)) for a finite a > 0, exact, from the fp32 bits.
__device__ __forceinline__ int floor_log2_f32(float a) {
  uint32_t b = __float_as_uint(a);
  int ef = (int)((b >> 23) & 0xFFu);
  if (ef) return ef - 127;
  return (31 - __clz((int)(b & 0x7FFFFFu))) - 149;
}

// 2^-E as fp32 for E in [-127, 127] (exact).
__device__ __forceinline__ float exp2_neg(int E) {
  int f = 127 - E;  // in [0, 254]
  return __uint_as_float(f == 0 ? 0x00400000u : ((uint32_t)f << 23));
}

// Largest normal exponent of each element format: the MX scale rule sets
// E = floor(log2(amax)) - emax so that the block maximum lands in the top binade.
__device__ __forceinline__ int fmt_emax(int fmt) { return fmt == FMT_E2M1 ? 2 : (fmt == FMT_E4M3 ? 8 : 15); }

// Two fp32 -> packed e2m1x2 (RNE, saturating). lo -> low nibble, hi -> high nibble.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint32_t out;
  asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n mov.b32 %0, {t, t, t, t};\n}"
      : "=r"(out) : "f"(hi), "f"(lo));
  return out & 0xFFu;
}

// Two fp32 -> packed e4m3x2 (RNE, saturating). lo -> low byte, hi -> high byte.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t out;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(out) : "f"(hi), "f"(lo));
  return (uint32_t)out;
}

// One e2m1 code (low nibble) -> its value as fp32 (exact).
__device__ __forceinline__ float e2m1_to_f32(uint32_t code) {
  uint32_t h;
  asm("{\n .reg .b8 t;\n cvt.u8.u32 t, %1;\n cvt.rn.f16x2.e2m1x2 %0, t;\n}" : "=r"(h) : "r"(code & 0xFu));
  return __half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu)));
}

// ---------------------------------------------------------------------------
// Activation functions (aiter PR 6259 Motivation, PR 4471 Motivation)
// sigmoid(z) = 1 / (1 + 2^(-z * log2 e)) with the hardware exp2 and reciprocal
// (no cancellation: a few ulp).
// tanh: the int4 SiTUv2 page builds it as 2 * sigmoid(2z) - 1, which saturates to
// +-1 at both ends; in fp32 that difference cancels for small z (the sigmoid's
// ~1e-7 absolute error becomes ~4e-4 relative at the |u| / linear_beta of small
// activations). For |z| < 1/4 the odd Taylor series of tanh,
//   z - z^3/3 + 2 z^5/15 - 17 z^7/315 + 62 z^9/2835,
// is used instead (truncation below 2e-8 relative there); above 1/4 the
// cancellation costs at most ~2e-6 relative.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float fast_sigmoid(float z) {
  float e, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(-1.4426950408889634f * z));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + e));
  return r;
}

__device__ __forceinline__ float tanh_act(float z) {
  if (fabsf(z) < 0.25f) {
    const float z2 = z * z;
    float p = 62.0f / 2835.0f;
    p = fmaf(p, z2, -17.0f / 315.0f);
    p = fmaf(p, z2, 2.0f / 15.0f);
    p = fmaf(p, z2, -1.0f / 3.0f);
    return fmaf(z * z2, p, z);
  }
  return 2.0f * fast_sigmoid(2.0f * z) - 1.0f;
}

// Per-call constants of the activation: -2 log2(e) / beta, -2 log2(e) / lbeta and
// beta * lbeta (formed once per thread instead of two divisions per value).
struct ActK {
  float nb2, nlb2, blb;
};
__device__ __forceinline__ ActK act_consts(float beta, float lbeta) {
  return ActK{-2.0f * 1.4426950408889634f / beta, -2.0f * 1.4426950408889634f / lbeta, beta * lbeta};
}

// kAccurate: tanh_act (the bf16 intermediate of the a16 path keeps 8 bits of every
// value). Otherwise (fp8 / fp4 intermediates) tanh(z) = (1 - e^-2z) / (1 + e^-2z),
// whose worst relative error (~4e-4 at small z, from the cancellation) lies far
// inside the fp8 / fp4 steps the intermediate is requantised to, and the three
// factors of SiTUv2 share one reciprocal:
//   y = beta * lbeta * (1 - e1)(1 - e3) / ((1 + e1)(1 + e2)(1 + e3)),
//   e1 = e^(-2g/beta), e2 = e^(-g), e3 = e^(-2u/lbeta),
// three exp2 and one reciprocal per value. e1 and e3 are capped at 2^40 (tanh is
// -1 to within 2^-39 there) so that the denominator stays finite; sigmoid(g) for
// g < -27 is below what that form resolves and takes the per-factor form.
template <bool kAccurate = true>
__device__ __forceinline__ float act_apply(int act, float g, float u, float beta, float lbeta, const ActK& k) {
  if (act == ACT_SILU) return g * fast_sigmoid(g) * u;
  if (kAccurate) return beta * tanh_act(g / beta) * fast_sigmoid(g) * (lbeta * tanh_act(u / lbeta));
  if (g < -27.0f) {
    const float tg = 2.0f * fast_sigmoid(2.0f * g / beta) - 1.0f;
    const float tu = 2.0f * fast_sigmoid(2.0f * u / lbeta) - 1.0f;
    return beta * tg * fast_sigmoid(g) * (lbeta * tu);
  }
  float e1, e2, e3, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e1) : "f"(fminf(g * k.nb2, 40.0f)));
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e2) : "f"(-1.4426950408889634f * g));
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e3) : "f"(fminf(u * k.nlb2, 40.0f)));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"((1.0f + e1) * (1.0f + e2) * (1.0f + e3)));
  return k.blb * ((1.0f - e1) * (1.0f - e3)) * r;
}

// ---------------------------------------------------------------------------
// Warp and block helpers
// ---------------------------------------------------------------------------
// Block-wide exclusive scan of one int per thread (blockDim.x <= 1024).
__device__ __forceinline__ int block_exclusive_scan(int v, int* smem32, int* total) {
  int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) smem32[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? smem32[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xFFFFFFFFu, w, o);
      if (lane >= o) w += y;
    }
    smem32[lane] = w;  // inclusive prefix of warp sums
  }
  __syncthreads();
  int before = (warp > 0 ? smem32[warp - 1] : 0) + x - v;
  *total = smem32[nw - 1];
  __syncthreads();
  return before;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// Warp-cooperative 1x32 block quantisation: lane l holds element l of the block.
// Returns the lane's code in the low bits (f16 bits / e4m3 byte / e2m1 nibble)
// and the block's e8m0 scale byte in *scale. Rule: amax == 0 -> scale 127 and
// +0 codes; else E = floor(log2 amax) - emax (clamped to [-127,127]) and
// code = RNE(v * 2^-E), saturating.
__device__ __forceinline__ uint32_t block_quant_lane(float v, int fmt, uint32_t* scale) {
  float amax = warp_max(fabsf(v));
  if (amax == 0.0f) {
    *scale = 127u;
    return 0u;
  }
  int E = floor_log2_f32(amax) - fmt_emax(fmt);
  E = E < -127 ? -127 : (E > 127 ? 127 : E);
  *scale = (uint32_t)(E + 127);
  float q = __fmul_rn(v, exp2_neg(E));
  if (fmt == FMT_F16) return (uint32_t)__half_as_ushort(__float2half_rn(q));
  if (fmt == FMT_E4M3) return cvt_e4m3x2(q, 0.0f) & 0xFFu;
  return cvt_e2m1x2(q, 0.0f) & 0xFu;
}

// Store one lane's code of a quantised 32-block: bytes per element 2 (f16),
// 1 (e4m3) or 1/2 (e2m1, lanes pair up into bytes). dst points at the block.
__device__ __forceinline__ void block_store_lane(uint8_t* dst, uint32_t code, int fmt, int lane) {
  if (fmt == FMT_F16) {
    reinterpret_cast<uint16_t*>(dst)[lane] = (uint16_t)code;
  } else if (fmt == FMT_E4M3) {
    dst[lane] = (uint8_t)code;
  } else {
    uint32_t nb = __shfl_down_sync(0xFFFFFFFFu, code, 1);
    if ((lane & 1) == 0) dst[lane >> 1] = (uint8_t)(code | (nb << 4));
  }
}

__host__ __device__ __forceinline__ int fmt_bytes_per_32(int fmt) { return fmt == FMT_F16 ? 64 : (fmt == FMT_E4M3 ? 32 : 16); }

// ---------------------------------------------------------------------------
// mbarrier / TMA (inline PTX). Every wait is bounded: on timeout it records
// DEV_ERR_TIMEOUT and returns false, so no kernel can spin forever.
// ---------------------------------------------------------------------------
// Dynamic shared memory this launch was given (bytes).
__device__ __forceinline__ uint32_t dynamic_smem_bytes() {
  uint32_t n;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(n));
  return n;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}" :: "r"(smem_u32(bar)) : "memory");
}

// Arrive without release semantics: for barriers that only hand back a buffer
// whose contents this thread has finished reading (nothing it wrote is published).
__device__ __forceinline__ void mbar_arrive_relaxed(uint64_t* bar) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.relaxed.cta.shared::cta.b64 st, [%0];\n}" :: "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}"
               :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
               : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}

// try_wait that may suspend the thread in hardware until the phase completes or
// hint_ns have passed: a waiting warp takes no issue slots from the warps that
// share its scheduler, and wakes when the barrier completes.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
               : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns) : "memory");
  return ok != 0;
}

// Bounded waits. The pipelines hand each stage through two or three barriers,
// so a waiting thread must wake at once, and warps that wait must not steal
// issue slots from the TMA and MMA threads: each poll suspends in hardware
// (woken by the phase completing) for at most MOE_SUSPEND_NS. The bound is
// wall-clock (%globaltimer): MOE_WAIT_NS, 2 s by default.
#ifndef MOE_WAIT_NS
#define MOE_WAIT_NS 2000000000ull
#endif
#ifndef MOE_SUSPEND_NS
#define MOE_SUSPEND_NS 1000000u
#endif

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait with an explicit wall-clock limit (ns).
__device__ __forceinline__ bool mbar_wait_limit(uint64_t* bar, uint32_t parity, int* err, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    if (mbar_try_wait_suspend(bar, parity, MOE_SUSPEND_NS)) return true;
    if (global_ns() - t0 > limit_ns) break;
  }
  set_error(err, DEV_ERR_TIMEOUT);
  return false;
}

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* err) {
  return mbar_wait_limit(bar, parity, err, MOE_WAIT_NS);
}

// Wait that drains instead of hanging: once any thread of the CTA has timed
// out (*abort set), every later wait returns false at once, so all warps run
// to the end of their loops and the CTA exits.
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t* bar, uint32_t parity, int* err, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    if (mbar_try_wait_suspend(bar, parity, MOE_SUSPEND_NS)) return true;
    if (*abort) return false;
    if (global_ns() - t0 > MOE_WAIT_NS) break;
  }
  *abort = 1;
  set_error(err, DEV_ERR_TIMEOUT);
  return false;
}

// 1-D bulk copy global -> shared (16-byte aligned addresses, size % 16 == 0).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               :: "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* m, int x, int y, int z, uint64_t* bar) {
  asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
               :: "r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* m, int x, int y, int z, int w, uint64_t* bar) {
  asm volatile("cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];"
               :: "r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
               : "memory");
}


}  // namespace moe
