// Prepacked stage-2 weights for the few-rows kernels.
//
// The plain w2 layout [E, H, I/2] gives the stage-2 TMA 64-byte pieces of rows
// that lie I/2 bytes apart (K tile 128 = 64 bytes of a row), a pattern HBM
// serves well below its copy rate. The packed copy stores, for each expert e,
// 128-row tile ht of H and 128-element chunk kc of I, the tile's 128 rows of
// that chunk as one contiguous 8 KB block:
//   codes  byte ((((e * HT + ht) * KC + kc) * 128 + r) * 64 + j)
//          = w2[e, 128 * ht + r, 64 * kc + j]                     (HT = H/128, KC = I/128)
// and the e8m0 scales of that block as one 512-byte chunk in the layout the
// tensor-core scale copy reads (row r, 32-block b of the chunk):
//   scales byte (((e * HT + ht) * KC + kc) * 512 + 16 * (r % 32) + 4 * (r / 32) + b)
//          = w2_scale[e, 128 * ht + r, 4 * kc + b]
// With swz (the layout for the kind::mxf4 kernels), each block is stored as the
// shared-memory image those kernels read -- K-major rows of 64 bytes with the
// 64-byte swizzle: 16-byte chunk c of row r at chunk c ^ ((r / 2) % 4) -- so one
// 8 KB bulk copy lands it ready for the MMA. Without swz (kind::mxf8f6f4, which
// takes the codes through the unpacking TMA) rows are stored in order.
// The aiter pages keep the weights plain ("Add an opt-in a4w4 SiTUv2 MoE
// path...", Three tuner defects item 2 compares decoded values, never bytes);
// the packed copy is an addition, the plain layout stays the contract.
#include "common.cuh"
#include "kernels.h"

namespace moe {

__global__ void __launch_bounds__(256) prepack_w2_kernel(const uint8_t* __restrict__ w2, const uint8_t* __restrict__ w2s,
                                                         int E, int H, int I, int swz, uint8_t* __restrict__ pc,
                                                         uint8_t* __restrict__ ps) {
  const int HT = H / 128, KC = I / 128;
  const long nblk = (long)E * HT * KC;  // 8 KB code blocks = 512-byte scale chunks
  const long n16 = nblk * 512;          // 16-byte pieces of the packed codes
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n16 + nblk * 128; i += (long)gridDim.x * blockDim.x) {
    if (i < n16) {
      const long blk = i / 512;
      const int q = (int)(i % 512);      // piece within the block: row q / 4, bytes 16 * (q % 4)
      const int r = q / 4, j = 16 * (q % 4);
      const int kc = (int)(blk % KC);
      const long eh = blk / KC;          // e * HT + ht
      const long e = eh / HT, ht = eh % HT;
      const uint8_t* src = w2 + ((size_t)e * H + 128 * ht + r) * (I / 2) + 64 * kc + j;
      const int cdst = swz ? ((q % 4) ^ ((r >> 1) & 3)) : q % 4;  // destination 16-byte chunk of the row
      *reinterpret_cast<uint4*>(pc + ((size_t)blk * 128 + r) * 64 + 16 * cdst) = *reinterpret_cast<const uint4*>(src);
    } else {
      const long k = i - n16;            // one thread per (chunk, row): its 4 scale bytes
      const long blk = k / 128;
      const int r = (int)(k % 128);
      const int kc = (int)(blk % KC);
      const long eh = blk / KC;
      const long e = eh / HT, ht = eh % HT;
      const uint8_t* src = w2s + ((size_t)e * H + 128 * ht + r) * (I / 32) + 4 * kc;
      uint8_t* dst = ps + (size_t)blk * 512 + 16 * (r % 32) + 4 * (r / 32);
      *reinterpret_cast<uint32_t*>(dst) = *reinterpret_cast<const uint32_t*>(src);
    }
  }
}

cudaError_t launch_prepack_w2(const uint8_t* w2, const uint8_t* w2s, int E, int H, int I, int swz, uint8_t* pc,
                              uint8_t* ps, int num_sms, cudaStream_t st) {
  const long work = (long)E * (H / 128) * (I / 128) * (512 + 128);
  long blocks = (work + 255) / 256;
  const long cap = (long)num_sms * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  prepack_w2_kernel<<<(unsigned)blocks, 256, 0, st>>>(w2, w2s, E, H, I, swz, pc, ps);
  return cudaGetLastError();
}

}  // namespace moe
