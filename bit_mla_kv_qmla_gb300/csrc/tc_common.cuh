// tc_common.cuh - pieces shared by the tensor-core decode kernels: the split
// planner, bounded waits, binary16 dequantization helpers and the swizzled
// shared-memory row store of the MMA operand tiles.
#pragma once

#include "plan.cuh"
#include "tc_ptx.cuh"

namespace qmla {
namespace tc {

using namespace ptx;

constexpr uint64_t kWaitNs = 1000000000ull;  // 1 s per wait

__device__ __forceinline__ bool wait_noabort(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer() - t0 > kWaitNs) return false;
  return true;
}
// All lanes of the warp agree on the outcome of a wait, so that the warp stays
// converged for the warp-synchronous tensor-memory instructions that follow.
__device__ __forceinline__ bool warp_ok(bool v) { return __all_sync(0xffffffffu, v); }

// Binary16 of a small integer field without a shift: OR the field, sitting
// at its bit position p inside each half-word, into the mantissa of 2^(10+p)
// ("magic" exponent), so that the value reads 2^(10+p) + field; subtracting
// 2^(10+p) leaves the field exactly.  Fields at bit 10 and above would reach
// the exponent, so those come from the word shifted right once.
__device__ __forceinline__ __half2 field_h2(uint32_t w, uint32_t mask, uint16_t magic) {
  const uint32_t mm = uint32_t(magic) * 0x10001u;
  const uint32_t v = (w & mask) | mm;
  return __hsub2(*reinterpret_cast<const __half2*>(&v),
                 *reinterpret_cast<const __half2*>(&mm));
}
// Four pairs of binary16 values (channels 2k, 2k+1) from 8 INT4 codes packed
// even-low / odd-high: x = code * s + z (exact on the quantizer's grid).
__device__ __forceinline__ void dq_int4(uint32_t w, __half2 s2, __half2 z2, uint32_t* out) {
  const uint32_t w8 = w >> 8;
  const __half2 c[4] = {field_h2(w, 0x000F000Fu, 0x6400), field_h2(w, 0x00F000F0u, 0x5400),
                        field_h2(w8, 0x000F000Fu, 0x6400), field_h2(w8, 0x00F000F0u, 0x5400)};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const __half2 h = __hfma2(c[k], s2, z2);
    out[k] = *reinterpret_cast<const uint32_t*>(&h);
  }
}
// Eight pairs from 16 INT2 codes.
__device__ __forceinline__ void dq_int2(uint32_t w, __half2 s2, __half2 z2, uint32_t* out) {
  const uint32_t w10 = w >> 10;
  const __half2 c[8] = {field_h2(w, 0x00030003u, 0x6400),   field_h2(w, 0x000C000Cu, 0x5C00),
                        field_h2(w, 0x00300030u, 0x5400),   field_h2(w, 0x00C000C0u, 0x4C00),
                        field_h2(w, 0x03000300u, 0x4400),   field_h2(w10, 0x00030003u, 0x6400),
                        field_h2(w10, 0x000C000Cu, 0x5C00), field_h2(w10, 0x00300030u, 0x5400)};
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const __half2 h = __hfma2(c[k], s2, z2);
    out[k] = *reinterpret_cast<const uint32_t*>(&h);
  }
}
__device__ __forceinline__ void split_sz(uint32_t sz, __half2& s2, __half2& z2) {
  const __half s = __ushort_as_half(uint16_t(sz & 0xffffu));
  const __half z = __ushort_as_half(uint16_t(sz >> 16));
  s2 = __halves2half2(s, s);
  z2 = __halves2half2(z, z);
}
// 16 channels (8 words) into row `row` of an SW128 [rows][64 fp16] region,
// logical 16-byte granules 2*seg and 2*seg+1.
__device__ __forceinline__ void st_row16(unsigned char* region, int row, int seg,
                                         const uint32_t* v) {
  unsigned char* r = region + (row >> 3) * 1024 + (row & 7) * 128;
  *reinterpret_cast<uint4*>(r + (((2 * seg) ^ (row & 7)) << 4)) =
      make_uint4(v[0], v[1], v[2], v[3]);
  *reinterpret_cast<uint4*>(r + (((2 * seg + 1) ^ (row & 7)) << 4)) =
      make_uint4(v[4], v[5], v[6], v[7]);
}

// Validity of blocks j0 .. j0+31 of sequence b as a bit mask (bit k: block
// j0+k exists in the piece and its id lies inside the pool).  One coalesced
// load per warp for 32 tiles keeps global-memory latency out of the per-tile
// path.  Called by a full warp.
__device__ __forceinline__ uint32_t valid_mask(const DecodeArgs& a, int b, int j0, int j1) {
  const int j = j0 + int(threadIdx.x & 31);
  bool ok = false;
  if (j < j1) {
    const int32_t blk = a.block_table[int64_t(b) * a.max_blocks_per_seq + j];
    ok = blk >= 0 && blk < a.num_blocks;
  }
  return __ballot_sync(0xffffffffu, ok);
}

}  // namespace tc

// Launch the one-warp planner that writes the split plan into the workspace.
cudaError_t launch_plan(const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_decode_tc16(const DecodeArgs& a, cudaStream_t stream);

}  // namespace qmla
