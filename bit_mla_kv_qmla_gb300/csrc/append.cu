// append.cu - quantize-and-pack of new tokens into the paged low-bit cache.
//
// The two quantizers of "QuantMLA: INT4 (and INT2) for both halves of the MLA
// cache" (flowchart: content quant INT4 or INT2, RoPE quant INT4): each token's
// 512-channel content latent and 64-channel RoPE key are cut into 64-channel
// groups, each stored as binary16 (scale, zero) plus packed integer codes.
// Scale and zero lie on the group's binary16-exact grid and codes are rounded
// half to even, as specified in qmla.h; every step uses an explicitly rounded
// intrinsic, so the result is bit-exact and independent of compiler
// contraction.
//
// One CTA per new token, one warp per 64-channel group (8 content + 1 RoPE),
// each lane holding two consecutive channels.  The whole append is one pass
// over the new tokens: it is launch-bound for decode-sized appends.

#include "qmla_internal.cuh"

namespace qmla {
namespace {

__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Scale and zero of a group on its binary16-exact grid: the smallest power of
// two u = 2^E (E in [-24, 5]) with integers Z = floor(mn/u) and
// M = max(1, ceil((mx - Z*u) / (levels*u))) such that |Z| <= 2047 and
// |Z + levels*M| <= 2047.  Every dequantized value (Z + c*M)*u is then exactly
// a binary16 number, so the tensor cores multiply exactly the value the
// quantizer defines.  Warp uniform.  Every step is exact, so no rounding mode
// matters and no binary64 division is needed: mn and mx (bfloat16 values)
// scale by 2^-E exactly in binary64, Z is the floor of the scaled minimum,
// N = mx/u - Z is an exact binary64 difference (N >= 0 since Z <= mn/u <=
// mx/u), and M = ceil(N / levels) = ceil(ceil(N) / levels) is an integer
// division.
__device__ __forceinline__ void group_grid(float mn, float mx, int levels, float& s, float& z) {
  const double d = double(mx) - double(mn);  // exact
  int E = (d > 0.0) ? max(-24, ilogb(d) - 12) : -24;
  for (;; ++E) {
    const double a_mn = ldexp(double(mn), -E), a_mx = ldexp(double(mx), -E);  // exact
    const double Zd = floor(a_mn);
    // |Z| and N beyond 2^40 fail the bounds below anyway; clamp before the
    // integer conversion
    const int64_t Z = int64_t(fmin(fmax(Zd, -1099511627776.0), 1099511627776.0));
    const double N = fmin(a_mx - Zd, 1099511627776.0);  // exact below the clamp
    int64_t M = (int64_t(ceil(N)) + levels - 1) / levels;
    if (M < 1) M = 1;
    const bool ok = (Z >= -2047 && Z <= 2047) && (Z + levels * M <= 2047);
    if (ok || E >= 5) {
      int64_t Zc = Z, Mc = M;
      if (!ok) {  // outside the |x| < 32768 precondition: clamp into range
        Zc = Z < -2047 ? -2047 : (Z > 2047 ? 2047 : Z);
        const int64_t mmax = (2047 - Zc) / levels;
        Mc = M > mmax ? mmax : M;
        if (Mc < 1) Mc = 1;
      }
      z = ldexpf(float(Zc), E);  // exact
      s = ldexpf(float(Mc), E);  // exact
      return;
    }
  }
}

// Quantize the warp's group; lane holds channels 2*lane and 2*lane+1 (x0, x1).
// Returns the two codes and (scale, zero) as binary16 bits.
__device__ __forceinline__ void quantize_pair(float x0, float x1, int bits, uint32_t& c0,
                                              uint32_t& c1, uint16_t& s_bits,
                                              uint16_t& z_bits) {
  const float mn = warp_min(fminf(x0, x1));
  const float mx = warp_max(fmaxf(x0, x1));
  const int levels = (1 << bits) - 1;
  float sf, zf;
  group_grid(mn, mx, levels, sf, zf);
  s_bits = __half_as_ushort(__float2half_rn(sf));
  z_bits = __half_as_ushort(__float2half_rn(zf));
  const float lv = float(levels);
  const float t0 = rintf(__fdiv_rn(__fsub_rn(x0, zf), sf));
  const float t1 = rintf(__fdiv_rn(__fsub_rn(x1, zf), sf));
  c0 = uint32_t(fminf(fmaxf(t0, 0.0f), lv));
  c1 = uint32_t(fminf(fmaxf(t1, 0.0f), lv));
}

// Pack: the lane's even channel goes to position j of the low half-word, its
// odd channel to position j of the high half-word, j = lane % (codes per
// half-word); OR-reduce across the lanes sharing a word.
__device__ __forceinline__ uint32_t pack_word(uint32_t c0, uint32_t c1, int bits, int lane) {
  const int per_half = 16 / bits;  // 4 (INT4) or 8 (INT2) lanes share a word
  const int j = lane % per_half;
  uint32_t w = (c0 << (bits * j)) | (c1 << (16 + bits * j));
  for (int o = 1; o < per_half; o <<= 1) w |= __shfl_xor_sync(0xffffffffu, w, o);
  return w;
}

// `advance` (one new token per sequence only): the CTA of sequence b also
// adds 1 to positions[b] once all of its threads have read it.
__global__ void __launch_bounds__(288) append_kernel(
    int fmt, uint8_t* __restrict__ blocks, int64_t num_blocks, const int32_t* __restrict__ table,
    int max_blocks, int32_t* positions, int n_new, const __nv_bfloat16* __restrict__ latent,
    const __nv_bfloat16* __restrict__ rope, int32_t* status, bool advance) {
  // a decode launched after this kernel as a programmatic dependent may start
  // its prologue now (it waits for this grid before reading anything)
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tok = blockIdx.x;  // b * n_new + i
  const int b = tok / n_new, i = tok % n_new;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the lane's two channels of this warp's group (issued first: independent
  // of the block-table lookups below)
  __nv_bfloat162 v;
  if (warp < 8) {
    v = reinterpret_cast<const __nv_bfloat162*>(latent + int64_t(tok) * kDc + warp * kG)[lane];
  } else {
    v = reinterpret_cast<const __nv_bfloat162*>(rope + int64_t(tok) * kDr)[lane];
  }
  const int64_t pos = int64_t(positions[b]) + i;
  if (advance) {
    __syncthreads();  // every thread has read positions[b]
    if (threadIdx.x == 0) positions[b] = int32_t(pos + 1);
  }
  const int64_t jb = pos / kT;
  if (pos < 0 || jb >= max_blocks) {
    if (threadIdx.x == 0) set_status(status, QMLA_STATUS_BAD_LEN);
    return;
  }
  const int32_t blk_id = table[int64_t(b) * max_blocks + jb];
  if (blk_id < 0 || blk_id >= num_blocks) {
    if (threadIdx.x == 0) set_status(status, QMLA_STATUS_BAD_BLOCK);
    return;
  }
  const Geom G = geom(fmt);
  const int slot = int(pos % kT);
  uint8_t* blk = blocks + int64_t(blk_id) * G.block;


  if (fmt == QMLA_BF16) {
    uint8_t* dst;
    if (warp < 8) {
      const int h = warp / 4, gi = warp % 4;
      dst = blk + h * G.half + G.content_off + (gi * kT + slot) * 128 + lane * 4;
    } else {
      const int h = lane / 16;  // lane holds RoPE channels 2*lane, 2*lane+1
      dst = blk + h * G.half + G.rope_off + slot * 64 + (lane % 16) * 4;
    }
    *reinterpret_cast<__nv_bfloat162*>(dst) = v;
    return;
  }

  const float x0 = __bfloat162float(v.x), x1 = __bfloat162float(v.y);
  const int bits = (warp < 8) ? G.cbits : 4;
  uint32_t c0, c1;
  uint16_t s_bits, z_bits;
  quantize_pair(x0, x1, bits, c0, c1, s_bits, z_bits);
  const uint32_t word = pack_word(c0, c1, bits, lane);
  const int per_word_lanes = 16 / bits;  // lanes per 32-bit word
  const int w = lane / per_word_lanes;
  const uint32_t sz = uint32_t(s_bits) | (uint32_t(z_bits) << 16);
  if (warp < 8) {
    const int h = warp / 4, gi = warp % 4;
    uint8_t* half = blk + h * G.half;
    if (lane % per_word_lanes == 0)
      reinterpret_cast<uint32_t*>(half + G.content_off + (gi * kT + slot) * G.code_bytes)[w] = word;
    if (lane == 0) reinterpret_cast<uint32_t*>(half + G.sz_off + (gi * kT + slot) * 4)[0] = sz;
  } else {
    // RoPE: 8 words of 8 channels; words 0-3 -> half 0, words 4-7 -> half 1
    if (lane % 4 == 0) {
      const int h = w / 4;
      reinterpret_cast<uint32_t*>(blk + h * G.half + G.rope_off + slot * 16)[w % 4] = word;
    }
    if (lane == 0) reinterpret_cast<uint32_t*>(blk + G.rope_sz_off + slot * 4)[0] = sz;
  }
}

}  // namespace

__global__ void advance_kernel(int32_t* positions, int batch, int n_new) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < batch) positions[b] += n_new;
}

cudaError_t launch_append(int fmt, uint8_t* blocks, int64_t num_blocks, const int32_t* table,
                          int max_blocks, int32_t* positions, int batch, int n_new,
                          const __nv_bfloat16* latent, const __nv_bfloat16* rope,
                          int32_t* status, bool advance, cudaStream_t stream) {
  const int64_t ntok = int64_t(batch) * n_new;
  if (ntok == 0) return cudaSuccess;
  // one token per sequence: the append CTA advances its own position;
  // several: a second kernel does, after every CTA has read the positions
  const bool fused = advance && n_new == 1;
  append_kernel<<<dim3(unsigned(ntok)), 288, 0, stream>>>(
      fmt, blocks, num_blocks, table, max_blocks, positions, n_new, latent, rope, status, fused);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || !advance || fused) return e;
  advance_kernel<<<dim3(unsigned((batch + 255) / 256)), 256, 0, stream>>>(positions, batch, n_new);
  return cudaGetLastError();
}

}  // namespace qmla
