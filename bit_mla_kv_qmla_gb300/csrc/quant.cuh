// quant.cuh - the quantize-and-pack of one token (used by append.cu).
//
// The two quantizers of "QuantMLA: INT4 (and INT2) for both halves of the MLA
// cache" (flowchart: content quant INT4 or INT2, RoPE quant INT4): each
// token's 512-channel content latent and 64-channel RoPE key are cut into
// 64-channel groups, each stored as binary16 (scale, zero) plus packed
// integer codes.  Scale and zero lie on the group's binary16-exact grid and
// codes are rounded half to even, as specified in qmla.h; every step uses an
// explicitly rounded intrinsic, so the result is bit-exact and independent of
// compiler contraction.  One warp handles one group, each lane two
// consecutive channels.
#pragma once

#include "qmla_internal.cuh"

namespace qmla {
namespace quant {

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
// quantizer defines.  Warp uniform.  Every step is exact in binary32 and
// integer arithmetic (no binary64, which is slow here): mn and mx are
// bfloat16 values, so mn/u and mx/u (|.| <= 2^12 for E >= ilogb(m) - 11, m =
// max |x|, or a division by at most 32 at the top exponent) are binary32
// numbers -- bfloat16's 8 significant bits stay above binary32's subnormal
// granularity even after that division; Z is the floor of the scaled
// minimum; since Z is an integer, ceil(mx/u - Z) = ceil(mx/u) - Z = N >= 0
// (Z <= mn/u <= mx/u); and M = ceil(N / levels) is an integer division.
__device__ __forceinline__ void group_grid(float mn, float mx, int levels, float& s, float& z) {
  // start: a lower bound on the exponent found (the difference rounded down)
  const float d = __fsub_rd(mx, mn);
  int E = (d > 0.0f) ? max(-24, ilogbf(d) - 12) : -24;
  // No E below ilogb(m) - 11 can pass: u <= m/4096 puts |Z| or Z + levels*M
  // (>= mx/u) above 2047.  Starting there skips those iterations and finds
  // the same E.
  const float m = fmaxf(fabsf(mn), fabsf(mx));
  if (m > 0.0f) E = max(E, min(ilogbf(m) - 11, 5));
  for (;; ++E) {
    const float inv_u = __int_as_float((127 - E) << 23);  // 2^-E, a normal number
    const float a_mn = mn * inv_u, a_mx = mx * inv_u;     // exact
    // magnitudes beyond 2^29 fail the bounds below anyway; clamp before the
    // integer conversions so that N stays an int
    const int Z = int(fminf(fmaxf(floorf(a_mn), -536870912.0f), 536870912.0f));
    const int C = int(fminf(fmaxf(ceilf(a_mx), -536870912.0f), 536870912.0f));
    const int N = C - Z;  // = ceil(mx/u - Z) while unclamped
    int M = (N + levels - 1) / levels;
    if (M < 1) M = 1;
    const bool ok = (Z >= -2047 && Z <= 2047) && (int64_t(Z) + int64_t(levels) * M <= 2047);
    if (ok || E >= 5) {
      int Zc = Z, Mc = M;
      if (!ok) {  // outside the |x| < 32768 precondition: clamp into range
        Zc = Z < -2047 ? -2047 : (Z > 2047 ? 2047 : Z);
        const int mmax = (2047 - Zc) / levels;
        Mc = M > mmax ? mmax : M;
        if (Mc < 1) Mc = 1;
      }
      const float u = __int_as_float((127 + E) << 23);  // 2^E
      z = float(Zc) * u;  // exact
      s = float(Mc) * u;  // exact
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

// One warp quantizes and stores group g of a token (g 0-7: content groups,
// 8: the RoPE key, INT4 or INT2 by format) at slot `slot` of block `blk`;
// lane holds the group's channels 2*lane and 2*lane+1 in v.
__device__ __forceinline__ void store_group(int fmt, uint8_t* blk, int slot, int g,
                                            __nv_bfloat162 v, int lane) {
  const Geom G = geom(fmt);
  if (fmt == QMLA_BF16) {
    uint8_t* dst;
    if (g < 8) {
      const int h = g / 4, gi = g % 4;
      dst = blk + h * G.half + G.content_off + (gi * kT + slot) * 128 + lane * 4;
    } else {
      const int h = lane / 16;  // lane holds RoPE channels 2*lane, 2*lane+1
      dst = blk + h * G.half + G.rope_off + slot * 64 + (lane % 16) * 4;
    }
    *reinterpret_cast<__nv_bfloat162*>(dst) = v;
    return;
  }
  const float x0 = __bfloat162float(v.x), x1 = __bfloat162float(v.y);
  const int bits = (g < 8) ? G.cbits : G.rbits;
  uint32_t c0, c1;
  uint16_t s_bits, z_bits;
  quantize_pair(x0, x1, bits, c0, c1, s_bits, z_bits);
  const uint32_t word = pack_word(c0, c1, bits, lane);
  const int per_word_lanes = 16 / bits;  // lanes per 32-bit word
  const int w = lane / per_word_lanes;
  const uint32_t sz = uint32_t(s_bits) | (uint32_t(z_bits) << 16);
  if (g < 8) {
    const int h = g / 4, gi = g % 4;
    uint8_t* half = blk + h * G.half;
    if (lane % per_word_lanes == 0)
      reinterpret_cast<uint32_t*>(half + G.content_off + (gi * kT + slot) * G.code_bytes)[w] = word;
    if (lane == 0) reinterpret_cast<uint32_t*>(half + G.sz_off + (gi * kT + slot) * 4)[0] = sz;
  } else {
    // RoPE: 8 words of 8 channels (INT4) or 4 of 16 (INT2); the first half
    // of the words (channels 0-31) goes to block half 0, the rest to half 1
    if (lane % per_word_lanes == 0) {
      const int words_per_half = bits;  // 32 channels / (32 / bits)
      const int h = w / words_per_half;
      reinterpret_cast<uint32_t*>(blk + h * G.half + G.rope_off + slot * G.rope_bytes)
          [w % words_per_half] = word;
    }
    if (lane == 0) reinterpret_cast<uint32_t*>(blk + G.rope_sz_off + slot * 4)[0] = sz;
  }
}

}  // namespace quant
}  // namespace qmla
