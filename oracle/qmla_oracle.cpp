// qmla_oracle.cpp - CPU oracle for the low-bit MLA cache write and decode.
//
// TEST INFRASTRUCTURE ONLY.  This file is the slow, plain restatement of what
// the library computes, used to check the CUDA path.  Only the test suite, the
// smoke check and the CPU-baseline leg of the benchmark may load it; the
// library itself never does.  It shares no code, header, table or constant
// generator with the CUDA path: the block layout and rounding rules are
// re-derived here from their written specification.
//
// What it follows:
//  * "QuantMLA: INT4 (and INT2) for both halves of the MLA cache" (TL;DR and
//    mermaid flowchart): each token stores a content latent and a decoupled
//    RoPE key; content is quantized to INT4 or INT2, the RoPE key to INT4;
//    dequantization happens inside attention.
//  * Same page, "Key findings": generic quantizers treat the content latent
//    and the RoPE key as one tensor with one bit width.  The formats C4R2
//    and C2R2 (RoPE key at INT2, the same 64-channel groups and grid) are
//    that comparison: the RoPE codes shrink from 16 to 8 bytes per token and
//    block half, everything else keeps its place.
//  * Same page, "Key findings": the learned transforms are folded into the
//    weights offline, so inputs here are already transformed.
//  * Parameters the pages leave open, fixed by this library: 64-channel
//    groups, asymmetric quantization with binary16 scale and zero per
//    (token, group), 64-token cache blocks, absorbed-query decode
//    s_t = (q_c . c_t + q_r . k_t) * scale, LSE in natural log.
//
// Precision: the quantizer chooses scale and zero on a binary16-exact grid
// (binary64 arithmetic with directed rounding taken from the CPU's own FPU via
// fesetround) and computes codes in binary32; attention runs in binary64 on
// the dequantized values.
// Build flags must include -frounding-math -ffp-contract=off.

#include <algorithm>
#include <cfenv>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <vector>

namespace {

constexpr int kDc = 512;   // content latent channels
constexpr int kDr = 64;    // RoPE key channels
constexpr int kGroup = 64; // channels per quantization group
constexpr int kSlots = 64; // token slots per block

enum Format { C4R4 = 0, C2R4 = 1, BF16 = 2, C4R2 = 3, C2R2 = 4 };
enum Round { RN = 0, RD = 1, RU = 2 };

float from_bits(uint32_t u) { float f; std::memcpy(&f, &u, 4); return f; }

// bfloat16 -> binary32: the bfloat16 bits are the upper half of the binary32.
float bf16_to_f32(uint16_t b) { return from_bits(uint32_t(b) << 16); }

// binary16 -> binary32 (exact).
float f16_to_f32(uint16_t h) {
  const int sign = (h >> 15) & 1, e = (h >> 10) & 0x1f, m = h & 0x3ff;
  double v;
  if (e == 0) v = std::ldexp(double(m), -24);                       // subnormal
  else if (e == 31) v = m ? std::numeric_limits<double>::quiet_NaN()
                          : std::numeric_limits<double>::infinity();
  else v = std::ldexp(double(m | 0x400), e - 25);                   // normal
  return float(sign ? -v : v);
}

// binary32 -> binary16 with the given IEEE rounding direction, written from
// the definition: find the two representable magnitudes around |x| and pick
// one; ties (round-to-nearest only) go to the even significand.
uint16_t f32_to_f16(float x, int mode) {
  if (std::isnan(x)) return 0x7e00;
  const bool neg = std::signbit(x);
  if (std::isinf(x)) return neg ? 0xfc00 : 0x7c00;
  const double a = std::fabs(double(x));
  // rounding of the magnitude: toward +inf on the magnitude means "up"
  bool mag_up;  // for directed modes
  if (mode == RD) mag_up = neg; else mag_up = !neg;  // RU: up for positive
  const uint16_t sbit = neg ? 0x8000 : 0;
  if (a == 0.0) return sbit;
  const double max_finite = 65504.0;
  // quantum of the binade containing a
  double q;
  if (a < std::ldexp(1.0, -14)) {
    q = std::ldexp(1.0, -24);
  } else {
    int e;
    std::frexp(a, &e);           // a = f * 2^e, f in [0.5, 1)
    q = std::ldexp(1.0, e - 11); // 11 significant bits
  }
  const double lo = std::floor(a / q) * q;
  const double hi = (lo == a) ? a : lo + q;
  double m;
  if (lo == hi) {
    m = lo;
  } else if (mode == RN) {
    const double dlo = a - lo, dhi = hi - a;
    if (dlo < dhi) m = lo;
    else if (dhi < dlo) m = hi;
    else m = (std::fmod(lo / q, 2.0) == 0.0) ? lo : hi;  // tie: even
  } else {
    m = mag_up ? hi : lo;
  }
  if (m > max_finite) {
    // beyond the largest finite binary16: RN overflows past the midpoint
    // 65520 (already decided by the tie rule above: hi = 65536 is "even"),
    // directed modes overflow only in their own direction.
    if (mode == RN) return sbit | 0x7c00;
    return mag_up ? (sbit | 0x7c00) : (sbit | 0x7bff);
  }
  if (m < std::ldexp(1.0, -14)) {
    return sbit | uint16_t(m / std::ldexp(1.0, -24));  // subnormal (or zero)
  }
  int e;
  const double f = std::frexp(m, &e);  // m = f * 2^e
  const int exp_field = e - 1 + 15;
  const int mant = int(f * 2048.0) - 1024;
  return sbit | uint16_t(exp_field << 10) | uint16_t(mant);
}

// binary32 subtraction and division with an explicit rounding direction,
// executed by the FPU under fesetround (volatile keeps the compiler from
// folding or reordering them).
float f32_sub(float a, float b, int mode) {
  const int old = std::fegetround();
  std::fesetround(mode == RU ? FE_UPWARD : mode == RD ? FE_DOWNWARD : FE_TONEAREST);
  volatile float va = a, vb = b;
  volatile float r = va - vb;
  std::fesetround(old);
  return r;
}
float f32_div(float a, float b, int mode) {
  const int old = std::fegetround();
  std::fesetround(mode == RU ? FE_UPWARD : mode == RD ? FE_DOWNWARD : FE_TONEAREST);
  volatile float va = a, vb = b;
  volatile float r = va / vb;
  std::fesetround(old);
  return r;
}

// binary64 subtraction and division with an explicit rounding direction.
double f64_sub(double a, double b, int mode) {
  const int old = std::fegetround();
  std::fesetround(mode == RU ? FE_UPWARD : mode == RD ? FE_DOWNWARD : FE_TONEAREST);
  volatile double va = a, vb = b;
  volatile double r = va - vb;
  std::fesetround(old);
  return r;
}
double f64_div(double a, double b, int mode) {
  const int old = std::fegetround();
  std::fesetround(mode == RU ? FE_UPWARD : mode == RD ? FE_DOWNWARD : FE_TONEAREST);
  volatile double va = a, vb = b;
  volatile double r = va / vb;
  std::fesetround(old);
  return r;
}

// Round half to even to an integer-valued float.
float rint_even(float t) {
  const float fl = std::floor(t);
  const float d = t - fl;  // exact for |t| < 2^23
  if (d < 0.5f) return fl;
  if (d > 0.5f) return fl + 1.0f;
  return (std::fmod(fl, 2.0f) == 0.0f) ? fl : fl + 1.0f;
}

// The binary16-exact grid of a group: the smallest power of two u = 2^E,
// E in [-24, 5], with integers Z = floor(mn / u) and
// M = max(1, ceil((mx - Z*u) / (levels*u))) such that |Z| <= 2047 and
// |Z + levels*M| <= 2047.  Every grid point (Z + c*M)*u, 0 <= c <= levels,
// is then an integer of at most 11 bits times a power of two: exactly
// representable in binary16.  E starts at a lower bound (the range needs
// levels*M*u >= mx - mn with levels*M <= 4094, so u >= (mx - mn) / 2^12); the
// quotient for M is rounded up, so the bounds hold even when it is inexact.
// Inputs with |x| >= 32768 (outside the precondition) take E = 5 with Z and M
// clamped into range.
void grid_for(float mn, float mx, int levels, int* E_out, double* Z_out, double* M_out) {
  const double d = f64_sub(mx, mn, RD);
  int E = (d > 0.0) ? std::max(-24, std::ilogb(d) - 12) : -24;
  for (;; ++E) {
    const double u = std::ldexp(1.0, E);
    double Z = std::floor(double(mn) / u);
    double M = std::ceil(f64_div(f64_sub(mx, Z * u, RU), levels * u, RU));
    if (M < 1.0) M = 1.0;
    const bool ok = std::fabs(Z) <= 2047.0 && std::fabs(Z + levels * M) <= 2047.0;
    if (ok || E >= 5) {
      if (!ok) {
        Z = std::min(2047.0, std::max(-2047.0, Z));
        M = std::max(1.0, std::min(M, std::floor((2047.0 - Z) / levels)));
      }
      *E_out = E;
      *Z_out = Z;
      *M_out = M;
      return;
    }
  }
}

// Quantize one group of n values to `bits` bits: binary16 scale s = M*u and
// zero z = Z*u on the group's binary16-exact grid, and integer codes
// c = clamp(rint((x - z) / s), 0, levels) in binary32.
void quantize_group(const float* x, int n, int bits, uint16_t* s_out,
                    uint16_t* z_out, uint8_t* codes) {
  const int levels = (1 << bits) - 1;
  float mn = x[0], mx = x[0];
  for (int i = 1; i < n; ++i) {
    if (x[i] < mn) mn = x[i];
    if (x[i] > mx) mx = x[i];
  }
  int E;
  double Z, M;
  grid_for(mn, mx, levels, &E, &Z, &M);
  const uint16_t z = f32_to_f16(float(Z * std::ldexp(1.0, E)), RN);  // exact
  const uint16_t s = f32_to_f16(float(M * std::ldexp(1.0, E)), RN);  // exact
  const float zf = f16_to_f32(z), sf = f16_to_f32(s);
  for (int i = 0; i < n; ++i) {
    const float t = f32_div(f32_sub(x[i], zf, RN), sf, RN);
    float c = rint_even(t);
    if (c < 0.0f) c = 0.0f;
    if (c > float(levels)) c = float(levels);
    codes[i] = uint8_t(c);
  }
  *s_out = s;
  *z_out = z;
}

// Pack codes of `nch` consecutive channels (a multiple of 32/bits) into
// little-endian 32-bit words: even channels in the low half-word, odd channels
// in the high half-word, each half in increasing channel order.
void pack_codes(const uint8_t* codes, int nch, int bits, uint8_t* out) {
  const int per_word = 32 / bits, half = per_word / 2;
  for (int w = 0; w < nch / per_word; ++w) {
    uint32_t word = 0;
    for (int k = 0; k < per_word; ++k) {
      const int ch = (k < half) ? 2 * k : 2 * (k - half) + 1;
      word |= uint32_t(codes[w * per_word + ch]) << (bits * k);
    }
    for (int byte = 0; byte < 4; ++byte) out[w * 4 + byte] = uint8_t(word >> (8 * byte));
  }
}

void unpack_codes(const uint8_t* in, int nch, int bits, uint8_t* codes) {
  const int per_word = 32 / bits, half = per_word / 2;
  const uint32_t mask = (1u << bits) - 1;
  for (int w = 0; w < nch / per_word; ++w) {
    uint32_t word = 0;
    for (int byte = 0; byte < 4; ++byte) word |= uint32_t(in[w * 4 + byte]) << (8 * byte);
    for (int k = 0; k < per_word; ++k) {
      const int ch = (k < half) ? 2 * k : 2 * (k - half) + 1;
      codes[w * per_word + ch] = uint8_t((word >> (bits * k)) & mask);
    }
  }
}

int content_bits(int fmt) { return (fmt == C4R4 || fmt == C4R2) ? 4 : 2; }
int rope_bits(int fmt) { return (fmt == C4R2 || fmt == C2R2) ? 2 : 4; }
size_t code_bytes_per_group(int fmt) { return size_t(kGroup * content_bits(fmt) / 8); }
// RoPE code bytes of one token in one block half (32 channels)
size_t rope_code_bytes(int fmt) { return size_t(32 * rope_bits(fmt) / 8); }
size_t half_bytes(int fmt) {
  if (fmt == BF16) return size_t(4 * kSlots * kGroup * 2 + kSlots * 32 * 2);
  return 4 * kSlots * code_bytes_per_group(fmt) + kSlots * rope_code_bytes(fmt) + 4 * kSlots * 4;
}
size_t block_bytes(int fmt) {
  if (fmt == BF16) return 2 * half_bytes(fmt);
  return 2 * half_bytes(fmt) + kSlots * 4;
}

// Byte offsets inside a block (see the layout specification).
size_t off_content_codes(int fmt, int g, int slot) {
  const int h = g / 4, gi = g % 4;
  return h * half_bytes(fmt) + (size_t(gi) * kSlots + slot) * code_bytes_per_group(fmt);
}
size_t off_rope_codes(int fmt, int h, int slot) {
  return h * half_bytes(fmt) + 4 * kSlots * code_bytes_per_group(fmt) +
         size_t(slot) * rope_code_bytes(fmt);
}
size_t off_content_sz(int fmt, int g, int slot) {
  const int h = g / 4, gi = g % 4;
  return h * half_bytes(fmt) + 4 * kSlots * code_bytes_per_group(fmt) +
         kSlots * rope_code_bytes(fmt) + (size_t(gi) * kSlots + slot) * 4;
}
size_t off_rope_sz(int fmt, int slot) { return 2 * half_bytes(fmt) + size_t(slot) * 4; }
size_t off_bf16_content(int g, int slot) {
  const int h = g / 4, gi = g % 4;
  return h * half_bytes(BF16) + (size_t(gi) * kSlots + slot) * kGroup * 2;
}
size_t off_bf16_rope(int h, int slot) {
  return h * half_bytes(BF16) + 4 * kSlots * kGroup * 2 + size_t(slot) * 32 * 2;
}

void put_u16(uint8_t* p, uint16_t v) { p[0] = uint8_t(v); p[1] = uint8_t(v >> 8); }
uint16_t get_u16(const uint8_t* p) { return uint16_t(p[0] | (p[1] << 8)); }

// Write one token (576 bf16 values: 512 content then 64 RoPE) into `slot`.
void write_token(int fmt, uint8_t* blk, int slot, const uint16_t* lat, const uint16_t* rope) {
  if (fmt == BF16) {
    for (int c = 0; c < kDc; ++c) put_u16(blk + off_bf16_content(c / 64, slot) + (c % 64) * 2, lat[c]);
    for (int j = 0; j < kDr; ++j) put_u16(blk + off_bf16_rope(j / 32, slot) + (j % 32) * 2, rope[j]);
    return;
  }
  float x[kGroup];
  uint8_t codes[kGroup];
  uint16_t s, z;
  const int cb = content_bits(fmt);
  for (int g = 0; g < kDc / kGroup; ++g) {
    for (int i = 0; i < kGroup; ++i) x[i] = bf16_to_f32(lat[g * kGroup + i]);
    quantize_group(x, kGroup, cb, &s, &z, codes);
    pack_codes(codes, kGroup, cb, blk + off_content_codes(fmt, g, slot));
    put_u16(blk + off_content_sz(fmt, g, slot), s);
    put_u16(blk + off_content_sz(fmt, g, slot) + 2, z);
  }
  // the RoPE key: one 64-channel group; channels 0-31 go to half 0, 32-63 to half 1
  const int rb = rope_bits(fmt);
  for (int i = 0; i < kDr; ++i) x[i] = bf16_to_f32(rope[i]);
  quantize_group(x, kDr, rb, &s, &z, codes);
  pack_codes(codes, 32, rb, blk + off_rope_codes(fmt, 0, slot));
  pack_codes(codes + 32, 32, rb, blk + off_rope_codes(fmt, 1, slot));
  put_u16(blk + off_rope_sz(fmt, slot), s);
  put_u16(blk + off_rope_sz(fmt, slot) + 2, z);
}

// Dequantize one token: x_hat = float(code) * float(s) + float(z), the
// multiply and the add each rounded to nearest binary32 (no fused multiply-add).
void read_token(int fmt, const uint8_t* blk, int slot, float* out576) {
  if (fmt == BF16) {
    for (int c = 0; c < kDc; ++c) out576[c] = bf16_to_f32(get_u16(blk + off_bf16_content(c / 64, slot) + (c % 64) * 2));
    for (int j = 0; j < kDr; ++j) out576[kDc + j] = bf16_to_f32(get_u16(blk + off_bf16_rope(j / 32, slot) + (j % 32) * 2));
    return;
  }
  uint8_t codes[kGroup];
  const int cb = content_bits(fmt);
  for (int g = 0; g < kDc / kGroup; ++g) {
    unpack_codes(blk + off_content_codes(fmt, g, slot), kGroup, cb, codes);
    const float s = f16_to_f32(get_u16(blk + off_content_sz(fmt, g, slot)));
    const float z = f16_to_f32(get_u16(blk + off_content_sz(fmt, g, slot) + 2));
    for (int i = 0; i < kGroup; ++i) {
      const float prod = float(codes[i]) * s;
      out576[g * kGroup + i] = prod + z;
    }
  }
  const int rb = rope_bits(fmt);
  unpack_codes(blk + off_rope_codes(fmt, 0, slot), 32, rb, codes);
  unpack_codes(blk + off_rope_codes(fmt, 1, slot), 32, rb, codes + 32);
  const float s = f16_to_f32(get_u16(blk + off_rope_sz(fmt, slot)));
  const float z = f16_to_f32(get_u16(blk + off_rope_sz(fmt, slot) + 2));
  for (int j = 0; j < kDr; ++j) {
    const float prod = float(codes[j]) * s;
    out576[kDc + j] = prod + z;
  }
}

// Attention over tokens [t0, t1) of one sequence for H heads, in binary64.
// Writes O[H][512] (normalized) and LSE[H]; empty ranges give O = 0, LSE = -inf.
void attend_range(int fmt, const uint8_t* blocks, const int32_t* table_row, int t0, int t1,
                  int H, const uint16_t* qc, const uint16_t* qr, double scale,
                  double* O, double* lse) {
  const int n = t1 - t0;
  for (int h = 0; h < H; ++h) {
    lse[h] = -std::numeric_limits<double>::infinity();
    for (int c = 0; c < kDc; ++c) O[size_t(h) * kDc + c] = 0.0;
  }
  if (n <= 0) return;
  const size_t bb = block_bytes(fmt);
  std::vector<float> xt(size_t(n) * (kDc + kDr));
  for (int t = t0; t < t1; ++t) {
    const uint8_t* blk = blocks + size_t(table_row[t / kSlots]) * bb;
    read_token(fmt, blk, t % kSlots, &xt[size_t(t - t0) * (kDc + kDr)]);
  }
  std::vector<double> q(kDc + kDr), sc(n);
  for (int h = 0; h < H; ++h) {
    for (int c = 0; c < kDc; ++c) q[c] = bf16_to_f32(qc[size_t(h) * kDc + c]);
    for (int j = 0; j < kDr; ++j) q[kDc + j] = bf16_to_f32(qr[size_t(h) * kDr + j]);
    double m = -std::numeric_limits<double>::infinity();
    for (int t = 0; t < n; ++t) {
      const float* x = &xt[size_t(t) * (kDc + kDr)];
      double acc = 0.0;
      for (int c = 0; c < kDc + kDr; ++c) acc += q[c] * double(x[c]);
      sc[t] = acc * scale;
      if (sc[t] > m) m = sc[t];
    }
    double l = 0.0;
    for (int t = 0; t < n; ++t) l += std::exp(sc[t] - m);
    const double L = m + std::log(l);
    lse[h] = L;
    double* o = O + size_t(h) * kDc;
    for (int t = 0; t < n; ++t) {
      const double p = std::exp(sc[t] - L);
      const float* x = &xt[size_t(t) * (kDc + kDr)];
      for (int c = 0; c < kDc; ++c) o[c] += p * double(x[c]);
    }
  }
}

}  // namespace

extern "C" {

uint16_t oracle_f32_to_f16(float x, int mode) { return f32_to_f16(x, mode); }
float oracle_f16_to_f32(uint16_t h) { return f16_to_f32(h); }
float oracle_f32_sub(float a, float b, int mode) { return f32_sub(a, b, mode); }
float oracle_f32_div(float a, float b, int mode) { return f32_div(a, b, mode); }
double oracle_f64_sub(double a, double b, int mode) { return f64_sub(a, b, mode); }
double oracle_f64_div(double a, double b, int mode) { return f64_div(a, b, mode); }
void oracle_grid_for(float mn, float mx, int levels, int* E, double* Z, double* M) {
  grid_for(mn, mx, levels, E, Z, M);
}

size_t oracle_block_bytes(int fmt) {
  if (fmt < 0 || fmt > 4) return 0;
  return block_bytes(fmt);
}

// Vectorised binary32 -> binary16 for exhaustive comparisons.
void oracle_f32_to_f16_array(const float* x, int64_t n, int mode, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = f32_to_f16(x[i], mode);
}

void oracle_quantize_group(const float* x, int n, int bits, uint16_t* s, uint16_t* z,
                           uint8_t* codes) {
  quantize_group(x, n, bits, s, z, codes);
}
void oracle_pack_codes(const uint8_t* codes, int nch, int bits, uint8_t* out) {
  pack_codes(codes, nch, bits, out);
}
void oracle_unpack_codes(const uint8_t* in, int nch, int bits, uint8_t* codes) {
  unpack_codes(in, nch, bits, codes);
}

// Mirror of qmla_append: returns the number of tokens skipped because their
// slot lies outside the block table or their block id outside the pool.
int oracle_append(int fmt, uint8_t* blocks, int64_t num_blocks, const int32_t* block_table,
                  int max_blocks_per_seq, const int32_t* positions, int batch, int n_new,
                  const uint16_t* latent, const uint16_t* rope) {
  int skipped = 0;
  const size_t bb = block_bytes(fmt);
  for (int b = 0; b < batch; ++b) {
    for (int i = 0; i < n_new; ++i) {
      const int64_t pos = int64_t(positions[b]) + i;
      const int64_t jb = pos / kSlots;
      if (pos < 0 || jb >= max_blocks_per_seq) { ++skipped; continue; }
      const int32_t blk = block_table[size_t(b) * max_blocks_per_seq + jb];
      if (blk < 0 || blk >= num_blocks) { ++skipped; continue; }
      write_token(fmt, blocks + size_t(blk) * bb, int(pos % kSlots),
                  latent + (size_t(b) * n_new + i) * kDc, rope + (size_t(b) * n_new + i) * kDr);
    }
  }
  return skipped;
}

// Dequantized token (576 floats: 512 content then 64 RoPE) of slot `slot`
// of the block at `blk`.
void oracle_read_token(int fmt, const uint8_t* blk, int slot, float* out576) {
  read_token(fmt, blk, slot, out576);
}

// Full decode: O [batch][H][512] and LSE [batch][H] in binary64.
void oracle_decode(int fmt, const uint8_t* blocks, const int32_t* block_table,
                   int max_blocks_per_seq, const int32_t* seq_lens, int batch, int H,
                   const uint16_t* q_c, const uint16_t* q_r, double scale, double* out,
                   double* lse) {
  for (int b = 0; b < batch; ++b) {
    attend_range(fmt, blocks, block_table + size_t(b) * max_blocks_per_seq, 0, seq_lens[b], H,
                 q_c + size_t(b) * H * kDc, q_r + size_t(b) * H * kDr, scale,
                 out + size_t(b) * H * kDc, lse + size_t(b) * H);
  }
}

// Merge of split partials (O_i normalized, LSE_i):
//   LSE = ln sum_i exp(LSE_i),  O = sum_i exp(LSE_i - LSE) * O_i.
void oracle_merge(int nsplit, int H, const double* part_o, const double* part_lse, double* out,
                  double* lse) {
  for (int h = 0; h < H; ++h) {
    double m = -std::numeric_limits<double>::infinity();
    for (int i = 0; i < nsplit; ++i) m = std::fmax(m, part_lse[size_t(i) * H + h]);
    double* o = out + size_t(h) * kDc;
    for (int c = 0; c < kDc; ++c) o[c] = 0.0;
    if (std::isinf(m) && m < 0) { lse[h] = m; continue; }
    double sum = 0.0;
    for (int i = 0; i < nsplit; ++i) sum += std::exp(part_lse[size_t(i) * H + h] - m);
    const double L = m + std::log(sum);
    lse[h] = L;
    for (int i = 0; i < nsplit; ++i) {
      const double w = std::exp(part_lse[size_t(i) * H + h] - L);
      if (w == 0.0) continue;
      const double* oi = part_o + (size_t(i) * H + h) * kDc;
      for (int c = 0; c < kDc; ++c) o[c] += w * oi[c];
    }
  }
}

// Decode of one sequence with its context cut into `nsplit` contiguous
// ranges of equal block count, each attended separately, then merged.
void oracle_decode_split(int fmt, const uint8_t* blocks, const int32_t* table_row, int L,
                         int H, const uint16_t* q_c, const uint16_t* q_r, double scale,
                         int nsplit, double* out, double* lse) {
  std::vector<double> po(size_t(nsplit) * H * kDc), pl(size_t(nsplit) * H);
  const int nblk = (L + kSlots - 1) / kSlots;
  for (int i = 0; i < nsplit; ++i) {
    const int b0 = int(int64_t(nblk) * i / nsplit), b1 = int(int64_t(nblk) * (i + 1) / nsplit);
    const int t0 = b0 * kSlots, t1 = std::min(L, b1 * kSlots);
    attend_range(fmt, blocks, table_row, t0, t1, H, q_c, q_r, scale,
                 &po[size_t(i) * H * kDc], &pl[size_t(i) * H]);
  }
  oracle_merge(nsplit, H, po.data(), pl.data(), out, lse);
}

}  // extern "C"
