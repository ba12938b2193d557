// decode_tc16.cu - tensor-core (tcgen05) decode over the low-bit paged cache,
// 16 absorbed query heads.
//
// The "native low-bit MLA attention kernel" of "QuantMLA: INT4 (and INT2) for
// both halves of the MLA cache" (flowchart node "Low-bit kernel: dequant
// inside attention") for the small-head-count case.  With 16 heads the
// product is too thin for heads on the MMA's M dimension (M >= 64), so the
// tokens go there instead:
//   QK : S^T[128 tok x 16 heads] = K[128 tok x 576] (A, smem, K-major)
//                                 x Q^T              (B, smem, 16 rows)
//   PV : O^T[512 ch x 16 heads] += C^T[512 ch x 128 tok] (A, the same smem
//        tile read MN-major, 4 slices of 128 channels) x P^T (B, smem)
// One CTA per SM; tensor memory holds S^T (16 columns) and O^T (4 x 16).
// The softmax runs over tokens, i.e. across the 128 lanes of S^T: per-head
// maxima are reduced with warp shuffles and across the four softmax warps
// through shared memory; row sums are kept per lane and reduced once per
// piece.  Rescaling of O^T is lazy (only when a maximum grows by more than 8
// in log2 units).
//
// Warp roles (14 warps): 0 bulk-copy producer (whole blocks), 1 MMA issuer,
// 2-5 softmax (thread = token lane), 6-13 dequantization.  Binary16 operands
// (exact on the quantizer's grid), binary32 accumulation.  Waits are bounded;
// a timeout raises an abort flag and QMLA_STATUS_TIMEOUT.

#include <cfloat>

#include "tc_common.cuh"

namespace qmla {
namespace {

using namespace ptx;
using namespace tc;

constexpr int kThreads = 448;
constexpr int kMmaWarp = 1;
constexpr int kSoftmaxWarp0 = 2;
constexpr int kDequantWarp0 = 6;
constexpr int kDequantThreads = 256;
constexpr int kH = 16;                                 // heads

constexpr uint32_t kTmemCols = 128;
constexpr uint32_t kColS = 0, kColO = 64;              // S^T 4 x 16 (partial sums), O^T 4 x 16

constexpr uint32_t kChunk = 16384;                     // [128 tok][64 ch] fp16 SW128
constexpr uint32_t kSmK = 0;                           // 8 content chunks + RoPE chunk
constexpr uint32_t kSmQ = kSmK + 9 * kChunk;           // 9 x [16 heads][128 B]
constexpr uint32_t kSmP = kSmQ + 9 * 2048;             // 2 x [16 heads][128 B] (P^T)
constexpr uint32_t kSmStage = kSmP + 2 * 2048;         // 2 x one whole block
constexpr uint32_t kStage = 20736;                     // largest block (C4R4)
constexpr uint32_t kSmRed = kSmStage + 2 * kStage;     // [4 warps][16] max, [4][16] sum
constexpr uint32_t kSmBar = kSmRed + 512;
constexpr uint32_t kNumBars = 11;
constexpr uint32_t kSmTslot = kSmBar + 8 * kNumBars;
constexpr uint32_t kSmAbort = kSmTslot + 4;
constexpr uint32_t kSmBytes = kSmAbort + 12;
constexpr uint32_t kSmDyn = kSmBytes + 1024;

enum : uint32_t {
  B_STAGE_FULL = 0, B_STAGE_EMPTY = 2, B_K_FULL = 4, B_K_EMPTY = 5, B_S_FULL = 6,
  B_P_FULL = 7, B_PV_DONE = 8, B_Q_FULL = 9, B_DRAIN = 10
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__global__ void __launch_bounds__(kThreads, 1) decode_tc16_kernel(DecodeArgs a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb0 = smem_u32(sm);
  auto BAR = [&](uint32_t i) { return sb0 + kSmBar + 8 * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kSmAbort);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int worker = blockIdx.x;
  const Geom G = geom(a.fmt);

  if (threadIdx.x == 0) {
    for (uint32_t i = 0; i < 2; ++i) {
      mbar_init(BAR(B_STAGE_FULL + i), 1);
      mbar_init(BAR(B_STAGE_EMPTY + i), kDequantThreads / 32);
    }
    mbar_init(BAR(B_K_FULL), kDequantThreads / 32);
    mbar_init(BAR(B_K_EMPTY), 1);
    mbar_init(BAR(B_S_FULL), 1);
    mbar_init(BAR(B_P_FULL), 128);
    mbar_init(BAR(B_PV_DONE), 1);
    mbar_init(BAR(B_Q_FULL), 128);
    mbar_init(BAR(B_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(sb0 + kSmTslot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *reinterpret_cast<volatile uint32_t*>(sm + kSmTslot);
  const int2 wr = a.ws.wrange[worker];

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    uint32_t u = 0;  // block counter
    bool ok = true;
    for (int s = wr.x; ok && s <= wr.y; ++s) {
      const int4 pc = a.ws.pieces[s];
      for (int jb = pc.y; ok && jb < pc.z; jb += 32) {
        const int n = min(32, pc.z - jb);
        const int32_t my_blk =
            (lane < n) ? a.block_table[int64_t(pc.x) * a.max_blocks_per_seq + jb + lane] : -1;
        for (int k = 0; k < n; ++k, ++u) {
          const int32_t blk = __shfl_sync(0xffffffffu, my_blk, k);
          bool got = true;
          if (lane == 0) {
            const uint32_t st = u & 1u, par = (u >> 1) & 1u;
            got = mbar_wait(BAR(B_STAGE_EMPTY + st), par ^ 1u, abort_flag, kWaitNs);
            if (got) {
              if (blk >= 0 && blk < a.num_blocks) {
                mbar_arrive_expect_tx(BAR(B_STAGE_FULL + st), uint32_t(G.block));
                bulk_g2s(sb0 + kSmStage + st * kStage, a.blocks + int64_t(blk) * G.block,
                         uint32_t(G.block), BAR(B_STAGE_FULL + st));
              } else {
                set_status(a.status, QMLA_STATUS_BAD_BLOCK);
                mbar_arrive_expect_tx(BAR(B_STAGE_FULL + st), 0u);
              }
            }
          }
          if (!warp_ok(got)) {
            ok = false;
            break;
          }
        }
      }
    }
    if (lane == 0)
      for (uint32_t v = (u >= 2 ? u - 2 : 0); v < u; ++v)
        wait_noabort(BAR(B_STAGE_FULL + (v & 1u)), (v >> 1) & 1u);
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_qk = idesc_f16(128, kH, false, false);
      const uint32_t idesc_pv = idesc_f16(128, kH, true, false);
      // operand descriptors; an offset inside the tile advances the 16-byte
      // address field (shared memory < 256 KB: no carry out of the field)
      const uint64_t dK = smem_desc(sb0 + kSmK, 16, 1024, kSwizzle128B);
      const uint64_t dQ = smem_desc(sb0 + kSmQ, 16, 1024, kSwizzle128B);
      const uint64_t dC = smem_desc(sb0 + kSmK, kChunk, 1024, kSwizzle128B);
      const uint64_t dP = smem_desc(sb0 + kSmP, 16, 1024, kSwizzle128B);
      uint32_t t = 0, piece = 0;
      bool ok = true;
      for (int s = wr.x; ok && s <= wr.y; ++s) {
        const int4 pc = a.ws.pieces[s];
        if (pc.z <= pc.y) continue;
        if (!mbar_wait(BAR(B_Q_FULL), piece & 1u, abort_flag, kWaitNs)) break;
        ++piece;
        for (int jt = pc.y; jt < pc.z; jt += 2, ++t) {
          if (!mbar_wait(BAR(B_K_FULL), t & 1u, abort_flag, kWaitNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // four independent partial sums over k-steps 9p..9p+8, issued round
          // robin: chained MMAs into one accumulator serialize on its latency
#pragma unroll
          for (uint32_t i = 0; i < 9; ++i) {
#pragma unroll
            for (uint32_t p = 0; p < 4; ++p) {
              const uint32_t ks = 9 * p + i, c = ks >> 2, koff = (ks & 3u) * 32u;
              mma_ss(tbase + kColS + kH * p, dK + ((c * kChunk + koff) >> 4),
                     dQ + ((c * 2048 + koff) >> 4), idesc_qk, i > 0 ? 1u : 0u);
            }
          }
          mma_commit(BAR(B_S_FULL));
          if (!mbar_wait(BAR(B_P_FULL), t & 1u, abort_flag, kWaitNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const bool first = (jt == pc.y);
#pragma unroll
          for (uint32_t ks = 0; ks < 8; ++ks) {
#pragma unroll
            for (uint32_t mk = 0; mk < 4; ++mk)
              mma_ss(tbase + kColO + kH * mk, dC + ((2 * mk * kChunk + ks * 2048) >> 4),
                     dP + (((ks >> 2) * 2048 + (ks & 3u) * 32u) >> 4), idesc_pv,
                     (first && ks == 0) ? 0u : 1u);
          }
          mma_commit(BAR(B_PV_DONE));
          mma_commit(BAR(B_K_EMPTY));
        }
      }
      mma_commit(BAR(B_DRAIN));
      wait_noabort(BAR(B_DRAIN), 0);
    }
  } else if (warp >= kSoftmaxWarp0 && warp < kDequantWarp0) {
    // ------------------------------------------------------------ softmax
    const uint32_t quad = uint32_t(warp & 3);
    const int r = int(quad * 32) + lane;  // token row of S^T / channel row of O^T
    const int sw = warp - kSoftmaxWarp0;  // 0..3
    const uint32_t lane_base = (quad * 32u) << 16;
    const float c2 = a.scale * 1.4426950408889634f;
    float* red_max = reinterpret_cast<float*>(sm + kSmRed);
    float* red_sum = red_max + 4 * kH;
    uint32_t t = 0;
    bool ok = true;
    for (int s = wr.x; ok && s <= wr.y; ++s) {
      const int4 pc = a.ws.pieces[s];
      const int b = pc.x;
      if (pc.z <= pc.y) {
        for (int i = threadIdx.x - kSoftmaxWarp0 * 32; i < kH * kDc; i += 128)
          a.ws.part_o[int64_t(s) * kH * kDc + i] = 0.f;
        if (r < kH) a.ws.part_lse[int64_t(s) * kH + r] = -INFINITY;
        continue;
      }
      const int L = seq_len_clamped(a, b);
      // Q^T of this piece: 16 heads x 576 channels, binary16, SW128 K-major
      for (int i = threadIdx.x - kSoftmaxWarp0 * 32; i < kH * 72; i += 128) {
        const int h = i / 72, sgm = i % 72;  // 8-channel segment
        const __nv_bfloat16* src =
            (sgm < 64) ? a.q_c + (int64_t(b) * kH + h) * kDc + sgm * 8
                       : a.q_r + (int64_t(b) * kH + h) * kDr + (sgm - 64) * 8;
        const uint4 v = *reinterpret_cast<const uint4*>(src);
        const uint32_t in[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          o[k] = pack_half2(__uint_as_float(in[k] << 16), __uint_as_float(in[k] & 0xffff0000u));
        const int c = sgm >> 3, g = sgm & 7;
        unsigned char* row = sm + kSmQ + c * 2048 + (h >> 3) * 1024 + (h & 7) * 128;
        *reinterpret_cast<uint4*>(row + ((g ^ (h & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
      }
      fence_proxy_async_smem();
      mbar_arrive(BAR(B_Q_FULL));

      float m_used[kH], l_part[kH];
#pragma unroll
      for (int h = 0; h < kH; ++h) {
        m_used[h] = -INFINITY;
        l_part[h] = 0.0f;
      }
      uint32_t vmask = 0;
      for (int jt = pc.y; jt < pc.z; jt += 2, ++t) {
        if (((jt - pc.y) & 31) == 0) vmask = valid_mask(a, b, jt, pc.z);
        // validity of this lane's token row
        const int bi = r >> 6, jj = jt + bi;
        const bool blk_ok = jj < pc.z && ((vmask >> ((jj - pc.y) & 31)) & 1u);
        const bool row_ok = blk_ok && (r & 63) < min(kT, L - jj * kT);
        if (!warp_ok(mbar_wait(BAR(B_S_FULL), t & 1u, abort_flag, kWaitNs))) {
          ok = false;
          break;
        }
        tc_fence_after();
        float sv[kH];
        {
          uint32_t q0[32], q1[32];
          tmem_ld32(tbase + lane_base + kColS, q0);
          tmem_ld32(tbase + lane_base + kColS + 32, q1);
          tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < kH; ++h) {
            const float v = (__uint_as_float(q0[h]) + __uint_as_float(q0[16 + h])) +
                            (__uint_as_float(q1[h]) + __uint_as_float(q1[16 + h]));
            sv[h] = row_ok ? v * c2 : -INFINITY;
          }
        }
        // per-head maximum over the 128 token rows
        float wm[kH];
#pragma unroll
        for (int h = 0; h < kH; ++h) wm[h] = warp_max(sv[h]);
        if (lane == 0) {
#pragma unroll
          for (int h = 0; h < kH; h += 4)
            *reinterpret_cast<float4*>(red_max + sw * kH + h) =
                make_float4(wm[h], wm[h + 1], wm[h + 2], wm[h + 3]);
        }
        named_bar_sync(1, 128);
        float mt[kH];
#pragma unroll
        for (int h = 0; h < kH; h += 4) {
          const float4 v0 = *reinterpret_cast<const float4*>(red_max + 0 * kH + h);
          const float4 v1 = *reinterpret_cast<const float4*>(red_max + 1 * kH + h);
          const float4 v2 = *reinterpret_cast<const float4*>(red_max + 2 * kH + h);
          const float4 v3 = *reinterpret_cast<const float4*>(red_max + 3 * kH + h);
          mt[h] = fmaxf(fmaxf(v0.x, v1.x), fmaxf(v2.x, v3.x));
          mt[h + 1] = fmaxf(fmaxf(v0.y, v1.y), fmaxf(v2.y, v3.y));
          mt[h + 2] = fmaxf(fmaxf(v0.z, v1.z), fmaxf(v2.z, v3.z));
          mt[h + 3] = fmaxf(fmaxf(v0.w, v1.w), fmaxf(v2.w, v3.w));
        }
        // lazy rescale: identical decisions in every thread
        bool any = false;
        float alpha[kH];
#pragma unroll
        for (int h = 0; h < kH; ++h) {
          const bool need = mt[h] > m_used[h] + 8.0f;
          alpha[h] = need ? ex2_approx(m_used[h] - mt[h]) : 1.0f;
          if (need) m_used[h] = mt[h];
          any |= need;
        }
        if (any) {
#pragma unroll
          for (int h = 0; h < kH; ++h) l_part[h] *= alpha[h];
          if (jt > pc.y) {  // O^T holds earlier tiles (P.V of the previous tile is done)
#pragma unroll 1
            for (uint32_t mk = 0; mk < 4; ++mk) {
              uint32_t o[16];
              tmem_ld16(tbase + lane_base + kColO + kH * mk, o);
              tmem_wait_ld();
#pragma unroll
              for (int h = 0; h < kH; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * alpha[h]);
              tmem_st16(tbase + lane_base + kColO + kH * mk, o);
            }
            tmem_wait_st();
          }
        }
        // P^T[h][r] = 2^(s - m) as binary16 into the SW128 K-major B tile
        unsigned char* preg = sm + kSmP + (r >> 6) * 2048;
        const int tk = r & 63;
#pragma unroll
        for (int h = 0; h < kH; ++h) {
          const float p = ex2_approx(sv[h] - (m_used[h] == -INFINITY ? 0.0f : m_used[h]));
          l_part[h] += p;
          unsigned char* row = preg + (h >> 3) * 1024 + (h & 7) * 128;
          *reinterpret_cast<__half*>(row + ((((tk >> 3) ^ (h & 7))) << 4) + (tk & 7) * 2) =
              __float2half_rn(p);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(BAR(B_P_FULL));
      }
      if (!ok) break;
      // epilogue: row sums over the 128 lanes, normalized partial O, LSE
      if (!warp_ok(mbar_wait(BAR(B_PV_DONE), (t - 1) & 1u, abort_flag, kWaitNs))) break;
      tc_fence_after();
      float lsum[kH];
#pragma unroll
      for (int h = 0; h < kH; ++h) lsum[h] = warp_sum_f(l_part[h]);
      if (lane == 0) {
#pragma unroll
        for (int h = 0; h < kH; h += 4)
          *reinterpret_cast<float4*>(red_sum + sw * kH + h) =
              make_float4(lsum[h], lsum[h + 1], lsum[h + 2], lsum[h + 3]);
      }
      named_bar_sync(1, 128);
      float inv[kH];
#pragma unroll
      for (int h = 0; h < kH; ++h) {
        const float l = red_sum[h] + red_sum[kH + h] + red_sum[2 * kH + h] + red_sum[3 * kH + h];
        inv[h] = l > 0.0f ? 1.0f / l : 0.0f;
        if (r == h)
          a.ws.part_lse[int64_t(s) * kH + h] =
              l > 0.0f ? (m_used[h] + log2f(l)) * 0.6931471805599453f : -INFINITY;
      }
#pragma unroll 1
      for (uint32_t mk = 0; mk < 4; ++mk) {
        uint32_t o[16];
        tmem_ld16(tbase + lane_base + kColO + kH * mk, o);
        tmem_wait_ld();
        float* dst = a.ws.part_o + int64_t(s) * kH * kDc + 128 * mk + r;
#pragma unroll
        for (int h = 0; h < kH; ++h) dst[h * kDc] = __uint_as_float(o[h]) * inv[h];
      }
      tc_fence_before();
      named_bar_sync(1, 128);  // red_sum is read by all before the next piece reuses it
    }
  } else if (warp >= kDequantWarp0) {
    // ------------------------------------------------------------ dequant
    const int dt = int(threadIdx.x) - kDequantWarp0 * 32;
    uint32_t t = 0, u = 0;
    bool ok = true;
    for (int s = wr.x; ok && s <= wr.y; ++s) {
      const int4 pc = a.ws.pieces[s];
      const int L = seq_len_clamped(a, pc.x);
      uint32_t vmask = 0;
      for (int jt = pc.y; jt < pc.z; jt += 2, ++t) {
        if (((jt - pc.y) & 31) == 0) vmask = valid_mask(a, pc.x, jt, pc.z);
        if (!warp_ok(mbar_wait(BAR(B_K_EMPTY), (t & 1u) ^ 1u, abort_flag, kWaitNs))) {
          ok = false;
          break;
        }
        for (int bi = 0; bi < 2; ++bi) {
          const int j = jt + bi;
          const bool present = j < pc.z;
          int nvalid = 0;
          const unsigned char* stg = sm + kSmStage + (u & 1u) * kStage;
          if (present) {
            if (!warp_ok(mbar_wait(BAR(B_STAGE_FULL + (u & 1u)), (u >> 1) & 1u, abort_flag,
                                   kWaitNs))) {
              ok = false;
              break;
            }
            nvalid = ((vmask >> ((j - pc.y) & 31)) & 1u) ? min(kT, L - j * kT) : 0;
          }
          // thread dt owns token tt and 16-channel segment seg of every group
          // (8 tokens x 4 segments per warp: conflict-free reads and writes);
          // loads are unconditional and invalid tokens are zeroed by a select,
          // so the unrolled groups' loads can all be in flight together
          {
            const int tt = (dt >> 2) & 63, seg = dt & 3;
            const bool valid = tt < nvalid;
            const int row = 64 * bi + tt;
#pragma unroll
            for (int g = 0; g < 8; ++g) {
              const unsigned char* half = stg + (g >> 2) * G.half;
              const int gi = g & 3;
              __half2 s2, z2;
              split_sz(*reinterpret_cast<const uint32_t*>(half + G.sz_off + (gi * 64 + tt) * 4), s2,
                       z2);
              uint32_t v[8];
              if (G.cbits == 4) {
                const uint2 w = *reinterpret_cast<const uint2*>(half + gi * 2048 + tt * 32 + seg * 8);
                dq_int4(w.x, s2, z2, v);
                dq_int4(w.y, s2, z2, v + 4);
              } else {
                dq_int2(*reinterpret_cast<const uint32_t*>(half + gi * 1024 + tt * 16 + seg * 4), s2,
                        z2, v);
              }
#pragma unroll
              for (int k = 0; k < 8; ++k) v[k] = valid ? v[k] : 0u;
              st_row16(sm + kSmK + g * kChunk, row, seg, v);
            }
            // RoPE (INT4): the same token and segment of the 64 RoPE channels
            {
              __half2 s2, z2;
              split_sz(*reinterpret_cast<const uint32_t*>(stg + G.rope_sz_off + tt * 4), s2, z2);
              const uint2 w = *reinterpret_cast<const uint2*>(stg + (seg >> 1) * G.half + G.rope_off +
                                                              tt * 16 + (seg & 1) * 8);
              uint32_t v[8];
              dq_int4(w.x, s2, z2, v);
              dq_int4(w.y, s2, z2, v + 4);
#pragma unroll
              for (int k = 0; k < 8; ++k) v[k] = valid ? v[k] : 0u;
              st_row16(sm + kSmK + 8 * kChunk, row, seg, v);
            }
          }
          if (present) {
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(B_STAGE_EMPTY + (u & 1u)));
            ++u;
          }
        }
        if (!ok) break;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(B_K_FULL));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) set_status(a.status, QMLA_STATUS_TIMEOUT);
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_decode_tc16(const DecodeArgs& a, cudaStream_t stream) {
  static int smem_attr_done[kMaxDevices];
  cudaError_t e = launch_plan(a, stream);
  if (e != cudaSuccess) return e;
  e = ensure_smem_attr(decode_tc16_kernel, int(kSmDyn), smem_attr_done);
  if (e != cudaSuccess) return e;
  decode_tc16_kernel<<<dim3(unsigned(a.workers)), kThreads, kSmDyn, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace qmla
