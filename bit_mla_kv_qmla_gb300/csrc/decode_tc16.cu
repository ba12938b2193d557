// decode_tc16.cu - tensor-core (tcgen05) decode over the low-bit paged cache,
// 16 absorbed query heads.
//
// The "native low-bit MLA attention kernel" of "QuantMLA: INT4 (and INT2) for
// both halves of the MLA cache" (flowchart node "Low-bit kernel: dequant
// inside attention") for the small-head-count case.  With 16 heads the
// product is too thin for heads on the MMA's M dimension (M >= 64), so the
// 128 tokens of a tile (two cache blocks) go there instead:
//   QK : S^T[128 tok x 16 heads] = K[128 tok x 576] (A, tensor memory)
//                                 x Q^T              (B, smem, 16 rows)
//   PV : O^T[512 ch x 16 heads] += C^T[512 ch x 128 tok] (A, smem, read
//        MN-major in 4 slices of 128 channels) x P^T (B, smem)
// The dequantization warps write every binary16 value twice: into tensor
// memory (lane = token) for QK and into a swizzled shared-memory tile for PV.
// K in tensor memory keeps half of the MMA operand traffic out of shared
// memory and lets QK of a tile chase its dequantization: a tile is two work
// items (half 0 of both blocks: content channels 0-255 and RoPE 0-31; half 1:
// content 256-511 and RoPE 32-63), each with full/empty barriers.  The
// shared-memory content tile of a half goes to one of three 64 KB groups, so
// the dequantization of a tile's first half overlaps the softmax and P.V
// products of the previous tile.  The packed codes need no staging in shared
// memory: the dequantization threads load them straight from global memory
// (32 bytes per token and group in one 256-bit load), one half-tile ahead of
// use, with block ids fetched 32 blocks at a time well ahead.
//
// At M=128, N=16 an MMA costs a roughly fixed ~50 cycles to issue, so the
// MMA count (36 QK + 32 PV per tile) and every wait/commit around them set the
// pace.  Two converged warps issue them, one for QK and one for P.V (an
// elected lane issues each instruction), with few synchronization points per
// tile.
//
// The softmax runs over tokens, i.e. across the 128 lanes of S^T.  A tile
// first checks, with one OR-barrier, whether any score exceeds the running
// maximum by more than kLazy = 15 (log2 units; P < 2^15 stays inside
// binary16's range, row sums and O are binary32); only then are per-head
// maxima reduced and O^T rescaled (lazy rescaling).  Row sums are kept per
// lane and reduced once per piece.
//
// Warp roles (14 warps): 0 QK issuer, 1 P.V issuer, 2-5 softmax (thread =
// token lane), 6-13 dequantization (two warps per lane quarter).  Binary16 operands (exact on the quantizer's grid), binary32
// accumulation.  Waits are bounded; a timeout raises an abort flag and
// QMLA_STATUS_TIMEOUT.

#include <cfloat>

#include "tc_common.cuh"

namespace qmla {
namespace {

using namespace ptx;
using namespace tc;

constexpr int kThreads = 448;
constexpr int kQkWarp = 0;
constexpr int kPvWarp = 1;
constexpr int kSoftmaxWarp0 = 2;
constexpr int kDequantWarp0 = 6;
constexpr int kH = 16;  // heads
// lazy-rescale margin (log2 units): P = 2^(s - m) < 2^15
constexpr float kLazy = 15.0f;

// tensor memory columns (32-bit); K holds binary16 pairs (channel 2j, 2j+1)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColK = 0;       // content chunk c (64 channels) at 32c
constexpr uint32_t kColRope = 256;  // RoPE channels, 32 columns
constexpr uint32_t kColS = 288;     // S^T: 4 partial sums x 16
constexpr uint32_t kColO = 352;     // O^T: 4 slices of 128 channels x 16

// shared memory
constexpr uint32_t kChunk = 16384;                   // [128 tok][64 ch] fp16, SW128
constexpr uint32_t kGroup = 4 * kChunk;              // content tile of one half
constexpr uint32_t kSmV = 0;                         // 3 groups
constexpr uint32_t kSmQ = kSmV + 3 * kGroup;         // 9 x [16 heads][128 B]
constexpr uint32_t kSmP = kSmQ + 9 * 2048;           // 2 buffers x 2 x [16 heads][128 B]
constexpr uint32_t kSmRed = kSmP + 2 * 4096;         // [4][16] max, [4][16] sum
constexpr uint32_t kSmBar = kSmRed + 512;
enum : uint32_t {
  B_K_FULL = 0,                  // [2] per half
  B_K_EMPTY = B_K_FULL + 2,      // [2]
  B_V_EMPTY = B_K_EMPTY + 2,     // [3] per content group
  B_S_FULL = B_V_EMPTY + 3,
  B_S_EMPTY = B_S_FULL + 1,
  B_P_FULL = B_S_EMPTY + 1,      // [2] per P buffer
  B_PV_DONE = B_P_FULL + 2,      // [2] per tile parity
  B_Q_FULL = B_PV_DONE + 2,
  B_DRAIN_QK = B_Q_FULL + 1,
  B_DRAIN_PV = B_DRAIN_QK + 1,
  kNumBars = B_DRAIN_PV + 1
};
constexpr uint32_t kSmTslot = kSmBar + 8 * kNumBars;
constexpr uint32_t kSmAbort = kSmTslot + 4;
// in-kernel split plan: the scanner state, this worker's pieces (slot order)
// and its slot range
constexpr int kPlanCap = 64;  // pieces per worker <= batch <= kPlanCap
constexpr uint32_t kSmPlanSt = (kSmAbort + 12 + 15) & ~15u;
constexpr uint32_t kSmPieces = (kSmPlanSt + uint32_t(sizeof(PlanState)) + 15) & ~15u;
constexpr uint32_t kSmWr = kSmPieces + 16 * kPlanCap;
constexpr uint32_t kSmBytes = kSmWr + 8;
constexpr uint32_t kSmDyn = kSmBytes + 1024;
static_assert(kSmDyn <= 232448, "shared memory budget");

// Packed codes of one half-tile for one dequantization thread: two content
// groups (codes and scale/zero) and, in the first half, 32 RoPE channels
// (codes, scale/zero).
struct HalfCodes {
  uint32_t c0[8], c1[8];
  uint32_t sz0, sz1, rope[4], rsz;
};
__device__ __forceinline__ void ld_nc_v8(const void* p, uint32_t* r) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "l"(p));
}
__device__ __forceinline__ void ld_nc_v4(const void* p, uint32_t* r) {
  asm volatile("ld.global.nc.L1::no_allocate.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "l"(p));
}
__device__ __forceinline__ uint32_t ld_nc_b32(const void* p) {
  uint32_t a;
  asm volatile("ld.global.nc.L1::no_allocate.b32 %0, [%1];" : "=r"(a) : "l"(p));
  return a;
}
// Issue the loads of half h for token tt and column half dw of block `blk`
// (nullptr: nothing to load; the scale/zero words read as 0, which turns
// every dequantized value into +0 whatever the codes hold).
template <int kCBits>
__device__ __forceinline__ void load_half(HalfCodes& L, const uint8_t* blk, const Geom& G, int h,
                                          int dw, int tt) {
  if (blk == nullptr) {
    L.sz0 = L.sz1 = L.rsz = 0u;
    return;
  }
  const uint8_t* half = blk + h * G.half;
  const int g0 = 2 * dw;
  if (kCBits == 4) {
    ld_nc_v8(half + g0 * 2048 + tt * 32, L.c0);
    ld_nc_v8(half + (g0 + 1) * 2048 + tt * 32, L.c1);
  } else {
    ld_nc_v4(half + g0 * 1024 + tt * 16, L.c0);
    ld_nc_v4(half + (g0 + 1) * 1024 + tt * 16, L.c1);
  }
  L.sz0 = ld_nc_b32(half + G.sz_off + (g0 * 64 + tt) * 4);
  L.sz1 = ld_nc_b32(half + G.sz_off + ((g0 + 1) * 64 + tt) * 4);
  if (h == 0) {  // RoPE channels 32dw .. 32dw+31: the RoPE words of block half dw
    ld_nc_v4(blk + dw * G.half + G.rope_off + tt * 16, L.rope);
    L.rsz = ld_nc_b32(blk + G.rope_sz_off + tt * 4);
  }
}
// Channels 32*part .. 32*part+31 of one content group as 16 words of
// binary16 pairs (channel 2k low, 2k+1 high).
template <int kCBits>
__device__ __forceinline__ void dq_group_part(const uint32_t* c, uint32_t sz, int part,
                                              uint32_t* v) {
  __half2 s2, z2;
  split_sz(sz, s2, z2);
  if (kCBits == 4) {
#pragma unroll
    for (int w = 0; w < 4; ++w) dq_int4(c[4 * part + w], s2, z2, v + 4 * w);
  } else {
#pragma unroll
    for (int w = 0; w < 2; ++w) dq_int2(c[2 * part + w], s2, z2, v + 8 * w);
  }
}

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

template <int kCBits>
__global__ void __launch_bounds__(kThreads, 1) decode_tc16_kernel(DecodeArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // offset from the shared array itself, so that every access stays a
  // shared-memory access
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb0 = smem_u32(sm);
  auto BAR = [&](uint32_t i) { return sb0 + kSmBar + 8 * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kSmAbort);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int worker = blockIdx.x;
  constexpr bool kBF16 = kCBits == 16;  // uncompressed cache (rows converted to binary16)
  const Geom G = geom(kCBits == 4 ? QMLA_C4R4 : kCBits == 2 ? QMLA_C2R4 : QMLA_BF16);

  if (threadIdx.x == 0) {
    for (uint32_t h = 0; h < 2; ++h) {
      mbar_init(BAR(B_K_FULL + h), 8);  // every dequantization warp
      mbar_init(BAR(B_K_EMPTY + h), 1);
      mbar_init(BAR(B_P_FULL + h), 128);
    }
    for (uint32_t g = 0; g < 3; ++g) mbar_init(BAR(B_V_EMPTY + g), 1);
    mbar_init(BAR(B_S_FULL), 1);
    mbar_init(BAR(B_S_EMPTY), 4);  // every softmax warp
    mbar_init(BAR(B_PV_DONE + 0), 1);
    mbar_init(BAR(B_PV_DONE + 1), 1);
    mbar_init(BAR(B_Q_FULL), 128);
    mbar_init(BAR(B_DRAIN_QK), 1);
    mbar_init(BAR(B_DRAIN_PV), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kQkWarp) {
    tmem_alloc(sb0 + kSmTslot, kTmemCols);
    tmem_relinquish();
  } else if (warp == kPvWarp) {
    // The kernel is launched as a programmatic dependent of the one before it
    // (an append, say), so the set-up above overlaps that kernel's tail.  No
    // thread reads global memory before this wait: the other warps read only
    // after the barrier below.
    asm volatile("griddepcontrol.wait;" ::: "memory");
  }
  if (warp == kPvWarp && a.fused_plan) {
    // This worker's pieces, computed here by one warp scanning seq_lens with
    // the same functions as the planner kernel (worker 0 also publishes the
    // per-sequence merge table).  A worker's slots are consecutive, one per
    // sequence it touches, so they fit kPlanCap when batch <= kPlanCap.
    PlanState& st = *reinterpret_cast<PlanState*>(sm + kSmPlanSt);
    int4* plist = reinterpret_cast<int4*>(sm + kSmPieces);
    const int64_t N = plan_total(a);
    if (lane == 0) {
      st.total_blocks = N;
      st.carry_blocks = 0;
      st.carry_slots = 0;
      st.next_seq = 0;
    }
    __syncwarp();
    int first = -1, cnt = 0;
    while (plan_next(a, st, worker, worker == 0)) {
      const int n = st.n;
      if (n > 0) {
        if (first < 0) first = st.list[0].slot;
        if (lane < n) {
          const Piece pc = st.list[lane];
          const int k = pc.slot - first;
          if (k >= 0 && k < kPlanCap) plist[k] = make_int4(pc.b, pc.j0, pc.j1, 0);
        }
        cnt += n;
      }
      __syncwarp();  // the next chunk rewrites st.list
    }
    if (lane == 0) {
      if (cnt > kPlanCap) set_status(a.status, QMLA_STATUS_BAD_LEN);
      *reinterpret_cast<int2*>(sm + kSmWr) =
          (first < 0 || cnt > kPlanCap) ? make_int2(0, -1) : make_int2(first, first + cnt - 1);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *reinterpret_cast<volatile uint32_t*>(sm + kSmTslot);
  // the merge kernel that follows may be scheduled now (it waits for this
  // grid to complete before it reads anything)
  if (threadIdx.x == 0) griddep_launch_dependents();
  const int2 wr = a.fused_plan ? *reinterpret_cast<const int2*>(sm + kSmWr) : a.ws.wrange[worker];
  // piece s of this worker: (sequence, first block, end block)
  const int4* plist = reinterpret_cast<const int4*>(sm + kSmPieces);
  auto piece_at = [&](int s) -> int4 { return a.fused_plan ? plist[s - wr.x] : a.ws.pieces[s]; };

  if (warp == kQkWarp) {
    // ------------------------------------------------------------ QK^T issuer
    // k-step ks of every content chunk accumulates into partial sum ks, so the
    // four products of a chunk are independent of one another; RoPE k-steps
    // 0-1 come with half 0, 2-3 with half 1
    const uint32_t idesc = idesc_f16(128, kH, false, false);
    // operand descriptor; an offset inside the tile advances the 16-byte
    // address field (shared memory < 256 KB: no carry out of the field)
    const uint64_t dQ = smem_desc(sb0 + kSmQ, 16, 1024, kSwizzle128B);
    uint32_t t = 0, piece = 0;
    bool ok = true;
    for (int s = wr.x; ok && s <= wr.y; ++s) {
      const int4 pc = piece_at(s);
      if (pc.z <= pc.y) continue;
      if (!warp_ok(mbar_wait(BAR(B_Q_FULL), piece & 1u, abort_flag, kWaitNs))) break;
      ++piece;
      for (int jt = pc.y; jt < pc.z; jt += 2, ++t) {
        // the softmax has read the previous tile's scores
        if (!warp_ok(mbar_wait(BAR(B_S_EMPTY), (t & 1u) ^ 1u, abort_flag, kWaitNs))) {
          ok = false;
          break;
        }
#pragma unroll
        for (uint32_t h = 0; h < 2; ++h) {
          if (!warp_ok(mbar_wait(BAR(B_K_FULL + h), t & 1u, abort_flag, kWaitNs))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (uint32_t i = 0; i < 16; ++i) {  // content chunk 4h + i/4, k-step i%4
            const uint32_t c = 4 * h + (i >> 2), ks = i & 3u;
            mma_ts_warp(tbase + kColS + kH * ks, tbase + kColK + 32 * c + 8 * ks,
                        dQ + ((c * 2048 + 32 * ks) >> 4), idesc, c > 0 ? 1u : 0u);
          }
          // RoPE: the low-bit dequantization writes all of it with half 0
          // (half 1 is the one on the critical path), the BF16 one half each
          constexpr uint32_t kRopeSteps = kBF16 ? 2 : 4;
          if (kBF16 || h == 0) {
#pragma unroll
            for (uint32_t ks = kBF16 ? 2 * h : 0; ks < (kBF16 ? 2 * h : 0) + kRopeSteps; ++ks)
              mma_ts_warp(tbase + kColS + kH * ks, tbase + kColRope + 8 * ks,
                          dQ + ((8 * 2048 + 32 * ks) >> 4), idesc, 1u);
          }
          mma_commit_warp(BAR(B_K_EMPTY + h));
        }
        if (!ok) break;
        mma_commit_warp(BAR(B_S_FULL));
      }
    }
    mma_commit_warp(BAR(B_DRAIN_QK));
    if (lane == 0) wait_noabort(BAR(B_DRAIN_QK), 0);
    __syncwarp();
  } else if (warp == kPvWarp) {
    // ------------------------------------------------------------ P.V issuer
    // in two halves of the channels; half hv of tile t reads content group
    // (2t + hv) mod 3 and frees it for the dequantization when done
    const uint32_t idesc = idesc_f16(128, kH, true, false);
    const uint64_t dV = smem_desc(sb0 + kSmV, kChunk, 1024, kSwizzle128B);
    const uint64_t dP = smem_desc(sb0 + kSmP, 16, 1024, kSwizzle128B);
    uint32_t t = 0;
    bool ok = true;
    for (int s = wr.x; ok && s <= wr.y; ++s) {
      const int4 pc = piece_at(s);
      for (int jt = pc.y; jt < pc.z; jt += 2, ++t) {
        if (!warp_ok(mbar_wait(BAR(B_P_FULL + (t & 1u)), (t >> 1) & 1u, abort_flag, kWaitNs))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const bool first = (jt == pc.y);
        const uint32_t pbuf = (t & 1u) * 4096u;
#pragma unroll
        for (uint32_t hv = 0; hv < 2; ++hv) {
          const uint32_t grp = (2 * t + hv) % 3;
#pragma unroll
          for (uint32_t i = 0; i < 16; ++i) {  // k-step i/2, slice 2hv + i%2
            const uint32_t ks = i >> 1, m2 = i & 1u, mk = 2 * hv + m2;
            mma_ss_warp(tbase + kColO + kH * mk,
                        dV + ((grp * kGroup + 2 * m2 * kChunk + ks * 2048) >> 4),
                        dP + ((pbuf + (ks >> 2) * 2048 + (ks & 3u) * 32u) >> 4), idesc,
                        (first && ks == 0) ? 0u : 1u);
          }
          mma_commit_warp(BAR(B_V_EMPTY + grp));
        }
        mma_commit_warp(BAR(B_PV_DONE + (t & 1u)));
      }
    }
    mma_commit_warp(BAR(B_DRAIN_PV));
    if (lane == 0) wait_noabort(BAR(B_DRAIN_PV), 0);
    __syncwarp();
  } else if (warp >= kSoftmaxWarp0 && warp < kDequantWarp0) {
    // ------------------------------------------------------------ softmax
    const uint32_t quad = uint32_t(warp & 3);
    const int r = int(quad * 32) + lane;  // token row of S^T / channel row of O^T
    const int sw = warp - kSoftmaxWarp0;  // 0..3
    const uint32_t lane_base = (quad * 32u) << 16;
    const float c2 = a.scale * 1.4426950408889634f;
    float* red_max = reinterpret_cast<float*>(sm + kSmRed);
    float* red_sum = red_max + 4 * kH;
    // Q^T of sequence b: 16 heads x 576 channels, binary16, SW128 K-major.
    // A thread's nine 16-byte segments are all loaded (q_load) before any is
    // converted and stored (q_store), so staging waits for one load latency,
    // and other work can run between the two halves.
    constexpr int kSeg = kH * 72 / 128;  // 8-channel segments per thread
    const int qi0 = threadIdx.x - kSoftmaxWarp0 * 32;
    auto q_load = [&](int b, uint4 (&qv)[kSeg]) {
#pragma unroll
      for (int k = 0; k < kSeg; ++k) {
        const int i = qi0 + 128 * k, h = i / 72, sgm = i % 72;
        const __nv_bfloat16* src =
            (sgm < 64) ? a.q_c + (int64_t(b) * kH + h) * kDc + sgm * 8
                       : a.q_r + (int64_t(b) * kH + h) * kDr + (sgm - 64) * 8;
        qv[k] = *reinterpret_cast<const uint4*>(src);
      }
    };
    auto q_store = [&](const uint4 (&qv)[kSeg]) {
      bool bad = false;  // a query value beyond binary16's range
#pragma unroll
      for (int k = 0; k < kSeg; ++k) {
        const int i = qi0 + 128 * k, h = i / 72, sgm = i % 72;
        const uint32_t in[4] = {qv[k].x, qv[k].y, qv[k].z, qv[k].w};
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          o[e] = pack_half2(__uint_as_float(in[e] << 16), __uint_as_float(in[e] & 0xffff0000u));
          bad |= (o[e] & 0x7fffu) == 0x7c00u || (o[e] & 0x7fff0000u) == 0x7c000000u;
        }
        const int c = sgm >> 3, g = sgm & 7;
        unsigned char* row = sm + kSmQ + c * 2048 + (h >> 3) * 1024 + (h & 7) * 128;
        *reinterpret_cast<uint4*>(row + ((g ^ (h & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
      }
      if (bad) set_status(a.status, QMLA_STATUS_BAD_QUERY);
      fence_proxy_async_smem();
      mbar_arrive(BAR(B_Q_FULL));
    };
    uint32_t t = 0;
    bool ok = true;
    bool q_staged = false;  // the current piece's Q is already in shared memory
    for (int s = wr.x; ok && s <= wr.y; ++s) {
      const int4 pc = piece_at(s);
      const int b = pc.x;
      if (pc.z <= pc.y) {
        q_staged = false;
        for (int i = threadIdx.x - kSoftmaxWarp0 * 32; i < kH * kDc; i += 128)
          a.ws.part_o[int64_t(s) * kH * kDc + i] = 0.f;
        if (r < kH) a.ws.part_lse[int64_t(s) * kH + r] = -INFINITY;
        continue;
      }
      const int L = seq_len_clamped(a, b);
      // the QK products of the previous piece completed before its epilogue
      if (!q_staged) {
        uint4 qv[kSeg];
        q_load(b, qv);
        q_store(qv);
      }
      const int4 pn = (s < wr.y) ? piece_at(s + 1) : make_int4(0, 0, 0, 0);  // next piece
      float m_used[kH], l_part[kH];
#pragma unroll
      for (int h = 0; h < kH; ++h) {
        m_used[h] = -INFINITY;
        l_part[h] = 0.0f;
      }
      uint32_t vmask = 0;
      for (int jt = pc.y; jt < pc.z; jt += 2, ++t) {
        if (((jt - pc.y) & 31) == 0) vmask = valid_mask(a, b, jt, pc.z);
        if (jt + 2 >= pc.z && pn.z > pn.y) {
          // last tile: the next piece's queries into L2 (18 KB, 144 lines of
          // 128 bytes), to be staged during this piece's epilogue
          prefetch_l2(reinterpret_cast<const char*>(a.q_c + int64_t(pn.x) * kH * kDc) + 128 * qi0);
          if (qi0 < 16)
            prefetch_l2(reinterpret_cast<const char*>(a.q_r + int64_t(pn.x) * kH * kDr) + 128 * qi0);
        }
        // validity of this lane's token row
        const int bi = r >> 6, jj = jt + bi;
        const bool blk_ok = jj < pc.z && ((vmask >> ((jj - pc.y) & 31)) & 1u);
        const bool row_ok = blk_ok && (r & 63) < min(kT, L - jj * kT);
        // scores of tile t; P buffer t&1 was last read by the P.V products of
        // tile t-2 (PV_DONE[b] completes for tiles b, b+2, ...), so the
        // softmax of tile t overlaps the P.V products of tile t-1
        bool got = warp_ok(mbar_wait(BAR(B_S_FULL), t & 1u, abort_flag, kWaitNs));
        if (got && t > 1)
          got = warp_ok(mbar_wait(BAR(B_PV_DONE + (t & 1u)), ((t >> 1) & 1u) ^ 1u, abort_flag,
                                  kWaitNs));
        float sv[kH];
#pragma unroll
        for (int h = 0; h < kH; ++h) sv[h] = -INFINITY;
        if (got) {
          tc_fence_after();
          uint32_t q0[32], q1[32];
          tmem_ld32(tbase + lane_base + kColS, q0);
          tmem_ld32(tbase + lane_base + kColS + 32, q1);
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR(B_S_EMPTY));
#pragma unroll
          for (int h = 0; h < kH; ++h) {
            const float v = (__uint_as_float(q0[h]) + __uint_as_float(q0[16 + h])) +
                            (__uint_as_float(q1[h]) + __uint_as_float(q1[16 + h]));
            sv[h] = row_ok ? v * c2 : -INFINITY;
          }
        }
        // lazy rescale: the per-head maxima are only reduced when some score
        // exceeds the maximum in use by more than kLazy; every thread then takes
        // the same decisions.  All four warps take the same barriers whatever
        // their waits returned: a failed wait forces the rare path, which
        // checks for it.
        bool over = !got;
#pragma unroll
        for (int h = 0; h < kH; ++h) over |= sv[h] > m_used[h] + kLazy;
        if (named_bar_or(1, 128, over)) {
          if (named_bar_or(1, 128, !got)) {
            ok = false;
            break;
          }
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
          float alpha[kH];
#pragma unroll
          for (int h = 0; h < kH; h += 4) {
            const float4 v0 = *reinterpret_cast<const float4*>(red_max + 0 * kH + h);
            const float4 v1 = *reinterpret_cast<const float4*>(red_max + 1 * kH + h);
            const float4 v2 = *reinterpret_cast<const float4*>(red_max + 2 * kH + h);
            const float4 v3 = *reinterpret_cast<const float4*>(red_max + 3 * kH + h);
            const float mt[4] = {fmaxf(fmaxf(v0.x, v1.x), fmaxf(v2.x, v3.x)),
                                 fmaxf(fmaxf(v0.y, v1.y), fmaxf(v2.y, v3.y)),
                                 fmaxf(fmaxf(v0.z, v1.z), fmaxf(v2.z, v3.z)),
                                 fmaxf(fmaxf(v0.w, v1.w), fmaxf(v2.w, v3.w))};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const bool need = mt[e] > m_used[h + e] + kLazy;
              alpha[h + e] = need ? ex2_approx(m_used[h + e] - mt[e]) : 1.0f;
              if (need) m_used[h + e] = mt[e];
            }
          }
#pragma unroll
          for (int h = 0; h < kH; ++h) l_part[h] *= alpha[h];
          if (jt > pc.y) {  // O^T holds earlier tiles of this piece
            // the P.V products of tile t-1 must have landed in O^T first
            // (uniform: every softmax thread is in this branch)
            if (!warp_ok(mbar_wait(BAR(B_PV_DONE + ((t - 1) & 1u)), ((t - 1) >> 1) & 1u,
                                   abort_flag, kWaitNs))) {
              ok = false;  // abort raised: every role unwinds
            }
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
          // red_max is rewritten only after every softmax thread has passed
          // this point: the next tile's scores need this tile's P first
        }
        // P^T[h][r] = 2^(s - m) as binary16 into the SW128 K-major B tile
        unsigned char* preg = sm + kSmP + (t & 1u) * 4096u + (r >> 6) * 2048;
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
        mbar_arrive(BAR(B_P_FULL + (t & 1u)));
      }
      // every softmax warp reaches this barrier (the loop is left together)
      if (named_bar_or(1, 128, !ok)) {
        ok = false;
        break;
      }
      // epilogue: row sums over the 128 lanes, normalized partial O, LSE
      const bool got = warp_ok(mbar_wait(BAR(B_PV_DONE + ((t - 1) & 1u)), ((t - 1) >> 1) & 1u,
                                         abort_flag, kWaitNs));
      if (named_bar_or(1, 128, !got)) break;
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
      // The next piece's queries (from L2): every QK product of this piece,
      // the only reader of Q^T, completed before its last scores were read;
      // the next piece's first QK then runs while the partial O is written.
      q_staged = pn.z > pn.y;
      if (q_staged) {
        uint4 qv[kSeg];
        q_load(pn.x, qv);
        q_store(qv);
      }
      // 1/l with the approximate reciprocal (1 ulp): the exact one costs a
      // long instruction sequence per head on the piece's critical path
      float inv[kH];
      float l_r = 0.0f, m_r = 0.0f;  // row sum and maximum of head r (threads r < 16)
#pragma unroll
      for (int h = 0; h < kH; ++h) {
        const float l = red_sum[h] + red_sum[kH + h] + red_sum[2 * kH + h] + red_sum[3 * kH + h];
        inv[h] = l > 0.0f ? rcp_approx(l) : 0.0f;
        if (r == h) {
          l_r = l;
          m_r = m_used[h];
        }
      }
      if (r < kH)
        a.ws.part_lse[int64_t(s) * kH + r] =
            l_r > 0.0f ? (m_r + log2f(l_r)) * 0.6931471805599453f : -INFINITY;
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
  } else if (warp >= kDequantWarp0 && kBF16) {
    // ------------------------------------------------------------ BF16 rows
    // The same split as the dequantization below (lane quarter q, column
    // half dw; content groups 4h+2dw, 4h+2dw+1 and RoPE channels
    // 32h+16dw .. +15 of half h), but the rows only change type: each item
    // (a 64-channel group row of 128 B, or 16 RoPE channels) is loaded one
    // item ahead, converted bfloat16 -> binary16 (exact for cache values in
    // binary16's normal range) and stored to tensor memory and shared memory.
    // Binary16 rather than bfloat16 operands because P is the other operand
    // of P.V: P in bfloat16 (8 significant bits) misses the 1e-2 output
    // tolerance at long contexts, P in binary16 (11) does not.
    const int q = warp & 3, dw = (warp - kDequantWarp0) >> 2;
    const int r = 32 * q + lane, bi = q >> 1, tt = r & 63;
    const uint32_t lane_base = uint32_t(32 * q) << 16;
    const uint32_t vrow_off = uint32_t((r >> 3) * 1024 + (r & 7) * 128);
    const int sw7 = r & 7;
    uint32_t t = 0;
    bool ok = true;
    for (int s = wr.x; ok && s <= wr.y; ++s) {
      const int4 pc = piece_at(s);
      if (pc.z <= pc.y) continue;
      const int L = seq_len_clamped(a, pc.x);
      const int32_t* btab = a.block_table + int64_t(pc.x) * a.max_blocks_per_seq;
      // rows of this thread's token in the tile starting at jt (nullptr: none
      // or a bad block id, read as zeros)
      auto tile_rows = [&](int jt) -> const uint8_t* {
        const int j = jt + bi;
        if (j >= pc.z) return nullptr;
        const int32_t blk = btab[j];
        if (blk < 0 || blk >= a.num_blocks) {
          if (lane == 0) set_status(a.status, QMLA_STATUS_BAD_BLOCK);
          return nullptr;
        }
        return (tt < min(kT, L - j * kT)) ? a.blocks + int64_t(blk) * G.block : nullptr;
      };
      // item k of half h: 0, 1 content groups 2dw+k; 2 the RoPE segment
      auto load_item = [&](const uint8_t* blk, int h, int k, uint32_t (&w)[32]) {
        if (blk == nullptr) {
#pragma unroll
          for (int e = 0; e < 32; ++e) w[e] = 0u;
          return;
        }
        const uint8_t* half = blk + h * G.half;
        if (k < 2) {
          const uint8_t* row = half + ((2 * dw + k) * 64 + tt) * 128;
#pragma unroll
          for (int i = 0; i < 4; ++i) ld_nc_v8(row + 32 * i, w + 8 * i);
        } else {
          ld_nc_v8(half + G.rope_off + tt * 64 + dw * 32, w);
        }
      };
      const uint8_t* rows_cur = tile_rows(pc.y);
      uint32_t nxt[32];
      load_item(rows_cur, 0, 0, nxt);
      for (int jt = pc.y; jt < pc.z; jt += 2, ++t) {
        const uint8_t* rows_next = tile_rows(jt + 2);
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          const uint32_t hn = 2 * t + uint32_t(h), grp = hn % 3;
          bool got = mbar_wait(BAR(B_K_EMPTY + h), (t & 1u) ^ 1u, abort_flag, kWaitNs);
          got = got && mbar_wait(BAR(B_V_EMPTY + grp), ((hn / 3) & 1u) ^ 1u, abort_flag, kWaitNs);
          if (!warp_ok(got)) {
            ok = false;
            break;
          }
          unsigned char* vgrp = sm + kSmV + grp * kGroup + vrow_off;
#pragma unroll 1
          for (int k = 0; k < 3; ++k) {
            uint32_t cur[32];
#pragma unroll
            for (int e = 0; e < 32; ++e)
              cur[e] = pack_half2(__uint_as_float(nxt[e] << 16),
                                  __uint_as_float(nxt[e] & 0xffff0000u));
            // the next item: this half's next one, else the next half's first
            if (k < 2)
              load_item(rows_cur, h, k + 1, nxt);
            else if (h == 0)
              load_item(rows_cur, 1, 0, nxt);
            else
              load_item(rows_next, 0, 0, nxt);
            if (k < 2) {
              const int c = 4 * h + 2 * dw + k;
              tmem_st32(tbase + lane_base + kColK + 32 * c, cur);
              unsigned char* row = vgrp + (c & 3) * kChunk;
#pragma unroll
              for (int g = 0; g < 8; ++g)
                *reinterpret_cast<uint4*>(row + ((g ^ sw7) << 4)) =
                    make_uint4(cur[4 * g], cur[4 * g + 1], cur[4 * g + 2], cur[4 * g + 3]);
            } else {
              uint32_t v[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) v[e] = cur[e];
              tmem_st8(tbase + lane_base + kColRope + 16 * h + 8 * dw, v);
            }
          }
          tmem_wait_st();
          fence_proxy_async_smem();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR(B_K_FULL + h));
        }
        if (!ok) break;
        rows_cur = rows_next;
      }
    }
  } else if (warp >= kDequantWarp0) {
    // ------------------------------------------------------------ dequant
    // warp: lane quarter q (tensor-memory lanes 32q..32q+31 = token rows) and
    // column half dw.  Rows 0-63 come from the tile's first block, 64-127 from
    // its second.  For half h the warp dequantizes content groups 4h+2dw and
    // 4h+2dw+1 of its tokens, and with half 0 also RoPE channels 32dw ..
    // 32dw+31, which keeps half 1 -- the half that waits for the previous
    // tile's P.V and holds up this tile's QK -- short.  The loads of the next
    // half-tile of the piece are issued before the current one is processed.
    const int q = warp & 3, dw = (warp - kDequantWarp0) >> 2;
    const int r = 32 * q + lane, bi = q >> 1, tt = r & 63;
    const uint32_t lane_base = uint32_t(32 * q) << 16;
    const uint32_t vrow_off = uint32_t((r >> 3) * 1024 + (r & 7) * 128);  // row r of a chunk
    const int sw7 = r & 7;
    uint32_t t = 0;  // tiles of this worker before the current piece
    bool ok = true;
    for (int s = wr.x; ok && s <= wr.y; ++s) {
      const int4 pc = piece_at(s);
      if (pc.z <= pc.y) continue;
      const int L = seq_len_clamped(a, pc.x);
      const int32_t* btab = a.block_table + int64_t(pc.x) * a.max_blocks_per_seq;
      // block ids of blocks jb0 .. jb0+63 of the piece, one per lane in two
      // registers; the next 32 are loaded 16 tiles before they are needed, so
      // no code load waits on a block-table load
      int jb0 = pc.y;
      int32_t ids_a = (jb0 + lane < pc.z) ? btab[jb0 + lane] : -1;
      int32_t ids_b = (jb0 + 32 + lane < pc.z) ? btab[jb0 + 32 + lane] : -1;
      // block of this thread's rows in the tile starting at jt (nullptr: none,
      // or a bad block id), and the number of valid token rows in it
      auto tile_block = [&](int jt, int& nvalid) -> const uint8_t* {
        const int j = jt + bi, k = j - jb0;  // k < 64, the same in the whole warp
        const int32_t va = __shfl_sync(0xffffffffu, ids_a, k & 31);
        const int32_t vb = __shfl_sync(0xffffffffu, ids_b, k & 31);
        nvalid = 0;
        if (j >= pc.z) return nullptr;
        const int32_t blk = k < 32 ? va : vb;
        if (blk < 0 || blk >= a.num_blocks) {
          if (lane == 0) set_status(a.status, QMLA_STATUS_BAD_BLOCK);
          return nullptr;
        }
        nvalid = min(kT, L - j * kT);
        return a.blocks + int64_t(blk) * G.block;
      };
      int nv_cur;
      const uint8_t* blk_cur = tile_block(pc.y, nv_cur);
      HalfCodes cur, nxt;
      load_half<kCBits>(nxt, (blk_cur && tt < nv_cur) ? blk_cur : nullptr, G, 0, dw, tt);
      for (int jt = pc.y; jt < pc.z; jt += 2, ++t) {
        if (jt >= jb0 + 32) {
          jb0 += 32;
          ids_a = ids_b;
          ids_b = (jb0 + 32 + lane < pc.z) ? btab[jb0 + 32 + lane] : -1;
        }
        int nv_next = 0;
        const uint8_t* blk_next = tile_block(jt + 2, nv_next);
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          cur = nxt;
          if (h == 0)
            load_half<kCBits>(nxt, (blk_cur && tt < nv_cur) ? blk_cur : nullptr, G, 1, dw, tt);
          else
            load_half<kCBits>(nxt, (blk_next && tt < nv_next) ? blk_next : nullptr, G, 0, dw, tt);
          const uint32_t hn = 2 * t + uint32_t(h), grp = hn % 3;
          bool got = mbar_wait(BAR(B_K_EMPTY + h), (t & 1u) ^ 1u, abort_flag, kWaitNs);
          got = got && mbar_wait(BAR(B_V_EMPTY + grp), ((hn / 3) & 1u) ^ 1u, abort_flag, kWaitNs);
          if (!warp_ok(got)) {
            ok = false;
            break;
          }
          unsigned char* vgrp = sm + kSmV + grp * kGroup + vrow_off;
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int c = 4 * h + 2 * dw + cc;
            unsigned char* row = vgrp + (c & 3) * kChunk;
            // 32 channels (16 words) at a time
#pragma unroll
            for (int part = 0; part < 2; ++part) {
              uint32_t v[16];
              dq_group_part<kCBits>(cc ? cur.c1 : cur.c0, cc ? cur.sz1 : cur.sz0, part, v);
              tmem_st16(tbase + lane_base + kColK + 32 * c + 16 * part, v);
#pragma unroll
              for (int g = 0; g < 4; ++g)
                *reinterpret_cast<uint4*>(row + (((4 * part + g) ^ sw7) << 4)) =
                    make_uint4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
            }
          }
          if (h == 0) {
            // RoPE channels 32dw .. 32dw+31 (INT4)
            __half2 s2, z2;
            split_sz(cur.rsz, s2, z2);
            uint32_t v[16];
#pragma unroll
            for (int w = 0; w < 4; ++w) dq_int4(cur.rope[w], s2, z2, v + 4 * w);
            tmem_st16(tbase + lane_base + kColRope + 16 * dw, v);
          }
          tmem_wait_st();
          fence_proxy_async_smem();
          tc_fence_before();
          __syncwarp();
          // (the test hook withholds the first half's arrival of this worker)
          if (lane == 0 && !(a.withhold && t == 0 && h == 0)) mbar_arrive(BAR(B_K_FULL + h));
        }
        if (!ok) break;
        blk_cur = blk_next;
        nv_cur = nv_next;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) set_status(a.status, QMLA_STATUS_TIMEOUT);
  if (warp == kQkWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_decode_tc16(const DecodeArgs& a, cudaStream_t stream) {
  static int smem_attr_done[kMaxDevices], smem_attr_done2[kMaxDevices],
      smem_attr_done_bf16[kMaxDevices];
  // Up to kPlanCap sequences the kernel plans its own pieces; beyond that a
  // worker may touch more sequences than its shared-memory list holds, and
  // the planner kernel writes the plan to the workspace instead.
  DecodeArgs b = a;
  b.fused_plan = a.batch <= kPlanCap ? 1 : 0;
  // A second piece costs a worker about three blocks of context (the
  // queries' staging, the pipeline refill and the epilogue).
  b.piece_cost = 3;
  cudaError_t e = cudaSuccess;
  if (!b.fused_plan) {
    e = launch_plan(b, stream);
    if (e != cudaSuccess) return e;
  }
  auto kernel = (a.fmt == QMLA_C4R4)   ? decode_tc16_kernel<4>
                : (a.fmt == QMLA_C2R4) ? decode_tc16_kernel<2>
                                       : decode_tc16_kernel<16>;
  e = ensure_smem_attr(kernel, int(kSmDyn),
                       a.fmt == QMLA_C4R4   ? smem_attr_done
                       : a.fmt == QMLA_C2R4 ? smem_attr_done2
                                            : smem_attr_done_bf16);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(a.workers));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmDyn;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, b);
}

}  // namespace qmla
