// decode_tc.cu - tensor-core (tcgen05) decode over the low-bit paged cache,
// 128 absorbed query heads.
//
// The "native low-bit MLA attention kernel" of "QuantMLA: INT4 (and INT2) for
// both halves of the MLA cache" (flowchart node "Low-bit kernel: dequant
// inside attention"; "Key findings"): packed blocks are unpacked and
// dequantized in shared memory and consumed directly by the tensor cores.
//
// Work split.  O for 128 heads x 512 channels in binary32 fills the whole
// 512-column tensor memory of an SM, so one work unit runs on a cluster of
// two CTAs: CTA r owns content channels 256r..256r+255 and RoPE channels
// 32r..32r+31, which is exactly one contiguous half of every cache block.
//   QK : S_r[128 heads x 64 tok] = Qc_r (A, tensor memory) x K_r^T (B, smem)
//                                + Qr_r (A, smem)          x R_r^T (B, smem)
//        the softmax of heads 64r..64r+63 runs on CTA r: each CTA sends the
//        partial scores of the other CTA's heads (16 KB per tile) through
//        cluster shared memory with asynchronous remote stores that complete
//        on the receiver's mbarrier, adds the partials it receives for its
//        own heads, and sends back those heads' P rows (binary16, 8 KB) with
//        their rescale factors, so both CTAs end up with the full P tile;
//   PV : O_r[128 x 256] += P (A, smem) x C_r (B, the same dequantized smem
//        tile read MN-major).
// Tensor memory per CTA: O_r cols 0-255, Qc_r cols 256-383, S double buffer
// cols 384-511.
//
// Warp roles (14 warps): 0 bulk-copy producer, 1 MMA issuer, 2-5 softmax
// (thread = head), 6-13 dequantization.  Dequantized operands are binary16
// (code*scale + zero, exact by construction of the quantizer's grid);
// queries are converted bf16 -> binary16; accumulation is binary32.
//
// The same kernel serves the uncompressed BF16 cache, the baseline the
// low-bit formats are compared with: nothing is dequantized; the
// "dequantization" warps load each tile's rows straight from HBM (256-bit
// loads, one tile ahead), convert them bfloat16 -> binary16 (exact for cache
// values in binary16's normal range; P, the other operand of P.V, needs
// binary16's 11 significant bits at long contexts) and store them into the
// swizzled operand tile; the producer warp has nothing to do.
// The softmax is online in base 2 with lazy rescaling: O and l are rescaled
// only when a tile's maximum exceeds the running one by more than 8
// (P <= 256).  Every wait is bounded in time; on timeout the CTA raises an
// abort flag, all roles unwind, and QMLA_STATUS_TIMEOUT is reported.

#include <cfloat>

#include "tc_common.cuh"

namespace qmla {
namespace tc {
// ---------------------------------------------------------------- planner
// One warp writes the split plan: merge table, piece descriptors per slot
// and the slot range of each worker.
__global__ void __launch_bounds__(32) plan_kernel(DecodeArgs a) {
  const int lane = threadIdx.x;
  const int64_t N = plan_total(a);
  const int64_t P = plan_workers(N, a.workers);
  // a worker that owns only piece-cost blocks (or none) has no piece
  for (int64_t w = lane; w < a.workers; w += 32) a.ws.wrange[w] = make_int2(0, -1);
  __syncwarp();
  int64_t carry_blocks = 0;
  int carry_slots = 0;
  for (int b0 = 0; b0 < a.batch; b0 += 32) {
    const int b = b0 + lane;
    const int nb = (b < a.batch) ? seq_blocks(a, b, false) : 0;
    const int ext = plan_extent(a, nb);
    const int incl = warp_incl_scan(ext);
    const int64_t S = carry_blocks + (incl - ext) + a.piece_cost;  // first real block
    int np = 0;
    int64_t pf = 0;
    if (nb > 0) {
      pf = plan_owner(S, N, P);
      np = int(plan_owner(S + nb - 1, N, P) - pf + 1);
    }
    const int np_incl = warp_incl_scan(np);
    const int base = carry_slots + (np_incl - np);
    if (b < a.batch) a.ws.seq_table[b] = make_int2(base, np);
    for (int i = 0; i < np; ++i) {
      const int64_t w = pf + i;
      const int64_t w0 = plan_start(w, N, P), w1 = plan_start(w + 1, N, P);
      const int j0 = int(max(w0 - S, int64_t(0))), j1 = int(min(w1 - S, int64_t(nb)));
      a.ws.pieces[base + i] = make_int4(b, j0, j1, 0);
      // the worker's first piece: its range starts inside this sequence's
      // extent (piece cost included); its last: the range ends before the
      // next sequence's first real block
      if (w0 >= S - a.piece_cost) a.ws.wrange[w].x = base + i;
      if (w1 <= S + nb + a.piece_cost) a.ws.wrange[w].y = base + i;
    }
    carry_blocks += __shfl_sync(0xffffffffu, incl, 31);
    carry_slots += __shfl_sync(0xffffffffu, np_incl, 31);
  }
}

}  // namespace tc

// The planner kernel is defined once, here, for both tensor-core decodes.
cudaError_t launch_plan(const DecodeArgs& a, cudaStream_t stream) {
  tc::plan_kernel<<<1, 32, 0, stream>>>(a);
  return cudaGetLastError();
}

namespace {

using namespace ptx;
using namespace tc;

// ---------------------------------------------------------------- layout
constexpr int kThreads = 448;
constexpr int kMmaWarp = 1;
constexpr int kSoftmaxWarp0 = 2;
constexpr int kDequantWarp0 = 6;
constexpr int kDequantThreads = 256;

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0, kColQ = 256, kColS = 384;

constexpr uint32_t kSmQr = 0;                        // [128 heads][128 B] SW128, 16 KB
constexpr uint32_t kSmK = 16384;                     // 2 x K tile
constexpr uint32_t kChunk = 8192;                    // [64 tok][64 ch] fp16 SW128
constexpr uint32_t kKTile = 5 * kChunk;              // 4 content chunks + RoPE chunk
constexpr uint32_t kStages = 4;                      // bulk-copy ring depth
constexpr uint32_t kSmStage = kSmK + 2 * kKTile;     // kStages x staging
constexpr uint32_t kStage = 10240 + 256;             // largest half + RoPE scale/zero
constexpr uint32_t kSmX = kSmStage + kStages * kStage;  // 2 x received partial scores
constexpr uint32_t kX = 64 * 64 * 4;                 // [64 own heads][64 tok] fp32
constexpr uint32_t kSmPt = kSmX + 2 * kX;            // 2 x P tile
constexpr uint32_t kPt = 128 * 128;                  // [128 heads][64 tok] fp16 SW128
constexpr uint32_t kSmAlpha = kSmPt + 2 * kPt;       // 2 x [64] received rescale factors
constexpr uint32_t kSmLx = kSmAlpha + 2 * 256;       // [64] received row sums (per piece)
constexpr uint32_t kPx = 64 * 128 + 64 * 4;          // P rows + rescale factors per tile
constexpr uint32_t kSmBar = kSmLx + 256;
constexpr uint32_t kNumBars = 27;
constexpr uint32_t kSmTslot = kSmBar + 8 * kNumBars;
constexpr uint32_t kSmAbort = kSmTslot + 4;
constexpr uint32_t kSmBytes = kSmAbort + 60;
constexpr uint32_t kSmDyn = kSmBytes + 1024;         // slack for 1 KB alignment

// barrier indices
enum : uint32_t {
  B_STAGE_FULL = 0, B_STAGE_EMPTY = 4, B_K_FULL = 8, B_K_EMPTY = 10, B_S_FULL = 12,
  B_P_FULL = 14, B_PV_DONE = 16, B_X_FULL = 18, B_X_EMPTY = 20, B_Q_FULL = 22, B_DRAIN = 23,
  B_PX_FULL = 24, B_LX_FULL = 26
};
static_assert(kSmPt % 1024 == 0, "SW128 operand tiles are 1 KB aligned");

__device__ __forceinline__ void ld_nc_v8(const void* p, uint32_t* r) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "l"(p));
}

// ---------------------------------------------------------------- kernel
template <bool kBF16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_tc128_kernel(DecodeArgs a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb0 = smem_u32(sm);
  auto BAR = [&](uint32_t i) { return sb0 + kSmBar + 8 * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kSmAbort);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
  const int pair = blockIdx.x >> 1;
  const Geom G = geom(a.fmt);

  if (threadIdx.x == 0) {
    for (uint32_t i = 0; i < kStages; ++i) {
      mbar_init(BAR(B_STAGE_FULL + i), 1);
      mbar_init(BAR(B_STAGE_EMPTY + i), kDequantThreads / 32);
    }
    for (uint32_t i = 0; i < 2; ++i) {
      mbar_init(BAR(B_K_FULL + i), kDequantThreads / 32);
      mbar_init(BAR(B_K_EMPTY + i), 1);
      mbar_init(BAR(B_S_FULL + i), 1);
      mbar_init(BAR(B_P_FULL + i), 128);
      mbar_init(BAR(B_PV_DONE + i), 1);
      mbar_init(BAR(B_X_FULL + i), 1);
      mbar_init(BAR(B_X_EMPTY + i), 64);  // the peer's 64 owning threads
      mbar_init(BAR(B_PX_FULL + i), 1);
    }
    mbar_init(BAR(B_Q_FULL), 128);
    mbar_init(BAR(B_DRAIN), 1);
    mbar_init(BAR(B_LX_FULL), 1);
    // the first exchanges are expected before the peer can send them
    mbar_arrive_expect_tx(BAR(B_X_FULL + 0), kX);
    mbar_arrive_expect_tx(BAR(B_X_FULL + 1), kX);
    mbar_arrive_expect_tx(BAR(B_PX_FULL + 0), kPx);
    mbar_arrive_expect_tx(BAR(B_PX_FULL + 1), kPx);
    mbar_arrive_expect_tx(BAR(B_LX_FULL), 256);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(sb0 + kSmTslot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers are initialized before any remote arrive
  tc_fence_after();
  const uint32_t tbase = *reinterpret_cast<volatile uint32_t*>(sm + kSmTslot);
  const int2 wr = a.ws.wrange[pair];

  if (warp == 0 && !kBF16) {
    // ------------------------------------------------------------ producer
    uint32_t t = 0;
    bool ok = true;
    for (int s = wr.x; ok && s <= wr.y; ++s) {
      const int4 pc = a.ws.pieces[s];
      for (int jb = pc.y; ok && jb < pc.z; jb += 32) {
        const int n = min(32, pc.z - jb);
        const int32_t my_blk =
            (lane < n) ? a.block_table[int64_t(pc.x) * a.max_blocks_per_seq + jb + lane] : -1;
        for (int k = 0; k < n; ++k, ++t) {
          const int32_t blk = __shfl_sync(0xffffffffu, my_blk, k);
          bool got = true;
          if (lane == 0) {
            const uint32_t st = t % kStages, par = (t / kStages) & 1u;
            got = mbar_wait(BAR(B_STAGE_EMPTY + st), par ^ 1u, abort_flag, kWaitNs);
            if (got) {
              const uint32_t dst = sb0 + kSmStage + st * kStage;
              if (blk >= 0 && blk < a.num_blocks) {
                const unsigned char* src = a.blocks + int64_t(blk) * G.block;
                mbar_arrive_expect_tx(BAR(B_STAGE_FULL + st), uint32_t(G.half) + 256u);
                bulk_g2s(dst, src + rank * G.half, uint32_t(G.half), BAR(B_STAGE_FULL + st));
                bulk_g2s(dst + G.half, src + G.rope_sz_off, 256u, BAR(B_STAGE_FULL + st));
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
    // copies still in flight must land before the CTA can exit
    if (lane == 0)
      for (uint32_t u = (t >= kStages ? t - kStages : 0); u < t; ++u)
        wait_noabort(BAR(B_STAGE_FULL + u % kStages), (u / kStages) & 1u);
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop converged and an elected lane issues each
    // instruction (single-lane issue behind waits and branches costs several
    // times more per MMA).
    const uint32_t idesc_qk = idesc_f16(128, 64, false, false);
    const uint32_t idesc_pv = idesc_f16(128, 256, false, true);
    // operand descriptors; an offset advances the 16-byte address field
    const uint64_t dKt = smem_desc(sb0 + kSmK, 16, 1024, kSwizzle128B);
    const uint64_t dCt = smem_desc(sb0 + kSmK, kChunk, 1024, kSwizzle128B);
    const uint64_t dQr = smem_desc(sb0 + kSmQr, 16, 1024, kSwizzle128B);
    const uint64_t dPt = smem_desc(sb0 + kSmPt, 16, 1024, kSwizzle128B);
    uint32_t t = 0, piece = 0;
    bool ok = true;
    auto issue_pv = [&](uint32_t tt, bool first) {
      const uint32_t sb = tt & 1u;
#pragma unroll
      for (uint32_t kk = 0; kk < 4; ++kk) {
        mma_ss_warp(tbase + kColO, dPt + ((sb * kPt + kk * 32) >> 4),
                    dCt + ((sb * kKTile + kk * 2048) >> 4), idesc_pv,
                    (first && kk == 0) ? 0u : 1u);
      }
      mma_commit_warp(BAR(B_PV_DONE + sb));
      mma_commit_warp(BAR(B_K_EMPTY + sb));
    };
    for (int s = wr.x; ok && s <= wr.y; ++s) {
      const int4 pc = a.ws.pieces[s];
      if (pc.z <= pc.y) continue;
      if (!warp_ok(mbar_wait(BAR(B_Q_FULL), piece & 1u, abort_flag, kWaitNs))) break;
      ++piece;
      tc_fence_after();
      for (int j = pc.y; j < pc.z; ++j, ++t) {
        const uint32_t sb = t & 1u, par = (t >> 1) & 1u;
        bool got = mbar_wait(BAR(B_K_FULL + sb), par, abort_flag, kWaitNs);
        got = got && (t < 2 || mbar_wait(BAR(B_PV_DONE + sb), par ^ 1u, abort_flag, kWaitNs));
        if (!warp_ok(got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t dk = dKt + ((sb * kKTile) >> 4);
        const uint32_t d = tbase + kColS + 64 * sb;
#pragma unroll
        for (uint32_t kc = 0; kc < 16; ++kc)
          mma_ts_warp(d, tbase + kColQ + 8 * kc, dk + (((kc >> 2) * kChunk + (kc & 3) * 32) >> 4),
                      idesc_qk, kc > 0 ? 1u : 0u);
#pragma unroll
        for (uint32_t kr = 0; kr < 2; ++kr)
          mma_ss_warp(d, dQr + ((kr * 32) >> 4), dk + ((4 * kChunk + kr * 32) >> 4), idesc_qk, 1u);
        mma_commit_warp(BAR(B_S_FULL + sb));
        if (j > pc.y) {
          const uint32_t tp = t - 1;
          if (!warp_ok(mbar_wait(BAR(B_P_FULL + (tp & 1u)), (tp >> 1) & 1u, abort_flag,
                                 kWaitNs))) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv(tp, j - 1 == pc.y);
        }
      }
      if (!ok) break;
      const uint32_t tp = t - 1;
      if (!warp_ok(mbar_wait(BAR(B_P_FULL + (tp & 1u)), (tp >> 1) & 1u, abort_flag, kWaitNs)))
        break;
      tc_fence_after();
      issue_pv(tp, pc.z - 1 == pc.y);
    }
    // no MMA may be in flight when tensor memory is released
    mma_commit_warp(BAR(B_DRAIN));
    if (lane == 0) wait_noabort(BAR(B_DRAIN), 0);
    __syncwarp();
  } else if (warp >= kSoftmaxWarp0 && warp < kDequantWarp0) {
    // ------------------------------------------------------------ softmax
    // thread = head h (tensor-memory lane).  CTA r owns heads 64r..64r+63
    // (lane quarters 2r, 2r+1): their softmax runs here.  The other two warps
    // send the peer the partial scores of the peer's heads and then take the
    // peer's P rows and rescale factors for them.
    const uint32_t quad = uint32_t(warp & 3);
    const int h = int(quad * 32) + lane;
    const bool own = (quad >> 1) == rank;
    const int hx = h & 63;  // row of h in the exchange buffers of its owner
    const uint32_t lane_base = (quad * 32u) << 16;
    const float c2 = a.scale * 1.4426950408889634f;  // scores to log2 units
    // row h of a P tile (SW128 K-major, 64 tokens = 128 B)
    const uint32_t prow = kSmPt + uint32_t(h >> 3) * 1024u + uint32_t(h & 7) * 128u;
    uint32_t t = 0, piece = 0;
    bool ok = true;
    for (int s = wr.x; ok && s <= wr.y; ++s) {
      const int4 pc = a.ws.pieces[s];
      const int b = pc.x;
      if (pc.z <= pc.y) {  // no block: an empty partial (the planner produces none)
        for (int c = 0; c < 256; ++c) a.ws.part_o[(int64_t(s) * 128 + h) * kDc + 256 * rank + c] = 0.f;
        if (own) a.ws.part_lse[int64_t(s) * 128 + h] = -INFINITY;
        continue;
      }
      const int L = seq_len_clamped(a, b);
      // queries of this piece: Qc half -> tensor memory, Qr half -> smem
      {
        const __nv_bfloat16* qrow = a.q_c + (int64_t(b) * 128 + h) * kDc + 256 * rank;
#pragma unroll 1
        for (int c0 = 0; c0 < 256; c0 += 64) {
          uint32_t w[32];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint4 v = *reinterpret_cast<const uint4*>(qrow + c0 + 8 * i);
            const uint32_t in[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k)
              w[4 * i + k] = pack_half2(__uint_as_float(in[k] << 16),
                                        __uint_as_float(in[k] & 0xffff0000u));
          }
          tmem_st32(tbase + lane_base + kColQ + c0 / 2, w);
        }
        const __nv_bfloat16* rrow = a.q_r + (int64_t(b) * 128 + h) * kDr + 32 * rank;
        unsigned char* qr = sm + kSmQr + (h >> 3) * 1024 + (h & 7) * 128;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const uint4 v = *reinterpret_cast<const uint4*>(rrow + 8 * g);
          const uint32_t in[4] = {v.x, v.y, v.z, v.w};
          uint32_t o[4];
#pragma unroll
          for (int k = 0; k < 4; ++k)
            o[k] = pack_half2(__uint_as_float(in[k] << 16), __uint_as_float(in[k] & 0xffff0000u));
          *reinterpret_cast<uint4*>(qr + ((g ^ (h & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
        fence_proxy_async_smem();
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(BAR(B_Q_FULL));
      }
      float m_run = -INFINITY, l_run = 0.0f;  // own heads
      uint32_t vmask = 0;
      for (int j = pc.y; j < pc.z; ++j, ++t) {
        if (((j - pc.y) & 31) == 0) vmask = valid_mask(a, b, j, pc.z);
        const uint32_t sb = t & 1u, par = (t >> 1) & 1u;
        if (!warp_ok(mbar_wait(BAR(B_S_FULL + sb), par, abort_flag, kWaitNs))) {
          ok = false;
          break;
        }
        tc_fence_after();
        float sv[64];
        {
          uint32_t r0[32], r1[32];
          tmem_ld32(tbase + lane_base + kColS + 64 * sb, r0);
          tmem_ld32(tbase + lane_base + kColS + 64 * sb + 32, r1);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            sv[i] = __uint_as_float(r0[i]);
            sv[32 + i] = __uint_as_float(r1[i]);
          }
        }
        float alpha = 1.0f;
        if (!own) {
          // --- the peer's head: send its partial scores, take back P and the
          // rescale factor.  (The peer writes P into this CTA's tile only after
          // these scores arrive, and they leave only after this CTA's QK of
          // tile t, i.e. after its P.V of tile t-2 read that tile parity.)
          if (!warp_ok(mbar_wait<true>(BAR(B_X_EMPTY + sb), par ^ 1u, abort_flag, kWaitNs))) {
            ok = false;
            break;
          }
          {
            const uint32_t xrow = mapa(sb0 + kSmX + sb * kX + uint32_t(hx) * 256u, peer);
            const uint32_t pbar = mapa(BAR(B_X_FULL + sb), peer);
#pragma unroll
            for (int q = 0; q < 16; ++q)
              st_async_v4(xrow + ((uint32_t(q) ^ uint32_t(hx & 15)) << 4), sv[4 * q],
                          sv[4 * q + 1], sv[4 * q + 2], sv[4 * q + 3], pbar);
          }
          if (!warp_ok(mbar_wait<true>(BAR(B_PX_FULL + sb), par, abort_flag, kWaitNs))) {
            ok = false;
            break;
          }
          alpha = *reinterpret_cast<const volatile float*>(sm + kSmAlpha + sb * 256 + hx * 4);
          // expect this buffer's next exchange (tile t+2) before the peer can
          // send it: the peer sends it only after scores this thread sends
          // later have arrived
          if (hx == 0) mbar_arrive_expect_tx(BAR(B_PX_FULL + sb), kPx);
        } else {
          // --- this CTA's head: add the peer's partial, softmax, send P back
          if (!warp_ok(mbar_wait<true>(BAR(B_X_FULL + sb), par, abort_flag, kWaitNs))) {
            ok = false;
            break;
          }
          const uint32_t xrow = kSmX + sb * kX + uint32_t(hx) * 256u;
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const float4 v = *reinterpret_cast<const float4*>(sm + xrow + ((q ^ (hx & 15)) << 4));
            sv[4 * q] += v.x;
            sv[4 * q + 1] += v.y;
            sv[4 * q + 2] += v.z;
            sv[4 * q + 3] += v.w;
          }
          // this CTA's buffer sb is read: expect the exchange two tiles ahead
          // and tell the peer it may send it
          if (hx == 0) mbar_arrive_expect_tx(BAR(B_X_FULL + sb), kX);
          mbar_arrive_remote(mapa(BAR(B_X_EMPTY + sb), peer));

          // tokens of this tile head h may see (its query's prefix in a
          // multi-token query decode)
          const int nvalid =
              ((vmask >> ((j - pc.y) & 31)) & 1u) ? min(kT, visible_tokens(a, h, L) - j * kT) : 0;
#pragma unroll
          for (int i = 0; i < 64; ++i) sv[i] *= c2;
          if (nvalid < 64) {
#pragma unroll
            for (int i = 0; i < 64; ++i) sv[i] = (i < nvalid) ? sv[i] : -INFINITY;
          }
          float mx8[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            mx8[k] = fmaxf(fmaxf(fmaxf(sv[8 * k], sv[8 * k + 1]), fmaxf(sv[8 * k + 2], sv[8 * k + 3])),
                           fmaxf(fmaxf(sv[8 * k + 4], sv[8 * k + 5]), fmaxf(sv[8 * k + 6], sv[8 * k + 7])));
          }
          const float mt = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                 fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
          if (mt > m_run + 8.0f) {
            alpha = exp2f(m_run - mt);
            m_run = mt;
          }
          l_run *= alpha;
          uint32_t pk[32];
          float ls4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
          const float msub = (mt == -INFINITY) ? 0.0f : m_run;  // all masked: every p is 0
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float p0 = ex2_approx(sv[2 * i] - msub);
            const float p1 = ex2_approx(sv[2 * i + 1] - msub);
            ls4[i & 3] += p0 + p1;
            pk[i] = pack_half2(p0, p1);
          }
          l_run += (ls4[0] + ls4[1]) + (ls4[2] + ls4[3]);
          // P row h into this CTA's tile and the peer's, the factor to the peer
          const uint32_t pl = prow + sb * kPt;
          const uint32_t pr = mapa(sb0 + pl, peer);
          const uint32_t pbar = mapa(BAR(B_PX_FULL + sb), peer);
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            const uint32_t off = uint32_t((g ^ (h & 7)) << 4);
            *reinterpret_cast<uint4*>(sm + pl + off) =
                make_uint4(pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
            st_async_u32x4(pr + off, pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3], pbar);
          }
          st_async_f32(mapa(sb0 + kSmAlpha + sb * 256 + hx * 4, peer), alpha, pbar);
        }
        // rescale this CTA's O rows of head h (its 256 channels) when the
        // maximum moved; the P.V products of tile t-1 must have landed first
        if (__any_sync(0xffffffffu, alpha != 1.0f) && j > pc.y) {
          const uint32_t tp = t - 1;
          if (!warp_ok(mbar_wait(BAR(B_PV_DONE + (tp & 1u)), (tp >> 1) & 1u, abort_flag,
                                 kWaitNs))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (uint32_t c0 = 0; c0 < 256; c0 += 32) {
            uint32_t o[32];
            tmem_ld32(tbase + lane_base + kColO + c0, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(tbase + lane_base + kColO + c0, o);
          }
          tmem_wait_st();
        }
        // this tile's P rows (written here or by the peer) reach the tensor
        // cores through the async proxy
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(BAR(B_P_FULL + sb));
      }
      if (!ok) break;
      // epilogue: normalized partial O (this CTA's 256 channels) and LSE
      const uint32_t tl = t - 1;
      if (!warp_ok(mbar_wait(BAR(B_PV_DONE + (tl & 1u)), (tl >> 1) & 1u, abort_flag, kWaitNs)))
        break;
      tc_fence_after();
      float l = l_run;
      if (own) {
        st_async_f32(mapa(sb0 + kSmLx + hx * 4, peer), l_run, mapa(BAR(B_LX_FULL), peer));
        a.ws.part_lse[int64_t(s) * 128 + h] =
            l_run > 0.0f ? (m_run + log2f(l_run)) * 0.6931471805599453f : -INFINITY;
      } else {
        if (!warp_ok(mbar_wait<true>(BAR(B_LX_FULL), piece & 1u, abort_flag, kWaitNs))) break;
        l = *reinterpret_cast<const volatile float*>(sm + kSmLx + hx * 4);
        __syncwarp();
        if (hx == 0) mbar_arrive_expect_tx(BAR(B_LX_FULL), 256);
      }
      ++piece;
      const float inv = l > 0.0f ? 1.0f / l : 0.0f;
      float* orow = a.ws.part_o + (int64_t(s) * 128 + h) * kDc + 256 * rank;
#pragma unroll 1
      for (uint32_t c0 = 0; c0 < 256; c0 += 32) {
        uint32_t o[32];
        tmem_ld32(tbase + lane_base + kColO + c0, o);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          *reinterpret_cast<float4*>(orow + c0 + i) =
              make_float4(__uint_as_float(o[i]) * inv, __uint_as_float(o[i + 1]) * inv,
                          __uint_as_float(o[i + 2]) * inv, __uint_as_float(o[i + 3]) * inv);
      }
      tc_fence_before();
    }
  } else if (warp >= kDequantWarp0 && kBF16) {
    // ------------------------------------------------------------ BF16 rows
    // thread dt owns token tt and 16-channel segment seg of each of the 4
    // groups of this half (and, dt < 128, a 16-channel RoPE segment); the
    // rows of the next tile are in flight while this tile's are stored
    const int dt = int(threadIdx.x) - kDequantWarp0 * 32;
    const int tt = (dt >> 2) & 63, seg = dt & 3;
    const int rtt = dt >> 1, rseg = dt & 1;  // RoPE (dt < 128)
    uint32_t t = 0;
    bool ok = true;
    for (int s = wr.x; ok && s <= wr.y; ++s) {
      const int4 pc = a.ws.pieces[s];
      if (pc.z <= pc.y) continue;
      const int L = seq_len_clamped(a, pc.x);
      const int32_t* btab = a.block_table + int64_t(pc.x) * a.max_blocks_per_seq;
      // rows of block j of this CTA's half, or nullptr (past the piece or a
      // bad block id: zeros); n = valid token rows
      auto half_of = [&](int j, int& n) -> const uint8_t* {
        n = 0;
        if (j >= pc.z) return nullptr;
        const int32_t blk = btab[j];
        if (blk < 0 || blk >= a.num_blocks) {
          if (dt == 0) set_status(a.status, QMLA_STATUS_BAD_BLOCK);
          return nullptr;
        }
        n = min(kT, L - j * kT);
        return a.blocks + int64_t(blk) * G.block + rank * G.half;
      };
      auto load_rows = [&](const uint8_t* hb, int n, uint32_t (&c)[4][8], uint32_t (&r)[8]) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          if (hb && tt < n) {
            ld_nc_v8(hb + (g * 64 + tt) * 128 + seg * 32, c[g]);
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) c[g][e] = 0u;
          }
        }
        if (dt < 128 && hb && rtt < n) {
          ld_nc_v8(hb + G.rope_off + rtt * 64 + rseg * 32, r);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) r[e] = 0u;
        }
      };
      int n_cur;
      const uint8_t* hb_cur = half_of(pc.y, n_cur);
      uint32_t cn[4][8], rn[8];
      load_rows(hb_cur, n_cur, cn, rn);
      for (int j = pc.y; j < pc.z; ++j, ++t) {
        uint32_t cc[4][8], rc[8];
#pragma unroll
        for (int g = 0; g < 4; ++g)
#pragma unroll
          for (int e = 0; e < 8; ++e) cc[g][e] = cn[g][e];
#pragma unroll
        for (int e = 0; e < 8; ++e) rc[e] = rn[e];
        int n_next;
        const uint8_t* hb_next = half_of(j + 1, n_next);
        load_rows(hb_next, n_next, cn, rn);
        const uint32_t kb = t & 1u;
        if (!warp_ok(mbar_wait(BAR(B_K_EMPTY + kb), ((t >> 1) & 1u) ^ 1u, abort_flag, kWaitNs))) {
          ok = false;
          break;
        }
        unsigned char* kt = sm + kSmK + kb * kKTile;
        auto to_f16 = [](uint32_t (&w)[8]) {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            w[e] = pack_half2(__uint_as_float(w[e] << 16), __uint_as_float(w[e] & 0xffff0000u));
        };
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          to_f16(cc[g]);
          st_row16(kt + g * kChunk, tt, seg, cc[g]);
        }
        if (dt < 128) {
          to_f16(rc);
          st_row16(kt + 4 * kChunk, rtt, rseg, rc);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(B_K_FULL + kb));
      }
    }
  } else if (warp >= kDequantWarp0) {
    // ------------------------------------------------------------ dequant
    const int dt = int(threadIdx.x) - kDequantWarp0 * 32;
    uint32_t t = 0;
    bool ok = true;
    for (int s = wr.x; ok && s <= wr.y; ++s) {
      const int4 pc = a.ws.pieces[s];
      const int L = seq_len_clamped(a, pc.x);
      uint32_t vmask = 0;
      for (int j = pc.y; j < pc.z; ++j, ++t) {
        if (((j - pc.y) & 31) == 0) vmask = valid_mask(a, pc.x, j, pc.z);
        const uint32_t st = t % kStages, kb = t & 1u;
        bool got = mbar_wait(BAR(B_STAGE_FULL + st), (t / kStages) & 1u, abort_flag, kWaitNs);
        got = got && mbar_wait(BAR(B_K_EMPTY + kb), ((t >> 1) & 1u) ^ 1u, abort_flag, kWaitNs);
        if (!warp_ok(got)) {
          ok = false;
          break;
        }
        const int nvalid = ((vmask >> ((j - pc.y) & 31)) & 1u) ? min(kT, L - j * kT) : 0;
        const unsigned char* stg = sm + kSmStage + st * kStage;
        unsigned char* kt = sm + kSmK + kb * kKTile;
        // content: thread dt owns token tt and 16-channel segment seg of each of
        // the 4 groups of this half; unconditional loads, invalid tokens zeroed
        {
          const int tt = (dt >> 2) & 63, seg = dt & 3;
          const bool valid = tt < nvalid;
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            __half2 s2, z2;
            split_sz(*reinterpret_cast<const uint32_t*>(stg + G.sz_off + (g * 64 + tt) * 4), s2,
                     z2);
            uint32_t v[8];
            if (G.cbits == 4) {
              const uint2 w = *reinterpret_cast<const uint2*>(stg + g * 2048 + tt * 32 + seg * 8);
              dq_int4(w.x, s2, z2, v);
              dq_int4(w.y, s2, z2, v + 4);
            } else {
              dq_int2(*reinterpret_cast<const uint32_t*>(stg + g * 1024 + tt * 16 + seg * 4), s2, z2,
                      v);
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = valid ? v[k] : 0u;
            st_row16(kt + g * kChunk, tt, seg, v);
          }
        }
        // RoPE: 64 tokens x 2 segments of 16 channels (INT4)
        if (dt < 128) {
          const int tt = dt >> 1, seg = dt & 1;
          uint32_t v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
          if (tt < nvalid) {
            __half2 s2, z2;
            split_sz(*reinterpret_cast<const uint32_t*>(stg + G.half + tt * 4), s2, z2);
            const uint2 w = *reinterpret_cast<const uint2*>(stg + G.rope_off + tt * 16 + seg * 8);
            dq_int4(w.x, s2, z2, v);
            dq_int4(w.y, s2, z2, v + 4);
          }
          st_row16(kt + 4 * kChunk, tt, seg, v);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(BAR(B_K_FULL + kb));
          mbar_arrive(BAR(B_STAGE_EMPTY + st));
        }
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
  cluster_sync();  // no CTA leaves while its peer may still touch its shared memory
}

}  // namespace

cudaError_t launch_decode_tc128(const DecodeArgs& a, cudaStream_t stream) {
  static int smem_attr_done[kMaxDevices], smem_attr_done_bf16[kMaxDevices];
  cudaError_t e = launch_plan(a, stream);
  if (e != cudaSuccess) return e;
  const bool bf16 = a.fmt == QMLA_BF16;
  auto kernel = bf16 ? decode_tc128_kernel<true> : decode_tc128_kernel<false>;
  e = ensure_smem_attr(kernel, int(kSmDyn), bf16 ? smem_attr_done_bf16 : smem_attr_done);
  if (e != cudaSuccess) return e;
  kernel<<<dim3(unsigned(2 * a.workers)), kThreads, kSmDyn, stream>>>(a);
  return cudaGetLastError();
}

int tc_workers(int sms, int heads) {
  if (heads == 16) return sms > 0 ? sms : 1;
  return sms / 2 > 0 ? sms / 2 : 1;
}

bool tc_supported(int fmt, int heads) {
  return (heads == 128 || heads == 16) &&
         (fmt == QMLA_C4R4 || fmt == QMLA_C2R4 || fmt == QMLA_BF16);
}

cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t stream) {
  return a.heads == 16 ? launch_decode_tc16(a, stream) : launch_decode_tc128(a, stream);
}

}  // namespace qmla
