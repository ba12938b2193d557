// decode_tc.cu - tensor-core (tcgen05) decode over the low-bit paged cache,
// 128 query heads (128 absorbed heads, or the 128 query rows of a
// multi-token query step), and the split planner of both tensor-core decodes.
//
// The "native low-bit MLA attention kernel" of "QuantMLA: INT4 (and INT2) for
// both halves of the MLA cache" (flowchart node "Low-bit kernel: dequant
// inside attention"; "Key findings"): packed blocks are unpacked and
// dequantized on chip and consumed directly by the tensor cores.
//
// Work split.  A work unit (a range of cache blocks of one sequence, in tiles
// of two blocks = 128 tokens) runs on a cluster of two CTAs.  CTA r
//   * computes the scores and the softmax of heads 64r .. 64r+63 over all 576
//     channels, tokens on the MMA's M:
//       S^T[128 tok x 64 heads] = K[128 tok x 576] (A) x Q_r^T (B, smem),
//     so the scores of its heads are complete in its own tensor memory and
//     no partial score ever crosses between the CTAs;
//   * accumulates O of all 128 heads over its half of the content channels,
//     256r .. 256r+255, heads on M:
//       O_r[128 heads x 256 ch] += P[128 heads x 128 tok] (A, smem) x
//                                  C_r[128 tok x 256 ch] (B, smem),
//     for which it needs the other CTA's P rows: 16 KB per tile and
//     direction through cluster shared memory, with the rescale factors.
// O of 128 heads x 512 channels in binary32 would fill all 512 columns of an
// SM's tensor memory, which is why O is split by channel.  Each CTA
// dequantizes all 576 channels of every token (the two CTAs read the same
// packed blocks at the same time; the second read hits L2).
//
// Operand placement (the tensor core reads shared memory at 128 B/clock, so
// an MMA whose operands both come from shared memory at N = 64 would wait
// for its operands; A from tensor memory avoids that):
//   tensor memory: O_r (256 columns), S^T (64), and the A operand of QK for
//     the content channels of the other CTA's half (4 x 32 columns), the RoPE
//     channels (32) and one content chunk of this CTA's half (32);
//   shared memory: Q_r^T (72 KB), P (32 KB), and a ring of seven 16 KB
//     content chunks of this CTA's half (K for QK read K-major, the same bytes
//     C_r for P.V read MN-major).  A tile's four chunks sit in slots 0-3
//     (even tiles) or 3-6 (odd tiles): slot 3 is the one chunk of a tile that
//     is written after the previous tile's P.V has released it, and the copy
//     in tensor memory lets QK run before that.
//
// Pipeline: the MMA warp issues QK of tile t, then P.V of tile t-1, so the
// softmax of tile t-1 and its P exchange overlap the tensor core's QK of
// tile t, and the dequantization of tile t+1 overlaps the P.V of tile t-1.
//
// Warp roles (20 warps, five warpgroups): 0 MMA issuer, 1 P exchanger (2-3
// idle); 4-11 softmax (thread = token row of S^T; two warps per
// tensor-memory lane quarter, 32 heads each); 12-19 dequantization (thread =
// token row; two warps per lane quarter).  The first warpgroup hands part of
// its registers to the other four (setmaxnreg): 48 + 104 (softmax) + 112
// (dequantization) per thread of each sub-partition's five warps, within the
// launch's 96 x 5, for the low-bit formats (the dequantization warps hold a
// tile's packed codes a tile ahead of use), 64 + 104 + 104 for BF16 rows
// (measured best of the splits that fit).  Binary16 operands (exact on the
// quantizer's grid), binary32 accumulation.  The softmax is online in base 2 with lazy
// rescaling: the running maximum of a head only moves when a score exceeds
// it by more than kLazy = 15 (P < 2^15, inside binary16's range; row sums
// and O are binary32).  Every
// wait is bounded in time; on timeout the CTA raises an abort flag, all
// roles unwind and QMLA_STATUS_TIMEOUT is reported.
//
// The same kernel serves the uncompressed BF16 cache, the baseline the
// low-bit formats are compared with: the rows are loaded and converted
// bfloat16 -> binary16 instead of dequantized.

#include <cfloat>

#include "tc_common.cuh"

namespace qmla {
namespace tc {
// ---------------------------------------------------------------- planner
// One warp writes the split plan: merge table, piece descriptors per slot
// and the slot range of each worker.
__global__ void __launch_bounds__(32) plan_kernel(DecodeArgs a) {
  const int lane = threadIdx.x;
  // Launched as a programmatic dependent of the kernel before it (the append
  // that advances seq_lens, say): the decode after it may be scheduled now,
  // and nothing is read before that kernel has completed.
  if (lane == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tc::plan_kernel, a);
}

namespace {

using namespace ptx;
using namespace tc;

// ---------------------------------------------------------------- layout
constexpr int kThreads = 20 * 32;
constexpr int kMmaWarp = 0;
constexpr int kXchgWarp = 1;   // moves this CTA's P rows to the peer
constexpr int kSmxWarp0 = 4;   // 8 softmax warps (warpgroups 1-2)
constexpr int kDqWarp0 = 12;   // 8 dequantization warps (warpgroups 3-4)
// registers per thread at launch (__launch_bounds__ at 20 warps; the
// launcher checks the compiled kernel's count) and of the issuer warpgroup,
// the softmax and the dequantization warps after setmaxnreg; the BF16 rows
// need no codes held ahead of use
constexpr uint32_t kRegsLaunch = 96;
template <int kCBits>
struct RegSplit {
  static constexpr uint32_t idle = kCBits == 16 ? 64 : 48, smx = 104, dq = kCBits == 16 ? 104 : 112;
  static_assert(128 * idle + 256 * smx + 256 * dq <= kThreads * kRegsLaunch,
                "register split within the launch allocation");
};

// tensor memory (32-bit columns)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;    // O_r: lane = head, 256 channels
constexpr uint32_t kColS = 256;  // S^T: lane = token, 64 heads
constexpr uint32_t kColK = 320;  // K units u = 0..5 at 320 + 32u, lane = token, binary16 pairs:
                                 // 0-3 the other half's content chunks, 4 this half's late
                                 // chunk, 5 the 64 RoPE channels

// shared memory
constexpr uint32_t kQChunk = 8192;  // [64 heads][64 ch] binary16, SW128 K-major
constexpr uint32_t kAtom = 16384;   // [128 rows][64] binary16, SW128
constexpr uint32_t kSmQ = 0;                                  // 9 chunks: content 0-7, RoPE
constexpr uint32_t kSmP = kSmQ + 9 * kQChunk;                 // 2 atoms: heads 0-63, 64-127
constexpr uint32_t kSmRing = kSmP + 2 * kAtom;                // 7 content chunk slots
constexpr uint32_t kSlots = 7;
constexpr uint32_t kPkt = 272;  // rescale packet: [64] factors + a 16-byte flag
constexpr uint32_t kSmAlphaIn = kSmRing + kSlots * kAtom;     // [2][packet] from the peer
constexpr uint32_t kSmAlphaOwn = kSmAlphaIn + 2 * kPkt;       // [64] this CTA's factors
constexpr uint32_t kSmM = kSmAlphaOwn + 256;                  // [64] running maxima (log2 units)
constexpr uint32_t kSmLIn = kSmM + 256;                       // [64] the peer's row sums
constexpr uint32_t kSmLOwn = kSmLIn + 256;                    // [64] this CTA's row sums
constexpr uint32_t kSmRed = kSmLOwn + 256;                    // [4 lane quarters][64] partials
constexpr uint32_t kSmBar = kSmRed + 1024;
enum : uint32_t {
  B_Q_FULL = 0,  // this piece's queries staged (8 dequantization warps)
  B_S_FULL,      // QK of a tile complete (commit)
  B_S_EMPTY,     // the softmax has read the scores (8 softmax warps)
  B_KT_FULL,     // [3] K unit pair k (units k, 3+k) of a tile written (8 dequantization warps)
  B_KT_EMPTY = B_KT_FULL + 3,  // [3] the QK products reading unit pair k complete (commit)
  B_RING_FULL = B_KT_EMPTY + 3,  // a tile's three early ring chunks written (8 dequantization warps)
  B_LATE_FULL,   // a tile's late ring chunk (slot 3) written (4 dequantization warps)
  B_PV_DONE,     // P.V of a tile complete: its ring slots and P free (commit)
  B_P_LOCAL,     // this CTA's P rows of a tile written (8 softmax warps)
  B_SRC_FREE,    // the bulk copy of those rows to the peer has read them (exchanger)
  B_P_FULL,      // a tile's local P rows written and O rescaled (8 softmax warps)
  B_PX_FULL,     // the peer's P rows arrived (1 arming arrival + bytes)
  B_PFREE,       // the peer's P.V of a tile complete (1 remote arrival)
  B_AX0,         // the peer's rescale packet of an even / odd tile arrived
  B_AX1,         //   (1 arming arrival + bytes each)
  B_O_EMPTY,     // the epilogue has read O (8 softmax warps)
  B_LX_FULL,     // the peer's row sums arrived (1 arming arrival + bytes)
  B_DRAIN,
  kNumBars
};
constexpr uint32_t kSmTslot = kSmBar + 8 * kNumBars;
constexpr uint32_t kSmAbort = kSmTslot + 4;
constexpr uint32_t kSmBytes = kSmAbort + 12;
constexpr uint32_t kSmDyn = kSmBytes + 1024;  // slack for 1 KB alignment
constexpr uint32_t kPx = 128 * 64 * 2;  // P rows of one CTA's heads per tile
// A head's running maximum before its first score (log2 units): finite, so
// that scores minus it stay exact enough to find the first maximum, and far
// below any score of binary16 operands that the softmax can represent.
constexpr float kMaxUnset = -32768.0f;
// Lazy rescaling: a head's running maximum moves only when a score exceeds it
// by more than this (log2 units).  P = 2^d then stays below 2^15, exact in
// binary16's range; a smaller margin rescales far more often on coarse (INT2)
// keys, whose scores spread more.
constexpr float kLazy = 15.0f;
static_assert(kSmP % 1024 == 0 && kSmRing % 1024 == 0, "SW128 operand tiles are 1 KB aligned");
static_assert(kSmBar % 8 == 0, "mbarrier alignment");
static_assert(kSmDyn <= 232448, "shared memory budget");

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
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.b32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
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
// Either half of a binary16 pair is infinite.
__device__ __forceinline__ bool h2_inf(uint32_t w) {
  return (w & 0x7fffu) == 0x7c00u || (w & 0x7fff0000u) == 0x7c000000u;
}

// Packed codes of one 64-channel unit of one token: a content group (INT4:
// 8 words, INT2: 4) or the 64 RoPE channels (INT4: two 16-byte halves), and
// the (scale, zero) word.  A zero scale/zero word makes every value +0,
// whatever the codes hold.
struct Unit {
  uint32_t c[8];
  uint32_t sz;
};
template <int kCBits>
__device__ __forceinline__ void load_content(Unit& u, const uint8_t* blk, const Geom& G, int grp,
                                             int slot) {
#pragma unroll
  for (int e = 0; e < 8; ++e) u.c[e] = 0u;
  u.sz = 0u;
  if (blk == nullptr) return;
  const uint8_t* half = blk + (grp >> 2) * G.half;
  const int g = grp & 3;
  if (kCBits == 4)
    ld_nc_v8(half + g * 2048 + slot * 32, u.c);
  else
    ld_nc_v4(half + g * 1024 + slot * 16, u.c);
  u.sz = ld_nc_b32(half + G.sz_off + (g * 64 + slot) * 4);
}
__device__ __forceinline__ void load_rope(Unit& u, const uint8_t* blk, const Geom& G, int slot) {
#pragma unroll
  for (int e = 0; e < 8; ++e) u.c[e] = 0u;
  u.sz = 0u;
  if (blk == nullptr) return;
  ld_nc_v4(blk + G.rope_off + slot * 16, u.c);
  ld_nc_v4(blk + G.half + G.rope_off + slot * 16, u.c + 4);
  u.sz = ld_nc_b32(blk + G.rope_sz_off + slot * 4);
}
// Channels 32*part .. 32*part+31 of a unit as 16 binary16 pairs (channel
// 2k low, 2k+1 high).  The RoPE unit is INT4 in both halves.
template <int kCBits>
__device__ __forceinline__ void dq_half(const Unit& u, int part, uint32_t (&v)[16]) {
  __half2 s2, z2;
  split_sz(u.sz, s2, z2);
  if (kCBits == 4) {
#pragma unroll
    for (int w = 0; w < 4; ++w) dq_int4(u.c[4 * part + w], s2, z2, v + 4 * w);
  } else {
#pragma unroll
    for (int w = 0; w < 2; ++w) dq_int2(u.c[2 * part + w], s2, z2, v + 8 * w);
  }
}
// BF16 cache: 64 bfloat16 values of a content group row (128 B) or of the
// RoPE key (two 64 B halves), converted to binary16 pairs.
__device__ __forceinline__ void load_bf16_content(uint32_t (&w)[32], const uint8_t* blk,
                                                  const Geom& G, int grp, int slot) {
  if (blk == nullptr) {
#pragma unroll
    for (int e = 0; e < 32; ++e) w[e] = 0u;
    return;
  }
  const uint8_t* row = blk + (grp >> 2) * G.half + ((grp & 3) * 64 + slot) * 128;
#pragma unroll
  for (int i = 0; i < 4; ++i) ld_nc_v8(row + 32 * i, w + 8 * i);
}
__device__ __forceinline__ void load_bf16_rope(uint32_t (&w)[32], const uint8_t* blk,
                                               const Geom& G, int slot) {
  if (blk == nullptr) {
#pragma unroll
    for (int e = 0; e < 32; ++e) w[e] = 0u;
    return;
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint8_t* row = blk + h * G.half + G.rope_off + slot * 64;
    ld_nc_v8(row, w + 16 * h);
    ld_nc_v8(row + 32, w + 16 * h + 8);
  }
}
__device__ __forceinline__ void bf16_to_f16(uint32_t (&w)[32]) {
#pragma unroll
  for (int e = 0; e < 32; ++e)
    w[e] = pack_half2(__uint_as_float(w[e] << 16), __uint_as_float(w[e] & 0xffff0000u));
}
// 64 channels into row `row_off` (precomputed row offset) of an SW128 atom.
__device__ __forceinline__ void st_row64(unsigned char* atom, uint32_t row_off, int sw7,
                                         const uint32_t (&v)[32]) {
#pragma unroll
  for (int g = 0; g < 8; ++g)
    *reinterpret_cast<uint4*>(atom + row_off + ((g ^ sw7) << 4)) =
        make_uint4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
}
// Channels 32*part .. 32*part+31 of a row.
__device__ __forceinline__ void st_row32(unsigned char* atom, uint32_t row_off, int sw7, int part,
                                         const uint32_t (&v)[16]) {
#pragma unroll
  for (int g = 0; g < 4; ++g)
    *reinterpret_cast<uint4*>(atom + row_off + (((4 * part + g) ^ sw7) << 4)) =
        make_uint4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
}
// A unit of packed codes, dequantized, into tensor-memory columns `col`
// (32 columns, lane = this thread's token row) or into a ring atom row.
template <int kCBits>
__device__ __forceinline__ void unit_to_tmem(const Unit& u, bool rope, uint32_t taddr) {
#pragma unroll
  for (int part = 0; part < 2; ++part) {
    uint32_t v[16];
    if (rope)
      dq_half<4>(u, part, v);
    else
      dq_half<kCBits>(u, part, v);
    tmem_st16(taddr + 16u * part, v);
  }
}
template <int kCBits>
__device__ __forceinline__ void unit_to_ring(const Unit& u, unsigned char* atom, uint32_t row_off,
                                             int sw7) {
#pragma unroll
  for (int part = 0; part < 2; ++part) {
    uint32_t v[16];
    dq_half<kCBits>(u, part, v);
    st_row32(atom, row_off, sw7, part, v);
  }
}

// Tiles of the worker: tile i of piece s covers blocks j0 + 2i, j0 + 2i + 1.
__device__ __forceinline__ int piece_tiles(const int4& pc) {
  return pc.z > pc.y ? (pc.z - pc.y + 1) >> 1 : 0;
}

// ---------------------------------------------------------------- kernel
template <int kCBits>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_tc128_kernel(DecodeArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb0 = smem_u32(sm);
  auto BAR = [&](uint32_t i) { return sb0 + kSmBar + 8 * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kSmAbort);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
  const int pair = blockIdx.x >> 1;
  constexpr bool kBF16 = kCBits == 16;
  const Geom G = geom(kCBits == 4 ? QMLA_C4R4 : kCBits == 2 ? QMLA_C2R4 : QMLA_BF16);

  if (threadIdx.x == 0) {
    mbar_init(BAR(B_Q_FULL), 8);
    mbar_init(BAR(B_S_FULL), 1);
    mbar_init(BAR(B_S_EMPTY), 8);
    for (uint32_t k = 0; k < 3; ++k) {
      mbar_init(BAR(B_KT_FULL + k), 8);
      mbar_init(BAR(B_KT_EMPTY + k), 1);
    }
    mbar_init(BAR(B_RING_FULL), 8);
    mbar_init(BAR(B_LATE_FULL), 4);
    mbar_init(BAR(B_PV_DONE), 1);
    mbar_init(BAR(B_P_LOCAL), 8);
    mbar_init(BAR(B_SRC_FREE), 1);
    mbar_init(BAR(B_P_FULL), 8);
    mbar_init(BAR(B_PX_FULL), 1);
    mbar_init(BAR(B_PFREE), 1);
    mbar_init(BAR(B_AX0), 1);
    mbar_init(BAR(B_AX1), 1);
    mbar_init(BAR(B_O_EMPTY), 8);
    mbar_init(BAR(B_LX_FULL), 1);
    mbar_init(BAR(B_DRAIN), 1);
    // the first exchanges are expected before the peer can send them
    mbar_arrive_expect_tx(BAR(B_PX_FULL), kPx);
    mbar_arrive_expect_tx(BAR(B_AX0), kPkt);
    mbar_arrive_expect_tx(BAR(B_AX1), kPkt);
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
  // The kernel is launched as a programmatic dependent of the planner: the
  // set-up above overlaps it, and no thread reads global memory before the
  // planner (and, through its own wait, the kernel before it) has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the merge kernel that follows may be scheduled now (it waits for this
  // grid to complete before it reads anything)
  if (threadIdx.x == 0) griddep_launch_dependents();
  const int2 wr = a.ws.wrange[pair];

  if (warp < kSmxWarp0) {
    // the first warpgroup (all four warps at this one instruction) gives up
    // registers; only its first warp has work
    setmaxnreg_to<kRegsLaunch, RegSplit<kCBits>::idle>();
  }
  if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop converged and an elected lane issues each
    // instruction.
    const uint32_t idq = idesc_f16(128, 64, false, false);
    const uint32_t idp = idesc_f16(128, 256, true, true);
    // operand descriptors; an offset advances the 16-byte address field
    const uint64_t dQ = smem_desc(sb0 + kSmQ, 16, 1024, kSwizzle128B);
    const uint64_t dK = smem_desc(sb0 + kSmRing, 16, 1024, kSwizzle128B);
    const uint64_t dV = smem_desc(sb0 + kSmRing, kAtom, 1024, kSwizzle128B);
    const uint64_t dP = smem_desc(sb0 + kSmP, kAtom, 1024, kSwizzle128B);
    uint32_t t = 0, pq = 0;
    bool ok = true;
    // P.V of the previous tile, issued after QK of the next one
    bool pend = false, pfirst = false;
    uint32_t pt = 0, ppq = 0;
    auto issue_pv = [&]() -> bool {
      bool got = mbar_wait(BAR(B_P_FULL), pt & 1u, abort_flag, kWaitNs);
      got = got && mbar_wait(BAR(B_LATE_FULL), pt & 1u, abort_flag, kWaitNs);
      got = got && mbar_wait<true>(BAR(B_PX_FULL), pt & 1u, abort_flag, kWaitNs);
      // the first tile of a piece overwrites O: the last piece's epilogue has read it
      if (pfirst && ppq > 0)
        got = got && mbar_wait(BAR(B_O_EMPTY), (ppq - 1) & 1u, abort_flag, kWaitNs);
      if (!warp_ok(got)) return false;
      // the peer sends the next tile's rows only after this tile's P.V
      if (lane == 0) mbar_arrive_expect_tx(BAR(B_PX_FULL), kPx);
      tc_fence_after();
      const uint32_t vbase = (pt & 1u) ? 3u * kAtom : 0u;
#pragma unroll
      for (uint32_t kt = 0; kt < 8; kt += 4)
        mma_ss_warp_x4(tbase + kColO, dP + ((kt * 2048u) >> 4), dV + ((vbase + kt * 2048u) >> 4),
                       idp, (pfirst && kt == 0) ? 0u : 1u, 2048u >> 4, 2048u >> 4);
      mma_commit_warp(BAR(B_PV_DONE));
      return true;
    };
    for (int s = wr.x; ok && s <= wr.y; ++s) {
      const int4 pc = a.ws.pieces[s];
      const int nt = piece_tiles(pc);
      if (nt == 0) continue;
      if (!warp_ok(mbar_wait(BAR(B_Q_FULL), pq & 1u, abort_flag, kWaitNs))) {
        ok = false;
        break;
      }
      for (int i = 0; i < nt; ++i, ++t) {
        if (!warp_ok(t == 0 || mbar_wait(BAR(B_S_EMPTY), (t - 1) & 1u, abort_flag, kWaitNs))) {
          ok = false;
          break;
        }
        const uint32_t odd = t & 1u;
        const uint32_t lc = odd ? 0u : 3u;  // this half's chunk in slot 3
        // QK from tensor memory, unit pair by unit pair as the dequantization
        // writes them: pair k is the other half's chunk k and unit 3+k (the
        // other half's chunk 3, this half's late chunk, RoPE); each pair is
        // released as soon as its products complete
#pragma unroll 1
        for (uint32_t k = 0; k < 3; ++k) {
          if (!warp_ok(mbar_wait(BAR(B_KT_FULL + k), t & 1u, abort_flag, kWaitNs))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (uint32_t h = 0; h < 2; ++h) {
            const uint32_t u = k + 3u * h;
            const uint32_t qc = u < 4 ? 4u * peer + u : (u == 4 ? 4u * rank + lc : 8u);
            mma_ts_warp_x4(tbase + kColS, tbase + kColK + 32u * u, dQ + ((qc * kQChunk) >> 4), idq,
                           u ? 1u : 0u, 8u, 32u >> 4);
          }
          mma_commit_warp(BAR(B_KT_EMPTY + k));
        }
        if (!ok) break;
        // QK from the ring: this half's three early chunks
        if (!warp_ok(mbar_wait(BAR(B_RING_FULL), t & 1u, abort_flag, kWaitNs))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t base = odd ? 3u : 0u;
#pragma unroll 1
        for (uint32_t e = 0; e < 3; ++e) {
          const uint32_t c = e + odd;
          mma_ss_warp_x4(tbase + kColS, dK + (((base + c) * kAtom) >> 4),
                         dQ + (((4u * rank + c) * kQChunk) >> 4), idq, 1u, 32u >> 4, 32u >> 4);
        }
        mma_commit_warp(BAR(B_S_FULL));
        if (pend && !issue_pv()) {
          ok = false;
          break;
        }
        pend = true;
        pt = t;
        pfirst = i == 0;
        ppq = pq;
      }
      ++pq;
    }
    if (ok && pend) issue_pv();
    // no MMA may be in flight when tensor memory is released
    mma_commit_warp(BAR(B_DRAIN));
    if (lane == 0) wait_noabort(BAR(B_DRAIN), 0);
    __syncwarp();
  } else if (warp == kXchgWarp) {
    // ------------------------------------------------------------ exchanger
    // One bulk copy per tile moves this CTA's P rows (its 64 heads, 16 KB)
    // into the peer's P tile, once the peer's P.V of the previous tile has
    // released it; the softmax warps never wait for the transfer.
    const uint32_t src = sb0 + kSmP + rank * kAtom;
    const uint32_t dst = mapa(src, peer);
    const uint32_t pbar = mapa(BAR(B_PX_FULL), peer);
    uint32_t t = 0;
    bool ok = true;
    for (int s = wr.x; ok && s <= wr.y; ++s) {
      const int nt = piece_tiles(a.ws.pieces[s]);
      for (int i = 0; i < nt; ++i, ++t) {
        bool got = mbar_wait(BAR(B_P_LOCAL), t & 1u, abort_flag, kWaitNs);
        got = got && (t == 0 || mbar_wait<true>(BAR(B_PFREE), (t - 1) & 1u, abort_flag, kWaitNs));
        if (!warp_ok(got)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          bulk_s2c(dst, src, kPx, pbar);
          bulk_commit_and_wait_read();
          mbar_arrive(BAR(B_SRC_FREE));
        }
        __syncwarp();
        // this CTA's P.V of tile t has read the peer's rows: the peer may send the next
        if (!warp_ok(mbar_wait(BAR(B_PV_DONE), t & 1u, abort_flag, kWaitNs))) {
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive_remote(mapa(BAR(B_PFREE), peer));
      }
    }
  } else if (warp < kSmxWarp0) {
    // idle warps of the first warpgroup
  } else if (warp < kDqWarp0) {
    // ------------------------------------------------------------ softmax
    setmaxnreg_to<kRegsLaunch, RegSplit<kCBits>::smx>();
    // thread = token row tt of S^T (its lane quarter's tensor-memory lanes);
    // the warp holds 32 of this CTA's 64 heads.  For O (lane = head) the same
    // thread stands for head tt.
    const int sw = warp - kSmxWarp0;  // 0..7
    const uint32_t quad = uint32_t(warp & 3);
    const int hh = sw >> 2;            // this CTA's heads 32hh .. 32hh+31
    const int tt = int(quad) * 32 + lane;
    const uint32_t lane_base = (quad * 32u) << 16;
    const bool o_own = (quad >> 1) == rank;  // O rows of this lane quarter: this CTA's heads
    const int oh = int(quad & 1u) * 32 + lane;  // head within its owner's 64
    const float c2 = a.scale * 1.4426950408889634f;  // scores to log2 units
    float* m_run = reinterpret_cast<float*>(sm + kSmM);
    float* red = reinterpret_cast<float*>(sm + kSmRed);
    float* al_own = reinterpret_cast<float*>(sm + kSmAlphaOwn);
    float* l_own = reinterpret_cast<float*>(sm + kSmLOwn);
    const float* l_in = reinterpret_cast<const float*>(sm + kSmLIn);
    const uint32_t prow = kSmP + rank * kAtom + uint32_t(tt >> 3) * 1024u + uint32_t(tt & 7) * 128u;
    auto rescale_o = [&](float al) {
      // this warp's 128 of the 256 O columns of row tt
#pragma unroll 1
      for (uint32_t c0 = 128u * hh; c0 < 128u * hh + 128u; c0 += 32) {
        uint32_t o[32];
        tmem_ld32(tbase + lane_base + kColO + c0, o);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * al);
        tmem_st32(tbase + lane_base + kColO + c0, o);
      }
      tmem_wait_st();
    };
    uint32_t t = 0, pq = 0;
    bool ok = true;
    for (int s = wr.x; ok && s <= wr.y; ++s) {
      const int4 pc = a.ws.pieces[s];
      const int nt = piece_tiles(pc);
      if (nt == 0) {  // no block: an empty partial (the planner produces none)
        for (int c = 0; c < 128; ++c)
          a.ws.part_o[(int64_t(s) * 128 + tt) * kDc + 256 * rank + 128 * hh + c] = 0.f;
        if (quad == 0) a.ws.part_lse[int64_t(s) * 128 + 64 * rank + 32 * hh + lane] = -INFINITY;
        continue;
      }
      const int b = pc.x;
      const int L = seq_len_clamped(a, b);
      if (quad == 0) m_run[32 * hh + lane] = kMaxUnset;
      named_bar_sync(2, 256);
      float l[32];
#pragma unroll
      for (int h = 0; h < 32; ++h) l[h] = 0.0f;
      uint32_t vmask = 0;
      for (int i = 0; i < nt; ++i, ++t) {
        const int jt = pc.y + 2 * i;
        if (((2 * i) & 31) == 0) vmask = valid_mask(a, b, jt, pc.z);
        const int j = jt + (tt >> 6);
        const bool row_ok =
            j < pc.z && ((vmask >> ((j - pc.y) & 31)) & 1u) && (tt & 63) < L - j * kT;
        bool got = ok && warp_ok(mbar_wait(BAR(B_S_FULL), t & 1u, abort_flag, kWaitNs));
        // d = score in log2 units minus the running maximum of its head
        float d[32];
        auto load_d = [&]() {
          tc_fence_after();
          uint32_t r32[32];
          tmem_ld32(tbase + lane_base + kColS + 32u * hh, r32);
          tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < 32; h += 4) {
            const float4 m = *reinterpret_cast<const float4*>(m_run + 32 * hh + h);
            d[h] = fmaf(__uint_as_float(r32[h]), c2, -m.x);
            d[h + 1] = fmaf(__uint_as_float(r32[h + 1]), c2, -m.y);
            d[h + 2] = fmaf(__uint_as_float(r32[h + 2]), c2, -m.z);
            d[h + 3] = fmaf(__uint_as_float(r32[h + 3]), c2, -m.w);
          }
          if (!row_ok) {
#pragma unroll
            for (int h = 0; h < 32; ++h) d[h] = -INFINITY;
          } else if (a.q_heads > 0) {
            // multi-token query: the last q_len - 1 positions are not visible to
            // every row.  Virtual head v (query v / q_heads) sees positions up to
            // L - q_len + v / q_heads, so position pos = L - q_len + 1 + e is
            // hidden from v exactly when v < (e + 1) q_heads: a prefix of this
            // thread's heads, found without a division per head.
            const int e = j * kT + (tt & 63) - (L - a.q_len + 1);
            if (e >= 0) {
              const int hcut = (e + 1) * a.q_heads - (64 * int(rank) + 32 * hh);
#pragma unroll
              for (int h = 0; h < 32; ++h)
                if (h < hcut) d[h] = -INFINITY;
            }
          }
        };
        if (got) {
          load_d();
        } else {
#pragma unroll
          for (int h = 0; h < 32; ++h) d[h] = -INFINITY;
        }
        ok = ok && got;
        // lazy rescale: a head's maximum only moves when one of its scores
        // exceeds it by more than kLazy (an unset maximum is kMaxUnset, below any
        // score); the decisions are the same in every thread.  All eight
        // warps take every barrier below whatever their waits returned: a
        // failed wait forces the rare path, which leaves the loop together.
        float dmax = d[0];
#pragma unroll
        for (int h = 1; h < 32; ++h) dmax = fmaxf(dmax, d[h]);
        bool rescaled = false;
        if (named_bar_or(1, 256, !ok || dmax > kLazy)) {
          if (named_bar_or(1, 256, !ok)) break;
          float mine = -INFINITY;
#pragma unroll
          for (int h = 0; h < 32; ++h) {
            const float v = warp_max(d[h]);
            if (lane == h) mine = v;
          }
          red[quad * 64 + 32 * hh + lane] = mine;
          named_bar_sync(2, 256);
          if (quad == 0) {  // one warp per head half moves the maxima
            const int hl = 32 * hh + lane;
            const float dm = fmaxf(fmaxf(red[hl], red[64 + hl]), fmaxf(red[128 + hl], red[192 + hl]));
            const bool need = dm > kLazy;
            al_own[hl] = need ? ex2_approx(-dm) : 1.0f;  // ~0 when the maximum was unset
            if (need) m_run[hl] += dm;
          }
          named_bar_sync(2, 256);
          // the scores again, against the new maxima (exact, where the step
          // from an unset maximum was not)
          load_d();
#pragma unroll
          for (int h = 0; h < 32; h += 4) {
            const float4 f = *reinterpret_cast<const float4*>(al_own + 32 * hh + h);
            l[h] *= f.x;
            l[h + 1] *= f.y;
            l[h + 2] *= f.z;
            l[h + 3] *= f.w;
          }
          rescaled = i > 0;  // O holds earlier tiles of this piece
        }
        // the scores are read: the next tile's QK may overwrite them
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(B_S_EMPTY));
        // P = 2^d as binary16 pairs, row sums per head
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float p0 = ex2_approx(d[2 * k]);
          const float p1 = ex2_approx(d[2 * k + 1]);
          l[2 * k] += p0;
          l[2 * k + 1] += p1;
          pk[k] = pack_half2(p0, p1);
        }
        // rescale packet for the peer's O rows of this CTA's heads: a flag
        // and the factors, sent as soon as the decision is made
        if (sw == 0 && lane <= 16) {
          float4 f = make_float4(1.0f, 1.0f, 1.0f, 1.0f);
          if (lane == 16)
            f.x = rescaled ? 1.0f : 0.0f;
          else if (rescaled)
            f = *reinterpret_cast<const float4*>(al_own + 4 * lane);
          st_async_v4(mapa(sb0 + kSmAlphaIn + (t & 1u) * kPkt + 16 * lane, peer), f.x, f.y, f.z, f.w,
                      mapa(BAR(B_AX0 + (t & 1u)), peer));
        }
        // The P tile is free, and O holds the previous tile, once this CTA's
        // P.V of tile t-1 has completed and the copy of its rows to the peer
        // has read them.
        if (t > 0) {
          got = warp_ok(mbar_wait(BAR(B_PV_DONE), (t - 1) & 1u, abort_flag, kWaitNs));
          got = got && warp_ok(mbar_wait(BAR(B_SRC_FREE), (t - 1) & 1u, abort_flag, kWaitNs));
          ok = ok && got;
        }
        if (!ok) continue;  // the next tile's barriers take every warp out together
        tc_fence_after();
        if (o_own) {
          if (rescaled) {
            const float al = al_own[oh];
            if (__any_sync(0xffffffffu, al != 1.0f)) rescale_o(al);
          }
        } else {
          // the peer's packet: rescale this CTA's O rows of the peer's heads
          got = warp_ok(mbar_wait<true>(BAR(B_AX0 + (t & 1u)), (t >> 1) & 1u, abort_flag, kWaitNs));
          if (got) {
            const float* pkt = reinterpret_cast<const float*>(sm + kSmAlphaIn + (t & 1u) * kPkt);
            const float al = pkt[oh];
            const bool flag = pkt[64] != 0.0f;
            // the peer's packet two tiles ahead goes to this buffer
            if (hh == 0 && (quad & 1u) == 0 && lane == 0)
              mbar_arrive_expect_tx(BAR(B_AX0 + (t & 1u)), kPkt);
            if (flag && i > 0 && __any_sync(0xffffffffu, al != 1.0f)) rescale_o(al);
          }
          ok = ok && got;
        }
        // P row tt of this CTA's heads into its own P atom
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const uint32_t off = prow + uint32_t(((4 * hh + g) ^ (tt & 7)) << 4);
          *reinterpret_cast<uint4*>(sm + off) =
              make_uint4(pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(B_P_LOCAL));
        tc_fence_before();
        __syncwarp();
        if (ok && lane == 0) mbar_arrive(BAR(B_P_FULL));
      }
      // every softmax warp reaches this barrier (the loop is left together)
      if (named_bar_or(1, 256, !ok)) {
        ok = false;
        break;
      }
      // epilogue: row sums, LSE, normalized partial O of this CTA's channels
      bool got = warp_ok(mbar_wait(BAR(B_PV_DONE), (t - 1) & 1u, abort_flag, kWaitNs));
      if (named_bar_or(1, 256, !got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float mine = 0.0f;
#pragma unroll
      for (int h = 0; h < 32; ++h) {
        const float v = warp_sum_f(l[h]);
        if (lane == h) mine = v;
      }
      red[quad * 64 + 32 * hh + lane] = mine;
      named_bar_sync(2, 256);
      if (quad == 0) {
        const int hl = 32 * hh + lane;
        const float ls = (red[hl] + red[64 + hl]) + (red[128 + hl] + red[192 + hl]);
        l_own[hl] = ls;
        a.ws.part_lse[int64_t(s) * 128 + 64 * rank + hl] =
            ls > 0.0f ? (m_run[hl] + log2f(ls)) * 0.6931471805599453f : -INFINITY;
      }
      named_bar_sync(2, 256);
      if (sw == 0 && lane < 16) {
        const float4 v = *reinterpret_cast<const float4*>(l_own + 4 * lane);
        st_async_v4(mapa(sb0 + kSmLIn + 16 * lane, peer), v.x, v.y, v.z, v.w,
                    mapa(BAR(B_LX_FULL), peer));
      }
      got = warp_ok(mbar_wait<true>(BAR(B_LX_FULL), pq & 1u, abort_flag, kWaitNs));
      if (named_bar_or(1, 256, !got)) {
        ok = false;
        break;
      }
      // the peer sends the next piece's sums only after that piece's tiles
      if (sw == 0 && lane == 0) mbar_arrive_expect_tx(BAR(B_LX_FULL), 256);
      const float lr = o_own ? l_own[oh] : l_in[oh];
      const float inv = lr > 0.0f ? 1.0f / lr : 0.0f;
      float* orow = a.ws.part_o + (int64_t(s) * 128 + tt) * kDc + 256 * rank;
#pragma unroll 1
      for (uint32_t c0 = 128u * hh; c0 < 128u * hh + 128u; c0 += 32) {
        uint32_t o[32];
        tmem_ld32(tbase + lane_base + kColO + c0, o);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 32; k += 4)
          *reinterpret_cast<float4*>(orow + c0 + k) =
              make_float4(__uint_as_float(o[k]) * inv, __uint_as_float(o[k + 1]) * inv,
                          __uint_as_float(o[k + 2]) * inv, __uint_as_float(o[k + 3]) * inv);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_O_EMPTY));
      ++pq;
    }
  } else {
    // ------------------------------------------------------------ dequant
    setmaxnreg_to<kRegsLaunch, RegSplit<kCBits>::dq>();
    // thread = token row tt of the tile (tensor-memory lane); rows 0-63 come
    // from the tile's first block, 64-127 from its second.  Units per tile:
    //   dh 0: A (tensor memory) the other half's chunks 0, 1, 2;
    //         B (ring) this half's early chunks 0 and 1 of the tile;
    //   dh 1: A the other half's chunk 3, this half's late chunk, RoPE;
    //         B this half's third early chunk; C the previous tile's late
    //         chunk into ring slot 3 (after that tile's predecessor's P.V).
    const int dw = warp - kDqWarp0, dh = dw >> 2;
    const uint32_t quad = uint32_t(warp & 3);
    const int tt = int(quad) * 32 + lane, bi = tt >> 6, slot = tt & 63;
    const uint32_t lane_base = (quad * 32u) << 16;
    const uint32_t row_off = uint32_t(tt >> 3) * 1024u + uint32_t(tt & 7) * 128u;
    const int sw7 = tt & 7;
    const int qt = int(threadIdx.x) - kDqWarp0 * 32;  // 0..255
    // this piece's queries (this CTA's 64 heads), binary16, SW128 K-major
    auto stage_q = [&](int b) {
      bool bad = false;
#pragma unroll 1
      for (int r0 = 0; r0 < 18; r0 += 9) {
        uint4 qv[9];
#pragma unroll
        for (int k = 0; k < 9; ++k) {
          const int idx = qt + 256 * (r0 + k), h = idx / 72, sg = idx % 72;
          const int64_t hv = int64_t(b) * 128 + 64 * int(rank) + h;
          const __nv_bfloat16* src =
              sg < 64 ? a.q_c + hv * kDc + sg * 8 : a.q_r + hv * kDr + (sg - 64) * 8;
          qv[k] = *reinterpret_cast<const uint4*>(src);
        }
#pragma unroll
        for (int k = 0; k < 9; ++k) {
          const int idx = qt + 256 * (r0 + k), h = idx / 72, sg = idx % 72;
          const uint32_t in[4] = {qv[k].x, qv[k].y, qv[k].z, qv[k].w};
          uint32_t o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            o[e] = pack_half2(__uint_as_float(in[e] << 16), __uint_as_float(in[e] & 0xffff0000u));
            bad |= h2_inf(o[e]);
          }
          const int c = sg >> 3, g = sg & 7;
          unsigned char* row = sm + kSmQ + c * kQChunk + (h >> 3) * 1024 + (h & 7) * 128;
          *reinterpret_cast<uint4*>(row + ((g ^ (h & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
      if (bad) set_status(a.status, QMLA_STATUS_BAD_QUERY);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_Q_FULL));
    };
    unsigned char* ring = sm + kSmRing;
    uint32_t t = 0;
    bool ok = true;
    // this thread's row block in the previous tile (its late chunk goes to slot 3)
    const uint8_t* prev_blk = nullptr;
    // Packed codes: the A units of a tile are loaded while the previous tile's
    // B units are processed, the B units (and the previous tile's late chunk)
    // while its own A units are.  Block ids come 32 at a time from lane
    // registers, so no code load waits for a block-table load.
    // A units in processing order (pair k = 0, 1, 2), rotated down as they
    // are consumed so that one copy of the unit code serves all three; B
    // units: dh 0 two early chunks, dh 1 one early chunk and the previous
    // tile's late chunk.  Each set is loaded as soon as the previous tile has
    // consumed it, about a tile ahead of its use.
    Unit ua0, ua1, ua2, ub0, ub1;
    auto load_a = [&](const uint8_t* blk, uint32_t t2) {
      if constexpr (!kBF16) {
        if (dh == 0) {
          load_content<kCBits>(ua0, blk, G, 4 * int(peer) + 0, slot);
          load_content<kCBits>(ua1, blk, G, 4 * int(peer) + 1, slot);
          load_content<kCBits>(ua2, blk, G, 4 * int(peer) + 2, slot);
        } else {
          load_content<kCBits>(ua0, blk, G, 4 * int(peer) + 3, slot);
          load_content<kCBits>(ua1, blk, G, 4 * int(rank) + ((t2 & 1u) ? 0 : 3), slot);
          load_rope(ua2, blk, G, slot);
        }
      }
    };
    for (int s = wr.x; ok && s <= wr.y; ++s) {
      const int4 pc = a.ws.pieces[s];
      const int nt = piece_tiles(pc);
      if (nt == 0) continue;
      const int L = seq_len_clamped(a, pc.x);
      const int32_t* btab = a.block_table + int64_t(pc.x) * a.max_blocks_per_seq;
      // block ids of blocks jb0 .. jb0+63 of the piece, one per lane in two registers
      int jb0 = pc.y;
      int32_t ids_a = (jb0 + lane < pc.z) ? btab[jb0 + lane] : -1;
      int32_t ids_b = (jb0 + 32 + lane < pc.z) ? btab[jb0 + 32 + lane] : -1;
      // block of this thread's row in tile i2 (nullptr: no such row, a bad
      // block id, or a token past the sequence: read as zeros); called by the
      // whole warp
      auto tile_block = [&](int i2) -> const uint8_t* {
        const int j = pc.y + 2 * i2 + bi, k = j - jb0;  // 0 <= k < 64
        const int32_t va = __shfl_sync(0xffffffffu, ids_a, k & 31);
        const int32_t vb = __shfl_sync(0xffffffffu, ids_b, k & 31);
        if (j >= pc.z) return nullptr;
        const int32_t blk = k < 32 ? va : vb;
        if (blk < 0 || blk >= a.num_blocks) {
          if (lane == 0 && (dw == 0 || dw == 2)) set_status(a.status, QMLA_STATUS_BAD_BLOCK);
          return nullptr;
        }
        return slot < L - j * kT ? a.blocks + int64_t(blk) * G.block : nullptr;
      };
      const uint8_t* blk = tile_block(0);
      load_a(blk, t);
      auto load_b = [&](const uint8_t* b_blk, const uint8_t* c_blk, uint32_t t2) {
        if constexpr (!kBF16) {
          const uint32_t o2 = t2 & 1u;
          if (dh == 0) {
            load_content<kCBits>(ub0, b_blk, G, 4 * int(rank) + 0 + int(o2), slot);
            load_content<kCBits>(ub1, b_blk, G, 4 * int(rank) + 1 + int(o2), slot);
          } else {
            load_content<kCBits>(ub0, b_blk, G, 4 * int(rank) + 2 + int(o2), slot);
            // the late chunk of tile t2-1 (slot 3 after tile t2's B units)
            load_content<kCBits>(ub1, c_blk, G, 4 * int(rank) + (o2 ? 3 : 0), slot);
          }
        }
      };
      load_b(blk, prev_blk, t);
      const uint8_t* blk_next = nt > 1 ? tile_block(1) : nullptr;
      for (int i = 0; i < nt; ++i, ++t) {
        if (pc.y + 2 * i - jb0 >= 32) {  // slide the window (tile i+1 stays inside it)
          jb0 += 32;
          ids_a = ids_b;
          ids_b = (jb0 + 32 + lane < pc.z) ? btab[jb0 + 32 + lane] : -1;
        }
        if (i == 0) {
          // this piece's queries, once every QK product of the previous piece is done
          if (!warp_ok(t == 0 || mbar_wait(BAR(B_S_FULL), (t - 1) & 1u, abort_flag, kWaitNs))) {
            ok = false;
            break;
          }
          stage_q(pc.x);
        }
        const uint32_t odd = t & 1u;
        const uint32_t base = odd ? 3u : 0u;
        const uint32_t late_prev = odd ? 3u : 0u;  // the previous tile's late chunk
        // ---- A: tensor-memory unit pairs, each once the previous tile's QK
        // products on it are complete
#pragma unroll 1
        for (int k = 0; k < 3; ++k) {
          if (!warp_ok(t == 0 ||
                       mbar_wait(BAR(B_KT_EMPTY + k), (t - 1) & 1u, abort_flag, kWaitNs))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t taddr = tbase + lane_base + kColK + 32u * uint32_t(dh == 0 ? k : 3 + k);
          if constexpr (!kBF16) {
            const Unit u = ua0;
            ua0 = ua1;
            ua1 = ua2;
            unit_to_tmem<kCBits>(u, dh == 1 && k == 2, taddr);
          } else {
            uint32_t v[32];
            if (dh == 1 && k == 2)
              load_bf16_rope(v, blk, G, slot);
            else
              load_bf16_content(v, blk, G,
                                dh == 0 ? 4 * int(peer) + k
                                        : (k == 0 ? 4 * int(peer) + 3 : 4 * int(rank) + (odd ? 0 : 3)),
                                slot);
            bf16_to_f16(v);
            tmem_st32(taddr, v);
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          // (the test hook withholds the first arrival of the first CTA of each pair)
          if (lane == 0 && !(a.withhold && t == 0 && rank == 0)) mbar_arrive(BAR(B_KT_FULL + k));
        }
        if (!ok) break;
        // ---- the next tile's A codes
        if (i + 1 < nt) load_a(blk_next, t + 1);
        // ---- B: this half's early chunks into the ring (slots of tile t-2)
        if (!warp_ok(t < 2 || mbar_wait(BAR(B_PV_DONE), t & 1u, abort_flag, kWaitNs))) {
          ok = false;
          break;
        }
        if constexpr (!kBF16) {
          unit_to_ring<kCBits>(ub0, ring + (base + (dh == 0 ? 0u : 2u) + odd) * kAtom, row_off, sw7);
          if (dh == 0) unit_to_ring<kCBits>(ub1, ring + (base + 1u + odd) * kAtom, row_off, sw7);
        } else {
#pragma unroll 1
          for (int k = 0; k < (dh == 0 ? 2 : 1); ++k) {
            const uint32_t c = (dh == 0 ? uint32_t(k) : 2u) + odd;
            uint32_t v[32];
            load_bf16_content(v, blk, G, 4 * int(rank) + int(c), slot);
            bf16_to_f16(v);
            st_row64(ring + (base + c) * kAtom, row_off, sw7, v);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(B_RING_FULL));
        // ---- C: the previous tile's late chunk into slot 3 (freed with tile t-2's P.V)
        if (dh == 1 && t >= 1) {
          if constexpr (!kBF16) {
            unit_to_ring<kCBits>(ub1, ring + 3u * kAtom, row_off, sw7);
          } else {
            uint32_t v[32];
            load_bf16_content(v, prev_blk, G, 4 * int(rank) + int(late_prev), slot);
            bf16_to_f16(v);
            st_row64(ring + 3u * kAtom, row_off, sw7, v);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR(B_LATE_FULL));
        }
        // ---- the next tile's B codes and this tile's late chunk
        if (i + 1 < nt) load_b(blk_next, blk, t + 1);
        prev_blk = blk;
        blk = blk_next;
        blk_next = i + 2 < nt ? tile_block(i + 2) : nullptr;
      }
    }
    // the last tile's late chunk (tile t-1), once tile t-2's P.V has freed slot 3
    if (ok && dh == 1 && t >= 1) {
      const uint32_t lc = ((t - 1) & 1u) ? 0u : 3u;
      uint32_t v[32];
      if constexpr (!kBF16)
        load_content<kCBits>(ub1, prev_blk, G, 4 * int(rank) + int(lc), slot);
      else
        load_bf16_content(v, prev_blk, G, 4 * int(rank) + int(lc), slot);
      const bool got = t < 2 || mbar_wait(BAR(B_PV_DONE), t & 1u, abort_flag, kWaitNs);
      if (warp_ok(got)) {
        if constexpr (!kBF16) {
          unit_to_ring<kCBits>(ub1, ring + 3u * kAtom, row_off, sw7);
        } else {
          bf16_to_f16(v);
          st_row64(ring + 3u * kAtom, row_off, sw7, v);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(B_LATE_FULL));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    if (threadIdx.x == 0) set_status(a.status, QMLA_STATUS_TIMEOUT);
    // Unwinding: the peer may have sent rows or sums this CTA never waited
    // for.  Give stores still in flight time to land before the cluster
    // barrier lets either CTA leave.
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 100000ull) {
    }
  }
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
  cluster_sync();  // no CTA leaves while its peer may still touch its shared memory
}

}  // namespace

cudaError_t launch_decode_tc128(const DecodeArgs& a, cudaStream_t stream) {
  static int done4[kMaxDevices], done2[kMaxDevices], done16[kMaxDevices];
  DecodeArgs b = a;
  // A second piece costs a worker about three tiles (the pipeline's drain
  // and refill, the epilogue, the queries' staging; measured by the charge
  // that makes the 64-sequence ragged workload fastest); the split charges
  // it six blocks.
  b.piece_cost = 6;
  cudaError_t e = launch_plan(b, stream);
  if (e != cudaSuccess) return e;
  auto kernel = a.fmt == QMLA_C4R4   ? decode_tc128_kernel<4>
                : a.fmt == QMLA_C2R4 ? decode_tc128_kernel<2>
                                     : decode_tc128_kernel<16>;
  e = ensure_smem_attr(kernel, int(kSmDyn),
                       a.fmt == QMLA_C4R4 ? done4 : a.fmt == QMLA_C2R4 ? done2 : done16,
                       int(kRegsLaunch));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(2 * a.workers));
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
