// plan.cuh - device side of the split plan shared by the decode kernels.
//
// The context of every sequence is attended in pieces (split-KV); the pieces
// are merged afterwards by log-sum-exp.  All sequences' 64-token blocks are
// concatenated in sequence order and cut into min(P, N) near-equal contiguous
// ranges, one per worker, so every worker gets the same number of blocks
// whatever the length mix.  Optionally every non-empty sequence counts a few
// extra blocks at its start (the piece cost), so that a worker that starts a
// second piece, and pays for that piece's start and epilogue, gets less
// context; a worker may then own no real block and has no piece.  One warp
// scans seq_lens (32 sequences per step) with warp prefix sums; no host-side
// copy of the lengths is needed.
#pragma once

#include "qmla_internal.cuh"

namespace qmla {

__device__ __forceinline__ int warp_incl_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Clamped number of blocks of sequence b (flags over-long or negative lengths).
__device__ __forceinline__ int seq_blocks(const DecodeArgs& a, int b, bool flag) {
  int L = a.seq_lens[b];
  const int cap = min(a.max_seq_len, a.max_blocks_per_seq * kT);
  if (L < 0 || L > cap) {
    if (flag) set_status(a.status, QMLA_STATUS_BAD_LEN);
    L = max(0, min(L, cap));
  }
  return blocks_of(L);
}
__device__ __forceinline__ int seq_len_clamped(const DecodeArgs& a, int b) {
  const int cap = min(a.max_seq_len, a.max_blocks_per_seq * kT);
  return max(0, min(a.seq_lens[b], cap));
}

// Cached tokens virtual head v attends to in a sequence of L tokens (a prefix
// of them in a multi-token query decode; possibly <= 0: none).
__device__ __forceinline__ int visible_tokens(const DecodeArgs& a, int v, int L) {
  return a.q_heads > 0 ? L - (a.q_len - 1 - v / a.q_heads) : L;
}

// One piece of work: blocks [j0, j1) of sequence b, partial result to `slot`.
struct Piece {
  int b, j0, j1, slot;
};

// Scanner state kept in shared memory by the scanning warp.
struct PlanState {
  int64_t total_blocks;  // N
  int64_t carry_blocks;  // blocks of sequences before the current chunk
  int carry_slots;       // pieces of sequences before the current chunk
  int next_seq;          // first sequence of the next chunk
  int n;                 // pieces found in the last chunk
  Piece list[32];
};

// Extent of a sequence of nb blocks in the split: its blocks plus the piece
// cost (none for an empty sequence).
__device__ __forceinline__ int plan_extent(const DecodeArgs& a, int nb) {
  return nb > 0 ? nb + a.piece_cost : 0;
}

// Called by ONE full warp: total extent N of all sequences.
__device__ __forceinline__ int64_t plan_total(const DecodeArgs& a) {
  const int lane = threadIdx.x & 31;
  int64_t tot = 0;
  for (int b0 = 0; b0 < a.batch; b0 += 32) {
    const int b = b0 + lane;
    const int nb = (b < a.batch) ? seq_blocks(a, b, true) : 0;
    tot += warp_sum(plan_extent(a, nb));
  }
  return tot;
}

// Called by ONE full warp: scan the next chunk of 32 sequences and list the
// pieces worker w owns there.  Worker 0 also publishes the per-sequence merge
// table.  Returns false when no sequence is left or the worker range is past.
__device__ __forceinline__ bool plan_next(const DecodeArgs& a, PlanState& st, int64_t w,
                                          bool publish) {
  const int lane = threadIdx.x & 31;
  const int64_t N = st.total_blocks, P = plan_workers(N, a.workers);
  const int64_t g0 = (w < P) ? plan_start(w, N, P) : N;
  const int64_t g1 = (w < P) ? plan_start(w + 1, N, P) : N;
  if (lane == 0) st.n = 0;
  __syncwarp();
  if (st.next_seq >= a.batch || (!publish && st.carry_blocks >= g1)) return false;
  const int b = st.next_seq + lane;
  const int nb = (b < a.batch) ? seq_blocks(a, b, false) : 0;
  const int ext = plan_extent(a, nb);
  const int incl = warp_incl_scan(ext);
  // the sequence's real blocks start after its piece cost
  const int64_t S = st.carry_blocks + (incl - ext) + a.piece_cost;
  int np = 0;
  int64_t pf = 0;
  if (nb > 0) {
    pf = plan_owner(S, N, P);
    const int64_t pl = plan_owner(S + nb - 1, N, P);
    np = int(pl - pf + 1);
  }
  const int np_incl = warp_incl_scan(np);
  const int base = st.carry_slots + (np_incl - np);
  if (publish && b < a.batch) a.ws.seq_table[b] = make_int2(base, np);
  const bool mine = nb > 0 && S < g1 && S + nb > g0;
  const unsigned ballot = __ballot_sync(0xffffffffu, mine);
  if (mine) {
    const int idx = __popc(ballot & ((1u << lane) - 1));
    Piece p;
    p.b = b;
    p.j0 = int(max(g0 - S, int64_t(0)));
    p.j1 = int(min(g1 - S, int64_t(nb)));
    p.slot = base + int(w - pf);
    st.list[idx] = p;
  }
  const int chunk_blocks = __shfl_sync(0xffffffffu, incl, 31);
  const int chunk_slots = __shfl_sync(0xffffffffu, np_incl, 31);
  __syncwarp();
  if (lane == 0) {
    st.n = __popc(ballot);
    st.carry_blocks += chunk_blocks;
    st.carry_slots += chunk_slots;
    st.next_seq += 32;
  }
  __syncwarp();
  return true;
}

}  // namespace qmla
