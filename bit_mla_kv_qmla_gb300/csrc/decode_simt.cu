// decode_simt.cu - CUDA-core decode over the low-bit paged cache.
//
// Serves every head count that is a multiple of 16 (the tensor-core kernels
// cover the MLA shapes 16 and 128) and every cache format.  It computes the
// decode formula of qmla.h in binary32: each 32-token sub-tile is unpacked
// and dequantized into shared memory (x_hat = code*scale + zero, multiply and
// add each rounded to nearest, as specified), scores and the running softmax
// are kept per head, and the content latent is accumulated into O in
// registers.  Dequantization happens inside the attention kernel, as the
// "Low-bit kernel" node of the flowchart of "QuantMLA: INT4 (and INT2) for
// both halves of the MLA cache" describes; nothing is expanded to a 16-bit
// cache in global memory.
//
// Grid: (workers P, head groups H/16); 256 threads; each worker walks its
// share of the context (plan.cuh) and writes one partial per piece.

#include <cfloat>

#include "plan.cuh"

namespace qmla {
namespace {

constexpr int kHG = 16;       // heads per CTA
constexpr int kTT = 32;       // tokens per sub-tile
constexpr int kLD = 577;      // padded row of 576 channels (bank spread)
constexpr int kThreads = 256;

struct SimtShared {
  float q[kHG][kLD];
  float x[kTT][kLD];
  float p[kTT][kHG];
  float alpha[kHG];
  float m[kHG];
  float l[kHG];
};

// Dequantize 8 consecutive channels (segment seg of 72: 64 content + 8 RoPE)
// of token `slot` of block `blk` into out[8].
__device__ __forceinline__ void dequant8(const Geom& G, const uint8_t* blk, int slot, int seg,
                                         float* out) {
  if (G.fmt == QMLA_BF16) {
    const uint8_t* src;
    if (seg < 64) {
      const int g = seg / 8;
      src = blk + (g / 4) * G.half + G.content_off + ((g % 4) * kT + slot) * 128 + (seg % 8) * 16;
    } else {
      const int r = seg - 64;
      src = blk + (r / 4) * G.half + G.rope_off + slot * 64 + (r % 4) * 16;
    }
    const uint4 v = *reinterpret_cast<const uint4*>(src);
    const uint32_t wds[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      out[2 * k] = __uint_as_float(wds[k] << 16);
      out[2 * k + 1] = __uint_as_float(wds[k] & 0xffff0000u);
    }
    return;
  }
  uint32_t word, sz;
  int bits, first;  // first channel of the segment inside its word
  if (seg < 64) {
    const int g = seg / 8, h = g / 4, gi = g % 4;
    const uint8_t* half = blk + h * G.half;
    bits = G.cbits;
    const int ch = (seg % 8) * 8;  // channel inside the group
    const int per_word = 32 / bits;
    word = reinterpret_cast<const uint32_t*>(half + G.content_off +
                                             (gi * kT + slot) * G.code_bytes)[ch / per_word];
    first = ch % per_word;
    sz = *reinterpret_cast<const uint32_t*>(half + G.sz_off + (gi * kT + slot) * 4);
  } else {
    const int r = seg - 64;  // RoPE channels 8r .. 8r+7, block half r / 4
    bits = G.rbits;
    const int ch = (r % 4) * 8;  // channel inside the half's 32
    const int per_word = 32 / bits;
    word = reinterpret_cast<const uint32_t*>(blk + (r / 4) * G.half + G.rope_off +
                                             slot * G.rope_bytes)[ch / per_word];
    first = ch % per_word;
    sz = *reinterpret_cast<const uint32_t*>(blk + G.rope_sz_off + slot * 4);
  }
  const float s = __half2float(__ushort_as_half(uint16_t(sz & 0xffff)));
  const float z = __half2float(__ushort_as_half(uint16_t(sz >> 16)));
  const int per_half = 16 / bits;
  const uint32_t mask = (1u << bits) - 1;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int cw = first + k;  // channel inside the word
    const int pos = (cw >> 1) + (cw & 1) * per_half;
    const uint32_t code = (word >> (bits * pos)) & mask;
    out[k] = __fadd_rn(__fmul_rn(float(code), s), z);
  }
}

__global__ void __launch_bounds__(kThreads) decode_simt_kernel(DecodeArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SimtShared& S = *reinterpret_cast<SimtShared*>(smem_raw);
  __shared__ PlanState st;
  __shared__ int s_more;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int w = blockIdx.x, hg = blockIdx.y;
  const Geom G = geom(a.fmt);

  if (warp == 0) {
    const int64_t N = plan_total(a);
    if (lane == 0) {
      st.total_blocks = N;
      st.carry_blocks = 0;
      st.carry_slots = 0;
      st.next_seq = 0;
    }
    __syncwarp();
  }
  __syncthreads();
  const bool publish = (w == 0 && hg == 0);

  while (true) {
    if (warp == 0) {
      const bool more = plan_next(a, st, w, publish);
      if (lane == 0) s_more = more;
    }
    __syncthreads();
    if (!s_more) break;
    const int npieces = st.n;
    for (int k = 0; k < npieces; ++k) {
      const Piece pc = st.list[k];
      const int b = pc.b;
      const int L = seq_len_clamped(a, b);
      // queries of this head group, binary32
      for (int i = tid; i < kHG * (kDc + kDr); i += kThreads) {
        const int h = i / (kDc + kDr), c = i % (kDc + kDr);
        const int64_t hq = int64_t(b) * a.heads + hg * kHG + h;
        S.q[h][c] = (c < kDc) ? __bfloat162float(a.q_c[hq * kDc + c])
                              : __bfloat162float(a.q_r[hq * kDr + (c - kDc)]);
      }
      if (tid < kHG) {
        S.m[tid] = -FLT_MAX;
        S.l[tid] = 0.0f;
      }
      float acc[kHG][2];
#pragma unroll
      for (int h = 0; h < kHG; ++h) acc[h][0] = acc[h][1] = 0.0f;
      __syncthreads();

      for (int j = pc.j0; j < pc.j1; ++j) {
        const int32_t blk_id = a.block_table[int64_t(b) * a.max_blocks_per_seq + j];
        if (blk_id < 0 || blk_id >= a.num_blocks) {
          if (tid == 0) set_status(a.status, QMLA_STATUS_BAD_BLOCK);
          continue;
        }
        const uint8_t* blk = a.blocks + int64_t(blk_id) * G.block;
        const int n_valid = min(kT, L - j * kT);
        for (int t0 = 0; t0 < n_valid; t0 += kTT) {
          const int nv = min(kTT, n_valid - t0);
          // 1. unpack + dequantize the sub-tile
          for (int it = tid; it < kTT * 72; it += kThreads) {
            const int t = it / 72, seg = it % 72;
            float v[8];
            if (t < nv) {
              dequant8(G, blk, t0 + t, seg, v);
            } else {
#pragma unroll
              for (int k2 = 0; k2 < 8; ++k2) v[k2] = 0.0f;
            }
            const int c0 = (seg < 64) ? seg * 8 : kDc + (seg - 64) * 8;
#pragma unroll
            for (int k2 = 0; k2 < 8; ++k2) S.x[t][c0 + k2] = v[k2];
          }
          __syncthreads();
          // 2. scores: thread (h, token lane) for tokens tl and tl + 16
          {
            const int h = tid / 16, tl = tid % 16;
            float s0 = 0.0f, s1 = 0.0f;
            for (int c = 0; c < kDc + kDr; ++c) {
              const float qv = S.q[h][c];
              s0 = fmaf(qv, S.x[tl][c], s0);
              s1 = fmaf(qv, S.x[tl + 16][c], s1);
            }
            // tokens virtual head hg*kHG+h may see (a prefix of them in a
            // multi-token query decode)
            const int vis = visible_tokens(a, hg * kHG + h, L) - (j * kT + t0);
            S.p[tl][h] = (tl < nv && tl < vis) ? s0 * a.scale : -INFINITY;
            S.p[tl + 16][h] = (tl + 16 < nv && tl + 16 < vis) ? s1 * a.scale : -INFINITY;
          }
          __syncthreads();
          // 3. online softmax: warp handles heads 2*warp, 2*warp+1; lane = token
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int h = 2 * warp + hh;
            const float v = S.p[lane][h];
            float mt = v;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
            const float m_old = S.m[h];
            // -inf only while a multi-token query's head has seen no token
            const float m_new = fmaxf(m_old, mt);
            const float p = m_new == -INFINITY ? 0.0f : __expf(v - m_new);
            float ps = p;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
            __syncwarp();
            S.p[lane][h] = p;
            if (lane == 0) {
              const float al = m_new == -INFINITY ? 1.0f : __expf(m_old - m_new);
              S.alpha[h] = al;
              S.m[h] = m_new;
              S.l[h] = S.l[h] * al + ps;
            }
          }
          __syncthreads();
          // 4. O[h][c0..c0+1] = alpha*O + sum_t p[t][h] * x[t][c]
          {
            const int c0 = 2 * tid;
#pragma unroll
            for (int h = 0; h < kHG; ++h) {
              const float al = S.alpha[h];
              acc[h][0] *= al;
              acc[h][1] *= al;
            }
            for (int t = 0; t < nv; ++t) {
              const float x0 = S.x[t][c0], x1 = S.x[t][c0 + 1];
#pragma unroll
              for (int h = 0; h < kHG; ++h) {
                const float p = S.p[t][h];
                acc[h][0] = fmaf(p, x0, acc[h][0]);
                acc[h][1] = fmaf(p, x1, acc[h][1]);
              }
            }
          }
          __syncthreads();
        }
      }
      // epilogue: normalized partial O and LSE of this piece
      {
        const int c0 = 2 * tid;
#pragma unroll
        for (int h = 0; h < kHG; ++h) {
          const float l = S.l[h];
          const float inv = (l > 0.0f) ? 1.0f / l : 0.0f;
          const int hq = hg * kHG + h;
          float2 o = make_float2(acc[h][0] * inv, acc[h][1] * inv);
          *reinterpret_cast<float2*>(a.ws.part_o + (int64_t(pc.slot) * a.heads + hq) * kDc + c0) = o;
        }
        if (tid < kHG) {
          const float l = S.l[tid];
          a.ws.part_lse[int64_t(pc.slot) * a.heads + hg * kHG + tid] =
              (l > 0.0f) ? S.m[tid] + logf(l) : -INFINITY;
        }
      }
      __syncthreads();
    }
    __syncthreads();
  }
}

}  // namespace

int simt_workers(int sms) { return 2 * sms; }

cudaError_t launch_decode_simt(const DecodeArgs& a, cudaStream_t stream) {
  static int smem_attr_done[kMaxDevices];
  const size_t smem = sizeof(SimtShared);
  cudaError_t e = ensure_smem_attr(decode_simt_kernel, int(smem), smem_attr_done);
  if (e != cudaSuccess) return e;
  dim3 grid(unsigned(a.workers), unsigned(a.heads / kHG));
  decode_simt_kernel<<<grid, kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace qmla
