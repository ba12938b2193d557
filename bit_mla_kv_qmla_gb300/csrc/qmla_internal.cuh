// qmla_internal.cuh - layout constants and shared device helpers of the CUDA
// path.  The byte layout implemented here is the one specified in qmla.h.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include "qmla.h"

namespace qmla {

constexpr int kDc = QMLA_D_C;
constexpr int kDr = QMLA_D_R;
constexpr int kG = QMLA_GROUP;
constexpr int kT = QMLA_BLOCK_TOKENS;

// Per-format byte geometry of a 64-token block.
struct Geom {
  int fmt;
  int cbits;        // content code bits (4, 2; 16 = bf16)
  int code_bytes;   // bytes of one content group of one token (32, 16, 128)
  int half;         // bytes of one half-block
  int content_off;  // offset of content codes inside a half (0)
  int rope_off;     // offset of RoPE codes inside a half
  int sz_off;       // offset of content scale/zero inside a half
  int rope_sz_off;  // offset of the shared RoPE scale/zero inside the block
  int block;        // bytes of a block
  int rbits;        // RoPE code bits (4, 2; 16 = bf16)
  int rope_bytes;   // bytes of one token's 32 RoPE channels in a half (16, 8, 64)
};

__host__ __device__ constexpr Geom geom(int fmt) {
  return fmt == QMLA_C4R4 ? Geom{QMLA_C4R4, 4, 32, 10240, 0, 8192, 9216, 20480, 20736, 4, 16}
       : fmt == QMLA_C2R4 ? Geom{QMLA_C2R4, 2, 16, 6144, 0, 4096, 5120, 12288, 12544, 4, 16}
       : fmt == QMLA_C4R2 ? Geom{QMLA_C4R2, 4, 32, 9728, 0, 8192, 8704, 19456, 19712, 2, 8}
       : fmt == QMLA_C2R2 ? Geom{QMLA_C2R2, 2, 16, 5632, 0, 4096, 4608, 11264, 11520, 2, 8}
                          : Geom{QMLA_BF16, 16, 128, 36864, 0, 32768, -1, -1, 73728, 16, 64};
}

// Device status word: OR in a bit (relaxed; read by the host after a sync).
__device__ __forceinline__ void set_status(int32_t* status, int bits) {
  if (status) atomicOr(status, bits);
}

// Number of 64-token blocks of a sequence of length L.
__host__ __device__ __forceinline__ int blocks_of(int L) { return (L + kT - 1) / kT; }

// Split plan.  The blocks of all sequences, concatenated in sequence order,
// are cut into Pe = min(P, N) contiguous ranges of near-equal size, one per
// worker (CTA or CTA pair), so every planned worker owns at least one block;
// workers >= Pe get nothing.  Worker w < Pe owns global blocks
// [start(w), start(w+1)) with start(w) = floor(w*N/Pe).  A worker range that
// touches k sequences produces k partial results ("pieces"); the pieces of
// sequence b get consecutive slots base_b .. base_b + n_b - 1.
__host__ __device__ __forceinline__ int64_t plan_workers(int64_t N, int64_t P) {
  return N < P ? N : P;
}
__host__ __device__ __forceinline__ int64_t plan_start(int64_t w, int64_t N, int64_t Pe) {
  return Pe > 0 ? (w * N) / Pe : 0;
}
// Worker owning global block g (0 <= g < N, Pe >= 1).
__host__ __device__ __forceinline__ int64_t plan_owner(int64_t g, int64_t N, int64_t Pe) {
  return ((g + 1) * Pe - 1) / N;
}

// Workspace layout for the decode (each region 256-byte aligned):
//   seq table  [B] int2   (first slot, number of pieces) per sequence
//   part LSE   [slots][H] float
//   part O     [slots][H][512] float
//   pieces     [slots] int4 (sequence, first block, end block, 0) per slot
//   worker     [slots] int2 (first slot, last slot) per worker (P <= slots)
struct Workspace {
  int2* seq_table;
  float* part_lse;
  float* part_o;
  int4* pieces;
  int2* wrange;
};
__host__ __device__ __forceinline__ size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
__host__ __device__ __forceinline__ size_t workspace_bytes(int batch, int heads, int slots) {
  return align256(size_t(batch) * sizeof(int2)) + align256(size_t(slots) * heads * sizeof(float)) +
         align256(size_t(slots) * heads * kDc * sizeof(float)) +
         align256(size_t(slots) * sizeof(int4)) + align256(size_t(slots) * sizeof(int2));
}
__host__ __device__ __forceinline__ Workspace carve(void* ws, int batch, int heads, int slots) {
  char* p = static_cast<char*>(ws);
  Workspace w;
  w.seq_table = reinterpret_cast<int2*>(p);
  p += align256(size_t(batch) * sizeof(int2));
  w.part_lse = reinterpret_cast<float*>(p);
  p += align256(size_t(slots) * heads * sizeof(float));
  w.part_o = reinterpret_cast<float*>(p);
  p += align256(size_t(slots) * heads * kDc * sizeof(float));
  w.pieces = reinterpret_cast<int4*>(p);
  p += align256(size_t(slots) * sizeof(int4));
  w.wrange = reinterpret_cast<int2*>(p);
  return w;
}

// Arguments shared by the decode kernels.
struct DecodeArgs {
  int fmt;
  const uint8_t* blocks;
  int64_t num_blocks;
  const int32_t* block_table;
  int max_blocks_per_seq;
  const int32_t* seq_lens;
  int max_seq_len;
  int batch;
  int heads;
  const __nv_bfloat16* q_c;
  const __nv_bfloat16* q_r;
  float scale;
  Workspace ws;
  int workers;  // P
  int32_t* status;
  // The kernel plans its own pieces (no planner launch); set by the
  // launchers that support it.
  int fused_plan = 0;
  // Cost of starting a piece, in blocks: the split counts this many extra
  // blocks at the start of every non-empty sequence, so a worker whose range
  // crosses into another sequence gets that much less context.
  int piece_cost = 0;
  // Multi-token query decode: heads = q_len * q_heads virtual heads, virtual
  // head v being head v % q_heads of query v / q_heads; query i sits at
  // position L - q_len + i and attends only to tokens up to it.  q_heads = 0:
  // one query per sequence, every cached token visible.
  int q_len = 1;
  int q_heads = 0;
  // Test hook (qmla_decode_timeout_test only): the 16-head tensor-core
  // kernel's dequantization warps withhold their first arrival, so that the
  // bounded waits run out and the kernel reports QMLA_STATUS_TIMEOUT.
  int withhold = 0;
};

// Raise a kernel's dynamic shared-memory limit once per device (the
// attribute is per function and device; repeating it costs a runtime call on
// every launch).  `done` is the caller's own per-device record for this kernel.
constexpr int kMaxDevices = 64;
// regs > 0: the kernel hands registers between warpgroups with setmaxnreg
// on the assumption that it launches with `regs` per thread; a build that
// compiled it to another count is refused here (its register increases
// would wait on registers nobody released) instead of launched.
template <typename K>
inline cudaError_t ensure_smem_attr(K* kernel, int bytes, int (&done)[kMaxDevices],
                                    int regs = 0) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDevices && done[dev] >= bytes) return cudaSuccess;
  if (regs > 0) {
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kernel);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != regs) return cudaErrorInvalidDeviceFunction;
  }
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev >= 0 && dev < kMaxDevices) done[dev] = bytes;
  return e;
}

// Kernel launchers (each defined next to its kernel).  They return a
// cudaError_t from the launch.
cudaError_t launch_append(int fmt, uint8_t* blocks, int64_t num_blocks, const int32_t* table,
                          int max_blocks, int32_t* positions, int batch, int n_new,
                          const __nv_bfloat16* latent, const __nv_bfloat16* rope,
                          int32_t* status, bool advance, cudaStream_t stream);
int simt_workers(int sms);
cudaError_t launch_decode_simt(const DecodeArgs& a, cudaStream_t stream);
int tc_workers(int sms, int heads);
bool tc_supported(int fmt, int heads);
cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_combine(const Workspace& ws, int batch, int heads, __nv_bfloat16* out,
                           float* lse, cudaStream_t stream);

}  // namespace qmla
