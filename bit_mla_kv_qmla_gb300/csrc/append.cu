// append.cu - quantize-and-pack of new tokens into the paged low-bit cache.
//
// The two quantizers of "QuantMLA: INT4 (and INT2) for both halves of the MLA
// cache" (flowchart: content quant INT4 or INT2, RoPE quant INT4), written in
// quant.cuh.  One CTA per new token, one warp per 64-channel group (8 content
// + 1 RoPE), each lane holding two consecutive channels.  The whole append is
// one pass over the new tokens: it is launch-bound for decode-sized appends.

#include "quant.cuh"

namespace qmla {
namespace {

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
  quant::store_group(fmt, blocks + int64_t(blk_id) * G.block, int(pos % kT), warp, v, lane);
}

__global__ void advance_kernel(int32_t* positions, int batch, int n_new) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < batch) positions[b] += n_new;
}

}  // namespace

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
