// qmla_api.cu - the exported C ABI (declared and documented in qmla.h).
//
// Host code only: argument validation, choice of kernel, split planning
// constants and launches on the caller's stream.  No allocation, no global
// state beyond what the CUDA runtime keeps per function.

#include <cstdio>

#include "qmla_internal.cuh"

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
bool known_format(int f) {
  return f == QMLA_C4R4 || f == QMLA_C2R4 || f == QMLA_BF16 || f == QMLA_C4R2 || f == QMLA_C2R2;
}

int device_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

bool heads_served(int fmt, int heads) {
  return qmla::tc_supported(fmt, heads) || (heads > 0 && heads <= 256 && heads % 16 == 0);
}

// Partial slots a decode can need: one per sequence plus one per worker
// boundary that falls inside a sequence.
int max_slots(int batch, int heads, int sms) {
  const int w = qmla::simt_workers(sms) > qmla::tc_workers(sms, heads)
                    ? qmla::simt_workers(sms) : qmla::tc_workers(sms, heads);
  return batch + w;
}

int append_impl(int format, void* blocks, int64_t num_blocks, const int32_t* block_table,
                int32_t max_blocks_per_seq, int32_t* positions, int32_t batch, int32_t n_new,
                const void* latent, const void* rope_k, int32_t* status_dev, void* stream,
                bool advance, bool launch = true) {
  if (!known_format(format)) return QMLA_ERR_UNSUPPORTED;
  if (batch < 0 || n_new < 0 || max_blocks_per_seq < 0 || num_blocks < 1)
    return QMLA_ERR_INVALID_ARG;
  if (int64_t(batch) * n_new == 0) return QMLA_OK;
  if (int64_t(batch) * n_new > 0x7fffffffLL) return QMLA_ERR_CAPACITY;
  if (!blocks || !block_table || !positions || !latent || !rope_k || !status_dev)
    return QMLA_ERR_INVALID_ARG;
  if (!aligned(blocks, 256) || !aligned(latent, 4) || !aligned(rope_k, 4) ||
      !aligned(block_table, 4) || !aligned(positions, 4) || !aligned(status_dev, 4))
    return QMLA_ERR_INVALID_ARG;
  if (max_blocks_per_seq == 0) return QMLA_ERR_INVALID_ARG;
  if (!launch) return QMLA_OK;
  cudaError_t e = qmla::launch_append(
      format, static_cast<uint8_t*>(blocks), num_blocks, block_table, max_blocks_per_seq,
      positions, batch, n_new, static_cast<const __nv_bfloat16*>(latent),
      static_cast<const __nv_bfloat16*>(rope_k), status_dev, advance,
      static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QMLA_OK : QMLA_ERR_CUDA;
}
// The decode; q_len > 1: `heads` is q_len * q_heads virtual heads of a
// multi-token query step (qmla_decode_multi).
int decode_impl(int format, const void* blocks, int64_t num_blocks, const int32_t* block_table,
                int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t max_seq_len,
                int32_t batch, int32_t heads, int32_t q_len, int32_t q_heads, const void* q_c,
                const void* q_r, float softmax_scale, void* out, float* lse, void* workspace,
                size_t workspace_bytes, int32_t* status_dev, void* stream, int withhold = 0,
                bool launch = true) {
  if (!known_format(format)) return QMLA_ERR_UNSUPPORTED;
  if (batch < 0 || max_seq_len < 0 || max_blocks_per_seq < 0 || num_blocks < 1)
    return QMLA_ERR_INVALID_ARG;
  if (!heads_served(format, heads)) return QMLA_ERR_UNSUPPORTED;
  if (batch == 0) return QMLA_OK;
  if (!blocks || !block_table || !seq_lens || !q_c || !q_r || !out || !lse || !workspace ||
      !status_dev)
    return QMLA_ERR_INVALID_ARG;
  if (!aligned(blocks, 256) || !aligned(workspace, 256) || !aligned(q_c, 16) ||
      !aligned(q_r, 16) || !aligned(out, 16) || !aligned(lse, 4) || !aligned(seq_lens, 4) ||
      !aligned(block_table, 4) || !aligned(status_dev, 4))
    return QMLA_ERR_INVALID_ARG;
  if (max_blocks_per_seq == 0) return QMLA_ERR_INVALID_ARG;
  const int sms = device_sms();
  if (sms <= 0) return QMLA_ERR_CUDA;
  const int slots = max_slots(batch, heads, sms);
  if (workspace_bytes < qmla::workspace_bytes(batch, heads, slots)) return QMLA_ERR_WORKSPACE;
  if (!launch) return QMLA_OK;

  qmla::DecodeArgs a;
  a.fmt = format;
  a.blocks = static_cast<const uint8_t*>(blocks);
  a.num_blocks = num_blocks;
  a.block_table = block_table;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.seq_lens = seq_lens;
  a.max_seq_len = max_seq_len;
  a.batch = batch;
  a.heads = heads;
  a.q_c = static_cast<const __nv_bfloat16*>(q_c);
  a.q_r = static_cast<const __nv_bfloat16*>(q_r);
  a.scale = softmax_scale;
  a.ws = qmla::carve(workspace, batch, heads, slots);
  a.status = status_dev;
  a.q_len = q_len;
  a.q_heads = q_len > 1 ? q_heads : 0;
  a.withhold = withhold;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  // 16 query rows of a multi-token query step go to the CUDA-core kernel:
  // the 16-head tensor-core kernel has no causal mask (it would cost the
  // single-token decode its hot loop's room)
  if (qmla::tc_supported(format, heads) && !(q_len > 1 && heads == 16)) {
    a.workers = qmla::tc_workers(sms, heads);
    e = qmla::launch_decode_tc(a, s);
  } else {
    a.workers = qmla::simt_workers(sms);
    e = qmla::launch_decode_simt(a, s);
  }
  if (e != cudaSuccess) return QMLA_ERR_CUDA;
  e = qmla::launch_combine(a.ws, batch, heads, static_cast<__nv_bfloat16*>(out), lse, s);
  return e == cudaSuccess ? QMLA_OK : QMLA_ERR_CUDA;
}

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

// Offsets of qmla_decode_step's packed host buffers (qmla.h).
void step_layout(int32_t batch, int32_t heads, int32_t n_new, size_t* o) {
  const size_t B = size_t(batch), H = size_t(heads), n = size_t(n_new);
  size_t off = 0;
  o[0] = o[1] = 0;
  if (n_new > 0) {
    o[0] = off;
    off = up256(off + B * n * QMLA_D_C * 2);
    o[1] = off;
    off = up256(off + B * n * QMLA_D_R * 2);
  }
  o[2] = off;
  off = up256(off + B * H * QMLA_D_C * 2);
  o[3] = off;
  o[4] = off + B * H * QMLA_D_R * 2;
  o[5] = 0;
  o[6] = up256(B * H * QMLA_D_C * 2);
  o[7] = o[6] + B * H * 4;
}

}  // namespace

extern "C" {

size_t qmla_block_bytes(int format) {
  if (!known_format(format)) return 0;
  return size_t(qmla::geom(format).block);
}

const char* qmla_error_string(int code) {
  switch (code) {
    case QMLA_OK: return "ok";
    case QMLA_ERR_INVALID_ARG: return "invalid argument";
    case QMLA_ERR_UNSUPPORTED: return "unsupported format or shape";
    case QMLA_ERR_CAPACITY: return "request exceeds a fixed capacity";
    case QMLA_ERR_WORKSPACE: return "workspace too small";
    case QMLA_ERR_CUDA: return "CUDA runtime error";
    case QMLA_ERR_DEVICE: return "device status flag set";
    default: return "unknown error";
  }
}

int qmla_append(int format, void* blocks, int64_t num_blocks, const int32_t* block_table,
                int32_t max_blocks_per_seq, const int32_t* positions, int32_t batch, int32_t n_new,
                const void* latent, const void* rope_k, int32_t* status_dev, void* stream) {
  // positions are only read on this path
  return append_impl(format, blocks, num_blocks, block_table, max_blocks_per_seq,
                     const_cast<int32_t*>(positions), batch, n_new, latent, rope_k, status_dev,
                     stream, false);
}

int qmla_append_advance(int format, void* blocks, int64_t num_blocks,
                        const int32_t* block_table, int32_t max_blocks_per_seq,
                        int32_t* positions, int32_t batch, int32_t n_new, const void* latent,
                        const void* rope_k, int32_t* status_dev, void* stream) {
  return append_impl(format, blocks, num_blocks, block_table, max_blocks_per_seq, positions,
                     batch, n_new, latent, rope_k, status_dev, stream, true);
}

size_t qmla_decode_workspace_bytes(int format, int32_t batch, int32_t heads, int32_t max_seq_len) {
  if (!known_format(format) || batch < 0 || max_seq_len < 0 || !heads_served(format, heads))
    return 0;
  const int sms = device_sms();
  if (sms <= 0) return 0;
  return qmla::workspace_bytes(batch, heads, max_slots(batch, heads, sms));
}

int qmla_decode(int format, const void* blocks, int64_t num_blocks, const int32_t* block_table,
                int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t max_seq_len,
                int32_t batch, int32_t heads, const void* q_c, const void* q_r,
                float softmax_scale, void* out, float* lse, void* workspace,
                size_t workspace_bytes, int32_t* status_dev, void* stream) {
  return decode_impl(format, blocks, num_blocks, block_table, max_blocks_per_seq, seq_lens,
                     max_seq_len, batch, heads, 1, 0, q_c, q_r, softmax_scale, out, lse,
                     workspace, workspace_bytes, status_dev, stream);
}

int qmla_decode_multi(int format, const void* blocks, int64_t num_blocks,
                      const int32_t* block_table, int32_t max_blocks_per_seq,
                      const int32_t* seq_lens, int32_t max_seq_len, int32_t batch, int32_t heads,
                      int32_t q_len, const void* q_c, const void* q_r, float softmax_scale,
                      void* out, float* lse, void* workspace, size_t workspace_bytes,
                      int32_t* status_dev, void* stream) {
  if (q_len < 1 || heads < 1 || int64_t(heads) * q_len > 0x7fffffff) return QMLA_ERR_INVALID_ARG;
  return decode_impl(format, blocks, num_blocks, block_table, max_blocks_per_seq, seq_lens,
                     max_seq_len, batch, heads * q_len, q_len, heads, q_c, q_r, softmax_scale,
                     out, lse, workspace, workspace_bytes, status_dev, stream);
}

int qmla_decode_timeout_test(int format, const void* blocks, int64_t num_blocks,
                             const int32_t* block_table, int32_t max_blocks_per_seq,
                             const int32_t* seq_lens, int32_t max_seq_len, int32_t batch,
                             int32_t heads, const void* q_c, const void* q_r,
                             float softmax_scale, void* out, float* lse, void* workspace,
                             size_t workspace_bytes, int32_t* status_dev, void* stream) {
  // only the tensor-core kernels (low-bit formats) carry the hook
  if ((heads != 16 && heads != 128) || (format != QMLA_C4R4 && format != QMLA_C2R4))
    return QMLA_ERR_UNSUPPORTED;
  return decode_impl(format, blocks, num_blocks, block_table, max_blocks_per_seq, seq_lens,
                     max_seq_len, batch, heads, 1, 0, q_c, q_r, softmax_scale, out, lse,
                     workspace, workspace_bytes, status_dev, stream, 1);
}

int qmla_decode_step_layout(int32_t batch, int32_t heads, int32_t n_new, size_t* offsets) {
  if (!offsets || batch < 0 || heads < 0 || n_new < 0) return QMLA_ERR_INVALID_ARG;
  step_layout(batch, heads, n_new, offsets);
  return QMLA_OK;
}

size_t qmla_decode_step_workspace_bytes(int format, int32_t batch, int32_t heads, int32_t n_new,
                                        int32_t max_seq_len) {
  if (n_new < 0) return 0;
  const size_t dws = qmla_decode_workspace_bytes(format, batch, heads, max_seq_len);
  if (dws == 0) return 0;
  size_t o[8];
  step_layout(batch, heads, n_new, o);
  return up256(o[4]) + up256(o[7]) + dws;
}

int qmla_decode_step(int format, void* blocks, int64_t num_blocks, const int32_t* block_table,
                     int32_t max_blocks_per_seq, int32_t* seq_lens, int32_t max_seq_len,
                     int32_t batch, int32_t heads, int32_t n_new, const void* h_in,
                     float softmax_scale, void* h_out, void* workspace, size_t workspace_bytes,
                     int32_t* status_dev, void* stream) {
  if (batch < 0 || heads < 0 || n_new < 0) return QMLA_ERR_INVALID_ARG;
  if (!h_in || !h_out || !workspace) return QMLA_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return QMLA_ERR_INVALID_ARG;
  const size_t need = qmla_decode_step_workspace_bytes(format, batch, heads, n_new, max_seq_len);
  if (need == 0) {
    if (!known_format(format) || !heads_served(format, heads)) return QMLA_ERR_UNSUPPORTED;
    return max_seq_len < 0 ? QMLA_ERR_INVALID_ARG : QMLA_ERR_CUDA;
  }
  if (workspace_bytes < need) return QMLA_ERR_WORKSPACE;
  if (batch == 0) return QMLA_OK;
  size_t o[8];
  step_layout(batch, heads, n_new, o);
  uint8_t* d_in = static_cast<uint8_t*>(workspace);
  uint8_t* d_out = d_in + up256(o[4]);
  uint8_t* d_ws = d_out + up256(o[7]);
  const size_t dws = need - up256(o[4]) - up256(o[7]);
  // every argument checked before anything is enqueued
  int r = n_new > 0 ? append_impl(format, blocks, num_blocks, block_table, max_blocks_per_seq,
                                  seq_lens, batch, n_new, d_in + o[0], d_in + o[1], status_dev,
                                  stream, true, false)
                    : QMLA_OK;
  if (r != QMLA_OK) return r;
  r = decode_impl(format, blocks, num_blocks, block_table, max_blocks_per_seq, seq_lens,
                  max_seq_len, batch, heads, 1, 0, d_in + o[2], d_in + o[3], softmax_scale,
                  d_out + o[5], reinterpret_cast<float*>(d_out + o[6]), d_ws, dws, status_dev,
                  stream, 0, false);
  if (r != QMLA_OK) return r;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(d_in, h_in, o[4], cudaMemcpyHostToDevice, s) != cudaSuccess)
    return QMLA_ERR_CUDA;
  if (n_new > 0) {
    r = append_impl(format, blocks, num_blocks, block_table, max_blocks_per_seq, seq_lens, batch,
                    n_new, d_in + o[0], d_in + o[1], status_dev, stream, true);
    if (r != QMLA_OK) return r;
  }
  r = decode_impl(format, blocks, num_blocks, block_table, max_blocks_per_seq, seq_lens,
                  max_seq_len, batch, heads, 1, 0, d_in + o[2], d_in + o[3], softmax_scale,
                  d_out + o[5], reinterpret_cast<float*>(d_out + o[6]), d_ws, dws, status_dev,
                  stream);
  if (r != QMLA_OK) return r;
  if (cudaMemcpyAsync(h_out, d_out, o[7], cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return QMLA_ERR_CUDA;
  return cudaStreamSynchronize(s) == cudaSuccess ? QMLA_OK : QMLA_ERR_CUDA;
}

int qmla_read_status(const int32_t* status_dev, void* stream) {
  if (!status_dev) return QMLA_ERR_INVALID_ARG;
  int32_t v = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&v, status_dev, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return QMLA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return QMLA_ERR_CUDA;
  return v == 0 ? QMLA_OK : QMLA_ERR_DEVICE;
}

}  // extern "C"
