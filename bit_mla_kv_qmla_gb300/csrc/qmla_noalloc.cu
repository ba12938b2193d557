// qmla_noalloc.cu - qmla_decode_noalloc: the decode with its scratch memory
// (split partials and merge table) taken from a fixed array that lives in
// the library's own device memory, so the call needs no workspace from the
// caller and allocates nothing.
//
// Some callers cannot allocate device memory where they call the decode: a
// serving loop that must not call cudaMalloc once it is running (cudaMalloc
// synchronizes the device and can fail under memory pressure), or a plugin
// whose host hands it a stream and expects it only to enqueue work.  They
// pass inputs and outputs as usual; the scratch below is shared by all calls.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds QMLA_NOALLOC_SCRATCH_BYTES of it until the process exits.
// Host code cannot use the variable's name as a device pointer, so the first
// call on each device looks its device address up with cudaGetSymbolAddress
// (that device current) and keeps it.  Nothing in the scratch must start at
// zero: the decode writes every merge-table entry and every partial it reads.

#include <mutex>

#include "qmla_internal.cuh"

namespace {

constexpr size_t kScratchBytes = QMLA_NOALLOC_SCRATCH_BYTES;
__device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (set up once).
int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return QMLA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return QMLA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return QMLA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return QMLA_OK;
}

bool is_aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" int qmla_decode_noalloc(int format, const void* blocks, int64_t num_blocks,
                                   const int32_t* block_table, int32_t max_blocks_per_seq,
                                   const int32_t* seq_lens, int32_t max_seq_len, int32_t batch,
                                   int32_t heads, const void* q_c, const void* q_r,
                                   float softmax_scale, void* out, float* lse,
                                   int32_t* status_dev, void* stream) {
  if (format != QMLA_C4R4 && format != QMLA_C2R4 && format != QMLA_BF16 &&
      format != QMLA_C4R2 && format != QMLA_C2R2)
    return QMLA_ERR_UNSUPPORTED;
  if (batch < 0 || max_seq_len < 0 || max_blocks_per_seq < 0 || num_blocks < 1)
    return QMLA_ERR_INVALID_ARG;
  const bool tc = qmla::tc_supported(format, heads);
  if (!tc && !(heads > 0 && heads <= 256 && heads % 16 == 0)) return QMLA_ERR_UNSUPPORTED;
  if (batch == 0) return QMLA_OK;
  if (!blocks || !block_table || !seq_lens || !q_c || !q_r || !out || !lse || !status_dev)
    return QMLA_ERR_INVALID_ARG;
  if (!is_aligned(blocks, 256) || !is_aligned(q_c, 16) || !is_aligned(q_r, 16) ||
      !is_aligned(out, 16) || !is_aligned(lse, 4) || !is_aligned(seq_lens, 4) ||
      !is_aligned(block_table, 4) || !is_aligned(status_dev, 4) || max_blocks_per_seq == 0)
    return QMLA_ERR_INVALID_ARG;

  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      sms <= 0)
    return QMLA_ERR_CUDA;
  // As many workers as the decode normally uses, or the largest count whose
  // partials still fit the scratch (the scratch need grows with the worker
  // count, so a binary search finds it); a batch whose merge table and one
  // partial per sequence do not fit is rejected.
  int workers = tc ? qmla::tc_workers(sms, heads) : qmla::simt_workers(sms);
  if (qmla::workspace_bytes(batch, heads, batch + 1) > kScratchBytes) return QMLA_ERR_CAPACITY;
  if (qmla::workspace_bytes(batch, heads, batch + workers) > kScratchBytes) {
    int lo = 1, hi = workers;  // fits at lo, not at hi
    while (hi - lo > 1) {
      const int mid = lo + (hi - lo) / 2;
      if (qmla::workspace_bytes(batch, heads, batch + mid) <= kScratchBytes)
        lo = mid;
      else
        hi = mid;
    }
    workers = lo;
  }

  void* scratch = nullptr;
  const int rc = scratch_for_current_device(&scratch);
  if (rc != QMLA_OK) return rc;

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
  a.ws = qmla::carve(scratch, batch, heads, batch + workers);
  a.workers = workers;
  a.status = status_dev;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = tc ? qmla::launch_decode_tc(a, s) : qmla::launch_decode_simt(a, s);
  if (e != cudaSuccess) return QMLA_ERR_CUDA;
  e = qmla::launch_combine(a.ws, batch, heads, static_cast<__nv_bfloat16*>(out), lse, s);
  return e == cudaSuccess ? QMLA_OK : QMLA_ERR_CUDA;
}
