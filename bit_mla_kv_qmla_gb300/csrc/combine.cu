// combine.cu - log-sum-exp merge of the split-KV partials.
//
// Each piece i of a sequence holds a normalized partial O_i and its LSE_i;
// the full result is LSE = ln sum_i exp(LSE_i) and
// O = sum_i exp(LSE_i - LSE) * O_i, written as bfloat16 O and binary32 LSE
// (computed as sum_i w_i O_i / sum_i w_i with w_i = exp(LSE_i - max_j LSE_j),
// the maximum kept running over the pieces).
// A sequence with no piece (length 0) gets O = 0 and LSE = -inf.
// Grid (batch, heads), 128 threads, 4 channels per thread.

#include <cfloat>

#include "qmla_internal.cuh"

namespace qmla {
namespace {

__global__ void __launch_bounds__(128) combine_kernel(Workspace ws, int heads,
                                                      __nv_bfloat16* __restrict__ out,
                                                      float* __restrict__ lse) {
  const int b = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  // launched as a programmatic dependent of the decode: wait until the
  // decode grid has completed and its partials are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int2 ent = ws.seq_table[b];
  const int base = ent.x, n = ent.y;
  const float* plse = ws.part_lse + int64_t(base) * heads + h;
  const float4* po = reinterpret_cast<const float4*>(ws.part_o + (int64_t(base) * heads + h) * kDc) + tid;
  const int64_t ostride = int64_t(heads) * kDc / 4;  // float4s from one piece to the next
  // one pass with a running maximum, eight pieces at a time: the LSEs and
  // partial outputs of up to eight pieces are loaded before any is used, so a
  // sequence with at most eight pieces costs one round of loads
  constexpr int kU = 8;
  float m = -INFINITY, sum = 0.0f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i0 = 0; i0 < n; i0 += kU) {
    float l[kU];
    float4 o[kU];
#pragma unroll
    for (int k = 0; k < kU; ++k) {
      const bool in = i0 + k < n;
      l[k] = in ? plse[int64_t(i0 + k) * heads] : -INFINITY;
      o[k] = in ? po[int64_t(i0 + k) * ostride] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float mc = m;
#pragma unroll
    for (int k = 0; k < kU; ++k) mc = fmaxf(mc, l[k]);
    if (mc > -INFINITY) {
      const float sc = __expf(m - mc);  // 0 while m is still -inf
      sum *= sc;
      acc.x *= sc;
      acc.y *= sc;
      acc.z *= sc;
      acc.w *= sc;
#pragma unroll
      for (int k = 0; k < kU; ++k) {
        const float wgt = __expf(l[k] - mc);  // 0 for empty pieces and padding
        sum += wgt;
        acc.x = fmaf(wgt, o[k].x, acc.x);
        acc.y = fmaf(wgt, o[k].y, acc.y);
        acc.z = fmaf(wgt, o[k].z, acc.z);
        acc.w = fmaf(wgt, o[k].w, acc.w);
      }
      m = mc;
    }
  }
  float L = -INFINITY;
  if (m > -INFINITY) {
    const float inv = 1.0f / sum;
    acc.x *= inv;
    acc.y *= inv;
    acc.z *= inv;
    acc.w *= inv;
    L = m + logf(sum);
  }
  __nv_bfloat162* dst = reinterpret_cast<__nv_bfloat162*>(out + (int64_t(b) * heads + h) * kDc) + 2 * tid;
  dst[0] = __floats2bfloat162_rn(acc.x, acc.y);
  dst[1] = __floats2bfloat162_rn(acc.z, acc.w);
  if (tid == 0) lse[int64_t(b) * heads + h] = L;
}

}  // namespace

cudaError_t launch_combine(const Workspace& ws, int batch, int heads, __nv_bfloat16* out,
                           float* lse, cudaStream_t stream) {
  if (batch == 0) return cudaSuccess;
  // Programmatic dependent launch: the combine's CTAs may be scheduled while
  // the decode's last CTAs finish (the decode signals early), which hides
  // the launch latency between the two kernels.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(batch), unsigned(heads));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel, ws, heads, out, lse);
}

}  // namespace qmla
