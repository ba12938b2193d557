// decode_tc.cu - tensor-core (tcgen05) decode kernels.  Placeholder until the
// kernels land: no head count is served here yet.
#include "qmla_internal.cuh"

namespace qmla {
int tc_workers(int sms, int heads) { (void)heads; return sms / 2; }
bool tc_supported(int fmt, int heads) { (void)fmt; (void)heads; return false; }
cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t stream) {
  (void)a; (void)stream;
  return cudaErrorNotSupported;
}
}  // namespace qmla
