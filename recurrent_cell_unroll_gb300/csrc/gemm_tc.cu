// placeholder: replaced by the tcgen05 GEMM
#include "tc.h"
namespace rcu {
bool tc_gemm_supported(int, int) { return false; }
cudaError_t launch_tc_gemm(const __nv_bfloat16 *, int, const __nv_bfloat16 *, int, const float *,
                           float *, int, int, const int32_t *, int, int, int, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace rcu
