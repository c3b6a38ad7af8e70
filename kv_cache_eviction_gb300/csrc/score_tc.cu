// tcgen05 (5th-generation tensor core) path of the window scoring and of the
// CriticalKV V*W_O row norm.  Placeholder until the kernels land: reports
// "not supported" so the CUDA-core path runs.
#include "kv_internal.cuh"

namespace kv {

bool score_tc_supported(const Shape&) { return false; }
size_t score_tc_ws(const Shape&, int) { return 0; }
cudaError_t launch_score_tc(const Shape&, int, int, const void*, const void*, const void*, float*,
                            char*, cudaStream_t) {
  return cudaErrorNotSupported;
}
bool crit_tc_supported(const Shape&, int) { return false; }
cudaError_t launch_crit_tc(const Shape&, const void*, const void*, int, float*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace kv
