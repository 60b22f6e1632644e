// Prefill path (tcgen05 / TMEM / TMA). Placeholder until the kernel lands: never selected.
#include "internal.h"

namespace w4a16 {

bool prefill_supported(const GemmArgs &) { return false; }

void prefill_make_plan(int64_t, int64_t, int64_t, int, int, w4a16_plan_t *p) {
  p->path = W4A16_PATH_PREFILL;
}

cudaError_t launch_gemm_prefill(const GemmArgs &, const w4a16_plan_t &) {
  return cudaErrorNotSupported;
}

cudaError_t prefill_take_device_error(uint32_t *err) {
  *err = 0;
  return cudaSuccess;
}

cudaError_t prefill_set_wait_limit_ns(uint64_t) { return cudaSuccess; }

}  // namespace w4a16
