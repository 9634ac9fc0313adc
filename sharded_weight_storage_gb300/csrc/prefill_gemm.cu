// tcgen05 / TMEM block-scaled FP8 prefill GEMM (m > 64).
#include "sws_internal.h"

namespace sws {

int launch_prefill(const PrefillLaunch& a, cudaStream_t s) {
  (void)a;
  (void)s;
  return fail(SWS_E_UNSUPPORTED, "prefill GEMM (m > 64) is not built yet");
}

}  // namespace sws
