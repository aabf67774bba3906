// prefill.cu -- dense prefill (t >= 256) on the tensor cores.
#include "../../include/tq1.h"
#include "tq1_internal.h"

namespace tq1 {

int launch_prefill(const uint8_t*, const uint8_t*, float*, int64_t, int64_t, int64_t, void*, size_t, cudaStream_t,
                   unsigned*) {
  return TQ1_ERR_UNSUPPORTED;
}

}  // namespace tq1
