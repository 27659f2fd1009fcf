#include "smla_internal.h"
namespace smla {
smla_status_t launch_sparse_prefill(const void*, int, const uint8_t*, int64_t, const float*, int, const uint32_t*, int,
                                    const uint32_t*, int, int, float, uint16_t*, unsigned*, cudaStream_t) {
  return fail(SMLA_ERR_UNSUPPORTED, "sparse prefill not built yet");
}
}
