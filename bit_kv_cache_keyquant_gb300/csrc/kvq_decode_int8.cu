// placeholder until the int8 decode kernel lands
#include "kvq_internal.h"
namespace kvq {
cudaError_t launch_decode_int8(const kvq_config *, const kvq_int8_cache *, const void *, const DecodePlan &, void *,
                              cudaStream_t) {
    return cudaErrorNotSupported;
}
}  // namespace kvq
