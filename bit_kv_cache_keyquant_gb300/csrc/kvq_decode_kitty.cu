// placeholder until the kitty decode kernel lands
#include "kvq_internal.h"
namespace kvq {
cudaError_t launch_decode_kitty(const kvq_config *, const kvq_kitty_cache *, const void *, const DecodePlan &, void *,
                              cudaStream_t) {
    return cudaErrorNotSupported;
}
}  // namespace kvq
