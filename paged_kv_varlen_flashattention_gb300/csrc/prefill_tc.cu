// Tensor-core (tcgen05) prefill kernel -- not yet enabled: every sequence runs on the
// split-KV kernel until this path is in place.
#include <cstdio>

#include "pa_internal.h"

namespace pa {
bool prefill_supported(const Args&) { return false; }
int prefill_rows_threshold() { return 32; }
int launch_prefill(const Args&, unsigned int*, char* msg, size_t msg_len) {
    snprintf(msg, msg_len, "tensor-core prefill kernel not built");
    return PA_ERR_UNSUPPORTED;
}
}  // namespace pa
