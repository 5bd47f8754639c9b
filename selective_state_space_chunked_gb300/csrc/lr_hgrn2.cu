// lr_hgrn2.cu -- HGRN2 chunked matrix-state recurrence (tcgen05 / TMEM / TMA).
// Placeholder until the kernel lands: every call reports LR_ERR_UNSUPPORTED.
#include "lr_internal.h"

namespace lr {

int hgrn2_workspace(int64_t, int64_t, int64_t, size_t *bytes) {
    *bytes = 0;
    return LR_OK;
}

int hgrn2_launch(const void *, const void *, const void *, const void *, const float *, void *,
                 float *, int64_t, int64_t, int64_t, void *, cudaStream_t) {
    return LR_ERR_UNSUPPORTED;
}

int hgrn2_status_read_and_clear(int *status) {
    *status = 0;
    return LR_OK;
}

}  // namespace lr
