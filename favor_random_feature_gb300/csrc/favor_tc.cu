// favor_tc.cu -- tensor-core (tcgen05) path; filled in below.
#include "favor_internal.h"

namespace favor {
bool tc_supported(const Problem &) { return false; }
int tc_forward(const void *, const void *, const void *, const float *, float *, const Problem &,
               cudaStream_t) {
    return FAVOR_ERR_UNSUPPORTED;
}
}  // namespace favor
