// Weight gradient on the tensor cores (NHWC bf16): planned, not yet enabled.
#include "problem.h"

namespace gbconv {

bool wgrad_tc_supported(const Problem&) { return false; }
int64_t wgrad_tc_workspace(const Problem&) { return 0; }
gbconv_status launch_wgrad_tc(const Problem&, const void*, const void*, void*, float*, void*, const Launch&) {
  return GBCONV_EUNSUPPORTED;
}
bool wgrad_tc_describe(const Problem&, char*, size_t) { return false; }

}  // namespace gbconv
