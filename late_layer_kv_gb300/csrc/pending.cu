// pending.cu -- entry points whose kernels are not built yet.
#include "abi_common.h"

using namespace rf;

extern "C" size_t ridgefill_fit_workspace_size(const rf_fit_args*) { return 0; }
extern "C" rf_status ridgefill_fit(const rf_fit_args*, void*, size_t, void*) {
  return fail(RF_ERR_SHAPE, "ridgefill_fit is not available in this build");
}
