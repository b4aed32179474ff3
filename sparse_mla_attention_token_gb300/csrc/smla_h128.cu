// tcgen05 kernel for H = 128 (not yet enabled: the planner routes H = 128 to
// the small-head kernel until this kernel passes parity).
#include <cuda_runtime.h>

#include "smla_internal.h"

namespace smla {

bool h128_supported(int64_t, int32_t, int32_t) { return false; }

int launch_h128(const FwdParams&, void*) { return static_cast<int>(cudaErrorNotSupported); }

int h128_error_word(unsigned int** addr) {
  *addr = nullptr;
  return 0;
}

}  // namespace smla
