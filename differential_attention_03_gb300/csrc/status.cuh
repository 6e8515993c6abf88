// Status codes shared by kernels and host code (values match diffattn.h).
#pragma once

#include <cstdint>

namespace da {

constexpr int kStatusOk = 0;
constexpr int kStatusTimeout = 7;  // DIFFATTN_ERR_TIMEOUT

// Budget of one in-kernel wait.  Every legitimate wait in these kernels lasts
// microseconds; one second leaves room for time-slicing with other contexts
// while still ending a wait on a phase that will never complete.
constexpr uint64_t kWaitBudgetNs = 1000000000ull;

}  // namespace da
