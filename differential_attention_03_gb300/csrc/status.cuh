// Status codes shared by kernels and host code (values match diffattn.h).
#pragma once

#include <cstdint>

namespace da {

constexpr int kStatusOk = 0;
constexpr int kStatusTimeout = 7;  // DIFFATTN_ERR_TIMEOUT
constexpr int kStatusSmemAlign = 9;  // a kernel found its shared memory misaligned (read as DIFFATTN_ERR_CUDA)

// Budget of one in-kernel wait, in SM clock cycles (about one second at the
// 2.07 GHz maximum clock, two at 1 GHz).  Every legitimate wait in these
// kernels lasts microseconds; this leaves room for time-slicing with other
// contexts while still ending a wait on a phase that will never complete.
constexpr uint64_t kWaitBudgetCycles = 2000000000ull;

}  // namespace da
