// fa_status.h -- values kernels write into their device status word.
#pragma once

namespace fa {
constexpr int kStatusTimeout = 4;   // a bounded wait ran out (FA_ERR_TIMEOUT in include/fa.h)
constexpr int kStatusLayout = 7;    // shared-memory base not aligned as the kernel needs
}  // namespace fa
