// api_internal.cuh -- error reporting shared by the C-ABI translation units.
#pragma once
#include "../../include/sf_gdn.h"

namespace sfg {
// Records a printf-style message as the calling thread's sf_last_error() and returns s.
sf_status report(sf_status s, const char* fmt, ...);
}  // namespace sfg
