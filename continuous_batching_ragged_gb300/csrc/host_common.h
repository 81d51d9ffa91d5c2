// Host-side helpers shared by the library's translation units: the calling
// thread's last error message and status plumbing.
#pragma once

#include <cstdarg>
#include <cstdio>
#include <string>

#include "cb.h"

namespace cb {

// Records `msg` as the calling thread's last error and returns `status`.
cb_status fail(cb_status status, const char* fmt, ...);

}  // namespace cb
