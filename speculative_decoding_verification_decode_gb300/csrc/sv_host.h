// Host helpers shared by the library's translation units (not part of the ABI).
#pragma once
#include "../../include/sv.h"

namespace svh {

// Records a printf-style message for sv_last_error() and returns `s`.
sv_status fail(sv_status s, const char* fmt, ...);
// Clears the message at the start of an entry point.
void clear_error();

}  // namespace svh
