// tl_unbound_error.h -- the message of the last failure that has no handle to
// keep it (a refused create, a refused or failed allocation-free forward),
// per host thread; tiled_linear_last_error(NULL) returns it.
#pragma once
#include <string>

namespace tl {
void set_unbound_error(const std::string& why);
const char* unbound_error();
}  // namespace tl
