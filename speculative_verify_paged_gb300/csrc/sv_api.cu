// Library-wide host state: the per-thread error message.
#include "sv_common.cuh"

namespace sv {
std::string &last_error() {
  thread_local std::string msg;
  return msg;
}
}  // namespace sv

extern "C" const char *sv_last_error_string(void) { return sv::last_error().c_str(); }
