// Library-wide host state: the per-thread error message and the count of
// kernel launches.
#include "sv_common.cuh"

namespace sv {
std::string &last_error() {
  thread_local std::string msg;
  return msg;
}
std::atomic<unsigned long long> &launch_counter() {
  static std::atomic<unsigned long long> n{0};
  return n;
}
}  // namespace sv

extern "C" const char *sv_last_error_string(void) { return sv::last_error().c_str(); }

extern "C" unsigned long long sv_kernel_launches(void) { return sv::launch_counter().load(); }
