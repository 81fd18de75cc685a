// Library-wide host state: the per-thread error message, the count of
// kernel launches, and the test hooks of the bounded waits.
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
namespace {
std::atomic<unsigned long long> g_wait_ns{0};
std::atomic<unsigned> g_withhold{0};
}  // namespace
uint64_t wait_limit_ns() {
  const unsigned long long v = g_wait_ns.load(std::memory_order_relaxed);
  return v ? v : kWaitLimitNs;
}
unsigned test_withhold() { return g_withhold.load(std::memory_order_relaxed); }
}  // namespace sv

extern "C" void sv_test_hooks(unsigned long long wait_limit_ns, unsigned withhold) {
  sv::g_wait_ns.store(wait_limit_ns, std::memory_order_relaxed);
  sv::g_withhold.store(withhold, std::memory_order_relaxed);
}

extern "C" const char *sv_last_error_string(void) { return sv::last_error().c_str(); }

extern "C" unsigned long long sv_kernel_launches(void) { return sv::launch_counter().load(); }
