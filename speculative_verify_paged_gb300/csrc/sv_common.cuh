// Shared host/device helpers of libspecverify: error reporting, dtype loads,
// and thin inline-PTX wrappers for the sm_100-family asynchronous machinery
// (mbarrier, bulk copies, tensor-map copies, cluster shared memory).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <cstdarg>
#include <cstdio>
#include <string>
#include <atomic>
#include <utility>

#include "../../include/specverify.h"

namespace sv {

// ----------------------------------------------------------------- host ---

// Top-p filter (topp.cu): rows0 rows in0 -> out0, then rows1 rows in1 -> out1,
// each [rows][V] of `dtype`; arguments already checked by the caller.
sv_status launch_topp_filter(sv_dtype dtype, const void *in0, void *out0, int rows0, const void *in1, void *out1,
                             int rows1, int V, float temperature, float top_p, int32_t *status, cudaStream_t s);

// Wait limit for device waits of later launches (sv_test_hooks; default
// kWaitLimitNs) and the signals a test asks launches to withhold.
uint64_t wait_limit_ns();
unsigned test_withhold();

// Per-thread message of the last failed call.
std::string &last_error();
// kernels this library launched successfully in this process
std::atomic<unsigned long long> &launch_counter();

inline sv_status fail(sv_status st, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  last_error() = buf;
  return st;
}

inline sv_status ok() {
  last_error().clear();
  return SV_OK;
}

inline sv_status check_launch(const char *what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(SV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return ok();
}

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline int dtype_bytes(sv_dtype t) {
  switch (t) {
    case SV_F32: return 4;
    case SV_BF16: return 2;
    case SV_F16: return 2;
    case SV_FP8_E4M3: return 1;
  }
  return 0;
}

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// --------------------------------------------------------------- device ---

template <int DT> struct Elem;
template <> struct Elem<SV_F32> { using T = float; };
template <> struct Elem<SV_BF16> { using T = __nv_bfloat16; };
template <> struct Elem<SV_F16> { using T = __half; };

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }

__device__ __forceinline__ void atomic_or_status(int32_t *st, int32_t bits) {
  if (st) atomicOr(st, bits);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Every spin-wait on an mbarrier gives up after this many nanoseconds of
// wall time (read from %globaltimer); callers then report SV_DEV_TIMEOUT and
// stop waiting for the rest of the launch.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbarrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t phase) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(phase)
      : "memory");
  return done != 0;
}

// try_wait that lets the hardware suspend the thread (up to ~65 us) until
// the phase completes, instead of spinning.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t phase) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(phase), "r"(0x10000u)
      : "memory");
  return done != 0;
}

// Bounded wait: returns false (and the caller reports SV_DEV_TIMEOUT) if the
// phase did not complete within limit_ns.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t phase, uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, phase)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, phase)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

// 1-D bulk copy global -> this CTA's shared memory, completion on `bar`.
// dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ------------------------------------------------------ cluster helpers ---

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// Address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa(const void *p, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_u32(p)), "r"(rank));
  return out;
}

__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ int ld_dsmem_s32(uint32_t addr) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// --------------------------------------------- programmatic launches ---
// pdl_wait(): the grids before this one in the stream have completed and
// their memory is visible. pdl_trigger(): the next launch of the stream may
// be scheduled while this grid drains. Kernels call both first, except where
// a kernel reads only inputs no kernel of the library writes (lengths, block
// table, new K/V rows, logits): those loads may come before the wait, and
// every write still comes after it. Data that the previous kernel writes
// (a work order, a partition, ancestor masks, accepted counts) is read after
// the wait with plain loads, never __ldg: that kernel may still have been
// writing it when this grid started, so it is not read-only data for this
// grid, and a read-only load may be scheduled as if it were.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch with programmatic stream serialization (and a cluster shape when
// cluster > 1).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                            int cluster, Args &&...args) {
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = (unsigned)n;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  if (e == cudaSuccess) launch_counter().fetch_add(1, std::memory_order_relaxed);
  return e;
}

// ----------------------------------------------------- warp reductions ---

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace sv
