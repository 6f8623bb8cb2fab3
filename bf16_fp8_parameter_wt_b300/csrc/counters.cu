// The consumer side of the completion counters: a bounded device-side wait
// until every listed rank's counter has reached its target (the receiver of
// a one-sided transfer engine counts immediates until it has seen as many
// as it expects, "RDMA point-to-point communication for LLM systems",
// ImmCounter). Counters are compared modulo 2^32, so they may wrap.
#include <string>

#include "plan.h"

namespace wt {
namespace {

constexpr int kMaxWaitRanks = 1000;

struct WaitArgs {
  const uint32_t* counters;
  int32_t* status;
  uint64_t limit_ns;
  int32_t n;
  uint32_t targets[kMaxWaitRanks];
};

__device__ __forceinline__ uint32_t ld_acquire_gpu_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__global__ void __launch_bounds__(256) wait_counters_kernel(const __grid_constant__ WaitArgs a) {
  int ok = 1;
  const uint64_t t0 = now_ns();
  for (int i = threadIdx.x; i < a.n && ok; i += blockDim.x) {
    while ((int32_t)(ld_acquire_gpu_u32(a.counters + i) - a.targets[i]) < 0) {
      if (now_ns() - t0 > a.limit_ns) {
        ok = 0;
        break;
      }
      __nanosleep(256);
    }
  }
  ok = __syncthreads_and(ok);
  if (threadIdx.x == 0) *a.status = ok ? 0 : (int32_t)WT_ERR_TIMEOUT;
}

__global__ void __launch_bounds__(256) add_counts_kernel(uint32_t* counters, const uint32_t* counts, int32_t n,
                                                        const int32_t* error_word) {
  // launched as a programmatic dependent: let the next launch begin, then
  // wait until the preparation before this kernel has completed and its
  // stores are visible (returns at once after an ordinary launch)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // a launch whose waits gave up stored only part of its blocks: count none
  if (error_word && (*reinterpret_cast<const volatile int32_t*>(error_word) & kErrTimeout)) return;
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const uint32_t c = counts[i];
    if (c) asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(counters + i), "r"(c) : "memory");
  }
}

}  // namespace

cudaError_t launch_add_counts(uint32_t* counters, const uint32_t* counts, int32_t n, const int32_t* error_word,
                              cudaStream_t s, bool pdl) {
  if (n <= 0) return cudaSuccess;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, add_counts_kernel, counters, counts, n, error_word);
}

}  // namespace wt

using namespace wt;

extern "C" wt_status wt_wait_counters(const uint32_t* counters, int32_t n, const uint32_t* targets,
                                      uint64_t limit_ns, int32_t* status, void* stream) {
  if (n < 0 || n > kMaxWaitRanks) {
    set_error("wt_wait_counters: n must be in [0, " + std::to_string(kMaxWaitRanks) + "]");
    return WT_ERR_INVALID_ARGUMENT;
  }
  if (!status || (n > 0 && (!counters || !targets))) {
    set_error("wt_wait_counters: NULL counters, targets or status");
    return WT_ERR_INVALID_ARGUMENT;
  }
  if (reinterpret_cast<uintptr_t>(counters) % 4 || reinterpret_cast<uintptr_t>(status) % 4) {
    set_error("wt_wait_counters: counters and status must be 4-byte aligned");
    return WT_ERR_ALIGNMENT;
  }
  WaitArgs a;
  a.counters = counters;
  a.status = status;
  a.limit_ns = limit_ns;
  a.n = n;
  for (int32_t i = 0; i < n; ++i) a.targets[i] = targets[i];
  wait_counters_kernel<<<1, 256, 0, static_cast<cudaStream_t>(stream)>>>(a);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error(std::string("wt_wait_counters: launch: ") + cudaGetErrorString(e));
    return WT_ERR_CUDA;
  }
  return WT_OK;
}
