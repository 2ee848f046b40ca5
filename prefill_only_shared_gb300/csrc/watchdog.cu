// Bounded device wait on a flag: the time limit and error path that every
// pipeline wait in libsp's kernels uses, exposed so that failure reporting
// can be exercised without a fault (a flag that nothing sets runs out).
#include "common.cuh"
#include "launch.h"

namespace sp {
namespace {

__global__ void wait_flag_kernel(const volatile unsigned* flag, unsigned expect,
                                 unsigned long long limit_ns, unsigned* err) {
  const unsigned long long t0 = globaltimer();
  while (*flag != expect) {
    if (globaltimer() - t0 > limit_ns) {
      raise_error(err, kErrTimeout);
      return;
    }
    __nanosleep(1000);
  }
}

}  // namespace

cudaError_t wait_flag_run(const unsigned* flag, unsigned expect, unsigned long long limit_ns,
                          unsigned* err, void* stream) {
  if (limit_ns < 1000ull) limit_ns = 1000ull;
  if (limit_ns > kWaitLimitNs) limit_ns = kWaitLimitNs;
  wait_flag_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(flag, expect, limit_ns, err);
  return cudaGetLastError();
}

}  // namespace sp
