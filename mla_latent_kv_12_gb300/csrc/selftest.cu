// Failure-detection self-test: one CTA waits on an mbarrier that nothing will
// ever complete, through the same bounded wait (mbar_wait) every kernel of the
// library uses, with a caller-chosen limit.  The wait gives up, the kernel
// records MLA_DEVICE_TIMEOUT in the status word and returns normally, so the
// context stays usable -- the behaviour every kernel relies on when a peer,
// a copy or an MMA never signals.  No fault, trap or endless loop is involved.
#include "mla_internal.h"
#include "tc_common.cuh"

namespace mla {
namespace {

__global__ void bounded_wait_kernel(long long limit_cycles, int32_t* status, long long* waited) {
  __shared__ __align__(8) uint64_t never;   // initialised for one arrival that never comes
  if (threadIdx.x == 0) {
    tc::mbar_init(&never, 1);
    tc::fence_mbar_init();
  }
  __syncthreads();
  const long long t0 = clock64();
  const bool ok = tc::mbar_wait_warp(&never, 0, limit_cycles);
  const long long t1 = clock64();
  if (threadIdx.x == 0) {
    if (!ok && status) atomicOr(status, MLA_DEVICE_TIMEOUT);
    if (waited) *waited = t1 - t0;
  }
}

}  // namespace

cudaError_t launch_bounded_wait(long long limit_cycles, int32_t* status, long long* waited, cudaStream_t stream) {
  bounded_wait_kernel<<<1, 32, 0, stream>>>(limit_cycles, status, waited);
  return cudaGetLastError();
}

}  // namespace mla
