// msa_waittest.cu -- the bounded-wait exit, exercised on purpose.
//
// Every wait in the library's kernels is bounded: when a phase does not
// complete in time the kernel sets MSA_ERR_TIMEOUT, waits (again bounded) for
// the copies it has in flight, frees its tensor memory and returns, leaving
// the context usable.  This kernel takes that exit deliberately: it allocates
// tensor memory, starts a bulk copy into shared memory, then waits with a
// short limit on an mbarrier that nothing completes.
#include "msa_device.cuh"
#include "msa_launch.h"
#include "msa_tcgen05.cuh"

namespace msa {

namespace {

__device__ __align__(16) uint8_t g_wait_src[256];   // the bulk copy's source

__global__ void __launch_bounds__(64) wait_timeout_kernel(unsigned long long limit_ns,
                                                          unsigned* err) {
  __shared__ __align__(128) uint8_t buf[256];
  __shared__ uint64_t never, landed;
  __shared__ uint32_t tmem_slot;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(&never, 1);
    mbar_init(&landed, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&tmem_slot, 32);
    tc::tmem_relinquish();
  }
  tc::fence_before_thread_sync();
  __syncthreads();
  tc::fence_after_thread_sync();
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&landed, sizeof(buf));
    bulk_load(buf, g_wait_src, sizeof(buf), &landed);
    if (!mbar_wait_limit(&never, 0, limit_ns)) {
      flag_error(err, MSA_ERR_TIMEOUT);
      // the exit every kernel takes: the copies in flight land first
      (void)mbar_wait(&landed, 0);
    }
  }
  tc::fence_before_thread_sync();
  __syncthreads();
  tc::fence_after_thread_sync();
  if (warp == 1) tc::tmem_dealloc(tmem_slot, 32);
}

}  // namespace

cudaError_t launch_wait_timeout(unsigned long long limit_ns, unsigned* err, cudaStream_t stream) {
  return launch_pdl(wait_timeout_kernel, dim3(1), dim3(64), 0, stream, false, limit_ns, err);
}

}  // namespace msa
