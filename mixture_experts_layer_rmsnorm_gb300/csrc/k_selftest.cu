// k_selftest.cu -- a self-test of the error path of the bounded device waits.
//
// One CTA of two warps: warp 0 waits on an mbarrier phase that nothing
// completes (the wait of the expert GEMMs' rings), warp 1 on a flag that
// nothing sets (the wait of their stream-K partial sums).  Both give up after
// timeout_ns; a wait that gives up records MOE_ERR_TIMEOUT and this kernel's
// id in the workspace error word, and the kernel returns normally, so the
// CUDA context stays usable.  Nothing faults, traps or hangs.
#include "bounded_wait.cuh"
#include "moe_kernels.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(64) selftest_wait_kernel(int32_t* err, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int32_t* flag = err + 8;  // a word of the error area that no kernel sets
  if (threadIdx.x == 0) {
    err[0] = 0;
    err[1] = 0;
    *flag = 0;
    ptx::mbar_init(&bar, 1);
    abort_flag = 0;
    ptx::fence_barrier_init();
  }
  __syncthreads();
  const int never = 0;  // each wait runs its full time: no early abort
  bool ok;
  if (warp == 0)
    ok = __all_sync(0xFFFFFFFFu, ptx::mbar_wait(&bar, 0, timeout_ns, &never));
  else
    ok = wait_flag(flag, &never, timeout_ns);
  if (!ok && lane == 0) raise_timeout(err, &abort_flag, kKernSelfTest);
}

}  // namespace

cudaError_t launch_selftest_wait(int32_t* err, uint64_t timeout_ns, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 64, 0, stream>>>(err, timeout_ns);
  return cudaGetLastError();
}

}  // namespace moe
