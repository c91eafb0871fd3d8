// selftest.cu -- exercises the failure path of the kernels' bounded barrier waits on
// the GPU without faulting it: one thread waits on an mbarrier that nothing arrives on,
// through the wait routine the tcgen05 kernels use (bounded by its poll cap, and left
// as soon as the CTA's abort flag is up), while another warp raises that flag after a
// given number of clock cycles.  The wait gives up, the kernel records
// PISA_ERR_DEVICE_TIMEOUT in the status word and returns; the context stays usable.
#include "api.cuh"
#include "tc.cuh"

namespace pisa {

__global__ void __launch_bounds__(64) selftest_wait_kernel(int* status, long long delay_cycles) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  volatile int* abort = &abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // one arrival completes a phase; none ever comes
    abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!mbar_wait(&bar, 0, abort)) set_status(status, PISA_ERR_DEVICE_TIMEOUT);
  } else if (threadIdx.x == 32) {
    const long long t0 = clock64();
    while (clock64() - t0 < delay_cycles) {
    }
    *abort = 1;
  }
}

cudaError_t launch_selftest_wait(int* status, long long delay_cycles, cudaStream_t s) {
  selftest_wait_kernel<<<1, 64, 0, s>>>(status, delay_cycles);
  note_launch();
  return cudaGetLastError();
}

}  // namespace pisa
