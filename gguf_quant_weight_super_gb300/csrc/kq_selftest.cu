// kq_selftest.cu -- the library's bounded waits, made to run out on purpose.
//
// Every wait in the kernels is bounded: an mbarrier wait (a copy that never
// lands) and a grid-barrier wait (a CTA that never arrives) give up after a
// poll limit, set the device error word and let the kernel return, so the
// context stays usable.  This self-test exercises exactly those two functions
// (mbar_wait, grid_wait of kq_ptx.cuh) on a flag that nothing ever sets, with
// a short limit (a few milliseconds), and reports the error code it observed.
#include "kq_internal.h"

namespace kq {
namespace {

__device__ int g_selftest_error = 0;
__device__ int g_selftest_counter = 0;

__global__ void selftest_wait_kernel(int kind, uint32_t max_polls) {
  __shared__ __align__(8) uint64_t bar;
  if (kind == 0) {
    if (threadIdx.x == 0) {
      mbar_init(&bar, 1);  // one arrival expected; none ever comes
      fence_mbar_init();
    }
    __syncthreads();
    mbar_wait(&bar, 0, &g_selftest_error, max_polls);
  } else if (threadIdx.x == 0) {
    grid_wait(&g_selftest_counter, 1, &g_selftest_error, max_polls);  // no CTA arrives
  }
}

}  // namespace

cudaError_t run_selftest_wait(int kind, int* observed, cudaStream_t st) {
  const int zero = 0;
  cudaError_t e = cudaMemcpyToSymbolAsync(g_selftest_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess)
    e = cudaMemcpyToSymbolAsync(g_selftest_counter, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return e;
  selftest_wait_kernel<<<1, 32, 0, st>>>(kind, 1u << 12);
  e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaMemcpyFromSymbolAsync(observed, g_selftest_error, sizeof(int), 0,
                                                      cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  return e;
}

}  // namespace kq
