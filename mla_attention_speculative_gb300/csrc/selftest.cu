// Failure-path self-test (mla_selftest_bounded_wait).
//
// One thread waits on a shared-memory barrier that nothing ever signals.  The
// wait is the same bounded wait every tcgen05 kernel of the library uses: it
// gives up after its limit (about a second), records its site in a status
// word and lets the kernel finish, so the context stays usable.  No fault,
// trap or endless loop is involved.

#include "mla_internal.h"
#include "sm103_ptx.cuh"

namespace mla {
using namespace sm103;

static __device__ int g_selftest_status;

namespace {
__global__ void __launch_bounds__(32) wait_selftest_sm103() {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    fence_mbar_init();
    if (!mbar_wait(b, 0)) atomicCAS(&g_selftest_status, 0, kSelftestSite);
  }
}
}  // namespace

cudaError_t launch_wait_selftest(cudaStream_t stream) {
  wait_selftest_sm103<<<1, 32, 0, stream>>>();
  return cudaGetLastError();
}

int selftest_device_status(bool clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_selftest_status, sizeof(int)) != cudaSuccess) return -1;
  if (clear && v != 0) {
    const int z = 0;
    if (cudaMemcpyToSymbol(g_selftest_status, &z, sizeof(int)) != cudaSuccess) return -1;
  }
  return v;
}

}  // namespace mla
