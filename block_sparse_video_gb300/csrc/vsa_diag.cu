// Diagnostics: exercise the bounded-wait failure path of the kernels without
// faulting the GPU. Every CTA waits on an mbarrier that nothing ever arrives
// on; the first wait to reach the time limit records VSA_ERR_DEVICE_TIMEOUT in
// the error words and raises the abort flag, and the remaining CTAs see the
// flag and return at once.
#include "kernels.cuh"
#include "ptx.cuh"
#include "vsa.h"

namespace {

__global__ void never_arrives_kernel(unsigned int* err) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = vsa::smem_u32(&bar);
  if (threadIdx.x == 0) {
    vsa::mbar_init(b, 1);
    vsa::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) vsa::mbar_wait(b, 0, err, 0xD1A6u + blockIdx.x);
  __syncthreads();
}

}  // namespace

extern "C" vsa_status_t vsa_diag_wait_timeout(vsa_plan_t plan, void* workspace, int n_ctas,
                                              void* stream) {
  if (!plan || !workspace || n_ctas < 1 || n_ctas > 65535) return VSA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned int* err = static_cast<unsigned int*>(workspace);  // error words sit at offset 0
  if (cudaMemsetAsync(err, 0, 16, st) != cudaSuccess) return VSA_ERR_CUDA;
  never_arrives_kernel<<<n_ctas, 32, 0, st>>>(err);
  return cudaGetLastError() == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
}
