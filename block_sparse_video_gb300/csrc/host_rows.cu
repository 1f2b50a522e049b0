// Row copies by SM loads and stores between pinned host memory and the device,
// for the host-buffer pipeline: the first head group's inputs are gathered and
// the last group's output scattered while nothing else runs on the device.
// SM accesses keep the host link busy with 16-byte requests from every SM and
// lose far less to short rows than a strided copy-engine copy does.
#include "host_rows.cuh"

namespace vsa {
namespace {

// blockIdx.y selects the tensor. Row r of tensor t: width bytes at
// src[t] + r * src_pitch go to dst[t] + r * dst_pitch. Widths, pitches and
// bases are multiples of 16 bytes (checked by the launcher).
__global__ void __launch_bounds__(512) copy_rows_kernel(HostRows a) {
  const int t = blockIdx.y;
  const uint8_t* __restrict__ src = a.src[t];
  uint8_t* __restrict__ dst = a.dst[t];
  const size_t per_row = a.width / 16;
  const size_t n = per_row * a.rows;
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const size_t r = i / per_row, c = i - r * per_row;
    const uint4 x = *reinterpret_cast<const uint4*>(src + r * a.src_pitch + c * 16);
    *reinterpret_cast<uint4*>(dst + r * a.dst_pitch + c * 16) = x;
  }
}

}  // namespace

cudaError_t launch_copy_host_rows(const HostRows& a, int num_sms, cudaStream_t stream) {
  if (a.tensors < 1 || a.tensors > 4 || a.width == 0 || a.width % 16 || a.src_pitch % 16 || a.dst_pitch % 16 ||
      a.src_pitch < a.width || a.dst_pitch < a.width)
    return cudaErrorInvalidValue;
  for (int t = 0; t < a.tensors; ++t)
    if (!a.src[t] || !a.dst[t] || reinterpret_cast<uintptr_t>(a.src[t]) % 16 || reinterpret_cast<uintptr_t>(a.dst[t]) % 16)
      return cudaErrorInvalidValue;
  if (a.rows == 0) return cudaSuccess;
  // A few CTAs per SM keep enough 16-byte requests in flight to fill the link.
  const dim3 grid(static_cast<unsigned>(2 * num_sms), static_cast<unsigned>(a.tensors));
  copy_rows_kernel<<<grid, 512, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace vsa
