// Row copies between pinned host memory and device memory by SM loads and
// stores over the host link, for the host-buffer pipeline's first and last
// head groups (nothing else runs on the device then). Declared apart from the
// attention kernels.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace vsa {

// Up to four tensors in one launch. Row r of tensor t: width bytes at
// src[t] + r * src_pitch go to dst[t] + r * dst_pitch. Addresses are
// device-side (for host memory: its device view); width, pitches and bases
// are multiples of 16 bytes.
struct HostRows {
  const uint8_t* src[4];
  uint8_t* dst[4];
  size_t src_pitch = 0;
  size_t dst_pitch = 0;
  size_t width = 0;
  size_t rows = 0;
  int tensors = 0;
};
cudaError_t launch_copy_host_rows(const HostRows& a, int num_sms, cudaStream_t stream);

}  // namespace vsa
