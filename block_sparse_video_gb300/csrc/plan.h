// The host-side plan behind the opaque vsa_plan_t handle of include/vsa.h.
#pragma once
#include <cstddef>
#include <vector>
#include <cuda_runtime.h>

#include "kernels.cuh"
#include "vsa.h"

// Head-group pipeline of the host-buffer path: group g's inputs are copied in
// while group g - 1 computes and group g - 2's output is copied out. Groups
// ramp up in width (4, 6, then 8 heads) so that the first group, whose copy
// nothing hides, is small, while the later ones keep copy rows wide.
struct HostPipe {
  static constexpr int kMaxWidth = 8;  // heads in the widest group
  std::vector<int> widths;             // heads per group, in order; one entry: no pipeline
  vsa_plan* sub[kMaxWidth + 1] = {};   // sub[w]: the plan of a w-head group (where used)
  int max_width = 0;
  cudaStream_t s_in = nullptr, s_out = nullptr;  // created on first use
  cudaEvent_t entry = nullptr, in_ready[2] = {}, fwd_done[2] = {}, out_done[2] = {};
};

struct vsa_plan {
  vsa_shape_t shape;
  int device;
  int subblock;         // 0: VSA (coarse branch + top-k); 1: SubBlock routing, no coarse term
  int coarse_tc;        // VSA: 1 when the coarse branch runs on the tcgen05 kernel
  double sparsity;      // SubBlock plans: fraction of video key tiles that may be dropped
  vsa::Geometry g;
  size_t off_err, off_pq, off_pk, off_pv, off_coarse, off_idx, off_redo, off_fq, off_fk, off_vf, ws_bytes;
  int num_sms;          // SM count of `device`, read on the first forward
  size_t tensor_bytes;  // one bf16 [B, N, H, 128] tensor
  cudaEvent_t events[4];
  bool have_events;
  HostPipe* pipe;       // host-buffer path (null for the plans of head groups)
};
