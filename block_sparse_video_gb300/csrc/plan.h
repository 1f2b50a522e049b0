// The host-side plan behind the opaque vsa_plan_t handle of include/vsa.h.
#pragma once
#include <cstddef>
#include <cuda_runtime.h>

#include "kernels.cuh"
#include "vsa.h"

struct vsa_plan {
  vsa_shape_t shape;
  int device;
  int subblock;         // 0: VSA (coarse branch + top-k); 1: SubBlock routing, no coarse term
  double sparsity;      // SubBlock plans: fraction of video key tiles that may be dropped
  vsa::Geometry g;
  size_t off_err, off_pq, off_pk, off_pv, off_coarse, off_idx, off_redo, off_fq, off_fk, ws_bytes;
  int num_sms;          // SM count of `device`, read on the first forward
  size_t tensor_bytes;  // one bf16 [B, N, H, 128] tensor
  cudaEvent_t events[4];
  bool have_events;
};
