// Host side of the C ABI declared in include/vsa.h: shape validation, the
// plan, the workspace layout, tensor-map encoding and the kernel launches.
// The plan is host memory only; every device buffer belongs to the caller.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>

#include <nvtx3/nvToolsExt.h>

#include "kernels.cuh"
#include "vsa.h"

#include "host_rows.cuh"
#include "plan.h"

namespace {

constexpr size_t kAlign = 256;
constexpr int64_t kMaxTokens = int64_t(1) << 26;  // keeps token rows and TMA coordinates in int32

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// Tensor map over a bf16 [B, N, H, 128] tensor; one box = 64 channels x 64
// tokens of one (batch, head), 128-byte swizzled (the tcgen05 operand layout).
// Out-of-range token rows read as zeros.
bool encode_bnhd(CUtensorMap* map, const void* ptr, const vsa::Geometry& g) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(vsa::kHeadDim), static_cast<cuuint64_t>(g.H),
                              static_cast<cuuint64_t>(g.N), static_cast<cuuint64_t>(g.B)};
  const cuuint64_t head = static_cast<cuuint64_t>(vsa::kHeadDim) * 2;
  const cuuint64_t row = static_cast<cuuint64_t>(vsa::input_row_stride(g)) * 2;  // bytes between token rows
  const cuuint64_t strides[3] = {head, row, row * static_cast<cuuint64_t>(g.N)};
  const cuuint32_t box[4] = {64, 1, 64, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map over the tcgen05 coarse kernel's score rows read back as bf16
// probabilities: per CTA slot, 64 rows of `tp` floats, each row's bytes
// holding tp bf16 hi values then tp bf16 lo values ({tp keys, 2 planes, 64
// rows, slots}); one box = 64 keys x 1 plane x 64 rows, 128-byte swizzled.
bool encode_prob_rows(CUtensorMap* map, const void* ptr, int tp, int slots) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(tp), 2, 64, static_cast<cuuint64_t>(slots)};
  const cuuint64_t plane = static_cast<cuuint64_t>(tp) * 2;
  const cuuint64_t strides[3] = {plane, 2 * plane, 128 * plane};
  const cuuint32_t box[4] = {64, 1, 64, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map over `rows` bf16 rows of 128 channels per (batch, head), for B H
// of them ({128, rows, B H, 1}); one box = 64 channels x 64 rows, 128-byte
// swizzled. Rows past `rows` read as zeros.
bool encode_rows(CUtensorMap* map, const void* ptr, int rows, int bh) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(vsa::kHeadDim), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(bh), 1};
  const cuuint64_t row = static_cast<cuuint64_t>(vsa::kHeadDim) * 2;
  const cuuint64_t strides[3] = {row, row * rows, row * rows * static_cast<cuuint64_t>(bh)};
  const cuuint32_t box[4] = {64, 64, 1, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

bool aligned(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

// Selects the plan's device for the duration of a call.
struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) { ok = false; return; }
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
  }
  ~DeviceGuard() {
    if (ok && prev >= 0) cudaSetDevice(prev);
  }
};

// NVTX range around the enqueueing of one call (or one kernel launch): a
// profiler attributes the kernels launched inside it to the range. Without a
// profiler attached the calls do nothing.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

vsa_status_t record(const vsa_plan* p, int i, cudaStream_t s) {
  if (!p->have_events) return VSA_OK;
  return cudaEventRecord(p->events[i], s) == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* vsa_status_string(vsa_status_t s) {
  switch (s) {
    case VSA_OK: return "ok";
    case VSA_ERR_INVALID_ARG: return "invalid argument";
    case VSA_ERR_UNSUPPORTED: return "unsupported shape";
    case VSA_ERR_CUDA: return "CUDA error";
    case VSA_ERR_DEVICE_TIMEOUT: return "a bounded wait inside a kernel timed out";
    case VSA_ERR_INTERNAL: return "internal error";
  }
  return "unknown status";
}

}  // extern "C"

namespace {

// Shared by vsa_plan_create (VSA selection) and vsa_plan_create_subblock.
vsa_status_t create_plan(const vsa_shape_t* shape, int device, bool subblock, double sparsity,
                         vsa_plan_t* out) {
  if (!shape || !out) return VSA_ERR_INVALID_ARG;
  *out = nullptr;
  const vsa_shape_t s = *shape;
  if (s.batch < 1 || s.num_heads < 1 || s.len_text < 0 || s.len_audio < 0 || s.len_video < 1 ||
      device < 0)
    return VSA_ERR_INVALID_ARG;
  if (subblock) {
    if (!(std::isfinite(sparsity) && sparsity >= 0.0 && sparsity < 1.0)) return VSA_ERR_INVALID_ARG;
  } else if (!(std::isfinite(s.keep_fraction) && s.keep_fraction > 0.0 && s.keep_fraction <= 1.0)) {
    return VSA_ERR_INVALID_ARG;
  }
  if (s.head_dim != vsa::kHeadDim) return VSA_ERR_UNSUPPORTED;
  const int64_t prefix = s.len_text + s.len_audio;
  const int64_t n = prefix + s.len_video;
  if (n > kMaxTokens || s.num_heads > 1024 || s.batch > 65535) return VSA_ERR_UNSUPPORTED;

  vsa::Geometry g;
  g.B = s.batch;
  g.H = s.num_heads;
  g.P = static_cast<int>(prefix);
  g.Lv = static_cast<int>(s.len_video);
  g.N = static_cast<int>(n);
  g.T = static_cast<int>((s.len_video + vsa::kTile - 1) / vsa::kTile);
  g.TP = static_cast<int>((prefix + vsa::kTile - 1) / vsa::kTile);
  int64_t k;
  if (subblock) {
    // at most floor(s T) key tiles dropped (IEEE double); the kept count rounded up to
    // a multiple of 8 tiles and capped at T
    const int64_t dropped = static_cast<int64_t>(std::floor(sparsity * static_cast<double>(g.T)));
    const int64_t need = g.T - dropped;
    k = (need + 7) / 8 * 8;
  } else {
    // "rounded to a whole number of tiles": round half up, in IEEE double, clamped to [1, T]
    k = static_cast<int64_t>(std::floor(s.keep_fraction * static_cast<double>(g.T) + 0.5));
  }
  if (k < 1) k = 1;
  if (k > g.T) k = g.T;
  g.k = static_cast<int>(k);
  if (static_cast<int64_t>(g.B) * g.H > 65535) return VSA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(g.B) * g.H * (g.TP + g.T) >= (int64_t(1) << 31)) return VSA_ERR_UNSUPPORTED;
  int rows = 0;
  const bool coarse_tc = !subblock && vsa::coarse_tc_supported(g);
  if (subblock ? vsa::subblock_router_smem_bytes(g, &rows) == 0
               : !coarse_tc && vsa::coarse_smem_bytes(g, &rows) == 0)
    return VSA_ERR_UNSUPPORTED;  // T too large for the selection kernel's shared memory

  vsa_plan* p = new (std::nothrow) vsa_plan;
  if (!p) return VSA_ERR_INTERNAL;
  std::memset(p, 0, sizeof(*p));
  p->shape = s;
  p->device = device;
  p->subblock = subblock ? 1 : 0;
  p->coarse_tc = coarse_tc ? 1 : 0;
  p->sparsity = subblock ? sparsity : 0.0;
  p->g = g;
  // VSA: pooled q, k, v and the coarse output, fp32 [B, H, T, 128] each.
  // SubBlock: 16-token sub-block means of q and k, fp32 [B, H, 4T, 128] each.
  const size_t pooled = static_cast<size_t>(g.B) * g.H * g.T * vsa::kHeadDim * sizeof(float);
  const size_t idx = static_cast<size_t>(g.B) * g.H * g.T * g.k * sizeof(int32_t);
  size_t off = 0;
  p->off_err = off;  off += kAlign;
  p->off_pq = off;   off += align_up(subblock ? 4 * pooled : pooled);
  p->off_pk = off;   off += align_up(subblock ? 4 * pooled : pooled);
  p->off_pv = off;   off += subblock ? 0 : align_up(pooled);
  p->off_coarse = off; off += subblock ? 0 : align_up(pooled);
  p->off_idx = off;  off += align_up(idx);
  p->off_redo = off; off += align_up(static_cast<size_t>(g.B) * g.H * (g.TP + g.T) * sizeof(int32_t));
  // SubBlock: the sub-block means again, as bf16 hi/lo mma fragments (512 bytes per padded sub-row)
  const size_t frag = subblock ? static_cast<size_t>(g.B) * g.H * vsa::subblock_rows_padded(g) * 512 : 0;
  p->off_fq = off;   off += align_up(frag);
  p->off_fk = off;   off += align_up(frag);
  // VSA: the pooled Q, K, V again as bf16 hi/lo rows plus the score rows of the
  // tcgen05 coarse kernel, or the pooled K and V as mma fragments for the other one
  p->off_vf = off;
  off += subblock ? 0
                  : align_up(coarse_tc ? vsa::coarse_tc_operand_bytes(g) + vsa::coarse_tc_scratch_bytes(g)
                                       : vsa::coarse_vfrag_bytes(g));
  p->ws_bytes = off;
  p->tensor_bytes = static_cast<size_t>(g.B) * g.N * g.H * vsa::kHeadDim * 2;
  *out = p;
  return VSA_OK;
}

void destroy_plan(vsa_plan* p);

// The host-buffer path pipelines head groups of up to 8 heads (host only: the streams
// and events are created on the first call).
// Head widths of the pipeline's groups. Up to 8 heads: two halves. Beyond:
// 4, 6, then 8 heads per group, the remainder last, split into (r - 2, 2)
// when it has 4 heads or more. The ramp keeps the first group's copy-in
// (which nothing hides) short and each later copy no longer than the forward
// of the group before it; 8-head groups copy 2 KB host rows, wide enough for
// the copy engines to run near the link rate. The 2-head tail keeps the last
// copy-out (which nothing hides either) short.
std::vector<int> head_group_widths(int H) {
  std::vector<int> w;
  if (H <= 1) return {H};
  if (H <= HostPipe::kMaxWidth) return {(H + 1) / 2, H / 2};
  int left = H;
  for (int step = 0; left > 0; ++step) {
    const int want = step == 0 ? 4 : step == 1 ? 6 : HostPipe::kMaxWidth;
    const int take = want < left ? want : left;
    w.push_back(take);
    left -= take;
  }
  if (w.back() >= 4) {
    w.back() -= 2;
    w.push_back(2);
  }
  return w;
}

vsa_status_t make_pipe(vsa_plan* p, bool subblock) {
  HostPipe* pipe = new (std::nothrow) HostPipe;
  if (!pipe) return VSA_ERR_INTERNAL;
  p->pipe = pipe;
  pipe->widths = head_group_widths(p->g.H);
  if (pipe->widths.size() == 1) return VSA_OK;
  vsa_shape_t s = p->shape;
  for (int w : pipe->widths) {
    if (w > pipe->max_width) pipe->max_width = w;
    if (pipe->sub[w]) continue;
    s.num_heads = w;
    vsa_plan_t sub = nullptr;
    const vsa_status_t st = create_plan(&s, p->device, subblock, p->sparsity, &sub);
    if (st != VSA_OK) return st;
    pipe->sub[w] = sub;
  }
  return VSA_OK;
}

void destroy_plan(vsa_plan* p) {
  if (!p) return;
  if (HostPipe* pipe = p->pipe) {
    for (vsa_plan* sub : pipe->sub) destroy_plan(sub);  // null entries are skipped
    if (pipe->s_in) {
      int prev = -1;
      cudaGetDevice(&prev);
      cudaSetDevice(p->device);
      cudaStreamDestroy(pipe->s_in);
      cudaStreamDestroy(pipe->s_out);
      cudaEventDestroy(pipe->entry);
      for (int i = 0; i < 2; ++i) {
        cudaEventDestroy(pipe->in_ready[i]);
        cudaEventDestroy(pipe->fwd_done[i]);
        cudaEventDestroy(pipe->out_done[i]);
      }
      if (prev >= 0) cudaSetDevice(prev);
    }
    delete pipe;
  }
  delete p;
}

}  // namespace

extern "C" {

namespace {

vsa_status_t create_with_pipe(const vsa_shape_t* shape, int device, bool subblock, double sparsity,
                              vsa_plan_t* out) {
  vsa_status_t st = create_plan(shape, device, subblock, sparsity, out);
  if (st != VSA_OK) return st;
  st = make_pipe(*out, subblock);
  if (st != VSA_OK) {
    destroy_plan(*out);
    *out = nullptr;
  }
  return st;
}

}  // namespace

vsa_status_t vsa_plan_create(const vsa_shape_t* shape, int device, vsa_plan_t* out) {
  return create_with_pipe(shape, device, false, 0.0, out);
}

vsa_status_t vsa_plan_create_subblock(const vsa_shape_t* shape, double sparsity, int device, vsa_plan_t* out) {
  return create_with_pipe(shape, device, true, sparsity, out);
}

vsa_status_t vsa_plan_info(vsa_plan_t plan, int64_t* n_tiles, int64_t* k, size_t* workspace_bytes) {
  if (!plan) return VSA_ERR_INVALID_ARG;
  if (n_tiles) *n_tiles = plan->g.T;
  if (k) *k = plan->g.k;
  if (workspace_bytes) *workspace_bytes = plan->ws_bytes;
  return VSA_OK;
}

vsa_status_t vsa_plan_set_stage_events(vsa_plan_t plan, void* const* events) {
  if (!plan) return VSA_ERR_INVALID_ARG;
  if (!events) {
    plan->have_events = false;
    return VSA_OK;
  }
  for (int i = 0; i < 4; ++i) {
    if (!events[i]) return VSA_ERR_INVALID_ARG;
    plan->events[i] = static_cast<cudaEvent_t>(events[i]);
  }
  plan->have_events = true;
  return VSA_OK;
}

}  // extern "C"

namespace {

// The forward behind vsa_forward (pool_ready = false: clears every counter and
// error word, then pools Q/K/V) and vsa_forward_preprocessed (pool_ready = true:
// the pooled statistics and word 7 come from vsa_preprocess and are kept).
// Output layout: null `rows` means the packed [B, N, H, 128] tensor `out`.
// Lengths: null means the plan's own; otherwise device memory read by the kernels.
// in_row_stride: elements between token rows of q, k, v and gate (0: packed, H * 128).
vsa_status_t forward_impl(vsa_plan_t plan, const void* q, const void* k, const void* v, const void* gate,
                          void* out, void* workspace, size_t workspace_bytes, void* stream,
                          bool pool_ready, const vsa_output_rows_t* rows = nullptr,
                          const vsa_lengths_t* lengths = nullptr, int64_t in_row_stride = 0) {
  if (!plan || !q || !k || !v || !out || !workspace) return VSA_ERR_INVALID_ARG;
  if (lengths && !aligned(lengths, 8)) return VSA_ERR_INVALID_ARG;
  if (!gate && !plan->subblock) return VSA_ERR_INVALID_ARG;  // SubBlock routing has no gate
  if (workspace_bytes < plan->ws_bytes || !aligned(workspace, kAlign)) return VSA_ERR_INVALID_ARG;
  if (in_row_stride < 0 || (in_row_stride > 0 && (in_row_stride < static_cast<int64_t>(plan->g.H) * vsa::kHeadDim ||
                                                   in_row_stride % 8 != 0)))
    return VSA_ERR_INVALID_ARG;
  if (in_row_stride > (int64_t(1) << 24)) return VSA_ERR_UNSUPPORTED;
  const void* ins[4] = {q, k, v, gate};
  // bytes one input spans: B * N rows of in_row_stride elements, the last one read up to its H * 128 channels
  const size_t tb = in_row_stride == 0 ? plan->tensor_bytes
                                       : (static_cast<size_t>(plan->g.B) * plan->g.N - 1) *
                                                 static_cast<size_t>(in_row_stride) * 2 +
                                             static_cast<size_t>(plan->g.H) * vsa::kHeadDim * 2;
  // bytes the output spans: the packed tensor, or B * out_rows rows of out_row_stride elements
  size_t out_span = tb;
  if (rows) {
    if (rows->out_rows < 1 || rows->out_row_stride < static_cast<int64_t>(plan->g.H) * vsa::kHeadDim ||
        rows->out_row_stride % 8 != 0)
      return VSA_ERR_INVALID_ARG;
    if (!rows->out_row_map && rows->out_rows < plan->g.N) return VSA_ERR_INVALID_ARG;
    if (rows->out_row_map && !aligned(rows->out_row_map, 4)) return VSA_ERR_INVALID_ARG;
    if (rows->out_row_stride > (int64_t(1) << 24) || rows->out_rows > kMaxTokens * 4) return VSA_ERR_UNSUPPORTED;
    out_span = (static_cast<size_t>(plan->g.B) * rows->out_rows - 1) * static_cast<size_t>(rows->out_row_stride) * 2 +
               static_cast<size_t>(plan->g.H) * vsa::kHeadDim * 2;
  }
  for (const void* x : ins) {
    if (!x) continue;
    if (!aligned(x, 16)) return VSA_ERR_INVALID_ARG;
    if (overlaps(x, tb, out, out_span)) return VSA_ERR_INVALID_ARG;
    if (overlaps(x, tb, workspace, plan->ws_bytes)) return VSA_ERR_INVALID_ARG;
  }
  if (!aligned(out, 16) || overlaps(out, out_span, workspace, plan->ws_bytes)) return VSA_ERR_INVALID_ARG;

  DeviceGuard guard(plan->device);
  if (!guard.ok) return VSA_ERR_CUDA;
  NvtxRange range(plan->subblock ? "vsa_forward (SubBlock)" : "vsa_forward");
  vsa::Geometry g = plan->g;
  g.row_stride = in_row_stride;
  CUtensorMap mq, mk, mv, mg;
  // without a gate (SubBlock routing) the gate map points at q; the kernel never reads it
  if (!encode_bnhd(&mq, q, g) || !encode_bnhd(&mk, k, g) || !encode_bnhd(&mv, v, g) ||
      !encode_bnhd(&mg, gate ? gate : q, g))
    return VSA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  unsigned int* err = reinterpret_cast<unsigned int*>(ws + plan->off_err);
  float* pq = reinterpret_cast<float*>(ws + plan->off_pq);
  float* pk = reinterpret_cast<float*>(ws + plan->off_pk);
  float* pv = reinterpret_cast<float*>(ws + plan->off_pv);
  float* coarse = reinterpret_cast<float*>(ws + plan->off_coarse);
  int32_t* idx = reinterpret_cast<int32_t*>(ws + plan->off_idx);

  if (plan->num_sms == 0 &&
      cudaDeviceGetAttribute(&plan->num_sms, cudaDevAttrMultiProcessorCount, plan->device) != cudaSuccess)
    return VSA_ERR_CUDA;
  // Error words: 0-2 (first error, detail, abort flag), 3 (bad output row map entry), 4 (redo
  // count), 5-6 (the fine kernels' work counters), 7 (bad preprocessing map entry, kept when the
  // preprocessing just wrote it) and 9 (device lengths outside the capacity).
  if (cudaMemsetAsync(err, 0, pool_ready ? 28 : 40, st) != cudaSuccess) return VSA_ERR_CUDA;
  if (pool_ready && cudaMemsetAsync(err + 8, 0, 8, st) != cudaSuccess) return VSA_ERR_CUDA;
  vsa::DeviceLengths dl;
  if (lengths) {
    dl.len = reinterpret_cast<const long long*>(lengths);
    dl.keep = plan->shape.keep_fraction;
    dl.sparsity = plan->subblock ? plan->sparsity : -1.0;
    dl.invalid = err + 9;
  }
  vsa_status_t rs = record(plan, 0, st);
  if (rs != VSA_OK) return rs;
  const __nv_bfloat16* qb = static_cast<const __nv_bfloat16*>(q);
  const __nv_bfloat16* kb = static_cast<const __nv_bfloat16*>(k);
  if (plan->subblock) {
    NvtxRange r_sel("vsa_subpool + vsa_subblock_router");
    // sub-block means are always taken here: the preprocessing pools 64-token tiles
    if (vsa::launch_subpool(g, qb, kb, pq, pk, ws + plan->off_fq, ws + plan->off_fk, dl, st) != cudaSuccess)
      return VSA_ERR_CUDA;
    if ((rs = record(plan, 1, st)) != VSA_OK) return rs;
    // the sub-pool's bf16 rows: hi then lo, spad rows per (b, h), in each of the q and k buffers
    const int spad = vsa::subblock_rows_padded(g);
    const size_t lo_off = static_cast<size_t>(g.B) * g.H * spad * vsa::kHeadDim * 2;
    CUtensorMap maps[4];
    if (!encode_rows(&maps[0], ws + plan->off_fq, spad, g.B * g.H) ||
        !encode_rows(&maps[1], ws + plan->off_fq + lo_off, spad, g.B * g.H) ||
        !encode_rows(&maps[2], ws + plan->off_fk, spad, g.B * g.H) ||
        !encode_rows(&maps[3], ws + plan->off_fk + lo_off, spad, g.B * g.H))
      return VSA_ERR_CUDA;
    if (vsa::launch_subblock_router(g, maps, idx, err, dl, st) != cudaSuccess)
      return VSA_ERR_CUDA;
  } else {
    NvtxRange r_sel("vsa_pool + vsa_coarse_topk");
    if (!pool_ready &&
        vsa::launch_pool(g, qb, kb, static_cast<const __nv_bfloat16*>(v), pq, pk, pv, dl, st) != cudaSuccess)
      return VSA_ERR_CUDA;
    if ((rs = record(plan, 1, st)) != VSA_OK) return rs;
    if (plan->coarse_tc) {
      uint8_t* ops = ws + plan->off_vf;
      const int tp = vsa::coarse_tc_padded(g);
      const size_t plane = static_cast<size_t>(g.B) * g.H * tp * vsa::kHeadDim * 2;
      const int slots = vsa::coarse_tc_units(g) < vsa::kCoarseTcMaxSlots ? vsa::coarse_tc_units(g)
                                                                         : vsa::kCoarseTcMaxSlots;
      float* scratch = reinterpret_cast<float*>(ops + vsa::coarse_tc_operand_bytes(g));
      CUtensorMap maps[7];
      for (int i = 0; i < 6; ++i)
        if (!encode_rows(&maps[i], ops + i * plane, tp, g.B * g.H)) return VSA_ERR_CUDA;
      if (!encode_prob_rows(&maps[6], scratch, tp, slots)) return VSA_ERR_CUDA;
      if (vsa::launch_split(g, pq, pk, pv, ops, dl, st) != cudaSuccess ||
          vsa::launch_coarse_tc(g, maps, scratch, coarse, idx, err, dl, plan->num_sms, st) != cudaSuccess)
        return VSA_ERR_CUDA;
    } else if (vsa::launch_coarse_topk(g, pq, pk, pv, coarse, idx, ws + plan->off_vf, dl, st) != cudaSuccess) {
      return VSA_ERR_CUDA;
    }
  }
  if ((rs = record(plan, 2, st)) != VSA_OK) return rs;
  vsa::FineArgs a;
  a.gate = static_cast<const __nv_bfloat16*>(gate);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.coarse = plan->subblock ? nullptr : coarse;
  a.dl = dl;
  if (rows) {
    a.out_row_map = rows->out_row_map;
    a.out_rows = rows->out_rows;
    a.out_row_stride = rows->out_row_stride;
  } else {
    a.out_row_map = nullptr;
  }
  a.tile_index = idx;
  a.err = err;
  a.redo_count = reinterpret_cast<int*>(err + 4);
  a.redo_list = reinterpret_cast<int32_t*>(ws + plan->off_redo);
  a.work_counters = reinterpret_cast<int*>(err + 5);
  {
    NvtxRange r_fine("vsa_fine_attn");
    if (vsa::launch_fine(g, mq, mk, mv, mg, a, plan->num_sms, st) != cudaSuccess) return VSA_ERR_CUDA;
  }
  return record(plan, 3, st);
}

// Bytes spanned by one projection input: B * rows_in rows of row_stride elements,
// the last one read up to its H * 128 channels.
size_t projection_span(const vsa::Geometry& g, int64_t rows_in, int64_t row_stride) {
  return (static_cast<size_t>(g.B) * rows_in - 1) * static_cast<size_t>(row_stride) * 2 +
         static_cast<size_t>(g.H) * vsa::kHeadDim * 2;
}

}  // namespace

extern "C" {

vsa_status_t vsa_forward(vsa_plan_t plan, const void* q, const void* k, const void* v,
                         const void* gate, void* out, void* workspace, size_t workspace_bytes,
                         void* stream) {
  return forward_impl(plan, q, k, v, gate, out, workspace, workspace_bytes, stream, false);
}

vsa_status_t vsa_forward_preprocessed(vsa_plan_t plan, const void* q, const void* k, const void* v,
                                      const void* gate, void* out, void* workspace,
                                      size_t workspace_bytes, void* stream) {
  return forward_impl(plan, q, k, v, gate, out, workspace, workspace_bytes, stream, true);
}

vsa_status_t vsa_forward_lengths(vsa_plan_t plan, const vsa_lengths_t* lengths, const void* q, const void* k,
                                 const void* v, const void* gate, void* out, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  if (!lengths) return VSA_ERR_INVALID_ARG;
  return forward_impl(plan, q, k, v, gate, out, workspace, workspace_bytes, stream, false, nullptr, lengths);
}

vsa_status_t vsa_forward_ex(vsa_plan_t plan, const vsa_forward_args_t* a, void* workspace,
                            size_t workspace_bytes, void* stream) {
  if (!a) return VSA_ERR_INVALID_ARG;
  void* out = a->rows ? a->rows->out : a->out;
  return forward_impl(plan, a->q, a->k, a->v, a->gate, out, workspace, workspace_bytes, stream, a->preprocessed != 0,
                      a->rows, a->lengths, a->in_row_stride);
}

vsa_status_t vsa_forward_rows(vsa_plan_t plan, const void* q, const void* k, const void* v, const void* gate,
                              const vsa_output_rows_t* out, int32_t preprocessed, void* workspace,
                              size_t workspace_bytes, void* stream) {
  if (!out || !out->out) return VSA_ERR_INVALID_ARG;
  return forward_impl(plan, q, k, v, gate, out->out, workspace, workspace_bytes, stream, preprocessed != 0, out);
}

vsa_status_t vsa_preprocess(vsa_plan_t plan, const vsa_preprocess_args_t* args, void* workspace,
                            size_t workspace_bytes, void* stream) {
  if (!plan || !args || !workspace) return VSA_ERR_INVALID_ARG;
  const vsa_preprocess_args_t& x = *args;
  const vsa::Geometry& g = plan->g;
  if (workspace_bytes < plan->ws_bytes || !aligned(workspace, kAlign)) return VSA_ERR_INVALID_ARG;
  const void* ins[4] = {x.q_in, x.k_in, x.v_in, x.gate_in};
  void* outs[4] = {x.q_out, x.k_out, x.v_out, x.gate_out};
  if (x.rows_in < 1 || x.row_stride < static_cast<int64_t>(g.H) * vsa::kHeadDim || x.row_stride % 8 != 0)
    return VSA_ERR_INVALID_ARG;
  if (!x.src_row && x.rows_in < g.N) return VSA_ERR_INVALID_ARG;
  if (x.rows_in > kMaxTokens * 4 || x.row_stride > (int64_t(1) << 24)) return VSA_ERR_UNSUPPORTED;
  if (x.src_row && !aligned(x.src_row, 4)) return VSA_ERR_INVALID_ARG;
  if (!x.q_norm_weight || !x.k_norm_weight || !aligned(x.q_norm_weight, 4) || !aligned(x.k_norm_weight, 4))
    return VSA_ERR_INVALID_ARG;
  if (!(std::isfinite(x.eps) && x.eps > 0.f)) return VSA_ERR_INVALID_ARG;
  if (x.rope_dim < 0 || x.rope_dim > vsa::kHeadDim || x.rope_dim % 16 != 0) return VSA_ERR_INVALID_ARG;
  if (x.rope_dim > 0 && (!x.rope_cos || !x.rope_sin || !aligned(x.rope_cos, 16) || !aligned(x.rope_sin, 16)))
    return VSA_ERR_INVALID_ARG;
  const size_t span = projection_span(g, x.rows_in, x.row_stride);
  const size_t tb = plan->tensor_bytes;
  for (int i = 0; i < 4; ++i) {
    if (!ins[i] || !outs[i] || !aligned(ins[i], 16) || !aligned(outs[i], 16)) return VSA_ERR_INVALID_ARG;
    if (overlaps(outs[i], tb, workspace, plan->ws_bytes)) return VSA_ERR_INVALID_ARG;
    for (int j = 0; j < 4; ++j) {
      if (overlaps(outs[i], tb, ins[j], span)) return VSA_ERR_INVALID_ARG;
      if (j > i && overlaps(outs[i], tb, outs[j], tb)) return VSA_ERR_INVALID_ARG;
    }
  }

  DeviceGuard guard(plan->device);
  if (!guard.ok) return VSA_ERR_CUDA;
  NvtxRange range("vsa_preprocess");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  unsigned int* err = reinterpret_cast<unsigned int*>(ws + plan->off_err);
  // a preprocessing starts a new call sequence: every error word and counter (0-9) starts at zero
  if (cudaMemsetAsync(err, 0, 40, st) != cudaSuccess) return VSA_ERR_CUDA;
  vsa::PreprocessArgs a;
  for (int i = 0; i < 4; ++i) {
    a.in[i] = static_cast<const __nv_bfloat16*>(ins[i]);
    a.out[i] = static_cast<__nv_bfloat16*>(outs[i]);
  }
  a.rows_in = x.rows_in;
  a.row_stride = x.row_stride;
  a.src_row = x.src_row;
  a.q_norm_weight = x.q_norm_weight;
  a.k_norm_weight = x.k_norm_weight;
  a.eps = x.eps;
  a.rope_dim = x.rope_dim;
  a.rope_interleaved = x.rope_interleaved;
  a.rope_cos = x.rope_cos;
  a.rope_sin = x.rope_sin;
  if (x.lengths) {
    if (!aligned(x.lengths, 8)) return VSA_ERR_INVALID_ARG;
    a.dl.len = reinterpret_cast<const long long*>(x.lengths);
    a.dl.keep = plan->shape.keep_fraction;
    a.dl.sparsity = plan->subblock ? plan->sparsity : -1.0;
    a.dl.invalid = err + 9;
  }
  // a SubBlock plan pools 16-token sub-blocks in its forward: no tile pooling here
  a.pooled[0] = plan->subblock ? nullptr : reinterpret_cast<float*>(ws + plan->off_pq);
  a.pooled[1] = plan->subblock ? nullptr : reinterpret_cast<float*>(ws + plan->off_pk);
  a.pooled[2] = plan->subblock ? nullptr : reinterpret_cast<float*>(ws + plan->off_pv);
  a.err = err;
  return vsa::launch_preprocess(g, a, st) == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
}

namespace {

// Layout of head group gi inside the host path's device buffer. Groups
// alternate between two slots; every group lays its five tensors out at the
// widest group's tensor stride, whatever its own width, so a group's inputs
// never overlap the output region of the group two before it (which the
// copy-out stream may still be reading while those inputs are copied in).
struct GroupLayout {
  int first_head, heads, slot;
  size_t off[5];        // q, k, v, gate, out
  size_t tensor_bytes;  // this group's tensors
  size_t ws_off, ws_bytes;
};

GroupLayout group_layout(const vsa_plan* p, int gi) {
  const HostPipe* pipe = p->pipe;
  GroupLayout L{};
  const size_t tstride = align_up(pipe->sub[pipe->max_width]->tensor_bytes);
  const size_t slot_bytes = 5 * tstride;
  for (int i = 0; i < gi; ++i) L.first_head += pipe->widths[i];
  L.heads = pipe->widths[gi];
  L.slot = gi & 1;
  for (int i = 0; i < 5; ++i) L.off[i] = L.slot * slot_bytes + i * tstride;
  L.tensor_bytes = pipe->sub[L.heads]->tensor_bytes;
  L.ws_off = 2 * slot_bytes;
  size_t ws = 0;
  for (const vsa_plan* sub : pipe->sub)
    if (sub && sub->ws_bytes > ws) ws = sub->ws_bytes;
  L.ws_bytes = ws;
  return L;
}

size_t pipe_bytes(const vsa_plan* p) {
  const HostPipe* pipe = p->pipe;
  if (!pipe || pipe->widths.size() == 1) return 5 * align_up(p->tensor_bytes) + p->ws_bytes;
  const GroupLayout L = group_layout(p, 0);
  return L.ws_off + L.ws_bytes;
}

// Device-side address of host memory the device can read (pinned or
// registered), else null.
const uint8_t* device_view_of_host(const void* h) {
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, h) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (attr.type != cudaMemoryTypeHost || !attr.devicePointer) return nullptr;
  return static_cast<const uint8_t*>(attr.devicePointer);
}

vsa_status_t ensure_streams(HostPipe* pipe) {
  if (pipe->s_in) return VSA_OK;
  bool ok = cudaStreamCreateWithFlags(&pipe->s_in, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&pipe->s_out, cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreateWithFlags(&pipe->entry, cudaEventDisableTiming) == cudaSuccess;
  for (int i = 0; i < 2 && ok; ++i)
    ok = cudaEventCreateWithFlags(&pipe->in_ready[i], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&pipe->fwd_done[i], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&pipe->out_done[i], cudaEventDisableTiming) == cudaSuccess;
  return ok ? VSA_OK : VSA_ERR_CUDA;
}

}  // namespace

vsa_status_t vsa_plan_host_path_bytes(vsa_plan_t plan, size_t* bytes) {
  if (!plan || !bytes) return VSA_ERR_INVALID_ARG;
  *bytes = pipe_bytes(plan);
  return VSA_OK;
}

vsa_status_t vsa_plan_host_path_group(vsa_plan_t plan, int32_t group, int32_t* n_groups, int32_t* first_head,
                                      int32_t* heads, size_t* offsets, size_t* tensor_bytes,
                                      size_t* workspace_offset, size_t* workspace_bytes) {
  if (!plan) return VSA_ERR_INVALID_ARG;
  const HostPipe* pipe = plan->pipe;
  const bool piped = pipe && pipe->widths.size() > 1;
  const int32_t ng = piped ? static_cast<int32_t>(pipe->widths.size()) : 1;
  if (n_groups) *n_groups = ng;
  if (!n_groups || !first_head || !heads || !offsets || !tensor_bytes || !workspace_offset || !workspace_bytes)
    return VSA_ERR_INVALID_ARG;
  if (group < 0 || group >= ng) return VSA_ERR_INVALID_ARG;
  if (!piped) {
    const size_t slot = align_up(plan->tensor_bytes);
    *first_head = 0;
    *heads = plan->g.H;
    for (int i = 0; i < 5; ++i) offsets[i] = i * slot;
    *tensor_bytes = plan->tensor_bytes;
    *workspace_offset = 5 * slot;
    *workspace_bytes = plan->ws_bytes;
    return VSA_OK;
  }
  const GroupLayout L = group_layout(plan, group);
  *first_head = L.first_head;
  *heads = L.heads;
  for (int i = 0; i < 5; ++i) offsets[i] = L.off[i];
  *tensor_bytes = L.tensor_bytes;
  *workspace_offset = L.ws_off;
  *workspace_bytes = L.ws_bytes;
  return VSA_OK;
}

vsa_status_t vsa_forward_host(vsa_plan_t plan, const void* q, const void* k, const void* v,
                              const void* gate, void* out, void* device_buffer,
                              size_t device_buffer_bytes, void* stream) {
  if (!plan || !q || !k || !v || !out || !device_buffer) return VSA_ERR_INVALID_ARG;
  if (!gate && !plan->subblock) return VSA_ERR_INVALID_ARG;
  if (device_buffer_bytes < pipe_bytes(plan) || !aligned(device_buffer, kAlign)) return VSA_ERR_INVALID_ARG;
  DeviceGuard guard(plan->device);
  if (!guard.ok) return VSA_ERR_CUDA;
  NvtxRange range("vsa_forward_host");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* d = static_cast<uint8_t*>(device_buffer);
  const void* hin[4] = {q, k, v, gate};
  HostPipe* pipe = plan->pipe;
  if (!pipe || pipe->widths.size() == 1) {
    const size_t tb = plan->tensor_bytes, slot = align_up(tb);
    for (int i = 0; i < 4; ++i)
      if (hin[i] && cudaMemcpyAsync(d + i * slot, hin[i], tb, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return VSA_ERR_CUDA;
    vsa_status_t s = vsa_forward(plan, d, d + slot, d + 2 * slot, gate ? d + 3 * slot : nullptr, d + 4 * slot,
                                 d + 5 * slot, plan->ws_bytes, stream);
    if (s != VSA_OK) return s;
    if (cudaMemcpyAsync(out, d + 4 * slot, tb, cudaMemcpyDeviceToHost, st) != cudaSuccess) return VSA_ERR_CUDA;
    return cudaStreamSynchronize(st) == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
  }

  // Head groups: group g's q/k/v/gate rows (its heads' 256-byte slices of every
  // host row) are copied in on s_in, its forward runs on the caller's stream,
  // and its output is copied out on s_out, two groups' buffers alternating.
  // The first group's rows are gathered by a kernel reading the host memory
  // when every input is pinned, and the last group's output is written by a
  // kernel when `out` is pinned; the rest go through strided copies that hide
  // under the neighbouring groups' forwards.
  vsa_status_t rs = ensure_streams(pipe);
  if (rs != VSA_OK) return rs;
  if (plan->num_sms == 0 &&
      cudaDeviceGetAttribute(&plan->num_sms, cudaDevAttrMultiProcessorCount, plan->device) != cudaSuccess)
    return VSA_ERR_CUDA;
  const vsa::Geometry& g = plan->g;
  const size_t rows = static_cast<size_t>(g.B) * g.N;
  const size_t host_pitch = static_cast<size_t>(g.H) * vsa::kHeadDim * 2;
  const int n_in = gate ? 4 : 3;
  const uint8_t* dev_in[4] = {nullptr, nullptr, nullptr, nullptr};
  bool gather_first = true;
  for (int i = 0; i < n_in && gather_first; ++i) {
    dev_in[i] = device_view_of_host(hin[i]);
    gather_first = dev_in[i] && reinterpret_cast<uintptr_t>(dev_in[i]) % 16 == 0;
  }
  uint8_t* dev_out = const_cast<uint8_t*>(device_view_of_host(out));
  const bool scatter_last = dev_out && reinterpret_cast<uintptr_t>(dev_out) % 16 == 0;
  auto cuda = [](cudaError_t e) { return e == cudaSuccess; };
  if (!cuda(cudaEventRecord(pipe->entry, st)) || !cuda(cudaStreamWaitEvent(pipe->s_in, pipe->entry, 0)))
    return VSA_ERR_CUDA;
  // Ordering (each stream runs in issue order): the copy-in of group gi waits
  // for the forward of gi - 2 (the last reader of its slot's inputs); the
  // forward of gi waits for its copy-in and for the copy-out of gi - 2 (the
  // last reader of its slot's output); the copy-out of gi waits for its
  // forward. The copy-out of gi - 2 may still run during the copy-in of gi,
  // which is why group_layout keeps inputs and outputs apart in every slot.
  const int groups = static_cast<int>(pipe->widths.size());
  for (int gi = 0; gi < groups; ++gi) {
    const GroupLayout L = group_layout(plan, gi);
    const int s = L.slot, h0 = L.first_head;
    vsa_plan* sub = pipe->sub[L.heads];
    const size_t width = static_cast<size_t>(sub->g.H) * vsa::kHeadDim * 2;
    uint8_t* const t[5] = {d + L.off[0], d + L.off[1], d + L.off[2], d + L.off[3], d + L.off[4]};
    uint8_t* ws = d + L.ws_off;
    // inputs: slot s is free once the forward of group gi - 2 has read it
    if (gi >= 2 && !cuda(cudaStreamWaitEvent(pipe->s_in, pipe->fwd_done[s], 0))) return VSA_ERR_CUDA;
    if (gi == 0 && gather_first) {
      vsa::HostRows a{};
      for (int i = 0; i < n_in; ++i) {
        a.src[i] = dev_in[i] + h0 * 256;
        a.dst[i] = t[i];
      }
      a.src_pitch = host_pitch;
      a.dst_pitch = width;
      a.width = width;
      a.rows = rows;
      a.tensors = n_in;
      if (!cuda(vsa::launch_copy_host_rows(a, plan->num_sms, pipe->s_in))) return VSA_ERR_CUDA;
    } else {
      for (int i = 0; i < n_in; ++i)
        if (!cuda(cudaMemcpy2DAsync(t[i], width, static_cast<const uint8_t*>(hin[i]) + h0 * 256,
                                    host_pitch, width, rows, cudaMemcpyHostToDevice, pipe->s_in)))
          return VSA_ERR_CUDA;
    }
    if (!cuda(cudaEventRecord(pipe->in_ready[s], pipe->s_in))) return VSA_ERR_CUDA;
    // forward: after its inputs, and after group gi - 2's output left slot s
    if (!cuda(cudaStreamWaitEvent(st, pipe->in_ready[s], 0))) return VSA_ERR_CUDA;
    if (gi >= 2 && !cuda(cudaStreamWaitEvent(st, pipe->out_done[s], 0))) return VSA_ERR_CUDA;
    rs = vsa_forward(sub, t[0], t[1], t[2], gate ? t[3] : nullptr, t[4], ws, L.ws_bytes, stream);
    if (rs != VSA_OK) return rs;
    if (!cuda(cudaEventRecord(pipe->fwd_done[s], st))) return VSA_ERR_CUDA;
    // output; the last group's, which nothing hides, is written by a kernel when `out` is pinned
    if (!cuda(cudaStreamWaitEvent(pipe->s_out, pipe->fwd_done[s], 0))) return VSA_ERR_CUDA;
    if (gi == groups - 1 && scatter_last) {
      vsa::HostRows a{};
      a.src[0] = t[4];
      a.dst[0] = dev_out + h0 * 256;
      a.src_pitch = width;
      a.dst_pitch = host_pitch;
      a.width = width;
      a.rows = rows;
      a.tensors = 1;
      if (!cuda(vsa::launch_copy_host_rows(a, plan->num_sms, pipe->s_out))) return VSA_ERR_CUDA;
    } else if (!cuda(cudaMemcpy2DAsync(static_cast<uint8_t*>(out) + h0 * 256, host_pitch, t[4], width,
                                       width, rows, cudaMemcpyDeviceToHost, pipe->s_out))) {
      return VSA_ERR_CUDA;
    }
    if (!cuda(cudaEventRecord(pipe->out_done[s], pipe->s_out))) return VSA_ERR_CUDA;
  }
  for (int s = 0; s < 2 && s < groups; ++s)
    if (!cuda(cudaStreamWaitEvent(st, pipe->out_done[s], 0))) return VSA_ERR_CUDA;
  return cudaStreamSynchronize(st) == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
}

vsa_status_t vsa_debug_views(vsa_plan_t plan, void* workspace, const float** pooled_q,
                             const float** pooled_k, const float** pooled_v,
                             const int32_t** tile_index, const float** coarse) {
  if (!plan || !workspace) return VSA_ERR_INVALID_ARG;
  const uint8_t* ws = static_cast<const uint8_t*>(workspace);
  if (pooled_q) *pooled_q = reinterpret_cast<const float*>(ws + plan->off_pq);
  if (pooled_k) *pooled_k = reinterpret_cast<const float*>(ws + plan->off_pk);
  if (pooled_v) *pooled_v = plan->subblock ? nullptr : reinterpret_cast<const float*>(ws + plan->off_pv);
  if (tile_index) *tile_index = reinterpret_cast<const int32_t*>(ws + plan->off_idx);
  if (coarse) *coarse = plan->subblock ? nullptr : reinterpret_cast<const float*>(ws + plan->off_coarse);
  return VSA_OK;
}

vsa_status_t vsa_check(vsa_plan_t plan, void* workspace, void* stream) {
  if (!plan || !workspace) return VSA_ERR_INVALID_ARG;
  DeviceGuard guard(plan->device);
  if (!guard.ok) return VSA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return VSA_ERR_CUDA;
  unsigned int words[10] = {0, 0, 0, 0, 0, 0, 0, 0, 0, 0};
  if (cudaMemcpy(words, static_cast<uint8_t*>(workspace) + plan->off_err, sizeof(words),
                 cudaMemcpyDeviceToHost) != cudaSuccess)
    return VSA_ERR_CUDA;
  if (words[0] == static_cast<unsigned int>(VSA_ERR_DEVICE_TIMEOUT)) return VSA_ERR_DEVICE_TIMEOUT;
  if (words[0] != 0) return VSA_ERR_INTERNAL;
  if (words[7] != 0) return VSA_ERR_INVALID_ARG;  // a preprocessing map entry outside its buffer
  if (words[3] != 0) return VSA_ERR_INVALID_ARG;  // an output map entry outside the output rows
  if (words[9] != 0) return VSA_ERR_INVALID_ARG;  // device lengths outside the plan's capacity
  return VSA_OK;
}

void vsa_plan_destroy(vsa_plan_t plan) { destroy_plan(plan); }

}  // extern "C"
