// Tile mean-pool (HBM-bound). For every video tile j of every batch, the mean
// of Q, K and V over the tile's valid tokens, in fp32 ("UniServe: serving
// FastH3 at its fastest", section "Fused attention preprocessing": tile
// pooling over valid tokens into FP32 pooled statistics). A second kernel
// takes 16-token runs of Q and K for the SubBlock router (the SGLang Diffusion benchmark page (MiniMax-H3 on 8x H200),
// section "How SubBlock Sparse Attention Works": four 16-token sub-blocks per 64-token
// block); a run past the end of a ragged last block is empty and its mean is
// written as 0.
//
// A token row holds all heads: H x 128 bf16 = H x 16 sixteen-byte vectors. A
// CTA of 128 threads owns 128 consecutive vectors of the row (8 channels per
// thread, always inside one head) and walks the tile's rows, keeping eight
// independent 16-byte loads in flight per thread. Reads are fully coalesced;
// each thread writes its 8 means as two float4 stores.
#include "kernels.cuh"

namespace vsa {
namespace {

constexpr int kPoolThreads = 128;
constexpr int kUnroll = 8;

__device__ __forceinline__ void accumulate(float (&acc)[8], const uint4& w) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc[2 * i] += __uint_as_float(u[i] << 16);
    acc[2 * i + 1] += __uint_as_float(u[i] & 0xFFFF0000u);
  }
}

// kLen-token runs: run t of batch b covers video tokens kLen t .. kLen t + n - 1
// (n = min(kLen, Lv - kLen t), possibly <= 0); blockIdx.z picks q, k or v.
// With device lengths, the grid covers the plan's capacity and runs past the
// actual video return at once.
template <int kLen>
__global__ void __launch_bounds__(kPoolThreads)
pool_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
            const __nv_bfloat16* __restrict__ v, float* __restrict__ pq, float* __restrict__ pk,
            float* __restrict__ pv, Geometry cap, DeviceLengths dl) {
  const int H = cap.H, N = cap.N, T = cap.T;
  const DynGeom dg = dyn_geom(cap, dl);
  if (!dg.valid) {
    if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0) *dl.invalid = 1u;
    return;
  }
  const int P = dg.P, Lv = dg.Lv;
  const int vec = blockIdx.y * kPoolThreads + threadIdx.x;  // 16-byte vector within a row
  const int row_vecs = H * (kHeadDim / 8);
  const int bt = blockIdx.x;  // b * T + t (T runs per batch)
  const int b = bt / T, t = bt % T;
  const __nv_bfloat16* src = blockIdx.z == 0 ? q : (blockIdx.z == 1 ? k : v);
  float* dst = blockIdx.z == 0 ? pq : (blockIdx.z == 1 ? pk : pv);
  if (vec >= row_vecs || t >= dg.T) return;
  const int n = min(kLen, Lv - t * kLen);
  const int h = vec / (kHeadDim / 8);
  const int d0 = (vec % (kHeadDim / 8)) * 8;
  float4* out = reinterpret_cast<float4*>(dst + ((static_cast<size_t>(b) * H + h) * T + t) * kHeadDim + d0);
  if (n <= 0) {  // empty sub-block of a ragged last block
    out[0] = out[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  const size_t row_stride = static_cast<size_t>(input_row_stride(cap) / 8);  // in uint4 units
  const uint4* base = reinterpret_cast<const uint4*>(src) +
                      (static_cast<size_t>(b) * N + P + static_cast<size_t>(t) * kLen) * row_stride +
                      vec;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  int r = 0;
  for (; r + kUnroll <= n; r += kUnroll) {
    uint4 w[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) w[u] = __ldg(base + static_cast<size_t>(r + u) * row_stride);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) accumulate(acc, w[u]);
  }
  for (; r < n; ++r) accumulate(acc, __ldg(base + static_cast<size_t>(r) * row_stride));
  const float fn = static_cast<float>(n);
  out[0] = make_float4(__fdiv_rn(acc[0], fn), __fdiv_rn(acc[1], fn), __fdiv_rn(acc[2], fn),
                       __fdiv_rn(acc[3], fn));
  out[1] = make_float4(__fdiv_rn(acc[4], fn), __fdiv_rn(acc[5], fn), __fdiv_rn(acc[6], fn),
                       __fdiv_rn(acc[7], fn));
}

// bf16 hi/lo split of x (x ~ hi + lo with hi = bf16(x), lo = bf16(x - hi)),
// packed as bf16x2 words of two consecutive channels
__device__ __forceinline__ void split_pair(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// 16-token sub-block means of q and k for the SubBlock router: fp32 rows
// [B, H, 4T, 128] (runs < 4T), and the same values split into bf16 hi + lo
// (x ~ hi + lo, hi = bf16(x), lo = bf16(x - hi)) as two row-major bf16
// tensors [B, H, spad, 128] (hi rows, then lo rows, in the `frag` buffer).
// Sub-row `run` of (b, h) is sub-block `run` of the video, in token order.
// These rows are the router's tensor-core operands, loaded by TMA. Rows are
// padded to spad per (b, h); runs past the video (n <= 0) are zeros in both
// forms.
__global__ void __launch_bounds__(kPoolThreads)
subpool_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
               float* __restrict__ pq, float* __restrict__ pk, uint4* __restrict__ fq, uint4* __restrict__ fk,
               Geometry cap, DeviceLengths dl, int spad) {
  constexpr int kLen = kTile / 4;
  // the request's prefix and video length (the capacity's layout: H, N, T, spad)
  const DynGeom dg = dyn_geom(cap, dl);
  if (!dg.valid) return;  // reported by the router
  const int H = cap.H, P = dg.P, Lv = dg.Lv, N = cap.N, T = cap.T;
  const int vec = blockIdx.y * kPoolThreads + threadIdx.x;  // 16-byte vector within a row
  const int row_vecs = H * (kHeadDim / 8);
  const int b = blockIdx.x / spad, run = blockIdx.x % spad;
  const __nv_bfloat16* src = blockIdx.z == 0 ? q : k;
  float* dst = blockIdx.z == 0 ? pq : pk;
  uint4* frag = blockIdx.z == 0 ? fq : fk;
  const bool active = vec < row_vecs;
  const int n = min(kLen, Lv - run * kLen);
  const int h = vec / (kHeadDim / 8);
  const int d0 = (vec % (kHeadDim / 8)) * 8;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  if (active && n > 0) {
    const size_t row_stride = static_cast<size_t>(input_row_stride(cap) / 8);  // in uint4 units
    const uint4* base = reinterpret_cast<const uint4*>(src) +
                        (static_cast<size_t>(b) * N + P + static_cast<size_t>(run) * kLen) * row_stride + vec;
    int r = 0;
    for (; r + kUnroll <= n; r += kUnroll) {
      uint4 w[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) w[u] = __ldg(base + static_cast<size_t>(r + u) * row_stride);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) accumulate(acc, w[u]);
    }
    for (; r < n; ++r) accumulate(acc, __ldg(base + static_cast<size_t>(r) * row_stride));
    const float fn = static_cast<float>(n);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = __fdiv_rn(acc[i], fn);
  }
  if (active && run < 4 * T) {
    float4* out = reinterpret_cast<float4*>(dst + ((static_cast<size_t>(b) * H + h) * 4 * T + run) * kHeadDim + d0);
    out[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    out[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
  // bf16 hi and lo rows: this thread's channels d0 .. d0 + 7 of sub-row `run`
  if (!active) return;
  uint32_t hi[4], lo[4];
#pragma unroll
  for (int t4 = 0; t4 < 4; ++t4) split_pair(acc[2 * t4], acc[2 * t4 + 1], hi[t4], lo[t4]);
  const size_t rows = static_cast<size_t>(cap.B) * H * spad;  // hi rows, then as many lo rows
  const size_t at = ((static_cast<size_t>(b) * H + h) * spad + run) * (kHeadDim / 8) + d0 / 8;
  frag[at] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
  frag[rows * (kHeadDim / 8) + at] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
}

}  // namespace

cudaError_t launch_pool(const Geometry& g, const __nv_bfloat16* q, const __nv_bfloat16* k,
                        const __nv_bfloat16* v, float* pooled_q, float* pooled_k,
                        float* pooled_v, const DeviceLengths& dl, cudaStream_t stream) {
  const int row_vecs = g.H * (kHeadDim / 8);
  dim3 grid(g.B * g.T, (row_vecs + kPoolThreads - 1) / kPoolThreads, 3);
  pool_kernel<kTile><<<grid, kPoolThreads, 0, stream>>>(q, k, v, pooled_q, pooled_k, pooled_v, g, dl);
  return cudaGetLastError();
}

int subblock_rows_padded(const Geometry& g) { return (4 * g.T + 127) / 128 * 128; }

cudaError_t launch_subpool(const Geometry& g, const __nv_bfloat16* q, const __nv_bfloat16* k, float* sub_q,
                           float* sub_k, void* frag_q, void* frag_k, const DeviceLengths& dl, cudaStream_t stream) {
  const int row_vecs = g.H * (kHeadDim / 8);
  const int spad = subblock_rows_padded(g);
  dim3 grid(g.B * spad, (row_vecs + kPoolThreads - 1) / kPoolThreads, 2);
  subpool_kernel<<<grid, kPoolThreads, 0, stream>>>(q, k, sub_q, sub_k, static_cast<uint4*>(frag_q),
                                                    static_cast<uint4*>(frag_k), g, dl, spad);
  return cudaGetLastError();
}

}  // namespace vsa
