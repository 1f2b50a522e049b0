// Tile mean-pool (HBM-bound). For every video tile j of every batch, the mean
// of Q, K and V over the tile's valid tokens, in fp32 ("UniServe: serving
// FastH3 at its fastest", section "Fused attention preprocessing": tile
// pooling over valid tokens into FP32 pooled statistics). The same kernel
// with 16-token runs gives the SubBlock router's sub-block means of Q and K
// (section "How SubBlock Sparse Attention Works": four 16-token sub-blocks
// per 64-token block); a run past the end of a ragged last block is empty and
// its mean is written as 0.
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
template <int kLen>
__global__ void __launch_bounds__(kPoolThreads)
pool_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
            const __nv_bfloat16* __restrict__ v, float* __restrict__ pq, float* __restrict__ pk,
            float* __restrict__ pv, int B, int H, int P, int Lv, int N, int T) {
  const int vec = blockIdx.y * kPoolThreads + threadIdx.x;  // 16-byte vector within a row
  const int row_vecs = H * (kHeadDim / 8);
  const int bt = blockIdx.x;  // b * T + t (T runs per batch)
  const int b = bt / T, t = bt % T;
  const __nv_bfloat16* src = blockIdx.z == 0 ? q : (blockIdx.z == 1 ? k : v);
  float* dst = blockIdx.z == 0 ? pq : (blockIdx.z == 1 ? pk : pv);
  if (vec >= row_vecs) return;
  const int n = min(kLen, Lv - t * kLen);
  const int h = vec / (kHeadDim / 8);
  const int d0 = (vec % (kHeadDim / 8)) * 8;
  float4* out = reinterpret_cast<float4*>(dst + ((static_cast<size_t>(b) * H + h) * T + t) * kHeadDim + d0);
  if (n <= 0) {  // empty sub-block of a ragged last block
    out[0] = out[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  const size_t row_stride = static_cast<size_t>(row_vecs);  // in uint4 units
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

}  // namespace

cudaError_t launch_pool(const Geometry& g, const __nv_bfloat16* q, const __nv_bfloat16* k,
                        const __nv_bfloat16* v, float* pooled_q, float* pooled_k,
                        float* pooled_v, cudaStream_t stream) {
  const int row_vecs = g.H * (kHeadDim / 8);
  dim3 grid(g.B * g.T, (row_vecs + kPoolThreads - 1) / kPoolThreads, 3);
  pool_kernel<kTile><<<grid, kPoolThreads, 0, stream>>>(q, k, v, pooled_q, pooled_k, pooled_v, g.B, g.H,
                                                        g.P, g.Lv, g.N, g.T);
  return cudaGetLastError();
}

cudaError_t launch_subpool(const Geometry& g, const __nv_bfloat16* q, const __nv_bfloat16* k, float* sub_q,
                           float* sub_k, cudaStream_t stream) {
  const int row_vecs = g.H * (kHeadDim / 8);
  const int runs = 4 * g.T;  // four 16-token sub-blocks per video tile
  dim3 grid(g.B * runs, (row_vecs + kPoolThreads - 1) / kPoolThreads, 2);
  pool_kernel<kTile / 4><<<grid, kPoolThreads, 0, stream>>>(q, k, nullptr, sub_q, sub_k, nullptr, g.B, g.H,
                                                            g.P, g.Lv, g.N, runs);
  return cudaGetLastError();
}

}  // namespace vsa
