// SubBlock router: the block-sparse selection of "UniServe: serving FastH3 at
// its fastest", section "How SubBlock Sparse Attention Works". Each 64-token
// block is split into four 16-token sub-blocks on the query and key side
// (n_q = n_k = 4). A pooled log-sum-exp score estimates each key block's
// unnormalised softmax mass for each query block and head, and the router
// keeps the k highest-scoring key blocks.
//
// Readings where the page is silent:
//   * each pair of sub-blocks (a of query block i, b of key block j) stands
//     for n_a * n_b token pairs at the logit q_a . k_b / sqrt(128), where q_a
//     and k_b are the sub-block means. So
//       score(i, j) = log sum_{a,b} n_a n_b exp(q_a . k_b / sqrt(128))
//     over non-empty sub-blocks, exact when Q and K are constant on each
//     sub-block;
//   * routing covers video query blocks over the T video key blocks;
//   * selection is the k largest fp32 scores, ties to the lower block,
//     stored ascending.
//
// A CTA owns R query blocks (4R query sub-rows) of one (batch, head) and keeps
// their R x T block scores in shared memory. Key sub-rows stream through a
// padded 64-row chunk (16 key blocks). The sub-block logits come from split
// TF32 tensor-core products (fp32-level error, as in the coarse kernel).
// Every m16n8 product tile is reduced at once in registers:
//   * its 16 x 8 sub-block logits are 4 query blocks x 2 key blocks of 4 x 4
//     pairs;
//   * the 16 values of one pair of blocks sit in 8 lanes (lane bits 0, 2 and
//     3 vary), so each log-sum-exp takes three shuffle rounds.
// The warp-per-row radix select of the coarse kernel then picks each row's top k.
#include <cmath>

#include "kernels.cuh"
#include "tf32_select.cuh"

namespace vsa {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 64;            // key sub-rows staged per step (16 key blocks)
constexpr int kQPad = kHeadDim + 4;   // padded rows: conflict-free fragment loads
constexpr size_t kSmemBudget = 220 * 1024;
constexpr int kSub = 16;              // tokens per sub-block

__device__ __forceinline__ void load_rows(float* dst, const float* src, int first, int count, int rows) {
  for (int e = threadIdx.x; e < rows * (kHeadDim / 4); e += kThreads) {
    const int r = e / (kHeadDim / 4), c4 = e % (kHeadDim / 4);
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (first + r < count)
      x = __ldg(reinterpret_cast<const float4*>(src + static_cast<size_t>(first + r) * kHeadDim) + c4);
    *reinterpret_cast<float4*>(dst + r * kQPad + 4 * c4) = x;
  }
}

constexpr int kChunkF4PerThread = kChunk * (kHeadDim / 4) / kThreads;

__device__ __forceinline__ void fetch_chunk(float4 (&pre)[kChunkF4PerThread], const float* src, int first,
                                            int count) {
#pragma unroll
  for (int i = 0; i < kChunkF4PerThread; ++i) {
    const int e = threadIdx.x + i * kThreads;
    const int r = e / (kHeadDim / 4), c4 = e % (kHeadDim / 4);
    pre[i] = first + r < count
                 ? __ldg(reinterpret_cast<const float4*>(src + static_cast<size_t>(first + r) * kHeadDim) + c4)
                 : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

__device__ __forceinline__ void stash_chunk(float* dst, const float4 (&pre)[kChunkF4PerThread]) {
#pragma unroll
  for (int i = 0; i < kChunkF4PerThread; ++i) {
    const int e = threadIdx.x + i * kThreads;
    const int r = e / (kHeadDim / 4), c4 = e % (kHeadDim / 4);
    *reinterpret_cast<float4*>(dst + r * kQPad + 4 * c4) = pre[i];
  }
}

// ln(number of valid tokens of sub-block s), -inf for an empty one
__device__ __forceinline__ float ln_count(int s, int Lv) {
  const int n = min(kSub, Lv - kSub * s);
  return n >= kSub ? 2.772588722239781f : (n > 0 ? logf(static_cast<float>(n)) : -INFINITY);
}

template <int R>
__global__ void __launch_bounds__(kThreads, 1)
subblock_router_kernel(const float* __restrict__ sub_q, const float* __restrict__ sub_k,
                       int32_t* __restrict__ tile_index, int T, int Lv, int k, int spad) {
  constexpr int MT = R / 4;                 // m16 tiles of query sub-rows
  const int bstride = spad / 4 + 4;         // block-score row stride (floats)
  extern __shared__ __align__(16) float smem[];
  float* S = smem;                          // [R][bstride] block scores
  float* sq = S + R * bstride;              // [16 MT][kQPad] query sub-block means
  float* sx = sq + 16 * MT * kQPad;         // [kChunk][kQPad] key sub-block means
  int* hist = reinterpret_cast<int*>(sx + kChunk * kQPad);  // [kWarps][kBins]

  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const int g = lane >> 2, t4 = lane & 3;
  const int q0 = blockIdx.x * R;            // first query block of this CTA
  const size_t bh = blockIdx.y;
  const int n_sub = 4 * T;
  const float* gq = sub_q + bh * n_sub * kHeadDim;
  const float* gk = sub_k + bh * n_sub * kHeadDim;
  const float scale = 0.08838834764831845f;  // 1/sqrt(128)

  load_rows(sq, gq, 4 * q0, n_sub, 16 * MT);

  // warp w: key columns 8 (w % 8) .. + 7 of each chunk, m16 tiles w / 8, w / 8 + 2, ...
  const int nt = warp % 8, mg = warp / 8;
  // ln n of this lane's query sub-rows (16 m + g and 16 m + g + 8 of the CTA's 4R)
  float lnq[MT][2];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int h = 0; h < 2; ++h) lnq[m][h] = ln_count(4 * q0 + 16 * m + g + 8 * h, Lv);

  float4 pre[kChunkF4PerThread];
  fetch_chunk(pre, gk, 0, n_sub);
  for (int c0 = 0; c0 < spad; c0 += kChunk) {
    __syncthreads();
    stash_chunk(sx, pre);
    __syncthreads();
    if (c0 + kChunk < spad) fetch_chunk(pre, gk, c0 + kChunk, n_sub);  // in flight during the products
    const int col = c0 + 8 * nt + 2 * t4;  // this lane's two key sub-rows: col, col + 1
    const float lnk0 = ln_count(col, Lv), lnk1 = ln_count(col + 1, Lv);
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      if ((m & 1) != mg) continue;  // warp-uniform: this warp's m16 tiles are mg, mg + 2, ...
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      const float* kb = sx + (8 * nt + g) * kQPad;
#pragma unroll 4
      for (int kk = 0; kk < kHeadDim; kk += 8) {
        uint32_t bh0, bl0, bh1, bl1;
        split_tf32(kb[kk + t4], bh0, bl0);
        split_tf32(kb[kk + t4 + 4], bh1, bl1);
        uint32_t ah[4], al[4];
        load_a_split(sq + 16 * m * kQPad + kk, kQPad, 16, g, t4, ah, al);
        mma_split(acc, ah, al, bh0, bh1, bl0, bl1);
      }
      // acc: (row g, cols 2t4, 2t4+1), (row g+8, same cols). Row g belongs to
      // query block 4m + g/4, row g+8 to 4m + 2 + g/4; columns 2t4, 2t4+1 to
      // key block c0/4 + 2nt + t4/2.
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float x0 = acc[2 * h] * scale + lnq[m][h] + lnk0;
        const float x1 = acc[2 * h + 1] * scale + lnq[m][h] + lnk1;
        float mx = fmaxf(x0, x1);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        float sum = 0.f;
        if (mx > -INFINITY) sum = expf(x0 - mx) + expf(x1 - mx);
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 4);
        sum += __shfl_xor_sync(0xffffffffu, sum, 8);
        const int lb = 4 * m + 2 * h + g / 4;  // query block within the CTA
        if ((g & 3) == 0 && (t4 & 1) == 0 && lb < R)
          S[lb * bstride + c0 / 4 + 2 * nt + t4 / 2] = mx > -INFINITY ? mx + logf(sum) : -INFINITY;
      }
    }
  }
  __syncthreads();

  for (int r = warp; r < R; r += kWarps)
    if (q0 + r < T)
      warp_select_topk(S + r * bstride, T, k, hist + warp * kBins,
                       tile_index + (bh * T + q0 + r) * static_cast<size_t>(k), lane);
}

size_t smem_for(int r, int spad) {
  return (static_cast<size_t>(r) * (spad / 4 + 4) + static_cast<size_t>(4 * r) * kQPad +
          static_cast<size_t>(kChunk) * kQPad + kWarps * kBins) * sizeof(float);
}

int pick_rows(int spad) {
  for (int r = 16; r >= 4; r /= 2)
    if (smem_for(r, spad) <= kSmemBudget) return r;
  return 0;
}

int sub_pad(int T) { return (4 * T + kChunk - 1) / kChunk * kChunk; }

template <int R>
cudaError_t launch_rows(const Geometry& g, const float* sub_q, const float* sub_k, int32_t* tile_index,
                        size_t smem, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(subblock_router_kernel<R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid((g.T + R - 1) / R, g.B * g.H);
  subblock_router_kernel<R><<<grid, kThreads, smem, stream>>>(sub_q, sub_k, tile_index, g.T, g.Lv, g.k,
                                                              sub_pad(g.T));
  return cudaGetLastError();
}

}  // namespace

size_t subblock_router_smem_bytes(const Geometry& g, int* rows_per_cta) {
  const int r = pick_rows(sub_pad(g.T));
  if (rows_per_cta) *rows_per_cta = r;
  return r ? smem_for(r, sub_pad(g.T)) : 0;
}

cudaError_t launch_subblock_router(const Geometry& g, const float* sub_q, const float* sub_k,
                                   int32_t* tile_index, cudaStream_t stream) {
  int r = 0;
  const size_t smem = subblock_router_smem_bytes(g, &r);
  switch (r) {
    case 16: return launch_rows<16>(g, sub_q, sub_k, tile_index, smem, stream);
    case 8: return launch_rows<8>(g, sub_q, sub_k, tile_index, smem, stream);
    case 4: return launch_rows<4>(g, sub_q, sub_k, tile_index, smem, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace vsa
