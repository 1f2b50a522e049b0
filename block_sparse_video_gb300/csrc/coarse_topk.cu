// Coarse tile attention fused with the top-k tile selection.
//
// For each (batch, head) and each video query tile t ("UniServe: serving
// FastH3 at its fastest", section "The FastH3 workload"):
//   s[t][j] = pooled_q[t] . pooled_k[j] / sqrt(128)         over all T video tiles
//   selection(t) = the k largest s[t][j], ties to the lower j, ascending
//   coarse[t] = sum_j softmax_j(s[t][.]) * pooled_v[j]
// The scores live only in shared memory.
//
// A CTA owns R query tiles of one (b, h) and keeps their R x T score rows in
// shared memory. Pooled K (then V) tiles stream through a padded smem chunk of
// 64 rows. Both products run on the tensor cores (mma.sync m16n8k8, tf32) with
// each fp32 operand split into a tf32 head and a tf32 remainder: a*b is taken
// as hi*hi + hi*lo + lo*hi, which leaves out only the lo*lo term (relative size
// ~2^-22), so the scores carry fp32-level error and the selection is an integer
// decision taken on them. Selection is a warp-per-row radix select over the
// order-preserving integer image of the fp32 scores: four passes of 8-bit
// digits, each a 256-bin shared-memory histogram of the keys that still match
// the digits fixed so far, then an in-order compaction that writes the selected
// tile ids ascending. Results are deterministic: the histograms are counts, and
// the compaction follows tile order.
#include "kernels.cuh"
#include "tf32_select.cuh"

namespace vsa {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 64;            // pooled tiles staged per step
constexpr int kQPad = kHeadDim + 4;   // q rows and K chunk rows (floats): conflict-free fragment loads
constexpr int kVPad = kHeadDim + 8;   // V chunk rows
constexpr size_t kSmemBudget = 220 * 1024;

__device__ __forceinline__ void load_rows(float* dst, const float* src, int first, int count, int rows,
                                          int pad) {
  // rows [first, first + rows) of a [count, 128] fp32 array into padded smem; zero past count
  for (int e = threadIdx.x; e < rows * (kHeadDim / 4); e += kThreads) {
    const int r = e / (kHeadDim / 4), c4 = e % (kHeadDim / 4);
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (first + r < count)
      x = __ldg(reinterpret_cast<const float4*>(src + static_cast<size_t>(first + r) * kHeadDim) + c4);
    *reinterpret_cast<float4*>(dst + r * pad + 4 * c4) = x;
  }
}

// Next K or V chunk, fetched into registers (one float4 per thread and step)
// while the current chunk is in use, then stored into the padded smem rows.
constexpr int kChunkF4PerThread = kChunk * (kHeadDim / 4) / kThreads;
static_assert(kChunkF4PerThread * kThreads == kChunk * (kHeadDim / 4), "chunk staging");

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

__device__ __forceinline__ void stash_chunk(float* dst, const float4 (&pre)[kChunkF4PerThread], int pad) {
#pragma unroll
  for (int i = 0; i < kChunkF4PerThread; ++i) {
    const int e = threadIdx.x + i * kThreads;
    const int r = e / (kHeadDim / 4), c4 = e % (kHeadDim / 4);
    *reinterpret_cast<float4*>(dst + r * pad + 4 * c4) = pre[i];
  }
}

// With device lengths the grid and the layout strides are the plan's capacity
// (T_cap tiles per (b, h), k_cap kept tiles per row, score rows of tpad_cap);
// the actual T and k come from the lengths, and CTAs past the actual T return.
template <int R>
__global__ void __launch_bounds__(kThreads, 1)
coarse_topk_kernel(const float* __restrict__ pooled_q, const float* __restrict__ pooled_k,
                   const float* __restrict__ pooled_v, float* __restrict__ coarse,
                   int32_t* __restrict__ tile_index, Geometry cap, DeviceLengths dl, int tpad_cap) {
  constexpr int MT = R >= 16 ? R / 16 : 1;  // m16 row tiles (R = 8 leaves rows 8-15 empty)
  const DynGeom dg = dyn_geom(cap, dl);
  const int T = dg.T, k = dg.k, T_cap = cap.T, k_cap = cap.k;
  if (!dg.valid) {
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *dl.invalid = 1u;  // also without a pool launch
    return;
  }
  if (static_cast<int>(blockIdx.x) * R >= T) return;  // uniform per CTA
  const int tpad = (T + kChunk - 1) / kChunk * kChunk;
  const int sstride = tpad_cap + 4;         // score row stride: conflict-free A-fragment reads
  extern __shared__ __align__(16) float smem[];
  float* S = smem;                          // [R][sstride] scores, then probabilities
  float* sq = S + R * sstride;              // [16 MT][kQPad] pooled queries
  float* sx = sq + 16 * MT * kQPad;         // [kChunk][kVPad] pooled K (row stride kQPad) or V chunk
  float* sl = sx + kChunk * kVPad;          // [R] softmax denominators
  int* hist = reinterpret_cast<int*>(sl + R);  // [kWarps][kBins] radix histograms

  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const int g = lane >> 2, t4 = lane & 3;
  const int t0 = blockIdx.x * R;
  const size_t bh = blockIdx.y;
  const float* gq = pooled_q + bh * T_cap * kHeadDim;
  const float* gk = pooled_k + bh * T_cap * kHeadDim;
  const float* gv = pooled_v + bh * T_cap * kHeadDim;
  const float scale = 0.08838834764831845f;  // 1/sqrt(128)
  const int rows = min(R, T - t0);           // query tiles of this CTA

  load_rows(sq, gq, t0, t0 + rows, 16 * MT, kQPad);

  // ---- scores: warp w computes key columns 8 (w % 8) .. + 7 of each chunk for
  // row tile w / 8 (warps of a row tile that does not exist idle here)
  float4 pre[kChunkF4PerThread];
  fetch_chunk(pre, gk, 0, T);
  const int s_nt = warp % 8, s_m = warp / 8;
  for (int c0 = 0; c0 < tpad; c0 += kChunk) {
    __syncthreads();
    stash_chunk(sx, pre, kQPad);
    __syncthreads();
    if (c0 + kChunk < tpad) fetch_chunk(pre, gk, c0 + kChunk, T);  // in flight during the products
    if (s_m < MT) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      const float* kb = sx + (8 * s_nt + g) * kQPad;
#pragma unroll 4
      for (int kk = 0; kk < kHeadDim; kk += 8) {
        uint32_t bh0, bl0, bh1, bl1;
        split_tf32(kb[kk + t4], bh0, bl0);
        split_tf32(kb[kk + t4 + 4], bh1, bl1);
        uint32_t ah[4], al[4];
        load_a_split(sq + 16 * s_m * kQPad + kk, kQPad, 16, g, t4, ah, al);
        mma_split(acc, ah, al, bh0, bh1, bl0, bl1);
      }
      const int col = c0 + 8 * s_nt + 2 * t4;
      const int r0 = 16 * s_m + g;
      if (r0 < R) *reinterpret_cast<float2*>(S + r0 * sstride + col) = make_float2(acc[0] * scale, acc[1] * scale);
      if (r0 + 8 < R)
        *reinterpret_cast<float2*>(S + (r0 + 8) * sstride + col) = make_float2(acc[2] * scale, acc[3] * scale);
    }
  }
  fetch_chunk(pre, gv, 0, T);  // first V chunk, in flight during the selection
  __syncthreads();

  // ---- per row: radix select of the k-th largest key, ordered compaction, softmax
  const unsigned full = 0xffffffffu;
  for (int r = warp; r < R; r += kWarps) {
    float* row = S + r * sstride;
    const int t = t0 + r;
    if (t < T)
      warp_select_topk(row, T, k, hist + warp * kBins, tile_index + (bh * T_cap + t) * static_cast<size_t>(k_cap),
                       lane);
    // softmax over the T tiles (probabilities overwrite the scores)
    float m = -INFINITY;
    for (int j = lane; j < T; j += 32) m = fmaxf(m, row[j]);
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(full, m, o));
    float l = 0.f;
    for (int j = lane; j < tpad; j += 32) {
      const float p = j < T ? expf(row[j] - m) : 0.f;
      row[j] = p;
      l += p;
    }
    for (int o = 16; o; o >>= 1) l += __shfl_xor_sync(full, l, o);
    if (lane == 0) sl[r] = l;
  }

  // ---- coarse[t] = sum_j p[t][j] * pooled_v[j] / l[t]; warp w owns dims 8w .. 8w + 7
  static_assert(kWarps * 8 == kHeadDim, "one 8-dim column tile per warp");
  float o[MT][4];
#pragma unroll
  for (int m = 0; m < MT; ++m) o[m][0] = o[m][1] = o[m][2] = o[m][3] = 0.f;
  for (int c0 = 0; c0 < tpad; c0 += kChunk) {
    __syncthreads();
    stash_chunk(sx, pre, kVPad);
    __syncthreads();
    if (c0 + kChunk < tpad) fetch_chunk(pre, gv, c0 + kChunk, T);
#pragma unroll 2
    for (int kk = 0; kk < kChunk; kk += 8) {
      const int n = 8 * warp + g;
      uint32_t bh0, bl0, bh1, bl1;
      split_tf32(sx[(kk + t4) * kVPad + n], bh0, bl0);
      split_tf32(sx[(kk + t4 + 4) * kVPad + n], bh1, bl1);
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        uint32_t ah[4], al[4];
        load_a_split(S + 16 * m * sstride + c0 + kk, sstride, R - 16 * m, g, t4, ah, al);
        mma_split(o[m], ah, al, bh0, bh1, bl0, bl1);
      }
    }
  }
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int r = 16 * m + g + 8 * half;
      if (r < rows) {
        const float inv = 1.0f / sl[r];
        float* dst = coarse + (bh * T_cap + t0 + r) * kHeadDim;
        *reinterpret_cast<float2*>(dst + 8 * warp + 2 * t4) = make_float2(o[m][2 * half] * inv, o[m][2 * half + 1] * inv);
      }
    }
}

size_t smem_for(int r, int tpad) {
  const int mt = r >= 16 ? r / 16 : 1;
  return (static_cast<size_t>(r) * (tpad + 4) + static_cast<size_t>(16 * mt) * kQPad +
          static_cast<size_t>(kChunk) * kVPad + r + kWarps * kBins) * sizeof(float);
}

int pick_rows(int tpad) {
  for (int r = 32; r >= 8; r /= 2)
    if (smem_for(r, tpad) <= kSmemBudget) return r;
  return 0;
}

}  // namespace

size_t coarse_smem_bytes(const Geometry& g, int* rows_per_cta) {
  const int tpad = (g.T + kChunk - 1) / kChunk * kChunk;
  const int r = pick_rows(tpad);
  if (rows_per_cta) *rows_per_cta = r;
  if (r == 0) return 0;
  return smem_for(r, tpad);
}

cudaError_t launch_coarse_topk(const Geometry& g, const float* pooled_q, const float* pooled_k,
                               const float* pooled_v, float* coarse, int32_t* tile_index,
                               const DeviceLengths& dl, cudaStream_t stream) {
  int r = 0;
  const size_t smem = coarse_smem_bytes(g, &r);
  if (r == 0) return cudaErrorInvalidValue;
  const int tpad = (g.T + kChunk - 1) / kChunk * kChunk;
  dim3 grid((g.T + r - 1) / r, g.B * g.H);
  cudaError_t e = cudaSuccess;
  switch (r) {
    case 32:
      e = cudaFuncSetAttribute(coarse_topk_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess)
        coarse_topk_kernel<32><<<grid, kThreads, smem, stream>>>(pooled_q, pooled_k, pooled_v, coarse, tile_index, g, dl, tpad);
      break;
    case 16:
      e = cudaFuncSetAttribute(coarse_topk_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess)
        coarse_topk_kernel<16><<<grid, kThreads, smem, stream>>>(pooled_q, pooled_k, pooled_v, coarse, tile_index, g, dl, tpad);
      break;
    default:
      e = cudaFuncSetAttribute(coarse_topk_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess)
        coarse_topk_kernel<8><<<grid, kThreads, smem, stream>>>(pooled_q, pooled_k, pooled_v, coarse, tile_index, g, dl, tpad);
      break;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace vsa
