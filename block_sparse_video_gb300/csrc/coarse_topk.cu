// Coarse tile attention fused with the top-k tile selection.
//
// For each (batch, head) and each video query tile t ("UniServe: serving
// FastH3 at its fastest", section "The FastH3 workload"):
//   s[t][j] = pooled_q[t] . pooled_k[j] / sqrt(128)         over all T video tiles
//   selection(t) = the k largest s[t][j], ties to the lower j, ascending
//   coarse[t] = sum_j softmax_j(s[t][.]) * pooled_v[j]
// The scores live only in shared memory. Everything is fp32 FFMA: the
// selection is an integer decision taken in fp32.
//
// A CTA owns R query tiles of one (b, h) and keeps their R x T score rows in
// shared memory. Pooled K (then V) tiles stream through a padded smem chunk of
// 64 rows. Selection is a warp-per-row radix select over the order-preserving
// integer image of the fp32 scores: four passes of 8-bit digits, each a
// 256-bin shared-memory histogram of the keys that still match the digits
// fixed so far, then an in-order compaction that writes the selected tile ids
// ascending. Results are deterministic: the histograms are counts, and the
// compaction follows tile order.
#include "kernels.cuh"

namespace vsa {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 64;        // pooled tiles staged per step
constexpr int kPad = kHeadDim + 4;  // padded smem row (floats): conflict-free float4 reads
constexpr size_t kSmemBudget = 220 * 1024;
constexpr int kBins = 256;          // radix-select histogram, one per warp

// Order-preserving map from fp32 to uint32 (larger float -> larger key);
// -0 and +0 map to the same key.
__device__ __forceinline__ uint32_t order_key(float s) {
  uint32_t u = __float_as_uint(s);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ void load_rows(float* dst, const float* src, int first, int count,
                                          int rows) {
  // rows [first, first + rows) of a [count, 128] fp32 array into padded smem; zero past count
  for (int e = threadIdx.x; e < rows * (kHeadDim / 4); e += kThreads) {
    const int r = e / (kHeadDim / 4), c4 = e % (kHeadDim / 4);
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (first + r < count)
      x = __ldg(reinterpret_cast<const float4*>(src + static_cast<size_t>(first + r) * kHeadDim) + c4);
    *reinterpret_cast<float4*>(dst + r * kPad + 4 * c4) = x;
  }
}

template <int R>
__global__ void __launch_bounds__(kThreads, 1)
coarse_topk_kernel(const float* __restrict__ pooled_q, const float* __restrict__ pooled_k,
                   const float* __restrict__ pooled_v, float* __restrict__ coarse,
                   int32_t* __restrict__ tile_index, int T, int k, int tpad) {
  extern __shared__ __align__(16) float smem[];
  float* S = smem;                    // [R][tpad] scores, then probabilities
  float* sq = S + R * tpad;           // [R][kPad] pooled queries
  float* sx = sq + R * kPad;          // [kChunk][kPad] pooled K or V chunk
  float* sl = sx + kChunk * kPad;     // [R] softmax denominators
  int* hist = reinterpret_cast<int*>(sl + R);  // [kWarps][kBins] radix histograms

  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const int t0 = blockIdx.x * R;
  const size_t bh = blockIdx.y;
  const float* gq = pooled_q + bh * T * kHeadDim;
  const float* gk = pooled_k + bh * T * kHeadDim;
  const float* gv = pooled_v + bh * T * kHeadDim;
  const float scale = 0.08838834764831845f;  // 1/sqrt(128)

  load_rows(sq, gq, t0, T, R);

  // ---- scores: thread -> one query row, KPT keys of each chunk
  constexpr int TPR = kThreads / R;   // threads per query row
  constexpr int KPT = kChunk / TPR;   // keys per thread per chunk
  const int my_r = tid / TPR, my_k = tid % TPR;
  for (int c0 = 0; c0 < tpad; c0 += kChunk) {
    __syncthreads();
    load_rows(sx, gk, c0, T, kChunk);
    __syncthreads();
    float acc[KPT];
#pragma unroll
    for (int i = 0; i < KPT; ++i) acc[i] = 0.f;
    const float* qrow = sq + my_r * kPad;
#pragma unroll 4
    for (int d = 0; d < kHeadDim; d += 4) {
      const float4 a = *reinterpret_cast<const float4*>(qrow + d);
#pragma unroll
      for (int i = 0; i < KPT; ++i) {
        const float4 b = *reinterpret_cast<const float4*>(sx + (my_k + TPR * i) * kPad + d);
        acc[i] = fmaf(a.x, b.x, acc[i]);
        acc[i] = fmaf(a.y, b.y, acc[i]);
        acc[i] = fmaf(a.z, b.z, acc[i]);
        acc[i] = fmaf(a.w, b.w, acc[i]);
      }
    }
#pragma unroll
    for (int i = 0; i < KPT; ++i) S[my_r * tpad + c0 + my_k + TPR * i] = acc[i] * scale;
  }
  __syncthreads();

  // ---- per row: radix select of the k-th largest key, ordered compaction, softmax
  const unsigned full = 0xffffffffu;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int r = warp; r < R; r += kWarps) {
    float* row = S + r * tpad;
    const int t = t0 + r;
    if (t < T) {
      // radix select, 8 bits per pass from the top: prefix holds the digits of
      // the k-th largest key fixed so far, rem how many keys above it are
      // still to be taken among those that match the prefix
      int* h = hist + warp * kBins;
      uint32_t prefix = 0u, pmask = 0u;
      int rem = k;
#pragma unroll 1
      for (int shift = 24; shift >= 0; shift -= 8) {
#pragma unroll
        for (int b = lane; b < kBins; b += 32) h[b] = 0;
        __syncwarp();
        for (int j = lane; j < T; j += 32) {
          const uint32_t key = order_key(row[j]);
          if ((key & pmask) == prefix) atomicAdd(&h[(key >> shift) & 0xFFu], 1);
        }
        __syncwarp();
        // lane l owns bins 255 - 8l .. 248 - 8l (descending); find the bin where
        // the count from the top first reaches rem
        int c[8], lsum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) { c[i] = h[255 - 8 * lane - i]; lsum += c[i]; }
        int incl = lsum;  // inclusive prefix over lanes 0..lane
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(full, incl, o);
          if (lane >= o) incl += y;
        }
        const int excl = incl - lsum;
        const unsigned hit = __ballot_sync(full, excl < rem && incl >= rem);
        const int src = __ffs(hit) - 1;
        int digit = 0, above = 0;
        if (lane == src) {
          int run = excl;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (run + c[i] >= rem) { digit = 255 - 8 * lane - i; above = run; break; }
            run += c[i];
          }
        }
        digit = __shfl_sync(full, digit, src);
        above = __shfl_sync(full, above, src);
        prefix |= static_cast<uint32_t>(digit) << shift;
        pmask |= 0xFFu << shift;
        rem -= above;
        __syncwarp();
      }
      const uint32_t thr = prefix;  // the k-th largest key
      const int need_eq = rem;      // how many keys equal to thr are taken (lowest tile ids first)
      int written = 0, eq_seen = 0;
      int32_t* dst = tile_index + (bh * T + t) * static_cast<size_t>(k);
      for (int base = 0; base < T; base += 32) {
        const int j = base + lane;
        const uint32_t key = j < T ? order_key(row[j]) : 0u;
        const bool is_gt = j < T && key > thr;
        const bool is_eq = j < T && key == thr;
        const unsigned eqb = __ballot_sync(full, is_eq);
        const bool sel = is_gt || (is_eq && eq_seen + __popc(eqb & lt_mask) < need_eq);
        const unsigned selb = __ballot_sync(full, sel);
        if (sel) dst[written + __popc(selb & lt_mask)] = j;
        written += __popc(selb);
        eq_seen += __popc(eqb);
      }
    }
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

  // ---- coarse[t] = sum_j p[t][j] * pooled_v[j] / l[t]
  constexpr int RPT = R / kWarps;  // query rows per thread
  const int d4 = lane;             // dims 4*d4 .. 4*d4+3
  float4 acc[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c0 = 0; c0 < tpad; c0 += kChunk) {
    __syncthreads();
    load_rows(sx, gv, c0, T, kChunk);
    __syncthreads();
#pragma unroll 4
    for (int j = 0; j < kChunk; ++j) {
      const float4 vv = *reinterpret_cast<const float4*>(sx + j * kPad + 4 * d4);
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        const float p = S[(warp * RPT + i) * tpad + c0 + j];
        acc[i].x = fmaf(p, vv.x, acc[i].x);
        acc[i].y = fmaf(p, vv.y, acc[i].y);
        acc[i].z = fmaf(p, vv.z, acc[i].z);
        acc[i].w = fmaf(p, vv.w, acc[i].w);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int r = warp * RPT + i;
    const int t = t0 + r;
    if (t < T) {
      const float inv = 1.0f / sl[r];
      float4 o = acc[i];
      o.x *= inv; o.y *= inv; o.z *= inv; o.w *= inv;
      reinterpret_cast<float4*>(coarse + (bh * T + t) * kHeadDim)[d4] = o;
    }
  }
}

int pick_rows(int tpad) {
  for (int r = 32; r >= 8; r /= 2) {
    const size_t bytes = (static_cast<size_t>(r) * tpad + static_cast<size_t>(r) * kPad +
                          static_cast<size_t>(kChunk) * kPad + r + kWarps * kBins) * sizeof(float);
    if (bytes <= kSmemBudget) return r;
  }
  return 0;
}

}  // namespace

size_t coarse_smem_bytes(const Geometry& g, int* rows_per_cta) {
  const int tpad = (g.T + kChunk - 1) / kChunk * kChunk;
  const int r = pick_rows(tpad);
  if (rows_per_cta) *rows_per_cta = r;
  if (r == 0) return 0;
  return (static_cast<size_t>(r) * tpad + static_cast<size_t>(r) * kPad +
          static_cast<size_t>(kChunk) * kPad + r + kWarps * kBins) * sizeof(float);
}

cudaError_t launch_coarse_topk(const Geometry& g, const float* pooled_q, const float* pooled_k,
                               const float* pooled_v, float* coarse, int32_t* tile_index,
                               cudaStream_t stream) {
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
        coarse_topk_kernel<32><<<grid, kThreads, smem, stream>>>(pooled_q, pooled_k, pooled_v, coarse, tile_index, g.T, g.k, tpad);
      break;
    case 16:
      e = cudaFuncSetAttribute(coarse_topk_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess)
        coarse_topk_kernel<16><<<grid, kThreads, smem, stream>>>(pooled_q, pooled_k, pooled_v, coarse, tile_index, g.T, g.k, tpad);
      break;
    default:
      e = cudaFuncSetAttribute(coarse_topk_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess)
        coarse_topk_kernel<8><<<grid, kThreads, smem, stream>>>(pooled_q, pooled_k, pooled_v, coarse, tile_index, g.T, g.k, tpad);
      break;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace vsa
