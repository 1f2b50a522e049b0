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
// shared memory. Pooled K (then V) tiles stream through a smem chunk of 64
// rows. Both products run on the tensor cores with each fp32 operand split
// into a head and a remainder, a*b = hi*hi + hi*lo + lo*hi:
//   * both as bf16 m16n8k16 MMAs on bf16 hi/lo fragments (~2^-16 relative),
//     with fp32 accumulation;
//   * scores: every warp builds its query tile's fragments once, in
//     registers, and each K chunk is converted once, at staging;
//   * coarse product: the pooled V comes as fragments from vfrag_kernel, and
//     each chunk's probabilities are converted once into fragments shared by
//     the warps.
// Score errors of ~2^-16 relative sit far inside the 1e-3 tie band of the
// selection, which is an integer decision taken on the fp32 scores. Selection is a warp-per-row radix select over the
// order-preserving integer image of the fp32 scores: four passes of 8-bit
// digits, each a 256-bin shared-memory histogram of the keys that still match
// the digits fixed so far, then an in-order compaction that writes the selected
// tile ids ascending. Results are deterministic: the histograms are counts, and
// the compaction follows tile order.
#include "kernels.cuh"
#include "rank_helpers.cuh"

namespace vsa {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 64;            // pooled tiles staged per step
constexpr int kVPad = kHeadDim + 8;   // staging area: 64 rows of kVPad floats (K fragments or V fragments)
constexpr int kVfPerThread = kChunk / 16 * 16 * 32 / kThreads;  // V fragment uint4s per thread per chunk
constexpr size_t kSmemBudget = 220 * 1024;

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

// The staged K chunk (64 pooled key tiles x 128 channels, from the register
// prefetch) as bf16 hi/lo B fragments of m16n8k16: uint4 {hi a, hi b, lo a,
// lo b} at [n-tile (8 keys)][ks (16 channels)][lane], a = channels 2 t4, 2 t4 + 1
// of key g of the n-tile, b = the same + 8.
__device__ __forceinline__ void stash_chunk_frag(uint32_t* dst, const float4 (&pre)[kChunkF4PerThread]) {
#pragma unroll
  for (int i = 0; i < kChunkF4PerThread; ++i) {
    const int e = threadIdx.x + i * kThreads;
    const int r = e / (kHeadDim / 4), c4 = e % (kHeadDim / 4);  // key row, channels 4 c4 .. 4 c4 + 3
    const int ks = c4 / 4, half = (c4 % 4) / 2, t4 = 2 * (c4 % 2);
    uint32_t h0, l0, h1, l1;
    split_bf16_pair(pre[i].x, pre[i].y, h0, l0);
    split_bf16_pair(pre[i].z, pre[i].w, h1, l1);
    uint32_t* w = dst + (((r / 8) * (kHeadDim / 16) + ks) * 32 + 4 * (r % 8) + t4) * 4;
    w[half] = h0;
    w[2 + half] = l0;
    w[4 + half] = h1;
    w[4 + 2 + half] = l1;
  }
}

template <int R>
__global__ void __launch_bounds__(kThreads, 1)
coarse_topk_kernel(const float* __restrict__ pooled_q, const float* __restrict__ pooled_k,
                   const uint4* __restrict__ vfrag, float* __restrict__ coarse,
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
  float* sx = S + R * sstride;              // K chunk (bf16 hi/lo fragments) or V chunk [kChunk][kVPad]
  float* sl = sx + kChunk * kVPad;          // [R] softmax denominators
  int* hist = reinterpret_cast<int*>(sl + R);  // [kWarps][kBins] radix histograms

  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const int g = lane >> 2, t4 = lane & 3;
  const int t0 = blockIdx.x * R;
  const size_t bh = blockIdx.y;
  const float* gq = pooled_q + bh * T_cap * kHeadDim;
  const float* gk = pooled_k + bh * T_cap * kHeadDim;
  // pooled V as bf16 hi/lo B fragments: [tpad_cap / 16 key steps][16 dim tiles][32 lanes]
  const uint4* gvf = vfrag + bh * (static_cast<size_t>(tpad_cap) / 16) * 16 * 32;
  const float scale = 0.08838834764831845f;  // 1/sqrt(128)
  const int rows = min(R, T - t0);           // query tiles of this CTA

  // ---- scores: warp w computes key columns 8 (w % 8) .. + 7 of each chunk for
  // row tile w / 8 (warps of a row tile that does not exist idle here)
  float4 pre[kChunkF4PerThread];
  fetch_chunk(pre, gk, 0, T);
  const int s_nt = warp % 8, s_m = warp / 8;
  // this warp's query rows 16 s_m + g and + 8 as bf16 hi/lo A fragments, built once
  uint4 aq[kHeadDim / 16][2];
#pragma unroll
  for (int ks = 0; ks < kHeadDim / 16; ++ks)
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int row = 16 * s_m + g + 8 * hr;
      float2 xa = make_float2(0.f, 0.f), xb = make_float2(0.f, 0.f);
      if (s_m < MT && row < rows) {
        const float* src = gq + static_cast<size_t>(t0 + row) * kHeadDim + 16 * ks + 2 * t4;
        xa = __ldg(reinterpret_cast<const float2*>(src));
        xb = __ldg(reinterpret_cast<const float2*>(src + 8));
      }
      uint32_t ha, la, hb, lb;
      split_bf16_pair(xa.x, xa.y, ha, la);
      split_bf16_pair(xb.x, xb.y, hb, lb);
      aq[ks][hr] = make_uint4(ha, hb, la, lb);
    }
  uint32_t* kfrag = reinterpret_cast<uint32_t*>(sx);
  const uint32_t kb = static_cast<uint32_t>(__cvta_generic_to_shared(sx)) +
                      ((s_nt * (kHeadDim / 16)) * 32 + lane) * 16;
  for (int c0 = 0; c0 < tpad; c0 += kChunk) {
    __syncthreads();
    stash_chunk_frag(kfrag, pre);
    __syncthreads();
    if (c0 + kChunk < tpad) fetch_chunk(pre, gk, c0 + kChunk, T);  // in flight during the products
    if (s_m < MT) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < kHeadDim / 16; ++ks) mma_bf16x3(acc, aq[ks][0], aq[ks][1], lds128(kb + ks * 512));
      const int col = c0 + 8 * s_nt + 2 * t4;
      const int r0 = 16 * s_m + g;
      if (r0 < R) *reinterpret_cast<float2*>(S + r0 * sstride + col) = make_float2(acc[0] * scale, acc[1] * scale);
      if (r0 + 8 < R)
        *reinterpret_cast<float2*>(S + (r0 + 8) * sstride + col) = make_float2(acc[2] * scale, acc[3] * scale);
    }
  }
  uint4 vpre[kVfPerThread];
  auto fetch_v = [&](int c0) {
#pragma unroll
    for (int i = 0; i < kVfPerThread; ++i) vpre[i] = __ldg(gvf + (c0 / 16) * 512 + threadIdx.x + i * kThreads);
  };
  fetch_v(0);  // first V chunk, in flight during the selection
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
  static_assert(MT * 4 * 2 * 32 * 16 <= kWarps * kBins * 4, "probability fragments fit over the histograms");
  uint4* vsm = reinterpret_cast<uint4*>(sx);    // this chunk's V fragments [4 key steps][16 dim tiles][32]
  uint4* psm = reinterpret_cast<uint4*>(hist);  // its probability fragments [MT][4 key steps][2][32]
  float o[MT][4];
#pragma unroll
  for (int m = 0; m < MT; ++m) o[m][0] = o[m][1] = o[m][2] = o[m][3] = 0.f;
  for (int c0 = 0; c0 < tpad; c0 += kChunk) {
    __syncthreads();  // the selection, or the previous chunk's products, are done
#pragma unroll
    for (int i = 0; i < kVfPerThread; ++i) vsm[threadIdx.x + i * kThreads] = vpre[i];
    // probabilities of rows 16 m + g (+ 8) and keys c0 + 16 ks + 2 t4 .. (+ 8) as A fragments
    for (int idx = tid; idx < MT * 4 * 2 * 32; idx += kThreads) {
      const int ln = idx % 32, hr = (idx / 32) % 2, ks = (idx / 64) % 4, m = idx / 256;
      const int row = 16 * m + ln / 4 + 8 * hr;
      const int key = c0 + 16 * ks + 2 * (ln % 4);
      float2 xa = make_float2(0.f, 0.f), xb = make_float2(0.f, 0.f);
      if (row < R) {
        xa = *reinterpret_cast<const float2*>(S + row * sstride + key);
        xb = *reinterpret_cast<const float2*>(S + row * sstride + key + 8);
      }
      uint32_t ha, la, hb, lb;
      split_bf16_pair(xa.x, xa.y, ha, la);
      split_bf16_pair(xb.x, xb.y, hb, lb);
      psm[idx] = make_uint4(ha, hb, la, lb);
    }
    __syncthreads();
    if (c0 + kChunk < tpad) fetch_v(c0 + kChunk);
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      const uint4 bf = vsm[(ks * 16 + warp) * 32 + lane];
#pragma unroll
      for (int m = 0; m < MT; ++m)
        mma_bf16x3(o[m], psm[((m * 4 + ks) * 2) * 32 + lane], psm[((m * 4 + ks) * 2 + 1) * 32 + lane], bf);
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

// The pooled V of every (b, h) as bf16 hi/lo B fragments of m16n8k16 for the
// coarse product: uint4 {hi b0, hi b1, lo b0, lo b1} at [key step ks (16
// tiles)][dim tile nt (8 dims)][lane], b0 = tiles 16 ks + 2 t4, + 1 and b1 =
// the same + 8, of dim 8 nt + g. Tiles past the request's T are zeros.
__global__ void __launch_bounds__(256)
vfrag_kernel(const float* __restrict__ pooled_v, uint4* __restrict__ vfrag, Geometry cap, DeviceLengths dl,
             int tpad_cap) {
  const DynGeom dg = dyn_geom(cap, dl);
  if (!dg.valid) return;
  const size_t per_bh = static_cast<size_t>(tpad_cap) / 16 * 16 * 32;
  const size_t idx = static_cast<size_t>(blockIdx.x) * 256 + threadIdx.x;
  if (idx >= per_bh * cap.B * cap.H) return;
  const size_t bh = idx / per_bh;
  const int within = static_cast<int>(idx % per_bh);
  const int ln = within % 32, nt = (within / 32) % 16, ks = within / 512;
  const int dim = 8 * nt + ln / 4, k0 = 16 * ks + 2 * (ln % 4);
  const float* src = pooled_v + bh * cap.T * kHeadDim + dim;
  auto val = [&](int key) { return key < dg.T ? __ldg(src + static_cast<size_t>(key) * kHeadDim) : 0.f; };
  uint32_t ha, la, hb, lb;
  split_bf16_pair(val(k0), val(k0 + 1), ha, la);
  split_bf16_pair(val(k0 + 8), val(k0 + 9), hb, lb);
  vfrag[idx] = make_uint4(ha, hb, la, lb);
}

size_t smem_for(int r, int tpad) {
  const int mt = r >= 16 ? r / 16 : 1;
  (void)mt;
  return (static_cast<size_t>(r) * (tpad + 4) + static_cast<size_t>(kChunk) * kVPad + r + kWarps * kBins) *
         sizeof(float);
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

size_t coarse_vfrag_bytes(const Geometry& g) {
  const size_t tpad = (g.T + kChunk - 1) / kChunk * kChunk;
  return static_cast<size_t>(g.B) * g.H * tpad * 512;  // 128 dims x (hi + lo) x 2 bytes per tile
}

cudaError_t launch_coarse_topk(const Geometry& g, const float* pooled_q, const float* pooled_k,
                               const float* pooled_v, float* coarse, int32_t* tile_index, void* vfrag,
                               const DeviceLengths& dl, cudaStream_t stream) {
  int r = 0;
  const size_t smem = coarse_smem_bytes(g, &r);
  if (r == 0) return cudaErrorInvalidValue;
  const int tpad = (g.T + kChunk - 1) / kChunk * kChunk;
  {
    const size_t n = coarse_vfrag_bytes(g) / 16;
    vfrag_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(pooled_v, static_cast<uint4*>(vfrag), g,
                                                                           dl, tpad);
  }
  const uint4* vf = static_cast<const uint4*>(vfrag);
  dim3 grid((g.T + r - 1) / r, g.B * g.H);
  cudaError_t e = cudaSuccess;
  switch (r) {
    case 32:
      e = cudaFuncSetAttribute(coarse_topk_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess)
        coarse_topk_kernel<32><<<grid, kThreads, smem, stream>>>(pooled_q, pooled_k, vf, coarse, tile_index, g, dl, tpad);
      break;
    case 16:
      e = cudaFuncSetAttribute(coarse_topk_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess)
        coarse_topk_kernel<16><<<grid, kThreads, smem, stream>>>(pooled_q, pooled_k, vf, coarse, tile_index, g, dl, tpad);
      break;
    default:
      e = cudaFuncSetAttribute(coarse_topk_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess)
        coarse_topk_kernel<8><<<grid, kThreads, smem, stream>>>(pooled_q, pooled_k, vf, coarse, tile_index, g, dl, tpad);
      break;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace vsa
