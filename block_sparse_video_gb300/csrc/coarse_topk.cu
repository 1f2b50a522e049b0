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
// shared memory. Both products run on the tensor cores with each fp32 operand
// split into a head and a remainder, a*b = hi*hi + hi*lo + lo*hi, as bf16
// m16n8k16 MMAs on bf16 hi/lo fragments (~2^-16 relative) with fp32
// accumulation:
//   * scores: every warp builds its query tiles' fragments once, in
//     registers, and streams its key columns' fragments (written once per
//     forward by frag_kernel) from L2, one 64-key chunk ahead;
//   * coarse product: the softmax pass rewrites each probability row in place
//     as A fragments (each fragment holds four keys of one row, so a row's
//     16-key segment becomes its four fragments), and every warp streams its
//     8 dims' V fragments from L2, one chunk ahead.
// Neither product loop stages through shared memory or waits at a barrier.
// Score errors of ~2^-16 relative sit far inside the 1e-3 tie band of the
// selection, which is an integer decision taken on the fp32 scores. Selection
// is a warp per row: a counting search for a threshold with exactly k scores
// at or above it, and where the row has equal scores at the cut, a radix
// select over the order-preserving integer image of the scores (four 8-bit
// digit passes with shared-memory histograms) followed by an in-order
// compaction. Both write the selected tile ids ascending and give the same
// set; results are deterministic.
#include "kernels.cuh"
#include "rank_helpers.cuh"

namespace vsa {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 64;  // key tiles per step of the product loops
constexpr size_t kSmemBudget = 220 * 1024;

// Fragment streams in global memory, per (b, h), for tpad_cap key tiles:
//   K (score B operand): uint4 {hi a, hi b, lo a, lo b} at [n-tile (8 keys)][ks
//     (16 channels)][lane], a = channels 16 ks + 2 t4, + 1 of key 8 n-tile + g,
//     b = the same + 8;
//   V (coarse-product B operand): uint4 {hi b0, hi b1, lo b0, lo b1} at [key
//     step (16 tiles)][dim tile nt (8 dims)][lane], b0 = tiles 16 ks + 2 t4, + 1
//     and b1 = the same + 8, of dim 8 nt + g.
// Both are tpad_cap x 512 bytes per (b, h); tiles past the request's T are
// zeros.
__device__ __forceinline__ size_t frag_per_bh(int tpad_cap) { return static_cast<size_t>(tpad_cap) * 32; }

template <int R>
__global__ void __launch_bounds__(kThreads, 1)
coarse_topk_kernel(const float* __restrict__ pooled_q, const uint4* __restrict__ kfrag,
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
  // Row stride: 16 floats past a multiple of 32, so that the two rows a quarter
  // warp reads together in the coarse product sit in disjoint banks.
  const int sstride = tpad_cap + 16;
  extern __shared__ __align__(16) float smem[];
  float* S = smem;                             // [R][sstride] scores, then probability fragments
  float* sl = S + R * sstride;                 // [R] softmax denominators
  int* hist = reinterpret_cast<int*>(sl + R);  // [kWarps][kBins] radix histograms (fallback select)

  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const int g = lane >> 2, t4 = lane & 3;
  const int t0 = blockIdx.x * R;
  const size_t bh = blockIdx.y;
  const float* gq = pooled_q + bh * T_cap * kHeadDim;
  const uint4* gkf = kfrag + bh * frag_per_bh(tpad_cap);
  const uint4* gvf = vfrag + bh * frag_per_bh(tpad_cap);
  const float scale = 0.08838834764831845f;  // 1/sqrt(128)
  const int rows = min(R, T - t0);           // query tiles of this CTA

  // ---- scores: warp w computes key columns 8 (w % 8) .. + 7 of each chunk for
  // row tile w / 8 (warps of a row tile that does not exist idle here)
  const int s_nt = warp % 8, s_m = warp / 8;
  if (s_m < MT) {
    // this warp's query rows 16 s_m + g and + 8 as bf16 hi/lo A fragments, built once
    uint4 aq[kHeadDim / 16][2];
#pragma unroll
    for (int ks = 0; ks < kHeadDim / 16; ++ks)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int row = 16 * s_m + g + 8 * hr;
        float2 xa = make_float2(0.f, 0.f), xb = make_float2(0.f, 0.f);
        if (row < rows) {
          const float* src = gq + static_cast<size_t>(t0 + row) * kHeadDim + 16 * ks + 2 * t4;
          xa = __ldg(reinterpret_cast<const float2*>(src));
          xb = __ldg(reinterpret_cast<const float2*>(src + 8));
        }
        uint32_t ha, la, hb, lb;
        split_bf16_pair(xa.x, xa.y, ha, la);
        split_bf16_pair(xb.x, xb.y, hb, lb);
        aq[ks][hr] = make_uint4(ha, hb, la, lb);
      }
    // the key fragments of n-tile c0 / 8 + s_nt; each slot is refilled with the
    // next chunk's fragment as soon as it has been read
    auto kf_at = [&](int c0, int ks) { return gkf + ((c0 / 8 + s_nt) * (kHeadDim / 16) + ks) * 32 + lane; };
    uint4 kf[kHeadDim / 16];
#pragma unroll
    for (int ks = 0; ks < kHeadDim / 16; ++ks) kf[ks] = __ldg(kf_at(0, ks));
    const int r0 = 16 * s_m + g;
    for (int c0 = 0; c0 < tpad; c0 += kChunk) {
      const bool more = c0 + kChunk < tpad;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < kHeadDim / 16; ++ks) {
        mma_bf16x3(acc, aq[ks][0], aq[ks][1], kf[ks]);
        if (more) kf[ks] = __ldg(kf_at(c0 + kChunk, ks));
      }
      const int col = c0 + 8 * s_nt + 2 * t4;
      if (r0 < R) *reinterpret_cast<float2*>(S + r0 * sstride + col) = make_float2(acc[0] * scale, acc[1] * scale);
      if (r0 + 8 < R)
        *reinterpret_cast<float2*>(S + (r0 + 8) * sstride + col) = make_float2(acc[2] * scale, acc[3] * scale);
    }
  }
  // this warp's first V fragments, in flight during the selection
  static_assert(kWarps * 8 == kHeadDim, "one 8-dim column tile per warp");
  auto vf_at = [&](int c0, int ks) { return gvf + ((c0 / 16 + ks) * (kHeadDim / 8) + warp) * 32 + lane; };
  uint4 vf[kChunk / 16];
#pragma unroll
  for (int ks = 0; ks < kChunk / 16; ++ks) vf[ks] = __ldg(vf_at(0, ks));
  __syncthreads();

  // ---- per row: top-k selection, then softmax written back as A fragments
  const unsigned full = 0xffffffffu;
  for (int r = warp; r < R; r += kWarps) {
    float* row = S + r * sstride;
    const int t = t0 + r;
    // key columns past T (zero-padded keys) are never selected and carry no mass
    for (int j = T + lane; j < tpad; j += 32) row[j] = -INFINITY;
    __syncwarp();
    if (t < T)
      warp_select_topk_count(row, T, tpad, k, hist + warp * kBins,
                             tile_index + (bh * T_cap + t) * static_cast<size_t>(k_cap), lane);
    float m = -INFINITY;
    for (int j = lane; j < T; j += 32) m = fmaxf(m, row[j]);
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(full, m, o));
    // lane-owned 16-key segments: p = exp(s - m), then the segment's four
    // fragments {hi a, hi b, lo a, lo b} (a = keys 2 t4, 2 t4 + 1; b = + 8)
    // in place of its 16 scores
    float l = 0.f;
    for (int seg = lane; seg < tpad / 16; seg += 32) {
      float4* q4 = reinterpret_cast<float4*>(row + 16 * seg);
      float p[16];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 x = q4[i];
        p[4 * i] = expf(x.x - m);
        p[4 * i + 1] = expf(x.y - m);
        p[4 * i + 2] = expf(x.z - m);
        p[4 * i + 3] = expf(x.w - m);
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) l += p[i];
      uint4* f4 = reinterpret_cast<uint4*>(q4);
#pragma unroll
      for (int tt = 0; tt < 4; ++tt) {
        uint32_t ha, la, hb, lb;
        split_bf16_pair(p[2 * tt], p[2 * tt + 1], ha, la);
        split_bf16_pair(p[2 * tt + 8], p[2 * tt + 9], hb, lb);
        f4[tt] = make_uint4(ha, hb, la, lb);
      }
    }
    for (int o = 16; o; o >>= 1) l += __shfl_xor_sync(full, l, o);
    if (lane == 0) sl[r] = l;
  }
  __syncthreads();

  // ---- coarse[t] = sum_j p[t][j] * pooled_v[j] / l[t]; warp w owns dims 8w .. 8w + 7
  float o[MT][4];
#pragma unroll
  for (int mm = 0; mm < MT; ++mm) o[mm][0] = o[mm][1] = o[mm][2] = o[mm][3] = 0.f;
  const uint32_t s_base = static_cast<uint32_t>(__cvta_generic_to_shared(S));
  for (int c0 = 0; c0 < tpad; c0 += kChunk) {
    const bool more = c0 + kChunk < tpad;
#pragma unroll
    for (int ks = 0; ks < kChunk / 16; ++ks) {
#pragma unroll
      for (int mm = 0; mm < MT; ++mm) {
        const int ra = 16 * mm + g, rb = ra + 8;
        const uint32_t off = static_cast<uint32_t>((c0 + 16 * ks + 4 * t4) * 4);
        const uint4 fa = ra < R ? lds128(s_base + static_cast<uint32_t>(ra * sstride * 4) + off) : make_uint4(0, 0, 0, 0);
        const uint4 fb = rb < R ? lds128(s_base + static_cast<uint32_t>(rb * sstride * 4) + off) : make_uint4(0, 0, 0, 0);
        mma_bf16x3(o[mm], fa, fb, vf[ks]);
      }
      if (more) vf[ks] = __ldg(vf_at(c0 + kChunk, ks));
    }
  }
#pragma unroll
  for (int mm = 0; mm < MT; ++mm)
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int r = 16 * mm + g + 8 * half;
      if (r < rows) {
        const float inv = 1.0f / sl[r];
        float* dst = coarse + (bh * T_cap + t0 + r) * kHeadDim;
        *reinterpret_cast<float2*>(dst + 8 * warp + 2 * t4) = make_float2(o[mm][2 * half] * inv, o[mm][2 * half + 1] * inv);
      }
    }
}

// The pooled K and V of every (b, h) as the fragment streams described above:
// entries [0, n) are K fragments, [n, 2n) V fragments, n = B H tpad_cap 32.
__global__ void __launch_bounds__(256)
frag_kernel(const float* __restrict__ pooled_k, const float* __restrict__ pooled_v, uint4* __restrict__ kfrag,
            uint4* __restrict__ vfrag, Geometry cap, DeviceLengths dl, int tpad_cap) {
  const DynGeom dg = dyn_geom(cap, dl);
  if (!dg.valid) return;
  const size_t per_bh = frag_per_bh(tpad_cap);
  const size_t n = per_bh * cap.B * cap.H;
  size_t idx = static_cast<size_t>(blockIdx.x) * 256 + threadIdx.x;
  if (idx >= 2 * n) return;
  const bool is_v = idx >= n;
  if (is_v) idx -= n;
  const size_t bh = idx / per_bh;
  const int within = static_cast<int>(idx % per_bh);
  const int ln = within % 32, gg = ln / 4, tt = ln % 4;
  uint32_t ha, la, hb, lb;
  if (!is_v) {
    const int ks = (within / 32) % (kHeadDim / 16), nt = within / 256;
    const int key = 8 * nt + gg, ch = 16 * ks + 2 * tt;
    float2 a = make_float2(0.f, 0.f), b = make_float2(0.f, 0.f);
    if (key < dg.T) {
      const float* src = pooled_k + (bh * cap.T + key) * kHeadDim + ch;
      a = __ldg(reinterpret_cast<const float2*>(src));
      b = __ldg(reinterpret_cast<const float2*>(src + 8));
    }
    split_bf16_pair(a.x, a.y, ha, la);
    split_bf16_pair(b.x, b.y, hb, lb);
    kfrag[idx] = make_uint4(ha, hb, la, lb);
  } else {
    const int nt = (within / 32) % (kHeadDim / 8), ks = within / 512;
    const int dim = 8 * nt + gg, k0 = 16 * ks + 2 * tt;
    const float* src = pooled_v + bh * cap.T * kHeadDim + dim;
    auto val = [&](int key) { return key < dg.T ? __ldg(src + static_cast<size_t>(key) * kHeadDim) : 0.f; };
    split_bf16_pair(val(k0), val(k0 + 1), ha, la);
    split_bf16_pair(val(k0 + 8), val(k0 + 9), hb, lb);
    vfrag[idx] = make_uint4(ha, hb, la, lb);
  }
}

size_t smem_for(int r, int tpad) {
  return (static_cast<size_t>(r) * (tpad + 16) + r + kWarps * kBins) * sizeof(float);
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
  return 2 * static_cast<size_t>(g.B) * g.H * tpad * 512;  // K and V: 128 channels x (hi + lo) x 2 bytes per tile
}

cudaError_t launch_coarse_topk(const Geometry& g, const float* pooled_q, const float* pooled_k,
                               const float* pooled_v, float* coarse, int32_t* tile_index, void* vfrag,
                               const DeviceLengths& dl, cudaStream_t stream) {
  int r = 0;
  const size_t smem = coarse_smem_bytes(g, &r);
  if (r == 0) return cudaErrorInvalidValue;
  const int tpad = (g.T + kChunk - 1) / kChunk * kChunk;
  const size_t n_frag = coarse_vfrag_bytes(g) / 32;  // uint4 entries of each stream
  uint4* kf = static_cast<uint4*>(vfrag);
  const uint4* vf = kf + n_frag;
  frag_kernel<<<static_cast<unsigned>((2 * n_frag + 255) / 256), 256, 0, stream>>>(pooled_k, pooled_v, kf,
                                                                                 kf + n_frag, g, dl, tpad);
  dim3 grid((g.T + r - 1) / r, g.B * g.H);
  cudaError_t e = cudaSuccess;
  switch (r) {
    case 32:
      e = cudaFuncSetAttribute(coarse_topk_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess)
        coarse_topk_kernel<32><<<grid, kThreads, smem, stream>>>(pooled_q, kf, vf, coarse, tile_index, g, dl, tpad);
      break;
    case 16:
      e = cudaFuncSetAttribute(coarse_topk_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess)
        coarse_topk_kernel<16><<<grid, kThreads, smem, stream>>>(pooled_q, kf, vf, coarse, tile_index, g, dl, tpad);
      break;
    default:
      e = cudaFuncSetAttribute(coarse_topk_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess)
        coarse_topk_kernel<8><<<grid, kThreads, smem, stream>>>(pooled_q, kf, vf, coarse, tile_index, g, dl, tpad);
      break;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace vsa
