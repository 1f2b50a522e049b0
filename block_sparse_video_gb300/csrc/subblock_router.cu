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
// their R x T block scores in shared memory.
//
// Operands. The sub-pool kernel leaves every sub-block mean split into bf16
// hi + lo (x ~ hi + lo, ~2^-16 relative), already in mma.sync m16n8k16
// fragment order. So the products are bf16 tensor-core MMAs,
//   q . k ~ hi.hi + hi.lo + lo.hi,
// with fp32 accumulation. That is about 2^-16 relative error on each logit,
// against the 1e-3 tie band of the selection. No operand is converted in the
// inner loop. The CTA's query fragments (R/2 x 4 KB) come in one bulk copy,
// and each warp keeps its own m16 tile's fragments in registers.
// Key fragments stream through a two-slot ring of CH-sub-row chunks, filled by
// bulk copies that complete on mbarriers.
//
// The sub-pool kernel permutes sub-rows inside each group of 4 blocks (see
// pool.cu). A warp's tile is one m16 tile (4 query blocks) by two n8 tiles
// (4 key blocks), and each lane then holds 8 of the 16 logits of one (query
// block, key block) pair; lane ^ 16 holds the other 8. The log-sum-exp is
// lane-local plus one shuffle for the maximum and one for the sum. It runs in
// log2 units (ex2 and lg2 on the MUFU pipe), which ranks in the same order.
// The coarse kernel's warp-per-row selection then picks each row's top k: the
// counting threshold search, with the radix select where scores tie at the
// cut. With device lengths the router scores the request's tiles only and
// writes its selections at the plan's strides.
#include <cmath>

#include "kernels.cuh"
#include "ptx.cuh"
#include "rank_helpers.cuh"

namespace vsa {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kTile8Bytes = 8 * 32 * 16;          // fragments of 8 sub-rows x 128 channels: 4 KB
constexpr size_t kSmemBudget = 220 * 1024;
constexpr int kSub = 16;                          // tokens per sub-block
constexpr unsigned int kDetailRouterQ = 0x700, kDetailRouterK = 0x710;

// log2(number of valid tokens of sub-block s), -inf for an empty one
__device__ __forceinline__ float lg_count(int s, int Lv) {
  const int n = min(kSub, Lv - kSub * s);
  return n >= kSub ? 4.f : (n > 0 ? __log2f(static_cast<float>(n)) : -INFINITY);
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// R query blocks per CTA (R/4 m16 tiles), CH key sub-rows per chunk (CH/16
// n-pairs). Warp w takes m16 tile w / (CH/16) and n-pair w % (CH/16) of each
// chunk; warps past R/4 m16 tiles idle.
template <int R, int CH>
__global__ void __launch_bounds__(kThreads, 1)
subblock_router_kernel(const uint4* __restrict__ frag_q, const uint4* __restrict__ frag_k,
                       int32_t* __restrict__ tile_index, unsigned int* err, Geometry cap, DeviceLengths dl,
                       int spad) {
  constexpr int MT = R / 4;
  constexpr int NP = CH / 16;
  constexpr int kChunkBytes = CH / 8 * kTile8Bytes;
  // The request's tiles (the plan's own, or the device lengths'); the layouts
  // (fragment rows spad, selections [T_cap][k_cap], shared-memory rows) are
  // the plan's.
  const DynGeom dg = dyn_geom(cap, dl);
  if (!dg.valid) {
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *dl.invalid = 1u;
    return;
  }
  const int T = dg.T, Lv = dg.Lv, k = dg.k;
  if (static_cast<int>(blockIdx.x) * R >= T) return;  // uniform per CTA, before any copy
  const int bstride = spad / 4 + 4;                 // block-score row stride (floats)
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* s_kbuf = smem;                           // [2][kChunkBytes] key fragments
  uint8_t* s_q = smem + 2 * kChunkBytes;            // [R/2 tile8][kTile8Bytes] query fragments
  float* S = reinterpret_cast<float*>(s_q + (R / 2) * kTile8Bytes);  // [R][bstride] block scores
  uint64_t* bars = reinterpret_cast<uint64_t*>(S + R * bstride);     // q, k slot 0, k slot 1
  int* hist = reinterpret_cast<int*>(smem);         // [kWarps][kBins], over the key ring after the products

  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const int g = lane >> 2, t4 = lane & 3;
  const int q0 = blockIdx.x * R;                    // first query block of this CTA
  const size_t bh = blockIdx.y;
  const size_t tiles_per_bh = static_cast<size_t>(spad) / 8;
  const uint8_t* gq = reinterpret_cast<const uint8_t*>(frag_q + bh * tiles_per_bh * 256);
  const uint8_t* gk = reinterpret_cast<const uint8_t*>(frag_k + bh * tiles_per_bh * 256);
  const float scale_log2 = 0.08838834764831845f * 1.4426950408889634f;  // log2(e) / sqrt(128)
  const int n_chunks = (4 * T + CH - 1) / CH;       // chunks holding the request's key sub-rows
  const uint32_t bar_q = smem_u32(bars), bar_k0 = smem_u32(bars + 1);

  if (tid == 0) {
    mbar_init(bar_q, 1);
    mbar_init(bar_k0, 1);
    mbar_init(bar_k0 + 8, 1);
    fence_barrier_init();
  }
  __syncthreads();
  int issued = 0;  // key chunks whose copy thread 0 has issued
  if (tid == 0) {
    // query sub-rows 4 q0 .. 4 q0 + 4R: R/2 tile8s, contiguous (within spad for every CTA)
    mbar_arrive_expect_tx(bar_q, (R / 2) * kTile8Bytes);
    bulk_load(smem_u32(s_q), gq + static_cast<size_t>(q0 / 2) * kTile8Bytes, (R / 2) * kTile8Bytes, bar_q);
    for (; issued < 2 && issued < n_chunks; ++issued) {
      mbar_arrive_expect_tx(bar_k0 + 8 * issued, kChunkBytes);
      bulk_load(smem_u32(s_kbuf + issued * kChunkBytes), gk + static_cast<size_t>(issued) * kChunkBytes,
                kChunkBytes, bar_k0 + 8 * issued);
    }
  }

  const int m = warp / NP, np = warp % NP;
  const bool has_work = m < MT;
  // this lane's pair: query block 4 m + (g & 3) of the CTA, key block 4 np + t4 of each chunk;
  // its query sub-blocks are a0 = 2 (g >> 2) (row g) and a0 + 1 (row g + 8)
  const int qsub = 4 * (q0 + 4 * m + (g & 3)) + 2 * (g >> 2);
  const float lq0 = lg_count(qsub, Lv), lq1 = lg_count(qsub + 1, Lv);
  const uint32_t qa = smem_u32(s_q + (2 * m) * kTile8Bytes) + lane * 16;

  bool ok = mbar_wait(bar_q, 0, err, kDetailRouterQ);
  // this warp's m16 tile is the same for every chunk: its A fragments stay in registers
  uint4 aq[kHeadDim / 16][2];
#pragma unroll
  for (int ks = 0; ks < kHeadDim / 16; ++ks) {
    aq[ks][0] = (ok && has_work) ? lds128(qa + ks * 512) : make_uint4(0, 0, 0, 0);                // rows g
    aq[ks][1] = (ok && has_work) ? lds128(qa + kTile8Bytes + ks * 512) : make_uint4(0, 0, 0, 0);  // rows g + 8
  }
  for (int c = 0; c < n_chunks; ++c) {
    const int slot = c & 1;
    ok = ok && mbar_wait(bar_k0 + 8 * slot, (c >> 1) & 1, err, kDetailRouterK);
    if (ok && has_work) {
      const int kblk = c * (CH / 4) + 4 * np + t4;  // key block of this lane
      float lk[4];
#pragma unroll
      for (int sb = 0; sb < 4; ++sb) lk[sb] = lg_count(4 * kblk + sb, Lv);
      const uint32_t kb = smem_u32(s_kbuf + slot * kChunkBytes + (2 * np) * kTile8Bytes) + lane * 16;
      float acc[2][4];
#pragma unroll
      for (int ni = 0; ni < 2; ++ni) acc[ni][0] = acc[ni][1] = acc[ni][2] = acc[ni][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < kHeadDim / 16; ++ks) {
        const uint4 t0 = aq[ks][0], t1 = aq[ks][1];
#pragma unroll
        for (int ni = 0; ni < 2; ++ni) {
          const uint4 bf = lds128(kb + ni * kTile8Bytes + ks * 512);  // {hi b0, hi b1, lo b0, lo b1}
          mma_bf16x3(acc[ni], t0, t1, bf);
        }
      }
      // acc[ni][e] (e < 2): row g, key sub-block 2 ni + e; acc[ni][2 + e]: row g + 8
      float x[8];
#pragma unroll
      for (int ni = 0; ni < 2; ++ni)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          x[4 * ni + e] = fmaf(acc[ni][e], scale_log2, lq0 + lk[2 * ni + e]);
          x[4 * ni + 2 + e] = fmaf(acc[ni][2 + e], scale_log2, lq1 + lk[2 * ni + e]);
        }
      float mx = x[0];
#pragma unroll
      for (int i = 1; i < 8; ++i) mx = fmaxf(mx, x[i]);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      float sum = 0.f;
      if (mx > -INFINITY) {
#pragma unroll
        for (int i = 0; i < 8; ++i) sum += ex2(x[i] - mx);
      }
      sum += __shfl_xor_sync(0xffffffffu, sum, 16);
      if (g < 4)
        S[(4 * m + g) * bstride + kblk] = mx > -INFINITY ? mx + lg2(sum) : -INFINITY;
    }
    __syncthreads();  // every warp is done with this slot
    if (tid == 0 && ok && c + 2 < n_chunks) {
      mbar_arrive_expect_tx(bar_k0 + 8 * slot, kChunkBytes);
      bulk_load(smem_u32(s_kbuf + slot * kChunkBytes), gk + static_cast<size_t>(c + 2) * kChunkBytes,
                kChunkBytes, bar_k0 + 8 * slot);
      ++issued;
    }
  }
  if (!__syncthreads_and(ok)) {
    // gave up: let the copies already issued land before the CTA ends. Thread 0
    // issued them all; the last two chunks are the latest phase of each slot.
    if (tid == 0) {
      mbar_wait_drain(bar_q, 0, kWaitLimitNs);
      for (int c = max(0, issued - 2); c < issued; ++c)
        mbar_wait_drain(bar_k0 + 8 * (c & 1), (c >> 1) & 1, kWaitLimitNs);
    }
    return;
  }

  // Key blocks T .. n_chunks * CH / 4 - 1 hold only empty sub-blocks and
  // scored -inf above, as the counting select requires of a row's padding.
  for (int r = warp; r < R; r += kWarps)
    if (q0 + r < T)
      warp_select_topk_count(S + r * bstride, T, n_chunks * CH / 4, k, hist + warp * kBins,
                             tile_index + (bh * cap.T + q0 + r) * static_cast<size_t>(cap.k), lane);
}

int sub_pad(int T) { return (4 * T + 127) / 128 * 128; }  // as subblock_rows_padded

// chunk length for R query blocks per CTA: enough n-pairs to give each of the 16 warps a tile
int chunk_for(int r) { return r == 16 ? 64 : 128; }

size_t smem_for(int r, int spad) {
  return 2 * static_cast<size_t>(chunk_for(r) / 8) * kTile8Bytes + static_cast<size_t>(r / 2) * kTile8Bytes +
         static_cast<size_t>(r) * (spad / 4 + 4) * sizeof(float) + 4 * sizeof(uint64_t);
}

int pick_rows(int spad) {
  for (int r = 16; r >= 4; r /= 2)
    if (smem_for(r, spad) <= kSmemBudget) return r;
  return 0;
}

template <int R, int CH>
cudaError_t launch_rows(const Geometry& g, const void* frag_q, const void* frag_k, int32_t* tile_index,
                        unsigned int* err, const DeviceLengths& dl, size_t smem, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(subblock_router_kernel<R, CH>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid((g.T + R - 1) / R, g.B * g.H);
  subblock_router_kernel<R, CH><<<grid, kThreads, smem, stream>>>(static_cast<const uint4*>(frag_q),
                                                                  static_cast<const uint4*>(frag_k), tile_index,
                                                                  err, g, dl, sub_pad(g.T));
  return cudaGetLastError();
}

}  // namespace

size_t subblock_router_smem_bytes(const Geometry& g, int* rows_per_cta) {
  const int r = pick_rows(sub_pad(g.T));
  if (rows_per_cta) *rows_per_cta = r;
  return r ? smem_for(r, sub_pad(g.T)) : 0;
}

cudaError_t launch_subblock_router(const Geometry& g, const void* frag_q, const void* frag_k,
                                   int32_t* tile_index, unsigned int* err, const DeviceLengths& dl,
                                   cudaStream_t stream) {
  int r = 0;
  const size_t smem = subblock_router_smem_bytes(g, &r);
  switch (r) {
    case 16: return launch_rows<16, 64>(g, frag_q, frag_k, tile_index, err, dl, smem, stream);
    case 8: return launch_rows<8, 128>(g, frag_q, frag_k, tile_index, err, dl, smem, stream);
    case 4: return launch_rows<4, 128>(g, frag_q, frag_k, tile_index, err, dl, smem, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace vsa
