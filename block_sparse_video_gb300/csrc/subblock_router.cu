// SubBlock router: the block-sparse selection of the SGLang Diffusion benchmark page (MiniMax-H3 on 8x H200),
// section "How SubBlock Sparse Attention Works". Each 64-token
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
// A CTA owns R query blocks (N = 4R query sub-rows) of one (batch, head) and
// keeps their R x T block scores in shared memory.
//
// Products on the tcgen05 tensor cores. The sub-pool kernel leaves every
// sub-block mean split into bf16 hi + lo rows (x ~ hi + lo, ~2^-16
// relative), so q . k ~ hi.hi + hi.lo + lo.hi: three bf16 MMAs accumulating
// in fp32 in TMEM, about 2^-16 relative error on each logit against the 1e-3
// tie band of the selection. The product is transposed, as for the fine
// kernel's scores:
//   L^T[128 key sub-rows x N query sub-rows] = K_chunk . Q^T     (M = 128)
// so a TMEM lane holds one key sub-row and a column one query sub-row.
//
// Warp roles (E = N / 4 score warps, then two more):
//   * warp E loads by TMA (four issuing lanes, one 8 KB box each) the CTA's
//     query rows (hi and lo, once) and the key chunks (each chunk's hi rows,
//     then its lo rows) through a 3-stage ring of 32 KB;
//   * warps E + 1 and E + 2 issue the MMAs, converged with one elected lane
//     each: every chunk's 24 products split between them, each into its own
//     accumulator of N columns (two interleaving issuers keep the tensor pipe
//     busy where one leaves it idle between N = 64 MMAs); warp E + 1 owns TMEM
//     (two such accumulator pairs, taken by chunk in turn);
//   * warps 0 .. E - 1 read each accumulator pair (warp w: TMEM lanes 32 (w %
//     4) .. + 31, the 16 columns of group w / 4: 4 query blocks), add its two
//     halves and fold them into
//     block scores, in log2 units (ex2 and lg2 on the MUFU pipe, which ranks
//     in the same order). Per query block, the 4 lanes of a key block (lanes
//     4j .. 4j + 3, one key sub-row each) first agree on the maximum logit
//     (two shuffle steps), then each sums 2^(x - max) over its 4 query
//     sub-rows and the sums meet in two more shuffle steps: no branch, and
//     an all-empty block (every x = -inf) ends at -inf.
// The same warps then pick each row's top k with the coarse kernel's
// selection: the counting threshold search, with the radix select where
// scores tie at the cut. With device lengths the router scores the
// request's tiles only and writes its selections at the plan's strides.
#include <cmath>

#include "kernels.cuh"
#include "ptx.cuh"
#include "rank_helpers.cuh"

namespace vsa {
namespace {

constexpr int kSub = 16;                                      // tokens per sub-block
constexpr int kChunkRows = 128;                               // key sub-rows per chunk: the MMA's M
constexpr uint32_t kStageBytes = kChunkRows * kHeadDim * 2;   // a chunk's hi or lo rows: 32 KB
constexpr int kStages = 3;
constexpr int kAcc = 2;                                       // TMEM accumulator pairs, by chunk
constexpr uint32_t kQBytes = 64 * kHeadDim * 2;               // a 64-row box pair, hi or lo: 16 KB
constexpr size_t kSmemBudget = 225 * 1024;
constexpr unsigned int kDetailQ = 0x700, kDetailK = 0x710, kDetailKEmpty = 0x720, kDetailAcc = 0x730,
                       kDetailAccEmpty = 0x740;
// shared memory, from a 1024-byte aligned base: Q hi, Q lo, the K ring, the
// block scores [R][bstride], then the barriers and the TMEM slot
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + 2 * kQBytes;
constexpr uint32_t kOffS = kOffK + kStages * kStageBytes;
constexpr int kBarQ = 0, kBarKFull = 1, kBarKEmpty = kBarKFull + kStages, kBarAccFull = kBarKEmpty + kStages,
              kBarAccEmpty = kBarAccFull + kAcc, kNumBars = kBarAccEmpty + kAcc;
constexpr uint32_t kTailBytes = kNumBars * 8 + 16;

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

template <int R>
__host__ __device__ constexpr int score_warps() { return R; }  // N / 4: one warp per 16 accumulator columns and lane quarter
template <int R>
__host__ __device__ constexpr int router_threads() { return 32 * (score_warps<R>() + 3); }

template <int R>
__global__ void __launch_bounds__(router_threads<R>(), 1)
subblock_router_kernel(const __grid_constant__ CUtensorMap map_q_hi, const __grid_constant__ CUtensorMap map_q_lo,
                       const __grid_constant__ CUtensorMap map_k_hi, const __grid_constant__ CUtensorMap map_k_lo,
                       int32_t* __restrict__ tile_index, unsigned int* err, Geometry cap, DeviceLengths dl,
                       int spad) {
  constexpr int N = 4 * R;                             // query sub-rows per CTA: the MMA's N
  constexpr int kEpiWarps = score_warps<R>();
  constexpr int kWarpTma = kEpiWarps, kWarpMma = kEpiWarps + 1;  // MMA issuers: kWarpMma and kWarpMma + 1
  constexpr int kCols = 16;                            // accumulator columns per score thread: 4 query blocks
  constexpr uint32_t kTmemCols = 2 * kAcc * N < 32 ? 32 : 2 * kAcc * N;  // per chunk: one accumulator per issuer
  static_assert((kTmemCols & (kTmemCols - 1)) == 0 && kTmemCols <= 512, "TMEM allocation");
  static_assert(kEpiWarps * kCols == 4 * N && N <= 64, "16 columns per score warp; query rows within one box");
  static_assert(kEpiWarps * kBins * 4 <= kStages * kStageBytes, "selection histograms fit over the K ring");
  // The request's tiles (the plan's own, or the device lengths'); the layouts
  // (sub-rows spad, selections [T_cap][k_cap]) are the plan's.
  const DynGeom dg = dyn_geom(cap, dl);
  if (!dg.valid) {
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *dl.invalid = 1u;
    return;
  }
  const int T = dg.T, Lv = dg.Lv, k = dg.k;
  const int q0 = blockIdx.x * R;                       // first query block of this CTA
  if (q0 >= T) return;                                 // uniform per CTA, before any barrier or copy
  const int bstride = spad / 4 + 4;                    // block-score row stride (floats)
  const int n_chunks = (4 * T + kChunkRows - 1) / kChunkRows;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  float* S = reinterpret_cast<float*>(smem + kOffS);
  const uint32_t bar0 = sbase + kOffS + static_cast<uint32_t>(R * bstride * 4);
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + kOffS + R * bstride * 4 + kNumBars * 8);
  int* hist = reinterpret_cast<int*>(smem + kOffK);    // [kEpiWarps][kBins], once the products are done

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int bh = blockIdx.y;
  if (tid == 0) {
    mbar_init(bar(kBarQ), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarKFull + s), 1);
      mbar_init(bar(kBarKEmpty + s), 2);  // both MMA issuers read every stage
    }
    for (int a = 0; a < kAcc; ++a) {
      mbar_init(bar(kBarAccFull + a), 2);  // one commit per issuer
      mbar_init(bar(kBarAccEmpty + a), kEpiWarps);
    }
    fence_barrier_init();
  }
  if (warp == kWarpMma) tmem_alloc(smem_u32(tslot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  bool ok = true;

  if (warp == kWarpTma) {
    // ------------------------------------------------------------ TMA loads (lanes 0-3)
    // Each of lanes 0-3 issues one 8 KB box of every stage (channel half
    // lane >> 1, row group lane & 1): one issuing thread keeps too few bytes
    // in flight to feed the products. Each lane waits for the stage itself;
    // lane 0 arms the full barrier. A box may land before the arming: the
    // transaction count may run negative until the arrive, and the phase
    // cannot complete before it.
    if (lane < 4) {
      const int half = lane >> 1, rg = lane & 1;
      int issued = 0;  // K stages issued
      if (lane == 0) mbar_arrive_expect_tx(bar(kBarQ), 2 * kQBytes);
      // Q: lane l loads channel half l & 1 of the hi (l < 2) or lo rows
      tma_load_4d(sbase + kOffQ + (lane >> 1) * kQBytes + (lane & 1) * 8192, (lane >> 1) ? &map_q_lo : &map_q_hi,
                  64 * (lane & 1), 4 * q0, bh, 0, bar(kBarQ));
      for (int i = 0; i < 2 * n_chunks; ++i) {
        const int st = i % kStages;
        // the stage's previous use (stage i - kStages) must have been read by its MMAs
        if (i >= kStages && !mbar_wait(bar(kBarKEmpty + st), ((i / kStages) - 1) & 1, err, kDetailKEmpty)) {
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(bar(kBarKFull + st), kStageBytes);
        const CUtensorMap* m = (i & 1) ? &map_k_lo : &map_k_hi;
        tma_load_4d(sbase + kOffK + st * kStageBytes + half * 16384 + rg * 8192, m, 64 * half,
                    kChunkRows * (i / 2) + 64 * rg, bh, 0, bar(kBarKFull + st));
        issued = i + 1;
      }
      if (!ok) {
        // gave up: let the copies already issued land before the CTA ends
        mbar_wait_drain(bar(kBarQ), 0, kWaitLimitNs);
        for (int i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
          mbar_wait_drain(bar(kBarKFull + i % kStages), (i / kStages) & 1, kWaitLimitNs);
      }
    }
  } else if (warp == kWarpMma || warp == kWarpMma + 1) {
    // ------------------------------------------------------------ MMA issue (two converged warps)
    // The chunk's 24 products split over two issuing warps, each into its own
    // accumulator of the pair (the score warps add the two): a single issuer
    // leaves the tensor pipe idle between its N = 64 MMAs, two interleave.
    //   issuer 0: hi . hi over k-steps 0-7, then lo . hi over k-steps 0-3;
    //   issuer 1: hi . lo over k-steps 0-7, then lo . hi over k-steps 4-7.
    const int w = warp - kWarpMma;
    const uint32_t idesc = idesc_bf16_f32(128, N, 0, 0);
    const uint64_t dq_hi = smem_desc_sw128(sbase + kOffQ, 16, 1024);
    const uint64_t dq_lo = smem_desc_sw128(sbase + kOffQ + kQBytes, 16, 1024);
    const uint64_t dq_b = w == 0 ? dq_hi : dq_lo;  // the B rows of this issuer's hi-stage products
    ok = mbar_wait_warp(bar(kBarQ), 0, err, kDetailQ);
    for (int c = 0; c < n_chunks && ok; ++c) {
      const int a = c % kAcc;
      // accumulator pair a was last read by the epilogue of chunk c - kAcc
      if (c >= kAcc) ok = mbar_wait_warp(bar(kBarAccEmpty + a), ((c / kAcc) - 1) & 1, err, kDetailAccEmpty);
      const uint32_t d = tbase + static_cast<uint32_t>((2 * a + w) * N);
      for (int part = 0; part < 2 && ok; ++part) {  // the chunk's hi rows, then its lo rows
        const int i = 2 * c + part, st = i % kStages;
        ok = mbar_wait_warp(bar(kBarKFull + st), (i / kStages) & 1, err, kDetailK);
        if (!ok) break;
        tc_fence_after();
        const uint64_t dk = smem_desc_sw128(sbase + kOffK + st * kStageBytes, 16, 1024);
        if (part == 0) {
#pragma unroll
          for (int s = 0; s < kHeadDim / 16; ++s) {
            const uint32_t koff = ((s >> 2) * 16384 + (s & 3) * 32) >> 4;
            const uint32_t qoff = ((s >> 2) * 8192 + (s & 3) * 32) >> 4;
            umma_bf16_elect(d, dk + koff, dq_b + qoff, idesc, s > 0 ? 1u : 0u);  // hi . hi or hi . lo
          }
        } else {
#pragma unroll
          for (int j = 0; j < kHeadDim / 32; ++j) {
            const int s = 4 * w + j;
            const uint32_t koff = ((s >> 2) * 16384 + (s & 3) * 32) >> 4;
            const uint32_t qoff = ((s >> 2) * 8192 + (s & 3) * 32) >> 4;
            umma_bf16_elect(d, dk + koff, dq_hi + qoff, idesc, 1u);  // lo . hi, half of the k-steps
          }
        }
        umma_commit_elect(bar(kBarKEmpty + st));  // the stage may be refilled once both issuers are done
      }
      if (ok) umma_commit_elect(bar(kBarAccFull + a));
    }
  } else {
    // ------------------------------------------------------------ block scores (warps 0 .. E - 1)
    const unsigned full = 0xffffffffu;
    const int quarter = warp % 4, col0 = (warp / 4) * kCols;
    const int r = 32 * quarter + lane;                 // key sub-row within a chunk (TMEM lane)
    const uint32_t taddr = tbase + (static_cast<uint32_t>(32 * quarter) << 16) + static_cast<uint32_t>(col0);
    const float scale_log2 = 0.08838834764831845f * 1.4426950408889634f;  // log2(e) / sqrt(128)
    float lq[kCols];                                   // log2 token counts of this thread's query sub-rows
#pragma unroll
    for (int j = 0; j < kCols; ++j) lq[j] = lg_count(4 * q0 + col0 + j, Lv);
    for (int c = 0; c < n_chunks && ok; ++c) {
      const int a = c % kAcc;
      ok = mbar_wait_warp(bar(kBarAccFull + a), (c / kAcc) & 1, err, kDetailAcc);
      if (!ok) break;
      tc_fence_after();
      uint32_t v[kCols], v1[kCols];
      tmem_ld16(taddr + static_cast<uint32_t>(2 * a * N), v);
      tmem_ld16(taddr + static_cast<uint32_t>((2 * a + 1) * N), v1);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarAccEmpty + a));  // the MMAs of chunk c + kAcc may overwrite it
      // logit x = acc / sqrt(128) + log2 n_q + log2 n_k, in log2 units; the key
      // sub-row's count is added to the maximum, not to every element
      const float lk = lg_count(kChunkRows * c + r, Lv);
      float* srow = S + (col0 / 4) * bstride + (kChunkRows / 4) * c + r / 4;
#pragma unroll
      for (int jb = 0; jb < kCols / 4; ++jb) {
        float x[4];
#pragma unroll
        for (int t = 0; t < 4; ++t)
          x[t] = fmaf(__uint_as_float(v[4 * jb + t]) + __uint_as_float(v1[4 * jb + t]), scale_log2, lq[4 * jb + t]);
        float mb = fmax3(x[0], x[1], fmaxf(x[2], x[3])) + lk;
        mb = fmaxf(mb, __shfl_xor_sync(full, mb, 1));
        mb = fmaxf(mb, __shfl_xor_sync(full, mb, 2));
        const float off = (mb > -INFINITY ? mb : 0.f) - lk;   // an all-empty block: 2^-inf = 0 below
        float w = (ex2(x[0] - off) + ex2(x[1] - off)) + (ex2(x[2] - off) + ex2(x[3] - off));
        w += __shfl_xor_sync(full, w, 1);
        w += __shfl_xor_sync(full, w, 2);
        if ((lane & 3) == 0) srow[jb * bstride] = (mb > -INFINITY ? mb : 0.f) + lg2(w);
      }
    }
  }
  // every product and score is done; the K ring is idle and holds the histograms
  ok = __syncthreads_and(ok);
  if (ok && warp < kEpiWarps) {
    // key blocks T .. n_chunks * 32 - 1 hold only empty sub-blocks and scored
    // -inf above, as the counting select requires of a row's padding
    for (int rq = warp; rq < R; rq += kEpiWarps)
      if (q0 + rq < T)
        warp_select_topk_count(S + rq * bstride, T, n_chunks * (kChunkRows / 4), k, hist + warp * kBins,
                               tile_index + (static_cast<size_t>(bh) * cap.T + q0 + rq) * cap.k, lane);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) tmem_dealloc(tbase, kTmemCols);
}

int sub_pad(int T) { return (4 * T + 127) / 128 * 128; }  // as subblock_rows_padded

size_t smem_for(int r, int spad) {
  return 1024 + kOffS + static_cast<size_t>(r) * (spad / 4 + 4) * sizeof(float) + kTailBytes;
}

int pick_rows(int spad) {
  for (int r = 16; r >= 8; r /= 2)
    if (smem_for(r, spad) <= kSmemBudget) return r;
  return 0;
}

template <int R>
cudaError_t launch_rows(const Geometry& g, const CUtensorMap (&maps)[4], int32_t* tile_index, unsigned int* err,
                        const DeviceLengths& dl, size_t smem, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(subblock_router_kernel<R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid((g.T + R - 1) / R, g.B * g.H);
  subblock_router_kernel<R><<<grid, router_threads<R>(), smem, stream>>>(maps[0], maps[1], maps[2], maps[3], tile_index, err,
                                                              g, dl, sub_pad(g.T));
  return cudaGetLastError();
}

}  // namespace

size_t subblock_router_smem_bytes(const Geometry& g, int* rows_per_cta) {
  const int r = pick_rows(sub_pad(g.T));
  if (rows_per_cta) *rows_per_cta = r;
  return r ? smem_for(r, sub_pad(g.T)) : 0;
}

cudaError_t launch_subblock_router(const Geometry& g, const CUtensorMap (&maps)[4], int32_t* tile_index,
                                   unsigned int* err, const DeviceLengths& dl, cudaStream_t stream) {
  int r = 0;
  const size_t smem = subblock_router_smem_bytes(g, &r);
  switch (r) {
    case 16: return launch_rows<16>(g, maps, tile_index, err, dl, smem, stream);
    case 8: return launch_rows<8>(g, maps, tile_index, err, dl, smem, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace vsa
