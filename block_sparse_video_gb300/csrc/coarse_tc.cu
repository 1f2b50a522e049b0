// Coarse tile attention fused with the top-k tile selection, both products on
// the tcgen05 tensor cores.
//
// For each (batch, head) and each video query tile t ("UniServe: serving
// FastH3 at its fastest", section "The FastH3 workload"):
//   s[t][j] = pooled_q[t] . pooled_k[j] / sqrt(128)        over all T video tiles
//   selection(t) = the k largest s[t][j], ties to the lower j, ascending
//   coarse[t] = sum_j softmax_j(s[t][.]) * pooled_v[j]
//
// Operands. A split kernel writes the pooled Q, K and V again as bf16 rows of
// a head plus a remainder (x ~ hi + lo, ~2^-16 relative), so that each fp32
// product is hi.hi + hi.lo + lo.hi: three bf16 MMAs accumulating in fp32 in
// TMEM. Rows past the request's T are zeros.
//
// Work unit: 64 query tiles of one (batch, head). The grid is persistent (one
// CTA per SM at most, units taken in a fixed stride), and each CTA owns a
// scratch row buffer in global memory (64 rows of T_pad floats, L2-resident).
// Per unit, three phases separated by CTA barriers:
//   A. scores, transposed so that the MMA has M = 128:
//        S^T[128 keys x 64 queries] = Kbar_chunk . Qbar^T      (A, B K-major)
//      for each 128-key chunk; four warps move each chunk from TMEM (lane =
//      key, column = query), scaled by 1/sqrt(128), into the scratch rows;
//   B. one warp per query row (rows handed out one at a time, as a row's cost
//      varies with its search): the row copied into shared memory and read
//      from there (rows of up to 1,280 keys) or held in registers, the exact
//      top-k (a
//      counting threshold search; the radix select where scores tie at the
//      cut), the row maximum m, l = sum_j exp(s_j - m), and p_j = exp(s_j - m)
//      written back over the row's own bytes as bf16 hi then bf16 lo rows;
//   C. the coarse product, transposed the same way:
//        C^T[128 dims x 64 queries] = Vbar_chunk^T . P^T       (A MN-major, B K-major)
//      accumulated over the chunks, with P loaded back by TMA; four warps
//      divide by l and store coarse rows.
// Score errors of ~2^-16 relative sit far inside the selection's 1e-3 tie
// band; the selection itself is an integer decision on the fp32 scores.
//
// Warp roles: warp 0 issues the TMA loads (four issuing lanes, one 8 KB box
// each) through a ring of 32 KB stages; warps 1 and 2 issue the MMAs,
// converged with one elected lane each, splitting every chunk's 24 products
// between two accumulators (a single issuer leaves the pipe idle between
// N = 64 MMAs); warps from 4 move scores and outputs out of TMEM (per lane
// quarter, a share of the 64 columns each); every warp runs phase B. Rows of up
// to 1,280 keys: 24 warps (16 movers), the row read from shared memory in
// phase B; longer rows: 12 warps (8 movers), the row held in registers. Every
// wait is bounded.
#include <cmath>

#include "kernels.cuh"
#include "ptx.cuh"
#include "rank_helpers.cuh"

namespace vsa {
namespace {

// Two builds: rows of up to 1,280 keys (NM <= 10) stay in shared memory in
// phase B, so the CTA runs 24 warps of at most 80 registers (twice the warps
// to hide a row's dependent chain); longer rows are held in registers by 12
// warps of up to 168 registers.
__host__ __device__ constexpr bool smem_rows(int nm) { return nm <= 10; }
__host__ __device__ constexpr int threads_of(int nm) { return smem_rows(nm) ? 768 : 384; }
constexpr int kRows = 64;                     // query tiles per unit: the MMA's N
constexpr int kChunk = 128;                   // key tiles per chunk: the MMA's M
constexpr int kStages = 5;                    // ring stages of 32 KB
constexpr uint32_t kStageBytes = kChunk * kHeadDim * 2;
constexpr uint32_t kQBytes = 2 * kRows * kHeadDim * 2;  // Qbar hi and lo, 64 rows each
constexpr int kWarpTma = 0, kWarpMma = 1, kWarpEpi0 = 4;
// TMEM movers from warp 4: lane quarter warp % 4, column group (warp - 4) / 4
__host__ __device__ constexpr int epi_warps_of(int nm) { return smem_rows(nm) ? 16 : 8; }
constexpr uint32_t kTmemCols = 256;           // two accumulator pairs of 64 columns
constexpr unsigned int kDetailQ = 0xE00, kDetailFull = 0xE10, kDetailEmpty = 0xE20, kDetailAcc = 0xE30,
                       kDetailAccEmpty = 0xE40, kDetailC = 0xE50, kDetailRow = 0xE60;

// shared memory from a 1024-byte aligned base: Qbar hi/lo, the ring (which
// holds the staged score rows in phase B), then the row sums, the selection
// histograms, the barriers and the TMEM slot
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffRing = kOffQ + kQBytes;
constexpr uint32_t kOffL = kOffRing + kStages * kStageBytes;
constexpr uint32_t kOffHist = kOffL + kRows * 4;
__host__ __device__ constexpr uint32_t off_bar_of(int nm) { return kOffHist + (threads_of(nm) / 32) * kBins * 4; }
constexpr int kBarQ = 0, kBarFull = 1, kBarEmpty = kBarFull + kStages, kBarAccFull = kBarEmpty + kStages,
              kBarAccEmpty = kBarAccFull + 2, kBarC = kBarAccEmpty + 2, kBarRow = kBarC + 1;
// kBarRow: the staged score row of each warp in phase B
__host__ __device__ constexpr int num_bars_of(int nm) { return kBarRow + threads_of(nm) / 32; }
__host__ __device__ constexpr uint32_t off_slot_of(int nm) { return off_bar_of(nm) + num_bars_of(nm) * 8; }
__host__ __device__ constexpr uint32_t smem_bytes_of(int nm) { return off_slot_of(nm) + 16 + 1024; }  // + alignment slack
static_assert(smem_bytes_of(5) <= 227 * 1024 && smem_bytes_of(10) <= 227 * 1024 && smem_bytes_of(18) <= 227 * 1024,
              "shared memory");
// phase B, rows in shared memory: one 128 NM-key buffer a warp in the ring
static_assert(24 * 128 * 10 * 4 <= kStages * kStageBytes, "staged rows fit the ring");

struct CoarseParams {
  Geometry cap;             // the plan's geometry: T_cap, k_cap and the layouts
  DeviceLengths dl;
  int tp_cap;               // padded rows per (b, h) of the hi/lo operands and of a scratch row
  int n_units;              // B * H * ceil(T_cap / 64)
  float* scratch;           // [grid][64][tp_cap] floats
  float* coarse;            // [B, H, T_cap, 128]
  int32_t* tile_index;      // [B, H, T_cap, k_cap]
  unsigned int* err;
};

// A query row as a warp sees it: lane l takes keys 128 m + 4 l .. + 3 as one
// float4 for m < NM (-inf past T), one coalesced 16-byte access per m.

// Exclusive prefix sum of a small per-lane count over the warp, and the total.
__device__ __forceinline__ int warp_exclusive_scan(int x, int lane, int& total) {
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  total = __shfl_sync(0xffffffffu, incl, 31);
  return incl - x;
}

// The k largest entries of the row, written ascending to dst[0 .. k): the
// same set, with ties to the lower index, as warp_select_topk_count (a
// counting search for a threshold with exactly k entries at or above it; the
// radix select where entries tie at the cut or a score is not finite). h: kBins
// ints of shared memory for the radix select.
__device__ __forceinline__ float f4_at(const float4& v, int e) {
  return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
}

// row(m): lane l's keys 128 m + 4 l .. + 3 as a float4 (-inf past T), from
// registers or from shared memory. Returns the row's maximum, taken with its
// moments (NaN when k >= T, where no moments are taken).
template <int NM, typename Row>
__device__ __forceinline__ float select_topk(const Row& row, int T, int k, int* h, int32_t* dst, int lane) {
  const unsigned full = 0xffffffffu;
  if (k >= T) {
    for (int j = lane; j < T; j += 32) dst[j] = j;
    return __int_as_float(0x7fffffff);  // no moments taken: NaN
  }
  // Row moments. Slices m holding only keys < T take no per-entry test; the
  // slice with the row's end skips the -inf entries past T. Four partial sums
  // a lane keep the dependent chains short. A score that is not finite (or
  // sums that overflow) sends the row to the radix select.
  float mn[2] = {INFINITY, INFINITY}, mxv[2] = {-INFINITY, -INFINITY};
  float a1[4] = {0.f, 0.f, 0.f, 0.f}, a2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int m = 0; m < NM; ++m) {
    if (128 * m + 128 <= T) {
      const float4 vm = row(m);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float x = f4_at(vm, e);
        mn[e & 1] = fminf(mn[e & 1], x);
        mxv[e & 1] = fmaxf(mxv[e & 1], x);
        a1[e] += x;
        a2[e] = fmaf(x, x, a2[e]);
      }
    } else if (128 * m < T) {
      const float4 vm = row(m);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float x = f4_at(vm, e);
        if (128 * m + 4 * lane + e < T) {
          mn[e & 1] = fminf(mn[e & 1], x);
          mxv[e & 1] = fmaxf(mxv[e & 1], x);
          a1[e] += x;
          a2[e] = fmaf(x, x, a2[e]);
        }
      }
    }
  }
  float vmin = fminf(mn[0], mn[1]), vmax = fmaxf(mxv[0], mxv[1]);
  float s1 = (a1[0] + a1[1]) + (a1[2] + a1[3]), s2 = (a2[0] + a2[1]) + (a2[2] + a2[3]);
  // a lane with no key has vmin > vmax and zero sums: nothing to flag (a NaN
  // key leaves the extremes alone but not the sum)
  const bool has_key = vmin <= vmax || s1 != s1;
  const bool bad =
      has_key && !(fabsf(vmin) <= 3.0e38f && fabsf(vmax) <= 3.0e38f && fabsf(s1) <= 3.0e38f && s2 <= 3.0e38f);
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    vmin = fminf(vmin, __shfl_xor_sync(full, vmin, o));
    vmax = fmaxf(vmax, __shfl_xor_sync(full, vmax, o));
    s1 += __shfl_xor_sync(full, s1, o);
    s2 += __shfl_xor_sync(full, s2, o);
  }
  auto count_ge = [&](float x) {  // -inf past T never counts (x > vmin >= -inf)
    int c = 0;
#pragma unroll
    for (int m = 0; m < NM; ++m)
      if (128 * m < T) {  // slices past T hold -inf only
        const float4 vm = row(m);
        c += (vm.x >= x) + (vm.y >= x) + (vm.z >= x) + (vm.w >= x);
      }
    return static_cast<int>(__reduce_add_sync(full, static_cast<unsigned>(c)));
  };
  float theta = 0.f;
  bool found = false;
  if (!__any_sync(full, bad) && k >= 1) {
    float lo = vmin, hi = nextafterf(vmax, INFINITY);
    float flo = static_cast<float>(T - k), fhi = static_cast<float>(-k);
    int kept = 0;
    const float mean = s1 / static_cast<float>(T);
    const float sd = sqrtf(fmaxf(s2 / static_cast<float>(T) - mean * mean, 0.f));
    float x = mean + normcdfinvf(1.f - static_cast<float>(k) / static_cast<float>(T)) * sd;
#pragma unroll 1
    for (int it = 0; it < 48; ++it) {
      if (it > 0) x = lo + (hi - lo) * __fdividef(flo, flo - fhi);  // a trial point: any x in (lo, hi) is valid
      if (!(x > lo && x < hi)) x = 0.5f * (lo + hi);
      if (!(x > lo && x < hi)) break;
      const int c = count_ge(x);
      if (c == k) {
        theta = x;
        found = true;
        break;
      }
      if (c > k) {
        lo = x;
        flo = static_cast<float>(c - k);
        if (kept > 0) fhi *= 0.5f;
        kept = 1;
      } else {
        hi = x;
        fhi = static_cast<float>(c - k);
        if (kept < 0) flo *= 0.5f;
        kept = -1;
      }
    }
  }
  if (found) {
    // in key order: lane-major, then the lane's four keys; one ballot per key
    // slot gives every lane the count of selected keys in the lanes before it
    const unsigned lt_mask = (1u << lane) - 1u;
    int written = 0;
#pragma unroll
    for (int m = 0; m < NM; ++m) {
      if (128 * m >= T) break;  // slices past T hold -inf only
      const float4 vm = row(m);
      const bool s0 = vm.x >= theta, s1b = vm.y >= theta, s2b = vm.z >= theta, s3 = vm.w >= theta;
      const unsigned b0 = __ballot_sync(full, s0), b1 = __ballot_sync(full, s1b), b2 = __ballot_sync(full, s2b),
                     b3 = __ballot_sync(full, s3);  // -inf past T never reaches theta
      int pos = written + __popc(b0 & lt_mask) + __popc(b1 & lt_mask) + __popc(b2 & lt_mask) + __popc(b3 & lt_mask);
      const int key = 128 * m + 4 * lane;
      if (s0) dst[pos++] = key;
      if (s1b) dst[pos++] = key + 1;
      if (s2b) dst[pos++] = key + 2;
      if (s3) dst[pos] = key + 3;
      written += __popc(b0) + __popc(b1) + __popc(b2) + __popc(b3);
    }
    return vmax;
  }
  // radix select, 8 bits per pass from the top, over the order-preserving
  // integer image of the scores (-0 and +0 alike)
  uint32_t prefix = 0u, pmask = 0u;
  int rem = k;
#pragma unroll 1
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int b = lane; b < kBins; b += 32) h[b] = 0;
    __syncwarp();
#pragma unroll
    for (int m = 0; m < NM; ++m) {
      const float4 vm = row(m);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (128 * m + 4 * lane + e < T) {
          const uint32_t key = order_key(f4_at(vm, e));
          if ((key & pmask) == prefix) atomicAdd(&h[(key >> shift) & 0xFFu], 1);
        }
    }
    __syncwarp();
    int c[8], lsum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) { c[i] = h[255 - 8 * lane - i]; lsum += c[i]; }
    int incl = lsum;
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
  // every key above the k-th largest, and the lowest `rem` keys equal to it
  int written = 0, eq_seen = 0;
#pragma unroll
  for (int m = 0; m < NM; ++m) {
    bool gt[4], eq[4];
    int n_eq = 0;
    const float4 vm = row(m);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const bool in = 128 * m + 4 * lane + e < T;
      const uint32_t key = in ? order_key(f4_at(vm, e)) : 0u;
      gt[e] = in && key > prefix;
      eq[e] = in && key == prefix;
      n_eq += eq[e];
    }
    int eq_total;
    int eq_before = eq_seen + warp_exclusive_scan(n_eq, lane, eq_total);
    bool sel[4];
    int cnt = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      sel[e] = gt[e] || (eq[e] && eq_before < rem);
      eq_before += eq[e];
      cnt += sel[e];
    }
    int total;
    int pos = written + warp_exclusive_scan(cnt, lane, total);
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (sel[e]) dst[pos++] = 128 * m + 4 * lane + e;
    written += total;
    eq_seen += eq_total;
  }
  return vmax;
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

template <int NM>
__global__ void __launch_bounds__(threads_of(NM), 1)
coarse_tc_kernel(const __grid_constant__ CUtensorMap map_qh, const __grid_constant__ CUtensorMap map_ql,
                 const __grid_constant__ CUtensorMap map_kh, const __grid_constant__ CUtensorMap map_kl,
                 const __grid_constant__ CUtensorMap map_vh, const __grid_constant__ CUtensorMap map_vl,
                 const __grid_constant__ CUtensorMap map_p, const CoarseParams p) {
  const DynGeom dg = dyn_geom(p.cap, p.dl);
  if (!dg.valid) {
    if (blockIdx.x == 0 && threadIdx.x == 0) *p.dl.invalid = 1u;
    return;
  }
  constexpr int kThreads = threads_of(NM), kWarps = kThreads / 32, kEpiWarps = epi_warps_of(NM);
  constexpr int kMoverCols = 4 * kRows / kEpiWarps;  // query columns a mover takes
  constexpr bool kSmemRows = smem_rows(NM);
  constexpr uint32_t kOffBar = off_bar_of(NM), kOffSlot = off_slot_of(NM);
  const int T = dg.T, k = dg.k, T_cap = p.cap.T, k_cap = p.cap.k;
  const int n_chunks = (T + kChunk - 1) / kChunk;
  const int groups_cap = (T_cap + kRows - 1) / kRows;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  float* l_row = reinterpret_cast<float*>(smem + kOffL);
  int* hist = reinterpret_cast<int*>(smem + kOffHist);
  auto bar = [&](int i) { return sbase + kOffBar + 8u * static_cast<uint32_t>(i); };
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + kOffSlot);
  int* next_row = reinterpret_cast<int*>(smem + kOffSlot + 4);  // phase B: rows handed out so far

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  unsigned int* err = p.err;
  if (tid == 0) {
    mbar_init(bar(kBarQ), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarFull + s), 1);
      mbar_init(bar(kBarEmpty + s), 2);  // both issuers read every stage
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar(kBarAccFull + a), 2);  // one commit per issuer
      mbar_init(bar(kBarAccEmpty + a), kEpiWarps);
    }
    mbar_init(bar(kBarC), 2);
    for (int i = 0; i < kWarps; ++i) mbar_init(bar(kBarRow + i), 1);
    fence_barrier_init();
  }
  if (warp == kWarpMma) tmem_alloc(smem_u32(tslot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  float* rows = p.scratch + static_cast<size_t>(blockIdx.x) * kRows * p.tp_cap;  // this CTA's scratch rows
  const float scale = 0.08838834764831845f;  // 1/sqrt(128)
  bool failed = false;

  // Ring positions and accumulator-pair uses, counted alike by every warp
  // over all units: phase A takes 2 stages (K hi, K lo) and one accumulator
  // pair per chunk, phase C 3 stages (V hi, V lo, P hi + lo) per chunk.
  uint32_t ring0 = 0, acc0 = 0, units_done = 0;
  uint32_t rows_staged = 0;  // score rows this warp has taken in phase B, over all units
  for (int u = blockIdx.x; u < p.n_units; u += gridDim.x) {
    const int bh = u / groups_cap;
    const int q0 = (u - bh * groups_cap) * kRows;
    if (q0 >= T) continue;  // uniform: a query group past the request's tiles
    const int n_rows = min(kRows, T - q0);

    // ------------------------------------------------------------ phase A: scores
    if (warp == kWarpTma) {
      bool lane_failed = false;
      if (lane < 4) {
        const int half = lane >> 1, rg = lane & 1;
        if (lane == 0) mbar_arrive_expect_tx(bar(kBarQ), kQBytes);
        // Qbar: lane l loads channel half l & 1 of the hi (l < 2) or lo rows
        tma_load_4d(sbase + kOffQ + (lane >> 1) * (kQBytes / 2) + (lane & 1) * 8192, (lane >> 1) ? &map_ql : &map_qh,
                    64 * (lane & 1), q0, bh, 0, bar(kBarQ));
        for (int i = 0; i < 2 * n_chunks && !lane_failed; ++i) {
          const uint32_t r = ring0 + i;
          const int st = r % kStages;
          if (r >= kStages && !mbar_wait(bar(kBarEmpty + st), ((r / kStages) - 1) & 1, err, kDetailEmpty)) {
            lane_failed = true;
            break;
          }
          if (lane == 0) mbar_arrive_expect_tx(bar(kBarFull + st), kStageBytes);
          tma_load_4d(sbase + kOffRing + st * kStageBytes + half * 16384 + rg * 8192, (i & 1) ? &map_kl : &map_kh,
                      64 * half, kChunk * (i / 2) + 64 * rg, bh, 0, bar(kBarFull + st));
        }
      }
      failed = __any_sync(0xffffffffu, lane_failed);
    } else if (warp == kWarpMma || warp == kWarpMma + 1) {
      // issuer 0: hi.hi over k-steps 0-7, then lo.hi over 0-3; issuer 1:
      // hi.lo over 0-7, then lo.hi over 4-7
      const int w = warp - kWarpMma;
      const uint32_t idesc = idesc_bf16_f32(128, kRows, 0, 0);
      const uint64_t dq_hi = smem_desc_sw128(sbase + kOffQ, 16, 1024);
      const uint64_t dq_lo = smem_desc_sw128(sbase + kOffQ + kQBytes / 2, 16, 1024);
      const uint64_t dq_b = w == 0 ? dq_hi : dq_lo;
      failed = !mbar_wait_warp(bar(kBarQ), units_done & 1, err, kDetailQ);
      for (int c = 0; c < n_chunks && !failed; ++c) {
        const uint32_t au = acc0 + c;
        const int a = au & 1;
        if (au >= 2 && !mbar_wait_warp(bar(kBarAccEmpty + a), ((au / 2) - 1) & 1, err, kDetailAccEmpty)) {
          failed = true;
          break;
        }
        const uint32_t d = tbase + static_cast<uint32_t>((2 * a + w) * kRows);
        for (int part = 0; part < 2; ++part) {
          const uint32_t r = ring0 + 2 * c + part;
          const int st = r % kStages;
          if (!mbar_wait_warp(bar(kBarFull + st), (r / kStages) & 1, err, kDetailFull)) {
            failed = true;
            break;
          }
          tc_fence_after();
          const uint64_t dk = smem_desc_sw128(sbase + kOffRing + st * kStageBytes, 16, 1024);
          if (part == 0) {
#pragma unroll
            for (int s = 0; s < kHeadDim / 16; ++s) {
              const uint32_t koff = ((s >> 2) * 16384 + (s & 3) * 32) >> 4;
              const uint32_t qoff = ((s >> 2) * 8192 + (s & 3) * 32) >> 4;
              umma_bf16_elect(d, dk + koff, dq_b + qoff, idesc, s > 0 ? 1u : 0u);
            }
          } else {
#pragma unroll
            for (int j = 0; j < kHeadDim / 32; ++j) {
              const int s = 4 * w + j;
              const uint32_t koff = ((s >> 2) * 16384 + (s & 3) * 32) >> 4;
              const uint32_t qoff = ((s >> 2) * 8192 + (s & 3) * 32) >> 4;
              umma_bf16_elect(d, dk + koff, dq_hi + qoff, idesc, 1u);
            }
          }
          umma_commit_elect(bar(kBarEmpty + st));
        }
        if (!failed) umma_commit_elect(bar(kBarAccFull + a));
      }
    } else if (warp >= kWarpEpi0 && warp < kWarpEpi0 + kEpiWarps) {
      // lane quarter q (TMEM lane = key 128 c + 32 q + lane), columns kMoverCols ch ..
      const int q = warp % 4, ch = (warp - kWarpEpi0) / 4;
      const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;
      for (int c = 0; c < n_chunks && !failed; ++c) {
        const uint32_t au = acc0 + c;
        const int a = au & 1;
        if (!mbar_wait_warp(bar(kBarAccFull + a), (au / 2) & 1, err, kDetailAcc)) {
          failed = true;
          break;
        }
        tc_fence_after();
        const int key = kChunk * c + 32 * q + lane;
#pragma unroll
        for (int part = 0; part < kMoverCols / 16; ++part) {
          const int col = kMoverCols * ch + 16 * part;
          uint32_t x0[16], x1[16];
          tmem_ld16(tbase + lane_off + static_cast<uint32_t>(2 * a * kRows + col), x0);
          tmem_ld16(tbase + lane_off + static_cast<uint32_t>((2 * a + 1) * kRows + col), x1);
          tmem_wait_ld();
          if (key < T) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int r = col + j;
              if (r < n_rows)
                rows[static_cast<size_t>(r) * p.tp_cap + key] =
                    (__uint_as_float(x0[j]) + __uint_as_float(x1[j])) * scale;
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarAccEmpty + a));
      }
      // phase B copies the score rows into shared memory through the async proxy
      fence_proxy_async_global();
    }
    if (tid == 0) *next_row = 0;  // read in phase B, after the barrier below
    ring0 += 2 * n_chunks;
    acc0 += n_chunks;
    failed = __syncthreads_or(failed);
    if (failed) break;

    // ------------------------------------------------------------ phase B: selection, softmax, P
    // mx: the row's maximum as the selection took it (the same fmaxf over the
    // same entries, so the same value), or NaN to take it here
    auto softmax_row = [&](auto&& rowf, float* row, int r, float mx) {
      if (mx != mx) {
        mx = -INFINITY;
#pragma unroll
        for (int m = 0; m < NM; ++m)
          if (128 * m < T) {
            const float4 vm = rowf(m);
            mx = fmaxf(mx, fmaxf(fmaxf(vm.x, vm.y), fmaxf(vm.z, vm.w)));
          }
#pragma unroll
        for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      }
      // p = exp(s - max) = 2^((s - max) log2 e); entries past T give 2^-inf = 0
      const float nmx = -mx * 1.4426950408889634f;
      float l = 0.f;
      __syncwarp();  // every lane has read the row before it is overwritten
      uint2* ph = reinterpret_cast<uint2*>(row);                 // the row's first half: p hi, 4 keys per uint2
      uint2* pl = reinterpret_cast<uint2*>(row + p.tp_cap / 2);  // second half: p lo
#pragma unroll
      for (int m = 0; m < NM; ++m) {
        if (128 * m < kChunk * n_chunks) {
          const float4 vm = rowf(m);
          const float e0 = ex2_approx(fmaf(vm.x, 1.4426950408889634f, nmx));
          const float e1 = ex2_approx(fmaf(vm.y, 1.4426950408889634f, nmx));
          const float e2 = ex2_approx(fmaf(vm.z, 1.4426950408889634f, nmx));
          const float e3 = ex2_approx(fmaf(vm.w, 1.4426950408889634f, nmx));
          l += (e0 + e1) + (e2 + e3);
          uint32_t h01, l01, h23, l23;
          split_bf16_pair(e0, e1, h01, l01);
          split_bf16_pair(e2, e3, h23, l23);
          ph[32 * m + lane] = make_uint2(h01, h23);
          pl[32 * m + lane] = make_uint2(l01, l23);
        }
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
      if (lane == 0) l_row[r] = l;
    };
    if constexpr (kSmemRows) {
      // each warp copies its row into its own buffer in the ring (idle in this
      // phase), marks the entries past T as -inf, and reads it from there
      const uint32_t buf = sbase + kOffRing + static_cast<uint32_t>(warp) * (NM * 512u);
      const uint32_t row_bytes = (static_cast<uint32_t>(T) * 4u + 15u) & ~15u;
      // rows are handed out one at a time (a row's cost varies with its search)
      for (int r = warp; r < n_rows && !failed; ++rows_staged) {
        float* row = rows + static_cast<size_t>(r) * p.tp_cap;
        if (lane == 0) {
          fence_proxy_async_smem();  // the buffer's earlier reads come before the copy overwrites it
          mbar_arrive_expect_tx(bar(kBarRow + warp), row_bytes);
          bulk_load(buf, row, row_bytes, bar(kBarRow + warp));
        }
        if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarRow + warp), rows_staged & 1u, err, kDetailRow))) {
          failed = true;
          break;
        }
#pragma unroll
        for (int m = 0; m < NM; ++m) {
          const int j = 128 * m + 4 * lane;
          if (j + 3 >= T)
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (j + e >= T) st_shared_f32(buf + 4u * static_cast<uint32_t>(j + e), -INFINITY);
        }
        __syncwarp();
        auto rowf = [&](int m) { return ld_shared_f4(buf + 16u * static_cast<uint32_t>(32 * m + lane)); };
        const float mx = select_topk<NM>(rowf, T, k, hist + warp * kBins,
                                         p.tile_index + (static_cast<size_t>(bh) * T_cap + q0 + r) * k_cap, lane);
        softmax_row(rowf, row, r, mx);
        int nr = 0;
        if (lane == 0) nr = kWarps + atomicAdd(next_row, 1);
        r = __shfl_sync(0xffffffffu, nr, 0);
      }
    } else {
      for (int r = warp; r < n_rows;) {
        float* row = rows + static_cast<size_t>(r) * p.tp_cap;
        float4 v[NM];
#pragma unroll
        for (int m = 0; m < NM; ++m) {
          const int j = 128 * m + 4 * lane;  // T_pad is a multiple of 128, so j + 3 < T_pad
          v[m] = j < T ? reinterpret_cast<const float4*>(row)[32 * m + lane]
                       : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
          if (j + 3 >= T) {  // the row's ragged end: entries past T are -inf
            if (j + 1 >= T) v[m].y = -INFINITY;
            if (j + 2 >= T) v[m].z = -INFINITY;
            if (j + 3 >= T) v[m].w = -INFINITY;
          }
        }
        auto rowf = [&](int m) { return v[m]; };
        const float mx = select_topk<NM>(rowf, T, k, hist + warp * kBins,
                                         p.tile_index + (static_cast<size_t>(bh) * T_cap + q0 + r) * k_cap, lane);
        softmax_row(rowf, row, r, mx);
        int nr = 0;
        if (lane == 0) nr = kWarps + atomicAdd(next_row, 1);
        r = __shfl_sync(0xffffffffu, nr, 0);
      }
    }
    // P is read back by TMA (the async proxy): order these generic writes before it,
    // and the reads of the staged rows before the TMA writes of phase C
    fence_proxy_async_global();
    fence_proxy_async_smem();
    failed = __syncthreads_or(failed);
    if (failed) break;

    // ------------------------------------------------------------ phase C: coarse product
    if (warp == kWarpTma) {
      bool lane_failed = false;
      if (lane < 4) {
        const int half = lane >> 1, kh = lane & 1;
        for (int i = 0; i < 3 * n_chunks && !lane_failed; ++i) {
          const uint32_t r = ring0 + i;
          const int st = r % kStages, c = i / 3, part = i % 3;
          if (r >= kStages && !mbar_wait(bar(kBarEmpty + st), ((r / kStages) - 1) & 1, err, kDetailEmpty)) {
            lane_failed = true;
            break;
          }
          if (lane == 0) mbar_arrive_expect_tx(bar(kBarFull + st), kStageBytes);
          const uint32_t dst = sbase + kOffRing + st * kStageBytes + half * 16384 + kh * 8192;
          if (part < 2) {
            // Vbar rows: dims half `half`, keys 64 kh .. + 63 of the chunk
            tma_load_4d(dst, part ? &map_vl : &map_vh, 64 * half, kChunk * c + 64 * kh, bh, 0, bar(kBarFull + st));
          } else {
            // P: plane `half` (hi, lo), keys 64 kh .. + 63 of the chunk, all 64 rows
            tma_load_4d(dst, &map_p, kChunk * c + 64 * kh, half, 0, static_cast<int>(blockIdx.x), bar(kBarFull + st));
          }
        }
      }
      failed = __any_sync(0xffffffffu, lane_failed);
    } else if (warp == kWarpMma || warp == kWarpMma + 1) {
      // issuer 0: Vhi.Phi over k-steps 0-7, then Vlo.Phi over 0-3; issuer 1:
      // Vhi.Plo over 0-7, then Vlo.Phi over 4-7; each into its own
      // accumulator of 64 columns, summed in the epilogue
      const int w = warp - kWarpMma;
      const uint32_t idesc = idesc_bf16_f32(128, kRows, 1, 0);
      const uint32_t d = tbase + static_cast<uint32_t>(w * kRows);
      for (int c = 0; c < n_chunks && !failed; ++c) {
        const uint32_t r = ring0 + 3 * c;
        const int sv_hi = r % kStages, sv_lo = (r + 1) % kStages, sp = (r + 2) % kStages;
        if (!mbar_wait_warp(bar(kBarFull + sv_hi), (r / kStages) & 1, err, kDetailFull) ||
            !mbar_wait_warp(bar(kBarFull + sv_lo), ((r + 1) / kStages) & 1, err, kDetailFull) ||
            !mbar_wait_warp(bar(kBarFull + sp), ((r + 2) / kStages) & 1, err, kDetailFull)) {
          failed = true;
          break;
        }
        tc_fence_after();
        const uint32_t pbase = sbase + kOffRing + sp * kStageBytes;
        const uint64_t dp_hi = smem_desc_sw128(pbase, 16, 1024);
        const uint64_t dp_lo = smem_desc_sw128(pbase + 16384, 16, 1024);
        const uint64_t dv_hi = smem_desc_sw128(sbase + kOffRing + sv_hi * kStageBytes, 16384, 1024);
        const uint64_t dv_lo = smem_desc_sw128(sbase + kOffRing + sv_lo * kStageBytes, 16384, 1024);
        const uint64_t dp_b = w == 0 ? dp_hi : dp_lo;
#pragma unroll
        for (int s = 0; s < kChunk / 16; ++s) {
          const uint32_t voff = (s * 2048) >> 4;
          const uint32_t poff = ((s >> 2) * 8192 + (s & 3) * 32) >> 4;
          umma_bf16_elect(d, dv_hi + voff, dp_b + poff, idesc, (c > 0 || s > 0) ? 1u : 0u);
        }
        umma_commit_elect(bar(kBarEmpty + sv_hi));
#pragma unroll
        for (int j = 0; j < kChunk / 32; ++j) {
          const int s = 4 * w + j;
          const uint32_t voff = (s * 2048) >> 4;
          const uint32_t poff = ((s >> 2) * 8192 + (s & 3) * 32) >> 4;
          umma_bf16_elect(d, dv_lo + voff, dp_hi + poff, idesc, 1u);
        }
        umma_commit_elect(bar(kBarEmpty + sv_lo));
        umma_commit_elect(bar(kBarEmpty + sp));
      }
      if (!failed) umma_commit_elect(bar(kBarC));
    } else if (warp >= kWarpEpi0 && warp < kWarpEpi0 + kEpiWarps) {
      // lane quarter q (TMEM lane = head dim 32 q + lane), columns kMoverCols ch ..
      const int q = warp % 4, ch = (warp - kWarpEpi0) / 4;
      const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;
      const int dim = 32 * q + lane;
      if (!mbar_wait_warp(bar(kBarC), units_done & 1, err, kDetailC)) {
        failed = true;
      } else {
        tc_fence_after();
#pragma unroll
        for (int part = 0; part < kMoverCols / 16; ++part) {
          const int col = kMoverCols * ch + 16 * part;
          uint32_t x0[16], x1[16];
          tmem_ld16(tbase + lane_off + static_cast<uint32_t>(col), x0);
          tmem_ld16(tbase + lane_off + static_cast<uint32_t>(kRows + col), x1);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int r = col + j;
            if (r < n_rows)
              p.coarse[(static_cast<size_t>(bh) * T_cap + q0 + r) * kHeadDim + dim] =
                  (__uint_as_float(x0[j]) + __uint_as_float(x1[j])) / l_row[r];
          }
        }
        tc_fence_before();
      }
    }
    ring0 += 3 * n_chunks;
    ++units_done;
    failed = __syncthreads_or(failed);
    if (failed) break;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) tmem_dealloc(tbase, kTmemCols);
}

// The pooled q, k, v (fp32 [B, H, T_cap, 128]) as bf16 hi and lo rows
// ([B H][tp_cap][128] each, x ~ hi + lo), rows past the request's T zero.
// One thread per 8 channels of one row of one tensor.
__global__ void __launch_bounds__(256)
split_kernel(const float* __restrict__ pq, const float* __restrict__ pk, const float* __restrict__ pv,
             uint4* __restrict__ out, Geometry cap, DeviceLengths dl, int tp_cap) {
  const DynGeom dg = dyn_geom(cap, dl);
  if (!dg.valid) return;  // reported by the coarse kernel
  const size_t per_tensor = static_cast<size_t>(cap.B) * cap.H * tp_cap * (kHeadDim / 8);
  size_t idx = static_cast<size_t>(blockIdx.x) * 256 + threadIdx.x;
  if (idx >= 3 * per_tensor) return;
  const int tensor = static_cast<int>(idx / per_tensor);
  idx -= tensor * per_tensor;
  const int c8 = static_cast<int>(idx % (kHeadDim / 8));
  const size_t row = idx / (kHeadDim / 8);
  const int t = static_cast<int>(row % tp_cap);
  const size_t bh = row / tp_cap;
  float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (t < dg.T) {
    const float* src = (tensor == 0 ? pq : tensor == 1 ? pk : pv) + (bh * cap.T + t) * kHeadDim + 8 * c8;
    const float4 a = __ldg(reinterpret_cast<const float4*>(src));
    const float4 b = __ldg(reinterpret_cast<const float4*>(src) + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
  uint32_t hi[4], lo[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) split_bf16_pair(x[2 * i], x[2 * i + 1], hi[i], lo[i]);
  // tensor-major: [tensor][hi, lo][B H][tp_cap][128]
  out[(2 * tensor) * per_tensor + idx] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
  out[(2 * tensor + 1) * per_tensor + idx] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
}

template <int NM>
cudaError_t launch_nm(const CUtensorMap (&maps)[7], const CoarseParams& p, int grid, cudaStream_t stream) {
  constexpr uint32_t kSmemBytes = smem_bytes_of(NM);
  cudaError_t e = cudaFuncSetAttribute(coarse_tc_kernel<NM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  coarse_tc_kernel<NM><<<grid, threads_of(NM), kSmemBytes, stream>>>(maps[0], maps[1], maps[2], maps[3], maps[4],
                                                              maps[5], maps[6], p);
  return cudaGetLastError();
}

}  // namespace

int coarse_tc_padded(const Geometry& g) { return (g.T + kChunk - 1) / kChunk * kChunk; }

bool coarse_tc_supported(const Geometry& g) { return g.T <= kCoarseTcMaxT; }

int coarse_tc_units(const Geometry& g) { return g.B * g.H * ((g.T + kRows - 1) / kRows); }

size_t coarse_tc_operand_bytes(const Geometry& g) {
  return 6 * static_cast<size_t>(g.B) * g.H * coarse_tc_padded(g) * kHeadDim * 2;
}

size_t coarse_tc_scratch_bytes(const Geometry& g) {
  const int slots = coarse_tc_units(g) < kCoarseTcMaxSlots ? coarse_tc_units(g) : kCoarseTcMaxSlots;
  return static_cast<size_t>(slots) * kRows * coarse_tc_padded(g) * sizeof(float);
}

cudaError_t launch_split(const Geometry& g, const float* pq, const float* pk, const float* pv, void* operands,
                         const DeviceLengths& dl, cudaStream_t stream) {
  const int tp = coarse_tc_padded(g);
  const size_t n = 3 * static_cast<size_t>(g.B) * g.H * tp * (kHeadDim / 8);
  split_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(pq, pk, pv, static_cast<uint4*>(operands),
                                                                           g, dl, tp);
  return cudaGetLastError();
}

cudaError_t launch_coarse_tc(const Geometry& g, const CUtensorMap (&maps)[7], float* scratch, float* coarse,
                             int32_t* tile_index, unsigned int* err, const DeviceLengths& dl, int num_sms,
                             cudaStream_t stream) {
  CoarseParams p;
  p.cap = g;
  p.dl = dl;
  p.tp_cap = coarse_tc_padded(g);
  p.n_units = coarse_tc_units(g);
  p.scratch = scratch;
  p.coarse = coarse;
  p.tile_index = tile_index;
  p.err = err;
  int grid = p.n_units < num_sms ? p.n_units : num_sms;
  if (grid > kCoarseTcMaxSlots) grid = kCoarseTcMaxSlots;
  // a query row's scores in NM float4 registers per lane (the same results
  // for any NM that holds the row: entries past T take no part)
  static_assert(kCoarseTcMaxT <= 128 * 18, "rows held in at most 18 float4 registers per lane");
  if (g.T <= 128 * 5) return launch_nm<5>(maps, p, grid, stream);
  if (g.T <= 128 * 10) return launch_nm<10>(maps, p, grid, stream);
  return launch_nm<18>(maps, p, grid, stream);
}

}  // namespace vsa
