// Device helpers shared by the kernels that rank pooled tiles (the coarse
// attention + top-k, and the SubBlock router):
//   * fp32 products on the tensor cores with mma.sync bf16 m16n8k16, each
//     operand split into a bf16 head and a bf16 remainder so that a*b is
//     hi*hi + hi*lo + lo*hi, dropping only the lo*lo term (~2^-16 relative);
//   * a warp-per-row exact top-k: a radix select over the order-preserving
//     integer image of the fp32 scores, four passes of 8-bit digits each
//     counted in a 256-bin shared-memory histogram, then an in-order
//     compaction that writes the selected indices ascending (ties to the
//     lower index; deterministic);
//   * a faster warp top-k for rows without ties at the cut: a search for a
//     threshold with exactly k scores at or above it, counting with compares
//     and warp reductions only (no shared-memory atomics); rows where no such
//     threshold exists (equal scores at the cut) or that hold a non-finite
//     score fall back to the radix select, so the result is the same set.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

namespace vsa {

constexpr int kBins = 256;  // radix-select histogram bins (one histogram per warp)

// Order-preserving map from fp32 to uint32 (larger float -> larger key);
// -0 and +0 map to the same key.
__device__ __forceinline__ uint32_t order_key(float s) {
  uint32_t u = __float_as_uint(s);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// bf16 hi/lo split of two consecutive values (x ~ hi + lo, hi = bf16(x),
// lo = bf16(x - hi)), packed as bf16x2 words
__device__ __forceinline__ void split_bf16_pair(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// c += a b from bf16 hi/lo fragments in the m16n8k16 "tile8" form: t0, t1 =
// {hi a, hi b, lo a, lo b} of A rows g and g + 8 (a = k 2 t4, 2 t4 + 1; b = the
// same + 8), bf = the same form of B column g. Small terms first.
__device__ __forceinline__ void mma_bf16x3(float (&c)[4], const uint4& t0, const uint4& t1, const uint4& bf) {
  mma_bf16(c, t0.z, t1.z, t0.w, t1.w, bf.x, bf.y);   // lo . hi
  mma_bf16(c, t0.x, t1.x, t0.y, t1.y, bf.z, bf.w);   // hi . lo
  mma_bf16(c, t0.x, t1.x, t0.y, t1.y, bf.x, bf.y);   // hi . hi
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(addr));
  return r;
}

// The k largest of row[0 .. T) by one warp: their indices, ascending, into
// dst[0 .. k). Equal scores go to the lower index. h: this warp's kBins ints
// of shared memory.
__device__ __forceinline__ void warp_select_topk(const float* row, int T, int k, int* h, int32_t* dst,
                                                 int lane) {
  const unsigned full = 0xffffffffu;
  const unsigned lt_mask = (1u << lane) - 1u;
  // radix select, 8 bits per pass from the top: prefix holds the digits of
  // the k-th largest key fixed so far, rem how many keys above it are
  // still to be taken among those that match the prefix
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

// The k largest of row[0 .. T), as warp_select_topk, for rows whose entries
// T .. tpad - 1 hold -inf (tpad >= T a multiple of 4, row 16-byte aligned). The
// count c(x) = #{j : row[j] >= x} falls as x rises; the search keeps lo with
// c(lo) > k and hi with c(hi) < k. The first try is the row's mean plus its
// standard deviation times the normal quantile of 1 - k/T; later tries are the
// point where the straight line between (lo, c(lo) - k) and (hi, c(hi) - k)
// crosses zero, with the Illinois rule (an end kept twice in a row has its
// value halved), so the bracket keeps shrinking from both sides. Emulated on
// 1,134-score rows with k = 227 (normal, log-normal, log-sum-exp-like and
// bimodal scores), this takes 4-7 counting passes on average, against 9-14
// for plain interpolation with a midpoint every third try. A try with
// c(x) == k separates the k-th largest score from the (k+1)-th: the k scores
// >= x are the selection, the same set the radix select returns. Brackets that
// can no longer be split (equal scores at the cut), non-finite scores and the
// iteration limit hand the row to warp_select_topk.
__device__ __forceinline__ void warp_select_topk_count(const float* row, int T, int tpad, int k, int* h,
                                                       int32_t* dst, int lane) {
  const unsigned full = 0xffffffffu;
  if (k >= T) {
    for (int j = lane; j < T; j += 32) dst[j] = j;
    return;
  }
  float vmin = INFINITY, vmax = -INFINITY, s1 = 0.f, s2 = 0.f;
  bool bad = false;
  for (int j = lane; j < T; j += 32) {
    const float x = row[j];
    vmin = fminf(vmin, x);
    vmax = fmaxf(vmax, x);
    s1 += x;
    s2 = fmaf(x, x, s2);
    bad |= !(fabsf(x) <= 3.0e38f);  // NaN or +-inf (or close to overflow)
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    vmin = fminf(vmin, __shfl_xor_sync(full, vmin, o));
    vmax = fmaxf(vmax, __shfl_xor_sync(full, vmax, o));
    s1 += __shfl_xor_sync(full, s1, o);
    s2 += __shfl_xor_sync(full, s2, o);
  }
  float theta = 0.f;
  bool found = false;
  if (!__any_sync(full, bad) && k >= 1) {
    const float4* r4 = reinterpret_cast<const float4*>(row);
    const int n4 = tpad / 4;
    auto count_ge = [&](float x) {
      int c = 0;
      for (int i = lane; i < n4; i += 32) {
        const float4 v = r4[i];
        c += (v.x >= x) + (v.y >= x) + (v.z >= x) + (v.w >= x);
      }
      return static_cast<int>(__reduce_add_sync(full, static_cast<unsigned>(c)));
    };
    float lo = vmin, hi = nextafterf(vmax, INFINITY);
    float flo = static_cast<float>(T - k), fhi = static_cast<float>(-k);  // c - k at the ends (Illinois weights)
    int kept = 0;                                                         // +1: lo moved last, -1: hi
    const float mean = s1 / static_cast<float>(T);
    const float sd = sqrtf(fmaxf(s2 / static_cast<float>(T) - mean * mean, 0.f));
    float x = mean + normcdfinvf(1.f - static_cast<float>(k) / static_cast<float>(T)) * sd;
#pragma unroll 1
    for (int it = 0; it < 48; ++it) {
      if (it > 0) x = lo + (hi - lo) * (flo / (flo - fhi));
      if (!(x > lo && x < hi)) x = 0.5f * (lo + hi);
      if (!(x > lo && x < hi)) break;  // lo and hi adjacent: equal scores at the cut
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
  if (!found) {
    warp_select_topk(row, T, k, h, dst, lane);
    return;
  }
  const unsigned lt_mask = (1u << lane) - 1u;
  int written = 0;
  for (int base = 0; base < T; base += 32) {
    const int j = base + lane;
    const bool sel = j < T && row[j] >= theta;
    const unsigned selb = __ballot_sync(full, sel);
    if (sel) dst[written + __popc(selb & lt_mask)] = j;
    written += __popc(selb);
  }
}

}  // namespace vsa
