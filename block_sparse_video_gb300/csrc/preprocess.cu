// Fused attention preprocessing (HBM-bound), per "UniServe: serving FastH3 at
// its fastest", section "Fused attention preprocessing". One pass over the
// projected rows does all of the following:
//   * learned Q/K RMSNorm;
//   * partial RoPE;
//   * tile packing (gathering each attention token's projection row, so that
//     capacity padding never reaches a later kernel);
//   * the gate copy;
//   * the FP32 tile pooling of the packed Q, K and V over each video tile's
//     valid tokens.
// The packed bf16 tensors and the pooled statistics land directly in the
// buffers the coarse and fine kernels read. Section "The Kernel Layer" of
// the SGLang Diffusion benchmark page (MiniMax-H3 on 8x H200) fixes two details: the normalised value is rounded to bf16 before RoPE is applied,
// and the rotary width (96 of 128 channels there).
//
// Conventions where the page is silent:
//   * the norm runs per (token, head) over the head's 128 channels, with one
//     weight per (head, channel);
//   * RoPE rotates channels [0, rope_dim) and passes the rest through;
//   * pairs are (2i, 2i+1) or (i, i + rope_dim/2);
//   * the pair (a, b) becomes (a cos - b sin, a sin + b cos), with cos and
//     sin read from per-token tables.
//
// Work split: a CTA owns one 64-row tile of the attention sequence (a prefix
// tile or a video tile) for up to 8 heads. Its rows stream through a 3-stage
// shared-memory ring. A stage holds 2 rows x 4 tensors x 8 heads (16 KB) plus
// the two rows' RoPE cos/sin. A producer thread fills the ring with untiled
// bulk copies, completing on the stage's full barrier: one copy per
// projection row and tensor (the 8-head slice, 2 KB contiguous), and one per
// table for the stage's two rows. Four consumer warps work only from shared
// memory, so each row's chain has no global-memory latency in it. A thread
// owns 8 channels (16 bytes) of one head. The 16 threads of a head reduce the
// sum of squares with shuffles. The thread writes the four packed rows with
// 16-byte stores, keeps the Q/K/V tile sums in registers, and releases the
// stage on its empty barrier. The two rows of a stage are independent chains
// the compiler interleaves. Three CTAs fit on an SM, which keeps up to six
// stages (about 100 KB) of loads in flight per SM without holding them in
// registers.
#include "kernels.cuh"
#include "ptx.cuh"

namespace vsa {
namespace {

constexpr int kHeadsPerCta = 8;
constexpr int kVecPerHead = kHeadDim / 8;
constexpr int kConsumers = kHeadsPerCta * kVecPerHead;  // 128 threads, 4 warps
constexpr int kPreThreads = kConsumers + 32;            // + the producer warp
constexpr int kRowsPerStage = 2;
constexpr int kStages = 3;
constexpr int kSlice = kHeadsPerCta * kHeadDim * 2;            // one row's 8-head slice of one tensor: 2 KB
constexpr int kTableRow = kHeadDim / 2 * 4;                     // cos or sin of one row, at most 256 B
constexpr int kTableOff = kRowsPerStage * 4 * kSlice;           // 16 KB of rows, then cos, then sin
constexpr int kStageBytes = kTableOff + 2 * kRowsPerStage * kTableRow;
constexpr int kRingBytes = kStages * kStageBytes;
constexpr int kWeightBytes = 2 * kHeadsPerCta * kHeadDim * 4;
constexpr size_t kPreSmem = kRingBytes + kWeightBytes + kTile * 4 + 2 * kStages * 8;

__device__ __forceinline__ void unpack(const uint4& w, float (&x)[8]) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(u[i] << 16);
    x[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ float round_bf16(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

// bf16-valued floats -> packed bf16 pairs (exact: the values are bf16 already)
__device__ __forceinline__ uint4 pack(const float (&x)[8]) {
  uint32_t u[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    u[i] = (__float_as_uint(x[2 * i]) >> 16) | (__float_as_uint(x[2 * i + 1]) & 0xFFFF0000u);
  return make_uint4(u[0], u[1], u[2], u[3]);
}

__device__ __forceinline__ float group_sum16(float v, unsigned mask) {
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) v += __shfl_xor_sync(mask, v, o);
  return v;
}

__device__ __forceinline__ float4 ld_shared_f4(uint32_t addr) {
  float4 r;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
               : "r"(addr));
  return r;
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(addr));
  return r;
}

constexpr unsigned int kDetailPreFull = 0x500;
constexpr unsigned int kDetailPreEmpty = 0x600;

__global__ void __launch_bounds__(kPreThreads, 3)
preprocess_kernel(PreprocessArgs a, Geometry cap) {
  // the plan's geometry is the layout (buffer rows N, pooled tiles T per (b, h)); with device
  // lengths the request's own P, Lv, T, TP place the tiles, and the tiles past them return
  const int H = cap.H, N = cap.N, T = cap.T;
  const DynGeom dg = dyn_geom(cap, a.dl);
  if (!dg.valid) {
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *a.dl.invalid = 1u;
    return;
  }
  const int P = dg.P, Lv = dg.Lv, TP = dg.TP;
  extern __shared__ __align__(128) uint8_t smem[];
  float* s_w = reinterpret_cast<float*>(smem + kRingBytes);          // [2][8][128]
  int* s_src = reinterpret_cast<int*>(smem + kRingBytes + kWeightBytes);
  const uint32_t ring = smem_u32(smem);
  const uint32_t bars = smem_u32(smem + kRingBytes + kWeightBytes + kTile * 4);
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (kStages + s); };

  const int tiles = cap.TP + cap.T;  // grid tiles per batch (the capacity)
  const int b = blockIdx.x / tiles;
  const int tile = blockIdx.x % tiles;
  if (tile >= TP + dg.T) return;      // uniform per CTA
  const bool video = tile >= TP;
  const int n0 = video ? P + (tile - TP) * kTile : tile * kTile;
  const int rows = video ? min(kTile, Lv - (tile - TP) * kTile) : min(kTile, P - n0);
  const int h_first = blockIdx.y * kHeadsPerCta;
  const int nh = min(kHeadsPerCta, H - h_first);
  const int n_stages = (rows + kRowsPerStage - 1) / kRowsPerStage;
  const int tid = threadIdx.x;

  // this tile's projection rows; an entry outside [0, rows_in) becomes -1 (a zero row)
  if (tid < rows) {
    const int n = n0 + tid;
    long long src = a.src_row ? static_cast<long long>(a.src_row[static_cast<size_t>(b) * N + n]) : n;
    if (src < 0 || src >= a.rows_in) {
      atomicCAS(a.err + 7, 0u, static_cast<unsigned int>(n) + 1u);
      src = -1;
    }
    s_src[tid] = static_cast<int>(src);
  }
  // weights as [tensor][head][half of the 8 channels][16 threads][4]: a warp's float4 reads are conflict-free
  for (int i = tid; i < nh * kHeadDim; i += kPreThreads) {
    const int hh = i / kHeadDim, c = i % kHeadDim;
    const int dst = ((hh * 2 + (c / 4) % 2) * kVecPerHead + c / 8) * 4 + c % 4;
    s_w[dst] = a.q_norm_weight[static_cast<size_t>(h_first) * kHeadDim + i];
    s_w[kHeadsPerCta * kHeadDim + dst] = a.k_norm_weight[static_cast<size_t>(h_first) * kHeadDim + i];
  }
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), kConsumers / 32);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (tid >= kConsumers) {
    // ---------------- producer: one thread streams the rows into the ring
    if (tid != kConsumers) return;
    const uint32_t slice = static_cast<uint32_t>(nh) * kHeadDim * 2;
    const size_t in_row = static_cast<size_t>(a.row_stride);
    const size_t in_base = static_cast<size_t>(b) * a.rows_in;
    const size_t col = static_cast<size_t>(h_first) * kHeadDim;
    int it = 0;
    for (; it < n_stages; ++it) {
      const int s = it % kStages;
      if (it >= kStages && !mbar_wait(empty_bar(s), ((it / kStages) - 1) & 1, a.err, kDetailPreEmpty))
        break;
      const int r_lo = it * kRowsPerStage, r_hi = min(rows, r_lo + kRowsPerStage);
      const uint32_t table_bytes = static_cast<uint32_t>((r_hi - r_lo) * a.rope_dim / 2 * 4);
      uint32_t bytes = 2 * table_bytes;
      for (int r = r_lo; r < r_hi; ++r)
        if (s_src[r] >= 0) bytes += 4 * slice;
      mbar_arrive_expect_tx(full_bar(s), bytes);
      if (table_bytes) {
        const size_t t_off = static_cast<size_t>(n0 + r_lo) * (a.rope_dim / 2);
        bulk_load(ring + s * kStageBytes + kTableOff, a.rope_cos + t_off, table_bytes, full_bar(s));
        bulk_load(ring + s * kStageBytes + kTableOff + kRowsPerStage * kTableRow, a.rope_sin + t_off,
                  table_bytes, full_bar(s));
      }
      for (int r = r_lo; r < r_hi; ++r) {
        const int src = s_src[r];
        if (src < 0) continue;
        const size_t off = (in_base + src) * in_row + col;
#pragma unroll
        for (int t = 0; t < 4; ++t)
          bulk_load(ring + s * kStageBytes + ((r - r_lo) * 4 + t) * kSlice, a.in[t] + off, slice, full_bar(s));
      }
    }
    if (it < n_stages) {
      // gave up: let the copies already issued land before the CTA ends
      for (int j = max(0, it - kStages); j < it; ++j)
        mbar_wait_drain(full_bar(j % kStages), (j / kStages) & 1, kWaitLimitNs);
    }
    return;
  }

  // ---------------- consumers
  const int lane = tid & 31;
  const unsigned mask = 0xFFFFu << (lane & 16);
  const int h_local = tid / kVecPerHead;
  const bool active = h_local < nh;  // whole 16-lane groups
  const int h = h_first + h_local;
  const int j = tid % kVecPerHead;
  const int d0 = j * 8;
  const int rd = a.rope_dim, half = rd / 2;
  const bool rotated = d0 < rd;
  // interleaved: this thread's 4 pairs use angles d0/2 .. d0/2 + 3
  // half split: this thread's 8 channels use angles p0 .. p0 + 7, partner lane +-half/8
  const bool first_half = d0 < half;
  const int p0 = a.rope_interleaved ? d0 / 2 : (first_half ? d0 : d0 - half);
  const int partner = a.rope_interleaved ? lane : (rotated ? (first_half ? lane + half / 8 : lane - half / 8) : lane);
  const uint32_t w_q = smem_u32(s_w) + static_cast<uint32_t>((h_local * 2 * kVecPerHead + j) * 16);
  const uint32_t w_k = w_q + kHeadsPerCta * kHeadDim * 4;
  const uint32_t my_off = static_cast<uint32_t>(h_local * kHeadDim * 2 + d0 * 2);

  float acc_q[8], acc_k[8], acc_v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc_q[i] = acc_k[i] = acc_v[i] = 0.f;
  const size_t row_elems = static_cast<size_t>(H) * kHeadDim;
  const size_t col = static_cast<size_t>(h) * kHeadDim + d0;
  const uint4 zero = make_uint4(0, 0, 0, 0);

  for (int it = 0; it < n_stages; ++it) {
    const int s = it % kStages;
    if (!mbar_wait_warp(full_bar(s), (it / kStages) & 1, a.err, kDetailPreFull)) return;
    const int r_lo = it * kRowsPerStage;
    const uint32_t stage = ring + s * kStageBytes;
    if (active) {
      bool live[kRowsPerStage];
      float q[kRowsPerStage][8], k[kRowsPerStage][8], ssq[kRowsPerStage], ssk[kRowsPerStage];
      uint4 wv[kRowsPerStage], wg[kRowsPerStage];
      // the rows' chains are independent; each step runs over both rows so that they overlap
#pragma unroll
      for (int u = 0; u < kRowsPerStage; ++u) {
        const int r = r_lo + u;
        live[u] = r < rows;
        const bool ok = live[u] && s_src[r] >= 0;
        const uint32_t base = stage + u * 4 * kSlice + my_off;
        unpack(ok ? ld_shared_v4(base) : zero, q[u]);
        unpack(ok ? ld_shared_v4(base + kSlice) : zero, k[u]);
        wv[u] = ok ? ld_shared_v4(base + 2 * kSlice) : zero;
        wg[u] = ok ? ld_shared_v4(base + 3 * kSlice) : zero;
        ssq[u] = 0.f;
        ssk[u] = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          ssq[u] = fmaf(q[u][i], q[u][i], ssq[u]);
          ssk[u] = fmaf(k[u][i], k[u][i], ssk[u]);
        }
      }
#pragma unroll
      for (int u = 0; u < kRowsPerStage; ++u) {
        ssq[u] = group_sum16(ssq[u], mask);
        ssk[u] = group_sum16(ssk[u], mask);
      }
      {
        const float4 q0 = ld_shared_f4(w_q), q1 = ld_shared_f4(w_q + kVecPerHead * 16);
        const float4 k0 = ld_shared_f4(w_k), k1 = ld_shared_f4(w_k + kVecPerHead * 16);
        const float fq[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        const float fk[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
#pragma unroll
        for (int u = 0; u < kRowsPerStage; ++u) {
          const float rq = rsqrtf(fmaf(ssq[u], 1.f / kHeadDim, a.eps));
          const float rk = rsqrtf(fmaf(ssk[u], 1.f / kHeadDim, a.eps));
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            q[u][i] = round_bf16(q[u][i] * rq * fq[i]);
            k[u][i] = round_bf16(k[u][i] * rk * fk[i]);
          }
        }
      }
      if (rd > 0) {
#pragma unroll
        for (int u = 0; u < kRowsPerStage; ++u) {
          const uint32_t tc = stage + kTableOff + static_cast<uint32_t>((u * half + p0) * 4);
          const uint32_t ts = tc + kRowsPerStage * kTableRow;
          if (a.rope_interleaved) {
            if (rotated) {
              const float4 c = ld_shared_f4(tc), sn = ld_shared_f4(ts);
              const float cc[4] = {c.x, c.y, c.z, c.w}, ss[4] = {sn.x, sn.y, sn.z, sn.w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float qa = q[u][2 * i], qb = q[u][2 * i + 1], ka = k[u][2 * i], kb = k[u][2 * i + 1];
                q[u][2 * i] = round_bf16(fmaf(qa, cc[i], -qb * ss[i]));
                q[u][2 * i + 1] = round_bf16(fmaf(qa, ss[i], qb * cc[i]));
                k[u][2 * i] = round_bf16(fmaf(ka, cc[i], -kb * ss[i]));
                k[u][2 * i + 1] = round_bf16(fmaf(ka, ss[i], kb * cc[i]));
              }
            }
          } else {
            // every lane of the head takes part in the exchange; only rotated lanes use it
            const uint4 mq = pack(q[u]), mk = pack(k[u]);
            uint4 oq, ok4;
            oq.x = __shfl_sync(mask, mq.x, partner); oq.y = __shfl_sync(mask, mq.y, partner);
            oq.z = __shfl_sync(mask, mq.z, partner); oq.w = __shfl_sync(mask, mq.w, partner);
            ok4.x = __shfl_sync(mask, mk.x, partner); ok4.y = __shfl_sync(mask, mk.y, partner);
            ok4.z = __shfl_sync(mask, mk.z, partner); ok4.w = __shfl_sync(mask, mk.w, partner);
            if (rotated) {
              float pq[8], pk[8];
              unpack(oq, pq);
              unpack(ok4, pk);
              const float4 c0 = ld_shared_f4(tc), c1 = ld_shared_f4(tc + 16);
              const float4 s0 = ld_shared_f4(ts), s1 = ld_shared_f4(ts + 16);
              const float cc[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
              const float ss[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                if (first_half) {  // this lane holds a, the partner b: a' = a cos - b sin
                  q[u][i] = round_bf16(fmaf(q[u][i], cc[i], -pq[i] * ss[i]));
                  k[u][i] = round_bf16(fmaf(k[u][i], cc[i], -pk[i] * ss[i]));
                } else {           // this lane holds b, the partner a: b' = a sin + b cos
                  q[u][i] = round_bf16(fmaf(pq[i], ss[i], q[u][i] * cc[i]));
                  k[u][i] = round_bf16(fmaf(pk[i], ss[i], k[u][i] * cc[i]));
                }
              }
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kRowsPerStage; ++u) {
        if (!live[u]) continue;
        const size_t out_off = (static_cast<size_t>(b) * N + n0 + r_lo + u) * row_elems + col;
        *reinterpret_cast<uint4*>(a.out[0] + out_off) = pack(q[u]);
        *reinterpret_cast<uint4*>(a.out[1] + out_off) = pack(k[u]);
        *reinterpret_cast<uint4*>(a.out[2] + out_off) = wv[u];
        *reinterpret_cast<uint4*>(a.out[3] + out_off) = wg[u];
        if (video) {
          float v[8];
          unpack(wv[u], v);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            acc_q[i] += q[u][i];
            acc_k[i] += k[u][i];
            acc_v[i] += v[i];
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_bar(s));
  }
  if (!video || !active || a.pooled[0] == nullptr) return;
  const int t = tile - TP;
  const float fn = static_cast<float>(rows);
  const size_t po = ((static_cast<size_t>(b) * H + h) * T + t) * kHeadDim + d0;
  auto store_mean = [&](float* dst, const float (&acc)[8]) {
    float4* o = reinterpret_cast<float4*>(dst + po);
    o[0] = make_float4(__fdiv_rn(acc[0], fn), __fdiv_rn(acc[1], fn), __fdiv_rn(acc[2], fn),
                       __fdiv_rn(acc[3], fn));
    o[1] = make_float4(__fdiv_rn(acc[4], fn), __fdiv_rn(acc[5], fn), __fdiv_rn(acc[6], fn),
                       __fdiv_rn(acc[7], fn));
  };
  store_mean(a.pooled[0], acc_q);
  store_mean(a.pooled[1], acc_k);
  store_mean(a.pooled[2], acc_v);
}

}  // namespace

cudaError_t launch_preprocess(const Geometry& g, const PreprocessArgs& a, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(preprocess_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kPreSmem));
  if (e != cudaSuccess) return e;
  dim3 grid(g.B * (g.TP + g.T), (g.H + kHeadsPerCta - 1) / kHeadsPerCta);
  preprocess_kernel<<<grid, kPreThreads, kPreSmem, stream>>>(a, g);
  return cudaGetLastError();
}

}  // namespace vsa
