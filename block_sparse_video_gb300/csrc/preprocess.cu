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
// buffers the coarse and fine kernels read. Section "The Kernel Layer" fixes
// two details: the normalised value is rounded to bf16 before RoPE is applied,
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
// tile or a video tile) for 8 heads. A thread owns 8 channels (one 16-byte
// vector) of one head, and the 16 threads of a head reduce the sum of squares
// with shuffles. Each thread walks the tile's rows with two rows' loads in
// flight (8 x 16 B), writes the four packed rows, and keeps the Q/K/V tile
// sums of its 8 channels in registers.
#include "kernels.cuh"

namespace vsa {
namespace {

constexpr int kPreThreads = 128;  // 8 heads x 16 vectors
constexpr int kVecPerHead = kHeadDim / 8;

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

__global__ void __launch_bounds__(kPreThreads, 4)
preprocess_kernel(PreprocessArgs a, int H, int P, int Lv, int N, int T, int TP) {
  __shared__ int s_src[kTile];
  __shared__ __align__(16) float s_w[2][kPreThreads / kVecPerHead][kHeadDim];  // this CTA's heads' norm weights
  const int tiles = TP + T;
  const int b = blockIdx.x / tiles;
  const int tile = blockIdx.x % tiles;
  const bool video = tile >= TP;
  const int n0 = video ? P + (tile - TP) * kTile : tile * kTile;
  const int rows = video ? min(kTile, Lv - (tile - TP) * kTile) : min(kTile, P - n0);

  // this tile's projection rows; an entry outside [0, rows_in) becomes -1 (a zero row)
  if (threadIdx.x < rows) {
    const int n = n0 + threadIdx.x;
    long long src = a.src_row ? static_cast<long long>(a.src_row[static_cast<size_t>(b) * N + n]) : n;
    if (src < 0 || src >= a.rows_in) {
      atomicCAS(a.err + 7, 0u, static_cast<unsigned int>(n) + 1u);
      src = -1;
    }
    s_src[threadIdx.x] = static_cast<int>(src);
  }
  {
    const int h_first = blockIdx.y * (kPreThreads / kVecPerHead);
    const int n_w = min(kPreThreads / kVecPerHead, H - h_first) * kHeadDim;
    for (int i = threadIdx.x; i < n_w; i += kPreThreads) {
      s_w[0][0][i] = a.q_norm_weight[static_cast<size_t>(h_first) * kHeadDim + i];
      s_w[1][0][i] = a.k_norm_weight[static_cast<size_t>(h_first) * kHeadDim + i];
    }
  }
  __syncthreads();

  const int vec = blockIdx.y * kPreThreads + threadIdx.x;
  if (vec >= H * kVecPerHead) return;  // whole 16-lane groups leave together
  const int lane = threadIdx.x & 31;
  const unsigned mask = 0xFFFFu << (lane & 16);
  const int h = vec / kVecPerHead;
  const int d0 = (vec % kVecPerHead) * 8;
  const int h_local = threadIdx.x / kVecPerHead;

  const int rd = a.rope_dim, half = rd / 2;
  const bool rotated = d0 < rd;
  // interleaved: this thread's 4 pairs use angles d0/2 .. d0/2 + 3
  // half split: this thread's 8 channels use angles p0 .. p0 + 7, partner lane +-half/8
  const bool first_half = d0 < half;
  const int p0 = a.rope_interleaved ? d0 / 2 : (first_half ? d0 : d0 - half);
  const int partner = a.rope_interleaved ? lane : (rotated ? (first_half ? lane + half / 8 : lane - half / 8) : lane);

  float acc_q[8], acc_k[8], acc_v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc_q[i] = acc_k[i] = acc_v[i] = 0.f;

  const size_t in_row = static_cast<size_t>(a.row_stride);
  const size_t in_base = static_cast<size_t>(b) * a.rows_in;
  const size_t col = static_cast<size_t>(h) * kHeadDim + d0;
  const uint4 zero = make_uint4(0, 0, 0, 0);

  for (int r0 = 0; r0 < rows; r0 += 2) {
    uint4 w[2][4];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int r = r0 + u;
      const int src = r < rows ? s_src[r] : -1;
#pragma unroll
      for (int t = 0; t < 4; ++t)
        w[u][t] = src >= 0 ? __ldg(reinterpret_cast<const uint4*>(a.in[t] + (in_base + src) * in_row + col))
                           : zero;
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int r = r0 + u;
      if (r >= rows) break;  // uniform across the CTA
      const int n = n0 + r;
      float q[8], k[8];
      unpack(w[u][0], q);
      unpack(w[u][1], k);
      float ssq = 0.f, ssk = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        ssq = fmaf(q[i], q[i], ssq);
        ssk = fmaf(k[i], k[i], ssk);
      }
      ssq = group_sum16(ssq, mask);
      ssk = group_sum16(ssk, mask);
      const float rq = rsqrtf(fmaf(ssq, 1.f / kHeadDim, a.eps));
      const float rk = rsqrtf(fmaf(ssk, 1.f / kHeadDim, a.eps));
      {
        const float4* wq = reinterpret_cast<const float4*>(&s_w[0][h_local][d0]);
        const float4* wk = reinterpret_cast<const float4*>(&s_w[1][h_local][d0]);
        const float4 q0 = wq[0], q1 = wq[1], k0 = wk[0], k1 = wk[1];
        const float fq[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        const float fk[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          q[i] = round_bf16(q[i] * rq * fq[i]);
          k[i] = round_bf16(k[i] * rk * fk[i]);
        }
      }
      if (rd > 0) {
        const size_t trow = static_cast<size_t>(n) * half;
        if (a.rope_interleaved) {
          if (rotated) {
            const float4 c = __ldg(reinterpret_cast<const float4*>(a.rope_cos + trow + p0));
            const float4 s = __ldg(reinterpret_cast<const float4*>(a.rope_sin + trow + p0));
            const float cc[4] = {c.x, c.y, c.z, c.w}, ss[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float qa = q[2 * i], qb = q[2 * i + 1], ka = k[2 * i], kb = k[2 * i + 1];
              q[2 * i] = round_bf16(fmaf(qa, cc[i], -qb * ss[i]));
              q[2 * i + 1] = round_bf16(fmaf(qa, ss[i], qb * cc[i]));
              k[2 * i] = round_bf16(fmaf(ka, cc[i], -kb * ss[i]));
              k[2 * i + 1] = round_bf16(fmaf(ka, ss[i], kb * cc[i]));
            }
          }
        } else {
          // every lane of the head takes part in the exchange; only rotated lanes use it
          const uint4 mq = pack(q), mk = pack(k);
          uint4 oq, ok;
          oq.x = __shfl_sync(mask, mq.x, partner); oq.y = __shfl_sync(mask, mq.y, partner);
          oq.z = __shfl_sync(mask, mq.z, partner); oq.w = __shfl_sync(mask, mq.w, partner);
          ok.x = __shfl_sync(mask, mk.x, partner); ok.y = __shfl_sync(mask, mk.y, partner);
          ok.z = __shfl_sync(mask, mk.z, partner); ok.w = __shfl_sync(mask, mk.w, partner);
          if (rotated) {
            float pq[8], pk[8], cc[8], ss[8];
            unpack(oq, pq);
            unpack(ok, pk);
            const float4* tc = reinterpret_cast<const float4*>(a.rope_cos + trow + p0);
            const float4* ts = reinterpret_cast<const float4*>(a.rope_sin + trow + p0);
            const float4 c0 = __ldg(tc), c1 = __ldg(tc + 1), s0 = __ldg(ts), s1 = __ldg(ts + 1);
            cc[0] = c0.x; cc[1] = c0.y; cc[2] = c0.z; cc[3] = c0.w;
            cc[4] = c1.x; cc[5] = c1.y; cc[6] = c1.z; cc[7] = c1.w;
            ss[0] = s0.x; ss[1] = s0.y; ss[2] = s0.z; ss[3] = s0.w;
            ss[4] = s1.x; ss[5] = s1.y; ss[6] = s1.z; ss[7] = s1.w;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              if (first_half) {  // this lane holds a, the partner b: a' = a cos - b sin
                q[i] = round_bf16(fmaf(q[i], cc[i], -pq[i] * ss[i]));
                k[i] = round_bf16(fmaf(k[i], cc[i], -pk[i] * ss[i]));
              } else {           // this lane holds b, the partner a: b' = a sin + b cos
                q[i] = round_bf16(fmaf(pq[i], ss[i], q[i] * cc[i]));
                k[i] = round_bf16(fmaf(pk[i], ss[i], k[i] * cc[i]));
              }
            }
          }
        }
      }
      const size_t out_off = (static_cast<size_t>(b) * N + n) * static_cast<size_t>(H) * kHeadDim + col;
      *reinterpret_cast<uint4*>(a.out[0] + out_off) = pack(q);
      *reinterpret_cast<uint4*>(a.out[1] + out_off) = pack(k);
      *reinterpret_cast<uint4*>(a.out[2] + out_off) = w[u][2];
      *reinterpret_cast<uint4*>(a.out[3] + out_off) = w[u][3];
      if (video) {
        float v[8];
        unpack(w[u][2], v);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          acc_q[i] += q[i];
          acc_k[i] += k[i];
          acc_v[i] += v[i];
        }
      }
    }
  }
  if (!video) return;
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
  const int row_vecs = g.H * kVecPerHead;
  dim3 grid(g.B * (g.TP + g.T), (row_vecs + kPreThreads - 1) / kPreThreads);
  preprocess_kernel<<<grid, kPreThreads, 0, stream>>>(a, g.H, g.P, g.Lv, g.N, g.T, g.TP);
  return cudaGetLastError();
}

}  // namespace vsa
