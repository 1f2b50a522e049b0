// Fine attention of the VSA forward, with the gated coarse add fused into the
// epilogue ("UniServe: serving FastH3 at its fastest", sections "The FastH3
// workload" and "Fused output combination").
//
// One CTA processes one 64-token query tile:
//   * a prefix (text/audio) query tile attends to every key tile: the TP
//     prefix tiles, then the T video tiles; its output is the attention alone;
//   * a video query tile t attends to the TP prefix tiles and to its k selected
//     video tiles; its output adds sigmoid(gate) * coarse[t] per channel.
// Key tiles are processed two at a time (a 128-key block).
//
// Formulation: transposed, so that both tensor-core products have M = 128
// with a 64-row query tile:
//   S^T[128 keys x 64 queries] = K_blk[128 x 128] . Q^T           (A, B K-major)
//   O^T[128 dims x 64 queries] += V_blk^T[128 x 128 keys] . P^T   (A, B MN-major)
// S^T and O^T live in tensor memory (TMEM lane = key, resp. head dim; column =
// query). Each softmax thread owns one key lane for 32 query columns, so
// masking a ragged or absent key tile is a per-thread select. The online
// softmax keeps, per query column, a reference m (log2 units) shared by every
// lane; a block whose scores all stay below m + 8 (P <= 256) needs no cross-
// lane work. Otherwise (always on the first block) a slow path reduces the
// exact block maximum across the 128 lanes, raises m, and rescales the row
// sums and O^T. Row sums are per-lane partials, reduced once at the end.
//
// Warp roles (320 threads): warp 0 issues TMA loads (Q once; K and V blocks
// into 3- and 2-stage rings); warp 1 owns TMEM and issues tcgen05.mma; warps
// 2-5 and 6-9 are two softmax warpgroups (query columns 0-31 and 32-63) that
// also run the epilogue. Every wait is bounded (see ptx.cuh).
#include "kernels.cuh"
#include "ptx.cuh"

namespace vsa {
namespace {

constexpr int kThreads = 320;
constexpr int kNumK = 3;
constexpr int kNumV = 2;
constexpr uint32_t kQBytes = 64 * kHeadDim * 2;    // 16 KB
constexpr uint32_t kKVBytes = 128 * kHeadDim * 2;  // 32 KB, one 128-key block
constexpr uint32_t kPBytes = 128 * 64 * 2;         // 16 KB
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS1 = 64;  // S^T buffer b at column b * kColS1
constexpr uint32_t kColO = 128;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P never exceeds 2^8

constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kQBytes;
constexpr uint32_t kOffV = kOffK + kNumK * kKVBytes;
constexpr uint32_t kOffP = kOffV + kNumV * kKVBytes;
constexpr uint32_t kOffBar = kOffP + 2 * kPBytes;
constexpr uint32_t kOffRed = kOffBar + 256;
constexpr uint32_t kOffSlot = kOffRed + 2 * 32 * 4 * 4;
constexpr uint32_t kSmemBytes = kOffSlot + 16 + 1024;  // + 1024-byte alignment slack

// barrier indices
constexpr int kBarQ = 0;
constexpr int kBarKFull = 1;
constexpr int kBarKEmpty = kBarKFull + kNumK;
constexpr int kBarVFull = kBarKEmpty + kNumK;
constexpr int kBarVEmpty = kBarVFull + kNumV;
constexpr int kBarSFull = kBarVEmpty + kNumV;
constexpr int kBarSEmpty = kBarSFull + 2;
constexpr int kBarPFull = kBarSEmpty + 2;
constexpr int kBarPEmpty = kBarPFull + 2;
constexpr int kNumBars = kBarPEmpty + 2;
static_assert(kNumBars * 8 <= 256, "barrier area");

struct FineParams {
  int B, H, P, Lv, N, T, TP, k;
  int n_prefix_items;
  float scale_log2;
  const __nv_bfloat16* gate;
  __nv_bfloat16* out;
  const float* coarse;
  const int32_t* tile_index;
  unsigned int* err;
};

struct Item {
  int b, h, t;
  bool video;
  int q_row0, q_valid;
  int n_kv;
  const int32_t* list;  // selected video tiles, or null: every video tile in order
};

__device__ __forceinline__ Item decode_item(const FineParams& p, int item) {
  Item it;
  if (item < p.n_prefix_items) {
    it.video = false;
    it.b = item / (p.H * p.TP);
    const int rem = item % (p.H * p.TP);
    it.h = rem / p.TP;
    it.t = rem % p.TP;
    it.q_row0 = it.t * kTile;
    it.q_valid = min(kTile, p.P - it.q_row0);
    it.n_kv = p.TP + p.T;
    it.list = nullptr;
  } else {
    const int v = item - p.n_prefix_items;
    it.video = true;
    it.b = v / (p.H * p.T);
    const int rem = v % (p.H * p.T);
    it.h = rem / p.T;
    it.t = rem % p.T;
    it.q_row0 = p.P + it.t * kTile;
    it.q_valid = min(kTile, p.Lv - it.t * kTile);
    it.n_kv = p.TP + p.k;
    it.list = p.tile_index + ((static_cast<size_t>(it.b) * p.H + it.h) * p.T + it.t) * p.k;
  }
  return it;
}

// Valid keys of key tile `ti` of an item whose video tile id is `jv`.
__device__ __forceinline__ int kv_tile_len(const FineParams& p, const Item& it, int ti, int jv) {
  if (ti >= it.n_kv) return 0;
  if (ti < p.TP) return min(kTile, p.P - ti * kTile);
  return min(kTile, p.Lv - jv * kTile);
}

__device__ __forceinline__ int kv_tile_id(const Item& it, int tp, int ti) {
  if (ti < tp || ti >= it.n_kv) return 0;
  return it.list ? __ldg(it.list + (ti - tp)) : ti - tp;
}

// Reduce 32 per-lane column values across the warp; afterwards lane c holds the
// reduction of column c. The input array is consumed.
template <bool kMax>
__device__ __forceinline__ float reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = upper ? v[i] : v[i + o];
      const float keep = upper ? v[i + o] : v[i];
      const float recv = __shfl_xor_sync(0xffffffffu, send, o);
      v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
    }
  }
  return v[0];
}

__device__ __forceinline__ bool warp_any(bool x) { return __any_sync(0xffffffffu, x); }

__global__ void __launch_bounds__(kThreads, 1)
fine_attn_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                 const __grid_constant__ CUtensorMap map_v, const FineParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t s_base = smem_u32(smem);
  const uint32_t sQ = s_base + kOffQ;
  const uint32_t sK = s_base + kOffK;
  const uint32_t sV = s_base + kOffV;
  const uint32_t sP = s_base + kOffP;
  auto bar = [&](int i) { return s_base + kOffBar + 8u * static_cast<uint32_t>(i); };
  float* red = reinterpret_cast<float*>(smem + kOffRed);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + kOffSlot);

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  unsigned int* err = p.err;
  const Item it = decode_item(p, blockIdx.x);
  const int nblk = (it.n_kv + 1) / 2;

  if (tid == 0) {
    mbar_init(bar(kBarQ), 1);
    for (int s = 0; s < kNumK; ++s) { mbar_init(bar(kBarKFull + s), 1); mbar_init(bar(kBarKEmpty + s), 1); }
    for (int s = 0; s < kNumV; ++s) { mbar_init(bar(kBarVFull + s), 1); mbar_init(bar(kBarVEmpty + s), 1); }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kBarSFull + s), 1);
      mbar_init(bar(kBarSEmpty + s), 8);
      mbar_init(bar(kBarPFull + s), 8);
      mbar_init(bar(kBarPEmpty + s), 1);
    }
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tslot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    bool failed = abort_raised(err);
    if (lane == 0 && !failed) {
      prefetch_tensor_map(&map_q);
      prefetch_tensor_map(&map_k);
      prefetch_tensor_map(&map_v);
      mbar_arrive_expect_tx(bar(kBarQ), kQBytes);
      for (int c = 0; c < 2; ++c)
        tma_load_4d(sQ + c * 8192, &map_q, 64 * c, it.h, it.q_row0, it.b, bar(kBarQ));
    }
    // window of 32 selected tile ids (video items), prefetched one window ahead
    int wbase = 0;
    int win = 0, win_next = 0;
    if (it.list) {
      win = lane < p.k ? __ldg(it.list + lane) : 0;
      win_next = 32 + lane < p.k ? __ldg(it.list + 32 + lane) : 0;
    }
    auto tile_row = [&](int ti) -> int {
      if (ti >= it.n_kv) return p.N;  // absent: fully out of bounds, TMA fills zeros
      if (ti < p.TP) return ti * kTile;
      const int pos = ti - p.TP;
      int j = pos;
      if (it.list) {
        while (pos >= wbase + 32) {
          wbase += 32;
          win = win_next;
          win_next = wbase + 32 + lane < p.k ? __ldg(it.list + wbase + 32 + lane) : 0;
        }
        j = __shfl_sync(0xffffffffu, win, pos - wbase);
      }
      return p.P + j * kTile;
    };
    int prev_ra = 0, prev_rb = 0;
    for (int step = 0; step <= nblk && !failed; ++step) {
      int ra = 0, rb = 0;
      if (step < nblk) {
        ra = tile_row(2 * step);
        rb = tile_row(2 * step + 1);
        if (lane == 0) {
          const int s = step % kNumK;
          const uint32_t par = ((step / kNumK) & 1) ^ 1;
          if (mbar_wait(bar(kBarKEmpty + s), par, err, 0x100u)) {
            const uint32_t dst = sK + s * kKVBytes;
            mbar_arrive_expect_tx(bar(kBarKFull + s), kKVBytes);
            for (int c = 0; c < 2; ++c) {
              tma_load_4d(dst + c * 16384, &map_k, 64 * c, it.h, ra, it.b, bar(kBarKFull + s));
              tma_load_4d(dst + c * 16384 + 8192, &map_k, 64 * c, it.h, rb, it.b, bar(kBarKFull + s));
            }
          } else {
            failed = true;
          }
        }
      }
      if (step >= 1 && lane == 0 && !failed) {
        const int vb = step - 1;
        const int s = vb % kNumV;
        const uint32_t par = ((vb / kNumV) & 1) ^ 1;
        if (mbar_wait(bar(kBarVEmpty + s), par, err, 0x200u)) {
          const uint32_t dst = sV + s * kKVBytes;
          mbar_arrive_expect_tx(bar(kBarVFull + s), kKVBytes);
          for (int c = 0; c < 2; ++c) {
            tma_load_4d(dst + c * 16384, &map_v, 64 * c, it.h, prev_ra, it.b, bar(kBarVFull + s));
            tma_load_4d(dst + c * 16384 + 8192, &map_v, 64 * c, it.h, prev_rb, it.b, bar(kBarVFull + s));
          }
        } else {
          failed = true;
        }
      }
      failed = __shfl_sync(0xffffffffu, failed, 0);
      prev_ra = ra;
      prev_rb = rb;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16_f32(128, 64, 0, 0);
      const uint32_t id_o = idesc_bf16_f32(128, 64, 1, 1);
      auto issue_pv = [&](int j) -> bool {
        const int vs = j % kNumV, pb = j & 1;
        if (!mbar_wait(bar(kBarVFull + vs), (j / kNumV) & 1, err, 0x300u)) return false;
        if (!mbar_wait(bar(kBarPFull + pb), (j >> 1) & 1, err, 0x400u)) return false;
        tc_fence_after();
        const uint32_t va = sV + vs * kKVBytes, pa = sP + pb * kPBytes;
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const uint64_t a = smem_desc_sw128(va + s * 2048, 16384, 1024);
          const uint64_t b = smem_desc_sw128(pa + s * 2048, 8192, 1024);
          umma_bf16(tbase + kColO, a, b, id_o, (j > 0 || s > 0) ? 1u : 0u);
        }
        umma_commit(bar(kBarVEmpty + vs));
        umma_commit(bar(kBarPEmpty + pb));
        return true;
      };
      bool ok = mbar_wait(bar(kBarQ), 0, err, 0x500u);
      for (int i = 0; i < nblk && ok; ++i) {
        const int ks = i % kNumK, sb = i & 1;
        ok = mbar_wait(bar(kBarKFull + ks), (i / kNumK) & 1, err, 0x600u) &&
             mbar_wait(bar(kBarSEmpty + sb), ((i >> 1) & 1) ^ 1, err, 0x700u);
        if (!ok) break;
        tc_fence_after();
        const uint32_t ka = sK + ks * kKVBytes;
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const uint64_t a = smem_desc_sw128(ka + (s >> 2) * 16384 + (s & 3) * 32, 16, 1024);
          const uint64_t b = smem_desc_sw128(sQ + (s >> 2) * 8192 + (s & 3) * 32, 16, 1024);
          umma_bf16(tbase + sb * kColS1, a, b, id_s, s > 0 ? 1u : 0u);
        }
        umma_commit(bar(kBarKEmpty + ks));
        umma_commit(bar(kBarSFull + sb));
        if (i >= 1) ok = issue_pv(i - 1);
      }
      if (ok) issue_pv(nblk - 1);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int wg = (warp - 2) / 4;          // query columns 32*wg .. 32*wg+31
    const int q4 = warp % 4;                // TMEM lane quarter this warp may access
    const int r = 32 * q4 + lane;           // key lane (softmax), head dim (epilogue)
    const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
    const uint32_t bar_id = 1 + wg;
    const float sl2 = p.scale_log2;
    float m[32], l[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) { m[c] = -INFINITY; l[c] = 0.f; }
    bool failed = false;
    int j_cur = kv_tile_id(it, p.TP, r >> 6);
    for (int i = 0; i < nblk; ++i) {
      const int sb = i & 1;
      const int ti = 2 * i + (r >> 6);
      const int j_nxt = kv_tile_id(it, p.TP, ti + 2);
      const bool valid = (r & 63) < kv_tile_len(p, it, ti, j_cur);
      j_cur = j_nxt;

      failed = warp_any(failed || !mbar_wait(bar(kBarSFull + sb), (i >> 1) & 1, err, 0x800u));
      float s[32];
      if (!failed) {
        tc_fence_after();
        uint32_t raw[32];
        tmem_ld32(tbase + lane_off + sb * kColS1 + 32 * wg, raw);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 32; ++c) s[c] = __uint_as_float(raw[c]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarSEmpty + sb));
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) s[c] = 0.f;
      }
      float t[32];
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        t[c] = valid ? fmaf(s[c], sl2, -m[c]) : -INFINITY;
        mx = fmaxf(mx, t[c]);
      }
      if (named_bar_or(bar_id, 128, failed || mx > kRescaleThreshold)) {
        if (named_bar_or(bar_id, 128, failed)) { failed = true; break; }
        // slow path: exact block maximum per query column across the 128 key lanes
        float u[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) u[c] = valid ? s[c] * sl2 : -INFINITY;
        const float wmax = reduce_scatter32<true>(u, lane);
        red[(wg * 32 + lane) * 4 + q4] = wmax;
        named_bar_sync(bar_id, 128);
        float alpha[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float4 x = reinterpret_cast<const float4*>(red)[wg * 32 + c];
          const float bm = fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w));
          const float mn = fmaxf(m[c], bm);
          alpha[c] = ex2_approx(m[c] - mn);
          l[c] *= alpha[c];
          m[c] = mn;
        }
        if (i > 0) {
          // O^T must hold every PV product issued so far: wait for PV of block
          // i-1 on its P-buffer barrier (PV of block i-3 is already known to be
          // complete, so this parity wait cannot alias an older phase; tcgen05
          // MMAs complete in issue order).
          const int pj = i - 1;
          failed = warp_any(!mbar_wait(bar(kBarPEmpty + (pj & 1)), (pj >> 1) & 1, err, 0x900u));
          if (!failed) {
            tc_fence_after();
            uint32_t o[32];
            tmem_ld32(tbase + lane_off + kColO + 32 * wg, o);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha[c]);
            tmem_st32(tbase + lane_off + kColO + 32 * wg, o);
            tmem_wait_st();
            tc_fence_before();
          }
        }
#pragma unroll
        for (int c = 0; c < 32; ++c) t[c] = valid ? fmaf(s[c], sl2, -m[c]) : -INFINITY;
      }
      uint32_t pk[16];
#pragma unroll
      for (int c = 0; c < 32; c += 2) {
        const float p0 = ex2_approx(t[c]), p1 = ex2_approx(t[c + 1]);
        l[c] += p0;
        l[c + 1] += p1;
        pk[c / 2] = pack_bf16x2(p0, p1);
      }
      failed = warp_any(failed || !mbar_wait(bar(kBarPEmpty + sb), ((i >> 1) & 1) ^ 1, err, 0xA00u));
      if (!failed) {
        const uint32_t row = sP + sb * kPBytes + r * 128;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const uint32_t chunk = static_cast<uint32_t>((4 * wg + cc) ^ (r & 7));
          st_shared_v4(row + chunk * 16, pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarPFull + sb));
      }
    }
    // ---- epilogue: out = O / l (+ sigmoid(gate) * coarse on video rows)
    if (!named_bar_or(bar_id, 128, failed)) {
      const float lw = reduce_scatter32<false>(l, lane);
      red[(wg * 32 + lane) * 4 + q4] = lw;
      named_bar_sync(bar_id, 128);
      const int pj = nblk - 1;  // the last PV product (see the rescale above)
      failed = warp_any(!mbar_wait(bar(kBarPEmpty + (pj & 1)), (pj >> 1) & 1, err, 0xB00u));
      if (!failed) {
        tc_fence_after();
        uint32_t o[32];
        tmem_ld32(tbase + lane_off + kColO + 32 * wg, o);
        tmem_wait_ld();
        const int d = r;
        float cz = 0.f;
        if (it.video)
          cz = __ldg(p.coarse + ((static_cast<size_t>(it.b) * p.H + it.h) * p.T + it.t) * kHeadDim + d);
#pragma unroll 4
        for (int c = 0; c < 32; ++c) {
          const int qc = 32 * wg + c;
          if (qc < it.q_valid) {
            const float4 x = reinterpret_cast<const float4*>(red)[wg * 32 + c];
            const float lsum = (x.x + x.y) + (x.z + x.w);
            float val = __uint_as_float(o[c]) / lsum;
            const size_t off =
                ((static_cast<size_t>(it.b) * p.N + it.q_row0 + qc) * p.H + it.h) * kHeadDim + d;
            if (it.video) {
              const float g = __bfloat162float(p.gate[off]);
              val += cz / (1.0f + __expf(-g));
            }
            p.out[off] = __float2bfloat16_rn(val);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tbase, kTmemCols);
}

}  // namespace

size_t fine_smem_bytes() { return kSmemBytes; }

cudaError_t launch_fine(const Geometry& g, const CUtensorMap& map_q, const CUtensorMap& map_k,
                        const CUtensorMap& map_v, const FineArgs& a, cudaStream_t stream) {
  FineParams p;
  p.B = g.B; p.H = g.H; p.P = g.P; p.Lv = g.Lv; p.N = g.N; p.T = g.T; p.TP = g.TP; p.k = g.k;
  p.n_prefix_items = g.B * g.H * g.TP;
  p.scale_log2 = 1.4426950408889634f * 0.08838834764831845f;
  p.gate = a.gate;
  p.out = a.out;
  p.coarse = a.coarse;
  p.tile_index = a.tile_index;
  p.err = a.err;
  const long long n_items = static_cast<long long>(g.B) * g.H * (g.TP + g.T);
  cudaError_t e = cudaFuncSetAttribute(fine_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  fine_attn_kernel<<<static_cast<unsigned>(n_items), kThreads, kSmemBytes, stream>>>(map_q, map_k,
                                                                                     map_v, p);
  return cudaGetLastError();
}

}  // namespace vsa
