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
// query). Each softmax thread owns one key lane for 16 query columns, so
// masking a ragged or absent key tile is a per-thread select. The online
// softmax keeps, per query column, a reference m (log2 units) shared by every
// lane; a block whose scores all stay below m + 8 (P <= 256) needs no cross-
// lane work. Otherwise (always on the first block) a slow path reduces the
// exact block maximum across the 128 lanes, raises m, and rescales the row
// sums and O^T. Row sums are per-lane partials, reduced once at the end.
//
// Warp roles (640 threads): warp 0 issues the TMA loads of Q and of the K
// blocks (3-stage ring), warp 19 those of the V blocks (2-stage ring), four
// lanes each issuing one 8 KB box; warp 1 owns TMEM and issues the S^T
// products, warp 18 the O^T products; warps 2-17 are four softmax warpgroups
// (16 query columns each) that also run the epilogue. Spreading the columns
// over 16 warps shortens each warp's per-block dependency chain. Every wait
// is bounded (see ptx.cuh).
#include "kernels.cuh"
#include "ptx.cuh"

namespace vsa {
namespace {

constexpr int kSoftmaxWGs = 4;               // softmax warpgroups, each kCols query columns
constexpr int kCols = 64 / kSoftmaxWGs;
constexpr int kThreads = 32 * (4 + 4 * kSoftmaxWGs);  // 20 warps
constexpr int kWarpProducer = 0;             // Q, then the K ring
constexpr int kWarpMmaS = 1;                 // also owns the TMEM allocation
constexpr int kWarpSoftmax0 = 2;             // warps 2 .. 2 + 4*kSoftmaxWGs - 1
constexpr int kWarpMmaPV = kWarpSoftmax0 + 4 * kSoftmaxWGs;
constexpr int kWarpProducerV = kWarpMmaPV + 1;  // the V ring
static_assert(kCols == 16, "the softmax code below is written for 16 columns per warpgroup");
constexpr int kNumK = 3;
constexpr int kNumV = 2;
constexpr uint32_t kQBytes = 64 * kHeadDim * 2;    // 16 KB
constexpr uint32_t kKVBytes = 128 * kHeadDim * 2;  // 32 KB, one 128-key block
constexpr uint32_t kPBytes = 128 * 64 * 2;         // 16 KB
constexpr uint32_t kTmemCols = 256;
constexpr int kNumS = 3;                 // S^T buffers in TMEM
constexpr int kNumP = 3;                 // P^T buffers in shared memory
constexpr uint32_t kColS1 = 64;          // S^T buffer b at column b * kColS1
constexpr uint32_t kColO = kNumS * kColS1;
constexpr float kRescaleThreshold = 8.0f;  // exact mode: rescale when P would exceed 2^8
constexpr float kFastLimitSum = 18446744073709551616.0f;  // 2^64: fast-pass bound on P (and on each row sum)

constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kQBytes;
constexpr uint32_t kOffV = kOffK + kNumK * kKVBytes;
constexpr uint32_t kOffP = kOffV + kNumV * kKVBytes;
constexpr uint32_t kOffBar = kOffP + kNumP * kPBytes;
constexpr uint32_t kOffRed = kOffBar + 256;
constexpr uint32_t kOffSlot = kOffRed + 64 * 4 * 4;  // [64 query columns][4 lane quarters] fp32
constexpr uint32_t kSmemBytes = kOffSlot + 16 + 1024;  // + 1024-byte alignment slack

// barrier indices
constexpr int kBarQ = 0;
constexpr int kBarKFull = 1;
constexpr int kBarKEmpty = kBarKFull + kNumK;
constexpr int kBarVFull = kBarKEmpty + kNumK;
constexpr int kBarVEmpty = kBarVFull + kNumV;
constexpr int kBarSFull = kBarVEmpty + kNumV;
constexpr int kBarSEmpty = kBarSFull + kNumS;
constexpr int kBarPFull = kBarSEmpty + kNumS;
constexpr int kBarPEmpty = kBarPFull + kNumP;
constexpr int kNumBars = kBarPEmpty + kNumP;
static_assert(kNumBars * 8 <= 256, "barrier area");
static_assert(kColO + 64 <= kTmemCols, "TMEM columns");
static_assert(kNumS == kNumP, "the softmax loop walks the S^T and P^T rings with one slot counter");

struct FineParams {
  int B, H, P, Lv, N, T, TP, k;
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

// Items are ordered head by head: for each (batch, head), its TP prefix query
// tiles (the long, dense items) and then its T video query tiles. The CTAs in
// flight at any time then read the K/V of one or two heads, which stay resident
// in L2; taking all prefix items first would stream every head's K/V at once.
__device__ __forceinline__ Item decode_item(const FineParams& p, int item) {
  Item it;
  const int per_head = p.TP + p.T;
  const int bh = item / per_head;
  const int local = item - bh * per_head;
  it.b = bh / p.H;
  it.h = bh - it.b * p.H;
  if (local < p.TP) {
    it.video = false;
    it.t = local;
    it.q_row0 = it.t * kTile;
    it.q_valid = min(kTile, p.P - it.q_row0);
    it.n_kv = p.TP + p.T;
    it.list = nullptr;
  } else {
    it.video = true;
    it.t = local - p.TP;
    it.q_row0 = p.P + it.t * kTile;
    it.q_valid = min(kTile, p.Lv - it.t * kTile);
    it.n_kv = p.TP + p.k;
    it.list = p.tile_index + ((static_cast<size_t>(it.b) * p.H + it.h) * p.T + it.t) * p.k;
  }
  return it;
}

// One halving step of the warp reduce-scatter: lanes with bit O set keep the
// upper half of the live columns, the others the lower half, combined with the
// half their partner (lane ^ O) gave away.
template <bool kMax, int O, int N>
__device__ __forceinline__ void reduce_scatter_step(float (&v)[N], int lane) {
  const bool upper = (lane & O) != 0;
#pragma unroll
  for (int i = 0; i < O; ++i) {
    const float send = upper ? v[i] : v[i + O];
    const float keep = upper ? v[i + O] : v[i];
    const float recv = __shfl_xor_sync(0xffffffffu, send, O);
    v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
  }
}

// Reduce 16 per-lane column values across the warp; afterwards lanes c and
// c + 16 hold the reduction of column c. The input array is consumed.
template <bool kMax>
__device__ __forceinline__ float reduce_scatter16(float (&v)[16], int lane) {
  reduce_scatter_step<kMax, 8>(v, lane);
  reduce_scatter_step<kMax, 4>(v, lane);
  reduce_scatter_step<kMax, 2>(v, lane);
  reduce_scatter_step<kMax, 1>(v, lane);
  const float other = __shfl_xor_sync(0xffffffffu, v[0], 16);
  return kMax ? fmaxf(v[0], other) : v[0] + other;
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

  volatile uint32_t* redo_flag = tslot + 1;  // set when the fast pass must be redone exactly
  if (warp == kWarpMmaS) tmem_alloc(smem_u32(tslot), kTmemCols);

  for (int pass = 0; pass < 2; ++pass) {
  // Pass 0 is the fast mode: after the first block, the per-column softmax
  // reference stays fixed and blocks need no warpgroup vote. It is valid while
  // every P = 2^(score - reference) stays below kFastLimitSum (P, the row sums
  // and O then stay finite, and exact in relative terms). A thread whose row
  // sums end at or above that bound flags the item, and the CTA reruns it in
  // pass 1 with the exact per-block rescaling.
  const bool exact = pass > 0;
  if (tid == 0) {
    if (pass > 0) {
      for (int i = 0; i < kNumBars; ++i) mbar_inval(bar(i));
    } else {
      *redo_flag = 0u;
    }
    mbar_init(bar(kBarQ), 1);
    for (int s = 0; s < kNumK; ++s) { mbar_init(bar(kBarKFull + s), 1); mbar_init(bar(kBarKEmpty + s), 1); }
    for (int s = 0; s < kNumV; ++s) { mbar_init(bar(kBarVFull + s), 1); mbar_init(bar(kBarVEmpty + s), 1); }
    for (int s = 0; s < kNumS; ++s) {
      mbar_init(bar(kBarSFull + s), 1);
      mbar_init(bar(kBarSEmpty + s), 4 * kSoftmaxWGs);
    }
    for (int s = 0; s < kNumP; ++s) {
      mbar_init(bar(kBarPFull + s), 4 * kSoftmaxWGs);
      mbar_init(bar(kBarPEmpty + s), 1);
    }
    fence_barrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  if (warp == kWarpProducer || warp == kWarpProducerV) {
    // ------------------------------------------------------------ TMA producers
    // Lanes 0-3 of each producer warp issue the four 8 KB boxes of a block (tile
    // a/b x channel half): several issuing threads keep far more bytes in flight
    // than one thread can.
    bool failed = abort_raised(err);
    if (warp == kWarpProducer && lane == 0 && !failed) {
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
    // K and V come from separate warps so that a full V ring never delays K.
    const bool v_warp = warp == kWarpProducerV;
    const CUtensorMap* map = v_warp ? &map_v : &map_k;
    const uint32_t ring = v_warp ? sV : sK;
    const int nstage = v_warp ? kNumV : kNumK;
    const int bar_full = v_warp ? kBarVFull : kBarKFull;
    const int bar_empty = v_warp ? kBarVEmpty : kBarKEmpty;
    const int box_tile = (lane >> 1) & 1, box_half = lane & 1;  // this lane's box within a block
    const uint32_t box_off = box_half * 16384 + box_tile * 8192;
    for (int blk = 0; blk < nblk && !failed; ++blk) {
      const int ra = tile_row(2 * blk);
      const int rb = tile_row(2 * blk + 1);
      const int s = blk % nstage;
      bool ok = true;
      if (lane == 0) {
        ok = mbar_wait(bar(bar_empty + s), ((blk / nstage) & 1) ^ 1, err, v_warp ? 0x200u : 0x100u, 128);
        if (ok) mbar_arrive_expect_tx(bar(bar_full + s), kKVBytes);
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) { failed = true; break; }
      if (lane < 4)
        tma_load_4d(ring + s * kKVBytes + box_off, map, 64 * box_half, it.h, box_tile ? rb : ra, it.b,
                    bar(bar_full + s));
    }
  } else if (warp == kWarpMmaS) {
    // ------------------------------------------------------------ S^T = K Q^T issuer
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16_f32(128, 64, 0, 0);
      const uint64_t dk0 = smem_desc_sw128(sK, 16, 1024);
      const uint64_t dq0 = smem_desc_sw128(sQ, 16, 1024);
      bool ok = mbar_wait(bar(kBarQ), 0, err, 0x500u, 64);
      for (int i = 0; i < nblk && ok; ++i) {
        const int ks = i % kNumK, sb = i % kNumS;
        ok = mbar_wait(bar(kBarKFull + ks), (i / kNumK) & 1, err, 0x600u, 64) &&
             mbar_wait(bar(kBarSEmpty + sb), ((i / kNumS) & 1) ^ 1, err, 0x700u, 64);
        if (!ok) break;
        tc_fence_after();
        const uint64_t dk = dk0 + ((ks * kKVBytes) >> 4);
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const uint32_t koff = ((s >> 2) * 16384 + (s & 3) * 32) >> 4;
          const uint32_t qoff = ((s >> 2) * 8192 + (s & 3) * 32) >> 4;
          umma_bf16(tbase + sb * kColS1, dk + koff, dq0 + qoff, id_s, s > 0 ? 1u : 0u);
        }
        umma_commit(bar(kBarKEmpty + ks));
        umma_commit(bar(kBarSFull + sb));
      }
    }
    __syncwarp();
  } else if (warp == kWarpMmaPV) {
    // ------------------------------------------------------------ O^T += V^T P^T issuer
    if (lane == 0) {
      const uint32_t id_o = idesc_bf16_f32(128, 64, 1, 1);
      const uint64_t dv0 = smem_desc_sw128(sV, 16384, 1024);
      const uint64_t dp0 = smem_desc_sw128(sP, 8192, 1024);
      for (int j = 0; j < nblk; ++j) {
        const int vs = j % kNumV, pb = j % kNumP;
        if (!mbar_wait(bar(kBarVFull + vs), (j / kNumV) & 1, err, 0x300u, 32)) break;
        if (!mbar_wait(bar(kBarPFull + pb), (j / kNumP) & 1, err, 0x400u, 32)) break;
        tc_fence_after();
        const uint64_t dv = dv0 + ((vs * kKVBytes) >> 4);
        const uint64_t dp = dp0 + ((pb * kPBytes) >> 4);
#pragma unroll
        for (int s = 0; s < 8; ++s)
          umma_bf16(tbase + kColO, dv + ((s * 2048) >> 4), dp + ((s * 2048) >> 4), id_o,
                    (j > 0 || s > 0) ? 1u : 0u);
        umma_commit(bar(kBarVEmpty + vs));
        umma_commit(bar(kBarPEmpty + pb));
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int wg = (warp - kWarpSoftmax0) / 4;  // query columns kCols*wg .. kCols*wg + kCols-1
    const int q4 = warp % 4;                     // TMEM lane quarter this warp may access
    const int r = 32 * q4 + lane;                // key lane (softmax), head dim (epilogue)
    const int col0 = kCols * wg;
    const int key_row = r & 63, key_slot = r >> 6;
    const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
    const uint32_t bar_id = 1 + wg;
    const float sl2 = p.scale_log2;
    // Only two key tiles can be ragged: the last prefix tile, and video tile T-1,
    // which (selections being ascending) can only be the item's last key tile.
    const int prefix_tail = p.TP > 0 ? p.P - (p.TP - 1) * kTile : kTile;
    const int video_tail = p.Lv - (p.T - 1) * kTile;
    const bool last_is_ragged =
        video_tail < kTile && (it.list == nullptr || __ldg(it.list + p.k - 1) == p.T - 1);
    // Per column pair: -reference (log2 units) and this lane's partial row sums.
    float2 nm2[kCols / 2], l2[kCols / 2];
#pragma unroll
    for (int j = 0; j < kCols / 2; ++j) {
      nm2[j] = make_float2(INFINITY, INFINITY);
      l2[j] = make_float2(0.f, 0.f);
    }
    const float2 sl2v = make_float2(sl2, sl2);
    // Blocks that may hold masked key lanes: the one with the ragged last prefix
    // tile, and the last block (an absent second tile, or ragged video tile T-1).
    const int ragged_prefix_blk = (p.TP > 0 && prefix_tail < kTile) ? (p.TP - 1) / 2 : -1;
    bool failed = false;
    // ---- general block: masking, and (exact pass or first block) the exact
    // per-column block maximum with rescaling. st / ph: S^T and P^T ring slot
    // of block i and its phase parity (the two rings have equal depth).
    auto general_block = [&](const int i, const int st, const uint32_t ph) {
      const int ti = 2 * i + key_slot;
      bool valid = ti < it.n_kv;
      if (ti == p.TP - 1) valid = key_row < prefix_tail;
      if (ti == it.n_kv - 1 && last_is_ragged) valid = valid && key_row < video_tail;

      failed = warp_any(failed || !mbar_wait(bar(kBarSFull + st), ph, err, 0x800u));
      float s[kCols];
      if (!failed) {
        tc_fence_after();
        uint32_t raw[kCols];
        tmem_ld16(tbase + lane_off + st * kColS1 + col0, raw);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < kCols; ++c) s[c] = __uint_as_float(raw[c]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarSEmpty + st));
      } else {
#pragma unroll
        for (int c = 0; c < kCols; ++c) s[c] = 0.f;
      }
      if (!valid) {  // masked key lane (ragged or absent tile): contributes nothing
#pragma unroll
        for (int c = 0; c < kCols; ++c) s[c] = -INFINITY;
      }
      // t = s * log2(e)/sqrt(128) - reference
      float t[kCols];
#pragma unroll
      for (int j = 0; j < kCols / 2; ++j) {
        const float2 tt = __ffma2_rn(make_float2(s[2 * j], s[2 * j + 1]), sl2v, nm2[j]);
        t[2 * j] = tt.x;
        t[2 * j + 1] = tt.y;
      }
      bool slow = false;
      if (exact || i == 0) {
        const float mxall = fmax3(fmax3(fmax3(t[0], t[1], t[2]), fmax3(t[3], t[4], t[5]), fmax3(t[6], t[7], t[8])),
                                  fmax3(t[9], t[10], t[11]), fmax3(fmax3(t[12], t[13], t[14]), t[15], -INFINITY));
        slow = named_bar_or(bar_id, 128, failed || mxall > kRescaleThreshold);
      }
      if (slow) {
        if (named_bar_or(bar_id, 128, failed)) { failed = true; return; }
        // slow path: exact block maximum per query column across the 128 key lanes
        float u[kCols];
#pragma unroll
        for (int c = 0; c < kCols; ++c) u[c] = s[c] * sl2;
        const float wmax = reduce_scatter16<true>(u, lane);
        if (lane < kCols) red[(wg * kCols + lane) * 4 + q4] = wmax;
        named_bar_sync(bar_id, 128);
        float alpha[kCols];
#pragma unroll
        for (int j = 0; j < kCols / 2; ++j) {
          const float4 x0 = reinterpret_cast<const float4*>(red)[wg * kCols + 2 * j];
          const float4 x1 = reinterpret_cast<const float4*>(red)[wg * kCols + 2 * j + 1];
          const float bm0 = fmaxf(fmaxf(x0.x, x0.y), fmaxf(x0.z, x0.w));
          const float bm1 = fmaxf(fmaxf(x1.x, x1.y), fmaxf(x1.z, x1.w));
          const float n0 = fminf(nm2[j].x, -bm0), n1 = fminf(nm2[j].y, -bm1);
          alpha[2 * j] = ex2_approx(n0 - nm2[j].x);
          alpha[2 * j + 1] = ex2_approx(n1 - nm2[j].y);
          l2[j] = make_float2(l2[j].x * alpha[2 * j], l2[j].y * alpha[2 * j + 1]);
          nm2[j] = make_float2(n0, n1);
        }
        if (i > 0) {
          // O^T must hold every PV product issued so far: wait for PV of block
          // i-1 on its P-buffer barrier (PV of block i-1-kNumP is already known
          // to be complete, so this parity wait cannot alias an older phase;
          // tcgen05 MMAs complete in issue order).
          const int pst = st == 0 ? kNumP - 1 : st - 1;
          const uint32_t pph = st == 0 ? ph ^ 1u : ph;
          failed = warp_any(!mbar_wait(bar(kBarPEmpty + pst), pph, err, 0x900u));
          if (!failed) {
            tc_fence_after();
            uint32_t o[kCols];
            tmem_ld16(tbase + lane_off + kColO + col0, o);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < kCols; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha[c]);
            tmem_st16(tbase + lane_off + kColO + col0, o);
            tmem_wait_st();
            tc_fence_before();
          }
        }
#pragma unroll
        for (int j = 0; j < kCols / 2; ++j) {
          const float2 tt = __ffma2_rn(make_float2(s[2 * j], s[2 * j + 1]), sl2v, nm2[j]);
          t[2 * j] = tt.x;
          t[2 * j + 1] = tt.y;
        }
      }
      uint32_t pk[kCols / 2];
#pragma unroll
      for (int j = 0; j < kCols / 2; ++j) {
        const float p0 = ex2_approx(t[2 * j]), p1 = ex2_approx(t[2 * j + 1]);
        l2[j] = __fadd2_rn(l2[j], make_float2(p0, p1));
        pk[j] = pack_bf16x2(p0, p1);
      }
      failed = warp_any(failed || !mbar_wait(bar(kBarPEmpty + st), ph ^ 1u, err, 0xA00u));
      if (!failed) {
        const uint32_t prow = sP + st * kPBytes + r * 128;
#pragma unroll
        for (int cc = 0; cc < kCols / 8; ++cc) {
          const uint32_t chunk = static_cast<uint32_t>((col0 / 8 + cc) ^ (r & 7));
          st_shared_v4(prow + chunk * 16, pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarPFull + st));
      }
    };
    // ---- fast-pass block: no masked lanes, fixed reference, no cross-lane work.
    // Returns false once a wait has failed.
    auto fast_block = [&](const int st, const uint32_t ph) -> bool {
      if (warp_any(!mbar_wait(bar(kBarSFull + st), ph, err, 0x800u))) return false;
      tc_fence_after();
      uint32_t raw[kCols];
      tmem_ld16(tbase + lane_off + st * kColS1 + col0, raw);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarSEmpty + st));
      uint32_t pk[kCols / 2];
#pragma unroll
      for (int j = 0; j < kCols / 2; ++j) {
        const float2 t = __ffma2_rn(make_float2(__uint_as_float(raw[2 * j]), __uint_as_float(raw[2 * j + 1])),
                                    sl2v, nm2[j]);
        const float p0 = ex2_approx(t.x), p1 = ex2_approx(t.y);
        l2[j] = __fadd2_rn(l2[j], make_float2(p0, p1));
        pk[j] = pack_bf16x2(p0, p1);
      }
      if (warp_any(!mbar_wait(bar(kBarPEmpty + st), ph ^ 1u, err, 0xA00u))) return false;
      const uint32_t prow = sP + st * kPBytes + r * 128;
#pragma unroll
      for (int cc = 0; cc < kCols / 8; ++cc) {
        const uint32_t chunk = static_cast<uint32_t>((col0 / 8 + cc) ^ (r & 7));
        st_shared_v4(prow + chunk * 16, pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarPFull + st));
      return true;
    };
    // The epilogue's gate and coarse inputs come from HBM: all of them are
    // requested together, right after the last block, so that their latency
    // overlaps the drain of the last O^T product (loading them inside the store
    // loop serialised one HBM round trip per column).
    const size_t row_stride = static_cast<size_t>(p.H) * kHeadDim;
    const size_t out_base = (static_cast<size_t>(it.b) * p.N + it.q_row0) * row_stride +
                            static_cast<size_t>(it.h) * kHeadDim + r;
    float gv[kCols];
    float cz = 0.f;
    auto prefetch_gate = [&]() {
#pragma unroll
      for (int c = 0; c < kCols; ++c) gv[c] = 0.f;
      if (it.video) {
        cz = __ldg(p.coarse + ((static_cast<size_t>(it.b) * p.H + it.h) * p.T + it.t) * kHeadDim + r);
#pragma unroll
        for (int c = 0; c < kCols; ++c)
          if (col0 + c < it.q_valid)
            gv[c] = __bfloat162float(__ldg(p.gate + out_base + static_cast<size_t>(col0 + c) * row_stride));
      }
    };
    if (exact) {
      for (int i = 0; i < nblk && !failed; ++i) general_block(i, i % kNumS, (i / kNumS) & 1);
      prefetch_gate();
    } else {
      general_block(0, 0, 0u);
      // fast blocks 1 .. nblk-2, the ragged-prefix block (if any) excepted
      int st = 1 % kNumS;
      uint32_t ph = 0;
      for (int i = 1; i < nblk - 1 && !failed; ++i) {
        if (i == ragged_prefix_blk) {
          general_block(i, st, ph);
        } else if (!fast_block(st, ph)) {
          failed = true;
        }
        if (++st == kNumS) { st = 0; ph ^= 1u; }
      }
      if (nblk > 1 && !failed) general_block(nblk - 1, (nblk - 1) % kNumS, ((nblk - 1) / kNumS) & 1);
      prefetch_gate();
    }
    // The fast pass is valid while every P stayed below 2^kFastLimit: P >= 0, so
    // one larger P (or an overflow to inf) leaves a partial row sum at or above
    // that bound (a NaN fails the comparison too).
    bool overflow = false;
    if (!exact) {
#pragma unroll
      for (int j = 0; j < kCols / 2; ++j)
        overflow = overflow || !(l2[j].x < kFastLimitSum) || !(l2[j].y < kFastLimitSum);
    }
    float l[kCols];
#pragma unroll
    for (int j = 0; j < kCols / 2; ++j) {
      l[2 * j] = l2[j].x;
      l[2 * j + 1] = l2[j].y;
    }
    // ---- epilogue: out = O / l (+ sigmoid(gate) * coarse on video rows)
    if (named_bar_or(bar_id, 128, overflow && !failed)) *redo_flag = 1u;  // rerun in exact mode
    if (!named_bar_or(bar_id, 128, failed)) {
      const float lw = reduce_scatter16<false>(l, lane);
      if (lane < kCols) red[(wg * kCols + lane) * 4 + q4] = lw;
      named_bar_sync(bar_id, 128);
      const int pj = nblk - 1;  // the last PV product (see the rescale above)
      failed = warp_any(!mbar_wait(bar(kBarPEmpty + pj % kNumP), (pj / kNumP) & 1, err, 0xB00u));
      if (!failed) {
        tc_fence_after();
        uint32_t o[kCols];
        tmem_ld16(tbase + lane_off + kColO + col0, o);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < kCols; ++c) {
          const int qc = col0 + c;
          if (qc < it.q_valid) {
            const float4 x = reinterpret_cast<const float4*>(red)[wg * kCols + c];
            const float lsum = (x.x + x.y) + (x.z + x.w);
            float val = __fdividef(__uint_as_float(o[c]), lsum);
            if (it.video) val += __fdividef(cz, 1.0f + __expf(-gv[c]));
            p.out[out_base + static_cast<size_t>(qc) * row_stride] = __float2bfloat16_rn(val);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*redo_flag == 0u) break;  // uniform: read after the barrier by every thread
  }  // pass

  if (warp == kWarpMmaS) tmem_dealloc(*tslot, kTmemCols);
}

}  // namespace

size_t fine_smem_bytes() { return kSmemBytes; }

cudaError_t launch_fine(const Geometry& g, const CUtensorMap& map_q, const CUtensorMap& map_k,
                        const CUtensorMap& map_v, const FineArgs& a, cudaStream_t stream) {
  FineParams p;
  p.B = g.B; p.H = g.H; p.P = g.P; p.Lv = g.Lv; p.N = g.N; p.T = g.T; p.TP = g.TP; p.k = g.k;
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
