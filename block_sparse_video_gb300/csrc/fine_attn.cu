// Fine attention of the VSA forward, with the gated coarse add fused into the
// epilogue ("UniServe: serving FastH3 at its fastest", sections "The FastH3
// workload" and "Fused output combination").
//
// Work items are 64-token query tiles:
//   * a prefix (text/audio) query tile attends to every key tile: the TP
//     prefix tiles, then the T video tiles; its output is the attention alone;
//   * a video query tile t attends to the TP prefix tiles and to its k selected
//     video tiles; its output adds sigmoid(gate) * coarse[t] per channel. With
//     no coarse input (the SubBlock router's selection, section "How SubBlock
//     Sparse Attention Works") the output is the attention alone.
// Key tiles are processed two at a time (a 128-key block).
//
// Persistent kernel: one CTA per SM takes items from a global counter until
// they run out. Every ring (Q, K, V, S^T, P^T, O^T) keeps its slot counters
// across items, so the loads of the next item start while the current one
// finishes and no CTA start-up or drain sits between items.
//
// Formulation: transposed, so that both tensor-core products have M = 128
// with a 64-row query tile:
//   S^T[128 keys x 64 queries] = K_blk[128 x 128] . Q^T           (A, B K-major)
//   O^T[128 dims x 64 queries] += V_blk^T[128 x 128 keys] . P^T   (A, B MN-major)
// S^T and O^T live in tensor memory (TMEM lane = key, resp. head dim; column =
// query). Each softmax thread owns one key lane for 16 query columns, so
// masking a ragged or absent key tile is a per-thread select.
//
// Online softmax. The fast kernel fixes the reference m (log2 units) to 0, so
// P = 2^score, and never rescales. Softmax does not depend on m. P (bf16) and
// the row sums and O^T (fp32) keep their relative precision at any scale
// between the limits, so the fast result is valid while every P stays below
// kFastLimitSum (2^64) and every row sum stays at or above kFastMinSum (2^-60;
// below it, P values that still matter could be subnormal). Both are checked
// on each lane's partial row sums: P >= 0, so one P at or above 2^64 leaves
// its lane's partial above the bound, and partials at or above 2^-60 make the
// row sum so too (a lane whose own keys all score far below the rest of the
// row fails the floor alone and only costs a redo). An item that fails is
// appended to a redo list. The exact kernel (the same code, exact mode) then
// recomputes the redo list with per-block rescaling. Its reference starts at
// the first block's exact maximum. A later block whose scores all stay below
// m + 8 (P <= 256) needs no cross-lane work; otherwise the exact block maximum
// is reduced across the 128 lanes, m is raised, and the row sums and O^T are
// rescaled. Row sums are per-lane partials, reduced once per item.
//
// Warp roles (640 threads): warp 0 fetches the items, loads each item's Q tile
// as soon as it has fetched it (two buffers, alternating by item) and issues
// the TMA loads of the K blocks (3-stage ring), warp 19 those of the V blocks
// (2-stage ring), four lanes each issuing one 8 KB box; warp 1 owns TMEM and
// issues the S^T products, warp 18 the O^T products (two TMEM accumulators,
// alternating by item; P^T in a 2-stage ring), each MMA warp converged with
// one elected lane issuing; warps 2-17
// are four softmax warpgroups (16 query columns each) that also run the
// epilogue. Every wait is bounded (see ptx.cuh); a named barrier
// is always reached by all of its threads.
#include "kernels.cuh"
#include "ptx.cuh"

namespace vsa {
namespace {

constexpr int kSoftmaxWGs = 4;               // softmax warpgroups, each kCols query columns
constexpr int kCols = 64 / kSoftmaxWGs;
constexpr int kThreads = 32 * (4 + 4 * kSoftmaxWGs);  // 20 warps
constexpr int kWarpProducer = 0;             // item fetch, then the K ring
constexpr int kWarpMmaS = 1;                 // also owns the TMEM allocation and loads Q
constexpr int kWarpSoftmax0 = 2;             // warps 2 .. 2 + 4*kSoftmaxWGs - 1
constexpr int kWarpMmaPV = kWarpSoftmax0 + 4 * kSoftmaxWGs;
constexpr int kWarpProducerV = kWarpMmaPV + 1;  // the V ring
constexpr int kSoftmaxWarps = 4 * kSoftmaxWGs;
static_assert(kCols == 16, "the softmax code below is written for 16 columns per warpgroup");
constexpr int kNumK = 3;
constexpr int kNumV = 2;
constexpr int kNumQ = 2;                           // Q buffers, alternating by item
constexpr uint32_t kQBytes = 64 * kHeadDim * 2;    // 16 KB
constexpr uint32_t kKVBytes = 128 * kHeadDim * 2;  // 32 KB, one 128-key block
constexpr uint32_t kPBytes = 128 * 64 * 2;         // 16 KB
constexpr uint32_t kTmemCols = 512;
constexpr int kNumS = 3;                 // S^T buffers in TMEM
constexpr int kNumP = 2;                 // P^T buffers in shared memory
constexpr int kNumO = 2;                 // O^T accumulators in TMEM, alternating by item
constexpr uint32_t kColS1 = 64;          // S^T buffer b at column b * kColS1
constexpr uint32_t kColO = kNumS * kColS1;  // O^T accumulator a at column kColO + 64 a
constexpr int kItemSlots = 8;            // item ring between the fetching warp and the others
constexpr int kItemReaders = 3 + kSoftmaxWarps;  // V loader, both MMA issuers, softmax warps
constexpr float kRescaleThreshold = 8.0f;  // exact mode: rescale when P would exceed 2^8
constexpr float kFastLimitSum = 18446744073709551616.0f;  // 2^64: fast-mode bound on P (and on each row sum)
constexpr float kFastMinSum = 8.673617379884035e-19f;       // 2^-60: fast-mode floor on each row sum
constexpr uint32_t kBarSoftmaxAll = 1 + kSoftmaxWGs;  // named barrier over all softmax warps

constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kNumQ * kQBytes;
constexpr uint32_t kOffV = kOffK + kNumK * kKVBytes;
constexpr uint32_t kOffP = kOffV + kNumV * kKVBytes;
constexpr uint32_t kOffBar = kOffP + kNumP * kPBytes;
constexpr uint32_t kOffRed = kOffBar + 512;
constexpr uint32_t kOffItems = kOffRed + 64 * 4 * 4;  // red: [64 query columns][4 lane quarters] fp32
constexpr uint32_t kOffSlot = kOffItems + kItemSlots * 4;
constexpr uint32_t kOffGeo = kOffSlot + 16;            // this forward's geometry (FineGeo)
constexpr uint32_t kSmemBytes = kOffGeo + 32 + 1024;   // + 1024-byte alignment slack

// barrier indices
constexpr int kBarQFull = 0;              // + item % kNumQ
constexpr int kBarQEmpty = kBarQFull + kNumQ;
// A K slot is released by the S-full barrier of the block that read it (the
// same commit, so no separate barrier), a V slot by the P-empty barrier of its
// block: one commit per MMA group. Each loader waits on those barriers in
// block order, so none of its parity waits can fall two phases behind.
constexpr int kBarKFull = kBarQEmpty + kNumQ;
constexpr int kBarVFull = kBarKFull + kNumK;
constexpr int kBarSFull = kBarVFull + kNumV;
constexpr int kBarSEmpty = kBarSFull + kNumS;
constexpr int kBarPFull = kBarSEmpty + kNumS;
constexpr int kBarPEmpty = kBarPFull + kNumP;
constexpr int kBarOEmpty = kBarPEmpty + kNumP;
constexpr int kBarItemFull = kBarOEmpty + kNumO;
constexpr int kBarItemEmpty = kBarItemFull + kItemSlots;
// Device lengths: a V box that reaches rows past the request's tokens lands
// here first; the V loader clears those rows, then completes the slot's full
// barrier itself.
constexpr int kBarVClear = kBarItemEmpty + kItemSlots;
constexpr int kNumBars = kBarVClear + 1;
static_assert(kNumBars * 8 <= 512, "barrier area");
static_assert(kColO + kNumO * 64 <= kTmemCols, "TMEM columns");
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

// Geometry of the plan: the capacity when lengths come from the device. N is
// the buffer rows per batch, T and k the layout strides of the coarse rows and
// tile selections; P, Lv, TP, T, k and n_items are this forward's own unless
// dl.len is set (then FineGeo holds the actual ones).
struct FineParams {
  int B, H, P, Lv, N, T, TP, k;
  int n_items;          // B * H * (TP + T)
  DeviceLengths dl;
  float scale_log2;
  const __nv_bfloat16* gate;
  __nv_bfloat16* out;
  const float* coarse;  // null: no gated coarse term on video rows (SubBlock routing)
  const int32_t* out_row_map;  // null: token n of batch b -> out row b * N + n; else row b * out_rows + map[b * N + n]
  long long out_rows;          // output rows per batch
  long long out_row_stride;    // elements between output rows
  long long in_row_stride;     // elements between token rows of the gate (and of q, k, v via the tensor maps)
  const int32_t* tile_index;
  unsigned int* err;
  int* work_counter;    // next work index to hand out (zeroed before the launch)
  int* redo_count;      // fast mode: items appended; exact mode: items to process
  int* redo_list;
};

// This forward's geometry, computed once per CTA into shared memory.
struct FineGeo {
  int P, Lv, T, TP, k, n_items;
};

__device__ __forceinline__ FineGeo fine_geo(const FineParams& p) {
  Geometry cap;
  cap.B = p.B; cap.H = p.H; cap.P = p.P; cap.Lv = p.Lv; cap.N = p.N; cap.T = p.T; cap.TP = p.TP; cap.k = p.k;
  const DynGeom d = dyn_geom(cap, p.dl);
  return FineGeo{d.P, d.Lv, d.T, d.TP, d.k, d.valid ? p.B * p.H * (d.TP + d.T) : 0};
}

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
__device__ __forceinline__ Item decode_item(const FineParams& p, const FineGeo& G, int item) {
  Item it;
  const int per_head = G.TP + G.T;
  const int bh = item / per_head;
  const int local = item - bh * per_head;
  it.b = bh / p.H;
  it.h = bh - it.b * p.H;
  if (local < G.TP) {
    it.video = false;
    it.t = local;
    it.q_row0 = it.t * kTile;
    it.q_valid = min(kTile, G.P - it.q_row0);
    it.n_kv = G.TP + G.T;
    it.list = nullptr;
  } else {
    it.video = true;
    it.t = local - G.TP;
    it.q_row0 = G.P + it.t * kTile;
    it.q_valid = min(kTile, G.Lv - it.t * kTile);
    it.n_kv = G.TP + G.k;
    // selections are stored at the plan's strides (T and k of the capacity)
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

// kExact = false: the fast kernel over all items; kExact = true: the exact
// kernel over the redo list the fast kernel wrote.
template <bool kExact>
__global__ void __launch_bounds__(kThreads, 1)
fine_attn_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                 const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_g,
                 const FineParams p) {
  const FineGeo geo = fine_geo(p);
  const int n_work = kExact ? *reinterpret_cast<const volatile int*>(p.redo_count) : geo.n_items;
  if (n_work <= 0) return;  // uniform: nothing to do (the exact kernel's usual case)

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
  volatile int* items = reinterpret_cast<volatile int*>(smem + kOffItems);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + kOffSlot);
  FineGeo* s_geo = reinterpret_cast<FineGeo*>(smem + kOffGeo);

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  unsigned int* err = p.err;

  if (tid == 0) {
    *s_geo = geo;
    for (int s = 0; s < kNumQ; ++s) {
      mbar_init(bar(kBarQFull + s), 1);
      mbar_init(bar(kBarQEmpty + s), 1);
    }
    for (int s = 0; s < kNumK; ++s) mbar_init(bar(kBarKFull + s), 1);
    for (int s = 0; s < kNumV; ++s) mbar_init(bar(kBarVFull + s), 1);
    for (int s = 0; s < kNumS; ++s) {
      mbar_init(bar(kBarSFull + s), 1);
      mbar_init(bar(kBarSEmpty + s), kSoftmaxWarps);
    }
    for (int s = 0; s < kNumP; ++s) {
      mbar_init(bar(kBarPFull + s), kSoftmaxWarps);
      mbar_init(bar(kBarPEmpty + s), 1);
    }
    for (int s = 0; s < kNumO; ++s) mbar_init(bar(kBarOEmpty + s), kSoftmaxWarps);
    for (int s = 0; s < kItemSlots; ++s) {
      mbar_init(bar(kBarItemFull + s), 1);
      mbar_init(bar(kBarItemEmpty + s), kItemReaders);
    }
    mbar_init(bar(kBarVClear), 1);
    fence_barrier_init();
  }
  if (warp == kWarpMmaS) tmem_alloc(smem_u32(tslot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const FineGeo& G = *s_geo;

  // Item n of this CTA (n = 0, 1, ...) sits in ring slot n % kItemSlots; -1
  // ends the sequence. Read by lane 0 of each reading warp, then broadcast.
  auto read_item = [&](int n, bool& ok) -> int {
    int item = -1;
    if (lane == 0) {
      const int s = n % kItemSlots;
      ok = ok && mbar_wait(bar(kBarItemFull + s), (n / kItemSlots) & 1, err, 0xC00u, 64);
      if (ok) {
        item = items[s];
        mbar_arrive(bar(kBarItemEmpty + s));
      }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    return __shfl_sync(0xffffffffu, item, 0);
  };

  if (warp == kWarpProducer || warp == kWarpProducerV) {
    // ------------------------------------------------------------ TMA producers
    // Lanes 0-3 of each producer warp issue the four 8 KB boxes of a block (tile
    // a/b x channel half): several issuing threads keep far more bytes in flight
    // than one thread can. K and V come from separate warps so that a full V
    // ring never delays K.
    const bool v_warp = warp == kWarpProducerV;
    bool ok = !abort_raised(err);
    if (!v_warp && lane == 0 && ok) {
      prefetch_tensor_map(&map_q);
      prefetch_tensor_map(&map_k);
      prefetch_tensor_map(&map_v);
    }
    const CUtensorMap* map = v_warp ? &map_v : &map_k;
    const uint32_t ring = v_warp ? sV : sK;
    const int nstage = v_warp ? kNumV : kNumK;
    const int bar_full = v_warp ? kBarVFull : kBarKFull;
    const int box_tile = (lane >> 1) & 1, box_half = lane & 1;  // this lane's box within a block
    const uint32_t box_off = box_half * 16384 + box_tile * 8192;
    int slot = 0;        // ring slot of the next block (counting over all items)
    uint32_t g = 0;      // blocks loaded so far, over all items
    uint32_t n_clear = 0;  // V blocks that went through the clearing barrier
    // With device lengths, rows past the request's N (up to the buffer's rows)
    // are capacity padding with arbitrary contents. Their key lanes are masked
    // (P = 0), but 0 * NaN is NaN in the P.V product, so V rows past N are
    // cleared in shared memory before the product reads them. Only the
    // ragged last prefix tile and the ragged last video tile can reach them.
    // (Without device lengths those rows are outside the tensor map and read
    // as zeros.)
    const bool clear_v = v_warp && p.dl.len != nullptr;
    const int n_req = G.P + G.Lv;
    auto kept_rows = [&](int row) { return (!clear_v || row >= p.N) ? kTile : max(0, min(kTile, n_req - row)); };
    for (int n = 0; ok; ++n) {
      int item;
      if (!v_warp) {
        // fetch the next item and publish it to the other warps
        item = -1;
        if (lane == 0) {
          const int s = n % kItemSlots;
          ok = mbar_wait(bar(kBarItemEmpty + s), ((n / kItemSlots) & 1) ^ 1, err, 0xD00u, 64);
          if (ok) {
            const int w = atomicAdd(p.work_counter, 1);
            item = w < n_work ? (kExact ? __ldg(p.redo_list + w) : w) : -1;
            items[s] = item;
            mbar_arrive(bar(kBarItemFull + s));
          }
          // The item's Q tile, into buffer n % kNumQ as soon as the item is
          // known: that buffer was last read by the S^T products of item
          // n - kNumQ, which completed before this warp could load the K
          // blocks of item n - 1 (the S^T products run in item order).
          if (ok && item >= 0) {
            const int qb = n % kNumQ;
            if (n >= kNumQ) ok = mbar_wait(bar(kBarQEmpty + qb), ((n - kNumQ) / kNumQ) & 1, err, 0x510u, 64);
            if (ok) {
              const Item qi = decode_item(p, G, item);
              mbar_arrive_expect_tx(bar(kBarQFull + qb), kQBytes);
              for (int c = 0; c < 2; ++c)
                tma_load_4d(sQ + qb * kQBytes + c * 8192, &map_q, 64 * c, qi.h, qi.q_row0, qi.b, bar(kBarQFull + qb));
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        item = __shfl_sync(0xffffffffu, item, 0);
      } else {
        item = read_item(n, ok);
      }
      if (!ok || item < 0) break;
      const Item it = decode_item(p, G, item);
      const int nblk = (it.n_kv + 1) / 2;
      if (!v_warp && lane == 0) {
        // Into L2 ahead of use: for a video item, its gate tile and coarse
        // row (read by the epilogue, an item's duration later).
        if (it.video && p.coarse) {
          tma_prefetch_l2_4d(&map_g, 0, it.h, it.q_row0, it.b);
          tma_prefetch_l2_4d(&map_g, 64, it.h, it.q_row0, it.b);
          bulk_prefetch_l2(p.coarse + ((static_cast<size_t>(it.b) * p.H + it.h) * p.T + it.t) * kHeadDim,
                           kHeadDim * sizeof(float));
        }
      }
      // Token row of key tile ti of this item (p.N, the buffer rows, for an absent tile: the TMA
      // box is then fully out of bounds and reads as zeros).
      auto tile_row = [&](int ti) -> int {
        if (ti >= it.n_kv) return p.N;
        if (ti < G.TP) return ti * kTile;
        return G.P + (it.list ? __ldg(it.list + (ti - G.TP)) : ti - G.TP) * kTile;
      };
      // Rows are worked out 32 blocks at a time, lane l taking block base + l,
      // so that each block only needs two shuffles here (this warp's loop is on
      // the critical path).
      int row_a = 0, row_b = 0;
      for (int blk = 0; blk < nblk; ++blk) {
        if ((blk & 31) == 0) {
          row_a = tile_row(2 * (blk + lane));
          row_b = tile_row(2 * (blk + lane) + 1);
        }
        const int ra = __shfl_sync(0xffffffffu, row_a, blk & 31);
        const int rb = __shfl_sync(0xffffffffu, row_b, blk & 31);
        // Each issuing lane waits for the slot itself (no broadcast round trip);
        // lane 0 arms the full barrier. A box may land before the arming: the
        // transaction count may run negative until the arrive, and the phase
        // cannot complete before it.
        // The slot's previous block, gp = g - nstage, must have been read: a K
        // slot via S-full of that block, a V slot via its P-empty (the first
        // nstage blocks wait for nothing). The parity wait cannot alias: the
        // next completion of that barrier needs a block this warp has not
        // loaded yet, and the one before it was waited for when block gp was
        // loaded.
        const uint32_t gp = g - static_cast<uint32_t>(nstage);  // wraps for the first nstage blocks
        const int rel_bar = v_warp ? kBarPEmpty + gp % kNumP : kBarSFull + gp % kNumS;
        const uint32_t rel_par = v_warp ? (gp / kNumP) & 1u : (gp / kNumS) & 1u;
        const int keep_a = kept_rows(ra), keep_b = kept_rows(rb);
        const bool clear = keep_a < kTile || keep_b < kTile;  // warp-uniform
        const uint32_t land = clear ? bar(kBarVClear) : bar(bar_full + slot);
        bool lane_ok = true;
        if (lane < 4) {
          if (g >= static_cast<uint32_t>(nstage))
            lane_ok = mbar_wait(bar(rel_bar), rel_par, err, v_warp ? 0x200u : 0x100u);
          if (lane_ok) {
            if (lane == 0) mbar_arrive_expect_tx(land, kKVBytes);
            tma_load_4d(ring + slot * kKVBytes + box_off, map, 64 * box_half, it.h, box_tile ? rb : ra, it.b, land);
          }
        }
        if (!__all_sync(0xffffffffu, lane_ok)) { ok = false; break; }
        if (clear) {
          // every lane observes the boxes landing before it overwrites rows of them
          lane_ok = mbar_wait(bar(kBarVClear), n_clear & 1u, err, 0x210u);
          ++n_clear;
          if (!__all_sync(0xffffffffu, lane_ok)) { ok = false; break; }
          // a row is 128 bytes whatever the swizzle: clear rows keep .. 63 of each
          // affected tile, in both channel halves, 16 bytes per store
          for (int tb = 0; tb < 2; ++tb) {
            const int keep = tb ? keep_b : keep_a;
            const int chunks = (kTile - keep) * 8;  // per channel half
            for (int c = lane; c < 2 * chunks; c += 32) {
              const int half = c >= chunks ? 1 : 0, rem = c - half * chunks;
              st_shared_v4(ring + slot * kKVBytes + half * 16384 + tb * 8192 + (keep + rem / 8) * 128 + (rem % 8) * 16,
                           0u, 0u, 0u, 0u);
            }
          }
          fence_proxy_async_smem();  // the products read shared memory through the async proxy
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(bar_full + slot));  // no bytes pending: completes the phase
        }
        if (++slot == nstage) slot = 0;
        ++g;
      }
    }
  } else if (warp == kWarpMmaS) {
    // ------------------------------------------------------------ S^T = K Q^T issuer
    // The whole warp runs the loop (warp-uniform descriptors); one elected lane
    // issues the products and commits. Item n reads Q buffer n % kNumQ (loaded
    // by the item-fetching warp) and releases it after its last S^T product.
    bool ok = true;
    const uint32_t id_s = idesc_bf16_f32(128, 64, 0, 0);
    const uint64_t dk0 = smem_desc_sw128(sK, 16, 1024);
    uint32_t g = 0;  // blocks issued so far, over all items
    for (int n = 0; ok; ++n) {
      const int item = read_item(n, ok);
      if (!ok || item < 0) break;
      const Item it = decode_item(p, G, item);
      const int nblk = (it.n_kv + 1) / 2;
      const int qb = n % kNumQ;
      const uint64_t dq0 = smem_desc_sw128(sQ + qb * kQBytes, 16, 1024);
      ok = mbar_wait_warp(bar(kBarQFull + qb), (n / kNumQ) & 1, err, 0x500u, 64);
      for (int i = 0; i < nblk && ok; ++i, ++g) {
        const int ks = g % kNumK, sb = g % kNumS;
        ok = mbar_wait_warp(bar(kBarKFull + ks), (g / kNumK) & 1, err, 0x600u, 64) &&
             mbar_wait_warp(bar(kBarSEmpty + sb), ((g / kNumS) & 1) ^ 1, err, 0x700u, 64);
        if (!ok) break;
        tc_fence_after();
        const uint64_t dk = dk0 + ((ks * kKVBytes) >> 4);
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const uint32_t koff = ((s >> 2) * 16384 + (s & 3) * 32) >> 4;
          const uint32_t qoff = ((s >> 2) * 8192 + (s & 3) * 32) >> 4;
          umma_bf16_elect(tbase + sb * kColS1, dk + koff, dq0 + qoff, id_s, s > 0 ? 1u : 0u);
        }
        umma_commit_elect(bar(kBarSFull + sb));  // also releases K slot ks
      }
      if (!ok) break;
      // Q buffer qb stays in use until the item's last S^T product completes
      umma_commit_elect(bar(kBarQEmpty + qb));
    }
  } else if (warp == kWarpMmaPV) {
    // ------------------------------------------------------------ O^T += V^T P^T issuer
    // converged warp, elected lane issues (as for S^T)
    bool ok = true;
    uint32_t g = 0;  // blocks issued so far, over all items
    const uint32_t id_o = idesc_bf16_f32(128, 64, 1, 1);
    const uint64_t dv0 = smem_desc_sw128(sV, 16384, 1024);
    const uint64_t dp0 = smem_desc_sw128(sP, 8192, 1024);
    for (int n = 0; ok; ++n) {
      const int item = read_item(n, ok);
      if (!ok || item < 0) break;
      const Item it = decode_item(p, G, item);
      const int nblk = (it.n_kv + 1) / 2;
      const uint32_t ob = n % kNumO;
      // accumulator ob was last read by the epilogue of item n - kNumO
      if (n >= kNumO) ok = mbar_wait_warp(bar(kBarOEmpty + ob), ((n - kNumO) / kNumO) & 1, err, 0x310u, 32);
      for (int j = 0; j < nblk && ok; ++j, ++g) {
        const int vs = g % kNumV, pb = g % kNumP;
        ok = mbar_wait_warp(bar(kBarVFull + vs), (g / kNumV) & 1, err, 0x300u, 32) &&
             mbar_wait_warp(bar(kBarPFull + pb), (g / kNumP) & 1, err, 0x400u, 32);
        if (!ok) break;
        tc_fence_after();
        const uint64_t dv = dv0 + ((vs * kKVBytes) >> 4);
        const uint64_t dp = dp0 + ((pb * kPBytes) >> 4);
#pragma unroll
        for (int s = 0; s < 8; ++s)
          umma_bf16_elect(tbase + kColO + ob * 64, dv + ((s * 2048) >> 4), dp + ((s * 2048) >> 4), id_o,
                          (j > 0 || s > 0) ? 1u : 0u);
        umma_commit_elect(bar(kBarPEmpty + pb));  // also releases V slot vs
      }
    }
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
    const float2 sl2v = make_float2(sl2, sl2);
    // Only two key tiles can be ragged: the last prefix tile, and video tile T-1,
    // which (selections being ascending) can only be the item's last key tile.
    // Worked out from the geometry where they are needed, so that the block loops
    // hold no register for them.
    auto prefix_tail = [&]() { return G.TP > 0 ? G.P - (G.TP - 1) * kTile : kTile; };
    auto video_tail = [&]() { return G.Lv - (G.T - 1) * kTile; };
    // Blocks that may hold masked key lanes: the one with the ragged last prefix
    // tile, and the last block (an absent second tile, or ragged video tile T-1).
    const int ragged_prefix_blk = (G.TP > 0 && prefix_tail() < kTile) ? (G.TP - 1) / 2 : -1;
    bool failed = false;
    uint32_t gs = 0;  // blocks consumed so far, over all items
    for (int n = 0;; ++n) {
      bool ok = true;
      const int item = read_item(n, ok);
      failed = failed || !ok;
      // all softmax warps read the same item sequence; agree on stopping
      if (named_bar_or(kBarSoftmaxAll, 32 * kSoftmaxWarps, failed || item < 0)) break;
      Item it = decode_item(p, G, item);
      const int nblk = (it.n_kv + 1) / 2;
      const bool last_is_ragged =
          video_tail() < kTile && (it.list == nullptr || __ldg(it.list + G.k - 1) == G.T - 1);
      // Per column pair: -reference (log2 units) and this lane's partial row sums.
      float2 nm2[kCols / 2], l2[kCols / 2];
#pragma unroll
      for (int j = 0; j < kCols / 2; ++j) {
        nm2[j] = kExact ? make_float2(INFINITY, INFINITY) : make_float2(0.f, 0.f);
        l2[j] = make_float2(0.f, 0.f);
      }
      // ---- general block: masking, and (exact mode) the exact per-column block
      // maximum with rescaling. g: the block's ring counter.
      auto general_block = [&](const int i, const uint32_t g) {
        const int st = g % kNumS, pt = g % kNumP;
        const uint32_t ph = (g / kNumS) & 1, pph = (g / kNumP) & 1;
        const int ti = 2 * i + key_slot;
        bool valid = ti < it.n_kv;
        if (ti == G.TP - 1) valid = key_row < prefix_tail();
        if (ti == it.n_kv - 1 && last_is_ragged) valid = valid && key_row < video_tail();

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
        if (kExact) {
          const float mxall =
              fmax3(fmax3(fmax3(t[0], t[1], t[2]), fmax3(t[3], t[4], t[5]), fmax3(t[6], t[7], t[8])),
                    fmax3(t[9], t[10], t[11]), fmax3(fmax3(t[12], t[13], t[14]), t[15], -INFINITY));
          slow = named_bar_or(bar_id, 128, failed || mxall > kRescaleThreshold);
        }
        if (slow) {
          // slow path: exact block maximum per query column across the 128 key lanes.
          // A failed warp runs it on zeros (its outputs are void) and so meets
          // the same named barriers as the others; the item's end reports it.
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
          // every warp has read the block maxima before red is written again: in
          // exact mode by the next slow block; in fast mode only the item's end
          // writes red, after the all-softmax barrier there
          if (kExact) named_bar_sync(bar_id, 128);
          if (i > 0 && !failed) {
            // O^T must hold every PV product issued so far: wait for PV of block
            // g-1 on its P-buffer barrier (PV of block g-1-kNumP is already known
            // to be complete, so this parity wait cannot alias an older phase;
            // tcgen05 MMAs complete in issue order).
            const uint32_t gp = g - 1;
            failed = warp_any(!mbar_wait(bar(kBarPEmpty + gp % kNumP), (gp / kNumP) & 1, err, 0x900u));
            if (!failed) {
              tc_fence_after();
              uint32_t o[kCols];
              const uint32_t ocol = tbase + lane_off + kColO + static_cast<uint32_t>(n % kNumO) * 64 + col0;
              tmem_ld16(ocol, o);
              tmem_wait_ld();
#pragma unroll
              for (int c = 0; c < kCols; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha[c]);
              tmem_st16(ocol, o);
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
        failed = warp_any(failed || !mbar_wait(bar(kBarPEmpty + pt), pph ^ 1u, err, 0xA00u));
        if (!failed) {
          const uint32_t prow = sP + pt * kPBytes + r * 128;
#pragma unroll
          for (int cc = 0; cc < kCols / 8; ++cc) {
            const uint32_t chunk = static_cast<uint32_t>((col0 / 8 + cc) ^ (r & 7));
            st_shared_v4(prow + chunk * 16, pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kBarPFull + pt));
        }
      };
      // ---- fast-mode block: no masked lanes, fixed reference, no cross-lane
      // work. st / ph, pt / pph: S^T and P^T ring slots and phase parities.
      // Returns false once a wait has failed.
      auto fast_block = [&](const int st, const uint32_t ph, const int pt, const uint32_t pph) -> bool {
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
        if (warp_any(!mbar_wait(bar(kBarPEmpty + pt), pph ^ 1u, err, 0xA00u))) return false;
        const uint32_t prow = sP + pt * kPBytes + r * 128;
#pragma unroll
        for (int cc = 0; cc < kCols / 8; ++cc) {
          const uint32_t chunk = static_cast<uint32_t>((col0 / 8 + cc) ^ (r & 7));
          st_shared_v4(prow + chunk * 16, pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarPFull + pt));
        return true;
      };
      // The epilogue's gate and coarse inputs were prefetched into L2 when the
      // item was fetched; they are requested together, before the wait for the
      // item's last PV product. Each lane loads them in the layout of its output
      // stores: tokens col0 + tr and col0 + tr + 8, channels kc .. kc + 7.
      const int tr = lane >> 2;
      const int kc = 32 * q4 + 8 * (lane & 3);
      uint4 g8[2];     // gate, 8 bf16 per token
      float4 cz8[2];   // the coarse row's 8 channels
      long long my_row = 0;  // output row of query column col0 + (lane % kCols)
      auto prefetch_gate = [&]() {
        g8[0] = g8[1] = make_uint4(0u, 0u, 0u, 0u);
        cz8[0] = cz8[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (it.video && p.coarse) {
          const float4* crow = reinterpret_cast<const float4*>(
              p.coarse + ((static_cast<size_t>(it.b) * p.H + it.h) * p.T + it.t) * kHeadDim + kc);
          cz8[0] = __ldg(crow);
          cz8[1] = __ldg(crow + 1);
#pragma unroll
          for (int j = 0; j < 2; ++j)
            if (col0 + tr + 8 * j < it.q_valid)
              g8[j] = __ldg(reinterpret_cast<const uint4*>(
                  p.gate +
                  (static_cast<size_t>(it.b) * p.N + it.q_row0 + col0 + tr + 8 * j) * static_cast<size_t>(p.in_row_stride) +
                  static_cast<size_t>(it.h) * kHeadDim + kc));
        }
        const int qc = col0 + (lane % kCols);
        my_row = it.q_row0 + qc;
        if (p.out_row_map && qc < it.q_valid)
          my_row = __ldg(p.out_row_map + static_cast<size_t>(it.b) * p.N + it.q_row0 + qc);
      };
      if (kExact) {
        // every block, even after a failure, so that all warps meet the same
        // named barriers (a failed warp skips the work)
        for (int i = 0; i < nblk; ++i) general_block(i, gs + i);
      } else {
        // fast blocks 0 .. nblk-2, the ragged-prefix block (if any) excepted;
        // in fast mode the general blocks use no named barrier
        uint32_t g = gs;
        for (int i = 0; i < nblk - 1 && !failed; ++i, ++g) {
          if (i == ragged_prefix_blk) {
            general_block(i, g);
          } else if (!fast_block(g % kNumS, (g / kNumS) & 1, g % kNumP, (g / kNumP) & 1)) {
            failed = true;
          }
        }
        if (!failed) general_block(nblk - 1, gs + nblk - 1);
      }
      // decoded again: nothing of the item but n_kv is held through the block loops
      it = decode_item(p, G, item);
      const uint32_t ob = n % kNumO;
      // The fast mode is valid while every P stayed below kFastLimitSum: P >= 0,
      // so one larger P (or an overflow to inf) leaves a partial row sum at or
      // above that bound (a NaN fails the comparison too). Partials at or above
      // kFastMinSum keep every P that matters out of the subnormal range.
      // Only the item's valid query columns count: the others are never stored
      // (with device lengths their Q rows may be padding with any contents).
      bool overflow = false;
      if (!kExact) {
#pragma unroll
        for (int j = 0; j < kCols / 2; ++j)
          overflow = overflow ||
                     (col0 + 2 * j < it.q_valid && !(l2[j].x < kFastLimitSum && l2[j].x >= kFastMinSum)) ||
                     (col0 + 2 * j + 1 < it.q_valid && !(l2[j].y < kFastLimitSum && l2[j].y >= kFastMinSum));
      }
      // one barrier in the common case; a second tells a failure from an overflow
      if (named_bar_or(kBarSoftmaxAll, 32 * kSoftmaxWarps, failed || overflow)) {
        if (named_bar_or(kBarSoftmaxAll, 32 * kSoftmaxWarps, failed)) break;
        if (!kExact && tid == 32 * kWarpSoftmax0) {  // some column left the fast bounds
          const int pos = atomicAdd(p.redo_count, 1);  // at most once per item: pos < n_items
          p.redo_list[pos] = item;
        }
      }
      // ---- epilogue: out = O / l (+ sigmoid(gate) * coarse on video rows, unless
      // there is no coarse term: SubBlock routing)
      float l[kCols];
#pragma unroll
      for (int j = 0; j < kCols / 2; ++j) {
        l[2 * j] = l2[j].x;
        l[2 * j + 1] = l2[j].y;
      }
      const float lw = reduce_scatter16<false>(l, lane);
      if (lane < kCols) red[(wg * kCols + lane) * 4 + q4] = lw;
      named_bar_sync(bar_id, 128);
      // after the named barriers (which wait for a warp's outstanding loads),
      // so that these L2 reads overlap the drain of the last O^T product
      prefetch_gate();
      const uint32_t gl = gs + nblk - 1;  // the item's last PV product (see the rescale above)
      failed = warp_any(!mbar_wait(bar(kBarPEmpty + gl % kNumP), (gl / kNumP) & 1, err, 0xB00u));
      if (!failed) {
        tc_fence_after();
        uint32_t o[kCols];
        tmem_ld16(tbase + lane_off + kColO + ob * 64 + col0, o);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarOEmpty + ob));  // accumulator ob may be reused
        // Each warp stages O (fp32) in its own 2 KB of the P^T ring, then reads
        // it back eight channels a lane, so that the gate loads and the
        // output stores are 16 bytes a lane: two a lane per item instead of one
        // 2-byte access per lane and column. The ring is idle here: the item's
        // last PV product has completed, and the next P^T is written after the
        // all-softmax barrier at the next item's start. Word (column c, channel
        // d) sits at 32 c + ((d + 4 (c & 1)) mod 32): both the column-wise writes
        // and the 16-byte reads are free of bank conflicts.
        const uint32_t stage = sP + static_cast<uint32_t>(warp - kWarpSoftmax0) * 2048u;
#pragma unroll
        for (int c = 0; c < kCols; ++c) {
          const uint32_t w = 32u * c + ((static_cast<uint32_t>(lane) + 4u * (c & 1)) & 31u);
          st_shared_f32(stage + 4u * w, __uint_as_float(o[c]));
        }
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int c = tr + 8 * j;
          const int qc = col0 + c;
          const long long row = __shfl_sync(0xffffffffu, my_row, c);
          const uint32_t w0 = (8u * static_cast<uint32_t>(lane & 3) + 4u * (c & 1)) & 31u;
          const float4 v0 = ld_shared_f4(stage + 4u * (32u * c + w0));
          const float4 v1 = ld_shared_f4(stage + 4u * (32u * c + ((w0 + 4u) & 31u)));
          if (qc < it.q_valid) {
            const float4 x = reinterpret_cast<const float4*>(red)[wg * kCols + c];
            const float lsum = (x.x + x.y) + (x.z + x.w);
            float val[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) val[e] = __fdividef(val[e], lsum);
            if (it.video && p.coarse) {
              const float cz[8] = {cz8[0].x, cz8[0].y, cz8[0].z, cz8[0].w, cz8[1].x, cz8[1].y, cz8[1].z, cz8[1].w};
              const uint32_t gw[4] = {g8[j].x, g8[j].y, g8[j].z, g8[j].w};
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const float gv = __uint_as_float((e & 1) ? (gw[e / 2] & 0xffff0000u) : (gw[e / 2] << 16));
                val[e] += __fdividef(cz[e], 1.0f + __expf(-gv));
              }
            }
            if (row >= 0 && row < p.out_rows) {
              *reinterpret_cast<uint4*>(p.out + (static_cast<size_t>(it.b) * p.out_rows + row) * p.out_row_stride +
                                        static_cast<size_t>(it.h) * kHeadDim + kc) =
                  make_uint4(pack_bf16x2(val[0], val[1]), pack_bf16x2(val[2], val[3]),
                             pack_bf16x2(val[4], val[5]), pack_bf16x2(val[6], val[7]));
            } else if (q4 == 0 && (lane & 3) == 0) {  // a map entry outside the output: skipped and reported (token + 1)
              atomicCAS(err + 3, 0u, static_cast<unsigned int>(it.q_row0 + qc) + 1u);
            }
          }
        }
      }
      // every warp has read the row sums before red is written again
      named_bar_sync(bar_id, 128);
      gs += nblk;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMmaS) tmem_dealloc(*tslot, kTmemCols);
}

}  // namespace

size_t fine_smem_bytes() { return kSmemBytes; }

cudaError_t launch_fine(const Geometry& g, const CUtensorMap& map_q, const CUtensorMap& map_k,
                        const CUtensorMap& map_v, const CUtensorMap& map_gate, const FineArgs& a, int num_sms,
                        cudaStream_t stream) {
  FineParams p;
  p.B = g.B; p.H = g.H; p.P = g.P; p.Lv = g.Lv; p.N = g.N; p.T = g.T; p.TP = g.TP; p.k = g.k;
  p.n_items = g.B * g.H * (g.TP + g.T);  // the capacity's, for the grid; the kernels use FineGeo
  p.dl = a.dl;
  p.scale_log2 = 1.4426950408889634f * 0.08838834764831845f;
  p.gate = a.gate;
  p.out = a.out;
  p.out_row_map = a.out_row_map;
  p.out_rows = a.out_row_map ? a.out_rows : g.N;
  p.out_row_stride = a.out_row_stride > 0 ? a.out_row_stride : static_cast<long long>(g.H) * kHeadDim;
  p.in_row_stride = input_row_stride(g);
  p.coarse = a.coarse;
  p.tile_index = a.tile_index;
  p.err = a.err;
  p.redo_count = a.redo_count;
  p.redo_list = a.redo_list;
  const int grid = p.n_items < num_sms ? p.n_items : num_sms;
  cudaError_t e = cudaFuncSetAttribute(fine_attn_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(fine_attn_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  p.work_counter = a.work_counters;
  fine_attn_kernel<false><<<grid, kThreads, kSmemBytes, stream>>>(map_q, map_k, map_v, map_gate, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // Items whose fast-mode softmax left its range: recomputed with exact
  // rescaling (an empty list costs one launch whose CTAs return at once).
  p.work_counter = a.work_counters + 1;
  fine_attn_kernel<true><<<grid, kThreads, kSmemBytes, stream>>>(map_q, map_k, map_v, map_gate, p);
  return cudaGetLastError();
}

}  // namespace vsa
