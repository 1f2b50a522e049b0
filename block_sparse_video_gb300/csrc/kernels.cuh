// Internal interface between the C-ABI host code and the kernels.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace vsa {

constexpr int kTile = 64;
constexpr int kHeadDim = 128;

// Problem geometry shared by the kernels. Token layout is [B, N, H, 128] with
// the prefix (text then audio, P tokens) first and Lv video tokens after it.
struct Geometry {
  int B = 0, H = 0;
  int P = 0;   // prefix tokens (text + audio)
  int Lv = 0;  // video tokens
  int N = 0;   // P + Lv
  int T = 0;   // video tiles, ceil(Lv / 64)
  int TP = 0;  // prefix tiles, ceil(P / 64)
  int k = 0;   // kept video tiles per video query tile
  // Elements between consecutive token rows of q, k, v and gate; 0 means
  // H * 128 (packed). A larger stride reads H heads out of a wider row, e.g.
  // one rank's head slice of the full projection.
  long long row_stride = 0;
};

__host__ __device__ __forceinline__ long long input_row_stride(const Geometry& g) {
  return g.row_stride > 0 ? g.row_stride : static_cast<long long>(g.H) * kHeadDim;
}

// Lengths read on the device (a capacity plan's forward): the plan's geometry
// is the capacity (buffer rows per batch N, tiles T, kept tiles k: the layout
// strides); the actual text/audio/video lengths come from `len` (3 x int64)
// and must satisfy text, audio >= 0, 1 <= video <= Lv, text + audio <= P.
struct DeviceLengths {
  const long long* len = nullptr;  // null: the plan's own lengths
  double keep = 0.0;               // keep fraction (the actual k is derived from the actual T)
  double sparsity = -1.0;          // >= 0: SubBlock routing's sparsity (its own rule for k)
  unsigned int* invalid = nullptr; // set to 1 when the lengths are outside the capacity
};

// Actual geometry of one forward: the plan's, or the one the device lengths give.
struct DynGeom {
  int P, Lv, T, TP, k;
  bool valid;
};

__device__ __forceinline__ DynGeom dyn_geom(const Geometry& cap, const DeviceLengths& dl) {
  DynGeom d{cap.P, cap.Lv, cap.T, cap.TP, cap.k, true};
  if (!dl.len) return d;
  const long long text = dl.len[0], audio = dl.len[1], video = dl.len[2];
  if (text < 0 || audio < 0 || video < 1 || video > cap.Lv || text + audio > cap.P) {
    d.valid = false;
    return d;
  }
  d.P = static_cast<int>(text + audio);
  d.Lv = static_cast<int>(video);
  d.T = (d.Lv + kTile - 1) / kTile;
  d.TP = (d.P + kTile - 1) / kTile;
  int k;
  if (dl.sparsity >= 0.0) {
    // SubBlock: at most floor(s T) tiles dropped (IEEE double), the kept count
    // rounded up to a multiple of 8
    const int need = d.T - static_cast<int>(floor(dl.sparsity * static_cast<double>(d.T)));
    k = (need + 7) / 8 * 8;
  } else {
    // "rounded to a whole number of tiles": round half up in IEEE double
    k = static_cast<int>(floor(dl.keep * static_cast<double>(d.T) + 0.5));
  }
  d.k = k < 1 ? 1 : (k > d.T ? d.T : k);  // clamped to [1, T]
  return d;
}

// Tile pool: mean over the valid tokens of each video tile of q, k and v.
// pooled_* are fp32 [B, H, T, 128] (T of the plan: the layout stride).
cudaError_t launch_pool(const Geometry& g, const __nv_bfloat16* q, const __nv_bfloat16* k,
                        const __nv_bfloat16* v, float* pooled_q, float* pooled_k,
                        float* pooled_v, const DeviceLengths& dl, cudaStream_t stream);

// Fused attention preprocessing: Q/K RMSNorm, partial RoPE, packing of the
// projection rows into [B, N, H, 128], gate copy and the Q/K/V tile pooling.
struct PreprocessArgs {
  const __nv_bfloat16* in[4];  // q, k, v, gate projections: row r of batch b at in + (b*rows_in + r)*row_stride
  long long rows_in;           // projection rows per batch
  long long row_stride;        // elements between projection rows
  const int32_t* src_row;      // int32 [B, N] or null (row n)
  const float* q_norm_weight;  // fp32 [H, 128]
  const float* k_norm_weight;
  float eps;
  int rope_dim;                // multiple of 16 in [0, 128]
  int rope_interleaved;        // pairs (2i, 2i+1) if nonzero, else (i, i + rope_dim/2)
  const float* rope_cos;       // fp32 [N, rope_dim/2]
  const float* rope_sin;
  __nv_bfloat16* out[4];       // packed q, k, v, gate, bf16 [B, N, H, 128]
  float* pooled[3];            // fp32 [B, H, T, 128]; null: no pooling
  unsigned int* err;           // error words; word 7 records the first bad map entry (token + 1)
  DeviceLengths dl;            // request lengths read on the device (null: the plan's)
};
cudaError_t launch_preprocess(const Geometry& g, const PreprocessArgs& a, cudaStream_t stream);

// Coarse attention over pooled tiles fused with the top-k tile selection.
// coarse fp32 [B, H, T, 128]; tile_index int32 [B, H, T, k] ascending.
size_t coarse_smem_bytes(const Geometry& g, int* rows_per_cta);
// vfrag: workspace of coarse_vfrag_bytes(g) for the pooled K and V in mma
// fragment form (written by a first, small kernel of the launch).
size_t coarse_vfrag_bytes(const Geometry& g);
cudaError_t launch_coarse_topk(const Geometry& g, const float* pooled_q, const float* pooled_k,
                               const float* pooled_v, float* coarse, int32_t* tile_index, void* vfrag,
                               const DeviceLengths& dl, cudaStream_t stream);

// Coarse attention + top-k with both products on the tcgen05 tensor cores,
// for up to kCoarseTcMaxT video tiles (longer videos take the kernel above).
// launch_split writes the pooled q, k, v as bf16 hi/lo rows (`operands`:
// [q, k, v][hi, lo][B H][coarse_tc_padded(g)][128], coarse_tc_operand_bytes);
// launch_coarse_tc reads them through `maps` (q hi, q lo, k hi, k lo, v hi,
// v lo: {128 channels, padded rows, B H, 1}, boxes of 64 x 64, 128-byte
// swizzled; then the scratch rows as bf16 {padded keys, 2 planes, 64 rows,
// slots}, boxes of 64 keys x 1 x 64 rows) and keeps its score rows in
// `scratch` (coarse_tc_scratch_bytes: one 64-row buffer per CTA).
constexpr int kCoarseTcMaxT = 2304;  // a query row of scores fits 72 registers per lane
constexpr int kCoarseTcMaxSlots = 160;  // CTAs of the persistent grid, at most
int coarse_tc_padded(const Geometry& g);
bool coarse_tc_supported(const Geometry& g);
int coarse_tc_units(const Geometry& g);
size_t coarse_tc_operand_bytes(const Geometry& g);
size_t coarse_tc_scratch_bytes(const Geometry& g);
cudaError_t launch_split(const Geometry& g, const float* pooled_q, const float* pooled_k, const float* pooled_v,
                         void* operands, const DeviceLengths& dl, cudaStream_t stream);
cudaError_t launch_coarse_tc(const Geometry& g, const CUtensorMap (&maps)[7], float* scratch, float* coarse,
                             int32_t* tile_index, unsigned int* err, const DeviceLengths& dl, int num_sms,
                             cudaStream_t stream);

// SubBlock routing: 16-token sub-block means of q and k (fp32 [B, H, 4T, 128],
// empty sub-blocks of a ragged last tile as 0, plus the same values split into
// bf16 hi + lo rows: frag_* holds hi [B, H, spad, 128] then lo [B, H, spad,
// 128], spad = subblock_rows_padded(g), 512 bytes per sub-row in all), then
// the k video key tiles of highest estimated softmax mass per video query tile
// (tile_index int32 [B, H, T, k], ascending).
int subblock_rows_padded(const Geometry& g);
// With device lengths (dl.len, dl.sparsity set) g is the capacity: both
// kernels keep its layout and work on the request's tiles.
cudaError_t launch_subpool(const Geometry& g, const __nv_bfloat16* q, const __nv_bfloat16* k, float* sub_q,
                           float* sub_k, void* frag_q, void* frag_k, const DeviceLengths& dl, cudaStream_t stream);
size_t subblock_router_smem_bytes(const Geometry& g, int* rows_per_cta);
// maps: the sub-pool's bf16 rows as TMA views {128 channels, spad rows, B H,
// 1}, boxes of 64 channels x 64 rows, 128-byte swizzled: q hi, q lo, k hi,
// k lo.
cudaError_t launch_subblock_router(const Geometry& g, const CUtensorMap (&maps)[4], int32_t* tile_index,
                                   unsigned int* err, const DeviceLengths& dl, cudaStream_t stream);

// Fine attention: prefix query tiles over every key, video query tiles over
// the prefix plus their selected video tiles; epilogue adds sigmoid(gate) *
// coarse on video rows and writes bf16 out.
// Launches two persistent kernels of num_sms CTAs (at most one per item): the
// fast one over every item, then the exact one over the items the fast one
// appended to the redo list.
struct FineArgs {
  const __nv_bfloat16* gate;
  __nv_bfloat16* out;          // row r of batch b at out + (b * out_rows + r) * out_row_stride
  const int32_t* out_row_map;  // null: token n -> row n (out_rows = N); else row map[b * N + n]
  long long out_rows = 0;
  long long out_row_stride = 0;  // 0: num_heads * 128
  const float* coarse;         // null: no gated coarse term (SubBlock routing)
  const int32_t* tile_index;
  unsigned int* err;   // error words in the workspace; word 3 records the first bad output map entry
  int* redo_count;     // zero before the launch
  int* redo_list;      // int32 [B * H * (TP + T)]
  int* work_counters;  // 2 counters, zero before the launch
  DeviceLengths dl;
};

size_t fine_smem_bytes();
cudaError_t launch_fine(const Geometry& g, const CUtensorMap& map_q, const CUtensorMap& map_k,
                        const CUtensorMap& map_v, const CUtensorMap& map_gate, const FineArgs& a, int num_sms,
                        cudaStream_t stream);

}  // namespace vsa
