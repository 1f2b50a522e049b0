/*
 * vsa.h - C ABI of the GB300 (sm_103a) video sparse attention (VSA) forward.
 *
 * The operation is the attention of one joint text+audio+video DiT layer as
 * "UniServe: serving FastH3 at its fastest" defines it:
 *   - section "The FastH3 workload": the sequence is processed in tiles of 64
 *     tokens; text and audio queries attend to every key; video queries attend
 *     to every text and audio key and to the highest-scoring fraction (20% in
 *     FastH3) of video key tiles, rounded to a whole number of tiles; a coarse
 *     branch attends over mean-pooled tiles, and a learned gate adds its
 *     output to the fine sparse-attention output;
 *   - section "Fused attention preprocessing": tiles are pooled over their
 *     valid tokens into FP32 pooled statistics;
 *   - section "Fused output combination": O_i = O_i^fine + G_i * O^coarse_tile(i);
 *   - section "Benchmarks / Setup": the top-k video tiles are selected exactly.
 *
 * Conventions fixed by this library where the page leaves them open:
 *   - memory order of the segments is text | audio | video (prefix P = text +
 *     audio tokens, then Lv video tokens, N = P + Lv); video tokens arrive
 *     tile-contiguous: video tile j is tokens P + 64j .. P + 64j + n_j - 1,
 *     T = ceil(Lv / 64) tiles, the last one may be ragged (n_j < 64);
 *   - tile score s[t][j] = (mean-pooled Q of tile t) . (mean-pooled K of tile
 *     j) / sqrt(128), computed in fp32; the coarse softmax runs over all T
 *     video tiles; prefix tokens are not tiles of the coarse branch;
 *   - k = max(1, min(T, floor(keep_fraction * T + 0.5))) in IEEE double;
 *     equal scores go to the lower tile index; selections are stored in
 *     ascending tile order;
 *   - G = sigmoid(gate) per channel; text/audio rows get no coarse term;
 *   - softmax scale 1/sqrt(128) in both branches.
 *
 * Data layout: q, k, v, gate and out are contiguous bf16 tensors of shape
 * [batch, N, num_heads, 128] (token-major, heads interleaved: the natural
 * output of the Q/K/V/gate projections), 16-byte aligned. All device buffers
 * are owned by the caller; the library owns only the host-side plan.
 *
 * Errors: argument errors are returned synchronously and nothing is launched.
 * CUDA errors at launch come back as VSA_ERR_CUDA. Every wait inside the
 * kernels is bounded; a wait that runs out records VSA_ERR_DEVICE_TIMEOUT in
 * the workspace's error words (the kernels then finish early), which
 * vsa_check() reports. The library never aborts the process.
 *
 * Threading: a plan may be used from one host thread at a time. Concurrent
 * forwards on different streams need different workspaces.
 */
#ifndef VSA_H_
#define VSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  VSA_OK = 0,
  VSA_ERR_INVALID_ARG = 1,    /* null pointer, bad length, keep fraction outside (0, 1], ... */
  VSA_ERR_UNSUPPORTED = 2,    /* head_dim other than 128, sizes beyond the supported range */
  VSA_ERR_CUDA = 3,           /* a CUDA runtime/driver call failed */
  VSA_ERR_DEVICE_TIMEOUT = 4, /* a bounded wait inside a kernel ran out (reported by vsa_check) */
  VSA_ERR_INTERNAL = 5
} vsa_status_t;

/* Problem shape. head_dim must be 128. len_text and len_audio may be 0;
 * len_video must be >= 1. keep_fraction in (0, 1]. batch, num_heads >= 1. */
typedef struct {
  int32_t batch;
  int32_t num_heads;
  int32_t head_dim;
  int64_t len_text;
  int64_t len_audio;
  int64_t len_video;
  double keep_fraction;
} vsa_shape_t;

typedef struct vsa_plan* vsa_plan_t; /* opaque, host memory, owned by the library */

/* "vsa_plan": validate a shape and precompute T, k, the workspace size and the
 * launch configuration for `device`. Host only: touches no GPU state and
 * allocates no device memory, so it may run on a machine without a GPU.
 * On success *out receives a plan to release with vsa_plan_destroy. */
vsa_status_t vsa_plan_create(const vsa_shape_t* shape, int device, vsa_plan_t* out);

/* A plan whose selection is the SubBlock router (the SGLang Diffusion benchmark page (MiniMax-H3 on 8x H200),
 * section "How SubBlock Sparse Attention Works") in place of the
 * coarse branch. Each 64-token tile splits into four 16-token sub-blocks on
 * the query and key side. The estimated softmax mass of video key tile j for
 * video query tile i is
 *   score(i, j) = log sum_{a,b} n_a n_b exp(q_a . k_b / sqrt(128))
 * over the non-empty sub-blocks a of tile i and b of tile j, where q_a and k_b
 * are the sub-block means and n_a, n_b their token counts. Each video query
 * tile keeps the k video key tiles of highest score (ties to the lower tile,
 * ascending).
 *
 * `sparsity` in [0, 1) is the fraction of key tiles that may be dropped:
 * k = min(T, 8 * ceil((T - floor(sparsity * T)) / 8)), with the floor in IEEE
 * double. Text and audio stay dense as in the VSA forward. There is no coarse
 * branch: vsa_forward on this plan computes out = fine attention, and its gate
 * argument is ignored and may be NULL. shape->keep_fraction is ignored.
 *
 * The forward enqueues four kernels: sub-block pooling of Q and K, the
 * router, and the fine attention's fast and exact passes. vsa_debug_views
 * returns the sub-block means (fp32 [batch, num_heads, 4T, 128], empty
 * sub-blocks of a ragged last tile as 0) as pooled_q and pooled_k, NULL for
 * pooled_v and coarse, and the selection as tile_index [batch, num_heads, T, k].
 * vsa_preprocess on this plan packs the tensors but pools nothing. Otherwise
 * as vsa_plan_create. */
vsa_status_t vsa_plan_create_subblock(const vsa_shape_t* shape, double sparsity, int device, vsa_plan_t* out);

/* Number of video tiles T, kept tiles per query tile k, and the device
 * workspace vsa_forward needs, in bytes. Any output pointer may be NULL. */
vsa_status_t vsa_plan_info(vsa_plan_t plan, int64_t* n_tiles, int64_t* k, size_t* workspace_bytes);

/* The VSA forward: out = fine attention (+ sigmoid(gate) * coarse on video rows).
 *   q, k, v, gate : device, bf16 [batch, N, num_heads, 128], read only
 *   out           : device, bf16 [batch, N, num_heads, 128], written; must not
 *                   alias any input
 *   workspace     : device, >= workspace_bytes from vsa_plan_info, 256-byte
 *                   aligned; holds pooled statistics, tile selections, the
 *                   coarse output and the error words; contents on entry are
 *                   ignored (the forward clears what must start at zero)
 *   stream        : cudaStream_t to launch on (NULL = legacy default stream)
 * Enqueues five kernels (tile pool; the pooled K and V in tensor-core fragment form;
 * coarse attention + top-k; fine attention with the gated combination fused
 * into its epilogue; the fine attention's exact pass over the query tiles whose
 * fast pass left its numeric range, which returns at once when there are none)
 * and returns without synchronising. It
 * allocates nothing and reads no device data on the host. The first call on a
 * plan reads the device's SM count (cudaDeviceGetAttribute). */
vsa_status_t vsa_forward(vsa_plan_t plan, const void* q, const void* k, const void* v,
                         const void* gate, void* out, void* workspace, size_t workspace_bytes,
                         void* stream);

/* Lengths of one request, read by the kernels at run time (device memory,
 * 8-byte aligned): the token counts of the text, audio and video segments. */
typedef struct {
  int64_t len_text;
  int64_t len_audio;
  int64_t len_video;
} vsa_lengths_t;

/* Fused attention preprocessing ("UniServe: serving FastH3 at its fastest",
 * section "Fused attention preprocessing"; section "The Kernel Layer" of
 * the SGLang Diffusion benchmark page (MiniMax-H3 on 8x H200) gives the
 * rotary width of 96 channels and the rounding of the normalised value before
 * RoPE). One pass over the projected Q/K/V/gate rows does the following:
 *   - packs each attention token's row into the [batch, N, num_heads, 128]
 *     layout the forward reads;
 *   - applies RMSNorm to Q and K, per token and head over the head's 128
 *     channels: y = x / sqrt(mean(x^2) + eps) * weight[head][channel];
 *   - rounds the result to bf16 and rotates channels [0, rope_dim) of every
 *     head: the pair (a, b) at token n becomes (a cos - b sin, a sin + b cos),
 *     with cos and sin from the tables; the result is rounded to bf16 (RNE);
 *   - copies V and the gate;
 *   - writes the FP32 tile means of the packed Q, K and V (over each video
 *     tile's valid tokens) into the workspace, where vsa_forward_preprocessed
 *     reads them.
 * Padding rows of the projection buffer are never read unless the map points
 * at them. */
typedef struct {
  /* Projections, device, bf16. Channel c of head h of projection row r of
   * batch b is at ptr + (b * rows_in + r) * row_stride + h * 128 + c (elements).
   * 16-byte aligned. The four may share one buffer (e.g. one merged projection
   * with row_stride = 4 * num_heads * 128). */
  const void* q_in;
  const void* k_in;
  const void* v_in;
  const void* gate_in;
  int64_t rows_in;    /* projection rows per batch (capacity, may include padding), >= 1 */
  int64_t row_stride; /* elements between projection rows: >= num_heads * 128, multiple of 8 */
  /* Device int32 [batch, N]: the projection row of attention token n (segments
   * text | audio | video). NULL means row n (then rows_in >= N). An entry outside
   * [0, rows_in) gives a zero row, and vsa_check reports VSA_ERR_INVALID_ARG. */
  const int32_t* src_row;
  const float* q_norm_weight; /* device fp32 [num_heads, 128] */
  const float* k_norm_weight; /* device fp32 [num_heads, 128] */
  float eps;                  /* > 0 */
  int32_t rope_dim;           /* rotated channels per head: multiple of 16 in [0, 128] */
  int32_t rope_interleaved;   /* nonzero: pairs (2i, 2i+1); zero: pairs (i, i + rope_dim/2) */
  /* Device fp32 [N, rope_dim / 2], 16-byte aligned: cos and sin of the angle
   * of pair i at attention token n (any 1-D or 3-D position encoding). Unused
   * when rope_dim = 0. */
  const float* rope_cos;
  const float* rope_sin;
  /* Outputs, device bf16 [batch, N, num_heads, 128], 16-byte aligned. They must
   * not overlap one another, any input or the workspace. */
  void* q_out;
  void* k_out;
  void* v_out;
  void* gate_out;
  /* Device lengths of the request (see vsa_forward_lengths), or NULL for the
   * plan's own. With lengths the plan's shape is the capacity: N above is the
   * plan's row count (the src_row stride, the RoPE table rows and the output
   * rows per batch), and only the request's tokens are written. */
  const vsa_lengths_t* lengths;
} vsa_preprocess_args_t;

/* Enqueue the fused preprocessing on `stream`. `workspace` is this plan's
 * forward workspace (vsa_plan_info): the pooled statistics go there, and its
 * error words are cleared first. Argument
 * errors are returned synchronously and nothing is launched. Allocates nothing,
 * does not synchronise and reads no device data on the host, so it is
 * capture-safe. */
vsa_status_t vsa_preprocess(vsa_plan_t plan, const vsa_preprocess_args_t* args, void* workspace,
                            size_t workspace_bytes, void* stream);

/* vsa_forward for inputs packed by vsa_preprocess into the same workspace on
 * the same stream: skips the tile pool (the pooled statistics are already in
 * the workspace) and keeps the preprocessing's error report for vsa_check.
 * Three kernels; otherwise as vsa_forward. */
vsa_status_t vsa_forward_preprocessed(vsa_plan_t plan, const void* q, const void* k, const void* v,
                                      const void* gate, void* out, void* workspace,
                                      size_t workspace_bytes, void* stream);


/* The forward of a request whose lengths live in DEVICE memory, inside a
 * capacity-padded buffer ("UniServe: serving FastH3 at its fastest", section
 * "Architecture": workspaces are allocated once for the largest shape and
 * smaller shapes run on views of it; CUDA graphs are captured once per shape
 * bucket and address each request through device-side tensors).
 *
 * The plan's shape is the capacity. q, k, v, gate and out are bf16
 * [batch, N_cap, num_heads, 128] with N_cap = the plan's text + audio + video.
 * The request's tokens occupy rows 0 .. N - 1 of each batch (text, then audio,
 * then video, N = len_text + len_audio + len_video). The kernels read
 * *lengths when they run, so one captured graph of this call serves every
 * request that fits the capacity: write the next request's lengths into the
 * same device buffer and replay.
 *
 * Requirements and effects:
 *   - 0 <= len_text, 0 <= len_audio, len_text + len_audio <= the plan's
 *     len_text + len_audio, and 1 <= len_video <= the plan's len_video.
 *     Otherwise nothing is computed, out is untouched and vsa_check reports
 *     VSA_ERR_INVALID_ARG;
 *   - k follows the plan's rule for the request's T: max(1, min(T,
 *     floor(keep_fraction * T + 0.5))); for a SubBlock plan, the kept count
 *     T - floor(sparsity * T) rounded up to a multiple of 8, capped at T;
 *   - rows N .. N_cap - 1 of q, k, v and gate (capacity padding) may hold
 *     anything, NaN and Inf included: a ragged tile's 64-row loads read
 *     some of them, and the forward masks their keys, clears their V rows in
 *     shared memory before the P.V product, and never stores or votes on
 *     their query rows, so no padding value reaches the output;
 *   - rows N .. N_cap - 1 of out are not written;
 *   - the workspace and its views (vsa_debug_views) keep the plan's layout:
 *     the request's tiles are the first T rows of each [T_cap] block, and
 *     its selections the first k entries of each row of k_cap.
 * SubBlock plans (gate may be NULL) run their four kernels the same way: the
 * sub-block pool and the router read the lengths too. Otherwise as
 * vsa_forward (capture-safe, five kernels). */
vsa_status_t vsa_forward_lengths(vsa_plan_t plan, const vsa_lengths_t* lengths, const void* q, const void* k,
                                 const void* v, const void* gate, void* out, void* workspace,
                                 size_t workspace_bytes, void* stream);

/* Where the forward writes its output rows. The combined rows can go straight
 * into another layout, such as the send buffer of the output all-to-all that
 * restores sequence sharding ("UniServe: serving FastH3 at its fastest",
 * section "Fused output combination": the combination kernel writes each row
 * directly into its position in the send buffer). Attention token n of batch
 * b (segments text | audio | video) is written to row
 *   out_row_map[b * N + n]        (or n when out_row_map is NULL)
 * of batch b. Channel c of head h of output row r of batch b is at
 *   out + (b * out_rows + r) * out_row_stride + h * 128 + c   (elements, bf16).
 * When sequence shards are contiguous row ranges, the rank-major send buffer
 * is the sequence order itself. out_row_map is then the map that packed the
 * rows (vsa_preprocess_args_t.src_row), and out_row_stride is num_heads * 128.
 * Rows no token maps to are left untouched. A map entry outside
 * [0, out_rows) skips that row, and vsa_check reports VSA_ERR_INVALID_ARG. */
typedef struct {
  void* out;                   /* device bf16, 16-byte aligned; must not overlap the inputs or the workspace */
  int64_t out_rows;            /* rows per batch, >= 1 (>= N without a map) */
  int64_t out_row_stride;      /* elements between rows: >= num_heads * 128, multiple of 8 */
  const int32_t* out_row_map;  /* device int32 [batch, N], or NULL */
} vsa_output_rows_t;

/* vsa_forward (preprocessed = 0) or vsa_forward_preprocessed (preprocessed != 0)
 * writing its rows through `out` as described above. Same errors, same
 * kernels, capture-safe. */
vsa_status_t vsa_forward_rows(vsa_plan_t plan, const void* q, const void* k, const void* v, const void* gate,
                              const vsa_output_rows_t* out, int32_t preprocessed, void* workspace,
                              size_t workspace_bytes, void* stream);

/* The general forward: every option of the entry points above in one call.
 *   q, k, v, gate : as vsa_forward (gate may be NULL for a SubBlock plan), or
 *                   head slices of wider rows (in_row_stride)
 *   out           : packed bf16 [batch, N, num_heads, 128] output, used when
 *                   rows is NULL
 *   rows          : output rows (vsa_forward_rows), or NULL
 *   lengths       : device lengths of the request (vsa_forward_lengths), or
 *                   NULL for the plan's own
 *   preprocessed  : nonzero when q, k, v, gate and the pooled statistics come
 *                   from vsa_preprocess on this workspace and stream
 *   in_row_stride : elements between consecutive token rows of q, k, v and
 *                   gate; 0 means num_heads * 128 (packed). Otherwise a
 *                   multiple of 8, >= num_heads * 128 and <= 2^24: channel c
 *                   of head h of token n of batch b is read at
 *                   x + (b * N + n) * in_row_stride + h * 128 + c. This is the
 *                   head split of "UniServe: serving FastH3 at its fastest",
 *                   section "The FastH3 workload" (each of 4 GPUs attends for
 *                   14 of the 56 heads): a plan of num_heads = 14 given
 *                   q + 14 r * 128 and in_row_stride = 56 * 128 computes heads
 *                   14 r .. 14 r + 13 of a 56-head projection in place, and
 *                   rows (out_row_stride = 56 * 128, out + 14 r * 128) writes
 *                   them into the matching head slice of a 56-head output.
 * With lengths, preprocessed and rows together, one captured graph runs the
 * whole serving step: pack and normalise a request from its capacity-padded
 * projection buffer, attend, and write the combined rows into the all-to-all
 * send layout, for any request the capacity holds. */
typedef struct {
  const void* q;
  const void* k;
  const void* v;
  const void* gate;
  void* out;
  const vsa_output_rows_t* rows;
  const vsa_lengths_t* lengths;
  int32_t preprocessed;
  int64_t in_row_stride;
} vsa_forward_args_t;

vsa_status_t vsa_forward_ex(vsa_plan_t plan, const vsa_forward_args_t* args, void* workspace,
                            size_t workspace_bytes, void* stream);

/* Same forward on HOST buffers (q, k, v, gate read, out written, all bf16
 * [batch, N, num_heads, 128]; pinned memory makes the copies asynchronous; the
 * gate may be NULL for a SubBlock plan). `device_buffer` (>= host_path_bytes
 * from vsa_plan_host_path_bytes, 256-byte aligned) receives the inputs, the
 * output and the workspace.
 *
 * With two or more heads the work is pipelined over head groups (up to 8
 * heads: two halves; beyond, groups of 4, 6, then 8 heads, the rest last,
 * split into a group and a final 2-head group when it has 4 heads or more):
 *   * each group's heads are copied in on a library-owned stream (strided
 *     copies of each host row's slice). When q, k, v (and gate) are pinned or
 *     registered host memory, the first group's slices are instead gathered by
 *     a kernel that reads the host memory directly;
 *   * the group's forward runs on `stream`;
 *   * its output is copied out on a second library-owned stream (the last
 *     group's, when out is pinned, by a kernel writing the host memory);
 *   * two groups' device buffers alternate.
 * The results equal vsa_forward's bit for bit. The two streams and their
 * events are created on the first call and released by vsa_plan_destroy.
 * Synchronises `stream` before returning; device-side errors are not reported
 * here. */
vsa_status_t vsa_plan_host_path_bytes(vsa_plan_t plan, size_t* bytes);

/* Where vsa_forward_host places head group `group` in its device buffer
 * (host only; touches no GPU). *n_groups receives the number of groups.
 * Group `group` covers heads [*first_head, *first_head + *heads); its q, k,
 * v, gate and output are bf16 [batch, N, *heads, 128] tensors of
 * *tensor_bytes bytes at byte offsets offsets[0..4] (5 entries, caller
 * storage); the workspace its forward uses is [*workspace_offset,
 * *workspace_offset + *workspace_bytes), shared by every group. Groups
 * alternate between two slots and each slot keeps inputs and output apart at
 * the widest group's tensor stride. The call order behind the layout: the
 * copy-in of group g waits for the forward of group g - 2; the forward of g
 * waits for its own copy-in and for the copy-out of g - 2; the copy-out of g
 * waits for the forward of g; each of the three streams runs in order.
 * Returns VSA_ERR_INVALID_ARG for a NULL pointer or a group outside
 * [0, *n_groups) (*n_groups is still set when n_groups is non-NULL). */
vsa_status_t vsa_plan_host_path_group(vsa_plan_t plan, int32_t group, int32_t* n_groups, int32_t* first_head,
                                      int32_t* heads, size_t* offsets, size_t* tensor_bytes,
                                      size_t* workspace_offset, size_t* workspace_bytes);

vsa_status_t vsa_forward_host(vsa_plan_t plan, const void* q, const void* k, const void* v,
                              const void* gate, void* out, void* device_buffer,
                              size_t device_buffer_bytes, void* stream);

/* Device pointers to the intermediates a forward leaves in `workspace`:
 *   pooled_q/k/v : fp32 [batch, num_heads, T, 128] tile means
 *   tile_index   : int32 [batch, num_heads, T, k] selected video tiles, ascending
 *   coarse       : fp32 [batch, num_heads, T, 128] coarse-branch output
 * Any output pointer may be NULL. */
vsa_status_t vsa_debug_views(vsa_plan_t plan, void* workspace, const float** pooled_q,
                             const float** pooled_k, const float** pooled_v,
                             const int32_t** tile_index, const float** coarse);

/* Synchronise `stream` and report the device error words of `workspace`:
 * VSA_OK; VSA_ERR_DEVICE_TIMEOUT if a bounded wait gave up; VSA_ERR_INVALID_ARG
 * if the last vsa_preprocess met a map entry outside its projection buffer,
 * the last vsa_forward_rows an output map entry outside its rows, or the last
 * vsa_forward_lengths lengths outside the plan's capacity. */
vsa_status_t vsa_check(vsa_plan_t plan, void* workspace, void* stream);

/* Optional per-kernel timing. When `events` is non-NULL, each vsa_forward
 * records events[0] before the pool kernel, events[1] before the coarse/top-k
 * kernel, events[2] before the attention kernel and events[3] after it, on
 * the forward's stream. The four cudaEvent_t handles are owned by the caller;
 * pass NULL to stop recording. */
vsa_status_t vsa_plan_set_stage_events(vsa_plan_t plan, void* const* events);

/* Diagnostics: launch `n_ctas` CTAs that each wait on a barrier nothing ever
 * completes, using the same bounded wait as the forward's kernels, with the
 * error words of `workspace` (a workspace of this plan). The first wait gives up
 * after its time limit (2 s) and records VSA_ERR_DEVICE_TIMEOUT; the other CTAs
 * observe the abort flag and return. vsa_check(plan, workspace, stream) then
 * reports VSA_ERR_DEVICE_TIMEOUT. Exercises failure detection without any GPU
 * fault; returns without synchronising. */
vsa_status_t vsa_diag_wait_timeout(vsa_plan_t plan, void* workspace, int n_ctas, void* stream);

/* Size of the library-owned workspace used by vsa_forward_static_workspace:
 * 64 MiB, enough for one GPU's head share of a 5 s request (14 heads, 36,288
 * video tokens: 54 MB) or anything whose workspace_bytes (vsa_plan_info) fits. */
#define VSA_STATIC_WORKSPACE_BYTES (64u * 1024u * 1024u)

/* The forward for callers that cannot allocate device memory (a serving engine
 * that budgets all device memory at start-up, a plugin interface without an
 * allocator, a latency-critical path that must not call cudaMalloc). The
 * paper has no counterpart to this entry point.
 *   q, k, v, gate, out, stream: as for vsa_forward; the caller still owns them.
 * The scratch is a file-scope device array of VSA_STATIC_WORKSPACE_BYTES inside
 * the library; every GPU that loads the library holds it until the process
 * exits. The call allocates nothing (no cudaMalloc, cudaFree or allocating
 * library routine).
 * Returns VSA_ERR_UNSUPPORTED, without launching, if the plan's workspace_bytes
 * exceed VSA_STATIC_WORKSPACE_BYTES.
 * The first call for a plan on a given device resolves the array's device
 * address (cudaGetSymbolAddress, once per device), which may also load the
 * library's device code and back the array on that device; make that first
 * call before any stream capture. The address is kept for the life of the
 * process: do not use this entry point on a device after cudaDeviceReset.
 * All calls share the one array, which keeps the previous call's contents (the
 * forward clears what must start at zero and overwrites the rest): calls whose
 * work overlaps on the GPU (different streams, or host threads, without
 * ordering between them) race on it. Device-side wait timeouts land in the
 * array's error words: vsa_check_static_workspace reports them. */
vsa_status_t vsa_forward_static_workspace(vsa_plan_t plan, const void* q, const void* k,
                                          const void* v, const void* gate, void* out,
                                          void* stream);

/* vsa_check for the library-owned array of vsa_forward_static_workspace:
 * synchronises `stream` and reports the error words the last forward on this
 * plan's device left in that array (VSA_OK, VSA_ERR_DEVICE_TIMEOUT, ...). Like
 * the forward, it allocates nothing; the paper has no counterpart. */
vsa_status_t vsa_check_static_workspace(vsa_plan_t plan, void* stream);

/* vsa_diag_wait_timeout on the library-owned array: lets a test of the
 * static-workspace path exercise its error report without a GPU fault. */
vsa_status_t vsa_diag_wait_timeout_static(vsa_plan_t plan, int n_ctas, void* stream);

void vsa_plan_destroy(vsa_plan_t plan);

const char* vsa_status_string(vsa_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* VSA_H_ */
