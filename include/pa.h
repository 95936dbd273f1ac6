/*
 * pa.h -- C ABI of libpa.so, a PagedAttention forward pass for one GB300 GPU.
 *
 * What the library computes
 * -------------------------
 * PagedAttentionOperation, "Constraints": softmax attention of a batch of
 * query tokens over a KV cache kept as fixed-size blocks. For sequence b,
 * query token i in [0, q_b) and head h in [0, H):
 *
 *   G      = H / Hk                         (GQA: H % Hk == 0)
 *   kvh    = h / G                          (contiguous head groups)
 *   p      = L_b - q_b + i                  (prefix = max(0, L_b - q_b), the
 *                                            mask-alignment rule of the
 *                                            MASK_TYPE_NORM_COMPRESS bullets)
 *   K_b[j] = key_cache  [block_tables[b][j / bs], j % bs, kvh, :]
 *   V_b[j] = value_cache[block_tables[b][j / bs], j % bs, kvh, :]
 *   s_j    = scale * <q[b,i,h,:], K_b[j]> + bias(h, i, j),   j in [0, L_b)
 *   out[b,i,h,:] = sum_j softmax(s)_j * V_b[j]
 *
 * where L_b = context_lens[b] counts the whole KV length including the
 * current query tokens, and bias is
 *   PA_MASK_NONE           0
 *   PA_MASK_ALIBI          alibi_slopes[h] * (j - p)
 *   PA_MASK_NORM_COMPRESS  sigma = max(0, L_b - 2048);
 *                          0 if j < sigma, else mask[p - sigma][j - sigma]
 *                          (the shared 2048 x 2048 causal mask: strict upper
 *                          triangle a large negative fill, diagonal and lower
 *                          triangle 0; the shift keeps both indices inside the
 *                          mask for any L_b, so sequences longer than 2048 need
 *                          nothing extra from the caller).
 *   PA_MASK_NORM           mask[b][i][j], the model's own additive mask
 *                          ("How to select a mask", PA_ENCODER restrictions
 *                          page), given per sequence as fp16
 *                          [batch][max_seqlen_q][max_blocks_per_seq * bs];
 *                          the kernels read the entries with i < q_b and
 *                          j < L_b only.
 * The mask value is added to the scaled score, not substituted by -inf, and is
 * not scaled. The kernels read the compressed mask only above the diagonal
 * (j > p): the pages fix the diagonal and the lower triangle at 0.
 *
 * The split-KV path follows SparseAttnSharedkvMetadata ("功能说明" and the
 * `metadata` output): a task list gives each CTA its (batch, head group, query
 * tile, KV-block range); CTAs that cover part of a sequence's KV write a
 * partial result, and a reduction pass merges the partials by log-sum-exp.
 *
 * Conventions
 * -----------
 * - Every function returns a pa_status; nothing is thrown across the ABI.
 * - pa_plan is pure host code. pa_forward is asynchronous on the caller's
 *   stream, allocates nothing and never synchronises.
 * - Tensors are dense row-major; fp16 is IEEE binary16. "device" pointers are
 *   CUDA global memory of the current device; the caller owns all memory.
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,      /* a constraint of the pages or of this ABI is violated */
  PA_ERR_UNSUPPORTED = 2,      /* a valid mode this build does not implement */
  PA_ERR_BUFFER_TOO_SMALL = 3, /* work/combine capacity or workspace too small */
  PA_ERR_CUDA = 4,             /* a CUDA runtime call or launch failed */
  PA_ERR_BLOCK_INDEX = 5,      /* a device-side block-table entry outside [0, num_blocks) */
  PA_ERR_TIMEOUT = 6           /* a bounded device-side wait ran out */
} pa_status;

/* Mask types. 5 is MASK_TYPE_NORM_COMPRESS as numbered by the pages; the
 * pages name UNDEFINED, NORM and ALIBI without numbers, so 0/1/2 are ours.
 * 4 (a spec-decoding mask whose contents the pages do not describe) returns
 * PA_ERR_UNSUPPORTED. */
typedef enum pa_mask_type {
  PA_MASK_NONE = 0,
  PA_MASK_NORM = 1,
  PA_MASK_ALIBI = 2,
  PA_MASK_SPEC = 4,
  PA_MASK_NORM_COMPRESS = 5
} pa_mask_type;

#define PA_COMPRESS_MASK_SIZE 2048
#define PA_MAX_BATCH 2048
#define PA_MAX_HEAD_SIZE 576
#define PA_FMA_MAX_ROWS 8
#define PA_TC_TILE_ROWS 64
#define PA_PF_TILE_ROWS 128
#define PA_PF_PAIR_ROWS 256
#define PA_STATUS_BYTES 256

/* Status bits written by the kernels into the first word of the workspace. */
#define PA_STATUS_BIT_BLOCK_INDEX 1u
#define PA_STATUS_BIT_TIMEOUT 2u
#define PA_STATUS_BIT_WORKSPACE 4u
#define PA_STATUS_BIT_PLAN 8u /* pa_plan_device: a length breaks a constraint */

/*
 * Problem description shared by pa_plan and pa_forward.
 *
 *   batch               B, 0 < B <= 2048 (PagedAttentionOperation "Constraints")
 *   num_heads           H > 0
 *   kv_heads            Hk > 0, H % Hk == 0 (GQA condition of both pages)
 *   head_size_k/_v      hk, hv in (0, 576] and multiples of 16; a size above
 *                       256 needs block_size <= 128 ("Constraints")
 *   block_size          bs, a multiple of 16; <= 128 when max_seqlen_q > 1
 *                       (parallel decoding)
 *   num_blocks          physical blocks in each cache
 *   max_blocks_per_seq  row length of block_tables, >= ceil(max L_b / bs)
 *   max_seqlen_q        largest q_b (0 is read as 1); the max_seqlen_q
 *                       attribute of SparseAttnSharedkvMetadata
 *   mask_type           a pa_mask_type
 *   chunk_blocks        KV blocks per split, > 0; or 0 for the automatic rule
 *   num_sms             streaming multiprocessors of the target GPU (> 0 when
 *                       chunk_blocks == 0)
 *   scale               QK scale; <= 0 selects 1/sqrt(hk) (SCALE_TYPE_TOR)
 */
typedef struct pa_config {
  int32_t batch;
  int32_t num_heads;
  int32_t kv_heads;
  int32_t head_size_k;
  int32_t head_size_v;
  int32_t block_size;
  int32_t num_blocks;
  int32_t max_blocks_per_seq;
  int32_t max_seqlen_q;
  int32_t mask_type;
  int32_t chunk_blocks;
  int32_t num_sms;
  float scale;
} pa_config;

/*
 * The work list (the `metadata` of SparseAttnSharedkvMetadata, restated).
 *
 * Rows. The query rows of one (b, kvh) pair are R_b = G * q_b rows ordered
 * token-major: row r is query token i = r / G of head h = kvh * G + r % G.
 * A launch uses one tile height TR for every sequence:
 *   TR = G * max_seqlen_q   if that is <= PA_FMA_MAX_ROWS (CUDA-core path)
 *   TR = PA_PF_PAIR_ROWS    if G * max_seqlen_q > PA_PF_TILE_ROWS and
 *                           hk = hv in {64, 128}  (prefill: two query tiles
 *                                                  sharing each K/V tile)
 *   TR = PA_PF_TILE_ROWS    if G * max_seqlen_q > PA_TC_TILE_ROWS and
 *                           hk = hv in {64, 128}       (prefill-shaped tiles)
 *   TR = PA_TC_TILE_ROWS    otherwise                      (tensor-core path)
 * and sequence b has QT_b = ceil(R_b / TR) tiles; tile qt covers rows
 * [qt * TR, min(R_b, (qt + 1) * TR)).
 *
 * Chunk. NB_b = ceil(L_b / bs). With chunk_blocks > 0, c = chunk_blocks.
 * Otherwise
 *   W     = sum_b NB_b * Hk * QT_b
 *   k     = 8 if TR <= PA_FMA_MAX_ROWS, else 2
 *   c_bal = ceil(W / (k * num_sms))
 *   RT    = min(TR, G * max_seqlen_q)   (rows a full tile really holds)
 *   c_min = ceil(64 * RT * hv / (bs * (hk + hv)))
 *   c0    = max(1, c_bal, c_min)
 * and c = c0 when TR <= PA_FMA_MAX_ROWS. For wider tiles (tcgen05 kernels, one
 * CTA per SM, so items run in waves of num_sms) the wave fit follows:
 *   items(x) = sum_b Hk * QT_b * ceil(NB_b / x)
 *   c = the x in [c0, min(2 * c0, c0 + 31, max(c0, max_b NB_b))] with the
 *       least ceil(items(x) / num_sms) * x, the smallest such x on a tie
 * (c_bal aims at about k work items per SM so that variable lengths
 * balance: eight for the CUDA-core and mma.sync kernels, of which several CTAs
 * share an SM, two for the tcgen05 kernel, which holds an SM alone and pays a
 * longer fixed cost per item; c_min keeps the partial results that a split
 * writes and re-reads below about a sixteenth of the KV bytes of the split;
 * the wave fit lengthens the chunk a little when that saves a nearly empty
 * last wave of items, waves x chunk standing for the launch's time.)
 * Sequence b has S_b = ceil(NB_b / c) splits; split s covers KV blocks
 * [s * c, min(NB_b, (s + 1) * c)).
 *
 * Items. One item per (b, kvh, qt, s), in lexicographic order of that tuple
 * (b slowest, s fastest); CTA x of the attention kernel runs item x. Each item
 * is PA_WORK_INTS int32:
 *   [0] b          [1] kvh        [2] row_begin   [3] row_end
 *   [4] kb_begin   [5] kb_end     [6] q_start     [7] slot
 * row_begin/row_end are the tile's row range, q_start = sum_{b' < b} q_b' is
 * the index of the sequence's first query token, and slot is -1 when S_b == 1
 * (the item writes `out` directly) or else the index of the first partial row
 * the item writes. Partial rows are numbered consecutively in item order over
 * the items with S_b > 1, each such item taking row_end - row_begin rows, so
 * the S_b splits of one tile sit at slot_0 + s * (row_end - row_begin).
 *
 * Combine entries. One per (b, kvh, qt) with S_b > 1, in the same order; each
 * is PA_COMBINE_INTS int32:
 *   [0] b   [1] kvh   [2] first_item (index of split 0's item)   [3] S_b
 *
 * Workspace. PA_STATUS_BYTES of status first (word 0 collects PA_STATUS_BIT_*
 * flags), then P * hv fp16 partial outputs (already divided by their softmax
 * sum, so within the range of V), then P fp32 log-sum-exps in natural-log
 * units, where P is the number of partial rows; each part starts on a
 * 256-byte boundary.
 */
#define PA_WORK_INTS 8
#define PA_COMBINE_INTS 4

/*
 * pa_plan -- validate a batch and build its work list (host only).
 *
 * context_lens  host int32 [batch], 1 <= q_b <= L_b.
 * q_seqlens     host int32 [batch], 1 <= q_b <= max(1, max_seqlen_q); NULL
 *               means every q_b = 1. With NORM_COMPRESS q_b <= 2048.
 * work          host int32 [work_cap * PA_WORK_INTS], or NULL to query sizes.
 * combine       host int32 [comb_cap * PA_COMBINE_INTS], or NULL.
 * n_items, n_combine, workspace_bytes   outputs (may be NULL).
 * Returns PA_ERR_BUFFER_TOO_SMALL (after writing the counts) when a non-NULL
 * buffer is too small. Writes nothing else on error.
 */
pa_status pa_plan(const pa_config* cfg, const int32_t* context_lens, const int32_t* q_seqlens,
                  int32_t* work, int64_t work_cap, int64_t* n_items,
                  int32_t* combine, int64_t comb_cap, int64_t* n_combine,
                  size_t* workspace_bytes);

/*
 * pa_forward -- run attention for one planned batch (device, asynchronous).
 *
 * query         device fp16 [sum q_b, H, hk]
 * key_cache     device fp16 [num_blocks, bs, Hk, hk]; 16-byte aligned
 * value_cache   device fp16 [num_blocks, bs, Hk, hv]; 16-byte aligned. Or
 *               exactly key_cache (requires hv <= hk): the shared-KV layout,
 *               one cache whose K row also carries V, V_b[j] being the first
 *               hv dims of K_b[j] (the latent cache of MLA-style models, K of
 *               576 dims and V of 512 in the head-size rule of the
 *               "Constraints" page). Every kernel then fetches each row once
 *               and reads V from the K rows it already holds.
 * block_tables  device int32 [batch, max_blocks_per_seq]
 * context_lens  device int32 [batch]
 * q_seqlens     device int32 [batch], or NULL when every q_b = 1
 * mask          device fp16 [2048, 2048] for NORM_COMPRESS, or
 *               [batch, max_seqlen_q, max_blocks_per_seq * bs] for NORM;
 *               non-NULL exactly for those two types
 * alibi_slopes  device fp32 [H]; non-NULL exactly for ALIBI
 * work/combine  device copies of pa_plan's lists (same cfg, same lengths)
 * workspace     device, >= pa_plan's workspace_bytes, 256-byte aligned; its
 *               status word must be zero before the first call (see
 *               pa_status_clear) and is only ever OR-ed by the kernels
 * out           fp16 [sum q_b, H, hv], 16-byte aligned: device memory, or
 *               pinned host memory mapped into the device's address space
 *               (the kernels then store the result straight into host
 *               memory, with no copy afterwards)
 * stream        a cudaStream_t (NULL = legacy default stream)
 *
 * Host-side errors return before anything is enqueued. Block-table entries
 * outside [0, num_blocks) are never dereferenced: the kernel skips their
 * copies, leaving the affected outputs undefined, and sets
 * PA_STATUS_BIT_BLOCK_INDEX, which pa_status_read reports. Launches: the
 * attention kernel, then, when n_combine > 0, the reduction kernel as its
 * programmatic dependent.
 */
pa_status pa_forward(const pa_config* cfg, const void* query, const void* key_cache,
                     const void* value_cache, const int32_t* block_tables,
                     const int32_t* context_lens, const int32_t* q_seqlens, const void* mask,
                     const float* alibi_slopes, const int32_t* work, int64_t n_items,
                     const int32_t* combine, int64_t n_combine, void* workspace,
                     size_t workspace_bytes, void* out, void* stream);

/*
 * pa_forward_noalloc -- pa_forward without a caller-provided workspace.
 *
 * The reference pages have no counterpart to this call; it exists for callers
 * that cannot allocate device memory: code whose device memory is owned by a
 * pool or an inference runtime that forbids ad-hoc allocations while serving,
 * and latency-critical loops that cannot afford the implicit synchronisation a
 * cudaMalloc/cudaFree may cause. It allocates nothing: the workspace is a fixed
 * device array of PA_NOALLOC_SCRATCH_BYTES inside libpa.so, which every GPU that
 * loads the library holds until the process exits.
 *
 * Arguments are those of pa_forward, except:
 * workspace_bytes  the size pa_plan reported for this batch; more than
 *                  PA_NOALLOC_SCRATCH_BYTES returns PA_ERR_BUFFER_TOO_SMALL
 *                  before anything is enqueued.
 * status           device uint32 or NULL; when non-NULL it receives, on the
 *                  stream, the status word of this call (PA_STATUS_BIT_* flags).
 *
 * The first call on a device, with that device current, looks up the array's
 * device address (cudaGetSymbolAddress) and caches it; make that first call
 * before any stream capture. Each call runs pa_forward's host-side checks
 * first (a rejected call enqueues nothing and leaves `status` unwritten), then
 * zeroes the array's status word on the stream before launching. All calls on a device share the one array, so calls
 * whose work overlaps on the GPU (other streams, other host threads) race.
 * Calls no cudaMalloc, cudaFree or allocating library routine.
 */
#define PA_NOALLOC_SCRATCH_BYTES (32u << 20)
pa_status pa_forward_noalloc(const pa_config* cfg, const void* query, const void* key_cache,
                             const void* value_cache, const int32_t* block_tables,
                             const int32_t* context_lens, const int32_t* q_seqlens,
                             const void* mask, const float* alibi_slopes, const int32_t* work,
                             int64_t n_items, const int32_t* combine, int64_t n_combine,
                             size_t workspace_bytes, uint32_t* status, void* out, void* stream);

/*
 * Planning on the device. The work list depends on the context lengths, which
 * change every decode step; pa_plan needs them on the host. The three calls
 * below keep the whole step on the GPU instead: pa_plan_device builds the
 * same lists as pa_plan (bit for bit, same rule) from device-resident
 * lengths, and pa_forward_device_plan launches grids sized by the list
 * capacities, whose CTAs past the device-side counts return at once. The
 * launches of a step then no longer depend on the lengths, so a caller can
 * record plan + forward once (e.g. as a CUDA graph, the analogue of the
 * graph-launch mode the operator pages mention for their metadata operator)
 * and replay it after updating the lengths in place.
 *
 * pa_plan_bounds (host): capacities that hold the lists of any lengths the
 *   configuration admits, and a workspace size that holds their partial
 *   rows. With tiles T = batch * Hk * ceil(G * max_seqlen_q / TR):
 *   comb_cap = T; work_cap = T * ceil(max_blocks_per_seq / chunk_blocks) for
 *   an explicit chunk, else 8 * num_sms + T (the automatic chunk, the wave
 *   fit included, is at least W / (8 * num_sms)); workspace for
 *   work_cap * TR partial rows. Fails with PA_ERR_INVALID_ARG when the
 *   automatic chunk is asked for with num_sms <= 0, as pa_plan_device does.
 */
pa_status pa_plan_bounds(const pa_config* cfg, int64_t* work_cap, int64_t* comb_cap,
                         size_t* workspace_bytes);

/*
 * pa_plan_device -- pa_plan on the GPU (asynchronous, one small kernel).
 *
 * context_lens, q_seqlens  int32 [batch] the device can read: device memory, or
 *                pinned host memory mapped into its address space;
 *                q_seqlens may be NULL
 * work, combine  device int32 [work_cap * PA_WORK_INTS], [comb_cap * PA_COMBINE_INTS],
 *                16-byte aligned
 * counts         device int32 [PA_PLAN_COUNTS]: items, combine entries,
 *                partial rows, error (0 ok, 1 a length breaks a constraint, 2
 *                a capacity is too small)
 * workspace      the workspace of the forward pass that follows; on an error
 *                the kernel sets PA_STATUS_BIT_PLAN (lengths) or
 *                PA_STATUS_BIT_WORKSPACE (capacity) in its status word and
 *                writes zero counts, so the forward pass does nothing.
 * Host-side checks (configuration, pointers) return before any launch.
 */
#define PA_PLAN_COUNTS 4
pa_status pa_plan_device(const pa_config* cfg, const int32_t* context_lens,
                         const int32_t* q_seqlens, int32_t* work, int64_t work_cap,
                         int32_t* combine, int64_t comb_cap, int32_t* counts, void* workspace,
                         void* stream);

/*
 * pa_forward_device_plan -- pa_forward over the lists of pa_plan_device.
 * Arguments as pa_forward, with the capacities in place of the list lengths
 * and `counts` the planner's device counts. Launches work_cap attention CTAs
 * and comb_cap combine CTAs whatever the counts.
 */
pa_status pa_forward_device_plan(const pa_config* cfg, const void* query, const void* key_cache,
                                 const void* value_cache, const int32_t* block_tables,
                                 const int32_t* context_lens, const int32_t* q_seqlens,
                                 const void* mask, const float* alibi_slopes,
                                 const int32_t* work, int64_t work_cap, const int32_t* combine,
                                 int64_t comb_cap, const int32_t* counts, void* workspace,
                                 size_t workspace_bytes, void* out, void* stream);

/* Zero the status word of a workspace (enqueued on stream). */
pa_status pa_status_clear(void* workspace, void* stream);

/* Wait for stream, read the status word into *bits (may be NULL) and map it to
 * PA_OK, PA_ERR_TIMEOUT, PA_ERR_BLOCK_INDEX, PA_ERR_BUFFER_TOO_SMALL or
 * PA_ERR_INVALID_ARG (PA_STATUS_BIT_PLAN). */
pa_status pa_status_read(const void* workspace, void* stream, uint32_t* bits);

/* Static description of a status code. */
const char* pa_status_string(pa_status s);

#ifdef __cplusplus
}
#endif
#endif /* PA_H */
