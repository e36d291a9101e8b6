/*
 * zl.h — C ABI of the coalesced attention engine (GB300, sm_103a).
 *
 * The engine runs, in one fused launch on one GPU, bidirectional (non-causal) DiT
 * attention over a heterogeneous work list: whole varlen-packed sequences next to
 * distributed-attention shards, each shard cut by its configuration theta=(q,h,k)
 * into a query-row range, a head subset and a KV chunk ("Zellige: Moldable Sequence
 * Placement for Mixed Image-Video DiT Training": newx.sg abstract — the coalesced
 * attention engine executes whole sequences alongside distributed-attention shards;
 * pith.science review, "What carries the argument" — theta splits queries, heads and
 * key/value states, and the engine schedules and fuses whole sequences and shards
 * on shared ranks).  Attention is exact softmax attention (pith.science review,
 * "Assumptions": FlashAttention [7]); k-split shards emit a partial O plus its
 * log-sum-exp, and zl_merge_partials combines them as a ring-attention executor
 * ([19]) would across ranks.
 *
 * Conventions shared by every call
 *  - Q, K, V, dO are bf16 tensors packed as [T, H, d] (token-major, head, then head
 *    dim contiguous; row stride H*d elements).  d is 64 or 128.  Every sequence is a
 *    contiguous run of tokens [seq_offset, seq_offset + seq_len).
 *  - All ranges are half-open and relative to the item's sequence start.
 *  - The CALLER owns every device buffer passed in (inputs, outputs, workspace).  The
 *    library owns a zl_plan: its host copy, its device tile lists, item table and
 *    status word.  fwd / merge / bwd never allocate.
 *  - Device pointers must be 16-byte aligned (ZL_ERR_ALIGN otherwise).
 *  - Every launch is asynchronous on the given stream (a cudaStream_t passed as
 *    void*; NULL = legacy default stream).  A plan keeps one scheduler counter per
 *    kernel, so launches that use the same plan must be ordered (one stream, or
 *    ordered by events).
 *  - No call throws; every call returns a zl_status.  A launch error is ZL_ERR_CUDA
 *    and leaves the CUDA error state for the caller to inspect.
 *  - Plans are bound to the device that was current when zl_plan_worklist ran; a launch
 *    or status query with another device current returns ZL_ERR_INVALID_ARG.
 *
 * Output arenas (element offsets; the planner assigns every offset left at -1)
 *  - o (bf16): one [|q|, |h|, d] block per non-k-split item and per merge group.  An
 *    item (or group) that covers its whole sequence (all rows, all heads) is placed
 *    in place, at element seq_offset*H*d, so whole sequences come out packed exactly
 *    like Q.  Other blocks follow after T*H*d.
 *  - o_partial (fp32): one [|q|, |h|, d] block per k-split (emit_lse=1) item.
 *  - lse (fp32, natural log): one [|h|, |q|] block per item and per merge group; a
 *    whole-sequence block sits at seq_offset*H, other blocks after T*H.
 *  - dq (fp32): one [|q|, |h|, d] block per item; dk, dv (fp32, same layout as each
 *    other): one [|kv|, |h|, d] block per item.  Whole items sit in place at
 *    seq_offset*H*d.  Each item writes only its own blocks, so overlapping shards
 *    never race; a q-split item's dK/dV and a k-split item's dQ are that shard's
 *    partial contributions (a distributed run would reduce them across ranks).
 */
#ifndef ZL_H
#define ZL_H

#include <stdint.h>

#if defined(__GNUC__)
#define ZL_API __attribute__((visibility("default")))
#else
#define ZL_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ZL_OK = 0,
  ZL_ERR_INVALID_ARG = 1,  /* bad descriptor, size or null pointer                     */
  ZL_ERR_ALIGN = 2,        /* pointer or offset breaks the 16-byte rule               */
  ZL_ERR_CUDA = 3,         /* a CUDA runtime/driver call or kernel launch failed      */
  ZL_ERR_TIMEOUT = 4,      /* a bounded device-side wait gave up (see status word)    */
  ZL_ERR_UNSUPPORTED = 5,  /* e.g. head_dim not in {64,128}, device is not sm_103     */
  ZL_ERR_NO_MEMORY = 6     /* plan allocation failed                                  */
} zl_status;

/* One work-list entry: a whole sequence or a theta=(q,h,k) shard of one sequence.
 * emit_lse = 1 marks a k-split shard: it writes an fp32 partial O (normalised by its
 * own chunk's softmax sum) plus its LSE, to be merged.  emit_lse items with the same
 * (seq_offset, seq_len, q range, h range) form one merge group, in list order.
 * out_offset: element offset of the item's O block in `o` (emit_lse = 0) or in
 * `o_partial` (emit_lse = 1); -1 = planner assigns.  Must be a multiple of 8.
 * lse_offset: element offset of the item's LSE block in `lse`; -1 = planner assigns. */
typedef struct {
  int64_t seq_offset;
  int32_t seq_len;
  int32_t q_lo, q_hi;
  int32_t h_lo, h_hi;
  int32_t kv_lo, kv_hi;
  int32_t emit_lse;
  int64_t out_offset;
  int64_t lse_offset;
} zl_work_item;

typedef struct zl_plan zl_plan;

/* Flag for zl_plan_worklist: build the host tables only (no device upload).  Such a
 * plan answers the zl_plan_* queries but cannot be launched. */
#define ZL_PLAN_HOST_ONLY 1u
/* Test flag (failure detection): the forward launch announces its first K tile (the
 * backward launch its first K/V tile) but never issues the copy, so a bounded device
 * wait runs out (after ~20M cycles) and zl_get_device_status reports ZL_ERR_TIMEOUT;
 * nothing faults or hangs. */
#define ZL_PLAN_TEST_WITHHOLD_LOAD 2u
/* (Flag value 4 is not used; zl_plan_worklist rejects flags it does not know.) */
/* Fused local k-merge.  A merge group (emit_lse items sharing sequence, rows and heads)
 * whose KV chunks tile one contiguous range is computed by the forward launch as a
 * single item over that range: its final O (bf16) and LSE go straight into the group's
 * blocks, which is the merge's result up to rounding (softmax over the union of the
 * chunks equals the LSE-weighted combine of the chunks; "Zellige", pith.science review,
 * "What carries the argument", k split of theta).  The members' own partial O and LSE
 * blocks are then neither allocated nor written (their resolved out_offset and
 * lse_offset are -1; offsets given in the work list are ignored), and
 * zl_merge_partials skips the group.  Groups with a gap between chunks are merged as
 * usual.  The backward is unchanged: each member keeps its gradient ownership and reads
 * the group's final O and LSE. */
#define ZL_PLAN_FUSE_LOCAL_KMERGE 8u
/* Deterministic dQ.  By default the backward's CTAs add their dQ contributions into the
 * fp32 accumulator in whatever order they reach a query block, so dQ may differ in its
 * last bits from run to run (dK, dV, O and LSE never do).  With this flag every
 * accumulator element receives its contributions in a fixed order, KV tile 0, 1, 2, ...
 * of its item and head, so dQ is bitwise reproducible for the same plan and inputs.
 * How: each drain warp of a KV tile waits (bounded) until a per-(query block, warp)
 * turn counter equals the tile's KV-block index, adds its rows, and passes the turn on
 * (index + 1) when it moves to its next block.
 * The backward tiles of each cost are listed block-major (KV block, then work-list
 * order), so the tiles of one item and head are claimed in ascending KV order and far
 * apart: a tile waits only on tiles claimed before it, held by running CTAs, and
 * rarely at all.  The workspace grows by one int32 per (128-row query block, 32-row
 * warp slice) of the accumulator, zeroed with it by zl_bwd_preprocess. */
#define ZL_PLAN_DETERMINISTIC_DQ 16u

/* Validate a work list and build its tile lists (host C++), then upload them to the
 * current device.
 * Passage: pith.science review, "What carries the argument" (theta=(q,h,k) cuts a
 * sequence into query-row, head and KV shards; the engine schedules whole sequences and
 * shards that share a rank in a fixed order and fuses them into shared launches).
 *   items[n_items]: descriptors (host memory, read only; not retained).
 *   n_heads H >= 1, head_dim d in {64, 128}, total_tokens T >= 1 (Q/K/V have T rows).
 * Tiles: forward = (item, head, 256 query rows, run as two 128-row sub-tiles);
 * backward = (item, head, 128 KV rows).
 * Each list is sorted longest-first (cost = KV blocks for forward, query blocks for
 * backward), ties in work-list order, and a persistent grid of one CTA per SM claims
 * tiles in that order from an atomic counter.
 * Errors: ZL_ERR_INVALID_ARG for a range outside its sequence, lo > hi, a head range
 * outside [0,H), a sequence outside [0,T), a negative offset other than -1, or a merge
 * group whose KV chunks overlap; ZL_ERR_ALIGN for out_offset not a multiple of 8;
 * ZL_ERR_UNSUPPORTED for d not in {64,128}; ZL_ERR_NO_MEMORY / ZL_ERR_CUDA on
 * allocation or copy failure.  On error *out is set to NULL. */
ZL_API zl_status zl_plan_worklist(const zl_work_item* items, int32_t n_items, int32_t n_heads,
                           int32_t head_dim, int64_t total_tokens, uint32_t flags,
                           zl_plan** out);

/* Passage: as zl_plan_worklist and zl_merge_partials.  zl_plan_worklist with the merge
 * groups chosen by the caller instead of formed from equal (sequence, q range, h range)
 * keys in list order.  Group g holds the emit_lse items
 * group_item_ids[group_ptr[g] .. group_ptr[g+1]) (host arrays; group_ptr has n_groups + 1
 * entries, group_ptr[0] = 0), merged in that member order.  Every emit_lse item must be
 * in exactly one group; the members of a group must share sequence, q range and h range,
 * and their KV chunks must be disjoint.  A group is one exact attention problem over the
 * union of its members' chunks: its merged O and LSE are the final outputs its members'
 * backward reads, so two groups over the same rows and heads are two separate problems
 * (e.g. two KV subsets of one sequence).  The groups are fixed here rather than given to
 * zl_merge_partials because the plan places each group's output block and the backward of
 * every member reads it.  Errors: as zl_plan_worklist, and ZL_ERR_INVALID_ARG for a
 * malformed group_ptr, an item id out of range, a member without emit_lse, an emit_lse
 * item in no group or in two, or members with different keys. */
ZL_API zl_status zl_plan_worklist_groups(const zl_work_item* items, int32_t n_items, int32_t n_heads,
                                         int32_t head_dim, int64_t total_tokens, uint32_t flags,
                                         const int32_t* group_item_ids, const int32_t* group_ptr,
                                         int32_t n_groups, zl_plan** out);

/* Free a plan (host and device parts).  (Library mechanics; no passage.)  NULL is ignored.  Must not be called while a
 * launch that uses the plan is still running. */
ZL_API void zl_plan_destroy(zl_plan* plan);

/* Element counts of every arena the caller must allocate for this plan (any pointer
 * may be NULL).  Passage: as zl_plan_worklist (every item and shard owns its blocks).  workspace_bytes: scratch for zl_coalesced_attn_bwd (row sums D, the
 * fp32 dQ accumulator and, with ZL_PLAN_DETERMINISTIC_DQ, its turn counters). */
ZL_API zl_status zl_plan_arena_sizes(const zl_plan* plan, int64_t* o_elems, int64_t* o_partial_elems,
                              int64_t* lse_elems, int64_t* dq_elems, int64_t* dkv_elems,
                              int64_t* workspace_bytes);

/* Passage: as zl_plan_worklist.  Resolved placement of item i: its descriptor with offsets filled in, plus
 * fin_out_offset / fin_lse_offset (where its FINAL O, dO and LSE live in `o` / `lse`:
 * its own block, or its merge group's block for an emit_lse item), dq_offset and
 * dkv_offset (its gradient blocks), and group (merge group index or -1). */
ZL_API zl_status zl_plan_item(const zl_plan* plan, int32_t i, zl_work_item* resolved,
                       int64_t* fin_out_offset, int64_t* fin_lse_offset, int64_t* dq_offset,
                       int64_t* dkv_offset, int32_t* group);

/* (Library mechanics, standing in for a device-side bounds checker; no passage.)
 * Host-side dry run of the plan: every block and workspace range that a launch with
 * this plan would touch lies inside the arena sizes of zl_plan_arena_sizes, and every
 * tile addresses an existing item, head and block.  ZL_OK or ZL_ERR_INVALID_ARG.  Works
 * on host-only plans (no GPU needed). */
ZL_API zl_status zl_plan_check_bounds(const zl_plan* plan);

/* Passage: as zl_plan_worklist.  Counts: which = 0 forward tiles, 1 backward tiles, 2 merge groups, 3 items (of the
 * work list), 4 merge groups that zl_merge_partials combines (2 minus those fused into
 * the forward by ZL_PLAN_FUSE_LOCAL_KMERGE). */
ZL_API zl_status zl_plan_count(const zl_plan* plan, int32_t which, int64_t* count);

/* Passage: as zl_plan_worklist (the fixed order in which shared launches take the work).
 * Copy a tile list to host memory as n x 4 int32 {item, head, block, cost}, in the
 * order the scheduler hands tiles out.  which = 0 forward, 1 backward. */
ZL_API zl_status zl_plan_tiles(const zl_plan* plan, int32_t which, int32_t* out, int64_t n);

/* Passage: as zl_merge_partials.  Merge group g: member item ids (up to cap written), member count, and the group's
 * final O / LSE offsets in `o` / `lse`. */
ZL_API zl_status zl_plan_group(const zl_plan* plan, int32_t g, int32_t* members, int32_t cap,
                        int32_t* n_members, int64_t* out_offset, int64_t* lse_offset);

/* Passage: newx.sg page, Abstract (the coalesced attention engine runs whole sequences
 * alongside distributed-attention shards); pith.science review, "What carries the
 * argument" (whole sequences and shards fused on a shared rank) and "Assumptions & free
 * parameters" (exact attention, FlashAttention [7]).
 * Forward: one persistent launch over every forward tile of the plan (sm_103a:
 * TMA-staged Q/K/V tiles, tcgen05 MMA with TMEM accumulators for S = Q K^T and
 * O += P V, online softmax with base-2 exponent, LSE epilogue).
 *   q, k, v: bf16 [T, H, d] device pointers (read only).
 *   o: bf16 arena (see above) for emit_lse = 0 items; may be NULL if there are none.
 *   o_partial: fp32 arena for emit_lse = 1 items; may be NULL if there are none.
 *   lse: fp32 arena; every item writes its LSE block (partial LSE for emit_lse items).
 *   scale: softmax scale applied to Q K^T (1/sqrt(d) for DiT attention).
 * Items with an empty KV range write O = 0 and LSE = -inf.
 * Tokens that belong to no item (gaps, padding) and other items' tokens may hold any
 * values, NaN and Inf included: the last, partial 128-row tile of an item reads the
 * tokens that follow it, but their scores are masked, their output rows are never
 * stored, and the value rows past the item's KV range are zeroed in shared memory before
 * the P V product reads them (a zero weight times NaN would still be NaN). */
ZL_API zl_status zl_coalesced_attn_fwd(const zl_plan* plan, const void* q, const void* k,
                                const void* v, void* o, float* o_partial, float* lse,
                                float scale, void* stream);

/* Passage: pith.science review, "What carries the argument" (the k of theta splits the
 * key/value states) and its ref. [19], ring attention, which combines per-chunk partial
 * outputs by their log-sum-exp weights; the pages do not print the combine.
 * Merge every k-split group of the plan: with M = max_c LSE_c,
 * LSE = M + ln sum_c exp(LSE_c - M) and O = sum_c exp(LSE_c - LSE) O_c.
 * Reads o_partial and the members' LSE blocks from lse_partial; writes the group's bf16
 * O block into o and its LSE block into lse_out (lse_out may equal lse_partial: the
 * planner keeps member and group blocks disjoint).  A row whose chunks are all empty
 * gets O = 0, LSE = -inf.  HBM-bound, one warp per (row, head). */
ZL_API zl_status zl_merge_partials(const zl_plan* plan, const float* o_partial,
                            const float* lse_partial, void* o, float* lse_out, void* stream);

/* Passage: newx.sg page, Abstract (DiT training on image and video data: the engine runs
 * the training step's attention, so its gradient too); pith.science review, "What carries
 * the argument" (theta shards; a shard's gradients are its own block's contribution).
 * Backward of every item, using each item's FINAL output and LSE (for k-split items,
 * the merged group's O and global LSE):
 *   D_i = rowsum(dO_i * O_i);  P_ij = exp(s_ij - LSE_i);  dS_ij = P_ij (dO_i.V_j - D_i);
 *   dV_j = sum_i P_ij dO_i;  dK_j = scale sum_i dS_ij Q_i;  dQ_i = scale sum_j dS_ij K_j,
 * every sum over the item's own rows x KV chunk.
 *   q, k, v: as for the forward.  o, d_o: bf16, `o`-arena layout (final outputs and
 *   their gradients).  lse: fp32 `lse` arena holding the final LSE blocks.
 *   dq, dk, dv: fp32 gradient arenas (written, not accumulated).
 *   workspace: device scratch of zl_plan_arena_sizes' workspace_bytes (16-byte aligned).
 * Launches: row sums D + zeroing of the dQ accumulator; the persistent tcgen05
 * backward over (item, head, 128 KV rows) tiles; the dQ finalisation (scale).
 * As for the forward, tokens outside an item may hold any values: the rows of K, V and Q
 * past an item's KV or query range in a partial tile are zeroed in shared memory before
 * any product reads them, and dO is read through per-item maps that end at the item. */
ZL_API zl_status zl_coalesced_attn_bwd(const zl_plan* plan, const void* q, const void* k,
                                const void* v, const void* o, const void* d_o,
                                const float* lse, float* dq, float* dk, float* dv,
                                void* workspace, float scale, void* stream);

/* Passage: as zl_coalesced_attn_bwd.
 * The three launches of zl_coalesced_attn_bwd, callable one by one (same arguments,
 * same order of use); zl_coalesced_attn_bwd is exactly these three in sequence.
 *   zl_bwd_preprocess: D_i = rowsum(dO_i * O_i) into the workspace and zeroing of the
 *     workspace's fp32 dQ accumulator (and turn counters) (HBM-bound, one warp per
 *     (row, head)).
 *   zl_bwd_main: the persistent tcgen05 backward over (item, head, 128 KV rows) tiles;
 *     writes dk, dv and accumulates unscaled dQ in the workspace.
 *   zl_bwd_finalize: dq = scale * accumulator, per item block. */
ZL_API zl_status zl_bwd_preprocess(const zl_plan* plan, const void* o, const void* d_o, void* workspace,
                                   void* stream);
ZL_API zl_status zl_bwd_main(const zl_plan* plan, const void* q, const void* k, const void* v,
                             const void* d_o, const float* lse, float* dk, float* dv, void* workspace,
                             float scale, void* stream);
ZL_API zl_status zl_bwd_finalize(const zl_plan* plan, float* dq, void* workspace, float scale,
                                 void* stream);

/* Forward launch that allocates no device memory (no counterpart in the paper; it
 * serves callers that cannot call cudaMalloc, e.g. code whose host framework owns all
 * device memory through its own pool, or an embedding that forbids device allocation
 * after start-up, and so cannot create a zl_plan, which uploads its tables to memory
 * the library allocates).
 *   Arguments: the work list and sizes as for zl_plan_worklist, then the buffers and
 *   scale as for zl_coalesced_attn_fwd.  Output placement is exactly the planner's
 *   default, so outputs land where a plan built from the same list would put them (ask
 *   a host-only plan, ZL_PLAN_HOST_ONLY, for the offsets and arena sizes).
 *   Scratch: the item table, tile list, scheduler counter and status word live in a
 *   fixed 8 MiB array compiled into the library; every GPU that loads the library holds
 *   it until the process exits.  Capacity: 112 bytes per work item plus 16 bytes per
 *   forward tile (256 query rows of one head), each table rounded up to 256 bytes,
 *   within 8 MiB - 256 bytes: about 65 000 items of one tile each, or about 520 000
 *   tiles over a few items.  A larger list is rejected with ZL_ERR_INVALID_ARG before
 *   any device work.
 *   The first call on a device (of this or of zl_noalloc_get_device_status) looks up that
 *   array's device address (once per device, with the device current); make that first
 *   call before any stream capture.
 *   Every call shares the array and zeroes the counter and status word itself, so calls
 *   whose launches overlap on the GPU (different streams, different threads) race on
 *   it: order them.  A bounded device wait that gives up is recorded in the array's
 *   status word: read it with zl_noalloc_get_device_status after the call and before the
 *   next one (the next call clears it).
 *   Calls no cudaMalloc/cudaFree or other allocating routine. */
ZL_API zl_status zl_coalesced_attn_fwd_noalloc(const zl_work_item* items, int32_t n_items, int32_t n_heads,
                                               int32_t head_dim, int64_t total_tokens, const void* q,
                                               const void* k, const void* v, void* o, float* o_partial,
                                               float* lse, float scale, void* stream);

/* Status word of zl_coalesced_attn_fwd_noalloc on the current device (no counterpart in
 * the paper): synchronises `stream`, stores in *device_status ZL_OK or the first error
 * the last call's kernel recorded (ZL_ERR_TIMEOUT when a bounded wait gave up; the kernel
 * then stopped cleanly instead of hanging, and its outputs are incomplete), and clears
 * the word.  Allocates nothing.  ZL_ERR_INVALID_ARG for a NULL device_status. */
ZL_API zl_status zl_noalloc_get_device_status(void* stream, int32_t* device_status);

/* (Library mechanics: failure detection by bounded device waits; no passage.)
 * Read and clear the plan's device status word (synchronises `stream`).  *device_status
 * receives ZL_OK or the first error a kernel recorded (ZL_ERR_TIMEOUT when a bounded
 * wait gave up; the kernel then stopped cleanly instead of hanging). */
ZL_API zl_status zl_get_device_status(const zl_plan* plan, void* stream, int32_t* device_status);

/* Static text for a status code.  (Library mechanics; no passage.) */
ZL_API const char* zl_status_string(zl_status status);

/* Library version, e.g. 100 for 0.1.0.  (Library mechanics; no passage.) */
ZL_API int32_t zl_version(void);

/* ------------------------------------------------------------------------------------
 * Host placement slice (no GPU): the catalog cut and the filler packing of the
 * two-stage planner ("Zellige", pith.science review, "Free parameters" and the referee
 * report on Eq. (8): the cut is the Fisher grouping under which the log run times of
 * whole sequences vary least inside each set; a filler goes to the rank whose tighter
 * resource, compute headroom against F or memory headroom against M_cap, stays the
 * most open).  The anchors' own placement (an exact CP-SAT model in
 * the pages) is not part of this library: the packing takes the anchors' per-rank time
 * and memory as given.
 * ---------------------------------------------------------------------------------- */

/* One bucket of a sequence catalog: sequences of one length, how many there are in the
 * batch, and the time and memory of one such sequence run whole on one rank. */
typedef struct {
  int64_t seq_len;
  int32_t count;  /* >= 1 */
  double time;    /* > 0, finite */
  double mem;     /* >= 0 */
} zl_bucket;

/* Passage: pith.science review, "Assumptions & free parameters" (catalog cut k*, Eq. 4:
 * the split that minimises the within-set dispersion of log whole-sequence times).
 * Catalog cut.  buckets[n_buckets] sorted by time ascending (host memory, read only).
 * With x_b = ln time_b and the count-weighted means mu_F, mu_A of x over buckets
 * [0, k) and [k, n), the cut k in 1..n-1 minimises
 *   D(k) = sum_{b<k} count_b (x_b - mu_F)^2 + sum_{b>=k} count_b (x_b - mu_A)^2;
 * *k_star = that k (smallest on ties): buckets [0, k*) are fillers, [k*, n) anchors.
 * A single bucket gives k* = 1 (all fillers), D = 0.  *dispersion (may be NULL)
 * receives D(k*).  ZL_ERR_INVALID_ARG for n < 1, a count < 1, a time not positive and
 * finite, or buckets out of order. */
ZL_API zl_status zl_catalog_cut(const zl_bucket* buckets, int32_t n_buckets, int32_t* k_star, double* dispersion);

/* Passage: pith.science review, "What carries the argument" (whole filler sequences
 * packed greedily by a bottleneck score) and its referee report on Eq. (8).
 * Filler packing.  Places fillers s = 0..n_fillers-1 (time filler_time[s], memory
 * filler_mem[s]; host arrays) whole on n_ranks ranks that already carry rank_time[r],
 * rank_mem[r] (the anchors' load; NULL = zeros).  Fillers go in decreasing time (ties:
 * lower index first), each to the rank with the largest bottleneck score
 *   min((F - L_r - t) / F, (M_cap - M_r - m) / M_cap)     (ties: lowest rank)
 * with L_r, M_r the rank's time and memory so far.  A filler whose best score is below
 * -1e-9 (negative beyond the rounding of an exact fit) is placed all the same and
 * counted in *n_overflow.  F <= 0 selects
 * max(max_r rank_time[r], (sum_r rank_time[r] + sum_s filler_time[s]) / n_ranks).
 * Outputs (host): assign[n_fillers] the rank of each filler; final_time[n_ranks] and
 * final_mem[n_ranks] (may be NULL); *n_overflow, *makespan = max_r final time (may be
 * NULL).  ZL_ERR_INVALID_ARG for n_ranks < 1, M_cap not positive and finite, F not
 * finite, or a negative or non-finite time or memory. */
ZL_API zl_status zl_pack_fillers(const double* filler_time, const double* filler_mem, int32_t n_fillers,
                                 int32_t n_ranks, const double* rank_time, const double* rank_mem, double F,
                                 double M_cap, int32_t* assign, double* final_time, double* final_mem,
                                 int32_t* n_overflow, double* makespan);

#ifdef __cplusplus
}
#endif

#endif /* ZL_H */
