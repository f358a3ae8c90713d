/*
 * ep.h - C ABI of the GB300 (sm_103a) MoE expert-parallel dispatch/combine
 * library (libep_gb300.so).
 *
 * The hot path has four steps, each one entry point below:
 *   ep_get_dispatch_layout  count tokens per rank / node / expert and build
 *                           is_token_in_rank from the router's top-k map
 *   ep_notify_dispatch      prefix sums: rank and channel prefix matrices,
 *                           receive counts and offsets, and the row map
 *   ep_dispatch             copy every token row (and its top-k ids, weights
 *                           and source info) into each destination's region
 *   ep_combine              gather the rows back and sum them in fp32
 *
 * Pages the operations come from (cited by title and section):
 *   [IN] "notify_dispatch (internode.cu)" notes on DeepEP: sm0 stages 3-6 and
 *        sm1..x stages 1-3.
 *   [CH] "cuda】deepep": channels as a partition of each rank's tokens.
 *   [RT] mscclpp src/ext/ep/ht_runtime.cc: MoEHighThroughputRuntime::
 *        getDispatchLayout, intranode/internodeNotifyDispatch,
 *        intranode/internodeDispatch, intranode/internodeCombine.
 *   [AR] "CUDA与DeepEP：分布式MoE系统中的高效通信机制解析": 2.2 rank-to-node
 *        mapping, 3.2 reductions and prefix sums, 4.1 SrcInfo, 4.2 combine.
 *
 * Model.  R "ranks" are logical partitions of ONE GPU's memory.  Every
 * rank-indexed array is stacked along a leading rank axis on the same device
 * (x is [R][T][H], topk_idx is [R][T][K], ...).  Sending to rank r is a store
 * into r's region of one receive pool; nothing crosses a GPU boundary.
 *
 * Notation: R ranks, N = max(1, R/8) nodes (node of rank r is r/8, [AR] 2.2),
 * T tokens per rank, K top-k slots, E experts, E_loc = E/R experts per rank,
 * H hidden size in bf16 elements, C channels.  Channel c of a rank holds its
 * tokens [min(c*q, T), min((c+1)*q, T)) with q = ceil(T/C) ([CH]).
 *
 * Conventions for every call:
 *   - All array arguments are DEVICE pointers (cudaMalloc / torch memory)
 *     unless marked "host".  Arrays are dense, C-order, 16-byte aligned.
 *   - The caller owns and allocates every buffer.  Apart from
 *     ep_sync_status's 4-byte read-back, no call allocates, frees or keeps
 *     state between calls.
 *   - Calls are asynchronous on `stream` (0 = legacy default stream) and
 *     return after enqueueing.  The host checks arguments first and returns
 *     EP_ERR_INVALID_ARG without enqueueing anything when they are wrong.
 *   - Errors found on the device (receive capacity exceeded, a wait that ran
 *     out, inputs that disagree) are OR-ed as EP_DEV_* bits into the
 *     caller's `status` word; the kernels never trap.  ep_sync_status turns
 *     the word into an ep_status_t.  Zero the word before the first call.
 *   - Outputs are a pure function of the inputs: re-running a call gives
 *     byte-identical results (no atomics decide any output value).
 */
#ifndef EP_GB300_H
#define EP_GB300_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    EP_OK = 0,
    EP_ERR_INVALID_ARG = -1,   /* a size, pointer or alignment rule is broken */
    EP_ERR_CUDA = -2,          /* a CUDA runtime call failed */
    EP_ERR_CAPACITY = -3,      /* receive pool smaller than the rows to place */
    EP_ERR_TIMEOUT = -4,       /* a bounded device wait ran out */
    EP_ERR_INCONSISTENT = -5,  /* count inputs disagree with is_token_in_rank */
    EP_ERR_INPUT = -6          /* an expert id outside [-1, E) */
} ep_status_t;

/* Bits the kernels OR into the device status word. */
#define EP_DEV_CAPACITY 0x1
#define EP_DEV_TIMEOUT 0x2
#define EP_DEV_INCONSISTENT 0x4
#define EP_DEV_INPUT 0x8

/* Problem shape.  Rules (EP_ERR_INVALID_ARG otherwise):
 *   1 <= R <= 32, and R % 8 == 0 when R > 8 (whole nodes of 8 ranks);
 *   T >= 0, R * T < 2^30;  1 <= K <= 32;  E >= R and E % R == 0, E <= 8192;
 *   H >= 8 and H % 8 == 0 (rows are whole 16-byte vectors, [RT] asserts
 *   (hidden * elem) % sizeof(int4) == 0);  1 <= C <= 4096;
 *   expert_alignment >= 1. */
typedef struct {
    int32_t num_ranks;        /* R */
    int32_t num_tokens;       /* T, tokens per source rank */
    int32_t num_topk;         /* K */
    int32_t num_experts;      /* E */
    int32_t hidden;           /* H, bf16 elements per token row */
    int32_t num_channels;     /* C */
    int32_t expert_alignment; /* per-expert receive counts round up to this */
} ep_shape_t;

/* Human-readable name of a status code.  Never NULL. */
const char* ep_status_string(ep_status_t status);

/* EP_OK when `shape` obeys the rules above, else EP_ERR_INVALID_ARG. */
ep_status_t ep_check_shape(const ep_shape_t* shape);

/* Number of nodes N = max(1, R/8), or -1 for an invalid shape. */
int32_t ep_num_nodes(const ep_shape_t* shape);

/* Bytes of device scratch ep_notify_dispatch needs (its `workspace`), or 0
 * for an invalid shape.  The workspace must be zero before its first use. */
size_t ep_notify_workspace_bytes(const ep_shape_t* shape);

/* ------------------------------------------------------------------------
 * Step 1 - layout.  [RT] getDispatchLayout; the three count vectors are the
 * ones [IN] sm0 stage 3 packs for each destination node.
 *
 *   topk_idx                 in   int64 [R][T][K]  expert id in [0,E), or -1
 *                                                   for an empty slot
 *   num_tokens_per_rank      out  int32 [R][R]     [s][r]: tokens of s with
 *                                                   at least one expert on r
 *   num_tokens_per_rdma_rank out  int32 [R][N]     [s][n]: tokens of s with
 *                                                   an expert on node n
 *   num_tokens_per_expert    out  int32 [R][E]     [s][e]: slots of s naming
 *                                                   e (a repeated id counts
 *                                                   every time)
 *   is_token_in_rank         out  uint8 [R][T][R]  1 when token (s,t) has an
 *                                                   expert on rank r, else 0
 *   status                   in/out int32 device status word
 * Expert e lives on rank e / E_loc.  An id outside [-1, E) sets EP_DEV_INPUT
 * and is ignored.  Every output element is written (no pre-zeroing needed).
 */
ep_status_t ep_get_dispatch_layout(const ep_shape_t* shape, const int64_t* topk_idx,
                                   int32_t* num_tokens_per_rank,
                                   int32_t* num_tokens_per_rdma_rank,
                                   int32_t* num_tokens_per_expert,
                                   uint8_t* is_token_in_rank, int32_t* status,
                                   cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Step 2 - notify.  [IN] sm1..x stages 1-3 (per-channel counts and their
 * prefix) and sm0 stage 6 (per-rank prefix over global source rank, node
 * prefix, per-expert totals rounded up to expert_alignment); [RT]
 * intranodeNotifyDispatch / internodeNotifyDispatch for the outputs' names
 * and shapes.  One kernel: per (source rank, channel) block a count and the
 * prefix over the earlier channels of the same source rank (recounted
 * directly for small sources, a decoupled-lookback scan otherwise); the
 * offset contributed by earlier source ranks comes from the per-rank counts,
 * as in the pages' notify.
 *
 * Inputs (as produced by step 1):
 *   is_token_in_rank           uint8 [R][T][R]
 *   num_tokens_per_rank        int32 [R][R]
 *   num_tokens_per_rdma_rank   int32 [R][N]
 *   num_tokens_per_expert      int32 [R][E]
 * Outputs:
 *   rank_prefix_matrix         int32 [R src][R dst]  sum over s' <= s of
 *                                                     num_tokens_per_rank[s'][r]
 *   gbl_channel_prefix_matrix  int32 [R src][R dst][C] tokens of s in
 *                                                     channels <= c sent to r
 *   rdma_channel_prefix_matrix int32 [R src][N][C]   same, per node
 *   recv_gbl_rank_prefix_sum   int32 [R dst][R src]  transpose of
 *                                                     rank_prefix_matrix
 *   recv_rdma_rank_prefix_sum  int32 [R dst][N]      [r][m]: sum over m' <= m
 *                                                     of what rank m'*8 + r%8
 *                                                     sends to node r/8
 *   recv_channel_offset        int32 [R dst][R src][C] first row of block
 *                                                     (s,c) in r's region
 *   num_recv_tokens            int32 [R]             rows rank r receives
 *   num_rdma_recv_tokens       int32 [R]             last column of
 *                                                     recv_rdma_rank_prefix_sum
 *   num_recv_tokens_per_expert int32 [R][E_loc]      per local expert,
 *                                                     rounded up to alignment
 *   recv_base                  int64 [R+1]           region of rank r starts at
 *                                                     pool row recv_base[r];
 *                                                     recv_base[R] = total rows
 *   send_pos                   int32 [R src][T][R dst] row of (s,t) inside r's
 *                                                     region, or -1
 *   workspace                  device scratch of ep_notify_workspace_bytes()
 *                              bytes, zero-filled once before its first use
 *                              (e.g. one cudaMemset); every call leaves it
 *                              ready for the next, so it is never cleared
 *                              again.  One workspace may serve calls of any
 *                              shape in turn, but not two calls at once.
 *   host_num_recv_tokens       optional (may be NULL): int32 [R+1] in
 *                              host-mapped pinned memory (cudaHostAlloc with
 *                              cudaHostAllocMapped, or any device-visible
 *                              pointer); receives num_recv_tokens and the
 *                              total, so the host can size its buffers after a
 *                              stream sync without another copy
 * Rows of r's region are ordered by (source rank, channel, token), which is
 * (source rank, token) order.  If the count inputs disagree with
 * is_token_in_rank, EP_DEV_INCONSISTENT is set and the outputs are
 * unspecified (dispatch and combine still never touch memory outside their
 * buffers).  A bounded wait that runs out sets EP_DEV_TIMEOUT.
 */
ep_status_t ep_notify_dispatch(const ep_shape_t* shape, const uint8_t* is_token_in_rank,
                               const int32_t* num_tokens_per_rank,
                               const int32_t* num_tokens_per_rdma_rank,
                               const int32_t* num_tokens_per_expert,
                               int32_t* rank_prefix_matrix, int32_t* gbl_channel_prefix_matrix,
                               int32_t* rdma_channel_prefix_matrix,
                               int32_t* recv_gbl_rank_prefix_sum,
                               int32_t* recv_rdma_rank_prefix_sum, int32_t* recv_channel_offset,
                               int32_t* num_recv_tokens, int32_t* num_rdma_recv_tokens,
                               int32_t* num_recv_tokens_per_expert, int64_t* recv_base,
                               int32_t* send_pos, void* workspace, size_t workspace_bytes,
                               int32_t* status, int32_t* host_num_recv_tokens,
                               cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Steps 1 and 2 in one call: ep_get_dispatch_layout followed by
 * ep_notify_dispatch on its outputs ([RT] getDispatchLayout then
 * intranode/internodeNotifyDispatch; [IN] sm0 stages 3 and 6, sm1..x stages
 * 1-3).  Every output of both calls is written, with the same values.  Always
 * one kernel, in one of two forms (ep_layout_notify_fused tells which):
 *
 *   cluster form (R <= 16, T <= 1024, R*T <= 8192, and a thread-block
 *   cluster of R CTAs fits on the device): CTA s counts source rank s's tokens and keeps one
 *   ballot word per 32 tokens and destination in shared memory; the counts
 *   are exchanged through distributed shared memory and one cluster barrier,
 *   so no workspace traffic and no second pass over is_token_in_rank.
 *
 *   tiled form (every other shape): CTAs work on tiles of tokens of one
 *   source rank, numbered in (source rank, tile) order - a CTA's first tile
 *   is its block index, later ones come from a ticket ([CH] channels are
 *   tiles of the same kind); per-rank counts pass through a single-pass
 *   scan ([AR] 3.2) - decoupled lookback within each source, per-source
 *   totals in self-counting 64-bit words - whose exclusive prefix is
 *   directly each tile's first row in every destination's region; the
 *   per-source results come from each source's last tile, the per-expert
 *   counts from the add that completes each counter word, the per-rank
 *   results from the last tile.  A tile waits only for tiles with smaller
 *   numbers, every wait is bounded.
 *
 * Arguments: topk_idx and the four layout outputs as for
 * ep_get_dispatch_layout; the notify outputs and host_num_recv_tokens as for
 * ep_notify_dispatch.  send_pos must be 16-byte aligned.  An expert id
 * outside [-1, E) sets EP_DEV_INPUT and is ignored.
 *   workspace        device scratch of at least
 *                    ep_layout_notify_workspace_bytes(shape) bytes, 16-byte
 *                    aligned, zero-filled once before its first use; every
 *                    call leaves it ready for the next, so it is never
 *                    cleared again.  It may serve calls of any shape in turn
 *                    (size it for the largest), and ep_layout_notify_dispatch
 *                    calls too, but not two calls at once, and not
 *                    ep_notify_dispatch (whose workspace holds other data:
 *                    zero it again before switching).
 */
ep_status_t ep_layout_notify(const ep_shape_t* shape, const int64_t* topk_idx,
                             int32_t* num_tokens_per_rank, int32_t* num_tokens_per_rdma_rank,
                             int32_t* num_tokens_per_expert, uint8_t* is_token_in_rank,
                             int32_t* rank_prefix_matrix, int32_t* gbl_channel_prefix_matrix,
                             int32_t* rdma_channel_prefix_matrix, int32_t* recv_gbl_rank_prefix_sum,
                             int32_t* recv_rdma_rank_prefix_sum, int32_t* recv_channel_offset,
                             int32_t* num_recv_tokens, int32_t* num_rdma_recv_tokens,
                             int32_t* num_recv_tokens_per_expert, int64_t* recv_base,
                             int32_t* send_pos, void* workspace, size_t workspace_bytes,
                             int32_t* status, int32_t* host_num_recv_tokens, cudaStream_t stream);

/* Bytes of workspace ep_layout_notify (and ep_layout_notify_dispatch) needs
 * for `shape`, or 0 for an invalid shape: a 256-byte header, 2 MiB + 64 KiB
 * of per-expert counter words (64-bit, [32][8192] + [8192]), 18 KiB of
 * per-source totals (two banks of 32 * 36 64-bit words) and 8 * (R + N) bytes
 * per tile, counting tiles of 256 tokens (T rounded up to 32 when smaller;
 * doubled, up to 8192, while there would be more than 16384 tiles). */
size_t ep_layout_notify_workspace_bytes(const ep_shape_t* shape);

/* Which kernel ep_layout_notify runs for this shape on the current device:
 * 1 = the cluster form, 2 = the tiled form (both are one launch), -1 for an
 * invalid shape. */
int32_t ep_layout_notify_fused(const ep_shape_t* shape);

/* ------------------------------------------------------------------------
 * ep_notify_dispatch without a caller-provided workspace.  The paper has no
 * counterpart; this exists for callers that cannot allocate device memory -
 * for example code running inside a host framework that owns every device
 * allocation and hands a plugin only the tensors it must fill, or a serving
 * loop that forbids allocation after start-up - and so have no way to supply
 * the workspace.
 *
 * Same arguments, outputs and errors as ep_notify_dispatch, minus
 * `workspace` / `workspace_bytes`.  The scratch is a 1 MiB array compiled
 * into the library (a static __device__ array); every GPU that loads the
 * library holds it until the process exits.  A shape whose workspace
 * (ep_notify_workspace_bytes) exceeds 1 MiB - that is, 256 + R*C*(R+N)*8
 * bytes - is refused with EP_ERR_INVALID_ARG before anything is enqueued.
 * The call allocates and frees nothing.
 *
 * The first call on each device looks up the array's device address (a
 * cudaGetSymbolAddress with that device current) and caches it for the life
 * of the process; make that first call before any stream capture.  The
 * cached address belongs to the device's primary context: after
 * cudaDeviceReset, or from another context on the same device, it no longer
 * names the library's array, so do not use this entry point there.  All
 * calls share the one array and
 * each clears it on `stream` before use, so two calls whose executions
 * overlap on the GPU (different streams without ordering, or concurrent
 * host threads) race on it and give undefined results; order them.
 */
ep_status_t ep_notify_dispatch_noalloc(
    const ep_shape_t* shape, const uint8_t* is_token_in_rank,
    const int32_t* num_tokens_per_rank, const int32_t* num_tokens_per_rdma_rank,
    const int32_t* num_tokens_per_expert, int32_t* rank_prefix_matrix,
    int32_t* gbl_channel_prefix_matrix, int32_t* rdma_channel_prefix_matrix,
    int32_t* recv_gbl_rank_prefix_sum, int32_t* recv_rdma_rank_prefix_sum,
    int32_t* recv_channel_offset, int32_t* num_recv_tokens, int32_t* num_rdma_recv_tokens,
    int32_t* num_recv_tokens_per_expert, int64_t* recv_base, int32_t* send_pos, int32_t* status,
    int32_t* host_num_recv_tokens, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Step 3 - dispatch.  [RT] intranodeDispatch / internodeDispatch (receive
 * side: recv_x, recv_topk_idx, recv_topk_weights, source index), [AR] 4.1
 * (SrcInfo {src_rank, src_idx}).  Token (s,t) is copied to pool row
 * recv_base[r] + send_pos[s][t][r] for every r with send_pos >= 0.
 *
 *   x              in  bf16 bits (uint16) [R][T][H]
 *   topk_idx       in  int64 [R][T][K]
 *   topk_w         in  fp32  [R][T][K]
 *   send_pos       in  int32 [R][T][R]   from ep_notify_dispatch
 *   recv_base      in  int64 [R+1]       from ep_notify_dispatch (device)
 *   capacity_rows  rows allocated in the four recv_* arrays; a row at or
 *                  beyond it is not written and EP_DEV_CAPACITY is set.
 *                  R*T*min(K,R) always suffices.
 *   recv_x         out bf16 [capacity_rows][H]   bit copies of x rows
 *   recv_topk_idx  out int64 [capacity_rows][K]  local expert id (e - r*E_loc)
 *                      where expert e lives on the receiving rank r, else -1
 *   recv_topk_w    out fp32 [capacity_rows][K]   the slot's weight where its
 *                      expert lives on r, else 0
 *   recv_src_info  out int32 [capacity_rows][2]  (source rank, source token)
 *   sched          optional (may be NULL): one device uint64, zero before
 *                  the first call (e.g. one cudaMemset), left zero by every
 *                  call.  Given, the CTAs take row parts from it as a counter
 *                  once their first ring-full is done, so CTAs on SMs that
 *                  write faster take more (the pages' static split leaves
 *                  the whole call waiting on the slowest SM); NULL keeps the
 *                  static split, and so does a call whose CTAs have no more
 *                  row parts than their ring holds (small calls).  Calls whose executions may overlap on the
 *                  GPU (different streams, concurrent host threads) need one
 *                  sched word each.  Results are the same either way.
 * Rows beyond recv_base[R] are left untouched.
 * Cached mode ([RT] intranodeDispatch / internodeDispatch with cachedMode,
 * where the top-k is not dispatched): a handle (send_pos, recv_base) from an
 * earlier ep_notify_dispatch stays valid for any later step with the same
 * routing, so layout and notify can be skipped.  Pass topk_idx, topk_w,
 * recv_topk_idx and recv_topk_w all as NULL to move only the rows;
 * recv_src_info may be NULL in any mode.
 * Kernels of this library overlap their launch with the preceding kernel in
 * the stream (programmatic dependent launch), and ep_dispatch starts reading
 * x before that kernel has finished; it waits for the row map before writing
 * anything.  So x must be complete by the time the step's kernels start,
 * which holds for any producer enqueued earlier in the stream unless that
 * producer itself releases its dependents early (griddepcontrol).
 */
ep_status_t ep_dispatch(const ep_shape_t* shape, const uint16_t* x, const int64_t* topk_idx,
                        const float* topk_w, const int32_t* send_pos, const int64_t* recv_base,
                        int64_t capacity_rows, uint16_t* recv_x, int64_t* recv_topk_idx,
                        float* recv_topk_w, int32_t* recv_src_info, int32_t* status, uint64_t* sched,
                        cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Step 3, FP8 rows.  [RT] intranodeDispatch / internodeDispatch take x with
 * an element size of 1 byte plus x_scales (num_scales fp32 per token) and
 * return recv_x_scales beside recv_x; the FP8 scale buffer is one of the
 * per-channel buffers sized in their asserts.  Same placement, top-k and
 * cached-mode rules as ep_dispatch; rows are H bytes (H % 16 == 0 here).
 * The bytes are copied as they are: quantising to and from e4m3 is the
 * caller's (the expert's) job.
 *
 *   x              in  uint8 [R][T][H]              FP8 (e4m3) activations
 *   x_scales       in  fp32  [R][T][num_scales]     or NULL when num_scales == 0
 *   num_scales     0 .. 4096 scales per token (for example one per 128 elements)
 *   recv_x         out uint8 [capacity_rows][H]
 *   recv_x_scales  out fp32  [capacity_rows][num_scales] (or NULL when 0)
 * other arguments as in ep_dispatch.
 */
ep_status_t ep_dispatch_fp8(const ep_shape_t* shape, const uint8_t* x, const float* x_scales,
                            int32_t num_scales, const int64_t* topk_idx, const float* topk_w,
                            const int32_t* send_pos, const int64_t* recv_base, int64_t capacity_rows,
                            uint8_t* recv_x, float* recv_x_scales, int64_t* recv_topk_idx,
                            float* recv_topk_w, int32_t* recv_src_info, int32_t* status,
                            uint64_t* sched, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Steps 1 to 3 in one launch: ep_layout_notify followed by ep_dispatch on
 * its row map ([RT] internodeNotifyDispatch then internodeDispatch; where
 * the pages hand notify's results to dispatch through per-channel head/tail
 * words, here one `ready` word of the workspace carries the call's sequence
 * number).  The dispatch CTAs load their first ring-full of x rows, take
 * tiles of the tiled layout + notify form (see ep_layout_notify) from its
 * ticket until none is left, wait - bounded, EP_DEV_TIMEOUT - until the
 * row map of the call is complete, and copy.  A CTA waits only on tiles taken
 * by CTAs that are already running, so the launch needs no co-residency.
 * Every output of ep_layout_notify and of ep_dispatch is written, with the
 * same values as the two calls.
 *
 * Arguments: topk_idx, the four layout outputs, the eleven notify outputs,
 * workspace / workspace_bytes (as for ep_layout_notify, the same workspace
 * may serve both calls in turn) and host_num_recv_tokens as for
 * ep_layout_notify; x, capacity_rows, recv_x, recv_src_info (may be NULL)
 * and sched as for ep_dispatch.  topk_w, recv_topk_idx and recv_topk_w
 * carry the top-k fields as in ep_dispatch, or are all three NULL (then only
 * rows and source info move).  With R*T == 0 only the layout + notify
 * outputs are written.
 */
ep_status_t ep_layout_notify_dispatch(
    const ep_shape_t* shape, const int64_t* topk_idx, const float* topk_w, const uint16_t* x,
    int32_t* num_tokens_per_rank, int32_t* num_tokens_per_rdma_rank, int32_t* num_tokens_per_expert,
    uint8_t* is_token_in_rank, int32_t* rank_prefix_matrix, int32_t* gbl_channel_prefix_matrix,
    int32_t* rdma_channel_prefix_matrix, int32_t* recv_gbl_rank_prefix_sum, int32_t* recv_rdma_rank_prefix_sum,
    int32_t* recv_channel_offset, int32_t* num_recv_tokens, int32_t* num_rdma_recv_tokens,
    int32_t* num_recv_tokens_per_expert, int64_t* recv_base, int32_t* send_pos, void* workspace,
    size_t workspace_bytes, int64_t capacity_rows, uint16_t* recv_x, int64_t* recv_topk_idx, float* recv_topk_w,
    int32_t* recv_src_info, int32_t* status, uint64_t* sched, int32_t* host_num_recv_tokens,
    cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Step 4 - combine.  [RT] intranodeCombine / internodeCombine (combined_x is
 * bf16, combined_topk_weights fp32), [AR] 4.2 (each received row returns to
 * its (src_rank, src_idx)).  For every source token (s,t):
 *   combined_x[s][t][h] = bf16_rne( sum over r ascending with
 *                          send_pos[s][t][r] >= 0 of float(y[recv_base[r] +
 *                          send_pos[s][t][r]][h]) ), starting from +0.0f;
 *   combined_w[s][t][k] = the same fp32 sum over y_w, not rounded.
 * A token with no destination combines to +0.  The sum is unweighted (an
 * expert applies its routing weights before combine).
 *
 *   y           in  bf16 bits [pool rows][H]  expert outputs, one per
 *                   received row (recv_x itself for an identity expert);
 *                   must be a valid array whenever R*T > 0
 *   y_w         in  fp32 [pool rows][K]; may be NULL when combined_w is
 *   y_rows      rows allocated in y (and y_w); a contribution whose row is
 *               at or beyond it is skipped and EP_DEV_CAPACITY is set
 *   send_pos    in  int32 [R][T][R]
 *   recv_base   in  int64 [R+1] (device)
 *   combined_x  out bf16 [R][T][H]
 *   combined_w  out fp32 [R][T][K], or NULL to skip the weights
 * Empty arrays (zero elements) may be passed as NULL in every call.
 */
ep_status_t ep_combine(const ep_shape_t* shape, const uint16_t* y, const float* y_w,
                       int64_t y_rows, const int32_t* send_pos, const int64_t* recv_base,
                       uint16_t* combined_x, float* combined_w, int32_t* status,
                       cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Low-latency layout (per-expert packed).  The pages name this second mode
 * and give only its transport ([RT] "Intra-node LL fast path setup": peer
 * pointers for LL dispatch/combine; LL combine's proxy threads); its data
 * layout here is a plain reading:
 *   - every non-masked top-k slot (s,t,k) naming expert e is one row of e's
 *     receive buffer: a token travels once per expert, not once per rank;
 *   - a buffer holds expert_capacity rows (R*T suffices when a token never
 *     names an expert twice); rows are in ascending (source rank, token,
 *     slot) order; a slot whose row would reach the capacity is dropped and
 *     EP_DEV_CAPACITY is set;
 *   - combine applies the routing weights (LL combine takes the top-k
 *     weights): combined_x[s][t] = bf16_rne(acc), acc = +0 and then, for each
 *     valid slot k ascending, acc = fma(topk_w[s][t][k], y[e_k][row_k], acc)
 *     (one rounding per step).
 * Buffers are indexed by global expert e = r*E_loc + j, so [E][cap] is the
 * same memory as [R][E_loc][cap] ([E_loc, R*T, H] per rank).
 *
 * ep_ll_layout
 *   topk_idx               in  int64 [R][T][K]
 *   num_tokens_per_expert  in  int32 [R][E]  (from ep_get_dispatch_layout or
 *                              ep_layout_notify), or NULL: then one
 *                              thread-block cluster of R CTAs counts the
 *                              slots itself and exchanges each source's
 *                              per-expert totals through distributed shared
 *                              memory.  NULL needs R <= 16, R*E <= 16384 and
 *                              such a cluster to fit on the device, else
 *                              EP_ERR_INVALID_ARG.
 *   expert_capacity        rows per expert buffer (>= 0)
 *   slot_pos               out int32 [R][T][K]  row in the slot's expert
 *                                                buffer, or -1
 *   layout_range           out int32 [E][R][2]  (first row, rows) of each
 *                                                source rank in the buffer
 *   count                  out int32 [E]        rows in each buffer (before
 *                                                any capacity drop)
 * ep_ll_dispatch (sched as for ep_dispatch)
 *   x [R][T][H] bf16, topk_idx, slot_pos (from ep_ll_layout) ->
 *   recv_x [E][expert_capacity][H] bf16, recv_src_info [E][expert_capacity][2]
 *   (source rank, token; may be NULL).  Rows not written are left as they are.
 * ep_ll_combine
 *   y [E][expert_capacity][H] bf16 (expert outputs, recv_x for an identity
 *   expert), topk_idx, topk_w [R][T][K] fp32, slot_pos -> combined_x [R][T][H].
 */
ep_status_t ep_ll_layout(const ep_shape_t* shape, const int64_t* topk_idx,
                         const int32_t* num_tokens_per_expert, int32_t expert_capacity,
                         int32_t* slot_pos, int32_t* layout_range, int32_t* count, int32_t* status,
                         cudaStream_t stream);
ep_status_t ep_ll_dispatch(const ep_shape_t* shape, const uint16_t* x, const int64_t* topk_idx,
                           const int32_t* slot_pos, int32_t expert_capacity, uint16_t* recv_x,
                           int32_t* recv_src_info, int32_t* status, uint64_t* sched,
                           cudaStream_t stream);
ep_status_t ep_ll_combine(const ep_shape_t* shape, const uint16_t* y, int32_t expert_capacity,
                          const int64_t* topk_idx, const float* topk_w, const int32_t* slot_pos,
                          uint16_t* combined_x, int32_t* status, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Waits for `stream`, reads the device status word (a 4-byte copy into host
 * memory owned by this call), and maps its bits to a status: EP_OK,
 * EP_ERR_TIMEOUT, EP_ERR_CAPACITY, EP_ERR_INPUT or EP_ERR_INCONSISTENT (in
 * that priority), or EP_ERR_CUDA when the wait or copy fails.  The word is
 * not cleared.
 */
ep_status_t ep_sync_status(const int32_t* status, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Testing hook for failure detection.  Runs ep_notify_dispatch on its
 * lookback path (whatever the shape) with the block at scan position
 * `stall_block` (-1: none) withholding its published prefix and every wait
 * bounded by `wait_limit_us` microseconds.  The blocks that wait
 * on it give up, set EP_DEV_TIMEOUT and exit, so the context stays usable.
 * Output contents are undefined after such a run.
 */
ep_status_t ep_debug_notify_dispatch_stall(
    const ep_shape_t* shape, const uint8_t* is_token_in_rank,
    const int32_t* num_tokens_per_rank, const int32_t* num_tokens_per_rdma_rank,
    const int32_t* num_tokens_per_expert, int32_t* rank_prefix_matrix,
    int32_t* gbl_channel_prefix_matrix, int32_t* rdma_channel_prefix_matrix,
    int32_t* recv_gbl_rank_prefix_sum, int32_t* recv_rdma_rank_prefix_sum,
    int32_t* recv_channel_offset, int32_t* num_recv_tokens, int32_t* num_rdma_recv_tokens,
    int32_t* num_recv_tokens_per_expert, int64_t* recv_base, int32_t* send_pos, void* workspace,
    size_t workspace_bytes, int32_t* status, int32_t stall_block, int32_t wait_limit_us,
    cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Testing hook for failure detection in dispatch.  Runs ep_dispatch (same
 * arguments) with CTA `stall_cta` withholding every ring-slot release (with
 * `sched` given, that CTA then keeps taking units from the counter, leaving
 * them undone, until it runs dry, so the word still ends at zero) and
 * every device wait bounded by `wait_limit_us` microseconds (1 .. 2e6).  That
 * CTA's producer gives up waiting for a free slot, its storer gives up
 * waiting for the next unit, both set EP_DEV_TIMEOUT and the CTA exits after
 * its in-flight bulk copies have completed, so the context stays usable.
 * The other CTAs finish normally.  Output contents are undefined after such a
 * run.  A shape whose CTAs all fit their units in the ring never waits for a
 * slot, and then nothing times out.
 */
ep_status_t ep_debug_dispatch_stall(const ep_shape_t* shape, const uint16_t* x, const int64_t* topk_idx,
                                    const float* topk_w, const int32_t* send_pos, const int64_t* recv_base,
                                    int64_t capacity_rows, uint16_t* recv_x, int64_t* recv_topk_idx,
                                    float* recv_topk_w, int32_t* recv_src_info, int32_t* status,
                                    uint64_t* sched, int32_t stall_cta, int32_t wait_limit_us,
                                    cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Testing hook for the tiled form of ep_layout_notify.  Runs it whatever the
 * shape, with tiles of `tile_tokens` tokens (0: the default; else a multiple
 * of 32 in [32, 8192]; the workspace must then hold what that tile size
 * needs: 256 + 2 MiB + 64 KiB + 18 KiB + 8 * (R + N) * R * ceil(T / tile)
 * bytes), tile number `stall_tile` (-1: none) withholding its lookback words
 * and its source-total adds, and every wait bounded by `wait_limit_us`
 * microseconds (1 .. 2e6).
 * Tiles that wait on the withheld words give up, set EP_DEV_TIMEOUT and go
 * on, so the context stays usable; outputs are undefined after such a run.
 */
ep_status_t ep_debug_layout_notify_tiled(
    const ep_shape_t* shape, const int64_t* topk_idx, int32_t* num_tokens_per_rank,
    int32_t* num_tokens_per_rdma_rank, int32_t* num_tokens_per_expert, uint8_t* is_token_in_rank,
    int32_t* rank_prefix_matrix, int32_t* gbl_channel_prefix_matrix, int32_t* rdma_channel_prefix_matrix,
    int32_t* recv_gbl_rank_prefix_sum, int32_t* recv_rdma_rank_prefix_sum, int32_t* recv_channel_offset,
    int32_t* num_recv_tokens, int32_t* num_rdma_recv_tokens, int32_t* num_recv_tokens_per_expert,
    int64_t* recv_base, int32_t* send_pos, void* workspace, size_t workspace_bytes, int32_t* status,
    int32_t* host_num_recv_tokens, int32_t tile_tokens, int32_t stall_tile, int32_t wait_limit_us,
    cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Testing hook for failure detection in ep_layout_notify_dispatch.  Same
 * arguments (no host_num_recv_tokens), with the layout + notify tile of
 * ticket `stall_tile` (>= 0) withholding its lookback words and every wait
 * bounded by `wait_limit_us` microseconds (1 .. 2e6).  The tiles that wait
 * on it give up and go on (EP_DEV_TIMEOUT); the row map is then wrong but
 * dispatch still writes no row outside the receive arrays; the context stays
 * usable and a later call is exact.  Output contents are undefined after
 * such a run.
 */
ep_status_t ep_debug_layout_notify_dispatch_stall(
    const ep_shape_t* shape, const int64_t* topk_idx, const float* topk_w, const uint16_t* x,
    int32_t* num_tokens_per_rank, int32_t* num_tokens_per_rdma_rank, int32_t* num_tokens_per_expert,
    uint8_t* is_token_in_rank, int32_t* rank_prefix_matrix, int32_t* gbl_channel_prefix_matrix,
    int32_t* rdma_channel_prefix_matrix, int32_t* recv_gbl_rank_prefix_sum, int32_t* recv_rdma_rank_prefix_sum,
    int32_t* recv_channel_offset, int32_t* num_recv_tokens, int32_t* num_rdma_recv_tokens,
    int32_t* num_recv_tokens_per_expert, int64_t* recv_base, int32_t* send_pos, void* workspace,
    size_t workspace_bytes, int64_t capacity_rows, uint16_t* recv_x, int64_t* recv_topk_idx, float* recv_topk_w,
    int32_t* recv_src_info, int32_t* status, uint64_t* sched, int32_t stall_tile, int32_t wait_limit_us,
    cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* EP_GB300_H */
