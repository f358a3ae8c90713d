// Host-side interface between the C ABI (ep_api.cu) and the kernel launchers.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace ep {

struct Shape {
    int R, T, K, E, H, C, align;
    int N;      // nodes: max(1, R / 8)
    int E_loc;  // experts per rank
    long long row_bytes() const { return 2LL * H; }
};

// SM count of the current device (0 on error).
int device_sm_count();

// Whether one thread-block cluster of `cluster` CTAs of `kernel` (threads,
// dynamic shared bytes) can be resident on the current device.  Asked once
// per device and configuration, then cached; sets the kernel's attributes
// through prepare_kernel (dynamic shared size above 48 KB, non-portable
// cluster size above 8).
bool cluster_fits(const void* kernel, int cluster, int threads, size_t smem);

cudaError_t launch_layout(const Shape& sh, const int64_t* topk_idx, int32_t* num_tokens_per_rank,
                          int32_t* num_tokens_per_rdma_rank, int32_t* num_tokens_per_expert,
                          uint8_t* is_token_in_rank, int32_t* status, cudaStream_t stream);

struct NotifyArgs {
    const uint8_t* is_token_in_rank;
    const int32_t* num_tokens_per_rank;
    const int32_t* num_tokens_per_rdma_rank;
    const int32_t* num_tokens_per_expert;
    int32_t* rank_prefix_matrix;
    int32_t* gbl_channel_prefix_matrix;
    int32_t* rdma_channel_prefix_matrix;
    int32_t* recv_gbl_rank_prefix_sum;
    int32_t* recv_rdma_rank_prefix_sum;
    int32_t* recv_channel_offset;
    int32_t* num_recv_tokens;
    int32_t* num_rdma_recv_tokens;
    int32_t* num_recv_tokens_per_expert;
    int64_t* recv_base;
    int32_t* send_pos;
    int32_t* status;
    int32_t* host_num_recv_tokens;
};

size_t notify_workspace_bytes(const Shape& sh);

// Size of the library's static notify scratch (ep_notify_dispatch_noalloc).
constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;

// Device address of that scratch on the current device (looked up once per
// device, then cached).
cudaError_t notify_noalloc_scratch(void** out);

// `workspace` must hold notify_workspace_bytes(sh) bytes and be zero before
// its first use; calls keep it valid for the next call.  With
// clear_workspace the launcher zeroes it on `stream` first.  force_lookback
// keeps the inter-block lookback scan even for small sources (test hooks).
// stall_block < 0 for normal runs.
cudaError_t launch_notify(const Shape& sh, const NotifyArgs& a, void* workspace, bool clear_workspace,
                          bool force_lookback, int stall_block, long long wait_limit_ns,
                          cudaStream_t stream);

// CTAs of `kernel` (threads, dynamic shared bytes) one SM holds at once on
// the current device (0 on error); asked once per device and configuration.
int max_blocks_per_sm(const void* kernel, int threads, size_t smem);

// Layout and notify in one launch for any shape: the tiled form.  Tiles of
// `tile_tokens` tokens (0: the default for the shape; else a multiple of 32,
// at most 8192); the workspace holds tiled_workspace_bytes(sh, TT) bytes with
// its first tiled_workspace_zero_bytes() zero before the first call (every
// call leaves them zero).  stall_tile >= 0 (test hook): that tile never
// publishes its lookback words.
int tiled_tile_tokens(const Shape& sh, int requested);
int tiled_sizing_tokens(const Shape& sh);
size_t tiled_workspace_bytes(const Shape& sh, int TT);
size_t tiled_workspace_zero_bytes();
cudaError_t launch_layout_notify_tiled(const Shape& sh, const int64_t* topk_idx, int32_t* num_tokens_per_rank,
                                       int32_t* num_tokens_per_rdma_rank, int32_t* num_tokens_per_expert,
                                       uint8_t* is_token_in_rank, const NotifyArgs& a, void* workspace,
                                       int tile_tokens, int stall_tile, long long wait_limit_ns,
                                       cudaStream_t stream);

// Layout and notify in one launch (a cluster of R CTAs).  Usable when R <= 16,
// T <= 8192 and such a cluster fits on the current device.
bool layout_notify_fused_ok(const Shape& sh);
cudaError_t launch_layout_notify(const Shape& sh, const int64_t* topk_idx, int32_t* num_tokens_per_rank,
                                 int32_t* num_tokens_per_rdma_rank, int32_t* num_tokens_per_expert,
                                 uint8_t* is_token_in_rank, const NotifyArgs& a, cudaStream_t stream);

// x rows are H * x_elem_bytes bytes (2: bf16, 1: FP8); x_scales /
// recv_x_scales ([tokens|rows][num_scales] fp32) may be NULL.
// stall_release_cta >= 0 (test hook): that CTA's storer never frees a ring
// slot, so its producer's bounded wait runs out (EP_DEV_TIMEOUT).
// sched: 8-byte unit counter for dynamic assignment (zero before the call,
// zero after it), or NULL for the static split.
cudaError_t launch_dispatch(const Shape& sh, const void* x, int x_elem_bytes, const float* x_scales,
                            int num_scales, const int64_t* topk_idx, const float* topk_w,
                            const int32_t* send_pos, const int64_t* recv_base, int64_t capacity_rows,
                            void* recv_x, float* recv_x_scales, int64_t* recv_topk_idx,
                            float* recv_topk_w, int32_t* recv_src_info, int32_t* status,
                            unsigned long long* sched, cudaStream_t stream, int stall_release_cta = -1,
                            long long wait_limit_ns = 1000000000LL);

// Layout, notify and dispatch in one launch (the tiled layout + notify inside
// the dispatch grid; see ep_layout_notify_dispatch).  Top-k fields travel
// when topk_w is given.
cudaError_t launch_layout_notify_dispatch(const Shape& sh, const int64_t* topk_idx, const float* topk_w,
                                          const uint16_t* x, int32_t* num_tokens_per_rank,
                                          int32_t* num_tokens_per_rdma_rank, int32_t* num_tokens_per_expert,
                                          uint8_t* is_token_in_rank, const NotifyArgs& a, void* workspace,
                                          int64_t capacity_rows, uint16_t* recv_x, int64_t* recv_topk_idx,
                                          float* recv_topk_w, int32_t* recv_src_info, int32_t* status,
                                          unsigned long long* sched, int tile_tokens, int stall_tile,
                                          long long wait_limit_ns, cudaStream_t stream);

cudaError_t launch_combine(const Shape& sh, const uint16_t* y, const float* y_w, int64_t y_rows,
                           const int32_t* send_pos, const int64_t* recv_base, uint16_t* combined_x,
                           float* combined_w, int32_t* status, cudaStream_t stream);

// Low-latency (per-expert packed) layout: row of every top-k slot in its
// expert's buffer of `cap` rows (-1 when masked or beyond cap), per-source
// ranges [E][R][2] and per-expert counts [E].
cudaError_t launch_ll_layout(const Shape& sh, const int64_t* topk_idx, const int32_t* num_tokens_per_expert,
                             int cap, int32_t* slot_pos, int32_t* layout_range, int32_t* count,
                             int32_t* status, cudaStream_t stream);

// The same without the per-expert count input: one cluster of R CTAs counts
// and exchanges the per-source totals through distributed shared memory.
// Usable when R <= 16, R * E <= 16384 and such a cluster fits.
bool ll_layout_counting_ok(const Shape& sh);
cudaError_t launch_ll_layout_counting(const Shape& sh, const int64_t* topk_idx, int cap, int32_t* slot_pos,
                                      int32_t* layout_range, int32_t* count, int32_t* status,
                                      cudaStream_t stream);

// LL dispatch / combine share the dispatch and combine kernels; rows are
// resolved from (topk_idx, slot_pos) as expert * cap + pos.
cudaError_t launch_ll_dispatch(const Shape& sh, const uint16_t* x, const int64_t* topk_idx,
                               const int32_t* slot_pos, int cap, uint16_t* recv_x,
                               int32_t* recv_src_info, int32_t* status, unsigned long long* sched,
                               cudaStream_t stream);
cudaError_t launch_ll_combine(const Shape& sh, const uint16_t* y, int cap, const int64_t* topk_idx,
                              const float* topk_w, const int32_t* slot_pos, uint16_t* combined_x,
                              int32_t* status, cudaStream_t stream);

}  // namespace ep
