// C ABI of libep_gb300.so (declared in include/ep.h): argument checks on the
// host, then one launch per step on the caller's stream.
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "ep.h"
#include "ep_device.cuh"
#include "ep_internal.h"

namespace ep {

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_sm_mu;
int g_sm_count[kMaxDevices] = {};

struct KernelState {
    const void* kernel;
    int dev;
    size_t smem_limit;  // dynamic shared bytes allowed so far
    bool max_shared, nonportable;
};
std::mutex g_kernel_mu;
KernelState g_kernels[256];
int g_kernel_count = 0;
}  // namespace

int device_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < kMaxDevices) {
        std::lock_guard<std::mutex> lock(g_sm_mu);
        if (g_sm_count[dev] > 0) return g_sm_count[dev];
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < kMaxDevices) {
        std::lock_guard<std::mutex> lock(g_sm_mu);
        g_sm_count[dev] = sms;
    }
    return sms;
}

cudaError_t prepare_kernel(const void* kernel, size_t smem, bool max_shared, bool nonportable_cluster) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_kernel_mu);
    KernelState* st = nullptr;
    for (int i = 0; i < g_kernel_count; ++i)
        if (g_kernels[i].kernel == kernel && g_kernels[i].dev == dev) st = &g_kernels[i];
    KernelState fresh = {kernel, dev, 48 * 1024, false, false};
    KernelState& k = st != nullptr ? *st : fresh;
    if (max_shared && !k.max_shared) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        k.max_shared = true;
    }
    if (smem > k.smem_limit) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        k.smem_limit = smem;
    }
    if (nonportable_cluster && !k.nonportable) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        k.nonportable = true;
    }
    if (st == nullptr && g_kernel_count < 256) g_kernels[g_kernel_count++] = fresh;
    return cudaSuccess;
}

namespace {
struct FitKey {
    const void* kernel;
    int dev, cluster, threads;
    size_t smem;
    bool fits;
};
std::mutex g_fit_mu;
FitKey g_fit_cache[128];
int g_fit_count = 0;
}  // namespace

bool cluster_fits(const void* kernel, int cluster, int threads, size_t smem) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lock(g_fit_mu);
    for (int i = 0; i < g_fit_count; ++i) {
        const FitKey& k = g_fit_cache[i];
        if (k.kernel == kernel && k.dev == dev && k.cluster == cluster && k.threads == threads && k.smem == smem)
            return k.fits;
    }
    // the same attribute cache as the launches, so the shared-memory limit only grows
    bool fits = prepare_kernel(kernel, smem, false, cluster > 8) == cudaSuccess;
    if (fits) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(cluster));
        cfg.blockDim = dim3(static_cast<unsigned>(threads));
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = static_cast<unsigned>(cluster);
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        fits = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) == cudaSuccess && clusters > 0;
        cudaGetLastError();  // a refused query leaves no sticky error behind
    }
    if (g_fit_count < 128) g_fit_cache[g_fit_count++] = FitKey{kernel, dev, cluster, threads, smem, fits};
    return fits;
}

namespace {
struct OccKey {
    const void* kernel;
    int dev, threads;
    size_t smem;
    int blocks;
};
std::mutex g_occ_mu;
OccKey g_occ_cache[64];
int g_occ_count = 0;
}  // namespace

int max_blocks_per_sm(const void* kernel, int threads, size_t smem) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lock(g_occ_mu);
    for (int i = 0; i < g_occ_count; ++i) {
        const OccKey& k = g_occ_cache[i];
        if (k.kernel == kernel && k.dev == dev && k.threads == threads && k.smem == smem) return k.blocks;
    }
    int blocks = 0;
    if (prepare_kernel(kernel, smem, false, false) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kernel, threads, smem) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    if (g_occ_count < 64) g_occ_cache[g_occ_count++] = OccKey{kernel, dev, threads, smem, blocks};
    return blocks;
}

namespace {

bool make_shape(const ep_shape_t* s, Shape* out) {
    if (s == nullptr) return false;
    const long long R = s->num_ranks, T = s->num_tokens, K = s->num_topk, E = s->num_experts,
                    H = s->hidden, C = s->num_channels, A = s->expert_alignment;
    if (R < 1 || R > 32) return false;
    if (R > kNodeSize && R % kNodeSize != 0) return false;
    if (T < 0 || R * T >= (1LL << 30)) return false;
    if (K < 1 || K > 32) return false;
    if (E < R || E % R != 0 || E > 8192) return false;
    if (H < 8 || H % 8 != 0 || H > (1 << 24)) return false;
    if (C < 1 || C > 4096) return false;
    if (A < 1) return false;
    out->R = static_cast<int>(R);
    out->T = static_cast<int>(T);
    out->K = static_cast<int>(K);
    out->E = static_cast<int>(E);
    out->H = static_cast<int>(H);
    out->C = static_cast<int>(C);
    out->align = static_cast<int>(A);
    out->N = R <= kNodeSize ? 1 : static_cast<int>(R / kNodeSize);
    out->E_loc = static_cast<int>(E / R);
    return true;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned8(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 7u) == 0; }
bool aligned4(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// An array of `n` elements: any pointer (even NULL) when empty, else non-NULL
// and aligned to `align` bytes.
bool array_ok(const void* p, long long n, unsigned align) {
    if (n == 0) return true;
    return p != nullptr && (reinterpret_cast<uintptr_t>(p) & (align - 1u)) == 0;
}

ep_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? EP_OK : EP_ERR_CUDA; }

ep_status_t notify_common(const ep_shape_t* shape, const uint8_t* is_token_in_rank,
                          const int32_t* num_tokens_per_rank, const int32_t* num_tokens_per_rdma_rank,
                          const int32_t* num_tokens_per_expert, int32_t* rank_prefix_matrix,
                          int32_t* gbl_channel_prefix_matrix, int32_t* rdma_channel_prefix_matrix,
                          int32_t* recv_gbl_rank_prefix_sum, int32_t* recv_rdma_rank_prefix_sum,
                          int32_t* recv_channel_offset, int32_t* num_recv_tokens,
                          int32_t* num_rdma_recv_tokens, int32_t* num_recv_tokens_per_expert,
                          int64_t* recv_base, int32_t* send_pos, void* workspace,
                          size_t workspace_bytes, int32_t* status, int32_t* host_num_recv_tokens,
                          bool clear_workspace, bool force_lookback, int stall_block,
                          long long wait_limit_ns, cudaStream_t stream) {
    Shape sh;
    if (!make_shape(shape, &sh)) return EP_ERR_INVALID_ARG;
    const long long tok_rank = static_cast<long long>(sh.R) * sh.T * sh.R;
    if (!array_ok(is_token_in_rank, tok_rank, 16) || !aligned4(num_tokens_per_rank) ||
        !aligned4(num_tokens_per_rdma_rank) || !aligned4(num_tokens_per_expert) ||
        !aligned4(rank_prefix_matrix) || !aligned4(gbl_channel_prefix_matrix) ||
        !aligned4(rdma_channel_prefix_matrix) || !aligned4(recv_gbl_rank_prefix_sum) ||
        !aligned4(recv_rdma_rank_prefix_sum) || !aligned4(recv_channel_offset) ||
        !aligned4(num_recv_tokens) || !aligned4(num_rdma_recv_tokens) ||
        !aligned4(num_recv_tokens_per_expert) || !aligned8(recv_base) ||
        !array_ok(send_pos, tok_rank, 4) || !aligned16(workspace) || !aligned4(status))
        return EP_ERR_INVALID_ARG;
    if (host_num_recv_tokens != nullptr && !aligned4(host_num_recv_tokens)) return EP_ERR_INVALID_ARG;
    if (workspace_bytes < notify_workspace_bytes(sh)) return EP_ERR_INVALID_ARG;
    NotifyArgs a;
    a.is_token_in_rank = is_token_in_rank;
    a.num_tokens_per_rank = num_tokens_per_rank;
    a.num_tokens_per_rdma_rank = num_tokens_per_rdma_rank;
    a.num_tokens_per_expert = num_tokens_per_expert;
    a.rank_prefix_matrix = rank_prefix_matrix;
    a.gbl_channel_prefix_matrix = gbl_channel_prefix_matrix;
    a.rdma_channel_prefix_matrix = rdma_channel_prefix_matrix;
    a.recv_gbl_rank_prefix_sum = recv_gbl_rank_prefix_sum;
    a.recv_rdma_rank_prefix_sum = recv_rdma_rank_prefix_sum;
    a.recv_channel_offset = recv_channel_offset;
    a.num_recv_tokens = num_recv_tokens;
    a.num_rdma_recv_tokens = num_rdma_recv_tokens;
    a.num_recv_tokens_per_expert = num_recv_tokens_per_expert;
    a.recv_base = recv_base;
    a.send_pos = send_pos;
    a.status = status;
    a.host_num_recv_tokens = host_num_recv_tokens;
    return from_cuda(
        launch_notify(sh, a, workspace, clear_workspace, force_lookback, stall_block, wait_limit_ns,
                      stream));
}

// Pointer checks shared by the one-call layout + notify entry points; fills
// the notify outputs of `a`.
ep_status_t layout_notify_args(const Shape& sh, const int64_t* topk_idx, int32_t* num_tokens_per_rank,
                               int32_t* num_tokens_per_rdma_rank, int32_t* num_tokens_per_expert,
                               uint8_t* is_token_in_rank, int32_t* rank_prefix_matrix,
                               int32_t* gbl_channel_prefix_matrix, int32_t* rdma_channel_prefix_matrix,
                               int32_t* recv_gbl_rank_prefix_sum, int32_t* recv_rdma_rank_prefix_sum,
                               int32_t* recv_channel_offset, int32_t* num_recv_tokens,
                               int32_t* num_rdma_recv_tokens, int32_t* num_recv_tokens_per_expert,
                               int64_t* recv_base, int32_t* send_pos, int32_t* status,
                               int32_t* host_num_recv_tokens, NotifyArgs* a) {
    const long long tokens = static_cast<long long>(sh.R) * sh.T;
    if (!array_ok(topk_idx, tokens * sh.K, 16) || !aligned4(num_tokens_per_rank) ||
        !aligned4(num_tokens_per_rdma_rank) || !aligned4(num_tokens_per_expert) ||
        !array_ok(is_token_in_rank, tokens * sh.R, 16) || !array_ok(send_pos, tokens * sh.R, 16) ||
        !aligned4(status) || !aligned4(rank_prefix_matrix) || !aligned4(gbl_channel_prefix_matrix) ||
        !aligned4(rdma_channel_prefix_matrix) || !aligned4(recv_gbl_rank_prefix_sum) ||
        !aligned4(recv_rdma_rank_prefix_sum) || !aligned4(recv_channel_offset) || !aligned4(num_recv_tokens) ||
        !aligned4(num_rdma_recv_tokens) || !aligned4(num_recv_tokens_per_expert) || !aligned8(recv_base))
        return EP_ERR_INVALID_ARG;
    if (host_num_recv_tokens != nullptr && !aligned4(host_num_recv_tokens)) return EP_ERR_INVALID_ARG;
    a->rank_prefix_matrix = rank_prefix_matrix;
    a->gbl_channel_prefix_matrix = gbl_channel_prefix_matrix;
    a->rdma_channel_prefix_matrix = rdma_channel_prefix_matrix;
    a->recv_gbl_rank_prefix_sum = recv_gbl_rank_prefix_sum;
    a->recv_rdma_rank_prefix_sum = recv_rdma_rank_prefix_sum;
    a->recv_channel_offset = recv_channel_offset;
    a->num_recv_tokens = num_recv_tokens;
    a->num_rdma_recv_tokens = num_rdma_recv_tokens;
    a->num_recv_tokens_per_expert = num_recv_tokens_per_expert;
    a->recv_base = recv_base;
    a->send_pos = send_pos;
    a->status = status;
    a->host_num_recv_tokens = host_num_recv_tokens;
    return EP_OK;
}

// Which kernel ep_layout_notify runs: 1 = one thread-block cluster of R CTAs
// (R <= 16, T <= 1024, R * T <= 8192 and the cluster fits: there it is as
// fast as the tiled form or faster, e.g. 10.0 vs 10.3 us at R = 16, T = 128
// and 11.7 vs 12.3 us at T = 512; with more tokens per CTA it falls behind,
// 13.5 vs 12.3 us at T = 1024), 2 = the tiled form (any shape).
constexpr long long kClusterMaxTokensPerRank = 1024;
constexpr long long kClusterMaxTokens = 8192;

int layout_notify_form(const Shape& sh) {
    if (sh.T <= kClusterMaxTokensPerRank && static_cast<long long>(sh.R) * sh.T <= kClusterMaxTokens &&
        layout_notify_fused_ok(sh))
        return 1;
    return 2;
}

}  // namespace
// Argument checks and launch shared by ep_dispatch and its stall test hook.
ep_status_t dispatch_common(const ep_shape_t* shape, const uint16_t* x, const int64_t* topk_idx,
                            const float* topk_w, const int32_t* send_pos, const int64_t* recv_base,
                            int64_t capacity_rows, uint16_t* recv_x, int64_t* recv_topk_idx,
                            float* recv_topk_w, int32_t* recv_src_info, int32_t* status,
                            uint64_t* sched, cudaStream_t stream, int stall_cta, long long wait_limit_ns);

}  // namespace ep

extern "C" {

const char* ep_status_string(ep_status_t status) {
    switch (status) {
        case EP_OK: return "ok";
        case EP_ERR_INVALID_ARG: return "invalid argument";
        case EP_ERR_CUDA: return "CUDA runtime error";
        case EP_ERR_CAPACITY: return "receive capacity exceeded";
        case EP_ERR_TIMEOUT: return "device wait timed out";
        case EP_ERR_INCONSISTENT: return "count inputs disagree with is_token_in_rank";
        case EP_ERR_INPUT: return "expert id outside [-1, num_experts)";
    }
    return "unknown status";
}

ep_status_t ep_check_shape(const ep_shape_t* shape) {
    ep::Shape sh;
    return ep::make_shape(shape, &sh) ? EP_OK : EP_ERR_INVALID_ARG;
}

int32_t ep_num_nodes(const ep_shape_t* shape) {
    ep::Shape sh;
    return ep::make_shape(shape, &sh) ? sh.N : -1;
}

size_t ep_notify_workspace_bytes(const ep_shape_t* shape) {
    ep::Shape sh;
    return ep::make_shape(shape, &sh) ? ep::notify_workspace_bytes(sh) : 0;
}

ep_status_t ep_get_dispatch_layout(const ep_shape_t* shape, const int64_t* topk_idx,
                                   int32_t* num_tokens_per_rank, int32_t* num_tokens_per_rdma_rank,
                                   int32_t* num_tokens_per_expert, uint8_t* is_token_in_rank,
                                   int32_t* status, cudaStream_t stream) {
    ep::Shape sh;
    if (!ep::make_shape(shape, &sh)) return EP_ERR_INVALID_ARG;
    const long long tokens = static_cast<long long>(sh.R) * sh.T;
    if (!ep::array_ok(topk_idx, tokens * sh.K, 16) || !ep::aligned4(num_tokens_per_rank) ||
        !ep::aligned4(num_tokens_per_rdma_rank) || !ep::aligned4(num_tokens_per_expert) ||
        !ep::array_ok(is_token_in_rank, tokens * sh.R, 16) || !ep::aligned4(status))
        return EP_ERR_INVALID_ARG;
    return ep::from_cuda(ep::launch_layout(sh, topk_idx, num_tokens_per_rank, num_tokens_per_rdma_rank,
                                           num_tokens_per_expert, is_token_in_rank, status, stream));
}

ep_status_t ep_notify_dispatch(const ep_shape_t* shape, const uint8_t* is_token_in_rank,
                               const int32_t* num_tokens_per_rank,
                               const int32_t* num_tokens_per_rdma_rank,
                               const int32_t* num_tokens_per_expert, int32_t* rank_prefix_matrix,
                               int32_t* gbl_channel_prefix_matrix,
                               int32_t* rdma_channel_prefix_matrix,
                               int32_t* recv_gbl_rank_prefix_sum,
                               int32_t* recv_rdma_rank_prefix_sum, int32_t* recv_channel_offset,
                               int32_t* num_recv_tokens, int32_t* num_rdma_recv_tokens,
                               int32_t* num_recv_tokens_per_expert, int64_t* recv_base,
                               int32_t* send_pos, void* workspace, size_t workspace_bytes,
                               int32_t* status, int32_t* host_num_recv_tokens,
                               cudaStream_t stream) {
    return ep::notify_common(shape, is_token_in_rank, num_tokens_per_rank, num_tokens_per_rdma_rank,
                             num_tokens_per_expert, rank_prefix_matrix, gbl_channel_prefix_matrix,
                             rdma_channel_prefix_matrix, recv_gbl_rank_prefix_sum,
                             recv_rdma_rank_prefix_sum, recv_channel_offset, num_recv_tokens,
                             num_rdma_recv_tokens, num_recv_tokens_per_expert, recv_base, send_pos,
                             workspace, workspace_bytes, status, host_num_recv_tokens, false, false, -1,
                             ep::kDefaultWaitLimitNs, stream);
}

int32_t ep_layout_notify_fused(const ep_shape_t* shape) {
    ep::Shape sh;
    if (!ep::make_shape(shape, &sh)) return -1;
    return ep::layout_notify_form(sh);
}

size_t ep_layout_notify_workspace_bytes(const ep_shape_t* shape) {
    ep::Shape sh;
    if (!ep::make_shape(shape, &sh)) return 0;
    return ep::tiled_workspace_bytes(sh, ep::tiled_sizing_tokens(sh));
}

ep_status_t ep_layout_notify(const ep_shape_t* shape, const int64_t* topk_idx,
                             int32_t* num_tokens_per_rank, int32_t* num_tokens_per_rdma_rank,
                             int32_t* num_tokens_per_expert, uint8_t* is_token_in_rank,
                             int32_t* rank_prefix_matrix, int32_t* gbl_channel_prefix_matrix,
                             int32_t* rdma_channel_prefix_matrix, int32_t* recv_gbl_rank_prefix_sum,
                             int32_t* recv_rdma_rank_prefix_sum, int32_t* recv_channel_offset,
                             int32_t* num_recv_tokens, int32_t* num_rdma_recv_tokens,
                             int32_t* num_recv_tokens_per_expert, int64_t* recv_base,
                             int32_t* send_pos, void* workspace, size_t workspace_bytes,
                             int32_t* status, int32_t* host_num_recv_tokens, cudaStream_t stream) {
    ep::Shape sh;
    if (!ep::make_shape(shape, &sh)) return EP_ERR_INVALID_ARG;
    ep::NotifyArgs a = {};
    const ep_status_t st = ep::layout_notify_args(
        sh, topk_idx, num_tokens_per_rank, num_tokens_per_rdma_rank, num_tokens_per_expert, is_token_in_rank,
        rank_prefix_matrix, gbl_channel_prefix_matrix, rdma_channel_prefix_matrix, recv_gbl_rank_prefix_sum,
        recv_rdma_rank_prefix_sum, recv_channel_offset, num_recv_tokens, num_rdma_recv_tokens,
        num_recv_tokens_per_expert, recv_base, send_pos, status, host_num_recv_tokens, &a);
    if (st != EP_OK) return st;
    if (!ep::aligned16(workspace) || workspace_bytes < ep::tiled_workspace_bytes(sh, ep::tiled_sizing_tokens(sh)))
        return EP_ERR_INVALID_ARG;
    if (ep::layout_notify_form(sh) == 1)
        return ep::from_cuda(ep::launch_layout_notify(sh, topk_idx, num_tokens_per_rank, num_tokens_per_rdma_rank,
                                                      num_tokens_per_expert, is_token_in_rank, a, stream));
    return ep::from_cuda(ep::launch_layout_notify_tiled(sh, topk_idx, num_tokens_per_rank, num_tokens_per_rdma_rank,
                                                        num_tokens_per_expert, is_token_in_rank, a, workspace, 0,
                                                        -1, ep::kDefaultWaitLimitNs, stream));
}

ep_status_t ep_debug_layout_notify_tiled(
    const ep_shape_t* shape, const int64_t* topk_idx, int32_t* num_tokens_per_rank,
    int32_t* num_tokens_per_rdma_rank, int32_t* num_tokens_per_expert, uint8_t* is_token_in_rank,
    int32_t* rank_prefix_matrix, int32_t* gbl_channel_prefix_matrix, int32_t* rdma_channel_prefix_matrix,
    int32_t* recv_gbl_rank_prefix_sum, int32_t* recv_rdma_rank_prefix_sum, int32_t* recv_channel_offset,
    int32_t* num_recv_tokens, int32_t* num_rdma_recv_tokens, int32_t* num_recv_tokens_per_expert,
    int64_t* recv_base, int32_t* send_pos, void* workspace, size_t workspace_bytes, int32_t* status,
    int32_t* host_num_recv_tokens, int32_t tile_tokens, int32_t stall_tile, int32_t wait_limit_us,
    cudaStream_t stream) {
    ep::Shape sh;
    if (!ep::make_shape(shape, &sh)) return EP_ERR_INVALID_ARG;
    if (tile_tokens != 0 && (tile_tokens < 32 || tile_tokens > 8192 || tile_tokens % 32 != 0))
        return EP_ERR_INVALID_ARG;
    if (wait_limit_us < 1 || wait_limit_us > 2000000) return EP_ERR_INVALID_ARG;
    ep::NotifyArgs a = {};
    const ep_status_t st = ep::layout_notify_args(
        sh, topk_idx, num_tokens_per_rank, num_tokens_per_rdma_rank, num_tokens_per_expert, is_token_in_rank,
        rank_prefix_matrix, gbl_channel_prefix_matrix, rdma_channel_prefix_matrix, recv_gbl_rank_prefix_sum,
        recv_rdma_rank_prefix_sum, recv_channel_offset, num_recv_tokens, num_rdma_recv_tokens,
        num_recv_tokens_per_expert, recv_base, send_pos, status, host_num_recv_tokens, &a);
    if (st != EP_OK) return st;
    const int sized = tile_tokens > 0 ? tile_tokens : ep::tiled_sizing_tokens(sh);
    if (!ep::aligned16(workspace) || workspace_bytes < ep::tiled_workspace_bytes(sh, sized)) return EP_ERR_INVALID_ARG;
    return ep::from_cuda(ep::launch_layout_notify_tiled(sh, topk_idx, num_tokens_per_rank, num_tokens_per_rdma_rank,
                                                        num_tokens_per_expert, is_token_in_rank, a, workspace, tile_tokens,
                                                        stall_tile, static_cast<long long>(wait_limit_us) * 1000LL,
                                                        stream));
}

}  // extern "C"

namespace ep {
namespace {

// Argument checks and launch shared by ep_layout_notify_dispatch and its
// stall test hook.
ep_status_t layout_notify_dispatch_common(
    const ep_shape_t* shape, const int64_t* topk_idx, const float* topk_w, const uint16_t* x,
    int32_t* num_tokens_per_rank, int32_t* num_tokens_per_rdma_rank, int32_t* num_tokens_per_expert,
    uint8_t* is_token_in_rank, int32_t* rank_prefix_matrix, int32_t* gbl_channel_prefix_matrix,
    int32_t* rdma_channel_prefix_matrix, int32_t* recv_gbl_rank_prefix_sum, int32_t* recv_rdma_rank_prefix_sum,
    int32_t* recv_channel_offset, int32_t* num_recv_tokens, int32_t* num_rdma_recv_tokens,
    int32_t* num_recv_tokens_per_expert, int64_t* recv_base, int32_t* send_pos, void* workspace,
    size_t workspace_bytes, int64_t capacity_rows, uint16_t* recv_x, int64_t* recv_topk_idx, float* recv_topk_w,
    int32_t* recv_src_info, int32_t* status, uint64_t* sched, int32_t* host_num_recv_tokens, int stall_tile,
    long long wait_limit_ns, cudaStream_t stream) {
    Shape sh;
    if (!make_shape(shape, &sh)) return EP_ERR_INVALID_ARG;
    NotifyArgs a = {};
    const ep_status_t st = layout_notify_args(
        sh, topk_idx, num_tokens_per_rank, num_tokens_per_rdma_rank, num_tokens_per_expert, is_token_in_rank,
        rank_prefix_matrix, gbl_channel_prefix_matrix, rdma_channel_prefix_matrix, recv_gbl_rank_prefix_sum,
        recv_rdma_rank_prefix_sum, recv_channel_offset, num_recv_tokens, num_rdma_recv_tokens,
        num_recv_tokens_per_expert, recv_base, send_pos, status, host_num_recv_tokens, &a);
    if (st != EP_OK) return st;
    if (!aligned16(workspace) || workspace_bytes < tiled_workspace_bytes(sh, tiled_sizing_tokens(sh)))
        return EP_ERR_INVALID_ARG;
    if (capacity_rows < 0) return EP_ERR_INVALID_ARG;
    const long long tokens = static_cast<long long>(sh.R) * sh.T;
    const long long cap = capacity_rows;
    // top-k fields: weights in, both receive arrays out - or all three NULL
    const bool topk_given = topk_w != nullptr || recv_topk_idx != nullptr || recv_topk_w != nullptr;
    if (topk_given && (!array_ok(topk_w, tokens * sh.K, 4) || !array_ok(recv_topk_idx, cap * sh.K, 8) ||
                       !array_ok(recv_topk_w, cap * sh.K, 4) || (tokens > 0 && topk_w == nullptr) ||
                       (cap > 0 && (recv_topk_idx == nullptr || recv_topk_w == nullptr))))
        return EP_ERR_INVALID_ARG;
    if (!array_ok(x, tokens * sh.H, 16) || !array_ok(recv_x, cap * sh.H, 16) ||
        (recv_src_info != nullptr && !aligned8(recv_src_info)) || (sched != nullptr && !aligned8(sched)))
        return EP_ERR_INVALID_ARG;
    return from_cuda(launch_layout_notify_dispatch(
        sh, topk_idx, topk_w, x, num_tokens_per_rank, num_tokens_per_rdma_rank, num_tokens_per_expert,
        is_token_in_rank, a, workspace, capacity_rows, recv_x, recv_topk_idx, recv_topk_w, recv_src_info, status,
        reinterpret_cast<unsigned long long*>(sched), 0, stall_tile, wait_limit_ns, stream));
}

}  // namespace
}  // namespace ep

extern "C" {

ep_status_t ep_layout_notify_dispatch(
    const ep_shape_t* shape, const int64_t* topk_idx, const float* topk_w, const uint16_t* x,
    int32_t* num_tokens_per_rank, int32_t* num_tokens_per_rdma_rank, int32_t* num_tokens_per_expert,
    uint8_t* is_token_in_rank, int32_t* rank_prefix_matrix, int32_t* gbl_channel_prefix_matrix,
    int32_t* rdma_channel_prefix_matrix, int32_t* recv_gbl_rank_prefix_sum, int32_t* recv_rdma_rank_prefix_sum,
    int32_t* recv_channel_offset, int32_t* num_recv_tokens, int32_t* num_rdma_recv_tokens,
    int32_t* num_recv_tokens_per_expert, int64_t* recv_base, int32_t* send_pos, void* workspace,
    size_t workspace_bytes, int64_t capacity_rows, uint16_t* recv_x, int64_t* recv_topk_idx, float* recv_topk_w,
    int32_t* recv_src_info, int32_t* status, uint64_t* sched, int32_t* host_num_recv_tokens,
    cudaStream_t stream) {
    return ep::layout_notify_dispatch_common(
        shape, topk_idx, topk_w, x, num_tokens_per_rank, num_tokens_per_rdma_rank, num_tokens_per_expert,
        is_token_in_rank, rank_prefix_matrix, gbl_channel_prefix_matrix, rdma_channel_prefix_matrix,
        recv_gbl_rank_prefix_sum, recv_rdma_rank_prefix_sum, recv_channel_offset, num_recv_tokens,
        num_rdma_recv_tokens, num_recv_tokens_per_expert, recv_base, send_pos, workspace, workspace_bytes,
        capacity_rows, recv_x, recv_topk_idx, recv_topk_w, recv_src_info, status, sched, host_num_recv_tokens, -1,
        ep::kDefaultWaitLimitNs, stream);
}

ep_status_t ep_debug_layout_notify_dispatch_stall(
    const ep_shape_t* shape, const int64_t* topk_idx, const float* topk_w, const uint16_t* x,
    int32_t* num_tokens_per_rank, int32_t* num_tokens_per_rdma_rank, int32_t* num_tokens_per_expert,
    uint8_t* is_token_in_rank, int32_t* rank_prefix_matrix, int32_t* gbl_channel_prefix_matrix,
    int32_t* rdma_channel_prefix_matrix, int32_t* recv_gbl_rank_prefix_sum, int32_t* recv_rdma_rank_prefix_sum,
    int32_t* recv_channel_offset, int32_t* num_recv_tokens, int32_t* num_rdma_recv_tokens,
    int32_t* num_recv_tokens_per_expert, int64_t* recv_base, int32_t* send_pos, void* workspace,
    size_t workspace_bytes, int64_t capacity_rows, uint16_t* recv_x, int64_t* recv_topk_idx, float* recv_topk_w,
    int32_t* recv_src_info, int32_t* status, uint64_t* sched, int32_t stall_tile, int32_t wait_limit_us,
    cudaStream_t stream) {
    if (stall_tile < 0 || wait_limit_us < 1 || wait_limit_us > 2000000) return EP_ERR_INVALID_ARG;
    return ep::layout_notify_dispatch_common(
        shape, topk_idx, topk_w, x, num_tokens_per_rank, num_tokens_per_rdma_rank, num_tokens_per_expert,
        is_token_in_rank, rank_prefix_matrix, gbl_channel_prefix_matrix, rdma_channel_prefix_matrix,
        recv_gbl_rank_prefix_sum, recv_rdma_rank_prefix_sum, recv_channel_offset, num_recv_tokens,
        num_rdma_recv_tokens, num_recv_tokens_per_expert, recv_base, send_pos, workspace, workspace_bytes,
        capacity_rows, recv_x, recv_topk_idx, recv_topk_w, recv_src_info, status, sched, nullptr, stall_tile,
        static_cast<long long>(wait_limit_us) * 1000LL, stream);
}

ep_status_t ep_notify_dispatch_noalloc(
    const ep_shape_t* shape, const uint8_t* is_token_in_rank, const int32_t* num_tokens_per_rank,
    const int32_t* num_tokens_per_rdma_rank, const int32_t* num_tokens_per_expert,
    int32_t* rank_prefix_matrix, int32_t* gbl_channel_prefix_matrix,
    int32_t* rdma_channel_prefix_matrix, int32_t* recv_gbl_rank_prefix_sum,
    int32_t* recv_rdma_rank_prefix_sum, int32_t* recv_channel_offset, int32_t* num_recv_tokens,
    int32_t* num_rdma_recv_tokens, int32_t* num_recv_tokens_per_expert, int64_t* recv_base,
    int32_t* send_pos, int32_t* status, int32_t* host_num_recv_tokens, cudaStream_t stream) {
    ep::Shape sh;
    if (!ep::make_shape(shape, &sh)) return EP_ERR_INVALID_ARG;
    // The shape must fit the fixed scratch; larger shapes are refused here,
    // before anything is enqueued.
    if (ep::notify_workspace_bytes(sh) > ep::kNoAllocScratchBytes) return EP_ERR_INVALID_ARG;
    void* scratch = nullptr;
    if (ep::notify_noalloc_scratch(&scratch) != cudaSuccess) return EP_ERR_CUDA;
    return ep::notify_common(shape, is_token_in_rank, num_tokens_per_rank, num_tokens_per_rdma_rank,
                             num_tokens_per_expert, rank_prefix_matrix, gbl_channel_prefix_matrix,
                             rdma_channel_prefix_matrix, recv_gbl_rank_prefix_sum,
                             recv_rdma_rank_prefix_sum, recv_channel_offset, num_recv_tokens,
                             num_rdma_recv_tokens, num_recv_tokens_per_expert, recv_base, send_pos,
                             scratch, ep::kNoAllocScratchBytes, status, host_num_recv_tokens, true, false, -1,
                             ep::kDefaultWaitLimitNs, stream);
}

ep_status_t ep_debug_notify_dispatch_stall(
    const ep_shape_t* shape, const uint8_t* is_token_in_rank, const int32_t* num_tokens_per_rank,
    const int32_t* num_tokens_per_rdma_rank, const int32_t* num_tokens_per_expert,
    int32_t* rank_prefix_matrix, int32_t* gbl_channel_prefix_matrix,
    int32_t* rdma_channel_prefix_matrix, int32_t* recv_gbl_rank_prefix_sum,
    int32_t* recv_rdma_rank_prefix_sum, int32_t* recv_channel_offset, int32_t* num_recv_tokens,
    int32_t* num_rdma_recv_tokens, int32_t* num_recv_tokens_per_expert, int64_t* recv_base,
    int32_t* send_pos, void* workspace, size_t workspace_bytes, int32_t* status,
    int32_t stall_block, int32_t wait_limit_us, cudaStream_t stream) {
    if (wait_limit_us < 1 || wait_limit_us > 2000000) return EP_ERR_INVALID_ARG;
    return ep::notify_common(shape, is_token_in_rank, num_tokens_per_rank, num_tokens_per_rdma_rank,
                             num_tokens_per_expert, rank_prefix_matrix, gbl_channel_prefix_matrix,
                             rdma_channel_prefix_matrix, recv_gbl_rank_prefix_sum,
                             recv_rdma_rank_prefix_sum, recv_channel_offset, num_recv_tokens,
                             num_rdma_recv_tokens, num_recv_tokens_per_expert, recv_base, send_pos,
                             workspace, workspace_bytes, status, nullptr, false, true, stall_block,
                             static_cast<long long>(wait_limit_us) * 1000LL, stream);
}

ep_status_t ep_dispatch(const ep_shape_t* shape, const uint16_t* x, const int64_t* topk_idx,
                        const float* topk_w, const int32_t* send_pos, const int64_t* recv_base,
                        int64_t capacity_rows, uint16_t* recv_x, int64_t* recv_topk_idx,
                        float* recv_topk_w, int32_t* recv_src_info, int32_t* status, uint64_t* sched,
                        cudaStream_t stream) {
    return ep::dispatch_common(shape, x, topk_idx, topk_w, send_pos, recv_base, capacity_rows, recv_x,
                               recv_topk_idx, recv_topk_w, recv_src_info, status, sched, stream, -1,
                               ep::kDefaultWaitLimitNs);
}

ep_status_t ep_debug_dispatch_stall(const ep_shape_t* shape, const uint16_t* x, const int64_t* topk_idx,
                                    const float* topk_w, const int32_t* send_pos, const int64_t* recv_base,
                                    int64_t capacity_rows, uint16_t* recv_x, int64_t* recv_topk_idx,
                                    float* recv_topk_w, int32_t* recv_src_info, int32_t* status,
                                    uint64_t* sched, int32_t stall_cta, int32_t wait_limit_us,
                                    cudaStream_t stream) {
    if (stall_cta < 0 || wait_limit_us < 1 || wait_limit_us > 2000000) return EP_ERR_INVALID_ARG;
    return ep::dispatch_common(shape, x, topk_idx, topk_w, send_pos, recv_base, capacity_rows, recv_x,
                               recv_topk_idx, recv_topk_w, recv_src_info, status, sched, stream, stall_cta,
                               static_cast<long long>(wait_limit_us) * 1000LL);
}

}  // extern "C"

namespace ep {

ep_status_t dispatch_common(const ep_shape_t* shape, const uint16_t* x, const int64_t* topk_idx,
                            const float* topk_w, const int32_t* send_pos, const int64_t* recv_base,
                            int64_t capacity_rows, uint16_t* recv_x, int64_t* recv_topk_idx,
                            float* recv_topk_w, int32_t* recv_src_info, int32_t* status,
                            uint64_t* sched, cudaStream_t stream, int stall_cta, long long wait_limit_ns) {
    ep::Shape sh;
    if (!ep::make_shape(shape, &sh)) return EP_ERR_INVALID_ARG;
    if (capacity_rows < 0) return EP_ERR_INVALID_ARG;
    const long long tokens = static_cast<long long>(sh.R) * sh.T;
    const long long cap = capacity_rows;
    // Cached mode ([RT] intranodeDispatch with cachedMode): the four top-k
    // arrays are all NULL and only rows (and optionally source info) move.
    const bool topk_given = topk_idx != nullptr || topk_w != nullptr || recv_topk_idx != nullptr ||
                            recv_topk_w != nullptr;
    if (topk_given && (!ep::array_ok(topk_idx, tokens * sh.K, 8) || !ep::array_ok(topk_w, tokens * sh.K, 4) ||
                       !ep::array_ok(recv_topk_idx, cap * sh.K, 8) || !ep::array_ok(recv_topk_w, cap * sh.K, 4) ||
                       (tokens > 0 && (topk_idx == nullptr || topk_w == nullptr)) ||
                       (cap > 0 && (recv_topk_idx == nullptr || recv_topk_w == nullptr))))
        return EP_ERR_INVALID_ARG;
    if (!ep::array_ok(x, tokens * sh.H, 16) || !ep::array_ok(send_pos, tokens * sh.R, 4) ||
        !ep::aligned8(recv_base) || !ep::array_ok(recv_x, cap * sh.H, 16) ||
        (recv_src_info != nullptr && !ep::aligned8(recv_src_info)) || !ep::aligned4(status) ||
        (sched != nullptr && !ep::aligned8(sched)))
        return EP_ERR_INVALID_ARG;
    return ep::from_cuda(ep::launch_dispatch(sh, x, 2, nullptr, 0, topk_idx, topk_w, send_pos, recv_base,
                                             capacity_rows, recv_x, nullptr, recv_topk_idx, recv_topk_w,
                                             recv_src_info, status,
                                             reinterpret_cast<unsigned long long*>(sched), stream, stall_cta,
                                             wait_limit_ns));
}

}  // namespace ep

extern "C" {

ep_status_t ep_dispatch_fp8(const ep_shape_t* shape, const uint8_t* x, const float* x_scales,
                            int32_t num_scales, const int64_t* topk_idx, const float* topk_w,
                            const int32_t* send_pos, const int64_t* recv_base, int64_t capacity_rows,
                            uint8_t* recv_x, float* recv_x_scales, int64_t* recv_topk_idx,
                            float* recv_topk_w, int32_t* recv_src_info, int32_t* status,
                            uint64_t* sched, cudaStream_t stream) {
    ep::Shape sh;
    if (!ep::make_shape(shape, &sh)) return EP_ERR_INVALID_ARG;
    if (sched != nullptr && !ep::aligned8(sched)) return EP_ERR_INVALID_ARG;
    if (capacity_rows < 0 || sh.H % 16 != 0 || num_scales < 0 || num_scales > 4096) return EP_ERR_INVALID_ARG;
    const long long tokens = static_cast<long long>(sh.R) * sh.T;
    const long long cap = capacity_rows;
    const bool topk_given = topk_idx != nullptr || topk_w != nullptr || recv_topk_idx != nullptr ||
                            recv_topk_w != nullptr;
    if (topk_given && (!ep::array_ok(topk_idx, tokens * sh.K, 8) || !ep::array_ok(topk_w, tokens * sh.K, 4) ||
                       !ep::array_ok(recv_topk_idx, cap * sh.K, 8) || !ep::array_ok(recv_topk_w, cap * sh.K, 4) ||
                       (tokens > 0 && (topk_idx == nullptr || topk_w == nullptr)) ||
                       (cap > 0 && (recv_topk_idx == nullptr || recv_topk_w == nullptr))))
        return EP_ERR_INVALID_ARG;
    if (num_scales > 0 && (!ep::array_ok(x_scales, tokens * num_scales, 4) ||
                           !ep::array_ok(recv_x_scales, cap * num_scales, 4) ||
                           (tokens > 0 && x_scales == nullptr) || (cap > 0 && recv_x_scales == nullptr)))
        return EP_ERR_INVALID_ARG;
    if (!ep::array_ok(x, tokens * sh.H, 16) || !ep::array_ok(send_pos, tokens * sh.R, 4) ||
        !ep::aligned8(recv_base) || !ep::array_ok(recv_x, cap * sh.H, 16) ||
        (recv_src_info != nullptr && !ep::aligned8(recv_src_info)) || !ep::aligned4(status))
        return EP_ERR_INVALID_ARG;
    return ep::from_cuda(ep::launch_dispatch(sh, x, 1, num_scales > 0 ? x_scales : nullptr, num_scales,
                                             topk_idx, topk_w, send_pos, recv_base, capacity_rows, recv_x,
                                             num_scales > 0 ? recv_x_scales : nullptr, recv_topk_idx,
                                             recv_topk_w, recv_src_info, status,
                                             reinterpret_cast<unsigned long long*>(sched), stream));
}

ep_status_t ep_combine(const ep_shape_t* shape, const uint16_t* y, const float* y_w,
                       int64_t y_rows, const int32_t* send_pos, const int64_t* recv_base,
                       uint16_t* combined_x, float* combined_w, int32_t* status,
                       cudaStream_t stream) {
    ep::Shape sh;
    if (!ep::make_shape(shape, &sh)) return EP_ERR_INVALID_ARG;
    if (y_rows < 0) return EP_ERR_INVALID_ARG;
    const long long tokens = static_cast<long long>(sh.R) * sh.T;
    // y (and y_w when combined_w is requested) hold y_rows rows; the kernel
    // never reads a row at or beyond y_rows.
    if (!ep::array_ok(y, y_rows * sh.H, 16) || !ep::array_ok(send_pos, tokens * sh.R, 4) ||
        !ep::aligned8(recv_base) || !ep::array_ok(combined_x, tokens * sh.H, 16) ||
        !ep::aligned4(status))
        return EP_ERR_INVALID_ARG;
    if (combined_w != nullptr && !ep::array_ok(y_w, y_rows * sh.K, 4)) return EP_ERR_INVALID_ARG;
    if (!ep::array_ok(combined_w, combined_w ? tokens * sh.K : 0, 4)) return EP_ERR_INVALID_ARG;
    return ep::from_cuda(ep::launch_combine(sh, y, y_w, y_rows, send_pos, recv_base, combined_x,
                                            combined_w, status, stream));
}

ep_status_t ep_ll_layout(const ep_shape_t* shape, const int64_t* topk_idx,
                         const int32_t* num_tokens_per_expert, int32_t expert_capacity,
                         int32_t* slot_pos, int32_t* layout_range, int32_t* count, int32_t* status,
                         cudaStream_t stream) {
    ep::Shape sh;
    if (!ep::make_shape(shape, &sh) || expert_capacity < 0) return EP_ERR_INVALID_ARG;
    const long long tokens = static_cast<long long>(sh.R) * sh.T;
    if (!ep::array_ok(topk_idx, tokens * sh.K, 8) || !ep::array_ok(slot_pos, tokens * sh.K, 4) ||
        !ep::aligned4(layout_range) || !ep::aligned4(count) || !ep::aligned4(status))
        return EP_ERR_INVALID_ARG;
    if (num_tokens_per_expert == nullptr) {  // counting form: one cluster counts for itself
        if (!ep::ll_layout_counting_ok(sh)) return EP_ERR_INVALID_ARG;
        return ep::from_cuda(ep::launch_ll_layout_counting(sh, topk_idx, expert_capacity, slot_pos, layout_range,
                                                           count, status, stream));
    }
    if (!ep::aligned4(num_tokens_per_expert)) return EP_ERR_INVALID_ARG;
    return ep::from_cuda(ep::launch_ll_layout(sh, topk_idx, num_tokens_per_expert, expert_capacity, slot_pos,
                                              layout_range, count, status, stream));
}

ep_status_t ep_ll_dispatch(const ep_shape_t* shape, const uint16_t* x, const int64_t* topk_idx,
                           const int32_t* slot_pos, int32_t expert_capacity, uint16_t* recv_x,
                           int32_t* recv_src_info, int32_t* status, uint64_t* sched, cudaStream_t stream) {
    ep::Shape sh;
    if (!ep::make_shape(shape, &sh) || expert_capacity < 0) return EP_ERR_INVALID_ARG;
    if (sched != nullptr && !ep::aligned8(sched)) return EP_ERR_INVALID_ARG;
    const long long tokens = static_cast<long long>(sh.R) * sh.T;
    const long long rows = static_cast<long long>(sh.E) * expert_capacity;
    if (!ep::array_ok(x, tokens * sh.H, 16) || !ep::array_ok(topk_idx, tokens * sh.K, 8) ||
        !ep::array_ok(slot_pos, tokens * sh.K, 4) || !ep::array_ok(recv_x, rows * sh.H, 16) ||
        (recv_src_info != nullptr && !ep::aligned8(recv_src_info)) || !ep::aligned4(status))
        return EP_ERR_INVALID_ARG;
    return ep::from_cuda(ep::launch_ll_dispatch(sh, x, topk_idx, slot_pos, expert_capacity, recv_x,
                                                recv_src_info, status,
                                                reinterpret_cast<unsigned long long*>(sched), stream));
}

ep_status_t ep_ll_combine(const ep_shape_t* shape, const uint16_t* y, int32_t expert_capacity,
                          const int64_t* topk_idx, const float* topk_w, const int32_t* slot_pos,
                          uint16_t* combined_x, int32_t* status, cudaStream_t stream) {
    ep::Shape sh;
    if (!ep::make_shape(shape, &sh) || expert_capacity < 0) return EP_ERR_INVALID_ARG;
    const long long tokens = static_cast<long long>(sh.R) * sh.T;
    const long long rows = static_cast<long long>(sh.E) * expert_capacity;
    if (!ep::array_ok(y, rows * sh.H, 16) || !ep::array_ok(topk_idx, tokens * sh.K, 8) ||
        !ep::array_ok(topk_w, tokens * sh.K, 4) || !ep::array_ok(slot_pos, tokens * sh.K, 4) ||
        !ep::array_ok(combined_x, tokens * sh.H, 16) || !ep::aligned4(status))
        return EP_ERR_INVALID_ARG;
    return ep::from_cuda(ep::launch_ll_combine(sh, y, expert_capacity, topk_idx, topk_w, slot_pos, combined_x,
                                               status, stream));
}

ep_status_t ep_sync_status(const int32_t* status, cudaStream_t stream) {
    if (!ep::aligned4(status)) return EP_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return EP_ERR_CUDA;
    int32_t h = 0;
    if (cudaMemcpy(&h, status, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return EP_ERR_CUDA;
    if (h & EP_DEV_TIMEOUT) return EP_ERR_TIMEOUT;
    if (h & EP_DEV_CAPACITY) return EP_ERR_CAPACITY;
    if (h & EP_DEV_INPUT) return EP_ERR_INPUT;
    if (h & EP_DEV_INCONSISTENT) return EP_ERR_INCONSISTENT;
    return EP_OK;
}

}  // extern "C"
