// Step 1 - layout counting ([RT] getDispatchLayout; count vectors of [IN]
// notify_dispatch sm0 stage 3).
//
// One thread-block cluster per source rank s.  The cluster's CTAs split s's
// tokens; each thread takes one token, reads its K expert ids, builds the
// R-bit destination mask, writes the is_token_in_rank row, and adds to
// shared-memory histograms (experts by smem atomics, ranks and nodes by warp
// ballot + popc).  CTA 0 of the cluster then sums the CTAs' histograms
// through distributed shared memory and writes the counts - no global
// atomics and no pre-zeroed outputs.
#include <cooperative_groups.h>

#include "ep_device.cuh"
#include "ep_internal.h"

namespace cg = cooperative_groups;

namespace ep {
namespace {

constexpr int kLayoutThreads = 256;
constexpr int kMaxClusterCtas = 8;       // portable cluster size
constexpr int kTokensPerCtaTarget = 1024;

__global__ void __launch_bounds__(kLayoutThreads)
layout_kernel(const int64_t* __restrict__ topk_idx, int R, int T, int K, int E, int N, int E_loc,
              int tokens_per_cta, int32_t* __restrict__ num_tokens_per_rank,
              int32_t* __restrict__ num_tokens_per_rdma_rank,
              int32_t* __restrict__ num_tokens_per_expert, uint8_t* __restrict__ is_token_in_rank,
              int32_t* status) {
    extern __shared__ int32_t hist[];  // [E] experts | [R] ranks | [N] nodes
    cg::cluster_group cluster = cg::this_cluster();
    const int part = static_cast<int>(cluster.block_rank());
    const int parts = static_cast<int>(cluster.num_blocks());
    const int s = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31;
    const int bins = E + R + N;
    int32_t* h_expert = hist;
    int32_t* h_rank = hist + E;
    int32_t* h_node = h_rank + R;
    griddep_launch_dependents();
    for (int i = tid; i < bins; i += blockDim.x) hist[i] = 0;
    griddep_wait();  // top-k ids written by the preceding kernel are visible
    __syncthreads();

    const int t_begin = min(T, part * tokens_per_cta);
    const int t_end = min(T, t_begin + tokens_per_cta);
    int rank_acc = 0, node_acc = 0;  // lane r (lane n) accumulates rank r (node n)
    bool bad = false;
    for (int base = t_begin; base < t_end; base += blockDim.x) {
        const int t = base + tid;
        uint32_t mask = 0;
        if (t < t_end) {
            mask = token_rank_mask(topk_idx + (static_cast<int64_t>(s) * T + t) * K, K, E, E_loc, h_expert, bad);
            write_membership_row(is_token_in_rank + (static_cast<int64_t>(s) * T + t) * R, mask, R);
        }
        const uint32_t node_mask = node_bits(mask, R, N);
        for (int r = 0; r < R; ++r) {
            const unsigned b = __ballot_sync(0xffffffffu, (mask >> r) & 1u);
            if (lane == r) rank_acc += __popc(b);
        }
        for (int n = 0; n < N; ++n) {
            const unsigned b = __ballot_sync(0xffffffffu, (node_mask >> n) & 1u);
            if (lane == n) node_acc += __popc(b);
        }
    }
    if (lane < R && rank_acc) atomicAdd(&h_rank[lane], rank_acc);
    if (lane < N && node_acc) atomicAdd(&h_node[lane], node_acc);
    if (bad) flag_error(status, EP_DEV_INPUT);

    if (parts > 1)
        cluster.sync();  // every CTA's partial histogram is complete and visible
    else
        __syncthreads();
    if (part == 0) {
        for (int i = tid; i < bins; i += blockDim.x) {
            int32_t sum = 0;
            for (int j = 0; j < parts; ++j) sum += cluster.map_shared_rank(hist, j)[i];
            if (i < E)
                num_tokens_per_expert[static_cast<int64_t>(s) * E + i] = sum;
            else if (i < E + R)
                num_tokens_per_rank[static_cast<int64_t>(s) * R + (i - E)] = sum;
            else
                num_tokens_per_rdma_rank[static_cast<int64_t>(s) * N + (i - E - R)] = sum;
        }
    }
    if (parts > 1) cluster.sync();  // keep every histogram alive until CTA 0 has read it
}

}  // namespace

cudaError_t launch_layout(const Shape& sh, const int64_t* topk_idx, int32_t* num_tokens_per_rank,
                          int32_t* num_tokens_per_rdma_rank, int32_t* num_tokens_per_expert,
                          uint8_t* is_token_in_rank, int32_t* status, cudaStream_t stream) {
    int parts = (sh.T + kTokensPerCtaTarget - 1) / kTokensPerCtaTarget;
    parts = parts < 1 ? 1 : (parts > kMaxClusterCtas ? kMaxClusterCtas : parts);
    const int tokens_per_cta = (sh.T + parts - 1) / parts;
    const size_t smem = sizeof(int32_t) * static_cast<size_t>(sh.E + sh.R + sh.N);
    return launch_pdl(layout_kernel, dim3(parts, sh.R, 1), dim3(kLayoutThreads, 1, 1), smem, stream,
                      static_cast<unsigned>(parts), false, topk_idx, sh.R, sh.T, sh.K, sh.E, sh.N, sh.E_loc,
                      tokens_per_cta, num_tokens_per_rank, num_tokens_per_rdma_rank,
                      num_tokens_per_expert, is_token_in_rank, status);
}

}  // namespace ep
