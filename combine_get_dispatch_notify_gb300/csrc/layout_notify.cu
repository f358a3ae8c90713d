// Steps 1 and 2 in one launch: layout counting ([RT] getDispatchLayout; the
// count vectors of [IN] notify_dispatch sm0 stage 3) followed by the notify
// prefix sums ([IN] sm1..x stages 1-3 and sm0 stage 6; [RT]
// intranode/internodeNotifyDispatch).  Same outputs as the two separate
// kernels.
//
// One thread-block cluster of R CTAs; CTA s owns source rank s and, for the
// per-destination results, destination rank s.  Every phase spreads its
// items over all threads of the CTA (up to 1024), so that the latencies of
// one thread's steps overlap with the other warps' work.
//   A. One thread per (token, pair of top-k slots): the ids go into a shared
//      expert histogram and their destination ranks into the token's mask
//      (shared atomicOr).  Then one warp per 32-token block writes the
//      is_token_in_rank rows and stores one ballot word per destination rank
//      and per node: bit t%32 of ballot (t/32, v) says whether token t goes
//      to v.  Nothing else about a token is kept.
//   B. One warp per value v scans the ballots' popcounts into an exclusive
//      prefix per 32-token block and the source total (the layout counts).
//   C. Every CTA stores its totals into each CTA's shared memory, and the
//      counts of the experts living on rank d into CTA d's, through
//      distributed shared memory (remote stores, nothing waits on them); one
//      cluster barrier later each CTA holds every source's totals and the
//      per-source counts of its own experts, and computes from local shared
//      memory the rows earlier sources send to each destination (rank
//      prefix matrix), the column sums (receive counts, recv_base), the
//      node-level prefix and its experts' totals.
//   D. The channel prefix matrices and send_pos follow from the ballots in
//      O(1) per element: the prefix of v before token t is the block prefix
//      plus the popcount of the ballot bits below t.  send_pos is written in
//      16-byte stores, fully coalesced.
// No global atomics, no workspace and no inter-CTA waits other than the one
// cluster barrier, which the hardware completes once every CTA of the
// cluster has arrived (all of them are co-scheduled).  Counts come from the
// same pass that builds is_token_in_rank, so they cannot disagree.
#include <cooperative_groups.h>

#include "ep_device.cuh"
#include "ep_internal.h"

namespace cg = cooperative_groups;

namespace ep {
namespace {

constexpr int kMaxThreads = 1024;
constexpr int kMinThreads = 256;
constexpr int kMaxRanks = 16;     // the cluster holds one CTA per rank
constexpr int kMaxTokens = 8192;  // ballots of one source stay in shared memory

struct LayoutNotifyArgs {
    const int64_t* topk_idx;
    int32_t* num_tokens_per_rank;
    int32_t* num_tokens_per_rdma_rank;
    int32_t* num_tokens_per_expert;
    uint8_t* is_token_in_rank;
    NotifyArgs a;  // outputs of the notify step (its count-input fields are unused)
    int R, T, K, E, N, E_loc, C, q, align, V, J;
    uint32_t eloc_magic;  // ceil(2^32 / E_loc): e / E_loc = umulhi(e, magic) for e < 8192, E_loc >= 2
};

// Tokens of this source routed to value v (rank, or node R+n) before token t.
__device__ __forceinline__ int32_t prefix_before(const uint32_t* bal, const int32_t* pre,
                                                 const int32_t* tot, int V, int T, int v, int t) {
    if (t >= T) return tot[v];
    const int j = t >> 5;
    return pre[j * V + v] + __popc(bal[j * V + v] & ((1u << (t & 31)) - 1u));
}

// One expert id: histogram and rank bit.  An id outside [-1, E) sets `bad`.
__device__ __forceinline__ void add_expert(const LayoutNotifyArgs& p, long long e, int32_t* hist,
                                           uint32_t& mask, bool& bad) {
    if (e >= 0 && e < p.E) {
        const uint32_t u = static_cast<uint32_t>(e);
        mask |= 1u << (p.E_loc == 1 ? u : __umulhi(u, p.eloc_magic));
        atomicAdd(&hist[u], 1);
    } else if (e != -1) {
        bad = true;
    }
}

__global__ void __launch_bounds__(kMaxThreads) layout_notify_kernel(LayoutNotifyArgs p) {
    // [E] expert histogram | [R][V] every source's totals | [R][E_loc] every
    // source's counts of this rank's experts | [32] cross-source offsets |
    // [T] token masks | [J][V] ballots | [J][V] exclusive block prefixes
    extern __shared__ __align__(16) int32_t smem[];
    cg::cluster_group cluster = cg::this_cluster();
    const int R = p.R, T = p.T, K = p.K, E = p.E, N = p.N, V = p.V, J = p.J, C = p.C, E_loc = p.E_loc;
    const int s = static_cast<int>(blockIdx.x);  // grid = one cluster, CTA s = source s
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = static_cast<int>(blockDim.x), warps = B >> 5;
    int32_t* hist = smem;
    int32_t* all_tot = hist + E;
    int32_t* my_experts = all_tot + R * V;
    int32_t* cross = my_experts + R * E_loc;
    uint32_t* tmask = reinterpret_cast<uint32_t*>(cross + 32);
    uint32_t* bal = tmask + T;
    int32_t* pre = reinterpret_cast<int32_t*>(bal + J * V);
    int32_t* tot = all_tot + s * V;  // this source's totals

    griddep_launch_dependents();
    for (int i = tid; i < E; i += B) hist[i] = 0;
    for (int i = tid; i < T; i += B) tmask[i] = 0u;
    griddep_wait();  // top-k ids written by the preceding kernel are visible
    const int64_t* ids = p.topk_idx + static_cast<int64_t>(s) * T * K;
    const int P2 = (K + 1) >> 1;  // pairs of slots per token
    if (tid == 0 && T * P2 > B) prefetch_l2(ids, static_cast<size_t>(T) * K * sizeof(int64_t));
    __syncthreads();

    // A1. thread per (token, pair of slots): histogram and the token's rank mask
    bool bad = false;
    {
        const int pk = tid % P2, tpi = B / P2;  // tokens per sweep of the CTA
        if (tid < tpi * P2) {
            if ((K & 1) == 0) {
                const longlong2* ids2 = reinterpret_cast<const longlong2*>(ids);
                for (int t = tid / P2; t < T; t += tpi) {
                    const longlong2 e2 = __ldg(ids2 + static_cast<int64_t>(t) * P2 + pk);
                    uint32_t m = 0;
                    add_expert(p, e2.x, hist, m, bad);
                    add_expert(p, e2.y, hist, m, bad);
                    if (m) atomicOr(&tmask[t], m);
                }
            } else {
                for (int t = tid / P2; t < T; t += tpi) {
                    const int64_t* row = ids + static_cast<int64_t>(t) * K + 2 * pk;
                    const long long e0 = __ldg(row);
                    const long long e1 = 2 * pk + 1 < K ? __ldg(row + 1) : -1;
                    uint32_t m = 0;
                    add_expert(p, e0, hist, m, bad);
                    add_expert(p, e1, hist, m, bad);
                    if (m) atomicOr(&tmask[t], m);
                }
            }
        }
    }
    if (bad) flag_error(p.a.status, EP_DEV_INPUT);
    __syncthreads();

    // A2. warp per 32-token block: membership rows and one ballot per value
    for (int j = warp; j < J; j += warps) {
        const int t = j * kWarp + lane;
        const uint32_t mask = t < T ? tmask[t] : 0u;
        if (t < T) write_membership_row(p.is_token_in_rank + (static_cast<int64_t>(s) * T + t) * R, mask, R);
        const uint32_t bits = mask | (node_bits(mask, R, N) << R);
        for (int v = 0; v < V; ++v) {
            const unsigned b = __ballot_sync(0xffffffffu, (bits >> v) & 1u);
            if (lane == v) bal[j * V + v] = b;
        }
    }
    __syncthreads();

    // B. exclusive prefix over 32-token blocks, per value; lane L takes a run
    //    of consecutive blocks
    const int per = (J + kWarp - 1) / kWarp;
    for (int v = warp; v < V; v += warps) {
        const int j0 = min(lane * per, J), j1 = min(j0 + per, J);
        int32_t sum = 0;
        for (int j = j0; j < j1; ++j) sum += __popc(bal[j * V + v]);
        int32_t inc = sum;
#pragma unroll
        for (int o = 1; o < kWarp; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        int32_t run = inc - sum;
        for (int j = j0; j < j1; ++j) {
            pre[j * V + v] = run;
            run += __popc(bal[j * V + v]);
        }
        if (lane == kWarp - 1) tot[v] = inc;
    }
    __syncthreads();

    // C. exchange: totals to every CTA, expert counts to the experts' rank
    for (int i = tid; i < R * V; i += B) {
        const int c = i / V, v = i - c * V;
        if (c != s) cluster.map_shared_rank(all_tot, c)[s * V + v] = tot[v];
    }
    for (int e = tid; e < E; e += B) {
        const int d = E_loc == 1 ? e : static_cast<int>(__umulhi(static_cast<uint32_t>(e), p.eloc_magic));
        cluster.map_shared_rank(my_experts, d)[s * E_loc + (e - d * E_loc)] = hist[e];
    }
    cluster.sync();  // every CTA's stores into this CTA's shared memory are visible

    // layout counts of source s; cross-source results from local shared memory
    for (int i = tid; i < E; i += B) p.num_tokens_per_expert[static_cast<int64_t>(s) * E + i] = hist[i];
    if (tid < R) {
        const int r = tid;
        p.num_tokens_per_rank[static_cast<int64_t>(s) * R + r] = tot[r];
        int32_t before = 0;  // rows that earlier source ranks send to r
        for (int s2 = 0; s2 < s; ++s2) before += all_tot[s2 * V + r];
        cross[r] = before;
        p.a.rank_prefix_matrix[static_cast<int64_t>(s) * R + r] = before + tot[r];
        p.a.recv_gbl_rank_prefix_sum[static_cast<int64_t>(r) * R + s] = before + tot[r];
    } else if (tid < V) {
        p.num_tokens_per_rdma_rank[static_cast<int64_t>(s) * N + (tid - R)] = tot[tid];
    }
    const int d = s;  // this CTA also writes the results of destination rank d
    if (warp == 1) {
        // lane r: rows rank r receives from all sources; recv_base[d] is the
        // sum over lanes below d
        int32_t col = 0;
        if (lane < R)
            for (int s2 = 0; s2 < R; ++s2) col += all_tot[s2 * V + lane];
        int32_t inc = col;
#pragma unroll
        for (int o = 1; o < kWarp; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        if (lane == d) {
            p.a.num_recv_tokens[d] = col;
            p.a.recv_base[d] = inc - col;
            if (p.a.host_num_recv_tokens) p.a.host_num_recv_tokens[d] = col;
        }
        if (d == R - 1 && lane == R - 1) {
            p.a.recv_base[R] = inc;
            if (p.a.host_num_recv_tokens) p.a.host_num_recv_tokens[R] = inc;
        }
        if (p.a.host_num_recv_tokens) __threadfence_system();
    } else if (warp == 2 && lane == 0) {
        // node-level receive prefix: d receives for its node from the
        // same-GPU-index peer m*8 + d%8 of every node m
        int32_t run = 0;
        for (int m = 0; m < N; ++m) {
            run += all_tot[(m * kNodeSize + d % kNodeSize) * V + R + d / kNodeSize];
            p.a.recv_rdma_rank_prefix_sum[static_cast<int64_t>(d) * N + m] = run;
        }
        p.a.num_rdma_recv_tokens[d] = run;
    }
    // per-expert totals of the experts on rank d, rounded up to the alignment
    for (int i = tid; i < E_loc; i += B) {
        long long sum = 0;
        for (int s2 = 0; s2 < R; ++s2) sum += my_experts[s2 * E_loc + i];
        sum = (sum + p.align - 1) / p.align * p.align;
        p.a.num_recv_tokens_per_expert[d * E_loc + i] = static_cast<int32_t>(sum);
    }
    __syncthreads();  // cross[] is complete

    // D. channel prefix matrices and receive offsets of source s
    for (int i = tid; i < V * C; i += B) {
        const int v = i / C, c = i - v * C;
        const int ta = static_cast<int>(min(static_cast<long long>(c) * p.q, static_cast<long long>(T)));
        const int tb = min(ta + p.q, T);
        const int32_t incl = prefix_before(bal, pre, tot, V, T, v, tb);
        if (v < R) {
            p.a.gbl_channel_prefix_matrix[(static_cast<int64_t>(s) * R + v) * C + c] = incl;
            p.a.recv_channel_offset[(static_cast<int64_t>(v) * R + s) * C + c] =
                cross[v] + prefix_before(bal, pre, tot, V, T, v, ta);
        } else {
            p.a.rdma_channel_prefix_matrix[(static_cast<int64_t>(s) * N + (v - R)) * C + c] = incl;
        }
    }
    // send_pos[s][t][r]: row of (s,t) inside r's region, or -1; thread per
    // (token, 4 ranks), one 16-byte store each
    int32_t* send_pos = p.a.send_pos + static_cast<int64_t>(s) * T * R;
    if ((R & 3) == 0) {
        const int qpt = R >> 2, tpi = B / qpt;
        const int r0 = (tid % qpt) * 4;
        if (tid < tpi * qpt) {
            for (int t = tid / qpt; t < T; t += tpi) {
                const int j = t >> 5;
                const uint32_t bit = 1u << (t & 31), below = bit - 1u;
                int32_t o[4];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const uint32_t b = bal[j * V + r0 + h];
                    o[h] = (b & bit) ? cross[r0 + h] + pre[j * V + r0 + h] + __popc(b & below) : -1;
                }
                *reinterpret_cast<int4*>(send_pos + static_cast<int64_t>(t) * R + r0) =
                    make_int4(o[0], o[1], o[2], o[3]);
            }
        }
    } else {
        for (int i = tid; i < T * R; i += B) {
            const int t = i / R, r = i - t * R;
            const int j = t >> 5;
            const uint32_t bit = 1u << (t & 31);
            const uint32_t b = bal[j * V + r];
            send_pos[i] = (b & bit) ? cross[r] + pre[j * V + r] + __popc(b & (bit - 1u)) : -1;
        }
    }
}

size_t fused_smem_bytes(const Shape& sh) {
    const size_t V = static_cast<size_t>(sh.R + sh.N);
    const size_t J = (static_cast<size_t>(sh.T) + kWarp - 1) / kWarp;
    return sizeof(int32_t) *
           (static_cast<size_t>(sh.E) + sh.R * V + static_cast<size_t>(sh.E) + 32 + sh.T + 2 * J * V);
}

// Threads: one per (token, pair of slots), a multiple of 32 within [256, 1024].
int fused_threads(const Shape& sh) {
    const long long items = static_cast<long long>(sh.T) * ((sh.K + 1) / 2);
    long long b = (items + kWarp - 1) / kWarp * kWarp;
    return static_cast<int>(b < kMinThreads ? kMinThreads : (b > kMaxThreads ? kMaxThreads : b));
}

}  // namespace

bool layout_notify_fused_ok(const Shape& sh) {
    if (sh.R > kMaxRanks || sh.T > kMaxTokens) return false;
    return cluster_fits(reinterpret_cast<const void*>(layout_notify_kernel), sh.R, fused_threads(sh),
                        fused_smem_bytes(sh));
}

cudaError_t launch_layout_notify(const Shape& sh, const int64_t* topk_idx, int32_t* num_tokens_per_rank,
                                 int32_t* num_tokens_per_rdma_rank, int32_t* num_tokens_per_expert,
                                 uint8_t* is_token_in_rank, const NotifyArgs& a, cudaStream_t stream) {
    LayoutNotifyArgs p;
    p.topk_idx = topk_idx;
    p.num_tokens_per_rank = num_tokens_per_rank;
    p.num_tokens_per_rdma_rank = num_tokens_per_rdma_rank;
    p.num_tokens_per_expert = num_tokens_per_expert;
    p.is_token_in_rank = is_token_in_rank;
    p.a = a;
    p.R = sh.R;
    p.T = sh.T;
    p.K = sh.K;
    p.E = sh.E;
    p.N = sh.N;
    p.E_loc = sh.E_loc;
    p.C = sh.C;
    p.q = (sh.T + sh.C - 1) / sh.C;
    p.align = sh.align;
    p.V = sh.R + sh.N;
    p.J = (sh.T + kWarp - 1) / kWarp;
    p.eloc_magic = sh.E_loc >= 2 ? static_cast<uint32_t>(((1ull << 32) + sh.E_loc - 1) / sh.E_loc) : 0u;
    return launch_pdl(layout_notify_kernel, dim3(static_cast<unsigned>(sh.R)), dim3(fused_threads(sh)),
                      fused_smem_bytes(sh), stream, static_cast<unsigned>(sh.R), false, p);
}

}  // namespace ep
