// Low-latency (per-expert packed) layout: the row of every top-k slot inside
// its expert's receive buffer.  The pages describe only this mode's transport
// ([RT] "Intra-node LL fast path setup"); the reading implemented here: each
// non-masked slot (s,t,k) naming expert e is one row of e's buffer, rows in
// ascending (source rank, token, slot) order.
//
// One CTA per source rank s.  Its T*K slots, in (t,k) order, are split into
// one contiguous segment per warp.  Pass 1: each warp walks its segment 32
// slots at a time; __match_any_sync groups the lanes naming the same expert,
// and the group's lowest lane adds the group size to the warp's shared
// counter for that expert.  Then, per expert, an exclusive prefix over the
// warps.  Pass 2: each warp rewalks its segment; a slot's row is
// base(s,e) + warp prefix + the lanes of its group below it, and the group's
// lowest lane advances the counter.  base(s,e) = slots that earlier source
// ranks send to e, summed from num_tokens_per_expert.  Deterministic, no
// global atomics, no waits.
//
// Counting form (no num_tokens_per_expert input): the R CTAs form one
// thread-block cluster; after pass 1 each CTA stores its per-expert totals
// into the shared memory of every later source's CTA (distributed shared
// memory), and one cluster barrier later base(s,e) is summed from local
// shared memory.
#include <cooperative_groups.h>

#include "ep_device.cuh"
#include "ep_internal.h"

namespace cg = cooperative_groups;

namespace ep {
namespace {

constexpr int kLlThreads = 1024;
constexpr int kCounterBudget = 48 * 1024;  // shared bytes for the per-warp counters
constexpr int kMaxClusterRanks = 16;
constexpr int kMaxExchangeInts = 16384;    // R * E totals exchanged in the counting form

struct LlLayoutArgs {
    const int64_t* topk_idx;
    const int32_t* num_tokens_per_expert;  // [R][E]
    int32_t* slot_pos;                     // [R][T][K]
    int32_t* layout_range;                 // [E][R][2]
    int32_t* count;                        // [E]
    int32_t* status;
    int R, T, K, E, cap, warps;
};

// kCounting: base(s,e) from the cluster's exchanged totals instead of
// num_tokens_per_expert (grid = one cluster of R CTAs).
template <bool kCounting>
__global__ void __launch_bounds__(kLlThreads, 1) ll_layout_kernel(LlLayoutArgs p) {
    extern __shared__ int32_t cnt[];  // [warps][E], then (counting form) [R][E] totals
    const int s = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int W = p.warps, E = p.E;
    griddep_launch_dependents();
    for (int i = tid; i < W * E; i += blockDim.x) cnt[i] = 0;
    griddep_wait();  // top-k ids and per-expert counts are visible from here on
    __syncthreads();

    const long long items = static_cast<long long>(p.T) * p.K;
    const long long seg = (items + W - 1) / W;
    const long long lo = warp < W ? warp * seg : items;
    const long long hi = lo + seg < items ? lo + seg : items;
    const int64_t* ids = p.topk_idx + static_cast<long long>(s) * items;
    int32_t* my = cnt + warp * E;
    const unsigned lt = lanemask_lt();
    bool bad = false;

    // pass 1: per-warp counts per expert
    if (warp < W) {
        for (long long b = lo; b < hi; b += kWarp) {
            const long long i = b + lane;
            long long e = i < hi ? __ldg(ids + i) : -1;
            if (e < -1 || e >= E) {
                bad = true;
                e = -1;
            }
            const unsigned m = __match_any_sync(0xffffffffu, e);
            if (e >= 0 && (m & lt) == 0u) my[e] += __popc(m);
        }
    }
    __syncthreads();
    // exclusive prefix over warps, per expert; in the counting form this
    // source's totals go to every later source's CTA, one cluster barrier
    // later each CTA holds the totals of all earlier sources
    int32_t* totals = cnt + W * E;  // counting form: [R][E], row s' = totals of source s'
    if (kCounting) {
        cg::cluster_group cluster = cg::this_cluster();
        for (int e = tid; e < E; e += blockDim.x) {
            int32_t run = 0;
            for (int w = 0; w < W; ++w) {
                const int32_t c = cnt[w * E + e];
                cnt[w * E + e] = run;
                run += c;
            }
            totals[s * E + e] = run;
            for (int c = s + 1; c < p.R; ++c) cluster.map_shared_rank(totals, c)[s * E + e] = run;
        }
        cluster.sync();
    }
    // ranges, totals, consistency
    for (int e = tid; e < E; e += blockDim.x) {
        int32_t run = 0, base = 0;
        if (kCounting) {
            run = totals[s * E + e];
            for (int s2 = 0; s2 < s; ++s2) base += totals[s2 * E + e];
        } else {
            for (int w = 0; w < W; ++w) {
                const int32_t c = cnt[w * E + e];
                cnt[w * E + e] = run;
                run += c;
            }
#pragma unroll 8
            for (int s2 = 0; s2 < s; ++s2) base += __ldg(p.num_tokens_per_expert + static_cast<long long>(s2) * E + e);
            if (run != __ldg(p.num_tokens_per_expert + static_cast<long long>(s) * E + e))
                flag_error(p.status, EP_DEV_INCONSISTENT);
        }
        p.layout_range[(static_cast<long long>(e) * p.R + s) * 2 + 0] = base;
        p.layout_range[(static_cast<long long>(e) * p.R + s) * 2 + 1] = run;
        if (s == p.R - 1) p.count[e] = base + run;
        // pass 2 starts every warp's counter at base + its prefix
        for (int w = 0; w < W; ++w) cnt[w * E + e] += base;
    }
    __syncthreads();
    // pass 2: rows
    bool dropped = false;
    if (warp < W) {
        for (long long b = lo; b < hi; b += kWarp) {
            const long long i = b + lane;
            long long e = i < hi ? __ldg(ids + i) : -1;
            if (e < -1 || e >= E) e = -1;
            const unsigned m = __match_any_sync(0xffffffffu, e);
            int32_t row = -1;
            if (e >= 0) {
                row = my[e] + __popc(m & lt);
                if (row >= p.cap) {
                    dropped = true;
                    row = -1;
                }
            }
            __syncwarp();
            if (e >= 0 && (m & lt) == 0u) my[e] += __popc(m);
            __syncwarp();
            if (i < hi) p.slot_pos[static_cast<long long>(s) * items + i] = row;
        }
    }
    if (bad) flag_error(p.status, EP_DEV_INPUT);
    if (dropped) flag_error(p.status, EP_DEV_CAPACITY);
}

}  // namespace

namespace {

int ll_warps(const Shape& sh) {
    const int warps = kCounterBudget / static_cast<int>(sizeof(int32_t) * sh.E);
    return warps < 1 ? 1 : (warps > kLlThreads / kWarp ? kLlThreads / kWarp : warps);
}

LlLayoutArgs ll_args(const Shape& sh, const int64_t* topk_idx, const int32_t* num_tokens_per_expert, int cap,
                     int32_t* slot_pos, int32_t* layout_range, int32_t* count, int32_t* status) {
    LlLayoutArgs p;
    p.topk_idx = topk_idx;
    p.num_tokens_per_expert = num_tokens_per_expert;
    p.slot_pos = slot_pos;
    p.layout_range = layout_range;
    p.count = count;
    p.status = status;
    p.R = sh.R;
    p.T = sh.T;
    p.K = sh.K;
    p.E = sh.E;
    p.cap = cap;
    p.warps = ll_warps(sh);
    return p;
}

size_t ll_counting_smem(const Shape& sh) {
    return sizeof(int32_t) * (static_cast<size_t>(ll_warps(sh)) + sh.R) * sh.E;
}

}  // namespace

cudaError_t launch_ll_layout(const Shape& sh, const int64_t* topk_idx, const int32_t* num_tokens_per_expert,
                             int cap, int32_t* slot_pos, int32_t* layout_range, int32_t* count,
                             int32_t* status, cudaStream_t stream) {
    const LlLayoutArgs p = ll_args(sh, topk_idx, num_tokens_per_expert, cap, slot_pos, layout_range, count, status);
    const size_t smem = sizeof(int32_t) * static_cast<size_t>(p.warps) * sh.E;
    return launch_pdl(ll_layout_kernel<false>, dim3(sh.R), dim3(kLlThreads), smem, stream, 0, false, p);
}

bool ll_layout_counting_ok(const Shape& sh) {
    if (sh.R > kMaxClusterRanks || static_cast<long long>(sh.R) * sh.E > kMaxExchangeInts) return false;
    return cluster_fits(reinterpret_cast<const void*>(ll_layout_kernel<true>), sh.R, kLlThreads,
                        ll_counting_smem(sh));
}

cudaError_t launch_ll_layout_counting(const Shape& sh, const int64_t* topk_idx, int cap, int32_t* slot_pos,
                                      int32_t* layout_range, int32_t* count, int32_t* status,
                                      cudaStream_t stream) {
    const LlLayoutArgs p = ll_args(sh, topk_idx, nullptr, cap, slot_pos, layout_range, count, status);
    return launch_pdl(ll_layout_kernel<true>, dim3(sh.R), dim3(kLlThreads), ll_counting_smem(sh), stream,
                      static_cast<unsigned>(sh.R), false, p);
}

}  // namespace ep
