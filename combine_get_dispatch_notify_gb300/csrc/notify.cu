// Step 2 - notify prefix sums ([IN] notify_dispatch: sm1..x stages 1-3 and
// sm0 stage 6; [RT] intranode/internodeNotifyDispatch for names and shapes).
//
// Grid = 1 + R*C CTAs, roles taken from an atomic ticket in launch order:
//   ticket 0      the per-rank results, which depend only on the exchanged
//                 counts ([IN] sm0 stage 6): rank prefix matrix and its
//                 transpose, receive counts, node-level prefix, per-expert
//                 totals rounded up to the alignment, recv_base;
//   ticket 1+b    block b = (source rank s, channel c), in (s, c) order:
//     1. count the channel's tokens per destination rank and per node (warp
//        ballot + popc) - [IN] sm1..x stage 1;
//     2. get the exclusive within-source prefix (channel prefix matrices,
//        [IN] stages 2-3): for small sources by recounting the earlier
//        channels of the source directly (no block waits on another, roles
//        come from blockIdx); otherwise publish the aggregate and look back
//        over the earlier channels of the same source (decoupled lookback,
//        one warp per value reading 32 predecessors per probe);
//     3. start row of the block in destination r's region = tokens every
//        earlier source rank sends to r (summed from num_tokens_per_rank, as
//        the pages' notify derives receive offsets from exchanged counts) +
//        the within-source prefix; then rewalk the channel and write
//        send_pos = start + running index, staged through shared memory so
//        the global writes are coalesced.
// The last channel of each source checks that its totals equal the count
// inputs (EP_DEV_INCONSISTENT otherwise).  A block waits only on blocks with
// smaller tickets, which are already running; every wait gives up after a
// deadline and sets EP_DEV_TIMEOUT.
#include <mutex>

#include "ep_device.cuh"
#include "ep_internal.h"

// Fixed scratch for ep_notify_dispatch_noalloc, for callers that cannot
// allocate device memory.  Every GPU that loads the library holds these
// bytes until the process exits.  All calls share it.
static __device__ __align__(256) unsigned char g_notify_noalloc_scratch[ep::kNoAllocScratchBytes];

namespace ep {
namespace {

constexpr int kNotifyThreads = 256;
constexpr int kNotifyWarps = kNotifyThreads / kWarp;
constexpr int kWorkspaceHeader = 256;  // ticket word, padded

// Workspace state survives between calls, so no call has to clear it (only
// a fresh workspace must be zero).  The 64-bit ticket word holds [63:32] the
// sequence number of the last completed call and [31:0] the tickets taken by
// the running call; the block that takes the last ticket stores the next
// sequence number with a zero count.  Lookback words carry the sequence
// number of the call that wrote them, so words left by earlier calls read as
// "not yet published":  [63:32] sequence, [31:30] flag, [29:0] value.
constexpr unsigned kFlagAggregate = 1u;
constexpr unsigned kFlagPrefix = 2u;
constexpr unsigned long long kValMask = (1ull << 30) - 1;

__device__ __forceinline__ unsigned long long pack_word(unsigned seq, unsigned flag, uint32_t val) {
    return (static_cast<unsigned long long>(seq) << 32) | (static_cast<unsigned long long>(flag) << 30) |
           (static_cast<unsigned long long>(val) & kValMask);
}
__device__ __forceinline__ unsigned word_seq(unsigned long long w) { return static_cast<unsigned>(w >> 32); }
__device__ __forceinline__ unsigned word_flag(unsigned long long w) {
    return static_cast<unsigned>((w >> 30) & 3u);
}
__device__ __forceinline__ uint32_t word_val(unsigned long long w) {
    return static_cast<uint32_t>(w & kValMask);
}

struct NotifyKernelArgs {
    NotifyArgs a;
    unsigned long long* ticket; // see the workspace state note above
    unsigned long long* words; // [R*C][V], V = R + N values per block
    int R, T, E, C, N, E_loc, align, q, V;
    int recount;  // 1: recount earlier channels of the source instead of looking back
    int stall_block;
    long long wait_limit_ns;
};

// Nonzero bytes of a little-endian word -> 4 bits.
__device__ __forceinline__ uint32_t bytes_to_bits4(uint32_t x) {
    x = __vcmpne4(x, 0u);
    return (x & 1u) | ((x >> 7) & 2u) | ((x >> 14) & 4u) | ((x >> 21) & 8u);
}

// Token row of is_token_in_rank (R bytes) -> R-bit mask.
__device__ __forceinline__ uint32_t load_mask(const uint8_t* row, int R) {
    uint32_t m = 0;
    if ((R & 15) == 0) {
        for (int w = 0; w < R / 16; ++w) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(row + 16 * w));
            m |= (bytes_to_bits4(v.x) | (bytes_to_bits4(v.y) << 4) | (bytes_to_bits4(v.z) << 8) |
                  (bytes_to_bits4(v.w) << 12))
                 << (16 * w);
        }
    } else if ((R & 3) == 0) {
        for (int w = 0; w < R / 4; ++w)
            m |= bytes_to_bits4(__ldg(reinterpret_cast<const uint32_t*>(row + 4 * w))) << (4 * w);
    } else {
        for (int r = 0; r < R; ++r) m |= (__ldg(row + r) != 0 ? 1u : 0u) << r;
    }
    return m;
}

// Ticket 0: the per-rank results ([IN] sm0 stage 6), from the count inputs
// only.  All inputs are loaded up front by many threads, then summed.
__device__ void per_rank_results(const NotifyKernelArgs& p, int32_t* s_nrecv,
                                 int32_t (*s_ntpr)[33]) {
    const NotifyArgs& a = p.a;
    const int R = p.R, N = p.N, tid = threadIdx.x;
    for (int i = tid; i < R * R; i += blockDim.x) s_ntpr[i / R][i % R] = __ldg(a.num_tokens_per_rank + i);
    // per-expert receive counts (expert e = r * E_loc + j), rounded up to the alignment
    for (int e = tid; e < p.E; e += blockDim.x) {
        long long sum = 0;
#pragma unroll 8
        for (int s = 0; s < R; ++s) sum += __ldg(a.num_tokens_per_expert + static_cast<int64_t>(s) * p.E + e);
        sum = (sum + p.align - 1) / p.align * p.align;
        a.num_recv_tokens_per_expert[e] = static_cast<int32_t>(sum);
    }
    // node-level receive prefix: rank r receives for its node from the
    // same-GPU-index peer m*8 + r%8 of every node m
    for (int r = tid; r < R; r += blockDim.x) {
        int32_t run = 0;
        for (int m = 0; m < N; ++m) {
            const int peer = m * kNodeSize + r % kNodeSize;
            run += __ldg(a.num_tokens_per_rdma_rank + static_cast<int64_t>(peer) * N + r / kNodeSize);
            a.recv_rdma_rank_prefix_sum[static_cast<int64_t>(r) * N + m] = run;
        }
        a.num_rdma_recv_tokens[r] = run;
    }
    __syncthreads();
    // prefix of per-rank counts over global source rank
    for (int r = tid; r < R; r += blockDim.x) {
        int32_t run = 0;
        for (int s = 0; s < R; ++s) {
            run += s_ntpr[s][r];
            a.rank_prefix_matrix[static_cast<int64_t>(s) * R + r] = run;
            a.recv_gbl_rank_prefix_sum[static_cast<int64_t>(r) * R + s] = run;
        }
        a.num_recv_tokens[r] = run;
        s_nrecv[r] = run;
    }
    __syncthreads();
    if (tid == 0) {
        long long acc = 0;
        a.recv_base[0] = 0;
        for (int r = 0; r < R; ++r) {
            acc += s_nrecv[r];
            a.recv_base[r + 1] = acc;
            if (a.host_num_recv_tokens) a.host_num_recv_tokens[r] = s_nrecv[r];
        }
        if (a.host_num_recv_tokens) {
            a.host_num_recv_tokens[R] = static_cast<int32_t>(acc);
            __threadfence_system();
        }
    }
}

// Exclusive prefix of value v over blocks [seg_lo, b) (one warp).  Lanes read
// 32 predecessors at once; the nearest published inclusive prefix ends the
// walk, and the segment start acts as one with value 0.
// A thread's waits share one deadline, set by the first of them that keeps
// polling (0 until then: a block whose words are all there reads no timer).
__device__ __forceinline__ bool notify_wait_expired(long long& deadline, long long limit_ns) {
    const long long now = globaltimer_ns();
    if (deadline == 0) {
        deadline = now + limit_ns;
        return false;
    }
    return now > deadline;
}

__device__ uint32_t segment_lookback(const NotifyKernelArgs& p, unsigned seq, int b, int seg_lo, int v,
                                     int lane, long long& deadline, bool& timed_out) {
    uint32_t excl = 0;
    for (int j0 = b - 1; j0 >= seg_lo; j0 -= kWarp) {
        const int j = j0 - lane;
        unsigned long long word = pack_word(seq, kFlagPrefix, 0);
        if (j >= seg_lo) {
            const unsigned long long* w = p.words + static_cast<int64_t>(j) * p.V + v;
            word = ld_relaxed_u64(w);
            uint32_t polls = 0;
            while (word_seq(word) != seq) {  // not yet published by this call
                if ((++polls & 15u) == 0 && notify_wait_expired(deadline, p.wait_limit_ns)) {
                    timed_out = true;
                    word = pack_word(seq, kFlagPrefix, 0);
                    break;
                }
                __nanosleep(32);
                word = ld_relaxed_u64(w);
            }
        }
        const unsigned pm = __ballot_sync(0xffffffffu, word_flag(word) == kFlagPrefix);
        const uint32_t val = word_val(word);
        if (pm != 0u) {
            const int k = __ffs(pm) - 1;
            excl += __reduce_add_sync(0xffffffffu, lane <= k ? val : 0u);
            break;
        }
        excl += __reduce_add_sync(0xffffffffu, val);
    }
    return excl;
}

__global__ void __launch_bounds__(kNotifyThreads) notify_kernel(NotifyKernelArgs p) {
    extern __shared__ int32_t tile[];  // [kNotifyThreads][R + 1] send_pos staging
    __shared__ int s_ticket;
    __shared__ unsigned s_seq;
    __shared__ int32_t s_ntpr[32][33];
    __shared__ int32_t s_count[64];    // block totals: ranks, then nodes
    __shared__ int32_t s_segex[64];    // exclusive within-source prefix per value
    __shared__ int32_t s_start[32];    // start row of this block in each region
    __shared__ int32_t s_run[32];      // running count inside the channel
    __shared__ int32_t s_warp[kNotifyWarps][33];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int R = p.R, N = p.N, C = p.C, V = p.V, T = p.T;
    griddep_launch_dependents();
    griddep_wait();  // the layout outputs are complete from here on
    if (p.recount) {  // no block waits on another: roles straight from blockIdx
        if (tid == 0) {
            s_ticket = static_cast<int>(blockIdx.x);
            s_seq = 0u;
        }
    } else if (tid == 0) {
        const unsigned long long old = atomicAdd(p.ticket, 1ull);
        const unsigned taken = static_cast<unsigned>(old & 0xffffffffull);
        const unsigned seq = static_cast<unsigned>(old >> 32) + 1u;
        if (taken == gridDim.x - 1u)  // last ticket of this call: arm the next call
            atomicExch(p.ticket, static_cast<unsigned long long>(seq) << 32);
        if (taken >= gridDim.x) flag_error(p.a.status, EP_DEV_INCONSISTENT);  // workspace not zeroed
        s_ticket = taken < gridDim.x ? static_cast<int>(taken) : -1;
        s_seq = seq;
    }
    if (tid < 64) {
        s_count[tid] = 0;
        s_segex[tid] = 0;
    }
    if (tid < 32) s_run[tid] = 0;
    __syncthreads();
    if (s_ticket < 0) return;
    const unsigned seq = s_seq;
    if (s_ticket == 0) {
        per_rank_results(p, s_run, s_ntpr);
        return;
    }
    const int b = s_ticket - 1, s = b / C, c = b % C;
    const int t0 = min(c * p.q, T), t1 = min(t0 + p.q, T);
    const uint8_t* in_rank = p.a.is_token_in_rank + static_cast<int64_t>(s) * T * R;

    // tokens every earlier source rank sends to r (independent loads, issued early)
    int32_t cross = 0;
    if (tid < R) {
#pragma unroll 8
        for (int s2 = 0; s2 < s; ++s2) cross += __ldg(p.a.num_tokens_per_rank + static_cast<int64_t>(s2) * R + tid);
    }

    if (p.recount) {
        // 1'+2'. small sources: count the channel (-> s_count) and, directly,
        //        every earlier channel of the same source (-> s_segex)
        int pre_r = 0, agg_r = 0, pre_n = 0, agg_n = 0;
        for (int base = 0; base < t1; base += kNotifyThreads) {
            const int t = base + tid;
            const uint32_t m = t < t1 ? load_mask(in_rank + static_cast<int64_t>(t) * R, R) : 0u;
            const uint32_t mp = t < t0 ? m : 0u, ma = t < t0 ? 0u : m;
            const uint32_t nmp = node_bits(mp, R, N), nma = node_bits(ma, R, N);
            for (int r = 0; r < R; ++r) {
                const unsigned bp = __ballot_sync(0xffffffffu, (mp >> r) & 1u);
                const unsigned ba = __ballot_sync(0xffffffffu, (ma >> r) & 1u);
                if (lane == r) {
                    pre_r += __popc(bp);
                    agg_r += __popc(ba);
                }
            }
            for (int n = 0; n < N; ++n) {
                const unsigned bp = __ballot_sync(0xffffffffu, (nmp >> n) & 1u);
                const unsigned ba = __ballot_sync(0xffffffffu, (nma >> n) & 1u);
                if (lane == n) {
                    pre_n += __popc(bp);
                    agg_n += __popc(ba);
                }
            }
        }
        if (lane < R && (pre_r | agg_r)) {
            atomicAdd(&s_segex[lane], pre_r);
            atomicAdd(&s_count[lane], agg_r);
        }
        if (lane < N && (pre_n | agg_n)) {
            atomicAdd(&s_segex[R + lane], pre_n);
            atomicAdd(&s_count[R + lane], agg_n);
        }
        __syncthreads();
    } else {
        // 1. per-rank / per-node counts of the channel
        int rank_acc = 0, node_acc = 0;
        for (int base = t0; base < t1; base += kNotifyThreads) {
            const int t = base + tid;
            const uint32_t m = t < t1 ? load_mask(in_rank + static_cast<int64_t>(t) * R, R) : 0u;
            const uint32_t nm = node_bits(m, R, N);
            for (int r = 0; r < R; ++r) {
                const unsigned bb = __ballot_sync(0xffffffffu, (m >> r) & 1u);
                if (lane == r) rank_acc += __popc(bb);
            }
            for (int n = 0; n < N; ++n) {
                const unsigned bb = __ballot_sync(0xffffffffu, (nm >> n) & 1u);
                if (lane == n) node_acc += __popc(bb);
            }
        }
        if (lane < R && rank_acc) atomicAdd(&s_count[lane], rank_acc);
        if (lane < N && node_acc) atomicAdd(&s_count[R + lane], node_acc);
        __syncthreads();

        // 2. publish the aggregate (the first channel of a source publishes its
        //    inclusive prefix directly), then look back within the source rank
        unsigned long long* mine = p.words + static_cast<int64_t>(b) * V;
        if (tid < V && b != p.stall_block)
            st_relaxed_u64(mine + tid, pack_word(seq, c == 0 ? kFlagPrefix : kFlagAggregate,
                                                 static_cast<uint32_t>(s_count[tid])));
        __syncthreads();
        bool timed_out = false;
        long long deadline = 0;  // set by the first wait that keeps polling
        for (int v = warp; v < V; v += kNotifyWarps) {
            const uint32_t ex = c == 0 ? 0u : segment_lookback(p, seq, b, s * C, v, lane, deadline, timed_out);
            if (lane == 0) {
                s_segex[v] = static_cast<int32_t>(ex);
                if (c != 0 && b != p.stall_block)
                    st_relaxed_u64(mine + v, pack_word(seq, kFlagPrefix, ex + static_cast<uint32_t>(s_count[v])));
            }
        }
        if (__any_sync(0xffffffffu, timed_out) && lane == 0) flag_error(p.a.status, EP_DEV_TIMEOUT);
        __syncthreads();

    }

    // 3. outputs of the block; the last channel checks the totals
    if (tid < V) {
        const int32_t incl = s_segex[tid] + s_count[tid];
        bool bad = false;
        if (tid < R) {
            const int r = tid;
            p.a.gbl_channel_prefix_matrix[(static_cast<int64_t>(s) * R + r) * C + c] = incl;
            p.a.recv_channel_offset[(static_cast<int64_t>(r) * R + s) * C + c] = cross + s_segex[r];
            s_start[r] = cross + s_segex[r];
            if (c == C - 1) bad = incl != __ldg(p.a.num_tokens_per_rank + static_cast<int64_t>(s) * R + r);
        } else {
            const int n = tid - R;
            p.a.rdma_channel_prefix_matrix[(static_cast<int64_t>(s) * N + n) * C + c] = incl;
            if (c == C - 1)
                bad = incl != __ldg(p.a.num_tokens_per_rdma_rank + static_cast<int64_t>(s) * N + n);
        }
        if (bad) flag_error(p.a.status, EP_DEV_INCONSISTENT);
    }
    __syncthreads();

    // 4. send_pos = start row + running index of the token among the
    //    channel's tokens routed to the same rank
    int32_t* send_pos = p.a.send_pos + static_cast<int64_t>(s) * T * R;
    const int stride = R + 1;
    const unsigned lt = lanemask_lt();
    for (int base = t0; base < t1; base += kNotifyThreads) {
        const int t = base + tid;
        const uint32_t m = t < t1 ? load_mask(in_rank + static_cast<int64_t>(t) * R, R) : 0u;
        for (int r = 0; r < R; ++r) {
            const unsigned bb = __ballot_sync(0xffffffffu, (m >> r) & 1u);
            if (lane == r) s_warp[warp][r] = __popc(bb);
        }
        __syncthreads();
        if (tid < R) {
            int32_t run = s_run[tid];
            for (int w = 0; w < kNotifyWarps; ++w) {
                const int32_t cnt = s_warp[w][tid];
                s_warp[w][tid] = run;
                run += cnt;
            }
            s_run[tid] = run;
        }
        __syncthreads();
        for (int r = 0; r < R; ++r) {
            const unsigned bb = __ballot_sync(0xffffffffu, (m >> r) & 1u);
            tile[tid * stride + r] =
                ((m >> r) & 1u) ? s_start[r] + s_warp[warp][r] + __popc(bb & lt) : -1;
        }
        __syncthreads();
        const int n_int = min(kNotifyThreads, t1 - base) * R;
        int32_t* dst = send_pos + static_cast<int64_t>(base) * R;
        for (int i = tid; i < n_int; i += kNotifyThreads) dst[i] = tile[(i / R) * stride + (i % R)];
        __syncthreads();
    }
}

}  // namespace

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};
}  // namespace

// Device address of the static scratch on the current device.  The first call
// on a device looks the address up (with that device current) and caches it.
// A host-side reference to the array is only a stand-in, never a device
// address, so kernels must be given this pointer instead.
cudaError_t notify_noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_notify_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return cudaSuccess;
}

size_t notify_workspace_bytes(const Shape& sh) {
    const size_t V = static_cast<size_t>(sh.R + sh.N);
    return kWorkspaceHeader + static_cast<size_t>(sh.R) * sh.C * V * sizeof(unsigned long long);
}

cudaError_t launch_notify(const Shape& sh, const NotifyArgs& a, void* workspace, bool clear_workspace,
                          bool force_lookback, int stall_block, long long wait_limit_ns,
                          cudaStream_t stream) {
    if (clear_workspace) {
        const cudaError_t e = cudaMemsetAsync(workspace, 0, notify_workspace_bytes(sh), stream);
        if (e != cudaSuccess) return e;
    }
    NotifyKernelArgs p;
    p.a = a;
    p.ticket = static_cast<unsigned long long*>(workspace);
    p.words = reinterpret_cast<unsigned long long*>(static_cast<char*>(workspace) + kWorkspaceHeader);
    p.R = sh.R;
    p.T = sh.T;
    p.E = sh.E;
    p.C = sh.C;
    p.N = sh.N;
    p.E_loc = sh.E_loc;
    p.align = sh.align;
    p.q = (sh.T + sh.C - 1) / sh.C;
    p.V = sh.R + sh.N;
    p.stall_block = stall_block;
    // Small sources (a source's membership rows fit in 8 KB) recount earlier
    // channels directly: no inter-block waits and no workspace traffic.
    // force_lookback (the test hooks) keeps the lookback path on any shape.
    p.recount = (!force_lookback && static_cast<long long>(sh.T) * sh.R <= 8 * 1024) ? 1 : 0;
    p.wait_limit_ns = wait_limit_ns;
    const size_t smem = sizeof(int32_t) * kNotifyThreads * static_cast<size_t>(sh.R + 1);
    const unsigned blocks = 1u + static_cast<unsigned>(sh.R * sh.C);
    return launch_pdl(notify_kernel, dim3(blocks), dim3(kNotifyThreads), smem, stream, 0, false, p);
}

}  // namespace ep
