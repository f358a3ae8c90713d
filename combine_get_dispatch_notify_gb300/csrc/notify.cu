// Step 2 - notify prefix sums ([IN] notify_dispatch: sm1..x stages 1-3 and
// sm0 stage 6; [RT] intranode/internodeNotifyDispatch for names and shapes).
//
// One CTA per (source rank s, channel c) block, R*C blocks in (s, c) order,
// which is also the order rows appear in every receive region.  A block
//   1. counts, per destination rank and per destination node, the tokens of
//      its channel (warp ballot + popc);
//   2. publishes that aggregate and looks back over earlier blocks
//      (single-pass decoupled lookback, one thread per rank / node value) to
//      get two exclusive prefixes at once: within its source rank (channel
//      prefix matrices) and global (start row of the block in each
//      destination region = recv_channel_offset);
//   3. rewalks its tokens and writes send_pos = block start + running index,
//      staged through shared memory so the global writes are coalesced.
// Block order comes from an atomic ticket, so a block only ever waits on
// blocks that are already running.  The last block to finish computes the
// small per-rank results (rank prefix matrix, node prefix, per-expert
// totals, recv_base) from the exchanged counts and cross-checks them with
// the scan.  Every wait gives up after a deadline and sets EP_DEV_TIMEOUT.
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
constexpr int kWorkspaceHeader = 256;  // two counters, padded

// Lookback word: [63:62] flag, [61:31] within-source prefix, [30:0] global prefix.
constexpr unsigned long long kFlagAggregate = 1ull;
constexpr unsigned long long kFlagPrefix = 2ull;
constexpr unsigned long long kMask31 = (1ull << 31) - 1;

__device__ __forceinline__ unsigned long long pack_word(unsigned long long flag, uint32_t seg,
                                                        uint32_t glob) {
    return (flag << 62) | ((static_cast<unsigned long long>(seg) & kMask31) << 31) |
           (static_cast<unsigned long long>(glob) & kMask31);
}
__device__ __forceinline__ uint32_t word_seg(unsigned long long w) {
    return static_cast<uint32_t>((w >> 31) & kMask31);
}
__device__ __forceinline__ uint32_t word_glob(unsigned long long w) {
    return static_cast<uint32_t>(w & kMask31);
}

struct NotifyKernelArgs {
    NotifyArgs a;
    unsigned* counters;        // [0] ticket, [1] finished blocks
    unsigned long long* words; // [R*C][V]
    int R, T, E, C, N, E_loc, align, q, V;
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

__device__ __forceinline__ uint32_t node_bits(uint32_t m, int R, int N) {
    if (R <= kNodeSize) return m != 0u ? 1u : 0u;
    uint32_t nm = 0;
    for (int n = 0; n < N; ++n) nm |= ((m >> (kNodeSize * n)) & 0xffu) ? (1u << n) : 0u;
    return nm;
}

__device__ void finish(const NotifyKernelArgs& p, int32_t* s_nrecv) {
    const NotifyArgs& a = p.a;
    const int R = p.R, N = p.N, C = p.C, V = p.V, tid = threadIdx.x;
    bool inconsistent = false;
    // [IN] sm0 stage 6: prefix of per-rank counts over global source rank.
    for (int r = tid; r < R; r += blockDim.x) {
        int32_t run = 0;
        for (int s = 0; s < R; ++s) {
            run += a.num_tokens_per_rank[static_cast<int64_t>(s) * R + r];
            a.rank_prefix_matrix[static_cast<int64_t>(s) * R + r] = run;
            a.recv_gbl_rank_prefix_sum[static_cast<int64_t>(r) * R + s] = run;
            const unsigned long long w =
                ld_acquire_u64(p.words + (static_cast<int64_t>(s) * C + C - 1) * V + r);
            if (word_glob(w) != static_cast<uint32_t>(run)) inconsistent = true;
        }
        a.num_recv_tokens[r] = run;
        s_nrecv[r] = run;
    }
    // Node-level receive prefix: rank r receives for its node from the
    // same-GPU-index peer m*8 + r%8 of every node m.
    for (int r = tid; r < R; r += blockDim.x) {
        int32_t run = 0;
        for (int m = 0; m < N; ++m) {
            const int peer = m * kNodeSize + r % kNodeSize;
            run += a.num_tokens_per_rdma_rank[static_cast<int64_t>(peer) * N + r / kNodeSize];
            a.recv_rdma_rank_prefix_sum[static_cast<int64_t>(r) * N + m] = run;
        }
        a.num_rdma_recv_tokens[r] = run;
    }
    for (int i = tid; i < R * N; i += blockDim.x) {
        const int s = i / N, n = i % N;
        const unsigned long long w =
            ld_acquire_u64(p.words + (static_cast<int64_t>(s) * C + C - 1) * V + R + n);
        if (word_seg(w) != static_cast<uint32_t>(a.num_tokens_per_rdma_rank[i])) inconsistent = true;
    }
    // Per-expert receive counts, rounded up to the alignment.
    for (int i = tid; i < R * p.E_loc; i += blockDim.x) {
        const int r = i / p.E_loc, j = i % p.E_loc;
        long long sum = 0;
        for (int s = 0; s < R; ++s)
            sum += a.num_tokens_per_expert[static_cast<int64_t>(s) * p.E + r * p.E_loc + j];
        sum = (sum + p.align - 1) / p.align * p.align;
        a.num_recv_tokens_per_expert[i] = static_cast<int32_t>(sum);
    }
    if (inconsistent) flag_error(a.status, EP_DEV_INCONSISTENT);
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

__global__ void __launch_bounds__(kNotifyThreads) notify_kernel(NotifyKernelArgs p) {
    extern __shared__ int32_t tile[];  // [kNotifyThreads][R + 1] send_pos staging
    __shared__ int s_block, s_last;
    __shared__ int32_t s_count[64];    // block totals: ranks, then nodes
    __shared__ int32_t s_start[32];    // global start row of this block, per rank
    __shared__ int32_t s_run[32];      // running count inside the channel
    __shared__ int32_t s_warp[kNotifyWarps][33];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int R = p.R, N = p.N, C = p.C, V = p.V, T = p.T;
    if (tid == 0) s_block = static_cast<int>(atomicAdd(p.counters, 1u));
    if (tid < 64) s_count[tid] = 0;
    if (tid < 32) s_run[tid] = 0;
    __syncthreads();
    const int b = s_block, s = b / C, c = b % C;
    const int t0 = min(c * p.q, T), t1 = min(t0 + p.q, T);
    const uint8_t* in_rank = p.a.is_token_in_rank + static_cast<int64_t>(s) * T * R;

    // 1. per-rank / per-node counts of the channel ([IN] sm1..x stage 1)
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

    // 2. publish, look back, publish the inclusive prefix ([IN] stages 2-3)
    if (tid < V) {
        const int v = tid;
        const uint32_t agg = static_cast<uint32_t>(s_count[v]);
        unsigned long long* mine = p.words + static_cast<int64_t>(b) * V + v;
        uint32_t ex_seg = 0, ex_glob = 0;
        if (b != p.stall_block) {
            if (b == 0) {
                st_release_u64(mine, pack_word(kFlagPrefix, agg, agg));
            } else {
                st_release_u64(mine, pack_word(kFlagAggregate, agg, agg));
                const long long deadline = globaltimer_ns() + p.wait_limit_ns;
                bool timed_out = false;
                for (int j = b - 1; j >= 0 && !timed_out; --j) {
                    const unsigned long long* w = p.words + static_cast<int64_t>(j) * V + v;
                    unsigned long long word = ld_acquire_u64(w);
                    uint32_t polls = 0;
                    while ((word >> 62) == 0ull) {
                        if ((++polls & 15u) == 0 && globaltimer_ns() > deadline) {
                            timed_out = true;
                            break;
                        }
                        __nanosleep(64);
                        word = ld_acquire_u64(w);
                    }
                    if (timed_out) break;
                    ex_glob += word_glob(word);
                    if (j / C == s) ex_seg += word_seg(word);
                    if ((word >> 62) == kFlagPrefix) break;
                }
                if (timed_out) flag_error(p.a.status, EP_DEV_TIMEOUT);
                st_release_u64(mine, pack_word(kFlagPrefix, ex_seg + agg, ex_glob + agg));
            }
            if (v < R) {
                p.a.gbl_channel_prefix_matrix[(static_cast<int64_t>(s) * R + v) * C + c] =
                    static_cast<int32_t>(ex_seg + agg);
                p.a.recv_channel_offset[(static_cast<int64_t>(v) * R + s) * C + c] =
                    static_cast<int32_t>(ex_glob);
            } else {
                p.a.rdma_channel_prefix_matrix[(static_cast<int64_t>(s) * N + (v - R)) * C + c] =
                    static_cast<int32_t>(ex_seg + agg);
            }
        }
        if (v < R) s_start[v] = static_cast<int32_t>(ex_glob);
    }
    __syncthreads();

    // 3. send_pos = block start + running index of the token among the
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

    // last block to finish computes the per-rank results
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(p.counters + 1, 1u) == gridDim.x - 1u;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    finish(p, s_run);  // s_run is free now: reuse it for the per-rank totals
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

cudaError_t launch_notify(const Shape& sh, const NotifyArgs& a, void* workspace, int stall_block,
                          long long wait_limit_ns, cudaStream_t stream) {
    const size_t ws_bytes = notify_workspace_bytes(sh);
    cudaError_t e = cudaMemsetAsync(workspace, 0, ws_bytes, stream);
    if (e != cudaSuccess) return e;
    NotifyKernelArgs p;
    p.a = a;
    p.counters = static_cast<unsigned*>(workspace);
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
    p.wait_limit_ns = wait_limit_ns;
    const size_t smem = sizeof(int32_t) * kNotifyThreads * static_cast<size_t>(sh.R + 1);
    const int blocks = sh.R * sh.C;
    notify_kernel<<<blocks, kNotifyThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace ep
