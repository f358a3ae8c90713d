// Layout + notify over tiles of tokens, for any number of CTAs.
//
// The same results as the layout step ([RT] getDispatchLayout; the count
// vectors of [IN] notify_dispatch sm0 stage 3) followed by notify ([IN]
// sm1..x stages 1-3 and sm0 stage 6), computed by CTAs that each take tiles
// of up to TT tokens of one source rank, tiles numbered in (source rank,
// tile) order: a CTA's first tile is its block index, its later ones come
// from an atomic ticket counter:
//   A. thread per (token, pair of top-k slots), up to 8 pairs of a thread
//      loaded at once: expert histogram in shared memory and the token's rank
//      mask; warp per 32 tokens writes the is_token_in_rank rows and gets
//      one ballot word per destination rank / node (a 32x32 bit transpose of
//      the tokens' masks), whose popcounts are the tile's counts;
//   B. warp per value (rank or node): the exclusive prefix of every 32-token
//      block inside the tile;
//   C. two-level single-pass scan ([AR] 3.2: prefix sums by a block scan):
//      a tile publishes its counts, and adds them into its source's total
//      words (one 64-bit atomic per value: the tiles that have added in the
//      high half, the running total in the low half); adds its histogram into
//      its source's expert counter words the same way; looks back
//      over the earlier tiles of its own source (decoupled lookback, 32
//      predecessors per probe, every value at once) and adds the totals of
//      the earlier source ranks, each read once all of that source's tiles
//      have added into it.  Tiles are ordered by source rank first, so the
//      result - the global exclusive prefix of rank r at the tile - is
//      exactly the row, inside r's receive region, of the tile's first token
//      routed to r;
//   D. the tile's outputs: send_pos of its tokens; the channel boundaries
//      inside it (recv_channel_offset at a channel's first token,
//      gbl/rdma_channel_prefix_matrix at its end); for the source's last
//      tile the source's counts and rank prefix;
//   E. the last tile - it holds the global prefix at the very end - writes
//      the receive counts, recv_base and the node-level receive prefix; the
//      thread whose add completed a source's expert counter word writes that
//      count out, clears the word for the next call and adds the count into
//      the call's word for the expert, whose R-th add does the same for the
//      per-expert receive count.
// Only steps C and E wait, and only on tiles with smaller numbers (earlier
// tiles of the source; the tiles of earlier sources), which publish what is
// waited for before they wait on anything.  A smaller number is either the
// first tile of a CTA with a smaller block index - dispatched before this
// CTA, as blocks are dispatched in index order (the order a single-pass scan
// with decoupled look-back relies on), so already running or done - or a
// ticket taken earlier by a running CTA, which works on it after its current
// (smaller) tile.  So the scan needs no co-residency and finishes in a few
// probes whatever the number of tiles; every wait is bounded
// (EP_DEV_TIMEOUT).
#pragma once

#include "ep_device.cuh"
#include "ep_internal.h"

namespace ep {

constexpr int kTiledMaxValues = 64;  // R + N <= 32 + 4
constexpr int kLbSlots = 32;         // predecessors read per lookback probe
constexpr int kAccRanks = 32;
constexpr int kAccExperts = 8192;
constexpr int kBankWords = 32 * 36;  // source total words of one call: [R][V], R <= 32, V <= 36

// Workspace of the tiled form, all offsets in bytes from its start:
//   header     ticket word, the finished-tiles counter and the `ready` word;
//   acc        expert counter words of the running call (64-bit: tiles that
//              have added in [63:32], count in [31:0]), per source
//              [32][8192] and summed over sources [8192], whatever the shape
//              (so a later call of another shape finds them zero);
//   banks      two banks of source total words [32 * 36] (64-bit: tiles in
//              [63:32], total in [31:0]); a call adds into the bank of its
//              sequence number's parity, and its first tile clears the other
//              one for the next call;
//   words      within-source lookback words [n_tiles][V], tagged with the
//              writing call's sequence number, so what an earlier call of any
//              shape left there never reads as this call's.
// The header, acc and banks must be zero before the first call; every call
// leaves the header counters and acc zero, and the next call's bank.
struct TiledWorkspace {
    size_t ticket, finished, ready, acc, acc_all, banks, words, total;
};

inline TiledWorkspace tiled_workspace_layout(int R, int N, long long n_tiles) {
    TiledWorkspace w;
    const size_t V = static_cast<size_t>(R + N);
    w.ticket = 0;
    w.finished = 12;
    w.ready = 16;
    w.acc = 256;
    w.acc_all = w.acc + sizeof(unsigned long long) * static_cast<size_t>(kAccRanks) * kAccExperts;
    w.banks = w.acc_all + sizeof(unsigned long long) * static_cast<size_t>(kAccExperts);
    w.words = w.banks + sizeof(unsigned long long) * 2 * static_cast<size_t>(kBankWords);
    w.total = w.words + sizeof(unsigned long long) * static_cast<size_t>(n_tiles) * V;
    return w;
}

struct TiledLnArgs {
    const int64_t* topk_idx;
    int32_t* num_tokens_per_rank;
    int32_t* num_tokens_per_rdma_rank;
    int32_t* num_tokens_per_expert;
    uint8_t* is_token_in_rank;
    NotifyArgs a;  // outputs of the notify step (its count-input fields are unused)
    unsigned long long* ticket;  // [63:32] sequence number of the last call, [31:0] tickets taken
    unsigned* finished;          // tiles whose outputs are written, this call (signal_ready)
    unsigned long long* ready;   // sequence number of the last call whose row map is complete
    unsigned long long* acc;      // [32][8192] per-source expert counter words of the running call
    unsigned long long* acc_all;  // [8192] expert counter words summed over sources
    unsigned long long* banks;   // [2][32 * 36] source total words, by call parity
    unsigned long long* words;   // [n_tiles][V] lookback words, within each source
    int R, T, K, E, N, E_loc, C, q, align, V, TT, tps, n_tiles;
    int Ep, Vp;           // E and V rounded up to 4 (shared-memory row strides)
    uint32_t eloc_magic;  // ceil(2^32 / E_loc): e / E_loc = umulhi(e, magic) for e < 8192, E_loc >= 2
    int stall_tile;       // test hook: this tile never publishes its lookback words (-1: none)
    int signal_ready;     // 1: count finished tiles and publish `ready` (a dispatch waits on it)
    long long wait_limit_ns;
};

// Tagged word: [63:32] sequence number of the writing call, [31:30] flag,
// [29:0] value.  A word of another call reads as "not yet published".  The
// word is the whole message - nothing else is read on the strength of it -
// so it is stored and polled with relaxed gpu-scope accesses, as are the
// source total words.
constexpr unsigned kLbAggregate = 1u;
constexpr unsigned kLbPrefix = 2u;

__device__ __forceinline__ unsigned long long lb_pack(unsigned seq, unsigned flag, uint32_t val) {
    return (static_cast<unsigned long long>(seq) << 32) | (static_cast<unsigned long long>(flag) << 30) |
           (static_cast<unsigned long long>(val) & ((1ull << 30) - 1));
}
__device__ __forceinline__ int32_t lb_val(unsigned long long w) {
    return static_cast<int32_t>(w & ((1ull << 30) - 1));
}

// A thread's waits in one tile share one deadline, set by the first of them
// that keeps polling (0 until then: a tile whose words are all there reads
// no timer).  True once it has passed.
__device__ __forceinline__ bool wait_expired(long long& deadline, long long limit_ns) {
    const long long now = globaltimer_ns();
    if (deadline == 0) {
        deadline = now + limit_ns;
        return false;
    }
    return now > deadline;
}

// Reads a tagged word of call `seq`, waiting (bounded) until it is published.
// On timeout returns a prefix word of value 0 and sets `timed_out`.
__device__ __forceinline__ unsigned long long lb_wait(const unsigned long long* w, unsigned seq, long long limit_ns,
                                                      long long& deadline, bool& timed_out) {
    unsigned long long word = ld_relaxed_u64(w);
    uint32_t polls = 0;
    while (static_cast<unsigned>(word >> 32) != seq) {
        if ((++polls & 15u) == 0 && wait_expired(deadline, limit_ns)) {
            timed_out = true;
            return lb_pack(seq, kLbPrefix, 0);
        }
        __nanosleep(32);
        word = ld_relaxed_u64(w);
    }
    return word;
}

// Total of a source once all `tiles` of its tiles have added into its word
// (waiting, bounded); on timeout 0 and `timed_out` set.
__device__ __forceinline__ int32_t bank_wait(const unsigned long long* w, unsigned tiles, long long limit_ns,
                                             long long& deadline, bool& timed_out) {
    unsigned long long word = ld_relaxed_u64(w);
    uint32_t polls = 0;
    while (static_cast<unsigned>(word >> 32) != tiles) {
        if ((++polls & 15u) == 0 && wait_expired(deadline, limit_ns)) {
            timed_out = true;
            return 0;
        }
        __nanosleep(32);
        word = ld_relaxed_u64(w);
    }
    return static_cast<int32_t>(word & 0xffffffffull);
}

// Dynamic shared memory of one tile, in 4-byte words: the expert histogram
// (E rounded up to 4), token masks [TT], ballots and block prefixes [TT/32]
// [Vp] with Vp = V rounded up to 4, so the rows of 4 ranks are 16-byte
// aligned.
inline int tiled_pad4(int x) { return (x + 3) & ~3; }
inline size_t tiled_smem_words(int E, int TT, int V) {
    const size_t J = static_cast<size_t>(TT) / kWarp;
    return static_cast<size_t>(tiled_pad4(E)) + TT + 2 * J * tiled_pad4(V);
}

struct TiledShared {
    int32_t cnt[kTiledMaxValues];  // the tile's count per value
    int32_t wex[kTiledMaxValues];  // exclusive prefix within the source
    int32_t xs[kTiledMaxValues];   // rows earlier source ranks send to each value
    int32_t fin[kTiledMaxValues];
    uint32_t lb[kLbSlots][kTiledMaxValues];  // low halves of the words of one lookback probe
    int ticket;
    unsigned seq;
};

// Tickets: a CTA's first tile is its block index; every CTA takes one ticket
// per tile it works on (a CTA without a first tile, one ticket), max(n_tiles,
// grid) tickets in all, and ticket t names tile grid + t (none once that is
// n_tiles or more).  A ticket also carries the call's sequence number (the
// previous call's, in the high half, plus one).  Decodes a ticket taken by
// this thread into sh.seq and sh.ticket (the CTA's next tile, or -1); the
// ticket that completes the count arms the next call.
__device__ __forceinline__ void tiled_ticket_done(const TiledLnArgs& p, TiledShared& sh, unsigned long long old) {
    const unsigned taken = static_cast<unsigned>(old & 0xffffffffull);
    const unsigned seq = static_cast<unsigned>(old >> 32) + 1u;
    const unsigned total = max(static_cast<unsigned>(p.n_tiles), gridDim.x);
    if (taken == total - 1u) atomicExch(p.ticket, static_cast<unsigned long long>(seq) << 32);
    if (taken >= total) flag_error(p.a.status, EP_DEV_INCONSISTENT);  // workspace not zeroed
    const long long next = static_cast<long long>(gridDim.x) + taken;
    sh.ticket = next < p.n_tiles ? static_cast<int>(next) : -1;
    sh.seq = seq;
}

// Prefix of value v before local token lt of the tile (0 <= lt <= ntok).
__device__ __forceinline__ int32_t tiled_prefix_at(const uint32_t* bal, const int32_t* pre, const int32_t* cnt,
                                                   int V, int ntok, int v, int lt) {
    if (lt >= ntok) return cnt[v];
    const int j = lt >> 5;
    return pre[j * V + v] + __popc(bal[j * V + v] & ((1u << (lt & 31)) - 1u));
}

// One top-k id: its bin of the shared histogram and its rank bit.  An id
// outside [-1, E) sets `bad` and is ignored.
__device__ __forceinline__ void tiled_count_id(const TiledLnArgs& p, long long e, int32_t* hist, uint32_t& mask,
                                               bool& bad) {
    if (e >= 0 && e < p.E) {
        const uint32_t u = static_cast<uint32_t>(e);
        mask |= 1u << (p.E_loc == 1 ? u : __umulhi(u, p.eloc_magic));
        atomicAdd(&hist[u], 1);
    } else if (e != -1) {
        bad = true;
    }
}

// 32 x 32 bit transpose across a warp: on return lane c holds, in bit i,
// bit c of lane i's input.  Five exchanges of half-blocks with the partner
// lane (lane ^ j), halving the block size each time.
__device__ __forceinline__ uint32_t warp_transpose32(uint32_t x, int lane) {
    constexpr uint32_t kMask[5] = {0x0000ffffu, 0x00ff00ffu, 0x0f0f0f0fu, 0x33333333u, 0x55555555u};
#pragma unroll
    for (int k = 0; k < 5; ++k) {
        const int j = 16 >> k;
        const uint32_t m = kMask[k];
        const uint32_t y = __shfl_xor_sync(0xffffffffu, x, j);
        x = (lane & j) ? ((x & ~m) | ((y & ~m) >> j)) : ((x & m) | ((y & m) << j));
    }
    return x;
}

// Hint: bring the top-k ids of tile b into L2 (a CTA's first tile, whose
// loads start straight away).
__device__ __forceinline__ void tiled_prefetch_ids(const TiledLnArgs& p, int b) {
    if (b >= p.n_tiles) return;
    const int s = b / p.tps, j = b - s * p.tps;
    const int t0 = j * p.TT, t1 = min(t0 + p.TT, p.T);
    if (t1 > t0)
        prefetch_l2(p.topk_idx + (static_cast<int64_t>(s) * p.T + t0) * p.K,
                    static_cast<size_t>(t1 - t0) * p.K * sizeof(int64_t));
}

// Expert e of source s after this tile's add (h: the tile's count; o_src:
// the source's counter word before it).  The add that completed the source's
// word writes its count out, clears it and adds the source's count into the
// call's word for e, whose R-th add writes the per-expert receive count
// (rounded up to the alignment) out and clears that word.  One call-wide add
// per source and expert, not per tile, keeps the call's words uncontended.
// The two halves: the source's word (returns whether this add completed it,
// and the call's word before the source's count went in), then the call's.
__device__ __forceinline__ bool tiled_expert_source(const TiledLnArgs& p, int s, int e, int32_t h,
                                                    unsigned long long o_src, int32_t& total,
                                                    unsigned long long& o_all) {
    if (static_cast<unsigned>(o_src >> 32) != static_cast<unsigned>(p.tps - 1)) return false;
    total = static_cast<int32_t>(o_src) + h;
    p.num_tokens_per_expert[static_cast<int64_t>(s) * p.E + e] = total;
    p.acc[static_cast<int64_t>(s) * kAccExperts + e] = 0ull;
    o_all = atomicAdd(p.acc_all + e, (1ull << 32) | static_cast<uint32_t>(total));
    return true;
}
__device__ __forceinline__ void tiled_expert_call(const TiledLnArgs& p, int e, int32_t total,
                                                  unsigned long long o_all) {
    if (static_cast<unsigned>(o_all >> 32) == static_cast<unsigned>(p.R - 1)) {
        const long long c = static_cast<long long>(static_cast<int32_t>(o_all)) + total;
        p.a.num_recv_tokens_per_expert[e] = static_cast<int32_t>((c + p.align - 1) / p.align * p.align);
        p.acc_all[e] = 0ull;
    }
}
__device__ __forceinline__ void tiled_expert_done(const TiledLnArgs& p, int s, int e, int32_t h,
                                                  unsigned long long o_src) {
    int32_t total = 0;
    unsigned long long o_all = 0;
    if (tiled_expert_source(p, s, e, h, o_src, total, o_all)) tiled_expert_call(p, e, total, o_all);
}

// One tile b (of source b / tps); returns the CTA's next tile, or -1.  Thread
// `taker` takes the next ticket as the tile starts and reads it (the call's
// sequence number with it) only once the tile's counts are in, so its round
// trip overlaps the tile's loads.  `dyn` holds tiled_smem_words() words.
// Every thread of the CTA calls it; blockDim.x is a multiple of 32.
__device__ inline int tiled_tile(const TiledLnArgs& p, TiledShared& sh, int32_t* dyn, int b, int taker) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = static_cast<int>(blockDim.x), warps = B >> 5;
    const int R = p.R, N = p.N, V = p.V, K = p.K, T = p.T, E = p.E, C = p.C;
    const int s = b / p.tps, j = b - s * p.tps;
    const bool last_tile = j == p.tps - 1;
    const int t0 = j * p.TT, t1 = min(t0 + p.TT, T), ntok = max(t1 - t0, 0);
    const int Jt = (ntok + kWarp - 1) / kWarp;
    const int J = p.TT / kWarp;
    const int Vp = p.Vp;
    int32_t* hist = dyn;
    uint32_t* tmask = reinterpret_cast<uint32_t*>(hist + p.Ep);
    uint32_t* bal = tmask + p.TT;
    int32_t* pre = reinterpret_cast<int32_t*>(bal + J * Vp);
    const long long limit = p.wait_limit_ns;
    long long deadline = 0;  // set by the first wait that keeps polling
    bool timed_out = false;
    unsigned long long ticket = 0;
    if (tid == taker) ticket = atomicAdd(p.ticket, 1ull);

    for (int i = tid; i < E; i += B) hist[i] = 0;
    for (int i = tid; i < ntok; i += B) tmask[i] = 0u;
    if (tid < V) {
        sh.fin[tid] = 0;
        sh.xs[tid] = 0;
        sh.cnt[tid] = 0;
    }
    __syncthreads();

    // A1. thread per (token, pair of slots), up to 8 pairs loaded at once;
    //     a thread keeps its pair and steps through tokens (no division)
    bool bad = false;
    {
        const int P2 = (K + 1) >> 1;
        const int tpi = B / P2;  // tokens per sweep of the CTA
        if (tid < tpi * P2) {
            const int pk = tid % P2;
            const int64_t* ids = p.topk_idx + (static_cast<int64_t>(s) * T + t0) * K + 2 * pk;
            constexpr int kU = 8;
            for (int t = tid / P2; t < ntok; t += kU * tpi) {
                long long e0[kU], e1[kU];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int tt = t + u * tpi;
                    e0[u] = -1;
                    e1[u] = -1;
                    if (tt < ntok) {
                        const int64_t* row = ids + static_cast<int64_t>(tt) * K;
                        if ((K & 1) == 0) {
                            const longlong2 v2 = __ldg(reinterpret_cast<const longlong2*>(row));
                            e0[u] = v2.x;
                            e1[u] = v2.y;
                        } else {
                            e0[u] = __ldg(row);
                            e1[u] = 2 * pk + 1 < K ? __ldg(row + 1) : -1;
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int tt = t + u * tpi;
                    if (tt >= ntok) break;
                    uint32_t m = 0;
                    tiled_count_id(p, e0[u], hist, m, bad);
                    tiled_count_id(p, e1[u], hist, m, bad);
                    if (m) atomicOr(&tmask[tt], m);
                }
            }
        }
    }
    if (bad) flag_error(p.a.status, EP_DEV_INPUT);
    __syncthreads();

    // A2. warp per 32-token block: membership rows and one ballot word per
    //     value (bit i: token i of the block goes to it), all values at once by
    //     a bit transpose of the 32 tokens' masks (ranks, then nodes when
    //     they fit in the same word; otherwise one ballot per node)
    const bool nodes_in_word = R + N <= kWarp;
    for (int jj = warp; jj < Jt; jj += warps) {
        const int lt = jj * kWarp + lane;
        const uint32_t mask = lt < ntok ? tmask[lt] : 0u;
        if (lt < ntok)
            write_membership_row(p.is_token_in_rank + (static_cast<int64_t>(s) * T + t0 + lt) * R, mask, R);
        const uint32_t nb = node_bits(mask, R, N);
        const uint32_t word = nodes_in_word ? (mask | (nb << R)) : mask;
        const uint32_t tr = warp_transpose32(word, lane);
        if (lane < V) {
            bal[jj * Vp + lane] = tr;
            if (tr) atomicAdd(&sh.cnt[lane], __popc(tr));  // the tile's count per value
        }
        if (!nodes_in_word) {
            for (int n = 0; n < N; ++n) {
                const unsigned bb = __ballot_sync(0xffffffffu, (nb >> n) & 1u);
                if (lane == 0) {
                    bal[jj * Vp + R + n] = bb;
                    if (bb) atomicAdd(&sh.cnt[R + n], __popc(bb));
                }
            }
        }
    }
    if (tid == taker) tiled_ticket_done(p, sh, ticket);
    __syncthreads();
    const unsigned seq = sh.seq;
    unsigned long long* bank = p.banks + (seq & 1u) * kBankWords;  // this call's source totals
    if (b == 0) {  // the previous call is complete: its bank is the next call's
        unsigned long long* other = p.banks + ((seq + 1u) & 1u) * kBankWords;
        for (int i = tid; i < kBankWords; i += B) other[i] = 0ull;
    }

    // C1. publish the tile's counts at once (the first tile of a source: its
    //     inclusive prefix) and add them into the source's totals, before the
    //     block prefixes below, so the tiles after it can read them sooner
    const bool withhold = b == p.stall_tile;
    unsigned long long* mine = p.words + static_cast<int64_t>(b) * V;
    if (tid < V && !withhold) {
        const uint32_t c = static_cast<uint32_t>(sh.cnt[tid]);
        st_relaxed_u64(mine + tid, lb_pack(seq, j == 0 ? kLbPrefix : kLbAggregate, c));
        atomicAdd(bank + s * V + tid, (1ull << 32) | c);
    }

    // B. warp per value: exclusive prefix of each 32-token block
    {
        const int per = (Jt + kWarp - 1) / kWarp;
        for (int v = warp; v < V; v += warps) {
            const int j0 = min(lane * per, Jt), j1 = min(j0 + per, Jt);
            int32_t sum = 0;
            for (int jj = j0; jj < j1; ++jj) sum += __popc(bal[jj * Vp + v]);
            int32_t inc = sum;
#pragma unroll
            for (int o = 1; o < kWarp; o <<= 1) {
                const int32_t y = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += y;
            }
            int32_t run = inc - sum;
            for (int jj = j0; jj < j1; ++jj) {
                pre[jj * Vp + v] = run;
                run += __popc(bal[jj * Vp + v]);
            }
        }
    }

    // C. two-level scan: (1, above) the counts are published and added into
    //    the source's totals; (2) look back over the source's earlier tiles;
    //    (3) sum the totals of the earlier sources.
    // The tile's expert counts into the source's and the call's counter
    // words, every expert whether its count is zero or not; with no more
    // experts than threads the adds go out here and their results (which
    // say whether this add completed the word) are read in E2
    const bool experts_early = E <= B;
    unsigned long long ex_src = 0;
    int32_t ex_h = 0;
    if (experts_early && tid < E) {
        ex_h = hist[tid];
        ex_src = atomicAdd(p.acc + static_cast<int64_t>(s) * kAccExperts + tid,
                           (1ull << 32) | static_cast<uint32_t>(ex_h));
    }
    const int Bl = B - kWarp;  // threads of the lookback loads
    // the totals of the earlier sources (word i = s2 * V + v of the bank):
    // first loads issued now, checked after the lookback, so the two round
    // trips overlap
    constexpr int kTotalsAhead = 4;
    const int n_totals = s * V;
    unsigned long long tw[kTotalsAhead];
#pragma unroll
    for (int k = 0; k < kTotalsAhead; ++k) {
        const int i = tid + k * B;
        tw[k] = i < n_totals ? ld_relaxed_u64(bank + i) : 0ull;
    }
    int32_t wex = 0;  // thread v < V: exclusive prefix of value v within the source
    if (j > 0) {
        const int seg_lo = s * p.tps;  // first tile of the source
        for (int r0 = 0;; r0 += kLbSlots) {
            // thread walks pairs (slot, value) i = tid, tid + Bl, ... without dividing
            int slot = tid / V, v = tid - (tid / V) * V;
            for (int i = tid; tid < Bl && i < kLbSlots * V; i += Bl, slot += Bl / V, v += Bl % V) {
                if (v >= V) {
                    v -= V;
                    ++slot;
                }
                if (sh.fin[v]) continue;
                const int pj = b - 1 - r0 - slot;  // before the source's first tile: prefix 0
                const unsigned long long word =
                    pj >= seg_lo ? lb_wait(p.words + static_cast<int64_t>(pj) * V + v, seq, limit, deadline, timed_out)
                                 : lb_pack(seq, kLbPrefix, 0);
                sh.lb[slot][v] = static_cast<uint32_t>(word);  // [31:30] flag, [29:0] value
            }
            __syncthreads();
            if (tid < V && !sh.fin[tid]) {
                for (int slot = 0; slot < kLbSlots; ++slot) {
                    const uint32_t lo = sh.lb[slot][tid];
                    wex += static_cast<int32_t>(lo & ((1u << 30) - 1));
                    if ((lo >> 30) == kLbPrefix) {
                        sh.fin[tid] = 1;
                        break;
                    }
                }
            }
            if (!__syncthreads_or(tid < V && !sh.fin[tid])) break;
        }
    }
    if (tid < V) {
        sh.wex[tid] = wex;
        if (!withhold) {
            const uint32_t incl = static_cast<uint32_t>(wex + sh.cnt[tid]);
            if (j > 0) st_relaxed_u64(mine + tid, lb_pack(seq, kLbPrefix, incl));
        }
    }
    {
        const unsigned tps = static_cast<unsigned>(p.tps);
#pragma unroll
        for (int k = 0; k < kTotalsAhead; ++k) {
            const int i = tid + k * B;
            if (i < n_totals) {
                const int32_t t = static_cast<unsigned>(tw[k] >> 32) == tps
                                      ? static_cast<int32_t>(tw[k] & 0xffffffffull)
                                      : bank_wait(bank + i, tps, limit, deadline, timed_out);
                atomicAdd(&sh.xs[i % V], t);
            }
        }
        for (int i = tid + kTotalsAhead * B; i < n_totals; i += B)
            atomicAdd(&sh.xs[i % V], bank_wait(bank + i, tps, limit, deadline, timed_out));
    }
    __syncthreads();

    // the source's half of the expert words now (the adds went out in C), so
    // the call-wide add's round trip overlaps step D; its result is read in E2
    bool ex_done = false;
    int32_t ex_total = 0;
    unsigned long long ex_all = 0;
    if (experts_early && tid < E) ex_done = tiled_expert_source(p, s, tid, ex_h, ex_src, ex_total, ex_all);

    // D1. send_pos[s][t][r]: row of (s,t) inside r's region, or -1.  A
    //     thread keeps 4 ranks (their row offsets in registers) and steps
    //     through tokens; 16-byte loads of ballots and prefixes, 16-byte stores
    int32_t* send_pos = p.a.send_pos + (static_cast<int64_t>(s) * T + t0) * R;
    if ((R & 3) == 0) {
        const int qpt = R >> 2, tpi = B / qpt;
        if (tid < tpi * qpt) {
            const int r0 = (tid % qpt) * 4;
            const int32_t o0 = sh.xs[r0] + sh.wex[r0], o1 = sh.xs[r0 + 1] + sh.wex[r0 + 1];
            const int32_t o2 = sh.xs[r0 + 2] + sh.wex[r0 + 2], o3 = sh.xs[r0 + 3] + sh.wex[r0 + 3];
            for (int lt = tid / qpt; lt < ntok; lt += tpi) {
                const int jj = lt >> 5;
                const uint32_t bit = 1u << (lt & 31), below = bit - 1u;
                const uint4 bb = *reinterpret_cast<const uint4*>(bal + jj * Vp + r0);
                const int4 pp = *reinterpret_cast<const int4*>(pre + jj * Vp + r0);
                int4 o;
                o.x = (bb.x & bit) ? o0 + pp.x + __popc(bb.x & below) : -1;
                o.y = (bb.y & bit) ? o1 + pp.y + __popc(bb.y & below) : -1;
                o.z = (bb.z & bit) ? o2 + pp.z + __popc(bb.z & below) : -1;
                o.w = (bb.w & bit) ? o3 + pp.w + __popc(bb.w & below) : -1;
                *reinterpret_cast<int4*>(send_pos + static_cast<int64_t>(lt) * R + r0) = o;
            }
        }
    } else {
        for (int i = tid; i < ntok * R; i += B) {
            const int lt = i / R, r = i - lt * R;
            const int jj = lt >> 5;
            const uint32_t bit = 1u << (lt & 31);
            const uint32_t bb = bal[jj * Vp + r];
            send_pos[i] = (bb & bit) ? sh.xs[r] + sh.wex[r] + pre[jj * Vp + r] + __popc(bb & (bit - 1u)) : -1;
        }
    }
    // D2. channel boundaries owned by this tile: boundary c sits at token
    //     min(c*q, T) (c = 0..C); a tile owns those inside it, the source's
    //     last tile also those at T.  Channel c starts at boundary c and ends
    //     at boundary c + 1.
    {
        int c_lo, c_hi;
        if (p.q == 0) {  // T == 0: every boundary is token 0, in the only tile
            c_lo = 0;
            c_hi = C;
        } else {
            c_lo = (t0 + p.q - 1) / p.q;
            c_hi = last_tile ? C : min((t1 + p.q - 1) / p.q - 1, C);
        }
        const int nc = c_hi - c_lo + 1;
        for (int i = tid; i < nc * V; i += B) {
            const int c = c_lo + i / V, v = i - (i / V) * V;
            const long long x = min(static_cast<long long>(c) * p.q, static_cast<long long>(T));
            const int32_t within = sh.wex[v] + tiled_prefix_at(bal, pre, sh.cnt, Vp, ntok, v, static_cast<int>(x - t0));
            if (v < R) {
                if (c < C) p.a.recv_channel_offset[(static_cast<int64_t>(v) * R + s) * C + c] = sh.xs[v] + within;
                if (c > 0) p.a.gbl_channel_prefix_matrix[(static_cast<int64_t>(s) * R + v) * C + c - 1] = within;
            } else if (c > 0) {
                p.a.rdma_channel_prefix_matrix[(static_cast<int64_t>(s) * N + (v - R)) * C + c - 1] = within;
            }
        }
    }
    // D3. the source's counts and rank prefix (its last tile holds its totals)
    if (last_tile && tid < V) {
        const int32_t total = sh.wex[tid] + sh.cnt[tid];
        if (tid < R) {
            p.num_tokens_per_rank[static_cast<int64_t>(s) * R + tid] = total;
            p.a.rank_prefix_matrix[static_cast<int64_t>(s) * R + tid] = sh.xs[tid] + total;
            p.a.recv_gbl_rank_prefix_sum[static_cast<int64_t>(tid) * R + s] = sh.xs[tid] + total;
        } else {
            p.num_tokens_per_rdma_rank[static_cast<int64_t>(s) * N + (tid - R)] = total;
        }
    }

    // E1. per-rank results: the last ticket holds the global prefix at the end
    if (b == p.n_tiles - 1) {
        if (warp == 0) {
            const int32_t col = lane < R ? sh.xs[lane] + sh.wex[lane] + sh.cnt[lane] : 0;
            int32_t inc = col;
#pragma unroll
            for (int o = 1; o < kWarp; o <<= 1) {
                const int32_t y = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += y;
            }
            if (lane < R) {
                p.a.num_recv_tokens[lane] = col;
                p.a.recv_base[lane] = inc - col;
                if (p.a.host_num_recv_tokens) p.a.host_num_recv_tokens[lane] = col;
            }
            if (lane == R - 1) {
                p.a.recv_base[R] = inc;
                if (p.a.host_num_recv_tokens) p.a.host_num_recv_tokens[R] = inc;
            }
            if (p.a.host_num_recv_tokens) __threadfence_system();
        } else if (warp == 1 && lane < R) {
            // node-level receive prefix: rank r receives for its node from the
            // same-GPU-index peer m*8 + r%8 of every node m
            const int r = lane;
            int32_t run = 0;
            for (int m = 0; m < N; ++m) {
                const int peer = m * kNodeSize + r % kNodeSize;
                run += bank_wait(bank + peer * V + R + r / kNodeSize, static_cast<unsigned>(p.tps), limit, deadline,
                                 timed_out);
                p.a.recv_rdma_rank_prefix_sum[static_cast<int64_t>(r) * N + m] = run;
            }
            p.a.num_rdma_recv_tokens[r] = run;
        }
    }
    if (timed_out) flag_error(p.a.status, EP_DEV_TIMEOUT);

    // E2. the add that completed a source's expert counter word (its
    //     tps-th) has made its thread write the count out, clear the word and
    //     pass the count on to the call's word; the call's R-th add writes
    //     the per-expert receive count (see tiled_expert_done)
    if (experts_early) {
        if (ex_done) tiled_expert_call(p, tid, ex_total, ex_all);
    } else {
        constexpr int kBatch = 4;
        for (int e0 = tid; e0 < E; e0 += kBatch * B) {
            unsigned long long o_src[kBatch];
            int32_t h[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int e = e0 + u * B;
                h[u] = e < E ? hist[e] : 0;
                const unsigned long long add = (1ull << 32) | static_cast<uint32_t>(h[u]);
                o_src[u] = e < E ? atomicAdd(p.acc + static_cast<int64_t>(s) * kAccExperts + e, add) : 0ull;
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u)
                if (e0 + u * B < E) tiled_expert_done(p, s, e0 + u * B, h[u], o_src[u]);
        }
    }
    if (p.signal_ready) {
        // the row map (send_pos, recv_base) is complete once every tile is here
        __syncthreads();
        if (tid == 0) {
            __threadfence();
            if (atomicAdd(p.finished, 1u) == static_cast<unsigned>(p.n_tiles - 1)) {
                atomicExch(p.finished, 0u);
                __threadfence();
                st_release_u64(p.ready, static_cast<unsigned long long>(seq));
            }
        }
    }
    __syncthreads();  // shared state is reused by the CTA's next tile
    return sh.ticket;
}

// Fills the argument block (host).  `workspace` is laid out by
// tiled_workspace_layout(); TT a multiple of 32.
inline TiledLnArgs tiled_args(const Shape& sh, int TT, const int64_t* topk_idx, int32_t* num_tokens_per_rank,
                              int32_t* num_tokens_per_rdma_rank, int32_t* num_tokens_per_expert,
                              uint8_t* is_token_in_rank, const NotifyArgs& a, void* workspace) {
    TiledLnArgs p;
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
    p.Ep = tiled_pad4(sh.E);
    p.Vp = tiled_pad4(p.V);
    p.TT = TT;
    p.tps = sh.T > 0 ? (sh.T + TT - 1) / TT : 1;
    p.n_tiles = sh.R * p.tps;
    p.eloc_magic = sh.E_loc >= 2 ? static_cast<uint32_t>(((1ull << 32) + sh.E_loc - 1) / sh.E_loc) : 0u;
    p.stall_tile = -1;
    p.signal_ready = 0;
    p.wait_limit_ns = kDefaultWaitLimitNs;
    const TiledWorkspace w = tiled_workspace_layout(sh.R, sh.N, p.n_tiles);
    char* base = static_cast<char*>(workspace);
    p.ticket = reinterpret_cast<unsigned long long*>(base + w.ticket);
    p.finished = reinterpret_cast<unsigned*>(base + w.finished);
    p.ready = reinterpret_cast<unsigned long long*>(base + w.ready);
    p.acc = reinterpret_cast<unsigned long long*>(base + w.acc);
    p.acc_all = reinterpret_cast<unsigned long long*>(base + w.acc_all);
    p.banks = reinterpret_cast<unsigned long long*>(base + w.banks);
    p.words = reinterpret_cast<unsigned long long*>(base + w.words);
    return p;
}

}  // namespace ep
