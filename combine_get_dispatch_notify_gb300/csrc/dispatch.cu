// Step 3 - dispatch ([RT] intranode/internodeDispatch receive side; [AR] 4.1
// SrcInfo).  Token (s,t) goes to pool row recv_base[r] + send_pos[s][t][r]
// of every rank r it is routed to.
//
// Persistent CTAs (2 per SM, 3 for rows of 8 KB or less) walk work units
// (token, row part): with a stride of the grid, or - when the caller passes a
// `sched` counter and CTAs have more units than ring slots - the first
// ring-full with that stride and every later unit from the counter, so CTAs
// on SMs that write faster take more.  Each CTA runs a shared-memory ring of
// `slots` buffers fed by the TMA engine (bulk, non-tensor copies):
//   warp 0 (producer): issues the bulk global->shared copies of its first
//        ring-full of row parts before waiting on notify (x is an input, so
//        at small sizes all of x is in shared memory by the time the row map
//        exists); then per unit reads the send_pos row (lane r = rank r),
//        writes the destination rows into the slot descriptor and, for units
//        beyond the first ring-full, waits for a free slot and issues the
//        copy.  A slot's "full" mbarrier completes on two arrivals (copy
//        armed, descriptor written) plus the copy's bytes;
//   warp 1 (storer, one thread): waits "full", issues one bulk
//        shared->global copy per destination, commits them as a bulk group,
//        and frees the slot of the unit `lag` groups back once that group
//        has been read out (up to 6 groups in flight, the rest of the ring
//        is load-ahead);
//   warps 2-3 (metadata): write recv_topk_idx / recv_topk_w / recv_src_info
//        for the destination rows of each token with plain stores.
// Each row is read from HBM once and written once per destination; no
// atomics decide placement (send_pos is precomputed by notify; the counter
// only decides which CTA copies a unit, so results do not depend on it).  Every wait
// is bounded; a wait that runs out sets EP_DEV_TIMEOUT and the CTA drains its
// in-flight copies before exiting.
#include "ep_device.cuh"
#include "ep_internal.h"
#include "ln_tiled.cuh"

namespace ep {
namespace {

constexpr int kDispatchThreads = 128;
constexpr int kMaxSlots = 16;
constexpr int kSmemPerSm = 200 * 1024;    // ring bytes per SM, split over its CTAs
constexpr int kMaxPartBytes = 32 * 1024;
constexpr int kStoreLag = 6;  // bulk store groups in flight per CTA

struct SlotDesc {
    int n;               // destinations in rows[], -1 = end of stream
    uint32_t bytes;      // bytes of this part
    long long part_off;  // byte offset of the part inside the row
    long long rows[32];  // pool row per destination (-1 = skip)
};

struct DispatchArgs {
    const uint8_t* x;
    const int64_t* topk_idx;
    const float* topk_w;
    const int32_t* send_pos;
    const int64_t* recv_base;
    long long capacity;
    uint8_t* recv_x;
    int64_t* recv_topk_idx;
    float* recv_topk_w;
    int32_t* recv_src_info;
    const int32_t* ll_slot_pos;  // low-latency layout: [R*T][K] row in the slot's expert buffer, else NULL
    long long ll_cap;            // rows per expert buffer (low-latency layout)
    int E;
    const float* x_scales;   // [R*T][num_scales] or NULL (FP8 rows)
    float* recv_x_scales;    // [capacity][num_scales] or NULL
    int num_scales;
    int32_t* status;
    int R, T, K, E_loc, parts, slots;
    uint32_t part_bytes;
    long long row_bytes;
    long long num_units;
    long long wait_limit_ns;
    int stall_release_cta;  // test hook: this CTA's storer never frees a slot (-1: none)
    unsigned long long* sched;  // unit counter (dynamic assignment), or NULL (static)
    int coherent;  // 1: send_pos / recv_base are written by this same launch (read through L2)
};

// Destination row this lane stands for, or -1: lane r = rank r through
// send_pos, or in the low-latency layout lane k = top-k slot k, whose row is
// expert * cap + slot_pos.  Rows outside the receive arrays are refused and
// reported.
__device__ __forceinline__ long long lane_row(const DispatchArgs& p, const long long* base, long long g,
                                              int lane) {
    if (p.ll_slot_pos != nullptr) {
        if (lane >= p.K) return -1;
        const long long e = __ldg(p.topk_idx + g * p.K + lane);
        const int32_t pos = __ldg(p.ll_slot_pos + g * p.K + lane);
        if (e < 0 || pos < 0) return -1;
        if (e >= p.E || pos >= p.ll_cap) {
            flag_error(p.status, EP_DEV_INCONSISTENT);
            return -1;
        }
        return e * p.ll_cap + pos;
    }
    if (lane >= p.R) return -1;
    const int32_t sp = p.coherent ? __ldcg(p.send_pos + g * p.R + lane) : __ldg(p.send_pos + g * p.R + lane);
    if (sp < 0) return -1;
    const long long row = base[lane] + sp;
    if (row >= p.capacity) {
        flag_error(p.status, EP_DEV_CAPACITY);
        return -1;
    }
    if (row >= base[lane + 1]) {
        flag_error(p.status, EP_DEV_INCONSISTENT);
        return -1;
    }
    return row;
}

// cp.async.bulk.wait_group.read takes an immediate: dispatch on the lag.
__device__ __forceinline__ void bulk_wait_read_lag(int lag) {
    switch (lag) {
        case 1: bulk_wait_read<1>(); break;
        case 2: bulk_wait_read<2>(); break;
        case 3: bulk_wait_read<3>(); break;
        case 4: bulk_wait_read<4>(); break;
        case 5: bulk_wait_read<5>(); break;
        default: bulk_wait_read<6>(); break;
    }
}

// Shared-memory ring of one CTA and its unit schedule.
struct Ring {
    int S;
    uint8_t* data;
    uint64_t* full;
    uint64_t* empty;
    SlotDesc* desc;
    long long* base;
    bool dynamic;
    long long P0;  // units this CTA takes with the static stride
    int pre;       // of them, loaded before the dependency wait
    unsigned long long dyn_units, last_grab;
};

// Bytes of the ring region (data, mbarriers, descriptors, recv_base copy).
__host__ __device__ inline size_t ring_bytes(int slots, uint32_t part_bytes) {
    return static_cast<size_t>(slots) * part_bytes + 2 * slots * sizeof(uint64_t) + slots * sizeof(SlotDesc) +
           33 * sizeof(long long);
}

// Unit assignment.  Static: CTA b takes units b, b + grid, ...
// Dynamic (counter): CTA b takes its first P0 units that way (they are the
// ones loaded before the dependency wait), and every later unit from the
// counter, so CTAs on faster SMs take more of them.  Each CTA's producer
// keeps one counter grab in flight and ends on exactly one grab past the
// end; the grab that sees the last value of the call resets the counter,
// so every call leaves it zero for the next.
// With fewer units per CTA than ring slots there is (almost) nothing left
// to balance after the first ring-full, and the counter's grabs would only
// add their latency: such calls keep the static split.
__device__ __forceinline__ Ring ring_setup(const DispatchArgs& p, uint8_t* smem) {
    Ring rg;
    rg.S = p.slots;
    rg.data = smem;
    rg.full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(rg.S) * p.part_bytes);
    rg.empty = rg.full + rg.S;
    rg.desc = reinterpret_cast<SlotDesc*>(rg.empty + rg.S);
    rg.base = reinterpret_cast<long long*>(rg.desc + rg.S);
    const long long per_cta = p.num_units / gridDim.x;
    rg.dynamic = p.sched != nullptr && per_cta > rg.S;
    const long long units_here =
        blockIdx.x < p.num_units ? (p.num_units - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    rg.P0 = rg.dynamic ? (per_cta < rg.S ? per_cta : rg.S) : units_here;
    rg.pre = static_cast<int>(rg.P0 < rg.S ? rg.P0 : rg.S);
    rg.dyn_units = rg.dynamic ? static_cast<unsigned long long>(p.num_units - rg.P0 * gridDim.x) : 0ull;
    rg.last_grab = rg.dyn_units + gridDim.x - 1;  // value of the call's final grab
    return rg;
}

// mbarrier set-up, then the first ring-full of row parts: x is an input of
// the step, not written by layout or notify, so it is loaded while the row
// map is still being computed.
__device__ __forceinline__ void ring_prologue(const DispatchArgs& p, const Ring& rg) {
    const int tid = threadIdx.x;
    if (tid == 0) {
        for (int i = 0; i < rg.S; ++i) {
            mbar_init(&rg.full[i], 2);  // arrivals: row part armed, descriptor written
            mbar_init(&rg.empty[i], 1);
        }
        fence_mbarrier_init();
    }
    __syncthreads();
    if (tid == 0) {
        long long u = blockIdx.x;
        for (int i = 0; i < rg.pre; ++i, u += gridDim.x) {
            const long long g = u / p.parts;
            const long long off = (u - g * p.parts) * static_cast<long long>(p.part_bytes);
            const long long left = p.row_bytes - off;
            const uint32_t bytes = left < p.part_bytes ? static_cast<uint32_t>(left) : p.part_bytes;
            mbar_arrive_expect_tx(&rg.full[i], bytes);
            bulk_g2s(rg.data + static_cast<size_t>(i) * p.part_bytes, p.x + g * p.row_bytes + off, bytes,
                     &rg.full[i]);
        }
    }
}

// The row map never became available (a bounded wait ran out): give the
// prefetched slots their second arrival, wait for their copies, and keep the
// counter's grab count exact (units are left undone), then return.
__device__ void ring_abort(const DispatchArgs& p, const Ring& rg) {
    if (threadIdx.x != 0) return;
    for (int i = 0; i < rg.pre; ++i) mbar_arrive(&rg.full[i]);
    for (int i = 0; i < rg.pre; ++i)
        if (!mbar_wait(&rg.full[i], 0, globaltimer_ns() + p.wait_limit_ns)) flag_error(p.status, EP_DEV_TIMEOUT);
    if (rg.dynamic) {
        unsigned long long grab = atomicAdd(p.sched, 1ull);
        for (;;) {
            if (grab == rg.last_grab) {
                atomicExch(p.sched, 0ull);
                break;
            }
            if (grab >= rg.dyn_units) break;
            grab = atomicAdd(p.sched, 1ull);
        }
    }
}

// Producer, storer and metadata roles, once base[] holds recv_base.
__device__ void dispatch_roles(const DispatchArgs& p, const Ring& rg) {
    const int S = rg.S;
    uint8_t* data = rg.data;
    uint64_t* full = rg.full;
    uint64_t* empty = rg.empty;
    SlotDesc* desc = rg.desc;
    const long long* base = rg.base;
    const bool dynamic = rg.dynamic;
    const long long P0 = rg.P0;
    const int pre = rg.pre;
    const unsigned long long dyn_units = rg.dyn_units, last_grab = rg.last_grab;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (warp == 0) {
        // ---------------- producer ----------------
        int k = 0;  // units (then the end marker) handed to the storer
        bool ok = true;
        unsigned long long grab = 0;  // lane 0: value of the counter grab in flight
        bool grab_pending = false;
        if (dynamic && lane == 0) {
            grab = atomicAdd(p.sched, 1ull);  // in flight while the static units are handed over
            grab_pending = true;
        }
        for (;;) {
            long long u;
            if (k < P0) {
                u = blockIdx.x + static_cast<long long>(k) * gridDim.x;
            } else if (!dynamic) {
                break;
            } else {
                unsigned long long got = grab;
                if (lane == 0) {
                    grab_pending = false;
                    if (got == last_grab) {
                        atomicExch(p.sched, 0ull);
                    } else if (got < dyn_units) {
                        grab = atomicAdd(p.sched, 1ull);  // the next one, in flight during this unit
                        grab_pending = true;
                    }
                }
                got = __shfl_sync(0xffffffffu, got, 0);
                if (got >= dyn_units) break;
                u = P0 * gridDim.x + static_cast<long long>(got);
            }
            const long long g = u / p.parts;
            const int part = static_cast<int>(u - g * p.parts);
            const long long row = lane_row(p, base, g, lane);
            const unsigned valid = __ballot_sync(0xffffffffu, row >= 0);
            const int slot = k % S;
            const long long off = static_cast<long long>(part) * p.part_bytes;
            const long long left = p.row_bytes - off;
            const uint32_t bytes = left < p.part_bytes ? static_cast<uint32_t>(left) : p.part_bytes;
            if (k >= pre) {  // not prefetched: wait for the slot, then load
                bool got = true;
                if (lane == 0)
                    got = mbar_wait(&empty[slot], ((k / S) - 1) & 1, globaltimer_ns() + p.wait_limit_ns);
                if (!__shfl_sync(0xffffffffu, got, 0)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(&full[slot], bytes);
                    bulk_g2s(data + static_cast<size_t>(slot) * p.part_bytes, p.x + g * p.row_bytes + off,
                             bytes, &full[slot]);
                }
            }
            if (row >= 0) desc[slot].rows[__popc(valid & lanemask_lt())] = row;
            if (lane == 0) {
                desc[slot].n = __popc(valid);
                desc[slot].bytes = bytes;
                desc[slot].part_off = off;
            }
            __syncwarp();  // every lane's descriptor writes precede the release below
            if (lane == 0) mbar_arrive(&full[slot]);
            ++k;
        }
        if (ok) {  // end-of-stream marker (both arrivals, no data)
            const int slot = k % S;
            bool got = true;
            if (k >= S && lane == 0)
                got = mbar_wait(&empty[slot], ((k / S) - 1) & 1, globaltimer_ns() + p.wait_limit_ns);
            if (__shfl_sync(0xffffffffu, got, 0)) {
                if (lane == 0) {
                    desc[slot].n = -1;
                    mbar_arrive(&full[slot]);
                    mbar_arrive(&full[slot]);
                }
                ++k;
            } else {
                ok = false;
            }
        }
        if (lane == 0) {
            if (!ok) flag_error(p.status, EP_DEV_TIMEOUT);
            // A wait that ran out left this CTA's grabs unfinished: keep grabbing
            // (the units are left undone) until one lands past the end, so the
            // call's grab count, and with it the counter reset, stay exact.
            while (grab_pending) {
                if (grab == last_grab) {
                    atomicExch(p.sched, 0ull);
                    grab_pending = false;
                } else if (grab >= dyn_units) {
                    grab_pending = false;
                } else {
                    grab = atomicAdd(p.sched, 1ull);
                }
            }
            // Drain: the newest phase armed on each slot has completed, so no
            // bulk copy into shared memory outlives the CTA.  (A wait can only
            // run out after every prefetched unit was handed over, so no phase
            // is left with one arrival.)
            for (int x = 0; x < S; ++x) {
                const int phases = k > x ? (k - x + S - 1) / S : 0;
                if (phases > 0 &&
                    !mbar_wait(&full[x], (phases - 1) & 1, globaltimer_ns() + p.wait_limit_ns))
                    flag_error(p.status, EP_DEV_TIMEOUT);
            }
        }
    } else if (warp == 1) {
        // ---------------- storer ----------------
        // Up to `lag` bulk groups stay in flight; the other slots are
        // load-ahead for the producer, which waits for unit k - S's slot and
        // so never for a unit it has not handed over (lag <= S - 1).
        const int lag = S - 1 < kStoreLag ? S - 1 : kStoreLag;
        if (lane == 0) {
            for (int k = 0;; ++k) {
                const int slot = k % S;
                if (!mbar_wait(&full[slot], (k / S) & 1, globaltimer_ns() + p.wait_limit_ns)) {
                    flag_error(p.status, EP_DEV_TIMEOUT);
                    break;
                }
                const int n = desc[slot].n;
                if (n < 0) break;
                fence_proxy_async_smem();
                const uint8_t* src = data + static_cast<size_t>(slot) * p.part_bytes;
                const uint32_t bytes = desc[slot].bytes;
                const long long off = desc[slot].part_off;
                for (int j = 0; j < n; ++j) {
                    const long long row = desc[slot].rows[j];
                    if (row >= 0) bulk_s2g(p.recv_x + row * p.row_bytes + off, src, bytes);
                }
                bulk_commit();
                if (k >= lag) {  // unit k - lag's group has been read out: free its slot
                    bulk_wait_read_lag(lag);
                    if (static_cast<int>(blockIdx.x) != p.stall_release_cta) mbar_arrive(&empty[(k - lag) % S]);
                }
            }
            bulk_wait_all();
        }
    } else {
        // ---------------- metadata ----------------
        // (cached mode passes no top-k arrays; recv_src_info may be omitted too)
        const bool with_topk = p.recv_topk_idx != nullptr;
        const bool with_src = p.recv_src_info != nullptr;
        const bool with_scales = p.recv_x_scales != nullptr;
        const int mw = warp - 2;
        int i = 0;
        for (long long u = blockIdx.x; (with_topk || with_src || with_scales) && u < p.num_units;
             u += gridDim.x) {
            if (u % p.parts != 0) continue;
            if ((i++ & 1) != mw) continue;
            const long long g = u / p.parts;
            const int s = static_cast<int>(g / p.T), t = static_cast<int>(g - static_cast<long long>(s) * p.T);
            const long long my_row = lane_row(p, base, g, lane);
            long long e = -1;
            float w = 0.0f;
            int owner = -1;
            if (with_topk && lane < p.K) {
                e = __ldg(p.topk_idx + g * p.K + lane);
                w = __ldg(p.topk_w + g * p.K + lane);
                owner = e >= 0 ? static_cast<int>(e / p.E_loc) : -1;
            }
            // the token's FP8 scales, loaded once (lane j holds scales j, j+32, ...)
            constexpr int kScaleRegs = 4;
            const bool scales_in_regs = with_scales && p.num_scales <= kScaleRegs * kWarp;
            float sc[kScaleRegs];
#pragma unroll
            for (int c = 0; c < kScaleRegs; ++c) {
                const int j = lane + c * kWarp;
                sc[c] = (scales_in_regs && j < p.num_scales) ? __ldg(p.x_scales + g * p.num_scales + j) : 0.0f;
            }
            unsigned m = __ballot_sync(0xffffffffu, my_row >= 0);
            while (m) {
                const int r = __ffs(m) - 1;  // rank r (or, low-latency layout, slot r)
                m &= m - 1;
                const long long row = __shfl_sync(0xffffffffu, my_row, r);
                if (with_topk && lane < p.K) {
                    const bool here = owner == r;
                    p.recv_topk_idx[row * p.K + lane] = here ? e - static_cast<long long>(r) * p.E_loc : -1;
                    p.recv_topk_w[row * p.K + lane] = here ? w : 0.0f;
                }
                if (with_src && lane == 0) *reinterpret_cast<int2*>(p.recv_src_info + row * 2) = make_int2(s, t);
                if (scales_in_regs) {  // the token's FP8 block scales travel with its row
#pragma unroll
                    for (int c = 0; c < kScaleRegs; ++c) {
                        const int j = lane + c * kWarp;
                        if (j < p.num_scales) p.recv_x_scales[row * p.num_scales + j] = sc[c];
                    }
                } else if (with_scales) {
                    for (int j = lane; j < p.num_scales; j += kWarp)
                        p.recv_x_scales[row * p.num_scales + j] = __ldg(p.x_scales + g * p.num_scales + j);
                }
            }
        }
    }
}


// Layout, notify and dispatch in one launch ([RT] internodeNotifyDispatch
// followed by internodeDispatch; the pages' notify hands its results to
// dispatch through per-channel head/tail words, here through one `ready`
// word).  The dispatch CTAs load their first ring-full of x rows, then work
// on layout + notify tiles as the tiled form's kernel does (see ln_tiled.cuh:
// the first tile by block index, later ones by ticket) until none is left,
// then wait - bounded - until the call's row map is complete and run the
// dispatch roles on it, reading send_pos and recv_base through L2 since this
// launch wrote them.  A CTA waits only on tiles of CTAs that are already
// running, so no co-residency is needed.
__global__ void __launch_bounds__(kDispatchThreads)
layout_notify_dispatch_kernel(DispatchArgs p, TiledLnArgs ln, uint32_t tile_smem_off) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ TiledShared sh;
    __shared__ int s_ok;
    griddep_launch_dependents();
    const Ring rg = ring_setup(p, smem);
    ring_prologue(p, rg);
    griddep_wait();  // top-k ids written by the preceding kernel are visible
    // Thread 0 is held while its row copies are taken in, thread 32 while the
    // ids prefetch is: a third thread takes the tickets.
    if (threadIdx.x == kWarp) tiled_prefetch_ids(ln, static_cast<int>(blockIdx.x));
    int32_t* dyn = reinterpret_cast<int32_t*>(smem + tile_smem_off);
    int b = blockIdx.x < static_cast<unsigned>(ln.n_tiles) ? static_cast<int>(blockIdx.x) : -1;
    if (b < 0) {  // no tile of its own: one ticket, for the call's sequence number
        if (threadIdx.x == 2 * kWarp) tiled_ticket_done(ln, sh, atomicAdd(ln.ticket, 1ull));
        __syncthreads();
    }
    while (b >= 0) b = tiled_tile(ln, sh, dyn, b, 2 * kWarp);
    const unsigned long long seq = sh.seq;
    if (threadIdx.x == 0) {
        const long long deadline = globaltimer_ns() + p.wait_limit_ns;
        unsigned long long w = ld_acquire_u64(ln.ready);
        uint32_t polls = 0;
        bool ok = true;
        while (w != seq) {
            if ((++polls & 15u) == 0 && globaltimer_ns() > deadline) {
                ok = false;
                break;
            }
            __nanosleep(64);
            w = ld_acquire_u64(ln.ready);
        }
        if (!ok) flag_error(p.status, EP_DEV_TIMEOUT);
        s_ok = ok;
    }
    __syncthreads();
    if (!s_ok) {
        ring_abort(p, rg);
        return;
    }
    if (threadIdx.x <= p.R) rg.base[threadIdx.x] = __ldcg(p.recv_base + threadIdx.x);
    __syncthreads();
    dispatch_roles(p, rg);
}

__global__ void __launch_bounds__(kDispatchThreads) dispatch_kernel(DispatchArgs p) {
    extern __shared__ __align__(128) uint8_t smem[];
    griddep_launch_dependents();
    const Ring rg = ring_setup(p, smem);
    ring_prologue(p, rg);
    griddep_wait();  // send_pos / recv_base from notify are visible from here on
    if (p.recv_base != nullptr && threadIdx.x <= p.R) rg.base[threadIdx.x] = p.recv_base[threadIdx.x];
    __syncthreads();
    dispatch_roles(p, rg);
}

}  // namespace

namespace {

// Sizes the ring for the row bytes in `p` (leaving `extra_per_cta` shared
// bytes per CTA for other uses) and returns the grid and dynamic shared bytes.
cudaError_t size_dispatch(DispatchArgs& p, long long tokens, size_t extra_per_cta, long long* grid_out,
                          size_t* smem_out) {
    const int sms = device_sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const long long row_bytes = p.row_bytes;
    // Two CTAs (two storer threads) per SM for rows above 8 KB; three for
    // smaller rows (FP8 at H = 7168), whose stores are too small for two
    // threads to issue at full bandwidth.
    const int ctas_per_sm = row_bytes <= 8192 ? 3 : 2;
    const long long grid_target = static_cast<long long>(sms) * ctas_per_sm;
    // Row parts: at most 32 KB, and split further (down to 2 KB) while there
    // are fewer than 8 units per CTA (4 for rows of 8 KB or less, whose
    // halves are too small to pay for the extra units).  Parts are
    // multiples of 16 bytes.
    long long part = row_bytes < kMaxPartBytes ? row_bytes : kMaxPartBytes;
    auto units_for = [&](long long pb) { return tokens * ((row_bytes + pb - 1) / pb); };
    const long long min_units = (row_bytes <= 8192 ? 4 : 8) * grid_target;
    while (part > 2048 && units_for(part) < min_units) part = ((part / 2) + 15) / 16 * 16;
    const int parts = static_cast<int>((row_bytes + part - 1) / part);
    const long long avail = kSmemPerSm / ctas_per_sm - static_cast<long long>(extra_per_cta);
    int slots = static_cast<int>(avail / part);
    slots = slots < 2 ? 2 : (slots > kMaxSlots ? kMaxSlots : slots);
    p.parts = parts;
    p.slots = slots;
    p.part_bytes = static_cast<uint32_t>(part);
    p.num_units = tokens * parts;
    *smem_out = ring_bytes(slots, p.part_bytes);
    *grid_out = p.num_units < grid_target ? p.num_units : grid_target;
    return cudaSuccess;
}

// Sizes the ring for the row bytes in `p` and launches.
cudaError_t launch_dispatch_args(DispatchArgs& p, long long tokens, cudaStream_t stream) {
    long long grid = 0;
    size_t smem = 0;
    const cudaError_t e = size_dispatch(p, tokens, 0, &grid, &smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(dispatch_kernel, dim3(static_cast<unsigned>(grid)), dim3(kDispatchThreads), smem,
                      stream, 0, true, p);
}

DispatchArgs base_args(const Shape& sh, int32_t* status) {
    DispatchArgs p = {};
    p.status = status;
    p.wait_limit_ns = kDefaultWaitLimitNs;
    p.stall_release_cta = -1;
    p.sched = nullptr;
    p.R = sh.R;
    p.T = sh.T;
    p.K = sh.K;
    p.E = sh.E;
    p.E_loc = sh.E_loc;
    return p;
}

}  // namespace

cudaError_t launch_dispatch(const Shape& sh, const void* x, int x_elem_bytes, const float* x_scales,
                            int num_scales, const int64_t* topk_idx, const float* topk_w,
                            const int32_t* send_pos, const int64_t* recv_base, int64_t capacity_rows,
                            void* recv_x, float* recv_x_scales, int64_t* recv_topk_idx,
                            float* recv_topk_w, int32_t* recv_src_info, int32_t* status,
                            unsigned long long* sched, cudaStream_t stream, int stall_release_cta,
                            long long wait_limit_ns) {
    const long long tokens = static_cast<long long>(sh.R) * sh.T;
    if (tokens == 0) return cudaSuccess;
    DispatchArgs p = base_args(sh, status);
    p.sched = sched;
    p.stall_release_cta = stall_release_cta;
    p.wait_limit_ns = wait_limit_ns;
    p.x = static_cast<const uint8_t*>(x);
    p.x_scales = x_scales;
    p.recv_x_scales = recv_x_scales;
    p.num_scales = num_scales;
    p.topk_idx = topk_idx;
    p.topk_w = topk_w;
    p.send_pos = send_pos;
    p.recv_base = recv_base;
    p.capacity = capacity_rows;
    p.recv_x = static_cast<uint8_t*>(recv_x);
    p.recv_topk_idx = recv_topk_idx;
    p.recv_topk_w = recv_topk_w;
    p.recv_src_info = recv_src_info;
    p.row_bytes = static_cast<long long>(sh.H) * x_elem_bytes;
    return launch_dispatch_args(p, tokens, stream);
}

cudaError_t launch_layout_notify_dispatch(const Shape& sh, const int64_t* topk_idx, const float* topk_w,
                                          const uint16_t* x, int32_t* num_tokens_per_rank,
                                          int32_t* num_tokens_per_rdma_rank, int32_t* num_tokens_per_expert,
                                          uint8_t* is_token_in_rank, const NotifyArgs& a, void* workspace,
                                          int64_t capacity_rows, uint16_t* recv_x, int64_t* recv_topk_idx,
                                          float* recv_topk_w, int32_t* recv_src_info, int32_t* status,
                                          unsigned long long* sched, int tile_tokens, int stall_tile,
                                          long long wait_limit_ns, cudaStream_t stream) {
    const long long tokens = static_cast<long long>(sh.R) * sh.T;
    if (tokens == 0)  // nothing to dispatch: layout + notify alone
        return launch_layout_notify_tiled(sh, topk_idx, num_tokens_per_rank, num_tokens_per_rdma_rank,
                                          num_tokens_per_expert, is_token_in_rank, a, workspace, tile_tokens,
                                          stall_tile, wait_limit_ns, stream);
    const int TT = tiled_tile_tokens(sh, tile_tokens);
    TiledLnArgs ln = tiled_args(sh, TT, topk_idx, num_tokens_per_rank, num_tokens_per_rdma_rank,
                                num_tokens_per_expert, is_token_in_rank, a, workspace);
    ln.stall_tile = stall_tile;
    ln.wait_limit_ns = wait_limit_ns;
    ln.signal_ready = 1;
    DispatchArgs p = base_args(sh, status);
    p.sched = sched;
    p.wait_limit_ns = wait_limit_ns;
    p.coherent = 1;
    p.x = reinterpret_cast<const uint8_t*>(x);
    p.topk_idx = topk_w != nullptr ? topk_idx : nullptr;  // top-k fields travel only with weights
    p.topk_w = topk_w;
    p.send_pos = a.send_pos;
    p.recv_base = a.recv_base;
    p.capacity = capacity_rows;
    p.recv_x = reinterpret_cast<uint8_t*>(recv_x);
    p.recv_topk_idx = recv_topk_idx;
    p.recv_topk_w = recv_topk_w;
    p.recv_src_info = recv_src_info;
    p.row_bytes = sh.row_bytes();
    const size_t tile_smem = sizeof(int32_t) * tiled_smem_words(sh.E, TT, sh.R + sh.N);
    long long grid = 0;
    size_t ring = 0;
    cudaError_t e = size_dispatch(p, tokens, tile_smem + sizeof(TiledShared) + 1024, &grid, &ring);
    if (e != cudaSuccess) return e;
    const size_t off = (ring + 15) / 16 * 16;
    return launch_pdl(layout_notify_dispatch_kernel, dim3(static_cast<unsigned>(grid)), dim3(kDispatchThreads),
                      off + tile_smem, stream, 0, true, p, ln, static_cast<uint32_t>(off));
}

cudaError_t launch_ll_dispatch(const Shape& sh, const uint16_t* x, const int64_t* topk_idx,
                               const int32_t* slot_pos, int cap, uint16_t* recv_x,
                               int32_t* recv_src_info, int32_t* status, unsigned long long* sched,
                               cudaStream_t stream) {
    const long long tokens = static_cast<long long>(sh.R) * sh.T;
    if (tokens == 0) return cudaSuccess;
    DispatchArgs p = base_args(sh, status);
    p.sched = sched;
    p.x = reinterpret_cast<const uint8_t*>(x);
    p.topk_idx = topk_idx;
    p.ll_slot_pos = slot_pos;
    p.ll_cap = cap;
    p.capacity = static_cast<long long>(sh.E) * cap;
    p.recv_x = reinterpret_cast<uint8_t*>(recv_x);
    p.recv_src_info = recv_src_info;
    p.row_bytes = sh.row_bytes();
    return launch_dispatch_args(p, tokens, stream);
}

}  // namespace ep
