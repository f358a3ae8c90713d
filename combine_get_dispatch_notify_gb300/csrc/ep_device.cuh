// Device helpers shared by the sm_103a kernels: inline PTX for mbarriers,
// bulk (TMA) copies, acquire/release words, streaming loads, bounded waits.
#pragma once

#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

#include "ep.h"

namespace ep {

constexpr int kWarp = 32;
constexpr int kNodeSize = 8;                       // ranks per node (NUM_MAX_NVL_PEERS)
constexpr long long kDefaultWaitLimitNs = 1000000000LL;  // 1 s: every device wait gives up after this

__device__ __forceinline__ void flag_error(int32_t* status, int bits) {
    atomicOr(reinterpret_cast<int*>(status), bits);
}

__device__ __forceinline__ long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return static_cast<long long>(t);
}

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// ---- gpu-scope acquire / release on 64-bit words (decoupled lookback) ----
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// ---- gpu-scope relaxed 64-bit words: for a word that is itself the whole
// message (no other data is read on the strength of it) ----
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// ---- streaming 16-byte loads (read-only for the kernel's lifetime) ----
__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_v4(void* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// ---- mbarrier (shared::cta) ----
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_addr(bar)),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of `parity` to complete; false when `deadline` passes first.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, long long deadline) {
    uint32_t polls = 0;
    while (!mbar_try_wait(bar, parity)) {
        if ((++polls & 63u) == 0 && globaltimer_ns() > deadline) return false;
    }
    return true;
}

// ---- bulk async copies (TMA engine, non-tensor form) ----
// global -> shared, completion counted on an mbarrier (bytes multiple of 16,
// both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_addr(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// shared -> global, tracked by the issuing thread's bulk async-groups.
__device__ __forceinline__ void bulk_s2g(void* gmem_dst, const void* smem_src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gmem_dst),
                 "r"(smem_addr(smem_src)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// All but the newest `N` groups have finished reading shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// All groups have fully completed (writes performed).
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- programmatic dependent launch ----
// Wait until the preceding kernel in the stream has completed and its writes
// are visible (returns at once when this launch was not programmatic).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Allow the next kernel in the stream to be scheduled; it still waits in
// griddep_wait() for this grid to finish before touching shared data.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- cluster barrier split into its two halves ----
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---- per-token routing helpers (layout counting) ----

__device__ __forceinline__ void count_expert(long long e, int E, int E_loc, int32_t* h_expert,
                                             uint32_t& mask, bool& bad) {
    if (e >= 0 && e < E) {
        mask |= 1u << (static_cast<int>(e) / E_loc);
        atomicAdd(&h_expert[e], 1);
    } else if (e != -1) {
        bad = true;
    }
}

// Reads the K expert ids of one token, adds each valid id to the shared
// expert histogram and returns the R-bit destination-rank mask (expert e lives
// on rank e / E_loc).  An id outside [-1, E) sets `bad` and is ignored.  Up
// to 16 ids are loaded before any is used, so their loads are in flight
// together.  For even K the ids of a token start 16-byte aligned.
__device__ __forceinline__ uint32_t token_rank_mask(const int64_t* ids, int K, int E, int E_loc,
                                                    int32_t* h_expert, bool& bad) {
    constexpr int kBatch = 16;
    uint32_t mask = 0;
    for (int k0 = 0; k0 < K; k0 += kBatch) {
        const int n = min(K - k0, kBatch);
        long long e[kBatch];
        if ((K & 1) == 0) {
#pragma unroll
            for (int i = 0; i < kBatch / 2; ++i)
                if (2 * i < n) {
                    const longlong2 v = __ldg(reinterpret_cast<const longlong2*>(ids + k0) + i);
                    e[2 * i] = v.x;
                    e[2 * i + 1] = v.y;
                }
        } else {
#pragma unroll
            for (int i = 0; i < kBatch; ++i)
                if (i < n) e[i] = __ldg(ids + k0 + i);
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i)
            if (i < n) count_expert(e[i], E, E_loc, h_expert, mask, bad);
    }
    return mask;
}

// Hint: bring [p, p + bytes) into L2 with bulk prefetches issued by one
// thread (the 16-byte-aligned interior; the ragged ends are left out).
__device__ __forceinline__ void prefetch_l2(const void* p, size_t bytes) {
    const uintptr_t a = (reinterpret_cast<uintptr_t>(p) + 15u) & ~uintptr_t(15);
    const uintptr_t b = (reinterpret_cast<uintptr_t>(p) + bytes) & ~uintptr_t(15);
    constexpr uintptr_t kChunk = 1u << 16;
    for (uintptr_t c = a; c < b; c += kChunk) {
        const uint32_t n = static_cast<uint32_t>(b - c < kChunk ? b - c : kChunk);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(c), "r"(n) : "memory");
    }
}

// Rank mask -> node mask (node of rank r is r / 8).
__device__ __forceinline__ uint32_t node_bits(uint32_t m, int R, int N) {
    if (R <= kNodeSize) return m != 0u ? 1u : 0u;
    uint32_t nm = 0;
    for (int n = 0; n < N; ++n) nm |= ((m >> (kNodeSize * n)) & 0xffu) ? (1u << n) : 0u;
    return nm;
}

// 4 mask bits -> 4 bytes holding 0 or 1 (bit i -> byte i, little-endian).
__device__ __forceinline__ uint32_t bits4_to_bytes(uint32_t b) {
    return (b & 1u) | ((b & 2u) << 7) | ((b & 4u) << 14) | ((b & 8u) << 21);
}

// Writes one is_token_in_rank row (R bytes of 0/1) from the rank mask.
__device__ __forceinline__ void write_membership_row(uint8_t* row, uint32_t mask, int R) {
    if ((R & 15) == 0) {
        for (int w = 0; w < R / 16; ++w) {
            const uint32_t m = mask >> (16 * w);
            uint4 v;
            v.x = bits4_to_bytes(m & 0xfu);
            v.y = bits4_to_bytes((m >> 4) & 0xfu);
            v.z = bits4_to_bytes((m >> 8) & 0xfu);
            v.w = bits4_to_bytes((m >> 12) & 0xfu);
            *reinterpret_cast<uint4*>(row + 16 * w) = v;
        }
    } else if ((R & 3) == 0) {
        for (int w = 0; w < R / 4; ++w)
            *reinterpret_cast<uint32_t*>(row + 4 * w) = bits4_to_bytes((mask >> (4 * w)) & 0xfu);
    } else {
        for (int r = 0; r < R; ++r) row[r] = static_cast<uint8_t>((mask >> r) & 1u);
    }
}

}  // namespace ep

namespace ep {

// Host: sets what a launch of `kernel` with `smem` dynamic shared bytes needs
// on the current device (the largest shared / smallest L1 split when
// `max_shared`, the dynamic shared limit above 48 KB, non-portable cluster
// sizes), once per kernel and device; later launches find it done.
cudaError_t prepare_kernel(const void* kernel, size_t smem, bool max_shared, bool nonportable_cluster);

// Host: launch `kernel` as a programmatic dependent of the previous work in
// `stream` (its prologue may overlap the predecessor's tail).  `max_shared`
// asks for the largest shared-memory / smallest L1 split (kernels that stage
// data in shared memory); other kernels keep the default split, which gives
// their loads more L1.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, unsigned cluster_x, bool max_shared,
                              Args&&... args) {
    const cudaError_t e =
        prepare_kernel(reinterpret_cast<const void*>(kernel), smem, max_shared, cluster_x > 8);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    unsigned n = 1;
    if (cluster_x > 0) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = cluster_x;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        n = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace ep
