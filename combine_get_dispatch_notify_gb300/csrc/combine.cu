// Step 4 - combine ([RT] intranode/internodeCombine; [AR] 4.2 combine
// routing).  combined_x[s][t] = bf16_rne(sum over contributing ranks r, in
// ascending order, of float(y[recv_base[r] + send_pos[s][t][r]])).
//
// Work unit = (token, column slice of 32 lanes x 2 chunks x 16 bytes).  A
// warp reads the token's send_pos row (lane r = rank r), compacts the
// contributing rows in ascending rank order into shared memory, then each
// lane loads its two 16-byte chunks from up to 4 contributing rows at a time
// (8 independent loads in flight per lane), accumulates in fp32 in rank
// order, rounds to bf16 and stores.  The chunks of a lane are 512 bytes
// apart, so every load instruction of a warp covers a contiguous 512-byte
// segment; slices of one token go to neighbouring warps.  Three 256-thread
// CTAs per SM with the default L1/shared split (the gather uses L1 for the
// row map).  No atomics: the result is deterministic and bit-identical to a
// sequential fp32 sum in the same order.
#include <cuda_bf16.h>

#include "ep_device.cuh"
#include "ep_internal.h"

namespace ep {
namespace {

constexpr int kCombineThreads = 256;
constexpr int kCombineWarps = kCombineThreads / kWarp;
constexpr int kCombineBlocksPerSm = 3;
constexpr int kBatch = 4;  // contributing rows loaded together
constexpr int kCpl = 2;    // 16-byte chunks per lane per unit

struct CombineArgs {
    const uint8_t* y;
    const float* y_w;
    const int32_t* send_pos;
    const int64_t* recv_base;
    uint8_t* out;
    float* out_w;
    int32_t* status;
    long long y_rows;
    // low-latency layout: rows come from (topk_idx, slot_pos) as expert * cap +
    // slot_pos, and each contribution is weighted by its routing weight
    const int64_t* topk_idx;
    const float* topk_w;
    const int32_t* ll_slot_pos;
    long long ll_cap;
    int E;
    int R, K;
    long long row_bytes;
    int chunks;  // 16-byte chunks per row
    int slices;  // ceil(chunks / (32 * kCpl))
    long long num_units;
};

__device__ __forceinline__ void add_bf16x8(float (&acc)[8], const uint4& v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc[2 * i] += __uint_as_float(w[i] << 16);
        acc[2 * i + 1] += __uint_as_float(w[i] & 0xffff0000u);
    }
}

__device__ __forceinline__ uint4 pack_bf16x8(const float (&acc)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
        w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// acc += w * v per element, one fused multiply-add (rounded once) per step.
__device__ __forceinline__ void fma_bf16x8(float (&acc)[8], float w, const uint4& v) {
    const uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc[2 * i] = __fmaf_rn(w, __uint_as_float(x[i] << 16), acc[2 * i]);
        acc[2 * i + 1] = __fmaf_rn(w, __uint_as_float(x[i] & 0xffff0000u), acc[2 * i + 1]);
    }
}

template <bool kWeighted>
__global__ void __launch_bounds__(kCombineThreads, kCombineBlocksPerSm)
combine_kernel(CombineArgs p) {
    __shared__ long long s_base[33];
    __shared__ long long s_rows[kCombineWarps][32];
    __shared__ float s_wts[kCombineWarps][32];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    griddep_launch_dependents();
    griddep_wait();  // the expert outputs and the row map are visible from here on
    if (!kWeighted && tid <= p.R) s_base[tid] = p.recv_base[tid];
    __syncthreads();
    long long* rows = s_rows[warp];
    float* wts = s_wts[warp];
    const long long warps_total = static_cast<long long>(gridDim.x) * kCombineWarps;

    for (long long u = static_cast<long long>(blockIdx.x) * kCombineWarps + warp; u < p.num_units;
         u += warps_total) {
        const long long g = u / p.slices;
        const int slice = static_cast<int>(u - g * p.slices);
        long long row = -1;
        float wt = 0.0f;
        if (kWeighted) {  // lane k = top-k slot k
            if (lane < p.K) {
                const long long e = __ldg(p.topk_idx + g * p.K + lane);
                const int32_t pos = __ldg(p.ll_slot_pos + g * p.K + lane);
                if (e >= 0 && pos >= 0) {
                    if (e >= p.E || pos >= p.ll_cap) {
                        flag_error(p.status, EP_DEV_INCONSISTENT);
                    } else {
                        row = e * p.ll_cap + pos;
                        wt = __ldg(p.topk_w + g * p.K + lane);
                    }
                }
            }
        } else {  // lane r = rank r
            const int32_t sp = lane < p.R ? __ldg(p.send_pos + g * p.R + lane) : -1;
            if (sp >= 0) {
                row = s_base[lane] + sp;
                if (row >= p.y_rows) {
                    flag_error(p.status, EP_DEV_CAPACITY);
                    row = -1;
                } else if (row >= s_base[lane + 1]) {
                    flag_error(p.status, EP_DEV_INCONSISTENT);
                    row = -1;
                }
            }
        }
        const unsigned valid = __ballot_sync(0xffffffffu, row >= 0);
        const int n = __popc(valid);
        if (row >= 0) {
            rows[__popc(valid & lanemask_lt())] = row;
            if (kWeighted) wts[__popc(valid & lanemask_lt())] = wt;
        }
        __syncwarp();

        const int ch0 = slice * kWarp * kCpl + lane;
        {
            float acc[kCpl][8];
#pragma unroll
            for (int c = 0; c < kCpl; ++c)
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[c][i] = 0.0f;
            for (int j0 = 0; j0 < n; j0 += kBatch) {
                uint4 v[kCpl][kBatch];
#pragma unroll
                for (int i = 0; i < kBatch; ++i)
#pragma unroll
                    for (int c = 0; c < kCpl; ++c)
                        if (j0 + i < n && ch0 + c * kWarp < p.chunks)
                            v[c][i] = ld_nc_v4(p.y + rows[j0 + i] * p.row_bytes + static_cast<long long>(ch0 + c * kWarp) * 16);
#pragma unroll
                for (int i = 0; i < kBatch; ++i)
#pragma unroll
                    for (int c = 0; c < kCpl; ++c)
                        if (j0 + i < n && ch0 + c * kWarp < p.chunks) {
                            if (kWeighted)
                                fma_bf16x8(acc[c], wts[j0 + i], v[c][i]);
                            else
                                add_bf16x8(acc[c], v[c][i]);
                        }
            }
#pragma unroll
            for (int c = 0; c < kCpl; ++c)
                if (ch0 + c * kWarp < p.chunks)
                    st_v4(p.out + g * p.row_bytes + static_cast<long long>(ch0 + c * kWarp) * 16, pack_bf16x8(acc[c]));
        }
        if (!kWeighted && slice == 0 && p.out_w != nullptr && lane < p.K) {
            float w = 0.0f;
            for (int j = 0; j < n; ++j) w += __ldg(p.y_w + rows[j] * p.K + lane);
            p.out_w[g * p.K + lane] = w;
        }
        __syncwarp();
    }
}

}  // namespace

namespace {

template <bool kWeighted>
cudaError_t launch_combine_args(CombineArgs& p, const Shape& sh, cudaStream_t stream) {
    const long long tokens = static_cast<long long>(sh.R) * sh.T;
    const int sms = device_sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    p.R = sh.R;
    p.K = sh.K;
    p.E = sh.E;
    p.row_bytes = sh.row_bytes();
    p.chunks = static_cast<int>(p.row_bytes / 16);
    p.slices = (p.chunks + kWarp * kCpl - 1) / (kWarp * kCpl);
    p.num_units = tokens * p.slices;
    const long long want = (p.num_units + kCombineWarps - 1) / kCombineWarps;
    const long long cap = static_cast<long long>(sms) * kCombineBlocksPerSm;
    const long long grid = want < cap ? want : cap;
    return launch_pdl(combine_kernel<kWeighted>, dim3(static_cast<unsigned>(grid)), dim3(kCombineThreads), 0,
                      stream, 0, false, p);
}

}  // namespace

cudaError_t launch_combine(const Shape& sh, const uint16_t* y, const float* y_w, int64_t y_rows,
                           const int32_t* send_pos, const int64_t* recv_base, uint16_t* combined_x,
                           float* combined_w, int32_t* status, cudaStream_t stream) {
    if (static_cast<long long>(sh.R) * sh.T == 0) return cudaSuccess;
    CombineArgs p = {};
    p.y = reinterpret_cast<const uint8_t*>(y);
    p.y_w = y_w;
    p.send_pos = send_pos;
    p.recv_base = recv_base;
    p.out = reinterpret_cast<uint8_t*>(combined_x);
    p.out_w = combined_w;
    p.status = status;
    p.y_rows = y_rows;
    return launch_combine_args<false>(p, sh, stream);
}

cudaError_t launch_ll_combine(const Shape& sh, const uint16_t* y, int cap, const int64_t* topk_idx,
                              const float* topk_w, const int32_t* slot_pos, uint16_t* combined_x,
                              int32_t* status, cudaStream_t stream) {
    if (static_cast<long long>(sh.R) * sh.T == 0) return cudaSuccess;
    CombineArgs p = {};
    p.y = reinterpret_cast<const uint8_t*>(y);
    p.out = reinterpret_cast<uint8_t*>(combined_x);
    p.status = status;
    p.y_rows = static_cast<long long>(sh.E) * cap;
    p.topk_idx = topk_idx;
    p.topk_w = topk_w;
    p.ll_slot_pos = slot_pos;
    p.ll_cap = cap;
    return launch_combine_args<true>(p, sh, stream);
}

}  // namespace ep
