// Combine: y[t] = sum over kept slots j of G[t, j] * out[pos[t, j]]
// ("Mixture-of-Experts (MoE) Architecture and Expert Parallelism", section 2: the
// layer output is the gate-weighted sum of the selected experts' outputs; "EP Math
// - Expert Parallelism (MoE)", "The combine all-to-all: the return trip": the k
// returned vectors are weighted by the gates and summed; "Token drop": a dropped
// slot contributes nothing).
//
// The reverse all-to-all and the weighted reduction are one gather: one warp per
// token reads its k expert-output rows (16-byte vector loads, all k issued before
// the arithmetic), accumulates in fp32 in slot order and rounds once on the store.
// No atomics, so the result is deterministic. Expert outputs are read in their own
// dtype (bf16 or fp32); a lane handles 8 consecutive elements of the row.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

template <typename TAct>
struct Vec16;
template <>
struct Vec16<float> {
    __device__ static void unpack(const uint4& v, float* f) {
        f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
    }
    __device__ static uint4 pack(const float* f) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
    }
};
template <>
struct Vec16<__nv_bfloat16> {
    __device__ static void unpack(const uint4& v, float* f) {
        f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
        f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z); f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
    }
    __device__ static uint4 pack(const float* f) {
        return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                          pack_bf16x2(f[6], f[7]));
    }
};

template <typename T>
__device__ __forceinline__ void store8(T* p, const float* f);
template <>
__device__ __forceinline__ void store8<float>(float* p, const float* f) {
    reinterpret_cast<uint4*>(p)[0] = Vec16<float>::pack(f);
    reinterpret_cast<uint4*>(p)[1] = Vec16<float>::pack(f + 4);
}
template <>
__device__ __forceinline__ void store8<__nv_bfloat16>(__nv_bfloat16* p, const float* f) {
    *reinterpret_cast<uint4*>(p) = Vec16<__nv_bfloat16>::pack(f);
}

// d must be a multiple of 8 here (16-byte bf16 rows); fp32 rows of d % 8 == 4 use the 4-wide kernel.
// Each step a lane covers 32 bytes of every kept slot's row (16 bf16 or 8 fp32
// values) and issues all KMAX slots' loads before the first multiply-add, so up
// to KMAX x 32 bytes per lane are in flight.
template <typename TOut, typename TY, int KMAX>
__global__ void __launch_bounds__(256) combine_kernel(const TOut* __restrict__ out, const float* __restrict__ gate,
                                                      const int32_t* __restrict__ pos, TY* __restrict__ y, int T,
                                                      int k, int d, int64_t max_rows, int32_t* status) {
    constexpr int EPL = 32 / int(sizeof(TOut));  // elements per lane per step
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T) return;
    int p = -1;
    float g = 0.f;
    if (lane < k) {
        p = pos[size_t(t) * k + lane];
        g = gate[size_t(t) * k + lane];
        if (p >= max_rows) {
            set_status(status, MOE_DEV_ERR_INDEX);
            p = -1;
        }
    }
    int src[KMAX];
    float gj[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        src[j] = __shfl_sync(0xFFFFFFFFu, p, j);
        gj[j] = __shfl_sync(0xFFFFFFFFu, g, j);
        if (j >= k) src[j] = -1;
    }
    // UNR column steps are loaded before any arithmetic, so a lane keeps UNR x KMAX x 32
    // bytes in flight even when k is small (k = 2: 256 bytes).
    constexpr int UNR = KMAX >= 8 ? 1 : 8 / KMAX;
    // column slice blockIdx.y of gridDim.y, in whole warp steps of 32 * EPL columns
    const int steps = (d + 32 * EPL - 1) / (32 * EPL);
    const int per = (steps + gridDim.y - 1) / gridDim.y;
    const int cbeg = blockIdx.y * per * 32 * EPL, cend = min(d, cbeg + per * 32 * EPL);
    for (int c00 = cbeg + lane * EPL; c00 < cend; c00 += 32 * EPL * UNR) {
        uint4 raw[UNR][KMAX][2];
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
            const int c0 = c00 + u * 32 * EPL;
            const bool full = c0 + EPL <= d;
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                if (src[j] >= 0 && c0 < cend) {
                    const uint4* rp = reinterpret_cast<const uint4*>(out + size_t(src[j]) * d + c0);
                    raw[u][j][0] = __ldg(rp);
                    raw[u][j][1] = full ? __ldg(rp + 1) : make_uint4(0, 0, 0, 0);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
            const int c0 = c00 + u * 32 * EPL;
            if (c0 >= cend) break;
            const bool full = c0 + EPL <= d;
            float acc[EPL];
#pragma unroll
            for (int q = 0; q < EPL; ++q) acc[q] = 0.f;
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                if (src[j] >= 0) {
                    float f[EPL];
                    if constexpr (sizeof(TOut) == 2) {
                        Vec16<__nv_bfloat16>::unpack(raw[u][j][0], f);
                        Vec16<__nv_bfloat16>::unpack(raw[u][j][1], f + 8);
                    } else {
                        Vec16<float>::unpack(raw[u][j][0], f);
                        Vec16<float>::unpack(raw[u][j][1], f + 4);
                    }
#pragma unroll
                    for (int q = 0; q < EPL; ++q) acc[q] = fmaf(gj[j], f[q], acc[q]);
                }
            }
#pragma unroll
            for (int h = 0; h < EPL / 8; ++h)
                if (full || h == 0) store8<TY>(y + size_t(t) * d + c0 + 8 * h, acc + 8 * h);
        }
    }
}

// fp32 rows whose length is a multiple of 4 but not of 8.
__global__ void __launch_bounds__(256) combine_kernel_f32x4(const float* __restrict__ out, const float* __restrict__ gate,
                                                            const int32_t* __restrict__ pos, float* __restrict__ y,
                                                            int T, int k, int d, int64_t max_rows, int32_t* status) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T) return;
    int p = -1;
    float g = 0.f;
    if (lane < k) {
        p = pos[size_t(t) * k + lane];
        g = gate[size_t(t) * k + lane];
        if (p >= max_rows) {
            set_status(status, MOE_DEV_ERR_INDEX);
            p = -1;
        }
    }
    int src[MOE_MAX_K];
    float gj[MOE_MAX_K];
#pragma unroll
    for (int j = 0; j < MOE_MAX_K; ++j) {
        src[j] = __shfl_sync(0xFFFFFFFFu, p, j);
        gj[j] = __shfl_sync(0xFFFFFFFFu, g, j);
    }
    for (int c = lane * 4; c < d; c += 32 * 4) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < MOE_MAX_K; ++j) {
            if (j >= k || src[j] < 0) continue;
            float f[4];
            Vec16<float>::unpack(__ldg(reinterpret_cast<const uint4*>(out + size_t(src[j]) * d + c)), f);
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[q] = fmaf(gj[j], f[q], acc[q]);
        }
        *reinterpret_cast<uint4*>(y + size_t(t) * d + c) = Vec16<float>::pack(acc);
    }
}

template <typename TOut, typename TY>
void launch_k(dim3 grid, const void* out, const float* gate, const int32_t* pos, void* y, int T, int k, int d,
              int64_t max_rows, int32_t* status, cudaStream_t stream) {
    const TOut* o = static_cast<const TOut*>(out);
    TY* yy = static_cast<TY*>(y);
    if (k <= 2) combine_kernel<TOut, TY, 2><<<grid, 256, 0, stream>>>(o, gate, pos, yy, T, k, d, max_rows, status);
    else if (k <= 4) combine_kernel<TOut, TY, 4><<<grid, 256, 0, stream>>>(o, gate, pos, yy, T, k, d, max_rows, status);
    else if (k <= 8) combine_kernel<TOut, TY, 8><<<grid, 256, 0, stream>>>(o, gate, pos, yy, T, k, d, max_rows, status);
    else combine_kernel<TOut, TY, 16><<<grid, 256, 0, stream>>>(o, gate, pos, yy, T, k, d, max_rows, status);
}

}  // namespace

cudaError_t launch_combine(int act_dtype, int out_dtype, const void* out, const float* gate, const int32_t* pos,
                           void* y, int T, int d, int k, int64_t rows, int32_t* status, cudaStream_t stream) {
    const int64_t max_rows = rows;
    // token blocks of 8 warps; small batches also split each row into column slices of
    // at least 512 elements, until about two CTAs per SM are in flight
    const int nb = (T + 7) / 8;
    const int want = (2 * device_sm_count() + nb - 1) / nb;
    const int cap = d / 512 > 1 ? d / 512 : 1;
    const dim3 grid(unsigned(nb), unsigned(want < cap ? (want > 1 ? want : 1) : cap));
    if (act_dtype == MOE_F32) {
        if (d % 8 == 0)
            launch_k<float, float>(grid, out, gate, pos, y, T, k, d, max_rows, status, stream);
        else
            combine_kernel_f32x4<<<nb, 256, 0, stream>>>(static_cast<const float*>(out), gate, pos,
                                                           static_cast<float*>(y), T, k, d, max_rows, status);
    } else if (out_dtype == MOE_F32) {
        launch_k<float, __nv_bfloat16>(grid, out, gate, pos, y, T, k, d, max_rows, status, stream);
    } else {
        launch_k<__nv_bfloat16, __nv_bfloat16>(grid, out, gate, pos, y, T, k, d, max_rows, status, stream);
    }
    return cudaGetLastError();
}

}  // namespace moe
