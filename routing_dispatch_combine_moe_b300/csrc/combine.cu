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
// No atomics, so the result is deterministic.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

template <typename TAct>
struct Vec16;
template <>
struct Vec16<float> {
    static constexpr int N = 4;
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
    static constexpr int N = 8;
    __device__ static void unpack(const uint4& v, float* f) {
        f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
        f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z); f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
    }
    __device__ static uint4 pack(const float* f) {
        return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                          pack_bf16x2(f[6], f[7]));
    }
};

template <typename TAct>
__global__ void __launch_bounds__(256) combine_kernel(const uint4* __restrict__ out, const float* __restrict__ gate,
                                                      const int32_t* __restrict__ pos, uint4* __restrict__ y, int T,
                                                      int k, int vec_per_row, int64_t max_rows, int32_t* status) {
    using V = Vec16<TAct>;
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
    for (int v = lane; v < vec_per_row; v += 32) {
        uint4 raw[MOE_MAX_K];
#pragma unroll
        for (int j = 0; j < MOE_MAX_K; ++j)
            if (j < k && src[j] >= 0) raw[j] = __ldg(out + size_t(src[j]) * vec_per_row + v);
        float acc[V::N];
#pragma unroll
        for (int q = 0; q < V::N; ++q) acc[q] = 0.f;
#pragma unroll
        for (int j = 0; j < MOE_MAX_K; ++j) {
            if (j < k && src[j] >= 0) {
                float f[V::N];
                V::unpack(raw[j], f);
#pragma unroll
                for (int q = 0; q < V::N; ++q) acc[q] = fmaf(gj[j], f[q], acc[q]);
            }
        }
        y[size_t(t) * vec_per_row + v] = V::pack(acc);
    }
}

}  // namespace

cudaError_t launch_combine(int act_dtype, const void* out, const float* gate, const int32_t* pos, void* y, int T,
                           int d, int k, int32_t* status, cudaStream_t stream) {
    const int act_bytes = act_dtype == MOE_F32 ? 4 : 2;
    const int vec_per_row = int(int64_t(d) * act_bytes / 16);
    const int64_t max_rows = int64_t(T) * k;
    const int grid = (T + 7) / 8;
    if (act_dtype == MOE_F32)
        combine_kernel<float><<<grid, 256, 0, stream>>>(static_cast<const uint4*>(out), gate, pos,
                                                        static_cast<uint4*>(y), T, k, vec_per_row, max_rows, status);
    else
        combine_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(static_cast<const uint4*>(out), gate, pos,
                                                                static_cast<uint4*>(y), T, k, vec_per_row,
                                                                max_rows, status);
    return cudaGetLastError();
}

}  // namespace moe
