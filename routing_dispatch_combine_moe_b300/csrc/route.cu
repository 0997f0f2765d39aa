// Router: fp32 logits H = x W_g (+ b), KeepTopK in registers with warp shuffles,
// softmax over the kept logits ("Mixture-of-Experts (MoE) Architecture and Expert
// Parallelism", section 2 "The Gating Network Formulation").
//
// One CTA of 256 threads owns 32 tokens and every expert. The logits are a small
// fp32 GEMM [32 x d] x [d x E_pad] done on the FMA units: chunks of d are staged
// through shared memory (x transposed so one 16-byte load gives a thread its four
// tokens), each thread accumulates 4 tokens x 8 experts over one K-slice, and the
// K-slices are summed in a fixed order. A running sum is folded every 256 products
// so the fp32 rounding error of a 7168-long dot product stays near 1e-7.
// The 32 logit rows then go to the 8 warps (4 tokens each): every lane holds
// E_pad/32 logits, and k rounds of a shuffle arg-max (ties to the lower expert id)
// pick the slots in descending order; the kept softmax uses expf in fp32.
#include "common.cuh"
#include "kernels.h"

#include <float.h>

namespace moe {
namespace {

constexpr int kTM = 32;       // tokens per CTA
constexpr int kThreads = 256;
constexpr int kRT = 4;        // tokens per thread
constexpr int kRE = 8;        // experts per thread
constexpr int kXStride = kTM + 4;  // padded row of the transposed x tile (floats)

template <int EG>
struct RouteShape {
    static constexpr int KS = 32 / EG;                  // K-slices per CTA
    static constexpr int EPASS = kRE * EG;              // padded expert count
    static constexpr int KC = (8 * KS > 32) ? 8 * KS : 32;  // d-chunk staged per step
    static constexpr int EPS = KC / KS;                 // elements per slice per chunk
    static constexpr int FOLD = (256 / EPS) > 0 ? 256 / EPS : 1;  // chunks per partial sum
    static constexpr int VPL = (EPASS + 31) / 32;       // logits per lane in the top-k
    static constexpr size_t smem_x = size_t(KC) * kXStride * 4;
    static constexpr size_t smem_w = size_t(KC) * EPASS * 4;
    static constexpr size_t smem_red = size_t(KS) * kTM * EPASS * 4;
    static constexpr size_t smem = smem_x + smem_w + smem_red;
};

template <typename TAct>
struct ActVec;
template <>
struct ActVec<float> {
    static constexpr int N = 4;  // elements per 16-byte vector
    __device__ static void to_f32(const uint4& v, float* o) {
        o[0] = __uint_as_float(v.x); o[1] = __uint_as_float(v.y);
        o[2] = __uint_as_float(v.z); o[3] = __uint_as_float(v.w);
    }
};
template <>
struct ActVec<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static void to_f32(const uint4& v, float* o) {
        o[0] = bf16_lo(v.x); o[1] = bf16_hi(v.x); o[2] = bf16_lo(v.y); o[3] = bf16_hi(v.y);
        o[4] = bf16_lo(v.z); o[5] = bf16_hi(v.z); o[6] = bf16_lo(v.w); o[7] = bf16_hi(v.w);
    }
};

template <typename TAct, int EG>
__global__ void __launch_bounds__(kThreads) route_kernel(const TAct* __restrict__ x, const float* __restrict__ Wg,
                                                         const float* __restrict__ bias, int T, int d, int E, int k,
                                                         int32_t* __restrict__ topk_idx,
                                                         float* __restrict__ topk_gate) {
    using S = RouteShape<EG>;
    constexpr int KS = S::KS, EPASS = S::EPASS, KC = S::KC, EPS = S::EPS;
    constexpr int VN = ActVec<TAct>::N;
    constexpr int XV = (kTM * KC / VN + kThreads - 1) / kThreads;     // x vectors per thread per chunk
    constexpr int WN = (KC * EPASS + kThreads - 1) / kThreads;        // Wg floats per thread per chunk

    extern __shared__ __align__(16) unsigned char smem_raw[];
    float* xs = reinterpret_cast<float*>(smem_raw);                          // [KC][kXStride]
    float* wsm = reinterpret_cast<float*>(smem_raw + S::smem_x);             // [KC][EPASS]
    float* red = reinterpret_cast<float*>(smem_raw + S::smem_x + S::smem_w); // [KS][kTM][EPASS]

    const int tid = threadIdx.x;
    const int eg = tid % EG;
    const int s = (tid / EG) % KS;
    const int tg = tid / (EG * KS);
    const int t0 = blockIdx.x * kTM;
    const int nchunks = (d + KC - 1) / KC;

    uint4 xr[XV];
    float wr[WN];

    auto load_chunk = [&](int c) {
        const int k0 = c * KC;
#pragma unroll
        for (int v = 0; v < XV; ++v) {
            const int vi = tid + v * kThreads;          // vector index inside the chunk
            const int tok = vi / (KC / VN), col = (vi % (KC / VN)) * VN;
            uint4 val = make_uint4(0, 0, 0, 0);
            if (vi < kTM * KC / VN && t0 + tok < T && k0 + col < d)
                val = __ldg(reinterpret_cast<const uint4*>(x + size_t(t0 + tok) * d + k0 + col));
            xr[v] = val;
        }
#pragma unroll
        for (int v = 0; v < WN; ++v) {
            const int wi = tid + v * kThreads;
            const int row = wi / EPASS, e = wi % EPASS;
            float val = 0.f;
            if (wi < KC * EPASS && k0 + row < d && e < E) val = __ldg(Wg + size_t(k0 + row) * E + e);
            wr[v] = val;
        }
    };
    auto store_chunk = [&]() {
#pragma unroll
        for (int v = 0; v < XV; ++v) {
            const int vi = tid + v * kThreads;
            if (vi < kTM * KC / VN) {
                const int tok = vi / (KC / VN), col = (vi % (KC / VN)) * VN;
                float f[VN];
                ActVec<TAct>::to_f32(xr[v], f);
#pragma unroll
                for (int q = 0; q < VN; ++q) xs[(col + q) * kXStride + tok] = f[q];
            }
        }
#pragma unroll
        for (int v = 0; v < WN; ++v) {
            const int wi = tid + v * kThreads;
            if (wi < KC * EPASS) wsm[wi] = wr[v];
        }
    };

    float acc[kRT][kRE], tot[kRT][kRE];
#pragma unroll
    for (int r = 0; r < kRT; ++r)
#pragma unroll
        for (int c = 0; c < kRE; ++c) acc[r][c] = tot[r][c] = 0.f;

    load_chunk(0);
    store_chunk();
    __syncthreads();
    for (int c = 0; c < nchunks; ++c) {
        if (c + 1 < nchunks) load_chunk(c + 1);
#pragma unroll
        for (int m = 0; m < EPS; ++m) {
            const int i = s + KS * m;
            const float4 xv = *reinterpret_cast<const float4*>(xs + i * kXStride + tg * kRT);
            const float4 w0 = *reinterpret_cast<const float4*>(wsm + i * EPASS + eg * kRE);
            const float4 w1 = *reinterpret_cast<const float4*>(wsm + i * EPASS + eg * kRE + 4);
            const float xa[4] = {xv.x, xv.y, xv.z, xv.w};
            const float wa[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
            for (int r = 0; r < kRT; ++r)
#pragma unroll
                for (int q = 0; q < kRE; ++q) acc[r][q] = fmaf(xa[r], wa[q], acc[r][q]);
        }
        if ((c + 1) % S::FOLD == 0) {
#pragma unroll
            for (int r = 0; r < kRT; ++r)
#pragma unroll
                for (int q = 0; q < kRE; ++q) { tot[r][q] += acc[r][q]; acc[r][q] = 0.f; }
        }
        __syncthreads();
        if (c + 1 < nchunks) {
            store_chunk();
            __syncthreads();
        }
    }
#pragma unroll
    for (int r = 0; r < kRT; ++r)
#pragma unroll
        for (int q = 0; q < kRE; ++q) tot[r][q] += acc[r][q];

    // K-slice partials -> shared memory, then summed in slice order per logit.
#pragma unroll
    for (int r = 0; r < kRT; ++r)
#pragma unroll
        for (int q = 0; q < kRE; ++q) red[(s * kTM + tg * kRT + r) * EPASS + eg * kRE + q] = tot[r][q];
    __syncthreads();

    const int warp = tid >> 5, lane = tid & 31;
    for (int tl = warp * (kTM / 8); tl < (warp + 1) * (kTM / 8); ++tl) {
        const int t = t0 + tl;
        if (t >= T) break;
        float v[S::VPL];
        int ids[S::VPL];
#pragma unroll
        for (int m = 0; m < S::VPL; ++m) {
            const int e = lane + 32 * m;
            ids[m] = e;
            float h = -INFINITY;
            if (e < E) {
                h = 0.f;
#pragma unroll
                for (int q = 0; q < KS; ++q) h += red[(q * kTM + tl) * EPASS + e];
                if (bias) h += __ldg(bias + e);
            }
            v[m] = h;
        }
        float my_val = -INFINITY;
        int my_idx = 0;
        for (int j = 0; j < k; ++j) {
            float bv = -INFINITY;
            int bi = 0x7FFFFFFF;
#pragma unroll
            for (int m = 0; m < S::VPL; ++m)
                if (v[m] > bv || (v[m] == bv && ids[m] < bi)) { bv = v[m]; bi = ids[m]; }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
                const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, off);
                if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
            }
            if (bi >= E) bi = 0;  // only reachable with NaN logits; keeps the index in range
            if (lane == j) { my_val = bv; my_idx = bi; }
#pragma unroll
            for (int m = 0; m < S::VPL; ++m)
                if (ids[m] == bi) v[m] = -INFINITY;
        }
        const float vmax = __shfl_sync(0xFFFFFFFFu, my_val, 0);
        const float ex = (lane < k) ? expf(my_val - vmax) : 0.f;
        float sum = 0.f;
        for (int j = 0; j < k; ++j) sum += __shfl_sync(0xFFFFFFFFu, ex, j);
        if (lane < k) {
            topk_idx[size_t(t) * k + lane] = my_idx;
            topk_gate[size_t(t) * k + lane] = ex / sum;
        }
    }
}

template <typename TAct, int EG>
cudaError_t launch_route_eg(const void* x, const float* Wg, const float* bias, int T, int d, int E, int k,
                            int32_t* idx, float* gate, cudaStream_t stream) {
    using S = RouteShape<EG>;
    auto kern = route_kernel<TAct, EG>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(S::smem));
    if (err != cudaSuccess) return err;
    const int grid = (T + kTM - 1) / kTM;
    kern<<<grid, kThreads, S::smem, stream>>>(static_cast<const TAct*>(x), Wg, bias, T, d, E, k, idx, gate);
    return cudaGetLastError();
}

template <typename TAct>
cudaError_t launch_route_t(const void* x, const float* Wg, const float* bias, int T, int d, int E, int k,
                           int32_t* idx, float* gate, cudaStream_t stream) {
    const int groups = (E + kRE - 1) / kRE;
    if (groups <= 1) return launch_route_eg<TAct, 1>(x, Wg, bias, T, d, E, k, idx, gate, stream);
    if (groups <= 2) return launch_route_eg<TAct, 2>(x, Wg, bias, T, d, E, k, idx, gate, stream);
    if (groups <= 4) return launch_route_eg<TAct, 4>(x, Wg, bias, T, d, E, k, idx, gate, stream);
    if (groups <= 8) return launch_route_eg<TAct, 8>(x, Wg, bias, T, d, E, k, idx, gate, stream);
    if (groups <= 16) return launch_route_eg<TAct, 16>(x, Wg, bias, T, d, E, k, idx, gate, stream);
    return launch_route_eg<TAct, 32>(x, Wg, bias, T, d, E, k, idx, gate, stream);
}

}  // namespace

cudaError_t launch_route(int act_dtype, const void* x, const float* Wg, const float* bias, int T, int d, int E,
                         int k, int32_t* topk_idx, float* topk_gate, cudaStream_t stream) {
    if (act_dtype == MOE_F32) return launch_route_t<float>(x, Wg, bias, T, d, E, k, topk_idx, topk_gate, stream);
    return launch_route_t<__nv_bfloat16>(x, Wg, bias, T, d, E, k, topk_idx, topk_gate, stream);
}

}  // namespace moe
