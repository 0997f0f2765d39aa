// Grouped expert FFN for fp32 experts on the FMA units. fp32 inputs would go
// through TF32 on the tensor cores, whose ~1e-3 relative product error is far
// above what an fp32 layer is expected to deliver, so the fp32 path stays on
// exactly-rounded FFMA.
//
// Same schedule idea as the tensor-core path: the tile list (expert, M tile,
// N tile) is built on the device from `offsets`; a CTA computes one 64x64 output
// tile with 256 threads (4x4 outputs each) from 16-deep K chunks staged through
// shared memory. SwiGLU keeps a gate and an up accumulator per output and applies
// silu(g) * u in the epilogue; ReLU applies max(., 0); the down projection stores
// the plain product.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int TM = 64, TN = 64, TK = 16, kThreads = 256;
enum Mode : int { kSwiGLU = 0, kPlain = 1, kReLU = 2 };

struct SimtParams {
    const float* A;          // [rows, K]
    const float* B;          // [E*R, K]
    float* C;                // [rows, ldc]
    const int32_t* offsets;  // [E+1]
    const int32_t* counts;   // [E] rows used at the start of each segment, or null (all of it)
    int E, K, R, F, ldc, n_out, n_tiles;
};

template <int MODE>
__global__ void __launch_bounds__(kThreads) grouped_sgemm_kernel(const SimtParams p) {
    constexpr int NB = (MODE == kSwiGLU) ? 2 : 1;
    __shared__ int off[MOE_MAX_E + 1];
    __shared__ int end[MOE_MAX_E];
    __shared__ int tile[MOE_MAX_E + 1];
    __shared__ __align__(16) float As[TK][TM + 4];
    __shared__ __align__(16) float Bs[NB][TK][TN + 4];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int E = p.E;
    if (warp == 0) {
        for (int e0 = 0; e0 <= E; e0 += 32)
            if (e0 + lane <= E) off[e0 + lane] = __ldg(p.offsets + e0 + lane);
        __syncwarp();
        for (int e0 = 0; e0 < E; e0 += 32) {
            const int e = e0 + lane;
            if (e < E) {
                const int seg = off[e + 1] - off[e];
                end[e] = off[e] + (p.counts ? min(max(__ldg(p.counts + e), 0), seg) : seg);
            }
        }
        __syncwarp();
        int run = 0;
        for (int e0 = 0; e0 < E; e0 += 32) {
            const int e = e0 + lane;
            const int v = e < E ? (end[e] - off[e] + TM - 1) / TM : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += n;
            }
            if (e < E) tile[e] = run + incl - v;
            run += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
        if (lane == 0) tile[E] = run;
    }
    __syncthreads();
    const int t = blockIdx.x;
    if (t >= tile[E] * p.n_tiles) return;
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tile[mid] * p.n_tiles <= t) lo = mid; else hi = mid - 1;
    }
    const int e = lo;
    const int local = t - tile[e] * p.n_tiles;
    const int mte = tile[e + 1] - tile[e];
    const int nt = local / mte, mt = local - nt * mte;
    const int m0 = off[e] + mt * TM, m_end = end[e];
    const int n0 = nt * TN;

    const int tx = tid % 16, ty = tid / 16;  // 4 output columns x 4 rows each
    float acc[NB][4][4];
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[b][i][j] = 0.f;

    for (int k0 = 0; k0 < p.K; k0 += TK) {
        // A tile: 64 rows x 16 k, stored transposed (As[k][m]).
#pragma unroll
        for (int v = 0; v < (TM * TK) / kThreads; ++v) {
            const int li = tid + v * kThreads;
            const int r = li / TK, c = li % TK;
            const int row = m0 + r, kk = k0 + c;
            As[c][r] = (row < m_end && kk < p.K) ? __ldg(p.A + size_t(row) * p.K + kk) : 0.f;
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
#pragma unroll
            for (int v = 0; v < (TN * TK) / kThreads; ++v) {
                const int li = tid + v * kThreads;
                const int r = li / TK, c = li % TK;
                const int n = n0 + r, kk = k0 + c;
                const int brow = e * p.R + (b ? p.F : 0) + n;
                Bs[b][c][r] = (n < p.n_out && kk < p.K) ? __ldg(p.B + size_t(brow) * p.K + kk) : 0.f;
            }
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < TK; ++kk) {
            const float4 a4 = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
            const float a[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                const float4 b4 = *reinterpret_cast<const float4*>(&Bs[b][kk][tx * 4]);
                const float bb[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[b][i][j] = fmaf(a[i], bb[j], acc[b][i][j]);
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = m0 + ty * 4 + i;
        if (row >= m_end) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx * 4 + j;
            if (n >= p.n_out) continue;
            float v = acc[0][i][j];
            if (MODE == kSwiGLU) v = v / (1.0f + expf(-v)) * acc[NB - 1][i][j];
            if (MODE == kReLU) v = fmaxf(v, 0.f);
            p.C[size_t(row) * p.ldc + n] = v;
        }
    }
}

template <int MODE>
cudaError_t launch_mode(const SimtParams& p, int64_t rows_max, cudaStream_t stream) {
    const int64_t grid = ((rows_max + TM - 1) / TM + p.E) * int64_t(p.n_tiles);
    grouped_sgemm_kernel<MODE><<<unsigned(grid > 0 ? grid : 1), kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ffn_simt(const FfnArgs& a, cudaStream_t stream, cudaEvent_t mid_event) {
    const int64_t rows_max = a.rows;
    const bool swiglu = a.expert_kind == MOE_EXPERT_SWIGLU;
    SimtParams p{};
    p.offsets = a.offsets;
    p.counts = a.counts;
    p.E = a.E;
    p.F = a.F;
    // Up projection.
    p.A = static_cast<const float*>(a.xperm);
    p.B = static_cast<const float*>(a.W13);
    p.C = static_cast<float*>(a.h);
    p.K = a.d;
    p.R = swiglu ? 2 * a.F : a.F;
    p.ldc = a.F;
    p.n_out = a.F;
    p.n_tiles = (a.F + TN - 1) / TN;
    cudaError_t err = swiglu ? launch_mode<kSwiGLU>(p, rows_max, stream) : launch_mode<kReLU>(p, rows_max, stream);
    if (err != cudaSuccess) return err;
    if (mid_event) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if ((err = cudaStreamIsCapturing(stream, &cs)) != cudaSuccess) return err;
        err = cs == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(mid_event, stream, cudaEventRecordExternal)
                                                  : cudaEventRecord(mid_event, stream);
        if (err != cudaSuccess) return err;
    }
    // Down projection.
    p.A = static_cast<const float*>(a.h);
    p.B = static_cast<const float*>(a.W2);
    p.C = static_cast<float*>(a.out);
    p.K = a.F;
    p.R = a.d;
    p.F = 0;
    p.ldc = a.d;
    p.n_out = a.d;
    p.n_tiles = (a.d + TN - 1) / TN;
    return launch_mode<kPlain>(p, rows_max, stream);
}

}  // namespace moe
