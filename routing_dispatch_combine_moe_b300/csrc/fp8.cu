// FP8 dispatch ("MoE Expert Parallelism Sizing: Traffic, Capacity, Fabric", "First-order
// dispatch and combine bytes" and "Decode": the dispatched rows travel as FP8 with
// scale tensors, half the bytes of BF16, while the combine stays wide).
//
// Wire format of one routed row: d e4m3 codes plus one fp32 scale 2^s per 128-element
// block (the last block of a row may be shorter). s is the smallest integer with
// amax / 2^s <= 448, so every x / 2^s is in e4m3's finite range and rounds (to nearest,
// ties to even, sign kept) without saturating; the receiver's q * 2^s is exact in
// bf16. Shared experts are replicated, not dispatched: their rows are copied from x.
//
//   gather_fp8_kernel   one warp per token: each half-warp takes one 128-element block
//                       (16 lanes x 8 bf16), reduces its amax with shuffles, picks s,
//                       converts its 8 values, and writes the 8 codes (and the scale)
//                       to each of the token's kept routed rows;
//   dequant_fp8_kernel  one warp per dispatched row: codes x scale back to bf16 rows
//                       for the expert GEMMs (the receiving side).
//
// Row-scaled format (the FP8 up projection's input): the same rule with one block per
// row, so a row has one scale 2^s; every kept row of a token, routed or shared, gets the
// codes, and the expert GEMM reads them as they are (the scale is applied to its fp32
// accumulator). The expert weights take the same format, one scale per weight row.
//   gather_fp8_row_kernel  one CTA per token: amax over the row, then the codes to
//                          each kept row and the scale;
//   quantize_rows_cta_kernel / quantize_rows_kernel   a bf16 matrix row by row (one
//                          CTA per row held in registers, read once; one warp per row
//                          for short or very long rows): the W13 and W2 weights (once),
//                          and h between the two expert GEMMs when the down projection
//                          runs on e4m3 too.
#include <cuda_fp8.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

// Smallest s with amax / 2^s <= 448 (448 = 0.875 * 2^9); amax = m * 2^e, m in [0.5, 1).
__device__ __forceinline__ int block_exponent(float amax) {
    if (!(amax > 0.f)) return 0;
    int e;
    const float m = frexpf(amax, &e);
    return e - 9 + (m > 0.875f ? 1 : 0);
}

// e4m3 codes of the 8 bf16 values of `raw` divided by 2^s, packed little-end first.
__device__ __forceinline__ uint2 e4m3_pack8(const uint4 raw, int s) {
    const float f[8] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y),
                        bf16_lo(raw.z), bf16_hi(raw.z), bf16_lo(raw.w), bf16_hi(raw.w)};
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t c = __nv_cvt_float_to_fp8(ldexpf(f[i], -s), __NV_SATFINITE, __NV_E4M3);
        if (i < 4) lo |= c << (8 * i);
        else hi |= c << (8 * (i - 4));
    }
    return make_uint2(lo, hi);
}

__device__ __forceinline__ float absmax8(const uint4 raw) {
    const float m0 = fmaxf(fmaxf(fabsf(bf16_lo(raw.x)), fabsf(bf16_hi(raw.x))),
                           fmaxf(fabsf(bf16_lo(raw.y)), fabsf(bf16_hi(raw.y))));
    const float m1 = fmaxf(fmaxf(fabsf(bf16_lo(raw.z)), fabsf(bf16_hi(raw.z))),
                           fmaxf(fabsf(bf16_lo(raw.w)), fabsf(bf16_hi(raw.w))));
    return fmaxf(m0, m1);
}

// Scale exponent of one bf16 row of vpr 16-byte pieces, read by the 32 lanes of a warp.
__device__ __forceinline__ int row_exponent(const uint4* __restrict__ src, int vpr, int lane) {
    float am = 0.f;
    for (int v = lane; v < vpr; v += 32) am = fmaxf(am, absmax8(__ldg(src + v)));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, off));
    return block_exponent(am);
}

// One CTA of 128 threads per token, so that a decode-sized batch still spreads over the
// SMs: the row's amax is reduced over the CTA, then every thread converts its 16-byte
// pieces and writes them to each kept row of the token.
__global__ void __launch_bounds__(128) gather_fp8_row_kernel(const uint4* __restrict__ x,
                                                             const int32_t* __restrict__ pos, int T, int K, int d,
                                                             int64_t max_rows, uint8_t* __restrict__ xq,
                                                             float* __restrict__ xscale, int32_t* status) {
    __shared__ int dst[MOE_MAX_K];
    __shared__ float am_w[4];
    const int t = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int vpr = d / 8;
    if (tid < K) {
        int r = pos[size_t(t) * K + tid];
        if (r >= max_rows) {
            set_status(status, MOE_DEV_ERR_INDEX);
            r = -1;
        }
        dst[tid] = r < 0 ? -1 : r;
    }
    const uint4* src = x + size_t(t) * vpr;
    float am = 0.f;
    for (int v = tid; v < vpr; v += 128) am = fmaxf(am, absmax8(__ldg(src + v)));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, off));
    if (lane == 0) am_w[warp] = am;
    __syncthreads();
    const int s = block_exponent(fmaxf(fmaxf(am_w[0], am_w[1]), fmaxf(am_w[2], am_w[3])));
    for (int v = tid; v < vpr; v += 128) {
        const uint2 c = e4m3_pack8(__ldg(src + v), s);
        for (int j = 0; j < K; ++j) {
            const int r = dst[j];
            if (r >= 0) *reinterpret_cast<uint2*>(xq + size_t(r) * d + size_t(v) * 8) = c;
        }
    }
    if (tid < K && dst[tid] >= 0) xscale[dst[tid]] = ldexpf(1.f, s);
}

__global__ void __launch_bounds__(256) quantize_rows_kernel(const uint4* __restrict__ w, int64_t n_rows, int d,
                                                            uint8_t* __restrict__ q, float* __restrict__ scale) {
    const int lane = threadIdx.x & 31;
    const int64_t r = int64_t(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (r >= n_rows) return;
    const int vpr = d / 8;
    const uint4* src = w + size_t(r) * vpr;
    const int s = row_exponent(src, vpr, lane);
    for (int v = lane; v < vpr; v += 32)
        *reinterpret_cast<uint2*>(q + size_t(r) * d + size_t(v) * 8) = e4m3_pack8(__ldg(src + v), s);
    if (lane == 0) scale[r] = ldexpf(1.f, s);
}

// One CTA of 256 threads per row, for rows of at most 256 * VPT 16-byte pieces: each
// thread keeps its VPT pieces in registers, so the row is read from memory once; the
// amax is reduced over the CTA, then the same registers are converted and stored.
template <int VPT>
__global__ void __launch_bounds__(256) quantize_rows_cta_kernel(const uint4* __restrict__ w, int d,
                                                                uint8_t* __restrict__ q, float* __restrict__ scale) {
    __shared__ float am_w[8];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t r = blockIdx.x;
    const int vpr = d / 8;
    const uint4* src = w + size_t(r) * vpr;
    uint4 raw[VPT];
    float am = 0.f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int v = tid + 256 * i;
        raw[i] = v < vpr ? __ldg(src + v) : make_uint4(0, 0, 0, 0);
        am = fmaxf(am, absmax8(raw[i]));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, off));
    if (lane == 0) am_w[warp] = am;
    __syncthreads();
    am = am_w[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) am = fmaxf(am, am_w[i]);
    const int s = block_exponent(am);
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int v = tid + 256 * i;
        if (v < vpr) *reinterpret_cast<uint2*>(q + size_t(r) * d + size_t(v) * 8) = e4m3_pack8(raw[i], s);
    }
    if (tid == 0) scale[r] = ldexpf(1.f, s);
}

__global__ void __launch_bounds__(256) gather_fp8_kernel(const uint4* __restrict__ x,
                                                         const int32_t* __restrict__ topk_idx,
                                                         const int32_t* __restrict__ pos, int T, int K, int d,
                                                         int E_routed, int64_t max_rows, uint8_t* __restrict__ xq,
                                                         float* __restrict__ xscale, uint4* __restrict__ xperm,
                                                         int32_t* status) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T) return;
    const int nb = (d + 127) / 128, vpr = d / 8;  // 16-byte pieces per bf16 row
    int p = -1, shared_dst = -1;
    if (lane < K) {
        const size_t a = size_t(t) * K + lane;
        const int r = pos[a], e = topk_idx[a];
        if (r >= max_rows) {
            set_status(status, MOE_DEV_ERR_INDEX);
        } else if (r >= 0) {
            if (e >= 0 && e < E_routed) p = r;
            else shared_dst = r;
        }
    }
    int dst[MOE_MAX_K], sdst[MOE_MAX_K];
#pragma unroll
    for (int j = 0; j < MOE_MAX_K; ++j) {
        dst[j] = __shfl_sync(0xFFFFFFFFu, p, j);
        sdst[j] = __shfl_sync(0xFFFFFFFFu, shared_dst, j);
    }
    const uint4* src = x + size_t(t) * vpr;
    // each iteration covers two 128-element blocks: lanes 0-15 and 16-31
    for (int v0 = 0; v0 < vpr; v0 += 32) {
        const int v = v0 + lane;
        const bool ok = v < vpr;
        const uint4 raw = ok ? __ldg(src + v) : make_uint4(0, 0, 0, 0);
        // shared experts take the bf16 row as it is
#pragma unroll
        for (int j = 0; j < MOE_MAX_K; ++j)
            if (j < K && sdst[j] >= 0 && ok) xperm[size_t(sdst[j]) * vpr + v] = raw;
        float am = absmax8(raw);
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, off));
        const int s = block_exponent(am);
        const uint2 c = e4m3_pack8(raw, s);
        const int blk = v0 / 16 + (lane >> 4);  // 128-element block of this half-warp
        const bool writes_scale = (lane & 15) == 0 && blk < nb;
#pragma unroll
        for (int j = 0; j < MOE_MAX_K; ++j) {
            if (j < K && dst[j] >= 0) {
                if (ok) *reinterpret_cast<uint2*>(xq + size_t(dst[j]) * d + size_t(v) * 8) = c;
                if (writes_scale) xscale[size_t(dst[j]) * nb + blk] = ldexpf(1.f, s);
            }
        }
    }
}

__global__ void __launch_bounds__(256) dequant_fp8_kernel(const uint8_t* __restrict__ xq,
                                                          const float* __restrict__ xscale,
                                                          const int32_t* __restrict__ row_src,
                                                          const int32_t* __restrict__ topk_idx,
                                                          const int32_t* __restrict__ offsets, int n_offsets,
                                                          int d, int E_routed, int64_t rows,
                                                          uint4* __restrict__ xperm) {
    const int lane = threadIdx.x & 31;
    const int64_t r = int64_t(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (r >= rows || r >= offsets[n_offsets]) return;
    const int a = row_src[r];
    if (a < 0) return;                         // padding row (zeroed by the dispatch)
    const int e = topk_idx[a];
    if (e < 0 || e >= E_routed) return;        // shared expert: the row came from x
    const int nb = (d + 127) / 128, vpr = d / 8;
    const uint8_t* q = xq + size_t(r) * d;
    // each lane converts 8 codes (8 bytes) per step into one 16-byte bf16 piece
    for (int v = lane; v < vpr; v += 32) {
        const uint2 c = *reinterpret_cast<const uint2*>(q + size_t(v) * 8);
        const float sc = xscale[size_t(r) * nb + (v * 8) / 128];
        float f[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t w = i < 4 ? c.x : c.y;
            const __nv_fp8_storage_t code = __nv_fp8_storage_t((w >> (8 * (i & 3))) & 0xFFu);
            const __half_raw h = __nv_cvt_fp8_to_halfraw(code, __NV_E4M3);
            f[i] = __half2float(__half(h)) * sc;
        }
        xperm[size_t(r) * vpr + v] = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                                                pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
    }
}

// bf16 values of the 8 e4m3 codes of `c` times the scale sc (exact: q * 2^s is a bf16).
__device__ __forceinline__ uint4 e4m3_unpack8(const uint2 c, float sc) {
    float f[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t w = i < 4 ? c.x : c.y;
        const __nv_fp8_storage_t code = __nv_fp8_storage_t((w >> (8 * (i & 3))) & 0xFFu);
        const __half_raw h = __nv_cvt_fp8_to_halfraw(code, __NV_E4M3);
        f[i] = __half2float(__half(h)) * sc;
    }
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7]));
}

// The deduplicated dispatch's receiving side with FP8 send rows: one warp per token; each
// kept routed assignment's row is the dequantized send row of (token, rank of its expert),
// each shared expert's row is x[t].
__global__ void __launch_bounds__(256) fanout_fp8_kernel(const uint4* __restrict__ x,
                                                         const uint8_t* __restrict__ xq,
                                                         const float* __restrict__ xscale,
                                                         const int32_t* __restrict__ topk_idx,
                                                         const int32_t* __restrict__ pos,
                                                         const int32_t* __restrict__ send_pos,
                                                         uint4* __restrict__ xperm, int T, int K, int E_routed, int D,
                                                         int d, int64_t max_rows, int64_t max_send, int32_t* status) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T) return;
    const int nb = (d + 127) / 128, vpr = d / 8;
    int dst = -1, src = -1;  // src >= 0: send row; src == -2: x[t]
    if (lane < K) {
        const size_t a = size_t(t) * K + lane;
        const int p = pos[a], e = topk_idx[a];
        if (p >= 0 && p < max_rows) {
            if (e >= 0 && e < E_routed) {
                const int sr = send_pos[size_t(t) * D + e / (E_routed / D)];
                if (sr >= 0 && sr < max_send) {
                    dst = p;
                    src = sr;
                } else {
                    set_status(status, MOE_DEV_ERR_INDEX);
                }
            } else {
                dst = p;
                src = -2;
            }
        } else if (p >= max_rows) {
            set_status(status, MOE_DEV_ERR_INDEX);
        }
    }
    for (int j = 0; j < K; ++j) {
        const int dj = __shfl_sync(0xFFFFFFFFu, dst, j);
        const int sj = __shfl_sync(0xFFFFFFFFu, src, j);
        if (dj < 0) continue;
        uint4* to = xperm + size_t(dj) * vpr;
        if (sj == -2) {
            const uint4* from = x + size_t(t) * vpr;
            for (int v = lane; v < vpr; v += 32) to[v] = __ldg(from + v);
        } else {
            const uint8_t* q = xq + size_t(sj) * d;
            const float* sc = xscale + size_t(sj) * nb;
            for (int v = lane; v < vpr; v += 32)
                to[v] = e4m3_unpack8(*reinterpret_cast<const uint2*>(q + size_t(v) * 8), __ldg(sc + (v * 8) / 128));
        }
    }
}

// The deduplicated dispatch's receiving side with row-scaled FP8 send rows (the FP8
// GEMM's format): one warp per token; each kept routed assignment's codes and row scale
// are copied from the send row of (token, rank of its expert), and each shared expert's
// row is x[t] quantized by the same row rule (shared experts are replicated: they read x).
__global__ void __launch_bounds__(256) fanout_fp8_row_kernel(const uint4* __restrict__ x,
                                                             const uint8_t* __restrict__ sq,
                                                             const float* __restrict__ sscale,
                                                             const int32_t* __restrict__ topk_idx,
                                                             const int32_t* __restrict__ pos,
                                                             const int32_t* __restrict__ send_pos,
                                                             uint8_t* __restrict__ xq, float* __restrict__ xscale,
                                                             int T, int K, int E_routed, int D, int d,
                                                             int64_t max_rows, int64_t max_send, int32_t* status) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T) return;
    const int vpr = d / 8;  // 8-code pieces of a row; 16-byte bf16 pieces of x
    int dst = -1, src = -1;  // src >= 0: send row; src == -2: x[t]
    if (lane < K) {
        const size_t a = size_t(t) * K + lane;
        const int p = pos[a], e = topk_idx[a];
        if (p >= 0 && p < max_rows) {
            if (e >= 0 && e < E_routed) {
                const int sr = send_pos[size_t(t) * D + e / (E_routed / D)];
                if (sr >= 0 && sr < max_send) {
                    dst = p;
                    src = sr;
                } else {
                    set_status(status, MOE_DEV_ERR_INDEX);
                }
            } else {
                dst = p;
                src = -2;
            }
        } else if (p >= max_rows) {
            set_status(status, MOE_DEV_ERR_INDEX);
        }
    }
    const uint4* row = x + size_t(t) * vpr;
    bool have_s = false;  // the row exponent of x[t], taken at its first shared slot
    int s_x = 0;
    for (int j = 0; j < K; ++j) {
        const int dj = __shfl_sync(0xFFFFFFFFu, dst, j);
        const int sj = __shfl_sync(0xFFFFFFFFu, src, j);
        if (dj < 0) continue;
        uint2* to = reinterpret_cast<uint2*>(xq + size_t(dj) * d);
        if (sj == -2) {
            if (!have_s) {
                s_x = row_exponent(row, vpr, lane);
                have_s = true;
            }
            for (int v = lane; v < vpr; v += 32) to[v] = e4m3_pack8(__ldg(row + v), s_x);
            if (lane == 0) xscale[dj] = ldexpf(1.f, s_x);
        } else {
            // d % 16 == 0: both rows are whole 16-byte pieces
            const uint4* from = reinterpret_cast<const uint4*>(sq + size_t(sj) * d);
            uint4* to16 = reinterpret_cast<uint4*>(xq + size_t(dj) * d);
            for (int v = lane; v < d / 16; v += 32) to16[v] = from[v];
            if (lane == 0) xscale[dj] = sscale[sj];
        }
    }
}

}  // namespace

cudaError_t launch_fp8_send_rows(const void* x, const int32_t* send_pos, int T, int D, int d, int64_t max_send,
                                 uint8_t* sq, float* sscale, int32_t* status, cudaStream_t stream) {
    // the per-token row quantizer with the D send slots of each token as its destinations
    gather_fp8_row_kernel<<<T, 128, 0, stream>>>(static_cast<const uint4*>(x), send_pos, T, D, d, max_send, sq,
                                                  sscale, status);
    return cudaGetLastError();
}

cudaError_t launch_fp8_row_fanout(const void* x, const uint8_t* sq, const float* sscale, const int32_t* topk_idx,
                                  const int32_t* pos, const int32_t* send_pos, uint8_t* xq, float* xscale, int T,
                                  int K, int E_routed, int D, int d, int64_t max_rows, int64_t max_send,
                                  int32_t* status, cudaStream_t stream) {
    fanout_fp8_row_kernel<<<(T + 7) / 8, 256, 0, stream>>>(static_cast<const uint4*>(x), sq, sscale, topk_idx, pos,
                                                            send_pos, xq, xscale, T, K, E_routed, D, d, max_rows,
                                                            max_send, status);
    return cudaGetLastError();
}

cudaError_t launch_fp8_send(const void* x, const int32_t* slots, const int32_t* send_pos, int T, int D, int d,
                            int64_t max_send, uint8_t* xq, float* xscale, int32_t* status, cudaStream_t stream) {
    // the slots array stands for the ids: slot r of a token holds r (a "routed" expert of
    // the D ranks) or -1, so every send row is quantized and none is copied as it is
    gather_fp8_kernel<<<(T + 7) / 8, 256, 0, stream>>>(static_cast<const uint4*>(x), slots, send_pos, T, D, d, D,
                                                        max_send, xq, xscale, nullptr, status);
    return cudaGetLastError();
}

cudaError_t launch_fp8_fanout(const void* x, const uint8_t* xq, const float* xscale, const int32_t* topk_idx,
                              const int32_t* pos, const int32_t* send_pos, void* xperm, int T, int K, int E_routed,
                              int D, int d, int64_t max_rows, int64_t max_send, int32_t* status,
                              cudaStream_t stream) {
    fanout_fp8_kernel<<<(T + 7) / 8, 256, 0, stream>>>(static_cast<const uint4*>(x), xq, xscale, topk_idx, pos,
                                                        send_pos, static_cast<uint4*>(xperm), T, K, E_routed, D, d,
                                                        max_rows, max_send, status);
    return cudaGetLastError();
}

cudaError_t launch_fp8_dispatch(const Fp8Args& a, cudaStream_t stream) {
    if (a.per_row) {
        gather_fp8_row_kernel<<<a.T, 128, 0, stream>>>(static_cast<const uint4*>(a.x), a.pos, a.T, a.K, a.d, a.rows,
                                                        a.xq, a.xscale, a.status);
        return cudaGetLastError();
    }
    gather_fp8_kernel<<<(a.T + 7) / 8, 256, 0, stream>>>(static_cast<const uint4*>(a.x), a.topk_idx, a.pos, a.T,
                                                          a.K, a.d, a.E_routed, a.rows, a.xq, a.xscale,
                                                          static_cast<uint4*>(a.xperm), a.status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || !a.dequant) return e;
    if (a.rows > 0)
        dequant_fp8_kernel<<<unsigned((a.rows + 7) / 8), 256, 0, stream>>>(a.xq, a.xscale, a.row_src, a.topk_idx,
                                                                            a.offsets, a.n_experts, a.d,
                                                                            a.E_routed, a.rows,
                                                                            static_cast<uint4*>(a.xperm));
    return cudaGetLastError();
}

cudaError_t launch_quantize_rows_fp8(const void* w, int64_t n_rows, int d, uint8_t* q, float* scale,
                                     cudaStream_t stream) {
    if (n_rows <= 0) return cudaSuccess;
    const uint4* src = static_cast<const uint4*>(w);
    const int vpr = d / 8;
    // rows of up to 16384 elements: one CTA per row, read once; longer rows: one warp per row
    if (n_rows <= int64_t(INT32_MAX) && vpr > 256 * 4 && vpr <= 256 * 8)
        quantize_rows_cta_kernel<8><<<unsigned(n_rows), 256, 0, stream>>>(src, d, q, scale);
    else if (n_rows <= int64_t(INT32_MAX) && vpr > 256 * 2 && vpr <= 256 * 4)
        quantize_rows_cta_kernel<4><<<unsigned(n_rows), 256, 0, stream>>>(src, d, q, scale);
    else if (n_rows <= int64_t(INT32_MAX) && vpr > 256 && vpr <= 256 * 2)
        quantize_rows_cta_kernel<2><<<unsigned(n_rows), 256, 0, stream>>>(src, d, q, scale);
    else
        quantize_rows_kernel<<<unsigned((n_rows + 7) / 8), 256, 0, stream>>>(src, n_rows, d, q, scale);
    return cudaGetLastError();
}

}  // namespace moe
