// Router: fp32 logits H = x W_g (+ b), KeepTopK in registers with warp shuffles,
// softmax over the kept logits ("Mixture-of-Experts (MoE) Architecture and Expert
// Parallelism", section 2 "The Gating Network Formulation").
//
// For bf16 activations and E >= 64 the logits come from the tensor cores
// (route_tc.cu); otherwise they are an fp32 GEMM [T x d] x [d x E] on the FMA units
// (exactly rounded products and sums), as follows. A CTA of 8 warps stages chunks of 16 elements of x (transposed)
// and of W_g through double-buffered shared memory; lanes own 4 tokens each, so W_g
// values are warp-wide broadcasts, and warps own 8 experts each (warps along experts
// = 1, 2, 4 or 8 for E <= 8, 16, 32 or more; the rest of the 8 warps run along
// tokens). Each thread keeps a 4 x 8 register tile. d is split into KS slices,
// chosen on the host so the CTA count fills the SMs evenly; each slice writes its
// partial logits, and the top-k kernel (one warp per token) adds the KS partials in
// slice order, adds the bias, and selects. Running sums are folded every 256
// products to keep the fp32 error of a long dot product near 1e-7.
//
// KeepTopK: k rounds of a warp arg-max over the logits held in registers, equal
// values won by the lower expert id; slot j is the (j+1)-th largest. Inside the layer
// forward the top-k writers also add each assignment to the dispatch's per-block
// expert histogram (RouteCounts), so the dispatch needs no count pass.
#include "common.cuh"
#include "kernels.h"

#include <mutex>

namespace moe {
namespace {

// ------------------------------------------------------------------ shared pieces
template <typename TAct>
struct Act16;
template <>
struct Act16<float> {
    static constexpr int N = 4;
    __device__ static void to_f32(const uint4& v, float* o) {
        o[0] = __uint_as_float(v.x); o[1] = __uint_as_float(v.y);
        o[2] = __uint_as_float(v.z); o[3] = __uint_as_float(v.w);
    }
};
template <>
struct Act16<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static void to_f32(const uint4& v, float* o) {
        o[0] = bf16_lo(v.x); o[1] = bf16_hi(v.x); o[2] = bf16_lo(v.y); o[3] = bf16_hi(v.y);
        o[4] = bf16_lo(v.z); o[5] = bf16_hi(v.z); o[6] = bf16_lo(v.w); o[7] = bf16_hi(v.w);
    }
};

// The dispatch histogram the layer forward has the router fill: hist[e * nblk + b]
// counts the assignments of expert e among assignments [256 b, 256 (b + 1)) (the count
// kernel's blocks), zeroed beforehand; integer atomics, so the counts do not depend on
// their order. A null hist leaves the counting to the dispatch. A non-null near_ties
// (zeroed beforehand) counts the tokens whose k-th and (k+1)-th largest selectable
// logits are a near tie (see is_near_tie).
struct RouteCounts {
    int32_t* hist;
    int nblk;
    int32_t* near_ties;
};

__device__ __forceinline__ void count_assignment(const RouteCounts c, int e, int64_t a) {
    if (c.hist) atomicAdd(c.hist + size_t(e) * c.nblk + size_t(a / kDispatchBlock), 1);
}

// A near tie of the selection: the k-th largest logit vk and the (k+1)-th vn (-inf
// when there is none) differ by less than 1e-6 of the larger magnitude, so another
// rounding of the logits could select a different set of experts.
__device__ __forceinline__ bool is_near_tie(float vk, float vn) {
    return (vk - vn) < 1e-6f * fmaxf(fabsf(vk), fabsf(vn));
}

// Top-k of the logits held by a warp (lane l holds experts l + 32 m, m < VPL, with
// -inf for padding), then the kept softmax; lane j < k writes slot j.
template <int VPL>
__device__ __forceinline__ void topk_softmax_store(float (&v)[VPL], int lane, int E, int k, int n_shared,
                                                   int32_t* idx_out, float* gate_out, const RouteCounts cnt,
                                                   int64_t a0) {
    float my_val = -INFINITY;
    int my_idx = 0;
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int bi = 0x7FFFFFFF;
#pragma unroll
        for (int m = 0; m < VPL; ++m) {
            const int e = lane + 32 * m;
            if (v[m] > bv || (v[m] == bv && e < bi)) { bv = v[m]; bi = e; }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
            const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, off);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if (bi >= E) bi = 0;  // only reachable with NaN logits; keeps the index in range
        if (lane == j) { my_val = bv; my_idx = bi; }
#pragma unroll
        for (int m = 0; m < VPL; ++m)
            if (lane + 32 * m == bi) v[m] = -INFINITY;
    }
    if (cnt.near_ties) {  // the (k+1)-th largest: one more arg-max round, value only
        float nv = -INFINITY;
#pragma unroll
        for (int m = 0; m < VPL; ++m) nv = fmaxf(nv, v[m]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) nv = fmaxf(nv, __shfl_xor_sync(0xFFFFFFFFu, nv, off));
        const float vk = __shfl_sync(0xFFFFFFFFu, my_val, k - 1);
        if (lane == 0 && is_near_tie(vk, nv)) atomicAdd(cnt.near_ties, 1);
    }
    const float vmax = __shfl_sync(0xFFFFFFFFu, my_val, 0);
    const float ex = (lane < k) ? expf(my_val - vmax) : 0.f;
    float sum = 0.f;
    for (int j = 0; j < k; ++j) sum += __shfl_sync(0xFFFFFFFFu, ex, j);
    if (lane < k) {
        idx_out[lane] = my_idx;
        gate_out[lane] = ex / sum;
        count_assignment(cnt, my_idx, a0 + lane);
    } else if (lane < k + n_shared) {  // shared experts follow the routed slots, gate 1
        idx_out[lane] = E + (lane - k);
        gate_out[lane] = 1.0f;
        count_assignment(cnt, E + (lane - k), a0 + lane);
    }
}

// Two fp32 fused multiply-adds in one instruction (Blackwell's packed f32x2 FMA):
// c0 = fma(a, b0, c0), c1 = fma(a, b1, c1), each rounded to nearest exactly like fmaf,
// with half the instructions to issue.
__device__ __forceinline__ void fma2_rn(float a, float b0, float b1, float& c0, float& c1) {
    uint64_t aa, bb, cc;
    asm("mov.b64 %0, {%1, %1};" : "=l"(aa) : "f"(a));
    asm("mov.b64 %0, {%1, %2};" : "=l"(bb) : "f"(b0), "f"(b1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(cc) : "f"(c0), "f"(c1));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(cc) : "l"(aa), "l"(bb));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(c0), "=f"(c1) : "l"(cc));
}

// ------------------------------------------------------------------ logits GEMM
// CTA of 8 warps: WE warps along experts (8 experts each), 8/WE warps along tokens
// (128 tokens each, 4 per lane).
constexpr int kGK = 16;    // d elements per staged chunk

template <int WE>
struct GemmShape {
    static constexpr int WT = 8 / WE;
    static constexpr int TT = 128 * WT;   // tokens per CTA
    static constexpr int TE = 8 * WE;     // experts per CTA
    static constexpr int XS = TT + 4;     // padded transposed-x row (floats)
    static constexpr size_t smem = size_t(2) * kGK * XS * 4 + size_t(2) * kGK * TE * 4;
};

template <typename TAct, int WE>
__global__ void __launch_bounds__(256, WE == 1 ? 1 : 2) route_gemm_kernel(const TAct* __restrict__ x,
                                                                         const float* __restrict__ Wg, int T, int d,
                                                                         int E, int k_slice,
                                                                         float* __restrict__ partial) {
    using G = GemmShape<WE>;
    constexpr int VN = Act16<TAct>::N;
    constexpr int XV = G::TT * kGK / VN / 256;              // x vectors per thread per chunk
    constexpr int WN = kGK * G::TE / 4;                      // W_g float4s per chunk
    constexpr int WV = (WN + 255) / 256;
    extern __shared__ __align__(16) float sm[];
    float* xs = sm;                                          // [2][kGK][XS]
    float* ws = sm + 2 * kGK * G::XS;                        // [2][kGK][TE]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int wexp = warp % WE, wtok = warp / WE;
    const int t0 = blockIdx.x * G::TT, e0 = blockIdx.y * G::TE;
    const int kb = blockIdx.z * k_slice;
    const int ke = min(d, kb + k_slice);
    const int nchunks = ke > kb ? (ke - kb + kGK - 1) / kGK : 0;
    const bool w_vec = (E % 4) == 0;

    uint4 xr[XV];
    float4 wr[WV];
    auto load = [&](int c) {
        const int k0 = kb + c * kGK;
#pragma unroll
        for (int i = 0; i < XV; ++i) {
            const int vi = tid + i * 256;
            const int tok = vi / (kGK / VN), col = (vi % (kGK / VN)) * VN;
            uint4 val = make_uint4(0, 0, 0, 0);
            if (t0 + tok < T && k0 + col < ke)
                val = __ldg(reinterpret_cast<const uint4*>(x + size_t(t0 + tok) * d + k0 + col));
            xr[i] = val;
        }
#pragma unroll
        for (int i = 0; i < WV; ++i) {
            const int wi = tid + i * 256;
            const int row = wi / (G::TE / 4), col = (wi % (G::TE / 4)) * 4;
            float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
            if (wi < WN && k0 + row < ke) {
                const float* src = Wg + size_t(k0 + row) * E + e0 + col;
                if (w_vec && e0 + col + 4 <= E) {
                    val = __ldg(reinterpret_cast<const float4*>(src));
                } else {
                    if (e0 + col + 0 < E) val.x = __ldg(src + 0);
                    if (e0 + col + 1 < E) val.y = __ldg(src + 1);
                    if (e0 + col + 2 < E) val.z = __ldg(src + 2);
                    if (e0 + col + 3 < E) val.w = __ldg(src + 3);
                }
            }
            wr[i] = val;
        }
    };
    auto store = [&](int buf) {
        float* xb = xs + buf * kGK * G::XS;
#pragma unroll
        for (int i = 0; i < XV; ++i) {
            const int vi = tid + i * 256;
            const int tok = vi / (kGK / VN), col = (vi % (kGK / VN)) * VN;
            float f[VN];
            Act16<TAct>::to_f32(xr[i], f);
#pragma unroll
            for (int q = 0; q < VN; ++q) xb[(col + q) * G::XS + tok] = f[q];
        }
        float* wb = ws + buf * kGK * G::TE;
#pragma unroll
        for (int i = 0; i < WV; ++i) {
            const int wi = tid + i * 256;
            if (wi < WN) *reinterpret_cast<float4*>(wb + wi * 4) = wr[i];
        }
    };

    float acc[4][8], tot[4][8];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[r][q] = tot[r][q] = 0.f;

    if (nchunks > 0) {
        load(0);
        store(0);
    }
    __syncthreads();
    const int xoff = wtok * 128 + lane * 4;
    for (int c = 0; c < nchunks; ++c) {
        const int buf = c & 1;
        if (c + 1 < nchunks) load(c + 1);
        const float* xb = xs + buf * kGK * G::XS;
        const float* wb = ws + buf * kGK * G::TE;
#pragma unroll
        for (int i = 0; i < kGK; ++i) {
            const float4 xv = *reinterpret_cast<const float4*>(xb + i * G::XS + xoff);
            const float4 w0 = *reinterpret_cast<const float4*>(wb + i * G::TE + wexp * 8);
            const float4 w1 = *reinterpret_cast<const float4*>(wb + i * G::TE + wexp * 8 + 4);
            const float xa[4] = {xv.x, xv.y, xv.z, xv.w};
            const float wa[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int q = 0; q < 8; q += 2) fma2_rn(xa[r], wa[q], wa[q + 1], acc[r][q], acc[r][q + 1]);
        }
        if ((c + 1) % (256 / kGK) == 0) {
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int q = 0; q < 8; ++q) { tot[r][q] += acc[r][q]; acc[r][q] = 0.f; }
        }
        if (c + 1 < nchunks) store(buf ^ 1);
        __syncthreads();
    }
    // partial[z][t][e]
    float* out = partial + size_t(blockIdx.z) * T * E;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int t = t0 + xoff + r;
        if (t >= T) continue;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int e = e0 + wexp * 8 + q;
            if (e < E) out[size_t(t) * E + e] = tot[r][q] + acc[r][q];
        }
    }
}

// Group-limited selection: the E experts form G contiguous groups of E/G; each group is
// scored by its largest logit, the M best groups are kept (equal scores: lower group
// first) and every other logit is set to -inf before KeepTopK. G <= 32: lane g holds
// group g's score.
template <int VPL>
__device__ __forceinline__ void limit_groups(float (&v)[VPL], int lane, int E, int G, int M) {
    const int gs = E / G;
    float score = -INFINITY;
    if (gs % 32 == 0) {
        // every register slot q lies in one group, q / (gs / 32): reduce the slots over the
        // warp (independent reductions) and take each group's largest
        float wq[VPL];
#pragma unroll
        for (int q = 0; q < VPL; ++q) wq[q] = lane + 32 * q < E ? v[q] : -INFINITY;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
#pragma unroll
            for (int q = 0; q < VPL; ++q) wq[q] = fmaxf(wq[q], __shfl_xor_sync(0xFFFFFFFFu, wq[q], off));
        const int qpg = gs / 32;
#pragma unroll
        for (int q = 0; q < VPL; ++q)
            if (q / qpg == lane) score = fmaxf(score, wq[q]);
    } else {
        for (int g = 0; g < G; ++g) {
            float m = -INFINITY;
#pragma unroll
            for (int q = 0; q < VPL; ++q) {
                const int e = lane + 32 * q;
                if (e < E && e / gs == g) m = fmaxf(m, v[q]);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
            if (lane == g) score = m;
        }
    }
    uint32_t kept = 0;
    for (int r = 0; r < M; ++r) {
        float bv = (lane < G && !((kept >> lane) & 1u)) ? score : -INFINITY;
        int bi = (lane < G && !((kept >> lane) & 1u)) ? lane : 0x7FFFFFFF;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
            const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, off);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if (bi < G) kept |= 1u << bi;
    }
#pragma unroll
    for (int q = 0; q < VPL; ++q) {
        const int e = lane + 32 * q;
        if (e < E && !((kept >> (e / gs)) & 1u)) v[q] = -INFINITY;
    }
}

// One warp per token (4 per CTA): the KS partial logits of each of the lane's VPL
// experts are loaded UB slices at a time (VPL * UB loads in flight) and added in slice
// order, then the bias; then the optional group limit and KeepTopK + kept softmax.
template <int VPL>
__global__ void __launch_bounds__(128) route_topk_kernel(const float* __restrict__ partial, int KS,
                                                         const float* __restrict__ bias, int T, int E, int k,
                                                         int n_shared, int n_groups, int topk_groups,
                                                         int32_t* __restrict__ topk_idx,
                                                         float* __restrict__ topk_gate, const RouteCounts cnt) {
    constexpr int UB = VPL >= 16 ? 4 : (VPL >= 4 ? 8 : 32 / VPL);
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * 4 + (threadIdx.x >> 5);
    if (t >= T) return;
    // Padding lanes (e >= E) start at -inf, which the finite partials do not change.
    // Every load is unconditional (indices clamped into range) so that all VPL * UB of
    // them are in flight before the first add; slices past KS add zero.
    float v[VPL];
#pragma unroll
    for (int q = 0; q < VPL; ++q) v[q] = (lane + 32 * q < E) ? 0.f : -INFINITY;
    const float* base = partial + size_t(t) * E;
    for (int z0 = 0; z0 < KS; z0 += UB) {
        float pz[VPL][UB];
#pragma unroll
        for (int q = 0; q < VPL; ++q) {
            const int e = min(lane + 32 * q, E - 1);
#pragma unroll
            for (int u = 0; u < UB; ++u) pz[q][u] = __ldg(base + size_t(min(z0 + u, KS - 1)) * T * E + e);
        }
#pragma unroll
        for (int q = 0; q < VPL; ++q)
#pragma unroll
            for (int u = 0; u < UB; ++u) v[q] += (z0 + u < KS) ? pz[q][u] : 0.f;
    }
    if (bias) {
#pragma unroll
        for (int q = 0; q < VPL; ++q)
            if (lane + 32 * q < E) v[q] += __ldg(bias + lane + 32 * q);
    }
    if (topk_groups > 0 && topk_groups < n_groups) limit_groups<VPL>(v, lane, E, n_groups, topk_groups);
    const int K = k + n_shared;
    topk_softmax_store<VPL>(v, lane, E, k, n_shared, topk_idx + size_t(t) * K, topk_gate + size_t(t) * K, cnt,
                            int64_t(t) * K);
}

// ------------------------------------------------------------------ small E, fused
// For E <= 32 with W_g small (d * E * 4 <= 128 KB, e.g. 4096 x 8) one kernel does the
// logits, KeepTopK and the softmax. A CTA takes 16 tokens; thread (tok, ks) of a 16 x 16
// grid sums the products of token tok over the ks-th sixteenth of d into EB partial
// logits (x in 16-byte pieces; each W_g row is read by 16 threads at once, so it comes
// from L1 as one sector per load). The 16 partials of a logit are then added in ks
// order through shared memory by thread (tok, 0), which also selects the top k (equal
// logits: lower id), applies the optional group limit and the kept softmax, exactly
// as the warp-wide path does. Deterministic: every sum has a fixed order.
template <int EB>
__device__ __forceinline__ void topk_softmax_thread(float (&v)[EB], int E, int k, int n_shared, int n_groups,
                                                    int topk_groups, int32_t* idx_out, float* gate_out,
                                                    const RouteCounts cnt, int64_t a0) {
    if (topk_groups > 0 && topk_groups < n_groups) {
        const int gs = E / n_groups;
        uint32_t kept = 0;
        for (int r = 0; r < topk_groups; ++r) {
            float best = -INFINITY;
            int bg = -1;
            for (int g = 0; g < n_groups; ++g) {
                if ((kept >> g) & 1u) continue;
                float m = -INFINITY;
#pragma unroll
                for (int e = 0; e < EB; ++e)
                    if (e < E && e / gs == g) m = fmaxf(m, v[e]);
                if (bg < 0 || m > best) { best = m; bg = g; }
            }
            kept |= 1u << bg;
        }
#pragma unroll
        for (int e = 0; e < EB; ++e)
            if (e < E && !((kept >> (e / gs)) & 1u)) v[e] = -INFINITY;
    }
    uint32_t taken = 0;
    float val[MOE_MAX_K];
    int id[MOE_MAX_K];
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int bi = -1;
#pragma unroll
        for (int e = 0; e < EB; ++e)
            if (e < E && !((taken >> e) & 1u) && (bi < 0 || v[e] > bv)) { bv = v[e]; bi = e; }
        if (bi < 0) bi = 0;  // only reachable with NaN logits; keeps the index in range
        taken |= 1u << bi;
        val[j] = bv;
        id[j] = bi;
    }
    if (cnt.near_ties) {  // the (k+1)-th largest of the logits not taken
        float nv = -INFINITY;
#pragma unroll
        for (int e = 0; e < EB; ++e)
            if (e < E && !((taken >> e) & 1u)) nv = fmaxf(nv, v[e]);
        if (is_near_tie(val[k - 1], nv)) atomicAdd(cnt.near_ties, 1);
    }
    float ex[MOE_MAX_K];
    float sum = 0.f;
    for (int j = 0; j < k; ++j) {
        ex[j] = expf(val[j] - val[0]);
        sum += ex[j];
    }
    for (int j = 0; j < k; ++j) {
        idx_out[j] = id[j];
        gate_out[j] = ex[j] / sum;
        count_assignment(cnt, id[j], a0 + j);
    }
    for (int j = 0; j < n_shared; ++j) {
        idx_out[k + j] = E + j;
        gate_out[k + j] = 1.0f;
        count_assignment(cnt, E + j, a0 + k + j);
    }
}

template <typename TAct, int EB>
__global__ void __launch_bounds__(256) route_small_kernel(const TAct* __restrict__ x, const float* __restrict__ Wg,
                                                          const float* __restrict__ bias, int T, int d, int E, int k,
                                                          int n_shared, int n_groups, int topk_groups, bool wvec,
                                                          int32_t* __restrict__ topk_idx,
                                                          float* __restrict__ topk_gate, const RouteCounts cnt) {
    constexpr int VN = Act16<TAct>::N, UV = 4;
    extern __shared__ __align__(16) float smw[];        // W_g [d][E], then the partial logits
    float (*red)[16][EB + 1] = reinterpret_cast<float (*)[16][EB + 1]>(smw + size_t(d) * E);
    const int tid = threadIdx.x, tok = tid & 15, ks = tid >> 4;
    // W_g once per CTA into shared memory (coalesced, independent loads)
    const int nw = d * E;
    if (wvec) {  // asynchronous 16-byte copies, all in flight at once
        const float4* src = reinterpret_cast<const float4*>(Wg);
        for (int i = tid; i < nw / 4; i += 256)
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smw + 4 * i)), "l"(src + i)
                         : "memory");
        asm volatile("cp.async.wait_all;" ::: "memory");
    } else {
        for (int i = tid; i < nw; i += 256) smw[i] = __ldg(Wg + i);
    }
    __syncthreads();
    const int t = blockIdx.x * 16 + tok;
    const int vpr = d / VN;                 // 16-byte pieces per row
    const int per = (vpr + 15) / 16;        // pieces per sixteenth
    const int v0 = ks * per, v1 = min(vpr, v0 + per);
    float acc[EB];
#pragma unroll
    for (int e = 0; e < EB; ++e) acc[e] = 0.f;
    if (t < T) {
        const uint4* row = reinterpret_cast<const uint4*>(x + size_t(t) * d);
        for (int vb = v0; vb < v1; vb += UV) {
            uint4 raw[UV];
#pragma unroll
            for (int u = 0; u < UV; ++u) raw[u] = vb + u < v1 ? __ldg(row + vb + u) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int u = 0; u < UV; ++u) {
                if (vb + u >= v1) break;
                float xv[VN];
                Act16<TAct>::to_f32(raw[u], xv);
#pragma unroll
                for (int q = 0; q < VN; ++q) {
                    const float* wrow = smw + size_t((vb + u) * VN + q) * E;
                    if (wvec) {  // E == EB: EB/4 vector reads per row
#pragma unroll
                        for (int e4 = 0; e4 < EB / 4; ++e4) {
                            const float4 w4 = reinterpret_cast<const float4*>(wrow)[e4];
                            acc[4 * e4 + 0] = fmaf(xv[q], w4.x, acc[4 * e4 + 0]);
                            acc[4 * e4 + 1] = fmaf(xv[q], w4.y, acc[4 * e4 + 1]);
                            acc[4 * e4 + 2] = fmaf(xv[q], w4.z, acc[4 * e4 + 2]);
                            acc[4 * e4 + 3] = fmaf(xv[q], w4.w, acc[4 * e4 + 3]);
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < EB; ++e)
                            if (e < E) acc[e] = fmaf(xv[q], wrow[e], acc[e]);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int e = 0; e < EB; ++e) red[ks][tok][e] = acc[e];
    __syncthreads();
    if (ks != 0 || t >= T) return;
    float h[EB];
#pragma unroll
    for (int e = 0; e < EB; ++e) {
        float sum = 0.f;
        for (int q = 0; q < 16; ++q) sum += red[q][tok][e];
        h[e] = e < E ? sum + (bias ? __ldg(bias + e) : 0.f) : -INFINITY;
    }
    const int K = k + n_shared;
    topk_softmax_thread<EB>(h, E, k, n_shared, n_groups, topk_groups, topk_idx + size_t(t) * K,
                            topk_gate + size_t(t) * K, cnt, int64_t(t) * K);
}

constexpr int kSmallRouteWBytes = 128 << 10;  // W_g bytes the fused small-E router holds

template <typename TAct, int EB>
cudaError_t launch_small(const void* x, const float* Wg, const float* bias, int T, int d, int E, int k, int S,
                         int G, int M, int32_t* idx, float* gate, const RouteCounts cnt, cudaStream_t stream) {
    auto kern = route_small_kernel<TAct, EB>;
    constexpr size_t max_smem = size_t(kSmallRouteWBytes) + sizeof(float) * 16 * 16 * (EB + 1);
    static PerContext<int> smem_set;
    const cudaError_t attr_err = set_smem_limit_once(smem_set, kern, max_smem);
    if (attr_err != cudaSuccess) return attr_err;
    const size_t smem = sizeof(float) * (size_t(d) * E + 16 * 16 * (EB + 1));
    const bool wvec = E == EB && (reinterpret_cast<uintptr_t>(Wg) & 15) == 0;
    kern<<<(T + 15) / 16, 256, smem, stream>>>(static_cast<const TAct*>(x), Wg, bias, T, d, E, k, S, G, M, wvec, idx,
                                               gate, cnt);
    return cudaGetLastError();
}

template <typename TAct>
cudaError_t launch_small_t(const void* x, const float* Wg, const float* bias, int T, int d, int E, int k, int S,
                           int G, int M, int32_t* idx, float* gate, const RouteCounts cnt, cudaStream_t stream) {
    if (E <= 4) return launch_small<TAct, 4>(x, Wg, bias, T, d, E, k, S, G, M, idx, gate, cnt, stream);
    if (E <= 8) return launch_small<TAct, 8>(x, Wg, bias, T, d, E, k, S, G, M, idx, gate, cnt, stream);
    if (E <= 16) return launch_small<TAct, 16>(x, Wg, bias, T, d, E, k, S, G, M, idx, gate, cnt, stream);
    return launch_small<TAct, 32>(x, Wg, bias, T, d, E, k, S, G, M, idx, gate, cnt, stream);
}

int warps_along_experts(int E) { return E <= 8 ? 1 : E <= 16 ? 2 : E <= 32 ? 4 : 8; }

template <typename TAct, int WE>
cudaError_t launch_gemm(const void* x, const float* Wg, int T, int d, int E, int slice, int ks, float* scratch,
                        cudaStream_t stream) {
    using G = GemmShape<WE>;
    auto kern = route_gemm_kernel<TAct, WE>;
    static PerContext<int> smem_set;
    const cudaError_t attr_err = set_smem_limit_once(smem_set, kern, G::smem);
    if (attr_err != cudaSuccess) return attr_err;
    const dim3 grid((T + G::TT - 1) / G::TT, (E + G::TE - 1) / G::TE, ks);
    kern<<<grid, 256, G::smem, stream>>>(static_cast<const TAct*>(x), Wg, T, d, E, slice, scratch);
    return cudaGetLastError();
}

template <typename TAct>
cudaError_t launch_gemm_t(const void* x, const float* Wg, int T, int d, int E, int slice, int ks, float* scratch,
                          cudaStream_t stream) {
    switch (warps_along_experts(E)) {
        case 1: return launch_gemm<TAct, 1>(x, Wg, T, d, E, slice, ks, scratch, stream);
        case 2: return launch_gemm<TAct, 2>(x, Wg, T, d, E, slice, ks, scratch, stream);
        case 4: return launch_gemm<TAct, 4>(x, Wg, T, d, E, slice, ks, scratch, stream);
        default: return launch_gemm<TAct, 8>(x, Wg, T, d, E, slice, ks, scratch, stream);
    }
}

int slice_len(int d, int ks) { return ((d + ks - 1) / ks + kGK - 1) / kGK * kGK; }

}  // namespace

// Up to 64 slices while the partial logits stay within 16 MB (4M floats); at least 8.
int route_max_slices(int T, int E) {
    const int64_t te = int64_t(T > 0 ? T : 1) * (E > 0 ? E : 1);
    const int64_t m = (int64_t(1) << 22) / te;
    return m < 8 ? 8 : (m > 64 ? 64 : int(m));
}

int route_k_slices(int T, int d, int E) {
    const int we = warps_along_experts(E);
    const int tt = 128 * (8 / we), te = 8 * we;
    const int64_t tiles = int64_t((T + tt - 1) / tt) * ((E + te - 1) / te);
    const int sms = device_sm_count();
    // Pick the slice count whose waves of CTAs finish soonest, charging the partial
    // logits' HBM round trip against larger counts.
    int best = 1;
    double best_cost = 1e300;
    for (int ks = 1; ks <= route_max_slices(T, E); ++ks) {
        const int slice = slice_len(d, ks);
        if (ks > 1 && slice < 64) break;
        if (ks > 1 && int64_t(slice) * (ks - 1) >= d) continue;  // the last slice would be empty
        const int64_t ctas = tiles * ks;
        const double waves = double((ctas + sms - 1) / sms);
        const double compute = waves * double(tt) * te * slice / 128.0 + waves * 2000.0;  // SM clocks
        const double traffic = double(ks) * T * E * 8.0 / 3200.0;                        // ~3.2 KB per GPU clock
        const double cost = compute + traffic;
        if (cost < best_cost * 0.999) {
            best_cost = cost;
            best = ks;
        }
    }
    return best;
}

// The fused small-E kernel while W_g stays in L1 (E <= 32, d * E * 4 <= 128 KB).
bool route_uses_small_kernel(int d, int E) { return E <= 32 && int64_t(d) * E * 4 <= kSmallRouteWBytes; }

cudaError_t launch_route(int act_dtype, const void* x, const float* Wg, const float* bias, int T, int d, int E,
                         int k, int n_shared, int n_groups, int topk_groups, int32_t* topk_idx, float* topk_gate,
                         float* scratch, int32_t* hist, int32_t* near_ties, int32_t* status, cudaStream_t stream) {
    const RouteCounts cnt{hist, dispatch_blocks(int64_t(T) * (k + n_shared)), near_ties};
    if (route_uses_small_kernel(d, E))
        return act_dtype == MOE_F32
                   ? launch_small_t<float>(x, Wg, bias, T, d, E, k, n_shared, n_groups, topk_groups, topk_idx,
                                           topk_gate, cnt, stream)
                   : launch_small_t<__nv_bfloat16>(x, Wg, bias, T, d, E, k, n_shared, n_groups, topk_groups,
                                                   topk_idx, topk_gate, cnt, stream);
    int ks = 0;
    cudaError_t e;
    if (route_uses_tc(act_dtype, d, E)) {
        void* wsplit = reinterpret_cast<unsigned char*>(scratch) + route_partial_bytes_max(T, E);
        e = launch_route_tc(x, Wg, T, d, E, scratch, wsplit, status, &ks, stream);
    } else {
        ks = route_k_slices(T, d, E);
        const int slice = slice_len(d, ks);
        e = act_dtype == MOE_F32 ? launch_gemm_t<float>(x, Wg, T, d, E, slice, ks, scratch, stream)
                                 : launch_gemm_t<__nv_bfloat16>(x, Wg, T, d, E, slice, ks, scratch, stream);
    }
    if (e != cudaSuccess) return e;
    const int g2 = (T + 3) / 4;
    const int S = n_shared, G = n_groups, M = topk_groups;
    if (E <= 32) route_topk_kernel<1><<<g2, 128, 0, stream>>>(scratch, ks, bias, T, E, k, S, G, M, topk_idx, topk_gate, cnt);
    else if (E <= 64) route_topk_kernel<2><<<g2, 128, 0, stream>>>(scratch, ks, bias, T, E, k, S, G, M, topk_idx, topk_gate, cnt);
    else if (E <= 128) route_topk_kernel<4><<<g2, 128, 0, stream>>>(scratch, ks, bias, T, E, k, S, G, M, topk_idx, topk_gate, cnt);
    else if (E <= 256) route_topk_kernel<8><<<g2, 128, 0, stream>>>(scratch, ks, bias, T, E, k, S, G, M, topk_idx, topk_gate, cnt);
    else route_topk_kernel<16><<<g2, 128, 0, stream>>>(scratch, ks, bias, T, E, k, S, G, M, topk_idx, topk_gate, cnt);
    return cudaGetLastError();
}

}  // namespace moe
