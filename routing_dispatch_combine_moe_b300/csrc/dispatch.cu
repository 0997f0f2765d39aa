// Dispatch: group the T*k token-to-expert assignments by expert, drop the overflow
// past the per-expert capacity in token order, and gather the kept rows of x into
// one contiguous send buffer ("EP Math - Expert Parallelism (MoE)": "The dispatch
// all-to-all: bytes on the wire", "Capacity factor: fixing buffer sizes", "Token
// drop: what overflow costs"; "MoE Expert Parallelism Sizing": the drop happens
// before the exchange, in "Capacity semantics decide what crosses the wire").
//
// Four launches, all deterministic:
//   1. count   - per 256-assignment block, a per-expert histogram built with
//                warp-aggregated shared-memory atomics (__match_any_sync leaders);
//                stored expert-major, hist[e][block].
//   2. scan    - one CTA: per expert an exclusive scan over blocks (so hist becomes
//                "assignments of e in earlier blocks"), then block-wide scans of the
//                kept counts (row offsets), of the dropped counts (drop-list offsets)
//                and the virtual-rank chunk offsets.
//   3. scatter - per block again: an assignment's rank among its expert's
//                assignments is the scanned block prefix + the counts of earlier warps
//                in the block + its rank among equal ids in its warp (match_any +
//                popc of the lower lanes). Rank < capacity gives its row; otherwise it
//                is dropped. Writes pos, row_src and the drop list.
//   4. gather  - one warp per token copies x[t] once from HBM into each of its kept
//                rows with 16-byte vector loads and stores.
// Because rows are ordered (expert, token), virtual rank r's rows (experts
// [r E/D, (r+1) E/D)) form one contiguous chunk: the layout of an all-to-all input buffer, which
// holds a separate chunk for every destination rank.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kWarps = kDispatchBlock / 32;

__global__ void __launch_bounds__(kDispatchBlock) count_kernel(const int32_t* __restrict__ topk_idx, int64_t A,
                                                               int E, int nblk, int32_t* __restrict__ hist,
                                                               int32_t* status) {
    __shared__ int sh[MOE_MAX_E];
    const int tid = threadIdx.x, lane = tid & 31;
    for (int e = tid; e < E; e += kDispatchBlock) sh[e] = 0;
    __syncthreads();
    const int64_t a = int64_t(blockIdx.x) * kDispatchBlock + tid;
    int e = -1;
    if (a < A) {
        e = topk_idx[a];
        if (e < 0 || e >= E) {
            set_status(status, MOE_DEV_ERR_INDEX);
            e = -1;
        }
    }
    const unsigned active = __ballot_sync(0xFFFFFFFFu, e >= 0);
    if (e >= 0) {
        const unsigned peers = __match_any_sync(active, e);
        if (lane == __ffs(peers) - 1) atomicAdd(&sh[e], __popc(peers));
    }
    __syncthreads();
    for (int ee = tid; ee < E; ee += kDispatchBlock) hist[size_t(ee) * nblk + blockIdx.x] = sh[ee];
}

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int n = __shfl_up_sync(0xFFFFFFFFu, v, off);
        if (lane >= off) v += n;
    }
    return v;
}

// Exclusive scan of one int per thread across a 1024-thread block; returns the
// exclusive prefix and writes the block total to *total (shared).
__device__ int block_excl_scan(int v, int* warp_sums, int* total) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int incl = warp_incl_scan(v, lane);
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int ws = warp_sums[lane];
        const int wi = warp_incl_scan(ws, lane);
        warp_sums[lane] = wi - ws;
        if (lane == 31) *total = wi;
    }
    __syncthreads();
    const int r = warp_sums[warp] + incl - v;
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(1024) scan_kernel(int E, int E_capped, int D, int nblk, int64_t capacity,
                                                    int32_t* __restrict__ hist, int32_t* __restrict__ counts_routed,
                                                    int32_t* __restrict__ counts_kept, int32_t* __restrict__ offsets,
                                                    int32_t* __restrict__ drop_offsets,
                                                    int32_t* __restrict__ rank_offsets,
                                                    int32_t* __restrict__ n_dropped) {
    __shared__ int routed[MOE_MAX_E];
    __shared__ int offs[MOE_MAX_E + 1];
    __shared__ int warp_sums[32];
    __shared__ int totals[2];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    for (int e = warp; e < E; e += 32) {
        int run = 0;
        int32_t* row = hist + size_t(e) * nblk;
        for (int b0 = 0; b0 < nblk; b0 += 32) {
            const int b = b0 + lane;
            const int v = b < nblk ? row[b] : 0;
            const int incl = warp_incl_scan(v, lane);
            if (b < nblk) row[b] = run + incl - v;
            run += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
        if (lane == 0) routed[e] = run;
    }
    __syncthreads();

    const int cr = tid < E ? routed[tid] : 0;
    const int ck = (capacity < 0 || tid >= E_capped || cr <= capacity) ? cr : int(capacity);
    const int off = block_excl_scan(ck, warp_sums, &totals[0]);
    const int doff = block_excl_scan(cr - ck, warp_sums, &totals[1]);
    if (tid < E) {
        counts_routed[tid] = cr;
        counts_kept[tid] = ck;
        offsets[tid] = off;
        drop_offsets[tid] = doff;
        offs[tid] = off;
    }
    if (tid == 0) {
        offsets[E] = totals[0];
        offs[E] = totals[0];
        *n_dropped = totals[1];
    }
    __syncthreads();
    if (tid <= D) rank_offsets[tid] = offs[tid * (E_capped / D)];
}

__global__ void __launch_bounds__(kDispatchBlock) scatter_kernel(const int32_t* __restrict__ topk_idx, int64_t A,
                                                                 int E, int E_capped, int nblk, int64_t capacity,
                                                                 const int32_t* __restrict__ hist,
                                                                 const int32_t* __restrict__ offsets,
                                                                 const int32_t* __restrict__ drop_offsets,
                                                                 int32_t* __restrict__ pos,
                                                                 int32_t* __restrict__ row_src,
                                                                 int32_t* __restrict__ drop_list) {
    __shared__ int cnt[kWarps][MOE_MAX_E];
    const int tid = threadIdx.x, warp = tid >> 5;
    for (int i = tid; i < kWarps * E; i += kDispatchBlock) (&cnt[0][0])[(i / E) * MOE_MAX_E + (i % E)] = 0;
    __syncthreads();
    const int64_t a = int64_t(blockIdx.x) * kDispatchBlock + tid;
    int e = -1;
    if (a < A) {
        e = topk_idx[a];
        if (e < 0 || e >= E) e = -1;
    }
    const unsigned active = __ballot_sync(0xFFFFFFFFu, e >= 0);
    int rank_in_warp = 0;
    if (e >= 0) {
        const unsigned peers = __match_any_sync(active, e);
        rank_in_warp = __popc(peers & lanemask_lt());
        if (rank_in_warp == 0) cnt[warp][e] = __popc(peers);
    }
    __syncthreads();
    if (a >= A) return;
    if (e < 0) {
        pos[a] = -1;
        return;
    }
    int rank = hist[size_t(e) * nblk + blockIdx.x] + rank_in_warp;
    for (int w = 0; w < warp; ++w) rank += cnt[w][e];
    if (capacity < 0 || e >= E_capped || rank < capacity) {
        const int row = offsets[e] + rank;
        pos[a] = row;
        row_src[row] = int32_t(a);
    } else {
        pos[a] = -1;
        drop_list[drop_offsets[e] + (rank - int(capacity))] = int32_t(a);
    }
}

// One warp per token: x[t] is read once and written to each of its kept rows.
__global__ void __launch_bounds__(256) gather_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ pos,
                                                     uint4* __restrict__ xperm, int T, int k, int vec_per_row,
                                                     int64_t max_rows) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T) return;
    int p = -1;
    if (lane < k) {
        p = pos[size_t(t) * k + lane];
        if (p >= max_rows) p = -1;
    }
    int dst[MOE_MAX_K];
#pragma unroll
    for (int j = 0; j < MOE_MAX_K; ++j) dst[j] = __shfl_sync(0xFFFFFFFFu, p, j);
    const uint4* src = x + size_t(t) * vec_per_row;
    constexpr int U = 8;  // 16-byte pieces per lane in flight
    for (int v0 = lane; v0 < vec_per_row; v0 += 32 * U) {
        uint4 buf[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = v0 + 32 * u;
            if (v < vec_per_row) buf[u] = __ldg(src + v);
        }
#pragma unroll
        for (int j = 0; j < MOE_MAX_K; ++j) {
            if (j < k && dst[j] >= 0) {
                uint4* d = xperm + size_t(dst[j]) * vec_per_row;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int v = v0 + 32 * u;
                    if (v < vec_per_row) d[v] = buf[u];
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_dispatch(const DispatchArgs& a, cudaStream_t stream) {
    const int64_t A = int64_t(a.T) * a.k;
    const int nblk = dispatch_blocks(A);
    count_kernel<<<nblk, kDispatchBlock, 0, stream>>>(a.topk_idx, A, a.E, nblk, a.hist, a.status);
    scan_kernel<<<1, 1024, 0, stream>>>(a.E, a.E_capped, a.D, nblk, a.capacity, a.hist, a.counts_routed,
                                        a.counts_kept, a.offsets, a.drop_offsets, a.rank_offsets, a.n_dropped);
    scatter_kernel<<<nblk, kDispatchBlock, 0, stream>>>(a.topk_idx, A, a.E, a.E_capped, nblk, a.capacity, a.hist,
                                                        a.offsets, a.drop_offsets, a.pos, a.row_src, a.drop_list);
    const int vec_per_row = int(int64_t(a.d) * a.act_bytes / 16);
    gather_kernel<<<(a.T + 7) / 8, 256, 0, stream>>>(static_cast<const uint4*>(a.x), a.pos,
                                                      static_cast<uint4*>(a.xperm), a.T, a.k, vec_per_row, A);
    return cudaGetLastError();
}

}  // namespace moe
