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
//                stored expert-major, hist[e][block]. Skipped when the router has
//                already counted (the layer forward: integer atomics from the top-k
//                writers into the zeroed histogram give the same counts).
//   2. scan    - a warp per expert scans its row of block counts (so hist becomes
//                "assignments of e in earlier blocks"); the last CTA to finish then
//                scans the kept counts (row offsets), the dropped counts (drop-list
//                offsets) and the virtual-rank chunk offsets.
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

// quiet_empty: an id of -1 marks "no assignment" and is skipped without a flag.
__global__ void __launch_bounds__(kDispatchBlock) count_kernel(const int32_t* __restrict__ topk_idx, int64_t A,
                                                               int E, int nblk, int32_t* __restrict__ hist,
                                                               int32_t* status, int quiet_empty = 0) {
    __shared__ int sh[MOE_MAX_E];
    const int tid = threadIdx.x, lane = tid & 31;
    for (int e = tid; e < E; e += kDispatchBlock) sh[e] = 0;
    __syncthreads();
    const int64_t a = int64_t(blockIdx.x) * kDispatchBlock + tid;
    int e = -1;
    if (a < A) {
        e = topk_idx[a];
        if (e < 0 || e >= E) {
            if (!(quiet_empty && e == -1)) set_status(status, MOE_DEV_ERR_INDEX);
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

// Scan, over ceil(E / 32) CTAs of 32 warps: warp w of CTA c turns expert e = 32 c + w's
// row of block counts into its exclusive scan (so hist[e][b] becomes "assignments of e
// in earlier blocks") and writes the row total to counts_routed[e]. Each CTA then
// takes a ticket; the last one to finish (no CTA waits for another) reads all totals
// back and scans the kept counts (row offsets), the dropped counts (drop-list
// offsets), the routed counts and the virtual-rank chunk offsets. With one CTA no
// ticket is needed (ticket may be null); otherwise *ticket starts at 0 and is left at 0.
__global__ void __launch_bounds__(1024) scan_kernel(int E, int E_capped, int D, int nblk, int64_t capacity,
                                                    int padded, int32_t* __restrict__ hist,
                                                    int32_t* __restrict__ counts_routed,
                                                    int32_t* __restrict__ counts_kept, int32_t* __restrict__ offsets,
                                                    int32_t* __restrict__ drop_offsets,
                                                    int32_t* __restrict__ routed_offsets,
                                                    int32_t* __restrict__ rank_offsets,
                                                    int32_t* __restrict__ n_dropped, int32_t* ticket) {
    __shared__ int offs[MOE_MAX_E + 1];
    __shared__ int warp_sums[32];
    __shared__ int totals[3];
    __shared__ int is_last;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // this warp's expert: SB chunks of 32 blocks loaded before they are scanned
    constexpr int SB = 8;
    const int e = int(blockIdx.x) * 32 + warp;
    if (e < E) {
        int32_t* row = hist + size_t(e) * nblk;
        int run = 0;
        for (int b0 = 0; b0 < nblk; b0 += 32 * SB) {
            int v[SB];
#pragma unroll
            for (int j = 0; j < SB; ++j) {
                const int b = b0 + 32 * j + lane;
                v[j] = b < nblk ? row[b] : 0;
            }
#pragma unroll
            for (int j = 0; j < SB; ++j) {
                if (b0 + 32 * j >= nblk) break;  // no blocks left (uniform over the warp)
                const int b = b0 + 32 * j + lane;
                const int incl = warp_incl_scan(v[j], lane);
                if (b < nblk) row[b] = run + incl - v[j];
                run += __shfl_sync(0xFFFFFFFFu, incl, 31);
            }
        }
        if (lane == 0) counts_routed[e] = run;
    }
    if (gridDim.x > 1) {
        __threadfence();
        __syncthreads();
        if (tid == 0) is_last = atomicAdd(ticket, 1) == int(gridDim.x) - 1;
        __syncthreads();
        if (!is_last) return;
        __threadfence();
    } else {
        __syncthreads();
    }

    const int cr = tid < E ? __ldcg(counts_routed + tid) : 0;
    const int ck = (capacity < 0 || tid >= E_capped || cr <= capacity) ? cr : int(capacity);
    const int scanned = block_excl_scan(ck, warp_sums, &totals[0]);
    const int doff = block_excl_scan(cr - ck, warp_sums, &totals[1]);
    const int roff = block_excl_scan(cr, warp_sums, &totals[2]);
    // padded layout: every expert owns `capacity` rows
    const int off = padded ? tid * int(capacity) : scanned;
    if (tid < E) {
        counts_kept[tid] = ck;
        offsets[tid] = off;
        drop_offsets[tid] = doff;
        routed_offsets[tid] = roff;
        offs[tid] = off;
    }
    if (tid == 0) {
        const int end = padded ? E * int(capacity) : totals[0];
        offsets[E] = end;
        offs[E] = end;
        routed_offsets[E] = totals[2];
        *n_dropped = totals[1];
        if (gridDim.x > 1) *ticket = 0;
    }
    __syncthreads();
    if (tid <= D) rank_offsets[tid] = offs[tid * (E_capped / D)];
}

// fp32 bits mapped so that unsigned order is value order (negatives flipped, the
// sign bit set on non-negatives); -0 sorts just below +0.
__device__ __forceinline__ uint32_t order_key(float g) {
    const uint32_t b = __float_as_uint(g);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// With `elist` set (gate drop policy) it only lists each expert's assignments in
// token order at elist[routed_offsets[e] + rank], with their gates' order keys at the
// same place of elist + A; select_kernel then places them.
__global__ void __launch_bounds__(kDispatchBlock) scatter_kernel(const int32_t* __restrict__ topk_idx, int64_t A,
                                                                 int E, int E_capped, int nblk, int64_t capacity,
                                                                 const int32_t* __restrict__ hist,
                                                                 const int32_t* __restrict__ offsets,
                                                                 const int32_t* __restrict__ drop_offsets,
                                                                 const int32_t* __restrict__ routed_offsets,
                                                                 int32_t* __restrict__ elist,
                                                                 const float* __restrict__ topk_gate,
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
    if (elist) {
        elist[routed_offsets[e] + rank] = int32_t(a);
        elist[A + routed_offsets[e] + rank] = int32_t(order_key(topk_gate[a]));
        return;
    }
    if (capacity < 0 || e >= E_capped || rank < capacity) {
        const int row = offsets[e] + rank;
        pos[a] = row;
        row_src[row] = int32_t(a);
    } else {
        pos[a] = -1;
        drop_list[drop_offsets[e] + (rank - int(capacity))] = int32_t(a);
    }
}

constexpr int kSelThreads = 512;
constexpr int kSelKeys = 9216;  // keys of one expert cached in shared memory (36 KB)

// Block-wide exclusive scan of one int per thread (kSelThreads threads); *total gets the sum.
__device__ int sel_excl_scan(int v, int* warp_sums, int* total) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int incl = warp_incl_scan(v, lane);
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int ws = lane < kSelThreads / 32 ? warp_sums[lane] : 0;
        const int wi = warp_incl_scan(ws, lane);
        if (lane < kSelThreads / 32) warp_sums[lane] = wi - ws;
        if (lane == 31) *total = wi;
    }
    __syncthreads();
    const int r = warp_sums[warp] + incl - v;
    __syncthreads();
    return r;
}

// Gate drop policy, one CTA per expert. The expert's n routed assignments are listed
// in token order with their gates' order keys (scatter_kernel). Kept are the keys
// above thr, the keep_n-th largest key, plus the first need_eq keys equal to it in
// token order; thr is found by a most-significant-digit-first radix select (digits
// of 11, 11 and 10 bits over 2048 shared bins, the bin crossing the wanted rank found
// by a block suffix scan). The keys sit in shared memory when they fit. A final pass
// scans, per 512-key chunk, the packed pair (greater, equal) to place every
// assignment: kept_before = greater_before + min(equal_before, need_eq); kept rows go
// to the expert's rows in token order, the rest to the drop list in token order.
__global__ void __launch_bounds__(kSelThreads) select_kernel(const int32_t* __restrict__ elist, int64_t A,
                                                             const int32_t* __restrict__ routed_offsets,
                                                             const int32_t* __restrict__ counts_routed,
                                                             const int32_t* __restrict__ counts_kept,
                                                             const int32_t* __restrict__ offsets,
                                                             const int32_t* __restrict__ drop_offsets,
                                                             int32_t* __restrict__ pos,
                                                             int32_t* __restrict__ row_src,
                                                             int32_t* __restrict__ drop_list) {
    __shared__ uint32_t skey[kSelKeys];
    __shared__ int hist[2048];
    __shared__ int warp_sums[32];
    __shared__ int totals[2];
    __shared__ int sel_bin, sel_rank;
    const int e = blockIdx.x, tid = threadIdx.x;
    const int n = counts_routed[e], keep_n = counts_kept[e];
    const int32_t* list = elist + routed_offsets[e];
    const uint32_t* gkey = reinterpret_cast<const uint32_t*>(elist + A) + routed_offsets[e];
    const int base = offsets[e], dbase = drop_offsets[e];
    const bool cached = n <= kSelKeys;
    const bool partial = keep_n > 0 && keep_n < n;
    if (cached && partial)
        for (int i = tid; i < n; i += kSelThreads) skey[i] = gkey[i];
    __syncthreads();
    auto key_at = [&](int i) -> uint32_t { return cached ? skey[i] : __ldg(gkey + i); };

    uint32_t thr = 0;
    int need_eq = 0;
    if (partial) {
        uint32_t prefix = 0, mask = 0;
        int rank = keep_n;  // 1-based rank, from the largest, of the last kept key
#pragma unroll
        for (int pass = 0; pass < 3; ++pass) {
            const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
            const uint32_t dmask = pass == 2 ? 0x3FFu : 0x7FFu;
            for (int b = tid; b < 2048; b += kSelThreads) hist[b] = 0;
            __syncthreads();
            for (int i = tid; i < n; i += kSelThreads) {
                const uint32_t key = key_at(i);
                if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & dmask], 1);
            }
            __syncthreads();
            // thread t owns bins 4t..4t+3; count the keys in all higher bins
            int own = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) own += hist[4 * tid + q];
            const int below = sel_excl_scan(own, warp_sums, &totals[0]);  // keys in the bins of lower threads
            int cum = totals[0] - below - own;                             // keys in the bins of higher threads
            for (int q = 3; q >= 0; --q) {
                const int b = 4 * tid + q;
                const int h = hist[b];
                if (cum < rank && cum + h >= rank) {
                    sel_bin = b;
                    sel_rank = rank - cum;
                }
                cum += h;
            }
            __syncthreads();
            prefix |= uint32_t(sel_bin) << shift;
            mask |= dmask << shift;
            rank = sel_rank;
            __syncthreads();
        }
        thr = prefix;
        need_eq = rank;
    }

    int carry_gt = 0, carry_eq = 0;
    for (int i0 = 0; i0 < n; i0 += kSelThreads) {
        const int i = i0 + tid;
        const bool valid = i < n;
        const int a = valid ? list[i] : 0;
        int kept_before;
        bool keep;
        if (keep_n >= n) {
            keep = valid;
            kept_before = i;
        } else if (keep_n == 0) {
            keep = false;
            kept_before = 0;
        } else {
            const uint32_t key = valid ? key_at(i) : 0u;
            const bool gt = valid && key > thr, eq = valid && key == thr;
            const int packed = (gt ? 1 << 16 : 0) | (eq ? 1 : 0);
            const int excl = sel_excl_scan(packed, warp_sums, &totals[0]);
            const int gt_before = carry_gt + (excl >> 16), eq_before = carry_eq + (excl & 0xFFFF);
            keep = gt || (eq && eq_before < need_eq);
            kept_before = gt_before + min(eq_before, need_eq);
            carry_gt += totals[0] >> 16;
            carry_eq += totals[0] & 0xFFFF;
        }
        if (keep) {
            pos[a] = base + kept_before;
            row_src[base + kept_before] = a;
        } else if (valid) {
            pos[a] = -1;
            drop_list[dbase + (i - kept_before)] = a;
        }
    }
}

// Padded layout: rows [offsets[e] + kept, offsets[e] + capacity) of expert e are
// zeroed and marked as holding no assignment. Grid (ceil(capacity / 8), E): one
// warp per row, 16-byte stores.
__global__ void __launch_bounds__(256) pad_rows_kernel(const int32_t* __restrict__ counts_kept,
                                                       const int32_t* __restrict__ offsets, int capacity,
                                                       uint4* __restrict__ xperm, int vec_per_row,
                                                       int32_t* __restrict__ row_src) {
    const int e = blockIdx.y, lane = threadIdx.x & 31;
    const int i = blockIdx.x * 8 + (threadIdx.x >> 5);  // row within the segment
    if (i >= capacity || i < counts_kept[e]) return;
    const int64_t r = int64_t(offsets[e]) + i;
    uint4* row = xperm + r * vec_per_row;
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (int v = lane; v < vec_per_row; v += 32) row[v] = z;
    if (lane == 0) row_src[r] = -1;
}

// One warp per token and column slice (blockIdx.y of gridDim.y): the slice of x[t] is
// read once and written to each of the token's kept rows. Small batches split the row
// over several warps so that enough of them are in flight.
__global__ void __launch_bounds__(256) gather_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ pos,
                                                     uint4* __restrict__ xperm, int T, int k, int vec_per_row,
                                                     int64_t max_rows) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T) return;
    const int per = (vec_per_row + gridDim.y - 1) / gridDim.y;
    const int vbeg = blockIdx.y * per, vend = min(vec_per_row, vbeg + per);
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
    for (int v0 = vbeg + lane; v0 < vend; v0 += 32 * U) {
        uint4 buf[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = v0 + 32 * u;
            if (v < vend) buf[u] = __ldg(src + v);
        }
#pragma unroll
        for (int j = 0; j < MOE_MAX_K; ++j) {
            if (j < k && dst[j] >= 0) {
                uint4* d = xperm + size_t(dst[j]) * vec_per_row;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int v = v0 + 32 * u;
                    if (v < vend) d[v] = buf[u];
                }
            }
        }
    }
}

// Gather by bulk copies: one thread per CTA moves each of its tokens' x row into
// shared memory with one bulk copy (completion counted on an mbarrier) and writes it
// to each of the token's kept rows with one bulk store per row, so the copy engine
// moves whole rows and the SM only issues. Tokens t = blockIdx.x + i * gridDim.x go
// through kGbBufs row buffers: while one buffer's stores drain, the next row loads.
// Rows are row_bytes long (a multiple of 16, as are the addresses).
constexpr int kGbBufs = 3;

__device__ __forceinline__ void bulk_load_row(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void bulk_store_row(void* dst, const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_addr(src)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Waits until at most N committed bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Waits until every committed bulk group has completed, its writes included.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__global__ void __launch_bounds__(32) gather_bulk_kernel(const unsigned char* __restrict__ x,
                                                         const int32_t* __restrict__ pos,
                                                         unsigned char* __restrict__ xperm, int T, int k,
                                                         uint32_t row_bytes, int64_t max_rows, int32_t* status) {
    extern __shared__ __align__(128) unsigned char gb_rows[];
    __shared__ uint64_t full[kGbBufs];
    if (threadIdx.x != 0) return;
    for (int b = 0; b < kGbBufs; ++b) mbar_init(&full[b], 1);
    fence_barrier_init();
    fence_proxy_async_smem();
    const int first = int(blockIdx.x), step = int(gridDim.x);
    const int n = first < T ? (T - 1 - first) / step + 1 : 0;  // tokens of this CTA
    int issued = 0;                                             // loads issued: tokens [0, issued)
    auto load = [&]() {
        const int b = issued % kGbBufs;
        mbar_arrive_expect_tx(&full[b], row_bytes);
        bulk_load_row(gb_rows + size_t(b) * row_bytes, x + size_t(first + issued * step) * row_bytes, row_bytes,
                      &full[b]);
        ++issued;
    };
    // bounded wait for load i; false after the time limit
    auto wait_load = [&](int i) {
        const unsigned long long t0 = globaltimer_ns();
        while (!mbar_try_wait(&full[i % kGbBufs], uint32_t(i / kGbBufs) & 1u))
            if (globaltimer_ns() - t0 > kWaitTimeoutNs) return false;
        return true;
    };
    while (issued < kGbBufs - 1 && issued < n) load();
    int i = 0;
    for (; i < n; ++i) {
        if (!wait_load(i)) {
            set_status(status, MOE_DEV_ERR_TIMEOUT);
            break;
        }
        fence_proxy_async_smem();
        const int b = i % kGbBufs;
        const int t = first + i * step;
        for (int j = 0; j < k; ++j) {
            const int p = __ldg(pos + size_t(t) * k + j);
            if (p >= 0 && p < max_rows)
                bulk_store_row(xperm + size_t(p) * row_bytes, gb_rows + size_t(b) * row_bytes, row_bytes);
        }
        bulk_commit();
        // the buffer of token i - 1 is free once every group but the newest has read it
        bulk_wait_read<1>();
        if (issued < n) load();
    }
    bulk_wait_all();
    // loads still in flight after a timeout must land before the CTA's shared memory goes
    for (int j = i; j < issued; ++j) wait_load(j);
}

}  // namespace

dim3 gather_grid(int T, int vec_per_row);

// Rows a bulk-copy gather CTA holds (kGbBufs of them) must fit its shared memory; small
// batches keep the warp gather, whose column slices spread one token over several SMs.
bool gather_uses_bulk(int T, int64_t row_bytes) { return T >= 512 && row_bytes * kGbBufs <= 96 * 1024; }

cudaError_t launch_gather(const void* x, const int32_t* pos, void* xperm, int T, int k, int64_t row_bytes,
                          int64_t max_rows, int32_t* status, cudaStream_t stream) {
    if (gather_uses_bulk(T, row_bytes)) {
        const size_t smem = size_t(kGbBufs) * size_t(row_bytes);
        static PerContext<int> smem_set;
        const cudaError_t e = set_smem_limit_once(smem_set, gather_bulk_kernel, 96 * 1024);
        if (e != cudaSuccess) return e;
        const int per_sm = int((200 * 1024) / (smem + 1024));
        const int ctas = T < device_sm_count() * per_sm ? T : device_sm_count() * per_sm;
        gather_bulk_kernel<<<ctas, 32, smem, stream>>>(static_cast<const unsigned char*>(x), pos,
                                                       static_cast<unsigned char*>(xperm), T, k, uint32_t(row_bytes),
                                                       max_rows, status);
        return cudaGetLastError();
    }
    const int vec_per_row = int(row_bytes / 16);
    gather_kernel<<<gather_grid(T, vec_per_row), 256, 0, stream>>>(static_cast<const uint4*>(x), pos,
                                                                   static_cast<uint4*>(xperm), T, k, vec_per_row,
                                                                   max_rows);
    return cudaGetLastError();
}

// Token blocks of 8 warps, times column slices of at least 64 pieces, until about two
// CTAs per SM are in flight.
dim3 gather_grid(int T, int vec_per_row) {
    const int nb = (T + 7) / 8;
    const int want = (2 * device_sm_count() + nb - 1) / nb;
    const int cap = vec_per_row / 64 > 1 ? vec_per_row / 64 : 1;
    return dim3(unsigned(nb), unsigned(want < cap ? (want > 1 ? want : 1) : cap));
}

cudaError_t launch_dispatch(const DispatchArgs& a, cudaStream_t stream) {
    const int64_t A = int64_t(a.T) * a.k;
    const int nblk = dispatch_blocks(A);
    const bool by_gate = a.drop_policy == MOE_DROP_LOW_GATE && a.capacity >= 0;
    const bool padded = a.layout == MOE_LAYOUT_PADDED;
    const int vec_per_row = int(int64_t(a.d) * a.act_bytes / 16);
    const int64_t rows = padded ? int64_t(a.E) * a.capacity : A;
    if (!a.counted) count_kernel<<<nblk, kDispatchBlock, 0, stream>>>(a.topk_idx, A, a.E, nblk, a.hist, a.status);
    scan_kernel<<<(a.E + 31) / 32, 1024, 0, stream>>>(a.E, a.E_capped, a.D, nblk, a.capacity, padded ? 1 : 0,
                                                       a.hist, a.counts_routed, a.counts_kept, a.offsets,
                                                       a.drop_offsets, a.routed_offsets, a.rank_offsets, a.n_dropped,
                                                       a.scan_ticket);
    scatter_kernel<<<nblk, kDispatchBlock, 0, stream>>>(a.topk_idx, A, a.E, a.E_capped, nblk, a.capacity, a.hist,
                                                        a.offsets, a.drop_offsets, a.routed_offsets,
                                                        by_gate ? a.elist : nullptr, a.topk_gate, a.pos, a.row_src,
                                                        a.drop_list);
    if (by_gate)
        select_kernel<<<a.E, kSelThreads, 0, stream>>>(a.elist, A, a.routed_offsets, a.counts_routed,
                                                       a.counts_kept, a.offsets, a.drop_offsets, a.pos, a.row_src,
                                                       a.drop_list);
    if (padded && a.capacity > 0)
        pad_rows_kernel<<<dim3(unsigned((a.capacity + 7) / 8), unsigned(a.E)), 256, 0, stream>>>(
            a.counts_kept, a.offsets, int(a.capacity),
                                                 static_cast<uint4*>(a.xperm), vec_per_row, a.row_src);
    if (!a.skip_gather) {
        const cudaError_t e = launch_gather(a.x, a.pos, a.xperm, a.T, a.k, int64_t(vec_per_row) * 16, rows, a.status,
                                            stream);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

namespace {

// Deduplicated dispatch ("MoE Expert Parallelism Sizing", "First-order dispatch and
// combine bytes", the deduplicated rows): token t sends its row once to each virtual
// rank holding one of its kept routed assignments, and the receiving rank copies it
// to each of its expert rows. Launches:
//   1. mask    - per token, the set of ranks its kept routed assignments live on,
//                written as D slots (slot r = r, or -1 when nothing goes to r);
//   2-4.       - count / scan / scatter over those T*D slots with D "experts" and no
//                capacity: send counts, send offsets, and each (token, rank) pair's
//                send row, rank-major and in token order inside a rank;
//   5. gather  - x rows into the send buffer (one warp per token, one read of x[t]);
//   6. fan-out - the receiving side: every kept assignment's row is copied from the
//                send row of (token, rank of its expert); shared experts (ids past the
//                routed ones) are replicated, so their rows come from x itself.
__global__ void __launch_bounds__(256) dedup_mask_kernel(const int32_t* __restrict__ topk_idx,
                                                         const int32_t* __restrict__ pos, int T, int K,
                                                         int E_routed, int D, int32_t* __restrict__ slots) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= T) return;
    const int per_rank = E_routed / D;
    uint32_t mask = 0;
    for (int j = 0; j < K; ++j) {
        const int e = topk_idx[size_t(t) * K + j];
        if (pos[size_t(t) * K + j] >= 0 && e >= 0 && e < E_routed) mask |= 1u << (e / per_rank);
    }
    for (int r = 0; r < D; ++r) slots[size_t(t) * D + r] = ((mask >> r) & 1u) ? r : -1;
}

__global__ void __launch_bounds__(256) fanout_kernel(const uint4* __restrict__ x, const uint4* __restrict__ xsend,
                                                     const int32_t* __restrict__ topk_idx,
                                                     const int32_t* __restrict__ pos,
                                                     const int32_t* __restrict__ send_pos, uint4* __restrict__ xperm,
                                                     int T, int K, int E_routed, int D, int vec_per_row,
                                                     int64_t max_rows, int64_t max_send, int32_t* status) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T) return;
    int dst = -1, src = -1;  // src >= 0: send row; src == -2: x[t]
    if (lane < K) {
        const size_t a = size_t(t) * K + lane;
        const int p = pos[a], e = topk_idx[a];
        if (p >= 0 && p < max_rows) {
            if (e >= 0 && e < E_routed) {
                const int s = send_pos[size_t(t) * D + e / (E_routed / D)];
                if (s >= 0 && s < max_send) {
                    dst = p;
                    src = s;
                } else {
                    set_status(status, MOE_DEV_ERR_INDEX);
                }
            } else {
                dst = p;
                src = -2;
            }
        }
    }
    for (int j = 0; j < K; ++j) {
        const int dj = __shfl_sync(0xFFFFFFFFu, dst, j);
        const int sj = __shfl_sync(0xFFFFFFFFu, src, j);
        if (dj < 0) continue;
        const uint4* from = sj == -2 ? x + size_t(t) * vec_per_row : xsend + size_t(sj) * vec_per_row;
        uint4* to = xperm + size_t(dj) * vec_per_row;
        for (int v = lane; v < vec_per_row; v += 32) to[v] = __ldg(from + v);
    }
}

}  // namespace

cudaError_t launch_dedup(const DedupArgs& a, cudaStream_t stream) {
    const int64_t A2 = int64_t(a.T) * a.D;
    const int nblk = dispatch_blocks(A2);
    const int vec_per_row = int(int64_t(a.d) * a.act_bytes / 16);
    dedup_mask_kernel<<<(a.T + 255) / 256, 256, 0, stream>>>(a.topk_idx, a.pos, a.T, a.K, a.E_routed, a.D, a.slots);
    count_kernel<<<nblk, kDispatchBlock, 0, stream>>>(a.slots, A2, a.D, nblk, a.hist, a.status, 1);
    scan_kernel<<<1, 1024, 0, stream>>>(a.D, a.D, 1, nblk, -1, 0, a.hist, a.send_counts, a.kept_scratch,
                                        a.send_offsets, a.drop_offsets, a.routed_offsets, a.rank_offsets,
                                        a.n_dropped, nullptr);
    scatter_kernel<<<nblk, kDispatchBlock, 0, stream>>>(a.slots, A2, a.D, a.D, nblk, -1, a.hist, a.send_offsets,
                                                        a.drop_offsets, a.routed_offsets, nullptr, nullptr,
                                                        a.send_pos, a.send_src, nullptr);
    if (a.fp8_rows) {
        const cudaError_t e1 = launch_fp8_send_rows(a.x, a.send_pos, a.T, a.D, a.d, A2, static_cast<uint8_t*>(a.xsend),
                                                    a.xsend_scale, a.status, stream);
        if (e1 != cudaSuccess) return e1;
        return launch_fp8_row_fanout(a.x, static_cast<const uint8_t*>(a.xsend), a.xsend_scale, a.topk_idx, a.pos,
                                     a.send_pos, a.xq, a.xscale, a.T, a.K, a.E_routed, a.D, a.d, a.rows, A2,
                                     a.status, stream);
    }
    if (a.fp8) {
        const cudaError_t e1 = launch_fp8_send(a.x, a.slots, a.send_pos, a.T, a.D, a.d, A2,
                                               static_cast<uint8_t*>(a.xsend), a.xsend_scale, a.status, stream);
        if (e1 != cudaSuccess) return e1;
        return launch_fp8_fanout(a.x, static_cast<const uint8_t*>(a.xsend), a.xsend_scale, a.topk_idx, a.pos,
                                 a.send_pos, a.xperm, a.T, a.K, a.E_routed, a.D, a.d, a.rows, A2, a.status, stream);
    }
    const cudaError_t ge = launch_gather(a.x, a.send_pos, a.xsend, a.T, a.D, int64_t(vec_per_row) * 16, A2, a.status,
                                         stream);
    if (ge != cudaSuccess) return ge;
    fanout_kernel<<<(a.T + 7) / 8, 256, 0, stream>>>(static_cast<const uint4*>(a.x),
                                                      static_cast<const uint4*>(a.xsend), a.topk_idx, a.pos,
                                                      a.send_pos, static_cast<uint4*>(a.xperm), a.T, a.K,
                                                      a.E_routed, a.D, vec_per_row, a.rows, A2, a.status);
    return cudaGetLastError();
}

}  // namespace moe
