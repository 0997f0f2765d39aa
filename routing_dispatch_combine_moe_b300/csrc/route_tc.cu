// Router logits H = x W_g on the 5th-generation tensor cores, for bf16 activations and
// E >= 64 ("Mixture-of-Experts (MoE) Architecture and Expert Parallelism", section 2
// "The Gating Network Formulation": H(x) = x W_g). The logits must stay as accurate as
// an fp32 dot product, because KeepTopK and the softmax are decided on them:
//
// * W_g (fp32) is split exactly into three bf16 terms, W_g = hi + mid + lo with
//   hi = bf16(w), mid = bf16(w - hi), lo = bf16(w - hi - mid): each rounding leaves a
//   remainder of at most 8 significant bits for the next term, so the sum is w itself.
//   Every product of a bf16 x with a bf16 term is exact in fp32.
// * The tensor core's fp32 accumulation loses a little with every instruction it
//   adds into its accumulator, in proportion to the accumulator's size. So each chunk
//   of 128 elements of K goes into a fresh TMEM accumulator (24 MMAs: 8 K steps x 3
//   terms), and the epilogue warps add the chunk sums into fp32 registers in chunk
//   order. A chunk sum is about sqrt(128 / d) of a logit, so its rounding is that much
//   smaller than that of one accumulator over all of d. Measured at T = 4096, d = 7168,
//   E = 256: gate error 3.7e-7 against float64 (3.0e-7 on the FMA units), 6.3e-7 with
//   256-element chunks, 1.3e-6 with 512; one accumulator over all of d gave 6.8e-6.
//
// Pairs of SMs (cta_group::2, M = 256 tokens): each SM loads its 128 tokens of x and
// half of the tile's N experts' three terms, so the W_g bytes each SM reads per token
// are half of a one-SM tile's. Warp 0 issues the TMA copies into a 3-stage ring of
// 64-element K blocks, one thread of warp 1 of the even CTA issues the pair MMAs into
// two accumulators (chunk c into c % 2), and warps 2-9 fold them: warp w reads TMEM
// lane quarter w % 4 (its 32 tokens) and half (w - 2) / 4 of the N columns. K is split
// into KS slices over the grid; each slice writes its partial logits
// partial[z][t][e] and the top-k kernel adds them in slice order.
//
// Every mbarrier wait is bounded (MOE_DEV_ERR_TIMEOUT in the status word, then the
// kernel drains its copies and MMAs, frees its tensor memory and returns).
#include <cstdlib>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int RT_BK = 64;          // K elements per stage: 128 bytes of bf16 per row
constexpr int RT_STAGES = 3;
constexpr int RT_THREADS = 320;    // warp 0 TMA, warp 1 MMA, warps 2-9 epilogue
constexpr int RT_EPI_WARPS = 8;    // per CTA; 16 arrivals free an accumulator
constexpr int RT_TILE_M = 256;     // tokens per pair

template <int N>
struct RtCfg {
    static constexpr int NH = N / 2;                   // experts each SM loads; columns each epilogue warp folds
    static constexpr int A_BYTES = 128 * RT_BK * 2;    // 16 KB of x
    static constexpr int B_TERM = NH * RT_BK * 2;      // one term's rows
    static constexpr int B_BYTES = 3 * B_TERM;
    static constexpr int STAGE = A_BYTES + B_BYTES;
    static constexpr uint32_t TMEM_COLS = 2 * N;       // two accumulators of N fp32 columns
    static constexpr uint32_t IDESC = idesc_bf16_f32(256, N);
};

struct RtSmem {
    uint64_t full[RT_STAGES];
    uint64_t empty[RT_STAGES];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
};

template <int N>
constexpr size_t rt_smem_bytes() {
    return 1024 + size_t(RT_STAGES) * RtCfg<N>::STAGE + sizeof(RtSmem);
}

// Bounded wait that ignores the abort flag (used only to drain in-flight work).
__device__ __forceinline__ void rt_drain_wait(uint64_t* bar, uint32_t parity) {
    const unsigned long long t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kWaitTimeoutNs) break;
    }
}

// W_g [d, E] fp32 -> three bf16 terms [3][E][d] (K-major rows per expert), through a
// 32 x 32 shared-memory transpose so both sides are coalesced.
__global__ void __launch_bounds__(256) split_router_weights_kernel(const float* __restrict__ Wg, int d, int E,
                                                                   __nv_bfloat16* __restrict__ out) {
    __shared__ float tile[32][33];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const int e0 = blockIdx.x * 32, k0 = blockIdx.y * 32;
#pragma unroll
    for (int r = ty; r < 32; r += 8) {
        const int k = k0 + r, e = e0 + tx;
        tile[r][tx] = (k < d && e < E) ? __ldg(Wg + size_t(k) * E + e) : 0.f;
    }
    __syncthreads();
    const size_t plane = size_t(E) * d;
#pragma unroll
    for (int r = ty; r < 32; r += 8) {
        const int e = e0 + r, k = k0 + tx;
        if (e >= E || k >= d) continue;
        const float w = tile[tx][r];
        const __nv_bfloat16 hi = __float2bfloat16_rn(w);
        const float r1 = w - __bfloat162float(hi);
        const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
        const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
        const size_t o = size_t(e) * d + k;
        out[o] = hi;
        out[plane + o] = mid;
        out[2 * plane + o] = lo;
    }
}

template <int N>
__global__ void __launch_bounds__(RT_THREADS, 1) route_tc_kernel(const __grid_constant__ CUtensorMap mapX,
                                                                 const __grid_constant__ CUtensorMap mapW, int T,
                                                                 int d, int E, int tiles_m, int tiles_n, int k_slice,
                                                                 int kb_per_chunk, float* __restrict__ partial,
                                                                 int32_t* status) {
    using C = RtCfg<N>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* base =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* sA = base;
    unsigned char* sB = base + RT_STAGES * C::A_BYTES;
    RtSmem& S = *reinterpret_cast<RtSmem*>(base + RT_STAGES * C::STAGE);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = int(blockIdx.x >> 1);
    const int mt = pair % tiles_m;
    const int nt = (pair / tiles_m) % tiles_n;
    const int z = pair / (tiles_m * tiles_n);
    const int t0 = mt * RT_TILE_M + int(rank) * 128;  // this SM's tokens
    const int e0 = nt * N + int(rank) * C::NH;         // this SM's experts (B rows)
    const int kbeg = z * k_slice;
    const int kend = min(d, kbeg + k_slice);
    const int nkb = kend > kbeg ? (kend - kbeg + RT_BK - 1) / RT_BK : 0;
    const int nchunks = (nkb + kb_per_chunk - 1) / kb_per_chunk;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < RT_STAGES; ++s) {
            mbar_init(&S.full[s], 1);
            mbar_init(&S.empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&S.tmem_full[a], 1);
            mbar_init(&S.tmem_empty[a], 2 * RT_EPI_WARPS);
        }
        mbar_init(&S.mma_done, 1);
        S.abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
        tma_prefetch_desc(&mapX);
        tma_prefetch_desc(&mapW);
    }
    if (warp == 1) {
        tmem_alloc_pair(&S.tmem_base, C::TMEM_COLS);
        tmem_relinquish_pair();
    }
    __syncwarp();
    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();

    const uint32_t tmem_base = S.tmem_base;
    volatile int* abort_flag = &S.abort_flag;
    const uint32_t full_base = mapa_shared(smem_addr(&S.full[0]), 0);

    if (warp == 0) {
        if (lane == 0) {
            uint32_t armed_mask = 0, armed_par = 0;
            int s = 0;
            uint32_t ph = 0;
            for (int kb = 0; kb < nkb; ++kb) {
                if (!mbar_wait(&S.empty[s], ph ^ 1u, abort_flag, status)) break;
                const int k0 = kbeg + kb * RT_BK;
                const uint32_t bar = full_base + uint32_t(s) * 8u;
                if (leader) mbar_arrive_expect_tx(&S.full[s], 2 * C::STAGE);
                tma_load_2d_pair(sA + s * C::A_BYTES, &mapX, bar, k0, t0);
                tma_load_3d_pair(sB + s * C::B_BYTES, &mapW, bar, k0, e0, 0);  // hi, mid, lo rows
                armed_mask |= 1u << s;
                armed_par = (armed_par & ~(1u << s)) | (ph << s);
                if (++s == RT_STAGES) { s = 0; ph ^= 1u; }
            }
            // Every armed stage must land before the CTA may exit; the even CTA's full
            // barriers also count the odd CTA's bytes, and the final cluster barrier
            // keeps the odd CTA alive until this drain is done.
            if (leader)
                for (int q = 0; q < RT_STAGES; ++q)
                    if (armed_mask & (1u << q)) rt_drain_wait(&S.full[q], (armed_par >> q) & 1u);
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            int s = 0;
            uint32_t ph = 0;
            for (int c = 0; c < nchunks; ++c) {
                const int acc = c & 1;
                const uint32_t aph = (c >> 1) & 1;
                if (!mbar_wait(&S.tmem_empty[acc], aph ^ 1u, abort_flag, status)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + uint32_t(acc * N);
                const int kb_end = min(nkb, (c + 1) * kb_per_chunk);
                bool ok = true;
                for (int kb = c * kb_per_chunk; kb < kb_end; ++kb) {
                    if (!mbar_wait(&S.full[s], ph, abort_flag, status)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_addr = smem_addr(sA + s * C::A_BYTES);
                    const uint32_t b_addr = smem_addr(sB + s * C::B_BYTES);
                    const uint64_t adesc = sw128_kmajor_desc(a_addr);
                    const uint64_t bdesc[3] = {sw128_kmajor_desc(b_addr), sw128_kmajor_desc(b_addr + C::B_TERM),
                                               sw128_kmajor_desc(b_addr + 2 * C::B_TERM)};
                    const bool first_block = kb == c * kb_per_chunk;
#pragma unroll
                    for (int ks = 0; ks < RT_BK / 16; ++ks) {
#pragma unroll
                        for (int term = 0; term < 3; ++term)
                            umma_bf16_pair(d_tmem, adesc + 2 * ks, bdesc[term] + 2 * ks, C::IDESC,
                                           (first_block && ks == 0 && term == 0) ? 0u : 1u);
                    }
                    umma_commit_pair_multicast(&S.empty[s], 0x3);
                    if (++s == RT_STAGES) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                umma_commit_pair_multicast(&S.tmem_full[acc], 0x3);
            }
            umma_commit_pair_multicast(&S.mma_done, 0x1);
            rt_drain_wait(&S.mma_done, 0);
        }
    } else {
        // Epilogue: warp w folds TMEM lanes 32 (w % 4) .. (its 32 tokens) and columns
        // [h NH, (h + 1) NH) of each chunk's accumulator into fp32 registers.
        const int q = warp & 3;
        const int h = (warp - 2) >> 2;
        const uint32_t empty_base = mapa_shared(smem_addr(&S.tmem_empty[0]), 0);
        float run[C::NH];
#pragma unroll
        for (int j = 0; j < C::NH; ++j) run[j] = 0.f;
        bool ok = true;
        for (int c = 0; c < nchunks; ++c) {
            const int acc = c & 1;
            const uint32_t aph = (c >> 1) & 1;
            ok = mbar_wait(&S.tmem_full[acc], aph, abort_flag, status);
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (!ok) break;
            tc_fence_after();
            const uint32_t taddr = tmem_base + (uint32_t(q * 32) << 16) + uint32_t(acc * N + h * C::NH);
#pragma unroll
            for (int j = 0; j < C::NH / 32; ++j) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(taddr + j * 32, v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) run[j * 32 + i] += __uint_as_float(v[i]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(empty_base + uint32_t(acc) * 8u);
        }
        // The pair tile is 256 tokens x N experts: each CTA's accumulator holds its own
        // 128 tokens against all N experts (columns 0..N/2-1 from the even CTA's B rows,
        // the rest from the odd CTA's).
        const int t = t0 + q * 32 + lane;
        if (ok && t < T) {
            float* row = partial + (size_t(z) * T + t) * E;
            const int ec = nt * N + h * C::NH;
            if (ec + C::NH <= E && (E & 3) == 0) {
#pragma unroll
                for (int j = 0; j < C::NH; j += 4)
                    *reinterpret_cast<float4*>(row + ec + j) = make_float4(run[j], run[j + 1], run[j + 2], run[j + 3]);
            } else {
#pragma unroll
                for (int j = 0; j < C::NH; ++j)
                    if (ec + j < E) row[ec + j] = run[j];
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    }
}

// K elements per fresh accumulator (128); MOE_ROUTE_TC_CHUNK (a multiple of 64, read
// once per process) overrides it for accuracy experiments.
int chunk_kblocks() {
    static const int v = [] {
        const char* e = getenv("MOE_ROUTE_TC_CHUNK");
        int c = e ? atoi(e) : 128;
        if (c < RT_BK || c % RT_BK) c = 128;
        return c / RT_BK;
    }();
    return v;
}

template <int N>
cudaError_t launch_n(const CUtensorMap& mX, const CUtensorMap& mW, int T, int d, int E, int tiles_m, int tiles_n,
                     int ks, int slice, float* partial, int32_t* status, cudaStream_t stream) {
    auto kern = route_tc_kernel<N>;
    constexpr size_t smem = rt_smem_bytes<N>();
    static PerContext<int> smem_set;
    const cudaError_t attr_err = set_smem_limit_once(smem_set, kern, smem);
    if (attr_err != cudaSuccess) return attr_err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(2 * tiles_m * tiles_n * ks));
    cfg.blockDim = dim3(RT_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, mX, mW, T, d, E, tiles_m, tiles_n, slice, chunk_kblocks(), partial,
                              status);
}

int tile_n(int E) { return E <= 64 ? 64 : (E <= 128 ? 128 : 256); }

}  // namespace

bool route_uses_tc(int act_dtype, int d, int E) {
    static const int mode = [] {
        const char* e = getenv("MOE_ROUTE_TC");
        return e ? atoi(e) : -1;
    }();
    if (act_dtype != MOE_BF16 || E < 64 || d % 8 != 0 || route_uses_small_kernel(d, E)) return false;
    return mode != 0;
}

size_t route_tc_weight_bytes(int d, int E) { return (size_t(3) * E * d * 2 + 255) & ~size_t(255); }

int route_tc_slices(int T, int d, int E) {
    const int tiles = ((T + RT_TILE_M - 1) / RT_TILE_M) * ((E + tile_n(E) - 1) / tile_n(E));
    const int chunk = chunk_kblocks() * RT_BK;
    const int chunks = (d + chunk - 1) / chunk;
    int ks = (device_sm_count() / 2) / tiles;
    ks = ks < 1 ? 1 : ks;
    ks = ks > chunks ? chunks : ks;
    const int cap = route_max_slices(T, E);
    ks = ks > cap ? cap : ks;
    const int per = (chunks + ks - 1) / ks;  // chunks per slice; no slice left empty
    return (chunks + per - 1) / per;
}

cudaError_t launch_route_tc(const void* x, const float* Wg, int T, int d, int E, float* partial,
                            void* wsplit, int32_t* status, int* ks_out, cudaStream_t stream) {
    __nv_bfloat16* w3 = static_cast<__nv_bfloat16*>(wsplit);
    split_router_weights_kernel<<<dim3(unsigned((E + 31) / 32), unsigned((d + 31) / 32)), 256, 0, stream>>>(Wg, d, E,
                                                                                                           w3);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    const int N = tile_n(E);
    CUtensorMap mX, mW;
    if ((err = make_tensor_map_sw128(&mX, x, 2, uint64_t(d), uint64_t(T), 1, 128, 1)) != cudaSuccess) return err;
    if ((err = make_tensor_map_sw128(&mW, w3, 2, uint64_t(d), uint64_t(E), 3, uint32_t(N / 2), 3)) != cudaSuccess)
        return err;
    const int tiles_m = (T + RT_TILE_M - 1) / RT_TILE_M;
    const int tiles_n = (E + N - 1) / N;
    const int ks = route_tc_slices(T, d, E);
    const int chunk = chunk_kblocks() * RT_BK;
    const int chunks = (d + chunk - 1) / chunk;
    const int slice = ((chunks + ks - 1) / ks) * chunk;
    *ks_out = ks;
    switch (N) {
        case 64: return launch_n<64>(mX, mW, T, d, E, tiles_m, tiles_n, ks, slice, partial, status, stream);
        case 128: return launch_n<128>(mX, mW, T, d, E, tiles_m, tiles_n, ks, slice, partial, status, stream);
        default: return launch_n<256>(mX, mW, T, d, E, tiles_m, tiles_n, ks, slice, partial, status, stream);
    }
}

}  // namespace moe
