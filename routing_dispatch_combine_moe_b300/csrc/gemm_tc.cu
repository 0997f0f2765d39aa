// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05) for bf16
// experts (and, with e4m3 rows and weights, kind::f8f6f4 on the swapped pairs for the
// up projection and optionally the down projection): the only dense contraction of the layer ("EP Math - Expert Parallelism
// (MoE)", "What expert parallelism actually shards": every expert is a complete FFN
// with private weights; the gated three-matrix form is the one in "MoE Expert
// Parallelism Sizing", "Memory residency for the same shape").
//
//   up   : h[r, :]   = act(xperm[r, :] . W13[e]^T)   SwiGLU: silu(g) * u, fused in the epilogue
//   down : out[r, :] = h[r, :] . W2[e]^T
// for every dispatched row r of expert e (rows [offsets[e], offsets[e+1])).
//
// Persistent, warp-specialised kernels, one CTA per SM (192 threads); three variants:
//   grouped_gemm_kernel<PAIR=false>: one SM per 128x256 output tile (tcgen05
//               cta_group::1, M=128).
//   grouped_gemm_kernel<PAIR=true>: clusters of two SMs share a 256x256 tile
//               (cta_group::2, M=256): each SM loads its own 128 rows of A and half of
//               the 256 B rows (the gate half or the up half for SwiGLU), so a stage is
//               32 KB per SM instead of 48 KB and six stages fit; one thread of the
//               even CTA issues the pair MMA, which writes each SM's 128 accumulator
//               rows into its own TMEM.
//   grouped_gemm_swap_kernel: SM pairs with the operands swapped (weights as A,
//               dispatched rows as B, N <= 256 rows per tile); see its own comment.
// gemm_variant() picks one per projection.
// Roles per CTA:
//   warp 0      TMA producer: 128x64 A tile + 256x64 B tile per stage, 128-byte
//               swizzle, 4-stage ring of 48 KB stages guarded by full/empty mbarriers.
//   warp 1      allocates 512 TMEM columns (two 128x256 fp32 accumulators) and one
//               thread issues tcgen05.mma (M=128, N=256, K=16) per 16-wide K slice,
//               committing each stage back to the producer and each finished tile
//               to the epilogue.
//   warps 2-5   epilogue: tcgen05.ld of their 32-lane quarter, activation in fp32,
//               one rounding to bf16, masked stores (rows past the expert's end and
//               columns past N are not written). Double-buffered accumulators let
//               the epilogue of tile i overlap the MMAs of tile i+1.
// The tile list is derived on the device from `offsets` (no host sync): tiles are
// (expert, N tile, M tile) with the M tile fastest, so the CTAs working at the same
// time share one weight tile through L2. An A tile that starts near the end of an
// expert reads the next expert's rows (or zero fill past the buffer); those rows
// are never stored. For SwiGLU the B stage holds 128 gate rows followed by the 128
// matching up rows, so each thread's accumulator row has g and u side by side.
// Every mbarrier wait is bounded; on a timeout the kernel flags MOE_DEV_ERR_TIMEOUT,
// drains its copies and MMAs, frees TMEM and exits.
//
// Output kinds (OUT): the up epilogue stores h in bf16 (kOutBF16) or split into
// hi = bf16(h) and lo = bf16(h - hi) as interleaved 64-column blocks [hi | lo] of a
// [rows, 2F] matrix (kOutHiLo). In the latter case the down projection runs over 2F
// columns of A while the producer loads each 64-wide weight K-block twice (once for
// hi, once for lo), so out = hi.W2 + lo.W2 with exact bf16 products and fp32
// accumulation. The down epilogue stores bf16 (kOutBF16) or fp32 (kOutF32).
#include "common.cuh"
#include "kernels.h"

#include <cstdlib>
#include <mutex>

namespace moe {
namespace {

constexpr int BK = 64, MMA_N = 256;
constexpr int A_STAGE = 128 * BK * 2;  // 16 KB: 128 rows of A per SM
constexpr int TMEM_COLS = 512;
constexpr int kThreads = 192;

enum Mode : int { kSwiGLU = 0, kPlain = 1, kReLU = 2 };
enum Out : int { kOutBF16 = 0, kOutHiLo = 1, kOutF32 = 2 };

template <bool PAIR>
struct Cfg {
    static constexpr int STAGES = PAIR ? 6 : 4;
    static constexpr int B_ROWS = PAIR ? MMA_N / 2 : MMA_N;  // B rows this SM loads per stage
    static constexpr int B_STAGE = B_ROWS * BK * 2;
    static constexpr int STAGE_BYTES = A_STAGE + B_STAGE;     // bytes landing in this SM per stage
    static constexpr int TILE_M = PAIR ? 256 : 128;           // rows of one output tile
    static constexpr uint32_t IDESC = idesc_bf16_f32(TILE_M, MMA_N);
    static constexpr int EPI_WARPS_TOTAL = PAIR ? 8 : 4;      // arrivals that free an accumulator
};

struct Params {
    const int32_t* offsets;  // [E+1]
    const int32_t* counts;   // [E] rows used at the start of each segment, or null (all of it)
    void* C;                 // output, row stride ldc (bf16, or fp32 for a kOutF32 down projection)
    int ldc;                 // elements
    int n_out;               // valid output columns
    int E;
    int K;                   // reduction length of A
    int b_k_shift;           // B's K block = A's K block >> b_k_shift (1 when A holds hi|lo pairs)
    int R;                   // rows per expert in B
    int F;                   // SwiGLU: up rows start at e*R + F
    int n_tiles;             // output column tiles
    int32_t* status;
    int skip_arrive;         // failure-path test: never signal the first finished accumulator
    const float* xscale;     // e4m3 inputs: scale of each row of B (swapped pairs) ...
    const float* wscale;     // ... and of each weight row
    // Swapped pairs, modes without SwiGLU: the split of the last partial wave's tiles
    // over k (null: never split). split_part holds split_slots slots of fp32 partials,
    // split_tickets 2 * split_slots counters that are zero at launch and left zero.
    float* split_part;
    int32_t* split_tickets;
    int split_slots;
};

template <int STAGES>
struct Smem {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
    int off[MOE_MAX_E + 1];
    int end[MOE_MAX_E];  // off[e] + rows of expert e that are computed
    int tile[MOE_MAX_E + 1];
};

template <bool PAIR>
constexpr size_t smem_bytes() {
    return 1024 /*alignment slack*/ + size_t(Cfg<PAIR>::STAGES) * Cfg<PAIR>::STAGE_BYTES +
           sizeof(Smem<Cfg<PAIR>::STAGES>);
}

__device__ __forceinline__ void decode_tile(int t, const int* tile, int E, int n_tiles, int& e, int& mt, int& nt) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tile[mid] * n_tiles <= t) lo = mid; else hi = mid - 1;
    }
    e = lo;
    const int local = t - tile[e] * n_tiles;
    const int mte = tile[e + 1] - tile[e];
    nt = local / mte;
    mt = local - nt * mte;
}

// Bounded wait that ignores the abort flag (used only to drain in-flight work).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
    const unsigned long long t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kWaitTimeoutNs) break;
    }
}

// silu(g) = g / (1 + e^-g) with the fast exponential and division intrinsics: their
// few-ulp fp32 error is far below the bf16 rounding (or the hi/lo split) that h gets.
__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// Stores 32 consecutive bf16 values (packed in pk[16]) at dst, the first n_valid of them.
__device__ __forceinline__ void store_bf16x32(uint16_t* dst, const uint32_t (&pk)[16], int n_valid) {
    if (n_valid >= 32) {
        uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
        for (int j = 0; j < 4; ++j) d4[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (j < n_valid) dst[j] = (j & 1) ? uint16_t(pk[j >> 1] >> 16) : uint16_t(pk[j >> 1] & 0xFFFFu);
    }
}

// Stores 32 activations: one bf16 rounding (kOutBF16), or the hi/lo pair into the
// interleaved [hi | lo] 64-column blocks of a [rows, 2F] matrix (kOutHiLo).
template <int OUT>
__device__ __forceinline__ void store_hidden(uint16_t* row_ptr, int col0, int n_out, const float (&h)[32]) {
    uint32_t hi[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) hi[j] = pack_bf16x2(h[2 * j], h[2 * j + 1]);
    if constexpr (OUT != kOutHiLo) {
        store_bf16x32(row_ptr + col0, hi, n_out - col0);
    } else {
        uint32_t lo[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
            lo[j] = pack_bf16x2(h[2 * j] - bf16_lo(hi[j]), h[2 * j + 1] - bf16_hi(hi[j]));
        const int blk = col0 >> 6, within = col0 & 63;
        store_bf16x32(row_ptr + 128 * blk + within, hi, n_out - col0);
        store_bf16x32(row_ptr + 128 * blk + 64 + within, lo, n_out - col0);
    }
}

// Epilogue of one accumulator tile for the 32 TMEM lanes (= rows) of this warp.
template <int MODE, int OUT>
__device__ __forceinline__ void epilogue_tile(const Params& p, uint32_t tbase, int row, bool row_ok, int nt) {
    if (MODE == kSwiGLU) {
        uint16_t* crow = static_cast<uint16_t*>(p.C) + size_t(row) * p.ldc;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            uint32_t g[32], u[32];
            tmem_ld_32x32b_x32(tbase + c * 32, g);
            tmem_ld_32x32b_x32(tbase + MMA_N / 2 + c * 32, u);
            tmem_ld_wait();
            const int col0 = nt * (MMA_N / 2) + c * 32;
            if (row_ok && col0 < p.n_out) {
                float h[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) h[j] = silu_f(__uint_as_float(g[j])) * __uint_as_float(u[j]);
                store_hidden<OUT>(crow, col0, p.n_out, h);
            }
        }
    } else if (MODE == kReLU) {
        uint16_t* crow = static_cast<uint16_t*>(p.C) + size_t(row) * p.ldc;
#pragma unroll 1
        for (int c = 0; c < MMA_N / 32; ++c) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(tbase + c * 32, v);
            tmem_ld_wait();
            const int col0 = nt * MMA_N + c * 32;
            if (row_ok && col0 < p.n_out) {
                float h[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) h[j] = fmaxf(__uint_as_float(v[j]), 0.f);
                store_hidden<OUT>(crow, col0, p.n_out, h);
            }
        }
    } else {
#pragma unroll 1
        for (int c = 0; c < MMA_N / 32; ++c) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(tbase + c * 32, v);
            tmem_ld_wait();
            const int col0 = nt * MMA_N + c * 32;
            if (row_ok && col0 < p.n_out) {
                if constexpr (OUT == kOutF32) {
                    float* crow = static_cast<float*>(p.C) + size_t(row) * p.ldc + col0;
                    if (col0 + 32 <= p.n_out) {
                        uint4* d4 = reinterpret_cast<uint4*>(crow);
#pragma unroll
                        for (int j = 0; j < 8; ++j) d4[j] = make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (col0 + j < p.n_out) crow[j] = __uint_as_float(v[j]);
                    }
                } else {
                    uint32_t pk[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        pk[j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
                    store_bf16x32(static_cast<uint16_t*>(p.C) + size_t(row) * p.ldc + col0, pk, p.n_out - col0);
                }
            }
        }
    }
}

template <int MODE, int OUT, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_kernel(const __grid_constant__ CUtensorMap mapA,
                                                                   const __grid_constant__ CUtensorMap mapB,
                                                                   const Params p) {
    using C = Cfg<PAIR>;
    constexpr int STAGES = C::STAGES;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* sA = base;
    unsigned char* sB = base + STAGES * A_STAGE;
    Smem<STAGES>& S = *reinterpret_cast<Smem<STAGES>*>(base + STAGES * C::STAGE_BYTES);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = p.E;
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;  // 0 = the CTA that issues the MMAs
    const bool leader = rank == 0;
    const int unit = PAIR ? int(blockIdx.x >> 1) : int(blockIdx.x);
    const int n_units = PAIR ? int(gridDim.x >> 1) : int(gridDim.x);

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&S.full[s], 1);
            mbar_init(&S.empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&S.tmem_full[a], 1);
            mbar_init(&S.tmem_empty[a], C::EPI_WARPS_TOTAL);
        }
        mbar_init(&S.mma_done, 1);
        S.abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
        tma_prefetch_desc(&mapA);
        tma_prefetch_desc(&mapB);
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            tmem_alloc_pair(&S.tmem_base, TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(&S.tmem_base, TMEM_COLS);
            tmem_relinquish();
        }
    }
    if (warp == 2) {
        for (int e0 = 0; e0 <= E; e0 += 32) {
            const int e = e0 + lane;
            if (e <= E) S.off[e] = __ldg(p.offsets + e);
        }
        __syncwarp();
        for (int e0 = 0; e0 < E; e0 += 32) {
            const int e = e0 + lane;
            if (e < E) {
                const int seg = S.off[e + 1] - S.off[e];
                S.end[e] = S.off[e] + (p.counts ? min(max(__ldg(p.counts + e), 0), seg) : seg);
            }
        }
        __syncwarp();
        int run = 0;
        for (int e0 = 0; e0 < E; e0 += 32) {
            const int e = e0 + lane;
            const int v = e < E ? (S.end[e] - S.off[e] + C::TILE_M - 1) / C::TILE_M : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += n;
            }
            if (e < E) S.tile[e] = run + incl - v;
            run += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
        if (lane == 0) S.tile[E] = run;
    }
    __syncwarp();
    tc_fence_before();
    if constexpr (PAIR) cluster_sync_all(); else __syncthreads();
    tc_fence_after();

    const uint32_t tmem_base = S.tmem_base;
    const int total = S.tile[E] * p.n_tiles;
    const int nkb = (p.K + BK - 1) / BK;
    volatile int* abort_flag = &S.abort_flag;
    // Barriers the peer signals live in the even CTA.
    const uint32_t full_base = PAIR ? mapa_shared(smem_addr(&S.full[0]), 0) : smem_addr(&S.full[0]);

    if (warp == 0) {
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            uint32_t armed_mask = 0, armed_par = 0;
            // The dispatched rows of an expert are re-read by every N tile: keep them in L2.
            // Weight tiles are shared by the CTAs running the same N tile at the same time.
            const uint64_t pol_a = l2_policy_evict_last();
            for (int t = unit; t < total; t += n_units) {
                int e, mt, nt;
                decode_tile(t, S.tile, E, p.n_tiles, e, mt, nt);
                const int m0 = S.off[e] + mt * C::TILE_M + int(rank) * 128;
                bool ok = true;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(&S.empty[s], ph ^ 1u, abort_flag, p.status)) { ok = false; break; }
                    const int k0 = kb * BK;
                    const int kB = (kb >> p.b_k_shift) * BK;
                    unsigned char* a_dst = sA + s * A_STAGE;
                    unsigned char* b_dst = sB + s * C::B_STAGE;
                    if constexpr (PAIR) {
                        const uint32_t bar = full_base + uint32_t(s) * 8u;
                        if (leader) mbar_arrive_expect_tx(&S.full[s], 2 * C::STAGE_BYTES);
                        tma_load_2d_pair_hint(a_dst, &mapA, bar, k0, m0, pol_a);
                        int r0;
                        if (MODE == kSwiGLU) r0 = e * p.R + nt * (MMA_N / 2) + (rank ? p.F : 0);
                        else r0 = e * p.R + nt * MMA_N + int(rank) * (MMA_N / 2);
                        tma_load_2d_pair(b_dst, &mapB, bar, kB, r0);
                    } else {
                        mbar_arrive_expect_tx(&S.full[s], C::STAGE_BYTES);
                        tma_load_2d_hint(a_dst, &mapA, &S.full[s], k0, m0, pol_a);
                        if (MODE == kSwiGLU) {
                            const int r0 = e * p.R + nt * (MMA_N / 2);
                            tma_load_2d(b_dst, &mapB, &S.full[s], kB, r0);
                            tma_load_2d(b_dst + C::B_STAGE / 2, &mapB, &S.full[s], kB, r0 + p.F);
                        } else {
                            tma_load_2d(b_dst, &mapB, &S.full[s], kB, e * p.R + nt * MMA_N);
                        }
                    }
                    armed_mask |= 1u << s;
                    armed_par = (armed_par & ~(1u << s)) | (ph << s);
                    if (++s == STAGES) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
            }
            // Every armed stage must land before the CTA may exit. The even CTA's full
            // barriers also count the odd CTA's bytes; the final cluster barrier keeps
            // the odd CTA alive until this drain is done.
            if (leader)
                for (int q = 0; q < STAGES; ++q)
                    if (armed_mask & (1u << q)) drain_wait(&S.full[q], (armed_par >> q) & 1u);
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            int s = 0;
            uint32_t ph = 0;
            int i = 0;
            for (int t = unit; t < total; t += n_units, ++i) {
                const int acc = i & 1;
                const uint32_t aph = (i >> 1) & 1;
                if (!mbar_wait(&S.tmem_empty[acc], aph ^ 1u, abort_flag, p.status)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * MMA_N;
                bool ok = true;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(&S.full[s], ph, abort_flag, p.status)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t adesc = sw128_kmajor_desc(smem_addr(sA + s * A_STAGE));
                    const uint64_t bdesc = sw128_kmajor_desc(smem_addr(sB + s * C::B_STAGE));
#pragma unroll
                    for (int ks = 0; ks < BK / 16; ++ks) {
                        if constexpr (PAIR)
                            umma_bf16_pair(d_tmem, adesc + 2 * ks, bdesc + 2 * ks, C::IDESC, (kb | ks) != 0 ? 1u : 0u);
                        else
                            umma_bf16(d_tmem, adesc + 2 * ks, bdesc + 2 * ks, C::IDESC, (kb | ks) != 0 ? 1u : 0u);
                    }
                    if constexpr (PAIR) umma_commit_pair_multicast(&S.empty[s], 0x3);
                    else umma_commit(&S.empty[s]);
                    if (++s == STAGES) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                if (!(p.skip_arrive && i == 0)) {
                    if constexpr (PAIR) umma_commit_pair_multicast(&S.tmem_full[acc], 0x3);
                    else umma_commit(&S.tmem_full[acc]);
                }
            }
            if constexpr (PAIR) umma_commit_pair_multicast(&S.mma_done, 0x1);
            else umma_commit(&S.mma_done);
            drain_wait(&S.mma_done, 0);
        }
    } else {
        // Epilogue: warps 2..5 own TMEM lane quarters (warp % 4) = rows of this SM's half.
        const int q = warp & 3;
        const int r_in_tile = q * 32 + lane;
        const uint32_t empty_base = PAIR ? mapa_shared(smem_addr(&S.tmem_empty[0]), 0) : 0u;
        int i = 0;
        for (int t = unit; t < total; t += n_units, ++i) {
            int e, mt, nt;
            decode_tile(t, S.tile, E, p.n_tiles, e, mt, nt);
            const int acc = i & 1;
            const uint32_t aph = (i >> 1) & 1;
            bool ok = mbar_wait(&S.tmem_full[acc], aph, abort_flag, p.status);
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (!ok) break;
            tc_fence_after();
            const int row = S.off[e] + mt * C::TILE_M + int(rank) * 128 + r_in_tile;
            const bool row_ok = row < S.end[e];
            const uint32_t tbase = tmem_base + (uint32_t(q * 32) << 16) + acc * MMA_N;
            epilogue_tile<MODE, OUT>(p, tbase, row, row_ok, nt);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (PAIR) mbar_arrive_cluster(empty_base + uint32_t(acc) * 8u);
                else mbar_arrive(&S.tmem_empty[acc]);
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    if constexpr (PAIR) cluster_sync_all(); else __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        if constexpr (PAIR) tmem_dealloc_pair(tmem_base, TMEM_COLS);
        else tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ swapped operands
// SM pairs (cta_group::2, M = 256) with the weights as the MMA's A operand and the
// dispatched rows as B. The 256 rows of a pair tile are output features: each SM
// loads 128 weight rows (SwiGLU: 64 gate rows and the 64 matching up rows). The N
// columns are up to 256 consecutive rows of one expert, N rounded up to a multiple
// of 32 on the expert's last tile, split N/2 + N/2 between the two SMs. An expert's
// row count then costs at most 31 idle columns, where the row-major pair tile costs up
// to 255 idle rows; per stage each SM lands 16 KB of weights and its N/2 rows (at
// most 16 KB; six stages), one copy for each. The
// accumulator holds features on TMEM lanes and rows on columns, so each epilogue
// thread owns one feature and stores it for 32 rows at a time: a warp writes 32
// consecutive features of one row per store. For SwiGLU, warps holding up values
// (lanes 64-127) pass them through shared memory to the warps holding the matching
// gate values (lanes 0-63).
constexpr int SW_STAGES = 6;
constexpr int SW_A_STAGE = 128 * BK * 2;          // 16 KB: 128 weight rows per SM
constexpr int SW_B_BIG = 128 * BK * 2;            // 16 KB: up to 128 dispatched rows per SM
constexpr int SW_STAGE_SMEM = SW_A_STAGE + SW_B_BIG;
constexpr int SW_TILE_N = 256;
constexpr int SW_ROW_MAPS = SW_TILE_N / 32;        // row boxes of 16, 32, ..., 128 rows

// Tensor maps over the dispatched rows, one per box height 16 (i + 1): a tile of N
// rows loads exactly its N / 2 rows per SM with one copy per stage.
struct RowMaps {
    CUtensorMap m[SW_ROW_MAPS];
};

struct SwapXchg {
    float v[2][32][33];     // up values for 32 rows x 32 features, per gate warp
    float sx[SW_TILE_N];    // e4m3 inputs: the scales of the tile's rows (0 past its end)
    int split_last;         // this CTA's k range was the last of its tile to finish
};

constexpr size_t swap_smem_bytes() {
    return 1024 + size_t(SW_STAGES) * SW_STAGE_SMEM + sizeof(Smem<SW_STAGES>) + sizeof(SwapXchg);
}

// Named barrier 1 over the four epilogue warps (128 threads); the second form also
// returns whether `v` holds in every one of them.
__device__ __forceinline__ void epi_bar_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ bool epi_bar_and(bool v) {
    uint32_t r;
    asm volatile(
        "{\n"
        " .reg .pred p, q;\n"
        " setp.ne.u32 p, %1, 0;\n"
        " bar.red.and.pred q, 1, 128, p;\n"
        " selp.u32 %0, 1, 0, q;\n"
        "}\n"
        : "=r"(r)
        : "r"(uint32_t(v))
        : "memory");
    return r != 0;
}

// Token-row tile mt of expert e: first row, rows used, and N. The expert's rows are
// split into ceil(rows / 256) tiles of equal width (rounded up to 32; the last one
// takes what is left), so no tile is a thin remainder: a tile's time is bounded
// below by the load latency of its weight stream whatever its N, and a thin tile
// would pay that for little work. A pair MMA takes N as a multiple of 32 in
// [32, 256] (each SM supplies N/2 rows, a multiple of 16).
__device__ __forceinline__ void swap_tile_rows(const int* off, const int* end, int e, int mt, int& start, int& len,
                                               int& n) {
    const int rows = end[e] - off[e];
    const int tiles = (rows + SW_TILE_N - 1) / SW_TILE_N;
    const int width = ((rows + tiles - 1) / tiles + 31) & ~31;
    start = off[e] + mt * width;
    len = min(width, end[e] - start);
    n = (len + 31) & ~31;
}

// Split of the last partial wave over k. When the tiles leave the last wave of pairs at
// most half busy, each of its `rem` tiles is cut into `parts` consecutive ranges of
// k-blocks that run on pairs which would otherwise idle; every range leaves its fp32
// accumulator in a slot of split_part, and the range that finishes last (an atomic
// ticket per tile and SM, no waiting) sums the slots in range order, so the result does
// not depend on which range finishes last. The work items are the `full` whole tiles,
// then rem * parts ranges, at most one per pair.
constexpr int SW_SPLIT_MAX = 4;         // ranges per tile
constexpr int SW_SPLIT_MIN_KB = 8;      // k-blocks per range at least
constexpr int SW_SPLIT_SLOT = 2 * SW_TILE_N * 128;  // floats per slot: both SMs, 128 features x 256 rows

struct SplitPlan {
    int full, rem, parts;
    __device__ int items() const { return full + rem * parts; }
};

__device__ __forceinline__ SplitPlan plan_split(const Params& p, int total, int n_units, int nkb, bool allowed) {
    SplitPlan sp{total, 0, 1};
    const int r = total % n_units;
    if (!allowed || p.split_part == nullptr || r == 0 || 2 * r > n_units) return sp;
    const int parts = min(min(n_units / r, SW_SPLIT_MAX), min(p.split_slots / r, nkb / SW_SPLIT_MIN_KB));
    if (parts >= 2) sp = SplitPlan{total - r, r, parts};
    return sp;
}

// Work item u: tile t and k-blocks [kb0, kb1); slot = the partial slot of a range (-1 for a
// whole tile), tile r = slot / parts of the split ones, range slot % parts.
struct SwapItem {
    int t, kb0, kb1, slot;
};

__device__ __forceinline__ SwapItem swap_item(int u, const SplitPlan& sp, int nkb) {
    if (u < sp.full) return SwapItem{u, 0, nkb, -1};
    const int j = u - sp.full, part = j % sp.parts;
    return SwapItem{sp.full + j / sp.parts, part * nkb / sp.parts, (part + 1) * nkb / sp.parts, j};
}

template <int OUT>
__device__ __forceinline__ void store_one(const Params& p, int row, int f, float v) {
    if constexpr (OUT == kOutF32) {
        static_cast<float*>(p.C)[size_t(row) * p.ldc + f] = v;
    } else {
        uint16_t* c = static_cast<uint16_t*>(p.C) + size_t(row) * p.ldc;
        const __nv_bfloat16 hi = __float2bfloat16_rn(v);
        if constexpr (OUT == kOutHiLo) {
            const int col = 128 * (f >> 6) + (f & 63);
            c[col] = __bfloat16_as_ushort(hi);
            c[col + 64] = __bfloat16_as_ushort(__float2bfloat16_rn(v - __bfloat162float(hi)));
        } else {
            c[f] = __bfloat16_as_ushort(hi);
        }
    }
}

// F8: weights and rows are e4m3 codes (kind::f8f6f4, 128 K elements per 128-byte stage
// row); the epilogue multiplies each accumulator by its weight row's scale and its
// row's scale, both powers of two, before the activation.
template <int MODE, int OUT, bool F8>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_swap_kernel(const __grid_constant__ CUtensorMap mapW,
                                                                        const __grid_constant__ RowMaps mapX,
                                                                        const Params p) {
    constexpr int STAGES = SW_STAGES;
    constexpr int BKE = F8 ? 128 : BK;  // K elements per stage: 128 bytes of every row
    constexpr int EPI_WARPS_TOTAL = 8;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* sA = base;
    unsigned char* sB = base + STAGES * SW_A_STAGE;
    Smem<STAGES>& S = *reinterpret_cast<Smem<STAGES>*>(base + STAGES * SW_STAGE_SMEM);
    SwapXchg& X = *reinterpret_cast<SwapXchg*>(base + STAGES * SW_STAGE_SMEM + sizeof(Smem<STAGES>));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = p.E;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int unit = int(blockIdx.x >> 1);
    const int n_units = int(gridDim.x >> 1);

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&S.full[s], 1);
            mbar_init(&S.empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&S.tmem_full[a], 1);
            mbar_init(&S.tmem_empty[a], EPI_WARPS_TOTAL);
        }
        mbar_init(&S.mma_done, 1);
        S.abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
        tma_prefetch_desc(&mapW);
        for (int i = 0; i < SW_ROW_MAPS; ++i) tma_prefetch_desc(&mapX.m[i]);
    }
    if (warp == 1) {
        tmem_alloc_pair(&S.tmem_base, TMEM_COLS);
        tmem_relinquish_pair();
    }
    if (warp == 2) {
        for (int e0 = 0; e0 <= E; e0 += 32) {
            const int e = e0 + lane;
            if (e <= E) S.off[e] = __ldg(p.offsets + e);
        }
        __syncwarp();
        for (int e0 = 0; e0 < E; e0 += 32) {
            const int e = e0 + lane;
            if (e < E) {
                const int seg = S.off[e + 1] - S.off[e];
                S.end[e] = S.off[e] + (p.counts ? min(max(__ldg(p.counts + e), 0), seg) : seg);
            }
        }
        __syncwarp();
        int run = 0;
        for (int e0 = 0; e0 < E; e0 += 32) {
            const int e = e0 + lane;
            const int v = e < E ? (S.end[e] - S.off[e] + SW_TILE_N - 1) / SW_TILE_N : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += n;
            }
            if (e < E) S.tile[e] = run + incl - v;
            run += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
        if (lane == 0) S.tile[E] = run;
    }
    __syncwarp();
    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();

    const uint32_t tmem_base = S.tmem_base;
    const int total = S.tile[E] * p.n_tiles;
    const int nkb = (p.K + BKE - 1) / BKE;
    volatile int* abort_flag = &S.abort_flag;
    const uint32_t full_base = mapa_shared(smem_addr(&S.full[0]), 0);
    const SplitPlan sp = plan_split(p, total, n_units, nkb, MODE != kSwiGLU);
    const int n_items = sp.items();

    if (warp == 0) {
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            uint32_t armed_mask = 0, armed_par = 0;
            // An expert's rows are re-read by every feature tile: keep them in L2.
            const uint64_t pol_x = l2_policy_evict_last();
            for (int u = unit; u < n_items; u += n_units) {
                const SwapItem it = swap_item(u, sp, nkb);
                int e, mt, nt, start, len, n;
                decode_tile(it.t, S.tile, E, p.n_tiles, e, mt, nt);
                swap_tile_rows(S.off, S.end, e, mt, start, len, n);
                const CUtensorMap* mx = &mapX.m[(n >> 5) - 1];  // box of n / 2 rows
                const int xrow = start + int(rank) * (n >> 1);
                const uint32_t stage_tx = uint32_t(SW_A_STAGE + (n >> 1) * BK * 2);
                // SwiGLU: feature row wf of the gate and up halves (a 3-D map over [2E, F, d]);
                // otherwise row w0 of [E * R, d]
                const int wf = nt * 128 + int(rank) * 64;
                const int w0 = e * p.R + nt * 256 + int(rank) * 128;
                bool ok = true;
                for (int kb = it.kb0; kb < it.kb1; ++kb) {
                    if (!mbar_wait(&S.empty[s], ph ^ 1u, abort_flag, p.status)) { ok = false; break; }
                    const int kW = (kb >> p.b_k_shift) * BKE;
                    const int kX = kb * BKE;
                    unsigned char* a_dst = sA + s * SW_A_STAGE;
                    unsigned char* b_dst = sB + s * SW_B_BIG;
                    const uint32_t bar = full_base + uint32_t(s) * 8u;
                    if (leader) mbar_arrive_expect_tx(&S.full[s], 2 * stage_tx);
                    if (MODE == kSwiGLU) {
                        // one 3-D box: 64 gate rows of expert e, then the 64 matching up rows
                        tma_load_3d_pair(a_dst, &mapW, bar, kW, wf, 2 * e);
                    } else {
                        tma_load_2d_pair(a_dst, &mapW, bar, kW, w0);
                    }
                    tma_load_2d_pair_hint(b_dst, mx, bar, kX, xrow, pol_x);
                    armed_mask |= 1u << s;
                    armed_par = (armed_par & ~(1u << s)) | (ph << s);
                    if (++s == STAGES) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
            }
            if (leader)
                for (int q = 0; q < STAGES; ++q)
                    if (armed_mask & (1u << q)) drain_wait(&S.full[q], (armed_par >> q) & 1u);
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            int s = 0;
            uint32_t ph = 0;
            int i = 0;
            for (int u = unit; u < n_items; u += n_units, ++i) {
                const SwapItem it = swap_item(u, sp, nkb);
                int e, mt, nt, start, len, n;
                decode_tile(it.t, S.tile, E, p.n_tiles, e, mt, nt);
                swap_tile_rows(S.off, S.end, e, mt, start, len, n);
                const uint32_t idesc = F8 ? idesc_e4m3_f32(256, uint32_t(n)) : idesc_bf16_f32(256, uint32_t(n));
                const int acc = i & 1;
                const uint32_t aph = (i >> 1) & 1;
                if (!mbar_wait(&S.tmem_empty[acc], aph ^ 1u, abort_flag, p.status)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * SW_TILE_N;
                bool ok = true;
                for (int kb = it.kb0; kb < it.kb1; ++kb) {
                    if (!mbar_wait(&S.full[s], ph, abort_flag, p.status)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t adesc = sw128_kmajor_desc(smem_addr(sA + s * SW_A_STAGE));
                    const uint64_t bdesc = sw128_kmajor_desc(smem_addr(sB + s * SW_B_BIG));
                    // four K slices of 32 bytes per 128-byte row (descriptor addresses in 16-byte units)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        const uint32_t accum = (kb != it.kb0 || ks != 0) ? 1u : 0u;
                        if constexpr (F8)
                            umma_f8_pair(d_tmem, adesc + 2 * ks, bdesc + 2 * ks, idesc, accum);
                        else
                            umma_bf16_pair(d_tmem, adesc + 2 * ks, bdesc + 2 * ks, idesc, accum);
                    }
                    umma_commit_pair_multicast(&S.empty[s], 0x3);
                    if (++s == STAGES) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                if (!(p.skip_arrive && i == 0)) umma_commit_pair_multicast(&S.tmem_full[acc], 0x3);
            }
            umma_commit_pair_multicast(&S.mma_done, 0x1);
            drain_wait(&S.mma_done, 0);
        }
    } else {
        // Epilogue: warps 2..5 own TMEM lane quarters q = warp % 4 (features of this SM).
        // Each tile's columns go in chunks of 32: the TMEM load of the next chunk is in
        // flight while the current one is processed, and the accumulator is handed back
        // to the MMA warp as soon as its last chunk is in registers.
        const int q = warp & 3;
        const int te = (warp - 2) * 32 + lane;  // 0..127 over the four epilogue warps
        const int fl = q * 32 + lane;           // this thread's TMEM lane: feature of the SM's 128
        const uint32_t empty_base = mapa_shared(smem_addr(&S.tmem_empty[0]), 0);
        int i = 0;
        for (int u = unit; u < n_items; u += n_units, ++i) {
            const SwapItem it = swap_item(u, sp, nkb);
            int e, mt, nt, start, len, n;
            decode_tile(it.t, S.tile, E, p.n_tiles, e, mt, nt);
            swap_tile_rows(S.off, S.end, e, mt, start, len, n);
            const int acc = i & 1;
            const uint32_t aph = (i >> 1) & 1;
            const int w = q & 1;
            const bool gate_warp = q < 2;
            // feature of this thread's TMEM lane, in [0, n_out) when it is stored
            const int f = MODE == kSwiGLU ? nt * 128 + int(rank) * 64 + w * 32 + lane
                                          : nt * 256 + int(rank) * 128 + q * 32 + lane;
            float wsc = 1.f;
            if constexpr (F8) {
                // e4m3 inputs: the weight row's scale and the tile's row scales, read
                // before the accumulator wait so that their latency hides behind it (the
                // previous tile's last barrier has passed every read of X.sx)
                if (f < p.n_out)
                    wsc = __ldg(p.wscale + size_t(e) * p.R + (MODE == kSwiGLU && !gate_warp ? p.F : 0) + f);
                X.sx[te] = te < len ? __ldg(p.xscale + start + te) : 0.f;
                X.sx[te + 128] = te + 128 < len ? __ldg(p.xscale + start + te + 128) : 0.f;
            }
            bool ok = mbar_wait(&S.tmem_full[acc], aph, abort_flag, p.status);
            ok = __all_sync(0xFFFFFFFFu, ok);
            // All four epilogue warps agree before the shared-memory hand-off (and the
            // row scales) below.
            if (MODE == kSwiGLU || F8) ok = epi_bar_and(ok);
            if (!ok) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + (uint32_t(q * 32) << 16) + acc * SW_TILE_N;
            auto release = [&]() {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(empty_base + uint32_t(acc) * 8u);
            };
            auto chunk = [&](int c0, uint32_t(&v)[32]) {
                if constexpr (MODE != kSwiGLU) {
                    if (it.slot >= 0) {
                        // a k range: its raw fp32 accumulator goes to the range's slot, laid
                        // out [SM][row / 4][feature][row % 4] so that each thread stores
                        // (and the reducer loads) four rows of its feature at once and a warp
                        // covers 512 contiguous bytes
                        float4* dst = reinterpret_cast<float4*>(p.split_part + size_t(it.slot) * SW_SPLIT_SLOT +
                                                                size_t(rank) * (SW_TILE_N * 128)) +
                                      (c0 >> 2) * 128 + fl;
#pragma unroll
                        for (int g = 0; g < 8; ++g)
                            if (c0 + 4 * g < len)
                                __stcg(dst + g * 128, make_float4(__uint_as_float(v[4 * g]), __uint_as_float(v[4 * g + 1]),
                                                                  __uint_as_float(v[4 * g + 2]), __uint_as_float(v[4 * g + 3])));
                        return;
                    }
                }
                if constexpr (F8) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * (wsc * X.sx[c0 + j]));
                }
                if constexpr (MODE == kSwiGLU) {
                    // Warps q and q + 2 hold the gate and up values of the same 32 features;
                    // each hands the other half a chunk through shared memory, so both
                    // compute 16 of the chunk's 32 rows.
                    if (gate_warp) {
#pragma unroll
                        for (int j = 16; j < 32; ++j) X.v[w][j][lane] = __uint_as_float(v[j]);
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j) X.v[w][j][lane] = __uint_as_float(v[j]);
                    }
                    epi_bar_sync();
                    const int j0 = gate_warp ? 0 : 16;
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int j = j0 + jj;
                        const float mine = __uint_as_float(gate_warp ? v[jj] : v[16 + jj]);
                        const float other = X.v[w][j][lane];
                        const float g = gate_warp ? mine : other;
                        const float u = gate_warp ? other : mine;
                        if (c0 + j < len && f < p.n_out) store_one<OUT>(p, start + c0 + j, f, silu_f(g) * u);
                    }
                    epi_bar_sync();
                } else if (f < p.n_out) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if (c0 + j < len) {
                            float x = __uint_as_float(v[j]);
                            if (MODE == kReLU) x = fmaxf(x, 0.f);
                            store_one<OUT>(p, start + c0 + j, f, x);
                        }
                    }
                }
            };
            uint32_t va[32], vb[32];
            tmem_ld_32x32b_x32(tbase, va);
            tmem_ld_wait();
#pragma unroll 1
            for (int c0 = 0; c0 < n; c0 += 64) {
                const bool more1 = c0 + 32 < n;
                if (more1) tmem_ld_32x32b_x32(tbase + c0 + 32, vb);
                else release();
                chunk(c0, va);
                if (!more1) break;
                tmem_ld_wait();
                const bool more2 = c0 + 64 < n;
                if (more2) tmem_ld_32x32b_x32(tbase + c0 + 64, va);
                else release();
                chunk(c0 + 32, vb);
                if (more2) tmem_ld_wait();
            }
            if constexpr (MODE != kSwiGLU) {
                if (it.slot >= 0) {
                    // Ticket of this tile and SM: the range that counts last sums all the
                    // ranges' slots, in range order, and applies the epilogue.
                    const int r = it.slot / sp.parts;
                    __threadfence();
                    epi_bar_sync();
                    if (te == 0) {
                        int32_t* ticket = p.split_tickets + 2 * r + int(rank);
                        __threadfence();
                        const bool last = atomicAdd(ticket, 1) == sp.parts - 1;
                        if (last) *ticket = 0;  // every range has counted: zero for the next launch
                        X.split_last = last;
                    }
                    epi_bar_sync();
                    if (X.split_last) {
                        __threadfence();
                        const float4* src = reinterpret_cast<const float4*>(p.split_part +
                                                                            size_t(r) * sp.parts * SW_SPLIT_SLOT +
                                                                            size_t(rank) * (SW_TILE_N * 128)) +
                                            fl;
                        // 16 rows per step, every range's values for them loaded before any
                        // is added, then summed in range order
                        constexpr int G = 4;  // float4 groups of rows per step
#pragma unroll 1
                        for (int c0 = 0; c0 < len; c0 += 4 * G) {
                            float4 a[SW_SPLIT_MAX][G];
#pragma unroll
                            for (int r2 = 0; r2 < SW_SPLIT_MAX; ++r2)
#pragma unroll
                                for (int g = 0; g < G; ++g)
                                    a[r2][g] = (r2 < sp.parts && c0 + 4 * g < len)
                                                   ? __ldcg(src + r2 * (SW_SPLIT_SLOT / 4) + ((c0 >> 2) + g) * 128)
                                                   : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                            for (int g = 0; g < G; ++g) {
                                float4 sum = a[0][g];
#pragma unroll
                                for (int r2 = 1; r2 < SW_SPLIT_MAX; ++r2) {
                                    if (r2 < sp.parts) {
                                        sum.x += a[r2][g].x;
                                        sum.y += a[r2][g].y;
                                        sum.z += a[r2][g].z;
                                        sum.w += a[r2][g].w;
                                    }
                                }
                                const float s4[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    const int c = c0 + 4 * g + j;
                                    if (c < len && f < p.n_out) {
                                        float x = s4[j];
                                        if constexpr (F8) x *= wsc * X.sx[c];
                                        if (MODE == kReLU) x = fmaxf(x, 0.f);
                                        store_one<OUT>(p, start + c, f, x);
                                    }
                                }
                            }
                        }
                    }
                }
            }
            // plain mode has no barrier inside the chunks: keep X.sx until every warp is done
            if constexpr (F8 && MODE != kSwiGLU) epi_bar_sync();
        }
    }

    __syncwarp();
    tc_fence_before();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host side
// 2-D tensor map over a row-major [rows, inner] matrix of bf16 (or bytes, u8), box =
// 128 bytes x box_rows, 128-byte swizzle, zero fill out of bounds.
cudaError_t make_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows,
                     bool u8 = false) {
    return make_tensor_map_sw128(map, base, u8 ? 1 : 2, inner, rows, 1, box_rows, 1);
}

// 3-D map over SwiGLU weights [E, 2, F, inner] seen as [2E, F, inner]: box = 128 bytes x
// 64 feature rows x both halves (gate, up) of one expert, 128-byte swizzle.
cudaError_t make_gate_up_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t F, uint64_t E, bool u8) {
    return make_tensor_map_sw128(map, base, u8 ? 1 : 2, inner, F, 2 * E, 64, 2);
}

cudaError_t make_row_maps(RowMaps* maps, const void* base, uint64_t inner, uint64_t rows, bool u8 = false) {
    for (int i = 0; i < SW_ROW_MAPS; ++i) {
        const cudaError_t err = make_map(&maps->m[i], base, inner, rows, uint32_t(16 * (i + 1)), u8);
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

template <int MODE, int OUT, bool PAIR>
cudaError_t launch_kernel(const CUtensorMap& mA, const CUtensorMap& mB, const Params& p, int grid,
                          cudaStream_t stream) {
    auto kern = grouped_gemm_kernel<MODE, OUT, PAIR>;
    constexpr size_t smem = smem_bytes<PAIR>();
    static PerContext<int> smem_set;
    const cudaError_t attr_err = set_smem_limit_once(smem_set, kern, smem);
    if (attr_err != cudaSuccess) return attr_err;
    if constexpr (PAIR) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(unsigned(grid));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        // The grid is persistent: never launch more pairs than can be resident at once.
        static PerContext<int> resident;
        int max_clusters = 0;
        resident.get(&max_clusters, [&](int* n) {
            if (cudaOccupancyMaxActiveClusters(n, kern, &cfg) != cudaSuccess || *n <= 0) *n = device_sm_count() / 2;
            return cudaSuccess;
        });
        if (int(cfg.gridDim.x) > 2 * max_clusters) cfg.gridDim.x = unsigned(2 * max_clusters);
        return cudaLaunchKernelEx(&cfg, kern, mA, mB, p);
    } else {
        kern<<<grid, kThreads, smem, stream>>>(mA, mB, p);
        return cudaGetLastError();
    }
}

enum Variant : int { kOneSM = 0, kPairRows = 1, kPairSwap = 2 };

// Which kernel runs a projection; MOE_GEMM_PAIR=0/1/2 forces one (read once per
// process). One SM per 128x256 tile keeps the tensor pipe about 70% busy: each SM
// lands 48 KB per k-block and four stages cover little load latency. SM pairs land
// 32 KB per SM, but a 256-row tile that starts near an expert's end leaves up to
// 255 rows idle; the swapped pair tile (features x rows) leaves at most 31 idle
// columns per expert. Measured on B300 (layer step, bf16): the swapped pairs win
// when experts average 128 rows or more without a capacity (T=2048, d=4096, E=8,
// k=2: 1.167 ms against 1.186 ms; T=4096, d=7168, E=256, k=8: 4.50 ms against
// 4.70 ms); one SM per tile wins for decode-sized batches (128 tokens, 257 experts:
// 3.43 against 3.54 ms) and under a capacity with skewed loads (Zipf 1.2, E=64,
// capacity factor 1.25: 0.315 against 0.327 ms), where most experts hold few rows.
int gemm_variant(int64_t rows_max, int E, int64_t capacity) {
    static int forced = [] {
        const char* v = getenv("MOE_GEMM_PAIR");
        return v ? atoi(v) : -1;
    }();
    if (forced >= 0 && forced <= 2) return forced;
    return (capacity < 0 && rows_max >= int64_t(E) * 128) ? kPairSwap : kOneSM;
}

int grid_for(int64_t rows_max, int E, int n_tiles, bool pair) {
    const int tile_m = pair ? 256 : 128;
    const int64_t upper = ((rows_max + tile_m - 1) / tile_m + E) * int64_t(n_tiles) * (pair ? 2 : 1);
    int sms = device_sm_count();
    if (pair) sms &= ~1;
    int64_t g = upper < sms ? upper : sms;
    if (pair) g = (g + 1) & ~int64_t(1);
    return int(g > 0 ? g : (pair ? 2 : 1));
}

template <int MODE, int OUT, bool F8 = false>
cudaError_t launch_swap(const CUtensorMap& mW, const RowMaps& mX, const Params& p,
                        int64_t rows_max, int E, cudaStream_t stream) {
    auto kern = grouped_gemm_swap_kernel<MODE, OUT, F8>;
    constexpr size_t smem = swap_smem_bytes();
    static PerContext<int> smem_set;
    const cudaError_t attr_err = set_smem_limit_once(smem_set, kern, smem);
    if (attr_err != cudaSuccess) return attr_err;
    const int64_t tiles = ((rows_max + SW_TILE_N - 1) / SW_TILE_N + E) * int64_t(p.n_tiles);
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // Persistent grid: never more pairs than can be resident at once.
    static PerContext<int> resident;
    int max_clusters = 0;
    cfg.gridDim = dim3(2);
    resident.get(&max_clusters, [&](int* n) {
        if (cudaOccupancyMaxActiveClusters(n, kern, &cfg) != cudaSuccess || *n <= 0) *n = device_sm_count() / 2;
        return cudaSuccess;
    });
    const int64_t pairs = tiles < max_clusters ? tiles : max_clusters;
    cfg.gridDim = dim3(unsigned(2 * (pairs > 0 ? pairs : 1)));
    return cudaLaunchKernelEx(&cfg, kern, mW, mX, p);
}

template <int MODE, int OUT>
cudaError_t launch_mode(const CUtensorMap& mA, const CUtensorMap& mB, const Params& p, int64_t rows_max, int E,
                        bool pair, cudaStream_t stream) {
    const int grid = grid_for(rows_max, E, p.n_tiles, pair);
    return pair ? launch_kernel<MODE, OUT, true>(mA, mB, p, grid, stream)
                : launch_kernel<MODE, OUT, false>(mA, mB, p, grid, stream);
}

}  // namespace

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

cudaError_t make_tensor_map_sw128(CUtensorMap* map, const void* base, uint32_t esz, uint64_t inner, uint64_t rows,
                                  uint64_t depth, uint32_t box_rows, uint32_t box_depth) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {inner, rows, depth};
    const cuuint64_t strides[2] = {inner * esz, rows * inner * esz};
    const cuuint32_t box[3] = {128u / esz, box_rows, box_depth};
    const cuuint32_t estr[3] = {1, 1, 1};
    const cuuint32_t rank = depth > 1 || box_depth > 1 ? 3 : 2;
    const CUresult r = enc(map, esz == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank,
                           const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int ffn_tc_variant(int64_t rows, int E, int64_t capacity) { return gemm_variant(rows, E, capacity); }

// MOE_DEBUG_SKIP_ARRIVE=1 (read once per process) makes every grouped-GEMM launch leave
// its first finished accumulator unsignalled: the epilogue's bounded wait then runs out,
// the kernel flags MOE_DEV_ERR_TIMEOUT, drains its copies and MMAs, frees TMEM and
// returns. It exists to test that failure path; nothing else sets it.
int debug_skip_arrive() {
    static const int v = [] {
        const char* e = getenv("MOE_DEBUG_SKIP_ARRIVE");
        return e && atoi(e) != 0 ? 1 : 0;
    }();
    return v;
}

// MOE_GEMM_SPLITK=0 (read once per process) turns the split of the last partial wave
// over k off, for comparisons; it is on otherwise.
bool gemm_splitk_enabled() {
    static const bool v = [] {
        const char* e = getenv("MOE_GEMM_SPLITK");
        return !(e && atoi(e) == 0);
    }();
    return v;
}

cudaError_t launch_ffn_tc(const FfnArgs& a, cudaStream_t stream, cudaEvent_t mid_event) {
    const int64_t rows_max = a.rows;
    const bool split_h = a.precision == MOE_PRECISION_SPLIT_H;
    const bool f32_out = a.precision != MOE_PRECISION_BF16;
    const int variant = gemm_variant(rows_max, a.E, a.capacity);
    const bool pair = variant == kPairRows;
    const bool swap = variant == kPairSwap;
    const uint32_t b_rows = pair ? MMA_N / 2 : MMA_N;  // rows of one B box
    CUtensorMap mA, mB;
    RowMaps mX;
    cudaError_t err;
    Params p{};
    p.offsets = a.offsets;
    p.counts = a.counts;
    p.E = a.E;
    p.status = a.status;
    p.F = a.F;
    p.skip_arrive = debug_skip_arrive();
    if (a.split_part && a.split_tickets && a.split_slots > 0 && gemm_splitk_enabled()) {
        p.split_part = a.split_part;
        p.split_tickets = a.split_tickets;
        p.split_slots = a.split_slots;
    }

    // Up projection: A = xperm [rows, d]; B = W13 [E*R, d]; C = h.
    const bool swiglu = a.expert_kind == MOE_EXPERT_SWIGLU;
    const int R = swiglu ? 2 * a.F : a.F;
    p.C = a.h;
    p.ldc = split_h ? 2 * a.F : a.F;
    p.n_out = a.F;
    p.K = a.d;
    p.b_k_shift = 0;
    p.R = R;
    if (a.in_fp8) {
        // e4m3 rows and weights: always the swapped pairs
        p.xscale = a.xscale;
        p.wscale = a.w13_scale;
        err = swiglu ? make_gate_up_map(&mA, a.W13, a.d, a.F, a.E, true)
                     : make_map(&mA, a.W13, a.d, uint64_t(a.E) * R, 128, true);
        if (err != cudaSuccess) return err;
        if ((err = make_row_maps(&mX, a.xperm, a.d, rows_max, true)) != cudaSuccess) return err;
        p.n_tiles = swiglu ? (a.F + 127) / 128 : (a.F + 255) / 256;
        if (swiglu)
            err = split_h ? launch_swap<kSwiGLU, kOutHiLo, true>(mA, mX, p, rows_max, a.E, stream)
                          : launch_swap<kSwiGLU, kOutBF16, true>(mA, mX, p, rows_max, a.E, stream);
        else
            err = split_h ? launch_swap<kReLU, kOutHiLo, true>(mA, mX, p, rows_max, a.E, stream)
                          : launch_swap<kReLU, kOutBF16, true>(mA, mX, p, rows_max, a.E, stream);
        p.xscale = p.wscale = nullptr;
    } else if (swap) {
        // weights as the MMA's A operand: a 3-D box of 64 gate + 64 up rows, or 128-row boxes
        err = swiglu ? make_gate_up_map(&mA, a.W13, a.d, a.F, a.E, false)
                     : make_map(&mA, a.W13, a.d, uint64_t(a.E) * R, 128);
        if (err != cudaSuccess) return err;
        if ((err = make_row_maps(&mX, a.xperm, a.d, rows_max)) != cudaSuccess) return err;
        p.n_tiles = swiglu ? (a.F + 127) / 128 : (a.F + 255) / 256;
        if (swiglu)
            err = split_h ? launch_swap<kSwiGLU, kOutHiLo>(mA, mX, p, rows_max, a.E, stream)
                          : launch_swap<kSwiGLU, kOutBF16>(mA, mX, p, rows_max, a.E, stream);
        else
            err = split_h ? launch_swap<kReLU, kOutHiLo>(mA, mX, p, rows_max, a.E, stream)
                          : launch_swap<kReLU, kOutBF16>(mA, mX, p, rows_max, a.E, stream);
    } else {
        if ((err = make_map(&mA, a.xperm, a.d, rows_max, 128)) != cudaSuccess) return err;
        if ((err = make_map(&mB, a.W13, a.d, uint64_t(a.E) * R, swiglu ? MMA_N / 2 : b_rows)) != cudaSuccess)
            return err;
        p.n_tiles = swiglu ? (a.F + MMA_N / 2 - 1) / (MMA_N / 2) : (a.F + MMA_N - 1) / MMA_N;
        if (swiglu)
            err = split_h ? launch_mode<kSwiGLU, kOutHiLo>(mA, mB, p, rows_max, a.E, pair, stream)
                          : launch_mode<kSwiGLU, kOutBF16>(mA, mB, p, rows_max, a.E, pair, stream);
        else
            err = split_h ? launch_mode<kReLU, kOutHiLo>(mA, mB, p, rows_max, a.E, pair, stream)
                          : launch_mode<kReLU, kOutBF16>(mA, mB, p, rows_max, a.E, pair, stream);
    }
    if (err != cudaSuccess) return err;
    if (mid_event) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if ((err = cudaStreamIsCapturing(stream, &cs)) != cudaSuccess) return err;
        err = cs == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(mid_event, stream, cudaEventRecordExternal)
                                                  : cudaEventRecord(mid_event, stream);
        if (err != cudaSuccess) return err;
    }

    // Down projection: A = h [rows, F] (split: [rows, 2F] hi|lo blocks); B = W2 [E*d, F].
    const int kA = split_h ? 2 * a.F : a.F;
    p.C = a.out;
    p.ldc = a.d;
    p.n_out = a.d;
    p.K = kA;
    p.b_k_shift = split_h ? 1 : 0;
    p.R = a.d;
    p.n_tiles = (a.d + MMA_N - 1) / MMA_N;
    if (a.h_fp8) {
        // h quantized per row (its bf16 value, as stored) into e4m3 codes + row scales,
        // then the down projection on e4m3 against e4m3 W2: always the swapped pairs
        if ((err = launch_quantize_rows_fp8(a.h, rows_max, a.F, a.hq, a.hscale, stream)) != cudaSuccess) return err;
        p.xscale = a.hscale;
        p.wscale = a.w2_scale;
        if ((err = make_map(&mA, a.W2, a.F, uint64_t(a.E) * a.d, 128, true)) != cudaSuccess) return err;
        if ((err = make_row_maps(&mX, a.hq, a.F, rows_max, true)) != cudaSuccess) return err;
        return launch_swap<kPlain, kOutF32, true>(mA, mX, p, rows_max, a.E, stream);
    }
    if (swap) {
        if ((err = make_map(&mA, a.W2, a.F, uint64_t(a.E) * a.d, 128)) != cudaSuccess) return err;
        if ((err = make_row_maps(&mX, a.h, kA, rows_max)) != cudaSuccess) return err;
        return f32_out ? launch_swap<kPlain, kOutF32>(mA, mX, p, rows_max, a.E, stream)
                       : launch_swap<kPlain, kOutBF16>(mA, mX, p, rows_max, a.E, stream);
    }
    if ((err = make_map(&mA, a.h, kA, rows_max, 128)) != cudaSuccess) return err;
    if ((err = make_map(&mB, a.W2, a.F, uint64_t(a.E) * a.d, b_rows)) != cudaSuccess) return err;
    return f32_out ? launch_mode<kPlain, kOutF32>(mA, mB, p, rows_max, a.E, pair, stream)
                   : launch_mode<kPlain, kOutBF16>(mA, mB, p, rows_max, a.E, pair, stream);
}

}  // namespace moe
