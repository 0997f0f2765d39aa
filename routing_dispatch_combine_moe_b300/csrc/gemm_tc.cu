// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05) for bf16
// experts: the only dense contraction of the layer ("EP Math - Expert Parallelism
// (MoE)", "What expert parallelism actually shards": each expert is a full FFN with
// its own weights; the gated three-matrix form is the one in "MoE Expert
// Parallelism Sizing", "Memory residency for the same shape").
//
//   up   : h[r, :]   = act(xperm[r, :] . W13[e]^T)   SwiGLU: silu(g) * u, fused in the epilogue
//   down : out[r, :] = h[r, :] . W2[e]^T
// for every dispatched row r of expert e (rows [offsets[e], offsets[e+1])).
//
// Persistent, warp-specialised kernel, one CTA per SM (192 threads):
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
#include "common.cuh"
#include "kernels.h"

#include <mutex>

namespace moe {
namespace {

constexpr int BM = 128, BK = 64, MMA_N = 256, STAGES = 4;
constexpr int A_STAGE = BM * BK * 2;     // 16 KB
constexpr int B_STAGE = MMA_N * BK * 2;  // 32 KB
constexpr int STAGE_BYTES = A_STAGE + B_STAGE;
constexpr int TMEM_COLS = 512;
constexpr int kThreads = 192;
constexpr uint32_t IDESC = idesc_bf16_f32(BM, MMA_N);

enum Mode : int { kSwiGLU = 0, kPlain = 1, kReLU = 2 };

struct Params {
    const int32_t* offsets;  // [E+1]
    __nv_bfloat16* C;        // output, row stride ldc
    int ldc;                 // elements
    int n_out;               // valid output columns
    int E;
    int K;                   // reduction length
    int R;                   // rows per expert in B
    int F;                   // SwiGLU: up rows start at e*R + F
    int n_tiles;             // output column tiles
    int32_t* status;
};

struct Smem {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
    int off[MOE_MAX_E + 1];
    int tile[MOE_MAX_E + 1];
};

constexpr size_t kSmemBytes = 1024 /*alignment slack*/ + size_t(STAGES) * STAGE_BYTES + sizeof(Smem);

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

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + __expf(-g)); }

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_kernel(const __grid_constant__ CUtensorMap mapA,
                                                                   const __grid_constant__ CUtensorMap mapB,
                                                                   const Params p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* sA = base;
    unsigned char* sB = base + STAGES * A_STAGE;
    Smem& S = *reinterpret_cast<Smem*>(base + STAGES * STAGE_BYTES);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = p.E;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&S.full[s], 1);
            mbar_init(&S.empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&S.tmem_full[a], 1);
            mbar_init(&S.tmem_empty[a], 4);
        }
        mbar_init(&S.mma_done, 1);
        S.abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
        tma_prefetch_desc(&mapA);
        tma_prefetch_desc(&mapB);
    }
    if (warp == 1) {
        tmem_alloc(&S.tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 2) {
        for (int e0 = 0; e0 <= E; e0 += 32) {
            const int e = e0 + lane;
            if (e <= E) S.off[e] = __ldg(p.offsets + e);
        }
        __syncwarp();
        int run = 0;
        for (int e0 = 0; e0 < E; e0 += 32) {
            const int e = e0 + lane;
            const int v = e < E ? (S.off[e + 1] - S.off[e] + BM - 1) / BM : 0;
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
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem_base = S.tmem_base;
    const int total = S.tile[E] * p.n_tiles;
    const int nkb = (p.K + BK - 1) / BK;
    volatile int* abort_flag = &S.abort_flag;

    if (warp == 0) {
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            uint32_t armed_mask = 0, armed_par = 0;
            // The dispatched rows of an expert are re-read by every N tile: keep them in L2.
            // Weight tiles are shared by the CTAs running the same N tile at the same time.
            const uint64_t pol_a = l2_policy_evict_last();
            for (int t = blockIdx.x; t < total; t += gridDim.x) {
                int e, mt, nt;
                decode_tile(t, S.tile, E, p.n_tiles, e, mt, nt);
                const int m0 = S.off[e] + mt * BM;
                bool ok = true;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(&S.empty[s], ph ^ 1u, abort_flag, p.status)) { ok = false; break; }
                    mbar_arrive_expect_tx(&S.full[s], STAGE_BYTES);
                    const int k0 = kb * BK;
                    tma_load_2d_hint(sA + s * A_STAGE, &mapA, &S.full[s], k0, m0, pol_a);
                    if (MODE == kSwiGLU) {
                        const int r0 = e * p.R + nt * (MMA_N / 2);
                        tma_load_2d(sB + s * B_STAGE, &mapB, &S.full[s], k0, r0);
                        tma_load_2d(sB + s * B_STAGE + B_STAGE / 2, &mapB, &S.full[s], k0, r0 + p.F);
                    } else {
                        tma_load_2d(sB + s * B_STAGE, &mapB, &S.full[s], k0, e * p.R + nt * MMA_N);
                    }
                    armed_mask |= 1u << s;
                    armed_par = (armed_par & ~(1u << s)) | (ph << s);
                    if (++s == STAGES) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
            }
            // Every armed stage must land before the CTA may exit.
            for (int q = 0; q < STAGES; ++q)
                if (armed_mask & (1u << q)) drain_wait(&S.full[q], (armed_par >> q) & 1u);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int i = 0;
            for (int t = blockIdx.x; t < total; t += gridDim.x, ++i) {
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
                    const uint64_t bdesc = sw128_kmajor_desc(smem_addr(sB + s * B_STAGE));
#pragma unroll
                    for (int ks = 0; ks < BK / 16; ++ks)
                        umma_bf16(d_tmem, adesc + 2 * ks, bdesc + 2 * ks, IDESC, (kb | ks) != 0 ? 1u : 0u);
                    umma_commit(&S.empty[s]);
                    if (++s == STAGES) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                umma_commit(&S.tmem_full[acc]);
            }
            umma_commit(&S.mma_done);
            drain_wait(&S.mma_done, 0);
        }
    } else {
        // Epilogue: warps 2..5 own TMEM lane quarters (warp % 4).
        const int q = warp & 3;
        const int r_in_tile = q * 32 + lane;
        int i = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++i) {
            int e, mt, nt;
            decode_tile(t, S.tile, E, p.n_tiles, e, mt, nt);
            const int acc = i & 1;
            const uint32_t aph = (i >> 1) & 1;
            bool ok = mbar_wait(&S.tmem_full[acc], aph, abort_flag, p.status);
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (!ok) break;
            tc_fence_after();
            const int row = S.off[e] + mt * BM + r_in_tile;
            const bool row_ok = row < S.off[e + 1];
            const uint32_t tbase = tmem_base + (uint32_t(q * 32) << 16) + acc * MMA_N;
            __nv_bfloat16* crow = p.C + size_t(row) * p.ldc;
            if (MODE == kSwiGLU) {
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t g[32], u[32];
                    tmem_ld_32x32b_x32(tbase + c * 32, g);
                    tmem_ld_32x32b_x32(tbase + MMA_N / 2 + c * 32, u);
                    tmem_ld_wait();
                    const int col0 = nt * (MMA_N / 2) + c * 32;
                    if (row_ok) {
                        uint32_t pk[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const float h0 = silu_f(__uint_as_float(g[2 * j])) * __uint_as_float(u[2 * j]);
                            const float h1 = silu_f(__uint_as_float(g[2 * j + 1])) * __uint_as_float(u[2 * j + 1]);
                            pk[j] = pack_bf16x2(h0, h1);
                        }
                        if (col0 + 32 <= p.n_out) {
                            uint4* dst = reinterpret_cast<uint4*>(crow + col0);
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                        } else {
                            for (int j = 0; j < 32 && col0 + j < p.n_out; ++j) {
                                const uint16_t b = (j & 1) ? uint16_t(pk[j >> 1] >> 16) : uint16_t(pk[j >> 1] & 0xFFFFu);
                                reinterpret_cast<uint16_t*>(crow)[col0 + j] = b;
                            }
                        }
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
                        uint32_t pk[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            float a0 = __uint_as_float(v[2 * j]), a1 = __uint_as_float(v[2 * j + 1]);
                            if (MODE == kReLU) { a0 = fmaxf(a0, 0.f); a1 = fmaxf(a1, 0.f); }
                            pk[j] = pack_bf16x2(a0, a1);
                        }
                        if (col0 + 32 <= p.n_out) {
                            uint4* dst = reinterpret_cast<uint4*>(crow + col0);
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                        } else {
                            for (int j = 0; j < 32 && col0 + j < p.n_out; ++j) {
                                const uint16_t b = (j & 1) ? uint16_t(pk[j >> 1] >> 16) : uint16_t(pk[j >> 1] & 0xFFFFu);
                                reinterpret_cast<uint16_t*>(crow)[col0 + j] = b;
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.tmem_empty[acc]);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host side
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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

// 2-D bf16 tensor map over a row-major [rows, inner] matrix, box = 64 x box_rows,
// 128-byte swizzle, zero fill out of bounds.
cudaError_t make_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {inner * 2};
    const cuuint32_t box[2] = {uint32_t(BK), box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int MODE>
cudaError_t launch_mode(const CUtensorMap& mA, const CUtensorMap& mB, const Params& p, int grid,
                        cudaStream_t stream) {
    auto kern = grouped_gemm_kernel<MODE>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemBytes));
    });
    if (attr_err != cudaSuccess) return attr_err;
    kern<<<grid, kThreads, kSmemBytes, stream>>>(mA, mB, p);
    return cudaGetLastError();
}

int grid_for(int64_t rows_max, int E, int n_tiles) {
    const int64_t upper = ((rows_max + BM - 1) / BM + E) * int64_t(n_tiles);
    const int sms = device_sm_count();
    return int(upper < sms ? (upper > 0 ? upper : 1) : sms);
}

}  // namespace

cudaError_t launch_ffn_tc(const FfnArgs& a, cudaStream_t stream, cudaEvent_t mid_event) {
    const int64_t rows_max = int64_t(a.T) * a.k;
    CUtensorMap mA, mB;
    cudaError_t err;
    Params p{};
    p.offsets = a.offsets;
    p.E = a.E;
    p.status = a.status;
    p.F = a.F;

    // Up projection: A = xperm [rows, d]; B = W13 [E*R, d].
    const bool swiglu = a.expert_kind == MOE_EXPERT_SWIGLU;
    const int R = swiglu ? 2 * a.F : a.F;
    if ((err = make_map(&mA, a.xperm, a.d, rows_max, BM)) != cudaSuccess) return err;
    if ((err = make_map(&mB, a.W13, a.d, uint64_t(a.E) * R, swiglu ? MMA_N / 2 : MMA_N)) != cudaSuccess) return err;
    p.C = static_cast<__nv_bfloat16*>(a.h);
    p.ldc = a.F;
    p.n_out = a.F;
    p.K = a.d;
    p.R = R;
    p.n_tiles = swiglu ? (a.F + MMA_N / 2 - 1) / (MMA_N / 2) : (a.F + MMA_N - 1) / MMA_N;
    err = swiglu ? launch_mode<kSwiGLU>(mA, mB, p, grid_for(rows_max, a.E, p.n_tiles), stream)
                 : launch_mode<kReLU>(mA, mB, p, grid_for(rows_max, a.E, p.n_tiles), stream);
    if (err != cudaSuccess) return err;
    if (mid_event && (err = cudaEventRecord(mid_event, stream)) != cudaSuccess) return err;

    // Down projection: A = h [rows, F]; B = W2 [E*d, F].
    if ((err = make_map(&mA, a.h, a.F, rows_max, BM)) != cudaSuccess) return err;
    if ((err = make_map(&mB, a.W2, a.F, uint64_t(a.E) * a.d, MMA_N)) != cudaSuccess) return err;
    p.C = static_cast<__nv_bfloat16*>(a.out);
    p.ldc = a.d;
    p.n_out = a.d;
    p.K = a.F;
    p.R = a.d;
    p.n_tiles = (a.d + MMA_N - 1) / MMA_N;
    return launch_mode<kPlain>(mA, mB, p, grid_for(rows_max, a.E, p.n_tiles), stream);
}

}  // namespace moe
