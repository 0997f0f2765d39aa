// Launchers of the CUDA kernels (host side). Each enqueues on `stream` and returns
// the launch's cudaError_t; argument checks happen in the C ABI layer before these.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

namespace moe {

// Assignments per dispatch block: the histogram, scan and scatter kernels all cut
// the T*k assignments into blocks of this many, in assignment order.
constexpr int kDispatchBlock = 256;
// Rows per tensor-core tile; the scan also emits per-expert tile offsets at this size.
constexpr int kTileM = 128;

inline int dispatch_blocks(int64_t assignments) {
    return int((assignments + kDispatchBlock - 1) / kDispatchBlock);
}

// Router. The logits are summed from up to route_max_slices(T, E) split-K partials
// held in `scratch`; the tensor-core router also keeps W_g's three bf16 terms there.
int route_max_slices(int T, int E);
bool route_uses_small_kernel(int d, int E);  // one fused launch instead of logits + top-k
int route_k_slices(int T, int d, int E);
// Logits on the tensor cores (bf16 x, E >= 64, not the small-E kernel; MOE_ROUTE_TC=0
// keeps them on the FMA units).
bool route_uses_tc(int act_dtype, int d, int E);
size_t route_tc_weight_bytes(int d, int E);  // [3][E][d] bf16, 256-byte rounded
int route_tc_slices(int T, int d, int E);
inline size_t route_partial_bytes_max(int T, int E) {
    return (size_t(route_max_slices(T, E)) * size_t(T) * size_t(E) * sizeof(float) + 255) & ~size_t(255);
}
inline size_t route_scratch_bytes(int act_dtype, int T, int d, int E) {
    return route_partial_bytes_max(T, E) + (route_uses_tc(act_dtype, d, E) ? route_tc_weight_bytes(d, E) : 0);
}
// Splits W_g into its three bf16 terms in `wsplit`, then writes ks_out split-K partial
// logits [ks][T][E] into `partial` from the tensor cores.
cudaError_t launch_route_tc(const void* x, const float* Wg, int T, int d, int E, float* partial, void* wsplit,
                            int32_t* status, int* ks_out, cudaStream_t stream);
// topk_idx / topk_gate have k + n_shared slots per token; the shared slots hold
// experts E..E+n_shared-1 with gate 1. With 0 < topk_groups < n_groups the selection
// is limited to the topk_groups best of n_groups contiguous expert groups. A non-null
// hist (zeroed, [(E + n_shared) * dispatch_blocks(T * (k + n_shared))]) receives the
// dispatch's per-block expert counts, so the dispatch can skip its count kernel. A
// non-null near_ties (one zeroed int) receives the number of tokens whose k-th and
// (k+1)-th largest selectable fp32 logits differ by less than 1e-6 relative.
// `status` (nullable) receives MOE_DEV_ERR_TIMEOUT from the tensor-core router's bounded waits.
cudaError_t launch_route(int act_dtype, const void* x, const float* Wg, const float* bias, int T, int d, int E,
                         int k, int n_shared, int n_groups, int topk_groups, int32_t* topk_idx, float* topk_gate,
                         float* scratch, int32_t* hist, int32_t* near_ties, int32_t* status, cudaStream_t stream);

struct DispatchArgs {
    int T, d, E, k, D;  // E: all experts (routed + shared), k: all slots per token
    int E_capped;       // experts [0, E_capped) are routed: held to the capacity, split over D ranks
    int64_t capacity;  // < 0: dropless
    int drop_policy;   // MOE_DROP_*
    int layout;        // MOE_LAYOUT_*
    int act_bytes;
    const float* topk_gate;  // [T*k], read by the gate drop policy
    const void* x;
    const int32_t* topk_idx;
    int32_t* counts_routed;
    int32_t* counts_kept;
    int32_t* offsets;
    int32_t* rank_offsets;
    int32_t* pos;
    int32_t* row_src;
    int32_t* drop_list;
    int32_t* n_dropped;
    void* xperm;
    // workspace pieces
    int32_t* status;
    int32_t* hist;         // [E * nblk]
    int32_t* drop_offsets; // [E]
    int32_t* routed_offsets; // [E+1] exclusive scan of the routed counts (gate policy)
    int32_t* elist;          // [2*T*k] each expert's assignments in token order, then their gate keys (gate policy)
    int32_t* scan_ticket;    // one int, 0 on entry (left at 0): orders the scan's CTAs when E > 32
    bool skip_gather;        // leave xperm to launch_dedup
    bool counted;            // hist already holds the counts (the router filled it)
};

cudaError_t launch_dispatch(const DispatchArgs& a, cudaStream_t stream);

// Deduplicated send buffer and the receiving side's fan-out into xperm.
struct DedupArgs {
    int T, d, K, E_routed, D;  // K: slots per token; experts [0, E_routed) split over D ranks
    int act_bytes;
    int64_t rows;              // rows of xperm
    const void* x;
    const int32_t* topk_idx;   // [T*K]
    const int32_t* pos;        // [T*K] from launch_dispatch
    int32_t* send_counts;      // [D]
    int32_t* send_offsets;     // [D+1]
    int32_t* send_pos;         // [T*D]
    int32_t* send_src;         // [T*D]
    void* xsend;               // [T*D, d] act, or (fp8) its e4m3 codes [T*D, d] uint8
    float* xsend_scale;        // fp8: [T*D, ceil(d/128)] block scales of the send rows; fp8_rows: [T*D]
    bool fp8;                  // send rows as e4m3 + per-128 block scales; the fan-out dequantizes
    bool fp8_rows;             // send rows as e4m3 + one scale per row; the fan-out copies codes + scale
    uint8_t* xq;               // fp8_rows: [rows, d] the expert rows' codes (the FP8 GEMM's input) ...
    float* xscale;             // ... and their row scales [rows]
    void* xperm;
    int32_t* status;
    // scratch
    int32_t* slots;            // [T*D]
    int32_t* hist;             // [D * ceil(T*D / 256)]
    int32_t* kept_scratch;     // [D]
    int32_t* drop_offsets;     // [D]
    int32_t* routed_offsets;   // [D+1]
    int32_t* rank_offsets;     // [2]
    int32_t* n_dropped;        // [1]
};

cudaError_t launch_dedup(const DedupArgs& a, cudaStream_t stream);

// FP8 dispatch: e4m3 rows with power-of-two per-128 block scales for the kept routed
// assignments (shared experts' rows copied from x into xperm), then, with `dequant`,
// the receiving side's bf16 rows in xperm.
struct Fp8Args {
    int T, d, K, E_routed, n_experts;  // K: slots per token; n_experts: routed + shared
    int64_t rows;                      // rows of xq / xscale / xperm
    const void* x;
    const int32_t* topk_idx;
    const int32_t* pos;
    const int32_t* row_src;
    const int32_t* offsets;            // [n_experts + 1]; rows [0, offsets[n_experts]) are dispatched
    uint8_t* xq;                       // [rows, d]
    float* xscale;                     // [rows, ceil(d / 128)], or [rows] with per_row
    void* xperm;
    bool dequant;
    bool per_row;                      // one scale per row, codes to every kept row (the FP8 GEMM input)
    int32_t* status;
};

cudaError_t launch_fp8_dispatch(const Fp8Args& a, cudaStream_t stream);
// The deduplicated dispatch's FP8 legs: x rows quantized once per (token, rank) slot into
// the send buffer (slots[t*D + r] = r or -1, send_pos from the send-map scatter), and the
// receiving side's fan-out: each kept routed assignment's row dequantized from its send
// row into xperm (exactly q * 2^s), shared experts' rows copied from x.
cudaError_t launch_fp8_send(const void* x, const int32_t* slots, const int32_t* send_pos, int T, int D, int d,
                            int64_t max_send, uint8_t* xq, float* xscale, int32_t* status, cudaStream_t stream);
cudaError_t launch_fp8_fanout(const void* x, const uint8_t* xq, const float* xscale, const int32_t* topk_idx,
                              const int32_t* pos, const int32_t* send_pos, void* xperm, int T, int K, int E_routed,
                              int D, int d, int64_t max_rows, int64_t max_send, int32_t* status,
                              cudaStream_t stream);
// The same two legs in the FP8 GEMM's format: each send row quantized by the row rule
// (codes [T*D, d], one scale per send row), and the fan-out copying each kept routed
// assignment's codes and scale into xq [rows, d] / xscale [rows]; shared experts' rows are
// x[t] quantized by the same rule.
cudaError_t launch_fp8_send_rows(const void* x, const int32_t* send_pos, int T, int D, int d, int64_t max_send,
                                 uint8_t* sq, float* sscale, int32_t* status, cudaStream_t stream);
cudaError_t launch_fp8_row_fanout(const void* x, const uint8_t* sq, const float* sscale, const int32_t* topk_idx,
                                  const int32_t* pos, const int32_t* send_pos, uint8_t* xq, float* xscale, int T,
                                  int K, int E_routed, int D, int d, int64_t max_rows, int64_t max_send,
                                  int32_t* status, cudaStream_t stream);
// Row-scaled e4m3 codes [n_rows, d] and scales [n_rows] of a bf16 matrix [n_rows, d].
cudaError_t launch_quantize_rows_fp8(const void* w, int64_t n_rows, int d, uint8_t* q, float* scale,
                                     cudaStream_t stream);

// `out_dtype` is the dtype of the expert outputs (MOE_F32 or MOE_BF16), `act_dtype` that of y.
cudaError_t launch_combine(int act_dtype, int out_dtype, const void* out, const float* gate, const int32_t* pos,
                           void* y, int T, int d, int k, int64_t rows, int32_t* status, cudaStream_t stream);

struct FfnArgs {
    int T, d, E, k, F;
    int64_t rows;      // rows of xperm / h / out
    int64_t capacity;  // per-expert row cap, or -1 (dropless); a hint for the kernel choice
    int expert_kind;
    int act_dtype;
    int precision;  // MOE_PRECISION_*
    const void* xperm;      // bf16 rows, or e4m3 codes with in_fp8
    const int32_t* offsets;
    const int32_t* counts;  // [E] rows computed at the start of each segment, or null (whole segments)
    bool in_fp8;            // up projection on e4m3 rows and weights (row-scaled)
    const float* xscale;    // [rows] with in_fp8
    const float* w13_scale; // [E * R] with in_fp8 (W13 then holds e4m3 codes)
    bool h_fp8;             // h quantized per row, down projection on e4m3 (W2 then holds e4m3 codes)
    uint8_t* hq;            // [rows, F] with h_fp8
    float* hscale;          // [rows] with h_fp8
    const float* w2_scale;  // [E * d] with h_fp8
    const void* W13;
    const void* W2;
    void* h;
    void* out;
    int32_t* status;
    // Swapped-pair GEMMs without SwiGLU: fp32 partial slots for the split of the last
    // partial wave over k, and their tickets (zero at launch, left zero); null: no split.
    float* split_part;
    int32_t* split_tickets;
    int split_slots;
};

// The workspace share of that split: kGemmSplitSlots slots of kGemmSplitSlotBytes (two
// SMs x 128 features x 256 rows of fp32) and two int32 tickets per slot.
constexpr int kGemmSplitSlots = 96;
constexpr size_t kGemmSplitSlotBytes = size_t(2) * 256 * 128 * sizeof(float);
constexpr size_t kGemmSplitTicketBytes = size_t(2) * kGemmSplitSlots * sizeof(int32_t);

// tcgen05 kernel a bf16 projection runs: 0 one SM per tile, 1 SM pairs on row
// tiles, 2 SM pairs with swapped operands.
int ffn_tc_variant(int64_t rows, int E, int64_t capacity);
// bf16 experts on the tensor cores (tcgen05 + TMA).
cudaError_t launch_ffn_tc(const FfnArgs& a, cudaStream_t stream, cudaEvent_t mid_event);
// fp32 experts on the FMA units.
cudaError_t launch_ffn_simt(const FfnArgs& a, cudaStream_t stream, cudaEvent_t mid_event);

// Tensor map for TMA over a row-major [depth, rows, inner] array of bf16 (esz 2) or
// bytes (esz 1): box = 128 bytes x box_rows x box_depth, 128-byte swizzle, zero fill
// out of bounds (a 2-D map when depth and box_depth are 1).
cudaError_t make_tensor_map_sw128(CUtensorMap* map, const void* base, uint32_t esz, uint64_t inner, uint64_t rows,
                                  uint64_t depth, uint32_t box_rows, uint32_t box_depth);

// Streaming-multiprocessor count of the current device (cached per device).
int device_sm_count();

// Key of the CUDA context current on this thread: the driver's unique context id
// (a context re-created after cudaDeviceReset gets a new one), or the device index
// with the top bit set where the driver does not report ids.
uint64_t current_context_key();

// A value set up once per CUDA context and then reused: kernel attributes, occupancy
// figures and module symbol addresses belong to the context they were made in, so a
// second device, or a context re-created after a reset, sets up its own. `make`
// returns the setup's cudaError_t, which is cached with the value. Thread-safe.
template <typename T>
class PerContext {
public:
    template <typename Make>
    cudaError_t get(T* out, Make&& make) {
        const uint64_t key = current_context_key();
        std::lock_guard<std::mutex> lock(mu_);
        for (int i = 0; i < n_; ++i)
            if (keys_[i] == key) {
                *out = vals_[i];
                return errs_[i];
            }
        T v{};
        const cudaError_t e = make(&v);
        if (n_ < kSlots) {  // beyond kSlots contexts the setup simply runs on every call
            keys_[n_] = key;
            vals_[n_] = v;
            errs_[n_] = e;
            ++n_;
        }
        *out = v;
        return e;
    }

private:
    static constexpr int kSlots = 64;
    std::mutex mu_;
    int n_ = 0;
    uint64_t keys_[kSlots] = {};
    T vals_[kSlots] = {};
    cudaError_t errs_[kSlots] = {};
};

// Raises a kernel's dynamic shared-memory limit once per context.
template <typename Kernel>
cudaError_t set_smem_limit_once(PerContext<int>& cache, Kernel kern, size_t bytes) {
    int unused = 0;
    return cache.get(&unused, [&](int*) {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes));
    });
}

}  // namespace moe
