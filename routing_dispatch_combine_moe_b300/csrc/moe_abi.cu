// The C ABI (include/moe.h): argument checks, workspace layout and the launch
// sequences of the hot path. Every entry point validates on the host, returns a
// MOE_* code synchronously, and otherwise only enqueues work on the caller's
// stream.
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "common.cuh"
#include "kernels.h"

namespace moe {

thread_local std::string g_last_cuda_error;

int device_sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

uint64_t current_context_key() {
    using GetCurrentFn = CUresult (*)(CUcontext*);
    using GetIdFn = CUresult (*)(CUcontext, unsigned long long*);
    static GetCurrentFn get_current = nullptr;
    static GetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetIdFn>(p);
    });
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
    const uint64_t fallback = (uint64_t(1) << 63) | uint64_t(uint32_t(dev));
    if (!get_current || !get_id) return fallback;
    // No context current yet (nothing has touched the device on this thread): the
    // device key stands in; the setup that follows makes the primary context current.
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return fallback;
    return uint64_t(id) & ~(uint64_t(1) << 63);
}

namespace {

constexpr size_t kAlign = 256;

inline size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }

int fail_cuda(cudaError_t e, const char* where) {
    g_last_cuda_error = std::string(where) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
    return MOE_ERR_CUDA;
}

inline int act_bytes(const moe_config* c) { return c->act_dtype == MOE_F32 ? 4 : 2; }

// All experts (routed + shared) and all slots per token (routed + shared).
inline int n_experts(const moe_config* c) { return c->E + c->n_shared; }
inline int n_slots(const moe_config* c) { return c->k + c->n_shared; }

// Rows of the dispatched-row buffers: every kept assignment (packed), or a fixed
// `capacity` rows per expert (padded).
inline int64_t rows_cap(const moe_config* c) {
    return c->layout == MOE_LAYOUT_PADDED ? int64_t(n_experts(c)) * c->capacity : int64_t(c->T) * n_slots(c);
}

inline bool bf16_experts(const moe_config* c) {
    return c->act_dtype == MOE_BF16 && c->expert_kind != MOE_EXPERT_IDENTITY;
}

// bf16 experts with h carried as hi|lo pairs.
inline bool split_h(const moe_config* c) { return bf16_experts(c) && c->precision == MOE_PRECISION_SPLIT_H; }

// dtype of the expert-output rows the combine reads.
inline int out_dtype(const moe_config* c) {
    return (bf16_experts(c) && c->precision != MOE_PRECISION_BF16) ? MOE_F32 : c->act_dtype;
}

// The FP8 wire formats: block-scaled rows turned back into bf16, or row-scaled rows for the FP8 GEMM.
inline bool fp8_blocks(const moe_config* c) { return c->dispatch_dtype == MOE_DISPATCH_FP8; }
inline bool fp8_gemm(const moe_config* c) { return c->dispatch_dtype == MOE_DISPATCH_FP8_GEMM; }
// h quantized per row and the down projection on e4m3 (with the FP8 up projection).
inline bool fp8_h(const moe_config* c) { return fp8_gemm(c) && c->precision == MOE_PRECISION_FP8_H; }

// Rows of W13 per expert: gate and up rows for SwiGLU, W1's rows for ReLU.
inline int64_t w13_rows(const moe_config* c) { return c->expert_kind == MOE_EXPERT_SWIGLU ? 2 * int64_t(c->F) : c->F; }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int validate(const moe_config* c) {
    if (!c) return MOE_ERR_ARG;
    if (c->T < 1 || c->d < 1 || c->E < 1 || c->k < 1 || c->D < 1) return MOE_ERR_ARG;
    if (c->act_dtype != MOE_F32 && c->act_dtype != MOE_BF16) return MOE_ERR_ARG;
    if (c->expert_kind != MOE_EXPERT_IDENTITY && c->expert_kind != MOE_EXPERT_RELU &&
        c->expert_kind != MOE_EXPERT_SWIGLU)
        return MOE_ERR_ARG;
    if (c->precision != MOE_PRECISION_BF16 && c->precision != MOE_PRECISION_F32_OUT &&
        c->precision != MOE_PRECISION_SPLIT_H && c->precision != MOE_PRECISION_FP8_H)
        return MOE_ERR_ARG;
    if (c->n_shared < 0) return MOE_ERR_ARG;
    if (c->k > c->E) return MOE_ERR_ARG;
    if (c->E % c->D != 0) return MOE_ERR_ARG;
    if (c->expert_kind != MOE_EXPERT_IDENTITY && c->F < 1) return MOE_ERR_ARG;
    if (c->drop_policy != MOE_DROP_TOKEN_ORDER && c->drop_policy != MOE_DROP_LOW_GATE) return MOE_ERR_ARG;
    if (c->layout != MOE_LAYOUT_PACKED && c->layout != MOE_LAYOUT_PADDED) return MOE_ERR_ARG;
    if (n_experts(c) > MOE_MAX_E || n_slots(c) > MOE_MAX_K) return MOE_ERR_UNSUPPORTED;
    if (c->layout == MOE_LAYOUT_PADDED && (c->capacity < 0 || c->n_shared != 0)) return MOE_ERR_UNSUPPORTED;
    if (c->n_groups < 0 || c->topk_groups < 0 || (c->dedup != 0 && c->dedup != 1)) return MOE_ERR_ARG;
    if (c->topk_groups > 0) {
        if (c->n_groups < 1 || c->E % c->n_groups != 0 || c->topk_groups > c->n_groups ||
            int64_t(c->k) > int64_t(c->topk_groups) * (c->E / c->n_groups))
            return MOE_ERR_ARG;
        if (c->n_groups > 32) return MOE_ERR_UNSUPPORTED;
    }
    if (c->dedup && c->D > MOE_MAX_K) return MOE_ERR_UNSUPPORTED;
    if (c->dispatch_dtype != MOE_DISPATCH_ACT && c->dispatch_dtype != MOE_DISPATCH_FP8 &&
        c->dispatch_dtype != MOE_DISPATCH_FP8_GEMM)
        return MOE_ERR_ARG;
    if ((fp8_blocks(c) || fp8_gemm(c)) && c->act_dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    if (fp8_gemm(c) && c->expert_kind == MOE_EXPERT_IDENTITY) return MOE_ERR_UNSUPPORTED;
    if (fp8_gemm(c) && c->d % 16 != 0) return MOE_ERR_ALIGN;  // e4m3 rows of d bytes, 16-byte aligned
    // the FP8 hidden activation goes with the FP8 up projection (bf16 activations), h rows of F bytes
    if (c->precision == MOE_PRECISION_FP8_H && c->act_dtype == MOE_BF16 && c->expert_kind != MOE_EXPERT_IDENTITY) {
        if (!fp8_gemm(c)) return MOE_ERR_UNSUPPORTED;
        if (c->F % 16 != 0) return MOE_ERR_ALIGN;
    }
    if (int64_t(c->T) * n_slots(c) > int64_t(INT32_MAX) || rows_cap(c) > int64_t(INT32_MAX))
        return MOE_ERR_UNSUPPORTED;
    if ((int64_t(c->d) * act_bytes(c)) % 16 != 0) return MOE_ERR_ALIGN;
    if (c->expert_kind != MOE_EXPERT_IDENTITY && (int64_t(c->F) * act_bytes(c)) % 16 != 0) return MOE_ERR_ALIGN;
    if (split_h(c) && c->F % 64 != 0) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

struct Layout {
    size_t status, near_ties, split_tickets, split_part, hist, drop_offsets, routed_offsets, elist, route_partial, topk_idx, topk_gate, counts_routed, counts_kept, offsets, rank_offsets,
        n_dropped, pos, row_src, drop_list, xperm, h, out, x_stage, y_stage;
    // deduplicated dispatch (cfg->dedup): scratch in the dispatch part, outputs in the forward part
    size_t dd_slots, dd_hist, dd_kept, dd_drop, dd_routed, dd_rank, dd_ndrop;
    size_t send_counts, send_offsets, send_pos, send_src, xsend, xsend_scale;
    size_t xq, xscale;  // FP8 dispatch
    size_t hq, hscale;  // FP8 hidden activation
    size_t dispatch_end, forward_end, host_end;
};

Layout layout(const moe_config* c) {
    Layout L{};
    const int64_t A = int64_t(c->T) * n_slots(c);
    const int N = n_experts(c);
    const int nblk = dispatch_blocks(A);
    const size_t b = size_t(act_bytes(c));
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align_up(o + bytes);
        return at;
    };
    L.status = take(2 * sizeof(int32_t));  // the status word, then the dispatch scan's ticket
    L.near_ties = take(sizeof(int32_t));
    L.split_tickets = take(bf16_experts(c) ? kGemmSplitTicketBytes : 0);
    L.hist = take(sizeof(int32_t) * size_t(N) * nblk);
    L.drop_offsets = take(sizeof(int32_t) * size_t(N));
    L.routed_offsets = take(sizeof(int32_t) * size_t(N + 1));
    L.elist = take(c->drop_policy == MOE_DROP_LOW_GATE ? 2 * sizeof(int32_t) * A : 0);  // ids, then gate keys
    const bool dd = c->dedup != 0;
    const size_t TD = size_t(c->T) * size_t(c->D);
    L.dd_slots = take(dd ? sizeof(int32_t) * TD : 0);
    L.dd_hist = take(dd ? sizeof(int32_t) * size_t(c->D) * size_t(dispatch_blocks(int64_t(TD))) : 0);
    L.dd_kept = take(dd ? sizeof(int32_t) * size_t(c->D) : 0);
    L.dd_drop = take(dd ? sizeof(int32_t) * size_t(c->D) : 0);
    L.dd_routed = take(dd ? sizeof(int32_t) * size_t(c->D + 1) : 0);
    L.dd_rank = take(dd ? sizeof(int32_t) * 2 : 0);
    L.dd_ndrop = take(dd ? sizeof(int32_t) : 0);
    L.dispatch_end = o;
    L.route_partial = take(route_scratch_bytes(c->act_dtype, c->T, c->d, c->E));
    L.topk_idx = take(sizeof(int32_t) * A);
    L.topk_gate = take(sizeof(float) * A);
    L.counts_routed = take(sizeof(int32_t) * size_t(N));
    L.counts_kept = take(sizeof(int32_t) * size_t(N));
    L.offsets = take(sizeof(int32_t) * size_t(N + 1));
    L.rank_offsets = take(sizeof(int32_t) * size_t(c->D + 1));
    L.n_dropped = take(sizeof(int32_t));
    const size_t R = size_t(rows_cap(c));
    L.pos = take(sizeof(int32_t) * A);
    L.row_src = take(sizeof(int32_t) * (R > size_t(A) ? R : size_t(A)));
    L.drop_list = take(sizeof(int32_t) * A);
    L.xperm = take(b * R * size_t(c->d));
    if (c->expert_kind != MOE_EXPERT_IDENTITY) {
        L.h = take(split_h(c) ? 2 * 2 * R * size_t(c->F) : b * R * size_t(c->F));
        L.out = take((out_dtype(c) == MOE_F32 ? 4 : b) * R * size_t(c->d));
        L.split_part = take(bf16_experts(c) ? kGemmSplitSlots * kGemmSplitSlotBytes : 0);
    } else {
        L.h = 0;
        L.out = L.xperm;
    }
    L.send_counts = take(dd ? sizeof(int32_t) * size_t(c->D) : 0);
    L.send_offsets = take(dd ? sizeof(int32_t) * size_t(c->D + 1) : 0);
    L.send_pos = take(dd ? sizeof(int32_t) * TD : 0);
    L.send_src = take(dd ? sizeof(int32_t) * TD : 0);
    L.xsend = take(dd ? b * TD * size_t(c->d) : 0);  // with FP8: the send rows' e4m3 codes
    // the send rows' scales: per 128-element block, or (FP8 GEMM rows) one per row
    L.xsend_scale = take(dd && fp8_blocks(c) ? sizeof(float) * TD * size_t((c->d + 127) / 128)
                         : dd && fp8_gemm(c) ? sizeof(float) * TD
                                             : 0);
    L.xq = take((fp8_blocks(c) && !dd) || fp8_gemm(c) ? R * size_t(c->d) : 0);
    L.xscale = take(fp8_blocks(c) && !dd ? sizeof(float) * R * size_t((c->d + 127) / 128)
                    : fp8_gemm(c) ? sizeof(float) * R
                                  : 0);
    L.hq = take(fp8_h(c) ? R * size_t(c->F) : 0);
    L.hscale = take(fp8_h(c) ? sizeof(float) * R : 0);
    L.forward_end = o;
    L.x_stage = take(b * size_t(c->T) * c->d);
    L.y_stage = take(b * size_t(c->T) * c->d);
    L.host_end = o;
    return L;
}

template <typename T>
T* at(void* ws, size_t off) {
    return reinterpret_cast<T*>(static_cast<unsigned char*>(ws) + off);
}

void fill_view(const moe_config* c, void* ws, moe_workspace_view* v) {
    const Layout L = layout(c);
    v->status = at<int32_t>(ws, L.status);
    v->topk_idx = at<int32_t>(ws, L.topk_idx);
    v->topk_gate = at<float>(ws, L.topk_gate);
    v->map.counts_routed = at<int32_t>(ws, L.counts_routed);
    v->map.counts_kept = at<int32_t>(ws, L.counts_kept);
    v->map.offsets = at<int32_t>(ws, L.offsets);
    v->map.rank_offsets = at<int32_t>(ws, L.rank_offsets);
    v->map.pos = at<int32_t>(ws, L.pos);
    v->map.row_src = at<int32_t>(ws, L.row_src);
    v->map.drop_list = at<int32_t>(ws, L.drop_list);
    v->map.n_dropped = at<int32_t>(ws, L.n_dropped);
    v->xperm = at<void>(ws, L.xperm);
    v->h = c->expert_kind == MOE_EXPERT_IDENTITY ? nullptr : at<void>(ws, L.h);
    v->out = at<void>(ws, L.out);
    const bool dd = c->dedup != 0;
    v->send.send_counts = dd ? at<int32_t>(ws, L.send_counts) : nullptr;
    v->send.send_offsets = dd ? at<int32_t>(ws, L.send_offsets) : nullptr;
    v->send.send_pos = dd ? at<int32_t>(ws, L.send_pos) : nullptr;
    v->send.send_src = dd ? at<int32_t>(ws, L.send_src) : nullptr;
    v->xsend = dd ? at<void>(ws, L.xsend) : nullptr;
    const bool f8 = fp8_blocks(c) || fp8_gemm(c);
    // FP8 with the deduplicated dispatch: the codes and scales are the send rows'
    v->xq = f8 ? at<uint8_t>(ws, dd && fp8_blocks(c) ? L.xsend : L.xq) : nullptr;
    v->xscale = f8 ? at<float>(ws, dd && fp8_blocks(c) ? L.xsend_scale : L.xscale) : nullptr;
    v->hq = fp8_h(c) ? at<uint8_t>(ws, L.hq) : nullptr;
    v->hscale = fp8_h(c) ? at<float>(ws, L.hscale) : nullptr;
    v->n_near_ties = at<int32_t>(ws, L.near_ties);
    v->xsend_scale = dd && f8 ? at<float>(ws, L.xsend_scale) : nullptr;
}

// Standalone moe_expert_ffn(_fp8) workspace: the status word, the GEMM split's tickets
// and partial slots (bf16 experts), then (FP8 hidden activation) h's codes and row scales.
struct FfnLayout {
    size_t split_tickets, split_part, hq, hscale, end;
};
FfnLayout ffn_layout(const moe_config* c) {
    FfnLayout F{};
    F.split_tickets = kAlign;
    F.split_part = align_up(F.split_tickets + (bf16_experts(c) ? kGemmSplitTicketBytes : 0));
    F.hq = align_up(F.split_part + (bf16_experts(c) ? kGemmSplitSlots * kGemmSplitSlotBytes : 0));
    const size_t R = size_t(rows_cap(c));
    F.hscale = align_up(F.hq + (fp8_h(c) ? R * size_t(c->F) : 0));
    F.end = align_up(F.hscale + (fp8_h(c) ? sizeof(float) * R : 0));
    return F;
}

int run_route(const moe_config* c, const void* x, const float* Wg, const float* bias, int32_t* idx, float* gate,
              float* scratch, cudaStream_t s, int32_t* hist = nullptr, int32_t* near_ties = nullptr,
              int32_t* status = nullptr) {
    const cudaError_t e = launch_route(c->act_dtype, x, Wg, bias, c->T, c->d, c->E, c->k, c->n_shared, c->n_groups,
                                       c->topk_groups, idx, gate, scratch, hist, near_ties, status, s);
    return e == cudaSuccess ? MOE_OK : fail_cuda(e, "moe_route");
}

int run_dispatch(const moe_config* c, const void* x, const int32_t* idx, const float* gate, const moe_dispatch_map* m,
                 void* xperm, void* ws, cudaStream_t s, bool skip_gather = false, bool counted = false) {
    const Layout L = layout(c);
    DispatchArgs a{};
    a.T = c->T; a.d = c->d; a.E = n_experts(c); a.k = n_slots(c); a.D = c->D;
    a.E_capped = c->E;
    a.capacity = c->capacity;
    a.drop_policy = c->drop_policy;
    a.layout = c->layout;
    a.topk_gate = gate;
    a.act_bytes = act_bytes(c);
    a.x = x;
    a.topk_idx = idx;
    a.counts_routed = m->counts_routed;
    a.counts_kept = m->counts_kept;
    a.offsets = m->offsets;
    a.rank_offsets = m->rank_offsets;
    a.pos = m->pos;
    a.row_src = m->row_src;
    a.drop_list = m->drop_list;
    a.n_dropped = m->n_dropped;
    a.xperm = xperm;
    a.status = at<int32_t>(ws, L.status);
    a.scan_ticket = at<int32_t>(ws, L.status) + 1;  // the int after the status word, zeroed with it
    a.hist = at<int32_t>(ws, L.hist);
    a.drop_offsets = at<int32_t>(ws, L.drop_offsets);
    a.routed_offsets = at<int32_t>(ws, L.routed_offsets);
    a.elist = c->drop_policy == MOE_DROP_LOW_GATE ? at<int32_t>(ws, L.elist) : nullptr;
    a.skip_gather = skip_gather;
    a.counted = counted;
    const cudaError_t e = launch_dispatch(a, s);
    return e == cudaSuccess ? MOE_OK : fail_cuda(e, "moe_dispatch");
}

// Deduplicated send buffer + fan-out into xperm; the scratch lives in the dispatch part of ws.
// xsend_scale: the send rows' scales with an FP8 dispatch dtype; xq, xscale: the expert
// rows' codes and row scales with MOE_DISPATCH_FP8_GEMM (xperm is then not written).
int run_dedup(const moe_config* c, const void* x, const int32_t* idx, const int32_t* pos, const moe_send_map* m,
              void* xsend, void* xperm, void* ws, cudaStream_t s, float* xsend_scale = nullptr,
              uint8_t* xq = nullptr, float* xscale = nullptr) {
    const Layout L = layout(c);
    DedupArgs a{};
    a.T = c->T; a.d = c->d; a.K = n_slots(c); a.E_routed = c->E; a.D = c->D;
    a.act_bytes = act_bytes(c);
    a.rows = rows_cap(c);
    a.x = x;
    a.topk_idx = idx;
    a.pos = pos;
    a.send_counts = m->send_counts;
    a.send_offsets = m->send_offsets;
    a.send_pos = m->send_pos;
    a.send_src = m->send_src;
    a.xsend = xsend;
    a.xsend_scale = xsend_scale;
    a.fp8 = fp8_blocks(c);
    a.fp8_rows = fp8_gemm(c);
    a.xq = xq;
    a.xscale = xscale;
    a.xperm = xperm;
    a.status = at<int32_t>(ws, L.status);
    a.slots = at<int32_t>(ws, L.dd_slots);
    a.hist = at<int32_t>(ws, L.dd_hist);
    a.kept_scratch = at<int32_t>(ws, L.dd_kept);
    a.drop_offsets = at<int32_t>(ws, L.dd_drop);
    a.routed_offsets = at<int32_t>(ws, L.dd_routed);
    a.rank_offsets = at<int32_t>(ws, L.dd_rank);
    a.n_dropped = at<int32_t>(ws, L.dd_ndrop);
    const cudaError_t e = launch_dedup(a, s);
    return e == cudaSuccess ? MOE_OK : fail_cuda(e, "moe_dispatch_dedup");
}

int run_fp8(const moe_config* c, const void* x, const int32_t* idx, const moe_dispatch_map* m, uint8_t* xq,
            float* xscale, void* xperm, void* ws, cudaStream_t s) {
    const Layout L = layout(c);
    Fp8Args a{};
    a.T = c->T; a.d = c->d; a.K = n_slots(c); a.E_routed = c->E; a.n_experts = n_experts(c);
    a.rows = rows_cap(c);
    a.x = x;
    a.topk_idx = idx;
    a.pos = m->pos;
    a.row_src = m->row_src;
    a.offsets = m->offsets;
    a.xq = xq;
    a.xscale = xscale;
    a.xperm = xperm;
    a.per_row = fp8_gemm(c);
    a.dequant = xperm != nullptr && !a.per_row;
    a.status = at<int32_t>(ws, L.status);
    const cudaError_t e = launch_fp8_dispatch(a, s);
    return e == cudaSuccess ? MOE_OK : fail_cuda(e, "moe_dispatch_fp8");
}

// Byte offset of the weight scales inside an FP8 W13 buffer (after the codes).
inline size_t fp8_weight_scale_offset(const moe_config* c) {
    return align_up(size_t(n_experts(c)) * size_t(w13_rows(c)) * size_t(c->d));
}

// Same for an FP8 W2 buffer.
inline size_t fp8_w2_scale_offset(const moe_config* c) {
    return align_up(size_t(n_experts(c)) * size_t(c->d) * size_t(c->F));
}

// xscale: the rows' scales when cfg is MOE_DISPATCH_FP8_GEMM (xperm then holds their
// e4m3 codes and W13 the FP8 weight buffer).
int run_ffn(const moe_config* c, const void* xperm, const int32_t* offsets, const int32_t* counts, const void* W13,
            const void* W2, void* h, void* out, int32_t* status, cudaStream_t s, cudaEvent_t mid,
            const float* xscale = nullptr, uint8_t* hq = nullptr, float* hscale = nullptr,
            float* split_part = nullptr, int32_t* split_tickets = nullptr) {
    FfnArgs a{};
    if (bf16_experts(c) && split_part && split_tickets) {
        a.split_part = split_part;
        a.split_tickets = split_tickets;
        a.split_slots = kGemmSplitSlots;
    }
    if (fp8_gemm(c)) {
        a.in_fp8 = true;
        a.xscale = xscale;
        a.w13_scale = reinterpret_cast<const float*>(static_cast<const unsigned char*>(W13) +
                                                     fp8_weight_scale_offset(c));
    }
    if (fp8_h(c)) {
        a.h_fp8 = true;
        a.hq = hq;
        a.hscale = hscale;
        a.w2_scale = reinterpret_cast<const float*>(static_cast<const unsigned char*>(W2) + fp8_w2_scale_offset(c));
    }
    a.T = c->T; a.d = c->d; a.E = n_experts(c); a.k = n_slots(c); a.F = c->F;
    a.rows = rows_cap(c);
    a.capacity = c->capacity;
    a.expert_kind = c->expert_kind;
    a.act_dtype = c->act_dtype;
    a.precision = c->precision;
    a.xperm = xperm;
    a.offsets = offsets;
    a.counts = counts;
    a.W13 = W13;
    a.W2 = W2;
    a.h = h;
    a.out = out;
    a.status = status;
    if (a.rows == 0) {  // padded layout with capacity 0: no rows, nothing to compute
        if (!mid) return MOE_OK;
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        cudaError_t e = cudaStreamIsCapturing(s, &cs);
        if (e == cudaSuccess)
            e = cs == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(mid, s, cudaEventRecordExternal)
                                                    : cudaEventRecord(mid, s);
        return e == cudaSuccess ? MOE_OK : fail_cuda(e, "cudaEventRecord");
    }
    const cudaError_t e = c->act_dtype == MOE_BF16 ? launch_ffn_tc(a, s, mid) : launch_ffn_simt(a, s, mid);
    return e == cudaSuccess ? MOE_OK : fail_cuda(e, "moe_expert_ffn");
}

// Records events[i] on s. Under stream capture the record becomes an event node of
// the graph (external record), so the timestamps exist when the graph is replayed.
int record(void* const* events, int n, int i, cudaStream_t s) {
    if (!events || i >= n || !events[i]) return MOE_OK;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cs);
    if (e != cudaSuccess) return fail_cuda(e, "cudaStreamIsCapturing");
    e = cs == cudaStreamCaptureStatusActive
            ? cudaEventRecordWithFlags(static_cast<cudaEvent_t>(events[i]), s, cudaEventRecordExternal)
            : cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s);
    return e == cudaSuccess ? MOE_OK : fail_cuda(e, "cudaEventRecord");
}

int forward(const moe_config* c, const void* x, const float* Wg, const float* bias, const void* W13, const void* W2,
            void* y, void* ws, size_t ws_bytes, cudaStream_t s, void* const* events, int n_events) {
    int rc = validate(c);
    if (rc != MOE_OK) return rc;
    if (!x || !Wg || !y || !ws) return MOE_ERR_ARG;
    if (c->expert_kind != MOE_EXPERT_IDENTITY && (!W13 || !W2)) return MOE_ERR_ARG;
    if (!aligned16(x) || !aligned16(y) || !aligned4(Wg) || (bias && !aligned4(bias)) || !aligned16(ws))
        return MOE_ERR_ALIGN;
    if (W13 && (!aligned16(W13) || !aligned16(W2))) return MOE_ERR_ALIGN;
    const Layout L = layout(c);
    if (ws_bytes < L.forward_end) return MOE_ERR_WORKSPACE;
    moe_workspace_view v{};
    fill_view(c, ws, &v);
    // The router also counts each expert's assignments per dispatch block (the fused
    // route + count) and the near-tie tokens: one memset clears the status word, the
    // near-tie count, the expert GEMM split's tickets and that histogram, which follow
    // each other at the start of the workspace.
    const size_t hist_end = L.hist + sizeof(int32_t) * size_t(n_experts(c)) *
                                         size_t(dispatch_blocks(int64_t(c->T) * n_slots(c)));
    cudaError_t e = cudaMemsetAsync(ws, 0, hist_end, s);
    if (e != cudaSuccess) return fail_cuda(e, "cudaMemsetAsync(status, histogram)");
    if ((rc = record(events, n_events, 0, s)) != MOE_OK) return rc;
    if ((rc = run_route(c, x, Wg, bias, v.topk_idx, v.topk_gate, at<float>(ws, L.route_partial), s,
                        at<int32_t>(ws, L.hist), v.n_near_ties, v.status)) != MOE_OK)
        return rc;
    if ((rc = record(events, n_events, 1, s)) != MOE_OK) return rc;
    const bool f8 = fp8_blocks(c) || fp8_gemm(c);
    if ((rc = run_dispatch(c, x, v.topk_idx, v.topk_gate, &v.map, v.xperm, ws, s, c->dedup != 0 || f8, true)) !=
        MOE_OK)
        return rc;
    // with the deduplicated dispatch the FP8 rows travel in the send buffer (run_dedup)
    if (f8 && !c->dedup &&
        (rc = run_fp8(c, x, v.topk_idx, &v.map, v.xq, v.xscale, fp8_gemm(c) ? nullptr : v.xperm, ws, s)) != MOE_OK)
        return rc;
    if (c->dedup && (rc = run_dedup(c, x, v.topk_idx, v.map.pos, &v.send, v.xsend, v.xperm, ws, s, v.xsend_scale,
                                    fp8_gemm(c) ? v.xq : nullptr, fp8_gemm(c) ? v.xscale : nullptr)) != MOE_OK)
        return rc;
    if ((rc = record(events, n_events, 2, s)) != MOE_OK) return rc;
    if (c->expert_kind != MOE_EXPERT_IDENTITY) {
        cudaEvent_t mid = (events && n_events > 3) ? static_cast<cudaEvent_t>(events[3]) : nullptr;
        // Padded layout: the GEMMs skip each segment's padding rows (only kept rows are
        // ever combined), so those rows of `out` are left unwritten by the forward.
        const int32_t* used = c->layout == MOE_LAYOUT_PADDED ? v.map.counts_kept : nullptr;
        const void* rows = fp8_gemm(c) ? static_cast<const void*>(v.xq) : v.xperm;
        if ((rc = run_ffn(c, rows, v.map.offsets, used, W13, W2, v.h, v.out, v.status, s, mid, v.xscale, v.hq,
                          v.hscale, bf16_experts(c) ? at<float>(ws, L.split_part) : nullptr,
                          bf16_experts(c) ? at<int32_t>(ws, L.split_tickets) : nullptr)) != MOE_OK)
            return rc;
    } else if ((rc = record(events, n_events, 3, s)) != MOE_OK) {
        return rc;
    }
    if ((rc = record(events, n_events, 4, s)) != MOE_OK) return rc;
    e = launch_combine(c->act_dtype, out_dtype(c), v.out, v.topk_gate, v.map.pos, y, c->T, c->d, n_slots(c),
                       rows_cap(c), v.status, s);
    if (e != cudaSuccess) return fail_cuda(e, "moe_combine");
    return record(events, n_events, 5, s);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int64_t moe_capacity(int32_t T, int32_t k, int32_t E, int64_t cf_num, int64_t cf_den, int64_t min_capacity) {
    if (T <= 0 || k <= 0 || E <= 0 || cf_den <= 0 || cf_num < 0) return -1;
    // ceil(cf_num * T * k / (cf_den * E)) without overflow for realistic sizes (128-bit product).
    const __int128 num = static_cast<__int128>(cf_num) * T * k;
    const __int128 den = static_cast<__int128>(cf_den) * E;
    __int128 c = (num + den - 1) / den;
    if (c < min_capacity) c = min_capacity;
    if (c > INT64_MAX) c = INT64_MAX;
    return static_cast<int64_t>(c);
}

int moe_validate_config(const moe_config* cfg) { return validate(cfg); }

int64_t moe_rows_capacity(const moe_config* cfg) { return validate(cfg) == MOE_OK ? rows_cap(cfg) : -1; }

size_t moe_dispatch_workspace_bytes(const moe_config* cfg) {
    return validate(cfg) == MOE_OK ? layout(cfg).dispatch_end : 0;
}

size_t moe_ffn_workspace_bytes(const moe_config* cfg) { return validate(cfg) == MOE_OK ? ffn_layout(cfg).end : 0; }

size_t moe_workspace_bytes(const moe_config* cfg) { return validate(cfg) == MOE_OK ? layout(cfg).forward_end : 0; }

size_t moe_workspace_bytes_host(const moe_config* cfg) {
    return validate(cfg) == MOE_OK ? layout(cfg).host_end : 0;
}

int moe_workspace_get_view(const moe_config* cfg, void* ws, size_t ws_bytes, moe_workspace_view* view) {
    const int rc = validate(cfg);
    if (rc != MOE_OK) return rc;
    if (!ws || !view) return MOE_ERR_ARG;
    if (ws_bytes < layout(cfg).forward_end) return MOE_ERR_WORKSPACE;
    fill_view(cfg, ws, view);
    return MOE_OK;
}

int moe_kernels_per_forward(const moe_config* cfg) {
    if (validate(cfg) != MOE_OK) return 0;
    // router (which also counts) + (scan, scatter, [select], [pad], gather) + (up, down) + combine
    const int select = cfg->drop_policy == MOE_DROP_LOW_GATE && cfg->capacity >= 0 ? 1 : 0;
    const int pad = cfg->layout == MOE_LAYOUT_PADDED && cfg->capacity > 0 ? 1 : 0;
    const int ffn = cfg->expert_kind == MOE_EXPERT_IDENTITY || rows_cap(cfg) == 0 ? 0 : 2;
    const int dedup = cfg->dedup ? 5 : 0;  // mask, count, scan, scatter, fan-out (the gather goes to xsend)
    // dequant (the gather quantizes; FP8_GEMM rows are used as they are; with dedup the fan-out dequantizes)
    const int fp8 = fp8_blocks(cfg) && !cfg->dedup ? 1 : 0;
    const int fp8h = fp8_h(cfg) && ffn ? 1 : 0;  // h quantized between the two GEMMs
    // fused; or logits + top-k; or (tensor cores) W_g's split + logits + top-k
    const int route = route_uses_small_kernel(cfg->d, cfg->E) ? 1 : (route_uses_tc(cfg->act_dtype, cfg->d, cfg->E) ? 3 : 2);
    return route + 3 + select + pad + dedup + fp8 + fp8h + ffn + 1;
}

size_t moe_route_workspace_bytes(const moe_config* cfg) {
    return validate(cfg) == MOE_OK ? route_scratch_bytes(cfg->act_dtype, cfg->T, cfg->d, cfg->E) : 0;
}

int moe_route(const moe_config* cfg, const void* x, const float* Wg, const float* bias, int32_t* topk_idx,
              float* topk_gate, void* ws, size_t ws_bytes, moe_stream_t stream) {
    const int rc = validate(cfg);
    if (rc != MOE_OK) return rc;
    if (!x || !Wg || !topk_idx || !topk_gate) return MOE_ERR_ARG;
    const size_t need = route_scratch_bytes(cfg->act_dtype, cfg->T, cfg->d, cfg->E);
    if (need && !ws) return MOE_ERR_ARG;
    if (!aligned16(x) || !aligned4(Wg) || (bias && !aligned4(bias)) || !aligned4(topk_idx) || !aligned4(topk_gate) ||
        (ws && !aligned16(ws)))
        return MOE_ERR_ALIGN;
    if (ws_bytes < need) return MOE_ERR_WORKSPACE;
    return run_route(cfg, x, Wg, bias, topk_idx, topk_gate, static_cast<float*>(ws), stream);
}

int moe_dispatch(const moe_config* cfg, const void* x, const int32_t* topk_idx, const float* topk_gate,
                 const moe_dispatch_map* map, void* xperm, void* ws, size_t ws_bytes, moe_stream_t stream) {
    const int rc = validate(cfg);
    if (rc != MOE_OK) return rc;
    // xperm may be NULL only when there are no rows (padded layout, capacity 0)
    if (!x || !topk_idx || !map || (!xperm && rows_cap(cfg) > 0) || !ws) return MOE_ERR_ARG;
    if (cfg->drop_policy == MOE_DROP_LOW_GATE && cfg->capacity >= 0 && !topk_gate) return MOE_ERR_ARG;
    if (!map->counts_routed || !map->counts_kept || !map->offsets || !map->rank_offsets || !map->pos ||
        !map->row_src || !map->drop_list || !map->n_dropped)
        return MOE_ERR_ARG;
    if (!aligned16(x) || !aligned16(xperm) || !aligned16(ws)) return MOE_ERR_ALIGN;
    if (ws_bytes < layout(cfg).dispatch_end) return MOE_ERR_WORKSPACE;
    // the status word and the scan's ticket after it
    const cudaError_t e = cudaMemsetAsync(ws, 0, 2 * sizeof(int32_t), stream);
    if (e != cudaSuccess) return fail_cuda(e, "cudaMemsetAsync(status)");
    return run_dispatch(cfg, x, topk_idx, topk_gate, map, xperm, ws, stream);
}

int moe_dispatch_dedup(const moe_config* cfg, const void* x, const int32_t* topk_idx, const int32_t* pos,
                       const moe_send_map* map, void* xsend, void* xperm, void* ws, size_t ws_bytes,
                       moe_stream_t stream) {
    const int rc = validate(cfg);
    if (rc != MOE_OK) return rc;
    if (!cfg->dedup || fp8_blocks(cfg) || fp8_gemm(cfg)) return MOE_ERR_ARG;
    if (!x || !topk_idx || !pos || !map || !ws || !map->send_counts || !map->send_offsets || !map->send_pos ||
        !map->send_src || !xsend || (!xperm && rows_cap(cfg) > 0))
        return MOE_ERR_ARG;
    if (!aligned16(x) || !aligned16(xsend) || (xperm && !aligned16(xperm)) || !aligned4(topk_idx) || !aligned4(pos) ||
        !aligned16(ws))
        return MOE_ERR_ALIGN;
    if (ws_bytes < layout(cfg).dispatch_end) return MOE_ERR_WORKSPACE;
    const cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(int32_t), stream);
    if (e != cudaSuccess) return fail_cuda(e, "cudaMemsetAsync(status)");
    return run_dedup(cfg, x, topk_idx, pos, map, xsend, xperm, ws, stream);
}

int moe_dispatch_dedup_fp8(const moe_config* cfg, const void* x, const int32_t* topk_idx, const int32_t* pos,
                           const moe_send_map* map, uint8_t* xsend_q, float* xsend_scale, void* xperm, void* ws,
                           size_t ws_bytes, moe_stream_t stream) {
    const int rc = validate(cfg);
    if (rc != MOE_OK) return rc;
    if (!cfg->dedup || !fp8_blocks(cfg)) return MOE_ERR_ARG;
    if (!x || !topk_idx || !pos || !map || !ws || !map->send_counts || !map->send_offsets || !map->send_pos ||
        !map->send_src || !xsend_q || !xsend_scale || (!xperm && rows_cap(cfg) > 0))
        return MOE_ERR_ARG;
    if (!aligned16(x) || !aligned16(xsend_q) || !aligned4(xsend_scale) || (xperm && !aligned16(xperm)) ||
        !aligned4(topk_idx) || !aligned4(pos) || !aligned16(ws))
        return MOE_ERR_ALIGN;
    if (ws_bytes < layout(cfg).dispatch_end) return MOE_ERR_WORKSPACE;
    const cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(int32_t), stream);
    if (e != cudaSuccess) return fail_cuda(e, "cudaMemsetAsync(status)");
    return run_dedup(cfg, x, topk_idx, pos, map, xsend_q, xperm, ws, stream, xsend_scale);
}

int moe_dispatch_dedup_fp8_gemm(const moe_config* cfg, const void* x, const int32_t* topk_idx, const int32_t* pos,
                                const moe_send_map* map, uint8_t* xsend_q, float* xsend_scale, uint8_t* xq,
                                float* xscale, void* ws, size_t ws_bytes, moe_stream_t stream) {
    const int rc = validate(cfg);
    if (rc != MOE_OK) return rc;
    if (!cfg->dedup || !fp8_gemm(cfg)) return MOE_ERR_ARG;
    const bool rows = rows_cap(cfg) > 0;
    if (!x || !topk_idx || !pos || !map || !ws || !map->send_counts || !map->send_offsets || !map->send_pos ||
        !map->send_src || !xsend_q || !xsend_scale || (rows && (!xq || !xscale)))
        return MOE_ERR_ARG;
    if (!aligned16(x) || !aligned16(xsend_q) || !aligned4(xsend_scale) || (xq && !aligned16(xq)) ||
        (xscale && !aligned4(xscale)) || !aligned4(topk_idx) || !aligned4(pos) || !aligned16(ws))
        return MOE_ERR_ALIGN;
    if (ws_bytes < layout(cfg).dispatch_end) return MOE_ERR_WORKSPACE;
    const cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(int32_t), stream);
    if (e != cudaSuccess) return fail_cuda(e, "cudaMemsetAsync(status)");
    return run_dedup(cfg, x, topk_idx, pos, map, xsend_q, nullptr, ws, stream, xsend_scale, xq, xscale);
}

int moe_dispatch_fp8(const moe_config* cfg, const void* x, const int32_t* topk_idx, const moe_dispatch_map* map,
                     uint8_t* xq, float* xscale, void* xperm, void* ws, size_t ws_bytes, moe_stream_t stream) {
    const int rc = validate(cfg);
    if (rc != MOE_OK) return rc;
    if (!fp8_blocks(cfg) && !fp8_gemm(cfg)) return MOE_ERR_ARG;
    if (fp8_gemm(cfg) && xperm) return MOE_ERR_ARG;
    const bool rows = rows_cap(cfg) > 0;
    if (!x || !topk_idx || !map || !map->pos || !map->row_src || !map->offsets || !ws || (rows && (!xq || !xscale)))
        return MOE_ERR_ARG;
    if (!aligned16(x) || (xperm && !aligned16(xperm)) || (xq && !aligned16(xq)) || (xscale && !aligned4(xscale)) ||
        !aligned16(ws))
        return MOE_ERR_ALIGN;
    if (ws_bytes < layout(cfg).dispatch_end) return MOE_ERR_WORKSPACE;
    const cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(int32_t), stream);
    if (e != cudaSuccess) return fail_cuda(e, "cudaMemsetAsync(status)");
    return run_fp8(cfg, x, topk_idx, map, xq, xscale, xperm, ws, stream);
}

int moe_expert_ffn(const moe_config* cfg, const void* xperm, const int32_t* offsets, const void* W13, const void* W2,
                   void* h, void* out, void* ws, size_t ws_bytes, moe_stream_t stream) {
    const int rc = validate(cfg);
    if (rc != MOE_OK) return rc;
    if (cfg->expert_kind == MOE_EXPERT_IDENTITY || fp8_gemm(cfg)) return MOE_ERR_ARG;
    if (!offsets || !W13 || !W2 || !ws) return MOE_ERR_ARG;
    if ((!xperm || !h || !out) && rows_cap(cfg) > 0) return MOE_ERR_ARG;
    if (!aligned16(xperm) || !aligned16(W13) || !aligned16(W2) || !aligned16(h) || !aligned16(out) ||
        !aligned16(ws))
        return MOE_ERR_ALIGN;
    const FfnLayout FL = ffn_layout(cfg);
    if (ws_bytes < FL.end) return MOE_ERR_WORKSPACE;
    // the status word and the GEMM split's tickets
    int32_t* status = static_cast<int32_t*>(ws);
    const cudaError_t e = cudaMemsetAsync(status, 0, FL.split_part, stream);
    if (e != cudaSuccess) return fail_cuda(e, "cudaMemsetAsync(status, split tickets)");
    return run_ffn(cfg, xperm, offsets, nullptr, W13, W2, h, out, status, stream, nullptr, nullptr, nullptr, nullptr,
                   at<float>(ws, FL.split_part), at<int32_t>(ws, FL.split_tickets));
}

size_t moe_fp8_weight_bytes(const moe_config* cfg) {
    if (validate(cfg) != MOE_OK || !fp8_gemm(cfg)) return 0;
    return fp8_weight_scale_offset(cfg) + sizeof(float) * size_t(n_experts(cfg)) * size_t(w13_rows(cfg));
}

int moe_quantize_weights_fp8(const moe_config* cfg, const void* W13, void* W13_fp8, moe_stream_t stream) {
    const int rc = validate(cfg);
    if (rc != MOE_OK) return rc;
    if (!fp8_gemm(cfg) || !W13 || !W13_fp8) return MOE_ERR_ARG;
    if (!aligned16(W13) || !aligned16(W13_fp8)) return MOE_ERR_ALIGN;
    unsigned char* q = static_cast<unsigned char*>(W13_fp8);
    const cudaError_t e = launch_quantize_rows_fp8(W13, int64_t(n_experts(cfg)) * w13_rows(cfg), cfg->d, q,
                                                   reinterpret_cast<float*>(q + fp8_weight_scale_offset(cfg)),
                                                   stream);
    return e == cudaSuccess ? MOE_OK : fail_cuda(e, "moe_quantize_weights_fp8");
}

size_t moe_fp8_w2_bytes(const moe_config* cfg) {
    if (validate(cfg) != MOE_OK || !fp8_h(cfg)) return 0;
    return fp8_w2_scale_offset(cfg) + sizeof(float) * size_t(n_experts(cfg)) * size_t(cfg->d);
}

int moe_quantize_w2_fp8(const moe_config* cfg, const void* W2, void* W2_fp8, moe_stream_t stream) {
    const int rc = validate(cfg);
    if (rc != MOE_OK) return rc;
    if (!fp8_h(cfg) || !W2 || !W2_fp8) return MOE_ERR_ARG;
    if (!aligned16(W2) || !aligned16(W2_fp8)) return MOE_ERR_ALIGN;
    unsigned char* q = static_cast<unsigned char*>(W2_fp8);
    const cudaError_t e = launch_quantize_rows_fp8(W2, int64_t(n_experts(cfg)) * cfg->d, cfg->F, q,
                                                   reinterpret_cast<float*>(q + fp8_w2_scale_offset(cfg)), stream);
    return e == cudaSuccess ? MOE_OK : fail_cuda(e, "moe_quantize_w2_fp8");
}

int moe_expert_ffn_fp8(const moe_config* cfg, const uint8_t* xq, const float* xscale, const int32_t* offsets,
                       const void* W13_fp8, const void* W2, void* h, void* out, void* ws, size_t ws_bytes,
                       moe_stream_t stream) {
    const int rc = validate(cfg);
    if (rc != MOE_OK) return rc;
    if (!fp8_gemm(cfg)) return MOE_ERR_ARG;
    if (!offsets || !W13_fp8 || !W2 || !ws) return MOE_ERR_ARG;
    if ((!xq || !xscale || !h || !out) && rows_cap(cfg) > 0) return MOE_ERR_ARG;
    if (!aligned16(xq) || !aligned4(xscale) || !aligned16(W13_fp8) || !aligned16(W2) || !aligned16(h) ||
        !aligned16(out) || !aligned16(ws))
        return MOE_ERR_ALIGN;
    const FfnLayout FL = ffn_layout(cfg);
    if (ws_bytes < FL.end) return MOE_ERR_WORKSPACE;
    // the status word and the GEMM split's tickets
    int32_t* status = static_cast<int32_t*>(ws);
    const cudaError_t e = cudaMemsetAsync(status, 0, FL.split_part, stream);
    if (e != cudaSuccess) return fail_cuda(e, "cudaMemsetAsync(status, split tickets)");
    return run_ffn(cfg, xq, offsets, nullptr, W13_fp8, W2, h, out, status, stream, nullptr, xscale,
                   fp8_h(cfg) ? at<uint8_t>(ws, FL.hq) : nullptr, fp8_h(cfg) ? at<float>(ws, FL.hscale) : nullptr,
                   at<float>(ws, FL.split_part), at<int32_t>(ws, FL.split_tickets));
}

int moe_combine(const moe_config* cfg, const void* out, const float* topk_gate, const int32_t* pos, void* y,
                int32_t* status, moe_stream_t stream) {
    const int rc = validate(cfg);
    if (rc != MOE_OK) return rc;
    if ((!out && rows_cap(cfg) > 0) || !topk_gate || !pos || !y) return MOE_ERR_ARG;
    if (!aligned16(out) || !aligned16(y) || !aligned4(topk_gate) || !aligned4(pos)) return MOE_ERR_ALIGN;
    const cudaError_t e = launch_combine(cfg->act_dtype, out_dtype(cfg), out, topk_gate, pos, y, cfg->T, cfg->d,
                                         n_slots(cfg), rows_cap(cfg), status, stream);
    return e == cudaSuccess ? MOE_OK : fail_cuda(e, "moe_combine");
}

int moe_layer_forward(const moe_config* cfg, const void* x, const float* Wg, const float* bias, const void* W13,
                      const void* W2, void* y, void* ws, size_t ws_bytes, moe_stream_t stream) {
    return forward(cfg, x, Wg, bias, W13, W2, y, ws, ws_bytes, stream, nullptr, 0);
}

int moe_layer_forward_traced(const moe_config* cfg, const void* x, const float* Wg, const float* bias,
                             const void* W13, const void* W2, void* y, void* ws, size_t ws_bytes,
                             moe_stream_t stream, void* const* events, int32_t n_events) {
    if (!events || n_events < 6) return MOE_ERR_ARG;
    return forward(cfg, x, Wg, bias, W13, W2, y, ws, ws_bytes, stream, events, n_events);
}

int moe_layer_forward_host_async(const moe_config* cfg, const void* x_host, const float* Wg, const float* bias,
                                 const void* W13, const void* W2, void* y_host, void* ws, size_t ws_bytes,
                                 moe_stream_t stream) {
    int rc = validate(cfg);
    if (rc != MOE_OK) return rc;
    if (!x_host || !y_host || !ws) return MOE_ERR_ARG;
    const Layout L = layout(cfg);
    if (ws_bytes < L.host_end) return MOE_ERR_WORKSPACE;
    const size_t bytes = size_t(act_bytes(cfg)) * cfg->T * cfg->d;
    void* xs = at<void>(ws, L.x_stage);
    void* ys = at<void>(ws, L.y_stage);
    cudaError_t e = cudaMemcpyAsync(xs, x_host, bytes, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return fail_cuda(e, "cudaMemcpyAsync(x)");
    if ((rc = forward(cfg, xs, Wg, bias, W13, W2, ys, ws, ws_bytes, stream, nullptr, 0)) != MOE_OK) return rc;
    e = cudaMemcpyAsync(y_host, ys, bytes, cudaMemcpyDeviceToHost, stream);
    return e == cudaSuccess ? MOE_OK : fail_cuda(e, "cudaMemcpyAsync(y)");
}

int moe_layer_forward_host(const moe_config* cfg, const void* x_host, const float* Wg, const float* bias,
                           const void* W13, const void* W2, void* y_host, void* ws, size_t ws_bytes,
                           moe_stream_t stream) {
    const int rc = moe_layer_forward_host_async(cfg, x_host, Wg, bias, W13, W2, y_host, ws, ws_bytes, stream);
    if (rc != MOE_OK) return rc;
    const cudaError_t e = cudaStreamSynchronize(stream);
    return e == cudaSuccess ? MOE_OK : fail_cuda(e, "cudaStreamSynchronize");
}

int moe_read_status(const int32_t* status_dev, int32_t* flags_host, moe_stream_t stream) {
    if (!status_dev) return MOE_ERR_ARG;
    int32_t h = 0;
    cudaError_t e = cudaMemcpyAsync(&h, status_dev, sizeof(h), cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return fail_cuda(e, "cudaMemcpyAsync(status)");
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return fail_cuda(e, "cudaStreamSynchronize");
    if (flags_host) *flags_host = h;
    return h == 0 ? MOE_OK : MOE_ERR_DEVICE;
}

const char* moe_status_string(int code) {
    switch (code) {
        case MOE_OK: return "ok";
        case MOE_ERR_ARG: return "invalid argument";
        case MOE_ERR_ALIGN: return "pointer or activation row not 16-byte aligned";
        case MOE_ERR_WORKSPACE: return "workspace too small";
        case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
        case MOE_ERR_CUDA: return "CUDA runtime error";
        case MOE_ERR_DEVICE: return "device reported an error";
        default: return "unknown status";
    }
}

const char* moe_last_cuda_error(void) { return g_last_cuda_error.c_str(); }

const char* moe_ffn_kernel_name(const moe_config* cfg) {
    if (validate(cfg) != MOE_OK || cfg->expert_kind == MOE_EXPERT_IDENTITY) return "";
    if (cfg->act_dtype == MOE_F32) return "grouped_sgemm_kernel";
    if (fp8_gemm(cfg)) return "grouped_gemm_swap_kernel<e4m3>";
    switch (ffn_tc_variant(rows_cap(cfg), n_experts(cfg), cfg->capacity)) {
        case 1: return "grouped_gemm_kernel<pair>";
        case 2: return "grouped_gemm_swap_kernel";
        default: return "grouped_gemm_kernel";
    }
}

int moe_version(void) { return 202; }

}  // extern "C"
