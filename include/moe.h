/*
 * moe.h - C ABI of the B300 (sm_103a) library for the forward pass of one
 * top-k-routed Mixture-of-Experts FFN layer on one GPU.
 *
 * What the layer computes (sources, by page title and section):
 *   - "Mixture-of-Experts (MoE) Architecture and Expert Parallelism",
 *     section 2 "The Gating Network Formulation":
 *       H(x) = x W_g (+ eps),  G(x) = Softmax(KeepTopK(H(x), k)),
 *       y = sum over the k kept experts i of G_i(x) * Expert_i(x).
 *   - "EP Math - Expert Parallelism (MoE)": "The dispatch all-to-all" and
 *     "The combine all-to-all" (each of the T*k assignments is a d-vector sent to
 *     its expert and returned), "Capacity factor: fixing buffer sizes"
 *     (C = f*T*k/E, rounded up) and "Token drop: what overflow costs" (overflow is
 *     not processed and contributes zero; the caller's residual carries x).
 *   - "MoE Expert Parallelism Sizing: Traffic, Capacity, Fabric",
 *     "First-order dispatch and combine bytes": an all-to-all input buffer holds
 *     one contiguous chunk per destination rank.
 *
 * On one GPU the dispatch and combine all-to-alls are on-device permutations:
 * dispatched rows are grouped by expert, experts ascending, tokens ascending
 * within an expert, so rank r of D virtual ranks (experts [r*E/D,(r+1)*E/D))
 * owns one contiguous chunk of rows.
 *
 * Shared experts: with S = cfg.n_shared > 0, experts E..E+S-1 are shared: every token
 * also uses each of them with gate 1, after its k routed slots (the pages' decode
 * example sends each token to 8 routed experts plus the shared one). Below, "slots"
 * K = k + S and "experts" N = E + S; capacity limits only the routed experts, and the
 * D virtual ranks split the routed experts, the shared rows following rank D-1's.
 *
 * Conventions for every entry point:
 *   - Pointers named *_host are host memory; every other pointer is device
 *     memory on the current CUDA device, allocated and owned by the caller. The
 *     library allocates no memory and keeps no per-call state; scratch lives in
 *     a caller-provided workspace.
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) without host synchronisation, so a sequence of calls can be
 *     captured in a CUDA graph. Exceptions: moe_read_status and
 *     moe_layer_forward_host (see their comments); moe_layer_forward_host_async
 *     enqueues host copies, which a graph capture can hold only with pinned buffers.
 *   - Argument errors are returned synchronously as a MOE_ERR_* code before any
 *     work is enqueued. Errors found on the device (an expert id or row index
 *     out of range, a bounded wait that gave up) set bits in a device status
 *     word (MOE_DEV_* flags) instead; read it with moe_read_status.
 *   - Layouts are row-major. Activation rows (x, dispatched rows, expert
 *     outputs, y) must start on 16-byte boundaries: d * sizeof(act) % 16 == 0
 *     and every activation pointer 16-byte aligned. Index arrays are int32.
 *   - The functions are thread-safe; the same workspace must not be used by two
 *     calls that may overlap on the GPU.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* a cudaStream_t */

/* Return codes. */
#define MOE_OK 0
#define MOE_ERR_ARG 1         /* null pointer, non-positive size, k > E, E % D != 0, ... */
#define MOE_ERR_ALIGN 2       /* pointer or activation row not 16-byte aligned */
#define MOE_ERR_WORKSPACE 3   /* workspace smaller than the matching *_workspace_bytes */
#define MOE_ERR_UNSUPPORTED 4 /* valid request this build does not implement (limits below) */
#define MOE_ERR_CUDA 5        /* a CUDA runtime call failed; moe_last_cuda_error() says which */
#define MOE_ERR_DEVICE 6      /* moe_read_status found device error flags */

/* Device status flags (bits of the device status word). */
#define MOE_DEV_ERR_INDEX 0x1   /* an expert id or row index out of range was skipped */
#define MOE_DEV_ERR_TIMEOUT 0x2 /* a bounded pipeline wait gave up; that kernel's output is incomplete */

/* Activation dtypes and expert kinds. */
#define MOE_F32 0
#define MOE_BF16 1
#define MOE_EXPERT_IDENTITY 0 /* Expert_e(x) = x (routing + dispatch + combine only) */
#define MOE_EXPERT_RELU 1     /* relu(x W1) W2 */
#define MOE_EXPERT_SWIGLU 2   /* (silu(x W_gate) * (x W_up)) W_down, silu(z) = z / (1 + e^-z) */

/* Precision of the bf16 expert path (ignored for fp32 activations and identity experts). */
#define MOE_PRECISION_BF16 0    /* h and the expert outputs are each rounded once to bf16 (fewest bytes) */
#define MOE_PRECISION_F32_OUT 1 /* h rounded once to bf16, expert outputs kept in fp32 */
#define MOE_PRECISION_SPLIT_H 2 /* h carried as a bf16 pair (hi = bf16(h), lo = bf16(h - hi)); both halves go
                                   through the down projection against the same weights; expert outputs in
                                   fp32: y then carries essentially only its own final rounding */
#define MOE_PRECISION_FP8_H 3   /* MOE_DISPATCH_FP8_GEMM only: h, as the bf16 value the up projection stores,
                                   quantized per row to e4m3 (one power-of-two scale per row, the rule of the
                                   FP8 rows), and the down projection on tcgen05 kind::f8f6f4 against e4m3 W2
                                   with one scale per output channel (moe_quantize_w2_fp8); expert outputs in
                                   fp32. Needs F % 16 == 0 */

/* What an expert past its capacity drops (capacity >= 0 only). */
#define MOE_DROP_TOKEN_ORDER 0 /* keep the first `capacity` assignments by token index */
#define MOE_DROP_LOW_GATE 1    /* keep the `capacity` assignments with the largest gates, equal gates
                                  to the lower token ("MoE Expert Parallelism Sizing", "Capacity
                                  semantics decide what crosses the wire": drops by selected probability) */

/* Row layout of the dispatched rows. */
#define MOE_LAYOUT_PACKED 0 /* kept rows back to back: expert e's rows are [offsets[e], offsets[e+1]) */
#define MOE_LAYOUT_PADDED 1 /* a fixed segment of `capacity` rows per expert, [e*C, (e+1)*C), the kept rows
                               first and zero rows after ("EP Math", "Capacity factor": a dense
                               [E, C, d] buffer with under-full experts padded); needs capacity >= 0
                               and n_shared == 0. offsets[e] = e*C, so the experts run on all C rows. */

/* Wire format of the dispatched rows. */
#define MOE_DISPATCH_ACT 0 /* rows in the activation dtype */
#define MOE_DISPATCH_FP8 1 /* routed rows as e4m3 codes with one power-of-two fp32 scale per 128-element
                              block ("MoE Expert Parallelism Sizing", "First-order dispatch and combine
                              bytes": FP8 dispatch halves the row, the combine stays wide); the receiving
                              side turns them back into bf16 rows (exact); bf16 activations only */
#define MOE_DISPATCH_FP8_GEMM 2 /* every dispatched row (routed and shared) as e4m3 codes with one
                              power-of-two fp32 scale per row, consumed as they are by an FP8 up
                              projection (tcgen05 kind::f8f6f4: e4m3 x e4m3 products, fp32
                              accumulation) against e4m3 W13 with one power-of-two scale per output
                              channel (moe_quantize_weights_fp8); h, W2 and the down projection stay
                              bf16. One scale per row, not per 128-element block, so that the GEMM can
                              apply it after the K loop. bf16 activations, ReLU or SwiGLU experts,
                              d % 16 == 0; with dedup see moe_dispatch_dedup_fp8_gemm */

/* Limits of this build. */
#define MOE_MAX_K 16        /* experts per token, routed plus shared */
#define MOE_MAX_E 512       /* experts, routed plus shared */

typedef struct moe_config {
    int32_t T;           /* tokens (rows of x), >= 1 */
    int32_t d;           /* hidden size, >= 1 */
    int32_t E;           /* routed experts; E + n_shared <= MOE_MAX_E */
    int32_t k;           /* routed experts kept per token, 1..E; k + n_shared <= MOE_MAX_K */
    int32_t F;           /* expert FFN width (ignored for identity experts) */
    int32_t D;           /* virtual expert-parallel ranks over the routed experts, E % D == 0 (1 = none) */
    int32_t act_dtype;   /* MOE_F32 or MOE_BF16: x, dispatched rows, h, expert outputs, y */
    int32_t expert_kind; /* MOE_EXPERT_* */
    int32_t precision;   /* MOE_PRECISION_*; SPLIT_H needs F % 64 == 0 */
    int32_t n_shared;    /* shared experts S >= 0: experts E..E+S-1, used by every token with gate 1 */
    int64_t capacity;    /* tokens each expert keeps; < 0 = dropless (see moe_capacity) */
    int32_t drop_policy; /* MOE_DROP_* */
    int32_t layout;      /* MOE_LAYOUT_* */
    int32_t n_groups;    /* G: routed experts form G contiguous groups of E/G (used with topk_groups) */
    int32_t topk_groups; /* M: 0 < M < G limits each token to the M groups with the largest best logit
                          * ("MoE Expert Parallelism Sizing", "First-order dispatch and combine
                          * bytes": node-limited / group-limited routing); 0 = no limit. Needs
                          * E % G == 0, G <= 32, k <= M * E / G. */
    int32_t dedup;       /* 1: moe_layer_forward sends each token once per virtual rank (the
                          * deduplicated dispatch, see moe_dispatch_dedup) and fans the send rows
                          * out into the expert rows; D <= 16. 0: rows go straight from x. */
    int32_t dispatch_dtype; /* MOE_DISPATCH_*; the FP8 formats need bf16 activations; with dedup
                             * the deduplicated send rows travel in the FP8 format (see
                             * moe_dispatch_dedup_fp8 and moe_dispatch_dedup_fp8_gemm) */
} moe_config;

/* Where the dispatch writes its routing map (all device int32 arrays). */
typedef struct moe_dispatch_map {
    int32_t* counts_routed; /* [N]   assignments routed to each expert */
    int32_t* counts_kept;   /* [N]   min(counts_routed, capacity) (shared experts: all T) */
    int32_t* offsets;       /* [N+1] rows of expert e are [offsets[e], offsets[e+1]): the exclusive scan of
                             * counts_kept (packed), or e * capacity (padded; the segment's first
                             * counts_kept[e] rows hold assignments, the rest are padding) */
    int32_t* rank_offsets;  /* [D+1] offsets[r*E/D]: virtual rank r's send chunk is [rank_offsets[r], rank_offsets[r+1]) */
    int32_t* pos;           /* [T*K] row of assignment t*K+j, or -1 if it was dropped */
    int32_t* row_src;       /* [rows] assignment t*K+j held by each row (-1 on padding rows); entries
                               [0, offsets[N]) are written; rows = moe_rows_capacity(cfg) */
    int32_t* drop_list;     /* [T*K] dropped assignments, ordered by (expert, token); [0, n_dropped) written */
    int32_t* n_dropped;     /* [1]   number of dropped assignments */
} moe_dispatch_map;

/* Pointers into a moe_layer_forward workspace (all device memory inside it). */
/* The deduplicated send buffer's map (all device int32 arrays). */
typedef struct moe_send_map {
    int32_t* send_counts;  /* [D]   rows sent to virtual rank r: tokens with a kept routed assignment there */
    int32_t* send_offsets; /* [D+1] exclusive scan; send_offsets[D] = rows sent in all */
    int32_t* send_pos;     /* [T*D] send row of (token t, rank r) at t*D + r, or -1 */
    int32_t* send_src;     /* [T*D] t*D + r held by each send row; entries [0, send_offsets[D]) written */
} moe_send_map;

typedef struct moe_workspace_view {
    int32_t* status;     /* device status word (MOE_DEV_* flags) */
    int32_t* topk_idx;   /* [T*K] */
    float* topk_gate;    /* [T*K] */
    moe_dispatch_map map;
    void* xperm;         /* [rows, d] act: dispatched rows (the dispatch "send buffer") */
    void* h;             /* expert hidden activations, see moe_expert_ffn (NULL for identity) */
    void* out;           /* expert outputs, see moe_expert_ffn (aliases xperm for identity); in the
                          * padded layout the forward computes kept rows only and leaves the
                          * padding rows of out unwritten */
    moe_send_map send;   /* cfg->dedup only (NULL pointers otherwise) */
    void* xsend;         /* [T*D, d] act: the deduplicated send buffer (cfg->dedup only); with
                          * an FP8 dispatch dtype it holds the send rows' e4m3 codes [T*D, d] uint8 */
    uint8_t* xq;         /* [rows, d] e4m3 codes of the dispatched rows (MOE_DISPATCH_FP8: routed rows;
                          * MOE_DISPATCH_FP8_GEMM: all rows); with cfg->dedup and MOE_DISPATCH_FP8 the
                          * send rows' codes [T*D, d] (= xsend); NULL for MOE_DISPATCH_ACT */
    float* xscale;       /* their scales: [rows, ceil(d/128)] block scales (MOE_DISPATCH_FP8; with
                          * cfg->dedup [T*D, ceil(d/128)] of the send rows) or [rows] row scales
                          * (MOE_DISPATCH_FP8_GEMM); NULL for MOE_DISPATCH_ACT */
    uint8_t* hq;         /* [rows, F] e4m3 codes of h (MOE_PRECISION_FP8_H only, else NULL) */
    float* hscale;       /* [rows] their row scales (MOE_PRECISION_FP8_H only, else NULL) */
    int32_t* n_near_ties; /* one int the forward's router writes: tokens whose k-th and (k+1)-th
                           * largest selectable fp32 logits differ by less than 1e-6 of the larger
                           * magnitude (a near tie, where another valid rounding of the logits could
                           * select other experts) */
    float* xsend_scale;  /* cfg->dedup with an FP8 dispatch dtype: the send rows' scales,
                          * [T*D, ceil(d/128)] block scales (MOE_DISPATCH_FP8, = xscale) or [T*D]
                          * row scales (MOE_DISPATCH_FP8_GEMM); NULL otherwise */
} moe_workspace_view;

/* ------------------------------------------------------------------ sizing */

/* Per-expert capacity ceil(cf_num * T * k / (cf_den * E)), floored at min_capacity,
 * in exact integer arithmetic ("EP Math", "Capacity factor": C = f T k / E rounded
 * up; "MoE Expert Parallelism Sizing", "Cross-framework notes": a minimum
 * capacity). The capacity factor is cf_num / cf_den. Returns -1 on bad arguments
 * (cf_den <= 0, cf_num < 0, T, k or E <= 0). */
int64_t moe_capacity(int32_t T, int32_t k, int32_t E, int64_t cf_num, int64_t cf_den, int64_t min_capacity);

/* MOE_OK if the config is valid and supported, else the code the entry points would return. */
int moe_validate_config(const moe_config* cfg);

/* Rows of the dispatched-row buffers (xperm, h, out): T*K packed, N*capacity padded
 * (-1 for an invalid config). */
int64_t moe_rows_capacity(const moe_config* cfg);

/* Workspace bytes each entry point needs (0 when cfg is invalid). */
size_t moe_route_workspace_bytes(const moe_config* cfg);
size_t moe_dispatch_workspace_bytes(const moe_config* cfg);
size_t moe_ffn_workspace_bytes(const moe_config* cfg);
size_t moe_workspace_bytes(const moe_config* cfg);      /* moe_layer_forward */
size_t moe_workspace_bytes_host(const moe_config* cfg); /* moe_layer_forward_host */

/* Fill `view` with the buffers moe_layer_forward keeps inside `ws`. Pure host
 * arithmetic on the pointer; touches no memory. */
int moe_workspace_get_view(const moe_config* cfg, void* ws, size_t ws_bytes, moe_workspace_view* view);

/* Number of kernels one moe_layer_forward enqueues for this config. */
int moe_kernels_per_forward(const moe_config* cfg);

/* ------------------------------------------------------------ the hot path */

/* Router: logits H = x W_g (+ bias) in fp32, KeepTopK and the softmax over the kept
 * logits ("Mixture-of-Experts (MoE) Architecture and Expert Parallelism", section 2).
 *   x         [T, d] act dtype
 *   Wg        [d, E] fp32 (the page's W_g in R^{d x E})
 *   bias      [E] fp32 added to every token's logits before KeepTopK, or NULL
 *   topk_idx  [T, K] int32 out: kept experts, slot 0 = largest logit; equal logits
 *             rank the lower expert id first; slots k..K-1 hold the shared experts
 *   topk_gate [T, K] fp32 out: G = exp(H_j - H_max) / sum over kept slots (1 for shared)
 *   ws        scratch of moe_route_workspace_bytes(cfg) bytes: the logits are summed
 *             from split-K partials kept there (and, on the tensor-core path, W_g's
 *             three bf16 terms).
 * Logits are fp32-accurate sums of exact products (x is promoted exactly), summed in a
 * fixed order, so the result is deterministic. For bf16 x and E >= 64 (unless the
 * small-E kernel applies) they come from the tensor cores: W_g is split exactly into
 * three bf16 terms (hi + mid + lo = W_g), each 128-element chunk of d accumulates in a
 * fresh fp32 tensor-memory accumulator, and the chunk sums are added in fp32 in chunk
 * order; otherwise from fp32 FMAs, folded every 256 products. A bounded wait of the
 * tensor-core kernel that gives up ends it early (MOE_DEV_ERR_TIMEOUT in the forward's
 * status word; this stage entry point has no status word). */
int moe_route(const moe_config* cfg, const void* x, const float* Wg, const float* bias,
              int32_t* topk_idx, float* topk_gate, void* ws, size_t ws_bytes, moe_stream_t stream);

/* Dispatch: groups the T*k assignments by expert, keeps `capacity` of each
 * expert's assignments (MOE_DROP_TOKEN_ORDER: the first ones by token;
 * MOE_DROP_LOW_GATE: the largest gates, equal gates by token) and gathers the kept
 * rows of x into `xperm`, in token order inside each expert's segment
 * ("EP Math": "The dispatch all-to-all", "Capacity factor", "Token drop").
 *   x        [T, d] act;  topk_idx [T, K] int32 (ids outside [0, N) are skipped
 *            and flagged MOE_DEV_ERR_INDEX)
 *   topk_gate [T, K] fp32, read only by MOE_DROP_LOW_GATE with a capacity (else may be NULL)
 *   map      output arrays (see moe_dispatch_map)
 *   xperm    [rows, d] act out (rows = moe_rows_capacity(cfg)): row r = x[row_src[r] / K], zero on
 *            padding rows; rows [0, offsets[N]) written. May be NULL when rows is 0.
 *   ws       >= moe_dispatch_workspace_bytes(cfg) bytes; its first 4 bytes are the
 *            device status word, which this call clears first.
 * Bit-exact and deterministic: the result does not depend on scheduling. */
int moe_dispatch(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                 const float* topk_gate, const moe_dispatch_map* map, void* xperm, void* ws,
                 size_t ws_bytes, moe_stream_t stream);

/* Deduplicated dispatch ("MoE Expert Parallelism Sizing", "First-order dispatch and
 * combine bytes", the deduplicated rows: a token crosses to each destination node
 * once). With D virtual ranks (rank r holds routed experts [r E/D, (r+1) E/D)),
 * token t sends its row once to every rank that holds one of its kept routed
 * assignments; send rows are rank-major and in token order inside a rank (rank r's
 * chunk is [send_offsets[r], send_offsets[r+1])). The receiving side then copies
 * each send row to the token's expert rows on that rank; shared experts are
 * replicated, so their rows come from x. The result in xperm equals what
 * moe_dispatch's gather writes.
 *   x        [T, d] act;  topk_idx [T, K] int32;  pos [T*K] int32 from moe_dispatch
 *   map      output arrays (see moe_send_map)
 *   xsend    [T*D, d] act out (rows [0, send_offsets[D]) written)
 *   xperm    [rows, d] act out (rows = moe_rows_capacity(cfg)): the kept assignments' rows
 *   ws       >= moe_dispatch_workspace_bytes(cfg) bytes (cfg->dedup set); its first 4
 *            bytes are the device status word, cleared by this call.
 * Needs 1 <= D <= 16. Bit-exact and deterministic. */
int moe_dispatch_dedup(const moe_config* cfg, const void* x, const int32_t* topk_idx, const int32_t* pos,
                       const moe_send_map* map, void* xsend, void* xperm, void* ws, size_t ws_bytes,
                       moe_stream_t stream);

/* The deduplicated dispatch with FP8 send rows, for cfg->dedup with MOE_DISPATCH_FP8
 * ("MoE Expert Parallelism Sizing", "First-order dispatch and combine bytes": the
 * deduplicated rows, and the FP8 rows with their scale tensors): the same send map as
 * moe_dispatch_dedup, but each send row is the token's row quantized once, per
 * 128-element block, by the rule of moe_dispatch_fp8 (e4m3 codes and a power-of-two
 * scale per block), so the bytes crossing to other ranks are d + 4 * ceil(d/128) per
 * send row. The receiving side turns each kept routed assignment's send row back into
 * bf16 (exactly q * 2^s) as it fans it out into xperm; shared experts' rows come from x.
 * xperm then equals what moe_dispatch_fp8 writes for the same map.
 *   x, topk_idx, pos, map, xperm, ws: as for moe_dispatch_dedup
 *   xsend_q     [T*D, d] uint8 out: the send rows' codes (rows [0, send_offsets[D]) written)
 *   xsend_scale [T*D, ceil(d/128)] fp32 out: their block scales
 * MOE_ERR_ARG unless cfg->dedup and MOE_DISPATCH_FP8 (and then moe_dispatch_dedup
 * rejects the config). Bit-exact and deterministic. */
int moe_dispatch_dedup_fp8(const moe_config* cfg, const void* x, const int32_t* topk_idx, const int32_t* pos,
                           const moe_send_map* map, uint8_t* xsend_q, float* xsend_scale, void* xperm, void* ws,
                           size_t ws_bytes, moe_stream_t stream);

/* The deduplicated dispatch in the FP8 GEMM's format, for cfg->dedup with
 * MOE_DISPATCH_FP8_GEMM (the same pages and passages as moe_dispatch_dedup_fp8): the
 * same send map, each send row the token's row quantized once by the row rule of
 * moe_dispatch_fp8 (e4m3 codes and one power-of-two scale per row: d + 4 bytes per send
 * row). The receiving side copies each kept routed assignment's send-row codes and scale
 * into its expert row of xq / xscale, as they are; shared experts' rows are x quantized by
 * the same rule. xq and xscale then equal what moe_dispatch_fp8 writes for the same map,
 * and feed moe_expert_ffn_fp8.
 *   x, topk_idx, pos, map, ws: as for moe_dispatch_dedup
 *   xsend_q     [T*D, d] uint8 out: the send rows' codes (rows [0, send_offsets[D]) written)
 *   xsend_scale [T*D] fp32 out: their row scales
 *   xq          [rows, d] uint8 out, xscale [rows] fp32 out: the expert rows' codes and scales
 *               (may be NULL when rows = moe_rows_capacity(cfg) is 0)
 * MOE_ERR_ARG unless cfg->dedup and MOE_DISPATCH_FP8_GEMM. Bit-exact and deterministic. */
int moe_dispatch_dedup_fp8_gemm(const moe_config* cfg, const void* x, const int32_t* topk_idx, const int32_t* pos,
                                const moe_send_map* map, uint8_t* xsend_q, float* xsend_scale, uint8_t* xq,
                                float* xscale, void* ws, size_t ws_bytes, moe_stream_t stream);

/* FP8 dispatch of the rows a moe_dispatch with the same cfg mapped (its pos, row_src
 * and offsets).
 * MOE_DISPATCH_FP8: each token row is quantized once, per 128-element block, to e4m3 codes
 * with the scale 2^s, s the smallest integer with amax/2^s <= 448 (round to nearest,
 * ties to even, sign kept), and written to each of its kept routed rows
 * ("MoE Expert Parallelism Sizing", "First-order dispatch and combine bytes": the
 * FP8 dispatch row with its scale tensors). Shared experts are replicated: their rows
 * are copied from x into xperm. With xperm non-NULL the receiving side also turns the
 * routed rows back into bf16 (exactly q * 2^s).
 *   x       [T, d] bf16;  topk_idx [T, K];  map: pos, row_src and offsets from moe_dispatch
 *   xq      [rows, d] uint8 out;  xscale [rows, ceil(d/128)] fp32 out (rows = moe_rows_capacity)
 *   xperm   [rows, d] bf16 out, or NULL (shared rows then need a moe_dispatch gather)
 *   ws      >= moe_dispatch_workspace_bytes(cfg); its first 4 bytes are the status word,
 *           cleared by this call.
 * MOE_DISPATCH_FP8_GEMM: the same rule over the whole row (one scale 2^s per token row),
 * and every kept row, routed or shared, receives the codes: xq [rows, d] uint8 and
 * xscale [rows] fp32 out; xperm must be NULL (the FP8 up projection reads xq as it is).
 * Needs one of the two FP8 dispatch dtypes. Bit-exact and deterministic. */
int moe_dispatch_fp8(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                     const moe_dispatch_map* map, uint8_t* xq, float* xscale, void* xperm, void* ws,
                     size_t ws_bytes, moe_stream_t stream);

/* Grouped expert FFN over the dispatched rows: for each expert e, rows
 * [offsets[e], offsets[e+1]) of xperm go through Expert_e ("EP Math", "What expert
 * parallelism actually shards": every expert is a complete FFN with private weights).
 *   xperm   [rows, d] act;  offsets [N+1] int32 (from moe_dispatch), offsets[N] <= rows.
 *           xperm, h and out may be NULL when rows (moe_rows_capacity) is 0.
 *   W13     SwiGLU: [N, 2F, d] act, rows [0,F) = W_gate^T, rows [F,2F) = W_up^T;
 *           ReLU:   [N, F, d]  act (W1^T).   (The usual linear-layer layout.)
 *   W2      [N, d, F] act (W_down^T / W2^T)
 *   h       out: hidden activation of each row, [rows, F] act; under MOE_PRECISION_SPLIT_H
 *           [rows, 2F] bf16: for every 64-column block b of h the 64 "hi" values at
 *           columns [128b, 128b+64) and the 64 "lo" values at [128b+64, 128b+128).
 *   out     out: expert output of each row, [rows, d]; fp32 under MOE_PRECISION_F32_OUT
 *           and MOE_PRECISION_SPLIT_H with bf16 activations, else the act dtype.
 * bf16 runs on the tensor cores (bf16 x bf16 products, fp32 accumulation); fp32
 * runs on the fp32 FMA units. Requires F * sizeof(act) % 16 == 0 besides the row
 * rule. ws >= moe_ffn_workspace_bytes(cfg); its first 4 bytes are the status word
 * (cleared). With bf16 experts it also holds the tickets (cleared on every call) and
 * fp32 partial slots of the split over k: when the tiles of a swapped-pair projection
 * without SwiGLU leave their last wave of SM pairs at most half busy, each tile of that
 * wave is cut into up to 4 ranges of k that run on idle pairs, and the range that
 * finishes last sums the ranges' partials in range order (deterministic; the sums are
 * associated differently from an uncut tile's). A MOE_DISPATCH_FP8_GEMM config takes
 * moe_expert_ffn_fp8 instead (MOE_ERR_ARG here). */
int moe_expert_ffn(const moe_config* cfg, const void* xperm, const int32_t* offsets,
                   const void* W13, const void* W2, void* h, void* out,
                   void* ws, size_t ws_bytes, moe_stream_t stream);

/* Bytes of the FP8 up-projection weights of a MOE_DISPATCH_FP8_GEMM config: the e4m3
 * codes of W13 ([N, R, d] uint8, R = 2F for SwiGLU, F for ReLU), then, at the next
 * 256-byte boundary, one fp32 scale per weight row ([N, R]). 0 for other configs. */
size_t moe_fp8_weight_bytes(const moe_config* cfg);

/* Quantizes the bf16 W13 [N, R, d] (layout as in moe_expert_ffn) into that buffer:
 * each weight row (one output channel) gets the scale 2^s, s the smallest integer with
 * amax/2^s <= 448, and the codes round(w / 2^s) to the nearest e4m3 value (ties to
 * even, sign kept). W13_fp8 holds moe_fp8_weight_bytes(cfg) bytes, 16-byte aligned.
 * Needs cfg->dispatch_dtype == MOE_DISPATCH_FP8_GEMM. Bit-exact and deterministic. */
int moe_quantize_weights_fp8(const moe_config* cfg, const void* W13, void* W13_fp8, moe_stream_t stream);

/* Bytes of the FP8 down-projection weights of a MOE_PRECISION_FP8_H config: the e4m3
 * codes of W2 ([N, d, F] uint8), then, at the next 256-byte boundary, one fp32 scale per
 * row of W2 (output channel, [N, d]). 0 for other configs. */
size_t moe_fp8_w2_bytes(const moe_config* cfg);

/* Quantizes the bf16 W2 [N, d, F] into that buffer, each row (output channel) by the
 * rule of moe_quantize_weights_fp8. Needs cfg->precision == MOE_PRECISION_FP8_H.
 * Bit-exact and deterministic. */
int moe_quantize_w2_fp8(const moe_config* cfg, const void* W2, void* W2_fp8, moe_stream_t stream);

/* moe_expert_ffn for a MOE_DISPATCH_FP8_GEMM config: the up projection runs on the
 * e4m3 rows and weights (tcgen05 kind::f8f6f4 on SM pairs), its fp32 accumulator
 * multiplied by the row scale and the weight row's scale before the activation; h is
 * stored as for moe_expert_ffn (bf16, or a hi/lo pair under MOE_PRECISION_SPLIT_H) and
 * the down projection is the bf16 one.
 *   xq      [rows, d] uint8 e4m3 codes;  xscale [rows] fp32 row scales (moe_dispatch_fp8)
 *   W13_fp8 moe_quantize_weights_fp8's buffer;  W2 [N, d, F] bf16, or under MOE_PRECISION_FP8_H
 *           moe_quantize_w2_fp8's buffer (h is then quantized per row between the two GEMMs)
 *   offsets, h, out as in moe_expert_ffn;  ws >= moe_ffn_workspace_bytes(cfg) (under
 *   MOE_PRECISION_FP8_H it also holds h's codes and scales). */
int moe_expert_ffn_fp8(const moe_config* cfg, const uint8_t* xq, const float* xscale, const int32_t* offsets,
                       const void* W13_fp8, const void* W2, void* h, void* out, void* ws, size_t ws_bytes,
                       moe_stream_t stream);

/* Combine: y[t] = sum over slots j < K with pos[t*K+j] >= 0 of topk_gate[t*K+j] * out[pos[t*K+j]],
 * with `out` in the dtype moe_expert_ffn writes (see there; the activation dtype for
 * identity experts),
 * summed in fp32 in slot order and rounded once ("Mixture-of-Experts (MoE)
 * Architecture and Expert Parallelism", section 2; "EP Math", "The combine
 * all-to-all"; "Token drop": a dropped slot adds nothing and the gates are not
 * renormalised). A row index >= rows is skipped and flagged in `status` if
 * status is not NULL. Deterministic, no atomics.
 *   out [rows, d]; topk_gate [T, K] fp32; pos [T, K] int32; y [T, d] act out. */
int moe_combine(const moe_config* cfg, const void* out, const float* topk_gate,
                const int32_t* pos, void* y, int32_t* status, moe_stream_t stream);

/* The whole layer: route, dispatch, expert FFN, combine. Intermediates live in ws
 * (layout: moe_workspace_get_view). ws >= moe_workspace_bytes(cfg); the status word
 * is cleared at the start. W13/W2 may be NULL for identity experts. Under
 * MOE_DISPATCH_FP8_GEMM, W13 is moe_quantize_weights_fp8's buffer, and under
 * MOE_PRECISION_FP8_H W2 is moe_quantize_w2_fp8's. y [T, d] act. */
int moe_layer_forward(const moe_config* cfg, const void* x, const float* Wg, const float* bias,
                      const void* W13, const void* W2, void* y, void* ws, size_t ws_bytes,
                      moe_stream_t stream);

/* moe_layer_forward that also records CUDA events between its stages, for timing:
 * events[0] before the router, [1] after it, [2] after the dispatch, [3] after the
 * expert up-projection, [4] after the down-projection, [5] after the combine
 * (for identity experts [3] and [4] are recorded right after [2]). `events` holds
 * cudaEvent_t handles; n_events >= 6 (the first 6 are used). */
int moe_layer_forward_traced(const moe_config* cfg, const void* x, const float* Wg,
                             const float* bias, const void* W13, const void* W2, void* y,
                             void* ws, size_t ws_bytes, moe_stream_t stream,
                             void* const* events, int32_t n_events);

/* The whole layer from and to host memory: copies x_host into the workspace,
 * runs moe_layer_forward, copies y back into y_host, all on `stream`, and
 * synchronises the stream before returning (so y_host is ready). x_host and
 * y_host should be page-locked for asynchronous copies. ws >=
 * moe_workspace_bytes_host(cfg). The weights stay device pointers. */
int moe_layer_forward_host(const moe_config* cfg, const void* x_host, const float* Wg,
                           const float* bias, const void* W13, const void* W2, void* y_host,
                           void* ws, size_t ws_bytes, moe_stream_t stream);

/* moe_layer_forward_host without the final synchronisation: the copy in, the layer and
 * the copy out are enqueued on `stream` and the call returns; y_host is ready once the
 * stream reaches that point (cudaStreamSynchronize, or an event). With page-locked
 * host buffers the copies run on the copy engines, so a caller that keeps two batches
 * in flight on two streams (each with its own workspace and y_host) overlaps one
 * batch's copies with the other's kernels. Same arguments as moe_layer_forward_host. */
int moe_layer_forward_host_async(const moe_config* cfg, const void* x_host, const float* Wg,
                                 const float* bias, const void* W13, const void* W2, void* y_host,
                                 void* ws, size_t ws_bytes, moe_stream_t stream);

/* moe_dispatch without a workspace, for callers that cannot give the library device
 * memory for scratch: for example a serving loop that must not allocate device
 * memory once it runs (cudaMalloc can synchronise the device and stall a step), or a
 * plugin whose host framework owns every device buffer and passes in only the
 * tensors. The pages have no counterpart of this entry point; it exists for such
 * callers.
 *
 * Same arguments, outputs and results as moe_dispatch, minus ws/ws_bytes. Its
 * scratch (histogram and offsets, 4 * (N * ceil(T*K/256) + 2N + 1) bytes, plus 8*T*K
 * under MOE_DROP_LOW_GATE, plus a small header) lives in one device array of
 * MOE_STATIC_SCRATCH_BYTES inside the
 * library, which every GPU that loads the library keeps until the process exits.
 * The call allocates nothing (no cudaMalloc, no cudaFree, no allocating library
 * routine) and returns MOE_ERR_WORKSPACE when a config needs more scratch than that.
 * The first call in each device context looks up the array's device address there
 * (cudaGetSymbolAddress, with the device current): once per device, and once more if
 * cudaDeviceReset re-creates the device's context; make that first call before any
 * stream capture. All calls share the one array: calls that may overlap on the GPU
 * (other streams, other threads) race and must be serialised by the caller. Expert
 * ids outside [0, E) are skipped, as in moe_dispatch, but there is no status word to
 * report them through. */
#define MOE_STATIC_SCRATCH_BYTES (1u << 20)
int moe_dispatch_static(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                        const float* topk_gate, const moe_dispatch_map* map, void* xperm,
                        moe_stream_t stream);

/* ----------------------------------------------------------- diagnostics */

/* Synchronises `stream`, copies the status word at `status_dev` to *flags_host
 * (may be NULL) and returns MOE_OK if it is zero, MOE_ERR_DEVICE otherwise.
 * For diagnostics, not for the hot path. */
int moe_read_status(const int32_t* status_dev, int32_t* flags_host, moe_stream_t stream);

/* Human-readable text of a return code. */
const char* moe_status_string(int code);

/* Text of the last CUDA error this thread saw inside the library ("" if none). */
const char* moe_last_cuda_error(void);

/* Name of the kernel moe_expert_ffn / moe_layer_forward run for this config's
 * expert GEMMs ("" for identity experts or an invalid config): the fp32 FMA
 * kernel, or one of the three tcgen05 variants (one SM per 128x256 tile, SM pairs
 * on 256-row tiles, SM pairs with swapped operands); under MOE_DISPATCH_FP8_GEMM the
 * e4m3 swapped-pair kernel of the up projection. The environment variable
 * MOE_GEMM_PAIR=0/1/2 forces a bf16 tcgen05 variant. Static storage; never freed. */
const char* moe_ffn_kernel_name(const moe_config* cfg);

/* Environment switches (read once per process):
 *   MOE_GEMM_PAIR=0/1/2    force the tcgen05 expert-GEMM variant (see moe_ffn_kernel_name);
 *   MOE_GEMM_SPLITK=0      never split the expert GEMMs' last partial wave over k (see
 *                          moe_expert_ffn), for comparisons;
 *   MOE_ROUTE_TC=0         keep the router's logits on the FMA units for every config;
 *   MOE_ROUTE_TC_CHUNK=n   elements of d per fresh accumulator on the tensor-core router
 *                          (a multiple of 64; default 128), for accuracy experiments;
 *   MOE_DEBUG_SKIP_ARRIVE=1 failure-path test only: the grouped GEMMs leave their first
 *                          finished accumulator unsignalled, so their bounded wait runs
 *                          out (2 s) and MOE_DEV_ERR_TIMEOUT is set in the status word;
 *                          the kernels drain, free tensor memory and return. */

/* Library version, major * 10000 + minor * 100 + patch. */
int moe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */
