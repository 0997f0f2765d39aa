"""Thin ctypes binding of libmoe.so (include/moe.h), same names as the C entry points.

Argument marshalling only: tensors become device pointers, the current torch CUDA
stream becomes the cudaStream_t, non-zero return codes become MoeError. Every step
of the layer runs in the library's CUDA kernels; there is no fallback, and loading
fails loudly when the shared library has not been built.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from fractions import Fraction

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "moe.h")

MOE_OK, MOE_ERR_ARG, MOE_ERR_ALIGN, MOE_ERR_WORKSPACE = 0, 1, 2, 3
MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_DEVICE = 4, 5, 6
MOE_DEV_ERR_INDEX, MOE_DEV_ERR_TIMEOUT = 0x1, 0x2
MOE_F32, MOE_BF16 = 0, 1
MOE_EXPERT_IDENTITY, MOE_EXPERT_RELU, MOE_EXPERT_SWIGLU = 0, 1, 2
MOE_PRECISION_BF16, MOE_PRECISION_F32_OUT, MOE_PRECISION_SPLIT_H, MOE_PRECISION_FP8_H = 0, 1, 2, 3
PRECISIONS = {"bf16": MOE_PRECISION_BF16, "f32_out": MOE_PRECISION_F32_OUT, "split_h": MOE_PRECISION_SPLIT_H,
              "fp8_h": MOE_PRECISION_FP8_H}
MOE_DROP_TOKEN_ORDER, MOE_DROP_LOW_GATE = 0, 1
DROP_POLICIES = {"token": MOE_DROP_TOKEN_ORDER, "gate": MOE_DROP_LOW_GATE}
MOE_LAYOUT_PACKED, MOE_LAYOUT_PADDED = 0, 1
LAYOUTS = {"packed": MOE_LAYOUT_PACKED, "padded": MOE_LAYOUT_PADDED}
MOE_DISPATCH_ACT, MOE_DISPATCH_FP8, MOE_DISPATCH_FP8_GEMM = 0, 1, 2
DISPATCH_DTYPES = {"act": MOE_DISPATCH_ACT, "fp8": MOE_DISPATCH_FP8, "fp8_gemm": MOE_DISPATCH_FP8_GEMM}
MOE_MAX_K, MOE_MAX_E = 16, 512
EXPERT_KINDS = {"identity": MOE_EXPERT_IDENTITY, "relu": MOE_EXPERT_RELU, "swiglu": MOE_EXPERT_SWIGLU}
ACT_DTYPES = {"f32": MOE_F32, "bf16": MOE_BF16}

_p = ctypes.c_void_p
_i32, _i64, _sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str, detail: str = ""):
        self.code = code
        msg = f"{where}: {status_string(code)} (code {code})"
        if detail:
            msg += f": {detail}"
        super().__init__(msg)


class moe_config(ctypes.Structure):
    _fields_ = [("T", _i32), ("d", _i32), ("E", _i32), ("k", _i32), ("F", _i32), ("D", _i32),
                ("act_dtype", _i32), ("expert_kind", _i32), ("precision", _i32), ("n_shared", _i32),
                ("capacity", _i64), ("drop_policy", _i32), ("layout", _i32), ("n_groups", _i32),
                ("topk_groups", _i32), ("dedup", _i32), ("dispatch_dtype", _i32)]


class moe_dispatch_map(ctypes.Structure):
    _fields_ = [(n, _p) for n in ("counts_routed", "counts_kept", "offsets", "rank_offsets", "pos",
                                  "row_src", "drop_list", "n_dropped")]


class moe_send_map(ctypes.Structure):
    _fields_ = [(n, _p) for n in ("send_counts", "send_offsets", "send_pos", "send_src")]


class moe_workspace_view(ctypes.Structure):
    _fields_ = [("status", _p), ("topk_idx", _p), ("topk_gate", _p), ("map", moe_dispatch_map),
                ("xperm", _p), ("h", _p), ("out", _p), ("send", moe_send_map), ("xsend", _p), ("xq", _p),
                ("xscale", _p), ("hq", _p), ("hscale", _p), ("n_near_ties", _p), ("xsend_scale", _p)]


_SIGNATURES = {
    "moe_capacity": (_i64, [_i32, _i32, _i32, _i64, _i64, _i64]),
    "moe_validate_config": (ctypes.c_int, [ctypes.POINTER(moe_config)]),
    "moe_rows_capacity": (_i64, [ctypes.POINTER(moe_config)]),
    "moe_dispatch_workspace_bytes": (_sz, [ctypes.POINTER(moe_config)]),
    "moe_ffn_workspace_bytes": (_sz, [ctypes.POINTER(moe_config)]),
    "moe_workspace_bytes": (_sz, [ctypes.POINTER(moe_config)]),
    "moe_workspace_bytes_host": (_sz, [ctypes.POINTER(moe_config)]),
    "moe_workspace_get_view": (ctypes.c_int, [ctypes.POINTER(moe_config), _p, _sz, ctypes.POINTER(moe_workspace_view)]),
    "moe_kernels_per_forward": (ctypes.c_int, [ctypes.POINTER(moe_config)]),
    "moe_route_workspace_bytes": (_sz, [ctypes.POINTER(moe_config)]),
    "moe_route": (ctypes.c_int, [ctypes.POINTER(moe_config), _p, _p, _p, _p, _p, _p, _sz, _p]),
    "moe_dispatch": (ctypes.c_int, [ctypes.POINTER(moe_config), _p, _p, _p, ctypes.POINTER(moe_dispatch_map), _p, _p,
                                    _sz, _p]),
    "moe_expert_ffn": (ctypes.c_int, [ctypes.POINTER(moe_config), _p, _p, _p, _p, _p, _p, _p, _sz, _p]),
    "moe_combine": (ctypes.c_int, [ctypes.POINTER(moe_config), _p, _p, _p, _p, _p, _p]),
    "moe_layer_forward": (ctypes.c_int, [ctypes.POINTER(moe_config), _p, _p, _p, _p, _p, _p, _p, _sz, _p]),
    "moe_layer_forward_traced": (ctypes.c_int, [ctypes.POINTER(moe_config), _p, _p, _p, _p, _p, _p, _p, _sz, _p,
                                                ctypes.POINTER(_p), _i32]),
    "moe_layer_forward_host": (ctypes.c_int, [ctypes.POINTER(moe_config), _p, _p, _p, _p, _p, _p, _p, _sz, _p]),
    "moe_layer_forward_host_async": (ctypes.c_int, [ctypes.POINTER(moe_config), _p, _p, _p, _p, _p, _p, _p, _sz,
                                                    _p]),
    "moe_dispatch_dedup": (ctypes.c_int, [ctypes.POINTER(moe_config), _p, _p, _p, ctypes.POINTER(moe_send_map), _p,
                                          _p, _p, _sz, _p]),
    "moe_dispatch_dedup_fp8": (ctypes.c_int, [ctypes.POINTER(moe_config), _p, _p, _p, ctypes.POINTER(moe_send_map),
                                              _p, _p, _p, _p, _sz, _p]),
    "moe_dispatch_dedup_fp8_gemm": (ctypes.c_int, [ctypes.POINTER(moe_config), _p, _p, _p,
                                                   ctypes.POINTER(moe_send_map), _p, _p, _p, _p, _p, _sz, _p]),
    "moe_dispatch_fp8": (ctypes.c_int, [ctypes.POINTER(moe_config), _p, _p, ctypes.POINTER(moe_dispatch_map), _p,
                                        _p, _p, _p, _sz, _p]),
    "moe_fp8_weight_bytes": (_sz, [ctypes.POINTER(moe_config)]),
    "moe_quantize_weights_fp8": (ctypes.c_int, [ctypes.POINTER(moe_config), _p, _p, _p]),
    "moe_fp8_w2_bytes": (_sz, [ctypes.POINTER(moe_config)]),
    "moe_quantize_w2_fp8": (ctypes.c_int, [ctypes.POINTER(moe_config), _p, _p, _p]),
    "moe_expert_ffn_fp8": (ctypes.c_int, [ctypes.POINTER(moe_config), _p, _p, _p, _p, _p, _p, _p, _p, _sz, _p]),
    "moe_dispatch_static": (ctypes.c_int, [ctypes.POINTER(moe_config), _p, _p, _p, ctypes.POINTER(moe_dispatch_map),
                                           _p, _p]),
    "moe_read_status": (ctypes.c_int, [_p, ctypes.POINTER(_i32), _p]),
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_last_cuda_error": (ctypes.c_char_p, []),
    "moe_version": (ctypes.c_int, []),
    "moe_ffn_kernel_name": (ctypes.c_char_p, [ctypes.POINTER(moe_config)]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded shared library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m routing_dispatch_combine_moe_b300.build`")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def status_string(code: int) -> str:
    return lib().moe_status_string(code).decode()


def _check(code: int, where: str):
    if code != MOE_OK:
        detail = lib().moe_last_cuda_error().decode() if code == MOE_ERR_CUDA else ""
        raise MoeError(code, where, detail)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


# ------------------------------------------------------------------ config
def make_config(T, d, E, k, F=0, D=1, act="bf16", expert="swiglu", capacity=None, precision="f32_out",
                n_shared=0, drop_policy="token", layout="packed", n_groups=0, topk_groups=0,
                dedup=False, dispatch_dtype="act") -> moe_config:
    """A moe_config; ``capacity`` None (dropless) or a non-negative integer."""
    return moe_config(T=T, d=d, E=E, k=k, F=F, D=D, act_dtype=ACT_DTYPES[act],
                      expert_kind=EXPERT_KINDS[expert], precision=PRECISIONS[precision], n_shared=n_shared,
                      capacity=-1 if capacity is None else int(capacity),
                      drop_policy=DROP_POLICIES[drop_policy], layout=LAYOUTS[layout], n_groups=n_groups,
                      topk_groups=topk_groups, dedup=int(bool(dedup)),
                      dispatch_dtype=DISPATCH_DTYPES[dispatch_dtype])


def out_dtype(cfg) -> torch.dtype:
    """dtype of the expert-output rows moe_expert_ffn writes for this config."""
    if cfg.act_dtype == MOE_F32:
        return torch.float32
    if cfg.expert_kind != MOE_EXPERT_IDENTITY and cfg.precision != MOE_PRECISION_BF16:
        return torch.float32
    return torch.bfloat16


def hidden_cols(cfg) -> int:
    """Columns of the h buffer moe_expert_ffn writes (2F in the split-h bf16 mode)."""
    if cfg.act_dtype == MOE_BF16 and cfg.precision == MOE_PRECISION_SPLIT_H:
        return 2 * cfg.F
    return cfg.F


def moe_capacity(T, k, E, capacity_factor, min_capacity=0) -> int:
    f = Fraction(capacity_factor)
    c = lib().moe_capacity(T, k, E, f.numerator, f.denominator, min_capacity)
    if c < 0:
        raise MoeError(MOE_ERR_ARG, "moe_capacity")
    return int(c)


def config_for(w, capacity="auto") -> moe_config:
    """moe_config of a workload (see workloads.Workload)."""
    if capacity == "auto":
        capacity = None if w.capacity_factor is None else moe_capacity(w.T, w.k, w.E, w.capacity_factor,
                                                                       w.min_capacity)
    return make_config(w.T, w.d, w.E, w.k, w.F, w.D, w.act, w.expert, capacity, w.precision, w.n_shared,
                       w.drop_policy, w.layout, w.n_groups, w.topk_groups, w.dedup, w.dispatch_dtype)


def moe_validate_config(cfg) -> int:
    return lib().moe_validate_config(ctypes.byref(cfg))


def moe_rows_capacity(cfg) -> int:
    """Rows of the dispatched-row buffers (xperm, h, out, row_src) for this config."""
    r = lib().moe_rows_capacity(ctypes.byref(cfg))
    if r < 0:
        raise MoeError(moe_validate_config(cfg), "moe_rows_capacity")
    return int(r)


def moe_workspace_bytes(cfg) -> int:
    return lib().moe_workspace_bytes(ctypes.byref(cfg))


def moe_workspace_bytes_host(cfg) -> int:
    return lib().moe_workspace_bytes_host(ctypes.byref(cfg))


def moe_dispatch_workspace_bytes(cfg) -> int:
    return lib().moe_dispatch_workspace_bytes(ctypes.byref(cfg))


def moe_ffn_workspace_bytes(cfg) -> int:
    return lib().moe_ffn_workspace_bytes(ctypes.byref(cfg))


def moe_kernels_per_forward(cfg) -> int:
    return lib().moe_kernels_per_forward(ctypes.byref(cfg))


def workspace(cfg, device="cuda", host=False) -> torch.Tensor:
    """A uint8 device tensor of the workspace size (memory from torch's allocator)."""
    n = moe_workspace_bytes_host(cfg) if host else moe_workspace_bytes(cfg)
    if n == 0:
        _check(moe_validate_config(cfg), "workspace")
    return torch.empty(n, dtype=torch.uint8, device=device)


@dataclass
class WorkspaceView:
    status: int
    topk_idx: int
    topk_gate: int
    counts_routed: int
    counts_kept: int
    offsets: int
    rank_offsets: int
    pos: int
    row_src: int
    drop_list: int
    n_dropped: int
    xperm: int
    h: int | None
    out: int
    send_counts: int | None = None
    send_offsets: int | None = None
    send_pos: int | None = None
    send_src: int | None = None
    xsend: int | None = None
    xq: int | None = None
    xscale: int | None = None
    hq: int | None = None
    hscale: int | None = None
    n_near_ties: int | None = None
    xsend_scale: int | None = None


def moe_workspace_get_view(cfg, ws: torch.Tensor) -> WorkspaceView:
    v = moe_workspace_view()
    _check(lib().moe_workspace_get_view(ctypes.byref(cfg), _ptr(ws), ws.numel(), ctypes.byref(v)),
           "moe_workspace_get_view")
    m = v.map
    sm = v.send
    return WorkspaceView(v.status, v.topk_idx, v.topk_gate, m.counts_routed, m.counts_kept, m.offsets,
                         m.rank_offsets, m.pos, m.row_src, m.drop_list, m.n_dropped, v.xperm, v.h, v.out,
                         sm.send_counts, sm.send_offsets, sm.send_pos, sm.send_src, v.xsend, v.xq, v.xscale,
                         v.hq, v.hscale, v.n_near_ties, v.xsend_scale)


# ------------------------------------------------------------------ hot path
def moe_route_workspace_bytes(cfg) -> int:
    return lib().moe_route_workspace_bytes(ctypes.byref(cfg))


def moe_route(cfg, x, Wg, bias, topk_idx, topk_gate, ws=None, stream=None):
    """``ws``: a uint8 device tensor of moe_route_workspace_bytes(cfg) bytes (None when that is 0)."""
    n = 0 if ws is None else ws.numel()
    _check(lib().moe_route(ctypes.byref(cfg), _ptr(x), _ptr(Wg), _ptr(bias), _ptr(topk_idx), _ptr(topk_gate),
                           _ptr(ws), n, _stream(stream)), "moe_route")


def dispatch_map(counts_routed, counts_kept, offsets, rank_offsets, pos, row_src, drop_list, n_dropped):
    return moe_dispatch_map(*[_ptr(t) for t in (counts_routed, counts_kept, offsets, rank_offsets, pos, row_src,
                                                drop_list, n_dropped)])


def moe_dispatch(cfg, x, topk_idx, dmap: moe_dispatch_map, xperm, ws, stream=None, topk_gate=None):
    """``topk_gate`` is read only by the gate drop policy with a capacity."""
    _check(lib().moe_dispatch(ctypes.byref(cfg), _ptr(x), _ptr(topk_idx), _ptr(topk_gate), ctypes.byref(dmap),
                              _ptr(xperm), _ptr(ws), ws.numel(), _stream(stream)), "moe_dispatch")


def send_map(send_counts, send_offsets, send_pos, send_src):
    return moe_send_map(*[_ptr(t) for t in (send_counts, send_offsets, send_pos, send_src)])


def moe_dispatch_dedup(cfg, x, topk_idx, pos, smap: moe_send_map, xsend, xperm, ws, stream=None):
    """Deduplicated send buffer (one row per token and destination rank) and its fan-out into xperm."""
    _check(lib().moe_dispatch_dedup(ctypes.byref(cfg), _ptr(x), _ptr(topk_idx), _ptr(pos), ctypes.byref(smap),
                                    _ptr(xsend), _ptr(xperm), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_dispatch_dedup")


def moe_dispatch_dedup_fp8(cfg, x, topk_idx, pos, smap: moe_send_map, xsend_q, xsend_scale, xperm, ws, stream=None):
    """Deduplicated send buffer as e4m3 codes + per-128 block scales, dequantized into xperm by the fan-out."""
    _check(lib().moe_dispatch_dedup_fp8(ctypes.byref(cfg), _ptr(x), _ptr(topk_idx), _ptr(pos), ctypes.byref(smap),
                                        _ptr(xsend_q), _ptr(xsend_scale), _ptr(xperm), _ptr(ws), ws.numel(),
                                        _stream(stream)), "moe_dispatch_dedup_fp8")


def moe_dispatch_dedup_fp8_gemm(cfg, x, topk_idx, pos, smap: moe_send_map, xsend_q, xsend_scale, xq, xscale, ws,
                                stream=None):
    """Deduplicated send buffer as e4m3 codes + one scale per row; the fan-out copies them into
    the expert rows' xq / xscale (the FP8 GEMM's input)."""
    _check(lib().moe_dispatch_dedup_fp8_gemm(ctypes.byref(cfg), _ptr(x), _ptr(topk_idx), _ptr(pos),
                                             ctypes.byref(smap), _ptr(xsend_q), _ptr(xsend_scale), _ptr(xq),
                                             _ptr(xscale), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_dispatch_dedup_fp8_gemm")


def moe_dispatch_fp8(cfg, x, topk_idx, dmap: moe_dispatch_map, xq, xscale, xperm, ws, stream=None):
    """FP8 (e4m3, power-of-two scales per 128-element block, or per row for "fp8_gemm")
    rows of a moe_dispatch map; xperm may be None (and must be for "fp8_gemm")."""
    _check(lib().moe_dispatch_fp8(ctypes.byref(cfg), _ptr(x), _ptr(topk_idx), ctypes.byref(dmap), _ptr(xq),
                                  _ptr(xscale), _ptr(xperm), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_dispatch_fp8")


def moe_dispatch_static(cfg, x, topk_idx, dmap: moe_dispatch_map, xperm, stream=None, topk_gate=None):
    """moe_dispatch with the library's built-in scratch array (no workspace argument)."""
    _check(lib().moe_dispatch_static(ctypes.byref(cfg), _ptr(x), _ptr(topk_idx), _ptr(topk_gate),
                                     ctypes.byref(dmap), _ptr(xperm), _stream(stream)), "moe_dispatch_static")


def moe_expert_ffn(cfg, xperm, offsets, W13, W2, h, out, ws, stream=None):
    _check(lib().moe_expert_ffn(ctypes.byref(cfg), _ptr(xperm), _ptr(offsets), _ptr(W13), _ptr(W2), _ptr(h),
                                _ptr(out), _ptr(ws), ws.numel(), _stream(stream)), "moe_expert_ffn")


def moe_fp8_weight_bytes(cfg) -> int:
    """Bytes of the FP8 W13 buffer of an "fp8_gemm" config (codes, then row scales)."""
    return lib().moe_fp8_weight_bytes(ctypes.byref(cfg))


def moe_quantize_weights_fp8(cfg, W13, W13_fp8, stream=None):
    _check(lib().moe_quantize_weights_fp8(ctypes.byref(cfg), _ptr(W13), _ptr(W13_fp8), _stream(stream)),
           "moe_quantize_weights_fp8")


def fp8_weights(cfg, W13, stream=None) -> torch.Tensor:
    """The FP8 W13 buffer (uint8, on W13's device) of an "fp8_gemm" config."""
    q = torch.empty(moe_fp8_weight_bytes(cfg), dtype=torch.uint8, device=W13.device)
    moe_quantize_weights_fp8(cfg, W13, q, stream)
    return q


def fp8_weight_parts(cfg, W13_fp8, N: int, R: int, d: int):
    """Views of an FP8 W13 buffer: codes [N, R, d] uint8 and row scales [N, R] fp32."""
    n = N * R * d
    off = (n + 255) // 256 * 256
    return W13_fp8[:n].view(N, R, d), W13_fp8[off:off + 4 * N * R].view(torch.float32).view(N, R)


def moe_fp8_w2_bytes(cfg) -> int:
    """Bytes of the FP8 W2 buffer of an "fp8_h" config (codes, then row scales)."""
    return lib().moe_fp8_w2_bytes(ctypes.byref(cfg))


def moe_quantize_w2_fp8(cfg, W2, W2_fp8, stream=None):
    _check(lib().moe_quantize_w2_fp8(ctypes.byref(cfg), _ptr(W2), _ptr(W2_fp8), _stream(stream)),
           "moe_quantize_w2_fp8")


def fp8_w2(cfg, W2, stream=None) -> torch.Tensor:
    """The FP8 W2 buffer (uint8, on W2's device) of an "fp8_h" config."""
    q = torch.empty(moe_fp8_w2_bytes(cfg), dtype=torch.uint8, device=W2.device)
    moe_quantize_w2_fp8(cfg, W2, q, stream)
    return q


def moe_expert_ffn_fp8(cfg, xq, xscale, offsets, W13_fp8, W2, h, out, ws, stream=None):
    _check(lib().moe_expert_ffn_fp8(ctypes.byref(cfg), _ptr(xq), _ptr(xscale), _ptr(offsets), _ptr(W13_fp8),
                                    _ptr(W2), _ptr(h), _ptr(out), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_expert_ffn_fp8")


def moe_combine(cfg, out, topk_gate, pos, y, status=None, stream=None):
    _check(lib().moe_combine(ctypes.byref(cfg), _ptr(out), _ptr(topk_gate), _ptr(pos), _ptr(y), _ptr(status),
                             _stream(stream)), "moe_combine")


def moe_layer_forward(cfg, x, Wg, bias, W13, W2, y, ws, stream=None):
    _check(lib().moe_layer_forward(ctypes.byref(cfg), _ptr(x), _ptr(Wg), _ptr(bias), _ptr(W13), _ptr(W2), _ptr(y),
                                   _ptr(ws), ws.numel(), _stream(stream)), "moe_layer_forward")


def moe_layer_forward_traced(cfg, x, Wg, bias, W13, W2, y, ws, events, stream=None):
    """``events``: six torch.cuda.Event(enable_timing=True), recorded between stages."""
    for ev in events:
        if ev.cuda_event == 0:  # created lazily by torch; record once to materialise
            ev.record()
    arr = (_p * len(events))(*[ev.cuda_event for ev in events])
    _check(lib().moe_layer_forward_traced(ctypes.byref(cfg), _ptr(x), _ptr(Wg), _ptr(bias), _ptr(W13), _ptr(W2),
                                          _ptr(y), _ptr(ws), ws.numel(), _stream(stream), arr, len(events)),
           "moe_layer_forward_traced")


def moe_layer_forward_host(cfg, x_host, Wg, bias, W13, W2, y_host, ws, stream=None):
    _check(lib().moe_layer_forward_host(ctypes.byref(cfg), _ptr(x_host), _ptr(Wg), _ptr(bias), _ptr(W13), _ptr(W2),
                                        _ptr(y_host), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_layer_forward_host")


def moe_layer_forward_host_async(cfg, x_host, Wg, bias, W13, W2, y_host, ws, stream=None):
    """moe_layer_forward_host without the final sync: y_host is ready once `stream` gets there."""
    _check(lib().moe_layer_forward_host_async(ctypes.byref(cfg), _ptr(x_host), _ptr(Wg), _ptr(bias), _ptr(W13),
                                              _ptr(W2), _ptr(y_host), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_layer_forward_host_async")


def moe_read_status(status_ptr: int, stream=None) -> int:
    """Synchronises the stream and returns the device status flags (0 = fine)."""
    flags = _i32(0)
    code = lib().moe_read_status(status_ptr, ctypes.byref(flags), _stream(stream))
    if code not in (MOE_OK, MOE_ERR_DEVICE):
        _check(code, "moe_read_status")
    return int(flags.value)


def moe_version() -> int:
    return lib().moe_version()


def exported_symbols() -> list[str]:
    """Function names declared in include/moe.h."""
    import re
    text = open(HEADER_PATH).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(moe_\w+)\s*\(", text, flags=re.M)))


def moe_ffn_kernel_name(cfg) -> str:
    """Kernel the expert GEMMs of this config run on ("" for identity experts)."""
    return lib().moe_ffn_kernel_name(ctypes.byref(cfg)).decode()
