"""The C ABI on the host: the library loads, exports every declared symbol, sizes
workspaces and rejects bad arguments with the documented codes before touching a GPU.

Nothing here launches a kernel: every call below fails validation (or is pure host
arithmetic), so the pointers passed are never dereferenced.
"""
import ctypes

import pytest
import torch

from routing_dispatch_combine_moe_b300 import abi, sizing
from routing_dispatch_combine_moe_b300 import workloads as wl

A16, MIS = 0x10000, 0x10001  # fake device addresses: 16-byte aligned / misaligned


def test_library_exports_every_declared_symbol():
    lib = abi.lib()
    names = abi.exported_symbols()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/moe.h but not exported"
    assert abi.moe_version() >= 100


def test_capacity_exact_integer_rounding():
    assert abi.moe_capacity(8192, 2, 64, "1.25") == 320
    assert abi.moe_capacity(10, 1, 3, "1") == 4
    assert abi.moe_capacity(10, 1, 3, "0.9") == 3
    assert abi.moe_capacity(16, 2, 8, "1", min_capacity=6) == 6
    for T, k, E, f in [(4096, 8, 256, "1.1"), (1000, 3, 7, "1.33"), (5, 2, 64, "0.5")]:
        assert abi.moe_capacity(T, k, E, f) == sizing.capacity(T, k, E, f)
    assert abi.lib().moe_capacity(10, 1, 3, 1, 0, 0) == -1
    assert abi.lib().moe_capacity(0, 1, 3, 1, 1, 0) == -1


def cfg(**kw):
    base = dict(T=64, d=128, E=8, k=2, F=64, D=1, act="bf16", expert="swiglu", capacity=None)
    base.update(kw)
    return abi.make_config(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(), abi.MOE_OK),
    (dict(k=9), abi.MOE_ERR_ARG),
    (dict(k=0), abi.MOE_ERR_ARG),
    (dict(T=0), abi.MOE_ERR_ARG),
    (dict(E=8, D=3), abi.MOE_ERR_ARG),
    (dict(F=0), abi.MOE_ERR_ARG),
    (dict(F=0, expert="identity"), abi.MOE_OK),
    (dict(E=300, k=2), abi.MOE_OK),
    (dict(E=600, k=2), abi.MOE_ERR_UNSUPPORTED),
    (dict(E=64, k=17), abi.MOE_ERR_UNSUPPORTED),
    (dict(d=100), abi.MOE_ERR_ALIGN),       # 200 bytes per bf16 row
    (dict(d=100, act="f32"), abi.MOE_OK),   # 400 bytes per fp32 row
    (dict(F=36), abi.MOE_ERR_ALIGN),
    (dict(F=36, expert="identity"), abi.MOE_OK),
    (dict(precision="split_h"), abi.MOE_OK),
    (dict(precision="split_h", F=72), abi.MOE_ERR_UNSUPPORTED),  # split h needs F % 64 == 0
    (dict(precision="split_h", F=72, act="f32"), abi.MOE_OK),      # fp32 ignores the precision mode
    (dict(precision="f32_out", F=72), abi.MOE_OK),
    (dict(precision="bf16", F=72), abi.MOE_OK),
])
def test_validate_config(kw, code):
    assert abi.moe_validate_config(cfg(**kw)) == code


def test_validate_rejects_unknown_precision_and_bad_shared_counts():
    c = cfg()
    c.precision = 7
    assert abi.moe_validate_config(c) == abi.MOE_ERR_ARG
    assert abi.moe_validate_config(cfg(n_shared=-1)) == abi.MOE_ERR_ARG
    assert abi.moe_validate_config(cfg(n_shared=2)) == abi.MOE_OK
    assert abi.moe_validate_config(cfg(E=256, k=8, n_shared=1)) == abi.MOE_OK       # 257 experts, 9 slots
    assert abi.moe_validate_config(cfg(E=510, k=2, n_shared=3)) == abi.MOE_ERR_UNSUPPORTED
    assert abi.moe_validate_config(cfg(E=64, k=15, n_shared=2)) == abi.MOE_ERR_UNSUPPORTED


def test_drop_policy_and_layout_validation():
    assert abi.moe_validate_config(cfg(capacity=16, drop_policy="gate")) == abi.MOE_OK
    assert abi.moe_validate_config(cfg(drop_policy="gate")) == abi.MOE_OK          # dropless: nothing to select
    assert abi.moe_validate_config(cfg(capacity=16, layout="padded")) == abi.MOE_OK
    assert abi.moe_validate_config(cfg(capacity=0, layout="padded")) == abi.MOE_OK
    assert abi.moe_validate_config(cfg(layout="padded")) == abi.MOE_ERR_UNSUPPORTED  # padded needs a capacity
    assert abi.moe_validate_config(cfg(capacity=16, layout="padded", n_shared=1)) == abi.MOE_ERR_UNSUPPORTED
    for field, bad in (("drop_policy", 2), ("layout", -1)):
        c = cfg()
        setattr(c, field, bad)
        assert abi.moe_validate_config(c) == abi.MOE_ERR_ARG


def test_rows_capacity_and_kernel_counts():
    assert abi.moe_rows_capacity(cfg()) == 64 * 2
    assert abi.moe_rows_capacity(cfg(n_shared=1)) == 64 * 3
    assert abi.moe_rows_capacity(cfg(capacity=5)) == 64 * 2                 # packed: T*K whatever C is
    assert abi.moe_rows_capacity(cfg(capacity=5, layout="padded")) == 8 * 5
    assert abi.moe_rows_capacity(cfg(capacity=100, layout="padded")) == 8 * 100  # may exceed T*K
    assert abi.moe_rows_capacity(cfg(capacity=0, layout="padded")) == 0
    with pytest.raises(abi.MoeError):
        abi.moe_rows_capacity(cfg(k=9))
    # cfg(): E=8, d=128, so the router is one fused launch; the router also counts the
    # dispatch histogram, so the dispatch is scan, scatter and gather
    assert abi.moe_kernels_per_forward(cfg()) == 7
    assert abi.moe_kernels_per_forward(cfg(capacity=5, drop_policy="gate")) == 8
    assert abi.moe_kernels_per_forward(cfg(capacity=5, drop_policy="gate", layout="padded")) == 9
    assert abi.moe_kernels_per_forward(cfg(capacity=0, layout="padded")) == 5   # no rows: no padding, no GEMMs
    assert abi.moe_kernels_per_forward(cfg(expert="identity", F=0)) == 5
    # bf16 and E >= 64: W_g's split, tensor-core split-K logits, top-k; fp32: FMA logits + top-k
    assert abi.moe_kernels_per_forward(cfg(E=64, d=1024)) == 9
    assert abi.moe_kernels_per_forward(cfg(E=64, d=1024, act="f32")) == 8


def test_padded_workspace_holds_n_times_c_rows():
    big = cfg(capacity=100, layout="padded")     # 800 rows against T*K = 128
    v = abi.moe_workspace_view()
    base = 1 << 40
    n = abi.moe_workspace_bytes(big)
    assert abi.lib().moe_workspace_get_view(ctypes.byref(big), base, n, ctypes.byref(v)) == 0
    assert v.h - v.xperm >= 800 * 128 * 2 and base + n - v.out >= 800 * 128 * 4
    assert v.map.drop_list - v.map.row_src >= 800 * 4


def test_shared_experts_size_the_routing_arrays():
    base, shared = cfg(E=8, k=2), cfg(E=8, k=2, n_shared=1)
    vb, vs = abi.moe_workspace_view(), abi.moe_workspace_view()
    lib, b0 = abi.lib(), 1 << 40
    assert lib.moe_workspace_get_view(ctypes.byref(base), b0, abi.moe_workspace_bytes(base), ctypes.byref(vb)) == 0
    assert lib.moe_workspace_get_view(ctypes.byref(shared), b0, abi.moe_workspace_bytes(shared), ctypes.byref(vs)) == 0
    # xperm holds T*K rows: 64 * 3 with one shared slot against 64 * 2
    assert (vs.out - vs.xperm) - (vb.out - vb.xperm) >= 64 * 128 * 2 - 256


def test_split_h_workspace_holds_hi_lo_pairs_and_fp32_outputs():
    fast, acc = cfg(precision="bf16"), cfg(precision="split_h")
    A = 64 * 2
    vf, va = abi.moe_workspace_view(), abi.moe_workspace_view()
    base = 1 << 40
    lib = abi.lib()
    assert lib.moe_workspace_get_view(ctypes.byref(fast), base, abi.moe_workspace_bytes(fast), ctypes.byref(vf)) == 0
    assert lib.moe_workspace_get_view(ctypes.byref(acc), base, abi.moe_workspace_bytes(acc), ctypes.byref(va)) == 0
    assert vf.out - vf.h >= A * 64 * 2 and va.out - va.h >= A * 2 * 64 * 2
    assert base + abi.moe_workspace_bytes(acc) - va.out >= A * 128 * 4
    assert abi.out_dtype(acc) == torch.float32 and abi.out_dtype(fast) == torch.bfloat16
    assert abi.hidden_cols(acc) == 128 and abi.hidden_cols(fast) == 64
    mid = cfg(precision="f32_out")
    assert abi.out_dtype(mid) == torch.float32 and abi.hidden_cols(mid) == 64
    assert abi.out_dtype(cfg(precision="split_h", expert="identity", F=0)) == torch.bfloat16


def test_workspace_sizes_and_layout():
    for name in wl.WORKLOAD_ORDER:
        w = wl.WORKLOADS[name]
        c = abi.config_for(w)
        fwd, host = abi.moe_workspace_bytes(c), abi.moe_workspace_bytes_host(c)
        disp = abi.moe_dispatch_workspace_bytes(c)
        A = w.T * w.k
        assert 0 < disp < fwd < host
        assert host - fwd >= 2 * w.T * w.d * w.act_bytes
        assert fwd >= A * w.d * w.act_bytes * (1 if w.expert == "identity" else 2)
        base = 1 << 40
        v = abi.lib()
        view = abi.moe_workspace_view()
        assert v.moe_workspace_get_view(ctypes.byref(c), base, fwd, ctypes.byref(view)) == abi.MOE_OK
        ptrs = [view.status, view.topk_idx, view.topk_gate, view.map.counts_routed, view.map.counts_kept,
                view.map.offsets, view.map.rank_offsets, view.map.n_dropped, view.map.pos, view.map.row_src,
                view.map.drop_list, view.xperm]
        assert all(p % 256 == 0 and base <= p < base + fwd for p in ptrs)
        assert view.status == base
        if w.expert == "identity":
            assert view.out == view.xperm and not view.h
        else:
            assert view.xperm < view.h < view.out < base + fwd
            assert view.out + A * w.d * w.act_bytes <= base + fwd
        assert v.moe_workspace_get_view(ctypes.byref(c), base, fwd - 1, ctypes.byref(view)) == abi.MOE_ERR_WORKSPACE
        small_router = w.E <= 32 and w.d * w.E * 4 <= 128 * 1024  # one fused router launch instead of two
        tc_router = w.act == "bf16" and w.E >= 64 and not small_router  # W_g's split kernel comes first
        assert abi.moe_kernels_per_forward(c) == ((6 if w.expert == "identity" else 8) + (5 if w.dedup else 0)
                                                  + (1 if w.dispatch_dtype == "fp8" and not w.dedup else 0)
                                                  + (1 if w.precision == "fp8_h" else 0)  # h quantized between GEMMs
                                                  - (1 if small_router else 0) + (1 if tc_router else 0))


def test_entry_points_reject_bad_arguments_on_the_host():
    lib = abi.lib()
    c = cfg()
    bad = cfg(k=9)
    ref = ctypes.byref
    # route
    nc = abi.moe_route_workspace_bytes(c)
    assert lib.moe_route(ref(bad), A16, A16, None, A16, A16, A16, nc, None) == abi.MOE_ERR_ARG
    assert lib.moe_route(ref(c), None, A16, None, A16, A16, A16, nc, None) == abi.MOE_ERR_ARG
    assert lib.moe_route(ref(c), MIS, A16, None, A16, A16, A16, nc, None) == abi.MOE_ERR_ALIGN
    big = cfg(E=64, k=2)  # the split-K partial logits live in the route workspace
    nr = abi.moe_route_workspace_bytes(big)
    assert nr >= 64 * 64 * 4 and abi.moe_route_workspace_bytes(c) >= 64 * 8 * 4
    assert lib.moe_route(ref(big), A16, A16, None, A16, A16, None, 0, None) == abi.MOE_ERR_ARG
    assert lib.moe_route(ref(big), A16, A16, None, A16, A16, A16, nr - 1, None) == abi.MOE_ERR_WORKSPACE
    # dispatch
    m = abi.moe_dispatch_map(*([A16] * 8))
    nbytes = abi.moe_dispatch_workspace_bytes(c)
    assert lib.moe_dispatch(ref(c), A16, A16, None, ref(m), A16, A16, nbytes - 1, None) == abi.MOE_ERR_WORKSPACE
    assert lib.moe_dispatch(ref(c), A16, A16, None, ref(m), MIS, A16, nbytes, None) == abi.MOE_ERR_ALIGN
    m0 = abi.moe_dispatch_map(*([A16] * 7 + [None]))
    assert lib.moe_dispatch(ref(c), A16, A16, None, ref(m0), A16, A16, nbytes, None) == abi.MOE_ERR_ARG
    # the gate drop policy with a capacity needs the gates
    g = cfg(capacity=16, drop_policy="gate")
    ng = abi.moe_dispatch_workspace_bytes(g)
    assert ng >= nbytes + 64 * 2 * 4  # plus the per-expert assignment lists
    assert lib.moe_dispatch(ref(g), A16, A16, None, ref(m), A16, A16, ng, None) == abi.MOE_ERR_ARG
    assert lib.moe_dispatch_static(ref(g), A16, A16, None, ref(m), A16, None) == abi.MOE_ERR_ARG
    # expert ffn
    assert lib.moe_expert_ffn(ref(cfg(expert="identity", F=0)), A16, A16, A16, A16, A16, A16, A16, 256,
                              None) == abi.MOE_ERR_ARG
    assert lib.moe_expert_ffn(ref(c), A16, A16, A16, A16, MIS, A16, A16, 256, None) == abi.MOE_ERR_ALIGN
    assert lib.moe_expert_ffn(ref(c), A16, A16, A16, A16, A16, A16, A16, 255, None) == abi.MOE_ERR_WORKSPACE
    # combine
    assert lib.moe_combine(ref(c), A16, A16, None, A16, None, None) == abi.MOE_ERR_ARG
    assert lib.moe_combine(ref(c), A16, A16, A16, MIS, None, None) == abi.MOE_ERR_ALIGN
    # layer
    n = abi.moe_workspace_bytes(c)
    assert lib.moe_layer_forward(ref(c), A16, A16, None, None, A16, A16, A16, n, None) == abi.MOE_ERR_ARG
    assert lib.moe_layer_forward(ref(c), A16, A16, None, A16, A16, A16, A16, n - 1, None) == abi.MOE_ERR_WORKSPACE
    assert lib.moe_layer_forward(ref(c), MIS, A16, None, A16, A16, A16, A16, n, None) == abi.MOE_ERR_ALIGN
    evs = (ctypes.c_void_p * 6)(*([A16] * 6))
    assert lib.moe_layer_forward_traced(ref(c), A16, A16, None, A16, A16, A16, A16, n, None, evs,
                                        5) == abi.MOE_ERR_ARG
    nh = abi.moe_workspace_bytes_host(c)
    assert lib.moe_layer_forward_host(ref(c), A16, A16, None, A16, A16, A16, A16, nh - 1,
                                      None) == abi.MOE_ERR_WORKSPACE
    assert lib.moe_read_status(None, None, None) == abi.MOE_ERR_ARG


def test_status_strings():
    for code in range(7):
        assert abi.status_string(code)
    assert abi.status_string(99) == "unknown status"


def test_ffn_kernel_name_follows_the_variant_choice():
    from routing_dispatch_combine_moe_b300 import workloads as wl
    name = lambda n: abi.moe_ffn_kernel_name(abi.config_for(wl.WORKLOADS[n]))
    assert name("tiny_f32") == "grouped_sgemm_kernel"
    assert name("dsv3_route_only") == ""                      # identity experts
    assert name("mixtral_bf16") == "grouped_gemm_swap_kernel"  # dropless, 512 rows per expert
    assert name("zipf_cf125") == "grouped_gemm_kernel"         # under a capacity
    assert name("dsv3_decode") == "grouped_gemm_kernel"        # ~4.5 rows per expert
    assert abi.moe_ffn_kernel_name(cfg(k=9)) == ""


def test_group_limit_and_dedup_validation():
    ok = abi.MOE_OK
    assert abi.moe_validate_config(cfg(E=16, k=4, n_groups=4, topk_groups=2)) == ok
    assert abi.moe_validate_config(cfg(E=16, k=4, n_groups=4, topk_groups=4)) == ok   # no limit in effect
    assert abi.moe_validate_config(cfg(E=16, k=4, n_groups=4)) == ok                  # groups alone: ignored
    assert abi.moe_validate_config(cfg(E=16, k=4, n_groups=5, topk_groups=2)) == abi.MOE_ERR_ARG  # 16 % 5
    assert abi.moe_validate_config(cfg(E=16, k=4, n_groups=4, topk_groups=5)) == abi.MOE_ERR_ARG  # M > G
    assert abi.moe_validate_config(cfg(E=16, k=5, n_groups=4, topk_groups=1)) == abi.MOE_ERR_ARG  # k > M*E/G
    assert abi.moe_validate_config(cfg(E=64, k=2, n_groups=64, topk_groups=2)) == abi.MOE_ERR_UNSUPPORTED
    assert abi.moe_validate_config(cfg(E=16, k=2, D=4, dedup=True)) == ok
    assert abi.moe_validate_config(cfg(E=64, k=2, D=32, dedup=True)) == abi.MOE_ERR_UNSUPPORTED   # D > 16
    c = cfg()
    c.dedup = 2
    assert abi.moe_validate_config(c) == abi.MOE_ERR_ARG


def test_dedup_workspace_and_kernel_count():
    plain, dd = cfg(E=16, k=2, D=4), cfg(E=16, k=2, D=4, dedup=True)
    assert abi.moe_kernels_per_forward(dd) == abi.moe_kernels_per_forward(plain) + 5
    assert abi.moe_dispatch_workspace_bytes(dd) > abi.moe_dispatch_workspace_bytes(plain)
    v = abi.moe_workspace_view()
    base = 1 << 40
    n = abi.moe_workspace_bytes(dd)
    assert abi.lib().moe_workspace_get_view(ctypes.byref(dd), base, n, ctypes.byref(v)) == 0
    assert v.xsend and v.send.send_pos and base + n - v.xsend >= 64 * 4 * 128 * 2
    vp = abi.moe_workspace_view()
    assert abi.lib().moe_workspace_get_view(ctypes.byref(plain), base, abi.moe_workspace_bytes(plain),
                                            ctypes.byref(vp)) == 0
    assert not vp.xsend and not vp.send.send_pos
    m = abi.send_map(*([None] * 4))
    A16 = 1 << 20
    assert abi.lib().moe_dispatch_dedup(ctypes.byref(plain), A16, A16, A16, ctypes.byref(m), A16, A16, A16,
                                        1 << 20, None) == abi.MOE_ERR_ARG  # cfg.dedup not set
    assert abi.lib().moe_dispatch_dedup(ctypes.byref(dd), A16, A16, A16, ctypes.byref(m), A16, A16, A16,
                                        1 << 20, None) == abi.MOE_ERR_ARG  # null map arrays


def test_fp8_dispatch_validation_and_workspace():
    f8 = cfg(dispatch_dtype="fp8")
    assert abi.moe_validate_config(f8) == abi.MOE_OK
    assert abi.moe_validate_config(cfg(act="f32", dispatch_dtype="fp8")) == abi.MOE_ERR_UNSUPPORTED
    # the deduplicated dispatch sends its rows as FP8: same kernel count as the bf16 dedup
    # (the send gather quantizes, the fan-out dequantizes), the send codes and scales in
    # the view; moe_dispatch_dedup rejects it, moe_dispatch_dedup_fp8 takes it
    ddf = cfg(D=4, dedup=True, dispatch_dtype="fp8")
    dd = cfg(D=4, dedup=True)
    assert abi.moe_validate_config(ddf) == abi.MOE_OK
    assert abi.moe_kernels_per_forward(ddf) == abi.moe_kernels_per_forward(dd)
    vd = abi.moe_workspace_view()
    nd = abi.moe_workspace_bytes(ddf)
    assert abi.lib().moe_workspace_get_view(ctypes.byref(ddf), 1 << 40, nd, ctypes.byref(vd)) == 0
    assert vd.xq == vd.xsend and vd.xscale and vd.xscale >= vd.xsend + 64 * 4 * 128
    assert vd.xsend_scale == vd.xscale
    m = abi.moe_send_map(*([A16] * 4))
    assert abi.lib().moe_dispatch_dedup(ctypes.byref(ddf), A16, A16, A16, ctypes.byref(m), A16, A16, A16, nd,
                                        None) == abi.MOE_ERR_ARG
    assert abi.lib().moe_dispatch_dedup_fp8(ctypes.byref(dd), A16, A16, A16, ctypes.byref(m), A16, A16, A16, A16,
                                            nd, None) == abi.MOE_ERR_ARG          # not an FP8 config
    assert abi.lib().moe_dispatch_dedup_fp8(ctypes.byref(ddf), A16, A16, A16, ctypes.byref(m), MIS, A16, A16, A16,
                                            nd, None) == abi.MOE_ERR_ALIGN
    assert abi.lib().moe_dispatch_dedup_fp8(ctypes.byref(ddf), A16, A16, A16, ctypes.byref(m), A16, A16, A16, A16,
                                            abi.moe_dispatch_workspace_bytes(ddf) - 1, None) == abi.MOE_ERR_WORKSPACE
    # with the FP8 GEMM's format the send rows carry one scale each and the fan-out fills
    # the expert rows' codes and scales (xq, xscale), not xperm
    ddg = cfg(D=4, dedup=True, dispatch_dtype="fp8_gemm")
    assert abi.moe_validate_config(ddg) == abi.MOE_OK
    assert abi.moe_kernels_per_forward(ddg) == abi.moe_kernels_per_forward(dd)
    ng = abi.moe_workspace_bytes(ddg)
    vg = abi.moe_workspace_view()
    assert abi.lib().moe_workspace_get_view(ctypes.byref(ddg), 1 << 40, ng, ctypes.byref(vg)) == 0
    assert vg.xq and vg.xq != vg.xsend and vg.xscale - vg.xq >= 64 * 2 * 128      # expert rows' codes
    assert vg.xsend_scale - vg.xsend >= 64 * 4 * 128                              # T*D send rows of d codes
    assert (1 << 40) + ng - vg.xsend_scale >= 64 * 4 * 4                          # T*D row scales
    vp = abi.moe_workspace_view()
    assert abi.lib().moe_workspace_get_view(ctypes.byref(dd), 1 << 40, abi.moe_workspace_bytes(dd),
                                            ctypes.byref(vp)) == 0
    assert not vp.xsend_scale                                                     # bf16 send rows
    lib = abi.lib()
    dg = abi.moe_dispatch_workspace_bytes(ddg)
    assert lib.moe_dispatch_dedup(ctypes.byref(ddg), A16, A16, A16, ctypes.byref(m), A16, A16, A16, dg,
                                  None) == abi.MOE_ERR_ARG
    assert lib.moe_dispatch_dedup_fp8(ctypes.byref(ddg), A16, A16, A16, ctypes.byref(m), A16, A16, A16, A16,
                                      dg, None) == abi.MOE_ERR_ARG
    assert lib.moe_dispatch_dedup_fp8_gemm(ctypes.byref(ddf), A16, A16, A16, ctypes.byref(m), A16, A16, A16, A16,
                                           A16, dg, None) == abi.MOE_ERR_ARG     # block-scaled config
    assert lib.moe_dispatch_dedup_fp8_gemm(ctypes.byref(ddg), A16, A16, A16, ctypes.byref(m), A16, A16, None, A16,
                                           A16, dg, None) == abi.MOE_ERR_ARG     # no expert-row codes
    assert lib.moe_dispatch_dedup_fp8_gemm(ctypes.byref(ddg), A16, A16, A16, ctypes.byref(m), A16, MIS, A16, A16,
                                           A16, dg, None) == abi.MOE_ERR_ALIGN
    assert lib.moe_dispatch_dedup_fp8_gemm(ctypes.byref(ddg), A16, A16, A16, ctypes.byref(m), A16, A16, A16, A16,
                                           A16, dg - 1, None) == abi.MOE_ERR_WORKSPACE
    c = cfg()
    c.dispatch_dtype = 5
    assert abi.moe_validate_config(c) == abi.MOE_ERR_ARG
    assert abi.moe_kernels_per_forward(f8) == abi.moe_kernels_per_forward(cfg()) + 1
    v = abi.moe_workspace_view()
    base = 1 << 40
    n = abi.moe_workspace_bytes(f8)
    assert abi.lib().moe_workspace_get_view(ctypes.byref(f8), base, n, ctypes.byref(v)) == 0
    assert v.xq and v.xscale and v.xscale - v.xq >= 64 * 2 * 128      # rows x d codes
    assert base + n - v.xscale >= 64 * 2 * 1 * 4                      # rows x ceil(d/128) scales
    m = abi.dispatch_map(*([None] * 8))
    assert abi.lib().moe_dispatch_fp8(ctypes.byref(cfg()), 1 << 20, 1 << 20, ctypes.byref(m), 1 << 20, 1 << 20,
                                      None, 1 << 20, 1 << 20, None) == abi.MOE_ERR_ARG   # not an fp8 config



def test_fp8_gemm_validation_workspace_and_weight_bytes():
    g = cfg(dispatch_dtype="fp8_gemm")
    assert abi.moe_validate_config(g) == abi.MOE_OK
    assert abi.moe_validate_config(cfg(dispatch_dtype="fp8_gemm", expert="relu")) == abi.MOE_OK
    assert abi.moe_validate_config(cfg(act="f32", dispatch_dtype="fp8_gemm")) == abi.MOE_ERR_UNSUPPORTED
    assert abi.moe_validate_config(cfg(F=0, expert="identity", dispatch_dtype="fp8_gemm")) == \
        abi.MOE_ERR_UNSUPPORTED
    assert abi.moe_validate_config(cfg(precision="split_h", dispatch_dtype="fp8_gemm")) == abi.MOE_OK
    assert abi.moe_validate_config(cfg(d=136, dispatch_dtype="fp8_gemm")) == abi.MOE_ERR_ALIGN  # 136-byte code rows
    assert abi.moe_validate_config(cfg(d=136)) == abi.MOE_OK
    # the quantizing gather replaces the plain one: same kernel count as the bf16 layer
    assert abi.moe_kernels_per_forward(g) == abi.moe_kernels_per_forward(cfg())
    v = abi.moe_workspace_view()
    base = 1 << 40
    n = abi.moe_workspace_bytes(g)
    assert abi.lib().moe_workspace_get_view(ctypes.byref(g), base, n, ctypes.byref(v)) == 0
    rows = 64 * 2
    assert v.xq and v.xscale and v.xscale - v.xq >= rows * 128 and base + n - v.xscale >= rows * 4
    # weight buffer: N*R*d codes, the next 256-byte boundary, N*R fp32 scales
    codes = 8 * 128 * 128
    assert abi.moe_fp8_weight_bytes(g) == (codes + 255) // 256 * 256 + 4 * 8 * 128
    relu = cfg(dispatch_dtype="fp8_gemm", expert="relu", F=80)
    assert abi.moe_fp8_weight_bytes(relu) == (8 * 80 * 128 + 255) // 256 * 256 + 4 * 8 * 80
    assert abi.moe_fp8_weight_bytes(cfg()) == 0 and abi.moe_fp8_weight_bytes(cfg(dispatch_dtype="fp8")) == 0
    assert abi.moe_ffn_kernel_name(g) == "grouped_gemm_swap_kernel<e4m3>"
    lib = abi.lib()
    # the bf16 FFN entry refuses an fp8_gemm config, the FP8 entry any other config
    assert lib.moe_expert_ffn(ctypes.byref(g), A16, A16, A16, A16, A16, A16, A16, 1 << 20, None) == abi.MOE_ERR_ARG
    assert lib.moe_expert_ffn_fp8(ctypes.byref(cfg()), A16, A16, A16, A16, A16, A16, A16, A16, 1 << 20,
                                  None) == abi.MOE_ERR_ARG
    assert lib.moe_expert_ffn_fp8(ctypes.byref(g), None, A16, A16, A16, A16, A16, A16, A16, 1 << 20,
                                  None) == abi.MOE_ERR_ARG
    assert lib.moe_expert_ffn_fp8(ctypes.byref(g), MIS, A16, A16, A16, A16, A16, A16, A16, 1 << 20,
                                  None) == abi.MOE_ERR_ALIGN
    assert lib.moe_expert_ffn_fp8(ctypes.byref(g), A16, A16, A16, A16, A16, A16, A16, A16, 16,
                                  None) == abi.MOE_ERR_WORKSPACE
    assert lib.moe_quantize_weights_fp8(ctypes.byref(cfg()), A16, A16, None) == abi.MOE_ERR_ARG
    assert lib.moe_quantize_weights_fp8(ctypes.byref(g), A16, MIS, None) == abi.MOE_ERR_ALIGN
    m = abi.dispatch_map(*([None] * 8))
    m.pos = m.row_src = m.offsets = A16
    # the row-scaled format feeds the FP8 GEMM directly: no bf16 rows to write
    assert lib.moe_dispatch_fp8(ctypes.byref(g), A16, A16, ctypes.byref(m), A16, A16, A16, A16, 1 << 20,
                                None) == abi.MOE_ERR_ARG


def test_fp8_h_validation_workspace_and_w2_bytes():
    h8 = cfg(dispatch_dtype="fp8_gemm", precision="fp8_h")
    assert abi.moe_validate_config(h8) == abi.MOE_OK
    assert abi.moe_validate_config(cfg(precision="fp8_h")) == abi.MOE_ERR_UNSUPPORTED        # needs the FP8 up GEMM
    assert abi.moe_validate_config(cfg(dispatch_dtype="fp8_gemm", precision="fp8_h", F=72)) == abi.MOE_ERR_ALIGN
    assert abi.moe_validate_config(cfg(precision="fp8_h", act="f32")) == abi.MOE_OK   # fp32 ignores the mode
    assert abi.out_dtype(h8) == torch.float32 and abi.hidden_cols(h8) == 64
    g = cfg(dispatch_dtype="fp8_gemm")
    assert abi.moe_kernels_per_forward(h8) == abi.moe_kernels_per_forward(g) + 1
    # W2 buffer: N*d*F codes, the next 256-byte boundary, N*d fp32 scales
    assert abi.moe_fp8_w2_bytes(h8) == (8 * 128 * 64 + 255) // 256 * 256 + 4 * 8 * 128
    assert abi.moe_fp8_w2_bytes(g) == 0
    # the FFN workspace: the status word, the GEMM split's tickets (two per slot) and fp32
    # partial slots (2 SMs x 128 features x 256 rows each), then h's codes and scales
    rows = 64 * 2
    split = 1024 + 96 * 2 * 128 * 256 * 4
    assert abi.moe_ffn_workspace_bytes(h8) >= split + rows * 64 + rows * 4
    assert abi.moe_ffn_workspace_bytes(g) == split
    assert abi.moe_ffn_workspace_bytes(cfg(act="f32", expert="relu")) == 256  # FMA experts: no split
    v = abi.moe_workspace_view()
    base = 1 << 40
    n = abi.moe_workspace_bytes(h8)
    assert abi.lib().moe_workspace_get_view(ctypes.byref(h8), base, n, ctypes.byref(v)) == 0
    assert v.hq and v.hscale and v.hscale - v.hq >= rows * 64 and base + n - v.hscale >= rows * 4
    assert abi.lib().moe_workspace_get_view(ctypes.byref(g), base, abi.moe_workspace_bytes(g), ctypes.byref(v)) == 0
    assert not v.hq and not v.hscale
    lib = abi.lib()
    assert lib.moe_quantize_w2_fp8(ctypes.byref(g), A16, A16, None) == abi.MOE_ERR_ARG
    assert lib.moe_quantize_w2_fp8(ctypes.byref(h8), MIS, A16, None) == abi.MOE_ERR_ALIGN
    assert lib.moe_expert_ffn_fp8(ctypes.byref(h8), A16, A16, A16, A16, A16, A16, A16, A16, 256,
                                  None) == abi.MOE_ERR_WORKSPACE

