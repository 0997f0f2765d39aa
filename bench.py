"""Benchmark of the MoE layer forward (route -> dispatch -> expert FFN -> combine).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one moe_layer_forward over one batch of the workload (default: the
DeepSeek-V3-shaped bf16 layer, T=4096, d=7168, E=256 routed experts, k=8, SwiGLU
F=2048, 22.5 GB of expert weights), inputs and weights resident in HBM, timed with
CUDA events on the launching stream. Under
torchrun each rank runs an independent replica on its own GPU (the layer needs no
cross-GPU exchange on one device; see the design notes), so the job processes
N * T tokens per step and the step time is the max over ranks.

Prints ONE JSON line on rank 0. `--impl reference` times the float64 CPU oracle on
a bounded token sample of the same workload on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from routing_dispatch_combine_moe_b300 import abi, sizing  # noqa: E402
from routing_dispatch_combine_moe_b300 import workloads as wl  # noqa: E402

METRIC = "MoE-layer tokens/s"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "dsv3_full"
STAGES = ["route", "dispatch", "expert_up", "expert_down", "combine"]
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
L2_FLUSH_BYTES = 256 << 20  # twice the 126 MB L2


# ------------------------------------------------------------------ distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, local, backend="nccl"):
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        if backend == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group(backend)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(value: float, world: int, device) -> float:
    """Max of a float over ranks (identity at world size 1)."""
    if world == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank: int, steps: int, world: int, max_seconds: float) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return tokens_per_rank * steps * world / max_seconds


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-i",
                 str(self.gpu_index), "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ peaks / traffic
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def versions(device) -> dict:
    """Software and hardware the numbers come from."""
    v = {"torch": torch.__version__, "cuda_runtime": torch.version.cuda, "library": abi.lib().moe_version(),
         "gpu": torch.cuda.get_device_name(device), "sms": torch.cuda.get_device_properties(device).multi_processor_count,
         "host_cores": os.cpu_count()}
    try:
        import pynvml
        pynvml.nvmlInit()
        drv = pynvml.nvmlSystemGetDriverVersion()
        v["driver"] = drv.decode() if isinstance(drv, bytes) else drv
    except Exception:  # noqa: BLE001 - the versions are informative only
        v["driver"] = None
    return v


def file_sha(path: str) -> str:
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def load_traffic(workload: str, kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel source is unchanged."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    rec = d.get(workload, {}).get(kernel)
    if not rec:
        return None
    src = os.path.join(ROOT, "routing_dispatch_combine_moe_b300", "csrc", rec["source"])
    if not os.path.exists(src) or file_sha(src) != rec["source_sha"]:
        return None
    return rec["bytes_per_launch"]


# ------------------------------------------------------------------ algorithmic work
def fp8_row_bytes(d: int, per_row: bool = False) -> int:
    """Wire bytes of one FP8-dispatched row: d e4m3 codes and a 4-byte scale per 128-element
    block (or one per row, the FP8-GEMM format)."""
    return d + 4 * (1 if per_row else (d + 127) // 128)


def algorithmic(w, rows: int, out_bytes: int, h_cols: int, rows_sent: int = 0, routed_rows: int = 0,
                active_experts: int | None = None) -> dict:
    """Algorithmic work per launch: flops of the formulas, bytes each kernel must move at least.

    The expert GEMMs read the weights of the experts that hold at least one row
    (`active_experts`, default all of them): an expert with no rows needs none of its
    weights, and the kernels skip it.

    With the deduplicated dispatch the rows travel x -> send buffer -> expert rows: x is
    read once, each send row written once and read once, each expert row written once.
    With the FP8 dispatch each routed row is written as codes + scales, read back and
    written as a bf16 row. With the FP8 GEMM every row is written once as codes + its
    scale (instead of a bf16 row) and the up projection reads those and the e4m3 weights;
    with dedup too, the send rows are codes + one scale as well.
    """
    b = w.act_bytes
    up, down = sizing.expert_gemm_flops(rows, w.d, w.F, w.expert)
    ident = w.expert == "identity"
    f8g = w.dispatch_dtype == "fp8_gemm"
    dispatch = sizing.dispatch_hbm_bytes(w.T, w.d, rows, b) + (2 * rows_sent * w.d * b if w.dedup else 0)
    if w.dispatch_dtype == "fp8" and w.dedup:  # the send rows travel as codes + block scales
        dispatch += 2 * rows_sent * (fp8_row_bytes(w.d) - w.d * b)
    elif w.dispatch_dtype == "fp8":
        dispatch += 2 * routed_rows * fp8_row_bytes(w.d)
    if f8g:  # x read once, each row written as codes + one scale
        dispatch = dispatch - rows * w.d * b + rows * fp8_row_bytes(w.d, per_row=True)
        if w.dedup:  # the send rows written and read as codes + one scale each
            dispatch += 2 * rows_sent * (fp8_row_bytes(w.d, per_row=True) - w.d * b)
    up_in = rows * fp8_row_bytes(w.d, per_row=True) if f8g else rows * w.d * b
    n_w = w.n_experts if active_experts is None else active_experts
    w13_bytes = n_w * w.w13_rows * (w.d + 4) if f8g else n_w * w.w13_rows * w.d * b
    # FP8 hidden activation: the down stage also quantizes h (reads it in bf16, writes codes
    # + a scale per row) and then reads those and the e4m3 W2
    f8h = w.precision == "fp8_h"
    w2_bytes = n_w * w.d * (w.F + 4) if f8h else n_w * w.d * w.F * b
    down_in = rows * h_cols * b + 2 * rows * (w.F + 4) if f8h else rows * h_cols * b
    return dict(
        route_flops=sizing.router_flops(w.T, w.d, w.E),
        route_bytes=w.T * w.d * b + w.d * w.E * 4 + w.T * w.slots * 8,
        dispatch_bytes=dispatch,
        # the combine's algorithmic bytes: every kept expert row read once in the
        # activation dtype, y written once; with fp32 expert outputs it moves rows * d
        # * 4 instead (combine_bytes_moved)
        combine_bytes=rows * w.d * b + w.T * w.d * b,
        combine_bytes_moved=rows * w.d * (b if ident else out_bytes) + w.T * w.d * b,
        up_flops=up, down_flops=down,
        up_bytes=0 if ident else w13_bytes + up_in + rows * h_cols * b,
        down_bytes=0 if ident else w2_bytes + down_in + rows * w.d * out_bytes,
    )


# ------------------------------------------------------------------ CPU oracle timing
def oracle_tokens_per_s(w, inp, tokens: int, seed: int = 0, cache=None, threads: int | None = None,
                        cache_budget: float = 16e9) -> dict:
    """Times the float64 oracle on `tokens` tokens of the workload.

    Expert weights are converted to float64 once ("model load", untimed) and kept in
    `cache` across calls; experts this sample does not use are dropped from the cache
    first whenever it holds more than `cache_budget` bytes. `threads` limits the BLAS
    thread pools (None: all host cores).
    """
    from oracle import moe_oracle as orc  # the timed CPU baseline is the oracle, as it stands
    from oracle.packed import expert_fn, f64

    rng = np.random.default_rng(seed)
    sel = np.sort(rng.choice(w.T, size=min(tokens, w.T), replace=False))
    x = f64(inp["x"][torch.as_tensor(sel, device=inp["x"].device)])
    Wg, bias = f64(inp["Wg"]), f64(inp.get("bias"))
    cache = {} if cache is None else cache
    fn = expert_fn(w.expert, inp.get("W13"), inp.get("W2"), w.F, cache=cache,
                   fp8_up=w.dispatch_dtype == "fp8_gemm", fp8_h=w.precision == "fp8_h")
    grouped = 0 < w.topk_groups < w.n_groups
    if w.expert != "identity":  # model load: the experts this sample uses, converted once
        H = orc.router_logits(x, Wg, bias)
        idx = orc.keep_topk_grouped(H, w.k, w.n_groups, w.topk_groups) if grouped else orc.keep_topk(H, w.k)
        need = [int(e) for e in np.unique(idx)] + list(range(w.E, w.n_experts))
        per_expert = (w.w13_rows + w.F) * w.d * 8
        if len(cache) * per_expert > cache_budget:
            for e in [e for e in cache if e not in set(need)]:
                del cache[e]
        for e in need:
            fn(e, np.zeros((1, w.d)))
    cap = orc.expert_capacity(len(sel), w.k, w.E, w.capacity_factor, w.min_capacity)

    def run():
        res = orc.moe_forward(x, Wg, w.k, fn, capacity=cap, bias=bias, D=w.D, n_shared=w.n_shared,
                              drop_policy=w.drop_policy, layout=w.layout, n_groups=w.n_groups,
                              topk_groups=w.topk_groups, dispatch_dtype=w.dispatch_dtype)
        if w.dedup:
            orc.dedup_send(res["idx"], res["pos"], w.E, w.D)

    if threads is None:
        t0 = time.perf_counter()
        run()
        dt = time.perf_counter() - t0
        used = cpu_threads()
    else:
        with blas_threads(threads):
            t0 = time.perf_counter()
            run()
            dt = time.perf_counter() - t0
            used = cpu_threads()
    return dict(value=len(sel) / dt, seconds=dt, tokens=len(sel), cores=used)


def _openblas():
    """numpy's own OpenBLAS thread getter and setter, found among the loaded libraries
    (for hosts without threadpoolctl); (None, None) when there is none."""
    import ctypes
    try:
        paths = {line.split()[-1] for line in open("/proc/self/maps") if "openblas" in line and ".so" in line}
    except OSError:
        return None, None
    for path in sorted(paths):
        try:
            lib = ctypes.CDLL(path)
        except OSError:
            continue
        for suffix in ("64_", "", "_64"):
            for prefix in ("scipy_openblas_", "openblas_"):
                get = getattr(lib, f"{prefix}get_num_threads{suffix}", None)
                put = getattr(lib, f"{prefix}set_num_threads{suffix}", None)
                if get is not None and put is not None:
                    get.restype = ctypes.c_int
                    put.argtypes = [ctypes.c_int]
                    return get, put
    return None, None


def cpu_threads() -> int:
    """Threads the oracle's BLAS calls use."""
    try:
        from threadpoolctl import threadpool_info
        n = max((i.get("num_threads", 1) for i in threadpool_info()), default=1)
        return int(n)
    except Exception:
        get, _ = _openblas()
        return int(get()) if get is not None else (os.cpu_count() or 1)


class blas_threads:
    """Limits the BLAS thread pools to n threads inside the block (threadpoolctl, else
    numpy's OpenBLAS setter, else nothing)."""

    def __init__(self, n: int):
        self.n, self.ctx, self.old = n, None, None

    def __enter__(self):
        try:
            from threadpoolctl import threadpool_limits
            self.ctx = threadpool_limits(limits=self.n)
            self.ctx.__enter__()
        except ImportError:
            get, put = _openblas()
            if put is not None:
                self.old = get()
                put(self.n)
                self.put = put
        return self

    def __exit__(self, *exc):
        if self.ctx is not None:
            self.ctx.__exit__(*exc)
        elif self.old is not None:
            self.put(self.old)


def oracle_sample_tokens(w, max_tokens: int = 2048, mem_budget: float = 16e9) -> int:
    """Tokens per oracle sample, bounded so the float64 copies of the experts it touches fit mem_budget."""
    if w.expert == "identity":
        return min(w.T, max_tokens)
    per_expert = (w.w13_rows + w.F) * w.d * 8
    if w.E * per_expert <= mem_budget:
        return min(w.T, max_tokens)
    return max(1, min(w.T, max_tokens, int(mem_budget / per_expert) // w.k))


# ------------------------------------------------------------------ arms
def run_ours(args, w, world, rank, local):
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    inp = wl.make_inputs(w, seed=rank, device=device)
    cfg = abi.config_for(w)
    # the FP8-GEMM layer takes its up weights as the library's e4m3 buffer (quantized
    # once, like a model load, before any timing)
    w13 = abi.fp8_weights(cfg, inp["W13"]) if w.dispatch_dtype == "fp8_gemm" else inp.get("W13")
    w2 = abi.fp8_w2(cfg, inp["W2"]) if w.precision == "fp8_h" else inp.get("W2")
    ws = abi.workspace(cfg, device)
    y = torch.empty(w.T, w.d, dtype=w.torch_act, device=device)
    stream = torch.cuda.current_stream(device)

    def step(events=None):
        if events is None:
            abi.moe_layer_forward(cfg, inp["x"], inp["Wg"], inp.get("bias"), w13, w2, y, ws)
        else:
            abi.moe_layer_forward_traced(cfg, inp["x"], inp["Wg"], inp.get("bias"), w13, w2, y, ws, events)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    view = abi.moe_workspace_get_view(cfg, ws)
    flags = abi.moe_read_status(view.status)
    if flags:
        raise RuntimeError(f"device status flags {flags:#x} after warm-up")
    base = ws.data_ptr()
    N = w.n_experts
    offs = ws[view.offsets - base:view.offsets - base + 4 * (N + 1)].view(torch.int32).cpu().numpy()
    rank_offs = ws[view.rank_offsets - base:view.rank_offsets - base + 4 * (w.D + 1)].view(torch.int32).cpu().numpy()
    counts = ws[view.counts_routed - base:view.counts_routed - base + 4 * w.E].view(torch.int32).cpu().numpy()
    kept = ws[view.counts_kept - base:view.counts_kept - base + 4 * N].view(torch.int32).cpu().numpy()
    n_dropped = int(ws[view.n_dropped - base:view.n_dropped - base + 4].view(torch.int32).cpu()[0])
    near_ties = int(ws[view.n_near_ties - base:view.n_near_ties - base + 4].view(torch.int32).cpu()[0])
    rows = int(kept.sum())          # rows holding an assignment: the algorithmic work
    rows_computed = int(offs[-1])   # rows the expert GEMMs run over (padding included)

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    for ev in events:  # materialise the event handles before timing
        for e in ev:
            e.record(stream)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device) if args.cold_l2 else None
    torch.cuda.synchronize()

    def timed_step(i):
        if flush is not None:  # overwrite twice the L2 before the step, outside its events
            flush.fill_(float(i))
        step(events[i])
    # The K timed steps are captured once into a CUDA graph and replayed, so small
    # layers are not timed as CPU launch latency; eager launches if capture fails.
    graph, launch_mode = None, "eager"
    if args.graph:
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                for i in range(args.steps):
                    timed_step(i)
            graph.replay()  # one untimed replay of the captured steps
            torch.cuda.synchronize()
            launch_mode = "cuda_graph"
        except Exception as exc:  # noqa: BLE001 - report and fall back
            graph, launch_mode = None, f"eager (graph capture failed: {type(exc).__name__})"
            torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        barrier(world)
        torch.cuda.synchronize()
        start.record(stream)
        if graph is not None:
            graph.replay()
        else:
            for i in range(args.steps):
                timed_step(i)
        end.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    total_ms = start.elapsed_time(end)
    stage_ms = {s: float(np.mean([ev[j].elapsed_time(ev[j + 1]) for ev in events])) for j, s in enumerate(STAGES)}
    # per-step times from the first to the last stage event of each step
    step_times = np.array([ev[0].elapsed_time(ev[len(STAGES)]) for ev in events])
    if args.cold_l2:  # the flushes between steps are not the layer's time: sum the steps themselves
        total_ms = float(step_times.sum())
    flags = abi.moe_read_status(view.status)
    max_ms = reduce_max(total_ms, world, device)

    # End to end through the host-buffer entry points: every step copies its x in from
    # pinned host memory, runs the layer and copies its y out. First one batch at a time
    # (moe_layer_forward_host, synchronous); then two batches in flight on two streams
    # (moe_layer_forward_host_async, one workspace and one y buffer per stream), so that
    # one batch's copies run on the copy engines under the other's kernels.
    x_host = inp["x"].cpu().pin_memory()
    fwd_args = (inp["Wg"], inp.get("bias"), w13, w2)
    ws_h = [abi.workspace(cfg, device, host=True) for _ in range(2)]
    y_h = [torch.empty_like(x_host).pin_memory() for _ in range(2)]
    streams = [torch.cuda.Stream(device) for _ in range(2)]
    for _ in range(max(1, args.warmup)):
        abi.moe_layer_forward_host(cfg, x_host, *fwd_args, y_h[0], ws_h[0])
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        abi.moe_layer_forward_host(cfg, x_host, *fwd_args, y_h[0], ws_h[0])
    e2e_sync_s = reduce_max(time.perf_counter() - t0, world, device)
    for i in range(max(2, args.warmup)):
        abi.moe_layer_forward_host_async(cfg, x_host, *fwd_args, y_h[i % 2], ws_h[i % 2], streams[i % 2])
    for st in streams:
        st.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for i in range(args.steps):
        abi.moe_layer_forward_host_async(cfg, x_host, *fwd_args, y_h[i % 2], ws_h[i % 2], streams[i % 2])
    for st in streams:
        st.synchronize()
    e2e_s = reduce_max(time.perf_counter() - t0, world, device)
    del ws_h
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cache = {}
        n_tok = oracle_sample_tokens(w)
        r = oracle_tokens_per_s(w, inp, n_tok, cache=cache)
        # the same oracle on one thread: on the same sample when the all-core run was
        # short, else on a sample scaled down by the core count
        n1 = n_tok if r["seconds"] < 5 else max(1, int(round(n_tok / max(1, r["cores"]))))
        r1 = oracle_tokens_per_s(w, inp, n1, cache=cache, threads=1)
        cpu = {"value": r["value"], "unit": UNIT, "cores": r["cores"], "kind": "oracle",
               "sample": f"{r['tokens']} random tokens of the workload, float64 numpy oracle "
                         f"(route, dispatch, experts, combine), {r['seconds']:.2f} s; expert weights converted "
                         f"to float64 once before timing",
               "single_thread": {"value": r1["value"], "unit": UNIT, "cores": r1["cores"],
                                 "sample": f"{r1['tokens']} random tokens, {r1['seconds']:.2f} s"}}

    if rank != 0:
        return None
    out_bytes = torch.tensor([], dtype=abi.out_dtype(cfg)).element_size()
    dedup = None
    if w.dedup:
        send_counts = ws[view.send_counts - base:view.send_counts - base + 4 * w.D].view(torch.int32).cpu().numpy()
        rows_sent = int(send_counts.sum())
        dedup = {"rows_sent": rows_sent, "ranks_per_token": rows_sent / w.T,
                 "remote_send_bytes": int((rows_sent - send_counts[0]) * w.d * w.act_bytes),
                 "remote_bytes_without_dedup": sizing.remote_dispatch_bytes(rank_offs, w.d, w.act_bytes),
                 "uniform_routing_ranks_per_token": sizing.expected_nodes_touched(w.k, w.D)}
    routed_rows = int(kept[:w.E].sum())
    fp8 = None
    if w.dispatch_dtype == "fp8":
        sent = dedup["rows_sent"] if dedup else routed_rows  # with dedup the FP8 rows are the send rows
        fp8 = {"wire_bytes": sent * fp8_row_bytes(w.d), "bf16_wire_bytes": sent * w.d * 2,
               "ratio": fp8_row_bytes(w.d) / (w.d * 2)}
        if dedup:
            dedup["remote_send_bytes_fp8"] = int((dedup["rows_sent"] - int(send_counts[0])) * fp8_row_bytes(w.d))
    if w.dispatch_dtype == "fp8_gemm":
        sent = dedup["rows_sent"] if dedup else rows  # with dedup the FP8 rows on the wire are the send rows
        fp8 = {"format": "e4m3 codes + one power-of-two scale per row, read as they are by the e4m3 up GEMM",
               "wire_bytes": sent * fp8_row_bytes(w.d, True), "bf16_wire_bytes": sent * w.d * 2,
               "ratio": fp8_row_bytes(w.d, True) / (w.d * 2)}
        if dedup:
            dedup["remote_send_bytes_fp8"] = int((dedup["rows_sent"] - int(send_counts[0])) *
                                                 fp8_row_bytes(w.d, True))
    work = algorithmic(w, rows, out_bytes, abi.hidden_cols(cfg), dedup["rows_sent"] if dedup else 0, routed_rows,
                       active_experts=int((kept > 0).sum()))
    peaks, peak_src = load_peaks()
    value = job_throughput(w.T, args.steps, world, max_ms / 1e3)
    dc_bytes = work["dispatch_bytes"] + work["combine_bytes"]
    dc_moved = work["dispatch_bytes"] + work["combine_bytes_moved"]
    dc_ms = stage_ms["dispatch"] + stage_ms["combine"]
    gemm_ms = stage_ms["expert_up"] + stage_ms["expert_down"]
    gemm_flops = work["up_flops"] + work["down_flops"]
    gemm_bytes = work["up_bytes"] + work["down_bytes"]
    # dominant kernel of the step; a GEMM is tensor-bound when its arithmetic
    # intensity (algorithmic flops / algorithmic bytes) is above the measured ridge
    # point (bf16 peak / HBM bandwidth), else HBM-bound on its weight stream
    ridge = float(peaks["bf16_tflops"]) * 1e12 / (float(peaks["hbm_gbs"]) * 1e9)
    ffn_kernel = abi.moe_ffn_kernel_name(cfg)
    f8g = w.dispatch_dtype == "fp8_gemm"
    # e4m3 up projection: the swapped-pair kernel on FP8; the down projection is the bf16 variant
    down_kernel = abi.moe_ffn_kernel_name(abi.config_for(wl.scaled(w, dispatch_dtype="act"))) if f8g else ffn_kernel
    f8h = w.precision == "fp8_h"
    if f8h:
        down_kernel = ffn_kernel
    up_name = "%s<%s> (up)" % (ffn_kernel, "SwiGLU" if w.expert == "swiglu" else "ReLU")
    # peak of each contraction in its own dtype: e4m3 takes the measured bf16 peak times
    # the nominal fp8 / bf16 ratio (4.5 / 2.25 PFLOP/s dense)
    up_peak_scale = 2.0 if f8g else 1.0
    down_peak_scale = 2.0 if f8h else 1.0

    def gemm_entry(name, flops, nbytes):
        if nbytes and flops / nbytes < ridge:
            return (name, "hbm", nbytes)
        return (name, "tensor", flops)

    # the ridge test in the contraction's own dtype (its peak is up_/down_peak_scale x bf16)
    up_entry = gemm_entry(up_name, work["up_flops"] / up_peak_scale, work["up_bytes"])
    if up_entry[1] == "tensor":
        up_entry = (up_name, "tensor", work["up_flops"])
    down_name = "%s<Plain> (down%s)" % (down_kernel, ", with the h quantization" if f8h else "")
    down_entry = gemm_entry(down_name, work["down_flops"] / down_peak_scale, work["down_bytes"])
    if down_entry[1] == "tensor":
        down_entry = (down_name, "tensor", work["down_flops"])

    kernel_work = {
        "route": ("route_gemm_kernel + route_topk_kernel", "alu", work["route_flops"]),
        "dispatch": ("dispatch (scan+scatter+gather; the router counts)", "hbm", work["dispatch_bytes"]),
        "expert_up": up_entry,
        "expert_down": down_entry,
        "combine": ("combine_kernel", "hbm", work["combine_bytes"]),
    }
    dom = max(STAGES, key=lambda s: stage_ms[s])
    kname, bound, amount = kernel_work[dom]
    dom_s = stage_ms[dom] / 1e3
    if bound == "tensor" and ((dom == "expert_up" and f8g) or (dom == "expert_down" and f8h)):
        peak = float(peaks["bf16_tflops"]) * 2.0
        roof = {"bound": "tensor", "achieved": amount / dom_s / 1e12, "peak": peak, "unit": "TFLOP/s",
                "peak_source": f"{peak_src} bf16 burst x 2 (nominal e4m3 / bf16 dense ratio)"}
    elif bound == "tensor":
        peak = float(peaks["bf16_tflops"])
        roof = {"bound": "tensor", "achieved": amount / dom_s / 1e12, "peak": peak, "unit": "TFLOP/s",
                "peak_source": f"{peak_src} bf16 burst"}
    elif bound == "hbm":
        peak = float(peaks["hbm_gbs"])
        roof = {"bound": "hbm", "achieved": amount / dom_s / 1e9, "peak": peak, "unit": "GB/s",
                "peak_source": f"{peak_src} copy bandwidth"}
    else:
        fp32_peak = 148 * 128 * 2 * float(peaks.get("sm_max_mhz", 2032.0)) * 1e6 / 1e12
        roof = {"bound": "alu", "achieved": amount / dom_s / 1e12, "peak": fp32_peak, "unit": "TFLOP/s",
                "peak_source": "148 SMs x 128 FP32 lanes x 2 flop x max SM clock"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["kernel"] = kname
    roof["algorithmic"] = amount
    roof["ridge_flop_per_byte"] = ridge
    roof["traffic"] = load_traffic(w.name, dom)
    roof["ms_per_launch"] = stage_ms[dom]

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": max_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 up, bf16 down" if f8g else w.act,
        "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "d": w.d, "E": w.E, "k": w.k, "F": w.F, "expert": w.expert,
                   "n_shared": w.n_shared,
                   "capacity": None if cfg.capacity < 0 else int(cfg.capacity), "D_virtual": w.D,
                   "precision": w.precision, "drop_policy": w.drop_policy, "layout": w.layout,
                   "n_groups": w.n_groups, "topk_groups": w.topk_groups, "dedup": w.dedup,
                   "dispatch_dtype": w.dispatch_dtype,
                   "parallelism": f"replicas{world}" if world > 1 else "single-gpu",
                   "l2": ("flushed: %d MB written between timed steps, outside the steps' events; "
                          % (L2_FLUSH_BYTES >> 20) if args.cold_l2 else "") +
                         "inputs larger than L2: the step streams %.2f GB of expert weights and %.0f MB of "
                         "dispatched rows" % (w.n_experts * (w.w13_rows * (1 if f8g else w.act_bytes)
                                                              + w.F * w.act_bytes) * w.d / 1e9
                                              if w.expert != "identity" else 0.0,
                                              rows * w.d * w.act_bytes / 1e6)},
        "roofline": roof,
        "dispatch_combine_gbs": dc_bytes / (dc_ms / 1e3) / 1e9 if dc_ms > 0 else None,
        "dispatch_combine_frac_hbm": (dc_bytes / (dc_ms / 1e3) / 1e9) / float(peaks["hbm_gbs"]) if dc_ms > 0 else None,
        "grouped_gemm_tflops": gemm_flops / (gemm_ms / 1e3) / 1e12 if gemm_ms > 0 and gemm_flops else None,
        "grouped_gemm_frac_bf16_peak": (gemm_flops / (gemm_ms / 1e3) / 1e12) / float(peaks["bf16_tflops"])
        if gemm_ms > 0 and gemm_flops else None,
        # against what the GEMMs can reach at their arithmetic intensity: min(bf16 peak,
        # AI x HBM bandwidth) with AI = algorithmic flops / algorithmic bytes (weights,
        # rows in, rows out)
        "grouped_gemm_frac_attainable": (gemm_flops / (gemm_ms / 1e3) / 1e12) /
        min(float(peaks["bf16_tflops"]), gemm_flops / gemm_bytes * float(peaks["hbm_gbs"]) / 1e3)
        if gemm_ms > 0 and gemm_flops and gemm_bytes else None,
        "grouped_gemm_arith_intensity": gemm_flops / gemm_bytes if gemm_bytes else None,
        "dispatch_combine_bytes": dc_bytes,
        "dispatch_combine_moved": {
            "bytes": dc_moved, "gbs": dc_moved / (dc_ms / 1e3) / 1e9 if dc_ms > 0 else None,
            "frac_hbm": (dc_moved / (dc_ms / 1e3) / 1e9) / float(peaks["hbm_gbs"]) if dc_ms > 0 else None,
            "why": "the bytes the kernels move: the combine reads the expert rows in their stored dtype "
                   "(fp32 with the f32_out precision) instead of the activation dtype"},
        "stage_ms": stage_ms,
        "step_ms": {"median": float(np.median(step_times)), "p95": float(np.percentile(step_times, 95)),
                    "min": float(step_times.min()), "max": float(step_times.max())},
        "routing": {"rows": rows, "rows_computed": rows_computed, "dropped": n_dropped, "near_ties": near_ties,
                    "dedup": dedup,
                    "fp8_dispatch": fp8,
                    "group_limit": [w.topk_groups, w.n_groups] if 0 < w.topk_groups < w.n_groups else None, "hist": sizing.histogram_summary(counts),
                    "rank_imbalance": sizing.imbalance_ratio(np.diff(rank_offs)),
                    "remote_dispatch_bytes": sizing.remote_dispatch_bytes(rank_offs, w.d, w.act_bytes),
                    "pages_dispatch_bytes": sizing.dispatch_bytes_per_direction(w.T, w.slots, w.d, w.act_bytes,
                                                                                w.D if w.D > 1 else None)},
        "device_status": flags,
        "clocks": clocks.summary(),
        "e2e": {"value": job_throughput(w.T, args.steps, world, e2e_s), "unit": UNIT,
                "h2d_bytes_per_step": w.T * w.d * w.act_bytes, "d2h_bytes_per_step": w.T * w.d * w.act_bytes,
                "api": "moe_layer_forward_host_async, two batches in flight on two streams",
                "one_batch_at_a_time": job_throughput(w.T, args.steps, world, e2e_sync_s)},
        "gpu_launches": abi.moe_kernels_per_forward(cfg) * args.steps,
        "launch": launch_mode,
        "cpu_baseline": cpu,
        "versions": versions(device),
    }
    return line


def run_reference(args, w, world, rank):
    """The float64 CPU oracle on bounded token samples of the same workload."""
    if rank != 0:
        return None
    inp = wl.make_inputs(w, seed=0, device="cuda" if torch.cuda.is_available() else "cpu")
    per_step = []
    cache = {}
    tokens = min(args.ref_tokens, oracle_sample_tokens(w))
    # a new token sample every step while every expert's float64 weights fit the cache;
    # otherwise (the DeepSeek-V3 shapes) the same sample each step, so that the weights
    # are converted once
    fits = w.expert == "identity" or w.n_experts * (w.w13_rows + w.F) * w.d * 8 <= 16e9
    for i in range(args.warmup + args.steps):
        r = oracle_tokens_per_s(w, inp, tokens, seed=i if fits else 0, cache=cache)
        if i >= args.warmup:
            per_step.append(r)
    tokens = sum(r["tokens"] for r in per_step)
    secs = sum(r["seconds"] for r in per_step)
    value = tokens / secs
    cores = per_step[0]["cores"]
    sample = (f"each step: {per_step[0]['tokens']} random tokens of the workload "
              f"({'a new sample per step' if fits else 'the same sample every step'}) through the float64 "
              f"numpy oracle (route, dispatch, experts, combine); expert weights converted to float64 once, "
              f"untimed")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": secs / len(per_step) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "d": w.d, "E": w.E, "k": w.k, "F": w.F, "expert": w.expert},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=wl.WORKLOAD_ORDER)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-tokens", type=int, default=8)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", dest="graph", action="store_false",
                    help="launch the timed steps eagerly instead of replaying a CUDA graph")
    ap.add_argument("--cold-l2", action="store_true",
                    help="overwrite 256 MB (twice the L2) before every timed step, outside its events; the "
                         "value then sums the steps' own times")
    ap.add_argument("--drop-policy", choices=["token", "gate"], default=None,
                    help="override the workload's drop policy (capacity workloads)")
    ap.add_argument("--layout", choices=["packed", "padded"], default=None,
                    help="override the workload's row layout (padded needs a capacity)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_env()
    w = wl.WORKLOADS[args.workload]
    changes = {k: v for k, v in (("drop_policy", args.drop_policy), ("layout", args.layout)) if v is not None}
    if changes:
        w = wl.scaled(w, **changes)
    if args.impl == "reference":
        line = run_reference(args, w, world, rank)
    else:
        init_dist(world, local)
        line = run_ours(args, w, world, rank, local)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
