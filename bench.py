"""Benchmark of the AWQ W4A16 linear forward on GB300.

Metric: AWQ W4A16 GEMM throughput -- TFLOP/s and effective weight GB/s
(packed weights + scales + zero points per call) -- over M from 1 to 8192,
with the fraction of each kernel family's roofline.

Default workload (one "step", ``--workload full``): every measured
configuration of the layer, 55 forward calls, group_size 128 unless stated:
  * decode on 7B-class projection shapes: M in {1, 4, 16} x (K, N) in
    {(4096, 4096), (4096, 12288), (4096, 22016), (11008, 4096)}, no bias;
  * prefill on the 7B-class shapes: M in {512, 2048, 8192} x (K, N) in
    {(4096, 12288), (4096, 22016), (11008, 4096)}, bias on M = 512 and 8192;
  * full-row grouping: x [8, 256, 4096] (M = 2048), K = N = 4096,
    group_size -1, with bias;
  * the 70B-class M sweep: (K, N) in {(8192, 10240), (8192, 57344),
    (28672, 8192)} x M in {1, 2, 4, 8, 16, 32, 64, 128, 512, 2048, 8192}.
Every call has its own weight copy (4.9 GB of distinct weights per step, far
more than the 129 MB L2), so each call reads its weights cold.

    python bench.py [--steps K] [--warmup W] [--impl native|reference]
    python bench.py --workload decode-7b | prefill-7b | sweep-70b | fullrow-3d
    python bench.py --sweep --workload all    # per-problem table, every path
    python bench.py --sweep --workload quantize   # awq_quantize_rtn / awq_pack GB/s
    python bench.py --sweep --workload gidx       # g_idx forward: table and sorted (act-order) forms
    python bench.py --sweep --workload shard      # column/row-sharded layer on one GPU

Timing: the calls of a step are grouped by kernel family -- the decode
kernel (HBM-bound) and the tcgen05 paths (tensor-bound) -- and each group is
one CUDA graph of back-to-back launches. The timed region replays K steps
between a barrier + synchronize on both sides, with a CUDA event on the
launching stream before each group's graph and after the last, so every
family's own time inside the timed region is measured, and with it its
roofline fraction. Per-call times (``per_problem``) come from separate graphs
with an event pair around every call, replayed after the timed region.
Clocks are sampled with nvidia-smi during the timed region. Under torchrun
every rank runs the same workload on its own GPU (replicas, weak scaling) and
rank 0 prints one JSON line with the max time over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "AWQ W4A16 GEMM TFLOP/s and weight GB/s vs M (1..8192), % of roofline, 1xGB300"

# DRAM bytes per launch of a kernel family, from one ncu capture of that
# workload (dram__bytes_read.sum + dram__bytes_write.sum, mean over one step's
# launches of the family), valid only while the kernel sources hash to what
# was captured. Keys: (workload, family).
NCU_TRAFFIC = {
    # (workload, family) -> mean DRAM read + write per launch (decode) or per
    # call (tcgen05: the call's launches summed) from one ncu capture of the
    # first eager pass, valid while the kernel sources hash as below
    ("full", "decode"): {
        "bytes_per_launch": 95182626,
        "sources": {
            "bit_weight_quantized_awq_gb300/csrc/awq_decode.cu":
                "04892afcc1dfe943d76ab2e33aa4952a13742311b4d2a0aaa11975962480911b",
            "bit_weight_quantized_awq_gb300/csrc/awq_device.cuh":
                "b046a423a76b51de6cd65483cbd97acc326bc2776db731410fa58a96f2482a61",
        },
        "summary": "profiles/decode_kernel_decode-7b.md (30 decode launches of one pass of the full workload)",
    },
    ("full", "tcgen05"): {
        "bytes_per_launch": 814108508,
        "sources": {
            "bit_weight_quantized_awq_gb300/csrc/awq_prefill.cu":
                "8d5cb8990dee65c09a5da74d86d8c036efcf871663e02b8f5a691edac2a43ed6",
            "bit_weight_quantized_awq_gb300/csrc/awq_tcgen05.cuh":
                "7583bdc482c3f999df48aafe74db217e2c2055ec6f41779622d85db462730d4a",
            "bit_weight_quantized_awq_gb300/csrc/awq_dequant.cu":
                "8062f0eddd6c436eb4452f43d9a64097041ee680fec5a9281620994bd0f23bdf",
            "bit_weight_quantized_awq_gb300/csrc/awq_device.cuh":
                "b046a423a76b51de6cd65483cbd97acc326bc2776db731410fa58a96f2482a61",
        },
        "summary": "profiles/full_step_launches_and_traffic.md (25 calls of one pass, per call)",
    },
}


def ncu_traffic(workload, family):
    """(bytes per launch, note) of the committed capture, or (None, why)."""
    import hashlib
    rec = NCU_TRAFFIC.get((workload, family))
    if rec is None:
        return None, f"no ncu capture of the {family} family on this workload"
    root = os.path.dirname(os.path.abspath(__file__))
    for rel, digest in rec["sources"].items():
        try:
            with open(os.path.join(root, rel), "rb") as f:
                if hashlib.sha256(f.read()).hexdigest() != digest:
                    return None, f"{rel} changed since the capture"
        except OSError:
            return None, f"{rel} not readable"
    return rec["bytes_per_launch"], rec["summary"]

DECODE_SHAPES = [(4096, 4096), (4096, 12288), (4096, 22016), (11008, 4096)]
PREFILL_SHAPES = [(4096, 12288), (4096, 22016), (11008, 4096)]
SWEEP_SHAPES = [(8192, 10240), (8192, 57344), (28672, 8192)]
SWEEP_M = [1, 2, 4, 8, 16, 32, 64, 128, 512, 2048, 8192]

WORKLOADS = {
    # name -> list of (M, K, N, group_size, bias)
    "decode-7b": [(M, K, N, 128, False) for M in (1, 4, 16) for (K, N) in DECODE_SHAPES],
    "prefill-7b": [(M, K, N, 128, M != 2048) for M in (512, 2048, 8192) for (K, N) in PREFILL_SHAPES],
    "fullrow-3d": [(2048, 4096, 4096, -1, True)],
    "sweep-70b": [(M, K, N, 128, False) for (K, N) in SWEEP_SHAPES for M in SWEEP_M],
}
WORKLOADS["full"] = (WORKLOADS["decode-7b"] + WORKLOADS["prefill-7b"] + WORKLOADS["fullrow-3d"]
                     + WORKLOADS["sweep-70b"])
DEFAULT_WORKLOAD = "full"
L2_BYTES = 129 * 1024 * 1024


def weight_bytes(K, N, g):
    g = K if g == -1 else g
    G = K // g
    return K * N // 2 + G * N * 2 + G * N // 2


def algo_bytes(M, K, N, g, bias):
    """Algorithmic HBM bytes of one call: weights + scales + zeros + x + y (+ bias)."""
    return weight_bytes(K, N, g) + 2 * M * K + 2 * M * N + (2 * N if bias else 0)


def flops(M, K, N):
    return 2 * M * K * N


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


# --------------------------------------------------------------------------
# distributed plumbing (replicas: no data-path collective)
# --------------------------------------------------------------------------

def dist_env():
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def aggregate_ranks(elapsed_s: float, units: float, device) -> tuple[float, float]:
    """(max elapsed, summed units) over all ranks; identity without a process
    group. The whole-job number is units of all ranks over the slowest rank."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return elapsed_s, units
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(device):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()
    if device.type == "cuda":
        torch.cuda.synchronize(device)


# --------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 50):
        self.gpu_index, self.interval_ms = gpu_index, interval_ms
        self.proc = self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms={self.interval_ms}"],
                stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], [], set()
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
                for name, v in zip(self.NAMES, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(name)
            except (ValueError, IndexError):
                continue
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------
# native arm
# --------------------------------------------------------------------------

def build_inputs(problems, device, min_bytes):
    """Copies of the workload on the device: each copy gives every problem
    its own weights, x, bias and y; enough copies that one pass over all of
    them reads at least `min_bytes` of distinct weights."""
    from bit_weight_quantized_awq_gb300.synthetic import make_activations, make_problem
    cache = {}
    per_step = sum(weight_bytes(K, N, g) for (M, K, N, g, b) in problems)
    copies = max(1, -(-min_bytes // per_step))
    sets = []
    for _ in range(copies):
        items = []
        for idx, (M, K, N, g, bias) in enumerate(problems):
            key = (K, N, g)
            if key not in cache:
                cache[key] = make_problem(1, K, N, g, bias=True, seed=0)
            w = cache[key]
            items.append({
                "shape": (M, K, N, g, bias),
                "x": make_activations(M, K, seed=1000 + idx).to(device),
                "qweight": w.qweight.to(device),
                "qzeros": w.qzeros.to(device),
                "scales": w.scales.to(device),
                "bias": w.bias.to(device) if bias else None,
                "y": torch.empty((M, N), dtype=torch.float16, device=device),
            })
        sets.append(items)
    return sets


def launch(item, path, stream_handle):
    from bit_weight_quantized_awq_gb300 import awq_linear_forward_path
    M, K, N, g, _ = item["shape"]
    b = item["bias"]
    return awq_linear_forward_path(item["x"].data_ptr(), item["qweight"].data_ptr(),
                                   item["qzeros"].data_ptr(), item["scales"].data_ptr(),
                                   None if b is None else b.data_ptr(), item["y"].data_ptr(),
                                   M, K, N, g, stream_handle, int(path))


def capture_step(items, path, stream, with_events=True):
    """One CUDA graph for one pass over `items`; returns (graph, event pairs)."""
    handle = stream.cuda_stream
    evs = []
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for it in items:
            if with_events:
                e0 = torch.cuda.Event(enable_timing=True, external=True)
                e1 = torch.cuda.Event(enable_timing=True, external=True)
                e0.record(stream)
            st = launch(it, path, handle)
            if st != 0:
                raise RuntimeError(f"launch failed with status {st} for {it['shape']}")
            if with_events:
                e1.record(stream)
                evs.append((e0, e1))
    return graph, evs


def kernels_per_call(M, K, N, g, path_value: int) -> int:
    """Kernel launches one forward call makes on `path_value`, as the library
    plans them (awq_forward_launches: the persistent kernel, the stream-K sum
    kernel when a tile is split, dequant windows)."""
    import bit_weight_quantized_awq_gb300 as awq
    n = awq.awq_forward_launches(M, K, N, g, path_value)
    if n < 0:
        raise RuntimeError(f"no launch plan for M={M} K={K} N={N} g={g} path={path_value}")
    return n


# kernel families of a step: the decode kernel (bound by HBM) and the tcgen05
# paths -- the fused prefill kernel and the dequantise-then-GEMM path, whose
# GEMM core is the same tensor-core pipeline (bound by the tensor cores)
FAMILY_OF_PATH = {1: "generic", 2: "decode", 3: "tcgen05", 4: "tcgen05"}


def call_paths(problems, path):
    """The path every call takes (the library's automatic choice unless a
    path is forced)."""
    import bit_weight_quantized_awq_gb300 as awq
    from bit_weight_quantized_awq_gb300 import Path
    if path != Path.AUTO:
        return [int(path)] * len(problems)
    return [awq.awq_select_path(p[0], p[1], p[2], p[3]) for p in problems]


def group_by_family(paths):
    """[(family, [problem indices])], decode first, in problem order within each."""
    order = ["decode", "generic", "tcgen05"]
    fams = {}
    for i, pth in enumerate(paths):
        fams.setdefault(FAMILY_OF_PATH[pth], []).append(i)
    return [(f, fams[f]) for f in order if f in fams]


def run_native(args, problems, device):
    import bit_weight_quantized_awq_gb300 as awq
    from bit_weight_quantized_awq_gb300 import Path
    awq.load_library()
    path = Path[args.path.upper()]
    paths = call_paths(problems, path)
    fams = group_by_family(paths)
    sets = build_inputs(problems, device, 2 * L2_BYTES)
    stream = torch.cuda.Stream(device)
    handle = stream.cuda_stream
    # eager pass first: allocates the per-stream scratch area before capture
    with torch.cuda.stream(stream):
        for items in sets:
            for it in items:
                st = launch(it, path, handle)
                if st != 0:
                    raise RuntimeError(f"status {st} for {it['shape']}")
    stream.synchronize()
    st = awq.awq_last_device_status(handle)
    if st != 0:
        raise RuntimeError(awq.awq_status_string(st))

    # timed graphs hold nothing but the launches of one family, so that
    # consecutive kernels may overlap as they would in a model (programmatic
    # dependent launch); a second set with an event pair around every launch
    # times each call on its own, after the timed region
    graphs = [[capture_step([items[i] for i in idx], path, stream, False)[0] for (_, idx) in fams]
              for items in sets]
    use_events = True
    try:
        ev_graphs = [[capture_step([items[i] for i in idx], path, stream, True) for (_, idx) in fams]
                     for items in sets]
    except Exception:
        use_events = False
        ev_graphs = []
    # CUDAGraph.replay() launches on the current stream: make it `stream`,
    # the stream the timing events are recorded on
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            for g in graphs[i % len(graphs)]:
                g.replay()
    torch.cuda.synchronize(device)

    nf = len(fams)
    marks = [[torch.cuda.Event(enable_timing=True) for _ in range(nf + 1)] for _ in range(args.steps)]
    ws, rank, local = dist_env()
    barrier(device)
    with ClockSampler(torch.cuda.current_device() if ws == 1 else local) as clk:
        barrier(device)
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                for f, g in enumerate(graphs[i % len(graphs)]):
                    marks[i][f].record(stream)
                    g.replay()
                marks[i][nf].record(stream)
        barrier(device)
    clocks = clk.summary()
    elapsed = marks[0][0].elapsed_time(marks[-1][nf]) / 1e3
    # each family's own time inside the timed region (summed over the steps)
    fam_s = [sum(marks[i][f].elapsed_time(marks[i][f + 1]) for i in range(args.steps)) / 1e3
             for f in range(nf)]

    st = awq.awq_last_device_status(handle)
    if st != 0:
        raise RuntimeError(awq.awq_status_string(st))

    wbytes = sum(weight_bytes(K, N, g) for (M, K, N, g, b) in problems)
    fl = sum(flops(M, K, N) for (M, K, N, g, b) in problems)
    abytes = sum(algo_bytes(*p) for p in problems)
    max_el, tot_wbytes = aggregate_ranks(elapsed, wbytes * args.steps, device)
    _, tot_flops = aggregate_ranks(elapsed, fl * args.steps, device)
    fam_max = [aggregate_ranks(t, 0.0, device)[0] for t in fam_s]

    per_problem = None
    if use_events:
        per_problem = [[] for _ in problems]
        with torch.cuda.stream(stream):
            for rep in range(3):
                for gs in ev_graphs:
                    for (g, _) in gs:
                        g.replay()
                stream.synchronize()
                if rep == 0:
                    continue   # warm-up pass
                for gs in ev_graphs:
                    for (_, evs), (_, idx) in zip(gs, fams):
                        for j, (e0, e1) in zip(idx, evs):
                            per_problem[j].append(e0.elapsed_time(e1) / 1e3)
    launches_per_call = [kernels_per_call(p[0], p[1], p[2], p[3], pth) for p, pth in zip(problems, paths)]
    return {"elapsed": max_el, "tot_wbytes": tot_wbytes, "tot_flops": tot_flops,
            "wbytes": wbytes, "flops": fl, "abytes": abytes, "clocks": clocks,
            "per_problem": per_problem, "copies": len(sets), "graph_events": use_events,
            "paths": paths, "families": fams, "family_s": fam_max,
            "launches_per_call": launches_per_call,
            "launches": args.steps * sum(launches_per_call),
            "sets": sets}


def run_e2e(args, problems, device, sets, steps):
    """The same metric through the public torch API from host buffers. Every
    step copies each call's activations from pinned host memory to the
    device, runs the layer once per problem (`linear_forward`, eager) into
    its slice of a device output buffer, and reads every output back into
    pinned host memory. The copies run on two copy streams and overlap the
    computation, call by call. The device buffers are double-buffered by
    step parity, so a step's input copies wait only for the forwards of two
    steps back that read the same buffer, not for the step before. Events
    order the rest: call j's input copy, its forward and its output copy;
    a forward also waits for the output copy of two steps back that read
    its y buffer."""
    from bit_weight_quantized_awq_gb300 import Path, linear_forward
    items = sets[0]
    x_sizes = [it["x"].numel() for it in items]
    y_sizes = [it["y"].numel() for it in items]
    xh = torch.empty(sum(x_sizes), dtype=torch.float16).pin_memory()
    yh = torch.empty(sum(y_sizes), dtype=torch.float16).pin_memory()
    xd = [torch.empty(sum(x_sizes), dtype=torch.float16, device=device) for _ in range(2)]
    yd = [torch.empty(sum(y_sizes), dtype=torch.float16, device=device) for _ in range(2)]
    xs, ys, xhs, yhs = [[], []], [[], []], [], []
    o = 0
    for it, n in zip(items, x_sizes):
        xh[o:o + n].copy_(it["x"].reshape(-1).cpu())
        for b in range(2):
            xs[b].append(xd[b][o:o + n].view(it["x"].shape))
        xhs.append(xh[o:o + n].view(it["x"].shape))
        o += n
    o = 0
    for it, n in zip(items, y_sizes):
        for b in range(2):
            ys[b].append(yd[b][o:o + n].view(it["y"].shape))
        yhs.append(yh[o:o + n].view(it["y"].shape))
        o += n
    path = Path[args.path.upper()]
    h2d = xh.numel() * 2
    d2h = yh.numel() * 2
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    s_c = torch.cuda.current_stream(device)
    n = len(items)
    ev_in = [[torch.cuda.Event() for _ in range(n)] for _ in range(2)]     # x_j on the device
    ev_c = [[torch.cuda.Event() for _ in range(n)] for _ in range(2)]      # forward j done
    ev_out = [[torch.cuda.Event() for _ in range(n)] for _ in range(2)]    # y_j read back
    used = [False, False]
    step_no = [0]

    def one_step():
        b = step_no[0] & 1
        for j, it in enumerate(items):
            with torch.cuda.stream(s_in):
                if used[b]:
                    s_in.wait_event(ev_c[b][j])
                xs[b][j].copy_(xhs[j], non_blocking=True)
                ev_in[b][j].record(s_in)
            s_c.wait_event(ev_in[b][j])
            if used[b]:
                s_c.wait_event(ev_out[b][j])
            linear_forward(xs[b][j], it["qweight"], it["qzeros"], it["scales"], it["bias"],
                           it["shape"][3], path=path, out=ys[b][j])
            ev_c[b][j].record(s_c)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_c[b][j])
                yhs[j].copy_(ys[b][j], non_blocking=True)
                ev_out[b][j].record(s_out)
        used[b] = True
        step_no[0] += 1

    def drain():
        for st in (s_in, s_c, s_out):
            st.synchronize()

    for _ in range(max(3, args.warmup // 10)):
        one_step()
    drain()
    barrier(device)
    t0 = time.perf_counter()
    for _ in range(steps):
        one_step()
    drain()
    barrier(device)
    return time.perf_counter() - t0, h2d, d2h


# --------------------------------------------------------------------------
# oracle (CPU baseline and reference arm)
# --------------------------------------------------------------------------

def oracle_inputs(problems, cache, idx, col_words=None):
    """(x, qweight, qzeros, scales, bias) of problem `idx` for the oracle, over
    all columns or the first `col_words` packed words, cached."""
    import numpy as np
    from bit_weight_quantized_awq_gb300.synthetic import make_activations, make_problem
    M, K, N, g, bias = problems[idx]
    key = (K, N, g)
    if key not in cache:
        w = make_problem(1, K, N, g, bias=True, seed=0)
        cache[key] = (w.qweight.numpy(), w.qzeros.numpy(), w.scales.numpy(), w.bias.numpy())
    if ("x", idx) not in cache:
        cache[("x", idx)] = make_activations(M, K, seed=1000 + idx).numpy()
    qw, qz, sc, b = cache[key]
    n_words = N // 8 if col_words is None else min(col_words, N // 8)
    skey = ("slice", key, n_words)
    if skey not in cache:
        cache[skey] = (np.ascontiguousarray(qw[:, :n_words]), np.ascontiguousarray(qz[:, :n_words]),
                       np.ascontiguousarray(sc[:, :8 * n_words]), np.ascontiguousarray(b[:8 * n_words]))
    qws, qzs, scs, bs = cache[skey]
    return cache[("x", idx)], qws, qzs, scs, (bs if bias else None)


def oracle_step(problems, cache, col_words=None, which=None, max_rows=None):
    """The oracle on the problems (all of them, or only index `which`), over
    all columns or the first `col_words` packed words, and all rows or the
    first `max_rows`. Returns the flops it performed (2 x rows x K x columns)."""
    import numpy as np
    import oracle
    done = 0
    for idx in (range(len(problems)) if which is None else [which]):
        M, K, N, g, _ = problems[idx]
        x, qws, qzs, scs, bs = oracle_inputs(problems, cache, idx, col_words)
        rows = None if max_rows is None or max_rows >= M else np.arange(max_rows, dtype=np.int64)
        oracle.forward(x, qws, qzs, scs, bs, g, rows=rows)
        done += 2 * (M if rows is None else len(rows)) * K * qws.shape[1] * 8
    return done


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


# fp64 multiply-adds above which a whole step is too slow for the host cores
CPU_FULL_STEP_MACS = 2e10
CPU_SAMPLE_ROWS = 8
CPU_SAMPLE_COL_FRACTION = 8


def cpu_baseline(problems, budget_s=12.0):
    """The oracle on whole steps of the workload (every problem, every row and
    column), repeated until about `budget_s` has passed; TFLOP/s. When a
    whole step holds more than CPU_FULL_STEP_MACS multiply-adds (the prefill
    workloads: hours of fp64 work), every problem runs on its first
    CPU_SAMPLE_ROWS rows and the first 1/CPU_SAMPLE_COL_FRACTION of its
    columns instead, and the time of a whole call is extrapolated from the
    timed dequantisation and the timed rows (both linear in the columns)."""
    import oracle
    oracle.build()
    cache = {}
    oracle_step(problems, cache, col_words=1)   # input generation stays outside the timing
    macs = sum(M * K * N for (M, K, N, _, _) in problems)
    cores, model = os.cpu_count(), cpu_model()
    if macs <= CPU_FULL_STEP_MACS:
        t0 = time.perf_counter()
        done, steps = 0, 0
        while True:
            done += oracle_step(problems, cache)
            steps += 1
            if time.perf_counter() - t0 > budget_s:
                break
        el = time.perf_counter() - t0
        return {"value": done / el / 1e12, "unit": "TFLOP/s", "cores": cores, "cpu_model": model,
                "kind": "oracle",
                "sample": f"{steps} full step(s) of the workload ({len(problems)} problems, all rows "
                          f"and columns), fp64 oracle on {cores} threads ({model}), {el:.1f} s"}
    # T(rows) = T_dequant + rows * T_row: the oracle dequantises W16 once per
    # call, then spends the same time on every row. Both parts are timed.
    import oracle as orc
    t_start = time.perf_counter()
    done, full_s, passes = 0, 0.0, 0
    while True:
        for i, (M, K, N, g, _) in enumerate(problems):
            r = min(M, CPU_SAMPLE_ROWS)
            words = max(1, N // 8 // CPU_SAMPLE_COL_FRACTION)
            _x, qws, qzs, scs, _b = oracle_inputs(problems, cache, i, words)
            t0 = time.perf_counter()
            orc.dequant(qws, qzs, scs, g)
            t_deq = time.perf_counter() - t0
            t0 = time.perf_counter()
            oracle_step(problems, cache, col_words=words, which=i, max_rows=r)
            t_r = time.perf_counter() - t0
            per_row = max(t_r - t_deq, 0.0) / r
            full_s += (t_deq + M * per_row) * (N // 8) / words
            done += flops(M, K, N)
        passes += 1
        if time.perf_counter() - t_start > budget_s:
            break
    el = time.perf_counter() - t_start
    return {"value": done / full_s / 1e12, "unit": "TFLOP/s", "cores": cores, "cpu_model": model,
            "kind": "oracle",
            "sample": f"{passes} pass(es) over the {len(problems)} problems, each on its first "
                      f"{CPU_SAMPLE_ROWS} rows and first 1/{CPU_SAMPLE_COL_FRACTION} of the columns; "
                      f"a whole call extrapolated as (T_dequant + M x (T_rows - T_dequant) / rows) "
                      f"x columns / sampled columns, with the oracle's dequant timed alone; fp64 oracle "
                      f"on {cores} threads ({model}), {el:.1f} s"}


REF_SAMPLE_WORDS = 8      # first 64 output columns
REF_SAMPLE_ROWS = 64      # first 64 rows


def run_reference(args, problems):
    """--impl reference: the oracle on this workload, timed on the host
    cores. Each step is one problem (in rotation) over its first 64 rows and
    its first 8 packed words (64 output columns), so that K + W steps end
    within minutes; TFLOP/s of the work done."""
    import oracle
    oracle.build()
    cache = {}
    kw = dict(col_words=REF_SAMPLE_WORDS, max_rows=REF_SAMPLE_ROWS)
    # inputs of the problems the steps will use, generated outside the timing
    for i in sorted({i % len(problems) for i in range(max(args.steps, args.warmup))}):
        oracle_step(problems, cache, which=i, **kw)
    for i in range(args.warmup):
        oracle_step(problems, cache, which=i % len(problems), **kw)
    t0 = time.perf_counter()
    done = 0
    for i in range(args.steps):
        done += oracle_step(problems, cache, which=i % len(problems), **kw)
    el = time.perf_counter() - t0
    value = done / el / 1e12
    cores, model = os.cpu_count(), cpu_model()
    sample = (f"each step: one of the {len(problems)} problems in rotation, its first {REF_SAMPLE_ROWS} "
              f"rows and first {8 * REF_SAMPLE_WORDS} output columns; fp64 oracle on {cores} threads "
              f"({model})")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "problems": len(problems)},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "cpu_model": model,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


# --------------------------------------------------------------------------
# sweep: per-problem table of every path that can take the shape
# --------------------------------------------------------------------------

def run_sweep(args, device, peaks):
    import bit_weight_quantized_awq_gb300 as awq
    from bit_weight_quantized_awq_gb300 import Path
    awq.load_library()
    out = open(args.sweep_out, "w") if args.sweep_out else None
    names = list(WORKLOADS) if args.workload == "all" else [args.workload]
    stream = torch.cuda.Stream(device)
    handle = stream.cuda_stream
    for wl in names:
        for prob in WORKLOADS[wl]:
            M, K, N, g, bias = prob
            for path in (Path.DECODE, Path.PREFILL, Path.DEQUANT_GEMM, Path.GENERIC):
                if not awq.awq_path_supported(M, K, N, g, path):
                    continue
                if path == Path.GENERIC and flops(M, K, N) > 2e11:
                    continue
                sets = build_inputs([prob], device, 2 * L2_BYTES)
                with torch.cuda.stream(stream):
                    for s in sets:
                        launch(s[0], path, handle)
                stream.synchronize()
                reps = max(3, min(200, int(2e-3 / max(1e-7, flops(M, K, N) / 1e15))))
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph, stream=stream):
                    for r in range(reps):
                        st = launch(sets[r % len(sets)][0], path, handle)
                        if st != 0:
                            raise RuntimeError(f"status {st} capturing {prob} on {path.name}")
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(stream):
                    graph.replay()
                    stream.synchronize()
                    e0.record(stream)
                    graph.replay()
                    e1.record(stream)
                torch.cuda.synchronize(device)
                t = e0.elapsed_time(e1) / 1e3 / reps
                row = {"workload": wl, "M": M, "K": K, "N": N, "g": g, "bias": bias,
                       "path": path.name.lower(), "us": t * 1e6,
                       "tflops": flops(M, K, N) / t / 1e12,
                       "weight_gbs": weight_bytes(K, N, g) / t / 1e9,
                       "hbm_frac": algo_bytes(*prob) / t / 1e9 / peaks["hbm_gbs"],
                       "tc_frac": flops(M, K, N) / t / 1e12 / peaks["bf16_tflops"]}
                print(json.dumps(row), file=sys.stderr, flush=True)
                if out:
                    out.write(json.dumps(row) + "\n")
                    out.flush()
                del sets, graph
                torch.cuda.empty_cache()
    if out:
        out.close()


# --------------------------------------------------------------------------
# sweep of the step before the forward: awq_quantize_rtn and awq_pack
# --------------------------------------------------------------------------

QUANTIZE_SHAPES = DECODE_SHAPES + SWEEP_SHAPES


def run_quantize_sweep(args, device, peaks):
    """Effective GB/s of awq_quantize_rtn (fp16 W + scales + zeros read, packed
    codes written) and awq_pack (one code byte read, half a byte written) on
    the 7B and 70B projection shapes, g = 128, back-to-back launches over two
    copies of the inputs, against the measured HBM copy bandwidth."""
    import bit_weight_quantized_awq_gb300 as awq
    awq.load_library()
    out = open(args.sweep_out, "w") if args.sweep_out else None
    stream = torch.cuda.Stream(device)
    h = stream.cuda_stream
    g = 128
    for (K, N) in QUANTIZE_SHAPES:
        G = K // g
        gen = torch.Generator(device=device).manual_seed(0)
        sets = []
        for _ in range(2):
            W = (torch.randn((K, N), device=device, generator=gen) * 0.02).half()
            sc = (torch.rand((G, N), device=device, generator=gen) * 9e-3 + 1e-3).half()
            qz = torch.randint(-2**31, 2**31 - 1, (G, N // 8), dtype=torch.int32, device=device,
                               generator=gen)
            codes = torch.randint(0, 16, (K, N), dtype=torch.uint8, device=device, generator=gen)
            qw = torch.empty((K, N // 8), dtype=torch.int32, device=device)
            sets.append((W, sc, qz, codes, qw))
        cases = {
            "quantize_rtn": (lambda st: awq.awq_quantize_rtn(st[0].data_ptr(), st[1].data_ptr(),
                                                             st[2].data_ptr(), st[4].data_ptr(),
                                                             K, N, g, h),
                             2 * K * N + 2 * G * N + G * N // 2 + K * N // 2),
            "pack": (lambda st: awq.awq_pack(st[3].data_ptr(), st[4].data_ptr(), K, N, h),
                     K * N + K * N // 2),
        }
        for name, (fn, nbytes) in cases.items():
            with torch.cuda.stream(stream):
                for st in sets:
                    if fn(st) != 0:
                        raise RuntimeError(f"{name} failed on {(K, N)}")
            stream.synchronize()
            reps = 20
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                for r in range(reps):
                    fn(sets[r % 2])
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                graph.replay()
                stream.synchronize()
                e0.record(stream)
                graph.replay()
                e1.record(stream)
            torch.cuda.synchronize(device)
            t = e0.elapsed_time(e1) / 1e3 / reps
            row = {"workload": "quantize", "kernel": name, "K": K, "N": N, "g": g,
                   "us": t * 1e6, "gbs": nbytes / t / 1e9, "hbm_frac": nbytes / t / 1e9 / peaks["hbm_gbs"]}
            print(json.dumps(row), file=sys.stderr, flush=True)
            if out:
                out.write(json.dumps(row) + "\n")
                out.flush()
            del graph
        del sets
        torch.cuda.empty_cache()
    if out:
        out.close()


def run_gidx_sweep(args, device, peaks):
    """The g_idx variant with an act-order table (each group holds 128 rows,
    scattered by a permutation) on 7B-class shapes, two ways: the table read
    as is (awq_linear_forward_gidx: the layer dequantised whole, then the
    GEMM core) and the rows sorted by group once (awq_linear_forward_sorted:
    x's columns gathered, then the grouped kernels). TFLOP/s and the binding
    roofline fraction, back-to-back calls over two weight copies."""
    import bit_weight_quantized_awq_gb300 as awq
    awq.load_library()
    out = open(args.sweep_out, "w") if args.sweep_out else None
    stream = torch.cuda.Stream(device)
    h = stream.cuda_stream
    for (K, N) in [(4096, 12288), (11008, 4096)]:
        G = K // 128
        for M in (1, 16, 512, 2048, 8192):
            gen = torch.Generator(device=device).manual_seed(0)
            sets = []
            for _ in range(2):
                qw = torch.randint(-2**31, 2**31 - 1, (K, N // 8), dtype=torch.int32, device=device, generator=gen)
                qz = torch.randint(-2**31, 2**31 - 1, (G, N // 8), dtype=torch.int32, device=device, generator=gen)
                sc = (torch.rand((G, N), device=device, generator=gen) * 9e-3 + 1e-3).half()
                perm = torch.randperm(K, device=device, generator=gen)
                gi = (torch.arange(K, device=device) // 128)[perm].to(torch.int32).contiguous()
                with torch.cuda.stream(stream):
                    qs, sperm, _ = awq.prepare_act_order(qw, gi, G)
                sets.append((qw, qz, sc, gi, qs, sperm))
            x = torch.randn((M, K), device=device, generator=gen).half()
            y = torch.empty((M, N), device=device, dtype=torch.float16)
            forms = {
                "table": lambda st: awq.awq_linear_forward_gidx(x.data_ptr(), st[0].data_ptr(), st[1].data_ptr(),
                                                                st[2].data_ptr(), st[3].data_ptr(), None,
                                                                y.data_ptr(), M, K, N, G, h),
                "sorted": lambda st: awq.awq_linear_forward_sorted(x.data_ptr(), st[5].data_ptr(), st[4].data_ptr(),
                                                                   st[1].data_ptr(), st[2].data_ptr(), None,
                                                                   y.data_ptr(), M, K, N, 128, h),
            }
            for form, fn in forms.items():
                with torch.cuda.stream(stream):
                    for st in sets:
                        if fn(st) != 0:
                            raise RuntimeError(f"gidx forward ({form}) failed on {(M, K, N)}")
                stream.synchronize()
                reps = max(3, min(50, int(2e-3 / max(1e-7, flops(M, K, N) / 1e15))))
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph, stream=stream):
                    for r in range(reps):
                        fn(sets[r % 2])
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(stream):
                    graph.replay()
                    stream.synchronize()
                    e0.record(stream)
                    graph.replay()
                    e1.record(stream)
                torch.cuda.synchronize(device)
                t = e0.elapsed_time(e1) / 1e3 / reps
                row = {"workload": "gidx", "form": form, "M": M, "K": K, "N": N, "G": G, "us": t * 1e6,
                       "tflops": flops(M, K, N) / t / 1e12,
                       "tc_frac": flops(M, K, N) / t / 1e12 / peaks["bf16_tflops"],
                       "hbm_frac": algo_bytes(M, K, N, 128, False) / t / 1e9 / peaks["hbm_gbs"]}
                print(json.dumps(row), file=sys.stderr, flush=True)
                if out:
                    out.write(json.dumps(row) + "\n")
                    out.flush()
                del graph
            del sets
            torch.cuda.empty_cache()
    if out:
        out.close()


def run_shard_sweep(args, device, peaks):
    """Sharded layer on one GPU (the shards one after another): the 70B-class
    shapes split 2 or 4 ways by columns and by group-aligned rows, against
    the unsharded forward; weight GB/s or TFLOP/s of the whole sharded
    forward, CUDA graph of back-to-back forwards over two weight copies. At
    M = 1 the column shards are timed twice: gathered in place (every shard
    writing its slice of one output) and as separate outputs concatenated."""
    import bit_weight_quantized_awq_gb300 as awq
    from bit_weight_quantized_awq_gb300.shard import (column_parallel_forward, row_parallel_forward,
                                                      split_columns, split_rows)
    awq.load_library()
    out = open(args.sweep_out, "w") if args.sweep_out else None
    stream = torch.cuda.Stream(device)
    g = 128
    for (K, N) in SWEEP_SHAPES:
        for M in (1, 16, 2048):
            gen = torch.Generator(device=device).manual_seed(0)
            G = K // g
            copies = []
            for _ in range(2):
                qw = torch.randint(-2**31, 2**31 - 1, (K, N // 8), dtype=torch.int32, device=device, generator=gen)
                qz = torch.randint(-2**31, 2**31 - 1, (G, N // 8), dtype=torch.int32, device=device, generator=gen)
                sc = (torch.rand((G, N), device=device, generator=gen) * 9e-3 + 1e-3).half()
                b = (torch.randn((N,), device=device, generator=gen) * 0.1).half()
                copies.append((qw, qz, sc, b))
            x = torch.randn((M, K), device=device, generator=gen).half()
            modes = [("unsharded", 1), ("columns", 2), ("columns", 4), ("rows", 2), ("rows", 4)]
            if M == 1:
                # the single-token gather in place against separate outputs
                # concatenated afterwards
                modes[3:3] = [("columns_concat", 2), ("columns_concat", 4)]
            for mode, parts in modes:
                if mode == "unsharded":
                    fns = [lambda c=c: awq.linear_forward(x, c[0], c[1], c[2], c[3], g) for c in copies]
                elif mode == "columns":
                    sh = [split_columns(c[0], c[1], c[2], c[3], parts) for c in copies]
                    fns = [lambda s=s: column_parallel_forward(x, s, g) for s in sh]
                elif mode == "columns_concat":
                    sh = [split_columns(c[0], c[1], c[2], c[3], parts) for c in copies]
                    fns = [lambda s=s: torch.cat([awq.linear_forward(x, *t, g) for t in s], dim=-1) for s in sh]
                else:
                    sh = [(split_rows(c[0], c[1], c[2], g, parts), c[3]) for c in copies]
                    fns = [lambda s=s: row_parallel_forward(x, s[0], s[1]) for s in sh]
                with torch.cuda.stream(stream):
                    for f in fns:
                        f()
                stream.synchronize()
                reps = 10
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph, stream=stream):
                    for r in range(reps):
                        fns[r % 2]()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(stream):
                    graph.replay()
                    stream.synchronize()
                    e0.record(stream)
                    graph.replay()
                    e1.record(stream)
                torch.cuda.synchronize(device)
                t = e0.elapsed_time(e1) / 1e3 / reps
                row = {"workload": "shard", "mode": mode, "parts": parts, "M": M, "K": K, "N": N,
                       "us": t * 1e6, "weight_gbs": weight_bytes(K, N, g) / t / 1e9,
                       "tflops": flops(M, K, N) / t / 1e12,
                       "hbm_frac": algo_bytes(M, K, N, g, True) / t / 1e9 / peaks["hbm_gbs"],
                       "tc_frac": flops(M, K, N) / t / 1e12 / peaks["bf16_tflops"]}
                print(json.dumps(row), file=sys.stderr, flush=True)
                if out:
                    out.write(json.dumps(row) + "\n")
                    out.flush()
                del graph
            del copies
            torch.cuda.empty_cache()
    if out:
        out.close()


# --------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser(description=__doc__,
                                 formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=list(WORKLOADS) + ["all", "quantize", "gidx", "shard"])
    ap.add_argument("--path", default="auto", choices=["auto", "generic", "decode", "prefill", "dequant_gemm"])
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--sweep-out", default=None)
    ap.add_argument("--e2e-steps", type=int, default=0, help="0: about one second of steps")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    ws, rank, local = dist_env()
    if args.impl == "reference":
        if rank == 0:
            run_reference(args, WORKLOADS[args.workload if args.workload in WORKLOADS else DEFAULT_WORKLOAD])
        return

    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", torch.cuda.current_device())
    peaks = load_peaks()

    if args.sweep:
        if args.workload == "quantize":
            run_quantize_sweep(args, device, peaks)
        elif args.workload == "gidx":
            run_gidx_sweep(args, device, peaks)
        elif args.workload == "shard":
            run_shard_sweep(args, device, peaks)
        else:
            run_sweep(args, device, peaks)
        return
    if args.workload in ("quantize", "gidx", "shard"):
        ap.error(f"--workload {args.workload} is a sweep (--sweep)")

    problems = WORKLOADS[args.workload]
    r = run_native(args, problems, device)
    step_s = r["elapsed"] / args.steps
    e2e_steps = args.e2e_steps if args.e2e_steps else max(3, min(200, int(1.0 / max(step_s, 1e-6))))
    e2e_el, h2d, d2h = run_e2e(args, problems, device, r["sets"], e2e_steps)
    e2e_el, e2e_units = aggregate_ranks(e2e_el, r["flops"] * e2e_steps, device)

    paths = r["paths"]
    rooflines = family_rooflines(r, problems, args, peaks)
    # the roofline of the family that takes most of the step's time
    roof = max(rooflines, key=lambda x: x["share_of_step"]) if rooflines else None
    per = None
    if r["per_problem"]:
        per = []
        for p, pth, ts in zip(problems, paths, r["per_problem"]):
            a_s = statistics.mean(ts)
            per.append({"M": p[0], "K": p[1], "N": p[2], "g": p[3], "bias": p[4],
                        "path": FAMILY_OF_PATH.get(pth, "?") if pth != 4 else "dequant_gemm",
                        "us_isolated": round(a_s * 1e6, 3),
                        "tflops": round(flops(p[0], p[1], p[2]) / a_s / 1e12, 2),
                        "weight_gbs": round(weight_bytes(p[1], p[2], p[3]) / a_s / 1e9, 1),
                        "hbm_frac": round(algo_bytes(*p) / a_s / 1e9 / peaks["hbm_gbs"], 4),
                        "tc_frac": round(flops(p[0], p[1], p[2]) / a_s / 1e12 / peaks["bf16_tflops"], 4)})

    line = {
        "metric": METRIC, "value": r["tot_flops"] / r["elapsed"] / 1e12, "unit": "TFLOP/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": r["elapsed"] / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic",
        "config": {"workload": args.workload, "problems": len(problems),
                   "shapes_M_K_N_g_bias": [list(p) for p in problems], "path": args.path,
                   "paths_auto": paths,
                   "l2": f"inputs larger than L2: {r['copies']} weight copies, "
                         f"{r['wbytes'] * r['copies'] / 2**20:.0f} MiB of distinct weights",
                   "parallelism": f"replicas x{ws}",
                   "timing": "one CUDA graph per kernel family per step, replayed back to back; CUDA "
                             "events on the launching stream around every family's graph in the timed "
                             "region; per_problem: separate graphs with an event pair per call, replayed "
                             "after the timed region"},
        "weight_gbs": r["tot_wbytes"] / r["elapsed"] / 1e9,
        "roofline": roof,
        "rooflines": rooflines,
        "per_problem": per,
        "e2e": {"value": e2e_units / e2e_el / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "api": "bit_weight_quantized_awq_gb300.linear_forward, eager; per step and call a "
                       "host-to-device copy of x from pinned memory and a device-to-host copy of y into "
                       "pinned memory, on two copy streams overlapping the computation (device x and y "
                       "double-buffered by step parity)"},
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(problems)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def family_rooflines(r, problems, args, peaks):
    """One roofline block per kernel family of the step, from that family's
    own time inside the timed region: the decode kernel against the measured
    HBM copy bandwidth (algorithmic bytes per launch / average launch
    duration; one launch per decode call), the tcgen05 paths against the
    measured dense bf16 peak (fp16's nominal rate equals bf16's; algorithmic
    flops per call / average call duration, a call being the fused prefill
    kernel or the dequant + GEMM-core pair, with the stream-K sum kernel
    where a tile is split)."""
    out = []
    total = sum(r["family_s"])
    for (fam, idx), t in zip(r["families"], r["family_s"]):
        calls = len(idx) * args.steps
        launches = sum(r["launches_per_call"][i] for i in idx) * args.steps
        traffic, traffic_note = ncu_traffic(args.workload, fam)
        if fam == "decode":
            nbytes = sum(algo_bytes(*problems[i]) for i in idx) * args.steps
            launch_s = t / launches
            achieved = nbytes / launches / launch_s / 1e9
            out.append({"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                        "traffic_source": traffic_note,
                        "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json hbm_gbs)",
                        "kernel": "decode_kernel", "calls_per_step": len(idx),
                        "bytes_per_launch_avg": nbytes / launches, "launch_us_avg": launch_s * 1e6,
                        "share_of_step": t / total,
                        "how": "algorithmic bytes (packed weights + scales + zero points + x + y) per "
                               "launch / (the family's time in the timed region / its launches)"})
        elif fam == "tcgen05":
            fl = sum(flops(*problems[i][:3]) for i in idx) * args.steps
            call_s = t / calls
            tf = fl / calls / call_s / 1e12
            out.append({"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                        "frac": tf / peaks["bf16_tflops"],
                        "frac_of_sustained": tf / peaks["bf16_tflops_sustained"],
                        "traffic": traffic, "traffic_source": traffic_note,
                        "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json bf16_tflops, burst; "
                                       "fp16 = bf16 nominal)",
                        "kernel": "prefill_kernel (fused, or GEMM core after dequant_kernel)",
                        "calls_per_step": len(idx), "launches_per_step": launches // args.steps,
                        "flops_per_call_avg": fl / calls, "call_us_avg": call_s * 1e6,
                        "share_of_step": t / total,
                        "how": "algorithmic flops per call / (the family's time in the timed region / "
                               "its calls)"})
    return out


if __name__ == "__main__":
    main()
