#!/usr/bin/env python3
"""Benchmark of the W4A4 prefill matmul on GB300 (one JSON line on stdout).

Workload (the dense attention-projection GEMM the headline metric is quoted on):
M = 512 tokens (one micro-batch), K = 5120, N = 5120; H32-rotated Q4_0 weights
(bf16 N(0, 0.02) source), fp32 activations N(0, 1) with 1% outlier channels x20.
One step = the whole hot path on one batch: rotate + int4-quantise the
activations, then the block-scaled W4A4 GEMM (fp32 output).  Weight packing runs
once per model and is timed separately.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``--impl reference`` times the CPU oracle (``oracle/``) on the host cores on a
bounded row sample of the same workload.  Under torchrun (N > 1) every rank
runs an independent replica (the path has no exchange step), the step time is
the max over ranks and ``value`` counts the work of all ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth_inputs as si  # noqa: E402

METRIC = "W4A4 GEMM effective TOPS and prefill tok/s at M=512; % of int8 tensor peak"
UNIT = "TOPS"  # effective: 2*M*N*K integer ops per second
L2_BYTES = 129 * 2 ** 20


def env_rank():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("LOCAL_RANK", "0"))


# ----------------------------------------------------------------------------- replicas (N > 1)
def max_over_ranks(ms: float, world: int, device=None) -> float:
    """The slowest replica's time, returned on every rank (all_reduce MAX; the
    process group must be up when world > 1)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replay_steps(first: int, count: int, nsets: int, replay_cycle, replay_one) -> None:
    """Run steps first .. first + count - 1, step i on input set i % nsets: a
    whole cycle of sets (replay_cycle(), sets 0 .. nsets - 1 in order) where one
    starts at set 0 and fits, else one step (replay_one(set index))."""
    i = first
    while count > 0:
        if i % nsets == 0 and count >= nsets:
            replay_cycle()
            i, count = i + nsets, count - nsets
        else:
            replay_one(i % nsets)
            i, count = i + 1, count - 1


def whole_job_value(world: int, ops_per_replica: float, ms_per_step: float) -> float:
    """Throughput of the whole job: the work of all replicas over the slowest one's step time."""
    return world * ops_per_replica / (ms_per_step * 1e-3) / 1e12


def emit(line: dict | None, rank: int) -> bool:
    """Rank 0 alone prints the JSON line."""
    if line is None or rank != 0:
        return False
    print(json.dumps(line), flush=True)
    return True


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []
        self._t = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self) -> dict:
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- oracle arm
def oracle_sample_step(d: dict, wp: dict, rows: np.ndarray) -> float:
    """One oracle pass (activation rotate + quantise, block-scaled product) over `rows`."""
    import oracle
    t0 = time.perf_counter()
    ap = oracle.quantize_activations(d["x"][rows])
    oracle.w4a4_matmul(wp, ap)
    return time.perf_counter() - t0


def cpu_rows_for_budget(d, wp, budget_s: float) -> tuple[np.ndarray, float]:
    """Pick a row sample whose oracle pass takes about budget_s seconds."""
    M = d["x"].shape[0]
    t1 = oracle_sample_step(d, wp, np.arange(1))
    t4 = oracle_sample_step(d, wp, np.arange(4))
    per_row = max((t4 - t1) / 3.0, 1e-4)
    n = int(min(M, max(1, budget_s / per_row)))
    return np.arange(n), per_row


def run_reference(args, shape) -> dict:
    rank, world, _ = env_rank()
    if rank != 0:
        sys.exit(0)
    import oracle
    d = si.dense_inputs(shape.name)
    wp = oracle.pack_weights(d["w_bf16"])
    rows, _ = cpu_rows_for_budget(d, wp, budget_s=6.0)
    for _ in range(args.warmup):
        oracle_sample_step(d, wp, rows)
    times = [oracle_sample_step(d, wp, rows) for _ in range(args.steps)]
    t = sum(times) / len(times)
    ops = 2.0 * len(rows) * shape.N * shape.K
    value = ops / t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int4 codes, f64 block-scaled sum", "data": "synthetic",
        "config": {"workload": shape.what, "M": shape.M, "K": shape.K, "N": shape.N,
                   "sample_rows": int(len(rows))},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                         "sample": f"{len(rows)} of {shape.M} activation rows x all {shape.N} weight rows per step "
                                   f"(numpy; BLAS matmuls threaded over the host cores, elementwise work on one)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return line


# ----------------------------------------------------------------------------- GPU arm
def read_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f)
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "sm_max_mhz": 2070.0, "fallback": True}


def source_digest(*names: str) -> str:
    """sha256 over kernel sources, to tie an ncu traffic figure to the kernel it was taken on."""
    import hashlib
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "hadamard_rotated_w4a4_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(summary: str, sources: tuple[str, ...]) -> tuple[float | None, str]:
    """DRAM bytes per launch recorded in a profiles/ summary, if its kernel sources are unchanged.

    The summary carries the lines ``traffic_bytes_per_launch: <int>`` and
    ``kernel_sources_sha256: <digest>``; a digest that no longer matches the
    sources means the counters describe an older kernel, and the traffic is null.
    """
    p = os.path.join(ROOT, "profiles", summary)
    if not os.path.exists(p):
        return None, f"profiles/{summary} missing"
    kv = {}
    with open(p) as f:
        for line in f:
            line = line.strip().strip("`")
            if ":" in line:
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
    digest = source_digest(*sources)
    if kv.get("kernel_sources_sha256") != digest:
        return None, f"profiles/{summary} was taken on other kernel sources"
    try:
        return float(kv["traffic_bytes_per_launch"]), f"profiles/{summary} (ncu dram__bytes_read+write)"
    except (KeyError, ValueError):
        return None, f"profiles/{summary} has no traffic line"


# the files that define each kernel's device code (the internal host header is left out)
GEMM_SOURCES = ("gemm_tc.cu", "w4a4_device.cuh")
ACT_SOURCES = ("act_quant.cu", "w4a4_device.cuh")


def graph_time(fn, n: int = 20, reps: int = 5) -> float:
    """Device milliseconds per call of fn(i, stream): n calls captured in one CUDA graph,
    the graph replayed `reps` times between CUDA events on the capturing stream (best kept).

    Timing a replayed graph measures the kernels themselves: a Python loop of short
    launches would time the host's launch rate instead.
    """
    import torch
    fn(0, torch.cuda.current_stream())  # any one-time set-up happens outside the capture
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for i in range(n):
                fn(i, s)
    with torch.cuda.stream(s):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = float("inf")
    for _ in range(reps):
        with torch.cuda.stream(s):
            e0.record(s)
            g.replay()
            e1.record(s)
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1) / n)
    return best


def moe_extra(dev) -> dict:
    """The expert-routed workload (1024 tokens, 128 experts, top-8): activation
    quantisation and w4a4_gemm_id for gate/up (K2048 -> N768, activations per
    token) and down (K768 -> N2048, activations per token-slot), device time."""
    import torch
    import hadamard_rotated_w4a4_gb300 as w4
    mi = si.moe_inputs("c4")
    s = mi["shape"]
    ids = torch.from_numpy(np.ascontiguousarray(mi["ids"], dtype=np.int32)).to(dev)
    out = {"workload": s.what}
    for name, wkey, xkey, N, per_slot in (("gate", "wg_bf16", "x_gate", s.N_gate, False),
                                          ("down", "wd_bf16", "x_down", s.N_down, True)):
        w = torch.from_numpy(mi[wkey].reshape(s.E * N, -1).view(np.int16)).to(dev).view(torch.bfloat16)
        wq = w4.h32_q4_0_pack_weights(w)
        del w
        x = torch.from_numpy(mi[xkey]).to(dev)
        K = x.shape[1]
        aq = w4.alloc_act4(x.shape[0], K, dev)
        ws = torch.zeros(w4.w4a4_gemm_id_workspace_bytes(s.M, s.top_k, s.E, K), dtype=torch.uint8, device=dev)
        y = torch.empty(s.M, s.top_k, N, dtype=torch.float32, device=dev)
        act_ms = graph_time(lambda i, st: w4.w4a4_rotate_quantize_act(x, out=aq, stream=st))
        gid_ms = graph_time(lambda i, st: w4.w4a4_gemm_id(wq, s.E, aq, ids, s.top_k, per_slot, y=y, ws=ws, stream=st))
        ops = 2.0 * s.M * s.top_k * N * K
        out[name] = {"K": K, "N": N, "act_ms": act_ms, "gemm_id_ms": gid_ms,
                     "gemm_id_effective_tops": ops / (gid_ms * 1e-3) / 1e12,
                     "weight_mb": s.E * N * K * 0.5625 / 1e6}
        w4.w4a4_gemm_id_status(ws)
        del wq, x, aq, ws, y
    del mi
    torch.cuda.empty_cache()
    return out


def prefill_proxy(dev, stream, nrep: int) -> dict:
    """GEMM-only prefill proxy for one dense layer at 512 tokens.

    A dense layer of the pages' 27B model at hidden 5120 / FFN 17408 runs, per
    512-token micro-batch: 4 attention projections (taken at K5120 N5120),
    gate and up (K5120 N17408) and down (K17408 N5120), with 4 activation
    quantisations (attention input, attention output, FFN input at K5120; FFN
    hidden at K17408).  tok/s = 512 / (sum of those kernel times).  It leaves
    out attention, norms and everything else in a layer: not comparable with
    whole-model prompt rates.
    """
    import torch
    import hadamard_rotated_w4a4_gb300 as w4

    out = {}
    for name, rows in (("c1", 512), ("c2", 512), ("c3", 512)):
        d = si.dense_inputs(name)
        w = torch.from_numpy(d["w_bf16"].view(np.int16)).to(dev).view(torch.bfloat16)
        x = torch.from_numpy(np.ascontiguousarray(d["x"][:rows])).to(dev)
        del d
        N, K = w.shape
        set_bytes = N * K * 1.5 + N * K // 8 + rows * K * 5.5 + rows * N * 4  # incl. both expanded operands
        nsets = max(2, int(np.ceil(2.2 * L2_BYTES / set_bytes)))
        wq0 = w4.h32_q4_0_pack_weights(w)
        del w
        sets = []
        for i in range(nsets):
            wq = w4.alloc_q4_0(N, K, dev)
            wq.codes.copy_(wq0.codes)
            wq.scales_buf.copy_(wq0.scales_buf)
            wq.sums_buf.copy_(wq0.sums_buf)
            if wq.expanded is not None:
                wq.expanded.copy_(wq0.expanded)
            sets.append((wq, x.clone(), w4.alloc_act4(rows, K, dev), torch.empty(rows, N, device=dev)))
        del wq0
        for s_ in sets:
            w4.w4a4_rotate_quantize_act(s_[1], out=s_[2])
        gws = torch.zeros(max(16, w4.w4a4_gemm_workspace_bytes(rows, N, K)), dtype=torch.uint8, device=dev)
        out[name] = {
            "act_ms": graph_time(lambda i, st: w4.w4a4_rotate_quantize_act(sets[i % nsets][1], out=sets[i % nsets][2],
                                                                            stream=st), nrep),
            "gemm_ms": graph_time(lambda i, st: w4.w4a4_gemm(sets[i % nsets][0], sets[i % nsets][2],
                                                             y=sets[i % nsets][3], ws=gws, stream=st), nrep),
        }
        del gws
        del sets
        torch.cuda.empty_cache()
    layer_ms = (4 * out["c1"]["gemm_ms"] + 2 * out["c2"]["gemm_ms"] + out["c3"]["gemm_ms"]
                + 3 * out["c1"]["act_ms"] + out["c3"]["act_ms"])
    return {"value": 512.0 / (layer_ms * 1e-3), "unit": "tok/s per layer", "layer_ms": layer_ms,
            "what": "512 / (4 GEMM K5120xN5120 + 2 GEMM K5120xN17408 + 1 GEMM K17408xN5120 + 3 act K5120 "
                    "+ 1 act K17408), M=512; GEMM-only, not a whole-model rate",
            "kernels_ms": out}


def run_probes() -> dict:
    """int8 / fp8 tensor and fp32 FMA throughput on this GPU (ops/s), via libw4a4_probes.so."""
    import ctypes
    from hadamard_rotated_w4a4_gb300 import build as b
    try:
        b.build(probes=True)
        lib = ctypes.CDLL(b.PROBE_LIB)
    except Exception as e:  # noqa: BLE001
        return {"error": str(e)}
    lib.w4a4_probe_mma_sync.argtypes, lib.w4a4_probe_mma_sync.restype = [ctypes.c_int, ctypes.c_int], ctypes.c_double
    lib.w4a4_probe_ffma.argtypes, lib.w4a4_probe_ffma.restype = [ctypes.c_int, ctypes.c_int], ctypes.c_double
    lib.w4a4_probe_tcgen05_f8.argtypes, lib.w4a4_probe_tcgen05_f8.restype = [ctypes.c_int], ctypes.c_double
    out = {
        "int8_mma_sync_tops": lib.w4a4_probe_mma_sync(0, 4096) / 1e12,
        "fp8_mma_sync_tflops": lib.w4a4_probe_mma_sync(1, 4096) / 1e12,
        "int4_mma_sync_tops": lib.w4a4_probe_mma_sync(2, 4096) / 1e12,
        "fp32_ffma_tflops": lib.w4a4_probe_ffma(0, 20000) / 1e12,
        "fp32_ffma2_tflops": lib.w4a4_probe_ffma(1, 20000) / 1e12,
        "fp8_tcgen05_tflops": lib.w4a4_probe_tcgen05_f8(20000) / 1e12,
    }
    return out


def run_ours(args, shape) -> dict | None:
    import torch
    import hadamard_rotated_w4a4_gb300 as w4

    rank, world, local = env_rank()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device() if world == 1 else local)
    w4.load_library(build_if_missing=True)
    stream = torch.cuda.current_stream()
    M, K, N = shape.M, shape.K, shape.N

    # ---- inputs: one seeded draw, copied into enough sets that a step never finds its inputs in L2
    d = si.dense_inputs(shape.name)
    w_dev = torch.from_numpy(d["w_bf16"].view(np.int16)).to(dev).view(torch.bfloat16)
    x0 = torch.from_numpy(d["x"]).to(dev)
    # per set: fp32 activations, weight codes + scales/sums + expanded operand,
    # activation codes + scales + expanded operand, fp32 output
    set_bytes = M * K * 4 + N * K // 2 + N * K // 16 + N * K + M * K // 2 + M * K // 8 + M * K + M * N * 4
    nsets = max(2, int(np.ceil(2.2 * L2_BYTES / set_bytes)))
    e_pack0, e_pack1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_pack0.record(stream)
    wq0 = w4.h32_q4_0_pack_weights(w_dev)
    e_pack1.record(stream)
    torch.cuda.synchronize()
    pack_ms = e_pack0.elapsed_time(e_pack1)
    # the converter's importance-weighted packing of the same weights (a synthetic
    # importance vector; once per model, like the plain packing)
    imx_ms = None
    if not args.no_exact and world == 1:
        imp = torch.from_numpy(np.random.default_rng(7).uniform(0, 3, K).astype(np.float32) ** 4).to(dev)
        wq_imx = w4.h32_q4_0_pack_weights_imatrix(w_dev, imp)  # warm-up
        e_pack0.record(stream)
        w4.h32_q4_0_pack_weights_imatrix(w_dev, imp, out=wq_imx)
        e_pack1.record(stream)
        torch.cuda.synchronize()
        imx_ms = e_pack0.elapsed_time(e_pack1)
        del wq_imx, imp
    sets = []
    for i in range(nsets):
        wq = w4.alloc_q4_0(N, K, dev)
        wq.codes.copy_(wq0.codes)
        wq.scales_buf.copy_(wq0.scales_buf)
        wq.sums_buf.copy_(wq0.sums_buf)
        if wq.expanded is not None:
            wq.expanded.copy_(wq0.expanded)
        xs = x0.clone()
        aq = w4.alloc_act4(M, K, dev)
        y = torch.empty(M, N, dtype=torch.float32, device=dev)
        sets.append((wq, xs, aq, y))
    del w_dev
    torch.cuda.synchronize()

    gws = torch.zeros(max(16, w4.w4a4_gemm_workspace_bytes(M, N, K)), dtype=torch.uint8, device=dev)

    def step(i, st=None):
        wq, xs, aq, y = sets[i % nsets]
        w4.w4a4_rotate_quantize_act(xs, out=aq, stream=st)
        w4.w4a4_gemm(wq, aq, y=y, ws=gws, stream=st)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    # The timed steps replay CUDA graphs (one per input set, each the step's two
    # kernels) so that the host's per-call cost does not pace the device; the
    # end-to-end steps below go through the public calls one by one.
    # One graph per input set, and one that runs a whole cycle of sets (fewer
    # graph launches between steps); a run of K steps replays whole cycles, then
    # single steps for the remainder, always in set order.
    gstream = torch.cuda.Stream()
    graphs = []
    for i in range(nsets):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(gstream):
            with torch.cuda.graph(g, stream=gstream):
                step(i, gstream)
        graphs.append(g)
    cycle = torch.cuda.CUDAGraph()
    with torch.cuda.stream(gstream):
        with torch.cuda.graph(cycle, stream=gstream):
            for i in range(nsets):
                step(i, gstream)

    def run_steps(first, count):
        replay_steps(first, count, nsets, cycle.replay, lambda k: graphs[k].replay())

    with torch.cuda.stream(gstream):
        run_steps(0, args.warmup)
    torch.cuda.synchronize()

    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index or 0) as clk:
        with torch.cuda.stream(gstream):
            t0.record(gstream)
            run_steps(args.warmup, args.steps)
            t1.record(gstream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    total_ms = t0.elapsed_time(t1)

    # per-kernel device time: each kernel back to back over the same rotating input sets,
    # events only around the loops (on the launching stream)
    # per-kernel device time: each kernel alone, replayed from a CUDA graph over the
    # same rotating input sets (events on the replaying stream)
    nk = max(nsets, 16)
    act_avg = graph_time(lambda i, st: w4.w4a4_rotate_quantize_act(sets[i % nsets][1], out=sets[i % nsets][2],
                                                                    stream=st), nk)
    gemm_avg = graph_time(lambda i, st: w4.w4a4_gemm(sets[i % nsets][0], sets[i % nsets][2], y=sets[i % nsets][3],
                                                     ws=gws, stream=st), nk)
    # the exact path (int8 activations) on the same sets: the pages' comparison
    exact = None
    if not args.no_exact and world == 1:
        a8s = [w4.alloc_act8(M, K, dev) for _ in range(nsets)]
        ws8 = torch.zeros(max(16, w4.w4a8_gemm_workspace_bytes(M, N, K)), dtype=torch.uint8, device=dev)
        act8_avg = graph_time(lambda i, st: w4.w4a8_rotate_quantize_act(sets[i % nsets][1], out=a8s[i % nsets],
                                                                         stream=st), nk)
        gemm8_avg = graph_time(lambda i, st: w4.w4a8_gemm(sets[i % nsets][0], a8s[i % nsets], y=sets[i % nsets][3],
                                                          ws=ws8, stream=st), nk)
        exact = {"what": "rotated Q4_0 x int8 activations (the pages' exact path), same workload",
                 "act_ms": act8_avg, "gemm_ms": gemm8_avg,
                 "gemm_effective_tops": 2.0 * M * N * K / (gemm8_avg * 1e-3) / 1e12,
                 "w4a4_speedup": (act8_avg + gemm8_avg) / (act_avg + gemm_avg)}
        del a8s, ws8
    # the rotate-only route (bf16 activations, not quantised) on the same sets
    rotate_only = None
    if not args.no_exact and world == 1:
        a16s = [w4.alloc_act16(M, K, dev) for _ in range(nsets)]
        ws16 = torch.zeros(max(16, w4.w4a16_gemm_workspace_bytes(M, N, K)), dtype=torch.uint8, device=dev)
        act16_avg = graph_time(lambda i, st: w4.w4a16_rotate_act(sets[i % nsets][1], out=a16s[i % nsets], stream=st),
                               nk)
        gemm16_avg = graph_time(lambda i, st: w4.w4a16_gemm(sets[i % nsets][0], a16s[i % nsets],
                                                            y=sets[i % nsets][3], ws=ws16, stream=st), nk)
        rotate_only = {"what": "rotated Q4_0 x rotated bf16 activations, not quantised (the pages' rotate-only "
                               "route), same workload",
                       "act_ms": act16_avg, "gemm_ms": gemm16_avg,
                       "gemm_effective_tops": 2.0 * M * N * K / (gemm16_avg * 1e-3) / 1e12,
                       "w4a4_speedup": (act16_avg + gemm16_avg) / (act_avg + gemm_avg)}
        del a16s, ws16
    # a drafter's verification batch: the first 8 tokens of the workload
    verify = None
    if not args.no_verify and world == 1:
        x8 = sets[0][1][:8].contiguous()
        a4v = w4.w4a4_rotate_quantize_act(x8)
        y8 = torch.empty(8, N, dtype=torch.float32, device=dev)
        wsv = torch.zeros(max(16, w4.w4a4_gemm_workspace_bytes(8, N, K)), dtype=torch.uint8, device=dev)
        tc_ms = graph_time(lambda i, st: w4.w4a4_gemm(sets[i % nsets][0], a4v, y=y8, ws=wsv, stream=st), nk)
        sm_ms = graph_time(lambda i, st: w4.w4a4_gemm_small_m(sets[i % nsets][0], a4v, y=y8, stream=st), nk)
        wbytes = N * K // 2 + N * (K // 32) * 2
        verify = {"what": "8-token verification batch, same weights", "tensor_core_ms": tc_ms, "small_m_ms": sm_ms,
                  "small_m_weight_gbs": wbytes / (sm_ms * 1e-3) / 1e9}
        del x8, a4v, y8, wsv
    w4.w4a4_check()
    total_ms = max_over_ranks(total_ms, world, dev)
    ms_per_step = total_ms / args.steps
    ops = 2.0 * M * N * K
    value = whole_job_value(world, ops, ms_per_step)

    # ---- end to end through the public API: host activations in, host output back, every step.
    # Each step copies its own fp32 activations in from pinned host memory and reads its
    # fp32 result back.  The copies run on their own streams with two device buffers each,
    # so step i's kernels overlap the input copy of step i + 1 and the read-back of step
    # i - 1 (events order every buffer's reuse).
    x_host = torch.from_numpy(d["x"]).pin_memory()
    y_hosts = [torch.empty(M, N, dtype=torch.float32).pin_memory() for _ in range(2)]
    wq_e, aq_e = sets[0][0], sets[0][2]
    xbufs = [sets[0][1], sets[1][1]]
    ybufs = [sets[0][3], sets[1][3]]
    s_in, s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i):
        j = i % 2
        s_in.wait_event(ev_cmp[j])  # step i - 2 has finished reading this input buffer
        with torch.cuda.stream(s_in):
            xbufs[j].copy_(x_host, non_blocking=True)
        ev_in[j].record(s_in)
        s_cmp.wait_event(ev_in[j])
        s_cmp.wait_event(ev_out[j])  # step i - 2's result has been read back from this buffer
        w4.w4a4_rotate_quantize_act(xbufs[j], out=aq_e, stream=s_cmp)
        w4.w4a4_gemm(wq_e, aq_e, y=ybufs[j], ws=gws, stream=s_cmp)
        ev_cmp[j].record(s_cmp)
        s_out.wait_event(ev_cmp[j])
        with torch.cuda.stream(s_out):
            y_hosts[j].copy_(ybufs[j], non_blocking=True)
        ev_out[j].record(s_out)

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(s_in)
    for i in range(args.steps):
        e2e_step(i)
    for st in (s_in, s_cmp):
        a1_wait = torch.cuda.Event()
        a1_wait.record(st)
        s_out.wait_event(a1_wait)
    a1.record(s_out)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e2e_ms = max_over_ranks(a0.elapsed_time(a1), world, dev) / args.steps
    e2e_value = whole_job_value(world, ops, e2e_ms)
    # the results read back are the device results of the last two steps
    assert torch.equal(y_hosts[(args.steps - 1) % 2], ybufs[(args.steps - 1) % 2].cpu())

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return None

    peaks = read_peaks()
    probes = run_probes() if not args.no_probes else {}
    B = K // 32
    a_exp = sets[0][2].expanded is not None and wq0.expanded is not None
    # GEMM roofline: the per-block scale fold on the fp32 pipe.  Per (m, n, block) it
    # takes two fp32-pipe operations (the product by d_w, with the offset correction
    # folded in, and the fused multiply-add with d_a): 4 flops in the FMA convention.
    fold_flops = 4.0 * M * N * B
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
    fp32_peak = sm_count * 128 * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
    gemm_traffic, gemm_traffic_src = profiled_traffic(f"gemm_tc_{shape.name}.md", GEMM_SOURCES)
    act_traffic, act_traffic_src = profiled_traffic(f"act_rotate_quantize_{shape.name}.md", ACT_SOURCES)
    gemm_roof = {"bound": "alu", "achieved": fold_flops / (gemm_avg * 1e-3) / 1e12, "peak": fp32_peak,
                 "unit": "TFLOP/s", "frac": None, "traffic": gemm_traffic, "traffic_source": gemm_traffic_src,
                 # each operand read as its expanded form (1 byte per element) when the GEMM uses it, else as codes
                 "algorithmic_bytes": float((N * K if wq0.expanded is not None else N * K // 2) + N * B * 4
                                            + (M * K if a_exp else M * K // 2) + M * B * 4 + M * N * 4),
                 "kernel": "w4a4_gemm_tc_kernel",
                 "peak_source": f"derived: {sm_count} SMs x 128 fp32 lanes x 2 flops x {peaks.get('sm_max_mhz', 2070.0)} MHz"}
    gemm_roof["frac"] = gemm_roof["achieved"] / gemm_roof["peak"]
    # fp32 in; codes, scales and (when allocated) the expanded operand out
    act_bytes = M * K * 4 + M * K // 2 + M * B * 4 + (M * K if a_exp else 0)
    act_roof = {"bound": "hbm", "achieved": act_bytes / (act_avg * 1e-3) / 1e9, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "kernel": "act_rotate_quantize_kernel", "traffic": act_traffic,
                "traffic_source": act_traffic_src, "algorithmic_bytes": float(act_bytes),
                "peak_source": "MEASURED_PEAKS.json hbm_gbs (measured)" if not peaks.get("fallback") else "fallback"}
    act_roof["frac"] = act_roof["achieved"] / act_roof["peak"]
    eff_tops_gemm = ops / (gemm_avg * 1e-3) / 1e12
    int8_peak = probes.get("int8_mma_sync_tops") if probes else None
    proxy = None
    if not args.no_proxy and world == 1:
        proxy = prefill_proxy(dev, stream, 16)
    moe = None
    if not args.no_moe and world == 1:
        moe = moe_extra(dev)

    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        wp = oracle.pack_weights(d["w_bf16"])
        rows, _ = cpu_rows_for_budget(d, wp, budget_s=args.cpu_budget)
        tc = oracle_sample_step(d, wp, rows)
        cpu = {"value": 2.0 * len(rows) * N * K / tc / 1e12, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"{len(rows)} of {M} activation rows x all {N} weight rows, one pass "
                         f"(numpy; BLAS matmuls threaded, elementwise single-threaded)", "seconds": tc}

    clocks = clk.summary()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "s4", "data": "synthetic",
        "config": {"workload": shape.what, "M": M, "K": K, "N": N,
                   "l2": f"inputs larger than L2: {nsets} input sets ({nsets * set_bytes / 2**20:.0f} MiB) "
                         f"rotated across steps", "launch": "CUDA-graph replays: whole cycles of the input sets (two kernels per step), single steps for the rest",
                   "parallelism": "replicas" if world > 1 else "single"},
        "roofline": gemm_roof,
        "roofline_act": act_roof,
        "gemm_effective_tops": eff_tops_gemm,
        "pct_int8_peak": (eff_tops_gemm / int8_peak) if int8_peak else None,
        "prefill_tok_s_proxy": proxy,
        "moe": moe,
        "exact_path": exact,
        "rotate_only": rotate_only,
        "verification_batch": verify,
        "kernel_ms": {"act_rotate_quantize": act_avg, "gemm": gemm_avg},
        "pack_weights_ms": pack_ms,
        "pack_weights_imatrix_ms": imx_ms,
        "probes": probes,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": int(M * K * 4),
                "d2h_bytes_per_step": int(M * N * 4), "ms_per_step": e2e_ms,
                "copies": "every step: pinned H2D of its fp32 activations, D2H of its fp32 output; "
                          "copy and compute streams overlap adjacent steps"},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
    }
    if world > 1:
        torch.distributed.destroy_process_group()
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="c1", choices=["c1", "c2", "c3"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-probes", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--no-proxy", action="store_true", help="skip the per-layer prefill proxy")
    ap.add_argument("--no-moe", action="store_true", help="skip the expert-routed workload timing")
    ap.add_argument("--no-exact", action="store_true", help="skip the exact-path (int8 activations) timing")
    ap.add_argument("--no-verify", action="store_true", help="skip the 8-token verification-batch timing")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    shape = si.DENSE[args.config]
    line = run_reference(args, shape) if args.impl == "reference" else run_ours(args, shape)
    emit(line, env_rank()[0])


if __name__ == "__main__":
    main()
