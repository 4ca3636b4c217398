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
import datetime
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
    """Samples nvidia-smi clocks and throttle reasons (every 100 ms) while kernels run.

    Each sample carries nvidia-smi's own timestamp; ``summary(t0, t1)`` keeps the
    samples taken between two host wall-clock times (the load window)."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[tuple[float, str]] = []
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
            self.lines.append((time.time(), line.strip()))

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    @staticmethod
    def parse(lines, t0: float | None = None, t1: float | None = None) -> dict:
        """Median SM clock, max clock and the throttle reasons seen in the samples
        read between host times t0 and t1 (all samples when not given)."""
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t_read, ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 10:
                continue
            try:  # nvidia-smi's own time of the sample (local time); the read time if unparsable
                t = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                t = t_read
            if (t0 is not None and t < t0) or (t1 is not None and t > t1):
                continue
            try:
                sm.append(float(parts[2]))
                smax.append(float(parts[3]))
                power.append(float(parts[4]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[6:10]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_median": statistics.median(power)}

    def summary(self, t0: float | None = None, t1: float | None = None) -> dict:
        return self.parse(self.lines, t0, t1)


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


def fold_peak_tflops(peaks: dict, sm_count: int) -> float:
    """fp32-pipe peak in the FMA convention (2 flops per FMA): SMs x 128 lanes x 2 x max SM clock."""
    return sm_count * 128 * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12


def gemm_algorithmic_bytes(w_rows: int, K: int, a_rows: int, y_rows: int, N: int) -> int:
    """The GEMM's algorithmic HBM bytes: weight codes + fp16 scales, activation codes + fp32
    scales, fp32 output (the expanded operands and the block sums are derived copies, left out)."""
    B = K // 32
    return w_rows * K // 2 + w_rows * B * 2 + a_rows * K // 2 + a_rows * B * 4 + y_rows * N * 4


def act_algorithmic_bytes(M: int, K: int) -> int:
    """The activation kernel's algorithmic HBM bytes: fp32 in, int4 codes + fp32 scales out."""
    return M * K * 4 + M * K // 2 + M * (K // 32) * 4


def gemm_roofline(ms: float, pairs: int, K: int, hbm_bytes: int, peaks: dict, sm_count: int) -> dict:
    """Both bounds of a GEMM launch: the scale fold on the fp32 pipe (2 FMAs = 4 flops per
    output and block) and the algorithmic bytes against the measured copy bandwidth."""
    fold_flops = 4.0 * pairs * (K // 32)
    fpk = fold_peak_tflops(peaks, sm_count)
    fold = fold_flops / (ms * 1e-3) / 1e12
    gbs = hbm_bytes / (ms * 1e-3) / 1e9
    return {"ms": ms, "effective_tops": 2.0 * pairs * K / (ms * 1e-3) / 1e12,
            "fold": {"achieved": fold, "peak": fpk, "unit": "TFLOP/s", "frac": fold / fpk,
                     "work": "2 fp32 FMAs (4 flops) per output and 32-block"},
            "hbm": {"algorithmic_bytes": hbm_bytes, "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": gbs / peaks["hbm_gbs"]}}


def act_roofline(ms: float, M: int, K: int, peaks: dict, expanded: bool) -> dict:
    b = act_algorithmic_bytes(M, K)
    gbs = b / (ms * 1e-3) / 1e9
    return {"ms": ms, "algorithmic_bytes": b, "expanded_write_bytes": M * K if expanded else 0,
            "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"]}


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
GEMM_SOURCES = ("gemm_grp.cu", "tc_ptx.cuh", "w4a4_device.cuh")
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


def act_time(dev, x0, expanded: bool, nrep: int = 20) -> float:
    """Device milliseconds per activation-kernel call on x0's shape, over input and
    output sets that together exceed L2 by 2.2x (the kernel touches nothing else)."""
    import torch
    import hadamard_rotated_w4a4_gb300 as w4
    M, K = x0.shape
    touched = M * K * 4 + M * K // 2 + M * (K // 32) * 4 + (M * K if expanded else 0)
    nsets = max(2, int(np.ceil(2.2 * L2_BYTES / touched)))
    xs = [x0.clone() for _ in range(nsets)]
    outs = [w4.alloc_act4(M, K, dev, expanded=expanded) for _ in range(nsets)]
    ms = graph_time(lambda i, st: w4.w4a4_rotate_quantize_act(xs[i % nsets], out=outs[i % nsets], stream=st), nrep)
    del xs, outs
    torch.cuda.empty_cache()
    return ms


def verify_extra(dev, name: str, peaks: dict | None = None, nrep: int = 20) -> dict:
    """A drafter's 8-token verification batch on a dense config's weights: the
    general GEMM (whole-tile schedule) and the small-M kernel, each replayed from a
    CUDA graph over weight sets that together exceed L2."""
    import torch
    import hadamard_rotated_w4a4_gb300 as w4
    peaks = peaks or read_peaks()
    d = si.dense_inputs(name)
    w = torch.from_numpy(d["w_bf16"].view(np.int16)).to(dev).view(torch.bfloat16)
    x8 = torch.from_numpy(np.ascontiguousarray(d["x"][:8])).to(dev)
    del d
    N, K = w.shape
    wq0 = w4.h32_q4_0_pack_weights(w)
    del w
    wbytes = N * K // 2 + N * (K // 32) * 2
    nsets = max(2, int(np.ceil(2.2 * L2_BYTES / wbytes)))
    sets = []
    for _ in range(nsets):
        wq = w4.alloc_q4_0(N, K, dev)
        wq.codes.copy_(wq0.codes)
        wq.scales_buf.copy_(wq0.scales_buf)
        wq.sums_buf.copy_(wq0.sums_buf)
        sets.append(wq)
    del wq0
    a4v = w4.w4a4_rotate_quantize_act(x8)
    y8 = torch.empty(8, N, dtype=torch.float32, device=dev)
    wsv = torch.zeros(max(16, w4.w4a4_gemm_workspace_bytes(8, N, K)), dtype=torch.uint8, device=dev)
    tc_ms = graph_time(lambda i, st: w4.w4a4_gemm(sets[i % nsets], a4v, y=y8, ws=wsv, stream=st), nrep)
    sm_ms = graph_time(lambda i, st: w4.w4a4_gemm_small_m(sets[i % nsets], a4v, y=y8, stream=st), nrep)
    gbs = wbytes / (sm_ms * 1e-3) / 1e9
    out = {"what": f"8-token verification batch on the {name} weights (K{K} N{N})", "tensor_core_ms": tc_ms,
           "small_m_ms": sm_ms, "small_m_weight_gbs": gbs,
           "roofline": {"bound": "hbm", "algorithmic_bytes": wbytes, "achieved": gbs, "peak": peaks["hbm_gbs"],
                        "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"]},
           "l2": f"{nsets} weight sets rotated"}
    del sets, a4v, y8, wsv
    torch.cuda.empty_cache()
    return out


def moe_extra(dev, peaks: dict | None = None) -> dict:
    """The expert-routed workload (1024 tokens, 128 experts, top-8): activation
    quantisation and w4a4_gemm_id for gate/up (K2048 -> N768, activations per
    token) and down (K768 -> N2048, activations per token-slot), device time."""
    import torch
    import hadamard_rotated_w4a4_gb300 as w4
    mi = si.moe_inputs("c4")
    s = mi["shape"]
    peaks = peaks or read_peaks()
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
    ids = torch.from_numpy(np.ascontiguousarray(mi["ids"], dtype=np.int32)).to(dev)
    out = {"workload": s.what}
    for name, wkey, xkey, N, per_slot in (("gate", "wg_bf16", "x_gate", s.N_gate, False),
                                          ("down", "wd_bf16", "x_down", s.N_down, True)):
        w = torch.from_numpy(mi[wkey].reshape(s.E * N, -1).view(np.int16)).to(dev).view(torch.bfloat16)
        wq0 = w4.h32_q4_0_pack_weights(w)
        del w
        x0 = torch.from_numpy(mi[xkey]).to(dev)
        K = x0.shape[1]
        # two input sets (weights, activations, output), each above 129 MB, rotated across calls
        sets = []
        for _ in range(2):
            wq = w4.alloc_q4_0(s.E * N, K, dev)
            wq.codes.copy_(wq0.codes)
            wq.scales_buf.copy_(wq0.scales_buf)
            wq.sums_buf.copy_(wq0.sums_buf)
            # the routed product reads the int4 codes: no expanded activation operand
            sets.append((wq, x0.clone(), w4.alloc_act4(x0.shape[0], K, dev, expanded=False),
                         torch.empty(s.M, s.top_k, N, dtype=torch.float32, device=dev)))
        del wq0, x0
        ws = torch.zeros(w4.w4a4_gemm_id_workspace_bytes(s.M, s.top_k, s.E, K), dtype=torch.uint8, device=dev)
        act_ms = act_time(dev, sets[0][1], expanded=False)
        gid_ms = graph_time(lambda i, st: w4.w4a4_gemm_id(sets[i % 2][0], s.E, sets[i % 2][2], ids, s.top_k, per_slot,
                                                          y=sets[i % 2][3], ws=ws, stream=st))
        aq = sets[0][2]
        ops = 2.0 * s.M * s.top_k * N * K
        a_rows = s.M * s.top_k if per_slot else s.M
        out[name] = {"K": K, "N": N, "act_ms": act_ms, "gemm_id_ms": gid_ms,
                     "gemm_id_effective_tops": ops / (gid_ms * 1e-3) / 1e12,
                     "weight_mb": s.E * N * K * 0.5625 / 1e6,
                     "l2": "GEMM: 2 input sets rotated, each larger than L2; activation kernel: its own "
                           "input/output sets, together 2.2x L2",
                     "roofline": gemm_roofline(gid_ms, s.M * s.top_k * N, K,
                                               gemm_algorithmic_bytes(s.E * N, K, a_rows, s.M * s.top_k, N),
                                               peaks, sm_count),
                     "act_roofline": act_roofline(act_ms, a_rows, K, peaks, aq.expanded is not None)}
        w4.w4a4_gemm_id_status(ws)
        del sets, aq, ws
    del mi
    torch.cuda.empty_cache()
    return out


def time_dense(dev, name: str, rows: int, nrep: int) -> dict:
    """Device times of the activation kernel and the GEMM on the first `rows` tokens of a
    dense config, each replayed from a CUDA graph over input sets that together exceed L2."""
    import torch
    import hadamard_rotated_w4a4_gb300 as w4

    d = si.dense_inputs(name)
    w = torch.from_numpy(d["w_bf16"].view(np.int16)).to(dev).view(torch.bfloat16)
    x = torch.from_numpy(np.ascontiguousarray(d["x"][:rows])).to(dev)
    del d
    N, K = w.shape
    set_bytes = N * K // 2 + N * K // 8 + rows * K * 5.5 + rows * N * 4  # codes, scales/sums, activations, Y
    nsets = max(2, int(np.ceil(2.2 * L2_BYTES / set_bytes)))
    wq0 = w4.h32_q4_0_pack_weights(w)
    del w
    sets = []
    for _ in range(nsets):
        wq = w4.alloc_q4_0(N, K, dev)
        wq.codes.copy_(wq0.codes)
        wq.scales_buf.copy_(wq0.scales_buf)
        wq.sums_buf.copy_(wq0.sums_buf)
        sets.append((wq, x.clone(), w4.alloc_act4(rows, K, dev), torch.empty(rows, N, device=dev)))
    del wq0
    for s_ in sets:
        w4.w4a4_rotate_quantize_act(s_[1], out=s_[2])
    gws = torch.zeros(max(16, w4.w4a4_gemm_workspace_bytes(rows, N, K)), dtype=torch.uint8, device=dev)
    out = {
        "M": rows, "K": K, "N": N,
        "act_ms": act_time(dev, x, expanded=True, nrep=nrep),
        "gemm_ms": graph_time(lambda i, st: w4.w4a4_gemm(sets[i % nsets][0], sets[i % nsets][2],
                                                         y=sets[i % nsets][3], ws=gws, stream=st), nrep),
    }
    del gws, sets
    torch.cuda.empty_cache()
    return out


def prefill_proxy(dev, nrep: int) -> tuple[dict, dict]:
    """GEMM-only prefill proxy for one dense layer at 512 tokens, and the full-size c3 times.

    A dense layer of the pages' 27B model at hidden 5120 / FFN 17408 runs, per
    512-token micro-batch: 4 attention projections (taken at K5120 N5120),
    gate and up (K5120 N17408) and down (K17408 N5120), with 4 activation
    quantisations (attention input, attention output, FFN input at K5120; FFN
    hidden at K17408).  tok/s = 512 / (sum of those kernel times).  It leaves
    out attention, norms and everything else in a layer: not comparable with
    whole-model prompt rates.
    """
    out = {name: time_dense(dev, name, 512, nrep) for name in ("c1", "c2", "c3")}
    layer_ms = (4 * out["c1"]["gemm_ms"] + 2 * out["c2"]["gemm_ms"] + out["c3"]["gemm_ms"]
                + 3 * out["c1"]["act_ms"] + out["c3"]["act_ms"])
    proxy = {"value": 512.0 / (layer_ms * 1e-3), "unit": "tok/s per layer", "layer_ms": layer_ms,
             "what": "512 / (4 GEMM K5120xN5120 + 2 GEMM K5120xN17408 + 1 GEMM K17408xN5120 + 3 act K5120 "
                     "+ 1 act K17408), M=512; GEMM-only, not a whole-model rate",
             "kernels_ms": out}
    return proxy, {"c2": out["c2"], "c3": time_dense(dev, "c3", si.DENSE["c3"].M, nrep)}


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


def run_pipeline_probes() -> dict:
    """Latency and rate probes behind the super-tile GEMM's design (single CTA, clock64
    cycles): back-to-back tcgen05 MMA issue, TMEM load + wait, the bare MMA-to-fold
    barrier handshake, and the fold loop alone.  A profiling aid, not in the bench line."""
    import ctypes
    from hadamard_rotated_w4a4_gb300 import build as b
    b.build(probes=True)
    lib = ctypes.CDLL(b.PROBE_LIB)
    lib.w4a4_probe_mma_rate.argtypes = [ctypes.c_int] * 4 + [ctypes.POINTER(ctypes.c_double)]
    lib.w4a4_probe_tmem_ld.argtypes, lib.w4a4_probe_tmem_ld.restype = [ctypes.c_int] * 3, ctypes.c_double
    lib.w4a4_probe_pipe.argtypes, lib.w4a4_probe_pipe.restype = [ctypes.c_int] * 2, ctypes.c_double
    lib.w4a4_probe_fold.argtypes, lib.w4a4_probe_fold.restype = [ctypes.c_int] * 2, ctypes.c_double
    out = {}
    for n in (64, 128, 256):
        for name, flags in (("no_swizzle", 8), ("sw128", 8 | 256)):
            o = (ctypes.c_double * 2)()
            rc = lib.w4a4_probe_mma_rate(n, 1, 2000, flags, o)
            out[f"mma_issue_cycles_n{n}_{name}"] = o[1] if rc == 0 else None
    for x8, nm in ((0, "x4"), (1, "x8")):
        out[f"tmem_ld_wait_cycles_16x256b_{nm}_8warps"] = lib.w4a4_probe_tmem_ld(x8, 8, 2000)
    out["handshake_cycles_per_block_n256_2buf"] = lib.w4a4_probe_pipe(2000, 1)
    for mode, nm in ((0, "8warps"), (1, "8warps_no_tmem_loads"), (2, "8warps_no_scale_loads"),
                     (3, "8warps_fma_only"), (4, "16warps")):
        out[f"fold_cycles_per_128x256_block_{nm}"] = lib.w4a4_probe_fold(2000, mode)
    lib.w4a4_probe_fold_mma.argtypes = [ctypes.c_int] * 3 + [ctypes.POINTER(ctypes.c_double)]
    for mp, tp in ((0, 0), (1, 0), (0, 2)):
        o = (ctypes.c_double * 2)()
        if lib.w4a4_probe_fold_mma(2000, mp, tp, o) == 0:
            out[f"fold_beside_issuers_mma{mp}_copies{tp}"] = {"beside_issuers": o[0], "other_warps": o[1]}
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
        tr0 = time.time()
        with torch.cuda.stream(gstream):
            t0.record(gstream)
            run_steps(args.warmup, args.steps)
            t1.record(gstream)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        total_ms = t0.elapsed_time(t1)
        # Load window: the same steps (whole cycles of the input sets) replayed for at
        # least 0.6 s right after the timed region, so that the clock samples (every
        # 100 ms) see the kernels under load; its time per step cross-checks ms_per_step.
        w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        nwin = 0
        tw0 = time.time()
        with torch.cuda.stream(gstream):
            w0.record(gstream)
            while True:
                for _ in range(max(1, 256 // nsets)):
                    cycle.replay()
                    nwin += nsets
                gstream.synchronize()
                if time.time() - tw0 >= 0.6:
                    break
            w1.record(gstream)
        torch.cuda.synchronize()
        tw1 = time.time()
    window_ms_per_step = w0.elapsed_time(w1) / nwin

    # per-kernel device time: each kernel back to back over the same rotating input sets,
    # events only around the loops (on the launching stream)
    # per-kernel device time: each kernel alone, replayed from a CUDA graph over the
    # same rotating input sets (events on the replaying stream)
    nk = max(nsets, 16)
    act_avg = graph_time(lambda i, st: w4.w4a4_rotate_quantize_act(sets[i % nsets][1], out=sets[i % nsets][2],
                                                                    stream=st), nk)
    gemm_avg = graph_time(lambda i, st: w4.w4a4_gemm(sets[i % nsets][0], sets[i % nsets][2], y=sets[i % nsets][3],
                                                     ws=gws, stream=st), nk)
    # the optional expanded weight copy (1 byte per weight beside the Q4_0 codes):
    # the same GEMM when it loads that copy instead of converting the codes
    expanded_w = None
    if not args.no_exact and world == 1:
        wxs = [w4.h32_q4_0_pack_weights(w_dev, expanded=True) for _ in range(nsets)]
        gemm_wx = graph_time(lambda i, st: w4.w4a4_gemm(wxs[i % nsets], sets[i % nsets][2], y=sets[i % nsets][3],
                                                        ws=gws, stream=st), nk)
        expanded_w = {"what": "the same GEMM reading the optional expanded weight copy (2.9x the Q4_0 footprint) "
                              "instead of converting the codes, over as many rotating weight sets",
                      "gemm_ms": gemm_wx, "speedup_vs_codes": gemm_avg / gemm_wx}
        del wxs
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
    del w_dev
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
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
    a_exp = sets[0][2].expanded is not None
    gemm_traffic, gemm_traffic_src = profiled_traffic(f"gemm_grp_{shape.name}.md", GEMM_SOURCES)
    act_traffic, act_traffic_src = profiled_traffic(f"act_rotate_quantize_{shape.name}.md", ACT_SOURCES)
    # the dominant kernel (the GEMM): bound by the per-block scale fold on the fp32 pipe
    g1 = gemm_roofline(gemm_avg, M * N, K, gemm_algorithmic_bytes(N, K, M, M, N), peaks, sm_count)
    gemm_roof = {"bound": "alu", "achieved": g1["fold"]["achieved"], "peak": g1["fold"]["peak"], "unit": "TFLOP/s",
                 "frac": g1["fold"]["frac"], "traffic": gemm_traffic, "traffic_source": gemm_traffic_src,
                 "work": g1["fold"]["work"], "algorithmic_bytes": g1["hbm"]["algorithmic_bytes"],
                 "hbm_frac": g1["hbm"]["frac"], "kernel": "w4a4_grp_kernel",
                 "peak_source": f"derived: {sm_count} SMs x 128 fp32 lanes x 2 flops x "
                                f"{peaks.get('sm_max_mhz', 2070.0)} MHz (the FMA-convention peak; the probe "
                                f"measures fma.rn.f32x2 at 79.7 TFLOP/s)"}
    a1 = act_roofline(act_avg, M, K, peaks, a_exp)
    act_roof = {"bound": "hbm", **{k: a1[k] for k in ("achieved", "peak", "unit", "frac", "algorithmic_bytes",
                                                      "expanded_write_bytes")},
                "kernel": "act_rotate_quantize_tma_kernel", "traffic": act_traffic,
                "traffic_source": act_traffic_src,
                "peak_source": "MEASURED_PEAKS.json hbm_gbs (measured)" if not peaks.get("fallback") else "fallback"}
    eff_tops_gemm = ops / (gemm_avg * 1e-3) / 1e12
    int8_peak = probes.get("int8_mma_sync_tops") if probes else None
    proxy, dense_cfg = None, {}
    if not args.no_proxy and world == 1:
        proxy, dense_cfg = prefill_proxy(dev, 16)
    moe = None
    if not args.no_moe and world == 1:
        moe = moe_extra(dev, peaks)
    verify_c3 = None
    if not args.no_verify and world == 1 and shape.name != "c3":
        verify_c3 = verify_extra(dev, "c3", peaks)
    # every config's kernels against their bounds (algorithmic bytes; expanded writes apart)
    rooflines = {"c1": {"gemm": g1, "act": a1}}
    for name, t in dense_cfg.items():
        rooflines[name] = {"M": t["M"], "K": t["K"], "N": t["N"],
                           "gemm": gemm_roofline(t["gemm_ms"], t["M"] * t["N"], t["K"],
                                                 gemm_algorithmic_bytes(t["N"], t["K"], t["M"], t["M"], t["N"]),
                                                 peaks, sm_count),
                           "act": act_roofline(t["act_ms"], t["M"], t["K"], peaks, True)}
    if moe:
        for part in ("gate", "down"):
            rooflines[f"c4_{part}"] = {"gemm": moe[part]["roofline"], "act": moe[part]["act_roofline"]}

    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        wp = oracle.pack_weights(d["w_bf16"])
        rows, _ = cpu_rows_for_budget(d, wp, budget_s=args.cpu_budget)
        tc = oracle_sample_step(d, wp, rows)
        cpu = {"value": 2.0 * len(rows) * N * K / tc / 1e12, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"{len(rows)} of {M} activation rows x all {N} weight rows, one pass "
                         f"(numpy; BLAS matmuls threaded, elementwise single-threaded)", "seconds": tc}

    clocks = clk.summary(tr0, tw1)
    clocks["samples_under_load"] = clocks.pop("samples")
    clocks["window"] = {"seconds": tw1 - tw0, "steps": nwin, "ms_per_step": window_ms_per_step,
                        "what": "clock samples of the timed steps and of a load window right after them "
                                "(the same steps replayed for >= 0.6 s)"}
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
        "rooflines": rooflines,
        "gemm_effective_tops": eff_tops_gemm,
        "int8_mma_sync_peak_ratio": (eff_tops_gemm / int8_peak) if int8_peak else None,
        "prefill_tok_s_proxy": proxy,
        "moe": moe,
        "exact_path": exact,
        "expanded_weights": expanded_w,
        "rotate_only": rotate_only,
        "verification_batch": verify,
        "verification_batch_c3": verify_c3,
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
    ap.add_argument("--moe-only", action="store_true",
                    help="time only the expert-routed workload and print its figures (a profiling aid, "
                         "not the benchmark line)")
    ap.add_argument("--verify-only", action="store_true",
                    help="time only the 8-token verification batch on --config's weights and print its "
                         "figures (a profiling aid, not the benchmark line)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.moe_only:
        import torch
        import hadamard_rotated_w4a4_gb300 as w4
        w4.load_library(build_if_missing=True)
        print(json.dumps({"moe": moe_extra(torch.device("cuda", torch.cuda.current_device()))}), flush=True)
        return
    if args.verify_only:
        import torch
        import hadamard_rotated_w4a4_gb300 as w4
        w4.load_library(build_if_missing=True)
        dev = torch.device("cuda", torch.cuda.current_device())
        print(json.dumps({"verification_batch": verify_extra(dev, args.config)}), flush=True)
        return
    shape = si.DENSE[args.config]
    line = run_reference(args, shape) if args.impl == "reference" else run_ours(args, shape)
    emit(line, env_rank()[0])


if __name__ == "__main__":
    main()
