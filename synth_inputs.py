"""Seeded synthetic inputs for the W4A4 prefill matmul workloads.

This module is shared by the CPU oracle (``oracle/``), the tests and
``bench.py``.  It only draws random numbers and lays them out; it holds none of
the method's arithmetic (no rotation, no quantisation, no dot products), so the
oracle and the CUDA path stay independent of each other.

Recipe (numpy ``default_rng(seed)``; draws taken in this order: weights,
activations, outlier channels, routing ids):

* weights  ~ N(0, 1) * 0.02 as fp32, then rounded to bf16 (round to nearest
  even); shape [N][K] (each output row is K-contiguous) or [E][N][K] for experts;
* activations ~ N(0, 1) fp32 [M][K]; the FFN-down shape draws SiLU(g) * u with
  g, u ~ N(0, 1) instead, the input that reaches a down projection;
* outlier channels: ``rng.choice(K, n, replace=False)`` columns scaled x20, the
  few large activation channels whose effect the Hadamard rotation is there to
  spread (engine docs "The lean option: ROCmFP4, ROCmI4 and Hadamard Q4_0",
  section "Hadamard-rotated Q4_0: W4A4 prompt processing");
* routing ids: per token, ``rng.choice(E, top_k, replace=False)`` (uniform,
  without replacement).

The shapes follow the pages' dense 27B-class model (hidden 5120, FFN 17408,
512- and 1024-token micro-batches) and a 128-expert top-8 MoE.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class DenseShape:
    name: str
    M: int
    K: int
    N: int
    n_outliers: int
    silu_act: bool = False
    what: str = ""


@dataclass(frozen=True)
class MoEShape:
    name: str
    M: int
    E: int
    top_k: int
    K_gate: int
    N_gate: int
    K_down: int
    N_down: int
    n_outliers_gate: int
    n_outliers_down: int
    what: str = ""


DENSE = {
    "c0": DenseShape("c0", 64, 256, 256, 2, what="tiny correctness GEMM M64 K256 N256"),
    "c1": DenseShape("c1", 512, 5120, 5120, 51, what="dense attention projection M512 K5120 N5120"),
    "c2": DenseShape("c2", 512, 5120, 17408, 51, what="dense FFN gate/up M512 K5120 N17408"),
    "c3": DenseShape("c3", 1024, 17408, 5120, 174, silu_act=True,
                     what="dense FFN down M1024 K17408 N5120, SiLU(g)*u activations"),
}

MOE = {
    "c4": MoEShape("c4", 1024, 128, 8, 2048, 768, 768, 2048, 16, 6,
                   what="MoE MUL_MAT_ID: 1024 tokens, 128 experts, top-8; "
                        "gate/up K2048->N768 (act per token), down K768->N2048 (act per token-slot)"),
    # small expert problem for brute-force style checks
    "moe_tiny": MoEShape("moe_tiny", 24, 4, 2, 64, 48, 64, 40, 1, 1, what="4 experts, top-2"),
}


def round_to_bf16(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """fp32 -> bf16 with round-to-nearest-even; returns (uint16 bits, fp32 values).

    Input preparation only (weights are bf16 tensors).  Inputs are finite.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    back = (r.astype(np.uint32) << 16).view(np.float32)
    return r, back


def _outliers(rng: np.random.Generator, x: np.ndarray, n: int) -> np.ndarray:
    if n <= 0:
        return np.zeros(0, dtype=np.int64)
    cols = rng.choice(x.shape[1], n, replace=False)
    x[:, cols] *= np.float32(20.0)
    return np.sort(cols)


def dense_inputs(shape: DenseShape | str, seed: int = 0) -> dict:
    """Weights (bf16 bits + exact fp32 values) and fp32 activations for a dense GEMM."""
    if isinstance(shape, str):
        shape = DENSE[shape]
    rng = np.random.default_rng(seed)
    w = rng.standard_normal((shape.N, shape.K), dtype=np.float32) * np.float32(0.02)
    w_bits, w_f32 = round_to_bf16(w)
    del w
    if shape.silu_act:
        g = rng.standard_normal((shape.M, shape.K), dtype=np.float32)
        u = rng.standard_normal((shape.M, shape.K), dtype=np.float32)
        x = (g / (np.float32(1.0) + np.exp(-g))) * u
        x = x.astype(np.float32)
        del g, u
    else:
        x = rng.standard_normal((shape.M, shape.K), dtype=np.float32)
    cols = _outliers(rng, x, shape.n_outliers)
    return {"shape": shape, "w_bf16": w_bits, "w": w_f32, "x": x, "outlier_cols": cols}


def random_dense(M: int, K: int, N: int, seed: int, n_outliers: int | None = None,
                 w_scale: float = 0.02) -> dict:
    """Same recipe at an arbitrary shape (for ragged / edge-case parity tests)."""
    rng = np.random.default_rng(seed)
    w = rng.standard_normal((N, K), dtype=np.float32) * np.float32(w_scale)
    w_bits, w_f32 = round_to_bf16(w)
    x = rng.standard_normal((M, K), dtype=np.float32)
    if n_outliers is None:
        n_outliers = max(1, (2 * K) // 256) if K >= 32 else 0
    cols = _outliers(rng, x, min(n_outliers, K))
    return {"w_bf16": w_bits, "w": w_f32, "x": x, "outlier_cols": cols}


def moe_inputs(shape: MoEShape | str, seed: int = 0) -> dict:
    """Expert weights for both projections, both activation sets and routing ids."""
    if isinstance(shape, str):
        shape = MOE[shape]
    s = shape
    rng = np.random.default_rng(seed)
    wg = rng.standard_normal((s.E, s.N_gate, s.K_gate), dtype=np.float32) * np.float32(0.02)
    wg_bits, wg_f32 = round_to_bf16(wg)
    del wg
    wd = rng.standard_normal((s.E, s.N_down, s.K_down), dtype=np.float32) * np.float32(0.02)
    wd_bits, wd_f32 = round_to_bf16(wd)
    del wd
    xg = rng.standard_normal((s.M, s.K_gate), dtype=np.float32)
    xd = rng.standard_normal((s.M * s.top_k, s.K_down), dtype=np.float32)
    cg = _outliers(rng, xg, s.n_outliers_gate)
    cd = _outliers(rng, xd, s.n_outliers_down)
    ids = np.stack([rng.choice(s.E, s.top_k, replace=False) for _ in range(s.M)]).astype(np.int32)
    return {"shape": s, "wg_bf16": wg_bits, "wg": wg_f32, "wd_bf16": wd_bits, "wd": wd_f32,
            "x_gate": xg, "x_down": xd, "ids": ids, "outlier_cols_gate": cg, "outlier_cols_down": cd}


def skewed_ids(M: int, E: int, top_k: int, seed: int, hot: int = 0) -> np.ndarray:
    """Routing where every token picks expert ``hot`` first (one expert gets all tokens,
    several experts get none)."""
    rng = np.random.default_rng(seed)
    out = np.empty((M, top_k), dtype=np.int32)
    others = np.array([e for e in range(E) if e != hot])
    for t in range(M):
        out[t, 0] = hot
        if top_k > 1:
            out[t, 1:] = rng.choice(others[: max(top_k - 1, len(others) // 4)], top_k - 1, replace=False)
    return out
