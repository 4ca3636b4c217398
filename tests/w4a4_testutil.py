"""Shared helpers for the GPU parity tests: move seeded inputs to the device, run
the CUDA path through the binding, and compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import hadamard_rotated_w4a4_gb300 as w4

#: max_i |Y - Y_ref| / max(|Y_ref,i|, FLOOR * max|Y_ref|) must not exceed REL_TOL
REL_TOL = 1e-3
FLOOR = 1e-3


def device() -> torch.device:
    assert torch.cuda.is_available(), "gpu tests need a CUDA device"
    w4.load_library(build_if_missing=True)
    return torch.device("cuda:0")


def bf16_tensor(bits: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


def f32_tensor(x: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(dev)


def weights_np(wq: w4.Q4_0Weights) -> dict:
    torch.cuda.synchronize()
    return {"codes": wq.codes.cpu().numpy(), "d16": wq.scales.cpu().numpy(), "sums": wq.sums.cpu().numpy()}


def act_np(aq: w4.Act4) -> dict:
    torch.cuda.synchronize()
    return {"codes": aq.codes.cpu().numpy(), "d_a": aq.scales.cpu().numpy()}


def assert_weights_bit_exact(gpu: dict, ref: dict, rows=None) -> None:
    gc, gd = gpu["codes"], gpu["d16"]
    if rows is not None:
        gc, gd = gc[rows], gd[rows]
    assert gc.shape == ref["codes"].shape
    bad = np.argwhere(gc != ref["codes"])
    assert len(bad) == 0, f"{len(bad)} code bytes differ, first at {bad[:5].tolist()}"
    assert np.array_equal(gd.view(np.uint16), np.asarray(ref["d16"], dtype=np.float16).view(np.uint16))
    # the derived block sums agree with the codes themselves: sum_j (q_j - 8)
    gs = gpu["sums"] if rows is None else gpu["sums"][rows]
    q = gc.reshape(gc.shape[0], -1, 16)
    want = ((q & 0x0F).astype(np.int64) + (q >> 4)).sum(axis=-1) - 256
    assert np.array_equal(gs.astype(np.int64), want)


def assert_act_bit_exact(gpu: dict, ref: dict) -> None:
    bad = np.argwhere(gpu["codes"] != ref["codes"])
    assert len(bad) == 0, f"{len(bad)} code bytes differ, first at {bad[:5].tolist()}"
    assert np.array_equal(gpu["d_a"].view(np.uint32), np.asarray(ref["d_a"], dtype=np.float32).view(np.uint32))


def assert_close(Y, R, tol: float = REL_TOL) -> float:
    Y = np.asarray(Y, dtype=np.float64)
    R = np.asarray(R, dtype=np.float64)
    assert Y.shape == R.shape
    if R.size == 0:
        return 0.0
    floor = FLOOR * max(np.abs(R).max(), 1e-30)
    err = np.abs(Y - R) / np.maximum(np.abs(R), floor)
    worst = float(err.max())
    assert worst <= tol, f"max relative error {worst:.3e} > {tol:.1e} at {np.unravel_index(err.argmax(), err.shape)}"
    return worst
