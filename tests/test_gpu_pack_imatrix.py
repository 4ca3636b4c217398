"""GPU parity of the importance-weighted Q4_0 packer against the CPU oracle.

The packer picks, per block, the scale with the least importance-weighted
error; the GPU evaluates the candidate errors in fp32, the oracle in fp64, so on
near-ties the two may keep different (equally good) scales.  Bar: every GPU
block is valid (its codes are the Q4_0 code rule's for its stored scale, its
sums match its codes), its weighted error is within 1e-4 (relative) of the
oracle's, and at least 99% of the blocks carry the oracle's scale and codes bit
for bit.
"""
import numpy as np
import pytest
import torch

import hadamard_rotated_w4a4_gb300 as w4
import oracle
import synth_inputs as si
from w4a4_testutil import assert_close, bf16_tensor, device, f32_tensor, weights_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return device()


def _code_rule(y32: np.ndarray, d16: np.ndarray) -> np.ndarray:
    d = d16.astype(np.float32)
    inv = np.zeros_like(d)
    nz = d != 0
    inv[nz] = np.float32(1.0) / d[nz]
    v = (y32 * inv[..., None]).astype(np.float32)
    return np.clip(np.copysign(np.floor(np.abs(v.astype(np.float64)) + 0.5), v) + 8, 0, 15).astype(np.int64)


def _check(dev, w_bits, imp, rotate, rows=None, min_same=0.99):
    N, K = w_bits.shape
    B = K // 32
    imp_t = f32_tensor(imp, dev) if imp is not None else None
    wq = w4.h32_q4_0_pack_weights_imatrix(bf16_tensor(w_bits, dev), imp_t, rotate=rotate)
    g = weights_np(wq)
    rows = np.arange(N) if rows is None else np.asarray(rows)
    wf = (w_bits[rows].astype(np.uint32) << 16).view(np.float32)
    y = oracle.rotate_h32(wf) if rotate else wf
    om = oracle.effective_importance(imp, K, rotate)
    ref = oracle.quantize_weights_q4_0_weighted(y, om[None, :])
    gq = oracle.unpack_nibbles(g["codes"][rows]).astype(np.int64).reshape(len(rows), B, 32)
    gd = g["d16"][rows].view(np.float16)
    yb = y.reshape(len(rows), B, 32)
    # valid: the code rule for the stored scale, and the sums of those codes
    assert np.array_equal(gq, _code_rule(yb, gd))
    assert np.array_equal(g["sums"][rows].astype(np.int64), (gq - 8).sum(axis=-1))
    # optimal within the fp32 evaluation of the errors
    from oracle.quant import _clean_weights
    omb = np.stack([_clean_weights(om[32 * b:32 * b + 32]) for b in range(B)])
    rq = ref["codes"].astype(np.int64).reshape(len(rows), B, 32)
    rd = ref["d16"]
    e_gpu = (omb[None] * (yb - gd.astype(np.float64)[..., None] * (gq - 8)) ** 2).sum(-1)
    e_ref = (omb[None] * (yb - rd.astype(np.float64)[..., None] * (rq - 8)) ** 2).sum(-1)
    assert np.all(e_gpu <= e_ref * (1 + 1e-4) + 1e-30), float(np.max(e_gpu / np.maximum(e_ref, 1e-30)))
    same = (gd.view(np.uint16) == rd.view(np.uint16)) & np.all(gq == rq, axis=-1)
    assert same.mean() >= min_same, same.mean()
    return wq, e_gpu, same


@pytest.mark.parametrize("rotate", [True, False])
@pytest.mark.parametrize("N,K", [(8, 32), (40, 256), (130, 1024)])
def test_weighted_pack_matches_oracle(dev, N, K, rotate):
    rng = np.random.default_rng(N + K)
    d = si.random_dense(4, K, N, seed=N * 3 + K)
    imp = rng.uniform(0, 4, K) ** 3
    imp[rng.random(K) < 0.05] = 0.0
    _check(dev, d["w_bf16"], imp, rotate)


def test_weighted_pack_edge_weights(dev):
    """Negative and non-finite importances count as 0; a block of zeros as
    uniform; no imatrix is uniform importance."""
    rng = np.random.default_rng(60)
    K, N = 256, 24
    d = si.random_dense(4, K, N, seed=61)
    imp = rng.uniform(0.5, 2.0, K)
    imp[:32] = 0.0
    imp[40] = -3.0
    imp[41] = np.inf
    imp[42] = np.nan
    _check(dev, d["w_bf16"], imp, rotate=False)
    _check(dev, d["w_bf16"], imp, rotate=True)
    _check(dev, d["w_bf16"], None, rotate=False)
    _check(dev, d["w_bf16"], None, rotate=True)


def test_rotated_imatrix_does_nothing_on_gpu(dev):
    """The pages' observation on the rotated file, through the CUDA path: the
    rotated importance is flat in each block, so the scales match those made
    with no imatrix at all."""
    rng = np.random.default_rng(62)
    d = si.random_dense(4, 1024, 200, seed=63)
    imp = f32_tensor(rng.uniform(0, 10, 1024) ** 3, dev)
    a = weights_np(w4.h32_q4_0_pack_weights_imatrix(bf16_tensor(d["w_bf16"], dev), imp, rotate=True))
    b = weights_np(w4.h32_q4_0_pack_weights_imatrix(bf16_tensor(d["w_bf16"], dev), None, rotate=True))
    assert np.mean(a["d16"].view(np.uint16) == b["d16"].view(np.uint16)) >= 0.99


def test_weighted_pack_lowers_the_weighted_error_and_feeds_the_gemm(dev):
    """Unrotated weights with skewed importance: the weighted scales cut the
    importance-weighted error against the plain Q4_0 scales, and the packed
    weights run through the W4A4 product like any other Q4_0 weights."""
    rng = np.random.default_rng(64)
    M, K, N = 64, 512, 96
    d = si.random_dense(M, K, N, seed=65)
    imp = np.where(rng.random(K) < 0.1, 50.0, 1.0)
    wq = w4.h32_q4_0_pack_weights_imatrix(bf16_tensor(d["w_bf16"], dev), f32_tensor(imp, dev), rotate=False)
    wp = w4.h32_q4_0_pack_weights(bf16_tensor(d["w_bf16"], dev), rotate=False)
    wf = (d["w_bf16"].astype(np.uint32) << 16).view(np.float32).astype(np.float64)

    def werr(pack):
        g = weights_np(pack)
        q = oracle.unpack_nibbles(g["codes"]).astype(np.float64).reshape(N, K // 32, 32) - 8
        deq = (q * g["d16"].view(np.float16).astype(np.float64)[..., None]).reshape(N, K)
        return float((imp[None, :] * (wf - deq) ** 2).sum())

    assert werr(wq) < 0.95 * werr(wp)
    a = w4.w4a4_rotate_quantize_act(f32_tensor(d["x"], dev), rotate=False)
    Y = w4.w4a4_gemm(wq, a).cpu().numpy()
    g = weights_np(wq)
    R = oracle.w4a4_matmul({"codes": g["codes"], "d16": g["d16"].view(np.float16)},
                           oracle.quantize_activations(d["x"], rotate=False))
    assert_close(Y, R)


def test_weighted_pack_full_size_sampled(dev):
    """The dense attention projection's weights (N = K = 5120), rotated, with a
    synthetic importance vector; sampled rows against the oracle."""
    dd = si.dense_inputs("c1")
    K = dd["shape"].K
    rng = np.random.default_rng(66)
    imp = rng.uniform(0, 3, K) ** 4
    rows = np.sort(rng.choice(dd["shape"].N, 24, replace=False))
    _check(dev, dd["w_bf16"], imp, rotate=True, rows=rows)
    w4.w4a4_check()
