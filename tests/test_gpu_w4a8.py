"""GPU parity of the exact path (rotated Q4_0 weights x int8 activations)
against the CPU oracle.

Bar: int8 codes, scales and integer partials bit-exact; outputs within a
relative error of 1e-3 of the oracle's fp64 product (floor 1e-3 * max|Y|).
"""
import os

import numpy as np
import pytest
import torch

import hadamard_rotated_w4a4_gb300 as w4
import oracle
import synth_inputs as si
from w4a4_testutil import assert_close, bf16_tensor, device, f32_tensor

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module")
def dev():
    return device()


def _act8_np(a: w4.Act8) -> dict:
    torch.cuda.synchronize()
    return {"q": a.codes.cpu().numpy(), "d_a": a.scales.cpu().numpy()}


def _assert_act8(gpu: dict, ref: dict) -> None:
    bad = np.argwhere(gpu["q"] != ref["q"])
    assert len(bad) == 0, f"{len(bad)} int8 codes differ, first at {bad[:5].tolist()}"
    assert np.array_equal(gpu["d_a"].view(np.uint32), np.asarray(ref["d_a"], np.float32).view(np.uint32))


@pytest.mark.parametrize("rotate", [True, False])
# (600, 8192): more 32-block chunks than the kernel has warps, so every warp reuses its TMA ring
@pytest.mark.parametrize("M,K", [(64, 256), (1, 32), (3, 96), (129, 1024), (7, 5120), (33, 736), (600, 8192)])
def test_act8_bit_exact(dev, M, K, rotate):
    d = si.random_dense(M, K, 8, seed=M * 7 + K)
    a = w4.w4a8_rotate_quantize_act(f32_tensor(d["x"], dev), rotate=rotate)
    _assert_act8(_act8_np(a), oracle.quantize_activations_int8(d["x"], rotate=rotate))


def test_act8_strided_rows(dev):
    d = si.random_dense(40, 512, 8, seed=9)
    big = torch.zeros(40, 512 + 64, dtype=torch.float32, device=dev)
    big[:, :512] = f32_tensor(d["x"], dev)
    a = w4.w4a8_rotate_quantize_act(big[:, :512])
    _assert_act8(_act8_np(a), oracle.quantize_activations_int8(d["x"]))


def test_act8_hand_blocks(dev):
    from test_oracle_pins import read_golden
    cases = read_golden(os.path.join(GOLDEN, "int8_act_hand_blocks.txt"))
    x = np.stack([c[2] for c in cases]).astype(np.float32)
    a = _act8_np(w4.w4a8_rotate_quantize_act(f32_tensor(x, dev), rotate=False))
    for i, (name, dval, _, codes) in enumerate(cases):
        assert float(a["d_a"][i, 0]) == dval, name
        assert np.array_equal(a["q"][i].astype(np.int64), codes), name


SHAPES = [(64, 256, 256), (1, 32, 1), (3, 64, 5), (129, 96, 130), (130, 1024, 260), (257, 160, 64), (17, 5120, 33)]


def _pair(dev, d, rotate=True):
    wq = w4.h32_q4_0_pack_weights(bf16_tensor(d["w_bf16"], dev), rotate=rotate)
    a = w4.w4a8_rotate_quantize_act(f32_tensor(d["x"], dev), rotate=rotate)
    return wq, a


@pytest.mark.parametrize("M,K,N", SHAPES)
def test_w4a8_partials_bit_exact(dev, M, K, N):
    d = si.random_dense(M, K, N, seed=M + 2 * K + N)
    wq, a = _pair(dev, d)
    P = w4.w4a8_gemm_partials(wq, a).cpu().numpy()
    ref = oracle.block_partials(oracle.pack_weights(d["w_bf16"]), oracle.quantize_activations_int8(d["x"]))
    bad = np.argwhere(P != ref)
    assert len(bad) == 0, f"{len(bad)} partials differ, first {bad[:5].tolist()}"


def test_w4a8_partials_extreme_values(dev):
    """Every partial at its largest magnitude: (q_w - 8) = -8 against q_a = +-127."""
    K = 128
    w = np.full((3, K), -8.0, dtype=np.float32)
    x = np.zeros((3, K), dtype=np.float32)
    x[0], x[1] = 127.0, -127.0
    x[2, ::2], x[2, 1::2] = 127.0, -127.0
    wq = w4.h32_q4_0_pack_weights(f32_tensor(w, dev), rotate=False)
    a = w4.w4a8_rotate_quantize_act(f32_tensor(x, dev), rotate=False)
    P = w4.w4a8_gemm_partials(wq, a).cpu().numpy()
    ref = oracle.block_partials(oracle.pack_weights(w, rotate=False), oracle.quantize_activations_int8(x, rotate=False))
    assert np.abs(ref).max() == 32512
    assert np.array_equal(P, ref)


@pytest.mark.parametrize("rotate", [True, False])
@pytest.mark.parametrize("M,K,N", SHAPES)
def test_w4a8_gemm_matches_oracle(dev, M, K, N, rotate):
    d = si.random_dense(M, K, N, seed=5 * M + K + N)
    wq, a = _pair(dev, d, rotate)
    Y = w4.w4a8_gemm(wq, a).cpu().numpy()
    R = oracle.w4a8_matmul(oracle.pack_weights(d["w_bf16"], rotate), oracle.quantize_activations_int8(d["x"], rotate))
    assert_close(Y, R)


def test_w4a8_refuses_int4_and_mixed_rotation(dev):
    d = si.random_dense(4, 64, 8, seed=2)
    wq = w4.h32_q4_0_pack_weights(bf16_tensor(d["w_bf16"], dev), rotate=True)
    a = w4.w4a8_rotate_quantize_act(f32_tensor(d["x"], dev), rotate=False)
    with pytest.raises(w4.W4A4Error) as e:
        w4.w4a8_gemm(wq, a)
    assert e.value.status_name == "W4A4_ERR_MISMATCH"


@pytest.mark.parametrize("cfg", ["c1", "c3"])
def test_w4a8_full_size(dev, cfg):
    d = si.dense_inputs(cfg)
    s = d["shape"]
    wq = w4.h32_q4_0_pack_weights(bf16_tensor(d["w_bf16"], dev))
    a = w4.w4a8_rotate_quantize_act(f32_tensor(d["x"], dev))
    ap = oracle.quantize_activations_int8(d["x"])
    _assert_act8(_act8_np(a), ap)
    ws = torch.zeros(max(16, w4.w4a8_gemm_workspace_bytes(s.M, s.N, s.K)), dtype=torch.uint8, device=dev)
    Y1 = w4.w4a8_gemm(wq, a, ws=ws)
    Y2 = w4.w4a8_gemm(wq, a, ws=ws)
    w4.w4a4_check()
    assert torch.equal(Y1, Y2)
    rng = np.random.default_rng(1)
    rows = np.sort(rng.choice(s.M, 6, replace=False))
    R = oracle.w4a8_matmul(oracle.pack_weights(d["w_bf16"]), {"q": ap["q"][rows], "d_a": ap["d_a"][rows]})
    assert_close(Y1[torch.from_numpy(rows).to(dev)].cpu().numpy(), R)
    # integer partials on a cropped slice
    P = w4.w4a8_gemm_partials(wq.head(128), w4.Act8(a.codes[:64], a.scales_buf, 64, s.K, True)).cpu().numpy()
    Pr = oracle.block_partials(oracle.pack_weights(d["w_bf16"][:128]), {"q": ap["q"][:64]})
    assert np.array_equal(P, Pr)
