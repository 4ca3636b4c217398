"""GPU parity of the rotate-only route (rotated Q4_0 weights x rotated
activations that were not quantised, carried as bf16) against the CPU oracle.

Bar: the bf16 activations bit-exact (the same fp32 rotation, then round to
nearest even); outputs within a relative error of 1e-3 of the oracle's fp64
product (floor 1e-3 * max|Y|): the tensor core sums each block's 32 bf16
products in fp32, a rounding the fp64 oracle does not make.
"""
import numpy as np
import pytest
import torch

import hadamard_rotated_w4a4_gb300 as w4
import oracle
import synth_inputs as si
from w4a4_testutil import assert_close, bf16_tensor, device, f32_tensor

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return device()


def _x16_np(a: w4.Act16) -> np.ndarray:
    torch.cuda.synchronize()
    return a.values.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("rotate", [True, False])
# (600, 8192): more 32-block chunks than the kernel has warps, so every warp reuses its TMA ring
@pytest.mark.parametrize("M,K", [(64, 256), (1, 32), (3, 96), (129, 1024), (7, 5120), (33, 736), (600, 8192)])
def test_act16_bit_exact(dev, M, K, rotate):
    d = si.random_dense(M, K, 8, seed=M * 11 + K)
    a = w4.w4a16_rotate_act(f32_tensor(d["x"], dev), rotate=rotate)
    ref = oracle.rotate_activations_bf16(d["x"], rotate=rotate)["x16"]
    got = _x16_np(a)
    bad = np.argwhere(got != ref)
    assert len(bad) == 0, f"{len(bad)} bf16 values differ, first at {bad[:5].tolist()}"


def test_act16_strided_rows_and_ties(dev):
    d = si.random_dense(40, 512, 8, seed=10)
    x = d["x"].copy()
    # exact bf16 ties after no rotation: low 16 bits 0x8000
    x[0, :64] = (np.arange(64, dtype=np.uint32) << 16 | np.uint32(0x3F808000)).view(np.float32)
    big = torch.zeros(40, 512 + 64, dtype=torch.float32, device=dev)
    big[:, :512] = f32_tensor(x, dev)
    for rotate in (True, False):
        a = w4.w4a16_rotate_act(big[:, :512], rotate=rotate)
        assert np.array_equal(_x16_np(a), oracle.rotate_activations_bf16(x, rotate=rotate)["x16"])


SHAPES = [(64, 256, 256), (1, 32, 1), (3, 64, 5), (129, 96, 130), (130, 1024, 260), (257, 160, 64), (17, 5120, 33)]


@pytest.mark.parametrize("rotate", [True, False])
@pytest.mark.parametrize("M,K,N", SHAPES)
def test_w4a16_gemm_matches_oracle(dev, M, K, N, rotate):
    d = si.random_dense(M, K, N, seed=7 * M + K + N)
    wq = w4.h32_q4_0_pack_weights(bf16_tensor(d["w_bf16"], dev), rotate=rotate)
    a = w4.w4a16_rotate_act(f32_tensor(d["x"], dev), rotate=rotate)
    Y = w4.w4a16_gemm(wq, a).cpu().numpy()
    R = oracle.w4a16_matmul(oracle.pack_weights(d["w_bf16"], rotate), oracle.rotate_activations_bf16(d["x"], rotate))
    assert_close(Y, R)


def test_w4a16_extreme_values(dev):
    """Largest codes and scales the route meets: every weight code 0 (q - 8 = -8)
    or 15, activations spanning many binades; still within the bar."""
    rng = np.random.default_rng(40)
    M, K, N = 40, 512, 136
    w = (rng.choice([-1.0, 1.0], (N, K)) * 10.0 ** rng.uniform(-3, 2, (N, 1))).astype(np.float32)
    x = (rng.standard_normal((M, K)) * 10.0 ** rng.uniform(-4, 4, (M, K // 32)).repeat(32, axis=1)).astype(np.float32)
    wb = oracle.round_bf16(w)
    wq = w4.h32_q4_0_pack_weights(bf16_tensor(wb, dev), rotate=False)
    a = w4.w4a16_rotate_act(f32_tensor(x, dev), rotate=False)
    Y = w4.w4a16_gemm(wq, a).cpu().numpy()
    R = oracle.w4a16_matmul(oracle.pack_weights(wb, False), oracle.rotate_activations_bf16(x, False))
    assert_close(Y, R)


def test_w4a16_refuses_other_activations_and_mixed_rotation(dev):
    d = si.random_dense(4, 64, 8, seed=3)
    wq = w4.h32_q4_0_pack_weights(bf16_tensor(d["w_bf16"], dev), rotate=True)
    a = w4.w4a16_rotate_act(f32_tensor(d["x"], dev), rotate=False)
    with pytest.raises(w4.W4A4Error) as e:
        w4.w4a16_gemm(wq, a)
    assert e.value.status_name == "W4A4_ERR_MISMATCH"
    # a descriptor tagged as int4 activations is refused before anything is read
    import ctypes
    bad = w4._Act16Desc(a.values.data_ptr(), 4, 64, w4.TAG_ACT4 | 1)
    y = torch.empty(4, 8, device=dev)
    st = w4.load_library().w4a16_gemm(ctypes.byref(wq.desc()), ctypes.byref(bad), y.data_ptr(), 8, None, 0, None)
    assert w4.STATUS[st] == "W4A4_ERR_INVALID_ARG"


def test_w4a16_graph_replay_and_workspace_reuse(dev):
    d = si.random_dense(300, 1024, 520, seed=41)
    wq = w4.h32_q4_0_pack_weights(bf16_tensor(d["w_bf16"], dev))
    x = f32_tensor(d["x"], dev)
    a = w4.w4a16_rotate_act(x)
    y = torch.empty(300, 520, device=dev)
    ws = torch.zeros(max(16, w4.w4a16_gemm_workspace_bytes(300, 520, 1024)), dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        w4.w4a16_rotate_act(x, out=a, stream=s)
        w4.w4a16_gemm(wq, a, y=y, ws=ws, stream=s)
    s.synchronize()
    ref = y.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        w4.w4a16_rotate_act(x, out=a, stream=s)
        w4.w4a16_gemm(wq, a, y=y, ws=ws, stream=s)
    for _ in range(3):
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y, ref)
    w4.w4a4_check()
    R = oracle.w4a16_matmul(oracle.pack_weights(d["w_bf16"]), oracle.rotate_activations_bf16(d["x"]))
    assert_close(ref.cpu().numpy(), R)


@pytest.mark.parametrize("cfg", ["c1", "c3"])
def test_w4a16_full_size(dev, cfg):
    d = si.dense_inputs(cfg)
    s = d["shape"]
    wq = w4.h32_q4_0_pack_weights(bf16_tensor(d["w_bf16"], dev))
    a = w4.w4a16_rotate_act(f32_tensor(d["x"], dev))
    ap = oracle.rotate_activations_bf16(d["x"])
    assert np.array_equal(_x16_np(a), ap["x16"])
    ws = torch.zeros(max(16, w4.w4a16_gemm_workspace_bytes(s.M, s.N, s.K)), dtype=torch.uint8, device=dev)
    Y1 = w4.w4a16_gemm(wq, a, ws=ws)
    Y2 = w4.w4a16_gemm(wq, a, ws=ws)
    w4.w4a4_check()
    assert torch.equal(Y1, Y2)
    rng = np.random.default_rng(2)
    rows = np.sort(rng.choice(s.M, 6, replace=False))
    R = oracle.w4a16_matmul(oracle.pack_weights(d["w_bf16"]), {"xr": ap["xr"][rows]})
    assert_close(Y1[torch.from_numpy(rows).to(dev)].cpu().numpy(), R)
