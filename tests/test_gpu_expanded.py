"""The expanded operands: the e4m3 bytes of q - 8 the packers and the import
write beside the Q4_0 codes, and the offset codes a + 8 the activation kernel
writes beside the int4 codes, which the dense GEMM loads straight into the
tensor-core operand layout.

Bar: the expanded bytes bit-exact against the codes (the oracle's, through the
sign-and-magnitude rule for weights, pad rows zero; a + 8 for activations); the
GEMM with them bit-identical to the GEMM that converts the codes itself (same
MMA operands, same fold)."""
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


def _expected_bytes(q: np.ndarray) -> np.ndarray:
    """q [rows][K] codes 0..15 -> [round_up(rows, 8)][K] bytes: q - 8 >= 0 -> q - 8, else 0x80 | (8 - q)."""
    rows, K = q.shape
    v = q.astype(np.int64) - 8
    e = np.where(v >= 0, v, 0x80 | (-v)).astype(np.uint8)
    out = np.zeros(((rows + 7) // 8 * 8, K), dtype=np.uint8)
    out[:rows] = e
    return out


def _expanded_np(wq: w4.Q4_0Weights) -> np.ndarray:
    torch.cuda.synchronize()
    r8 = (wq.rows + 7) // 8 * 8
    return wq.expanded[: r8 * wq.K].view(r8, wq.K).cpu().numpy()


@pytest.mark.parametrize("rotate", [True, False])
@pytest.mark.parametrize("N,K", [(8, 32), (13, 256), (130, 1024), (5, 5120)])
def test_pack_writes_expanded_bytes(dev, N, K, rotate):
    d = si.random_dense(4, K, N, seed=N + K)
    wq = w4.h32_q4_0_pack_weights(bf16_tensor(d["w_bf16"], dev), rotate=rotate, expanded=True)
    ref = oracle.pack_weights(d["w_bf16"], rotate)
    assert np.array_equal(_expanded_np(wq), _expected_bytes(ref["q"].astype(np.int64)))


def test_weighted_pack_and_import_write_expanded_bytes(dev):
    d = si.random_dense(4, 512, 37, seed=5)
    imp = np.random.default_rng(6).uniform(0, 2, 512).astype(np.float32)
    wq = w4.h32_q4_0_pack_weights_imatrix(bf16_tensor(d["w_bf16"], dev), f32_tensor(imp, dev), expanded=True)
    torch.cuda.synchronize()
    q = oracle.unpack_nibbles(wq.codes.cpu().numpy()).astype(np.int64)
    assert np.array_equal(_expanded_np(wq), _expected_bytes(q))
    # import: canonical 18-byte blocks of the same weights
    blocks = oracle.q4_0_to_aos(wq.codes.cpu().numpy(), wq.scales.cpu().numpy())
    wi = w4.q4_0_import(torch.from_numpy(np.ascontiguousarray(blocks).reshape(-1)).to(dev), 512, expanded=True)
    assert np.array_equal(_expanded_np(wi), _expected_bytes(q))


SHAPES = [(64, 256, 256), (1, 32, 1), (3, 64, 5), (129, 96, 130), (300, 1024, 520), (257, 160, 64), (17, 5120, 33),
          (512, 512, 1000)]


@pytest.mark.parametrize("M,K,N", SHAPES)
@pytest.mark.parametrize("stream_k", [True, False])
def test_gemm_with_expanded_weights_is_bit_identical(dev, M, K, N, stream_k):
    d = si.random_dense(M, K, N, seed=3 * M + K + N)
    wq = w4.h32_q4_0_pack_weights(bf16_tensor(d["w_bf16"], dev), expanded=True)
    assert wq.expanded is not None
    a = w4.w4a4_rotate_quantize_act(f32_tensor(d["x"], dev))
    ws = True if stream_k else None
    y_exp = w4.w4a4_gemm(wq, a, ws=ws)
    y_cnv = w4.w4a4_gemm(wq.without_expanded(), a, ws=ws)
    torch.cuda.synchronize()
    w4.w4a4_check()
    assert torch.equal(y_exp, y_cnv), float((y_exp - y_cnv).abs().max())
    R = oracle.w4a4_matmul(oracle.pack_weights(d["w_bf16"]), oracle.quantize_activations(d["x"]))
    assert_close(y_exp.cpu().numpy(), R)


def test_gemm_expanded_on_a_row_slice(dev):
    """head(): a slice of the rows keeps the same expanded buffer (the 8-row groups
    past the slice are valid memory, their rows never stored)."""
    d = si.random_dense(40, 512, 300, seed=9)
    wq = w4.h32_q4_0_pack_weights(bf16_tensor(d["w_bf16"], dev), expanded=True)
    a = w4.w4a4_rotate_quantize_act(f32_tensor(d["x"], dev))
    y = w4.w4a4_gemm(wq.head(131), a)
    y_ref = w4.w4a4_gemm(wq, a)[:, :131]
    torch.cuda.synchronize()
    assert torch.equal(y, y_ref)


@pytest.mark.parametrize("cfg", ["c1", "c3"])
def test_gemm_expanded_full_size(dev, cfg):
    d = si.dense_inputs(cfg)
    s = d["shape"]
    wq = w4.h32_q4_0_pack_weights(bf16_tensor(d["w_bf16"], dev), expanded=True)
    a = w4.w4a4_rotate_quantize_act(f32_tensor(d["x"], dev))
    ws = torch.zeros(max(16, w4.w4a4_gemm_workspace_bytes(s.M, s.N, s.K)), dtype=torch.uint8, device=dev)
    y1 = w4.w4a4_gemm(wq, a, ws=ws)
    y2 = w4.w4a4_gemm(wq.without_expanded(), a, ws=ws)
    torch.cuda.synchronize()
    w4.w4a4_check()
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("name,act_per_slot", [("moe_tiny", False), ("moe_tiny", True), ("c4", False), ("c4", True)])
def test_routed_gemm_with_expanded_weights_is_bit_identical(dev, name, act_per_slot):
    mi = si.moe_inputs(name, seed=4)
    s = mi["shape"]
    w, x, N = (mi["wd_bf16"], mi["x_down"], s.N_down) if act_per_slot else (mi["wg_bf16"], mi["x_gate"], s.N_gate)
    wq = w4.h32_q4_0_pack_weights(bf16_tensor(w.reshape(s.E * N, -1), dev), expanded=True)
    aq = w4.w4a4_rotate_quantize_act(f32_tensor(x, dev))
    ids = torch.from_numpy(np.ascontiguousarray(mi["ids"], dtype=np.int32)).to(dev)
    y1 = w4.w4a4_gemm_id(wq, s.E, aq, ids, s.top_k, act_per_slot)
    y2 = w4.w4a4_gemm_id(wq.without_expanded(), s.E, aq, ids, s.top_k, act_per_slot)
    torch.cuda.synchronize()
    w4.w4a4_check()
    assert torch.equal(y1, y2)


# ---------------------------------------------------------------- expanded activations
def _act_expanded_np(a: w4.Act4) -> np.ndarray:
    torch.cuda.synchronize()
    return a.expanded[: a.rows * a.K].view(a.rows, a.K).cpu().numpy()


@pytest.mark.parametrize("rotate", [True, False])
@pytest.mark.parametrize("M,K", [(1, 32), (7, 256), (65, 1024), (300, 160), (600, 8192)])
def test_act_writes_expanded_bytes(dev, M, K, rotate):
    d = si.random_dense(M, K, 1, seed=M + 7 * K)
    a = w4.w4a4_rotate_quantize_act(f32_tensor(d["x"], dev), rotate=rotate)
    ref = oracle.quantize_activations(d["x"], rotate)
    assert np.array_equal(_act_expanded_np(a), (ref["q"].astype(np.int64) + 8).astype(np.uint8))


def test_act_expanded_bytes_strided_rows(dev):
    """Rows with a stride (ldx > K) take the other activation kernel; same bytes."""
    d = si.random_dense(37, 512, 1, seed=11)
    x = torch.zeros(37, 640, dtype=torch.float32, device=dev)
    x[:, :512] = f32_tensor(d["x"], dev)
    a = w4.w4a4_rotate_quantize_act(x[:, :512])
    ref = oracle.quantize_activations(d["x"])
    assert np.array_equal(_act_expanded_np(a), (ref["q"].astype(np.int64) + 8).astype(np.uint8))


ACT_SHAPES = [(64, 256, 256), (1, 32, 1), (3, 64, 5), (129, 96, 130), (300, 1024, 520), (257, 160, 64),
              (17, 5120, 33), (512, 512, 1000), (600, 8192, 64)]


@pytest.mark.parametrize("M,K,N", ACT_SHAPES)
@pytest.mark.parametrize("stream_k", [True, False])
def test_gemm_with_expanded_activations_is_bit_identical(dev, M, K, N, stream_k):
    d = si.random_dense(M, K, N, seed=5 * M + K + N)
    wq = w4.h32_q4_0_pack_weights(bf16_tensor(d["w_bf16"], dev), expanded=True)
    a = w4.w4a4_rotate_quantize_act(f32_tensor(d["x"], dev))
    assert a.expanded is not None and wq.expanded is not None
    ws = True if stream_k else None
    y_ax = w4.w4a4_gemm(wq, a, ws=ws)                    # both operands expanded
    y_wx = w4.w4a4_gemm(wq, a.without_expanded(), ws=ws)  # weights expanded, activations converted
    torch.cuda.synchronize()
    w4.w4a4_check()
    assert torch.equal(y_ax, y_wx), float((y_ax - y_wx).abs().max())
    R = oracle.w4a4_matmul(oracle.pack_weights(d["w_bf16"]), oracle.quantize_activations(d["x"]))
    assert_close(y_ax.cpu().numpy(), R)


def test_gemm_expanded_activations_on_a_row_slice(dev):
    """Act4.head(): the slice keeps the expanded buffer; rows past it are valid memory and never stored."""
    d = si.random_dense(300, 512, 96, seed=12)
    wq = w4.h32_q4_0_pack_weights(bf16_tensor(d["w_bf16"], dev), expanded=True)
    a = w4.w4a4_rotate_quantize_act(f32_tensor(d["x"], dev))
    y = w4.w4a4_gemm(wq, a.head(131))
    y_ref = w4.w4a4_gemm(wq, a)[:131]
    torch.cuda.synchronize()
    assert torch.equal(y, y_ref)


@pytest.mark.parametrize("cfg", ["c1", "c2", "c3"])
def test_gemm_expanded_activations_full_size(dev, cfg):
    d = si.dense_inputs(cfg)
    s = d["shape"]
    wq = w4.h32_q4_0_pack_weights(bf16_tensor(d["w_bf16"], dev), expanded=True)
    a = w4.w4a4_rotate_quantize_act(f32_tensor(d["x"], dev))
    ws = torch.zeros(max(16, w4.w4a4_gemm_workspace_bytes(s.M, s.N, s.K)), dtype=torch.uint8, device=dev)
    y1 = w4.w4a4_gemm(wq, a, ws=ws)
    y2 = w4.w4a4_gemm(wq, a.without_expanded(), ws=ws)
    torch.cuda.synchronize()
    w4.w4a4_check()
    assert torch.equal(y1, y2)
