"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bar: codes, scales and integer partials bit-exact; outputs within a relative
error of 1e-3 of the oracle's fp64 product (floor 1e-3 * max|Y| on the
denominator), on seeded inputs of the workloads' shapes and distributions.
"""
import os

import numpy as np
import pytest
import torch

import hadamard_rotated_w4a4_gb300 as w4
import oracle
import synth_inputs as si
from w4a4_testutil import (act_np, assert_act_bit_exact, assert_close, assert_weights_bit_exact, bf16_tensor,
                           device, f32_tensor, weights_np)

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module")
def dev():
    return device()


# ------------------------------------------------------------------ activations
@pytest.mark.parametrize("rotate", [True, False])
# (600, 8192): more 32-block chunks than the kernel has warps, so every warp reuses its TMA ring
@pytest.mark.parametrize("M,K", [(64, 256), (1, 32), (3, 96), (129, 1024), (7, 5120), (33, 736), (600, 8192)])
def test_act_bit_exact(dev, M, K, rotate):
    d = si.random_dense(M, K, 8, seed=M * 1000 + K)
    aq = w4.w4a4_rotate_quantize_act(f32_tensor(d["x"], dev), rotate=rotate)
    assert_act_bit_exact(act_np(aq), oracle.quantize_activations(d["x"], rotate=rotate))
    assert aq.rotated == rotate


def test_act_config0(dev):
    d = si.dense_inputs("c0")
    aq = w4.w4a4_rotate_quantize_act(f32_tensor(d["x"], dev))
    assert_act_bit_exact(act_np(aq), oracle.quantize_activations(d["x"]))


def test_act_strided_rows(dev):
    d = si.random_dense(40, 512, 8, seed=5)
    big = torch.zeros(40, 512 + 64, dtype=torch.float32, device=dev)
    big[:, :512] = f32_tensor(d["x"], dev)
    aq = w4.w4a4_rotate_quantize_act(big[:, :512])
    assert_act_bit_exact(act_np(aq), oracle.quantize_activations(d["x"]))


def test_act_ties_and_hand_blocks(dev):
    # unrotated half-integer values: every element is an exact rounding tie or an integer
    rng = np.random.default_rng(11)
    x = (rng.integers(-14, 15, size=(16, 256)) / 2.0).astype(np.float32)
    x[:, ::32] = 7.0  # amax 7 in every block -> d_a = 1: y * (1/d_a) = y exactly
    aq = w4.w4a4_rotate_quantize_act(f32_tensor(x, dev), rotate=False)
    assert_act_bit_exact(act_np(aq), oracle.quantize_activations(x, rotate=False))
    from test_oracle_pins import read_golden
    for name, dval, vals, codes in read_golden(os.path.join(GOLDEN, "int4_act_hand_blocks.txt")):
        aq = w4.w4a4_rotate_quantize_act(f32_tensor(vals[None, :], dev), rotate=False)
        g = act_np(aq)
        q = oracle.act_codes_from_nibbles(oracle.unpack_nibbles(g["codes"]))[0]
        assert np.array_equal(q, codes), name
        assert float(g["d_a"][0, 0]) == dval, name


def test_act_zero_and_huge_range_rows(dev):
    rng = np.random.default_rng(12)
    x = rng.standard_normal((6, 128)).astype(np.float32)
    x[0] = 0.0
    x[1] *= np.float32(1e-30)
    x[2] *= np.float32(1e30)
    x[3, :32] = 0.0
    aq = w4.w4a4_rotate_quantize_act(f32_tensor(x, dev))
    assert_act_bit_exact(act_np(aq), oracle.quantize_activations(x))


# ------------------------------------------------------------------ weights
@pytest.mark.parametrize("rotate", [True, False])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("N,K", [(256, 256), (1, 32), (5, 96), (130, 1024)])
def test_pack_bit_exact(dev, N, K, dtype, rotate):
    d = si.random_dense(4, K, N, seed=N * 7 + K)
    if dtype == "bf16":
        wt, ref_in = bf16_tensor(d["w_bf16"], dev), d["w_bf16"]
    else:
        wf = (d["w"] * np.float32(1.7)).astype(np.float32)  # not bf16-representable values
        wt, ref_in = f32_tensor(wf, dev), wf
    wq = w4.h32_q4_0_pack_weights(wt, rotate=rotate)
    ref = oracle.pack_weights(ref_in, rotate=rotate)
    assert_weights_bit_exact(weights_np(wq), ref)


def test_pack_hand_blocks_and_ties(dev):
    from test_oracle_pins import read_golden
    for name, dval, vals, codes in read_golden(os.path.join(GOLDEN, "q4_0_hand_blocks.txt")):
        wq = w4.h32_q4_0_pack_weights(f32_tensor(vals[None, :], dev), rotate=False)
        g = weights_np(wq)
        assert np.array_equal(oracle.unpack_nibbles(g["codes"])[0].astype(np.int64), codes), name
        assert float(g["d16"][0, 0]) == float(np.float16(dval)), name
    # many exact magnitude ties (lowest index must win) and half-way values
    rng = np.random.default_rng(13)
    w = (rng.integers(-16, 17, size=(64, 256)) / 2.0).astype(np.float32)
    wq = w4.h32_q4_0_pack_weights(f32_tensor(w, dev), rotate=False)
    assert_weights_bit_exact(weights_np(wq), oracle.pack_weights(w, rotate=False))


def test_import_is_bit_for_bit(dev):
    d = si.random_dense(4, 512, 96, seed=3)
    ref = oracle.pack_weights(d["w_bf16"])
    aos = oracle.q4_0_to_aos(ref["codes"], ref["d16"])
    wq = w4.q4_0_import(torch.from_numpy(aos.reshape(-1)).to(dev), K=512, rotated=True)
    assert_weights_bit_exact(weights_np(wq), ref)
    assert wq.rotated


# ------------------------------------------------------------------ partials and products
SHAPES = [(64, 256, 256), (1, 32, 1), (3, 64, 5), (129, 96, 130), (130, 1024, 260), (257, 160, 64), (17, 5120, 33)]


def _gpu_pair(dev, d, rotate=True):
    wq = w4.h32_q4_0_pack_weights(bf16_tensor(d["w_bf16"], dev), rotate=rotate)
    aq = w4.w4a4_rotate_quantize_act(f32_tensor(d["x"], dev), rotate=rotate)
    return wq, aq


@pytest.mark.parametrize("M,K,N", SHAPES)
def test_partials_bit_exact(dev, M, K, N):
    d = si.random_dense(M, K, N, seed=M + K + N)
    wq, aq = _gpu_pair(dev, d)
    P = w4.w4a4_gemm_partials(wq, aq).cpu().numpy()
    ref = oracle.block_partials(oracle.pack_weights(d["w_bf16"]), oracle.quantize_activations(d["x"]))
    bad = np.argwhere(P != ref)
    assert len(bad) == 0, f"{len(bad)} partials differ, first {bad[:5].tolist()}"


def test_partials_extreme_values(dev):
    """Every block at the largest |P| = 8 * 7 * 32 = 1792 and sign pattern mixes."""
    K = 256
    x = np.zeros((4, K), dtype=np.float32)
    w = np.zeros((4, K), dtype=np.float32)
    x[0], w[0] = 7.0, -8.0    # q_a = 7, q_w - 8 = -8 everywhere (unrotated)
    x[1], w[1] = -7.0, -8.0
    x[2, ::2], x[2, 1::2] = 7.0, -7.0
    w[2, ::2], w[2, 1::2] = -8.0, 7.0
    x[3] = np.arange(K) % 15 - 7.0
    w[3] = np.arange(K) % 16 - 8.0
    wq = w4.h32_q4_0_pack_weights(f32_tensor(w, dev), rotate=False)
    aq = w4.w4a4_rotate_quantize_act(f32_tensor(x, dev), rotate=False)
    P = w4.w4a4_gemm_partials(wq, aq).cpu().numpy()
    ref = oracle.block_partials(oracle.pack_weights(w, rotate=False), oracle.quantize_activations(x, rotate=False))
    assert np.abs(ref).max() == 1792
    assert np.array_equal(P, ref)


@pytest.mark.parametrize("rotate", [True, False])
@pytest.mark.parametrize("M,K,N", SHAPES)
def test_gemm_matches_oracle(dev, M, K, N, rotate):
    d = si.random_dense(M, K, N, seed=3 * M + K + N)
    wq, aq = _gpu_pair(dev, d, rotate)
    Y = w4.w4a4_gemm(wq, aq).cpu().numpy()
    R = oracle.w4a4_matmul(oracle.pack_weights(d["w_bf16"], rotate), oracle.quantize_activations(d["x"], rotate))
    assert_close(Y, R)


def test_gemm_config0_and_accuracy_report(dev):
    d = si.dense_inputs("c0")
    wq, aq = _gpu_pair(dev, d)
    Y = w4.w4a4_gemm(wq, aq).cpu().numpy()
    wp, ap = oracle.pack_weights(d["w_bf16"]), oracle.quantize_activations(d["x"])
    assert_close(Y, oracle.w4a4_matmul(wp, ap))
    P = w4.w4a4_gemm_partials(wq, aq).cpu().numpy()
    assert np.array_equal(P, oracle.block_partials(wp, ap))


def test_gemm_output_row_stride(dev):
    d = si.random_dense(20, 128, 40, seed=21)
    wq, aq = _gpu_pair(dev, d)
    ybig = torch.full((20, 48), 7.0, dtype=torch.float32, device=dev)
    w4.w4a4_gemm(wq, aq, y=ybig[:, :40])
    yb = ybig.cpu().numpy()
    assert np.all(yb[:, 40:] == 7.0)
    assert_close(yb[:, :40], oracle.w4a4_matmul(oracle.pack_weights(d["w_bf16"]), oracle.quantize_activations(d["x"])))


def test_gemm_zero_operands(dev):
    x = np.zeros((5, 64), dtype=np.float32)
    w = np.random.default_rng(1).standard_normal((9, 64)).astype(np.float32)
    wq = w4.h32_q4_0_pack_weights(f32_tensor(w, dev))
    aq = w4.w4a4_rotate_quantize_act(f32_tensor(x, dev))
    assert np.all(w4.w4a4_gemm(wq, aq).cpu().numpy() == 0.0)
    wq0 = w4.h32_q4_0_pack_weights(f32_tensor(np.zeros((9, 64), np.float32), dev))
    aq1 = w4.w4a4_rotate_quantize_act(f32_tensor(w[:5], dev))
    assert np.all(w4.w4a4_gemm(wq0, aq1).cpu().numpy() == 0.0)


def test_gemm_refuses_mixed_rotation(dev):
    d = si.random_dense(4, 64, 8, seed=2)
    wq = w4.h32_q4_0_pack_weights(bf16_tensor(d["w_bf16"], dev), rotate=True)
    aq = w4.w4a4_rotate_quantize_act(f32_tensor(d["x"], dev), rotate=False)
    with pytest.raises(w4.W4A4Error) as e:
        w4.w4a4_gemm(wq, aq)
    assert e.value.status_name == "W4A4_ERR_MISMATCH"


def test_empty_activation_rows(dev):
    d = si.random_dense(1, 64, 8, seed=2)
    wq = w4.h32_q4_0_pack_weights(bf16_tensor(d["w_bf16"], dev))
    aq = w4.w4a4_rotate_quantize_act(torch.empty(0, 64, dtype=torch.float32, device=dev))
    y = w4.w4a4_gemm(wq, aq)
    assert y.shape == (0, 8)


# ------------------------------------------------------------------ stream-K schedule
# Shapes whose whole tiles would leave SMs idle: the K stages of all tiles are
# split evenly over the CTAs and cut tiles are summed from a workspace.
SK_SHAPES = [(300, 1024, 640), (64, 2048, 128), (1024, 17408, 640), (512, 5120, 5120)]


@pytest.mark.parametrize("M,K,N", SK_SHAPES)
def test_stream_k_matches_oracle_and_is_deterministic(dev, M, K, N):
    need = w4.w4a4_gemm_workspace_bytes(M, N, K)
    assert need > 0, "the split schedule should apply at this shape"
    d = si.dense_inputs("c1") if (M, K, N) == (512, 5120, 5120) else si.random_dense(M, K, N, seed=M + 7 * K + N)
    wq, aq = _gpu_pair(dev, d)
    ws = torch.zeros(need, dtype=torch.uint8, device=dev)
    y1 = w4.w4a4_gemm(wq, aq, ws=ws)
    y2 = w4.w4a4_gemm(wq, aq, ws=ws)  # the tickets of the first launch are stale for the second
    y_whole = w4.w4a4_gemm(wq, aq, ws=None)
    w4.w4a4_check()
    assert torch.equal(y1, y2), "stream-K result changed between identical launches"
    rng = np.random.default_rng(M)
    rows = np.arange(M) if M * N <= 300 * 640 else np.sort(rng.choice(M, 24, replace=False))
    R = oracle.w4a4_matmul(oracle.pack_weights(d["w_bf16"]), oracle.quantize_activations(d["x"][rows]))
    ridx = torch.from_numpy(rows).to(dev)
    assert_close(y1[ridx].cpu().numpy(), R)
    assert_close(y_whole[ridx].cpu().numpy(), R)


def test_stream_k_order_does_not_depend_on_timing(dev):
    """Which CTA of a cut tile arrives last (and so sums the parts, its own from
    registers, with or without depositing it) varies with timing; the sum is always
    taken in CTA order, so every launch gives the same bits.  Launches run beside
    a concurrent matmul on another stream to vary the arrival order."""
    M, K, N = 512, 5120, 5120
    d = si.dense_inputs("c1")
    wq, aq = _gpu_pair(dev, d)
    ws = torch.zeros(w4.w4a4_gemm_workspace_bytes(M, N, K), dtype=torch.uint8, device=dev)
    ref = w4.w4a4_gemm(wq, aq, ws=ws)
    side = torch.cuda.Stream()
    big = torch.randn(4096, 4096, device=dev)
    for i in range(10):
        if i % 2:
            with torch.cuda.stream(side):
                big = (big @ big).clamp_(-1, 1)
        y = w4.w4a4_gemm(wq, aq, ws=ws)
        torch.cuda.synchronize()
        assert torch.equal(y, ref), f"launch {i} differs"
    w4.w4a4_check()


def test_stream_k_under_cuda_graph_replay(dev):
    """A captured split-schedule GEMM replays correctly: the tickets return to zero after every launch."""
    M, K, N = 300, 1024, 640
    d = si.random_dense(M, K, N, seed=77)
    wq, aq = _gpu_pair(dev, d)
    ws = torch.zeros(w4.w4a4_gemm_workspace_bytes(M, N, K), dtype=torch.uint8, device=dev)
    y = torch.empty(M, N, dtype=torch.float32, device=dev)
    w4.w4a4_gemm(wq, aq, y=y, ws=ws)  # set-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            w4.w4a4_gemm(wq, aq, y=y, ws=ws, stream=s)
    first = None
    for _ in range(3):
        y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        cur = y.clone()
        if first is None:
            first = cur
        assert torch.equal(cur, first)
    w4.w4a4_check()
    R = oracle.w4a4_matmul(oracle.pack_weights(d["w_bf16"]), oracle.quantize_activations(d["x"]))
    assert_close(first.cpu().numpy(), R)
    # the tickets (10 tiles x 8 warps x 4 bytes at the start of the workspace) are back at zero
    assert torch.count_nonzero(ws[:1 << 20]).item() == 0


def test_stream_k_workspace_reused_across_shapes(dev):
    shapes = [(300, 1024, 640), (64, 2048, 128), (300, 1024, 640)]
    ws = torch.zeros(max(w4.w4a4_gemm_workspace_bytes(M, N, K) for M, K, N in shapes), dtype=torch.uint8, device=dev)
    for i, (M, K, N) in enumerate(shapes):
        d = si.random_dense(M, K, N, seed=40 + i)
        wq, aq = _gpu_pair(dev, d)
        Y = w4.w4a4_gemm(wq, aq, ws=ws).cpu().numpy()
        assert_close(Y, oracle.w4a4_matmul(oracle.pack_weights(d["w_bf16"]), oracle.quantize_activations(d["x"])))


def test_stream_k_short_workspace_refused(dev):
    d = si.random_dense(300, 1024, 640, seed=3)
    wq, aq = _gpu_pair(dev, d)
    with pytest.raises(w4.W4A4Error) as e:
        w4.w4a4_gemm(wq, aq, ws=torch.zeros(64, dtype=torch.uint8, device=dev))
    assert e.value.status_name == "W4A4_ERR_WORKSPACE"


# ------------------------------------------------------------------ full-size workloads
@pytest.mark.parametrize("cfg", ["c1", "c2", "c3"])
def test_full_size_dense(dev, cfg):
    d = si.dense_inputs(cfg)
    s = d["shape"]
    xt = f32_tensor(d["x"], dev)
    wq = w4.h32_q4_0_pack_weights(bf16_tensor(d["w_bf16"], dev))
    aq = w4.w4a4_rotate_quantize_act(xt)
    Y = w4.w4a4_gemm(wq, aq)
    # activations: every code and scale
    ap = oracle.quantize_activations(d["x"])
    assert_act_bit_exact(act_np(aq), ap)
    # weights: a sample of rows
    rng = np.random.default_rng(0)
    rows = np.sort(rng.choice(s.N, 384, replace=False))
    wp_rows = oracle.pack_weights(d["w_bf16"][rows])
    assert_weights_bit_exact(weights_np(wq), wp_rows, rows=rows)
    # integer partials on a cropped slice: first 128 activation rows x 256 weight rows, all of K
    wsub = wq.head(256)
    asub = aq.head(128)
    P = w4.w4a4_gemm_partials(wsub, asub).cpu().numpy()
    wp_head = oracle.pack_weights(d["w_bf16"][:256])
    ap_head = {"q": ap["q"][:128], "d_a": ap["d_a"][:128]}
    assert np.array_equal(P, oracle.block_partials(wp_head, ap_head))
    # outputs: sampled rows, every column
    mrows = np.sort(rng.choice(s.M, 6, replace=False))
    wp_all = oracle.pack_weights(d["w_bf16"])
    R = oracle.w4a4_matmul(wp_all, ap, m_idx=mrows)
    assert_close(Y[torch.from_numpy(mrows).to(dev)].cpu().numpy(), R)


# ------------------------------------------------------------------ MUL_MAT_ID
def _moe_gpu(dev, w_bits, E, N, x, ids, top_k, act_per_slot, ws=None):
    wq = w4.h32_q4_0_pack_weights(bf16_tensor(w_bits.reshape(E * N, -1), dev))
    aq = w4.w4a4_rotate_quantize_act(f32_tensor(x, dev))
    idt = torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32)).to(dev)
    if ws is None:
        ws = torch.empty(w4.w4a4_gemm_id_workspace_bytes(ids.shape[0], top_k, E, x.shape[1]), dtype=torch.uint8, device=dev)
    y = w4.w4a4_gemm_id(wq, E, aq, idt, top_k, act_per_slot, ws=ws)
    return y, ws


@pytest.mark.parametrize("act_per_slot", [False, True])
def test_moe_tiny_full_compare(dev, act_per_slot):
    mi = si.moe_inputs("moe_tiny", seed=1)
    s = mi["shape"]
    w, x, N = (mi["wd_bf16"], mi["x_down"], s.N_down) if act_per_slot else (mi["wg_bf16"], mi["x_gate"], s.N_gate)
    y, ws = _moe_gpu(dev, w, s.E, N, x, mi["ids"], s.top_k, act_per_slot)
    w4.w4a4_gemm_id_status(ws)
    R = oracle.w4a4_matmul_id(oracle.pack_weights(w.reshape(s.E * N, -1)), s.E, oracle.quantize_activations(x),
                              mi["ids"], act_per_slot)
    assert_close(y.cpu().numpy(), R)


@pytest.mark.parametrize("act_per_slot", [False, True])
def test_moe_config4(dev, act_per_slot):
    mi = si.moe_inputs("c4")
    s = mi["shape"]
    w, x, N = (mi["wd_bf16"], mi["x_down"], s.N_down) if act_per_slot else (mi["wg_bf16"], mi["x_gate"], s.N_gate)
    y, ws = _moe_gpu(dev, w, s.E, N, x, mi["ids"], s.top_k, act_per_slot)
    w4.w4a4_gemm_id_status(ws)
    yn = y.cpu().numpy()
    rng = np.random.default_rng(1)
    toks = np.sort(rng.choice(s.M, 48, replace=False))
    cols = np.sort(rng.choice(N, 256, replace=False))
    wp = oracle.pack_weights(w.reshape(s.E * N, -1))
    ap = oracle.quantize_activations(x)
    R = oracle.w4a4_matmul_id(wp, s.E, ap if act_per_slot else ap, mi["ids"], act_per_slot, n_idx=cols)
    assert_close(yn[toks][:, :, cols], R[toks])


def test_moe_skewed_routing(dev):
    E, N, K, M, k = 16, 64, 128, 300, 3
    ids = si.skewed_ids(M, E, k, seed=4, hot=5)  # expert 5: 300 rows (3 tiles); most others none
    rng = np.random.default_rng(6)
    w = si.round_to_bf16(rng.standard_normal((E, N, K)).astype(np.float32) * np.float32(0.02))[0]
    x = rng.standard_normal((M, K)).astype(np.float32)
    y, ws = _moe_gpu(dev, w, E, N, x, ids, k, False)
    w4.w4a4_gemm_id_status(ws)
    R = oracle.w4a4_matmul_id(oracle.pack_weights(w.reshape(E * N, K)), E, oracle.quantize_activations(x), ids, False)
    assert_close(y.cpu().numpy(), R)


@pytest.mark.parametrize("act_per_slot", [False, True])
def test_moe_few_tiles_long_k(dev, act_per_slot):
    # 4 experts x 1 tile of 2 weight sub-tiles, K 4096 (32 stages): 128 stream-K units,
    # fewer than the SMs, so the routed schedule cuts them over 128 CTAs and the rest idle
    E, N, K, M, k = 4, 256, 4096, 16, 2
    rng = np.random.default_rng(21)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(M)]).astype(np.int32)
    w = si.round_to_bf16(rng.standard_normal((E, N, K)).astype(np.float32) * np.float32(0.02))[0]
    x = rng.standard_normal((M * k if act_per_slot else M, K)).astype(np.float32)
    y, ws = _moe_gpu(dev, w, E, N, x, ids, k, act_per_slot)
    w4.w4a4_gemm_id_status(ws)
    R = oracle.w4a4_matmul_id(oracle.pack_weights(w.reshape(E * N, K)), E, oracle.quantize_activations(x), ids,
                              act_per_slot)
    assert_close(y.cpu().numpy(), R)


def test_moe_bad_ids_flagged_and_zeroed(dev):
    mi = si.moe_inputs("moe_tiny", seed=2)
    s = mi["shape"]
    ids = mi["ids"].copy()
    ids[3, 1] = -1
    ids[7, 0] = s.E
    y, ws = _moe_gpu(dev, mi["wg_bf16"], s.E, s.N_gate, mi["x_gate"], ids, s.top_k, False)
    with pytest.raises(w4.W4A4Error) as e:
        w4.w4a4_gemm_id_status(ws)
    assert e.value.status_name == "W4A4_ERR_DEVICE_FLAG"
    yn = y.cpu().numpy()
    assert np.all(yn[3, 1] == 0) and np.all(yn[7, 0] == 0)
    good = ids.copy()
    good[3, 1] = 0
    good[7, 0] = 0
    R = oracle.w4a4_matmul_id(oracle.pack_weights(mi["wg_bf16"].reshape(s.E * s.N_gate, -1)), s.E,
                              oracle.quantize_activations(mi["x_gate"]), good, False)
    mask = np.ones(ids.shape, bool)
    mask[3, 1] = mask[7, 0] = False
    assert_close(yn[mask], R[mask])
    # the next call on the same workspace clears the flag
    y2, ws = _moe_gpu(dev, mi["wg_bf16"], s.E, s.N_gate, mi["x_gate"], good, s.top_k, False, ws=ws)
    w4.w4a4_gemm_id_status(ws)
