"""The routed product without a caller workspace (w4a4_gemm_id_static).

That entry point keeps its routing scratch in a fixed device array inside the
library, for callers that cannot allocate at the call site.  The GPU tests call
it twice in a row through the C ABI and compare both results with
w4a4_gemm_id on the same inputs.  The file name sorts last, so the suite also
runs it after every other test; it passes alone in a fresh process as well.
"""
import ctypes

import numpy as np
import pytest

import hadamard_rotated_w4a4_gb300 as w4
import synth_inputs as si
from hadamard_rotated_w4a4_gb300 import _Act4Desc, _Q4_0Desc

FAKE = 0x10000  # aligned, never dereferenced: the call below fails validation first


def test_oversized_problem_refused_before_launch():
    lib = w4.load_library(build_if_missing=True)
    E, N, K, M, k = 8, 64, 4096, 16384, 2  # 32768 routed rows x 2048 code bytes: > 64 MiB of scratch
    assert w4.w4a4_gemm_id_workspace_bytes(M, k, E, K) > w4.GEMM_ID_STATIC_SCRATCH_BYTES
    wd = _Q4_0Desc(FAKE, FAKE, FAKE, E * N, K, w4.TAG_Q4_0 | 1)
    ad = _Act4Desc(FAKE, FAKE, M, K, w4.TAG_ACT4 | 1)
    s = lib.w4a4_gemm_id_static(ctypes.byref(wd), E, N, ctypes.byref(ad), FAKE, M, k, 0, FAKE, None)
    assert w4.STATUS[s] == "W4A4_ERR_WORKSPACE"
    assert b"fixed" in lib.w4a4_last_error()


@pytest.fixture(scope="module")
def dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from w4a4_testutil import device
    return device()


CASES = [("moe_tiny", False), ("moe_tiny", True), ("c4", False), ("c4", True)]


@pytest.mark.gpu
@pytest.mark.parametrize("name,act_per_slot", CASES)
def test_static_scratch_matches_workspace_variant(dev, name, act_per_slot):
    import torch
    from w4a4_testutil import assert_close, bf16_tensor, f32_tensor

    mi = si.moe_inputs(name, seed=3)
    s = mi["shape"]
    w, x, N = (mi["wd_bf16"], mi["x_down"], s.N_down) if act_per_slot else (mi["wg_bf16"], mi["x_gate"], s.N_gate)
    K = x.shape[1]
    assert w4.w4a4_gemm_id_workspace_bytes(s.M, s.top_k, s.E, K) <= w4.GEMM_ID_STATIC_SCRATCH_BYTES
    wq = w4.h32_q4_0_pack_weights(bf16_tensor(w.reshape(s.E * N, -1), dev))
    aq = w4.w4a4_rotate_quantize_act(f32_tensor(x, dev))
    ids = torch.from_numpy(np.ascontiguousarray(mi["ids"], dtype=np.int32)).to(dev)

    want = w4.w4a4_gemm_id(wq, s.E, aq, ids, s.top_k, act_per_slot)
    y1 = torch.full((s.M, s.top_k, N), float("nan"), device=dev)
    y2 = torch.full((s.M, s.top_k, N), float("nan"), device=dev)
    w4.w4a4_gemm_id_static(wq, s.E, aq, ids, s.top_k, act_per_slot, y1)
    w4.w4a4_gemm_id_static(wq, s.E, aq, ids, s.top_k, act_per_slot, y2)
    w4.w4a4_check()
    # the same kernels on the same inputs: the results agree bit for bit
    assert torch.equal(y1, want)
    assert torch.equal(y2, want)


@pytest.mark.gpu
def test_static_scratch_zeroes_rows_of_bad_ids(dev):
    """Ids outside [0, E) zero their output rows through the fixed scratch too, and
    every other row is the workspace variant's, bit for bit; the call after it,
    with good ids, is unaffected by what the bad call left in the scratch."""
    import torch
    from w4a4_testutil import bf16_tensor, f32_tensor

    mi = si.moe_inputs("moe_tiny", seed=2)
    s = mi["shape"]
    wq = w4.h32_q4_0_pack_weights(bf16_tensor(mi["wg_bf16"].reshape(s.E * s.N_gate, -1), dev))
    aq = w4.w4a4_rotate_quantize_act(f32_tensor(mi["x_gate"], dev))
    bad = mi["ids"].astype(np.int32).copy()
    bad[3, 1] = -1
    bad[7, 0] = s.E
    bad[0, s.top_k - 1] = 1 << 20
    ids_bad = torch.from_numpy(bad).to(dev)
    ids_good = torch.from_numpy(np.ascontiguousarray(mi["ids"], dtype=np.int32)).to(dev)

    ws = torch.empty(w4.w4a4_gemm_id_workspace_bytes(s.M, s.top_k, s.E, s.K_gate), dtype=torch.uint8, device=dev)
    want = w4.w4a4_gemm_id(wq, s.E, aq, ids_bad, s.top_k, False, ws=ws)
    with pytest.raises(w4.W4A4Error):
        w4.w4a4_gemm_id_status(ws)
    y = torch.full((s.M, s.top_k, s.N_gate), float("nan"), device=dev)
    w4.w4a4_gemm_id_static(wq, s.E, aq, ids_bad, s.top_k, False, y)
    w4.w4a4_check()
    mask = torch.from_numpy((bad < 0) | (bad >= s.E)).to(dev)
    assert int(mask.sum()) == 3
    assert torch.all(y[mask] == 0)
    assert torch.equal(y, want)

    y_good = torch.full((s.M, s.top_k, s.N_gate), float("nan"), device=dev)
    w4.w4a4_gemm_id_static(wq, s.E, aq, ids_good, s.top_k, False, y_good)
    w4.w4a4_check()
    assert torch.equal(y_good, w4.w4a4_gemm_id(wq, s.E, aq, ids_good, s.top_k, False))
