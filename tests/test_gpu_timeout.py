"""A bounded pipeline wait that runs out, on the GPU, without a fault or a hang.

The test hook w4a4_debug_set_wait_limit shortens the super-tile GEMM's wait
bound to 50 us and holds its producer back for 5 ms: the MMA issuer, the
converters and the workers each give up on their first wait, the CTA winds down
(no copy or MMA is in flight) and returns, and w4a4_check reports
W4A4_ERR_TIMEOUT.  With the defaults restored, the next call on the same inputs
is correct again (compared with the oracle).
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


@pytest.fixture
def short_waits():
    w4.w4a4_debug_set_wait_limit(50_000, 5_000_000)
    yield
    w4.w4a4_debug_set_wait_limit(0, 0)


def test_gemm_wait_runs_out_then_recovers(dev):
    d = si.random_dense(200, 1024, 384, seed=21)
    wq = w4.h32_q4_0_pack_weights(bf16_tensor(d["w_bf16"], dev))
    a = w4.w4a4_rotate_quantize_act(f32_tensor(d["x"], dev))
    assert a.expanded is not None  # the super-tile kernel serves this call
    w4.w4a4_check()
    try:
        w4.w4a4_debug_set_wait_limit(50_000, 5_000_000)
        y = w4.w4a4_gemm(wq, a, ws=None)
        with pytest.raises(w4.W4A4Error) as e:
            w4.w4a4_check()
        assert e.value.status_name == "W4A4_ERR_TIMEOUT"
    finally:
        w4.w4a4_debug_set_wait_limit(0, 0)
    w4.w4a4_check()  # the condition was cleared by the check that reported it
    y = w4.w4a4_gemm(wq, a, ws=None)
    w4.w4a4_check()
    R = oracle.w4a4_matmul(oracle.pack_weights(d["w_bf16"]), oracle.quantize_activations(d["x"]))
    assert_close(y.cpu().numpy(), R)


def test_routed_wait_runs_out_then_recovers(dev):
    mi = si.moe_inputs("moe_tiny", seed=5)
    s = mi["shape"]
    wq = w4.h32_q4_0_pack_weights(bf16_tensor(mi["wg_bf16"].reshape(s.E * s.N_gate, -1), dev))
    aq = w4.w4a4_rotate_quantize_act(f32_tensor(mi["x_gate"], dev))
    ids = torch.from_numpy(np.ascontiguousarray(mi["ids"], dtype=np.int32)).to(dev)
    w4.w4a4_check()
    try:
        w4.w4a4_debug_set_wait_limit(50_000, 5_000_000)
        w4.w4a4_gemm_id(wq, s.E, aq, ids, s.top_k, False)
        with pytest.raises(w4.W4A4Error) as e:
            w4.w4a4_check()
        assert e.value.status_name == "W4A4_ERR_TIMEOUT"
    finally:
        w4.w4a4_debug_set_wait_limit(0, 0)
    y = w4.w4a4_gemm_id(wq, s.E, aq, ids, s.top_k, False)
    w4.w4a4_check()
    R = oracle.w4a4_matmul_id(oracle.pack_weights(mi["wg_bf16"].reshape(s.E * s.N_gate, -1)), s.E,
                              oracle.quantize_activations(mi["x_gate"]), mi["ids"], False)
    assert_close(y.cpu().numpy(), R)
