"""GPU parity of the small-batch kernel (1 to 8 activation rows): bit for bit
the tensor-core kernel's whole-tile result, and within 1e-3 of the oracle."""
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


@pytest.mark.parametrize("M", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("K,N", [(256, 256), (4096, 33), (5120, 130), (17408, 96)])
def test_small_m_bit_exact_with_tensor_core_kernel(dev, M, K, N):
    d = si.random_dense(M, K, N, seed=M * 31 + K + N)
    wq = w4.h32_q4_0_pack_weights(bf16_tensor(d["w_bf16"], dev))
    aq = w4.w4a4_rotate_quantize_act(f32_tensor(d["x"], dev))
    ys = w4.w4a4_gemm_small_m(wq, aq)
    yt = w4.w4a4_gemm(wq, aq, ws=None)
    torch.cuda.synchronize()
    assert torch.equal(ys, yt), f"max |diff| {float((ys - yt).abs().max())}"
    R = oracle.w4a4_matmul(oracle.pack_weights(d["w_bf16"]), oracle.quantize_activations(d["x"]))
    assert_close(ys.cpu().numpy(), R)


def test_small_m_row_stride_and_unrotated(dev):
    d = si.random_dense(4, 512, 40, seed=8)
    wq = w4.h32_q4_0_pack_weights(bf16_tensor(d["w_bf16"], dev), rotate=False)
    aq = w4.w4a4_rotate_quantize_act(f32_tensor(d["x"], dev), rotate=False)
    big = torch.full((4, 48), 3.0, dtype=torch.float32, device=dev)
    w4.w4a4_gemm_small_m(wq, aq, y=big[:, :40])
    yb = big.cpu().numpy()
    assert np.all(yb[:, 40:] == 3.0)
    R = oracle.w4a4_matmul(oracle.pack_weights(d["w_bf16"], False), oracle.quantize_activations(d["x"], False))
    assert_close(yb[:, :40], R)


def test_small_m_refuses_nine_rows(dev):
    d = si.random_dense(9, 64, 8, seed=2)
    wq = w4.h32_q4_0_pack_weights(bf16_tensor(d["w_bf16"], dev))
    aq = w4.w4a4_rotate_quantize_act(f32_tensor(d["x"], dev))
    with pytest.raises(w4.W4A4Error) as e:
        w4.w4a4_gemm_small_m(wq, aq)
    assert e.value.status_name == "W4A4_ERR_UNSUPPORTED"
