"""The arithmetic premises of the tensor-core path, checked on the CPU.

The GEMM computes each block's integer dot product on the fp8 tensor cores and
removes the activations' offset inside the fold's first fused multiply-add.
Those steps are exact only if:
* every 4-bit value v is the e4m3 value v * 2^-9 (bytes 0x00..0x0F linear, 0x80
  the sign), so that the expanded weight bytes (q - 8) and activation bytes
  (a + 8) stand for exactly those integers;
* a block's 32 products, and every partial sum of them in any order, are exact
  in fp32;
* the offset term -d_w * 8 * S_w (d_w an fp16 scale, S_w a block's code sum) is
  exact in fp32, so that fma(D, d_w, -d_w 8 S_w) rounds once, to fl(d_w * P).

The e4m3 decoder below follows the format's definition (1 sign bit, 4 exponent
bits with bias 7, 3 mantissa bits, subnormals at exponent 0, 0x7F / 0xFF NaN);
torch's float8_e4m3fn conversion cross-checks it.
"""
import numpy as np
import pytest


def e4m3(byte: int) -> float:
    s = -1.0 if byte & 0x80 else 1.0
    e = (byte >> 3) & 0xF
    m = byte & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * m * 2.0 ** -9  # subnormal: m / 8 * 2^(1 - 7)
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def test_decoder_matches_torch_float8_e4m3fn():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8_e4m3fn in this torch")
    b = torch.arange(256, dtype=torch.uint8)
    t = b.view(torch.float8_e4m3fn).float().numpy()
    mine = np.array([e4m3(i) for i in range(256)])
    nan = np.isnan(mine)
    assert np.array_equal(nan, np.isnan(t))
    assert np.array_equal(mine[~nan], t[~nan].astype(np.float64))


def test_nibble_values_are_exact_e4m3_values():
    for v in range(16):
        assert e4m3(v) == v * 2.0 ** -9
        assert e4m3(0x80 | v) == -v * 2.0 ** -9


def test_expanded_weight_bytes_encode_q_minus_8():
    # the packers' expanded byte: q - 8 >= 0 -> q - 8, else 0x80 | (8 - q)
    for q in range(16):
        byte = q - 8 if q >= 8 else 0x80 | (8 - q)
        assert e4m3(byte) == (q - 8) * 2.0 ** -9


def test_expanded_activation_bytes_encode_a_plus_8():
    # the activation kernel's expanded byte: the two's complement nibble XOR 8
    for a in range(-8, 8):
        nibble = a & 0xF
        byte = nibble ^ 0x8
        assert byte == a + 8
        assert e4m3(byte) == (a + 8) * 2.0 ** -9


def test_block_sums_are_exact_in_fp32_in_any_order():
    rng = np.random.default_rng(0)
    for trial in range(2000):
        w = rng.integers(-8, 8, 32)   # q - 8
        u = rng.integers(0, 16, 32)   # a + 8 (the offset operand), or signed below
        if trial % 2:
            u = rng.integers(-8, 8, 32)
        if trial < 8:  # the largest magnitudes
            w = np.full(32, -8)
            u = np.full(32, 15 if trial % 2 == 0 else -8)
        exact = int(np.dot(w, u))
        prods = (w.astype(np.float32) * np.float32(2.0 ** -9)) * (u.astype(np.float32) * np.float32(2.0 ** -9))
        for order in (np.arange(32), rng.permutation(32), np.arange(32)[::-1]):
            acc = np.float32(0.0)
            for i in order:
                acc = np.float32(acc + prods[i])
            assert float(acc) == exact * 2.0 ** -18, (trial, exact, float(acc))


def _fp16_values(rng, n):
    bits = rng.integers(0, 0x7C00, n).astype(np.uint16)  # finite, positive
    return bits.view(np.float16).astype(np.float64)


def test_offset_term_is_exact_in_fp32():
    rng = np.random.default_rng(1)
    edges = np.array([6.0e-8, 6.1035e-5, 65504.0, 1.0, 2.0 ** -14]).astype(np.float16).astype(np.float64)
    d = np.concatenate([_fp16_values(rng, 20000), edges])  # fp16 values only, smallest subnormal to largest
    s = rng.integers(-256, 257, d.size)
    s[:4] = [-256, 256, 0, 255]
    term = -d * 8.0 * s                       # exact in fp64 (11 + 3 + 9 significant bits)
    assert np.array_equal(term.astype(np.float32).astype(np.float64), term)
    # the kernel forms it as (d_w 2^18) * (S_w 2^-15) in fp32: both factors and the product are exact
    a = (d * 2.0 ** 18).astype(np.float32)
    b = (s * 2.0 ** -15).astype(np.float32)
    assert np.array_equal(a.astype(np.float64), d * 2.0 ** 18)
    assert np.array_equal(b.astype(np.float64), s * 2.0 ** -15)
    assert np.array_equal((-a * b).astype(np.float64), term)


def test_first_fold_fma_rounds_once_to_dw_times_p():
    # t = fma(D 2^-18, d_w 2^18, -d_w 8 S_w) with D = P + 8 S_w: the exact value of
    # the fma's product-plus-addend is d_w * P, so its one rounding is fl32(d_w * P)
    rng = np.random.default_rng(2)
    for _ in range(20000):
        q = rng.integers(0, 16, 32) - 8
        a = rng.integers(-8, 8, 32)
        P = int(np.dot(q, a))
        S = int(q.sum())
        D = P + 8 * S
        dw = float(_fp16_values(rng, 1)[0])
        exact = (D * 2.0 ** -18) * (dw * 2.0 ** 18) + (-dw * 8.0 * S)  # every step exact in fp64
        assert exact == dw * P
        assert np.float32(exact) == np.float32(dw * P)
