"""Pins for the CPU oracle: each test ties it to something other than itself --
exact rational arithmetic, an independent construction, a closed form worked out
from the method's definition, hand-worked values (tests/golden/), or brute-force
Python loops on tiny inputs.

Method: engine docs "The lean option: ROCmFP4, ROCmI4 and Hadamard Q4_0",
sections "Hadamard-rotated Q4_0: W4A4 prompt processing" and "MoE: W4A4 on the
experts".
"""
import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth_inputs as si


# ---------------------------------------------------------------- helpers (independent)
def hadamard_recursive(n: int) -> np.ndarray:
    """Sylvester construction H_{2n} = [[H, H], [H, -H]], built without popcounts."""
    H = np.array([[1]], dtype=np.int64)
    while H.shape[0] < n:
        H = np.block([[H, H], [H, -H]])
    return H


H32 = hadamard_recursive(32)


def read_golden(path):
    cases = []
    with open(path) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            name, d, vals, codes = [x.strip() for x in line.split("|")]
            cases.append((name, float(d), np.array([float(v) for v in vals.split()], dtype=np.float32),
                          np.array([int(c) for c in codes.split()])))
    return cases


# ---------------------------------------------------------------- the rotation
def test_c_is_nearest_fp32_to_inv_sqrt32():
    c = Fraction(float(oracle.C_H32))
    bits = int(np.float32(oracle.C_H32).view(np.uint32))
    ulp = Fraction(2) ** (((bits >> 23) & 0xFF) - 127 - 23)
    # c - ulp/2 < 1/sqrt(32) < c + ulp/2  <=>  squares bracket 1/32
    assert (c - ulp / 2) ** 2 < Fraction(1, 32) < (c + ulp / 2) ** 2
    assert bits == 0x3E3504F3


def test_sylvester_matches_recursive_construction_and_is_orthogonal():
    H = oracle.sylvester_h32()
    assert np.array_equal(H, H32)
    assert np.array_equal(H @ H.T, 32 * np.eye(32, dtype=np.int64))
    assert np.array_equal(H, H.T)


def test_butterfly_equals_dense_product_on_integers():
    rng = np.random.default_rng(1)
    x = rng.integers(-1000, 1001, size=(50, 32))
    got = oracle.fwht32(x.astype(np.float32))
    want = x @ H32.T  # |sums| <= 32000: exact in fp32
    assert np.array_equal(got.astype(np.int64), want)
    assert np.array_equal(oracle.fwht32(x.astype(np.int64)), want)


def test_butterfly_of_ones_is_32_e0():
    u = oracle.fwht32(np.ones(32, dtype=np.float32))
    e = np.zeros(32, dtype=np.float32)
    e[0] = 32
    assert np.array_equal(u, e)


def test_rotation_preserves_dot_products_fp64():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((8, 256))
    w = rng.standard_normal((8, 256))
    rx = oracle.rotate_h32(x, dtype=np.float64)
    rw = oracle.rotate_h32(w, dtype=np.float64)
    lhs = (rx * rw).sum(axis=1)
    rhs = (x * w).sum(axis=1)
    assert np.allclose(lhs, rhs, rtol=1e-12, atol=1e-12)
    # orthogonal and symmetric: rotating twice is the identity
    assert np.allclose(oracle.rotate_h32(rx, dtype=np.float64), x, atol=1e-13)


def test_rotation_fp32_within_rounding_bound_of_exact():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((64, 128)) * 3).astype(np.float32)
    y32 = oracle.rotate_h32(x).astype(np.float64)
    exact = (x.astype(np.float64).reshape(64, 4, 32) @ H32.T.astype(np.float64)) / math.sqrt(32)
    l1 = np.abs(x.astype(np.float64)).reshape(64, 4, 32).sum(-1, keepdims=True)
    bound = 8 * 2.0 ** -24 * l1  # five rounded adds plus one rounded multiply per element
    assert np.all(np.abs(y32.reshape(64, 4, 32) - exact) <= bound)


# ---------------------------------------------------------------- quantisers, hand-worked
def test_q4_0_hand_worked_blocks(golden_dir):
    cases = read_golden(os.path.join(golden_dir, "q4_0_hand_blocks.txt"))
    assert len(cases) == 4
    for name, d, vals, codes in cases:
        qz = oracle.quantize_weights_q4_0(vals[None, :])
        assert float(qz["d32"][0, 0]) == d, name
        assert np.array_equal(qz["codes"][0].astype(np.int64), codes), name


def test_int4_hand_worked_blocks(golden_dir):
    cases = read_golden(os.path.join(golden_dir, "int4_act_hand_blocks.txt"))
    assert len(cases) == 3
    for name, d, vals, codes in cases:
        qa = oracle.quantize_act_int4(vals[None, :])
        assert float(qa["d_a"][0, 0]) == d, name
        assert np.array_equal(qa["q"][0].astype(np.int64), codes), name


def test_round_half_away_against_exact_rationals():
    vals = [0.5, -0.5, 1.5, -1.5, 2.5, -2.5, 0.49999997, -0.49999997, 7.4999995, 3.0000002,
            -6.5, 1e-8, -0.0, 0.0, 7.5, -7.5]
    got = oracle.round_half_away(np.array(vals, dtype=np.float32))
    for v, g in zip(vals, got):
        f = Fraction(float(np.float32(v)))
        r = math.floor(abs(f) + Fraction(1, 2))
        assert g == (r if f >= 0 else -r), v


# ---------------------------------------------------------------- quantisers, closed forms
def test_unit_vectors_closed_form():
    """x = e_j in one block: rotated y_i = c * H[i][j]; all magnitudes tie, the
    lowest index (i = 0, H[0][j] = +1) is m, so d = -c/8 and the weight codes are
    0 where H[i][j] = +1 and 16 -> 15 (clamped) where H[i][j] = -1; the int4
    codes are 7 * H[i][j].  Writing the weight values q - 8 as -1/2 - 15/2 H[i][k],
    P[activation e_j][weight e_k] = -1680 [j == k] - 112 [j == 0]."""
    E = np.eye(32, dtype=np.float32)
    wp = oracle.pack_weights(E)  # rows are weight vectors e_j
    ap = oracle.quantize_activations(E)
    c = np.float32(oracle.C_H32)
    for j in range(32):
        want_w = np.where(H32[:, j] == 1, 0, 15)
        assert np.array_equal(wp["q"][j].astype(np.int64), want_w)
        assert wp["d32"][j, 0] == np.float32(-c / np.float32(8))
        assert np.array_equal(ap["q"][j].astype(np.int64), 7 * H32[:, j])
    P = oracle.block_partials(wp, ap)[:, :, 0]  # P[m = activation e_j][n = weight e_k]
    for ja in range(32):
        for kw in range(32):
            assert P[ja, kw] == -1680 * (ja == kw) - 112 * (ja == 0)
            # and by brute force on the sign patterns
            wv = np.where(H32[:, kw] == 1, -8, 7)
            assert P[ja, kw] == int((wv * 7 * H32[:, ja]).sum())


def test_constant_blocks_closed_form():
    """Weight block constant alpha, activation block constant beta: y = 32 alpha c e0,
    weight codes (0, 8, 8, ...), int4 codes (+-7, 0, ...), P = -56 sign(beta), and
    d_w d_a P = (y_w / -8)(|y_a| / 7)(-56 sign beta) = 32 alpha beta (up to the
    fp16 scale), the exact product."""
    rng = np.random.default_rng(4)
    B = 8
    alpha = rng.uniform(0.1, 2.0, B) * rng.choice([-1, 1], B)
    beta = rng.uniform(0.1, 2.0, B) * rng.choice([-1, 1], B)
    w = np.repeat(alpha, 32).astype(np.float32)[None, :]
    x = np.repeat(beta, 32).astype(np.float32)[None, :]
    wp = oracle.pack_weights(w)
    ap = oracle.quantize_activations(x)
    for b in range(B):
        qw = wp["q"][0, 32 * b:32 * b + 32].astype(np.int64)
        qa = ap["q"][0, 32 * b:32 * b + 32].astype(np.int64)
        assert qw[0] == 0 and np.all(qw[1:] == 8)
        assert qa[0] == 7 * np.sign(beta[b]) and np.all(qa[1:] == 0)
    P = oracle.block_partials(wp, ap)[0, 0]
    assert np.array_equal(P, -56 * np.sign(beta).astype(np.int64))
    Y = oracle.w4a4_matmul(wp, ap)[0, 0]
    exact = float(np.sum(32 * np.float32(alpha).astype(np.float64) * np.float32(beta).astype(np.float64)))
    scale = float(np.sum(np.abs(32 * alpha * beta)))
    assert abs(Y - exact) <= 2.0 ** -10 * scale


def test_q4_0_round_trip_bounds_random():
    rng = np.random.default_rng(5)
    y = (rng.standard_normal((200, 256)) * rng.uniform(1e-3, 10, (200, 1))).astype(np.float32)
    qz = oracle.quantize_weights_q4_0(y)
    q = qz["codes"].reshape(200, 8, 32).astype(np.float64)
    d = qz["d32"].astype(np.float64)[..., None]
    yb = y.reshape(200, 8, 32).astype(np.float64)
    err = np.abs(yb - d * (q - 8))
    v = yb / d
    dd = np.broadcast_to(np.abs(d), err.shape)
    inside = np.abs(v) <= 7.49  # not clamped: error at most half a step
    assert np.all(err[inside] <= 0.5 * dd[inside] * (1 + 2.0 ** -20))
    assert np.all(err <= dd * (1 + 2.0 ** -20))  # clamped (+8 -> 15): at most one step
    # the signed-max element maps to code 0
    idx = np.argmax(np.abs(yb), axis=-1)
    assert np.all(np.take_along_axis(q, idx[..., None], -1) == 0)
    # fp16 stored scale within 2^-11 relative (normal fp16 range)
    d16 = qz["d16"].astype(np.float64)
    rel = np.abs(d16 - qz["d32"]) / np.abs(qz["d32"])
    assert np.all(rel <= 2.0 ** -11)


def test_int4_round_trip_bounds_random():
    rng = np.random.default_rng(6)
    y = (rng.standard_normal((200, 256)) * rng.uniform(1e-3, 10, (200, 1))).astype(np.float32)
    qa = oracle.quantize_act_int4(y)
    q = qa["q"].reshape(200, 8, 32).astype(np.float64)
    d = qa["d_a"].astype(np.float64)[..., None]
    yb = y.reshape(200, 8, 32).astype(np.float64)
    assert np.all(np.abs(yb - d * q) <= 0.5 * d * (1 + 2.0 ** -20))
    idx = np.argmax(np.abs(yb), axis=-1)
    assert np.all(np.abs(np.take_along_axis(q, idx[..., None], -1)) == 7)
    assert q.min() >= -7  # -8 is never produced (|y / d_a| <= 7 up to rounding)


def test_activation_scale_invariance_powers_of_two():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((16, 128)).astype(np.float32)
    base = oracle.quantize_activations(x)
    for k in (-3, 5):
        s = np.float32(2.0 ** k)
        sc = oracle.quantize_activations(x * s)
        assert np.array_equal(sc["codes"], base["codes"])
        assert np.array_equal(sc["d_a"], base["d_a"] * s)


# ---------------------------------------------------------------- nibble formats
def test_q_xor_8_is_q_minus_8_exhaustive():
    for q in range(16):
        n = q ^ 8
        signed = n - 16 if n >= 8 else n
        assert signed == q - 8
        assert int(oracle.weight_codes_from_nibbles(np.array([q]))[0]) == q - 8
    for v in range(-8, 8):
        assert int(oracle.act_codes_from_nibbles(np.array([v & 0xF]))[0]) == v


def test_nibble_packing_brute_force():
    rng = np.random.default_rng(8)
    nib = rng.integers(0, 16, size=(3, 96)).astype(np.uint8)
    packed = oracle.pack_nibbles(nib)
    for r in range(3):
        for b in range(3):
            for i in range(16):
                byte = int(nib[r, 32 * b + i]) | (int(nib[r, 32 * b + i + 16]) << 4)
                assert packed[r, 16 * b + i] == byte
    assert np.array_equal(oracle.unpack_nibbles(packed), nib)


def test_q4_0_aos_brute_force():
    rng = np.random.default_rng(9)
    codes = rng.integers(0, 256, size=(2, 48)).astype(np.uint8)  # N=2, K=96
    d16 = rng.standard_normal((2, 3)).astype(np.float16)
    aos = oracle.q4_0_to_aos(codes, d16)
    for n in range(2):
        for b in range(3):
            want = struct.pack("<e", float(d16[n, b])) + bytes(codes[n, 16 * b:16 * b + 16].tolist())
            assert bytes(aos[n, b].tolist()) == want
    c2, d2 = oracle.q4_0_from_aos(aos)
    assert np.array_equal(c2, codes) and np.array_equal(d2.view(np.uint16), d16.view(np.uint16))


# ---------------------------------------------------------------- products, brute force
def _tiny(seed, M=3, N=4, K=64):
    d = si.random_dense(M, K, N, seed=seed)
    return d, oracle.pack_weights(d["w_bf16"]), oracle.quantize_activations(d["x"])


def test_partials_brute_force():
    d, wp, ap = _tiny(10)
    P = oracle.block_partials(wp, ap)
    wq, aq = wp["q"], ap["q"]
    for m in range(3):
        for n in range(4):
            for b in range(2):
                s = 0
                for j in range(32):
                    s += (int(wq[n, 32 * b + j]) - 8) * int(aq[m, 32 * b + j])
                assert P[m, n, b] == s


def test_w4a4_matmul_brute_force():
    d, wp, ap = _tiny(11)
    Y = oracle.w4a4_matmul(wp, ap)
    wq, aq = wp["q"], ap["q"]
    for m in range(3):
        for n in range(4):
            acc = Fraction(0)
            for b in range(2):
                s = sum((int(wq[n, 32 * b + j]) - 8) * int(aq[m, 32 * b + j]) for j in range(32))
                acc += Fraction(float(wp["d16"][n, b])) * Fraction(float(ap["d_a"][m, b])) * s
            assert abs(Y[m, n] - float(acc)) <= 1e-15 * max(1.0, abs(float(acc)))
    # selected rows / columns agree with the full product
    Ys = oracle.w4a4_matmul(wp, ap, m_idx=[2, 0], n_idx=[3, 1])
    assert np.array_equal(Ys, Y[np.ix_([2, 0], [3, 1])])


def test_exact_matmul_brute_force():
    d, _, _ = _tiny(12)
    R = oracle.exact_matmul(d["x"], d["w_bf16"])
    for m in range(3):
        for n in range(4):
            s = math.fsum(float(d["x"][m, k]) * float(d["w"][n, k]) for k in range(64))
            assert abs(R[m, n] - s) <= 1e-12 * max(1.0, abs(s))


@pytest.mark.parametrize("act_per_slot", [False, True])
def test_matmul_id_reduces_to_dense_per_token_slot(act_per_slot):
    mi = si.moe_inputs("moe_tiny", seed=3)
    s = mi["shape"]
    if act_per_slot:
        w, x, N = mi["wd_bf16"], mi["x_down"], s.N_down
    else:
        w, x, N = mi["wg_bf16"], mi["x_gate"], s.N_gate
    wp = oracle.pack_weights(w.reshape(s.E * N, -1))
    ap = oracle.quantize_activations(x)
    Y = oracle.w4a4_matmul_id(wp, s.E, ap, mi["ids"], act_per_slot)
    wq, aq = wp["q"], ap["q"]
    K = x.shape[1]
    for t in range(s.M):
        for slot in range(s.top_k):
            e = int(mi["ids"][t, slot])
            r = t * s.top_k + slot if act_per_slot else t
            for n in (0, N // 2, N - 1):
                acc = 0.0
                for b in range(K // 32):
                    p = sum((int(wq[e * N + n, 32 * b + j]) - 8) * int(aq[r, 32 * b + j]) for j in range(32))
                    acc += float(wp["d16"][e * N + n, b]) * float(ap["d_a"][r, b]) * p
                assert abs(Y[t, slot, n] - acc) <= 1e-12 * max(1.0, abs(acc))


# ---------------------------------------------------------------- the pages' accuracy claim
def test_rotation_reduces_w4a4_error_on_outlier_activations():
    """The rotation spreads a block's few large values before 4-bit rounding, so on
    activations with outlier channels the rotated product is closer to the exact one."""
    d = si.dense_inputs("c0")
    R = oracle.exact_matmul(d["x"], d["w_bf16"])
    Yr = oracle.w4a4_matmul(oracle.pack_weights(d["w_bf16"]), oracle.quantize_activations(d["x"]))
    Yu = oracle.w4a4_matmul(oracle.pack_weights(d["w_bf16"], rotate=False),
                            oracle.quantize_activations(d["x"], rotate=False))
    err_r = np.linalg.norm(Yr - R) / np.linalg.norm(R)
    err_u = np.linalg.norm(Yu - R) / np.linalg.norm(R)
    assert err_r < err_u


# ---------------------------------------------------------------- the exact int8 path
def test_int8_hand_worked_blocks(golden_dir):
    for name, d, vals, codes in read_golden(os.path.join(golden_dir, "int8_act_hand_blocks.txt")):
        out = oracle.quantize_act_int8(vals[None, :])
        assert float(out["d_a"][0, 0]) == d, name
        assert np.array_equal(out["q"][0].astype(np.int64), codes), name


def test_int8_round_trip_bounds_and_amax():
    rng = np.random.default_rng(21)
    y = (rng.standard_normal((64, 256)) * rng.uniform(0.01, 50, (64, 1))).astype(np.float32)
    out = oracle.quantize_act_int8(y)
    q = out["q"].astype(np.float64).reshape(64, 8, 32)
    d = out["d_a"].astype(np.float64)[..., None]
    yb = y.astype(np.float64).reshape(64, 8, 32)
    # |y - d q| <= d / 2 (plus the fp32 rounding of y * (1/d))
    assert np.all(np.abs(yb - d * q) <= d * (0.5 + 1e-5))
    # the element of largest magnitude maps to +-127
    idx = np.argmax(np.abs(yb), axis=-1)
    top = np.take_along_axis(q, idx[..., None], axis=-1)[..., 0]
    assert np.all(np.abs(top) == 127)
    assert np.abs(q).max() <= 127


def test_int8_scale_invariance_powers_of_two():
    rng = np.random.default_rng(22)
    x = rng.standard_normal((8, 128)).astype(np.float32)
    a = oracle.quantize_activations_int8(x)
    for k in (-3, 5):
        b = oracle.quantize_activations_int8((x * np.float32(2.0 ** k)).astype(np.float32))
        assert np.array_equal(a["q"], b["q"])
        assert np.array_equal(b["d_a"], (a["d_a"] * np.float32(2.0 ** k)).astype(np.float32))


def test_w4a8_matmul_brute_force():
    rng = np.random.default_rng(23)
    w = rng.standard_normal((4, 64)).astype(np.float32)
    x = rng.standard_normal((3, 64)).astype(np.float32)
    wp = oracle.pack_weights(w)
    ap = oracle.quantize_activations_int8(x)
    Y = oracle.w4a8_matmul(wp, ap)
    wq, aq = wp["q"], ap["q"]
    for m in range(3):
        for n in range(4):
            acc = Fraction(0)
            for b in range(2):
                s = sum((int(wq[n, 32 * b + j]) - 8) * int(aq[m, 32 * b + j]) for j in range(32))
                acc += Fraction(float(wp["d16"][n, b])) * Fraction(float(ap["d_a"][m, b])) * s
            assert abs(Y[m, n] - float(acc)) <= 1e-15 * max(1.0, abs(float(acc)))
    P = oracle.block_partials(wp, ap)
    for m in range(3):
        for n in range(4):
            for b in range(2):
                s = sum((int(wq[n, 32 * b + j]) - 8) * int(aq[m, 32 * b + j]) for j in range(32))
                assert P[m, n, b] == s


def test_w4a8_constant_blocks_closed_form():
    """Weight block constant alpha, activation block constant beta: rotated, the
    activation block is (32 beta c, 0, ...), int8 codes (+-127, 0, ...), and
    P = -8 * (+-127) = -1016 sign(beta); d_w d_a P = 32 alpha beta up to the fp16 scale."""
    rng = np.random.default_rng(24)
    B = 6
    alpha = rng.uniform(0.1, 2.0, B) * rng.choice([-1, 1], B)
    beta = rng.uniform(0.1, 2.0, B) * rng.choice([-1, 1], B)
    w = np.repeat(alpha, 32).astype(np.float32)[None, :]
    x = np.repeat(beta, 32).astype(np.float32)[None, :]
    wp = oracle.pack_weights(w)
    ap = oracle.quantize_activations_int8(x)
    for b in range(B):
        qa = ap["q"][0, 32 * b:32 * b + 32].astype(np.int64)
        assert qa[0] == 127 * np.sign(beta[b]) and np.all(qa[1:] == 0)
    P = oracle.block_partials(wp, ap)[0, 0]
    assert np.array_equal(P, -1016 * np.sign(beta).astype(np.int64))
    Y = oracle.w4a8_matmul(wp, ap)[0, 0]
    exact = float(np.sum(32 * np.float32(alpha).astype(np.float64) * np.float32(beta).astype(np.float64)))
    assert abs(Y - exact) <= 2.0 ** -10 * float(np.sum(np.abs(32 * alpha * beta)))


def test_int8_path_is_closer_than_int4_to_the_exact_product():
    """Against the product of the (exact) Q4_0 weights with the unrounded rotated
    activations, eight-bit activations lose far less than four-bit ones."""
    d = si.random_dense(16, 512, 24, seed=25)
    wp = oracle.pack_weights(d["w_bf16"])
    w_deq = ((wp["q"].astype(np.float64) - 8).reshape(24, 16, 32)
             * wp["d16"].astype(np.float64)[..., None]).reshape(24, 512)
    ref = oracle.exact_matmul(oracle.rotate_h32(d["x"]), w_deq)
    e4 = np.abs(oracle.w4a4_matmul(wp, oracle.quantize_activations(d["x"])) - ref).mean()
    e8 = np.abs(oracle.w4a8_matmul(wp, oracle.quantize_activations_int8(d["x"])) - ref).mean()
    assert e8 < 0.1 * e4


# ---------------------------------------------------------------- rotate-only route (bf16 activations)
def test_bf16_rounding_hand_worked():
    """Round to nearest even at the bf16 boundary (7 stored mantissa bits): the
    fp32 values halfway between two bf16 neighbours go to the even one."""
    cases = [
        (1.0, 0x3F80),
        (1.0 + 2.0 ** -8, 0x3F80),            # halfway 1 .. 1 + 2^-7, mantissa 0 is even
        (1.0 + 3 * 2.0 ** -8, 0x3F82),        # halfway 1 + 2^-7 .. 1 + 2^-6, mantissa 2 is even
        (1.0 + 2.0 ** -8 + 2.0 ** -20, 0x3F81),  # just past halfway rounds up
        (-2.5, 0xC020),
        (0.0, 0x0000),
        (-0.0, 0x8000),
        (2.0 ** -133, 0x0001),                # smallest bf16 subnormal, exact
        (float(np.float32(3.3895314e38)), 0x7F7F),  # largest finite bf16, exact
        (float(np.finfo(np.float32).max), 0x7F80),  # rounds past it: infinity
    ]
    v = np.array([c[0] for c in cases], dtype=np.float32)
    got = oracle.round_bf16(v)
    assert [int(g) for g in got] == [c[1] for c in cases]
    # widening is exact: bf16 bits -> fp32 value with the low half zero
    assert np.array_equal(oracle.bf16_to_f32(got[:8]).view(np.uint32), got[:8].astype(np.uint32) << 16)


def test_bf16_rounding_matches_torch_conversion():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(31)
    v = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** rng.integers(-30, 30, 20000),
        # every fp32 whose low 16 bits are exactly 0x8000 (ties) or next to it
        (rng.integers(0, 0x7F7F, 4000).astype(np.uint32) << 16 | np.uint32(0x8000)).view(np.float32),
        (rng.integers(0, 0x7F7F, 4000).astype(np.uint32) << 16 | np.uint32(0x7FFF)).view(np.float32),
        (rng.integers(0, 0x7F7F, 4000).astype(np.uint32) << 16 | np.uint32(0x8001)).view(np.float32),
    ]).astype(np.float32)
    v = np.concatenate([v, -v])
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.round_bf16(v), ref)


def test_rotate_only_unit_vectors_hand_derived():
    """e_i in a block rotates to c * (column i of H32): every entry +-c, and
    c = 0x3E3504F3 rounds to the bf16 0x3E35 (low half 0x04F3 < 0x8000)."""
    x = np.zeros((32, 64), dtype=np.float32)
    for i in range(32):
        x[i, 32 + i] = 1.0
    r = oracle.rotate_activations_bf16(x)
    assert np.all(r["x16"][:, :32] == 0)
    want = np.where(H32.T > 0, 0x3E35, 0xBE35).astype(np.uint16)
    assert np.array_equal(r["x16"][:, 32:], want)
    # without the rotation the route is the plain bf16 rounding of x
    y = np.random.default_rng(32).standard_normal((3, 96)).astype(np.float32)
    assert np.array_equal(oracle.rotate_activations_bf16(y, rotate=False)["x16"], oracle.round_bf16(y))


def test_w4a16_matmul_brute_force():
    rng = np.random.default_rng(33)
    w = rng.standard_normal((4, 64)).astype(np.float32)
    x = rng.standard_normal((3, 64)).astype(np.float32) * 3
    wp = oracle.pack_weights(w)
    ap = oracle.rotate_activations_bf16(x)
    Y = oracle.w4a16_matmul(wp, ap)
    wq = wp["q"]
    xr = [[struct.unpack("<f", struct.pack("<I", int(h) << 16))[0] for h in row] for row in ap["x16"]]
    for m in range(3):
        for n in range(4):
            acc = Fraction(0)
            for b in range(2):
                s = sum(Fraction(xr[m][32 * b + j]) * (int(wq[n, 32 * b + j]) - 8) for j in range(32))
                acc += Fraction(float(wp["d16"][n, b])) * s
            assert abs(Y[m, n] - float(acc)) <= 1e-14 * max(1.0, abs(float(acc)))
    Ys = oracle.w4a16_matmul(wp, ap, m_idx=[1], n_idx=[3, 0])
    assert np.array_equal(Ys, Y[np.ix_([1], [3, 0])])


def test_w4a16_reduces_to_plain_matmul_on_exact_inputs():
    """Weights that Q4_0 stores exactly (each block d (q - 8) with a code 0 at
    the signed max, fp16 d) and bf16 activations, no rotation: the route's
    product is the ordinary matmul x @ w^T."""
    rng = np.random.default_rng(34)
    N, M, K = 5, 4, 128
    B = K // 32
    q = rng.integers(0, 16, (N, B, 32))
    q[:, :, 0] = 0                                   # value -8 d: the signed max
    q[:, :, 1:] = np.clip(q[:, :, 1:], 1, 15)        # |q - 8| <= 7 elsewhere
    d = np.float16(rng.uniform(0.01, 0.2, (N, B)) * rng.choice([-1, 1], (N, B))).astype(np.float32)
    w = (d[..., None] * (q - 8)).astype(np.float32).reshape(N, K)
    x = oracle.bf16_to_f32(oracle.round_bf16(rng.standard_normal((M, K)).astype(np.float32)))
    wp = oracle.pack_weights(w, rotate=False)
    assert np.array_equal(wp["q"].reshape(N, B, 32), q) and np.array_equal(wp["d16"].astype(np.float32), d)
    Y = oracle.w4a16_matmul(wp, oracle.rotate_activations_bf16(x, rotate=False))
    ref = x.astype(np.float64) @ w.astype(np.float64).T
    assert np.allclose(Y, ref, rtol=1e-13, atol=1e-13)


def test_w4a16_constant_blocks_closed_form():
    """Unrotated: weight block constant alpha (codes 0 everywhere, d = -alpha/8)
    and activation block constant beta (bf16-exact): Y = sum_b 32 d (-8) beta."""
    rng = np.random.default_rng(35)
    B = 5
    alpha = np.float32(rng.uniform(0.1, 2.0, B) * rng.choice([-1, 1], B))
    beta = oracle.bf16_to_f32(oracle.round_bf16(np.float32(rng.uniform(0.1, 2.0, B) * rng.choice([-1, 1], B))))
    w = np.repeat(alpha, 32).astype(np.float32)[None, :]
    x = np.repeat(beta, 32).astype(np.float32)[None, :]
    wp = oracle.pack_weights(w, rotate=False)
    assert np.all(wp["q"] == 0)
    Y = oracle.w4a16_matmul(wp, oracle.rotate_activations_bf16(x, rotate=False))[0, 0]
    d = wp["d16"][0].astype(np.float64)
    assert Y == pytest.approx(float(np.sum(32 * d * -8 * beta.astype(np.float64))), rel=1e-15)
    assert abs(Y - float(np.sum(32 * alpha.astype(np.float64) * beta))) <= 2.0 ** -10 * float(np.sum(np.abs(32 * alpha * beta)))


def test_rotate_only_is_closer_than_int8_to_the_exact_product():
    """Against the exact Q4_0 weights times the unrounded rotated activations,
    bf16 activations lose less than the int8 codes of the exact path."""
    d = si.random_dense(16, 512, 24, seed=36)
    wp = oracle.pack_weights(d["w_bf16"])
    w_deq = ((wp["q"].astype(np.float64) - 8).reshape(24, 16, 32)
             * wp["d16"].astype(np.float64)[..., None]).reshape(24, 512)
    ref = oracle.exact_matmul(oracle.rotate_h32(d["x"]), w_deq)
    e8 = np.abs(oracle.w4a8_matmul(wp, oracle.quantize_activations_int8(d["x"])) - ref).mean()
    e16 = np.abs(oracle.w4a16_matmul(wp, oracle.rotate_activations_bf16(d["x"])) - ref).mean()
    assert e16 < 0.5 * e8


# ---------------------------------------------------------------- importance-weighted Q4_0 (converter)
def _nearest_error(y, w, d):
    """Independent restatement: error of scale d with each code the nearest integer in -8..7 (fp64)."""
    y = np.asarray(y, np.float64)
    c = np.clip(np.floor(y / d + 0.5), -8, 7)
    return float(np.sum(w * (y - d * c) ** 2))


def test_rotate_importance_is_the_block_mean():
    """Every entry of H32 is +-1, so diag(Hn D Hn^T)_i = sum_j imp_j / 32."""
    rng = np.random.default_rng(50)
    imp = rng.uniform(0, 5, 256)
    r = oracle.rotate_importance(imp)
    want = np.repeat(imp.reshape(8, 32).mean(axis=1), 32)
    assert np.allclose(r, want, rtol=1e-14, atol=0)
    # a one-hot block spreads evenly; the trace (total importance) is kept
    one = np.zeros(64)
    one[37] = 3.0
    assert np.allclose(oracle.rotate_importance(one), np.r_[np.zeros(32), np.full(32, 3.0 / 32)], rtol=1e-14, atol=1e-17)
    assert oracle.rotate_importance(imp).sum() == pytest.approx(imp.sum(), rel=1e-14)


def test_weighted_scale_beats_a_dense_scan():
    """No scale on a fine grid (nor next to d*) has a smaller weighted error."""
    rng = np.random.default_rng(51)
    for trial in range(12):
        y = (rng.standard_normal(32) * (1 + 5 * (trial % 3 == 0) * (np.arange(32) == trial))).astype(np.float32)
        w = rng.uniform(0, 3, 32) if trial % 2 else np.ones(32)
        d = oracle.weighted_block_scale(y, w)
        e = _nearest_error(y, w, d)
        a = float(np.max(np.abs(y)))
        grid = np.concatenate([np.linspace(-a / 4, -a / 20, 20000), np.linspace(a / 20, a / 4, 20000)])
        scan = min(_nearest_error(y, w, g) for g in grid)
        assert e <= scan * (1 + 1e-12), (trial, e, scan)
        for f in (1 - 1e-7, 1 + 1e-7):
            assert e <= _nearest_error(y, w, d * f) * (1 + 1e-12)


def test_weighted_q4_0_exact_blocks_and_plain_scale():
    """A block Q4_0 holds exactly keeps error 0 (its plain scale); elsewhere the
    weighted choice is never worse than the plain scale under the same code
    rule, and clearly better on average for Gaussian blocks."""
    rng = np.random.default_rng(52)
    q = rng.integers(1, 16, (6, 32))
    q[:, 0] = 0
    d0 = np.float16(rng.uniform(0.02, 0.5, 6) * rng.choice([-1, 1], 6)).astype(np.float32)
    y = (d0[:, None] * (q - 8)).astype(np.float32)
    r = oracle.quantize_weights_q4_0_weighted(y, np.ones(32))
    assert np.array_equal(r["d16"][:, 0].astype(np.float32), d0) and np.array_equal(r["codes"], q)
    y = rng.standard_normal((400, 32)).astype(np.float32)
    w = rng.uniform(0.1, 2.0, (400, 32))
    r = oracle.quantize_weights_q4_0_weighted(y, w)
    plain = oracle.quantize_weights_q4_0(y)
    ew, ep = [], []
    for i in range(400):
        cw = r["codes"][i].astype(np.float64) - 8
        ew.append(np.sum(w[i] * (y[i] - np.float64(r["d16"][i, 0]) * cw) ** 2))
        dp = np.float32(plain["d16"][i, 0])
        cp = np.clip(np.copysign(np.floor(np.abs(y[i] * (np.float32(1) / dp)) + 0.5), y[i] * (np.float32(1) / dp)), -8, 7)
        ep.append(np.sum(w[i] * (y[i] - np.float64(dp) * cp) ** 2))
    ew, ep = np.array(ew), np.array(ep)
    assert np.all(ew <= ep * (1 + 1e-12))
    assert ew.mean() < 0.9 * ep.mean()


def test_weighted_q4_0_power_of_two_weight_invariance():
    rng = np.random.default_rng(53)
    y = rng.standard_normal((50, 64)).astype(np.float32)
    w = rng.uniform(0, 2, (50, 64))
    a = oracle.quantize_weights_q4_0_weighted(y, w)
    b = oracle.quantize_weights_q4_0_weighted(y, w * 8.0)
    assert np.array_equal(a["codes"], b["codes"]) and np.array_equal(a["d16"], b["d16"])


def test_rotated_imatrix_does_nothing():
    """The pages: on the rotated file an imatrix does nothing, Q4_0 having one
    scale per 32 values.  With the matching change the rotated importance is
    flat inside every block, so the weighted choice is the unweighted one."""
    rng = np.random.default_rng(54)
    w = rng.standard_normal((20, 256)).astype(np.float32)
    imp = rng.uniform(0, 10, 256) ** 3
    a = oracle.pack_weights_imatrix(w, imp, rotate=True)
    b = oracle.pack_weights_imatrix(w, np.ones(256), rotate=True)
    same = np.all(a["q"].reshape(20, 8, 32) == b["q"].reshape(20, 8, 32), axis=-1) & (a["d16"] == b["d16"])
    assert same.mean() >= 0.99
    # unrotated, the same importance does move the scales
    c = oracle.pack_weights_imatrix(w, imp, rotate=False)
    d = oracle.pack_weights_imatrix(w, np.ones(256), rotate=False)
    assert np.mean(c["d16"] != d["d16"]) > 0.3


def test_effective_importance_cleans_before_rotating():
    imp = np.r_[np.full(32, 2.0), [-1.0, np.nan, np.inf] + [4.0] * 29]
    e = oracle.effective_importance(imp, 64, rotate=True)
    assert np.allclose(e[:32], 2.0, rtol=1e-14) and np.allclose(e[32:], 4.0 * 29 / 32, rtol=1e-14)
    assert np.array_equal(oracle.effective_importance(None, 64, rotate=False), np.ones(64))
