"""The seeded input recipe (synth_inputs.py) does what its description says:
shapes, determinism, bf16 rounding, the weights' scale, the ×20 outlier
channels, the SiLU(g)·u draw and distinct routing ids."""
import numpy as np
import pytest

import synth_inputs as si


def test_same_seed_same_inputs_and_different_seed_different_inputs():
    a, b = si.dense_inputs("c0", seed=0), si.dense_inputs("c0", seed=0)
    assert np.array_equal(a["w_bf16"], b["w_bf16"]) and np.array_equal(a["x"], b["x"])
    c = si.dense_inputs("c0", seed=1)
    assert not np.array_equal(a["x"], c["x"])


def test_bf16_rounding_bits_and_values_agree():
    x = np.random.default_rng(3).standard_normal(4096).astype(np.float32)
    bits, vals = si.round_to_bf16(x)
    assert bits.dtype == np.uint16
    assert np.array_equal((bits.astype(np.uint32) << 16).view(np.float32), vals)
    # nearest: no bf16 value lies strictly closer than the chosen one
    up = ((bits.astype(np.uint32) + 1) << 16).view(np.float32)
    dn = ((bits.astype(np.uint32) - 1) << 16).view(np.float32)
    err = np.abs(vals.astype(np.float64) - x)
    assert np.all(err <= np.abs(up.astype(np.float64) - x)) and np.all(err <= np.abs(dn.astype(np.float64) - x))


@pytest.mark.parametrize("name", ["c0", "c1"])
def test_dense_shapes_scale_and_outliers(name):
    d = si.dense_inputs(name)
    s = d["shape"]
    assert d["w_bf16"].shape == (s.N, s.K) and d["w_bf16"].dtype == np.uint16
    assert d["x"].shape == (s.M, s.K) and d["x"].dtype == np.float32
    assert abs(float(d["w"].std()) - 0.02) < 0.02 * 0.05
    cols = np.asarray(d["outlier_cols"])
    assert cols.size == s.n_outliers == len(set(cols.tolist()))
    assert cols.min() >= 0 and cols.max() < s.K
    # the outlier columns carry 20x the spread of the others
    rest = np.setdiff1d(np.arange(s.K), cols)
    ratio = float(d["x"][:, cols].std() / d["x"][:, rest].std())
    assert 17.0 < ratio < 23.0, ratio


def test_outlier_fraction_is_one_percent_of_channels():
    assert si.DENSE["c0"].n_outliers == 2  # 2 of 256 for the tiny case
    for name in ("c1", "c2", "c3"):
        s = si.DENSE[name]
        assert s.n_outliers == s.K // 100


def test_silu_product_activations():
    shape = si.DenseShape("t", 256, 512, 32, 5, silu_act=True)
    d = si.dense_inputs(shape, seed=4)
    rest = np.setdiff1d(np.arange(shape.K), np.asarray(d["outlier_cols"]))
    x = d["x"][:, rest].astype(np.float64)
    # SiLU(g) * u with u ~ N(0, 1) independent of g: mean 0, and E[x^2] = E[SiLU(g)^2]
    g = np.random.default_rng(0).standard_normal(2_000_000)
    e_silu2 = float(np.mean((g / (1.0 + np.exp(-g))) ** 2))
    assert abs(float(x.mean())) < 0.02
    assert abs(float((x ** 2).mean()) - e_silu2) < 0.05 * e_silu2


@pytest.mark.parametrize("name", ["moe_tiny", "c4"])
def test_moe_ids_distinct_per_token_and_shapes(name):
    mi = si.moe_inputs(name)
    s = mi["shape"]
    ids = mi["ids"]
    assert ids.shape == (s.M, s.top_k) and ids.dtype == np.int32
    assert ids.min() >= 0 and ids.max() < s.E
    assert all(len(set(r.tolist())) == s.top_k for r in ids)
    assert mi["wg_bf16"].shape == (s.E, s.N_gate, s.K_gate)
    assert mi["wd_bf16"].shape == (s.E, s.N_down, s.K_down)
    assert mi["x_gate"].shape == (s.M, s.K_gate)
    assert mi["x_down"].shape == (s.M * s.top_k, s.K_down)
    if name == "c4":  # uniform routing: every expert is used, about M * top_k / E times
        counts = np.bincount(ids.ravel(), minlength=s.E)
        assert counts.min() > 0 and abs(float(counts.mean()) - s.M * s.top_k / s.E) < 1e-9
