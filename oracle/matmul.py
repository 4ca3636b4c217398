"""Block-scaled W4A4 dot products -- oracle side.

Source: engine docs "The lean option: ROCmFP4, ROCmI4 and Hadamard Q4_0",
section "Hadamard-rotated Q4_0: W4A4 prompt processing" (int4 weights times int4
activations, a Q4_0 code q standing for q - 8, one scale per 32 values) and
section "MoE: W4A4 on the experts" (the same product on the expert matmuls,
MUL_MAT_ID).  Written out:

    P[m][n][b] = sum_{j<32} (q_w[n][32b+j] - 8) * q_a[m][32b+j]     (integers)
    Y[m][n]    = sum_b d_w[n][b] * d_a[m][b] * P[m][n][b]

with d_w the stored fp16 weight scale and d_a the fp32 activation scale.  Here
Y is evaluated in fp64: every term d_w * d_a * P is exact in fp64 (11 + 24 + 12
significant bits), only the sum over b rounds.

For MUL_MAT_ID, token t's slot s uses expert e = ids[t][s]: output row (t, s)
is the dense product of expert e's weights with activation row t (the gate/up
projections, one activation row per token) or row t * top_k + s (the down
projection, one activation row per token-slot).
"""
from __future__ import annotations

import numpy as np

from .quant import act_codes_from_nibbles, unpack_nibbles, weight_codes_from_nibbles


def _wvals(wp: dict) -> np.ndarray:
    q = wp["q"] if "q" in wp else unpack_nibbles(wp["codes"])
    return weight_codes_from_nibbles(q)


def _avals(ap: dict) -> np.ndarray:
    if "q" in ap:
        return np.asarray(ap["q"], dtype=np.int64)
    return act_codes_from_nibbles(unpack_nibbles(ap["codes"]))


def block_partials(wp: dict, ap: dict, m_idx=None, n_idx=None) -> np.ndarray:
    """Integer per-block dot products P [M][N][K/32] (int64).

    With int4 activations |P| <= 2048; with the int8 activations of the exact
    path (``quantize_activations_int8``) |P| <= 32 * 8 * 127 = 32512.
    """
    wv = _wvals(wp)
    av = _avals(ap)
    if m_idx is not None:
        av = av[np.asarray(m_idx)]
    if n_idx is not None:
        wv = wv[np.asarray(n_idx)]
    M, K = av.shape
    N = wv.shape[0]
    B = K // 32
    P = np.einsum("mbj,nbj->mnb", av.reshape(M, B, 32), wv.reshape(N, B, 32))
    assert np.abs(P).max(initial=0) <= (2048 if np.abs(av).max(initial=0) <= 8 else 32512)
    return P


def _matmul_vals(av: np.ndarray, da: np.ndarray, wv: np.ndarray, dw: np.ndarray) -> np.ndarray:
    """Y = sum_b d_w d_a P_b for integer code values av [M][K], wv [N][K] (fp64)."""
    M, K = av.shape
    N = wv.shape[0]
    B = K // 32
    av = av.astype(np.float64).reshape(M, B, 32)
    wv = wv.astype(np.float64).reshape(N, B, 32)
    da = np.asarray(da, dtype=np.float64)
    dw = np.asarray(dw, dtype=np.float64)
    Y = np.zeros((M, N), dtype=np.float64)
    for b in range(B):
        # integer-valued fp64 matmul: every partial sum is an integer < 2^53, so exact
        Pb = av[:, b, :] @ wv[:, b, :].T
        Y += (da[:, b][:, None] * dw[:, b][None, :]) * Pb
    return Y


def w4a4_matmul(wp: dict, ap: dict, m_idx=None, n_idx=None) -> np.ndarray:
    """Y [M][N] in fp64; optionally only rows ``m_idx`` and columns ``n_idx``."""
    wv, dw = _wvals(wp), np.asarray(wp["d16"])
    av, da = _avals(ap), np.asarray(ap["d_a"])
    if m_idx is not None:
        m_idx = np.asarray(m_idx)
        av, da = av[m_idx], da[m_idx]
    if n_idx is not None:
        n_idx = np.asarray(n_idx)
        wv, dw = wv[n_idx], dw[n_idx]
    return _matmul_vals(av, da, wv, dw)


def w4a8_matmul(wp: dict, ap8: dict, m_idx=None, n_idx=None) -> np.ndarray:
    """The exact path's product, rotated Q4_0 weights times int8 activations:
    Y = sum_b d_w d_a P with P = sum_j (q_w - 8) q_a, q_a in -127..127 (fp64).
    The same block-scaled sum as ``w4a4_matmul``; only the activation codes differ."""
    return w4a4_matmul(wp, ap8, m_idx, n_idx)


def w4a16_matmul(wp: dict, ap16: dict, m_idx=None, n_idx=None) -> np.ndarray:
    """The rotate-only route: rotated Q4_0 weights times rotated activations that
    were not quantised (bf16 values xr from ``rotate_activations_bf16``):

        Y[m][n] = sum_b d_w[n][b] * sum_{j<32} xr[m][32b+j] * (q_w[n][32b+j] - 8)

    in fp64.  Each product xr * (q - 8) has at most 8 + 4 significant bits and
    each d_w * (block sum) is exact in fp64 for the value ranges here; the sums
    over j and b round only in fp64.
    """
    wv, dw = _wvals(wp), np.asarray(wp["d16"], dtype=np.float64)
    xr = np.asarray(ap16["xr"], dtype=np.float64)
    if m_idx is not None:
        xr = xr[np.asarray(m_idx)]
    if n_idx is not None:
        n_idx = np.asarray(n_idx)
        wv, dw = wv[n_idx], dw[n_idx]
    M, K = xr.shape
    N = wv.shape[0]
    B = K // 32
    xb = xr.reshape(M, B, 32)
    wb = wv.astype(np.float64).reshape(N, B, 32)
    Y = np.zeros((M, N), dtype=np.float64)
    for b in range(B):
        Y += (xb[:, b, :] @ wb[:, b, :].T) * dw[:, b][None, :]
    return Y


def w4a4_matmul_id(wp_experts: dict, E: int, ap: dict, ids: np.ndarray,
                   act_per_slot: bool, n_idx=None) -> np.ndarray:
    """Expert-routed product: Y [M][top_k][N] in fp64.

    ``wp_experts`` holds all experts' weights stacked along rows (E * N rows):
    expert e owns rows e*N .. e*N + N - 1.  Each (token, slot) output row is an
    independent dense product; they are evaluated expert by expert.
    """
    ids = np.asarray(ids)
    M, top_k = ids.shape
    wv_all, dw_all = _wvals(wp_experts), np.asarray(wp_experts["d16"])
    av_all, da_all = _avals(ap), np.asarray(ap["d_a"])
    N = wv_all.shape[0] // E
    assert N * E == wv_all.shape[0]
    assert ids.min(initial=0) >= 0 and ids.max(initial=0) < E
    cols = np.arange(N) if n_idx is None else np.asarray(n_idx)
    Y = np.zeros((M, top_k, len(cols)), dtype=np.float64)
    for e in range(E):
        ts = np.argwhere(ids == e)  # (t, s) pairs routed to expert e
        if len(ts) == 0:
            continue
        rows = ts[:, 0] * top_k + ts[:, 1] if act_per_slot else ts[:, 0]
        Ye = _matmul_vals(av_all[rows], da_all[rows], wv_all[e * N + cols], dw_all[e * N + cols])
        Y[ts[:, 0], ts[:, 1]] = Ye
    return Y


def exact_matmul(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """The unquantised product sum_k x[m][k] * w[n][k] in fp64 (accuracy reports)."""
    w = np.asarray(w)
    if w.dtype == np.uint16:
        w = (w.astype(np.uint32) << 16).view(np.float32)
    return np.asarray(x, dtype=np.float64) @ np.asarray(w, dtype=np.float64).T
