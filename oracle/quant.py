"""Q4_0 weight quantiser and per-block int4 activation quantiser -- oracle side.

Sources (engine docs "The lean option: ROCmFP4, ROCmI4 and Hadamard Q4_0"):

* section "Hadamard-rotated Q4_0: W4A4 prompt processing": weights are plain
  Q4_0, read bit for bit; a Q4_0 code q stands for q - 8, and q ^ 8 read as a
  signed 4-bit number is exactly q - 8; only the activations are rounded to 4
  bits, after the same per-32-block rotation as the weights;
* section "MoE: W4A4 on the experts": Q4_0 has one scale per 32 values.

Readings where the pages are silent:

* weight block: m = the rotated value of largest magnitude, the lowest index
  on ties; d = m / -8 in fp32; id = 1/d (0 when d == 0); code
  q = clamp(round_half_away(fl(y * id)) + 8, 0, 15); the stored scale is d
  rounded to fp16 (nearest even); the codes use the fp32 d;
* activation block: a = max |y|; d_a = a / 7 in fp32, stored as fp32;
  id = 1/d_a (0 when d_a == 0); q = clamp(round_half_away(fl(y * id)), -8, 7);
* nibble order inside a block's 16 bytes: byte i holds element i in its low
  nibble and element i + 16 in its high nibble (the Q4_0 block layout); the
  activations use the same order, each code as a 4-bit two's complement nibble.

All rounding decisions are taken on fp32 values computed with one IEEE
operation per step, exactly as written; round_half_away is evaluated in fp64,
where |v| + 0.5 is exact for every fp32 v.
"""
from __future__ import annotations

import numpy as np

from .hadamard import rotate_h32


def round_half_away(v: np.ndarray) -> np.ndarray:
    """Round to the nearest integer, ties away from zero (returns float64)."""
    v64 = np.asarray(v, dtype=np.float64)
    return np.copysign(np.floor(np.abs(v64) + 0.5), v64)


def _blocks(y: np.ndarray) -> np.ndarray:
    K = y.shape[-1]
    assert K % 32 == 0, "K must be a multiple of 32"
    return y.reshape(y.shape[:-1] + (K // 32, 32))


def _safe_recip(d: np.ndarray) -> np.ndarray:
    out = np.zeros_like(d)
    nz = d != 0
    out[nz] = np.float32(1.0) / d[nz]
    return out


def quantize_weights_q4_0(y: np.ndarray) -> dict:
    """Q4_0-quantise fp32 values y [..., K] per 32-block.

    Returns codes (uint8 0..15, [..., K]), d32 (fp32 scale, [..., K/32]) and d16
    (the stored fp16 scale).
    """
    y = np.asarray(y, dtype=np.float32)
    blk = _blocks(y)
    idx = np.argmax(np.abs(blk), axis=-1)  # first index of the largest magnitude
    m = np.take_along_axis(blk, idx[..., None], axis=-1)[..., 0]
    d = (m / np.float32(-8.0)).astype(np.float32)
    inv = _safe_recip(d)
    v = (blk * inv[..., None]).astype(np.float32)
    q = np.clip(round_half_away(v) + 8.0, 0.0, 15.0).astype(np.uint8)
    return {"codes": q.reshape(y.shape), "d32": d, "d16": d.astype(np.float16)}


def quantize_act_int4(y: np.ndarray) -> dict:
    """int4-quantise fp32 values y [..., K] per 32-block.

    Returns q (int8 in -8..7, [..., K]) and d_a (fp32, [..., K/32]).
    """
    y = np.asarray(y, dtype=np.float32)
    blk = _blocks(y)
    a = np.max(np.abs(blk), axis=-1)
    d_a = (a / np.float32(7.0)).astype(np.float32)
    inv = _safe_recip(d_a)
    v = (blk * inv[..., None]).astype(np.float32)
    q = np.clip(round_half_away(v), -8.0, 7.0).astype(np.int8)
    return {"q": q.reshape(y.shape), "d_a": d_a}


def quantize_act_int8(y: np.ndarray) -> dict:
    """int8-quantise fp32 values y [..., K] per 32-block (the exact path's
    8-bit activations, engine docs page above, section "Hadamard-rotated Q4_0:
    W4A4 prompt processing": with W4A4 switched off the rotated file runs on
    the exact int8 path).

    Reading: a = max |y|; d_a = a / 127 in fp32; id = 1/d_a (0 when d_a == 0);
    q = clamp(round_half_away(fl(y * id)), -127, 127).  Returns q (int8,
    [..., K]) and d_a (fp32, [..., K/32]).
    """
    y = np.asarray(y, dtype=np.float32)
    blk = _blocks(y)
    a = np.max(np.abs(blk), axis=-1)
    d_a = (a / np.float32(127.0)).astype(np.float32)
    inv = _safe_recip(d_a)
    v = (blk * inv[..., None]).astype(np.float32)
    q = np.clip(round_half_away(v), -127.0, 127.0).astype(np.int8)
    return {"q": q.reshape(y.shape), "d_a": d_a}


def pack_nibbles(nib: np.ndarray) -> np.ndarray:
    """Pack 4-bit values (uint8 0..15, [..., K]) into [..., K/2] bytes, Q4_0 order."""
    blk = _blocks(np.asarray(nib, dtype=np.uint8))
    lo = blk[..., :16]
    hi = blk[..., 16:]
    packed = (lo | (hi << 4)).astype(np.uint8)
    return packed.reshape(nib.shape[:-1] + (nib.shape[-1] // 2,))


def unpack_nibbles(packed: np.ndarray) -> np.ndarray:
    """Inverse of ``pack_nibbles``: [..., K/2] bytes -> [..., K] values 0..15."""
    p = np.asarray(packed, dtype=np.uint8)
    Kh = p.shape[-1]
    assert Kh % 16 == 0
    blk = p.reshape(p.shape[:-1] + (Kh // 16, 16))
    out = np.concatenate([blk & 0x0F, blk >> 4], axis=-1)
    return out.reshape(p.shape[:-1] + (Kh * 2,))


def weight_codes_from_nibbles(nib: np.ndarray) -> np.ndarray:
    """Q4_0 code q -> the integer it stands for, q - 8 (int64)."""
    return np.asarray(nib, dtype=np.int64) - 8


def act_codes_from_nibbles(nib: np.ndarray) -> np.ndarray:
    """4-bit two's complement nibble -> signed integer in -8..7 (int64)."""
    n = np.asarray(nib, dtype=np.int64)
    return np.where(n >= 8, n - 16, n)


def q4_0_to_aos(codes_packed: np.ndarray, d16: np.ndarray) -> np.ndarray:
    """SoA (codes [N][K/2], fp16 scales [N][K/32]) -> canonical 18-byte blocks.

    Each block is the little-endian fp16 scale followed by its 16 code bytes;
    returns uint8 [N][K/32][18].
    """
    N, Kh = codes_packed.shape
    B = Kh // 16
    out = np.empty((N, B, 18), dtype=np.uint8)
    out[..., 0:2] = np.ascontiguousarray(d16, dtype="<f2").view(np.uint8).reshape(N, B, 2)
    out[..., 2:] = codes_packed.reshape(N, B, 16)
    return out


def q4_0_from_aos(blocks: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Canonical 18-byte blocks [N][B][18] -> (codes [N][16B], fp16 scales [N][B])."""
    blocks = np.asarray(blocks, dtype=np.uint8)
    N, B, _ = blocks.shape
    d16 = np.ascontiguousarray(blocks[..., 0:2]).view("<f2").reshape(N, B).astype(np.float16)
    codes = np.ascontiguousarray(blocks[..., 2:]).reshape(N, B * 16)
    return codes, d16


def _weights_fp32(w: np.ndarray) -> np.ndarray:
    w = np.asarray(w)
    if w.dtype == np.uint16:  # bf16 bit patterns: exact widening to fp32
        return (w.astype(np.uint32) << 16).view(np.float32)
    return w.astype(np.float32)


def pack_weights(w: np.ndarray, rotate: bool = True) -> dict:
    """Weights [N][K] (fp32 values or bf16 bits as uint16) -> rotated Q4_0.

    Returns codes (packed bytes [N][K/2]), d16 [N][K/32] (stored scales), d32
    and q (unpacked codes [N][K]).
    """
    wf = _weights_fp32(w)
    y = rotate_h32(wf) if rotate else wf
    qz = quantize_weights_q4_0(y)
    return {"codes": pack_nibbles(qz["codes"]), "d16": qz["d16"], "d32": qz["d32"],
            "q": qz["codes"], "rotated": bool(rotate)}


def quantize_activations(x: np.ndarray, rotate: bool = True) -> dict:
    """Activations [M][K] fp32 -> rotated int4 codes + fp32 per-block scales.

    Returns codes (packed bytes [M][K/2], two's complement nibbles), d_a
    [M][K/32] fp32 and q (int8 [M][K]).
    """
    xf = np.asarray(x, dtype=np.float32)
    y = rotate_h32(xf) if rotate else xf
    qa = quantize_act_int4(y)
    nib = (qa["q"].astype(np.int16) & 0x0F).astype(np.uint8)
    return {"codes": pack_nibbles(nib), "d_a": qa["d_a"], "q": qa["q"], "rotated": bool(rotate)}


def quantize_activations_int8(x: np.ndarray, rotate: bool = True) -> dict:
    """Activations [M][K] fp32 -> rotated int8 codes [M][K] + fp32 per-block scales."""
    xf = np.asarray(x, dtype=np.float32)
    y = rotate_h32(xf) if rotate else xf
    qa = quantize_act_int8(y)
    return {"codes8": qa["q"].copy(), "d_a": qa["d_a"], "q": qa["q"], "rotated": bool(rotate)}


def round_bf16(v: np.ndarray) -> np.ndarray:
    """fp32 values -> bf16 bit patterns (uint16), round to nearest, ties to even.

    Integer arithmetic on the fp32 bits: add 0x7FFF plus the lowest kept bit,
    keep the top 16 bits.  A finite value that rounds past the largest bf16
    becomes infinity, as IEEE rounding does.
    """
    bits = np.asarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    keep_lsb = (bits >> 16) & 1
    return ((bits + 0x7FFF + keep_lsb) >> 16).astype(np.uint16)


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> fp32 values (exact widening)."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def rotate_activations_bf16(x: np.ndarray, rotate: bool = True) -> dict:
    """The rotate-only route: activations [M][K] fp32 rotated per 32-block (the
    same fp32 rotation the quantisers see) and not rounded to 4 bits; they are
    carried as bf16 (round to nearest even), the tensor-core operand type.

    Returns x16 (bf16 bits [M][K]) and xr (their fp32 values).
    """
    xf = np.asarray(x, dtype=np.float32)
    y = rotate_h32(xf) if rotate else xf
    h = round_bf16(y)
    return {"x16": h, "xr": bf16_to_f32(h), "rotated": bool(rotate)}


# ---------------------------------------------------------------- importance-weighted Q4_0 (converter)
def rotate_importance(imp: np.ndarray) -> np.ndarray:
    """The importance the rotated input channels inherit (section "Hadamard-
    rotated Q4_0: W4A4 prompt processing": the converter gives the imatrix the
    matching change).  An imatrix keeps one value per input channel, the
    diagonal of E[x x^T]; with rotated inputs Hn x (Hn = H32 / sqrt 32, per
    block) that diagonal becomes diag(Hn diag(imp) Hn^T), evaluated here with
    the explicit matrices in fp64.
    """
    from .hadamard import sylvester_h32

    imp = np.asarray(imp, dtype=np.float64)
    K = imp.shape[-1]
    assert K % 32 == 0, "K must be a multiple of 32"
    Hn = sylvester_h32().astype(np.float64) / np.sqrt(32.0)
    out = np.empty_like(imp)
    for b in range(K // 32):
        A = Hn @ np.diag(imp[..., 32 * b:32 * b + 32]) @ Hn.T
        out[..., 32 * b:32 * b + 32] = np.diag(A)
    return out


def _clean_weights(w: np.ndarray) -> np.ndarray:
    w = np.asarray(w, dtype=np.float64)
    w = np.where(np.isfinite(w) & (w > 0), w, 0.0)
    return w if w.sum() > 0 else np.ones_like(w)


def _codes_for(y32: np.ndarray, d16: np.float16) -> np.ndarray:
    """The Q4_0 code rule for a stored scale: id = fl32(1/d) (0 if d == 0),
    q = clamp(round_half_away(fl32(y * id)) + 8, 0, 15)."""
    d = np.float32(d16)
    inv = np.float32(1.0) / d if d != 0 else np.float32(0.0)
    v = (y32 * inv).astype(np.float32)
    return np.clip(round_half_away(v) + 8.0, 0.0, 15.0).astype(np.int64)


def _weighted_error(y32: np.ndarray, w: np.ndarray, d16: np.float16) -> float:
    q = _codes_for(y32, d16)
    return float(np.sum(w * (y32.astype(np.float64) - float(d16) * (q - 8)) ** 2))


def weighted_block_scale(y32: np.ndarray, w: np.ndarray) -> float:
    """The real scale d minimising sum_j w_j (y_j - d c_j)^2 with every c_j the
    nearest integer to y_j / d in -8..7 (fp64; 0 for an all-zero block).

    With s = 1/d the nearest codes change only where some y_j s crosses a
    half-integer k + 1/2 (k = -8..6); between consecutive crossings the codes c
    are fixed and the best d is the weighted least-squares d = sum w y c /
    sum w c^2, with error sum w y^2 - (sum w y c)^2 / sum w c^2.  Every interval
    (each evaluated at its midpoint, plus one point beyond each end) is tried;
    the first largest (sum w y c)^2 / sum w c^2 wins.  When the winning codes
    avoid -8, (-d, -c) is an equally good twin: the sign of the plain Q4_0
    scale m / -8 is kept.
    """
    y = np.asarray(y32, dtype=np.float64)
    nz = y != 0
    if not nz.any():
        return 0.0
    ks = np.arange(-8, 7, dtype=np.float64) + 0.5
    bps = np.unique((ks[None, :] / y[nz][:, None]).ravel())
    pts = np.concatenate([[bps[0] - abs(bps[0]) - 1.0], (bps[:-1] + bps[1:]) / 2, [bps[-1] + abs(bps[-1]) + 1.0]])
    c = np.clip(np.rint(y[None, :] * pts[:, None]), -8, 7)
    num = (c * (w * y)[None, :]).sum(axis=1)
    den = (c * c * w[None, :]).sum(axis=1)
    ok = den > 0
    score = np.full(len(pts), -1.0)
    score[ok] = num[ok] ** 2 / den[ok]
    i = int(np.argmax(score))
    if not ok[i]:
        return 0.0
    d = float(num[i] / den[i])
    m = y[int(np.argmax(np.abs(y)))]
    if not np.any(c[i] == -8) and d * -m < 0:
        d = -d
    return d


def quantize_weights_q4_0_weighted(y: np.ndarray, omega: np.ndarray) -> dict:
    """Importance-weighted Q4_0 of fp32 values y [..., K] with per-element
    weights omega (broadcast against y; negative or non-finite weights count
    as 0, an all-zero block of weights as uniform).

    Per block: d* = weighted_block_scale; the stored fp16 scale is the best, by
    the weighted error under the code rule of ``_codes_for``, of (in order) the
    plain Q4_0 scale fp16(m / -8), fp16(d*) and the two fp16 neighbours of
    fp16(d*); the first smallest error wins.  Returns codes, d16.
    """
    y = np.asarray(y, dtype=np.float32)
    blk = _blocks(y)
    om = np.broadcast_to(np.asarray(omega, dtype=np.float64), y.shape)
    wblk = _blocks(om)
    plain = quantize_weights_q4_0(y)["d16"]
    flat_y = blk.reshape(-1, 32)
    flat_w = wblk.reshape(-1, 32)
    flat_p = np.asarray(plain).reshape(-1)
    d16 = np.empty(flat_y.shape[0], dtype=np.float16)
    codes = np.empty(flat_y.shape, dtype=np.uint8)
    for i in range(flat_y.shape[0]):
        yb, wb = flat_y[i], _clean_weights(flat_w[i])
        ds = np.float16(weighted_block_scale(yb, wb))
        cands = [flat_p[i], ds, np.nextafter(ds, np.float16(-np.inf)), np.nextafter(ds, np.float16(np.inf))]
        best, best_e = None, None
        for cd in cands:
            if not np.isfinite(cd):
                continue
            e = _weighted_error(yb, wb, cd)
            if best_e is None or e < best_e:
                best, best_e = cd, e
        d16[i] = best
        codes[i] = _codes_for(yb, best)
    return {"codes": codes.reshape(y.shape), "d16": d16.reshape(blk.shape[:-1])}


def effective_importance(imp, K: int, rotate: bool) -> np.ndarray:
    """The per-element weights of the weighted packer: imp [K] (None: ones) with
    negative or non-finite entries set to 0, then, when rotating, given the
    matching change (``rotate_importance``)."""
    imp = np.ones(K) if imp is None else np.asarray(imp, dtype=np.float64)
    imp = np.where(np.isfinite(imp) & (imp > 0), imp, 0.0)
    return rotate_importance(imp) if rotate else imp


def pack_weights_imatrix(w: np.ndarray, imp, rotate: bool = True) -> dict:
    """Weights [N][K] (fp32 or bf16 bits) and an importance vector imp [K] (or
    None) -> importance-weighted Q4_0: the weights rotated as in
    ``pack_weights`` and the importance given the matching change, or both as
    they are when rotate is False.  Returns codes (packed), d16, q."""
    wf = _weights_fp32(w)
    y = rotate_h32(wf) if rotate else wf
    om = effective_importance(imp, wf.shape[-1], rotate)
    qz = quantize_weights_q4_0_weighted(y, om[None, :])
    return {"codes": pack_nibbles(qz["codes"]), "d16": qz["d16"], "q": qz["codes"], "rotated": bool(rotate)}
