"""The 32-point Walsh-Hadamard rotation (H32) -- oracle side.

Source: engine docs "The lean option: ROCmFP4, ROCmI4 and Hadamard Q4_0",
section "Hadamard-rotated Q4_0: W4A4 prompt processing": a 32-point
Walsh-Hadamard rotation is applied to each 32-element block along K, to the
activations at run time and to the weights once, so that x.w = (Hx).(Hw) in
exact arithmetic.  For that identity H must be orthogonal, i.e. the +-1
Walsh-Hadamard matrix scaled by 1/sqrt(32).

Readings (the page names the transform but fixes neither its ordering nor the
floating-point evaluation order):

* natural (Sylvester) order: H[i][j] = (-1)^popcount(i & j);
* the rotation is evaluated as an unnormalised butterfly in the input's
  precision, stages h = 1, 2, 4, 8, 16 in that order, each pair
  (i, i+h) with i & h == 0 becoming (a + b, a - b); then every element is
  multiplied by c = fl32(1/sqrt(32)).  No fused multiply-add anywhere.

The quantiser's integer decisions are taken on these fp32 values, so this
evaluation order is part of what the CUDA path has to reproduce bit for bit.
"""
from __future__ import annotations

import numpy as np

#: fl32(1/sqrt(32)), the normalisation of the 32-point rotation.
C_H32 = np.float32(1.0 / np.sqrt(32.0))


def sylvester_h32() -> np.ndarray:
    """The +-1 Walsh-Hadamard matrix of order 32 in natural order, int64."""
    i = np.arange(32)
    bits = np.bitwise_and(i[:, None], i[None, :])
    parity = np.zeros_like(bits)
    for s in range(5):
        parity ^= (bits >> s) & 1
    return np.where(parity == 0, 1, -1).astype(np.int64)


def fwht32(v: np.ndarray) -> np.ndarray:
    """Unnormalised Walsh-Hadamard butterfly over the last axis (length 32).

    Works in the dtype of ``v`` (fp32 for the quantisers, fp64 for checks).
    Stage h pairs element i with i + h for every i whose bit h is clear.
    """
    v = np.asarray(v)
    assert v.shape[-1] == 32
    u = v.copy()
    lead = u.shape[:-1]
    h = 1
    while h < 32:
        # index i = hi * 2h + s * h + lo with s the bit of weight h
        t = u.reshape(lead + (32 // (2 * h), 2, h))
        a = t[..., 0, :]
        b = t[..., 1, :]
        u = np.stack([a + b, a - b], axis=-2).reshape(lead + (32,))
        h *= 2
    return u


def rotate_h32(x: np.ndarray, dtype=np.float32) -> np.ndarray:
    """Rotate every 32-element block along the last axis: y = fl(fwht32(x) * c).

    ``x`` has last dimension K, a multiple of 32.  In fp32 this is the value the
    quantisers round; in fp64 (``dtype=np.float64``) c is 1/sqrt(32) in fp64.
    """
    x = np.asarray(x, dtype=dtype)
    K = x.shape[-1]
    assert K % 32 == 0, "K must be a multiple of 32"
    blocks = x.reshape(x.shape[:-1] + (K // 32, 32))
    c = C_H32 if dtype == np.float32 else np.float64(1.0) / np.sqrt(np.float64(32.0))
    u = fwht32(blocks)
    y = u * np.asarray(c, dtype=dtype)
    return y.reshape(x.shape)
