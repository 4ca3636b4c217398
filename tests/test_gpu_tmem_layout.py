"""Register layout of the 16x256b TMEM load, which the dense fold uses.

The fold reads each 16-lane half of a warp's TMEM quarter with 16x256b loads:
thread t then holds rows t/4 and t/4 + 8 of the half, columns 2(t%4) and
2(t%4) + 1 of every 8-column group.  The probe writes lane * 256 + column with
the 32x32b store (one lane per thread) and reads it back with that load.
"""
import ctypes

import numpy as np
import pytest


@pytest.mark.gpu
def test_tmem_16x256b_register_layout():
    torch = pytest.importorskip("torch")
    assert torch.cuda.is_available()
    from hadamard_rotated_w4a4_gb300 import build as b
    b.build(probes=True)
    lib = ctypes.CDLL(b.PROBE_LIB)
    lib.w4a4_probe_tmem_layout.argtypes = [ctypes.c_void_p]
    lib.w4a4_probe_tmem_layout.restype = ctypes.c_int
    out = np.zeros((128, 8), dtype=np.uint32)
    assert lib.w4a4_probe_tmem_layout(out.ctypes.data) == 0
    want = np.zeros_like(out)
    for tid in range(128):
        w, t = divmod(tid, 32)
        for half in range(2):
            for j in range(4):
                row = 32 * w + 16 * half + t // 4 + 8 * (j // 2)
                col = 2 * (t % 4) + (j % 2)
                want[tid, 4 * half + j] = row * 256 + col
    seen = [[(int(v) // 256, int(v) % 256) for v in out[t]] for t in range(8)]
    assert np.array_equal(out, want), f"(lane, column) per register, threads 0-7: {seen}"
