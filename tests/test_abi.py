"""The C-ABI library loads, exports every symbol include/w4a4.h declares, and its
host-side argument checks return the documented statuses.  No call here reaches
a GPU: each one fails validation before anything is launched, so these run on a
machine without one."""
import ctypes
import os
import re

import pytest

import hadamard_rotated_w4a4_gb300 as w4
from hadamard_rotated_w4a4_gb300 import _Act4Desc, _Q4_0Desc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    return w4.load_library(build_if_missing=True)


def declared_functions():
    text = open(os.path.join(ROOT, "include", "w4a4.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"^\s*#.*$", "", text, flags=re.M)  # preprocessor lines (macros are not exports)
    return sorted(set(re.findall(r"\b(\w+)\s*\([^;{]*\)\s*;", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(w4.EXPORTS) == names


def test_abi_version_and_status_names(lib):
    assert lib.w4a4_abi_version() == 200
    for code, name in w4.STATUS.items():
        assert lib.w4a4_status_name(code).decode() == name


def test_size_queries(lib):
    assert lib.w4a4_q4_0_codes_bytes(5120, 5120) == 5120 * 2560
    assert lib.w4a4_q4_0_scales_bytes(3, 96) == 32  # 3 * 3 * 2 = 18 bytes, padded to 16
    assert lib.w4a4_act4_scales_bytes(2, 64) == 16
    assert lib.w4a4_q4_0_codes_bytes(4, 33) == 0   # K not a multiple of 32
    assert lib.w4a4_gemm_id_workspace_bytes(1024, 8, 128, 2048) >= 4 * (1024 * 8 + 3 * 128) + 1024 * 8 * (1024 + 256)


FAKE = 0x10000  # aligned, never dereferenced: every call below fails validation first


def q4(rows=64, K=256, rotated=True, tag=None):
    return _Q4_0Desc(FAKE, FAKE, FAKE, rows, K, tag if tag is not None else (w4.TAG_Q4_0 | (1 if rotated else 0)))


def a4(rows=64, K=256, rotated=True, tag=None):
    return _Act4Desc(FAKE, FAKE, rows, K, tag if tag is not None else (w4.TAG_ACT4 | (1 if rotated else 0)))


def status(lib, fn, *args):
    s = getattr(lib, fn)(*args)
    return w4.STATUS[s], lib.w4a4_last_error().decode()


def test_gemm_refuses_rotation_mismatch(lib):
    s, msg = status(lib, "w4a4_gemm", ctypes.byref(q4(rotated=True)), ctypes.byref(a4(rotated=False)), FAKE, 64, None, 0, None)
    assert s == "W4A4_ERR_MISMATCH" and "silently wrong" in msg
    s, _ = status(lib, "w4a4_gemm", ctypes.byref(q4(rotated=False)), ctypes.byref(a4(rotated=True)), FAKE, 64, None, 0, None)
    assert s == "W4A4_ERR_MISMATCH"


def test_gemm_refuses_k_mismatch_and_bad_tags(lib):
    s, _ = status(lib, "w4a4_gemm", ctypes.byref(q4(K=256)), ctypes.byref(a4(K=512)), FAKE, 64, None, 0, None)
    assert s == "W4A4_ERR_MISMATCH"
    s, _ = status(lib, "w4a4_gemm", ctypes.byref(q4(tag=w4.TAG_ACT4)), ctypes.byref(a4()), FAKE, 64, None, 0, None)
    assert s == "W4A4_ERR_INVALID_ARG"
    s, _ = status(lib, "w4a4_gemm", None, ctypes.byref(a4()), FAKE, 64, None, 0, None)
    assert s == "W4A4_ERR_INVALID_ARG"


def test_gemm_argument_checks(lib):
    s, _ = status(lib, "w4a4_gemm", ctypes.byref(q4(K=48)), ctypes.byref(a4(K=48)), FAKE, 64, None, 0, None)
    assert s == "W4A4_ERR_INVALID_ARG"
    s, _ = status(lib, "w4a4_gemm", ctypes.byref(q4()), ctypes.byref(a4()), FAKE, 32, None, 0, None)  # ldy < N
    assert s == "W4A4_ERR_INVALID_ARG"
    s, _ = status(lib, "w4a4_gemm", ctypes.byref(q4()), ctypes.byref(a4()), FAKE + 2, 64, None, 0, None)  # y not 4B aligned
    assert s == "W4A4_ERR_ALIGNMENT"
    bad = _Q4_0Desc(FAKE + 8, FAKE, FAKE, 64, 256, w4.TAG_Q4_0 | 1)
    s, _ = status(lib, "w4a4_gemm", ctypes.byref(bad), ctypes.byref(a4()), FAKE, 64, None, 0, None)
    assert s == "W4A4_ERR_ALIGNMENT"
    bad = _Q4_0Desc(FAKE, FAKE, FAKE + 4, 64, 256, w4.TAG_Q4_0 | 1)  # sums not 16-byte aligned
    s, _ = status(lib, "w4a4_gemm", ctypes.byref(bad), ctypes.byref(a4()), FAKE, 64, None, 0, None)
    assert s == "W4A4_ERR_ALIGNMENT"
    s, _ = status(lib, "w4a4_gemm", ctypes.byref(q4()), ctypes.byref(a4()), None, 64, None, 0, None)
    assert s == "W4A4_ERR_INVALID_ARG"


def test_empty_problems_are_no_ops(lib):
    s, _ = status(lib, "w4a4_gemm", ctypes.byref(q4(rows=0)), ctypes.byref(a4()), None, 0, None, 0, None)
    assert s == "W4A4_OK"
    s, _ = status(lib, "w4a4_gemm", ctypes.byref(q4()), ctypes.byref(a4(rows=0)), None, 64, None, 0, None)
    assert s == "W4A4_OK"
    d = _Act4Desc(FAKE, FAKE, 0, 0, 0)
    s, _ = status(lib, "w4a4_rotate_quantize_act", FAKE, 0, 256, 256, 1, ctypes.byref(d), None)
    assert s == "W4A4_OK" and d.rows == 0 and d.K == 256 and d.tag == w4.TAG_ACT4 | 1


def test_act_and_pack_argument_checks(lib):
    d = _Act4Desc(FAKE, FAKE, 0, 0, 0)
    assert status(lib, "w4a4_rotate_quantize_act", FAKE, 4, 100, 100, 1, ctypes.byref(d), None)[0] == "W4A4_ERR_INVALID_ARG"
    assert status(lib, "w4a4_rotate_quantize_act", FAKE, 4, 64, 32, 1, ctypes.byref(d), None)[0] == "W4A4_ERR_INVALID_ARG"
    assert status(lib, "w4a4_rotate_quantize_act", FAKE, 4, 64, 66, 1, ctypes.byref(d), None)[0] == "W4A4_ERR_ALIGNMENT"
    assert status(lib, "w4a4_rotate_quantize_act", FAKE, 4, 64, 64, 2, ctypes.byref(d), None)[0] == "W4A4_ERR_INVALID_ARG"
    assert status(lib, "w4a4_rotate_quantize_act", FAKE, 4, 64, 64, 1, None, None)[0] == "W4A4_ERR_INVALID_ARG"
    w = _Q4_0Desc(FAKE, FAKE, FAKE, 0, 0, 0)
    assert status(lib, "h32_q4_0_pack_weights", FAKE, 2, 4, 64, 64, 1, ctypes.byref(w), None)[0] == "W4A4_ERR_INVALID_ARG"
    assert status(lib, "h32_q4_0_pack_weights", FAKE, 0, 4, 64, 68, 1, ctypes.byref(w), None)[0] == "W4A4_ERR_ALIGNMENT"
    assert status(lib, "h32_q4_0_pack_weights", FAKE + 2, 0, 4, 64, 64, 1, ctypes.byref(w), None)[0] == "W4A4_ERR_ALIGNMENT"
    pw = "h32_q4_0_pack_weights_imatrix"
    assert status(lib, pw, FAKE, 0, 4, 64, 64, 1, FAKE + 4, ctypes.byref(w), None)[0] == "W4A4_ERR_ALIGNMENT"
    assert status(lib, pw, FAKE, 0, 4, 64, 64, 3, FAKE, ctypes.byref(w), None)[0] == "W4A4_ERR_INVALID_ARG"
    assert status(lib, pw, FAKE, 5, 4, 64, 64, 1, None, ctypes.byref(w), None)[0] == "W4A4_ERR_INVALID_ARG"
    s, _ = status(lib, pw, FAKE, 0, 0, 64, 64, 1, None, ctypes.byref(w), None)  # no rows: nothing to do
    assert s == "W4A4_OK" and w.tag == w4.TAG_Q4_0 | 1 and w.K == 64
    assert status(lib, "q4_0_import", FAKE + 1, 4, 64, 1, ctypes.byref(w), None)[0] == "W4A4_ERR_ALIGNMENT"
    assert status(lib, "q4_0_import", FAKE, 4, 64, 3, ctypes.byref(w), None)[0] == "W4A4_ERR_INVALID_ARG"


def test_gemm_id_argument_checks(lib):
    E, N, M, k = 4, 64, 8, 2
    ex = q4(rows=E * N)
    need = lib.w4a4_gemm_id_workspace_bytes(M, k, E, 256)

    def call(experts=ex, E=E, N=N, a=a4(rows=M), M=M, k=k, aps=0, ws_bytes=need, ws=FAKE):
        return status(lib, "w4a4_gemm_id", ctypes.byref(experts), E, N, ctypes.byref(a), FAKE, M, k, aps,
                      FAKE, ws, ws_bytes, None)[0]

    assert call(ws_bytes=need - 16) == "W4A4_ERR_WORKSPACE"
    assert call(ws=None) == "W4A4_ERR_INVALID_ARG"
    assert call(experts=q4(rows=E * N - 1)) == "W4A4_ERR_MISMATCH"
    assert call(a=a4(rows=M * k)) == "W4A4_ERR_MISMATCH"       # per-token rows expected
    assert call(a=a4(rows=M), aps=1) == "W4A4_ERR_MISMATCH"    # per-slot rows expected
    assert call(k=5) == "W4A4_ERR_INVALID_ARG"                 # top_k > E
    assert call(E=0) == "W4A4_ERR_INVALID_ARG"
    assert call(a=a4(rows=M, rotated=False)) == "W4A4_ERR_MISMATCH"
    assert call(ws=FAKE + 8) == "W4A4_ERR_ALIGNMENT"
    assert status(lib, "w4a4_gemm_id_status", None, None)[0] == "W4A4_ERR_INVALID_ARG"


def test_gemm_workspace_query_and_short_workspace(lib):
    # M300 x N640 x K1024: 10 tiles of 8 stages leave most SMs idle as whole tiles,
    # so the split schedule applies and wants a workspace
    need = lib.w4a4_gemm_workspace_bytes(300, 640, 1024)
    assert need > 0 and need % 16 == 0
    assert lib.w4a4_gemm_workspace_bytes(300, 640, 1000) == 0  # K not a multiple of 32
    s, msg = status(lib, "w4a4_gemm", ctypes.byref(q4(rows=640, K=1024)), ctypes.byref(a4(rows=300, K=1024)), FAKE,
                    640, FAKE, 16, None)
    assert s == "W4A4_ERR_WORKSPACE", msg
    s, _ = status(lib, "w4a4_gemm", ctypes.byref(q4(rows=640, K=1024)), ctypes.byref(a4(rows=300, K=1024)), FAKE,
                  640, FAKE + 8, need, None)
    assert s == "W4A4_ERR_ALIGNMENT"


def test_exact_path_validation(lib):
    assert lib.w4a4_act8_codes_bytes(3, 64) == 192
    assert lib.w4a4_act8_scales_bytes(3, 64) == 32  # 3 x 2 fp32, padded to 16 bytes
    a8 = _Act4Desc(FAKE, FAKE, 64, 256, w4.TAG_ACT8 | 1)
    # an int4 descriptor is not an int8 one
    s, _ = status(lib, "w4a8_gemm", ctypes.byref(q4()), ctypes.byref(a4()), FAKE, 64, None, 0, None)
    assert s == "W4A4_ERR_INVALID_ARG"
    s, _ = status(lib, "w4a8_gemm", ctypes.byref(q4(rotated=False)), ctypes.byref(a8), FAKE, 64, None, 0, None)
    assert s == "W4A4_ERR_MISMATCH"
    s, _ = status(lib, "w4a8_gemm_partials", ctypes.byref(q4(K=512)), ctypes.byref(a8), FAKE, None)
    assert s == "W4A4_ERR_MISMATCH"
    d = _Act4Desc(FAKE, FAKE, 0, 0, 0)
    assert status(lib, "w4a8_rotate_quantize_act", FAKE, 4, 100, 100, 1, ctypes.byref(d), None)[0] == "W4A4_ERR_INVALID_ARG"


def test_expanded_activation_operand_size_and_alignment(lib):
    # [round_up(rows, 8)][K] bytes, the buffer rounded to 16 bytes
    assert lib.w4a4_act4_expanded_bytes(512, 5120) == 512 * 5120
    assert lib.w4a4_act4_expanded_bytes(65, 256) == 72 * 256
    assert lib.w4a4_act4_expanded_bytes(1, 32) == 8 * 32
    assert lib.w4a4_act4_expanded_bytes(4, 33) == 0  # K not a multiple of 32
    # a misaligned expanded buffer is refused before any launch, by the quantiser and by the GEMM
    d = _Act4Desc(FAKE, FAKE, 0, 0, 0, FAKE + 8)
    assert status(lib, "w4a4_rotate_quantize_act", FAKE, 4, 64, 64, 1, ctypes.byref(d), None)[0] == "W4A4_ERR_ALIGNMENT"
    bad = _Act4Desc(FAKE, FAKE, 64, 256, w4.TAG_ACT4 | 1, FAKE + 4)
    s, msg = status(lib, "w4a4_gemm", ctypes.byref(q4()), ctypes.byref(bad), FAKE, 64, None, 0, None)
    assert s == "W4A4_ERR_ALIGNMENT" and "expanded" in msg
