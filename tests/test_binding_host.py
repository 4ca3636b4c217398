"""Host-side behaviour of the Python binding that needs no GPU."""
import pytest
import torch

import hadamard_rotated_w4a4_gb300 as w4


class _FakeLib:
    """Stands in for libw4a4.so: w4a4_check reports the given status."""

    def __init__(self, status: int):
        self.status = status

    def w4a4_check(self, stream):
        return self.status

    def w4a4_last_error(self):
        return b"w4a4_check: a bounded wait inside a GEMM kernel gave up"


@pytest.fixture
def cached_workspaces(monkeypatch):
    monkeypatch.setattr(w4, "_GEMM_WS", {(0, 7): torch.zeros(16, dtype=torch.uint8),
                                         (0, 9): torch.ones(16, dtype=torch.uint8)})
    return w4._GEMM_WS


def test_timeout_drops_cached_gemm_workspaces(monkeypatch, cached_workspaces):
    # a kernel that gave up can leave stream-K tickets standing in its workspace
    monkeypatch.setattr(w4, "load_library", lambda *a, **k: _FakeLib(8))
    with pytest.raises(w4.W4A4Error) as e:
        w4.w4a4_check(0)
    assert e.value.status_name == "W4A4_ERR_TIMEOUT"
    assert w4._GEMM_WS == {}


def test_ok_check_keeps_cached_gemm_workspaces(monkeypatch, cached_workspaces):
    monkeypatch.setattr(w4, "load_library", lambda *a, **k: _FakeLib(0))
    w4.w4a4_check(0)
    assert sorted(w4._GEMM_WS) == [(0, 7), (0, 9)]


def test_other_errors_keep_cached_gemm_workspaces(monkeypatch, cached_workspaces):
    monkeypatch.setattr(w4, "load_library", lambda *a, **k: _FakeLib(5))
    with pytest.raises(w4.W4A4Error):
        w4.w4a4_check(0)
    assert len(w4._GEMM_WS) == 2
