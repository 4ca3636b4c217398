"""hadamard_rotated_w4a4_gb300 -- Python binding of libw4a4.so.

The prefill matmul of a Hadamard-rotated Q4_0 model run as W4A4 (engine docs
"The lean option: ROCmFP4, ROCmI4 and Hadamard Q4_0", sections "Hadamard-rotated
Q4_0: W4A4 prompt processing" and "MoE: W4A4 on the experts"), on GB300.

This module only marshals arguments: every step runs in the CUDA library's
kernels.  PyTorch provides device memory (output tensors are allocated with
``torch.empty``) and the current CUDA stream.  If the library is missing the
calls raise; there is no CPU fallback.

Entry points (same names as the C ABI in ``include/w4a4.h``):

* ``h32_q4_0_pack_weights(w, rotate=True)`` -> :class:`Q4_0Weights`
* ``q4_0_import(blocks, K, rotated=True)`` -> :class:`Q4_0Weights`
* ``w4a4_rotate_quantize_act(x, rotate=True)`` -> :class:`Act4`
* ``w4a4_gemm(w, a)`` -> fp32 [M][N]
* ``w4a4_gemm_partials(w, a)`` -> int32 [M][N][K/32]
* ``w4a4_gemm_id(experts, E, a, ids, top_k, act_per_slot)`` -> fp32 [M][top_k][N]
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

from . import build as _build

__all__ = [
    "W4A4Error", "Q4_0Weights", "Act4", "load_library", "library_path",
    "h32_q4_0_pack_weights", "q4_0_import", "w4a4_rotate_quantize_act",
    "w4a4_gemm", "w4a4_gemm_workspace_bytes", "w4a4_gemm_partials", "w4a4_gemm_id", "w4a4_gemm_id_status",
    "w4a4_gemm_id_workspace_bytes", "w4a4_gemm_id_static", "w4a4_check", "STATUS",
    "Act8", "w4a8_rotate_quantize_act", "w4a8_gemm", "w4a8_gemm_partials", "w4a8_gemm_workspace_bytes",
    "w4a4_gemm_small_m",
]

STATUS = {
    0: "W4A4_OK", 1: "W4A4_ERR_INVALID_ARG", 2: "W4A4_ERR_ALIGNMENT", 3: "W4A4_ERR_MISMATCH",
    4: "W4A4_ERR_UNSUPPORTED", 5: "W4A4_ERR_CUDA", 6: "W4A4_ERR_DEVICE_FLAG", 7: "W4A4_ERR_WORKSPACE",
    8: "W4A4_ERR_TIMEOUT",
}
TAG_Q4_0 = 0x51340000
TAG_ACT4 = 0x41340000
TAG_ACT8 = 0x41380000
TAG_ACT16 = 0x41420000
TAG_ROTATED = 0x1

#: every symbol include/w4a4.h declares
EXPORTS = [
    "w4a4_q4_0_codes_bytes", "w4a4_q4_0_scales_bytes", "w4a4_q4_0_sums_bytes", "w4a4_q4_0_expanded_bytes",
    "w4a4_act4_codes_bytes",
    "w4a4_act4_scales_bytes", "w4a4_act4_expanded_bytes", "h32_q4_0_pack_weights", "q4_0_import", "w4a4_rotate_quantize_act", "w4a4_gemm", "w4a4_gemm_workspace_bytes",
    "w4a4_gemm_partials", "w4a4_gemm_id", "w4a4_gemm_id_workspace_bytes", "w4a4_gemm_id_status", "w4a4_gemm_id_static", "w4a4_check", "w4a4_last_error",
    "w4a4_status_name", "w4a4_abi_version", "w4a4_act8_codes_bytes", "w4a4_act8_scales_bytes", "w4a4_gemm_small_m",
    "w4a8_rotate_quantize_act", "w4a8_gemm", "w4a8_gemm_partials", "w4a8_gemm_workspace_bytes",
    "w4a4_act16_values_bytes", "w4a16_rotate_act", "w4a16_gemm", "w4a16_gemm_workspace_bytes",
    "h32_q4_0_pack_weights_imatrix", "w4a4_debug_set_wait_limit",
]


class W4A4Error(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        self.status_name = STATUS.get(status, f"status {status}")
        super().__init__(f"{self.status_name}: {message}")


class _Q4_0Desc(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("sums", ctypes.c_void_p),
                ("rows", ctypes.c_int64), ("K", ctypes.c_int64), ("tag", ctypes.c_uint32),
                ("expanded", ctypes.c_void_p)]


class _Act4Desc(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("rows", ctypes.c_int64),
                ("K", ctypes.c_int64), ("tag", ctypes.c_uint32), ("expanded", ctypes.c_void_p)]


class _Act16Desc(ctypes.Structure):
    _fields_ = [("values", ctypes.c_void_p), ("rows", ctypes.c_int64), ("K", ctypes.c_int64),
                ("tag", ctypes.c_uint32)]


_LIB = None


def library_path() -> str:
    return _build.LIB


def load_library(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libw4a4.so (built in-tree by ``hadamard_rotated_w4a4_gb300.build``)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError(f"{path} is missing: build it with `python -m hadamard_rotated_w4a4_gb300.build`")
        _build.build()
    lib = ctypes.CDLL(path)
    i64, vp, i32, u = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    for name in ("w4a4_q4_0_codes_bytes", "w4a4_q4_0_scales_bytes", "w4a4_q4_0_sums_bytes", "w4a4_q4_0_expanded_bytes",
                 "w4a4_act4_codes_bytes",
                 "w4a4_act4_scales_bytes", "w4a4_act4_expanded_bytes", "w4a4_act8_codes_bytes",
                 "w4a4_act8_scales_bytes"):
        f = getattr(lib, name)
        f.argtypes, f.restype = [i64, i64], u
    lib.h32_q4_0_pack_weights.argtypes = [vp, i32, i64, i64, i64, i32, ctypes.POINTER(_Q4_0Desc), vp]
    lib.h32_q4_0_pack_weights_imatrix.argtypes = [vp, i32, i64, i64, i64, i32, vp, ctypes.POINTER(_Q4_0Desc), vp]
    lib.q4_0_import.argtypes = [vp, i64, i64, i32, ctypes.POINTER(_Q4_0Desc), vp]
    lib.w4a4_rotate_quantize_act.argtypes = [vp, i64, i64, i64, i32, ctypes.POINTER(_Act4Desc), vp]
    lib.w4a4_gemm.argtypes = [ctypes.POINTER(_Q4_0Desc), ctypes.POINTER(_Act4Desc), vp, i64, vp, u, vp]
    lib.w4a4_gemm_workspace_bytes.argtypes, lib.w4a4_gemm_workspace_bytes.restype = [i64, i64, i64], u
    lib.w4a8_rotate_quantize_act.argtypes = [vp, i64, i64, i64, i32, ctypes.POINTER(_Act4Desc), vp]
    lib.w4a8_gemm.argtypes = [ctypes.POINTER(_Q4_0Desc), ctypes.POINTER(_Act4Desc), vp, i64, vp, u, vp]
    lib.w4a8_gemm_partials.argtypes = [ctypes.POINTER(_Q4_0Desc), ctypes.POINTER(_Act4Desc), vp, vp]
    lib.w4a8_gemm_workspace_bytes.argtypes, lib.w4a8_gemm_workspace_bytes.restype = [i64, i64, i64], u
    lib.w4a16_rotate_act.argtypes = [vp, i64, i64, i64, i32, ctypes.POINTER(_Act16Desc), vp]
    lib.w4a16_gemm.argtypes = [ctypes.POINTER(_Q4_0Desc), ctypes.POINTER(_Act16Desc), vp, i64, vp, u, vp]
    lib.w4a16_gemm_workspace_bytes.argtypes, lib.w4a16_gemm_workspace_bytes.restype = [i64, i64, i64], u
    lib.w4a4_gemm_small_m.argtypes = [ctypes.POINTER(_Q4_0Desc), ctypes.POINTER(_Act4Desc), vp, i64, vp]
    lib.w4a4_gemm_partials.argtypes = [ctypes.POINTER(_Q4_0Desc), ctypes.POINTER(_Act4Desc), vp, vp]
    lib.w4a4_gemm_id.argtypes = [ctypes.POINTER(_Q4_0Desc), i32, i64, ctypes.POINTER(_Act4Desc), vp, i64, i32, i32,
                                 vp, vp, u, vp]
    lib.w4a4_gemm_id_workspace_bytes.argtypes, lib.w4a4_gemm_id_workspace_bytes.restype = [i64, i32, i32, i64], u
    lib.w4a4_gemm_id_status.argtypes = [vp, vp]
    lib.w4a4_gemm_id_static.argtypes = [ctypes.POINTER(_Q4_0Desc), i32, i64, ctypes.POINTER(_Act4Desc), vp, i64, i32,
                                         i32, vp, vp]
    lib.w4a4_check.argtypes = [vp]
    lib.w4a4_debug_set_wait_limit.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
    lib.w4a4_debug_set_wait_limit.restype = None
    for name in ("h32_q4_0_pack_weights", "q4_0_import", "w4a4_rotate_quantize_act", "w4a4_gemm",
                 "w4a4_gemm_partials", "w4a4_gemm_id", "w4a4_gemm_id_status", "w4a4_check",
                 "w4a8_rotate_quantize_act", "w4a8_gemm", "w4a8_gemm_partials", "w4a4_gemm_small_m"):
        getattr(lib, name).restype = ctypes.c_int
    lib.w4a4_last_error.argtypes, lib.w4a4_last_error.restype = [], ctypes.c_char_p
    lib.w4a4_status_name.argtypes, lib.w4a4_status_name.restype = [ctypes.c_int], ctypes.c_char_p
    lib.w4a4_abi_version.argtypes, lib.w4a4_abi_version.restype = [], ctypes.c_int
    _LIB = lib
    return lib


def _check(status: int) -> None:
    if status != 0:
        msg = load_library().w4a4_last_error().decode(errors="replace")
        raise W4A4Error(status, msg)


def _stream(stream=None) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _cuda(t: torch.Tensor, name: str) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")


@dataclass
class Q4_0Weights:
    """Q4_0 weights in the library's layout: codes uint8 [rows][K/2], scales fp16 [rows][K/32],
    the derived per-block code sums int16 [rows][K/32] and, optionally, the expanded operand
    (e4m3 bytes of q - 8, [round_up(rows, 8)][K]) that lets the dense GEMM skip converting
    the weights."""
    codes: torch.Tensor
    scales_buf: torch.Tensor  # uint8 buffer (padded to 16 bytes) holding the fp16 scales
    sums_buf: torch.Tensor    # uint8 buffer (padded to 16 bytes) holding the int16 block sums
    rows: int
    K: int
    rotated: bool
    expanded: torch.Tensor | None = None  # uint8 buffer of w4a4_q4_0_expanded_bytes, or None

    @property
    def sums(self) -> torch.Tensor:
        n = self.rows * (self.K // 32)
        return self.sums_buf[: 2 * n].view(torch.int16).view(self.rows, self.K // 32)

    @property
    def scales(self) -> torch.Tensor:
        n = self.rows * (self.K // 32)
        return self.scales_buf[: 2 * n].view(torch.float16).view(self.rows, self.K // 32)

    @property
    def tag(self) -> int:
        return TAG_Q4_0 | (TAG_ROTATED if self.rotated else 0)

    def desc(self) -> _Q4_0Desc:
        return _Q4_0Desc(self.codes.data_ptr(), self.scales_buf.data_ptr(), self.sums_buf.data_ptr(), self.rows,
                         self.K, self.tag, self.expanded.data_ptr() if self.expanded is not None else None)

    def head(self, rows: int) -> "Q4_0Weights":
        """The first `rows` rows (views of the same buffers)."""
        return Q4_0Weights(self.codes[:rows], self.scales_buf, self.sums_buf, rows, self.K, self.rotated,
                           self.expanded)

    def without_expanded(self) -> "Q4_0Weights":
        """The same weights without the expanded operand (the GEMM then converts the codes)."""
        return Q4_0Weights(self.codes, self.scales_buf, self.sums_buf, self.rows, self.K, self.rotated)


@dataclass
class Act4:
    """int4 activations: codes uint8 [rows][K/2] (two's complement nibbles), scales fp32 [rows][K/32]
    and, optionally, the expanded operand (the offset codes a + 8 as bytes, [round_up(rows, 8)][K])
    that lets the dense GEMM, with expanded weights, skip converting the activations."""
    codes: torch.Tensor
    scales_buf: torch.Tensor
    rows: int
    K: int
    rotated: bool
    expanded: torch.Tensor | None = None  # uint8 buffer of w4a4_act4_expanded_bytes, or None

    @property
    def scales(self) -> torch.Tensor:
        n = self.rows * (self.K // 32)
        return self.scales_buf[: 4 * n].view(torch.float32).view(self.rows, self.K // 32)

    @property
    def tag(self) -> int:
        return TAG_ACT4 | (TAG_ROTATED if self.rotated else 0)

    def head(self, rows: int) -> "Act4":
        """The first `rows` rows (views of the same buffers)."""
        return Act4(self.codes[:rows], self.scales_buf, rows, self.K, self.rotated, self.expanded)

    def without_expanded(self) -> "Act4":
        """The same activations without the expanded operand (the GEMM then converts the codes)."""
        return Act4(self.codes, self.scales_buf, self.rows, self.K, self.rotated)

    def desc(self) -> _Act4Desc:
        return _Act4Desc(self.codes.data_ptr(), self.scales_buf.data_ptr(), self.rows, self.K, self.tag,
                         self.expanded.data_ptr() if self.expanded is not None else None)


def alloc_q4_0(rows: int, K: int, device, rotated: bool = True, expanded: bool = False) -> Q4_0Weights:
    """Buffers for Q4_0 weights.  expanded=True also allocates the optional expanded
    operand (1 byte per weight beside the 0.5-byte codes and the 0.125 bytes of
    scales and sums: 2.9x the Q4_0 footprint); the dense GEMM then loads it instead
    of converting the codes.  The codes stay the format of record either way."""
    lib = load_library()
    nc, ns = lib.w4a4_q4_0_codes_bytes(rows, K), lib.w4a4_q4_0_scales_bytes(rows, K)
    if K <= 0 or K % 32:
        raise W4A4Error(1, f"K={K} must be a positive multiple of 32")
    codes = torch.empty(max(nc, 16), dtype=torch.uint8, device=device)[:nc].view(rows, K // 2)
    sbuf = torch.empty(max(ns, 16), dtype=torch.uint8, device=device)
    ubuf = torch.empty(max(lib.w4a4_q4_0_sums_bytes(rows, K), 16), dtype=torch.uint8, device=device)
    ebuf = (torch.empty(max(lib.w4a4_q4_0_expanded_bytes(rows, K), 16), dtype=torch.uint8, device=device)
            if expanded else None)
    return Q4_0Weights(codes, sbuf, ubuf, rows, K, rotated, ebuf)


def alloc_act4(rows: int, K: int, device, rotated: bool = True, expanded: bool = True) -> Act4:
    lib = load_library()
    if K <= 0 or K % 32:
        raise W4A4Error(1, f"K={K} must be a positive multiple of 32")
    nc, ns = lib.w4a4_act4_codes_bytes(rows, K), lib.w4a4_act4_scales_bytes(rows, K)
    codes = torch.empty(max(nc, 16), dtype=torch.uint8, device=device)[:nc].view(rows, K // 2)
    sbuf = torch.empty(max(ns, 16), dtype=torch.uint8, device=device)
    ebuf = None
    if expanded:
        ne = lib.w4a4_act4_expanded_bytes(rows, K)
        ebuf = torch.empty(max(ne, 16), dtype=torch.uint8, device=device)
        ebuf[rows * K:].zero_()  # the pad rows are read into unused MMA columns only; keep them defined
    return Act4(codes, sbuf, rows, K, rotated, ebuf)


def h32_q4_0_pack_weights(w: torch.Tensor, rotate: bool = True, out: Q4_0Weights | None = None,
                          stream=None, expanded: bool = False) -> Q4_0Weights:
    """Rotate (H32 per 32-block along K) and Q4_0-pack weights w [N][K] (bf16 or fp32, CUDA).
    expanded=True also writes the optional expanded operand (see alloc_q4_0)."""
    _cuda(w, "w")
    if w.dim() != 2 or w.stride(1) != 1:
        raise ValueError("w must be a 2-D tensor with unit stride along K")
    dtype = {torch.bfloat16: 0, torch.float32: 1}.get(w.dtype)
    if dtype is None:
        raise ValueError("w must be bf16 or fp32")
    N, K = w.shape
    out = out or alloc_q4_0(N, K, w.device, rotate, expanded)
    d = out.desc()
    ldw = w.stride(0) if N > 1 else K  # a single row's stride is meaningless (may be 0)
    _check(load_library().h32_q4_0_pack_weights(w.data_ptr(), dtype, N, K, ldw, int(rotate),
                                                 ctypes.byref(d), _stream(stream)))
    out.rotated = bool(d.tag & TAG_ROTATED)
    return out


def h32_q4_0_pack_weights_imatrix(w: torch.Tensor, imatrix: torch.Tensor | None, rotate: bool = True,
                                  out: Q4_0Weights | None = None, stream=None, expanded: bool = False) -> Q4_0Weights:
    """As h32_q4_0_pack_weights, with each block's scale chosen against the importance vector
    imatrix (fp32 [K], CUDA, the unrotated input channels' importance; None = uniform)."""
    _cuda(w, "w")
    if w.dim() != 2 or w.stride(1) != 1:
        raise ValueError("w must be a 2-D tensor with unit stride along K")
    dtype = {torch.bfloat16: 0, torch.float32: 1}.get(w.dtype)
    if dtype is None:
        raise ValueError("w must be bf16 or fp32")
    N, K = w.shape
    if imatrix is not None:
        _cuda(imatrix, "imatrix")
        if imatrix.dtype != torch.float32 or imatrix.numel() != K or not imatrix.is_contiguous():
            raise ValueError("imatrix must be a contiguous fp32 tensor of K values")
    out = out or alloc_q4_0(N, K, w.device, rotate, expanded)
    d = out.desc()
    ldw = w.stride(0) if N > 1 else K
    _check(load_library().h32_q4_0_pack_weights_imatrix(
        w.data_ptr(), dtype, N, K, ldw, int(rotate), imatrix.data_ptr() if imatrix is not None else None,
        ctypes.byref(d), _stream(stream)))
    out.rotated = bool(d.tag & TAG_ROTATED)
    return out


def q4_0_import(blocks: torch.Tensor, K: int, rotated: bool = True, out: Q4_0Weights | None = None,
                stream=None, expanded: bool = False) -> Q4_0Weights:
    """Import canonical 18-byte Q4_0 blocks (uint8 CUDA tensor, N * K/32 * 18 bytes) bit for bit."""
    _cuda(blocks, "blocks")
    if blocks.dtype != torch.uint8 or not blocks.is_contiguous():
        raise ValueError("blocks must be a contiguous uint8 tensor")
    if K <= 0 or K % 32 or blocks.numel() % (18 * (K // 32)):
        raise W4A4Error(1, "blocks size is not a multiple of a row of K/32 blocks")
    N = blocks.numel() // (18 * (K // 32))
    out = out or alloc_q4_0(N, K, blocks.device, rotated, expanded)
    d = out.desc()
    _check(load_library().q4_0_import(blocks.data_ptr(), N, K, int(rotated), ctypes.byref(d), _stream(stream)))
    out.rotated = bool(rotated)
    return out


def w4a4_rotate_quantize_act(x: torch.Tensor, rotate: bool = True, out: Act4 | None = None,
                             stream=None) -> Act4:
    """Rotate (H32) and int4-quantise fp32 activations x [M][K] (CUDA) per 32-block."""
    _cuda(x, "x")
    if x.dtype != torch.float32 or x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be a 2-D fp32 tensor with unit stride along K")
    M, K = x.shape
    out = out or alloc_act4(M, K, x.device, rotate)
    d = out.desc()
    ldx = x.stride(0) if M > 1 else K
    _check(load_library().w4a4_rotate_quantize_act(x.data_ptr(), M, K, ldx, int(rotate),
                                                    ctypes.byref(d), _stream(stream)))
    out.rotated = bool(rotate)
    return out


def w4a4_gemm_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load_library().w4a4_gemm_workspace_bytes(M, N, K))


_GEMM_WS: dict = {}


def gemm_workspace(M: int, N: int, K: int, device, stream=None, need: int | None = None) -> torch.Tensor | None:
    """A zero-initialised GEMM workspace kept per (device, stream), grown on demand.

    One per stream, because calls sharing a workspace must not overlap on the GPU.
    ``need`` overrides the size query (the exact path has its own).
    """
    if need is None:
        need = w4a4_gemm_workspace_bytes(M, N, K)
    if need == 0:
        return None
    key = (torch.device(device).index, _stream(stream))
    ws = _GEMM_WS.get(key)
    if ws is None or ws.numel() < need:
        ws = torch.zeros(need, dtype=torch.uint8, device=device)
        _GEMM_WS[key] = ws
    return ws


def w4a4_gemm(w: Q4_0Weights, a: Act4, y: torch.Tensor | None = None, ws: torch.Tensor | None | bool = True,
              stream=None) -> torch.Tensor:
    """Y[m][n] = sum_b d_w[n][b] d_a[m][b] P[m][n][b] (fp32 [M][N]).

    ws: True = the cached per-stream workspace (stream-K where it pays), a tensor
    = that workspace (zero before its first use), None/False = whole-tile schedule.
    """
    if y is None:
        y = torch.empty(a.rows, w.rows, dtype=torch.float32, device=w.codes.device)
    _cuda(y, "y")
    if y.dtype != torch.float32 or y.dim() != 2 or y.stride(1) != 1:
        raise ValueError("y must be a 2-D fp32 tensor with unit stride along N")
    ldy = y.stride(0) if y.shape[0] > 1 else max(w.rows, 1)
    if ws is True:
        ws = gemm_workspace(a.rows, w.rows, w.K, y.device, stream)
    elif ws is False:
        ws = None
    ws_ptr, ws_bytes = (ws.data_ptr(), ws.numel() * ws.element_size()) if ws is not None else (None, 0)
    _check(load_library().w4a4_gemm(ctypes.byref(w.desc()), ctypes.byref(a.desc()), y.data_ptr(), ldy, ws_ptr,
                                    ws_bytes, _stream(stream)))
    return y


def w4a4_gemm_small_m(w: Q4_0Weights, a: Act4, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """w4a4_gemm for 1 to 8 activation rows (a verification batch): the weight-streaming kernel,
    bit for bit the tensor-core kernel's whole-tile result."""
    if y is None:
        y = torch.empty(a.rows, w.rows, dtype=torch.float32, device=w.codes.device)
    _cuda(y, "y")
    if y.dtype != torch.float32 or y.dim() != 2 or y.stride(1) != 1:
        raise ValueError("y must be a 2-D fp32 tensor with unit stride along N")
    ldy = y.stride(0) if y.shape[0] > 1 else max(w.rows, 1)
    _check(load_library().w4a4_gemm_small_m(ctypes.byref(w.desc()), ctypes.byref(a.desc()), y.data_ptr(), ldy,
                                            _stream(stream)))
    return y


def w4a4_gemm_partials(w: Q4_0Weights, a: Act4, P: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Exact per-block integer partials P[m][n][b] (int32), from the tensor-core main loop."""
    if P is None:
        P = torch.empty(a.rows, w.rows, w.K // 32, dtype=torch.int32, device=w.codes.device)
    _cuda(P, "P")
    _check(load_library().w4a4_gemm_partials(ctypes.byref(w.desc()), ctypes.byref(a.desc()), P.data_ptr(),
                                             _stream(stream)))
    return P


def w4a4_gemm_id_workspace_bytes(M: int, top_k: int, E: int, K: int) -> int:
    return int(load_library().w4a4_gemm_id_workspace_bytes(M, top_k, E, K))


def w4a4_gemm_id(experts: Q4_0Weights, E: int, a: Act4, ids: torch.Tensor, top_k: int, act_per_slot: bool,
                 y: torch.Tensor | None = None, ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Expert-routed product: y [M][top_k][N], N = experts.rows // E."""
    _cuda(ids, "ids")
    if ids.dtype != torch.int32 or not ids.is_contiguous() or ids.dim() != 2 or ids.shape[1] != top_k:
        raise ValueError("ids must be a contiguous int32 [M][top_k] tensor")
    M = ids.shape[0]
    N = experts.rows // E
    if y is None:
        y = torch.empty(M, top_k, N, dtype=torch.float32, device=ids.device)
    need = w4a4_gemm_id_workspace_bytes(M, top_k, E, a.K)
    if ws is None:
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=ids.device)
    _check(load_library().w4a4_gemm_id(ctypes.byref(experts.desc()), E, N, ctypes.byref(a.desc()), ids.data_ptr(),
                                       M, top_k, int(act_per_slot), y.data_ptr(), ws.data_ptr(),
                                       ws.numel() * ws.element_size(), _stream(stream)))
    return y


#: bytes of the library's fixed routing scratch, per device
GEMM_ID_STATIC_SCRATCH_BYTES = 64 << 20


def w4a4_gemm_id_static(experts: Q4_0Weights, E: int, a: Act4, ids: torch.Tensor, top_k: int, act_per_slot: bool,
                        y: torch.Tensor, stream=None) -> torch.Tensor:
    """w4a4_gemm_id with the library's fixed routing scratch instead of a workspace.

    Nothing is allocated: the caller passes the output ``y`` [M][top_k][N].
    Calls that may overlap on the GPU share the scratch and race.
    """
    _cuda(ids, "ids")
    if ids.dtype != torch.int32 or not ids.is_contiguous() or ids.dim() != 2 or ids.shape[1] != top_k:
        raise ValueError("ids must be a contiguous int32 [M][top_k] tensor")
    _cuda(y, "y")
    if y.dtype != torch.float32 or not y.is_contiguous() or tuple(y.shape) != (ids.shape[0], top_k, experts.rows // E):
        raise ValueError("y must be a contiguous float32 [M][top_k][N] tensor")
    _check(load_library().w4a4_gemm_id_static(ctypes.byref(experts.desc()), E, experts.rows // E,
                                              ctypes.byref(a.desc()), ids.data_ptr(), ids.shape[0], top_k,
                                              int(act_per_slot), y.data_ptr(), _stream(stream)))
    return y


def w4a4_check(stream=None) -> None:
    """Synchronise and raise W4A4Error(W4A4_ERR_TIMEOUT) if a GEMM kernel gave up on a bounded wait.

    A kernel that gave up may leave stream-K arrival tickets standing in its
    workspace, and a later call on that workspace would then finish its cut
    tiles wrongly.  So on a timeout every cached per-stream workspace is dropped
    (the next call allocates a zeroed one); a workspace the caller passed in
    must be zeroed by the caller before it is used again.
    """
    status = load_library().w4a4_check(_stream(stream))
    if status == 8:  # W4A4_ERR_TIMEOUT
        _GEMM_WS.clear()
    _check(status)


def w4a4_debug_set_wait_limit(wait_ns: int = 0, producer_delay_ns: int = 0) -> None:
    """Test hook: the super-tile GEMM's pipeline-wait bound and a producer delay ((0, 0): defaults)."""
    load_library().w4a4_debug_set_wait_limit(int(wait_ns), int(producer_delay_ns))


def w4a4_gemm_id_status(ws: torch.Tensor, stream=None) -> None:
    """Synchronise and raise W4A4Error(W4A4_ERR_DEVICE_FLAG) if the last gemm_id on ws saw a bad id."""
    _check(load_library().w4a4_gemm_id_status(ws.data_ptr(), _stream(stream)))


# ---------------------------------------------------------------- the exact path (int8 activations)
@dataclass
class Act8:
    """int8 activations of the exact path: codes int8 [rows][K] (element order), scales fp32 [rows][K/32]."""
    codes: torch.Tensor
    scales_buf: torch.Tensor
    rows: int
    K: int
    rotated: bool

    @property
    def scales(self) -> torch.Tensor:
        n = self.rows * (self.K // 32)
        return self.scales_buf[: 4 * n].view(torch.float32).view(self.rows, self.K // 32)

    @property
    def tag(self) -> int:
        return TAG_ACT8 | (TAG_ROTATED if self.rotated else 0)

    def desc(self) -> _Act4Desc:
        return _Act4Desc(self.codes.data_ptr(), self.scales_buf.data_ptr(), self.rows, self.K, self.tag)


def alloc_act8(rows: int, K: int, device, rotated: bool = True) -> Act8:
    lib = load_library()
    if K <= 0 or K % 32:
        raise W4A4Error(1, f"K={K} must be a positive multiple of 32")
    nc, ns = lib.w4a4_act8_codes_bytes(rows, K), lib.w4a4_act8_scales_bytes(rows, K)
    codes = torch.empty(max(nc, 16), dtype=torch.int8, device=device)[:nc].view(rows, K)
    sbuf = torch.empty(max(ns, 16), dtype=torch.uint8, device=device)
    return Act8(codes, sbuf, rows, K, rotated)


def w4a8_rotate_quantize_act(x: torch.Tensor, rotate: bool = True, out: Act8 | None = None, stream=None) -> Act8:
    """Rotate (H32) and int8-quantise fp32 activations x [M][K] (CUDA) per 32-block (d_a = amax / 127)."""
    _cuda(x, "x")
    if x.dtype != torch.float32 or x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be a 2-D fp32 tensor with unit stride along K")
    M, K = x.shape
    out = out or alloc_act8(M, K, x.device, rotate)
    d = out.desc()
    ldx = x.stride(0) if M > 1 else K
    _check(load_library().w4a8_rotate_quantize_act(x.data_ptr(), M, K, ldx, int(rotate), ctypes.byref(d),
                                                    _stream(stream)))
    out.rotated = bool(rotate)
    return out


def w4a8_gemm_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load_library().w4a8_gemm_workspace_bytes(M, N, K))


def w4a8_gemm(w: Q4_0Weights, a: Act8, y: torch.Tensor | None = None, ws: torch.Tensor | None | bool = True,
              stream=None) -> torch.Tensor:
    """The exact path: Y[m][n] = sum_b d_w d_a P with int8 activations (fp32 [M][N]); ws as for w4a4_gemm."""
    if y is None:
        y = torch.empty(a.rows, w.rows, dtype=torch.float32, device=w.codes.device)
    _cuda(y, "y")
    if y.dtype != torch.float32 or y.dim() != 2 or y.stride(1) != 1:
        raise ValueError("y must be a 2-D fp32 tensor with unit stride along N")
    ldy = y.stride(0) if y.shape[0] > 1 else max(w.rows, 1)
    if ws is True:
        ws = gemm_workspace(a.rows, w.rows, w.K, y.device, stream, need=w4a8_gemm_workspace_bytes(a.rows, w.rows, w.K))
    elif ws is False:
        ws = None
    ws_ptr, ws_bytes = (ws.data_ptr(), ws.numel() * ws.element_size()) if ws is not None else (None, 0)
    _check(load_library().w4a8_gemm(ctypes.byref(w.desc()), ctypes.byref(a.desc()), y.data_ptr(), ldy, ws_ptr,
                                    ws_bytes, _stream(stream)))
    return y


def w4a8_gemm_partials(w: Q4_0Weights, a: Act8, P: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Exact per-block integer partials of the exact path, P[m][n][b] (int32)."""
    if P is None:
        P = torch.empty(a.rows, w.rows, w.K // 32, dtype=torch.int32, device=w.codes.device)
    _cuda(P, "P")
    _check(load_library().w4a8_gemm_partials(ctypes.byref(w.desc()), ctypes.byref(a.desc()), P.data_ptr(),
                                             _stream(stream)))
    return P


# ---------------------------------------------------------------- the rotate-only route (bf16 activations)
@dataclass
class Act16:
    """Rotated activations that were not quantised: bf16 values [rows][K] (element order)."""
    values: torch.Tensor
    rows: int
    K: int
    rotated: bool

    @property
    def tag(self) -> int:
        return TAG_ACT16 | (TAG_ROTATED if self.rotated else 0)

    def desc(self) -> _Act16Desc:
        return _Act16Desc(self.values.data_ptr(), self.rows, self.K, self.tag)


def alloc_act16(rows: int, K: int, device, rotated: bool = True) -> Act16:
    lib = load_library()
    if K <= 0 or K % 32:
        raise W4A4Error(1, f"K={K} must be a positive multiple of 32")
    nv = lib.w4a4_act16_values_bytes(rows, K)
    buf = torch.empty(max(nv, 16), dtype=torch.uint8, device=device)
    return Act16(buf[: 2 * rows * K].view(torch.bfloat16).view(rows, K), rows, K, rotated)


def w4a16_rotate_act(x: torch.Tensor, rotate: bool = True, out: Act16 | None = None, stream=None) -> Act16:
    """Rotate (H32) fp32 activations x [M][K] (CUDA) per 32-block and store them as bf16, not quantised."""
    _cuda(x, "x")
    if x.dtype != torch.float32 or x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be a 2-D fp32 tensor with unit stride along K")
    M, K = x.shape
    out = out or alloc_act16(M, K, x.device, rotate)
    d = out.desc()
    ldx = x.stride(0) if M > 1 else K
    _check(load_library().w4a16_rotate_act(x.data_ptr(), M, K, ldx, int(rotate), ctypes.byref(d), _stream(stream)))
    out.rotated = bool(rotate)
    return out


def w4a16_gemm_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load_library().w4a16_gemm_workspace_bytes(M, N, K))


def w4a16_gemm(w: Q4_0Weights, a: Act16, y: torch.Tensor | None = None, ws: torch.Tensor | None | bool = True,
               stream=None) -> torch.Tensor:
    """The rotate-only route: Y[m][n] = sum_b d_w sum_j y (q_w - 8) with bf16 activations (fp32 [M][N])."""
    if y is None:
        y = torch.empty(a.rows, w.rows, dtype=torch.float32, device=w.codes.device)
    _cuda(y, "y")
    if y.dtype != torch.float32 or y.dim() != 2 or y.stride(1) != 1:
        raise ValueError("y must be a 2-D fp32 tensor with unit stride along N")
    ldy = y.stride(0) if y.shape[0] > 1 else max(w.rows, 1)
    if ws is True:
        ws = gemm_workspace(a.rows, w.rows, w.K, y.device, stream, need=w4a16_gemm_workspace_bytes(a.rows, w.rows, w.K))
    elif ws is False:
        ws = None
    ws_ptr, ws_bytes = (ws.data_ptr(), ws.numel() * ws.element_size()) if ws is not None else (None, 0)
    _check(load_library().w4a16_gemm(ctypes.byref(w.desc()), ctypes.byref(a.desc()), y.data_ptr(), ldy, ws_ptr,
                                     ws_bytes, _stream(stream)))
    return y
