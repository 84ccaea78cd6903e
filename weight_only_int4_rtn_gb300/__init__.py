"""GB300 (sm_103a) weight-only INT4 round-to-nearest quantization and W4A16 GEMM.

A thin ctypes binding over the C ABI in ``include/w4a16.h`` (the in-tree
library ``libw4a16.so``).  Every function here only marshals arguments:
shapes, dtypes and devices are checked from metadata, device buffers come
from PyTorch, and each call is one launch of the library's CUDA kernels on
the current PyTorch stream.  There is no CPU path: a missing library or a
non-CUDA tensor raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libw4a16.so")
GROUP = 128

W4A16_OK = 0
W4A16_ERR_INVALID_ARG = 1
W4A16_ERR_UNSUPPORTED = 2
W4A16_ERR_ALIGNMENT = 3
W4A16_ERR_WORKSPACE = 4
W4A16_ERR_NO_VARIANT = 5
W4A16_ERR_CUDA = 6
W4A16_ERR_TIMEOUT = 7

# (name, restype, argtypes) of every symbol the C header declares.
_c_int64, _c_size, _vp = ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p
class GemmProblem(ctypes.Structure):
    """Mirror of w4a16_gemm_problem (include/w4a16.h)."""
    _fields_ = [("A", ctypes.c_void_p), ("packed", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("bias_or_null", ctypes.c_void_p), ("Y", ctypes.c_void_p),
                ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("epilogue", ctypes.c_int)]


EPILOGUE_NONE = 0
EPILOGUE_SWIGLU = 1


class QuantizeProblem(ctypes.Structure):
    """Mirror of w4a16_quantize_problem (include/w4a16.h)."""
    _fields_ = [("W_bf16", ctypes.c_void_p), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("packed_out", ctypes.c_void_p), ("scales_out", ctypes.c_void_p)]


MAX_GROUP = 8

SIGNATURES = [
    ("w4a16_status_string", ctypes.c_char_p, [ctypes.c_int]),
    ("w4a16_packed_bytes", _c_size, [_c_int64, _c_int64]),
    ("w4a16_scales_bytes", _c_size, [_c_int64, _c_int64, ctypes.c_int]),
    ("w4a16_quantize", ctypes.c_int, [_vp, _c_int64, _c_int64, ctypes.c_int, _vp, _vp, _vp]),
    ("w4a16_quantize_sr", ctypes.c_int,
     [_vp, _c_int64, _c_int64, ctypes.c_int, ctypes.c_uint64, _vp, _vp, _vp]),
    ("w4a16_tune_grouped", ctypes.c_int,
     [ctypes.POINTER(GemmProblem), ctypes.c_int, ctypes.c_int, _vp, ctypes.POINTER(ctypes.c_int)]),
    ("w4a16_set_grouped_variant", ctypes.c_int, [ctypes.POINTER(GemmProblem), ctypes.c_int, ctypes.c_int]),
    ("w8a16_packed_bytes", _c_size, [_c_int64, _c_int64]),
    ("w8a16_quantize", ctypes.c_int, [_vp, _c_int64, _c_int64, ctypes.c_int, _vp, _vp, _vp]),
    ("w8a16_gemm_workspace_bytes", _c_size, [_c_int64, _c_int64, _c_int64]),
    ("w8a16_gemm", ctypes.c_int,
     [_vp, _c_int64, _c_int64, _c_int64, _vp, _vp, ctypes.c_int, _vp, _vp, _vp, _c_size, _vp]),
    ("w8a16_variant_count", ctypes.c_int, []),
    ("w8a16_variant_name", ctypes.c_char_p, [ctypes.c_int]),
    ("w8a16_variant_eligible", ctypes.c_int, [ctypes.c_int, _c_int64, _c_int64, _c_int64]),
    ("w8a16_variant_workspace_bytes", _c_size, [ctypes.c_int, _c_int64, _c_int64, _c_int64]),
    ("w8a16_select_variant", ctypes.c_int, [_c_int64, _c_int64, _c_int64]),
    ("w8a16_gemm_variant", ctypes.c_int,
     [ctypes.c_int, _vp, _c_int64, _c_int64, _c_int64, _vp, _vp, ctypes.c_int, _vp, _vp, _vp,
      _c_size, _vp]),
    ("fp4a16_packed_bytes", _c_size, [_c_int64, _c_int64]),
    ("fp4a16_scales_bytes", _c_size, [ctypes.c_int, _c_int64, _c_int64]),
    ("fp4a16_quantize", ctypes.c_int, [ctypes.c_int, _vp, _c_int64, _c_int64, _vp, _vp, _vp, _vp]),
    ("fp4a16_gemm_workspace_bytes", _c_size, [ctypes.c_int, _c_int64, _c_int64, _c_int64]),
    ("fp4a16_gemm", ctypes.c_int,
     [ctypes.c_int, _vp, _c_int64, _c_int64, _c_int64, _vp, _vp, _vp, _vp, _vp, _vp, _c_size, _vp]),
    ("fp4a16_variant_count", ctypes.c_int, []),
    ("fp4a16_variant_name", ctypes.c_char_p, [ctypes.c_int]),
    ("fp4a16_variant_eligible", ctypes.c_int, [ctypes.c_int, _c_int64, _c_int64, _c_int64]),
    ("fp4a16_variant_workspace_bytes", _c_size, [ctypes.c_int, _c_int64, _c_int64, _c_int64]),
    ("fp4a16_select_variant", ctypes.c_int, [_c_int64, _c_int64, _c_int64]),
    ("fp4a16_gemm_variant", ctypes.c_int,
     [ctypes.c_int, ctypes.c_int, _vp, _c_int64, _c_int64, _c_int64, _vp, _vp, _vp, _vp, _vp, _vp,
      _c_size, _vp]),
    ("w4a16_gemm_workspace_bytes", _c_size, [_c_int64, _c_int64, _c_int64]),
    ("w4a16_gemm_workspace_bytes_max", _c_size, [_c_int64, _c_int64, _c_int64]),
    ("w4a16_workspace_init", ctypes.c_int, [_vp, _c_size, _vp]),
    ("w4a16_gemm", ctypes.c_int,
     [_vp, _c_int64, _c_int64, _c_int64, _vp, _vp, ctypes.c_int, _vp, _vp, _vp, _c_size, _vp]),
    ("w4a16_gemm_f16", ctypes.c_int,
     [_vp, _c_int64, _c_int64, _c_int64, _vp, _vp, ctypes.c_int, _vp, _vp, _vp, _c_size, _vp]),
    ("w4a16_quantize_grouped", ctypes.c_int,
     [ctypes.POINTER(QuantizeProblem), ctypes.c_int, ctypes.c_int, _vp]),
    ("w4a16_gemm_grouped_workspace_bytes", _c_size,
     [ctypes.POINTER(GemmProblem), ctypes.c_int, ctypes.c_int]),
    ("w4a16_gemm_grouped", ctypes.c_int,
     [ctypes.POINTER(GemmProblem), ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp,
      _c_size, _vp]),
    ("w4a16_variant_count", ctypes.c_int, []),
    ("w4a16_variant_name", ctypes.c_char_p, [ctypes.c_int]),
    ("w4a16_variant_eligible", ctypes.c_int, [ctypes.c_int, _c_int64, _c_int64, _c_int64]),
    ("w4a16_variant_workspace_bytes", _c_size, [ctypes.c_int, _c_int64, _c_int64, _c_int64]),
    ("w4a16_select_variant", ctypes.c_int, [_c_int64, _c_int64, _c_int64]),
    ("w4a16_variant_schedule", ctypes.c_int,
     [ctypes.c_int, _c_int64, _c_int64, _c_int64, ctypes.c_int, ctypes.POINTER(ctypes.c_int)]),
    ("w4a16_gemm_variant", ctypes.c_int,
     [ctypes.c_int, _vp, _c_int64, _c_int64, _c_int64, _vp, _vp, ctypes.c_int, _vp, _vp, _vp,
      _c_size, _vp]),
    ("w4a16_gemm_swiglu", ctypes.c_int,
     [_vp, _c_int64, _c_int64, _c_int64, _vp, _vp, ctypes.c_int, _vp, _vp, _vp, _c_size, _vp]),
    ("w4a16_gemm_swiglu_workspace_bytes", _c_size, [_c_int64, _c_int64, _c_int64]),
    ("w4a16_gemm_swiglu_variant", ctypes.c_int,
     [ctypes.c_int, _vp, _c_int64, _c_int64, _c_int64, _vp, _vp, ctypes.c_int, _vp, _vp, _vp,
      _c_size, _vp]),
    ("w4a16_gemm_variant_f16", ctypes.c_int,
     [ctypes.c_int, _vp, _c_int64, _c_int64, _c_int64, _vp, _vp, ctypes.c_int, _vp, _vp, _vp,
      _c_size, _vp]),
    ("w4a16_tune", ctypes.c_int, [_c_int64, _c_int64, _c_int64, _vp, ctypes.POINTER(ctypes.c_int)]),
    ("w4a16_table_set", ctypes.c_int, [_c_int64, _c_int64, _c_int64, ctypes.c_int]),
    ("w4a16_tune_swiglu", ctypes.c_int, [_c_int64, _c_int64, _c_int64, _vp, ctypes.POINTER(ctypes.c_int)]),
    ("w8a16_tune", ctypes.c_int, [_c_int64, _c_int64, _c_int64, _vp, ctypes.POINTER(ctypes.c_int)]),
    ("fp4a16_tune", ctypes.c_int,
     [ctypes.c_int, _c_int64, _c_int64, _c_int64, _vp, ctypes.POINTER(ctypes.c_int)]),
    ("w4a16_swiglu_table_set", ctypes.c_int, [_c_int64, _c_int64, _c_int64, ctypes.c_int]),
    ("w8a16_table_set", ctypes.c_int, [_c_int64, _c_int64, _c_int64, ctypes.c_int]),
    ("fp4a16_table_set", ctypes.c_int, [_c_int64, _c_int64, _c_int64, ctypes.c_int]),
    ("w4a16_table_clear", None, []),
    ("w4a16_table_save", ctypes.c_int, [ctypes.c_char_p]),
    ("w4a16_table_load", ctypes.c_int, [ctypes.c_char_p]),
    ("w4a16_get_device_error", ctypes.c_int, [_vp]),
    ("w4a16_set_wait_timeout_ns", None, [ctypes.c_uint64]),
    ("w4a16_set_weights_static", None, [ctypes.c_int]),
    ("w4a16_weights_static", ctypes.c_int, []),
    ("w4a16_selftest_wait_timeout", ctypes.c_int, [ctypes.c_uint64, _vp]),
    ("w4a16_launch_count", ctypes.c_uint64, []),
    ("w4a16_last_error_detail", ctypes.c_char_p, []),
    ("w4a16_packed_rowmajor_bytes", _c_size, [_c_int64, _c_int64]),
    ("w4a16_repack_rowmajor", ctypes.c_int, [_vp, _c_int64, _c_int64, _vp, _vp]),
    ("w4a16_selftest_quotient", ctypes.c_int, [ctypes.c_int, _vp, _vp]),
    ("w4a16_gemm_noalloc", ctypes.c_int,
     [_vp, _c_int64, _c_int64, _c_int64, _vp, _vp, ctypes.c_int, _vp, _vp, _vp]),
]

_lib = None
_lib_lock = threading.Lock()


class W4A16Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        with _lib_lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"{LIB_PATH} is not built; run `python -c \"import __graft_entry__ as g; g.build()\"`")
                handle = ctypes.CDLL(LIB_PATH)
                for name, res, args in SIGNATURES:
                    fn = getattr(handle, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = handle
    return _lib


def status_string(status: int) -> str:
    try:
        return lib().w4a16_status_string(status).decode()
    except Exception:   # library missing: still give a readable message
        return f"status {status}"


def _check(status: int, what: str) -> None:
    if status != W4A16_OK:
        if status == W4A16_ERR_CUDA:
            what = f"{what} [{lib().w4a16_last_error_detail().decode()}]"
        raise W4A16Error(status, what)


def _stream_handle(device: torch.device, stream=None) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream)


def _require_cuda(t: torch.Tensor, name: str, dtype: torch.dtype) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (no CPU path), got {t.device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


# ------------------------------------------------------------------ sizes
def w4a16_packed_bytes(N: int, K: int) -> int:
    return lib().w4a16_packed_bytes(N, K)


def w4a16_scales_bytes(N: int, K: int, group: int = GROUP) -> int:
    return lib().w4a16_scales_bytes(N, K, group)


def w4a16_gemm_workspace_bytes(M: int, N: int, K: int) -> int:
    return lib().w4a16_gemm_workspace_bytes(M, N, K)


def w4a16_gemm_workspace_bytes_max(M: int, N: int, K: int) -> int:
    return lib().w4a16_gemm_workspace_bytes_max(M, N, K)


# --------------------------------------------------------------- quantize
def w4a16_quantize(W: torch.Tensor, group: int = GROUP, packed: torch.Tensor | None = None,
                   scales: torch.Tensor | None = None, stream=None, seed: int | None = None):
    """Quantize ``W[N, K]`` (bf16, CUDA).  Returns ``(packed, scales)``:
    ``packed`` is the 1-D uint8 tiled code storage of w4a16_packed_bytes(N, K)
    bytes, ``scales`` fp16 ``[K/128, N]``; outputs are allocated when not
    given.  Round to nearest (w4a16_quantize), or, with an unsigned 64-bit
    ``seed``, seeded stochastic rounding with the same scales
    (w4a16_quantize_sr)."""
    if seed is not None and not 0 <= int(seed) < (1 << 64):
        raise ValueError("seed must be an unsigned 64-bit integer")
    _require_cuda(W, "W", torch.bfloat16)
    if W.dim() != 2:
        raise ValueError("W must be [N, K]")
    N, K = W.shape
    nbytes = lib().w4a16_packed_bytes(N, K)
    if packed is None:
        packed = torch.empty(nbytes, dtype=torch.uint8, device=W.device)
    if scales is None:
        scales = torch.empty((max(K // group, 0), N), dtype=torch.float16, device=W.device)
    _require_cuda(packed, "packed", torch.uint8)
    _require_cuda(scales, "scales", torch.float16)
    if packed.numel() != nbytes or scales.numel() * group != N * K:
        raise ValueError("output buffers have the wrong size")
    if seed is None:
        st = lib().w4a16_quantize(W.data_ptr(), N, K, group, packed.data_ptr(), scales.data_ptr(),
                                  _stream_handle(W.device, stream))
        _check(st, "w4a16_quantize")
    else:
        st = lib().w4a16_quantize_sr(W.data_ptr(), N, K, group, int(seed), packed.data_ptr(),
                                     scales.data_ptr(), _stream_handle(W.device, stream))
        _check(st, "w4a16_quantize_sr")
    return packed, scales


def w4a16_repack_rowmajor(packed_rowmajor: torch.Tensor, N: int, K: int,
                          packed: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Row-major packed codes (uint8 ``[N, K/2]`` or 1-D with N*K/2 bytes;
    byte j of row n: code 2j low nibble, 2j+1 high nibble) to the tiled
    storage the GEMM reads (w4a16_repack_rowmajor).  Returns ``packed`` (1-D
    uint8, w4a16_packed_bytes(N, K) bytes), allocated when not given."""
    _require_cuda(packed_rowmajor, "packed_rowmajor", torch.uint8)
    if packed_rowmajor.numel() != lib().w4a16_packed_rowmajor_bytes(N, K):
        raise ValueError("packed_rowmajor must hold N * K / 2 bytes")
    nbytes = lib().w4a16_packed_bytes(N, K)
    if packed is None:
        packed = torch.empty(nbytes, dtype=torch.uint8, device=packed_rowmajor.device)
    _require_cuda(packed, "packed", torch.uint8)
    if packed.numel() != nbytes:
        raise ValueError("packed must hold w4a16_packed_bytes(N, K) bytes")
    _check(lib().w4a16_repack_rowmajor(packed_rowmajor.data_ptr(), N, K, packed.data_ptr(),
                                       _stream_handle(packed.device, stream)),
           "w4a16_repack_rowmajor")
    return packed


def selftest_quotient(mode: int, device=None) -> dict:
    """Run w4a16_selftest_quotient (0: INT4 scales, 1: INT8 scales, 2: NVFP4
    steps) on ``device`` and return its counts: pairs checked, codes that
    differ, quotients that differ in the normal range and anywhere
    (synchronises)."""
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
    counts = torch.zeros(4, dtype=torch.int64, device=dev)
    _check(lib().w4a16_selftest_quotient(int(mode), counts.data_ptr(), _stream_handle(dev)),
           "w4a16_selftest_quotient")
    c = [int(v) for v in counts.cpu().tolist()]
    return dict(checked=c[0], code_mismatches=c[1], quotient_mismatches_normal=c[2],
                quotient_mismatches=c[3])


# ------------------------------------------------------------------- GEMM
class Workspace:
    """A zero-initialised device workspace that grows on demand.  One per
    (device, stream): GEMMs that may run concurrently need separate ones."""

    def __init__(self):
        self._buf: dict = {}

    def get(self, device: torch.device, stream_handle: int, nbytes: int) -> torch.Tensor | None:
        if nbytes == 0:
            return None
        key = (device.index, stream_handle)
        buf = self._buf.get(key)
        if buf is None or buf.numel() < nbytes:
            buf = torch.zeros(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
            self._buf[key] = buf
        return buf


_default_ws = Workspace()


def w4a16_gemm(A: torch.Tensor, packed: torch.Tensor, scales: torch.Tensor,
               bias: torch.Tensor | None = None, Y: torch.Tensor | None = None,
               workspace: torch.Tensor | None = None, group: int = GROUP, stream=None,
               variant: int | None = None) -> torch.Tensor:
    """``Y[M, N] = A[M, K] @ dequant(packed, scales)^T + bias`` on the GPU, in
    the activation type of ``A`` (bf16: w4a16_gemm; fp16: w4a16_gemm_f16);
    ``bias`` and ``Y`` take the same type.

    ``variant`` forces one entry of the kernel catalogue (tests, tuning);
    otherwise the library's per-shape table chooses."""
    if not isinstance(A, torch.Tensor):
        raise TypeError("A must be a torch.Tensor")
    act = A.dtype if A.dtype in (torch.bfloat16, torch.float16) else torch.bfloat16
    _require_cuda(A, "A", act)
    _require_cuda(packed, "packed", torch.uint8)
    _require_cuda(scales, "scales", torch.float16)
    if A.dim() != 2 or scales.dim() != 2:
        raise ValueError("A and scales must be 2-D")
    M, K = A.shape
    N = scales.shape[1]
    if scales.shape[0] * group != K:
        raise ValueError("scales must be [K/128, N]")
    if packed.numel() != lib().w4a16_packed_bytes(N, K):
        raise ValueError("packed must hold w4a16_packed_bytes(N, K) bytes of tiled codes")
    if bias is not None:
        _require_cuda(bias, "bias", act)
        if bias.numel() != N:
            raise ValueError("bias must have N elements")
    if Y is None:
        Y = torch.empty((M, N), dtype=act, device=A.device)
    _require_cuda(Y, "Y", act)
    if Y.shape != (M, N):
        raise ValueError("Y must be [M, N]")
    sh = _stream_handle(A.device, stream)
    L = lib()
    need = (L.w4a16_gemm_workspace_bytes(M, N, K) if variant is None
            else L.w4a16_variant_workspace_bytes(variant, M, N, K))
    if workspace is None:
        workspace = _default_ws.get(A.device, sh, need)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    bias_ptr = bias.data_ptr() if bias is not None else None
    f16 = act == torch.float16
    if variant is None:
        fn = L.w4a16_gemm_f16 if f16 else L.w4a16_gemm
        st = fn(A.data_ptr(), M, N, K, packed.data_ptr(), scales.data_ptr(), group,
                bias_ptr, Y.data_ptr(), ws_ptr, ws_bytes, sh)
    else:
        fn = L.w4a16_gemm_variant_f16 if f16 else L.w4a16_gemm_variant
        st = fn(variant, A.data_ptr(), M, N, K, packed.data_ptr(), scales.data_ptr(), group,
                bias_ptr, Y.data_ptr(), ws_ptr, ws_bytes, sh)
    _check(st, "w4a16_gemm_f16" if f16 else "w4a16_gemm")
    return Y


def w4a16_gemm_swiglu(A: torch.Tensor, packed: torch.Tensor, scales: torch.Tensor,
                      bias: torch.Tensor | None = None, Y: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None, group: int = GROUP, stream=None,
                      variant: int | None = None) -> torch.Tensor:
    """``Y[M, N/2] = silu(y[:, 1::2]) * y[:, 0::2]`` with ``y = A @
    dequant(packed, scales)^T + bias`` in fp32 (bf16 A, bias and Y): the
    weight's rows interleave up (even rows) and gate (odd rows).  ``variant``
    forces one tcgen05 entry of the catalogue."""
    _require_cuda(A, "A", torch.bfloat16)
    _require_cuda(packed, "packed", torch.uint8)
    _require_cuda(scales, "scales", torch.float16)
    if A.dim() != 2 or scales.dim() != 2:
        raise ValueError("A and scales must be 2-D")
    M, K = A.shape
    N = scales.shape[1]
    if scales.shape[0] * group != K:
        raise ValueError("scales must be [K/128, N]")
    if N % 2 != 0:
        raise ValueError("N must be even (interleaved up and gate rows)")
    if packed.numel() != lib().w4a16_packed_bytes(N, K):
        raise ValueError("packed must hold w4a16_packed_bytes(N, K) bytes of tiled codes")
    if bias is not None:
        _require_cuda(bias, "bias", torch.bfloat16)
        if bias.numel() != N:
            raise ValueError("bias must have N elements")
    if Y is None:
        Y = torch.empty((M, N // 2), dtype=torch.bfloat16, device=A.device)
    _require_cuda(Y, "Y", torch.bfloat16)
    if Y.shape != (M, N // 2):
        raise ValueError("Y must be [M, N/2]")
    sh = _stream_handle(A.device, stream)
    L = lib()
    need = (L.w4a16_gemm_swiglu_workspace_bytes(M, N, K) if variant is None
            else L.w4a16_variant_workspace_bytes(variant, M, N, K))
    if workspace is None:
        workspace = _default_ws.get(A.device, sh, need)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    bias_ptr = bias.data_ptr() if bias is not None else None
    if variant is None:
        st = L.w4a16_gemm_swiglu(A.data_ptr(), M, N, K, packed.data_ptr(), scales.data_ptr(),
                                 group, bias_ptr, Y.data_ptr(), ws_ptr, ws_bytes, sh)
    else:
        st = L.w4a16_gemm_swiglu_variant(variant, A.data_ptr(), M, N, K, packed.data_ptr(),
                                         scales.data_ptr(), group, bias_ptr, Y.data_ptr(), ws_ptr,
                                         ws_bytes, sh)
    _check(st, "w4a16_gemm_swiglu")
    return Y


# ------------------------------------------------------------ INT8 (W8A16)
def w8a16_quantize(W: torch.Tensor, group: int = GROUP, packed: torch.Tensor | None = None,
                   scales: torch.Tensor | None = None, stream=None):
    """RTN INT8 quantize ``W[N, K]`` (bf16, CUDA).  Returns ``(packed,
    scales)``: 1-D uint8 tiled codes of w8a16_packed_bytes(N, K) bytes and fp16
    scales ``[K/128, N]``."""
    _require_cuda(W, "W", torch.bfloat16)
    if W.dim() != 2:
        raise ValueError("W must be [N, K]")
    N, K = W.shape
    nbytes = lib().w8a16_packed_bytes(N, K)
    if packed is None:
        packed = torch.empty(nbytes, dtype=torch.uint8, device=W.device)
    if scales is None:
        scales = torch.empty((max(K // group, 0), N), dtype=torch.float16, device=W.device)
    _require_cuda(packed, "packed", torch.uint8)
    _require_cuda(scales, "scales", torch.float16)
    if packed.numel() != nbytes or scales.numel() * group != N * K:
        raise ValueError("output buffers have the wrong size")
    _check(lib().w8a16_quantize(W.data_ptr(), N, K, group, packed.data_ptr(), scales.data_ptr(),
                                _stream_handle(W.device, stream)), "w8a16_quantize")
    return packed, scales


def w8a16_gemm(A: torch.Tensor, packed: torch.Tensor, scales: torch.Tensor,
               bias: torch.Tensor | None = None, Y: torch.Tensor | None = None,
               workspace: torch.Tensor | None = None, group: int = GROUP, stream=None,
               variant: int | None = None) -> torch.Tensor:
    """``Y[M, N] = A[M, K] @ dequant8(packed, scales)^T + bias`` (bf16) on
    the GPU; ``variant`` forces one entry of the INT8 catalogue."""
    _require_cuda(A, "A", torch.bfloat16)
    _require_cuda(packed, "packed", torch.uint8)
    _require_cuda(scales, "scales", torch.float16)
    if A.dim() != 2 or scales.dim() != 2:
        raise ValueError("A and scales must be 2-D")
    M, K = A.shape
    N = scales.shape[1]
    if scales.shape[0] * group != K:
        raise ValueError("scales must be [K/128, N]")
    if packed.numel() != lib().w8a16_packed_bytes(N, K):
        raise ValueError("packed must hold w8a16_packed_bytes(N, K) bytes of tiled codes")
    if bias is not None:
        _require_cuda(bias, "bias", torch.bfloat16)
        if bias.numel() != N:
            raise ValueError("bias must have N elements")
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _require_cuda(Y, "Y", torch.bfloat16)
    if Y.shape != (M, N):
        raise ValueError("Y must be [M, N]")
    sh = _stream_handle(A.device, stream)
    L = lib()
    need = (L.w8a16_gemm_workspace_bytes(M, N, K) if variant is None
            else L.w8a16_variant_workspace_bytes(variant, M, N, K))
    if workspace is None:
        workspace = _default_ws.get(A.device, sh, need)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    bias_ptr = bias.data_ptr() if bias is not None else None
    if variant is None:
        st = L.w8a16_gemm(A.data_ptr(), M, N, K, packed.data_ptr(), scales.data_ptr(), group,
                          bias_ptr, Y.data_ptr(), ws_ptr, ws_bytes, sh)
    else:
        st = L.w8a16_gemm_variant(variant, A.data_ptr(), M, N, K, packed.data_ptr(),
                                  scales.data_ptr(), group, bias_ptr, Y.data_ptr(), ws_ptr,
                                  ws_bytes, sh)
    _check(st, "w8a16_gemm")
    return Y


# ----------------------------------------------------------------- groups
# ------------------------------------------------- FP4 (MXFP4, NVFP4)
FP4_FORMATS = {"mxfp4": 1, "nvfp4": 2}


def _fp4_format(fmt) -> int:
    if isinstance(fmt, str):
        if fmt not in FP4_FORMATS:
            raise ValueError(f"unknown FP4 format {fmt!r}: one of {sorted(FP4_FORMATS)}")
        return FP4_FORMATS[fmt]
    if fmt not in FP4_FORMATS.values():
        raise ValueError(f"unknown FP4 format {fmt!r}")
    return int(fmt)


def fp4a16_quantize(W: torch.Tensor, fmt="mxfp4", packed: torch.Tensor | None = None,
                    scales: torch.Tensor | None = None, tensor_scale: torch.Tensor | None = None,
                    stream=None):
    """FP4 quantize ``W[N, K]`` (bf16, CUDA) as ``fmt`` ("mxfp4" or
    "nvfp4").  Returns ``(packed, scales, tensor_scale)``: 1-D uint8 tiled
    E2M1 codes (fp4a16_packed_bytes), uint8 scale codes ``[K/32, N]`` (E8M0)
    or ``[K/16, N]`` (E4M3), and for NVFP4 a float32 pair ``(g, amax)`` on the
    device (None for MXFP4)."""
    f = _fp4_format(fmt)
    _require_cuda(W, "W", torch.bfloat16)
    if W.dim() != 2:
        raise ValueError("W must be [N, K]")
    N, K = W.shape
    L = lib()
    nbytes = L.fp4a16_packed_bytes(N, K)
    blk = 32 if f == 1 else 16
    if packed is None:
        packed = torch.empty(nbytes, dtype=torch.uint8, device=W.device)
    if scales is None:
        scales = torch.empty((max(K // blk, 0), N), dtype=torch.uint8, device=W.device)
    if f == 2 and tensor_scale is None:
        tensor_scale = torch.empty(2, dtype=torch.float32, device=W.device)
    _require_cuda(packed, "packed", torch.uint8)
    _require_cuda(scales, "scales", torch.uint8)
    if f == 2:
        _require_cuda(tensor_scale, "tensor_scale", torch.float32)
        if tensor_scale.numel() != 2:
            raise ValueError("tensor_scale must hold 2 floats")
    if packed.numel() != nbytes or scales.numel() != L.fp4a16_scales_bytes(f, N, K):
        raise ValueError("output buffers have the wrong size")
    ts_ptr = tensor_scale.data_ptr() if f == 2 else None
    _check(L.fp4a16_quantize(f, W.data_ptr(), N, K, packed.data_ptr(), scales.data_ptr(), ts_ptr,
                             _stream_handle(W.device, stream)), "fp4a16_quantize")
    return packed, scales, (tensor_scale if f == 2 else None)


def fp4a16_gemm(A: torch.Tensor, packed: torch.Tensor, scales: torch.Tensor, fmt="mxfp4",
                tensor_scale: torch.Tensor | None = None, bias: torch.Tensor | None = None,
                Y: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                stream=None, variant: int | None = None) -> torch.Tensor:
    """``Y[M, N] = g * (A[M, K] @ D^T) + bias`` (bf16) on the GPU, D the
    dequantized FP4 weight (E2M1 code times its block scale), g NVFP4's tensor
    scale (``tensor_scale[0]``); ``variant`` forces one entry of the FP4
    catalogue."""
    f = _fp4_format(fmt)
    _require_cuda(A, "A", torch.bfloat16)
    _require_cuda(packed, "packed", torch.uint8)
    _require_cuda(scales, "scales", torch.uint8)
    if A.dim() != 2 or scales.dim() != 2:
        raise ValueError("A and scales must be 2-D")
    M, K = A.shape
    N = scales.shape[1]
    if scales.shape[0] * (32 if f == 1 else 16) != K:
        raise ValueError("scales must be [K/32, N] (mxfp4) or [K/16, N] (nvfp4)")
    L = lib()
    if packed.numel() != L.fp4a16_packed_bytes(N, K):
        raise ValueError("packed must hold fp4a16_packed_bytes(N, K) bytes of tiled codes")
    if f == 2:
        if tensor_scale is None:
            raise ValueError("nvfp4 needs the tensor scale written by fp4a16_quantize")
        _require_cuda(tensor_scale, "tensor_scale", torch.float32)
    if bias is not None:
        _require_cuda(bias, "bias", torch.bfloat16)
        if bias.numel() != N:
            raise ValueError("bias must have N elements")
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _require_cuda(Y, "Y", torch.bfloat16)
    if Y.shape != (M, N):
        raise ValueError("Y must be [M, N]")
    sh = _stream_handle(A.device, stream)
    need = (L.fp4a16_gemm_workspace_bytes(f, M, N, K) if variant is None
            else L.fp4a16_variant_workspace_bytes(variant, M, N, K))
    if workspace is None:
        workspace = _default_ws.get(A.device, sh, need)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    bias_ptr = bias.data_ptr() if bias is not None else None
    ts_ptr = tensor_scale.data_ptr() if f == 2 else None
    if variant is None:
        st = L.fp4a16_gemm(f, A.data_ptr(), M, N, K, packed.data_ptr(), scales.data_ptr(), ts_ptr,
                           bias_ptr, Y.data_ptr(), ws_ptr, ws_bytes, sh)
    else:
        st = L.fp4a16_gemm_variant(variant, f, A.data_ptr(), M, N, K, packed.data_ptr(),
                                   scales.data_ptr(), ts_ptr, bias_ptr, Y.data_ptr(), ws_ptr,
                                   ws_bytes, sh)
    _check(st, "fp4a16_gemm")
    return Y


def fp4a16_variant_count() -> int:
    return lib().fp4a16_variant_count()


def fp4a16_variant_name(variant: int) -> str | None:
    n = lib().fp4a16_variant_name(variant)
    return n.decode() if n is not None else None


def fp4a16_variant_eligible(variant: int, M: int, N: int, K: int) -> bool:
    return bool(lib().fp4a16_variant_eligible(variant, M, N, K))


def fp4a16_select_variant(M: int, N: int, K: int) -> int:
    return lib().fp4a16_select_variant(M, N, K)


def w4a16_quantize_grouped(weights, outs=None, stream=None):
    """RTN-quantize several bf16 weights in one launch.  Returns a list of
    ``(packed, scales)`` as ``w4a16_quantize`` would (``outs`` may supply
    those buffers)."""
    if not 1 <= len(weights) <= MAX_GROUP:
        raise ValueError(f"1 .. {MAX_GROUP} weights")
    given = outs
    outs, probs = [], (QuantizeProblem * len(weights))()
    for i, W in enumerate(weights):
        _require_cuda(W, "W", torch.bfloat16)
        N, K = W.shape
        if given is not None:
            packed, scales = given[i]
            _require_cuda(packed, "packed", torch.uint8)
            _require_cuda(scales, "scales", torch.float16)
            if packed.numel() != lib().w4a16_packed_bytes(N, K) or scales.shape != (K // GROUP, N):
                raise ValueError("packed / scales of the wrong size")
        else:
            packed = torch.empty(lib().w4a16_packed_bytes(N, K), dtype=torch.uint8, device=W.device)
            scales = torch.empty((K // GROUP, N), dtype=torch.float16, device=W.device)
        probs[i] = QuantizeProblem(W.data_ptr(), N, K, packed.data_ptr(), scales.data_ptr())
        outs.append((packed, scales))
    _check(lib().w4a16_quantize_grouped(probs, len(weights), GROUP,
                                        _stream_handle(weights[0].device, stream)),
           "w4a16_quantize_grouped")
    return outs


def _gemm_problems(As, packeds, scales_list, biases, Ys, epilogues=None):
    n = len(As)
    if not 1 <= n <= MAX_GROUP or not (len(packeds) == len(scales_list) == n):
        raise ValueError(f"1 .. {MAX_GROUP} problems with matching argument lists")
    act = As[0].dtype if As[0].dtype in (torch.bfloat16, torch.float16) else torch.bfloat16
    biases = biases if biases is not None else [None] * n
    Ys = Ys if Ys is not None else [None] * n
    epilogues = epilogues if epilogues is not None else [EPILOGUE_NONE] * n
    probs, outs = (GemmProblem * n)(), []
    for i in range(n):
        A, packed, scales, bias, Y = As[i], packeds[i], scales_list[i], biases[i], Ys[i]
        epi = int(epilogues[i])
        _require_cuda(A, "A", act)
        _require_cuda(packed, "packed", torch.uint8)
        _require_cuda(scales, "scales", torch.float16)
        M, K = A.shape
        N = scales.shape[1]
        if scales.shape[0] * GROUP != K:
            raise ValueError("scales must be [K/128, N]")
        if packed.numel() != lib().w4a16_packed_bytes(N, K):
            raise ValueError("packed must hold w4a16_packed_bytes(N, K) bytes of tiled codes")
        if bias is not None:
            _require_cuda(bias, "bias", act)
        ncols = N // 2 if epi == EPILOGUE_SWIGLU else N
        if Y is None:
            Y = torch.empty((M, ncols), dtype=act, device=A.device)
        _require_cuda(Y, "Y", act)
        if Y.shape != (M, ncols):
            raise ValueError(f"Y of problem {i} must be [{M}, {ncols}]")
        probs[i] = GemmProblem(A.data_ptr(), packed.data_ptr(), scales.data_ptr(),
                               bias.data_ptr() if bias is not None else None, Y.data_ptr(), M, N, K,
                               epi)
        outs.append(Y)
    return probs, outs, act


def w4a16_tune_grouped(shapes, act=torch.bfloat16, stream=None, device=None) -> int:
    """Choose the grouped-GEMM plan for these ``(M, N, K)`` (or ``(M, N, K,
    epilogue)``) shapes by measurement and memoize it (later
    ``w4a16_gemm_grouped`` calls of the same shapes use it).  Returns the
    chosen variant id."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    # only the shapes are read; the pointers must still be 16-byte aligned
    # and non-null for the argument checks
    probs, dummy = _shape_problems(shapes, dev)
    n = len(shapes)
    out = ctypes.c_int(-1)
    _check(lib().w4a16_tune_grouped(probs, n, 1 if act == torch.float16 else 0,
                                    _stream_handle(dev, stream), ctypes.byref(out)),
           "w4a16_tune_grouped")
    return out.value


def _shape_problems(shapes, device):
    n = len(shapes)
    if not 1 <= n <= MAX_GROUP:
        raise ValueError(f"1 .. {MAX_GROUP} shapes")
    probs = (GemmProblem * n)()
    dummy = torch.empty(256, dtype=torch.uint8, device=device)
    for i, shp in enumerate(shapes):
        M, N, K = shp[:3]
        epi = shp[3] if len(shp) > 3 else EPILOGUE_NONE
        probs[i] = GemmProblem(dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(), None,
                               dummy.data_ptr(), M, N, K, epi)
    return probs, dummy


def w4a16_set_grouped_variant(shapes, variant: int, device=None) -> None:
    """Memoize ``variant`` (with its per-problem schedules) as the plan of
    grouped launches of these ``(M, N, K)`` shapes, as a tuned choice."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    probs, _keep = _shape_problems(shapes, dev)
    _check(lib().w4a16_set_grouped_variant(probs, len(shapes), variant), "w4a16_set_grouped_variant")


def w4a16_gemm_grouped(As, packeds, scales_list, biases=None, Ys=None, workspace=None,
                       stream=None, variant=None, epilogues=None):
    """Independent W4A16 GEMMs ``Y_i = A_i @ dequant(W_i)^T + bias_i`` in one
    launch (bf16 or fp16 activations, all of one type).  ``epilogues[i] ==
    EPILOGUE_SWIGLU`` gives problem i the SwiGLU epilogue (interleaved
    up/gate rows, ``Y_i`` of ``[M, N/2]``, bf16).  Returns the Y's."""
    probs, outs, act = _gemm_problems(As, packeds, scales_list, biases, Ys, epilogues)
    n = len(outs)
    L = lib()
    v = -1 if variant is None else variant
    need = L.w4a16_gemm_grouped_workspace_bytes(probs, n, v)
    sh = _stream_handle(As[0].device, stream)
    if workspace is None:
        workspace = _default_ws.get(As[0].device, sh, need)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(L.w4a16_gemm_grouped(probs, n, GROUP, 1 if act == torch.float16 else 0, v, ws_ptr,
                                ws_bytes, sh), "w4a16_gemm_grouped")
    return outs


# --------------------------------------------------------------- variants
def w4a16_variant_count() -> int:
    return lib().w4a16_variant_count()


def w4a16_variant_name(variant: int) -> str | None:
    n = lib().w4a16_variant_name(variant)
    return None if n is None else n.decode()


def w4a16_variant_eligible(variant: int, M: int, N: int, K: int) -> bool:
    return bool(lib().w4a16_variant_eligible(variant, M, N, K))


def w4a16_variant_workspace_bytes(variant: int, M: int, N: int, K: int) -> int:
    return lib().w4a16_variant_workspace_bytes(variant, M, N, K)


def w4a16_select_variant(M: int, N: int, K: int) -> int:
    return lib().w4a16_select_variant(M, N, K)


def w4a16_variant_schedule(variant: int, M: int, N: int, K: int, num_sms: int = 0) -> dict:
    """The launch the library would make for `variant` on this shape (host
    only): grid, dp_tiles, sk_units, cluster, team (row-block kernel)."""
    out = (ctypes.c_int * 5)()
    _check(lib().w4a16_variant_schedule(variant, M, N, K, num_sms, out), "w4a16_variant_schedule")
    return dict(grid=out[0], dp_tiles=out[1], sk_units=out[2], cluster=out[3], team=out[4])


def variant_id(name: str) -> int:
    for i in range(w4a16_variant_count()):
        if w4a16_variant_name(i) == name:
            return i
    raise KeyError(name)


def w4a16_tune(M: int, N: int, K: int, stream=None, device=None) -> int:
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    out = ctypes.c_int(-1)
    _check(lib().w4a16_tune(M, N, K, _stream_handle(dev, stream), ctypes.byref(out)), "w4a16_tune")
    return out.value


def w4a16_tune_swiglu(M: int, N: int, K: int, stream=None, device=None) -> int:
    """Choose the SwiGLU-epilogue GEMM's variant for this shape by measurement
    (w4a16_tune_swiglu); returns the id."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    out = ctypes.c_int(-1)
    _check(lib().w4a16_tune_swiglu(M, N, K, _stream_handle(dev, stream), ctypes.byref(out)),
           "w4a16_tune_swiglu")
    return out.value


def w8a16_tune(M: int, N: int, K: int, stream=None, device=None) -> int:
    """Choose the INT8 GEMM's variant for this shape by measurement."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    out = ctypes.c_int(-1)
    _check(lib().w8a16_tune(M, N, K, _stream_handle(dev, stream), ctypes.byref(out)), "w8a16_tune")
    return out.value


def fp4a16_tune(M: int, N: int, K: int, fmt="mxfp4", stream=None, device=None) -> int:
    """Choose the FP4 GEMM's variant for this shape by measurement (timed with
    ``fmt``'s scales; the entry serves both formats)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    out = ctypes.c_int(-1)
    _check(lib().fp4a16_tune(_fp4_format(fmt), M, N, K, _stream_handle(dev, stream),
                             ctypes.byref(out)), "fp4a16_tune")
    return out.value


def w4a16_table_set(M: int, N: int, K: int, variant: int) -> None:
    _check(lib().w4a16_table_set(M, N, K, variant), "w4a16_table_set")


def w4a16_swiglu_table_set(M: int, N: int, K: int, variant: int) -> None:
    _check(lib().w4a16_swiglu_table_set(M, N, K, variant), "w4a16_swiglu_table_set")


def w8a16_table_set(M: int, N: int, K: int, variant: int) -> None:
    _check(lib().w8a16_table_set(M, N, K, variant), "w8a16_table_set")


def fp4a16_table_set(M: int, N: int, K: int, variant: int) -> None:
    _check(lib().fp4a16_table_set(M, N, K, variant), "fp4a16_table_set")


def w4a16_table_clear() -> None:
    lib().w4a16_table_clear()


def w4a16_table_save(path: str) -> None:
    _check(lib().w4a16_table_save(path.encode()), "w4a16_table_save")


def w4a16_table_load(path: str) -> None:
    _check(lib().w4a16_table_load(path.encode()), "w4a16_table_load")


# ------------------------------------------------------------ diagnostics
def w4a16_get_device_error(stream=None, device=None) -> int:
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    return lib().w4a16_get_device_error(_stream_handle(dev, stream))


def w4a16_set_wait_timeout_ns(ns: int) -> None:
    lib().w4a16_set_wait_timeout_ns(ns)


def w4a16_selftest_wait_timeout(timeout_ns: int, stream=None, device=None) -> None:
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    _check(lib().w4a16_selftest_wait_timeout(timeout_ns, _stream_handle(dev, stream)),
           "w4a16_selftest_wait_timeout")


def w4a16_set_weights_static(enable: bool) -> None:
    """Declare the GEMM weights static (w4a16_set_weights_static): no kernel
    that can run just before a GEMM on its stream writes that GEMM's packed
    codes or scales, so the GEMM may start copying them early."""
    lib().w4a16_set_weights_static(1 if enable else 0)


def w4a16_weights_static() -> bool:
    return bool(lib().w4a16_weights_static())


def w4a16_launch_count() -> int:
    return lib().w4a16_launch_count()
