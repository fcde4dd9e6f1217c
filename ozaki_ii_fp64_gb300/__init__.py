"""Ozaki scheme II FP64 emulation on GB300 FP4 tensor cores: Python binding.

A thin ctypes layer over libozemu.so (``include/ozemu.h``).  The functions
named ``ozemu_*`` mirror the C ABI one to one (ints for device pointers and
streams); the short-named helpers (``dgemm``, ``igemm_s8``, ``split_rows_f64``
...) only marshal torch CUDA tensors into those calls.  Every step of the
computation runs in the library's CUDA kernels; there is no fallback: if the
library cannot be built or loaded, importing the binding's functions raises.
"""

import ctypes
import os

from . import build as _build

OZEMU_OK = 0
OZEMU_ERR_INVALID_ARG = -1
OZEMU_ERR_K_OVERFLOW = -2
OZEMU_ERR_ALLOC = -3
OZEMU_ERR_CUDA = -4
OZEMU_ERR_NONFINITE = -5
OZEMU_ERR_TIMEOUT = -6
OZEMU_ERR_UNSUPPORTED = -7
OZEMU_ERR_SCRATCH_TOO_SMALL = -8
OZEMU_ERR_RANGE = -9

_STATUS_NAMES = {
    0: "OZEMU_OK", -1: "OZEMU_ERR_INVALID_ARG", -2: "OZEMU_ERR_K_OVERFLOW", -3: "OZEMU_ERR_ALLOC",
    -4: "OZEMU_ERR_CUDA", -5: "OZEMU_ERR_NONFINITE", -6: "OZEMU_ERR_TIMEOUT", -7: "OZEMU_ERR_UNSUPPORTED",
    -8: "OZEMU_ERR_SCRATCH_TOO_SMALL", -9: "OZEMU_ERR_RANGE",
}


class OzemuError(RuntimeError):
    def __init__(self, code, what=""):
        self.code = code
        super().__init__("%s failed: %s (%d)" % (what, _STATUS_NAMES.get(code, "?"), code))


_lib = None

_I = ctypes.c_int
_P = ctypes.c_void_p
_S = ctypes.c_size_t

_SIGNATURES = {
    "ozemu_igemm_s8": (_I, [_I, _I, _I, _P, _P, _P, _P]),
    "ozemu_igemm_s4s8": (_I, [_I, _I, _I, _P, _P, _P, _P]),
    "ozemu_four_plane_bytes": (_S, [_I, _I]),
    "ozemu_split_rows_s4": (_I, [_I, _I, _P, _I, _P, _P]),
    "ozemu_split_cols_s8_four": (_I, [_I, _I, _P, _I, _P, _P]),
    "ozemu_dgemm": (_I, [_I, _I, _I, _P, _I, _P, _I, _P, _I, _I, _P]),
    "ozemu_max_moduli": (_I, []),
    "ozemu_moduli": (_I, [_I, _P]),
    "ozemu_bit_budget": (_I, [_I, _I, _P, _P]),
    "ozemu_plane_bytes": (_S, [_I, _I, _I]),
    "ozemu_residue_bytes": (_S, [_I, _I, _I]),
    "ozemu_split_rows_f64": (_I, [_I, _I, _P, _I, _I, _I, _P, _P, _P]),
    "ozemu_split_cols_f64": (_I, [_I, _I, _P, _I, _I, _I, _P, _P, _P]),
    "ozemu_split_rows_s8": (_I, [_I, _I, _P, _I, _P, _P]),
    "ozemu_split_cols_s8": (_I, [_I, _I, _P, _I, _P, _P]),
    "ozemu_residue_gemm": (_I, [_I, _I, _I, _I, _P, _P, _P, _P]),
    "ozemu_limb_gemm_s32": (_I, [_I, _I, _I, _P, _P, _P, _I, _P]),
    "ozemu_crt_f64": (_I, [_I, _I, _I, _P, _P, _P, _P, _I, _P]),
    "ozemu_get_status": (_I, [_P]),
    "ozemu_release": (None, []),
    "ozemu_dgemm_noalloc": (_I, [_I, _I, _I, _P, _I, _P, _I, _P, _I, _I, _P]),
    "ozemu_res8_bytes": (_S, [_I, _I, _I]),
    "ozemu_split_rows_f64_res8": (_I, [_I, _I, _P, _I, _I, _I, _P, _P, _P]),
    "ozemu_split_cols_f64_res8": (_I, [_I, _I, _P, _I, _I, _I, _P, _P, _P]),
    "ozemu_residue_gemm_i8": (_I, [_I, _I, _I, _I, _P, _P, _P, _P]),
    "ozemu_narrow_max_n": (_I, []),
    "ozemu_dgemm_host": (_I, [_I, _I, _I, _P, _I, _P, _I, _P, _I, _I, _P]),
    "ozemu_residues_narrow_f64": (_I, [_I, _I, _I, _I, _P, _I, _P, _I, _P, _P, _P, _P]),
    "ozemu_moduli_2limb": (_I, [_I, _P]),
    "ozemu_bit_budget_2limb": (_I, [_I, _I, _P, _P]),
    "ozemu_plane_bytes_2limb": (_S, [_I, _I, _I]),
    "ozemu_split_rows_f64_2limb": (_I, [_I, _I, _P, _I, _I, _I, _P, _P, _P]),
    "ozemu_split_cols_f64_2limb": (_I, [_I, _I, _P, _I, _I, _I, _P, _P, _P]),
    "ozemu_residue_gemm_2limb": (_I, [_I, _I, _I, _I, _P, _P, _P, _P]),
    "ozemu_crt_f64_2limb": (_I, [_I, _I, _I, _P, _P, _P, _P, _I, _P]),
    "ozemu_dgemm_2limb": (_I, [_I, _I, _I, _P, _I, _P, _I, _P, _I, _I, _P]),
    "ozemu_dgemm_host_2limb": (_I, [_I, _I, _I, _P, _I, _P, _I, _P, _I, _I, _P]),
    "ozemu_get_status_noalloc": (_I, [_P]),
    "ozemu_set_workspace_limit": (_I, [_S]),
    "ozemu_workspace_limit": (_S, []),
    "ozemu_probe_wait_timeout": (_I, [ctypes.c_ulonglong, _P]),
    "ozemu_max_moduli_mixed": (_I, []),
    "ozemu_single_digit_moduli_mixed": (_I, []),
    "ozemu_moduli_mixed": (_I, [_I, _P]),
    "ozemu_bit_budget_mixed": (_I, [_I, _I, _P, _P]),
    "ozemu_plane_bytes_mixed": (_S, [_I, _I, _I]),
    "ozemu_products_mixed": (_I, [_I]),
    "ozemu_split_rows_f64_mixed": (_I, [_I, _I, _P, _I, _I, _I, _P, _P, _P]),
    "ozemu_split_cols_f64_mixed": (_I, [_I, _I, _P, _I, _I, _I, _P, _P, _P]),
    "ozemu_residue_gemm_mixed": (_I, [_I, _I, _I, _I, _P, _P, _P, _P]),
    "ozemu_crt_f64_mixed": (_I, [_I, _I, _I, _P, _P, _P, _P, _I, _P]),
    "ozemu_dgemm_mixed": (_I, [_I, _I, _I, _P, _I, _P, _I, _P, _I, _I, _P]),
    "ozemu_dgemm_host_mixed": (_I, [_I, _I, _I, _P, _I, _P, _I, _P, _I, _I, _P]),
}


def library_path():
    return _build.lib_path()


def load(build_if_needed=True):
    """Load libozemu.so (building it first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    if not _build.is_current():
        if not build_if_needed:
            raise ImportError("libozemu.so is missing or stale; run ozaki_ii_fp64_gb300.build.build()")
        _build.build()
    lib = ctypes.CDLL(_build.lib_path())
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _call(name, *args):
    return getattr(load(), name)(*args)


# ---------------------------------------------------------------- raw C ABI

def ozemu_igemm_s8(m, n, k, A, B, C32, stream):
    return _call("ozemu_igemm_s8", m, n, k, A, B, C32, stream)


def ozemu_igemm_s4s8(m, n, k, A, B, C32, stream):
    return _call("ozemu_igemm_s4s8", m, n, k, A, B, C32, stream)


def ozemu_four_plane_bytes(rows, k):
    return _call("ozemu_four_plane_bytes", rows, k)


def ozemu_split_rows_s4(rows, k, X, ldx, planes, stream):
    return _call("ozemu_split_rows_s4", rows, k, X, ldx, planes, stream)


def ozemu_split_cols_s8_four(k, cols, X, ldx, planes, stream):
    return _call("ozemu_split_cols_s8_four", k, cols, X, ldx, planes, stream)


def ozemu_dgemm(m, n, k, A, lda, B, ldb, C, ldc, r, stream):
    return _call("ozemu_dgemm", m, n, k, A, lda, B, ldb, C, ldc, r, stream)


def ozemu_max_moduli():
    return _call("ozemu_max_moduli")


def ozemu_moduli(r):
    buf = (ctypes.c_int32 * max(r, 1))()
    st = _call("ozemu_moduli", r, ctypes.cast(buf, ctypes.c_void_p))
    if st != OZEMU_OK:
        raise OzemuError(st, "ozemu_moduli")
    return [int(x) for x in buf[:r]]


def ozemu_bit_budget(k, r):
    pa, pb = ctypes.c_int(0), ctypes.c_int(0)
    st = _call("ozemu_bit_budget", k, r, ctypes.byref(pa), ctypes.byref(pb))
    if st != OZEMU_OK:
        raise OzemuError(st, "ozemu_bit_budget")
    return pa.value, pb.value


def ozemu_plane_bytes(rows, k, r):
    return _call("ozemu_plane_bytes", rows, k, r)


def ozemu_residue_bytes(m, n, r):
    return _call("ozemu_residue_bytes", m, n, r)


def ozemu_split_rows_f64(rows, k, X, ldx, p, r, planes, shifts, stream):
    return _call("ozemu_split_rows_f64", rows, k, X, ldx, p, r, planes, shifts, stream)


def ozemu_split_cols_f64(k, cols, X, ldx, p, r, planes, shifts, stream):
    return _call("ozemu_split_cols_f64", k, cols, X, ldx, p, r, planes, shifts, stream)


def ozemu_split_rows_s8(rows, k, X, ldx, planes, stream):
    return _call("ozemu_split_rows_s8", rows, k, X, ldx, planes, stream)


def ozemu_split_cols_s8(k, cols, X, ldx, planes, stream):
    return _call("ozemu_split_cols_s8", k, cols, X, ldx, planes, stream)


def ozemu_residue_gemm(m, n, k, r, a_planes, b_planes, residues, stream):
    return _call("ozemu_residue_gemm", m, n, k, r, a_planes, b_planes, residues, stream)


def ozemu_limb_gemm_s32(m, n, k, a_planes, b_planes, C32, ldc, stream):
    return _call("ozemu_limb_gemm_s32", m, n, k, a_planes, b_planes, C32, ldc, stream)


def ozemu_res8_bytes(rows, k, r):
    return _call("ozemu_res8_bytes", rows, k, r)


def ozemu_split_rows_f64_res8(rows, k, X, ldx, p, r, res8, shifts, stream):
    return _call("ozemu_split_rows_f64_res8", rows, k, X, ldx, p, r, res8, shifts, stream)


def ozemu_split_cols_f64_res8(k, cols, X, ldx, p, r, res8, shifts, stream):
    return _call("ozemu_split_cols_f64_res8", k, cols, X, ldx, p, r, res8, shifts, stream)


def ozemu_residue_gemm_i8(m, n, k, r, a_res8, b_res8, residues, stream):
    return _call("ozemu_residue_gemm_i8", m, n, k, r, a_res8, b_res8, residues, stream)


def ozemu_dgemm_host(m, n, k, A, lda, B, ldb, C, ldc, r, stream):
    return _call("ozemu_dgemm_host", m, n, k, A, lda, B, ldb, C, ldc, r, stream)


def ozemu_narrow_max_n():
    return _call("ozemu_narrow_max_n")


def ozemu_residues_narrow_f64(m, n, k, r, A, lda, B, ldb, residues, shifts_a, shifts_b, stream):
    return _call("ozemu_residues_narrow_f64", m, n, k, r, A, lda, B, ldb, residues, shifts_a, shifts_b, stream)


def ozemu_crt_f64(m, n, r, residues, shifts_a, shifts_b, C, ldc, stream):
    return _call("ozemu_crt_f64", m, n, r, residues, shifts_a, shifts_b, C, ldc, stream)


def ozemu_get_status(stream):
    return _call("ozemu_get_status", stream)


def ozemu_release():
    _call("ozemu_release")


def ozemu_dgemm_noalloc(m, n, k, A, lda, B, ldb, C, ldc, r, stream):
    return _call("ozemu_dgemm_noalloc", m, n, k, A, lda, B, ldb, C, ldc, r, stream)


def ozemu_get_status_noalloc(stream):
    return _call("ozemu_get_status_noalloc", stream)


def ozemu_set_workspace_limit(nbytes):
    return _call("ozemu_set_workspace_limit", nbytes)


def ozemu_workspace_limit():
    return _call("ozemu_workspace_limit")


def ozemu_probe_wait_timeout(limit_ns, stream):
    return _call("ozemu_probe_wait_timeout", limit_ns, stream)


def ozemu_moduli_2limb(r):
    buf = (ctypes.c_int32 * max(r, 1))()
    st = _call("ozemu_moduli_2limb", r, ctypes.cast(buf, ctypes.c_void_p))
    if st != OZEMU_OK:
        raise OzemuError(st, "ozemu_moduli_2limb")
    return [int(x) for x in buf[:r]]


def ozemu_bit_budget_2limb(k, r):
    pa, pb = ctypes.c_int(0), ctypes.c_int(0)
    st = _call("ozemu_bit_budget_2limb", k, r, ctypes.byref(pa), ctypes.byref(pb))
    if st != OZEMU_OK:
        raise OzemuError(st, "ozemu_bit_budget_2limb")
    return pa.value, pb.value


def ozemu_plane_bytes_2limb(rows, k, r):
    return _call("ozemu_plane_bytes_2limb", rows, k, r)


def ozemu_split_rows_f64_2limb(rows, k, X, ldx, p, r, planes, shifts, stream):
    return _call("ozemu_split_rows_f64_2limb", rows, k, X, ldx, p, r, planes, shifts, stream)


def ozemu_split_cols_f64_2limb(k, cols, X, ldx, p, r, planes, shifts, stream):
    return _call("ozemu_split_cols_f64_2limb", k, cols, X, ldx, p, r, planes, shifts, stream)


def ozemu_residue_gemm_2limb(m, n, k, r, a_planes, b_planes, residues, stream):
    return _call("ozemu_residue_gemm_2limb", m, n, k, r, a_planes, b_planes, residues, stream)


def ozemu_crt_f64_2limb(m, n, r, residues, shifts_a, shifts_b, C, ldc, stream):
    return _call("ozemu_crt_f64_2limb", m, n, r, residues, shifts_a, shifts_b, C, ldc, stream)


def ozemu_dgemm_2limb(m, n, k, A, lda, B, ldb, C, ldc, r, stream):
    return _call("ozemu_dgemm_2limb", m, n, k, A, lda, B, ldb, C, ldc, r, stream)


def ozemu_dgemm_host_2limb(m, n, k, A, lda, B, ldb, C, ldc, r, stream):
    return _call("ozemu_dgemm_host_2limb", m, n, k, A, lda, B, ldb, C, ldc, r, stream)


def ozemu_max_moduli_mixed():
    return _call("ozemu_max_moduli_mixed")


def ozemu_single_digit_moduli_mixed():
    return _call("ozemu_single_digit_moduli_mixed")


def ozemu_moduli_mixed(r):
    buf = (ctypes.c_int32 * max(r, 1))()
    st = _call("ozemu_moduli_mixed", r, ctypes.cast(buf, ctypes.c_void_p))
    if st != OZEMU_OK:
        raise OzemuError(st, "ozemu_moduli_mixed")
    return [int(x) for x in buf[:r]]


def ozemu_bit_budget_mixed(k, r):
    pa, pb = ctypes.c_int(0), ctypes.c_int(0)
    st = _call("ozemu_bit_budget_mixed", k, r, ctypes.byref(pa), ctypes.byref(pb))
    if st != OZEMU_OK:
        raise OzemuError(st, "ozemu_bit_budget_mixed")
    return pa.value, pb.value


def ozemu_plane_bytes_mixed(rows, k, r):
    return _call("ozemu_plane_bytes_mixed", rows, k, r)


def ozemu_products_mixed(r):
    return _call("ozemu_products_mixed", r)


def ozemu_split_rows_f64_mixed(rows, k, X, ldx, p, r, planes, shifts, stream):
    return _call("ozemu_split_rows_f64_mixed", rows, k, X, ldx, p, r, planes, shifts, stream)


def ozemu_split_cols_f64_mixed(k, cols, X, ldx, p, r, planes, shifts, stream):
    return _call("ozemu_split_cols_f64_mixed", k, cols, X, ldx, p, r, planes, shifts, stream)


def ozemu_residue_gemm_mixed(m, n, k, r, a_planes, b_planes, residues, stream):
    return _call("ozemu_residue_gemm_mixed", m, n, k, r, a_planes, b_planes, residues, stream)


def ozemu_crt_f64_mixed(m, n, r, residues, shifts_a, shifts_b, C, ldc, stream):
    return _call("ozemu_crt_f64_mixed", m, n, r, residues, shifts_a, shifts_b, C, ldc, stream)


def ozemu_dgemm_mixed(m, n, k, A, lda, B, ldb, C, ldc, r, stream):
    return _call("ozemu_dgemm_mixed", m, n, k, A, lda, B, ldb, C, ldc, r, stream)


def ozemu_dgemm_host_mixed(m, n, k, A, lda, B, ldb, C, ldc, r, stream):
    return _call("ozemu_dgemm_host_mixed", m, n, k, A, lda, B, ldb, C, ldc, r, stream)


# ------------------------------------------------------- torch marshalling

def _torch():
    import torch
    return torch


def _stream(stream=None):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _check(st, what):
    if st != OZEMU_OK:
        raise OzemuError(st, what)


def _ld(t):
    """Leading dimension of a row-major 2-D tensor (unit inner stride)."""
    if t.dim() != 2:
        raise ValueError("expected a 2-D tensor")
    if t.numel() == 0:
        return max(t.shape[1], 1)
    if t.stride(1) != 1 and t.shape[1] > 1:
        raise ValueError("expected a row-major 2-D tensor")
    return max(t.stride(0), max(t.shape[1], 1))


def plane_layout(rows, k):
    """(rows_padded, row_bytes) of the limb-plane layout."""
    return (rows + 127) // 128 * 128, (k + 127) // 128 * 128 // 2


def dgemm(A, B, r, out=None, stream=None):
    """Emulated fp64 A @ B (cuda float64 row-major tensors) with r moduli."""
    torch = _torch()
    m, k = A.shape
    k2, n = B.shape
    if k != k2:
        raise ValueError("inner dimensions differ")
    C = torch.empty((m, n), dtype=torch.float64, device=A.device) if out is None else out
    _check(ozemu_dgemm(m, n, k, A.data_ptr(), _ld(A), B.data_ptr(), _ld(B), C.data_ptr(), _ld(C), r,
                       _stream(stream)), "ozemu_dgemm")
    return C


def dgemm_host(A, B, r, out=None, stream=None):
    """Emulated fp64 A @ B of CPU float64 tensors (pinned for overlap) through
    ozemu_dgemm_host; returns the CPU result after synchronising the stream."""
    torch = _torch()
    m, k = A.shape
    k2, n = B.shape
    if k != k2 or A.device.type != "cpu" or B.device.type != "cpu":
        raise ValueError("expected CPU matrices with matching inner dimension")
    C = torch.empty((m, n), dtype=torch.float64, pin_memory=A.is_pinned()) if out is None else out
    s = torch.cuda.current_stream() if stream is None else stream
    _check(ozemu_dgemm_host(m, n, k, A.data_ptr(), _ld(A), B.data_ptr(), _ld(B), C.data_ptr(), _ld(C), r,
                            s.cuda_stream), "ozemu_dgemm_host")
    s.synchronize()
    return C


def igemm_s8(A, B, out=None, stream=None):
    """Exact int32 A @ B of contiguous int8 cuda tensors."""
    torch = _torch()
    m, k = A.shape
    k2, n = B.shape
    if k != k2 or not A.is_contiguous() or not B.is_contiguous():
        raise ValueError("expected contiguous int8 matrices with matching inner dimension")
    C = torch.empty((m, n), dtype=torch.int32, device=A.device) if out is None else out
    _check(ozemu_igemm_s8(m, n, k, A.data_ptr(), B.data_ptr(), C.data_ptr(), _stream(stream)), "ozemu_igemm_s8")
    return C


def igemm_s4s8(A, B, out=None, stream=None):
    """Exact int32 A @ B of a contiguous int8 cuda tensor A holding INT4 values
    ([-8, 7]) and a contiguous int8 cuda tensor B (four FP4 products)."""
    torch = _torch()
    m, k = A.shape
    k2, n = B.shape
    if k != k2 or not A.is_contiguous() or not B.is_contiguous():
        raise ValueError("expected contiguous int8 matrices with matching inner dimension")
    C = torch.empty((m, n), dtype=torch.int32, device=A.device) if out is None else out
    _check(ozemu_igemm_s4s8(m, n, k, A.data_ptr(), B.data_ptr(), C.data_ptr(), _stream(stream)),
           "ozemu_igemm_s4s8")
    return C


def alloc_planes(rows, k, r, device):
    torch = _torch()
    return torch.empty(ozemu_plane_bytes(rows, k, r), dtype=torch.uint8, device=device)


def split_rows_f64(X, p, r, stream=None):
    """(planes, shifts) of the rows of a cuda float64 matrix."""
    torch = _torch()
    rows, k = X.shape
    planes = alloc_planes(rows, k, r, X.device)
    shifts = torch.empty(rows, dtype=torch.int32, device=X.device)
    _check(ozemu_split_rows_f64(rows, k, X.data_ptr(), _ld(X), p, r, planes.data_ptr(), shifts.data_ptr(),
                                _stream(stream)), "ozemu_split_rows_f64")
    return planes, shifts


def split_cols_f64(X, p, r, stream=None):
    """(planes, shifts) of the columns of a cuda float64 matrix."""
    torch = _torch()
    k, cols = X.shape
    planes = alloc_planes(cols, k, r, X.device)
    shifts = torch.empty(cols, dtype=torch.int32, device=X.device)
    _check(ozemu_split_cols_f64(k, cols, X.data_ptr(), _ld(X), p, r, planes.data_ptr(), shifts.data_ptr(),
                                _stream(stream)), "ozemu_split_cols_f64")
    return planes, shifts


def split_rows_s8(X, stream=None):
    rows, k = X.shape
    planes = alloc_planes(rows, k, 1, X.device)
    _check(ozemu_split_rows_s8(rows, k, X.data_ptr(), _ld(X), planes.data_ptr(), _stream(stream)),
           "ozemu_split_rows_s8")
    return planes


def split_cols_s8(X, stream=None):
    k, cols = X.shape
    planes = alloc_planes(cols, k, 1, X.device)
    _check(ozemu_split_cols_s8(k, cols, X.data_ptr(), _ld(X), planes.data_ptr(), _stream(stream)),
           "ozemu_split_cols_s8")
    return planes


def residue_gemm(m, n, k, r, a_planes, b_planes, out=None, stream=None):
    """uint8 residues [r][m][round_up(n, 16)] of the limb product."""
    torch = _torch()
    ldr = (n + 15) // 16 * 16
    res = torch.empty((r, m, ldr), dtype=torch.uint8, device=a_planes.device) if out is None else out
    _check(ozemu_residue_gemm(m, n, k, r, a_planes.data_ptr(), b_planes.data_ptr(), res.data_ptr(),
                              _stream(stream)), "ozemu_residue_gemm")
    return res


def split_rows_f64_res8(X, p, r, stream=None):
    """(int8 residues, shifts) of the rows of a cuda float64 matrix."""
    torch = _torch()
    rows, k = X.shape
    res = torch.empty(ozemu_res8_bytes(rows, k, r), dtype=torch.int8, device=X.device)
    shifts = torch.empty(rows, dtype=torch.int32, device=X.device)
    _check(ozemu_split_rows_f64_res8(rows, k, X.data_ptr(), _ld(X), p, r, res.data_ptr(), shifts.data_ptr(),
                                     _stream(stream)), "ozemu_split_rows_f64_res8")
    return res, shifts


def split_cols_f64_res8(X, p, r, stream=None):
    """(int8 residues, shifts) of the columns of a cuda float64 matrix."""
    torch = _torch()
    k, cols = X.shape
    res = torch.empty(ozemu_res8_bytes(cols, k, r), dtype=torch.int8, device=X.device)
    shifts = torch.empty(cols, dtype=torch.int32, device=X.device)
    _check(ozemu_split_cols_f64_res8(k, cols, X.data_ptr(), _ld(X), p, r, res.data_ptr(), shifts.data_ptr(),
                                     _stream(stream)), "ozemu_split_cols_f64_res8")
    return res, shifts


def residue_gemm_i8(m, n, k, r, a_res8, b_res8, out=None, stream=None):
    """Residues [r][m][round_up(n, 16)] by the INT8 mma.sync comparison path."""
    torch = _torch()
    ldr = (n + 15) // 16 * 16
    res = torch.empty((r, m, ldr), dtype=torch.uint8, device=a_res8.device) if out is None else out
    _check(ozemu_residue_gemm_i8(m, n, k, r, a_res8.data_ptr(), b_res8.data_ptr(), res.data_ptr(),
                                 _stream(stream)), "ozemu_residue_gemm_i8")
    return res


def limb_gemm_s32(m, n, k, a_planes, b_planes, out=None, stream=None):
    torch = _torch()
    C = torch.empty((m, n), dtype=torch.int32, device=a_planes.device) if out is None else out
    _check(ozemu_limb_gemm_s32(m, n, k, a_planes.data_ptr(), b_planes.data_ptr(), C.data_ptr(), _ld(C),
                               _stream(stream)), "ozemu_limb_gemm_s32")
    return C


def residues_narrow_f64(A, B, r, stream=None):
    """(residues, shifts_a, shifts_b) of A @ B for a narrow B (n <= 2) by the
    fused path: no limb planes."""
    torch = _torch()
    m, k = A.shape
    k2, n = B.shape
    if k != k2:
        raise ValueError("inner dimensions differ")
    res = torch.empty(ozemu_residue_bytes(m, n, r), dtype=torch.uint8, device=A.device)
    sa = torch.empty(m, dtype=torch.int32, device=A.device)
    sb = torch.empty(n, dtype=torch.int32, device=A.device)
    _check(ozemu_residues_narrow_f64(m, n, k, r, A.data_ptr(), _ld(A), B.data_ptr(), _ld(B), res.data_ptr(),
                                     sa.data_ptr(), sb.data_ptr(), _stream(stream)), "ozemu_residues_narrow_f64")
    return res.view(r, m, (n + 15) // 16 * 16), sa, sb


def crt_f64(m, n, r, residues, shifts_a, shifts_b, out=None, stream=None):
    torch = _torch()
    C = torch.empty((m, n), dtype=torch.float64, device=residues.device) if out is None else out
    _check(ozemu_crt_f64(m, n, r, residues.data_ptr(), shifts_a.data_ptr(), shifts_b.data_ptr(), C.data_ptr(),
                         _ld(C), _stream(stream)), "ozemu_crt_f64")
    return C


def get_status(stream=None):
    return ozemu_get_status(_stream(stream))


# ------------------------------------------------------ two-limb moduli

def dgemm_2limb(A, B, r, out=None, stream=None):
    """Emulated fp64 A @ B with r two-limb moduli (4 FP4 products each)."""
    torch = _torch()
    m, k = A.shape
    k2, n = B.shape
    if k != k2:
        raise ValueError("inner dimensions differ")
    C = torch.empty((m, n), dtype=torch.float64, device=A.device) if out is None else out
    _check(ozemu_dgemm_2limb(m, n, k, A.data_ptr(), _ld(A), B.data_ptr(), _ld(B), C.data_ptr(), _ld(C), r,
                             _stream(stream)), "ozemu_dgemm_2limb")
    return C


def dgemm_host_2limb(A, B, r, out=None, stream=None):
    """ozemu_dgemm_host_2limb of CPU float64 tensors (pinned for overlap);
    returns the CPU result after synchronising the stream."""
    torch = _torch()
    m, k = A.shape
    k2, n = B.shape
    if k != k2 or A.device.type != "cpu" or B.device.type != "cpu":
        raise ValueError("expected CPU matrices with matching inner dimension")
    C = torch.empty((m, n), dtype=torch.float64, pin_memory=A.is_pinned()) if out is None else out
    s = torch.cuda.current_stream() if stream is None else stream
    _check(ozemu_dgemm_host_2limb(m, n, k, A.data_ptr(), _ld(A), B.data_ptr(), _ld(B), C.data_ptr(), _ld(C), r,
                                  s.cuda_stream), "ozemu_dgemm_host_2limb")
    s.synchronize()
    return C


def split_rows_f64_2limb(X, p, r, stream=None):
    """(planes, shifts) of the rows of a cuda float64 matrix, two limbs."""
    torch = _torch()
    rows, k = X.shape
    planes = torch.empty(ozemu_plane_bytes_2limb(rows, k, r), dtype=torch.uint8, device=X.device)
    shifts = torch.empty(rows, dtype=torch.int32, device=X.device)
    _check(ozemu_split_rows_f64_2limb(rows, k, X.data_ptr(), _ld(X), p, r, planes.data_ptr(), shifts.data_ptr(),
                                      _stream(stream)), "ozemu_split_rows_f64_2limb")
    return planes, shifts


def split_cols_f64_2limb(X, p, r, stream=None):
    """(planes, shifts) of the columns of a cuda float64 matrix, two limbs."""
    torch = _torch()
    k, cols = X.shape
    planes = torch.empty(ozemu_plane_bytes_2limb(cols, k, r), dtype=torch.uint8, device=X.device)
    shifts = torch.empty(cols, dtype=torch.int32, device=X.device)
    _check(ozemu_split_cols_f64_2limb(k, cols, X.data_ptr(), _ld(X), p, r, planes.data_ptr(), shifts.data_ptr(),
                                      _stream(stream)), "ozemu_split_cols_f64_2limb")
    return planes, shifts


def residue_gemm_2limb(m, n, k, r, a_planes, b_planes, out=None, stream=None):
    """uint8 residues [r][m][round_up(n, 16)] of the two-limb product."""
    torch = _torch()
    ldr = (n + 15) // 16 * 16
    res = torch.empty((r, m, ldr), dtype=torch.uint8, device=a_planes.device) if out is None else out
    _check(ozemu_residue_gemm_2limb(m, n, k, r, a_planes.data_ptr(), b_planes.data_ptr(), res.data_ptr(),
                                    _stream(stream)), "ozemu_residue_gemm_2limb")
    return res


def crt_f64_2limb(m, n, r, residues, shifts_a, shifts_b, out=None, stream=None):
    torch = _torch()
    C = torch.empty((m, n), dtype=torch.float64, device=residues.device) if out is None else out
    _check(ozemu_crt_f64_2limb(m, n, r, residues.data_ptr(), shifts_a.data_ptr(), shifts_b.data_ptr(),
                               C.data_ptr(), _ld(C), _stream(stream)), "ozemu_crt_f64_2limb")
    return C


# --------------------------------------------------- mixed-digit moduli

def dgemm_mixed(A, B, r, out=None, stream=None):
    """Emulated fp64 A @ B with r mixed-digit moduli (one FP4 product for
    each single-digit modulus, four for each two-digit one)."""
    torch = _torch()
    m, k = A.shape
    k2, n = B.shape
    if k != k2:
        raise ValueError("inner dimensions differ")
    C = torch.empty((m, n), dtype=torch.float64, device=A.device) if out is None else out
    _check(ozemu_dgemm_mixed(m, n, k, A.data_ptr(), _ld(A), B.data_ptr(), _ld(B), C.data_ptr(), _ld(C), r,
                             _stream(stream)), "ozemu_dgemm_mixed")
    return C


def dgemm_host_mixed(A, B, r, out=None, stream=None):
    """ozemu_dgemm_host_mixed of CPU float64 tensors (pinned for overlap);
    returns the CPU result after synchronising the stream."""
    torch = _torch()
    m, k = A.shape
    k2, n = B.shape
    if k != k2 or A.device.type != "cpu" or B.device.type != "cpu":
        raise ValueError("expected CPU matrices with matching inner dimension")
    C = torch.empty((m, n), dtype=torch.float64, pin_memory=A.is_pinned()) if out is None else out
    s = torch.cuda.current_stream() if stream is None else stream
    _check(ozemu_dgemm_host_mixed(m, n, k, A.data_ptr(), _ld(A), B.data_ptr(), _ld(B), C.data_ptr(), _ld(C), r,
                                  s.cuda_stream), "ozemu_dgemm_host_mixed")
    s.synchronize()
    return C


def split_rows_f64_mixed(X, p, r, stream=None):
    """(planes, shifts) of the rows of a cuda float64 matrix, mixed digits."""
    torch = _torch()
    rows, k = X.shape
    planes = torch.empty(ozemu_plane_bytes_mixed(rows, k, r), dtype=torch.uint8, device=X.device)
    shifts = torch.empty(rows, dtype=torch.int32, device=X.device)
    _check(ozemu_split_rows_f64_mixed(rows, k, X.data_ptr(), _ld(X), p, r, planes.data_ptr(), shifts.data_ptr(),
                                      _stream(stream)), "ozemu_split_rows_f64_mixed")
    return planes, shifts


def split_cols_f64_mixed(X, p, r, stream=None):
    """(planes, shifts) of the columns of a cuda float64 matrix, mixed digits."""
    torch = _torch()
    k, cols = X.shape
    planes = torch.empty(ozemu_plane_bytes_mixed(cols, k, r), dtype=torch.uint8, device=X.device)
    shifts = torch.empty(cols, dtype=torch.int32, device=X.device)
    _check(ozemu_split_cols_f64_mixed(k, cols, X.data_ptr(), _ld(X), p, r, planes.data_ptr(), shifts.data_ptr(),
                                      _stream(stream)), "ozemu_split_cols_f64_mixed")
    return planes, shifts


def residue_gemm_mixed(m, n, k, r, a_planes, b_planes, out=None, stream=None):
    """uint8 residues [r][m][round_up(n, 16)] of the mixed-digit product."""
    torch = _torch()
    ldr = (n + 15) // 16 * 16
    res = torch.empty((r, m, ldr), dtype=torch.uint8, device=a_planes.device) if out is None else out
    _check(ozemu_residue_gemm_mixed(m, n, k, r, a_planes.data_ptr(), b_planes.data_ptr(), res.data_ptr(),
                                    _stream(stream)), "ozemu_residue_gemm_mixed")
    return res


def crt_f64_mixed(m, n, r, residues, shifts_a, shifts_b, out=None, stream=None):
    torch = _torch()
    C = torch.empty((m, n), dtype=torch.float64, device=residues.device) if out is None else out
    _check(ozemu_crt_f64_mixed(m, n, r, residues.data_ptr(), shifts_a.data_ptr(), shifts_b.data_ptr(),
                               C.data_ptr(), _ld(C), _stream(stream)), "ozemu_crt_f64_mixed")
    return C
