"""Python binding of libtfqmm, the MLX-affine quantized row product for GB300.

Argument marshalling only: every step of the product runs in the library's
CUDA kernels (``csrc/``).  The names and arguments follow ``include/tfqmm.h``.
Tensors may be passed as torch tensors (their ``data_ptr()`` is used) or as
raw integer addresses; ``stream`` is a ``torch.cuda.Stream``, a raw
``cudaStream_t`` integer, or None for torch's current stream.

The library must be built first (``mlx_affine_bit_gb300.build.build()``);
loading fails loudly when it is missing.  There is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
SO = os.path.join(HERE, "_build", "libtfqmm.so")
SO_DEBUG = os.path.join(HERE, "_build", "libtfqmm_debug.so")   # bounds-checking build (tfqmm_debug.h)
SO_TRACE = os.path.join(HERE, "_build", "libtfqmm_trace.so")   # phase-trace build (tfqmm_trace.h)

TF_OK = 0
STATUS = {
    -1: "TF_EINVAL_BITS", -2: "TF_EINVAL_GROUP", -3: "TF_EINVAL_ROWS", -4: "TF_EINVAL_STRIDE",
    -5: "TF_EINVAL_PTR", -6: "TF_EINVAL_SIZE", -7: "TF_ENARROW", -8: "TF_EGROUP",
    -9: "TF_ESTACK", -10: "TF_ECUDA", -11: "TF_EDEVICE", -12: "TF_EINVAL_FLAGS", -13: "TF_EGATHER",
    -14: "TF_EBOUNDS",
}
SYMBOLS = ("tf_qmm", "tf_qmm_ex", "tf_qmm_prompt", "tf_qmm_gather", "tf_qmm_noalloc", "tf_noalloc_status", "tf_qmm_stack", "tf_widen",
           "tf_widen_host", "tf_common_width", "tf_qmm_bytes", "tf_device_status", "tf_set_launch_mode",
           "tf_inject_stall", "tf_last_error_string", "tf_version")
TF_LAUNCH_PDL, TF_LAUNCH_EARLY_WEIGHTS, TF_LAUNCH_EARLY_X = 1, 2, 4
TF_OUT_BF16, TF_EPI_RELU2 = 1, 2


class TfError(RuntimeError):
    def __init__(self, rc: int, msg: str):
        super().__init__("%s (%d): %s" % (STATUS.get(rc, "?"), rc, msg))
        self.rc = rc


class TfRun(ctypes.Structure):
    _fields_ = [("W", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("biases", ctypes.c_void_p),
                ("N", ctypes.c_int), ("bits", ctypes.c_int), ("group", ctypes.c_int)]


class TfMember(ctypes.Structure):
    _fields_ = [("run", ctypes.c_int), ("src_col", ctypes.c_int), ("n_cols", ctypes.c_int),
                ("dst_col", ctypes.c_int)]


_lib = None
_debug_lib = None
_trace_lib = None


def lib():
    """The loaded libtfqmm (raises if it has not been built)."""
    global _lib
    if _lib is None:
        _lib = _load(SO)
    return _lib


def debug_lib():
    """The loaded bounds-checking build, libtfqmm_debug.so (same entry points, plus tf_debug_shrink_y)."""
    global _debug_lib
    if _debug_lib is None:
        _debug_lib = _load(SO_DEBUG)
        _debug_lib.tf_debug_shrink_y.argtypes = [ctypes.c_int]
        _debug_lib.tf_debug_shrink_y.restype = ctypes.c_int
    return _debug_lib


def trace_lib():
    """The loaded phase-trace build, libtfqmm_trace.so (same entry points, plus tf_trace_reset / tf_trace_read)."""
    global _trace_lib
    if _trace_lib is None:
        _trace_lib = _load(SO_TRACE)
        _trace_lib.tf_trace_reset.argtypes = []
        _trace_lib.tf_trace_reset.restype = ctypes.c_int
        _trace_lib.tf_trace_read.argtypes = [ctypes.c_void_p, ctypes.c_int]
        _trace_lib.tf_trace_read.restype = ctypes.c_int
    return _trace_lib


class using:
    """Context manager: the calls of this module go to library L (a build from
    debug_lib() or trace_lib()) inside the block."""

    def __init__(self, L):
        self.L = L

    def __enter__(self):
        global _lib
        self.old, _lib = _lib, self.L
        return self.L

    def __exit__(self, *exc):
        global _lib
        _lib = self.old
        return False


def _load(path):
    """Open one build of the library and declare its entry points' argument types."""
    if not os.path.exists(path):
        raise ImportError("%s is not built; run mlx_affine_bit_gb300.build.build()" % path)
    L = ctypes.CDLL(path)
    P, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    L.tf_qmm.argtypes = [P, i32, i32, P, P, P, i32, i32, i32, P, i64, P]
    L.tf_qmm_noalloc.argtypes = [P, i32, i32, P, P, P, i32, i32, i32, P, i64, P]
    L.tf_qmm_ex.argtypes = [P, i32, i32, P, P, P, i32, i32, i32, P, i64, i32, P]
    L.tf_qmm_prompt.argtypes = [P, i32, i32, P, P, P, i32, i32, i32, P, i64, i32, P]
    L.tf_qmm_gather.argtypes = [P, i32, i32, ctypes.POINTER(TfRun), i32, ctypes.POINTER(ctypes.c_int),
                                ctypes.POINTER(ctypes.c_int), i32, P, i64, i32, P]
    L.tf_qmm_stack.argtypes = [P, i32, i32, ctypes.POINTER(TfRun), i32,
                               ctypes.POINTER(TfMember), i32, P, i64, P]
    L.tf_widen.argtypes = [P, P, P, i32, i32, i32, i32, P, P, P, i32, i32, P]
    L.tf_widen_host.argtypes = [P, P, P, i32, i32, i32, i32, P, P, P, i32, i32]
    L.tf_common_width.argtypes = [P, P, i32, P, P]
    L.tf_qmm_bytes.argtypes = [i32, i32, i32, i32, P, P]
    L.tf_device_status.argtypes = []
    L.tf_noalloc_status.argtypes = []
    L.tf_set_launch_mode.argtypes = [i32]
    L.tf_inject_stall.argtypes = []
    L.tf_last_error_string.restype = ctypes.c_char_p
    L.tf_version.restype = ctypes.c_char_p
    for name in ("tf_qmm", "tf_qmm_ex", "tf_qmm_prompt", "tf_qmm_gather", "tf_qmm_noalloc", "tf_qmm_stack", "tf_widen",
                 "tf_widen_host", "tf_common_width", "tf_qmm_bytes", "tf_device_status", "tf_noalloc_status",
                 "tf_set_launch_mode", "tf_inject_stall"):
        getattr(L, name).restype = i32
    return L


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int) -> None:
    if rc != TF_OK:
        raise TfError(rc, lib().tf_last_error_string().decode())


def tf_qmm(x, rows, K, W, scales, biases, N, bits, group, y, y_stride, stream=None) -> None:
    _check(lib().tf_qmm(_ptr(x), rows, K, _ptr(W), _ptr(scales), _ptr(biases), N, bits, group,
                        _ptr(y), y_stride, _stream(stream)))


def tf_qmm_noalloc(x, rows, K, W, scales, biases, N, bits, group, y, y_stride, stream=None) -> None:
    """tf_qmm with no device allocation (fixed built-in scratch; see include/tfqmm.h)."""
    _check(lib().tf_qmm_noalloc(_ptr(x), rows, K, _ptr(W), _ptr(scales), _ptr(biases), N, bits,
                                group, _ptr(y), y_stride, _stream(stream)))


def tf_qmm_ex(x, rows, K, W, scales, biases, N, bits, group, y, y_stride, flags, stream=None) -> None:
    """tf_qmm with output flags (TF_OUT_BF16: y is bf16; TF_EPI_RELU2: squared ReLU)."""
    _check(lib().tf_qmm_ex(_ptr(x), rows, K, _ptr(W), _ptr(scales), _ptr(biases), N, bits, group,
                           _ptr(y), y_stride, flags, _stream(stream)))


def tf_qmm_prompt(x, rows, K, W, scales, biases, N, bits, group, y, y_stride, flags=0, stream=None) -> None:
    """Many-row product on the tcgen05 tensor cores, weights read once per 64 rows (see include/tfqmm.h)."""
    _check(lib().tf_qmm_prompt(_ptr(x), rows, K, _ptr(W), _ptr(scales), _ptr(biases), N, bits, group,
                               _ptr(y), y_stride, flags, _stream(stream)))


def tf_qmm_gather(x, x_rows, K, experts, slot_expert, slot_row, y, y_stride, flags=0, stream=None) -> None:
    """experts: [(W, scales, biases, N, bits, group)]; slot i: y row i = experts[slot_expert[i]] x row slot_row[i]."""
    ee = (TfRun * len(experts))(*[TfRun(_ptr(W), _ptr(s), _ptr(b), N, bits, g)
                                  for (W, s, b, N, bits, g) in experts])
    n = len(slot_expert)
    se = (ctypes.c_int * n)(*slot_expert)
    sr = (ctypes.c_int * len(slot_row))(*slot_row)
    _check(lib().tf_qmm_gather(_ptr(x), x_rows, K, ee, len(experts), se, sr, n, _ptr(y), y_stride, flags,
                               _stream(stream)))


def tf_qmm_stack(x, rows, K, runs, members, y, y_stride, stream=None) -> None:
    """runs: [(W, scales, biases, N, bits, group)]; members: [(run, src_col, n_cols, dst_col)]."""
    rr = (TfRun * len(runs))(*[TfRun(_ptr(W), _ptr(s), _ptr(b), N, bits, g)
                               for (W, s, b, N, bits, g) in runs])
    mm = (TfMember * len(members))(*[TfMember(*m) for m in members])
    _check(lib().tf_qmm_stack(_ptr(x), rows, K, rr, len(runs), mm, len(members), _ptr(y),
                              y_stride, _stream(stream)))


def tf_widen(W, scales, biases, N, K, bits, group, W_out, s_out, b_out, bits_out, group_out,
             stream=None) -> None:
    _check(lib().tf_widen(_ptr(W), _ptr(scales), _ptr(biases), N, K, bits, group, _ptr(W_out),
                          _ptr(s_out), _ptr(b_out), bits_out, group_out, _stream(stream)))


def tf_widen_host(W, scales, biases, N, K, bits, group, bits_out, group_out):
    """Widen / regroup on host numpy arrays (uint32 W, uint16 scales/biases); returns (W_out, s_out, b_out)."""
    import numpy as np
    W = np.ascontiguousarray(W, dtype=np.uint32)
    s = np.ascontiguousarray(scales, dtype=np.uint16)
    b = np.ascontiguousarray(biases, dtype=np.uint16)
    Wo = np.zeros((N, K * bits_out // 32), dtype=np.uint32)
    so = np.zeros((N, K // group_out), dtype=np.uint16)
    bo = np.zeros((N, K // group_out), dtype=np.uint16)
    _check(lib().tf_widen_host(W.ctypes.data, s.ctypes.data, b.ctypes.data, N, K, bits, group, Wo.ctypes.data,
                               so.ctypes.data, bo.ctypes.data, bits_out, group_out))
    return Wo, so, bo


def tf_common_width(bits_list, groups_list) -> tuple[int, int]:
    n = len(bits_list)
    b = (ctypes.c_int * n)(*bits_list)
    g = (ctypes.c_int * n)(*groups_list)
    bo, go = ctypes.c_int(), ctypes.c_int()
    _check(lib().tf_common_width(b, g, n, ctypes.byref(bo), ctypes.byref(go)))
    return bo.value, go.value


def tf_qmm_bytes(N, K, bits, group) -> tuple[int, int]:
    wb, sb = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().tf_qmm_bytes(N, K, bits, group, ctypes.byref(wb), ctypes.byref(sb)))
    return wb.value, sb.value


def tf_device_status() -> None:
    _check(lib().tf_device_status())


def tf_noalloc_status() -> None:
    """Raise TfError(TF_EDEVICE) if a tf_qmm_noalloc product gave up a bounded wait (clears it)."""
    _check(lib().tf_noalloc_status())


def tf_set_launch_mode(mode: int) -> int:
    """Set the launch mode (TF_LAUNCH_* bits) of later calls; returns the previous mode."""
    rc = lib().tf_set_launch_mode(mode)
    if rc < 0:
        _check(rc)
    return rc


def tf_inject_stall() -> None:
    """Test hook: the next product's first stage is withheld (its bounded wait runs out)."""
    _check(lib().tf_inject_stall())


def tf_version() -> str:
    return lib().tf_version().decode()


def qmm(x, W, scales, biases, bits, group, y=None, y_stride=None, stream=None):
    """Convenience wrapper on torch tensors: x [rows][K] bf16, W [N][K*bits/32] int32.

    Allocates y [rows][N] fp32 when not given, then calls tf_qmm.
    """
    import torch
    rows, K = x.shape
    N = W.shape[0]
    if y is None:
        y = torch.empty((rows, N), dtype=torch.float32, device=x.device)
        y_stride = N
    tf_qmm(x, rows, K, W, scales, biases, N, bits, group, y,
           y_stride if y_stride is not None else y.stride(0), stream)
    return y
