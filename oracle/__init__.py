"""fp64 CPU oracle for the MLX-affine quantized row product -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package.  The product path (``mlx_affine_bit_gb300``)
never imports it, and this package imports nothing from the product.

The arithmetic lives in ``oracle.c`` (plain C, fp64, one bit at a time); see
``oracle.h`` for the definitions and their sources.  This module only builds
the shared object with gcc and marshals numpy arrays to it.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
against hand-packed fixtures (``tests/golden/``), closed forms, exact integer
brute force and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")

OK, EINVAL, ENARROW, EGROUP = 0, -1, -2, -3


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (no fast-math, no FMA contraction)."""
    src = os.path.join(_HERE, "oracle.c")
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= max(
            os.path.getmtime(src), os.path.getmtime(os.path.join(_HERE, "oracle.h"))):
        return _SO
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _SO + ".tmp%d" % os.getpid()
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                           "-pthread", src, "-o", tmp, "-lm"])
    os.replace(tmp, _SO)
    return _SO


_lib = None


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i64, i32 = ctypes.c_int64, ctypes.c_int
        L.oracle_words_per_row.restype = i64
        L.oracle_words_per_row.argtypes = [i64, i32]
        L.oracle_code.restype = ctypes.c_uint32
        L.oracle_code.argtypes = [P, i64, i32, i64, i64]
        L.oracle_bf16.restype = ctypes.c_double
        L.oracle_bf16.argtypes = [ctypes.c_uint16]
        L.oracle_weights.restype = i32
        L.oracle_weights.argtypes = [P, P, P, i64, i64, i32, i32, i64, i64, P]
        L.oracle_qmm.restype = i32
        L.oracle_qmm.argtypes = [P, i32, i64, P, P, P, i64, i32, i32, P, i64, P, P, i32]
        L.oracle_widen.restype = i32
        L.oracle_widen.argtypes = [P, P, P, i64, i64, i32, i32, P, P, P, i32, i32]
        L.oracle_common_width.restype = i32
        L.oracle_common_width.argtypes = [P, P, i32, P, P]
        L.oracle_relu2.restype = None
        L.oracle_relu2.argtypes = [P, i64, P]
        _lib = L
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class OracleError(RuntimeError):
    def __init__(self, rc: int):
        super().__init__("oracle returned %d" % rc)
        self.rc = rc


def code(W, K: int, bits: int, n: int, k: int) -> int:
    W = _c(W, np.uint32)
    return int(lib().oracle_code(_p(W), K, bits, n, k))


def bf16(h: int) -> float:
    return float(lib().oracle_bf16(int(h)))


def weights(W, scales, biases, N, K, bits, group, n0=0, n1=None) -> np.ndarray:
    n1 = N if n1 is None else n1
    W, s, b = _c(W, np.uint32), _c(scales, np.uint16), _c(biases, np.uint16)
    out = np.empty((n1 - n0, K), dtype=np.float64)
    rc = lib().oracle_weights(_p(W), _p(s), _p(b), N, K, bits, group, n0, n1, _p(out))
    if rc:
        raise OracleError(rc)
    return out


def qmm(x, W, scales, biases, N, K, bits, group, cols=None, nthreads: int = 1):
    """(y64, absum), each [rows][ncols] float64, for the columns ``cols`` (default all)."""
    x = _c(x, np.uint16)
    rows = x.shape[0]
    W, s, b = _c(W, np.uint32), _c(scales, np.uint16), _c(biases, np.uint16)
    if cols is None:
        cptr, ncols = None, N
    else:
        cols = _c(cols, np.int64)
        cptr, ncols = _p(cols), cols.size
    y = np.empty((rows, ncols), dtype=np.float64)
    a = np.empty((rows, ncols), dtype=np.float64)
    rc = lib().oracle_qmm(_p(x), rows, K, _p(W), _p(s), _p(b), N, bits, group,
                          cptr, ncols, _p(y), _p(a), nthreads)
    if rc:
        raise OracleError(rc)
    return y, a


def widen(W, scales, biases, N, K, bits, group, bits_out, group_out):
    """(W_out, s_out, b_out) or raises OracleError(ENARROW / EGROUP / EINVAL)."""
    W, s, b = _c(W, np.uint32), _c(scales, np.uint16), _c(biases, np.uint16)
    Wo = np.zeros((N, K * bits_out // 32), dtype=np.uint32)
    so = np.zeros((N, K // group_out), dtype=np.uint16)
    bo = np.zeros((N, K // group_out), dtype=np.uint16)
    rc = lib().oracle_widen(_p(W), _p(s), _p(b), N, K, bits, group, _p(Wo), _p(so), _p(bo),
                            bits_out, group_out)
    if rc:
        raise OracleError(rc)
    return Wo, so, bo


def common_width(bits_list, groups_list):
    bl, gl = _c(bits_list, np.int32), _c(groups_list, np.int32)
    bo, go = np.zeros(1, np.int32), np.zeros(1, np.int32)
    rc = lib().oracle_common_width(_p(bl), _p(gl), bl.size, _p(bo), _p(go))
    if rc:
        raise OracleError(rc)
    return int(bo[0]), int(go[0])


# fp32-summation bound used for every floating-point comparison:
# |y - y64| <= (K * 2**-24 + 2**-20) * sum_k |x_k * w_k|.
def bound(absum: np.ndarray, K: int) -> np.ndarray:
    return (K * 2.0 ** -24 + 2.0 ** -20) * absum


def relu2(y: np.ndarray) -> np.ndarray:
    """max(y, 0)^2 elementwise, in fp64 (the squared-ReLU output epilogue)."""
    y = _c(y, np.float64)
    out = np.empty_like(y)
    lib().oracle_relu2(_p(y), y.size, _p(out))
    return out


def bf16_ulp(a: np.ndarray) -> np.ndarray:
    """One bf16 ulp at magnitude a (8 significant bits; 0 where a == 0)."""
    a = np.abs(np.asarray(a, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 7), 0.0)


def bound_out(y64: np.ndarray, absum: np.ndarray, K: int, relu2_epi: bool, bf16_out: bool):
    """(target, bound) of an output with options, from the fp32 bound B of the
    product v: squared ReLU moves the error to B*(2|v| + B) plus one fp32
    rounding of the square; a bf16 output adds one bf16 ulp (as the pages bound
    bf16 outputs)."""
    B = bound(absum, K)
    t, Bt = y64, B
    if relu2_epi:
        t = relu2(y64)
        Bt = B * (2 * np.abs(y64) + B) + 2.0 ** -24 * (np.maximum(y64, 0) + B) ** 2
    if bf16_out:
        Bt = Bt + bf16_ulp(np.abs(t) + Bt)
    return t, Bt
