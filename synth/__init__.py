"""Seeded synthetic inputs shared by the tests, the bench and the smoke check.

This module holds random-number generation and the workload recipes only.  It
contains none of the quantized product's arithmetic: it never decodes a code,
dequantizes a weight or forms a dot product, and neither the oracle nor the
CUDA library imports it.

Generator
---------
SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014; the constants are those of Vigna's public-domain
``splitmix64.c``).  Output ``i`` (0-based) of a stream whose state starts at
``base`` is ``mix(base + (i + 1) * GAMMA)``, so a stream is counter based and
is evaluated vectorised with numpy.  Each array of a workload draws from its
own stream: ``base = mix(seed * GAMMA ^ tag)``.

Value recipes
-------------
* uniform ``U(lo, hi)``: ``u = (r >> 11) * 2**-53`` in fp64, ``lo + (hi-lo)*u``.
* normal ``N(0, 1)``: Box-Muller, ``sqrt(-2 ln(1-u1)) * cos(2 pi u2)`` from the
  even and odd outputs of one stream, in fp64.
* every real value is rounded fp64 -> fp32 (numpy's round-to-nearest-even
  cast) and then fp32 -> bf16 (round to nearest even on the bit pattern).
* packed codes: codes drawn i.i.d. uniform on ``[0, 2**bits)`` and packed low
  code first into a contiguous little-endian bitstream have i.i.d. uniform
  bits, so a packed row is drawn directly as uniform 32-bit words (each 64-bit
  output gives its low word, then its high word).  That is exactly the
  distribution the workloads call for, with no packer in the generator.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# Stream tags: one independent stream per array of a workload.
TAG_W, TAG_SCALE, TAG_BIAS_U, TAG_X = 1, 2, 3, 4

BITS = (2, 3, 4, 5, 6, 8)
GROUPS = (32, 64, 128)


def _mix(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _base(seed: int, tag: int) -> np.uint64:
    with np.errstate(over="ignore"):
        s = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) * GAMMA ^ np.uint64(tag)
    return _mix(np.array([s], dtype=np.uint64))[0]


def draws(seed: int, tag: int, n: int, start: int = 0) -> np.ndarray:
    """Outputs ``start .. start+n-1`` of stream (seed, tag) as uint64."""
    base = _base(seed, tag)
    idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(base + idx * GAMMA)


def uniform01(seed: int, tag: int, n: int, start: int = 0) -> np.ndarray:
    r = draws(seed, tag, n, start)
    return (r >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(seed: int, tag: int, n: int) -> np.ndarray:
    u = uniform01(seed, tag, 2 * n)
    u1, u2 = u[0::2], u[1::2]
    return np.sqrt(-2.0 * np.log1p(-u1)) * np.cos(2.0 * math.pi * u2)


def f32_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest even) and return the uint16 patterns."""
    b = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))
    return (r >> np.uint64(16)).astype(np.uint16)


def to_bf16(v64: np.ndarray) -> np.ndarray:
    return f32_to_bf16_bits(np.asarray(v64, dtype=np.float64).astype(np.float32))


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """bf16 patterns -> fp32 values (exact: the pattern is the top half)."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def packed_words(seed: int, n_rows: int, words_per_row: int) -> np.ndarray:
    n = n_rows * words_per_row
    r = draws(seed, TAG_W, (n + 1) // 2)
    w = np.empty(2 * r.size, dtype=np.uint32)
    w[0::2] = (r & np.uint64(0xFFFFFFFF)).astype(np.uint32)
    w[1::2] = (r >> np.uint64(32)).astype(np.uint32)
    return w[:n].reshape(n_rows, words_per_row)


@dataclass
class Matrix:
    """One MLX-affine quantized matrix: W [N][K*bits/32] u32, scales/biases [N][K/G] bf16."""
    N: int
    K: int
    bits: int
    group: int
    W: np.ndarray
    scales: np.ndarray
    biases: np.ndarray
    seed: int = 0


def make_matrix(N: int, K: int, bits: int, group: int, seed: int,
                scale_lo: float, scale_hi: float,
                bias_mult: float | None = None,
                bias_u: tuple[float, float] = (0.9, 1.1)) -> Matrix:
    """Seeded synthetic matrix.

    ``bias = -scale * bias_mult * U(bias_u)`` with ``bias_mult`` defaulting to
    ``2**(bits-1)``; the product is formed from the fp32 scale before that is
    rounded to bf16, and then rounded itself.
    """
    assert K % group == 0 and (K * bits) % 32 == 0
    ng = N * (K // group)
    W = packed_words(seed, N, K * bits // 32)
    s32 = (scale_lo + (scale_hi - scale_lo) * uniform01(seed, TAG_SCALE, ng)).astype(np.float32)
    mult = float(2 ** (bits - 1)) if bias_mult is None else float(bias_mult)
    u = bias_u[0] + (bias_u[1] - bias_u[0]) * uniform01(seed, TAG_BIAS_U, ng)
    b64 = -s32.astype(np.float64) * mult * u
    return Matrix(N, K, bits, group, W,
                  f32_to_bf16_bits(s32).reshape(N, K // group),
                  to_bf16(b64).reshape(N, K // group), seed)


def make_x(rows: int, K: int, seed: int) -> np.ndarray:
    """bf16 activations x ~ N(0,1), [rows][K] uint16 patterns."""
    return to_bf16(normal(seed, TAG_X, rows * K)).reshape(rows, K)


# ----------------------------------------------------------------------------
# Workloads: the shapes, sizes and value distributions of the pages' checks.
# ----------------------------------------------------------------------------

def single_matrix():
    """N=256, K=1024, 4-bit g64, one row, seed 0; bias = -8*s*U(0.8,1.2)."""
    m = make_matrix(256, 1024, 4, 64, 0, 0.002, 0.02, bias_mult=8.0, bias_u=(0.8, 1.2))
    return m, make_x(1, 1024, 0)


def width_sweep_cases():
    """(bits, group, seed) of the 4096x4096 one-row sweep; seeds 1..18 bits-major."""
    out, seed = [], 1
    for b in BITS:
        for g in GROUPS:
            out.append((b, g, seed))
            seed += 1
    return out


def width_sweep_matrix(bits: int, group: int, seed: int, N: int = 4096, K: int = 4096):
    return make_matrix(N, K, bits, group, seed, 0.001, 0.03)


DECODE_SHAPES = ((12288, 2048, 19), (2048, 12288, 20))   # (N, K, seed), 6-bit g32
DECODE_ROWS = (1, 2, 3, 8, 16)


def decode_matrix(N: int, K: int, seed: int):
    return make_matrix(N, K, 6, 32, seed, 0.001, 0.03)


@dataclass
class StackMember:
    bits: int
    group: int
    n_cols: int
    seed: int


# The mixed-width fused projection (4/64, 5/128, 5/128, 6/64).  The first three
# members widen and regroup to one 5-bit g64 run of 6192 columns (not a
# multiple of 32, so it runs untiled); the last is a 6-bit g64 run of 48
# columns; the output row stride is 6240.
STACK_MEMBERS = (StackMember(4, 64, 4096, 21), StackMember(5, 128, 2048, 22),
                 StackMember(5, 128, 48, 23), StackMember(6, 64, 48, 24))
STACK_K = 2048
STACK_ROWS = (1, 16)


def stack_member_matrices(K: int = STACK_K, members=STACK_MEMBERS):
    return [make_matrix(m.n_cols, K, m.bits, m.group, m.seed, 0.001, 0.03) for m in members]


LMHEAD_N = 248320
LMHEAD_K = 2048
LMHEAD_CASES = ((6, 32, 31), (4, 64, 32))
LMHEAD_ROWS = (1, 16)


def lmhead_matrix(bits: int, group: int, seed: int, N: int = LMHEAD_N, K: int = LMHEAD_K):
    return make_matrix(N, K, bits, group, seed, 0.001, 0.02)


def algorithmic_bytes(N: int, K: int, bits: int, group: int, rows: int) -> int:
    """Codes + scales/biases + x + y bytes of one product."""
    return N * K * bits // 8 + N * (K // group) * 4 + rows * K * 2 + rows * N * 4
