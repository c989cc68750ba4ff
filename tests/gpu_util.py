"""Helpers for the GPU parity tests: device copies, calls through the C ABI,
and comparison with the fp64 oracle."""
import os

import numpy as np
import torch

import oracle
import synth
import mlx_affine_bit_gb300 as tf

DEV = torch.device("cuda:0")


def dev(a: np.ndarray) -> torch.Tensor:
    """numpy bit patterns -> device tensor of the same width (int16/int32)."""
    a = np.ascontiguousarray(a)
    view = {np.dtype(np.uint16): np.int16, np.dtype(np.uint32): np.int32}[a.dtype]
    return torch.from_numpy(a.view(view)).to(DEV)


class DevMatrix:
    def __init__(self, m):
        self.m = m
        self.W, self.s, self.b = dev(m.W), dev(m.scales), dev(m.biases)


def run_qmm(dm: DevMatrix, xd: torch.Tensor, y_stride=None, fill=float("nan"), y=None):
    m = dm.m
    rows = xd.shape[0]
    ys = m.N if y_stride is None else y_stride
    if y is None:
        y = torch.full((rows, ys), fill, dtype=torch.float32, device=DEV)
    tf.tf_qmm(xd, rows, m.K, dm.W, dm.s, dm.b, m.N, m.bits, m.group, y, ys)
    return y


NTHREADS = os.cpu_count() or 8


def _bias_part(m, x: np.ndarray, cols) -> np.ndarray:
    """sum_g bias[n][g] * sum_{k in g} x[r][k] in fp64, [rows][ncols]: the part of
    the product that does not scale with the scales (for the 1%-off control)."""
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    sx = xf.reshape(x.shape[0], m.K // m.group, m.group).sum(axis=2)
    b = synth.bf16_bits_to_f32(m.biases if cols is None else m.biases[cols]).astype(np.float64)
    return sx @ b.T


def oracle_check(m, x: np.ndarray, y_gpu: np.ndarray, cols=None, control: bool = False):
    """Worst |y - y64| / bound over the given columns (all if None); asserts <= 1.

    With control=True also returns the 1%-off negative control (TensorFold PR
    #788, tf-affine-ref commit: a reference whose scales are 1 % off must fail
    the bound): the max over the columns of |y_gpu - y64(scales * 1.01)| / bound,
    asserted > 1.  y64(scales * 1.01) = y64 + 0.01 * (y64 - bias part) exactly
    in real arithmetic.  Returns worst, or (worst, control)."""
    y64, absum = oracle.qmm(x, m.W, m.scales, m.biases, m.N, m.K, m.bits, m.group, cols=cols,
                            nthreads=NTHREADS)
    yg = (y_gpu if cols is None else y_gpu[:, cols]).astype(np.float64)
    assert np.all(np.isfinite(yg)), "non-finite GPU output"
    B = oracle.bound(absum, m.K)
    worst = float(np.max(np.abs(yg - y64) / B))
    assert worst <= 1.0, "worst err/bound %.4f" % worst
    if not control:
        return worst
    ysq = y64 - _bias_part(m, x, cols)
    ctrl = float(np.max(np.abs(yg - (y64 + 0.01 * ysq)) / B))
    assert ctrl > 1.0, "1%%-off control stays inside the bound (max ratio %.3f)" % ctrl
    return worst, ctrl


def full_cols(N: int, seed: int):
    """All columns (None) unless TFQ_PARITY_COLS=n asks for a sample of n."""
    n = os.environ.get("TFQ_PARITY_COLS")
    return None if not n else sample_cols(N, int(n), seed)


def sample_cols(N: int, n: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    c = set(rng.choice(N, size=min(n, N), replace=False).tolist())
    c.update([0, N - 1, min(N - 1, 127), min(N - 1, 128)])
    return np.array(sorted(c), dtype=np.int64)
