"""Helpers for the GPU parity tests: device copies, calls through the C ABI,
and comparison with the fp64 oracle."""
import numpy as np
import torch

import oracle
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


def oracle_check(m, x: np.ndarray, y_gpu: np.ndarray, cols=None) -> float:
    """Worst |y - y64| / bound over the given columns (all if None); asserts <= 1."""
    y64, absum = oracle.qmm(x, m.W, m.scales, m.biases, m.N, m.K, m.bits, m.group, cols=cols,
                            nthreads=8)
    yg = y_gpu if cols is None else y_gpu[:, cols]
    err = np.abs(yg.astype(np.float64) - y64)
    ratio = err / oracle.bound(absum, m.K)
    worst = float(np.max(ratio))
    assert np.all(np.isfinite(yg)), "non-finite GPU output"
    assert worst <= 1.0, "worst err/bound %.4f" % worst
    return worst


def control_ratio(m, x: np.ndarray, y_gpu: np.ndarray, cols=None) -> float:
    """Max over columns of |y_gpu - y64(scales*1.01)| / bound: the 1%-off control."""
    zero = np.zeros_like(m.biases)
    y64, absum = oracle.qmm(x, m.W, m.scales, m.biases, m.N, m.K, m.bits, m.group, cols=cols,
                            nthreads=8)
    ysq, _ = oracle.qmm(x, m.W, m.scales, zero, m.N, m.K, m.bits, m.group, cols=cols, nthreads=8)
    yg = y_gpu if cols is None else y_gpu[:, cols]
    return float(np.max(np.abs(yg - (y64 + 0.01 * ysq)) / oracle.bound(absum, m.K)))


def sample_cols(N: int, n: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    c = set(rng.choice(N, size=min(n, N), replace=False).tolist())
    c.update([0, N - 1, min(N - 1, 127), min(N - 1, 128)])
    return np.array(sorted(c), dtype=np.int64)
