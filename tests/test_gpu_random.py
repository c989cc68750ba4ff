"""Seeded random shapes through the C ABI against the fp64 oracle: widths,
groups, odd column counts, K that is not a multiple of 256 (the producer's
plain-copy path), 1-20 rows, strides and output options; one row of every
case is also checked against the same row computed alone."""
import os

import numpy as np
import pytest
import torch

import oracle
import synth
import mlx_affine_bit_gb300 as tf
from tests.gpu_util import DEV, DevMatrix, dev, sample_cols

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    yield
    torch.cuda.synchronize()
    tf.tf_device_status()


def _cases(n=None, seed=2024):
    # TFQ_RANDOM_CASES widens the sample (40 by default, so the suite stays quick).
    n = int(os.environ.get("TFQ_RANDOM_CASES", "40")) if n is None else n
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        bits = int(rng.choice([2, 3, 4, 5, 6, 8]))
        group = int(rng.choice([32, 64, 128]))
        K = group * int(rng.integers(1, 6144 // group + 1))
        N = int(rng.integers(1, 5000))
        rows = int(rng.choice([1, 1, 2, 3, 5, 8, 11, 16, 20]))
        pad = int(rng.choice([0, 0, 3, 64]))
        flags = int(rng.choice([0, 0, 1, 2, 3]))
        out.append((i, bits, group, K, N, rows, pad, flags))
    return out


@pytest.mark.parametrize("i,bits,group,K,N,rows,pad,flags", _cases())
def test_random_shape(i, bits, group, K, N, rows, pad, flags):
    m = synth.make_matrix(N, K, bits, group, 500 + i, 0.001, 0.03)
    dm = DevMatrix(m)
    x = synth.make_x(rows, K, 600 + i)
    xd = dev(x)
    bf = bool(flags & tf.TF_OUT_BF16)
    stride = N + pad
    fill = -9 if bf else float("nan")
    y = torch.full((rows, stride), fill, dtype=torch.int16 if bf else torch.float32, device=DEV)
    tf.tf_qmm_ex(xd, rows, K, dm.W, dm.s, dm.b, N, bits, group, y, stride, flags)
    r = rows // 2
    one = torch.full((1, N), fill, dtype=y.dtype, device=DEV)
    tf.tf_qmm_ex(xd[r:r + 1].contiguous(), 1, K, dm.W, dm.s, dm.b, N, bits, group, one, N, flags)
    assert torch.equal(y[r, :N], one[0])
    if pad:
        tail = y[:, N:]
        assert torch.all(tail == -9) if bf else torch.all(torch.isnan(tail))
    cols = sample_cols(N, 32, i)
    y64, absum = oracle.qmm(x, m.W, m.scales, m.biases, N, K, bits, group, cols=cols, nthreads=8)
    t, B = oracle.bound_out(y64, absum, K, bool(flags & tf.TF_EPI_RELU2), bf)
    if bf:
        h = y[:, cols].cpu().numpy().view(np.uint16).astype(np.uint32) << 16
        got = h.view(np.float32).astype(np.float64)
    else:
        got = y[:, cols].cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    assert np.all(np.abs(got - t) <= B), float(np.max(np.abs(got - t) / np.maximum(B, 1e-300)))
