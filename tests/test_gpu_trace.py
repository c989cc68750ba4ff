"""The phase-trace build (libtfqmm_trace.so, TF_TRACE): one record per CTA of
every row-kernel launch, its phases in order, and products bit-identical to the
product library's."""
import numpy as np
import pytest
import torch

import synth
import mlx_affine_bit_gb300 as tf
from mlx_affine_bit_gb300 import build
from tests.gpu_util import DEV, DevMatrix, dev, run_qmm

pytestmark = pytest.mark.gpu

ENTER, TMA0, LAND0, RELEASE, XLOADED, STAGE0, EXIT = range(2, 9)


@pytest.fixture(scope="module")
def trace_lib():
    import __graft_entry__
    __graft_entry__.build()
    build.build_trace()
    return tf.trace_lib()


@pytest.mark.parametrize("mode", [0, tf.TF_LAUNCH_EARLY_WEIGHTS, tf.TF_LAUNCH_EARLY_WEIGHTS | tf.TF_LAUNCH_EARLY_X])
def test_trace_records(trace_lib, mode):
    shapes = [(4096, 4096, 2, 32, 1), (300, 2048, 6, 32, 3), (12288, 2048, 4, 64, 16)]
    mats = [DevMatrix(synth.make_matrix(N, K, b, g, 900 + i, 0.001, 0.03)) for i, (N, K, b, g, r) in enumerate(shapes)]
    xs = [dev(synth.make_x(r, K, 910 + i)) for i, (N, K, b, g, r) in enumerate(shapes)]
    want = [run_qmm(dm, xd) for dm, xd in zip(mats, xs)]
    L = trace_lib
    with tf.using(L):
        old = tf.tf_set_launch_mode(mode)
        try:
            assert L.tf_trace_reset() == 0
            got = [run_qmm(dm, xd) for dm, xd in zip(mats, xs)]
            torch.cuda.synchronize()
            tf.tf_device_status()
        finally:
            tf.tf_set_launch_mode(old)
        buf = np.zeros((1 << 16, 9), dtype=np.uint64)
        n = L.tf_trace_read(buf.ctypes.data, buf.shape[0])
    for a, b in zip(want, got):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert n > 0
    buf = buf[:n].astype(np.int64)
    seqs = sorted(set(buf[:, 0].tolist()))
    assert seqs == list(range(len(shapes)))            # one launch each, numbered in order
    for s in seqs:
        r = buf[buf[:, 0] == s]
        blocks = (r[:, 1] & 0xFFFFFFFF).tolist()
        assert len(blocks) == len(set(blocks))          # one record per CTA
        assert np.all(r[:, ENTER] > 0) and np.all(r[:, EXIT] >= r[:, ENTER])
        assert np.all(r[:, RELEASE] > 0) and np.all(r[:, RELEASE] <= r[:, EXIT])
        w = r[r[:, XLOADED] > 0]                        # CTAs that had an item
        assert len(w) > 0
        landed = w[w[:, LAND0] > 0]                     # the producer waited for its first stage
        assert np.all(landed[:, LAND0] >= landed[:, TMA0]) and np.all(w[:, TMA0] >= w[:, ENTER])
        assert np.all(w[:, XLOADED] >= w[:, ENTER]) and np.all(w[:, STAGE0] >= w[:, XLOADED])
        assert np.all(w[:, EXIT] >= w[:, STAGE0])
