"""Out-of-bounds evidence without a sanitizer: the bounds-checking debug build
(libtfqmm_debug.so, TF_DEBUG_BOUNDS) checks every shared- and global-memory
index its kernels compute and reports a violation as TF_EBOUNDS, and guard
bands of sentinel words after every output buffer stay untouched.

The edge shapes are the ones where an index is most likely to slip: one
column, ragged column tails (17, 33, 6192), K of one group or not a multiple
of a stage (32, 96, 1536), 3- and 5-bit rows whose 32-wide groups are an odd
number of words (TensorFold PR #788, the lane-kernel formats commit), split K,
stacks with a column map, gathers, windows past 16 rows and bf16 outputs.
"""
import contextlib

import numpy as np
import pytest
import torch

import synth
import mlx_affine_bit_gb300 as tf
from tests.gpu_util import DEV, DevMatrix, dev, oracle_check

pytestmark = pytest.mark.gpu

GUARD = 64                    # sentinel words after each output buffer
SENT = -7777.25


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.synchronize()
    tf.tf_device_status()
    with use(tf.debug_lib()):
        tf.tf_device_status()


@contextlib.contextmanager
def use(L):
    """Route the binding's calls to library build L for the block."""
    old = tf._lib
    tf._lib = L
    try:
        yield
    finally:
        tf._lib = old


def guarded_y(rows, stride, dtype=torch.float32):
    """y of rows x stride elements followed by GUARD sentinel elements."""
    buf = torch.full((rows * stride + GUARD,), SENT if dtype == torch.float32 else -3, dtype=dtype, device=DEV)
    return buf, buf[:rows * stride].view(rows, stride)


def check_guard(buf, n, dtype=torch.float32):
    tail = buf[n:]
    want = SENT if dtype == torch.float32 else -3
    assert torch.all(tail == want), "guard band written"


def product(dm, xd, rows, stride=None, flags=0):
    m = dm.m
    stride = m.N if stride is None else stride
    dt = torch.int16 if flags & tf.TF_OUT_BF16 else torch.float32
    buf, y = guarded_y(rows, stride, dt)
    tf.tf_qmm_ex(xd, rows, m.K, dm.W, dm.s, dm.b, m.N, m.bits, m.group, y, stride, flags)
    torch.cuda.synchronize()
    check_guard(buf, rows * stride, dt)
    return y


EDGE = [(1, 32, 3, 32, 1), (17, 96, 5, 32, 2), (33, 1536, 3, 32, 3), (33, 1536, 5, 32, 16), (6192, 2048, 5, 64, 1),
        (6192, 2048, 3, 32, 16), (17, 1536, 5, 128, 5), (2048, 12288, 6, 32, 16), (2048, 12288, 3, 32, 1),
        (300, 4096, 8, 64, 9), (129, 4096, 2, 128, 1), (4096, 4096, 4, 64, 2)]


@pytest.mark.parametrize("N,K,bits,group,rows", EDGE)
@pytest.mark.parametrize("mode", [0, 6])
def test_debug_build_edge_shapes(N, K, bits, group, rows, mode):
    # Every index in range (no TF_EBOUNDS), the same bits as the release
    # build, within the oracle bound, and the guard band after y untouched.
    m = synth.make_matrix(N, K, bits, group, 600 + N % 97 + K % 89 + bits, 0.001, 0.03)
    dm = DevMatrix(m)
    x = synth.make_x(rows, K, 601 + rows)
    xd = dev(x)
    stride = N + 3
    old = tf.tf_set_launch_mode(mode)
    try:
        ref = product(dm, xd, rows, stride)
        with use(tf.debug_lib()):
            old_d = tf.tf_set_launch_mode(mode)
            got = product(dm, xd, rows, stride)
            tf.tf_set_launch_mode(old_d)
            tf.tf_device_status()
    finally:
        tf.tf_set_launch_mode(old)
    assert torch.equal(got.view(torch.int32), ref.view(torch.int32))
    assert torch.all(got[:, N:] == SENT)                     # the stride gap
    oracle_check(m, x, got[:, :N].cpu().numpy())


def test_debug_build_stack_gather_windows_options_noalloc():
    K = 2048
    mats = [synth.make_matrix(N, K, b, g, 620 + i, 0.001, 0.03)
            for i, (N, b, g) in enumerate([(4096, 4, 64), (48, 6, 64), (2000, 3, 128), (17, 5, 32)])]
    dms = [DevMatrix(m) for m in mats]
    x = synth.make_x(40, K, 621)
    xd = dev(x)
    runs = [(dm.W, dm.s, dm.b, m.N, m.bits, m.group) for dm, m in zip(dms, mats)]
    total = sum(m.N for m in mats)
    members, off = [], 0
    for i, m in enumerate(mats):
        members.append((i, 0, m.N, off))
        off += m.N
    se = [i % 4 for i in range(21)]
    sr = [(7 * i) % 40 for i in range(21)]

    def calls():
        out = []
        buf, y = guarded_y(3, total)
        tf.tf_qmm_stack(xd, 3, K, runs, members, y, total)
        out.append((buf, y, 3 * total, torch.float32))
        buf, y = guarded_y(21, 4096)
        tf.tf_qmm_gather(xd, 40, K, runs, se, sr, y, 4096, 0)
        out.append((buf, y, 21 * 4096, torch.float32))
        m, dm = mats[2], dms[2]
        buf, y = guarded_y(40, m.N, torch.int16)
        tf.tf_qmm_ex(xd, 40, K, dm.W, dm.s, dm.b, m.N, m.bits, m.group, y, m.N, tf.TF_OUT_BF16 | tf.TF_EPI_RELU2)
        out.append((buf, y, 40 * m.N, torch.int16))
        buf, y = guarded_y(17, m.N)
        tf.tf_qmm_noalloc(xd[:17].contiguous(), 17, K, dm.W, dm.s, dm.b, m.N, m.bits, m.group, y, m.N)
        out.append((buf, y, 17 * m.N, torch.float32))
        torch.cuda.synchronize()
        for buf, y, n, dt in out:
            check_guard(buf, n, dt)
        return [y for (_, y, _, _) in out]

    ref = calls()
    with use(tf.debug_lib()):
        got = calls()
        tf.tf_device_status()
        tf.tf_noalloc_status()
    for a, b in zip(ref, got):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_bounds_checker_reports_and_skips():
    # The checker is live: with y declared two rows short, the stores to the
    # last two rows fail the check, are skipped (the caller's memory keeps its
    # sentinel) and are reported as TF_EBOUNDS; the next call is clean.
    m = synth.make_matrix(300, 1024, 5, 64, 640, 0.001, 0.03)
    dm = DevMatrix(m)
    xd = dev(synth.make_x(5, 1024, 641))
    L = tf.debug_lib()
    with use(L):
        assert L.tf_debug_shrink_y(2) == 0
        buf, y = guarded_y(5, 300)
        tf.tf_qmm(xd, 5, 1024, dm.W, dm.s, dm.b, 300, 5, 64, y, 300)
        torch.cuda.synchronize()
        with pytest.raises(tf.TfError) as e:
            tf.tf_device_status()
        assert e.value.rc == -14
        assert torch.all(y[3:] == SENT) and not torch.any(y[:3] == SENT)
        tf.tf_qmm(xd, 5, 1024, dm.W, dm.s, dm.b, 300, 5, 64, y, 300)
        torch.cuda.synchronize()
        tf.tf_device_status()
        assert not torch.any(y == SENT)
        check_guard(buf, 5 * 300)


@pytest.mark.parametrize("b0,g0,b1,g1", [(3, 32, 5, 32), (5, 128, 6, 64), (2, 64, 8, 32)])
def test_widen_guard_bands(b0, g0, b1, g1):
    # tf_widen writes exactly W_out, s_out and b_out: the sentinel words after
    # each stay untouched (both builds).
    N, K = 37, 96 if g0 == 32 else 384
    m = synth.make_matrix(N, K, b0, g0, 650 + b0, 0.001, 0.03)
    dm = DevMatrix(m)
    for L in (tf.lib(), tf.debug_lib()):
        nw, ng = N * K * b1 // 32, N * (K // g1)
        Wb = torch.full((nw + GUARD,), -5, dtype=torch.int32, device=DEV)
        sb = torch.full((ng + GUARD,), -5, dtype=torch.int16, device=DEV)
        bb = torch.full((ng + GUARD,), -5, dtype=torch.int16, device=DEV)
        with use(L):
            tf.tf_widen(dm.W, dm.s, dm.b, N, K, b0, g0, Wb[:nw], sb[:ng], bb[:ng], b1, g1)
            torch.cuda.synchronize()
            tf.tf_device_status()
        assert torch.all(Wb[nw:] == -5) and torch.all(sb[ng:] == -5) and torch.all(bb[ng:] == -5)
        want = tf.tf_widen_host(m.W, m.scales, m.biases, N, K, b0, g0, b1, g1)
        assert np.array_equal(Wb[:nw].cpu().numpy().view(np.uint32), want[0].reshape(-1))
        assert np.array_equal(sb[:ng].cpu().numpy().view(np.uint16), want[1].reshape(-1))
