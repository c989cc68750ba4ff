"""tf_qmm_noalloc: the product for callers that cannot let a library allocate
device memory (graph capture, engines that pool all memory up front, fixed
footprints).  It must give exactly what tf_qmm gives, call after call, while
its scratch comes from the fixed array built into the library.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import synth
import mlx_affine_bit_gb300 as tf
from tests.gpu_util import DEV, DevMatrix, dev, oracle_check, run_qmm, sample_cols

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def _noalloc(dm, xd):
    m = dm.m
    rows = xd.shape[0]
    y = torch.full((rows, m.N), float("nan"), dtype=torch.float32, device=DEV)
    tf.tf_qmm_noalloc(xd, rows, m.K, dm.W, dm.s, dm.b, m.N, m.bits, m.group, y, m.N)
    return y


# (N, K, bits, group, rows): split-K shapes use the fixed scratch; the others don't.
CASES = [(2048, 12288, 6, 32, 16), (2048, 12288, 4, 64, 1), (4096, 4096, 3, 128, 3),
         (300, 2048, 5, 64, 2)]


@pytest.mark.parametrize("N,K,bits,group,rows", CASES)
def test_noalloc_matches_tf_qmm_twice(N, K, bits, group, rows):
    m = synth.make_matrix(N, K, bits, group, 400 + bits, 0.001, 0.03)
    dm = DevMatrix(m)
    x = synth.make_x(rows, K, 401 + rows)
    xd = dev(x)
    ref = run_qmm(dm, xd)
    for _ in range(2):                       # two calls in a row share the scratch
        got = _noalloc(dm, xd)
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int32), ref.view(torch.int32))
    oracle_check(m, x, got.cpu().numpy(), sample_cols(N, 24, 5))


def test_noalloc_refuses_beyond_its_scratch():
    # 16 rows x 16384 columns x 6 chunks of split-K partials (6.3 MB) is beyond
    # the fixed scratch: refused on the host before any launch.  The buffers
    # are real and as large as the shape claims, so even a planner that chose
    # not to split K here would launch on valid memory.
    N, K, bits, group, rows = 16384, 12288, 2, 32, 16
    W = torch.zeros((N, K * bits // 32), dtype=torch.int32, device=DEV)
    s = torch.zeros((N, K // group), dtype=torch.int16, device=DEV)
    x = torch.zeros((rows, K), dtype=torch.int16, device=DEV)
    y = torch.zeros((rows, N), dtype=torch.float32, device=DEV)
    with pytest.raises(tf.TfError) as e:
        tf.tf_qmm_noalloc(x, rows, K, W, s, s, N, bits, group, y, N)
    assert e.value.rc == -6 and "scratch" in str(e.value)
    torch.cuda.synchronize()


@pytest.mark.parametrize("rows", [17, 40])
def test_noalloc_rows_past_16(rows):
    # More than 16 rows run as 16-row windows over the shared scratch (split K
    # at 2048 x 12288): the same bits as tf_qmm, twice in a row.
    m = synth.make_matrix(2048, 12288, 5, 64, 420 + rows, 0.001, 0.03)
    dm = DevMatrix(m)
    x = synth.make_x(rows, m.K, 421 + rows)
    xd = dev(x)
    ref = run_qmm(dm, xd)
    for _ in range(2):
        got = _noalloc(dm, xd)
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int32), ref.view(torch.int32))
    oracle_check(m, x, got.cpu().numpy(), sample_cols(m.N, 16, rows))


def test_noalloc_reports_a_bounded_wait_that_ran_out():
    # A withheld first stage (test hook) makes the kernel's bounded wait run
    # out: tf_noalloc_status reports TF_EDEVICE once, and the next call is right.
    m = synth.make_matrix(256, 1024, 4, 64, 430, 0.001, 0.03)
    dm = DevMatrix(m)
    x = synth.make_x(2, m.K, 431)
    xd = dev(x)
    torch.cuda.synchronize()
    tf.tf_noalloc_status()                     # starts clean
    tf.tf_inject_stall()
    _noalloc(dm, xd)                           # about 2 s: the first stage never arrives
    torch.cuda.synchronize()
    with pytest.raises(tf.TfError) as e:
        tf.tf_noalloc_status()
    assert e.value.rc == -11
    tf.tf_noalloc_status()                     # reading cleared it
    ref = run_qmm(dm, xd)
    got = _noalloc(dm, xd)
    torch.cuda.synchronize()
    tf.tf_noalloc_status()
    assert torch.equal(got.view(torch.int32), ref.view(torch.int32))
    oracle_check(m, x, got.cpu().numpy())
