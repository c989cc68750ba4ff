"""Failure detection without a GPU fault: a withheld stage makes the kernel's
bounded wait run out; the kernel records it in the device status word and
completes, the host reads TF_EDEVICE, and the next call is correct again."""
import pytest
import torch

import synth
import mlx_affine_bit_gb300 as tf
from tests.gpu_util import DevMatrix, dev, oracle_check, run_qmm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("N,K,bits,group", [(256, 1024, 4, 64), (40, 96, 3, 32)])
def test_bounded_wait_runs_out_and_is_reported(N, K, bits, group):
    m = synth.make_matrix(N, K, bits, group, 160, 0.001, 0.03)
    dm = DevMatrix(m)
    x = synth.make_x(2, K, 161)
    xd = dev(x)
    torch.cuda.synchronize()
    tf.tf_device_status()                      # starts clean
    tf.tf_inject_stall()
    run_qmm(dm, xd)                            # its first stage never arrives: about 2 s
    torch.cuda.synchronize()
    with pytest.raises(tf.TfError) as e:
        tf.tf_device_status()
    assert e.value.rc == -11
    tf.tf_device_status()                      # reading cleared it
    y = run_qmm(dm, xd)                        # the context is usable and the next call right
    torch.cuda.synchronize()
    tf.tf_device_status()
    oracle_check(m, x, y.cpu().numpy())
