"""tf_qmm_prompt: the many-row product on the tcgen05 tensor cores.

Bars (TensorFold PR #788, the 2-bit affine_mm and tf-affine-ref commits, which gate
the prompt-side product row by row against windows of 1 to 65 rows):
  (i)  every output within (K*2^-24 + 2^-20) * sum|x*w| of the fp64 product, with
       the 1%-off negative control outside it;
  (ii) every row of a 129-row call equals the same row computed in windows of 1, 2,
       3, 8, 16, 17, 33, 64 and 65 rows, bit for bit, at every window position;
  (iii) strided and bf16 / squared-ReLU outputs equal the contiguous fp32 result's.
"""
import numpy as np
import pytest
import torch

import synth
import mlx_affine_bit_gb300 as tf
from tests.gpu_util import DEV, DevMatrix, dev, full_cols, oracle_check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    yield
    torch.cuda.synchronize()
    tf.tf_device_status()


def prompt(dm, xd, stride=None, flags=0, fill=float("nan")):
    m = dm.m
    rows = xd.shape[0]
    stride = m.N if stride is None else stride
    dt = torch.int16 if flags & tf.TF_OUT_BF16 else torch.float32
    y = torch.full((rows, stride), -3 if dt == torch.int16 else fill, dtype=dt, device=DEV)
    tf.tf_qmm_prompt(xd, rows, m.K, dm.W, dm.s, dm.b, m.N, m.bits, m.group, y, stride, flags)
    return y


@pytest.mark.parametrize("bits", (2, 3, 4, 5, 6, 8))
@pytest.mark.parametrize("group", (32, 64, 128))
def test_prompt_widths_full(bits, group):
    # a ragged last column tile, two K chunks, 65 rows (two windows)
    N, K, rows = 300, 4096, 65
    m = synth.make_matrix(N, K, bits, group, 800 + 3 * bits + group, 0.001, 0.03)
    x = synth.make_x(rows, K, 801 + bits)
    y = prompt(DevMatrix(m), dev(x)).cpu().numpy()
    oracle_check(m, x, y)


@pytest.mark.parametrize("N,K,bits,group,rows", [(2048, 2048, 6, 32, 64), (4096, 2048, 4, 64, 33),
                                                 (1000, 6144, 3, 128, 17)])
def test_prompt_full_size_with_control(N, K, bits, group, rows):
    m = synth.make_matrix(N, K, bits, group, 820 + bits, 0.001, 0.03)
    x = synth.make_x(rows, K, 821 + rows)
    y = prompt(DevMatrix(m), dev(x)).cpu().numpy()
    worst, ctrl = oracle_check(m, x, y, full_cols(N, bits), control=True)
    print("prompt %dx%d %d/g%d rows %d worst %.4f control %.2f" % (N, K, bits, group, rows, worst, ctrl))


@pytest.mark.parametrize("bits,group", [(6, 32), (2, 128), (5, 64)])
def test_prompt_windows_bit_exact(bits, group):
    # Every row of a 129-row call equals the same row in windows of 1..65 rows at
    # every position the window sizes allow (start every 7 rows).
    N, K, rows = 260, 2048, 129
    m = synth.make_matrix(N, K, bits, group, 840 + bits, 0.001, 0.03)
    dm = DevMatrix(m)
    x = synth.make_x(rows, K, 841)
    xd = dev(x)
    full = prompt(dm, xd)
    for w in (1, 2, 3, 8, 16, 17, 33, 64, 65):
        for p0 in list(range(0, rows - w + 1, 7)) + [rows - w]:
            yw = prompt(dm, xd[p0:p0 + w].contiguous())
            assert torch.equal(yw.view(torch.int32), full[p0:p0 + w].view(torch.int32)), (w, p0)
    oracle_check(m, x, full.cpu().numpy())


@pytest.mark.parametrize("K", [2048, 4096])   # 4096: two chunks over 3 column tiles, so split and folded
@pytest.mark.parametrize("flags", [tf.TF_EPI_RELU2, tf.TF_OUT_BF16, tf.TF_OUT_BF16 | tf.TF_EPI_RELU2])
def test_prompt_output_options_and_stride(flags, K):
    N, rows = 300, 20
    m = synth.make_matrix(N, K, 4, 64, 860, 0.001, 0.03)
    dm = DevMatrix(m)
    xd = dev(synth.make_x(rows, K, 861))
    v = prompt(dm, xd)
    if flags & tf.TF_EPI_RELU2:
        v = torch.clamp(v, min=0) * torch.clamp(v, min=0)
    want = v.to(torch.bfloat16).view(torch.int16) if flags & tf.TF_OUT_BF16 else v
    stride = N + 11
    got = prompt(dm, xd, stride=stride, flags=flags, fill=-99.0)
    if flags & tf.TF_OUT_BF16:
        assert torch.equal(got[:, :N], want)
        assert torch.all(got[:, N:] == -3)
    else:
        assert torch.equal(got[:, :N].view(torch.int32), want.view(torch.int32))
        assert torch.all(got[:, N:] == -99.0)


def test_prompt_refusals():
    m = synth.make_matrix(64, 1024, 4, 64, 870, 0.001, 0.03)
    dm = DevMatrix(m)
    xd = dev(synth.make_x(2, 1024, 871))
    y = torch.zeros((2, 64), dtype=torch.float32, device=DEV)
    with pytest.raises(tf.TfError) as e:            # K not a multiple of 2048
        tf.tf_qmm_prompt(xd, 2, 1024, dm.W, dm.s, dm.b, 64, 4, 64, y, 64, 0)
    assert e.value.rc == -6
    m2 = synth.make_matrix(64, 2048, 4, 64, 872, 0.001, 0.03)
    dm2 = DevMatrix(m2)
    xd2 = dev(synth.make_x(2, 2048, 873))
    s_off = torch.zeros(m2.scales.size + 8, dtype=torch.int16, device=DEV)[1:1 + m2.scales.size]
    with pytest.raises(tf.TfError) as e:            # scales not 16-byte aligned
        tf.tf_qmm_prompt(xd2, 2, 2048, dm2.W, s_off, dm2.b, 64, 4, 64, y, 64, 0)
    assert e.value.rc == -5


@pytest.mark.parametrize("bits,group", [(4, 64), (6, 32)])
def test_prompt_chunk_split_bit_exact(bits, group):
    # A matrix of more column tiles than SMs runs whole-K items (chunk sums in
    # registers); its first 300 columns alone run as chunk-split items whose
    # partials a fold sums.  Both follow C_0 + C_1 + ... and agree bit for bit.
    N, K, rows = 160 * 128, 6144, 40
    m = synth.make_matrix(N, K, bits, group, 880 + bits, 0.001, 0.03)
    xd = dev(synth.make_x(rows, K, 881))
    wide = prompt(DevMatrix(m), xd)
    n = 300
    sub = synth.Matrix(n, K, bits, group, np.ascontiguousarray(m.W[:n]), np.ascontiguousarray(m.scales[:n]),
                       np.ascontiguousarray(m.biases[:n]), m.seed)
    narrow = prompt(DevMatrix(sub), xd)
    assert torch.equal(narrow.view(torch.int32), wide[:, :n].view(torch.int32))
    oracle_check(sub, synth.make_x(rows, K, 881), narrow.cpu().numpy())
