"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Bars (TensorFold PR #788 row-kernel and tf-affine-ref commits):
  (i)   every output within (K*2^-24 + 2^-20) * sum|x*w| of the fp64 product;
  (ii)  each row alone equals the same row in 2-, 3-, 8- and 16-row windows,
        bit for bit, at every window position;
  (iii) strided and stacked outputs equal the contiguous result bit for bit,
        with the gap columns untouched;
  and the negative control: the oracle with scales 1 % off lies outside the
  bound on some column, asserted for every full-size workload.

Full-size workloads are checked on every output column (TFQ_PARITY_COLS=n
samples n columns instead, for quick runs).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import mlx_affine_bit_gb300 as tf
from tests.gpu_util import DEV, DevMatrix, dev, full_cols, oracle_check, run_qmm, sample_cols

pytestmark = pytest.mark.gpu

BITS = (2, 3, 4, 5, 6, 8)
GROUPS = (32, 64, 128)


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    yield
    torch.cuda.synchronize()
    tf.tf_device_status()


def test_single_matrix_full():
    m, x = synth.single_matrix()
    y = run_qmm(DevMatrix(m), dev(x)).cpu().numpy()
    worst, ctrl = oracle_check(m, x, y, control=True)
    print("single matrix worst err/bound %.4f, 1%%-off control %.2f" % (worst, ctrl))


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("group", GROUPS)
@pytest.mark.parametrize("N,K,rows", [(300, 1536, 3), (257, 2048, 11), (33, 1024, 16)])
def test_widths_small_full(bits, group, N, K, rows):
    # several column tiles, a ragged column tail, 2-4 K chunks; G=128 at K=1536
    # takes the producer-copy path (K not a multiple of 8*G).
    m = synth.make_matrix(N, K, bits, group, 500 + bits * 7 + group, 0.001, 0.03)
    x = synth.make_x(rows, K, 77 + rows)
    y = run_qmm(DevMatrix(m), dev(x)).cpu().numpy()
    oracle_check(m, x, y)


@pytest.mark.parametrize("bits,group,seed", synth.width_sweep_cases())
def test_width_sweep_4096(bits, group, seed):
    m = synth.width_sweep_matrix(bits, group, seed)
    x = synth.make_x(1, m.K, seed)
    y = run_qmm(DevMatrix(m), dev(x)).cpu().numpy()
    worst, ctrl = oracle_check(m, x, y, full_cols(m.N, seed), control=True)
    print("sweep %d/g%d worst err/bound %.4f, control %.2f" % (bits, group, worst, ctrl))


@pytest.mark.parametrize("N,K,seed", synth.DECODE_SHAPES)
def test_decode_windows_bit_exact(N, K, seed):
    m = synth.decode_matrix(N, K, seed)
    dm = DevMatrix(m)
    x = synth.make_x(16, K, seed)
    xd = dev(x)
    alone = [run_qmm(dm, xd[r:r + 1].contiguous()) for r in range(16)]
    for w in (2, 3, 8, 16):
        for p0 in range(0, 16 - w + 1):
            yw = run_qmm(dm, xd[p0:p0 + w].contiguous())
            for i in range(w):
                assert torch.equal(yw[i].view(torch.int32), alone[p0 + i][0].view(torch.int32)), (w, p0, i)
    # Rows of every window equal the rows alone (above), so the 16-row output
    # covers the 1-, 2-, 3- and 8-row cases too: every column against the oracle.
    y16 = run_qmm(dm, xd).cpu().numpy()
    assert torch.equal(torch.from_numpy(y16[0:1]).view(torch.int32), alone[0].cpu().view(torch.int32))
    worst, ctrl = oracle_check(m, x, y16, full_cols(N, seed), control=True)
    _, ctrl1 = oracle_check(m, x[0:1], y16[0:1], full_cols(N, seed), control=True)
    print("decode %dx%d worst err/bound %.4f, control r16 %.2f r1 %.2f" % (N, K, worst, ctrl, ctrl1))


@pytest.mark.parametrize("rows", list(range(1, 17)))
def test_every_row_count_matches_alone(rows):
    m = synth.make_matrix(200, 2048, 5, 64, 9, 0.001, 0.03)
    dm = DevMatrix(m)
    x = synth.make_x(rows, m.K, 900 + rows)
    xd = dev(x)
    y = run_qmm(dm, xd)
    for r in range(rows):
        assert torch.equal(y[r].view(torch.int32), run_qmm(dm, xd[r:r + 1].contiguous())[0].view(torch.int32))
    oracle_check(m, x, y.cpu().numpy())


@pytest.mark.parametrize("bits,group", [(6, 32), (3, 128), (8, 64)])
def test_strided_equals_contiguous(bits, group):
    N, K, rows = 500, 2048, 5
    m = synth.make_matrix(N, K, bits, group, 31, 0.001, 0.03)
    dm = DevMatrix(m)
    xd = dev(synth.make_x(rows, K, 31))
    yc = run_qmm(dm, xd)
    stride = N + 37
    ys = run_qmm(dm, xd, y_stride=stride, fill=-1234.5)
    assert torch.equal(ys[:, :N].view(torch.int32), yc.view(torch.int32))
    assert torch.all(ys[:, N:] == -1234.5)


@pytest.mark.parametrize("N,K,rows", [(1, 32, 1), (17, 96, 2), (16, 64, 16), (129, 4096, 1)])
def test_edge_shapes(N, K, rows):
    for bits in (3, 8):
        m = synth.make_matrix(N, K, bits, 32, 3 * N + K, 0.001, 0.03)
        x = synth.make_x(rows, K, N)
        oracle_check(m, x, run_qmm(DevMatrix(m), dev(x)).cpu().numpy())


def test_extreme_codes_and_zero_x():
    from tests.packing import pack
    N, K = 40, 512
    for bits in BITS:
        codes = np.full((N, K), (1 << bits) - 1)
        codes[::3] = 0
        m = synth.make_matrix(N, K, bits, 64, 1, 0.001, 0.03)
        m.W = pack(codes, bits)
        x = synth.make_x(2, K, 5)
        oracle_check(m, x, run_qmm(DevMatrix(m), dev(x)).cpu().numpy())
        y0 = run_qmm(DevMatrix(m), dev(np.zeros((1, K), np.uint16))).cpu().numpy()
        assert np.all(y0 == 0.0)


def test_integer_dot_exact():
    # s=1, b=0, small integer x: every partial sum is an integer below 2^24, so
    # the GPU result is exactly the integer dot product.
    from tests.packing import pack
    rng = np.random.default_rng(3)
    N, K = 64, 1024
    for bits in BITS:
        codes = rng.integers(0, 1 << bits, size=(N, K))
        xi = rng.integers(-3, 4, size=(4, K))
        m = synth.make_matrix(N, K, bits, 32, 2, 0.001, 0.03)
        m.W = pack(codes, bits)
        m.scales = synth.to_bf16(np.ones((N, K // 32)))
        m.biases = synth.to_bf16(np.zeros((N, K // 32)))
        y = run_qmm(DevMatrix(m), dev(synth.to_bf16(xi.astype(np.float64)))).cpu().numpy()
        assert np.array_equal(y.astype(np.int64), xi @ codes.T)


# ------------------------------------------------------------ widen & stack --

@pytest.mark.parametrize("b0,g0,b1,g1", [(4, 64, 5, 64), (5, 128, 5, 64), (2, 128, 8, 32),
                                         (3, 32, 6, 32), (6, 64, 6, 64), (5, 64, 8, 32)])
def test_widen_matches_oracle(b0, g0, b1, g1):
    N, K = 70, 1024
    m = synth.make_matrix(N, K, b0, g0, 40 + b0 + g0, 0.001, 0.03)
    dm = DevMatrix(m)
    Wo = torch.zeros((N, K * b1 // 32), dtype=torch.int32, device=DEV)
    so = torch.zeros((N, K // g1), dtype=torch.int16, device=DEV)
    bo = torch.zeros_like(so)
    tf.tf_widen(dm.W, dm.s, dm.b, N, K, b0, g0, Wo, so, bo, b1, g1)
    rW, rs, rb = oracle.widen(m.W, m.scales, m.biases, N, K, b0, g0, b1, g1)
    assert np.array_equal(Wo.cpu().numpy().view(np.uint32), rW)
    assert np.array_equal(so.cpu().numpy().view(np.uint16), rs)
    assert np.array_equal(bo.cpu().numpy().view(np.uint16), rb)


def test_widen_refusals():
    m = synth.make_matrix(4, 256, 5, 64, 1, 0.001, 0.03)
    dm = DevMatrix(m)
    out = torch.zeros(4096, dtype=torch.int32, device=DEV)
    for (b1, g1, code) in ((4, 64, -7), (5, 128, -8), (7, 64, -1)):
        with pytest.raises(tf.TfError) as e:
            tf.tf_widen(dm.W, dm.s, dm.b, 4, 256, 5, 64, out, out, out, b1, g1)
        assert e.value.rc == code


def _widen_dev(m, bits, group):
    Wo = torch.zeros((m.N, m.K * bits // 32), dtype=torch.int32, device=DEV)
    so = torch.zeros((m.N, m.K // group), dtype=torch.int16, device=DEV)
    bo = torch.zeros_like(so)
    dm = DevMatrix(m)
    tf.tf_widen(dm.W, dm.s, dm.b, m.N, m.K, m.bits, m.group, Wo, so, bo, bits, group)
    return Wo, so, bo


@pytest.mark.parametrize("rows", synth.STACK_ROWS)
def test_fused_stack(rows):
    K = synth.STACK_K
    mats = synth.stack_member_matrices()
    # runs: members 0-2 widen to 5-bit g64 (6192 columns), member 3 is 6-bit g64 (48)
    parts = [_widen_dev(m, 5, 64) for m in mats[:3]]
    W5 = torch.cat([p[0] for p in parts]).contiguous()
    s5 = torch.cat([p[1] for p in parts]).contiguous()
    b5 = torch.cat([p[2] for p in parts]).contiguous()
    m6 = DevMatrix(mats[3])
    runs = [(W5, s5, b5, 6192, 5, 64), (m6.W, m6.s, m6.b, 48, 6, 64)]
    stride = 6240
    x = synth.make_x(rows, K, 60 + rows)
    xd = dev(x)
    members = [(0, 0, 4096, 0), (0, 4096, 2048, 4096), (0, 6144, 48, 6144), (1, 0, 48, 6192)]
    y = torch.full((rows, stride), float("nan"), dtype=torch.float32, device=DEV)
    tf.tf_qmm_stack(xd, rows, K, runs, members, y, stride)
    # each run equals its own contiguous product bit for bit
    y5 = torch.empty((rows, 6192), dtype=torch.float32, device=DEV)
    tf.tf_qmm(xd, rows, K, W5, s5, b5, 6192, 5, 64, y5, 6192)
    y6 = torch.empty((rows, 48), dtype=torch.float32, device=DEV)
    tf.tf_qmm(xd, rows, K, m6.W, m6.s, m6.b, 48, 6, 64, y6, 48)
    assert torch.equal(y[:, :6192].view(torch.int32), y5.view(torch.int32))
    assert torch.equal(y[:, 6192:].view(torch.int32), y6.view(torch.int32))
    # and every member is within the bound of the oracle on its unwidened
    # matrix, on every column, with the 1%-off control outside it
    yn = y.cpu().numpy()
    off = 0
    for m in mats:
        worst, ctrl = oracle_check(m, x, yn[:, off:off + m.N], full_cols(m.N, m.seed), control=True)
        print("stack r%d member %d/g%d (%d cols) worst %.4f, control %.2f" % (rows, m.bits, m.group, m.N, worst, ctrl))
        off += m.N
    # non-adjacent destinations through the column map
    members2 = [(0, 4096, 2048, 0), (1, 0, 48, 2048), (0, 0, 4096, 2096), (0, 6144, 48, 6192)]
    y2 = torch.full((rows, stride), float("nan"), dtype=torch.float32, device=DEV)
    tf.tf_qmm_stack(xd, rows, K, runs, members2, y2, stride)
    assert torch.equal(y2[:, 0:2048].view(torch.int32), y5[:, 4096:6144].view(torch.int32))
    assert torch.equal(y2[:, 2048:2096].view(torch.int32), y6.view(torch.int32))
    assert torch.equal(y2[:, 2096:6192].view(torch.int32), y5[:, :4096].view(torch.int32))
    assert torch.equal(y2[:, 6192:].view(torch.int32), y5[:, 6144:].view(torch.int32))


def test_stack_refusals():
    m = synth.make_matrix(64, 256, 4, 64, 1, 0.001, 0.03)
    dm = DevMatrix(m)
    xd = dev(synth.make_x(1, 256, 1))
    y = torch.zeros((1, 200), dtype=torch.float32, device=DEV)
    runs = [(dm.W, dm.s, dm.b, 64, 4, 64)]
    for members in ([(0, 0, 65, 0)], [(1, 0, 8, 0)], [(0, 0, 32, 0), (0, 32, 32, 16)],
                    [(0, 0, 32, 190)], [(0, 0, 32, 0), (0, 16, 8, 100)]):
        with pytest.raises(tf.TfError) as e:
            tf.tf_qmm_stack(xd, 1, 256, runs, members, y, 200)
        assert e.value.rc == -9


# ------------------------------------------------------------------- LM head --

@pytest.mark.parametrize("bits,group,seed", synth.LMHEAD_CASES)
def test_lmhead(bits, group, seed):
    m = synth.lmhead_matrix(bits, group, seed)
    dm = DevMatrix(m)
    x = synth.make_x(16, m.K, seed)
    xd = dev(x)
    y1 = run_qmm(dm, xd[0:1].contiguous())
    y16 = run_qmm(dm, xd)
    assert torch.equal(y16[0].view(torch.int32), y1[0].view(torch.int32))
    cols = full_cols(m.N, seed)
    y1n = y1.cpu().numpy()
    w1, c1 = oracle_check(m, x[0:1], y1n, cols, control=True)
    w16, c16 = oracle_check(m, x, y16.cpu().numpy(), cols, control=True)
    print("LM head %d/g%d worst r1 %.4f r16 %.4f, control r1 %.2f r16 %.2f" % (bits, group, w1, w16, c1, c16))


@pytest.mark.parametrize("bits,group", [(2, 64), (3, 128), (4, 32), (5, 64), (6, 32), (8, 128)])
def test_sixteen_rows_two_tiles(bits, group):
    # 2048 columns over K = 8192 at 16 rows take two m-tiles per item with one
    # consumer group (split K); every row equals the row computed alone (a
    # one-row plan) bit for bit and meets the tolerance.
    N, K = 2048, 8192
    m = synth.make_matrix(N, K, bits, group, 170 + bits, 0.001, 0.03)
    dm = DevMatrix(m)
    x = synth.make_x(16, K, 171)
    xd = dev(x)
    y = run_qmm(dm, xd)
    for r in (0, 5, 15):
        alone = run_qmm(dm, xd[r:r + 1].contiguous())
        assert torch.equal(y[r].view(torch.int32), alone[0].view(torch.int32)), r
    oracle_check(m, x, y.cpu().numpy(), sample_cols(N, 24, bits))


@pytest.mark.parametrize("bits,group", [(4, 32), (5, 32), (6, 32), (4, 128), (6, 64)])
def test_offset_codes_keep_margin(bits, group):
    # 4-6-bit codes enter the tensor cores as 128 + c (the bias term takes the
    # 128 * sum(x) back), which raises the rounding of the group products.  At
    # a short K, where the tolerance is tightest, the worst error stays well
    # inside it (an fp32 model of the arithmetic gives about 0.02 of it).
    N, K = 512, 256
    m = synth.make_matrix(N, K, bits, group, 160 + bits, 0.001, 0.03)
    x = synth.make_x(4, K, 161)
    y = run_qmm(DevMatrix(m), dev(x)).cpu().numpy()
    worst = oracle_check(m, x, y)
    assert worst < 0.25, worst


@pytest.mark.parametrize("mode", [1, 2, 6])
def test_launch_modes_bit_identical(mode):
    # A back-to-back sequence of products (including a split-K shape) gives the
    # same bits with programmatic dependent launch as with plain launches.
    mats = [synth.make_matrix(N, K, b, g, 70 + i, 0.001, 0.03)
            for i, (N, K, b, g) in enumerate([(4096, 4096, 4, 64), (2048, 12288, 6, 32),
                                              (300, 2048, 3, 128), (4096, 4096, 8, 32)])]
    dms = [DevMatrix(m) for m in mats]
    xs = [dev(synth.make_x(3, m.K, 80 + i)) for i, m in enumerate(mats)]
    ref = [run_qmm(dm, x) for dm, x in zip(dms, xs)]
    old = tf.tf_set_launch_mode(mode)
    try:
        for _ in range(3):
            got = [run_qmm(dm, x) for dm, x in zip(dms, xs)]
            for a, b in zip(ref, got):
                assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    finally:
        tf.tf_set_launch_mode(old)


@pytest.mark.parametrize("bits,group", [(2, 128), (3, 32), (4, 64), (5, 32), (5, 128), (6, 32)])
@pytest.mark.parametrize("rows", [1, 3, 8, 16])
def test_plans_bit_identical(bits, group, rows):
    # 12304 columns take the widest plan (two m-tiles per item, or one with 16
    # rows; two consumer groups where the stages fit; an odd item count),
    # slices of 1024 and 1040 columns the one-m-tile, two-CTA plans: the shared
    # columns agree bit for bit.
    N, K = 12304, 2048
    m = synth.make_matrix(N, K, bits, group, 40 + bits, 0.001, 0.03)
    dm = DevMatrix(m)
    x = synth.make_x(rows, K, 41 + rows)
    xd = dev(x)
    y = run_qmm(dm, xd)
    for c0, n in ((0, 1024), (N - 1040, 1040)):
        ys = torch.full((rows, n), float("nan"), dtype=torch.float32, device=DEV)
        tf.tf_qmm(xd, rows, K, dm.W[c0:c0 + n], dm.s[c0:c0 + n], dm.b[c0:c0 + n], n, bits, group, ys, n)
        assert torch.equal(ys.view(torch.int32), y[:, c0:c0 + n].contiguous().view(torch.int32)), c0
    oracle_check(m, x, y.cpu().numpy(), sample_cols(N, 48, bits))


@pytest.mark.parametrize("mode", [0, 1, 2, 6])
def test_stack_launch_modes_bit_identical(mode):
    # Under programmatic dependent launch the runs of a stack overlap (the
    # first releases the rest only after its dependency wait; a split-K run
    # keeps the ordinary ordering).  Every run still equals its own product.
    K = 8192
    shapes = [(4096, 4, 64), (64, 5, 32), (48, 6, 64), (2000, 3, 128)]
    mats = [synth.make_matrix(N, K, b, g, 90 + i, 0.001, 0.03) for i, (N, b, g) in enumerate(shapes)]
    dms = [DevMatrix(m) for m in mats]
    x = synth.make_x(3, K, 95)
    xd = dev(x)
    runs = [(dm.W, dm.s, dm.b, m.N, m.bits, m.group) for dm, m in zip(dms, mats)]
    members, off = [], 0
    for i, m in enumerate(mats):
        members.append((i, 0, m.N, off))
        off += m.N
    ref = [run_qmm(dm, xd) for dm in dms]
    old = tf.tf_set_launch_mode(mode)
    try:
        for _ in range(3):
            y = torch.full((3, off), float("nan"), dtype=torch.float32, device=DEV)
            tf.tf_qmm_stack(xd, 3, K, runs, members, y, off)
            c = 0
            for r, m in zip(ref, mats):
                assert torch.equal(y[:, c:c + m.N].contiguous().view(torch.int32), r.view(torch.int32))
                c += m.N
    finally:
        tf.tf_set_launch_mode(old)


def test_early_x_writes_wait_for_the_previous_product():
    # Under early-x launches a product computes before the previous kernel
    # finishes but writes only after it: products that write the same output
    # back to back leave the last one's result (write-after-write order), also
    # when the later product is much smaller (it would otherwise finish first).
    shapes = [(4096, 4096, 8, 32), (4096, 256, 2, 128), (4096, 2048, 4, 64)]
    mats = [synth.make_matrix(N, K, b, g, 190 + i, 0.001, 0.03) for i, (N, K, b, g) in enumerate(shapes)]
    dms = [DevMatrix(m) for m in mats]
    xs = [dev(synth.make_x(1, m.K, 191 + i)) for i, m in enumerate(mats)]
    refs = [run_qmm(dm, x) for dm, x in zip(dms, xs)]
    old = tf.tf_set_launch_mode(tf.TF_LAUNCH_EARLY_WEIGHTS | tf.TF_LAUNCH_EARLY_X)
    try:
        y = torch.zeros((1, 4096), dtype=torch.float32, device=DEV)
        for rep in range(30):
            order = [0, 1, 2] if rep % 2 == 0 else [2, 0, 1]
            for i in order:
                m = mats[i]
                tf.tf_qmm(xs[i], 1, m.K, dms[i].W, dms[i].s, dms[i].b, m.N, m.bits, m.group, y, m.N)
            torch.cuda.synchronize()
            assert torch.equal(y.view(torch.int32), refs[order[-1]].view(torch.int32)), rep
    finally:
        tf.tf_set_launch_mode(old)
    tf.tf_device_status()


@pytest.mark.parametrize("bits,group,rows", [(6, 32, 1), (4, 64, 1), (3, 32, 2), (6, 32, 16), (4, 128, 16)])
def test_two_group_plans_repeatable(bits, group, rows):
    # The two-consumer-group plans (three to eight ring stages; each group
    # skips the other's stages) give the same bits on every call and never
    # trip a bounded wait.
    N, K = 24832, 2048
    m = synth.make_matrix(N, K, bits, group, 110 + bits, 0.001, 0.02)
    dm = DevMatrix(m)
    x = synth.make_x(rows, K, 111)
    xd = dev(x)
    ref = run_qmm(dm, xd)
    for _ in range(20):
        y = run_qmm(dm, xd)
        assert torch.equal(y.view(torch.int32), ref.view(torch.int32))
    torch.cuda.synchronize()
    tf.tf_device_status()
    oracle_check(m, x, ref.cpu().numpy(), sample_cols(N, 32, bits))


OPTION_SHAPES = [(4, 64, 300, 2048), (6, 32, 12304, 2048), (3, 128, 2048, 12288)]


@pytest.mark.parametrize("bits,group,N,K", OPTION_SHAPES)
def test_output_options_product_full(bits, group, N, K):
    # The output options apply their epilogue to this fp32 product bit for bit
    # (test_output_options): every column of it against the oracle, with the
    # 1%-off control outside the bound.
    m = synth.make_matrix(N, K, bits, group, 130 + bits, 0.001, 0.03)
    x = synth.make_x(16, K, 131)
    v = run_qmm(DevMatrix(m), dev(x)).cpu().numpy()
    worst, ctrl = oracle_check(m, x, v, full_cols(N, bits), control=True)
    print("options product %d/g%d %dx%d worst %.4f, control %.2f" % (bits, group, N, K, worst, ctrl))


def _bf16_bits_to_f64(t: torch.Tensor) -> np.ndarray:
    h = t.cpu().numpy().view(np.uint16).astype(np.uint32) << 16
    return h.view(np.float32).astype(np.float64)


@pytest.mark.parametrize("flags", [tf.TF_EPI_RELU2, tf.TF_OUT_BF16, tf.TF_OUT_BF16 | tf.TF_EPI_RELU2])
@pytest.mark.parametrize("bits,group,N,K", OPTION_SHAPES)
def test_output_options(flags, bits, group, N, K):
    # fp32 or bf16 output, with or without the squared-ReLU epilogue: within
    # the bound of the oracle's product passed through the same epilogue, equal
    # to the epilogue of the fp32 result bit for bit, and each row alone equal
    # to the same row of a 16-row window.
    m = synth.make_matrix(N, K, bits, group, 130 + bits, 0.001, 0.03)
    dm = DevMatrix(m)
    x = synth.make_x(16, K, 131)
    xd = dev(x)
    bf = bool(flags & tf.TF_OUT_BF16)
    dt = torch.int16 if bf else torch.float32

    def call(xs):
        y = torch.zeros((xs.shape[0], N), dtype=dt, device=DEV)
        tf.tf_qmm_ex(xs, xs.shape[0], K, dm.W, dm.s, dm.b, N, bits, group, y, N, flags)
        return y

    y16 = call(xd)
    v = run_qmm(dm, xd)                                     # the fp32 product
    if flags & tf.TF_EPI_RELU2:
        v = torch.clamp(v, min=0) * torch.clamp(v, min=0)
    want = v.to(torch.bfloat16).view(torch.int16) if bf else v
    assert torch.equal(y16.view(torch.int16 if bf else torch.int32), want.view(torch.int16 if bf else torch.int32))
    for r in (0, 7, 15):
        assert torch.equal(call(xd[r:r + 1].contiguous())[0], y16[r])
    cols = sample_cols(N, 40, bits)
    y64, absum = oracle.qmm(x, m.W, m.scales, m.biases, N, K, bits, group, cols=cols, nthreads=8)
    t, B = oracle.bound_out(y64, absum, K, bool(flags & tf.TF_EPI_RELU2), bf)
    got = _bf16_bits_to_f64(y16[:, cols]) if bf else y16[:, cols].cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - t) <= B)


@pytest.mark.parametrize("flags", [0, tf.TF_OUT_BF16 | tf.TF_EPI_RELU2])
def test_gather_equals_dense(flags):
    # Indexed slots over four experts (mixed widths, one with fewer columns):
    # every slot equals its expert's product on its x row alone, bit for bit;
    # columns past an expert's N stay untouched.
    K, x_rows, n_slots = 2048, 6, 37
    shapes = [(256, 4, 64), (256, 6, 32), (256, 3, 128), (160, 5, 64)]
    mats = [synth.make_matrix(N, K, b, g, 140 + i, 0.001, 0.03) for i, (N, b, g) in enumerate(shapes)]
    dms = [DevMatrix(m) for m in mats]
    x = synth.make_x(x_rows, K, 141)
    xd = dev(x)
    rng = np.random.default_rng(142)
    se = rng.integers(0, 4, n_slots).tolist()
    sr = rng.integers(0, x_rows, n_slots).tolist()
    bf = bool(flags & tf.TF_OUT_BF16)
    dt = torch.int16 if bf else torch.float32
    stride = 264
    y = torch.full((n_slots, stride), -7, dtype=torch.int16, device=DEV) if bf else \
        torch.full((n_slots, stride), float("nan"), dtype=torch.float32, device=DEV)
    experts = [(dm.W, dm.s, dm.b, m.N, m.bits, m.group) for dm, m in zip(dms, mats)]
    tf.tf_qmm_gather(xd, x_rows, K, experts, se, sr, y, stride, flags)
    for i in range(n_slots):
        m, dm = mats[se[i]], dms[se[i]]
        one = torch.zeros((1, m.N), dtype=dt, device=DEV)
        tf.tf_qmm_ex(xd[sr[i]:sr[i] + 1].contiguous(), 1, K, dm.W, dm.s, dm.b, m.N, m.bits, m.group, one, m.N,
                     flags)
        assert torch.equal(y[i, :m.N], one[0]), i
        tail = y[i, m.N:]
        if bf:
            assert torch.all(tail == -7)
        else:
            assert torch.all(torch.isnan(tail))
    # every expert's dense product on every x row and column against the
    # oracle, with the 1%-off control (each slot equals one of these rows)
    for e, (m, dm) in enumerate(zip(mats, dms)):
        yd = torch.zeros((x_rows, m.N), dtype=torch.float32, device=DEV)
        tf.tf_qmm(xd, x_rows, K, dm.W, dm.s, dm.b, m.N, m.bits, m.group, yd, m.N)
        oracle_check(m, x, yd.cpu().numpy(), control=True)
    # and the slots themselves (with their output options) for a few slots
    for i in (0, 5, 36):
        m = mats[se[i]]
        cols = sample_cols(m.N, 24, i)
        y64, absum = oracle.qmm(x[sr[i]:sr[i] + 1], m.W, m.scales, m.biases, m.N, K, m.bits, m.group, cols=cols)
        t, B = oracle.bound_out(y64, absum, K, bool(flags & tf.TF_EPI_RELU2), bf)
        got = _bf16_bits_to_f64(y[i:i + 1, cols]) if bf else y[i:i + 1, cols].cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got - t) <= B)


@pytest.mark.parametrize("rows", [17, 33, 65])
@pytest.mark.parametrize("flags", [0, tf.TF_OUT_BF16 | tf.TF_EPI_RELU2])
def test_rows_past_16(rows, flags):
    # More than 16 rows run as 16-row windows: every row equals the same row
    # computed alone, bit for bit, and the product stays within the bound.
    m = synth.make_matrix(700, 2048, 5, 64, 170, 0.001, 0.03)
    dm = DevMatrix(m)
    x = synth.make_x(rows, m.K, 171 + rows)
    xd = dev(x)
    bf = bool(flags & tf.TF_OUT_BF16)
    dt = torch.int16 if bf else torch.float32

    def call(xs):
        y = torch.zeros((xs.shape[0], m.N), dtype=dt, device=DEV)
        tf.tf_qmm_ex(xs, xs.shape[0], m.K, dm.W, dm.s, dm.b, m.N, m.bits, m.group, y, m.N, flags)
        return y

    y = call(xd)
    for r in (0, 15, 16, rows - 1):
        assert torch.equal(call(xd[r:r + 1].contiguous())[0], y[r]), r
    if flags == 0:
        y2 = run_qmm(dm, xd)                                   # tf_qmm takes any row count too
        assert torch.equal(y2.view(torch.int32), y.view(torch.int32))
    cols = sample_cols(m.N, 24, rows)
    y64, absum = oracle.qmm(x, m.W, m.scales, m.biases, m.N, m.K, m.bits, m.group, cols=cols, nthreads=8)
    t, B = oracle.bound_out(y64, absum, m.K, bool(flags & tf.TF_EPI_RELU2), bf)
    got = _bf16_bits_to_f64(y[:, cols]) if bf else y[:, cols].cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - t) <= B)
