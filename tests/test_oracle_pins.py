"""Pins of the fp64 oracle to facts outside itself (CPU only).

* unpack: hand-packed golden bytes, single-bit brute force over every stream
  position (codes straddling words at 3/5/6 bits included), and the
  independent test packer on random codes;
* bf16 decode: every finite pattern against torch's bfloat16 conversion;
* product: exact rational brute force (fractions.Fraction), closed forms
  (integer dot product with s=1, b=0; bias-only with zero codes; per-group
  scales), invariants (scaling, linearity, column/row placement);
* widen: identical fp64 weights bit for bit for every admitted pair, identity,
  refusals, common width.
A plausible slip in the oracle (bit order, a dropped bias, a wrong group index,
a transposed operand, a swapped scale/bias) fails at least one test here.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth
from tests.packing import pack, pack_row, row_bytes

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "packing.txt")
BITS = (2, 3, 4, 5, 6, 8)
GROUPS = (32, 64, 128)


def _golden():
    out = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        f = dict(kv.split("=") for kv in line.split())
        out.append((int(f["bits"]), [int(c) for c in f["codes"].split(",")],
                    bytes(int(b, 16) for b in f["bytes"].split(","))))
    return out


@pytest.mark.parametrize("bits,codes,raw", _golden())
def test_golden_packing(bits, codes, raw):
    # The golden bytes, repeated to fill one 32-code row, decode to the codes.
    reps = 32 // len(codes)
    row = np.frombuffer(raw * reps, dtype=np.uint8).copy().view(np.uint32)
    for i in range(32):
        assert oracle.code(row, 32, bits, 0, i) == codes[i % len(codes)]
    # ...and the independent test packer writes exactly those bytes.
    assert row_bytes(pack_row(codes * reps, bits)).tobytes() == raw * reps


@pytest.mark.parametrize("bits", BITS)
def test_single_bit_positions(bits):
    K = 64
    nbits = K * bits
    for p in range(nbits):
        acc = 1 << p
        row = np.array([(acc >> (32 * w)) & 0xFFFFFFFF for w in range(nbits // 32)],
                       dtype=np.uint32)
        for k in range(K):
            want = (1 << (p % bits)) if k == p // bits else 0
            assert oracle.code(row, K, bits, 0, k) == want, (p, k)


@pytest.mark.parametrize("bits", BITS)
def test_random_codes_roundtrip(bits):
    rng = np.random.default_rng(bits)
    N, K = 3, 128
    codes = rng.integers(0, 1 << bits, size=(N, K))
    W = pack(codes, bits)
    for n in range(N):
        for k in range(K):
            assert oracle.code(W, K, bits, n, k) == codes[n, k]


def test_bf16_decode_all_patterns():
    torch = pytest.importorskip("torch")
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    finite = np.isfinite(ref)
    got = np.array([oracle.bf16(int(v)) for v in h[finite]])
    assert np.array_equal(got, ref[finite])


def _exact_y(x_bits, codes, s_bits, b_bits, group):
    """Exact rational y and sum|x*w| from decoded values (Fraction arithmetic)."""
    xf = synth.bf16_bits_to_f32(x_bits).astype(np.float64)
    sf = synth.bf16_bits_to_f32(s_bits).astype(np.float64)
    bf = synth.bf16_bits_to_f32(b_bits).astype(np.float64)
    rows, K = xf.shape
    N = codes.shape[0]
    y = [[Fraction(0)] * N for _ in range(rows)]
    a = [[Fraction(0)] * N for _ in range(rows)]
    for r in range(rows):
        for n in range(N):
            for k in range(K):
                w = Fraction(sf[n, k // group]) * int(codes[n, k]) + Fraction(bf[n, k // group])
                t = Fraction(xf[r, k]) * w
                y[r][n] += t
                a[r][n] += abs(t)
    return y, a


@pytest.mark.parametrize("bits,group", [(b, g) for b in BITS for g in GROUPS])
def test_brute_force_exact(bits, group):
    rng = np.random.default_rng(100 * bits + group)
    N, K, rows = 3, 2 * group, 2
    codes = rng.integers(0, 1 << bits, size=(N, K))
    W = pack(codes, bits)
    s = synth.to_bf16(rng.uniform(0.001, 0.03, size=(N, K // group)))
    b = synth.to_bf16(-synth.bf16_bits_to_f32(s) * 2 ** (bits - 1) * rng.uniform(0.9, 1.1, s.shape))
    x = synth.to_bf16(rng.standard_normal((rows, K)))
    y64, absum = oracle.qmm(x, W, s, b, N, K, bits, group)
    ye, ae = _exact_y(x, codes, s, b, group)
    for r in range(rows):
        for n in range(N):
            # sequential fp64 sum: |err| <= K * 2^-53 * sum|terms| (plus exact products)
            tol = (K + 2) * 2.0 ** -53 * float(ae[r][n])
            assert abs(Fraction(y64[r, n]) - ye[r][n]) <= Fraction(tol)
            assert abs(Fraction(absum[r, n]) - ae[r][n]) <= Fraction(tol)


def test_integer_dot_closed_form():
    # s = 1, b = 0, small integer x: y is the exact integer dot product.
    rng = np.random.default_rng(7)
    for bits in BITS:
        N, K, G = 4, 128, 32
        codes = rng.integers(0, 1 << bits, size=(N, K))
        xi = rng.integers(-8, 9, size=(2, K))
        x = synth.to_bf16(xi.astype(np.float64))
        one = synth.to_bf16(np.ones((N, K // G)))
        zero = synth.to_bf16(np.zeros((N, K // G)))
        y64, _ = oracle.qmm(x, pack(codes, bits), one, zero, N, K, bits, G)
        want = xi @ codes.T
        assert np.array_equal(y64, want.astype(np.float64))


def test_bias_only_closed_form():
    # codes all zero: y = sum_g b_g * sum_{k in g} x_k (distinct b per group).
    N, K, G, bits = 2, 128, 32, 5
    W = pack(np.zeros((N, K), dtype=int), bits)
    s = synth.to_bf16(np.full((N, K // G), 0.5))
    bv = np.array([[1, -2, 3, -4], [0.5, 0.25, -1, 2]])
    b = synth.to_bf16(bv)
    xi = np.arange(K, dtype=np.float64).reshape(1, K) % 7 - 3
    x = synth.to_bf16(xi)
    y64, _ = oracle.qmm(x, W, s, b, N, K, bits, G)
    want = [sum(bv[n, g] * xi[0, g * G:(g + 1) * G].sum() for g in range(K // G)) for n in range(N)]
    assert np.array_equal(y64[0], np.array(want))


def test_group_index_and_scale_vs_bias():
    # Per-group scales 1,2,4,8 with all-ones codes and all-ones x: y = 32*(1+2+4+8) + 32*sum(b).
    N, K, G, bits = 1, 128, 32, 3
    W = pack(np.ones((N, K), dtype=int), bits)
    s = synth.to_bf16(np.array([[1.0, 2.0, 4.0, 8.0]]))
    b = synth.to_bf16(np.array([[0.0, 0.0, 0.0, 16.0]]))
    x = synth.to_bf16(np.ones((1, K)))
    y64, absum = oracle.qmm(x, W, s, b, N, K, bits, G)
    assert y64[0, 0] == 32 * 15 + 32 * 16
    assert absum[0, 0] == y64[0, 0]
    # a distinct x per group exposes k/G vs k%G slips
    xg = synth.to_bf16(np.repeat(np.array([[1.0, 0.0, 0.0, 0.0]]), G, axis=1))
    y64, _ = oracle.qmm(xg, W, s, b, N, K, bits, G)
    assert y64[0, 0] == 32 * 1.0


def test_scaling_and_linearity_invariants():
    m = synth.make_matrix(8, 256, 6, 64, 5, 0.001, 0.03)
    x = synth.make_x(3, 256, 5)
    y, _ = oracle.qmm(x, m.W, m.scales, m.biases, m.N, m.K, m.bits, m.group)
    s2 = synth.to_bf16(2.0 * synth.bf16_bits_to_f32(m.scales))
    b2 = synth.to_bf16(2.0 * synth.bf16_bits_to_f32(m.biases))
    y2, _ = oracle.qmm(x, m.W, s2, b2, m.N, m.K, m.bits, m.group)
    assert np.array_equal(y2, 2.0 * y)
    # each output row depends on its own x row only; each column on its own W row
    y1, _ = oracle.qmm(x[1:2], m.W, m.scales, m.biases, m.N, m.K, m.bits, m.group)
    assert np.array_equal(y1[0], y[1])
    yc, _ = oracle.qmm(x, m.W, m.scales, m.biases, m.N, m.K, m.bits, m.group, cols=[5, 2])
    assert np.array_equal(yc[:, 0], y[:, 5]) and np.array_equal(yc[:, 1], y[:, 2])
    perm = np.array([3, 0, 7, 1, 2, 6, 5, 4])
    yp, _ = oracle.qmm(x, m.W[perm], m.scales[perm], m.biases[perm], m.N, m.K, m.bits, m.group)
    assert np.array_equal(yp, y[:, perm])


def test_refusals():
    m = synth.make_matrix(2, 64, 4, 32, 1, 0.001, 0.03)
    x = synth.make_x(1, 64, 1)
    for bits, group, K in ((7, 32, 64), (4, 48, 96), (4, 64, 96)):
        with pytest.raises(oracle.OracleError):
            oracle.qmm(x[:, :K] if K <= 64 else np.zeros((1, K), np.uint16),
                       np.zeros((2, K * bits // 32 + 1), np.uint32), m.scales, m.biases,
                       2, K, bits, group)


# ---------------------------------------------------------------- widen ----

WIDEN_PAIRS = [(b0, g0, b1, g1) for b0 in BITS for g0 in GROUPS for b1 in BITS for g1 in GROUPS
               if b1 >= b0 and g0 % g1 == 0]


@pytest.mark.parametrize("b0,g0,b1,g1", WIDEN_PAIRS)
def test_widen_same_fp64_weights(b0, g0, b1, g1):
    N, K = 3, 256
    m = synth.make_matrix(N, K, b0, g0, 1000 + b0 * 10 + g0, 0.001, 0.03)
    Wo, so, bo = oracle.widen(m.W, m.scales, m.biases, N, K, b0, g0, b1, g1)
    w0 = oracle.weights(m.W, m.scales, m.biases, N, K, b0, g0)
    w1 = oracle.weights(Wo, so, bo, N, K, b1, g1)
    assert np.array_equal(w0.view(np.uint64), w1.view(np.uint64))
    for k in (0, 1, K // 2 + 3, K - 1):
        assert oracle.code(Wo, K, b1, 1, k) == oracle.code(m.W, K, b0, 1, k)
    if (b0, g0) == (b1, g1):
        assert np.array_equal(Wo, m.W) and np.array_equal(so, m.scales)


def test_widen_refusals_and_common_width():
    m = synth.make_matrix(2, 256, 5, 64, 3, 0.001, 0.03)
    with pytest.raises(oracle.OracleError) as e:
        oracle.widen(m.W, m.scales, m.biases, 2, 256, 5, 64, 4, 64)
    assert e.value.rc == oracle.ENARROW
    with pytest.raises(oracle.OracleError) as e:
        oracle.widen(m.W, m.scales, m.biases, 2, 256, 5, 64, 5, 128)
    assert e.value.rc == oracle.EGROUP
    with pytest.raises(oracle.OracleError) as e:
        oracle.widen(m.W, m.scales, m.biases, 2, 256, 5, 64, 7, 64)
    assert e.value.rc == oracle.EINVAL
    assert oracle.common_width([4, 5, 5, 6], [64, 128, 128, 64]) == (6, 64)
    assert oracle.common_width([4, 5, 5], [64, 128, 128]) == (5, 64)
    assert oracle.common_width([2], [128]) == (2, 128)
    with pytest.raises(oracle.OracleError):
        oracle.common_width([4, 7], [64, 64])


def test_negative_control_exceeds_bound():
    # A reference whose scales are 1% off moves y by 0.01 * sum_k x*s*q; on the
    # single-matrix workload that must exceed the fp32 bound on some column.
    m, x = synth.single_matrix()
    y, absum = oracle.qmm(x, m.W, m.scales, m.biases, m.N, m.K, m.bits, m.group)
    zero = np.zeros_like(m.biases)
    ysq, _ = oracle.qmm(x, m.W, m.scales, zero, m.N, m.K, m.bits, m.group)
    ratio = np.abs(0.01 * ysq) / oracle.bound(absum, m.K)
    assert ratio.max() > 1.0


def test_relu2_closed_form():
    # max(v, 0)^2 at values whose squares are exact: negatives and zeros give 0.
    y = np.array([-3.0, -0.0, 0.0, 0.5, 2.0, 1e-3, -1e300, 3.0])
    assert oracle.relu2(y).tolist() == [0.0, 0.0, 0.0, 0.25, 4.0, 1e-6, 0.0, 9.0]


def test_relu2_monotone_and_even_part():
    v = np.linspace(-5, 5, 1001)
    r = oracle.relu2(v)
    assert np.all(np.diff(r) >= 0) and np.all(r[v <= 0] == 0)
    # on v > 0 it is the square: relu2(v) * relu2(1/v) == 1 up to rounding
    pos = v[v > 0]
    assert np.allclose(oracle.relu2(pos) * oracle.relu2(1 / pos), 1.0, rtol=1e-15, atol=0)


@pytest.mark.parametrize("h", [0x3F80, 0x4300, 0x3A83, 0x7F00, 0x0080])
def test_bf16_ulp_is_the_spacing_of_adjacent_patterns(h):
    # one ulp at a bf16 value = the gap to the next bit pattern (same exponent)
    a, b = oracle.bf16(h), oracle.bf16(h + 1)
    assert oracle.bf16_ulp(np.array([a]))[0] == b - a
