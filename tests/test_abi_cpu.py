"""CPU-only checks of the C ABI: the library builds and loads, exports every
symbol include/tfqmm.h declares, and refuses bad arguments on the host before
any CUDA call.  Also runs the host build of the kernel's code unpack."""
import os
import re
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def tf():
    from mlx_affine_bit_gb300.build import build
    build()
    import mlx_affine_bit_gb300 as tf
    tf.lib()
    return tf


def test_exports_every_declared_symbol(tf):
    hdr = open(os.path.join(ROOT, "include", "tfqmm.h")).read()
    declared = set(re.findall(r"^(?:int|const char \*)\s*(tf_\w+)\s*\(", hdr, re.M))
    assert {"tf_qmm", "tf_qmm_stack", "tf_widen"} <= declared
    out = subprocess.check_output(["nm", "-D", "--defined-only", tf.SO]).decode()
    exported = set(re.findall(r"\sT\s(tf_\w+)$", out, re.M))
    assert declared <= exported, declared - exported
    for name in declared:
        getattr(tf.lib(), name)


def test_debug_build_exports(tf):
    # The bounds-checking build exports every entry point of both headers.
    names = set()
    for h in ("tfqmm.h", "tfqmm_debug.h"):
        names |= set(re.findall(r"^(?:int|const char \*)\s*(tf_\w+)\s*\(",
                                open(os.path.join(ROOT, "include", h)).read(), re.M))
    assert "tf_debug_shrink_y" in names
    out = subprocess.check_output(["nm", "-D", "--defined-only", tf.SO_DEBUG]).decode()
    exported = set(re.findall(r"\sT\s(tf_\w+)$", out, re.M))
    assert names <= exported, names - exported
    assert tf.debug_lib().tf_debug_shrink_y(17) == -3


def test_trace_build_exports(tf):
    # The phase-trace build (made on request) exports every entry point of
    # tfqmm.h and tfqmm_trace.h; the product library exports no trace entry.
    from mlx_affine_bit_gb300 import build
    so = build.build_trace()
    names = set()
    for h in ("tfqmm.h", "tfqmm_trace.h"):
        names |= set(re.findall(r"^(?:int|const char \*)\s*(tf_\w+)\s*\(",
                                open(os.path.join(ROOT, "include", h)).read(), re.M))
    assert {"tf_trace_reset", "tf_trace_read"} <= names
    out = subprocess.check_output(["nm", "-D", "--defined-only", so]).decode()
    exported = set(re.findall(r"\sT\s(tf_\w+)$", out, re.M))
    assert names <= exported, names - exported
    L = tf.trace_lib()
    for name in names:
        getattr(L, name)
    prod = subprocess.check_output(["nm", "-D", "--defined-only", tf.SO]).decode()
    assert "tf_trace_" not in prod


A = 4096  # a 16-byte aligned stand-in address; no call below reaches the device


@pytest.mark.parametrize("kw,code", [
    (dict(bits=7), -1), (dict(bits=1), -1),
    (dict(group=48), -2), (dict(group=64, K=96), -2), (dict(K=16, group=32), -2),
    (dict(rows=0), -3), (dict(rows=65537), -3),
    (dict(y_stride=255), -4),
    (dict(x=0), -5), (dict(W=0), -5), (dict(x=A + 8), -5), (dict(W=A + 4), -5), (dict(y=A + 2), -5),
    (dict(N=0, y_stride=0), -6),
])
def test_tf_qmm_refusals(tf, kw, code):
    args = dict(x=A, rows=1, K=1024, W=A, s=A, b=A, N=256, bits=4, group=64, y=A, y_stride=256)
    args.update(kw)
    rc = tf.lib().tf_qmm(args["x"], args["rows"], args["K"], args["W"], args["s"], args["b"],
                         args["N"], args["bits"], args["group"], args["y"], args["y_stride"], None)
    assert rc == code, tf.lib().tf_last_error_string()
    assert tf.lib().tf_last_error_string()


def test_widen_refusals_on_host(tf):
    L = tf.lib()
    assert L.tf_widen(A, A, A, 4, 256, 5, 64, A, A, A, 4, 64, None) == -7
    assert L.tf_widen(A, A, A, 4, 256, 5, 64, A, A, A, 5, 128, None) == -8
    assert L.tf_widen(A, A, A, 4, 256, 5, 32, A, A, A, 5, 64, None) == -8
    assert L.tf_widen(A, A, A, 4, 256, 5, 64, A, A, A, 7, 64, None) == -1


def test_stack_refusals_on_host(tf):
    runs = [(A, A, A, 64, 4, 64)]
    for members in ([(0, 0, 65, 0)], [(1, 0, 8, 0)], [(0, 0, 32, 0), (0, 32, 32, 16)],
                    [(0, 0, 32, 190)]):
        with pytest.raises(tf.TfError) as e:
            tf.tf_qmm_stack(A, 1, 256, runs, members, A, 200, stream=0)
        assert e.value.rc == -9


def test_bytes_and_common_width(tf):
    assert tf.tf_qmm_bytes(248320, 2048, 6, 32) == (248320 * 2048 * 6 // 8, 248320 * 64 * 2)
    assert tf.tf_common_width([4, 5, 5, 6], [64, 128, 128, 64]) == (6, 64)
    assert tf.tf_common_width([4, 5, 5], [64, 128, 128]) == (5, 64)
    with pytest.raises(tf.TfError):
        tf.tf_common_width([4, 7], [64, 64])
    assert "sm_103a" in tf.tf_version()


def test_unpack_host_build(tmp_path):
    exe = str(tmp_path / "unpack_test")
    subprocess.check_call(["g++", "-O1", "-std=c++17", os.path.join(ROOT, "tests", "unpack_host_test.cpp"),
                           "-o", exe])
    out = subprocess.check_output([exe]).decode()
    assert "PASS" in out


def test_planner_host(tmp_path):
    # Every launch plan over a grid of shapes, widths, groups, row counts and SM
    # counts, with and without overlapping products, fits shared memory (half
    # the SM for the overlap plans), has a ring of 2-8 stages, uses an
    # instantiated kernel, gives two consumer groups only one K slice and three
    # stages, and covers K with whole teams of CTAs.  Host code only (stubbed
    # launchers).
    import shutil
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "planner_test")
    subprocess.check_call([nvcc, "-std=c++17", "-O1", "-I" + os.path.join(ROOT, "mlx_affine_bit_gb300", "csrc"),
                           "-gencode", "arch=compute_103a,code=sm_103a",
                           os.path.join(ROOT, "tests", "planner_host_test.cu"), "-o", exe])
    out = subprocess.check_output([exe]).decode()
    assert "PASS" in out, out


def test_prompt_layout_host(tmp_path):
    # The prompt kernel's static plan for every width and group: shared memory
    # within a CTA's limit and above half an SM (one CTA and one tensor-memory
    # allocation per SM), aligned regions and pitches, whole accumulator sets, and
    # the register cap within the schedulers' files.  Host code only.
    import shutil
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "prompt_test")
    subprocess.check_call([nvcc, "-std=c++17", "-O1", "-I" + os.path.join(ROOT, "mlx_affine_bit_gb300", "csrc"),
                           "-gencode", "arch=compute_103a,code=sm_103a",
                           os.path.join(ROOT, "tests", "prompt_host_test.cu"), "-o", exe])
    out = subprocess.check_output([exe]).decode()
    assert "PASS" in out, out


def test_every_kernel_instantiated(tf):
    # 6 widths x 3 groups x row buckets {1, 2, 4, 8, 16} x one m-tile per item, and
    # buckets up to 8 rows with two m-tiles and one or two consumer groups, and
    # 16 rows with one m-tile and two groups or two m-tiles and one group: every host
    # launch stub is in the library.
    out = subprocess.check_output(["nm", "-C", "--defined-only", tf.SO]).decode()
    for bits in (2, 3, 4, 5, 6, 8):
        for group in (32, 64, 128):
            for rb in (1, 2, 4, 8, 16):
                for mt, cg in (((1, 1), (2, 1), (2, 2)) if rb <= 8 else ((1, 1), (1, 2), (2, 1))):
                    name = "tfq::qmm_kernel<%d, %d, %d, %d, %d>(" % (bits, group, rb, mt, cg)
                    assert name in out, name


def test_output_option_refusals_on_host(tf):
    L = tf.lib()
    # unknown flag bits; bf16 y needs 2-byte alignment only, fp32 y 4-byte
    assert L.tf_qmm_ex(A, 1, 1024, A, A, A, 256, 4, 64, A, 256, 4, None) == -12
    assert L.tf_qmm_ex(A, 1, 1024, A, A, A, 256, 4, 64, A + 2, 256, 0, None) == -5
    assert L.tf_qmm_ex(A, 65537, 1024, A, A, A, 256, 4, 64, A, 256, 1, None) == -3
    assert L.tf_qmm_ex(A, 1, 1024, A, A, A, 256, 4, 64, A, 255, 3, None) == -4


@pytest.mark.parametrize("slot_expert,slot_row,code", [
    ([0, 2], [0, 0], -13),        # a missing expert
    ([0, 1], [0, 3], -13),        # a missing x row (x_rows = 3)
    ([0, -1], [0, 0], -13),
    ([], [], -13),                # no slots
])
def test_gather_refusals_on_host(tf, slot_expert, slot_row, code):
    experts = [(A, A, A, 64, 4, 64), (A, A, A, 64, 5, 32)]
    with pytest.raises(tf.TfError) as e:
        tf.tf_qmm_gather(A, 3, 256, experts, slot_expert, slot_row, A, 64, 0, stream=0)
    assert e.value.rc == code


def test_gather_stride_and_flags_refused(tf):
    experts = [(A, A, A, 64, 4, 64), (A, A, A, 96, 5, 32)]
    with pytest.raises(tf.TfError) as e:      # y_stride below the used expert's N
        tf.tf_qmm_gather(A, 3, 256, experts, [1], [0], A, 64, 0, stream=0)
    assert e.value.rc == -4
    with pytest.raises(tf.TfError) as e:
        tf.tf_qmm_gather(A, 3, 256, experts, [0], [0], A, 96, 8, stream=0)
    assert e.value.rc == -12


def test_stack_keeps_16_rows(tf):
    with pytest.raises(tf.TfError) as e:
        tf.tf_qmm_stack(A, 17, 256, [(A, A, A, 64, 4, 64)], [(0, 0, 64, 0)], A, 64, stream=0)
    assert e.value.rc == -3


WIDEN_PAIRS = [(b0, g0, b1, g1) for b0 in (2, 3, 4, 5, 6, 8) for b1 in (2, 3, 4, 5, 6, 8) if b1 >= b0
               for g0 in (32, 64, 128) for g1 in (32, 64, 128) if g0 % g1 == 0]


@pytest.mark.parametrize("b0,g0,b1,g1", WIDEN_PAIRS)
def test_widen_host_equals_oracle(tf, b0, g0, b1, g1):
    # The host widen re-packs every code at the wider width and copies scales
    # and biases to each finer group: byte for byte the oracle's widen.
    import oracle
    import synth
    N, K = 9, 384
    m = synth.make_matrix(N, K, b0, g0, 700 + 11 * b0 + g0 + b1, 0.001, 0.03)
    got = tf.tf_widen_host(m.W, m.scales, m.biases, N, K, b0, g0, b1, g1)
    want = oracle.widen(m.W, m.scales, m.biases, N, K, b0, g0, b1, g1)
    for a, b in zip(got, want):
        assert a.dtype == b.dtype and np.array_equal(a, b)


def test_widen_host_refusals(tf):
    import synth
    m = synth.make_matrix(4, 256, 5, 64, 1, 0.001, 0.03)
    for (b1, g1, code) in ((4, 64, -7), (5, 128, -8), (7, 64, -1), (5, 48, -2)):
        with pytest.raises(tf.TfError) as e:
            tf.tf_widen_host(m.W, m.scales, m.biases, 4, 256, 5, 64, b1, g1)
        assert e.value.rc == code
