"""The stage layout's row pad (seg_pad_words in qmm_common.h) against a model of
the consumers' shared-memory code loads.

A warp's 32 lanes are 8 rows g x 4 quarters q of an m-tile; lane (g, q) of run
m reads, in row g + 8h, the 32-bit words from ((q*G/4 + 8m) * bits) / 32 on: one
word (2/4-bit), two words as two loads (3/5/6/8-bit), or, for 4/8-bit with two or
more runs a group, the group's words as one 8- or 16-byte vector load.  6-bit
lanes of groups 32 / 128 with q even / q < 2 load the second word first.  The
model counts the distinct words each bank serves per access phase (32, 16 or 8
lanes for 4, 8 or 16 bytes); the chosen pad must reach the smallest worst case
over the pads a TMA box allows (multiples of 4 words)."""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SEG = 256
PROBE = r'''
#include <cstdio>
#include "qmm_common.h"
int main() {
    const int bits[] = {2, 3, 4, 5, 6, 8}, groups[] = {32, 64, 128};
    for (int b : bits) for (int g : groups) printf("%d %d %d\n", b, g, tfq::seg_pad_words(b, g));
}
'''


def _pads(tmp_path):
    src = tmp_path / "pad.cpp"
    src.write_text(PROBE)
    exe = str(tmp_path / "pad")
    inc = os.path.join(ROOT, "mlx_affine_bit_gb300", "csrc")
    cuda_inc = "/usr/local/cuda/include"
    if not os.path.exists(os.path.join(cuda_inc, "cuda.h")):
        pytest.skip("cuda.h not available")
    subprocess.check_call(["g++", "-std=c++17", "-I" + inc, "-I" + cuda_inc, str(src), "-o", exe])
    out = subprocess.check_output([exe]).decode().split()
    vals = list(map(int, out))
    return {(vals[i], vals[i + 1]): vals[i + 2] for i in range(0, len(vals), 3)}


def _swap(bits, group, q):
    return bits == 6 and ((group == 32 and q % 2 == 0) or (group == 128 and q < 2))


def _worst(bits, group, pad):
    """Worst bank multiplicity (distinct words on one bank in one phase) of a warp's loads."""
    segw = SEG * bits // 32
    rw = segw + pad
    qg, runs = group // 4, group // 32
    vec = bits in (4, 8) and runs >= 2
    worst = 0

    def phase_worst(addrs, width):
        per = 32 // width                      # lanes per phase
        w = 0
        for p0 in range(0, 32, per):
            banks = {}
            for lane in range(p0, p0 + per):
                for j in range(width):
                    a = addrs[lane] + j
                    banks.setdefault(a % 32, set()).add(a)
            w = max(w, max(len(v) for v in banks.values()))
        return w

    for gi in range(SEG // group):
        woff = gi * group * bits // 32
        for h in (0, 8):
            if vec:
                vw = runs * bits // 4                          # words of the lane's runs
                step = 4 if vw >= 4 else 2
                for v in range(0, vw, step):
                    addrs = [((l >> 2) + h) * rw + woff + (((l & 3) * qg * bits) >> 5) + v for l in range(32)]
                    worst = max(worst, phase_worst(addrs, step))
                continue
            nwords = 1 if bits in (2, 4) else 2
            for m in range(runs):
                for j in range(nwords):
                    addrs = []
                    for l in range(32):
                        g, q = l >> 2, l & 3
                        wo = ((q * qg + 8 * m) * bits) >> 5
                        jj = (1 - j) if (nwords == 2 and _swap(bits, group, q)) else j
                        addrs.append((g + h) * rw + woff + wo + jj)
                    worst = max(worst, phase_worst(addrs, 1))
    return worst


def test_chosen_pads_reach_the_least_conflicts(tmp_path):
    pads = _pads(tmp_path)
    assert len(pads) == 18
    for (bits, group), pad in pads.items():
        assert pad % 4 == 0 and 4 <= pad <= 16, (bits, group, pad)
        best = min(_worst(bits, group, p) for p in (4, 8, 12, 16))
        assert _worst(bits, group, pad) == best, (bits, group, pad, best)


def test_six_bit_word_order_is_conflict_free():
    # with the per-lane word order the 6-bit loads meet no bank twice at any group
    for group in (32, 64, 128):
        assert _worst(6, group, 4) == 1, group
