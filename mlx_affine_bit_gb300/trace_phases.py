"""Phase times of the one-row width sweep from the phase-trace build.

    python -m mlx_affine_bit_gb300.trace_phases [--steps 6] [--skip 2]

Builds libtfqmm_trace.so (TF_TRACE, include/tfqmm_trace.h) when needed and runs
the width sweep step -- one-row products N = K = 4096 at every width and group
(18 products, the seeded matrices of the bench) -- `steps` times under two launch
modes: "dependent x" (programmatic dependent launch with the weights streamed
before the dependency wait, x read after it) and "early x" (x read before it too;
each product waits only before its first write).  For every product of the steps
after the first `skip`, each CTA's record gives its phases; the script prints, per
mode and width, the median over those CTAs of

    entry->issued   kernel entry to the producer's first stage issued
    issued->landed  that stage's TMA flight (nan where the producer does not wait
                    for it: early-x launches of one or two rows)
    entry->release  entry to consumer thread 0 past the dependency wait
    entry->x        entry to the first x slice placed and summed
    x->stage0       x placed to the first stage's group products done
    stage0->exit    the rest of the CTA's work (later stages, fold, stores)
    CTA             entry to exit

and the step share: the median gap between the previous product's last CTA exit
and this product's last CTA exit (the time the product adds to the step).
Times are %globaltimer nanoseconds; the trace's own stores add a little to each.
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

PHASES = ("entry->issued", "issued->landed", "entry->release", "entry->x", "x->stage0", "stage0->exit", "CTA")
SLOTS = 9
ENTER, TMA0, LAND0, RELEASE, XLOADED, STAGE0, EXIT = range(2, 9)


def phase_table(rec: np.ndarray) -> dict:
    """Per-CTA phase durations (us) of one launch's records (rows of SLOTS words)."""
    t = rec.astype(np.float64) / 1e3
    ok = (t[:, EXIT] > 0) & (t[:, ENTER] > 0)
    t = t[ok]
    d = {
        "entry->issued": t[:, TMA0] - t[:, ENTER],
        "issued->landed": np.where(t[:, LAND0] > 0, t[:, LAND0] - t[:, TMA0], np.nan),
        "entry->release": t[:, RELEASE] - t[:, ENTER],
        "entry->x": t[:, XLOADED] - t[:, ENTER],
        "x->stage0": t[:, STAGE0] - t[:, XLOADED],
        "stage0->exit": t[:, EXIT] - t[:, STAGE0],
        "CTA": t[:, EXIT] - t[:, ENTER],
    }
    return {k: v for k, v in d.items()}


def run(steps: int, skip: int) -> str:
    import torch

    import synth
    import mlx_affine_bit_gb300 as tf
    from mlx_affine_bit_gb300 import build

    build.build_trace()
    L = tf.trace_lib()
    dev = torch.device("cuda", 0)
    N = K = 4096
    cases = synth.width_sweep_cases()
    mats = []
    for (bits, group, seed) in cases:
        m = synth.make_matrix(N, K, bits, group, seed, 0.001, 0.03)
        mats.append((bits, group, torch.from_numpy(m.W.view(np.int32)).to(dev),
                     torch.from_numpy(m.scales.view(np.int16)).to(dev),
                     torch.from_numpy(m.biases.view(np.int16)).to(dev)))
    x = torch.from_numpy(synth.make_x(1, K, 1).view(np.int16)).to(dev)
    ys = [torch.empty((1, N), dtype=torch.float32, device=dev) for _ in mats]
    st = torch.cuda.Stream()
    modes = (("dependent x", tf.TF_LAUNCH_EARLY_WEIGHTS),
             ("early x", tf.TF_LAUNCH_EARLY_WEIGHTS | tf.TF_LAUNCH_EARLY_X))
    out = []
    with tf.using(L):
        for (name, mode) in modes:
            old = tf.tf_set_launch_mode(mode)
            torch.cuda.synchronize()
            if L.tf_trace_reset() != 0:
                raise RuntimeError("tf_trace_reset failed")
            with torch.cuda.stream(st):
                for _ in range(steps):
                    for (bits, group, W, s, b), y in zip(mats, ys):
                        tf.tf_qmm(x, 1, K, W, s, b, N, bits, group, y, N, st)
            torch.cuda.synchronize()
            tf.tf_set_launch_mode(old)
            tf.tf_device_status()
            buf = np.zeros((1 << 16, SLOTS), dtype=np.uint64)
            n = L.tf_trace_read(buf.ctypes.data, buf.shape[0])
            if n < 0:
                raise RuntimeError("tf_trace_read failed")
            buf = buf[:n]
            seq = buf[:, 0].astype(np.int64)
            nl = len(mats) * steps
            last_exit = np.array([buf[seq == i][:, EXIT].max() for i in range(nl)], dtype=np.float64) / 1e3
            rows = []
            for w, (bits, group, *_r) in enumerate(mats):
                per = {k: [] for k in PHASES}
                share = []
                for sidx in range(skip, steps):
                    i = sidx * len(mats) + w
                    d = phase_table(buf[seq == i])
                    for k in PHASES:
                        per[k].extend(d[k].tolist())
                    if i > 0:
                        share.append(last_exit[i] - last_exit[i - 1])
                rows.append((bits, group, {k: float(np.nanmedian(v)) if np.any(np.isfinite(v)) else float("nan")
                                           for k, v in per.items()}, float(np.median(share))))
            step = [last_exit[(s + 1) * len(mats) - 1] - last_exit[s * len(mats) - 1] for s in range(max(skip, 1), steps)]
            out.append("### %s (medians over steps %d..%d; step %.1f us from last exit to last exit)\n"
                       % (name, skip, steps - 1, float(np.median(step))))
            out.append("| bits/G | " + " | ".join(PHASES) + " | step share |")
            out.append("|---" * (len(PHASES) + 2) + "|")
            for (bits, group, med, sh) in rows:
                out.append("| %d/%d | " % (bits, group) + " | ".join("%.2f" % med[k] for k in PHASES) + " | %.2f |" % sh)
            out.append("")
    return "\n".join(out)


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--steps", type=int, default=6)
    ap.add_argument("--skip", type=int, default=2, help="steps left out of the medians (warm-up)")
    a = ap.parse_args()
    print(run(a.steps, a.skip))


if __name__ == "__main__":
    main()
