"""Writes the golden fixtures under tests/golden/ from the oracle alone.

Inputs: the packed.rs (hanzo-kernel 0.2.42) test fixture -- `mod tests`: LENS = [5, 40, 1,
33, 70], HEADS = 2, qkv = rnd(T * 3 * HEADS * 64, seed 7, amp 1.0) (xorshift64), tables(128)
with base 10000, scale 64^-0.5, inputs rounded to bf16 before the f64 composite sees them,
windows None / 8 / 64 (fn forward). The expected values are the oracle's (fp64), stored with
17 significant digits; they are a regression fixture, not a pin of the oracle.

Run from the repository root:  python tests/golden/make_golden.py
"""

import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import synth  # noqa: E402

ROWS = (0, 4, 5, 44, 45, 46, 78, 79, 110, 148)


def main():
    orc = oracle.get()
    for w in (0, 8, 64):
        wl = synth.p1_fixture("bf16", w)
        out, lse = orc.attend(wl.qkv, wl.cos, wl.sin, wl.cu, wl.H, w, wl.scale, "bf16")
        path = os.path.join(HERE, f"p1_fixture_bf16_w{w}.txt")
        with open(path, "w") as f:
            f.write(f"# packed.rs mod tests fixture, bf16 inputs, window {w or 'None'}\n")
            f.write("# written by tests/golden/make_golden.py from the fp64 oracle\n")
            f.write(f"lens {' '.join(str(x) for x in synth.P1_LENS)}\n")
            f.write(f"heads {wl.H}\nwindow {w}\nscale {wl.scale!r}\n")
            for h in range(wl.H):
                f.write(f"lse {h} " + " ".join(f"{v:.17g}" for v in lse[h]) + "\n")
            for a in ROWS:
                f.write(f"out {a} " + " ".join(f"{v:.17g}" for v in out[a]) + "\n")
        print("wrote", path)


if __name__ == "__main__":
    main()
