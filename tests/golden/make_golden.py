"""Write the stored expected values under tests/golden/ from the CPU oracle only.

The pages print no worked numeric example for this method (they report ratios,
accuracies and speedups only), so the stored values here are the oracle's own
results on the small decode workload (context 4096, block 64, fp32, two needle
blocks; "Faster Than Flash" Sec. 1-3 for the scan-then-attend decode, "How Much
Dense Attention is Necessary?" Sec. 2.1 for exact attention on the selected
support).  They pin the oracle against accidental change: any later change to
its arithmetic has to regenerate them, with the passage that justifies it.

Run:  python tests/golden/make_golden.py
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import synth  # noqa: E402


def c1_decode_lines():
    wl = synth.WORKLOADS["c1"]
    x = synth.make_inputs(wl)
    idx, cnt, s, _ = oracle.decode_select(x.q, x.k, wl)
    rows = [(0, 0, h) for h in range(wl.Hq)]
    out, lse = oracle.attend(x.q, x.k, x.v, wl.Hkv, wl.L, wl.L - wl.T, wl.Bk, wl.scale, rows, idx, cnt)
    lines = ["# c1 decode: B=1 T=1 Hq=4 Hkv=1 d=64 L=4096 Bk=64 k=8, fp32, seed %d" % wl.seed,
             "needles " + " ".join(str(b) for b in np.nonzero(x.needle_mask[0])[0]),
             "selected " + " ".join(str(b) for b in idx[0, : cnt[0]]),
             "scores " + " ".join("%.17g" % v for v in s[0])]
    for h in range(wl.Hq):
        lines.append("lse %d %.17g" % (h, lse[h]))
        lines.append("out %d " % h + " ".join("%.17g" % v for v in out[h]))
    return lines


def c1_token_decode_lines():
    """Head-collapsed token-level support on the small decode workload at 512 tokens
    ("How Much Dense Attention is Necessary?" Sec. 2.1-2.2): the mass of the selected
    tokens, the selection (top-32 + tokens 0 and 511) and the outputs over it."""
    wl = synth.WORKLOADS["c1"].replace(L=512, k=32)
    x = synth.make_inputs(wl)
    P = oracle.token_mass_decode(x.q, x.k, wl.Hkv, wl.L, wl.scale)
    idx, cnt = oracle.token_select(P, wl.k)
    sel = idx[0, : cnt[0]]
    rows = [(0, 0, h) for h in range(wl.Hq)]
    out, lse = oracle.token_attend(x.q, x.k, x.v, wl.Hkv, wl.L, wl.scale, idx, cnt, rows)
    lines = ["# c1 token decode: B=1 T=1 Hq=4 Hkv=1 d=64 L=512, top-32 tokens + 0 + 511, fp32, seed %d" % wl.seed,
             "selected " + " ".join(str(j) for j in sel),
             "mass " + " ".join("%.17g" % P[0, j] for j in sel),
             "masssum %.17g" % P[0].sum()]
    for h in range(wl.Hq):
        lines.append("lse %d %.17g" % (h, lse[h]))
        lines.append("out %d " % h + " ".join("%.17g" % v for v in out[h]))
    return lines


def main():
    with open(os.path.join(HERE, "c1_decode.txt"), "w") as f:
        f.write("\n".join(c1_decode_lines()) + "\n")
    with open(os.path.join(HERE, "c1_token_decode.txt"), "w") as f:
        f.write("\n".join(c1_token_decode_lines()) + "\n")


if __name__ == "__main__":
    main()
