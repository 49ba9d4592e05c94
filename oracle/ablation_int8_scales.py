"""Scale-granularity ablation of the int8 model, on the oracle (CPU).

TEST INFRASTRUCTURE ONLY: runs the oracle, never the CUDA library.

The quantized GPT-2 abstract reports that one scale per activation row
degraded the output and that scales per 64 consecutive coordinates raised
greedy agreement with the binary32 model from 87 to 120 of 128 prefixes
(pretrained weights, which are not available here).  This script measures
the same agreement on a seeded synthetic GPT-2 124M checkpoint for:

  quant 1  group-64 weight and activation scales (the deployed design)
  quant 3  one weight scale per output row, group-64 activation scales
  quant 4  one weight scale per output row and one scale per projection
           input (the rejected first design)

Protocol: the binary32 model runs greedily from a 16-token seeded prompt
for 128 positions; each int8 model is fed the same 128 tokens (teacher
forcing) and its greedy choice at every position is compared with the
binary32 choice.  Prints one JSON line per model.

    python -m oracle.ablation_int8_scales [--positions 128] [--variant plain|rich|outlier_channels]
"""
from __future__ import annotations

import argparse
import json
import time

import numpy as np

from oracle import Oracle
from stream_decode_gb300 import synth


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--positions", type=int, default=128)
    ap.add_argument("--variant", default="plain", choices=["plain", "rich", "outlier_channels"])
    args = ap.parse_args()
    s = synth.GPT2_124M
    n = min(args.positions, s.max_pos)
    w = synth.checkpoint(s, synth.SEED_124M, args.variant)
    o = Oracle()
    prompt = list(synth.tokens(s.vocab, 16))
    t0 = time.time()
    ref_logits, ref_ch, _ = o.model(s, w, 0).session(prompt + [-1] * (n - 16), n)
    seq = prompt + [int(c) for c in ref_ch[15:n - 1]]
    out = [{"quant": 0, "name": "binary32", "seconds": round(time.time() - t0, 1)}]
    top2 = np.sort(ref_logits, axis=1)[:, -2:]
    margin = top2[:, 1] - top2[:, 0]
    for q, name in ((1, "group-64 weights and activations"), (3, "per-row weights, group-64 activations"),
                    (4, "per-row weights and activations")):
        t0 = time.time()
        lg, ch, _ = o.model(s, w, q).session(seq, n)
        agree = int((ch == ref_ch).sum())
        err = float(np.abs(lg - ref_logits).max())
        out.append({"quant": q, "name": name, "agree": agree, "of": n, "max_abs_logit_diff": err,
                    "median_top2_margin_binary32": float(np.median(margin)),
                    "seconds": round(time.time() - t0, 1)})
    for r in out:
        print(json.dumps(r), flush=True)


if __name__ == "__main__":
    main()
