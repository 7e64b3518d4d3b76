"""Writes zipf_exp_probs_b_seed3.txt: the selection bias (exp_probs_b) of the 512-row prefill
workload, calibrated so that the share of routed slots each expert receives follows Zipf(1.1)
over a seeded permutation of the 256 experts (water-filled at 1/top_k, since a token picks an
expert at most once).

It calls only the oracle (router logits and the top-k rule) and the input generator.  The
calibration runs on the workload's own 512 state rows: logits are computed once, then the bias is
moved toward the target in log-share space for a fixed number of rounds.

    python tests/golden/make_zipf_bias.py
"""
import os
import sys
from dataclasses import replace

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402

ROUNDS, STEP = 400, 0.02


def main():
    cfg = synth.CONFIGS["c3_prefill_512"]
    case = synth.Case(replace(cfg, bias="normal"))
    logits = oracle.prelude_and_route(case)["logits"]
    target = synth.zipf_targets(cfg)
    slots = cfg.rows * cfg.top_k
    b = np.zeros(cfg.experts)
    for _ in range(ROUNDS):
        idx = oracle.topk_desc(oracle.selection_scores(logits, b.astype(np.float32)), cfg.top_k)
        share = np.bincount(idx.ravel(), minlength=cfg.experts) / slots
        b += STEP * (np.log(target) - np.log(share + 0.25 / slots))
        b -= b.mean()
    b32 = b.astype(np.float32)
    idx = oracle.topk_desc(oracle.selection_scores(logits, b32), cfg.top_k)
    share = np.bincount(idx.ravel(), minlength=cfg.experts) / slots
    tv = 0.5 * np.abs(share - target).sum()
    path = synth.ZIPF_BIAS_FILE
    with open(path, "w") as fh:
        fh.write("# exp_probs_b for the 512-row Zipf(1.1) prefill workload (seed 3), float32 values\n")
        fh.write(f"# written by tests/golden/make_zipf_bias.py: {ROUNDS} rounds, step {STEP}; on the workload's "
                 f"rows the slot shares are within total-variation {tv:.4f} of the target\n")
        fh.write(f"# top expert share {share.max():.4f} (target {target.max():.4f}); experts touched "
                 f"{int((share > 0).sum())}\n")
        for v in b32:
            fh.write(f"{float(v):.9g}\n")
    print(f"wrote {path}: TV {tv:.4f}, touched {(share > 0).sum()}")


if __name__ == "__main__":
    main()
