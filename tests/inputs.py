"""Test inputs: the generator's workloads with near-tied router rows redrawn.

A score-routed row whose selection scores (sigmoid(logit) + bias, f32) have two values within
``margin`` of each other among the top_k + 1 largest is redrawn (a new attempt number for that state
row only): such a near-tie could put different experts, or the same experts in a different slot
order, in the top_k of two correct implementations.  The margins come from the oracle.
"""
from __future__ import annotations

import numpy as np

import oracle
import synth

MARGIN = 1e-5


def tie_free(cfg, margin: float = MARGIN, max_rounds: int = 50):
    """Returns (case, stages) with every row's selection margin >= margin; stages are the oracle's
    prelude + routing outputs for all rows of the returned case."""
    if isinstance(cfg, str):
        cfg = synth.CONFIGS[cfg]
    case = synth.Case(cfg)
    st = oracle.prelude_and_route(case)
    if cfg.is_hash:
        return case, st
    for _ in range(max_rounds):
        bad = np.flatnonzero(st["margin"] < margin)
        if bad.size == 0:
            return case, st
        att = case.attempts.copy()
        att[bad] += 1
        case = case.with_attempts(att)
        part = oracle.prelude_and_route(case, rows=bad)
        for k, v in part.items():
            if k != "rows" and isinstance(v, np.ndarray) and v.shape[:1] == (len(bad),):
                st[k][bad] = v
    raise RuntimeError("could not draw a tie-free workload")


def sample_rows(rows: int, n: int, seed: int = 0) -> np.ndarray:
    """First, last and a seeded spread of rows in between."""
    if rows <= n:
        return np.arange(rows)
    rng = np.random.default_rng(seed)
    mid = rng.choice(np.arange(1, rows - 1), size=n - 2, replace=False)
    return np.sort(np.concatenate([[0, rows - 1], mid]))


def substages(st: dict, rows: np.ndarray) -> dict:
    out = {}
    for k, v in st.items():
        out[k] = v[rows] if isinstance(v, np.ndarray) and v.ndim >= 1 and k != "rows" else v
    out["rows"] = np.asarray(st["rows"])[rows]
    return out


def compare_state(got: np.ndarray, ref: np.ndarray, rel_l2: float = 1e-3, max_frac: float = 1e-2):
    """The output-state tolerance: relative L2 <= rel_l2 and max |delta| <= max_frac * RMS(ref)."""
    got = got.astype(np.float64)
    diff = got - ref
    rl2 = np.linalg.norm(diff) / np.linalg.norm(ref)
    rms = np.sqrt(np.mean(ref * ref))
    mx = np.abs(diff).max()
    assert rl2 <= rel_l2, f"relative L2 {rl2:.3e} > {rel_l2}"
    assert mx <= max_frac * rms, f"max |delta| {mx:.3e} > {max_frac} * RMS {rms:.3e}"
    return rl2, mx / rms


def compare_dot(got: np.ndarray, ref: np.ndarray, x: np.ndarray, w: np.ndarray, tau: float, what: str = ""):
    """A tolerance for f32 dot products ref = x @ w.T, scaled by each entry's condition.

    An entry's f32 error is bounded by a multiple of sum_d |x_d * w_d| (the rounding of every
    partial sum and of x itself is relative to that magnitude, not to the result), so the bar is
    |got - ref| <= tau * (|x| @ |w|.T).  Entries near zero after cancellation get the same absolute
    slack as their terms deserve.  Returns the largest |delta| / bound ratio seen (<= 1 passes)."""
    cond = np.abs(x.astype(np.float64)) @ np.abs(w.astype(np.float64)).T
    diff = np.abs(got.astype(np.float64) - ref)
    ratio = diff / (tau * cond + 1e-30)
    worst = np.unravel_index(np.argmax(ratio), ratio.shape)
    assert ratio[worst] <= 1.0, (f"{what} |delta| {diff[worst]:.3e} at {worst} > {tau:g} x condition "
                                 f"{cond[worst]:.3e} (ratio {ratio[worst]:.2f})")
    return float(ratio[worst])


def compare_scaled(got: np.ndarray, ref: np.ndarray, cond: np.ndarray, tau: float, what: str = ""):
    """|got - ref| <= tau * cond elementwise, cond an entry's own error scale (the magnitude its
    inputs carry before any cancellation); the message names the worst entry."""
    diff = np.abs(got.astype(np.float64) - ref)
    ratio = diff / (tau * cond + 1e-30)
    worst = np.unravel_index(np.argmax(ratio), ratio.shape)
    assert ratio[worst] <= 1.0, (f"{what} |delta| {diff[worst]:.3e} at {worst} (got {got[worst]:.8g}, ref "
                                 f"{ref[worst]:.8g}) > {tau:g} x scale {cond[worst]:.3e}")
    return float(ratio[worst])
