"""The bench's algorithmic byte models (CPU): the per-kernel byte figures its JSON line reports."""
from dataclasses import replace

import numpy as np

import bench
import synth


def _c1_indices():
    return np.array([[3, 17, 40, 99, 150, 201]], np.int32)  # 6 distinct routed experts, like c1's draw


def test_decode_bytes_match_the_reported_figures():
    cfg = synth.CONFIGS["c1_decode_b1"]
    wm = bench.work_model(cfg, _c1_indices())
    assert wm["groups"] == 7
    nbytes, _ = bench.kernel_work("decode", wm, cfg)
    assert nbytes == 355_680_256                         # 355.7 MB per launch (bf16)
    mx = replace(cfg, weights="mxfp8")
    wmx = bench.work_model(mx, _c1_indices())
    assert abs(wmx["w_gateup"] / wm["w_gateup"] - (1 + 1 / 32) / 2) < 1e-9
    assert abs(wmx["w_down"] / wm["w_down"] - (1 + 1 / 32) / 2) < 1e-9
    nbytes_mx, _ = bench.kernel_work("decode", wmx, mx)
    assert nbytes_mx == 185_024_512                      # 184.7 MB of forward bytes + the act/y trips


def test_hc_sublayer_bytes():
    cfg = synth.CONFIGS["c4_prefill_4096"]
    pre, post = bench.hc_sublayer_bytes(cfg)
    R, D, HC, M = cfg.rows, cfg.hidden, cfg.hc, cfg.mix
    assert pre == R * HC * D * 4 + M * HC * D * 2 + D * 4 + R * D * 4 + R * (2 * HC + HC * HC) * 4
    assert post == R * D * 4 + 2 * R * HC * D * 4 + R * (HC + HC * HC) * 4
    assert post == 604_307_456 and pre == 336_740_352  # the figures of the 4096-row table
