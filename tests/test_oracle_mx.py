"""Pins of the oracle's MXFP8 weight decoding (the quantised-expert mode of the block).

The format is the OCP Microscaling (MX) one with E4M3 elements: one E8M0 power-of-two scale per 32
consecutive elements of a row.  The decoder (``e4m3_to_float``, ``e8m0_to_float``,
``mxfp8_to_float``) is checked against values fixed by the format's definition, and against the
generator's encoder (synth/gen.c, written separately from the same definition): every finite
code survives encode(decode(code)), and decode(encode(v)) stays within half a step of v."""
import math

import numpy as np
import pytest

import oracle
import synth
from dataclasses import replace
from oracle import moe_ffn as O


def test_e4m3_fixed_points():
    known = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x0F: 1.875 * 2.0 ** -6,
             0x38: 1.0, 0x39: 1.125, 0x3C: 1.5, 0x40: 2.0, 0x48: 4.0, 0x77: 240.0, 0x7E: 448.0,
             0xB8: -1.0, 0xC0: -2.0, 0xFE: -448.0}
    got = O.e4m3_to_float(np.array(list(known), np.uint8))
    assert np.array_equal(got, np.array(list(known.values())))
    assert math.copysign(1.0, O.e4m3_to_float(np.array([0x80], np.uint8))[0]) == -1.0  # -0
    assert np.all(np.isnan(O.e4m3_to_float(np.array([0x7F, 0xFF], np.uint8))))


def test_e8m0_fixed_points():
    got = O.e8m0_to_float(np.array([127, 128, 130, 120, 0, 254, 255], np.uint8))
    assert np.array_equal(got[:6], [1.0, 2.0, 8.0, 2.0 ** -7, 2.0 ** -127, 2.0 ** 127])
    assert np.isnan(got[6])


def test_every_finite_code_round_trips_through_the_generator_encoder():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF, 0x80)], np.uint8)
    vals = O.e4m3_to_float(codes)
    # blocks of 32 values whose largest magnitude is 448, so the shared scale is 2^0 (code 127)
    pad = (-len(vals)) % 31
    v = np.concatenate([vals, np.zeros(pad)]).reshape(-1, 31)
    blocks = np.concatenate([np.full((v.shape[0], 1), 448.0), v], axis=1).astype(np.float32)
    q, s = synth.quantize_mxfp8(blocks)
    assert np.all(s == 127)
    assert np.array_equal(q.reshape(-1, 32)[:, 1:].ravel()[: len(codes)], codes)


def test_decode_of_encode_is_within_half_a_step():
    rng = np.random.default_rng(7)
    v = (rng.standard_normal(32 * 400) * np.exp2(rng.integers(-20, 10, 32 * 400))).astype(np.float32)
    q, s = synth.quantize_mxfp8(v)
    X = O.e8m0_to_float(np.repeat(s, 32))
    deq = O.mxfp8_to_float(q.reshape(400, 32), s.reshape(400, 1)).ravel()
    a = np.abs(v.astype(np.float64))
    # the shared exponent puts every block's largest value in [256, 512) X
    amax = a.reshape(400, 32).max(axis=1)
    assert np.all((amax / X[::32] >= 256) & (amax / X[::32] < 512))
    within = a <= 448 * X
    bound = np.maximum(2.0 ** -4 * a, 2.0 ** -10 * X)  # half a step: relative 2^-4 (3 bits), 2^-10 X below 2^-6 X
    assert np.all(np.abs(deq - v)[within] <= bound[within])
    assert np.array_equal(deq[~within], np.sign(v[~within]) * 448 * X[~within])  # saturation


def test_scales_apply_per_block_of_32_along_the_row():
    q = np.full((2, 64), 0x38, np.uint8)  # every element 1.0
    s = np.array([[127, 130], [120, 1]], np.uint8)
    got = O.mxfp8_to_float(q, s)
    for r in range(2):
        for k in range(64):
            assert got[r, k] == 2.0 ** (int(s[r, k // 32]) - 127)


def test_mx_workload_is_the_bf16_one_up_to_quantisation():
    cfg = synth.CONFIGS["c0_tiny"]
    case_b = synth.Case(cfg)
    case_m = synth.Case(replace(cfg, weights="mxfp8"))
    # the same draws: an MX element is within 2^-4 of bf16's value, or 1/8 for a block maximum
    # clamped to 448 X (the format's rule puts it in [256, 512) X), plus bf16's own rounding
    g_b = O.bf16_to_float(case_b.expert_matrix("gate", 5))
    g_m = O.expert_weights(case_m, "gate", 5)
    assert np.all(np.abs(g_m - g_b) <= 0.126 * np.abs(g_b) + 2.0 ** -20)
    assert not np.array_equal(g_m, g_b)
    a = oracle.forward_ffn_rows(case_b)["out_state"]
    b = oracle.forward_ffn_rows(case_m)["out_state"]
    rel = np.linalg.norm(a - b) / np.linalg.norm(a)
    assert 1e-5 < rel < 0.05, rel
