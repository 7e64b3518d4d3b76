"""Pins of the CPU oracle to facts outside itself: closed forms, hand-worked values,
invariants, special cases that reduce to textbook results, and brute force on tiny inputs.

Each stage of ``forward_ffn_rows`` (docs.rs "hf2q 0.1.3 .../deepseek4/ffn_forward.rs") has at
least one pin that a dropped term, a wrong sign or index, or a transposed operand would fail.
"""
import itertools
import math

import numpy as np
import pytest

import oracle
import synth
from oracle import moe_ffn as O

RNG = np.random.default_rng(12345)


# ---- RMSNorm (rms_norm_no_scale_f32, rms_norm) ------------------------------------------------

def test_rms_no_scale_constant_vector_closed_form():
    eps = 1e-6
    for c in (-3.0, 0.25, 7.5):
        x = np.full((1, 37), c)
        y = O.rms_norm_no_scale(x, eps)
        assert np.allclose(y, np.sign(c) / math.sqrt(1 + eps / (c * c)), rtol=1e-15, atol=0)


def test_rms_norm_hand_value_and_weight():
    x = np.array([[3.0, 4.0]])        # mean square 12.5
    w = np.array([2.0, -1.0])
    y = O.rms_norm(x, w, 0.5)          # sqrt(13) in the denominator
    assert np.allclose(y, [[6 / math.sqrt(13), -4 / math.sqrt(13)]], rtol=1e-15)


# ---- HC mix (raw_matmul "HC FFN function") -----------------------------------------------------

def test_hc_mixes_brute_force_and_flat_index():
    hc, hidden, M = 2, 3, 8
    xn = RNG.standard_normal((2, hc * hidden))
    fn = RNG.standard_normal((M, hc * hidden))
    got = O.hc_mixes(xn, fn)
    for r in range(2):
        for m in range(M):
            ref = 0.0
            for h in range(hc):
                for d in range(hidden):
                    ref += xn[r, h * hidden + d] * fn[m, h * hidden + d]
            assert abs(got[r, m] - ref) < 1e-12


# ---- split + Sinkhorn (dispatch_hc_split_sinkhorn) ---------------------------------------------

def test_split_zero_inputs_give_half_one_and_uniform():
    hc = 4
    pre, post, comb = O.hc_split_sinkhorn(np.zeros((3, 24)), np.array([1.7, -2.0, 3.0]), np.zeros(24), hc, 20)
    assert np.all(pre == 0.5) and np.all(post == 1.0)
    assert np.allclose(comb, 0.25, rtol=0, atol=1e-15)


def test_split_segments_scale_and_base():
    hc = 2
    mixes = np.array([[0.3, -0.7, 1.1, 0.4, 0.0, 0.0, 0.0, 0.0]])
    scale = np.array([2.0, -3.0, 5.0])
    base = np.array([0.1, 0.2, -0.5, 0.6, 0.0, 0.0, 0.0, 0.0])
    pre, post, comb = O.hc_split_sinkhorn(mixes, scale, base, hc, 20)
    s = lambda v: 1 / (1 + math.exp(-v))
    assert np.allclose(pre, [[s(0.3 * 2 + 0.1), s(-0.7 * 2 + 0.2)]], rtol=1e-15)
    assert np.allclose(post, [[2 * s(1.1 * -3 - 0.5), 2 * s(0.4 * -3 + 0.6)]], rtol=1e-15)
    assert np.allclose(comb, 0.5, atol=1e-15)


def test_sinkhorn_one_sweep_hand_worked_2x2():
    # a = [[0, ln 2], [ln 3, 0]]: exp(a - rowmax) = [[1/2, 1], [1, 1/3]]; rows -> [[1/3, 2/3], [3/4, 1/4]];
    # columns sum to 13/12 and 11/12 -> [[4/13, 8/11], [9/13, 3/11]].
    mixes = np.zeros((1, 8))
    mixes[0, 4:] = [0.0, math.log(2), math.log(3), 0.0]
    _, _, comb = O.hc_split_sinkhorn(mixes, np.ones(3), np.zeros(8), 2, 1)
    assert np.allclose(comb[0], [[4 / 13, 8 / 11], [9 / 13, 3 / 11]], rtol=1e-14)
    _, _, c0 = O.hc_split_sinkhorn(mixes, np.ones(3), np.zeros(8), 2, 0)
    assert np.allclose(c0[0], [[0.5, 1.0], [1.0, 1 / 3]], rtol=1e-15)


def test_sinkhorn_last_sweep_is_columns():
    mixes = RNG.standard_normal((5, 24))
    _, _, comb = O.hc_split_sinkhorn(mixes, np.ones(3), np.zeros(24), 4, 3)
    assert np.allclose(comb.sum(axis=1), 1.0, atol=1e-14)


def test_sinkhorn_doubly_stochastic_is_fixed_point():
    P = (0.5 * np.eye(4) + 0.3 * np.roll(np.eye(4), 1, axis=1) + 0.15 * np.roll(np.eye(4), 3, axis=1)
         + 0.05 * np.roll(np.eye(4), 2, axis=1))
    mixes = np.zeros((1, 24))
    mixes[0, 8:] = np.log(P).ravel() + 0.37   # a constant shift cancels
    _, _, comb = O.hc_split_sinkhorn(mixes, np.ones(3), np.zeros(24), 4, 20)
    assert np.allclose(comb[0], P, atol=1e-15)


def test_sinkhorn_hc1_is_one():
    pre, post, comb = O.hc_split_sinkhorn(RNG.standard_normal((3, 3)), np.ones(3), np.zeros(3), 1, 20)
    assert np.all(comb == 1.0)


def test_sinkhorn_invariant_tiny_workload_1e5():
    st = oracle.prelude_and_route(synth.Case(synth.CONFIGS["c0_tiny"]))
    comb = st["comb"]
    assert np.abs(comb.sum(axis=2) - 1).max() < 1e-5
    assert np.abs(comb.sum(axis=1) - 1).max() < 1e-5
    assert np.all(comb > 0)


# ---- hc_pre / hc_post ----------------------------------------------------------------------------

def test_hc_pre_one_hot_and_brute_force():
    state = RNG.standard_normal((2, 3, 5))
    pre = np.array([[0.0, 1.0, 0.0], [0.2, -0.5, 0.9]])
    got = O.hc_pre(state, pre)
    assert np.array_equal(got[0], state[0, 1])
    ref = sum(pre[1, h] * state[1, h] for h in range(3))
    assert np.allclose(got[1], ref, rtol=1e-15)


def test_hc_post_orientation_and_post_term():
    state = RNG.standard_normal((1, 3, 4))
    comb = np.array([[[0.0, 1.0, 0.0], [0.0, 0.0, 2.0], [5.0, 0.0, 0.0]]])   # not symmetric
    out = O.hc_post(np.zeros((1, 4)), state, np.zeros((1, 3)), comb)
    assert np.allclose(out[0, 0], state[0, 1]) and np.allclose(out[0, 1], 2 * state[0, 2])
    assert np.allclose(out[0, 2], 5 * state[0, 0])
    f = RNG.standard_normal((1, 4))
    out2 = O.hc_post(f, state, np.array([[1.0, 0.0, -2.0]]), comb)
    assert np.allclose(out2 - out, [[f[0], 0 * f[0], -2 * f[0]]], rtol=1e-15)


# ---- routing -------------------------------------------------------------------------------------

# ---- router projection (raw_matmul "MoE gate") ---------------------------------------------------

def test_router_logits_brute_force_rows_are_experts():
    # logits[r, e] = sum_d x[r, d] * gate[e, d]: gate rows are experts (a transposed operand or a
    # sum over the wrong axis fails; the shapes are chosen so that both would still run)
    x = RNG.standard_normal((3, 5))
    g = RNG.standard_normal((5, 5))
    got = O.router_logits(x, g)
    for r in range(3):
        for e in range(5):
            assert abs(got[r, e] - sum(x[r, d] * g[e, d] for d in range(5))) < 1e-12
    assert not np.allclose(got, x @ g)


def test_router_logits_of_the_tiny_workload_by_loops():
    # the block's logits are the dots of its own ffn_norm rows with the widened gate rows
    case = synth.Case(synth.CONFIGS["c0_tiny"])
    st = oracle.prelude_and_route(case)
    gate = synth.bf16_bits_to_f32(case.gate).astype(np.float64)
    xf = st["ffn_norm"]
    c = case.cfg
    for r in range(c.rows):
        for e in range(c.experts):
            ref = 0.0
            for d in range(c.hidden):
                ref += xf[r, d] * gate[e, d]
            assert abs(st["logits"][r, e] - ref) < 1e-12 * (1 + abs(ref))


class _HandCase:
    """A one-row block with hc = 1 and zero HC weights (so pre = sigmoid(0) = 1/2), written out."""

    def __init__(self, state_row, norm_w, gate_rows, eps=0.0):
        hidden = len(state_row)
        experts = len(gate_rows)
        from types import SimpleNamespace
        self.cfg = SimpleNamespace(rows=1, hc=1, hidden=hidden, experts=experts, top_k=1, rms_eps=eps,
                                   sinkhorn_iters=20, is_hash=False, vocab=16)
        self.state = np.asarray(state_row, np.float32).reshape(1, 1, hidden)
        self.hc_fn = np.zeros((3, hidden), np.uint16)
        self.hc_scale = np.ones(3, np.float32)
        self.hc_base = np.zeros(3, np.float32)
        self.ffn_norm = np.asarray(norm_w, np.float32)
        self.gate = _bf16_bits(gate_rows)
        self.exp_probs_b = np.zeros(experts, np.float32)
        self.token_ids = np.zeros(1, np.int32)
        self.tid2eid = None


def test_router_reads_the_normalised_input():
    # state [4, 3, 0, 0] -> ffn_input = pre * state = [2, 1.5, 0, 0]; mean square 1.5625, so with
    # eps 0 the RMS is 1.25 and ffn_norm = [1.6, 1.2, 0, 0] * w = [0.8, 1.8, 0, 0] for
    # w = [0.5, 1.5, 1, 1].  Gate rows e0 = d0, e1 = d1: logits [0.8, 1.8] choose expert 1, while
    # the same projection of ffn_input ([2, 1.5]), of the state ([4, 3]) or of the unweighted
    # normalised input ([1.6, 1.2]) would choose expert 0.
    case = _HandCase([4.0, 3.0, 0.0, 0.0], [0.5, 1.5, 1.0, 1.0],
                     [[1.0, 0.0, 0.0, 0.0], [0.0, 1.0, 0.0, 0.0]])
    st = oracle.prelude_and_route(case)
    assert np.allclose(st["pre"], 0.5, rtol=0, atol=0)
    assert np.allclose(st["ffn_input"], [[2.0, 1.5, 0.0, 0.0]], rtol=1e-15)
    assert np.allclose(st["ffn_norm"], [[0.8, 1.8, 0.0, 0.0]], rtol=1e-15)
    assert np.allclose(st["logits"], [[0.8, 1.8]], rtol=1e-15)
    assert st["indices"].tolist() == [[1]] and st["weights"].tolist() == [[1.0]]
    # the eps term sits inside the square root of the norm: eps = 0.4375 makes the RMS sqrt(2)
    st = oracle.prelude_and_route(_HandCase([4.0, 3.0, 0.0, 0.0], [1.0, 1.0, 1.0, 1.0],
                                            [[1.0, 0.0, 0.0, 0.0], [0.0, 1.0, 0.0, 0.0]], eps=0.4375))
    assert np.allclose(st["logits"], [[2 / math.sqrt(2), 1.5 / math.sqrt(2)]], rtol=1e-15)


def test_score_route_brute_force_subsets_tiny():
    case = synth.Case(synth.CONFIGS["c0_tiny"])
    st = oracle.prelude_and_route(case)
    logits, b = st["logits"], case.exp_probs_b.astype(np.float64)
    s = 1 / (1 + np.exp(-logits))
    for r in range(case.cfg.rows):
        best = max(itertools.combinations(range(16), 2), key=lambda S: sum(s[r, e] + b[e] for e in S))
        assert set(best) == set(st["indices"][r].tolist())
        chosen = s[r, st["indices"][r]]
        assert np.allclose(st["weights"][r], chosen / chosen.sum(), rtol=1e-14)
        v = s[r, st["indices"][r]] + b[st["indices"][r]]
        assert v[0] >= v[1]                       # slots in descending biased score
    assert np.allclose(st["weights"].sum(axis=1), 1.0, atol=1e-12)


def test_score_route_bias_selects_but_does_not_weight():
    logits = np.array([[2.0, 1.0, 0.0, -1.0]])
    bias = np.array([0.0, 0.0, 0.0, 0.9], np.float32)
    idx, w = O.score_route(logits, bias, 2)
    # sigmoid(-1)+0.9 = 1.169 > sigmoid(2) = 0.881 > sigmoid(1) = 0.731: expert 3 first, expert 1 out
    assert idx.tolist() == [[3, 0]]
    s0, s3 = 1 / (1 + math.exp(-2)), 1 / (1 + math.exp(1))
    assert np.allclose(w, [[s3 / (s0 + s3), s0 / (s0 + s3)]], rtol=1e-14)


def test_score_route_ties_go_to_lower_index_and_topk_all():
    idx, _ = O.score_route(np.zeros((1, 5)), np.zeros(5, np.float32), 3)
    assert idx.tolist() == [[0, 1, 2]]
    logits = RNG.standard_normal((3, 8))
    idx, w = O.score_route(logits, np.zeros(8, np.float32), 8)
    assert all(sorted(r) == list(range(8)) for r in idx.tolist())
    s = 1 / (1 + np.exp(-logits))
    assert np.allclose(np.sort(w, axis=1), np.sort(s / s.sum(axis=1, keepdims=True), axis=1), rtol=1e-14)


def test_selection_margin():
    logits = np.log(np.array([[0.5, 0.3, 0.2, 0.1]]) / (1 - np.array([[0.5, 0.3, 0.2, 0.1]])))
    m = O.selection_margin(logits, np.zeros(4, np.float32), 2)
    assert abs(m[0] - 0.1) < 1e-6     # gaps 0.2, 0.1 among the top 3


def test_hash_route_is_table_lookup():
    logits = RNG.standard_normal((3, 8))
    table = np.array([[1, 5], [7, 0], [2, 2], [6, 3]], np.int32)
    idx, w = O.hash_route(logits, np.array([3, 0, 1], np.int32), table, vocab=4)
    assert idx.tolist() == [[6, 3], [1, 5], [7, 0]]
    s = 1 / (1 + np.exp(-logits))
    assert np.allclose(w[0], s[0, [6, 3]] / s[0, [6, 3]].sum(), rtol=1e-14)


def test_hash_route_invalid_entries_and_tokens_are_masked():
    logits = RNG.standard_normal((3, 8))
    table = np.array([[1, -1], [9, 2]], np.int32)
    idx, w = O.hash_route(logits, np.array([0, 1, 5], np.int32), table, vocab=2)
    assert idx.tolist() == [[1, -1], [9, 2], [-1, -1]]
    assert w[0, 1] == 0 and w[0, 0] == 1.0 and w[1, 0] == 0 and w[1, 1] == 1.0
    assert np.all(w[2] == 0)
    safe, valid = O.sanitize(idx, 8)
    assert safe.tolist() == [[1, 0], [0, 2], [0, 0]] and valid.tolist() == [[True, False], [False, True], [False, False]]


def test_hash_workload_matches_table():
    cfg = synth.MoeConfig("hash_tiny", rows=5, hidden=64, experts=16, top_k=3, inter=32, shared_inter=32,
                          vocab=100, token_range=100, layer=0, seed=11)
    case = synth.Case(cfg)
    st = oracle.prelude_and_route(case)
    assert np.array_equal(st["indices"], case.tid2eid[case.token_ids])
    assert np.allclose(st["weights"].sum(axis=1), 1.0, atol=1e-12)


# ---- experts and the whole block ---------------------------------------------------------------

def test_swiglu_closed_forms():
    assert O.swiglu(np.array([0.0]), np.array([5.0]))[0] == 0.0
    assert abs(O.swiglu(np.array([1.0]), np.array([2.0]))[0] - 2 / (1 + math.exp(-1))) < 1e-15
    assert abs(O.swiglu(np.array([-2.0]), np.array([1.0]))[0] - (-2 / (1 + math.exp(2)))) < 1e-15


def _dense_block(case):
    """Every expert evaluated for every row with a mask of route weights (brute force)."""
    c = case.cfg
    st = oracle.prelude_and_route(case)
    xf = st["ffn_norm"]
    mask = np.zeros((c.rows, c.experts))
    for r in range(c.rows):
        for k in range(c.top_k):
            e = st["indices"][r, k]
            if 0 <= e < c.experts:
                mask[r, e] += st["weights"][r, k]
    f = np.zeros((c.rows, c.hidden))
    for e in range(c.experts):
        G, U, D = (O.bf16_to_float(case.expert_matrix(w, e)) for w in ("gate", "up", "down"))
        for r in range(c.rows):
            g = np.array([np.dot(xf[r], G[i]) for i in range(c.inter)])
            u = np.array([np.dot(xf[r], U[i]) for i in range(c.inter)])
            a = g / (1 + np.exp(-g)) * u
            f[r] += mask[r, e] * np.array([np.dot(a, D[d]) for d in range(c.hidden)])
    Gs, Us, Ds = (O.bf16_to_float(m) for m in (case.gate_sh, case.up_sh, case.down_sh))
    for r in range(c.rows):
        g, u = Gs @ xf[r], Us @ xf[r]
        f[r] += (g / (1 + np.exp(-g)) * u) @ Ds.T
    out = np.empty((c.rows, c.hc, c.hidden))
    for r in range(c.rows):
        for i in range(c.hc):
            out[r, i] = st["post"][r, i] * f[r] + sum(st["comb"][r, i, j] * st["state"][r, j] for j in range(c.hc))
    return f, out


def test_dense_masked_equals_sparse_tiny():
    case = synth.Case(synth.CONFIGS["c0_tiny"])
    st = oracle.forward_ffn_rows(case)
    f, out = _dense_block(case)
    assert np.allclose(st["ffn_output"], f, rtol=1e-12, atol=1e-13)
    assert np.allclose(st["out_state"], out, rtol=1e-12, atol=1e-13)


def test_zero_route_weights_give_shared_only():
    case = synth.Case(synth.CONFIGS["c0_tiny"])
    st = oracle.prelude_and_route(case)
    st["weights"] = np.zeros_like(st["weights"])
    full = oracle.forward_ffn_rows(case, stages=st)
    Gs, Us, Ds = (O.bf16_to_float(m) for m in (case.gate_sh, case.up_sh, case.down_sh))
    xf = st["ffn_norm"]
    g, u = xf @ Gs.T, xf @ Us.T
    assert np.allclose(full["ffn_output"], (g / (1 + np.exp(-g)) * u) @ Ds.T, rtol=1e-13)


def test_zero_hc_weights_reduce_to_mean_stream_plus_f():
    # hc_fn = 0 and hc_base = 0: pre = 1/2, post = 1, comb = 1/hc, so out_i = f + mean_j state_j
    case = synth.Case(synth.CONFIGS["c0_tiny"])
    case.hc_fn = np.zeros_like(case.hc_fn)
    case.hc_base = np.zeros_like(case.hc_base)
    st = oracle.forward_ffn_rows(case)
    assert np.allclose(st["ffn_input"], 0.5 * case.state.astype(np.float64).sum(axis=1), rtol=1e-14)
    ref = st["ffn_output"][:, None, :] + case.state.astype(np.float64).mean(axis=1, keepdims=True)
    assert np.allclose(st["out_state"], ref, rtol=1e-13, atol=1e-14)


def test_f32_oracle_agrees_with_f64():
    case = synth.Case(synth.CONFIGS["c0_tiny"])
    a = oracle.forward_ffn_rows(case)["out_state"]
    b = oracle.forward_ffn_rows(case, dtype=np.float32)["out_state"]
    assert np.linalg.norm(a - b) / np.linalg.norm(a) < 1e-5


@pytest.mark.parametrize("rows", [[0], [2, 3]])
def test_row_subset_equals_full(rows):
    case = synth.Case(synth.CONFIGS["c0_tiny"])
    full = oracle.forward_ffn_rows(case)
    part = oracle.forward_ffn_rows(case, rows=rows)
    assert np.allclose(full["out_state"][rows], part["out_state"], rtol=1e-14, atol=1e-15)


# ---- HC prelude of a sublayer (attention_forward.rs and ffn_forward.rs, the same five stages) ----

def _bf16_bits(x):
    # exact for values representable in bf16 (0, +-1, powers of two)
    return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_hc_sublayer_pre_hand_worked_hc1():
    # hc = 1, hidden = 2, state [3, 4] (mean square 12.5), eps 0; the mix rows pick the two state
    # columns for pre and post and give comb zero: pre = s(3/sqrt(12.5)), post = 2 s(4/sqrt(12.5)),
    # comb = [[1]], x = pre * [3, 4], x_norm = [3, 4] / sqrt(12.5) * w
    state = np.array([[[3.0, 4.0]]])
    fn = _bf16_bits([[1.0, 0.0], [0.0, 1.0], [0.0, 0.0]])
    w = np.array([2.0, -0.5])
    got = O.hc_sublayer_pre(state, fn, np.ones(3), np.zeros(3), w, hc=1, iters=20, eps=0.0)
    a, b = 3 / math.sqrt(12.5), 4 / math.sqrt(12.5)
    pre = 1 / (1 + math.exp(-a))
    assert abs(got["pre"][0, 0] - pre) < 1e-15
    assert abs(got["post"][0, 0] - 2 / (1 + math.exp(-b))) < 1e-15
    assert got["comb"].shape == (1, 1, 1) and got["comb"][0, 0, 0] == 1.0
    assert np.allclose(got["x"], [[3 * pre, 4 * pre]], rtol=1e-15)
    assert np.allclose(got["x_norm"], [[a * 2.0, b * -0.5]], rtol=1e-14)


def test_hc_sublayer_pre_equal_streams_closed_form():
    # every stream equal to s: x = P s with P = sum_h pre_h, so x_norm = P s / sqrt(P^2 ms + eps) * w
    hc, hidden, eps = 4, 64, 1e-3
    s = RNG.standard_normal((3, hidden))
    state = np.repeat(s[:, None, :], hc, axis=1)
    fn = _bf16_bits(np.where(RNG.random(((2 + hc) * hc, hc * hidden)) < 0.5, 0.0, 0.0625))
    base = RNG.standard_normal((2 + hc) * hc) * 0.1
    w = 1 + 0.05 * RNG.standard_normal(hidden)
    got = O.hc_sublayer_pre(state, fn, np.ones(3), base, w, hc=hc, iters=20, eps=eps)
    P = got["pre"].sum(axis=1, keepdims=True)
    ms = (s * s).mean(axis=1, keepdims=True)
    assert np.allclose(got["x_norm"], P * s / np.sqrt(P * P * ms + eps) * w, rtol=1e-13)
    # and the mixes are the dots of the flat row scaled by its RMS over hc*hidden (= RMS of s)
    m_ref = np.array([[sum(s[r, d] * O.bf16_to_float(fn)[m, h * hidden + d] for h in range(hc) for d in range(hidden))
                       for m in range((2 + hc) * hc)] for r in range(3)]) / np.sqrt(ms + eps)
    assert np.allclose(got["mixes"], m_ref, rtol=1e-12)


def test_hc_sublayer_pre_zero_weights_give_half_sum():
    case = synth.Case(synth.CONFIGS["c0_tiny"])
    a = case.attn_hc()
    st = case.state.astype(np.float64)
    got = O.hc_sublayer_pre(st, np.zeros_like(a["hc_fn"]), a["hc_scale"], np.zeros_like(a["hc_base"]), a["norm"],
                            hc=4, iters=20, eps=1e-6)
    assert np.all(got["pre"] == 0.5) and np.all(got["post"] == 1.0)
    assert np.allclose(got["comb"], 0.25, atol=1e-15)
    assert np.allclose(got["x"], 0.5 * st.sum(axis=1), rtol=1e-15)


def test_hc_sublayer_pre_with_ffn_weights_is_the_ffn_prelude():
    # the FFN sublayer runs the same stages: with its weights the sublayer prelude gives the
    # block's own pre, post, comb, ffn_input and ffn_norm
    case = synth.Case(synth.CONFIGS["c0_tiny"])
    c = case.cfg
    st = oracle.prelude_and_route(case)
    got = O.hc_sublayer_pre(case.state, case.hc_fn, case.hc_scale, case.hc_base, case.ffn_norm, c.hc,
                            c.sinkhorn_iters, c.rms_eps)
    for k, ref in (("pre", "pre"), ("post", "post"), ("comb", "comb"), ("x", "ffn_input"), ("x_norm", "ffn_norm")):
        assert np.array_equal(got[k], st[ref]), k
