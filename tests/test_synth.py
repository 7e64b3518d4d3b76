"""The workload generator: determinism, independence of streams, and the shape of its
distributions (it holds none of the block's arithmetic)."""
import numpy as np

import synth


def test_deterministic_and_offset_consistent():
    a = synth.normal_f32(7, synth.T_STATE, 1000)
    b = synth.normal_f32(7, synth.T_STATE, 1000)
    assert np.array_equal(a, b)
    c = synth.normal_f32(7, synth.T_STATE, 500, start=500)
    assert np.array_equal(a[500:], c)
    assert not np.array_equal(a, synth.normal_f32(8, synth.T_STATE, 1000))
    assert not np.array_equal(a, synth.normal_f32(7, synth.T_GATE, 1000))


def test_normal_moments_and_tails():
    z = synth.normal_f32(3, synth.T_GATE, 1 << 22).astype(np.float64)
    assert abs(z.mean()) < 3e-3
    assert abs(z.std() - 1.0) < 3e-3
    k = np.mean((z - z.mean()) ** 4) / z.var() ** 2 - 3  # a normal's excess kurtosis is 0
    assert abs(k) < 0.03
    # tails of a true normal: P(|z| > 3.5) = 4.65e-4, P(|z| > 4) = 6.33e-5 (unbounded, unlike a
    # sum of a few uniforms); counts within 5 binomial standard deviations
    for t, p in ((3.5, 4.6525e-4), (4.0, 6.3342e-5)):
        n, c = z.size, int(np.sum(np.abs(z) > t))
        assert abs(c - n * p) < 5 * np.sqrt(n * p), (t, c, n * p)
    assert np.abs(z).max() > 4.5


def test_normal_against_the_normal_cdf():
    # Kolmogorov-Smirnov distance of 2^20 draws from Phi, written with math.erf
    import math
    z = np.sort(synth.normal_f32(11, synth.T_STATE, 1 << 20).astype(np.float64))
    cdf = 0.5 * (1.0 + np.vectorize(math.erf)(z / math.sqrt(2.0)))
    n = z.size
    d = max(np.max(np.arange(1, n + 1) / n - cdf), np.max(cdf - np.arange(n) / n))
    assert d < 1.63 / np.sqrt(n)  # the 1 % critical value


def test_pairs_split_across_calls_and_rows():
    # an odd start takes the second member of a pair; row draws equal flat draws of the same stream
    a = synth.normal_f32(9, synth.T_STATE, 4099)
    for s0, n in ((1, 7), (2047, 3), (2048, 2051), (4097, 2)):
        assert np.array_equal(a[s0:s0 + n], synth.normal_f32(9, synth.T_STATE, n, start=s0))
    rows = synth.normal_rows_f32(9, synth.T_STATE, np.zeros(2, np.int32), 2049)
    assert np.array_equal(rows.ravel(), a[: 2 * 2049])


def test_bf16_is_round_to_nearest_even_of_f32_draw():
    n = 4096
    f = synth.normal_f32(5, synth.T_HC_FN, n, 0.0, 0.02)
    b = synth.normal_bf16(5, synth.T_HC_FN, n, 0.02)
    # independent RNE: pick the nearer of the two bf16 neighbours, ties to even mantissa
    u = f.view(np.uint32).astype(np.uint64)
    lo = (u >> 16) << 16
    hi = lo + (1 << 16)
    dlo = np.abs(f.astype(np.float64) - (lo.astype(np.uint32)).view(np.float32).astype(np.float64))
    dhi = np.abs((hi.astype(np.uint32)).view(np.float32).astype(np.float64) - f.astype(np.float64))
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (((lo >> 16) & 1) == 1))
    ref = np.where(pick_hi, hi >> 16, lo >> 16).astype(np.uint16)
    assert np.array_equal(ref, b)


def test_gain_applied_before_rounding():
    f = synth.normal_f32(5, synth.T_GATE, 64, 0.0, 0.02).astype(np.float64) * 3.0
    b = synth.bf16_bits_to_f32(synth.normal_bf16(5, synth.T_GATE, 64, 0.02, gain=3.0))
    assert np.max(np.abs(b - f) / np.abs(f)) <= 2.0 ** -8


def test_uniform_int_range_and_distinct_rows():
    t = synth.uniform_i32(1, synth.T_TOKENS, 100000, 0, 129280)
    assert t.min() >= 0 and t.max() < 129280
    assert abs(t.mean() / 129280 - 0.5) < 0.01
    rows = synth.distinct_rows_i32(2, synth.T_TID2EID, 5000, 6, 256)
    assert rows.min() >= 0 and rows.max() < 256
    assert all(len(set(r)) == 6 for r in rows)
    counts = np.bincount(rows.ravel(), minlength=256)
    assert counts.min() > 0.7 * counts.mean()


def test_permutation():
    p = synth.permutation(4, synth.T_HOT, 256)
    assert sorted(p.tolist()) == list(range(256))
    assert not np.array_equal(p, np.arange(256))


def test_case_shapes_tiny():
    c = synth.Case(synth.CONFIGS["c0_tiny"])
    cfg = c.cfg
    assert c.state.shape == (4, 4, 256) and c.state.dtype == np.float32
    assert c.hc_fn.shape == (24, 1024) and c.hc_fn.dtype == np.uint16
    assert c.gate.shape == (16, 256)
    assert c.expert_matrix("gate", 3).shape == (128, 256)
    assert c.expert_matrix("down", 3).shape == (256, 128)
    assert c.token_ids.max() < 1024
    blk = np.empty(2 * cfg.inter * cfg.hidden, np.uint16)
    c.expert_block("up", 2, 2, blk)
    assert np.array_equal(blk[: cfg.inter * cfg.hidden].reshape(cfg.inter, cfg.hidden), c.expert_matrix("up", 2))


def test_attempts_redraw_only_that_row():
    cfg = synth.CONFIGS["c0_tiny"]
    a = synth.Case(cfg)
    b = synth.Case(cfg, attempts=np.array([0, 1, 0, 0]))
    assert np.array_equal(a.state[0], b.state[0]) and np.array_equal(a.state[2:], b.state[2:])
    assert not np.array_equal(a.state[1], b.state[1])


def test_hot_experts_scaled():
    cfg = synth.MoeConfig("hot_tiny", rows=2, hidden=64, experts=16, top_k=2, inter=32, shared_inter=32,
                          vocab=64, token_range=64, seed=9, hot_experts=3)
    c = synth.Case(cfg)
    plain = synth.Case(synth.MoeConfig("cold_tiny", rows=2, hidden=64, experts=16, top_k=2, inter=32,
                                       shared_inter=32, vocab=64, token_range=64, seed=9))
    g, g0 = synth.bf16_bits_to_f32(c.gate), synth.bf16_bits_to_f32(plain.gate)
    assert len(c.hot) == 3
    for e in range(16):
        if e in c.hot:
            assert np.allclose(g[e], 3 * g0[e], rtol=2 ** -7, atol=0)
        else:
            assert np.array_equal(g[e], g0[e])


def test_zipf_targets_capped_and_normalised():
    p = synth.zipf_targets(synth.CONFIGS["c3_prefill_512"])
    assert abs(p.sum() - 1) < 1e-12
    assert p.max() <= 1 / 6 + 1e-12
    order = np.sort(p)[::-1]
    # below the cap the shares follow rank^-1.1
    assert abs(order[5] / order[10] - (11 / 6) ** 1.1) < 1e-9


def test_mx_experts_chunked_equal_per_expert_and_deterministic():
    # upload_mx draws experts in chunks; each chunk must equal the per-expert matrices
    from dataclasses import replace
    cfg = replace(synth.CONFIGS["c0_tiny"], weights="mxfp8")
    c = synth.Case(cfg)
    per = cfg.inter * cfg.hidden
    q = np.empty(3 * per, np.uint8)
    s = np.empty(3 * per // 32, np.uint8)
    c.expert_block_mx("down", 4, 3, q, s)
    for k in range(3):
        eq, es = c.expert_matrix_mx("down", 4 + k)
        assert eq.shape == (cfg.hidden, cfg.inter) and es.shape == (cfg.hidden, cfg.inter // 32)
        assert np.array_equal(q[k * per:(k + 1) * per], eq.ravel())
        assert np.array_equal(s[k * per // 32:(k + 1) * per // 32], es.ravel())
    q2, s2 = synth.Case(cfg).expert_matrix_mx("down", 5)
    assert np.array_equal(q2, c.expert_matrix_mx("down", 5)[0]) and np.array_equal(s2, c.expert_matrix_mx("down", 5)[1])
    sq, ss = c.shared_mx("gate")
    assert sq.shape == (cfg.shared_inter, cfg.hidden) and ss.shape == (cfg.shared_inter, cfg.hidden // 32)
