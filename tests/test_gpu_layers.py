"""GPU tests of several layers in one submission (moe_ffn_forward_layers) and of capturing this
library's entry points in a caller's CUDA graph.

The chain's output must equal the same layers called one by one, bit for bit (same kernels on
the same inputs; every reduction order is fixed), and each layer must match the oracle on the
state it was given.  Layers 0-2 of the tiny config route by hash, layer 3 by score."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
import synth
from synth.device import upload
from tests.inputs import compare_state

pytestmark = pytest.mark.gpu

BASE = synth.CONFIGS["c0_tiny"]


def _layer_cases(rows):
    """One Case per layer (distinct weights), all on the same token ids."""
    cases = [synth.Case(replace(BASE, rows=rows, layer=l, seed=BASE.seed + 17 * l)) for l in range(BASE.n_layers)]
    for c in cases[1:]:
        c.token_ids = cases[0].token_ids
    return cases


def _handle(cases, max_rows):
    from deepseek_v4_moe_gb300 import MoeFFN, config_from
    devs = [upload(c) for c in cases]
    m = MoeFFN(config_from(BASE, max_rows=max_rows), {l: d["weights"] for l, d in enumerate(devs)})
    return m, devs


@pytest.mark.parametrize("rows,first,n", [(1, 0, 4), (4, 0, 4), (4, 2, 2), (40, 0, 4), (40, 1, 3)])
def test_chain_equals_layer_by_layer_and_oracle(rows, first, n):
    cases = _layer_cases(rows)
    m, devs = _handle(cases, max(rows, 8))
    state, tok = devs[0]["state"], devs[0]["token_ids"]
    ins, outs = [], []
    cur = state
    for l in range(first, first + n):
        ins.append(cur)
        cur = m.forward(cur, tok, l)
        outs.append(cur)
    torch.cuda.synchronize()
    chain = m.forward_layers(state, tok, first, n)
    torch.cuda.synchronize()
    assert torch.equal(chain, outs[-1]), "chain differs from the layers called one by one"
    # every layer against the oracle on the state it was given
    for l, (x, y) in zip(range(first, first + n), zip(ins, outs)):
        case = cases[l]
        case.state = x.cpu().numpy()
        ref = oracle.forward_ffn_rows(case)
        if not case.cfg.is_hash:
            assert ref["margin"].min() > 1e-6, "a near-tie in the chained state"
        compare_state(y.cpu().numpy(), ref["out_state"])
    # a replay reads the buffers' new contents
    state.copy_(torch.flip(state, dims=[0]))
    cur = state
    for l in range(first, first + n):
        cur = m.forward(cur, tok, l)
    again = m.forward_layers(state, tok, first, n, out=chain)
    torch.cuda.synchronize()
    assert torch.equal(again, cur)
    assert m.status() == 0
    m.close()


def test_chain_graph_cache_evicts_and_stays_correct():
    cases = _layer_cases(4)
    m, devs = _handle(cases, 8)
    state, tok = devs[0]["state"], devs[0]["token_ids"]
    ref = m.forward(m.forward(state, tok, 0), tok, 1)
    outs = [torch.empty_like(state) for _ in range(10)]  # ten argument sets: more than the cache keeps
    for rep in range(2):
        for o in outs:
            m.forward_layers(state, tok, 0, 2, out=o)
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o, ref)
    assert m.status() == 0
    m.close()


def test_chain_rejects_bad_ranges():
    from deepseek_v4_moe_gb300 import MoeFFN, MoeFFNError, config_from
    from deepseek_v4_moe_gb300 import _lib as L
    cases = _layer_cases(4)
    devs = [upload(c) for c in cases[:2]]
    m = MoeFFN(config_from(BASE, max_rows=8), {0: devs[0]["weights"], 1: devs[1]["weights"]})
    state, tok = devs[0]["state"], devs[0]["token_ids"]
    for first, n, code in ((0, 0, L.ERR_LAYER_RANGE), (3, 2, L.ERR_LAYER_RANGE), (-1, 2, L.ERR_LAYER_RANGE),
                           (1, 2, L.ERR_NO_WEIGHTS)):
        with pytest.raises(MoeFFNError) as e:
            m.forward_layers(state, tok, first, n)
        assert e.value.code == code, (first, n)
    with pytest.raises(MoeFFNError) as e:
        m.forward_layers(state, tok, 0, 2, out=state)
    assert e.value.code == L.ERR_ALIAS
    torch.cuda.synchronize()
    assert m.status() == 0
    m.close()


@pytest.mark.parametrize("rows", [4, 24])
def test_full_layer_step_captured_in_a_torch_graph(rows):
    # a decode step of two layers as a model would run it: attention HC prelude, the caller's
    # attention (a stand-in in plain torch: an elementwise map of x_norm, so that its own kernels
    # are deterministic too), attention HC post, then the FFN block; captured once in a torch CUDA
    # graph and replayed, it must give the eager result bit for bit
    cases = _layer_cases(rows)
    m, devs = _handle(cases, 32)
    a = cases[0].attn_hc()

    def to_dev(x):
        return torch.from_numpy(x.view(np.int16) if x.dtype == np.uint16 else x).cuda()

    for l in (0, 1):
        m.set_attn_hc(l, {k: to_dev(a[k]) for k in ("hc_fn", "hc_base", "hc_scale", "norm")})
    tok = devs[0]["token_ids"]
    state = devs[0]["state"].clone()

    def step(x):
        for l in (0, 1):
            p = m.hc_pre(x, l, "attn")
            x = m.hc_post(torch.tanh(p["x_norm"]) * 0.5, x, p["post"], p["comb"])
            x = m.forward(x, tok, l)
        return x

    eager = step(state)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(state)  # warm-up on the side stream before capture
    torch.cuda.current_stream().wait_stream(s)
    with torch.cuda.graph(g):
        out = step(state)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    state.copy_(torch.flip(state, dims=[0]))
    g.replay()
    eager2 = step(state)
    torch.cuda.synchronize()
    assert torch.equal(out, eager2)
    assert m.status() == 0
    m.close()
