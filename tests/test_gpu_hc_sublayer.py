"""GPU parity of the hyper-connection prelude and post of a sublayer (moe_ffn_hc_pre /
moe_ffn_hc_post) against the oracle: the attention sublayer (docs.rs "hf2q 0.1.3
.../deepseek4/attention_forward.rs": HC attention function, split + Sinkhorn, hc_pre, attn_norm,
and hc_post on the output projection) and the FFN sublayer's prelude on its own.  Rows <= 4 take
the split-K mix kernel, larger batches the tensor-core split GEMM; both are covered, with tails
that are not whole tiles."""
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
CASES = {
    "tiny": (BASE, [1, 2, 4, 5, 33, 300]),
    "full_width": (replace(BASE, hidden=4096, seed=31), [1, 4, 130]),
    "hc2_d384": (replace(BASE, hc=2, hidden=384, seed=32), [3, 70]),
    "hc1_d128": (replace(BASE, hc=1, hidden=128, seed=33), [1, 9]),
}
PARAMS = [(n, r) for n, (_, rows) in CASES.items() for r in rows]


def _dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def _attn_handle(cfg, max_rows, layer=1):
    from deepseek_v4_moe_gb300 import MoeFFN, config_from
    case = synth.Case(replace(cfg, rows=max_rows))
    a = case.attn_hc()
    w = {k: _dev(a[k]) for k in ("hc_fn", "hc_base", "hc_scale", "norm")}
    m = MoeFFN(config_from(cfg, max_rows=max_rows), {})
    m.set_attn_hc(layer, w)
    return m, case, w


def _check_pre(got, ref):
    for k in ("pre", "post", "comb"):
        g = got[k].cpu().numpy()
        assert np.allclose(g, ref[k], rtol=1e-5, atol=1e-6), k
    assert np.allclose(got["x_norm"].cpu().numpy(), ref["x_norm"], rtol=1e-4, atol=1e-5)
    compare_state(got["x_norm"].cpu().numpy(), ref["x_norm"])


@pytest.mark.parametrize("name,rows", PARAMS, ids=[f"{n}-r{r}" for n, r in PARAMS])
def test_attn_hc_pre_and_post_against_oracle(name, rows):
    cfg, all_rows = CASES[name]
    m, case, _ = _attn_handle(cfg, max(all_rows))
    c = case.cfg
    a = case.attn_hc()
    state = case.state[:rows]
    ref = oracle.hc_sublayer_pre(state, a["hc_fn"], a["hc_scale"], a["hc_base"], a["norm"], c.hc,
                                 c.sinkhorn_iters, c.rms_eps)
    st = _dev(state)
    got = m.hc_pre(st, layer=1, sublayer="attn")
    torch.cuda.synchronize()
    _check_pre(got, ref)
    # hc_post on the attention output stand-in, with the device's own post and comb (f32) given to
    # both sides, so the comparison isolates the post
    f = a["attn_out"][:rows]
    post, comb = got["post"].cpu().numpy(), got["comb"].cpu().numpy()
    out = m.hc_post(_dev(f), st, got["post"], got["comb"])
    torch.cuda.synchronize()
    ref_out = oracle.moe_ffn.hc_post(f.astype(np.float64), state.astype(np.float64), post.astype(np.float64),
                                     comb.astype(np.float64))
    o = out.cpu().numpy()
    assert np.allclose(o, ref_out, rtol=1e-5, atol=2e-5)
    compare_state(o, ref_out)
    assert m.status() == 0
    m.close()


@pytest.mark.parametrize("rows", [3, 40])
def test_ffn_sublayer_hc_pre_is_the_block_prelude(rows):
    from deepseek_v4_moe_gb300 import MoeFFN, config_from
    case = synth.Case(replace(BASE, rows=rows))
    c = case.cfg
    dev = upload(case)
    m = MoeFFN(config_from(c), {c.layer: dev["weights"]})
    got = m.hc_pre(dev["state"], layer=c.layer, sublayer="ffn")
    torch.cuda.synchronize()
    st = oracle.prelude_and_route(case)
    _check_pre(got, dict(pre=st["pre"], post=st["post"], comb=st["comb"], x_norm=st["ffn_norm"]))
    m.close()


def test_attn_hc_full_size_sampled_rows():
    # 4096 rows of hidden 4096 (268 MB of state), the size the bench times; the oracle checks a
    # sample of rows (the prelude and post are row-independent)
    cfg = replace(synth.CONFIGS["c4_prefill_4096"], experts=16, inter=128, shared_inter=128)
    m, case, _ = _attn_handle(cfg, 4096, layer=2)
    c = case.cfg
    a = case.attn_hc()
    st = _dev(case.state)
    got = m.hc_pre(st, layer=2, sublayer="attn")
    out = m.hc_post(_dev(a["attn_out"]), st, got["post"], got["comb"])
    torch.cuda.synchronize()
    sample = np.array([0, 1, 127, 128, 1000, 2047, 2048, 4000, 4094, 4095])
    ref = oracle.hc_sublayer_pre(case.state[sample], a["hc_fn"], a["hc_scale"], a["hc_base"], a["norm"], c.hc,
                                 c.sinkhorn_iters, c.rms_eps)
    _check_pre({k: v[torch.from_numpy(sample).cuda()] for k, v in got.items()}, ref)
    post, comb = got["post"].cpu().numpy()[sample], got["comb"].cpu().numpy()[sample]
    ref_out = oracle.moe_ffn.hc_post(a["attn_out"][sample].astype(np.float64),
                                     case.state[sample].astype(np.float64), post.astype(np.float64),
                                     comb.astype(np.float64))
    o = out.cpu().numpy()[sample]
    assert np.allclose(o, ref_out, rtol=1e-5, atol=2e-5)
    assert m.status() == 0
    m.close()


def test_hc_entry_points_reject_bad_calls():
    from deepseek_v4_moe_gb300 import MoeFFNError
    from deepseek_v4_moe_gb300 import _lib as L
    m, case, _ = _attn_handle(BASE, 8, layer=1)
    st = _dev(case.state[:4])
    with pytest.raises(MoeFFNError) as e:
        m.hc_pre(st, layer=0, sublayer="attn")          # no attention weights on layer 0
    assert e.value.code == L.ERR_NO_WEIGHTS
    with pytest.raises(MoeFFNError) as e:
        m.hc_pre(st, layer=1, sublayer="ffn")           # the handle has no FFN weights
    assert e.value.code == L.ERR_NO_WEIGHTS
    with pytest.raises(MoeFFNError) as e:
        m.hc_pre(st, layer=9, sublayer="attn")
    assert e.value.code == L.ERR_LAYER_RANGE
    with pytest.raises(MoeFFNError) as e:
        m.hc_pre(_dev(case.state[:8]).repeat(2, 1, 1), layer=1, sublayer="attn")  # 16 rows > max_rows 8
    assert e.value.code == L.ERR_ROWS_RANGE
    got = m.hc_pre(st, layer=1, sublayer="attn")
    with pytest.raises(MoeFFNError) as e:
        m.hc_post(_dev(case.attn_hc()["attn_out"][:4]), st, got["post"], got["comb"], out=st)
    assert e.value.code == L.ERR_ALIAS
    # no kernel ran for the rejected calls: the accepted one completes with a clean status
    torch.cuda.synchronize()
    assert m.status() == 0
    m.close()
