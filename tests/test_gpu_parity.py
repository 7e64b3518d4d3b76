"""GPU path vs the CPU oracle on the five workloads, through the C ABI.

Bar: routed expert indices bit-exact (every row, slot order included), route weights and HC
pre/post/comb to 1e-5 relative, and the output state within relative L2 1e-3 and
max |delta| <= 1e-2 * RMS(output), on every row of every workload (the 4096-row prefill included:
the oracle evaluates the experts expert by expert, so all rows cost seconds of f64 BLAS).
"""
import gc

import numpy as np
import pytest
import torch

import oracle
import synth
from synth.device import upload
from tests.inputs import compare_dot, compare_scaled, compare_state, tie_free

pytestmark = pytest.mark.gpu

LOGIT_TAU = 1e-6


def _run(name, cuda_lib):
    from deepseek_v4_moe_gb300 import MoeFFN, config_from
    case, st = tie_free(name)
    cfg = case.cfg
    dev = upload(case)
    m = MoeFFN(config_from(cfg), {cfg.layer: dev["weights"]})
    out = m.forward(dev["state"], dev["token_ids"], cfg.layer)
    torch.cuda.synchronize()
    res = dict(out=out.cpu().numpy(), status=m.status())
    for k in ("indices", "weights", "pre", "post", "comb", "logits", "ffn_norm"):
        res[k] = m.debug(k)
    m.close()
    del dev, out, m
    gc.collect()
    torch.cuda.empty_cache()
    return case, st, res


@pytest.mark.parametrize("name", list(synth.CONFIGS))
def test_parity(name, cuda_lib):
    case, st, res = _run(name, cuda_lib)
    cfg = case.cfg
    assert res["status"] == 0
    assert np.array_equal(res["indices"], st["indices"]), "routed indices differ"
    assert np.allclose(res["weights"], st["weights"], rtol=1e-5, atol=1e-6)
    assert np.allclose(res["weights"].sum(axis=1), 1.0, atol=1e-5)
    for k in ("pre", "post", "comb"):
        assert np.allclose(res[k], st[k], rtol=1e-5, atol=1e-6), k
    # ffn_norm = rs * w * sum_h pre_h * state_h: with pre held to 1e-5 relative, an entry's error is
    # bounded by 1e-5 of rs |w| sum_h pre_h |state_h| (its terms before cancellation) plus 1e-5 of
    # itself (the RMS scale); 2e-5 of that sum is the bar
    st64 = case.state.astype(np.float64)
    rs = 1.0 / np.sqrt(np.mean(st["ffn_input"] ** 2, axis=1, keepdims=True) + cfg.rms_eps)
    cond = rs * np.abs(case.ffn_norm.astype(np.float64)) * np.einsum("rh,rhd->rd", st["pre"], np.abs(st64))
    compare_scaled(res["ffn_norm"], st["ffn_norm"], cond + np.abs(st["ffn_norm"]), 2e-5, "ffn_norm")
    # logits: f32 sums over hidden = 4096 products; the bar is relative to sum |x_d * g_ed| (see
    # compare_dot), with tau = 1e-6 ~ 16 units of f32 rounding over the normalised input
    compare_dot(res["logits"], st["logits"], st["ffn_norm"], synth.bf16_bits_to_f32(case.gate), LOGIT_TAU, "logits")
    ref = oracle.forward_ffn_rows(case, stages=st)
    compare_state(res["out"], ref["out_state"])
    # and row by row: no row may hide behind the others' agreement
    for r in range(cfg.rows):
        compare_state(res["out"][r], ref["out_state"][r], rel_l2=1e-3, max_frac=1e-2)
    if cfg.rows > 4:
        assert len(np.unique(st["indices"])) > 0.5 * cfg.experts
