"""GPU path vs the CPU oracle on the five workloads, through the C ABI.

Bar: routed expert indices bit-exact (every row, slot order included), route weights and HC
pre/post/comb to 1e-5 relative, and the output state within relative L2 1e-3 and
max |delta| <= 1e-2 * RMS(output).  At full shape the oracle evaluates the experts for a seeded
sample of rows (first, last and a spread), and the prelude/routing for every row.
"""
import gc

import numpy as np
import pytest
import torch

import oracle
import synth
from synth.device import upload
from tests.inputs import compare_dot, compare_state, sample_rows, substages, tie_free

pytestmark = pytest.mark.gpu

LOGIT_TAU = 1e-6
SAMPLE = {"c0_tiny": 4, "c1_decode_b1": 1, "c2_decode_b4_hash": 4, "c3_prefill_512": 12, "c4_prefill_4096": 12}


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
    assert np.allclose(res["ffn_norm"], st["ffn_norm"], rtol=1e-4, atol=1e-5)
    # logits: f32 sums over hidden = 4096 products; the bar is relative to sum |x_d * g_ed| (see
    # compare_dot), with tau = 1e-6 ~ 16 units of f32 rounding over the normalised input
    compare_dot(res["logits"], st["logits"], st["ffn_norm"], synth.bf16_bits_to_f32(case.gate), LOGIT_TAU, "logits")
    rows = sample_rows(cfg.rows, SAMPLE[name], seed=cfg.seed)
    ref = oracle.forward_ffn_rows(case, stages=substages(st, rows))
    compare_state(res["out"][rows], ref["out_state"])
    if cfg.rows > 4:  # the sample covers the hot / popular experts too
        assert len(np.unique(st["indices"])) > 0.5 * cfg.experts
