"""GPU path against the oracle on configurations away from the workloads' shapes (tiny, fast):
hc of 1, 2 and 3 (mix widths 3, 8 and 15; a mix chunk narrower than 512 columns), hidden 128 and
384 (router chunks and K splits that are not the defaults), 512 experts (router passes beyond
256 experts and two router weight tiles), and top_k 8 at four rows, whose 32 routed slots can
make 33 expert groups (the decode kernel's second group-table register).  Each on the decode
kernel (rows <= 4) and on the prefill path."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
import synth
from synth.device import upload
from tests.inputs import compare_state, tie_free

pytestmark = pytest.mark.gpu

BASE = synth.CONFIGS["c0_tiny"]

CASES = {
    "hc2_e32_k3": replace(BASE, hc=2, experts=32, top_k=3, seed=11),
    "hc1_d128": replace(BASE, hc=1, hidden=128, seed=12),
    "hc4_e512_k8": replace(BASE, experts=512, top_k=8, seed=13),
    "hc4_e512_k8_hash": replace(BASE, experts=512, top_k=8, layer=0, seed=14),
    "hc3_d384_e48_k4": replace(BASE, hc=3, hidden=384, experts=48, top_k=4, inter=256, shared_inter=256, seed=15),
}
ROWS = {
    "hc2_e32_k3": [1, 4, 40],
    "hc1_d128": [2, 9],
    "hc4_e512_k8": [4, 130],
    "hc4_e512_k8_hash": [4, 20],
    "hc3_d384_e48_k4": [3, 70],
}
PARAMS = [(name, rows) for name in CASES for rows in ROWS[name]]


@pytest.mark.parametrize("name,rows", PARAMS, ids=[f"{n}-r{r}" for n, r in PARAMS])
def test_config_against_oracle(name, rows, cuda_lib):
    from deepseek_v4_moe_gb300 import MoeFFN, config_from
    case, st = tie_free(replace(CASES[name], rows=rows, name=f"{name}_r{rows}"))
    cfg = case.cfg
    dev = upload(case)
    m = MoeFFN(config_from(cfg), {cfg.layer: dev["weights"]})
    out = m.forward(dev["state"], dev["token_ids"], cfg.layer)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    res = {k: m.debug(k) for k in ("indices", "weights", "pre", "post", "comb")}
    status = m.status()
    m.close()
    assert status == 0
    assert np.array_equal(res["indices"], st["indices"]), "routed indices differ"
    assert np.allclose(res["weights"], st["weights"], rtol=1e-5, atol=1e-6)
    for k in ("pre", "post", "comb"):
        assert np.allclose(res[k], st[k], rtol=1e-5, atol=1e-6), k
    ref = oracle.forward_ffn_rows(case, stages=st)
    compare_state(got, ref["out_state"])


def test_top_k8_four_rows_fill_33_groups():
    # the hash case at four rows draws 32 distinct experts from 512 with overwhelming likelihood:
    # together with the shared expert that is the largest group count the decode kernel handles
    case, st = tie_free(replace(CASES["hc4_e512_k8_hash"], rows=4, name="g33"))
    idx = st["indices"]
    assert len(np.unique(idx[(idx >= 0) & (idx < case.cfg.experts)])) == 32
