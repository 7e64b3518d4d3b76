"""GPU parity of the block on MXFP8 experts (moe_ffn_set_mxfp8_experts) against the oracle, which
decodes the same codes and scales by the format's definition.  Rows <= 4 stream the codes in the
decode kernel; larger batches run the tensor-core path on the exact bf16 expansion made at
registration."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
import synth
from synth.device import upload, upload_mx
from tests.inputs import compare_state, tie_free

pytestmark = pytest.mark.gpu

TINY = replace(synth.CONFIGS["c0_tiny"], weights="mxfp8")


def _run(cfg, rows, with_bf16=True, max_rows=None):
    from deepseek_v4_moe_gb300 import MoeFFN, config_from
    case, st = tie_free(replace(cfg, rows=rows, name=f"{cfg.name}_mx_r{rows}"))
    c = case.cfg
    dev = upload(case)
    w = dict(dev["weights"])
    if not with_bf16:
        for k in ("gate_exps", "up_exps", "down_exps", "gate_sh", "up_sh", "down_sh"):
            w.pop(k)
    m = MoeFFN(config_from(c, max_rows=max_rows or rows), {c.layer: w})
    m.set_mxfp8_experts(c.layer, upload_mx(case))
    out = m.forward(dev["state"], dev["token_ids"], c.layer)
    torch.cuda.synchronize()
    got, idx, status = out.cpu().numpy(), m.debug("indices"), m.status()
    m.close()
    return case, st, got, idx, status


@pytest.mark.parametrize("rows", [1, 2, 3, 4, 5, 40, 130])
def test_mx_tiny_against_oracle(rows):
    case, st, got, idx, status = _run(TINY, rows)
    assert status == 0
    assert np.array_equal(idx, st["indices"])
    compare_state(got, oracle.forward_ffn_rows(case, stages=st)["out_state"])


@pytest.mark.parametrize("rows", [1, 40])
def test_mx_without_bf16_experts(rows):
    case, st, got, idx, status = _run(TINY, rows, with_bf16=False)
    assert status == 0
    compare_state(got, oracle.forward_ffn_rows(case, stages=st)["out_state"])


def test_forward_before_mx_registration_is_rejected():
    from deepseek_v4_moe_gb300 import MoeFFN, MoeFFNError, config_from
    from deepseek_v4_moe_gb300 import _lib as L
    case = synth.Case(replace(TINY, rows=4))
    dev = upload(case)
    w = {k: v for k, v in dev["weights"].items() if k not in ("gate_exps", "up_exps", "down_exps", "gate_sh",
                                                               "up_sh", "down_sh")}
    m = MoeFFN(config_from(case.cfg), {case.cfg.layer: w})
    with pytest.raises(MoeFFNError) as e:
        m.forward(dev["state"], dev["token_ids"], case.cfg.layer)
    assert e.value.code == L.ERR_NO_WEIGHTS
    m.close()


def test_mx_full_shape_prefill():
    # hidden 4096, inter 2048, 32 experts, 512 rows: every weight tile of the tensor-core path at its
    # real shape, every row compared
    cfg = replace(synth.PROFILE_CONFIGS["p_prefill_512_e32"], weights="mxfp8")
    case, st, got, idx, status = _run(cfg, cfg.rows)
    assert status == 0
    assert np.array_equal(idx, st["indices"])
    ref = oracle.forward_ffn_rows(case, stages=st)["out_state"]
    compare_state(got, ref)
    for r in range(cfg.rows):
        compare_state(got[r], ref[r])


@pytest.mark.parametrize("name", ["c1_decode_b1", "c2_decode_b4_hash"])
def test_mx_full_shape_decode(name):
    cfg = replace(synth.CONFIGS[name], weights="mxfp8")
    case, st, got, idx, status = _run(cfg, cfg.rows)
    assert status == 0
    assert np.array_equal(idx, st["indices"])
    compare_state(got, oracle.forward_ffn_rows(case, stages=st)["out_state"])
