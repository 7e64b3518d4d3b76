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


# hidden 640: K splits of 5 chunks, so a row's scales for one split are 10 bytes at a 2-byte offset
# (copied with plain loads), and the last pair of 128-row down tiles is half past the matrix; inter 384:
# 12 scale bytes a row (4-byte copies)
RAGGED = replace(TINY, hidden=640, inter=384, shared_inter=384, seed=31)


@pytest.mark.parametrize("rows", [1, 4])
def test_mx_decode_ragged_splits(rows):
    case, st, got, idx, status = _run(RAGGED, rows)
    assert status == 0
    assert np.array_equal(idx, st["indices"])
    compare_state(got, oracle.forward_ffn_rows(case, stages=st)["out_state"])


@pytest.mark.parametrize("what", ["code", "scale"])
@pytest.mark.parametrize("rows", [1, 4, 40])
def test_mx_nan_weight(what, rows):
    # one NaN element in the shared expert's gate: its act entry is NaN, so is every element of the
    # FFN output and of the new state, and the status reports it.  At four rows a NaN code or a NaN
    # scale (E8M0 255) sends the layer from the tensor-core decode kernel (its f16 weights hold
    # neither) to the CUDA-core one, which one row uses anyway; 40 rows run the tensor-core GEMMs,
    # whose act planes must carry the NaN too.
    from deepseek_v4_moe_gb300 import MoeFFN, config_from
    case, st = tie_free(replace(TINY, rows=rows, name=f"c0_mx_nan_{what}_r{rows}"))
    c = case.cfg
    dev = upload(case)
    mx = upload_mx(case)
    if what == "code":
        mx["gate_sh"][3, 17] = 0x7F
    else:
        mx["gate_sh_scale"][5, 1] = 0xFF
    m = MoeFFN(config_from(c, max_rows=rows), {c.layer: dict(dev["weights"])})
    m.set_mxfp8_experts(c.layer, mx)
    out = m.forward(dev["state"], dev["token_ids"], c.layer)
    torch.cuda.synchronize()
    got, status = out.cpu().numpy(), m.status()
    m.close()
    assert status & 0x4
    assert np.isnan(got).all()


@pytest.mark.parametrize("span", [22, 23])
def test_mx_decode_scale_span(span):
    # one scale of the shared gate moved `span` binades below the layer's largest: at 22 the f16
    # weights of the tensor-core decode are still exact (the smallest code times it is 2^-24 in f16);
    # at 23 the layer decodes on the CUDA-core kernel.  Both match the oracle on the same scales.
    from deepseek_v4_moe_gb300 import MoeFFN, config_from
    case, st = tie_free(replace(TINY, rows=4, name=f"c0_mx_span{span}"))
    c = case.cfg
    dev = upload(case)
    mx = upload_mx(case)
    smax = max(int(v.max()) for k, v in mx.items() if k.endswith("_scale"))
    q, sc = case.shared_mx("gate")
    sc = sc.copy()
    sc[7, 3] = smax - span
    mx["gate_sh_scale"][7, 3] = smax - span
    orig = case.shared_mx
    case.shared_mx = lambda which: (q, sc) if which == "gate" else orig(which)
    m = MoeFFN(config_from(c, max_rows=c.rows), {c.layer: dict(dev["weights"])})
    m.set_mxfp8_experts(c.layer, mx)
    out = m.forward(dev["state"], dev["token_ids"], c.layer)
    torch.cuda.synchronize()
    got, status = out.cpu().numpy(), m.status()
    m.close()
    assert status == 0
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
