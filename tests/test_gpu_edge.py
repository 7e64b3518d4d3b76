"""Edge cases of the GPU path at tiny shapes (hidden 256, 16 experts, top-2, inter 128) against the
oracle: ragged row counts on both paths, hash routing with invalid table entries and token ids,
every row on one expert (and most experts empty), repeated calls, and the host-side error codes."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
import synth
from synth.device import upload
from tests.inputs import compare_state, tie_free

pytestmark = pytest.mark.gpu

TINY = synth.CONFIGS["c0_tiny"]


def _run(case, max_rows=None, layer=None):
    from deepseek_v4_moe_gb300 import MoeFFN, config_from
    cfg = case.cfg
    dev = upload(case)
    m = MoeFFN(config_from(cfg, max_rows or cfg.rows), {cfg.layer: dev["weights"]})
    out = m.forward(dev["state"], dev["token_ids"], cfg.layer if layer is None else layer)
    torch.cuda.synchronize()
    res = dict(out=out.cpu().numpy(), status=m.status(), indices=m.debug("indices"), weights=m.debug("weights"),
               ffn_output=m.debug("ffn_output"))
    return m, dev, res


@pytest.mark.parametrize("rows", [1, 2, 3, 5, 17, 129, 300])
def test_ragged_rows_score(rows, cuda_lib):
    case, st = tie_free(replace(TINY, rows=rows, name=f"tiny{rows}"))
    m, dev, res = _run(case)
    ref = oracle.forward_ffn_rows(case, stages=st)
    assert res["status"] == 0
    assert np.array_equal(res["indices"], ref["indices"])
    compare_state(res["out"], ref["out_state"])
    m.close()


@pytest.mark.parametrize("rows", [3, 9])
def test_hash_with_invalid_entries(rows, cuda_lib):
    cfg = replace(TINY, rows=rows, layer=0, name=f"hash{rows}")
    case = synth.Case(cfg)
    case.token_ids[0] = 7
    case.tid2eid[7] = [-1, 5]          # invalid first slot
    case.token_ids[1] = 9
    case.tid2eid[9] = [999, 3]         # out of range expert
    case.token_ids[2] = cfg.vocab + 5  # token outside the vocabulary: both slots masked
    m, dev, res = _run(case)
    ref = oracle.forward_ffn_rows(case)
    assert res["status"] & 0x1 and res["status"] & 0x2
    assert np.array_equal(res["indices"], ref["indices"])
    assert np.allclose(res["weights"], ref["weights"], rtol=1e-5, atol=1e-6)
    compare_state(res["out"], ref["out_state"])
    m.close()


def test_one_expert_takes_every_row(cuda_lib):
    cfg = replace(TINY, rows=200, name="hot1")
    case = synth.Case(cfg)
    case.exp_probs_b = np.zeros(16, np.float32)
    case.exp_probs_b[11] = 5.0         # expert 11 first in every row; most others get nothing
    case, st = tie_free_case(case)
    m, dev, res = _run(case)
    ref = oracle.forward_ffn_rows(case, stages=st)
    assert np.all(res["indices"][:, 0] == 11)
    assert np.array_equal(res["indices"], ref["indices"])
    compare_state(res["out"], ref["out_state"])
    m.close()


def tie_free_case(case):
    st = oracle.prelude_and_route(case)
    for _ in range(20):
        bad = st["margin"] < 1e-5
        if not bad.any():
            return case, st
        att = case.attempts.copy()
        att[bad] += 1
        bias = case.exp_probs_b
        case = case.with_attempts(att)
        case.exp_probs_b = bias
        st = oracle.prelude_and_route(case)
    raise RuntimeError("ties")


def test_repeat_calls_are_identical_and_counters_reset(cuda_lib):
    case, st = tie_free(replace(TINY, rows=64, name="rep"))
    from deepseek_v4_moe_gb300 import MoeFFN, config_from
    dev = upload(case)
    m = MoeFFN(config_from(case.cfg), {case.cfg.layer: dev["weights"]})
    outs = [m.forward(dev["state"], None, case.cfg.layer).cpu().numpy() for _ in range(3)]
    small = m.forward(dev["state"][:3].contiguous(), None, case.cfg.layer).cpu().numpy()
    again = m.forward(dev["state"], None, case.cfg.layer).cpu().numpy()
    assert m.status() == 0
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2]) and np.array_equal(outs[0], again)
    ref = oracle.forward_ffn_rows(case, stages=st)
    compare_state(outs[0], ref["out_state"])
    compare_state(small, ref["out_state"][:3])
    m.close()


def test_decode_row_counts_interleaved(cuda_lib):
    # One handle, decode calls of 4, 1, 2, 3, 4 and 2 rows in turn: each row count runs its own
    # instance of the persistent decode kernel, and every launch must leave its tickets and counters
    # at zero for the next one (the last CTA out resets them).
    case, st = tie_free(replace(TINY, rows=4, name="dec_interleave"))
    from deepseek_v4_moe_gb300 import MoeFFN, config_from
    dev = upload(case)
    m = MoeFFN(config_from(case.cfg), {case.cfg.layer: dev["weights"]})
    ref = oracle.forward_ffn_rows(case, stages=st)["out_state"]
    seen = {}
    for r in (4, 1, 2, 3, 4, 2):
        out = m.forward(dev["state"][:r].contiguous(), dev["token_ids"][:r].contiguous(), case.cfg.layer)
        got = out.cpu().numpy()
        assert m.status() == 0
        compare_state(got, ref[:r])
        if r in seen:
            assert np.array_equal(got, seen[r])  # same inputs, same bits
        seen[r] = got
    m.close()


def test_host_buffer_entry_point(cuda_lib):
    case, st = tie_free(replace(TINY, rows=6, name="host"))
    from deepseek_v4_moe_gb300 import MoeFFN, config_from
    dev = upload(case)
    m = MoeFFN(config_from(case.cfg), {case.cfg.layer: dev["weights"]})
    out = np.empty_like(case.state)
    m.forward_host(case.state, case.token_ids, case.cfg.layer, out)
    ref = oracle.forward_ffn_rows(case, stages=st)
    compare_state(out, ref["out_state"])
    m.close()


def test_error_codes(cuda_lib):
    from deepseek_v4_moe_gb300 import MoeFFN, MoeFFNError, config_from
    case = synth.Case(replace(TINY, rows=4, layer=0, name="err"))
    dev = upload(case)
    m = MoeFFN(config_from(case.cfg), {0: dev["weights"]})
    s = dev["state"]
    codes = []
    for kwargs in (dict(layer=4), dict(layer=3), dict(layer=0, token_ids=None)):
        try:
            m.forward(s, kwargs.get("token_ids", dev["token_ids"]), kwargs["layer"])
        except MoeFFNError as e:
            codes.append(e.code)
    assert codes == [-3, -12, -1]
    lib = m._lib
    assert lib.moe_ffn_forward(m._h, s.data_ptr(), dev["token_ids"].data_ptr(), 0, 0, s.data_ptr(), None) == -4
    assert lib.moe_ffn_forward(m._h, s.data_ptr(), dev["token_ids"].data_ptr(), 5, 0, s.data_ptr() + 4096, None) == -5
    assert lib.moe_ffn_forward(m._h, s.data_ptr(), dev["token_ids"].data_ptr(), 4, 0, s.data_ptr() + 4096, None) == -7
    assert lib.moe_ffn_forward(m._h, s.data_ptr() + 4, dev["token_ids"].data_ptr(), 1, 0,
                               torch.empty_like(s).data_ptr(), None) == -11
    assert m.status() == 0
    m.close()


def _tie_free_fixed(case, plant):
    """Redraws near-tied rows (new attempt numbers) while keeping the planted modification."""
    for _ in range(20):
        plant(case)
        st = oracle.prelude_and_route(case)
        bad = st["margin"] < 1e-5
        if not bad.any():
            return case, st
        att = case.attempts.copy()
        att[bad] += 1
        case = case.with_attempts(att)
    raise RuntimeError("ties")


@pytest.mark.parametrize("rows", [3, 40])
def test_outliers_and_activations_past_fp16_range(rows, cuda_lib):
    # state elements at +-12..20 sigma, one row scaled by 1e5 (values far past fp16's 65504), and the
    # ffn_norm weight scaled so that the SwiGLU output of most slots exceeds 65504 as well: both paths
    # must keep f32 range end to end (compared row by row, so the big row hides nothing)
    def plant(case):  # applied once to each freshly drawn case
        case.ffn_norm = (case.ffn_norm * 2000.0).astype(np.float32)
        case.state[0, 1, 5] = 20.0
        case.state[0, 2, 7] = -12.0
        case.state[1] *= 1e5
        case.state[-1, 3, :9] = 16.0

    cfg = replace(TINY, rows=rows, name=f"outl{rows}")
    case, st = _tie_free_fixed(synth.Case(cfg), plant)
    m, dev, res = _run(case)
    ref = oracle.forward_ffn_rows(case, stages=st)
    xf = st["ffn_norm"]
    act = oracle.moe_ffn.swiglu(xf @ oracle.moe_ffn.expert_weights(case, "gate", None).T,
                                xf @ oracle.moe_ffn.expert_weights(case, "up", None).T)
    assert np.mean(np.abs(act) > 65504) > 0.1, "the case must carry activations past fp16 range"
    assert res["status"] == 0
    assert np.array_equal(res["indices"], ref["indices"])
    for r in range(rows):
        compare_state(res["out"][r], ref["out_state"][r])
    m.close()


@pytest.mark.parametrize("rows", [3, 40])
def test_nonfinite_state_row_is_reported_and_contained(rows, cuda_lib):
    # a NaN in one state row: the device status carries the non-finite bit, that row's output is
    # not finite, and every other row still matches the oracle
    cfg = replace(TINY, rows=rows, name=f"nan{rows}")
    case, st = tie_free(cfg)
    ref = oracle.forward_ffn_rows(case, stages=st)
    case.state[1, 2, 3] = np.nan
    m, dev, res = _run(case)
    assert res["status"] & 0x4, f"status {res['status']:#x} lacks the non-finite bit"
    assert not np.isfinite(res["out"][1]).all()
    others = [r for r in range(rows) if r != 1]
    assert np.array_equal(res["indices"][others], ref["indices"][others])
    for r in others:
        compare_state(res["out"][r], ref["out_state"][r])
    m.close()
