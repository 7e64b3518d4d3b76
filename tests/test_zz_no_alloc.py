"""moe_ffn_hc_split_noalloc: the HC split for callers that cannot allocate device memory at call time
(graph capture, allocation-free serving loops, hosts whose pool owns the GPU).

Its scratch is a fixed array inside the library, shared by every call and keeping the last call's
contents, so it is checked on two calls in a row against the handle-based forward's pre/post/comb
(the same tolerance as the parity tests).  This file is collected last so that a stopping run has
already run every other test; it also passes on its own in a fresh process.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
import synth
from synth.device import upload

pytestmark = pytest.mark.gpu


def _split_noalloc(lib, case, dev):
    c = case.cfg
    rows = c.rows
    pre = torch.full((rows, c.hc), float("nan"), device="cuda")
    post = torch.full((rows, c.hc), float("nan"), device="cuda")
    comb = torch.full((rows, c.hc, c.hc), float("nan"), device="cuda")
    w = dev["weights"]
    stream = torch.cuda.current_stream()
    rc = lib.moe_ffn_hc_split_noalloc(dev["state"].data_ptr(), w["hc_fn"].data_ptr(), w["hc_scale"].data_ptr(),
                                      w["hc_base"].data_ptr(), rows, c.hc, c.hidden, c.sinkhorn_iters, c.rms_eps,
                                      pre.data_ptr(), post.data_ptr(), comb.data_ptr(), stream.cuda_stream)
    assert rc == 0, lib.moe_ffn_last_error(None)
    torch.cuda.synchronize()
    return pre.cpu().numpy(), post.cpu().numpy(), comb.cpu().numpy()


@pytest.mark.parametrize("rows", [4, 40])
def test_noalloc_split_matches_forward_twice(rows, cuda_lib):
    from deepseek_v4_moe_gb300 import MoeFFN, config_from
    case = synth.Case(replace(synth.CONFIGS["c0_tiny"], rows=rows))
    dev = upload(case)
    m = MoeFFN(config_from(case.cfg), {case.cfg.layer: dev["weights"]})
    m.forward(dev["state"], dev["token_ids"], case.cfg.layer)
    ref = [m.debug(k) for k in ("pre", "post", "comb")]
    m.close()
    for _ in range(2):
        got = _split_noalloc(cuda_lib, case, dev)
        for g, r in zip(got, ref):
            assert np.allclose(g, r, rtol=1e-5, atol=1e-6)


def test_noalloc_split_full_shape_against_oracle(cuda_lib):
    case = synth.Case(replace(synth.CONFIGS["c1_decode_b1"], rows=4))
    st = oracle.prelude_and_route(case)
    w = {k: torch.from_numpy(np.ascontiguousarray(getattr(case, k)).view(np.int16) if k == "hc_fn"
                             else np.ascontiguousarray(getattr(case, k))).cuda()
         for k in ("hc_fn", "hc_scale", "hc_base")}
    dev = {"weights": w, "state": torch.from_numpy(case.state).cuda()}
    for _ in range(2):
        pre, post, comb = _split_noalloc(cuda_lib, case, dev)
        assert np.allclose(pre, st["pre"], rtol=1e-5, atol=1e-6)
        assert np.allclose(post, st["post"], rtol=1e-5, atol=1e-6)
        assert np.allclose(comb, st["comb"], rtol=1e-5, atol=1e-6)


def _call_with_sized_buffers(lib, rows, hc, hidden):
    """Calls the split with buffers sized for (rows, hc, hidden), so that even a call the host
    accepted would stay inside its buffers."""
    M = (2 + hc) * hc
    state = torch.zeros(rows * hc * hidden, device="cuda")
    hc_fn = torch.zeros(M * hc * hidden, dtype=torch.int16, device="cuda")
    scale = torch.ones(3, device="cuda")
    base = torch.zeros(M, device="cuda")
    pre = torch.empty(rows * hc, device="cuda")
    post = torch.empty(rows * hc, device="cuda")
    comb = torch.empty(rows * hc * hc, device="cuda")
    rc = lib.moe_ffn_hc_split_noalloc(state.data_ptr(), hc_fn.data_ptr(), scale.data_ptr(), base.data_ptr(), rows,
                                      hc, hidden, 20, 1e-6, pre.data_ptr(), post.data_ptr(), comb.data_ptr(),
                                      torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return rc


def test_noalloc_split_rejects_rows_beyond_the_fixed_scratch(cuda_lib):
    from deepseek_v4_moe_gb300 import _lib
    # more rows than the fixed ticket array covers
    assert _call_with_sized_buffers(cuda_lib, 5000, 4, 4096) == _lib.ERR_ROWS_RANGE
    assert b"fixed scratch" in cuda_lib.moe_ffn_last_error(None)
    # within the row cap, but hc*hidden = 24192 is no multiple of 512, so the mix keeps 189 chunk
    # partials per output and row: 100 rows need about 1.2 MB, above the fixed 1 MiB
    assert _call_with_sized_buffers(cuda_lib, 100, 3, 8064) == _lib.ERR_ROWS_RANGE
    assert b"fixed 1 MiB scratch" in cuda_lib.moe_ffn_last_error(None)
