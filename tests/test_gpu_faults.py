"""Failure detection without a GPU fault: a bounded in-kernel wait made to run out on purpose.

Every wait inside the kernels gives up after a limit, sets the device timeout bit, stops its work,
waits (bounded) for its own copies and tensor-core operations in flight, frees its tensor memory and
returns; the handle stays usable.  A test hook (moe_ffn_set_fault_injection) makes one wait run out:
on the decode path a count that nothing reaches, on the tensor-core path an mbarrier that nothing
arrives at.  The forward then reports MOE_FFN_DEV_TIMEOUT, and the next forward on the same handle,
hook off, matches the oracle with a clean status.  This mirrors the guards of forward_ffn_rows
(docs.rs "hf2q 0.1.3 .../deepseek4/ffn_forward.rs"), which fail the call instead of running on."""
import time
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
TIMEOUT_BIT = 0x8


@pytest.mark.parametrize("rows,which", [(2, "decode"), (40, "gemm")])
def test_injected_wait_times_out_and_the_handle_recovers(rows, which, cuda_lib):
    from deepseek_v4_moe_gb300 import MoeFFN, config_from
    case, st = tie_free(replace(TINY, rows=rows, name=f"fault_{which}"))
    ref = oracle.forward_ffn_rows(case, stages=st)["out_state"]
    dev = upload(case)
    m = MoeFFN(config_from(case.cfg), {case.cfg.layer: dev["weights"]})
    good = m.forward(dev["state"], dev["token_ids"], case.cfg.layer).cpu().numpy()
    assert m.status() == 0
    compare_state(good, ref)

    m.set_fault_injection(which, wait_limit_us=20000)  # every wait bounded by 20 ms
    t0 = time.perf_counter()
    m.forward(dev["state"], dev["token_ids"], case.cfg.layer)
    status = m.status()  # synchronises: the kernels returned
    took = time.perf_counter() - t0
    assert status & TIMEOUT_BIT, f"status {status:#x} lacks the timeout bit"
    assert took < 10.0, f"the aborted forward took {took:.1f} s"

    m.set_fault_injection(None)
    for _ in range(2):  # the counters and the tensor memory were left clean
        again = m.forward(dev["state"], dev["token_ids"], case.cfg.layer).cpu().numpy()
        assert m.status() == 0
        compare_state(again, ref)
        assert np.array_equal(again, good)
    m.close()
    torch.cuda.synchronize()
