"""Uploads a workload's inputs to device tensors (torch), drawing the expert weights in chunks
through a pinned host buffer so that 12.9 GB never sit on the host at once."""
from __future__ import annotations

import numpy as np
import torch


def _dev(a: np.ndarray, device) -> torch.Tensor:
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def upload(case, device="cuda", chunk_experts: int = 16, experts: bool = True) -> dict:
    """Returns {"weights": {field: tensor}, "state": f32 [rows, hc, hidden], "token_ids": i32 [rows]}.
    bf16 tensors hold raw bit patterns (torch.int16).  With experts=False the six bf16 expert
    matrices are left out (a layer whose experts come in MXFP8)."""
    c = case.cfg
    w = {
        "hc_fn": _dev(case.hc_fn, device),
        "hc_base": _dev(case.hc_base, device),
        "hc_scale": _dev(case.hc_scale, device),
        "ffn_norm": _dev(case.ffn_norm, device),
        "gate": _dev(case.gate, device),
    }
    if experts:
        w.update(gate_sh=_dev(case.gate_sh, device), up_sh=_dev(case.up_sh, device), down_sh=_dev(case.down_sh, device))
    if case.exp_probs_b is not None:
        w["exp_probs_b"] = _dev(case.exp_probs_b, device)
    if case.tid2eid is not None:
        w["tid2eid"] = _dev(case.tid2eid, device)
    if not experts:
        return {"weights": w, "state": _dev(case.state, device), "token_ids": _dev(case.token_ids, device)}
    per = c.inter * c.hidden
    chunk = max(1, min(chunk_experts, c.experts))
    host = torch.empty(chunk * per, dtype=torch.int16, pin_memory=torch.cuda.is_available())
    host_np = host.numpy().view(np.uint16)
    for which in ("gate", "up", "down"):
        shape = (c.experts, c.hidden, c.inter) if which == "down" else (c.experts, c.inter, c.hidden)
        t = torch.empty(shape, dtype=torch.int16, device=device)
        flat = t.view(-1)
        for e0 in range(0, c.experts, chunk):
            n = min(chunk, c.experts - e0)
            case.expert_block(which, e0, n, host_np[: n * per])
            flat[e0 * per:(e0 + n) * per].copy_(host[: n * per], non_blocking=False)
        w[f"{which}_exps"] = t
    return {"weights": w, "state": _dev(case.state, device), "token_ids": _dev(case.token_ids, device)}


def upload_mx(case, device="cuda", chunk_experts: int = 16) -> dict:
    """The workload's expert matrices in MXFP8 (the same draws as ``upload``'s bf16 ones), as uint8
    device tensors named like the fields of ``moe_ffn_mxfp8_experts``: E4M3 codes in the bf16
    layouts and E8M0 scales [rows, K / 32], drawn in chunks through pinned host buffers."""
    c = case.cfg
    per = c.inter * c.hidden
    chunk = max(1, min(chunk_experts, c.experts))
    pin = torch.cuda.is_available()
    host_q = torch.empty(chunk * per, dtype=torch.uint8, pin_memory=pin)
    host_s = torch.empty(chunk * per // 32, dtype=torch.uint8, pin_memory=pin)
    hq, hs = host_q.numpy(), host_s.numpy()
    out = {}
    for which in ("gate", "up", "down"):
        rows, k = (c.hidden, c.inter) if which == "down" else (c.inter, c.hidden)
        q = torch.empty((c.experts, rows, k), dtype=torch.uint8, device=device)
        s = torch.empty((c.experts, rows, k // 32), dtype=torch.uint8, device=device)
        for e0 in range(0, c.experts, chunk):
            n = min(chunk, c.experts - e0)
            case.expert_block_mx(which, e0, n, hq[: n * per], hs[: n * per // 32])
            q.view(-1)[e0 * per:(e0 + n) * per].copy_(host_q[: n * per])
            s.view(-1)[e0 * per // 32:(e0 + n) * per // 32].copy_(host_s[: n * per // 32])
        out[f"{which}_exps"], out[f"{which}_exps_scale"] = q, s
        sq, ss = case.shared_mx(which)
        out[f"{which}_sh"] = torch.from_numpy(np.ascontiguousarray(sq)).to(device)
        out[f"{which}_sh_scale"] = torch.from_numpy(np.ascontiguousarray(ss)).to(device)
    return out
