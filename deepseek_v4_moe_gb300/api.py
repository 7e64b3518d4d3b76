"""Python face of the C ABI: a handle object over torch device tensors (marshalling only)."""
from __future__ import annotations

import ctypes
from typing import Mapping, Optional

import numpy as np
import torch

from . import _lib
from ._lib import (MXFP8_FIELDS, SUBLAYER_ATTN, SUBLAYER_FFN, MoeFfnConfig, MoeFfnHcWeights, MoeFfnLayerWeights,
                   MoeFfnMxfp8Experts, WEIGHT_FIELDS)

DEBUG_BUFFERS = {"pre": 0, "post": 1, "comb": 2, "ffn_norm": 3, "logits": 4, "indices": 5, "weights": 6,
                 "safe_indices": 7, "ffn_output": 8}

_BF16_FIELDS = {"hc_fn", "gate", "gate_exps", "up_exps", "down_exps", "gate_sh", "up_sh", "down_sh"}
_F32_FIELDS = {"hc_base", "hc_scale", "ffn_norm", "exp_probs_b"}


class MoeFFNError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"moe_ffn error {code}: {message}")
        self.code = code


def config_from(c, max_rows: Optional[int] = None) -> MoeFfnConfig:
    """A MoeFfnConfig from any object with the config's field names (e.g. synth.MoeConfig)."""
    return MoeFfnConfig(hidden=c.hidden, hc=c.hc, experts=c.experts, top_k=c.top_k, inter=c.inter,
                        shared_inter=c.shared_inter, vocab=c.vocab, n_layers=c.n_layers,
                        hash_layer_count=c.hash_layer_count, max_rows=max_rows or c.rows,
                        sinkhorn_iters=c.sinkhorn_iters, rms_eps=c.rms_eps)


def _check_weight(name: str, t: torch.Tensor):
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if name in _BF16_FIELDS and t.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise ValueError(f"{name} must hold bf16 values (torch.bfloat16 or raw 16-bit words)")
    if name in _F32_FIELDS and t.dtype != torch.float32:
        raise ValueError(f"{name} must be float32")
    if name == "tid2eid" and t.dtype != torch.int32:
        raise ValueError("tid2eid must be int32")


class MoeFFN:
    """One handle of the C library: weights of every layer, scratch for max_rows rows.

    ``layers`` maps a layer index to a dict of device tensors named like the fields of
    ``moe_ffn_layer_weights``; layers absent from the mapping have no weights.  The tensors must
    stay alive (and unchanged) for the life of the handle; the object keeps references.
    """

    def __init__(self, config: MoeFfnConfig, layers: Mapping[int, Mapping[str, torch.Tensor]]):
        self._lib = _lib.load()
        self.config = config
        self._keep = {int(k): dict(v) for k, v in layers.items()}
        arr = (MoeFfnLayerWeights * config.n_layers)()
        for l, w in self._keep.items():
            if not 0 <= l < config.n_layers:
                raise ValueError(f"layer {l} outside 0..{config.n_layers}")
            for name in WEIGHT_FIELDS:
                t = w.get(name)
                if t is not None:
                    _check_weight(name, t)
                    setattr(arr[l], name, t.data_ptr())
        h = ctypes.c_void_p()
        rc = self._lib.moe_ffn_init(ctypes.byref(config), arr, ctypes.byref(h))
        if rc != 0:
            raise MoeFFNError(rc, self._lib.moe_ffn_last_error(None).decode())
        self._h = h
        self.last_rows = 0

    def _err(self, rc: int):
        raise MoeFFNError(rc, self._lib.moe_ffn_last_error(self._h).decode())

    def forward(self, state: torch.Tensor, token_ids: Optional[torch.Tensor] = None, layer: int = 0,
                out: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
        """Enqueues the block on ``stream`` (default: the current stream); returns the output tensor."""
        c = self.config
        if state.dtype != torch.float32 or not state.is_cuda or not state.is_contiguous() or state.dim() != 3 \
                or state.shape[1:] != (c.hc, c.hidden):
            raise ValueError(f"state must be a contiguous CUDA float32 [rows, {c.hc}, {c.hidden}] tensor")
        if token_ids is not None and (token_ids.dtype != torch.int32 or not token_ids.is_cuda
                                      or token_ids.numel() != state.shape[0]):
            raise ValueError("token_ids must be a CUDA int32 tensor with one id per row")
        if out is None:
            out = torch.empty_like(state)
        s = stream if stream is not None else torch.cuda.current_stream(state.device)
        rc = self._lib.moe_ffn_forward(self._h, state.data_ptr(),
                                       token_ids.data_ptr() if token_ids is not None else None,
                                       state.shape[0], layer, out.data_ptr(), s.cuda_stream)
        if rc != 0:
            self._err(rc)
        self.last_rows = state.shape[0]
        return out

    def forward_layers(self, state: torch.Tensor, token_ids: Optional[torch.Tensor], first_layer: int, n_layers: int,
                       out: Optional[torch.Tensor] = None,
                       stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
        """Enqueues the blocks of n_layers consecutive layers, each on the previous one's output
        (one CUDA graph per argument set, captured by the first call); returns the final state."""
        self._check_state(state)
        if token_ids is not None and (token_ids.dtype != torch.int32 or not token_ids.is_cuda
                                      or token_ids.numel() != state.shape[0]):
            raise ValueError("token_ids must be a CUDA int32 tensor with one id per row")
        if out is None:
            out = torch.empty_like(state)
        s = stream if stream is not None else torch.cuda.current_stream(state.device)
        rc = self._lib.moe_ffn_forward_layers(self._h, state.data_ptr(),
                                              token_ids.data_ptr() if token_ids is not None else None,
                                              state.shape[0], first_layer, n_layers, out.data_ptr(), s.cuda_stream)
        if rc != 0:
            self._err(rc)
        self.last_rows = state.shape[0]
        return out

    def forward_host(self, state: np.ndarray, token_ids: Optional[np.ndarray], layer: int,
                     out: np.ndarray, stream: Optional[torch.cuda.Stream] = None) -> np.ndarray:
        """The block on host arrays (or pinned host tensors' numpy views); waits for completion."""
        s = stream if stream is not None else torch.cuda.current_stream()
        rows = state.shape[0]
        rc = self._lib.moe_ffn_forward_host(self._h, state.ctypes.data,
                                            token_ids.ctypes.data if token_ids is not None else None,
                                            rows, layer, out.ctypes.data, s.cuda_stream)
        if rc != 0:
            self._err(rc)
        self.last_rows = rows
        return out

    def set_mxfp8_experts(self, layer: int, experts: Mapping[str, torch.Tensor]):
        """Makes ``layer`` run on MXFP8 experts: uint8 device tensors named like the fields of
        ``moe_ffn_mxfp8_experts`` (E4M3 codes in the bf16 layouts, E8M0 scales per 32 elements)."""
        w = MoeFfnMxfp8Experts()
        for name in MXFP8_FIELDS:
            t = experts[name]
            if not t.is_cuda or not t.is_contiguous() or t.dtype != torch.uint8:
                raise ValueError(f"{name} must be a contiguous CUDA uint8 tensor")
            setattr(w, name, t.data_ptr())
        self._keep.setdefault(("mxfp8", int(layer)), {}).update(experts)
        rc = self._lib.moe_ffn_set_mxfp8_experts(self._h, layer, ctypes.byref(w))
        if rc != 0:
            self._err(rc)

    # ---- the hyper-connection prelude and post of a sublayer ----

    def set_attn_hc(self, layer: int, weights: Mapping[str, torch.Tensor]):
        """Registers the attention sublayer's HC weights of ``layer``: a dict with ``hc_fn`` (bf16
        [(2+hc)*hc, hc*hidden]), ``hc_base``, ``hc_scale`` and ``norm`` (f32) device tensors."""
        for name in ("hc_fn", "hc_base", "hc_scale", "norm"):
            t = weights[name]
            want = (torch.bfloat16, torch.int16, torch.uint16) if name == "hc_fn" else (torch.float32,)
            if not t.is_cuda or not t.is_contiguous() or t.dtype not in want:
                raise ValueError(f"attention {name} must be a contiguous CUDA tensor of "
                                 f"{'bf16 values' if name == 'hc_fn' else 'float32'}")
        self._keep.setdefault(("attn", int(layer)), {}).update(weights)
        w = MoeFfnHcWeights(hc_fn=weights["hc_fn"].data_ptr(), hc_base=weights["hc_base"].data_ptr(),
                            hc_scale=weights["hc_scale"].data_ptr(), norm=weights["norm"].data_ptr())
        rc = self._lib.moe_ffn_set_attn_hc(self._h, layer, ctypes.byref(w))
        if rc != 0:
            self._err(rc)

    def hc_pre(self, state: torch.Tensor, layer: int, sublayer: str = "attn",
               stream: Optional[torch.cuda.Stream] = None) -> dict:
        """Enqueues the HC prelude of ``sublayer`` ("attn" or "ffn"); returns device tensors
        x_norm [rows, hidden], pre, post [rows, hc] and comb [rows, hc, hc]."""
        c = self.config
        self._check_state(state)
        rows = state.shape[0]
        out = {"x_norm": torch.empty((rows, c.hidden), dtype=torch.float32, device=state.device),
               "pre": torch.empty((rows, c.hc), dtype=torch.float32, device=state.device),
               "post": torch.empty((rows, c.hc), dtype=torch.float32, device=state.device),
               "comb": torch.empty((rows, c.hc, c.hc), dtype=torch.float32, device=state.device)}
        sub = {"attn": SUBLAYER_ATTN, "ffn": SUBLAYER_FFN}[sublayer]
        s = stream if stream is not None else torch.cuda.current_stream(state.device)
        rc = self._lib.moe_ffn_hc_pre(self._h, layer, sub, state.data_ptr(), rows, out["x_norm"].data_ptr(),
                                      out["pre"].data_ptr(), out["post"].data_ptr(), out["comb"].data_ptr(),
                                      s.cuda_stream)
        if rc != 0:
            self._err(rc)
        return out

    def hc_post(self, f: torch.Tensor, state: torch.Tensor, post: torch.Tensor, comb: torch.Tensor,
                out: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
        """Enqueues hc_post of a sublayer body's output f [rows, hidden]; returns the new state."""
        c = self.config
        self._check_state(state)
        rows = state.shape[0]
        for name, t, shape in (("f", f, (rows, c.hidden)), ("post", post, (rows, c.hc)),
                               ("comb", comb, (rows, c.hc, c.hc))):
            if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != shape:
                raise ValueError(f"{name} must be a contiguous CUDA float32 {list(shape)} tensor")
        if out is None:
            out = torch.empty_like(state)
        s = stream if stream is not None else torch.cuda.current_stream(state.device)
        rc = self._lib.moe_ffn_hc_post(self._h, f.data_ptr(), state.data_ptr(), post.data_ptr(), comb.data_ptr(),
                                       rows, out.data_ptr(), s.cuda_stream)
        if rc != 0:
            self._err(rc)
        return out

    def _check_state(self, state: torch.Tensor):
        c = self.config
        if state.dtype != torch.float32 or not state.is_cuda or not state.is_contiguous() or state.dim() != 3 \
                or state.shape[1:] != (c.hc, c.hidden):
            raise ValueError(f"state must be a contiguous CUDA float32 [rows, {c.hc}, {c.hidden}] tensor")

    def status(self) -> int:
        rc = self._lib.moe_ffn_status(self._h)
        if rc < 0:
            self._err(rc)
        return rc

    def debug(self, name: str) -> np.ndarray:
        """An intermediate of the last forward, copied to the host."""
        c, r = self.config, self.last_rows
        shapes = {"pre": (r, c.hc), "post": (r, c.hc), "comb": (r, c.hc, c.hc), "ffn_norm": (r, c.hidden),
                  "logits": (r, c.experts), "indices": (r, c.top_k), "weights": (r, c.top_k),
                  "safe_indices": (r, c.top_k), "ffn_output": (r, c.hidden)}
        dt = {"indices": np.int32, "safe_indices": np.uint32}.get(name, np.float32)
        a = np.empty(shapes[name], dt)
        rc = self._lib.moe_ffn_debug_copy(self._h, DEBUG_BUFFERS[name], a.ctypes.data, a.nbytes)
        if rc != 0:
            self._err(rc)
        return a

    def set_stage_timing(self, enable: bool):
        rc = self._lib.moe_ffn_set_stage_timing(self._h, 1 if enable else 0)
        if rc != 0:
            self._err(rc)

    def set_fault_injection(self, which: str | None, wait_limit_us: int = 0):
        """Test hook: make one bounded in-kernel wait run out on later forwards ("decode": the decode
        kernel's last phase; "gemm": CTA 0 of the gate/up GEMM; None: off), with every in-kernel
        wait bounded by wait_limit_us (0: the kernels' defaults)."""
        code = {None: 0, "decode": 1, "gemm": 2}[which]
        rc = self._lib.moe_ffn_set_fault_injection(self._h, code, int(wait_limit_us))
        if rc != 0:
            self._err(rc)

    def stage_times(self) -> list[tuple[str, float]]:
        """(kernel name, ms) of each kernel of the last forward made with stage timing on."""
        ms = (ctypes.c_float * 16)()
        names = (ctypes.c_char_p * 16)()
        n = self._lib.moe_ffn_stage_times(self._h, ms, names, 16)
        if n < 0:
            self._err(n)
        return [(names[i].decode(), float(ms[i])) for i in range(n)]

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            self._lib.moe_ffn_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
