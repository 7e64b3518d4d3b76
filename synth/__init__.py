"""Seeded synthetic inputs for the DeepSeek-V4 routed-MoE FFN block.

This module draws numbers and nothing else: it holds none of the block's
arithmetic, and both the CPU oracle (tests) and the CUDA path (tests, bench)
take their inputs from it.  The drawing itself is plain C (``gen.c``), built
on first use, so that the 12.9 GB of full-shape expert weights are produced
in seconds and bit-identically on x86-64 and AArch64.

The five workloads are the ones the block is measured on: a tiny layer, a
B=1 score-routed decode, a B=4 hash-routed decode, a 512-row prefill whose
expert popularity follows Zipf(1.1), and a 4096-row prefill with eight hot
experts.  Distributions not fixed by the workload description follow the
tiny layer's (hc_base N(0,0.1), hc_scale [1,1,1], RMSNorm weights 1+N(0,0.05),
selection bias N(0,0.01), shared expert of the routed experts' shapes).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, replace
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_synth.so")
_SRC = os.path.join(_HERE, "gen.c")
_lib = None

# Tensor ids: each input tensor draws from its own stream.
T_STATE, T_HC_FN, T_HC_BASE, T_FFN_NORM, T_GATE, T_BIAS, T_TID2EID = 1, 2, 3, 4, 5, 6, 7
T_GATE_EXPS, T_UP_EXPS, T_DOWN_EXPS, T_GATE_SH, T_UP_SH, T_DOWN_SH = 8, 9, 10, 11, 12, 13
T_TOKENS, T_HOT, T_ZIPF_PERM = 14, 15, 16
T_HC_ATTN_FN, T_HC_ATTN_BASE, T_ATTN_NORM, T_ATTN_OUT = 17, 18, 19, 20

ZIPF_BIAS_FILE = os.path.join(os.path.dirname(_HERE), "tests", "golden", "zipf_exp_probs_b_seed3.txt")


def build(force: bool = False) -> str:
    """Compile gen.c into _synth.so (gcc, OpenMP, no fused multiply-add)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u64, u32, i64, i32, f64 = (ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int64,
                                   ctypes.c_int32, ctypes.c_double)
        vp = ctypes.c_void_p
        lib.synth_normal_f32.argtypes = [u64, u32, u32, u64, u64, f64, f64, vp]
        lib.synth_normal_bf16.argtypes = [u64, u32, u32, u64, u64, f64, f64, f64, vp]
        lib.synth_normal_rows_f32.argtypes = [u64, u32, vp, u64, u64, u64, f64, vp]
        lib.synth_uniform_i32.argtypes = [u64, u32, u32, u64, u64, i64, i64, vp]
        lib.synth_distinct_rows_i32.argtypes = [u64, u32, u64, u64, i32, i32, vp]
        lib.synth_distinct_rows_i32.restype = ctypes.c_int
        lib.synth_permutation.argtypes = [u64, u32, i32, vp]
        lib.synth_quantize_mxfp8.argtypes = [vp, u64, vp, vp]
        lib.synth_normal_mxfp8.argtypes = [u64, u32, u64, u64, f64, vp, vp]
        lib.synth_key.argtypes = [u64, u32, u32]
        lib.synth_key.restype = u64
        _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ---- raw draws -------------------------------------------------------------------------------

def normal_f32(seed, tensor, n, mean=0.0, sigma=1.0, start=0, attempt=0) -> np.ndarray:
    out = np.empty(n, np.float32)
    _load().synth_normal_f32(seed, tensor, attempt, start, n, mean, sigma, _ptr(out))
    return out


def normal_bf16(seed, tensor, n, sigma, start=0, gain=1.0, out: Optional[np.ndarray] = None) -> np.ndarray:
    """bf16 bit patterns (uint16) of N(0, sigma) draws times gain, rounded to nearest even."""
    if out is None:
        out = np.empty(n, np.uint16)
    assert out.dtype == np.uint16 and out.size == n
    _load().synth_normal_bf16(seed, tensor, 0, start, n, 0.0, sigma, gain, _ptr(out))
    return out


def quantize_mxfp8(v: np.ndarray):
    """MXFP8 (OCP MX, E4M3 elements, one E8M0 scale per 32 consecutive values) of float32 values,
    n a multiple of 32: (codes uint8 [n], scales uint8 [n / 32])."""
    v = np.ascontiguousarray(v, np.float32).ravel()
    assert v.size % 32 == 0
    q, s = np.empty(v.size, np.uint8), np.empty(v.size // 32, np.uint8)
    _load().synth_quantize_mxfp8(_ptr(v), v.size, _ptr(q), _ptr(s))
    return q, s


def normal_mxfp8(seed, tensor, n, sigma, start=0, out_q: Optional[np.ndarray] = None,
                 out_s: Optional[np.ndarray] = None):
    """MXFP8 of the N(0, sigma) draws that normal_bf16 rounds to bf16 (start, n multiples of 32)."""
    assert start % 32 == 0 and n % 32 == 0
    q = np.empty(n, np.uint8) if out_q is None else out_q
    s = np.empty(n // 32, np.uint8) if out_s is None else out_s
    assert q.dtype == np.uint8 and q.size == n and s.dtype == np.uint8 and s.size == n // 32
    _load().synth_normal_mxfp8(seed, tensor, start, n, sigma, _ptr(q), _ptr(s))
    return q, s


def normal_rows_f32(seed, tensor, attempts: np.ndarray, row_len, sigma=1.0) -> np.ndarray:
    attempts = np.ascontiguousarray(attempts, np.int32)
    out = np.empty((attempts.size, row_len), np.float32)
    _load().synth_normal_rows_f32(seed, tensor, _ptr(attempts), 0, attempts.size, row_len, sigma, _ptr(out))
    return out


def uniform_i32(seed, tensor, n, lo, hi, start=0, attempt=0) -> np.ndarray:
    out = np.empty(n, np.int32)
    _load().synth_uniform_i32(seed, tensor, attempt, start, n, lo, hi, _ptr(out))
    return out


def distinct_rows_i32(seed, tensor, rows, k, n_values) -> np.ndarray:
    out = np.empty((rows, k), np.int32)
    rc = _load().synth_distinct_rows_i32(seed, tensor, 0, rows, k, n_values, _ptr(out))
    if rc != 0:
        raise ValueError("k must be in 1..min(64, n_values)")
    return out


def permutation(seed, tensor, n) -> np.ndarray:
    out = np.empty(n, np.int32)
    _load().synth_permutation(seed, tensor, n, _ptr(out))
    return out


def bf16_bits_to_f32(u16: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 (a storage conversion, not arithmetic)."""
    return (u16.astype(np.uint32) << 16).view(np.float32)


# ---- workloads -------------------------------------------------------------------------------

@dataclass(frozen=True)
class MoeConfig:
    name: str
    rows: int
    hidden: int = 4096
    hc: int = 4
    experts: int = 256
    top_k: int = 6
    inter: int = 2048
    shared_inter: int = 2048
    vocab: int = 129280
    token_range: int = 129280
    n_layers: int = 4
    hash_layer_count: int = 3
    layer: int = 3
    seed: int = 1
    bias: str = "normal"          # "normal": N(0, 0.01); "zipf": calibrated table
    hot_experts: int = 0          # number of experts whose router rows are scaled by hot_gain
    hot_gain: float = 3.0
    sinkhorn_iters: int = 20
    rms_eps: float = 1e-6
    weight_sigma: float = 0.02
    weights: str = "bf16"         # expert matrices: "bf16", or "mxfp8" (the same draws in MXFP8)

    @property
    def mix(self) -> int:
        return (2 + self.hc) * self.hc

    @property
    def is_hash(self) -> bool:
        return self.layer < self.hash_layer_count

    @property
    def expert_bytes(self) -> int:
        return 3 * self.inter * self.hidden * 2


CONFIGS = {
    "c0_tiny": MoeConfig("c0_tiny", rows=4, hidden=256, experts=16, top_k=2, inter=128,
                         shared_inter=128, vocab=1024, token_range=1024, seed=0),
    "c1_decode_b1": MoeConfig("c1_decode_b1", rows=1, seed=1),
    "c2_decode_b4_hash": MoeConfig("c2_decode_b4_hash", rows=4, layer=0, seed=2),
    "c3_prefill_512": MoeConfig("c3_prefill_512", rows=512, seed=3, bias="zipf"),
    "c4_prefill_4096": MoeConfig("c4_prefill_4096", rows=4096, seed=4, hot_experts=8),
}


# Smaller variants for profiler captures (a few GB on the device): full hidden/inter, 32 experts.
PROFILE_CONFIGS = {
    "p_decode_b1_e32": MoeConfig("p_decode_b1_e32", rows=1, experts=32, seed=21),
    "p_decode_b4_e32": MoeConfig("p_decode_b4_e32", rows=4, experts=32, layer=0, seed=22),
    "p_prefill_512_e32": MoeConfig("p_prefill_512_e32", rows=512, experts=32, seed=23),
    # full router and HC shapes (256 experts, hidden 4096) with inter 128: 0.8 GB of expert weights
    "p_decode_b1_i128": MoeConfig("p_decode_b1_i128", rows=1, inter=128, shared_inter=128, seed=25),
    "p_prefill_4096_e32": MoeConfig("p_prefill_4096_e32", rows=4096, experts=32, seed=27),
    # 512 rows over all 256 experts with the Zipf bias, inter 512: the small expert tiles of the
    # 512-row prefill in 3.2 GB of expert weights
    "p_prefill_512_i512": MoeConfig("p_prefill_512_i512", rows=512, inter=512, shared_inter=512, seed=3,
                                    bias="zipf"),
    # 4096 rows with the 8 hot experts, inter 512: the 4096-row prefill's tiles in 3.2 GB of weights
    "p_prefill_4096_i512": MoeConfig("p_prefill_4096_i512", rows=4096, inter=512, shared_inter=512, seed=4,
                                     hot_experts=8),
}
ALL_CONFIGS = {**CONFIGS, **PROFILE_CONFIGS}


class Case:
    """All inputs of one workload, as host arrays.  Expert weights are drawn on demand.

    Layouts (row-major):  state f32 [rows, hc, hidden];  token_ids i32 [rows];
    hc_fn bf16 [(2+hc)*hc, hc*hidden];  hc_base f32 [(2+hc)*hc];  hc_scale f32 [3];
    ffn_norm f32 [hidden];  gate bf16 [experts, hidden];  exp_probs_b f32 [experts] (score layers);
    tid2eid i32 [vocab, top_k] (hash layers);  gate/up experts bf16 [experts, inter, hidden];
    down experts bf16 [experts, hidden, inter];  shared gate/up bf16 [shared_inter, hidden];
    shared down bf16 [hidden, shared_inter].
    """

    def __init__(self, cfg: MoeConfig, attempts: Optional[np.ndarray] = None, rows: Optional[int] = None):
        if rows is not None and rows != cfg.rows:
            cfg = replace(cfg, rows=rows)
        self.cfg = cfg
        c = cfg
        s = c.seed
        self.attempts = np.zeros(c.rows, np.int32) if attempts is None else np.asarray(attempts, np.int32).copy()
        self.state = normal_rows_f32(s, T_STATE, self.attempts, c.hc * c.hidden).reshape(c.rows, c.hc, c.hidden)
        self.token_ids = uniform_i32(s, T_TOKENS, c.rows, 0, c.token_range)
        self.hc_fn = normal_bf16(s, T_HC_FN, c.mix * c.hc * c.hidden, c.weight_sigma).reshape(c.mix, c.hc * c.hidden)
        self.hc_base = normal_f32(s, T_HC_BASE, c.mix, 0.0, 0.1)
        self.hc_scale = np.ones(3, np.float32)
        self.ffn_norm = normal_f32(s, T_FFN_NORM, c.hidden, 1.0, 0.05)
        gate = normal_bf16(s, T_GATE, c.experts * c.hidden, c.weight_sigma).reshape(c.experts, c.hidden)
        self.hot = np.zeros(0, np.int32)
        if c.hot_experts:
            self.hot = np.sort(permutation(s, T_HOT, c.experts)[: c.hot_experts])
            for e in self.hot:
                normal_bf16(s, T_GATE, c.hidden, c.weight_sigma, start=int(e) * c.hidden, gain=c.hot_gain,
                            out=gate[e])
        self.gate = gate
        self.exp_probs_b = None
        self.tid2eid = None
        if c.is_hash:
            self.tid2eid = distinct_rows_i32(s, T_TID2EID, c.vocab, c.top_k, c.experts)
        elif c.bias == "zipf":
            self.exp_probs_b = load_zipf_bias(c)
        else:
            self.exp_probs_b = normal_f32(s, T_BIAS, c.experts, 0.0, 0.01)
        n_sh = c.shared_inter * c.hidden
        self.gate_sh = normal_bf16(s, T_GATE_SH, n_sh, c.weight_sigma).reshape(c.shared_inter, c.hidden)
        self.up_sh = normal_bf16(s, T_UP_SH, n_sh, c.weight_sigma).reshape(c.shared_inter, c.hidden)
        self.down_sh = normal_bf16(s, T_DOWN_SH, n_sh, c.weight_sigma).reshape(c.hidden, c.shared_inter)

    # Expert weights: one [inter, hidden] (gate/up) or [hidden, inter] (down) matrix per expert.
    def expert_matrix(self, which: str, e: int, out: Optional[np.ndarray] = None) -> np.ndarray:
        c = self.cfg
        tensor = {"gate": T_GATE_EXPS, "up": T_UP_EXPS, "down": T_DOWN_EXPS}[which]
        n = c.inter * c.hidden
        m = normal_bf16(c.seed, tensor, n, c.weight_sigma, start=e * n, out=out)
        return m.reshape((c.hidden, c.inter) if which == "down" else (c.inter, c.hidden))

    def expert_block(self, which: str, e0: int, n_experts: int, out: np.ndarray) -> np.ndarray:
        """Fill out (uint16, n_experts * inter * hidden elements) with experts e0..e0+n_experts-1."""
        c = self.cfg
        tensor = {"gate": T_GATE_EXPS, "up": T_UP_EXPS, "down": T_DOWN_EXPS}[which]
        n = c.inter * c.hidden
        return normal_bf16(c.seed, tensor, n * n_experts, c.weight_sigma, start=e0 * n, out=out)

    # The expert matrices in MXFP8 (workloads with weights="mxfp8"): the same draws as the bf16
    # matrices, stored as E4M3 codes [rows, K] and E8M0 scales [rows, K / 32], K the contiguous axis.
    def expert_matrix_mx(self, which: str, e: int):
        c = self.cfg
        tensor = {"gate": T_GATE_EXPS, "up": T_UP_EXPS, "down": T_DOWN_EXPS}[which]
        n = c.inter * c.hidden
        q, s = normal_mxfp8(c.seed, tensor, n, c.weight_sigma, start=e * n)
        shape = (c.hidden, c.inter) if which == "down" else (c.inter, c.hidden)
        return q.reshape(shape), s.reshape(shape[0], shape[1] // 32)

    def expert_block_mx(self, which: str, e0: int, n_experts: int, out_q: np.ndarray, out_s: np.ndarray):
        """Fill out_q (n_experts * inter * hidden codes) and out_s (1/32 as many scales)."""
        c = self.cfg
        tensor = {"gate": T_GATE_EXPS, "up": T_UP_EXPS, "down": T_DOWN_EXPS}[which]
        n = c.inter * c.hidden
        return normal_mxfp8(c.seed, tensor, n * n_experts, c.weight_sigma, start=e0 * n, out_q=out_q, out_s=out_s)

    def shared_mx(self, which: str):
        c = self.cfg
        tensor = {"gate": T_GATE_SH, "up": T_UP_SH, "down": T_DOWN_SH}[which]
        q, s = normal_mxfp8(c.seed, tensor, c.shared_inter * c.hidden, c.weight_sigma)
        shape = (c.hidden, c.shared_inter) if which == "down" else (c.shared_inter, c.hidden)
        return q.reshape(shape), s.reshape(shape[0], shape[1] // 32)

    def attn_hc(self) -> dict:
        """The attention sublayer's hyper-connection weights, drawn like the FFN's: hc_attn_fn bf16
        [(2+hc)*hc, hc*hidden] N(0, weight_sigma), hc_attn_base f32 N(0, 0.1), hc_attn_scale ones,
        attn_norm f32 1 + N(0, 0.05); and attn_out f32 [rows, hidden] N(0, 1), a stand-in for the
        attention body's output that hc_post folds back into the state."""
        if getattr(self, "_attn", None) is None:
            c, s = self.cfg, self.cfg.seed
            self._attn = dict(
                hc_fn=normal_bf16(s, T_HC_ATTN_FN, c.mix * c.hc * c.hidden, c.weight_sigma).reshape(c.mix, c.hc * c.hidden),
                hc_base=normal_f32(s, T_HC_ATTN_BASE, c.mix, 0.0, 0.1),
                hc_scale=np.ones(3, np.float32),
                norm=normal_f32(s, T_ATTN_NORM, c.hidden, 1.0, 0.05),
                attn_out=normal_f32(s, T_ATTN_OUT, c.rows * c.hidden).reshape(c.rows, c.hidden))
        return self._attn

    def with_attempts(self, attempts: np.ndarray) -> "Case":
        return Case(self.cfg, attempts)


def load_zipf_bias(cfg: MoeConfig) -> np.ndarray:
    """Selection bias of the Zipf workload, written by tests/golden/make_zipf_bias.py."""
    if not os.path.exists(ZIPF_BIAS_FILE):
        raise FileNotFoundError(f"missing {ZIPF_BIAS_FILE}; run tests/golden/make_zipf_bias.py")
    vals = np.loadtxt(ZIPF_BIAS_FILE, dtype=np.float64, comments="#").astype(np.float32)
    if vals.shape != (cfg.experts,):
        raise ValueError("Zipf bias table has the wrong length")
    return vals


def zipf_targets(cfg: MoeConfig) -> np.ndarray:
    """Target share of routed slots per expert: Zipf(1.1) over a seeded permutation of the
    experts, water-filled so that no expert exceeds 1/top_k of the slots (an expert can be
    chosen at most once per token)."""
    e = cfg.experts
    perm = permutation(cfg.seed, T_ZIPF_PERM, e)
    p = np.empty(e)
    p[perm] = 1.0 / np.arange(1, e + 1) ** 1.1
    p /= p.sum()
    cap = 1.0 / cfg.top_k
    fixed = np.zeros(e, bool)
    for _ in range(e):
        over = (p > cap) & ~fixed
        if not over.any():
            break
        fixed |= over
        p[fixed] = cap
        free = ~fixed
        p[free] *= (1.0 - cap * fixed.sum()) / p[free].sum()
    return p
