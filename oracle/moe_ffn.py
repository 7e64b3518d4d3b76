"""CPU oracle of the DeepSeek-V4 routed-MoE FFN block with hyper-connections.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the bench's
``cpu_baseline`` / reference leg may import or run this module; the library path
never does.  It shares no code with the CUDA path: inputs come from ``synth``,
which holds none of the block's arithmetic.

Source: docs.rs page "hf2q 0.1.3 src/inference/models/deepseek4/ffn_forward.rs",
function ``forward_ffn_rows``.  That page is host code: it names each device stage
(its ``dispatch_*`` / ``raw_matmul`` / ``expert_matmul`` calls), their buffers,
shapes and dtypes, but prints no kernel body.  Each function below states the
stage it follows and, where the page leaves the arithmetic open, the reading
taken.  All arithmetic is float64 (``dtype`` can be set to float32 to measure the
effect of precision); bf16 weights are widened exactly.

Quantised experts: the page consumes the expert matrices as raw GGUF types without naming one.
The quantised mode here reads them as MXFP8 (OCP Microscaling: E4M3 codes, one E8M0 power-of-two
scale per 32 consecutive elements of a row); ``mxfp8_to_float`` decodes that format by its
definition, and the rest of the block is unchanged.

Parity unpinned (fixed by reading, not by the page): the orientation of the comb
matrix in hc_post (out_i = sum_j comb[i, j] * state_j), the Sinkhorn start, order and
iteration count (exp(a - rowmax); rows then columns; 20), the absence of any eps in
the Sinkhorn sums and in pre/post, and the hash-route weight rule
(sigmoid of the chosen logits, normalised).
"""
from __future__ import annotations

import numpy as np

F64 = np.float64


def bf16_to_float(u16: np.ndarray, dtype=F64) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) exactly: the bf16 value is the top half of an f32."""
    return (np.asarray(u16).astype(np.uint32) << 16).view(np.float32).astype(dtype)


def e4m3_to_float(q: np.ndarray, dtype=F64) -> np.ndarray:
    """OCP 8-bit floating point E4M3 codes (uint8) to values: sign bit 7; exponent field bits 3-6
    with bias 7; mantissa bits 0-2.  Exponent field 0: subnormal (m / 8) * 2^-6; else
    (1 + m / 8) * 2^(e - 7); exponent 15 with mantissa 7 is NaN (the format has no infinities)."""
    q = np.asarray(q).astype(np.int64)
    e, m = (q >> 3) & 0xF, q & 0x7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2((e - 7).astype(np.float64)))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(q & 0x80, -mag, mag).astype(dtype)


def e8m0_to_float(s: np.ndarray, dtype=F64) -> np.ndarray:
    """OCP MX E8M0 scale codes to values 2^(s - 127); code 255 is NaN."""
    s = np.asarray(s).astype(np.int64)
    return np.where(s == 255, np.nan, np.exp2((s - 127).astype(np.float64))).astype(dtype)


def mxfp8_to_float(q: np.ndarray, s: np.ndarray, dtype=F64) -> np.ndarray:
    """MXFP8 matrix [rows, K] (E4M3 codes) with scales [rows, K / 32]: element k of a row is its
    code's value times the scale of block k // 32.  Exact in float64."""
    v = e4m3_to_float(q, dtype).reshape(*q.shape[:-1], q.shape[-1] // 32, 32)
    return (v * e8m0_to_float(s, dtype)[..., None]).reshape(q.shape)


def expert_weights(case, which: str, e, dtype=F64) -> np.ndarray:
    """Matrix `which` (gate, up, down) of routed expert e, or of the shared expert when e is None,
    widened from the workload's storage (bf16, or MXFP8 when cfg.weights is "mxfp8")."""
    if getattr(case.cfg, "weights", "bf16") == "mxfp8":
        return mxfp8_to_float(*(case.shared_mx(which) if e is None else case.expert_matrix_mx(which, int(e))), dtype)
    if e is None:
        return bf16_to_float({"gate": case.gate_sh, "up": case.up_sh, "down": case.down_sh}[which], dtype)
    return bf16_to_float(case.expert_matrix(which, int(e)), dtype)


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


# ---- hyper-connection prelude -----------------------------------------------------------------

def rms_norm_no_scale(x: np.ndarray, eps: float) -> np.ndarray:
    """``rms_norm_no_scale_f32`` over the flattened [rows, hc*hidden] state:
    y = x / sqrt(mean(x^2) + eps), no weight."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps)


def hc_mixes(state_norm: np.ndarray, hc_fn: np.ndarray) -> np.ndarray:
    """``raw_matmul`` "HC FFN function": mixes[r, m] = sum_c state_norm[r, c] * hc_fn[m, c],
    c = h*hidden + d (the [rows, hc*hidden] flat view), m < (2+hc)*hc."""
    return state_norm @ hc_fn.T


def hc_split_sinkhorn(mixes: np.ndarray, hc_scale: np.ndarray, hc_base: np.ndarray, hc: int,
                      iters: int):
    """``dispatch_hc_split_sinkhorn``: (mixes, hc_scale, hc_base) -> (pre, post, comb).

    Reading: the (2+hc)*hc mixes split as [pre (hc) | post (hc) | comb (hc*hc, row-major
    i*hc + j)], the order of the call's outputs.  Segment s is scaled by hc_scale[s] before
    hc_base is added.  pre = sigmoid(a), post = 2*sigmoid(a).  comb starts at
    exp(a - max_j a[i, j]) and is then made doubly stochastic by ``iters`` Sinkhorn sweeps,
    each dividing every row by its sum and then every column by its sum.
    """
    dt = mixes.dtype
    a_pre = mixes[:, :hc] * hc_scale[0] + hc_base[:hc]
    a_post = mixes[:, hc:2 * hc] * hc_scale[1] + hc_base[hc:2 * hc]
    a_comb = (mixes[:, 2 * hc:] * hc_scale[2] + hc_base[2 * hc:]).reshape(-1, hc, hc)
    pre = sigmoid(a_pre)
    post = 2.0 * sigmoid(a_post)
    comb = np.exp(a_comb - a_comb.max(axis=2, keepdims=True))
    for _ in range(iters):
        comb = comb / comb.sum(axis=2, keepdims=True)   # each row i sums to 1
        comb = comb / comb.sum(axis=1, keepdims=True)   # each column j sums to 1
    return pre.astype(dt), post.astype(dt), comb.astype(dt)


def hc_pre(state: np.ndarray, pre: np.ndarray) -> np.ndarray:
    """``dispatch_hc_pre`` (state, pre) -> ffn_input [rows, hidden]:
    ffn_input[r, d] = sum_h pre[r, h] * state[r, h, d]."""
    return np.einsum("rh,rhd->rd", pre, state)


def rms_norm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """``rms_norm`` with the ffn_norm weight: y = x / sqrt(mean(x^2) + eps) * w."""
    return rms_norm_no_scale(x, eps) * w


# ---- router -------------------------------------------------------------------------------------

def router_logits(xf: np.ndarray, gate: np.ndarray) -> np.ndarray:
    """``raw_matmul`` "MoE gate": logits[r, e] = sum_d xf[r, d] * gate[e, d]."""
    return xf @ gate.T


def selection_scores(logits: np.ndarray, bias: np.ndarray) -> np.ndarray:
    """The values the top-k decision is taken on, in the pages' buffer precision (f32):
    the logits buffer is f32, score = sigmoid(logit) rounded to f32, plus the f32 bias,
    rounded to f32 (the correctly rounded f32 sum)."""
    l32 = np.asarray(logits).astype(np.float32).astype(F64)
    s32 = sigmoid(l32).astype(np.float32).astype(F64)
    return (s32 + np.asarray(bias, np.float32).astype(F64)).astype(np.float32)


def topk_desc(values: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest entries of each row, largest first; equal values go to the
    lower index (a stable sort of the negated values)."""
    order = np.argsort(-values.astype(F64), axis=1, kind="stable")
    return order[:, :k].astype(np.int32)


def score_route(logits: np.ndarray, bias: np.ndarray, top_k: int):
    """``dispatch_deepseek_moe_score_route`` (logits, exp_probs_b) -> (indices, weights).

    Scores are sigmoid(logits); the top_k experts are chosen on score + bias (slots in
    descending biased score); weights are the chosen *unbiased* scores normalised to sum 1.
    """
    idx = topk_desc(selection_scores(logits, bias), top_k)
    s = sigmoid(logits)
    chosen = np.take_along_axis(s, idx.astype(np.int64), axis=1)
    w = chosen / chosen.sum(axis=1, keepdims=True)
    return idx, w


def selection_margin(logits: np.ndarray, bias: np.ndarray, top_k: int) -> np.ndarray:
    """Smallest gap between consecutive values among the top_k+1 largest selection scores of
    each row (float64).  A row with a small margin has a near-tie that decides membership of
    or order in the top-k; the workload generator redraws such rows."""
    v = np.sort(selection_scores(logits, bias).astype(F64), axis=1)[:, ::-1]
    n = min(top_k + 1, v.shape[1])
    gaps = v[:, : n - 1] - v[:, 1:n]
    return gaps.min(axis=1) if gaps.shape[1] else np.full(v.shape[0], np.inf)


def hash_route(logits: np.ndarray, token_ids: np.ndarray, tid2eid: np.ndarray, vocab: int):
    """``dispatch_deepseek_moe_hash_route`` (logits, token ids, tid2eid) -> (indices, weights).

    indices = tid2eid[token] in table order.  Reading for the weights: sigmoid of the chosen
    logits, normalised over the valid slots.  A token outside [0, vocab) gives index -1 in
    every slot; a table entry outside [0, experts) stays as it is (sanitize masks it).
    """
    rows, k = token_ids.shape[0], tid2eid.shape[1]
    experts = logits.shape[1]
    idx = np.full((rows, k), -1, np.int32)
    ok = (token_ids >= 0) & (token_ids < vocab)
    idx[ok] = tid2eid[token_ids[ok]]
    valid = (idx >= 0) & (idx < experts)
    s = sigmoid(logits)
    chosen = np.where(valid, np.take_along_axis(s, np.where(valid, idx, 0).astype(np.int64), axis=1), 0.0)
    tot = chosen.sum(axis=1, keepdims=True)
    w = np.divide(chosen, tot, out=np.zeros_like(chosen), where=tot > 0)
    return idx, w


def sanitize(idx: np.ndarray, experts: int):
    """``dispatch_deepseek_moe_sanitize_indices``: i32 -> u32 "safe" indices.  Reading: a valid
    index is kept, an invalid one (<0 or >= experts) becomes 0; the weighted reduce, which reads
    the original indices, gives such a slot no weight."""
    valid = (idx >= 0) & (idx < experts)
    return np.where(valid, idx, 0).astype(np.uint32), valid


# ---- experts ------------------------------------------------------------------------------------

def swiglu(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """``dispatch_deepseek_moe_swiglu`` with no third operand: silu(g) * u = g * sigmoid(g) * u."""
    return g * sigmoid(g) * u


def expert_ffn(x: np.ndarray, G: np.ndarray, U: np.ndarray, Dn: np.ndarray) -> np.ndarray:
    """One expert on rows x [n, hidden]: gate and up projections (``expert_matmul`` / ``raw_matmul``
    "gate", "up"), SwiGLU, down projection: y = swiglu(x G^T, x U^T) Dn^T."""
    return swiglu(x @ G.T, x @ U.T) @ Dn.T


def weighted_reduce(idx: np.ndarray, w: np.ndarray, routed: np.ndarray, shared: np.ndarray,
                    experts: int) -> np.ndarray:
    """``dispatch_deepseek_moe_weighted_reduce`` (indices, weights, routed_down [rows, k, hidden],
    shared_down [rows, hidden]) -> ffn_output = sum over valid slots of w * routed + shared."""
    valid = (idx >= 0) & (idx < experts)
    wv = np.where(valid, w, 0.0)
    return np.einsum("rk,rkd->rd", wv, routed) + shared


def hc_post(f: np.ndarray, state: np.ndarray, post: np.ndarray, comb: np.ndarray) -> np.ndarray:
    """``dispatch_hc_post`` (ffn_output, state, post, comb) -> out_state [rows, hc, hidden]:
    out[r, i, d] = post[r, i] * f[r, d] + sum_j comb[r, i, j] * state[r, j, d]."""
    return post[:, :, None] * f[:, None, :] + np.einsum("rij,rjd->rid", comb, state)


# ---- the hyper-connection prelude of any sublayer -------------------------------------------------

def hc_sublayer_pre(state: np.ndarray, hc_fn: np.ndarray, hc_scale: np.ndarray, hc_base: np.ndarray,
                    norm_w: np.ndarray, hc: int, iters: int, eps: float, dtype=F64):
    """The HC prelude a sublayer runs on the state before its body, for the attention sublayer
    (docs.rs "hf2q 0.1.3 src/inference/models/deepseek4/attention_forward.rs": rms_norm_no_scale_f32,
    raw_matmul "HC attention function", dispatch_hc_split_sinkhorn, dispatch_hc_pre, then rms_norm
    with attn_norm) and the same five stages of the FFN sublayer (ffn_forward.rs, with the HC FFN
    function and ffn_norm).  state [rows, hc, hidden]; hc_fn bf16 bits [(2+hc)*hc, hc*hidden].
    Returns the pre, post and comb of the sublayer, its input x = hc_pre(state, pre) and the
    normalised input x_norm its body consumes.  The sublayer's output f is folded back by
    ``hc_post`` (the attention page's last stage, dispatch_hc_post on the output projection)."""
    state = state.astype(dtype)
    rows = state.shape[0]
    flat = state.reshape(rows, -1)
    mixes = hc_mixes(rms_norm_no_scale(flat, eps), bf16_to_float(hc_fn, dtype))
    pre, post, comb = hc_split_sinkhorn(mixes, hc_scale.astype(dtype), hc_base.astype(dtype), hc, iters)
    x = hc_pre(state, pre)
    x_norm = rms_norm(x, norm_w.astype(dtype), eps)
    return dict(mixes=mixes, pre=pre, post=post, comb=comb, x=x, x_norm=x_norm)


# ---- whole block --------------------------------------------------------------------------------

def prelude_and_route(case, dtype=F64, rows=None):
    """Stages up to and including sanitize, for all rows (or the given row indices)."""
    c = case.cfg
    sel = np.arange(c.rows) if rows is None else np.asarray(rows)
    state = case.state[sel].astype(dtype)
    flat = state.reshape(len(sel), c.hc * c.hidden)
    state_norm = rms_norm_no_scale(flat, c.rms_eps)
    mixes = hc_mixes(state_norm, bf16_to_float(case.hc_fn, dtype))
    pre, post, comb = hc_split_sinkhorn(mixes, case.hc_scale.astype(dtype), case.hc_base.astype(dtype),
                                        c.hc, c.sinkhorn_iters)
    ffn_input = hc_pre(state, pre)
    xf = rms_norm(ffn_input, case.ffn_norm.astype(dtype), c.rms_eps)
    logits = router_logits(xf, bf16_to_float(case.gate, dtype))
    if c.is_hash:
        idx, w = hash_route(logits, case.token_ids[sel], case.tid2eid, c.vocab)
        margin = np.full(len(sel), np.inf)
    else:
        idx, w = score_route(logits, case.exp_probs_b, c.top_k)
        margin = selection_margin(logits, case.exp_probs_b, c.top_k)
    safe, valid = sanitize(idx, c.experts)
    return dict(rows=sel, state=state, mixes=mixes, pre=pre, post=post, comb=comb, ffn_input=ffn_input,
                ffn_norm=xf, logits=logits, indices=idx, weights=w.astype(dtype), safe_indices=safe,
                valid=valid, margin=margin)


def forward_ffn_rows(case, dtype=F64, rows=None, stages=None):
    """The whole block for the selected rows (all by default): returns a dict of every stage's
    output, ending with ``out_state`` [n, hc, hidden].  Expert weights are drawn per expert from
    the workload generator and widened exactly to ``dtype``."""
    c = case.cfg
    st = prelude_and_route(case, dtype, rows) if stages is None else stages
    n = len(st["rows"])
    xf = st["ffn_norm"]
    routed = np.zeros((n, c.top_k, c.hidden), dtype)
    for e in np.unique(st["safe_indices"][st["valid"]]):
        r_k = np.argwhere((st["indices"] == e))
        G = expert_weights(case, "gate", e, dtype)
        U = expert_weights(case, "up", e, dtype)
        Dn = expert_weights(case, "down", e, dtype)
        y = expert_ffn(xf[r_k[:, 0]], G, U, Dn)
        routed[r_k[:, 0], r_k[:, 1]] = y
    shared = expert_ffn(xf, expert_weights(case, "gate", None, dtype), expert_weights(case, "up", None, dtype),
                        expert_weights(case, "down", None, dtype))
    f = weighted_reduce(st["indices"], st["weights"], routed, shared, c.experts)
    out = hc_post(f, st["state"], st["post"], st["comb"])
    st.update(routed_down=routed, shared_down=shared, ffn_output=f, out_state=out)
    return st
