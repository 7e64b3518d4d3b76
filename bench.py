"""Throughput of the GB300 MoE-FFN block (tokens/s per layer) on the synthetic workloads.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
                    [--extra | --no-extra]

One step = one forward of the whole block (HC prelude, router, experts, reduce, HC post) over one
batch of the workload, inputs resident in HBM, L2 flushed (a 256 MB write) before every step, each
step timed with CUDA events on the forward's stream.  Rank 0 prints one JSON line.  With N > 1
(torchrun) every rank runs its own replica of the workload (rows are independent: no collective
on the data path), the time is the max over ranks and the value counts every rank's tokens.

--impl reference times the CPU oracle instead (the only other arm: the pages ship no runnable
implementation), on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time
from dataclasses import replace

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE-FFN layer tokens/s (decode B=1/4, prefill 512) + % of HBM/TC roofline"
DEFAULT_WORKLOAD = "c1_decode_b1"
EXTRA_WORKLOADS = ["c2_decode_b4_hash", "c3_prefill_512", "c4_prefill_4096"]
FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def describe(cfg) -> str:
    route = "hash" if cfg.is_hash else "score"
    extra = {"c3_prefill_512": ", Zipf(1.1) expert popularity", "c4_prefill_4096": ", 8 hot experts (router rows x3)"}
    return (f"{cfg.name}: rows={cfg.rows}, hidden={cfg.hidden}, hc={cfg.hc}, experts={cfg.experts}, "
            f"top_k={cfg.top_k}, inter={cfg.inter}, shared expert inter={cfg.shared_inter}, {route} routing"
            f"{extra.get(cfg.name, '')}, seed {cfg.seed}"
            f"{', MXFP8 experts (E4M3, E8M0 scale per 32)' if cfg.weights == 'mxfp8' else ''}")


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---- algorithmic work ----------------------------------------------------------------------------

def work_model(cfg, indices: np.ndarray) -> dict:
    """Algorithmic bytes and flops of one forward from its routing (indices [rows, top_k])."""
    R, D, I, E, HC, M = cfg.rows, cfg.hidden, cfg.inter, cfg.experts, cfg.hc, cfg.mix
    valid = (indices >= 0) & (indices < E)
    groups = len(np.unique(indices[valid])) + 1          # touched routed experts + shared
    slots = int(valid.sum()) + R                          # (row, expert) pairs incl. shared
    wb = 1 + 1 / 32 if cfg.weights == "mxfp8" else 2    # bytes per expert weight: MXFP8 codes + scales, or bf16
    w_gateup = int(groups * 2 * I * D * wb)
    w_down = int(groups * D * I * wb)
    state = R * HC * D * 4
    small = M * HC * D * 2 + E * D * 2                    # hc_fn + router
    flops_experts = slots * 2 * 3 * I * D
    flops_router = R * (2 * E * D + 2 * M * HC * D)
    return dict(groups=groups, slots=slots, w_gateup=w_gateup, w_down=w_down, state=state, small=small,
                bytes_total=w_gateup + w_down + small + 2 * state, flops_total=flops_experts + flops_router,
                flops_gateup=slots * 2 * 2 * I * D, flops_down=slots * 2 * I * D)


def kernel_work(name: str, wm: dict, cfg) -> tuple[float, float]:
    """(algorithmic bytes, algorithmic flops) of one launch of a kernel of the forward."""
    R, D, I, HC, E, K = cfg.rows, cfg.hidden, cfg.inter, cfg.hc, cfg.experts, cfg.top_k
    slots = wm["slots"]
    if name == "decode":
        # the whole block in one launch: every touched expert once, hc_fn and the router, the state
        # read and written, the per-group act / y round trips
        return (wm["w_gateup"] + wm["w_down"] + wm["small"] + 2 * wm["state"] + slots * (I + D) * 4 * 2,
                wm["flops_gateup"] + wm["flops_down"] + 2 * R * (E + cfg.mix * HC) * D)
    # the tensor-core path's activations are f32 values held as two bf16 planes (4 B per element):
    # gate/up reads each slot's normalised input and writes its SwiGLU output; down reads that and
    # reduces into ffn_out, which is counted once (its R x hidden f32 result)
    if name == "gemm_gateup":
        return wm["w_gateup"] + slots * (D * 4 + I * 4), wm["flops_gateup"]
    if name == "gemm_down":
        return wm["w_down"] + slots * I * 4 + R * D * 4, wm["flops_down"]
    if name == "mix_gemm":
        return wm["state"] + cfg.mix * HC * D * 2, 2 * R * cfg.mix * HC * D
    if name == "mix_finish":
        return R * (cfg.mix + HC * (2 + HC)) * 4, 0.0
    if name == "prenorm":
        return wm["state"] + R * D * 4, 0.0
    if name == "router_gemm":
        return R * D * 4 + E * D * 2 + R * E * 4, 2 * R * E * D
    if name == "post":
        return 2 * wm["state"] + R * D * 4, 0.0  # state in, state out, ffn_out in
    if name == "scatter":
        return R * D * 4 + slots * D * 4, 0.0  # each normalised row read once, written per slot as hi + lo bf16
    return R * K * 4, 0.0


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch from ncu captures of the
# kernels as they stand, keyed by (kernel, rows, expert groups touched): the decode kernel streams
# every touched expert once, so a capture on the 32-expert profiling workload with the same
# routing width (6 routed + shared) carries the same bytes as the full workload.  A kernel change
# removes its entry until it is captured again.
NCU_TRAFFIC = {("decode", 1, 7): 354_256_128 + 3_561_728}


def roofline_entry(name: str, avg_ms: float, wm: dict, cfg, peaks: dict, peak_kind: str) -> dict:
    """The kernel's binding roofline: HBM bytes or tensor flops, whichever takes longer at peak."""
    nbytes, flops = kernel_work(name, wm, cfg)
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    s = avg_ms * 1e-3
    if t_tc > t_hbm:
        ach = flops / s / 1e12
        return dict(bound="tensor", achieved=round(ach, 1), peak=peaks["bf16_tflops"], unit="TFLOP/s",
                    frac=round(ach / peaks["bf16_tflops"], 4), alg=int(flops),
                    peak_source=f"{peak_kind} bf16_tflops (cuBLAS)")
    ach = nbytes / s / 1e9
    return dict(bound="hbm", achieved=round(ach, 1), peak=peaks["hbm_gbs"], unit="GB/s",
                frac=round(ach / peaks["hbm_gbs"], 4), alg=int(nbytes), peak_source=f"{peak_kind} hbm_gbs (copy)")


def max_over_ranks(x: float, dist, device) -> float:
    """The largest x over all ranks (the job's time is its slowest rank's); x itself with no group."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, rows_per_rank: int, steps: int, seconds: float) -> float:
    """Whole-job tokens/s: every rank's rows of every step over the slowest rank's time."""
    return world * rows_per_rank * steps / seconds


# ---- clocks ----------------------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                                          "-i", str(self.index), "-lms", "100"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---- our arm --------------------------------------------------------------------------------------

def run_ours(cfg, steps: int, warmup: int, device, rank: int, world: int, dist, peaks, peak_kind,
             want_e2e: bool, soak_s: float = 1.0) -> dict:
    import torch

    from deepseek_v4_moe_gb300 import MoeFFN, config_from
    from synth.device import upload

    case = synth.Case(cfg)
    mx = cfg.weights == "mxfp8"
    dev = upload(case, device, experts=not mx)
    m = MoeFFN(config_from(cfg), {cfg.layer: dev["weights"]})
    if mx:
        from synth.device import upload_mx
        m.set_mxfp8_experts(cfg.layer, upload_mx(case, device))
    stream = torch.cuda.Stream(device)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    out = torch.empty_like(dev["state"])
    tok = dev["token_ids"]

    def step():
        m.forward(dev["state"], tok, cfg.layer, out=out, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(max(warmup, 3)):
            flush.fill_(1.0)
            step()
    torch.cuda.synchronize(device)
    indices = m.debug("indices")
    wm = work_model(cfg, indices)

    sampler = ClockSampler(device.index if device.index is not None else 0)
    sampler.start()
    t_end = time.perf_counter() + soak_s  # load the GPU so the clock samples see this work
    with torch.cuda.stream(stream):
        while time.perf_counter() < t_end:
            flush.fill_(1.0)
            step()
            stream.synchronize()
    # ---- timed region: K steps, each bracketed by events on the forward's stream ----
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(device)
    wall0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(steps):
            flush.fill_(float(i))
            starts[i].record(stream)
            step()
            ends[i].record(stream)
    torch.cuda.synchronize(device)
    wall1 = time.perf_counter()
    if dist is not None:
        dist.barrier()
    clocks = sampler.stop()
    ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = max_over_ranks(float(sum(ms)), dist, device)
    res = dict(total_ms=total_ms, ms_per_step=total_ms / steps, median_ms=statistics.median(ms),
               value=job_rate(world, cfg.rows, steps, total_ms / 1e3), wall_s=wall1 - wall0, clocks=clocks, wm=wm)

    # ---- per-kernel durations: the same steps again with stage events ----
    m.set_stage_timing(True)
    per = {}
    n_kernels = 0
    with torch.cuda.stream(stream):
        for i in range(steps):
            flush.fill_(float(i))
            step()
            st = m.stage_times()
            n_kernels = len(st)
            for name, t in st:
                per.setdefault(name, []).append(t)
    m.set_stage_timing(False)
    kernels = []
    tot = sum(statistics.mean(v) for v in per.values())
    for name, v in per.items():
        avg = statistics.mean(v)
        rl = roofline_entry(name, avg, wm, cfg, peaks, peak_kind)
        kernels.append(dict(name=name, avg_us=round(avg * 1e3, 2), share=round(avg / tot, 4), bound=rl["bound"],
                            achieved=rl["achieved"], unit=rl["unit"], frac=rl["frac"], alg=rl["alg"]))
        per[name] = (v, rl)
    kernels.sort(key=lambda k: -k["avg_us"])
    top = kernels[0]
    res["kernels"] = kernels
    res["gpu_launches"] = n_kernels * steps
    rl = per[top["name"]][1]
    traffic = NCU_TRAFFIC.get((top["name"], cfg.rows, wm["groups"]))
    res["roofline"] = {"bound": rl["bound"], "kernel": top["name"], "achieved": rl["achieved"], "peak": rl["peak"],
                       "unit": rl["unit"], "frac": rl["frac"], "traffic": traffic, "peak_source": rl["peak_source"],
                       "alg_per_launch": rl["alg"],
                       "traffic_source": "ncu capture of decode_tc_kernel on p_decode_b1_e32 (same 7 expert groups)"
                       if traffic else None}
    # whole forward against its binding roofline
    t_hbm = wm["bytes_total"] / (peaks["hbm_gbs"] * 1e9)
    t_tc = wm["flops_total"] / (peaks["bf16_tflops"] * 1e12)
    step_s = res["ms_per_step"] / 1e3
    res["forward_roofline"] = {"alg_bytes": wm["bytes_total"], "alg_flops": wm["flops_total"],
                               "hbm_frac": round(t_hbm / step_s, 4), "tensor_frac": round(t_tc / step_s, 4),
                               "binding": "hbm" if t_hbm >= t_tc else "tensor",
                               "binding_frac": round(max(t_hbm, t_tc) / step_s, 4),
                               "distinct_experts": wm["groups"] - 1}

    if want_e2e:
        pin_in = torch.from_numpy(case.state.copy()).pin_memory()
        pin_tok = torch.from_numpy(case.token_ids.copy()).pin_memory()
        pin_out = torch.empty_like(pin_in).pin_memory()
        a_in, a_tok, a_out = pin_in.numpy(), pin_tok.numpy(), pin_out.numpy()
        for _ in range(max(warmup, 3)):
            m.forward_host(a_in, a_tok, cfg.layer, a_out, stream=stream)
        dts = []
        for i in range(steps):
            with torch.cuda.stream(stream):
                flush.fill_(float(i))
            stream.synchronize()
            t0 = time.perf_counter()
            m.forward_host(a_in, a_tok, cfg.layer, a_out, stream=stream)
            dts.append(time.perf_counter() - t0)
        e2e_s = max_over_ranks(sum(dts), dist, device)
        res["e2e"] = {"value": round(job_rate(world, cfg.rows, steps, e2e_s), 1), "unit": "tokens/s",
                      "h2d_bytes_per_step": int(a_in.nbytes + a_tok.nbytes), "d2h_bytes_per_step": int(a_out.nbytes),
                      "api": "moe_ffn_forward_host (pinned host buffers, synchronous)"}
    m.close()
    del dev, flush, out
    torch.cuda.empty_cache()
    return res


# ---- the hyper-connection prelude and post of a sublayer (attention), timed on their own ----------

HC_SUBLAYER_WORKLOADS = ["c1_decode_b1", "c4_prefill_4096"]
MX_WORKLOADS = ["c1_decode_b1", "c2_decode_b4_hash"]   # the same workloads on MXFP8 experts


def hc_sublayer_bytes(cfg) -> tuple[int, int]:
    """Algorithmic bytes of hc_pre (state once, hc_fn, norm weight, x_norm and pre/post/comb out)
    and of hc_post (f and state in, the new state out, post/comb in)."""
    R, D, HC, M = cfg.rows, cfg.hidden, cfg.hc, cfg.mix
    small = R * (2 * HC + HC * HC) * 4
    pre = R * HC * D * 4 + M * HC * D * 2 + D * 4 + R * D * 4 + small
    post = R * D * 4 + 2 * R * HC * D * 4 + R * (HC + HC * HC) * 4
    return pre, post


def run_hc_sublayer(cfg, steps: int, warmup: int, device, peaks) -> dict:
    """The attention sublayer's HC prelude (moe_ffn_hc_pre) and post (moe_ffn_hc_post) on the
    workload's state, L2 flushed before each, timed with CUDA events on their stream."""
    import torch

    from deepseek_v4_moe_gb300 import MoeFFN, config_from

    case = synth.Case(cfg)
    a = case.attn_hc()
    w = {k: torch.from_numpy(a[k].view(np.int16) if a[k].dtype == np.uint16 else a[k]).to(device)
         for k in ("hc_fn", "hc_base", "hc_scale", "norm")}
    m = MoeFFN(config_from(cfg), {})
    m.set_attn_hc(cfg.layer, w)
    state = torch.from_numpy(case.state).to(device)
    f = torch.from_numpy(a["attn_out"]).to(device)
    out = torch.empty_like(state)
    stream = torch.cuda.Stream(device)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    with torch.cuda.stream(stream):
        for i in range(max(warmup, 3) + steps):
            flush.fill_(float(i))
            timed = i >= max(warmup, 3)
            e = ev[i - max(warmup, 3)] if timed else None
            if timed:
                e[0].record(stream)
            p = m.hc_pre(state, cfg.layer, "attn", stream=stream)
            if timed:
                e[1].record(stream)
                # the post reads f and the state again: flush between, so it meets them in HBM
                flush.fill_(0.5)
                e[2].record(stream)
            m.hc_post(f, state, p["post"], p["comb"], out=out, stream=stream)
            if timed:
                e[3].record(stream)
    torch.cuda.synchronize(device)
    assert m.status() == 0
    pre_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    post_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in ev)
    m.close()
    b_pre, b_post = hc_sublayer_bytes(cfg)
    peak = peaks["hbm_gbs"]
    res = {}
    for name, ms, b in (("hc_pre", pre_ms, b_pre), ("hc_post", post_ms, b_post)):
        gbs = b / (ms * 1e-3) / 1e9
        res[name] = {"avg_us": round(ms * 1e3, 2), "alg_bytes": b, "achieved": round(gbs, 1), "unit": "GB/s",
                     "peak": peak, "frac": round(gbs / peak, 4),
                     "bound": "hbm" if cfg.rows > 4 else "latency (under 1 MB moved)"}
    res["rows"] = cfg.rows
    return res


# ---- several layers in one submission (moe_ffn_forward_layers) --------------------------------------

CHAIN_WORKLOADS = ["c1_decode_b1", "c2_decode_b4_hash"]
CHAIN_LAYERS = 4


def run_layer_chain(cfg, steps: int, warmup: int, device) -> dict:
    """CHAIN_LAYERS consecutive FFN blocks on the workload's rows, each on the previous one's
    output: launched one by one (eager) and as one captured chain (moe_ffn_forward_layers).  Every
    layer has weights of its own (the workload's generator with the seed offset per layer) and
    routes the way the workload's layer does; the L2 is flushed before each chain."""
    import torch

    from deepseek_v4_moe_gb300 import MoeFFN, config_from
    from synth.device import upload

    n = CHAIN_LAYERS
    ccfg = replace(cfg, n_layers=n, hash_layer_count=n if cfg.is_hash else 0)
    devs = [upload(synth.Case(replace(ccfg, seed=ccfg.seed + 1000 * l)), device) for l in range(n)]
    m = MoeFFN(config_from(ccfg), {l: d["weights"] for l, d in enumerate(devs)})
    state, tok = devs[0]["state"], devs[0]["token_ids"]
    bufs = [torch.empty_like(state), torch.empty_like(state)]
    out = torch.empty_like(state)
    stream = torch.cuda.Stream(device)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=device)

    def eager():
        x = state
        for l in range(n):
            x = m.forward(x, tok, l, out=bufs[l % 2], stream=stream)

    def chained():
        m.forward_layers(state, tok, 0, n, out=out, stream=stream)

    res = {}
    for name, fn in (("eager", eager), ("graph", chained)):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        with torch.cuda.stream(stream):
            for i in range(max(warmup, 3) + steps):
                flush.fill_(float(i))
                k = i - max(warmup, 3)
                if k >= 0:
                    ev[k][0].record(stream)
                fn()
                if k >= 0:
                    ev[k][1].record(stream)
        torch.cuda.synchronize(device)
        ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
        res[name] = {"us_per_layer": round(ms * 1e3 / n, 2), "tokens_per_s_per_layer": round(cfg.rows * n / (ms / 1e3), 1)}
    assert torch.equal(out, bufs[(n - 1) % 2]), "the chain differs from the layers launched one by one"
    assert m.status() == 0
    m.close()
    res.update(layers=n, rows=cfg.rows, weights="distinct per layer")
    del devs
    torch.cuda.empty_cache()
    return res


# ---- oracle (CPU baseline and reference arm) ------------------------------------------------------

class _CachedCase:
    """The workload with its expert matrices drawn up front, so the oracle's timing holds its own
    arithmetic only (the bf16 -> f64 widening included)."""

    def __init__(self, case, experts):
        self.__dict__.update(case.__dict__)
        self._cache = {(w, int(e)): case.expert_matrix(w, int(e)) for e in experts for w in ("gate", "up", "down")}

    def expert_matrix(self, which, e, out=None):
        return self._cache[(which, int(e))]


def oracle_rate(cfg, rows_sample: int, target_s: float):
    """Oracle tokens/s on `rows_sample` rows of the workload (full block per row), the forward over
    those rows repeated until `target_s` seconds of oracle work have been timed."""
    import oracle
    n = max(1, rows_sample)
    case = synth.Case(replace(cfg, rows=n))
    st = oracle.prelude_and_route(case)
    cached = _CachedCase(case, np.unique(st["indices"][(st["indices"] >= 0) & (st["indices"] < cfg.experts)]))
    dt, passes = 0.0, 0
    while dt < target_s:
        t0 = time.perf_counter()
        oracle.forward_ffn_rows(cached)
        dt += time.perf_counter() - t0
        passes += 1
    return n * passes / dt, dt, n, passes


def run_reference(cfg, steps: int, warmup: int, budget_s: float = 150.0) -> dict:
    import oracle
    per_step_rows = 1
    case = synth.Case(replace(cfg, rows=max(1, steps + warmup)))
    st_all = oracle.prelude_and_route(case)
    cached = _CachedCase(case, np.unique(st_all["indices"][(st_all["indices"] >= 0)
                                                          & (st_all["indices"] < cfg.experts)]))
    for i in range(warmup):
        oracle.forward_ffn_rows(cached, rows=[i])
    times = []
    t_start = time.perf_counter()
    for i in range(steps):
        t0 = time.perf_counter()
        oracle.forward_ffn_rows(cached, rows=[warmup + i])
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_start > budget_s:
            break
    total = sum(times)
    return dict(value=len(times) * per_step_rows / total, ms_per_step=1e3 * total / len(times), timed=len(times))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(synth.ALL_CONFIGS))
    ap.add_argument("--soak", type=float, default=1.0, help="seconds of untimed load before the timed steps")
    ap.add_argument("--no-e2e", dest="e2e", action="store_false", default=True)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--extra", dest="extra", action="store_true", default=True)
    ap.add_argument("--no-extra", dest="extra", action="store_false")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false", default=True)
    ap.add_argument("--weights", choices=["bf16", "mxfp8"], default="bf16",
                    help="expert weight format of the workload (mxfp8: a profiling and comparison mode)")
    ap.add_argument("--section", choices=["hc_sublayer", "layer_chain"], default=None,
                    help="time only this extra section on --workload and print its JSON (for profiling)")
    args = ap.parse_args()
    warmup = max(args.warmup, 3)
    cfg = replace(synth.ALL_CONFIGS[args.workload], weights=args.weights)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    peaks, peak_kind = load_peaks()
    config = {"workload": describe(cfg), "rows_per_rank": cfg.rows, "layer": cfg.layer,
              "l2": "flushed before every step (256 MB write)", "parallelism": f"replicas x{world}"}

    if args.impl == "reference":
        if rank != 0:
            return
        ref = run_reference(cfg, args.steps, warmup)
        cores = os.cpu_count()
        line = {"impl": "reference", "metric": METRIC, "value": round(ref["value"], 4), "unit": "tokens/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": warmup, "ms_per_step": round(ref["ms_per_step"], 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": config,
                "cpu_baseline": {"value": round(ref["value"], 4), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                 "sample": f"{ref['timed']} of {args.steps} steps timed (150 s budget), one row of the "
                                           f"workload per step, expert weights drawn before timing"},
                "e2e": {"value": round(ref["value"], 4), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    import torch
    dist = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl")
        dist = tdist
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)

    if args.section is not None:
        if args.section == "hc_sublayer":
            res = run_hc_sublayer(cfg, args.steps, warmup, device, peaks)
        else:
            res = run_layer_chain(cfg, args.steps, warmup, device)
        if rank == 0:
            print(json.dumps({"section": args.section, "workload": args.workload, **res}), flush=True)
        return
    main_res = run_ours(cfg, args.steps, warmup, device, rank, world, dist, peaks, peak_kind, want_e2e=args.e2e,
                        soak_s=args.soak)
    workloads = {}
    if args.extra:
        for name in EXTRA_WORKLOADS:
            if name == args.workload:
                continue
            c = synth.CONFIGS[name]
            r = run_ours(c, max(10, args.steps // 5), warmup, device, rank, world, dist, peaks, peak_kind,
                         want_e2e=False, soak_s=min(0.5, args.soak))
            workloads[name] = {"value": round(r["value"], 1), "unit": "tokens/s", "ms_per_step": round(r["ms_per_step"], 4),
                               "forward_roofline": r["forward_roofline"], "top_kernel": r["kernels"][0],
                               "kernels": r["kernels"], "clocks": r["clocks"]}
    mx = {}
    if args.extra:
        for name in MX_WORKLOADS:
            c = replace(synth.CONFIGS[name], weights="mxfp8")
            r = run_ours(c, max(10, args.steps // 5), warmup, device, rank, world, dist, peaks, peak_kind,
                         want_e2e=False, soak_s=min(0.5, args.soak))
            mx[name] = {"value": round(r["value"], 1), "unit": "tokens/s", "ms_per_step": round(r["ms_per_step"], 4),
                        "forward_roofline": r["forward_roofline"], "top_kernel": r["kernels"][0],
                        "clocks": r["clocks"], "weights": "MXFP8 (E4M3 + E8M0 per 32), 1.03 B per weight"}
    hc_sub = {}
    if args.extra:
        for name in HC_SUBLAYER_WORKLOADS:
            hc_sub[name] = run_hc_sublayer(synth.CONFIGS[name], 20, warmup, device, peaks)
    chain = {}
    if args.extra:
        for name in CHAIN_WORKLOADS:
            chain[name] = run_layer_chain(synth.CONFIGS[name], 20, warmup, device)
    cpu = None
    if rank == 0 and world == 1 and args.cpu_baseline:
        rate, dt, n, passes = oracle_rate(cfg, 8 if cfg.rows <= 4 else 4, 10.0)
        cpu = {"value": round(rate, 4), "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"{passes} passes over {n} rows of the workload's distribution (whole block per row, "
                         f"f64 NumPy), {dt:.1f} s timed; expert weights drawn before timing"}
    if rank == 0:
        line = {"metric": METRIC, "value": round(main_res["value"], 1), "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": warmup, "ms_per_step": round(main_res["ms_per_step"], 5),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16 weights, split-bf16 activations (hi + lo), f32 accumulate, f64 reductions",
                "data": "synthetic", "config": config, "roofline": main_res["roofline"],
                "forward_roofline": main_res["forward_roofline"], "kernels": main_res["kernels"],
                "cpu_baseline": cpu, "e2e": main_res.get("e2e"), "gpu_launches": main_res["gpu_launches"],
                "clocks": main_res["clocks"], "median_ms_per_step": round(main_res["median_ms"], 5),
                "workloads": workloads, "mxfp8_experts": mx, "hc_sublayer_attn": hc_sub, "layer_chain": chain}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
