#!/usr/bin/env python3
"""Benchmark of the FlashMap one-jump block-draft step on GB300.

One step = the whole hot path for one batch: the context-KV write of the verify
window's committed columns, the anchor row, the noise embedding and the DiT
(flashmap_draft_block), and the folded head with whole-block sampling
(flashmap_sample_block). Inputs are synthetic and resident in HBM; the step is
captured once in a CUDA graph and replayed; the timed region is bracketed by a
barrier and synchronizations and timed with CUDA events on the launch stream. Each
step streams ~3 GB of weights, far above the 129 MB L2, so nothing survives in L2
between steps.

Prints one JSON line (rank 0). --impl reference times the CPU oracle instead.
"""

from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from speculative_decoding_block_context_gb300 import synthetic as syn  # noqa: E402

METRIC = "drafted tokens/sec (batch x block_size / s)"
UNIT = "tokens/s"


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# --------------------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the GPU works."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.device = device
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        self.t_start = time.time()

    def stop(self, t0: float, t1: float) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for ln in f:
                parts = [p.strip() for p in ln.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        # samples are ~100 ms apart: keep those around the timed region
        n = len(rows)
        span = max(time.time() - self.t_start, 1e-3)
        sel = [r for i, r in enumerate(rows) if t0 - 0.3 <= self.t_start + span * i / max(n, 1) <= t1 + 0.3] or rows
        sm = [float(r[1]) for r in sel if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in sel if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[j] for r in sel for j in range(4) if r[5 + j].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(sel)}


# --------------------------------------------------------------------------- our arm


def algorithmic_bytes(cfg: dict, req: dict, deferred_write: bool = False) -> dict:
    """Bytes the step must move: every weight once (bf16, or e4m3 plus one float32
    scale per output channel), the context K/V of positions 0..p of every request, the
    window and anchor rows written, the logits. With the window write deferred into the
    draft the all-layer context K/V weight is read once for both (the separate write
    call reads it again)."""
    H, Lt, D, L, F, Vd, V, K = (cfg[k] for k in ("target_hidden", "num_target_layers", "hidden", "num_layers",
                                                 "intermediate", "draft_vocab_size", "vocab_size", "block_size"))
    es = 4 if cfg["act_dtype"] == "f32" else 2
    wes = 1 if cfg.get("weight_dtype") == "e4m3" else es  # e4m3 weights: one byte (+ a scale per row)
    Vd = Vd if 0 < Vd < V else V
    bs = req["bs"]
    w_write = ((D * Lt * H + (0 if deferred_write else 2 * L * D * D)) * wes
               + (D + (0 if deferred_write else 2 * L * D)) * 4 * (wes == 1)) if req["window"] else 0
    w_draft = ((D * H + 2 * L * D * D + D * H + L * (6 * D * D + 2 * D * F)) * wes + H * H * es
               + (D + 2 * L * D + D + L * (6 * D + D + F)) * 4 * (wes == 1))
    w_head = Vd * D * wes + Vd * 4 * (wes == 1)
    kv_row = L * 2 * D * (1 if cfg.get("kv_dtype") == "e4m3" else es)
    kv_read = sum((p + 1) * kv_row for p in req["anchor_pos"])
    n = cfg.get("num_steps", 1)
    if cfg.get("noise_path", 0) == 1:
        # the folded eigenbasis: one act-dtype (D x H) projection instead of the noise
        # factor L (H x H) and x_embed (D x H)
        w_draft += D * H * es - H * H * es - D * H * wes - D * 4 * (wes == 1)
    if n > 1:
        # several jumps: the anchor projection and context K/V once; per jump the DiT,
        # x_embed's projection, E^T (act dtype) and the float32 state read and written;
        # between jumps the full-vocabulary head (act dtype); no noise factor L; every
        # jump's cross-attention reads the context again
        R = bs * K
        w_draft = ((D * H + 2 * L * D * D) * wes + (D + 2 * L * D) * 4 * (wes == 1)
                   + n * ((D * H + L * (6 * D * D + 2 * D * F)) * wes + (D + L * (6 * D + D + F)) * 4 * (wes == 1)
                          + H * V * es + 2 * R * V * 4)
                   + (n - 1) * V * D * es)
        kv_read *= n
    rows_written = (sum(req["commit"]) if req["window"] else 0) + bs
    # a tree draft: the logits of every candidate block; the context is read once per
    # request (the candidates share it), the algorithmic minimum
    nc = req["tree"][0] if req.get("tree") else 1
    logits = bs * nc * K * Vd * 4
    x_in = (bs * (K + 1) * Lt * H * es) if req["window"] else 0
    full = bs * K * V * 4 if req["full_scatter"] else 0
    total = w_write + w_draft + w_head + kv_read + rows_written * kv_row + logits + x_in + full
    draft_sample = w_draft + w_head + kv_read + bs * kv_row + logits + full
    return {"weights": w_write + w_draft + w_head, "kv_read": kv_read, "total": total, "draft_sample": draft_sample}


def setup_ours(workload: str, device: str):
    from speculative_decoding_block_context_gb300 import _lib as F

    cfg = syn.model_config(workload)
    W, E, LM, rank = syn.make_model(cfg, device)
    model = F.flashmap_load_weights(cfg, W, E, LM, rank)
    torch.cuda.synchronize()
    del W, LM
    req = syn.make_requests(workload, device)
    bs, K = req["bs"], cfg["block_size"]
    dt = syn.torch_dtype(cfg["act_dtype"])
    code = F.DTYPE_CODES[cfg["kv_dtype"]]
    pool_t = torch.empty(F.flashmap_pool_bytes(cfg, req["num_pages"]), dtype=torch.uint8, device=device)
    pool = F.make_pool(pool_t, req["num_pages"], code)
    nc = req["tree"][0] if req["tree"] else 1  # drafted blocks per request
    max_rows = max(max(req["ctx"]) if req["prefill"] else 0, bs * (K + 1))
    ws = torch.empty(F.flashmap_workspace_size(model, bs * nc, min(max_rows, 4096)), dtype=torch.uint8,
                     device=device)
    i32 = dict(dtype=torch.int32, device=device)
    if req["prefill"]:
        for b in range(bs):
            X = req["prefill_hidden"][b]
            F.flashmap_write_context_kv(model, pool, X, 1, X.shape[0], req["req_pool_idx"][b : b + 1],
                                        torch.zeros(1, **i32), None, req["req_to_page"], None, ws)
        req.pop("prefill_hidden")
    else:
        syn.fill_pool_random(pool_t.view(syn.torch_dtype(cfg["kv_dtype"])), req["kv_generator_seed"])
    Vd = cfg["draft_vocab_size"] if 0 < cfg["draft_vocab_size"] < cfg["vocab_size"] else cfg["vocab_size"]
    st = dict(
        F=F, cfg=cfg, model=model, E=E, req=req, pool_t=pool_t, pool=pool, ws=ws,
        start=torch.tensor(req["ctx"], **i32), commit=torch.tensor(req["commit"], **i32),
        anchor_pos=torch.tensor(req["anchor_pos"], **i32),
        hidden=torch.empty((bs * nc * K, cfg["hidden"]), dtype=dt, device=device),
        tokens=torch.empty(bs * nc * K, dtype=torch.int64, device=device),
        logits=torch.empty((bs * nc * K, Vd), dtype=torch.float32, device=device),
        full=(torch.empty((bs * K, cfg["vocab_size"]), dtype=torch.float32, device=device)
              if req["full_scatter"] else None),
        window_loc=torch.empty(bs * (K + 1), dtype=torch.int64, device=device),
    )
    if req["tree"]:
        # every candidate block samples with its request's position, temperature and seed
        n, width = req["tree"]
        st["tree_in"] = {k: v.repeat_interleave(n) for k, v in (
            ("anchor_pos", st["anchor_pos"]), ("temperature", req["temperature"]), ("greedy", req["greedy"]),
            ("seeds", req["seeds"]))}
        st["tree_out"] = [torch.empty((bs, width - 1), dtype=torch.int64, device=device) for _ in range(2)] + \
            [torch.empty((bs, 2), dtype=torch.int64, device=device)]
    return st


def blocks_per_step(st: dict) -> int:
    """Drafted blocks of one step: one per request, or one per candidate of a tree draft."""
    return st["req"]["bs"] * (st["req"]["tree"][0] if st["req"]["tree"] else 1)


def draft_call(st: dict, stream=None) -> None:
    F, req = st["F"], st["req"]
    if req["tree"]:
        F.flashmap_draft_candidates(st["model"], st["pool"], req["bs"], req["tree"][0], req["anchor_ids"],
                                    st["anchor_pos"], req["req_pool_idx"], req["req_to_page"], req["seeds"], 1.0,
                                    st["hidden"], None, st["ws"], stream)
    else:
        F.flashmap_draft_block(st["model"], st["pool"], req["bs"], req["anchor_ids"], st["anchor_pos"],
                               req["req_pool_idx"], req["req_to_page"], req["seeds"], 1.0, st["hidden"], None,
                               st["ws"], stream)


def sample_call(st: dict, stream=None) -> None:
    F, req = st["F"], st["req"]
    if req["tree"]:
        t = st["tree_in"]
        F.flashmap_sample_block(st["model"], blocks_per_step(st), st["hidden"], t["anchor_pos"], t["temperature"],
                                t["greedy"], t["seeds"], req["step"], st["tokens"], st["logits"], st["full"],
                                st["ws"], stream)
        n, width = req["tree"]
        F.flashmap_build_tree(st["tokens"].view(req["bs"], n, -1), width, *st["tree_out"], stream)
    else:
        F.flashmap_sample_block(st["model"], req["bs"], st["hidden"], st["anchor_pos"], req["temperature"],
                                req["greedy"], req["seeds"], req["step"], st["tokens"], st["logits"], st["full"],
                                st["ws"], stream)


def deferred(st: dict) -> bool:
    """The verify-window write goes into the draft call (one context K/V GEMM for the
    window rows and the anchors) unless --separate-write asks for three calls; tree
    drafts keep the separate write."""
    return bool(st["req"]["window"]) and not st["req"]["tree"] and not st.get("separate_write")


def write_call(st: dict, stream=None) -> None:
    F, req, cfg = st["F"], st["req"], st["cfg"]
    F.flashmap_write_context_kv(st["model"], st["pool"], req["window_hidden"], req["bs"], cfg["block_size"] + 1,
                                req["req_pool_idx"], st["start"], st["commit"], req["req_to_page"], st["window_loc"],
                                st["ws"], stream)


def draft_with_write_call(st: dict, stream=None) -> None:
    F, req, cfg = st["F"], st["req"], st["cfg"]
    F.flashmap_draft_block_with_write(st["model"], st["pool"], req["window_hidden"], cfg["block_size"] + 1,
                                      st["start"], st["commit"], st["window_loc"], req["bs"], req["anchor_ids"],
                                      st["anchor_pos"], req["req_pool_idx"], req["req_to_page"], req["seeds"], 1.0,
                                      st["hidden"], None, st["ws"], stream)


def run_step(st: dict, stream=None) -> None:
    if deferred(st):
        draft_with_write_call(st, stream)
    else:
        if st["req"]["window"]:
            write_call(st, stream)
        draft_call(st, stream)
    sample_call(st, stream)


def roofline_entry(roof: dict, chain, hbm_peak: float, peak_src: str, ms_step: float, workload: str) -> dict:
    """The roofline object of the dominant kernel (the tcgen05 GEMM): from the GEMM
    chain timed as one graph where it applies, else from the eager per-launch events."""
    traffic = profiled_traffic(workload)
    out = {"bound": "hbm", "peak": hbm_peak, "unit": "GB/s", "peak_source": f"{peak_src} hbm_gbs",
           "kernel": "tc_linear_kernel (tcgen05 GEMM, every launch of a step)", "traffic": traffic,
           "traffic_source": ("ncu dram__bytes_read.sum + dram__bytes_write.sum per GEMM launch, from "
                              f"profiles/tc_linear_step_{workload}.md, whose kernel source hash matches csrc/gemm.cu"
                              if traffic is not None else "no ncu summary for the current csrc/gemm.cu")}
    if chain is not None:
        out.update(achieved=round(chain["achieved_gbs"], 1), frac=round(chain["achieved_gbs"] / hbm_peak, 4),
                   bytes_per_launch=round(chain["bytes_per_launch"]), us_per_launch=round(chain["us_per_launch"], 2),
                   launches_per_step=chain["launches"],
                   gemm_ms_per_step=round(chain["ms_chain"], 4),
                   gemm_time_within_step=bool(chain["ms_chain"] <= ms_step),
                   timing=("the step's GEMM launches alone (flashmap_profile_gemm_chain), one CUDA graph replayed "
                           "between one event pair; achieved = algorithmic bytes / graph time"))
    else:
        out.update(achieved=round(roof["achieved_gbs"], 1), frac=round(roof["achieved_gbs"] / hbm_peak, 4),
                   bytes_per_launch=round(roof["bytes_per_launch"]), us_per_launch=round(roof["ms_per_launch"] * 1e3, 2),
                   launches_per_step=roof["launches_per_step"],
                   timing="eager step with an event pair around every launch (several-jump drafts)")
    return out


def gemm_roofline(st: dict, stream: torch.cuda.Stream, hbm_peak: float, steps: int = 3) -> dict:
    """Event-timed launches of the tcgen05 GEMM over `steps` eager steps on the launch
    stream: algorithmic bytes (weights + activations read, float32 outputs written)
    per launch over the mean launch duration."""
    F = st["F"]
    es = 4 if st["cfg"]["act_dtype"] == "f32" else 2
    e4m3 = st["cfg"].get("weight_dtype") == "e4m3"
    with torch.cuda.stream(stream):
        F.flashmap_profile_start(st["model"], 100000)
        for _ in range(steps):
            run_step(st)
        recs = F.flashmap_profile_stop(st["model"], 100000)
    gem = [r for r in recs if r[0] == "gemm"]
    by_kind = {}
    for r in recs:
        by_kind[r[0]] = by_kind.get(r[0], 0.0) + r[5] / steps
    # e4m3 weights: one byte per element plus a float32 scale per channel, except the
    # noise factor L (square H x H), which stays bf16
    H = st["cfg"]["target_hidden"]

    V, D = st["cfg"]["vocab_size"], st["cfg"]["hidden"]
    act_shapes = {(H, H)}  # the noise factor L stays in act dtype; so do E^T and the full head of several jumps
    if st["cfg"].get("num_steps", 1) > 1:
        act_shapes = {(H, V), (V, D)}

    def wbytes(n, k):
        return n * k * es if not e4m3 or (n, k) in act_shapes else n * k + n * 4

    byts = sum(wbytes(n, k) + rows * k * es + rows * n * 4 for _, _, rows, n, k, _ in gem) / len(gem)
    ms = sum(r[5] for r in gem) / len(gem)
    achieved = byts / (ms * 1e-3) / 1e9
    return {"kernel": "tc_linear_kernel (tcgen05 GEMM, all launches of a step)", "bytes_per_launch": byts,
            "ms_per_launch": ms, "launches_per_step": len(gem) // steps, "achieved_gbs": achieved,
            "ms_by_kind_per_step": {k: round(v, 4) for k, v in sorted(by_kind.items())},
            "launches_per_step_total": len(recs) // steps}


def gemm_chain_roofline(st: dict, stream: torch.cuda.Stream, n: int = 30):
    """The step's tcgen05 GEMM launches alone (flashmap_profile_gemm_chain: the same
    shapes, weights and launch configuration, back to back with programmatic
    dependent launch), captured in one CUDA graph and replayed n times between one
    pair of events on the launch stream: algorithmic bytes per launch over the mean
    launch duration. None where the chain does not apply (several jumps)."""
    F, req, cfg = st["F"], st["req"], st["cfg"]
    if cfg.get("num_steps", 1) > 1:
        return None
    bs = blocks_per_step(st)
    window = cfg["block_size"] + 1 if req["window"] else 0
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        byts, launches = F.flashmap_profile_gemm_chain(st["model"], bs, window, st["hidden"], st["ws"])
        with torch.cuda.graph(g, stream=stream):
            F.flashmap_profile_gemm_chain(st["model"], bs, window, st["hidden"], st["ws"])
        for _ in range(3):
            g.replay()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(n):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    return {"bytes_per_chain": byts, "launches": launches, "ms_chain": ms, "bytes_per_launch": byts / launches,
            "us_per_launch": ms * 1e3 / launches, "achieved_gbs": byts / (ms * 1e-3) / 1e9}


def profiled_traffic(workload: str):
    """DRAM bytes per GEMM launch from the committed ncu summary of this workload, or
    None when there is none or csrc/gemm.cu changed since the counters were taken."""
    import hashlib

    path = os.path.join(ROOT, "profiles", f"tc_linear_step_{workload}.md")
    src = os.path.join(ROOT, "speculative_decoding_block_context_gb300", "csrc", "gemm.cu")
    try:
        kv = {}
        with open(path) as f:
            for ln in f:
                if ":" in ln and ln.split(":")[0] in ("traffic_bytes_per_launch", "kernel_source_sha256"):
                    k, v = ln.split(":", 1)
                    kv[k] = v.strip()
        with open(src, "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()
        return int(kv["traffic_bytes_per_launch"]) if kv.get("kernel_source_sha256") == sha else None
    except (OSError, KeyError, ValueError):
        return None


def phase_times(st: dict, stream: torch.cuda.Stream, n: int = 60) -> dict:
    """The step's three calls captured as separate graphs and replayed n times each,
    every replay timed with its own event pair on the launch stream: median and p90 in
    microseconds (write only when the workload writes a verify window)."""
    F, req, cfg = st["F"], st["req"], st["cfg"]
    bs, K = req["bs"], cfg["block_size"]
    calls = {}
    if req["window"]:
        calls["write"] = lambda: write_call(st)  # the separate write call, for reference
    calls["draft"] = lambda: draft_call(st)
    if deferred(st):
        calls["draft_with_write"] = lambda: draft_with_write_call(st)
    calls["sample"] = lambda: sample_call(st)  # a tree draft's sample phase includes the tree
    out = {}
    for name, fn in calls.items():
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            fn()
            with torch.cuda.graph(g, stream=stream):
                fn()
            for _ in range(3):
                g.replay()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        with torch.cuda.stream(stream):
            for a, b in ev:
                a.record(stream)
                g.replay()
                b.record(stream)
        torch.cuda.synchronize()
        us = np.array([a.elapsed_time(b) * 1e3 for a, b in ev])
        out[name] = {"median_us": round(float(np.median(us)), 1), "p90_us": round(float(np.percentile(us, 90)), 1)}
    return out


# Configurations the default (batch-1) run also times, each on its own model and pool
# after the batch-1 line is measured: batch 32 (ragged contexts), batch 128 (window
# write and full-vocabulary scatter), e4m3 weights at batch 64.
EXTRA_WORKLOADS = ("qwen3_8b_bs32", "qwen3_8b_bs128", "qwen3_8b_fp8_bs64")


def time_workload(workload: str, device: str, stream: torch.cuda.Stream, hbm_peak: float, steps: int = 20,
                  warmup: int = 3) -> dict:
    """One workload's step as a replayed CUDA graph (events around `steps` replays on
    the launch stream, after `warmup` replays), its per-call phases and its step
    roofline; the model and pool are released afterwards."""
    st = setup_ours(workload, device)
    F, cfg, req = st["F"], st["cfg"], st["req"]
    with torch.cuda.stream(stream):
        for _ in range(2):
            run_step(st)
    torch.cuda.synchronize()
    err = F.flashmap_get_device_error(st["model"])
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            run_step(st)
        for _ in range(warmup):
            graph.replay()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    phases = phase_times(st, stream, n=20)
    ab = algorithmic_bytes(cfg, req, deferred(st))
    tokens = blocks_per_step(st) * cfg["block_size"]
    out = {"ms_per_step": round(ms, 4), "value": round(tokens / (ms * 1e-3), 1), "unit": UNIT, "steps": steps,
           "batch": req["bs"], "dtype": cfg["act_dtype"], "weight_dtype": cfg["weight_dtype"],
           "context": {"min": min(req["ctx"]), "max": max(req["ctx"]), "mean": float(np.mean(req["ctx"]))},
           "phases": phases, "device_error": err,
           "step_roofline": {"algorithmic_bytes": ab["total"],
                             "achieved_gbs": round(ab["total"] / (ms * 1e-3) / 1e9, 1),
                             "frac_of_measured_hbm": round(ab["total"] / (ms * 1e-3) / 1e9 / hbm_peak, 4),
                             "frac_of_8tbs": round(ab["total"] / (ms * 1e-3) / 1e9 / 8000.0, 4)}}
    del graph, st
    torch.cuda.empty_cache()
    return out


def world_max(value: float, world: int, device) -> float:
    """The largest of every rank's value (the slowest rank's step time); identity at N=1."""
    if world <= 1:
        return float(value)
    t = torch.tensor([float(value)], device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank_step: int, world: int, ms_max: float) -> float:
    """Whole-job drafted tokens/s: every rank drafts its own batch (requests are
    sharded across ranks, weak scaling) and the job takes the slowest rank's time."""
    return tokens_per_rank_step * world / (ms_max * 1e-3)


def our_arm(args, rank: int, world: int) -> dict:
    device = f"cuda:{int(os.environ.get('LOCAL_RANK', '0'))}"
    torch.cuda.set_device(device)
    hbm_peak, tf_peak, peak_src = load_peaks()
    st = setup_ours(args.workload, device)
    st["separate_write"] = args.separate_write
    F, cfg, req = st["F"], st["cfg"], st["req"]
    bs, K = req["bs"], cfg["block_size"]
    stream = torch.cuda.Stream(device=device)
    # eager warm-up, then capture one step
    with torch.cuda.stream(stream):
        for _ in range(2):
            run_step(st)
    torch.cuda.synchronize()
    err = F.flashmap_get_device_error(st["model"])
    if err:
        raise RuntimeError(f"device error word {err} during warm-up")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            run_step(st)
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            graph.replay()
    torch.cuda.synchronize()
    t_ev0, t_ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    with torch.cuda.stream(stream):
        t_ev0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        t_ev1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    ms = world_max(t_ev0.elapsed_time(t_ev1) / args.steps, world, device)
    clocks = sampler.stop(t0, t1)
    tokens_per_step = blocks_per_step(st) * K * world
    value = job_throughput(blocks_per_step(st) * K, world, ms)

    # end to end through the public API with host buffers: pinned inputs copied in,
    # the step, the sampled token ids copied out, every step
    host_in = {k: req[k].cpu().pin_memory() for k in ("anchor_ids", "seeds", "temperature", "greedy")}
    host_in["anchor_pos"] = st["anchor_pos"].cpu().pin_memory()
    dev_in = {k: req[k] for k in ("anchor_ids", "seeds", "temperature", "greedy")}
    dev_in["anchor_pos"] = st["anchor_pos"]
    if req["window"]:
        host_in["window_hidden"] = req["window_hidden"].cpu().pin_memory()
        dev_in["window_hidden"] = req["window_hidden"]
    result = [st["tokens"]]
    if req["tree"]:  # candidates sample with per-block copies of the request inputs; the tree comes back
        for k, t in st["tree_in"].items():
            host_in["tree_" + k] = t.cpu().pin_memory()
            dev_in["tree_" + k] = t
        result = st["tree_out"][:2]
    tok_host = [torch.empty(t.shape, dtype=torch.int64).pin_memory() for t in result]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in tok_host)

    def e2e_loop(step_fn, n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(n):
                for k, t in host_in.items():
                    dev_in[k].copy_(t, non_blocking=True)
                step_fn()
                for h, t in zip(tok_host, result):
                    h.copy_(t, non_blocking=True)
            e1.record(stream)
        torch.cuda.synchronize()
        return world_max(e0.elapsed_time(e1) / n, world, device)

    # the three C-ABI calls (write, draft, sample) issued every step, no graph
    with torch.cuda.stream(stream):
        for _ in range(3):
            run_step(st)
    e2e_ms = e2e_loop(lambda: run_step(st), args.steps)
    # the same step replayed from the captured graph
    e2e_graph_ms = e2e_loop(graph.replay, args.steps)

    roof = gemm_roofline(st, stream, hbm_peak)
    chain = gemm_chain_roofline(st, stream)
    phases = phase_times(st, stream)
    ab = algorithmic_bytes(cfg, req, deferred(st))
    t_ds = (phases["draft"]["median_us"] + phases["sample"]["median_us"]) * 1e-6
    launches = roof["launches_per_step_total"]
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "draft_step_us": round(ms * 1e3, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": cfg["act_dtype"],
        "data": "synthetic (seeded random weights and inputs of the workload's shapes)",
        "config": {"workload": args.workload, "batch": bs, "block_size": K,
                   "context": {"min": min(req["ctx"]), "max": max(req["ctx"]),
                               "mean": float(np.mean(req["ctx"]))},
                   "window_write": ("deferred into the draft call" if deferred(st) else
                                    "its own call" if req["window"] else None),
                   "full_vocab_scatter": bool(req["full_scatter"]),
                   "tree": ({"candidates": req["tree"][0], "width": req["tree"][1]} if req["tree"] else None),
                   "parallelism": f"replicas x{world} (requests sharded, no collective)",
                   "l2": "inputs larger than L2 (weights alone ~3 GB per step)", "cuda_graph": True},
        "e2e": {"value": round(tokens_per_step / (e2e_ms * 1e-3), 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
                "how": "every step: pinned host inputs copied in, the step's C-ABI calls ("
                       + ("flashmap_draft_block_with_write, flashmap_sample_block" if deferred(st) else
                          "flashmap_write_context_kv, flashmap_draft_block, flashmap_sample_block" if req["window"] else
                          "flashmap_draft_block, flashmap_sample_block")
                       + ") made through the Python binding (no graph), token ids copied out"},
        "e2e_graph": {"value": round(tokens_per_step / (e2e_graph_ms * 1e-3), 1), "unit": UNIT,
                      "ms_per_step": round(e2e_graph_ms, 4),
                      "how": "the same copies around a replay of the step's captured CUDA graph"},
        "gpu_launches": launches * args.steps,
        "roofline": roofline_entry(roof, chain, hbm_peak, peak_src, ms, args.workload),
        "step_roofline": {"algorithmic_bytes": ab["total"], "achieved_gbs": round(ab["total"] / (ms * 1e-3) / 1e9, 1),
                          "frac_of_measured_hbm": round(ab["total"] / (ms * 1e-3) / 1e9 / hbm_peak, 4),
                          "frac_of_8tbs": round(ab["total"] / (ms * 1e-3) / 1e9 / 8000.0, 4)},
        # the draft step proper (draft + sample calls, each its own graph), against the
        # bytes it must move (the window write's weights and rows excluded)
        "phases": phases,
        "draft_sample_roofline": {"algorithmic_bytes": ab["draft_sample"],
                                  "us": round(t_ds * 1e6, 1),
                                  "frac_of_measured_hbm": round(ab["draft_sample"] / t_ds / 1e9 / hbm_peak, 4),
                                  "frac_of_8tbs": round(ab["draft_sample"] / t_ds / 1e9 / 8000.0, 4)},
        "breakdown_ms_per_step_eager": roof["ms_by_kind_per_step"],
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, budget_s=args.cpu_budget)
    if world == 1 and args.workload == "qwen3_8b_bs1" and not args.no_extra_configs:
        # the other configurations, timed after the batch-1 line (not part of its value)
        del graph, st
        torch.cuda.empty_cache()
        line["other_configs"] = {w: time_workload(w, device, stream, hbm_peak) for w in EXTRA_WORKLOADS}
    return line


# --------------------------------------------------------------------------- the oracle arm


def oracle_setup(workload: str, device: str, gen_model=None):
    """Numpy inputs for the oracle: weights, constants (gram replaced by the identity:
    the value of L does not change the work of a step), request inputs."""
    from oracle import flashmap_ref as ref

    cfg = syn.model_config(workload)
    if gen_model is None:
        W, E, LM, rank = syn.make_model(cfg, device)
    else:
        W, E, LM, rank = gen_model
    Wnp = {k: v.double().cpu().numpy() for k, v in W.items()}
    Enp = E.float().cpu().numpy()
    LMnp = LM.float().cpu().numpy()
    ocfg = ref.Config.from_dict(cfg)
    C = ref.load_constants(ocfg, Wnp, Enp, LMnp, rank.cpu().numpy(), skip_gram=True)
    C.extra["LM"] = LMnp  # the full-vocabulary head of a several-jump draft
    return ocfg, Wnp, Enp, C


def oracle_step(ref, ocfg, Wnp, Enp, C, req, b: int, ctx_kv, window_hidden) -> None:
    """One request's whole step on the CPU oracle: window write, anchor row, draft
    (every jump of a several-jump draft; every candidate block and the verify tree of a
    tree draft), folded head, sampling."""
    K = ocfg.block_size
    kc, vc = ctx_kv
    if req["window"]:
        m = req["commit"][b]
        kw, vw = ref.write_rows_kv(ocfg, Wnp, window_hidden[:m], req["ctx"][b] + np.arange(m))
        kc, vc = np.concatenate([kc, kw], 1), np.concatenate([vc, vw], 1)
    p = req["anchor_pos"][b]
    ka, va = ref.anchor_kv(ocfg, Wnp, Enp, [int(req["anchor_ids"][b])], [p])
    kc, vc = np.concatenate([kc, ka], 1), np.concatenate([vc, va], 1)
    seed = int(req["seeds"][b])
    n = req["tree"][0] if req.get("tree") else 1
    if ocfg.num_steps > 1:
        hids = ref.draft_requests_multi(ocfg, Wnp, C, Enp, C.extra["LM"], [(kc, vc)], [p], [seed], ocfg.num_steps)
    else:
        hids = ref.draft_requests(ocfg, Wnp, C, [(kc, vc)] * n, [p] * n, [seed] * n, 1.0, list(range(n)))
    toks = []
    for hid in hids:
        lg = ref.head_logits(C, hid)
        toks.append(ref.sample_rows(lg, [float(req["temperature"][b])] * K, [int(req["greedy"][b])] * K,
                                    [seed] * K, p + 1 + np.arange(K), req["step"], C.hot)[0])
    if req.get("tree"):
        ref.build_tree(np.stack(toks), req["tree"][1])


def time_oracle(workload: str, device: str, n_steps: int, budget_s: float = 90.0, warmup: int = 1,
                gen_model=None, req=None):
    """Times up to n_steps oracle steps (stopping once budget_s is spent, at least one),
    each one request of the workload: requests are independent, so a step of bs
    requests costs bs of these. Returns (seconds per request-step, steps timed)."""
    from oracle import flashmap_ref as ref

    ocfg, Wnp, Enp, C = oracle_setup(workload, device, gen_model)
    req = req or syn.make_requests(workload, device)
    rng = np.random.default_rng(0)
    L, nh, hd = ocfg.num_layers, ocfg.num_heads, ocfg.head_dim
    times = []
    spent = 0.0
    for i in range(warmup + n_steps):
        b = i % req["bs"]
        n = req["ctx"][b]
        # context keys/values of positions 0..ctx-1 (their values do not change the work)
        kc = rng.standard_normal((L, n, nh, hd)).astype(np.float32)
        vc = rng.standard_normal((L, n, nh, hd)).astype(np.float32)
        wh = req["window_hidden"][b].float().cpu().numpy() if req["window"] else None
        t0 = time.perf_counter()
        oracle_step(ref, ocfg, Wnp, Enp, C, req, b, (kc, vc), wh)
        dt = time.perf_counter() - t0
        if i >= warmup:
            times.append(dt)
            spent += dt
            if spent > budget_s:
                break
    return float(np.mean(times)), len(times)


def cores_used() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def tokens_per_request(workload: str) -> int:
    """Drafted tokens of one request-step: block_size, times the candidates of a tree draft."""
    tree = syn.WORKLOADS[workload].get("tree")
    return syn.model_config(workload)["block_size"] * (tree[0] if tree else 1)


def cpu_baseline(workload: str, budget_s: float = 30.0) -> dict:
    K = tokens_per_request(workload)
    sec, n = time_oracle(workload, "cuda", 3, budget_s=budget_s)
    return {"value": round(K / sec, 3), "unit": UNIT, "cores": cores_used(), "kind": "oracle",
            "sample": f"{n} request-steps of {workload} (window write + anchor + draft + head + sampling of one "
                      f"request, {K} tokens each) on the NumPy float64 oracle, {sec:.2f} s each; load-time "
                      f"constants untimed, the E^T E factor replaced by the identity for timing"}


def reference_arm(args) -> dict:
    K = tokens_per_request(args.workload)
    sec, n = time_oracle(args.workload, "cuda" if torch.cuda.is_available() else "cpu", max(1, args.steps),
                         budget_s=90.0, warmup=min(args.warmup, 1))
    value = K / sec
    sample = (f"{n} request-steps of {args.workload} on the NumPy float64 oracle, each one request's window "
              f"write, anchor row, draft, head and sampling ({K} tokens); requests are independent, so a batch "
              f"costs bs request-steps; stopped after 90 s of timed work")
    return {"metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": 0, "steps": n,
            "steps_requested": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 2),
            "higher_is_better": True, "impl": "reference", "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload},
            "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": cores_used(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def kernel_case(args) -> dict:
    """One tcgen05 GEMM timed alone over --steps launches: "gemm" is the batch-1 shape
    (16 activation rows x the all-layer context K/V weight, 40960 x 4096 bf16 = 335 MB,
    above L2; HBM-bound), "gemm2048" the batch-128 MLP shape (2048 rows x 12288 x 4096;
    tensor-bound), "head2048" the batch-128 folded head (2048 rows x 32768 draft
    vocabulary x 4096; tensor-bound)."""
    from speculative_decoding_block_context_gb300 import _lib as F

    hbm_peak, tf_peak, src = load_peaks()
    rows, n, k = {"gemm": (16, 40960, 4096), "gemm512": (512, 12288, 4096),
                  "gemm2048": (2048, 12288, 4096), "head2048": (2048, 32768, 4096)}[args.kernel_case]
    g = torch.Generator(device="cuda").manual_seed(0)
    x = torch.randn((rows, k), generator=g, device="cuda").to(torch.bfloat16)
    w = (torch.randn((n, k), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    out = torch.zeros((rows, n), dtype=torch.float32, device="cuda")
    for _ in range(max(args.warmup, 3)):
        F.flashmap_debug_linear(F.BF16, x, w, out)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        F.flashmap_debug_linear(F.BF16, x, w, out)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    byts = n * k * 2 + rows * k * 2 + rows * n * 4
    flops = 2.0 * rows * n * k
    return {"kernel_case": args.kernel_case, "shape": [rows, n, k], "us_per_launch": round(ms * 1e3, 2),
            "achieved_gbs": round(byts / (ms * 1e-3) / 1e9, 1), "peak_gbs": hbm_peak, "peak_source": src,
            "frac_hbm": round(byts / (ms * 1e-3) / 1e9 / hbm_peak, 4),
            "achieved_tflops": round(flops / (ms * 1e-3) / 1e12, 1), "peak_tflops": tf_peak,
            "frac_tensor": round(flops / (ms * 1e-3) / 1e12 / tf_peak, 4)}


def main() -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="qwen3_8b_bs1", choices=sorted(syn.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--separate-write", action="store_true",
                    help="run the verify-window write as its own call instead of deferring it into the draft")
    ap.add_argument("--no-extra-configs", action="store_true",
                    help="skip the batch-32, batch-128 and e4m3 batch-64 steps the default run also times")
    ap.add_argument("--cpu-budget", type=float, default=30.0)
    ap.add_argument("--kernel-case", choices=["gemm", "gemm512", "gemm2048", "head2048"], default=None,
                    help="time one kernel alone instead of the step (profiling case)")
    args = ap.parse_args()
    if args.kernel_case:
        print(json.dumps(kernel_case(args)), flush=True)
        return 0
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(reference_arm(args)), flush=True)
        return 0
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device(f"cuda:{os.environ.get('LOCAL_RANK', '0')}"))
    line = our_arm(args, rank, world)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
