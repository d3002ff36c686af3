"""Benchmark of the DARTree draft-tree build + verify round on one GB300.

One step = one dartree_round call (S1-S10: the draft-tree build and its
verification) over one batch of seeded synthetic inputs already resident in HBM. The default workload is the
Qwen3-4B-shaped single-request round (C=1, L=16, V=151936, H=2560, K=64, W=12,
B=64, bf16); the C=64 stress batch (H=4096, K=512) is measured in the same run
and reported under "c64". Prints one JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from dartree_inputs import (breadth_first_slot_depth, make_config, make_inputs, make_lm_head,  # noqa: E402
                            make_target_per_node)

MAIN_CFG = "cfg1_qwen3_4b_c1"
STRESS_CFG = "cfg4_c64_stress"
L2_BYTES = 129 * 1024 * 1024
CLOCKS_CSV = None  # where the clock samples of the timed region go (set by --clocks-csv)


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# --------------------------------------------------------------------------- algorithmic work (per round)
#
# The roofline numerator is the METHOD's work (the steps of one round as the method
# states them): base logits read once (S1), the stand-in head's weights and the
# candidates' embedding rows and block hidden rows (S2-S7), the projection flops of
# S3 (2 * C * sum_d P_d * H^2) and the contraction flops of S4, the target rows the
# walk reads (S10). W_q is counted once per round: it is the compulsory traffic of
# the per-depth projection (33.5 MB at H = 4096 stays in the 129 MB L2 between
# depths); the variant that re-reads it at every depth is reported beside it.
# What the implementation adds on top (the candidate rows copied for the G GEMM,
# the G or u bf16 pairs, the logits, the reassociated GEMM's extra flops) is
# reported separately as intermediate bytes and extra flops.

def parents(cfg):
    P = [1]
    for _ in range(cfg.L - 1):
        P.append(min(cfg.W, P[-1] * cfg.K))
    return P


def algorithmic(cfg, accepted_mean: float) -> dict:
    """Bytes and flops the method must touch once per round (roofline numerator)."""
    eb = 2 if cfg.dtype == "bf16" else 4
    C, L, V, H, K = cfg.C, cfg.L, cfg.V, cfg.H, cfg.K
    P = parents(cfg)
    topk_bytes = C * L * V * eb
    expand_bytes = (H * H * eb                # W_q once (compulsory)
                    + C * L * K * H * eb      # candidate embedding rows
                    + C * L * H * eb)         # block hidden rows
    rows_walked = (accepted_mean + 1) if cfg.rows == "node" else L
    verify_bytes = C * rows_walked * V * eb
    flops = 2 * C * H * H * sum(P) + 2 * C * K * H * sum(P)
    return dict(topk=topk_bytes, expand=expand_bytes, verify=verify_bytes, flops=flops,
                total=topk_bytes + expand_bytes + verify_bytes,
                total_wq_per_depth=topk_bytes + expand_bytes + (L - 1) * H * H * eb + verify_bytes)


# --------------------------------------------------------------------------- inputs

def device_inputs(cfg, torch):
    inp = make_inputs(cfg)

    def t(a):
        a = np.ascontiguousarray(a)
        if cfg.dtype == "bf16":
            return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
        return torch.from_numpy(a).cuda()

    x = dict(E=t(inp["E"]), Wq=t(inp["Wq"]), base=t(inp["base"]), hidden=t(inp["hidden"]),
             anchor=torch.from_numpy(inp["anchor"]).cuda())
    if cfg.rows == "position":
        x["target"] = t(inp["target"])
    else:
        x["target"] = t(make_target_per_node(cfg, inp, breadth_first_slot_depth(cfg)))
    return inp, x


# --------------------------------------------------------------------------- clocks

class Clocks:
    """nvidia-smi samples (every 200 ms) of the SM clock and throttle reasons while a
    measurement runs; the raw samples go to CLOCKS_CSV (--clocks-csv), by default a
    file in the temporary directory."""

    def __init__(self):
        self.p = None
        self.path = CLOCKS_CSV or os.path.join(tempfile.gettempdir(), f"dartree_bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.p = subprocess.Popen(
                ["nvidia-smi", "-i", os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0],
                 "--query-gpu=clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
                 "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                 "clocks_event_reasons.sw_power_cap", "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self) -> dict:
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        self.p.wait()
        self.f.close()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 7:
                    continue
                try:
                    sm.append(float(parts[0]))
                    mx = float(parts[1])
                except ValueError:
                    continue
                for n, v in zip(names, parts[3:7]):
                    if v.lower() == "active":
                        reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- GPU measurement

def time_steps(torch, fn, steps, warmup, flush):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        if flush is not None:
            flush.add_(1)
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record()
        fn()
        e.record()
        e.synchronize()
        times.append(s.elapsed_time(e))
    return np.array(times)  # ms


def graphed(torch, fn, use_graph=True):
    """fn captured in a CUDA graph (so host overhead does not show in device timings)."""
    fn()
    torch.cuda.synchronize()
    if not use_graph:
        return fn
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    graphed.keep.append(g)
    return g.replay


graphed.keep = []


def job_rate(ms_sum_local: float, steps: int, world: int, max_over_ranks=None):
    """Whole-job rounds/s of `world` ranks that each run their own replica of the
    workload (no exchange between them): the job's time for `steps` rounds is the
    slowest rank's. Returns (rounds/s over all ranks, ms per step)."""
    ms_sum = max_over_ranks(ms_sum_local) if max_over_ranks is not None else ms_sum_local
    ms = ms_sum / steps
    return world * 1e3 / ms, ms


def measure(cfg, steps, warmup, torch, dd, graphs=True, barrier=None):
    inp, x = device_inputs(cfg, torch)
    rows = dd.ROWS_PER_POSITION if cfg.rows == "position" else dd.ROWS_PER_NODE
    rnd = dd.Round(x["E"], x["Wq"], cfg.C, cfg.L, cfg.K, cfg.W, cfg.B, cfg.beta, rows)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")

    def step():
        rnd.run(x["base"], x["hidden"], x["anchor"], x["target"])

    step()
    torch.cuda.synchronize()
    if dd.read_status(rnd.ws) != 0:
        raise RuntimeError(f"device status {dd.read_status(rnd.ws)}")
    run = graphed(torch, step, graphs)
    clocks = Clocks()
    clocks.start()
    torch.cuda.synchronize()
    if barrier is not None:  # every rank starts (and ends) the timed steps together
        barrier()
    t_round = time_steps(torch, run, steps, warmup, flush)
    torch.cuda.synchronize()
    if barrier is not None:
        barrier()
    clk = clocks.stop()
    acc = rnd.out["accepted_len"].float().mean().item()

    # per-step breakdown through the individual entry points (same inputs, same stream)
    V = x["E"].shape[0]
    base2 = x["base"].view(cfg.C * cfg.L, V)
    t_topk = time_steps(torch, graphed(torch, lambda: dd.topk(base2, cfg.K, ws=rnd.ws), graphs), steps, warmup,
                        flush)
    t_verify = time_steps(torch, graphed(torch, lambda: dd.verify(rnd.tree, x["target"], rows, cfg.L, ws=rnd.ws),
                                         graphs), steps, warmup, flush)
    # per-kernel device time: the library brackets each launch with CUDA events on
    # its own stream while timing is on (same rounds, not graph-captured)
    n_prof = max(5, min(steps, 20))
    dd.timing(True)
    for _ in range(n_prof):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize()
    kt = dd.kernel_times()
    dd.timing(False)
    return dict(inp=inp, x=x, rnd=rnd, t_round=t_round, t_topk=t_topk, t_verify=t_verify, clocks=clk,
                accepted_mean=acc, rows=rows, kernel_times=kt, n_prof=n_prof)


E2E_STEPS = 200  # host-buffer rounds timed back to back (~25 ms at cfg1)


def measure_e2e(cfg, m, steps, torch, dd):
    """The same round through the C ABI's host session (dartree_host_stage /
    dartree_host_round, via dd.HostRounds): every step copies its inputs from pinned
    host memory and reads its result back into pinned host memory, all inside the
    timed region; step i + 1's inputs are copied on the session's copy stream while
    step i runs (two device input sets)."""
    x, rnd = m["x"], m["rnd"]
    h = {k: x[k].cpu().pin_memory() for k in dd.HostRounds.KEYS}
    outs = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in rnd.out.items()}
    hr = dd.HostRounds(rnd, h)
    h2d = hr.h2d_bytes()
    d2h = sum(v.numel() * v.element_size() for v in outs.values())

    def run_steps(n):
        hr.copy_in(0, h)
        for i in range(n):
            if i + 1 < n:
                hr.copy_in(i + 1, h)
            hr.run(i, outs)

    run_steps(3)
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record()  # (recorded on an idle device, before the first copy is enqueued)
    run_steps(steps)
    e.record()
    e.synchronize()
    ms = s.elapsed_time(e) / steps
    return ms, h2d, d2h


def measure_heap(cfg, m, steps, warmup, torch, dd, graphs=True):
    """The node-by-node heap -> correction baseline (one head evaluation per popped
    node, the same S1 and G projection) on the same inputs: us per build, and the
    ratio to the deferred round's p50 (build + verify)."""
    x = m["x"]
    h = dd.HeapRound(x["E"], x["Wq"], cfg.C, cfg.L, cfg.K, cfg.B, cfg.beta)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
    t = time_steps(torch, graphed(torch, lambda: h.run(x["base"], x["hidden"], x["anchor"]), graphs), steps, warmup,
                   flush)
    us = float(np.median(t)) * 1e3
    return {"heap_baseline_us": round(us, 2), "deferred_round_us": round(float(np.median(m["t_round"])) * 1e3, 2),
            "heap_over_deferred": round(us / (float(np.median(m["t_round"])) * 1e3), 3)}


def measure_sample(cfg, m, steps, warmup, torch, dd, hbm_peak, graphs=True, temperature=1.0, seed=2026):
    """Verification at temperature T (dartree_verify_sample) on the round's tree and
    target rows, beside greedy verification on the same inputs: us per call and the
    target bytes the draw reads (per-position rows: all C*L rows; per-node rows: the
    rows on the walked paths)."""
    x, rnd, rows = m["x"], m["rnd"], m["rows"]
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
    fn = lambda: dd.verify_sample(rnd.tree, x["target"], rows, cfg.L, temperature, seed, ws=rnd.ws)  # noqa: E731
    out = fn()
    torch.cuda.synchronize()
    walked = float(out["accepted_len"].float().mean().item()) + 1.0
    t = time_steps(torch, graphed(torch, fn, graphs), steps, warmup, flush)
    us = float(np.median(t)) * 1e3
    eb = 2 if cfg.dtype == "bf16" else 4
    nbytes = cfg.C * (cfg.L if cfg.rows == "position" else walked) * cfg.V * eb
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"us": round(us, 2), "greedy_verify_us": round(float(np.median(m["t_verify"])) * 1e3, 2),
            "temperature": temperature, "rows": cfg.rows, "accepted_mean": round(walked - 1.0, 3),
            "target_bytes": int(nbytes), "achieved_gbs": round(gbs, 1), "hbm_frac": round(gbs / hbm_peak, 4)}


def measure_lm_head(cfg, m, steps, warmup, torch, dd, hbm_peak, graphs=True):
    """The drafter's LM head fused with S1 (dartree_lm_head_topk) on the round's block
    hidden states and a stand-in W_lm [V, H]: us per call and the fraction of the
    measured copy bandwidth its bytes (W_lm once, the hidden rows) reach. Beside it,
    for context only, the unfused library path (torch matmul writing the logits,
    then torch.topk) on the same operands."""
    if cfg.dtype != "bf16":
        return None
    x = m["x"]
    R = cfg.C * cfg.L
    h = x["hidden"].view(R, cfg.H)
    W = torch.from_numpy(make_lm_head(cfg).view(np.int16)).cuda().view(torch.bfloat16)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
    ws = dd.new_workspace(dd.lib().dartree_lm_head_workspace_bytes(R, cfg.V, cfg.H, cfg.K))
    t = time_steps(torch, graphed(torch, lambda: dd.lm_head_topk(h, W, cfg.K, ws=ws), graphs), steps, warmup, flush)
    us = float(np.median(t)) * 1e3
    nbytes = cfg.V * cfg.H * 2 + R * cfg.H * 2
    t_lib = time_steps(torch, graphed(torch, lambda: torch.topk((h @ W.t()).float(), cfg.K, dim=1), graphs), steps,
                       warmup, flush)
    del W
    return {"us": round(us, 2), "rows": R, "V": cfg.V, "H": cfg.H, "K": cfg.K, "bytes": int(nbytes),
            "achieved_gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
            "hbm_frac": round(nbytes / (us * 1e-6) / 1e9 / hbm_peak, 4),
            "unfused_torch_us": round(float(np.median(t_lib)) * 1e3, 2)}


ATTN_SHAPE = dict(Hq=32, Hkv=8, D=128, N=2048, theta=1.0e6)   # a Qwen3-4B/8B attention layer, 2048 cached


def measure_attention(cfg, m, steps, warmup, torch, dd, hbm_peak, tf_peak, graphs=True):
    """One tree-attention layer of the verification pass (dartree_tree_attention) on the
    round's tree (S9's mask and positions) over a full 2048-token cache per request:
    us per call, the cache bytes it streams against the measured copy bandwidth, and
    its score + value flops (over every cached key and the tree) against bf16 peak."""
    tr = m["rnd"].tree
    C, S = tr["mask"].shape[0], tr["mask"].shape[1]
    Hq, Hkv, D, N = ATTN_SHAPE["Hq"], ATTN_SHAPE["Hkv"], ATTN_SHAPE["D"], ATTN_SHAPE["N"]
    gen = torch.Generator(device="cuda")
    gen.manual_seed(2026)
    r = lambda *shape: torch.randn(*shape, generator=gen, device="cuda").to(torch.bfloat16)  # noqa: E731
    q, kt, vt = r(C, S, Hq, D), r(C, S, Hkv, D), r(C, S, Hkv, D)
    kc, vtc = r(C, Hkv, N, D), r(C, Hkv, D, N)
    n_ctx = torch.full((C,), N, dtype=torch.int32, device="cuda")
    p = dd.AttnParams(C, S, Hq, Hkv, D, N, ATTN_SHAPE["theta"])
    import ctypes
    ws = dd.new_workspace(dd.lib().dartree_tree_attention_workspace_bytes(ctypes.byref(p)))
    fn = lambda: dd.tree_attention(q, kt, vt, kc, vtc, n_ctx, tr, ATTN_SHAPE["theta"], ws=ws)  # noqa: E731
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
    t = time_steps(torch, graphed(torch, fn, graphs), steps, warmup, flush)
    us = float(np.median(t)) * 1e3
    nbytes = C * Hkv * N * D * 2 * 2 + C * S * (Hq + 2 * Hkv) * D * 2 + C * S * Hq * D * 2
    flops = 2 * 2 * C * Hq * S * (N + S) * D
    del q, kt, vt, kc, vtc
    return {"us": round(us, 2), "C": C, "S": S, "Hq": Hq, "Hkv": Hkv, "D": D, "n_ctx": N, "bytes": int(nbytes),
            "achieved_gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
            "hbm_frac": round(nbytes / (us * 1e-6) / 1e9 / hbm_peak, 4),
            "tflops": round(flops / (us * 1e-6) / 1e12, 1),
            "tensor_frac": round(flops / (us * 1e-6) / 1e12 / tf_peak, 4)}


# DRAM bytes per launch (read + write) from one ncu capture of the current kernel on
# this workload; the C=64 contraction was captured on 8 requests and scaled by the
# requests processed (its traffic is per request).
# A kernel changed since its capture has no entry (traffic null).
NCU_TRAFFIC = {
    ("cfg1_qwen3_4b_c1", "expand_g_kernel"): 15566592,      # one launch = one round, full size
    ("cfg1_qwen3_4b_c1", "gemm_bf16_tc_kernel"): 23247360,
    ("cfg1_qwen3_4b_c1", "topk_rows_kernel"): 28392192,     # incl. the 13.1 MB L2 prefetch of W_q^T
    ("cfg4_c64_stress", "contract_tc_kernel"): 35337472 * 8,   # one launch over all 64 requests
    ("cfg4_c64_stress", "topk_stream_kernel"): 361796608 + 5478400,   # full size
}


def kernel_work(cfg, name, accepted_mean, g_path, fused_gather=False):
    """Work of a kernel family over ONE round: (bound, method work, intermediate
    bytes, extra flops). The method work is bytes ("hbm") or flops ("tensor") of the
    method's own steps that the family performs; the intermediates are what the
    implementation writes and reads back in between; extra flops are the flops the
    implementation does beyond the method's (the candidate-side G GEMM).
    fused_gather: the cluster top-K also copied the candidates' rows of E."""
    eb = 2 if cfg.dtype == "bf16" else 4
    C, L, V, H, K, W, B = cfg.C, cfg.L, cfg.V, cfg.H, cfg.K, cfg.W, cfg.B
    P = parents(cfg)
    proj_flops = 2 * C * sum(P) * H * H
    logits = sum(C * p * K * 4 for p in P)
    rows_walked = (accepted_mean + 1) if cfg.rows == "node" else L
    if name in ("topk_rows_kernel", "topk_stream_kernel"):
        copy = 2 * C * L * K * H * 2 if (fused_gather and name == "topk_rows_kernel") else 0
        return "hbm", C * L * V * eb, copy, 0
    if name == "gather_rows_kernel":
        return "hbm", 0, 2 * C * L * K * H * eb, 0
    if name == "rowmax_kernel":
        return "hbm", C * L * V * eb, 0, 0
    if name == "gemm_bf16_tc_kernel":
        if g_path:  # G = E[cand] W_q for all C*L*K candidates; S3's flops are the method's part
            g_flops = 2 * C * L * K * H * H
            return "tensor", proj_flops, C * L * K * H * 2 + 2 * C * L * K * H * 2, g_flops - proj_flops
        return "tensor", proj_flops, sum(2 * C * p * H * 2 for p in P), 0
    if name == "expand_g_kernel":  # S2, S4-S7 (and S8-S10 after the last depth) over G
        return "hbm", C * L * K * H * eb + C * L * H * eb, 2 * C * L * K * H * 2 + logits, 0
    if name == "contract_tc_kernel":  # S4: every depth's candidate rows against the u pair
        return "hbm", L * C * K * H * eb, L * C * 32 * H * 2 + logits, 0
    if name == "select_kernel":
        return "hbm", 0, logits, 0
    if name == "state_kernel":  # S7: the kept children's rows of E and H_d
        return "hbm", (L - 1) * C * (W + 1) * H * eb, (L - 1) * 2 * C * W * H * eb, 0
    if name == "walk_kernel":
        return "hbm", C * rows_walked * V * eb, 0, 0
    if name == "finish_kernel":
        return "hbm", 0, C * (L * W * 16 + (B + 1) * (B + 1) + (B + 1) * 20), 0
    return "hbm", 0, 0, 0


# Batches of at least this many requests expand as two halves on two streams.
SPLIT_MIN_C = 32


def kernel_roofline(cfg, m, hbm_peak, tf_peak):
    """Roofline of the kernel family with the largest device time per round:
    the method's work of one launch (the round's work / launches per round) over
    the average launch time. When the batch expands as two halves on two streams
    ("concurrent_halves": 2), a launch covers half of the requests and shares the
    GPU with its sibling, so its own rate understates the pair's."""
    kt, n = m["kernel_times"], m["n_prof"]
    g_path = "expand_g_kernel" in kt
    dom = max(kt, key=lambda k: kt[k][1])
    launches, ms_total = kt[dom]
    lpr = launches / n
    ms_launch = ms_total / launches
    fused = g_path and "gather_rows_kernel" not in kt
    bound, work_round, inter_round, extra_round = kernel_work(cfg, dom, m["accepted_mean"], g_path, fused)
    work, inter, extra = work_round / lpr, inter_round / lpr, extra_round / lpr
    traffic = NCU_TRAFFIC.get((cfg.name, dom))
    split = (not g_path) and cfg.C >= SPLIT_MIN_C and dom in ("contract_tc_kernel", "gemm_bf16_tc_kernel",
                                                               "select_kernel", "state_kernel")
    if split and traffic is not None:
        traffic //= 2  # the capture processed whole-batch launches; a launch here is half of them
    if bound == "tensor":
        achieved = work / (ms_launch * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": tf_peak, "unit": "TFLOP/s",
                "frac": round(achieved / tf_peak, 4), "traffic": traffic, "flops_per_launch": int(work)}
    else:
        achieved = work / (ms_launch * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(achieved / hbm_peak, 4), "traffic": traffic, "bytes_per_launch": int(work)}
    roof.update({"intermediate_bytes_per_launch": int(inter), "extra_flops_per_launch": int(extra),
                 "kernel": dom, "ms_per_launch": round(ms_launch, 5), "launches_per_round": lpr,
                 "share_of_kernel_time": round(ms_total / sum(v[1] for v in kt.values()), 4)})
    if split:
        roof["concurrent_halves"] = 2
    per_kernel = {k: {"launches_per_round": round(v[0] / n, 2), "ms_per_round": round(v[1] / n, 4)}
                  for k, v in sorted(kt.items(), key=lambda kv: -kv[1][1])}
    launches_per_round = sum(v[0] for v in kt.values()) / n
    return roof, per_kernel, launches_per_round


def roofline(cfg, m, hbm_peak):
    alg = algorithmic(cfg, m["accepted_mean"])
    parts = {"topk": (alg["topk"], float(np.median(m["t_topk"]))),
             "verify": (alg["verify"], float(np.median(m["t_verify"])))}
    t_round = float(np.median(m["t_round"]))
    rest = max(t_round - parts["topk"][1] - parts["verify"][1], 1e-6)
    parts["expand+prune+mask"] = (alg["expand"], rest)
    dom = max(parts, key=lambda k: parts[k][1])
    b, ms = parts[dom]
    achieved = b / (ms * 1e-3) / 1e9
    return dom, {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm_peak, "unit": "GB/s",
                 "frac": round(achieved / hbm_peak, 4), "traffic": None, "kernel": dom,
                 "bytes_per_launch": int(b), "ms_per_launch": round(ms, 4)}, alg, parts


# --------------------------------------------------------------------------- CPU oracle leg

def cpu_model() -> str:
    """The host CPU's name from /proc/cpuinfo (x86 'model name', else the Arm part
    numbers), or the platform's machine name."""
    import platform
    try:
        info = open("/proc/cpuinfo").read().splitlines()
    except OSError:
        info = []
    for key in ("model name", "Model name"):
        for line in info:
            if line.startswith(key):
                return line.split(":", 1)[1].strip()
    parts = {}
    for line in info:
        if ":" in line:
            k, v = (x.strip() for x in line.split(":", 1))
            if k in ("CPU implementer", "CPU part") and k not in parts:
                parts[k] = v
    if parts:
        return f"{platform.machine()} implementer {parts.get('CPU implementer', '?')} part {parts.get('CPU part', '?')}"
    return platform.machine()


def _oracle_rate(cfg, budget_s):
    """(rounds, seconds) of full oracle rounds (build + verify) within budget_s."""
    import oracle
    inp = make_inputs(cfg)
    t0 = time.time()
    n = 0
    while True:
        o = oracle.build(inp)
        if cfg.rows == "position":
            oracle.verify(o, inp["target"], cfg.dtype, cfg.rows, cfg.L)
        n += 1
        if time.time() - t0 > budget_s:
            break
    return n, time.time() - t0


def _oracle_rate_one_thread(cfg_name, budget_s):
    """The same in a child process whose BLAS and OpenMP pools have one thread."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1")
    code = ("import sys, json; sys.path.insert(0, %r); import bench; from dartree_inputs import make_config; "
            "n, dt = bench._oracle_rate(make_config(%r), %r); print(json.dumps([n, dt]))" % (ROOT, cfg_name, budget_s))
    try:
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                           timeout=budget_s * 10 + 120)
        n, dt = json.loads(r.stdout.strip().splitlines()[-1])
        return n, dt
    except Exception:
        return None


def cpu_baseline(cfg, budget_s=10.0, one_thread_s=5.0):
    n, dt = _oracle_rate(cfg, budget_s)
    out = {"value": round(n / dt, 4), "unit": "rounds/s", "cores": len(os.sched_getaffinity(0)),
           "kind": "oracle", "cpu": cpu_model(),
           "sample": f"{n} full oracle round(s) of {cfg.name} (build+verify, float64 numpy), {dt:.1f} s"}
    one = _oracle_rate_one_thread(cfg.name, one_thread_s)
    if one:
        out["value_one_thread"] = round(one[0] / one[1], 4)
        out["sample_one_thread"] = f"{one[0]} round(s) in {one[1]:.1f} s with one BLAS/OpenMP thread"
    return out


def cpu_baseline_stress(cfg, budget_requests=1):
    """Oracle on a bounded sample of the C=64 batch (one request), scaled to rounds/s."""
    import oracle
    inp = make_inputs(cfg, requests=list(range(budget_requests)))
    t0 = time.time()
    oracle.build(inp)
    dt = time.time() - t0
    per_round = dt * cfg.C / budget_requests
    return {"value": round(1.0 / per_round, 6), "unit": "rounds/s", "cores": len(os.sched_getaffinity(0)),
            "kind": "oracle",
            "sample": f"oracle build of {budget_requests} of {cfg.C} requests ({dt:.1f} s), scaled to the batch"}


def workload_config(cfg, graphs: bool, world: int) -> dict:
    """The `config` object of the JSON line, the same for both arms."""
    return {"workload": cfg.name, "C": cfg.C, "L": cfg.L, "V": cfg.V, "H": cfg.H, "K": cfg.K, "W": cfg.W,
            "B": cfg.B, "beta": cfg.beta, "l2": "flushed between timed steps (2x L2 write)",
            "cuda_graph": graphs, "parallelism": "replicas" if world > 1 else "single"}


# --------------------------------------------------------------------------- profiling mode

def profile_only(args):
    """Runs one entry point on one workload (for ncu); prints its device time."""
    import torch
    import diffusion_drafter_draft_gb300 as dd
    from diffusion_drafter_draft_gb300 import _build
    _build.build()
    cfg = make_config(args.config or MAIN_CFG)
    if args.C:
        cfg = cfg.replace(C=args.C)
    inp, x = device_inputs(cfg, torch)
    rows = dd.ROWS_PER_POSITION if cfg.rows == "position" else dd.ROWS_PER_NODE
    V = x["E"].shape[0]
    if args.only == "topk":
        ws = dd.new_workspace(256)
        base2 = x["base"].view(cfg.C * cfg.L, V)
        fn = lambda: dd.topk(base2, cfg.K, ws=ws)  # noqa: E731
    elif args.only == "lmhead":
        R = cfg.C * cfg.L
        W = torch.from_numpy(make_lm_head(cfg).view(np.int16)).cuda().view(torch.bfloat16)
        h = x["hidden"].view(R, cfg.H)
        ws = dd.new_workspace(dd.lib().dartree_lm_head_workspace_bytes(R, cfg.V, cfg.H, cfg.K))
        fn = lambda: dd.lm_head_topk(h, W, cfg.K, ws=ws)  # noqa: E731
    elif args.only == "attn":
        import ctypes
        rnd0 = dd.Round(x["E"], x["Wq"], cfg.C, cfg.L, cfg.K, cfg.W, cfg.B, cfg.beta, rows)
        rnd0.run(x["base"], x["hidden"], x["anchor"], x["target"])
        tr = rnd0.tree
        C, S = cfg.C, cfg.B + 1
        Hq, Hkv, D, N = ATTN_SHAPE["Hq"], ATTN_SHAPE["Hkv"], ATTN_SHAPE["D"], ATTN_SHAPE["N"]
        r_ = lambda *shape: torch.randn(*shape, device="cuda").to(torch.bfloat16)  # noqa: E731
        aq, akt, avt, akc, avc = r_(C, S, Hq, D), r_(C, S, Hkv, D), r_(C, S, Hkv, D), r_(C, Hkv, N, D), r_(C, Hkv, D, N)
        n_ctx = torch.full((C,), N, dtype=torch.int32, device="cuda")
        ap = dd.AttnParams(C, S, Hq, Hkv, D, N, ATTN_SHAPE["theta"])
        aws = dd.new_workspace(dd.lib().dartree_tree_attention_workspace_bytes(ctypes.byref(ap)))
        fn = lambda: dd.tree_attention(aq, akt, avt, akc, avc, n_ctx, tr, ATTN_SHAPE["theta"], ws=aws)  # noqa: E731
    elif args.only == "heap":
        h = dd.HeapRound(x["E"], x["Wq"], cfg.C, cfg.L, cfg.K, cfg.B, cfg.beta)
        fn = lambda: h.run(x["base"], x["hidden"], x["anchor"])  # noqa: E731
    else:
        rnd = dd.Round(x["E"], x["Wq"], cfg.C, cfg.L, cfg.K, cfg.W, cfg.B, cfg.beta, rows)
        fn = lambda: rnd.run(x["base"], x["hidden"], x["anchor"], x["target"])  # noqa: E731
    t = time_steps(torch, fn, args.steps, max(3, args.warmup), None)
    print(json.dumps({"only": args.only, "workload": cfg.name, "ms_median": float(np.median(t)),
                      "ms_min": float(np.min(t))}))


# --------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-stress", action="store_true")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--only", choices=["topk", "round", "heap", "lmhead", "attn"], default=None,
                    help="profiling mode: run just one entry point on --config and print its timing")
    ap.add_argument("--config", default=None, help="workload name for --only (default: the main workload)")
    ap.add_argument("--C", type=int, default=None, help="--only: override the number of requests (a smaller case)")
    ap.add_argument("--clocks-csv", default=None, help="file for the raw nvidia-smi clock samples of the timed region")
    args = ap.parse_args()
    global CLOCKS_CSV
    CLOCKS_CSV = args.clocks_csv
    if args.only:
        return profile_only(args)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    cfg = make_config(MAIN_CFG)

    if args.impl == "reference":
        if rank != 0:
            return
        vals = []
        t0 = time.time()
        import oracle
        inp = make_inputs(cfg)
        for _ in range(args.warmup):  # untimed
            oracle.verify(oracle.build(inp), inp["target"], cfg.dtype, cfg.rows, cfg.L)
        for _ in range(args.steps):
            s = time.time()
            o = oracle.build(inp)
            oracle.verify(o, inp["target"], cfg.dtype, cfg.rows, cfg.L)
            vals.append(time.time() - s)
        ms = float(np.mean(vals)) * 1e3
        v = 1e3 / ms
        print(json.dumps({
            "impl": "reference", "metric": "draft-tree rounds/sec (build+verify)", "value": round(v, 4),
            "unit": "rounds/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": workload_config(cfg, not args.no_graph, world),
            "cpu_baseline": {"value": round(v, 4), "unit": "rounds/s", "cores": len(os.sched_getaffinity(0)),
                             "kind": "oracle", "cpu": cpu_model(),
                             "sample": f"{args.steps} full rounds of {cfg.name}"},
            "e2e": {"value": round(v, 4), "unit": "rounds/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": round(time.time() - t0, 1)}))
        return

    import torch
    import diffusion_drafter_draft_gb300 as dd
    from diffusion_drafter_draft_gb300 import _build
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    _build.build()
    dd.lib()
    hbm_peak, tf_peak, peak_kind = _peaks()

    barrier = max_over_ranks = None
    if world > 1:
        import torch.distributed as dist

        def max_over_ranks(v):
            tt = torch.tensor([v], device="cuda")
            dist.all_reduce(tt, op=dist.ReduceOp.MAX)
            return float(tt.item())

        barrier = dist.barrier
    m = measure(cfg, args.steps, max(3, args.warmup), torch, dd, graphs=not args.no_graph, barrier=barrier)
    value, ms = job_rate(float(np.sum(m["t_round"])), args.steps, world, max_over_ranks)
    dom, _, alg, parts = roofline(cfg, m, hbm_peak)
    roof, per_kernel, lpr = kernel_roofline(cfg, m, hbm_peak, tf_peak)
    e2e_ms, h2d, d2h = measure_e2e(cfg, m, E2E_STEPS, torch, dd)
    heap = measure_heap(cfg, m, args.steps, max(3, args.warmup), torch, dd, graphs=not args.no_graph)
    sample = measure_sample(cfg, m, args.steps, max(3, args.warmup), torch, dd, hbm_peak, graphs=not args.no_graph)
    lmh = measure_lm_head(cfg, m, args.steps, max(3, args.warmup), torch, dd, hbm_peak, graphs=not args.no_graph)
    attn = measure_attention(cfg, m, args.steps, max(3, args.warmup), torch, dd, hbm_peak, tf_peak,
                             graphs=not args.no_graph)
    line = {
        "metric": "draft-tree rounds/sec (build+verify)", "value": round(value, 3), "unit": "rounds/s",
        "n_gpus": world, "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": round(ms, 5),
        "us_per_round_p50": round(float(np.median(m["t_round"])) * 1e3, 2),
        "us_per_round_p90": round(float(np.percentile(m["t_round"], 90)) * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": cfg.dtype,
        "data": "synthetic",
        "config": workload_config(cfg, not args.no_graph, world),
        "roofline": dict(roof, peak_kind=peak_kind),
        "round_hbm_frac": round(alg["total"] / (float(np.median(m["t_round"])) * 1e-3) / 1e9 / hbm_peak, 4),
        "round_tensor_frac": round(alg["flops"] / (float(np.median(m["t_round"])) * 1e-3) / 1e12 / tf_peak, 4),
        "breakdown_ms": {k: round(v[1], 4) for k, v in parts.items()},
        "kernels": per_kernel,
        "accepted_mean": m["accepted_mean"],
        "gpu_launches": int(round(lpr * args.steps)),
        "e2e": {"value": round(1e3 / e2e_ms, 3), "unit": "rounds/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h)},
        "clocks": m["clocks"],
        "heap_baseline": heap,
        "verify_sample": sample,
        "lm_head_topk": lmh,
        "tree_attention": attn,
    }
    del m
    torch.cuda.empty_cache()
    if not args.no_stress:
        scfg = make_config(STRESS_CFG)
        sm = measure(scfg, max(5, min(args.steps, 20)), 3, torch, dd, graphs=not args.no_graph)
        sdom, _, salg, sparts = roofline(scfg, sm, hbm_peak)
        sroof, sper_kernel, _ = kernel_roofline(scfg, sm, hbm_peak, tf_peak)
        sms = float(np.median(sm["t_round"]))
        line["c64"] = {"workload": scfg.name, "value": round(1e3 / sms, 3), "unit": "rounds/s",
                       "request_rounds_per_s": round(scfg.C * 1e3 / sms, 1), "us_per_round_p50": round(sms * 1e3, 1),
                       "roofline": dict(sroof, peak_kind=peak_kind),
                       "round_hbm_frac": round(salg["total"] / (sms * 1e-3) / 1e9 / hbm_peak, 4),
                       "round_hbm_frac_wq_per_depth": round(salg["total_wq_per_depth"] / (sms * 1e-3) / 1e9
                                                            / hbm_peak, 4),
                       "round_tensor_frac": round(salg["flops"] / (sms * 1e-3) / 1e12 / tf_peak, 4),
                       "breakdown_ms": {k: round(v[1], 4) for k, v in sparts.items()},
                       "kernels": sper_kernel,
                       "accepted_mean": sm["accepted_mean"], "clocks": sm["clocks"],
                       "verify_sample": measure_sample(scfg, sm, max(5, min(args.steps, 20)), 3, torch, dd,
                                                       hbm_peak, graphs=not args.no_graph),
                       "tree_attention": measure_attention(scfg, sm, max(5, min(args.steps, 20)), 3, torch, dd,
                                                           hbm_peak, tf_peak, graphs=not args.no_graph)}
        del sm
        torch.cuda.empty_cache()
    if rank == 0:
        line["cpu_baseline"] = cpu_baseline(cfg)
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
