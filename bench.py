"""Benchmark of one CSA / HCA attention-layer forward on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Default workload: CSA decode at V4-Pro shape, 128K context, batch 4 (one new
query token per sequence: index -> top-k -> attend over a given compressed
cache).  A step is one pass of every stage of the workload over one batch of
seeded synthetic inputs already resident in HBM.  Steps are CUDA-graph
replays; consecutive steps cycle through enough copies of the inputs that the
working set exceeds twice the L2, so no step reads another step's data from L2.

Prints one JSON line (rank 0).  With torchrun (N > 1) every rank runs an
independent replica of the workload ("replicas only": the path has no
exchange step) and the slowest rank's time counts.

--impl reference times the float64 CPU oracle (the only reference this method
has) on a bounded sample of the same workload on the host cores.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "CSA tokens/s (decode @128K ctx, prefill @32K) and % of HBM/tensor roofline"
DEFAULT_WORKLOAD = "csa_decode_128k"
L2_BYTES = 126 * 1024 * 1024


def kernel_source_sha():
    """First 12 hex digits of the sha256 over the kernel sources (csrc/*.cu, *.cuh),
    leaving out the lines that hold phase-trace marks (they compile to nothing
    outside the -DCSA_TRACE build, so they do not change the measured kernels)."""
    import glob
    import hashlib
    h = hashlib.sha256()
    for f in sorted(glob.glob(os.path.join(ROOT, "compressed_sparse_long_05_b300", "csrc", "*.cu*"))):
        for line in open(f, "rb"):
            if b"CSA_TRACE_MARK(" in line or b"CSA_TRACE_WALL(" in line:
                continue
            h.update(line)
    return h.hexdigest()[:12]


def profiled_traffic(cfg, stage):
    """DRAM bytes (read + write) per launch of `stage` from the committed ncu summaries.

    Lines in profiles/*.md of the form
        traffic <workload>[@T=<tokens>] <stage> <bytes> src=<sha>
    hold the counters of one capture.  They count only while the kernel sources
    still hash to <sha>; a capture of a shrunk prefill case (@T=...) is scaled
    to this workload's T (q, out and the streamed inputs grow in proportion).
    Returns (bytes or None, note).
    """
    import glob
    sha = kernel_source_sha()
    for f in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        for line in open(f):
            p = line.split()
            if len(p) != 5 or p[0] != "traffic" or p[2] != stage or not p[4].startswith("src="):
                continue
            wl, _, at = p[1].partition("@")
            if wl != cfg["name"].split("_T")[0] and wl != cfg["name"]:
                continue
            if p[4][4:] != sha:
                return None, f"{os.path.basename(f)}: kernel sources changed since the capture"
            nbytes = float(p[3])
            if at:
                k, v = at.split("=")
                nbytes *= cfg[k] / int(v)
                return int(nbytes), f"{os.path.basename(f)} (captured at {at}, scaled by {k})"
            return int(nbytes), os.path.basename(f)
    return None, "no capture of this kernel and workload"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained", d["bf16_tflops"]), "measured"
    return 6400.0, 1800.0, 1400.0, "fallback"


# ----------------------------------------------------------------------------
# algorithmic work per stage (bytes that must move, flops that must be done)
# ----------------------------------------------------------------------------


def _vis(t, m, N):
    return min(N, (t + 1) // m)


def row_bytes(cfg):
    d, r = cfg["d"], cfg["r"]
    return (d - r) + 4 + 2 * r if cfg["dtype"] == "mixed" else d * (4 if cfg["dtype"] == "f32" else 2)


def work(cfg):
    """{stage: (bytes, flops)} for one step of the workload (summed over its
    sequences, each at its own query positions)."""
    out = {}
    for L_b, pos in zip(cfg["lengths"], synth.configs.query_positions(cfg)):
        one = dict(cfg, B=1, lengths=[L_b])
        for st, (b, f) in _work_one(one, np.asarray(pos, dtype=np.int64)).items():
            b0, f0 = out.get(st, (0, 0.0))
            out[st] = (b0 + b, f0 + f)
    return out


def _work_one(cfg, t):
    B, Tq, N, m, d = 1, cfg["Tq"], cfg["N"], cfg["m"], cfg["d"]
    n_h, n_win = cfg["n_h"], cfg["n_win"]
    el = 4 if cfg["dtype"] == "f32" else 2
    rb = row_bytes(cfg)
    vis = np.minimum(N, (t + 1) // m)
    win = np.minimum(n_win, t + 1)
    out = {}
    kind = cfg["kind"]
    if kind.endswith("prefill"):
        T = cfg["T"]
        nt = 4 if kind == "csa_prefill" else 2
        cb = nt * T * d * el + N * d * el
        if cfg.get("index_keys") == "compressed":          # K^IComp from raw index rows
            cb += 4 * T * cfg["c_I"] * el + N * cfg["c_I"] * el
        out["compress"] = (B * cb, 0.0)
    if kind.startswith("csa"):
        H, c, k = cfg["H_I"], cfg["c_I"], cfg["k"]
        kb = (c // 2 + c // 16) if cfg["dtype"] == "mixed" else c * el
        pairs = int(vis.sum())
        out["index"] = (B * (N * kb + Tq * H * kb + Tq * H * 4 + Tq * N * 4), 2.0 * B * pairs * H * c)
        out["topk"] = (B * (pairs * 4 + Tq * k * 4), 0.0)
        if Tq == 1:
            ib, ifl = out.pop("index")
            tb, _ = out.pop("topk")
            out["index_topk"] = (ib + tb, ifl)
        rows = np.minimum(k, vis) + win
        out["attend"] = (B * (int(rows.sum()) * rb + int(np.minimum(k, vis).sum()) * 4 +
                              2 * Tq * n_h * d * el), 4.0 * B * int(rows.sum()) * n_h * d)
    else:
        rows = vis + win
        if kind == "hca_decode":
            gathered = B * int(rows.max()) * rb        # every query row of a sequence shares the rows
        else:
            gathered = B * (N + cfg["T_win"]) * rb
        out["attend"] = (gathered + 2 * B * Tq * n_h * d * el, 4.0 * B * int(rows.sum()) * n_h * d)
    return out


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------


class ClockSampler:
    """Samples SM clocks and clock-event (throttle) reasons while the timed region runs.

    Uses `nvidia-smi --query-gpu ... -lms` on this process's GPU (by UUID);
    falls back to NVML when nvidia-smi is missing.
    """

    QUERY = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev):
        self.dev = dev
        self.proc = None
        self.err = None
        try:
            u = str(torch.cuda.get_device_properties(dev).uuid)
            self.gpu_id = u if u.startswith("GPU-") else "GPU-" + u
        except Exception as e:  # pragma: no cover
            self.gpu_id, self.err = str(dev.index), repr(e)

    def __enter__(self):
        import subprocess
        import tempfile
        self.out = tempfile.TemporaryFile(mode="w+")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.out,
                stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception as e:
            self.err = repr(e)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            self.out.seek(0)
            for line in self.out:
                f = [x.strip() for x in line.split(",")]
                if len(f) < 8:
                    continue
                try:
                    sm.append(float(f[0]))
                    mx = float(f[1])
                except ValueError:
                    continue
                for nm, val in zip(names, f[4:8]):
                    if val.lower() == "active":
                        reasons.add(nm)
        except Exception as e:
            self.err = repr(e)
        res = {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
               "reasons": sorted(reasons), "samples": len(sm), "source": "nvidia-smi -lms 50"}
        if self.err:
            res["error"] = self.err
        return res


def max_over_ranks(value, device):
    """The largest of every rank's value (all ranks get it): the slowest rank's time counts."""
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def make_step(K, cfg, x, buf):
    """Stage callables of one step on inputs x (device tensors) with buffers buf."""
    from compressed_sparse_long_05_b300 import path as P
    m, r, n_win = cfg["m"], cfg["r"], cfg["n_win"]
    q0, wb, base = x["q_pos"], x["win_base"], cfg["rope_base"]
    kind = cfg["kind"]
    rot = bool(cfg.get("entry_rope"))
    stages = []
    if kind.endswith("prefill"):
        stages.append(("compress", lambda: P.compress_stage(cfg, x, buf)))
    ent = buf.entries if kind.endswith("prefill") else P._entries_arg(x)
    win = P._win_arg(x)
    if kind.startswith("csa") and cfg["Tq"] == 1:
        # decode: one call scores every entry and selects the top k (the index
        # kernel also builds the selector's first histogram)
        qI, qI_sf, Kt, K_sf = P._indexer_args(x, buf)
        stages.append(("index_topk", lambda: K.csa_index_topk(
            qI, x["w"], Kt, cfg["k"], m, q0, qI_sf=qI_sf, K_sf=K_sf, scores=buf.scores,
            idx=buf.idx, ws=buf.ws_topk)))
    elif kind.startswith("csa"):
        qI, qI_sf, Kt, K_sf = P._indexer_args(x, buf)
        stages.append(("index", lambda: K.csa_index(qI, x["w"], Kt, m, q0, qI_sf=qI_sf, K_sf=K_sf,
                                                    scores=buf.scores)))
        stages.append(("topk", lambda: K.csa_topk(buf.scores, cfg["k"], m, q0, idx=buf.idx)))
    if kind.startswith("csa"):
        stages.append(("attend", lambda: K.csa_attend(x["q"], ent, buf.idx, win, x["sink"], m, n_win,
                                                      wb, q0, r, base, out=buf.out, ws=buf.ws,
                                                      entries_rotated=rot)))
    else:
        stages.append(("attend", lambda: K.hca_attend(x["q"], ent, win, x["sink"], m, n_win, wb, q0,
                                                      r, base, out=buf.out, ws=buf.ws,
                                                      entries_rotated=rot)))
    return stages


def alloc_buffers(K, cfg, x, dev):
    from compressed_sparse_long_05_b300 import path as P
    buf = P.Buffers()
    B, Tq, N, d = cfg["B"], cfg["Tq"], cfg["N"], cfg["d"]
    kind = cfg["kind"]
    if kind.endswith("prefill"):
        buf.entries = torch.empty((B, N, d), dtype=x["q"].dtype, device=dev)
        if "CIa" in x:
            buf.K = torch.empty((B, N, cfg["c_I"]), dtype=x["CIa"].dtype, device=dev)
    if kind.startswith("csa"):
        buf.scores = torch.empty((B, Tq, N), dtype=torch.float32, device=dev)
        buf.idx = torch.empty((B, Tq, cfg["k"]), dtype=torch.int32, device=dev)
        dt = 3 if "qI_fp4" in x else 1
        nb = K.lib().csa_index_topk_workspace_size(B, Tq, N, dt)
        buf.ws_topk = torch.zeros(max(nb, 256), dtype=torch.uint8, device=dev)   # histograms start zero
    buf.out = torch.empty_like(x["q"])
    ent = buf.entries if kind.endswith("prefill") else P._entries_arg(x)
    nbytes = K.attend_workspace_size(x["q"], ent, P._win_arg(x), cfg.get("k", 0), cfg["m"],
                                     cfg["n_win"], cfg["r"], not kind.startswith("csa"))
    buf.ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
    return buf


def count_kernel_nodes(step, stream):
    """Kernels one step launches: kernel nodes of a captured graph of the step."""
    from cuda.bindings import runtime as rt
    g = torch.cuda.CUDAGraph(keep_graph=True)
    with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
        for _, f in step:
            f()
    err, _, n = rt.cudaGraphGetNodes(g.raw_cuda_graph(), 0)
    err, nodes, n = rt.cudaGraphGetNodes(g.raw_cuda_graph(), n)
    kern = 0
    for nd in nodes:
        e2, ty = rt.cudaGraphNodeGetType(nd)
        if ty == rt.cudaGraphNodeType.cudaGraphNodeTypeKernel:
            kern += 1
    g.reset()
    return kern


def config_dict(cfg):
    """The `config` object of a JSON line: the workload and its sizes."""
    out = {k: cfg[k] for k in ("B", "Tq", "N", "d", "r", "n_h", "m", "n_win") if k in cfg}
    for k in ("L", "T", "k", "H_I", "c_I"):
        if k in cfg:
            out[k] = cfg[k]
    if len(set(cfg["lengths"])) > 1:
        out["lengths"] = cfg["lengths"]
    out.update({"workload": cfg["name"], "kind": cfg["kind"], "storage": cfg["dtype"]})
    return out


def gpu_arm(args, cfg, rank, world, with_e2e=True):
    """Times `args.steps` steps of workload `cfg` on this rank's GPU; returns
    (JSON line fields, the first input copy)."""
    import compressed_sparse_long_05_b300 as K
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    K.lib()
    hbm_peak, tf_burst, tf_sust, peak_src = peaks()

    x0 = synth.make_inputs(cfg, seed=0, device=dev)
    wk = work(cfg)
    step_bytes = sum(b for b, _ in wk.values())
    copies = max(1, min(16, math.ceil(2 * L2_BYTES / max(1, step_bytes))))
    xs = [x0] + [synth.make_inputs(cfg, seed=s, device=dev) for s in range(1, copies)]
    bufs = [alloc_buffers(K, cfg, x, dev) for x in xs]
    steps = [make_step(K, cfg, x, b) for x, b in zip(xs, bufs)]

    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for w in range(max(3, args.warmup)):
            for _, f in steps[w % copies]:
                f()
    torch.cuda.synchronize()
    K.device_error()
    launches_per_step = count_kernel_nodes(steps[0], stream)

    # decode steps are a few microseconds: replay CUDA graphs so the host never
    # paces the GPU.  One graph runs a whole cycle over the input copies; single
    # step graphs cover the remainder, so exactly `steps` steps run.
    use_graph = cfg["kind"].endswith("decode")
    cycle, singles, inst_graphs, inst_events = None, [], [], []
    if use_graph:
        def capture(fns):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
                for f in fns:
                    f()
            return g
        cycle = capture([f for c in range(copies) for _, f in steps[c]])
        singles = [capture([f for _, f in steps[c]]) for c in range(copies)]
        for c in range(copies):
            ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(len(steps[c]) + 1)]
            gi = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gi, stream=stream, capture_error_mode="relaxed"):
                ev[0].record()
                for si, (_, f) in enumerate(steps[c]):
                    f()
                    ev[si + 1].record()
            inst_graphs.append(gi)
            inst_events.append(ev)
        torch.cuda.synchronize()
        cycle.replay()
        for g in singles:
            g.replay()
        torch.cuda.synchronize()

    def run_steps(n):
        if use_graph:
            for _ in range(n // copies):
                cycle.replay()
            for c in range(n % copies):
                singles[c].replay()
        else:
            for s_ in range(n):
                for _, f in steps[s_ % copies]:
                    f()

    # ---------------- timed region ----------------
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with clocks, torch.cuda.stream(stream):
        # keep the GPU busy while the host queues the timed steps, so that the
        # host's launch latency of the first graph replays is not timed as idle
        # device time (a short run of 20 steps would otherwise carry it)
        torch.cuda._sleep(4_000_000)
        e0.record()
        run_steps(args.steps)
        e1.record()
        e1.synchronize()
    torch.cuda.synchronize()
    ms_total = e0.elapsed_time(e1)
    if world > 1:
        ms_total = max_over_ranks(ms_total, dev)
        torch.distributed.barrier()
    K.device_error()

    # ---------------- per-stage durations ----------------
    # The same launches with an event recorded between stages, on the stream
    # they run on.  An event between two kernels keeps the second from
    # starting while the first drains, so the stage times add up to a little
    # more than the step time above (which lets consecutive kernels overlap).
    names = [n for n, _ in steps[0]]
    stage_ms = {n: [] for n in names}
    reps = min(args.steps, 200) if use_graph else min(args.steps, 5)
    with torch.cuda.stream(stream):
        for s in range(reps):
            if use_graph:
                inst_graphs[s % copies].replay()
                ev = inst_events[s % copies]
                ev[-1].synchronize()
                for si, n in enumerate(names):
                    stage_ms[n].append(ev[si].elapsed_time(ev[si + 1]))
            else:
                # keep the GPU busy while the host queues the stages, so the first
                # stage's time does not include the host's launch latency
                torch.cuda._sleep(2_000_000)
                evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
                evs[0].record()
                for si, (_, f) in enumerate(steps[s % copies]):
                    f()
                    evs[si + 1].record()
                evs[-1].synchronize()
                for si, n in enumerate(names):
                    stage_ms[n].append(evs[si].elapsed_time(evs[si + 1]))
    stage_avg = {n: float(np.mean(v)) for n, v in stage_ms.items()}

    # ---------------- end to end through the public API, host buffers ----------------
    e2e = e2e_leg(K, cfg, xs[0], bufs[0], stream, args, dev) if with_e2e else None
    bf16 = (bf16_scores_leg(K, cfg, xs[0], dev)
            if cfg["kind"] == "csa_decode" and cfg["dtype"] != "f32" else None)
    paged = (paged_leg(K, cfg, xs[0], dev)
             if cfg["kind"].endswith("decode") and cfg["dtype"] != "f32" else None)

    ms_step = ms_total / args.steps
    tokens_per_step = cfg["B"] * cfg["Tq"] * world
    value = tokens_per_step / (ms_step / 1e3)

    # roofline of the stage with the largest share of the step
    dom = max(stage_avg, key=stage_avg.get)
    b_dom, f_dom = wk[dom]
    traffic, traffic_note = profiled_traffic(cfg, dom)
    if cfg["kind"].endswith("decode") or f_dom == 0:
        achieved = b_dom / (stage_avg[dom] / 1e3) / 1e9
        roof = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": hbm_peak,
                "unit": "GB/s", "frac": round(achieved / hbm_peak, 4), "traffic": traffic,
                "traffic_source": traffic_note, "algorithmic_bytes": b_dom,
                "peak_source": peak_src + " (hbm_gbs, copy)"}
    else:
        achieved = f_dom / (stage_avg[dom] / 1e3) / 1e12
        roof = {"bound": "tensor", "kernel": dom, "achieved": round(achieved, 1), "peak": tf_sust,
                "unit": "TFLOP/s", "frac": round(achieved / tf_sust, 4), "traffic": traffic,
                "traffic_source": traffic_note, "algorithmic_flops": f_dom,
                "algorithmic_bytes": b_dom, "peak_source": peak_src + " (bf16_tflops_sustained)"}
    kernels = {}
    for n in names:
        b, f = wk[n]
        kernels[n] = {"ms": round(stage_avg[n], 5),
                      "share": round(stage_avg[n] / sum(stage_avg.values()), 4),
                      "GB/s": round(b / (stage_avg[n] / 1e3) / 1e9, 1),
                      "hbm_frac": round(b / (stage_avg[n] / 1e3) / 1e9 / hbm_peak, 4)}
        if f:
            tf = f / (stage_avg[n] / 1e3) / 1e12
            kernels[n]["TFLOP/s"] = round(tf, 1)
            kernels[n]["tensor_frac"] = round(tf / tf_sust, 4)
    step_frac_hbm = step_bytes / (ms_step / 1e3) / 1e9 / hbm_peak
    cfg_out = config_dict(cfg)
    cfg_out.update({"l2": f"inputs rotate over {copies} copies (> 2x L2 per cycle)"
                    if copies > 1 else "inputs larger than 2x L2", "graph": use_graph})
    line = {
        "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 6),
        "config": cfg_out, "roofline": roof, "step_hbm_frac": round(step_frac_hbm, 4),
        "kernels": kernels, "e2e": e2e, "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks.summary(),
    }
    if bf16:
        line["bf16_scores"] = bf16
    if paged:
        line["paged_kv_cache"] = paged
    x_first = xs[0]
    del xs, bufs, steps, cycle, singles, inst_graphs
    torch.cuda.synchronize()
    return line, x_first


def projection_leg(args, dev, tokens, g=16, d_g=1024, n_h=128, d=512, d_model=7168, reps=None):
    """The grouped output projection at V4-Pro shape (DeepSeek-V4 report,
    Chinese translation, §2.3.1 and §4.2.1: g = 16, d_g = 1024, d = 7168) for
    `tokens` rows: the [tokens, n_h*d] attention output through 16 grouped
    GEMMs to [tokens, g*d_g], then one GEMM to [tokens, d_model].  Synthetic
    bf16 inputs and weights.  Returns timing, roofline and launch counts."""
    import compressed_sparse_long_05_b300 as K
    hbm_peak, tf_burst, tf_sust, peak_src = peaks()
    gen = torch.Generator(device=dev).manual_seed(7)
    Kg = (n_h // g) * d
    A = torch.randn((tokens, n_h * d), generator=gen, device=dev).to(torch.bfloat16)
    Wg = (torch.randn((g, d_g, Kg), generator=gen, device=dev) * Kg ** -0.5).to(torch.bfloat16)
    Wo = (torch.randn((1, d_model, g * d_g), generator=gen, device=dev) * (g * d_g) ** -0.5).to(torch.bfloat16)
    y = torch.empty((tokens, g * d_g), dtype=torch.bfloat16, device=dev)
    z = torch.empty((tokens, d_model), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(device=dev)
    reps = reps or max(3, min(args.steps, 20))
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    t1, t2 = [], []
    with torch.cuda.stream(stream):
        for _ in range(3):
            K.csa_grouped_proj(A, Wg, C=y)
            K.csa_grouped_proj(y, Wo, C=z)
        for _ in range(reps):
            ev[0].record()
            K.csa_grouped_proj(A, Wg, C=y)
            ev[1].record()
            K.csa_grouped_proj(y, Wo, C=z)
            ev[2].record()
            ev[2].synchronize()
            t1.append(ev[0].elapsed_time(ev[1]))
            t2.append(ev[1].elapsed_time(ev[2]))
    K.device_error()
    ms1, ms2 = float(np.median(t1)), float(np.median(t2))
    f1 = 2.0 * tokens * g * Kg * d_g
    f2 = 2.0 * tokens * (g * d_g) * d_model
    b1 = 2 * (tokens * n_h * d + g * d_g * Kg + tokens * g * d_g)
    b2 = 2 * (tokens * g * d_g + d_model * g * d_g + tokens * d_model)
    out = {"tokens": tokens, "ms": round(ms1 + ms2, 5), "steps": reps,
           "grouped": {"ms": round(ms1, 5), "TFLOP/s": round(f1 / ms1 / 1e9, 1),
                       "GB/s": round(b1 / ms1 / 1e6, 1)},
           "final": {"ms": round(ms2, 5), "TFLOP/s": round(f2 / ms2 / 1e9, 1),
                     "GB/s": round(b2 / ms2 / 1e6, 1)},
           "gpu_launches": 2 * reps}
    if tokens >= 1024:
        ach = (f1 + f2) / ((ms1 + ms2) * 1e9)
        out["roofline"] = {"bound": "tensor", "achieved": round(ach, 1), "peak": tf_sust,
                           "unit": "TFLOP/s", "frac": round(ach / tf_sust, 4),
                           "peak_source": peak_src + " (bf16_tflops_sustained)"}
    else:
        ach = (b1 + b2) / ((ms1 + ms2) * 1e6)
        out["roofline"] = {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm_peak,
                           "unit": "GB/s", "frac": round(ach / hbm_peak, 4),
                           "peak_source": peak_src + " (hbm_gbs, copy)",
                           "note": "few tokens: the weights (369 MB) dominate the bytes"}
    del A, Wg, Wo, y, z
    torch.cuda.synchronize()
    return out


def bf16_scores_leg(K, cfg, x, dev, reps=200):
    """Index + top-k of a decode workload with the scores stored as bf16 (the
    pages' FP32 -> BF16 index-score quantisation) against float32 scores: the
    time of each (CUDA-graph replays, events on the launching stream) and the
    recall of the float32 selection."""
    from compressed_sparse_long_05_b300 import path as P
    qI, qI_sf, Kt, K_sf = P._indexer_args(x)
    B, N = cfg["B"], cfg["N"]
    stream = torch.cuda.Stream(device=dev)
    res = {}
    sel = {}
    for name, dt in (("f32", torch.float32), ("bf16", torch.bfloat16)):
        scores = torch.empty((B, 1, N), dtype=dt, device=dev)
        idx = torch.empty((B, 1, cfg["k"]), dtype=torch.int32, device=dev)
        ws = None
        with torch.cuda.stream(stream):
            for _ in range(3):
                _, _, ws = K.csa_index_topk(qI, x["w"], Kt, cfg["k"], cfg["m"], x["q_pos"], qI_sf=qI_sf,
                                            K_sf=K_sf, scores=scores, idx=idx, ws=ws, score_dtype=dt)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
            K.csa_index_topk(qI, x["w"], Kt, cfg["k"], cfg["m"], x["q_pos"], qI_sf=qI_sf, K_sf=K_sf,
                             scores=scores, idx=idx, ws=ws, score_dtype=dt)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for _ in range(10):
                g.replay()
            e0.record()
            for _ in range(reps):
                g.replay()
            e1.record()
        e1.synchronize()
        res[name + "_index_topk_ms"] = round(e0.elapsed_time(e1) / reps, 5)
        sel[name] = idx.cpu().numpy()
        del g
    K.device_error()
    rec = []
    for b in range(B):
        a32 = set(sel["f32"][b, 0].tolist()) - {-1}
        a16 = set(sel["bf16"][b, 0].tolist()) - {-1}
        rec.append(len(a32 & a16) / max(1, len(a32)))
    res["recall_of_f32_selection"] = round(float(np.mean(rec)), 5)
    res["speedup"] = round(res["f32_index_topk_ms"] / res["bf16_index_topk_ms"], 3)
    key_mb = sum(t.numel() * t.element_size() for t in (Kt, K_sf) if t is not None) / 1e6
    where = "stay in L2, so these are warm-cache times" if key_mb < 100 else "exceed L2"
    res["note"] = (f"one decode batch of the workload replayed on the same inputs (its {key_mb:.0f} MB of "
                   f"keys {where}); the pages report a 2x faster selector at 99.7% recall on the trained "
                   "model's scores")
    return res


def paged_leg(K, cfg, x, dev, reps=200):
    """One decode step of the workload through the paged KV cache (blocks of
    lcm(m, m') = 128 raw tokens handed out in scrambled order, window rows in a
    per-sequence ring) against the flat layout on the same inputs: the time of
    each (CUDA-graph replays, events on the launching stream) and whether the
    outputs are identical."""
    from compressed_sparse_long_05_b300 import path as P
    cache, views = P.PagedKVCache.from_inputs(cfg, x)
    xp = dict(x)
    xp.update(views)
    stream = torch.cuda.Stream(device=dev)
    res, outs = {}, {}
    for name, xx in (("flat", x), ("paged", xp)):
        buf = P.Buffers()
        with torch.cuda.stream(stream):
            for _ in range(3):
                P.forward(cfg, xx, buf)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
            P.forward(cfg, xx, buf)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for _ in range(10):
                g.replay()
            e0.record()
            for _ in range(reps):
                g.replay()
            e1.record()
        e1.synchronize()
        res[name + "_step_ms"] = round(e0.elapsed_time(e1) / reps, 5)
        outs[name] = buf.out.clone()
        del g
    K.device_error()
    res["identical_output"] = bool(torch.equal(outs["flat"], outs["paged"]))
    res["blocks"] = {"raw_tokens": cache.block_tokens, "csa_rows": cache.csa_rows,
                     "hca_rows": cache.hca_rows, "allocated": cache.num_blocks - cache.pool.free_count()}
    res["note"] = ("the same decode batch replayed on the same inputs for both layouts (warm L2); "
                   "blocks handed out round-robin over the sequences in shuffled order")
    cache.pool.close()
    return res


def e2e_leg(K, cfg, x, buf, stream, args, dev):
    """Same metric through the public API with per-step H2D of the step's new inputs
    (queries, indexer queries and weights; prefill also the raw rows and window)
    from pinned host memory and D2H of the output.

    Decode goes through ``path.GraphForward`` (copies and stages replayed as one
    graph).  Prefill goes through ``path.PipelinedForward``: a stream of
    independent prefill steps whose uploads and downloads overlap other steps'
    compute (each step still moves its own inputs and output).
    """
    from compressed_sparse_long_05_b300 import path as P
    names = ["q"] + (["qI", "w"] if "qI" in x else (["qI_fp4", "qI_sf", "w"] if "qI_fp4" in x else []))
    decode = cfg["kind"].endswith("decode")
    if not decode:
        names += [n for n in ("Ca", "Cb", "Za", "Zb", "C", "Z", "CIa", "CIb", "ZIa", "ZIb") if n in x]
        names += ["win"] if "win" in x else []
    n_steps = max(3, min(args.steps, 200 if decode else 3))
    if decode and cfg["kind"] == "csa_decode":
        # the C ABI's host-buffer decode step: every step copies its inputs from
        # pinned host memory, runs index, top-k and attention, copies the output
        # back, and the host waits for it
        host = {n: x[n].cpu().pin_memory() for n in names if n in x}
        host["q_pos"] = x["q_pos"][:, 0].contiguous().cpu().pin_memory()
        host["win_base"] = x["win_base"].cpu().pin_memory()
        mixed = "ent_nope" in x
        cache = {"sink": x["sink"],
                 "entries": (x["ent_nope"], x["ent_scale"], x["ent_rope"]) if mixed else x["entries"],
                 "win": (x["win_nope"], x["win_scale"], x["win_rope"]) if mixed else x["win"],
                 "K": x["K_fp4"] if mixed else x["K"]}
        if mixed:
            cache["K_sf"] = x["K_sf"]
        rates = {}
        with torch.cuda.stream(stream):
            for mode in ("eager", "graph"):
                step = K.DecodeStepHost(cache, host, cfg["k"], cfg["m"], cfg["n_win"], cfg["r"],
                                        cfg["rope_base"], graph=mode == "graph")
                for _ in range(3):
                    step()
                t0 = time.perf_counter()
                for _ in range(n_steps):
                    step()
                rates[mode] = (time.perf_counter() - t0) / n_steps
                h2d, d2h = step.h2d_bytes, step.d2h_bytes
                del step
        dt = rates["graph"]
        api = ("csa_decode_step_host (C ABI; per step: H2D of q, qI, w, positions from pinned host "
               "buffers, index, top-k, attention, D2H of the output; the call captured once into a "
               "CUDA graph and replayed, the host waits for each step; "
               f"issued eagerly from Python instead: {cfg['B'] * cfg['Tq'] / rates['eager']:.1f} tokens/s)")
        K.device_error()
    elif decode:
        fw = P.GraphForward(cfg, x, names, stream=stream)
        for _ in range(3):
            fw()
        t0 = time.perf_counter()
        for _ in range(n_steps):
            fw()
        dt = (time.perf_counter() - t0) / n_steps
        h2d, d2h = fw.h2d_bytes, fw.d2h_bytes
        api = "compressed_sparse_long_05_b300.path.GraphForward (H2D, every stage and D2H in one CUDA graph)"
        del fw
    else:
        host = {n: x[n].cpu().pin_memory() for n in names}
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        pf = P.PipelinedForward(cfg, x, names)
        d2h = pf.out_host[0].numel() * pf.out_host[0].element_size()
        for s_ in range(2):
            pf.submit(host)
        pf.wait(1)
        n_steps = max(n_steps, 8)
        t0 = time.perf_counter()
        first = pf.step
        for s_ in range(n_steps):
            pf.wait(first + s_ - 2)           # that step's output has arrived before its buffer is reused
            pf.submit(host)
        pf.wait(first + n_steps - 1)
        dt = (time.perf_counter() - t0) / n_steps
        api = ("compressed_sparse_long_05_b300.path.PipelinedForward (per step: H2D of its inputs, "
               "every stage, D2H of its output; transfers overlap other steps' compute)")
        del pf
    return {"value": round(cfg["B"] * cfg["Tq"] / dt, 1), "unit": "tokens/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": n_steps,
            "api": api}


# ----------------------------------------------------------------------------
# CPU oracle arm
# ----------------------------------------------------------------------------


def cpu_info():
    """(logical cores usable by this process, CPU model name)."""
    try:
        cores = len(os.sched_getaffinity(0))
    except Exception:
        cores = os.cpu_count() or 1
    model = "unknown"
    try:
        for line in open("/proc/cpuinfo"):
            if line.startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    return cores, model


def blas_threads():
    """(threads of numpy's BLAS pool, note).  Without threadpoolctl the pool
    size is not known: the logical core count is reported, with the reason."""
    try:
        from threadpoolctl import threadpool_info
        info = [i for i in threadpool_info() if i.get("user_api") == "blas"]
        if info:
            return max(int(i.get("num_threads", 1)) for i in info), "numpy BLAS pool (threadpoolctl)"
        note = "threadpoolctl saw no BLAS pool"
    except Exception as e:   # pragma: no cover - depends on the host
        note = f"threadpoolctl failed: {e!r}"[:160]
    return cpu_info()[0], note + "; reporting the logical cores"


def one_thread_rate(workload, budget_s):
    """The oracle's tokens/s with every BLAS/OpenMP pool held to one thread:
    a child process (the pool size is fixed when numpy loads) that generates
    the workload's inputs on the CPU and times a bounded sample."""
    import subprocess
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    code = ("import sys, json; sys.path.insert(0, %r); import bench, synth; "
            "cfg = synth.get(%r); x = bench.host_copy(synth.make_inputs(cfg, seed=0)); "
            "print(json.dumps(bench.oracle_sample(cfg, x, %r)[0]))" % (ROOT, workload, budget_s))
    try:
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                           timeout=120 + 4 * budget_s)
        return float(r.stdout.strip().splitlines()[-1])
    except Exception:
        return None


def oracle_sample(cfg, x_np, budget_s):
    """Runs the oracle on query rows of the workload until ~budget_s elapsed.

    Returns (tokens/s, description).  Prefill workloads count the compression
    of one batch row in full plus whole query rows of the rest.
    """
    from oracle import pipeline as OP
    kind = cfg["kind"]
    t_start = time.perf_counter()
    done_rows = 0
    ent = None
    if kind.endswith("prefill"):
        ent = OP.entries_of(cfg, x_np, 0)
    t_comp = time.perf_counter() - t_start
    rows_total = cfg["Tq"]
    rng = np.random.default_rng(0)
    order = rng.permutation(rows_total)
    t_rows = 0.0
    b = 0
    while True:
        t0 = time.perf_counter()
        i = int(order[done_rows % rows_total])
        OP.run_rows(cfg, x_np, b, [i], entries=ent)
        t_rows += time.perf_counter() - t0
        done_rows += 1
        if time.perf_counter() - t_start > budget_s or done_rows >= max(4 * rows_total, 100000):
            break
        if done_rows % rows_total == 0:
            b = (b + 1) % cfg["B"]
    per_row = t_rows / done_rows
    if kind.endswith("prefill"):
        # one full step per batch row = compression + every query row
        t_step_per_row = t_comp + per_row * rows_total
        tps = rows_total / t_step_per_row
        desc = (f"compression of one {cfg['T']}-token sequence in full ({t_comp:.2f}s) + "
                f"{done_rows} query rows of index/top-k/attend; tokens/s = T / (compress + T x "
                "per-row time), extrapolated from the sampled rows")
    else:
        tps = 1.0 / per_row
        desc = f"{done_rows} decode query rows (index over all N entries, top-k, attend)"
    return tps, desc


def cpu_baseline(cfg, x_np, budget_s):
    """The oracle timed on this host: its BLAS thread pool as it stands on a
    bounded sample of the workload (~2/3 of budget_s), and one thread in a
    child process (~1/3)."""
    cores, model = cpu_info()
    threads, note = blas_threads()
    tps, desc = oracle_sample(cfg, x_np, budget_s * 2 / 3)
    tps1 = one_thread_rate(cfg["name"], budget_s / 3) if cfg["name"] in synth.configs.WORKLOADS else None
    return {"value": round(tps, 4), "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": desc, "nproc": cores, "cpu_model": model,
            "value_1_thread": None if tps1 is None else round(tps1, 4),
            "threads_note": f"{note}; float64 numpy oracle: its row loop is serial Python, only "
                            "the BLAS matrix products use the pool"}


class _RowView:
    """Read-only view of a large tensor for the oracle: indexing down to a
    2-D (or smaller) slice returns that slice alone as a float32/int numpy
    array, so a sampled row never needs the whole tensor on the host."""

    def __init__(self, t):
        self.t = t

    def __getitem__(self, k):
        if isinstance(k, (np.ndarray, list)):          # a set of rows: fetch just those
            return _np(self.t[torch.as_tensor(np.asarray(k), device=self.t.device)])
        v = self.t[k]
        return _RowView(v) if v.dim() > 2 else _np(v)

    def __len__(self):
        return self.t.shape[0]


def _np(v):
    return v.float().cpu().numpy() if v.dtype in (torch.bfloat16, torch.float32) else v.cpu().numpy()


def host_copy(x):
    """Inputs as the oracle reads them: numpy copies, except that tensors above
    256 MB stay where they are behind a per-row view."""
    return {k: (_RowView(v) if v.numel() * v.element_size() > (256 << 20) else _np(v))
            for k, v in x.items()}


def reference_arm(args, cfg, rank, world):
    if rank != 0:
        return None
    x = synth.make_inputs(cfg, seed=0, device="cuda" if torch.cuda.is_available() else "cpu")
    xn = host_copy(x)
    del x
    # the oracle is slow by design: W short warm-up samples (at least 3, ~0.2 s
    # each), then up to 3 timed samples of --cpu-budget seconds whatever K is
    run_steps = max(1, min(args.steps, 3))
    per_step_budget = args.cpu_budget
    warm = max(3, args.warmup)
    for _ in range(warm):
        oracle_sample(cfg, xn, min(0.2, per_step_budget))
    vals = []
    desc = ""
    for s in range(run_steps):
        tps, desc = oracle_sample(cfg, xn, per_step_budget)
        vals.append(tps)
    value = float(np.mean(vals))
    tokens = cfg["B"] * cfg["Tq"]
    cores, model = cpu_info()
    cfg_out = config_dict(cfg)
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tokens/s",
            "n_gpus": world, "steps": run_steps, "steps_requested": args.steps, "warmup": warm,
            "ms_per_step": round(tokens / value * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": cfg_out,
            "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": blas_threads()[0],
                             "kind": "oracle", "nproc": cores, "cpu_model": model,
                             "sample": desc + f"; {run_steps} sample steps of ~{per_step_budget:.0f}s"},
            "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


PREFILL_WORKLOAD = "csa_prefill_32k"


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.configs.WORKLOADS))
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle CPU work")
    ap.add_argument("--no-prefill", action="store_true",
                    help="default workload only: skip the 32K-prefill half of the metric")
    ap.add_argument("--set", action="append", default=[], metavar="KEY=INT",
                    help="override a size of the workload (smaller cases for profiling)")
    args = ap.parse_args()
    over = {kv.split("=")[0]: int(kv.split("=")[1]) for kv in args.set}
    cfg = synth.scaled(args.workload, **over) if over else synth.get(args.workload)
    decode = cfg["kind"].endswith("decode")
    steps_given, warm_given = args.steps, args.warmup
    if args.steps is None:
        args.steps = 20000 if decode else 10
    if args.warmup is None:
        args.warmup = 50 if decode else 3
    args.warmup = max(3, args.warmup)
    # the metric is quoted at decode @128K and prefill @32K: the default run times both
    with_prefill = args.workload == DEFAULT_WORKLOAD and not over and not args.no_prefill
    pcfg = synth.get(PREFILL_WORKLOAD) if with_prefill else None
    pargs = argparse.Namespace(**vars(args))
    pargs.steps = steps_given if steps_given is not None else 10
    pargs.steps = max(3, min(pargs.steps, 20))
    pargs.warmup = max(3, min(warm_given if warm_given is not None else 3, 5))

    world = int(os.environ.get("WORLD_SIZE", 1))
    rank = int(os.environ.get("RANK", 0))
    if world > 1:
        backend = "nccl" if args.impl == "native" else "gloo"
        torch.distributed.init_process_group(backend)

    common = {"metric": METRIC, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
              "data": "synthetic"}
    if args.impl == "reference":
        line = reference_arm(args, cfg, rank, world)
        if rank == 0 and with_prefill:
            pline = reference_arm(pargs, pcfg, rank, world)
            line["prefill_32k"] = {k: pline[k] for k in ("value", "unit", "ms_per_step", "config",
                                                         "cpu_baseline")}
        if rank == 0:
            print(json.dumps(line), flush=True)
    else:
        fields, x0 = gpu_arm(args, cfg, rank, world)
        line = dict(common)
        line.update(fields)
        line["dtype"] = "bf16" if cfg["dtype"] != "f32" else "f32"
        if rank == 0 and world == 1:
            line["cpu_baseline"] = cpu_baseline(cfg, host_copy(x0), args.cpu_budget)
        del x0
        if with_prefill:
            pf, px0 = gpu_arm(pargs, pcfg, rank, world)
            pf = {k: pf[k] for k in ("value", "unit", "ms_per_step", "steps", "warmup", "config",
                                     "roofline", "kernels", "e2e", "gpu_launches", "clocks")}
            if rank == 0 and world == 1:
                pf["cpu_baseline"] = cpu_baseline(pcfg, host_copy(px0), args.cpu_budget)
            del px0
            line["prefill_32k"] = pf
            dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
            line["output_projection"] = {
                "what": "grouped output projection, V4-Pro shape (g=16, d_g=1024, d=7168), bf16",
                "prefill_32k": projection_leg(args, dev, 32768),
                "decode_b4": projection_leg(args, dev, 4)}
        if rank == 0:
            print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
