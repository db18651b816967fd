"""Per-phase timeline of one layer forward's kernels, from the phase-trace build.

    CSA_LIB_TRACE=1 python -m compressed_sparse_long_05_b300.trace [--workload NAME] [--reps R]

Builds (if needed) and loads ``lib/libcsa_b300_trace.so`` (the same sources
compiled with -DCSA_TRACE: kernels mark the SM clock at their phase
boundaries), runs R layer forwards of the workload, and prints for the index, top-k and
attention kernels when their CTAs start and end, and per phase the median
over launches and CTAs of the time since the CTA started, in microseconds
(SM cycles converted with the wall-clock span of each CTA).
"""

from __future__ import annotations

import argparse
import ctypes
import os
import sys

import numpy as np

# kernel -> (wall-clock entry slot, clock entry slot, clock exit slot, wall exit slot, phases)
KERNELS = {
    "index (index_tc_kernel or index_fp4_kernel)": (32, 33, 44, 43, {
        34: "barriers + TMEM allocated",
        45: "producer: first item's tiles known",
        46: "producer: first K-tile copy issued",
        47: "producer: first item's prefetch copies issued",
        35: "producer: first item's query group issued",
        36: "MMA: first K tile landed",
        37: "MMA: every MMA of the first item issued",
        38: "epilogue warp 2: first tiles folded",
        39: "epilogue warp 2: last tile folded",
        40: "epilogue warp 2: item's tiles done",
        41: "histogram flush start",
        42: "histogram flush end",
        57: "FP4: scale warp 2, first tile's scale atoms in tensor memory",
        58: "FP4: scale warp 2, last tile's scale atoms in tensor memory",
        59: "FP4: producer, every copy of the first item issued",
        60: "FP4: epilogue warp 4, its 21st tile: waits for the accumulator",
        61: "FP4: epilogue warp 4, its 21st tile: accumulator ready",
        62: "FP4: epilogue warp 4, its 21st tile: heads folded",
        63: "FP4: epilogue warp 4, its 21st tile: scores stored, histogram added, released",
    }),
    "top-k (topk2_kernel)": (48, 49, 56, 55, {
        50: "histogram read, cluster barrier passed",
        51: "threshold bin found",
        52: "candidates gathered",
        53: "radix passes done (k-th key known)",
        54: "indices written",
    }),
    "attention (attend_tc_kernel)": (0, 1, 22, 21, {
        2: "barriers + TMEM allocated",
        29: "MMA warp: first item's rows known",
        30: "MMA warp: first q box issued",
        3: "q TMA issued (MMA warp)",
        31: "gather warp 4: first item's rows known",
        4: "q landed (MMA warp)",
        5: "traced tile: row sources known (gather warp 4)",
        6: "traced tile: every row copy issued",
        7: "traced tile: rows landed",
        8: "traced tile: RoPE done, last chunk released",
        9: "traced tile: QK issued (all chunks in)",
        10: "traced tile: S in softmax warps",
        23: "traced tile: S read from TMEM",
        24: "traced tile: tile max exchanged (4 warps)",
        25: "traced tile: P computed in registers",
        11: "traced tile: P written",
        12: "traced tile: PV issued",
        13: "traced tile: row sums done",
        14: "epilogue: last PV done",
        15: "epilogue: O stored (single chunk or split mode)",
        16: "all roles done (before merge)",
        17: "merge: own partial staged as bf16",
        18: "merge: every chunk's (max, sum) received",
        19: "merge: copies issued, weights computed",
        20: "merge: this CTA's blocks received",
        26: "merge: outputs stored",
        27: "merge: own copies read",
    }),
}


def main():
    if os.environ.get("CSA_LIB_TRACE") != "1":
        os.environ["CSA_LIB_TRACE"] = "1"
        os.execv(sys.executable, [sys.executable, "-m", "compressed_sparse_long_05_b300.trace"] +
                 sys.argv[1:])
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import torch

    import synth
    from compressed_sparse_long_05_b300 import _lib, build, path as P

    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="csa_decode_128k")
    ap.add_argument("--reps", type=int, default=20)
    ap.add_argument("--tile", type=int, default=0,
                    help="which tile of each attention CTA its per-tile marks describe")
    ap.add_argument("--set", action="append", default=[], metavar="KEY=INT",
                    help="override a size of the workload")
    ap.add_argument("--paged", action="store_true",
                    help="decode through the paged KV cache (blocks in shuffled order)")
    args = ap.parse_args()
    build.build(trace=True)
    L = _lib.lib()
    over = {kv.split("=")[0]: int(kv.split("=")[1]) for kv in args.set}
    cfg = synth.scaled(args.workload, **over) if over else synth.get(args.workload)
    L.csa_trace_set_tile.argtypes = [ctypes.c_int]
    L.csa_trace_set_tile(args.tile)
    x = synth.make_inputs(cfg, seed=0, device="cuda")
    if args.paged:
        cache, views = P.PagedKVCache.from_inputs(cfg, x)
        x.update(views)
    buf = P.Buffers()
    P.forward(cfg, x, buf)                          # every stage once (sizes buffers)
    torch.cuda.synchronize()
    ncta, nslot = 160, 64
    host = (ctypes.c_longlong * (ncta * nslot))()
    L.csa_trace_read(host, ncta * nslot)            # clear
    rows = []
    for _ in range(args.reps):
        P.forward(cfg, x, buf)
        torch.cuda.synchronize()
        L.csa_trace_read(host, ncta * nslot)
        rows.append(np.frombuffer(host, dtype=np.int64).reshape(ncta, nslot).copy())
    a = np.stack(rows)                              # [reps, cta, slot]
    print(f"workload {cfg['name']}: {args.reps} forward passes; times in us")
    t0 = None
    for name, (w0, c0, c1, w1, phases) in KERNELS.items():
        live = (a[:, :, c0] > 0) & (a[:, :, c1] > a[:, :, c0]) & (a[:, :, w1] > a[:, :, w0])
        if not live.any():
            continue
        cyc = (a[:, :, c1] - a[:, :, c0]).astype(np.float64)
        wall = (a[:, :, w1] - a[:, :, w0]).astype(np.float64)
        ghz = np.median(cyc[live] / wall[live])
        starts = np.where(live, a[:, :, w0], np.iinfo(np.int64).max).min(axis=1)
        ends = np.where(live, a[:, :, w1], 0).max(axis=1)
        if t0 is None:
            t0 = starts
        print(f"\n{name}: {int(live[0].sum())} CTAs, SM clock {ghz:.3f} GHz; first CTA start "
              f"+{np.median(starts - t0) / 1e3:.2f}, last CTA end +{np.median(ends - t0) / 1e3:.2f} "
              f"(from the first traced kernel's start); CTA span median "
              f"{np.median(wall[live]) / 1e3:.2f}, max {wall[live].max() / 1e3:.2f}")
        print(f"  {'slot':>4}  {'median':>7}  {'p90':>7}  phase (time since the CTA's entry)")
        for slot, what in phases.items():
            m = live & (a[:, :, slot] > 0)
            if not m.any():
                continue
            us = (a[:, :, slot] - a[:, :, c0]).astype(np.float64)[m] / ghz / 1e3
            print(f"  {slot:>4}  {np.median(us):7.2f}  {np.percentile(us, 90):7.2f}  {what}")
        us = cyc[live] / ghz / 1e3
        print(f"  {c1:>4}  {np.median(us):7.2f}  {np.percentile(us, 90):7.2f}  exit")
    _lib.device_error()


if __name__ == "__main__":
    main()
