"""Token-tile sweep: writes the tile table the binding loads (tile_table.csv).

    python -m quantized_mixture_experts_moe_gb300.tune [--out PATH] [--workloads NAME ...]

In the manner of the tuned grouped-fmoe configuration rows (the aiter tuned
grouped-fmoe page, Changes: one row per model shape, TP degree and token
bucket 1-256, 1024, 4096, 8192), each workload's layer is run through
qmoe_moe_forward with the token tile pinned to 16, 112 and 224 rows.  Per
(shape, token bucket) the tile with the smaller total step time over the
bucket's workloads becomes a rule.

Checks, per workload:
  * the tiles' outputs agree to rel L2 < 5e-3 (they differ only in the order
    of fp32 sums; the tests compare each against the CPU oracle);
  * no K tile passes the end of K: every kernel steps K in 128-element tiles,
    so a shape with H % 256 or I % 128 is excluded rather than tuned.
"""

from __future__ import annotations

import argparse
import csv
import os
import statistics
import sys

import numpy as np
import torch

from quantized_mixture_experts_moe_gb300 import binding as qb
from quantized_mixture_experts_moe_gb300 import inputs as gen

TILES = (16, 112, 224)
BUCKETS = [(1, 256), (257, 1024), (1025, 4096), (4097, 8192), (8193, 2**31 - 1)]
DEFAULT_WORKLOADS = [
    "decode_T1", "decode_T4", "decode_T16", "decode_T64",
    "mxfp4_T256", "mxfp4_T1024", "mxfp4_T4096", "mxfp4_T8192",
    *[f"mxfp4_tp{tp}_T{T}" for tp in (2, 4) for T in (16, 256, 1024, 4096, 8192)],
    "w4a16_T2048", "w8a8_T8192", "w4a8_T8192",
]
L2_BYTES = 129 * 10**6


def bucket_of(T):
    return next(b for b in BUCKETS if b[0] <= T <= b[1])


def time_layer(w, t, out, status, ws, steps, flush):
    """Median step time (µs) of the whole layer through the public entry point."""
    dims = qb.dims(w.T, w.k, w.H, w.I, w.E)
    run = lambda: qb.qmoe_moe_forward(w.scheme, dims, t["x"], t["topk_ids"], t["topk_w"], t["w1"], t["w1_s"],
                                      t["w2"], t["w2_s"], out, status, ws)
    for _ in range(3):
        run()
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        if flush is not None:
            flush.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        run()
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b) * 1e3)
    assert int(status.item()) == 0, f"{w.name}: device status {int(status.item())}"
    return statistics.median(times)


def measure(w, steps=10):
    if w.H % 256 or w.I % 128:
        return None  # a 128-element K tile would pass the end of K
    dev = torch.device("cuda")
    d = gen.make_all(w)
    to = lambda a: torch.from_numpy(np.ascontiguousarray(a.view(np.int16) if a.dtype == np.uint16 else a)).to(dev)
    t = {k: to(v) for k, v in d.items()}
    if w.scheme == "mxfp4":
        t["w1"], t["w1_s"], t["w2"], t["w2_s"] = qb.prepack_mxfp4(t["w1"], t["w1_s"], t["w2"], t["w2_s"], w.H, w.I)
    elif w.scheme == "w4a16":
        t["w1"], t["w2"] = qb.prepack_w4a16(t["w1"], t["w1_s"], t["w2"], t["w2_s"], w.H, w.I)
        t["w1_s"] = t["w2_s"] = None
    # a step touching under 4x L2 of weights runs behind an L2 flush, so it streams them from HBM
    touched = len(np.unique(d["topk_ids"]))
    wbytes = dict(mxfp4=0.53, w4a16=0.56, w8a8=1.0, w4a8=0.5)[w.scheme]
    small = touched * 3 * w.H * w.I * wbytes < 4 * L2_BYTES
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev) if small else None
    res, outs = {}, {}
    dims = qb.dims(w.T, w.k, w.H, w.I, w.E)
    for nmax in TILES:
        qb.set_tile_rules([dict(H=w.H, I=w.I, E=w.E, k=w.k, t_min=w.T, t_max=w.T, nmax=nmax)])
        ws = qb.alloc_workspace(qb.forward_workspace_bytes(dims, w.scheme), dev)
        out = torch.empty((w.T, w.H), dtype=torch.int16, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        res[nmax] = time_layer(w, t, out, status, ws, steps, flush)
        outs[nmax] = (out.cpu().numpy().astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        del ws
    ref = outs[112]
    rel = max(float(np.linalg.norm(outs[n] - ref) / max(np.linalg.norm(ref), 1e-300)) for n in TILES)
    return dict(**{f"us_{n}": res[n] for n in TILES}, rel=rel)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--out", default=qb.TILE_TABLE_PATH)
    ap.add_argument("--workloads", nargs="*", default=DEFAULT_WORKLOADS)
    ap.add_argument("--steps", type=int, default=10)
    args = ap.parse_args(argv)
    groups = {}
    for name in args.workloads:
        w = gen.WORKLOADS[name]
        m = measure(w, args.steps)
        if m is None:
            print(f"{name}: excluded (K tiles would pass the end of K)", file=sys.stderr)
            continue
        ok = m["rel"] < 5e-3
        print(f"{name:22s} " + "  ".join(f"{n}: {m[f'us_{n}']:8.1f} us" for n in TILES) + "  rel L2 between tiles "
              f"{m['rel']:.2e} {'ok' if ok else 'MISMATCH'}", file=sys.stderr)
        if not ok:
            continue
        key = (w.scheme, w.H, w.I, w.E, w.k, bucket_of(w.T))
        g = groups.setdefault(key, dict(**{f"us_{n}": 0.0 for n in TILES}, reps=[]))
        for n in TILES:
            g[f"us_{n}"] += m[f"us_{n}"]
        g["reps"].append(w.T)
    qb.set_tile_rules([])
    rows = []
    for (scheme, H, I, E, k, (lo, hi)), g in sorted(groups.items(), key=lambda x: (x[0][:5], x[0][5][0])):
        nmax = min(TILES, key=lambda n: (g[f"us_{n}"], n != 112))  # ties keep the 112-row tile
        rows.append(dict(scheme=scheme, H=H, I=I, E=E, k=k, t_min=lo, t_max=hi, nmax=nmax,
                         t_measured=" ".join(map(str, g["reps"])), **{f"us_{n}": f"{g[f'us_{n}']:.1f}" for n in TILES}))
    with open(args.out, "w", newline="") as f:
        f.write("# token-tile table written by quantized_mixture_experts_moe_gb300.tune on "
                f"{torch.cuda.get_device_name()}: per (shape, token bucket) the tile with the smaller\n"
                "# summed step time over the bucket's measured token counts (us_16, us_112, us_224)\n")
        wr = csv.DictWriter(f, fieldnames=[*qb.TILE_TABLE_FIELDS, "t_measured", *[f"us_{n}" for n in TILES]])
        wr.writeheader()
        wr.writerows(rows)
    print(f"wrote {len(rows)} rules to {args.out}", file=sys.stderr)


if __name__ == "__main__":
    main()
