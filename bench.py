"""Benchmark of the affine 4-bit group-quantized product on one GB300 per rank.

Headline workload: the 4096x2048 product called 400 times (the pages'
per-call measurement, "Array.q4mv on Metal ..." bendlang/bend #1435,
Verification: a 4096x2048 product run 400 times, printing a hash of y).  One
step = the activation's group sums, then the 400 products queued as one stage
("Array.q4go/Array.q4wait ..." #1437, Change: queued products run
concurrently and none reads another's y), recorded as one stage graph and
launched once.  Each of the 400 products reads its own copy of the weights
(2.1 GB in all, many times the L2 cache), so every call streams its weights
from HBM and nothing read in one step is still cached in the next.

Also measured in the same run (as "extra"): the same 400 products as 400
dependent stages (each waits for the previous one: decode-like latency), the
248320x2048 output head, one synthetic 24-layer decode token (fused and
unfused stage graphs), the 4096x2048 product in every weight format
(groups of 32, 64 or 128 columns; f32, bf16 or f16 scale and bias), each as a
grouped launch of 256 products streaming from HBM, the batched product
(1, 2, 4 and 8 tokens sharing the 248320x2048 head's weights), and the pages'
own timing of the 4096x2048 product ((400-call - 1-call)/400, median of 6).
and the rows x cols x rows-per-item x mode sweep (GB/s and fraction of peak
per point, and the fast-mode error over every row of each point).

Output: one JSON line on rank 0.  --impl reference times the CPU oracle (the
plain C definition the library is tested against) on the same workload.
Multi-GPU runs are independent replicas (the product has no exchange step).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from affine_bit_group_gb300 import synth  # noqa: E402

CALLS = 400
GROUP = 256  # products per grouped launch (the library's limit)
MID_ROWS, MID_COLS = 4096, 2048
PEAK_FALLBACK_GBS = 6800.0


def product_bytes(rows: int, cols: int, group: int = 64, sb_bytes: int = 4) -> int:
    """Algorithmic bytes of one product: nibbles, scale and bias, x, xsum and y."""
    G = cols // group
    return rows * cols // 2 + 2 * sb_bytes * rows * G + 4 * cols + 4 * G + 4 * rows


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    return PEAK_FALLBACK_GBS, "fallback"


def code_sha256(path: str) -> str:
    """sha256 of a C/CUDA source's code: // comments, trailing blanks and empty
    lines removed, so that an edit of comments alone keeps a profile valid."""
    out = []
    with open(path) as f:
        for line in f:
            quote = False
            cut = len(line)
            for i, c in enumerate(line):
                if c == '"' and (i == 0 or line[i - 1] != "\\"):
                    quote = not quote
                elif not quote and line.startswith("//", i):
                    cut = i
                    break
            code = line[:cut].rstrip()
            if code:
                out.append(code)
    return hashlib.sha256("\n".join(out).encode()).hexdigest()


# Every source the product kernel's code and launch plan depend on: a profile
# recorded for one version of these stays valid only while none of them changes.
KERNEL_SOURCES = tuple(os.path.join("affine_bit_group_gb300", "csrc", f) for f in
                       ("q4mv_kernel.cuh", "abg_dev.cuh", "abg_kernels.cuh", "q4mv.cu", "q4mv_fixed.cu"))


def kernel_code_sha256(paths=None) -> str:
    """sha256 over the code (comments and blank lines removed) of the kernel's sources, in order."""
    h = hashlib.sha256()
    for rel in (paths or KERNEL_SOURCES):
        h.update(rel.encode() + b"\0" + code_sha256(os.path.join(ROOT, rel)).encode() + b"\n")
    return h.hexdigest()


def profile_traffic(profile: str):
    """DRAM bytes per launch from a committed ncu summary, or None once the kernel's code changed."""
    path = os.path.join(ROOT, "profiles", profile)
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.strip().startswith(("dram_bytes_per_launch", "kernel_code_sha256")):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.split()[0].strip("`")
    if vals.get("kernel_code_sha256") != kernel_code_sha256() or "dram_bytes_per_launch" not in vals:
        return None
    return float(vals["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_uuid: str | None):
        self.rows = []
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if device_uuid:
            cmd += ["-i", device_uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 8:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        if not self.rows:
            return None
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        reasons = set()
        for r in self.rows:
            for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"), r[4:]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(self.rows)}


def device_uuid():
    import torch
    try:
        u = torch.cuda.get_device_properties(0).uuid
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    except Exception:
        return None


def rotating_copies(m, copies: int):
    """`copies` device copies of one matrix (same bits; separate memory)."""
    import torch
    w = torch.from_numpy(m.w.view(np.int32)).cuda()
    s = torch.from_numpy(m.scale).cuda()
    b = torch.from_numpy(m.bias).cuda()
    return [(w.clone(), s.clone(), b.clone()) for _ in range(copies)]


def build_mid_graph(abg, mats, x, xsum, ys, calls, chained: bool, mode=0, host_io=None):
    """Group sums of x, then `calls` products: one stage (queued, independent)
    or one stage each (every product waits for the previous one).  With
    host_io = (x_host, y_host) the graph first copies x from pinned host
    memory and last copies the final product's y back there."""
    first = 0 if host_io is None else 1
    nodes = [] if host_io is None else [abg.Node.copy(0, host_io[0], x)]
    nodes.append(abg.Node.gsum(first, x, xsum))
    for i in range(calls):
        w, s, b = mats[i % len(mats)]
        y = ys[i % len(ys)]
        nodes.append(abg.Node.q4mv(first + 1 + i if chained else first + 1, w, s, b, y, MID_COLS, x=x, xsum=xsum))
    keep = [x, xsum] + ys + [t for m in mats for t in m]
    if host_io is not None:
        nodes.append(abg.Node.copy(nodes[-1].stage + 1, ys[(calls - 1) % len(ys)], host_io[1]))
        keep += list(host_io)
    return abg.StageGraph(nodes, mode=mode, keep=keep)


def time_graph(graph, stream, steps, warmup, sampler_uuid=None):
    """(ms per replay, clocks) with CUDA events on `stream`, synchronize on both sides."""
    import torch
    for _ in range(warmup):
        graph.launch(stream)
    torch.cuda.synchronize()
    sampler = ClockSampler(sampler_uuid) if sampler_uuid is not False else None
    time.sleep(0.3 if sampler else 0)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(steps):
        graph.launch(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    return e0.elapsed_time(e1) / steps, clocks


def run_ours(args, rank, world):
    import torch

    import affine_bit_group_gb300 as abg
    import oracle
    from affine_bit_group_gb300 import decode

    torch.cuda.set_device(0 if world == 1 else int(os.environ.get("LOCAL_RANK", rank)))
    stream = torch.cuda.Stream()
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    l2 = getattr(props, "L2_cache_size", 126 * 2 ** 20)
    peak, peak_kind = measured_peak()

    # ---------------------------------------------------------------- mid ---
    m, x_np = synth.mid()
    pbytes = product_bytes(MID_ROWS, MID_COLS)
    # one copy per product of the step: no product of a grouped launch or of
    # the next step finds its weights in L2
    copies = max(CALLS, math.ceil(3 * l2 / (m.nbytes)))
    mats = rotating_copies(m, copies)
    x = torch.from_numpy(x_np).cuda()
    xsum = torch.empty(MID_COLS // 64, dtype=torch.float32, device="cuda")
    ys = [torch.empty(MID_ROWS, dtype=torch.float32, device="cuda") for _ in range(CALLS)]
    g = build_mid_graph(abg, mats, x, xsum, ys, CALLS, chained=False)
    uuid = device_uuid()
    ms_step, clocks = time_graph(g, stream, args.steps, args.warmup, uuid if rank == 0 else False)
    y_last = ys[CALLS - 1]
    y_hash = oracle.hash32(y_last.cpu().numpy())
    if any(oracle.hash32(ys[i].cpu().numpy()) != y_hash for i in (0, 1, 199)):
        raise SystemExit("the 400 products do not all give the same bits")
    exp_hash = oracle.hash32(oracle.q4mv(*m.arrays(), x_np, oracle.gsum(x_np), MID_COLS))
    if y_hash != exp_hash:
        raise SystemExit(f"mid product hash {y_hash} differs from the oracle's {exp_hash}")
    step_bytes = CALLS * pbytes
    value = step_bytes / (ms_step * 1e-3) / 1e9
    us_per_product = ms_step * 1e3 / CALLS
    launches_per_step = g.launches

    # the dominant kernel alone: one grouped launch of 256 products (the
    # step's product launches are of this kind), timed with CUDA events on
    # the stream it runs on
    g1 = abg.StageGraph([abg.Node.q4mv(0, *mats[i % len(mats)], ys[i], MID_COLS, x=x, xsum=xsum)
                         for i in range(GROUP)], keep=[x, xsum] + ys)
    ms_launch, _ = time_graph(g1, stream, max(args.steps, 10), args.warmup, False)
    g1.close()
    achieved = GROUP * pbytes / (ms_launch * 1e-3) / 1e9

    # the same 400 products as 400 dependent stages (decode-like latency)
    gc = build_mid_graph(abg, mats, x, xsum, ys[:2], CALLS, chained=True)
    ms_chain, _ = time_graph(gc, stream, args.steps, args.warmup, False)
    chain = {"us_per_product": ms_chain * 1e3 / CALLS, "gbs": step_bytes / (ms_chain * 1e-3) / 1e9,
             "launches": gc.launches}
    gc.close()

    # ---------------------------------------------------------------- e2e ---
    # the same step as one stage graph that copies x in from pinned host
    # memory and the last product's y back out (copy nodes): one launch and
    # one synchronization per step, timed on the host
    x_host = torch.from_numpy(x_np).pin_memory()
    y_host = torch.empty(MID_ROWS, dtype=torch.float32).pin_memory()
    g.close()
    g = build_mid_graph(abg, mats, x, xsum, ys, CALLS, chained=False, host_io=(x_host, y_host))
    for _ in range(args.warmup):
        g.launch(stream)
        stream.synchronize()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        g.launch(stream)
        stream.synchronize()
    e2e_s = (time.perf_counter() - t0) / args.steps
    if oracle.hash32(y_host.numpy()) != exp_hash:
        raise SystemExit("the e2e step's host output differs from the oracle's")
    e2e = {"value": step_bytes / e2e_s / 1e9, "unit": "GB/s", "h2d_bytes_per_step": 4 * MID_COLS,
           "d2h_bytes_per_step": 4 * MID_ROWS, "ms_per_step": e2e_s * 1e3}
    g.close()
    del mats, g
    torch.cuda.empty_cache()

    extra = {"mid_chained": chain}
    if not args.no_extra:
        extra["head"] = bench_head(abg, stream, args, peak)
        extra["decode_token"] = bench_decode(abg, decode, stream, args)
        extra["formats"] = bench_formats(abg, stream, args, peak, l2)
        extra["batched"] = bench_batched(abg, stream, args)
        extra["pages_way"] = bench_pages_way(abg, stream, args)
        extra["gdn"] = bench_gdn(abg, stream, args)
        extra["atq"] = bench_atq(abg, stream, args)
        extra["sweep"] = bench_sweep(abg, stream, args, peak, l2)

    res = dict(value=value, ms_step=ms_step, us_per_product=us_per_product, achieved=achieved,
               launch_us=ms_launch * 1e3, clocks=clocks,
               e2e=e2e, extra=extra, launches=launches_per_step * args.steps, peak=peak, peak_kind=peak_kind,
               hash=y_hash, copies=copies)
    return res


def bench_head(abg, stream, args, peak):
    import torch
    m, hidden, wt = synth.head()
    rows, cols = m.rows, m.cols
    w = torch.from_numpy(m.w.view(np.int32)).cuda()
    s = torch.from_numpy(m.scale).cuda()
    b = torch.from_numpy(m.bias).cuda()
    h = torch.from_numpy(hidden).cuda()
    wtd = torch.from_numpy(wt).cuda()
    xn = torch.empty(cols, dtype=torch.float32, device="cuda")
    xs = torch.empty(cols // 64, dtype=torch.float32, device="cuda")
    y = torch.empty(rows, dtype=torch.float32, device="cuda")
    n = 20
    nodes = [abg.Node.rmsq(0, h, wtd, xn, xs)] + [abg.Node.q4mv(1 + i, w, s, b, y, cols, x=xn, xsum=xs)
                                                  for i in range(n)]
    g = abg.StageGraph(nodes, keep=[w, s, b, h, wtd, xn, xs, y])
    ms, _ = time_graph(g, stream, max(1, args.steps // 2), args.warmup, False)
    g.close()
    us = ms * 1e3 / n
    gbs = product_bytes(rows, cols) / (us * 1e-6) / 1e9
    return {"workload": "q4mv 248320x2048 output head, x = rmsq(hidden), 20 products per replay",
            "us_per_product": us, "gbs": gbs, "frac_of_measured_peak": gbs / peak}


def bench_formats(abg, stream, args, peak, l2):
    """The 4096x2048 product in each format: one grouped launch of 256 products,
    each on its own copy of the weights (the copies total many times L2)."""
    import torch

    import oracle
    out = {"workload": "q4mv 4096x2048, one grouped launch of 256 products per replay, weights from HBM"}
    for group in synth.GROUPS:
        for sb in synth.SB_TYPES:
            m, x_np = synth.fmt_case(group, sb, MID_ROWS, MID_COLS)
            sbb = 4 if sb == "f32" else 2
            pb = product_bytes(MID_ROWS, MID_COLS, group, sbb)
            copies = max(GROUP, math.ceil(3 * l2 / m.nbytes))
            w = torch.from_numpy(m.w.view(np.int32)).cuda()
            sc = torch.from_numpy(m.scale.view(np.int16) if sbb == 2 else m.scale).cuda()
            bi = torch.from_numpy(m.bias.view(np.int16) if sbb == 2 else m.bias).cuda()
            mats = [(w.clone(), sc.clone(), bi.clone()) for _ in range(copies)]
            x = torch.from_numpy(x_np).cuda()
            xs = torch.empty(MID_COLS // group, dtype=torch.float32, device="cuda")
            ys = [torch.empty(MID_ROWS, dtype=torch.float32, device="cuda") for _ in range(GROUP)]
            abg.gsum(x, xs, group=group)
            g = abg.StageGraph([abg.Node.q4mv(0, *mats[i % copies], ys[i], MID_COLS, x=x, xsum=xs, group=group,
                                              sb_type=sb) for i in range(GROUP)], keep=[x, xs] + ys)
            ms, _ = time_graph(g, stream, max(args.steps, 10), args.warmup, False)
            g.close()
            got = oracle.hash32(ys[GROUP - 1].cpu().numpy())
            exp = oracle.hash32(oracle.q4mv_ex(*m.arrays(), sb, group, x_np, oracle.gsum_ex(x_np, group), MID_COLS))
            if got != exp:
                raise SystemExit(f"format g{group} {sb}: hash {got} differs from the oracle's {exp}")
            us = ms * 1e3 / GROUP
            gbs = GROUP * pb / (ms * 1e-3) / 1e9
            out[f"g{group}_{sb}"] = {"us_per_product": round(us, 3), "gbs": round(gbs, 1),
                                     "frac_of_measured_peak": round(gbs / peak, 3), "bytes_per_product": pb}
            del mats, g, w, sc, bi
            torch.cuda.empty_cache()
    return out


def bench_batched(abg, stream, args):
    """The 248320x2048 head for a batch of T tokens (abg_q4mm): us per call and per
    token; every row of every token checked against the oracle."""
    import torch

    import oracle
    m, _, _ = synth.head()
    w = torch.from_numpy(m.w.view(np.int32)).cuda()
    s = torch.from_numpy(m.scale).cuda()
    b = torch.from_numpy(m.bias).cuda()
    pb = product_bytes(m.rows, m.cols)
    out = {"workload": "q4mm 248320x2048 head, T tokens per call (four or two tokens share a launch)"}
    for T in (1, 2, 4, 8):
        rng = np.random.default_rng([6, T])
        X_np = np.stack([synth.activations(rng, m.cols) for _ in range(T)])
        XS_np = np.stack([oracle.gsum(x) for x in X_np])
        X = torch.from_numpy(X_np).cuda()
        XS = torch.from_numpy(XS_np).cuda()
        Y = torch.empty(T * m.rows, dtype=torch.float32, device="cuda")
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                abg.q4mm(w, s, b, X, XS, Y, cols=m.cols, stream=stream)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            reps = max(3, args.steps // 2)
            for _ in range(reps):
                abg.q4mm(w, s, b, X, XS, Y, cols=m.cols, stream=stream)
            e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / reps
        got = Y.view(T, m.rows).cpu().numpy()
        exp = oracle.q4mm(*m.arrays(), X_np, XS_np, m.cols)
        if not np.array_equal(got.view(np.uint32), exp.view(np.uint32)):
            raise SystemExit(f"batched product T={T} differs from the oracle")
        out[f"T{T}"] = {"us_per_call": round(us, 2), "us_per_token": round(us / T, 2),
                        "token_gbs": round(T * pb / (us * 1e-6) / 1e9, 1)}
    del w, s, b
    torch.cuda.empty_cache()
    return out


SWEEP_ROWS = (512, 2048, 4096, 6144, 16384, 65536, 248320)
SWEEP_COLS = (2048, 4096, 6144)


def bench_sweep(abg, stream, args, peak, l2):
    """Every (rows, cols) point of the sweep, each rows-per-item setting, tree and
    fast mode: products queued as one stage over copies of the weights totalling
    more than 3x L2.  Also the fast-mode error over every row of each point,
    against the tree result: the largest |y_fast - y_tree| / A_r (A_r = sum over
    groups of |scale*d| + |bias*xsum|, the stated bound's scale), the largest
    |y_fast - y_tree| / |y_tree| over all rows, and the same over rows with
    |y_tree| >= 1e-3 A_r."""
    import torch

    import oracle
    out = {"workload": "sweep: seed [4, rows, cols]; products queued as one stage, weights > 3x L2", "points": []}
    for cols in SWEEP_COLS:
        for rows in SWEEP_ROWS:
            m, x_np = synth.sweep_point(rows, cols)
            pb = product_bytes(rows, cols)
            copies = int(min(600, max(2, math.ceil(3 * l2 / m.nbytes))))
            w = torch.from_numpy(m.w.view(np.int32)).cuda()
            sc = torch.from_numpy(m.scale).cuda()
            bi = torch.from_numpy(m.bias).cuda()
            mats = [(w.clone(), sc.clone(), bi.clone()) for _ in range(copies)]
            del w, sc, bi
            x = torch.from_numpy(x_np).cuda()
            xs = torch.empty(cols // 64, dtype=torch.float32, device="cuda")
            abg.gsum(x, xs)
            calls = max(copies, 8)
            ys = [torch.empty(rows, dtype=torch.float32, device="cuda") for _ in range(calls)]
            point = {"rows": rows, "cols": cols, "copies": copies}
            y_tree = y_fast = None
            for mode, mname in ((abg.TREE, "tree"), (abg.FAST, "fast")):
                for R in (1, 2, 4, 8):
                    g = abg.StageGraph([abg.Node.q4mv(0, *mats[i % copies], ys[i % len(ys)], cols, x=x, xsum=xs)
                                        for i in range(calls)], mode=mode, rows_per_warp=R, keep=[x, xs] + ys)
                    ms, _ = time_graph(g, stream, 3, 1, False)
                    g.close()
                    gbs = calls * pb / (ms * 1e-3) / 1e9
                    point[f"{mname}_R{R}_gbs"] = round(gbs, 1)
                    point[f"{mname}_R{R}_frac"] = round(gbs / peak, 3)
                    if R == 8:
                        y8 = ys[(calls - 1) % len(ys)].cpu().numpy().copy()
                        if mname == "tree":
                            y_tree = y8
                        else:
                            y_fast = y8
            xs_np = oracle.gsum(x_np)
            if oracle.hash32(y_tree) != oracle.hash32(oracle.q4mv(*m.arrays(), x_np, xs_np, cols)):
                raise SystemExit(f"sweep {rows}x{cols}: tree mode differs from the oracle")
            mag = oracle.q4mv_absmag(*m.arrays(), x_np, xs_np, cols)
            yt, yf = y_tree.astype(np.float64), y_fast.astype(np.float64)
            d = np.abs(yf - yt)
            nz = yt != 0
            keep = np.abs(yt) >= 1e-3 * mag
            point["fast_max_err_over_A"] = float(np.max(d / mag))
            point["fast_max_rel_err_all_rows"] = float(np.max(d[nz] / np.abs(yt[nz]))) if nz.any() else 0.0
            point["fast_max_rel_err"] = float(np.max(d[keep] / np.abs(yt[keep]))) if keep.any() else 0.0
            point["fast_rows_over_1e-5_rel"] = int(np.count_nonzero(d > 1e-5 * np.abs(yt)))
            out["points"].append(point)
            del mats, ys, x, xs
            torch.cuda.empty_cache()
    return out


def bench_pages_way(abg, stream, args):
    """The pages' timing of the 4096x2048 product: (400-call - 1-call) / 400, rounds
    alternating, median of 6, calls back to back on one stream, each call of a
    round on its own copy of the weights."""
    import torch
    m, x_np = synth.mid()
    l2 = getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 126 * 2 ** 20)
    copies = max(CALLS, math.ceil(3 * l2 / m.nbytes))
    mats = rotating_copies(m, copies)
    x = torch.from_numpy(x_np).cuda()
    xs = torch.empty(MID_COLS // 64, dtype=torch.float32, device="cuda")
    abg.gsum(x, xs)
    y = torch.empty(MID_ROWS, dtype=torch.float32, device="cuda")

    def run(n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(n):
            abg.q4mv(*mats[i % copies], x, xs, y, cols=MID_COLS, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    run(20)
    per = []
    for _ in range(6):
        t400 = run(CALLS)
        t1 = run(1)
        per.append((t400 - t1) / CALLS)
    us = statistics.median(per) * 1e3
    del mats
    torch.cuda.empty_cache()
    return {"workload": "4096x2048, 400 single-call launches back to back, (400-call - 1-call)/400, median of 6",
            "us_per_call": round(us, 3), "gbs": round(product_bytes(MID_ROWS, MID_COLS) / (us * 1e-6) / 1e9, 1)}


def time_calls_graph(fn, count: int, replays: int = 5) -> float:
    """us per call of `count` calls of fn(i, stream) captured in one CUDA graph
    (so the host's per-call cost is not timed), median over replays."""
    import torch
    cs = torch.cuda.Stream()
    cs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cs):
        fn(0, cs)  # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cs):
        for i in range(count):
            fn(i, cs)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    times = []
    for _ in range(replays):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(cs)
        with torch.cuda.stream(cs):
            g.replay()
        e1.record(cs)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) * 1e3 / count)
    del g
    return statistics.median(times)


def bench_gdn(abg, stream, args):
    """One token of the gated DeltaNet mixer (abg_gdn), 16 heads of 128 columns,
    4 conv taps: calls captured in a CUDA graph (the host's per-call cost not
    timed), each on its own copy of the state (S and the conv state rotate over
    copies totalling more than L2), us per token; the first call's outputs
    checked bit for bit against the oracle."""
    import torch

    import oracle
    c = synth.gdn_case(np.random.default_rng(21))
    H, D, K = c["S"].shape[0], c["S"].shape[1], c["conv"].shape[1]
    d = {k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in c.items()}
    l2 = getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 126 * 2 ** 20)
    copies = max(2, math.ceil(1.5 * l2 / (c["S"].nbytes + c["state"].nbytes)))
    Ss = [d["S"].clone() for _ in range(copies)]
    sts = [d["state"].clone() for _ in range(copies)]
    y = torch.empty(H * D, dtype=torch.float32, device="cuda")
    ys = torch.empty(H * D // 64, dtype=torch.float32, device="cuda")
    args_of = lambda i: (d["x"], d["conv"], sts[i], d["a"], d["b"], d["z"], d["A_log"], d["dt_bias"], d["nw"], Ss[i])
    abg.gdn(*args_of(0), y, ys, stream=stream)
    torch.cuda.synchronize()
    ey, eys, eS, est = oracle.gdn(**c)
    same = (np.array_equal(y.cpu().numpy().view(np.uint32), ey.view(np.uint32))
            and np.array_equal(ys.cpu().numpy().view(np.uint32), eys.view(np.uint32))
            and np.array_equal(Ss[0].cpu().numpy().view(np.uint32), eS.view(np.uint32))
            and np.array_equal(sts[0].cpu().numpy().view(np.uint32), est.view(np.uint32)))
    if not same:
        raise SystemExit("gdn differs from the oracle")
    us = time_calls_graph(lambda i, st: abg.gdn(*args_of(i % copies), y, ys, stream=st), 200)
    # algorithmic bytes: S and the conv state read and written once, x, conv,
    # z, the per-head scalars and the norm weights read, y and ysum written
    nbytes = 2 * c["S"].nbytes + 2 * c["state"].nbytes + c["x"].nbytes + c["conv"].nbytes + c["z"].nbytes + \
        4 * 4 * H + c["nw"].nbytes + 4 * H * D + 4 * H * D // 64
    del Ss, sts
    torch.cuda.empty_cache()
    return {"workload": f"gdn mixer, one token: {H} heads x {D} columns, {K} conv taps; state rotating over "
                        f"{copies} copies (> L2); 200 calls captured in one CUDA graph, median of 5 replays",
            "us_per_token": round(us, 3), "bytes_per_token": int(nbytes),
            "gbs": round(nbytes / (us * 1e-6) / 1e9, 1), "bit_exact": True}


def bench_atq(abg, stream, args):
    """One token of gated attention (abg_atq): 8 query heads over 2 key/value
    heads of 256 columns at position 2047 of 4096-row caches; calls captured in
    a CUDA graph, the caches rotating over copies larger than L2; us per token;
    the first call's outputs checked bit for bit against the oracle."""
    import torch

    import oracle
    c = synth.atq_case(np.random.default_rng(22))
    Hkv, P, D = c["Kc"].shape
    Hq, pos = c["q"].size // D, c["pos"]
    d = {k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in c.items() if k != "pos"}
    l2 = getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 126 * 2 ** 20)
    copies = max(2, math.ceil(1.5 * l2 / (2 * c["Kc"].nbytes)))
    Ks = [d["Kc"].clone() for _ in range(copies)]
    Vs = [d["Vc"].clone() for _ in range(copies)]
    y = torch.empty(Hq * D, dtype=torch.float32, device="cuda")
    ys = torch.empty(Hq * D // 64, dtype=torch.float32, device="cuda")
    args_of = lambda i: (d["q"], d["gate"], d["k"], d["v"], d["qn_w"], d["kn_w"], d["cos"], d["sin"], Ks[i], Vs[i])
    abg.atq(*args_of(0), y, ys, pos=pos, stream=stream)
    torch.cuda.synchronize()
    ey, eys, eK, eV = oracle.atq(**c)
    same = (np.array_equal(y.cpu().numpy().view(np.uint32), ey.view(np.uint32))
            and np.array_equal(ys.cpu().numpy().view(np.uint32), eys.view(np.uint32))
            and np.array_equal(Ks[0].cpu().numpy().view(np.uint32), eK.view(np.uint32))
            and np.array_equal(Vs[0].cpu().numpy().view(np.uint32), eV.view(np.uint32)))
    if not same:
        raise SystemExit("atq differs from the oracle")
    us = time_calls_graph(lambda i, st: abg.atq(*args_of(i % copies), y, ys, pos=pos, stream=st), 100)
    # algorithmic bytes: the caches' rows 0..pos read once (each group's rows
    # serve its query heads), one row of each written, the vectors
    nbytes = 2 * Hkv * (pos + 1) * D * 4 + 2 * Hkv * D * 4 + (2 * Hq + 2 * Hkv) * D * 4 + 2 * D * 4 + \
        D * 4 + Hq * D * 4 + Hq * D // 16
    del Ks, Vs
    torch.cuda.empty_cache()
    return {"workload": f"atq, one token: {Hq} query heads over {Hkv} kv heads x {D} columns at position {pos} of "
                        f"{P}-row caches; caches rotating over {copies} copies (> L2); 100 calls captured in one "
                        "CUDA graph, median of 5 replays",
            "us_per_token": round(us, 3), "bytes_per_token": int(nbytes),
            "gbs": round(nbytes / (us * 1e-6) / 1e9, 1), "bit_exact": True}


def bench_decode(abg, decode, stream, args):
    import torch
    model, h = synth.decode_model()
    dm = decode.DeviceModel.upload(model)
    del model
    h0 = torch.from_numpy(h).cuda()
    out = {"workload": "24 layers, hidden 2048, MLP 6144, 248320-row head; 169 products",
           "product_bytes": dm.product_bytes}
    for fused in (True, False):
        g, _ = decode.decode_token_graph(dm, h0, fused=fused)
        ms, _ = time_graph(g, stream, 50, 5, False)
        # wall time of launch + one sync, per token: median of 50 replays
        walls = []
        for _ in range(50):
            t0 = time.perf_counter()
            g.launch(stream)
            stream.synchronize()
            walls.append((time.perf_counter() - t0) * 1e3)
        key = "fused" if fused else "unfused"
        out[key] = {"gpu_ms_per_token": ms, "wall_ms_per_token": statistics.median(walls), "launches": g.launches,
                    "gbs": dm.product_bytes / (ms * 1e-3) / 1e9}
        g.close()
    # end to end: the fused token as one graph that copies the hidden vector in
    # from pinned host memory and the logits back out; wall time of launch +
    # one sync, median of 50 replays; the host logits checked against a replay
    # of the graph without copies
    h_host = torch.from_numpy(h).pin_memory()
    logits_host = torch.empty(dm.head.rows, dtype=torch.float32).pin_memory()
    h_dev = torch.empty_like(h0)
    g, o = decode.decode_token_graph(dm, h_dev, fused=True, host_io=(h_host, logits_host))
    walls = []
    for i in range(55):
        t0 = time.perf_counter()
        g.launch(stream)
        stream.synchronize()
        if i >= 5:
            walls.append((time.perf_counter() - t0) * 1e3)
    g.close()
    g2, o2 = decode.decode_token_graph(dm, h0, fused=True)
    g2.launch(stream)
    stream.synchronize()
    if not torch.equal(o2["logits"].cpu(), logits_host):
        raise SystemExit("the decode token's host logits differ from its device logits")
    g2.close()
    out["e2e"] = {"wall_ms_per_token": statistics.median(walls), "h2d_bytes": 4 * h.size,
                  "d2h_bytes": 4 * dm.head.rows}
    return out


def cpu_baseline(seconds: float = 10.0):
    """The oracle (plain C, one thread) on the 4096x2048 product, repeated for about `seconds`."""
    import oracle
    m, x = synth.mid()
    xs = oracle.gsum(x)
    oracle.q4mv(*m.arrays(), x, xs, MID_COLS)
    n, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        oracle.q4mv(*m.arrays(), x, xs, MID_COLS)
        n += 1
    dt = time.perf_counter() - t0
    return {"value": n * product_bytes(MID_ROWS, MID_COLS) / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} calls of the 4096x2048 product (single-threaded C oracle, {dt:.1f} s)"}


def _oracle_rows_worker(job):
    """One host process of the all-cores baseline: rows [r0, r1) of the 4096x2048
    product, repeated for `seconds`; returns (calls, rows per call)."""
    r0, r1, seconds = job
    import oracle
    m, x = synth.mid()
    xs = oracle.gsum(x)
    oracle.q4mv(*m.arrays(), x, xs, MID_COLS, row0=r0, n=r1 - r0)
    n, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        oracle.q4mv(*m.arrays(), x, xs, MID_COLS, row0=r0, n=r1 - r0)
        n += 1
    return n, r1 - r0, time.perf_counter() - t0


def cpu_all_cores(seconds: float = 10.0):
    """The same oracle on every host core: one spawned process per core, each on its
    own slice of the rows (the oracle itself is single-threaded C)."""
    import multiprocessing as mp
    cores = os.cpu_count() or 1
    bounds = [(MID_ROWS * i // cores, MID_ROWS * (i + 1) // cores, seconds) for i in range(cores)]
    with mp.get_context("spawn").Pool(cores) as pool:
        res = pool.map(_oracle_rows_worker, bounds)
    dt = max(r[2] for r in res)
    total = sum(n * product_bytes(rows, MID_COLS) for n, rows, _ in res)
    return {"value": total / dt / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"4096x2048 product, rows split over {cores} processes, {dt:.1f} s"}


def run_reference(args):
    """The oracle as the reference arm: each step is a bounded sample of the workload on the host."""
    import oracle
    m, x = synth.mid()
    xs = oracle.gsum(x)
    per_step = 20
    for _ in range(args.warmup):
        oracle.q4mv(*m.arrays(), x, xs, MID_COLS)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        xs = oracle.gsum(x)
        for _ in range(per_step):
            oracle.q4mv(*m.arrays(), x, xs, MID_COLS)
    dt = (time.perf_counter() - t0) / args.steps
    value = per_step * product_bytes(MID_ROWS, MID_COLS) / dt / 1e9
    sample = f"{per_step} of the step's {CALLS} products per step (single-threaded C oracle)"
    return {"metric": "q4mv achieved HBM GB/s", "value": value, "unit": "GB/s", "impl": "reference", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": config_dict(),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def config_dict(copies=None):
    return {"workload": "q4mv mid: 4096x2048, 400 calls queued as one stage per step (+ group sums of x), seed 1",
            "rows": MID_ROWS, "cols": MID_COLS, "calls_per_step": CALLS, "mode": "tree",
            "l2": f"inputs larger than L2: weights rotate over {copies} device copies" if copies else None,
            "parallelism": "replicas"}


def max_over_ranks(ms: float, world: int, device: str) -> float:
    """The slowest rank's step time (replicas run the same work; the job is as
    fast as its slowest replica).  Ends with a barrier."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.barrier()
    return float(t.item())


def job_value(ms_step: float, world: int) -> float:
    """Whole-job GB/s: every replica streams one step's products per step."""
    return world * CALLS * product_bytes(MID_ROWS, MID_COLS) / (ms_step * 1e-3) / 1e9


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extra", action="store_true", help="skip the head and decode-token measurements")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--only", choices=["head", "decode", "formats", "batched", "sweep", "pages_way", "gdn", "atq"],
                    default=None,
                    help="run one secondary workload alone and print its numbers (for profiling)")
    args = ap.parse_args()
    if args.only:
        import torch

        import affine_bit_group_gb300 as abg
        from affine_bit_group_gb300 import decode
        stream = torch.cuda.Stream()
        peak, _ = measured_peak()
        if args.only == "head":
            out = bench_head(abg, stream, args, peak)
        elif args.only == "decode":
            out = bench_decode(abg, decode, stream, args)
        elif args.only == "batched":
            out = bench_batched(abg, stream, args)
        elif args.only == "gdn":
            out = bench_gdn(abg, stream, args)
        elif args.only == "atq":
            out = bench_atq(abg, stream, args)
        elif args.only == "pages_way":
            out = bench_pages_way(abg, stream, args)
        elif args.only == "sweep":
            l2 = getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 126 * 2 ** 20)
            out = bench_sweep(abg, stream, args, peak, l2)
        else:
            l2 = getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 126 * 2 ** 20)
            out = bench_formats(abg, stream, args, peak, l2)
        print(json.dumps(out), flush=True)
        return
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if os.environ.get("ABG_BENCH_BACKEND") != "gloo" else "gloo")
    res = run_ours(args, rank, world)
    ms_step = max_over_ranks(res["ms_step"], world, "cuda")
    if rank != 0:
        return
    value = job_value(ms_step, world)
    traffic = profile_traffic("q4mv_mid_4096x2048.md")
    line = {
        "metric": "q4mv achieved HBM GB/s", "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": config_dict(res["copies"]),
        "us_per_product": res["us_per_product"],
        "frac_of_peak": {"measured": res["value"] / res["peak"], "nominal_8tbs": res["value"] / 8000.0},
        "hash32": res["hash"],
        "roofline": {"bound": "hbm", "achieved": res["achieved"], "peak": res["peak"], "unit": "GB/s",
                     "frac": res["achieved"] / res["peak"], "traffic": traffic, "peak_kind": res["peak_kind"],
                     "kernel": "q4mv_kernel<8,tree,bulk scale/bias>: one launch of 256 products of 4096x2048",
                     "bytes_per_launch": GROUP * product_bytes(MID_ROWS, MID_COLS),
                     "launch_us": res["launch_us"]},
        "clocks": res["clocks"], "e2e": res["e2e"], "gpu_launches": res["launches"], "extra": res["extra"],
    }
    if not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline()
        line["extra"]["cpu_all_cores"] = cpu_all_cores()
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
