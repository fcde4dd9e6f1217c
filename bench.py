#!/usr/bin/env python
"""Benchmark: emulated DGEMM TFLOP/s (2MNK/t) and % of FP4 roofline on one GB300.

One step = one pass of the whole hot path over one synthetic problem held in
HBM: deconstruction of A's rows and B's columns (scale, round, residues, FP4
limb planes), the FP4 limb GEMM with modular recombination, and the CRT +
scale back to fp64.  The default workload is M = N = K = 8192 with entries
u 2^e (u ~ U(-1, 1), e uniform in [-10, 10]) and r = 13 moduli.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on bounded samples

Under torchrun every rank runs its own replica (the problems are independent:
weak scaling, no data-path collective); rank 0 prints one JSON line.
"""

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import WORKLOADS, make_pair  # noqa: E402

METRIC = "emulated DGEMM TFLOP/s (2MNK/t) and % of FP4 roofline at 1 GB300"
FP4_OVER_BF16 = 13.5 / 2.25  # nominal dense FP4 : BF16 tensor ratio on GB300
NARROW_MAX_K = 1 << 24       # k limit of the fused narrow path
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
CPU_SAMPLE = 128        # sampled rows and columns of C per oracle step
CPU_MIN_SECONDS = 10.0  # bounded CPU baseline: repeat the sample at least this long


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ozemu", choices=["ozemu", "reference"])
    ap.add_argument("--workload", default="dgemm_8192_wide", choices=sorted(WORKLOADS))
    ap.add_argument("--r", type=int, default=None, help="override the number of moduli")
    ap.add_argument("--m", type=int, default=None, help="override M (same distribution and seed)")
    ap.add_argument("--n", type=int, default=None, help="override N")
    ap.add_argument("--k", type=int, default=None, help="override K")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-native", action="store_true")
    ap.add_argument("--no-compare", action="store_true", help="skip the INT8 residue-GEMM comparison")
    ap.add_argument("--no-igemm", action="store_true", help="skip the exact INT8 product leg (4096^3)")
    ap.add_argument("--no-two-limb", action="store_true", help="skip the two-limb moduli leg")
    ap.add_argument("--chunks", type=int, default=4,
                    help="row chunks of A in the timed step (1: the stages one after another)")
    return ap.parse_args()


ACC_SAMPLE = 24  # sampled entries of C for the exact error measurement


def bound_ratios(A_h, B_h, rows, cols, results):
    """max over sampled entries (i, j) of |C_ij - (AB)_ij| / (2 K 2^-53 (|A||B|)_ij)
    for each named result (arrays of the sampled entries), with the exact
    product (AB)_ij summed in rationals (every fp64 value is a dyadic
    rational, so the sum is exact)."""
    from fractions import Fraction
    k = A_h.shape[1]
    out = {name: 0.0 for name in results}
    for e, (i, j) in enumerate(zip(rows, cols)):
        a = A_h[i]
        b = B_h[:, j]
        exact = sum((Fraction(float(x)) * Fraction(float(y)) for x, y in zip(a, b)), Fraction(0))
        scale = 2.0 * k * 2.0 ** -53 * float(np.abs(a) @ np.abs(b))
        for name, vals in results.items():
            err = abs(Fraction(float(vals[e])) - exact)
            if scale > 0:
                out[name] = max(out[name], float(err) / scale)
    return out


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def max_over_ranks(x, dist, device):
    """Max of a float across all ranks (plain value when not distributed)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world_size, flop_per_step, steps, elapsed_ms):
    """Units all ranks processed over the slowest rank's time, in TFLOP/s."""
    return world_size * flop_per_step * steps / (elapsed_ms / 1e3) / 1e12


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        loaded = [s for s in sm if mx and s > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------- CPU oracle

CPU_SNIPPET = r"""
import json, sys, time
sys.path.insert(0, {root!r})
import numpy as np
import oracle
from workloads import WORKLOADS, make_pair, sample_indices
spec = dict(WORKLOADS[{name!r}]); spec.update({shape!r})
A, B = make_pair(spec["m"], spec["n"], spec["k"], spec["seed"], spec["dist"])
r = {r}
n_rows = min({ns}, spec["m"]); n_cols = min({ns}, spec["n"])
steps, total, t0 = 0, 0.0, time.time()
while True:
    rows = sample_indices(spec["m"], n_rows, seed=100 + steps)
    cols = sample_indices(spec["n"], n_cols, seed=200 + steps)
    t = time.time()
    oracle.dgemm_block(A, B, r, rows=rows, cols=cols)
    total += time.time() - t
    steps += 1
    if (({max_steps} and steps >= {max_steps}) or (not {max_steps} and total >= {min_s})):
        break
print(json.dumps(dict(seconds=total, steps=steps, rows=n_rows, cols=n_cols, k=spec["k"])))
"""


def cpu_oracle(name, r, min_seconds, max_steps=0, sample=CPU_SAMPLE, shape=None):
    """Times the oracle on bounded samples in a single-threaded subprocess."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = CPU_SNIPPET.format(root=ROOT, name=name, r=r, ns=sample, max_steps=max_steps, min_s=min_seconds,
                              shape=dict(shape or {}))
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=3600)
    if out.returncode != 0:
        raise RuntimeError(out.stderr[-2000:])
    d = json.loads(out.stdout.strip().splitlines()[-1])
    flops = 2.0 * d["rows"] * d["cols"] * d["k"] * d["steps"]
    d["tflops"] = flops / d["seconds"] / 1e12
    return d


# ------------------------------------------------------------------ GPU arm

def kernel_traffic(workload, chunks, bblocks):
    """DRAM bytes per launch of the limb GEMM from the committed ncu record,
    used only for the workload and row chunking it was captured on and only
    while the kernel sources are unchanged since the capture."""
    path = os.path.join(ROOT, "profiles", "limb_gemm_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    h = hashlib.sha256()
    for fn in ("gemm_fp4.cu", "common.cuh"):
        with open(os.path.join(ROOT, "ozaki_ii_fp64_gb300", "csrc", fn), "rb") as f:
            h.update(f.read())
    if d.get("source_sha256") != h.hexdigest() or d.get("workload") != workload or d.get("chunks") != chunks or d.get("b_blocks") != bblocks:
        return None
    return d


def gemm_kernel_name(n, k):
    """The limb-GEMM kernel the library picks for a residue product."""
    pair = n > 64 and os.environ.get("OZEMU_GEMM_PAIR", "1") != "0"
    if pair:
        return "limb_gemm_pair_kernel (CTA pair, 256x224 tiles)"
    bn = 16 if n <= 16 else 32 if n <= 32 else 64 if n <= 64 else 128
    return "limb_gemm_kernel<%d, residue> (one CTA, 128x%d tiles)" % (bn, bn)


def workload_name(args, spec):
    base = WORKLOADS[args.workload]
    if all(spec[x] == base[x] for x in ("m", "n", "k")):
        return args.workload
    return "%s@%dx%dx%d" % (args.workload, spec["m"], spec["n"], spec["k"])


def run_gpu(args):
    import torch
    import torch.distributed as dist
    import ozaki_ii_fp64_gb300 as oz

    ws, rank, local = dist_env()
    if ws > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", init_method="env://")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    oz.load()

    spec = dict(WORKLOADS[args.workload])
    for key in ("m", "n", "k"):
        if getattr(args, key):
            spec[key] = getattr(args, key)
    A_h, B_h = make_pair(spec["m"], spec["n"], spec["k"], spec["seed"], spec["dist"])
    if spec["kind"] != "dgemm":
        raise SystemExit("bench.py times the emulated DGEMM workloads")
    m, n, k = spec["m"], spec["n"], spec["k"]
    r = args.r or spec["r"]
    pA, pB = oz.ozemu_bit_budget(k, r)
    A = torch.from_numpy(A_h).to(dev)
    B = torch.from_numpy(B_h).to(dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    # Preallocated stage buffers: nothing is allocated in the timed region.
    ap = torch.empty(oz.ozemu_plane_bytes(m, k, r), dtype=torch.uint8, device=dev)
    bp = torch.empty(oz.ozemu_plane_bytes(n, k, r), dtype=torch.uint8, device=dev)
    sa = torch.empty(m, dtype=torch.int32, device=dev)
    sb = torch.empty(n, dtype=torch.int32, device=dev)
    res = torch.empty(oz.ozemu_residue_bytes(m, n, r), dtype=torch.uint8, device=dev)
    C = torch.empty((m, n), dtype=torch.float64, device=dev)
    # n <= ozemu_narrow_max_n(): the library's fused narrow path (what
    # ozemu_dgemm runs for such shapes); otherwise the limb-plane path.
    narrow = n <= oz.ozemu_narrow_max_n() and k <= NARROW_MAX_K and os.environ.get("OZEMU_NARROW", "1") != "0"

    def check(st, what):
        if st != 0:
            raise oz.OzemuError(st, what)

    def split_a():
        check(oz.ozemu_split_rows_f64(m, k, A.data_ptr(), k, pA, r, ap.data_ptr(), sa.data_ptr(), sh), "split A")

    def split_b():
        check(oz.ozemu_split_cols_f64(k, n, B.data_ptr(), n, pB, r, bp.data_ptr(), sb.data_ptr(), sh), "split B")

    def limb_gemm():
        check(oz.ozemu_residue_gemm(m, n, k, r, ap.data_ptr(), bp.data_ptr(), res.data_ptr(), sh), "limb gemm")

    def narrow_residues():
        check(oz.ozemu_residues_narrow_f64(m, n, k, r, A.data_ptr(), k, B.data_ptr(), n, res.data_ptr(),
                                           sa.data_ptr(), sb.data_ptr(), sh), "narrow residues")

    def crt():
        check(oz.ozemu_crt_f64(m, n, r, res.data_ptr(), sa.data_ptr(), sb.data_ptr(), C.data_ptr(), n, sh), "crt")

    # The bracketed stage (ev0 .. ev1) is the step's dominant kernel.
    if narrow:
        stages = [("narrow_residues", narrow_residues), ("crt", crt)]
        dominant = "narrow_residues"
        launches_per_step = 3  # B's column residues, fused pass over A, CRT
    else:
        stages = [("split_A", split_a), ("split_B", split_b), ("limb_gemm", limb_gemm), ("crt", crt)]
        dominant = "limb_gemm"
        launches_per_step = 5  # split rows, transpose, split rows of B^T, limb GEMM, CRT

    # The timed step.  Limb-plane path: the library's device-operand schedule
    # with the stage calls, pipelined over row chunks of A on three streams --
    # B's split (main stream), each chunk's split (split stream, from the
    # start), limb GEMM (main stream, bracketed by events) and CRT (CRT
    # stream, beside the next chunk's GEMM).  Narrow path: its two calls in
    # order.
    chunks = 1 if narrow else max(1, args.chunks)
    crows = m if chunks == 1 else ((m + chunks - 1) // chunks + 255) // 256 * 256
    chunk_bufs = []
    for row0 in range(0, m, crows):
        mc = min(crows, m - row0)
        chunk_bufs.append((row0, mc, torch.empty(oz.ozemu_plane_bytes(mc, k, r), dtype=torch.uint8, device=dev),
                           torch.empty(mc, dtype=torch.int32, device=dev),
                           torch.empty(oz.ozemu_residue_bytes(mc, n, r), dtype=torch.uint8, device=dev)))
    nch = len(chunk_bufs)
    s_split = torch.cuda.Stream(dev)
    s_crt = torch.cuda.Stream(dev)
    ev_start = torch.cuda.Event()
    evA = [torch.cuda.Event() for _ in range(nch)]
    evG = [torch.cuda.Event() for _ in range(nch)]
    evC = [torch.cuda.Event() for _ in range(nch)]
    if not narrow:
        launches_per_step = 2 + 3 * nch  # transpose + split of B; per chunk split, limb GEMM, CRT
    n_dominant = 1 if narrow else nch

    def step(gev=None):
        if narrow:
            if gev is not None:
                gev[0][0].record(stream)
            narrow_residues()
            if gev is not None:
                gev[0][1].record(stream)
            crt()
            return
        ev_start.record(stream)
        s_split.wait_event(ev_start)
        s_crt.wait_event(ev_start)
        split_b()
        for c, (row0, mc, apc, sac, resc) in enumerate(chunk_bufs):
            check(oz.ozemu_split_rows_f64(mc, k, A.data_ptr() + row0 * k * 8, k, pA, r, apc.data_ptr(),
                                          sac.data_ptr(), s_split.cuda_stream), "split A chunk")
            evA[c].record(s_split)
        for c, (row0, mc, apc, sac, resc) in enumerate(chunk_bufs):
            stream.wait_event(evA[c])
            if gev is not None:
                gev[c][0].record(stream)
            check(oz.ozemu_residue_gemm(mc, n, k, r, apc.data_ptr(), bp.data_ptr(), resc.data_ptr(), sh),
                  "limb gemm chunk")
            if gev is not None:
                gev[c][1].record(stream)
            evG[c].record(stream)
            s_crt.wait_event(evG[c])
            check(oz.ozemu_crt_f64(mc, n, r, resc.data_ptr(), sac.data_ptr(), sb.data_ptr(),
                                   C.data_ptr() + row0 * n * 8, n, s_crt.cuda_stream), "crt chunk")
            evC[c].record(s_crt)
        stream.wait_event(evC[nch - 1])
    nbc = 1  # B whole (column blocks are for host operands)

    def stage_times(which):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(which) + 1)]
        evs[0].record(stream)
        for i, (_, fn) in enumerate(which):
            fn()
            evs[i + 1].record(stream)
        torch.cuda.synchronize(dev)
        return {name: evs[i].elapsed_time(evs[i + 1]) for i, (name, _) in enumerate(which)}

    if not narrow:
        # Grow the library's cached workspace to the full-width column split
        # once, so that no later call (timed or staged) reallocates it.
        split_b()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if oz.ozemu_get_status(sh) != 0:
        raise SystemExit("device status not OK after warm-up")

    # Per-stage durations (one untimed pass, for the report only).
    stage_ms = stage_times(stages)
    C_staged = C.clone()

    # Timed region.
    gev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_dominant)]
           for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    t_start.record(stream)
    for i in range(args.steps):
        step(gev[i])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    if ws > 1:
        dist.barrier()
    elapsed_ms = t_start.elapsed_time(t_end)
    dom_ms = sum(a.elapsed_time(b) for g in gev for a, b in g) / args.steps  # per step
    status = oz.ozemu_get_status(sh)
    if status != 0:
        raise SystemExit("device status %d after the timed region" % status)
    if not torch.equal(C.view(torch.int64), C_staged.view(torch.int64)):
        raise SystemExit("the timed step's result differs from the stages run one after another")
    elapsed_ms = max_over_ranks(elapsed_ms, dist if ws > 1 else None, dev)

    ms_per_step = elapsed_ms / args.steps
    flop = 2.0 * m * n * k
    value = whole_job_tflops(ws, flop, args.steps, elapsed_ms)

    pk, pk_kind = peaks()
    fp4_peak = pk["bf16_tflops"] * FP4_OVER_BF16  # TFLOP/s, burst
    fp4_flop = 9.0 * r * flop
    if narrow:
        # HBM-bound: A and B read once, residues written once.
        kbytes = 8.0 * (m * k + k * n) + r * m * n
        achieved = kbytes / (dom_ms / 1e3) / 1e9
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": round(pk["hbm_gbs"], 1),
                    "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 4), "traffic": None,
                    "kernel": "dgemv_fused_kernel (fused deconstruction + product, narrow B)",
                    "peak_source": "%s HBM copy bandwidth" % pk_kind,
                    "algorithmic": "8 (mk + kn) + r m n bytes per launch"}
        bytes_alg = 8.0 * (m * k + k * n + m * n)
        t_roof = bytes_alg / (pk["hbm_gbs"] * 1e9)
    else:
        achieved = fp4_flop / (dom_ms / 1e3) / 1e12
        tr = kernel_traffic(workload_name(args, spec), nch, nbc)
        roofline = {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(fp4_peak, 1),
                    "unit": "TFLOP/s", "frac": round(achieved / fp4_peak, 4),
                    "traffic": (int(tr["bytes_per_launch"]) if tr else None),
                    "kernel": gemm_kernel_name(n, k),
                    "peak_source": "%s bf16 burst x %.0f (nominal FP4:BF16)" % (pk_kind, FP4_OVER_BF16),
                    "algorithmic": "9 r 2MNK FP4 flop per launch"}
        # Whole-step roofline: the slower of the FP4 term and the algorithmic
        # bytes at HBM peak.  K1 reads 8 B and writes 1.5 r B per input
        # element, K2 reads the planes once (1.5 r B per input element) and
        # writes r B per output, K3 reads r B and writes 8 B per output.
        bytes_alg = (m * k + k * n) * (8 + 3.0 * r) + m * n * (2.0 * r + 8)
        t_roof = max(fp4_flop / (fp4_peak * 1e12), bytes_alg / (pk["hbm_gbs"] * 1e9))
    pct_roof = 100.0 * t_roof / (ms_per_step / 1e3)

    line = {"metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_name(args, spec), "m": m, "n": n, "k": k, "r": r, "dist": spec["dist"],
                       "seed": spec["seed"], "path": "narrow (fused)" if narrow else "limb planes",
                       "row_chunks": nch, "b_column_blocks": nbc,
                       "l2": "inputs larger than L2 (%d MiB per operand), no flush" % (m * k * 8 >> 20)},
            "pct_fp4_roofline" if not narrow else "pct_io_roofline": round(pct_roof, 2), "roofline": roofline,
            "stage_ms": {kk: round(v, 3) for kk, v in stage_ms.items()},
            "gpu_launches": launches_per_step * args.steps, "clocks": clk}

    # The memory-bound stages alone (limb-plane path): median of repeated
    # launches, each after a write of 256 MiB (more than L2), against the
    # algorithmic bytes.  Deconstruction reads 8 B and writes 1.5 r B per input
    # element (B's transpose is extra traffic of this implementation, not in
    # the count); the CRT reads r B and writes 8 B per output.
    if not narrow:
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

        def median_ms(fn, reps=9):
            ts = []
            for _ in range(reps):
                with torch.cuda.stream(stream):
                    flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                torch.cuda.synchronize(dev)
                ts.append(e0.elapsed_time(e1))
            return statistics.median(ts)

        def mem_entry(name, fn, nbytes):
            t = median_ms(fn)
            gbs = nbytes / (t / 1e3) / 1e9
            return {"kernel": name, "ms": round(t, 4), "algorithmic_bytes": int(nbytes), "achieved": round(gbs, 1),
                    "peak": round(pk["hbm_gbs"], 1), "unit": "GB/s", "frac": round(gbs / pk["hbm_gbs"], 4)}

        line["memory_stages"] = {
            "deconstruct_A": mem_entry("split_rows_f64_kernel", split_a, (8.0 + 1.5 * r) * m * k),
            "deconstruct_B": mem_entry("transpose + split_rows_f64_kernel", split_b, (8.0 + 1.5 * r) * k * n),
            "reconstruct": mem_entry("crt_kernel", crt, (r + 8.0) * m * n)}
        del flush

    # The limb-plane path on the same narrow problem, for comparison.
    plane_stages = [("split_A", split_a), ("split_B", split_b), ("limb_gemm", limb_gemm), ("crt", crt)]
    if narrow:
        C_narrow = C.clone()
        stage_times(plane_stages)
        pl = stage_times(plane_stages)
        if not torch.equal(C.view(torch.int64), C_narrow.view(torch.int64)):
            raise SystemExit("narrow and limb-plane paths differ")
        line["limb_plane_path"] = {"stage_ms": {kk: round(v, 3) for kk, v in pl.items()},
                                   "ms_per_step": round(sum(pl.values()), 3),
                                   "narrow_speedup": round(sum(pl.values()) / ms_per_step, 2)}
        gemm_ms = pl["limb_gemm"]
    else:
        gemm_ms = dom_ms

    # End to end through the C ABI with host buffers: ozemu_dgemm_host copies
    # A and B in from pinned memory and C out, every step (pipelined with the
    # work inside the library).
    if not args.no_e2e:
        A_pin = torch.from_numpy(A_h).pin_memory()
        B_pin = torch.from_numpy(B_h).pin_memory()
        C_pin = torch.empty((m, n), dtype=torch.float64).pin_memory()

        def e2e_step():
            check(oz.ozemu_dgemm_host(m, n, k, A_pin.data_ptr(), k, B_pin.data_ptr(), n, C_pin.data_ptr(), n, r,
                                      sh), "dgemm_host")

        for _ in range(max(1, args.warmup)):
            e2e_step()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e_steps = max(1, min(args.steps, 5))
        e0.record(stream)
        for _ in range(e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e_ms = e0.elapsed_time(e1) / e_steps
        if oz.ozemu_get_status(sh) != 0:
            raise SystemExit("device status not OK after e2e")
        # the result must be the device-timed path's result
        if not torch.equal(C_pin.view(torch.int64), C.cpu().view(torch.int64)):
            raise SystemExit("e2e result differs from the staged result")
        line["e2e"] = {"value": round(ws * flop / (e_ms / 1e3) / 1e12, 3), "unit": "TFLOP/s",
                       "h2d_bytes_per_step": int(A_h.nbytes + B_h.nbytes), "d2h_bytes_per_step": int(m * n * 8),
                       "ms_per_step": round(e_ms, 3), "steps": e_steps}

    if not args.no_native:
        # Context: native fp64 GEMM (cuBLAS DGEMM/DGEMV via torch.matmul) on the
        # same GPU.  Warmed up on the same shape when that is cheap, median of
        # up to 5 calls.
        cheap = flop < 2e11
        if cheap:
            torch.matmul(A, B)
        else:
            torch.matmul(A[:512], B)
        torch.cuda.synchronize(dev)
        times = []
        for _ in range(5 if cheap else 1):
            n0 = torch.cuda.Event(enable_timing=True)
            n1 = torch.cuda.Event(enable_timing=True)
            n0.record(stream)
            C_native = torch.matmul(A, B)
            n1.record(stream)
            torch.cuda.synchronize(dev)
            times.append(n0.elapsed_time(n1))
        nat_ms = statistics.median(times)
        line["native_dgemm"] = {"tflops": round(flop / (nat_ms / 1e3) / 1e12, 3), "ms": round(nat_ms, 3),
                                "calls": len(times), "speedup_of_emulation": round(nat_ms / ms_per_step, 2)}

    # Accuracy on sampled entries against the exact product (rationals on the
    # host): the emulated result, native cuBLAS DGEMM and, below, the
    # two-limb result, each as a fraction of the 2 K 2^-53 |A||B| bound.
    acc_rng = np.random.default_rng(7)
    acc_rows = acc_rng.integers(0, m, size=ACC_SAMPLE)
    acc_cols = acc_rng.integers(0, n, size=ACC_SAMPLE)
    ri = torch.from_numpy(acc_rows).to(dev)
    ci = torch.from_numpy(acc_cols).to(dev)
    acc_results = {"emulated": C[ri, ci].cpu().numpy()}
    if not args.no_native:
        acc_results["native_dgemm"] = C_native[ri, ci].cpu().numpy()
        del C_native

    if not args.no_compare:
        # Comparison: the residue products as one INT8 GEMM per modulus on the
        # legacy mma.sync tensor path (the tcgen05 INT8 kind does not exist on
        # sm_103a), and cuBLASLt INT8 (torch._int_mm) on the same residue
        # matrices as a library reference.
        a8 = torch.empty(oz.ozemu_res8_bytes(m, k, r), dtype=torch.int8, device=dev)
        b8 = torch.empty(oz.ozemu_res8_bytes(n, k, r), dtype=torch.int8, device=dev)
        res8 = torch.empty_like(res)
        check(oz.ozemu_split_rows_f64_res8(m, k, A.data_ptr(), k, pA, r, a8.data_ptr(), sa.data_ptr(), sh), "res8 A")
        check(oz.ozemu_split_cols_f64_res8(k, n, B.data_ptr(), n, pB, r, b8.data_ptr(), sb.data_ptr(), sh), "res8 B")

        def i8_gemm():
            check(oz.ozemu_residue_gemm_i8(m, n, k, r, a8.data_ptr(), b8.data_ptr(), res8.data_ptr(), sh), "i8 gemm")

        i8_gemm()
        torch.cuda.synchronize(dev)
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(3):
            i8_gemm()
        c1.record(stream)
        torch.cuda.synchronize(dev)
        i8_ms = c0.elapsed_time(c1) / 3
        same = bool(torch.equal(res8, res))
        cmp = {"kernel": "residue_gemm_i8_kernel (mma.sync m16n8k32 s8)", "gemm_ms": round(i8_ms, 3),
               "fp4_limb_gemm_ms": round(gemm_ms, 3), "fp4_speedup": round(i8_ms / gemm_ms, 2),
               "int8_tops": round(r * flop / (i8_ms / 1e3) / 1e12, 1), "residues_identical": same}
        rows_p, k_p = (m + 127) // 128 * 128, (k + 127) // 128 * 128
        cols_p = (n + 127) // 128 * 128
        if hasattr(torch, "_int_mm") and m >= 32 and n >= 8:
            try:
                Am = a8.view(r, rows_p, k_p)[0]
                Bm = b8.view(r, cols_p, k_p)[0].t()
                torch._int_mm(Am, Bm)
                torch.cuda.synchronize(dev)
                c0.record(stream)
                for l in range(r):
                    torch._int_mm(a8.view(r, rows_p, k_p)[l], b8.view(r, cols_p, k_p)[l].t())
                c1.record(stream)
                torch.cuda.synchronize(dev)
                lt_ms = c0.elapsed_time(c1)
                cmp["cublaslt_int8_ms"] = round(lt_ms, 3)
                cmp["cublaslt_int8_tops"] = round(r * 2.0 * rows_p * cols_p * k_p / (lt_ms / 1e3) / 1e12, 1)
            except RuntimeError as exc:  # shape or build constraints of the library call
                cmp["cublaslt_int8"] = "unavailable: %s" % str(exc).splitlines()[0][:120]
        line["int8_comparison"] = cmp
        del a8, b8, res8

    if not args.no_igemm:
        # The exact INT8 x INT8 -> INT32 product (9 FP4 limb GEMMs) on the
        # 4096^3 int8 workload, beside cuBLASLt's INT8 GEMM on the same matrices.
        Ai_h, Bi_h = make_pair(4096, 4096, 4096, WORKLOADS["igemm_s8_4096"]["seed"], "int8")
        Ai = torch.from_numpy(Ai_h).to(dev)
        Bi = torch.from_numpy(Bi_h).to(dev)
        Ci = torch.empty((4096, 4096), dtype=torch.int32, device=dev)

        def igemm():
            check(oz.ozemu_igemm_s8(4096, 4096, 4096, Ai.data_ptr(), Bi.data_ptr(), Ci.data_ptr(), sh), "igemm")

        igemm()
        torch.cuda.synchronize(dev)
        times = []
        for _ in range(5):
            i0 = torch.cuda.Event(enable_timing=True)
            i1 = torch.cuda.Event(enable_timing=True)
            i0.record(stream)
            igemm()
            i1.record(stream)
            torch.cuda.synchronize(dev)
            times.append(i0.elapsed_time(i1))
        ig_ms = statistics.median(times)
        iflop = 2.0 * 4096 ** 3
        leg = {"ms": round(ig_ms, 3), "tops": round(iflop / (ig_ms / 1e3) / 1e12, 1),
               "fp4_frac": round(9 * iflop / (ig_ms / 1e3) / 1e12 / fp4_peak, 4),
               "launches": "split A rows, split B columns, limb GEMM (int32 epilogue)"}
        if hasattr(torch, "_int_mm"):
            ref = torch._int_mm(Ai, Bi)
            torch.cuda.synchronize(dev)
            i0 = torch.cuda.Event(enable_timing=True)
            i1 = torch.cuda.Event(enable_timing=True)
            i0.record(stream)
            torch._int_mm(Ai, Bi)
            i1.record(stream)
            torch.cuda.synchronize(dev)
            leg["exact_vs_cublaslt"] = bool(torch.equal(ref, Ci))
            leg["cublaslt_int8_ms"] = round(i0.elapsed_time(i1), 3)
        line["igemm_s8_4096"] = leg
        del Ai, Bi, Ci

    if not args.no_two_limb and not narrow:
        # The same product with the two-limb moduli (<= 113, 4 FP4 GEMMs per
        # modulus) through ozemu_dgemm_2limb, at the smallest r whose bit
        # budget reaches the three-limb run's.
        P3 = sum(oz.ozemu_bit_budget(k, r))
        r2 = None
        for cand in range(1, oz.ozemu_max_moduli() + 1):
            try:
                if sum(oz.ozemu_bit_budget_2limb(k, cand)) >= P3:
                    r2 = cand
                    break
            except oz.OzemuError:
                continue
        if r2 is not None:
            C2 = torch.empty((m, n), dtype=torch.float64, device=dev)

            def two_limb():
                check(oz.ozemu_dgemm_2limb(m, n, k, A.data_ptr(), k, B.data_ptr(), n, C2.data_ptr(), n, r2, sh),
                      "dgemm_2limb")

            for _ in range(2):
                two_limb()
            torch.cuda.synchronize(dev)
            times = []
            for _ in range(5):
                t0 = torch.cuda.Event(enable_timing=True)
                t1 = torch.cuda.Event(enable_timing=True)
                t0.record(stream)
                two_limb()
                t1.record(stream)
                torch.cuda.synchronize(dev)
                times.append(t0.elapsed_time(t1))
            st2 = oz.ozemu_get_status(sh)
            t2 = statistics.median(times)
            acc_results["two_limb"] = C2[ri, ci].cpu().numpy()
            pA2, pB2 = oz.ozemu_bit_budget_2limb(k, r2)

            # The stages one after another (CUDA events), for the limb GEMM's
            # roofline: 4 r 2MNK FP4 flop per launch.
            ap2 = torch.empty(oz.ozemu_plane_bytes_2limb(m, k, r2), dtype=torch.uint8, device=dev)
            bp2 = torch.empty(oz.ozemu_plane_bytes_2limb(n, k, r2), dtype=torch.uint8, device=dev)
            res2 = torch.empty(oz.ozemu_residue_bytes(m, n, r2), dtype=torch.uint8, device=dev)
            stages2 = [
                ("split_A", lambda: check(oz.ozemu_split_rows_f64_2limb(m, k, A.data_ptr(), k, pA2, r2, ap2.data_ptr(),
                                                                        sa.data_ptr(), sh), "split A 2")),
                ("split_B", lambda: check(oz.ozemu_split_cols_f64_2limb(k, n, B.data_ptr(), n, pB2, r2, bp2.data_ptr(),
                                                                        sb.data_ptr(), sh), "split B 2")),
                ("limb_gemm", lambda: check(oz.ozemu_residue_gemm_2limb(m, n, k, r2, ap2.data_ptr(), bp2.data_ptr(),
                                                                        res2.data_ptr(), sh), "gemm 2")),
                ("crt", lambda: check(oz.ozemu_crt_f64_2limb(m, n, r2, res2.data_ptr(), sa.data_ptr(), sb.data_ptr(),
                                                             C2.data_ptr(), n, sh), "crt 2"))]
            stage_times(stages2)
            st_ms = stage_times(stages2)
            e2e2 = None
            if not args.no_e2e:
                # End to end with host buffers (pinned), as the e2e entry above.
                def e2e2_step():
                    check(oz.ozemu_dgemm_host_2limb(m, n, k, A_pin.data_ptr(), k, B_pin.data_ptr(), n,
                                                    C_pin.data_ptr(), n, r2, sh), "dgemm_host_2limb")

                e2e2_step()
                torch.cuda.synchronize(dev)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(3):
                    e2e2_step()
                e1.record(stream)
                torch.cuda.synchronize(dev)
                e2_ms = e0.elapsed_time(e1) / 3
                if not torch.equal(C_pin.view(torch.int64), C2.cpu().view(torch.int64)):
                    raise SystemExit("two-limb e2e result differs from the device result")
                e2e2 = {"value": round(flop / (e2_ms / 1e3) / 1e12, 3), "unit": "TFLOP/s",
                        "ms_per_step": round(e2_ms, 3), "steps": 3}
            g2_tflops = 4.0 * r2 * flop / (st_ms["limb_gemm"] / 1e3) / 1e12
            line["two_limb"] = {
                "r": r2, "bit_budget": pA2 + pB2, "three_limb_bit_budget": P3,
                "fp4_gemms": 4 * r2, "three_limb_fp4_gemms": 9 * r, "ms": round(t2, 3),
                "tflops": round(flop / (t2 / 1e3) / 1e12, 2), "status": int(st2),
                "stage_ms": {kk: round(v, 3) for kk, v in st_ms.items()}, "e2e": e2e2,
                "limb_gemm_roofline": {"bound": "tensor", "achieved": round(g2_tflops, 1),
                                       "peak": round(fp4_peak, 1), "unit": "TFLOP/s",
                                       "frac": round(g2_tflops / fp4_peak, 4),
                                       "algorithmic": "4 r 2MNK FP4 flop per launch"}}
            del C2, ap2, bp2, res2

    if rank == 0:
        t_acc = time.time()
        ratios = bound_ratios(A_h, B_h, acc_rows, acc_cols, acc_results)
        line["accuracy"] = {"sample": "%d random entries of C, exact products summed in rationals on the host"
                                      % ACC_SAMPLE,
                            "max_err_over_bound": {kk: round(v, 6) for kk, v in ratios.items()},
                            "bound": "2 K 2^-53 (|A||B|)_ij", "seconds": round(time.time() - t_acc, 1)}
        if "two_limb" in ratios:
            line["accuracy"]["two_limb_r"] = line["two_limb"]["r"]

    if rank == 0 and not args.no_cpu_baseline:
        cb = cpu_oracle(args.workload, r, CPU_MIN_SECONDS, shape={"m": m, "n": n, "k": k})
        line["cpu_baseline"] = {"value": cb["tflops"], "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                                "sample": "%d steps of a %dx%d block of C at full K=%d (oracle, 1 thread), %.1f s"
                                          % (cb["steps"], cb["rows"], cb["cols"], cb["k"], cb["seconds"])}
    if rank == 0 and not args.no_cpu_baseline:
        # Context: native fp64 matmul on the host cores (numpy's BLAS) on a
        # block of the same product at the full K.
        rb = min(m, 1024)
        cbk = min(n, 1024)
        Ab = np.ascontiguousarray(A_h[:rb])
        Bb = np.ascontiguousarray(B_h[:, :cbk])
        Ab @ Bb
        t0 = time.perf_counter()
        reps = 0
        while True:
            Ab @ Bb
            reps += 1
            if time.perf_counter() - t0 > 1.0:
                break
        t_np = (time.perf_counter() - t0) / reps
        line["cpu_native_matmul"] = {"tflops": round(2.0 * rb * cbk * k / t_np / 1e12, 4), "unit": "TFLOP/s",
                                     "block": "%dx%d @ %dx%d" % (rb, k, k, cbk), "host_cores": os.cpu_count(),
                                     "kind": "numpy float64 matmul (context, not the oracle)"}
    if ws > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    spec = dict(WORKLOADS[args.workload])
    for key in ("m", "n", "k"):
        if getattr(args, key):
            spec[key] = getattr(args, key)
    shape = {"m": spec["m"], "n": spec["n"], "k": spec["k"]}
    r = args.r or spec.get("r", 13)
    # warm-up steps are bounded samples too; each step is one sample block.
    if args.warmup:
        cpu_oracle(args.workload, r, 0, max_steps=args.warmup, sample=32, shape=shape)
    cb = cpu_oracle(args.workload, r, 0, max_steps=args.steps, sample=32, shape=shape)
    value = cb["tflops"]
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(1e3 * cb["seconds"] / cb["steps"], 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": workload_name(args, spec), "m": spec["m"], "n": spec["n"], "k": spec["k"], "r": r,
                       "dist": spec["dist"], "seed": spec["seed"]},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                             "sample": "each step a %dx%d block of C at full K=%d (oracle, 1 thread)"
                                       % (cb["rows"], cb["cols"], cb["k"])},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
