#!/usr/bin/env python
"""Benchmark: emulated DGEMM TFLOP/s (2MNK/t) and % of FP4 roofline on one GB300.

One step = one pass of the whole hot path over one synthetic problem held in
HBM: deconstruction of A's rows and B's columns (scale, round, residues, FP4
digit planes), the FP4 digit GEMMs with modular recombination, and the CRT +
scale back to fp64.  The default workload is M = N = K = 8192 with entries
u 2^e (u ~ U(-1, 1), e uniform in [-10, 10]).

The headline family of moduli is the mixed-digit list (one FP4 product for
each single-digit modulus, four for each two-digit one) with the smallest r
whose bit budget reaches that of r three-limb moduli (9 products each) for
the workload; the three-limb and two-limb families are timed beside it on
the same problem, and the other workloads (256^3, the exact INT8 product at
4096^3, the GEMV at n = 1 and 8, K = 65536) follow as sub-records.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--family F]
  python bench.py --impl reference ...   # the CPU oracle on bounded samples

Under torchrun every rank runs its own replica (the problems are independent:
weak scaling, no data-path collective); rank 0 prints one JSON line.
"""

import argparse
import hashlib
import json
import math
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
SPLIT_INSTR_PER_ELEMENT = 222.0  # row split, mixed-digit r = 19: thread instructions per input element (ncu)
SPLIT_INSTR_R = 19
FAMILIES = ("mixed", "two", "three")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ozemu", choices=["ozemu", "reference"])
    ap.add_argument("--workload", default="dgemm_8192_wide", choices=sorted(WORKLOADS))
    ap.add_argument("--family", default="mixed", choices=FAMILIES,
                    help="moduli of the timed step: mixed-digit, two-limb or three-limb")
    ap.add_argument("--r", type=int, default=None, help="override the number of moduli of the timed step")
    ap.add_argument("--m", type=int, default=None, help="override M (same distribution and seed)")
    ap.add_argument("--n", type=int, default=None, help="override N")
    ap.add_argument("--k", type=int, default=None, help="override K")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-native", action="store_true")
    ap.add_argument("--no-compare", action="store_true", help="skip the INT8 residue-GEMM comparison")
    ap.add_argument("--no-families", action="store_true", help="skip the other moduli families")
    ap.add_argument("--no-workloads", action="store_true", help="skip the other workloads' sub-records")
    ap.add_argument("--no-accuracy", action="store_true")
    ap.add_argument("--chunks", type=int, default=4,
                    help="row chunks of A in the timed step (1: the stages one after another)")
    ap.add_argument("--schedule", default="pipelined", choices=["pipelined", "phased"],
                    help="pipelined: each chunk's CRT beside the next chunk's GEMM, chunk splits beside the "
                         "GEMMs; phased: all splits (A beside B), then the GEMMs, then the CRTs")
    return ap.parse_args()


# ------------------------------------------------------------ exact error
# The accuracy entries compare results with the exact product, computed here
# on the host without the oracle: each row of A (column of B) is cut into
# slices of integers below 2^beta times a power of two, with k 2^(2 beta) <=
# 2^53, so every slice-by-slice product is an exact float64 BLAS result, and
# the residual sum - C is rounded once by math.fsum.

def _beta(k):
    beta = 26
    while k * 4 ** beta > 2 ** 53:
        beta -= 1
    return beta


def _cut(X, beta):
    """(e, slices): X = sum_s slices[s] 2^(e - beta (s+1)) per row, exactly."""
    rem = np.array(X, dtype=np.float64, order="C")
    mx = np.max(np.abs(rem), axis=1) if rem.shape[1] else np.zeros(rem.shape[0])
    e = np.array([math.frexp(float(v))[1] if v else 0 for v in mx], dtype=np.int64)
    out = []
    while rem.any():
        sc = np.ldexp(1.0, beta * (len(out) + 1) - e)[:, None]
        q = np.trunc(rem * sc)
        rem -= q / sc
        out.append(q)
        if len(out) > 80:
            raise ArithmeticError("too many slices")
    return e, out


def _exact_terms(Ar, Bc, pairs):
    """Exact float64 terms whose sum is the product: for pairs=False the
    block Ar @ Bc (R x N), for pairs=True the entry-wise dot products of the
    rows of Ar with the columns of Bc."""
    beta = _beta(max(Ar.shape[1], 1))
    ea, sa = _cut(Ar, beta)
    eb, sb = _cut(Bc.T, beta)
    terms = []
    for s, qa in enumerate(sa):
        for t, qb in enumerate(sb):
            if pairs:
                terms.append(np.ldexp(np.einsum("ek,ek->e", qa, qb), ea + eb - beta * (s + t + 2)))
            else:
                terms.append(np.ldexp(qa @ qb.T, ea[:, None] + eb[None, :] - beta * (s + t + 2)))
    return terms


def exact_residuals(A, B, part, Cs):
    """[RN(exact - C) for C in Cs] for one part of the accuracy sample,
    exactly: ("rows", idx) whole rows, ("cols", idx) whole columns, ("pairs",
    (I, J)) entries.  The exact terms are formed once for all the Cs."""
    kind, idx = part
    Cs = [np.asarray(C, dtype=np.float64) for C in Cs]
    outs = [np.empty(C.shape) for C in Cs]

    def fold(T, sel):
        flat_T = T.reshape(T.shape[0], -1)
        for C, out in zip(Cs, outs):
            c = C[sel].reshape(-1)
            o = np.array([math.fsum(flat_T[:, j].tolist() + [-c[j]]) for j in range(c.size)])
            out[sel] = o.reshape(C[sel].shape)

    if kind == "pairs":
        I, J = idx
        for e0 in range(0, len(I), 512):
            fold(np.stack(_exact_terms(A[I[e0:e0 + 512]], B[:, J[e0:e0 + 512]], True)), np.s_[e0:e0 + 512])
        return outs
    if kind == "rows":
        for b0 in range(0, B.shape[1], 512):
            fold(np.stack(_exact_terms(A[idx], B[:, b0:b0 + 512], False)), np.s_[:, b0:b0 + 512])
    else:
        for b0 in range(0, A.shape[0], 512):
            fold(np.stack(_exact_terms(A[b0:b0 + 512], B[:, idx], False)), np.s_[b0:b0 + 512])
    return outs


def _absum(A, B, part):
    kind, idx = part
    if kind == "pairs":
        I, J = idx
        return np.einsum("ek,ek->e", np.abs(A[I]), np.abs(B[:, J].T))
    if kind == "rows":
        return np.abs(A[idx]) @ np.abs(B)
    return np.abs(A) @ np.abs(B[:, idx])


def bound_ratios(A_h, B_h, parts, results):
    """max over the sampled entries of |C_ij - (AB)_ij| / (2 K 2^-53 (|A||B|)_ij)
    for each named result; parts as accuracy_sample returns, results[name]
    a list of the entries of each part (as sample_values takes them)."""
    k = A_h.shape[1]
    names = list(results)
    out = {name: 0.0 for name in names}
    for p, part in enumerate(parts):
        bound = 2.0 * k * 2.0 ** -53 * _absum(A_h, B_h, part)
        res = exact_residuals(A_h, B_h, part, [results[name][p] for name in names])
        for name, rr in zip(names, res):
            rr = np.abs(rr)
            with np.errstate(divide="ignore", invalid="ignore"):
                ratio = np.where(bound > 0, rr / np.where(bound > 0, bound, 1.0), np.where(rr == 0, 0.0, np.inf))
            if ratio.size:
                out[name] = max(out[name], float(ratio.max()))
    return out


def accuracy_sample(m, n, full_rows, full_cols, n_entries, seed=7):
    """The sampled parts: ("rows", idx) whole rows, ("cols", idx) whole
    columns and ("pairs", (I, J)) random entries."""
    rng = np.random.default_rng(seed)
    fr = np.sort(rng.choice(m, size=min(full_rows, m), replace=False))
    fc = np.sort(rng.choice(n, size=min(full_cols, n), replace=False))
    return [("rows", fr), ("cols", fc), ("pairs", (rng.integers(0, m, n_entries), rng.integers(0, n, n_entries)))]


def sample_values(C, parts, dev):
    """The entries of a device matrix C for each sampled part (host arrays)."""
    import torch
    out = []
    for kind, idx in parts:
        if kind == "rows":
            out.append(C[torch.from_numpy(idx).to(dev)].cpu().numpy())
        elif kind == "cols":
            out.append(C[:, torch.from_numpy(idx).to(dev)].cpu().numpy())
        else:
            I, J = idx
            out.append(C[torch.from_numpy(I).to(dev), torch.from_numpy(J).to(dev)].cpu().numpy())
    return out


def sample_size(parts, m, n):
    return sum(len(idx) * (n if kind == "rows" else m) if kind != "pairs" else len(idx[0]) for kind, idx in parts)


# ------------------------------------------------------------------ misc

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
            return
        # nvidia-smi takes a moment to start: wait (up to 3 s) for its first
        # sample, so that the samples fall inside the region that follows.
        t0 = time.time()
        while time.time() - t0 < 3.0 and self.proc.poll() is None:
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.02)
        self._skip = 0
        with open(self.path) as f:
            self._skip = sum(1 for _ in f)  # samples taken before the region

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows, before = [], []
        with open(self.path) as f:
            for i, line in enumerate(f):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    (rows if i >= getattr(self, "_skip", 0) else before).append(parts)
        if not rows:  # a region shorter than the sampling interval: the last sample before it
            rows = before[-1:]
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
ceiling = {ceiling!r}
n_rows = min({ns}, spec["m"]); n_cols = min({ns}, spec["n"])
steps, total, t0 = 0, 0.0, time.time()
while True:
    rows = sample_indices(spec["m"], n_rows, seed=100 + {off} + steps)
    cols = sample_indices(spec["n"], n_cols, seed=200 + {off} + steps)
    t = time.time()
    oracle.dgemm_block(A, B, r, rows=rows, cols=cols, ceiling=ceiling)
    total += time.time() - t
    steps += 1
    if (({max_steps} and steps >= {max_steps}) or (not {max_steps} and total >= {min_s})):
        break
print(json.dumps(dict(seconds=total, steps=steps, rows=n_rows, cols=n_cols, k=spec["k"])))
"""


CEILING_OF = {"three": 256, "two": 113, "mixed": "mixed"}  # the oracle's name for each family's moduli


def cpu_oracle(name, r, min_seconds, max_steps=0, sample=CPU_SAMPLE, shape=None, family="three", procs=1):
    """Times the oracle on bounded samples in `procs` single-threaded
    subprocesses at once (each its own sample blocks); the throughput is their
    flops over the slowest one's time."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    children = []
    for i in range(procs):
        code = CPU_SNIPPET.format(root=ROOT, name=name, r=r, ns=sample, max_steps=max_steps, min_s=min_seconds,
                                  shape=dict(shape or {}), ceiling=CEILING_OF[family], off=1000 * i)
        children.append(subprocess.Popen([sys.executable, "-c", code], env=env, stdout=subprocess.PIPE,
                                         stderr=subprocess.PIPE, text=True))
    results = []
    for ch in children:
        out, err = ch.communicate(timeout=3600)
        if ch.returncode != 0:
            raise RuntimeError(err[-2000:])
        results.append(json.loads(out.strip().splitlines()[-1]))
    d = dict(results[0])
    d["steps"] = sum(x["steps"] for x in results)
    d["seconds"] = max(x["seconds"] for x in results)
    d["procs"] = procs
    flops = 2.0 * d["rows"] * d["cols"] * d["k"] * d["steps"]
    d["tflops"] = flops / d["seconds"] / 1e12
    return d


# ------------------------------------------------------------------ GPU arm

def kernel_traffic(workload, family, chunks, bblocks):
    """DRAM bytes per launch of the digit GEMM from the committed ncu record,
    used only for the workload, family and row chunking it was captured on
    and only while the kernel sources are unchanged since the capture."""
    path = os.path.join(ROOT, "profiles", "limb_gemm_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    h = hashlib.sha256()
    for fn in ("gemm_fp4.cu", "common.cuh"):
        with open(os.path.join(ROOT, "ozaki_ii_fp64_gb300", "csrc", fn), "rb") as f:
            h.update(f.read())
    if (d.get("source_sha256") != h.hexdigest() or d.get("workload") != workload or d.get("chunks") != chunks
            or d.get("b_blocks") != bblocks or d.get("family", "three") != family):
        return None
    return d


def bench_config(args, spec, r, products, bits):
    """The config dict both arms print: workload, shape, inputs and moduli."""
    m, k = spec["m"], spec["k"]
    return {"workload": workload_name(args, spec), "m": spec["m"], "n": spec["n"], "k": k, "dist": spec["dist"],
            "seed": spec["seed"], "family": args.family, "r": r, "fp4_products_per_output": products,
            "bit_budget": bits, "l2": "inputs larger than L2 (%d MiB per operand), no flush" % (m * k * 8 >> 20)}


def workload_name(args, spec):
    base = WORKLOADS[args.workload]
    if all(spec[x] == base[x] for x in ("m", "n", "k")):
        return args.workload
    return "%s@%dx%dx%d" % (args.workload, spec["m"], spec["n"], spec["k"])


class Family:
    """The C ABI entry points and product count of one moduli family."""

    SUFFIX = {"three": "", "two": "_2limb", "mixed": "_mixed"}
    NAME = {"three": "three-limb (9 FP4 products per modulus)",
            "two": "two-limb (4 FP4 products per modulus)",
            "mixed": "mixed-digit (1 FP4 product per single-digit modulus, 4 per two-digit one)"}

    def __init__(self, oz, key):
        self.oz = oz
        self.key = key
        sfx = self.SUFFIX[key]
        g = lambda base: getattr(oz, base + sfx)
        self.budget = g("ozemu_bit_budget")
        self.plane_bytes = g("ozemu_plane_bytes")
        self.split_rows = g("ozemu_split_rows_f64")
        self.split_cols = g("ozemu_split_cols_f64")
        self.residue_gemm = g("ozemu_residue_gemm")
        self.crt = g("ozemu_crt_f64")
        self.dgemm = g("ozemu_dgemm")
        self.dgemm_host = g("ozemu_dgemm_host")
        self.max_r = oz.ozemu_max_moduli_mixed() if key == "mixed" else oz.ozemu_max_moduli()

    def products(self, r):
        if self.key == "mixed":
            return self.oz.ozemu_products_mixed(r)
        return (9 if self.key == "three" else 4) * r

    def gemm_launches(self, r):
        if self.key == "mixed":
            single = self.oz.ozemu_single_digit_moduli_mixed()
            return 1 if r <= single else 2
        return 1

    def bits(self, k, r):
        try:
            return sum(self.budget(k, r))
        except self.oz.OzemuError:
            return -1

    def r_for(self, k, P):
        """Smallest r whose bit budget at inner dimension k reaches P."""
        for r in range(1, self.max_r + 1):
            if self.bits(k, r) >= P:
                return r
        return None


def time_ms(torch, stream, fn, reps=5, warm=1):
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return statistics.median(ts)


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
    t_bench0 = time.time()

    spec = dict(WORKLOADS[args.workload])
    for key in ("m", "n", "k"):
        if getattr(args, key):
            spec[key] = getattr(args, key)
    if spec["kind"] == "igemm":
        # The exact integer products alone (their own line; not the metric's workload).
        stream = torch.cuda.current_stream(dev)

        def check_int(st, what):
            if st != 0:
                raise oz.OzemuError(st, what)

        pk, pk_kind = peaks()
        legs = int_products(torch, oz, stream, stream.cuda_stream, check_int, dev, pk["bf16_tflops"] * FP4_OVER_BF16)
        if rank == 0:
            print(json.dumps({"metric": "exact INT8 x INT8 GEMM TOP/s (2MNK/t) at 4096^3", "unit": "TOP/s",
                              "value": legs["igemm_s8_4096"]["tops"], "higher_is_better": True, "n_gpus": ws,
                              "dtype": "int8", "data": "synthetic", "config": {"workload": args.workload},
                              "peak_source": "%s bf16 burst x %.0f" % (pk_kind, FP4_OVER_BF16),
                              "int_products": legs}))
        return
    if spec["kind"] != "dgemm":
        raise SystemExit("bench.py times the emulated DGEMM workloads")
    A_h, B_h = make_pair(spec["m"], spec["n"], spec["k"], spec["seed"], spec["dist"])
    m, n, k = spec["m"], spec["n"], spec["k"]
    fams = {key: Family(oz, key) for key in FAMILIES}
    three = fams["three"]
    P3 = three.bits(k, spec["r"])  # the budget the workload's r three-limb moduli give
    fam = fams[args.family]
    r = args.r or fam.r_for(k, P3)
    if r is None:
        raise SystemExit("no r of the %s family reaches P = %d at k = %d" % (args.family, P3, k))
    pA, pB = fam.budget(k, r)
    n_prod = fam.products(r)
    A = torch.from_numpy(A_h).to(dev)
    B = torch.from_numpy(B_h).to(dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    def check(st, what):
        if st != 0:
            raise oz.OzemuError(st, what)

    # Preallocated stage buffers: nothing is allocated in the timed region.
    ap = torch.empty(fam.plane_bytes(m, k, r), dtype=torch.uint8, device=dev)
    bp = torch.empty(fam.plane_bytes(n, k, r), dtype=torch.uint8, device=dev)
    sa = torch.empty(m, dtype=torch.int32, device=dev)
    sb = torch.empty(n, dtype=torch.int32, device=dev)
    res = torch.empty(oz.ozemu_residue_bytes(m, n, r), dtype=torch.uint8, device=dev)
    C = torch.empty((m, n), dtype=torch.float64, device=dev)
    # n <= ozemu_narrow_max_n() with the three-limb family: the fused narrow
    # path (what ozemu_dgemm runs for such shapes).
    narrow = (args.family == "three" and n <= oz.ozemu_narrow_max_n() and k <= NARROW_MAX_K
              and os.environ.get("OZEMU_NARROW", "1") != "0")

    def split_a():
        check(fam.split_rows(m, k, A.data_ptr(), k, pA, r, ap.data_ptr(), sa.data_ptr(), sh), "split A")

    def split_b():
        check(fam.split_cols(k, n, B.data_ptr(), n, pB, r, bp.data_ptr(), sb.data_ptr(), sh), "split B")

    def digit_gemm():
        check(fam.residue_gemm(m, n, k, r, ap.data_ptr(), bp.data_ptr(), res.data_ptr(), sh), "digit gemm")

    def narrow_residues():
        check(oz.ozemu_residues_narrow_f64(m, n, k, r, A.data_ptr(), k, B.data_ptr(), n, res.data_ptr(),
                                           sa.data_ptr(), sb.data_ptr(), sh), "narrow residues")

    def crt():
        check(fam.crt(m, n, r, res.data_ptr(), sa.data_ptr(), sb.data_ptr(), C.data_ptr(), n, sh), "crt")

    if narrow:
        stages = [("narrow_residues", narrow_residues), ("crt", crt)]
    else:
        stages = [("split_A", split_a), ("split_B", split_b), ("digit_gemm", digit_gemm), ("crt", crt)]

    # The timed step.  Digit-plane path: the library's device-operand
    # schedule with the stage calls, pipelined over row chunks of A on three
    # streams -- B's split (main stream), each chunk's split (split stream,
    # from the start), digit GEMM (main stream, bracketed by events) and CRT
    # (CRT stream, beside the next chunk's GEMM).  Narrow path: its two calls.
    chunks = 1 if narrow else max(1, args.chunks)
    crows = m if chunks == 1 else ((m + chunks - 1) // chunks + 255) // 256 * 256
    chunk_bufs = []
    for row0 in range(0, m, crows):
        mc = min(crows, m - row0)
        chunk_bufs.append((row0, mc, torch.empty(fam.plane_bytes(mc, k, r), dtype=torch.uint8, device=dev),
                           torch.empty(mc, dtype=torch.int32, device=dev),
                           torch.empty(oz.ozemu_residue_bytes(mc, n, r), dtype=torch.uint8, device=dev)))
    nch = len(chunk_bufs)
    s_split = torch.cuda.Stream(dev)
    s_crt = torch.cuda.Stream(dev)
    ev_start = torch.cuda.Event()
    evA = [torch.cuda.Event() for _ in range(nch)]
    evG = [torch.cuda.Event() for _ in range(nch)]
    evC = [torch.cuda.Event() for _ in range(nch)]
    if narrow:
        launches_per_step = 3  # B's column residues, fused pass over A, CRT
    else:
        launches_per_step = 2 + nch * (2 + fam.gemm_launches(r))  # B: column maxima + split; chunk: split, GEMMs, CRT
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
        # As the library enqueues them: the chunks' splits on the split
        # stream first, then B's split on the main stream.
        for c, (row0, mc, apc, sac, resc) in enumerate(chunk_bufs):
            check(fam.split_rows(mc, k, A.data_ptr() + row0 * k * 8, k, pA, r, apc.data_ptr(), sac.data_ptr(),
                                 s_split.cuda_stream), "split A chunk")
            evA[c].record(s_split)
        split_b()
        if args.schedule == "phased":
            # Splits of A beside B's, then the GEMMs back to back, then the CRTs.
            stream.wait_event(evA[nch - 1])
            for c, (row0, mc, apc, sac, resc) in enumerate(chunk_bufs):
                if gev is not None:
                    gev[c][0].record(stream)
                check(fam.residue_gemm(mc, n, k, r, apc.data_ptr(), bp.data_ptr(), resc.data_ptr(), sh),
                      "digit gemm chunk")
                if gev is not None:
                    gev[c][1].record(stream)
            for c, (row0, mc, apc, sac, resc) in enumerate(chunk_bufs):
                check(fam.crt(mc, n, r, resc.data_ptr(), sac.data_ptr(), sb.data_ptr(), C.data_ptr() + row0 * n * 8,
                              n, sh), "crt chunk")
            return
        for c, (row0, mc, apc, sac, resc) in enumerate(chunk_bufs):
            stream.wait_event(evA[c])
            if gev is not None:
                gev[c][0].record(stream)
            check(fam.residue_gemm(mc, n, k, r, apc.data_ptr(), bp.data_ptr(), resc.data_ptr(), sh),
                  "digit gemm chunk")
            if gev is not None:
                gev[c][1].record(stream)
            evG[c].record(stream)
            s_crt.wait_event(evG[c])
            check(fam.crt(mc, n, r, resc.data_ptr(), sac.data_ptr(), sb.data_ptr(), C.data_ptr() + row0 * n * 8, n,
                          s_crt.cuda_stream), "crt chunk")
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
    fp4_peak = pk["bf16_tflops"] * FP4_OVER_BF16  # TFLOP/s, burst: kernels timed alone (the legs below)
    # The timed step runs back to back for a long region under the power cap:
    # its GEMM takes the sustained figure (the burst one is reported beside it).
    step_long = elapsed_ms >= 250.0 and pk.get("bf16_tflops_sustained")
    fp4_peak_step = pk["bf16_tflops_sustained"] * FP4_OVER_BF16 if step_long else fp4_peak
    step_peak_kind = "sustained" if step_long else "burst"
    fp4_flop = n_prod * flop
    if narrow:
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
        tr = kernel_traffic(workload_name(args, spec), args.family, nch, nbc)
        roofline = {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(fp4_peak_step, 1),
                    "unit": "TFLOP/s", "frac": round(achieved / fp4_peak_step, 4),
                    "frac_of_burst_peak": round(achieved / fp4_peak, 4),
                    "traffic": (int(tr["bytes_per_launch"]) if tr else None),
                    "traffic_per": (tr.get("unit_of_launch", "launch") if tr else None),
                    "kernel": "limb_gemm_pair_kernel (CTA pair, 256x224 tiles), %d launch(es) per chunk"
                              % fam.gemm_launches(r),
                    "peak_source": "%s bf16 %s x %.0f (nominal FP4:BF16): timed inside %.0f ms of back-to-back "
                                   "steps" % (pk_kind, step_peak_kind, FP4_OVER_BF16, elapsed_ms),
                    "algorithmic": "%d FP4 products x 2MNK flop per chunk (%s)" % (n_prod, Family.NAME[args.family])}
        # Whole-step roofline: the slower of the FP4 term and the algorithmic
        # bytes at HBM peak.  Planes hold one nibble per digit plane.
        planes_per_elem = fam.plane_bytes(128, 128, r) / (128 * 64)
        bytes_alg = (m * k + k * n) * (8 + planes_per_elem) + m * n * (2.0 * r + 8)
        t_roof = max(fp4_flop / (fp4_peak_step * 1e12), bytes_alg / (pk["hbm_gbs"] * 1e9))
        t_roof_burst = max(fp4_flop / (fp4_peak * 1e12), bytes_alg / (pk["hbm_gbs"] * 1e9))
        # Context: the same step against the roofline of the three-limb list
        # (9 FP4 products per modulus) at the same bit budget.
        t_roof_three = fams["three"].products(spec["r"]) * flop / (fp4_peak_step * 1e12)
    pct_roof = 100.0 * t_roof / (ms_per_step / 1e3)

    line = {"metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": bench_config(args, spec, r, n_prod, pA + pB),
            "schedule": {"path": "narrow (fused)" if narrow else "digit planes", "row_chunks": nch,
                         "order": args.schedule,
                         "three_limb_r": spec["r"], "three_limb_bit_budget": P3},
            "pct_fp4_roofline" if not narrow else "pct_io_roofline": round(pct_roof, 2), "roofline": roofline,
            "stage_ms": {kk: round(v, 3) for kk, v in stage_ms.items()},
            "gpu_launches": launches_per_step * args.steps, "clocks": clk}
    if not narrow:
        line["pct_fp4_roofline_burst_peak"] = round(100.0 * t_roof_burst / (ms_per_step / 1e3), 2)
        line["pct_three_limb_fp4_roofline"] = round(100.0 * t_roof_three / (ms_per_step / 1e3), 2)

    # The memory-bound stages alone: median of repeated launches, each after
    # a write of 256 MiB (more than L2), against the algorithmic bytes.
    # Deconstruction reads 8 B and writes the digit planes per input element
    # (B's transpose is extra traffic of this implementation, not in the
    # count); the CRT reads r B and writes 8 B per output.
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

        pe = fam.plane_bytes(128, 128, r) / (128 * 128)  # plane bytes per input element
        line["memory_stages"] = {
            "deconstruct_A": mem_entry("split_rows_f64_kernel", split_a, (8.0 + pe) * m * k),
            "deconstruct_B": mem_entry("col_absmax_kernel + split_cols_f64_kernel", split_b, (8.0 + pe) * k * n),
            "reconstruct": mem_entry("crt_kernel", crt, (r + 8.0) * m * n)}
        del flush

    # End to end through the C ABI with host buffers: the family's
    # ozemu_dgemm_host call copies A and B in from pinned memory and C out,
    # every step (pipelined with the work inside the library).
    A_pin = B_pin = C_pin = None
    if not args.no_e2e:
        A_pin = torch.from_numpy(A_h).pin_memory()
        B_pin = torch.from_numpy(B_h).pin_memory()
        C_pin = torch.empty((m, n), dtype=torch.float64).pin_memory()

        def e2e_step():
            if narrow:
                check(oz.ozemu_dgemm_host(m, n, k, A_pin.data_ptr(), k, B_pin.data_ptr(), n, C_pin.data_ptr(), n, r,
                                          sh), "dgemm_host")
            else:
                check(fam.dgemm_host(m, n, k, A_pin.data_ptr(), k, B_pin.data_ptr(), n, C_pin.data_ptr(), n, r, sh),
                      "dgemm_host")

        e_steps = max(1, min(args.steps, 5))
        e_ms = time_ms(torch, stream, e2e_step, reps=e_steps, warm=max(1, args.warmup))
        if oz.ozemu_get_status(sh) != 0:
            raise SystemExit("device status not OK after e2e")
        if not torch.equal(C_pin.view(torch.int64), C.cpu().view(torch.int64)):
            raise SystemExit("e2e result differs from the staged result")
        line["e2e"] = {"value": round(ws * flop / (e_ms / 1e3) / 1e12, 3), "unit": "TFLOP/s",
                       "h2d_bytes_per_step": int(A_h.nbytes + B_h.nbytes), "d2h_bytes_per_step": int(m * n * 8),
                       "ms_per_step": round(e_ms, 3), "steps": e_steps,
                       "call": "ozemu_dgemm_host%s" % ("" if narrow else Family.SUFFIX[args.family])}

    C_native = None
    if not args.no_native:
        nat_ms, C_native = native_dgemm(torch, stream, A, B)
        line["native_dgemm"] = {"tflops": round(flop / (nat_ms / 1e3) / 1e12, 3), "ms": round(nat_ms, 3),
                                "speedup_of_emulation": round(nat_ms / ms_per_step, 2)}

    # Accuracy against the exact product: 16 full rows, 16 full columns and
    # 4096 random entries of C (every family below is checked on the same
    # entries).
    acc_parts = accuracy_sample(m, n, 16, 16, 4096)
    acc_results = {args.family: sample_values(C, acc_parts, dev)}
    if C_native is not None:
        acc_results["native_dgemm"] = sample_values(C_native, acc_parts, dev)
        del C_native

    # The same product through each family's ozemu_dgemm call (device
    # buffers), at the smallest r whose budget reaches the three-limb one,
    # with the stage times and the digit GEMM's roofline fraction.
    if not args.no_families and not narrow:
        line["families"] = {}
        Cf = torch.empty((m, n), dtype=torch.float64, device=dev)
        for key, fm in fams.items():
            rf = fm.r_for(k, P3) if key != args.family else r
            if rf is None:
                continue
            pAf, pBf = fm.budget(k, rf)
            ms_f = time_ms(torch, stream, lambda: check(fm.dgemm(m, n, k, A.data_ptr(), k, B.data_ptr(), n,
                                                                 Cf.data_ptr(), n, rf, sh), "dgemm family"))
            if oz.ozemu_get_status(sh) != 0:
                raise SystemExit("device status not OK after the %s family" % key)
            if key != args.family:
                acc_results[key] = sample_values(Cf, acc_parts, dev)
            apf = torch.empty(fm.plane_bytes(m, k, rf), dtype=torch.uint8, device=dev)
            bpf = torch.empty(fm.plane_bytes(n, k, rf), dtype=torch.uint8, device=dev)
            resf = torch.empty(oz.ozemu_residue_bytes(m, n, rf), dtype=torch.uint8, device=dev)
            stf = [("split_A", lambda: check(fm.split_rows(m, k, A.data_ptr(), k, pAf, rf, apf.data_ptr(),
                                                           sa.data_ptr(), sh), "split A")),
                   ("split_B", lambda: check(fm.split_cols(k, n, B.data_ptr(), n, pBf, rf, bpf.data_ptr(),
                                                           sb.data_ptr(), sh), "split B")),
                   ("digit_gemm", lambda: check(fm.residue_gemm(m, n, k, rf, apf.data_ptr(), bpf.data_ptr(),
                                                                resf.data_ptr(), sh), "gemm")),
                   ("crt", lambda: check(fm.crt(m, n, rf, resf.data_ptr(), sa.data_ptr(), sb.data_ptr(),
                                                Cf.data_ptr(), n, sh), "crt"))]
            stage_times(stf)
            st_ms = stage_times(stf)
            g_tflops = fm.products(rf) * flop / (st_ms["digit_gemm"] / 1e3) / 1e12
            rec = {"family": Family.NAME[key], "r": rf, "bit_budget": pAf + pBf,
                   "fp4_products_per_output": fm.products(rf), "ms": round(ms_f, 3),
                   "tflops": round(flop / (ms_f / 1e3) / 1e12, 2),
                   "stage_ms": {kk: round(v, 3) for kk, v in st_ms.items()},
                   "digit_gemm_roofline": {"bound": "tensor", "achieved": round(g_tflops, 1),
                                           "peak": round(fp4_peak, 1), "unit": "TFLOP/s",
                                           "frac": round(g_tflops / fp4_peak, 4)}}
            if not args.no_e2e:
                e_f = time_ms(torch, stream, lambda: check(fm.dgemm_host(m, n, k, A_pin.data_ptr(), k,
                                                                         B_pin.data_ptr(), n, C_pin.data_ptr(), n,
                                                                         rf, sh), "dgemm_host family"),
                              reps=3, warm=1)
                rec["e2e_tflops"] = round(flop / (e_f / 1e3) / 1e12, 2)
            line["families"][key] = rec
            del apf, bpf, resf
        del Cf

    if not args.no_compare and not narrow and not args.no_families:
        line["int8_comparison"] = int8_comparison(torch, oz, stream, sh, check, A, B, m, n, k, spec["r"], dev,
                                                  line)

    if not args.no_workloads:
        line["fp4_mma_rate"] = fp4_mma_rate(torch, oz, stream, sh, check, dev, clk, fp4_peak)
        line["workloads"] = other_workloads(torch, oz, fams, stream, sh, check, dev, args, pk, fp4_peak,
                                            line.get("native_dgemm"), clk)

    if rank == 0 and not args.no_accuracy:
        t_acc = time.time()
        ratios = bound_ratios(A_h, B_h, acc_parts, acc_results)
        line["accuracy"] = {"sample": "16 full rows, 16 full columns and 4096 random entries of C (%d entries), "
                                      "exact products from error-free slices summed by fsum on the host"
                                      % sample_size(acc_parts, m, n),
                            "max_err_over_bound": {kk: round(v, 6) for kk, v in ratios.items()},
                            "bound": "2 K 2^-53 (|A||B|)_ij", "seconds": round(time.time() - t_acc, 1)}

    if rank == 0 and not args.no_cpu_baseline:
        procs = max(1, min(16, os.cpu_count() or 1))
        cb = cpu_oracle(args.workload, r, CPU_MIN_SECONDS, shape={"m": m, "n": n, "k": k}, family=args.family,
                        procs=procs)
        line["cpu_baseline"] = {"value": cb["tflops"], "unit": "TFLOP/s", "cores": procs, "kind": "oracle",
                                "sample": "%d steps of %dx%d blocks of C at full K=%d over %d single-threaded "
                                          "processes (oracle, %s moduli, r=%d), %.1f s each"
                                          % (cb["steps"], cb["rows"], cb["cols"], cb["k"], procs, args.family, r,
                                             cb["seconds"])}
        # Context: native fp64 matmul on the host cores (numpy's BLAS) on a
        # block of the same product at the full K.
        rb, cbk = min(m, 1024), min(n, 1024)
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
    line["bench_seconds"] = round(time.time() - t_bench0, 1)
    if ws > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def native_dgemm(torch, stream, A, B):
    """cuBLAS DGEMM (torch.matmul on float64) on the same GPU: (ms, result)."""
    m, k = A.shape
    n = B.shape[1]
    cheap = 2.0 * m * n * k < 2e11
    if cheap:
        torch.matmul(A, B)
    else:
        torch.matmul(A[:min(m, 512)], B)
    torch.cuda.synchronize()
    times = []
    C = None
    for _ in range(5 if cheap else 1):
        n0, n1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n0.record(stream)
        C = torch.matmul(A, B)
        n1.record(stream)
        torch.cuda.synchronize()
        times.append(n0.elapsed_time(n1))
    return statistics.median(times), C


def int8_comparison(torch, oz, stream, sh, check, A, B, m, n, k, r, dev, line):
    """The three-limb residue products as one INT8 GEMM per modulus on the
    legacy mma.sync tensor path (the tcgen05 INT8 kind does not exist on
    sm_103a), beside the FP4 digit GEMM on the same residues and cuBLASLt
    INT8 (torch._int_mm) on the same residue matrices."""
    pA, pB = oz.ozemu_bit_budget(k, r)
    sa = torch.empty(m, dtype=torch.int32, device=dev)
    sb = torch.empty(n, dtype=torch.int32, device=dev)
    a8 = torch.empty(oz.ozemu_res8_bytes(m, k, r), dtype=torch.int8, device=dev)
    b8 = torch.empty(oz.ozemu_res8_bytes(n, k, r), dtype=torch.int8, device=dev)
    res8 = torch.empty(oz.ozemu_residue_bytes(m, n, r), dtype=torch.uint8, device=dev)
    res = torch.empty_like(res8)
    ap = torch.empty(oz.ozemu_plane_bytes(m, k, r), dtype=torch.uint8, device=dev)
    bp = torch.empty(oz.ozemu_plane_bytes(n, k, r), dtype=torch.uint8, device=dev)
    check(oz.ozemu_split_rows_f64_res8(m, k, A.data_ptr(), k, pA, r, a8.data_ptr(), sa.data_ptr(), sh), "res8 A")
    check(oz.ozemu_split_cols_f64_res8(k, n, B.data_ptr(), n, pB, r, b8.data_ptr(), sb.data_ptr(), sh), "res8 B")
    check(oz.ozemu_split_rows_f64(m, k, A.data_ptr(), k, pA, r, ap.data_ptr(), sa.data_ptr(), sh), "split A")
    check(oz.ozemu_split_cols_f64(k, n, B.data_ptr(), n, pB, r, bp.data_ptr(), sb.data_ptr(), sh), "split B")
    i8_ms = time_ms(torch, stream, lambda: check(oz.ozemu_residue_gemm_i8(m, n, k, r, a8.data_ptr(), b8.data_ptr(),
                                                                          res8.data_ptr(), sh), "i8 gemm"), reps=3)
    fp4_ms = time_ms(torch, stream, lambda: check(oz.ozemu_residue_gemm(m, n, k, r, ap.data_ptr(), bp.data_ptr(),
                                                                        res.data_ptr(), sh), "fp4 gemm"), reps=3)
    flop = 2.0 * m * n * k
    cmp = {"kernel": "residue_gemm_i8_kernel (mma.sync m16n8k32 s8)", "r": r, "gemm_ms": round(i8_ms, 3),
           "fp4_three_limb_gemm_ms": round(fp4_ms, 3), "fp4_speedup": round(i8_ms / fp4_ms, 2),
           "int8_tops": round(r * flop / (i8_ms / 1e3) / 1e12, 1), "residues_identical": bool(torch.equal(res8, res))}
    fam_gemm = line.get("families", {}).get(line["config"]["family"], {}).get("stage_ms", {}).get("digit_gemm")
    if fam_gemm:
        cmp["headline_family_gemm_ms"] = fam_gemm
    rows_p, k_p = (m + 127) // 128 * 128, (k + 127) // 128 * 128
    cols_p = (n + 127) // 128 * 128
    if hasattr(torch, "_int_mm") and m >= 32 and n >= 8:
        try:
            av, bv = a8.view(r, rows_p, k_p), b8.view(r, cols_p, k_p)
            lt_ms = time_ms(torch, stream, lambda: [torch._int_mm(av[l], bv[l].t()) for l in range(r)], reps=1)
            cmp["cublaslt_int8_ms"] = round(lt_ms, 3)
            cmp["cublaslt_int8_tops"] = round(r * 2.0 * rows_p * cols_p * k_p / (lt_ms / 1e3) / 1e12, 1)
        except RuntimeError as exc:  # shape or build constraints of the library call
            cmp["cublaslt_int8"] = "unavailable: %s" % str(exc).splitlines()[0][:120]
    return cmp


def fp4_mma_rate(torch, oz, stream, sh, check, dev, clk, fp4_peak):
    """The FP4 MMA rate the library's own kernel reaches when nothing else
    limits it: the three-limb CTA-pair digit GEMM (9 MMAs per stage, A reused
    from the collector) on planes of zero digits, 1024 x 4256 outputs (exactly
    76 pair tiles, one per SM pair) for each of r = 13 moduli at k = 16384,
    so every wave is full and the per-tile drain is a small share.  Reported
    per SM and clock against the SM clock sampled during the timed step."""
    m, n, k, r = 1024, 4256, 16384, 13
    ap = torch.zeros(oz.ozemu_plane_bytes(m, k, r), dtype=torch.uint8, device=dev)
    bp = torch.zeros(oz.ozemu_plane_bytes(n, k, r), dtype=torch.uint8, device=dev)
    res = torch.empty(oz.ozemu_residue_bytes(m, n, r), dtype=torch.uint8, device=dev)
    ms = time_ms(torch, stream, lambda: check(oz.ozemu_residue_gemm(m, n, k, r, ap.data_ptr(), bp.data_ptr(),
                                                                    res.data_ptr(), sh), "mma rate"), reps=5)
    flop = 9.0 * r * 2.0 * m * n * k
    tflops = flop / (ms / 1e3) / 1e12
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    out = {"tflops": round(tflops, 1), "ms": round(ms, 3), "shape": "%dx%dx%d, r=%d three-limb" % (m, n, k, r),
           "frac_of_roofline_peak": round(tflops / fp4_peak, 4), "sms": sms}
    if clk.get("sm_mhz"):
        out["mac_per_clk_per_sm_at_sampled_clock"] = round(tflops * 1e12 / 2 / (sms * clk["sm_mhz"] * 1e6), 0)
        out["sampled_sm_mhz"] = clk["sm_mhz"]
    return out


def int_products(torch, oz, stream, sh, check, dev, fp4_peak):
    """The exact integer products at 4096^3: INT8 x INT8 (nine FP4 limb
    products) beside cuBLASLt's INT8 GEMM, and INT4 x INT8 (four plane
    products)."""
    out = {}
    # The exact INT8 x INT8 -> INT32 product (9 FP4 limb GEMMs) on the 4096^3
    # int8 workload, beside cuBLASLt's INT8 GEMM on the same matrices.
    Ai_h, Bi_h = make_pair(4096, 4096, 4096, WORKLOADS["igemm_s8_4096"]["seed"], "int8")
    Ai = torch.from_numpy(Ai_h).to(dev)
    Bi = torch.from_numpy(Bi_h).to(dev)
    Ci = torch.empty((4096, 4096), dtype=torch.int32, device=dev)
    ig_ms = time_ms(torch, stream, lambda: check(oz.ozemu_igemm_s8(4096, 4096, 4096, Ai.data_ptr(), Bi.data_ptr(),
                                                                   Ci.data_ptr(), sh), "igemm"), reps=5)
    iflop = 2.0 * 4096 ** 3
    leg = {"ms": round(ig_ms, 3), "tops": round(iflop / (ig_ms / 1e3) / 1e12, 1),
           "roofline": {"bound": "tensor", "achieved": round(9 * iflop / (ig_ms / 1e3) / 1e12, 1),
                        "peak": round(fp4_peak, 1), "unit": "TFLOP/s",
                        "frac": round(9 * iflop / (ig_ms / 1e3) / 1e12 / fp4_peak, 4)},
           "launches": "split A rows, split B columns, limb GEMM (int32 epilogue)"}
    if hasattr(torch, "_int_mm"):
        ref = torch._int_mm(Ai, Bi)
        lt_ms = time_ms(torch, stream, lambda: torch._int_mm(Ai, Bi), reps=3)
        leg["exact_vs_cublaslt"] = bool(torch.equal(ref, Ci))
        leg["cublaslt_int8_ms"] = round(lt_ms, 3)
    out["igemm_s8_4096"] = leg
    del Ai, Bi, Ci

    # The exact INT4 x INT8 -> INT32 product in four FP4 products (the
    # encoding a b = sum_k g_k u_k(a) v_k(b)) at 4096^3, beside the INT8 x
    # INT8 product's nine on the same shape.
    A4_h, B4_h = make_pair(4096, 4096, 4096, 6, "int4_int8")
    A4 = torch.from_numpy(A4_h).to(dev)
    B4 = torch.from_numpy(B4_h).to(dev)
    C4 = torch.empty((4096, 4096), dtype=torch.int32, device=dev)
    s4_ms = time_ms(torch, stream, lambda: check(oz.ozemu_igemm_s4s8(4096, 4096, 4096, A4.data_ptr(), B4.data_ptr(),
                                                                     C4.data_ptr(), sh), "igemm_s4s8"), reps=5)
    leg4 = {"ms": round(s4_ms, 3), "tops": round(iflop / (s4_ms / 1e3) / 1e12, 1), "fp4_products": 4,
            "roofline": {"bound": "tensor", "achieved": round(4 * iflop / (s4_ms / 1e3) / 1e12, 1),
                         "peak": round(fp4_peak, 1), "unit": "TFLOP/s",
                         "frac": round(4 * iflop / (s4_ms / 1e3) / 1e12 / fp4_peak, 4)},
            "vs_int8_x_int8_9_products": round(ig_ms / s4_ms, 3),
            "launches": "split A rows (4 planes), split B columns (4 planes), plane GEMM (int32 epilogue)",
            "inputs": "A uniform in [-8, 7], B uniform int8, seed 6"}
    # Exactness on a sample of rows: float64 products of these integers are exact.
    rows = np.arange(0, 4096, 257)
    ref = A4_h[rows].astype(np.float64) @ B4_h.astype(np.float64)
    leg4["exact_on_sampled_rows"] = bool(np.array_equal(C4[torch.from_numpy(rows).to(dev)].cpu().numpy(),
                                                        ref.astype(np.int64)))
    out["igemm_s4s8_4096"] = leg4
    del A4, B4, C4
    return out


def other_workloads(torch, oz, fams, stream, sh, check, dev, args, pk, fp4_peak, head_native, clk):
    """Sub-records of the other workloads: each product through the
    library's call for the shape (three-limb with the fused narrow path for
    n <= 2; the headline family otherwise), device-timed, with its roofline
    fraction, the end-to-end call with host buffers, native cuBLAS DGEMM and
    a small exact accuracy sample; the GEMV records add the operational
    intensity against the OI* threshold."""
    out = {}
    fam = fams[args.family]
    native_tflops = None
    for name in ("dgemm_256_uniform", "dgemv_16384_n1", "dgemv_16384_n8", "dgemm_4096_k65536"):
        if name == args.workload:
            continue
        spec = WORKLOADS[name]
        m, n, k = spec["m"], spec["n"], spec["k"]
        A_h, B_h = make_pair(m, n, k, spec["seed"], spec["dist"])
        A = torch.from_numpy(A_h).to(dev)
        B = torch.from_numpy(B_h).to(dev)
        C = torch.empty((m, n), dtype=torch.float64, device=dev)
        flop = 2.0 * m * n * k
        P3 = fams["three"].bits(k, spec["r"])
        narrow = n <= oz.ozemu_narrow_max_n()
        rec = {"m": m, "n": n, "k": k, "dist": spec["dist"]}
        paths = {}
        for key, fm in fams.items():
            rf = fm.r_for(k, P3)
            if rf is None:
                continue
            t = time_ms(torch, stream, lambda: check(fm.dgemm(m, n, k, A.data_ptr(), k, B.data_ptr(), n,
                                                              C.data_ptr(), n, rf, sh), name), reps=5)
            paths[key] = {"r": rf, "fp4_products_per_output": fm.products(rf), "ms": round(t, 4),
                          "tflops": round(flop / (t / 1e3) / 1e12, 3)}
        if oz.ozemu_get_status(sh) != 0:
            raise SystemExit("device status not OK in %s" % name)
        best_key = "three" if narrow else args.family
        best = fams[best_key]
        rb = best.r_for(k, P3)
        rec["path"] = ("three-limb, fused narrow deconstruction + product" if narrow
                       else Family.NAME[best_key])
        rec["r"] = rb
        rec["ms"] = paths[best_key]["ms"]
        rec["tflops"] = paths[best_key]["tflops"]
        rec["paths"] = paths
        # the result whose accuracy is reported
        check(best.dgemm(m, n, k, A.data_ptr(), k, B.data_ptr(), n, C.data_ptr(), n, rb, sh), name)
        # roofline of the dominant kernel
        if narrow:
            res = torch.empty(oz.ozemu_residue_bytes(m, n, rb), dtype=torch.uint8, device=dev)
            sa = torch.empty(m, dtype=torch.int32, device=dev)
            sb = torch.empty(n, dtype=torch.int32, device=dev)
            t = time_ms(torch, stream, lambda: check(oz.ozemu_residues_narrow_f64(
                m, n, k, rb, A.data_ptr(), k, B.data_ptr(), n, res.data_ptr(), sa.data_ptr(), sb.data_ptr(), sh),
                "narrow"), reps=5)
            nbytes = 8.0 * (m * k + k * n) + rb * m * n
            gbs = nbytes / (t / 1e3) / 1e9
            rec["roofline"] = {"bound": "hbm", "kernel": "dgemv_fused_kernel", "ms": round(t, 4),
                               "achieved": round(gbs, 1), "peak": round(pk["hbm_gbs"], 1), "unit": "GB/s",
                               "frac": round(gbs / pk["hbm_gbs"], 4)}
        else:
            pA, pB = best.budget(k, rb)
            ap = torch.empty(best.plane_bytes(m, k, rb), dtype=torch.uint8, device=dev)
            bp = torch.empty(best.plane_bytes(n, k, rb), dtype=torch.uint8, device=dev)
            sa = torch.empty(m, dtype=torch.int32, device=dev)
            sb = torch.empty(n, dtype=torch.int32, device=dev)
            res = torch.empty(oz.ozemu_residue_bytes(m, n, rb), dtype=torch.uint8, device=dev)
            check(best.split_rows(m, k, A.data_ptr(), k, pA, rb, ap.data_ptr(), sa.data_ptr(), sh), "split")
            check(best.split_cols(k, n, B.data_ptr(), n, pB, rb, bp.data_ptr(), sb.data_ptr(), sh), "split")
            t = time_ms(torch, stream, lambda: check(best.residue_gemm(m, n, k, rb, ap.data_ptr(), bp.data_ptr(),
                                                                       res.data_ptr(), sh), "gemm"), reps=5)
            g = best.products(rb) * flop / (t / 1e3) / 1e12
            rec["roofline"] = {"bound": "tensor", "kernel": "digit GEMM", "ms": round(t, 4), "achieved": round(g, 1),
                               "peak": round(fp4_peak, 1), "unit": "TFLOP/s", "frac": round(g / fp4_peak, 4)}
            del ap, bp
        # end to end with host buffers
        A_pin = torch.from_numpy(A_h).pin_memory()
        B_pin = torch.from_numpy(B_h).pin_memory()
        C_pin = torch.empty((m, n), dtype=torch.float64).pin_memory()
        host = oz.ozemu_dgemm_host if narrow else best.dgemm_host
        e = time_ms(torch, stream, lambda: check(host(m, n, k, A_pin.data_ptr(), k, B_pin.data_ptr(), n,
                                                      C_pin.data_ptr(), n, rb, sh), "host"), reps=3)
        if not torch.equal(C_pin.view(torch.int64), C.cpu().view(torch.int64)):
            raise SystemExit("%s: e2e result differs from the device result" % name)
        rec["e2e"] = {"value": round(flop / (e / 1e3) / 1e12, 4), "unit": "TFLOP/s", "ms": round(e, 3),
                      "h2d_bytes_per_step": int(A_h.nbytes + B_h.nbytes), "d2h_bytes_per_step": int(m * n * 8)}
        if not args.no_native:
            nat_ms, Cn = native_dgemm(torch, stream, A, B)
            rec["native_dgemm"] = {"ms": round(nat_ms, 4), "tflops": round(flop / (nat_ms / 1e3) / 1e12, 3),
                                   "emulation_speedup": round(nat_ms / rec["ms"], 2)}
            if name == "dgemm_4096_k65536":
                native_tflops = flop / (nat_ms / 1e3) / 1e12
        if not args.no_accuracy:
            parts = accuracy_sample(m, n, 2, 2, 512, seed=11)
            vals = {"emulated": sample_values(C, parts, dev)}
            if not args.no_native:
                vals["native_dgemm"] = sample_values(Cn, parts, dev)
            rat = bound_ratios(A_h, B_h, parts, vals)
            rec["accuracy"] = {"entries": sample_size(parts, m, n),
                               "sample": "2 full rows, 2 full columns, 512 random entries",
                               "max_err_over_bound": {kk: round(v, 6) for kk, v in rat.items()}}
        rec["operational_intensity"] = round(flop / (8.0 * (m * k + k * n + m * n)), 4)
        out[name] = rec
        del A, B, C
        torch.cuda.empty_cache()
    out.update(int_products(torch, oz, stream, sh, check, dev, fp4_peak))

    # OI* of [TME4] abstract on this GPU: c_q r P_fp64 / (8 P_int), with c_q
    # the split kernel's thread instructions per input element and modulus
    # (ncu, r = 13), P_int the issue rate of the SMs (4 schedulers x 32 lanes
    # per clock) at the clock sampled during the headline step, and P_fp64
    # the native DGEMM rate measured here.
    nat = native_tflops or (head_native or {}).get("tflops")
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    c_q = SPLIT_INSTR_PER_ELEMENT / SPLIT_INSTR_R
    if nat:
        mhz = clk.get("sm_mhz") or 2070.0
        P_int = sms * 4 * 32 * mhz * 1e6
        oi = {}
        for name in ("dgemv_16384_n1", "dgemv_16384_n8"):
            if name in out:
                r = out[name]["r"]
                oi_star = c_q * r * nat * 1e12 / (8.0 * P_int)
                oi[name] = {"r": r, "oi_star": round(oi_star, 3), "operational_intensity":
                            out[name]["operational_intensity"],
                            "below_oi_star": out[name]["operational_intensity"] < oi_star}
        out["oi_star"] = {"c_q": round(c_q, 2), "c_q_source": "split kernel, %g thread instructions per element at "
                          "r = %d (ncu, profiles/split_crt_dgemm_4096_mixed.md)" % (SPLIT_INSTR_PER_ELEMENT,
                                                                                     SPLIT_INSTR_R),
                          "P_fp64_tflops": round(nat, 3), "P_int_per_s": P_int,
                          "P_int_source": "%d SMs x 4 schedulers x 32 lanes x %.0f MHz" % (sms, mhz),
                          "workloads": oi,
                          "formula": "OI* = c_q r P_fp64 / (8 P_int) flop per byte"}
    return out


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle  # the reference arm of this bench is the CPU oracle
    spec = dict(WORKLOADS[args.workload])
    for key in ("m", "n", "k"):
        if getattr(args, key):
            spec[key] = getattr(args, key)
    shape = {"m": spec["m"], "n": spec["n"], "k": spec["k"]}
    k = spec["k"]
    ceil = CEILING_OF[args.family]
    P3 = oracle.bit_budget(k, spec["r"])[0]
    r = args.r
    if r is None:
        r = next(x for x in range(1, 21) if _budget_or_none(oracle, k, x, ceil) is not None
                 and _budget_or_none(oracle, k, x, ceil) >= P3)
    products = sum(oracle.products_per_modulus(l, ceil) for l in range(r))
    bits = oracle.bit_budget(k, r, ceil)[0]
    # warm-up steps are bounded samples too; each step is one sample block.
    if args.warmup:
        cpu_oracle(args.workload, r, 0, max_steps=args.warmup, sample=32, shape=shape, family=args.family)
    cb = cpu_oracle(args.workload, r, 0, max_steps=args.steps, sample=32, shape=shape, family=args.family)
    value = cb["tflops"]
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(1e3 * cb["seconds"] / cb["steps"], 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": bench_config(args, spec, r, products, bits),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                             "sample": "each step a %dx%d block of C at full K=%d (oracle, %s moduli, r=%d, 1 thread)"
                                       % (cb["rows"], cb["cols"], cb["k"], args.family, r)},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _budget_or_none(oracle, k, r, ceil):
    try:
        return oracle.bit_budget(k, r, ceil)[0]
    except ValueError:
        return None


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
