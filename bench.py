"""Benchmark of the preshuffled-weight GEMM on GB300.

Default workload: the FP8 e4m3 per-tensor split-K decode sweep the pages
measure (M in {1,16} x N in {2048,16384}, K=7168; split_k from the dispatch
table), one step = the four GEMMs (mainloop + split-K reduce) back to back.
Metric: decode GEMM GB/s = algorithmic bytes (A + B + scales + Y) / time,
whole job over all ranks.  Other workloads (--workload): the other decode
scale modes, and the large-M shapes (metric TFLOP/s = 2MNK / time).

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
the host cores instead (a bounded sample of the same workload per step).
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import inputs  # noqa: E402

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------- workloads

def _wl(src, first, n, kind):
    """Cases first..first+n-1 of the seeded workload `src` of the inputs module
    (its shapes, splits and seeds, shared with the parity tests)."""
    cases = [dict(inputs.WORKLOADS[src]["cases"][first + i]) for i in range(n)]
    return dict(cases=cases, kind=kind, src=src, first=first)


WORKLOADS = {
    # M=1 N=2048 K=7168 with an explicit split_k of 4
    "fp8_tensor_decode_m1_n2048_k7168_split4": _wl("fp8_tensor_decode_m1_n2048_k7168_split4", 0, 1, "decode"),
    "fp8_tensor_decode_sweep_k7168": _wl("fp8_tensor_decode_sweep_k7168", 0, 4, "decode"),
    "large_bf16_54560x8192x8192": _wl("large_bf16_54560x8192x8192_fp8_4096x4096x8192", 0, 1, "large"),
    "large_fp8_4096x4096x8192": _wl("large_bf16_54560x8192x8192_fp8_4096x4096x8192", 1, 1, "large"),
    "fp8_block128_decode_sweep_k7168": _wl("fp8_block128_decode_sweep_k7168", 0, 4, "decode"),
    "mxfp8_decode_n16384_k7168": _wl("mx_mxfp8_mxfp4_n16384_k7168", 0, 2, "decode"),
    "mxfp4_decode_n16384_k7168": _wl("mx_mxfp8_mxfp4_n16384_k7168", 3, 2, "decode"),
    "large_mxfp8_4096x16384x7168": _wl("mx_mxfp8_mxfp4_n16384_k7168", 2, 1, "large"),
    "large_mxfp4_4096x16384x7168": _wl("mx_mxfp8_mxfp4_n16384_k7168", 5, 1, "large"),
    "mxfp8_b32_decode_n16384_k7168": _wl("mx_mxfp8_b32_n16384_k7168", 0, 2, "decode"),
    "large_mxfp8_b32_4096x16384x7168": _wl("mx_mxfp8_b32_n16384_k7168", 2, 1, "large"),
    "bf16_decode_sweep_k7168": _wl("bf16_decode_sweep_k7168", 0, 4, "decode"),
    "fp8_tensor_decode_m32_k7168": _wl("fp8_tensor_decode_m32_k7168", 0, 2, "decode"),
    "large_fp8_block128_4096x16384x7168": _wl("large_fp8_block128_4096x16384x7168", 0, 1, "large"),
    "large_fp8_block128_4096x8192x7168": _wl("large_fp8_block128_4096x8192x7168", 0, 1, "large"),
    "large_mxfp4_4096x8192x7168": _wl("large_mxfp4_4096x8192x7168", 0, 1, "large"),
    # fp8 activations against fp4 weights, on the MX shapes
    "mxfp4_fp8a_decode_n16384_k7168": _wl("mx_fp8a_fp4w_n16384_k7168", 0, 2, "decode"),
    "large_mxfp4_fp8a_4096x16384x7168": _wl("mx_fp8a_fp4w_n16384_k7168", 2, 1, "large"),
}
DEFAULT_WORKLOAD = "fp8_tensor_decode_sweep_k7168"
MX_MODES = ("mxfp8", "mxfp4", "mxfp8_b32", "mxfp4_fp8a")


def elem_bytes(mode, operand="a"):
    """Bytes per element of operand "a" (activations) or "b" (weights)."""
    if mode == "mxfp4_fp8a":
        return 0.5 if operand == "b" else 1.0
    return {"bf16": 2.0, "mxfp4": 0.5}.get(mode, 1.0)


def scale_bytes(mode, M, N, K):
    if mode == "fp8_tensor":
        return 8
    if mode == "fp8_block128":
        return 4 * (M + N // 128) * (K // 128)
    if mode == "mxfp8":
        return (M + N) * (K // 128)
    if mode in ("mxfp4", "mxfp8_b32", "mxfp4_fp8a"):
        return (M + N) * (K // 32)
    return 0


def algo_bytes(c, n=None):
    """A + B + scales + Y bytes of one GEMM (n restricts to the first n weight rows)."""
    M, N, K, mode = c["M"], c["N"] if n is None else n, c["K"], c["mode"]
    return int(M * K * elem_bytes(mode, "a") + N * K * elem_bytes(mode, "b") + scale_bytes(mode, M, N, K) + 2 * M * N)


def algo_flops(c, n=None):
    return 2.0 * c["M"] * (c["N"] if n is None else n) * c["K"]


def work(kind, c, n=None):
    """The metric's unit of work for one GEMM: bytes (decode) or flops (large)."""
    return algo_flops(c, n) if kind == "large" else algo_bytes(c, n)


METRIC = {"decode": ("decode GEMM GB/s", "GB/s", 1e9), "large": ("large GEMM TFLOP/s", "TFLOP/s", 1e12)}


def case_operands(wl, i):
    """Host operands of case i of a bench workload (seeded as in the inputs module)."""
    return inputs.workload_operands(wl["src"], wl["first"] + i)


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons in the background."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.proc, self.lines = index, None, []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[3:7]):
                if v.lower() in ("active", "1", "yes"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------- oracle arm

class OracleSample:
    """The oracle on a bounded sample of each case, calibrated once so that one
    pass costs about target_s seconds on `threads` host threads.

    Decode cases (M <= 32): all M rows against the first n weight rows (full
    K).  Large cases: the 256 seeded sample rows of A (rows 0 and M-1
    included, as in the parity tests) against the first n weight rows.  n is
    the same fraction of N for every case.  The rate (work / time) is what is
    reported; full-step times are extrapolated from it and labelled so."""

    def __init__(self, wl, host_ops, target_s, threads=None):
        import oracle
        self.oracle = oracle
        self.orc = {"bf16": oracle.BF16, "fp8_tensor": oracle.FP8_TENSOR, "fp8_block128": oracle.FP8_BLOCK128,
                    "mxfp8": oracle.MXFP8, "mxfp4": oracle.MXFP4, "mxfp8_b32": oracle.MXFP8_B32,
                    "mxfp4_fp8a": oracle.MXFP4_FP8A}
        self.wl, self.host_ops = wl, host_ops
        self.threads = threads or os.cpu_count() or 1
        self.large = wl["kind"] == "large"
        self.frac = 1.0 / 4096
        t, _ = self.run()
        self.frac = min(1.0, max(1.0 / 4096, self.frac * target_s / max(t, 1e-6)))

    def rows(self, c):
        return max(8, int(c["N"] * self.frac) // 8 * 8)

    def a_rows(self, c):
        return inputs.sample_rows(c["M"]) if self.large else None

    def run(self):
        t0 = time.perf_counter()
        nbytes = 0
        for c, (A, B, a_s, b_s) in zip(self.wl["cases"], self.host_ops):
            n = self.rows(c)
            bs = b_s
            if c["mode"] == "fp8_block128":
                bs = b_s[: (n + 127) // 128]
            elif c["mode"] in MX_MODES:
                bs = b_s[:n]
            rows = self.a_rows(c)
            self.oracle.gemm(self.orc[c["mode"]], A, B[:n], a_s, bs, M=c["M"], N=n, K=c["K"], rows=rows,
                             threads=self.threads)
            m = c["M"] if rows is None else len(rows)
            nbytes += work(self.wl["kind"], dict(c, M=m), n)
        return time.perf_counter() - t0, nbytes

    def threads_used(self):
        """The oracle shares output rows of A out over its threads: a case with
        fewer rows than threads uses only that many."""
        return max(min(self.threads, len(self.a_rows(c)) if self.large else c["M"]) for c in self.wl["cases"])

    def describe(self):
        what = "the 256 seeded sample rows of A" if self.large else "all M rows"
        return "first %s weight rows of the %s cases (%s, full K) per pass, %d host thread%s asked, at most %d " \
               "busy (the oracle shares rows of A out over threads)" % (
                   "/".join(str(self.rows(c)) for c in self.wl["cases"]), len(self.wl["cases"]), what,
                   self.threads, "" if self.threads == 1 else "s", self.threads_used())


def cpu_baseline(wl, host_ops, kind, unit, scale_u, step_work):
    """The oracle timed on the host cores twice -- single-threaded and on every
    core -- each on its own calibrated sample; value = the all-core rate."""
    out = {}
    for label, threads, target in (("all_cores", os.cpu_count() or 1, 10.0), ("single_thread", 1, 6.0)):
        ref = OracleSample(wl, host_ops, target, threads)
        t, nw = ref.run()
        passes = 1
        while t < 0.5 * target:      # a sample that is already the whole workload: repeat it
            dt, dw = ref.run()
            t, nw, passes = t + dt, nw + dw, passes + 1
        rate = nw / t
        out[label] = {"value": rate / scale_u, "unit": unit, "cores": ref.threads_used(),
                      "sample": ref.describe() + ", %d pass%s in %.2f s" % (passes, "" if passes == 1 else "es", t),
                      "full_step_s_extrapolated": step_work / rate}
    allc = out["all_cores"]
    return {"value": allc["value"], "unit": unit, "cores": allc["cores"], "kind": "oracle",
            "sample": allc["sample"], "single_thread": out["single_thread"],
            "full_step_s_extrapolated": {
                "all_cores": allc["full_step_s_extrapolated"],
                "single_thread": out["single_thread"]["full_step_s_extrapolated"],
                "how": "EXTRAPOLATED, not measured: sample time x (work of one full step / work of the "
                       "sample)%s" % (" (x M/256 for the rows of A)" if kind == "large" else "")},
            "host_cores": os.cpu_count()}


# ---------------------------------------------------------- multi-rank

def aggregate_ranks(ms, world, dist=None, device=None):
    """Timed-region milliseconds of the slowest rank (every rank calls it)."""
    if world <= 1:
        return ms
    import torch
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(steps, step_work, ms, world, unit_scale):
    """Work of all ranks over the slowest rank's time (replicas: weak scaling)."""
    return world * steps * step_work / (ms / 1e3) / unit_scale


# ----------------------------------------------------------- ncu traffic

TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def _code_only(text):
    """C/C++ source with its comments and all whitespace removed (string
    literals kept), so that edits to comments leave the digest unchanged."""
    import re
    tok = re.compile(r'"(?:\\.|[^"\\])*"|//[^\n]*|/\*.*?\*/|\s+', re.S)
    return tok.sub(lambda m: m.group(0) if m.group(0).startswith('"') else "", text)


def kernel_sources_digest(fg):
    """Digest of the library's kernel sources (code only, comments and
    whitespace ignored), to tell whether a stored ncu traffic figure still
    describes the kernels being timed."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(os.path.dirname(fg.__file__), "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh")):
            h.update(name.encode())
            h.update(_code_only(open(os.path.join(csrc, name), encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


def traffic(workload, fg):
    """DRAM bytes (read + write) per step of the dominant kernel from the
    committed ncu summary, or None when there is none for these sources."""
    try:
        rec = json.load(open(TRAFFIC_FILE)).get(workload)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("sources") != kernel_sources_digest(fg):
        return None
    return rec.get("dram_bytes_per_step")


# ------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None, help="timed steps (default per workload)")
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", default="fg", choices=["fg", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--rotate", type=int, default=None, help="operand copies cycled to keep L2 cold")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    wl = WORKLOADS[args.workload]
    kind = wl["kind"]
    if args.steps is None:
        args.steps = 3000 if kind == "decode" else 40
    if args.warmup is None:
        args.warmup = 20 if kind == "decode" else 5
    args.warmup = max(3, args.warmup)
    if args.rotate is None:
        args.rotate = 3 if kind == "decode" else (1 if wl["cases"][0]["M"] * wl["cases"][0]["K"] > 2e8 else 4)
    metric, unit, scale_u = METRIC[kind]

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    peaks = dict(FALLBACK_PEAKS)
    peaks_src = "fallback"
    if os.path.exists(PEAKS_FILE):
        try:
            peaks.update(json.load(open(PEAKS_FILE)))
            peaks_src = "measured"
        except ValueError:
            pass
    host_ops_fn = lambda: [case_operands(wl, i) for i in range(len(wl["cases"]))]  # noqa: E731
    dtype = {"bf16": "bf16", "fp8_tensor": "e4m3", "fp8_block128": "e4m3", "mxfp8": "e4m3",
             "mxfp4": "e2m1", "mxfp8_b32": "e4m3", "mxfp4_fp8a": "e4m3xe2m1"}[wl["cases"][0]["mode"]]

    if args.impl == "reference":
        if rank != 0:
            return
        host_ops = host_ops_fn()
        budget = 90.0 / max(1, args.steps + args.warmup)   # whole run ~1.5 min
        ref = OracleSample(wl, host_ops, budget)
        times, total = [], 0.0
        for s in range(args.warmup + args.steps):
            t, nw = ref.run()
            if s >= args.warmup:
                times.append(t)
                total += nw
        tsum = sum(times)
        value = total / tsum / scale_u
        line = {"metric": metric, "value": value, "unit": unit, "impl": "reference",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": 1000 * tsum / len(times), "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": args.workload, "cases": wl["cases"]},
                "cpu_baseline": {"value": value, "unit": unit, "cores": ref.threads_used(), "kind": "oracle",
                                 "sample": ref.describe()},
                "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    import torch
    import torch.distributed as dist

    import mx_gemm_gb300 as fg

    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)

    def to_dev(x):
        if x is None:
            return None
        x = np.ascontiguousarray(x)
        return torch.from_numpy(x.view(np.int16) if x.dtype == np.uint16 else x).to(dev)

    # operands: `rotate` copies of every activation and preshuffled weight
    host_ops = host_ops_fn()
    cases = []
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    for c, (A, B, a_s, b_s) in zip(wl["cases"], host_ops):
        dB, db_s = to_dev(B), to_dev(b_s)
        # enough weight copies that a case timed on its own cycles through
        # more than twice the L2 (a small weight would stay resident otherwise)
        wb = c["N"] * c["K"] * elem_bytes(c["mode"])
        R = max(1, args.rotate, -(-2 * l2_bytes // int(wb)) if kind == "decode" else 1)
        pbs = [fg.preshuffle_b(c["mode"], dB, db_s, K=c["K"]) for _ in range(R)]
        del dB
        dA0 = to_dev(A)
        dAs = [dA0] + [dA0.clone() for _ in range(R - 1 if kind == "large" else 0)]
        plan = fg.gemm_plan(c["mode"], c["M"], c["N"], c["K"], c.get("split_k", 0))
        S = plan["split_k"]
        ws_bytes = fg.gemm_workspace_size(c["mode"], c["M"], c["N"], c["K"], c.get("split_k", 0))
        ws = torch.empty(max(4, ws_bytes) // 4, dtype=torch.float32, device=dev)
        Y = torch.empty((c["M"], c["N"]), dtype=torch.bfloat16, device=dev)
        hA = torch.from_numpy(np.ascontiguousarray(A).view(np.int16) if A.dtype == np.uint16 else
                              np.ascontiguousarray(A)).pin_memory()
        ha_s = torch.from_numpy(np.ascontiguousarray(a_s)).pin_memory() if a_s is not None else None
        red_as = to_dev(a_s) if c["mode"] == "fp8_tensor" else None
        # calls pass the case's own split_k (0: the dispatch's choice, which may
        # be the balanced form that an explicit split would turn off)
        cases.append(dict(c=c, pbs=pbs, dAs=dAs, S=S, call_split=c.get("split_k", 0), ws=ws, Y=Y,
                          da_s=to_dev(a_s), hA=hA, ha_s=ha_s, plan=plan, work=work(kind, c), red_as=red_as))
    torch.cuda.synchronize()

    def one_case(x, r):
        st = torch.cuda.current_stream()
        pb = x["pbs"][r % len(x["pbs"])]
        dA = x["dAs"][r % len(x["dAs"])]
        fg.gemm(dA, pb, x["da_s"], split_k=x["call_split"], Y=x["Y"], workspace=x["ws"], stream=st)

    def step(r):
        for x in cases:
            one_case(x, r)

    def graph_of(fn, n):
        """Capture fn(0..n-1) into one CUDA graph (the launches of a decode
        step are short enough that host launch latency would otherwise show)."""
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=cap):
            for r in range(n):
                fn(r)
        torch.cuda.synchronize()
        g.replay()                          # one untimed replay
        torch.cuda.synchronize()
        return g

    def time_graph(g):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        st = torch.cuda.current_stream()
        e0.record(st)
        g.replay()
        e1.record(st)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    for w in range(args.warmup):
        step(w)
    torch.cuda.synchronize()
    if fg.get_error() != fg.FG_OK:
        raise RuntimeError("kernel error word set during warm-up")

    # ---------------- timed region: one replay of a graph of the K steps
    K = args.steps
    graph = graph_of(step, K)
    stream = torch.cuda.current_stream()
    clk = ClockSampler(local_rank)
    clk.start()
    time.sleep(0.2)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    graph.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = clk.stop()
    ms = t0.elapsed_time(t1)
    del graph
    ms = aggregate_ranks(ms, world, dist, dev)
    if fg.get_error() != fg.FG_OK:
        raise RuntimeError("kernel error word set during the timed region")
    step_work = sum(x["work"] for x in cases)
    value = whole_job_value(K, step_work, ms, world, scale_u)

    # ---------------- per case: the main kernel alone, back to back (a graph
    # of the same call repeated, CUDA events around its replay)
    per_case, main_ms = [], []
    for x in cases:
        n = max(20, min(K, 400))
        g = graph_of(lambda r, x=x: one_case(x, r), n)
        avg = time_graph(g) / n
        del g
        main_ms.append(avg)
        per_case.append({"mode": x["c"]["mode"], "M": x["c"]["M"], "N": x["c"]["N"], "K": x["c"]["K"],
                         "split_k": x["S"], "path": x["plan"]["path"], "kernel": x["plan"]["name"],
                         "us": round(avg * 1e3, 3),
                         unit.replace("/", "p"): round(x["work"] / (avg / 1e3) / scale_u, 1)})
    achieved = step_work / (sum(main_ms) / 1e3) / scale_u
    if kind == "decode":
        # The shape's own bandwidth wall: a device-to-device copy whose read +
        # write bytes equal the GEMM's algorithmic bytes, timed the same way
        # (back to back in a graph, cycling through buffers larger than twice
        # the L2), so each shape's GB/s sits beside what a plain stream of the
        # same size reaches.  The copy is an SM kernel (a float32 elementwise
        # op) rather than a memcpy node, which a graph may hand to a copy engine.
        for x, pc in zip(cases, per_case):
            nb = max(16, x["work"] // 2 // 16 * 16)
            R = max(2, -(-2 * l2_bytes // nb) + 1)
            src = [torch.zeros(nb // 4, dtype=torch.float32, device=dev) for _ in range(R)]
            dst = [torch.zeros(nb // 4, dtype=torch.float32, device=dev) for _ in range(R)]
            n = max(20, min(K, 400))
            g = graph_of(lambda r: torch.mul(src[(r + 1) % R], 1.0, out=dst[r % R]), n)
            cms = time_graph(g) / n
            del g, src, dst
            copy_gbs = 2 * nb / (cms / 1e3) / 1e9
            pc["copy_us"] = round(cms * 1e3, 3)
            pc["copy_GBps"] = round(copy_gbs, 1)
            pc["frac_of_copy"] = round(pc["GBps"] / copy_gbs, 4)
    if kind == "decode":
        bound, peak, psrc = "hbm", float(peaks["hbm_gbs"]), peaks_src + " hbm_gbs (burst copy)"
    else:
        # the measured bf16 rate times the nominal dense ratio of the operand
        # type (fp8 4.5 and fp4 13.5 vs bf16 2.25 PFLOP/s; fp8 x fp4 runs at
        # the fp8 rate): the burst figure for a timed region shorter than a
        # second, the sustained (power-capped) one for a longer region
        ratio = {"bf16": 1.0, "e4m3": 2.0, "e2m1": 6.0, "e4m3xe2m1": 2.0}[dtype]
        which = "bf16_tflops_sustained" if ms >= 1000.0 else "bf16_tflops"
        bound, peak = "tensor", ratio * float(peaks[which])
        psrc = peaks_src + " " + which + " (timed region %.0f ms)" % ms + (
            " x %g (%s/bf16 nominal dense ratio)" % (ratio, dtype) if ratio != 1 else "")

    # ---------------- end-to-end: the public API call per case with the
    # activation copied from pinned host memory before it and Y copied back
    # after it, every step -- once as a serving loop issues decode steps (a
    # CUDA graph; step s+1's inputs go over and step s-1's outputs come back
    # on copy streams while step s computes, two device buffer sets) and once
    # as plain eager calls, copies and GEMMs one after the other.
    E = max(3, K // 10)

    # The step's inputs (every case's activation and activation scales) sit in
    # one pinned host buffer and go over in one copy; the step's outputs come
    # back in one copy.  The GEMMs read and write views of the two device
    # buffers.
    def pack(tensors):
        offs, off = [], 0
        for t in tensors:
            offs.append(off)
            off += -(-t.numel() * t.element_size() // 256) * 256
        return offs, max(off, 256)

    ins = []
    for x in cases:
        ins.append(x["hA"])
        if x["ha_s"] is not None:
            ins.append(x["ha_s"])
    in_offs, in_bytes = pack(ins)
    h_in = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
    d_ins = [torch.empty(in_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    out_offs, out_bytes = pack([x["Y"] for x in cases])
    d_outs = [torch.empty(out_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    h_outs = [torch.empty(out_bytes, dtype=torch.uint8).pin_memory() for _ in range(2)]
    d_in, d_out, h_out = d_ins[0], d_outs[0], h_outs[0]

    def view(buf, off, like):
        n = like.numel() * like.element_size()
        return buf[off:off + n].view(like.dtype).view(like.shape)

    k = 0
    for i, x in enumerate(cases):
        view(h_in, in_offs[k], x["hA"]).copy_(x["hA"])
        x["e_A"] = [view(b, in_offs[k], x["hA"]) for b in d_ins]
        k += 1
        x["e_as"] = [None, None]
        if x["ha_s"] is not None:
            view(h_in, in_offs[k], x["ha_s"]).copy_(x["ha_s"])
            x["e_as"] = [view(b, in_offs[k], x["ha_s"]) for b in d_ins]
            k += 1
        x["e_Y"] = [view(b, out_offs[i], x["Y"]) for b in d_outs]
    h2d, d2h = in_bytes, out_bytes
    copy_in, copy_out = torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_pipeline(n):
        """n steps; step s uses buffer set s % 2.  Edges: H2D(s+1) after the
        GEMMs of s-1 (last readers of its set); GEMMs(s) after H2D(s) and after
        D2H(s-2) (last reader of its output set); D2H(s) after GEMMs(s)."""
        main = torch.cuda.current_stream()
        fork = torch.cuda.Event()
        fork.record(main)
        copy_in.wait_event(fork)
        copy_out.wait_event(fork)
        h2d_ev = [torch.cuda.Event() for _ in range(n)]
        done_ev = [torch.cuda.Event() for _ in range(n)]
        d2h_ev = [torch.cuda.Event() for _ in range(n)]
        with torch.cuda.stream(copy_in):
            d_ins[0].copy_(h_in, non_blocking=True)
            h2d_ev[0].record(copy_in)
        for s in range(n):
            b = s % 2
            if s + 1 < n:
                with torch.cuda.stream(copy_in):
                    if s >= 1:
                        copy_in.wait_event(done_ev[s - 1])
                    d_ins[(s + 1) % 2].copy_(h_in, non_blocking=True)
                    h2d_ev[s + 1].record(copy_in)
            main.wait_event(h2d_ev[s])
            if s >= 2:
                main.wait_event(d2h_ev[s - 2])
            for x in cases:
                fg.gemm(x["e_A"][b], x["pbs"][s % len(x["pbs"])], x["e_as"][b], split_k=x["call_split"], Y=x["e_Y"][b],
                        workspace=x["ws"], stream=main)
            done_ev[s].record(main)
            with torch.cuda.stream(copy_out):
                copy_out.wait_event(done_ev[s])
                h_outs[b].copy_(d_outs[b], non_blocking=True)
                d2h_ev[s].record(copy_out)
        main.wait_stream(copy_in)
        main.wait_stream(copy_out)

    def e2e_step(s):
        st = torch.cuda.current_stream()
        d_in.copy_(h_in, non_blocking=True)
        for x in cases:
            fg.gemm(x["e_A"][0], x["pbs"][s % len(x["pbs"])], x["e_as"][0], split_k=x["call_split"], Y=x["e_Y"][0],
                    workspace=x["ws"], stream=st)
        h_out.copy_(d_out, non_blocking=True)

    g_e2e = graph_of(lambda r: e2e_pipeline(E), 1)
    e2e_ms = aggregate_ranks(time_graph(g_e2e), world, dist, dev)
    del g_e2e
    # every step computes the same product (identical inputs, identical weight
    # copies): both host output buffers must hold the timed path's Y bit for bit
    for i, x in enumerate(cases):
        y_ref = x["Y"].cpu()
        for hb in h_outs:
            if not torch.equal(view(hb, out_offs[i], x["Y"]).view(torch.int16), y_ref.view(torch.int16)):
                raise RuntimeError("end-to-end output differs from the timed path's (case %d)" % i)
    e2e_value = whole_job_value(E, step_work, e2e_ms, world, scale_u)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s in range(E):
        e2e_step(s)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_eager = whole_job_value(E, step_work, aggregate_ranks(e0.elapsed_time(e1), world, dist, dev), world,
                                scale_u)

    # + the per-call A scale relayout of the large MX form
    launches_per_step = sum((2 if x["S"] > 8 else 1) +
                            (1 if x["plan"]["path"] == 1 and x["c"]["mode"] in MX_MODES else 0)
                            for x in cases)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, host_ops, kind, unit, scale_u, step_work)

    if rank == 0:
        wbytes = sum(x["c"]["N"] * x["c"]["K"] * elem_bytes(x["c"]["mode"]) for x in cases)
        abytes = sum(x["c"]["M"] * x["c"]["K"] * elem_bytes(x["c"]["mode"]) for x in cases)
        line = {
            "metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": dtype, "data": "synthetic",
            "config": {"workload": args.workload,
                       "shapes": [[x["c"]["M"], x["c"]["N"], x["c"]["K"]] for x in cases],
                       "l2": "inputs larger than L2: every case cycles through copies of its operands "
                             "(%s copies) so that more than twice the L2 (%d MB) passes between reuses; "
                             "%.0f MB of weights per step" % ("/".join(str(len(x["pbs"])) for x in cases),
                                                              l2_bytes // 10**6, wbytes / 1e6),
                       "parallelism": "replicas" if world > 1 else "single"},
            "per_case": per_case,
            "roofline": {"bound": bound, "achieved": round(achieved, 1), "peak": peak, "unit": unit,
                         "frac": round(achieved / peak, 4), "traffic": traffic(args.workload, fg),
                         "peak_source": psrc,
                         "kernel": "the GEMM's main kernel, per case timed back to back, work summed over "
                                   "the cases"},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "how": "public API calls with one pinned-host H2D of the step's activations and scales "
                           "and one D2H of its outputs every step, captured in one CUDA graph as a serving "
                           "loop: step s+1's H2D and step s-1's D2H run on copy streams while step s computes "
                           "(two device buffer sets); the first H2D and the last D2H are inside the timed region"},
            "e2e_eager": {"value": e2e_eager, "unit": unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                          "how": "the same calls issued eagerly from Python, each step's H2D, GEMMs and D2H "
                                 "one after the other on one stream"},
            "gpu_launches": launches_per_step * K,
            "clocks": clocks,
            "timed_region": "one CUDA-graph replay of the %d steps" % K,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
