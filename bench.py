#!/usr/bin/env python
"""Throughput of C = A_sparse @ B_dense on GB300, one JSON line on stdout.

Headline workload: A 8192 x 8192 int8 in 2:4 form (exactly two nonzeros in
every group of four along K), B 8192 x 4096 int8, C int32 (exact).  A step is
one spmm_24 call with A (already compressed) and B resident in HBM; the L2 is
flushed (256 MiB written) before every timed step.  Metric: effective
TFLOP/s = 2 * nnz * N / time.

The same line carries, per other workload (BCSR LLM-shaped, tile-vector-wise,
row-window CSR, fp16 2:4, 6:8 through overlapping 2:4 windows, a scrambled band
multiplied after Reverse Cuthill-McKee, SDDMM on the row-window pattern, the two
pruning builders, BCSR tiny), its own time, TFLOP/s, GB/s and roofline fraction.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs the same workload on its own GPU (independent
replicas: the path has no exchange step); time is the max over ranks and
`value` counts the work of all ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "SpMM effective TFLOP/s (2·nnz·N/time) and % of roofline, per sparse format"
HEADLINE = "mask24_int8"
EXTRA_WORKLOADS = ("bcsr_llm", "tvw", "wcsr_lognormal", "wcsr_clustered", "mask24_f16", "mask24_e4m3", "slide68_f16", "bcsr_rcm",
                   "sddmm_lognormal", "sddmm_lognormal_i8", "prune24_f16", "prune_tvw_f16", "bcsr_tiny")
FLUSH_BYTES = 256 << 20
# L2 -> SM gather ceiling (GB/s): 256-byte rows read at random row indices from a
# 24 MB L2-resident buffer, half-warp per row, 64 warps per SM, four rows in
# flight per half-warp; measured on this machine's GB300 (21.0 TB/s; streaming
# 16-byte loads over the same buffer reached 15.5 TB/s).  The gathering kernels
# (TVW's kept B rows, row-window and SDDMM rows) are reported against it beside
# their HBM / tensor roofline.
L2_GATHER_GBS = 21000.0
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------------ helpers
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def _code_only(src: str) -> str:
    """C/C++/CUDA source without comments or blank-line changes: what the compiler sees."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c == '"' or c == "'":                      # string or character literal
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "\n".join(line.rstrip() for line in "".join(out).splitlines() if line.strip())


def source_sha(*rel):
    """Hash of the kernel sources' code (comments and blank lines ignored), so a
    recorded DRAM traffic figure stays attached to the code it was measured on."""
    h = hashlib.sha256()
    for r in rel:
        with open(os.path.join(ROOT, r), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


KERNEL_SOURCES = {
    "sparse_spmm_kernel": ("sparse_dense_matrix_spmm_gb300/csrc/spmm24.cu", "sparse_dense_matrix_spmm_gb300/csrc/sm103.cuh"),
    "bcsr_spmm_kernel": ("sparse_dense_matrix_spmm_gb300/csrc/bcsr.cu", "sparse_dense_matrix_spmm_gb300/csrc/sm103.cuh"),
    "wcsr_spmm_kernel": ("sparse_dense_matrix_spmm_gb300/csrc/wcsr.cu", "sparse_dense_matrix_spmm_gb300/csrc/sm103.cuh"),
    "wcsr_tc_kernel": ("sparse_dense_matrix_spmm_gb300/csrc/wcsr.cu", "sparse_dense_matrix_spmm_gb300/csrc/sm103.cuh"),
    "wcsr_ts_kernel": ("sparse_dense_matrix_spmm_gb300/csrc/wcsr.cu", "sparse_dense_matrix_spmm_gb300/csrc/sm103.cuh"),
    "sddmm_kernel": ("sparse_dense_matrix_spmm_gb300/csrc/sddmm.cu",),
}


def measured_traffic(kernel, workload):
    """DRAM bytes per launch from a committed ncu capture, if the kernel is unchanged since."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(f"{kernel}|{workload}")
    if not e:
        return None
    try:
        if e.get("source_sha") != source_sha(*KERNEL_SOURCES[kernel]):
            return None
    except OSError:
        return None
    return e.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
                power.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None, "samples": len(sm), "reasons": sorted(reasons)}


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws, device):
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(ws, flops_per_step, steps, max_total_ms):
    """Throughput of the whole job: every rank ran `steps` steps of `flops_per_step`
    useful flops; the slowest rank's time is the job's time."""
    return ws * flops_per_step * steps / (max_total_ms / 1e3) / 1e12


# ------------------------------------------------------------------ workloads (ours)
def to_dev(bits, torch_dtype=None):
    import torch
    if bits.dtype == np.int8:
        return torch.from_numpy(np.ascontiguousarray(bits)).cuda()
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()
    return t.view(torch_dtype) if torch_dtype is not None else t


# Steps run again with the library's per-kernel trace on, for the kernels' own
# times and launch counts.  The timed steps themselves run without those events
# (a pair per kernel launch: about 9 us per headline step, 2.5%).
TRACED_STEPS = 5


def traced_pass(step, flush_buf, ws):
    import sparse_dense_matrix_spmm_gb300 as spmm
    spmm.trace_enable(True)
    timed_steps(step, TRACED_STEPS, 0, flush_buf, ws)


def timed_steps(step, steps, warmup, flush_buf, ws):
    """Warm up, then time exactly `steps` steps with CUDA events (L2 flushed before each)."""
    import torch
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in evs:
        flush_buf.zero_()
        a.record()
        step()
        b.record()
    torch.cuda.synchronize()
    barrier(ws)
    return sum(a.elapsed_time(b) for a, b in evs)


# Dense fp8 tensor rate relative to bf16 (nominal 4.5 vs 2.25 PFLOP/s): no fp8 GEMM
# is measured on this machine, so the fp8 peak is the measured bf16 figure times this.
FP8_OVER_BF16 = 2.0


def roofline(flops, alg_bytes, t_s, peaks, prefer=None, traffic=None, peak_kind="burst", peak_scale=1.0):
    """Roofline object for one kernel: bound = the larger of the two time floors.
    peak_scale multiplies the measured bf16 tensor peak (FP8_OVER_BF16 for fp8)."""
    P = peaks["bf16_tflops"] if peak_kind == "burst" else peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    P = P * peak_scale
    BW = peaks["hbm_gbs"]
    t_tensor = flops / (P * 1e12)
    t_hbm = alg_bytes / (BW * 1e9)
    bound = prefer or ("tensor" if t_tensor >= t_hbm else "hbm")
    if bound == "tensor":
        ach = flops / t_s / 1e12
        return {"bound": "tensor", "achieved": round(ach, 2), "peak": P, "unit": "TFLOP/s",
                "frac": round(ach / P, 4), "traffic": traffic}
    ach = alg_bytes / t_s / 1e9
    return {"bound": "hbm", "achieved": round(ach, 1), "peak": BW, "unit": "GB/s", "frac": round(ach / BW, 4),
            "traffic": traffic}


def run_headline(args, ws, rank, local, peaks, flush_buf):
    import torch
    import spmm_inputs as gen
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.config_problem(HEADLINE)
    M, K, N = p["M"], p["K"], p["N"]
    nnz = M * K // 2
    flops = 2.0 * nnz * N
    A = to_dev(p["A"])
    B = to_dev(p["B"])
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    # the format: compressed int8 values and metadata, plus the values widened to
    # fp16 once (a step widens only B)
    F = spmm.spmm_widen_24(spmm.spmm_compress_24(A))
    torch.cuda.synchronize()
    build_ms = (time.perf_counter() - t0) * 1e3
    del A
    Cd = torch.empty((M, N), dtype=torch.int32, device="cuda")
    wsz = spmm.spmm_24_workspace_size(F, N)
    wsp = torch.empty(wsz, dtype=torch.uint8, device="cuda")

    def step():
        spmm.spmm_24(F, B, Cd, wsp)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    spmm.trace_enable(False)
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    total_ms = timed_steps(step, args.steps, 0, flush_buf, ws)
    clocks = sampler.stop()
    traced_pass(step, flush_buf, ws)
    n_sp, ms_sp = spmm.trace_read(spmm._lib.KERNEL_SPARSE)
    n_wd, ms_wd = spmm.trace_read(spmm._lib.KERNEL_WIDEN)
    spmm.trace_enable(False)
    total_ms = max_over_ranks(total_ms, ws, "cuda")
    ms_step = total_ms / args.steps
    value = whole_job_tflops(ws, flops, args.steps, total_ms)
    t_kernel = ms_sp / max(n_sp, 1) / 1e3
    alg_bytes = nnz * 1 + M * K // 8 + K * N + M * N * 4
    rl = roofline(flops, alg_bytes, t_kernel, peaks, prefer="tensor",
                  traffic=measured_traffic("sparse_spmm_kernel", HEADLINE))
    rl["kernel"] = "sparse_spmm_kernel<dense B, int-exact>"
    rl["kernel_ms"] = round(t_kernel * 1e3, 4)
    rl["widen_ms"] = round(ms_wd / max(n_wd, 1), 4)

    # End to end through the public API: every step copies B in from pinned host
    # memory and the int32 C out to pinned host memory.  Consecutive steps overlap
    # on three streams (copy in / compute / copy out) with double-buffered device
    # and host buffers, as a serving loop would run them.  The per-step footprint
    # (B, widened operands, C: ~340 MB) is larger than L2, so no flush is needed.
    Bh = torch.from_numpy(p["B"]).pin_memory()
    Chs = [torch.empty((M, N), dtype=torch.int32).pin_memory() for _ in range(2)]
    Bds = [torch.empty_like(B) for _ in range(2)]
    Cds = [Cd, torch.empty_like(Cd)]
    s_cmp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_run(n):
        for i in range(n):
            j = i % 2
            if i >= 2:
                s_in.wait_event(ev_cmp[j])  # step i-2 is done reading Bds[j]
            with torch.cuda.stream(s_in):
                Bds[j].copy_(Bh, non_blocking=True)
                ev_in[j].record(s_in)
            s_cmp.wait_event(ev_in[j])
            if i >= 2:
                s_cmp.wait_event(ev_out[j])  # step i-2's C has left Cds[j]
            spmm.spmm_24(F, Bds[j], Cds[j], wsp)
            ev_cmp[j].record(s_cmp)
            s_out.wait_event(ev_cmp[j])
            with torch.cuda.stream(s_out):
                Chs[j].copy_(Cds[j], non_blocking=True)
                ev_out[j].record(s_out)
        s_cmp.wait_event(ev_out[(n - 1) % 2])
        s_cmp.wait_event(ev_in[(n - 1) % 2])

    n_e2e = max(3, min(args.steps, 10))
    e2e_run(2)
    torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_start.record(s_cmp)
    s_in.wait_stream(s_cmp)
    s_out.wait_stream(s_cmp)
    e2e_run(n_e2e)
    e_end.record(s_cmp)
    torch.cuda.synchronize()
    barrier(ws)
    e2e_ms = max_over_ranks(e_start.elapsed_time(e_end), ws, "cuda")
    e2e = {"value": round(whole_job_tflops(ws, flops, n_e2e, e2e_ms), 3), "unit": "TFLOP/s",
           "h2d_bytes_per_step": int(Bh.numel() * Bh.element_size()),
           "d2h_bytes_per_step": int(Chs[0].numel() * Chs[0].element_size()),
           "ms_per_step": round(e2e_ms / n_e2e, 4),
           "overlap": "copy in, compute and copy out of consecutive steps on three streams",
           "l2": "per-step footprint larger than L2, not flushed",
           "result_matches_device": bool(torch.equal(Chs[(n_e2e - 1) % 2], Cd.cpu()))}
    # the sparse kernel and one widening launch per call, counted over the traced steps
    launches = round((n_sp + n_wd) * args.steps / TRACED_STEPS) * ws
    return {"value": value, "ms_step": ms_step, "roofline": rl, "clocks": clocks, "e2e": e2e,
            "build_ms": build_ms, "launches": launches, "M": M, "K": K, "N": N, "nnz": nnz, "problem": p}


def run_extra(name, args, ws, peaks, flush_buf):
    """One of the other measured workloads: time, TFLOP/s, GB/s, roofline."""
    import torch
    import spmm_inputs as gen
    import sparse_dense_matrix_spmm_gb300 as spmm
    c = dict(gen.CONFIGS[name])
    if args.n:
        c["N"] = args.n
    steps = max(3, min(args.steps, 10))
    g = torch.Generator(device="cuda")
    g.manual_seed(int(c["seed"]))
    extra_fields = {}
    gathered = 0  # bytes a launch gathers from L2 row by row (reported against L2_GATHER_GBS)
    peak_scale = 1.0
    if c["kind"] == "bcsr":
        p = gen.bcsr_problem(c["M"], c["K"], 8, c["bh"], c["bw"], c["nnzb"], c["seed"], c["dtype"], c["std"])
        dt = torch.bfloat16 if c["dtype"] == "bf16" else torch.float16
        A = to_dev(p["A"], dt)
        Bx = torch.randn((c["K"], c["N"]), generator=g, device="cuda", dtype=torch.float32).to(dt)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        F = spmm.build_bcsr(A, c["bh"], c["bw"])
        torch.cuda.synchronize()
        build_ms = (time.perf_counter() - t0) * 1e3
        del A
        Cd = torch.empty((c["M"], c["N"]), dtype=torch.float32, device="cuda")
        nnz = F.nnzb * c["bh"] * c["bw"]
        alg = nnz * 2 + F.nnzb * 4 + (c["M"] // c["bh"] + 1) * 4 + c["K"] * c["N"] * 2 + c["M"] * c["N"] * 4
        kern, kid = "bcsr_spmm_kernel", spmm._lib.KERNEL_BCSR

        def step():
            spmm.spmm_bcsr(F, Bx, Cd)
    elif c["kind"] == "tvw":
        p = gen.config_problem(name, **({"N": args.n} if args.n else {}))
        A = to_dev(p["A"], torch.float16)
        Bx = to_dev(p["B"], torch.float16)
        tp = to_dev(p["tile_ptr"])
        cl = to_dev(p["cols"])
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        F = spmm.spmm_build_tvw(A, c["tile_rows"], tp, cl, Kp=c["keep"])
        torch.cuda.synchronize()
        build_ms = (time.perf_counter() - t0) * 1e3
        del A
        Cd = torch.empty((c["M"], c["N"]), dtype=torch.float32, device="cuda")
        nnz = c["M"] * c["keep"] // 2
        alg = nnz * 2 + c["M"] * c["keep"] // 8 + int(p["cols"].size) * 4 + c["K"] * c["N"] * 2 + \
            c["M"] * c["N"] * 4
        kern, kid = "sparse_spmm_kernel", spmm._lib.KERNEL_SPARSE
        # every (row tile, 128-column tile) gathers its tile's kept B rows: kept x N x 2 bytes per row tile
        gathered = int(np.diff(p["tile_ptr"]).sum()) * c["N"] * 2

        def step():
            spmm.spmm_tvw(F, Bx, Cd)
    elif c["kind"] == "24f":
        # the same recipe as the host generator, drawn on the device (the bench checks no values):
        # per 4-group one of the 6 position pairs, N(0,1) values; B N(0,1); fp16 or fp8 E4M3
        M, K = c["M"], c["K"]
        fp8 = c.get("dtype") == "e4m3"
        tdt = torch.float8_e4m3fn if fp8 else torch.float16
        pat = torch.tensor([0b0011, 0b0101, 0b1001, 0b0110, 0b1010, 0b1100], device="cuda")
        sel = pat[torch.randint(0, 6, (M, K // 4), generator=g, device="cuda")]
        bit = torch.arange(4, device="cuda")
        keep = ((sel[:, :, None] >> bit) & 1).bool().reshape(M, K)
        A = (torch.randn((M, K), generator=g, device="cuda") * keep).to(tdt)
        del sel, keep
        Bx = torch.randn((K, c["N"]), generator=g, device="cuda").to(tdt)
        if fp8:
            peak_scale = FP8_OVER_BF16
            extra_fields["peak_note"] = (f"fp8 peak derived: {FP8_OVER_BF16:g} x the measured bf16 burst "
                                         "(nominal dense fp8 : bf16 = 4.5 : 2.25 PFLOP/s)")
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        F = spmm.spmm_compress_24(A)
        torch.cuda.synchronize()
        build_ms = (time.perf_counter() - t0) * 1e3
        del A
        Cd = torch.empty((M, c["N"]), dtype=torch.float32, device="cuda")
        wsp = torch.empty(max(1, spmm.spmm_24_workspace_size(F, c["N"])), dtype=torch.uint8, device="cuda")
        nnz = M * K // 2
        es = 1 if fp8 else 2
        alg = nnz * es + M * K // 8 + K * c["N"] * es + M * c["N"] * 4
        kern, kid = "sparse_spmm_kernel", spmm._lib.KERNEL_SPARSE

        def step():
            spmm.spmm_24(F, Bx, Cd, wsp)
    elif c["kind"] == "sddmm":
        # sampled dense-dense product on the row-window workload's CSR pattern: A and Bt N(0,1) fp16
        # (fp32 out), or uniform int8 (exact int32 out)
        p = gen.config_problem(name)
        i8 = c["dtype"] == "i8"
        dt = torch.int8 if i8 else torch.float16
        val = torch.zeros(int(p["row_ptr"][-1]), dtype=torch.int8, device="cuda") if i8 else to_dev(p["val"], dt)
        S = spmm.CSR(c["M"], c["K"], int(p["row_ptr"][-1]), dt, to_dev(p["row_ptr"]), to_dev(p["col"]), val)
        Ax, Btx = (torch.from_numpy(p["A"]).cuda(), torch.from_numpy(p["Bt"]).cuda()) if i8 else \
            (to_dev(p["A"], dt), to_dev(p["Bt"], dt))
        out_d = torch.empty(S.nnz, dtype=torch.int32 if i8 else torch.float32, device="cuda")
        build_ms = 0.0
        nnz = S.nnz
        K_in = c["inner"]
        es = 1 if i8 else 2
        # pattern (row_ptr, col), A and Bt read once, one fp32 / int32 per entry written
        alg = (c["M"] + 1) * 4 + nnz * 4 + c["M"] * K_in * es + c["K"] * K_in * es + nnz * 4
        kern, kid = "sddmm_kernel", spmm._lib.KERNEL_SDDMM
        extra_fields["inner"] = K_in
        gathered = nnz * K_in * es  # one Bt row per entry

        def step():
            spmm.spmm_sddmm(S, Ax, Btx, out_d)
    elif c["kind"] == "rcm":
        # a scrambled band: RCM (host) on its pattern, P A P^T and its BCSR on the device; the step is
        # the permuted product (B gathered, BCSR, C scattered); context: BCSR of the scrambled matrix as is
        p = gen.config_problem(name, **({"N": args.n} if args.n else {}))
        n, bh = c["M"], c["bh"]
        nzm = (p["A"] & 0x7FFF) != 0
        row_ptr = np.concatenate([[0], np.cumsum(nzm.sum(axis=1))]).astype(np.int32)
        col = np.nonzero(nzm)[1].astype(np.int32)
        del nzm
        t0 = time.perf_counter()
        perm = spmm.rcm_order(n, row_ptr, col)
        extra_fields["rcm_host_ms"] = round((time.perf_counter() - t0) * 1e3, 2)
        A = to_dev(p["A"], torch.float16)
        Bx = to_dev(p["B"], torch.float16)
        permd = perm.cuda()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        F = spmm.build_bcsr(spmm.spmm_permute_sym(A, permd), bh, c["bw"])
        torch.cuda.synchronize()
        build_ms = (time.perf_counter() - t0) * 1e3
        Cd = torch.empty((n, c["N"]), dtype=torch.float32, device="cuda")
        wsp = torch.empty(spmm.spmm_bcsr_permuted_workspace_size(F, c["N"]), dtype=torch.uint8, device="cuda")
        # context: the scrambled matrix's own BCSR and product
        G = spmm.build_bcsr(A, bh, c["bw"])
        del A
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        for _ in range(2):
            spmm.spmm_bcsr(G, Bx, Cd)
        ev[0].record()
        for _ in range(3):
            spmm.spmm_bcsr(G, Bx, Cd)
        ev[1].record()
        torch.cuda.synchronize()
        extra_fields.update({"nnzb_scrambled": int(G.nnzb), "nnzb_permuted": int(F.nnzb),
                             "unpermuted_bcsr_ms": round(ev[0].elapsed_time(ev[1]) / 3, 4)})
        del G
        torch.cuda.empty_cache()
        nnz = F.nnzb * bh * c["bw"]
        # the BCSR kernel's own bytes: A' blocks + indices, B' read once, C' written once
        alg = nnz * 2 + F.nnzb * 4 + (n // bh + 1) * 4 + n * c["N"] * 2 + n * c["N"] * 4
        kern, kid = "bcsr_spmm_kernel", spmm._lib.KERNEL_BCSR

        def step():
            spmm.spmm_bcsr_permuted(F, permd, Bx, Cd, wsp)
    elif c["kind"] == "slide":
        # (2n-2):2n, the same recipe as the host generator drawn on the device: per group of 2n
        # two distinct zero positions, N(0,1) fp16 values elsewhere; B N(0,1) fp16
        M, K, n = c["M"], c["K"], c["n"]
        grp = 2 * n
        z0 = torch.randint(0, grp, (M, K // grp), generator=g, device="cuda")
        z1 = (z0 + 1 + torch.randint(0, grp - 1, (M, K // grp), generator=g, device="cuda")) % grp
        pos = torch.arange(grp, device="cuda")
        keep = ((pos != z0[..., None]) & (pos != z1[..., None])).reshape(M, K)
        A = torch.randn((M, K), generator=g, device="cuda").to(torch.float16) * keep
        del z0, z1, keep
        Bx = torch.randn((K, c["N"]), generator=g, device="cuda").to(torch.float16)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        F = spmm.spmm_build_slide(A, n)
        torch.cuda.synchronize()
        build_ms = (time.perf_counter() - t0) * 1e3
        # context: the dense fp16 GEMM (cuBLAS, fp16 out) of the same M x K x N on the unpruned shape
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        for _ in range(3):
            torch.mm(A, Bx)
        ev[0].record()
        for _ in range(5):
            torch.mm(A, Bx)
        ev[1].record()
        torch.cuda.synchronize()
        extra_fields["dense_cublas_fp16_ms"] = round(ev[0].elapsed_time(ev[1]) / 5, 4)
        del A
        Kl = F.K_lifted
        Cd = torch.empty((M, c["N"]), dtype=torch.float32, device="cuda")
        nnz = M * Kl // 2                      # = M K (n-1)/n stored nonzeros of the (2n-2):2n operand
        alg = nnz * 2 + M * Kl // 8 + K * c["N"] * 2 + M * c["N"] * 4
        kern, kid = "sparse_spmm_kernel", spmm._lib.KERNEL_SPARSE

        def step():
            spmm.spmm_slide(F, Bx, Cd)
    elif c["kind"] == "prune24":
        # magnitude pruning of a dense fp16 N(0,1) matrix into 2:4 (a builder: HBM-bound)
        M, K = c["M"], c["K"]
        A = torch.randn((M, K), generator=g, device="cuda").to(torch.float16)
        build_ms = 0.0
        nnz = M * K // 2
        flops = 0.0
        alg = M * K * 2 + nnz * 2 + M * K // 8
        kern, kid = "prune24_kernel", spmm._lib.KERNEL_PRUNE
        out = {}

        def step():
            out["F"] = spmm.spmm_prune_24(A)
    elif c["kind"] == "prunetvw":
        # magnitude pruning of a dense fp16 N(0,1) matrix into TVW (given kept columns; a builder)
        M, K, tr, keep = c["M"], c["K"], c["tile_rows"], c["keep"]
        A = torch.randn((M, K), generator=g, device="cuda").to(torch.float16)
        rng = np.random.default_rng(int(c["seed"]))
        n_t = -(-M // tr)
        cl = torch.from_numpy(np.concatenate([np.sort(rng.choice(K, keep, replace=False)) for _ in range(n_t)])
                              .astype(np.int32)).cuda()
        tp = torch.arange(0, n_t * keep + 1, keep, dtype=torch.int32, device="cuda")
        build_ms = 0.0
        nnz = M * keep // 2
        alg = M * keep * 2 + n_t * keep * 4 + nnz * 2 + M * keep // 8
        kern, kid = "tvw_build_kernel", None
        out = {}

        def step():
            out["F"] = spmm.spmm_prune_tvw(A, tr, tp, cl, Kp=keep)
    elif c["kind"] in ("wcsr", "wcsrc"):
        p = gen.config_problem(name, **({"N": args.n} if args.n else {}))
        dt = torch.float16
        csr = spmm.CSR(c["M"], c["K"], int(p["row_ptr"][-1]), dt, to_dev(p["row_ptr"]), to_dev(p["col"]),
                       to_dev(p["val"], dt))
        Bx = to_dev(p["B"], dt)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        F = spmm.build_wcsr(csr, 16, 32)
        torch.cuda.synchronize()
        build_ms = (time.perf_counter() - t0) * 1e3
        extra_fields["nonzeros_per_window_column"] = round(F.nnz / max(F.n_wcols, 1), 3)
        # the library's rule: tensor core when >= 4 nonzeros per window column and >= 384 per work unit
        tcore = F.nnz >= 4 * F.n_wcols and F.nnz >= 384 * F.n_units
        extra_fields["window_products"] = "tensor core" if tcore else "CUDA cores"
        # and of the tensor-core kernels, the streaming one for windows of <= 16 rows
        # and <= 32 steps per unit
        stream = F.h <= 16 and F.S <= 32
        wkern = ("wcsr_ts_kernel" if stream else "wcsr_tc_kernel") if tcore else "wcsr_spmm_kernel"
        Cd = torch.empty((c["M"], c["N"]), dtype=torch.float32, device="cuda")
        wsp = torch.zeros(max(1, spmm.spmm_wcsr_workspace_size(F, c["N"])), dtype=torch.uint8, device="cuda")
        nnz = csr.nnz
        # CSR-equivalent stored A (row_ptr, col, val) + B read once + C written once
        alg = (c["M"] + 1) * 4 + nnz * 4 + nnz * 2 + c["K"] * c["N"] * 2 + c["M"] * c["N"] * 4
        kern, kid = wkern, spmm._lib.KERNEL_WCSR
        # one B row per nonzero on CUDA cores, one per distinct window column on the tensor core
        gathered = (F.n_wcols if tcore else nnz) * c["N"] * 2

        def step():
            spmm.spmm_wcsr(F, Bx, Cd, wsp)
    else:
        raise ValueError(name)
    builder = c["kind"] in ("prune24", "prunetvw")
    flops = 0.0 if builder else 2.0 * nnz * (c["inner"] if c["kind"] == "sddmm" else c["N"])
    spmm.trace_enable(False)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    total_ms = timed_steps(step, steps, 0, flush_buf, ws)
    traced_pass(step, flush_buf, ws)
    # untraced builder: a check and a build kernel per call
    n, ms = spmm.trace_read(kid) if kid is not None else (2 * TRACED_STEPS, 0.0)
    if c["kind"] == "rcm":  # the row gather and scatter around each BCSR launch
        n_p, ms_p = spmm.trace_read(spmm._lib.KERNEL_PERMUTE)
        extra_fields["permute_kernels_ms_per_step"] = round(ms_p / TRACED_STEPS, 4)
        extra_fields["permute_launches"] = round(n_p * steps / TRACED_STEPS)
    spmm.trace_enable(False)
    total_ms = max_over_ranks(total_ms, ws, "cuda")
    # a builder without a traced kernel id (it synchronises inside): time the whole call
    t_kernel = ms / max(n, 1) / 1e3 if kid is not None else total_ms / steps / 1e3
    rl = roofline(flops, alg, t_kernel, peaks, prefer="hbm" if builder else None,
                  traffic=measured_traffic(kern, name), peak_scale=peak_scale)
    rl["kernel"] = kern
    rl["kernel_ms"] = round(t_kernel * 1e3, 4)
    if gathered:
        ach = gathered / t_kernel / 1e9
        extra_fields["l2_gather"] = {"bytes_per_launch": int(gathered), "achieved_gbs": round(ach, 1),
                                     "ceiling_gbs": L2_GATHER_GBS, "frac": round(ach / L2_GATHER_GBS, 4)}
    t_step = total_ms / steps / 1e3
    return {"workload": name, "ms_per_step": round(t_step * 1e3, 4),
            "tflops": round(ws * flops / t_step / 1e12, 3), "gbs": round(alg / t_step / 1e9, 1),
            "nnz": int(nnz), "build_ms": round(build_ms, 2), "roofline": rl, "launches": round(n * steps / TRACED_STEPS), **extra_fields}


# ------------------------------------------------------------------ CPU oracle legs
def oracle_sample_run(p, rows):
    import oracle
    F = oracle.compress24(p["A"], "i8")
    t0 = time.perf_counter()
    oracle.spmm24(F, p["B"], rows=rows)
    return time.perf_counter() - t0, F


def cpu_baseline(p, target_s=12.0):
    """The oracle (as it stands) on a bounded row sample of the headline workload."""
    import oracle
    F = oracle.compress24(p["A"], "i8")
    K, N = p["K"], p["N"]
    r = 8
    t0 = time.perf_counter()
    oracle.spmm24(F, p["B"], rows=(0, r))
    dt = time.perf_counter() - t0
    rows = int(min(p["M"], max(r, r * target_s / max(dt, 1e-3))))
    t0 = time.perf_counter()
    oracle.spmm24(F, p["B"], rows=(0, rows))
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * (K // 2) * N
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"rows 0..{rows - 1} of the {p['M']}x{K} int8 2:4 operand times the full {K}x{N} B "
                      f"(int64 accumulation), {dt:.1f} s"}


def _time_rows(run, total_rows, step, target_s):
    """Oracle time on rows [0, r): r grows from `step` until the run takes about
    target_s seconds (or covers every row); returns (r, seconds)."""
    r = min(step, total_rows)
    while True:
        t0 = time.perf_counter()
        run(r)
        dt = time.perf_counter() - t0
        if dt >= target_s or r >= total_rows:
            return r, dt
        grow = target_s / max(dt, 1e-3)
        r = min(total_rows, max(r + step, int(r * min(grow, 8.0)) // step * step))


def cpu_baseline_extra(name, target_s=2.0):
    """The oracle (as it stands, all host cores) on a bounded row sample of one of the
    other workloads, in the workload's own unit; the sample is stated."""
    import oracle
    import spmm_inputs as gen
    c = dict(gen.CONFIGS[name])
    kind = c["kind"]
    cores = oracle.num_threads()
    out = {"unit": "TFLOP/s", "cores": cores, "kind": "oracle"}
    if kind == "bcsr":
        Ns = min(c["N"], 512)
        p = gen.bcsr_problem(c["M"], c["K"], Ns, c["bh"], c["bw"], c["nnzb"], c["seed"], c["dtype"], c["std"])
        F = oracle.bcsr_build(p["A"], c["bh"], c["bw"], c["dtype"])
        r, dt = _time_rows(lambda r: oracle.bcsr_spmm(F, p["B"], rows=(0, r)), c["M"], c["bh"], target_s)
        nnz_r = int(F["row_ptr"][r // c["bh"]]) * c["bh"] * c["bw"]
        flops = 2.0 * nnz_r * Ns
        sample = f"rows 0..{r - 1} of {c['M']}, {Ns} of {c['N']} columns"
        if Ns < c["N"]:
            sample += (f"; extrapolated from the {Ns}-column slice to N = {c['N']} "
                       "(the oracle's time per column is constant, so the rate stands)")
    elif kind == "tvw":
        p = gen.config_problem(name)
        F = oracle.tvw_build(p["A"], c["tile_rows"], p["tile_ptr"], p["cols"], c["dtype"], Kp=c["keep"])
        r, dt = _time_rows(lambda r: oracle.tvw_spmm(F, p["B"], rows=(0, r)), c["M"], 8, target_s)
        flops = 2.0 * r * (c["keep"] // 2) * c["N"]
        sample = f"rows 0..{r - 1} of {c['M']}, all {c['N']} columns"
    elif kind in ("wcsr", "wcsrc"):
        p = gen.config_problem(name)
        F = oracle.wcsr_build(c["M"], c["K"], p["row_ptr"], p["col"], p["val"], c["dtype"], 16, 32)
        r, dt = _time_rows(lambda r: oracle.wcsr_spmm(F, p["B"], rows=(0, r)), c["M"], 256, target_s)
        flops = 2.0 * int(p["row_ptr"][r]) * c["N"]
        sample = f"rows 0..{r - 1} of {c['M']} (row-window form), all {c['N']} columns"
    elif kind == "24f":
        p = gen.config_problem(name)
        F = oracle.compress24(p["A"], c["dtype"])
        r, dt = _time_rows(lambda r: oracle.spmm24(F, p["B"], rows=(0, r)), c["M"], 4, target_s)
        flops = 2.0 * r * (c["K"] // 2) * c["N"]
        sample = f"rows 0..{r - 1} of {c['M']}, all {c['N']} columns ({c['dtype']}, fp64 sums)"
    elif kind == "slide":
        p = gen.config_problem(name)
        F = oracle.slide_build(p["A"], c["n"], c["dtype"])
        Kl = oracle.slide_lifted_k(c["K"], c["n"])
        G = {"M": F["M"], "K": Kl, "dtype": F["dtype"], "vals": F["vals"], "meta": F["meta"]}
        BL = oracle.slide_lift_b(p["B"], c["K"], c["n"])
        r, dt = _time_rows(lambda r: oracle.spmm24(G, BL, rows=(0, r)), c["M"], 4, target_s)
        flops = 2.0 * r * (Kl // 2) * c["N"]
        sample = f"rows 0..{r - 1} of {c['M']} of the lifted 2:4 operand, all {c['N']} columns"
    elif kind == "rcm":
        p = gen.config_problem(name)
        perm = oracle.rcm_dense(p["A"])
        F = oracle.bcsr_build(oracle.permute_sym(p["A"], perm, c["dtype"]), c["bh"], c["bw"], c["dtype"])
        Bp = np.ascontiguousarray(p["B"][perm])
        r, dt = _time_rows(lambda r: oracle.bcsr_spmm(F, Bp, rows=(0, r)), c["M"], c["bh"], target_s)
        flops = 2.0 * int(F["row_ptr"][r // c["bh"]]) * c["bh"] * c["bw"] * c["N"]
        sample = (f"rows 0..{r - 1} of {c['M']} of the BCSR of P A P^T (RCM order) times P B, all {c['N']} "
                  "columns (the permutations themselves untimed)")
    elif kind == "sddmm":
        p = gen.config_problem(name)
        rp, col = p["row_ptr"], p["col"]

        def run(r):
            if c["dtype"] == "i8":
                oracle.sddmm_i64(rp[:r + 1], col[:int(rp[r])], p["A"][:r], p["Bt"])
            else:
                oracle.sddmm(rp[:r + 1], col[:int(rp[r])], p["A"][:r], p["Bt"], c["dtype"])
        r, dt = _time_rows(run, c["M"], 256, target_s)
        flops = 2.0 * int(rp[r]) * c["inner"]
        sample = f"pattern rows 0..{r - 1} of {c['M']}, inner dimension {c['inner']}"
    elif kind in ("prune24", "prunetvw"):
        rng = np.random.default_rng(c["seed"])
        A = gen.normal_bits(rng, (c["M"], c["K"]), c["dtype"])
        out["unit"] = "GB/s"
        if kind == "prune24":
            r, dt = _time_rows(lambda r: oracle.prune24(A[:r], c["dtype"]), c["M"], 8, target_s)
            by = r * c["K"] * 2 + r * c["K"] // 2 * 2 + r * c["K"] // 8
        else:
            tr, keep = c["tile_rows"], c["keep"]
            n_t = -(-c["M"] // tr)
            cl = np.concatenate([np.sort(rng.choice(c["K"], keep, replace=False)) for _ in range(n_t)]).astype(np.int32)
            tp = np.arange(0, n_t * keep + 1, keep, dtype=np.int32)

            def run(r):
                t = r // tr
                oracle.prune_tvw(A[:r], tr, tp[:t + 1], cl[:t * keep], c["dtype"], Kp=keep)
            r, dt = _time_rows(run, c["M"], tr, target_s)
            by = r * keep * 2 + (r // tr) * keep * 4 + r * keep // 2 * 2 + r * keep // 8
        out.update({"value": round(by / dt / 1e9, 4),
                    "sample": f"rows 0..{r - 1} of the {c['M']}x{c['K']} dense matrix, {dt:.1f} s"})
        return out
    else:
        return None
    out.update({"value": round(flops / dt / 1e12, 6), "sample": f"{sample}, {dt:.1f} s"})
    return out


def run_reference(args, ws, rank):
    """--impl reference: the CPU oracle timed on the host cores, bounded sample per step."""
    if rank != 0:
        return 0
    import oracle
    import spmm_inputs as gen
    p = gen.config_problem(HEADLINE)
    F = oracle.compress24(p["A"], "i8")
    K, N = p["K"], p["N"]
    # size one step to about 2 s of CPU work
    t0 = time.perf_counter()
    oracle.spmm24(F, p["B"], rows=(0, 4))
    dt = time.perf_counter() - t0
    rows = int(min(p["M"], max(4, 4 * 2.0 / max(dt, 1e-3))))
    for i in range(args.warmup):
        oracle.spmm24(F, p["B"], rows=(0, rows))
    t0 = time.perf_counter()
    for i in range(args.steps):
        r0 = (i * rows) % (p["M"] - rows + 1)
        oracle.spmm24(F, p["B"], rows=(r0, r0 + rows))
    total = time.perf_counter() - t0
    flops = 2.0 * rows * (K // 2) * N
    value = flops * args.steps / total / 1e12
    sample = f"{rows} rows of the {p['M']}x{K} int8 2:4 operand times the full {K}x{N} B per step (int64)"
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "i8", "data": "synthetic",
            "config": {"workload": f"{HEADLINE}: A {p['M']}x{K} int8 2:4, B {K}x{N} int8, C int32",
                       "sample_rows": rows},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extra", action="store_true", help="skip the other formats")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", default=None,
                    help="run one workload (" + ", ".join(EXTRA_WORKLOADS) + ") "
                         "and print its result; "
                         "for profiling runs, not the benchmark line")
    ap.add_argument("--n", type=int, default=0, help="with --only: override the workload's N")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    ws, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, ws, rank)

    import torch
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    barrier(ws)
    import sparse_dense_matrix_spmm_gb300 as spmm
    spmm._lib.load()
    peaks, peak_src = load_peaks()
    flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    if args.only:
        r = run_extra(args.only, args, ws, peaks, flush_buf)
        if rank == 0:
            print(json.dumps({"only": args.only, **r}), flush=True)
        return 0
    h = run_headline(args, ws, rank, local, peaks, flush_buf)
    extra = []
    if not args.no_extra:
        for name in EXTRA_WORKLOADS:
            try:
                extra.append(run_extra(name, args, ws, peaks, flush_buf))
            except Exception as e:  # a format whose kernel is missing is reported, not hidden
                extra.append({"workload": name, "error": f"{type(e).__name__}: {e}"})
            torch.cuda.empty_cache()
    if spmm.last_device_error() != 0:
        raise RuntimeError("device error word set during the benchmark")
    if rank != 0:
        return 0
    cpu = None if args.no_cpu_baseline else cpu_baseline(h["problem"])
    if not args.no_cpu_baseline:
        # every other workload's oracle baseline, after all GPU timing (host work only)
        for e in extra:
            if "error" in e:
                continue
            try:
                e["cpu_baseline"] = cpu_baseline_extra(e["workload"])
            except Exception as ex:  # reported, not hidden
                e["cpu_baseline"] = {"error": f"{type(ex).__name__}: {ex}"}
    rl = h["roofline"]
    rl["peak_source"] = f"{peak_src} (MEASURED_PEAKS.json bf16 burst; fp16 tensor rate = bf16 rate)" \
        if rl["bound"] == "tensor" else peak_src
    line = {
        "metric": METRIC, "value": round(h["value"], 3), "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(h["ms_step"], 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "i8", "data": "synthetic",
        "config": {"workload": f"{HEADLINE}: A {h['M']}x{h['K']} int8 2:4 (2 nonzeros per 4-group), "
                               f"B {h['K']}x{h['N']} int8, C int32 exact",
                   "M": h["M"], "K": h["K"], "N": h["N"], "nnz": h["nnz"],
                   "compute": "fp16 sparse tensor core on int8-valued operands (A widened once when the format is built, B per step), fp32 partials over 2048-K chunks (< 2^24), int32 sum",
                   "l2": "flushed before every timed step (256 MiB write)", "parallelism": f"replicas x{ws}",
                   "build_ms": round(h["build_ms"], 2)},
        "roofline": rl, "cpu_baseline": cpu, "e2e": h["e2e"], "gpu_launches": h["launches"],
        "clocks": h["clocks"], "formats": extra,
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
