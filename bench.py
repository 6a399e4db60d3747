#!/usr/bin/env python
"""Benchmark: one step = the whole hot path (forward + backward) of exact
attention on one seeded synthetic workload, through the C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints ONE JSON line (rank 0).  ``value`` is forward+backward TFLOP/s
(algorithmic FLOPs: 4*B*H*N^2*d forward, halved for causal, x3.5 for
forward+backward; masked pairs are not counted) over all ranks, timed with
CUDA events on the launching stream, inputs resident in HBM, L2 flushed
between steps.  ``e2e`` is the same metric through ``fa_attention_host``
with pinned host buffers (copies inside the timed region).  Under torchrun
every rank runs its own replica of the workload (weak scaling, no data-path
collective); the time is the max over ranks.  ``per_config`` holds the
forward and forward+backward figures of every other configuration (a few
timed steps each, same loop).  Fractions of peak divide by the measured
dense-bf16 figure that matches the clock record of the timed region: the
burst figure when the SMs ran at their maximum clock, else the sustained one.

``--impl reference`` times the fp64 CPU oracle instead, on a bounded sample
of the same workload (one head truncated to ``--cpu-tokens`` tokens, the
sample ``cpu_baseline`` times too), on this machine's host cores.

``--fp8`` measures the FP8 forward instead: one step = the block
quantisation of Q, K and V (``fa_quantize_fp8``, three launches) and
``fa_fwd_fp8``; ``value`` is forward TFLOP/s over the step, the roofline is
the FP8 forward kernel against the dense-FP8 peak (the measured bf16
figure chosen as above x 2, the nominal fp8 : bf16 ratio).  ``--incoherent`` adds the
incoherent processing: Q and K go through ``fa_quantize_fp8_rotated`` with a
seeded random sign vector, and the forward is ``fa_fwd_fp8_rotated``.

``--tile-sweep`` times the forward at each tile shape ``fa_fwd_tiles`` offers
(query rows per CTA 128 / 256 x key rows per tile 64 / 128) on the workload
and prints one line with a ``sweep`` list (forward TFLOP/s per shape).

``--workload varlen_...`` measures a ragged batch (packed sequences of uneven
lengths): one step = ``fa_fwd_varlen`` + ``fa_bwd_varlen``; ``value`` is
forward+backward TFLOP/s over the visible (query, key) pairs.

``--workload decode_...`` measures the split-KV decode path instead: one step
= one ``fa_decode`` call (a few new query rows per sequence against a
resident key/value cache); ``value`` is GB/s of algorithmic traffic (Q, the
visible K and V rows read once, O and LSE written once) against the measured
HBM copy bandwidth.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "longctx_b1h16n16384d128"
FWD_BWD_FACTOR = 3.5          # forward + backward = forward x (1 + 2.5)
KERNEL_SOURCES = {"fa_fwd_kernel": "fa_fwd.cu", "fa_bwd64_kernel": "fa_bwd64.cu", "fa_bwd128_kernel": "fa_bwd128.cu",
                  "fa_fwd_kernel_fp8": "fa_fwd_fp8.cu", "fa_decode_kernel": "fa_decode.cu",
                  "fa_fwd_kernel_varlen": "fa_fwd.cu", "fa_bwd_varlen": ("fa_bwd.cu", "fa_bwd128.cu")}


# ---------------------------------------------------------------- distributed helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(backend):
    import torch.distributed as dist
    ws, rank, _ = dist_env()
    if ws > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return ws, rank


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def reduce_max(x: float, device=None) -> float:
    """Max of a float over ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank_step: float, world: int, step_s: float) -> float:
    """Aggregate throughput: the units every rank processed / the slowest rank's time."""
    return flops_per_rank_step * world / step_s / 1e12


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples every 200 ms during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
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
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        hi = max(sm)
        loaded = [s for s in sm if s >= 0.5 * hi] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- peaks / profiles
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def pick_peak(peaks, clk):
    """Dense-bf16 denominator for a kernel timed in this run.  The burst figure
    (a short cuBLAS run at the maximum SM clock) when the clock record of the
    timed region shows the SMs at their maximum clock with no power cap
    active; the sustained figure (a seconds-long cuBLAS loop, power-capped)
    otherwise, or when no clock record exists.  Returns (TFLOP/s, label)."""
    burst = float(peaks.get("bf16_tflops"))
    sustained = float(peaks.get("bf16_tflops_sustained", burst))
    sm = clk.get("sm_mhz") if clk else None
    mx = (clk.get("sm_max_mhz") if clk else None) or peaks.get("sm_max_mhz")
    capped = bool(clk) and "sw_power_cap" in clk.get("reasons", [])
    if sm is not None and mx and sm >= 0.95 * float(mx) and not capped:
        return burst, "bf16_tflops (burst: SM clock at its maximum during the timed region)"
    return sustained, "bf16_tflops_sustained (SM clock below its maximum or not recorded)"


def strip_comments(src: str) -> str:
    """C++ source without its comments (// to the end of the line, /* ... */),
    string and character literals kept as they are; the line breaks stay."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
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
            j = n if j < 0 else j + 2
            out.append("\n" * src.count("\n", i, j))
            i = j
        else:
            out.append(c)
            i += 1
    return "".join(out)


def source_digest(fname) -> str:
    """Digest of a kernel's source file(s) (a name or a tuple of names) and the
    shared device headers, over the code lines alone (comments, trailing blanks
    and empty lines left out): a change to a comment leaves the compiled
    kernel, and so its ncu record, as it was."""
    h = hashlib.sha256()
    files = {fname} if isinstance(fname, str) else set(fname)
    for f in sorted(files | {"fa_ptx.cuh", "fa_tiles.cuh"}):
        with open(os.path.join(ROOT, "io_aware_exact_09_gb300", "csrc", f), encoding="utf-8") as fh:
            code = [ln.rstrip() for ln in strip_comments(fh.read()).splitlines()]
            h.update("\n".join(ln for ln in code if ln).encode())
    return h.hexdigest()[:16]


def ncu_record(kernel: str, workload: str):
    """The committed ncu figures of `kernel` on `workload`, if they were taken
    on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rows = json.load(f)
    r = rows.get(kernel, {}).get(workload)
    if not r or r.get("source_digest") != source_digest(KERNEL_SOURCES[kernel]):
        return None
    return r


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch (read + write) from the committed ncu capture, or None."""
    r = ncu_record(kernel, workload)
    return None if r is None else r.get("bytes_per_launch")


def ncu_tensor_pipe(kernel: str, workload: str):
    """ncu's sm__pipe_tensor_cycles_active (% of peak) from the committed capture, or None."""
    r = ncu_record(kernel, workload)
    return None if r is None else r.get("tensor_pipe_active_pct")


# ---------------------------------------------------------------- CPU oracle baseline
def _oracle_case(w, n):
    import torch

    from synthetic import Workload, make_inputs
    sub = Workload(w.name, 1, 1, n, w.d, w.seed, causal=w.causal, input_scale=w.input_scale,
                   sparse_density=w.sparse_density)
    c = make_inputs(sub)
    kl = [max(1, int(n * 0.625))] if w.key_len_range is not None else None   # mean of U[128,512] / 512
    Q, K, V, dO = (c[k].to(torch.float64).numpy() for k in ("Q", "K", "V", "dO"))
    bm = None if c["block_mask"] is None else c["block_mask"].numpy()
    return Q, K, V, dO, kl, bm


def oracle_time(w, n):
    """One fp64 oracle forward+backward on one head of the workload truncated
    to its first n tokens: (TFLOP/s, seconds)."""
    import oracle
    from synthetic import algorithmic_fwd_flops
    Q, K, V, dO, kl, bm = _oracle_case(w, n)
    t0 = time.perf_counter()
    oracle.attention_bwd(Q, K, V, dO, w.softmax_scale, causal=w.causal, key_len=kl, block_mask=bm)
    dt = time.perf_counter() - t0
    fl = FWD_BWD_FACTOR * algorithmic_fwd_flops(1, 1, n, w.d, w.causal, kl, bm)
    return fl / dt / 1e12, dt


def oracle_sample_desc(w, n):
    return ("fp64 oracle fwd+bwd (materialised S and P), one head of %s truncated to its first %d tokens, "
            "d=%d" % (w.name, n, w.d))


def oracle_sample(w, n, budget_s: float = 0.0):
    """Time the fp64 oracle on the bounded sample of n tokens of one head,
    calling it repeatedly until about budget_s has passed (at least once).
    Returns (TFLOP/s, cores, description, seconds per call)."""
    import oracle
    dts, tfs = [], []
    t_end = time.perf_counter() + budget_s
    while not dts or time.perf_counter() < t_end:
        tf, dt = oracle_time(w, n)
        tfs.append(tf)
        dts.append(dt)
    dt = sum(dts) / len(dts)
    tf = sum(tfs) / len(tfs)
    desc = oracle_sample_desc(w, n) + ", %d call(s), %.2f s per call" % (len(dts), dt)
    return tf, oracle.num_threads(), desc, dt


def sample_tokens(w, requested):
    """Tokens of the CPU sample: the requested count, at most N."""
    return max(1, min(int(requested), w.N))


# ---------------------------------------------------------------- decode
def decode_bytes(w, kv_len):
    """Algorithmic bytes of one decode step: Q read, the visible K and V rows
    read once, O (bf16) and LSE (fp32) written once."""
    from synthetic import decode_visible_keys
    rows = w.B * w.H * w.Nq
    return rows * w.d * 2 + 2 * decode_visible_keys(w, kv_len) * w.d * 2 + rows * w.d * 2 + rows * 4


def _oracle_decode_case(w, B, H):
    import dataclasses

    import torch

    from synthetic import make_decode_inputs
    sub = dataclasses.replace(w, B=B, H=H)
    c = make_decode_inputs(sub)
    Q, K, V = (c[k].to(torch.float64).numpy() for k in ("Q", "K", "V"))
    kl = None if c["kv_len"] is None else c["kv_len"].tolist()
    return sub, Q, K, V, kl


def oracle_decode_sample(w, budget_s: float, BH=None):
    """Time the fp64 oracle decode on a bounded sample: the first B' batch
    entries with H' heads (same recipe, a smaller draw), at most ~2 GB of
    fp64 cache, called repeatedly for about budget_s.  Returns (GB/s of
    bf16-equivalent algorithmic bytes, cores, description, (B', H'))."""
    import oracle
    if BH is None:
        per_head = 2 * w.Nk * w.d * 8
        H = max(1, min(w.H, (2 << 30) // per_head))
        B = max(1, min(w.B, (2 << 30) // (per_head * H)))
    else:
        B, H = BH
    sub, Q, K, V, kl = _oracle_decode_case(w, B, H)
    dts = []
    t_end = time.perf_counter() + budget_s
    while not dts or time.perf_counter() < t_end:
        t0 = time.perf_counter()
        oracle.attention_decode(Q, K, V, w.softmax_scale, causal=w.causal, kv_len=kl)
        dts.append(time.perf_counter() - t0)
    dt = sum(dts) / len(dts)
    what = ("the whole of %s" % w.name if (B, H) == (w.B, w.H) else
            "the first %d batch entr%s x %d head(s) of %s (same recipe, smaller draw)"
            % (B, "y" if B == 1 else "ies", H, w.name))
    desc = "fp64 oracle decode of %s, %d calls, %.3f s per call" % (what, len(dts), dt)
    return decode_bytes(sub, kl) / dt / 1e9, oracle.num_threads(), desc, (B, H)


def run_decode(args, w):
    import torch

    ws_n, rank = init_dist("nccl")
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import io_aware_exact_09_gb300 as fa
    from synthetic import make_decode_inputs
    fa.build()
    B, H, Nq, Nk, d = w.B, w.H, w.Nq, w.Nk, w.d
    case = make_decode_inputs(w)
    Q, K, V = (case[k].to(dev).contiguous() for k in ("Q", "K", "V"))
    kl = None if case["kv_len"] is None else case["kv_len"].to(dev)
    kl_list = None if case["kv_len"] is None else case["kv_len"].tolist()
    O = torch.empty_like(Q)
    LSE = torch.empty((B, H, Nq), dtype=torch.float32, device=dev)
    wsn = fa.fa_decode_workspace_size(B, H, Nq, Nk, d, 0)
    ws = fa.workspace(wsn, dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    nbytes = decode_bytes(w, kl_list)

    def check(st, where):
        if st != 0:
            raise RuntimeError("%s failed: %s" % (where, fa.fa_status_string(st)))

    def step():
        check(fa.fa_decode(Q, K, V, O, LSE, B, H, Nq, Nk, d, w.softmax_scale, w.causal, kl, 0, ws, wsn, sp),
              "fa_decode")

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)     # 256 MiB > 129 MB L2
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    check(fa.fa_get_device_status(ws, sp), "device status after warm-up")

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    # one timed step is ~0.1-0.4 ms: repeat it so the clock sampler sees load
    reps = max(1, int(args.decode_reps))
    times = []
    barrier()
    torch.cuda.synchronize(dev)
    launches = 0
    for _ in range(args.steps):
        for _ in range(reps):
            flush.zero_()
            e0.record(stream)
            step()
            e1.record(stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1))
            launches += 2
    torch.cuda.synchronize(dev)
    barrier()
    clk = clocks.stop()
    check(fa.fa_get_device_status(ws, sp), "device status after timing")
    ms = reduce_max(sum(times) / len(times), dev)
    value = nbytes * ws_n / (ms / 1e3) / 1e9

    peaks, peak_src = measured_peaks()
    peak = float(peaks.get("hbm_gbs"))
    achieved = nbytes / (ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": "fa_decode_kernel + fa_decode_merge_kernel (one fa_decode call)",
                "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": ncu_traffic("fa_decode_kernel", w.name), "peak_source": "%s hbm_gbs" % peak_src}

    e2e = None
    if not args.no_e2e:
        # the cache stays resident (it is the decode state); each step copies
        # the new queries in and the outputs out through pinned host memory
        Qh = case["Q"].contiguous().pin_memory()
        Oh = torch.empty_like(Qh).pin_memory()
        Lh = torch.empty((B, H, Nq), dtype=torch.float32).pin_memory()
        Qd = torch.empty_like(Q)
        et = []
        for i in range(1 + max(3, min(args.steps, 10))):
            flush.zero_()
            e0.record(stream)
            Qd.copy_(Qh, non_blocking=True)
            check(fa.fa_decode(Qd, K, V, O, LSE, B, H, Nq, Nk, d, w.softmax_scale, w.causal, kl, 0, ws, wsn, sp),
                  "fa_decode")
            Oh.copy_(O, non_blocking=True)
            Lh.copy_(LSE, non_blocking=True)
            e1.record(stream)
            e1.synchronize()
            if i > 0:
                et.append(e0.elapsed_time(e1))
        e_ms = reduce_max(sum(et) / len(et), dev)
        e2e = {"value": nbytes * ws_n / (e_ms / 1e3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": Qh.numel() * 2, "d2h_bytes_per_step": Oh.numel() * 2 + Lh.numel() * 4,
               "ms_per_step": e_ms, "note": "key/value cache resident in HBM"}

    cpu = None
    if rank == 0 and ws_n == 1 and not args.no_cpu_baseline:
        gbs, cores, desc, _ = oracle_decode_sample(w, args.cpu_budget)
        cpu = {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": desc}

    if rank == 0:
        line = {
            "metric": "decode attention GB/s (bf16 K/V cache)", "value": value, "unit": "GB/s", "n_gpus": ws_n,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "B": B, "H": H, "Nq": Nq, "Nk": Nk, "d": d, "causal": w.causal,
                       "ragged_cache": kl is not None, "splits": "auto",
                       "parallelism": "replicas" if ws_n > 1 else "single",
                       "l2": "flushed between steps (cache larger than L2 too)",
                       "timed_calls": len(times)},
            "algorithmic_bytes_per_step": nbytes,
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clk,
            "gpu_launches": launches,
        }
        print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- FP8 forward
def run_fp8(args):
    import torch

    ws_n, rank = init_dist("nccl")
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import io_aware_exact_09_gb300 as fa
    from synthetic import WORKLOADS, algorithmic_fwd_flops, make_inputs
    fa.build()
    w = WORKLOADS[args.workload]
    B, H, N, d = w.B, w.H, w.N, w.d
    if d != 128:
        raise SystemExit("the FP8 forward needs d = 128")
    case = make_inputs(w, with_dO=False)
    Q, K, V = (case[k].to(dev).contiguous() for k in ("Q", "K", "V"))
    kl = None if case["key_len"] is None else case["key_len"].to(dev)
    bm = None if case["block_mask"] is None else case["block_mask"].contiguous().to(dev)
    T, Np = (N + 127) // 128, (N + 15) // 16 * 16
    Q8 = torch.empty((B, H, N, d), dtype=torch.uint8, device=dev)
    K8 = torch.empty_like(Q8)
    Vt8 = torch.empty((B, H, d, Np), dtype=torch.uint8, device=dev)
    sQ, sK, sV = (torch.empty((B, H, T), dtype=torch.float32, device=dev) for _ in range(3))
    O = torch.empty_like(Q)
    LSE = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    # incoherent processing: a seeded random sign vector (an input of the method)
    signs = None
    scale = w.softmax_scale
    if args.incoherent:
        g = torch.Generator().manual_seed(w.seed + 17)
        signs = torch.where(torch.rand(d, generator=g) < 0.5, -1, 1).to(torch.int8).to(dev)
    wsn = fa.fa_fwd_workspace_size(B, H, N, d)
    ws = fa.workspace(wsn, dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    flops = algorithmic_fwd_flops(B, H, N, d, w.causal,
                                  None if case["key_len"] is None else case["key_len"].tolist(),
                                  None if case["block_mask"] is None else case["block_mask"])

    def check(st, where):
        if st != 0:
            raise RuntimeError("%s failed: %s" % (where, fa.fa_status_string(st)))

    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]

    def step(record):
        if record:
            ev[0].record(stream)
        if signs is None:
            check(fa.fa_quantize_fp8(Q, Q8, sQ, B, H, N, d, False, sp), "fa_quantize_fp8 Q")
            check(fa.fa_quantize_fp8(K, K8, sK, B, H, N, d, False, sp), "fa_quantize_fp8 K")
        else:
            check(fa.fa_quantize_fp8_rotated(Q, Q8, sQ, signs, B, H, N, d, sp), "fa_quantize_fp8_rotated Q")
            check(fa.fa_quantize_fp8_rotated(K, K8, sK, signs, B, H, N, d, sp), "fa_quantize_fp8_rotated K")
        check(fa.fa_quantize_fp8(V, Vt8, sV, B, H, N, d, True, sp), "fa_quantize_fp8 V")
        if record:
            ev[1].record(stream)
        fwd = fa.fa_fwd_fp8 if signs is None else fa.fa_fwd_fp8_rotated
        check(fwd(Q8, K8, Vt8, sQ, sK, sV, O, LSE, B, H, N, d, scale, w.causal, kl, bm, ws, wsn, sp),
              "fa_fwd_fp8" if signs is None else "fa_fwd_fp8_rotated")
        if record:
            ev[2].record(stream)

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        step(False)
    torch.cuda.synchronize(dev)
    check(fa.fa_get_device_status(ws, sp), "device status after warm-up")
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    tq, tf_, tstep = [], [], []
    barrier()
    torch.cuda.synchronize(dev)
    launches = 0
    for _ in range(args.steps):
        flush.zero_()
        step(True)
        launches += 4
        ev[2].synchronize()
        tq.append(ev[0].elapsed_time(ev[1]))
        tf_.append(ev[1].elapsed_time(ev[2]))
        tstep.append(ev[0].elapsed_time(ev[2]))
    torch.cuda.synchronize(dev)
    barrier()
    clk = clocks.stop()
    check(fa.fa_get_device_status(ws, sp), "device status after timing")
    mq, mf, ms = (sum(x) / len(x) for x in (tq, tf_, tstep))
    step_ms = reduce_max(ms, dev)
    value = whole_job_tflops(flops, ws_n, step_ms / 1e3)
    peaks, peak_src = measured_peaks()
    peak16, peak_kind = pick_peak(peaks, clk)
    peak8 = 2.0 * peak16
    achieved = flops / (mf / 1e3) / 1e12
    roofline = {"bound": "tensor", "kernel": "fa_fwd_kernel<128, fp8>", "achieved": achieved, "peak": peak8,
                "unit": "TFLOP/s", "frac": achieved / peak8, "traffic": ncu_traffic("fa_fwd_kernel_fp8", w.name),
                "ncu_tensor_pipe_active_pct": ncu_tensor_pipe("fa_fwd_kernel_fp8", w.name),
                "peak_source": "%s %s x 2 (nominal dense fp8 : bf16 ratio 4.5 : 2.25)" % (peak_src, peak_kind)}
    e2e = None
    if not args.no_e2e:
        # the user's call from host memory: bf16 Q, K, V in, O and LSE out
        pin = lambda t: t.contiguous().pin_memory()
        Qh, Kh, Vh = (pin(case[k]) for k in ("Q", "K", "V"))
        Oh = torch.empty_like(Qh).pin_memory()
        Lh = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        et = []
        for i in range(1 + max(1, min(args.steps, 5))):
            e0.record(stream)
            Q.copy_(Qh, non_blocking=True)
            K.copy_(Kh, non_blocking=True)
            V.copy_(Vh, non_blocking=True)
            step(False)
            Oh.copy_(O, non_blocking=True)
            Lh.copy_(LSE, non_blocking=True)
            e1.record(stream)
            e1.synchronize()
            if i > 0:
                et.append(e0.elapsed_time(e1))
        e_ms = reduce_max(sum(et) / len(et), dev)
        nb = B * H * N * d * 2
        e2e = {"value": whole_job_tflops(flops, ws_n, e_ms / 1e3), "unit": "TFLOP/s",
               "h2d_bytes_per_step": 3 * nb, "d2h_bytes_per_step": nb + B * H * N * 4, "ms_per_step": e_ms}
    if rank == 0:
        line = {
            "metric": "attention fwd TFLOP/s (fp8 e4m3, block-quantised)", "value": value, "unit": "TFLOP/s",
            "n_gpus": ws_n, "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp8-e4m3", "data": "synthetic",
            "config": {"workload": w.name, "B": B, "H": H, "N": N, "d": d, "causal": w.causal, "path": "fp8 forward",
                       "incoherent_processing": bool(args.incoherent),
                       "parallelism": "replicas" if ws_n > 1 else "single", "l2": "flushed between steps"},
            "kernel_ms": {"fa_quant_fp8_kernel x3": mq, "fa_fwd_kernel<128, fp8>": mf},
            "fwd_kernel_tflops": achieved, "algorithmic_flops_per_step": flops,
            "roofline": roofline, "cpu_baseline": None, "e2e": e2e, "clocks": clk, "gpu_launches": launches,
        }
        print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- tile-size sweep
def run_tile_sweep(args):
    import torch

    ws_n, rank = init_dist("nccl")
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import io_aware_exact_09_gb300 as fa
    from synthetic import WORKLOADS, algorithmic_fwd_flops, make_inputs
    fa.build()
    w = WORKLOADS[args.workload]
    B, H, N, d = w.B, w.H, w.N, w.d
    case = make_inputs(w, with_dO=False)
    Q, K, V = (case[k].to(dev).contiguous() for k in ("Q", "K", "V"))
    kl = None if case["key_len"] is None else case["key_len"].to(dev)
    bm = None if case["block_mask"] is None else case["block_mask"].contiguous().to(dev)
    O = torch.empty_like(Q)
    LSE = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    wsn = fa.fa_fwd_workspace_size(B, H, N, d)
    ws = fa.workspace(wsn, dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    flops = algorithmic_fwd_flops(B, H, N, d, w.causal,
                                  None if case["key_len"] is None else case["key_len"].tolist(),
                                  None if case["block_mask"] is None else case["block_mask"])
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    out = []
    launches = 0
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    for bq, bk in ((256, 128), (256, 64), (128, 128), (128, 64)):
        def step():
            st = fa.fa_fwd_tiles(Q, K, V, O, LSE, B, H, N, d, w.softmax_scale, w.causal, kl, bm, bq, bk, ws, wsn, sp)
            if st != 0:
                raise RuntimeError("fa_fwd_tiles failed: %s" % fa.fa_status_string(st))
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize(dev)
        ts = []
        for _ in range(args.steps):
            flush.zero_()
            e0.record(stream)
            step()
            e1.record(stream)
            e1.synchronize()
            ts.append(e0.elapsed_time(e1))
            launches += 1
        ms = reduce_max(sum(ts) / len(ts), dev)
        out.append({"block_q": bq, "block_k": bk, "ms": ms, "tflops": whole_job_tflops(flops, ws_n, ms / 1e3)})
    clk = clocks.stop()
    if fa.fa_get_device_status(ws, sp) != 0:
        raise RuntimeError("device status after the sweep")
    peaks, peak_src = measured_peaks()
    peak, peak_kind = pick_peak(peaks, clk)
    best = max(out, key=lambda r: r["tflops"])
    if rank == 0:
        print(json.dumps({
            "metric": "attention fwd TFLOP/s (bf16) per tile shape", "value": best["tflops"], "unit": "TFLOP/s",
            "n_gpus": ws_n, "steps": args.steps, "warmup": args.warmup, "ms_per_step": best["ms"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "B": B, "H": H, "N": N, "d": d, "causal": w.causal,
                       "l2": "flushed between steps"},
            "sweep": out,
            "roofline": {"bound": "tensor", "kernel": "fa_fwd_kernel (best shape)", "achieved": best["tflops"] / ws_n,
                         "peak": peak, "unit": "TFLOP/s", "frac": best["tflops"] / ws_n / peak, "traffic": None,
                         "peak_source": "%s %s" % (peak_src, peak_kind)},
            "cpu_baseline": None, "e2e": None, "clocks": clk, "gpu_launches": launches}), flush=True)
    return 0


# ---------------------------------------------------------------- ragged batches
def oracle_varlen_sample(w, budget_s: float):
    """The fp64 oracle forward + backward of sequence 0 of the ragged workload,
    one head, called repeatedly for about budget_s: (TFLOP/s, cores, description)."""
    import oracle
    from synthetic import make_varlen_inputs, varlen_fwd_flops
    c = make_varlen_inputs(w)
    cq, ck = c["cu_q"].numpy(), c["cu_k"].numpy()
    f = lambda X, a, b: X[a:b, 0:1].double().numpy().transpose(1, 0, 2)[None]
    q, k, v = f(c["Q"], cq[0], cq[1]), f(c["K"], ck[0], ck[1]), f(c["V"], ck[0], ck[1])
    g = q * 0.5                       # any fixed dO of the right shape: the work does not depend on its values
    fl = FWD_BWD_FACTOR * varlen_fwd_flops([0, cq[1] - cq[0]], [0, ck[1] - ck[0]], 1, w.d, w.causal)
    dts = []
    t_end = time.perf_counter() + budget_s
    while not dts or time.perf_counter() < t_end:
        t0 = time.perf_counter()
        oracle.attention_bwd_rect(q, k, v, g, w.softmax_scale, causal=w.causal)
        dts.append(time.perf_counter() - t0)
    dt = sum(dts) / len(dts)
    desc = ("fp64 oracle forward + backward (materialised S and P) of sequence 0 (%d queries, %d keys), head 0, "
            "of %s, %d calls, %.3f s per call" % (cq[1] - cq[0], ck[1] - ck[0], w.name, len(dts), dt))
    return fl / dt / 1e12, oracle.num_threads(), desc


def run_varlen(args, w):
    import torch

    ws_n, rank = init_dist("nccl")
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import io_aware_exact_09_gb300 as fa
    from synthetic import make_varlen_inputs, varlen_fwd_flops
    fa.build()
    c = make_varlen_inputs(w)
    g = torch.Generator().manual_seed(w.seed + 1)
    dO_h = torch.randn(c["Q"].shape, generator=g).to(torch.bfloat16)
    Q, K, V = (c[k].to(dev).contiguous() for k in ("Q", "K", "V"))
    dO = dO_h.to(dev)
    cu_q, cu_k = c["cu_q"].to(dev), c["cu_k"].to(dev)
    B, H, d = w.B, w.H, w.d
    tq, tk = int(Q.shape[0]), int(K.shape[0])
    max_k = int((c["cu_k"][1:] - c["cu_k"][:-1]).max())
    O = torch.empty_like(Q)
    LSE = torch.empty((H, tq), dtype=torch.float32, device=dev)
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    wsn = fa.fa_fwd_workspace_size(1, 1, 1, d)
    ws = fa.workspace(wsn, dev)
    wsbn = fa.fa_bwd_varlen_workspace_size(H, tq, d)
    wsb = fa.workspace(wsbn, dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    flops_fwd = varlen_fwd_flops(c["cu_q"].tolist(), c["cu_k"].tolist(), H, d, w.causal)
    flops = FWD_BWD_FACTOR * flops_fwd

    def check(st, where):
        if st != 0:
            raise RuntimeError("%s failed: %s" % (where, fa.fa_status_string(st)))

    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]

    def step(record):
        if record:
            ev[0].record(stream)
        check(fa.fa_fwd_varlen(Q, K, V, O, LSE, cu_q, cu_k, B, H, tq, tk, c["max_q"], d, w.softmax_scale, w.causal,
                               ws, wsn, sp), "fa_fwd_varlen")
        if record is True:
            ev[1].record(stream)
        check(fa.fa_bwd_varlen(Q, K, V, O, LSE, dO, dQ, dK, dV, cu_q, cu_k, B, H, tq, tk, max_k, d, w.softmax_scale,
                               w.causal, wsb, wsbn, sp), "fa_bwd_varlen")
        if record:
            ev[2].record(stream)

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        step(False)
    torch.cuda.synchronize(dev)
    check(fa.fa_get_device_status(ws, sp), "device status after warm-up")
    check(fa.fa_get_device_status(wsb, sp), "device status after warm-up")
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    tf_, tb_, tstep = [], [], []
    barrier()
    torch.cuda.synchronize(dev)
    for _ in range(args.steps):
        flush.zero_()
        step(True)
        ev[2].synchronize()
        tf_.append(ev[0].elapsed_time(ev[1]))
        tb_.append(ev[1].elapsed_time(ev[2]))
    # the whole step with events at its ends only (an event between the calls
    # would keep the backward's first kernel from overlapping the forward's tail)
    for _ in range(args.steps):
        flush.zero_()
        step("ends")
        ev[2].synchronize()
        tstep.append(ev[0].elapsed_time(ev[2]))
    torch.cuda.synchronize(dev)
    barrier()
    clk = clocks.stop()
    check(fa.fa_get_device_status(ws, sp), "device status after timing")
    check(fa.fa_get_device_status(wsb, sp), "device status after timing")
    mf, mb, ms = (sum(x) / len(x) for x in (tf_, tb_, tstep))
    ms = reduce_max(ms, dev)
    value = whole_job_tflops(flops, ws_n, ms / 1e3)
    peaks, peak_src = measured_peaks()
    peak, peak_kind = pick_peak(peaks, clk)
    fwd_tf = flops_fwd / (mf / 1e3) / 1e12
    bwd_tf = 2.5 * flops_fwd / (mb / 1e3) / 1e12
    # the dominant launch sequence of the step is the backward (three kernels)
    dom_forward = mf >= mb
    achieved = fwd_tf if dom_forward else bwd_tf
    roofline = {"bound": "tensor",
                "kernel": ("fa_fwd_kernel<%d, varlen>" % d) if dom_forward else
                          ("fa_bwd_varlen (pre + %s<varlen> + convert)" % ("fa_bwd128_kernel" if d == 128 else
                                                                           "fa_bwd64_kernel")),
                "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": ncu_traffic("fa_fwd_kernel_varlen" if dom_forward else "fa_bwd_varlen", w.name),
                "ncu_tensor_pipe_active_pct": ncu_tensor_pipe("fa_fwd_kernel_varlen" if dom_forward else "fa_bwd_varlen",
                                                              w.name),
                "peak_source": "%s %s" % (peak_src, peak_kind)}
    e2e = None
    if not args.no_e2e:
        pin = lambda t: t.contiguous().pin_memory()
        Qh, Kh, Vh, dOh = (pin(x) for x in (c["Q"], c["K"], c["V"], dO_h))
        Oh = torch.empty_like(Qh).pin_memory()
        Lh = torch.empty((H, tq), dtype=torch.float32).pin_memory()
        dQh, dKh, dVh = torch.empty_like(Qh).pin_memory(), torch.empty_like(Kh).pin_memory(), \
            torch.empty_like(Vh).pin_memory()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        et = []
        # two untimed passes (the first copies through freshly pinned pages run
        # several times slower), then the median of the timed ones
        for i in range(2 + max(3, min(args.steps, 7))):
            e0.record(stream)
            for dst, src in ((Q, Qh), (K, Kh), (V, Vh), (dO, dOh)):
                dst.copy_(src, non_blocking=True)
            step(False)
            for dst, src in ((Oh, O), (Lh, LSE), (dQh, dQ), (dKh, dK), (dVh, dV)):
                dst.copy_(src, non_blocking=True)
            e1.record(stream)
            e1.synchronize()
            if i > 1:
                et.append(e0.elapsed_time(e1))
        e_ms = reduce_max(sorted(et)[len(et) // 2], dev)
        e2e = {"value": whole_job_tflops(flops, ws_n, e_ms / 1e3), "unit": "TFLOP/s",
               "h2d_bytes_per_step": (2 * tq + 2 * tk) * H * d * 2,
               "d2h_bytes_per_step": (2 * tq + 2 * tk) * H * d * 2 + H * tq * 4,
               "ms_per_step": e_ms, "note": "cu_seqlens stay resident"}
    cpu = None
    if rank == 0 and ws_n == 1 and not args.no_cpu_baseline:
        tf, cores, desc = oracle_varlen_sample(w, args.cpu_budget)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc}
    if rank == 0:
        line = {
            "metric": "attention fwd+bwd TFLOP/s (bf16, ragged batch)", "value": value, "unit": "TFLOP/s",
            "n_gpus": ws_n, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "B": B, "H": H, "d": d, "total_q": tq, "total_k": tk,
                       "max_seqlen_q": c["max_q"], "max_seqlen_k": max_k, "causal": w.causal,
                       "parallelism": "replicas" if ws_n > 1 else "single", "l2": "flushed between steps"},
            "fwd_tflops": fwd_tf, "bwd_tflops": bwd_tf, "fwd_frac_of_peak": fwd_tf / peak,
            "bwd_frac_of_peak": bwd_tf / peak, "kernel_ms": {"fa_fwd_varlen": mf, "fa_bwd_varlen": mb},
            "algorithmic_flops_per_step": flops, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "clocks": clk, "gpu_launches": 4 * args.steps,
        }
        print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- reference arm
def run_reference_decode(args, w):
    import oracle
    oracle.build()
    vals = []
    desc = cores = None
    _, _, _, BH = oracle_decode_sample(w, 0.0)
    for i in range(args.warmup + args.steps):
        gbs, cores, desc, _ = oracle_decode_sample(w, 3.0, BH)
        if i >= args.warmup:
            vals.append(gbs)
    v = statistics.median(vals)
    line = {"impl": "reference", "metric": "decode attention GB/s (bf16 K/V cache)", "value": v, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d,
                       "causal": w.causal},
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


def run_reference(args):
    ws, rank = init_dist("gloo")
    if rank != 0:
        return 0
    from synthetic import DECODE_WORKLOADS, VARLEN_WORKLOADS, WORKLOADS
    if args.workload in DECODE_WORKLOADS:
        return run_reference_decode(args, DECODE_WORKLOADS[args.workload])
    if args.workload in VARLEN_WORKLOADS:
        w = VARLEN_WORKLOADS[args.workload]
        import oracle
        oracle.build()
        vals = []
        for i in range(args.warmup + args.steps):
            tf, cores, desc = oracle_varlen_sample(w, 3.0)
            if i >= args.warmup:
                vals.append(tf)
        v = statistics.median(vals)
        print(json.dumps({"impl": "reference", "metric": "attention fwd+bwd TFLOP/s (bf16, ragged batch)", "value": v,
                          "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                          "data": "synthetic", "config": {"workload": w.name, "B": w.B, "H": w.H, "d": w.d},
                          "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                           "sample": desc},
                          "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
                          "gpu_launches": 0}), flush=True)
        return 0
    import oracle
    oracle.build()
    w = WORKLOADS[args.workload]
    vals, dts = [], []
    cores = None
    n = sample_tokens(w, args.cpu_tokens)
    # one oracle call on the bounded sample per step (the sample cpu_baseline times too)
    for i in range(args.warmup + args.steps):
        tf, cores, _, dt = oracle_sample(w, n)
        if i >= args.warmup:
            vals.append(tf)
            dts.append(dt)
    v = statistics.median(vals)
    desc = oracle_sample_desc(w, n) + ", %d call(s), %.2f s per call" % (len(dts), sum(dts) / len(dts))
    line = {"impl": "reference", "metric": "attention fwd+bwd TFLOP/s (bf16)", "value": v, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, args.gpus),
            "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- our arm
# The configurations the method is evaluated on besides the timed workload:
# each gets a short forward + backward timing in the same run.
PER_CONFIG = ("small_b1h2n128d64", "gpt2m_causal_b8h16n1024d64", "bertl_keypad_b16h16n512d64",
              "longctx_causal_b1h16n16384d128", "blocksparse_b2h16n8192d64")


def workload_config(w, n_gpus):
    """The `config` object of a square workload's line (both arms use it)."""
    return {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
            "key_padding": w.key_len_range is not None, "block_sparse": w.sparse_density is not None,
            "parallelism": "replicas" if n_gpus > 1 else "single", "l2": "flushed between steps"}


class SquareStep:
    """Device buffers of one square workload and its step: fa_fwd, then the
    three backward stages, each bracketed by CUDA events on the launching
    stream."""

    def __init__(self, fa, w, dev):
        import torch
        from synthetic import algorithmic_fwd_flops, make_inputs
        self.fa, self.w = fa, w
        B, H, N, d = w.B, w.H, w.N, w.d
        self.case = make_inputs(w)
        c = self.case
        self.Q, self.K, self.V, self.dO = (c[k].to(dev).contiguous() for k in ("Q", "K", "V", "dO"))
        self.kl = None if c["key_len"] is None else c["key_len"].to(dev)
        self.bm = None if c["block_mask"] is None else c["block_mask"].contiguous().to(dev)
        self.O = torch.empty_like(self.Q)
        self.LSE = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        self.dQ, self.dK, self.dV = (torch.empty_like(self.Q) for _ in range(3))
        self.wsb = fa.fa_bwd_workspace_size(B, H, N, d)
        self.wsf = fa.fa_fwd_workspace_size(B, H, N, d)
        self.ws_f = fa.workspace(self.wsf, dev)
        self.ws_b = fa.workspace(self.wsb, dev)
        self.stream = torch.cuda.current_stream(dev)
        self.flops_fwd = algorithmic_fwd_flops(B, H, N, d, w.causal,
                                               None if c["key_len"] is None else c["key_len"].tolist(),
                                               None if c["block_mask"] is None else c["block_mask"])
        self.ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        self.bwd_name = "fa_bwd128_kernel" if d == 128 else "fa_bwd64_kernel"

    def _check(self, st, where):
        if st != 0:
            raise RuntimeError("%s failed: %s" % (where, self.fa.fa_status_string(st)))

    def run(self, record):
        """One step; record: False, "ends" (events 0 and 4 only) or True (an event between calls)."""
        fa, w, s, ev = self.fa, self.w, self.stream.cuda_stream, self.ev
        B, H, N, d = w.B, w.H, w.N, w.d
        if record:
            ev[0].record(self.stream)
        self._check(fa.fa_fwd(self.Q, self.K, self.V, self.O, self.LSE, B, H, N, d, w.softmax_scale, w.causal,
                              self.kl, self.bm, self.ws_f, self.wsf, s), "fa_fwd")
        if record is True:
            ev[1].record(self.stream)
        self._check(fa.fa_bwd_preprocess(self.O, self.dO, B, H, N, d, self.ws_b, self.wsb, s), "fa_bwd_preprocess")
        if record is True:
            ev[2].record(self.stream)
        self._check(fa.fa_bwd_main(self.Q, self.K, self.V, self.LSE, self.dO, self.dK, self.dV, B, H, N, d,
                                   w.softmax_scale, w.causal, self.kl, self.bm, self.ws_b, self.wsb, s), "fa_bwd_main")
        if record is True:
            ev[3].record(self.stream)
        self._check(fa.fa_bwd_postprocess(self.dQ, B, H, N, d, w.softmax_scale, self.ws_b, self.wsb, s),
                    "fa_bwd_postprocess")
        if record:
            ev[4].record(self.stream)

    def status(self, where):
        for wsx in (self.ws_f, self.ws_b):
            self._check(self.fa.fa_get_device_status(wsx, self.stream.cuda_stream), where)

    def time(self, steps, warmup, flush, on_start=None):
        """Mean ms per stage over `steps` timed steps, then of the whole step
        over `steps` more (L2 flushed before each, outside the events).
        on_start runs after the warm-up, before timing."""
        import torch
        for _ in range(warmup):
            self.run(False)
        torch.cuda.synchronize()
        self.status("device status after warm-up")
        if on_start is not None:
            on_start()
        times = {"step": [], "step_staged": [], "fwd": [], "pre": [], "main": [], "post": []}
        barrier()
        torch.cuda.synchronize()
        for _ in range(steps):
            flush.zero_()
            self.run(True)
            ev = self.ev
            ev[4].synchronize()
            times["fwd"].append(ev[0].elapsed_time(ev[1]))
            times["pre"].append(ev[1].elapsed_time(ev[2]))
            times["main"].append(ev[2].elapsed_time(ev[3]))
            times["post"].append(ev[3].elapsed_time(ev[4]))
            times["step_staged"].append(ev[0].elapsed_time(ev[4]))
        # the step itself, timed with events at its ends only: an event between
        # two calls would separate kernels that otherwise overlap (each is
        # launched to be scheduled while the one before it drains)
        for _ in range(steps):
            flush.zero_()
            self.run("ends")
            self.ev[4].synchronize()
            times["step"].append(self.ev[0].elapsed_time(self.ev[4]))
        torch.cuda.synchronize()
        barrier()
        return {k: sum(v) / len(v) for k, v in times.items()}


def per_config_entry(st, mean, peak):
    """Forward and forward+backward figures of one configuration."""
    f = st.flops_fwd
    bwd_ms = mean["pre"] + mean["main"] + mean["post"]
    fwd_tf = f / (mean["fwd"] / 1e3) / 1e12
    bwd_tf = 2.5 * f / (bwd_ms / 1e3) / 1e12
    step_tf = FWD_BWD_FACTOR * f / (mean["step"] / 1e3) / 1e12
    return {"fwd_ms": mean["fwd"], "bwd_ms": bwd_ms, "bwd_main_ms": mean["main"], "fwd_bwd_ms": mean["step"],
            "fwd_tflops": fwd_tf, "bwd_tflops": bwd_tf, "fwd_bwd_tflops": step_tf,
            "fwd_frac_of_peak": fwd_tf / peak, "bwd_frac_of_peak": bwd_tf / peak,
            "fwd_bwd_frac_of_peak": step_tf / peak, "algorithmic_fwd_flops": f}


def run_ours(args):
    import torch

    ws_n, rank = init_dist("nccl")
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import io_aware_exact_09_gb300 as fa
    from synthetic import WORKLOADS
    fa.build()
    w = WORKLOADS[args.workload]
    B, H, N, d = w.B, w.H, w.N, w.d
    st = SquareStep(fa, w, dev)
    case, scale = st.case, w.softmax_scale
    flops_fwd = st.flops_fwd
    flops_step = FWD_BWD_FACTOR * flops_fwd
    flops_main = 2.5 * flops_fwd

    def check(s, where):
        if s != 0:
            raise RuntimeError("%s failed: %s" % (where, fa.fa_status_string(s)))

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)     # 256 MiB > 129 MB L2
    clocks = ClockSampler(local)

    def start_clocks():
        clocks.start()
        time.sleep(0.3)

    mean = st.time(args.steps, args.warmup, flush, on_start=start_clocks)
    clk = clocks.stop()
    st.status("device status after timing")
    launches = 4 * args.steps

    step_ms = reduce_max(mean["step"], dev)
    value = whole_job_tflops(flops_step, ws_n, step_ms / 1e3)
    fwd_tf = flops_fwd / (mean["fwd"] / 1e3) / 1e12
    bwd_tf = 2.5 * flops_fwd / ((mean["pre"] + mean["main"] + mean["post"]) / 1e3) / 1e12

    peaks, peak_src = measured_peaks()
    peak_tf, peak_kind = pick_peak(peaks, clk)
    # dominant kernel of the step
    bwd_name = st.bwd_name
    dom = bwd_name if mean["main"] >= mean["fwd"] else "fa_fwd_kernel"
    dom_ms = mean["main"] if dom == bwd_name else mean["fwd"]
    dom_flops = flops_main if dom == bwd_name else flops_fwd
    achieved = dom_flops / (dom_ms / 1e3) / 1e12
    roofline = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                "frac": achieved / peak_tf, "traffic": ncu_traffic(dom, w.name),
                "ncu_tensor_pipe_active_pct": ncu_tensor_pipe(dom, w.name),
                "kernel_ms": dom_ms, "algorithmic_flops_per_launch": dom_flops,
                "peak_source": "%s %s" % (peak_src, peak_kind)}

    # the other configurations, the same timing loop, a few steps each
    per_config = {}
    if not args.no_per_config and ws_n == 1:
        for name in PER_CONFIG:
            if name == w.name:
                continue
            sx = SquareStep(fa, WORKLOADS[name], dev)
            mx = sx.time(max(3, min(args.steps, 10)), 3, flush)
            sx.status("device status after timing " + name)
            per_config[name] = per_config_entry(sx, mx, peak_tf)
            del sx
        per_config[w.name] = per_config_entry(st, mean, peak_tf)

    # end-to-end through the host-buffer entry point (pinned memory, copies timed)
    e2e = None
    if not args.no_e2e:
        pin = lambda t: t.contiguous().pin_memory()
        Qh, Kh, Vh, dOh = (pin(case[k]) for k in ("Q", "K", "V", "dO"))
        Oh = torch.empty_like(Qh).pin_memory()
        Lh = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
        dQh, dKh, dVh = (torch.empty_like(Qh).pin_memory() for _ in range(3))
        klh = None if case["key_len"] is None else case["key_len"].contiguous()
        bmh = None if case["block_mask"] is None else case["block_mask"].contiguous()
        hws_n = fa.fa_host_workspace_size(B, H, N, d, 1)
        del flush
        hws = fa.workspace(hws_n, dev)
        stream = st.stream
        sp = stream.cuda_stream
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        et = []
        n_e2e = max(1, min(args.steps, 5))
        for i in range(1 + n_e2e):
            e0.record(stream)
            check(fa.fa_attention_host(Qh, Kh, Vh, dOh, Oh, Lh, dQh, dKh, dVh, B, H, N, d, scale, w.causal, klh,
                                       bmh, hws, hws_n, sp), "fa_attention_host")
            e1.record(stream)
            e1.synchronize()
            if i > 0:
                et.append(e0.elapsed_time(e1))
        e_ms = reduce_max(sum(et) / len(et), dev)
        nbytes = B * H * N * d * 2
        e2e = {"value": whole_job_tflops(flops_step, ws_n, e_ms / 1e3), "unit": "TFLOP/s",
               "h2d_bytes_per_step": 4 * nbytes + (0 if klh is None else 4 * B) + (0 if bmh is None else bmh.numel()),
               "d2h_bytes_per_step": 4 * nbytes + B * H * N * 4, "ms_per_step": e_ms}

    cpu = None
    if rank == 0 and ws_n == 1 and not args.no_cpu_baseline:
        tf, cores, desc, _ = oracle_sample(w, sample_tokens(w, args.cpu_tokens), budget_s=args.cpu_budget)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc}

    if rank == 0:
        line = {
            "metric": "attention fwd+bwd TFLOP/s (bf16)", "value": value, "unit": "TFLOP/s", "n_gpus": ws_n,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config(w, ws_n),
            "fwd_tflops": fwd_tf, "bwd_tflops": bwd_tf,
            "fwd_frac_of_peak": fwd_tf / peak_tf, "bwd_frac_of_peak": bwd_tf / peak_tf,
            "fwd_bwd_frac_of_peak": value / ws_n / peak_tf,
            "kernel_ms": {"fa_fwd_kernel": mean["fwd"], "fa_bwd_pre_kernel": mean["pre"],
                          bwd_name: mean["main"], "fa_bwd_convert_kernel": mean["post"]},
            "algorithmic_flops_per_step": flops_step,
            "roofline": roofline, "per_config": per_config, "cpu_baseline": cpu, "e2e": e2e, "clocks": clk,
            "gpu_launches": launches,
        }
        print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of repeated oracle calls behind cpu_baseline")
    ap.add_argument("--cpu-tokens", type=int, default=4096,
                    help="tokens of the one-head sample the oracle is timed on (both arms)")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the short timings of the other configurations")
    ap.add_argument("--fp8", action="store_true", help="measure the FP8 forward (d = 128 workloads)")
    ap.add_argument("--incoherent", action="store_true",
                    help="with --fp8: quantise Q and K with incoherent processing (Hadamard rotation)")
    ap.add_argument("--tile-sweep", action="store_true", help="time the forward at each tile shape")
    ap.add_argument("--decode-reps", type=int, default=20,
                    help="decode workloads: timed calls per step (each one is well under a millisecond)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    from synthetic import DECODE_WORKLOADS, VARLEN_WORKLOADS
    if args.workload in DECODE_WORKLOADS:
        return run_decode(args, DECODE_WORKLOADS[args.workload])
    if args.workload in VARLEN_WORKLOADS:
        return run_varlen(args, VARLEN_WORKLOADS[args.workload])
    if args.fp8:
        return run_fp8(args)
    if args.tile_sweep:
        return run_tile_sweep(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
