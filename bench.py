#!/usr/bin/env python
"""Attention throughput on GB300: TFLOPS of the fused forward + backward step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Workload (one "step" = one pass of the whole hot path over one batch): the training
shape B=4, Hq=Hkv=16, N=2048, d=128, bf16, non-causal, inputs i.i.d. N(0,1) drawn from a
seeded generator; the step runs attn_fwd then attn_bwd.  FLOPs: forward 4*B*Hq*N^2*d,
backward 2.5x that.  Multi-GPU: one process per GPU, every rank runs its own copy of the
workload (the path shards over independent (batch, head) units with no exchange), so
scaling is weak and ``value`` is the total over ranks divided by the slowest rank's time.

Printed: one JSON line on rank 0 (see the fields in ``main``).  ``--impl reference``
times the fp64 CPU oracle on a bounded sample of the same workload on the host cores.
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

METRIC = "attention fwd/bwd TFLOPS (BF16, d=128, 1×GB300) and fraction of 2.25 PF peak"
UNIT = "TFLOP/s"
NOMINAL_PEAK_TFLOPS = 2250.0
WORKLOAD = dict(name="train_fwd_bwd_B4_H16_N2048_d128", seed=2, B=4, Hq=16, Hkv=16, N=2048, d=128, causal=False)
FWD_SWEEP = (4096, 8192, 16384)          # forward-only lines at d=128, non-causal, B*N = 16384
L2_FLUSH_BYTES = 512 << 20
E2E_STREAMS = 2                           # end-to-end leg: batch chunks' kernels alternate over these streams


def fwd_flops(B, Hq, N, d, causal):
    return 4.0 * B * Hq * N * N * d * (0.5 if causal else 1.0)


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-sweep", action="store_true", help="skip the forward-only sequence sweep lines")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline leg")
    ap.add_argument("--profile", action="store_true",
                    help="short run for a profiler: warm-up plus the timed steps only (no e2e, sweep or CPU leg)")
    ap.add_argument("--case", default=None,
                    help="run one kernel configuration (see CASES) --warmup + --steps times and print its "
                         "median time: a small, single-kernel target for a profiler")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.steps < 1:
        ap.error("--steps must be >= 1")
    return args


# ------------------------------------------------------------------------------ ranks
def dist_env():
    """(rank, world, local_rank) from the torchrun environment (1 process = 1 GPU)."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def dist_init(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        os.environ.setdefault("MASTER_PORT", "29511")
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, value: float, device=None) -> float:
    """Largest value over all ranks (the slowest rank's time)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def combine(per_rank_units: float, world: int, max_seconds: float) -> float:
    """Whole-job throughput: units every rank processed / the slowest rank's time."""
    return per_rank_units * world / max_seconds if max_seconds > 0 else 0.0


# ------------------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clock / throttle samples every 200 ms while the timed region runs."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self._t = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self._t is not None:
                self._t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------------ helpers
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}, "fallback"


def recorded_traffic(kernel: str):
    """dram bytes per launch from the committed ncu summary, or None if the kernel's source
    changed since the counters were taken (the summary stores the source's sha256)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel)
    except (OSError, ValueError):
        return None
    if not rec:
        return None
    src = os.path.join(ROOT, "attention_attn_fwd_09_gb300", "csrc", rec["source"])
    try:
        with open(src, "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()
    except OSError:
        return None
    if sha != rec.get("sha256") or rec.get("workload") != WORKLOAD["name"]:
        return None
    return rec.get("bytes_per_launch")


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_sample(seconds_fwd: float = 6.0, seconds_bwd: float = 8.0):
    """Time the fp64 CPU oracle on whole heads of the workload until each leg has run for
    about the given time.  Returns (flops, seconds, description)."""
    os.environ.setdefault("OMP_NUM_THREADS", str(host_cores()))
    import oracle
    from attn_inputs import make_inputs
    w = WORKLOAD
    x = make_inputs(w["seed"], w["B"], w["Hq"], w["Hkv"], w["N"], w["d"], with_grad=True)
    scale = w["d"] ** -0.5
    oracle.build()
    ff = fwd_flops(1, 1, w["N"], w["d"], w["causal"])
    heads = [(b, h) for b in range(w["B"]) for h in range(w["Hq"])]
    flops, secs, nf, nb = 0.0, 0.0, 0, 0
    t0 = time.perf_counter()
    for bh in heads:
        oracle.attn_fwd(x["q"], x["k"], x["v"], w["causal"], scale, heads=[bh])
        nf += 1
        if time.perf_counter() - t0 >= seconds_fwd:
            break
    t1 = time.perf_counter()
    kv = [(b, h) for b in range(w["B"]) for h in range(w["Hkv"])]
    for bh in kv:
        oracle.attn_bwd(x["q"], x["k"], x["v"], x["do"], w["causal"], scale, kv_heads=[bh])
        nb += 1
        if time.perf_counter() - t1 >= seconds_bwd:
            break
    t2 = time.perf_counter()
    g = w["Hq"] // w["Hkv"]
    flops = nf * ff + nb * g * 2.5 * ff
    secs = t2 - t0
    desc = (f"fp64 oracle on {nf} of {len(heads)} query heads (forward) and {nb} of {len(kv)} key/value "
            f"heads (backward) of the workload, {secs:.1f} s")
    return flops, secs, desc


# ------------------------------------------------------------------------------ our arm
def varlen_lines(A, torch, dev, flush):
    """Lines for the packed mixed-length batch (65536 tokens in sequences of 256..8192, 16
    heads, d = 128): forward and backward, with the work longest first (the library's
    default) and in no particular order, causal and not.  Forward FLOPs 4*d*Hq*sum(nq*nk),
    halved for causal; backward 2.5 times that."""
    from attn_inputs import make_varlen_inputs, varlen_workload
    w = varlen_workload()
    x = make_varlen_inputs(w["seed"], w["lens"], w["lens"], w["Hq"], w["Hkv"], w["d"])
    q, k, v, cq, ck = (x[n].to(dev) for n in ("q", "k", "v", "cu_q", "cu_k"))
    do = torch.randn(q.shape, generator=torch.Generator(device=dev).manual_seed(8), device=dev).to(torch.bfloat16)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    bws = torch.empty((A.attn_bwd_varlen_workspace_size(len(w["lens"]), w["Hq"], w["Hkv"], q.shape[1], k.shape[1],
                                                         w["d"], False),), dtype=torch.uint8, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((w["Hq"], q.shape[1]), dtype=torch.float32, device=dev)
    ws = torch.empty((A.attn_fwd_varlen_workspace_size(len(w["lens"]), w["Hq"], w["Hkv"], q.shape[1], w["d"]),),
                     dtype=torch.uint8, device=dev)
    full = 4.0 * w["d"] * w["Hq"] * sum(n * n for n in w["lens"])
    res = {"sequences": len(w["lens"]), "tokens": int(q.shape[1]), "min_len": min(w["lens"]),
           "max_len": max(w["lens"])}
    def timed(call):
        for _ in range(3):
            call()
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(8)]
        for e in evs:
            flush.fill_(1.0)
            e[0].record()
            call()
            e[1].record()
        torch.cuda.synchronize()
        return statistics.median(e[0].elapsed_time(e[1]) for e in evs)

    scale = w["d"] ** -0.5
    for causal in (False, True):
        for order in (True, False):
            A.attn_set_varlen_order(order)
            fwd = lambda: A.attn_fwd_varlen(q, k, v, cq, ck, causal=causal, scale=scale, o=o, lse=lse, workspace=ws)
            bwd = lambda: A.attn_bwd_varlen(q, k, v, o, lse, do, cq, ck, causal=causal, scale=scale, dq=dq, dk=dk,
                                            dv=dv, workspace=bws)
            ms_f = timed(fwd)
            ms_b = timed(bwd)
            ff = full * (0.5 if causal else 1.0)
            res[f"{'causal' if causal else 'noncausal'}_{'longest_first' if order else 'unordered'}"] = {
                "fwd_ms": round(ms_f, 4), "fwd_tflops": round(ff / ms_f / 1e9, 1),
                "bwd_ms": round(ms_b, 4), "bwd_tflops": round(2.5 * ff / ms_b / 1e9, 1)}
    A.attn_set_varlen_order(True)
    if A.attn_device_status(True) != 0:
        raise RuntimeError("a kernel reported a timeout or bad offsets in the packed-sequence lines")
    return res


def wide_lines(A, torch, dev, flush):
    """Lines for wide heads: B=2, H=16, N=8192, d = 192 and 256, non-causal and causal; the
    forward (one-tile kernel, FLOPs 4*B*H*N^2*d, halved for causal) and the backward (the
    column-half kernel, 2.5 times the forward FLOPs, atomic dQ)."""
    res = {}
    B, H, N = 2, 16, 8192
    for d in (192, 256):
        g = torch.Generator(device=dev).manual_seed(9)
        q, k, v = (torch.randn((B, H, N, d), generator=g, device=dev).to(torch.bfloat16) for _ in range(3))
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        do = torch.randn((B, H, N, d), generator=g, device=dev).to(torch.bfloat16)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty((A.attn_bwd_workspace_size(B, H, H, N, d, False),), dtype=torch.uint8, device=dev)
        for causal in (False, True):
            call = lambda: A.attn_fwd(q, k, v, causal=causal, scale=d ** -0.5, o=o, lse=lse)
            for _ in range(3):
                call()
            evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(8)]
            for e in evs:
                flush.fill_(1.0)
                e[0].record()
                call()
                e[1].record()
            torch.cuda.synchronize()
            ms = statistics.median(e[0].elapsed_time(e[1]) for e in evs)
            tf = fwd_flops(B, H, N, d, causal) / ms / 1e9
            msb = _median_ms(torch, flush, lambda: A.attn_bwd(q, k, v, o, lse, do, causal=causal, scale=d ** -0.5,
                                                              dq=dq, dk=dk, dv=dv, workspace=ws))
            tfb = 2.5 * fwd_flops(B, H, N, d, causal) / msb / 1e9
            res[f"d{d}_{'causal' if causal else 'noncausal'}"] = {
                "ms": round(ms, 4), "tflops": round(tf, 1), "frac_of_2250": round(tf / NOMINAL_PEAK_TFLOPS, 4),
                "bwd_ms": round(msb, 4), "bwd_tflops": round(tfb, 1), "bwd_frac_of_2250": round(tfb / NOMINAL_PEAK_TFLOPS, 4)}
        del q, k, v, o, lse, do, dq, dk, dv, ws
    if A.attn_device_status(True) != 0:
        raise RuntimeError("a kernel reported a timeout in the wide-head lines")
    return res


def _median_ms(torch, flush, call, reps=8, warm=3):
    for _ in range(warm):
        call()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(reps)]
    for e in evs:
        if flush is not None:
            flush.fill_(1.0)
        e[0].record()
        call()
        e[1].record()
    torch.cuda.synchronize()
    return statistics.median(e[0].elapsed_time(e[1]) for e in evs)


def suite_lines(A, torch, dev, flush):
    """The measurement suite's other configurations (the training-shape step causal and not,
    atomic and deterministic; the forward sweep over N = 512 .. 16384,
    d = 64 and 128, causal and not; grouped / multi-query heads at N = 8192 with outlier
    inputs; the backward at N = 8192 and 16384, atomic and deterministic).  Each line:
    median ms over 8 calls (L2 flushed before each), TFLOP/s, and the roofline ceiling
    min(tensor peak, arithmetic intensity x HBM bandwidth) from MEASURED_PEAKS.json."""
    from attn_inputs import make_inputs
    peaks, _ = measured_peaks()
    tpeak, hbm = float(peaks["bf16_tflops"]), float(peaks["hbm_gbs"])

    def fwd_bytes(B, Hq, Hkv, N, d):
        return 2.0 * (2 * B * Hq * N * d + 2 * B * Hkv * N * d) + 4.0 * B * Hq * N

    res = {"sweep": {}, "gqa_outliers": {}, "bwd_long": {}, "train": {}}
    # The training-shape step (B=4, H=16, N=2048, d=128, seed 2), causal and not, atomic and
    # deterministic dQ: forward, backward and the step's TFLOP/s (3.5 x the forward FLOPs).
    x = make_inputs(2, 4, 16, 16, 2048, 128, with_grad=True)
    q, k, v, do = (x[nm].to(dev) for nm in ("q", "k", "v", "do"))
    o, lse = torch.empty_like(q), torch.empty((4, 16, 2048), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    for causal in (False, True):
        fl = fwd_flops(4, 16, 2048, 128, causal)
        msf = _median_ms(torch, flush, lambda: A.attn_fwd(q, k, v, causal=causal, scale=128 ** -0.5, o=o, lse=lse))
        for det in (False, True):
            ws = torch.empty((A.attn_bwd_workspace_size(4, 16, 16, 2048, 128, det),), dtype=torch.uint8, device=dev)
            msb = _median_ms(torch, flush, lambda: A.attn_bwd(q, k, v, o, lse, do, causal=causal, scale=128 ** -0.5,
                                                              deterministic=det, dq=dq, dk=dk, dv=dv, workspace=ws))
            res["train"][f"{'causal' if causal else 'noncausal'}_{'det' if det else 'atomic'}"] = {
                "fwd_ms": round(msf, 4), "bwd_ms": round(msb, 4), "fwd_tflops": round(fl / msf / 1e9, 1),
                "bwd_tflops": round(2.5 * fl / msb / 1e9, 1), "step_tflops": round(3.5 * fl / (msf + msb) / 1e9, 1)}
            del ws
    del x, q, k, v, do, o, lse, dq, dk, dv
    for d in (64, 128):
        for n in (512, 1024, 2048, 4096, 8192, 16384):
            b = 16384 // n
            g = torch.Generator(device=dev).manual_seed(3)
            q, k, v = (torch.randn((b, 16, n, d), generator=g, device=dev).to(torch.bfloat16) for _ in range(3))
            o, lse = torch.empty_like(q), torch.empty((b, 16, n), dtype=torch.float32, device=dev)
            for causal in (False, True):
                ms = _median_ms(torch, flush, lambda: A.attn_fwd(q, k, v, causal=causal, scale=d ** -0.5, o=o, lse=lse))
                fl = fwd_flops(b, 16, n, d, causal)
                ceil = min(tpeak, fl / fwd_bytes(b, 16, 16, n, d) * hbm / 1e3)
                res["sweep"][f"d{d}_N{n}_{'causal' if causal else 'noncausal'}"] = {
                    "B": b, "ms": round(ms, 4), "tflops": round(fl / ms / 1e9, 1), "ceiling_tflops": round(ceil, 1)}
            del q, k, v, o, lse
    for hkv in (8, 1):
        x = make_inputs(4, 2, 32, hkv, 8192, 128, recipe="outliers")
        q, k, v = (x[nm].to(dev) for nm in ("q", "k", "v"))
        o, lse = torch.empty_like(q), torch.empty((2, 32, 8192), dtype=torch.float32, device=dev)
        ms = _median_ms(torch, flush, lambda: A.attn_fwd(q, k, v, causal=True, scale=128 ** -0.5, o=o, lse=lse))
        fl = fwd_flops(2, 32, 8192, 128, True)
        res["gqa_outliers"][f"Hq32_Hkv{hkv}_N8192_causal"] = {"ms": round(ms, 4), "tflops": round(fl / ms / 1e9, 1)}
        del x, q, k, v, o, lse
    for n in (8192, 16384):
        g = torch.Generator(device=dev).manual_seed(5)
        q, k, v, do = (torch.randn((2, 16, n, 128), generator=g, device=dev).to(torch.bfloat16) for _ in range(4))
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        for causal in (False, True):
            o, lse = A.attn_fwd(q, k, v, causal=causal)
            for det in (False, True):
                ws = torch.empty((A.attn_bwd_workspace_size(2, 16, 16, n, 128, det),), dtype=torch.uint8, device=dev)
                ms = _median_ms(torch, flush, lambda: A.attn_bwd(q, k, v, o, lse, do, causal=causal, deterministic=det,
                                                                 dq=dq, dk=dk, dv=dv, workspace=ws))
                fl = 2.5 * fwd_flops(2, 16, n, 128, causal)
                res["bwd_long"][f"N{n}_{'causal' if causal else 'noncausal'}_{'det' if det else 'atomic'}"] = {
                    "ms": round(ms, 4), "tflops": round(fl / ms / 1e9, 1)}
                del ws
        del q, k, v, do, dq, dk, dv
    if A.attn_device_status(True) != 0:
        raise RuntimeError("a kernel reported a timeout in the suite lines")
    return res


def fp8_lines(A, torch, dev, flush):
    """FP8 forward (e4m3 Q/K/V with per-128-row block scales, d = 128) at the forward
    sweep's shapes (B = 16384 / N, 16 heads): TFLOP/s with the same FLOP count as the bf16
    forward, next to the bf16 forward on the same inputs, and the quantiser's bandwidth
    (2 bytes read and 1 written per element, plus the scales)."""
    peaks, _ = measured_peaks()
    res = {}
    for n in (4096, 8192, 16384):
        b = 16384 // n
        g = torch.Generator(device=dev).manual_seed(3)
        q, k, v = (torch.randn((b, 16, n, 128), generator=g, device=dev).to(torch.bfloat16) for _ in range(3))
        q8, sq = A.attn_quantize_fp8(q)
        k8, sk = A.attn_quantize_fp8(k)
        v8, sv = A.attn_quantize_fp8(v)
        o, lse = torch.empty_like(q), torch.empty((b, 16, n), dtype=torch.float32, device=dev)
        for causal in (False, True):
            ms = _median_ms(torch, flush, lambda: A.attn_fwd_fp8(q8, k8, v8, sq, sk, sv, causal=causal,
                                                                 scale=128 ** -0.5, o=o, lse=lse))
            ms16 = _median_ms(torch, flush, lambda: A.attn_fwd(q, k, v, causal=causal, scale=128 ** -0.5, o=o,
                                                               lse=lse))
            fl = fwd_flops(b, 16, n, 128, causal)
            res[f"N{n}_{'causal' if causal else 'noncausal'}"] = {
                "B": b, "ms": round(ms, 4), "tflops": round(fl / ms / 1e9, 1), "bf16_ms": round(ms16, 4),
                "bf16_tflops": round(fl / ms16 / 1e9, 1)}
        if n == 4096:
            msq = _median_ms(torch, flush, lambda: A.attn_quantize_fp8(q, q8, sq))
            nbytes = 3.0 * q.numel() + 4.0 * sq.numel()
            res["quantize_B4_H16_N4096"] = {"ms": round(msq, 4), "gbs": round(nbytes / msq / 1e6, 1),
                                            "frac_of_hbm": round(nbytes / msq / 1e6 / float(peaks["hbm_gbs"]), 4)}
        del q, k, v, q8, k8, v8, o, lse
    if A.attn_device_status(True) != 0:
        raise RuntimeError("a kernel reported a timeout in the FP8 lines")
    return res


def decode_lines(A, torch, dev, flush):
    """Decoding against a key/value cache (attn_fwd_kv): B=8, Hq=32, Hkv=8, Nk=8192, d=128,
    causal, Nq new queries per head.  The forward reads the whole cache once, so the line
    is reported as cache bandwidth: bytes of K and V (2*B*Hkv*Nk*d*2) plus Q, O and LSE,
    over the median time, against the measured HBM copy bandwidth."""
    from attn_inputs import make_inputs
    peaks, _ = measured_peaks()
    hbm = float(peaks["hbm_gbs"])
    B, Hq, Hkv, Nk, d = 8, 32, 8, 8192, 128
    x = make_inputs(6, B, Hq, Hkv, Nk, d)
    k, v = x["k"].to(dev), x["v"].to(dev)
    res = {}
    for nq in (1, 16, 128):
        q = x["q"][:, :, Nk - nq:].contiguous().to(dev)
        o = torch.empty_like(q)
        lse = torch.empty((B, Hq, nq), dtype=torch.float32, device=dev)
        ws = torch.empty((max(A.attn_fwd_kv_workspace_size(B, Hq, Hkv, nq, Nk, d), 16),), dtype=torch.uint8,
                         device=dev)
        # The cache (268 MB of K and V) is larger than L2, so no flush between calls: writing a
        # flush buffer right before a bandwidth-bound call leaves its dirty lines to drain to
        # HBM during the call.
        ms = _median_ms(torch, None, lambda: A.attn_fwd_kv(q, k, v, causal=True, scale=d ** -0.5, o=o, lse=lse,
                                                           workspace=ws))
        nbytes = 2.0 * B * Hkv * Nk * d * 2 + 2.0 * B * Hq * nq * d * 2 + 4.0 * B * Hq * nq
        gbs = nbytes / ms / 1e6
        res[f"Nq{nq}"] = {"ms": round(ms, 4), "cache_gbs": round(gbs, 1), "frac_of_hbm": round(gbs / hbm, 4),
                          "grouped": A.attn_fwd_kv_workspace_size(B, Hq, Hkv, nq, Nk, d) > 0}
    res["workload"] = "B8_Hq32_Hkv8_Nk8192_d128_causal"
    res["l2"] = "no flush: the 268 MB cache read per call is larger than L2"
    res["hbm_peak_gbs"] = hbm
    if A.attn_device_status(True) != 0:
        raise RuntimeError("a kernel reported a timeout in the decode lines")
    return res


def rescale_lines(A, torch, dev):
    """Conditional rescale on the grouped-head outlier workload (B=2, Hq=32, Hkv 8 and 1,
    N=8192, d=128, causal): the number of (row, key block) steps after a row's first block
    in which O was rescaled, with tau = 0 (every growth of the maximum) and tau = 8 (the
    default), counted once each outside any timed region."""
    from attn_inputs import make_inputs
    res = {}
    for hkv in (8, 1):
        x = make_inputs(4, 2, 32, hkv, 8192, 128, recipe="outliers")
        q, k, v = (x[nm].to(dev) for nm in ("q", "k", "v"))
        counts = {}
        for tau in (0.0, 8.0):
            A.attn_set_debug_knobs(tau=tau)
            A.attn_rescale_counter(True)
            A.attn_fwd(q, k, v, causal=True, scale=128 ** -0.5)
            counts[tau] = A.attn_rescale_counter(False)
        A.attn_set_debug_knobs()
        res[f"Hq32_Hkv{hkv}_N8192_causal"] = {
            "rescales_tau0": counts[0.0], "rescales_tau8": counts[8.0],
            "skipped_pct": round(100.0 * (1.0 - counts[8.0] / max(counts[0.0], 1)), 2)}
        del x, q, k, v
    if A.attn_device_status(True) != 0:
        raise RuntimeError("a kernel reported a timeout in the rescale lines")
    return res


def _case_table():
    """Single-configuration runs for a profiler (``--case NAME``): name -> (description,
    setup(A, torch, dev) -> callable)."""
    def fwd(b, h, hkv, n, d, causal, poly=0, recipe="normal", seed=3, persistent=False):
        def setup(A, torch, dev):
            from attn_inputs import make_inputs
            A.attn_set_fwd_persistent(persistent)
            x = make_inputs(seed, b, h, hkv, n, d, recipe=recipe)
            q, k, v = (x[nm].to(dev) for nm in ("q", "k", "v"))
            o, lse = torch.empty_like(q), torch.empty((b, h, n), dtype=torch.float32, device=dev)
            A.attn_set_debug_knobs(poly_per_16=poly)
            return lambda: A.attn_fwd(q, k, v, causal=causal, scale=d ** -0.5, o=o, lse=lse)
        return setup

    def bwd(b, h, n, d, causal, det=False, seed=5, tile=None):
        def setup(A, torch, dev):
            from attn_inputs import make_inputs
            if tile is not None:
                A.attn_set_bwd_query_tile(tile)
            x = make_inputs(seed, b, h, h, n, d, with_grad=True)
            q, k, v, do = (x[nm].to(dev) for nm in ("q", "k", "v", "do"))
            o, lse = A.attn_fwd(q, k, v, causal=causal)
            dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
            ws = torch.empty((A.attn_bwd_workspace_size(b, h, h, n, d, det),), dtype=torch.uint8, device=dev)
            return lambda: A.attn_bwd(q, k, v, o, lse, do, causal=causal, deterministic=det, dq=dq, dk=dk, dv=dv,
                                      workspace=ws)
        return setup

    def varlen(backward, causal):
        def setup(A, torch, dev):
            from attn_inputs import make_varlen_inputs, varlen_workload
            w = varlen_workload()
            x = make_varlen_inputs(w["seed"], w["lens"], w["lens"], w["Hq"], w["Hkv"], w["d"])
            q, k, v, cq, ck = (x[nm].to(dev) for nm in ("q", "k", "v", "cu_q", "cu_k"))
            o, lse = A.attn_fwd_varlen(q, k, v, cq, ck, causal=causal)
            if not backward:
                return lambda: A.attn_fwd_varlen(q, k, v, cq, ck, causal=causal, o=o, lse=lse)
            do = torch.randn(q.shape, generator=torch.Generator(device=dev).manual_seed(8),
                             device=dev).to(torch.bfloat16)
            return lambda: A.attn_bwd_varlen(q, k, v, o, lse, do, cq, ck, causal=causal)
        return setup

    def fwd_fp8(b, n, causal):
        def setup(A, torch, dev):
            g = torch.Generator(device=dev).manual_seed(3)
            q, k, v = (torch.randn((b, 16, n, 128), generator=g, device=dev).to(torch.bfloat16) for _ in range(3))
            (q8, sq), (k8, sk), (v8, sv) = (A.attn_quantize_fp8(t) for t in (q, k, v))
            o, lse = torch.empty_like(q), torch.empty((b, 16, n), dtype=torch.float32, device=dev)
            return lambda: A.attn_fwd_fp8(q8, k8, v8, sq, sk, sv, causal=causal, o=o, lse=lse)
        return setup

    def decode(nq, one_tile=True):
        def setup(A, torch, dev):
            from attn_inputs import make_inputs
            A.attn_set_decode_one_tile(one_tile)
            B, Hq, Hkv, Nk, d = 8, 32, 8, 8192, 128
            x = make_inputs(6, B, Hq, Hkv, Nk, d)
            k, v = x["k"].to(dev), x["v"].to(dev)
            q = x["q"][:, :, Nk - nq:].contiguous().to(dev)
            o = torch.empty_like(q)
            lse = torch.empty((B, Hq, nq), dtype=torch.float32, device=dev)
            ws = torch.empty((max(A.attn_fwd_kv_workspace_size(B, Hq, Hkv, nq, Nk, d), 16),), dtype=torch.uint8,
                             device=dev)
            return lambda: A.attn_fwd_kv(q, k, v, causal=True, o=o, lse=lse, workspace=ws)
        return setup

    return {
        "fwd_train_B4_H16_N2048": ("forward B4 H16 N2048 d128 non-causal (the training step's inputs)",
                                   fwd(4, 16, 16, 2048, 128, False, seed=2)),
        "fwd_d128_N8192_noncausal": ("forward B2 H16 N8192 d128 non-causal", fwd(2, 16, 16, 8192, 128, False)),
        "fwd_d128_N8192_noncausal_poly4": ("same, 4 of 16 exponentials on the FMA cubic",
                                           fwd(2, 16, 16, 8192, 128, False, poly=4)),
        "fwd_d128_N4096_noncausal": ("forward B4 H16 N4096 d128 non-causal", fwd(4, 16, 16, 4096, 128, False)),
        "fwd_d128_N2048_noncausal": ("forward B8 H16 N2048 d128 non-causal", fwd(8, 16, 16, 2048, 128, False)),
        "fwd_d128_N2048_persistent": ("same, persistent kernel", fwd(8, 16, 16, 2048, 128, False, persistent=True)),
        "fwd_d128_N4096_persistent": ("forward B4 H16 N4096 d128 non-causal, persistent kernel",
                                      fwd(4, 16, 16, 4096, 128, False, persistent=True)),
        "fwd_d128_N8192_persistent": ("forward B2 H16 N8192 d128 non-causal, persistent kernel",
                                      fwd(2, 16, 16, 8192, 128, False, persistent=True)),
        "fwd_d64_N8192_noncausal": ("forward B2 H16 N8192 d64 non-causal", fwd(2, 16, 16, 8192, 64, False)),
        "fwd_d64_N8192_causal": ("forward B2 H16 N8192 d64 causal", fwd(2, 16, 16, 8192, 64, True)),
        "fwd_d64_N4096_noncausal": ("forward B4 H16 N4096 d64 non-causal", fwd(4, 16, 16, 4096, 64, False)),
        "fwd_d64_N2048_noncausal": ("forward B4 H16 N2048 d64 non-causal", fwd(4, 16, 16, 2048, 64, False)),
        "fwd_d64_N16384_noncausal": ("forward B1 H16 N16384 d64 non-causal", fwd(1, 16, 16, 16384, 64, False)),
        "fwd_d256_N8192_noncausal": ("forward B2 H16 N8192 d256 non-causal (one-tile kernel)",
                                     fwd(2, 16, 16, 8192, 256, False, seed=9)),
        "fwd_gqa8_N8192_causal_outliers": ("forward B2 Hq32 Hkv8 N8192 d128 causal, outlier inputs",
                                           fwd(2, 32, 8, 8192, 128, True, recipe="outliers", seed=4)),
        "bwd_train_B4_H16_N2048": ("backward B4 H16 N2048 d128 non-causal", bwd(4, 16, 2048, 128, False, seed=2)),
        "bwd_N8192_noncausal": ("backward B2 H16 N8192 d128 non-causal", bwd(2, 16, 8192, 128, False)),
        "bwd_train_tile64": ("backward B4 H16 N2048 d128 non-causal, 64-row query tiles",
                             bwd(4, 16, 2048, 128, False, seed=2, tile=64)),
        "bwd_train_tile128": ("backward B4 H16 N2048 d128 non-causal, 128-row query tiles",
                              bwd(4, 16, 2048, 128, False, seed=2, tile=128)),
        "bwd_N8192_tile64": ("backward B2 H16 N8192 d128 non-causal, 64-row query tiles",
                             bwd(2, 16, 8192, 128, False, tile=64)),
        "bwd_N8192_causal_tile64": ("backward B2 H16 N8192 d128 causal, 64-row query tiles",
                                    bwd(2, 16, 8192, 128, True, tile=64)),
        "bwd_N8192_causal_tile128": ("backward B2 H16 N8192 d128 causal, 128-row query tiles",
                                     bwd(2, 16, 8192, 128, True, tile=128)),
        "bwd_N8192_det_tile64": ("backward B2 H16 N8192 d128 non-causal deterministic, 64-row query tiles",
                                 bwd(2, 16, 8192, 128, False, det=True, tile=64)),
        "bwd_d64_train_tile64": ("backward B4 H16 N2048 d64 non-causal, 64-row query tiles",
                                 bwd(4, 16, 2048, 64, False, seed=2, tile=64)),
        "bwd_d64_train_tile128": ("backward B4 H16 N2048 d64 non-causal, 128-row query tiles",
                                  bwd(4, 16, 2048, 64, False, seed=2, tile=128)),
        "bwd_d256_N8192_noncausal": ("backward B2 H16 N8192 d256 non-causal (column halves)",
                                     bwd(2, 16, 8192, 256, False)),
        "bwd_d192_N8192_noncausal": ("backward B2 H16 N8192 d192 non-causal (column halves)",
                                     bwd(2, 16, 8192, 192, False)),
        "bwd_N8192_noncausal_det": ("same, deterministic dQ", bwd(2, 16, 8192, 128, False, det=True)),
        "bwd_train_det": ("backward B4 H16 N2048 d128 non-causal, deterministic dQ",
                          bwd(4, 16, 2048, 128, False, det=True, seed=2)),
        "bwd_train_causal_det": ("backward B4 H16 N2048 d128 causal, deterministic dQ",
                                 bwd(4, 16, 2048, 128, True, det=True, seed=2)),
        "bwd_N8192_causal_det": ("backward B2 H16 N8192 d128 causal, deterministic dQ",
                                 bwd(2, 16, 8192, 128, True, det=True)),
        "bwd_N8192_causal": ("backward B2 H16 N8192 d128 causal", bwd(2, 16, 8192, 128, True)),
        "bwd_N16384_noncausal_det": ("backward B1 H16 N16384 d128 non-causal, deterministic dQ",
                                     bwd(1, 16, 16384, 128, False, det=True)),
        "bwd_N16384_noncausal": ("backward B1 H16 N16384 d128 non-causal", bwd(1, 16, 16384, 128, False)),
        "bwd_N16384_causal_det": ("backward B1 H16 N16384 d128 causal, deterministic dQ",
                                  bwd(1, 16, 16384, 128, True, det=True)),
        "varlen_fwd_noncausal": ("packed forward, 18 sequences (65536 tokens), H16 d128", varlen(False, False)),
        "varlen_bwd_noncausal": ("packed backward, same batch", varlen(True, False)),
        "fp8_fwd_N8192_noncausal": ("FP8 forward B2 H16 N8192 d128 non-causal", fwd_fp8(2, 8192, False)),
        "fp8_fwd_N4096_noncausal": ("FP8 forward B4 H16 N4096 d128 non-causal", fwd_fp8(4, 4096, False)),
        "decode_Nq1": ("grouped decode B8 Hq32 Hkv8 Nk8192 d128, 1 query", decode(1)),
        "decode_Nq16": ("grouped decode B8 Hq32 Hkv8 Nk8192 d128, 16 queries", decode(16)),
        "decode_Nq1_two_tile": ("same, 1 query, two-tile kernel", decode(1, False)),
        "decode_Nq16_two_tile": ("same, 16 queries, two-tile kernel", decode(16, False)),
    }


def run_case(args):
    """One configuration, --warmup untimed and --steps timed calls (CUDA events on the
    current stream, no L2 flush): a short, single-kernel program for ncu."""
    import torch
    import attention_attn_fwd_09_gb300 as A
    table = _case_table()
    if args.case not in table:
        raise SystemExit(f"unknown case {args.case!r}; cases: {', '.join(sorted(table))}")
    desc, setup = table[args.case]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    call = setup(A, torch, dev)
    for _ in range(args.warmup):
        call()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for e in evs:
        e[0].record()
        call()
        e[1].record()
    torch.cuda.synchronize()
    A.attn_set_debug_knobs()
    A.attn_set_decode_one_tile(True)
    A.attn_set_fwd_persistent(False)
    if A.attn_device_status(True) != 0:
        raise RuntimeError("a kernel reported a timeout")
    return {"case": args.case, "what": desc, "steps": args.steps, "warmup": args.warmup,
            "median_ms": round(statistics.median(e[0].elapsed_time(e[1]) for e in evs), 4)}


def run_ours(args):
    import torch

    rank, world, local_rank = dist_env()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = dist_init(world, "nccl")
    import attention_attn_fwd_09_gb300 as A
    from attn_inputs import make_inputs

    w = WORKLOAD
    B, Hq, Hkv, N, d, causal = w["B"], w["Hq"], w["Hkv"], w["N"], w["d"], w["causal"]
    scale = d ** -0.5
    x = make_inputs(w["seed"], B, Hq, Hkv, N, d, with_grad=True)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty((max(A.attn_bwd_workspace_size(B, Hq, Hkv, N, d, False), 16),), dtype=torch.uint8,
                     device=dev)
    flush = torch.empty((L2_FLUSH_BYTES // 4,), dtype=torch.float32, device=dev)

    def fwd():
        A.attn_fwd(q, k, v, causal=causal, scale=scale, o=o, lse=lse)

    def bwd():
        A.attn_bwd(q, k, v, o, lse, do, causal=causal, scale=scale, dq=dq, dk=dk, dv=dv, workspace=ws)

    fwd()
    try:
        bwd()
        has_bwd = True
    except A.AttnError as e:
        if e.code != -2:
            raise
        has_bwd = False
    for _ in range(args.warmup):
        fwd()
        if has_bwd:
            bwd()
    torch.cuda.synchronize()
    if A.attn_device_status(True) != 0:
        raise RuntimeError("a kernel reported a timeout during warm-up")

    ff = fwd_flops(B, Hq, N, d, causal)
    step_flops = ff * (3.5 if has_bwd else 1.0)
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    barrier(dist)
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        for i in range(K):
            flush.fill_(float(i))                 # > L2 between timed iterations
            ev[i][0].record()
            fwd()
            ev[i][1].record()
            if has_bwd:
                bwd()
            ev[i][2].record()
        torch.cuda.synchronize()
    barrier(dist)
    if A.attn_device_status(True) != 0:
        raise RuntimeError("a kernel reported a timeout during the timed region")
    fwd_ms = [e[0].elapsed_time(e[1]) for e in ev]
    bwd_ms = [e[1].elapsed_time(e[2]) for e in ev]
    step_ms = [e[0].elapsed_time(e[2]) for e in ev]
    total_s = max_over_ranks(dist, sum(step_ms) / 1e3, dev)
    value = combine(step_flops * K, world, total_s) / 1e12

    if args.profile:
        return {"profile": True, "fwd_ms": round(statistics.mean(fwd_ms), 4),
                "bwd_ms": round(statistics.mean(bwd_ms), 4) if has_bwd else None} if rank == 0 else None

    # End to end through the public API: pinned host inputs in, results back to the host.
    pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t)
    q_h, k_h, v_h, do_h = pin(x["q"]), pin(x["k"]), pin(x["v"]), pin(x["do"])
    outs_h = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in ((o, dq, dk, dv) if has_bwd else (o,))]
    h2d = sum(t.numel() * t.element_size() for t in ((q_h, k_h, v_h, do_h) if has_bwd else (q_h, k_h, v_h)))
    d2h = sum(t.numel() * t.element_size() for t in outs_h) + (lse.numel() * 4)
    lse_h = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
    ee = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    barrier(dist)
    torch.cuda.synchronize()
    for i in range(K):
        flush.fill_(float(i))
        ee[i][0].record()
        q.copy_(q_h, non_blocking=True)
        k.copy_(k_h, non_blocking=True)
        v.copy_(v_h, non_blocking=True)
        if has_bwd:
            do.copy_(do_h, non_blocking=True)
        fwd()
        if has_bwd:
            bwd()
        for t_h, t_d in zip(outs_h, (o, dq, dk, dv)):
            t_h.copy_(t_d, non_blocking=True)
        lse_h.copy_(lse, non_blocking=True)
        ee[i][1].record()
    torch.cuda.synchronize()
    barrier(dist)
    serial_s = max_over_ranks(dist, sum(e[0].elapsed_time(e[1]) for e in ee) / 1e3, dev)
    e2e_serial = combine(step_flops * K, world, serial_s) / 1e12

    # The same step pipelined the way a caller with host-resident data would run it: one
    # chunk per batch element; the input copies go in order on one copy stream, each chunk's
    # kernels on one of two compute streams once its inputs have landed, and the result copies
    # in order on a third stream, so that the two link directions and the kernels overlap.
    # Every chunk still copies its own inputs in and its results out inside the timed region.
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    streams = [torch.cuda.Stream(device=dev) for _ in range(E2E_STREAMS)]
    ws_s = [torch.empty((max(A.attn_bwd_workspace_size(1, Hq, Hkv, N, d, False), 16),), dtype=torch.uint8,
                        device=dev) for _ in streams] if has_bwd else []
    pe = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    main = torch.cuda.current_stream()
    barrier(dist)
    torch.cuda.synchronize()
    for i in range(K):
        flush.fill_(float(i))
        pe[i][0].record(main)
        for st in (s_in, s_out, *streams):
            st.wait_stream(main)
        for b in range(B):
            sl = slice(b, b + 1)
            cs = streams[b % len(streams)]
            with torch.cuda.stream(s_in):
                for t_d, t_h in zip((q, k, v, do) if has_bwd else (q, k, v), (q_h, k_h, v_h, do_h)):
                    t_d[sl].copy_(t_h[sl], non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(s_in)
            cs.wait_event(ev_in)
            with torch.cuda.stream(cs):
                A.attn_fwd(q[sl], k[sl], v[sl], causal=causal, scale=scale, o=o[sl], lse=lse[sl])
                if has_bwd:
                    A.attn_bwd(q[sl], k[sl], v[sl], o[sl], lse[sl], do[sl], causal=causal, scale=scale,
                               dq=dq[sl], dk=dk[sl], dv=dv[sl], workspace=ws_s[b % len(streams)])
                ev_c = torch.cuda.Event()
                ev_c.record(cs)
            s_out.wait_event(ev_c)
            with torch.cuda.stream(s_out):
                for t_h, t_d in zip(outs_h, (o, dq, dk, dv)):
                    t_h[sl].copy_(t_d[sl], non_blocking=True)
                lse_h[sl].copy_(lse[sl], non_blocking=True)
        for st in (s_in, s_out, *streams):
            main.wait_stream(st)
        pe[i][1].record(main)
    torch.cuda.synchronize()
    barrier(dist)
    if A.attn_device_status(True) != 0:
        raise RuntimeError("a kernel reported a timeout in the end-to-end leg")
    e2e_s = max_over_ranks(dist, sum(e[0].elapsed_time(e[1]) for e in pe) / 1e3, dev)
    e2e_value = combine(step_flops * K, world, e2e_s) / 1e12

    # The host link itself: one pinned-to-device copy of the step's input bytes and one
    # device-to-pinned copy of its output bytes, timed alone, as the ceiling of the leg above.
    link = {}
    for name, nbytes, to_dev in (("h2d", h2d, True), ("d2h", d2h, False)):
        hb = torch.empty((nbytes,), dtype=torch.uint8, pin_memory=True)
        db = torch.empty((nbytes,), dtype=torch.uint8, device=dev)
        for _ in range(3):
            (db.copy_(hb, non_blocking=True) if to_dev else hb.copy_(db, non_blocking=True))
        le = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(5)]
        for e in le:
            e[0].record()
            (db.copy_(hb, non_blocking=True) if to_dev else hb.copy_(db, non_blocking=True))
            e[1].record()
        torch.cuda.synchronize()
        link[f"{name}_gbs"] = round(nbytes / statistics.median(e[0].elapsed_time(e[1]) for e in le) / 1e6, 1)
        del hb, db
    # Both directions at once (two streams), as the pipelined leg runs them.
    hb_in = torch.empty((h2d,), dtype=torch.uint8, pin_memory=True)
    db_in = torch.empty((h2d,), dtype=torch.uint8, device=dev)
    hb_out = torch.empty((d2h,), dtype=torch.uint8, pin_memory=True)
    db_out = torch.empty((d2h,), dtype=torch.uint8, device=dev)
    sa, sb = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    both = []
    for r in range(8):
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(main)
        sa.wait_stream(main)
        sb.wait_stream(main)
        with torch.cuda.stream(sa):
            db_in.copy_(hb_in, non_blocking=True)
        with torch.cuda.stream(sb):
            hb_out.copy_(db_out, non_blocking=True)
        main.wait_stream(sa)
        main.wait_stream(sb)
        e1.record(main)
        torch.cuda.synchronize()
        if r >= 3:
            both.append(e0.elapsed_time(e1))
    del hb_in, db_in, hb_out, db_out
    # The slowest of the input copies, the result copies (or both at once) and the kernels
    # bounds a step whose copies and kernels overlap perfectly: the end-to-end ceiling here.
    h2d_ms, d2h_ms, both_ms = h2d / link["h2d_gbs"] / 1e6, d2h / link["d2h_gbs"] / 1e6, statistics.median(both)
    link["h2d_ms"], link["d2h_ms"], link["both_directions_ms"] = round(h2d_ms, 4), round(d2h_ms, 4), round(both_ms, 4)
    link["e2e_ceiling"] = round(step_flops / max(h2d_ms, d2h_ms, both_ms, statistics.mean(step_ms)) / 1e9, 1)

    # Forward-only lines at the lengths the forward target is stated for (d=128, non-causal).
    sweep = {}
    if not args.no_sweep:
        for n in FWD_SWEEP:
            b = 16384 // n
            g = torch.Generator(device=dev).manual_seed(3)
            qs = torch.randn((b, 16, n, 128), generator=g, device=dev).to(torch.bfloat16)
            ks = torch.randn((b, 16, n, 128), generator=g, device=dev).to(torch.bfloat16)
            vs = torch.randn((b, 16, n, 128), generator=g, device=dev).to(torch.bfloat16)
            os_, ls = torch.empty_like(qs), torch.empty((b, 16, n), dtype=torch.float32, device=dev)
            for _ in range(3):
                A.attn_fwd(qs, ks, vs, causal=False, scale=128 ** -0.5, o=os_, lse=ls)
            evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(8)]
            for e in evs:
                flush.fill_(1.0)
                e[0].record()
                A.attn_fwd(qs, ks, vs, causal=False, scale=128 ** -0.5, o=os_, lse=ls)
                e[1].record()
            torch.cuda.synchronize()
            ms = statistics.median(e[0].elapsed_time(e[1]) for e in evs)
            tf = fwd_flops(b, 16, n, 128, False) / ms / 1e9
            sweep[f"N{n}"] = {"B": b, "ms": round(ms, 4), "tflops": round(tf, 1),
                              "frac_of_2250": round(tf / NOMINAL_PEAK_TFLOPS, 4)}
            del qs, ks, vs, os_, ls
        if A.attn_device_status(True) != 0:
            raise RuntimeError("a kernel reported a timeout in the sweep")
        varlen = varlen_lines(A, torch, dev, flush)
        wide = wide_lines(A, torch, dev, flush)
        suite = suite_lines(A, torch, dev, flush)
        decode = decode_lines(A, torch, dev, flush)
        fp8 = fp8_lines(A, torch, dev, flush)
        rescale = rescale_lines(A, torch, dev)

    peaks, peak_src = measured_peaks()
    fwd_avg = statistics.mean(fwd_ms)
    bwd_avg = statistics.mean(bwd_ms) if has_bwd else 0.0
    dominant = "attn_bwd" if has_bwd and bwd_avg > fwd_avg else "attn_fwd_kernel"
    if dominant == "attn_fwd_kernel":
        achieved = ff / fwd_avg / 1e9
    else:
        achieved = 2.5 * ff / bwd_avg / 1e9
    peak = float(peaks["bf16_tflops"])
    roofline = {"bound": "tensor", "kernel": dominant, "achieved": round(achieved, 1), "peak": peak,
                "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                "peak_source": f"{peak_src} bf16 burst (MEASURED_PEAKS.json bf16_tflops)"
                if peak_src == "measured" else "fallback 1.9 PFLOP/s bf16 burst",
                "frac_of_2250": round(achieved / NOMINAL_PEAK_TFLOPS, 4),
                "traffic": recorded_traffic(dominant)}
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(statistics.mean(step_ms), 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1), bf16)",
        "config": {"workload": w["name"], "B": B, "Hq": Hq, "Hkv": Hkv, "seq_len": N, "head_dim": d,
                   "causal": causal, "passes": "fwd+bwd" if has_bwd else "fwd",
                   "l2": "512 MiB buffer written between timed iterations",
                   "parallelism": f"replicas x{world} (independent (batch, head) units)"},
        "fwd_ms": round(fwd_avg, 4), "bwd_ms": round(bwd_avg, 4) if has_bwd else None,
        "fwd_tflops": round(ff / fwd_avg / 1e9, 1),
        "bwd_tflops": round(2.5 * ff / bwd_avg / 1e9, 1) if has_bwd else None,
        "frac_of_2250": round(value / world / NOMINAL_PEAK_TFLOPS, 4),
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "pipelining": f"{B} batch chunks: inputs in order on one copy stream, kernels on {E2E_STREAMS} "
                              "streams, results in order on another copy stream",
                "serial_value": round(e2e_serial, 2), "host_link": link},
        "gpu_launches": K * (1 + (3 if has_bwd else 0)),
        "roofline": roofline,
        "clocks": clk.summary(),
        "fwd_sweep_d128_noncausal": sweep,
    }
    if not args.no_sweep:
        out["varlen_mixed_lengths"] = varlen
        out["fwd_wide_heads"] = wide
        out["suite"] = suite
        out["decode_kv_cache"] = decode
        out["fwd_fp8_e4m3"] = fp8
        out["rescale_skip_outliers"] = rescale
    if rank == 0 and world == 1 and not args.no_cpu:
        flops, secs, desc = oracle_sample()
        out["cpu_baseline"] = {"value": round(flops / secs / 1e12, 6), "unit": UNIT, "cores": host_cores(),
                               "kind": "oracle", "sample": desc}
    if dist is not None:
        dist.destroy_process_group()
    return out if rank == 0 else None


# ------------------------------------------------------------------------------ reference arm
def run_reference(args):
    """The fp64 CPU oracle as the reference arm, on the host cores, rank 0 only."""
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    os.environ.setdefault("OMP_NUM_THREADS", str(host_cores()))
    import oracle
    from attn_inputs import make_inputs
    w = WORKLOAD
    x = make_inputs(w["seed"], w["B"], w["Hq"], w["Hkv"], w["N"], w["d"], with_grad=True)
    scale = w["d"] ** -0.5
    oracle.build()
    ff = fwd_flops(1, 1, w["N"], w["d"], w["causal"])
    g = w["Hq"] // w["Hkv"]
    step_flops = ff + 2.5 * g * ff       # one query head forward + one key/value group backward

    def step(i):
        b, h = divmod(i % (w["B"] * w["Hkv"]), w["Hkv"])
        oracle.attn_fwd(x["q"], x["k"], x["v"], w["causal"], scale, heads=[(b, h * g)])
        oracle.attn_bwd(x["q"], x["k"], x["v"], x["do"], w["causal"], scale, kv_heads=[(b, h)])

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    secs = time.perf_counter() - t0
    value = step_flops * args.steps / secs / 1e12
    desc = (f"per step: fp64 oracle forward of one query head and backward of one key/value head "
            f"(B=1 slice of {w['name']})")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(secs / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1), bf16 inputs)",
        "config": {"workload": w["name"], "B": w["B"], "Hq": w["Hq"], "Hkv": w["Hkv"], "seq_len": w["N"],
                   "head_dim": w["d"], "causal": w["causal"], "passes": "fwd+bwd"},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": host_cores(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    args = parse_args(argv)
    if args.case is not None:
        out = run_case(args)
    else:
        out = run_reference(args) if args.impl == "reference" else run_ours(args)
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
