"""Benchmark: ring all-reduce on one GB300, P=8 logical ranks, 64 MiB per rank.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload f32_64mib|bf16_64mib|weak|ag_gemm|gemm_rs|fused_f32_64mib|
                                psum_f32_64mib|reduce_scatter_bf16_64mib|reduce_scatter_bidir_bf16_64mib]
                    [--P P] [--no-secondary]

One step = one ring all-reduce (reduce-scatter + all-gather, 2(P-1) ring
steps) over the workload's synthetic inputs, which are resident in HBM when
the timed region starts.  The in-place inputs are restored by a device copy
before every step, outside the CUDA events that time the step.  The metric is
GB/s of the ring schedule's algorithmic bytes 5(P-1)*N*e per all-reduce
(roofline (a)).  The `roofline` object is taken against the bytes that must
cross HBM, 2*P*N*e (roofline (b)), since most of the schedule's traffic stays
in L2; the fraction of (a) is reported beside it.

Multi-GPU (torchrun, one process per GPU): every rank runs an independent
replica of the workload on its own GPU (the logical ranks already live in
one GPU's HBM; there is no exchange between GPUs); value = the bytes all
replicas processed / the slowest replica's time.

--impl reference times the oracle (plain C) on all host cores, one thread per
column range of every chunk (bit-identical to the single-thread run), on the
full workload; rank 0 only.
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

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from ring_collectives_gb300 import synthetic  # noqa: E402

ES = {"f32": 4, "bf16": 2}
KERNEL_SOURCES = ["ring_collectives_gb300/csrc/ring_kernels.cu", "ring_collectives_gb300/csrc/ring_pair.cu",
                  "ring_collectives_gb300/csrc/ring_common.cuh", "ring_collectives_gb300/csrc/dev.cuh",
                  "ring_collectives_gb300/csrc/internal.h", "ring_collectives_gb300/csrc/api.cu",
                  "ring_collectives_gb300/csrc/tc.cuh"]
FOLD_SOURCES = ["ring_collectives_gb300/csrc/fold_kernels.cu", "ring_collectives_gb300/csrc/dev.cuh",
                "ring_collectives_gb300/csrc/internal.h", "ring_collectives_gb300/csrc/api.cu"]
ROW_WORKLOADS = ("fused_f32_64mib", "psum_f32_64mib", "reduce_scatter_bf16_64mib",
                 "reduce_scatter_bidir_bf16_64mib", "ppermute_f32_64mib", "all_gather_f32_8mib")


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="f32_64mib",
                    choices=["f32_64mib", "bf16_64mib", "weak", "ag_gemm", "gemm_rs"] + list(ROW_WORKLOADS))
    ap.add_argument("--P", type=int, default=8)
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--sweep", action="store_true",
                    help="(kept for old command lines: the default line always carries the weak-scaling sweep)")
    ap.add_argument("--n-per-rank", type=int, default=0,
                    help="override N per rank (a smaller case of the same workload, e.g. for profiling)")
    return ap.parse_args(argv)


def parse_args_for_tests(argv):
    return parse(argv)


def workload_spec(name, P, n_override=0):
    if name == "f32_64mib":
        spec = dict(name=name, P=8, N=16 << 20, dtype="f32")
    elif name == "bf16_64mib":
        spec = dict(name=name, P=8, N=32 << 20, dtype="bf16")
    else:
        spec = dict(name=name, P=P, N=(4 << 20) * P, dtype="f32")
    if n_override:
        spec["N"] = n_override - n_override % spec["P"]
    return spec


def ring_bytes(P, N, e):
    """Roofline (a): per rank, P-1 reduce-scatter steps of 2 reads + 1 write of
    a chunk and P-1 all-gather steps of 1 read + 1 write: 5(P-1)*N*e in all."""
    return 5 * (P - 1) * N * e


def min_bytes(P, N, e):
    """Roofline (b): read every input once, write every output once."""
    return 2 * P * N * e


def max_over_ranks(x: float, dist, device) -> float:
    """The slowest replica's time: all-reduce MAX of one float (NCCL tensors
    on the GPU, gloo tensors on the CPU); identity with one rank."""
    if dist is None:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replicas_value(world: int, bytes_per_replica: float, ms_max: float) -> float:
    """Whole-job throughput in GB/s: every replica moves bytes_per_replica in
    at most ms_max milliseconds."""
    return world * bytes_per_replica / (ms_max * 1e-3) / 1e9


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _strip_comments(src: str) -> str:
    """C/C++ source without comments or blank space, so that documentation
    edits do not count as kernel changes."""
    import re
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


def kernel_hash(sources=None):
    h = hashlib.sha256()
    for rel in (KERNEL_SOURCES if sources is None else sources):
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(_strip_comments(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload, sources=None, prefix="ring_allreduce_"):
    """DRAM bytes per launch of the timed kernel from the committed ncu
    summary profiles/<prefix><workload>.md, if it was taken on the current
    kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", f"{prefix}{workload}.md")
    if not os.path.exists(path):
        return None
    src_hash, traffic = None, None
    with open(path, encoding="utf-8") as f:
        for ln in f:
            if ln.startswith("kernel_source_sha256_16:"):
                src_hash = ln.split(":", 1)[1].strip()
            if ln.startswith("dram_bytes_per_launch:"):
                try:
                    traffic = int(ln.split(":", 1)[1].strip())
                except ValueError:
                    traffic = None
    return traffic if src_hash == kernel_hash(sources) else None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.rows = []
        self.proc = None
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.25)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for ln in self.proc.stdout:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) == 8:
                self.rows.append(parts)

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[4 + i].lower().startswith("active")})
        pw = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows), "power_w_max": max(pw) if pw else None}


# ------------------------------------------------------------------ oracle timing
def oracle_time(spec, seconds, warmup=0, steps=None, frac=16):
    """Times the oracle all-reduce on the host (single thread) on a bounded
    sample: the workload's P with N_s = N/frac elements per rank (the first N_s
    of each slot's seeded values).  Returns (GB/s of ring bytes, sample text, runs)."""
    import numpy as np

    import oracle
    oracle.build()
    P, N, dt = spec["P"], spec["N"], spec["dtype"]
    Ns = N // frac
    Ns -= Ns % P
    x = synthetic.workload(spec["name"], P=P, N=Ns)
    xn = x.view(torch.int16).numpy().view(np.uint16) if dt == "bf16" else x.numpy()
    times = []
    for _ in range(warmup):
        oracle.ring_allreduce(xn.copy(), dt)
    t_end = time.perf_counter() + seconds
    while True:
        buf = xn.copy()
        t0 = time.perf_counter()
        oracle.ring_allreduce(buf, dt)
        times.append(time.perf_counter() - t0)
        if (steps is not None and len(times) >= steps) or (steps is None and time.perf_counter() > t_end):
            break
    t = statistics.mean(times)
    gbs = ring_bytes(P, Ns, ES[dt]) / t / 1e9
    sample = (f"P={P}, {Ns} {dt} elements per rank (N/{frac} of the workload), single thread, "
              f"{len(times)} runs, mean taken")
    return gbs, sample, times


def oracle_time_threads(spec, seconds, threads=None, warmup=0, steps=None):
    """Times the unmodified oracle on all host cores: chunk k of every slot is
    cut into T equal column ranges, and range j of all P*P chunks forms
    sub-problem j, a ring all-reduce of P slots with chunk k still at chunk
    position k.  Each element keeps its chunk, hence its fold order, so the
    result is bit-identical to the single-thread run (checked once).  The T
    sub-problems run in T threads (the oracle's C calls release the GIL); the
    timed step includes the gather into sub-problems and the scatter back.
    Returns (GB/s of ring bytes, sample text, runs, threads used)."""
    import numpy as np

    import oracle
    oracle.build()
    P, N, dt = spec["P"], spec["N"], spec["dtype"]
    T = threads or (os.cpu_count() or 1)
    c = N // P
    T = max(1, min(T, c))
    x = synthetic.workload(spec["name"], P=P, N=N)
    xn = x.view(torch.int16).numpy().view(np.uint16) if dt == "bf16" else x.numpy()
    edges = [c * j // T for j in range(T + 1)]
    subs = [np.empty((P, P * (edges[j + 1] - edges[j])), dtype=xn.dtype) for j in range(T)]
    from concurrent.futures import ThreadPoolExecutor
    pool = ThreadPoolExecutor(max_workers=T)

    def part(v, j):
        sub = subs[j].reshape(P, P, -1)
        sub[...] = v[:, :, edges[j]:edges[j + 1]]
        oracle.ring_allreduce(subs[j], dt)
        v[:, :, edges[j]:edges[j + 1]] = sub

    def one(buf):
        v = buf.reshape(P, P, c)
        list(pool.map(lambda j: part(v, j), range(T)))
        return buf

    check = one(xn.copy())
    ident = bool(np.array_equal(check, oracle.ring_allreduce(xn.copy(), dt)))
    if not ident:
        raise AssertionError("threaded oracle decomposition changed the result")
    buf = np.empty_like(xn)
    for _ in range(warmup):
        np.copyto(buf, xn)
        one(buf)
    times = []
    t_end = time.perf_counter() + seconds
    while True:
        np.copyto(buf, xn)
        t0 = time.perf_counter()
        one(buf)
        times.append(time.perf_counter() - t0)
        if (steps is not None and len(times) >= steps) or (steps is None and time.perf_counter() > t_end):
            break
    pool.shutdown()
    t = statistics.mean(times)
    gbs = ring_bytes(P, N, ES[dt]) / t / 1e9
    sample = (f"P={P}, the full {N} {dt} elements per rank, {T} threads over column ranges of every chunk "
              f"(bit-identical to the single-thread oracle), {len(times)} runs, mean taken, "
              f"host {cpu_model()}, os.cpu_count()={os.cpu_count()}")
    return gbs, sample, times, T


def cpu_model():
    arm_parts = {"0xd4f": "Arm Neoverse-V2", "0xd40": "Arm Neoverse-V1", "0xd0c": "Arm Neoverse-N1"}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
                if line.lower().startswith("cpu part"):
                    part = line.split(":", 1)[1].strip()
                    return f"{arm_parts.get(part, 'aarch64')} (CPU part {part})"
    except OSError:
        pass
    import platform
    return platform.machine()


def run_reference(args, spec, rank, world):
    if rank != 0:
        return 0
    gbs, sample, times, T = oracle_time_threads(spec, seconds=0, warmup=args.warmup, steps=args.steps)
    line = {
        "impl": "reference", "metric": metric_name(spec), "value": round(gbs, 3), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * statistics.mean(times), 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": spec["dtype"], "data": "synthetic",
        "config": config_dict(spec, args.gpus),
        "cpu_baseline": {"value": round(gbs, 3), "unit": "GB/s", "cores": T, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(gbs, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def metric_name(spec):
    return (f"ring_allreduce GB/s (ring-schedule bytes 5(P-1)*N*e / time) and % HBM roofline, "
            f"P={spec['P']}, {spec['N'] * ES[spec['dtype']] >> 20} MiB/rank, {spec['dtype']}, 1xGB300 per replica")


def config_dict(spec, ngpus):
    return {"workload": f"ring_allreduce_{spec['name']}", "P": spec["P"], "N_per_rank": spec["N"],
            "bytes_per_rank": spec["N"] * ES[spec["dtype"]], "chunk_elems": spec["N"] // spec["P"],
            "replicas": ngpus, "parallelism": f"replicas{ngpus} (P logical ranks per GPU)",
            "l2": "inputs (P*64 MiB) larger than L2; restored by a device copy before every step, outside the events"}


# ------------------------------------------------------------------ GPU timing
def time_allreduce(rc, bufs, pristine, N, steps, warmup, stream):
    for _ in range(warmup):
        bufs.copy_(pristine)
        rc.ring_allreduce(bufs, N=N, stream=stream)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        bufs.copy_(pristine)
        starts[i].record(stream)
        rc.ring_allreduce(bufs, N=N, stream=stream)
        ends[i].record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def time_reduce_scatter(rc, bufs, out, pristine, N, steps, warmup, stream, fn=None):
    fn = rc.ring_reduce_scatter if fn is None else fn
    for _ in range(warmup):
        bufs.copy_(pristine)
        fn(bufs, out, N=N, stream=stream)
    torch.cuda.synchronize()
    ts = []
    for _ in range(steps):
        bufs.copy_(pristine)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn(bufs, out, N=N, stream=stream)
        b.record(stream)
        ts.append((a, b))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ts]


def bf16_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured burst"
    except Exception:
        return 1900.0, "fallback burst"


def cublas_same_shape(A, Bt, stream, args):
    """Context for the tensor-core rows: cuBLAS (torch.matmul, bf16 in and
    out, fp32 accumulate) on one GEMM with the row's M, N and total K, timed
    like the row (CUDA events per call, mean after warm-up).  Not on the
    product path; its own accumulation order differs."""
    out = torch.empty((A.shape[0], Bt.shape[0]), dtype=torch.bfloat16, device=A.device)
    for _ in range(max(args.warmup, 3)):
        torch.matmul(A, Bt.t(), out=out)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for x, y in ev:
        x.record(stream)
        torch.matmul(A, Bt.t(), out=out)
        y.record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(x.elapsed_time(y) for x, y in ev)
    flop = 2 * A.shape[0] * Bt.shape[0] * A.shape[1]
    return {"ms": round(ms, 4), "TFLOP/s": round(flop / (ms * 1e-3) / 1e12, 1),
            "shape": f"{A.shape[0]}x{Bt.shape[0]}x{A.shape[1]}", "call": "torch.matmul (cuBLAS), bf16"}


def plain_gemm_same_kernel(rc, A, Bt, stream, args):
    """Context for the tensor-core rows: the library's own CTA-pair GEMM
    (gemm_rs with P=1, i.e. C = A.B^T with no reduction) on the same M, N and
    total K, timed like the row."""
    a1, b1 = A.reshape(1, *A.shape), Bt.reshape(1, *Bt.shape)
    out = torch.empty((1, A.shape[0], Bt.shape[0]), dtype=torch.bfloat16, device=A.device)
    for _ in range(max(args.warmup, 3)):
        rc.gemm_rs(a1, b1, out, stream=stream)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for x, y in ev:
        x.record(stream)
        rc.gemm_rs(a1, b1, out, stream=stream)
        y.record(stream)
    torch.cuda.synchronize()
    if rc.ring_status(stream) != 0:
        raise RuntimeError(rc.ring_last_error())
    ms = statistics.mean(x.elapsed_time(y) for x, y in ev)
    flop = 2 * A.shape[0] * Bt.shape[0] * A.shape[1]
    return {"ms": round(ms, 4), "TFLOP/s": round(flop / (ms * 1e-3) / 1e12, 1),
            "shape": f"{A.shape[0]}x{Bt.shape[0]}x{A.shape[1]}", "call": "gemm_rs with P=1 (k_gemm_rs2)"}


def ag_gemm_secondary(rc, dev, stream, args):
    """All-gather + GEMM at P=8, shards [1024,4096], B [4096,4096] bf16 (tensor-bound)."""
    P, M_r, K, N = 8, 1024, 4096, 4096
    a, b = synthetic.ag_gemm_inputs(P=P, M_r=M_r, K=K, N=N)
    ad, bd = a.to(dev), b.to(dev)
    ag = torch.empty((P * M_r, K), dtype=torch.bfloat16, device=dev)
    C = torch.empty((P * M_r, N), dtype=torch.bfloat16, device=dev)
    for _ in range(args.warmup):
        rc.ag_gemm(ad, ag, bd, C, 3, stream=stream)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for x, y in ev:
        x.record(stream)
        rc.ag_gemm(ad, ag, bd, C, 3, stream=stream)
        y.record(stream)
    torch.cuda.synchronize()
    if rc.ring_status(stream) != 0:
        raise RuntimeError(rc.ring_last_error())
    ms = statistics.mean(x.elapsed_time(y) for x, y in ev)
    flop = 2 * P * M_r * N * K
    peak, kind = bf16_peak()
    tf = flop / (ms * 1e-3) / 1e12
    cb = cublas_same_shape(ag, bd, stream, args)
    own = plain_gemm_same_kernel(rc, ag, bd, stream, args)
    own["frac_of_cublas_same_shape"] = round(own["TFLOP/s"] / cb["TFLOP/s"], 4)
    # the same workload with the weight stored [K][N] (x @ W): MN-major B operand
    bkn = bd.t().contiguous()
    for _ in range(args.warmup):
        rc.ag_gemm_kn(ad, ag, bkn, C, 3, stream=stream)
    torch.cuda.synchronize()
    evk = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for x, y in evk:
        x.record(stream)
        rc.ag_gemm_kn(ad, ag, bkn, C, 3, stream=stream)
        y.record(stream)
    torch.cuda.synchronize()
    if rc.ring_status(stream) != 0:
        raise RuntimeError(rc.ring_last_error())
    ms_kn = statistics.mean(x.elapsed_time(y) for x, y in evk)
    tf_kn = flop / (ms_kn * 1e-3) / 1e12
    kn = {"ms": round(ms_kn, 4), "TFLOP/s": round(tf_kn, 1), "frac_bf16_peak": round(tf_kn / peak, 4),
          "frac_of_nk_layout": round(tf_kn / tf, 4), "call": "ag_gemm_kn (B [K][N], MN-major operand)"}
    return {"ag_gemm_p8_8192x4096x4096": {
        "ms": round(ms, 4), "TFLOP/s": round(tf, 1), "frac_bf16_peak": round(tf / peak, 4),
        "peak": peak, "peak_kind": kind, "flop_per_call": flop,
        "cublas_same_shape": cb, "frac_of_cublas_same_shape": round(tf / cb["TFLOP/s"], 4),
        "plain_gemm_same_kernel": own, "weight_kn_layout": kn,
        "note": "gather of the 8 shards (64 MiB) + C = A_g.B^T, one tcgen05 launch"}}


def gemm_rs_secondary(rc, dev, stream, args):
    """Matmul + ring reduce-scatter at P=8, A [8192,512] and B [4096,512] per
    rank (bf16): the mirror of the all-gather + GEMM workload, 275 GFLOP."""
    P, M, N, K = 8, 8192, 4096, 512
    a, _ = synthetic.ag_gemm_inputs(P=P, M_r=M, K=K, N=256, seed=11)
    b, _ = synthetic.ag_gemm_inputs(P=P, M_r=N, K=K, N=256, seed=12)
    ad, bd = a.to(dev), b.to(dev)
    out = torch.empty((P, M, N // P), dtype=torch.bfloat16, device=dev)
    for _ in range(args.warmup):
        rc.gemm_rs(ad, bd, out, stream=stream)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for x, y in ev:
        x.record(stream)
        rc.gemm_rs(ad, bd, out, stream=stream)
        y.record(stream)
    torch.cuda.synchronize()
    if rc.ring_status(stream) != 0:
        raise RuntimeError(rc.ring_last_error())
    ms = statistics.mean(x.elapsed_time(y) for x, y in ev)
    flop = 2 * P * M * N * K
    peak, kind = bf16_peak()
    tf = flop / (ms * 1e-3) / 1e12
    # the same flops as one GEMM: sum_q A_q.B_q^T = [A_0 .. A_7] . [B_0 .. B_7]^T (K = P*512)
    a_cat = ad.permute(1, 0, 2).reshape(M, P * K).contiguous()
    b_cat = bd.permute(1, 0, 2).reshape(N, P * K).contiguous()
    cb = cublas_same_shape(a_cat, b_cat, stream, args)
    own = plain_gemm_same_kernel(rc, a_cat, b_cat, stream, args)
    own["frac_of_cublas_same_shape"] = round(own["TFLOP/s"] / cb["TFLOP/s"], 4)
    return {"gemm_rs_p8_8192x4096x512": {
        "ms": round(ms, 4), "TFLOP/s": round(tf, 1), "frac_bf16_peak": round(tf / peak, 4), "peak": peak,
        "peak_kind": kind, "flop_per_call": flop,
        "cublas_same_shape": cb, "frac_of_cublas_same_shape": round(tf / cb["TFLOP/s"], 4),
        "plain_gemm_same_kernel": own,
        "note": "8 partial products folded in ring order in the epilogue; output [8,8192,512] bf16"}}


def weak_sweep(rc, dev, stream, args):
    """The weak-scaling workload: chunk N/P = 4M fp32 ~ U[-1,1) (seed 3), P in
    {2,4,8,16,32}; per P the all-reduce time, the time per ring step
    T/(2(P-1)), and GB/s and the fraction of the HBM roofline against the
    minimum bytes 2*P*N*e.  The inputs are drawn on the device by a seeded
    torch generator (timing does not depend on the values; parity at these
    sizes is tested against the oracle with the host-drawn bytes)."""
    out = {}
    peak = peaks()[0]
    for P in (2, 4, 8, 16, 32):
        N = (4 << 20) * P
        g = torch.Generator(device=dev).manual_seed(3)
        pr = torch.empty((P, N), dtype=torch.float32, device=dev).uniform_(-1.0, 1.0, generator=g)
        bf = torch.empty_like(pr)
        ts = time_allreduce(rc, bf, pr, N, max(3, min(args.steps, 10)), max(3, args.warmup), stream)
        if rc.ring_status(stream) != 0:
            raise RuntimeError(rc.ring_last_error())
        ms = statistics.mean(ts)
        gb_min = min_bytes(P, N, 4) / (ms * 1e-3) / 1e9
        out[f"P{P}"] = {"ms": round(ms, 4), "us_per_step": round(1e3 * ms / (2 * (P - 1)), 2),
                        "per_rank_step_bytes": 5 * (4 << 20) * 4 // 2,
                        "GB/s_ring_bytes": round(ring_bytes(P, N, 4) / (ms * 1e-3) / 1e9, 1),
                        "GB/s_min_bytes": round(gb_min, 1), "frac": round(gb_min / peak, 4),
                        "traffic": profiled_traffic("weak") if P == 8 else None}
        del pr, bf
        torch.cuda.empty_cache()
    return out


def ring_bound(rc, dev, stream, spec, ms):
    """What bounds the ring all-reduce, measured in this run.
    (1) The L2 step rates: the library's own copy and add loops
    (ring_debug_l2_rate) over buffers that stay in L2 (16 MiB each), in the
    ring's launch shape -- the fastest an all-gather step (copy) or a
    reduce-scatter step (add) can move data that is already on chip.  The
    schedule's bytes at those rates give the L2 floor of one all-reduce.
    (2) Where the time of one traced all-reduce goes: per-step stamps of every
    block (ring_debug_set_trace), as the share of block time spent waiting for
    the left neighbour and the mean time of the first step, the other
    reduce-scatter steps and the all-gather steps."""
    nb = 16 << 20
    a = torch.randn(nb // 4, device=dev)
    b = torch.randn(nb // 4, device=dev)
    d = torch.empty(nb // 4, device=dev)
    reps = 200
    rates = {}
    for name, bb, factor in (("copy", None, 2), ("add", b, 3)):
        rc.ring_debug_l2_rate(d, a, bb, reps=5, stream=stream)
        torch.cuda.synchronize()
        best = None
        for _ in range(5):
            x = torch.cuda.Event(enable_timing=True)
            y = torch.cuda.Event(enable_timing=True)
            x.record(stream)
            rc.ring_debug_l2_rate(d, a, bb, reps=reps, stream=stream)
            y.record(stream)
            torch.cuda.synchronize()
            t = x.elapsed_time(y)
            best = t if best is None else min(best, t)
        rates[name] = factor * nb * reps / (best * 1e-3) / 1e9
    P, N, e = spec["P"], spec["N"], ES[spec["dtype"]]
    c = N // P
    rs_bytes = 3 * (P - 1) * P * c * e
    ag_bytes = 2 * (P - 1) * P * c * e
    floor_ms = (rs_bytes / rates["add"] + ag_bytes / rates["copy"]) / 1e6
    out = {"l2_copy_GB/s": round(rates["copy"], 1), "l2_add_GB/s": round(rates["add"], 1),
           "l2_floor_ms": round(floor_ms, 4), "frac_of_l2_floor": round(floor_ms / ms, 4),
           "l2_probe": ("ring_debug_l2_rate: the ring's 32-byte vector copy / f32 add loop, 8 blocks x 128 "
                        "threads per SM, 16 MiB buffers resident in L2, 200 passes per launch, best of 5"),
           "l2_floor": "3(P-1)*N*e at the add rate + 2(P-1)*N*e at the copy rate (reduce-scatter + all-gather)"}
    # (2) one traced all-reduce
    x = host_workload(spec["name"], P=P, N=N)
    if x is not None:
        pr = x.to(dev)
        nsteps = 2 * (P - 1)
        words = 3 * nsteps * 8 * 1216 * 4   # generous: 3 stamps x steps x blocks (up to 4x the co-resident count)
        tb = torch.zeros(words, dtype=torch.int64, device=dev)
        rc.ring_allreduce(pr, stream=stream)     # warm
        pr.copy_(x.to(dev))
        torch.cuda.synchronize()
        rc.ring_debug_set_trace(tb)
        try:
            rc.ring_allreduce(pr, stream=stream)
            torch.cuda.synchronize()
        finally:
            rc.ring_debug_set_trace(None)
        if rc.ring_status(stream) != 0:
            raise RuntimeError(rc.ring_last_error())
        st = tb.view(-1, nsteps, 3).cpu().numpy().astype("float64")
        st = st[(st[:, :, 2] > 0).all(axis=1)]          # blocks that ran (all stamps written)
        if len(st):
            span = st[:, -1, 2] - st[:, 0, 0]
            wait = (st[:, 1:, 1] - st[:, 1:, 0]).sum(axis=1)
            step = st[:, :, 2] - st[:, :, 0]
            out.update({
                "trace_blocks": int(len(st)),
                "wait_share": round(float((wait / span).mean()), 4),
                "first_step_us": round(float(step[:, 0].mean()) / 1e3, 2),
                "rs_step_us": round(float(step[:, 1:P - 1].mean()) / 1e3, 2),
                "ag_step_us": round(float(step[:, P - 1:].mean()) / 1e3, 2),
                "trace": ("one all-reduce with ring_debug_set_trace: per block, waits for the left neighbour "
                          "(steps >= 1) over its first-wait-to-last-step span, mean over blocks; step times are "
                          "wait start to step end, mean over blocks")})
        del pr, tb
    del a, b, d
    torch.cuda.empty_cache()
    return out


def run_ours(args, spec, rank, world, dist):
    import ring_collectives_gb300 as rc
    import __graft_entry__
    __graft_entry__.build()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    P, N, dt = spec["P"], spec["N"], spec["dtype"]
    e = ES[dt]
    x = host_workload(spec["name"], P=P, N=N)
    pristine = x.to(dev)
    bufs = torch.empty_like(pristine)

    # one untimed call checks that the library ran cleanly on this GPU
    bufs.copy_(pristine)
    rc.ring_allreduce(bufs, stream=stream)
    if rc.ring_status(stream) != 0:
        raise RuntimeError(rc.ring_last_error())

    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        times = time_allreduce(rc, bufs, pristine, N, args.steps, args.warmup, stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    if rc.ring_status(stream) != 0:
        raise RuntimeError(rc.ring_last_error())
    ms = statistics.mean(times)
    ms_max = max_over_ranks(ms, dist, dev)

    # end to end through the host entry point: pinned host in -> device -> pinned host out
    h_in = x.pin_memory()
    h_out = torch.empty_like(h_in).pin_memory()
    e2e_steps = max(3, min(args.steps, 10))
    for _ in range(2):
        rc.ring_allreduce_host(h_in, h_out, bufs, stream=stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(e2e_steps):
        rc.ring_allreduce_host(h_in, h_out, bufs, stream=stream)
    b.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(a.elapsed_time(b) / e2e_steps, dist, dev)
    if rc.ring_status(stream) != 0:
        raise RuntimeError(rc.ring_last_error())

    secondary = {}
    if not args.no_secondary:
        secondary["ring_bound"] = ring_bound(rc, dev, stream, spec, ms)
    if not args.no_secondary and spec["name"] == "f32_64mib":
        # bf16 gradient-bucket workload: the all-reduce
        del h_in, h_out
        xb = host_workload("bf16_64mib")
        pb = xb.to(dev)
        bb = torch.empty_like(pb)
        Nb = xb.shape[1]
        tb = time_allreduce(rc, bb, pb, Nb, args.steps, args.warmup, stream)
        if rc.ring_status(stream) != 0:
            raise RuntimeError(rc.ring_last_error())
        mb = statistics.mean(tb)
        secondary["bf16_64mib_allreduce"] = {
            "ms": round(mb, 4), "GB/s": round(ring_bytes(8, Nb, 2) / mb / 1e6, 1),
            "frac_a": round(ring_bytes(8, Nb, 2) / mb / 1e6 / peaks()[0], 4),
            "frac": round(min_bytes(8, Nb, 2) / mb / 1e6 / peaks()[0], 4),
            "traffic": profiled_traffic("bf16_64mib")}
        del pb, bb
        # every other HBM-bound row of the hot path, each against its own minimum bytes
        for name in ROW_WORKLOADS:
            rs = row_spec(rc, name, dev, stream)
            secondary[name] = row_summary(rs, statistics.mean(row_time(rc, rs, args.steps, args.warmup, stream)))
            del rs
            torch.cuda.empty_cache()
        secondary.update(ag_gemm_secondary(rc, dev, stream, args))
        secondary.update(gemm_rs_secondary(rc, dev, stream, args))
        secondary["weak_scaling"] = weak_sweep(rc, dev, stream, args)

    if rank != 0:
        return 0
    peak, peak_kind = peaks()
    rb = ring_bytes(P, N, e)
    achieved = rb / (ms * 1e-3) / 1e9
    achieved_b = min_bytes(P, N, e) / (ms * 1e-3) / 1e9
    value = replicas_value(world, rb, ms_max)
    cpu_gbs, cpu_sample, _, cpu_T = oracle_time_threads(spec, seconds=args.cpu_seconds)
    cpu1_gbs, cpu1_sample, _ = oracle_time(spec, seconds=args.cpu_seconds / 2, frac=1)
    line = {
        "metric": metric_name(spec), "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dt, "data": "synthetic",
        "config": config_dict(spec, world),
        "frac_roofline_a": round(achieved / peak, 4),
        "frac_roofline_b": round(achieved_b / peak, 4),
        # The roofline object uses the bytes that must cross HBM, 2*P*N*e (one
        # read and one write of every element of every slot: 2*e bytes per
        # element-slot); the ring schedule's 5(P-1)*N*e (the value above) mostly
        # stays in L2, so against it the fraction exceeds 1 (frac_roofline_a).
        "roofline": {"bound": "hbm", "achieved": round(achieved_b, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved_b / peak, 4),
                     # the committed weak-scaling capture is for P=8
                     "traffic": profiled_traffic(spec["name"]) if spec["name"] != "weak" or P == 8 else None,
                     "peak_kind": f"{peak_kind} (MEASURED_PEAKS hbm_gbs, burst copy)",
                     "algorithmic_bytes_per_launch": min_bytes(P, N, e),
                     "algorithmic_bytes": "2*P*N*e: every element of every slot read once and written once",
                     "ring_schedule_bytes_per_launch": rb, "kernel": "k_ring (one launch per all-reduce)"},
        "cpu_baseline": {"value": round(cpu_gbs, 3), "unit": "GB/s", "cores": cpu_T, "kind": "oracle",
                         "sample": cpu_sample,
                         "single_thread": {"value": round(cpu1_gbs, 3), "cores": 1, "sample": cpu1_sample}},
        "e2e": {"value": round(replicas_value(world, rb, e2e_ms), 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": P * N * e, "d2h_bytes_per_step": P * N * e,
                "api": "ring_allreduce_host (pinned host slots in and out)"},
        "gpu_launches": args.steps,
        "gpu_launches_note": "one k_ring launch per timed step; the e2e leg adds one per step as well",
        "clocks": clocks.summary(),
        "ms_min": round(min(times), 4), "ms_median": round(statistics.median(times), 4),
    }
    if secondary:
        line["secondary"] = secondary
    print(json.dumps(line), flush=True)
    return 0


def run_ag_gemm(args, rank, world, dist):
    """--workload ag_gemm: the all-gather + GEMM (P=8 shards [1024,4096], B
    [4096,4096], bf16, fp32 accumulate) as its own line, in TFLOP/s."""
    import ring_collectives_gb300 as rc
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    if dist is not None:
        dist.barrier()
    with ClockSampler(dev.index) as clocks:
        if args.workload == "gemm_rs":
            key, res = next(iter(gemm_rs_secondary(rc, dev, stream, args).items()))
        else:
            key, res = next(iter(ag_gemm_secondary(rc, dev, stream, args).items()))
    ms = max_over_ranks(res["ms"], dist, dev)
    if rank != 0:
        return 0
    flop = res["flop_per_call"]
    peak, kind = bf16_peak()
    tf = flop / (res["ms"] * 1e-3) / 1e12
    if args.workload == "gemm_rs":
        metric = "gemm_rs TFLOP/s (P=8 partial products A_q.B_q^T + ring reduce-scatter), 8192x4096x512 per rank, bf16"
        cfg = {"workload": "gemm_rs_p8_m8192_n4096_k512", "P": 8, "replicas": world,
               "l2": "operands 96 MiB + output 64 MiB"}
        kern = "k_gemm_rs2 (CTA pairs)"
    else:
        metric = "ag_gemm TFLOP/s (all-gather of P=8 row shards + C = A_g.B^T), 8192x4096x4096 bf16"
        cfg = {"workload": "ag_gemm_p8_m1024_k4096_n4096", "P": 8, "rank": 3, "replicas": world,
               "l2": "operands 96 MiB + outputs 128 MiB, larger than L2"}
        kern = "k_ag_gemm2 (CTA pairs)"
    line = {
        "metric": metric,
        "value": round(world * flop / (ms * 1e-3) / 1e12, 1), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": cfg,
        "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(tf / peak, 4), "traffic": None, "peak_kind": kind,
                     "algorithmic_flop_per_launch": flop, "kernel": kern},
        "cublas_same_shape": res["cublas_same_shape"],
        "frac_of_cublas_same_shape": res["frac_of_cublas_same_shape"],
        "plain_gemm_same_kernel": res["plain_gemm_same_kernel"],
        "gpu_launches": args.steps, "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)
    return 0


_HOST_INPUTS = {}


def host_workload(name, **kw):
    """Seeded host inputs, drawn once per process (several rows share them)."""
    key = (name, tuple(sorted(kw.items())))
    if key not in _HOST_INPUTS:
        _HOST_INPUTS[key] = synthetic.workload(name, **kw)
    return _HOST_INPUTS[key]


def row_spec(rc, name, dev, stream):
    """Device inputs, the call and the byte counts of one HBM-bound row of
    the hot path (the --workload rows; the default line times them all)."""
    restore = True
    if name in ("fused_f32_64mib", "psum_f32_64mib", "ppermute_f32_64mib"):
        x = host_workload("f32_64mib")
        e, dt = 4, "f32"
    elif name == "all_gather_f32_8mib":
        x = host_workload("f32_64mib", N=2 << 20)   # shards of 2M fp32 (8 MiB); outputs 64 MiB per rank
        e, dt = 4, "f32"
    else:
        x = host_workload("bf16_64mib")
        e, dt = 2, "bf16"
    P, N = x.shape
    pr = x.contiguous().to(dev)
    bufs = torch.empty_like(pr)
    if name.startswith("fused") or name.startswith("psum"):
        fn = rc.ring_allreduce_fused if name.startswith("fused") else rc.ring_psum
        call = lambda: fn(bufs, stream=stream)        # noqa: E731
        alg = min_bytes(P, N, e)
        row_min = alg
        alg_text = "2*P*N*e (every input read once, every output written once)"
        row_min_text = alg_text
        kern, sources = "k_fold_reg (register form, P=8)", FOLD_SOURCES
        metric = (f"{'fused ring-order' if name.startswith('fused') else 'psum'} single-pass all-reduce GB/s "
                  f"(2*P*N*e / time), P=8, 64 MiB/rank, f32, 1xGB300 per replica")
    elif name.startswith("reduce_scatter"):
        out = torch.empty((P, N // P), dtype=pr.dtype, device=dev)
        fn = rc.ring_reduce_scatter if name == "reduce_scatter_bf16_64mib" else rc.ring_reduce_scatter_bidir
        call = lambda: fn(bufs, out, stream=stream)   # noqa: E731
        row_min = (P + 1) * N * e   # read every slot once, write one chunk per rank
        row_min_text = "(P+1)*N*e: every slot read once, one reduced chunk written per rank"
        alg = 3 * (P - 1) * N * e
        sources = KERNEL_SOURCES
        if name == "reduce_scatter_bf16_64mib":
            alg_text = "3(P-1)*N*e (per rank P-1 steps of 2 chunk reads + 1 chunk write)"
            kern = "k_ring (reduce-scatter mode)"
            metric = "ring reduce_scatter GB/s (3(P-1)*N*e / time), P=8, 64 MiB/rank, bf16, 1xGB300 per replica"
        else:
            alg_text = ("3(P-1)*N*e (P-1 steps of 2 half-chunk reads + 1 write per direction; the last write "
                        "goes to the owner's output)")
            kern = "k_ring (bidirectional reduce-scatter mode)"
            metric = ("bidirectional reduce_scatter GB/s (3(P-1)*N*e / time), P=8, 64 MiB/rank, bf16, "
                      "1xGB300 per replica")
    elif name == "ppermute_f32_64mib":
        restore = False
        call = lambda: rc.ring_ppermute_right(pr, bufs, stream=stream)   # noqa: E731
        alg = row_min = 2 * P * N * e
        alg_text = "2*P*n*e (every source slot read once, every destination slot written once)"
        row_min_text = alg_text
        kern, sources = "k_ppermute", KERNEL_SOURCES
        metric = "ppermute right-shift GB/s (2*P*n*e / time), P=8, 64 MiB/rank, f32, 1xGB300 per replica"
    else:
        restore = False
        out = torch.empty((P, P * N), dtype=pr.dtype, device=dev)
        call = lambda: rc.ring_all_gather(pr, out, stream=stream)   # noqa: E731
        alg = 2 * P * N * e + 2 * (P - 1) * P * N * e
        row_min = P * N * e + P * P * N * e
        row_min_text = "P*n*e + P^2*n*e: every shard read once, every output written once"
        alg_text = "2*P*n*e (own shard) + 2(P-1)*P*n*e (P-1 ring steps of a read and a write of n)"
        kern, sources = "k_ring (all-gather mode)", KERNEL_SOURCES
        metric = "ring all_gather GB/s (2P*n*e*P / time), P=8, 8 MiB shards, f32, 1xGB300 per replica"
    return dict(name=name, P=P, N=N, e=e, dt=dt, pr=pr, bufs=bufs, call=call, restore=restore, alg=alg,
                alg_text=alg_text, row_min=row_min, row_min_text=row_min_text, kern=kern, sources=sources,
                metric=metric)


def row_time(rc, spec, steps, warmup, stream):
    """Event times (ms) of `steps` calls after `warmup`; in-place inputs are
    restored by a device copy before every call, outside the events."""
    for _ in range(warmup):
        if spec["restore"]:
            spec["bufs"].copy_(spec["pr"])
        spec["call"]()
    torch.cuda.synchronize()
    ev = []
    for _ in range(steps):
        if spec["restore"]:
            spec["bufs"].copy_(spec["pr"])
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        spec["call"]()
        b.record(stream)
        ev.append((a, b))
    torch.cuda.synchronize()
    if rc.ring_status(stream) != 0:
        raise RuntimeError(rc.ring_last_error())
    return [a.elapsed_time(b) for a, b in ev]


def row_summary(spec, ms):
    """GB/s and roofline fractions of one row against its minimum bytes and
    its schedule's bytes, with the DRAM traffic of its committed profile."""
    peak = peaks()[0]
    gbs_min = spec["row_min"] / (ms * 1e-3) / 1e9
    return {"ms": round(ms, 4), "GB/s_min_bytes": round(gbs_min, 1), "frac": round(gbs_min / peak, 4),
            "GB/s_schedule_bytes": round(spec["alg"] / (ms * 1e-3) / 1e9, 1),
            "frac_schedule_bytes": round(spec["alg"] / (ms * 1e-3) / 1e9 / peak, 4),
            "min_bytes_per_launch": spec["row_min"], "min_bytes": spec["row_min_text"],
            "traffic": profiled_traffic(spec["name"], spec["sources"], prefix=""),
            "kernel": spec["kern"]}


def run_row(args, rank, world, dist):
    """--workload <row>: one HBM-bound row of the hot path on its own line,
    timed like the headline (inputs resident, restored by a device copy
    outside the events), against the row's algorithmic bytes."""
    import ring_collectives_gb300 as rc
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    spec = row_spec(rc, args.workload, dev, stream)
    if dist is not None:
        dist.barrier()
    with ClockSampler(dev.index) as clocks:
        times = row_time(rc, spec, args.steps, args.warmup, stream)
    ms = statistics.mean(times)
    ms_max = max_over_ranks(ms, dist, dev)
    if rank != 0:
        return 0
    peak, peak_kind = peaks()
    P, N, e, alg, row_min = spec["P"], spec["N"], spec["e"], spec["alg"], spec["row_min"]
    achieved = alg / (ms * 1e-3) / 1e9
    line = {
        "metric": spec["metric"], "value": round(replicas_value(world, alg, ms_max), 2), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": spec["dt"], "data": "synthetic",
        "config": {"workload": spec["name"], "P": P, "N_per_rank": N, "bytes_per_rank": N * e, "replicas": world,
                   "l2": ("inputs larger than L2; in-place inputs restored by a device copy before every "
                          "step, outside the events")},
        "frac_schedule_bytes": round(achieved / peak, 4),
        "frac_roofline_b": round(row_min / (ms * 1e-3) / 1e9 / peak, 4),
        # roofline against the bytes that must cross HBM (the row's minimum);
        # the schedule's own byte count is reported beside it
        "roofline": {"bound": "hbm", "achieved": round(row_min / (ms * 1e-3) / 1e9, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(row_min / (ms * 1e-3) / 1e9 / peak, 4),
                     "traffic": profiled_traffic(spec["name"], spec["sources"], prefix=""),
                     "peak_kind": f"{peak_kind} (MEASURED_PEAKS hbm_gbs, burst copy)",
                     "algorithmic_bytes_per_launch": row_min, "algorithmic_bytes": spec["row_min_text"],
                     "schedule_bytes_per_launch": alg, "schedule_bytes": spec["alg_text"], "kernel": spec["kern"]},
        "gpu_launches": args.steps, "clocks": clocks.summary(),
        "ms_min": round(min(times), 4), "ms_median": round(statistics.median(times), 4),
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.workload in ("ag_gemm", "gemm_rs"):
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the GEMM oracles are sampled checks, not "
                              "timed baselines; use the default all-reduce workload"}))
            return 0
        dist = None
        if world > 1:
            import torch.distributed as dist_mod
            dist_mod.init_process_group("nccl", device_id=torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0"))))
            dist = dist_mod
        try:
            return run_ag_gemm(args, rank, world, dist)
        finally:
            if dist is not None:
                dist.destroy_process_group()
    if args.workload in ROW_WORKLOADS:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the reference arm times the oracle on the "
                              "default all-reduce workload only"}))
            return 0
        dist = None
        if world > 1:
            import torch.distributed as dist_mod
            dist_mod.init_process_group("nccl", device_id=torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0"))))
            dist = dist_mod
        try:
            return run_row(args, rank, world, dist)
        finally:
            if dist is not None:
                dist.destroy_process_group()
    spec = workload_spec(args.workload, args.P, args.n_per_rank)
    if args.impl == "reference":
        return run_reference(args, spec, rank, world)
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist_mod.init_process_group("nccl", device_id=torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0"))))
        dist = dist_mod
    try:
        return run_ours(args, spec, rank, world, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
