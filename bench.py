#!/usr/bin/env python
"""Benchmark of the LoLA hybrid-attention hot path on one GB300 (or N, one process each).

One step = one lola_prefill over the workload the metric is quoted on: 4 sequences x 32
heads, n = 4096, d = D = 128, eta = lambda = 64, C = 64, bf16 inputs (K rows normalised to
norm sqrt(128)); inputs (402 MB) exceed the 129 MB L2.  `value` is prefill tokens/s per
layer (B * n / step time, summed over ranks).  The decode workload (64 x 32 heads, state
prefilled from a 4096-token prefix, then single-token steps) is timed in the same run and
reported under "decode".  Each rank runs its own replica (weak scaling, no collective
on the data path).

--impl reference times the CPU float64 oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "prefill & decode tokens/s per layer on 1 GB300; % of tensor/HBM roofline"
PREFILL = "w2_bf16_b4h32_n4096"
DECODE = "w4_bf16_decode_b64h32"


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="lola", choices=["lola", "reference"])
    p.add_argument("--decode-steps", type=int, default=64, help="timed decode steps")
    p.add_argument("--no-decode", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--decode-only", action="store_true", help="skip the prefill measurement")
    p.add_argument("--decode-batch", type=int, default=None, help="batch of the decode workload (profiling)")
    p.add_argument("--read-mask", type=int, default=0, choices=[0, 1, 2, 3],
                   help="read mask of the layer (1: state hidden, 2: cache hidden, 3: both)")
    p.add_argument("--sre-map", action="store_true",
                   help="also time lola_sre_map over the prefill's snapshots (reported under sre_map)")
    p.add_argument("--alloc", default="token", choices=["token", "chunk"],
                   help="allocation granularity of the prefill (chunk: the chunk-granular variant; "
                        "no decode line, the decode step is per token)")
    return p.parse_args()


# ---------------------------------------------------------------------------------------
# ranks
# ---------------------------------------------------------------------------------------

class Ranks:
    """One process per GPU (torchrun's RANK / LOCAL_RANK / WORLD_SIZE).  The path shards by
    (batch, head) with no data-path exchange, so N > 1 runs N replicas: a barrier brackets the
    timed region and the time is the maximum over ranks."""

    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = False
        self.cpu = False

    def init_gpu(self):
        import torch
        torch.cuda.set_device(self.local)
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group("nccl", device_id=torch.device("cuda", self.local))
            self.pg = True

    def init_cpu(self):
        """The same rank logic over gloo (multi-process tests without a GPU)."""
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group("gloo")
            self.pg = True
            self.cpu = True

    def barrier(self):
        if self.pg:
            import torch.distributed as dist
            dist.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        import torch.distributed as dist
        t = torch.tensor([x], dtype=torch.float64, device="cpu" if self.cpu else "cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            import torch.distributed as dist
            dist.destroy_process_group()


def whole_job_value(world: int, units_per_rank: float, ms_max: float) -> float:
    """Units per second over all ranks: every rank processed units_per_rank in at most ms_max."""
    return world * units_per_rank / (ms_max / 1e3)


# ---------------------------------------------------------------------------------------
# clocks and peaks
# ---------------------------------------------------------------------------------------

class Clocks:
    """nvidia-smi sampled every 200 ms during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            for line in open(self.path):
                f = [c.strip() for c in line.split(",")]
                if len(f) >= 9:
                    rows.append(f)
        finally:
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        reasons = set()
        for r in rows:
            for name, col in (("hw_slowdown", 5), ("hw_thermal_slowdown", 6), ("sw_thermal_slowdown", 7),
                              ("sw_power_cap", 8)):
                if r[col].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": num(rows[0][2]),
                "power_w_max": max((num(r[3]) or 0.0) for r in rows), "reasons": sorted(reasons),
                "samples": len(rows)}


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one ncu capture of
# the kernel on the workload named beside it, valid only for the kernel sources it was taken
# on: the digest of those files must match, otherwise the traffic is reported as null.
CSRC = os.path.join(ROOT, "sparse_exact_kv_gb300", "csrc")
NCU_TRAFFIC = {
    # w2 prefill (4 x 32 heads, n = 4096): mean of 3 select launches
    "select": {"sources": ["lola_select.cu", "lola_chain.cuh", "lola_internal.cuh"], "digest": "8ef752573e82a0a9",
               "bytes_per_launch": 409638656 + 132049067},
    # w4 decode captured at B = 32 (1024 heads, mean of 5 launches), scaled x2 to the B = 64 launch
    # (every byte is per head)
    "decode": {"sources": ["lola_decode.cu", "lola_chain.cuh", "lola_internal.cuh"], "digest": "850fe64c2562ac87",
               "bytes_per_launch": 2 * (206851584 + 56466483)},
}


def sources_digest(files) -> str:
    h = hashlib.sha1()
    for f in files:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic(kernel: str):
    e = NCU_TRAFFIC.get(kernel)
    if not e or sources_digest(e["sources"]) != e["digest"]:
        return None
    return e["bytes_per_launch"]


def peaks(sm_count: int):
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        src = "measured"
    else:
        p = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0}
        src = "fallback"
    mhz = float(p.get("sm_max_mhz", 2070.0))
    # float32 CUDA-core peak: SMs x 128 FP32 lanes x 2 flop (FMA) x max SM clock
    p["fp32_tflops"] = sm_count * 128 * 2 * mhz * 1e6 / 1e12
    p["source"] = src
    return p


# ---------------------------------------------------------------------------------------
# algorithmic work (per head-token), stated in the design notes
# ---------------------------------------------------------------------------------------

def select_flops_per_step(D, dv, lam):
    """Allocation chain per step (steady state): the evictee's H^T phi (2 D dv), the rank-1
    write of H (2 D dv), one Gram row phi_w . phi_i (2 lambda D), the N update of every
    candidate (2 lambda dv) and the SRE of the lambda + 1 candidates (4 (lambda + 1) dv)."""
    return 2 * D * dv + 2 * D * dv + 2 * lam * D + 2 * lam * dv + 4 * (lam + 1) * dv


def chunk_select_flops_per_chunk(D, dv, lam, C):
    """Chunk-granular allocation per chunk (steady state, lambda + C candidates, C written):
    every candidate's H^T phi (2 D dv) and s^T phi (2 D) and its SRE (4 dv), then the
    written keys' rank-1 terms (2 D dv + D each)."""
    P = lam + C
    return 2 * P * D * dv + 2 * P * D + 4 * P * dv + C * (2 * D * dv + D)


def output_flops_per_token(dk, dv, D, eta, lam):
    """Co-normalised read per query: softmax branch over eta + lambda exact keys
    (2 (eta + lambda)(dk + dv)) and the linear read H^T phi(q), phi(q)^T s (2 D dv + 2 D)."""
    return 2 * (eta + lam) * (dk + dv) + 2 * D * dv + 2 * D


def decode_bytes_per_head(d, D, eta, lam, io=2):
    """Algorithmic HBM bytes of one decode step of one head: H read + write, s read + write,
    the eta + lambda exact KV read, q, k, v in and y out, and the new KV written."""
    return 2 * 4 * D * d + 2 * 4 * D + (eta + lam) * 2 * d * io + 4 * d * io + 2 * d * io


# ---------------------------------------------------------------------------------------
# the CUDA path
# ---------------------------------------------------------------------------------------

def dev_tensor(a, dtype: str, dev):
    import numpy as np
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype == "bf16":
        t = t.view(torch.bfloat16)
    return t.to(dev)


def time_loop(fn, steps, stream):
    import torch
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def kernel_times(L, names):
    out = {}
    for k in names:
        ms, cnt = L.lola_kernel_time(k)
        if cnt:
            out[k] = {"launches": cnt, "total_ms": ms, "avg_ms": ms / cnt}
    return out


def sre_map_timing(L, lay, w, V, ws, stream, pk, reps=5):
    """lola_sre_map over the snapshots of the last prefill in ws (a diagnostic, section 4.4):
    device time per call and its FP32 rate on the algorithmic flops (every snapshot c scores
    the c * P keys before it: 2 D d_v + 2 D + 4 d_v each)."""
    import torch
    P = max(w.chunk, 128)
    nck = (w.n + P - 1) // P
    out = torch.empty(w.B, w.Hh, nck, w.n, dtype=torch.float32, device=V.device)
    L.lola_sre_map(lay.cfg, w.n, V, ws, out, stream)
    ms = time_loop(lambda: L.lola_sre_map(lay.cfg, w.n, V, ws, out, stream), reps, stream) / reps
    keys = sum(c * P for c in range(nck))
    fl = w.B * w.Hh * keys * (2 * w.D * w.d + 2 * w.D + 4 * w.d)
    tf = fl / (ms / 1e3) / 1e12
    return {"ms": ms, "achieved_tflops": tf, "frac_of_fp32_peak": tf / pk["fp32_tflops"], "snapshots": nck}


def traced_kernel_times(L, R, step, steps, stream, names):
    """Per-kernel device times over `steps` more steps with the library's launch tracing on
    (an event pair around every launch).  The timed loop runs without it, so the events do
    not sit between its launches; its launch count per step is the same."""
    L.lola_kernel_timing(True)
    R.barrier()
    time_loop(step, steps, stream)
    R.barrier()
    L.lola_kernel_timing(False)
    return kernel_times(L, names)


def run_prefill(L, R, args, pk):
    import torch
    import synth
    w = synth.WORKLOADS[PREFILL]
    x = synth.make_inputs(w)
    dev = torch.device("cuda", R.local)
    Q, K, V = (dev_tensor(getattr(x, a), w.dtype, dev) for a in "qkv")
    W = torch.from_numpy(x.W).to(dev)
    lay = L.Lola(w.B, w.Hh, w.d, w.D, w.eta, w.lam, chunk=w.chunk, dtype=torch.bfloat16, device=dev,
                 read_mask=args.read_mask, alloc=L.LOLA_ALLOC_CHUNK if args.alloc == "chunk" else L.LOLA_ALLOC_TOKEN)
    ws = lay.workspace_for(w.n)
    Y = torch.empty_like(V)
    wpos = torch.empty(w.B, w.Hh, w.n, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        L.lola_prefill(lay.cfg, w.n, Q, K, V, W, 0, Y, lay.state, wpos, ws, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    with Clocks(R.local) as clk:
        R.barrier()
        ms = time_loop(step, args.steps, stream)
        R.barrier()
    kt = traced_kernel_times(L, R, step, args.steps, stream, ["state_init", "phi", "select", "output"])
    sre = sre_map_timing(L, lay, w, V, ws, stream, pk) if args.sre_map else None
    ms = R.max(ms) / args.steps
    tokens = w.B * w.n
    res = {"workload": w, "ms": ms, "value": whole_job_value(R.world, tokens, ms), "kernels": kt, "clocks": clk.summary(),
           "launches": sum(v["launches"] for v in kt.values()), "sre_map": sre}
    heads = w.B * w.Hh
    sel = kt.get("select")
    if sel:
        if args.alloc == "chunk":   # chunk starts that score (the first eta / C only fill the window)
            fl = heads * max(0, w.n // w.chunk - w.eta // w.chunk) * chunk_select_flops_per_chunk(w.D, w.d, w.lam,
                                                                                                  w.chunk)
        else:
            fl = heads * w.n * select_flops_per_step(w.D, w.d, w.lam)
        ach = fl / (sel["avg_ms"] / 1e3) / 1e12
        if args.alloc == "chunk" and w.dtype == "bf16" and w.D == 128 and w.d == 128:
            # the candidates' products and the H update run on the tensor cores as split-bf16
            # passes (3 for the scoring, 2 for the write); the bound is the bf16 tensor peak
            nch = heads * max(0, w.n // w.chunk - w.eta // w.chunk)
            P = w.lam + w.chunk
            executed = nch * 2 * (3 * P * w.D * w.d + 2 * w.chunk * w.D * w.d)
            res["roofline"] = {"kernel": "select", "bound": "tensor", "achieved": ach, "peak": pk["bf16_tflops"],
                               "unit": "TFLOP/s", "frac": ach / pk["bf16_tflops"], "traffic": None,
                               "peak_source": "measured cuBLAS bf16 (burst)",
                               "executed_tensor_tflops": executed / (sel["avg_ms"] / 1e3) / 1e12}
        else:
            res["roofline"] = {"kernel": "select", "bound": "alu", "achieved": ach, "peak": pk["fp32_tflops"],
                               "unit": "TFLOP/s", "frac": ach / pk["fp32_tflops"],
                               "traffic": traffic("select") if args.alloc == "token" else None,
                               "peak_source": "derived: SMs x 128 FP32 lanes x 2 x max SM clock"}
    out = kt.get("output")
    if out:
        fl = heads * w.n * output_flops_per_token(w.d, w.d, w.D, w.eta, w.lam)
        ach = fl / (out["avg_ms"] / 1e3) / 1e12
        out["achieved_tflops"] = ach
        out["frac_of_bf16_peak"] = ach / pk["bf16_tflops"]
    phi = kt.get("phi")
    if phi:
        byts = heads * w.n * (w.d * 2 + w.D * 4)
        phi["achieved_gbs"] = byts / (phi["avg_ms"] / 1e3) / 1e9
    # end to end through the C ABI: every step's Q, K, V copied in from pinned host memory and
    # its Y copied back to pinned host memory.  The copies run on a copy stream into a second
    # set of device buffers, so step i + 1's inputs travel while step i computes (double
    # buffering); the timed region spans from before the first copy to after the last read-back.
    if not args.no_e2e:
        hq, hk, hv = (t.cpu().pin_memory() for t in (Q, K, V))
        hy = torch.empty(Y.shape, dtype=Y.dtype, pin_memory=True)
        bufs = [(Q, K, V, Y), tuple(torch.empty_like(t) for t in (Q, K, V, Y))]
        # inputs in and outputs out on two copy streams, so the two directions of the link
        # run at once
        cin, cout = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        copied = [torch.cuda.Event(), torch.cuda.Event()]
        done = [torch.cuda.Event(), torch.cuda.Event()]
        read = [torch.cuda.Event(), torch.cuda.Event()]

        def h2d(b):
            with torch.cuda.stream(cin):
                cin.wait_event(done[b])         # the compute that last read buffer b
                for dst, src in zip(bufs[b][:3], (hq, hk, hv)):
                    dst.copy_(src, non_blocking=True)
                copied[b].record(cin)

        def compute(b):
            stream.wait_event(copied[b])
            stream.wait_event(read[b])          # the copy-out of buffer b's previous output
            q_, k_, v_, y_ = bufs[b]
            L.lola_prefill(lay.cfg, w.n, q_, k_, v_, W, 0, y_, lay.state, wpos, ws, stream)
            done[b].record(stream)

        def d2h(b):
            with torch.cuda.stream(cout):
                cout.wait_event(done[b])
                hy.copy_(bufs[b][3], non_blocking=True)
                read[b].record(cout)

        def pipeline(nsteps):
            start = torch.cuda.Event(enable_timing=True)
            end = torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            start.record(stream)
            cin.wait_event(start)
            cout.wait_event(start)
            for b in (0, 1):
                read[b].record(cout)
                done[b].record(stream)
            h2d(0)
            for i in range(nsteps):
                b = i % 2
                if i + 1 < nsteps:
                    h2d(1 - b)
                compute(b)
                d2h(b)
            stream.wait_stream(cin)
            stream.wait_stream(cout)
            end.record(stream)
            torch.cuda.synchronize()
            return start.elapsed_time(end)

        pipeline(2)
        R.barrier()
        ems = R.max(pipeline(args.steps)) / args.steps
        res["e2e"] = {"value": whole_job_value(R.world, tokens, ems), "unit": "tokens/s", "ms_per_step": ems,
                      "h2d_bytes_per_step": 3 * Q.numel() * Q.element_size(),
                      "d2h_bytes_per_step": Y.numel() * Y.element_size(),
                      "overlap": "step i+1's inputs are copied in while step i computes and step i-1's output "
                                 "is copied out (two device buffers, one copy stream per direction)"}
    res["x"] = x
    return res


def run_decode(L, R, args, pk):
    import torch
    import synth
    w = synth.WORKLOADS[DECODE]
    if args.decode_batch:
        w = dataclasses.replace(w, B=args.decode_batch, decode_steps=args.warmup + args.decode_steps)
    x = synth.make_inputs(w)
    dev = torch.device("cuda", R.local)
    # the timed steps, then as many again with per-kernel tracing (each step advances the state)
    steps = min(args.decode_steps, (w.decode_steps - args.warmup) // 2)
    lay = L.Lola(w.B, w.Hh, w.d, w.D, w.eta, w.lam, chunk=w.chunk, dtype=torch.bfloat16, device=dev,
                 read_mask=args.read_mask)
    W = torch.from_numpy(x.W).to(dev)
    P = [dev_tensor(getattr(x, a)[:, :, :w.n], w.dtype, dev) for a in "qkv"]
    lay.prefill(*P, W)
    torch.cuda.synchronize()
    del P
    lay.workspace = None
    torch.cuda.empty_cache()
    nt = args.warmup + 2 * steps
    dq, dk, dv = (dev_tensor(getattr(x, a)[:, :, w.n:w.n + nt].transpose(2, 0, 1, 3), w.dtype, dev) for a in "qkv")
    y = torch.empty(w.B, w.Hh, w.d, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    it = [0]

    def step():
        i = it[0]
        L.lola_decode_step(lay.cfg, lay.state, W, 0, dq[i], dk[i], dv[i], y, None, stream)
        it[0] += 1

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    with Clocks(R.local) as clk:
        R.barrier()
        ms = time_loop(step, steps, stream)
        R.barrier()
    kt = traced_kernel_times(L, R, step, steps, stream, ["phi", "decode"])
    ms = R.max(ms) / steps
    heads = w.B * w.Hh
    res = {"metric": "decode tokens/s per layer", "value": whole_job_value(R.world, w.B, ms), "unit": "tokens/s",
           "ms_per_step": ms, "steps": steps,
           "config": {"workload": w.name, "B": w.B, "Hh": w.Hh, "d": w.d, "D": w.D, "eta": w.eta, "lambda": w.lam,
                      "prefix": w.n, "state_bytes": lola_state_bytes(L, lay), "read_mask": args.read_mask},
           "kernels": kt, "clocks": clk.summary(), "gpu_launches": sum(v["launches"] for v in kt.values())}
    dk_ = kt.get("decode")
    if dk_:
        byts = heads * decode_bytes_per_head(w.d, w.D, w.eta, w.lam)
        ach = byts / (dk_["avg_ms"] / 1e3) / 1e9
        res["roofline"] = {"kernel": "decode", "bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s",
                           "frac": ach / pk["hbm_gbs"], "traffic": traffic("decode"),
                           "algorithmic_bytes_per_launch": byts}
    return res


def lola_state_bytes(L, lay):
    return L.lola_state_bytes(lay.cfg)


# ---------------------------------------------------------------------------------------
# the CPU oracle
# ---------------------------------------------------------------------------------------

def oracle_sample(x, w, heads: int, read_mask: int = 0):
    """Runs the oracle on the first `heads` heads of the workload; returns (seconds, tokens, threads)."""
    from oracle import inc
    BH = w.B * w.Hh
    heads = min(heads, BH)
    sl = lambda a: a.reshape(BH, *a.shape[2:])[:heads]  # noqa: E731
    t0 = time.perf_counter()
    out = inc.run(sl(x.q), sl(x.k), sl(x.v), x.W, w.eta, w.lam, w.dtype, read_mask=read_mask)
    dt = time.perf_counter() - t0
    return dt, heads * w.n / w.Hh, out["threads"]


def cpu_baseline(x, w, read_mask: int = 0):
    """The oracle over every head of the prefill workload (about 35 core-seconds)."""
    heads = w.B * w.Hh
    dt, tokens, threads = oracle_sample(x, w, heads, read_mask)
    return {"value": tokens / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"all {heads} heads of {w.name}, full n={w.n} "
                      f"({tokens:g} token-equivalents in {dt:.2f} s)"}


def cpu_baseline_chunk(x, w, heads: int = 16):
    """The oracle's chunk-granular rule (one thread, float64) on the first `heads` heads of the
    prefill workload (about 0.4-0.6 s per head)."""
    import numpy as np
    import synth
    from oracle import lola_ref as Rf
    heads = min(heads, w.B * w.Hh)
    wide = (lambda a: synth.bf16_bits_to_f32(a).astype(np.float64)) if w.dtype == "bf16" else \
        (lambda a: a.astype(np.float64))
    t0 = time.perf_counter()
    for i in range(heads):
        b, h = divmod(i, w.Hh)
        Rf.lola_chunk_run(wide(x.q[b, h]), wide(x.k[b, h]), wide(x.v[b, h]), x.W, w.eta, w.lam, w.chunk)
    dt = time.perf_counter() - t0
    tokens = heads * w.n / w.Hh
    return {"value": tokens / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"chunk-granular rule on {heads} of {w.B * w.Hh} heads of {w.name}, full n={w.n} "
                      f"({tokens:g} token-equivalents in {dt:.2f} s)"}


def run_reference(args):
    R = Ranks()
    if R.rank != 0:
        return 0
    import synth
    w = synth.WORKLOADS[PREFILL]
    x = synth.make_inputs(w, B=1)         # one sequence's 32 heads: the sample is drawn from them
    heads = min(w.Hh, max(1, os.cpu_count() or 1))
    for _ in range(args.warmup):
        oracle_sample(x, x.w, heads, args.read_mask)
    times = []
    tokens = threads = 0
    for _ in range(args.steps):
        dt, tokens, threads = oracle_sample(x, x.w, heads, args.read_mask)
        times.append(dt)
    ms = 1e3 * sum(times) / len(times)
    value = tokens / (ms / 1e3)
    sample = f"each step: {heads} of {w.B * w.Hh} heads of {w.name}, full n={w.n}"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "Hh": w.Hh, "n": w.n, "d": w.d, "D": w.D, "eta": w.eta,
                       "lambda": w.lam, "chunk": w.chunk},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    import torch
    import sparse_exact_kv_gb300 as L
    R = Ranks()
    R.init_gpu()
    props = torch.cuda.get_device_properties(R.local)
    pk = peaks(props.multi_processor_count)
    if args.decode_only:
        dec = run_decode(L, R, args, pk)
        if R.rank == 0:
            print(json.dumps({"metric": "decode tokens/s per layer", **{k: v for k, v in dec.items() if k != "metric"}}))
        R.close()
        return 0
    pre = run_prefill(L, R, args, pk)
    w = pre["workload"]
    dec = None if args.no_decode or args.alloc == "chunk" else run_decode(L, R, args, pk)
    cpu = None
    if R.rank == 0 and not args.no_cpu:
        cpu = cpu_baseline(pre["x"], w, args.read_mask) if args.alloc == "token" else cpu_baseline_chunk(pre["x"], w)
    if R.rank == 0:
        launches = pre["launches"] * 1
        line = {
            "metric": METRIC, "value": pre["value"], "unit": "tokens/s", "n_gpus": R.world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": pre["ms"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "Hh": w.Hh, "n": w.n, "d": w.d, "D": w.D, "eta": w.eta,
                       "lambda": w.lam, "chunk": w.chunk, "l2": "inputs 402 MB > 129 MB L2, no flush",
                       "parallelism": f"replicas x{R.world}", "read_mask": args.read_mask, "alloc": args.alloc},
            "roofline": pre.get("roofline"), "cpu_baseline": cpu, "e2e": pre.get("e2e"), "gpu_launches": launches,
            "clocks": pre["clocks"], "kernels": pre["kernels"],
            **({"sre_map": pre["sre_map"]} if pre.get("sre_map") else {}),
            "peaks": {k: pk[k] for k in
                                                                        ("hbm_gbs", "bf16_tflops", "fp32_tflops",
                                                                         "source")},
            "decode": dec,
        }
        print(json.dumps(line))
    R.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
