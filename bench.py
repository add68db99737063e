#!/usr/bin/env python
"""Benchmark of the LoLA hybrid-attention hot path on one GB300 (or N, one process each).

One step = one lola_prefill over the long-prefill workload: 1 sequence x 8 heads, n = 131072,
d = D = 128, eta = lambda = 512, C = 256, bf16 inputs drawn from a per-channel AR(1) process
(rho = 0.9); the inputs (805 MB) exceed the 129 MB L2, so no flush is needed between steps.
`value` is prefill tokens/s per layer (B * n / step time, summed over ranks).

Beside it, in the same line:
  * `roofline`: the prefill's contraction flops (per head-token: phi of q and k, the softmax
    branch over eta + lambda keys, the linear read, the write, the evictee's SRE and one Gram
    row) over the whole step time, against the measured bf16 tensor-core peak; `kernels`
    carries each kernel's own roofline (the chain against the FP32 CUDA-core peak derived
    from unit counts and clock, the output pass against the bf16 peak, phi(K) against HBM);
  * `prefill_more`: the same measurement on the other prefill workloads (4 x 32 heads at
    n = 4096; 32 heads at n = 16384 with planted needle keys; the float32 head at n = 1024);
  * `decode`: 64 x 32 heads whose state was prefilled from a 4096-token prefix, then all
    1024 single-token steps, timed as whole passes from the restored post-prefix state;
  * `e2e`: the same prefill through the C ABI from pinned host buffers, copies included;
  * `cpu_baseline`: the float64 C oracle on a stated sample of the workload;
  * `hola`: the write-magnitude exact cache on a gated delta-rule state (4 x 32 heads,
    n = 4096, w = 64, C = 256, bf16), one lola_hola_prefill per step, with each of its four
    kernels' rooflines and its own float64 oracle baseline.

With N processes (torchrun) the global batch is N blocks of B sequences, block r drawn with
seed + r; rank r takes the contiguous slice of heads [r B Hh, (r + 1) B Hh) -- its block -- so
per-GPU work is fixed as N grows (weak scaling) and no data crosses GPUs.

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
PREFILL = "w5_bf16_h8_n131072_ar1"
MORE_PREFILL = ("w2_bf16_b4h32_n4096", "w3_bf16_h32_n16384_needle", "w1_f32_n1024")
DECODE = "w4_bf16_decode_b64h32"
# timed steps of the other prefill workloads (a fraction of a second each)
MORE_STEPS = {"w2_bf16_b4h32_n4096": 20, "w3_bf16_h32_n16384_needle": 10, "w1_f32_n1024": 20}
# tokens of each head the CPU oracle baseline runs (the sample), per prefill workload
CPU_SAMPLE_TOKENS = 16384


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=5)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="lola", choices=["lola", "reference"])
    p.add_argument("--workload", default=PREFILL, help="prefill workload of the headline value")
    p.add_argument("--n", type=int, default=None,
                   help="override the prefill workload's sequence length (profiling captures of the same kernels "
                        "on a shorter sequence; the line then names the shortened workload)")
    p.add_argument("--decode-passes", type=int, default=2,
                   help="timed decode passes (each: every decode step of the workload from the post-prefix state)")
    p.add_argument("--no-decode", action="store_true")
    p.add_argument("--no-more", action="store_true", help="skip the other prefill workloads")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-hola", action="store_true",
                   help="skip the write-magnitude cache layer (delta-rule state) line")
    p.add_argument("--hola-only", action="store_true", help="only the write-magnitude cache layer line (profiling)")
    p.add_argument("--decode-only", action="store_true", help="skip the prefill measurement")
    p.add_argument("--decode-batch", type=int, default=None, help="batch of the decode workload (profiling)")
    p.add_argument("--decode-steps", type=int, default=None, help="decode steps per pass (profiling)")
    p.add_argument("--read-mask", type=int, default=0, choices=[0, 1, 2, 3],
                   help="read mask of the layer (1: state hidden, 2: cache hidden, 3: both)")
    p.add_argument("--sre-map", action="store_true",
                   help="also time lola_sre_map over the prefill's snapshots (reported under sre_map)")
    p.add_argument("--score", default="sre", choices=["sre", "kernel_sq", "kernel_abs", "kernel_ratio", "attention"],
                   help="cache score (sre: the self-recall error; others: the scoring ablation's query-dependent "
                        "scores, frozen at eviction; no decode line)")
    p.add_argument("--alloc", default="token", choices=["token", "chunk"],
                   help="allocation granularity of the prefill (chunk: the chunk-granular variant; "
                        "no decode line, the decode step is per token)")
    return p.parse_args(argv)


# ---------------------------------------------------------------------------------------
# ranks
# ---------------------------------------------------------------------------------------

class Ranks:
    """One process per GPU (torchrun's RANK / LOCAL_RANK / WORLD_SIZE).  The path shards by
    (batch, head) with no data-path exchange: rank r runs its own block of sequences (see
    head_slice); a barrier brackets the timed region and the time is the maximum over ranks."""

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

    def gather_heads(self, local, total_heads: int):
        """Reassembles per-rank head slices (numpy arrays whose first axis is this rank's
        heads, head_slice order) into the whole [total_heads, ...] array on every rank.
        Used off the timed path (checks), never between kernels."""
        import numpy as np
        if not self.pg:
            return local
        import torch
        import torch.distributed as dist
        lo, hi = head_slice(total_heads, self.world, self.rank)
        assert local.shape[0] == hi - lo
        per = -(-total_heads // self.world)
        dev = "cpu" if self.cpu else "cuda"
        buf = torch.zeros((per,) + local.shape[1:], dtype=torch.from_numpy(local[:0]).dtype, device=dev)
        buf[: hi - lo] = torch.from_numpy(np.ascontiguousarray(local)).to(dev)
        parts = [torch.empty_like(buf) for _ in range(self.world)]
        dist.all_gather(parts, buf)
        out = []
        for r, t in enumerate(parts):
            a, b = head_slice(total_heads, self.world, r)
            out.append(t[: b - a].cpu().numpy())
        return np.concatenate(out, axis=0)

    def close(self):
        if self.pg:
            import torch.distributed as dist
            dist.destroy_process_group()


def head_slice(total_heads: int, world: int, rank: int) -> tuple[int, int]:
    """Contiguous slice [lo, hi) of the global heads owned by `rank`: the first
    total_heads % world ranks take one head more; every head is owned exactly once."""
    base, extra = divmod(total_heads, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def rank_inputs(w, rank: int):
    """This rank's block of the global batch: B sequences drawn with seed w.seed + rank
    (global heads [rank B Hh, (rank + 1) B Hh), the head_slice of rank over world B Hh heads)."""
    import synth
    return synth.make_inputs(w, seed=w.seed + rank)


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
        # the timed region starts once nvidia-smi has written its first sample: its start-up
        # (NVML initialisation) can hold the driver for seconds and stall the launches
        t0 = time.time()
        while self.proc is not None and time.time() - t0 < 15.0:
            if os.path.getsize(self.path) > 0 or self.proc.poll() is not None:
                break
            time.sleep(0.05)
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
# a kernel on the workload named in the key, valid only for the kernel sources it was taken on:
# the digest of those files must match, otherwise the traffic is reported as null.
CSRC = os.path.join(ROOT, "sparse_exact_kv_gb300", "csrc")
NCU_TRAFFIC = {
    # long prefill (8 heads): captured on the same configuration at n = 32768 (one launch each) and
    # scaled x4 to n = 131072 -- every kernel's traffic grows in proportion to the tokens (the
    # chain streams each key's rows once, the output pass reads one pool per 128-query tile)
    ("select", "w5_bf16_h8_n131072_ar1"): {"sources": ["lola_select.cu", "lola_chain.cuh", "lola_internal.cuh"],
                                           "digest": "745c94b1a3f6faf1", "bytes_per_launch": 4 * (207.87e6 + 27.81e6)},
    ("output", "w5_bf16_h8_n131072_ar1"): {"sources": ["lola_output_tc.cu", "lola_tc.cuh", "lola_internal.cuh"],
                                           "digest": "012ab2a4689683b4", "bytes_per_launch": 4 * (372.92e6 + 56.13e6)},
    ("phi", "w5_bf16_h8_n131072_ar1"): {"sources": ["lola_phi.cu", "lola_phi_tc.cuh", "lola_tc.cuh", "lola_internal.cuh"],
                                        "digest": "e53710d10f162473", "bytes_per_launch": 4 * (67.20e6 + 140.94e6)},
    ("phi_q", "w5_bf16_h8_n131072_ar1"): {"sources": ["lola_phi.cu", "lola_phi_tc.cuh", "lola_tc.cuh", "lola_internal.cuh"],
                                          "digest": "e53710d10f162473", "bytes_per_launch": 4 * (67.19e6 + 13.51e6)},
    # 4 x 32 heads, n = 4096: the output pass, one launch
    ("output", "w2_bf16_b4h32_n4096"): {"sources": ["lola_output_tc.cu", "lola_tc.cuh", "lola_internal.cuh"],
                                        "digest": "012ab2a4689683b4", "bytes_per_launch": 810.63e6 + 121.14e6},
    # w4 decode captured at B = 32 (1024 heads, mean of 5 launches), scaled x2 to the B = 64 launch
    # (every byte is per head)
    ("decode", "w4_bf16_decode_b64h32"): {"sources": ["lola_decode.cu", "lola_chain.cuh", "lola_internal.cuh"],
                                          "digest": "3f2a4be8572b1122", "bytes_per_launch": 2 * (206.91e6 + 56.62e6)},
    # the write-magnitude cache layer, 4 x 32 heads, n = 4096: one launch of each kernel
    ("hola_prep", "hola_bf16_b4h32_n4096"): {"sources": ["lola_hola.cu", "lola_chain.cuh", "lola_internal.cuh"],
                                             "digest": "2816d23cf95ee96f", "bytes_per_launch": 268.53e6 + 744.45e6},
    ("hola_cache", "hola_bf16_b4h32_n4096"): {"sources": ["lola_hola.cu", "lola_chain.cuh", "lola_internal.cuh"],
                                              "digest": "2816d23cf95ee96f", "bytes_per_launch": 1.98e6 + 0.0},
    ("hola_state", "hola_bf16_b4h32_n4096"): {"sources": ["lola_hola_tc.cu", "lola_tc.cuh", "lola_internal.cuh"],
                                              "digest": "5cb3c1dd5116a066", "bytes_per_launch": 675.40e6 + 240.09e6},
    ("hola_read", "hola_bf16_b4h32_n4096"): {"sources": ["lola_output_tc.cu", "lola_tc.cuh", "lola_internal.cuh"],
                                             "digest": "012ab2a4689683b4", "bytes_per_launch": 671.73e6 + 118.11e6},
}


def sources_digest(files) -> str:
    h = hashlib.sha1()
    for f in files:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic(kernel: str, workload: str):
    e = NCU_TRAFFIC.get((kernel, workload))
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
# algorithmic work per head-token (steady state: every query sees eta + lambda exact keys and
# every step writes one key), as the design notes state it
# ---------------------------------------------------------------------------------------

def contraction_flops(d, D, eta, lam):
    """The prefill's contraction flops per head-token, by term: the feature map of q and k
    (2 D d: W has D/2 rows), the softmax branch over eta + lambda keys (2 (eta + lambda)
    (d_k + d_v)), the linear read H^T phi(q), phi(q)^T s (2 D d_v + 2 D), the write
    phi v^T, phi (2 D d_v + D), the evictee's H^T phi and s^T phi (2 D d_v + 2 D) and one
    Gram row phi_w . phi_i over the cache (2 lambda D).  The lambda N / z refreshes and SREs
    (about 3 lambda d_v FMAs per step) are CUDA-core work, not counted."""
    return {"phi": 2 * D * d, "soft": 2 * (eta + lam) * (d + d), "read": 2 * D * d + 2 * D,
            "write": 2 * D * d + D, "sre_new": 2 * D * d + 2 * D, "gram": 2 * lam * D}


def chunk_select_flops_per_chunk(D, dv, lam, C):
    """Chunk-granular allocation per chunk (steady state, lambda + C candidates, C written):
    every candidate's H^T phi (2 D dv) and s^T phi (2 D) and its SRE (4 dv), then the
    written keys' rank-1 terms (2 D dv + D each)."""
    P = lam + C
    return 2 * P * D * dv + 2 * P * D + 4 * P * dv + C * (2 * D * dv + D)


def decode_bytes_per_head(d, D, eta, lam, io=2):
    """Algorithmic HBM bytes of one decode step of one head: H read + write, s read + write,
    the eta + lambda exact KV read, q, k, v in and y out, and the new KV written."""
    return 2 * 4 * D * d + 2 * 4 * D + (eta + lam) * 2 * d * io + 4 * d * io + 2 * d * io


def phi_k_bytes_per_row(d, D, io):
    """Algorithmic HBM bytes of phi(K) per key row: the row read, phi(k) written once in
    float32 (the selection's precision)."""
    return d * io + 4 * D


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
    the c * P keys before it: 2 D d_v + 2 D + 4 d_v each); and lola_sre_map_relative (the
    same map minus each key's SRE at first write, appendix G)."""
    import torch
    P = max(w.chunk, 128)
    nck = (w.n + P - 1) // P
    out = torch.empty(w.B, w.Hh, nck, w.n, dtype=torch.float32, device=V.device)
    base = torch.empty(w.B, w.Hh, w.n, dtype=torch.float32, device=V.device)
    L.lola_sre_map(lay.cfg, w.n, V, ws, out, stream)
    ms = time_loop(lambda: L.lola_sre_map(lay.cfg, w.n, V, ws, out, stream), reps, stream) / reps
    L.lola_sre_map_relative(lay.cfg, w.n, V, ws, out, base, stream)
    ms_rel = time_loop(lambda: L.lola_sre_map_relative(lay.cfg, w.n, V, ws, out, base, stream), reps, stream) / reps
    keys = sum(c * P for c in range(nck))
    fl = w.B * w.Hh * keys * (2 * w.D * w.d + 2 * w.D + 4 * w.d)
    tf = fl / (ms / 1e3) / 1e12
    return {"ms": ms, "achieved_tflops": tf, "frac_of_fp32_peak": tf / pk["fp32_tflops"], "snapshots": nck,
            "relative_ms": ms_rel}


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


def fixed_score_flops_per_key(d, D, eta):
    """The scoring ablation's score pass per key: over its eta window queries, q . k (2 d) and
    phi(q) . phi(k) (2 D)."""
    return eta * (2 * d + 2 * D)


def prefill_rooflines(w, kt, ms, pk, alloc="token", score="sre"):
    """The step's roofline (contraction flops over the whole step time against the measured
    bf16 peak) and each kernel's own."""
    heads = w.B * w.Hh
    ht = heads * w.n
    io = 2 if w.dtype == "bf16" else 4
    cf = contraction_flops(w.d, w.D, w.eta, w.lam)
    per_ht = sum(cf.values())
    ach = ht * per_ht / (ms / 1e3) / 1e12
    step = {"kernel": "prefill step (all kernels)", "bound": "tensor", "achieved": ach, "peak": pk["bf16_tflops"],
            "unit": "TFLOP/s", "frac": ach / pk["bf16_tflops"], "traffic": None,
            "flop_per_head_token": per_ht, "flop_terms": cf, "head_tokens": ht, "ms": ms,
            "peak_source": f"{pk['source']} cuBLAS bf16 (burst)"}
    tr = [traffic(k, w.name) for k in ("phi", "phi_q", "select", "output")]
    if all(t is not None for t in tr):
        step["traffic"] = sum(tr)
    per = {}
    sel = kt.get("select")
    if sel and score != "sre":
        f = fixed_score_flops_per_key(w.d, w.D, w.eta)
        a_ = ht * f / (sel["avg_ms"] / 1e3) / 1e12
        per["select"] = {"bound": "alu", "achieved": a_, "peak": pk["fp32_tflops"], "unit": "TFLOP/s",
                         "frac": a_ / pk["fp32_tflops"], "flop_per_head_token": f, "avg_ms": sel["avg_ms"],
                         "traffic": None, "what": "score pass + closed-form write steps + interval sums",
                         "peak_source": "derived: SMs x 128 FP32 lanes x 2 x max SM clock"}
    elif sel and alloc == "token":
        f = cf["sre_new"] + cf["write"] + cf["gram"]
        a_ = ht * f / (sel["avg_ms"] / 1e3) / 1e12
        per["select"] = {"bound": "alu", "achieved": a_, "peak": pk["fp32_tflops"], "unit": "TFLOP/s",
                         "frac": a_ / pk["fp32_tflops"], "flop_per_head_token": f, "avg_ms": sel["avg_ms"],
                         "traffic": traffic("select", w.name),
                         "peak_source": "derived: SMs x 128 FP32 lanes x 2 x max SM clock"}
    elif sel:
        nch = heads * max(0, w.n // w.chunk - w.eta // w.chunk)
        fl = nch * chunk_select_flops_per_chunk(w.D, w.d, w.lam, w.chunk)
        a_ = fl / (sel["avg_ms"] / 1e3) / 1e12
        P = w.lam + w.chunk
        executed = nch * 2 * (3 * P * w.D * w.d + 2 * w.chunk * w.D * w.d)
        per["select"] = {"bound": "tensor", "achieved": a_, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": a_ / pk["bf16_tflops"], "avg_ms": sel["avg_ms"], "traffic": None,
                         "executed_tensor_tflops": executed / (sel["avg_ms"] / 1e3) / 1e12,
                         "peak_source": f"{pk['source']} cuBLAS bf16 (burst)"}
    out = kt.get("output")
    if out:
        f = cf["soft"] + cf["read"]
        a_ = ht * f / (out["avg_ms"] / 1e3) / 1e12
        tc = w.dtype == "bf16"
        pkv = pk["bf16_tflops"] if tc else pk["fp32_tflops"]
        per["output"] = {"bound": "tensor" if tc else "alu", "achieved": a_, "peak": pkv, "unit": "TFLOP/s",
                         "frac": a_ / pkv, "flop_per_head_token": f, "avg_ms": out["avg_ms"],
                         "traffic": traffic("output", w.name)}
    phi = kt.get("phi")
    if phi:
        byts = ht * phi_k_bytes_per_row(w.d, w.D, io)
        a_ = byts / (phi["avg_ms"] / 1e3) / 1e9
        per["phi_k"] = {"bound": "hbm", "achieved": a_, "peak": pk["hbm_gbs"], "unit": "GB/s",
                        "frac": a_ / pk["hbm_gbs"], "bytes_per_launch": byts, "avg_ms": phi["avg_ms"],
                        "traffic": traffic("phi", w.name)}
    return step, per


def e2e_prefill(L, R, lay, w, Q, K, V, Y, W, wpos, ws, stream, steps):
    """End to end through the C ABI: every step's Q, K, V copied in from pinned host memory
    and its Y copied back to pinned host memory.  The copies run on one copy stream per
    direction into a second set of device buffers, so step i + 1's inputs travel while step i
    computes (double buffering); the timed region spans from before the first copy to after
    the last read-back."""
    import torch
    dev = Q.device
    hq, hk, hv = (t.cpu().pin_memory() for t in (Q, K, V))
    hy = torch.empty(Y.shape, dtype=Y.dtype, pin_memory=True)
    bufs = [(Q, K, V, Y), tuple(torch.empty_like(t) for t in (Q, K, V, Y))]
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
    ems = R.max(pipeline(steps)) / steps
    tokens = w.B * w.n
    out = {"value": whole_job_value(R.world, tokens, ems), "unit": "tokens/s", "ms_per_step": ems,
           "h2d_bytes_per_step": 3 * Q.numel() * Q.element_size(), "d2h_bytes_per_step": Y.numel() * Y.element_size(),
           "overlap": "step i+1's inputs are copied in while step i computes and step i-1's output "
                      "is copied out (two device buffers, one copy stream per direction)"}
    del bufs
    return out


PREFILL_KERNELS = ["state_init", "phi", "phi_q", "select", "output"]


def run_prefill(L, R, args, pk, name, steps, warmup, e2e=True, sre_map=False, n=None):
    import torch
    import synth
    w = synth.WORKLOADS[name]
    if n:
        w = dataclasses.replace(w, n=n, name=f"{w.name}[n={n}]")
    x = rank_inputs(w, R.rank)
    dev = torch.device("cuda", R.local)
    Q, K, V = (dev_tensor(getattr(x, a), w.dtype, dev) for a in "qkv")
    W = torch.from_numpy(x.W).to(dev)
    lay = L.Lola(w.B, w.Hh, w.d, w.D, w.eta, w.lam, chunk=w.chunk,
                 dtype=torch.bfloat16 if w.dtype == "bf16" else torch.float32, device=dev,
                 read_mask=args.read_mask, alloc=L.LOLA_ALLOC_CHUNK if args.alloc == "chunk" else L.LOLA_ALLOC_TOKEN,
                 score=args.score)
    ws = lay.workspace_for(w.n)
    Y = torch.empty_like(V)
    wpos = torch.empty(w.B, w.Hh, w.n, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        L.lola_prefill(lay.cfg, w.n, Q, K, V, W, 0, Y, lay.state, wpos, ws, stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    with Clocks(R.local) as clk:
        R.barrier()
        ms = time_loop(step, steps, stream)
        R.barrier()
    kt = traced_kernel_times(L, R, step, steps, stream, PREFILL_KERNELS)
    ms = R.max(ms) / steps
    tokens = w.B * w.n
    in_bytes = 3 * Q.numel() * Q.element_size()
    roof, per = prefill_rooflines(w, kt, ms, pk, args.alloc, args.score)
    res = {"workload": w, "ms": ms, "value": whole_job_value(R.world, tokens, ms), "kernels": kt,
           "clocks": clk.summary(), "launches_per_step": sum(v["launches"] for v in kt.values()) / steps,
           "roofline": roof, "kernel_rooflines": per,
           "l2": (f"inputs {in_bytes / 1e6:.0f} MB > 129 MB L2, no flush" if in_bytes > 129e6 else
                  f"inputs {in_bytes / 1e6:.1f} MB fit in L2 and are not flushed (small case)")}
    if sre_map:
        res["sre_map"] = sre_map_timing(L, lay, w, V, ws, stream, pk)
    if e2e:
        res["e2e"] = e2e_prefill(L, R, lay, w, Q, K, V, Y, W, wpos, ws, stream, steps)
    res["x"] = x
    return res


def summarize_prefill(p):
    w = p["workload"]
    return {"workload": w.name, "value": p["value"], "unit": "tokens/s", "ms_per_step": p["ms"],
            "dtype": w.dtype, "config": workload_config(w), "roofline": p["roofline"],
            "kernels": {k: {**v, **p["kernel_rooflines"].get(k if k != "phi" else "phi_k", {})}
                        for k, v in p["kernels"].items()},
            "clocks": p["clocks"], **({"e2e": p["e2e"]} if p.get("e2e") else {})}


def hola_flops(d, w, chunk):
    """Per head-token: the delta-rule state path's three d_k x d_v products (the prediction
    S^T k, the rank-one write, the read-out S^T q: 6 d^2, float32 CUDA cores) and the cache
    read's two products over its visible keys (w cached plus (C + 1) / 2 chunk tokens on
    average: 2 (w + (C + 1)/2)(d_k + d_v), bf16 tensor cores)."""
    return {"state": 6 * d * d, "read": 2 * (w + (chunk + 1) / 2) * (2 * d)}


def hola_prep_bytes_per_row(d):
    """HBM bytes of the row kernel per token and head: q, k in (bf16), unit q, k out (float32),
    RMS-scaled q, k out (bf16)."""
    return 2 * (2 * d) + 2 * (4 * d) + 2 * (2 * d)


def cpu_baseline_hola(x, tokens):
    """The float64 oracle on the first `tokens` tokens of every head of one sequence, threads
    over heads (spawned workers)."""
    import multiprocessing as mp
    import numpy as np
    heads = [(0, h) for h in range(x.Hh)]
    threads = min(len(heads), os.cpu_count() or 1)
    sub = dataclasses.replace(x, n=tokens, q=np.ascontiguousarray(x.q[:, :, :tokens]),
                              k=np.ascontiguousarray(x.k[:, :, :tokens]), v=np.ascontiguousarray(x.v[:, :, :tokens]),
                              alpha=np.ascontiguousarray(x.alpha[:, :, :tokens]),
                              beta=np.ascontiguousarray(x.beta[:, :, :tokens]))
    t0 = time.time()
    with mp.get_context("spawn").Pool(threads) as pool:
        pool.starmap(_hola_oracle_head, [(sub, bh) for bh in heads])
    el = time.time() - t0
    return {"value": tokens / el, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{x.Hh} heads of one sequence, first {tokens} tokens ({tokens} token-equivalents in {el:.2f} s)"}


def _hola_oracle_head(x, bh):
    from oracle import hola_ref
    hola_ref.hola_run(x, heads=[bh])


def run_hola(L, R, args, pk, steps=10):
    """The write-magnitude cache layer (a gated delta-rule state with a persistent top-w exact
    cache, B x Hh heads, n tokens, w, C as synth.HOLA_WORKLOAD): lola_hola_prefill steps."""
    import numpy as np
    import torch
    import synth
    wl = synth.HOLA_WORKLOAD
    x = synth.hola_inputs(wl["B"], wl["Hh"], wl["n"], wl["d"], w=wl["w"], chunk=wl["chunk"], dtype=wl["dtype"],
                          seed=R.rank)
    dev = torch.device("cuda", R.local)
    b16 = lambda a: torch.from_numpy(np.ascontiguousarray(a)).view(torch.bfloat16).to(dev)  # noqa: E731
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    n, d = x.n, x.d
    cfg = L.make_hola_config(x.B, x.Hh, d, x.w, x.chunk)
    Q, K, V = b16(x.q), b16(x.k), b16(x.v)
    rest = [f32(x.alpha), f32(x.beta), f32(x.gamma_q), f32(x.gamma_k), f32(x.sink), f32(x.gate)]
    ws = torch.empty(L.lola_hola_workspace_bytes(cfg, n), dtype=torch.uint8, device=dev)
    Y = torch.empty(x.B, x.Hh, n, d, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    step = lambda: L.lola_hola_prefill(cfg, n, Q, K, V, *rest, Y, ws, stream=stream)  # noqa: E731
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    with Clocks(R.local) as clk:
        R.barrier()
        ms = time_loop(step, steps, stream) / steps
        R.barrier()
    ms = R.max(ms)
    names = ["hola_prep", "hola_state", "hola_cache", "hola_read"]
    kt = traced_kernel_times(L, R, step, steps, stream, names)
    st, _ = L.lola_hola_status(cfg, n, ws, stream=stream)
    ht = x.B * x.Hh * n
    fl = hola_flops(d, x.w, x.chunk)
    kr = {}
    if "hola_state" in kt:
        t = kt["hola_state"]["avg_ms"]
        a = fl["state"] * ht / (t * 1e-3) / 1e12
        kr["hola_state"] = {"bound": "alu", "achieved": a, "peak": pk["fp32_tflops"], "unit": "TFLOP/s",
                            "frac": a / pk["fp32_tflops"], "flop_per_head_token": fl["state"],
                            "traffic": traffic("hola_state", wl["name"]),
                            "peak_source": "derived: SMs x 128 FP32 lanes x 2 x max SM clock"}
    if "hola_read" in kt:
        t = kt["hola_read"]["avg_ms"]
        a = fl["read"] * ht / (t * 1e-3) / 1e12
        kr["hola_read"] = {"bound": "tensor", "achieved": a, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                           "frac": a / pk["bf16_tflops"], "flop_per_head_token": fl["read"],
                           "traffic": traffic("hola_read", wl["name"])}
    if "hola_prep" in kt:
        t = kt["hola_prep"]["avg_ms"]
        a = hola_prep_bytes_per_row(d) * ht / (t * 1e-3) / 1e9
        kr["hola_prep"] = {"bound": "hbm", "achieved": a, "peak": pk["hbm_gbs"], "unit": "GB/s",
                           "frac": a / pk["hbm_gbs"], "bytes_per_row": hola_prep_bytes_per_row(d),
                           "traffic": traffic("hola_prep", wl["name"])}
    per_ht = fl["state"] + fl["read"]
    step_tf = per_ht * ht / (ms * 1e-3) / 1e12
    tr = [traffic(k, wl["name"]) for k in names]
    step_traffic = sum(tr) if all(t is not None for t in tr) else None
    out = {"metric": "prefill tokens/s per layer (write-magnitude cache on a delta-rule state)",
           "value": R.world * x.B * n / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms, "steps": steps,
           "status": int(st), "dtype": "bf16",
           "config": {"workload": wl["name"], "B": x.B, "Hh": x.Hh, "n": n, "d": d, "w": x.w, "chunk": x.chunk,
                      "inputs": "gauss q, k, v; alpha in (0.9, 1], beta in [0, 1)"},
           "roofline": {"kernel": "layer step (all kernels)", "bound": "tensor", "achieved": step_tf,
                        "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": step_tf / pk["bf16_tflops"],
                        "flop_per_head_token": per_ht, "flop_terms": fl, "traffic": step_traffic},
           "kernels": {k: {**v, **kr.get(k, {})} for k, v in kt.items()}, "clocks": clk.summary()}
    if R.rank == 0 and not args.no_cpu:
        out["cpu_baseline"] = cpu_baseline_hola(x, n)
    return out


def workload_config(w):
    return {"workload": w.name, "B": w.B, "Hh": w.Hh, "n": w.n, "d": w.d, "D": w.D, "eta": w.eta, "lambda": w.lam,
            "chunk": w.chunk, "inputs": w.kind}


def run_decode(L, R, args, pk):
    """The decode workload: the state is prefilled from the prefix, saved, and every timed pass
    restores it and runs all decode steps of the workload (one lola_decode_step per token)."""
    import torch
    import synth
    w = synth.WORKLOADS[DECODE]
    if args.decode_batch:
        w = dataclasses.replace(w, B=args.decode_batch)
    if args.decode_steps:
        w = dataclasses.replace(w, decode_steps=args.decode_steps)
    x = rank_inputs(w, R.rank)
    dev = torch.device("cuda", R.local)
    lay = L.Lola(w.B, w.Hh, w.d, w.D, w.eta, w.lam, chunk=w.chunk, dtype=torch.bfloat16, device=dev,
                 read_mask=args.read_mask)
    W = torch.from_numpy(x.W).to(dev)
    P = [dev_tensor(getattr(x, a)[:, :, :w.n], w.dtype, dev) for a in "qkv"]
    lay.prefill(*P, W)
    torch.cuda.synchronize()
    del P
    lay.workspace = None
    torch.cuda.empty_cache()
    saved = lay.state.clone()
    m = w.decode_steps
    dq, dk, dv = (dev_tensor(getattr(x, a)[:, :, w.n:w.n + m].transpose(2, 0, 1, 3), w.dtype, dev) for a in "qkv")
    y = torch.empty(w.B, w.Hh, w.d, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()

    def one_pass():
        for i in range(m):
            L.lola_decode_step(lay.cfg, lay.state, W, 0, dq[i], dk[i], dv[i], y, None, stream)

    def restore():
        lay.state.copy_(saved)

    for _ in range(max(1, args.warmup // 2)):
        restore()
        one_pass()
    torch.cuda.synchronize()
    total = 0.0
    with Clocks(R.local) as clk:
        R.barrier()
        for _ in range(args.decode_passes):
            restore()
            total += time_loop(one_pass, 1, stream)
        R.barrier()
    restore()
    kt = traced_kernel_times(L, R, one_pass, 1, stream, ["phi", "decode"])
    ms = R.max(total / args.decode_passes) / m          # per decode step
    heads = w.B * w.Hh
    res = {"metric": "decode tokens/s per layer", "value": whole_job_value(R.world, w.B, ms), "unit": "tokens/s",
           "ms_per_step": ms, "steps_per_pass": m, "passes": args.decode_passes,
           "config": {"workload": w.name, "B": w.B, "Hh": w.Hh, "d": w.d, "D": w.D, "eta": w.eta, "lambda": w.lam,
                      "prefix": w.n, "state_bytes": L.lola_state_bytes(lay.cfg), "read_mask": args.read_mask,
                      "l2": f"state {L.lola_state_bytes(lay.cfg) / 1e6:.0f} MB > 129 MB L2, no flush"},
           "kernels": kt, "clocks": clk.summary(), "gpu_launches": sum(v["launches"] for v in kt.values())}
    dk_ = kt.get("decode")
    if dk_:
        byts = heads * decode_bytes_per_head(w.d, w.D, w.eta, w.lam)
        ach = byts / (dk_["avg_ms"] / 1e3) / 1e9
        res["roofline"] = {"kernel": "decode", "bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s",
                           "frac": ach / pk["hbm_gbs"], "traffic": traffic("decode", w.name),
                           "algorithmic_bytes_per_launch": byts, "avg_ms": dk_["avg_ms"],
                           "peak_source": f"{pk['source']} copy bandwidth"}
        step_ms = ms
        res["roofline_step"] = {"achieved": byts / (step_ms / 1e3) / 1e9, "unit": "GB/s",
                                "frac": byts / (step_ms / 1e3) / 1e9 / pk["hbm_gbs"],
                                "note": "algorithmic bytes over the whole step (token feature map + decode kernel)"}
    return res


# ---------------------------------------------------------------------------------------
# the CPU oracle
# ---------------------------------------------------------------------------------------

def oracle_sample(x, w, heads: int, tokens: int, read_mask: int = 0):
    """Runs the oracle on the first `tokens` tokens of the first `heads` heads of the
    workload; returns (seconds, token-equivalents, threads): a token-equivalent is one token
    of all Hh heads."""
    from oracle import inc
    BH = w.B * w.Hh
    heads = min(heads, BH)
    tokens = min(tokens, w.n)
    sl = lambda a: a.reshape(BH, *a.shape[2:])[:heads, :tokens]  # noqa: E731
    t0 = time.perf_counter()
    out = inc.run(sl(x.q), sl(x.k), sl(x.v), x.W, w.eta, w.lam, w.dtype, read_mask=read_mask)
    dt = time.perf_counter() - t0
    return dt, heads * tokens / w.Hh, out["threads"]


def cpu_baseline(x, w, read_mask: int = 0):
    """The float64 oracle on the first CPU_SAMPLE_TOKENS tokens of every head of one sequence
    (threads over heads, one per host core at most)."""
    heads = min(w.B * w.Hh, w.Hh)
    dt, tokens, threads = oracle_sample(x, w, heads, CPU_SAMPLE_TOKENS, read_mask)
    return {"value": tokens / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{heads} heads of {w.name} (one sequence), first {min(CPU_SAMPLE_TOKENS, w.n)} tokens "
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


def cpu_baseline_fixed(x, w, kind: str, heads: int = 2, tokens: int = 2048):
    """The oracle's query-dependent-score rule (one thread, float64) on the first `tokens`
    tokens of the first `heads` heads."""
    import numpy as np
    import synth
    from oracle import lola_ref as Rf
    heads = min(heads, w.B * w.Hh)
    tokens = min(tokens, w.n)
    wide = (lambda a: synth.bf16_bits_to_f32(a).astype(np.float64)) if w.dtype == "bf16" else \
        (lambda a: a.astype(np.float64))
    t0 = time.perf_counter()
    for i in range(heads):
        b, h = divmod(i, w.Hh)
        Rf.lola_run_fixed_score(wide(x.q[b, h, :tokens]), wide(x.k[b, h, :tokens]), wide(x.v[b, h, :tokens]), x.W,
                                w.eta, w.lam, kind)
    dt = time.perf_counter() - t0
    te = heads * tokens / w.Hh
    return {"value": te / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{kind} rule on {heads} of {w.B * w.Hh} heads of {w.name}, first {tokens} tokens "
                      f"({te:g} token-equivalents in {dt:.2f} s)"}


# tokens per head of each reference-arm step (a bounded sample of the workload)
REFERENCE_SAMPLE_TOKENS = 4096


def run_reference(args):
    R = Ranks()
    if R.rank != 0:
        return 0
    import synth
    w = synth.WORKLOADS[args.workload]
    x = synth.make_inputs(w, n=min(w.n, REFERENCE_SAMPLE_TOKENS), B=1)   # the sample: one sequence's heads
    heads = w.Hh
    for _ in range(args.warmup):
        oracle_sample(x, x.w, heads, REFERENCE_SAMPLE_TOKENS, args.read_mask)
    times = []
    tokens = threads = 0
    for _ in range(args.steps):
        dt, tokens, threads = oracle_sample(x, x.w, heads, REFERENCE_SAMPLE_TOKENS, args.read_mask)
        times.append(dt)
    ms = 1e3 * sum(times) / len(times)
    value = tokens / (ms / 1e3)
    sample = (f"each step: all {heads} heads of one sequence of {w.name}, first {x.w.n} of n={w.n} tokens "
              f"(token-equivalents per second)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    import torch
    import sparse_exact_kv_gb300 as L
    R = Ranks()
    R.init_gpu()
    props = torch.cuda.get_device_properties(R.local)
    pk = peaks(props.multi_processor_count)
    if args.hola_only:
        hol = run_hola(L, R, args, pk)
        if R.rank == 0:
            print(json.dumps(hol))
        R.close()
        return 0
    if args.decode_only:
        dec = run_decode(L, R, args, pk)
        if R.rank == 0:
            print(json.dumps({"metric": "decode tokens/s per layer", **{k: v for k, v in dec.items() if k != "metric"}}))
        R.close()
        return 0
    pre = run_prefill(L, R, args, pk, args.workload, args.steps, args.warmup, e2e=not args.no_e2e,
                      sre_map=args.sre_map, n=args.n)
    w = pre["workload"]
    x = pre.pop("x")
    cpu = None
    if R.rank == 0 and not args.no_cpu:
        if args.score != "sre":
            cpu = cpu_baseline_fixed(x, w, args.score)
        elif args.alloc == "token":
            cpu = cpu_baseline(x, w, args.read_mask)
        else:
            cpu = cpu_baseline_chunk(x, w)
    del x
    more = []
    if not args.no_more and args.alloc == "token" and args.score == "sre":
        for name in MORE_PREFILL:
            if name == args.workload:
                continue
            import synth
            mw = synth.WORKLOADS[name]
            k = MORE_STEPS.get(name, 5)
            p = run_prefill(L, R, args, pk, name, k, max(3, args.warmup), e2e=False)
            p.pop("x")
            more.append({**summarize_prefill(p), "steps": k})
            torch.cuda.empty_cache()
    dec = None if args.no_decode or args.alloc == "chunk" or args.score != "sre" else run_decode(L, R, args, pk)
    hol = None if args.no_hola or args.n is not None else run_hola(L, R, args, pk)
    if R.rank == 0:
        kt = pre["kernels"]
        launches = int(round(pre["launches_per_step"] * args.steps))
        line = {
            "metric": METRIC, "value": pre["value"], "unit": "tokens/s", "n_gpus": R.world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": pre["ms"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": {**workload_config(w), "l2": pre["l2"],
                       "parallelism": f"heads sharded: rank r runs batch block r (seed + r), {R.world} rank(s)",
                       "read_mask": args.read_mask, "alloc": args.alloc, "score": args.score},
            "roofline": pre["roofline"], "cpu_baseline": cpu, "e2e": pre.get("e2e"), "gpu_launches": launches,
            "clocks": pre["clocks"],
            "kernels": {k: {**v, **pre["kernel_rooflines"].get(k if k != "phi" else "phi_k", {})}
                        for k, v in kt.items()},
            **({"sre_map": pre["sre_map"]} if pre.get("sre_map") else {}),
            "peaks": {k: pk[k] for k in ("hbm_gbs", "bf16_tflops", "fp32_tflops", "source")},
            "prefill_more": more,
            "decode": dec,
            "hola": hol,
        }
        print(json.dumps(line))
    R.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
