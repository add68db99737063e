"""Helpers for GPU-vs-oracle parity: run the CUDA path through the C ABI, run the oracle
on the same seeded inputs, and compare under the stated bars.

Bars (the LoLA hot-path contract): float32 runs must reproduce the oracle's decision log
exactly and outputs within max-abs 1e-4 and rel-L2 1e-4; bfloat16 runs may take another
decision only where the relative SRE gap to the oracle's best candidate is below 1e-3
(checked by replaying the GPU's decisions in the oracle), and outputs must be within
max-abs 2e-2 and rel-L2 1e-2 of the oracle's outputs along the GPU's trajectory."""
from __future__ import annotations

import numpy as np
import torch

from oracle import inc

TOL = {"f32": dict(max_abs=1e-4, rel_l2=1e-4), "bf16": dict(max_abs=2e-2, rel_l2=1e-2)}
GAP = 1e-3


def to_dev(x, dev, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype == "bf16":
        t = t.view(torch.bfloat16)
    return t.to(dev)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def run_prefill(L, x, eta, lam, chunk, n=None, dev="cuda", read_mask=0, alloc=0, score=0):
    """Prefill through the C ABI; returns (Y float64, write_pos, layer)."""
    w = x.w
    dt = w.dtype
    n = n or x.q.shape[2]
    lay = L.Lola(w.B, w.Hh, w.d, w.D, eta, lam, chunk=chunk,
                 dtype=torch.bfloat16 if dt == "bf16" else torch.float32, device=dev, read_mask=read_mask,
                 alloc=alloc, score=score)
    Q, K, V = (to_dev(getattr(x, a)[:, :, :n], dev, dt) for a in "qkv")
    W = torch.from_numpy(x.W).to(dev)
    wpos = torch.full((w.B, w.Hh, n), -7, dtype=torch.int32, device=dev)
    Y = lay.prefill(Q, K, V, W, write_pos=wpos)
    torch.cuda.synchronize()
    return to_f64(Y), wpos.cpu().numpy(), lay


def err_stats(got, ref):
    d = got - ref
    return float(np.abs(d).max()), float(np.linalg.norm(d) / max(np.linalg.norm(ref), 1e-300))


def check_outputs(got, ref, dtype, what="Y"):
    ma, rl = err_stats(got, ref)
    tol = TOL[dtype]
    assert ma <= tol["max_abs"] and rl <= tol["rel_l2"], f"{what}: max-abs {ma:.3e}, rel-L2 {rl:.3e} vs {tol}"
    return ma, rl


def check_final_state(st, ref, dtype, eta, n, heads=None):
    """The memory a prefill (or prefill + decode) leaves in the state, against the oracle's
    (free-running in float32, replayed along the GPU's log in bf16): H and s (float32 in both
    modes), the cache positions (exported sorted) and the window ring.  float32: max-abs
    1e-4 and rel-L2 1e-4 on H and s, unscaled.  bf16 workloads are long (up to 131072
    writes), where float32 accumulation alone moves an entry of s ~ 2000 by more than 1e-4,
    so their bar is relative: rel-L2 1e-4 and max-abs 1e-4 of the largest entry."""
    nref = ref["H"].reshape(-1, *ref["H"].shape[-2:]).shape[0]     # heads the oracle ran, in `heads` order
    heads = np.arange(nref) if heads is None else np.asarray(heads)
    H_ref = ref["H"].reshape(nref, *ref["H"].shape[-2:])
    s_ref = ref["s"].reshape(nref, -1)
    cache_ref = ref["cache"].reshape(nref, -1)
    for what, got, want in (("H", st["H"][heads], H_ref), ("s", st["s"][heads], s_ref)):
        ma, rl = err_stats(got.astype(np.float64), want)
        bound = 1e-4 if dtype == "f32" else 1e-4 * max(1.0, float(np.abs(want).max()))
        assert ma <= bound and rl <= 1e-4, f"final {what}: max-abs {ma:.3e} (bound {bound:.3e}), rel-L2 {rl:.3e}"
    for j, i in enumerate(heads):
        live = st["c_pos"][i][st["c_pos"][i] >= 0]
        assert list(live) == sorted(live), "cache not exported sorted by position"
        assert list(live) == [p for p in cache_ref[j] if p >= 0], f"head {i}: cache differs"
        assert st["n_cache"][i] == len(live)
        assert sorted(p for p in st["win_pos"][i] if p >= 0) == list(range(max(0, n - eta), n))
    assert (st["t"][heads] == n).all() and (st["status"][heads] == 0).all()


def check_decisions(x, wpos, eta, lam, n=None, nthreads=None, read_mask=0):
    """Validates the GPU decision log against the oracle; returns the oracle run along the
    GPU's trajectory (replay) and the free-running oracle (outputs read with read_mask)."""
    dt = x.w.dtype
    n = n or wpos.shape[-1]
    q, k, v = (getattr(x, a)[..., :n, :] for a in "qkv")
    free = inc.run(q, k, v, x.W, eta, lam, dt, nthreads=nthreads, read_mask=read_mask)
    if dt == "f32":
        diff = np.argwhere(free["write_pos"] != wpos)
        assert diff.size == 0, f"float32 decision log differs at (head..., step) {diff[:5].tolist()}"
        return free, free
    rep = inc.run(q, k, v, x.W, eta, lam, dt, replay=wpos, nthreads=nthreads, read_mask=read_mask)
    assert (rep["status"] == 0).all(), f"replay rejected the GPU log: status {np.unique(rep['status'])}"
    worst = float(np.max(rep["max_gap"]))
    assert worst < GAP, f"a GPU decision is {worst:.3e} (relative SRE) away from the best candidate"
    return rep, free
