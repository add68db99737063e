"""GPU parity of the write-magnitude exact cache on a gated delta-rule state (through the C
ABI) against the float64 oracle ``oracle/hola_ref.py``.

Method: "A Hippocampus for Linear Attention" (arXiv 2607.02303v1), reading notes sections
3.1-3.5.  The state path and the scores run in float32 on the GPU; the cache decisions are exact
given the scores (checked by replaying the oracle's cache rule on the GPU's scores, and against
the oracle's own scores wherever the decision is not a near tie); the read runs on tcgen05 from
bf16 RMS-scaled rows, so outputs follow the bf16 bar (max-abs 2e-2; rel-L2 1e-2 of the two
branches' magnitudes)."""
import numpy as np
import pytest
import torch

import synth
from oracle import hola_ref as HR

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_exact_kv_gb300 as lib
    return lib


def _bf16_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).view(torch.bfloat16).cuda()


def _to_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def run_hola(L, x: synth.HolaInputs, n=None):
    n = x.n if n is None else n
    B, Hh, d = x.B, x.Hh, x.d
    cfg = L.make_hola_config(B, Hh, d, x.w, x.chunk)
    Q, K, V = (_bf16_dev(getattr(x, a)[:, :, :n]) for a in "qkv")
    f = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    alpha, beta = f(x.alpha[:, :, :n]), f(x.beta[:, :, :n])
    ws = torch.empty(L.lola_hola_workspace_bytes(cfg, n), dtype=torch.uint8, device="cuda")
    Y = torch.empty(B, Hh, n, d, dtype=torch.bfloat16, device="cuda")
    S = torch.empty(B, Hh, d, d, dtype=torch.float32, device="cuda")
    sc = torch.empty(B, Hh, n, dtype=torch.float32, device="cuda")
    nck = (n + x.chunk - 1) // x.chunk
    cache = torch.empty(B, Hh, nck, max(x.w, 1), dtype=torch.int32, device="cuda")
    L.lola_hola_prefill(cfg, n, Q, K, V, alpha, beta, f(x.gamma_q), f(x.gamma_k), f(x.sink), f(x.gate), Y, ws,
                        S_out=S, scores=sc, cache=cache)
    st, words = L.lola_hola_status(cfg, n, ws)
    assert st == 0 and not any(words)
    return {"Y": _to_f64(Y), "S": S.cpu().numpy().astype(np.float64), "scores": sc.cpu().numpy().astype(np.float64),
            "cache": cache.cpu().numpy()[..., :x.w]}


def _gpu_caches(res, b, h, nck, w):
    return [np.sort(c[c >= 0]) for c in res["cache"][b, h, :nck, :w]]


def check_head(x, res, b, h, n):
    """Scores, cache decisions, final state and outputs of head (b, h) against the oracle."""
    q, k, v = (x.widened(a)[b, h, :n] for a in "qkv")
    al, be = x.alpha[b, h, :n].astype(np.float64), x.beta[b, h, :n].astype(np.float64)
    ys, m, _, S = HR.delta_state_run(q, k, v, al, be)
    # the state path in float32: scores and the final state to 1e-4 relative to their scale
    gm = res["scores"][b, h, :n]
    assert np.abs(gm - m).max() <= 1e-4 * max(1.0, np.abs(m).max())
    assert np.abs(res["S"][b, h] - S).max() <= 1e-4 * max(1.0, np.abs(S).max())
    nck = (n + x.chunk - 1) // x.chunk
    gc = _gpu_caches(res, b, h, nck, x.w)
    # the cache rule is exact given the scores: the oracle's rule on the GPU's scores
    for got, want in zip(gc, HR.topw_running(gm, x.w, x.chunk)):
        np.testing.assert_array_equal(got, want)
    # against the oracle's own scores: a different decision only at a near tie
    for c, (got, want) in enumerate(zip(gc, HR.topw_running(m, x.w, x.chunk))):
        if not np.array_equal(got, want):
            diff = np.setxor1d(got, want)
            lo = min(m[want].min(), m[got].min())
            assert np.all(np.abs(m[diff] - lo) <= 1e-4 * max(1.0, lo)), f"chunk {c}: decisions differ beyond a tie"
    # outputs with the GPU's decisions (bf16 bar)
    oc = HR.cache_read(q, k, v, gc, x.chunk, x.gamma_q, x.gamma_k, float(x.sink[h]))
    want = ys + float(x.gate[h]) * oc
    got = res["Y"][b, h, :n]
    err = np.abs(got - want)
    assert err.max() <= 2e-2, err.max()
    # rel-L2 against the two branches' magnitudes: y is a sum of the state read-out and the
    # gated cache read, each carrying its own rounding (the cache read's bf16 operands), so a
    # near-cancelling sum (a single token, say) is measured against the size of its terms
    scale = np.linalg.norm(np.abs(ys) + abs(float(x.gate[h])) * np.abs(oc))
    assert np.linalg.norm(got - want) <= 1e-2 * scale


@pytest.mark.parametrize("B,Hh,n,w,chunk,seed", [
    (1, 2, 300, 16, 128, 1),     # ragged last chunk, three chunks
    (2, 2, 513, 64, 256, 2),     # the notes' w and C, ragged
    (1, 3, 700, 128, 128, 3),    # the largest cache this build holds
    (1, 1, 200, 0, 128, 4),      # no persistent cache: chunk tokens and the sink only
    (1, 2, 1, 16, 256, 5),       # a single token
    (1, 1, 400, 128, 384, 6),    # w larger than the tokens before most chunk starts
])
def test_layer_matches_oracle(L, B, Hh, n, w, chunk, seed):
    x = synth.hola_inputs(B, Hh, n, 128, w=w, chunk=chunk, dtype="bf16", seed=seed)
    res = run_hola(L, x)
    for b in range(B):
        for h in range(Hh):
            check_head(x, res, b, h, n)


def test_pure_delta_rule_reduction(L):
    """gate = 0: the output is the delta-rule state's read-out alone."""
    x = synth.hola_inputs(1, 2, 333, 128, w=16, chunk=128, dtype="bf16", seed=8)
    x.gate[:] = 0.0
    res = run_hola(L, x)
    for h in range(2):
        q, k, v = (x.widened(a)[0, h] for a in "qkv")
        ys, _, _, _ = HR.delta_state_run(q, k, v, x.alpha[0, h].astype(np.float64), x.beta[0, h].astype(np.float64))
        assert np.abs(res["Y"][0, h] - ys).max() <= 2e-2
        assert np.linalg.norm(res["Y"][0, h] - ys) <= 1e-2 * np.linalg.norm(ys)


def test_workload_sampled_heads(L):
    """The 4 x 32-head workload at n = 4096 (w = 64, C = 256): every head runs on the GPU,
    two sampled heads are checked against the oracle in full."""
    wl = synth.HOLA_WORKLOAD
    x = synth.hola_inputs(wl["B"], wl["Hh"], wl["n"], wl["d"], w=wl["w"], chunk=wl["chunk"], dtype=wl["dtype"])
    res = run_hola(L, x)
    assert np.isfinite(res["Y"]).all()
    for b, h in [(0, 0), (3, 31)]:
        check_head(x, res, b, h, wl["n"])


def test_small_decays_split_a_chunk(L):
    """Decays far below 1 inside a chunk: the state path splits the chunk into passes wherever
    the running decay would fall below 2^-100 (and takes a decay below 2^-100 as 2^-100, a
    change of the state far below float32 resolution).  Scores, final state and outputs still
    follow the oracle's exact recurrence."""
    x = synth.hola_inputs(1, 2, 300, 128, w=16, chunk=128, dtype="bf16", seed=11)
    x.alpha[0, 0, [5, 9, 20, 70, 71, 72, 200]] = [1e-20, 1e-20, 1e-20, 1e-30, 1e-30, 1e-30, 1e-35]
    x.alpha[0, 1, 64:128] = 0.25                 # 0.25^64 = 2^-128: one chunk in two passes or more
    x.alpha[0, 1, 130] = 1e-40                   # below 2^-100 (taken as 2^-100)
    res = run_hola(L, x)
    for h in range(2):
        check_head(x, res, 0, h, 300)


def test_tied_scores_keep_the_older_tokens(L):
    """Many tokens with beta = 0 write nothing and score exactly 0: the cache decisions among
    those ties (older token stays) and against the rest follow the oracle's rule exactly."""
    x = synth.hola_inputs(1, 2, 700, 128, w=32, chunk=128, dtype="bf16", seed=12)
    r = np.random.default_rng(12)
    x.beta[0, 0, r.random(700) < 0.6] = 0.0      # most of head 0's tokens tie at score 0
    x.beta[0, 1, :] = 0.0                        # head 1: every score ties, the oldest w stay
    res = run_hola(L, x)
    for h in range(2):
        check_head(x, res, 0, h, 700)
    caches = _gpu_caches(res, 0, 1, (700 + 127) // 128, 32)
    for c, got in enumerate(caches):
        np.testing.assert_array_equal(got, np.arange(min(32, c * 128)))
