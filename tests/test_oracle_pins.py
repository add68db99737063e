"""Pins of the CPU oracle to facts fixed outside it: hand-derived worked examples,
closed forms the method reduces to, library routines, invariants and brute force.

Source of every rule: "LoLA: Low-Rank Linear Attention With Sparse Caching"
(arXiv 2505.23666v3) reading notes, sections 2.2-2.7."""
import json
import math
import os

import numpy as np
import pytest

import synth
from oracle import inc
from oracle import lola_ref as R

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        g = json.load(f)
    return {k: (np.array(v, dtype=np.float64) if isinstance(v, list) and k not in ("derivation",) else v)
            for k, v in g.items()}


def _all_forms(q, k, v, W, eta, lam, read_mask=0):
    """The three oracle formulations on one head (float32 inputs for the C form)."""
    a = R.lola_run(q, k, v, W, eta, lam, read_mask=read_mask)
    b = R.lola_set(q, k, v, W, eta, lam, read_mask=read_mask)
    c = inc.run(np.asarray(q, np.float32)[None], np.asarray(k, np.float32)[None],
                np.asarray(v, np.float32)[None], np.asarray(W, np.float32), eta, lam, "f32",
                read_mask=read_mask)
    c1 = {key: (val[0] if isinstance(val, np.ndarray) and val.ndim >= 1 else val) for key, val in c.items()}
    return a, b, c1


# ---------------------------------------------------------------------------
# feature map
# ---------------------------------------------------------------------------

def test_phi_matches_library_softmax():
    from scipy.special import softmax
    x = synth.gauss_inputs(1, 1, 17, 16, 12, "f32", seed=3)
    q = x.q[0, 0].astype(np.float64)
    W = x.W.astype(np.float64)
    z = q @ W.T
    want = np.concatenate([softmax(z, axis=-1), softmax(-z, axis=-1)], axis=-1)
    got = R.phi(q, W)
    np.testing.assert_allclose(got, want, rtol=1e-14, atol=0)
    assert (got > 0).all()
    np.testing.assert_allclose(got[:, :6].sum(-1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(got[:, 6:].sum(-1), 1.0, rtol=1e-14)


def test_phi_zero_weight_is_uniform():
    got = R.phi(np.random.default_rng(0).normal(size=(5, 8)), np.zeros((4, 8)))
    np.testing.assert_array_equal(got, np.full((5, 8), 0.25))


# ---------------------------------------------------------------------------
# SRE closed forms
# ---------------------------------------------------------------------------

def test_sre_zero_for_only_written_key():
    """A state holding only (k, v) recalls v exactly: H^T phi / phi^T s = v (phi.phi)/(phi.phi)."""
    rng = np.random.default_rng(1)
    W = rng.normal(size=(8, 16)) / 8
    k, v = rng.normal(size=16), rng.normal(size=16)
    p = R.phi(k, W)
    assert R.sre_sq(np.outer(p, v), p.copy(), p, v) < 1e-28


def test_sre_opposite_values_cancel():
    """Worked example of section 2.4: two keys with the same features and values +v, -v
    written together leave H = 0, so the read-out is 0 and each SRE equals ||v||."""
    rng = np.random.default_rng(2)
    W = rng.normal(size=(8, 16)) / 8
    k, v = rng.normal(size=16), rng.normal(size=16)
    p = R.phi(k, W)
    H = np.outer(p, v) + np.outer(p, -v)
    s = 2 * p
    np.testing.assert_allclose(math.sqrt(R.sre_sq(H, s, p, v)), np.linalg.norm(v), rtol=1e-14)
    np.testing.assert_allclose(math.sqrt(R.sre_sq(H, s, p, -v)), np.linalg.norm(v), rtol=1e-14)


def test_sre_empty_memory_is_value_norm():
    v = np.array([3.0, 4.0])
    assert R.sre_sq(np.zeros((4, 2)), np.zeros(4), np.full(4, 0.25), v) == 25.0


def test_opposite_values_read_out_zero_in_a_run():
    """Both keys written (eta = lambda = 0): the linear read-out after step 1 is 0."""
    rng = np.random.default_rng(4)
    W = rng.normal(size=(4, 8)) / 8
    kk, vv = rng.normal(size=8), rng.normal(size=8)
    q = rng.normal(size=(2, 8))
    k = np.stack([kk, kk])
    v = np.stack([vv, -vv])
    for out in _all_forms(q, k, v, W, 0, 0):
        np.testing.assert_allclose(out["Y"][1], 0.0, atol=1e-12)
        assert list(out["write_pos"]) == [0, 1]


# ---------------------------------------------------------------------------
# hand-derived worked examples (tests/golden)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["uniform_phi_mean_memory.json", "tie_breaks_to_older.json"])
def test_golden_worked_examples(name):
    g = _load(name)
    eta, lam = int(g["eta"]), int(g["lambda"])
    for out in _all_forms(g["q"], g["k"], g["v"], g["W"], eta, lam):
        assert list(out["write_pos"]) == [int(x) for x in g["write_pos"]]
        assert sorted(int(x) for x in out["cache"] if x >= 0) == [int(x) for x in g["final_cache"]]
        np.testing.assert_allclose(out["Y"], g["y"], rtol=1e-13, atol=1e-13)
        if "H" in g and "H" in out:
            np.testing.assert_allclose(out["H"], g["H"], rtol=1e-13)
            np.testing.assert_allclose(out["s"], g["s"], rtol=1e-13)
    for mask, want in g.get("y_read_mask", {}).items():
        for out in _all_forms(g["q"], g["k"], g["v"], g["W"], eta, lam, read_mask=int(mask)):
            assert list(out["write_pos"]) == [int(x) for x in g["write_pos"]]
            np.testing.assert_allclose(out["Y"], want, rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------------------
# closed forms the method reduces to
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("eta,lam", [(40, 0), (25, 15), (0, 40), (64, 64)])
def test_no_write_is_causal_softmax_attention(eta, lam):
    """eta + lambda >= n: nothing is ever written, so the method is full causal softmax
    attention; checked against torch's scaled_dot_product_attention (float64, CPU)."""
    import torch
    x = synth.gauss_inputs(1, 1, 40, 16, 16, "f32", seed=5)
    q, k, v = (x.widened(n)[0, 0] for n in "qkv")
    want = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(k)[None], torch.from_numpy(v)[None],
        is_causal=True)[0].numpy()
    for out in _all_forms(q, k, v, x.W, eta, lam):
        np.testing.assert_allclose(out["Y"], want, rtol=1e-12, atol=1e-12)
        assert (out["write_pos"] == -1).all()
    np.testing.assert_allclose(R.causal_softmax_attention(q, k, v), want, rtol=1e-12, atol=1e-12)


def test_zero_budget_is_linear_attention():
    """eta = lambda = 0: every token is written at its own step, so the output is the
    inclusive linear-attention recurrence of section 2.2 (Eqs. 3-5), here written as a
    running sum of outer products independent of the oracle's code."""
    x = synth.gauss_inputs(1, 1, 33, 8, 12, "f32", seed=6, dv=5)
    q, k, v = (x.widened(n)[0, 0] for n in "qkv")
    PQ, PK = R.phi(q, x.W), R.phi(k, x.W)
    S = np.cumsum(PK[:, :, None] * v[:, None, :], axis=0)     # H_t, (n, D, dv)
    z = np.cumsum(PK, axis=0)                                  # s_t
    want = np.einsum("td,tdv->tv", PQ, S) / np.einsum("td,td->t", PQ, z)[:, None]
    for out in _all_forms(q, k, v, x.W, 0, 0):
        np.testing.assert_allclose(out["Y"], want, rtol=1e-10, atol=1e-12)
        assert list(out["write_pos"]) == list(range(33))
    np.testing.assert_allclose(R.linear_attention(q, k, v, x.W), want, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("eta", [1, 4, 9])
def test_zero_cache_is_window_plus_linear(eta):
    """lambda = 0: sliding-window softmax over the last eta tokens plus a linear state over
    every token <= t - eta, one shared denominator; each token is written when it leaves."""
    x = synth.gauss_inputs(1, 1, 30, 8, 8, "f32", seed=7)
    q, k, v = (x.widened(n)[0, 0] for n in "qkv")
    want = R.window_plus_linear(q, k, v, x.W, eta)
    for out in _all_forms(q, k, v, x.W, eta, 0):
        np.testing.assert_allclose(out["Y"], want, rtol=1e-12, atol=1e-12)
        assert list(out["write_pos"]) == [-1] * eta + list(range(30 - eta))


# ---------------------------------------------------------------------------
# invariants and brute force
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("eta,lam", [(0, 0), (0, 3), (2, 0), (3, 2), (1, 5), (4, 4), (7, 1)])
@pytest.mark.parametrize("seed", [0, 1])
def test_three_forms_agree_brute_force(eta, lam, seed):
    """n <= 32: set-based brute force, running state and the incremental C form agree."""
    x = synth.gauss_inputs(1, 1, 32, 8, 8, "f32", seed=10 + seed, dv=6)
    q, k, v = (x.widened(n)[0, 0] for n in "qkv")
    a, b, c = _all_forms(q, k, v, x.W, eta, lam)
    assert np.array_equal(a["write_pos"], b["write_pos"])
    assert np.array_equal(a["write_pos"], c["write_pos"])
    np.testing.assert_allclose(b["Y"], a["Y"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(c["Y"], a["Y"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(c["H"], a["H"], rtol=1e-11, atol=1e-12)
    assert np.array_equal(np.array(sorted(c["cache"][c["cache"] >= 0])), a["cache"])


@pytest.mark.parametrize("eta,lam", [(0, 0), (3, 2), (5, 9), (16, 16)])
def test_exactly_once_accounting(eta, lam):
    """At every t the window, cache and written set are disjoint, cover {0..t}, the
    window holds min(t+1, eta) tokens, and (H, s) are the sums over the written set."""
    x = synth.gauss_inputs(1, 1, 40, 8, 8, "f32", seed=12)
    q, k, v = (x.widened(n)[0, 0] for n in "qkv")
    PK = R.phi(k, x.W)
    for t in (0, 1, eta, eta + lam, eta + lam + 1, 25, 39):
        if t >= 40:
            continue
        o = R.lola_run(q[:t + 1], k[:t + 1], v[:t + 1], x.W, eta, lam)
        win, cache = set(o["window"].tolist()), set(o["cache"].tolist())
        written = set(np.flatnonzero(o["write_step"] >= 0).tolist())
        assert not (win & cache) and not (win & written) and not (cache & written)
        assert win | cache | written == set(range(t + 1))
        assert len(win) == min(t + 1, eta)
        assert len(cache) <= lam
        wl = sorted(written)
        np.testing.assert_allclose(o["H"], PK[wl].T @ v[wl] if wl else 0.0, atol=1e-13)
        np.testing.assert_allclose(o["s"], PK[wl].sum(0) if wl else 0.0, atol=1e-13)


def test_prefix_consistency():
    """The rule is causal: running n + m tokens repeats the decisions and outputs of the
    first n (the decode step continues a prefill exactly)."""
    x = synth.gauss_inputs(2, 2, 200, 16, 16, "bf16", seed=13)
    full = inc.run(x.q, x.k, x.v, x.W, 8, 8, "bf16")
    part = inc.run(x.q[:, :, :150], x.k[:, :, :150], x.v[:, :, :150], x.W, 8, 8, "bf16")
    assert np.array_equal(full["write_pos"][..., :150], part["write_pos"])
    np.testing.assert_array_equal(full["Y"][..., :150, :], part["Y"])


def test_value_scaling_and_shift():
    """V -> cV scales Y and every SRE by c (decisions unchanged); V -> V + b shifts Y by b
    and leaves every SRE taken against a non-empty memory unchanged (the co-normalised
    weights sum to 1).  b is small so the one empty-memory decision keeps its order."""
    x = synth.gauss_inputs(1, 1, 120, 8, 8, "f32", seed=14)
    q, k, v = (x.widened(n)[0, 0] for n in "qkv")
    base = R.lola_run(q, k, v, x.W, 4, 6)
    sc = R.lola_run(q, k, 2.5 * v, x.W, 4, 6)
    assert np.array_equal(base["write_pos"], sc["write_pos"])
    np.testing.assert_allclose(sc["Y"], 2.5 * base["Y"], rtol=1e-12, atol=1e-12)
    b = 1e-3 * np.arange(1, 9)
    sh = R.lola_run(q, k, v + b, x.W, 4, 6)
    assert np.array_equal(base["write_pos"], sh["write_pos"])
    np.testing.assert_allclose(sh["Y"], base["Y"] + b, rtol=1e-11, atol=1e-11)


def test_bf16_inputs_widen_exactly():
    x = synth.gauss_inputs(1, 3, 64, 16, 16, "bf16", seed=15)
    a = inc.run(x.q, x.k, x.v, x.W, 4, 4, "bf16")
    f = [synth.bf16_bits_to_f32(getattr(x, n)) for n in "qkv"]
    b = inc.run(*f, x.W, 4, 4, "f32")
    assert np.array_equal(a["write_pos"], b["write_pos"])
    np.testing.assert_array_equal(a["Y"], b["Y"])


def test_replay_of_own_decisions_and_rejection():
    x = synth.gauss_inputs(1, 2, 100, 8, 8, "f32", seed=16)
    o = inc.run(x.q, x.k, x.v, x.W, 5, 5, "f32")
    r = inc.run(x.q, x.k, x.v, x.W, 5, 5, "f32", replay=o["write_pos"])
    assert (r["status"] == 0).all() and (r["mismatches"] == 0).all()
    np.testing.assert_array_equal(r["Y"], o["Y"])
    bad = o["write_pos"].copy()
    t = int(np.flatnonzero(bad[0, 0] >= 0)[3])
    bad[0, 0, t] = t    # token t is in the window at step t, never a candidate (eta = 5)
    assert inc.run(x.q, x.k, x.v, x.W, 5, 5, "f32", replay=bad)["status"][0, 0] == 1
    bad = o["write_pos"].copy()
    bad[0, 1, 0] = 0    # a write before any is due
    assert inc.run(x.q, x.k, x.v, x.W, 5, 5, "f32", replay=bad)["status"][0, 1] == 2


def test_replay_reports_gap_of_a_suboptimal_choice():
    """Replaying a non-best write reports its relative SRE gap to the best candidate."""
    x = synth.gauss_inputs(1, 1, 60, 8, 8, "f32", seed=17)
    q, k, v = (x.widened(n)[0, 0] for n in "qkv")
    o = R.lola_run(q, k, v, x.W, 2, 3)
    t0 = int(np.flatnonzero(o["write_pos"] >= 0)[0])
    cand = [j for j in range(t0 + 1) if o["write_step"][j] in (-1,) or o["write_step"][j] >= t0]
    cand = [j for j in cand if j <= t0 - 2]           # the pool at step t0: cache + evictee
    alt = [j for j in cand if j != o["write_pos"][t0]][0]
    rep = o["write_pos"].copy()
    rep[t0] = alt
    rep[t0 + 1:] = -2                                 # placeholder, trajectory diverges
    r = R.lola_run(q[:t0 + 1], k[:t0 + 1], v[:t0 + 1], x.W, 2, 3, replay=rep[:t0 + 1])
    assert r["mismatches"] == 1 and r["max_gap"] > 0


def test_state_element_formula():
    """Appendix B: min{t(d_k+d_v), (eta+lambda)(d_k+d_v) + D d_v + D}."""
    assert R.state_elements(10, 64, 64, 64, 64, 64) == 10 * 128
    assert R.state_elements(4096, 128, 128, 128, 64, 64) == 128 * 256 + 128 * 128 + 128


# ---------------------------------------------------------------------------
# read mask (appendix I, Table 12: what a query reads is restricted; the cache and the
# state are updated as always)
# ---------------------------------------------------------------------------

HIDE_STATE, HIDE_CACHE = 1, 2


@pytest.mark.parametrize("eta,lam", [(1, 3), (4, 4), (9, 2), (6, 40)])
def test_window_only_read_is_sliding_window_attention(eta, lam):
    """Both memories hidden: y_t is softmax attention over the last eta tokens, whatever the
    cache and the state hold (Table 12's window-only row)."""
    x = synth.gauss_inputs(1, 1, 48, 8, 8, "f32", seed=40 + eta, dv=6)
    q, k, v = (x.widened(n)[0, 0] for n in "qkv")
    ref = R.sliding_window_attention(q, k, v, eta)
    a, b, c = _all_forms(q, k, v, x.W, eta, lam, read_mask=HIDE_STATE | HIDE_CACHE)
    for o in (a, b, c):
        np.testing.assert_allclose(o["Y"], ref, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("mask", [HIDE_STATE, HIDE_CACHE, HIDE_STATE | HIDE_CACHE])
def test_read_mask_keeps_decisions_and_memory(mask):
    """The mask changes the read only: the decision log, H, s and the cache are those of
    the unmasked run, and at least one output row differs."""
    x = synth.gauss_inputs(1, 1, 60, 8, 8, "f32", seed=44, dv=6)
    q, k, v = (x.widened(n)[0, 0] for n in "qkv")
    base = R.lola_run(q, k, v, x.W, 5, 4)
    o = R.lola_run(q, k, v, x.W, 5, 4, read_mask=mask)
    assert np.array_equal(o["write_pos"], base["write_pos"])
    assert np.array_equal(o["cache"], base["cache"])
    np.testing.assert_array_equal(o["H"], base["H"])
    np.testing.assert_array_equal(o["s"], base["s"])
    assert np.abs(o["Y"] - base["Y"]).max() > 1e-6


def test_hide_state_with_empty_cache_is_sliding_window():
    """lambda = 0: the cache is empty, so hiding the state leaves the window alone."""
    x = synth.gauss_inputs(1, 1, 40, 8, 8, "f32", seed=46, dv=6)
    q, k, v = (x.widened(n)[0, 0] for n in "qkv")
    o = R.lola_run(q, k, v, x.W, 7, 0, read_mask=HIDE_STATE)
    np.testing.assert_allclose(o["Y"], R.sliding_window_attention(q, k, v, 7), rtol=1e-11, atol=1e-12)


def test_hide_cache_with_empty_cache_changes_nothing():
    """lambda = 0: there is no cache to hide; the read is the window plus the state."""
    x = synth.gauss_inputs(1, 1, 40, 8, 8, "f32", seed=47, dv=6)
    q, k, v = (x.widened(n)[0, 0] for n in "qkv")
    o = R.lola_run(q, k, v, x.W, 5, 0, read_mask=HIDE_CACHE)
    np.testing.assert_allclose(o["Y"], R.window_plus_linear(q, k, v, x.W, 5), rtol=1e-11, atol=1e-12)


def test_hide_cache_without_writes_is_sliding_window():
    """eta + lambda >= n: nothing is ever written, so hiding the cache leaves the window."""
    x = synth.gauss_inputs(1, 1, 30, 8, 8, "f32", seed=48, dv=6)
    q, k, v = (x.widened(n)[0, 0] for n in "qkv")
    o = R.lola_run(q, k, v, x.W, 6, 30, read_mask=HIDE_CACHE)
    assert (o["write_pos"] == -1).all()
    np.testing.assert_allclose(o["Y"], R.sliding_window_attention(q, k, v, 6), rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("mask", [HIDE_STATE, HIDE_CACHE])
@pytest.mark.parametrize("eta,lam", [(1, 5), (3, 2), (4, 4)])
def test_three_forms_agree_with_read_mask(mask, eta, lam):
    x = synth.gauss_inputs(1, 1, 32, 8, 8, "f32", seed=49 + lam, dv=6)
    q, k, v = (x.widened(n)[0, 0] for n in "qkv")
    a, b, c = _all_forms(q, k, v, x.W, eta, lam, read_mask=mask)
    assert np.array_equal(a["write_pos"], b["write_pos"]) and np.array_equal(a["write_pos"], c["write_pos"])
    np.testing.assert_allclose(b["Y"], a["Y"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(c["Y"], a["Y"], rtol=1e-11, atol=1e-12)


def test_read_mask_that_leaves_nothing_is_rejected():
    """With eta = 0 the window is empty: a nonzero mask could leave no term to read."""
    x = synth.gauss_inputs(1, 1, 8, 8, 8, "f32", seed=50, dv=6)
    q, k, v = (x.widened(n)[0, 0] for n in "qkv")
    with pytest.raises(ValueError):
        R.lola_run(q, k, v, x.W, 0, 3, read_mask=HIDE_CACHE)
    with pytest.raises(ValueError):
        inc.run(np.asarray(q, np.float32)[None], np.asarray(k, np.float32)[None], np.asarray(v, np.float32)[None],
                x.W, 0, 3, "f32", read_mask=HIDE_STATE)


# ---------------------------------------------------------------------------
# chunk-granular allocation (section 2.6, Eq. 15; readings in lola_chunk_run)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("eta,lam", [(1, 0), (1, 6), (3, 2), (5, 4), (6, 60)])
def test_chunk_mode_with_unit_chunks_is_the_per_token_rule(eta, lam):
    """C = 1: every step evicts one token before its read, as the per-token rule does."""
    x = synth.gauss_inputs(1, 1, 48, 8, 8, "f32", seed=70 + eta, dv=6)
    q, k, v = (x.widened(n)[0, 0] for n in "qkv")
    a = R.lola_run(q, k, v, x.W, eta, lam)
    b = R.lola_chunk_run(q, k, v, x.W, eta, lam, 1)
    assert np.array_equal(a["write_step"], b["write_step"])
    np.testing.assert_array_equal(b["Y"], a["Y"])
    np.testing.assert_array_equal(b["H"], a["H"])
    assert np.array_equal(a["cache"], b["cache"]) and np.array_equal(np.sort(a["window"]), b["window"])


@pytest.mark.parametrize("C,mult", [(4, 1), (4, 2), (8, 1), (8, 3)])
def test_chunk_mode_zero_cache_is_window_chunks_plus_linear(C, mult):
    """lambda = 0: every token leaving the window chunks is written; the read is the window
    chunks plus the linear state over everything before them."""
    x = synth.gauss_inputs(1, 1, 50, 8, 8, "f32", seed=75 + C, dv=6)
    q, k, v = (x.widened(n)[0, 0] for n in "qkv")
    o = R.lola_chunk_run(q, k, v, x.W, mult * C, 0, C)
    np.testing.assert_allclose(o["Y"], R.window_chunks_plus_linear(q, k, v, x.W, mult * C, C), rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("C,eta", [(4, 8), (8, 8), (16, 32)])
def test_chunk_mode_without_writes_is_causal_softmax(C, eta):
    """lambda >= n: nothing is written, the cache keeps every evicted key, so the read is
    causal softmax attention."""
    x = synth.gauss_inputs(1, 1, 40, 8, 8, "f32", seed=80 + C, dv=6)
    q, k, v = (x.widened(n)[0, 0] for n in "qkv")
    o = R.lola_chunk_run(q, k, v, x.W, eta, 40, C)
    assert (o["write_step"] == -1).all()
    np.testing.assert_allclose(o["Y"], R.causal_softmax_attention(q, k, v), rtol=1e-11, atol=1e-12)


def test_chunk_mode_golden_worked_example():
    """Hand-derived in tests/golden/chunk_allocation_mean_memory.json: with W = 0 the memory
    read-out is the mean of the written values, so every SRE is worked out by hand; the first
    scored start meets the empty-memory rule and a tie at the cut (the older token is written),
    the second a key the memory recalls exactly.  Every read weight is 1, so y_t is the running
    mean (each token read exactly once)."""
    with open(os.path.join(GOLDEN, "chunk_allocation_mean_memory.json")) as f:
        g = json.load(f)
    a = lambda key: np.asarray(g[key], dtype=np.float64)  # noqa: E731
    tr = []
    o = R.lola_chunk_run(a("q"), a("k"), a("v"), a("W"), g["eta"], g["lambda"], g["C"], trace=tr)
    assert len(tr) == len(g["decisions"])
    for (c0, sq, written, kept), want in zip(tr, g["decisions"]):
        assert c0 == want["start"]
        assert {int(j): x for j, x in want["sre_sq"].items()} == pytest.approx(sq, rel=1e-15, abs=1e-15)
        assert list(written) == want["written"] and sorted(kept) == want["kept"]
    assert o["write_step"].tolist() == g["write_step"]
    assert o["cache"].tolist() == g["final_cache"] and o["window"].tolist() == g["final_window"]
    np.testing.assert_allclose(o["H"], a("H"), rtol=1e-15)
    np.testing.assert_allclose(o["s"], a("s"), rtol=1e-15)
    np.testing.assert_allclose(o["Y"], a("y"), rtol=1e-14, atol=1e-15)


@pytest.mark.parametrize("C,eta,lam", [(4, 8, 6), (8, 8, 5), (8, 16, 12)])
def test_chunk_mode_keeps_the_highest_sre_and_writes_each_key_once(C, eta, lam):
    """Every scored decision keeps exactly lambda candidates, all with larger (SRE, position)
    than every written one; at the end window, cache and written set partition the tokens
    and (H, s) are the sums over the written set."""
    x = synth.gauss_inputs(1, 1, 64, 8, 8, "f32", seed=85 + C, dv=6)
    q, k, v = (x.widened(n)[0, 0] for n in "qkv")
    tr = []
    o = R.lola_chunk_run(q, k, v, x.W, eta, lam, C, trace=tr)
    assert tr, "no decision was scored"
    for c0, sq, written, kept in tr:
        assert c0 % C == 0 and len(kept) == lam and written
        assert max((sq[j], j) for j in written) < min((sq[j], j) for j in kept)
        assert all(o["write_step"][j] == c0 for j in written)
    written = set(np.flatnonzero(o["write_step"] >= 0).tolist())
    win, cache = set(o["window"].tolist()), set(o["cache"].tolist())
    assert not (win & cache) and not (win & written) and not (cache & written)
    assert win | cache | written == set(range(64))
    PK = R.phi(k, x.W)
    wl = sorted(written)
    np.testing.assert_allclose(o["H"], PK[wl].T @ v[wl], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(o["s"], PK[wl].sum(axis=0), rtol=1e-12, atol=1e-12)


def test_chunk_mode_value_scaling_and_shift():
    """Chunk mode: V -> cV scales Y by c and keeps every decision; V -> V + b shifts Y by b and
    keeps the decisions taken against a non-empty memory (the memory's read-out and every
    co-normalised read are weighted averages of values).  b is small so that the one
    empty-memory decision keeps its order."""
    x = synth.gauss_inputs(1, 1, 96, 8, 8, "f32", seed=93, dv=6)
    q, k, v = (x.widened(n)[0, 0] for n in "qkv")
    base = R.lola_chunk_run(q, k, v, x.W, 8, 6, 4)
    sc = R.lola_chunk_run(q, k, 3.0 * v, x.W, 8, 6, 4)
    assert np.array_equal(base["write_step"], sc["write_step"])
    np.testing.assert_allclose(sc["Y"], 3.0 * base["Y"], rtol=1e-12, atol=1e-12)
    b = 1e-3 * np.arange(1, 7)
    sh = R.lola_chunk_run(q, k, v + b, x.W, 8, 6, 4)
    assert np.array_equal(base["write_step"], sh["write_step"])
    np.testing.assert_allclose(sh["Y"], base["Y"] + b, rtol=1e-11, atol=1e-11)


def test_chunk_mode_needs_whole_window_chunks():
    x = synth.gauss_inputs(1, 1, 16, 8, 8, "f32", seed=90, dv=6)
    q, k, v = (x.widened(n)[0, 0] for n in "qkv")
    for eta, C in ((6, 4), (2, 4), (0, 1)):
        with pytest.raises(ValueError):
            R.lola_chunk_run(q, k, v, x.W, eta, 4, C)


def test_chunk_mode_replay_of_own_and_of_a_swapped_log():
    """Replaying the oracle's own log reproduces it with no gap; swapping one written and one
    kept candidate of a decision is followed and reported as that pair's SRE excess."""
    x = synth.gauss_inputs(1, 1, 64, 8, 8, "f32", seed=91, dv=6)
    q, k, v = (x.widened(n)[0, 0] for n in "qkv")
    tr = []
    own = R.lola_chunk_run(q, k, v, x.W, 8, 6, 8, trace=tr)
    rep = R.lola_chunk_run(q, k, v, x.W, 8, 6, 8, replay=own["write_step"])
    assert rep["max_gap"] == 0.0
    np.testing.assert_array_equal(rep["Y"], own["Y"])
    c0, sq, written, kept = tr[-1]
    w, kp = max(written, key=lambda j: (sq[j], j)), min(kept, key=lambda j: (sq[j], j))
    log = own["write_step"].copy()
    log[w], log[kp] = -1, c0
    tr2 = []
    swapped = R.lola_chunk_run(q, k, v, x.W, 8, 6, 8, replay=log, trace=tr2)
    expect = (math.sqrt(sq[kp]) - math.sqrt(sq[w])) / math.sqrt(sq[w])
    assert swapped["max_gap"] == pytest.approx(expect, rel=1e-12)
    bad = own["write_step"].copy()
    bad[w] = -1
    with pytest.raises(ValueError):
        R.lola_chunk_run(q, k, v, x.W, 8, 6, 8, replay=bad)


# ---------------------------------------------------------------------------
# SRE diagnostics (Fig. 3)
# ---------------------------------------------------------------------------

def test_sre_map_against_the_running_memory():
    """At every chunk start the map's memory is the run's (H, s) before that step: the
    per-token run replayed up to t gives the same SREs; zero columns for keys not held."""
    x = synth.gauss_inputs(1, 1, 48, 8, 8, "f32", seed=95, dv=6)
    q, k, v = (x.widened(n)[0, 0] for n in "qkv")
    o = R.lola_run(q, k, v, x.W, 4, 3)
    times = [0, 8, 16, 24, 32, 40, 48]
    m = R.sre_map(k, v, x.W, o["write_step"], times)
    assert (m[0] == 0).all()
    PK = R.phi(k, x.W)
    for c, t in enumerate(times):
        held = (o["write_step"] >= 0) & (o["write_step"] < t)
        assert (m[c][~held] == 0).all()
        if t == 0:
            continue
        pre = R.lola_run(q[:t], k[:t], v[:t], x.W, 4, 3)   # the memory after step t - 1
        for j in np.flatnonzero(held):
            assert m[c, j] == pytest.approx(math.sqrt(R.sre_sq(pre["H"], pre["s"], PK[j], v[j])), rel=1e-12)


def test_sre_map_single_written_key_is_zero():
    """A memory holding one key recalls it exactly (section 2.3): SRE 0 at the next time."""
    x = synth.gauss_inputs(1, 1, 4, 8, 8, "f32", seed=96, dv=6)
    k, v = x.widened("k")[0, 0], x.widened("v")[0, 0]
    m = R.sre_map(k, v, x.W, np.array([2, -1, -1, -1]), [2, 3])
    assert m[0, 0] == 0.0 and m[1, 0] == pytest.approx(0.0, abs=1e-12) and (m[:, 1:] == 0).all()


def test_sre_at_first_write_is_the_rank_one_shrink_of_the_score():
    """Writing (k, v) into (H, s) adds g v to H^T phi(k) and g to phi(k)^T s (g = |phi(k)|^2),
    so its SRE right after the write is its score just before times z / (z + g) (0 into an
    empty memory).  The baseline of the relative map (appendix G, Eq. 26) is checked against
    that closed form, with the pre-write memory taken from the running oracle."""
    x = synth.gauss_inputs(1, 1, 40, 8, 8, "f32", seed=97, dv=6)
    q, k, v = (x.widened(n)[0, 0] for n in "qkv")
    o = R.lola_run(q, k, v, x.W, 4, 3)
    base = R.sre_at_first_write(k, v, x.W, o["write_step"])
    PK = R.phi(k, x.W)
    written = np.flatnonzero(o["write_step"] >= 0)
    assert written.size >= 10
    for j in written:
        w = int(o["write_step"][j])
        pre = R.lola_run(q[:w], k[:w], v[:w], x.W, 4, 3)   # the memory before step w's write
        z = float(PK[j] @ pre["s"])
        g = float(PK[j] @ PK[j])
        score = math.sqrt(R.sre_sq(pre["H"], pre["s"], PK[j], v[j]))
        assert base[j] == pytest.approx(score * z / (z + g), rel=1e-10, abs=1e-13)
    assert (base[o["write_step"] < 0] == 0).all()


def test_sre_maps_golden_worked_example():
    """Hand-derived in tests/golden/sre_maps_mean_memory.json: with W = 0 the memory read-out
    is the mean of the held values, so the SRE map (Fig. 3), the first-write baseline (two keys
    written at one chunk start share their first memory) and the relative map (Fig. 10,
    Eq. 26) are worked out by hand."""
    with open(os.path.join(GOLDEN, "sre_maps_mean_memory.json")) as f:
        g = json.load(f)
    a = lambda key: np.asarray(g[key], dtype=np.float64)  # noqa: E731
    k, v, W, ws, times = a("k"), a("v"), a("W"), g["write_step"], g["times"]
    np.testing.assert_allclose(R.sre_map(k, v, W, ws, times), a("sre_map"), rtol=1e-15, atol=1e-15)
    np.testing.assert_allclose(R.sre_at_first_write(k, v, W, ws), a("sre_at_first_write"), rtol=1e-15, atol=1e-15)
    np.testing.assert_allclose(R.sre_map_relative(k, v, W, ws, times), a("sre_map_relative"), rtol=1e-14,
                               atol=1e-15)


def test_sre_map_relative_is_zero_right_after_the_write_and_tracks_later_writes():
    """Per token: at the time right after its write the relative SRE of a key is 0; later it
    is the map's SRE minus that baseline.  Chunk mode: the keys written at one chunk start
    share their first memory, so each one's baseline includes the others."""
    x = synth.gauss_inputs(1, 1, 48, 8, 8, "f32", seed=98, dv=6)
    q, k, v = (x.widened(n)[0, 0] for n in "qkv")
    o = R.lola_run(q, k, v, x.W, 4, 3)
    ws = o["write_step"]
    times = list(range(0, 49, 4))
    rel = R.sre_map_relative(k, v, x.W, ws, times)
    m = R.sre_map(k, v, x.W, ws, times)
    base = R.sre_at_first_write(k, v, x.W, ws)
    for j in np.flatnonzero(ws >= 0):
        right_after = R.sre_map_relative(k, v, x.W, ws, [int(ws[j]) + 1])
        assert right_after[0, j] == pytest.approx(0.0, abs=1e-12)
        for c, t in enumerate(times):
            expect = m[c, j] - base[j] if ws[j] < t else 0.0
            assert rel[c, j] == pytest.approx(expect, abs=1e-12)
    co = R.lola_chunk_run(q, k, v, x.W, 8, 6, 4)
    cws = co["write_step"]
    starts = np.unique(cws[cws >= 0])
    multi = [c0 for c0 in starts if (cws == c0).sum() > 1]
    assert multi, "no chunk start wrote more than one key"
    PK = R.phi(k, x.W)
    cbase = R.sre_at_first_write(k, v, x.W, cws)
    for c0 in multi:
        held = np.flatnonzero((cws >= 0) & (cws <= c0))
        H, s = PK[held].T @ v[held], PK[held].sum(axis=0)
        for j in np.flatnonzero(cws == c0):
            assert cbase[j] == pytest.approx(math.sqrt(R.sre_sq(H, s, PK[j], v[j])), rel=1e-12)
            alone = np.array([i for i in held if cws[i] < c0] + [j])
            Ha, sa = PK[alone].T @ v[alone], PK[alone].sum(axis=0)
            assert abs(cbase[j] - math.sqrt(R.sre_sq(Ha, sa, PK[j], v[j]))) > 1e-9



# ---------------------------------------------------------------------------
# Scoring ablation (section 4.4, Table 4): query-dependent scores in place of the SRE
# ---------------------------------------------------------------------------

def _top_lambda_write_steps(score, n, eta, lam):
    """Set definition with a score that never changes: at step t the evicted keys are
    {i : i + eta <= t}; the cache is the lam of them with the largest (score, position); a
    key is written at the first step at which it is evicted but not among those."""
    ws = np.full(n, -1, np.int64)
    for t in range(n):
        ev = [i for i in range(n) if i + eta <= t]
        keep = set(sorted(ev, key=lambda i: (score[i], i))[max(0, len(ev) - lam):])
        for i in ev:
            if i not in keep and ws[i] < 0:
                ws[i] = t
    return ws


def _closed_form_write_steps(score, n, eta, lam):
    """Per key, with no steps simulated: j is written once it has been evicted and lam keys of
    higher (score, position) have been evicted too, i.e. at step max(j, p) + eta with p the
    lam-th smallest position among the higher keys (at j + eta when lam = 0); never if that
    step is past the end or there are fewer than lam higher keys."""
    ws = np.full(n, -1, np.int64)
    for j in range(n):
        higher = sorted(i for i in range(n) if (score[i], i) > (score[j], j))
        if len(higher) < lam:
            continue
        p = higher[lam - 1] if lam > 0 else j
        t = max(j, p) + eta
        if t <= n - 1:
            ws[j] = t
    return ws


@pytest.mark.parametrize("kind", ["kernel_sq", "kernel_abs", "kernel_ratio", "attention"])
@pytest.mark.parametrize("eta,lam", [(4, 3), (1, 5), (6, 1)])
def test_fixed_score_rule_keeps_the_top_lambda_of_the_evicted(kind, eta, lam):
    """A frozen score makes the cache the lam highest-scored evicted keys at every step (the
    incremental write-the-minimum rule equals the set definition and the per-key closed
    form), and (H, s) are the sums over the written keys."""
    x = synth.gauss_inputs(1, 1, 36, 8, 8, "f32", seed=101, dv=6)
    q, k, v = (x.widened(n)[0, 0] for n in "qkv")
    o = R.lola_run_fixed_score(q, k, v, x.W, eta, lam, kind)
    assert np.array_equal(o["write_step"], _top_lambda_write_steps(o["score"], 36, eta, lam))
    assert np.array_equal(o["write_step"], _closed_form_write_steps(o["score"], 36, eta, lam))
    wl = np.flatnonzero(o["write_step"] >= 0)
    PK = R.phi(k, x.W)
    np.testing.assert_allclose(o["H"], PK[wl].T @ v[wl], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(o["s"], PK[wl].sum(axis=0), rtol=1e-12, atol=1e-12)


def test_fixed_score_decisions_do_not_depend_on_values():
    """The query-dependent scores read q and k only, so any other V gives the same write log
    (unlike the SRE, which is a value reconstruction error)."""
    x = synth.gauss_inputs(1, 1, 40, 8, 8, "f32", seed=102, dv=6)
    q, k, v = (x.widened(n)[0, 0] for n in "qkv")
    other = synth.gauss_inputs(1, 1, 40, 8, 8, "f32", seed=103, dv=6).widened("v")[0, 0]
    for kind in R.SCORE_KINDS:
        a = R.lola_run_fixed_score(q, k, v, x.W, 4, 3, kind)
        b = R.lola_run_fixed_score(q, k, other, x.W, 4, 3, kind)
        assert np.array_equal(a["write_step"], b["write_step"]), kind


def test_fixed_score_reductions():
    """lambda = 0 writes every evictee at once, whatever the score: the SRE run's window +
    linear result.  lambda >= n (nothing written): causal softmax attention."""
    x = synth.gauss_inputs(1, 1, 30, 8, 8, "f32", seed=104, dv=6)
    q, k, v = (x.widened(n)[0, 0] for n in "qkv")
    ref0 = R.lola_run(q, k, v, x.W, 5, 0)
    full = R.causal_softmax_attention(q, k, v)
    for kind in R.SCORE_KINDS:
        o = R.lola_run_fixed_score(q, k, v, x.W, 5, 0, kind)
        assert np.array_equal(o["write_step"], ref0["write_step"])
        np.testing.assert_allclose(o["Y"], ref0["Y"], rtol=1e-12, atol=1e-12)
        o = R.lola_run_fixed_score(q, k, v, x.W, 3, 30, kind)
        assert (o["write_step"] < 0).all()
        np.testing.assert_allclose(o["Y"], full, rtol=1e-11, atol=1e-12)


def test_window_scores_of_a_key_seen_by_one_query():
    """eta = 1: each key is read only by its own step's query, so its scores are those of
    one (e, l) pair: e = exp(q_j . k_j / sqrt(d_k)), l = phi(q_j) . phi(k_j)."""
    q = np.array([[1.0, 0.0], [0.5, -0.5]])
    k = np.array([[2.0, 1.0], [0.0, 1.0]])
    W = np.array([[1.0, 0.0]])
    e = np.exp(np.array([2.0, -0.5]) / math.sqrt(2.0))
    # phi(x) = [softmax(W x), softmax(-W x)] with one row: both halves are 1, so l = 2
    assert np.allclose(R.phi(q, W), 1.0)
    np.testing.assert_allclose(R.window_scores(q, k, W, 1, "attention"), e, rtol=1e-15)
    np.testing.assert_allclose(R.window_scores(q, k, W, 1, "kernel_sq"), (e - 2.0) ** 2, rtol=1e-14)
    np.testing.assert_allclose(R.window_scores(q, k, W, 1, "kernel_abs"), np.abs(e - 2.0), rtol=1e-14)
    np.testing.assert_allclose(R.window_scores(q, k, W, 1, "kernel_ratio"), 2.0 / e, rtol=1e-15)


def test_fixed_score_golden_worked_example():
    """Hand-derived in tests/golden/query_scores_two_axes.json: queries and keys on two axes
    make every softmax weight 1 or 2 and (W = 0) every linear weight 1, so the four scores,
    each kind's decisions (a tie between a cached key and the evictee included) and the reads
    are worked out by hand."""
    with open(os.path.join(GOLDEN, "query_scores_two_axes.json")) as f:
        g = json.load(f)
    a = lambda key: np.asarray(g[key], dtype=np.float64)  # noqa: E731
    for kind, want in g["kinds"].items():
        np.testing.assert_allclose(R.window_scores(a("q"), a("k"), a("W"), g["eta"], kind), want["score"],
                                   rtol=1e-15, atol=1e-15)
        o = R.lola_run_fixed_score(a("q"), a("k"), a("v"), a("W"), g["eta"], g["lambda"], kind)
        np.testing.assert_allclose(o["score"], want["score"], rtol=1e-15, atol=1e-15)
        assert o["write_pos"].tolist() == want["write_pos"], kind
        assert o["cache"].tolist() == want["final_cache"], kind
        assert sorted(o["window"].tolist()) == g["final_window"]
        np.testing.assert_allclose(o["Y"], a("y"), rtol=1e-14, atol=1e-15)


def test_fixed_score_replay_of_own_and_of_a_swapped_log():
    """Replaying the own log reproduces it with no gap; writing, at one decision, the lowest
    kept key instead of the written one is followed and reported as their relative score
    difference; a log that writes a non-candidate is refused."""
    x = synth.gauss_inputs(1, 1, 40, 8, 8, "f32", seed=105, dv=6)
    q, k, v = (x.widened(n)[0, 0] for n in "qkv")
    own = R.lola_run_fixed_score(q, k, v, x.W, 4, 3, "attention")
    rep = R.lola_run_fixed_score(q, k, v, x.W, 4, 3, "attention", replay=own["write_step"])
    assert rep["max_gap"] == 0.0 and rep["mismatches"] == 0
    np.testing.assert_array_equal(rep["Y"], own["Y"])
    sc, ws = own["score"], own["write_step"]
    # the last decision: its written key and the lowest key kept at that step
    t = int(ws.max())
    w = int(np.flatnonzero(ws == t)[0])
    kept = [i for i in range(40) if i + 4 <= t and (ws[i] < 0 or ws[i] > t) and i != w]
    kp = min(kept, key=lambda i: (sc[i], i))
    log = ws.copy()
    log[w], log[kp] = -1, t
    sw = R.lola_run_fixed_score(q, k, v, x.W, 4, 3, "attention", replay=log)
    assert sw["mismatches"] == 1
    assert sw["max_gap"] == pytest.approx((sc[kp] - sc[w]) / abs(sc[w]), rel=1e-12)
    bad = ws.copy()
    bad[w], bad[int(np.flatnonzero(ws < 0)[-1])] = -1, t   # a key still in the window
    with pytest.raises(ValueError):
        R.lola_run_fixed_score(q, k, v, x.W, 4, 3, "attention", replay=bad)

