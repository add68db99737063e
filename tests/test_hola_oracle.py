"""Pins of the write-magnitude-cache oracle (``oracle/hola_ref.py``) to closed forms, an
independent restatement of the gated delta rule and library attention.

Method: "A Hippocampus for Linear Attention" (arXiv 2607.02303v1), reading notes sections
3.1-3.5."""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import hola_ref as HR


def _rng(seed):
    return np.random.default_rng(seed)


def test_orthonormal_keys_are_recalled_exactly():
    """alpha = beta = 1 and orthonormal keys: every write sees a zero prediction (e = v,
    score = ||v||) and the final state recalls every value exactly (section 3.1, Eq. 1)."""
    n, dk, dv = 6, 8, 5
    Qm, _ = np.linalg.qr(_rng(1).standard_normal((dk, dk)))
    k = Qm[:n] * 3.0                              # scaled: the state path normalises keys
    v = _rng(2).standard_normal((n, dv))
    q = _rng(3).standard_normal((n, dk))
    ys, m, E, S = HR.delta_state_run(q, k, v, np.ones(n), np.ones(n))
    np.testing.assert_allclose(E, v, atol=1e-12)
    np.testing.assert_allclose(m, np.linalg.norm(v, axis=1), rtol=1e-12)
    np.testing.assert_allclose(S.T @ Qm[:n].T, v.T, atol=1e-12)


def test_zero_write_strength_leaves_the_state_empty():
    n, d = 9, 4
    r = _rng(4)
    q, k, v = r.standard_normal((3, n, d))
    ys, m, E, S = HR.delta_state_run(q, k, v, r.uniform(0.5, 1.0, n), np.zeros(n))
    assert not S.any() and not ys.any() and not m.any()
    np.testing.assert_array_equal(E, v)


def test_repeated_key_overwrites_its_value():
    """The delta rule replaces, it does not add: writing (k, v1) then (k, v2) with
    alpha = beta = 1 predicts v2 for k, and the second residual is v2 - v1."""
    k = np.array([[1.0, 2.0, 2.0], [1.0, 2.0, 2.0]])
    v = np.array([[1.0, -1.0], [3.0, 5.0]])
    ys, m, E, S = HR.delta_state_run(k, k, v, np.ones(2), np.ones(2))
    np.testing.assert_allclose(S.T @ (k[0] / 3.0), v[1], atol=1e-12)
    np.testing.assert_allclose(E[1], v[1] - v[0], atol=1e-12)
    np.testing.assert_allclose(ys[1], v[1], atol=1e-12)


def _householder_states(q, k, v, alpha, beta):
    """S_t = alpha_t (I - beta_t k^ k^T) S_{t-1} + beta_t k^ v_t^T, the same recurrence written as
    a decayed projection plus a rank-one write."""
    kh = k / np.linalg.norm(k, axis=1, keepdims=True)
    S = np.zeros((k.shape[1], v.shape[1]))
    out = []
    for t in range(len(k)):
        P = np.eye(k.shape[1]) - beta[t] * np.outer(kh[t], kh[t])
        S = alpha[t] * P @ S + beta[t] * np.outer(kh[t], v[t])
        out.append(S.copy())
    return out


def test_gated_delta_rule_matches_its_projection_form_and_the_score_is_the_write_norm():
    """Section 3.5's gated form against its projection restatement, and Eqs. 5-6: the score is
    the Frobenius norm of the correction, ||S_t - alpha_t S_{t-1}||_F = beta_t ||e_t||."""
    n, dk, dv = 12, 5, 3
    r = _rng(5)
    q, k = r.standard_normal((2, n, dk))
    v = r.standard_normal((n, dv))
    alpha, beta = r.uniform(0.8, 1.0, n), r.uniform(0.0, 1.0, n)
    ys, m, E, S = HR.delta_state_run(q, k, v, alpha, beta)
    Ss = _householder_states(q, k, v, alpha, beta)
    np.testing.assert_allclose(S, Ss[-1], atol=1e-12)
    qh = q / np.linalg.norm(q, axis=1, keepdims=True)
    for t in range(n):
        prev = Ss[t - 1] if t else np.zeros_like(S)
        np.testing.assert_allclose(np.linalg.norm(Ss[t] - alpha[t] * prev), m[t], rtol=1e-10, atol=1e-14)
        np.testing.assert_allclose(ys[t], Ss[t].T @ qh[t], atol=1e-12)


def test_running_cache_equals_the_sorted_definition_with_ties():
    """The token-by-token cache equals, at every chunk start, the w best of the tokens before it
    ranked by (higher score, older position): integer scores force many ties."""
    r = _rng(6)
    for w, chunk, n in [(4, 3, 40), (7, 8, 64), (1, 5, 23), (16, 4, 30)]:
        scores = r.integers(0, 5, n).astype(np.float64)
        a, b = HR.topw_running(scores, w, chunk), HR.topw_sorted(scores, w, chunk)
        assert len(a) == len(b) == (n + chunk - 1) // chunk
        for x, y in zip(a, b):
            np.testing.assert_array_equal(x, y)


def test_equal_scores_keep_the_oldest_tokens():
    caches = HR.topw_running(np.ones(50), 8, 10)
    np.testing.assert_array_equal(caches[-1], np.arange(8))
    assert len(caches[0]) == 0


def test_rms_scale_closed_form():
    x = np.full((1, 16), 2.0)
    np.testing.assert_allclose(HR.rms_scaled(x, np.ones(16)), 2.0 / math.sqrt(4.0 + HR.RMS_EPS), rtol=1e-15)
    g = np.arange(1.0, 17.0)
    np.testing.assert_allclose(HR.rms_scaled(x, g)[0], g * 2.0 / math.sqrt(4.0 + HR.RMS_EPS), rtol=1e-15)


def test_read_with_everything_cached_and_no_sink_is_causal_softmax():
    """w >= n and a sink of weight 0: every earlier token is visible, so the read is causal
    softmax attention on the RMS-scaled queries and keys (library SDPA)."""
    n, d, chunk = 20, 8, 6
    r = _rng(7)
    q, k, v = r.standard_normal((3, n, d))
    gq, gk = r.uniform(0.8, 1.2, d), r.uniform(0.8, 1.2, d)
    caches = HR.topw_running(r.standard_normal(n), n, chunk)
    out = HR.cache_read(q, k, v, caches, chunk, gq, gk, -1e9)
    qt = torch.from_numpy(HR.rms_scaled(q, gq))[None, None]
    kt = torch.from_numpy(HR.rms_scaled(k, gk))[None, None]
    want = torch.nn.functional.scaled_dot_product_attention(qt, kt, torch.from_numpy(v)[None, None], is_causal=True)
    np.testing.assert_allclose(out, want[0, 0].numpy(), atol=1e-12)


def test_sink_closed_form_on_one_token():
    q = np.array([[1.0, 0.0, 2.0, -1.0]])
    k = np.array([[0.5, 1.0, -1.0, 2.0]])
    v = np.array([[2.0, -3.0]])
    g = np.ones(4)
    logit = float(HR.rms_scaled(q, g)[0] @ HR.rms_scaled(k, g)[0]) / 2.0
    for sink in (-2.0, 0.0, 1.5):
        out = HR.cache_read(q, k, v, [np.zeros(0, dtype=np.int64)], 4, g, g, sink)
        np.testing.assert_allclose(out[0], v[0] / (1.0 + math.exp(sink - logit)), rtol=1e-14)


def test_read_is_causal_and_cache_changes_only_at_chunk_starts():
    """Query t reads nothing after t; a token enters the cache only for later chunks."""
    n, d, chunk, w = 24, 6, 8, 3
    x = synth.hola_inputs(1, 1, n, d, w=w, chunk=chunk, dtype="f32", seed=3)
    base = HR.hola_run(x)[(0, 0)]
    x.v[0, 0, 13] += 5.0
    x.k[0, 0, 13] += 1.0
    moved = HR.hola_run(x)[(0, 0)]
    np.testing.assert_array_equal(base["Y"][:13], moved["Y"][:13])
    for c, cache in enumerate(base["caches"]):
        assert (cache < c * chunk).all() and len(cache) == min(w, c * chunk)


def test_gate_zero_leaves_the_state_read_out():
    x = synth.hola_inputs(1, 2, 30, 8, w=4, chunk=8, dtype="f32", seed=4)
    x.gate[:] = 0.0
    for (b, h), r in HR.hola_run(x).items():
        np.testing.assert_array_equal(r["Y"], r["y_state"])


def test_hand_derived_worked_example():
    """Six tokens on two axes, derived by hand in tests/golden/hola_worked_example.json: the
    delta rule's residuals, decays and write strengths in exact fractions, a score tie at a chunk
    start (the older token stays), RMS-scaled logits with per-channel query scales, the sink and
    the gate."""
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", "hola_worked_example.json")) as f:
        g = json.load(f)
    a = lambda key: np.asarray(g[key], dtype=np.float64)  # noqa: E731
    out = HR.hola_head(a("q"), a("k"), a("v"), a("alpha"), a("beta"), a("gamma_q"), a("gamma_k"),
                       float(g["sink"]), float(g["gate"]), int(g["w"]), int(g["chunk"]))
    for key in ("scores", "S", "y_state", "o_cache", "Y"):
        np.testing.assert_allclose(out[key], a(key), rtol=1e-13, atol=1e-15, err_msg=key)
    for caches in (out["caches"], HR.topw_sorted(out["scores"], int(g["w"]), int(g["chunk"]))):
        assert [list(map(int, c)) for c in caches] == g["caches"]
