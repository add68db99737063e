"""The chunked form of the gated delta rule that the state kernel computes, restated in float64
numpy and checked against the oracle's token-by-token recurrence (``oracle/hola_ref.py``).

Method: "A Hippocampus for Linear Attention" (arXiv 2607.02303v1), reading notes sections 3.1 and
3.5: e_t = v_t - alpha_t S^T k^_t, S <- alpha_t S + beta_t k^_t e_t^T, read-out S^T q^_t, score
beta_t ||e_t||.  A pass over tokens [s0, s1) of a chunk starts from R_0 (the decay before it folded
in); with c_t the product of the pass's decays up to t and u'_t = beta_t e_t / c_t:
  (I + A') U' = W',  A'_tj = beta_t (k^_t . k^_j) (j < t),  W'_t = beta_t (v_t / c_t - R_0^T k^_t),
  y_t = c_t (R_0^T q^_t + sum_{j <= t} (q^_t . k^_j) u'_j),  m_t = ||c_t u'_t||,
  R_end = R_0 + sum_j k^_j u'_j^T,  S_end = c_{s1-1} R_end;
a pass ends before its running decay falls below 2^-100, and a decay below 2^-100 is taken as
2^-100.  This test pins that algebra (not the kernel: the GPU tests compare the kernel with the
oracle)."""
import numpy as np

import synth
from oracle import hola_ref as HR

MIN_C = 2.0 ** -100


def _unit(x):
    n = np.linalg.norm(x, axis=1, keepdims=True)
    return np.where(n > 0, x / np.where(n > 0, n, 1.0), 0.0)


def chunked_state(q, k, v, alpha, beta, chunk=64):
    n, dk = k.shape
    dv = v.shape[1]
    qh, kh = _unit(q), _unit(k)
    R, G = np.zeros((dk, dv)), 1.0
    y, m = np.zeros((n, dv)), np.zeros(n)
    passes = 0
    for c0 in range(0, n, chunk):
        mlen = min(chunk, n - c0)
        s0 = 0
        while s0 < mlen:
            a = np.maximum(alpha[c0 + s0:c0 + mlen], MIN_C)
            c = np.cumprod(a)
            below = np.nonzero(c < MIN_C)[0]
            s1 = s0 + (int(below[0]) if len(below) else mlen - s0)
            c = c[:s1 - s0]
            t = np.arange(c0 + s0, c0 + s1)
            R0 = G * R
            K, Q, V, b = kh[t], qh[t], v[t], beta[t]
            A = np.tril(b[:, None] * (K @ K.T), -1)
            W = b[:, None] * (V / c[:, None] - K @ R0)
            U = np.linalg.solve(np.eye(len(t)) + A, W)
            y[t] = c[:, None] * (Q @ R0 + np.tril(Q @ K.T) @ U)
            m[t] = np.linalg.norm(c[:, None] * U, axis=1)
            R = R0 + K.T @ U
            G = c[-1]
            s0 = s1
            passes += 1
    return y, m, G * R, passes


def _check(x, h, chunk=64, min_passes=None):
    q, k, v = (x.widened(a)[0, h] for a in "qkv")
    al, be = x.alpha[0, h].astype(np.float64), x.beta[0, h].astype(np.float64)
    ys, m, _, S = HR.delta_state_run(q, k, v, al, be)
    yc, mc, Sc, passes = chunked_state(q, k, v, al, be, chunk)
    scale = max(1.0, np.abs(S).max())
    np.testing.assert_allclose(yc, ys, atol=1e-9 * scale)
    np.testing.assert_allclose(mc, m, atol=1e-9 * max(1.0, np.abs(m).max()))
    np.testing.assert_allclose(Sc, S, atol=1e-9 * scale)
    if min_passes is not None:
        assert passes >= min_passes
    return passes


def test_chunked_form_equals_the_recurrence():
    """Decays near 1: one pass per chunk, ragged last chunk."""
    x = synth.hola_inputs(1, 2, 300, 32, w=8, chunk=128, dtype="f32", seed=21)
    for h in range(2):
        assert _check(x, h) == (300 + 63) // 64


def test_small_decays_split_a_chunk_into_passes():
    """Running decays below 2^-100 inside a chunk start new passes; the result is unchanged."""
    x = synth.hola_inputs(1, 2, 200, 32, w=8, chunk=128, dtype="f32", seed=22)
    x.alpha[0, 0, [5, 9, 20, 70, 71, 72]] = [1e-20, 1e-20, 1e-20, 1e-30, 1e-30, 1e-30]
    x.alpha[0, 1, 64:128] = 0.25          # 0.25^50 = 2^-100: the chunk needs two passes
    _check(x, 0, min_passes=(200 + 63) // 64 + 2)
    _check(x, 1, min_passes=(200 + 63) // 64 + 1)


def test_a_decay_below_the_floor_is_a_change_below_resolution():
    """A decay of 1e-40 taken as 2^-100: the state before it still enters only at ~1e-30 relative."""
    x = synth.hola_inputs(1, 1, 150, 16, w=4, chunk=128, dtype="f32", seed=23)
    x.alpha[0, 0, 100] = 1e-40
    _check(x, 0)
