"""CPU float64 oracle for the write-magnitude exact cache on a gated delta-rule state --
TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import this
module.  The CUDA library never calls it and shares no code with it.

Source: "A Hippocampus for Linear Attention: An Exact Memory for What the Recurrent State
Forgets" (arXiv 2607.02303v1), Chinese reading notes, method sections 3.1-3.5.  Per head, with
column vectors, S of shape (d_k, d_v), S_{-1} = 0:

* state path (section 3.1, Eq. 1, in the gated form of section 3.5): unit-L2 key k^_t, the
  residual of the decayed state's prediction e_t = v_t - alpha_t S_{t-1}^T k^_t, and the write
  S_t = alpha_t S_{t-1} + beta_t k^_t e_t^T; its read-out S_t^T q^_t with the unit-L2 query;
* write-magnitude score (section 3.3, Eqs. 5-6): m_t = beta_t ||e_t||_2, the Frobenius norm of
  the rank-one correction beta_t k^_t e_t^T (||k^_t|| = 1), fixed when the token is written;
* persistent cache (section 3.3): the w tokens with the highest fixed scores so far;
* cache read (section 3.3's visible set, section 3.4, Eq. 7): RMS-normalised query and key
  with their own scales gamma_q, gamma_k, temperature 1 over sqrt(d_k), a softmax over the
  persistent cache, the current chunk's tokens up to t and a null sink;
* output (section 3.2, Eq. 3: state prediction plus the non-parametric read-out, weighted by
  the per-head cache gate of section 3.5): y_t = S_t^T q^_t + lambda_h o_t.

Readings taken where the notes leave the step open (each is listed in the design notes):

* the cache changes only at chunk boundaries: the queries of chunk [c0, c0 + C) read the w best
  tokens among j < c0 plus the chunk's own tokens j <= t (so no token is read twice);
* ties in the score keep the older token (a new token enters only with a strictly larger score
  than the cache's worst entry; among equal scores the newest is the worst);
* RMS normalisation: x / sqrt(mean(x^2) + 1e-6), then the per-channel scale;
* the sink is a key whose logit is the head's ``sink`` value and whose value is zero;
* the state read-out uses S_t, after token t's write (as in the delta rule's output).
"""
from __future__ import annotations

import math

import numpy as np

RMS_EPS = 1e-6


def unit(x: np.ndarray) -> np.ndarray:
    """x / ||x||_2 along the last axis (float64)."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def rms_scaled(x: np.ndarray, gamma: np.ndarray) -> np.ndarray:
    """gamma * x / sqrt(mean(x^2) + eps) along the last axis (float64)."""
    x = np.asarray(x, dtype=np.float64)
    return np.asarray(gamma, dtype=np.float64) * x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + RMS_EPS)


def delta_state_run(q, k, v, alpha, beta):
    """The gated delta-rule state of one head (section 3.1, Eq. 1; section 3.5), token by token.

    q, k: (n, d_k); v: (n, d_v); alpha, beta: (n,).  Returns the state read-out S_t^T q^_t per
    token (n, d_v), the write-magnitude scores beta_t ||e_t|| (n,), the residuals e_t (n, d_v) and
    the final S (d_k, d_v)."""
    kh, qh = unit(k), unit(q)
    v = np.asarray(v, dtype=np.float64)
    n, dk = kh.shape
    S = np.zeros((dk, v.shape[1]))
    ys = np.zeros((n, v.shape[1]))
    m = np.zeros(n)
    E = np.zeros((n, v.shape[1]))
    for t in range(n):
        a, b = float(alpha[t]), float(beta[t])
        e = v[t] - a * (S.T @ kh[t])
        S = a * S + b * np.outer(kh[t], e)
        E[t] = e
        m[t] = b * np.linalg.norm(e)
        ys[t] = S.T @ qh[t]
    return ys, m, E, S


def topw_running(scores, w: int, chunk: int):
    """The persistent cache at every chunk start, kept token by token (section 3.3): a new token
    replaces the worst entry (lowest score, the newest among equal scores) when its score is
    strictly larger; the first w tokens fill the cache.  Returns one sorted position array per
    chunk start c0 = 0, C, 2C, ... < n (the tokens j < c0 it holds)."""
    n = len(scores)
    held: list[int] = []
    out = []
    for t in range(n):
        if t % chunk == 0:
            out.append(np.array(sorted(held), dtype=np.int64))
        if len(held) < w:
            held.append(t)
            continue
        if w == 0:
            continue
        worst = min(held, key=lambda j: (scores[j], -j))
        if scores[t] > scores[worst]:
            held.remove(worst)
            held.append(t)
    return out


def topw_sorted(scores, w: int, chunk: int):
    """The same caches by definition: at chunk start c0, the w tokens j < c0 ranked first by
    (higher score, older position)."""
    n = len(scores)
    out = []
    for c0 in range(0, n, chunk):
        order = sorted(range(c0), key=lambda j: (-scores[j], j))
        out.append(np.array(sorted(order[:w]), dtype=np.int64))
    return out


def cache_read(q, k, v, caches, chunk: int, gamma_q, gamma_k, sink: float):
    """The cache read-out of one head (section 3.4, Eq. 7): softmax over the persistent cache of
    the query's chunk, the chunk's tokens up to the query and the null sink (value 0)."""
    qt, kt = rms_scaled(q, gamma_q), rms_scaled(k, gamma_k)
    v = np.asarray(v, dtype=np.float64)
    n, d = qt.shape
    out = np.zeros((n, v.shape[1]))
    for t in range(n):
        c = t // chunk
        keys = np.concatenate([caches[c], np.arange(c * chunk, t + 1)])
        logits = kt[keys] @ qt[t] / math.sqrt(d)
        mx = max(logits.max(), sink)
        p = np.exp(logits - mx)
        out[t] = (p @ v[keys]) / (p.sum() + math.exp(sink - mx))
    return out


def hola_head(q, k, v, alpha, beta, gamma_q, gamma_k, sink: float, gate: float, w: int, chunk: int):
    """One head end to end: state path, scores, caches, cache read, output."""
    ys, m, _, S = delta_state_run(q, k, v, alpha, beta)
    caches = topw_running(m, w, chunk)
    oc = cache_read(q, k, v, caches, chunk, gamma_q, gamma_k, sink)
    return {"Y": ys + gate * oc, "y_state": ys, "o_cache": oc, "scores": m, "caches": caches, "S": S}


def hola_run(x, heads=None):
    """Every head of a ``synth.HolaInputs`` (or the listed (b, h) pairs)."""
    q, k, v = x.widened("q"), x.widened("k"), x.widened("v")
    out = {}
    pairs = heads if heads is not None else [(b, h) for b in range(x.B) for h in range(x.Hh)]
    for b, h in pairs:
        out[(b, h)] = hola_head(q[b, h], k[b, h], v[b, h], x.alpha[b, h].astype(np.float64),
                                x.beta[b, h].astype(np.float64), x.gamma_q, x.gamma_k, float(x.sink[h]),
                                float(x.gate[h]), x.w, x.chunk)
    return out
