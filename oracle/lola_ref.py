"""CPU float64 oracle for LoLA hybrid attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may
import this package.  The CUDA library never calls it and shares no code with it.

Source: "LoLA: Low-Rank Linear Attention With Sparse Caching" (arXiv 2505.23666v3),
Chinese reading notes, sections 2.1-2.7.  Per attention head:

* feature map (section 2.2, Eq. 3; the configured form): ``phi(x) = [softmax(W x), softmax(-W x)]``
  with ``W`` of shape (D/2, d_k), so ``phi(x)`` is strictly positive and each half sums to 1;
* linear memory (section 2.2, Eqs. 3-5): ``H += phi(k) v^T``, ``s += phi(k)``, read-out
  ``H^T phi(q) / (phi(q)^T s)``; only KV actually assigned to the state are added;
* self-recall error (section 2.3, Eq. 10): ``SRE(k, v | H, s) = || H^T phi(k) / (phi(k)^T s) - v ||_2``
  (the L2 norm, not its square);
* per-token allocation (section 2.4, Eqs. 11-13, "score, then write" as in appendix H):
  the new KV enters the sliding window; once the window holds more than eta entries the
  oldest one leaves and joins the candidates ``E = G ∪ {evictee}``; if ``|E| <= lambda`` all
  are kept, otherwise the lambda highest-SRE candidates (scored against the state *before*
  this step's write) stay in the sparse cache G and the rest are written into (H, s) once;
* co-normalised output (section 2.5, Eq. 14): one shared denominator over the linear
  memory, the sparse cache and the window, with ``a = exp(q^T k / sqrt(d_k))``.

Readings taken where the notes are silent (each is listed in the design notes):

* R0: the per-token rule above is the definition; the prefill chunk length C only
  schedules work and never changes which KV are kept (section 2.6's chunk-granular
  allocation is a different variant, not this one);
* the window includes the current token: ``W_t = {max(0, t-eta+1) .. t}``, evictee ``t-eta``;
* empty-state rule (section 2.6 notes that H = 0, s = 0 makes the SRE division undefined):
  when ``phi(k)^T s = 0`` the memory predicts 0, so ``SRE = ||v||``;
* exact capacity with ties broken towards the older token: among equal SREs the smaller
  position is written; SRE order is compared through SRE^2 (same order);
* the output is read after this step's write, with H_t, G_t and W_t (so every token
  <= t is in exactly one of window, cache, state);
* only the softmax branch carries the 1/sqrt(d_k) temperature; the linear branch is the
  plain ``phi(q)^T phi(k)``.  The max-subtraction in the output is for range only;
* read mask (appendix I, Table 12: a read-time ablation; the cache and the state are
  updated exactly as without it): bit 0 leaves the state's terms ``H^T phi(q)`` and
  ``phi(q)^T s`` out of the read, bit 1 the cache's keys; the window is always read, and
  a nonzero mask needs eta >= 1 (then the window holds the current token).

Scoring ablation (section 4.4, Table 4; appendix F, whose formulas the notes do not
reproduce): ``lola_run_fixed_score`` runs the per-token rule with one of four
query-dependent scores in place of the SRE, each accumulated while the key is in the window
and frozen from its eviction on.  Readings taken: e = exp(q . k / sqrt(d_k)) and
l = phi(q) . phi(k) are the two branches' unnormalised weights; the scores are sum (e - l)^2,
sum |e - l|, sum l / e and sum e over the key's window queries; a larger score keeps the key.

Diagnostics (not on the path): the SRE map (section 4.4, Fig. 3) -- every key's SRE against
the memory at chosen state times, 0 for keys it does not hold -- and the relative map
(appendix G, Fig. 10, Eq. 26): the SRE now minus the SRE at first write.  Reading taken for
the latter's baseline: the SRE against the first memory that holds the key, i.e. the
memory right after its write step (not the score it had just before the write).

Three formulations live here and in ``lola_inc.c``: ``lola_run`` (running H, s; all
SREs recomputed from H each step), ``lola_set`` (no running state: H is re-summed from
the written set every step) and the C incremental form.  Tests check that they agree,
and pin them to closed forms that the method reduces to.
"""
from __future__ import annotations

import math
from collections import deque

import numpy as np


def phi(x: np.ndarray, W: np.ndarray) -> np.ndarray:
    """Feature map ``[softmax(W x), softmax(-W x)]`` over the last axis of ``x`` (float64)."""
    z = np.asarray(x, dtype=np.float64) @ np.asarray(W, dtype=np.float64).T
    out = []
    for zz in (z, -z):
        e = np.exp(zz - zz.max(axis=-1, keepdims=True))
        out.append(e / e.sum(axis=-1, keepdims=True))
    return np.concatenate(out, axis=-1)


def sre_sq(H: np.ndarray, s: np.ndarray, phik: np.ndarray, v: np.ndarray) -> float:
    """Squared self-recall error of (k, v) against memory (H, s) (section 2.3, Eq. 10).

    Empty-memory reading: if ``phi(k)^T s == 0`` the memory predicts 0 and SRE = ||v||."""
    den = float(phik @ s)
    if den == 0.0:
        return float(v @ v)
    r = (H.T @ phik) / den - v
    return float(r @ r)


def _check_mask(eta: int, read_mask: int) -> None:
    if read_mask not in (0, 1, 2, 3) or (read_mask and eta < 1):
        raise ValueError(f"read mask {read_mask} with eta = {eta}: nothing would be left to read")


def _output(qt, phiq, exact, K, V, H_num, den_lin, scale):
    """Co-normalised read (section 2.5, Eq. 14).  ``H_num = H^T phi(q)``, ``den_lin = phi(q)^T s``."""
    if len(exact):
        idx = np.fromiter(exact, dtype=np.int64)
        a = (K[idx] @ qt) * scale
        m = a.max()
        w = np.exp(a - m)
        em = math.exp(-m)
        num = w @ V[idx] + em * H_num
        den = w.sum() + em * den_lin
    else:
        num, den = H_num, den_lin
    return num / den


def lola_run(q, k, v, W, eta: int, lam: int, replay=None, read_mask: int = 0):
    """Per-token LoLA on one head with a running (H, s); float64.

    ``q, k``: (n, d_k); ``v``: (n, d_v); ``W``: (D/2, d_k).  ``replay``: optional (n,)
    int array of the position written at each step (-1: none); when given, the oracle
    follows those decisions instead of its own and reports how far each was from its
    own best (relative SRE gap).  ``read_mask``: see the module notes (read time only).

    Returns a dict with Y (n, d_v), write_pos (n,), write_step (n,), H, s, cache
    (sorted positions), window (positions), min_gap (smallest relative SRE gap between
    the best and the second-best candidate over all decisions of a free run), max_gap
    and mismatches (replay only).
    """
    _check_mask(eta, read_mask)
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    n, dk = k.shape
    dv = v.shape[1]
    PQ, PK = phi(q, W), phi(k, W)
    D = PK.shape[1]
    scale = 1.0 / math.sqrt(dk)
    H = np.zeros((D, dv))
    s = np.zeros(D)
    window: deque[int] = deque()
    cache: list[int] = []
    write_pos = np.full(n, -1, np.int64)
    write_step = np.full(n, -1, np.int64)
    Y = np.zeros((n, dv))
    min_gap, max_gap, mismatches = math.inf, 0.0, 0
    for t in range(n):
        window.append(t)
        E = list(cache)
        if len(window) > eta:
            E.append(window.popleft())
        if len(E) <= lam:
            cache = E
            if replay is not None and replay[t] != -1:
                raise ValueError(f"replay writes at step {t} but no write is due")
        else:
            sq = {j: sre_sq(H, s, PK[j], v[j]) for j in E}
            best = min(E, key=lambda j: (sq[j], j))
            if len(E) > 1:
                second = min((j for j in E if j != best), key=lambda j: (sq[j], j))
                sb, s2 = math.sqrt(sq[best]), math.sqrt(sq[second])
                gap = (s2 - sb) / sb if sb > 0 else (math.inf if s2 > 0 else 0.0)
                min_gap = min(min_gap, gap)
            w = best
            if replay is not None:
                w = int(replay[t])
                if w not in sq:
                    raise ValueError(f"replay writes position {w} at step {t}, not a candidate")
                if w != best:
                    mismatches += 1
                    sb, sw = math.sqrt(sq[best]), math.sqrt(sq[w])
                    gap = (sw - sb) / sb if sb > 0 else (math.inf if sw > 0 else 0.0)
                    max_gap = max(max_gap, gap)
            H += np.outer(PK[w], v[w])
            s += PK[w]
            write_pos[t] = w
            write_step[w] = t
            cache = [j for j in E if j != w]
        exact = list(window) + ([] if read_mask & 2 else cache)
        if read_mask & 1:
            Y[t] = _output(q[t], PQ[t], exact, k, v, np.zeros(dv), 0.0, scale)
        else:
            Y[t] = _output(q[t], PQ[t], exact, k, v, H.T @ PQ[t], float(PQ[t] @ s), scale)
    return dict(Y=Y, write_pos=write_pos, write_step=write_step, H=H, s=s,
                cache=np.array(sorted(cache), np.int64), window=np.array(list(window), np.int64),
                min_gap=min_gap, max_gap=max_gap, mismatches=mismatches)


SCORE_KINDS = ("kernel_sq", "kernel_abs", "kernel_ratio", "attention")


def window_scores(q, k, W, eta: int, kind: str):
    """Query-dependent cache scores of the notes' scoring ablation (section 4.4, Table 4;
    appendix F), accumulated while key j is in the window, i.e. over the queries of steps
    t = j .. min(n, j + eta) - 1.  With e = exp(q_t . k_j / sqrt(d_k)) (the softmax branch's
    weight) and l = phi(q_t) . phi(k_j) (the linear branch's weight):
    kernel_sq = sum (e - l)^2, kernel_abs = sum |e - l|, kernel_ratio = sum l / e (large
    when the linear kernel over-weights the key), attention = sum e.  A larger score keeps
    the key exact."""
    if kind not in SCORE_KINDS:
        raise ValueError(f"unknown score {kind!r}")
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    n, dk = k.shape
    PQ, PK = phi(q, W), phi(k, W)
    scale = 1.0 / math.sqrt(dk)
    out = np.zeros(n)
    for j in range(n):
        for t in range(j, min(n, j + eta)):
            e = math.exp(float(q[t] @ k[j]) * scale)
            lin = float(PQ[t] @ PK[j])
            if kind == "kernel_sq":
                out[j] += (e - lin) ** 2
            elif kind == "kernel_abs":
                out[j] += abs(e - lin)
            elif kind == "kernel_ratio":
                out[j] += lin / e
            else:
                out[j] += e
    return out


def lola_run_fixed_score(q, k, v, W, eta: int, lam: int, kind: str, replay=None):
    """The per-token rule with a query-dependent score in place of the SRE (the notes'
    scoring ablation, section 4.4, Table 4).  Every key's score is complete when it leaves
    the window (``window_scores``) and never changes after, so no rescoring happens: at each
    eviction the candidates are the cache and the evictee, and when they exceed lambda the
    one with the lowest (score, position) is written (the older among equal scores).  The
    memory and the co-normalised read are those of ``lola_run``.  ``replay``: an optional
    (n,) per-key write step (-1: never) to follow instead of the own choice; a step whose
    replayed write is not one of its candidates, or a write due with none replayed, raises.
    Returns the same keys as ``lola_run`` plus ``score``; ``max_gap`` is the largest
    (score_written - score_lowest) / |score_lowest| over the replayed decisions."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    n, dk = k.shape
    dv = v.shape[1]
    if eta < 1:
        raise ValueError("a query-dependent score needs eta >= 1 (the key's queries are read in the window)")
    score = window_scores(q, k, W, eta, kind)
    PQ, PK = phi(q, W), phi(k, W)
    scale = 1.0 / math.sqrt(dk)
    H = np.zeros((PK.shape[1], dv))
    s = np.zeros(PK.shape[1])
    window: deque[int] = deque()
    cache: list[int] = []
    write_pos = np.full(n, -1, np.int64)
    write_step = np.full(n, -1, np.int64)
    Y = np.zeros((n, dv))
    due = {}
    if replay is not None:
        for j, st in enumerate(np.asarray(replay)):
            if st >= 0:
                if int(st) in due:
                    raise ValueError(f"replay writes two keys at step {int(st)}")
                due[int(st)] = j
    max_gap, mismatches = 0.0, 0
    for t in range(n):
        window.append(t)
        E = list(cache)
        if len(window) > eta:
            E.append(window.popleft())
        if replay is not None and (t in due) != (len(E) > lam):
            raise ValueError(f"replay and the capacity disagree on a write at step {t}")
        if len(E) > lam:
            w = min(E, key=lambda j: (score[j], j))
            if replay is not None:
                best, w = w, due[t]
                if w not in E:
                    raise ValueError(f"replay writes position {w} at step {t}, not a candidate")
                if w != best:
                    mismatches += 1
                    sb = score[best]
                    gap = (score[w] - sb) / abs(sb) if sb != 0 else (math.inf if score[w] != sb else 0.0)
                    max_gap = max(max_gap, gap)
            H += np.outer(PK[w], v[w])
            s += PK[w]
            write_pos[t] = w
            write_step[w] = t
            E = [j for j in E if j != w]
        cache = E
        Y[t] = _output(q[t], PQ[t], list(window) + cache, k, v, H.T @ PQ[t], float(PQ[t] @ s), scale)
    return dict(Y=Y, write_pos=write_pos, write_step=write_step, H=H, s=s, score=score,
                cache=np.array(sorted(cache), np.int64), window=np.array(list(window), np.int64),
                max_gap=max_gap, mismatches=mismatches)


def lola_set(q, k, v, W, eta: int, lam: int, read_mask: int = 0):
    """Brute-force LoLA with no running state (small n only).

    Every quantity is summed from explicit sets each step: the memory read-out for a
    key c is ``sum_{j in S} (phi_c . phi_j) v_j / sum_{j in S} phi_c . phi_j`` over the
    written set S, and the output's linear terms are ``sum_{j in S} (phi_q . phi_j) v_j``
    and ``sum_{j in S} phi_q . phi_j``.  Same decisions and outputs as ``lola_run`` in
    exact arithmetic (with the same read mask)."""
    _check_mask(eta, read_mask)
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    n, dk = k.shape
    PQ, PK = phi(q, W), phi(k, W)
    scale = 1.0 / math.sqrt(dk)
    written: list[int] = []
    cache: list[int] = []
    write_pos = np.full(n, -1, np.int64)
    write_step = np.full(n, -1, np.int64)
    Y = np.zeros((n, v.shape[1]))
    for t in range(n):
        win = list(range(max(0, t - eta + 1), t + 1))
        E = list(cache)
        if t - eta >= 0:
            E.append(t - eta)
        if len(E) <= lam:
            cache = E
        else:
            def err2(c):
                g = np.array([PK[c] @ PK[j] for j in written])
                if len(written) == 0 or g.sum() == 0.0:
                    return float(v[c] @ v[c])
                r = (g @ v[written]) / g.sum() - v[c]
                return float(r @ r)
            sq = {j: err2(j) for j in E}
            w = min(E, key=lambda j: (sq[j], j))
            written.append(w)
            write_pos[t] = w
            write_step[w] = t
            cache = [j for j in E if j != w]
        read = [] if read_mask & 1 else written
        gl = np.array([PQ[t] @ PK[j] for j in read]) if read else np.zeros(0)
        num_lin = gl @ v[read] if read else np.zeros(v.shape[1])
        Y[t] = _output(q[t], PQ[t], win + ([] if read_mask & 2 else cache), k, v, num_lin, float(gl.sum()), scale)
    return dict(Y=Y, write_pos=write_pos, write_step=write_step,
                cache=np.array(sorted(cache), np.int64), written=np.array(written, np.int64))


def lola_chunk_run(q, k, v, W, eta: int, lam: int, C: int, trace=None, replay=None):
    """Chunk-granular LoLA (section 2.6, Eq. 15, the notes' own prefill) on one head; float64.

    Readings (the notes call the mapping between eta, the window and the chunk length
    ambiguous; these are the ones taken): the sequence is cut into chunks of C tokens; the
    window holds the last eta / C chunks, the current one included (eta a positive
    multiple of C), so a query of chunk c reads its own chunk up to itself and the eta/C - 1
    chunks before it; every query of a chunk reads the state (H, s) and the cache as they
    stood when the chunk began; when a chunk begins (after the first eta/C), the oldest
    chunk of the previous window leaves it and joins the cache as candidates, each scored
    (SRE, Eq. 10, the empty-memory rule R3) against the current (H, s); if there are more
    than lambda, the lambda highest stay and the rest are written into (H, s) at once, the
    lowest SRE first and the older position first among equal ones.  With C = 1 this is the
    per-token rule (``lola_run``), final state included.

    Returns Y (n, d_v), write_step (n,): for every written key the start of the chunk
    before which it was written (the first query that reads it through the state), else
    -1; H, s and the final cache and window positions.  ``trace``: an optional list that
    receives (chunk start, {candidate: SRE^2}, written, kept) for every scored decision.
    ``replay``: another implementation's write_step; the oracle then writes, at every
    chunk start, the candidates that log says, checks that their count is the one due, and
    reports as max_gap the largest relative SRE excess of a written candidate over a kept
    one (0 when the log follows the oracle's own order; ValueError if it is not a valid
    decision)."""
    if C < 1 or eta < C or eta % C:
        raise ValueError(f"chunk mode needs eta a positive multiple of C (eta = {eta}, C = {C})")
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    n, dk = k.shape
    dv = v.shape[1]
    PQ, PK = phi(q, W), phi(k, W)
    D = PK.shape[1]
    scale = 1.0 / math.sqrt(dk)
    nwc = eta // C
    H = np.zeros((D, dv))
    s = np.zeros(D)
    cache: list[int] = []
    write_step = np.full(n, -1, np.int64)
    Y = np.zeros((n, dv))
    nch = (n + C - 1) // C
    max_gap = 0.0
    for c in range(nch):
        c0, c1 = c * C, min(n, (c + 1) * C)
        e = c - nwc          # the chunk that leaves the window as chunk c begins
        if e >= 0:
            E = list(cache) + list(range(e * C, (e + 1) * C))
            if len(E) <= lam:
                cache = E
            else:
                sq = {j: sre_sq(H, s, PK[j], v[j]) for j in E}
                order = sorted(E, key=lambda j: (sq[j], j))
                written, kept = order[:len(E) - lam], order[len(E) - lam:]
                if replay is not None:
                    written = [j for j in order if replay[j] == c0]   # added in (SRE, position) order
                    kept = [j for j in order if replay[j] != c0]
                    if len(written) != len(E) - lam:
                        raise ValueError(f"replay writes {len(written)} keys at {c0}, {len(E) - lam} are due")
                    for w in written:
                        for kp in kept:
                            if (sq[w], w) > (sq[kp], kp):
                                sw, sk = math.sqrt(sq[w]), math.sqrt(sq[kp])
                                max_gap = max(max_gap, (sw - sk) / sk if sk > 0 else math.inf)
                if trace is not None:
                    trace.append((c0, sq, written, kept))
                for j in written:
                    H += np.outer(PK[j], v[j])
                    s += PK[j]
                    write_step[j] = c0
                cache = sorted(kept)
        w0 = max(0, (c - nwc + 1) * C)
        for t in range(c0, c1):
            exact = list(range(w0, t + 1)) + cache
            Y[t] = _output(q[t], PQ[t], exact, k, v, H.T @ PQ[t], float(PQ[t] @ s), scale)
    win = list(range(max(0, (nch - nwc) * C), n)) if nch else []
    if replay is not None and not np.array_equal(np.asarray(replay), write_step):
        raise ValueError("replay writes a key that is not a candidate when it says")
    return dict(Y=Y, write_step=write_step, H=H, s=s, cache=np.array(sorted(cache), np.int64),
                window=np.array(win, np.int64), max_gap=max_gap)


def window_chunks_plus_linear(q, k, v, W, eta: int, C: int):
    """lambda = 0 in chunk mode: a query of chunk c reads softmax over its window chunks
    (chunks c - eta/C + 1 .. c, up to itself) and the linear state over every token
    before them, one shared denominator."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    n = q.shape[0]
    PQ, PK = phi(q, W), phi(k, W)
    t = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    wstart = np.maximum(0, (t // C - eta // C + 1) * C)
    in_win = (j <= t) & (j >= wstart)
    in_state = j < wstart
    a = (q @ k.T) / math.sqrt(q.shape[1])
    m = np.where(in_win, a, -np.inf).max(axis=1, keepdims=True)
    ws = np.where(in_win, np.exp(np.where(in_win, a, 0.0) - m), 0.0)
    wl = np.where(in_state, PQ @ PK.T, 0.0) * np.exp(-m)
    wt = ws + wl
    return (wt @ v) / wt.sum(axis=1, keepdims=True)


def sre_map(k, v, W, write_step, times):
    """Self-recall error of every key held by the linear memory at each state time (the
    notes' Fig. 3 diagnostic, section 4.4): out[c, j] = SRE(k_j, v_j | H_t, s_t) for
    t = times[c], where (H_t, s_t) is the memory before step t -- the sums of phi(k) v^T and
    phi(k) over the keys written before t (write_step[j] < t) -- and 0 for keys it does not
    hold (still exact in the window or cache, or not yet seen)."""
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    PK = phi(k, W)
    ws = np.asarray(write_step)
    out = np.zeros((len(times), k.shape[0]))
    for c, t in enumerate(times):
        held = np.flatnonzero((ws >= 0) & (ws < t))
        if held.size == 0:
            continue
        H = PK[held].T @ v[held]
        s = PK[held].sum(axis=0)
        for j in held:
            out[c, j] = math.sqrt(sre_sq(H, s, PK[j], v[j]))
    return out


def sre_at_first_write(k, v, W, write_step):
    """SRE of every written key against the first memory that holds it (the notes' appendix
    G, Eq. 26 baseline): the sums over the keys written at or before its own write step
    (write_step[i] <= write_step[j]; with chunk-granular allocation that includes the keys
    written at the same chunk start).  0 for keys never written."""
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    PK = phi(k, W)
    ws = np.asarray(write_step)
    out = np.zeros(k.shape[0])
    for w in np.unique(ws[ws >= 0]):
        held = np.flatnonzero((ws >= 0) & (ws <= w))
        H = PK[held].T @ v[held]
        s = PK[held].sum(axis=0)
        for j in np.flatnonzero(ws == w):
            out[j] = math.sqrt(sre_sq(H, s, PK[j], v[j]))
    return out


def sre_map_relative(k, v, W, write_step, times):
    """The relative SRE map (the notes' appendix G, Fig. 10, Eq. 26): for every key held by
    the memory at state time t = times[c], its SRE now minus its SRE at first write (a
    difference, not a ratio); 0 for keys the memory does not hold."""
    m = sre_map(k, v, W, write_step, times)
    base = sre_at_first_write(k, v, W, write_step)
    ws = np.asarray(write_step)
    out = np.zeros_like(m)
    for c, t in enumerate(times):
        held = (ws >= 0) & (ws < t)
        out[c, held] = m[c, held] - base[held]
    return out


# ---------------------------------------------------------------------------
# Closed forms the method reduces to (used as pins)
# ---------------------------------------------------------------------------

def causal_softmax_attention(q, k, v):
    """Textbook causal softmax attention, ``softmax(q k^T / sqrt(d_k))`` over j <= t."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    n = q.shape[0]
    a = (q @ k.T) / math.sqrt(q.shape[1])
    a = np.where(np.tril(np.ones((n, n), bool)), a, -np.inf)
    p = np.exp(a - a.max(axis=1, keepdims=True))
    return (p / p.sum(axis=1, keepdims=True)) @ v


def sliding_window_attention(q, k, v, eta: int):
    """Causal softmax attention restricted to the last eta tokens (inclusive):
    ``softmax(q k^T / sqrt(d_k))`` over t - eta < j <= t."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    n = q.shape[0]
    t = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    a = (q @ k.T) / math.sqrt(q.shape[1])
    a = np.where((j <= t) & (j > t - eta), a, -np.inf)
    p = np.exp(a - a.max(axis=1, keepdims=True))
    return (p / p.sum(axis=1, keepdims=True)) @ v


def linear_attention(q, k, v, W):
    """Causal linear attention with the inclusive recurrence of section 2.2 (Eqs. 3-5):
    ``y_t = sum_{j<=t} (phi_q . phi_j) v_j / sum_{j<=t} phi_q . phi_j``."""
    PQ, PK = phi(q, W), phi(k, W)
    A = np.tril(PQ @ PK.T)
    return (A @ np.asarray(v, np.float64)) / A.sum(axis=1, keepdims=True)


def window_plus_linear(q, k, v, W, eta: int):
    """lambda = 0: softmax over the last eta tokens (inclusive) and the linear state over
    every token <= t - eta, one shared denominator (the LoLCATs base, section 3.1)."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    n = q.shape[0]
    PQ, PK = phi(q, W), phi(k, W)
    t = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    in_win = (j <= t) & (j > t - eta)
    in_state = j <= t - eta
    a = (q @ k.T) / math.sqrt(q.shape[1])
    m = np.where(in_win, a, -np.inf).max(axis=1, keepdims=True)
    m = np.where(np.isfinite(m), m, 0.0)
    ws = np.where(in_win, np.exp(np.where(in_win, a, 0.0) - m), 0.0)
    wl = np.where(in_state, PQ @ PK.T, 0.0) * np.exp(-m)
    wt = ws + wl
    return (wt @ v) / wt.sum(axis=1, keepdims=True)


def state_elements(t: int, dk: int, dv: int, D: int, eta: int, lam: int) -> int:
    """Per-head element count of the persistent memory (appendix B):
    ``min{t (d_k + d_v), (eta + lambda)(d_k + d_v) + D d_v + D}``."""
    return min(t * (dk + dv), (eta + lam) * (dk + dv) + D * dv + D)
