"""Seeded synthetic inputs for the LoLA hot path.

This module only draws numbers: it holds none of the method's arithmetic. Both
the CPU oracle (through the tests and the benchmark) and the CUDA library are
fed from it, so both sides see bit-identical inputs.

Generator: a counter-based SplitMix64 stream (Steele, Lea and Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014) turned into standard
normals by the Box-Muller transform.  Value ``i`` of stream ``(seed, stream)``
depends only on those three integers, so any slice can be regenerated alone.

Workload recipes follow the five workload descriptions of the LoLA hot path:
Gaussian Q/K/V with an optional row normalisation of K (workload 2), planted
high-norm "needle" keys (workload 3), a random prefix followed by single-token
decode steps (workload 4) and per-channel AR(1) sequences (workload 5).  The
feature-map weight W is Gaussian with variance 1/64 in every workload.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function applied elementwise (uint64, wrapping)."""
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _stream_key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        base = np.array([(seed * 0x100000001B3 + stream * 0x5851F42D4C957F2D) & 0xFFFFFFFFFFFFFFFF],
                        dtype=np.uint64)
        return _mix(base + _GOLDEN)[0]


def uniform_bits(seed: int, stream: int, count: int, offset: int = 0) -> np.ndarray:
    """``count`` uint64 words of stream (seed, stream), starting at word ``offset``."""
    key = _stream_key(seed, stream)
    with np.errstate(over="ignore"):
        ctr = np.arange(offset + 1, offset + count + 1, dtype=np.uint64) * _GOLDEN + key
        return _mix(ctr)


def normal_reference(seed: int, stream: int, count: int) -> np.ndarray:
    """Readable numpy statement of the normal stream (float64): pair p takes words
    2p and 2p+1; u1 = (w >> 11 + 1) 2^-53 in (0, 1], u2 = (w >> 11) 2^-53, and
    z = sqrt(-2 ln u1) (cos, sin)(2 pi u2).  The C library computes the same
    values; this function is the definition it is tested against."""
    npairs = (count + 1) // 2
    bits = uniform_bits(seed, stream, 2 * npairs)
    u1 = ((bits[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
    u2 = (bits[1::2] >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    r = np.sqrt(-2.0 * np.log(u1))
    out = np.empty(2 * npairs, dtype=np.float64)
    out[0::2] = r * np.cos(2.0 * math.pi * u2)
    out[1::2] = r * np.sin(2.0 * math.pi * u2)
    return out[:count]


_LIB = None


def _lib():
    """Load (building on first use) the C generator next to this file."""
    global _LIB
    if _LIB is not None:
        return _LIB
    import ctypes
    import os
    import subprocess

    here = os.path.dirname(os.path.abspath(__file__))
    src = os.path.join(here, "synth_gen.c")
    so = os.path.join(here, "libsynth_gen.so")
    if not os.path.exists(so) or os.path.getmtime(so) < os.path.getmtime(src):
        tmp = so + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-shared", "-fPIC", "-pthread", src, "-o", tmp, "-lm"])
        os.replace(tmp, so)
    lib = ctypes.CDLL(so)
    lib.synth_normal.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64, ctypes.c_double,
                                 ctypes.c_int, ctypes.c_void_p, ctypes.c_int]
    lib.synth_normal.restype = None
    lib.synth_word.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64]
    lib.synth_word.restype = ctypes.c_uint64
    lib.synth_to_bf16.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
    lib.synth_to_bf16.restype = None
    lib.synth_ar1.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64, ctypes.c_int64,
                              ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int]
    lib.synth_ar1.restype = None
    _LIB = lib
    return lib


def _threads() -> int:
    import os
    return min(64, os.cpu_count() or 1)


def normal(seed: int, stream: int, count: int, scale: float = 1.0, out: str = "f64") -> np.ndarray:
    """``count`` values ``scale * N(0,1)`` of stream (seed, stream).

    ``out`` selects float64 ("f64"), float32 ("f32") or bf16 words ("bf16", uint16).
    """
    mode, dt = {"f64": (0, np.float64), "f32": (1, np.float32), "bf16": (2, np.uint16)}[out]
    a = np.empty(count, dtype=dt)
    _lib().synth_normal(seed, stream, count, scale, mode, a.ctypes.data, _threads())
    return a


# ---------------------------------------------------------------------------
# bf16 helpers (numpy has no bf16 type: bf16 values travel as uint16 words)
# ---------------------------------------------------------------------------

def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); returns uint16 words."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(f.shape, dtype=np.uint16)
    _lib().synth_to_bf16(f.ctypes.data, out.ctypes.data, f.size)
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 words to float32 (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ---------------------------------------------------------------------------
# Workloads
# ---------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hh: int
    n: int          # prefill length (workload 4: prefix length)
    d: int          # d_k = d_v
    D: int          # feature dimension (W has D/2 rows)
    eta: int
    lam: int
    chunk: int
    dtype: str      # "f32" or "bf16": storage type of Q, K, V and Y
    kind: str       # "gauss", "gauss_knorm", "needle", "decode", "ar1"
    decode_steps: int = 0
    seed: int = 0


WORKLOADS = {
    # 1 sequence, 1 head, fp32 inputs: the small fp32 case.
    "w1_f32_n1024": Workload("w1_f32_n1024", 1, 1, 1024, 64, 64, 64, 64, 64, "f32", "gauss"),
    # 4 x 32 heads, n = 4096, bf16, K rows normalised to norm sqrt(d).
    "w2_bf16_b4h32_n4096": Workload("w2_bf16_b4h32_n4096", 4, 32, 4096, 128, 128, 64, 64, 64,
                                    "bf16", "gauss_knorm"),
    # 1 x 32 heads, n = 16384, every 512th key scaled by 4.
    "w3_bf16_h32_n16384_needle": Workload("w3_bf16_h32_n16384_needle", 1, 32, 16384, 128, 128,
                                          256, 256, 128, "bf16", "needle"),
    # decode: 64 x 32 heads, 4096-token random prefix then 1024 single-token steps.
    "w4_bf16_decode_b64h32": Workload("w4_bf16_decode_b64h32", 64, 32, 4096, 128, 128, 64, 64, 64,
                                      "bf16", "decode", decode_steps=1024),
    # long prefill: 1 x 8 heads, n = 131072, AR(1) rho = 0.9 per channel.
    "w5_bf16_h8_n131072_ar1": Workload("w5_bf16_h8_n131072_ar1", 1, 8, 131072, 128, 128, 512, 512,
                                       256, "bf16", "ar1"),
}

# stream ids: one per tensor
_S_W, _S_Q, _S_K, _S_V = 1, 2, 3, 4


def feature_weight(seed: int, D: int, d: int) -> np.ndarray:
    """W in R^{(D/2) x d}, entries N(0, 1/64), float32."""
    return (normal(seed, _S_W, (D // 2) * d) / 8.0).astype(np.float32).reshape(D // 2, d)


def ar1_reference(seed: int, stream: int, rows: int, n: int, d: int, rho: float = 0.9) -> np.ndarray:
    """Readable statement of the AR(1) recipe (float64): x_0 = e_0 and
    x_t = rho x_{t-1} + sqrt(1-rho^2) e_t per (row, channel), e the normal stream in
    row-major (rows, n, d) order.  Stationary with unit variance."""
    from scipy.signal import lfilter

    e = normal_reference(seed, stream, rows * n * d).reshape(rows, n, d)
    drive = e * math.sqrt(1.0 - rho * rho)
    drive[:, 0, :] = e[:, 0, :]
    return lfilter([1.0], [1.0, -rho], drive, axis=1)


def _ar1(seed: int, stream: int, rows: int, n: int, d: int, rho: float = 0.9) -> np.ndarray:
    """The AR(1) recipe computed by the C library, float32 of shape (rows, n, d)."""
    lib = _lib()
    out = np.empty((rows, n, d), dtype=np.float32)
    lib.synth_ar1(seed, stream, rows, n, d, rho, out.ctypes.data, min(_threads(), rows))
    return out


def _tensor(w: Workload, n_total: int, seed: int, stream: int) -> np.ndarray:
    """One of Q, K, V in its storage type, shape (B, Hh, n_total, d)."""
    rows = w.B * w.Hh
    shape = (w.B, w.Hh, n_total, w.d)
    cnt = rows * n_total * w.d
    if w.kind == "ar1":
        x = _ar1(seed, stream, rows, n_total, w.d).reshape(shape)
    elif stream == _S_K and w.kind == "gauss_knorm":
        x = normal(seed, stream, cnt).reshape(shape)
        x = (x / np.linalg.norm(x, axis=-1, keepdims=True) * math.sqrt(w.d)).astype(np.float32)
    elif stream == _S_K and w.kind == "needle":
        x = normal(seed, stream, cnt, out="f32").reshape(shape)
        needle = ((np.arange(n_total) + 1) % 512) == 0
        x[:, :, needle, :] *= np.float32(4.0)
    else:
        return normal(seed, stream, cnt, out=w.dtype).reshape(shape)
    return to_bf16_bits(x) if w.dtype == "bf16" else x.astype(np.float32)


@dataclasses.dataclass
class Inputs:
    """One workload's inputs.  ``q``, ``k``, ``v`` hold the storage dtype:
    float32 arrays for "f32", uint16 bf16 words for "bf16".  ``W`` is float32."""
    w: Workload
    n_total: int
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    W: np.ndarray

    def widened(self, name: str) -> np.ndarray:
        """Exact float64 copy of q, k or v."""
        a = getattr(self, name)
        if self.w.dtype == "bf16":
            return bf16_bits_to_f32(a).astype(np.float64)
        return a.astype(np.float64)


def make_inputs(w: Workload, n: int | None = None, B: int | None = None, Hh: int | None = None,
                seed: int | None = None) -> Inputs:
    """Generate a workload's inputs, optionally at reduced (n, B, Hh) for small cases.

    For the decode workload the sequence holds the prefix followed by the decode tokens.
    """
    if n is not None or B is not None or Hh is not None:
        w = dataclasses.replace(w, n=n if n is not None else w.n, B=B if B is not None else w.B,
                                Hh=Hh if Hh is not None else w.Hh)
    seed = w.seed if seed is None else seed
    n_total = w.n + w.decode_steps
    q, k, v = (_tensor(w, n_total, seed, s) for s in (_S_Q, _S_K, _S_V))
    W = feature_weight(seed, w.D, w.d)
    return Inputs(w, n_total, q, k, v, W)


def gauss_inputs(B: int, Hh: int, n: int, d: int, D: int, dtype: str = "f32", seed: int = 0,
                 dv: int | None = None) -> Inputs:
    """Plain N(0,1) inputs of any small shape (tests).  ``dv`` defaults to d."""
    dv = d if dv is None else dv
    w = Workload(f"gauss_{B}x{Hh}x{n}", B, Hh, n, d, D, 0, 0, 1, dtype, "gauss", seed=seed)
    q = normal(seed, _S_Q, B * Hh * n * d, out=dtype).reshape(B, Hh, n, d)
    k = normal(seed, _S_K, B * Hh * n * d, out=dtype).reshape(B, Hh, n, d)
    v = normal(seed, _S_V, B * Hh * n * dv, out=dtype).reshape(B, Hh, n, dv)
    W = feature_weight(seed, D, d)
    return Inputs(w, n, q, k, v, W)


# ---------------------------------------------------------------------------
# The write-magnitude cache on a gated delta-rule state: per-token gates and the
# cache path's scales, drawn like every other input
# ---------------------------------------------------------------------------

_S_ALPHA, _S_BETA, _S_GQ, _S_GK, _S_SINK, _S_GATE = 5, 6, 7, 8, 9, 10


def uniform(seed: int, stream: int, count: int) -> np.ndarray:
    """``count`` values uniform in [0, 1) of stream (seed, stream): (word >> 11) 2^-53, float64."""
    return (uniform_bits(seed, stream, count) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


@dataclasses.dataclass
class HolaInputs:
    """Inputs of one delta-rule-state layer with a write-magnitude cache.  ``q``, ``k``, ``v``
    hold the storage dtype (as in ``Inputs``); the gates and scales are float32:
    ``alpha`` (decay) in (0.9, 1] and ``beta`` (write strength) in [0, 1) per (b, h, t),
    ``gamma_q``, ``gamma_k`` (cache-path scales, 1 + 0.1 N(0,1)) per channel, ``sink`` (the
    null entry's logit, N(0,1)) and ``gate`` (the cache read's weight, in [0.5, 1.5)) per head."""
    B: int
    Hh: int
    n: int
    d: int
    w: int
    chunk: int
    dtype: str
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    alpha: np.ndarray
    beta: np.ndarray
    gamma_q: np.ndarray
    gamma_k: np.ndarray
    sink: np.ndarray
    gate: np.ndarray

    def widened(self, name: str) -> np.ndarray:
        """Exact float64 copy of q, k or v."""
        a = getattr(self, name)
        if self.dtype == "bf16":
            return bf16_bits_to_f32(a).astype(np.float64)
        return a.astype(np.float64)


def hola_inputs(B: int, Hh: int, n: int, d: int, w: int = 64, chunk: int = 256, dtype: str = "bf16",
                seed: int = 0) -> HolaInputs:
    """Gaussian q, k, v and the gate / scale recipe above (no row normalisation: the layer
    normalises its keys and queries itself)."""
    cnt = B * Hh * n * d
    q = normal(seed, _S_Q, cnt, out=dtype).reshape(B, Hh, n, d)
    k = normal(seed, _S_K, cnt, out=dtype).reshape(B, Hh, n, d)
    v = normal(seed, _S_V, cnt, out=dtype).reshape(B, Hh, n, d)
    alpha = (1.0 - 0.1 * uniform(seed, _S_ALPHA, B * Hh * n)).astype(np.float32).reshape(B, Hh, n)
    beta = uniform(seed, _S_BETA, B * Hh * n).astype(np.float32).reshape(B, Hh, n)
    gamma_q = (1.0 + 0.1 * normal(seed, _S_GQ, d)).astype(np.float32)
    gamma_k = (1.0 + 0.1 * normal(seed, _S_GK, d)).astype(np.float32)
    sink = normal(seed, _S_SINK, Hh).astype(np.float32)
    gate = (0.5 + uniform(seed, _S_GATE, Hh)).astype(np.float32)
    return HolaInputs(B, Hh, n, d, w, chunk, dtype, q, k, v, alpha, beta, gamma_q, gamma_k, sink, gate)


# the write-magnitude cache workload: 4 x 32 heads, n = 4096, d = 128, cache w = 64, chunk 256
HOLA_WORKLOAD = dict(name="hola_bf16_b4h32_n4096", B=4, Hh=32, n=4096, d=128, w=64, chunk=256, dtype="bf16")
