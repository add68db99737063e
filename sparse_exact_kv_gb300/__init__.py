"""Python binding of liblola.so, the GB300 LoLA hybrid-attention library.

Argument marshalling only: every step of the method runs in the library's CUDA kernels.
The functions carry the C ABI's names (include/lola.h) and take torch tensors for the
device buffers; torch provides device memory and streams, nothing else.

If the shared library is missing or fails to load, importing this package raises: there
is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "liblola.so")

LOLA_OK = 0
LOLA_ERR_INVALID_ARG = -1
LOLA_ERR_UNSUPPORTED = -2
LOLA_ERR_WORKSPACE = -3
LOLA_ERR_CUDA = -4
LOLA_ERR_DEVICE = -5
LOLA_F32 = 0
LOLA_BF16 = 1
LOLA_READ_HIDE_STATE = 1
LOLA_READ_HIDE_CACHE = 2
LOLA_ALLOC_TOKEN = 0
LOLA_ALLOC_CHUNK = 1
LOLA_SCORE_SRE = 0
LOLA_SCORE_KERNEL_SQ = 1
LOLA_SCORE_KERNEL_ABS = 2
LOLA_SCORE_KERNEL_RATIO = 3
LOLA_SCORE_ATTENTION = 4
SCORES = {"sre": 0, "kernel_sq": 1, "kernel_abs": 2, "kernel_ratio": 3, "attention": 4}

# every symbol include/lola.h declares
EXPORTS = ("lola_version", "lola_status_string", "lola_last_cuda_error", "lola_check_config",
           "lola_state_layout_of", "lola_state_bytes", "lola_prefill_workspace_bytes", "lola_state_init",
           "lola_prefill", "lola_decode_step", "lola_read_status", "lola_kernel_timing", "lola_kernel_time",
           "lola_kernel_name", "lola_prefill_noalloc", "lola_selftest_bounded_wait", "lola_sre_map",
           "lola_sre_map_relative", "lola_hola_workspace_bytes", "lola_hola_prefill", "lola_hola_status")
# size of the fixed scratch array behind lola_prefill_noalloc (include/lola.h)
LOLA_NOALLOC_SCRATCH_BYTES = 32 << 20
KERNELS = ("state_init", "phi", "select", "output", "decode", "phi_q", "hola_prep", "hola_state", "hola_cache",
           "hola_read")


class lola_config(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("Hh", ctypes.c_int32), ("d_k", ctypes.c_int32),
                ("d_v", ctypes.c_int32), ("D", ctypes.c_int32), ("eta", ctypes.c_int32),
                ("lambda_", ctypes.c_int32), ("chunk", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("read_mask", ctypes.c_int32), ("alloc", ctypes.c_int32), ("score", ctypes.c_int32)]


class lola_hola_config(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("Hh", ctypes.c_int32), ("d_k", ctypes.c_int32), ("d_v", ctypes.c_int32),
                ("w", ctypes.c_int32), ("chunk", ctypes.c_int32), ("dtype", ctypes.c_int32)]


class lola_state_layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in
                ("head_bytes", "H", "s", "win_pos", "win_k", "win_v", "win_phi", "c_pos", "c_k", "c_v", "c_phi",
                 "c_N", "c_z", "ev", "tok_phi")]


class LolaError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = _lib.lola_status_string(status).decode()
        if status == LOLA_ERR_CUDA:
            msg += ": " + _lib.lola_last_cuda_error().decode()
        super().__init__(f"{where}: {msg} ({status})")
        self.status = status


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                          "(or python -m sparse_exact_kv_gb300._build)")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.c_void_p
    C = ctypes.POINTER(lola_config)
    HC = ctypes.POINTER(lola_hola_config)
    sig = {
        "lola_version": ([], ctypes.c_int32),
        "lola_status_string": ([ctypes.c_int32], ctypes.c_char_p),
        "lola_last_cuda_error": ([], ctypes.c_char_p),
        "lola_check_config": ([C], ctypes.c_int32),
        "lola_state_layout_of": ([C, ctypes.POINTER(lola_state_layout)], ctypes.c_int32),
        "lola_state_bytes": ([C], ctypes.c_size_t),
        "lola_prefill_workspace_bytes": ([C, ctypes.c_int32], ctypes.c_size_t),
        "lola_state_init": ([C, P, P], ctypes.c_int32),
        "lola_prefill": ([C, ctypes.c_int32, P, P, P, P, ctypes.c_int64, P, P, P, P, ctypes.c_size_t, P],
                         ctypes.c_int32),
        "lola_decode_step": ([C, P, P, ctypes.c_int64, P, P, P, P, P, P], ctypes.c_int32),
        "lola_read_status": ([C, P, P, P], ctypes.c_int32),
        "lola_kernel_timing": ([ctypes.c_int32], ctypes.c_int32),
        "lola_kernel_time": ([ctypes.c_int32, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64)],
                             ctypes.c_int32),
        "lola_kernel_name": ([ctypes.c_int32], ctypes.c_char_p),
        "lola_prefill_noalloc": ([C, ctypes.c_int32, P, P, P, P, ctypes.c_int64, P, P, P, P], ctypes.c_int32),
        "lola_selftest_bounded_wait": ([ctypes.c_int64, ctypes.POINTER(ctypes.c_int64), P], ctypes.c_int32),
        "lola_sre_map": ([C, ctypes.c_int32, P, P, ctypes.c_size_t, P, P], ctypes.c_int32),
        "lola_sre_map_relative": ([C, ctypes.c_int32, P, P, ctypes.c_size_t, P, P, P], ctypes.c_int32),
        "lola_hola_workspace_bytes": ([HC, ctypes.c_int32], ctypes.c_int64),
        "lola_hola_prefill": ([HC, ctypes.c_int32] + [P] * 14 + [ctypes.c_size_t, P], ctypes.c_int32),
        "lola_hola_status": ([HC, ctypes.c_int32, P, P, P], ctypes.c_int32),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    return lib


_lib = _load()


def make_config(B, Hh, d_k, d_v, D, eta, lam, chunk, dtype, read_mask=0, alloc=LOLA_ALLOC_TOKEN,
                score=LOLA_SCORE_SRE) -> lola_config:
    """``read_mask``: LOLA_READ_HIDE_STATE | LOLA_READ_HIDE_CACHE, memories left out of every
    query's read (the memory and the decisions are unchanged).  ``alloc``: LOLA_ALLOC_TOKEN
    (the per-token rule) or LOLA_ALLOC_CHUNK (chunk-granular allocation).  ``score``:
    LOLA_SCORE_SRE (the self-recall error) or one of the query-dependent scores of the scoring
    ablation (a LOLA_SCORE_* value or its name in SCORES)."""
    dt = dtype if isinstance(dtype, int) else {"f32": LOLA_F32, "bf16": LOLA_BF16,
                                               torch.float32: LOLA_F32, torch.bfloat16: LOLA_BF16}[dtype]
    sc = SCORES[score] if isinstance(score, str) else int(score)
    return lola_config(B, Hh, d_k, d_v, D, eta, lam, chunk, dt, read_mask, alloc, sc)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if isinstance(stream, int):          # a raw cudaStream_t (0: the legacy default stream)
        return ctypes.c_void_p(stream)
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status, where):
    if status != LOLA_OK:
        raise LolaError(status, where)


def lola_version() -> int:
    return _lib.lola_version()


def lola_status_string(status: int) -> str:
    return _lib.lola_status_string(status).decode()


def lola_check_config(cfg: lola_config) -> int:
    return _lib.lola_check_config(ctypes.byref(cfg))


def lola_state_layout_of(cfg: lola_config) -> lola_state_layout:
    out = lola_state_layout()
    _check(_lib.lola_state_layout_of(ctypes.byref(cfg), ctypes.byref(out)), "lola_state_layout_of")
    return out


def lola_state_bytes(cfg: lola_config) -> int:
    return _lib.lola_state_bytes(ctypes.byref(cfg))


def lola_prefill_workspace_bytes(cfg: lola_config, n: int) -> int:
    return _lib.lola_prefill_workspace_bytes(ctypes.byref(cfg), n)


def lola_state_init(cfg: lola_config, state: torch.Tensor, stream=None) -> None:
    _check(_lib.lola_state_init(ctypes.byref(cfg), _ptr(state), _stream(stream)), "lola_state_init")


def lola_prefill(cfg: lola_config, n: int, Q, K, V, W, w_head_stride: int, Y, state, write_pos, workspace,
                 stream=None) -> None:
    """Enqueue lola_prefill on ``stream`` (default: torch's current stream)."""
    _check(_lib.lola_prefill(ctypes.byref(cfg), n, _ptr(Q), _ptr(K), _ptr(V), _ptr(W), w_head_stride, _ptr(Y),
                             _ptr(state), _ptr(write_pos), _ptr(workspace),
                             workspace.numel() * workspace.element_size(), _stream(stream)), "lola_prefill")


def lola_prefill_noalloc(cfg: lola_config, n: int, Q, K, V, W, w_head_stride: int, Y, state, write_pos=None,
                         stream=None) -> None:
    """lola_prefill without a workspace: its scratch is the library's fixed device array
    (LOLA_NOALLOC_SCRATCH_BYTES), for callers that cannot allocate device memory."""
    _check(_lib.lola_prefill_noalloc(ctypes.byref(cfg), n, _ptr(Q), _ptr(K), _ptr(V), _ptr(W), w_head_stride,
                                     _ptr(Y), _ptr(state), _ptr(write_pos), _stream(stream)),
           "lola_prefill_noalloc")


def lola_decode_step(cfg: lola_config, state, W, w_head_stride: int, q, k, v, y, written_pos=None,
                     stream=None) -> None:
    _check(_lib.lola_decode_step(ctypes.byref(cfg), _ptr(state), _ptr(W), w_head_stride, _ptr(q), _ptr(k),
                                 _ptr(v), _ptr(y), _ptr(written_pos), _stream(stream)), "lola_decode_step")


def lola_read_status(cfg: lola_config, state, stream=None):
    """Synchronises the stream and returns (status, per-head status words as a list)."""
    BH = cfg.B * cfg.Hh
    buf = (ctypes.c_int32 * BH)()
    st = _lib.lola_read_status(ctypes.byref(cfg), _ptr(state), buf, _stream(stream))
    return st, list(buf)


def lola_kernel_timing(enable: bool) -> None:
    _check(_lib.lola_kernel_timing(1 if enable else 0), "lola_kernel_timing")


def lola_kernel_time(kernel) -> tuple[float, int]:
    """(total device ms, launches) of a kernel id or name since timing was enabled."""
    kid = KERNELS.index(kernel) if isinstance(kernel, str) else int(kernel)
    ms, cnt = ctypes.c_double(), ctypes.c_int64()
    _check(_lib.lola_kernel_time(kid, ctypes.byref(ms), ctypes.byref(cnt)), "lola_kernel_time")
    return ms.value, cnt.value


def lola_kernel_name(kid: int) -> str:
    return _lib.lola_kernel_name(kid).decode()


def lola_sre_map(cfg: lola_config, n: int, V, workspace, out, stream=None) -> None:
    """SRE of every key held by each snapshot of the last prefill in ``workspace`` (section
    4.4): ``out`` float32 [B, Hh, nck, n]."""
    _check(_lib.lola_sre_map(ctypes.byref(cfg), n, _ptr(V), _ptr(workspace), workspace.numel() * workspace.element_size(),
                             _ptr(out), _stream(stream)), "lola_sre_map")


def lola_sre_map_relative(cfg: lola_config, n: int, V, workspace, out, base, stream=None) -> None:
    """The relative SRE map (appendix G, Eq. 26): ``out`` float32 [B, Hh, nck, n] = the map
    minus each held key's SRE at first write, ``base`` float32 [B, Hh, n] = that SRE."""
    _check(_lib.lola_sre_map_relative(ctypes.byref(cfg), n, _ptr(V), _ptr(workspace),
                                      workspace.numel() * workspace.element_size(), _ptr(out), _ptr(base),
                                      _stream(stream)), "lola_sre_map_relative")


def lola_selftest_bounded_wait(limit_ns: int, stream=None):
    """Runs the kernels' bounded mbarrier wait on a barrier nothing completes; returns
    (status, nanoseconds waited): LOLA_ERR_DEVICE when the wait gave up as designed."""
    ns = ctypes.c_int64(0)
    st = _lib.lola_selftest_bounded_wait(int(limit_ns), ctypes.byref(ns), _stream(stream))
    return st, ns.value


# ---------------------------------------------------------------------------------------
# The write-magnitude exact cache on a gated delta-rule state (include/lola.h)
# ---------------------------------------------------------------------------------------

def make_hola_config(B, Hh, d, w, chunk, dtype=LOLA_BF16) -> lola_hola_config:
    return lola_hola_config(B, Hh, d, d, w, chunk, dtype)


def lola_hola_workspace_bytes(cfg: lola_hola_config, n: int) -> int:
    b = _lib.lola_hola_workspace_bytes(ctypes.byref(cfg), n)
    if b < 0:
        raise LolaError(int(b), "lola_hola_workspace_bytes")
    return int(b)


def lola_hola_prefill(cfg: lola_hola_config, n: int, Q, K, V, alpha, beta, gamma_q, gamma_k, sink, gate, Y,
                      workspace, S_out=None, scores=None, cache=None, stream=None) -> None:
    _check(_lib.lola_hola_prefill(ctypes.byref(cfg), n, _ptr(Q), _ptr(K), _ptr(V), _ptr(alpha), _ptr(beta),
                                  _ptr(gamma_q), _ptr(gamma_k), _ptr(sink), _ptr(gate), _ptr(Y), _ptr(S_out),
                                  _ptr(scores), _ptr(cache), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream)),
           "lola_hola_prefill")


def lola_hola_status(cfg: lola_hola_config, n: int, workspace, stream=None):
    """Synchronises the stream and returns (status, per-head status words as a list)."""
    buf = (ctypes.c_int32 * (cfg.B * cfg.Hh))()
    st = _lib.lola_hola_status(ctypes.byref(cfg), n, _ptr(workspace), buf, _stream(stream))
    return st, list(buf)


# ---------------------------------------------------------------------------------------
# Convenience: buffers allocated through torch, then the C ABI
# ---------------------------------------------------------------------------------------

class Lola:
    """One layer's LoLA memory for B x Hh heads: owns the state and the prefill workspace."""

    def __init__(self, B, Hh, d, D, eta, lam, chunk=64, dtype=torch.bfloat16, device="cuda", read_mask=0,
                 alloc=LOLA_ALLOC_TOKEN, score=LOLA_SCORE_SRE):
        self.cfg = make_config(B, Hh, d, d, D, eta, lam, chunk, dtype, read_mask, alloc, score)
        _check(lola_check_config(self.cfg), "config")
        self.dtype = dtype
        self.device = torch.device(device)
        self.state = torch.empty(lola_state_bytes(self.cfg), dtype=torch.uint8, device=self.device)
        self.workspace = None
        lola_state_init(self.cfg, self.state)

    def layout(self) -> lola_state_layout:
        return lola_state_layout_of(self.cfg)

    def workspace_for(self, n: int) -> torch.Tensor:
        need = lola_prefill_workspace_bytes(self.cfg, n)
        if self.workspace is None or self.workspace.numel() < need:
            self.workspace = torch.empty(need, dtype=torch.uint8, device=self.device)
        return self.workspace

    def prefill(self, Q, K, V, W, Y=None, write_pos=None, stream=None):
        """Q, K, V: [B, Hh, n, d] device tensors of the config's dtype; W: [D/2, d] float32."""
        n = Q.shape[2]
        if Y is None:
            Y = torch.empty_like(V)
        ws = self.workspace_for(n)
        lola_prefill(self.cfg, n, Q, K, V, W, 0, Y, self.state, write_pos, ws, stream)
        return Y

    def decode_step(self, q, k, v, W, y=None, written_pos=None, stream=None):
        """q, k, v: [B, Hh, d] device tensors; returns y [B, Hh, d]."""
        if y is None:
            y = torch.empty_like(v)
        lola_decode_step(self.cfg, self.state, W, 0, q, k, v, y, written_pos, stream)
        return y

    def read_state(self):
        """Host copies of every head's memory: dict of numpy arrays (H, s, window, cache)."""
        import numpy as np
        L = self.layout()
        c = self.cfg
        raw = self.state.view(c.B * c.Hh, L.head_bytes).cpu().numpy()
        io = np.uint16 if c.dtype == LOLA_BF16 else np.float32
        isz = 2 if c.dtype == LOLA_BF16 else 4

        def f(off, count, dt, size):
            return np.ascontiguousarray(raw[:, off: off + count * size]).view(dt)

        BH = c.B * c.Hh
        hdr = f(0, 16, np.int32, 4)
        return dict(t=hdr[:, 0], n_cache=hdr[:, 1], n_written=hdr[:, 2], status=hdr[:, 3],
                    H=f(L.H, c.D * c.d_v, np.float32, 4).reshape(BH, c.D, c.d_v),
                    s=f(L.s, c.D, np.float32, 4),
                    win_pos=f(L.win_pos, c.eta, np.int32, 4),
                    win_k=f(L.win_k, c.eta * c.d_k, io, isz).reshape(BH, c.eta, c.d_k),
                    win_v=f(L.win_v, c.eta * c.d_v, io, isz).reshape(BH, c.eta, c.d_v),
                    win_phi=f(L.win_phi, c.eta * c.D, np.float32, 4).reshape(BH, c.eta, c.D),
                    c_pos=f(L.c_pos, c.lambda_, np.int32, 4),
                    c_k=f(L.c_k, c.lambda_ * c.d_k, io, isz).reshape(BH, c.lambda_, c.d_k),
                    c_v=f(L.c_v, c.lambda_ * c.d_v, io, isz).reshape(BH, c.lambda_, c.d_v),
                    c_phi=f(L.c_phi, c.lambda_ * c.D, np.float32, 4).reshape(BH, c.lambda_, c.D),
                    c_N=f(L.c_N, c.lambda_ * c.d_v, np.float32, 4).reshape(BH, c.lambda_, c.d_v),
                    c_z=f(L.c_z, c.lambda_, np.float32, 4),
                    ev=f(L.ev, c.d_v + 1, np.float32, 4))
