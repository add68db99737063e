"""lola_prefill_noalloc: the prefill for callers that cannot allocate device memory when
they call in (a host runtime that owns the allocator, or a path that must not call
cudaMalloc/cudaFree because those can synchronise the device).  Its scratch is the
library's fixed device array, so it must give the same results as lola_prefill with a
caller-provided workspace, call after call, whatever the previous call left in the array.

This file is named to be collected last."""
import ctypes

import numpy as np
import pytest
import torch

import synth

from lola_parity import TOL, check_outputs, to_dev, to_f64


def _lib():
    import sparse_exact_kv_gb300 as L
    return L


def _run(L, x, eta, lam, chunk, noalloc):
    w = x.w
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    cfg = L.make_config(w.B, w.Hh, w.d, w.d, w.D, eta, lam, chunk, dt)
    n = x.q.shape[2]
    Q, K, V = (to_dev(getattr(x, a), "cuda", w.dtype) for a in "qkv")
    W = torch.from_numpy(x.W).cuda()
    Y = torch.empty_like(V)
    state = torch.empty(L.lola_state_bytes(cfg), dtype=torch.uint8, device="cuda")
    wpos = torch.empty(w.B, w.Hh, n, dtype=torch.int32, device="cuda")
    if noalloc:
        L.lola_prefill_noalloc(cfg, n, Q, K, V, W, 0, Y, state, wpos)
    else:
        ws = torch.empty(L.lola_prefill_workspace_bytes(cfg, n), dtype=torch.uint8, device="cuda")
        L.lola_prefill(cfg, n, Q, K, V, W, 0, Y, state, wpos, ws)
    torch.cuda.synchronize()
    return to_f64(Y), wpos.cpu().numpy(), state.cpu().numpy()


@pytest.mark.gpu
def test_noalloc_prefill_matches_workspace_prefill_on_consecutive_calls():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L = _lib()
    cases = [
        (synth.gauss_inputs(1, 3, 700, 128, 128, "bf16", seed=41), 32, 48, 64),
        (synth.gauss_inputs(2, 2, 500, 64, 64, "f32", seed=42), 16, 24, 32),
    ]
    first = None
    for x, eta, lam, chunk in cases:       # two noalloc calls in a row, different shapes
        Yr, wr, sr = _run(L, x, eta, lam, chunk, noalloc=False)
        Yn, wn, sn = _run(L, x, eta, lam, chunk, noalloc=True)
        assert np.array_equal(wn, wr)
        check_outputs(Yn, Yr, x.w.dtype, what="noalloc Y")
        np.testing.assert_array_equal(sn, sr)
        if first is None:
            first = (Yn, wn, sn)
    # the first case again, straight after the second: whatever the array still holds from
    # the earlier calls must not change a bit of the result
    x, eta, lam, chunk = cases[0]
    Y3, w3, s3 = _run(L, x, eta, lam, chunk, noalloc=True)
    Y4, w4, s4 = _run(L, x, eta, lam, chunk, noalloc=True)
    for got in ((Y3, w3, s3), (Y4, w4, s4)):
        for a, b in zip(got, first):
            np.testing.assert_array_equal(a, b)


def test_noalloc_rejects_problems_beyond_its_array():
    """Sizes whose scratch exceeds the fixed array are refused before anything runs."""
    L = _lib()
    cfg = L.make_config(4, 32, 128, 128, 128, 64, 64, 64, "bf16")
    n = 4096
    assert L.lola_prefill_workspace_bytes(cfg, n) > L.LOLA_NOALLOC_SCRATCH_BYTES
    P = ctypes.c_void_p(256)
    st = L._lib.lola_prefill_noalloc(ctypes.byref(cfg), n, P, P, P, P, 0, P, P, None, None)
    assert st == L.LOLA_ERR_WORKSPACE
