"""Host-side checks of the C ABI (no GPU needed): every symbol include/lola.h declares is
exported by liblola.so, configurations are validated, and the state layout holds the
appendix-B element count of the LoLA reading notes (arXiv 2505.23666v3)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="session")
def lib():
    import __graft_entry__
    __graft_entry__._build_module().build()
    import sparse_exact_kv_gb300 as L
    return L


def _declared():
    src = open(os.path.join(ROOT, "include", "lola.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(lola_\w+)\s*\(", src, flags=re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 11, names
    so = ctypes.CDLL(lib.LIB_PATH)
    for name in names:
        assert hasattr(so, name), f"{name} declared in lola.h but not exported"
    assert sorted(lib.EXPORTS) == names


def test_version_and_status_strings(lib):
    assert lib.lola_version() >= 100
    assert lib.lola_status_string(0) == "ok"
    assert "workspace" in lib.lola_status_string(lib.LOLA_ERR_WORKSPACE)


@pytest.mark.parametrize("bad", [
    dict(B=0), dict(Hh=-1), dict(D=63), dict(eta=-1), dict(lam=-2), dict(chunk=0), dict(dtype=7)])
def test_invalid_configs(lib, bad):
    kw = dict(B=2, Hh=4, d_k=128, d_v=128, D=128, eta=64, lam=64, chunk=64, dtype="bf16")
    kw.update(bad)
    cfg = lib.make_config(kw["B"], kw["Hh"], kw["d_k"], kw["d_v"], kw["D"], kw["eta"], kw["lam"], kw["chunk"],
                          kw["dtype"])
    assert lib.lola_check_config(cfg) == lib.LOLA_ERR_INVALID_ARG
    assert lib.lola_state_bytes(cfg) == 0


@pytest.mark.parametrize("bad", [dict(d_k=96, d_v=96, D=96), dict(D=64), dict(lam=2000), dict(chunk=48),
                                 dict(chunk=512), dict(chunk=8)])
def test_unsupported_configs(lib, bad):
    kw = dict(B=1, Hh=1, d_k=128, d_v=128, D=128, eta=64, lam=64, chunk=64, dtype="bf16")
    kw.update(bad)
    cfg = lib.make_config(kw["B"], kw["Hh"], kw["d_k"], kw["d_v"], kw["D"], kw["eta"], kw["lam"], kw["chunk"],
                          kw["dtype"])
    assert lib.lola_check_config(cfg) == lib.LOLA_ERR_UNSUPPORTED


@pytest.mark.parametrize("d,eta,lam,dtype", [(128, 64, 64, "bf16"), (64, 64, 64, "f32"), (128, 512, 512, "bf16"),
                                             (128, 0, 0, "f32"), (64, 7, 3, "bf16")])
def test_state_layout_holds_appendix_b_memory(lib, d, eta, lam, dtype):
    """State bytes >= (eta + lambda)(d_k + d_v) io + (D d_v + D) float32 per head; each
    region is 256-byte aligned and regions do not overlap."""
    from oracle.lola_ref import state_elements
    cfg = lib.make_config(3, 5, d, d, d, eta, lam, 64, dtype)
    assert lib.lola_check_config(cfg) == 0
    L = lib.lola_state_layout_of(cfg)
    io = 2 if dtype == "bf16" else 4
    kv = (eta + lam) * 2 * d
    min_bytes = kv * io + (d * d + d) * 4
    assert state_elements(10 ** 9, d, d, d, eta, lam) == kv + d * d + d
    assert L.head_bytes >= min_bytes
    assert lib.lola_state_bytes(cfg) == 15 * L.head_bytes
    regions = [(L.H, 4 * d * d), (L.s, 4 * d), (L.win_pos, 4 * eta), (L.win_k, io * eta * d), (L.win_v, io * eta * d),
               (L.win_phi, 4 * eta * d),
               (L.c_pos, 4 * lam), (L.c_k, io * lam * d), (L.c_v, io * lam * d), (L.c_phi, 4 * lam * d),
               (L.c_N, 4 * lam * d), (L.c_z, 4 * lam), (L.ev, 4 * (d + 1)), (L.tok_phi, 4 * 2 * d)]
    end = 64
    for off, size in regions:
        assert off % 256 == 0 and off >= end
        end = off + size
    assert end <= L.head_bytes


def test_workspace_size_grows_with_n(lib):
    cfg = lib.make_config(4, 32, 128, 128, 128, 64, 64, 64, "bf16")
    a = lib.lola_prefill_workspace_bytes(cfg, 1024)
    b = lib.lola_prefill_workspace_bytes(cfg, 4096)
    assert 0 < a < b
    assert lib.lola_prefill_workspace_bytes(cfg, 0) == 0


def test_null_and_misaligned_pointers_rejected_before_any_launch(lib):
    """Validation returns before anything touches the GPU: safe to call without one."""
    cfg = lib.make_config(1, 1, 64, 64, 64, 4, 4, 16, "f32")
    so = lib._lib
    P = ctypes.c_void_p
    st = so.lola_prefill(ctypes.byref(cfg), 16, None, P(256), P(256), P(256), 0, P(256), P(256), None, P(256),
                         1 << 30, None)
    assert st == lib.LOLA_ERR_INVALID_ARG
    st = so.lola_prefill(ctypes.byref(cfg), 16, P(258), P(256), P(256), P(256), 0, P(256), P(256), None, P(256),
                         1 << 30, None)
    assert st == lib.LOLA_ERR_INVALID_ARG
    st = so.lola_prefill(ctypes.byref(cfg), 0, P(256), P(256), P(256), P(256), 0, P(256), P(256), None, P(256),
                         1 << 30, None)
    assert st == lib.LOLA_ERR_INVALID_ARG
    st = so.lola_prefill(ctypes.byref(cfg), 16, P(256), P(256), P(256), P(256), 0, P(256), P(256), None, P(256),
                         16, None)
    assert st == lib.LOLA_ERR_WORKSPACE
    st = so.lola_decode_step(ctypes.byref(cfg), None, P(256), 0, P(256), P(256), P(256), P(256), None, None)
    assert st == lib.LOLA_ERR_INVALID_ARG
    st = so.lola_decode_step(ctypes.byref(cfg), P(256), P(256), -1, P(256), P(256), P(256), P(256), None, None)
    assert st == lib.LOLA_ERR_INVALID_ARG
    # a per-head W must start on a 16-byte boundary: the stride is a multiple of 4 floats
    st = so.lola_decode_step(ctypes.byref(cfg), P(256), P(256), 6, P(256), P(256), P(256), P(256), None, None)
    assert st == lib.LOLA_ERR_INVALID_ARG
    st = so.lola_prefill(ctypes.byref(cfg), 16, P(256), P(256), P(256), P(256), 6, P(256), P(256), None, P(256),
                         1 << 30, None)
    assert st == lib.LOLA_ERR_INVALID_ARG


def test_bounded_wait_selftest_rejects_bad_limits(lib):
    """The limit is checked before anything is enqueued (safe without a GPU)."""
    for bad in (0, -5, 10 ** 9 + 1):
        st, _ = lib.lola_selftest_bounded_wait(bad, stream=0)
        assert st == lib.LOLA_ERR_INVALID_ARG


def test_read_mask_validation(lib):
    """The read mask is 0..3 and, when nonzero, needs a window (eta >= 1)."""
    ok = lib.make_config(2, 4, 128, 128, 128, 64, 64, 64, "bf16", read_mask=lib.LOLA_READ_HIDE_STATE)
    assert lib.lola_check_config(ok) == 0
    both = lib.make_config(2, 4, 128, 128, 128, 1, 0, 64, "f32", read_mask=3)
    assert lib.lola_check_config(both) == 0
    assert lib.lola_check_config(lib.make_config(2, 4, 128, 128, 128, 64, 64, 64, "bf16", read_mask=4)) == \
        lib.LOLA_ERR_INVALID_ARG
    assert lib.lola_check_config(lib.make_config(2, 4, 128, 128, 128, 0, 64, 64, "bf16", read_mask=2)) == \
        lib.LOLA_ERR_INVALID_ARG
    # the mask changes neither the state layout nor the workspace
    base = lib.make_config(2, 4, 128, 128, 128, 64, 64, 64, "bf16")
    assert lib.lola_state_bytes(ok) == lib.lola_state_bytes(base)
    assert lib.lola_prefill_workspace_bytes(ok, 512) == lib.lola_prefill_workspace_bytes(base, 512)


def test_chunk_alloc_validation(lib):
    """Chunk-granular allocation needs whole window chunks and no read mask."""
    C = lib.LOLA_ALLOC_CHUNK
    ok = lib.make_config(2, 4, 128, 128, 128, 128, 64, 64, "bf16", alloc=C)
    assert lib.lola_check_config(ok) == 0
    for eta, chunk, mask in ((96, 64, 0), (32, 64, 0), (128, 64, 1)):
        cfg = lib.make_config(2, 4, 128, 128, 128, eta, 64, chunk, "bf16", read_mask=mask, alloc=C)
        assert lib.lola_check_config(cfg) == lib.LOLA_ERR_INVALID_ARG, (eta, chunk, mask)
    assert lib.lola_check_config(lib.make_config(2, 4, 128, 128, 128, 64, 64, 64, "bf16", alloc=2)) == \
        lib.LOLA_ERR_INVALID_ARG
    # the selection kernel's shared-memory plan fits the largest cache and chunk accepted, in both
    # builds (tensor-core bf16 at D = 128, CUDA-core float32)
    for dt in ("bf16", "f32"):
        for D in (64, 128):
            big = lib.make_config(1, 1, D, D, D, 256, 1024, 256, dt, alloc=C)
            assert lib.lola_check_config(big) == 0, (dt, D)
    # the decode step is per token: refused for a chunk-mode layer before anything runs
    P = ctypes.c_void_p
    st = lib._lib.lola_decode_step(ctypes.byref(ok), P(256), P(256), 0, P(256), P(256), P(256), P(256), None, None)
    assert st == lib.LOLA_ERR_UNSUPPORTED


def test_sre_map_validation(lib):
    """Null pointers and a workspace smaller than the prefill's are refused before any launch."""
    cfg = lib.make_config(1, 1, 64, 64, 64, 4, 4, 16, "f32")
    so = lib._lib
    P = ctypes.c_void_p
    assert so.lola_sre_map(ctypes.byref(cfg), 16, None, P(256), 1 << 30, P(256), None) == lib.LOLA_ERR_INVALID_ARG
    assert so.lola_sre_map(ctypes.byref(cfg), 0, P(256), P(256), 1 << 30, P(256), None) == lib.LOLA_ERR_INVALID_ARG
    assert so.lola_sre_map(ctypes.byref(cfg), 16, P(256), P(256), 16, P(256), None) == lib.LOLA_ERR_WORKSPACE
    rel = so.lola_sre_map_relative
    assert rel(ctypes.byref(cfg), 16, P(256), P(256), 1 << 30, P(256), None, None) == lib.LOLA_ERR_INVALID_ARG
    assert rel(ctypes.byref(cfg), 16, None, P(256), 1 << 30, P(256), P(256), None) == lib.LOLA_ERR_INVALID_ARG
    assert rel(ctypes.byref(cfg), 16, P(256), P(256), 16, P(256), P(256), None) == lib.LOLA_ERR_WORKSPACE
    assert rel(ctypes.byref(cfg), 16, P(256), P(256), 1 << 30, P(256), P(264), None) == lib.LOLA_ERR_INVALID_ARG


def test_query_dependent_score_validation(lib):
    """The scoring ablation's configs: a known score, a window (eta >= 1) and per-token
    allocation; the decode step is refused for such a layer before anything runs."""
    mk = lambda **kw: lib.make_config(1, 1, 64, 64, 64, kw.get("eta", 8), 8, 16, "f32",  # noqa: E731
                                      alloc=kw.get("alloc", 0), score=kw.get("score", 0))
    for sc in range(5):
        assert lib.lola_check_config(mk(score=sc)) == 0
    for name, val in lib.SCORES.items():
        assert lib.make_config(1, 1, 64, 64, 64, 8, 8, 16, "f32", score=name).score == val
    assert lib.lola_check_config(mk(score=5)) == lib.LOLA_ERR_INVALID_ARG
    assert lib.lola_check_config(mk(score=-1)) == lib.LOLA_ERR_INVALID_ARG
    assert lib.lola_check_config(mk(score=2, eta=0)) == lib.LOLA_ERR_INVALID_ARG
    assert lib.lola_check_config(mk(score=2, alloc=lib.LOLA_ALLOC_CHUNK)) == lib.LOLA_ERR_INVALID_ARG
    assert lib.lola_check_config(mk(score=0, eta=0)) == 0
    cfg = mk(score=4)
    P = ctypes.c_void_p
    st = lib._lib.lola_decode_step(ctypes.byref(cfg), P(256), P(256), 0, P(256), P(256), P(256), P(256), None, None)
    assert st == lib.LOLA_ERR_UNSUPPORTED
    # the float32 phi(Q) the scores read, the scores and the interval sums make the workspace larger
    assert lib.lola_prefill_workspace_bytes(cfg, 100) > lib.lola_prefill_workspace_bytes(mk(score=0), 100)


def test_write_magnitude_cache_layer_validation(lib):
    """The delta-rule cache layer's shapes and pointers are checked before anything is
    enqueued: bf16 rows of 128, w <= 128, chunk a multiple of 128; null or misaligned
    buffers are invalid; the optional outputs may be null."""
    P = ctypes.c_void_p
    ok = lib.make_hola_config(2, 3, 128, 64, 256)
    base = lib.lola_hola_workspace_bytes(ok, 1000)
    assert base > 0
    # the workspace grows with n and with the cache
    assert lib.lola_hola_workspace_bytes(ok, 2000) > base
    assert lib.lola_hola_workspace_bytes(lib.make_hola_config(2, 3, 128, 128, 256), 1000) > base
    for cfg, want in [(lib.make_hola_config(1, 1, 64, 16, 128), lib.LOLA_ERR_UNSUPPORTED),
                      (lib.make_hola_config(1, 1, 128, 129, 128), lib.LOLA_ERR_UNSUPPORTED),
                      (lib.make_hola_config(1, 1, 128, 16, 64), lib.LOLA_ERR_UNSUPPORTED),
                      (lib.make_hola_config(1, 1, 128, 16, 2048), lib.LOLA_ERR_UNSUPPORTED),
                      (lib.make_hola_config(1, 1, 128, 16, 128, lib.LOLA_F32), lib.LOLA_ERR_UNSUPPORTED),
                      (lib.make_hola_config(1, 1, 128, -1, 128), lib.LOLA_ERR_INVALID_ARG),
                      (lib.make_hola_config(0, 1, 128, 16, 128), lib.LOLA_ERR_INVALID_ARG),
                      (lib.make_hola_config(1, 1, 128, 16, 0), lib.LOLA_ERR_INVALID_ARG),
                      (lib.make_hola_config(1, 1, 128, 16, 128, 7), lib.LOLA_ERR_INVALID_ARG)]:
        assert lib._lib.lola_hola_workspace_bytes(ctypes.byref(cfg), 100) == want
    assert lib._lib.lola_hola_workspace_bytes(ctypes.byref(ok), 0) == lib.LOLA_ERR_INVALID_ARG
    bufs = [P(256)] * 10
    call = lambda b, ws=P(256), nbytes=base, n=1000, opt=(None, None, None): lib._lib.lola_hola_prefill(  # noqa: E731
        ctypes.byref(ok), n, *b, *opt, ws, nbytes, None)
    assert call(bufs, nbytes=base - 1) == lib.LOLA_ERR_WORKSPACE
    for i in range(10):
        b = list(bufs)
        b[i] = None
        assert call(b) == lib.LOLA_ERR_INVALID_ARG
        b[i] = P(258)
        assert call(b) == lib.LOLA_ERR_INVALID_ARG
    assert call(bufs, ws=None) == lib.LOLA_ERR_INVALID_ARG
    assert call(bufs, opt=(P(260), None, None)) == lib.LOLA_ERR_INVALID_ARG
    assert call(bufs, n=0) == lib.LOLA_ERR_INVALID_ARG
