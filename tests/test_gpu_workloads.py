"""Parity at the workloads' full sizes, in the launch configuration the benchmark times.

The GPU runs every head; the float64 oracle replays the GPU's decision log (every decision
must be a due candidate within 1e-3 relative SRE of the oracle's best) and gives the
outputs along that trajectory, which the GPU outputs must match within the bf16 bars.
Where the oracle would take minutes, a fixed sample of heads is checked; the sample is
stated in each test.  The float32 workload is checked free-running (exact decision log).

Method: "LoLA: Low-Rank Linear Attention With Sparse Caching" (arXiv 2505.23666v3),
reading notes sections 2.2-2.6."""
import numpy as np
import pytest
import torch

import synth
from oracle import inc

from lola_parity import GAP, check_final_state, check_outputs, run_prefill, to_dev, to_f64

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_exact_kv_gb300 as lib
    return lib


def _replay(x, wpos, eta, lam, heads, read_mask=0):
    """Oracle replay over a subset of heads (flattened indices)."""
    BH = x.w.B * x.w.Hh
    n = wpos.shape[-1]
    pick = lambda a: a.reshape(BH, *a.shape[2:])[heads]  # noqa: E731
    rep = inc.run(pick(x.q)[:, :n], pick(x.k)[:, :n], pick(x.v)[:, :n], x.W, eta, lam, x.w.dtype,
                  replay=wpos.reshape(BH, -1)[heads], read_mask=read_mask)
    assert (rep["status"] == 0).all(), np.unique(rep["status"])
    worst = float(np.max(rep["max_gap"]))
    assert worst < GAP, f"decision {worst:.3e} relative SRE away from the best"
    return rep


def _prefill_parity(L, name, heads=None, read_mask=0):
    w = synth.WORKLOADS[name]
    x = synth.make_inputs(w)
    Y, wpos, lay = run_prefill(L, x, w.eta, w.lam, w.chunk, read_mask=read_mask)
    BH = w.B * w.Hh
    heads = np.arange(BH) if heads is None else np.asarray(heads)
    rep = _replay(x, wpos, w.eta, w.lam, heads, read_mask=read_mask)
    check_outputs(Y.reshape(BH, w.n, w.d)[heads], rep["Y"], "bf16", what=name)
    st, words = L.lola_read_status(lay.cfg, lay.state)
    assert st == 0, words
    check_final_state(lay.read_state(), rep, "bf16", w.eta, w.n, heads=heads)
    return rep, wpos


def test_w2_full_every_head(L):
    """4 x 32 heads, n = 4096, eta = lambda = 64 (the benchmark's prefill): all 128 heads."""
    rep, _ = _prefill_parity(L, "w2_bf16_b4h32_n4096")
    assert rep["Y"].shape == (128, 4096, 128)


def test_w2_read_mask_full_every_head(L):
    """w2 with both the state and the cache hidden from every read (appendix I, Table 12's
    window-only row): the decisions equal the unmasked run's (the mask never changes the
    memory) and every head's outputs follow the oracle read with the same mask."""
    _, w_masked = _prefill_parity(L, "w2_bf16_b4h32_n4096", read_mask=3)
    w = synth.WORKLOADS["w2_bf16_b4h32_n4096"]
    x = synth.make_inputs(w)
    _, w_plain, _ = run_prefill(L, x, w.eta, w.lam, w.chunk)
    assert np.array_equal(w_masked, w_plain)


def test_w3_needles_full_every_head(L):
    """1 x 32 heads, n = 16384, eta = lambda = 256 (4-CTA clusters), planted high-norm keys."""
    _prefill_parity(L, "w3_bf16_h32_n16384_needle")


def test_w5_long_prefill_sampled_heads(L):
    """1 x 8 heads, n = 131072, eta = lambda = 512 (8-CTA clusters), AR(1) inputs: the GPU runs
    all 8 heads; the oracle replays heads 0 and 5 over all 131072 tokens."""
    _prefill_parity(L, "w5_bf16_h8_n131072_ar1", heads=[0, 5])


def test_w1_f32_full_free_running(L):
    """The float32 workload: the decision log equals the free-running oracle's."""
    w = synth.WORKLOADS["w1_f32_n1024"]
    x = synth.make_inputs(w)
    Y, wpos, lay = run_prefill(L, x, w.eta, w.lam, w.chunk)
    ref = inc.run(x.q, x.k, x.v, x.W, w.eta, w.lam, "f32")
    assert np.array_equal(wpos, ref["write_pos"])
    check_outputs(Y, ref["Y"], "f32")
    check_final_state(lay.read_state(), ref, "f32", w.eta, w.n)


def test_w4_decode_full_sampled_heads(L):
    """64 x 32 heads: prefill a 4096-token prefix on the GPU, then 1024 decode steps for all
    2048 heads; the oracle replays 16 fixed heads over the whole 5120 tokens."""
    w = synth.WORKLOADS["w4_bf16_decode_b64h32"]
    x = synth.make_inputs(w)
    dev = "cuda"
    lay = L.Lola(w.B, w.Hh, w.d, w.D, w.eta, w.lam, chunk=w.chunk, dtype=torch.bfloat16, device=dev)
    W = torch.from_numpy(x.W).to(dev)
    P = [to_dev(getattr(x, a)[:, :, :w.n], dev, "bf16") for a in "qkv"]
    wpre = torch.empty(w.B, w.Hh, w.n, dtype=torch.int32, device=dev)
    Ypre = lay.prefill(*P, W, write_pos=wpre)
    del P
    lay.workspace = None
    steps = w.decode_steps
    dq, dk, dv = (to_dev(getattr(x, a)[:, :, w.n:].transpose(2, 0, 1, 3), dev, "bf16") for a in "qkv")
    ys = torch.empty(steps, w.B, w.Hh, w.d, dtype=torch.bfloat16, device=dev)
    wps = torch.empty(steps, w.B, w.Hh, dtype=torch.int32, device=dev)
    for i in range(steps):
        lay.decode_step(dq[i], dk[i], dv[i], W, y=ys[i], written_pos=wps[i])
    torch.cuda.synchronize()
    st, words = L.lola_read_status(lay.cfg, lay.state)
    assert st == 0, [i for i, v in enumerate(words) if v][:5]
    BH = w.B * w.Hh
    heads = np.arange(0, BH, BH // 16)
    wall = np.concatenate([wpre.cpu().numpy().reshape(BH, w.n),
                           wps.cpu().numpy().reshape(steps, BH).T], axis=1)
    rep = _replay(x, wall, w.eta, w.lam, heads)
    Yall = np.concatenate([to_f64(Ypre).reshape(BH, w.n, w.d),
                           to_f64(ys).reshape(steps, BH, w.d).transpose(1, 0, 2)], axis=1)
    check_outputs(Yall[heads][:, w.n:], rep["Y"][:, w.n:], "bf16", what="decode outputs")
    check_outputs(Yall[heads][:, :w.n], rep["Y"][:, :w.n], "bf16", what="prefix outputs")


def _chunk_parity(L, name, heads):
    """Chunk-granular allocation at a workload's full size: the GPU runs every head; the float64
    chunk oracle replays the GPU's per-key log on the sampled heads."""
    from oracle import lola_ref as R
    w = synth.WORKLOADS[name]
    x = synth.make_inputs(w)
    Y, wlog, lay = run_prefill(L, x, w.eta, w.lam, w.chunk, alloc=L.LOLA_ALLOC_CHUNK)
    BH = w.B * w.Hh
    q, k, v = (x.widened(a).reshape(BH, w.n, -1) for a in "qkv")
    wl = wlog.reshape(BH, w.n)
    for h in heads:
        ref = R.lola_chunk_run(q[h], k[h], v[h], x.W, w.eta, w.lam, w.chunk, replay=wl[h])
        assert ref["max_gap"] < GAP, f"head {h}: a chunk decision {ref['max_gap']:.3e} away from the best"
        check_outputs(Y.reshape(BH, w.n, w.d)[h], ref["Y"], "bf16", what=f"{name} head {h}")
    st, words = L.lola_read_status(lay.cfg, lay.state)
    assert st == 0, words


def test_w2_chunk_allocation_sampled_heads(L):
    """w2 (4 x 32 heads, n = 4096, eta = lambda = C = 64) with chunk-granular allocation: the
    GPU runs all 128 heads; the chunk oracle replays heads 0, 77 and 127."""
    _chunk_parity(L, "w2_bf16_b4h32_n4096", heads=[0, 77, 127])


def test_w5_chunk_allocation_sampled_head(L):
    """w5 (8 heads, n = 131072, eta = lambda = 512, C = 256: window = two chunks, AR(1)
    inputs) with chunk-granular allocation: the GPU runs all 8 heads; the chunk oracle
    replays head 6 over all 512 chunk starts."""
    _chunk_parity(L, "w5_bf16_h8_n131072_ar1", heads=[6])


def test_w3_chunk_allocation_sampled_heads(L):
    """w3 (32 heads, n = 16384, eta = lambda = 256, C = 128: window = two chunks) with
    chunk-granular allocation and the planted needles: heads 3 and 30 replayed."""
    _chunk_parity(L, "w3_bf16_h32_n16384_needle", heads=[3, 30])
