"""fm_select_noalloc: the selection entry point that allocates nothing.

It takes no context and keeps its only scratch (the first-digit histogram) in
a fixed array inside the library, so its results must equal fm_select's on
the same inputs, call after call, although every call reuses the array the
previous call left behind. The CPU test checks the size limits; the GPU test
compares consecutive calls with fm_select (exact: selection is index work).
"""
import shutil

import numpy as np
import pytest

from oracle import srh_oracle as O

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and not __import__("os").path.exists(
    "/usr/local/cuda/bin/nvcc"), reason="nvcc not available")


@pytest.fixture(scope="module")
def abi():
    import __graft_entry__
    __graft_entry__.build()
    from sparse_retrieval_host_gb300 import abi as a
    return a


def _rejects(abi, match, **over):
    kw = dict(scores=256, batch=1, n=100, mode=abi.SRH_SELECT_TOPK, k=10, tau=0.5, clamp=0, max_select=64,
              sel=512, count=768, stream=0)
    kw.update(over)
    with pytest.raises(abi.SrhError) as ei:
        abi.fm_select_noalloc(**kw)
    assert ei.value.code == abi.SRH_ERR_INVALID
    assert match in str(ei.value), str(ei.value)


def test_noalloc_rejects_sizes_beyond_its_limits(abi):
    """Checked on the host before any GPU work (the dummy pointers are never used)."""
    _rejects(abi, f"batch={abi.SRH_NOALLOC_MAX_BATCH + 1}", batch=abi.SRH_NOALLOC_MAX_BATCH + 1)
    _rejects(abi, "batch=0", batch=0)
    _rejects(abi, "n=0", n=0)
    _rejects(abi, "max_select=4097", max_select=4097)
    _rejects(abi, "k=65", k=65)
    _rejects(abi, "clamp=65", mode=abi.SRH_SELECT_THRESH, clamp=65)
    _rejects(abi, "tau", mode=abi.SRH_SELECT_THRESH, tau=1.0)
    _rejects(abi, "mode", mode=7)
    _rejects(abi, "NULL", scores=None)


def _scores(kind, B, n, rng):
    if kind == "random":
        return rng.standard_normal((B, n)).astype(np.float32)
    if kind == "ties":
        return rng.choice(np.float32([-2.0, -0.0, 0.0, 0.5, 1.0, 1.0000001, 3.0]), size=(B, n))
    if kind == "tail":
        return (rng.standard_normal((B, n)) - 2.0).astype(np.float32)
    raise ValueError(kind)


@pytest.mark.gpu
def test_noalloc_matches_fm_select_on_consecutive_calls(abi):
    import torch
    torch.cuda.set_device(0)
    B, n, S = 4, 50001, 1024
    rng = np.random.default_rng(20261202)
    # (batch, mode, k, clamp, scores): the second call uses fewer rows and other
    # scores, so rows the first call left in the shared scratch must not leak in.
    calls = [
        (B, abi.SRH_SELECT_TOPK, 512, 0, _scores("random", B, n, rng)),
        (3, abi.SRH_SELECT_TOPK, 200, 0, _scores("ties", B, n, rng)),
        (B, abi.SRH_SELECT_THRESH, 512, 300, _scores("tail", B, n, rng)),
    ]
    dev = torch.device("cuda", 0)
    scores = [torch.from_numpy(c[4]).to(dev) for c in calls]
    outs = [(torch.full((B, S), -1, dtype=torch.int32, device=dev), torch.full((B,), -1, dtype=torch.int32,
                                                                                 device=dev)) for _ in calls]
    # The no-alloc calls back to back on one stream.
    for (b, mode, k, clamp, _), sc, (sel, cnt) in zip(calls, scores, outs):
        abi.fm_select_noalloc(sc, b, n, mode, k, 0.5, clamp, S, sel, cnt)
    torch.cuda.synchronize()

    cfg = abi.make_config(batch=B, layer_ratios=(128,), gpu_chunks=512, index_topk=512, context_len=4 * n,
                          max_select=S)
    ctx = abi.srh_create(cfg)
    try:
        for (b, mode, k, clamp, s_np), sc, (sel, cnt) in zip(calls, scores, outs):
            ref_sel = torch.full((B, S), -1, dtype=torch.int32, device=dev)
            ref_cnt = torch.full((B,), -1, dtype=torch.int32, device=dev)
            abi.fm_select(ctx, sc, n, mode, k, 0.5, clamp, ref_sel, ref_cnt)
            torch.cuda.synchronize()
            got_c, ref_c = cnt.cpu().numpy(), ref_cnt.cpu().numpy()
            assert np.array_equal(got_c[:b], ref_c[:b])
            assert np.all(got_c[b:] == -1)          # rows past the call's batch are untouched
            for r in range(b):
                m = int(ref_c[r])
                assert np.array_equal(sel[r, :m].cpu().numpy(), ref_sel[r, :m].cpu().numpy())
        # And the first call against the oracle's definition directly.
        s0 = calls[0][4]
        for r in range(B):
            assert np.array_equal(outs[0][0][r, :512].cpu().numpy(), O.select_topk(s0[r].astype(np.float64), 512))
    finally:
        abi.srh_destroy(ctx)


@pytest.mark.gpu
def test_noalloc_full_batch_reaches_the_last_scratch_row(abi):
    """At batch = SRH_NOALLOC_MAX_BATCH every row of the fixed scratch is used:
    two calls in a row (the second with other scores) against the oracle."""
    import torch
    torch.cuda.set_device(0)
    B, n, S, k = abi.SRH_NOALLOC_MAX_BATCH, 4097, 64, 16
    rng = np.random.default_rng(64)
    dev = torch.device("cuda", 0)
    for kind in ("random", "ties"):
        s_np = _scores(kind, B, n, rng)
        sel = torch.full((B, S), -1, dtype=torch.int32, device=dev)
        cnt = torch.full((B,), -1, dtype=torch.int32, device=dev)
        abi.fm_select_noalloc(torch.from_numpy(s_np).to(dev), B, n, abi.SRH_SELECT_TOPK, k, 0.5, 0, S, sel, cnt)
        torch.cuda.synchronize()
        got, got_c = sel.cpu().numpy(), cnt.cpu().numpy()
        assert np.all(got_c == k)
        for r in range(B):
            assert np.array_equal(got[r, :k], O.select_topk(s_np[r].astype(np.float64), k)), (kind, r)
