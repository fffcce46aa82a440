"""The Store flow on the device (kvswap_store) and the periodic selection
(DecodeStep.step(rescore=False)), through the C ABI, against the fp64 oracle."""
import numpy as np
import pytest
import torch

from srh_workload import configs as C
from srh_workload import generate as G

from helpers import ATTN_TOL, attn_err, fill, load_step_inputs, make_ds, make_oracle, spec_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _ref_step(ora, w, keys, t, pools, rescore=True):
    return ora.step(lambda b: keys[b], lambda b: G.fm_queries(w, t, b), lambda l, b: G.attn_q(w, t, l, b),
                    lambda l, b: G.window(w, l, b),
                    lambda l, b, idx: pools[(l, b)][np.asarray(idx, dtype=np.int64)], rescore=rescore)


def _new_rows(n, seed):
    return np.random.default_rng(seed).standard_normal((n, 512)).astype(np.float32) * 4


def test_store_updates_pool_and_the_staged_row_and_keeps_the_slot():
    w = C.TINY                                   # one swapped layer: cap 2048 > 512 slots
    pools = {(0, 0): G.pool(w, 0, 0)}
    ds = make_ds(w)
    try:
        keys = fill(ds, w, pools)
        ora = make_oracle(w)
        spec = spec_of(w)
        load_step_inputs(ds, w, 0)
        ds.step(spec)
        torch.cuda.synchronize()
        _ref_step(ora, w, keys, 0, pools)
        sel = ds.sel[0, :int(ds.count[0])].cpu().numpy()
        staged = int(sel[0])
        slot = int(ds.phys[0, 0, 0]) - 128
        fresh = int(np.setdiff1d(np.arange(w.n_chunks), sel)[0])
        new = _new_rows(2, 11)
        rows = torch.from_numpy(new).cuda()
        ds.store(0, 0, staged, rows[0:1])
        ds.store(0, 0, fresh, rows[1:2])
        torch.cuda.synchronize()
        view = ds.pool_view(0, 0)
        assert np.array_equal(view[staged], new[0]) and np.array_equal(view[fresh], new[1])
        assert np.array_equal(ds.staging[0, 0, slot].cpu().numpy(), new[0].astype(np.float16))   # fp16 staging
        pools[(0, 0)][staged] = new[0]
        pools[(0, 0)][fresh] = new[1]
        ora.store(0, 0, staged, 1)
        ora.store(0, 0, fresh, 1)
        misses0 = ds.stats()["misses"]
        # the same memory-indexer queries (one lookahead window): the same
        # selection, all hits, the stored chunk in its old slot, its new row used
        load_step_inputs(ds, w, 1)
        ds.step(spec)
        torch.cuda.synchronize()
        ref = _ref_step(ora, w, keys, 1, pools)
        st = ds.stats()
        assert st["misses"] == misses0
        assert st["d2h_bytes"] == 2 * 512 * 4
        assert int(ds.phys[0, 0, 0]) - 128 == slot
        err, rel = attn_err(ds.out[0, 0].cpu().numpy(), ref.out[(0, 0)])
        assert rel <= ATTN_TOL, (err, rel)
        assert ds.check_error() == 0
    finally:
        ds.close()


@pytest.mark.parametrize("before_first_stage", [True, False])
def test_store_on_a_layer_that_does_not_swap(before_first_stage):
    w = C.TINY.with_(gpu_chunks=2048)            # cap 2048 <= 2048 slots: resident, row c = chunk c
    pools = {(0, 0): G.pool(w, 0, 0)}
    ds = make_ds(w)
    try:
        keys = fill(ds, w, pools)
        assert not ds.swap[0]
        ora = make_oracle(w)
        spec = spec_of(w)
        new = _new_rows(3, 12)
        rows = torch.from_numpy(new).cuda()
        if not before_first_stage:
            load_step_inputs(ds, w, 0)
            ds.step(spec)
            _ref_step(ora, w, keys, 0, pools)
        ds.store(0, 0, 100, rows)                # chunks 100..102
        pools[(0, 0)][100:103] = new
        ora.store(0, 0, 100, 3)
        load_step_inputs(ds, w, 1)
        ds.step(spec)
        torch.cuda.synchronize()
        ref = _ref_step(ora, w, keys, 1, pools)
        assert np.array_equal(ds.staging[0, 0, 100:103].cpu().numpy(), new.astype(np.float16))
        err, rel = attn_err(ds.out[0, 0].cpu().numpy(), ref.out[(0, 0)])
        assert rel <= ATTN_TOL, (err, rel)
        assert ds.check_error() == 0
    finally:
        ds.close()


def test_storing_the_missing_chunks_clears_the_not_stored_error():
    from sparse_retrieval_host_gb300 import abi
    w = C.TINY
    pool = G.pool(w, 0, 0)
    ds = make_ds(w)
    try:
        from sparse_retrieval_host_gb300.runtime import bits_to_i16
        keys = G.keys(w, 0)
        ds.keys[0] = bits_to_i16(keys)
        ds.window[0, 0] = torch.from_numpy(G.window(w, 0, 0))
        view = ds.pool_view(0, 0)
        view[:1024] = pool[:1024]
        ds.mark_stored(0, 0, 0, 1024)            # the upper half was never stored
        spec = spec_of(w)
        load_step_inputs(ds, w, 0)
        ds.step(spec)
        assert ds.check_error() == abi.SRH_ERR_NOT_STORED
        sel = ds.sel[0, :int(ds.count[0])].cpu().numpy()
        assert (sel >= 1024).any()
        # the compressor's chunks arrive through the device store path
        ds.store(0, 0, 1024, torch.from_numpy(pool[1024:]).cuda())
        ora = make_oracle(w)                     # everything stored from here on
        load_step_inputs(ds, w, 1)
        ds.step(spec)
        torch.cuda.synchronize()
        assert ds.check_error() == 0
        ref = _ref_step(ora, w, [keys], 1, {(0, 0): pool})
        err, rel = attn_err(ds.out[0, 0].cpu().numpy(), ref.out[(0, 0)])
        assert rel <= ATTN_TOL, (err, rel)
        assert np.array_equal(view[1024:], pool[1024:])
    finally:
        ds.close()


def test_periodic_selection_matches_scoring_every_step():
    """The memory-indexer queries are held for a lookahead window, so scoring
    once per window gives the same bits as scoring at every step."""
    w = C.TINY.with_(steps=20)
    runs = []
    for periodic in (False, True):
        ds = make_ds(w)
        try:
            fill(ds, w)
            spec = spec_of(w)
            seq = []
            for t in range(w.steps):
                load_step_inputs(ds, w, t)
                ds.step(spec, rescore=(not periodic) or t % w.lookahead == 0)
                torch.cuda.synchronize()
                seq.append([x.clone() for x in (ds.sel, ds.count, ds.phys, ds.count_l, ds.out)])
            st = ds.stats()
            runs.append((seq, st["hits"], st["misses"]))
            assert ds.check_error() == 0
        finally:
            ds.close()
    (sa, ha, ma), (sb, hb, mb) = runs
    assert (ha, ma) == (hb, mb)
    for xa, xb in zip(sa, sb):
        for a, b in zip(xa, xb):
            assert torch.equal(a, b)


def test_fp16_staging_reports_pool_values_beyond_its_range():
    """Staged rows are kept as fp16: a pool value beyond +-65504 that reaches a
    staging slot -- by a store into a staged chunk, or by the miss gather of a
    chunk stored earlier -- is reported as SRH_ERR_RANGE; finite rows are not."""
    from sparse_retrieval_host_gb300 import abi
    w = C.TINY
    pools = {(0, 0): G.pool(w, 0, 0)}
    ds = make_ds(w)
    try:
        fill(ds, w, pools)
        load_step_inputs(ds, w, 0)
        ds.step(spec_of(w))
        torch.cuda.synchronize()
        assert ds.check_error() == abi.SRH_OK
        sel = ds.sel[0, :int(ds.count[0])].cpu().numpy()
        staged = int(sel[0])
        big = pools[(0, 0)][staged:staged + 1].copy()
        big[0, 7] = 1e5
        ds.store(0, 0, staged, torch.from_numpy(big).cuda())      # the staged row gets it
        torch.cuda.synchronize()
        assert ds.check_error() == abi.SRH_ERR_RANGE
        assert ds.check_error() == abi.SRH_OK
        ds.store(0, 0, staged, torch.from_numpy(pools[(0, 0)][staged:staged + 1].copy()).cuda())
        torch.cuda.synchronize()
        assert ds.check_error() == abi.SRH_OK
        # a chunk in no slot: the store writes the pool only, its miss gather converts the row
        fresh = int(np.setdiff1d(np.arange(w.n_chunks), sel)[0])
        big = pools[(0, 0)][fresh:fresh + 1].copy()
        big[0, 300] = -7e4
        ds.store(0, 0, fresh, torch.from_numpy(big).cuda())
        torch.cuda.synchronize()
        assert ds.check_error() == abi.SRH_OK
        s = np.zeros(tuple(ds.sel.shape), np.int32)
        s[0, 0] = fresh
        ds.sel.copy_(torch.from_numpy(s))
        ds.count.copy_(torch.ones_like(ds.count))
        ds.stage()
        torch.cuda.synchronize()
        assert ds.check_error() == abi.SRH_ERR_RANGE
        assert ds.check_error() == abi.SRH_OK
    finally:
        ds.close()
