"""GPU parity of each C-ABI call against the fp64 oracle on seeded inputs."""
import numpy as np
import pytest
import torch

from oracle import srh_oracle as O
from srh_workload import configs as C
from srh_workload import generate as G

from helpers import (ATTN_TOL, attn_err, check_selection, fill, load_step_inputs, make_ds, spec_of)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _w(**kw):
    base = dict(name="unit", code=50, context_len=8192, layer_ratios=(4,), gpu_chunks=512,
                index_topk=512, ensemble=C.ENSEMBLE_MAX, select_mode=C.SELECT_TOPK, tau=0.5,
                bias=0.0, n_heads=16, batch=1, steps=4, lookahead=2)
    base.update(kw)
    return C.Workload(**base)


# ----------------------------------------------------------------------------- fm_score
@pytest.mark.parametrize("w", [
    C.TINY,
    _w(context_len=4 * 1001 + 3, code=51),                          # ragged tail: n = 1002
    _w(context_len=4, code=52, index_topk=1, gpu_chunks=1),         # n = 1
    _w(context_len=131072, batch=3, code=53, ensemble=C.ENSEMBLE_MEAN, bias=-7.0),
    # 2^19 chunks in one call: the tensor-core kernel (from 2^18; smaller calls use the mma.sync one)
    _w(context_len=131072, batch=16, code=61, layer_ratios=(128,)),
    _w(context_len=4 * (4 * 32768 + 37), batch=4, code=62, layer_ratios=(128,), ensemble=C.ENSEMBLE_MEAN,
       bias=-7.0),
], ids=["tiny", "ragged", "n1", "b3_mean", "b16_tc", "b4_ragged_tc"])
def test_fm_score_matches_oracle(w):
    from sparse_retrieval_host_gb300.runtime import bits_to_i16
    ds = make_ds(w, layer_ratios=(4,))
    try:
        keys = [G.keys(w, b) for b in range(w.batch)]
        for b in range(w.batch):
            ds.keys[b] = bits_to_i16(keys[b])
        for t in (0, w.lookahead):
            for b in range(w.batch):
                ds.fm_q[b] = bits_to_i16(G.fm_queries(w, t, b))
            ds.score(spec_of(w))
            got = ds.scores.double().cpu().numpy()
            for b in range(w.batch):
                q = G.fm_queries(w, t, b)
                ref = O.score(keys[b], q, w.scale, [w.bias] * 3, w.ensemble)
                # a-priori bound of an fp32 dot product of 128 terms in any order
                # (unit roundoff 2^-23 allows truncating adders), then scale, bias
                # and the ensemble in fp32
                absdot = np.abs(O.bf16_to_f64(keys[b])) @ np.abs(O.bf16_to_f64(q)).reshape(24, 128).T
                bound = (w.scale * 128 * 2.0 ** -23 * absdot.max(axis=1)
                         + 8 * 2.0 ** -24 * (np.abs(ref) + abs(w.bias)))
                err = np.abs(got[b] - ref)
                assert np.all(err <= bound), (err.max(), bound[err.argmax()])
                if len(err) >= 100:
                    assert np.median(err) <= 1e-6
    finally:
        ds.close()


@pytest.mark.parametrize("w", [
    C.TINY,
    _w(context_len=4 * 1001 + 3, code=56),                          # ragged tail: n = 1002
    _w(context_len=131072, batch=2, code=57, ensemble=C.ENSEMBLE_MEAN, bias=-7.0),
], ids=["tiny", "ragged", "b2_mean"])
def test_fm_score_multi_matches_oracle(w):
    """One key set per memory indexer: indexer i scores key set i."""
    from sparse_retrieval_host_gb300.runtime import bits_to_i16
    ds = make_ds(w, layer_ratios=(4,), key_sets=3)
    try:
        keys = [G.keys_multi(w, b) for b in range(w.batch)]
        for b in range(w.batch):
            for i in range(3):
                ds.keys[i, b] = bits_to_i16(keys[b][i])
        for t in (0, w.lookahead):
            for b in range(w.batch):
                ds.fm_q[b] = bits_to_i16(G.fm_queries_multi(w, t, b))
            ds.score(spec_of(w))
            got = ds.scores.double().cpu().numpy()
            for b in range(w.batch):
                q = G.fm_queries_multi(w, t, b)
                ref = O.score_multi(keys[b], q, w.scale, [w.bias] * 3, w.ensemble)
                qf = np.abs(O.bf16_to_f64(q)).reshape(3, 8, 128)
                absdot = np.stack([np.abs(O.bf16_to_f64(keys[b][i])) @ qf[i].T for i in range(3)])
                bound = (w.scale * 128 * 2.0 ** -23 * absdot.max(axis=(0, 2))
                         + 8 * 2.0 ** -24 * (np.abs(ref) + abs(w.bias)))
                err = np.abs(got[b] - ref)
                assert np.all(err <= bound), (err.max(), bound[err.argmax()])
                if len(err) >= 100:
                    assert np.median(err) <= 1e-6
                # the needles of every indexer's own key set are found
                top = O.select_topk(ref, w.index_topk)
                assert np.isin(G.step_needles(w, t, b), top).all()
    finally:
        ds.close()


def _crafted_keys(n, rng):
    """Random keys plus chunks that exercise the quantizer's corners."""
    k = rng.standard_normal((n, 128)).astype(np.float32)
    k[0] = 0.0                                            # all zero: scale 0, zero codes
    k[1, :] = 1e-6 * (-1.0) ** np.arange(128)             # +-tiny: zero codes, the negative ones signed
    k[1, 7] = -3e4                                        # large amax, tiny negatives -> signed zeros
    k[2, ::2] = -k[2, ::2] * 1e-3                         # wide dynamic range, subnormal codes
    return G.f32_to_bf16_bits(k)


@pytest.mark.parametrize("w", [
    C.TINY,
    _w(context_len=4 * 1001 + 3, code=58),                          # ragged tail: n = 1002
    _w(context_len=131072, batch=2, code=59, ensemble=C.ENSEMBLE_MEAN, bias=-7.0),
], ids=["tiny", "ragged", "b2_mean"])
def test_fp8_keys_quantize_exactly_and_score_within_bound(w):
    from sparse_retrieval_host_gb300.runtime import bits_to_i16
    ds = make_ds(w, layer_ratios=(4,), key_format="fp8")
    try:
        keys = [G.keys(w, b) for b in range(w.batch)]
        keys[0] = np.concatenate([_crafted_keys(3, np.random.default_rng(5)), keys[0][3:]])
        for b in range(w.batch):
            ds.keys[b] = bits_to_i16(keys[b])
        ds.quantize_keys()
        codes = ds.codes.cpu().numpy()
        ks = ds.kscale.cpu().numpy()
        ref = [O.quantize_keys_fp8(keys[b]) for b in range(w.batch)]
        for b in range(w.batch):
            assert np.array_equal(ks[b], ref[b][1]), np.nonzero(ks[b] != ref[b][1])[0][:5]
            bad = np.nonzero(codes[b] != ref[b][0])
            assert bad[0].size == 0, (bad[0][:5], bad[1][:5], codes[b][bad][:5], ref[b][0][bad][:5])
        for t in (0, w.lookahead):
            for b in range(w.batch):
                ds.fm_q[b] = bits_to_i16(G.fm_queries(w, t, b))
            ds.score(spec_of(w))
            ds.select(spec_of(w))
            got = ds.scores.double().cpu().numpy()
            for b in range(w.batch):
                q = G.fm_queries(w, t, b)
                c8, k8 = ref[b]
                s_ref = O.score_fp8(c8, k8, q, w.scale, [w.bias] * 3, w.ensemble)
                deq = np.abs(O.e4m3_decode(c8))
                absdot = (deq @ np.abs(O.bf16_to_f64(q)).reshape(24, 128).T).max(axis=1) * k8.astype(np.float64)
                bound = w.scale * 130 * 2.0 ** -23 * absdot + 8 * 2.0 ** -24 * (np.abs(s_ref) + abs(w.bias))
                err = np.abs(got[b] - s_ref)
                assert np.all(err <= bound), (err.max(), bound[err.argmax()])
                sel_ref = O.select(s_ref, w.select_mode, w.index_topk, w.tau, w.clamp)
                cnt = int(ds.count[b])
                check_selection(w, s_ref, sel_ref, ds.sel[b, :cnt].cpu().numpy(), got[b])
                nd = G.step_needles(w, t, b)
                nd = nd[nd >= 3] if b == 0 else nd          # chunks 0-2 of sequence 0 were replaced
                assert np.isin(nd, ds.sel[b, :cnt].cpu().numpy()).all()
    finally:
        ds.close()


# ----------------------------------------------------------------------------- fm_select
def _select_case(name, n, rng):
    if name == "random":
        return rng.standard_normal(n).astype(np.float32)
    if name == "ties":
        return rng.choice(np.float32([-2.0, -0.0, 0.0, 0.5, 1.0, 1.0000001, 3.0]), size=n)
    if name == "equal":
        return np.zeros(n, np.float32)
    if name == "one_bin":     # everything in one 12-bit histogram bin: forces deeper radix passes
        return (1.0 + rng.random(n) * 1e-3).astype(np.float32)
    if name == "neg":
        return -np.abs(rng.standard_normal(n)).astype(np.float32)
    if name == "coarse":      # 64 distinct values: mid-sized digit buckets full of exact ties
        return (rng.integers(0, 64, n) * 0.125).astype(np.float32)
    if name == "wide":        # magnitudes from 1e-30 to 1e30: the fine buckets span thousands of digits
        return (rng.standard_normal(n) * 10.0 ** rng.integers(-30, 31, n)).astype(np.float32)
    raise ValueError(name)


@pytest.mark.parametrize("n", [1, 37, 2048, 65536, 262144])
@pytest.mark.parametrize("case", ["random", "ties", "equal", "one_bin", "neg", "coarse", "wide"])
def test_fm_select_topk_exact(n, case):
    from sparse_retrieval_host_gb300 import abi
    rng = np.random.default_rng(n + len(case))
    s = _select_case(case, n, rng)
    k = 512
    w = _w(context_len=4 * n, code=54)
    ds = make_ds(w, layer_ratios=(4,))
    try:
        ds.scores[0, :n] = torch.from_numpy(s)
        abi.fm_select(ds.ctx, ds.scores, n, abi.SRH_SELECT_TOPK, k, 0.5, 0, ds.sel, ds.count)
        cnt = int(ds.count[0])
        got = ds.sel[0, :cnt].cpu().numpy()
        ref = O.select_topk(s.astype(np.float64), k)
        assert cnt == len(ref)
        assert np.array_equal(got, ref)
    finally:
        ds.close()


@pytest.mark.parametrize("n,clamp,case", [(2048, 512, "random"), (262144, 512, "random"),
                                          (262144, 512, "neg"), (5000, 4, "ties"), (70000, 300, "ties"),
                                          (2048, 0, "random")])
def test_fm_select_threshold_exact(n, clamp, case):
    from sparse_retrieval_host_gb300 import abi
    rng = np.random.default_rng(n + clamp)
    s = _select_case(case, n, rng) - np.float32(2.5 if case == "random" else 0.0)
    w = _w(context_len=4 * n, code=55)
    ds = make_ds(w, layer_ratios=(4,))
    try:
        ds.scores[0, :n] = torch.from_numpy(s)
        abi.fm_select(ds.ctx, ds.scores, n, abi.SRH_SELECT_THRESH, 512, 0.5, clamp, ds.sel, ds.count)
        cnt = int(ds.count[0])
        got = ds.sel[0, :cnt].cpu().numpy()
        ref = O.select_threshold(s.astype(np.float64), 0.5, clamp)
        assert np.array_equal(got, ref)
    finally:
        ds.close()


def test_fm_select_uses_fresh_histogram_after_scores_change():
    """The scoring pass's histogram is used once; a second selection over other
    scores in the same buffer must rebuild it."""
    from sparse_retrieval_host_gb300 import abi
    from sparse_retrieval_host_gb300.runtime import bits_to_i16
    w = C.TINY
    ds = make_ds(w)
    try:
        keys = G.keys(w, 0)
        ds.keys[0] = bits_to_i16(keys)
        ds.fm_q[0] = bits_to_i16(G.fm_queries(w, 0, 0))
        ds.score(spec_of(w))
        ds.select(spec_of(w))
        s = np.random.default_rng(3).standard_normal(w.n_chunks).astype(np.float32)
        ds.scores[0] = torch.from_numpy(s)
        ds.select(spec_of(w))
        got = ds.sel[0, :int(ds.count[0])].cpu().numpy()
        assert np.array_equal(got, O.select_topk(s.astype(np.float64), w.index_topk))
    finally:
        ds.close()


# ----------------------------------------------------------------------------- kvswap_stage
def _trace(rng, n_steps, n, m_max, G_):
    """Selections (distinct ids) mixing repeats, fresh ids and returns of old ids,
    so some steps pop a slot whose chunk is selected later in the same list."""
    steps, hist = [], []
    for t in range(n_steps):
        m = int(rng.integers(0, m_max + 1))
        kind = t % 4
        if kind == 0 or not hist:
            ids = rng.choice(n, size=m, replace=False)
        elif kind == 1:
            prev = hist[-1]
            keep = prev[rng.random(len(prev)) < 0.7]
            fresh = rng.choice(n, size=m, replace=False)
            ids = np.concatenate([keep, fresh])
        elif kind == 2:
            old = np.concatenate(hist[-4:])
            ids = np.concatenate([rng.choice(n, size=m // 2, replace=False), old[::-1]])
        else:
            ids = np.concatenate([hist[0][::-1], rng.choice(n, size=m, replace=False)])
        _, first = np.unique(ids, return_index=True)
        ids = ids[np.sort(first)][:m_max]
        steps.append(ids.astype(np.int64))
        hist.append(ids)
    return steps


@pytest.mark.parametrize("G_,k,ctx_len", [(64, 48, 4 * 600), (512, 512, 8192), (40, 40, 4 * 90)])
def test_kvswap_stage_matches_list_lru(G_, k, ctx_len):
    ratios = (4, 128, 4, 8)
    w = _w(context_len=ctx_len, layer_ratios=ratios, gpu_chunks=G_, index_topk=k, batch=2, code=56)
    ds = make_ds(w, max_select=k)
    try:
        pools = {(l, b): G.pool(w, l, b) for l in range(w.n_layers) for b in range(w.batch)}
        fill(ds, w, pools)
        states = [[O.KvSwapLayerState(w.layer_cap(l), G_) for b in range(w.batch)] for l in range(w.n_layers)]
        for row in states:
            for st in row:
                st.host_ready[:] = 1
        rng = np.random.default_rng(G_ + k)
        traces = [_trace(rng, 24, w.n_chunks, k, G_) for _ in range(w.batch)]
        hits = misses = 0
        for t in range(24):
            sel = np.zeros((w.batch, ds.S), np.int32)
            cnt = np.zeros(w.batch, np.int32)
            for b in range(w.batch):
                ids = traces[b][t]
                sel[b, :len(ids)] = ids
                cnt[b] = len(ids)
            ds.sel.copy_(torch.from_numpy(sel))
            ds.count.copy_(torch.from_numpy(cnt))
            ds.stage()
            torch.cuda.synchronize()
            phys = ds.phys.cpu().numpy()
            cl = ds.count_l.cpu().numpy()
            staging = ds.staging.cpu().numpy()
            for l in range(w.n_layers):
                for b in range(w.batch):
                    lst = O.layer_chunks(traces[b][t], 4, ratios[l])
                    r = states[l][b].swap_in_selected(lst)
                    if states[l][b].swap_enabled:
                        hits += r.hits
                        misses += len(r.misses)
                    assert cl[l, b] == len(lst)
                    assert phys[l, b, :len(lst)].tolist() == r.phys, (t, l, b)
                    rows = staging[l, b][phys[l, b, :len(lst)] - 128]
                    # a staged row is the pool row rounded to nearest fp16
                    assert np.array_equal(rows, pools[(l, b)][lst].astype(np.float16)), (t, l, b)
        st = ds.stats()
        assert st["hits"] == hits and st["misses"] == misses
        assert st["h2d_bytes"] == misses * 2048
        assert ds.check_error() == 0
    finally:
        ds.close()


def test_kvswap_stage_replays_evictions_of_later_listed_chunks():
    """Lists whose new chunks come first and whose last entries are the chunks
    in the least recently used slots: each of those slots is popped before its
    chunk's turn, which then misses too. Step 2 has 60 such evictions pending at
    once (more than the warp replay holds: the one-thread replay), step 3 has
    ten (the warp replay); both match the oracle's list LRU, rows included."""
    G_, k = 128, 128
    w = _w(context_len=4 * 1024, layer_ratios=(4,), gpu_chunks=G_, index_topk=k, code=57)
    ds = make_ds(w, max_select=k)
    try:
        pool = G.pool(w, 0, 0)
        fill(ds, w, {(0, 0): pool})
        st = O.KvSwapLayerState(w.layer_cap(0), G_)
        st.host_ready[:] = 1
        lists = [list(range(128)), list(range(200, 260)) + list(range(60)),
                 list(range(300, 310)) + list(range(60, 70)) + list(range(200, 230))]
        for t, ids in enumerate(lists):
            sel = np.zeros((1, ds.S), np.int32)
            sel[0, :len(ids)] = ids
            ds.sel.copy_(torch.from_numpy(sel))
            ds.count.copy_(torch.from_numpy(np.array([len(ids)], np.int32)))
            ds.stage()
            torch.cuda.synchronize()
            r = st.swap_in_selected(ids)
            phys = ds.phys.cpu().numpy()[0, 0, :len(ids)]
            assert phys.tolist() == r.phys, t
            rows = ds.staging.cpu().numpy()[0, 0][phys - 128]
            assert np.array_equal(rows, pool[ids].astype(np.float16)), t
        s_ = ds.stats()
        assert s_["misses"] == st.misses and s_["hits"] == st.hits
        assert ds.check_error() == 0
    finally:
        ds.close()


def test_kvswap_stage_chained_back_to_back_matches_list_lru():
    """Two kvswap_stage calls chained back to back on one stream (each with its
    own selection and outputs, written before the first is issued): the second
    resolve may start while the first still runs, and reads the LRU state again
    if it changed after its early read. Both calls' phys match the oracle's list
    LRU, applied in order, over eight rounds with in-step evictions."""
    from sparse_retrieval_host_gb300 import abi
    G_, k = 64, 48
    w = _w(context_len=4 * 600, layer_ratios=(4, 4, 8), gpu_chunks=G_, index_topk=k, batch=2, code=58)
    ds = make_ds(w, max_select=k)
    try:
        fill(ds, w)
        states = [[O.KvSwapLayerState(w.layer_cap(l), G_) for b in range(w.batch)] for l in range(w.n_layers)]
        for row in states:
            for st in row:
                st.host_ready[:] = 1
        rng = np.random.default_rng(58)
        traces = [_trace(rng, 16, w.n_chunks, k, G_) for _ in range(w.batch)]
        sels = [torch.zeros_like(ds.sel) for _ in range(2)]
        cnts = [torch.zeros_like(ds.count) for _ in range(2)]
        phys = [torch.zeros_like(ds.phys) for _ in range(2)]
        cls = [torch.zeros_like(ds.count_l) for _ in range(2)]
        for r in range(8):
            for i in range(2):
                sel = np.zeros(tuple(ds.sel.shape), np.int32)
                cnt = np.zeros(w.batch, np.int32)
                for b in range(w.batch):
                    ids = traces[b][2 * r + i]
                    sel[b, :len(ids)] = ids
                    cnt[b] = len(ids)
                sels[i].copy_(torch.from_numpy(sel))
                cnts[i].copy_(torch.from_numpy(cnt))
            torch.cuda.synchronize()
            abi.srh_set_chained(ds.ctx, True)
            try:
                for i in range(2):
                    abi.kvswap_stage(ds.ctx, -1, sels[i], cnts[i], ds.staging, phys[i], cls[i])
            finally:
                abi.srh_set_chained(ds.ctx, False)
            torch.cuda.synchronize()
            for i in range(2):
                ph = phys[i].cpu().numpy()
                for l in range(w.n_layers):
                    for b in range(w.batch):
                        lst = O.layer_chunks(traces[b][2 * r + i], 4, w.layer_ratios[l])
                        res = states[l][b].swap_in_selected(lst)
                        assert ph[l, b, :len(lst)].tolist() == res.phys, (r, i, l, b)
        assert ds.check_error() == 0
    finally:
        ds.close()


@pytest.mark.parametrize("G_,k,policy", [
    (64, 24, dict(g_min=24, g_max=64, g_init=32, epoch=2, lo_permille=600, hi_permille=850, delta=8)),
    (96, 32, dict(g_min=32, g_max=80, g_init=80, epoch=1, lo_permille=300, hi_permille=500, delta=16)),
    (512, 128, dict(g_min=128, g_max=512, g_init=128, epoch=3, lo_permille=700, hi_permille=900, delta=64)),
])
def test_kvswap_stage_adaptive_capacity_matches_oracle(G_, k, policy):
    """Adaptive staging capacity: per step the slots, misses, staged rows and
    the capacity in use match the oracle's resizable LRU under the same policy;
    removing the policy restores every slot."""
    ratios = (4, 128, 4, 8)
    w = _w(context_len=4 * 700, layer_ratios=ratios, gpu_chunks=G_, index_topk=k, batch=2, code=58)
    ds = make_ds(w, max_select=k)
    try:
        pools = {(l, b): G.pool(w, l, b) for l in range(w.n_layers) for b in range(w.batch)}
        fill(ds, w, pools)
        states = [[O.KvSwapLayerState(w.layer_cap(l), G_) for b in range(w.batch)] for l in range(w.n_layers)]
        pol = O.AdaptivePolicy(**policy)
        for row in states:
            for st in row:
                st.host_ready[:] = 1
                if st.swap_enabled:
                    st.install_policy(pol)
        ds.set_adaptive(policy)
        rng = np.random.default_rng(G_ + 7 * k)
        n_steps = 30
        traces = [_trace(rng, n_steps, w.n_chunks, k, G_) for _ in range(w.batch)]
        seen = set()
        for t in range(n_steps):
            if t == n_steps - 6:
                ds.set_adaptive(None)
                for row in states:
                    for st in row:
                        if st.swap_enabled:
                            st.install_policy(None)
            sel = np.zeros((w.batch, ds.S), np.int32)
            cnt = np.zeros(w.batch, np.int32)
            for b in range(w.batch):
                ids = traces[b][t]
                sel[b, :len(ids)] = ids
                cnt[b] = len(ids)
            ds.sel.copy_(torch.from_numpy(sel))
            ds.count.copy_(torch.from_numpy(cnt))
            ds.stage()
            torch.cuda.synchronize()
            phys = ds.phys.cpu().numpy()
            cl = ds.count_l.cpu().numpy()
            staging = ds.staging.cpu().numpy()
            active = ds.active_slots()
            for l in range(w.n_layers):
                for b in range(w.batch):
                    st = states[l][b]
                    lst = O.layer_chunks(traces[b][t], 4, ratios[l])
                    g = st.active_capacity()
                    if st.swap_enabled:
                        lst = lst[:g]
                    r = st.swap_in_selected(lst)
                    assert cl[l, b] == len(lst), (t, l, b)
                    assert phys[l, b, :len(lst)].tolist() == r.phys, (t, l, b)
                    rows = staging[l, b][phys[l, b, :len(lst)] - 128]
                    # a staged row is the pool row rounded to nearest fp16
                    assert np.array_equal(rows, pools[(l, b)][lst].astype(np.float16)), (t, l, b)
                    assert active[l][b] == (st.capacity if st.swap_enabled else w.layer_cap(l)), (t, l, b)
                    if st.swap_enabled:
                        seen.add(st.capacity)
        assert len(seen) > 1, "the policy never changed the capacity"
        assert all(active[l][b] == G_ for l in range(w.n_layers) for b in range(w.batch) if states[l][b].swap_enabled)
        assert ds.check_error() == 0
    finally:
        ds.close()


def test_kvswap_not_stored_is_reported():
    """Section 故障排查, error 4: a selected chunk that was never stored."""
    from sparse_retrieval_host_gb300 import abi
    w = _w(context_len=4 * 300, layer_ratios=(4, 128), gpu_chunks=64, index_topk=32, code=57)
    ds = make_ds(w, max_select=32)
    try:
        ds.mark_stored(0, 0, 0, 100)
        ds.mark_stored(1, 0)
        sel = torch.zeros((1, ds.S), dtype=torch.int32)
        sel[0, :3] = torch.tensor([5, 7, 99])
        ds.sel.copy_(sel)
        ds.count.fill_(3)
        ds.stage()
        assert ds.check_error() == abi.SRH_OK
        sel[0, :3] = torch.tensor([5, 150, 99])
        ds.sel.copy_(sel)
        ds.stage()
        assert ds.check_error() == abi.SRH_ERR_NOT_STORED
        assert ds.check_error() == abi.SRH_OK       # the word clears after it is read
    finally:
        ds.close()


def test_kvswap_rejects_a_second_staging_buffer():
    from sparse_retrieval_host_gb300 import abi
    w = _w(context_len=4 * 300, gpu_chunks=64, index_topk=32, code=58)
    ds = make_ds(w, max_select=32)
    try:
        ds.mark_stored(0, 0)
        ds.count.fill_(0)
        ds.stage()
        other = torch.zeros_like(ds.staging)
        with pytest.raises(abi.SrhError):
            abi.kvswap_stage(ds.ctx, -1, ds.sel, ds.count, other, ds.phys, ds.count_l)
    finally:
        ds.close()


# ----------------------------------------------------------------------------- lsa_attend
@pytest.mark.parametrize("H", [16, 32, 64])
@pytest.mark.parametrize("counts,batch_layers,per_layer", [((0, 1, 31, 32), 1, False),
                                                           ((33, 200, 512, 97), 1, False),
                                                           ((512,) * 8, 20, False),
                                                           ((0, 1, 300, 512, 77, 130, 511, 2), 20, False),
                                                           ((5, 512, 260, 0), 6, True)])
def test_lsa_attend_matches_oracle(H, counts, batch_layers, per_layer):
    """All layers in one call (one wave of pair chunks, or stream-K tile ranges
    when the pairs do not fit one wave, with counts below the planned rows) or one
    call per layer (the single-layer plans)."""
    from sparse_retrieval_host_gb300.runtime import bits_to_i16
    B = len(counts)
    L = batch_layers
    w = _w(context_len=8192, layer_ratios=(4,) * L, gpu_chunks=600, index_topk=512, n_heads=H,
           batch=B, code=59)
    ds = make_ds(w, max_select=512)
    try:
        rng = np.random.default_rng(H * 7 + B + L)
        stg = rng.standard_normal((L, B, 600, 512), dtype=np.float32)
        win = rng.standard_normal((L, B, 128, 512), dtype=np.float32)
        q = G.f32_to_bf16_bits(rng.standard_normal((L, B, H, 512), dtype=np.float32))
        phys = np.zeros((L, B, ds.S), np.int32)
        for l in range(L):
            for b in range(B):
                phys[l, b, :counts[b]] = 128 + rng.choice(600, size=counts[b], replace=False)
        ds.staging.copy_(torch.from_numpy(stg))
        ds.window.copy_(torch.from_numpy(win))
        ds.q.copy_(bits_to_i16(q))
        ds.phys.copy_(torch.from_numpy(phys))
        ds.count_l.copy_(torch.from_numpy(np.tile(np.int32(counts), (L, 1))))
        if per_layer:
            for l in range(L):
                ds.attend(l)
        else:
            ds.attend()
        out = ds.out.cpu().numpy()
        worst = 0.0
        for l in range(L):
            for b in range(B):
                rows = np.concatenate([win[l, b], stg[l, b][phys[l, b, :counts[b]] - 128]])
                ref = O.attend(q[l, b], rows)
                _, rel = attn_err(out[l, b], ref)
                worst = max(worst, rel)
        assert worst <= ATTN_TOL, worst
        assert ds.check_error() == 0
    finally:
        ds.close()


def _attend_case(H, counts, L, scales, seed):
    """lsa_attend on random rows, row block (l, b) scaled by scales[(l * B + b) % len]."""
    from sparse_retrieval_host_gb300.runtime import bits_to_i16
    B = len(counts)
    w = _w(context_len=8192, layer_ratios=(4,) * L, gpu_chunks=600, index_topk=512, n_heads=H, batch=B, code=63)
    ds = make_ds(w, max_select=512)
    rng = np.random.default_rng(seed)
    stg = rng.standard_normal((L, B, 600, 512), dtype=np.float32)
    win = rng.standard_normal((L, B, 128, 512), dtype=np.float32)
    for l in range(L):
        for b in range(B):
            f = np.float32(scales[(l * B + b) % len(scales)])
            stg[l, b] *= f
            win[l, b] *= f
    q = G.f32_to_bf16_bits(rng.standard_normal((L, B, H, 512), dtype=np.float32))
    phys = np.zeros((L, B, ds.S), np.int32)
    for l in range(L):
        for b in range(B):
            phys[l, b, :counts[b]] = 128 + rng.choice(600, size=counts[b], replace=False)
    ds.staging.copy_(torch.from_numpy(stg))
    ds.window.copy_(torch.from_numpy(win))
    ds.q.copy_(bits_to_i16(q))
    ds.phys.copy_(torch.from_numpy(phys))
    ds.count_l.copy_(torch.from_numpy(np.tile(np.int32(counts), (L, 1))))
    return ds, stg, win, q, phys


@pytest.mark.parametrize("scales", [(8e3,), (1e-4,), (8e3, 1e-4, 1.0)], ids=["large", "small", "mixed"])
def test_lsa_attend_rows_far_from_unit_scale(scales):
    """Latent rows far from O(1): |e| around 1e4 (near fp16's top) and around
    1e-4 (partly fp16-subnormal), within one call and mixed across pairs; the
    pairs are split over several CTAs, so the fp16 partials and the merge run."""
    H, counts, L = 64, (512, 300, 33), 2
    ds, stg, win, q, phys = _attend_case(H, counts, L, scales, seed=5)
    try:
        ds.attend()
        out = ds.out.cpu().numpy()
        worst = 0.0
        for l in range(L):
            for b in range(len(counts)):
                rows = np.concatenate([win[l, b], stg[l, b][phys[l, b, :counts[b]] - 128]])
                _, rel = attn_err(out[l, b], O.attend(q[l, b], rows))
                worst = max(worst, rel)
        assert worst <= ATTN_TOL, worst
        assert ds.check_error() == 0
    finally:
        ds.close()


@pytest.mark.parametrize("where", ["staged_row", "window_row", "query"])
def test_lsa_attend_reports_values_beyond_fp16(where):
    """A latent or query value beyond +-65504 cannot become an fp16 tensor-core
    operand: the call reports SRH_ERR_RANGE (the word clears once read), and a
    later call on finite-range inputs is clean."""
    from sparse_retrieval_host_gb300 import abi
    from sparse_retrieval_host_gb300.runtime import bits_to_i16
    ds, stg, win, q, phys = _attend_case(32, (200, 7), 1, (1.0,), seed=9)
    try:
        ds.attend()
        assert ds.check_error() == abi.SRH_OK
        if where == "staged_row":
            ds.staging[0, 1, int(phys[0, 1, 3]) - 128, 17] = 1e5
        elif where == "window_row":
            ds.window[0, 0, 5, 300] = -7e4
        else:
            qq = q.copy()
            qq[0, 1, 2, 9] = G.f32_to_bf16_bits(np.array([2e5], np.float32))[0]
            ds.q.copy_(bits_to_i16(qq))
        ds.attend()
        assert ds.check_error() == abi.SRH_ERR_RANGE
        assert ds.check_error() == abi.SRH_OK
        ds.staging.copy_(torch.from_numpy(stg))
        ds.window.copy_(torch.from_numpy(win))
        ds.q.copy_(bits_to_i16(q))
        ds.attend()
        assert ds.check_error() == abi.SRH_OK
    finally:
        ds.close()


def test_create_host_alloc_failure_frees_everything():
    """An injected pinned-pool allocation failure (the last layer's, after the
    earlier layers' pools and device tables exist) gives SRH_ERR_NOMEM, and the
    failed creations leave neither device memory nor pinned host memory behind."""
    import os
    from sparse_retrieval_host_gb300 import abi

    def rss_bytes():
        with open("/proc/self/statm") as f:
            return int(f.read().split()[1]) * os.sysconf("SC_PAGE_SIZE")

    ratios = [4, 4, 128]
    kw = dict(batch=2, layer_ratios=ratios, gpu_chunks=1024, index_topk=512, context_len=1 << 20)
    ok = abi.srh_create(abi.make_config(**kw))            # a context of this shape can be made
    abi.srh_destroy(ok)
    torch.cuda.synchronize()
    free0, rss0 = torch.cuda.mem_get_info()[0], rss_bytes()
    for _ in range(4):   # each attempt pins 2 pools of 1 GiB before it fails
        with pytest.raises(abi.SrhError) as ei:
            abi.srh_create(abi.make_config(flags=abi.SRH_FLAG_TEST_FAIL_HOST_ALLOC, **kw))
        assert ei.value.code == abi.SRH_ERR_NOMEM
        assert "injected" in str(ei.value)
    torch.cuda.synchronize()
    free1, rss1 = torch.cuda.mem_get_info()[0], rss_bytes()
    assert abs(free1 - free0) < (8 << 20), (free0, free1)
    assert rss1 - rss0 < (256 << 20), (rss0, rss1)       # four leaks would be 8 GiB
