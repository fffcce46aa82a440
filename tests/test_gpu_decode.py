"""End-to-end decode steps through the C ABI against the fp64 oracle, the
residency invariant, and the swap counters."""
import os

import numpy as np
import pytest
import torch

from srh_workload import configs as C
from srh_workload import generate as G

from helpers import (ATTN_TOL, attn_err, check_selection, fill, load_step_inputs, make_ds,
                     make_oracle, spec_of)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _run_decode(w, steps, attend_layers=None, pools=None, policy=None, attend_seqs=None):
    """Run ``steps`` decode steps on GPU and oracle; returns (n_matched_steps, worst_attn_rel).
    With ``policy`` both sides run the adaptive staging capacity. Attention and
    staged rows are checked on ``attend_layers`` x ``attend_seqs`` (all by
    default); selections, slots and counters on every sequence and layer."""
    ds = make_ds(w)
    try:
        if pools is None and w.n_chunks <= 8192:
            pools = {(l, b): G.pool(w, l, b) for l in range(w.n_layers) for b in range(w.batch)}
        keys = fill(ds, w, pools)
        ora = make_oracle(w)
        caps_seen = set()
        if policy is not None:
            ds.set_adaptive(policy)
            from oracle import srh_oracle as O
            ora.install_policy(O.AdaptivePolicy(**policy))
        spec = spec_of(w)
        # Exact slot/LRU comparisons need the same selection ORDER on both sides
        # since the first step; the order of chunks whose scores differ by less
        # than the fp32 scoring error is not unique, so once it differs only the
        # order-free facts are compared (sets, staged rows, attention outputs).
        order_sync = True
        worst = 0.0
        matched = 0
        hits = misses = 0
        if pools is not None:
            rows_of = lambda l, b, idx: pools[(l, b)][np.asarray(idx, dtype=np.int64)]
        else:
            rows_of = lambda l, b, idx: G.pool_rows(w, l, b, idx)
        layers = range(w.n_layers) if attend_layers is None else attend_layers
        seqs = range(w.batch) if attend_seqs is None else attend_seqs
        for t in range(steps):
            load_step_inputs(ds, w, t)
            ds.step(spec)
            torch.cuda.synchronize()
            pairs = [(l, b) for l in layers for b in seqs]
            ref = ora.step(lambda b: keys[b], lambda b: G.fm_queries(w, t, b),
                           lambda l, b: G.attn_q(w, t, l, b), lambda l, b: G.window(w, l, b),
                           rows_of, attend_pairs=pairs)
            scores = ds.scores.double().cpu().numpy()
            sel = ds.sel.cpu().numpy()
            cnt = ds.count.cpu().numpy()
            same = True
            for b in range(w.batch):
                same &= check_selection(w, ref.scores[b], ref.sel[b], sel[b, :cnt[b]], scores[b])
                order_sync &= np.array_equal(sel[b, :cnt[b]], ref.sel[b])
            order_sync &= same
            phys = ds.phys.cpu().numpy()
            cl = ds.count_l.cpu().numpy()
            active = ds.active_slots() if policy is not None else None
            for l in range(w.n_layers):
                for b in range(w.batch):
                    if active is not None and order_sync and ds.swap[l]:
                        assert active[l][b] == ora.states[l][b].capacity, (t, l, b)
                        caps_seen.add(active[l][b])
                    if same:
                        assert sorted(ref.lists[l][b]) == sorted(
                            set((sel[b, :cnt[b]].astype(np.int64) * 4 // w.layer_ratios[l]).tolist()))
                    if order_sync:
                        assert cl[l, b] == len(ref.lists[l][b])
                        assert phys[l, b, :cl[l, b]].tolist() == ref.swap[l][b].phys, (t, l, b)
                        if ds.swap[l]:
                            hits += ref.swap[l][b].hits
                            misses += len(ref.swap[l][b].misses)
            # staged rows always hold the pool rows of the GPU's own selection, rounded to fp16
            stg = ds.staging
            for l in list(layers)[:3]:
                for b in seqs:
                    n_l = int(cl[l, b])
                    got = stg[l, b][torch.from_numpy(phys[l, b, :n_l] - 128).long().cuda()].cpu().numpy()
                    lst = np.asarray(sorted(set(sel[b, :cnt[b]] * 4 // w.layer_ratios[l])), dtype=np.int64)
                    want_rows = np.asarray(rows_of(l, b, lst), dtype=np.float32).astype(np.float16)   # fp16 staging
                    assert sorted(map(bytes, got)) == sorted(map(bytes, want_rows))
            if same:
                matched += 1
                out = ds.out.cpu().numpy()
                for (l, b), r in ref.out.items():
                    _, rel = attn_err(out[l, b], r)
                    worst = max(worst, rel)
        if order_sync:
            st = ds.stats()
            assert st["hits"] == hits and st["misses"] == misses
        if policy is not None:
            assert len(caps_seen) > 1, caps_seen     # compared while the orders agreed
        assert ds.check_error() == 0
        return matched, worst
    finally:
        ds.close()


def test_decode_tiny_all_steps():
    w = C.TINY
    matched, worst = _run_decode(w, w.steps)
    assert matched == w.steps
    assert worst <= ATTN_TOL, worst


def test_decode_ctx8k_full_stack():
    w = C.CTX8K
    matched, worst = _run_decode(w, 40)
    assert matched == 40
    assert worst <= ATTN_TOL, worst


def test_decode_batch_sweep_b4():
    w = C.batch_sweep(4)
    matched, worst = _run_decode(w, 20, attend_layers=[0, 7, 19])
    assert matched == 20
    assert worst <= ATTN_TOL, worst


@pytest.mark.skipif(os.environ.get("SRH_SKIP_LARGE") == "1", reason="large configs skipped")
@pytest.mark.parametrize("batch,steps,seqs", [(16, 4, (0, 9, 15)), (32, 3, (0, 17, 31))])
def test_decode_batch_sweep_large(batch, steps, seqs):
    """The batch rows where one step runs the tensor-core scoring kernel (2^18
    chunks and more per call) and the stream-K attention plan (more tiles than
    SMs) together: selections, slots and counters of every sequence and layer;
    attention and staged rows on sampled layers and sequences."""
    w = C.batch_sweep(batch)
    assert w.batch * w.n_chunks >= 1 << 18
    matched, worst = _run_decode(w, steps, attend_layers=[0, 11, 19], attend_seqs=seqs)
    assert matched == steps
    assert worst <= ATTN_TOL, worst


def test_decode_ctx8k_adaptive_capacity():
    """Adaptive staging capacity over the full 8K stack: per step the capacity
    in use, the slots and the outputs match the oracle under the same policy."""
    w = C.CTX8K
    policy = dict(g_min=512, g_max=1024, g_init=1024, epoch=4, lo_permille=800, hi_permille=950, delta=128)
    matched, worst = _run_decode(w, 40, attend_layers=[0, 19, 20, 40], policy=policy)
    assert matched == 40
    assert worst <= ATTN_TOL, worst


@pytest.mark.skipif(os.environ.get("SRH_SKIP_LARGE") == "1", reason="large configs skipped")
def test_decode_ctx256k_sampled():
    w = C.CTX256K
    matched, worst = _run_decode(w, 20, attend_layers=[0, 19, 20, 40])
    assert matched == 20
    assert worst <= ATTN_TOL, worst


@pytest.mark.skipif(os.environ.get("SRH_SKIP_LARGE") == "1", reason="large configs skipped")
def test_decode_ctx1m_sampled():
    w = C.CTX1M
    matched, worst = _run_decode(w, 12, attend_layers=[0, 20, 40])
    assert matched == 12
    assert worst <= ATTN_TOL, worst


def test_residency_changes_slots_never_outputs():
    """kestrel-llm-cuda 06, section 3.4 and the FlashMemory doc's 验证状态: swapping
    changes which slots hold a chunk, never the outputs (bitwise)."""
    swapped = C.TINY
    resident = swapped.with_(gpu_chunks=2048)
    outs = []
    for w in (swapped, resident):
        ds = make_ds(w)
        try:
            fill(ds, w)
            spec = spec_of(w)
            seq = []
            for t in range(w.steps):
                load_step_inputs(ds, w, t)
                ds.step(spec)
                seq.append(ds.out.clone())
            st = ds.stats()
            outs.append((torch.stack(seq).cpu(), st, ds.swap[0]))
        finally:
            ds.close()
    (a, sa, swa), (b, sb, swb) = outs
    assert swa and not swb
    assert sa["misses"] > 0 and sb["misses"] == 0
    assert torch.equal(a, b)


@pytest.mark.parametrize("parts,adaptive", [(False, False), (True, False), (False, True)],
                         ids=["one_graph", "three_graphs", "one_graph_adaptive"])
def test_graph_replay_equals_eager_steps(parts, adaptive):
    """Steps replayed from captured CUDA graphs give the same bits as eager
    calls (chained, through step(), and unchained, call by call): selections,
    slots, staged rows, outputs and the swap counters; with the adaptive
    capacity also the capacity decided on the device each step."""
    w = C.TINY.with_(steps=12)
    policy = None
    if adaptive:
        w = w.with_(gpu_chunks=1024, lookahead=4)
        policy = dict(g_min=512, g_max=1024, g_init=768, epoch=2, lo_permille=700, hi_permille=900, delta=128)
    runs = []
    for mode in ("eager", "graph", "unchained"):
        ds = make_ds(w)
        try:
            fill(ds, w)
            spec = spec_of(w)
            if policy is not None:
                ds.set_adaptive(policy)
            load_step_inputs(ds, w, 0)
            ds.step(spec)                       # one eager step before capture
            graphs = ds.capture(spec, parts=parts) if mode == "graph" else None
            seq = []
            for t in range(1, w.steps):
                load_step_inputs(ds, w, t)
                if mode == "unchained":
                    ds.score(spec)
                    ds.select(spec)
                    ds.stage(-1)
                    ds.attend(-1)
                elif graphs is None:
                    ds.step(spec)
                else:
                    for g in graphs:
                        g.replay()
                torch.cuda.synchronize()
                seq.append([x.clone() for x in (ds.sel, ds.count, ds.phys, ds.count_l, ds.out)])
                if policy is not None:
                    seq[-1].append(torch.tensor(ds.active_slots()))
            st = ds.stats()
            runs.append((seq, st["hits"], st["misses"], ds.staging.clone()))
            assert ds.check_error() == 0
        finally:
            ds.close()
    (sa, ha, ma, ga) = runs[0]
    for (sb, hb, mb, gb) in runs[1:]:
        assert (ha, ma) == (hb, mb)
        assert torch.equal(ga, gb)
        for xa, xb in zip(sa, sb):
            for a, b in zip(xa, xb):
                assert torch.equal(a, b)


def test_ties_follow_index_order():
    """Duplicated keys give exactly equal scores; both sides break ties by index."""
    from sparse_retrieval_host_gb300.runtime import bits_to_i16
    from oracle import srh_oracle as O
    w = C.TINY
    ds = make_ds(w)
    try:
        base = G.keys(w, 0)
        keys = base[np.arange(w.n_chunks) % 100]
        ds.keys[0] = bits_to_i16(keys)
        for t in (0, 8):
            ds.fm_q[0] = bits_to_i16(G.fm_queries(w, t, 0))
            ds.score(spec_of(w))
            ds.select(spec_of(w))
            ref_s = O.score(keys, G.fm_queries(w, t, 0), w.scale, [0.0] * 3, w.ensemble)
            ref = O.select_topk(ref_s, w.index_topk)
            got = ds.sel[0, :int(ds.count[0])].cpu().numpy()
            assert np.array_equal(np.sort(got), np.sort(ref))
            g = ds.scores[0].double().cpu().numpy()
            assert all(g[c] == g[c % 100] for c in range(w.n_chunks))
    finally:
        ds.close()


def test_device_wait_timeout_is_reported_and_context_stays_usable():
    """The kernels' bounded-wait path on its own: a wait that nothing completes gives
    up after its limit (wall-clock), the host reads SRH_ERR_TIMEOUT once, and the
    context's later steps equal, bit for bit, those of a context that never timed out."""
    import time
    from sparse_retrieval_host_gb300 import abi
    w = C.TINY
    results = []
    for inject in (False, True):
        ds = make_ds(w)
        try:
            fill(ds, w)
            spec = spec_of(w)
            for t in range(3):
                load_step_inputs(ds, w, t)
                if inject and t == 1:
                    torch.cuda.synchronize()
                    t0 = time.perf_counter()
                    abi.srh_selftest_wait_timeout(ds.ctx, 20000)
                    assert ds.check_error() == abi.SRH_ERR_TIMEOUT
                    waited = time.perf_counter() - t0
                    assert 0.015 <= waited < 5.0, waited
                    assert ds.check_error() == abi.SRH_OK   # the word was cleared
                ds.step(spec)
                torch.cuda.synchronize()
            assert ds.check_error() == abi.SRH_OK
            results.append([x.clone() for x in (ds.out, ds.sel, ds.count, ds.phys, ds.count_l)])
        finally:
            ds.close()
    for a, b in zip(*results):
        assert torch.equal(a, b)


def test_max_sizes_select_and_stage():
    """Largest supported S and G (4096) on one layer."""
    w = C.Workload(name="max", code=60, context_len=4 * 20000, layer_ratios=(4,), gpu_chunks=4096,
                   index_topk=4096, ensemble=C.ENSEMBLE_MAX, select_mode=C.SELECT_TOPK, tau=0.5,
                   bias=0.0, n_heads=64, batch=1, steps=3, lookahead=1)
    matched, worst = _run_decode(w, 3)
    assert matched == 3
    assert worst <= ATTN_TOL


def _lookahead_run(w, steps, attend_layers, graph):
    """The lookahead schedule on the GPU (eager or graph replays) beside the
    oracle's; returns per-step outputs and the number of steps compared."""
    ds = make_ds(w)
    try:
        pools = {(l, b): G.pool(w, l, b) for l in range(w.n_layers) for b in range(w.batch)}
        keys = fill(ds, w, pools)
        ora = make_oracle(w)
        spec = spec_of(w)
        rows_of = lambda l, b, idx: pools[(l, b)][np.asarray(idx, dtype=np.int64)]
        graphs = None
        outs, compared = [], 0
        in_force_same = True           # the GPU's selection in force has the oracle's set
        order_sync = True
        for t in range(steps):
            trig = t % w.lookahead == 0
            load_step_inputs(ds, w, t)
            if graph and graphs is None and t >= 1:
                graphs = ds.capture_lookahead(spec)
            if graphs is not None:
                ds.replay_lookahead(graphs, trig)
            else:
                ds.lookahead_step(spec, trig)
            torch.cuda.synchronize()
            outs.append(ds.out.clone())
            pairs = [(l, b) for l in attend_layers for b in range(w.batch)]
            ref = ora.lookahead_step(lambda b: keys[b], lambda b: G.fm_queries(w, t, b),
                                     lambda l, b: G.attn_q(w, t, l, b), lambda l, b: G.window(w, l, b),
                                     rows_of, attend_pairs=pairs, trigger=trig)
            if in_force_same:
                out = ds.out.cpu().numpy()
                for (l, b), r in ref.out.items():
                    _, rel = attn_err(out[l, b], r)
                    assert rel <= ATTN_TOL, (t, l, b, rel)
                compared += 1
            if trig:
                scores = ds.scores.double().cpu().numpy()
                sel = ds.sel.cpu().numpy()
                cnt = ds.count.cpu().numpy()
                same = True
                for b in range(w.batch):
                    same &= check_selection(w, ref.scores[b], ref.sel[b], sel[b, :cnt[b]], scores[b])
                    order_sync &= np.array_equal(sel[b, :cnt[b]], ref.sel[b])
                order_sync &= same
                in_force_same = same
                nxt = ds.in_force                 # the buffer the new selection was staged into
                phys = ds.phys2[nxt].cpu().numpy()
                cl = ds.count_l2[nxt].cpu().numpy()
                for l in range(w.n_layers):
                    for b in range(w.batch):
                        if order_sync:
                            assert cl[l, b] == len(ref.swap[l][b].phys)
                            assert phys[l, b, :cl[l, b]].tolist() == ref.swap[l][b].phys, (t, l, b)
        assert ds.check_error() == 0
        return outs, compared
    finally:
        ds.close()


def test_lookahead_schedule_matches_oracle():
    """Lookahead schedule over the 8K stack: the step's attention reads the
    selection in force while the new one is swapped in on a side stream; the
    outputs and the new slots match the oracle's schedule, and graph replays
    give the same bits as eager steps."""
    w = C.CTX8K.with_(lookahead=4)
    eager, n_cmp = _lookahead_run(w, 14, [0, 19, 20, 40], graph=False)
    assert n_cmp >= 10
    replay, _ = _lookahead_run(w, 14, [0, 40], graph=True)
    for a, b in zip(eager, replay):
        assert torch.equal(a, b)


def test_lookahead_needs_two_selections_of_slots():
    w = C.TINY                                     # GPU_CHUNKS = index_topk = 512
    ds = make_ds(w)
    try:
        fill(ds, w)
        with pytest.raises(ValueError):
            ds.lookahead_step(spec_of(w), True)
    finally:
        ds.close()


@pytest.mark.parametrize("ctx_len", [8192, 4 * 32768], ids=["n2048", "n32768_candidates"])
def test_replay_after_unconsumed_scoring_selects_right(ctx_len):
    """A graph captured while the score histogram was clean has no clearing
    step. If an eager scoring pass that no selection consumed runs before the
    replay, the replay's histogram counts keys twice; the select kernel (and
    the candidate pass) must notice and rebuild rather than select wrongly."""
    from sparse_retrieval_host_gb300 import abi
    w = C.TINY.with_(context_len=ctx_len)
    ds = make_ds(w)
    try:
        fill(ds, w)
        spec = spec_of(w)
        load_step_inputs(ds, w, 0)
        ds.step(spec)
        (g,) = ds.capture(spec)
        load_step_inputs(ds, w, 9)
        ds.score(spec)                      # scored, never selected
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        sel, cnt = ds.sel.clone(), ds.count.clone()
        ref_sel = torch.zeros_like(ds.sel)
        ref_cnt = torch.zeros_like(ds.count)
        abi.fm_select_noalloc(ds.scores, w.batch, ds.n, spec.select_mode, spec.k, spec.tau, spec.clamp, ds.S,
                              ref_sel, ref_cnt)
        torch.cuda.synchronize()
        assert torch.equal(cnt, ref_cnt)
        for b in range(w.batch):
            assert torch.equal(sel[b, :cnt[b]], ref_sel[b, :cnt[b]])
        assert ds.check_error() == 0
    finally:
        ds.close()


def test_host_loop_matches_eager_steps():
    """runtime.HostLoop and the library's native loop (srh_hostloop_*, through
    runtime.NativeHostLoop) -- pinned host inputs and outputs, copies of
    neighbouring steps overlapping the step in flight -- give, step for step,
    the bits of eager steps fed through the bound buffers."""
    from sparse_retrieval_host_gb300.runtime import HostLoop, NativeHostLoop, bits_to_i16
    w = C.TINY.with_(steps=10)
    n = 9
    h_fmq = [bits_to_i16(np.stack([G.fm_queries(w, t, b) for b in range(w.batch)])).pin_memory() for t in range(n)]
    h_q = [bits_to_i16(np.stack([np.stack([G.attn_q(w, t, l, b) for b in range(w.batch)])
                                 for l in range(w.n_layers)])).pin_memory() for t in range(n)]
    runs = []
    for mode in ("eager", "loop", "native"):
        ds = make_ds(w)
        try:
            fill(ds, w)
            spec = spec_of(w)
            load_step_inputs(ds, w, 0)
            ds.step(spec)                                   # set-up step
            outs = []
            if mode == "eager":
                for t in range(1, n):
                    ds.fm_q.copy_(h_fmq[t])
                    ds.q.copy_(h_q[t])
                    ds.step(spec)
                    outs.append((ds.out.cpu(), ds.sel.cpu(), ds.count.cpu()))
            else:
                loop = HostLoop(ds, spec) if mode == "loop" else NativeHostLoop(ds, spec)
                bufs = [(torch.empty(ds.out.shape).pin_memory(), torch.empty(ds.sel.shape, dtype=torch.int32).pin_memory(),
                         torch.empty(ds.count.shape, dtype=torch.int32).pin_memory()) for _ in range(1, n)]
                for i, t in enumerate(range(1, n)):
                    loop.step(i, h_fmq[t], h_q[t], *bufs[i])
                if mode == "native":
                    loop.wait(n - 3)                        # the second-to-last step's outputs
                loop.synchronize()
                if mode == "native":
                    loop.close()
                outs = bufs
            assert ds.check_error() == 0
            runs.append(outs)
        finally:
            ds.close()
    for run in runs[1:]:                                     # each loop against the eager steps
        for a, b in zip(runs[0], run):
            for x, y in zip(a, b):
                assert torch.equal(x, y)
