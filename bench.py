#!/usr/bin/env python3
"""Decode-step benchmark of the FlashMemory LSA + KV_SWAP hot path on GB300.

One "step" is one pass of the whole hot path -- fm_score, fm_select,
kvswap_stage (LRU resolve + miss gather) and lsa_attend over all sparse
layers -- for one batch of synthetic input, with inputs already resident in
HBM. Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config ctx8k]
  python bench.py --impl reference ...   # the fp64 CPU oracle, timed on the host

Timing: W warm-up steps, then K timed steps; the L2 is flushed before every
timed step (a 256 MiB buffer is written, then read back, so the L2 holds only
clean lines of it and the timed kernels pay no write-back of the flush), and
each step is bracketed by CUDA events on its stream, so the flush is outside
the timed spans. Multi-GPU (N > 1 under
torchrun) runs N independent replicas (weak scaling, no collective on the
data path); value = steps of all ranks / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from srh_workload import configs as C  # noqa: E402
from srh_workload import generate as G  # noqa: E402

TC_SCORE_MIN_CHUNKS = 1 << 18  # fm_score's tensor-core kernel from this many chunks per call (all sequences)
HOLD_CYCLES = 400_000          # ~0.2 ms device-side wait before eagerly timed calls
BASE_KERNELS = 5              # score, select, lru, gather, attend (+ the candidate pass)
COLLECT_MIN_N = 16384         # fm_select runs its candidate pass above this many chunks
Q_CYCLE = 16                  # distinct attention-query sets cycled through the steps
FLUSH_BYTES = 256 << 20       # > 2x the 126 MiB L2
METRIC = "decode steps/s"
SWEEP = ("ctx256k", "ctx1m", "batch128k_b1", "batch128k_b4", "batch128k_b8", "batch128k_b16", "batch128k_b32")
DTYPE = "bf16 scoring / fp16 attention operands / fp32 accumulate"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="ctx8k", choices=sorted(C.ALL))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample-steps", type=int, default=0, help="0 = auto")
    ap.add_argument("--quiet", action="store_true")
    ap.add_argument("--no-sweep", action="store_true", help="skip the other workloads' sub-records")
    ap.add_argument("--sweep", default=",".join(SWEEP), help="workloads measured beside the headline")
    ap.add_argument("--oracle-seconds", type=int, default=0, help=argparse.SUPPRESS)
    return ap.parse_args()


# --------------------------------------------------------------------------- distributed
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = os.environ.get("SRH_DIST_BACKEND", "nccl")
        dist.init_process_group(backend)
        return dist, rank, world, local
    return None, 0, 1, 0


def aggregate(dist, local_seconds: float, local_steps: int, device=None):
    """Max of the timed seconds and sum of the steps over ranks."""
    if dist is None:
        return local_seconds, local_steps
    import torch
    t = torch.tensor([local_seconds], dtype=torch.float64, device=device)
    s = torch.tensor([float(local_steps)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(s, op=dist.ReduceOp.SUM)
    return float(t.item()), int(s.item())


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 8:
                continue
            try:
                sm.append(float(p[0]))
                mx.append(float(p[1]))
            except ValueError:
                continue
            for nm, v in zip(names, p[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- peaks
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def code_hash(path: str) -> str:
    """sha256 (first 16 hex digits) of a C++/CUDA source with its comments and
    whitespace removed: a change to the code changes it, a change to the
    comments does not. String and character literals are kept as they are."""
    src = open(path, encoding="utf-8").read()
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            if not c.isspace():
                out.append(c)
            i += 1
    return hashlib.sha256("".join(out).encode("utf-8")).hexdigest()[:16]


def traffic_record(kernel: str, workload: str):
    """Measured DRAM bytes per launch from an ncu capture of this workload, if the
    kernel's code is unchanged since (profiles/traffic.json keys it by
    code_hash of the source and names the workload it was taken on)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f).get(kernel)
    if not rec or rec.get("workload") != workload:
        return None
    src = os.path.join(ROOT, "sparse_retrieval_host_gb300", "csrc", rec["source"])
    return rec if code_hash(src) == rec.get("source_code_hash") else None


# --------------------------------------------------------------------------- setup
def setup(w, device):
    import torch
    from sparse_retrieval_host_gb300.runtime import DecodeStep, StepSpec, bits_to_i16
    ds = DecodeStep(batch=w.batch, layer_ratios=w.layer_ratios, gpu_chunks=w.gpu_chunks,
                    index_topk=w.index_topk, context_len=w.context_len, n_heads=w.n_heads,
                    max_select=w.clamp)
    for l in range(w.n_layers):
        for b in range(w.batch):
            G.fill_pool(w, l, b, ds.pool_view(l, b))
            ds.mark_stored(l, b)
            ds.window[l, b] = torch.from_numpy(G.window(w, l, b))
    for b in range(w.batch):
        ds.keys[b] = bits_to_i16(G.keys(w, b))
    n_win = (w.steps + w.lookahead - 1) // w.lookahead
    fmq = np.stack([np.stack([G.fm_queries(w, i * w.lookahead, b) for b in range(w.batch)])
                    for i in range(n_win)])
    fm_q_all = bits_to_i16(fmq).to(device)
    nq = min(Q_CYCLE, w.steps)
    qs = np.stack([np.stack([np.stack([G.attn_q(w, t, l, b) for b in range(w.batch)])
                             for l in range(w.n_layers)]) for t in range(nq)])
    q_all = bits_to_i16(qs).to(device)
    spec = StepSpec(w.scale, [w.bias] * 3, w.ensemble, w.select_mode, w.index_topk, w.tau, w.clamp)
    return ds, spec, fm_q_all, q_all


def attn_bytes(w, count_l):
    """Algorithmic bytes of one lsa_attend launch with the pages' fp32 rows
    (2048 B per window or staged row) + q read + out written."""
    rows = count_l.sum() + w.n_layers * w.batch * C.WINDOW
    return int(rows) * C.KV_DIM * 4 + w.n_layers * w.batch * w.n_heads * C.KV_DIM * (2 + 4)


def attn_layout_bytes(w, count_l):
    """Bytes one lsa_attend launch must move with this layout: fp32 window rows
    (2048 B), fp16 staged rows (1024 B), q read and out written."""
    window = w.n_layers * w.batch * C.WINDOW
    return (window * C.KV_DIM * 4 + int(count_l.sum()) * C.KV_DIM * 2
            + w.n_layers * w.batch * w.n_heads * C.KV_DIM * (2 + 4))


def scoring_kernel(w) -> str:
    """Which fm_score kernel a call of this workload runs (one key set)."""
    if w.batch * w.n_chunks >= TC_SCORE_MIN_CHUNKS:
        return "score_tc_kernel (TMA + tcgen05)"
    return "score_kernel<1> (mma.sync)"


def launches_per_step(w, sm_count):
    """Our kernels per step: score, select, resolve, gather and attend (the
    attention kernel merges split pairs itself), plus fm_select's candidate
    pass when the workload scores more than COLLECT_MIN_N chunks; the gather
    runs only when some layer swaps (its capacity exceeds GPU_CHUNKS)."""
    collect = 1 if w.n_chunks > COLLECT_MIN_N else 0
    swapped = any(-(-w.context_len // r) > w.gpu_chunks for r in w.layer_ratios)
    return BASE_KERNELS + collect - (0 if swapped else 1)


def adaptive_policy(w):
    """Hit-rate policy for the adaptive-capacity run: from GPU_CHUNKS down to
    index_topk slots, one decision per lookahead window, shrink above a 90 %
    hit rate, grow below 80 %. None when the workload leaves no room."""
    swapped = any(-(-w.context_len // r) > w.gpu_chunks for r in w.layer_ratios)
    if not swapped or w.gpu_chunks <= w.index_topk:
        return None
    return dict(g_min=w.index_topk, g_max=w.gpu_chunks, g_init=w.gpu_chunks, epoch=w.lookahead,
                lo_permille=800, hi_permille=900, delta=max(1, w.gpu_chunks // 8))


def pass_bytes(w):
    """Algorithmic bytes of the scoring + selection pass: keys, the score write and
    up to two reads of the scores by the selection."""
    return w.batch * w.n_chunks * (C.INDEXER_DIM * 2 + 12)


def score_bytes(w):
    return w.batch * w.n_chunks * (C.INDEXER_DIM * 2 + 4)


# --------------------------------------------------------------------------- our arm
def run_ours(args, dist, rank, world, local):
    import torch
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    import __graft_entry__
    __graft_entry__.build()
    w = C.get(args.config)
    ds, spec, fm_q_all, q_all = setup(w, device)
    stream = torch.cuda.current_stream()
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=device)

    def bind(t):
        # the step's inputs into the buffers the graphs read (outside the timed span)
        ds.fm_q.copy_(fm_q_all[(t % w.steps) // w.lookahead])
        ds.q.copy_(q_all[t % q_all.shape[0]])

    def flush_l2():
        flush.zero_()
        flush.sum()

    for t in range(args.warmup):
        bind(t)
        ds.step(spec, stream)
    torch.cuda.synchronize()
    assert ds.check_error() == 0, "device error during warm-up"
    (graph,) = ds.capture(spec)
    parts = ds.capture(spec, parts=True)
    ds.reset_stats()

    # headline: K steps, each one graph launch, timed on the stream
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    with ClockSampler(local) as clk:
        for i in range(K):
            bind(args.warmup + i)
            flush_l2()
            ev[i][0].record(stream)
            graph.replay()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    assert ds.check_error() == 0, "device error during the timed steps"
    step_ms = [e0.elapsed_time(e1) for e0, e1 in ev]
    st = ds.stats()
    # the same steps with a warm L2 (no flush between them), for comparison only
    evw = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for i in range(K):
        bind(args.warmup + i)
        evw[i][0].record(stream)
        graph.replay()
        evw[i][1].record(stream)
    torch.cuda.synchronize()
    warm_ms = [e0.elapsed_time(e1) for e0, e1 in evw]

    # periodic selection: the memory indexer scores once per lookahead window and
    # the steps in between reuse the selection (same outputs for these inputs)
    (graph_reuse,) = ds.capture(spec, rescore=False)
    KP = K
    evp = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(KP)]
    for i in range(KP):
        t = args.warmup + K + i
        bind(t)
        flush_l2()
        evp[i][0].record(stream)
        (graph if t % w.lookahead == 0 else graph_reuse).replay()
        evp[i][1].record(stream)
    torch.cuda.synchronize()
    assert ds.check_error() == 0, "device error during the periodic-selection steps"
    periodic_ms = [e0.elapsed_time(e1) for e0, e1 in evp]

    # lookahead schedule: a trigger step swaps in its new selection on a side
    # stream while its attention reads the selection in force (not the headline:
    # the selection takes effect one step later)
    lookahead = None
    m_sel = w.index_topk if w.select_mode == C.SELECT_TOPK else w.clamp
    if w.gpu_chunks >= 2 * m_sel or not any(ds.swap):
        t0 = args.warmup + K + KP
        ds.lookahead_step(spec, True)             # eager first step (buffers, set-up)
        torch.cuda.synchronize()
        lgraphs = ds.capture_lookahead(spec)
        evl = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
        for i in range(K):
            t = t0 + 1 + i
            bind(t)
            flush_l2()
            evl[i][0].record(stream)
            ds.replay_lookahead(lgraphs, t % w.lookahead == 0)
            evl[i][1].record(stream)
        torch.cuda.synchronize()
        assert ds.check_error() == 0, "device error during the lookahead-schedule steps"
        la_ms = [e0.elapsed_time(e1) for e0, e1 in evl]
        trig_ms = [m for i, m in enumerate(la_ms) if (t0 + 1 + i) % w.lookahead == 0]
        lookahead = {
            "value": K / (sum(la_ms) / 1e3), "unit": "steps/s", "ms_per_step": statistics.mean(la_ms),
            "trigger_step_us": statistics.mean(trig_ms) * 1e3 if trig_ms else None,
            "note": f"indexer fires every {w.lookahead} steps; at a trigger step score + select + swap-in "
                    "run on a side stream beside the attention over the selection in force; the other "
                    "steps run the attention alone; one graph per step"}
    else:
        lookahead = {"value": None, "note": f"needs gpu_chunks >= {2 * m_sel} (two selections in flight)"}

    # adaptive staging capacity: the same steps with the hit-rate policy deciding
    # on the device; the policy is a launch argument, so the step is captured again
    adaptive = None
    policy = adaptive_policy(w)
    if policy is not None:
        ds.set_adaptive(policy)
        (graph_ad,) = ds.capture(spec)
        t0 = args.warmup + K + KP
        settle = 6 * policy["epoch"]
        for i in range(settle):                       # let the capacity settle (untimed)
            bind(t0 + i)
            graph_ad.replay()
        torch.cuda.synchronize()
        ds.reset_stats()
        eva = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
        for i in range(K):
            bind(t0 + settle + i)
            flush_l2()
            eva[i][0].record(stream)
            graph_ad.replay()
            eva[i][1].record(stream)
        torch.cuda.synchronize()
        assert ds.check_error() == 0, "device error during the adaptive-capacity steps"
        sta = ds.stats()
        act = ds.active_slots()
        swapped = [act[l][b] for l in range(ds.L) for b in range(ds.B) if ds.swap[l]]
        ada_ms = [e0.elapsed_time(e1) for e0, e1 in eva]
        sel_a = sta["hits"] + sta["misses"]
        adaptive = {
            "value": K / (sum(ada_ms) / 1e3), "unit": "steps/s", "ms_per_step": statistics.mean(ada_ms),
            "policy": policy,
            "lru_hit_rate": (sta["hits"] / sel_a) if sel_a else None,
            "staged_bytes_per_step": sta["h2d_bytes"] / K,
            "mean_active_slots": statistics.mean(swapped),
            "gpu_chunks": w.gpu_chunks,
            "staging_bytes_in_use": sum(swapped) * C.KV_DIM * 2,
            "staging_bytes_allocated": len(swapped) * w.gpu_chunks * C.KV_DIM * 2,
            "note": f"srh_set_adaptive; {settle} settling steps, then {K} timed steps of one graph each; "
                    "slots in use read after the timed steps"}
        ds.set_adaptive(None)

    # breakdown: the same steps as three graphs with events between the phases
    KB = min(K, 20)
    evb = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(KB)]
    counts, sel_counts = [], []
    for i in range(KB):
        bind(args.warmup + K + KP + i)
        flush_l2()
        e0, e1, e2, e3 = evb[i]
        e0.record(stream)
        parts[0].replay()
        e1.record(stream)
        parts[1].replay()
        e2.record(stream)
        parts[2].replay()
        e3.record(stream)
        e3.synchronize()
        counts.append(ds.count_l.cpu().numpy().copy())
        sel_counts.extend(int(c) for c in ds.count.cpu().numpy())
    assert ds.check_error() == 0, "device error during the breakdown steps"
    score_ms = [e[0].elapsed_time(e[1]) for e in evb]

    # the scoring + selection pass alone, eager calls queued behind the L2 flush and
    # a short device-side wait (the device is still busy when they are issued, so
    # the event spans are device time, without host or graph-launch latency)
    # The same for the whole step, call by call: these spans are the per-call
    # device times; the attention call's is the roofline's launch duration.
    sp_score, sp_select, sp_stage, sp_attn, sp_counts = [], [], [], [], []
    for i in range(10):
        bind(args.warmup + K + KP + KB + i)
        flush_l2()
        torch.cuda._sleep(HOLD_CYCLES)                  # the calls below are all queued before the GPU gets to them
        q = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        q[0].record(stream)
        ds.score(spec, stream)
        q[1].record(stream)
        ds.select(spec, stream)
        q[2].record(stream)
        ds.stage(-1, stream)
        q[3].record(stream)
        ds.attend(-1, stream)
        q[4].record(stream)
        q[4].synchronize()
        if i >= 2:
            sp_score.append(q[0].elapsed_time(q[1]))
            sp_select.append(q[1].elapsed_time(q[2]))
            sp_stage.append(q[2].elapsed_time(q[3]))
            sp_attn.append(q[3].elapsed_time(q[4]))
            sp_counts.append(ds.count_l.cpu().numpy().copy())

    ch_us = chained_pass_us(ds, spec, stream, flush, bind, args.warmup + K + KP + KB + 10)

    # one key set per memory indexer (fm_score_multi): the scoring call alone
    from sparse_retrieval_host_gb300 import abi
    keys3 = torch.empty((3,) + tuple(ds.keys.shape), dtype=ds.keys.dtype, device=device)
    keys3[:] = ds.keys
    multi_ms = []
    for i in range(6):
        flush_l2()
        torch.cuda._sleep(HOLD_CYCLES)
        m0, m1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        m0.record(stream)
        abi.fm_score_multi(ds.ctx, keys3, ds.n, ds.fm_q, spec.scale, spec.bias, spec.ensemble, ds.scores, stream)
        m1.record(stream)
        m1.synchronize()
        if i >= 1:
            multi_ms.append(m0.elapsed_time(m1))
    del keys3

    # fp8 (e4m3) indexer keys with per-chunk scales (fm_score_fp8): the scoring call alone
    codes = torch.empty(tuple(ds.keys.shape), dtype=torch.uint8, device=device)
    kscale = torch.empty(tuple(ds.keys.shape[:2]), dtype=torch.float32, device=device)
    abi.fm_quantize_keys(ds.ctx, ds.keys, ds.n, codes, kscale, stream)
    fp8_ms = []
    for i in range(6):
        flush_l2()
        torch.cuda._sleep(HOLD_CYCLES)
        m0, m1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        m0.record(stream)
        abi.fm_score_fp8(ds.ctx, codes, kscale, ds.n, ds.fm_q, spec.scale, spec.bias, spec.ensemble, ds.scores,
                         stream)
        m1.record(stream)
        m1.synchronize()
        if i >= 1:
            fp8_ms.append(m0.elapsed_time(m1))
    del codes, kscale
    stage_ms = [e[1].elapsed_time(e[2]) for e in evb]
    attn_ms = [e[2].elapsed_time(e[3]) for e in evb]
    local_s = sum(step_ms) / 1e3
    tot_s, tot_steps = aggregate(dist, local_s, K, device)

    result = None
    if rank == 0:
        peak, peak_kind = measured_peaks()
        a_bytes = [attn_bytes(w, c) for c in sp_counts]
        l_bytes = statistics.mean(attn_layout_bytes(w, c) for c in sp_counts)
        a_avg_ms = statistics.mean(sp_attn)
        achieved = statistics.mean(a_bytes) / (a_avg_ms / 1e3) / 1e9
        sel_total = st["hits"] + st["misses"]
        step_bytes = statistics.mean(a_bytes) + score_bytes(w)
        traffic = traffic_record("attend", w.name)
        result = {
            "metric": METRIC,
            "value": tot_steps / tot_s,
            "unit": "steps/s",
            "n_gpus": world,
            "steps": K,
            "warmup": args.warmup,
            "ms_per_step": statistics.mean(step_ms),
            "step_ms_spread": {
                "p50": statistics.median(step_ms), "max": max(step_ms),
                "lookahead_boundary": [[args.warmup + i, step_ms[i]] for i in range(K)
                                       if (args.warmup + i) % w.lookahead == 0],
                "note": "per-step device time; a lookahead-boundary step (new indexer queries) gathers "
                        "the new selection's misses from the pinned pool"},
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": DTYPE,
            "precision": "bf16 keys/queries scored on bf16 MMAs; f32 latents rounded to fp16 attention MMA operands "
                         "(tcgen05 kind::f16; staged rows kept as those fp16 values); f32 accumulate and softmax; "
                         "fp16 split partials",
            "data": "synthetic (seeded PCG64; shapes of the pages' workloads)",
            "config": {
                "workload": w.name, "context_len": w.context_len,
                "layers": f"{sum(1 for r in w.layer_ratios if r == 4)}x ratio-4 + "
                          f"{sum(1 for r in w.layer_ratios if r == 128)}x ratio-128",
                "n_chunks": w.n_chunks, "gpu_chunks": w.gpu_chunks, "index_topk": w.index_topk,
                "select": "topk" if w.select_mode == C.SELECT_TOPK else f"threshold tau={w.tau}",
                "ensemble": "max" if w.ensemble == C.ENSEMBLE_MAX else "mean",
                "heads": w.n_heads, "batch": w.batch, "lookahead": w.lookahead,
                "l2": "flushed before every timed step (256 MiB written then read back, outside the timed span)",
                "parallelism": f"replicas x{world}",
            },
            "gpu_launches": launches_per_step(w, torch.cuda.get_device_properties(device).multi_processor_count) * K,
            "roofline": {
                "kernel": "lsa_attend (attend_kernel, split pairs merged in the same kernel), device time per call",
                "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "peak_kind": peak_kind,
                "traffic": traffic["dram_bytes_per_launch"] if traffic else None,
                "algorithmic_bytes_per_launch": statistics.mean(a_bytes),
                "algorithmic_bytes_note": "the pages' fp32 rows: 2048 B per window or staged row, q and out",
                "avg_launch_us": a_avg_ms * 1e3,
                "layout": {"bytes_per_launch": l_bytes, "achieved": l_bytes / (a_avg_ms / 1e3) / 1e9,
                           "frac": l_bytes / (a_avg_ms / 1e3) / 1e9 / peak,
                           "note": "the bytes this layout reads: fp32 window rows, fp16 staged rows (1024 B)"},
            },
            "kernels_us": {"fm_score": statistics.mean(score_ms) * 1e3,
                           "fm_select+kvswap_stage": statistics.mean(stage_ms) * 1e3,
                           "lsa_attend": statistics.mean(attn_ms) * 1e3,
                           "note": f"phase spans of {KB} further steps replayed as three graphs (each span "
                                   "includes its graph launch)"},
            "calls_us": {"fm_score": statistics.median(sp_score) * 1e3,
                         "fm_select": statistics.median(sp_select) * 1e3,
                         "kvswap_stage": statistics.median(sp_stage) * 1e3,
                         "lsa_attend": statistics.median(sp_attn) * 1e3,
                         "note": "device time per call: eager calls queued behind the L2 flush and a device-side "
                                 "wait, unchained"},
            "score_gbs": score_bytes(w) / (statistics.mean(score_ms) / 1e3) / 1e9,
            "score_select_pass": {
                "score_us": statistics.median(sp_score) * 1e3, "select_us": statistics.median(sp_select) * 1e3,
                "bytes": pass_bytes(w),
                "gbs": pass_bytes(w) / ((statistics.median(sp_score) + statistics.median(sp_select)) / 1e3) / 1e9,
                "score_kernel_gbs": score_bytes(w) / (statistics.median(sp_score) / 1e3) / 1e9,
                "score_kernel": scoring_kernel(w),
                "frac": pass_bytes(w) / ((statistics.median(sp_score) + statistics.median(sp_select)) / 1e3) / 1e9
                / peak,
                "chained": {"us": ch_us, "gbs": pass_bytes(w) / ch_us / 1e3,
                            "frac": pass_bytes(w) / ch_us / 1e3 / peak,
                            "note": "as the decode step issues them: fm_select chained to fm_score (its kernel "
                                    "launched while the scoring kernel runs), one span"},
                "note": "fm_score then fm_select, eager and unchained (each call pays its launch), queued behind "
                        "the L2 flush; bytes = keys + score write + selection reads (256 + 12 per chunk and "
                        "sequence)"},
            "score_fp8_keys": {
                "us": statistics.median(fp8_ms) * 1e3,
                "gbs": w.batch * w.n_chunks * (C.INDEXER_DIM + 4 + 4) / (statistics.median(fp8_ms) / 1e3) / 1e9,
                "note": "fm_score_fp8: e4m3 codes + fp32 scale per chunk (132 B read, 4 B written), L2 flushed, "
                        "eager call queued behind a device-side wait"},
            "score_per_indexer_keys": {
                "us": statistics.median(multi_ms) * 1e3,
                "gbs": w.batch * w.n_chunks * (3 * C.INDEXER_DIM * 2 + 4) / (statistics.median(multi_ms) / 1e3) / 1e9,
                "note": "fm_score_multi, three key sets (one per memory indexer), L2 flushed, eager call queued "
                        "behind a device-side wait"},
            "step_hbm_gbs": step_bytes / (statistics.mean(step_ms) / 1e3) / 1e9,
            "warm_l2": {"value": K / (sum(warm_ms) / 1e3), "unit": "steps/s", "ms_per_step": statistics.mean(warm_ms),
                        "note": "the same graph-replayed steps without the L2 flush between them"},
            "lru_hit_rate": (st["hits"] / sel_total) if sel_total else None,
            "staged_bytes_per_step": st["h2d_bytes"] / K,
            "selected_per_step": st["selected"] / K,
            "selected_count": {
                "min": min(sel_counts), "median": statistics.median(sel_counts), "max": max(sel_counts),
                "hist": {str(c): sel_counts.count(c) for c in sorted(set(sel_counts))},
                "note": f"fm_select's count per sequence over {KB} breakdown steps"},
            "wall_s": wall,
            "adaptive_capacity": adaptive,
            "lookahead_schedule": lookahead,
            "periodic_selection": {
                "value": KP / (sum(periodic_ms) / 1e3), "unit": "steps/s",
                "ms_per_step": statistics.mean(periodic_ms),
                "note": f"score + select once per {w.lookahead}-step lookahead window, the other steps "
                        "reuse the selection (swap-in + attention only); not the headline"},
        }
        clk_sum = clk.summary()
        result["clocks"] = clk_sum
    if not args.no_e2e:
        e2e = run_e2e(args, w, ds, spec, graph)
        if result is not None:
            result["e2e"] = e2e
    link = host_link_gbs(device)
    gather = run_miss_gather(w, ds, stream, cold=False, link=link)
    gather_cold = run_miss_gather(w, ds, stream, cold=True, link=link)
    if result is not None:
        result["miss_gather"] = gather
        result["miss_gather_cold"] = gather_cold
    ds.close()
    del flush, fm_q_all, q_all
    torch.cuda.synchronize()
    if result is not None and world == 1 and not args.no_sweep:
        # the other workloads of the metric, one compact record each
        sweep = {}
        for name in [x for x in args.sweep.split(",") if x and x != w.name]:
            try:
                sweep[name] = sweep_record(name, args, device, link)
            except Exception as exc:   # a failed workload is reported, the headline stands
                sweep[name] = {"error": f"{type(exc).__name__}: {exc}"}
            torch.cuda.empty_cache()
        result["workloads"] = sweep
    return result


def host_link_gbs(device):
    """A plain pinned H2D copy of 256 MiB, best of 3: the host link's measured rate."""
    import torch
    src = torch.empty(64 << 20, dtype=torch.float32).pin_memory()
    dst = torch.empty(src.shape, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream()
    link = 0.0
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        dst.copy_(src, non_blocking=True)
        b.record(stream)
        b.synchronize()
        link = max(link, src.numel() * 4 / (a.elapsed_time(b) / 1e3) / 1e9)
    return link


def run_miss_gather(w, ds, stream, cold=False, link=None):
    """Host-link roofline of the miss gather: kvswap_stage calls in which every
    selected chunk of a swapped layer misses (disjoint chunk sets in turn, so the
    LRU always evicts a set staged earlier). Warm: every row's host pages were
    read once just before (the rows of the first chunk sets, read twice in
    turn). Cold: chunk sets from the top of the context that no step selected,
    read for the first time since their store (only where the context has
    room for them). Compared with a plain pinned H2D copy of 256 MiB."""
    import torch
    if not any(ds.swap):
        return None
    m = w.index_topk if w.select_mode == C.SELECT_TOPK else w.clamp
    n_sets = 3 if w.gpu_chunks >= 2 * m else 2
    R = 4 if cold else 6
    if cold and w.n_chunks < 64 * m:
        return {"value": None, "note": "context too small for rows unread since their store"}
    if w.n_chunks < n_sets * m:
        return None
    dev = ds.sel.device
    if cold:
        sets = [torch.arange(w.n_chunks - (i + 1) * m, w.n_chunks - i * m, dtype=torch.int32, device=dev)
                for i in range(R)]
    else:
        sets = [torch.arange(i * m, (i + 1) * m, dtype=torch.int32, device=dev) for i in range(n_sets)]

    def select_set(i):
        ds.sel[:, :m] = sets[i % len(sets)]
        ds.count.fill_(m)

    if not cold:
        for i in range(2 * n_sets):                     # fill the slots, then read every row once more
            select_set(i)
            ds.stage(-1, stream)
    torch.cuda.synchronize()
    ds.reset_stats()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(R)]
    for i in range(R):
        select_set(i if cold else 2 * n_sets + i)       # outside the timed span
        ev[i][0].record(stream)
        ds.stage(-1, stream)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    assert ds.check_error() == 0, "device error during the miss-gather measurement"
    st = ds.stats()
    secs = sum(e0.elapsed_time(e1) for e0, e1 in ev) / 1e3
    link = link if link is not None else host_link_gbs(dev)
    gbs = st["h2d_bytes"] / secs / 1e9
    return {"gbs": gbs, "host_link_gbs": link, "frac": gbs / link, "misses_per_call": st["misses"] / R,
            "hits": st["hits"], "us_per_call": secs / R * 1e6,
            "note": f"kvswap_stage (resolve + zero-copy gather) of {m} chunks per sequence, all missing in every "
                    f"swapped layer, {'rows not read since their store' if cold else 'rows read once before'}; "
                    f"host link = pinned cudaMemcpyAsync H2D of 256 MiB"}


def chained_pass_us(ds, spec, stream, flush, bind, t0, reps=6):
    """The scoring + selection pass as the decode step issues it: fm_score, then
    fm_select chained to it (its kernel launched while the scoring kernel runs),
    queued behind the L2 flush and a device-side wait; median span in us."""
    import torch
    from sparse_retrieval_host_gb300 import abi
    spans = []
    for i in range(reps):
        bind(t0 + i)
        flush.zero_()
        flush.sum()
        torch.cuda._sleep(HOLD_CYCLES)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        ds.score(spec, stream)
        abi.srh_set_chained(ds.ctx, True)
        ds.select(spec, stream)
        abi.srh_set_chained(ds.ctx, False)
        e1.record(stream)
        e1.synchronize()
        if i >= 1:
            spans.append(e0.elapsed_time(e1) * 1e3)
    assert ds.check_error() == 0, "device error during the chained pass"
    return statistics.median(spans)


def sweep_record(name, args, device, link):
    """A compact record of one more workload: graph-replayed steps with the L2
    flushed and warm, per-call device times (attention roofline, scoring +
    selection pass), the swap counters, and the miss gather on warm and cold rows."""
    import torch
    w = C.get(name)
    t0 = time.perf_counter()
    ds, spec, fm_q_all, q_all = setup(w, device)
    setup_s = time.perf_counter() - t0
    try:
        stream = torch.cuda.current_stream()
        flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=device)

        def bind(t):
            ds.fm_q.copy_(fm_q_all[(t % w.steps) // w.lookahead])
            ds.q.copy_(q_all[t % q_all.shape[0]])

        W, K = 3, 10
        for t in range(W):
            bind(t)
            ds.step(spec, stream)
        torch.cuda.synchronize()
        assert ds.check_error() == 0, "device error during warm-up"
        (graph,) = ds.capture(spec)
        ds.reset_stats()
        cold_ms, warm_ms = [], []
        # the timed steps straddle a lookahead boundary (new needles: misses)
        t_first = max(W, w.lookahead - K // 2)
        for flushed, out in ((True, cold_ms), (False, warm_ms)):
            ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
            for i in range(K):
                bind(t_first + i + (0 if flushed else w.lookahead))
                if flushed:
                    flush.zero_()
                    flush.sum()
                ev[i][0].record(stream)
                graph.replay()
                ev[i][1].record(stream)
            torch.cuda.synchronize()
            out.extend(e0.elapsed_time(e1) for e0, e1 in ev)
            if flushed:
                st = ds.stats()
        assert ds.check_error() == 0, "device error during the timed steps"
        sp = {"score": [], "select": [], "stage": [], "attend": []}
        counts, sel_counts = [], []
        for i in range(6):
            bind(t_first + 2 * w.lookahead + i)
            flush.zero_()
            flush.sum()
            torch.cuda._sleep(HOLD_CYCLES)
            q = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
            q[0].record(stream)
            ds.score(spec, stream)
            q[1].record(stream)
            ds.select(spec, stream)
            q[2].record(stream)
            ds.stage(-1, stream)
            q[3].record(stream)
            ds.attend(-1, stream)
            q[4].record(stream)
            q[4].synchronize()
            if i >= 1:
                for j, key in enumerate(("score", "select", "stage", "attend")):
                    sp[key].append(q[j].elapsed_time(q[j + 1]))
                counts.append(ds.count_l.cpu().numpy().copy())
                sel_counts.extend(int(c) for c in ds.count.cpu().numpy())
        assert ds.check_error() == 0, "device error during the per-call timing"
        ch_us = chained_pass_us(ds, spec, stream, flush, bind, t_first + 3 * w.lookahead)
        peak, _ = measured_peaks()
        a_us = statistics.median(sp["attend"]) * 1e3
        a_bytes = statistics.mean(attn_bytes(w, c) for c in counts)
        l_bytes = statistics.mean(attn_layout_bytes(w, c) for c in counts)
        p_us = (statistics.median(sp["score"]) + statistics.median(sp["select"])) * 1e3
        sel_total = st["hits"] + st["misses"]
        rec = {
            "value": K / (sum(cold_ms) / 1e3), "unit": "steps/s", "ms_per_step": statistics.mean(cold_ms),
            "warm_l2": {"value": K / (sum(warm_ms) / 1e3), "ms_per_step": statistics.mean(warm_ms)},
            "batch": w.batch, "context_len": w.context_len, "n_chunks": w.n_chunks,
            "lsa_attend": {"us": a_us, "algorithmic_bytes": a_bytes, "gbs": a_bytes / a_us / 1e3,
                           "frac": a_bytes / a_us / 1e3 / peak, "layout_bytes": l_bytes,
                           "layout_frac": l_bytes / a_us / 1e3 / peak},
            "score_select_pass": {"us": p_us, "score_us": statistics.median(sp["score"]) * 1e3,
                                  "select_us": statistics.median(sp["select"]) * 1e3,
                                  "score_kernel": scoring_kernel(w), "bytes": pass_bytes(w),
                                  "gbs": pass_bytes(w) / p_us / 1e3, "frac": pass_bytes(w) / p_us / 1e3 / peak,
                                  "chained": {"us": ch_us, "gbs": pass_bytes(w) / ch_us / 1e3,
                                              "frac": pass_bytes(w) / ch_us / 1e3 / peak}},
            "kvswap_stage_us": statistics.median(sp["stage"]) * 1e3,
            "lru_hit_rate": (st["hits"] / sel_total) if sel_total else None,
            "staged_bytes_per_step": st["h2d_bytes"] / K,
            "selected_count": {"min": min(sel_counts), "median": statistics.median(sel_counts),
                               "max": max(sel_counts)},
            "setup_s": setup_s,
            "steps": K, "warmup": W,
        }
        rec["miss_gather_warm"] = run_miss_gather(w, ds, stream, cold=False, link=link)
        rec["miss_gather_cold"] = run_miss_gather(w, ds, stream, cold=True, link=link)
        return rec
    finally:
        ds.close()
        torch.cuda.synchronize()


def run_e2e(args, w, ds, spec, graph):
    """Same steps through the public API with host buffers (runtime.HostLoop):
    every step copies its queries H2D from pinned memory and reads the attention
    output and the selection back D2H. The copies of neighbouring steps overlap
    the step in flight (two buffer sets, copy streams); the timed region spans
    all K steps, every step's copies included. The serial form (copy in, step,
    copy out, synchronize, one step at a time) is reported beside it."""
    import torch
    from sparse_retrieval_host_gb300.runtime import HostLoop, NativeHostLoop, bits_to_i16
    stream = torch.cuda.current_stream()
    nq = min(Q_CYCLE, w.steps)
    h_fmq = [bits_to_i16(np.stack([G.fm_queries(w, t, b) for b in range(w.batch)])).pin_memory()
             for t in range(0, w.steps, w.lookahead)]
    h_q = [bits_to_i16(np.stack([np.stack([G.attn_q(w, t, l, b) for b in range(w.batch)])
                                 for l in range(w.n_layers)])).pin_memory() for t in range(nq)]
    h_out = [torch.empty(ds.out.shape, dtype=torch.float32).pin_memory() for _ in range(2)]
    h_sel = [torch.empty(ds.sel.shape, dtype=torch.int32).pin_memory() for _ in range(2)]
    h_cnt = [torch.empty(ds.count.shape, dtype=torch.int32).pin_memory() for _ in range(2)]
    K = max(3, args.steps // 2)
    t0 = args.warmup + args.steps

    # serial: one step at a time through the bound buffers of the captured step
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(K):
        t = t0 + i
        ds.fm_q.copy_(h_fmq[(t % w.steps) // w.lookahead], non_blocking=True)
        ds.q.copy_(h_q[t % nq], non_blocking=True)
        graph.replay()
        h_out[0].copy_(ds.out, non_blocking=True)
        h_sel[0].copy_(ds.sel, non_blocking=True)
        h_cnt[0].copy_(ds.count, non_blocking=True)
        stream.synchronize()
    end.record(stream)
    end.synchronize()
    ms_serial = start.elapsed_time(end) / K

    def pipelined(loop, first):
        for i in range(2):                              # warm the loop's graphs
            t = first + i
            loop.step(i, h_fmq[(t % w.steps) // w.lookahead], h_q[t % nq], h_out[i & 1], h_sel[i & 1], h_cnt[i & 1])
        loop.synchronize()
        s_first = loop.s_in if hasattr(loop, "s_in") else stream
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t_host = time.perf_counter()
        start.record(s_first)
        for i in range(2, K + 2):
            t = first + i
            loop.step(i, h_fmq[(t % w.steps) // w.lookahead], h_q[t % nq], h_out[i & 1], h_sel[i & 1], h_cnt[i & 1])
        loop.synchronize()
        end.record(stream)
        end.synchronize()
        # the loop's streams are synchronized before `end` is recorded, so the
        # span is taken on the host clock as well and the larger one is kept
        return max(start.elapsed_time(end), (time.perf_counter() - t_host) * 1e3) / K

    # pipelined, native: the library's host loop (one call per step)
    nloop = NativeHostLoop(ds, spec)
    ms = pipelined(nloop, t0 + K)
    nloop.close()
    # pipelined, Python: runtime.HostLoop (torch streams and events)
    ms_py = pipelined(HostLoop(ds, spec), t0 + 2 * K + 2)
    h2d = ds.fm_q.numel() * 2 + ds.q.numel() * 2
    d2h = ds.out.numel() * 4 + ds.sel.numel() * 4 + ds.count.numel() * 4
    return {"value": 1e3 / ms, "unit": "steps/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": ms, "steps": K,
            "api": "srh_hostloop_* (runtime.NativeHostLoop): pinned host inputs and outputs, copies of neighbouring "
                   "steps overlap the step, one library call per step",
            "python_loop": {"value": 1e3 / ms_py, "ms_per_step": ms_py,
                            "note": "runtime.HostLoop: the same pipeline issued from Python (torch streams and events)"},
            "serial": {"value": 1e3 / ms_serial, "ms_per_step": ms_serial,
                       "note": "copy in, replay, copy out, synchronize: one step at a time"}}


# --------------------------------------------------------------------------- the oracle
def oracle_sample(w, n_steps):
    """Time the fp64 oracle on the first ``n_steps`` steps of workload ``w``."""
    from oracle import srh_oracle as O
    ora = O.DecodeOracle(context_len=w.context_len, layer_ratios=w.layer_ratios,
                         gpu_chunks=w.gpu_chunks, index_topk=w.index_topk, batch=w.batch,
                         scale=w.scale, bias=[w.bias] * 3, ensemble_mode=w.ensemble,
                         select_mode=w.select_mode, tau=w.tau, clamp=w.clamp)
    ora.mark_all_stored()
    keys = [G.keys(w, b) for b in range(w.batch)]
    small = w.n_chunks <= 8192
    pools = {(l, b): G.pool(w, l, b) for l in range(w.n_layers) for b in range(w.batch)} if small else None
    wins = {(l, b): G.window(w, l, b) for l in range(w.n_layers) for b in range(w.batch)}
    fmq = {t: [G.fm_queries(w, t, b) for b in range(w.batch)] for t in range(n_steps)}
    qs = {t: {(l, b): G.attn_q(w, t, l, b) for l in range(w.n_layers) for b in range(w.batch)}
          for t in range(n_steps)}
    rows = (lambda l, b, idx: pools[(l, b)][np.asarray(idx, dtype=np.int64)]) if small else \
        (lambda l, b, idx: G.pool_rows(w, l, b, idx))
    t0 = time.perf_counter()
    for t in range(n_steps):
        ora.step(lambda b: keys[b], lambda b: fmq[t][b], lambda l, b: qs[t][(l, b)],
                 lambda l, b: wins[(l, b)], rows)
    return time.perf_counter() - t0


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        n = max((i.get("num_threads", 1) for i in info), default=1)
        return int(n)
    except Exception:
        return None


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


ONE_THREAD_ENV = {"OMP_NUM_THREADS": "1", "OPENBLAS_NUM_THREADS": "1", "MKL_NUM_THREADS": "1",
                  "BLIS_NUM_THREADS": "1", "VECLIB_MAXIMUM_THREADS": "1"}


def oracle_seconds_subprocess(name, n_steps, one_thread):
    """Seconds of the oracle on the first ``n_steps`` steps of workload ``name``,
    timed in a fresh interpreter (its BLAS pinned to one thread when asked; the
    GPU is not touched)."""
    env = dict(os.environ)
    if one_thread:
        env.update(ONE_THREAD_ENV)
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--config", name, "--oracle-seconds",
                        str(n_steps)], capture_output=True, text=True, env=env, timeout=600)
    if r.returncode != 0:
        raise RuntimeError(r.stderr.strip()[-300:])
    return float(r.stdout.strip().splitlines()[-1])


def cpu_baseline(w, sample_steps=0):
    n = sample_steps or {"tiny": 256, "ctx8k": 96}.get(w.name, 8)
    cores = host_cores()
    secs_all = oracle_seconds_subprocess(w.name, n, one_thread=False)
    secs_one = oracle_seconds_subprocess(w.name, n, one_thread=True)
    return {"value": n / secs_all, "unit": "steps/s", "cores": cores, "kind": "oracle",
            "sample": f"first {n} decode steps of {w.name} (fp64 numpy oracle; input generation excluded)",
            "seconds": secs_all,
            "threading": "numpy's BLAS on every host core for the matrix products; selection, LRU and the step "
                         "loop are single-threaded Python",
            "blas_threads": blas_threads(),
            "single_thread": {"value": n / secs_one, "unit": "steps/s", "seconds": secs_one, "cores": 1}}


def run_reference(args, rank):
    if rank != 0:
        return None
    w = C.get(args.config)
    n = max(1, min(args.steps, args.cpu_sample_steps or {"tiny": 1000, "ctx8k": 200}.get(w.name, 8)))
    # warm-up: one step, untimed
    if args.warmup > 0:
        oracle_sample(w, 1)
    secs = oracle_sample(w, n)
    v = n / secs
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "steps/s", "n_gpus": 1,
            "steps": n, "warmup": args.warmup, "ms_per_step": secs / n * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name},
            "cpu_baseline": {"value": v, "unit": "steps/s", "cores": host_cores(), "kind": "oracle",
                             "blas_threads": blas_threads(),
                             "sample": f"{n} decode steps of {w.name} per timed run"},
            "e2e": {"value": v, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    if args.oracle_seconds:
        print(oracle_sample(C.get(args.config), args.oracle_seconds))
        return
    dist, rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        res = run_reference(args, rank)
    else:
        res = run_ours(args, dist, rank, world, local)
        if rank == 0 and res is not None and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(C.get(args.config), args.cpu_sample_steps)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
