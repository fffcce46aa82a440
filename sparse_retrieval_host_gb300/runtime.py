"""Device buffers for one decode loop and the four-call decode step.

``DecodeStep`` owns a library context (pinned pools, slot tables, scratch) and
the caller-side device tensors the C ABI reads and writes. ``step()`` issues
fm_score -> fm_select -> kvswap_stage -> lsa_attend on one stream (the miss
gathers go to a side stream when one is given), and ``capture()`` records the
step into CUDA graphs. ``HostLoop`` and ``NativeHostLoop`` run steps from pinned
host buffers: queries copied in, outputs and the selection copied out, the
copies of neighbouring steps overlapping the step (issued from Python, or by one
library call per step). PyTorch is used only to allocate device memory and to
name streams.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np
import torch

from . import abi

INDEXERS, IDX_HEADS, IDX_DIM = 3, 8, 128


@dataclass
class StepSpec:
    scale: float
    bias: Sequence[float]
    ensemble: int
    select_mode: int
    k: int
    tau: float
    clamp: int


class DecodeStep:
    def __init__(self, *, batch: int, layer_ratios: Sequence[int], gpu_chunks: int, index_topk: int,
                 context_len: int, n_heads: int, max_select: int = 0, src_ratio: int = 4,
                 pinned_cap_bytes: int = 0, allow_topk_reduction: bool = False,
                 device: str = "cuda", flags: int = 0, key_sets: int = 1, key_format: str = "bf16"):
        self.cfg = abi.make_config(batch=batch, layer_ratios=list(layer_ratios), gpu_chunks=gpu_chunks,
                                   index_topk=index_topk, context_len=context_len, src_ratio=src_ratio,
                                   pinned_cap_bytes=pinned_cap_bytes,
                                   allow_topk_reduction=allow_topk_reduction, max_select=max_select,
                                   flags=flags)
        self.ctx = abi.srh_create(self.cfg)
        self.B, self.L, self.G, self.H = batch, len(layer_ratios), gpu_chunks, n_heads
        self.layer_ratios = list(layer_ratios)
        self.S = abi.srh_max_select(self.ctx)
        self.n = (context_len + src_ratio - 1) // src_ratio
        self.caps = [abi.srh_layer_info(self.ctx, l)[0] for l in range(self.L)]
        self.swap = [abi.srh_layer_info(self.ctx, l)[1] for l in range(self.L)]
        dev = torch.device(device)
        B, L, G, H, S, n = self.B, self.L, self.G, self.H, self.S, self.n
        i16, f32, i32 = torch.int16, torch.float32, torch.int32
        # key_sets = 3: each memory indexer scores its own layer's keys (fm_score_multi)
        if key_sets not in (1, 3):
            raise ValueError("key_sets must be 1 or 3")
        self.key_sets = key_sets
        shape = (B, n, IDX_DIM) if key_sets == 1 else (3, B, n, IDX_DIM)
        self.keys = torch.zeros(shape, dtype=i16, device=dev)
        # key_format = "fp8": score e4m3 codes made by quantize_keys() from ``keys``
        if key_format not in ("bf16", "fp8") or (key_format == "fp8" and key_sets != 1):
            raise ValueError("key_format must be bf16, or fp8 with one key set")
        self.key_format = key_format
        if key_format == "fp8":
            self.codes = torch.zeros((B, n, IDX_DIM), dtype=torch.uint8, device=dev)
            self.kscale = torch.zeros((B, n), dtype=f32, device=dev)
        self.fm_q = torch.zeros((B, INDEXERS, IDX_HEADS, IDX_DIM), dtype=i16, device=dev)
        self.scores = torch.zeros((B, n), dtype=f32, device=dev)
        self.sel = torch.zeros((B, S), dtype=i32, device=dev)
        self.count = torch.zeros((B,), dtype=i32, device=dev)
        self.staging = torch.zeros((L, B, G, abi.KV_DIM), dtype=torch.float16, device=dev)   # fp16 staged rows
        self.phys = torch.zeros((L, B, S), dtype=i32, device=dev)
        self.count_l = torch.zeros((L, B), dtype=i32, device=dev)
        self.window = torch.zeros((L, B, abi.WINDOW, abi.KV_DIM), dtype=f32, device=dev)
        self.q = torch.zeros((L, B, H, abi.KV_DIM), dtype=i16, device=dev)
        self.out = torch.zeros((L, B, H, abi.KV_DIM), dtype=f32, device=dev)
        self._adaptive = None

    # ------------------------------------------------------------------ host pools
    def pool_view(self, layer: int, seq: int) -> np.ndarray:
        """numpy view of the pinned pool of (layer, seq): ``[cap][512]`` fp32."""
        addr = abi.srh_pool_host_ptr(self.ctx, layer, seq)
        cap = self.caps[layer]
        buf = (ctypes.c_float * (cap * abi.KV_DIM)).from_address(addr)
        return np.ctypeslib.as_array(buf).reshape(cap, abi.KV_DIM)

    def mark_stored(self, layer: int, seq: int, c0: int = 0, n: Optional[int] = None) -> None:
        if n is None:
            n = self.caps[layer] - c0
        abi.srh_mark_stored(self.ctx, layer, seq, c0, n)

    def store(self, layer: int, seq: int, c0: int, rows: torch.Tensor, stream=None) -> None:
        """Store flow on the device: ``rows`` [n][512] fp32 (CUDA) become chunks
        c0.. of (layer, seq) in the host pool (see kvswap_store)."""
        rows = rows.contiguous()
        abi.kvswap_store(self.ctx, layer, seq, c0, rows.shape[0], rows, stream)

    # ------------------------------------------------------------------ the step
    def quantize_keys(self, stream=None) -> None:
        """e4m3 codes and per-chunk scales of ``keys`` (once, for frozen keys)."""
        abi.fm_quantize_keys(self.ctx, self.keys, self.n, self.codes, self.kscale, stream)

    def score(self, spec: StepSpec, stream=None, fm_q=None) -> None:
        if self.key_format == "fp8":
            abi.fm_score_fp8(self.ctx, self.codes, self.kscale, self.n, self.fm_q if fm_q is None else fm_q,
                             spec.scale, spec.bias, spec.ensemble, self.scores, stream)
            return
        fn = abi.fm_score if self.key_sets == 1 else abi.fm_score_multi
        fn(self.ctx, self.keys, self.n, self.fm_q if fm_q is None else fm_q, spec.scale, spec.bias, spec.ensemble,
           self.scores, stream)

    def select(self, spec: StepSpec, stream=None) -> None:
        abi.fm_select(self.ctx, self.scores, self.n, spec.select_mode, spec.k, spec.tau, spec.clamp,
                      self.sel, self.count, stream)

    def stage(self, layer: int = -1, stream=None, side=None) -> None:
        abi.kvswap_stage(self.ctx, layer, self.sel, self.count, self.staging, self.phys, self.count_l,
                         stream, side)

    def attend(self, layer: int = -1, stream=None, q=None, out=None) -> None:
        abi.lsa_attend(self.ctx, layer, self.q if q is None else q, self.H, self.window, self.staging,
                       self.phys, self.count_l, self.out if out is None else out, stream)

    def step(self, spec: StepSpec, stream=None, side=None, fm_q=None, q=None, out=None,
             rescore: bool = True) -> None:
        """One decode step: the four C entry points in order, issued back to back
        on one stream, so their kernels are launched chained (each may start
        while the previous one finishes; see srh_set_chained).

        With ``rescore=False`` the step keeps the current selection (``sel``,
        ``count``) and runs only the swap-in and the attention: the memory
        indexer fires periodically, once per lookahead window (summary section
        "LSA 让模型预判 KV chunk"), not at every step."""
        # the step's first kernel waits for all earlier work on the stream; the
        # ones after it are chained
        try:
            if rescore:
                self.score(spec, stream, fm_q)
                abi.srh_set_chained(self.ctx, True)
                self.select(spec, stream)
                self.stage(-1, stream, side)
            else:
                self.stage(-1, stream, side)
                abi.srh_set_chained(self.ctx, True)
            self.attend(-1, stream, q, out)
        finally:
            abi.srh_set_chained(self.ctx, False)

    # ------------------------------------------------------------------ CUDA graphs
    def capture(self, spec: StepSpec, parts: bool = False, rescore: bool = True):
        """Record the decode step into CUDA graphs and return them.

        The graphs read the bound inputs (``fm_q``, ``q``) and write the bound
        outputs, so a caller copies each step's queries into those buffers and
        calls ``replay()``: one launch per step instead of one host call per
        kernel. Replays advance the LRU state like eager steps. Capture after at
        least one eager step (one-time set-up -- kernel attributes, resident
        fills of layers that do not swap -- happens there), and capture again
        after ``mark_stored`` on a layer that does not swap. With ``parts`` the
        step is recorded as three graphs (score; select + stage; attend) so the
        phases can be timed separately.
        """
        dev = self.keys.device
        s = torch.cuda.Stream(device=dev)
        s.wait_stream(torch.cuda.current_stream(dev))
        graphs = []

        def rec(fn):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                fn()
            graphs.append(g)

        if parts:
            rec(lambda: self.score(spec))
            rec(lambda: (self.select(spec), self.stage(-1)))
            rec(lambda: self.attend(-1))
        else:
            rec(lambda: self.step(spec, rescore=rescore))
        torch.cuda.current_stream(dev).wait_stream(s)
        return graphs

    # ------------------------------------------------------------------ lookahead schedule
    def _lookahead_setup(self, spec: StepSpec) -> None:
        """Two phys/count_l buffers (the selection in force and the one being
        staged) and the capacity check that makes the overlap safe."""
        m = spec.k if spec.select_mode == abi.SRH_SELECT_TOPK else spec.clamp
        g_lo = self.G if self._adaptive is None else self._adaptive["g_min"]
        if any(self.swap) and g_lo < 2 * m:
            raise ValueError(f"the lookahead schedule needs >= {2 * m} slots in use per swapped layer "
                             f"(two selections of up to {m} chunks); the capacity can drop to {g_lo}")
        if not hasattr(self, "phys2"):
            dev = self.keys.device
            self.phys2 = torch.zeros((2,) + tuple(self.phys.shape), dtype=torch.int32, device=dev)
            self.count_l2 = torch.zeros((2,) + tuple(self.count_l.shape), dtype=torch.int32, device=dev)
            self.in_force = 0
            self.side = torch.cuda.Stream(device=dev)

    def lookahead_step(self, spec: StepSpec, trigger: bool, stream=None, fm_q=None, q=None, out=None) -> None:
        """One step of the lookahead schedule. At a trigger step the memory
        indexer scores and selects from this step's queries and the selection
        is swapped in on a side stream, while the attention on ``stream`` reads
        the selection in force (staged at the previous trigger); the new one is
        in force from the next step on. Other steps run the attention alone.
        Before the first trigger no chunk is in force (window rows only).

        Safe because a swapped layer keeps at least two selections' worth of
        slots: the LRU then evicts only slots outside the selection in force,
        whose slots are the most recently used (checked on the first call)."""
        self._lookahead_setup(spec)
        dev = self.keys.device
        main = stream if stream is not None else torch.cuda.current_stream(dev)
        cur, nxt = self.in_force, 1 - self.in_force
        try:
            if trigger:
                self.side.wait_stream(main)
                self.score(spec, self.side, fm_q)
                abi.srh_set_chained(self.ctx, True)
                self.select(spec, self.side)
                abi.kvswap_stage(self.ctx, -1, self.sel, self.count, self.staging, self.phys2[nxt],
                                 self.count_l2[nxt], self.side, None)
                abi.srh_set_chained(self.ctx, False)
            abi.lsa_attend(self.ctx, -1, self.q if q is None else q, self.H, self.window, self.staging,
                           self.phys2[cur], self.count_l2[cur], self.out if out is None else out, main)
            if trigger:
                main.wait_stream(self.side)
        finally:
            abi.srh_set_chained(self.ctx, False)
        if trigger:
            self.in_force = nxt

    def capture_lookahead(self, spec: StepSpec):
        """CUDA graphs of the lookahead schedule: ``{(trigger, in_force): graph}``
        for the four combinations (the buffers alternate). Replay with
        ``replay_lookahead``. Capture after at least one eager step."""
        self._lookahead_setup(spec)
        dev = self.keys.device
        s = torch.cuda.Stream(device=dev)
        s.wait_stream(torch.cuda.current_stream(dev))
        keep = self.in_force
        graphs = {}
        for trig in (True, False):
            for cur in (0, 1):
                self.in_force = cur
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=s):
                    self.lookahead_step(spec, trig, stream=s)
                graphs[(trig, cur)] = g
        self.in_force = keep
        torch.cuda.current_stream(dev).wait_stream(s)
        return graphs

    def replay_lookahead(self, graphs, trigger: bool) -> None:
        graphs[(bool(trigger), self.in_force)].replay()
        if trigger:
            self.in_force = 1 - self.in_force

    # ------------------------------------------------------------------ status
    def set_adaptive(self, policy=None) -> None:
        """Adaptive staging capacity (srh_set_adaptive); ``policy`` is a mapping
        of g_min, g_max, g_init, epoch, lo_permille, hi_permille, delta, or None."""
        abi.srh_set_adaptive(self.ctx, policy)
        self._adaptive = dict(policy) if policy is not None else None

    def active_slots(self):
        """Slots in use per (layer, sequence) (srh_get_active_slots)."""
        return abi.srh_get_active_slots(self.ctx, self.L, self.B)

    def stats(self) -> dict:
        return abi.srh_get_stats(self.ctx)

    def reset_stats(self) -> None:
        abi.srh_reset_stats(self.ctx)

    def check_error(self) -> int:
        return abi.srh_check_error(self.ctx)

    def close(self) -> None:
        if getattr(self, "ctx", None):
            abi.srh_destroy(self.ctx)
            self.ctx = None

    def __del__(self):  # pragma: no cover
        try:
            self.close()
        except Exception:
            pass


class HostLoop:
    """Decode steps fed from pinned host memory and read back into it, with the
    copies of neighbouring steps overlapping the step in flight.

    Two sets of device input/output buffers alternate. Step i's queries are
    copied in on one stream while step i-1 runs, and step i-1's outputs
    (attention output, selection, count) are copied out on another while step
    i runs; each step is one graph replay on the compute stream, so the LRU
    state still advances in step order. A set is refilled only after the step
    that read it finished and its outputs left the device (stream events).
    """

    def __init__(self, ds: "DecodeStep", spec: StepSpec):
        self.ds = ds
        dev = ds.keys.device
        self.fm_q = [torch.zeros_like(ds.fm_q) for _ in range(2)]
        self.q = [torch.zeros_like(ds.q) for _ in range(2)]
        self.out = [torch.zeros_like(ds.out) for _ in range(2)]
        self.sel = [torch.zeros_like(ds.sel) for _ in range(2)]
        self.count = [torch.zeros_like(ds.count) for _ in range(2)]
        self.s_comp = torch.cuda.Stream(device=dev)
        self.s_in = torch.cuda.Stream(device=dev)
        self.s_out = torch.cuda.Stream(device=dev)
        self.ev_in = [torch.cuda.Event() for _ in range(2)]
        self.ev_done = [torch.cuda.Event() for _ in range(2)]
        self.ev_out = [torch.cuda.Event() for _ in range(2)]
        self.s_comp.wait_stream(torch.cuda.current_stream(dev))
        self.graphs = []
        for k in range(2):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.s_comp):
                ds.step(spec, self.s_comp, fm_q=self.fm_q[k], q=self.q[k], out=self.out[k])
                self.sel[k].copy_(ds.sel)
                self.count[k].copy_(ds.count)
            self.graphs.append(g)
        torch.cuda.current_stream(dev).wait_stream(self.s_comp)

    def step(self, i: int, h_fm_q: torch.Tensor, h_q: torch.Tensor, h_out: torch.Tensor, h_sel: torch.Tensor,
             h_count: torch.Tensor) -> None:
        """Issue step i: inputs from pinned ``h_fm_q``/``h_q``, outputs into pinned
        ``h_out``/``h_sel``/``h_count`` (ready once ``synchronize()`` returns, or
        two steps later). Asynchronous."""
        k = i & 1
        self.s_in.wait_event(self.ev_done[k])          # step i-2 finished reading set k
        with torch.cuda.stream(self.s_in):
            self.fm_q[k].copy_(h_fm_q, non_blocking=True)
            self.q[k].copy_(h_q, non_blocking=True)
        self.ev_in[k].record(self.s_in)
        self.s_comp.wait_event(self.ev_in[k])
        self.s_comp.wait_event(self.ev_out[k])         # step i-2's outputs left set k
        with torch.cuda.stream(self.s_comp):
            self.graphs[k].replay()
        self.ev_done[k].record(self.s_comp)
        self.s_out.wait_event(self.ev_done[k])
        with torch.cuda.stream(self.s_out):
            h_out.copy_(self.out[k], non_blocking=True)
            h_sel.copy_(self.sel[k], non_blocking=True)
            h_count.copy_(self.count[k], non_blocking=True)
        self.ev_out[k].record(self.s_out)

    def synchronize(self) -> None:
        for s in (self.s_in, self.s_comp, self.s_out):
            s.synchronize()


class NativeHostLoop:
    """The same pipelined loop as HostLoop, issued by the library in native code
    (srh_hostloop_*): two sets of device step buffers, each with a CUDA graph
    of one step captured by the library, copy-in and copy-out streams ordered by
    events. One call per step from Python. Single key set, bf16 keys."""

    def __init__(self, ds: "DecodeStep", spec: StepSpec):
        if ds.key_format != "bf16" or ds.key_sets != 1:
            raise ValueError("the native host loop scores one bf16 key set")
        self.ds = ds
        self.fm_q = [torch.zeros_like(ds.fm_q) for _ in range(2)]
        self.q = [torch.zeros_like(ds.q) for _ in range(2)]
        self.out = [torch.zeros_like(ds.out) for _ in range(2)]
        self.sel = [torch.zeros_like(ds.sel) for _ in range(2)]
        self.count = [torch.zeros_like(ds.count) for _ in range(2)]
        self.lp = abi.srh_hostloop_create(ds.ctx, ds.keys, ds.n, ds.scores, ds.staging, ds.phys, ds.count_l,
                                          ds.window, ds.H, spec.scale, spec.bias, spec.ensemble, spec.select_mode,
                                          spec.k, spec.tau, spec.clamp, self.fm_q, self.q, self.out, self.sel,
                                          self.count, torch.cuda.current_stream(ds.keys.device))

    def step(self, i: int, h_fm_q: torch.Tensor, h_q: torch.Tensor, h_out: torch.Tensor, h_sel: torch.Tensor,
             h_count: torch.Tensor) -> None:
        """Issue step i (consecutive i from 0): pinned host inputs and outputs,
        complete after ``wait(i)`` or ``synchronize()``. Asynchronous."""
        abi.srh_hostloop_step(self.ds.ctx, self.lp, i, h_fm_q, h_q, h_out, h_sel, h_count)

    def wait(self, i: int) -> None:
        abi.srh_hostloop_wait(self.ds.ctx, self.lp, i)

    def synchronize(self) -> None:
        abi.srh_hostloop_sync(self.ds.ctx, self.lp)

    def close(self) -> None:
        if self.lp:
            abi.srh_hostloop_destroy(self.lp)
            self.lp = None

    def __del__(self):  # pragma: no cover
        try:
            self.close()
        except Exception:
            pass


def bits_to_i16(a: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bit patterns as an int16 tensor (same bytes)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16))
