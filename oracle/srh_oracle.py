"""Plain fp64 CPU oracle of one FlashMemory LSA + KV_SWAP decode step.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline / reference legs of ``bench.py`` may import or run this module. It
shares no code with the CUDA path: it does not import the product package and
the product package does not import it. Inputs come from the seeded
generator in ``srh_workload`` (random draws only) or from hand-made cases.

The step, as the pages state it:
  1. score every compressed chunk by dotting 3 memory-indexer query sets
     against the frozen compressed indexer keys (PocketLLM
     "FlashMemory 1M 上下文显存优化使用文档", section "技术细节 / 架构概览", box
     "FlashMemory Runtime Scoring", steps 1-2; FlashMemory-DeepSeek-V4 summary,
     section "LSA 让模型预判 KV chunk");
  2. ensemble the three scores by max (OR-mode) or mean (same box, step 3;
     summary section "Memory Indexer 放哪里");
  3. select by top-k (index_topk = 512) or by a sigmoid threshold
     (same box, step 3; summary section "LSA 让模型预判 KV chunk");
  4. per sparse layer, resolve the selected chunks against the GPU staging
     slots with the pages' LRU (section "KV_SWAP 实现细节", the
     GgufKvSwapLayerState structure and the Swap-in flow);
  5. attention over the 128-row window plus the selected chunks
     (section "架构概览", box "Per-layer Sparse Attention", step 3, and
     "Memory Layout").

Readings taken where the pages are silent (each one is a choice, listed with
its reason in the design notes):
  * the 8 query heads of one indexer combine by max; logit = scale*max + b_i,
    scale = 1/sqrt(128);
  * MEAN ensembles logits (max is domain-free because the sigmoid is monotone);
  * the threshold test is strict and taken in the logit domain:
    sigmoid(s) > tau  <=>  s > ln(tau/(1-tau));
  * order and tie-break everywhere: score descending, then chunk index ascending;
    a threshold set larger than the clamp keeps its first ``clamp`` entries;
  * a layer of ratio r reuses the global selection through
    c -> floor(c*src_ratio/r), first occurrence kept;
  * the LRU list starts with every slot free, slot 0 at the back;
  * with GPU_CHUNKS below the selected count (allowed only by the test flag),
    a swapped layer keeps the first GPU_CHUNKS chunks of its list;
  * adaptive GPU_CHUNKS (listed by the pages as a future direction) resizes the
    slot range in use from the hit rate of a window of steps, by the rule of
    section 4c; slots are never moved, dropped slots forget their chunks;
  * attention is MQA over the 512-wide latent (K = V = row), scale 1/sqrt(512).

Parity pins (checks that do not reuse this code) live in ``tests/test_oracle_*.py``.

Parity unpinned against the method: the head reduction (max over the 8
heads), the logit scale and bias, and the MEAN domain (logits, not sigmoids).
The pages do not fix them; hand-worked cases pin the code only to the readings
stated above. Every other step has a pin fixed by the pages or by mathematics.
"""
from __future__ import annotations

import math
from collections import OrderedDict
from dataclasses import dataclass, field
from typing import Callable, Dict, List, Optional, Sequence, Tuple

import numpy as np

KV_DIM = 512
WINDOW = 128
N_INDEXERS = 3
INDEXER_HEADS = 8
INDEXER_DIM = 128

ENSEMBLE_MAX = 0
ENSEMBLE_MEAN = 1
SELECT_TOPK = 0
SELECT_THRESH = 1


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float64; exact."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# Pinned host memory (section "关键参数调优", item 2, PINNED_MIB: the formula
#   required_pinned_mib = sum(layer_compressed_cap * kv_dim * sizeof(float)) / 2^20
#   layer_compressed_cap = (context_length + ratio - 1) / ratio )
# ----------------------------------------------------------------------------
def compressed_cap(context_len: int, ratio: int) -> int:
    return (context_len + ratio - 1) // ratio


def layer_pinned_bytes(context_len: int, ratio: int, kv_dim: int = KV_DIM) -> int:
    return compressed_cap(context_len, ratio) * kv_dim * 4


def required_pinned_bytes(context_len: int, ratios: Sequence[int], kv_dim: int = KV_DIM) -> int:
    return sum(layer_pinned_bytes(context_len, r, kv_dim) for r in ratios)


def swap_enabled(compressed_cap_: int, gpu_chunks: int) -> bool:
    """A layer swaps only if its chunks do not all fit in the staging slots
    (section "故障排查", the note on ``reason=no_layer_with_compressed_cap_gt_gpu_chunks``)."""
    return compressed_cap_ > gpu_chunks


# ----------------------------------------------------------------------------
# 1-2. Scoring and ensemble
# ----------------------------------------------------------------------------
def head_dots(keys_bits: np.ndarray, q_bits: np.ndarray) -> np.ndarray:
    """s_{i,h}(c) = <Q[i,h,:], K[c,:]> for every chunk c: ``[n][3][8]``."""
    k = bf16_to_f64(keys_bits)                       # [n][128]
    q = bf16_to_f64(q_bits).reshape(N_INDEXERS * INDEXER_HEADS, INDEXER_DIM)
    return (k @ q.T).reshape(k.shape[0], N_INDEXERS, INDEXER_HEADS)


def indexer_logits(keys_bits, q_bits, scale: float, bias: Sequence[float]) -> np.ndarray:
    """s_i(c) = scale * max_h s_{i,h}(c) + b_i: ``[3][n]``."""
    d = head_dots(keys_bits, q_bits)
    per = d.max(axis=2)                              # max over the 8 heads
    b = np.asarray(bias, dtype=np.float64).reshape(1, N_INDEXERS)
    return (scale * per + b).T


def ensemble(logits: np.ndarray, mode: int) -> np.ndarray:
    """MAX: s = max_i s_i (OR-mode routing); MEAN: s = (s_0 + s_1 + s_2) / 3."""
    if mode == ENSEMBLE_MAX:
        return logits.max(axis=0)
    if mode == ENSEMBLE_MEAN:
        return logits.sum(axis=0) / N_INDEXERS
    raise ValueError(mode)


def score(keys_bits, q_bits, scale, bias, mode) -> np.ndarray:
    return ensemble(indexer_logits(keys_bits, q_bits, scale, bias), mode)


def indexer_logits_multi(keys3_bits, q_bits, scale: float, bias: Sequence[float]) -> np.ndarray:
    """One key set per indexer (section "限制与未来工作", Multi-layer compressed_k:
    each scorer reads its own layer's indexer keys):
    s_i(c) = scale * max_h <Q[i,h,:], K_i[c,:]> + b_i: ``[3][n]``."""
    q = bf16_to_f64(q_bits).reshape(N_INDEXERS, INDEXER_HEADS, INDEXER_DIM)
    rows = []
    for i in range(N_INDEXERS):
        k = bf16_to_f64(np.asarray(keys3_bits)[i])   # [n][128]
        rows.append(scale * (k @ q[i].T).max(axis=1) + float(bias[i]))
    return np.stack(rows)


def score_multi(keys3_bits, q_bits, scale, bias, mode) -> np.ndarray:
    return ensemble(indexer_logits_multi(keys3_bits, q_bits, scale, bias), mode)


# ----------------------------------------------------------------------------
# 1'. fp8 indexer keys (section "限制与未来工作": quantize the indexer keys to
#     fp8/int8 to cut the key stream; the scorer kernel has to change with it).
#     Reading: e4m3 codes (1 sign, 4 exponent bits with bias 7, 3 mantissa bits;
#     largest finite value 448; 0x7F/0xFF are NaN) with one fp32 scale per
#     chunk, scale_c = amax_c / 448; code = e4m3(K / scale_c), rounded to nearest
#     (ties to even) and saturated to +-448. The scale and the division are fp32
#     operations, the same ones the kernel performs, because they decide codes.
# ----------------------------------------------------------------------------
E4M3_MAX = 448.0


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """Value of each e4m3 code (uint8) as float64; NaN for 0x7F / 0xFF."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = np.where((c & 0x7F) == 0x7F, np.nan, val)
    return sign * val


def _e4m3_table():
    codes = np.arange(0x7F, dtype=np.uint8)          # non-negative finite codes, increasing values
    return codes, e4m3_decode(codes)


def e4m3_encode(x) -> np.ndarray:
    """Round each finite value to the nearest e4m3 value, ties to the even code,
    saturating at +-448, keeping the sign (a negative value that rounds to zero
    gives 0x80); fp32/fp64 inputs, NaN is not expected."""
    x = np.asarray(x, dtype=np.float64)
    codes, vals = _e4m3_table()
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.searchsorted(vals, a, side="left")       # first value >= a
    hi = np.minimum(hi, len(vals) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - vals[lo]
    d_hi = vals[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((codes[hi] & 1) == 0))
    out = np.where(pick_hi, codes[hi], codes[lo]).astype(np.uint8)
    out = np.where(vals[hi] == a, codes[hi], out).astype(np.uint8)
    return np.where(np.signbit(x), out | 0x80, out).astype(np.uint8)   # the sign is kept, -0 included


def quantize_keys_fp8(keys_bits: np.ndarray):
    """bf16 keys [n][128] -> (e4m3 codes [n][128] uint8, fp32 scale [n])."""
    k = (np.asarray(keys_bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
    amax = np.abs(k).max(axis=1).astype(np.float32)
    scale = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
    ratio = (k / safe[:, None]).astype(np.float32)     # fp32 division, as on the device
    codes = e4m3_encode(ratio)
    codes[scale == 0] = 0
    return codes, scale


def indexer_logits_fp8(codes: np.ndarray, kscale: np.ndarray, q_bits, scale: float,
                       bias: Sequence[float]) -> np.ndarray:
    """s_i(c) = scale * kscale_c * max_h <Q[i,h,:], e4m3(K8[c,:])> + b_i: ``[3][n]``."""
    k = e4m3_decode(codes)                            # [n][128], exact
    q = bf16_to_f64(q_bits).reshape(N_INDEXERS * INDEXER_HEADS, INDEXER_DIM)
    d = (k @ q.T).reshape(k.shape[0], N_INDEXERS, INDEXER_HEADS).max(axis=2)
    per = d * np.asarray(kscale, dtype=np.float64)[:, None]
    b = np.asarray(bias, dtype=np.float64).reshape(1, N_INDEXERS)
    return (scale * per + b).T


def score_fp8(codes, kscale, q_bits, scale, bias, mode) -> np.ndarray:
    return ensemble(indexer_logits_fp8(codes, kscale, q_bits, scale, bias), mode)


# ----------------------------------------------------------------------------
# 3. Selection
# ----------------------------------------------------------------------------
def threshold_logit(tau: float) -> float:
    """sigmoid(s) > tau  <=>  s > ln(tau / (1 - tau))."""
    return math.log(tau / (1.0 - tau))


def order_desc(s: np.ndarray) -> np.ndarray:
    """Chunk indices ordered by (score descending, index ascending)."""
    s = np.asarray(s, dtype=np.float64)
    return np.lexsort((np.arange(s.shape[0]), -s))


def select_topk(s: np.ndarray, k: int) -> np.ndarray:
    return order_desc(s)[:min(k, s.shape[0])].astype(np.int64)


def select_threshold(s: np.ndarray, tau: float, clamp: int) -> np.ndarray:
    t = threshold_logit(tau)
    o = order_desc(s)
    o = o[np.asarray(s)[o] > t]
    return o[:clamp].astype(np.int64)


def select(s, mode: int, k: int, tau: float, clamp: int) -> np.ndarray:
    if mode == SELECT_TOPK:
        return select_topk(s, k)
    if mode == SELECT_THRESH:
        return select_threshold(s, tau, clamp)
    raise ValueError(mode)


# ----------------------------------------------------------------------------
# 4a. All sparse layers reuse the one global selection (section "技术细节",
#     "FlashMemory vs Native Indexer": selection granularity is global).
# ----------------------------------------------------------------------------
def layer_chunks(sel: Sequence[int], src_ratio: int, layer_ratio: int) -> List[int]:
    out: List[int] = []
    seen = set()
    for c in sel:
        m = (int(c) * src_ratio) // layer_ratio
        if m not in seen:
            seen.add(m)
            out.append(m)
    return out


# ----------------------------------------------------------------------------
# 4b. KV_SWAP: GgufKvSwapLayerState and gguf_kv_swap_in_selected
#     (section "KV_SWAP 实现细节", data structure and Swap-in flow)
# ----------------------------------------------------------------------------
class NotStoredError(RuntimeError):
    """A selected chunk has not been stored to the host cache yet
    (section "故障排查", error 4)."""


@dataclass
class SwapResult:
    phys: List[int]                       # window + slot (or window + chunk when resident)
    misses: List[Tuple[int, int]]         # (logical chunk, slot) in processing order
    hits: int


class KvSwapLayerState:
    """One (layer, sequence) of the swap state.

    ``slot_lru`` is the pages' ``std::list<int>`` with front = most recently
    used; it is held as an ordered dict whose LAST item is the front and whose
    FIRST item is the back, so ``pop_back`` = ``popitem(last=False)``. All slots
    start free at the back, slot 0 outermost, so the first misses fill slots
    0, 1, 2, ...
    """

    def __init__(self, compressed_cap_: int, gpu_chunks: int, window: int = WINDOW):
        self.compressed_cap = compressed_cap_
        self.gpu_chunks = gpu_chunks
        self.window = window
        self.swap_enabled = swap_enabled(compressed_cap_, gpu_chunks)
        self.host_ready = np.zeros(compressed_cap_, dtype=np.uint8)
        self.gpu_slot_logical = [-1] * gpu_chunks
        self.slot_by_logical: Dict[int, int] = {}
        self.slot_lru: "OrderedDict[int, None]" = OrderedDict((s, None) for s in range(gpu_chunks))
        self.hits = 0
        self.misses = 0
        # adaptive capacity (section 4c below): slots [0, capacity) are in use
        self.capacity = gpu_chunks
        self.next_capacity = gpu_chunks
        self.policy: Optional["AdaptivePolicy"] = None
        self.ep_steps = self.ep_hits = self.ep_sel = 0

    # -- adaptive capacity -------------------------------------------------
    def install_policy(self, policy: Optional["AdaptivePolicy"]) -> None:
        """The next swap step runs with ``policy.g_init`` slots (all
        ``gpu_chunks`` when ``policy`` is None); the hit-rate window restarts."""
        if policy is not None:
            policy.check(self.gpu_chunks)
        self.policy = policy
        self.next_capacity = policy.g_init if policy is not None else self.gpu_chunks
        self.ep_steps = self.ep_hits = self.ep_sel = 0

    def set_capacity(self, g: int) -> None:
        """Resize the slot range in use to [0, g) without moving any row.
        Growing adds the new slots, empty, at the back of the LRU list (lowest
        index outermost), so they are taken before any slot that holds a
        chunk. Shrinking drops slots [g, capacity): their chunks are no longer
        staged; the kept slots keep their chunks and their LRU order."""
        assert 1 <= g <= self.gpu_chunks
        cur = self.capacity
        if g > cur:
            order = list(range(cur, g)) + list(self.slot_lru)
            self.slot_lru = OrderedDict((s, None) for s in order)
        elif g < cur:
            for s in range(g, cur):
                c = self.gpu_slot_logical[s]
                if c >= 0:
                    del self.slot_by_logical[c]
                    self.gpu_slot_logical[s] = -1
                del self.slot_lru[s]
        self.capacity = g
        self.next_capacity = g

    def active_capacity(self) -> int:
        """Slots the next swap step uses (a pending resize is applied first)."""
        if self.swap_enabled and self.next_capacity != self.capacity:
            self.set_capacity(self.next_capacity)
        return self.capacity if self.swap_enabled else self.gpu_chunks

    def _account(self, hits: int, selected: int) -> None:
        """Hit-rate window of the policy: after ``epoch`` swap steps the window's
        hits/selected decides the capacity of the steps that follow."""
        p = self.policy
        if p is None:
            return
        self.ep_steps += 1
        self.ep_hits += hits
        self.ep_sel += selected
        if self.ep_steps < p.epoch:
            return
        g = self.capacity
        if self.ep_hits * 1000 < p.lo_permille * self.ep_sel:
            g = min(p.g_max, g + p.delta)
        elif self.ep_hits * 1000 > p.hi_permille * self.ep_sel:
            g = max(p.g_min, g - p.delta)
        self.next_capacity = g
        self.ep_steps = self.ep_hits = self.ep_sel = 0

    def store(self, logical: int) -> None:
        """Store flow: the chunk now exists in the host cache; a resident copy stays."""
        self.host_ready[logical] = 1

    def swap_in_selected(self, logical_ids: Sequence[int]) -> SwapResult:
        phys: List[int] = []
        misses: List[Tuple[int, int]] = []
        hits = 0
        if not self.swap_enabled:
            # swap disabled: every chunk is resident at its own index
            for c in logical_ids:
                if not self.host_ready[c]:
                    raise NotStoredError(f"chunk {c} selected before it was stored")
                phys.append(self.window + int(c))
            return SwapResult(phys, misses, 0)
        self.active_capacity()
        for c in logical_ids:
            c = int(c)
            slot = self.slot_by_logical.get(c)
            if slot is not None:
                self.slot_lru.move_to_end(slot)          # LRU touch: move to front
                hits += 1
            else:
                if not self.host_ready[c]:
                    raise NotStoredError(f"chunk {c} selected before it was stored")
                slot, _ = self.slot_lru.popitem(last=False)   # LRU evict: pop_back
                old = self.gpu_slot_logical[slot]
                if old >= 0:
                    del self.slot_by_logical[old]
                self.gpu_slot_logical[slot] = c
                self.slot_by_logical[c] = slot
                self.slot_lru[slot] = None               # the filled slot is the front
                misses.append((c, slot))                 # H2D h_compressed_kv[c] -> slot
            phys.append(self.window + slot)
        self.hits += hits
        self.misses += len(misses)
        self._account(hits, len(logical_ids))
        return SwapResult(phys, misses, hits)


# ----------------------------------------------------------------------------
# 4c. Adaptive GPU_CHUNKS from the runtime LRU hit rate (section "未来优化方向",
#     item 4: the staging capacity follows the measured hit rate). The pages
#     name the direction only; the rule below is this implementation's reading.
# ----------------------------------------------------------------------------
@dataclass(frozen=True)
class AdaptivePolicy:
    """Per (layer, sequence) of a swapped layer: every ``epoch`` swap steps the
    hit rate h = hits/selected of those steps sets the capacity of the next
    steps: h < lo_permille/1000 grows it by ``delta`` (up to ``g_max``),
    h > hi_permille/1000 shrinks it by ``delta`` (down to ``g_min``), otherwise
    it stays. The comparisons are exact integers (hits*1000 against
    permille*selected), so a window with nothing selected changes nothing."""
    g_min: int
    g_max: int
    g_init: int
    epoch: int
    lo_permille: int
    hi_permille: int
    delta: int

    def check(self, gpu_chunks: int) -> None:
        assert 1 <= self.g_min <= self.g_init <= self.g_max <= gpu_chunks
        assert self.epoch >= 1 and self.delta >= 1
        assert 0 <= self.lo_permille <= self.hi_permille <= 1000


# ----------------------------------------------------------------------------
# 5. Attention over window + selected chunks (K = V = the 512-wide latent row)
# ----------------------------------------------------------------------------
def attend(q_bits: np.ndarray, rows: np.ndarray) -> np.ndarray:
    """o_h = sum_j softmax_j(<q_h, e_j> / sqrt(D)) e_j, all in fp64. ``[H][D]``."""
    q = bf16_to_f64(q_bits)
    e = np.asarray(rows, dtype=np.float64)
    z = (q @ e.T) / math.sqrt(e.shape[1])
    z = z - z.max(axis=1, keepdims=True)
    p = np.exp(z)
    return (p @ e) / p.sum(axis=1, keepdims=True)


# ----------------------------------------------------------------------------
# The decode step
# ----------------------------------------------------------------------------
@dataclass
class StepResult:
    scores: List[np.ndarray]              # [B] of [n] fp64
    sel: List[np.ndarray]                 # [B] of selected chunk ids, in order
    lists: List[List[List[int]]]          # [L][B] per-layer ordered chunk lists
    swap: List[List[SwapResult]]          # [L][B]
    out: Dict[Tuple[int, int], np.ndarray] = field(default_factory=dict)  # (l, b) -> [H][512]


class DecodeOracle:
    """Holds the per-(layer, sequence) swap state across decode steps."""

    def __init__(self, *, context_len: int, layer_ratios: Sequence[int], gpu_chunks: int,
                 index_topk: int, batch: int, scale: float, bias: Sequence[float],
                 ensemble_mode: int, select_mode: int, tau: float, clamp: int,
                 src_ratio: int = 4, window: int = WINDOW):
        self.context_len = context_len
        self.layer_ratios = list(layer_ratios)
        self.gpu_chunks = gpu_chunks
        self.index_topk = index_topk
        self.batch = batch
        self.scale = scale
        self.bias = list(bias)
        self.ensemble_mode = ensemble_mode
        self.select_mode = select_mode
        self.tau = tau
        self.clamp = clamp
        self.src_ratio = src_ratio
        self.window = window
        self.caps = [compressed_cap(context_len, r) for r in self.layer_ratios]
        self.states = [[KvSwapLayerState(cap, gpu_chunks, window) for _ in range(batch)]
                       for cap in self.caps]

    def install_policy(self, policy: Optional[AdaptivePolicy]) -> None:
        """Adaptive capacity (section 4c) for every swapped (layer, sequence)."""
        for row in self.states:
            for st in row:
                if st.swap_enabled:
                    st.install_policy(policy)

    def mark_all_stored(self) -> None:
        for row in self.states:
            for st in row:
                st.host_ready[:] = 1

    def store(self, layer: int, seq: int, c0: int, n: int) -> None:
        """Store flow (section "KV_SWAP 实现细节", Store): chunks [c0, c0+n) of
        (layer, seq) now exist in the host cache. The swap state is untouched: a
        chunk already in a staging slot keeps it. The new content itself is
        whatever the caller's ``pool_rows_of`` returns from now on."""
        for c in range(c0, c0 + n):
            self.states[layer][seq].store(c)

    def step(self, keys_of: Callable[[int], np.ndarray], fm_q_of: Callable[[int], np.ndarray],
             attn_q_of: Optional[Callable[[int, int], np.ndarray]] = None,
             window_of: Optional[Callable[[int, int], np.ndarray]] = None,
             pool_rows_of: Optional[Callable[[int, int, Sequence[int]], np.ndarray]] = None,
             attend_pairs: Optional[Sequence[Tuple[int, int]]] = None, rescore: bool = True) -> StepResult:
        """One decode step. With ``rescore=False`` the step reuses the previous
        step's scores and selection (the memory indexer fires periodically,
        summary section "LSA 让模型预判 KV chunk"): only the swap-in and the
        attention run."""
        if rescore or not hasattr(self, "_last"):
            scores, sels = [], []
            for b in range(self.batch):
                k = np.asarray(keys_of(b))
                sc = score_multi if k.ndim == 3 else score   # [3][n][128]: per-indexer key sets
                s = sc(k, fm_q_of(b), self.scale, self.bias, self.ensemble_mode)
                scores.append(s)
                sels.append(select(s, self.select_mode, self.index_topk, self.tau, self.clamp))
            self._last = (scores, sels)
        else:
            scores, sels = self._last
        lists, swaps = [], []
        for l, ratio in enumerate(self.layer_ratios):
            row_l, row_s = [], []
            for b in range(self.batch):
                lst = layer_chunks(sels[b], self.src_ratio, ratio)
                g = self.states[l][b].active_capacity()
                if self.states[l][b].swap_enabled and len(lst) > g:
                    # fewer slots in use than chunks listed (GPU_CHUNKS < index_topk,
                    # a test-only setting, or a small adaptive capacity): the layer
                    # keeps the first chunks of its list, as many as it has slots
                    lst = lst[:g]
                row_l.append(lst)
                row_s.append(self.states[l][b].swap_in_selected(lst))
            lists.append(row_l)
            swaps.append(row_s)
        res = StepResult(scores, sels, lists, swaps)
        if attend_pairs is None and attn_q_of is not None:
            attend_pairs = [(l, b) for l in range(len(self.layer_ratios)) for b in range(self.batch)]
        for (l, b) in attend_pairs or []:
            rows = np.concatenate([np.asarray(window_of(l, b), dtype=np.float64),
                                   np.asarray(pool_rows_of(l, b, lists[l][b]), dtype=np.float64)
                                   .reshape(-1, KV_DIM)], axis=0)
            res.out[(l, b)] = attend(attn_q_of(l, b), rows)
        return res

    def lookahead_step(self, keys_of, fm_q_of, attn_q_of=None, window_of=None, pool_rows_of=None,
                       attend_pairs=None, trigger: bool = True) -> StepResult:
        """One step of the lookahead schedule (summary section "LSA 让模型预判 KV
        chunk": the indexer predicts, from the current token, the chunks the
        coming window of steps needs; PocketLLM doc, section "未来优化方向",
        item 2: take the scoring off the step's critical path). At a trigger
        step the indexer scores and selects and the selection is swapped in,
        while the step's attention still reads the selection in force; the new
        selection is in force from the next step on. Other steps only attend.
        Before the first trigger no chunk is in force (window rows only).
        ``lists`` and ``out`` describe the selection in force during the step;
        ``sel``, ``scores`` and ``swap`` the new selection (trigger steps)."""
        cur = getattr(self, "_in_force", None)
        if cur is None:
            cur = [[[] for _ in range(self.batch)] for _ in self.layer_ratios]
        if trigger:
            new = self.step(keys_of, fm_q_of)
            res = StepResult(new.scores, new.sel, cur, new.swap)
            self._in_force = new.lists
        else:
            res = StepResult([], [], cur, [])
        if attend_pairs is None and attn_q_of is not None:
            attend_pairs = [(l, b) for l in range(len(self.layer_ratios)) for b in range(self.batch)]
        for (l, b) in attend_pairs or []:
            rows = np.asarray(window_of(l, b), dtype=np.float64)
            if cur[l][b]:
                rows = np.concatenate([rows, np.asarray(pool_rows_of(l, b, cur[l][b]), dtype=np.float64)
                                       .reshape(-1, KV_DIM)], axis=0)
            res.out[(l, b)] = attend(attn_q_of(l, b), rows)
        return res
