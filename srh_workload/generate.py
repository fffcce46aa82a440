"""Seeded synthetic inputs for the FlashMemory LSA + KV_SWAP decode step.

This module draws random inputs and nothing else: it holds none of the
method's arithmetic (no scoring, selection, LRU or attention). Both the CUDA
path and the fp64 oracle consume what it returns, so the two always see the
same bytes.

Every array is addressable piecewise: each block of rows has its own
``numpy.random.Generator(PCG64(SeedSequence(...)))`` keyed by
(seed, workload code, kind, indices), so a checker can regenerate any row of
a multi-GB pool without drawing the rest.

Recipe (plainest reading of the pages, sizes per ``srh_workload.configs``):
  * indexer keys ``K`` ~ N(0,1) rounded to bf16, ``[n][128]`` per sequence;
  * pool latents ~ N(0,1) fp32 ``[cap][512]`` per (layer, sequence);
  * window latents ~ N(0,1) fp32 ``[128][512]`` per (layer, sequence);
  * attention queries ~ N(0,1) rounded to bf16 ``[H][512]`` per
    (step, layer, sequence), fresh every step;
  * memory-indexer queries: per lookahead window and sequence, a set of
    ``n_needles`` distinct chunks drawn uniformly from ``[0, n)``; each of the
    3 indexers takes its own random permutation of the needles into its
    8 heads x 4 slots, and ``Q[i,h] = sum_j K[needle_{i,h,j}] + 0.5 * N(0, I)``
    (fp32 sum of the bf16 keys), rounded to bf16. Needles and noise are
    redrawn at each lookahead-window boundary, so queries repeat within a
    window (the lookahead indexer predicts a short decoding window ahead).
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from typing import Sequence

import numpy as np

from .configs import (INDEXER_DIM, INDEXER_HEADS, KV_DIM, N_INDEXERS, WINDOW,
                      Workload)

KIND_KEYS = 1
KIND_POOL = 2
KIND_WINDOW = 3
KIND_ATTNQ = 4
KIND_NEEDLES = 5
KIND_KEY_SET = 6       # key sets 1 and 2 of the per-indexer-keys variant

KEY_BLOCK = 1024     # key rows per generator
POOL_BLOCK = 32      # pool rows per generator
SLOTS_PER_HEAD = 4   # planted key directions per indexer head
NOISE_STD = 0.5


def _rng(w: Workload, kind: int, *idx: int) -> np.random.Generator:
    ss = np.random.SeedSequence([w.seed, w.code, kind, *[int(i) for i in idx]])
    return np.random.Generator(np.random.PCG64(ss))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32 (input preparation only)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------- keys
def key_block(w: Workload, seq: int, block: int) -> np.ndarray:
    n = w.n_chunks
    lo = block * KEY_BLOCK
    rows = min(KEY_BLOCK, n - lo)
    g = _rng(w, KIND_KEYS, seq, block)
    return f32_to_bf16_bits(g.standard_normal((rows, INDEXER_DIM), dtype=np.float32))


def keys(w: Workload, seq: int) -> np.ndarray:
    """bf16 bits ``[n][128]`` for one sequence."""
    n = w.n_chunks
    out = np.empty((n, INDEXER_DIM), dtype=np.uint16)
    for b in range((n + KEY_BLOCK - 1) // KEY_BLOCK):
        out[b * KEY_BLOCK:(b + 1) * KEY_BLOCK] = key_block(w, seq, b)
    return out


def key_rows(w: Workload, seq: int, idx: Sequence[int]) -> np.ndarray:
    idx = np.asarray(idx, dtype=np.int64)
    out = np.empty((len(idx), INDEXER_DIM), dtype=np.uint16)
    cache = {}
    for j, c in enumerate(idx):
        b = int(c) // KEY_BLOCK
        if b not in cache:
            cache[b] = key_block(w, seq, b)
        out[j] = cache[b][int(c) - b * KEY_BLOCK]
    return out


def key_set_block(w: Workload, i: int, seq: int, block: int) -> np.ndarray:
    """Block of key set i (set 0 is the shared key set of ``keys``)."""
    if i == 0:
        return key_block(w, seq, block)
    n = w.n_chunks
    lo = block * KEY_BLOCK
    rows = min(KEY_BLOCK, n - lo)
    g = _rng(w, KIND_KEY_SET, i, seq, block)
    return f32_to_bf16_bits(g.standard_normal((rows, INDEXER_DIM), dtype=np.float32))


def keys_multi(w: Workload, seq: int) -> np.ndarray:
    """bf16 bits ``[3][n][128]``: one key set per memory indexer (set 0 = ``keys``)."""
    n = w.n_chunks
    out = np.empty((N_INDEXERS, n, INDEXER_DIM), dtype=np.uint16)
    for i in range(N_INDEXERS):
        for b in range((n + KEY_BLOCK - 1) // KEY_BLOCK):
            out[i, b * KEY_BLOCK:(b + 1) * KEY_BLOCK] = key_set_block(w, i, seq, b)
    return out


def _key_set_rows(w: Workload, i: int, seq: int, idx) -> np.ndarray:
    idx = np.asarray(idx, dtype=np.int64)
    out = np.empty((len(idx), INDEXER_DIM), dtype=np.uint16)
    cache = {}
    for j, c in enumerate(idx):
        b = int(c) // KEY_BLOCK
        if b not in cache:
            cache[b] = key_set_block(w, i, seq, b)
        out[j] = cache[b][int(c) - b * KEY_BLOCK]
    return out


# --------------------------------------------------------------------------- pools
def pool_block(w: Workload, layer: int, seq: int, block: int) -> np.ndarray:
    cap = w.layer_cap(layer)
    lo = block * POOL_BLOCK
    rows = min(POOL_BLOCK, cap - lo)
    g = _rng(w, KIND_POOL, layer, seq, block)
    return g.standard_normal((rows, KV_DIM), dtype=np.float32)


def fill_pool(w: Workload, layer: int, seq: int, out: np.ndarray, threads: int | None = None) -> None:
    """Write the full pool ``[cap][512]`` fp32 of (layer, seq) into ``out``."""
    cap = w.layer_cap(layer)
    assert out.shape == (cap, KV_DIM) and out.dtype == np.float32
    nblk = (cap + POOL_BLOCK - 1) // POOL_BLOCK

    def work(b0: int, b1: int) -> None:
        for b in range(b0, b1):
            out[b * POOL_BLOCK:(b + 1) * POOL_BLOCK] = pool_block(w, layer, seq, b)

    threads = threads or min(16, os.cpu_count() or 1)
    if nblk < 64 or threads <= 1:
        work(0, nblk)
        return
    step = (nblk + threads - 1) // threads
    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(lambda i: work(i * step, min(nblk, (i + 1) * step)), range(threads)))


def pool(w: Workload, layer: int, seq: int) -> np.ndarray:
    out = np.empty((w.layer_cap(layer), KV_DIM), dtype=np.float32)
    fill_pool(w, layer, seq, out)
    return out


def pool_rows(w: Workload, layer: int, seq: int, idx: Sequence[int]) -> np.ndarray:
    idx = np.asarray(idx, dtype=np.int64)
    out = np.empty((len(idx), KV_DIM), dtype=np.float32)
    cache = {}
    for j, c in enumerate(idx):
        b = int(c) // POOL_BLOCK
        if b not in cache:
            cache[b] = pool_block(w, layer, seq, b)
        out[j] = cache[b][int(c) - b * POOL_BLOCK]
    return out


# --------------------------------------------------------------------------- window
def window(w: Workload, layer: int, seq: int) -> np.ndarray:
    g = _rng(w, KIND_WINDOW, layer, seq)
    return g.standard_normal((WINDOW, KV_DIM), dtype=np.float32)


# --------------------------------------------------------------------------- queries
def attn_q(w: Workload, step: int, layer: int, seq: int) -> np.ndarray:
    """bf16 bits ``[H][512]``: the attention query of (step, layer, seq)."""
    g = _rng(w, KIND_ATTNQ, step, layer, seq)
    return f32_to_bf16_bits(g.standard_normal((w.n_heads, KV_DIM), dtype=np.float32))


def _needle_plan(w: Workload, window_idx: int, seq: int):
    g = _rng(w, KIND_NEEDLES, window_idx, seq)
    n_nd = min(w.n_needles, w.n_chunks)
    nd = np.sort(g.choice(w.n_chunks, size=n_nd, replace=False)).astype(np.int64)
    per_head = INDEXER_HEADS * SLOTS_PER_HEAD
    plan = np.empty((N_INDEXERS, INDEXER_HEADS, SLOTS_PER_HEAD), dtype=np.int64)
    for i in range(N_INDEXERS):
        perm = g.permutation(n_nd)
        # every needle appears in each indexer; extra slots wrap around the set
        take = np.resize(perm, per_head)
        plan[i] = nd[take].reshape(INDEXER_HEADS, SLOTS_PER_HEAD)
    noise = g.standard_normal((N_INDEXERS, INDEXER_HEADS, INDEXER_DIM), dtype=np.float32)
    return nd, plan, noise


def fm_queries(w: Workload, step: int, seq: int) -> np.ndarray:
    """bf16 bits ``[3][8][128]``: memory-indexer queries of (step, seq)."""
    window_idx = step // w.lookahead
    _, plan, noise = _needle_plan(w, window_idx, seq)
    flat = plan.reshape(-1)
    k = bf16_bits_to_f32(key_rows(w, seq, flat)).reshape(N_INDEXERS, INDEXER_HEADS,
                                                          SLOTS_PER_HEAD, INDEXER_DIM)
    q = k.sum(axis=2, dtype=np.float32) + np.float32(NOISE_STD) * noise
    return f32_to_bf16_bits(q)


def fm_queries_multi(w: Workload, step: int, seq: int) -> np.ndarray:
    """Like ``fm_queries`` for per-indexer key sets: indexer i's needle
    directions are taken from key set i."""
    window_idx = step // w.lookahead
    _, plan, noise = _needle_plan(w, window_idx, seq)
    q = np.empty((N_INDEXERS, INDEXER_HEADS, INDEXER_DIM), dtype=np.float32)
    for i in range(N_INDEXERS):
        k = bf16_bits_to_f32(_key_set_rows(w, i, seq, plan[i].reshape(-1))).reshape(
            INDEXER_HEADS, SLOTS_PER_HEAD, INDEXER_DIM)
        q[i] = k.sum(axis=1, dtype=np.float32) + np.float32(NOISE_STD) * noise[i]
    return f32_to_bf16_bits(q)


def step_needles(w: Workload, step: int, seq: int) -> np.ndarray:
    return _needle_plan(w, step // w.lookahead, seq)[0]
