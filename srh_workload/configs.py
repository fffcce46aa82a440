"""Workload shapes for the FlashMemory LSA + KV_SWAP decode step.

Shapes only: no part of the method's arithmetic lives here. Both the CUDA path
(through the Python binding) and the fp64 oracle read these shapes, and the
seeded generator in ``srh_workload.generate`` draws the inputs for them.

Sources of the numbers (PocketLLM "FlashMemory 1M 上下文显存优化使用文档"):
  * 20 ratio-4 layers + 21 ratio-128 layers, kv_dim 512, window 128
    (section "关键参数调优", item 2, the pinned-size examples).
  * index_topk 512, GPU_CHUNKS 512/1024 (item 1 of the same section).
  * ensemble max|mean (section "配置说明", env ``..._FLASHMEMORY_ENSEMBLE``).
The sigmoid-threshold selector, the three memory indexers and the lookahead
window come from the FlashMemory-DeepSeek-V4 summary (wmrh.cn/news/1094,
sections "LSA 让模型预判 KV chunk" and "Memory Indexer 放哪里").
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Tuple

KV_DIM = 512          # latent row width (fp32)
WINDOW = 128          # sliding-window rows
N_INDEXERS = 3        # memory indexers (layers 10/12/20)
INDEXER_HEADS = 8     # query heads per indexer
INDEXER_DIM = 128     # indexer key width (bf16)
SRC_RATIO = 4         # the scored chunks are the ratio-4 compressed chunks

ENSEMBLE_MAX = 0
ENSEMBLE_MEAN = 1
SELECT_TOPK = 0
SELECT_THRESH = 1


def compressed_cap(context_len: int, ratio: int) -> int:
    """Chunks a layer of compression ``ratio`` holds for ``context_len`` tokens."""
    return (context_len + ratio - 1) // ratio


@dataclass(frozen=True)
class Workload:
    name: str
    code: int                      # small integer folded into the seed
    context_len: int
    layer_ratios: Tuple[int, ...]  # one entry per sparse layer
    gpu_chunks: int                # G, staging slots per layer and sequence
    index_topk: int                # k
    ensemble: int                  # ENSEMBLE_MAX / ENSEMBLE_MEAN
    select_mode: int               # SELECT_TOPK / SELECT_THRESH
    tau: float                     # sigmoid threshold (THRESH mode)
    bias: float                    # per-indexer logit bias b_i (same for all i)
    n_heads: int                   # attention heads H (MQA over the latent)
    batch: int
    steps: int                     # decode steps of the scenario
    lookahead: int                 # steps the needle set is held fixed
    n_needles: int = 32
    seed: int = 0

    @property
    def n_chunks(self) -> int:
        """Scored chunks n = ratio-4 compressed capacity."""
        return compressed_cap(self.context_len, SRC_RATIO)

    @property
    def n_layers(self) -> int:
        return len(self.layer_ratios)

    def layer_cap(self, layer: int) -> int:
        return compressed_cap(self.context_len, self.layer_ratios[layer])

    @property
    def layer_caps(self) -> Tuple[int, ...]:
        return tuple(self.layer_cap(l) for l in range(self.n_layers))

    @property
    def clamp(self) -> int:
        """Maximum selected count: k for top-k, G for the threshold selector."""
        return self.index_topk if self.select_mode == SELECT_TOPK else self.gpu_chunks

    @property
    def scale(self) -> float:
        return INDEXER_DIM ** -0.5

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


def _layers(n4: int, n128: int) -> Tuple[int, ...]:
    return (4,) * n4 + (128,) * n128


TINY = Workload(
    name="tiny", code=1, context_len=8192, layer_ratios=_layers(1, 0),
    gpu_chunks=512, index_topk=512, ensemble=ENSEMBLE_MAX, select_mode=SELECT_TOPK,
    tau=0.5, bias=0.0, n_heads=16, batch=1, steps=32, lookahead=8)

CTX8K = Workload(
    name="ctx8k", code=2, context_len=8192, layer_ratios=_layers(20, 21),
    gpu_chunks=1024, index_topk=512, ensemble=ENSEMBLE_MAX, select_mode=SELECT_TOPK,
    tau=0.5, bias=0.0, n_heads=64, batch=1, steps=64, lookahead=16)

CTX256K = Workload(
    name="ctx256k", code=3, context_len=262144, layer_ratios=_layers(20, 21),
    gpu_chunks=1024, index_topk=512, ensemble=ENSEMBLE_MAX, select_mode=SELECT_TOPK,
    tau=0.5, bias=0.0, n_heads=64, batch=1, steps=128, lookahead=16)

CTX1M = Workload(
    name="ctx1m", code=4, context_len=1048576, layer_ratios=_layers(20, 21),
    gpu_chunks=512, index_topk=512, ensemble=ENSEMBLE_MEAN, select_mode=SELECT_THRESH,
    tau=0.5, bias=-7.0, n_heads=64, batch=1, steps=128, lookahead=4)


def batch_sweep(batch: int) -> Workload:
    return Workload(
        name=f"batch128k_b{batch}", code=5, context_len=131072, layer_ratios=_layers(20, 0),
        gpu_chunks=768, index_topk=512, ensemble=ENSEMBLE_MAX, select_mode=SELECT_TOPK,
        tau=0.5, bias=0.0, n_heads=64, batch=batch, steps=64, lookahead=16)


BATCH_SIZES = (1, 4, 8, 16, 32)

ALL = {w.name: w for w in (TINY, CTX8K, CTX256K, CTX1M)}
for _b in BATCH_SIZES:
    ALL[batch_sweep(_b).name] = batch_sweep(_b)


def get(name: str) -> Workload:
    return ALL[name]
