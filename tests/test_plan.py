"""CPU checks of lsa_attend's static work split (srh_attend_plan_info, host
only): every plan keeps its invariants, never has more CTAs than SMs, and
spreads the rows' bytes evenly -- fp32 window rows count 2 KiB, fp16 staged
rows 1 KiB (the staging layout of kvswap_stage)."""
import shutil

import pytest

from srh_workload import configs as C

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and not __import__("os").path.exists(
    "/usr/local/cuda/bin/nvcc"), reason="nvcc not available")

MIN_CHUNK_KIB = 128      # the even share is never taken below one staged tile


@pytest.fixture(scope="module")
def abi():
    import __graft_entry__
    __graft_entry__.build()
    from sparse_retrieval_host_gb300 import abi as a
    return a


def _cfg(abi, w, **over):
    kw = dict(batch=w.batch, layer_ratios=w.layer_ratios, gpu_chunks=w.gpu_chunks, index_topk=w.index_topk,
              context_len=w.context_len)
    kw.update(over)
    return abi.make_config(**kw)


def _pair_kib(ctx_len, ratio, s):
    """KiB of one (layer, seq)'s rows: 128 window rows of 2 KiB, min(S, cap) staged rows of 1 KiB."""
    cap = (ctx_len + ratio - 1) // ratio
    return 2 * 128 + min(s, cap)


@pytest.mark.parametrize("name", sorted(C.ALL))
@pytest.mark.parametrize("sms", [152, 148, 132, 16])
def test_plans_keep_invariants_and_balance_bytes(abi, name, sms):
    w = C.ALL[name]
    s = w.index_topk
    scopes = [(-1, list(range(w.n_layers)))] + [(l, [l]) for l in sorted({w.layer_ratios.index(r) for r in
                                                                            set(w.layer_ratios)})]
    for layer, layers in scopes:
        info = abi.srh_attend_plan_info(_cfg(abi, w), sms, layer)
        assert info["valid"], (name, layer, info)
        assert 1 <= info["ctas"] <= sms
        pairs = [_pair_kib(w.context_len, w.layer_ratios[l], s) for l in layers for _ in range(w.batch)]
        even = max(-(-sum(pairs) // sms), MIN_CHUNK_KIB)
        if info["one_wave"]:
            # every pair on CTAs of its own, one tile (<= 128 rows, <= 256 KiB) per CTA
            assert info["ctas"] >= len(pairs) and info["segments"] == info["ctas"]
            assert info["max_cta_kib"] <= 256, (name, layer, info)
        else:
            # whole tiles, equal bytes to the nearest tile (a window tile is 256 KiB)
            assert info["max_cta_kib"] <= even + 256, (name, layer, info, even)


def test_ctx8k_step_is_one_wave_of_single_tiles(abi):
    """The 8K decode step at batch 1: 41 pairs (640 rows on the ratio-4 layers,
    192 on the ratio-128 layers) become 142 one-tile chunks; a ratio-128 pair's
    two chunks share its 320 KiB evenly (160 + 160 rather than 256 + 64)."""
    info = abi.srh_attend_plan_info(_cfg(abi, C.CTX8K), 152)
    assert info["one_wave"] and info["valid"]
    assert info["ctas"] == 142 and info["split_pairs"] == 41
    assert info["max_cta_kib"] == 256
    last = abi.srh_attend_plan_info(_cfg(abi, C.CTX8K), 152, C.CTX8K.n_layers - 1)
    assert last["ctas"] == 2 and last["max_cta_kib"] == 160


def test_spare_sms_split_window_tiles(abi):
    """With SMs to spare (20 ratio-4 pairs of 640 rows, 100 tiles, on 152 SMs)
    each pair gets a sixth CTA and no chunk holds more than 128 KiB."""
    info = abi.srh_attend_plan_info(_cfg(abi, C.ALL["batch128k_b1"]), 152)
    assert info["one_wave"] and info["valid"]
    assert info["ctas"] == 120 and info["max_cta_kib"] == 128


@pytest.mark.parametrize("batch,select", [(1, 1), (1, 4096), (64, 512), (3, 100)])
def test_edge_shapes(abi, batch, select):
    """One staged row per pair, the largest selection, a wide batch and an odd
    selection size: plans stay valid and within the SM count."""
    ratios = [4] * 3 + [128] * 2
    cfg = abi.make_config(batch=batch, layer_ratios=ratios, gpu_chunks=max(select, 512), index_topk=select,
                          context_len=1 << 20)
    for sms in (1, 7, 152):
        for layer in (-1, 0, 4):
            info = abi.srh_attend_plan_info(cfg, sms, layer)
            assert info["valid"] and 1 <= info["ctas"] <= sms, (batch, select, sms, layer, info)


def test_rejects_bad_arguments(abi):
    cfg = _cfg(abi, C.CTX8K)
    with pytest.raises(abi.SrhError):
        abi.srh_attend_plan_info(cfg, 0)
    with pytest.raises(abi.SrhError):
        abi.srh_attend_plan_info(cfg, 152, C.CTX8K.n_layers)
