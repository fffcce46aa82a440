"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each test checks one oracle function against what the pages print, a closed
form, an invariant, an independent brute-force formulation, or a library
routine. A plausible slip in the oracle (a dropped term, a wrong sign or
index, a transposed operand, a wrong tie-break) fails at least one of them.
"""
import math
import os
import random
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import srh_oracle as O
from srh_workload import configs as C
from srh_workload import generate as G

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


# --------------------------------------------------------------------------- pinned sizes
def _printed_close(value_mb: float, printed: str) -> bool:
    """True if ``value_mb`` rounds to the printed figure (its last printed digit)."""
    digits = len(printed.split(".")[1]) if "." in printed else 0
    p = float(printed)
    if digits == 0:
        # integers such as "134" or "2680" carry 2-3 significant digits on the page
        sig = len(printed.rstrip("0")) or 1
        unit = 10 ** (len(printed) - sig)
        return abs(value_mb - p) <= 0.5 * unit + 1e-9
    return abs(value_mb - p) <= 0.5 * 10 ** (-digits) + 1e-9


def test_pinned_formula_matches_page_examples():
    """Section "关键参数调优" item 2: per-layer pinned bytes and per-ratio totals."""
    n = 0
    for row in _golden_rows("pinned_sizes.txt"):
        if row[0] == "total":
            continue
        ctx, ratio, layers, cap = (int(x) for x in row[:4])
        per_mb, total_mb = row[4], row[5]
        assert O.compressed_cap(ctx, ratio) == cap
        per = O.layer_pinned_bytes(ctx, ratio)
        assert per == cap * 512 * 4
        assert _printed_close(per / 1e6, per_mb), (ctx, ratio, per / 1e6, per_mb)
        exact_total = O.required_pinned_bytes(ctx, [ratio] * layers) / 1e6
        # the page multiplies its rounded per-layer figure by the layer count
        assert abs(float(per_mb) * layers - float(total_mb)) <= 0.02 * float(total_mb) + 0.05
        assert abs(exact_total - float(total_mb)) <= 0.02 * float(total_mb) + 0.05
        n += 1
    assert n == 6


def test_pinned_grand_totals():
    """Grand totals ~87 MB / ~2.77 GB / ~11 GB for 20 ratio-4 + 21 ratio-128 layers."""
    ratios = [4] * 20 + [128] * 21
    for row in _golden_rows("pinned_sizes.txt"):
        if row[0] != "total":
            continue
        ctx, printed = int(row[1]), float(row[2])
        got = O.required_pinned_bytes(ctx, ratios) / 1e6
        assert abs(got - printed) <= 0.01 * printed + 0.5, (ctx, got, printed)


def test_compressed_cap_rounds_up():
    assert O.compressed_cap(64, 4) == 16
    assert O.compressed_cap(65, 4) == 17
    assert O.compressed_cap(1, 128) == 1
    assert O.compressed_cap(128, 128) == 1
    assert O.compressed_cap(129, 128) == 2
    assert O.compressed_cap(0, 4) == 0


def test_log_example_numbers():
    """Section "使用示例", 示例 1: pinned_mib=84, max_capacity=640, stats totals."""
    g = {r[0]: int(r[1]) for r in _golden_rows("log_example.txt")}
    cap = O.compressed_cap(g["context_len"], g["ratio"])
    n = g["swapped_layers"]
    assert O.swap_enabled(cap, g["gpu_chunks"])
    assert O.required_pinned_bytes(g["context_len"], [g["ratio"]] * n) // 2**20 == g["pinned_mib"]
    assert g["window"] + g["gpu_chunks"] == g["max_capacity"]
    assert n * g["gpu_chunks"] == g["gpu_chunks_total"]
    assert n * cap == g["compressed_cap_total"]
    # section "故障排查": 64-token context, ratio 4
    short = O.compressed_cap(g["short_context_len"], 4)
    assert short == g["short_compressed_cap"]
    assert not O.swap_enabled(short, g["short_gpu_chunks_disabled"])
    assert O.swap_enabled(short, g["short_gpu_chunks_enabled"])


# --------------------------------------------------------------------------- scoring
def _bf16_exact(bits: int) -> Fraction:
    """bf16 value as an exact rational, decoded field by field."""
    s, e, m = (bits >> 15) & 1, (bits >> 7) & 0xFF, bits & 0x7F
    assert e != 0xFF
    if e == 0:
        v = Fraction(m, 128) * Fraction(1, 2 ** 126)
    else:
        v = Fraction(128 + m, 128) * (Fraction(2) ** (e - 127))
    return -v if s else v


def test_head_dots_exact_against_rational_arithmetic():
    rng = np.random.default_rng(7)
    keys = G.f32_to_bf16_bits(rng.standard_normal((9, 128), dtype=np.float32))
    q = G.f32_to_bf16_bits(2.0 * rng.standard_normal((3, 8, 128), dtype=np.float32))
    d = O.head_dots(keys, q)
    assert d.shape == (9, 3, 8)
    for c in range(9):
        for i in range(3):
            for h in range(8):
                exact = sum(_bf16_exact(int(a)) * _bf16_exact(int(b))
                            for a, b in zip(keys[c], q[i, h]))
                assert Fraction(d[c, i, h]) == exact, (c, i, h)


def _bits(x):
    return G.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def test_logit_is_scaled_max_over_heads_plus_indexer_bias():
    # one chunk whose key is 2*e_0; head h of indexer i carries (i*8 + h + 1) * e_0
    key = np.zeros((1, 128), np.float32)
    key[0, 0] = 2.0
    q = np.zeros((3, 8, 128), np.float32)
    for i in range(3):
        for h in range(8):
            q[i, h, 0] = (-1.0) ** h * (i * 8 + h + 1)
    bias = [0.25, -1.0, 3.0]
    lg = O.indexer_logits(_bits(key), _bits(q), 0.5, bias)
    # largest head of indexer i: h = 6 (positive, even) -> 2 * (8i + 7)
    want = [0.5 * 2 * (8 * i + 7) + bias[i] for i in range(3)]
    assert np.array_equal(lg[:, 0], np.array(want))
    assert O.ensemble(lg, O.ENSEMBLE_MAX)[0] == max(want)
    assert O.ensemble(lg, O.ENSEMBLE_MEAN)[0] == pytest.approx(sum(want) / 3, abs=0)


def test_per_indexer_keys_exact_and_isolated():
    """Multi-layer compressed_k (限制与未来工作): indexer i scores key set i only.
    Exact against rational arithmetic; three equal sets give the shared-key
    score; changing set 1 moves only indexer 1's logits."""
    rng = np.random.default_rng(21)
    keys3 = G.f32_to_bf16_bits(rng.standard_normal((3, 7, 128), dtype=np.float32))
    q = G.f32_to_bf16_bits(rng.standard_normal((3, 8, 128), dtype=np.float32))
    bias = [0.5, -0.25, 1.0]
    lg = O.indexer_logits_multi(keys3, q, 0.5, bias)
    for i in range(3):
        for c in range(7):
            best = max(sum(_bf16_exact(int(a)) * _bf16_exact(int(b)) for a, b in zip(keys3[i, c], q[i, h]))
                       for h in range(8))
            assert Fraction(lg[i, c]) == Fraction(1, 2) * best + Fraction(bias[i]), (i, c)
    same = np.stack([keys3[0]] * 3)
    assert np.array_equal(O.indexer_logits_multi(same, q, 0.5, bias), O.indexer_logits(keys3[0], q, 0.5, bias))
    other = keys3.copy()
    other[1] = G.f32_to_bf16_bits(rng.standard_normal((7, 128), dtype=np.float32))
    lg2 = O.indexer_logits_multi(other, q, 0.5, bias)
    assert np.array_equal(lg2[0], lg[0]) and np.array_equal(lg2[2], lg[2])
    assert not np.array_equal(lg2[1], lg[1])


def test_e4m3_decode_follows_the_format():
    """e4m3: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits, no infinities,
    0x7F / 0xFF NaN; subnormals m * 2^-9."""
    want = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0, 0x39: 1.125,
            0x7E: 448.0, 0xB8: -1.0, 0xFE: -448.0}
    got = O.e4m3_decode(np.array(list(want), np.uint8))
    assert np.array_equal(got, np.array(list(want.values())))
    assert np.isnan(O.e4m3_decode(np.array([0x7F, 0xFF], np.uint8))).all()
    pos = O.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0)                       # 127 distinct, increasing values


def test_e4m3_encode_rounds_to_nearest_even_and_saturates():
    codes = np.arange(0x7F, dtype=np.uint8)
    vals = O.e4m3_decode(codes)
    assert np.array_equal(O.e4m3_encode(vals), codes)      # every value is its own code
    assert np.array_equal(O.e4m3_encode(-vals[1:]), codes[1:] | 0x80)
    mid = (vals[:-1] + vals[1:]) / 2                      # exact midpoints go to the even code
    even = np.where(codes[:-1] % 2 == 0, codes[:-1], codes[1:])
    assert np.array_equal(O.e4m3_encode(mid), even)
    assert np.array_equal(O.e4m3_encode(np.nextafter(mid, np.inf)), codes[1:])
    assert np.array_equal(O.e4m3_encode(np.nextafter(mid, -np.inf)), codes[:-1])
    assert list(O.e4m3_encode([449.0, 1e9, -1e9])) == [0x7E, 0x7E, 0xFE]
    assert list(O.e4m3_encode([-0.0, -2.0 ** -12])) == [0x80, 0x80]


def test_fp8_key_quantization_and_score():
    rng = np.random.default_rng(17)
    keys = G.f32_to_bf16_bits(rng.standard_normal((64, 128), dtype=np.float32))
    keys[5] = 0                                           # an all-zero key
    codes, ks = O.quantize_keys_fp8(keys)
    k = O.bf16_to_f64(keys)
    assert ks.dtype == np.float32 and ks[5] == 0 and not codes[5].any()
    amax_at = np.abs(k).argmax(axis=1)
    for c in range(64):
        if c == 5:
            continue
        assert codes[c, amax_at[c]] & 0x7F == 0x7E          # the largest element maps to +-448
        deq = O.e4m3_decode(codes[c]) * float(ks[c])
        assert np.all(np.abs(deq - k[c]) <= np.maximum(2.0 ** -4 * np.abs(k[c]), 2.0 ** -10 * float(ks[c])))
    q = G.f32_to_bf16_bits(rng.standard_normal((3, 8, 128), dtype=np.float32))
    lg = O.indexer_logits_fp8(codes, ks, q, 0.25, [0.5, 0.0, -1.0])
    deq = O.e4m3_decode(codes) * ks.astype(np.float64)[:, None]
    qq = O.bf16_to_f64(q)
    for i in range(3):
        want = 0.25 * np.max(deq @ qq[i].T, axis=1) + [0.5, 0.0, -1.0][i]
        assert np.allclose(lg[i], want, rtol=1e-13, atol=1e-13)


def _e4m3_exact(code: int) -> Fraction:
    """e4m3 value as an exact rational, from the format's fields: sign, 4
    exponent bits with bias 7, 3 mantissa bits; subnormals m * 2^-9."""
    s, e, m = (code >> 7) & 1, (code >> 3) & 0xF, code & 0x7
    assert (code & 0x7F) != 0x7F
    v = Fraction(m, 512) if e == 0 else Fraction(8 + m, 8) * Fraction(2) ** (e - 7)
    return -v if s else v


def _rne_f32(x: Fraction) -> Fraction:
    """Round a rational to the nearest binary32 value, ties to the even
    significand (normal and subnormal range; no overflow in these cases)."""
    if x == 0:
        return Fraction(0)
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1                                            # now 2^e <= a < 2^(e+1)
    ulp = Fraction(2) ** (max(e, -126) - 23)
    n, rem = divmod(a, ulp)
    n = int(n)
    if rem * 2 > ulp or (rem * 2 == ulp and n % 2 == 1):
        n += 1
    return n * ulp if x > 0 else -(n * ulp)


def _e4m3_rne(x: Fraction) -> int:
    """Nearest e4m3 code of a rational, ties to the even code, saturated at
    +-448, sign kept (searched over all 127 finite magnitudes)."""
    a = min(abs(x), Fraction(448))
    best = min(range(0x7F), key=lambda c: (abs(_e4m3_exact(c) - a), c & 1))
    return best | (0x80 if x < 0 else 0)


def test_fp8_quantizer_divides_in_fp32():
    """The codes are decided by the fp32 quotient K / kscale (the reading the
    device kernel follows): a crafted row whose fp32 quotient lands exactly on
    an e4m3 midpoint, where an fp64 quotient lies just above it and would give
    the next code. Expected codes come from exact rational arithmetic: kscale =
    rn32(amax / 448), quotient = rn32(K / kscale), code = the e4m3 value nearest
    to it (ties to even)."""
    row = np.zeros((1, 128), np.float32)
    vals = [7.5, 0.001373291015625, 0.0006866455078125, 0.00034332275390625, -0.001373291015625, 0.30078125, -2.0]
    row[0, :len(vals)] = vals
    bits = G.f32_to_bf16_bits(row)
    assert np.array_equal(G.bf16_bits_to_f32(bits), row)          # every value is a bf16 value
    codes, ks = O.quantize_keys_fp8(bits)
    kscale = _rne_f32(Fraction(7.5) / 448)
    assert Fraction(float(ks[0])) == kscale
    fp64_differs = 0
    for d in range(128):
        x = Fraction(float(row[0, d]))
        want = _e4m3_rne(_rne_f32(x / kscale))
        assert int(codes[0, d]) == want, (d, hex(int(codes[0, d])), hex(want))
        fp64_differs += _e4m3_rne(Fraction(float(x) / float(kscale))) != want
    assert int(codes[0, 1]) == 0x1A and int(codes[0, 4]) == 0x9A   # the midpoint 0.08203125 rounds to even
    assert fp64_differs >= 3                                        # an fp64 division gives other codes here


def test_fp8_logits_exact_against_rational_arithmetic():
    """s_i(c) = scale * kscale_c * max_h <Q[i,h], e4m3(K8[c])> + b_i, checked
    against exact rationals built from the code and bf16 bit fields. A dropped
    chunk scale, a scale applied inside the max, a wrong head or indexer index,
    or a missing bias fails it."""
    rng = np.random.default_rng(29)
    keys = G.f32_to_bf16_bits((rng.standard_normal((6, 128)) * rng.uniform(0.05, 20, (6, 1))).astype(np.float32))
    codes, ks = O.quantize_keys_fp8(keys)
    q = G.f32_to_bf16_bits(rng.standard_normal((3, 8, 128), dtype=np.float32))
    scale, bias = 128 ** -0.5, [0.75, -3.0, 0.0]
    lg = O.indexer_logits_fp8(codes, ks, q, scale, bias)
    for c in range(6):
        k = [_e4m3_exact(int(v)) for v in codes[c]]
        for i in range(3):
            best = max(sum(a * _bf16_exact(int(b)) for a, b in zip(k, q[i, h])) for h in range(8))
            term = Fraction(scale) * Fraction(float(ks[c])) * best
            exact = term + Fraction(bias[i])
            err = abs(Fraction(float(lg[i, c])) - exact)
            assert err <= (abs(term) + abs(Fraction(bias[i]))) * Fraction(1, 2 ** 50), (i, c)


def test_fp8_keys_still_find_the_needles():
    w = C.TINY
    codes, ks = O.quantize_keys_fp8(G.keys(w, 0))
    for t in (0, 8, 16):
        s = O.score_fp8(codes, ks, G.fm_queries(w, t, 0), w.scale, [0.0] * 3, w.ensemble)
        assert np.isin(G.step_needles(w, t, 0), O.select_topk(s, w.index_topk)).all()


def test_or_mode_max_threshold_is_union_of_indexers():
    """Summary section "Memory Indexer 放哪里": a chunk is recalled if ANY indexer recalls it."""
    rng = np.random.default_rng(3)
    keys = G.f32_to_bf16_bits(rng.standard_normal((500, 128), dtype=np.float32))
    q = G.f32_to_bf16_bits(rng.standard_normal((3, 8, 128), dtype=np.float32))
    lg = O.indexer_logits(keys, q, 128 ** -0.5, [-2.0, -2.5, -1.5])
    s = O.ensemble(lg, O.ENSEMBLE_MAX)
    for tau in (0.3, 0.5, 0.8):
        t = O.threshold_logit(tau)
        union = set(np.nonzero((lg > t).any(axis=0))[0].tolist())
        got = set(O.select_threshold(s, tau, 10 ** 9).tolist())
        assert got == union


def test_sigmoid_threshold_equivalence():
    rng = np.random.default_rng(11)
    s = rng.normal(0, 3, 4000)
    for tau in (0.1, 0.5, 0.9):
        t = O.threshold_logit(tau)
        keep = np.abs(s - t) > 1e-9
        sig = 1.0 / (1.0 + np.exp(-s))
        assert np.array_equal((sig > tau)[keep], (s > t)[keep])
    assert O.threshold_logit(0.5) == 0.0


# --------------------------------------------------------------------------- selection
def _rank_bruteforce(s):
    n = len(s)
    return [sum(1 for j in range(n) if s[j] > s[i] or (s[j] == s[i] and j < i)) for i in range(n)]


@pytest.mark.parametrize("n,k", [(1, 1), (7, 3), (33, 8), (64, 17), (64, 64), (20, 50)])
def test_topk_matches_rank_definition(n, k):
    rng = np.random.default_rng(n * 100 + k)
    s = rng.choice([-1.5, 0.0, 0.25, 2.0, 3.0], size=n) + rng.choice([0.0, 1e-3], size=n)
    rank = _rank_bruteforce(list(s))
    want = [i for _, i in sorted((r, i) for i, r in enumerate(rank))][:min(k, n)]
    assert O.select_topk(s, k).tolist() == want


def test_topk_k_at_least_n_selects_everything_in_order():
    s = np.array([0.5, 2.0, 0.5, -1.0, 2.0])
    assert O.select_topk(s, 5).tolist() == [1, 4, 0, 2, 3]
    assert O.select_topk(s, 99).tolist() == [1, 4, 0, 2, 3]


def test_threshold_is_strict_ordered_and_clamped():
    s = np.array([0.0, 1.0, -0.5, 3.0, 1.0, 1e-12, -1e-12])
    assert O.select_threshold(s, 0.5, 100).tolist() == [3, 1, 4, 5]
    assert O.select_threshold(s, 0.5, 2).tolist() == [3, 1]
    assert O.select_threshold(s, 0.5, 0).tolist() == []
    rng = np.random.default_rng(5)
    s = rng.choice([-1.0, 0.5, 0.75, 1.5], size=40)
    rank = _rank_bruteforce(list(s))
    over = sorted((rank[i], i) for i in range(40) if s[i] > 0.0)
    assert O.select_threshold(s, 0.5, 9).tolist() == [i for _, i in over][:9]


# --------------------------------------------------------------------------- ratio mapping
def test_layer_chunks_ratio_mapping():
    assert O.layer_chunks([5, 37, 33, 64, 3], 4, 4) == [5, 37, 33, 64, 3]
    assert O.layer_chunks([5, 37, 33, 64, 3], 4, 128) == [0, 1, 2]
    assert O.layer_chunks([40, 8, 9, 41], 4, 8) == [20, 4]
    assert O.layer_chunks([], 4, 128) == []


# --------------------------------------------------------------------------- LRU
def _lru_textbook(steps, G_):
    """Textbook LRU by timestamps: hit iff fewer than G other distinct chunks were
    referenced since the last reference (stack distance); a miss fills the lowest
    free slot, else the slot of the chunk referenced longest ago."""
    last, slot_of, out, t = {}, {}, [], 0
    for refs in steps:
        res = []
        for c in refs:
            if c in last:
                since = {x for x, tt in last.items() if tt > last[c]}
                hit_sd = len(since) < G_
            else:
                hit_sd = False
            hit = c in slot_of
            assert hit == hit_sd
            if hit:
                slot = slot_of[c]
            elif len(slot_of) < G_:
                slot = min(set(range(G_)) - set(slot_of.values()))
                slot_of[c] = slot
            else:
                victim = min(slot_of, key=lambda x: last[x])
                slot = slot_of.pop(victim)
                slot_of[c] = slot
            last[c] = t
            t += 1
            res.append((hit, slot))
        out.append(res)
    return out, slot_of


def _random_trace(seed, G_, universe, n_steps):
    r = random.Random(seed)
    steps, prev = [], []
    for _ in range(n_steps):
        m = r.randint(0, G_)
        keep = [c for c in prev if r.random() < 0.7]
        pool = [c for c in range(universe) if c not in keep]
        new = r.sample(pool, max(0, min(m - len(keep), len(pool))))
        refs = (keep + new)[:m]
        r.shuffle(refs)
        steps.append(refs)
        prev = refs
    return steps


@pytest.mark.parametrize("seed,G_,universe", [(0, 4, 9), (1, 8, 30), (2, 16, 40), (3, 5, 6), (4, 32, 200)])
def test_lru_matches_textbook_stack_distance(seed, G_, universe):
    steps = _random_trace(seed, G_, universe, 40)
    st = O.KvSwapLayerState(universe + G_ + 1, G_, window=128)
    st.host_ready[:] = 1
    want, resident = _lru_textbook(steps, G_)
    for refs, exp in zip(steps, want):
        r = st.swap_in_selected(refs)
        got = []
        miss_slots = dict(r.misses)
        for c, p in zip(refs, r.phys):
            got.append((c not in miss_slots, p - 128))
        assert got == exp
        assert r.hits + len(r.misses) == len(refs)
    assert {c: s for c, s in st.slot_by_logical.items()} == resident
    assert sorted(s for s in st.gpu_slot_logical if s >= 0) == sorted(resident)


def test_lru_evicts_a_chunk_selected_later_in_the_same_step():
    """The Swap-in flow walks the list in order: a miss may pop a slot whose chunk
    is selected further down the same list (then that chunk misses too)."""
    st = O.KvSwapLayerState(10, 2)
    st.host_ready[:] = 1
    r1 = st.swap_in_selected([1, 2])          # 1 -> slot 0, 2 -> slot 1; 1 is least recent
    assert r1.phys == [128, 129] and r1.hits == 0
    r2 = st.swap_in_selected([3, 1])          # 3 pops slot 0 (chunk 1); then 1 pops slot 1
    assert r2.misses == [(3, 0), (1, 1)] and r2.hits == 0
    assert r2.phys == [128, 129]


def test_lru_invariants_constant_selection_all_hits():
    st = O.KvSwapLayerState(5000, 1024)
    st.host_ready[:] = 1
    sel = list(np.random.default_rng(0).permutation(5000)[:512])
    r = st.swap_in_selected(sel)
    assert r.hits == 0 and len(r.misses) == 512
    assert [s for _, s in r.misses] == list(range(512))     # free slots fill in order
    for _ in range(3):
        r = st.swap_in_selected(sel)
        assert r.hits == 512 and not r.misses
    assert len(set(r.phys)) == 512


def test_lru_not_stored_error():
    st = O.KvSwapLayerState(10, 4)
    st.store(3)
    st.swap_in_selected([3])
    with pytest.raises(O.NotStoredError):
        st.swap_in_selected([3, 7])


def test_store_keeps_a_staged_chunk_and_enables_a_new_one():
    """Store flow (KV_SWAP 实现细节, Store): storing sets host_ready; a chunk that
    is already in a staging slot stays there (the store evicts nothing)."""
    st = O.KvSwapLayerState(10, 2)
    for c in (1, 2):
        st.store(c)
    r1 = st.swap_in_selected([1, 2])
    before = (dict(st.slot_by_logical), list(st.slot_lru), list(st.gpu_slot_logical))
    st.store(1)                                   # re-store a staged chunk
    st.store(5)                                   # a new chunk
    assert (dict(st.slot_by_logical), list(st.slot_lru), list(st.gpu_slot_logical)) == before
    r2 = st.swap_in_selected([1])                 # still staged: a hit in its old slot
    assert r2.hits == 1 and r2.phys == [r1.phys[0]]
    r3 = st.swap_in_selected([5])                 # now allowed; takes the least recent slot (chunk 2's)
    assert r3.misses == [(5, 1)]


def test_decode_oracle_store_and_periodic_selection():
    """DecodeOracle.store marks chunks of one (layer, seq) only; a step with
    rescore=False reuses the previous selection, so a repeated selection is all
    hits (the indexer fires once per lookahead window)."""
    w = C.TINY
    ora = O.DecodeOracle(context_len=w.context_len, layer_ratios=(4, 4), gpu_chunks=w.gpu_chunks,
                         index_topk=w.index_topk, batch=2, scale=w.scale, bias=[0.0] * 3,
                         ensemble_mode=w.ensemble, select_mode=w.select_mode, tau=w.tau, clamp=w.clamp)
    ora.store(1, 0, 10, 5)
    assert ora.states[1][0].host_ready[10:15].all() and not ora.states[1][0].host_ready[15]
    assert not ora.states[0][0].host_ready.any() and not ora.states[1][1].host_ready.any()
    ora.mark_all_stored()
    keys = [G.keys(w, b) for b in range(2)]
    r0 = ora.step(lambda b: keys[b], lambda b: G.fm_queries(w, 0, b))
    other = lambda b: G.fm_queries(w, 8, b)       # would change the selection if it were scored
    r1 = ora.step(lambda b: keys[b], other, rescore=False)
    for b in range(2):
        assert np.array_equal(r1.sel[b], r0.sel[b])
        assert r1.swap[0][b].hits == len(r1.lists[0][b]) and not r1.swap[0][b].misses
    r2 = ora.step(lambda b: keys[b], other)       # rescored: a new needle set
    assert not all(np.array_equal(r2.sel[b], r0.sel[b]) for b in range(2))


# --------------------------------------------------------------------------- adaptive capacity
def _stamp_lru_resizable(steps, caps, G_):
    """LRU by last-use keys over a slot range that can shrink or grow, written
    independently of the list form: a slot's key is (step, position) of its
    last use; slots free from the start have (-1, slot); slots added when the
    range grows at step t have (-(t + 2), slot), below every other key. A miss
    takes the slot in range with the smallest key; a dropped slot forgets its
    chunk."""
    key = {s: (-1, s) for s in range(G_)}
    chunk = {}
    g, out = G_, []
    for t, (refs, gt) in enumerate(zip(steps, caps)):
        if gt > g:
            for s in range(g, gt):
                key[s] = (-(t + 2), s)
        for s in range(gt, g):
            chunk.pop(s, None)
        g = gt
        res = []
        for p, c in enumerate(refs):
            where = [s for s in range(g) if chunk.get(s) == c]
            if where:
                s, hit = where[0], True
            else:
                s, hit = min(range(g), key=lambda x: key[x]), False
                chunk[s] = c
            key[s] = (t, p)
            res.append((hit, s))
        out.append(res)
    return out


@pytest.mark.parametrize("seed,G_,universe", [(0, 8, 20), (1, 16, 40), (2, 6, 9), (3, 32, 100)])
def test_adaptive_resize_matches_stamp_model(seed, G_, universe):
    r = random.Random(100 + seed)
    caps, g = [], G_
    for _ in range(60):
        if r.random() < 0.3:
            g = r.randint(1, G_)
        caps.append(g)
    steps = []
    prev = []
    for g in caps:
        m = r.randint(0, g)
        keep = [c for c in prev if r.random() < 0.6]
        pool = [c for c in range(universe) if c not in keep]
        refs = (keep + r.sample(pool, max(0, min(m - len(keep), len(pool)))))[:m]
        r.shuffle(refs)
        steps.append(refs)
        prev = refs
    want = _stamp_lru_resizable(steps, caps, G_)
    st = O.KvSwapLayerState(universe + G_ + 1, G_)
    st.host_ready[:] = 1
    for refs, g, exp in zip(steps, caps, want):
        st.set_capacity(g)
        res = st.swap_in_selected(refs)
        miss = dict(res.misses)
        assert [(c not in miss, p - 128) for c, p in zip(refs, res.phys)] == exp
        assert all(s < g for s in st.slot_by_logical.values())
        assert sorted(st.slot_lru) == list(range(g))


def test_adaptive_policy_hand_worked():
    """Capacity 8 slots, policy: start at 4, decide every 2 steps, grow below a
    50 % hit rate, shrink above 90 %, by 2 slots, within [2, 8]."""
    st = O.KvSwapLayerState(100, 8)
    st.host_ready[:] = 1
    st.install_policy(O.AdaptivePolicy(g_min=2, g_max=8, g_init=4, epoch=2, lo_permille=500,
                                       hi_permille=900, delta=2))
    trace = [
        # refs, capacity used, phys, hits
        ([0, 1, 2], 4, [128, 129, 130], 0),
        ([0, 1, 2], 4, [128, 129, 130], 3),   # window 3/6 = 50 %: neither below 50 % nor above 90 %
        ([0, 1, 2], 4, [128, 129, 130], 3),
        ([0, 1, 2], 4, [128, 129, 130], 3),   # window 6/6: shrink to 2
        ([0, 1], 2, [128, 129], 2),           # slots 2, 3 dropped with chunk 2
        ([5, 6], 2, [128, 129], 0),           # window 2/4 = 50 %: stays
        ([7, 8], 2, [128, 129], 0),
        ([9], 2, [128], 0),                   # window 0/3: grow to 4
        ([10], 4, [130], 0),                  # the new empty slots go first, lowest first
        ([8, 11, 12], 4, [129, 131, 128], 1), # 12 takes the least recent slot (chunk 9's); 1/4: grow to 6
        ([], 6, [], 0),
    ]
    for refs, g, phys, hits in trace:
        res = st.swap_in_selected(refs)
        assert (st.capacity, res.phys, res.hits) == (g, phys, hits), refs
    assert st.next_capacity == 6 and st.capacity == 6


def test_adaptive_fixed_range_is_plain_lru():
    """A policy pinned to the full range (or one that never fires) leaves the
    plain list LRU unchanged, step for step."""
    steps = _random_trace(9, 16, 50, 40)
    for pol in (O.AdaptivePolicy(16, 16, 16, 1, 0, 1000, 4), O.AdaptivePolicy(4, 16, 16, 3, 0, 1000, 4)):
        a = O.KvSwapLayerState(70, 16)
        b = O.KvSwapLayerState(70, 16)
        a.host_ready[:] = 1
        b.host_ready[:] = 1
        b.install_policy(pol)
        for refs in steps:
            ra, rb = a.swap_in_selected(refs), b.swap_in_selected(refs)
            assert (ra.phys, ra.misses, ra.hits) == (rb.phys, rb.misses, rb.hits)
        assert b.capacity == 16


def test_decode_oracle_keeps_list_prefix_under_small_capacity():
    """A step whose list is longer than the slots in use keeps the first chunks
    of the list, as many as the slots (and the attention uses those)."""
    w = C.TINY
    ora = O.DecodeOracle(context_len=w.context_len, layer_ratios=(4,), gpu_chunks=w.gpu_chunks,
                         index_topk=w.index_topk, batch=1, scale=w.scale, bias=[0.0] * 3,
                         ensemble_mode=w.ensemble, select_mode=w.select_mode, tau=w.tau, clamp=w.clamp)
    ora.mark_all_stored()
    ora.install_policy(O.AdaptivePolicy(100, w.gpu_chunks, 100, 1, 0, 1000, 1))
    keys = G.keys(w, 0)
    r = ora.step(lambda b: keys, lambda b: G.fm_queries(w, 0, b))
    assert len(r.lists[0][0]) == 100 and r.lists[0][0] == list(r.sel[0][:100])
    assert sorted(p - 128 for p in r.swap[0][0].phys) == list(range(100))


def test_gpu_chunks_below_topk_keeps_the_list_head_hand_trace():
    """GPU_CHUNKS < index_topk (rejected by default, [P1] 故障排查 error 2;
    allowed by the reduction flag): a swapped layer stages only the first
    GPU_CHUNKS chunks of its list. Hand-worked trace: 10 chunks whose key c is
    (c+1)*e_0, every query head e_0 (step 0) or -e_0 (step 1), so the top-5 is
    [9, 8, 7, 6, 5] then [0, 1, 2, 3, 4]; G = 3; layers of ratio 4 (cap 10) and
    ratio 8 (cap 5, list c -> c // 2), both swapped."""
    keys = np.zeros((10, 128), np.float32)
    keys[:, 0] = np.arange(1, 11)
    qa = np.zeros((3, 8, 128), np.float32)
    qa[:, :, 0] = 1.0
    kb, qpos, qneg = _bits(keys), _bits(qa), _bits(-qa)
    ora = O.DecodeOracle(context_len=40, layer_ratios=(4, 8), gpu_chunks=3, index_topk=5, batch=1,
                         scale=1.0, bias=[0.0] * 3, ensemble_mode=O.ENSEMBLE_MAX,
                         select_mode=O.SELECT_TOPK, tau=0.5, clamp=5)
    ora.mark_all_stored()
    win = np.zeros((128, 512))
    pool = np.arange(10 * 512, dtype=np.float64).reshape(10, 512) / 5000.0
    qa_bits = _bits(np.ones((16, 512), np.float32))
    rows_of = lambda l, b, idx: pool[np.asarray(idx, dtype=np.int64)] if len(idx) else np.zeros((0, 512))
    r0 = ora.step(lambda b: kb, lambda b: qpos, lambda l, b: qa_bits, lambda l, b: win, rows_of)
    assert list(r0.sel[0]) == [9, 8, 7, 6, 5]
    assert r0.lists[0][0] == [9, 8, 7]                      # ratio 4: the first three of five
    assert r0.lists[1][0] == [4, 3, 2]                      # ratio 8: [4,4,3,3,2] deduplicated, fits
    assert r0.swap[0][0].phys == [128, 129, 130] and r0.swap[0][0].misses == [(9, 0), (8, 1), (7, 2)]
    assert r0.swap[1][0].misses == [(4, 0), (3, 1), (2, 2)]
    # the attention reads the window and exactly the staged chunks
    want = O.attend(qa_bits, np.concatenate([win, pool[[9, 8, 7]]]))
    assert np.array_equal(r0.out[(0, 0)], want)
    r1 = ora.step(lambda b: kb, lambda b: qneg, lambda l, b: qa_bits, lambda l, b: win, rows_of)
    assert list(r1.sel[0]) == [0, 1, 2, 3, 4]
    assert r1.lists[0][0] == [0, 1, 2]
    assert r1.swap[0][0].misses == [(0, 0), (1, 1), (2, 2)] and r1.swap[0][0].hits == 0
    # ratio 8: [0,0,1,1,2] -> [0, 1, 2]; chunk 2 is still in slot 2 (a hit),
    # 0 and 1 take the least recent slots 0 (chunk 4) and 1 (chunk 3)
    assert r1.lists[1][0] == [0, 1, 2]
    assert r1.swap[1][0].misses == [(0, 0), (1, 1)] and r1.swap[1][0].hits == 1
    assert r1.swap[1][0].phys == [128, 129, 130]


def _small_oracle(w):
    ora = O.DecodeOracle(context_len=w.context_len, layer_ratios=w.layer_ratios, gpu_chunks=w.gpu_chunks,
                         index_topk=w.index_topk, batch=1, scale=w.scale, bias=[0.0] * 3,
                         ensemble_mode=w.ensemble, select_mode=w.select_mode, tau=w.tau, clamp=w.clamp)
    ora.mark_all_stored()
    return ora


def test_lookahead_schedule_is_the_plain_step_one_step_late():
    """Triggered at every step, the lookahead schedule attends at step t over
    the chunks that the indexer picked from step t-1's queries: the plain step
    fed step t-1's indexer queries and step t's attention queries gives the
    same output. Step 0 attends over the window rows alone (checked against
    torch's attention)."""
    w = C.TINY.with_(gpu_chunks=1024, lookahead=1, layer_ratios=(4, 128))
    keys = G.keys(w, 0)
    pools = {l: G.pool(w, l, 0) for l in range(2)}
    rows_of = lambda l, b, idx: pools[l][np.asarray(idx, dtype=np.int64)]
    win = lambda l, b: G.window(w, l, b)
    la, plain = _small_oracle(w), _small_oracle(w)
    for t in range(4):
        q_t = lambda l, b, t=t: G.attn_q(w, t, l, b)
        r = la.lookahead_step(lambda b: keys, lambda b, t=t: G.fm_queries(w, t, b), q_t, win, rows_of,
                              attend_pairs=[(0, 0), (1, 0)], trigger=True)
        if t == 0:
            for l in range(2):
                q = torch.from_numpy(O.bf16_to_f64(G.attn_q(w, 0, l, 0)))[None, :, None, :].transpose(1, 2)
                e = torch.from_numpy(win(l, 0).astype(np.float64))[None, None]
                ref = torch.nn.functional.scaled_dot_product_attention(q.transpose(1, 2), e, e)[0]
                assert np.allclose(r.out[(l, 0)], ref.numpy().reshape(r.out[(l, 0)].shape), rtol=1e-12, atol=1e-12)
            continue
        p = plain.step(lambda b: keys, lambda b, t=t: G.fm_queries(w, t - 1, b), q_t, win, rows_of,
                       attend_pairs=[(0, 0), (1, 0)])
        for l in range(2):
            assert r.lists[l][0] == p.lists[l][0]
            assert np.allclose(r.out[(l, 0)], p.out[(l, 0)], rtol=1e-13, atol=1e-13)


def test_lookahead_schedule_swaps_like_periodic_selection():
    """Between triggers the lookahead schedule resolves nothing; the periodic
    schedule resolves the same list again (all hits). Touching a list that was
    just resolved leaves the LRU order as it was, so both schedules stage the
    same slots at every trigger and end in the same state."""
    w = C.TINY.with_(gpu_chunks=1024, lookahead=3, layer_ratios=(4, 128))
    keys = G.keys(w, 0)
    la, per = _small_oracle(w), _small_oracle(w)
    for t in range(9):
        fq = lambda b, t=t: G.fm_queries(w, t, b)
        trig = t % w.lookahead == 0
        r = la.lookahead_step(lambda b: keys, fq, trigger=trig)
        p = per.step(lambda b: keys, fq, rescore=trig)
        if trig:
            for l in range(2):
                assert r.swap[l][0].phys == p.swap[l][0].phys and r.swap[l][0].misses == p.swap[l][0].misses
        else:
            assert all(p.swap[l][0].hits == len(p.lists[l][0]) for l in range(2) if per.states[l][0].swap_enabled)
    for l in range(2):
        a, b = la.states[l][0], per.states[l][0]
        assert (a.slot_by_logical, list(a.slot_lru), a.gpu_slot_logical) == \
               (b.slot_by_logical, list(b.slot_lru), b.gpu_slot_logical)


def test_swap_disabled_layer_is_identity_mapped():
    st = O.KvSwapLayerState(16, 16)
    st.host_ready[:] = 1
    assert not st.swap_enabled
    r = st.swap_in_selected([9, 0, 15])
    assert r.phys == [137, 128, 143] and r.hits == 0 and not r.misses


# --------------------------------------------------------------------------- attention
def test_attention_matches_torch_sdpa_float64():
    rng = np.random.default_rng(1)
    q = G.f32_to_bf16_bits(rng.standard_normal((16, 512), dtype=np.float32))
    rows = rng.standard_normal((200, 512))
    got = O.attend(q, rows)
    qt = torch.from_numpy(O.bf16_to_f64(q))[None, None]
    et = torch.from_numpy(rows)[None, None]
    want = torch.nn.functional.scaled_dot_product_attention(qt, et, et)[0, 0].numpy()
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)


def test_attention_special_cases():
    rng = np.random.default_rng(2)
    rows = rng.standard_normal((1, 512))
    q = G.f32_to_bf16_bits(rng.standard_normal((4, 512), dtype=np.float32))
    np.testing.assert_allclose(O.attend(q, rows), np.repeat(rows, 4, axis=0), rtol=0, atol=1e-15)
    rows = rng.standard_normal((37, 512))
    zero_q = np.zeros((3, 512), np.uint16)
    np.testing.assert_allclose(O.attend(zero_q, rows), np.repeat(rows.mean(0, keepdims=True), 3, 0),
                               rtol=1e-13, atol=1e-14)
    # two rows, logits differing by exactly ln 3 -> weights 3/4, 1/4
    e = np.zeros((2, 512))
    e[0, 0] = math.sqrt(512) * math.log(3.0)
    q1 = np.zeros((1, 512), np.float32)
    q1[0, 0] = 1.0
    o = O.attend(G.f32_to_bf16_bits(q1), e)
    assert o[0, 0] == pytest.approx(0.75 * e[0, 0], rel=1e-13)


# --------------------------------------------------------------------------- whole step
def _small_workload(**kw):
    base = dict(name="pin", code=99, context_len=256, layer_ratios=(4, 128), gpu_chunks=64,
                index_topk=64, ensemble=C.ENSEMBLE_MAX, select_mode=C.SELECT_TOPK, tau=0.5,
                bias=0.0, n_heads=16, batch=2, steps=6, lookahead=2, n_needles=4)
    base.update(kw)
    return C.Workload(**base)


def _run(w, attend=True):
    ora = O.DecodeOracle(context_len=w.context_len, layer_ratios=w.layer_ratios,
                         gpu_chunks=w.gpu_chunks, index_topk=w.index_topk, batch=w.batch,
                         scale=w.scale, bias=[w.bias] * 3, ensemble_mode=w.ensemble,
                         select_mode=w.select_mode, tau=w.tau, clamp=w.clamp)
    ora.mark_all_stored()
    keys = [G.keys(w, b) for b in range(w.batch)]
    pools = {(l, b): G.pool(w, l, b) for l in range(w.n_layers) for b in range(w.batch)}
    res = []
    for t in range(w.steps):
        res.append(ora.step(lambda b: keys[b], lambda b: G.fm_queries(w, t, b),
                            (lambda l, b: G.attn_q(w, t, l, b)) if attend else None,
                            lambda l, b: G.window(w, l, b),
                            lambda l, b, idx: pools[(l, b)][np.asarray(idx, dtype=np.int64)]))
    return ora, res, keys, pools


def test_topk_covering_all_chunks_is_dense_attention():
    w = _small_workload(index_topk=64, gpu_chunks=64)      # n = 64 chunks, all selected
    _, res, _, pools = _run(w)
    for t, r in enumerate(res):
        for b in range(w.batch):
            assert sorted(r.sel[b].tolist()) == list(range(64))
            rows = np.concatenate([G.window(w, 0, b), pools[(0, b)]]).astype(np.float64)
            qt = torch.from_numpy(O.bf16_to_f64(G.attn_q(w, t, 0, b)))[None, None]
            et = torch.from_numpy(rows)[None, None]
            want = torch.nn.functional.scaled_dot_product_attention(qt, et, et)[0, 0].numpy()
            np.testing.assert_allclose(r.out[(0, b)], want, rtol=1e-12, atol=1e-13)


def test_residency_changes_slots_never_outputs():
    """kestrel-llm-cuda 06, section 3.4: residency changes occupancy, never outputs."""
    swapped = _small_workload(index_topk=16, gpu_chunks=24)    # cap 64 > 24 -> swap
    resident = swapped.with_(gpu_chunks=64)                     # cap 64 <= 64 -> resident
    _, rs, _, _ = _run(swapped)
    _, rr, _, _ = _run(resident)
    saw_miss_after_start = False
    for t, (a, b) in enumerate(zip(rs, rr)):
        for key in a.out:
            assert np.array_equal(a.out[key], b.out[key])
        for bb in range(swapped.batch):
            assert a.swap[0][bb].phys != b.swap[0][bb].phys or not a.sel[bb].size
            if t > 0 and a.swap[0][bb].misses:
                saw_miss_after_start = True
    assert saw_miss_after_start


def test_needles_are_selected_by_every_ensemble():
    """The planted needles score far above the noise chunks, so top-k and the
    threshold selector (bias -7, tau 0.5) both recall them."""
    for w in (_small_workload(context_len=8192, index_topk=32, gpu_chunks=64, n_needles=8,
                              layer_ratios=(4,), steps=2, batch=1),
              _small_workload(context_len=8192, ensemble=C.ENSEMBLE_MEAN, select_mode=C.SELECT_THRESH,
                              bias=-7.0, gpu_chunks=512, n_needles=32, layer_ratios=(4,), steps=2,
                              batch=1)):
        _, res, _, _ = _run(w, attend=False)
        for t, r in enumerate(res):
            nd = set(G.step_needles(w, t, 0).tolist())
            assert nd <= set(r.sel[0].tolist())
