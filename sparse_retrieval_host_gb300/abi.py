"""ctypes binding of libsrh.so (include/srh.h): argument marshalling only.

Every function here has the name of the C entry point it calls. Tensors are
torch tensors on the CUDA device (or plain integers holding device pointers);
their pointers, sizes and the current stream are passed through unchanged and
all the work runs in the library's kernels. There is no CPU fallback: if the
library is missing, importing the package's runtime raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libsrh.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "srh.h")

SRH_OK = 0
SRH_ERR_INVALID = -1
SRH_ERR_PINNED_CAP = -2
SRH_ERR_NOT_STORED = -3
SRH_ERR_CUDA = -4
SRH_ERR_TIMEOUT = -5
SRH_ERR_NOMEM = -6
SRH_ERR_BOUNDS = -7
SRH_ERR_RANGE = -8
SRH_ENSEMBLE_MAX = 0
SRH_ENSEMBLE_MEAN = 1
SRH_SELECT_TOPK = 0
SRH_SELECT_THRESH = 1
SRH_FLAG_TEST_FAIL_HOST_ALLOC = 1
KV_DIM = 512
WINDOW = 128
SRH_NOALLOC_MAX_BATCH = 64
SRH_NOALLOC_MAX_N = 1 << 30


class SrhConfig(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int),
        ("n_layers", ctypes.c_int),
        ("kv_dim", ctypes.c_int),
        ("window", ctypes.c_int),
        ("gpu_chunks", ctypes.c_int),
        ("index_topk", ctypes.c_int),
        ("src_ratio", ctypes.c_int),
        ("layer_ratio", ctypes.POINTER(ctypes.c_int)),
        ("context_len", ctypes.c_longlong),
        ("pinned_cap_bytes", ctypes.c_size_t),
        ("allow_topk_reduction", ctypes.c_int),
        ("max_select", ctypes.c_int),
        ("flags", ctypes.c_uint),
    ]


class SrhStats(ctypes.Structure):
    _fields_ = [
        ("hits", ctypes.c_ulonglong),
        ("misses", ctypes.c_ulonglong),
        ("h2d_bytes", ctypes.c_ulonglong),
        ("d2h_bytes", ctypes.c_ulonglong),
        ("resident_fill_bytes", ctypes.c_ulonglong),
        ("stage_calls", ctypes.c_ulonglong),
        ("selected", ctypes.c_ulonglong),
        ("swapped_layers", ctypes.c_int),
        ("n_layers", ctypes.c_int),
    ]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


class SrhAdaptive(ctypes.Structure):
    """srh_adaptive: the hit-rate policy of the staging capacity."""
    _fields_ = [(name, ctypes.c_int) for name in
                ("enabled", "g_min", "g_max", "g_init", "epoch", "lo_permille", "hi_permille", "delta")]


class SrhError(RuntimeError):
    def __init__(self, code: int, where: str, detail: str = ""):
        self.code = code
        super().__init__(f"{where}: {error_string(code)} ({code}){': ' + detail if detail else ''}")


_vp = ctypes.c_void_p
_i = ctypes.c_int
_ll = ctypes.c_longlong
_f = ctypes.c_float

# (name, restype, argtypes) -- the order of include/srh.h
SIGNATURES = [
    ("srh_create", _i, [ctypes.POINTER(SrhConfig), ctypes.POINTER(_vp)]),
    ("srh_destroy", None, [_vp]),
    ("srh_pinned_required_bytes", _i, [ctypes.POINTER(SrhConfig), ctypes.POINTER(ctypes.c_ulonglong)]),
    ("srh_attend_plan_info", _i, [ctypes.POINTER(SrhConfig), _i, _i, ctypes.POINTER(_ll)]),
    ("srh_pool_host_ptr", ctypes.POINTER(_f), [_vp, _i, _i]),
    ("srh_mark_stored", _i, [_vp, _i, _i, _ll, _ll]),
    ("kvswap_store", _i, [_vp, _i, _i, _ll, _i, _vp, _vp]),
    ("srh_layer_info", _i, [_vp, _i, ctypes.POINTER(_ll), ctypes.POINTER(_i)]),
    ("srh_max_select", _i, [_vp]),
    ("fm_score", _i, [_vp, _vp, _i, _vp, _f, ctypes.POINTER(_f), _i, _vp, _vp]),
    ("fm_score_multi", _i, [_vp, _vp, _i, _vp, _f, ctypes.POINTER(_f), _i, _vp, _vp]),
    ("fm_quantize_keys", _i, [_vp, _vp, _i, _vp, _vp, _vp]),
    ("fm_score_fp8", _i, [_vp, _vp, _vp, _i, _vp, _f, ctypes.POINTER(_f), _i, _vp, _vp]),
    ("fm_select", _i, [_vp, _vp, _i, _i, _i, _f, _i, _vp, _vp, _vp]),
    ("fm_select_noalloc", _i, [_vp, _i, _i, _i, _i, _f, _i, _i, _vp, _vp, _vp, ctypes.c_char_p, ctypes.c_size_t]),
    ("kvswap_stage", _i, [_vp, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    ("lsa_attend", _i, [_vp, _i, _vp, _i, _vp, _vp, _vp, _vp, _vp, _vp]),
    ("srh_set_chained", _i, [_vp, _i]),
    ("srh_set_adaptive", _i, [_vp, ctypes.POINTER(SrhAdaptive)]),
    ("srh_get_active_slots", _i, [_vp, ctypes.POINTER(ctypes.c_int)]),
    ("srh_get_stats", _i, [_vp, ctypes.POINTER(SrhStats)]),
    ("srh_reset_stats", _i, [_vp]),
    ("srh_check_error", _i, [_vp]),
    ("srh_selftest_wait_timeout", _i, [_vp, _i, _vp]),
    ("srh_hostloop_create", _i, [_vp, _vp, _i, _vp, _vp, _vp, _vp, _vp, _i, _f, ctypes.POINTER(_f), _i, _i, _i, _f, _i,
                                 ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                                 ctypes.POINTER(_vp), _vp, ctypes.POINTER(_vp)]),
    ("srh_hostloop_step", _i, [_vp, _ll, _vp, _vp, _vp, _vp, _vp]),
    ("srh_hostloop_wait", _i, [_vp, _ll]),
    ("srh_hostloop_sync", _i, [_vp]),
    ("srh_hostloop_destroy", None, [_vp]),
    ("srh_error_string", ctypes.c_char_p, [_i]),
    ("srh_last_error", ctypes.c_char_p, [_vp]),
]

_lib: Optional[ctypes.CDLL] = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libsrh.so (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m sparse_retrieval_host_gb300.build` "
                           "(there is no CPU fallback)")
    lib = ctypes.CDLL(path)
    for name, res, args in SIGNATURES:
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def error_string(code: int) -> str:
    try:
        return load().srh_error_string(code).decode()
    except Exception:  # pragma: no cover - library not built
        return str(code)


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, where: str, ctx=None) -> int:
    if rc != SRH_OK:
        detail = load().srh_last_error(ctx).decode(errors="replace")
        raise SrhError(rc, where, detail)
    return rc


def make_config(*, batch: int, layer_ratios: Sequence[int], gpu_chunks: int, index_topk: int,
                context_len: int, src_ratio: int = 4, pinned_cap_bytes: int = 0,
                allow_topk_reduction: bool = False, max_select: int = 0, flags: int = 0):
    arr = (ctypes.c_int * len(layer_ratios))(*layer_ratios)
    cfg = SrhConfig(batch, len(layer_ratios), KV_DIM, WINDOW, gpu_chunks, index_topk, src_ratio,
                    ctypes.cast(arr, ctypes.POINTER(ctypes.c_int)), context_len, pinned_cap_bytes,
                    1 if allow_topk_reduction else 0, max_select, flags)
    cfg._keep = arr  # keep the ratio array alive with the struct
    return cfg


def srh_create(cfg: SrhConfig) -> int:
    out = _vp()
    _check(load().srh_create(ctypes.byref(cfg), ctypes.byref(out)), "srh_create")
    return out.value


def srh_destroy(ctx: int) -> None:
    load().srh_destroy(ctx)


def srh_pinned_required_bytes(cfg: SrhConfig) -> int:
    out = ctypes.c_ulonglong()
    _check(load().srh_pinned_required_bytes(ctypes.byref(cfg), ctypes.byref(out)), "srh_pinned_required_bytes")
    return out.value


def srh_attend_plan_info(cfg: SrhConfig, sm_count: int, layer: int = -1) -> dict:
    """srh_attend_plan_info: lsa_attend's work split for this configuration (host only)."""
    info = (_ll * 6)()
    _check(load().srh_attend_plan_info(ctypes.byref(cfg), sm_count, layer, info), "srh_attend_plan_info")
    return {"ctas": info[0], "segments": info[1], "split_pairs": info[2], "max_cta_kib": info[3],
            "one_wave": bool(info[4]), "valid": bool(info[5])}


def srh_pool_host_ptr(ctx: int, layer: int, seq: int) -> int:
    p = load().srh_pool_host_ptr(ctx, layer, seq)
    addr = ctypes.cast(p, ctypes.c_void_p).value
    if not addr:
        raise SrhError(SRH_ERR_INVALID, "srh_pool_host_ptr")
    return addr


def srh_mark_stored(ctx: int, layer: int, seq: int, c0: int, n: int) -> None:
    _check(load().srh_mark_stored(ctx, layer, seq, c0, n), "srh_mark_stored", ctx)


def kvswap_store(ctx, layer, seq, c0, n, rows, stream=None) -> None:
    _check(load().kvswap_store(ctx, layer, seq, c0, n, _ptr(rows), _stream(stream)), "kvswap_store", ctx)


def srh_layer_info(ctx: int, layer: int):
    cap, sw = _ll(), _i()
    _check(load().srh_layer_info(ctx, layer, ctypes.byref(cap), ctypes.byref(sw)), "srh_layer_info", ctx)
    return cap.value, bool(sw.value)


def srh_max_select(ctx: int) -> int:
    return load().srh_max_select(ctx)


def fm_score(ctx, keys, n, q, scale, bias3, ensemble, scores, stream=None) -> None:
    b = (ctypes.c_float * 3)(*[float(x) for x in bias3])
    _check(load().fm_score(ctx, _ptr(keys), n, _ptr(q), float(scale), b, ensemble, _ptr(scores),
                           _stream(stream)), "fm_score", ctx)


def fm_score_multi(ctx, keys3, n, q, scale, bias3, ensemble, scores, stream=None) -> None:
    b = (ctypes.c_float * 3)(*[float(x) for x in bias3])
    _check(load().fm_score_multi(ctx, _ptr(keys3), n, _ptr(q), float(scale), b, ensemble, _ptr(scores),
                                 _stream(stream)), "fm_score_multi", ctx)


def fm_quantize_keys(ctx, keys, n, codes, kscale, stream=None) -> None:
    _check(load().fm_quantize_keys(ctx, _ptr(keys), n, _ptr(codes), _ptr(kscale), _stream(stream)),
           "fm_quantize_keys", ctx)


def fm_score_fp8(ctx, codes, kscale, n, q, scale, bias3, ensemble, scores, stream=None) -> None:
    b = (ctypes.c_float * 3)(*[float(x) for x in bias3])
    _check(load().fm_score_fp8(ctx, _ptr(codes), _ptr(kscale), n, _ptr(q), float(scale), b, ensemble,
                               _ptr(scores), _stream(stream)), "fm_score_fp8", ctx)


def fm_select(ctx, scores, n, mode, k, tau, clamp, sel, count, stream=None) -> None:
    _check(load().fm_select(ctx, _ptr(scores), n, mode, k, float(tau), clamp, _ptr(sel), _ptr(count),
                            _stream(stream)), "fm_select", ctx)


def fm_select_noalloc(scores, batch, n, mode, k, tau, clamp, max_select, sel, count, stream=None) -> None:
    """fm_select with no context and no device allocation (scratch is a fixed
    array inside the library; see include/srh.h for the limits and sharing)."""
    buf = ctypes.create_string_buffer(256)
    rc = load().fm_select_noalloc(_ptr(scores), batch, n, mode, k, float(tau), clamp, max_select, _ptr(sel),
                                  _ptr(count), _stream(stream), buf, len(buf))
    if rc != SRH_OK:
        raise SrhError(rc, "fm_select_noalloc", buf.value.decode(errors="replace"))


def kvswap_stage(ctx, layer, sel, count, staging, phys, count_l, main=None, side=None) -> None:
    m = _stream(main)
    s = m if side is None else _stream(side)
    _check(load().kvswap_stage(ctx, layer, _ptr(sel), _ptr(count), _ptr(staging), _ptr(phys), _ptr(count_l),
                               m, s), "kvswap_stage", ctx)


def lsa_attend(ctx, layer, q, n_heads, window, staging, phys, count_l, out, stream=None) -> None:
    _check(load().lsa_attend(ctx, layer, _ptr(q), n_heads, _ptr(window), _ptr(staging), _ptr(phys),
                             _ptr(count_l), _ptr(out), _stream(stream)), "lsa_attend", ctx)


def srh_set_chained(ctx, on: bool) -> None:
    _check(load().srh_set_chained(ctx, 1 if on else 0), "srh_set_chained", ctx)


def srh_set_adaptive(ctx, policy=None) -> None:
    """policy: None (remove) or a mapping with the srh_adaptive fields except
    ``enabled``."""
    if policy is None:
        rc = load().srh_set_adaptive(ctx, None)
    else:
        p = SrhAdaptive(enabled=1, **dict(policy))
        rc = load().srh_set_adaptive(ctx, ctypes.byref(p))
    _check(rc, "srh_set_adaptive", ctx)


def srh_get_active_slots(ctx, n_layers: int, batch: int):
    """Slots in use per (layer, sequence), as a list of lists."""
    buf = (ctypes.c_int * (n_layers * batch))()
    _check(load().srh_get_active_slots(ctx, buf), "srh_get_active_slots", ctx)
    return [[buf[l * batch + b] for b in range(batch)] for l in range(n_layers)]


def srh_get_stats(ctx) -> dict:
    st = SrhStats()
    _check(load().srh_get_stats(ctx, ctypes.byref(st)), "srh_get_stats", ctx)
    return st.as_dict()


def srh_reset_stats(ctx) -> None:
    _check(load().srh_reset_stats(ctx), "srh_reset_stats", ctx)


def srh_hostloop_create(ctx, keys, n, scores, staging, phys, count_l, window, n_heads, scale, bias3, ensemble,
                        mode, k, tau, clamp, fm_q2, q2, out2, sel2, count2, stream=None) -> int:
    """The native host loop over two sets of step buffers (each argument ending
    in 2 is a pair of tensors). Returns its handle."""
    pair = lambda xs: (_vp * 2)(*[_ptr(x) for x in xs])
    b3 = (_f * 3)(*[float(v) for v in bias3])
    out = _vp()
    rc = load().srh_hostloop_create(ctx, _ptr(keys), n, _ptr(scores), _ptr(staging), _ptr(phys), _ptr(count_l),
                                    _ptr(window), n_heads, float(scale), b3, ensemble, mode, k, float(tau), clamp,
                                    pair(fm_q2), pair(q2), pair(out2), pair(sel2), pair(count2), _stream(stream),
                                    ctypes.byref(out))
    _check(rc, "srh_hostloop_create", ctx)
    return out.value


def srh_hostloop_step(ctx, lp, i, h_fm_q, h_q, h_out, h_sel, h_count) -> None:
    _check(load().srh_hostloop_step(lp, i, _ptr(h_fm_q), _ptr(h_q), _ptr(h_out), _ptr(h_sel), _ptr(h_count)),
           "srh_hostloop_step", ctx)


def srh_hostloop_wait(ctx, lp, i) -> None:
    _check(load().srh_hostloop_wait(lp, i), "srh_hostloop_wait", ctx)


def srh_hostloop_sync(ctx, lp) -> None:
    _check(load().srh_hostloop_sync(lp), "srh_hostloop_sync", ctx)


def srh_hostloop_destroy(lp) -> None:
    load().srh_hostloop_destroy(lp)


def srh_check_error(ctx) -> int:
    """Returns the code (does not raise): SRH_OK, SRH_ERR_NOT_STORED, SRH_ERR_BOUNDS, SRH_ERR_TIMEOUT or SRH_ERR_RANGE."""
    return load().srh_check_error(ctx)


def srh_selftest_wait_timeout(ctx, limit_us: int, stream=None) -> None:
    _check(load().srh_selftest_wait_timeout(ctx, int(limit_us), _stream(stream)), "srh_selftest_wait_timeout", ctx)


def srh_last_error(ctx) -> str:
    return load().srh_last_error(ctx).decode(errors="replace")


def header_functions(path: str = HEADER):
    """Names of the functions include/srh.h declares (for the export check)."""
    import re
    src = open(path, encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", src, flags=re.M)
    return [n for n in names if n not in ("if", "defined")]
