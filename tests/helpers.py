"""Shared test plumbing: build DecodeStep objects from workloads, fill them from
the seeded generator, drive the oracle on the same inputs, and compare."""
from __future__ import annotations

import numpy as np

from oracle import srh_oracle as O
from srh_workload import configs as C
from srh_workload import generate as G

# attention tolerance stated by the target: max|err| <= 2e-3 * max|ref|
ATTN_TOL = 2e-3
# selection: chunks whose oracle score lies within this of the cutoff may differ
SEL_BAND = 1e-5


def spec_of(w):
    from sparse_retrieval_host_gb300.runtime import StepSpec
    return StepSpec(w.scale, [w.bias] * 3, w.ensemble, w.select_mode, w.index_topk, w.tau, w.clamp)


def make_ds(w, **over):
    from sparse_retrieval_host_gb300.runtime import DecodeStep
    kw = dict(batch=w.batch, layer_ratios=w.layer_ratios, gpu_chunks=w.gpu_chunks,
              index_topk=w.index_topk, context_len=w.context_len, n_heads=w.n_heads,
              max_select=w.clamp)
    kw.update(over)
    return DecodeStep(**kw)


def fill(ds, w, pools=None):
    """Pools, window and keys of workload ``w`` into ``ds``. Returns the key arrays."""
    import torch
    from sparse_retrieval_host_gb300.runtime import bits_to_i16
    for l in range(w.n_layers):
        for b in range(w.batch):
            view = ds.pool_view(l, b)
            if pools is not None and (l, b) in pools:
                view[:] = pools[(l, b)]
            else:
                G.fill_pool(w, l, b, view)
            ds.mark_stored(l, b)
            ds.window[l, b] = torch.from_numpy(G.window(w, l, b))
    keys = [G.keys(w, b) for b in range(w.batch)]
    for b in range(w.batch):
        ds.keys[b] = bits_to_i16(keys[b])
    return keys


def load_step_inputs(ds, w, t):
    from sparse_retrieval_host_gb300.runtime import bits_to_i16
    for b in range(w.batch):
        ds.fm_q[b] = bits_to_i16(G.fm_queries(w, t, b))
        for l in range(w.n_layers):
            ds.q[l, b] = bits_to_i16(G.attn_q(w, t, l, b))


def make_oracle(w):
    ora = O.DecodeOracle(context_len=w.context_len, layer_ratios=w.layer_ratios,
                         gpu_chunks=w.gpu_chunks, index_topk=w.index_topk, batch=w.batch,
                         scale=w.scale, bias=[w.bias] * 3, ensemble_mode=w.ensemble,
                         select_mode=w.select_mode, tau=w.tau, clamp=w.clamp)
    ora.mark_all_stored()
    return ora


def selection_cutoff(w, s_ref, sel_ref):
    if w.select_mode == C.SELECT_THRESH:
        if len(sel_ref) >= w.clamp and len(sel_ref) > 0:
            return max(O.threshold_logit(w.tau), float(s_ref[sel_ref[-1]]))
        return O.threshold_logit(w.tau)
    return float(s_ref[sel_ref[-1]]) if len(sel_ref) else 0.0


def check_selection(w, s_ref, sel_ref, sel_gpu, scores_gpu):
    """Bit-exact except chunks within SEL_BAND of the cutoff; the GPU order must be
    (its own score desc, index asc). Returns True if the sets are identical."""
    cut = selection_cutoff(w, s_ref, sel_ref)
    a, b = set(sel_ref.tolist()), set(sel_gpu.tolist())
    for c in a ^ b:
        assert abs(s_ref[c] - cut) <= SEL_BAND, (c, s_ref[c], cut)
    assert len(b) == len(sel_gpu), "duplicate ids in the GPU selection"
    sg = scores_gpu[sel_gpu]
    for i in range(len(sel_gpu) - 1):
        assert sg[i] > sg[i + 1] or (sg[i] == sg[i + 1] and sel_gpu[i] < sel_gpu[i + 1]), i
    return a == b


def attn_err(out_gpu, ref):
    err = float(np.abs(out_gpu.astype(np.float64) - ref).max())
    return err, err / float(np.abs(ref).max())
