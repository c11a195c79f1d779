"""Helpers shared by the parity tests: run a bundle through the CUDA library and compare
with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
import synth

TOL_BF16 = 2e-3   # max |o_gpu - o_oracle| / RMS(o_oracle), bf16 caches
TOL_FP = 1e-2     # the same for FP8 / FP4 caches


def out_tol(params) -> float:
    return TOL_BF16 if (params["lat_fmt"] == "bf16" and params["swa_fmt"] == "bf16") else TOL_FP


def rel_err(o_gpu, o_ora) -> float:
    o_gpu = np.asarray(o_gpu, np.float64)
    rms = float(np.sqrt(np.mean(o_ora ** 2)))
    return float(np.max(np.abs(o_gpu - o_ora))) / rms


def decode_kwargs(dv, layer: int, K: int):
    """Keyword arguments of sparse_attention_csa2_gb300.DecodeLayer for one layer of a device bundle."""
    p, rows, cache, lay = dv["params"], dv["rows"], dv["cache"], dv["layers"][layer]
    kw = dict(seq_of_row=rows["seq_of_row"], n_visible=rows["n_visible"], q=lay["q"], q_pos=rows["q_pos"],
              latents=cache["lat"], lat_scale=cache["lat_scales"], swa=lay["swa"], swa_scale=lay["swa_scale"],
              swa_pos0=rows["swa_pos0"], window=p["W"], sink=lay["sink"], K=K, theta=p["theta"],
              softmax_scale=p["softmax_scale"], block_size=p["block_size"], n_keep=p["n_keep"])
    if lay["mode"] != "reuse":
        kw.update(q_idx=lay["q_idx"], w=lay["w"], k_idx=cache["k_idx"], k_scale=cache["k_scale"])
    return kw


def gpu_group(dv, K=None):
    """Runs every layer of a device bundle through csa2_fused_decode; returns the DecodeLayer objects."""
    import sparse_attention_csa2_gb300 as S
    K = dv["params"]["K"] if K is None else K
    layers, prev = [], None
    for l, lay in enumerate(dv["layers"]):
        kw = decode_kwargs(dv, l, K)
        if lay["mode"] == "reindex":
            kw.update(pool=prev.pool, n_pool=prev.n_pool)
        if lay["mode"] == "reuse":
            kw.update(idx=prev.idx, pool=prev.pool, n_pool=prev.n_pool)
        prev = S.DecodeLayer(lay["mode"], **kw)
        prev()
        layers.append(prev)
    torch.cuda.synchronize()
    return layers


def set_rows(inp, n_visible, q_pos=None):
    """Per-row visibility for a decode bundle (one row per sequence): n_visible[r] records
    visible, the query at q_pos (default n_visible), window rows ending at q_pos."""
    p, rows = inp["params"], inp["rows"]
    nv = np.asarray(n_visible, np.int32)
    qp = nv.astype(np.int64) if q_pos is None else np.asarray(q_pos, np.int64)
    rows["n_visible"] = nv
    rows["q_pos"] = qp
    rows["swa_pos0"] = np.maximum(qp - p["W"] + 1, 0)[: p["B"]]
    return inp


def check_idx_near_ties(idx_gpu, idx_ora, scores_ora, bound):
    """GPU and oracle selections may differ only by swaps across the K-boundary between
    entries whose oracle scores lie within `bound` of the oracle's K-th score.  Returns the
    number of swaps."""
    swaps = 0
    for r in range(idx_ora.shape[0]):
        a = set(int(x) for x in idx_gpu[r] if x >= 0)
        b = set(int(x) for x in idx_ora[r] if x >= 0)
        assert len(a) == len(b)
        if a == b:
            continue
        s = scores_ora[r]
        kth = min(s[j] for j in b)
        for j in a - b:
            assert s[j] >= kth - bound[r], (r, j, s[j], kth)
        for j in b - a:
            assert s[j] <= kth + bound[r], (r, j, s[j], kth)
        swaps += len(a - b)
    return swaps


def score_bound(inp, layer, rows=None):
    """Per-row fp32 accumulation bound for indexer scores: 1e-5 * sum_h w_h |q_h| max_j |k_j|."""
    p, rw, lay = inp["params"], inp["rows"], inp["layers"][layer]
    rows = range(p["Bq"]) if rows is None else rows
    out = []
    for r in rows:
        b = int(rw["seq_of_row"][r])
        qn = np.linalg.norm(O.bf16_to_f64(lay["q_idx"][r]), axis=1)
        kn = np.linalg.norm(O.keys_of(inp, b), axis=1).max()
        out.append(1e-5 * float(np.sum(np.asarray(lay["w"][r], np.float64) * qn)) * kn + 1e-6)
    return np.array(out)


def scores_by_position(ref_layer, n_records):
    """Oracle scores of one layer indexed by record position (-inf where the record is not a
    candidate): a full layer's rows as they are; a Reindex layer's pool slots placed at their
    positions."""
    s = ref_layer["scores"]
    if ref_layer["mode"] != "reindex":
        return s
    out = np.full((s.shape[0], n_records), -np.inf)
    pool, n_pool = ref_layer["pool"], ref_layer["n_pool"]
    for r in range(s.shape[0]):
        n = int(n_pool[r])
        out[r, pool[r, :n]] = s[r, :n]
    return out


def check_pool_near_ties(pool_gpu, n_pool_gpu, scores_ora, n_visible, bs, n_keep, bound):
    """A GPU block pool against the oracle's scores of the same rows.  The pool must list every
    visible position of its kept blocks in ascending order (-1 after them) and keep
    min(n_keep, blocks) blocks; the kept blocks may differ from the oracle's only by swaps
    across the n_keep boundary between blocks whose oracle block maxima lie within `bound` of
    the oracle's n_keep-th block maximum.  Returns the number of swapped blocks."""
    swaps = 0
    for r in range(len(n_visible)):
        nv = int(n_visible[r])
        _, bm, kept_ora = O.block_pool(scores_ora[r, :nv], bs, n_keep)
        n = int(n_pool_gpu[r])
        p = np.asarray(pool_gpu[r], np.int64)
        kept = np.unique(p[:n] // bs)
        expect = np.concatenate([np.arange(c * bs, min((c + 1) * bs, nv)) for c in kept])
        assert np.array_equal(p[:n], expect) and np.all(p[n:] == -1), r
        assert len(kept) == len(kept_ora), r
        a, b = set(int(c) for c in kept), set(int(c) for c in kept_ora)
        if a == b:
            continue
        kth = min(bm[c] for c in b)
        for c in a - b:
            assert bm[c] >= kth - bound[r], (r, c, bm[c], kth)
        for c in b - a:
            assert bm[c] <= kth + bound[r], (r, c, bm[c], kth)
        swaps += len(a - b)
    return swaps
