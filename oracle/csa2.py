"""The oracle's arithmetic, in numpy float64 (sources: the package docstring).

Two levels:

* the method's definitions, one function each (format decoders, indexer score,
  top-K order, block pool, RoPE, sink softmax, attention);
* row drivers that apply them to an input bundle from ``synth.make_inputs`` in
  the shape of the library's calls (index scores, block pool, top-K, sparse
  attention, one layer of a Full / Reindex / Reuse group).

Readings of points the pages leave open are stated where they are used.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "bf16_to_f64", "e4m3_to_f64", "e2m1_to_f64", "fp4_to_f64", "fp8_rows_to_f64", "mxfp4_to_f64",
    "index_scores", "topk_order", "topk_set", "block_max", "block_pool", "rope",
    "sink_softmax", "attend", "csa2_attention_row", "scored_positions",
    "keys_of", "latents_of", "swa_rows_of", "index_scores_rows", "topk_rows",
    "block_pool_rows", "sparse_attn_rows", "csa2_layer", "csa2_group",
]


# ================================================================ storage formats
def bf16_to_f64(bits) -> np.ndarray:
    """bf16 is the upper half of an IEEE-754 binary32: widen the 16-bit pattern and reinterpret."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def e4m3_to_f64(codes) -> np.ndarray:
    """OCP FP8 E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 is
    subnormal (m/8 * 2^-6); there are no infinities and S.1111.111 is NaN (largest finite 448).

    The pages name E4M3 as the FP4 group-scale format ("DeepSeek-V4.1-Flash explained",
    section 7; course, FP4 lesson, "What V4.1 changes") and FP8 for the local SWA cache;
    the bit layout is the OCP 8-bit floating-point specification's.
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def e2m1_to_f64(nibbles) -> np.ndarray:
    """E2M1: sign bit 3, two exponent bits (bias 1), one mantissa bit.  The non-negative
    magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4 and 6 (course, FP4 lesson, "Which values can E2M1
    represent?"); exponent 0 is subnormal (m * 0.5)."""
    n = np.asarray(nibbles).astype(np.int64) & 0xF
    sign = np.where(n & 0x8, -1.0, 1.0)
    e = (n >> 1) & 0x3
    m = (n & 1).astype(np.float64)
    mag = np.where(e == 0, m * 0.5, (1.0 + m / 2.0) * np.exp2(e - 1.0))
    return sign * mag


def fp4_to_f64(codes, scales, group: int) -> np.ndarray:
    """Dequantize FP4 main-KV records: value = E2M1 level x the E4M3 scale of its group
    (course FP4 lesson, section 3: a code picks a level and the group's shared scale sets its
    size; one E4M3 scale per 16 channels in section 7 of "DeepSeek-V4.1-Flash explained").

    codes [..., D/2] hold two codes per byte, the low nibble being the even channel;
    scales [..., D/group] hold one E4M3 code per group (the group size is a parameter:
    16 as the pages say, 32 for the long-context workload)."""
    codes = np.asarray(codes, dtype=np.uint8)
    lev = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), np.float64)
    lev[..., 0::2] = e2m1_to_f64(codes & 0xF)
    lev[..., 1::2] = e2m1_to_f64(codes >> 4)
    return lev * np.repeat(e4m3_to_f64(scales), group, axis=-1)


def mxfp4_to_f64(codes, exps) -> np.ndarray:
    """OCP MXFP4 (the pages' indexer precision: "DeepSeek-V4.1-Flash explained", section 7
    table, "Indexer queries and keys: OCP MXFP4"): blocks of 32 E2M1 elements share one
    UE8M0 scale 2^(e - 127), e = 255 being NaN (OCP Microscaling specification).  codes
    [..., D/2] two per byte, low nibble the even element; exps [..., D/32]."""
    codes = np.asarray(codes, dtype=np.uint8)
    e = np.asarray(exps, dtype=np.uint8).astype(np.float64)
    scale = np.where(e == 255, np.nan, np.exp2(e - 127.0))
    lev = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), np.float64)
    lev[..., 0::2] = e2m1_to_f64(codes & 0xF)
    lev[..., 1::2] = e2m1_to_f64(codes >> 4)
    return lev * np.repeat(scale, 32, axis=-1)


def fp8_rows_to_f64(codes, row_scale) -> np.ndarray:
    """FP8 row with one fp32 scale per row: value = E4M3(code) x scale."""
    return e4m3_to_f64(codes) * np.asarray(row_scale, np.float64)[..., None]


# ================================================================ the method
def index_scores(q_idx, w, keys) -> np.ndarray:
    """Lightning-indexer score of every given record:
    score_j = sum_h w_h * ReLU(q^I_h . k^I_j) over the indexer heads.

    The indexer sums the rectified query-key dot products of its 32 heads, each weighted
    ("Every layer, connected", "The global and index paths").  Reading: one indexer key per
    record, shared by all heads (the pages call the keys compact and give them no head index),
    no scaling or bias, and one weight per head for this query row.

    q_idx [HI, DI], w [HI], keys [n, DI] -> scores [n]."""
    dots = np.asarray(keys, np.float64) @ np.asarray(q_idx, np.float64).T  # [n, HI]
    return np.maximum(dots, 0.0) @ np.asarray(w, np.float64)


def topk_order(scores, k: int) -> np.ndarray:
    """Indices of the k highest scores, highest first, equal scores lowest index first.

    Top-K returns addresses, not scores, and ties go to the lower position (course,
    06 "Indexer and attention", the select_values example and its note).  -0.0 and +0.0
    compare equal."""
    s = np.asarray(scores, np.float64)
    order = np.lexsort((np.arange(s.shape[0]), -s))
    return order[:k]


def topk_set(scores, k: int) -> np.ndarray:
    """The selected indices as an ascending set (attention does not depend on their order)."""
    return np.sort(topk_order(scores, k))


def block_max(scores, bs: int) -> np.ndarray:
    """Score of every block of bs consecutive positions = the highest score in it; a partial
    last block uses the positions it has ("Every layer, connected", hierarchical figure: each
    block's score is the maximum score among its positions)."""
    s = np.asarray(scores, np.float64)
    return np.maximum.reduceat(s, np.arange(0, s.shape[0], bs)) if s.shape[0] else s


def block_pool(scores, bs: int, n_keep: int):
    """Hierarchical candidate pool of the first decoder indexer: score every visible position,
    score each block by its best position, keep the n_keep best blocks (ties to the lower block
    index, as for positions), and pool every position of the kept blocks, ascending
    ("DeepSeek-V4.1-Flash explained", section 3; course, 07 "Hierarchical indexing").

    scores [n_visible] -> (pool positions ascending, block maxima, kept block indices)."""
    n = len(scores)
    bm = block_max(scores, bs)
    kept = topk_set(bm, n_keep)
    pool = [np.arange(c * bs, min(n, (c + 1) * bs)) for c in kept]
    pool = np.concatenate(pool) if pool else np.zeros(0, np.int64)
    return pool, bm, kept


def scored_positions(n_visible: int, n_later: int, n_keep: int, bs: int) -> int:
    """Positions scored by one full-range indexer plus n_later indexers restricted to a pool of
    n_keep blocks of bs positions ("DeepSeek-V4.1-Flash explained", section 3)."""
    return n_visible + n_later * min(n_visible, n_keep * bs)


def rope(x, pos, theta: float, R: int, sign: int = 1) -> np.ndarray:
    """Rotary embedding of the last R coordinates: pair i = (D-R+2i, D-R+2i+1) turns by the
    angle sign*pos*theta^(-2i/R): (x, y) -> (x cos a - y sin a, x sin a + y cos a).

    RoPE acts on the last 64 dims (qk_rope_head_dim) and the output's rotary coordinates are
    turned back by position -i ("DeepSeek V4 Inside", layer-0 SWA and CSA sections; "Every
    layer, connected", "The query and output paths").  Readings: adjacent pairs, frequencies
    theta^(-2i/R) with theta = 1e4 (the pages print one pair only)."""
    x = np.array(x, dtype=np.float64, copy=True)
    D = x.shape[-1]
    i = np.arange(R // 2, dtype=np.float64)
    a = sign * float(pos) * np.power(float(theta), -2.0 * i / R)
    c, s = np.cos(a), np.sin(a)
    xe = x[..., D - R::2].copy()
    xo = x[..., D - R + 1::2].copy()
    x[..., D - R::2] = xe * c - xo * s
    x[..., D - R + 1::2] = xe * s + xo * c
    return x


def sink_softmax(z, z_sink):
    """Softmax with a sink logit in the denominator only: s_j = exp(z_j) / (sum_k exp(z_k) +
    exp(z')) ("DeepSeek V4 Inside", eq. (27)).  The weights sum to 1 - sink mass.
    Returns (weights, sink mass).  z_sink = -inf removes the sink."""
    e = np.exp(np.asarray(z, np.float64))
    es = math.exp(z_sink) if np.isfinite(z_sink) else 0.0
    den = e.sum() + es
    return e / den, es / den


def attend(q, keys, values, scale: float, sink) -> tuple[np.ndarray, np.ndarray]:
    """Softmax attention of every query head over the same rows, with one sink logit per head:
    logits z = scale * q_h . key_j; output sum_j s_j value_j with s from ``sink_softmax``.

    q [H, D], keys [n, D], values [n, D], sink [H] -> (o [H, D], sink mass [H])."""
    q = np.asarray(q, np.float64)
    z = scale * (q @ np.asarray(keys, np.float64).T)
    v = np.asarray(values, np.float64)
    H = q.shape[0]
    o = np.zeros((H, v.shape[1]))
    sm = np.zeros(H)
    for h in range(H):
        p, sm[h] = sink_softmax(z[h], float(sink[h]))
        o[h] = p @ v
    return o, sm


def csa2_attention_row(q, q_pos, sel_rows, swa_rows, sink, theta, R, scale):
    """Main attention of one query row: RoPE on the last R dims of every head of q at q_pos;
    the selected shared latents and the layer's sliding-window rows each serve as key and
    value at once (shared-KV MQA, one KV head); one sink logit per head; the output's rotary
    coordinates turned back by -q_pos ("DeepSeek V4 Inside", CSA section; "Every layer,
    connected", "The query and output paths" and "The global and index paths").

    Stored latents and window rows are taken as already rotated (the course FP4 lesson has
    the cache quantized after RoPE is applied), so only q is rotated here."""
    qr = rope(q, q_pos, theta, R)
    kv = np.concatenate([np.asarray(sel_rows, np.float64).reshape(-1, qr.shape[1]),
                         np.asarray(swa_rows, np.float64).reshape(-1, qr.shape[1])], 0)
    o, sm = attend(qr, kv, kv, scale, sink)
    return rope(o, q_pos, theta, R, sign=-1), sm


# ================================================================ row drivers
def keys_of(inp, b: int, positions=None) -> np.ndarray:
    """Decoded indexer keys of sequence b (all records, or the given positions)."""
    c, p = inp["cache"], inp["params"]
    k = c["k_idx"][b] if positions is None else c["k_idx"][b][positions]
    if p["key_fmt"] == "bf16":
        return bf16_to_f64(k)
    sc = c["k_scale"][b] if positions is None else c["k_scale"][b][positions]
    if p["key_fmt"] == "mxfp4":
        return mxfp4_to_f64(k, sc)
    return fp8_rows_to_f64(k, sc)


def latents_of(inp, b: int, positions) -> np.ndarray:
    """Decoded shared latents of sequence b at the given positions."""
    c, p = inp["cache"], inp["params"]
    if p["lat_fmt"] == "bf16":
        return bf16_to_f64(c["lat"][b][positions])
    return fp4_to_f64(c["lat"][b][positions], c["lat_scales"][b][positions], p["lat_group"])


def swa_rows_of(inp, layer: int, b: int, q_pos: int) -> np.ndarray:
    """The layer's own sliding-window rows seen by a query at q_pos: absolute positions
    max(q_pos-W+1, swa_pos0) .. q_pos, the current token included ("DeepSeek V4 Inside",
    layer-0 SWA: with a window of 2 the query attends to the previous token and to itself)."""
    p, rows, lay = inp["params"], inp["rows"], inp["layers"][layer]
    W = p["W"]
    pos0 = int(rows["swa_pos0"][b])
    if W == 0:
        return np.zeros((0, p["D"]))
    lo = max(q_pos - W + 1, pos0)
    r = np.arange(lo - pos0, q_pos - pos0 + 1)
    if p["swa_fmt"] == "bf16":
        return bf16_to_f64(lay["swa"][b][r])
    return fp8_rows_to_f64(lay["swa"][b][r], lay["swa_scale"][b][r])


def index_scores_rows(inp, layer: int, rows=None, cand=None, n_cand=None) -> np.ndarray:
    """Indexer scores of the given query rows (all rows by default).

    Without ``cand``: scores of records 0..N-1, with records at or beyond the row's
    n_visible excluded (-inf): selection is causal ("Every layer, connected", "The global and
    index paths"); the mask applies before selection.  With ``cand`` [Bq, L] (e.g. a pool):
    scores of the listed positions; entries beyond ``n_cand`` are -inf."""
    p, rw, lay = inp["params"], inp["rows"], inp["layers"][layer]
    rows = range(p["Bq"]) if rows is None else rows
    L = p["N"] if cand is None else cand.shape[1]
    out = np.full((len(rows), L), -np.inf)
    cache_keys = {}
    for i, r in enumerate(rows):
        b = int(rw["seq_of_row"][r])
        qi = bf16_to_f64(lay["q_idx"][r])
        w = np.asarray(lay["w"][r], np.float64)
        if cand is None:
            if b not in cache_keys:
                cache_keys = {b: keys_of(inp, b)}
            nv = int(rw["n_visible"][r])
            out[i, :nv] = index_scores(qi, w, cache_keys[b][:nv])
        else:
            nc = int(n_cand[r])
            out[i, :nc] = index_scores(qi, w, keys_of(inp, b, cand[r, :nc]))
    return out


def topk_rows(scores, n_valid, K: int, cand=None) -> np.ndarray:
    """Top-K of every row as the ascending set of record positions, -1 padded when fewer
    than K candidates are valid.  ``scores`` [rows, L]; the first n_valid[r] entries of row r
    are candidates; ``cand`` maps entry j to a record position (identity if None)."""
    rows = scores.shape[0]
    out = np.full((rows, K), -1, np.int64)
    for r in range(rows):
        nv = int(n_valid[r])
        sel = topk_set(scores[r, :nv], K)
        pos = sel if cand is None else cand[r, sel]
        out[r, :len(pos)] = pos
    return out


def block_pool_rows(scores, n_visible, bs: int, n_keep: int):
    """Block pool of every row (see ``block_pool``): pool [rows, n_keep*bs] ascending, -1
    padded, and the pool size of each row."""
    rows = scores.shape[0]
    pool = np.full((rows, n_keep * bs), -1, np.int64)
    n_pool = np.zeros(rows, np.int64)
    for r in range(rows):
        pl, _, _ = block_pool(scores[r, :int(n_visible[r])], bs, n_keep)
        pool[r, :len(pl)] = pl
        n_pool[r] = len(pl)
    return pool, n_pool


def sparse_attn_rows(inp, layer: int, idx, rows=None):
    """Main attention of the given rows over their selected records (``idx`` [rows, K], -1
    entries skipped) plus the layer's window rows.  -> (o [rows, H, D], sink mass [rows, H])."""
    p, rw, lay = inp["params"], inp["rows"], inp["layers"][layer]
    rows = range(p["Bq"]) if rows is None else rows
    H, D = p["H"], p["D"]
    o = np.zeros((len(rows), H, D))
    sm = np.zeros((len(rows), H))
    for i, r in enumerate(rows):
        b = int(rw["seq_of_row"][r])
        qp = int(rw["q_pos"][r])
        sel = np.asarray(idx[i])
        sel = sel[sel >= 0]
        o[i], sm[i] = csa2_attention_row(
            bf16_to_f64(lay["q"][r]), qp, latents_of(inp, b, sel), swa_rows_of(inp, layer, b, qp),
            lay["sink"], p["theta"], p["R"], p["softmax_scale"])
    return o, sm


def csa2_layer(inp, layer: int, prev=None, rows=None) -> dict:
    """One CSA2 layer in its mode ("DeepSeek-V4.1-Flash explained", section 2, mode table;
    section 3):

    * full      - fresh scores over every visible record, fresh top-K, attention;
    * full_pool - as full, and also the block pool for the later indexers (the first decoder
                  indexer selects its own top-K and builds the pool);
    * reindex   - scores of this layer's own indexer query over the pool of the preceding
                  full_pool layer only, fresh top-K from the pool, attention;
    * reuse     - no indexing; the selection of the immediately preceding layer, attention
                  with this layer's own query, window rows and sinks.

    ``prev`` is the result dict of the preceding layer of the group."""
    p, rw = inp["params"], inp["rows"]
    mode = inp["layers"][layer]["mode"]
    rows = list(range(p["Bq"])) if rows is None else list(rows)
    res = {"mode": mode, "rows": rows}
    if mode in ("full", "full_pool"):
        s = index_scores_rows(inp, layer, rows)
        nv = rw["n_visible"][rows]
        res["scores"] = s
        res["idx"] = topk_rows(s, nv, p["K"])
        if mode == "full_pool":
            res["pool"], res["n_pool"] = block_pool_rows(s, nv, p["block_size"], p["n_keep"])
    elif mode == "reindex":
        pool, n_pool = prev["pool"], prev["n_pool"]
        full_pool = np.full((p["Bq"], pool.shape[1]), -1, np.int64)
        full_n = np.zeros(p["Bq"], np.int64)
        full_pool[rows], full_n[rows] = pool, n_pool
        s = index_scores_rows(inp, layer, rows, cand=full_pool, n_cand=full_n)
        res["scores"] = s
        res["idx"] = topk_rows(s, n_pool, p["K"], cand=pool)
        res["pool"], res["n_pool"] = pool, n_pool
    elif mode == "reuse":
        res["idx"] = prev["idx"]
        res["pool"], res["n_pool"] = prev.get("pool"), prev.get("n_pool")
    else:
        raise ValueError(mode)
    res["o"], res["sink_mass"] = sparse_attn_rows(inp, layer, res["idx"], rows)
    return res


def csa2_group(inp, rows=None) -> list:
    """Every layer of a sharing group in order (a single full layer for plain decode)."""
    out, prev = [], None
    for l in range(len(inp["layers"])):
        prev = csa2_layer(inp, l, prev, rows)
        out.append(prev)
    return out
