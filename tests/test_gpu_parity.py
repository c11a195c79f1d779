"""Parity of the CUDA library with the CPU oracle, call by call, on seeded inputs.

Sizes span several tiles, segments and a ragged tail while keeping the oracle to seconds.
Bars: selected indices and pools bit-exact (grid mode, where every score is exact in fp32,
and whenever both sides select from the same fp32 scores); outputs within 2e-3 x RMS for
bf16 caches and 1e-2 x RMS for FP8/FP4 caches.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from csa2_testlib import (check_idx_near_ties, check_pool_near_ties, gpu_group, out_tol, rel_err, score_bound,
                          scores_by_position, set_rows)

pytestmark = pytest.mark.gpu

S = pytest.importorskip("sparse_attention_csa2_gb300")


def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def small(name, seed=7, mode="gauss", **kw):
    return synth.make_inputs(synth.scaled(synth.WORKLOADS[name], **kw), seed=seed, mode=mode)


# ------------------------------------------------------------------ index scores
@pytest.mark.parametrize("key_fmt", ["bf16", "fp8", "mxfp4"])
@pytest.mark.parametrize("mode", ["grid", "gauss"])
def test_index_scores(key_fmt, mode):
    _cuda()
    inp = small("batched_decode", seed=3, mode=mode, B=3, N=5003, key_fmt=key_fmt)
    set_rows(inp, [5003, 4321, 37])
    dv = synth.to_device(inp)
    c, lay, rw = dv["cache"], dv["layers"][0], dv["rows"]
    s, bmax = S.index_scores(lay["q_idx"], lay["w"], c["k_idx"], c["k_scale"], rw["seq_of_row"], rw["n_visible"],
                             block_size=64)
    s = s.cpu().numpy().astype(np.float64)
    ref = O.index_scores_rows(inp, 0)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(s), fin)
    if mode == "grid":
        assert np.array_equal(s[fin], ref[fin])
    else:
        bound = score_bound(inp, 0)
        assert np.all(np.abs(s - ref)[fin] <= np.repeat(bound[:, None], s.shape[1], 1)[fin])
    bm = bmax.cpu().numpy().astype(np.float64)
    for r in range(3):
        nv = int(inp["rows"]["n_visible"][r])
        ref_bm = O.block_max(s[r, :nv], 64)  # block maxima of the GPU's own scores: exact
        assert np.array_equal(bm[r, :len(ref_bm)], ref_bm)
        assert np.all(np.isneginf(bm[r, len(ref_bm):]))


@pytest.mark.parametrize("key_fmt", ["bf16", "fp8"])
def test_index_scores_heads_of_wide_magnitude(key_fmt):
    """q^I heads scaled by powers of two from 2^-100 to 2^60 (one head all zero), the head
    weights by the inverse: every head still weighs alike in the score, so a head whose
    magnitude the kernel mishandles (FP8 keys widen q^I to f16 with a per-head scale) shows."""
    _cuda()
    inp = small("batched_decode", seed=9, mode="gauss", B=2, N=3001, key_fmt=key_fmt)
    set_rows(inp, [3001, 1777])
    lay = inp["layers"][0]
    HI = lay["q_idx"].shape[1]
    ex = np.array([(-100, -60, -30, -8, 0, 7, 25, 60)[h % 8] for h in range(HI)], np.float64)
    q = O.bf16_to_f64(lay["q_idx"]) * np.exp2(ex)[None, :, None]
    q[:, 3, :] = 0.0
    lay["q_idx"] = synth.bf16_bits(torch.from_numpy(q.astype(np.float32)))
    lay["w"] = (np.asarray(lay["w"], np.float64) * np.exp2(-ex)[None, :]).astype(np.float32)
    dv = synth.to_device(inp)
    c, dl, rw = dv["cache"], dv["layers"][0], dv["rows"]
    s = S.index_scores(dl["q_idx"], dl["w"], c["k_idx"], c["k_scale"], rw["seq_of_row"], rw["n_visible"])
    s = s.cpu().numpy().astype(np.float64)
    ref = O.index_scores_rows(inp, 0)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(s), fin)
    bound = score_bound(inp, 0)
    assert np.all(np.abs(s - ref)[fin] <= np.repeat(bound[:, None], s.shape[1], 1)[fin])


def test_index_scores_over_candidates():
    _cuda()
    inp = small("hierarchical", seed=5, mode="grid", B=2, N=3000)
    rng = np.random.default_rng(0)
    L = 700
    cand = np.full((2, L), -1, np.int32)
    n_cand = np.array([700, 333], np.int32)
    for r in range(2):
        cand[r, :n_cand[r]] = np.sort(rng.choice(3000, n_cand[r], replace=False))
    dv = synth.to_device(inp)
    c, lay, rw = dv["cache"], dv["layers"][0], dv["rows"]
    s = S.index_scores(lay["q_idx"], lay["w"], c["k_idx"], c["k_scale"], rw["seq_of_row"], rw["n_visible"],
                       cand=torch.from_numpy(cand).cuda(), n_cand=torch.from_numpy(n_cand).cuda())
    ref = O.index_scores_rows(inp, 0, cand=cand.astype(np.int64), n_cand=n_cand)
    s = s.cpu().numpy().astype(np.float64)
    assert np.array_equal(np.isfinite(s), np.isfinite(ref))
    assert np.array_equal(s[np.isfinite(ref)], ref[np.isfinite(ref)])


# ------------------------------------------------------------------ top-K
@pytest.mark.parametrize("L,K", [(3001, 512), (100_003, 512), (70_000, 37), (600, 1024), (9, 4)])
def test_topk_exact_on_seeded_scores(L, K):
    _cuda()
    rows = 5
    sc = synth.integers((rows, L), 9, L % 97, -50, 50).float() / 4.0  # many ties
    sc[1] = synth.normal((L,), 9, 1)  # no ties
    sc[2, ::3] = -0.0
    sc[2, 1::3] = 0.0
    n_valid = np.array([L, L - 1, L // 2, min(K, L), 1], np.int32)
    idx = S.topk(sc.cuda(), torch.from_numpy(n_valid).cuda(), K).cpu().numpy()
    ref = O.topk_rows(sc.numpy().astype(np.float64), n_valid, K)
    assert np.array_equal(idx, ref)


def test_topk_with_candidate_map():
    _cuda()
    L, K = 5000, 300
    sc = synth.integers((2, L), 4, 1, 0, 9).float()
    cand = np.sort(np.random.default_rng(1).choice(10 ** 6, (2, L), replace=False), axis=1).astype(np.int32)
    n_valid = np.array([L, 1234], np.int32)
    idx = S.topk(sc.cuda(), torch.from_numpy(n_valid).cuda(), K, cand=torch.from_numpy(cand).cuda()).cpu().numpy()
    ref = O.topk_rows(sc.numpy().astype(np.float64), n_valid, K, cand=cand)
    assert np.array_equal(idx, ref)


# ------------------------------------------------------------------ block pool
@pytest.mark.parametrize("N,bs,keep", [(131_072, 64, 64), (5003, 64, 16), (1000, 16, 100), (777, 128, 3)])
def test_block_pool(N, bs, keep):
    _cuda()
    rows = 3
    sc = synth.integers((rows, N), 6, bs, -20, 20).float()
    n_vis = np.array([N, N - 5, max(1, N // 3)], np.int32)
    bm = np.full((rows, (N + bs - 1) // bs), -np.inf, np.float32)
    for r in range(rows):
        b = O.block_max(sc[r, :n_vis[r]].numpy().astype(np.float64), bs)
        bm[r, :len(b)] = b
    pool, n_pool = S.block_pool(torch.from_numpy(bm).cuda(), torch.from_numpy(n_vis).cuda(), bs, keep)
    ref_pool, ref_n = O.block_pool_rows(sc.numpy().astype(np.float64), n_vis, bs, keep)
    assert np.array_equal(n_pool.cpu().numpy(), ref_n)
    assert np.array_equal(pool.cpu().numpy(), ref_pool)


# ------------------------------------------------------------------ sparse attention
@pytest.mark.parametrize("lat_fmt,group,swa_fmt", [("bf16", 32, "bf16"), ("fp4", 32, "fp8"), ("fp4", 16, "bf16")])
def test_sparse_attn(lat_fmt, group, swa_fmt):
    _cuda()
    inp = small("batched_decode", seed=11, B=3, N=4000, lat_fmt=lat_fmt, lat_group=group, swa_fmt=swa_fmt)
    set_rows(inp, [4000, 3000, 100])
    rng = np.random.default_rng(2)
    K = 512
    idx = np.full((3, K), -1, np.int64)
    for r, nv in enumerate([4000, 3000, 100]):
        sel = np.sort(rng.choice(nv, min(K, nv), replace=False))
        idx[r, :len(sel)] = sel
    dv = synth.to_device(inp)
    c, lay, rw, p = dv["cache"], dv["layers"][0], dv["rows"], dv["params"]
    out, sm = S.sparse_attn(lay["q"], rw["q_pos"], rw["seq_of_row"], c["lat"], c["lat_scales"],
                            torch.from_numpy(idx.astype(np.int32)).cuda(), lay["swa"], lay["swa_scale"],
                            rw["swa_pos0"], p["W"], lay["sink"], p["theta"], p["softmax_scale"])
    o_ref, sm_ref = O.sparse_attn_rows(inp, 0, idx)
    err = rel_err(out.cpu().numpy(), o_ref)
    assert err <= out_tol(inp["params"]), err
    assert np.max(np.abs(sm.cpu().numpy() - sm_ref)) < 1e-4
    assert np.all(sm.cpu().numpy() < 1.0)  # the sink keeps the attention mass below one


# ------------------------------------------------------------------ fused decode layers
@pytest.mark.parametrize("key_fmt,lat_fmt,swa_fmt", [("bf16", "bf16", "bf16"), ("fp8", "fp4", "fp8"),
                                                     ("mxfp4", "fp4", "fp8")])
def test_fused_full_grid_exact_indices(key_fmt, lat_fmt, swa_fmt):
    _cuda()
    inp = small("batched_decode", seed=4, mode="grid", B=3, N=9001, key_fmt=key_fmt, lat_fmt=lat_fmt,
                swa_fmt=swa_fmt)
    set_rows(inp, [9001, 5000, 300])
    g = gpu_group(synth.to_device(inp))
    ref = O.csa2_group(inp)
    assert np.array_equal(g[0].idx.cpu().numpy(), ref[0]["idx"])
    assert rel_err(g[0].out.cpu().numpy(), ref[0]["o"]) <= out_tol(inp["params"])


def test_fused_full_gauss():
    _cuda()
    inp = small("batched_decode", seed=8, B=4, N=20_000)
    set_rows(inp, [20_000, 19_999, 12_345, 513])
    g = gpu_group(synth.to_device(inp))
    ref = O.csa2_group(inp)
    swaps = check_idx_near_ties(g[0].idx.cpu().numpy(), ref[0]["idx"], ref[0]["scores"], score_bound(inp, 0))
    assert swaps == 0
    assert rel_err(g[0].out.cpu().numpy(), ref[0]["o"]) <= out_tol(inp["params"])


@pytest.mark.parametrize("mode", ["grid", "gauss", "ties"])
@pytest.mark.parametrize("forced_seg,B,N,rows,K", [
    (40, 4, 50_000, [50_000, 49_999, 7_777, 300], 512),  # two waves of segments: lists, then the merge
    (40, 4, 50_000, [50_000, 49_999, 7_777, 300], 64),   # small K: the buffers prune and select often
    (0, 160, 3_000, None, 512),                          # more rows than SMs: one segment per row
    (1, 12, 200_000, None, 512),                         # one segment longer than the placement bitmap
])
def test_fused_full_fp8_streaming_scan(mode, forced_seg, B, N, rows, K):
    """FP8 keys over more work than one wave of the decode kernel's segments (each segment's
    keys kept in shared memory, one block per SM): the FULL layer takes the streaming FP8
    scan (per-warp top-K buffers, two blocks per SM), then the lists merge when a row has
    several segments.  Forcing 40 segments on 4 rows makes such a grid at a size the oracle
    finishes quickly; a 300-record row leaves most of its segments empty; one forced segment of
    200,000 records per row is longer than the bitmap that places a segment's survivors, so
    they are placed by the engine's searches instead.  Grid mode: indices
    bit-exact; Gaussian mode: near-tie swaps only (none on these seeds).  Ties: a zero indexer
    query makes every score 0, so each row keeps its lowest positions (every selection step
    decides by position alone)."""
    _cuda()
    inp = small("long_decode", seed=21, mode="grid" if mode == "ties" else mode, B=B, N=N, K=K)
    if mode == "ties":
        inp["layers"][0]["q_idx"][...] = 0
    if rows is not None:
        set_rows(inp, rows)
    if forced_seg:
        S.set_tuning(S.TUNE_SCAN_SEGMENTS, forced_seg)
    try:
        dv = synth.to_device(inp)
        with torch.profiler.profile(activities=[torch.profiler.ProfilerActivity.CUDA]) as prof:
            g = gpu_group(dv)
            torch.cuda.synchronize()
    finally:
        S.reset_tuning()
    kernels = [e.name for e in prof.events() if e.device_type == torch.autograd.DeviceType.CUDA]
    if kernels:  # (empty when the profiler cannot trace kernels on this machine)
        assert any("idx_fp8_stream_kernel" in k for k in kernels), sorted(set(kernels))
    ref = O.csa2_group(inp)
    idx = g[0].idx.cpu().numpy()
    if mode == "gauss":
        assert check_idx_near_ties(idx, ref[0]["idx"], ref[0]["scores"], score_bound(inp, 0)) == 0
    else:
        assert np.array_equal(idx, ref[0]["idx"])
    assert rel_err(g[0].out.cpu().numpy(), ref[0]["o"]) <= out_tol(inp["params"])


@pytest.mark.parametrize("mode,key_fmt", [("grid", "bf16"), ("gauss", "bf16"), ("grid", "fp8"), ("gauss", "fp8")])
def test_fused_hierarchical_group(mode, key_fmt):
    """FULL_POOL -> 3 x REINDEX -> 2 x REUSE.  Grid mode: pool and every layer's indices
    bit-exact.  Gaussian mode: the pool and every scoring layer's indices may differ from the
    oracle's only by near-tie swaps at the boundary (none on this seed), checked against the
    oracle's scores of that layer."""
    _cuda()
    inp = small("hierarchical", seed=12, mode=mode, B=2, N=9000, n_keep=16, n_hot_blocks=10, key_fmt=key_fmt)
    set_rows(inp, [9000, 7001])
    g = gpu_group(synth.to_device(inp))
    ref = O.csa2_group(inp)
    p = inp["params"]
    assert np.array_equal(g[0].n_pool.cpu().numpy(), ref[0]["n_pool"])
    if mode == "grid":
        assert np.array_equal(g[0].pool.cpu().numpy(), ref[0]["pool"])
    else:
        swaps = check_pool_near_ties(g[0].pool.cpu().numpy(), g[0].n_pool.cpu().numpy(), ref[0]["scores"],
                                     inp["rows"]["n_visible"], p["block_size"], p["n_keep"], score_bound(inp, 0))
        assert swaps == 0
    for l in range(len(ref)):
        gi = g[l].idx.cpu().numpy()
        if mode == "grid":
            assert np.array_equal(gi, ref[l]["idx"]), l
        elif ref[l]["mode"] != "reuse":
            swaps = check_idx_near_ties(gi, ref[l]["idx"], scores_by_position(ref[l], p["N"]), score_bound(inp, l))
            assert swaps == 0, l
        assert rel_err(g[l].out.cpu().numpy(), ref[l]["o"]) <= out_tol(inp["params"]), l
    # Reuse layers: the same selection as the last Reindex layer, different outputs
    assert np.array_equal(g[4].idx.cpu().numpy(), g[3].idx.cpu().numpy())
    o4, o5 = g[4].out.cpu().numpy(), g[5].out.cpu().numpy()
    assert np.max(np.abs(o4 - o5)) > 0.1 * np.sqrt(np.mean(o4 ** 2))


def test_fused_decode_is_deterministic_and_causal():
    _cuda()
    inp = small("batched_decode", seed=21, B=2, N=6000)
    set_rows(inp, [5000, 4000])
    a = gpu_group(synth.to_device(inp))
    b = gpu_group(synth.to_device(inp))
    assert torch.equal(a[0].idx, b[0].idx) and torch.equal(a[0].out, b[0].out)
    # records at or past n_visible do not matter
    inp["cache"]["k_idx"][:, 5000:] = inp["cache"]["k_idx"][:, 5000:][:, ::-1]
    inp["cache"]["lat"][:, 5000:] ^= np.uint16(0x0101)
    c = gpu_group(synth.to_device(inp))
    assert torch.equal(a[0].idx, c[0].idx) and torch.equal(a[0].out, c[0].out)
    assert int(a[0].idx.max()) < 5000


def test_decode_equals_prefill_row():
    _cuda()
    # a prefill chunk, and the same query rows run as decode rows with the same visibility
    wl = synth.scaled(synth.WORKLOADS["prefill_chunk"], N=2100, T=40, P0=2060)
    inp = synth.make_inputs(wl, seed=5)
    ref = O.csa2_layer(inp, 0, rows=[0, 17, 39])
    dv = synth.to_device(inp)
    g = gpu_group(dv)
    got = g[0].out.cpu().numpy()
    for i, t in enumerate([0, 17, 39]):
        assert rel_err(got[t][None], ref["o"][i][None]) <= 2e-3
        # decode call on the single row t (batch of one, sequence 0)
        one = {k: (v[t:t + 1] if k in ("q_pos", "n_visible", "seq_of_row") else v) for k, v in dv["rows"].items()}
        lay = dict(dv["layers"][0])
        for k in ("q_idx", "w", "q"):
            lay[k] = lay[k][t:t + 1].contiguous()
        d1 = dict(dv, rows=one, layers=[lay])
        d1["params"] = dict(dv["params"], Bq=1)
        g1 = gpu_group(d1)
        assert torch.equal(g1[0].idx[0], g[0].idx[t])
        assert rel_err(g1[0].out[0].cpu().numpy()[None], ref["o"][i][None]) <= 2e-3


# ------------------------------------------------------------------ prefill indexer (tcgen05, persistent)
@pytest.mark.parametrize("mode", ["grid", "gauss"])
def test_prefill_index_scores(mode):
    _cuda()
    wl = synth.scaled(synth.WORKLOADS["prefill_chunk"], N=3077, T=203, P0=2874)
    inp = synth.make_inputs(wl, seed=9, mode=mode)
    dv = synth.to_device(inp)
    c, lay, rw = dv["cache"], dv["layers"][0], dv["rows"]
    s = S.index_scores(lay["q_idx"], lay["w"], c["k_idx"], c["k_scale"], rw["seq_of_row"], rw["n_visible"])
    s = s.cpu().numpy().astype(np.float64)
    rows = [0, 1, 7, 8, 100, 201, 202]
    ref = O.index_scores_rows(inp, 0, rows=rows)
    got = s[rows]
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin)
    if mode == "grid":
        assert np.array_equal(got[fin], ref[fin])
    else:
        bound = score_bound(inp, 0, rows)
        assert np.all(np.abs(got - ref)[fin] <= np.repeat(bound[:, None], got.shape[1], 1)[fin])
    # every row: -inf exactly from its causal boundary on
    nv = inp["rows"]["n_visible"]
    assert all(np.isfinite(s[r, :nv[r]]).all() and np.isneginf(s[r, nv[r]:]).all() for r in range(wl.T))


# ------------------------------------------------------------------ MXFP4 keys for prefill
def test_expand_mxfp4_bit_exact():
    _cuda()
    rng = np.random.default_rng(70)
    n = 5000
    codes = rng.integers(0, 256, (n, 64)).astype(np.uint8)
    exps = rng.integers(0, 255, (n, 4)).astype(np.uint8)
    exps[:6, 0] = [0, 1, 100, 127, 200, 254]
    got = S.expand_mxfp4(torch.from_numpy(codes).cuda(), torch.from_numpy(exps).cuda())
    torch.cuda.synchronize()
    ref = O.bf16_round(O.mxfp4_to_f64(codes, exps).astype(np.float32))
    assert np.array_equal(got.cpu().view(torch.int16).numpy().view(np.uint16), ref)


@pytest.mark.parametrize("mode", ["grid", "gauss"])
def test_prefill_index_scores_mxfp4(mode):
    """A prefill chunk with MXFP4 keys: the keys expanded once to their exact bf16 values, then
    the tensor-core prefill indexer, against the oracle's scores of the MXFP4 keys."""
    _cuda()
    wl = synth.scaled(synth.WORKLOADS["prefill_chunk"], N=3077, T=203, P0=2874, key_fmt="mxfp4")
    inp = synth.make_inputs(wl, seed=71, mode=mode)
    dv = synth.to_device(inp)
    c, lay, rw = dv["cache"], dv["layers"][0], dv["rows"]
    keys = S.expand_mxfp4(c["k_idx"], c["k_scale"])
    s = S.index_scores(lay["q_idx"], lay["w"], keys, None, rw["seq_of_row"], rw["n_visible"])
    s = s.cpu().numpy().astype(np.float64)
    rows = [0, 1, 7, 8, 100, 201, 202]
    ref = O.index_scores_rows(inp, 0, rows=rows)
    got = s[rows]
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin)
    if mode == "grid":
        assert np.array_equal(got[fin], ref[fin])
    else:
        bound = score_bound(inp, 0, rows)
        assert np.all(np.abs(got - ref)[fin] <= np.repeat(bound[:, None], got.shape[1], 1)[fin])


# ------------------------------------------------------------------ attention kernels
# tiles + merge; rows with 32 heads; rows with 16 heads; pipelined rows (bf16 only, else tiles)
@pytest.mark.parametrize("kernel", [1, 2, 3, 4])
@pytest.mark.parametrize("lat_fmt,group,swa_fmt", [("bf16", 32, "bf16"), ("fp4", 32, "fp8")])
def test_attention_kernels_agree_with_the_oracle(kernel, lat_fmt, group, swa_fmt):
    """Every attention kernel (a block per (row, tile) with a merge kernel; a block per (row,
    head group) carrying the softmax across the row's tiles, plain or with the tiles' copies
    pipelined) against the oracle, on rows where a later tile's logits exceed the first
    (window) tile's by far more than the row kernels' rescale threshold, so their running
    reference moves and the accumulated output is rescaled; -1 pads and a short row included."""
    _cuda()
    inp = small("batched_decode", seed=31, B=3, N=4000, lat_fmt=lat_fmt, lat_group=group, swa_fmt=swa_fmt)
    set_rows(inp, [4000, 3000, 100])
    rng = np.random.default_rng(9)
    K = 512
    idx = np.full((3, K), -1, np.int64)
    for r, nv in enumerate([4000, 3000, 100]):
        sel = np.sort(rng.choice(nv, min(K, nv) - 3, replace=False))
        idx[r, :len(sel)] = sel
    if lat_fmt == "bf16":
        # records aligned with some heads' query (rotary dims left out): logits near 20 against ~0.1
        q = O.bf16_to_f64(inp["layers"][0]["q"][0])  # row 0, [64, 512]
        for j, h in enumerate((0, 17, 40)):
            v = 23.0 * q[h] / np.linalg.norm(q[h])  # logit ~ 23 * 0.875 ~ 20 for head h
            v[448:] = 0.0
            inp["cache"]["lat"][0, idx[0, 100 + j]] = synth.bf16_bits(torch.from_numpy(v.astype(np.float32)))
    dv = synth.to_device(inp)
    c, lay, rw, p = dv["cache"], dv["layers"][0], dv["rows"], dv["params"]
    S.set_tuning(S.TUNE_ATTN_ROWS, kernel)
    try:
        out, sm = S.sparse_attn(lay["q"], rw["q_pos"], rw["seq_of_row"], c["lat"], c["lat_scales"],
                                torch.from_numpy(idx.astype(np.int32)).cuda(), lay["swa"], lay["swa_scale"],
                                rw["swa_pos0"], p["W"], lay["sink"], p["theta"], p["softmax_scale"])
        torch.cuda.synchronize()
    finally:
        S.reset_tuning()
    o_ref, sm_ref = O.sparse_attn_rows(inp, 0, idx)
    err = rel_err(out.cpu().numpy(), o_ref)
    assert err <= out_tol(inp["params"]), err
    assert np.max(np.abs(sm.cpu().numpy() - sm_ref)) < 1e-4


@pytest.mark.parametrize("L,K", [(70_001, 512), (60_001, 512), (36_864, 512), (20_001, 512), (9_000, 1024), (4_099, 37)])
def test_topk_many_long_rows(L, K):
    """More rows than SMs, each far longer than K (the prefill chunk's shape): the radix
    selection over rows in memory, bit-exact against the oracle, with ties (quarter-step
    integers), +-0, rows of every visible length (including at most K) and a candidate map.
    Row strides both 16-byte aligned and not; rows up to 65,536 entries place the kept entries
    through bitmaps, longer ones (70,001) by counting and writing passes."""
    _cuda()
    rows = 200
    sc = synth.integers((rows, L), 13, L % 89, -300, 300).float() / 4.0
    sc[1::4] = synth.normal((len(range(1, rows, 4)), L), 13, 2)  # no ties
    sc[2, ::2] = -0.0
    sc[2, 1::2] = 0.0
    rng = np.random.default_rng(L)
    n_valid = rng.integers(1, L + 1, rows).astype(np.int32)
    n_valid[:4] = [L, L - 1, K, 1]
    idx = S.topk(sc.cuda(), torch.from_numpy(n_valid).cuda(), K).cpu().numpy()
    ref = O.topk_rows(sc.numpy().astype(np.float64), n_valid, K)
    assert np.array_equal(idx, ref)
    cand = np.sort(rng.choice(10 ** 7, (rows, L), replace=True), axis=1).astype(np.int32) + np.arange(L, dtype=np.int32)
    idx_c = S.topk(sc.cuda(), torch.from_numpy(n_valid).cuda(), K, cand=torch.from_numpy(cand).cuda()).cpu().numpy()
    assert np.array_equal(idx_c, O.topk_rows(sc.numpy().astype(np.float64), n_valid, K, cand=cand))
