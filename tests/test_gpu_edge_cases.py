"""Edge cases of the fused decode step against the oracle.

Segment counts: with one block per SM the scan splits a row into min(SMs / rows, N / 4096)
segments, so the batch size chooses the selection path: a cluster of 16 segments (B=2), of
9 (B=16), or more segments than a cluster holds, which write lists merged afterwards (B=5).
Short rows: rows with fewer visible records than K (every candidate kept, -1 padding), one
record, exactly K, K + 1, and a query whose window starts at position 0.
Grid-mode inputs make every indexer score exact, so the indices must be bit-identical.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as O
import synth
from csa2_testlib import gpu_group, out_tol, rel_err, set_rows

pytestmark = pytest.mark.gpu


def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def _check(inp, g, rows):
    ref = O.csa2_layer(inp, 0, None, rows)
    gi = g[0].idx.cpu().numpy()[rows]
    assert np.array_equal(gi, ref["idx"])
    assert rel_err(g[0].out.cpu().numpy()[rows], ref["o"]) <= out_tol(inp["params"])


@pytest.mark.parametrize("B", [2, 5, 16])
def test_segment_counts(B):
    _cuda()
    wl = synth.scaled(synth.WORKLOADS["batched_decode"], B=B, N=65536)
    inp = synth.make_inputs(wl, seed=20 + B, mode="grid")
    g = gpu_group(synth.to_device(inp))
    _check(inp, g, sorted({0, B // 2, B - 1}))


@pytest.mark.parametrize("key_fmt,lat_fmt,swa_fmt", [("bf16", "bf16", "bf16"), ("fp8", "fp4", "fp8")])
def test_short_rows(key_fmt, lat_fmt, swa_fmt):
    _cuda()
    wl = synth.scaled(synth.WORKLOADS["batched_decode"], B=7, N=20000, key_fmt=key_fmt, lat_fmt=lat_fmt,
                      swa_fmt=swa_fmt)
    inp = synth.make_inputs(wl, seed=31, mode="grid")
    K = inp["params"]["K"]
    set_rows(inp, [1, 100, K - 1, K, K + 1, 3 * K + 17, 20000])
    g = gpu_group(synth.to_device(inp))
    rows = list(range(7))
    _check(inp, g, rows)
    gi = g[0].idx.cpu().numpy()
    nv = inp["rows"]["n_visible"]
    for r in rows:
        kept = gi[r][gi[r] >= 0]
        assert len(kept) == min(K, int(nv[r]))
        assert np.all(np.diff(kept) > 0) and np.all(gi[r][len(kept):] == -1)


@pytest.mark.parametrize("B", [2, 5])
def test_segment_counts_without_clusters(B):
    """The same rows with the scan's cluster selection switched off: the segments write lists
    and the last segment of each row to finish merges them."""
    _cuda()
    import sparse_attention_csa2_gb300 as S
    wl = synth.scaled(synth.WORKLOADS["batched_decode"], B=B, N=65536)
    inp = synth.make_inputs(wl, seed=40 + B, mode="grid")
    S.set_tuning(S.TUNE_SCAN_CLUSTER, 0)
    try:
        g = gpu_group(synth.to_device(inp))
    finally:
        S.reset_tuning()
    _check(inp, g, sorted({0, B - 1}))
