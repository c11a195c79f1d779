"""Record-range split of one sequence's records (the multi-device decode of a long context),
run on one GPU: every range in turn through the library's split calls (range scores, range
candidates, merge, range attention partials, partial merge), against the oracle on the whole
sequence.  Grid-mode inputs make every score exact, so the merged indices must equal the
oracle's exactly; Gaussian inputs allow only near-tie swaps at the K-boundary.  Outputs:
within 1e-2 x RMS (FP8 / FP4 caches) of the oracle's attention over the merged selection.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from csa2_testlib import check_idx_near_ties, rel_err, score_bound, set_rows

pytestmark = pytest.mark.gpu

S = pytest.importorskip("sparse_attention_csa2_gb300")


def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _shards(dv, ranges):
    """Range k's local inputs: its slice of the keys and latents, the full query side."""
    p, rw, c, lay = dv["params"], dv["rows"], dv["cache"], dv["layers"][0]
    common = dict(q_idx=lay["q_idx"], w=lay["w"], q=lay["q"], q_pos=rw["q_pos"], seq_of_row=rw["seq_of_row"],
                  n_visible=rw["n_visible"], swa=lay["swa"], swa_scale=lay["swa_scale"], swa_pos0=rw["swa_pos0"],
                  window=p["W"], sink=lay["sink"], theta=p["theta"], softmax_scale=p["softmax_scale"])
    out = []
    for first, count in ranges:
        sl = slice(first, first + count)
        local = dict(common)
        local["k_idx"] = c["k_idx"][:, sl].contiguous()
        local["k_scale"] = None if c["k_scale"] is None else c["k_scale"][:, sl].contiguous()
        local["lat"] = c["lat"][:, sl].contiguous()
        local["lat_scale"] = None if c["lat_scales"] is None else c["lat_scales"][:, sl].contiguous()
        out.append(local)
    return out


@pytest.mark.parametrize("parts", [2, 3, 5])
@pytest.mark.parametrize("mode", ["grid", "gauss"])
def test_split_layer_matches_the_oracle(parts, mode):
    _cuda()
    from sparse_attention_csa2_gb300.shard import emulate_split, record_ranges
    N = 30011
    wl = synth.scaled(synth.WORKLOADS["long_decode"], B=3, N=N)
    inp = synth.make_inputs(wl, seed=50 + parts, mode=mode)
    # ragged visibility: a row seeing fewer records than one range holds, one seeing all
    set_rows(inp, [N, 17_003, 4_321])
    dv = synth.to_device(inp)
    ranges = record_ranges(N, parts)
    idx, out, sm = emulate_split(_shards(dv, ranges), ranges, inp["params"]["K"])
    torch.cuda.synchronize()
    ref = O.csa2_layer(inp, 0)
    gi = idx.cpu().numpy()
    if mode == "grid":
        assert np.array_equal(gi, ref["idx"])
    else:
        assert check_idx_near_ties(gi, ref["idx"], ref["scores"], score_bound(inp, 0)) == 0
    o_ref, sm_ref = O.sparse_attn_rows(inp, 0, gi.astype(np.int64))
    assert rel_err(out.cpu().numpy(), o_ref) <= 1e-2
    assert np.max(np.abs(sm.cpu().numpy() - sm_ref)) < 1e-4


def test_split_indices_equal_the_unsplit_layer():
    """The merged selection of a 4-way split equals the fused FULL layer's on the same inputs
    (grid mode: exact scores on both paths)."""
    _cuda()
    from csa2_testlib import gpu_group
    from sparse_attention_csa2_gb300.shard import emulate_split, record_ranges
    N = 24_000
    wl = synth.scaled(synth.WORKLOADS["long_decode"], B=2, N=N)
    inp = synth.make_inputs(wl, seed=61, mode="grid")
    dv = synth.to_device(inp)
    ranges = record_ranges(N, 4)
    idx, out, _ = emulate_split(_shards(dv, ranges), ranges, inp["params"]["K"])
    g = gpu_group(dv)
    assert torch.equal(idx, g[0].idx)
    ref = g[0].out.cpu().numpy().astype(np.float64)
    assert rel_err(out.cpu().numpy(), ref) <= 1e-2
