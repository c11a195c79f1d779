"""The encoder's CSA2 memory path on the GPU against the oracle: token pairs pooled by the
compressor (ratio 2), written as bf16 latent rows rotated at each entry's position, indexer
keys derived from the entries by a plain projection, and a decode query reading that memory
under the encoder's causal rule (an entry is visible once its last token is: (p + 1) // 2
entries).  Each stage is compared with the oracle's own stage; the decode stage runs the
fused CSA2 layer on the oracle-built memory.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as O
import synth
from csa2_testlib import check_idx_near_ties, gpu_group, out_tol, rel_err, score_bound

pytestmark = pytest.mark.gpu

S = pytest.importorskip("sparse_attention_csa2_gb300")

U = 2.0 ** -8  # bf16 unit roundoff


def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _bf16_bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("x_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rotate", [True, False])
def test_writer_bf16_rows_bit_exact(x_dtype, rotate):
    _cuda()
    rng = np.random.default_rng(60)
    n, rows = 3000, 5000
    x = (rng.standard_normal((n, 512)) * np.exp2(rng.integers(-8, 8, (n, 1)))).astype(np.float32)
    pos = rng.integers(0, 2_000_000, n).astype(np.int64)
    dst = rng.permutation(rows)[:n].astype(np.int64)
    xt = torch.from_numpy(x)
    if x_dtype == "bf16":
        xt = xt.to(torch.bfloat16)
        x = xt.float().numpy()
    cache = torch.full((rows, 512), 0x7FC1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    S.write_records(xt.cuda(), torch.from_numpy(dst).cuda(), cache, None, S.BF16,
                    pos=torch.from_numpy(pos).cuda() if rotate else None)
    torch.cuda.synchronize()
    ref, _ = O.write_records(x, pos if rotate else None, 10000.0, "bf16")
    got = _bf16_bits(cache)
    assert np.array_equal(got[dst], ref)
    untouched = np.setdiff1d(np.arange(rows), dst)
    assert np.all(got[untouched] == 0x7FC1)


@pytest.mark.parametrize("T,k_in,k_out", [(1, 64, 128), (37, 512, 128), (300, 512, 256), (4096, 1024, 512)])
def test_linear(T, k_in, k_out):
    _cuda()
    g = torch.Generator().manual_seed(T + k_in)
    x = torch.randn(T, k_in, generator=g).to(torch.bfloat16)
    w = (torch.randn(k_out, k_in, generator=g) / k_in ** 0.5).to(torch.bfloat16)
    out = S.linear(x.cuda(), w.cuda())
    torch.cuda.synchronize()
    ref = O.linear(x.float().numpy(), w.float().numpy())
    got = out.float().cpu().numpy().astype(np.float64)
    rms = np.sqrt(np.mean(ref ** 2))
    # one rounding to bf16 of an fp32 sum
    assert np.all(np.abs(got - ref) <= U * np.abs(ref) + 1e-4 * rms)


def _tokens(n_seq, T, seed):
    rng = np.random.default_rng(seed)
    kv = rng.standard_normal((n_seq, T, 512)).astype(np.float32)
    gate = (2.0 * rng.standard_normal((n_seq, T, 512))).astype(np.float32)
    w_ik = (rng.standard_normal((128, 512)) / np.sqrt(512)).astype(np.float32)
    w_ik = torch.from_numpy(w_ik).to(torch.bfloat16).float().numpy()  # weights are bf16 values
    return kv, gate, w_ik


def test_encoder_memory_chain():
    """compress -> bf16 rotated latents and unrotated entries -> keys, all on the GPU, against
    the oracle's chain: the GPU's float32 entries differ from the oracle's float64 ones by a
    few float32 ulps, which can move a bf16 rounding by one step."""
    _cuda()
    T = 20001
    kv, gate, w_ik = _tokens(1, T, 61)
    ref = O.encoder_memory(kv[0], gate[0], 2, w_ik)
    n = T // 2
    entries = S.compress(torch.from_numpy(kv[0]).cuda(), torch.from_numpy(gate[0]).cuda(), 2)
    pos = torch.arange(n, dtype=torch.int64, device="cuda") * 2 + 1
    rows = torch.arange(n, dtype=torch.int64, device="cuda")
    lat = torch.empty((n, 512), dtype=torch.bfloat16, device="cuda")
    plain = torch.empty((n, 512), dtype=torch.bfloat16, device="cuda")
    S.write_records(entries, rows, lat, None, S.BF16, pos=pos)
    S.write_records(entries, rows, plain, None, S.BF16)
    keys = S.linear(plain, torch.from_numpy(w_ik).to(torch.bfloat16).cuda())
    torch.cuda.synchronize()
    e_ref = ref["entries"].astype(np.float64)
    assert np.max(np.abs(entries.cpu().numpy() - e_ref)) <= 1e-5 * np.max(np.abs(e_ref))
    lr = O.bf16_to_f64(ref["lat"])
    assert np.all(np.abs(lat.float().cpu().numpy() - lr) <= 2 * U * np.abs(lr) + 1e-6)
    # keys: a one-step flip of the unrotated bf16 entry (entries near a bf16 rounding
    # boundary, about 2.6e-4 of them for a 1e-6 relative float32 difference) moves a key by at
    # most |w| 2^-7 |e| (<= 0.22 x 0.031 here, about 8e-3 of the keys' RMS); a key takes 0.13
    # such flips on average, so: within one bf16 step of the oracle's for almost all, and
    # within one step plus two worst-case flips for every one
    kr = O.bf16_to_f64(ref["k_idx"])
    rms = np.sqrt(np.mean(kr ** 2))
    d = np.abs(keys.float().cpu().numpy() - kr)
    assert np.mean(d <= 2 * U * np.abs(kr)) >= 0.99
    assert np.all(d <= 2 * U * np.abs(kr) + 2e-2 * rms)


def test_encoder_decode_over_compressed_memory():
    """A decode query at token position p of each sequence over the oracle-built encoder
    memory, with the encoder's causal rule (n_visible = (p + 1) // 2) and the token-level
    window: the fused CSA2 layer against the oracle layer."""
    _cuda()
    B, N = 4, 5000
    T = 2 * N
    wl = synth.scaled(synth.WORKLOADS["batched_decode"], B=B, N=N)
    inp = synth.make_inputs(wl, seed=62)
    kv, gate, w_ik = _tokens(B, T, 63)
    lat = np.empty((B, N, 512), np.uint16)
    keys = np.empty((B, N, 128), np.uint16)
    for b in range(B):
        m = O.encoder_memory(kv[b], gate[b], 2, w_ik)
        lat[b], keys[b] = m["lat"], m["k_idx"]
    inp["cache"]["lat"], inp["cache"]["k_idx"] = lat, keys
    # queries at the last token (every entry visible), one before it (the last entry holds a
    # future token), and odd / even positions inside the sequence
    q_pos = np.array([T - 1, T - 2, 3001, 3000], np.int64)
    n_vis = O.visible_entries(q_pos, 2).astype(np.int32)
    assert list(n_vis) == [N, N - 1, 1501, 1500]
    rows = inp["rows"]
    rows["n_visible"], rows["q_pos"] = n_vis, q_pos
    rows["swa_pos0"] = np.maximum(q_pos - inp["params"]["W"] + 1, 0)
    ref = O.csa2_layer(inp, 0, None, list(range(B)))
    g = gpu_group(synth.to_device(inp))[0]
    gi = g.idx.cpu().numpy()
    assert all(gi[r][gi[r] >= 0].max() < n_vis[r] for r in range(B))  # nothing beyond the causal rule
    scores = O.index_scores_rows(inp, 0)
    swaps = check_idx_near_ties(gi, ref["idx"], scores, score_bound(inp, 0))
    assert swaps == 0
    assert rel_err(g.out.cpu().numpy(), ref["o"]) <= out_tol(inp["params"])
