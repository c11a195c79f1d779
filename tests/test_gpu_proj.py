"""Parity of the projections around attention (low-rank query path, grouped low-rank output
projection) with the oracle, from tiny shapes with ragged token counts to the Flash shapes at
decode (32 tokens) and prefill (4096 tokens, sampled rows); and the attention's bf16 output,
the output projection's input.

Tolerance, from the arithmetic (bf16 keeps 8 significant bits: unit roundoff u = 2^-8): both
paths take bf16 inputs exactly; the kernels accumulate in fp32 (error far below what
follows), round the rank-sized intermediate (c * g_q, or y) to bf16 (relative error <= u per
element, spread about uniformly; summed over the next projection's K terms with random
weights it adds an error of standard deviation at most u / sqrt(3) of the output's RMS,
0.0023) and round the output to bf16 (<= u relative).  The bound checked per element is
u |ref| + 1.6e-2 RMS(ref): the output rounding plus seven standard deviations of the
intermediate's.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as O
import synth

pytestmark = pytest.mark.gpu

S = pytest.importorskip("sparse_attention_csa2_gb300")


def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _f(t):
    return t.float().cpu().numpy().astype(np.float64)


def _check(got, ref):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(ref ** 2))
    err = np.abs(got - ref)
    bound = 2.0 ** -8 * np.abs(ref) + 1.6e-2 * rms
    worst = float(np.max(err / bound))
    print(f"[worst {worst:.3f} of the bound]", end=" ")
    assert worst <= 1.0, f"worst error {worst:.3f} of the bound (max abs {err.max():.3e}, rms {rms:.3e})"
    return worst


def _query_ref(inp, rows, eps=1e-6):
    heads = inp["w_uq"].shape[0] // 512
    return O.query_proj(_f(inp["x"])[rows], _f(inp["w_dq"]), inp["g_q"].numpy(), _f(inp["w_uq"]),
                        inp["g_head"].numpy(), heads, eps)


def _run_query(inp, eps=1e-6, gains=True):
    d = {k: v.cuda() for k, v in inp.items()}
    q = S.query_proj(d["x"], d["w_dq"], d["w_uq"], d["g_q"] if gains else None, d["g_head"] if gains else None, eps)
    torch.cuda.synchronize()
    return q


# (tokens, hidden, q_rank, heads)
QUERY_SMALL = [(1, 256, 128, 1), (37, 512, 256, 2), (200, 1024, 512, 4), (300, 192, 384, 1)]


@pytest.mark.parametrize("T,hidden,q_rank,heads", QUERY_SMALL)
def test_query_proj_small(T, hidden, q_rank, heads):
    _cuda()
    shape = synth.ProjShape("t", tokens=T, hidden=hidden, q_rank=q_rank, heads=heads, groups=1, o_rank=128)
    inp = synth.projection_inputs(shape, seed=T + hidden)
    q = _run_query(inp)
    assert q.shape == (T, heads, 512) and q.dtype == torch.bfloat16
    _check(_f(q), _query_ref(inp, np.arange(T)))


def test_query_proj_without_gains_has_unit_head_rms():
    _cuda()
    shape = synth.ProjShape("t", tokens=50, hidden=512, q_rank=256, heads=3, groups=1, o_rank=128)
    inp = synth.projection_inputs(shape, seed=7)
    q = _f(_run_query(inp, eps=0.0, gains=False))
    ref = O.query_proj(_f(inp["x"]), _f(inp["w_dq"]), None, _f(inp["w_uq"]), None, 3, 0.0)
    _check(q, ref)
    assert np.allclose(np.sqrt(np.mean(q ** 2, -1)), 1.0, atol=4e-3)


@pytest.mark.parametrize("name", ["decode", "prefill"])
def test_query_proj_flash_shape(name):
    _cuda()
    shape = synth.PROJECTIONS[name]
    inp = synth.projection_inputs(shape, seed=3)
    q = _run_query(inp)
    T = shape.tokens
    rows = np.arange(T) if T <= 64 else np.array([0, 1, 127, 128, 255, 256, 1000, 2047, 3333, T - 1])
    _check(_f(q)[rows], _query_ref(inp, rows))


# (tokens, heads, groups, o_rank, hidden)
OUT_SMALL = [(5, 8, 2, 128, 256), (77, 8, 8, 256, 512), (260, 16, 4, 128, 384), (1, 4, 1, 128, 128)]


def _run_out(inp):
    d = {k: v.cuda() for k, v in inp.items()}
    out = S.out_proj(d["o"], d["w_oa"], d["w_ob"])
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("T,heads,groups,o_rank,hidden", OUT_SMALL)
def test_out_proj_small(T, heads, groups, o_rank, hidden):
    _cuda()
    shape = synth.ProjShape("t", tokens=T, hidden=hidden, q_rank=128, heads=heads, groups=groups, o_rank=o_rank)
    inp = synth.projection_inputs(shape, seed=T + heads)
    out = _run_out(inp)
    assert out.shape == (T, hidden) and out.dtype == torch.bfloat16
    _check(_f(out), O.out_proj(_f(inp["o"]), _f(inp["w_oa"]), _f(inp["w_ob"])))


@pytest.mark.parametrize("name", ["decode", "prefill"])
def test_out_proj_flash_shape(name):
    _cuda()
    shape = synth.PROJECTIONS[name]
    inp = synth.projection_inputs(shape, seed=4)
    out = _run_out(inp)
    T = shape.tokens
    rows = np.arange(T) if T <= 64 else np.array([0, 1, 127, 128, 255, 256, 1000, 2047, 3333, T - 1])
    _check(_f(out)[rows], O.out_proj(_f(inp["o"])[rows], _f(inp["w_oa"]), _f(inp["w_ob"])))


@pytest.mark.parametrize("ks", [1, 2, 8])
def test_split_counts_agree(ks):
    """The K split (a cluster reduction) changes only the fp32 summation order."""
    _cuda()
    shape = synth.ProjShape("t", tokens=32, hidden=1024, q_rank=256, heads=8, groups=8, o_rank=128)
    inp = synth.projection_inputs(shape, seed=12)
    S.set_tuning(S.TUNE_PROJ_KSPLIT, ks)
    try:
        out = _f(_run_out(inp))
        q = _f(_run_query(inp))
    finally:
        S.reset_tuning()
    _check(out, O.out_proj(_f(inp["o"]), _f(inp["w_oa"]), _f(inp["w_ob"])))
    _check(q, _query_ref(inp, np.arange(32)))


def test_attention_bf16_output_is_the_rounded_fp32_output():
    _cuda()
    inp = synth.make_inputs(synth.scaled(synth.WORKLOADS["batched_decode"], B=3, N=3000), seed=5)
    rng = np.random.default_rng(3)
    idx = np.stack([np.sort(rng.choice(3000, 512, replace=False)) for _ in range(3)]).astype(np.int32)
    dv = synth.to_device(inp)
    c, lay, rw, p = dv["cache"], dv["layers"][0], dv["rows"], dv["params"]
    args = (lay["q"], rw["q_pos"], rw["seq_of_row"], c["lat"], c["lat_scales"], torch.from_numpy(idx).cuda(),
            lay["swa"], lay["swa_scale"], rw["swa_pos0"], p["W"], lay["sink"], p["theta"], p["softmax_scale"])
    o32, _ = S.sparse_attn(*args)
    o16, _ = S.sparse_attn(*args, out_dtype=torch.bfloat16)
    assert o16.dtype == torch.bfloat16
    assert torch.equal(o32.to(torch.bfloat16), o16)
    # and the output projection takes it as it is
    w = synth.projection_inputs(synth.ProjShape("t", tokens=3), seed=8)
    out = S.out_proj(o16, w["w_oa"].cuda(), w["w_ob"].cuda())
    _check(_f(out), O.out_proj(_f(o16), _f(w["w_oa"]), _f(w["w_ob"])))
