"""Seeded synthetic inputs for the CSA2 attention step.

This package only draws random numbers and stores them in the cache formats the
step reads: bf16, OCP FP8 E4M3 with one fp32 scale per row, and FP4 E2M1 with
one E4M3 scale per group of 16 or 32 channels.  It holds none of the step's
arithmetic (no scoring, selection, attention or decoding of the formats), so
the CPU oracle and the CUDA library can both consume the bytes it returns
without sharing any code.

Every draw is reproducible from ``(seed, stream)``: large tensors are filled in
independent 4 Mi-element chunks, each from its own ``torch.Generator`` seeded by
``(seed, stream, chunk)``, so generation runs on all host cores and gives the
same bytes whatever the thread count.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

from .workloads import Workload, WORKLOADS, scaled, ProjShape, PROJECTIONS  # noqa: F401

_CHUNK = 1 << 22
_THREADS = max(1, min(16, os.cpu_count() or 1))


def _chunk_seed(seed: int, stream: int, chunk: int) -> int:
    return (seed * 1_000_003 + stream * 10_007 + chunk * 7_919 + 12_345) & 0x7FFF_FFFF_FFFF


def _fill(t: torch.Tensor, seed: int, stream: int, fn) -> torch.Tensor:
    flat = t.view(-1)
    n = flat.numel()
    nchunks = (n + _CHUNK - 1) // _CHUNK

    def work(c):
        g = torch.Generator().manual_seed(_chunk_seed(seed, stream, c))
        fn(flat[c * _CHUNK:min(n, (c + 1) * _CHUNK)], g)

    if nchunks <= 1:
        for c in range(nchunks):
            work(c)
    else:
        with ThreadPoolExecutor(_THREADS) as ex:
            list(ex.map(work, range(nchunks)))
    return t


def normal(shape, seed: int, stream: int, std: float = 1.0) -> torch.Tensor:
    """float32 N(0, std^2) samples."""
    t = torch.empty(shape, dtype=torch.float32)
    return _fill(t, seed, stream, lambda x, g: x.normal_(0.0, std, generator=g))


def uniform(shape, seed: int, stream: int, lo: float = 0.0, hi: float = 1.0) -> torch.Tensor:
    """float32 U[lo, hi) samples."""
    t = torch.empty(shape, dtype=torch.float32)
    return _fill(t, seed, stream, lambda x, g: x.uniform_(lo, hi, generator=g))


def integers(shape, seed: int, stream: int, lo: int, hi: int) -> torch.Tensor:
    """int32 samples uniform on the integers lo..hi (inclusive)."""
    t = torch.empty(shape, dtype=torch.int32)
    return _fill(t, seed, stream, lambda x, g: x.random_(lo, hi + 1, generator=g))


# ---------------------------------------------------------------- storage formats
def bf16_bits(x: torch.Tensor) -> np.ndarray:
    """Round float32 to bf16 (round to nearest even) and return the raw 16-bit patterns."""
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def e4m3_bits(x: torch.Tensor) -> np.ndarray:
    """Round float32 to OCP FP8 E4M3 (round to nearest even) and return the raw bytes.

    The caller keeps |x| <= 448; larger inputs would encode as NaN."""
    return x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def fp8_rows(x: torch.Tensor, unit_scale: bool = False):
    """Per-row FP8 encoding: scale = amax(row)/448 (1.0 when ``unit_scale``), codes = E4M3(x/scale)."""
    if unit_scale:
        scale = torch.ones(x.shape[:-1], dtype=torch.float32)
    else:
        amax = x.abs().amax(-1)
        scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    codes = e4m3_bits(x / scale.unsqueeze(-1))
    return codes, scale.numpy().astype(np.float32)


# The 127 non-negative finite E4M3 values in code order (codes 0x00..0x7E), decoded by torch.
_E4M3_POS = torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float32)
# Midpoints between consecutive E2M1 magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}.
_E2M1_MIDS = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], dtype=torch.float32)


def _fp4_encode_chunk(x: torch.Tensor, group: int):
    lead = x.shape[:-1]
    d = x.shape[-1]
    xg = x.reshape(*lead, d // group, group)
    amax = xg.abs().amax(-1)
    # scale code: the smallest E4M3 value >= amax/6, so no element clips.
    scode = torch.searchsorted(_E4M3_POS, (amax / 6.0).contiguous(), right=False).clamp_(max=126)
    sval = _E4M3_POS[scode]
    q = torch.where(sval.unsqueeze(-1) > 0, xg / sval.unsqueeze(-1).clamp(min=1e-30), torch.zeros_like(xg))
    mag = q.abs().contiguous()
    idx = torch.searchsorted(_E2M1_MIDS, mag, right=False)
    tie = (idx < 7) & (mag == _E2M1_MIDS[idx.clamp(max=6)])
    idx = torch.where(tie & (idx % 2 == 1), idx + 1, idx)  # ties go to the even code
    code = (idx | torch.where(q < 0, 8, 0)).to(torch.uint8).reshape(*lead, d)
    packed = (code[..., 0::2] | (code[..., 1::2] << 4)).to(torch.uint8)  # low nibble = even channel
    return packed.numpy(), scode.to(torch.uint8).numpy()


def _e2m1_codes(q: torch.Tensor) -> torch.Tensor:
    """E2M1 code of each value: nearest level, ties to the even code, saturating at 6."""
    mag = q.abs().contiguous()
    idx = torch.searchsorted(_E2M1_MIDS, mag, right=False)
    tie = (idx < 7) & (mag == _E2M1_MIDS[idx.clamp(max=6)])
    idx = torch.where(tie & (idx % 2 == 1), idx + 1, idx)
    return idx | torch.where(q < 0, 8, 0)


def mxfp4_blocks(x: torch.Tensor):
    """OCP MXFP4 encoding of float32 rows [..., D]: per block of 32 the shared UE8M0 scale
    2^(floor(log2 amax) - 2) (2 = the exponent of E2M1's largest value, 6 = 1.5 * 2^2; an
    all-zero block takes 2^-127), each element the nearest E2M1 level of x / scale, ties to
    the even code, saturating at 6.  Returns (codes [..., D/2] low nibble = even element,
    biased exponents [..., D/32] uint8)."""
    lead, d = x.shape[:-1], x.shape[-1]
    xb = x.reshape(*lead, d // 32, 32)
    amax = xb.abs().amax(-1)
    e = torch.where(amax > 0, torch.floor(torch.log2(amax.clamp(min=1e-38))) - 2, torch.full_like(amax, -127.0))
    e = e.clamp(-127, 127)
    q = xb / torch.exp2(e).unsqueeze(-1)
    code = _e2m1_codes(q).to(torch.uint8).reshape(*lead, d)
    packed = (code[..., 0::2] | (code[..., 1::2] << 4)).to(torch.uint8)
    return packed.numpy(), (e + 127).to(torch.uint8).numpy()


def mxfp4_round_trip(x: torch.Tensor) -> torch.Tensor:
    """The values of x's MXFP4 encoding, as float32 (exact)."""
    codes, exps = mxfp4_blocks(x)
    c = torch.from_numpy(codes).to(torch.int64)
    lv = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    def dec(n):
        m = lv[n & 7]
        return torch.where((n & 8) != 0, -m, m)
    vals = torch.stack([dec(c & 0xF), dec(c >> 4)], -1).reshape(*x.shape)
    sc = torch.exp2(torch.from_numpy(exps).to(torch.float32) - 127.0)
    return vals * sc.repeat_interleave(32, -1)


def fp4_groups(x: torch.Tensor, group: int):
    """FP4 encoding: E2M1 codes (two per byte, low nibble = even channel) and one E4M3
    scale code per ``group`` channels.  The scale is the smallest E4M3 value >= amax/6;
    each value rounds to the nearest E2M1 level, ties to the even code."""
    lead = x.shape[:-1]
    d = x.shape[-1]
    rows = x.reshape(-1, d)
    n = rows.shape[0]
    codes = np.empty((n, d // 2), np.uint8)
    scales = np.empty((n, d // group), np.uint8)
    step = max(1, _CHUNK // d)

    def work(r0):
        c, s = _fp4_encode_chunk(rows[r0:r0 + step], group)
        codes[r0:r0 + step] = c
        scales[r0:r0 + step] = s

    with ThreadPoolExecutor(_THREADS) as ex:
        list(ex.map(work, range(0, n, step)))
    return codes.reshape(*lead, d // 2), scales.reshape(*lead, d // group)


# ---------------------------------------------------------------- input bundles
def _stream(base: int, layer: int, k: int) -> int:
    return base + 100 * layer + k


def make_inputs(wl: Workload, seed: int, mode: str = "gauss") -> dict:
    """Build one seeded input bundle for ``wl``.

    ``mode='gauss'`` draws the distributions of the workload recipe; ``mode='grid'``
    draws indexer queries and keys on the integers [-4, 4] and indexer weights on
    {0, 1/16, ..., 1}, so every indexer score is exactly representable in fp32.

    Returns a dict with keys ``params``, ``rows``, ``cache`` and ``layers`` (a list,
    one entry per layer).  Arrays are numpy, in the storage formats.
    """
    assert mode in ("gauss", "grid")
    B, N, Bq = wl.B, wl.N, wl.Bq
    H, D, HI, DI, W = wl.H, wl.D, wl.HI, wl.DI, wl.W

    # ---- query rows: which sequence, which position, how many visible records
    if wl.T > 0:
        t = np.arange(wl.T, dtype=np.int64)
        q_pos = wl.P0 + t
        n_visible = (wl.P0 + t + 1).astype(np.int32)
        seq_of_row = np.zeros(wl.T, np.int32)
        wrows = wl.T + W - 1
        swa_pos0 = np.full(B, wl.P0 - W + 1, np.int64)
    else:
        q_pos = np.full(Bq, wl.q_pos, np.int64)
        n_visible = np.full(Bq, wl.N, np.int32)
        seq_of_row = np.arange(Bq, dtype=np.int32) % B
        wrows = W
        swa_pos0 = np.full(B, wl.q_pos - W + 1, np.int64)
    swa_pos0 = np.maximum(swa_pos0, 0)
    rows = dict(q_pos=q_pos, n_visible=n_visible, seq_of_row=seq_of_row, swa_pos0=swa_pos0, swa_rows=wrows)

    n_layers = wl.n_layers
    # ---- indexer queries (per layer that indexes) and weights
    layers = []
    q_idx0 = None
    for l in range(n_layers):
        lay = {}
        if wl.layer_mode(l) != "reuse":
            if mode == "grid":
                qi = integers((Bq, HI, DI), seed, _stream(10, l, 0), -4, 4).to(torch.float32)
                w = integers((Bq, HI), seed, _stream(10, l, 1), 0, 16).to(torch.float32) / 16.0
            else:
                qi = normal((Bq, HI, DI), seed, _stream(10, l, 0))
                if l > 0 and q_idx0 is not None:
                    qi = 0.7 * q_idx0 + 0.3 * qi  # later indexers correlated with the first
                w = uniform((Bq, HI), seed, _stream(10, l, 1))
            if l == 0:
                q_idx0 = qi
            if wl.key_fmt == "mxfp4":
                qi = mxfp4_round_trip(qi)  # the pages' MXFP4 indexer queries, exact in bf16
            lay["q_idx"] = bf16_bits(qi)
            lay["w"] = w.numpy().astype(np.float32)
        q = normal((Bq, H, D), seed, _stream(10, l, 2))
        lay["q"] = bf16_bits(q)
        swa = normal((B, wrows, D), seed, _stream(10, l, 3), std=D ** -0.5)
        if wl.swa_fmt == "bf16":
            lay["swa"] = bf16_bits(swa)
            lay["swa_scale"] = None
        else:
            lay["swa"], lay["swa_scale"] = fp8_rows(swa)
        lay["sink"] = normal((H,), seed, _stream(10, l, 4)).numpy().astype(np.float32)
        lay["mode"] = wl.layer_mode(l)
        layers.append(lay)

    # ---- shared indexer keys
    if mode == "grid":
        k = integers((B, N, DI), seed, 1, -4, 4).to(torch.float32)
    else:
        k = normal((B, N, DI), seed, 1)
        if wl.n_hot_blocks > 0:
            nb = (N + wl.block_size - 1) // wl.block_size
            # for every sequence: hot blocks get half the mean first-layer indexer query added
            hot = integers((B, wl.n_hot_blocks), seed, 2, 0, nb - 1).numpy()
            qmean = q_idx0[:B].mean(1)  # [B, DI]: row b is the first query row of sequence b
            for b in range(B):
                for c in np.unique(hot[b]):
                    k[b, c * wl.block_size:(c + 1) * wl.block_size] += 0.5 * qmean[b]
    if wl.key_fmt == "bf16":
        cache = dict(k_idx=bf16_bits(k), k_scale=None)
    elif wl.key_fmt == "mxfp4":
        codes, exps = mxfp4_blocks(k)
        cache = dict(k_idx=codes, k_scale=exps)
    else:
        codes, scale = fp8_rows(k, unit_scale=(mode == "grid"))
        cache = dict(k_idx=codes, k_scale=scale)
    del k

    # ---- shared latents (one 512-d latent per record: key and value at once)
    lat = normal((B, N, D), seed, 3, std=D ** -0.5)
    if wl.lat_fmt == "bf16":
        cache["lat"] = bf16_bits(lat)
        cache["lat_scales"] = None
    else:
        cache["lat"], cache["lat_scales"] = fp4_groups(lat, wl.lat_group)
    del lat

    params = dict(H=H, D=D, R=wl.R, HI=HI, DI=DI, K=wl.K, W=W, theta=wl.theta,
                  softmax_scale=D ** -0.5, key_fmt=wl.key_fmt, lat_fmt=wl.lat_fmt,
                  lat_group=wl.lat_group, swa_fmt=wl.swa_fmt, block_size=wl.block_size,
                  n_keep=wl.n_keep, B=B, N=N, Bq=Bq, mode=mode, seed=seed, name=wl.name)
    return dict(params=params, rows=rows, cache=cache, layers=layers)


# ---------------------------------------------------------------- device transfer
def _t(a, device):
    if a is None:
        return None
    if isinstance(a, np.ndarray):
        if a.dtype == np.uint16:  # bf16 bit patterns
            t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
        else:
            t = torch.from_numpy(np.ascontiguousarray(a))
        return t.to(device, non_blocking=False)
    return a


def to_device(inp: dict, device="cuda") -> dict:
    """The same bundle with every array as a torch tensor on ``device`` (bf16 bit patterns
    become torch.bfloat16; E4M3 / E2M1 codes stay uint8)."""
    out = {"params": dict(inp["params"])}
    out["rows"] = {k: (_t(v, device) if isinstance(v, np.ndarray) else v) for k, v in inp["rows"].items()}
    out["cache"] = {k: _t(v, device) for k, v in inp["cache"].items()}
    out["layers"] = [{k: (_t(v, device) if isinstance(v, np.ndarray) else v) for k, v in lay.items()}
                     for lay in inp["layers"]]
    return out


# ---------------------------------------------------------------- projections
def projection_inputs(shape, seed: int) -> dict:
    """Hidden states, attention outputs and random-init weights (N(0, 1/fan_in)) for the
    projections around attention, all bf16 tensors on the host, gains float32 near 1."""
    s = shape
    hd = s.heads * s.head_dim

    def bf(sh, stream, std):
        return normal(sh, seed, stream, std).to(torch.bfloat16)

    return {
        "x": bf((s.tokens, s.hidden), 1, 1.0),
        "w_dq": bf((s.q_rank, s.hidden), 2, s.hidden ** -0.5),
        "g_q": 1.0 + 0.1 * normal((s.q_rank,), seed, 3),
        "w_uq": bf((hd, s.q_rank), 4, s.q_rank ** -0.5),
        "g_head": 1.0 + 0.1 * normal((s.head_dim,), seed, 5),
        "o": bf((s.tokens, s.heads, s.head_dim), 6, 0.1),
        "w_oa": bf((s.groups, s.o_rank, hd // s.groups), 7, (hd // s.groups) ** -0.5),
        "w_ob": bf((s.hidden, s.groups * s.o_rank), 8, (s.groups * s.o_rank) ** -0.5),
    }
