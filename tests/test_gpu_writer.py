"""Parity of the cache writer (rotation by position, then FP4 group or FP8 row quantization)
with the oracle's writer: codes and scales byte for byte (a zero code's sign aside, both
encodings reading as 0), rows written at their destinations and no others, and an
out-of-range destination skipped and reported."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as O

pytestmark = pytest.mark.gpu

S = pytest.importorskip("sparse_attention_csa2_gb300")

CACHE_ROWS = 5000


def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _records(n, seed):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((n, 512)) * np.exp2(rng.integers(-10, 10, (n, 1)))).astype(np.float32)
    x[0] = 0.0                                    # all-zero record
    x[1, :] = 1e-30                               # below every E4M3 scale
    x[2, :16] = [6.0, 3.2, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -5.0, 4.0, 0.0, -0.0, 1.5, -6.0]
    x[3] *= 1e6                                   # group scales saturate at 448, values clip at 6 x 448
    x[4, ::2] = -x[4, 1::2]
    pos = rng.integers(0, 2_000_000, n).astype(np.int64)
    pos[:3] = [0, 1, 1_048_575]
    dst = rng.permutation(CACHE_ROWS)[:n].astype(np.int64)
    return x, pos, dst


def _zero_sign_free_fp4(c):
    lo, hi = c & 0xF, c >> 4
    lo = np.where(lo == 8, 0, lo)
    hi = np.where(hi == 8, 0, hi)
    return (lo | (hi << 4)).astype(np.uint8)


@pytest.mark.parametrize("fmt,group", [("fp4", 16), ("fp4", 32), ("fp8", 0)])
@pytest.mark.parametrize("x_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rotate", [True, False])
def test_writer_matches_oracle(fmt, group, x_dtype, rotate):
    _cuda()
    n = 1500
    x, pos, dst = _records(n, seed=3 + group)
    xt = torch.from_numpy(x)
    if x_dtype == "bf16":
        xt = xt.to(torch.bfloat16)
        x = xt.to(torch.float32).numpy()  # the values the writer sees
    dev = "cuda"
    if fmt == "fp4":
        codes = torch.full((CACHE_ROWS, 256), 0xAA, dtype=torch.uint8, device=dev)
        scales = torch.full((CACHE_ROWS, 512 // group), 0xAA, dtype=torch.uint8, device=dev)
        out_dtype = S.FP4_E2M1_G16 if group == 16 else S.FP4_E2M1_G32
    else:
        codes = torch.full((CACHE_ROWS, 512), 0xAA, dtype=torch.uint8, device=dev)
        scales = torch.full((CACHE_ROWS,), -7.0, dtype=torch.float32, device=dev)
        out_dtype = S.FP8_E4M3_ROWSCALE
    S.write_records(xt.to(dev), torch.from_numpy(dst).to(dev), codes, scales, out_dtype,
                    pos=torch.from_numpy(pos).to(dev) if rotate else None, theta=10000.0)
    torch.cuda.synchronize()
    rc, rs = O.write_records(x, pos if rotate else None, 10000.0, fmt, group or 16)
    gc, gs = codes.cpu().numpy(), scales.cpu().numpy()
    if fmt == "fp4":
        assert np.array_equal(_zero_sign_free_fp4(gc[dst]), _zero_sign_free_fp4(rc))
        assert np.array_equal(gs[dst], rs)
    else:
        assert np.array_equal(np.where(gc[dst] == 0x80, 0, gc[dst]), np.where(rc == 0x80, 0, rc))
        assert np.array_equal(gs[dst], rs)
    # rows not written keep their contents
    untouched = np.setdiff1d(np.arange(CACHE_ROWS), dst)
    assert np.all(gc[untouched] == 0xAA)
    if fmt == "fp8":
        assert np.all(gs[untouched] == -7.0)
    else:
        assert np.all(gs[untouched] == 0xAA)
    # the cache reads back the rotated records within the format's rounding
    xr = O.rotate_f32(x, pos, 10000.0) if rotate else x
    if fmt == "fp4":
        deq = O.fp4_to_f64(gc[dst], gs[dst], group)
        step = np.repeat(O.e4m3_to_f64(gs[dst]), group, -1)
        ok = np.abs(deq - xr) <= step + 1e-30
        ok[3] = True  # the saturated record clips by design
        assert ok.all()
    else:
        deq = O.fp8_rows_to_f64(gc[dst], gs[dst])
        assert np.all(np.abs(deq - xr) <= np.abs(xr) * 2.0 ** -4 + gs[dst][:, None] * 2.0 ** -10)


def test_writer_skips_and_reports_out_of_range_rows():
    _cuda()
    x, pos, dst = _records(8, seed=9)
    dst[5] = CACHE_ROWS  # out of range
    dev = "cuda"
    codes = torch.zeros((CACHE_ROWS, 256), dtype=torch.uint8, device=dev)
    scales = torch.zeros((CACHE_ROWS, 32), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    S.write_records(torch.from_numpy(x).to(dev), torch.from_numpy(dst).to(dev), codes, scales, S.FP4_E2M1_G16,
                    pos=torch.from_numpy(pos).to(dev), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 6  # CSA2_EDEVICE_INDEX
    rc, rs = O.write_records(x, pos, 10000.0, "fp4", 16)
    ok = np.arange(8) != 5
    assert np.array_equal(_zero_sign_free_fp4(codes.cpu().numpy()[dst[ok]]), _zero_sign_free_fp4(rc[ok]))


# ------------------------------------------------------------------ compressor
@pytest.mark.parametrize("ratio", [1, 2, 4, 8])
@pytest.mark.parametrize("x_dtype", ["f32", "bf16"])
def test_compressor_matches_oracle(ratio, x_dtype):
    _cuda()
    rng = np.random.default_rng(50 + ratio)
    T = 1000 * ratio + ratio - 1  # an incomplete last group: no entry
    kv = rng.standard_normal((T, 512)).astype(np.float32)
    gate = (rng.standard_normal((T, 512)) * 4).astype(np.float32)
    gate[0, :8] = 80.0  # a saturated gate: its token takes the whole weight of those channels
    kt, gt = torch.from_numpy(kv), torch.from_numpy(gate)
    if x_dtype == "bf16":
        kt, gt = kt.to(torch.bfloat16), gt.to(torch.bfloat16)
        kv, gate = kt.to(torch.float32).numpy(), gt.to(torch.float32).numpy()
    out = S.compress(kt.cuda(), gt.cuda(), ratio)
    torch.cuda.synchronize()
    ref = O.compress(kv, gate, ratio)
    got = out.cpu().numpy().astype(np.float64)
    assert got.shape == ref.shape == (T // ratio, 512)
    # fp32 softmax weights: error a few ulps of the largest token value
    assert np.max(np.abs(got - ref)) <= 1e-5 * np.max(np.abs(kv))
