"""Failure paths on the GPU, made to happen without faulting anything.

* A bounded device wait that runs out: the library's self-test waits on an mbarrier that
  nothing signals, through the same wait and reporting the tensor-core kernels use, with a
  short limit; the status word must read CSA2_ETIMEOUT and the context must stay usable.
* Out-of-range selected indices made on the host: attention skips them, reports
  CSA2_EDEVICE_INDEX, and its output equals the oracle's over the remaining entries.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from csa2_testlib import out_tol, rel_err, set_rows

pytestmark = pytest.mark.gpu

S = pytest.importorskip("sparse_attention_csa2_gb300")


def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_bounded_wait_times_out_and_reports():
    _cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    S.selftest_wait_timeout(status, tries=1000)
    assert S.read_device_status(status) == S.ETIMEOUT
    # the context is still usable: a normal call afterwards runs and is exact
    sc = synth.normal((2, 3001), 3, 1)
    nv = np.array([3001, 17], np.int32)
    idx = S.topk(sc.cuda(), torch.from_numpy(nv).cuda(), 64).cpu().numpy()
    assert np.array_equal(idx, O.topk_rows(sc.numpy().astype(np.float64), nv, 64))


def test_out_of_range_indices_are_skipped_and_reported():
    _cuda()
    N = 4000
    inp = synth.make_inputs(synth.scaled(synth.WORKLOADS["batched_decode"], B=2, N=N), seed=13)
    set_rows(inp, [N, 2500])
    rng = np.random.default_rng(5)
    K = 512
    idx = np.stack([np.sort(rng.choice(2500, K, replace=False)) for _ in range(2)]).astype(np.int64)
    bad = idx.copy()
    bad[0, [3, 100, 511]] = [N, N + 12345, 2 ** 31 - 1]  # past the cache
    bad[1, [0, 7]] = [-2, -(2 ** 31)]                     # negative, other than the -1 pad
    ref_idx = idx.copy()
    ref_idx[0, [3, 100, 511]] = -1
    ref_idx[1, [0, 7]] = -1
    dv = synth.to_device(inp)
    c, lay, rw, p = dv["cache"], dv["layers"][0], dv["rows"], dv["params"]
    args = (lay["q"], rw["q_pos"], rw["seq_of_row"], c["lat"], c["lat_scales"])
    tail = (lay["swa"], lay["swa_scale"], rw["swa_pos0"], p["W"], lay["sink"], p["theta"], p["softmax_scale"])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, _ = S.sparse_attn(*args, torch.from_numpy(bad.astype(np.int32)).cuda(), *tail, dev_status=status)
    assert S.read_device_status(status) == S.EDEVICE_INDEX
    o_ref, _ = O.sparse_attn_rows(inp, 0, ref_idx)
    assert rel_err(out.cpu().numpy(), o_ref) <= out_tol(inp["params"])
    # the same call with valid indices leaves the status word alone
    status.zero_()
    out2, _ = S.sparse_attn(*args, torch.from_numpy(idx.astype(np.int32)).cuda(), *tail, dev_status=status)
    assert S.read_device_status(status) == S.OK
    o_ref2, _ = O.sparse_attn_rows(inp, 0, idx)
    assert rel_err(out2.cpu().numpy(), o_ref2) <= out_tol(inp["params"])
