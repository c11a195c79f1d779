"""csa2_topk_static: the top-K entry point for callers that cannot allocate device memory.

Such callers (a framework that owns every allocation while it captures a stream, a runtime
with a fixed memory budget) have no workspace to hand over, so this entry point takes its
scratch from an array built into the library.  The test calls it through the C ABI, twice
in a row on different inputs, and checks each result against csa2_topk (which uses a
caller workspace): selected indices must be identical.  The file sorts last so that a run
stopping at the first failure has run every other test first.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


def _call_static(S, scores, n_valid, K):
    a = S.TopkArgs()
    a.scores, a.cand, a.n_valid = scores.data_ptr(), None, n_valid.data_ptr()
    a.n_rows, a.L, a.K = scores.shape[0], scores.shape[1], K
    idx = torch.full((a.n_rows, K), -7, dtype=torch.int32, device=scores.device)
    a.idx = idx.data_ptr()
    a.workspace, a.workspace_bytes = None, 0
    f = S._lib.csa2_topk_static
    f.argtypes = [C.POINTER(S.TopkArgs), C.c_void_p]
    f.restype = C.c_int
    status = f(C.byref(a), C.c_void_p(torch.cuda.current_stream().cuda_stream))
    return status, idx


def test_topk_static_matches_topk_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_attention_csa2_gb300 as S
    rows, L, K = 8, 100_003, 512  # several segments per row: the scratch array is used
    for call, seed in enumerate((21, 22)):
        sc = synth.integers((rows, L), seed, 5, -200, 200).float() / 8.0  # many ties
        sc[1] = synth.normal((L,), seed, 6)
        n_valid = torch.tensor([L, L - 1, L // 2, 700, 1, L, 3, L], dtype=torch.int32)
        sc_d, nv_d = sc.cuda(), n_valid.cuda()
        status, got = _call_static(S, sc_d, nv_d, K)
        assert status == 0, f"call {call}: status {status}"
        ref = S.topk(sc_d, nv_d, K)
        torch.cuda.synchronize()
        assert torch.equal(got, ref), f"call {call}: indices differ from csa2_topk"
        assert int((got[4] >= 0).sum()) == 1 and int(got[4, 0]) == 0
