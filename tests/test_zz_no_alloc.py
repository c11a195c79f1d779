"""csa2_topk_static: the top-K entry point for callers that cannot allocate device memory.

Such callers (a framework that owns every allocation while it captures a stream, a runtime
with a fixed memory budget) have no workspace to hand over, so this entry point takes its
scratch from an array built into the library.  The test calls it through the C ABI twice in
a row, with different shapes (8 rows with K = 512, then 2 rows with K = 1024 and another
segment count), so the second call reuses the shared array in a different layout; each result
must equal csa2_topk's (which uses a caller workspace) and the oracle's top-K of the same
scores, index for index.  A too-small workspace passed with the call is ignored.  The file
sorts last so that a run stopping at the first failure has run every other test first.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle as O
import synth

pytestmark = pytest.mark.gpu


def _call_static(S, scores, n_valid, K, junk_ws):
    a = S.TopkArgs()
    a.scores, a.cand, a.n_valid = scores.data_ptr(), None, n_valid.data_ptr()
    a.n_rows, a.L, a.K = scores.shape[0], scores.shape[1], K
    idx = torch.full((a.n_rows, K), -7, dtype=torch.int32, device=scores.device)
    a.idx = idx.data_ptr()
    # a real device buffer far smaller than csa2_topk would need: the static entry point
    # takes no workspace, so it must neither use nor reject it
    a.workspace, a.workspace_bytes = junk_ws.data_ptr(), junk_ws.numel()
    # several segments per row: csa2_topk would need a workspace, so the scratch array is used
    assert S._topk_ws(C.byref(a)) > junk_ws.numel()
    f = S._lib.csa2_topk_static
    f.argtypes = [C.POINTER(S.TopkArgs), C.c_void_p]
    f.restype = C.c_int
    status = f(C.byref(a), C.c_void_p(torch.cuda.current_stream().cuda_stream))
    return status, idx


def test_topk_static_matches_topk_and_oracle_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_attention_csa2_gb300 as S
    junk_ws = torch.zeros(16, dtype=torch.uint8, device="cuda")
    L = 100_003
    cases = [  # (seed, rows, K, n_valid)
        (21, 8, 512, [L, L - 1, L // 2, 700, 1, L, 3, L]),
        (22, 2, 1024, [L, L - 4321]),
    ]
    for call, (seed, rows, K, nv) in enumerate(cases):
        sc = synth.integers((rows, L), seed, 5, -200, 200).float() / 8.0  # many ties
        sc[1] = synth.normal((L,), seed, 6)                               # no ties
        n_valid = torch.tensor(nv, dtype=torch.int32)
        sc_d, nv_d = sc.cuda(), n_valid.cuda()
        status, got = _call_static(S, sc_d, nv_d, K, junk_ws)
        assert status == 0, f"call {call}: status {status}"
        ref = S.topk(sc_d, nv_d, K)
        torch.cuda.synchronize()
        assert torch.equal(got, ref), f"call {call}: indices differ from csa2_topk"
        ora = O.topk_rows(sc.numpy().astype(np.float64), n_valid.numpy(), K)
        assert np.array_equal(got.cpu().numpy(), ora), f"call {call}: indices differ from the oracle"
    assert int(junk_ws.sum()) == 0
