"""ds4a_topk_select_noalloc: top-k for callers that cannot allocate device
memory (for example a plugin inside a serving engine that has reserved the
GPU's memory for its own pool, or a runtime whose memory plan is fixed before
it starts).  It must give exactly what ds4a_topk_select gives with a workspace,
call after call, although every call reuses the same fixed scratch array.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from deepseek_v4_sparse_indexer_gb300 import _binding as B

pytestmark = pytest.mark.gpu


def _scores(R, N, seed):
    rng = np.random.default_rng(seed)
    x = (np.round(rng.standard_normal((R, 1, N)) * 64) / 64).astype(np.float32)   # some exact ties
    x[rng.random((R, 1, N)) < 0.02] = -np.inf
    return torch.from_numpy(x).cuda()


def _with_workspace(scores, n_rows, k):
    R, Q, N = scores.shape
    idx = torch.empty(R, Q, k, dtype=torch.int32, device="cuda")
    cnt = torch.empty(R, Q, dtype=torch.int32, device="cuda")
    ws = torch.empty(B.ds4a_workspace_bytes(B.DS4A_OP_TOPK_SELECT, R, Q, N, k), dtype=torch.uint8, device="cuda")
    B.ds4a_topk_select(scores, n_rows, k, idx, cnt, ws)
    return idx, cnt


def _no_alloc(lib, scores, n_rows, k):
    """Straight through the C ABI: plain device pointers, no workspace."""
    R, Q, N = scores.shape
    idx = torch.full((R, Q, k), 12345, dtype=torch.int32, device="cuda")
    cnt = torch.full((R, Q), -7, dtype=torch.int32, device="cuda")
    st = lib.ds4a_topk_select_noalloc(ctypes.c_void_p(scores.data_ptr()), ctypes.c_void_p(n_rows.data_ptr()), R, Q,
                                      N, k, ctypes.c_void_p(idx.data_ptr()), ctypes.c_void_p(cnt.data_ptr()),
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == B.DS4A_OK, B._strerror(st)
    return idx, cnt


def test_no_alloc_topk_matches_workspace_topk_on_two_calls_in_a_row():
    lib = B.load()
    # A large call, then a smaller one: the second must not see the first's
    # leftovers in the shared scratch.
    cases = [(64, 16384, 512, 1, None), (5, 3000, 100, 2, [3000, 2999, 100, 7, 0])]
    for R, N, k, seed, n in cases:
        scores = _scores(R, N, seed)
        n_rows = torch.tensor(n if n is not None else [N] * R, dtype=torch.int32, device="cuda")
        ref_idx, ref_cnt = _with_workspace(scores, n_rows, k)
        idx, cnt = _no_alloc(lib, scores, n_rows, k)
        torch.cuda.synchronize()
        assert torch.equal(cnt, ref_cnt)
        assert torch.equal(idx, ref_idx)
    st, flags = B.ds4a_get_device_status()
    assert st == B.DS4A_OK and flags == 0


def test_no_alloc_topk_rejects_requests_beyond_its_scratch():
    lib = B.load()
    R, N, k = 200, 1024, 512          # needs about 16 MiB of scratch; the array holds 8 MiB
    assert B.ds4a_workspace_bytes(B.DS4A_OP_TOPK_SELECT, R, 1, N, k) > B.DS4A_TOPK_NOALLOC_SCRATCH_BYTES
    scores = torch.zeros(R, 1, N, device="cuda")
    n_rows = torch.full((R,), N, dtype=torch.int32, device="cuda")
    idx = torch.full((R, 1, k), 9, dtype=torch.int32, device="cuda")
    cnt = torch.full((R, 1), 9, dtype=torch.int32, device="cuda")
    st = lib.ds4a_topk_select_noalloc(ctypes.c_void_p(scores.data_ptr()), ctypes.c_void_p(n_rows.data_ptr()), R, 1,
                                      N, k, ctypes.c_void_p(idx.data_ptr()), ctypes.c_void_p(cnt.data_ptr()), None)
    assert st == B.DS4A_EWORKSPACE
    torch.cuda.synchronize()
    assert torch.all(idx == 9) and torch.all(cnt == 9)     # nothing was launched
