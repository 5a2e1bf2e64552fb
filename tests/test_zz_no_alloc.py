"""ds4a_topk_select_noalloc: top-k for callers that cannot allocate device
memory (for example a plugin inside a serving engine that has reserved the
GPU's memory for its own pool, or a runtime whose memory plan is fixed before
it starts).  It must give exactly the oracle's selection -- and what
ds4a_topk_select gives with a workspace -- call after call, although every
call reuses the same fixed scratch array.

The cases take the path that uses the scratch (up to 76 (u,q) rows, each
longer than 2^19 scores: the rows are cut over several CTAs whose candidate
slots live in the scratch), back to back, so that the second call runs on what
the first left in the array; a batch that needs no scratch runs in between.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from deepseek_v4_sparse_indexer_gb300 import _binding as B

pytestmark = pytest.mark.gpu


def _scores(R, N, seed):
    rng = np.random.default_rng(seed)
    x = (np.round(rng.standard_normal((R, N)) * 64) / 64).astype(np.float32)   # some exact ties
    x[rng.random((R, N)) < 0.02] = -np.inf
    return x


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


def test_no_alloc_topk_matches_the_oracle_on_calls_in_a_row():
    lib = B.load()
    cases = [
        (3, 600000, 512, 1, None),                                  # scratch: 50 CTAs per row
        (100, 3000, 100, 3, None),                                  # no scratch: one CTA per row
        (5, 540000, 100, 2, [540000, 539999, 100, 7, 0]),          # scratch again, ragged, ties, -inf
    ]
    for R, N, k, seed, n in cases:
        x = _scores(R, N, seed)
        n_list = n if n is not None else [N] * R
        scores = torch.from_numpy(x).cuda().view(R, 1, N)
        n_rows = torch.tensor(n_list, dtype=torch.int32, device="cuda")
        ref_idx, ref_cnt = _with_workspace(scores, n_rows, k)
        idx, cnt = _no_alloc(lib, scores, n_rows, k)
        torch.cuda.synchronize()
        assert torch.equal(cnt, ref_cnt)
        assert torch.equal(idx, ref_idx)
        got_idx, got_cnt = idx.cpu().numpy(), cnt.cpu().numpy()
        for r in range(R):
            o_idx, _ = oracle.topk_select(x[r, :n_list[r]].astype(np.float64), k)
            c = int(got_cnt[r, 0])
            assert c == len(o_idx), (R, N, r)
            assert np.array_equal(got_idx[r, 0, :c], o_idx), (R, N, r)
            assert np.all(got_idx[r, 0, c:] == -1)
    st, flags = B.ds4a_get_device_status()
    assert st == B.DS4A_OK and flags == 0


def test_no_alloc_topk_scratch_covers_every_request_and_bad_arguments_launch_nothing():
    # The scratch is only used by up to 76 very long rows, and then by at
    # most 152 CTA slots: every size fits the fixed array.
    cap = B.DS4A_TOPK_NOALLOC_SCRATCH_BYTES
    for R, N, k in [(1, 1 << 24, 2048), (151, 1 << 20, 512), (76, 65536, 512), (4, 262144, 512), (200, 1 << 20, 512)]:
        assert B.ds4a_workspace_bytes(B.DS4A_OP_TOPK_SELECT, R, 1, N, k) <= cap, (R, N, k)
    lib = B.load()
    R, N = 4, 600000
    scores = torch.zeros(R, 1, N, device="cuda")
    n_rows = torch.full((R,), N, dtype=torch.int32, device="cuda")
    idx = torch.full((R, 1, 8), 9, dtype=torch.int32, device="cuda")
    cnt = torch.full((R, 1), 9, dtype=torch.int32, device="cuda")
    for k in (0, B.DS4A_MAX_TOP_K + 1):
        st = lib.ds4a_topk_select_noalloc(ctypes.c_void_p(scores.data_ptr()), ctypes.c_void_p(n_rows.data_ptr()), R,
                                          1, N, k, ctypes.c_void_p(idx.data_ptr()), ctypes.c_void_p(cnt.data_ptr()),
                                          None)
        assert st == B.DS4A_EINVAL
    torch.cuda.synchronize()
    assert torch.all(idx == 9) and torch.all(cnt == 9)     # nothing was launched
