"""Parity of the fused indexer score + top-k select (ds4a_indexer_topk: no
scores array; "DwarfStar(ds4.c) のアーキテクチャを読む" §3-3: the indexer keeps
only the top-k rows for the main attention) through the C ABI:

  * bit-identical idx and count to the two-call path (ds4a_indexer_score then
    ds4a_topk_select), itself checked against the oracle elsewhere;
  * the index sets against the fp64 oracle directly on sampled rows;
  * the cases that stress the running threshold: every row's score equal
    (all ties: the lowest rows win), scores rising with the row (every row
    beats the threshold: the candidate list holds the whole row), fewer
    visible rows than k, empty rows, NaN scores, causal prefill rows, and
    long rows split over many CTAs (the threshold shared between them)."""
import math

import numpy as np
import pytest
import torch

import oracle
from deepseek_v4_sparse_indexer_gb300 import DecodeStep, PrefillStep, _binding as B
from deepseek_v4_sparse_indexer_gb300.workloads import make_decode_inputs, make_prefill_inputs
from tests.parity_util import check_index_set, pool, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    yield
    torch.cuda.synchronize()


def device_ok():
    st, flags = B.ds4a_get_device_status()
    assert st == B.DS4A_OK and flags == 0, f"device status flags {flags}"


def both_paths(iq, w, ik, n_rows, k, q_pos=None, row_pos=None):
    U, Q = iq.shape[:2]
    N_cap = ik.shape[1]
    scores = torch.empty(U, Q, N_cap, device="cuda")
    B.ds4a_indexer_score(iq, w, ik, n_rows, scores, q_pos=q_pos, row_pos=row_pos)
    idx2 = torch.empty(U, Q, k, dtype=torch.int32, device="cuda")
    cnt2 = torch.empty(U, Q, dtype=torch.int32, device="cuda")
    ws2 = torch.empty(B.ds4a_workspace_bytes(B.DS4A_OP_TOPK_SELECT, U, Q, N_cap, k), dtype=torch.uint8, device="cuda")
    B.ds4a_topk_select(scores, n_rows, k, idx2, cnt2, ws2)
    idx1 = torch.full((U, Q, k), -7, dtype=torch.int32, device="cuda")
    cnt1 = torch.full((U, Q), -7, dtype=torch.int32, device="cuda")
    ws1 = torch.empty(B.ds4a_workspace_bytes(B.DS4A_OP_INDEXER_TOPK, U, Q, N_cap, k), dtype=torch.uint8, device="cuda")
    B.ds4a_indexer_topk(iq, w, ik, n_rows, k, idx1, cnt1, ws1, q_pos=q_pos, row_pos=row_pos)
    torch.cuda.synchronize()
    device_ok()
    assert torch.equal(cnt1, cnt2), (cnt1.flatten()[:8], cnt2.flatten()[:8])
    assert torch.equal(idx1, idx2)
    return idx1, cnt1, scores


def rand_case(U, Q, N_cap, seed, scale_rows=None):
    g = torch.Generator().manual_seed(seed)
    iq = (torch.randn(U, Q, 64, 128, generator=g) / math.sqrt(128)).to(torch.bfloat16)
    w = torch.rand(U, Q, 64, generator=g)
    ik = torch.randn(U, N_cap, 128, generator=g) / math.sqrt(128)
    if scale_rows is not None:
        ik = ik * scale_rows
    return iq.cuda(), w.cuda(), ik.to(torch.bfloat16).cuda()


def oracle_check(iq, w, ik, n_rows, idx, cnt, k, units, q_pos=None, row_pos=None):
    def one(uq):
        u, q = uq
        n = int(n_rows[u])
        kw = {}
        if q_pos is not None:
            kw = dict(q_pos=q_pos[u, q:q + 1].cpu().numpy(), row_pos=row_pos[u].cpu().numpy())
        ref = oracle.indexer_score(u16(iq[u, q:q + 1]), w[u, q:q + 1].cpu().numpy(), u16(ik[u, :max(n, 1)]), n,
                                   **kw)[0][:n]
        check_index_set(idx[u, q].cpu().numpy(), int(cnt[u, q]), ref, k)
    with pool() as p:
        list(p.map(one, units))


def test_fused_decode_ragged_rows_match_two_calls_and_oracle():
    U, N_cap, k = 6, 5000, 512
    iq, w, ik = rand_case(U, 1, N_cap, seed=70)
    n_rows = torch.tensor([5000, 4999, 600, 512, 100, 0], dtype=torch.int32, device="cuda")
    idx, cnt, _ = both_paths(iq, w, ik, n_rows, k)
    assert cnt.flatten().tolist() == [512, 512, 512, 512, 100, 0]
    oracle_check(iq, w, ik, n_rows, idx, cnt, k, [(u, 0) for u in range(U)])


def test_fused_many_units_and_k_extremes():
    U, N_cap = 200, 3000
    iq, w, ik = rand_case(U, 1, N_cap, seed=71)
    n_rows = torch.tensor([N_cap - (u % 9) * 300 for u in range(U)], dtype=torch.int32, device="cuda")
    for k in (1, 512, 2048):
        idx, cnt, _ = both_paths(iq, w, ik, n_rows, k)
    oracle_check(iq, w, ik, n_rows, idx, cnt, 2048, [(0, 0), (7, 0), (199, 0)])


def test_fused_long_rows_split_over_many_ctas():
    # 3 units x 300k rows: each unit's row is scanned by about 50 CTAs that share its threshold
    U, N_cap, k = 3, 300_000, 512
    iq, w, ik = rand_case(U, 1, N_cap, seed=72)
    heavy = torch.rand(U, N_cap, generator=torch.Generator().manual_seed(73)) < 0.05
    ik = torch.where(heavy.cuda()[..., None], ik * 4, ik)
    n_rows = torch.tensor([N_cap, N_cap - 1, 131_072], dtype=torch.int32, device="cuda")
    idx, cnt, _ = both_paths(iq, w, ik, n_rows, k)
    oracle_check(iq, w, ik, n_rows, idx, cnt, k, [(u, 0) for u in range(U)])


@pytest.mark.parametrize("k", [512, 1024])
def test_fused_all_equal_scores_take_the_lowest_rows(k):
    # every row a candidate: 20,000 pairs, more than either candidate cache
    # (6,144 at k <= 512, 12,288 above) holds, so the list is read in place
    U, N_cap = 3, 20_000
    iq, w, ik = rand_case(U, 1, N_cap, seed=74)
    ik = ik[:, :1].expand(U, N_cap, 128).contiguous()            # identical keys: every score equal
    n_rows = torch.tensor([20_000, k - 1, 9000], dtype=torch.int32, device="cuda")
    idx, cnt, _ = both_paths(iq, w, ik, n_rows, k)
    assert idx[0, 0].tolist() == list(range(k)) and int(cnt[1, 0]) == k - 1
    assert idx[2, 0].tolist() == list(range(k))


@pytest.mark.parametrize("k", [512, 1024])
def test_fused_rising_scores_keep_every_row_as_candidate(k):
    # key of row r scaled by (1 + r/N): every row beats the threshold of the rows before it
    U, N_cap = 2, 30_000
    ramp = (1 + torch.arange(N_cap, dtype=torch.float32) / N_cap)[None, :, None]
    iq, w, ik = rand_case(U, 1, N_cap, seed=75)
    base = ik[:, :1].float().abs()                                  # one positive key per unit
    iq = iq.abs()                                                   # positive dots: ReLU keeps all heads
    ik = (base * ramp.cuda()).to(torch.bfloat16)
    n_rows = torch.tensor([N_cap, N_cap], dtype=torch.int32, device="cuda")
    idx, cnt, scores = both_paths(iq, w, ik, n_rows, k)
    oracle_check(iq, w, ik, n_rows, idx, cnt, k, [(0, 0), (1, 0)])


def test_fused_nan_and_negative_scores():
    U, N_cap, k = 3, 4000, 256
    iq, w, ik = rand_case(U, 1, N_cap, seed=76)
    w = w.clone()
    w[0, 0, 5] = float("nan")                                       # every score of unit 0 NaN: nothing visible
    w[1] = -w[1]                                                    # all scores <= 0
    n_rows = torch.tensor([N_cap, N_cap, 3000], dtype=torch.int32, device="cuda")
    idx, cnt, _ = both_paths(iq, w, ik, n_rows, k)
    assert int(cnt[0, 0]) == 0 and torch.all(idx[0, 0] == -1)
    oracle_check(iq, w, ik, n_rows, idx, cnt, k, [(1, 0), (2, 0)])


@pytest.mark.parametrize("Q", [3, 9])
def test_fused_query_groups_with_causal_positions(Q):
    U, N_cap, k = 2, 6000, 512
    iq, w, ik = rand_case(U, Q, N_cap, seed=77 + Q)
    g = torch.Generator().manual_seed(Q)
    row_pos = torch.sort(torch.randint(0, 24000, (U, N_cap), generator=g), dim=1).values.to(torch.int32).cuda()
    q_pos = torch.randint(0, 24100, (U, Q), generator=g).to(torch.int32).cuda()
    q_pos[0, 0] = -1                                                # sees no row
    n_rows = torch.tensor([6000, 4321], dtype=torch.int32, device="cuda")
    idx, cnt, _ = both_paths(iq, w, ik, n_rows, k, q_pos=q_pos, row_pos=row_pos)
    assert int(cnt[0, 0]) == 0
    oracle_check(iq, w, ik, n_rows, idx, cnt, k, [(u, q) for u in range(U) for q in range(Q)], q_pos, row_pos)


def test_fused_steps_equal_the_two_call_steps():
    x = make_decode_inputs(40, 8192, device="cuda", seed=78, n_rows=[8192 - 37 * i for i in range(40)])
    a, b = DecodeStep(40, 8192, 512), DecodeStep(40, 8192, 512, fused=True)
    a(x)
    b(x)
    torch.cuda.synchronize()
    device_ok()
    assert torch.equal(a.idx, b.idx) and torch.equal(a.count, b.count) and torch.equal(a.out, b.out)
    xp = make_prefill_inputs(64, 3000, device="cuda", seed=79)
    pa, pb = PrefillStep(64, xp["ik"].shape[0], 512), PrefillStep(64, xp["ik"].shape[0], 512, fused=True)
    pa(xp)
    pb(xp)
    torch.cuda.synchronize()
    device_ok()
    assert torch.equal(pa.idx, pb.idx) and torch.equal(pa.count, pb.count) and torch.equal(pa.out, pb.out)


def test_fused_rejects_bad_arguments():
    iq, w, ik = rand_case(1, 1, 100, seed=80)
    n_rows = torch.tensor([100], dtype=torch.int32, device="cuda")
    idx = torch.empty(1, 1, 64, dtype=torch.int32, device="cuda")
    cnt = torch.empty(1, 1, dtype=torch.int32, device="cuda")
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(B.Ds4aError) as e:
        B.ds4a_indexer_topk(iq, w, ik, n_rows, 64, idx, cnt, small)
    assert e.value.status == B.DS4A_EWORKSPACE
