"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Small cases cover several tiles and ragged tails, every branch of the kernels
(query groups, split rows, candidate-list overflow, empty sets, out-of-range
indices), and stress inputs with a peaked softmax; the five workloads are
checked in full where the oracle finishes in seconds, and on sampled units /
queries at full size.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from deepseek_v4_sparse_indexer_gb300 import DecodeStep, DenseStep, PrefillStep, _binding as B
from deepseek_v4_sparse_indexer_gb300.workloads import WORKLOADS, make_decode_inputs, make_prefill_inputs
from tests.parity_util import (check_index_set, check_output, check_scores, pool, score_tolerance, u16)

pytestmark = pytest.mark.gpu
SCALE = 1.0 / math.sqrt(512)


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    yield
    torch.cuda.synchronize()


def device_ok():
    st, flags = B.ds4a_get_device_status()
    assert st == B.DS4A_OK and flags == 0, f"device status flags {flags}"


# ----------------------------------------------------------------------------
# decode: unit-level check shared by the tests below
# ----------------------------------------------------------------------------

def check_decode_unit(x, st, u, top_k, scale, check_sc=True):
    n = int(x["n_rows"][u])
    nraw = int(x["n_raw"][u])
    iq = u16(x["iq"][u])
    w = x["w"][u].cpu().numpy()
    ik = u16(x["ik"][u, :max(n, 1)])
    ref = oracle.indexer_score(iq[None], w[None], ik, n)[0][:n]
    gpu_s = st.scores[u, 0, :n].cpu().numpy()
    if check_sc:
        check_scores(gpu_s, ref, score_tolerance(iq, w, ik, n))
    cnt = int(st.count[u, 0])
    gidx = st.idx[u, 0].cpu().numpy()
    swaps = check_index_set(gidx, cnt, ref, top_k)
    rows = u16(x["rows"][u, :max(n, 1)])
    raw = u16(x["raw"][u])
    out, lse = oracle.sparse_attention(u16(x["q"][u]), rows, gidx[:cnt], raw, np.arange(nraw), scale)
    stats = check_output(st.out[u].cpu().numpy(), out, st.lse[u].cpu().numpy(), lse)
    stats["swaps"] = swaps
    return stats


def run_decode(x, top_k, scale=SCALE):
    U, N_cap = x["ik"].shape[:2]
    st = DecodeStep(U, N_cap, top_k)
    st(x, scale)
    torch.cuda.synchronize()
    device_ok()
    return st


# ----------------------------------------------------------------------------
# A1 indexer score
# ----------------------------------------------------------------------------

def test_indexer_scores_decode_ragged_and_untouched_tail():
    x = make_decode_inputs(3, 300, device="cuda", seed=1, n_rows=[300, 129, 1])
    scores = torch.full((3, 1, 300), 12345.0, device="cuda")
    B.ds4a_indexer_score(x["iq"].view(3, 1, 64, 128), x["w"].view(3, 1, 64), x["ik"], x["n_rows"], scores)
    torch.cuda.synchronize()
    device_ok()
    for u, n in enumerate([300, 129, 1]):
        iq, w, ik = u16(x["iq"][u]), x["w"][u].cpu().numpy(), u16(x["ik"][u])
        ref = oracle.indexer_score(iq[None], w[None], ik, n)[0]
        check_scores(scores[u, 0, :n].cpu().numpy(), ref[:n], score_tolerance(iq, w, ik, n))
        assert torch.all(scores[u, 0, n:] == 12345.0)


@pytest.mark.parametrize("Q", [2, 4, 6, 9])
def test_indexer_scores_query_groups_with_positions(Q):
    U, N_cap = 2, 400
    g = torch.Generator().manual_seed(Q)
    iq = (torch.randn(U, Q, 64, 128, generator=g) / math.sqrt(128)).to(torch.bfloat16).cuda()
    w = torch.rand(U, Q, 64, generator=g).cuda()
    ik = (torch.randn(U, N_cap, 128, generator=g) / math.sqrt(128)).to(torch.bfloat16).cuda()
    n_rows = torch.tensor([400, 333], dtype=torch.int32).cuda()
    row_pos = torch.sort(torch.randint(0, 2000, (U, N_cap), generator=g), dim=1).values.to(torch.int32).cuda()
    q_pos = torch.randint(0, 2100, (U, Q), generator=g).to(torch.int32).cuda()
    scores = torch.empty(U, Q, N_cap, device="cuda")
    B.ds4a_indexer_score(iq, w, ik, n_rows, scores, q_pos=q_pos, row_pos=row_pos)
    torch.cuda.synchronize()
    device_ok()
    for u in range(U):
        n = int(n_rows[u])
        iqn, wn, ikn = u16(iq[u]), w[u].cpu().numpy(), u16(ik[u])
        ref = oracle.indexer_score(iqn, wn, ikn, n, q_pos=q_pos[u].cpu().numpy(), row_pos=row_pos[u].cpu().numpy())
        for q in range(Q):
            tol = score_tolerance(iqn[q], wn[q], ikn, n)
            check_scores(scores[u, q, :n].cpu().numpy(), ref[q, :n], tol)


def _indexer_case(U, Q, N_cap, n_rows, seed, positions=False):
    g = torch.Generator().manual_seed(seed)
    iq = (torch.randn(U, Q, 64, 128, generator=g) / math.sqrt(128)).to(torch.bfloat16).cuda()
    w = (torch.rand(U, Q, 64, generator=g) * 2 - 0.5).cuda()
    ik = (torch.randn(U, N_cap, 128, generator=g) / math.sqrt(128)).to(torch.bfloat16).cuda()
    nr = torch.tensor(n_rows, dtype=torch.int32).cuda()
    q_pos = row_pos = None
    if positions:
        row_pos = torch.sort(torch.randint(0, 4 * N_cap, (U, N_cap), generator=g), dim=1).values.to(torch.int32).cuda()
        q_pos = torch.randint(0, 4 * N_cap + 8, (U, Q), generator=g).to(torch.int32).cuda()
    scores = torch.full((U, Q, N_cap), 12345.0, device="cuda")
    B.ds4a_indexer_score(iq, w, ik, nr, scores, q_pos=q_pos, row_pos=row_pos)
    torch.cuda.synchronize()
    return iq, w, ik, q_pos, row_pos, scores


def _check_indexer_unit(iq, w, ik, q_pos, row_pos, scores, u, n):
    iqn, wn, ikn = u16(iq[u]), w[u].cpu().numpy(), u16(ik[u])
    kw = {}
    if q_pos is not None:
        kw = dict(q_pos=q_pos[u].cpu().numpy(), row_pos=row_pos[u].cpu().numpy())
    ref = oracle.indexer_score(iqn, wn, ikn, n, **kw)
    for q in range(iq.shape[1]):
        check_scores(scores[u, q, :n].cpu().numpy(), ref[q, :n], score_tolerance(iqn[q], wn[q], ikn, n))
    assert torch.all(scores[u, :, n:] == 12345.0)


@pytest.mark.parametrize("U,Q,N_cap,n_rows,positions", [
    # one query (decode): 200 units x 3 tiles, so CTA shares end inside units
    (200, 1, 260, [260 - (u % 7) * 37 for u in range(200)], False),
    # query groups of 4 with a partial last group; shares cross groups and units,
    # and units with no rows or one row sit between full ones
    (5, 9, 3000, [3000, 1, 0, 2999, 1500], True),
])
def test_indexer_work_shares_cross_unit_and_group_boundaries(U, Q, N_cap, n_rows, positions):
    case = _indexer_case(U, Q, N_cap, n_rows, seed=U + Q, positions=positions)
    device_ok()
    units = range(U) if U <= 8 else [0, 1, 2, 3, 50, 99, 150, 198, 199]
    for u in units:
        _check_indexer_unit(*case, u, n_rows[u])


def test_indexer_row_count_out_of_range_is_clamped_and_flagged():
    U, Q, N_cap = 3, 5, 300
    iq, w, ik, q_pos, row_pos, scores = _indexer_case(U, Q, N_cap, [-4, N_cap + 7, 200], seed=35)
    st, flags = B.ds4a_get_device_status()
    assert st == B.DS4A_EDEVICE and flags & B.DS4A_DEV_BOUNDS
    _check_indexer_unit(iq, w, ik, q_pos, row_pos, scores, 0, 0)
    _check_indexer_unit(iq, w, ik, q_pos, row_pos, scores, 1, N_cap)
    _check_indexer_unit(iq, w, ik, q_pos, row_pos, scores, 2, 200)
    device_ok()


# ----------------------------------------------------------------------------
# A2 top-k on given scores: bit-exact against the oracle
# ----------------------------------------------------------------------------

def topk_case(rows_f32, n_rows, top_k, shift=0):
    """rows_f32: float32 [R, N_cap] (one unit per row); checks every row exactly.
    shift > 0 places the scores `shift` floats past a 16-byte boundary."""
    R, N_cap = rows_f32.shape
    if shift:
        buf = torch.zeros(R * N_cap + shift, dtype=torch.float32, device="cuda")
        buf[shift:] = torch.from_numpy(rows_f32).cuda().view(-1)
        s = buf[shift:].view(R, 1, N_cap)
    else:
        s = torch.from_numpy(rows_f32).cuda().view(R, 1, N_cap)
    nr = torch.tensor(n_rows, dtype=torch.int32).cuda()
    idx = torch.full((R, 1, top_k), 777, dtype=torch.int32, device="cuda")
    cnt = torch.full((R, 1), -5, dtype=torch.int32, device="cuda")
    ws = torch.empty(B.ds4a_workspace_bytes(B.DS4A_OP_TOPK_SELECT, R, 1, N_cap, top_k), dtype=torch.uint8,
                     device="cuda")
    B.ds4a_topk_select(s, nr, top_k, idx, cnt, ws)
    torch.cuda.synchronize()
    device_ok()
    for r in range(R):
        n = n_rows[r]
        ref_idx, _ = oracle.topk_select(rows_f32[r, :n].astype(np.float64), top_k)
        c = int(cnt[r, 0])
        got = idx[r, 0].cpu().numpy()
        assert c == len(ref_idx), (r, c, len(ref_idx))
        assert np.array_equal(got[:c], ref_idx), f"row {r}"
        assert np.all(got[c:] == -1)


def test_topk_random_and_ragged():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 5000)).astype(np.float32)
    topk_case(x, [5000, 4999, 513, 512, 77], 512)


def test_topk_ties_neginf_nan_and_signed_zero():
    rng = np.random.default_rng(1)
    x = (np.round(rng.standard_normal((4, 3000)) * 2) / 2).astype(np.float32)   # heavy ties
    x[0, rng.random(3000) < 0.3] = -np.inf
    x[1, rng.random(3000) < 0.1] = np.nan
    x[2] = 0.0
    x[2, ::2] = -0.0                                                          # -0 == +0: lower rows win
    x[2, 5:20] = 1.0
    x[3] = -np.abs(x[3])                                                      # all negative
    topk_case(x, [3000, 3000, 3000, 2999], 100)


@pytest.mark.parametrize("k", [1, 7, 2048])
def test_topk_k_extremes(k):
    rng = np.random.default_rng(k)
    x = rng.standard_normal((3, 4096)).astype(np.float32)
    topk_case(x, [4096, 1000, 3], k)


def test_topk_all_equal_small_and_overflowing_candidates():
    # 3000 equal scores fit the candidate list; 20000 overflow it (fallback path).
    topk_case(np.full((2, 3000), 0.5, np.float32), [3000, 2500], 512)
    topk_case(np.full((2, 20000), 0.25, np.float32), [20000, 19999], 512)


def test_topk_one_long_row_split_over_many_ctas():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((1, 262144)).astype(np.float32)
    x[0, rng.random(262144) < 0.05] *= 4
    topk_case(x, [262144], 512)


# Up to 16 rows of more than 4,096 scores: a cluster of eight CTAs per row
# filters its chunks against one sampled threshold; the CTAs exchange counts,
# a bucket histogram and the crossing bucket's keys through distributed shared
# memory and each writes its own rows (or CTA 0 selects from the whole row when
# the lists cannot decide).

def test_topk_cluster_rows_ties_neginf_nan_locality_and_short_rows():
    rng = np.random.default_rng(20)
    N = 100000
    x = rng.standard_normal((8, N)).astype(np.float32)
    x[1] = np.round(x[1] * 2) / 2                             # heavy ties at the k-th score
    x[2, rng.random(N) < 0.3] = -np.inf
    x[2, rng.random(N) < 0.1] = np.nan
    x[3] = 0.25                                               # all equal: slots overflow, exact pass
    x[4, N - 5000:] += 3.0                                    # the top rows crowded in the last chunk
    x[5, ::2] = -0.0
    x[5, 1::2] = 0.0
    x[5, 777] = 1.0
    topk_case(x, [N, N, N, N, N - 3, 9000, 8000, 513], 512)   # 8,000 and 513 rows: every row a candidate


@pytest.mark.parametrize("k", [1, 2048])
def test_topk_cluster_rows_k_extremes_and_odd_stride(k):
    rng = np.random.default_rng(21 + k)
    x = rng.standard_normal((3, 70001)).astype(np.float32)   # N_cap not a multiple of 4: scalar loads
    x[1, rng.random(70001) < 0.05] *= 4
    topk_case(x, [70001, 70000, 2047], k)


def test_topk_cluster_rows_nine_to_sixteen_rows_load_through_registers():
    # more than eight rows: the cluster CTAs load their chunks eight float4 per
    # thread (no bulk-copy ring); ties, -inf, NaN, crowding, ragged rows
    rng = np.random.default_rng(27)
    N = 100000
    x = rng.standard_normal((12, N)).astype(np.float32)
    x[1] = np.round(x[1] * 2) / 2
    x[2, rng.random(N) < 0.3] = -np.inf
    x[3, rng.random(N) < 0.1] = np.nan
    x[4, N - 5000:] += 3.0
    x[5] = 0.25                                               # all equal: exact pass by CTA 0
    x[6, rng.random(N) < 0.05] *= 4
    topk_case(x, [N, N, N, N, N, N, N - 7, 50001, 9000, 8193, 8192, 513], 512)


def test_topk_cluster_rows_longest_chunks_refill_the_ring():
    # five rows of 524,288 scores: eight CTAs per row, 65,536 scores each, eight
    # 32 KB bulk copies through a ring of four; ragged ends exercise the copy
    # rounded up to 16 bytes
    rng = np.random.default_rng(25)
    N = 524288
    x = rng.standard_normal((5, N)).astype(np.float32)
    x[1, rng.random(N) < 0.05] *= 4
    x[2, 300000:300100] = 9.0                                 # the top rows inside one copy
    x[3] = np.round(x[3] * 2) / 2
    topk_case(x, [N, 400001, 262147, N - 3, 100000], 512)


def test_topk_cluster_rows_sixteen_ctas_per_row():
    # up to four rows: sixteen CTAs per row (ties, -inf, NaN, all equal, ragged,
    # the top rows crowded into one CTA's chunk)
    rng = np.random.default_rng(28)
    N = 300000
    x = rng.standard_normal((4, N)).astype(np.float32)
    x[0] = np.round(x[0] * 2) / 2
    x[1, rng.random(N) < 0.3] = -np.inf
    x[1, rng.random(N) < 0.1] = np.nan
    x[2] = 0.125                                              # all equal: exact pass by CTA 0
    x[3, 120000:125000] += 3.0
    topk_case(x, [N, N - 1, 200003, 150001], 512)
    topk_case(x[:2].copy(), [N, 77777], 2048)


@pytest.mark.parametrize("shape", [(3, 100000), (160, 9000), (2, 600000)])
def test_topk_scores_not_16_byte_aligned(shape):
    # 4-byte aligned scores (the API's requirement) one float past a 16-byte
    # boundary: every kernel takes its scalar loads
    R, N = shape
    rng = np.random.default_rng(26 + R)
    x = rng.standard_normal((R, N)).astype(np.float32)
    topk_case(x, [N - (r % 3) * 7 for r in range(R)], 512, shift=1)


def test_topk_cluster_rows_all_candidates_and_sixteen_rows():
    rng = np.random.default_rng(22)
    x = rng.standard_normal((16, 9000)).astype(np.float32)
    x[::3, 4500:] += 1.0
    # rows of at most 8,192 scores take every visible row as a candidate
    topk_case(x, [9000 - (i % 7) * 700 for i in range(16)], 512)


# Rows of more than 2^19 scores in batches of up to 76 rows: every row is cut
# over several CTAs that filter their chunk against one sampled threshold into
# slots of their own in the workspace, and one CTA per row selects from the
# joined slots (or from the whole row when the slots cannot decide).

def test_topk_split_very_long_rows_ties_locality_and_short_rows():
    rng = np.random.default_rng(23)
    N = 600000
    x = rng.standard_normal((4, N)).astype(np.float32)
    x[1] = np.round(x[1] * 2) / 2                             # heavy ties at the k-th score
    x[2, N - 40000:] += 3.0                                   # the top rows crowded in the last chunks
    x[2, rng.random(N) < 0.2] = -np.inf
    x[3] = 0.5                                                # all equal: slots overflow, exact pass
    topk_case(x, [N, N - 1, 550000, 7000], 512)


@pytest.mark.parametrize("k", [1, 2048])
def test_topk_split_very_long_rows_k_extremes_and_odd_stride(k):
    rng = np.random.default_rng(24 + k)
    x = rng.standard_normal((2, 524289)).astype(np.float32)  # N_cap not a multiple of 4: scalar loads
    x[1, rng.random(524289) < 0.05] *= 4
    topk_case(x, [524289, 300000], k)


# Batches with at least as many rows as SMs take the one-CTA-per-row kernel
# (sampled threshold, candidate list, exact fallback over the row).

ROWS_MANY = 160      # > 152 SMs


def _many(rng, n_cap, lens):
    return [lens[i % len(lens)] for i in range(ROWS_MANY)]


def test_topk_rows_random_and_ragged():
    rng = np.random.default_rng(10)
    x = rng.standard_normal((ROWS_MANY, 20000)).astype(np.float32)
    x[::7] *= 1e-3                                   # narrow value range on some rows
    x[3::7][:, rng.random(20000) < 0.05] *= 4        # heavy tail on others
    topk_case(x, _many(rng, 20000, [20000, 19999, 4097, 4096, 3000, 513, 512, 77, 1, 0]), 512)


def test_topk_rows_between_32768_and_65536():
    # long rows through the 256-thread shape (candidates cached, bitmap output)
    rng = np.random.default_rng(17)
    x = rng.standard_normal((ROWS_MANY, 40000)).astype(np.float32)
    x[1::5][:, rng.random(40000) < 0.02] *= 6        # heavy tail
    x[2::5, 30000:] += 2.0                           # the top rows crowded at the end of the row
    topk_case(x, _many(rng, 40000, [40000, 39999, 32769, 32768, 20000, 512]), 512)


def test_topk_rows_longer_than_the_row_bitmap():
    # rows over 131,072 entries take the 512-thread shape and sort the chosen rows
    rng = np.random.default_rng(18)
    x = rng.standard_normal((ROWS_MANY, 140000)).astype(np.float32)
    x[1::4, 135000:] += 3.0                          # the top rows crowded at the end of the row
    x[2::4] = np.round(x[2::4] * 4) / 4              # heavy ties
    topk_case(x, _many(rng, 140000, [140000, 139999, 131073, 131072, 70000]), 512)


def test_topk_rows_ties_neginf_nan_signed_zero():
    rng = np.random.default_rng(11)
    x = (np.round(rng.standard_normal((ROWS_MANY, 12000)) * 2) / 2).astype(np.float32)   # heavy ties
    x[0::4][:, rng.random(12000) < 0.3] = -np.inf
    x[1::4][:, rng.random(12000) < 0.1] = np.nan
    x[2::4] = 0.0
    x[2::4, ::2] = -0.0
    x[2::4, 5:20] = 1.0
    x[3::4] = -np.abs(x[3::4])
    topk_case(x, _many(rng, 12000, [12000, 11999, 6000]), 100)


def test_topk_rows_all_equal_sorted_and_prefix_visible():
    rng = np.random.default_rng(12)
    x = np.empty((ROWS_MANY, 16384), np.float32)
    x[0::4] = 0.25                                              # all equal: candidate overflow
    x[1::4] = np.arange(16384, dtype=np.float32)                # ascending by row
    x[2::4] = -np.arange(16384, dtype=np.float32)               # descending by row
    x[3::4] = rng.standard_normal((ROWS_MANY // 4, 16384)).astype(np.float32)
    for r in range(3, ROWS_MANY, 4):                            # visible prefix, -inf after (causal)
        x[r, rng.integers(100, 16384):] = -np.inf
    topk_case(x, _many(rng, 16384, [16384, 16383, 9000]), 512)


# Batches of at least four rows per SM with k <= 512 take the 128-thread shape
# (2,048 candidates, the threshold aimed at 2k, eight CTAs per SM).
ROWS_LOTS = 640      # >= 4 x 152

@pytest.mark.parametrize("k", [1, 100, 512, 513])
def test_topk_rows_large_batches_small_shape(k):
    rng = np.random.default_rng(30 + k)
    N = 20000
    x = rng.standard_normal((ROWS_LOTS, N)).astype(np.float32)
    x[0::8] = np.round(x[0::8] * 2) / 2                          # heavy ties at the k-th score
    x[1::8][:, rng.random(N) < 0.3] = -np.inf
    x[2::8][:, rng.random(N) < 0.1] = np.nan
    x[3::8] = 0.25                                               # all equal: candidate overflow
    x[4::8, 15000:] += 3.0                                       # the top rows crowded at the end
    x[5::8][:, rng.random(N) < 0.05] *= 4                        # heavy tail
    lens = [N, N - 1, 4097, 2049, 2048, 513, 77, 0]
    topk_case(x, [lens[(r // 8) % len(lens)] for r in range(ROWS_LOTS)], k)


@pytest.mark.parametrize("k", [1, 2048])
def test_topk_rows_k_extremes_and_odd_stride(k):
    rng = np.random.default_rng(13 + k)
    x = rng.standard_normal((ROWS_MANY, 5001)).astype(np.float32)     # N_cap not a multiple of 4
    topk_case(x, _many(rng, 5001, [5001, 5000, 2048, 2047, 10]), k)


# ----------------------------------------------------------------------------
# A4 attention on given row sets
# ----------------------------------------------------------------------------

def attention_case(U, N_cap, top_k, seed, q_scale=1.0, n_raw=None):
    rng = np.random.default_rng(seed)
    x = make_decode_inputs(U, N_cap, device="cuda", seed=seed, q_scale=q_scale,
                           n_raw=n_raw if n_raw is not None else list(rng.integers(0, 129, U)))
    idx = np.full((U, top_k), -1, np.int32)
    cnt = rng.integers(0, top_k + 1, U).astype(np.int32)
    cnt[0] = top_k
    for u in range(U):
        idx[u, :cnt[u]] = np.sort(rng.choice(N_cap, size=cnt[u], replace=False))
    idx_t, cnt_t = torch.from_numpy(idx).cuda(), torch.from_numpy(cnt).cuda()
    out = torch.empty(U, 64, 512, device="cuda")
    lse = torch.empty(U, 64, device="cuda")
    nb = B.ds4a_workspace_bytes(B.DS4A_OP_SPARSE_ATTN_DECODE, U, 1, N_cap, top_k)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda") if nb else None
    B.ds4a_sparse_attn_decode(x["q"], x["rows"], idx_t, cnt_t, x["raw"], x["n_raw"], SCALE, out, lse, ws)
    torch.cuda.synchronize()
    device_ok()

    def one(u):
        nraw = int(x["n_raw"][u])
        ro, rl = oracle.sparse_attention(u16(x["q"][u]), u16(x["rows"][u]), idx[u, :cnt[u]], u16(x["raw"][u]),
                                         np.arange(nraw), SCALE)
        return check_output(out[u].cpu().numpy(), ro, lse[u].cpu().numpy(), rl)

    with pool() as p:
        return list(p.map(one, range(U)))


@pytest.mark.parametrize("q_scale", [1.0, 32.0])
def test_attention_split_rows_few_units(q_scale):
    attention_case(3, 2000, 512, seed=11, q_scale=q_scale)


@pytest.mark.parametrize("q_scale", [1.0, 32.0])
def test_attention_one_cta_per_unit(q_scale):
    attention_case(160, 700, 512, seed=12, q_scale=q_scale)


@pytest.mark.parametrize("U,top_k", [(152, 512), (305, 512), (457, 64), (40, 512), (17, 64), (9, 64), (16, 512),
                                     (1, 512), (19, 512), (20, 512), (19, 384), (3, 320)])
def test_attention_work_schedule(U, top_k):
    # Whole strided rounds of 152 units, then the remainder units' tiles cut
    # into equal shares: no remainder, one remainder unit over ten CTAs, three-
    # tile units, and fewer units than CTAs (pieces merged by a second kernel:
    # one-tile pieces, shares of several tiles, a single unit over ten CTAs,
    # 19 and 20 units of ten tiles, 19 units of eight, 3 units of seven).
    attention_case(U, 600, top_k, seed=40 + U)


@pytest.mark.parametrize("U", [2, 20])
def test_attention_largest_top_k_in_many_pieces(U):
    # top_k = 2,048: 34 tiles per unit.  Two units: 68 one-tile pieces, 34 per
    # unit (the most pieces a unit can have); twenty units: 680 tiles in 152
    # shares, merged.
    attention_case(U, 2500, 2048, seed=47 + U)


@pytest.mark.parametrize("scale", [-1 / math.sqrt(512), 0.0, 4 / math.sqrt(512)])
def test_attention_negative_zero_and_large_scale(scale):
    # A non-positive scale takes the general softmax path (the max is taken
    # after scaling); scale 0 gives the plain mean of the row set.
    U, N_cap, k = 5, 900, 256
    rng = np.random.default_rng(61)
    x = make_decode_inputs(U, N_cap, device="cuda", seed=61, n_raw=[128, 64, 0, 1, 100])
    cnt = np.array([256, 200, 64, 0, 129], np.int32)
    idx = np.full((U, k), -1, np.int32)
    for u in range(U):
        idx[u, :cnt[u]] = np.sort(rng.choice(N_cap, size=cnt[u], replace=False))
    out = torch.empty(U, 64, 512, device="cuda")
    lse = torch.empty(U, 64, device="cuda")
    ws = torch.empty(max(B.ds4a_workspace_bytes(B.DS4A_OP_SPARSE_ATTN_DECODE, U, 1, N_cap, k), 1),
                     dtype=torch.uint8, device="cuda")
    B.ds4a_sparse_attn_decode(x["q"], x["rows"], torch.from_numpy(idx).cuda(), torch.from_numpy(cnt).cuda(),
                              x["raw"], x["n_raw"], scale, out, lse, ws)
    torch.cuda.synchronize()
    device_ok()
    for u in range(U):
        ro, rl = oracle.sparse_attention(u16(x["q"][u]), u16(x["rows"][u]), idx[u, :cnt[u]], u16(x["raw"][u]),
                                         np.arange(int(x["n_raw"][u])), scale)
        check_output(out[u].cpu().numpy(), ro, lse[u].cpu().numpy(), rl)


def test_attention_raw_window_extremes_and_odd_k():
    attention_case(4, 300, 100, seed=13, n_raw=[0, 1, 127, 128])


def test_attention_empty_row_set():
    x = make_decode_inputs(2, 64, device="cuda", seed=3, n_raw=[0, 0])
    idx = torch.full((2, 512), -1, dtype=torch.int32, device="cuda")
    cnt = torch.zeros(2, dtype=torch.int32, device="cuda")
    out = torch.full((2, 64, 512), 7.0, device="cuda")
    lse = torch.zeros(2, 64, device="cuda")
    ws = torch.empty(B.ds4a_workspace_bytes(B.DS4A_OP_SPARSE_ATTN_DECODE, 2, 1, 64, 512), dtype=torch.uint8,
                     device="cuda")
    B.ds4a_sparse_attn_decode(x["q"], x["rows"], idx, cnt, x["raw"], x["n_raw"], SCALE, out, lse, ws)
    torch.cuda.synchronize()
    device_ok()
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


def test_attention_out_of_range_index_is_masked_and_flagged():
    U, N_cap = 160, 256
    x = make_decode_inputs(U, N_cap, device="cuda", seed=4, n_raw=[5] * U)
    rng = np.random.default_rng(4)
    idx = np.stack([np.sort(rng.choice(N_cap, 64, replace=False)) for _ in range(U)]).astype(np.int32)
    bad = idx.copy()
    bad[0, 3] = N_cap + 5
    bad[1, 0] = -3
    out = torch.empty(U, 64, 512, device="cuda")
    cnt = torch.full((U,), 64, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(B.ds4a_workspace_bytes(B.DS4A_OP_SPARSE_ATTN_DECODE, U, 1, N_cap, 64), 1),
                     dtype=torch.uint8, device="cuda")
    B.ds4a_sparse_attn_decode(x["q"], x["rows"], torch.from_numpy(bad).cuda(), cnt, x["raw"], x["n_raw"], SCALE,
                              out, None, ws)
    st, flags = B.ds4a_get_device_status()
    assert st == B.DS4A_EDEVICE and flags & B.DS4A_DEV_BOUNDS
    for u, keep in [(0, np.delete(idx[0], 3)), (1, idx[1, 1:]), (2, idx[2])]:
        ro, _ = oracle.sparse_attention(u16(x["q"][u]), u16(x["rows"][u]), keep, u16(x["raw"][u]), np.arange(5),
                                        SCALE)
        check_output(out[u].cpu().numpy(), ro)
    device_ok()


# ----------------------------------------------------------------------------
# Whole decode step
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("q_scale", [1.0, 32.0])
def test_decode_step_small_ragged(q_scale):
    x = make_decode_inputs(2, 1000, device="cuda", seed=21, n_rows=[1000, 555], n_raw=[128, 37], q_scale=q_scale)
    st = run_decode(x, 512)
    for u in range(2):
        check_decode_unit(x, st, u, 512, SCALE)


def test_decode_step_fewer_rows_than_k():
    x = make_decode_inputs(2, 700, device="cuda", seed=22, n_rows=[300, 0], n_raw=[128, 10])
    st = run_decode(x, 512)
    for u in range(2):
        check_decode_unit(x, st, u, 512, SCALE)
    assert int(st.count[1, 0]) == 0


@pytest.mark.parametrize("name", ["decode_1x1024", "decode_8x16384"])
def test_workload_decode_full(name):
    wl = WORKLOADS[name]
    x = make_decode_inputs(wl.units, wl.n_rows, device="cuda", seed=wl.seed)
    st = run_decode(x, wl.top_k)
    with pool() as p:
        list(p.map(lambda u: check_decode_unit(x, st, u, wl.top_k, SCALE), range(wl.units)))


@pytest.mark.slow
def test_workload_longctx_4x262144_full():
    wl = WORKLOADS["longctx_4x262144"]
    x = make_decode_inputs(wl.units, wl.n_rows, device="cuda", seed=wl.seed, heavy_frac=wl.heavy_frac,
                           heavy_scale=wl.heavy_scale)
    st = run_decode(x, wl.top_k)
    with pool() as p:
        list(p.map(lambda u: check_decode_unit(x, st, u, wl.top_k, SCALE), range(wl.units)))


@pytest.mark.slow
def test_workload_decode_32x43x65536_sampled():
    wl = WORKLOADS["decode_32x43x65536"]
    x = make_decode_inputs(wl.units, wl.n_rows, device="cuda", seed=wl.seed)
    st = run_decode(x, wl.top_k)
    units = [0, 1, 42, 687, 1000, wl.units - 1]
    with pool() as p:
        list(p.map(lambda u: check_decode_unit(x, st, u, wl.top_k, SCALE), units))
    # the configuration the bench times: the fused score + select, bit-identical
    # to score-then-select over all 1,376 units
    sf = DecodeStep(wl.units, wl.n_rows, wl.top_k, fused=True)
    sf(x, SCALE)
    torch.cuda.synchronize()
    device_ok()
    assert torch.equal(sf.count, st.count) and torch.equal(sf.idx, st.idx) and torch.equal(sf.out, st.out)
    del x, st, sf
    torch.cuda.empty_cache()


# ----------------------------------------------------------------------------
# Prefill chunk
# ----------------------------------------------------------------------------

def check_prefill_query(x, st, t, top_k, scale, np_in):
    q, iq, w, ik, rows, row_pos, q_pos, raw = np_in
    n = int(x["n_rows"][0])
    res = oracle.prefill_query(t, q, iq, w, ik, rows, n, row_pos, q_pos, raw, x["raw_pos0"], top_k, scale)
    gpu_s = st.scores[0, t].cpu().numpy()
    tol = score_tolerance(iq[t], w[t], ik, n)
    check_scores(gpu_s[:n], res["scores"][:n], tol)
    cnt = int(st.count[0, t])
    gidx = st.idx[0, t].cpu().numpy()
    check_index_set(gidx, cnt, res["scores"][:n], top_k)
    assert np.all(row_pos[gidx[:cnt]] <= q_pos[t])
    ro, rl = oracle.sparse_attention(q[t], rows, gidx[:cnt], raw, res["window"], scale)
    return check_output(st.out[t].cpu().numpy(), ro, st.lse[t].cpu().numpy(), rl)


def prefill_numpy(x):
    return (u16(x["q"]), u16(x["iq"]), x["w"].cpu().numpy(), u16(x["ik"]), u16(x["rows"]),
            x["row_pos"].cpu().numpy(), x["q_pos"].cpu().numpy(), u16(x["raw"]))


@pytest.mark.parametrize("T,prior,top_k,q_scale", [(64, 100, 32, 1.0), (37, 300, 512, 1.0), (64, 600, 256, 32.0)])
def test_prefill_small(T, prior, top_k, q_scale):
    x = make_prefill_inputs(T, prior, device="cuda", seed=T + prior, q_scale=q_scale)
    st = PrefillStep(T, x["ik"].shape[0], top_k)
    st(x, SCALE)
    torch.cuda.synchronize()
    device_ok()
    np_in = prefill_numpy(x)
    with pool() as p:
        list(p.map(lambda t: check_prefill_query(x, st, t, top_k, SCALE, np_in), range(T)))


@pytest.mark.slow
def test_workload_prefill_2048x65536_sampled():
    wl = WORKLOADS["prefill_2048x65536"]
    x = make_prefill_inputs(wl.queries, wl.extra["prior_rows"], device="cuda", seed=wl.seed)
    st = PrefillStep(wl.queries, x["ik"].shape[0], wl.top_k)
    st(x, SCALE)
    torch.cuda.synchronize()
    device_ok()
    np_in = prefill_numpy(x)
    ts = [0, 1, 2, 3, 4, 127, 128, 1000, 2043, 2044, 2046, 2047]
    with pool() as p:
        list(p.map(lambda t: check_prefill_query(x, st, t, wl.top_k, SCALE, np_in), ts))


# ----------------------------------------------------------------------------
# Ratio-128 layers: dense attention over all compressed rows (no indexer)
# ----------------------------------------------------------------------------

def dense_case(U, N_cap, n_rows, n_raw, seed, q_scale=1.0):
    x = make_decode_inputs(U, N_cap, device="cuda", seed=seed, n_rows=n_rows, n_raw=n_raw, q_scale=q_scale,
                           with_indexer=False)
    out = torch.full((U, 64, 512), float("nan"), device="cuda")
    lse = torch.full((U, 64), float("nan"), device="cuda")
    nb = B.ds4a_workspace_bytes(B.DS4A_OP_DENSE_ATTN_DECODE, U, 1, N_cap, 0)
    ws = torch.empty(max(nb, 1), dtype=torch.uint8, device="cuda") if nb else None
    B.ds4a_dense_attn_decode(x["q"], x["rows"], x["n_rows"], x["raw"], x["n_raw"], SCALE, out, lse, ws)
    torch.cuda.synchronize()
    return x, out, lse


def check_dense_unit(x, out, lse, u):
    n, nw = int(x["n_rows"][u]), int(x["n_raw"][u])
    ro, rl = oracle.dense_attention(u16(x["q"][u]), u16(x["rows"][u]), n, u16(x["raw"][u]), nw, SCALE)
    if n + nw == 0:
        assert torch.all(out[u] == 0) and torch.all(torch.isneginf(lse[u]))
        return
    check_output(out[u].cpu().numpy(), ro)
    assert np.allclose(lse[u].cpu().numpy(), rl, atol=1e-4, rtol=1e-5), u


@pytest.mark.parametrize("q_scale", [1.0, 32.0])
def test_dense_attention_small_ragged(q_scale):
    # 160 units: one item per unit (no split); ragged row counts cover partial tiles
    n_rows = [1000, 513, 0, 64, 65, 1] + [777] * 154
    n_raw = [128, 7, 0, 0, 128, 1] + [33] * 154
    x, out, lse = dense_case(160, 1000, n_rows, n_raw, seed=31, q_scale=q_scale)
    device_ok()
    for u in range(8):
        check_dense_unit(x, out, lse, u)


@pytest.mark.parametrize("U", [3, 24])
def test_dense_attention_few_units_split_rows(U):
    # fewer units than SMs: each unit's rows are split over several CTAs and
    # merged by a second kernel (3 and 24 units)
    n_rows = ([6000, 4500, 129] * 8)[:U]
    n_raw = ([128, 0, 5] * 8)[:U]
    x, out, lse = dense_case(U, 6000, n_rows, n_raw, seed=32)
    device_ok()
    for u in range(min(U, 6)):
        check_dense_unit(x, out, lse, u)


def test_dense_attention_row_count_out_of_range_is_clamped_and_flagged():
    U, N_cap = 2, 300
    x = make_decode_inputs(U, N_cap, device="cuda", seed=33, n_raw=[10, 10], with_indexer=False)
    nr = torch.tensor([N_cap + 7, 120], dtype=torch.int32, device="cuda")
    out = torch.empty(U, 64, 512, device="cuda")
    nb = B.ds4a_workspace_bytes(B.DS4A_OP_DENSE_ATTN_DECODE, U, 1, N_cap, 0)
    ws = torch.empty(max(nb, 1), dtype=torch.uint8, device="cuda")
    B.ds4a_dense_attn_decode(x["q"], x["rows"], nr, x["raw"], x["n_raw"], SCALE, out, None, ws)
    st, flags = B.ds4a_get_device_status()
    assert st == B.DS4A_EDEVICE and flags & B.DS4A_DEV_BOUNDS
    for u, n in [(0, N_cap), (1, 120)]:
        ro, _ = oracle.dense_attention(u16(x["q"][u]), u16(x["rows"][u]), n, u16(x["raw"][u]), 10, SCALE)
        check_output(out[u].cpu().numpy(), ro)
    device_ok()


def test_sparse_count_out_of_range_is_clamped_and_flagged():
    U, N_cap, k = 160, 256, 64
    x = make_decode_inputs(U, N_cap, device="cuda", seed=34, n_raw=[3] * U)
    rng = np.random.default_rng(34)
    idx = np.stack([np.sort(rng.choice(N_cap, k, replace=False)) for _ in range(U)]).astype(np.int32)
    cnt = torch.full((U,), k, dtype=torch.int32, device="cuda")
    cnt[0] = k + 9
    out = torch.empty(U, 64, 512, device="cuda")
    ws = torch.empty(max(B.ds4a_workspace_bytes(B.DS4A_OP_SPARSE_ATTN_DECODE, U, 1, N_cap, k), 1),
                     dtype=torch.uint8, device="cuda")
    B.ds4a_sparse_attn_decode(x["q"], x["rows"], torch.from_numpy(idx).cuda(), cnt, x["raw"], x["n_raw"], SCALE,
                              out, None, ws)
    st, flags = B.ds4a_get_device_status()
    assert st == B.DS4A_EDEVICE and flags & B.DS4A_DEV_BOUNDS
    ro, _ = oracle.sparse_attention(u16(x["q"][0]), u16(x["rows"][0]), idx[0], u16(x["raw"][0]), np.arange(3), SCALE)
    check_output(out[0].cpu().numpy(), ro)
    device_ok()


@pytest.mark.slow
def test_workload_dense_sampled():
    wl = WORKLOADS["dense_32x20x8192"]
    x = make_decode_inputs(wl.units, wl.n_rows, device="cuda", seed=wl.seed, with_indexer=False)
    step = DenseStep(wl.units, wl.n_rows)
    step(x)
    torch.cuda.synchronize()
    device_ok()
    units = [0, 1, wl.units // 2, wl.units - 1]
    with pool() as p:
        list(p.map(lambda u: check_dense_unit(x, step.out, step.lse, u), units))
