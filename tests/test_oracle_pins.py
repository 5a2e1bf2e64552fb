"""Pins of the fp64 oracle to facts outside itself (CPU only).

Each test checks the oracle against something it does not compute the same
way: hand-worked values (tests/golden), closed forms, invariants, library
routines on special cases (numpy float16 casts, torch bfloat16 casts, torch's
scaled_dot_product_attention), and brute force on tiny inputs.  A plausible
slip in the oracle (dropped ReLU, wrong sign, transposed operand, wrong
head/row index, wrong tie order, wrong window edge) fails at least one.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
H, D, HI, DI = oracle.N_HEAD, oracle.HEAD_DIM, oracle.N_INDEXER_HEAD, oracle.INDEXER_DIM


def bf16_bits(x):
    return torch.as_tensor(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def f16_bits(x):
    return np.asarray(x, np.float64).astype(np.float16).view(np.uint16)


def bits_bf16_to_f64(b):
    return torch.from_numpy(np.asarray(b, np.uint16).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def rng(seed):
    return np.random.default_rng(seed)


def rand_bf16(r, shape, scale):
    return bf16_bits(r.standard_normal(shape) * scale)


# ----------------------------------------------------------------------------
# Storage formats
# ----------------------------------------------------------------------------

def test_bf16_decode_named_values():
    assert oracle.bf16_to_double(0x3F80) == 1.0
    assert oracle.bf16_to_double(0xC000) == -2.0
    assert oracle.bf16_to_double(0x0001) == 2.0 ** -133       # smallest subnormal
    assert oracle.bf16_to_double(0x7F7F) == (2 - 2 ** -7) * 2.0 ** 127
    assert oracle.bf16_to_double(0x7F80) == math.inf
    assert math.isnan(oracle.bf16_to_double(0x7FC0))


def test_bf16_decode_all_patterns_match_torch():
    bits = np.arange(1 << 16, dtype=np.uint16)
    ref = bits_bf16_to_f64(bits)
    got = np.array([oracle.bf16_to_double(int(b)) for b in bits])
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.array_equal(ref[~both_nan], got[~both_nan])


def test_f16_decode_all_patterns_match_numpy():
    bits = np.arange(1 << 16, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_double(int(b)) for b in bits])
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.array_equal(ref[~both_nan], got[~both_nan])


def test_f16_round_matches_numpy_cast():
    """The raw tier stores rows rounded to f16 (§3-1); numpy's float64->float16
    cast is a correctly rounded (ties-to-even) reference."""
    r = rng(1)
    xs = np.concatenate([
        r.standard_normal(20000) * 0.05,
        r.standard_normal(2000) * 3e4,
        r.standard_normal(2000) * 1e-6,                         # subnormal range
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e9, -1e9,
                  2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -14, 1.0 + 2.0 ** -11,
                  1.0 + 3 * 2.0 ** -11, 2049.0, 2051.0]),
    ])
    with np.errstate(over="ignore"):
        ref = xs.astype(np.float16).view(np.uint16)
    got = np.array([oracle.double_to_f16(float(x)) for x in xs], dtype=np.uint16)
    assert np.array_equal(ref, got)


# ----------------------------------------------------------------------------
# A1 indexer score
# ----------------------------------------------------------------------------

def _load_indexer_golden():
    iq = np.zeros((HI, DI)); w = np.zeros(HI); ik = np.zeros((3, DI)); score = {}
    for line in open(os.path.join(GOLDEN, "indexer_hand_worked.txt")):
        line = line.split("#")[0].split()
        if not line:
            continue
        k = line[0]
        if k == "iq":
            iq[int(line[1]), int(line[2])] = float(line[3])
        elif k == "w":
            w[int(line[1])] = float(line[2])
        elif k == "ik":
            ik[int(line[1]), int(line[2])] = float(line[3])
        elif k == "score":
            score[int(line[1])] = float(line[2])
    return iq, w, ik, np.array([score[i] for i in range(3)])


def test_indexer_hand_worked_golden():
    iq, w, ik, expect = _load_indexer_golden()
    s = oracle.indexer_score(bf16_bits(iq)[None], w[None].astype(np.float32), bf16_bits(ik), 3)
    assert np.array_equal(s[0], expect)


def test_indexer_zero_weights_give_zero():
    r = rng(2)
    iq = rand_bf16(r, (2, HI, DI), 1 / math.sqrt(DI))
    ik = rand_bf16(r, (40, DI), 1 / math.sqrt(DI))
    s = oracle.indexer_score(iq, np.zeros((2, HI), np.float32), ik, 40)
    assert np.all(s == 0.0)


def test_indexer_relu_identity():
    """relu(x) - relu(-x) = x, so s(k) - s(-k) = sum_h w_h (q_h . k): the linear
    part, computed here with numpy's matrix product.  A dropped or misplaced
    ReLU, or a sign slip, breaks it."""
    r = rng(3)
    iq = rand_bf16(r, (1, HI, DI), 1 / math.sqrt(DI))
    ik = rand_bf16(r, (33, DI), 1 / math.sqrt(DI))
    w = r.uniform(-1, 1, (1, HI)).astype(np.float32)
    s_pos = oracle.indexer_score(iq, w, ik, 33)[0]
    s_neg = oracle.indexer_score(iq, w, ik ^ np.uint16(0x8000), 33)[0]   # exact negation of bf16
    lin = (bits_bf16_to_f64(ik) @ bits_bf16_to_f64(iq[0]).T) @ w[0].astype(np.float64)
    np.testing.assert_allclose(s_pos - s_neg, lin, rtol=1e-12, atol=1e-12)


def test_indexer_single_head_is_relu_of_dot():
    r = rng(4)
    iq = np.zeros((1, HI, DI), np.uint16)
    iq[0, 7] = rand_bf16(r, DI, 1.0)
    w = np.zeros((1, HI), np.float32); w[0, 7] = 1.0
    ik = rand_bf16(r, (50, DI), 1.0)
    s = oracle.indexer_score(iq, w, ik, 50)[0]
    dots = bits_bf16_to_f64(ik) @ bits_bf16_to_f64(iq[0, 7])
    np.testing.assert_allclose(s, np.maximum(dots, 0), rtol=1e-12, atol=1e-13)
    assert np.any(dots < 0) and np.all(s[dots < 0] == 0)


def test_indexer_positive_homogeneity_and_query_independence():
    r = rng(5)
    iq = rand_bf16(r, (3, HI, DI), 1 / math.sqrt(DI))
    w = r.uniform(0, 1, (3, HI)).astype(np.float32)
    ik = rand_bf16(r, (20, DI), 1 / math.sqrt(DI))
    both = oracle.indexer_score(iq, w, ik, 20)
    for q in range(3):
        alone = oracle.indexer_score(iq[q:q + 1], w[q:q + 1], ik, 20)[0]
        assert np.array_equal(both[q], alone)
    ik2 = bf16_bits(bits_bf16_to_f64(ik) * 2.0)          # x2 is exact in bf16
    np.testing.assert_allclose(oracle.indexer_score(iq, w, ik2, 20), 2 * both, rtol=1e-13)


def test_indexer_visibility():
    r = rng(6)
    iq = rand_bf16(r, (2, HI, DI), 1 / math.sqrt(DI))
    w = r.uniform(0, 1, (2, HI)).astype(np.float32)
    ik = rand_bf16(r, (16, DI), 1 / math.sqrt(DI))
    full = oracle.indexer_score(iq, w, ik, 16)
    part = oracle.indexer_score(iq, w, ik, 11)
    assert np.all(part[:, 11:] == -np.inf) and np.array_equal(part[:, :11], full[:, :11])
    row_pos = np.arange(16, dtype=np.int32) * 4 + 3
    q_pos = np.array([20, 63], np.int32)
    causal = oracle.indexer_score(iq, w, ik, 16, q_pos=q_pos, row_pos=row_pos)
    for q in range(2):
        vis = row_pos <= q_pos[q]
        assert np.array_equal(causal[q][vis], full[q][vis])
        assert np.all(causal[q][~vis] == -np.inf)


# ----------------------------------------------------------------------------
# A2 top-k
# ----------------------------------------------------------------------------

def brute_topk(s, k):
    """Row r is selected iff fewer than k visible rows beat it, where r' beats r
    when s[r'] > s[r], or s[r'] == s[r] and r' < r.  Counted pairwise, O(N^2)."""
    vis = [r for r in range(len(s)) if s[r] != -np.inf]
    sel = []
    for r in vis:
        beaten_by = sum(1 for q in vis if s[q] > s[r] or (s[q] == s[r] and q < r))
        if beaten_by < k:
            sel.append(r)
    return np.array(sorted(sel), dtype=np.int32)


@pytest.mark.parametrize("seed", range(12))
def test_topk_matches_pairwise_brute_force(seed):
    r = rng(100 + seed)
    n = int(r.integers(1, 65))
    k = int(r.integers(1, 70))
    s = np.round(r.standard_normal(n) * 3) / 2          # many exact ties
    s[r.random(n) < 0.15] = -np.inf
    idx, kth = oracle.topk_select(s, k)
    expect = brute_topk(s, k)
    assert np.array_equal(idx, expect)
    if len(expect):
        assert kth == min(s[expect])
    else:
        assert kth == -np.inf


def test_topk_fewer_rows_than_k_selects_all_visible():
    s = np.array([3.0, -np.inf, 1.0, 2.0, -np.inf])
    idx, kth = oracle.topk_select(s, 512)
    assert list(idx) == [0, 2, 3] and kth == 1.0


def test_topk_all_equal_takes_lowest_indices():
    idx, kth = oracle.topk_select(np.full(1000, 0.5), 512)
    assert np.array_equal(idx, np.arange(512)) and kth == 0.5


def test_topk_permutation_equivariance():
    r = rng(7)
    s = r.standard_normal(300)
    perm = r.permutation(300)
    idx, _ = oracle.topk_select(s, 37)
    idx_p, _ = oracle.topk_select(s[perm], 37)
    assert np.array_equal(np.sort(perm[idx_p]), idx)


# ----------------------------------------------------------------------------
# A4 attention
# ----------------------------------------------------------------------------

def test_attention_two_rows_golden():
    vals = {}
    for line in open(os.path.join(GOLDEN, "attention_two_rows.txt")):
        line = line.split("#")[0].split()
        if line:
            vals[line[0]] = [float(v) for v in line[1:]]
    q = bf16_bits([vals["q"]])
    comp = bf16_bits([vals["x1"]])
    raw = f16_bits([vals["x2"]])
    out, lse = oracle.sparse_attention(q, comp, [0], raw, [0], vals["scale"][0])
    np.testing.assert_allclose(out[0], vals["out"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, vals["lse"], rtol=0, atol=1e-15)


def test_attention_single_row_returns_it():
    r = rng(8)
    q = rand_bf16(r, (H, D), 1 / math.sqrt(D))
    rows = rand_bf16(r, (5, D), 1 / math.sqrt(D))
    out, lse = oracle.sparse_attention(q, rows, [3], None, [], 0.3)
    x = bits_bf16_to_f64(rows[3])
    assert np.array_equal(out, np.broadcast_to(x, (H, D)))
    np.testing.assert_allclose(lse, 0.3 * (bits_bf16_to_f64(q) @ x), rtol=1e-13)


def test_attention_two_rows_closed_form():
    r = rng(9)
    q = rand_bf16(r, (H, D), 1.0)
    rows = rand_bf16(r, (2, D), 1.0)
    scale = 1 / math.sqrt(D)
    out, lse = oracle.sparse_attention(q, rows, [0, 1], None, [], scale)
    qd, x = bits_bf16_to_f64(q), bits_bf16_to_f64(rows)
    delta = scale * (qd @ (x[1] - x[0]))
    expect = (x[0][None] + np.exp(delta)[:, None] * x[1][None]) / (1 + np.exp(delta))[:, None]
    np.testing.assert_allclose(out, expect, rtol=1e-12, atol=1e-14)
    l0 = scale * (qd @ x[0])
    np.testing.assert_allclose(lse, l0 + np.log1p(np.exp(delta)), rtol=1e-12)


def test_attention_zero_scale_is_mean_and_equal_logits_lse():
    r = rng(10)
    q = rand_bf16(r, (H, D), 1.0)
    comp = rand_bf16(r, (30, D), 1.0)
    raw = f16_bits(r.standard_normal((9, D)))
    sel = [4, 7, 11, 29]
    out, lse = oracle.sparse_attention(q, comp, sel, raw, [0, 8, 2], 0.0)
    rows = np.concatenate([bits_bf16_to_f64(comp[sel]), raw[[0, 8, 2]].view(np.float16).astype(np.float64)])
    np.testing.assert_allclose(out, np.broadcast_to(rows.mean(0), (H, D)), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(lse, np.log(7.0), rtol=1e-14)


def test_attention_weights_sum_to_one():
    """Rows all equal to one vector c: any convex combination returns c."""
    r = rng(11)
    q = rand_bf16(r, (H, D), 3.0)
    c = r.standard_normal(D)
    comp = np.tile(bf16_bits(c), (6, 1))
    out, _ = oracle.sparse_attention(q, comp, [0, 1, 2, 3, 4, 5], None, [], 0.7)
    np.testing.assert_allclose(out, np.broadcast_to(bits_bf16_to_f64(comp[0]), (H, D)), rtol=1e-13)


def test_attention_dominant_row():
    q = bf16_bits([[1.0, 0, 0, 0]])
    comp = bf16_bits([[0, 1, 2, 3], [50, -1, 0.5, 7], [0, -2, -3, 1]])
    out, _ = oracle.sparse_attention(q, comp, [0, 1, 2], None, [], 1.0)
    np.testing.assert_allclose(out[0], bits_bf16_to_f64(comp[1]), rtol=0, atol=1e-18)   # other weights ~e^-50


def test_attention_permutation_and_tier_invariance():
    r = rng(13)
    q = rand_bf16(r, (H, D), 1 / math.sqrt(D) * 8)
    comp = rand_bf16(r, (40, D), 1 / math.sqrt(D))
    raw = f16_bits(r.standard_normal((20, D)) / math.sqrt(D))
    sel = np.array([1, 5, 9, 12, 30, 39], np.int32)
    rsel = np.array([0, 3, 4, 19], np.int32)
    out, lse = oracle.sparse_attention(q, comp, sel, raw, rsel, 0.1)
    p1, p2 = r.permutation(len(sel)), r.permutation(len(rsel))
    out2, lse2 = oracle.sparse_attention(q, comp, sel[p1], raw, rsel[p2], 0.1)
    np.testing.assert_allclose(out2, out, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(lse2, lse, rtol=1e-13)
    # A value exact in both bf16 and fp16 gives the same result in either tier.
    small = bf16_bits(np.round(r.standard_normal((3, D)) * 8) / 8)
    small_f16 = f16_bits(bits_bf16_to_f64(small))
    a, _ = oracle.sparse_attention(q, small, [0, 1, 2], None, [], 0.1)
    b, _ = oracle.sparse_attention(q, None, [], small_f16, [0, 1, 2], 0.1)
    np.testing.assert_allclose(a, b, rtol=1e-14, atol=0)


def test_attention_full_selection_matches_torch_sdpa():
    """top_k >= N: sparse attention is dense attention over all rows + window;
    torch's scaled_dot_product_attention (float64, CPU) is the reference."""
    r = rng(14)
    n_comp, n_raw = 37, 11
    q = rand_bf16(r, (H, D), 1 / math.sqrt(D) * 4)
    comp = rand_bf16(r, (n_comp, D), 1 / math.sqrt(D))
    raw = f16_bits(r.standard_normal((n_raw, D)) / math.sqrt(D))
    scale = 1 / math.sqrt(D)
    out, lse = oracle.sparse_attention(q, comp, np.arange(n_comp), raw, np.arange(n_raw), scale)
    X = torch.from_numpy(np.concatenate([bits_bf16_to_f64(comp), raw.view(np.float16).astype(np.float64)]))
    Qt = torch.from_numpy(bits_bf16_to_f64(q))
    ref = torch.nn.functional.scaled_dot_product_attention(
        Qt[None, None], X[None, None], X[None, None], scale=scale)[0, 0].numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-14)
    ref_lse = torch.logsumexp(scale * (Qt @ X.T), dim=-1).numpy()
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12)


def test_attention_empty_set():
    q = rand_bf16(rng(15), (H, D), 1.0)
    out, lse = oracle.sparse_attention(q, None, [], None, [], 0.1)
    assert np.all(out == 0) and np.all(lse == -np.inf)


# ----------------------------------------------------------------------------
# Composition: decode unit, prefill query, raw window
# ----------------------------------------------------------------------------

def test_prefill_window_brute_force():
    for raw_pos0, n_raw_rows in [(0, 50), (100, 300), (1000, 128), (5, 3)]:
        for p in range(raw_pos0 - 3, raw_pos0 + n_raw_rows + 140):
            expect = [i for i in range(n_raw_rows) if p - 128 < raw_pos0 + i <= p]
            got = oracle.prefill_window(p, raw_pos0, n_raw_rows)
            assert list(got) == expect, (p, raw_pos0, n_raw_rows)


def test_prefill_query_equals_restricted_decode():
    """A prefill query is a decode over the rows finalised at or before its
    position, with its own 128-token window; the first query of the chunk sees
    only rows finalised before the chunk."""
    r = rng(16)
    prior, T = 40, 24
    n_cap = prior + T // 4
    row_pos = (np.arange(n_cap) * 4 + 3).astype(np.int32)
    P0 = 4 * prior
    q_pos = (P0 + np.arange(T)).astype(np.int32)
    q = rand_bf16(r, (T, H, D), 1 / math.sqrt(D))
    iq = rand_bf16(r, (T, HI, DI), 1 / math.sqrt(DI))
    w = r.uniform(0, 1, (T, HI)).astype(np.float32)
    ik = rand_bf16(r, (n_cap, DI), 1 / math.sqrt(DI))
    rows = rand_bf16(r, (n_cap, D), 1 / math.sqrt(D))
    raw_pos0 = P0 - 128
    raw = f16_bits(r.standard_normal((128 + T, D)) / math.sqrt(D))
    k = 7
    for t in [0, 1, 5, 13, T - 1]:
        res = oracle.prefill_query(t, q, iq, w, ik, rows, n_cap, row_pos, q_pos, raw, raw_pos0, k, 1 / math.sqrt(D))
        p = q_pos[t]
        vis = np.nonzero(row_pos <= p)[0]
        assert np.all(row_pos[res["idx"]] <= p)
        if t == 0:
            assert np.all(res["idx"] < prior)
        # Same thing as a decode over the visible prefix (rows are position-sorted).
        n_vis = len(vis)
        assert np.array_equal(vis, np.arange(n_vis))
        win = np.arange(t + 1, t + 129)
        dec = oracle.decode_unit(q[t], iq[t], w[t], ik[:n_vis], rows[:n_vis], n_vis, raw[win], 128, k, 1 / math.sqrt(D))
        assert np.array_equal(dec["idx"], res["idx"])
        assert np.array_equal(res["window"], win)
        np.testing.assert_allclose(dec["out"], res["out"], rtol=1e-13, atol=1e-16)


# ----------------------------------------------------------------------------
# Cache producer: compressor pooling and the raw-window push
# ----------------------------------------------------------------------------

def test_compressor_pool_two_rows_golden():
    vals = {}
    for line in open(os.path.join(GOLDEN, "compressor_pool_two_rows.txt")):
        line = line.split("#")[0].split()
        if line:
            vals[line[0]] = [float(v) for v in line[1:]]
    kv = np.array([vals["kv0"], vals["kv1"]], np.float32)
    sc = np.array([vals["s0"], vals["s1"]], np.float32)
    np.testing.assert_allclose(oracle.compressor_pool(kv, sc), vals["out"], rtol=0, atol=1e-7)


@pytest.mark.parametrize("ratio", [1, 4, 128])
def test_compressor_pool_equal_scores_give_the_mean_and_ratio_one_the_row(ratio):
    r = rng(60 + ratio)
    kv = r.standard_normal((ratio, 24)).astype(np.float32)
    sc = np.broadcast_to(r.standard_normal(24).astype(np.float32), (ratio, 24))
    out = oracle.compressor_pool(kv, sc)
    np.testing.assert_allclose(out, kv.astype(np.float64).mean(axis=0), rtol=1e-13, atol=1e-14)
    if ratio == 1:
        assert np.array_equal(out, kv[0].astype(np.float64))


def test_compressor_pool_matches_scipy_softmax_and_is_shift_invariant():
    special = pytest.importorskip("scipy.special")
    r = rng(70)
    for ratio in (4, 128):
        kv = r.standard_normal((ratio, 40)).astype(np.float32)
        # scores on a 2^-10 grid, |s| < 16: adding 64 below is exact in fp32
        sc = (np.round(np.clip(3 * r.standard_normal((ratio, 40)), -15, 15) * 1024) / 1024).astype(np.float32)
        ref = (special.softmax(sc.astype(np.float64), axis=0) * kv.astype(np.float64)).sum(axis=0)
        out = oracle.compressor_pool(kv, sc)
        np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)
        # adding one constant to a column's scores leaves it unchanged
        shifted = oracle.compressor_pool(kv, sc + np.float32(64.0))
        np.testing.assert_allclose(shifted, out, rtol=1e-12, atol=1e-13)


def test_compressor_pool_dominant_score_and_masked_column():
    r = rng(71)
    kv = r.standard_normal((4, 8)).astype(np.float32)
    sc = r.standard_normal((4, 8)).astype(np.float32)
    sc[2, :] += 200.0                                   # row 2 dominates every column
    out = oracle.compressor_pool(kv, sc)
    np.testing.assert_allclose(out, kv[2].astype(np.float64), rtol=0, atol=1e-60)
    sc[:, 5] = -np.inf                                  # no finite score: the column is 0
    out = oracle.compressor_pool(kv, sc)
    assert out[5] == 0.0
    # the pooled value lies within the column's range (a convex combination)
    sc = r.standard_normal((4, 8)).astype(np.float32)
    out = oracle.compressor_pool(kv, sc)
    assert np.all(out >= kv.min(axis=0) - 1e-12) and np.all(out <= kv.max(axis=0) + 1e-12)


def test_push_raw_keeps_the_last_128_rows_rounded_through_f16():
    r = rng(72)
    dim, cap = 16, oracle.N_SWA
    ring, n = np.zeros((cap, dim), np.uint16), 0
    pushed = []
    for t in range(300):
        kv = (r.standard_normal(dim) * 1e3).astype(np.float32)
        if t == 7:
            kv[:4] = [65520.0, -65520.0, 1e-8, 2.0 ** -24 * 1.5]   # overflow, underflow, subnormal tie
        ring, n = oracle.push_raw(ring, n, kv)
        pushed.append(kv.astype(np.float16).view(np.uint16))      # numpy's f32 -> f16 cast (round to nearest even)
        want = pushed[-cap:]
        assert n == len(want)
        assert np.array_equal(ring[:n], np.array(want)), t


# ----------------------------------------------------------------------------
# FP8 row store (E4M3 codes + one power-of-two scale per row)
# ----------------------------------------------------------------------------

def _torch_e4m3_decode(codes):
    """torch's own float8_e4m3fn decoding, an implementation independent of the oracle."""
    t = torch.from_numpy(np.asarray(codes, dtype=np.uint8).copy()).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def test_e4m3_decode_named_values():
    assert oracle.e4m3_to_double(0x38) == 1.0
    assert oracle.e4m3_to_double(0xB8) == -1.0
    assert oracle.e4m3_to_double(0x40) == 2.0
    assert oracle.e4m3_to_double(0x3F) == 1.875
    assert oracle.e4m3_to_double(0x7E) == 448.0               # largest finite
    assert oracle.e4m3_to_double(0x08) == 2.0 ** -6           # smallest normal
    assert oracle.e4m3_to_double(0x01) == 2.0 ** -9           # smallest subnormal
    assert oracle.e4m3_to_double(0x07) == 7 * 2.0 ** -9
    assert oracle.e4m3_to_double(0x00) == 0.0
    assert math.copysign(1.0, oracle.e4m3_to_double(0x80)) == -1.0
    assert math.isnan(oracle.e4m3_to_double(0x7F)) and math.isnan(oracle.e4m3_to_double(0xFF))


def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = _torch_e4m3_decode(codes)
    got = np.array([oracle.e4m3_to_double(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])
    assert not np.isinf(got).any()                               # the format has no infinities
    pos = got[:0x7F]
    assert np.all(np.diff(pos) > 0)                              # codes 0x00..0x7E increase strictly


def _e4m3_grid():
    vals = np.array([oracle.e4m3_to_double(c) for c in range(0x7F)])
    return vals                                                   # 0, 2^-9, ..., 448


def test_e4m3_encode_matches_torch_in_range():
    """Round to nearest, ties to even, against torch's float32 -> float8_e4m3fn
    cast on values it converts with one rounding: float32 values below 448,
    including every exact grid value and every midpoint between neighbours."""
    r = rng(40)
    grid = _e4m3_grid()
    mids = (grid[:-1] + grid[1:]) / 2
    rand = np.exp2(r.uniform(-13, np.log2(448), 4000)) * r.choice([-1, 1], 4000)
    xs = np.concatenate([grid, -grid, mids, -mids, rand]).astype(np.float32)
    xs = xs[np.abs(xs) < 448]
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.double_to_e4m3(float(x)) for x in xs], dtype=np.uint8)
    bad = np.nonzero(ref != got)[0]
    assert bad.size == 0, [(float(xs[i]), int(ref[i]), int(got[i])) for i in bad[:5]]


def test_e4m3_encode_saturates_rounds_ties_to_even_and_keeps_nan():
    assert oracle.double_to_e4m3(448.0) == 0x7E
    for big in (449.0, 464.0, 480.0, 1e6, math.inf):
        assert oracle.double_to_e4m3(big) == 0x7E
        assert oracle.double_to_e4m3(-big) == 0xFE
    assert oracle.double_to_e4m3(math.nan) == 0x7F
    assert oracle.double_to_e4m3(2.0 ** -10) == 0x00               # half the smallest subnormal: tie to 0
    assert oracle.double_to_e4m3(2.0 ** -10 * 1.001) == 0x01
    assert oracle.double_to_e4m3(3 * 2.0 ** -10) == 0x02           # tie between codes 1 and 2 -> even
    assert oracle.double_to_e4m3(1.0625) == 0x38                   # tie between 1 and 1.125 -> 1
    assert oracle.double_to_e4m3(1.1875) == 0x3A                   # tie between 1.125 and 1.25 -> 1.25
    assert oracle.double_to_e4m3(-0.0) == 0x80


def test_fp8_row_exponent_is_the_smallest_fitting_power_of_two():
    assert oracle.fp8_row_exponent(448.0) == 0
    assert oracle.fp8_row_exponent(448.0 * (1 + 2.0 ** -30)) == 1
    assert oracle.fp8_row_exponent(1.0) == -8
    assert oracle.fp8_row_exponent(0.0) == 0
    assert oracle.fp8_row_exponent(math.inf) == 0
    assert oracle.fp8_row_exponent(1e-40) == -126                 # clamped: the scale stays a normal fp32
    r = rng(41)
    for amax in np.exp2(r.uniform(-100, 100, 500)):
        e = oracle.fp8_row_exponent(float(amax))
        assert amax <= 448.0 * 2.0 ** e and not amax <= 448.0 * 2.0 ** (e - 1)


def test_quantize_rows_fp8_picks_the_nearest_scaled_code_by_brute_force():
    r = rng(42)
    rows = []
    for mag in (1e-3, 0.05, 1.0, 300.0, 7e4):
        rows.append(r.standard_normal(64) * mag)
    rows.append(np.zeros(64))
    special = r.standard_normal(64)
    special[3] = np.nan                                            # NaN does not set the scale
    special[5] = -0.0
    rows.append(special)
    x = np.array(rows, dtype=np.float32)
    codes, scale = oracle.quantize_rows_fp8(x)
    grid = _e4m3_grid()
    cand = np.concatenate([grid, -grid[1:]])
    cand_codes = np.concatenate([np.arange(0x7F), 0x80 | np.arange(1, 0x7F)])
    for i, row in enumerate(x.astype(np.float64)):
        amax = np.nanmax(np.abs(row))
        e = oracle.fp8_row_exponent(amax)
        assert scale[i] == 2.0 ** e
        for d, v in enumerate(row):
            c = int(codes[i, d])
            if np.isnan(v):
                assert c == 0x7F
                continue
            dist = np.abs(cand * scale[i] - v)
            best = cand_codes[dist == dist.min()]
            if v == 0:
                assert c in (0x00, 0x80)
                continue
            # nearest; a tie goes to the code with an even last bit
            assert c in best and (best.size == 1 or c % 2 == 0), (i, d, v, c, best)


def test_fp8_attention_equals_attention_on_the_stored_values():
    """Attention over the FP8 store equals the already pinned attention over
    bf16 rows holding the same values (every E4M3 value times a power of two in
    range is a bf16 value)."""
    r = rng(43)
    N, D = 40, 512
    x = (r.standard_normal((N, D)) / math.sqrt(D)).astype(np.float32)
    x[7] *= 300.0
    codes, scale = oracle.quantize_rows_fp8(x)
    vals = oracle.fp8_rows_to_double(codes, scale)
    bits = bf16_bits(vals)
    assert np.array_equal(bits_bf16_to_f64(bits), vals)              # exact in bf16
    q = rand_bf16(r, (64, D), 1.0)
    raw = f16_bits(r.standard_normal((9, D)) / math.sqrt(D))
    sel = np.array([3, 7, 0, 39, 12], dtype=np.int32)
    raw_sel = np.arange(9, dtype=np.int32)
    o8, l8 = oracle.sparse_attention_fp8(q, codes, scale, sel, raw, raw_sel, 1 / math.sqrt(D))
    ob, lb = oracle.sparse_attention(q, bits, sel, raw, raw_sel, 1 / math.sqrt(D))
    assert np.array_equal(o8, ob) and np.array_equal(l8, lb)
