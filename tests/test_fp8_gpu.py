"""Parity of the FP8 row store ("DwarfStar(ds4.c) のアーキテクチャを読む" §3-2:
the compressed row's FP8 quantisation round trip, read as E4M3 codes with one
power-of-two scale per row) with the fp64 oracle, through the C ABI:

  * ds4a_rows_to_fp8: codes and scales bit-exact against the oracle's
    quantiser (integer outputs);
  * attention over the FP8 store (decode and prefill): within the attention
    tolerances of the oracle run on the device's own selected set, and
    bit-identical to the bf16 path on rows holding the same values (the FP8
    gather expands every row to exactly those bf16 values).

The codes fed to the attention come from the oracle's quantiser on the CPU;
the device's quantiser is checked on its own."""
import math

import numpy as np
import pytest
import torch

import oracle
from deepseek_v4_sparse_indexer_gb300 import DecodeStep, PrefillStep, _binding as B
from deepseek_v4_sparse_indexer_gb300.workloads import (WORKLOADS, decode_rows_fp32_chunks, make_decode_inputs,
                                                        make_prefill_inputs, prefill_rows_fp32_chunks)
from tests.parity_util import check_index_set, check_output, check_scores, pool, score_tolerance, u16

pytestmark = pytest.mark.gpu

SCALE = 1.0 / math.sqrt(512)


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    yield
    torch.cuda.synchronize()


def device_ok():
    st, flags = B.ds4a_get_device_status()
    assert st == B.DS4A_OK and flags == 0, f"device status flags {flags}"


def quantize_on_device(x):
    x = x.contiguous().cuda()
    codes = torch.empty(x.shape[0], 512, dtype=torch.uint8, device="cuda")
    scale = torch.empty(x.shape[0], dtype=torch.float32, device="cuda")
    B.ds4a_rows_to_fp8(x, codes, scale)
    torch.cuda.synchronize()
    device_ok()
    return codes.cpu().numpy(), scale.cpu().numpy()


def special_rows():
    r = np.random.default_rng(50)
    rows = [r.standard_normal(512) * m for m in (1e-30, 1e-3, 0.044, 1.0, 448.0, 3e4, 1e37)]
    z = np.zeros(512)
    rows.append(z)
    a = r.standard_normal(512)
    a[17] = np.nan
    a[18] = -0.0
    rows.append(a)
    b = r.standard_normal(512)
    b[100] = np.inf                                 # amax infinite: scale 1, inf saturates
    b[101] = -np.inf
    rows.append(b)
    c = r.standard_normal(512) * 1e-3
    c[:64] = 448.0 * 2.0 ** -10 * (1 + np.arange(64) / 64)   # amax near a power-of-two boundary
    rows.append(c)
    d = np.full(512, np.nan)                        # every element NaN: amax 0, scale 1
    rows.append(d)
    e = np.exp2(r.uniform(-140, -127, 512)) * r.choice([-1, 1], 512)   # fp32 subnormals
    rows.append(e)
    return np.array(rows, dtype=np.float32)


@pytest.mark.parametrize("n", [1, 5, 1003])
def test_rows_to_fp8_bit_exact(n):
    r = np.random.default_rng(51 + n)
    x = (r.standard_normal((n, 512)) * np.exp2(r.uniform(-20, 20, (n, 1)))).astype(np.float32)
    if n > 20:
        sp = special_rows()
        x[:sp.shape[0]] = sp
    gc, gs = quantize_on_device(torch.from_numpy(x))
    oc, os_ = oracle.quantize_rows_fp8(x)
    assert np.array_equal(gs.view(np.uint32), os_.view(np.uint32)), np.nonzero(gs.view(np.uint32) != os_.view(np.uint32))
    bad = np.argwhere(gc != oc)
    assert bad.size == 0, [(int(i), int(j), float(x[i, j]), int(gc[i, j]), int(oc[i, j])) for i, j in bad[:5]]


def test_rows_to_fp8_zero_rows_is_a_no_op():
    B.ds4a_rows_to_fp8(torch.empty(0, 512, device="cuda"), torch.empty(0, 512, dtype=torch.uint8, device="cuda"),
                       torch.empty(0, device="cuda"))
    device_ok()


def fp8_store_from_oracle(chunks, shape):
    """Oracle-quantised FP8 store of the workload's fp32 rows: (codes, scales)
    as CUDA tensors of the given leading shape."""
    codes, scales = [], []
    for _, c in chunks:
        cc, ss = oracle.quantize_rows_fp8(c.numpy())
        codes.append(cc)
        scales.append(ss)
    codes = np.concatenate(codes).reshape(*shape, 512)
    scales = np.concatenate(scales).reshape(*shape)
    return torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda()


def stored_values_bf16(codes, scales):
    """The FP8 store's values as bf16 rows (exact: at most four significant bits)."""
    v = oracle.fp8_rows_to_double(codes.cpu().numpy().reshape(-1, 512), scales.cpu().numpy().reshape(-1))
    t = torch.from_numpy(v).to(torch.bfloat16)
    assert torch.equal(t.double(), torch.from_numpy(v)), "stored values not exact in bf16"
    return t.view(*codes.shape).cuda()


def fp8_attention_case(U, N_cap, top_k, seed, n_raw=None, q_scale=1.0):
    rng = np.random.default_rng(seed)
    x = make_decode_inputs(U, N_cap, device="cuda", seed=seed, q_scale=q_scale, with_indexer=False,
                           with_rows=False, n_raw=n_raw if n_raw is not None else list(rng.integers(0, 129, U)))
    rows8, rscale = fp8_store_from_oracle(decode_rows_fp32_chunks(U, N_cap, seed=seed), (U, N_cap))
    idx = np.full((U, top_k), -1, np.int32)
    cnt = rng.integers(0, top_k + 1, U).astype(np.int32)
    cnt[0] = min(top_k, N_cap)
    for u in range(U):
        cnt[u] = min(cnt[u], N_cap)
        idx[u, :cnt[u]] = np.sort(rng.choice(N_cap, size=cnt[u], replace=False))
    idx_t, cnt_t = torch.from_numpy(idx).cuda(), torch.from_numpy(cnt).cuda()
    nb = B.ds4a_workspace_bytes(B.DS4A_OP_SPARSE_ATTN_DECODE, U, 1, N_cap, top_k)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda") if nb else None
    out = torch.empty(U, 64, 512, device="cuda")
    lse = torch.empty(U, 64, device="cuda")
    B.ds4a_sparse_attn_decode_fp8(x["q"], rows8, rscale, idx_t, cnt_t, x["raw"], x["n_raw"], SCALE, out, lse, ws)
    torch.cuda.synchronize()
    device_ok()
    # the bf16 path on rows holding the same values: bit-identical
    rows16 = stored_values_bf16(rows8, rscale)
    out16 = torch.empty_like(out)
    lse16 = torch.empty_like(lse)
    B.ds4a_sparse_attn_decode(x["q"], rows16, idx_t, cnt_t, x["raw"], x["n_raw"], SCALE, out16, lse16, ws)
    torch.cuda.synchronize()
    device_ok()
    assert torch.equal(out, out16) and torch.equal(lse, lse16)
    codes_np, scale_np = rows8.cpu().numpy(), rscale.cpu().numpy()

    def one(u):
        nraw = int(x["n_raw"][u])
        ro, rl = oracle.sparse_attention_fp8(u16(x["q"][u]), codes_np[u], scale_np[u], idx[u, :cnt[u]],
                                             u16(x["raw"][u]), np.arange(nraw), SCALE)
        return check_output(out[u].cpu().numpy(), ro, lse[u].cpu().numpy(), rl)

    with pool() as p:
        return list(p.map(one, range(U)))


@pytest.mark.parametrize("q_scale", [1.0, 32.0])
def test_fp8_attention_split_rows_few_units(q_scale):
    fp8_attention_case(3, 2000, 512, seed=61, q_scale=q_scale)


def test_fp8_attention_one_cta_per_unit():
    fp8_attention_case(160, 700, 512, seed=62)


def test_fp8_attention_raw_window_extremes_odd_k_and_tiny_cache():
    fp8_attention_case(4, 300, 100, seed=63, n_raw=[0, 1, 127, 128])
    fp8_attention_case(2, 37, 64, seed=64, n_raw=[5, 0])          # fewer rows than top_k


def test_fp8_attention_out_of_range_index_is_masked_and_flagged():
    U, N_cap, k = 2, 256, 64
    x = make_decode_inputs(U, N_cap, device="cuda", seed=65, with_indexer=False, with_rows=False, n_raw=[3, 3])
    rows8, rscale = fp8_store_from_oracle(decode_rows_fp32_chunks(U, N_cap, seed=65), (U, N_cap))
    rng = np.random.default_rng(65)
    idx = np.stack([np.sort(rng.choice(N_cap, k, replace=False)) for _ in range(U)]).astype(np.int32)
    bad = idx.copy()
    bad[0, 5] = N_cap + 3
    cnt = torch.full((U,), k, dtype=torch.int32, device="cuda")
    out = torch.empty(U, 64, 512, device="cuda")
    ws = torch.empty(max(B.ds4a_workspace_bytes(B.DS4A_OP_SPARSE_ATTN_DECODE, U, 1, N_cap, k), 1),
                     dtype=torch.uint8, device="cuda")
    B.ds4a_sparse_attn_decode_fp8(x["q"], rows8, rscale, torch.from_numpy(bad).cuda(), cnt, x["raw"], x["n_raw"],
                                  SCALE, out, None, ws)
    st, flags = B.ds4a_get_device_status()
    assert st == B.DS4A_EDEVICE and flags & B.DS4A_DEV_BOUNDS
    keep = np.delete(idx[0], 5)
    ro, _ = oracle.sparse_attention_fp8(u16(x["q"][0]), rows8[0].cpu().numpy(), rscale[0].cpu().numpy(), keep,
                                        u16(x["raw"][0]), np.arange(3), SCALE)
    check_output(out[0].cpu().numpy(), ro)
    device_ok()


def test_fp8_decode_step_end_to_end():
    U, N_cap, k = 5, 1500, 512
    x = make_decode_inputs(U, N_cap, device="cuda", seed=66, with_rows=False, n_rows=[1500, 1499, 600, 512, 7])
    x["rows8"], x["row_scale"] = fp8_store_from_oracle(decode_rows_fp32_chunks(U, N_cap, seed=66), (U, N_cap))
    st = DecodeStep(U, N_cap, k, fp8=True)
    st(x, SCALE)
    torch.cuda.synchronize()
    device_ok()
    codes_np, scale_np = x["rows8"].cpu().numpy(), x["row_scale"].cpu().numpy()

    def one(u):
        n = int(x["n_rows"][u])
        iq, w, ik = u16(x["iq"][u]), x["w"][u].cpu().numpy(), u16(x["ik"][u, :n])
        ref = oracle.indexer_score(iq[None], w[None], ik, n)[0][:n]
        check_scores(st.scores[u, 0, :n].cpu().numpy(), ref, score_tolerance(iq, w, ik, n))
        cnt = int(st.count[u, 0])
        gidx = st.idx[u, 0].cpu().numpy()
        check_index_set(gidx, cnt, ref, k)
        ro, rl = oracle.sparse_attention_fp8(u16(x["q"][u]), codes_np[u], scale_np[u], gidx[:cnt], u16(x["raw"][u]),
                                             np.arange(int(x["n_raw"][u])), SCALE)
        return check_output(st.out[u].cpu().numpy(), ro, st.lse[u].cpu().numpy(), rl)

    with pool() as p:
        list(p.map(one, range(U)))


@pytest.mark.parametrize("T,prior", [(64, 1000), (129, 37)])
def test_fp8_prefill_matches_oracle(T, prior):
    x = make_prefill_inputs(T, prior, device="cuda", seed=T + prior + 7, with_rows=False)
    n_cap = x["ik"].shape[0]
    x["rows8"], x["row_scale"] = fp8_store_from_oracle(prefill_rows_fp32_chunks(n_cap, seed=T + prior + 7), (n_cap,))
    st = PrefillStep(T, n_cap, 512, fp8=True)
    st(x, SCALE)
    torch.cuda.synchronize()
    device_ok()
    q, iq, w, ik = u16(x["q"]), u16(x["iq"]), x["w"].cpu().numpy(), u16(x["ik"])
    row_pos, q_pos, raw = x["row_pos"].cpu().numpy(), x["q_pos"].cpu().numpy(), u16(x["raw"])
    codes_np, scale_np = x["rows8"].cpu().numpy(), x["row_scale"].cpu().numpy()
    n = int(x["n_rows"][0])

    def one(t):
        p = int(q_pos[t])
        s = oracle.indexer_score(iq[t:t + 1], w[t:t + 1], ik, n, q_pos=np.array([p], np.int32), row_pos=row_pos)[0]
        check_scores(st.scores[0, t, :n].cpu().numpy(), s[:n], score_tolerance(iq[t], w[t], ik, n))
        cnt = int(st.count[0, t])
        gidx = st.idx[0, t].cpu().numpy()
        check_index_set(gidx, cnt, s[:n], 512)
        win = oracle.prefill_window(p, x["raw_pos0"], raw.shape[0])
        ro, rl = oracle.sparse_attention_fp8(q[t], codes_np, scale_np, gidx[:cnt], raw, win, SCALE)
        return check_output(st.out[t].cpu().numpy(), ro, st.lse[t].cpu().numpy(), rl)

    with pool() as p:
        list(p.map(one, range(T)))


@pytest.mark.slow
def test_workload_decode_fp8_sampled():
    """The benchmarked FP8 decode workload, store built by the device quantiser
    (checked bit-exact against the oracle's on sampled units)."""
    wl = WORKLOADS["decode_fp8_32x43x65536"]
    x = make_decode_inputs(wl.units, wl.n_rows, device="cuda", seed=wl.seed, with_rows=False)
    rows8 = torch.empty(wl.units, wl.n_rows, 512, dtype=torch.uint8, device="cuda")
    rscale = torch.empty(wl.units, wl.n_rows, dtype=torch.float32, device="cuda")
    r8, rs = rows8.view(-1, 512), rscale.view(-1)
    units = [0, 1, wl.units // 2, wl.units - 1]
    first = {}                                       # fp32 rows of the sampled units, for the oracle
    for r0, c in decode_rows_fp32_chunks(wl.units, wl.n_rows, device="cuda", seed=wl.seed):
        B.ds4a_rows_to_fp8(c, r8[r0:r0 + c.shape[0]], rs[r0:r0 + c.shape[0]])
        u0, u1 = r0 // wl.n_rows, (r0 + c.shape[0]) // wl.n_rows
        for u in units:
            if u0 <= u < u1:
                first[u] = c[(u - u0) * wl.n_rows:(u - u0 + 1) * wl.n_rows].cpu().numpy()
    x["rows8"], x["row_scale"] = rows8, rscale
    st = DecodeStep(wl.units, wl.n_rows, wl.top_k, fp8=True)
    st(x, SCALE)
    torch.cuda.synchronize()
    device_ok()
    for u in units:
        oc, os_ = oracle.quantize_rows_fp8(first[u])
        assert np.array_equal(rows8[u].cpu().numpy(), oc) and np.array_equal(rscale[u].cpu().numpy(), os_)
        n = wl.n_rows
        iq, w, ik = u16(x["iq"][u]), x["w"][u].cpu().numpy(), u16(x["ik"][u])
        ref = oracle.indexer_score(iq[None], w[None], ik, n)[0]
        cnt = int(st.count[u, 0])
        gidx = st.idx[u, 0].cpu().numpy()
        check_index_set(gidx, cnt, ref, wl.top_k)
        ro, rl = oracle.sparse_attention_fp8(u16(x["q"][u]), oc, os_, gidx[:cnt], u16(x["raw"][u]), np.arange(128),
                                             SCALE)
        check_output(st.out[u].cpu().numpy(), ro, st.lse[u].cpu().numpy(), rl)


@pytest.mark.slow
def test_workload_prefill_fp8_sampled():
    """The benchmarked FP8 prefill chunk (2,048 queries over 65,536 + 512 rows),
    store built by the device quantiser, sampled queries against the oracle
    (the first and last query and spread ones; the store of the rows they
    select checked bit-exact against the oracle's quantiser)."""
    wl = WORKLOADS["prefill_fp8_2048x65536"]
    x = make_prefill_inputs(wl.queries, wl.extra["prior_rows"], device="cuda", seed=wl.seed, with_rows=False)
    n_cap = x["ik"].shape[0]
    rows8 = torch.empty(n_cap, 512, dtype=torch.uint8, device="cuda")
    rscale = torch.empty(n_cap, dtype=torch.float32, device="cuda")
    f32 = []
    for r0, c in prefill_rows_fp32_chunks(n_cap, device="cuda", seed=wl.seed):
        B.ds4a_rows_to_fp8(c, rows8[r0:r0 + c.shape[0]], rscale[r0:r0 + c.shape[0]])
        f32.append(c.cpu())
    x["rows8"], x["row_scale"] = rows8, rscale
    st = PrefillStep(wl.queries, n_cap, wl.top_k, fp8=True)
    st(x, SCALE)
    torch.cuda.synchronize()
    device_ok()
    q, iq, w, ik = u16(x["q"]), u16(x["iq"]), x["w"].cpu().numpy(), u16(x["ik"])
    row_pos, q_pos, raw = x["row_pos"].cpu().numpy(), x["q_pos"].cpu().numpy(), u16(x["raw"])
    codes_np, scale_np = rows8.cpu().numpy(), rscale.cpu().numpy()
    f32 = torch.cat(f32).numpy()
    n = int(x["n_rows"][0])
    queries = [0, 1, 700, 1023, 1536, wl.queries - 1]

    def one(t):
        p = int(q_pos[t])
        s = oracle.indexer_score(iq[t:t + 1], w[t:t + 1], ik, n, q_pos=np.array([p], np.int32), row_pos=row_pos)[0]
        check_scores(st.scores[0, t, :n].cpu().numpy(), s[:n], score_tolerance(iq[t], w[t], ik, n))
        cnt = int(st.count[0, t])
        gidx = st.idx[0, t].cpu().numpy()
        check_index_set(gidx, cnt, s[:n], wl.top_k)
        oc, os_ = oracle.quantize_rows_fp8(f32[gidx[:cnt]])
        assert np.array_equal(codes_np[gidx[:cnt]], oc) and np.array_equal(scale_np[gidx[:cnt]], os_)
        win = oracle.prefill_window(p, x["raw_pos0"], raw.shape[0])
        ro, rl = oracle.sparse_attention_fp8(q[t], codes_np, scale_np, gidx[:cnt], raw, win, SCALE)
        return check_output(st.out[t].cpu().numpy(), ro, st.lse[t].cpu().numpy(), rl)

    with pool() as p:
        list(p.map(one, queries))
