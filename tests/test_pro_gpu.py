"""The Pro shape ("DwarfStar(ds4.c) のアーキテクチャを読む" §2: 128 query heads,
indexer top_k 1,024; one KV head of 512-d rows, 128-row raw window as in
Flash) through the C ABI, against the fp64 oracle: the decode step (few units,
split rows; many units), a prefill chunk, dense attention and sampled units of
the Pro workload."""
import numpy as np
import pytest
import torch

import oracle
from deepseek_v4_sparse_indexer_gb300 import DecodeStep, DenseStep, PrefillStep
from deepseek_v4_sparse_indexer_gb300.workloads import WORKLOADS, make_decode_inputs, make_prefill_inputs
from tests.parity_util import check_output, pool, u16
from tests.test_parity_gpu import SCALE, check_decode_unit, check_prefill_query, device_ok

pytestmark = pytest.mark.gpu
H, K = 128, 1024


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    yield
    torch.cuda.synchronize()


def run_decode(x, top_k=K):
    U, N_cap = x["ik"].shape[:2]
    st = DecodeStep(U, N_cap, top_k, n_head=H)
    st(x, SCALE)
    torch.cuda.synchronize()
    device_ok()
    return st


def test_pro_decode_step_few_units_split_rows():
    x = make_decode_inputs(3, 3000, device="cuda", seed=41, n_rows=[3000, 1500, 700], n_raw=[128, 20, 0],
                           n_head=H)
    st = run_decode(x)
    for u in range(3):
        check_decode_unit(x, st, u, K, SCALE)


def test_pro_decode_step_many_units():
    U = 160
    n_rows = [1200, 1025, 1024, 999] + [1200] * (U - 4)
    n_raw = [128, 1, 77, 0] + [128] * (U - 4)
    x = make_decode_inputs(U, 1200, device="cuda", seed=42, n_rows=n_rows, n_raw=n_raw, n_head=H)
    st = run_decode(x)
    with pool() as p:
        list(p.map(lambda u: check_decode_unit(x, st, u, K, SCALE), [0, 1, 2, 3, 100, U - 1]))


def test_pro_prefill_chunk():
    T = 64
    x = make_prefill_inputs(T, 1500, device="cuda", seed=43, n_head=H)
    st = PrefillStep(T, x["ik"].shape[0], K, n_head=H)
    st(x, SCALE)
    torch.cuda.synchronize()
    device_ok()
    np_in = (u16(x["q"]), u16(x["iq"]), x["w"].cpu().numpy(), u16(x["ik"]), u16(x["rows"]),
             x["row_pos"].cpu().numpy(), x["q_pos"].cpu().numpy(), u16(x["raw"]))
    for t in (0, 1, 31, T - 1):
        check_prefill_query(x, st, t, K, SCALE, np_in)


def test_pro_dense_attention():
    U = 160
    n_rows = [900, 333, 0, 64] + [700] * (U - 4)
    n_raw = [128, 5, 0, 0] + [64] * (U - 4)
    x = make_decode_inputs(U, 900, device="cuda", seed=44, n_rows=n_rows, n_raw=n_raw, with_indexer=False,
                           n_head=H)
    st = DenseStep(U, 900, n_head=H)
    st(x, SCALE)
    torch.cuda.synchronize()
    device_ok()
    for u in (0, 1, 2, 3, U - 1):
        n, nw = n_rows[u], n_raw[u]
        ro, rl = oracle.dense_attention(u16(x["q"][u]), u16(x["rows"][u]), n, u16(x["raw"][u]), nw, SCALE)
        if n + nw == 0:
            assert torch.all(st.out[u] == 0) and torch.all(torch.isneginf(st.lse[u]))
            continue
        check_output(st.out[u].cpu().numpy(), ro, st.lse[u].cpu().numpy(), rl)


@pytest.mark.slow
def test_workload_pro_decode_sampled():
    wl = WORKLOADS["pro_decode_16x30x65536"]
    x = make_decode_inputs(wl.units, wl.n_rows, device="cuda", seed=wl.seed, n_head=wl.heads)
    st = run_decode(x, wl.top_k)
    with pool() as p:
        list(p.map(lambda u: check_decode_unit(x, st, u, wl.top_k, SCALE), [0, wl.units // 2, wl.units - 1]))
