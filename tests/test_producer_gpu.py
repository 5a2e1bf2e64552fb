"""Parity of the cache-producer kernels (through the C ABI) with the fp64 oracle:
the raw-window push with f16 rounding ("DwarfStar(ds4.c) のアーキテクチャを読む"
§3-1) and the compressor's per-column softmax pooling (§3-2)."""
import numpy as np
import pytest
import torch

import oracle
from deepseek_v4_sparse_indexer_gb300 import _binding as B

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    yield
    torch.cuda.synchronize()


def device_ok():
    st, flags = B.ds4a_get_device_status()
    assert st == B.DS4A_OK and flags == 0, f"device status flags {flags}"


def pool_tolerance(kv):
    """fp32 weights (expf, one rounding each) and up to `ratio` fp32 terms in
    the two sums: the pooled value is off by at most ~(ratio + 8) units of
    2^-24 of the column's largest |kv|; 2^-14 of it is a safe bound."""
    return np.abs(kv).max(axis=0) * 2.0 ** -14 + 1e-30


@pytest.mark.parametrize("ratio,width", [(1, 128), (4, 512), (4, 128), (128, 512), (7, 12)])
def test_compressor_pool_matches_oracle(ratio, width):
    rng = np.random.default_rng(ratio * 1000 + width)
    U = 5
    kv = rng.standard_normal((U, ratio, width)).astype(np.float32)
    sc = (3 * rng.standard_normal((U, ratio, width))).astype(np.float32)
    sc[0, :, 1] = -np.inf                                   # masked column -> 0
    sc[1, ratio // 2, :] += 80.0                            # one dominant row
    if ratio > 1:
        sc[2, 0, 3] = -np.inf                               # one masked row in a column
    out = torch.full((U, width), float("nan"), device="cuda")
    B.ds4a_compressor_pool(torch.from_numpy(kv).cuda(), torch.from_numpy(sc).cuda(), out)
    torch.cuda.synchronize()
    device_ok()
    got = out.cpu().numpy().astype(np.float64)
    for u in range(U):
        ref = oracle.compressor_pool(kv[u], sc[u])
        tol = pool_tolerance(kv[u])
        assert np.all(np.abs(got[u] - ref) <= tol), (u, float(np.max(np.abs(got[u] - ref) - tol)))
    assert got[0, 1] == 0.0


def test_push_raw_sequence_matches_the_oracle_window():
    """Positions 0..299 pushed one call at a time: after every push the ring
    holds the oracle's window (oldest first) rotated by the position."""
    rng = np.random.default_rng(90)
    U, steps = 3, 300
    raw = torch.zeros(U, 128, 512, dtype=torch.float16, device="cuda")
    n_raw = torch.zeros(U, dtype=torch.int32, device="cuda")
    win = [np.zeros((128, 512), np.uint16) for _ in range(U)]
    nwin = [0] * U
    for p in range(steps):
        kv = (rng.standard_normal((U, 512)) * 300).astype(np.float32)
        if p == 5:
            kv[0, :4] = [65520.0, -65520.0, 1e-8, 2.0 ** -24 * 1.5]   # overflow, underflow, subnormal tie
        pos = torch.full((U,), p, dtype=torch.int32, device="cuda")
        B.ds4a_kv_push_raw(torch.from_numpy(kv).cuda(), raw, pos, n_raw)
        for u in range(U):
            win[u], nwin[u] = oracle.push_raw(win[u], nwin[u], kv[u])
        if p in (0, 1, 126, 127, 128, 129, 200, steps - 1):
            torch.cuda.synchronize()
            ring = raw.view(torch.int16).cpu().numpy().view(np.uint16)
            assert n_raw.cpu().tolist() == nwin
            for u in range(U):
                n = nwin[u]
                slots = [(p - n + 1 + i) % 128 for i in range(n)]   # oldest first
                assert np.array_equal(ring[u][slots], win[u][:n]), (p, u)
    device_ok()


def test_push_raw_batch_with_strided_rings_and_a_bad_position():
    rng = np.random.default_rng(91)
    U = 4
    store = torch.zeros(U, 130, 512, dtype=torch.float16, device="cuda")     # unit stride 130 rows
    raw = store[:, :128]
    n_raw = torch.full((U,), 77, dtype=torch.int32, device="cuda")
    kv = (rng.standard_normal((U, 512)) * 10).astype(np.float32)
    pos = torch.tensor([0, 127, 1000, -1], dtype=torch.int32, device="cuda")
    B.ds4a_kv_push_raw(torch.from_numpy(kv).cuda(), raw, pos, n_raw)
    st, flags = B.ds4a_get_device_status()
    assert st == B.DS4A_EDEVICE and flags & B.DS4A_DEV_BOUNDS
    ring = store.view(torch.int16).cpu().numpy().view(np.uint16)
    for u, slot, n in [(0, 0, 1), (1, 127, 128), (2, 1000 % 128, 128)]:
        assert np.array_equal(ring[u, slot], kv[u].astype(np.float16).view(np.uint16))
        assert int(n_raw[u]) == n
    assert int(n_raw[3]) == 77 and not ring[3].any()        # the bad position wrote nothing
    device_ok()


@pytest.mark.slow
def test_workload_pool_32x20x128_full():
    """The benchmarked producer step (raw push + ratio-128 pooling of 640 units)
    in the bench's launch configuration, every unit against the oracle."""
    from deepseek_v4_sparse_indexer_gb300 import ProducerStep
    from deepseek_v4_sparse_indexer_gb300.workloads import WORKLOADS, make_pool_inputs
    wl = WORKLOADS["pool_32x20x128"]
    x = make_pool_inputs(wl.units, wl.n_rows, device="cuda", seed=wl.seed)
    st = ProducerStep(wl.units)
    st(x)
    torch.cuda.synchronize()
    device_ok()
    kv, sc, got = x["kv"].cpu().numpy(), x["score"].cpu().numpy(), st.out.cpu().numpy().astype(np.float64)
    for u in range(wl.units):
        ref = oracle.compressor_pool(kv[u], sc[u])
        assert np.all(np.abs(got[u] - ref) <= pool_tolerance(kv[u])), u
    # the new rows landed in ring slot pos % 128, rounded to f16
    slot = int(x["pos"][0]) % 128
    assert torch.equal(x["raw"][:, slot], x["row"].half())
