"""The C-ABI library builds, loads and exports every entry point include/ds4a.h
declares; host-side validation rejects bad arguments before touching a GPU.
CPU only: no call here launches a kernel or queries a device."""
import ctypes
import os
import re
import subprocess

import pytest

from deepseek_v4_sparse_indexer_gb300 import _binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ds4a.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ds4a_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return B.load()


def test_header_declares_the_four_ops():
    fns = declared_functions()
    for op in ("ds4a_indexer_score", "ds4a_topk_select", "ds4a_sparse_attn_decode", "ds4a_sparse_attn_prefill"):
        assert op in fns


def test_every_declared_symbol_is_exported(lib):
    fns = declared_functions()
    assert set(fns) == set(B.EXPORTS), "binding and header disagree"
    nm = subprocess.run(["nm", "-D", "--defined-only", B.lib_path()], capture_output=True, text=True, check=True)
    exported = set(re.findall(r"\bT (ds4a_\w+)$", nm.stdout, flags=re.M))
    for f in fns:
        assert f in exported, f
        assert hasattr(lib, f)


def test_version_and_strerror(lib):
    assert B.ds4a_version() >> 16 == 1
    for code in (0, -1, -2, -3, -4, -5, 7):
        assert lib.ds4a_strerror(code)


def test_workspace_sizes():
    assert B.ds4a_workspace_bytes(B.DS4A_OP_INDEXER_SCORE, 4, 1, 262144, 512) == 0
    # Top-k: only up to 76 rows, each longer than 2^19 scores, use a
    # workspace (candidate slots of the two or more CTAs a row is cut over: at
    # most 152 slots of up to 4,096 (key, row) pairs plus two counters each).
    slot = 4096 * 8 + 8
    assert B.ds4a_workspace_bytes(B.DS4A_OP_TOPK_SELECT, 8, 1, 16384, 512) == 0
    assert B.ds4a_workspace_bytes(B.DS4A_OP_TOPK_SELECT, 1376, 1, 65536, 512) == 0
    assert B.ds4a_workspace_bytes(B.DS4A_OP_TOPK_SELECT, 4, 1, 262144, 512) == 0
    assert B.ds4a_workspace_bytes(B.DS4A_OP_TOPK_SELECT, 77, 1, 1 << 20, 512) == 0
    assert B.ds4a_workspace_bytes(B.DS4A_OP_TOPK_SELECT, 2, 1, 1 << 20, 512) == 2 * 76 * slot
    assert B.ds4a_workspace_bytes(B.DS4A_OP_TOPK_SELECT, 60, 1, 600000, 512) == 60 * 2 * slot
    assert B.ds4a_workspace_bytes(B.DS4A_OP_TOPK_SELECT, 1, 1, 1 << 24, 2048) <= 152 * slot
    # Attention: two partial slots (64 x (512 + 2) fp32) per share, at most
    # 160 shares, at most one share per 64-row tile (10 tiles per unit at k = 512).
    slot = 64 * 514 * 4
    assert B.ds4a_workspace_bytes(B.DS4A_OP_SPARSE_ATTN_DECODE, 1376, 1, 65536, 512) == 2 * 160 * slot
    assert B.ds4a_workspace_bytes(B.DS4A_OP_SPARSE_ATTN_DECODE, 4, 1, 262144, 512) == 2 * 40 * slot
    assert B.ds4a_workspace_bytes(B.DS4A_OP_SPARSE_ATTN_DECODE, 17, 1, 65536, 512) == 2 * 160 * slot  # 170 tiles
    assert B.ds4a_workspace_bytes(B.DS4A_OP_SPARSE_ATTN_PREFILL, 1, 2048, 66048, 512) == 2 * 160 * slot
    assert B.ds4a_workspace_bytes(B.DS4A_OP_DENSE_ATTN_DECODE, 1, 1, 64, 0) == 2 * 3 * slot    # 1 + 2 tiles
    assert B.ds4a_workspace_bytes(B.DS4A_OP_DENSE_ATTN_DECODE | B.DS4A_OP_FLAG_128_HEADS, 3, 1, 8192, 0) == 2 * 160 * slot
    with pytest.raises(ValueError):
        B.ds4a_workspace_bytes(B.DS4A_OP_TOPK_SELECT, 1, 1, 10, 4096)
    with pytest.raises(ValueError):
        B.ds4a_workspace_bytes(9, 1, 1, 10, 512)


def _vp(x):
    return ctypes.c_void_p(x)


FAKE = 0x10000   # never dereferenced: validation fails before any device access


def test_indexer_score_rejects_bad_arguments(lib):
    f = lib.ds4a_indexer_score
    # null pointers
    assert f(None, _vp(FAKE), _vp(FAKE), 128, _vp(FAKE), None, None, _vp(FAKE), 1, 1, 10, None) == B.DS4A_EINVAL
    # q_pos without row_pos
    assert f(_vp(FAKE), _vp(FAKE), _vp(FAKE), 128, _vp(FAKE), _vp(FAKE), None, _vp(FAKE), 1, 1, 10,
             None) == B.DS4A_EINVAL
    # sizes
    assert f(_vp(FAKE), _vp(FAKE), _vp(FAKE), 128, _vp(FAKE), None, None, _vp(FAKE), 0, 1, 10, None) == B.DS4A_EINVAL
    # misaligned key base (TMA needs 16 bytes)
    assert f(_vp(FAKE), _vp(FAKE), _vp(FAKE + 2), 1280, _vp(FAKE), None, None, _vp(FAKE), 1, 1, 10,
             None) == B.DS4A_EINVAL
    # unit stride smaller than a unit
    assert f(_vp(FAKE), _vp(FAKE), _vp(FAKE), 128, _vp(FAKE), None, None, _vp(FAKE), 2, 1, 10, None) == B.DS4A_EINVAL


def test_topk_rejects_bad_arguments(lib):
    f = lib.ds4a_topk_select
    assert f(_vp(FAKE), _vp(FAKE), 1, 1, 100, 0, _vp(FAKE), _vp(FAKE), _vp(FAKE), 1 << 30, None) == B.DS4A_EINVAL
    assert f(_vp(FAKE), _vp(FAKE), 1, 1, 100, 4096, _vp(FAKE), _vp(FAKE), _vp(FAKE), 1 << 30, None) == B.DS4A_EINVAL
    N = 1 << 20                                         # one very long row: the split path needs a workspace
    need = B.ds4a_workspace_bytes(B.DS4A_OP_TOPK_SELECT, 1, 1, N, 8)
    assert need > 0
    assert f(_vp(FAKE), _vp(FAKE), 1, 1, N, 8, _vp(FAKE), _vp(FAKE), None, need, None) == B.DS4A_EWORKSPACE
    assert f(_vp(FAKE), _vp(FAKE), 1, 1, N, 8, _vp(FAKE), _vp(FAKE), _vp(FAKE), need - 1, None) == \
        B.DS4A_EWORKSPACE
    assert f(_vp(FAKE), _vp(FAKE), 1, 1, N, 8, _vp(FAKE), _vp(FAKE), _vp(FAKE + 16), need, None) == \
        B.DS4A_EWORKSPACE


def test_attention_rejects_bad_arguments(lib):
    d = lib.ds4a_sparse_attn_decode
    args = [_vp(FAKE), _vp(FAKE), 512 * 64, 64, _vp(FAKE), _vp(FAKE), 512, _vp(FAKE), 128 * 512, _vp(FAKE),
            ctypes.c_float(0.04), _vp(FAKE), None, 1, None, 0, None]
    bad = list(args); bad[0] = None
    assert d(*bad) == B.DS4A_EINVAL
    bad = list(args); bad[6] = 0
    assert d(*bad) == B.DS4A_EINVAL
    bad = list(args); bad[1] = _vp(FAKE + 8)            # rows not 16-byte aligned
    assert d(*bad) == B.DS4A_EINVAL
    bad = list(args); bad[10] = ctypes.c_float(float("nan"))
    assert d(*bad) == B.DS4A_EINVAL
    bad = list(args); bad[13] = 4                       # 4 units need split workspace
    bad[2] = 512 * 64
    assert d(*bad) == B.DS4A_EWORKSPACE
    p = lib.ds4a_sparse_attn_prefill
    assert p(_vp(FAKE), None, _vp(FAKE), 64, _vp(FAKE), _vp(FAKE), 512, _vp(FAKE), 0, 10, ctypes.c_float(0.1),
             _vp(FAKE), None, 300, None, 0, None) == B.DS4A_EINVAL


def test_injected_error_is_returned_once(lib):
    lib.ds4a_debug_inject_error(B.DS4A_ECUDA)
    f = lib.ds4a_indexer_score
    assert f(None, None, None, 0, None, None, None, None, 0, 0, 0, None) == B.DS4A_ECUDA
    assert f(None, None, None, 0, None, None, None, None, 0, 0, 0, None) == B.DS4A_EINVAL


def test_binding_raises_on_error_status():
    B.ds4a_debug_inject_error(B.DS4A_EDEVICE)
    with pytest.raises(B.Ds4aError) as e:
        B._check(B.load().ds4a_topk_select(None, None, 0, 0, 0, 0, None, None, None, 0, None), "topk")
    assert e.value.status == B.DS4A_EDEVICE
