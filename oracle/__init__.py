"""fp64 CPU oracle for the three-tier compressed-attention step (test infrastructure).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package.  The CUDA
library never imports or calls it; the two share no code.

The arithmetic lives in ``ds4a_oracle.c`` (plain C, double precision).  This
module loads it through ctypes and adds the bookkeeping a whole query needs:
which raw-window rows a query sees, and composing score -> select -> attend.

Sources:
  [ARCH]  "DwarfStar(ds4.c) のアーキテクチャを読む【第1回/全8回】" (Qiita),
          §2 DS4_SHAPE_FLASH, §3-1 raw sliding-window KV, §3-3 indexer.
  [NOTES] "antirez/ds4 深度阅读笔记", 固定模型形状.
"""
import ctypes
import os

import numpy as np

from .build import build_oracle

# The pages' fixed shape ([ARCH] §2, [NOTES] 固定模型形状).  The oracle keeps its
# own copy: it shares no constant with the CUDA library.
N_HEAD = 64            # n_head
HEAD_DIM = 512         # n_head_dim (one KV head: rows are 512-d key = value)
N_INDEXER_HEAD = 64    # n_indexer_head
INDEXER_DIM = 128      # n_indexer_head_dim
N_SWA = 128            # raw sliding window
TOP_K = 512            # n_indexer_top_k (Flash)

_lib = None


def lib():
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if _lib is None:
        path = build_oracle()
        L = ctypes.CDLL(path)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f32p = ctypes.POINTER(ctypes.c_float)
        f64p = ctypes.POINTER(ctypes.c_double)
        i32p = ctypes.POINTER(ctypes.c_int32)
        L.oracle_abi_version.restype = ctypes.c_int
        L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_to_double.restype = ctypes.c_double
        L.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_f16_to_double.restype = ctypes.c_double
        L.oracle_double_to_f16.argtypes = [ctypes.c_double]
        L.oracle_double_to_f16.restype = ctypes.c_uint16
        L.oracle_indexer_score.argtypes = [u16p, f32p, u16p, ctypes.c_int64, ctypes.c_int64,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           i32p, i32p, f64p]
        L.oracle_indexer_score.restype = None
        L.oracle_topk_select.argtypes = [f64p, ctypes.c_int64, ctypes.c_int, i32p, f64p]
        L.oracle_topk_select.restype = ctypes.c_int
        L.oracle_sparse_attention.argtypes = [u16p, ctypes.c_int, ctypes.c_int,
                                              u16p, i32p, ctypes.c_int,
                                              u16p, i32p, ctypes.c_int,
                                              ctypes.c_double, f64p, f64p]
        L.oracle_sparse_attention.restype = ctypes.c_int
        L.oracle_compressor_pool.argtypes = [f32p, f32p, ctypes.c_int, ctypes.c_int, f64p]
        L.oracle_compressor_pool.restype = None
        L.oracle_push_raw.argtypes = [u16p, ctypes.POINTER(ctypes.c_int), ctypes.c_int, ctypes.c_int, f32p]
        L.oracle_push_raw.restype = None
        u8p = ctypes.POINTER(ctypes.c_uint8)
        L.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_to_double.restype = ctypes.c_double
        L.oracle_double_to_e4m3.argtypes = [ctypes.c_double]
        L.oracle_double_to_e4m3.restype = ctypes.c_uint8
        L.oracle_fp8_row_exponent.argtypes = [ctypes.c_double]
        L.oracle_fp8_row_exponent.restype = ctypes.c_int
        L.oracle_quantize_rows_fp8.argtypes = [f32p, ctypes.c_int64, ctypes.c_int, u8p, f32p]
        L.oracle_quantize_rows_fp8.restype = None
        L.oracle_sparse_attention_fp8.argtypes = [u16p, ctypes.c_int, ctypes.c_int,
                                                  u8p, f32p, i32p, ctypes.c_int,
                                                  u16p, i32p, ctypes.c_int,
                                                  ctypes.c_double, f64p, f64p]
        L.oracle_sparse_attention_fp8.restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(a, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _u16(a):
    """Raw 16-bit storage words (bf16 or fp16 bit patterns) as a C-contiguous uint16 array."""
    a = np.asarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    if a.dtype == np.int16:
        a = a.view(np.uint16)
    assert a.dtype == np.uint16, a.dtype
    return np.ascontiguousarray(a)


# ----------------------------------------------------------------------------
# Scalars
# ----------------------------------------------------------------------------

def bf16_to_double(bits: int) -> float:
    return lib().oracle_bf16_to_double(bits)


def f16_to_double(bits: int) -> float:
    return lib().oracle_f16_to_double(bits)


def double_to_f16(x: float) -> int:
    return lib().oracle_double_to_f16(x)


# ----------------------------------------------------------------------------
# A1 / A2 / A4 on one unit or one query
# ----------------------------------------------------------------------------

def indexer_score(iq, w, ik, n_rows, q_pos=None, row_pos=None):
    """Scores [Q, N_cap] (float64) of one unit.

    iq: bf16 bits [Q, H_i, D_i]; w: float32 [Q, H_i]; ik: bf16 bits [N_cap, D_i].
    Rows r >= n_rows, and (with positions) rows with row_pos[r] > q_pos[q], get -inf.
    """
    iq = _u16(iq)
    ik = _u16(ik)
    w = np.ascontiguousarray(w, dtype=np.float32)
    Q, H, Di = iq.shape
    n_cap = ik.shape[0]
    assert ik.shape[1] == Di and w.shape == (Q, H)
    out = np.empty((Q, n_cap), dtype=np.float64)
    qp = None if q_pos is None else np.ascontiguousarray(q_pos, dtype=np.int32)
    rp = None if row_pos is None else np.ascontiguousarray(row_pos, dtype=np.int32)
    lib().oracle_indexer_score(_ptr(iq, ctypes.c_uint16), _ptr(w, ctypes.c_float),
                               _ptr(ik, ctypes.c_uint16), int(n_rows), n_cap, Q, H, Di,
                               _ptr(qp, ctypes.c_int32), _ptr(rp, ctypes.c_int32),
                               _ptr(out, ctypes.c_double))
    return out


def topk_select(scores, top_k):
    """(idx ascending int32 [m], kth score) for one query's score row (float64)."""
    s = np.ascontiguousarray(scores, dtype=np.float64)
    idx = np.empty(max(top_k, 1), dtype=np.int32)
    kth = ctypes.c_double(0.0)
    m = lib().oracle_topk_select(_ptr(s, ctypes.c_double), s.shape[0], int(top_k),
                                 _ptr(idx, ctypes.c_int32), ctypes.byref(kth))
    return idx[:m].copy(), kth.value


def sparse_attention(q, comp_rows, sel, raw_rows, raw_sel, scale):
    """(out [H, D] float64, lse [H] float64) of one query.

    q: bf16 bits [H, D]; comp_rows: bf16 bits [N, D] indexed by sel;
    raw_rows: fp16 bits [R, D] indexed by raw_sel.
    """
    q = _u16(q)
    H, D = q.shape
    comp_rows = _u16(comp_rows) if comp_rows is not None else np.zeros((1, D), np.uint16)
    raw_rows = _u16(raw_rows) if raw_rows is not None else np.zeros((1, D), np.uint16)
    sel = np.ascontiguousarray(sel if sel is not None else [], dtype=np.int32)
    raw_sel = np.ascontiguousarray(raw_sel if raw_sel is not None else [], dtype=np.int32)
    if sel.size:
        assert sel.max() < comp_rows.shape[0]
    if raw_sel.size:
        assert raw_sel.max() < raw_rows.shape[0]
    out = np.empty((H, D), dtype=np.float64)
    lse = np.empty(H, dtype=np.float64)
    sel_p = sel if sel.size else np.zeros(1, np.int32)
    raw_p = raw_sel if raw_sel.size else np.zeros(1, np.int32)
    rc = lib().oracle_sparse_attention(_ptr(q, ctypes.c_uint16), H, D,
                                       _ptr(comp_rows, ctypes.c_uint16), _ptr(sel_p, ctypes.c_int32), sel.size,
                                       _ptr(raw_rows, ctypes.c_uint16), _ptr(raw_p, ctypes.c_int32), raw_sel.size,
                                       float(scale), _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double))
    if rc != 0:
        raise ValueError("negative row index")
    return out, lse


# ----------------------------------------------------------------------------
# Whole query: score -> select -> attend
# ----------------------------------------------------------------------------

def prefill_window(p, raw_pos0, n_raw_rows, window=N_SWA):
    """Indices into a contiguous raw buffer (row i holds position raw_pos0 + i)
    of the raw rows query position p attends: positions in [p - window + 1, p].

    [ARCH] §3-1 keeps the last n_swa = 128 tokens in the raw tier; the row of
    the query's own token is pushed before attention, so the window ends at p.
    """
    lo = max(p - window + 1 - raw_pos0, 0)
    hi = min(p - raw_pos0, n_raw_rows - 1)
    if hi < lo:
        return np.zeros(0, dtype=np.int32)
    return np.arange(lo, hi + 1, dtype=np.int32)


def decode_unit(q, iq, w, ik, rows, n_rows, raw, n_raw, top_k, scale):
    """One decode query of one unit end to end.

    Returns dict(scores [N_cap], idx ascending, kth, out [H, D], lse [H]).
    raw: fp16 bits [W, D] ring; its first n_raw slots are valid (any order).
    """
    s = indexer_score(iq[None], w[None], ik, n_rows)[0]
    idx, kth = topk_select(s, top_k)
    out, lse = sparse_attention(q, rows, idx, raw, np.arange(n_raw, dtype=np.int32), scale)
    return dict(scores=s, idx=idx, kth=kth, out=out, lse=lse)


def prefill_query(t, q, iq, w, ik, rows, n_rows, row_pos, q_pos, raw, raw_pos0, top_k, scale):
    """Query t of a prefill chunk end to end (positions make it causal).

    q: bf16 bits [T, H, D]; iq [T, H_i, D_i]; w [T, H_i]; q_pos [T];
    rows / ik / row_pos over the unit's N_cap rows; raw: fp16 bits [n_raw_rows, D]
    holding positions raw_pos0, raw_pos0 + 1, ...
    """
    p = int(q_pos[t])
    s = indexer_score(iq[t:t + 1], w[t:t + 1], ik, n_rows,
                      q_pos=np.array([p], np.int32), row_pos=row_pos)[0]
    idx, kth = topk_select(s, top_k)
    win = prefill_window(p, raw_pos0, raw.shape[0])
    out, lse = sparse_attention(q[t], rows, idx, raw, win, scale)
    return dict(scores=s, idx=idx, kth=kth, out=out, lse=lse, window=win)


def dense_attention(q, rows, n_rows, raw, n_raw, scale):
    """Attention of a ratio-128 layer ([ARCH] §3-2: the 128:1 layers have no
    indexer and attend to every compressed row): the joint softmax over rows
    0 .. n_rows-1 and raw slots 0 .. n_raw-1, i.e. the attention definition
    with every row selected."""
    return sparse_attention(q, rows, np.arange(n_rows, dtype=np.int32), raw, np.arange(n_raw, dtype=np.int32), scale)


def attention_with_given_set(q, rows, idx, raw, raw_sel, scale):
    """The attention step alone on a row set chosen elsewhere (used to check the
    device's output on the device's own selected set)."""
    return sparse_attention(q, rows, np.asarray(idx, np.int32), raw, raw_sel, scale)


# ----------------------------------------------------------------------------
# Cache producer: raw-window push and compressor pooling ([ARCH] §3-1, §3-2)
# ----------------------------------------------------------------------------

def compressor_pool(kv, score):
    """One compressed row (float64 [width]) from a frontier of `ratio` rows:
    per column, a softmax of the scores over the rows weights the kv values.
    kv, score: float32 [ratio, width]."""
    kv = np.ascontiguousarray(kv, dtype=np.float32)
    score = np.ascontiguousarray(score, dtype=np.float32)
    assert kv.shape == score.shape and kv.ndim == 2
    ratio, width = kv.shape
    out = np.empty(width, dtype=np.float64)
    lib().oracle_compressor_pool(_ptr(kv, ctypes.c_float), _ptr(score, ctypes.c_float), ratio, width,
                                 _ptr(out, ctypes.c_double))
    return out


def push_raw(ring, n_raw, kv, cap=N_SWA):
    """Push one fp32 row into a raw window kept oldest first (f16 bits
    [cap, dim]); returns (ring, n_raw) after the push (the ring is a copy)."""
    ring = np.array(ring, dtype=np.uint16, copy=True)
    kv = np.ascontiguousarray(kv, dtype=np.float32)
    assert ring.ndim == 2 and ring.shape[0] == cap and ring.shape[1] == kv.shape[0]
    n = ctypes.c_int(int(n_raw))
    lib().oracle_push_raw(_ptr(ring, ctypes.c_uint16), ctypes.byref(n), cap, ring.shape[1],
                          _ptr(kv, ctypes.c_float))
    return ring, n.value


# ----------------------------------------------------------------------------
# FP8 row store ([ARCH] §3-2: the FP8 quantisation round trip of a new
# compressed row).  Read as E4M3 codes with one power-of-two scale per row.
# ----------------------------------------------------------------------------

def e4m3_to_double(code: int) -> float:
    return lib().oracle_e4m3_to_double(int(code) & 0xFF)


def double_to_e4m3(x: float) -> int:
    """Nearest E4M3 code (ties to even), saturating at +-448; NaN -> 0x7F."""
    return lib().oracle_double_to_e4m3(float(x))


def fp8_row_exponent(amax: float) -> int:
    """Smallest e with amax <= 448 * 2^e, within [-126, 127]; 0 for amax 0 or not finite."""
    return lib().oracle_fp8_row_exponent(float(amax))


def quantize_rows_fp8(x):
    """(codes uint8 [n, dim], row_scale float32 [n]) of fp32 rows x [n, dim]."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert x.ndim == 2
    n, dim = x.shape
    codes = np.empty((n, dim), dtype=np.uint8)
    scale = np.empty(n, dtype=np.float32)
    if n:
        lib().oracle_quantize_rows_fp8(_ptr(x, ctypes.c_float), n, dim, _ptr(codes, ctypes.c_uint8),
                                       _ptr(scale, ctypes.c_float))
    return codes, scale


def fp8_rows_to_double(codes, row_scale):
    """Stored values (float64 [n, dim]) of FP8 rows: e4m3(code) * row scale."""
    codes = np.asarray(codes, dtype=np.uint8)
    table = np.array([e4m3_to_double(c) for c in range(256)], dtype=np.float64)
    return table[codes] * np.asarray(row_scale, dtype=np.float64)[:, None]


def sparse_attention_fp8(q, codes, row_scale, sel, raw_rows, raw_sel, scale):
    """sparse_attention with the compressed rows in the FP8 store (codes uint8
    [N, D], row_scale float32 [N]); raw rows stay fp16 bits."""
    q = _u16(q)
    H, D = q.shape
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    row_scale = np.ascontiguousarray(row_scale, dtype=np.float32)
    assert codes.shape[1] == D and row_scale.shape == (codes.shape[0],)
    raw_rows = _u16(raw_rows) if raw_rows is not None else np.zeros((1, D), np.uint16)
    sel = np.ascontiguousarray(sel if sel is not None else [], dtype=np.int32)
    raw_sel = np.ascontiguousarray(raw_sel if raw_sel is not None else [], dtype=np.int32)
    if sel.size:
        assert sel.max() < codes.shape[0]
    if raw_sel.size:
        assert raw_sel.max() < raw_rows.shape[0]
    out = np.empty((H, D), dtype=np.float64)
    lse = np.empty(H, dtype=np.float64)
    sel_p = sel if sel.size else np.zeros(1, np.int32)
    raw_p = raw_sel if raw_sel.size else np.zeros(1, np.int32)
    rc = lib().oracle_sparse_attention_fp8(_ptr(q, ctypes.c_uint16), H, D, _ptr(codes, ctypes.c_uint8),
                                           _ptr(row_scale, ctypes.c_float), _ptr(sel_p, ctypes.c_int32), sel.size,
                                           _ptr(raw_rows, ctypes.c_uint16), _ptr(raw_p, ctypes.c_int32), raw_sel.size,
                                           float(scale), _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double))
    if rc != 0:
        raise ValueError("negative row index")
    return out, lse
