"""ctypes binding of libds4a.so: the C ABI's entry points under the same names.

Argument marshalling only: each function checks dtypes, shapes, devices and
contiguity of torch tensors, passes their device pointers, the sizes and the
current CUDA stream to the C entry point, and raises Ds4aError on a non-zero
status.  Every step of the computation runs in the library's CUDA kernels;
there is no CPU path.  If the shared library is missing or cannot be loaded,
load() raises: nothing falls back.
"""
import ctypes
import os

import torch

from . import build as _build

DS4A_OK = 0
DS4A_EINVAL = -1
DS4A_EUNSUPPORTED = -2
DS4A_ECUDA = -3
DS4A_EWORKSPACE = -4
DS4A_EDEVICE = -5
DS4A_DEV_TIMEOUT = 1
DS4A_DEV_BOUNDS = 2
DS4A_OP_INDEXER_SCORE = 0
DS4A_OP_TOPK_SELECT = 1
DS4A_OP_SPARSE_ATTN_DECODE = 2
DS4A_OP_SPARSE_ATTN_PREFILL = 3
DS4A_OP_DENSE_ATTN_DECODE = 4
DS4A_OP_INDEXER_TOPK = 5
DS4A_OP_FLAG_128_HEADS = 0x100

N_HEAD, HEAD_DIM, N_IDX_HEAD, IDX_DIM, N_SWA = 64, 512, 64, 128, 128

# The C entry points this binding (and include/ds4a.h) exposes.
EXPORTS = ("ds4a_strerror", "ds4a_version", "ds4a_workspace_bytes", "ds4a_get_device_status",
           "ds4a_debug_inject_error", "ds4a_debug_wait_timeout", "ds4a_indexer_score", "ds4a_topk_select",
           "ds4a_topk_select_noalloc", "ds4a_sparse_attn_decode", "ds4a_sparse_attn_prefill",
           "ds4a_dense_attn_decode", "ds4a_kv_push_raw", "ds4a_compressor_pool",
           "ds4a_sparse_attn_decode_heads", "ds4a_sparse_attn_prefill_heads", "ds4a_dense_attn_decode_heads",
           "ds4a_rows_to_fp8", "ds4a_sparse_attn_decode_fp8", "ds4a_sparse_attn_prefill_fp8", "ds4a_indexer_topk")
DS4A_TOPK_NOALLOC_SCRATCH_BYTES = 8 << 20
DS4A_MAX_TOP_K = 2048


class Ds4aError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: ds4a status {status} ({_strerror(status)})")


_lib = None
_vp, _i32, _i64, _f32, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t


def lib_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = True):
    """Load libds4a.so (building it with nvcc first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB_PATH
    if build_if_missing and not _build.up_to_date():
        _build.build()
    if not os.path.exists(path):
        raise RuntimeError(f"libds4a.so not found at {path}; build it with __graft_entry__.build()")
    L = ctypes.CDLL(path)
    L.ds4a_strerror.argtypes = [_i32]
    L.ds4a_strerror.restype = ctypes.c_char_p
    L.ds4a_version.restype = _i32
    L.ds4a_workspace_bytes.argtypes = [_i32, _i32, _i32, _i32, _i32]
    L.ds4a_workspace_bytes.restype = _sz
    L.ds4a_get_device_status.argtypes = [_vp, ctypes.POINTER(ctypes.c_uint)]
    L.ds4a_get_device_status.restype = _i32
    L.ds4a_debug_inject_error.argtypes = [_i32]
    L.ds4a_debug_inject_error.restype = None
    L.ds4a_debug_wait_timeout.argtypes = [ctypes.c_uint, _vp]
    L.ds4a_debug_wait_timeout.restype = _i32
    L.ds4a_indexer_score.argtypes = [_vp, _vp, _vp, _i64, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _vp]
    L.ds4a_indexer_score.restype = _i32
    L.ds4a_topk_select.argtypes = [_vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _sz, _vp]
    L.ds4a_topk_select.restype = _i32
    L.ds4a_topk_select_noalloc.argtypes = [_vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp]
    L.ds4a_topk_select_noalloc.restype = _i32
    L.ds4a_sparse_attn_decode.argtypes = [_vp, _vp, _i64, _i32, _vp, _vp, _i32, _vp, _i64, _vp, _f32, _vp, _vp,
                                          _i32, _vp, _sz, _vp]
    L.ds4a_dense_attn_decode.argtypes = [_vp, _vp, _i64, _i32, _vp, _vp, _i64, _vp, _f32, _vp, _vp, _i32, _vp, _sz,
                                         _vp]
    L.ds4a_dense_attn_decode.restype = _i32
    L.ds4a_kv_push_raw.argtypes = [_vp, _vp, _i64, _vp, _vp, _i32, _vp]
    L.ds4a_kv_push_raw.restype = _i32
    L.ds4a_compressor_pool.argtypes = [_vp, _vp, _i32, _i32, _vp, _i32, _vp]
    L.ds4a_compressor_pool.restype = _i32
    L.ds4a_sparse_attn_decode.restype = _i32
    L.ds4a_sparse_attn_prefill.argtypes = [_vp, _vp, _vp, _i32, _vp, _vp, _i32, _vp, _i32, _i32, _f32, _vp, _vp,
                                           _i32, _vp, _sz, _vp]
    L.ds4a_sparse_attn_prefill.restype = _i32
    L.ds4a_sparse_attn_decode_heads.argtypes = [_i32] + L.ds4a_sparse_attn_decode.argtypes
    L.ds4a_sparse_attn_decode_heads.restype = _i32
    L.ds4a_sparse_attn_prefill_heads.argtypes = [_i32] + L.ds4a_sparse_attn_prefill.argtypes
    L.ds4a_sparse_attn_prefill_heads.restype = _i32
    L.ds4a_dense_attn_decode_heads.argtypes = [_i32] + L.ds4a_dense_attn_decode.argtypes
    L.ds4a_dense_attn_decode_heads.restype = _i32
    L.ds4a_indexer_topk.argtypes = [_vp, _vp, _vp, _i64, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _sz,
                                    _vp]
    L.ds4a_indexer_topk.restype = _i32
    L.ds4a_rows_to_fp8.argtypes = [_vp, _i64, _vp, _vp, _vp]
    L.ds4a_rows_to_fp8.restype = _i32
    L.ds4a_sparse_attn_decode_fp8.argtypes = [_vp, _vp, _vp, _i64, _i32, _vp, _vp, _i32, _vp, _i64, _vp, _f32, _vp,
                                              _vp, _i32, _vp, _sz, _vp]
    L.ds4a_sparse_attn_decode_fp8.restype = _i32
    L.ds4a_sparse_attn_prefill_fp8.argtypes = [_vp, _vp, _vp, _vp, _i32, _vp, _vp, _i32, _vp, _i32, _i32, _f32, _vp,
                                               _vp, _i32, _vp, _sz, _vp]
    L.ds4a_sparse_attn_prefill_fp8.restype = _i32
    _lib = L
    return L


def _strerror(status):
    try:
        return load(build_if_missing=False).ds4a_strerror(status).decode()
    except Exception:
        return "?"


def _check(status, where):
    if status != DS4A_OK:
        raise Ds4aError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _req(t, name, dtype, dev=True):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if dev and not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


# ----------------------------------------------------------------------------
# Entry points (same names as the C ABI)
# ----------------------------------------------------------------------------

def ds4a_version():
    return load().ds4a_version()


def ds4a_workspace_bytes(op, U, Q, N_cap, top_k):
    n = load().ds4a_workspace_bytes(op, U, Q, N_cap, top_k)
    if n == ctypes.c_size_t(-1).value:
        raise ValueError("ds4a_workspace_bytes: sizes out of range")
    return n


def ds4a_get_device_status(stream=None):
    """(status, flags) after synchronising the stream; clears the device word."""
    flags = ctypes.c_uint(0)
    st = load().ds4a_get_device_status(_stream(stream), ctypes.byref(flags))
    return st, flags.value


def ds4a_debug_inject_error(code):
    load().ds4a_debug_inject_error(code)


def ds4a_debug_wait_timeout(limit_us, stream=None):
    """Device-side failure-path hook: a bounded wait that nothing completes
    gives up after limit_us and sets DS4A_DEV_TIMEOUT (no fault)."""
    _check(load().ds4a_debug_wait_timeout(int(limit_us), _stream(stream)), "ds4a_debug_wait_timeout")


def ds4a_indexer_score(iq, w, ik, n_rows, scores, q_pos=None, row_pos=None, stream=None):
    """iq bf16 [U,Q,64,128]; w f32 [U,Q,64]; ik bf16 [U,N_cap,128] (unit stride
    may exceed N_cap*128); n_rows i32 [U]; scores f32 [U,Q,N_cap] (written).
    q_pos i32 [U,Q] and row_pos i32 [U,N_cap] for a causal prefill chunk."""
    _req(iq, "iq", torch.bfloat16)
    _req(w, "w", torch.float32)
    _req(n_rows, "n_rows", torch.int32)
    _req(scores, "scores", torch.float32)
    if ik.dtype != torch.bfloat16 or not ik.is_cuda or ik.dim() != 3 or ik.stride(2) != 1 or ik.stride(1) != IDX_DIM:
        raise ValueError("ik: bf16 CUDA tensor [U, N_cap, 128] with contiguous rows")
    U, N_cap = ik.shape[0], ik.shape[1]
    Q = iq.shape[1]
    if iq.shape != (U, Q, N_IDX_HEAD, IDX_DIM) or w.shape != (U, Q, N_IDX_HEAD):
        raise ValueError("iq / w shape")
    if scores.shape != (U, Q, N_cap) or n_rows.shape != (U,):
        raise ValueError("scores / n_rows shape")
    if (q_pos is None) != (row_pos is None):
        raise ValueError("q_pos and row_pos go together")
    if q_pos is not None:
        _req(q_pos, "q_pos", torch.int32)
        _req(row_pos, "row_pos", torch.int32)
        if q_pos.shape != (U, Q) or row_pos.shape != (U, N_cap):
            raise ValueError("q_pos / row_pos shape")
    st = load().ds4a_indexer_score(_ptr(iq), _ptr(w), _ptr(ik), ik.stride(0), _ptr(n_rows), _ptr(q_pos),
                                   _ptr(row_pos), _ptr(scores), U, Q, N_cap, _stream(stream))
    _check(st, "ds4a_indexer_score")


def ds4a_topk_select(scores, n_rows, top_k, idx, count, ws, stream=None):
    """scores f32 [U,Q,N_cap]; n_rows i32 [U]; idx i32 [U,Q,top_k], count i32
    [U,Q] (written); ws uint8 CUDA tensor of ds4a_workspace_bytes(...) bytes."""
    _req(scores, "scores", torch.float32)
    _req(n_rows, "n_rows", torch.int32)
    _req(idx, "idx", torch.int32)
    _req(count, "count", torch.int32)
    U, Q, N_cap = scores.shape
    if idx.shape != (U, Q, top_k) or count.shape != (U, Q):
        raise ValueError("idx / count shape")
    st = load().ds4a_topk_select(_ptr(scores), _ptr(n_rows), U, Q, N_cap, top_k, _ptr(idx), _ptr(count), _ptr(ws),
                                 ws.numel() * ws.element_size() if ws is not None else 0, _stream(stream))
    _check(st, "ds4a_topk_select")


def ds4a_indexer_topk(iq, w, ik, n_rows, top_k, idx, count, ws, q_pos=None, row_pos=None, stream=None):
    """Indexer score and top-k select fused (no scores array): iq bf16
    [U,Q,64,128]; w f32 [U,Q,64]; ik bf16 [U,N_cap,128]; n_rows i32 [U]; idx
    i32 [U,Q,top_k] and count i32 [U,Q] (written); ws uint8 CUDA tensor of
    ds4a_workspace_bytes(DS4A_OP_INDEXER_TOPK, ...) bytes."""
    _req(iq, "iq", torch.bfloat16)
    _req(w, "w", torch.float32)
    _req(n_rows, "n_rows", torch.int32)
    _req(idx, "idx", torch.int32)
    _req(count, "count", torch.int32)
    if ik.dtype != torch.bfloat16 or not ik.is_cuda or ik.dim() != 3 or ik.stride(2) != 1 or ik.stride(1) != IDX_DIM:
        raise ValueError("ik: bf16 CUDA tensor [U, N_cap, 128] with contiguous rows")
    U, N_cap = ik.shape[0], ik.shape[1]
    Q = iq.shape[1]
    if iq.shape != (U, Q, N_IDX_HEAD, IDX_DIM) or w.shape != (U, Q, N_IDX_HEAD) or n_rows.shape != (U,):
        raise ValueError("iq / w / n_rows shape")
    if idx.shape != (U, Q, top_k) or count.shape != (U, Q):
        raise ValueError("idx / count shape")
    if (q_pos is None) != (row_pos is None):
        raise ValueError("q_pos and row_pos go together")
    if q_pos is not None:
        _req(q_pos, "q_pos", torch.int32)
        _req(row_pos, "row_pos", torch.int32)
        if q_pos.shape != (U, Q) or row_pos.shape != (U, N_cap):
            raise ValueError("q_pos / row_pos shape")
    st = load().ds4a_indexer_topk(_ptr(iq), _ptr(w), _ptr(ik), ik.stride(0), _ptr(n_rows), _ptr(q_pos), _ptr(row_pos),
                                  U, Q, N_cap, top_k, _ptr(idx), _ptr(count), _ptr(ws),
                                  ws.numel() * ws.element_size() if ws is not None else 0, _stream(stream))
    _check(st, "ds4a_indexer_topk")


def ds4a_topk_select_noalloc(scores, n_rows, top_k, idx, count, stream=None):
    """Same result as ds4a_topk_select, with no workspace argument: the scratch
    is the library's fixed 8 MiB device array.  For callers that cannot
    allocate device memory; calls on one device must not overlap on the GPU."""
    _req(scores, "scores", torch.float32)
    _req(n_rows, "n_rows", torch.int32)
    _req(idx, "idx", torch.int32)
    _req(count, "count", torch.int32)
    U, Q, N_cap = scores.shape
    if idx.shape != (U, Q, top_k) or count.shape != (U, Q):
        raise ValueError("idx / count shape")
    st = load().ds4a_topk_select_noalloc(_ptr(scores), _ptr(n_rows), U, Q, N_cap, top_k, _ptr(idx), _ptr(count),
                                         _stream(stream))
    _check(st, "ds4a_topk_select_noalloc")


def ds4a_sparse_attn_decode(q, rows, idx, count, raw, n_raw, scale, out, lse=None, ws=None, stream=None):
    """The 64-head call (see ds4a_sparse_attn_decode_heads)."""
    if q.dim() == 3 and q.shape[1] != N_HEAD:
        raise ValueError("q: 64 heads (use ds4a_sparse_attn_decode_heads for 128)")
    ds4a_sparse_attn_decode_heads(N_HEAD, q, rows, idx, count, raw, n_raw, scale, out, lse, ws, stream)


def ds4a_sparse_attn_decode_heads(n_head, q, rows, idx, count, raw, n_raw, scale, out, lse=None, ws=None,
                                  stream=None):
    """q bf16 [U,H,512] (H = 64, or 128 through ds4a_sparse_attn_decode_heads);
    rows bf16 [U,N_cap,512]; idx i32 [U,top_k]; count i32 [U]; raw fp16
    [U,128,512]; n_raw i32 [U]; out f32 [U,H,512]; lse f32 [U,H] or None; ws
    uint8 workspace or None."""
    _req(q, "q", torch.bfloat16)
    _req(idx, "idx", torch.int32)
    _req(count, "count", torch.int32)
    _req(n_raw, "n_raw", torch.int32)
    _req(out, "out", torch.float32)
    if rows.dtype != torch.bfloat16 or not rows.is_cuda or rows.dim() != 3 or rows.stride(2) != 1 \
            or rows.stride(1) != HEAD_DIM:
        raise ValueError("rows: bf16 CUDA tensor [U, N_cap, 512] with contiguous rows")
    if raw.dtype != torch.float16 or not raw.is_cuda or raw.dim() != 3 or raw.stride(2) != 1 \
            or raw.stride(1) != HEAD_DIM or raw.shape[1] != N_SWA:
        raise ValueError("raw: fp16 CUDA tensor [U, 128, 512] with contiguous rows")
    U = q.shape[0]
    top_k = idx.shape[1]
    if q.shape != (U, n_head, HEAD_DIM) or rows.shape[0] != U or idx.shape[0] != U or count.shape != (U,) \
            or raw.shape[0] != U or n_raw.shape != (U,) or out.shape != (U, n_head, HEAD_DIM):
        raise ValueError("shape mismatch")
    if lse is not None:
        _req(lse, "lse", torch.float32)
        if lse.shape != (U, n_head):
            raise ValueError("lse: [U, n_head]")
    st = load().ds4a_sparse_attn_decode_heads(int(n_head), _ptr(q), _ptr(rows), rows.stride(0), rows.shape[1], _ptr(idx),
                                        _ptr(count), top_k, _ptr(raw), raw.stride(0), _ptr(n_raw), float(scale),
                                        _ptr(out), _ptr(lse), U, _ptr(ws),
                                        ws.numel() * ws.element_size() if ws is not None else 0, _stream(stream))
    _check(st, "ds4a_sparse_attn_decode_heads")


def ds4a_dense_attn_decode(q, rows, n_rows, raw, n_raw, scale, out, lse=None, ws=None, stream=None):
    """The 64-head call (see ds4a_dense_attn_decode_heads)."""
    if q.dim() == 3 and q.shape[1] != N_HEAD:
        raise ValueError("q: 64 heads (use ds4a_dense_attn_decode_heads for 128)")
    ds4a_dense_attn_decode_heads(N_HEAD, q, rows, n_rows, raw, n_raw, scale, out, lse, ws, stream)


def ds4a_dense_attn_decode_heads(n_head, q, rows, n_rows, raw, n_raw, scale, out, lse=None, ws=None, stream=None):
    """q bf16 [U,64,512]; rows bf16 [U,N_cap,512]; n_rows i32 [U]; raw fp16
    [U,128,512]; n_raw i32 [U]; out f32 [U,64,512]; lse f32 [U,64] or None;
    ws uint8 workspace or None."""
    _req(q, "q", torch.bfloat16)
    _req(n_rows, "n_rows", torch.int32)
    _req(n_raw, "n_raw", torch.int32)
    _req(out, "out", torch.float32)
    if rows.dtype != torch.bfloat16 or not rows.is_cuda or rows.dim() != 3 or rows.stride(2) != 1 \
            or rows.stride(1) != HEAD_DIM:
        raise ValueError("rows: bf16 CUDA tensor [U, N_cap, 512] with contiguous rows")
    if raw.dtype != torch.float16 or not raw.is_cuda or raw.dim() != 3 or raw.stride(2) != 1 \
            or raw.stride(1) != HEAD_DIM or raw.shape[1] != N_SWA:
        raise ValueError("raw: fp16 CUDA tensor [U, 128, 512] with contiguous rows")
    U = q.shape[0]
    if q.shape != (U, n_head, HEAD_DIM) or rows.shape[0] != U or n_rows.shape != (U,) or raw.shape[0] != U \
            or n_raw.shape != (U,) or out.shape != (U, n_head, HEAD_DIM):
        raise ValueError("shape mismatch")
    if lse is not None:
        _req(lse, "lse", torch.float32)
        if lse.shape != (U, n_head):
            raise ValueError("lse: [U, n_head]")
    st = load().ds4a_dense_attn_decode_heads(int(n_head), _ptr(q), _ptr(rows), rows.stride(0), rows.shape[1], _ptr(n_rows), _ptr(raw),
                                       raw.stride(0), _ptr(n_raw), float(scale), _ptr(out), _ptr(lse), U, _ptr(ws),
                                       ws.numel() * ws.element_size() if ws is not None else 0, _stream(stream))
    _check(st, "ds4a_dense_attn_decode_heads")


def ds4a_sparse_attn_prefill(q, q_pos, rows, idx, count, raw, raw_pos0, scale, out, lse=None, ws=None, stream=None):
    """The 64-head call (see ds4a_sparse_attn_prefill_heads)."""
    if q.dim() == 3 and q.shape[1] != N_HEAD:
        raise ValueError("q: 64 heads (use ds4a_sparse_attn_prefill_heads for 128)")
    ds4a_sparse_attn_prefill_heads(N_HEAD, q, q_pos, rows, idx, count, raw, raw_pos0, scale, out, lse, ws, stream)


def ds4a_sparse_attn_prefill_heads(n_head, q, q_pos, rows, idx, count, raw, raw_pos0, scale, out, lse=None, ws=None,
                                   stream=None):
    """q bf16 [T,64,512]; q_pos i32 [T]; rows bf16 [N_cap,512]; idx i32
    [T,top_k]; count i32 [T]; raw fp16 [n_raw_rows,512] (row i = position
    raw_pos0 + i); out f32 [T,64,512]; lse f32 [T,64] or None."""
    _req(q, "q", torch.bfloat16)
    _req(q_pos, "q_pos", torch.int32)
    _req(rows, "rows", torch.bfloat16)
    _req(idx, "idx", torch.int32)
    _req(count, "count", torch.int32)
    _req(raw, "raw", torch.float16)
    _req(out, "out", torch.float32)
    T = q.shape[0]
    top_k = idx.shape[1]
    if q.shape != (T, n_head, HEAD_DIM) or q_pos.shape != (T,) or rows.dim() != 2 or rows.shape[1] != HEAD_DIM \
            or idx.shape[0] != T or count.shape != (T,) or raw.dim() != 2 or raw.shape[1] != HEAD_DIM \
            or out.shape != (T, n_head, HEAD_DIM):
        raise ValueError("shape mismatch")
    if lse is not None:
        _req(lse, "lse", torch.float32)
        if lse.shape != (T, n_head):
            raise ValueError("lse: [T, n_head]")
    st = load().ds4a_sparse_attn_prefill_heads(int(n_head), _ptr(q), _ptr(q_pos), _ptr(rows), rows.shape[0], _ptr(idx), _ptr(count),
                                         top_k, _ptr(raw), int(raw_pos0), raw.shape[0], float(scale), _ptr(out),
                                         _ptr(lse), T, _ptr(ws),
                                         ws.numel() * ws.element_size() if ws is not None else 0, _stream(stream))
    _check(st, "ds4a_sparse_attn_prefill_heads")


def ds4a_kv_push_raw(kv, raw, pos, n_raw, stream=None):
    """kv f32 [U,512]; raw fp16 [U,128,512] ring (written); pos i32 [U]; n_raw
    i32 [U] (written)."""
    _req(kv, "kv", torch.float32)
    _req(pos, "pos", torch.int32)
    _req(n_raw, "n_raw", torch.int32)
    if raw.dtype != torch.float16 or not raw.is_cuda or raw.dim() != 3 or raw.stride(2) != 1 \
            or raw.stride(1) != HEAD_DIM or raw.shape[1] != N_SWA:
        raise ValueError("raw: fp16 CUDA tensor [U, 128, 512] with contiguous rows")
    U = kv.shape[0]
    if kv.shape != (U, HEAD_DIM) or raw.shape[0] != U or pos.shape != (U,) or n_raw.shape != (U,):
        raise ValueError("shape mismatch")
    st = load().ds4a_kv_push_raw(_ptr(kv), _ptr(raw), raw.stride(0), _ptr(pos), _ptr(n_raw), U, _stream(stream))
    _check(st, "ds4a_kv_push_raw")


def ds4a_compressor_pool(kv, score, out, stream=None):
    """kv, score f32 [U,ratio,width]; out f32 [U,width] (written)."""
    _req(kv, "kv", torch.float32)
    _req(score, "score", torch.float32)
    _req(out, "out", torch.float32)
    if kv.dim() != 3 or score.shape != kv.shape or out.shape != (kv.shape[0], kv.shape[2]):
        raise ValueError("shape mismatch")
    U, ratio, width = kv.shape
    st = load().ds4a_compressor_pool(_ptr(kv), _ptr(score), ratio, width, _ptr(out), U, _stream(stream))
    _check(st, "ds4a_compressor_pool")


# ----------------------------------------------------------------------------
# FP8 row store
# ----------------------------------------------------------------------------

def _req_fp8_rows(rows8, row_scale, n_dims):
    if rows8.dtype != torch.uint8 or not rows8.is_cuda or rows8.dim() != n_dims or rows8.stride(-1) != 1 \
            or rows8.shape[-1] != HEAD_DIM or rows8.stride(-2) != HEAD_DIM:
        raise ValueError("rows8: uint8 CUDA tensor [..., N_cap, 512] of E4M3 codes with contiguous rows")
    if row_scale.dtype != torch.float32 or not row_scale.is_cuda or row_scale.stride(-1) != 1:
        raise ValueError("row_scale: float32 CUDA tensor, one scale per row")


def ds4a_rows_to_fp8(x, rows8, row_scale, stream=None):
    """x f32 [n,512] -> rows8 uint8 [n,512] E4M3 codes and row_scale f32 [n]
    (power-of-two scale per row), both written."""
    _req(x, "x", torch.float32)
    _req(rows8, "rows8", torch.uint8)
    _req(row_scale, "row_scale", torch.float32)
    n = x.shape[0]
    if x.shape != (n, HEAD_DIM) or rows8.shape != (n, HEAD_DIM) or row_scale.shape != (n,):
        raise ValueError("shape mismatch")
    st = load().ds4a_rows_to_fp8(_ptr(x), n, _ptr(rows8), _ptr(row_scale), _stream(stream))
    _check(st, "ds4a_rows_to_fp8")


def ds4a_sparse_attn_decode_fp8(q, rows8, row_scale, idx, count, raw, n_raw, scale, out, lse=None, ws=None,
                                stream=None):
    """ds4a_sparse_attn_decode with the compressed rows as the FP8 store:
    rows8 uint8 [U,N_cap,512] E4M3 codes, row_scale f32 [U,N_cap] laid out
    like the rows (unit u's scales start at u * rows8.stride(0) / 512)."""
    _req(q, "q", torch.bfloat16)
    _req(idx, "idx", torch.int32)
    _req(count, "count", torch.int32)
    _req(n_raw, "n_raw", torch.int32)
    _req(out, "out", torch.float32)
    _req_fp8_rows(rows8, row_scale, 3)
    if raw.dtype != torch.float16 or not raw.is_cuda or raw.dim() != 3 or raw.stride(2) != 1 \
            or raw.stride(1) != HEAD_DIM or raw.shape[1] != N_SWA:
        raise ValueError("raw: fp16 CUDA tensor [U, 128, 512] with contiguous rows")
    U, N_cap = rows8.shape[0], rows8.shape[1]
    top_k = idx.shape[1]
    if row_scale.dim() != 2 or row_scale.shape != (U, N_cap) or (U > 1 and
                                                               row_scale.stride(0) * HEAD_DIM != rows8.stride(0)):
        raise ValueError("row_scale: [U, N_cap] with unit stride rows8.stride(0) / 512")
    if q.shape != (U, N_HEAD, HEAD_DIM) or idx.shape[0] != U or count.shape != (U,) or raw.shape[0] != U \
            or n_raw.shape != (U,) or out.shape != (U, N_HEAD, HEAD_DIM):
        raise ValueError("shape mismatch")
    if lse is not None:
        _req(lse, "lse", torch.float32)
        if lse.shape != (U, N_HEAD):
            raise ValueError("lse: [U, 64]")
    st = load().ds4a_sparse_attn_decode_fp8(_ptr(q), _ptr(rows8), _ptr(row_scale), rows8.stride(0), N_cap, _ptr(idx),
                                            _ptr(count), top_k, _ptr(raw), raw.stride(0), _ptr(n_raw), float(scale),
                                            _ptr(out), _ptr(lse), U, _ptr(ws),
                                            ws.numel() * ws.element_size() if ws is not None else 0, _stream(stream))
    _check(st, "ds4a_sparse_attn_decode_fp8")


def ds4a_sparse_attn_prefill_fp8(q, q_pos, rows8, row_scale, idx, count, raw, raw_pos0, scale, out, lse=None,
                                 ws=None, stream=None):
    """ds4a_sparse_attn_prefill with the compressed rows as the FP8 store:
    rows8 uint8 [N_cap,512], row_scale f32 [N_cap]."""
    _req(q, "q", torch.bfloat16)
    _req(q_pos, "q_pos", torch.int32)
    _req(rows8, "rows8", torch.uint8)
    _req(row_scale, "row_scale", torch.float32)
    _req(idx, "idx", torch.int32)
    _req(count, "count", torch.int32)
    _req(raw, "raw", torch.float16)
    _req(out, "out", torch.float32)
    T = q.shape[0]
    top_k = idx.shape[1]
    if q.shape != (T, N_HEAD, HEAD_DIM) or q_pos.shape != (T,) or rows8.dim() != 2 or rows8.shape[1] != HEAD_DIM \
            or row_scale.shape != (rows8.shape[0],) or idx.shape[0] != T or count.shape != (T,) or raw.dim() != 2 \
            or raw.shape[1] != HEAD_DIM or out.shape != (T, N_HEAD, HEAD_DIM):
        raise ValueError("shape mismatch")
    if lse is not None:
        _req(lse, "lse", torch.float32)
        if lse.shape != (T, N_HEAD):
            raise ValueError("lse: [T, 64]")
    st = load().ds4a_sparse_attn_prefill_fp8(_ptr(q), _ptr(q_pos), _ptr(rows8), _ptr(row_scale), rows8.shape[0],
                                             _ptr(idx), _ptr(count), top_k, _ptr(raw), int(raw_pos0), raw.shape[0],
                                             float(scale), _ptr(out), _ptr(lse), T, _ptr(ws),
                                             ws.numel() * ws.element_size() if ws is not None else 0,
                                             _stream(stream))
    _check(st, "ds4a_sparse_attn_prefill_fp8")
