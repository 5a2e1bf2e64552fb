"""One pass of the three-tier compressed-attention step through the C ABI.

DecodeStep: U units (sequence x layer caches), one query each.
PrefillStep: one chunk of T queries of one sequence over a causal row store.
DenseStep: the ratio-128 layers' attention over all compressed rows (no
indexer, so no score or select).
ProducerStep: the cache producer at a ratio boundary: the raw-window push of
the new token, the compressor pooling of the frontier and (fp8=True) the FP8
store of the pooled row.

DecodeStep and PrefillStep with fp8=True read the compressed rows from the FP8
row store (x["rows8"] E4M3 codes, x["row_scale"] per-row scales) instead of
the bf16 rows; with fused=True they score and select in one call
(ds4a_indexer_topk: no scores array, the same selection).

Both own their outputs and workspaces (allocated once, reused every call, so a
call can be captured in a CUDA graph) and run indexer score -> top-k select ->
sparse attention on one CUDA stream, each op a C-ABI call into libds4a.so.
"""
import math

import torch

from . import _binding as B

DEFAULT_SCALE = 1.0 / math.sqrt(B.HEAD_DIM)


def _ws(nbytes, device):
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device) if nbytes else None


class DecodeStep:
    def __init__(self, U, N_cap, top_k=512, device="cuda", n_head=B.N_HEAD, fp8=False, fused=False):
        if fp8 and n_head != B.N_HEAD:
            raise ValueError("the FP8 row store is read with 64 query heads")
        self.U, self.N_cap, self.top_k, self.n_head, self.fp8, self.fused = U, N_cap, top_k, n_head, fp8, fused
        dev = torch.device(device)
        flag = B.DS4A_OP_FLAG_128_HEADS if n_head == 128 else 0
        self.scores = None if fused else torch.empty(U, 1, N_cap, dtype=torch.float32, device=dev)
        self.ws_fused = _ws(B.ds4a_workspace_bytes(B.DS4A_OP_INDEXER_TOPK, U, 1, N_cap, top_k), dev) if fused else None
        self.idx = torch.empty(U, 1, top_k, dtype=torch.int32, device=dev)
        self.count = torch.empty(U, 1, dtype=torch.int32, device=dev)
        self.out = torch.empty(U, n_head, B.HEAD_DIM, dtype=torch.float32, device=dev)
        self.lse = torch.empty(U, n_head, dtype=torch.float32, device=dev)
        self.ws_topk = None if fused else _ws(B.ds4a_workspace_bytes(B.DS4A_OP_TOPK_SELECT, U, 1, N_cap, top_k), dev)
        self.ws_attn = _ws(B.ds4a_workspace_bytes(B.DS4A_OP_SPARSE_ATTN_DECODE | flag, U, 1, N_cap, top_k), dev)

    def score(self, x, stream=None):
        iq, w = x["iq"].view(self.U, 1, B.N_IDX_HEAD, B.IDX_DIM), x["w"].view(self.U, 1, B.N_IDX_HEAD)
        if self.fused:
            B.ds4a_indexer_topk(iq, w, x["ik"], x["n_rows"], self.top_k, self.idx, self.count, self.ws_fused,
                                stream=stream)
            return
        B.ds4a_indexer_score(iq, w, x["ik"], x["n_rows"], self.scores, stream=stream)

    def select(self, x, stream=None):
        if self.fused:
            return                                   # done by score()
        B.ds4a_topk_select(self.scores, x["n_rows"], self.top_k, self.idx, self.count, self.ws_topk, stream=stream)

    def attend(self, x, scale=DEFAULT_SCALE, stream=None):
        idx, count = self.idx.view(self.U, self.top_k), self.count.view(self.U)
        if self.fp8:
            B.ds4a_sparse_attn_decode_fp8(x["q"], x["rows8"], x["row_scale"], idx, count, x["raw"], x["n_raw"], scale,
                                          self.out, self.lse, self.ws_attn, stream=stream)
            return
        B.ds4a_sparse_attn_decode_heads(self.n_head, x["q"], x["rows"], idx, count, x["raw"], x["n_raw"], scale,
                                        self.out, self.lse, self.ws_attn, stream=stream)

    def __call__(self, x, scale=DEFAULT_SCALE, stream=None):
        self.score(x, stream)
        self.select(x, stream)
        self.attend(x, scale, stream)
        return self.out


class PrefillStep:
    def __init__(self, T, N_cap, top_k=512, device="cuda", n_head=B.N_HEAD, fp8=False, fused=False):
        if fp8 and n_head != B.N_HEAD:
            raise ValueError("the FP8 row store is read with 64 query heads")
        self.T, self.N_cap, self.top_k, self.n_head, self.fp8, self.fused = T, N_cap, top_k, n_head, fp8, fused
        dev = torch.device(device)
        flag = B.DS4A_OP_FLAG_128_HEADS if n_head == 128 else 0
        self.scores = None if fused else torch.empty(1, T, N_cap, dtype=torch.float32, device=dev)
        self.ws_fused = _ws(B.ds4a_workspace_bytes(B.DS4A_OP_INDEXER_TOPK, 1, T, N_cap, top_k), dev) if fused else None
        self.idx = torch.empty(1, T, top_k, dtype=torch.int32, device=dev)
        self.count = torch.empty(1, T, dtype=torch.int32, device=dev)
        self.out = torch.empty(T, n_head, B.HEAD_DIM, dtype=torch.float32, device=dev)
        self.lse = torch.empty(T, n_head, dtype=torch.float32, device=dev)
        self.ws_topk = None if fused else _ws(B.ds4a_workspace_bytes(B.DS4A_OP_TOPK_SELECT, 1, T, N_cap, top_k), dev)
        self.ws_attn = _ws(B.ds4a_workspace_bytes(B.DS4A_OP_SPARSE_ATTN_PREFILL | flag, 1, T, N_cap, top_k), dev)

    def score(self, x, stream=None):
        T, N = self.T, self.N_cap
        iq, w = x["iq"].view(1, T, B.N_IDX_HEAD, B.IDX_DIM), x["w"].view(1, T, B.N_IDX_HEAD)
        ik, qp, rp = x["ik"].view(1, N, B.IDX_DIM), x["q_pos"].view(1, T), x["row_pos"].view(1, N)
        if self.fused:
            B.ds4a_indexer_topk(iq, w, ik, x["n_rows"], self.top_k, self.idx, self.count, self.ws_fused,
                                q_pos=qp, row_pos=rp, stream=stream)
            return
        B.ds4a_indexer_score(iq, w, ik, x["n_rows"], self.scores, q_pos=qp, row_pos=rp, stream=stream)

    def select(self, x, stream=None):
        if self.fused:
            return                                   # done by score()
        B.ds4a_topk_select(self.scores, x["n_rows"], self.top_k, self.idx, self.count, self.ws_topk, stream=stream)

    def attend(self, x, scale=DEFAULT_SCALE, stream=None):
        idx, count = self.idx.view(self.T, self.top_k), self.count.view(self.T)
        if self.fp8:
            B.ds4a_sparse_attn_prefill_fp8(x["q"], x["q_pos"], x["rows8"], x["row_scale"], idx, count, x["raw"],
                                           x["raw_pos0"], scale, self.out, self.lse, self.ws_attn, stream=stream)
            return
        B.ds4a_sparse_attn_prefill_heads(self.n_head, x["q"], x["q_pos"], x["rows"], idx, count, x["raw"],
                                         x["raw_pos0"], scale, self.out, self.lse, self.ws_attn, stream=stream)

    def __call__(self, x, scale=DEFAULT_SCALE, stream=None):
        self.score(x, stream)
        self.select(x, stream)
        self.attend(x, scale, stream)
        return self.out


class DenseStep:
    def __init__(self, U, N_cap, device="cuda", n_head=B.N_HEAD):
        self.U, self.N_cap, self.n_head = U, N_cap, n_head
        dev = torch.device(device)
        flag = B.DS4A_OP_FLAG_128_HEADS if n_head == 128 else 0
        self.out = torch.empty(U, n_head, B.HEAD_DIM, dtype=torch.float32, device=dev)
        self.lse = torch.empty(U, n_head, dtype=torch.float32, device=dev)
        self.ws_attn = _ws(B.ds4a_workspace_bytes(B.DS4A_OP_DENSE_ATTN_DECODE | flag, U, 1, N_cap, 0), dev)

    def attend(self, x, scale=DEFAULT_SCALE, stream=None):
        B.ds4a_dense_attn_decode_heads(self.n_head, x["q"], x["rows"], x["n_rows"], x["raw"], x["n_raw"], scale,
                                       self.out, self.lse, self.ws_attn, stream=stream)

    def __call__(self, x, scale=DEFAULT_SCALE, stream=None):
        self.attend(x, scale, stream)
        return self.out


class ProducerStep:
    def __init__(self, U, width=B.HEAD_DIM, device="cuda", fp8=False):
        if fp8 and width != B.HEAD_DIM:
            raise ValueError("the FP8 row store holds 512-wide rows")
        self.U, self.width, self.fp8 = U, width, fp8
        dev = torch.device(device)
        self.out = torch.empty(U, width, dtype=torch.float32, device=dev)
        self.rows8 = torch.empty(U, width, dtype=torch.uint8, device=dev) if fp8 else None
        self.row_scale = torch.empty(U, dtype=torch.float32, device=dev) if fp8 else None

    def push(self, x, stream=None):
        B.ds4a_kv_push_raw(x["row"], x["raw"], x["pos"], x["n_raw"], stream=stream)

    def pool(self, x, stream=None):
        B.ds4a_compressor_pool(x["kv"], x["score"], self.out, stream=stream)

    def store_fp8(self, stream=None):
        B.ds4a_rows_to_fp8(self.out, self.rows8, self.row_scale, stream=stream)

    def __call__(self, x, stream=None):
        self.push(x, stream)
        self.pool(x, stream)
        if self.fp8:
            self.store_fp8(stream)
        return self.out
