"""Seeded synthetic inputs shaped like the pages' workloads.

This module only builds inputs: it holds none of the step's arithmetic (no
scoring, selection or attention).  The tests feed the same tensors to the CUDA
library and to the fp64 oracle, and the benchmark uses them for timing.

Value recipe: every bf16/fp16 tensor is N(0,1)/sqrt(d) rounded to nearest
even, with d = 512 for queries, compressed rows and raw rows and d = 128 for
indexer queries and keys; indexer weights are U(0,1) fp32.  Compressed rows,
queries and indexer tensors are bf16; raw-window rows are fp16 (the raw tier is
kept rounded to f16: "DwarfStar(ds4.c) のアーキテクチャを読む" §3-1).

Workload shapes (query-token x layer units, compressed rows per unit):
  decode_1x1024          1 unit, 1,024 rows                  (small parity case)
  decode_8x16384         8 units, 16,384 rows
  decode_32x43x65536     32 sequences x 43 layers = 1,376 units, 65,536 rows
  prefill_2048x65536     one 2,048-query chunk over 65,536 prior rows + 512 rows
                         finalised inside the chunk (causal)
  longctx_4x262144       4 units, 262,144 rows, 5 % of indexer keys scaled x4
The shapes follow the pages: 43 layers, 64 heads x 512, indexer 64 x 128,
top_k 512, 128-row raw window (§2 DS4_SHAPE_FLASH); prefill advances in
2,048-token chunks and benchmarks reach depth 65,536 (the Qwen3.8-Flash-Next
on DwarfStar article, 測定条件); a 1M-token context holds ~250k ratio-4
compressed rows (§3-3).
"""
from dataclasses import dataclass, field
import math

import torch

N_HEAD = 64
HEAD_DIM = 512
N_IDX_HEAD = 64
IDX_DIM = 128
N_SWA = 128
COMPRESS_RATIO = 4


@dataclass
class Workload:
    name: str
    kind: str              # "decode", "prefill", "dense" (ratio-128 layers: all rows, no indexer)
                           # or "pool" (cache producer: raw push + compressor pooling; n_rows = ratio)
    units: int             # decode: sequences x layers; prefill: 1
    n_rows: int            # compressed rows per unit (prefill: prior + in-chunk)
    top_k: int = 512
    queries: int = 1       # queries per unit (prefill chunk length T)
    heavy_frac: float = 0.0
    heavy_scale: float = 4.0
    seed: int = 0
    heads: int = 64        # query heads (64 Flash, 128 Pro)
    fp8: bool = False      # compressed rows kept in the FP8 row store (E4M3 codes + row scales)
    extra: dict = field(default_factory=dict)

    @property
    def query_units(self) -> int:
        """Query-token x layer units one pass of the step processes."""
        return self.units * self.queries


WORKLOADS = {
    "decode_1x1024": Workload("decode_1x1024", "decode", 1, 1024),
    "decode_8x16384": Workload("decode_8x16384", "decode", 8, 16384),
    "decode_32x43x65536": Workload("decode_32x43x65536", "decode", 32 * 43, 65536),
    "prefill_2048x65536": Workload("prefill_2048x65536", "prefill", 1, 65536 + 512,
                                   queries=2048, extra=dict(prior_rows=65536)),
    "longctx_4x262144": Workload("longctx_4x262144", "decode", 4, 262144,
                                 heavy_frac=0.05),
    # Ratio-128 layers ("DwarfStar(ds4.c) のアーキテクチャを読む" §3-2: the odd
    # layers 3..41 of the Flash shape fold 128 tokens into one row and attend to
    # all rows): 32 sequences x 20 layers at 1M tokens of context = 8,192 rows.
    "dense_32x20x8192": Workload("dense_32x20x8192", "dense", 32 * 20, 8192, top_k=0),
    # Pro shape ("DwarfStar(ds4.c) のアーキテクチャを読む" §2: 128 heads, indexer
    # top_k 1,024; 61 layers, of which the even layers 2..60 are ratio-4
    # indexer layers): 16 sequences x 30 layers at depth 65,536 rows.
    "pro_decode_16x30x65536": Workload("pro_decode_16x30x65536", "decode", 16 * 30, 65536, top_k=1024,
                                       heads=128),
    # Cache producer at a ratio-128 boundary (§3-1, §3-2): for each of 32
    # sequences x 20 ratio-128 layers, push the new token's raw row and pool
    # the 128-row (kv, score) frontier of width 512 into one compressed row.
    "pool_32x20x128": Workload("pool_32x20x128", "pool", 32 * 20, 128, top_k=0),
    # The decode and prefill workloads with the compressed rows in the FP8 row
    # store (§3-2: the compressed row's FP8 round trip): the same fp32 values,
    # stored as E4M3 codes with one power-of-two scale per row.
    "decode_fp8_32x43x65536": Workload("decode_fp8_32x43x65536", "decode", 32 * 43, 65536, fp8=True),
    "prefill_fp8_2048x65536": Workload("prefill_fp8_2048x65536", "prefill", 1, 65536 + 512,
                                       queries=2048, extra=dict(prior_rows=65536), fp8=True),
}


def _gen(seed: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    # Distinct, reproducible stream per tensor: mix (seed, stream) into one 63-bit seed.
    g.manual_seed((seed * 0x9E3779B97F4A7C15 + stream * 0xBF58476D1CE4E5B9 + 1) & ((1 << 63) - 1))
    return g


def normal_fill_(dst: torch.Tensor, d: int, seed: int, stream: int, chunk_elems: int = 1 << 28):
    """Fill dst (bf16 or fp16, any device) with N(0,1)/sqrt(d), rounded to nearest even.

    Generates in fp32 chunks so multi-GB tensors need only a bounded temporary.
    """
    g = _gen(seed, stream, dst.device)
    flat = dst.view(-1)
    inv = 1.0 / math.sqrt(d)
    for s in range(0, flat.numel(), chunk_elems):
        n = min(chunk_elems, flat.numel() - s)
        t = torch.randn(n, generator=g, device=dst.device, dtype=torch.float32)
        t.mul_(inv)
        flat[s:s + n].copy_(t)
    return dst


def normal_fp32_chunks(n_rows: int, d: int, seed: int, stream: int, device="cpu", chunk_elems: int = 1 << 28):
    """The fp32 values normal_fill_ draws for a [n_rows, d] tensor with the same
    (seed, stream), before its rounding, chunk by chunk: yields (first_row,
    fp32 [rows, d]).  The FP8 row store is built from these values by the
    caller's own quantiser (this module does none of that arithmetic)."""
    assert chunk_elems % d == 0
    g = _gen(seed, stream, device)
    inv = 1.0 / math.sqrt(d)
    total = n_rows * d
    for s in range(0, total, chunk_elems):
        n = min(chunk_elems, total - s)
        t = torch.randn(n, generator=g, device=device, dtype=torch.float32)
        t.mul_(inv)
        yield s // d, t.view(-1, d)


def decode_rows_fp32_chunks(units, n_cap, device="cpu", seed=0):
    """The decode workload's compressed rows (make_decode_inputs' x["rows"]) as
    fp32 values before their bf16 rounding, in chunks of whole rows."""
    return normal_fp32_chunks(units * n_cap, HEAD_DIM, seed, 6, device)


def prefill_rows_fp32_chunks(n_cap, device="cpu", seed=0):
    """make_prefill_inputs' x["rows"] as fp32 values before rounding, in chunks."""
    return normal_fp32_chunks(n_cap, HEAD_DIM, seed, 16, device)


def uniform_fill_(dst: torch.Tensor, seed: int, stream: int):
    g = _gen(seed, stream, dst.device)
    dst.copy_(torch.rand(dst.shape, generator=g, device=dst.device, dtype=torch.float32))
    return dst


def apply_heavy_tail_(ik: torch.Tensor, frac: float, scale: float, seed: int, stream: int):
    """Scale a seeded fraction `frac` of the indexer keys (rows of the last-but-one
    dim) by `scale` (a power of two, so bf16 stays exact), giving the score
    distribution a heavy tail and sharp top-k boundaries."""
    g = _gen(seed, stream, ik.device)
    rows = ik.view(-1, ik.shape[-1])
    chunk = 1 << 22
    for s in range(0, rows.shape[0], chunk):
        n = min(chunk, rows.shape[0] - s)
        heavy = torch.rand(n, generator=g, device=ik.device) < frac
        seg = rows[s:s + n]
        seg[heavy] = seg[heavy] * scale
    return ik


def make_decode_inputs(units, n_cap, device="cpu", seed=0, n_rows=None, n_raw=None,
                       heavy_frac=0.0, heavy_scale=4.0, q_scale=1.0, with_indexer=True, n_head=N_HEAD,
                       with_rows=True):
    """Decode-step inputs for `units` independent (sequence x layer) caches.

    n_rows / n_raw: per-unit valid compressed rows / raw-window slots (int or
    list); default full.  q_scale multiplies the attention query (x32 gives a
    peaked softmax for stress cases).  with_indexer=False leaves out iq, w and
    ik (the ratio-128 layers have no indexer).  with_rows=False leaves out the
    bf16 rows (an FP8 row store is built from decode_rows_fp32_chunks instead).
    """
    dev = torch.device(device)
    bf, hf = torch.bfloat16, torch.float16
    x = {}
    x["q"] = normal_fill_(torch.empty(units, n_head, HEAD_DIM, dtype=bf, device=dev), HEAD_DIM, seed, 1)
    if q_scale != 1.0:
        x["q"].mul_(q_scale)
    if with_indexer:
        x["iq"] = normal_fill_(torch.empty(units, N_IDX_HEAD, IDX_DIM, dtype=bf, device=dev), IDX_DIM, seed, 2)
        x["w"] = uniform_fill_(torch.empty(units, N_IDX_HEAD, dtype=torch.float32, device=dev), seed, 3)
        x["ik"] = normal_fill_(torch.empty(units, n_cap, IDX_DIM, dtype=bf, device=dev), IDX_DIM, seed, 4)
        if heavy_frac > 0:
            apply_heavy_tail_(x["ik"], heavy_frac, heavy_scale, seed, 5)
    if with_rows:
        x["rows"] = normal_fill_(torch.empty(units, n_cap, HEAD_DIM, dtype=bf, device=dev), HEAD_DIM, seed, 6)
    x["raw"] = normal_fill_(torch.empty(units, N_SWA, HEAD_DIM, dtype=hf, device=dev), HEAD_DIM, seed, 7)
    nr = n_rows if n_rows is not None else n_cap
    nw = n_raw if n_raw is not None else N_SWA
    x["n_rows"] = torch.tensor([nr] * units if isinstance(nr, int) else list(nr), dtype=torch.int32, device=dev)
    x["n_raw"] = torch.tensor([nw] * units if isinstance(nw, int) else list(nw), dtype=torch.int32, device=dev)
    return x


def prefill_positions(T, prior_rows, ratio=COMPRESS_RATIO):
    """Positions of a prefill chunk that starts right after `prior_rows`
    ratio-4 compressed rows (one row per 4 tokens, "DwarfStar(ds4.c) の
    アーキテクチャを読む" §3-2).  Row i covers tokens ratio*i .. ratio*i+3 and
    is finalised at its last token; the chunk's queries are tokens P0..P0+T-1.

    Returns (q_pos [T], row_pos [prior_rows + T // ratio], P0).
    """
    P0 = ratio * prior_rows
    n_new = T // ratio
    i = torch.arange(prior_rows + n_new, dtype=torch.int64)
    row_pos = (ratio * i + (ratio - 1)).to(torch.int32)
    q_pos = (P0 + torch.arange(T, dtype=torch.int64)).to(torch.int32)
    return q_pos, row_pos, P0


def make_prefill_inputs(T, prior_rows, device="cpu", seed=0, q_scale=1.0, n_head=N_HEAD, with_rows=True):
    """Prefill-chunk inputs: T queries over prior_rows + T/4 compressed rows, and
    a contiguous fp16 raw buffer holding positions P0-128 .. P0+T-1."""
    dev = torch.device(device)
    bf, hf = torch.bfloat16, torch.float16
    q_pos, row_pos, P0 = prefill_positions(T, prior_rows)
    n_cap = row_pos.numel()
    x = {}
    x["q"] = normal_fill_(torch.empty(T, n_head, HEAD_DIM, dtype=bf, device=dev), HEAD_DIM, seed, 11)
    if q_scale != 1.0:
        x["q"].mul_(q_scale)
    x["iq"] = normal_fill_(torch.empty(T, N_IDX_HEAD, IDX_DIM, dtype=bf, device=dev), IDX_DIM, seed, 12)
    x["w"] = uniform_fill_(torch.empty(T, N_IDX_HEAD, dtype=torch.float32, device=dev), seed, 13)
    x["ik"] = normal_fill_(torch.empty(n_cap, IDX_DIM, dtype=bf, device=dev), IDX_DIM, seed, 14)
    if with_rows:
        x["rows"] = normal_fill_(torch.empty(n_cap, HEAD_DIM, dtype=bf, device=dev), HEAD_DIM, seed, 16)
    raw_pos0 = max(P0 - N_SWA, 0)
    n_raw_rows = P0 + T - raw_pos0
    x["raw"] = normal_fill_(torch.empty(n_raw_rows, HEAD_DIM, dtype=hf, device=dev), HEAD_DIM, seed, 17)
    x["q_pos"] = q_pos.to(dev)
    x["row_pos"] = row_pos.to(dev)
    x["n_rows"] = torch.tensor([n_cap], dtype=torch.int32, device=dev)
    x["raw_pos0"] = raw_pos0
    x["P0"] = P0
    return x


def as_u16(t: torch.Tensor):
    """The raw 16-bit storage of a bf16/fp16 tensor as a numpy uint16 array (CPU copy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view("uint16")


def make_pool_inputs(units, ratio, width=HEAD_DIM, device="cpu", seed=0):
    """Cache-producer inputs: a frontier of `ratio` (kv, score) rows per unit
    (fp32; kv ~ N(0,1)/sqrt(width), score ~ N(0,1)), the new token's row, a
    raw ring per unit and the position of the new token (a ratio boundary
    far into the context)."""
    dev = torch.device(device)
    x = {}
    x["kv"] = torch.empty(units, ratio, width, dtype=torch.float32, device=dev)
    normal_fill_(x["kv"], width, seed, 11)
    x["score"] = torch.empty(units, ratio, width, dtype=torch.float32, device=dev)
    normal_fill_(x["score"], 1, seed, 12)
    x["row"] = torch.empty(units, width, dtype=torch.float32, device=dev)
    normal_fill_(x["row"], width, seed, 13)
    x["raw"] = torch.zeros(units, N_SWA, HEAD_DIM, dtype=torch.float16, device=dev)
    x["n_raw"] = torch.full((units,), N_SWA, dtype=torch.int32, device=dev)
    x["pos"] = torch.full((units,), 128 * 8191 - 1, dtype=torch.int32, device=dev)
    return x
