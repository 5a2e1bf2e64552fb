"""Comparison rules for the CUDA path against the fp64 oracle (test helpers).

Index sets: the device's selected set G and the oracle's set O must have the
same size, and every row in their symmetric difference must score, by the
oracle, within 1e-5 relative of the oracle's k-th score (a near-tie that fp32
scoring may order either way).

Attention outputs: the oracle recomputes the attention on the device's own
selected set; then max |d| <= 2e-3 and, element-wise, |d| <= 1e-2 * max(|ref|,
rms(ref of that unit)).  The RMS floor keeps the relative bound meaningful for
outputs near zero (an attention output is a convex combination of rows, so an
element can be arbitrarily close to 0 while the unit's scale is not).
"""
import concurrent.futures as cf
import math
import os

import numpy as np
import torch

import oracle

INDEX_BAND = 1e-5
OUT_ATOL = 2e-3
OUT_RTOL = 1e-2


def u16(t):
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def pool():
    return cf.ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1)))


def score_tolerance(iq_u16, w, ik_u16, n_rows):
    """Bound on |fp32 device score - exact score| per row: (128 + 64 + 2) ulps of
    the absolute-value sum  sum_h |w_h| sum_d |iq_hd ik_rd|  (the worst case of
    fp32 accumulation over 128 products then 64 weighted heads)."""
    qd = np.abs(torch.from_numpy(iq_u16.view(np.int16)).view(torch.bfloat16).double().numpy())
    kd = np.abs(torch.from_numpy(ik_u16[:n_rows].view(np.int16)).view(torch.bfloat16).double().numpy())
    s_abs = (kd @ qd.T) @ np.abs(w.astype(np.float64))
    return 194 * 2.0 ** -24 * s_abs + 1e-30


def check_scores(gpu_scores, ref_scores, tol):
    g = np.asarray(gpu_scores, np.float64)
    r = np.asarray(ref_scores, np.float64)
    inv = np.isneginf(r)
    assert np.array_equal(np.isneginf(g), inv), "visibility mask differs"
    d = np.abs(g[~inv] - r[~inv])
    t = np.broadcast_to(tol, r.shape)[~inv]
    bad = d > t
    assert not bad.any(), f"{bad.sum()} scores off: max excess {(d - t).max():.3e}"
    return float(d.max()) if d.size else 0.0


def check_index_set(gpu_idx, gpu_count, ref_scores, top_k):
    """Returns the number of near-tie swaps accepted."""
    s = np.asarray(ref_scores, np.float64)
    o_idx, kth = oracle.topk_select(s, top_k)
    g = np.asarray(gpu_idx[:gpu_count], np.int64)
    assert gpu_count == len(o_idx), f"count {gpu_count} != oracle {len(o_idx)}"
    assert np.all(np.diff(g) > 0), "device indices not strictly ascending"
    assert np.all(np.asarray(gpu_idx[gpu_count:]) == -1), "padding must be -1"
    diff = np.setxor1d(g, o_idx)
    if diff.size:
        band = INDEX_BAND * abs(kth)
        off = np.abs(s[diff] - kth)
        assert np.all(off <= band), f"rows {diff[off > band][:8]} differ beyond the 1e-5 band"
    return int(diff.size)


def check_output(gpu_out, ref_out, gpu_lse=None, ref_lse=None):
    g = np.asarray(gpu_out, np.float64)
    r = np.asarray(ref_out, np.float64)
    d = np.abs(g - r)
    rms = math.sqrt(float(np.mean(r * r))) if r.size else 0.0
    assert np.all(np.isfinite(g)), "non-finite output"
    assert d.max() <= OUT_ATOL, f"max |d| {d.max():.3e} > {OUT_ATOL}"
    rel = d / np.maximum(np.abs(r), max(rms, 1e-30))
    assert rel.max() <= OUT_RTOL, f"max rel {rel.max():.3e} > {OUT_RTOL}"
    if gpu_lse is not None:
        gl, rl = np.asarray(gpu_lse, np.float64), np.asarray(ref_lse, np.float64)
        assert np.array_equal(np.isneginf(gl), np.isneginf(rl))
        fin = np.isfinite(rl)
        assert np.all(np.abs(gl[fin] - rl[fin]) <= 1e-4 * np.maximum(1, np.abs(rl[fin])))
    return dict(max_abs=float(d.max()), max_rel=float(rel.max()), rel_rms=float(d.max() / max(rms, 1e-30)))
