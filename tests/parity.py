"""Helpers of the GPU parity tests: run the library on a workload, compare with
the oracle.

Tolerance (logits): |gpu - oracle| <= ATOL + RTOL * |oracle| per element, with
ATOL = RTOL = 1e-3; -inf and NaN positions must match exactly; padding
columns [W, stride) and guard rows keep their sentinel bit for bit.

Top-k: every row's entries [min(k, n_r), k) are -1 exactly; entries
[0, min(k, n_r)) are distinct columns in [0, n_r); rows with n_r <= k hold
exactly {0..n_r-1}; otherwise the index set equals the oracle's except for
indices whose oracle logit lies within the logits tolerance of the oracle's
k-th largest value.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import sparse_attention_indexer_03_gb300 as sai

ATOL = 1e-3
RTOL = 1e-3
SENTINEL = 12345.0


def row_ctx(w, cap_table: bool = True) -> np.ndarray:
    """Row lengths by the oracle's rule (table capacity included or not)."""
    if cap_table:
        return oracle.row_context_lengths(w.context_lens, w.next_n, w.max_model_len,
                                          w.block_table.shape[1], w.page_size)
    return oracle.row_context_lengths(w.context_lens, w.next_n, w.max_model_len,
                                      w.max_model_len, 1)


def alloc_logits(rows: int, stride: int, guard_rows: int = 1, device="cuda") -> tuple:
    """Sentinel-filled [rows + 2 * guard_rows, stride] buffer and the [rows, stride] view."""
    buf = torch.full((rows + 2 * guard_rows, stride), SENTINEL, dtype=torch.float32, device=device)
    return buf, buf[guard_rows:guard_rows + rows]


def run_logits(w, dev=None, stride=None, guard_rows=1, status=None, kv_layout=None, logits=None):
    """Launch the library's logits on a workload; returns (buffer, view, dev)."""
    dev = dev or w.to_device()
    stride = stride or w.logits_stride
    if logits is None:
        buf, view = alloc_logits(w.rows, stride, guard_rows)
    else:
        buf, view = logits, logits
    sai.paged_mqa_logits(dev["q"], dev["kv"], w.page_size, dev["weights"], dev["context_lens"],
                         dev["block_table"], view, w.max_model_len, num_pages=w.pool.num_pages,
                         status=status, kv_layout=kv_layout or w.layout)
    return buf, view, dev


def run_topk(view, dev, w, k=None, indices=None):
    k = k or w.topk
    if indices is None:
        indices = torch.full((w.rows, k), -7, dtype=torch.int32, device="cuda")
    sai.top_k_per_row_decode(view, dev["context_lens"], w.next_n, w.max_model_len, k, indices)
    return indices


def oracle_logits(w, rows=None, W=None):
    return oracle.paged_mqa_logits(w.q, w.pool.ids, w.pool.data, w.pool.num_pages, w.page_size,
                                   w.weights, w.context_lens, w.block_table, w.next_n,
                                   W or w.max_model_len, layout=w.layout, rows=rows)


def assert_logits_close(gpu: np.ndarray, ref: np.ndarray, what: str = "logits"):
    gpu = np.asarray(gpu, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    ninf_g, ninf_r = np.isneginf(gpu), np.isneginf(ref)
    bad = np.argwhere(ninf_g != ninf_r)
    assert len(bad) == 0, f"{what}: -inf mask differs at {bad[:5].tolist()}"
    nan_g, nan_r = np.isnan(gpu), np.isnan(ref)
    bad = np.argwhere(nan_g != nan_r)
    assert len(bad) == 0, f"{what}: NaN mask differs at {bad[:5].tolist()}"
    fin = np.isfinite(ref)
    assert np.isfinite(gpu[fin]).all(), f"{what}: non-finite where oracle is finite"
    err = np.abs(gpu[fin] - ref[fin])
    lim = ATOL + RTOL * np.abs(ref[fin])
    if err.size:
        worst = np.argmax(err - lim)
        assert (err <= lim).all(), (f"{what}: {(err > lim).sum()} elements out of tolerance; worst "
                                    f"gpu={gpu[fin][worst]!r} oracle={ref[fin][worst]!r}")


def assert_untouched(buf: torch.Tensor, view: torch.Tensor, W: int, guard_rows: int):
    """Guard rows and padding columns [W, stride) still hold the sentinel."""
    if guard_rows:
        assert bool((buf[:guard_rows] == SENTINEL).all()), "guard row above written"
        assert bool((buf[-guard_rows:] == SENTINEL).all()), "guard row below written"
    if view.shape[1] > W:
        assert bool((view[:, W:] == SENTINEL).all()), "padding columns [W, stride) written"


def assert_topk_valid(gpu_idx: np.ndarray, ref_logits: np.ndarray, n_r: np.ndarray, k: int,
                      what: str = "top-k"):
    """Top-k rule against fp64 oracle logits (see module docstring)."""
    for i in range(gpu_idx.shape[0]):
        n = int(n_r[i])
        m = min(k, n)
        row = gpu_idx[i]
        assert (row[m:] == -1).all(), f"{what}: row {i} padding not -1"
        sel = row[:m]
        assert (sel >= 0).all() and (sel < n).all(), f"{what}: row {i} index out of [0, {n})"
        assert len(np.unique(sel)) == m, f"{what}: row {i} duplicate indices"
        if n <= k:
            assert set(sel.tolist()) == set(range(n)), f"{what}: row {i} short row not 0..n-1"
            continue
        vals = ref_logits[i, :n]
        kth = np.sort(vals)[::-1][k - 1]
        ref_set = set(oracle.top_k_per_row(vals[None, :], [n], k)[0].tolist())
        diff = ref_set.symmetric_difference(set(sel.tolist()))
        tol = ATOL + RTOL * abs(kth)
        for idx in diff:
            assert abs(vals[idx] - kth) <= tol, (
                f"{what}: row {i} index {idx} (oracle {vals[idx]}) not within tolerance of k-th {kth}")


def assert_topk_exact(gpu_idx: np.ndarray, fp32_logits: np.ndarray, n_r: np.ndarray, k: int):
    """GPU top-k run on the very values the oracle's top-k sees: identical sets."""
    ref = oracle.top_k_per_row(fp32_logits, n_r, k)
    for i in range(gpu_idx.shape[0]):
        m = min(k, int(n_r[i]))
        assert (gpu_idx[i, m:] == -1).all()
        assert set(gpu_idx[i, :m].tolist()) == set(ref[i, :m].tolist()), f"row {i}"
