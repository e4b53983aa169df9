"""GPU parity of `sai_top_k_per_row_decode` (through the C ABI).

Two checks per case: (1) on the library's own logits, the selected sets
against the fp64 oracle's with the tie tolerance; (2) on the oracle's logits
rounded to fp32 and uploaded, the sets exactly equal to the oracle's top-k of
those same values.  Short rows, -1 padding, ties and rows longer than the
shared-memory cache are covered.
"""
import numpy as np
import pytest
import torch

import synth
import sparse_attention_indexer_03_gb300 as sai
from parity import (assert_topk_exact, assert_topk_valid, oracle_logits, row_ctx, run_logits,
                    run_topk)

pytestmark = pytest.mark.gpu


def _both_checks(w, k=None):
    k = k or w.topk
    _, view, dev = run_logits(w)
    idx = run_topk(view, dev, w, k=k)
    ref = oracle_logits(w)
    n_r = row_ctx(w, cap_table=False)
    torch.cuda.synchronize()
    assert_topk_valid(idx.cpu().numpy(), ref, n_r, k)
    # Exact check on the oracle's own fp32 values.
    ref32 = torch.from_numpy(ref.astype(np.float32)).cuda()
    idx2 = run_topk(ref32, dev, w, k=k)
    torch.cuda.synchronize()
    assert_topk_exact(idx2.cpu().numpy(), ref.astype(np.float32), n_r, k)


def test_tiny():
    _both_checks(synth.tiny())


def test_decode():
    _both_checks(synth.decode())


@pytest.mark.slow
def test_mtp():
    _both_checks(synth.mtp())


@pytest.mark.parametrize("k", [1, 7, 64, 300, 2048])
def test_k_values_and_short_rows(k):
    w = synth.custom(batch=5, next_n=3, heads=64, page_size=16, context_lens=[0, 2, 299, 1500, 40],
                     max_model_len=1536, seed=k)
    _both_checks(w, k=k)


def _run_on_values(vals: np.ndarray, ctx: np.ndarray, next_n: int, k: int, W: int, stride=None):
    stride = stride or W
    rows = vals.shape[0]
    buf = torch.full((rows, stride), 777.0, dtype=torch.float32, device="cuda")
    buf[:, :vals.shape[1]] = torch.from_numpy(vals).cuda()
    cl = torch.from_numpy(ctx.astype(np.int32)).cuda()
    idx = torch.full((rows, k + 3), -7, dtype=torch.int32, device="cuda")
    sai.top_k_per_row_decode(buf, cl, next_n, W, k, idx)
    torch.cuda.synchronize()
    out = idx.cpu().numpy()
    assert (out[:, k:] == -7).all(), "entries past k written"
    return out[:, :k]


def test_ties_take_lowest_columns_in_order():
    W, k = 1000, 10
    vals = np.zeros((2, W), np.float32)
    vals[0, [5, 50, 500]] = 2.0               # 3 above, ties at 0 for the other 7
    vals[1, :] = -1.0
    vals[1, 999] = 3.0
    got = _run_on_values(vals, np.array([W, W]), 1, k, W)
    assert got[0].tolist() == [5, 50, 500, 0, 1, 2, 3, 4, 6, 7]
    assert got[1].tolist() == [999, 0, 1, 2, 3, 4, 5, 6, 7, 8]


def test_signed_zeros_infinities_and_extremes():
    W, k = 64, 6
    row = np.full(W, -np.inf, np.float32)
    row[[3, 9, 17, 30, 41, 50, 60]] = [0.0, -0.0, 1e-38, -1e-38, np.float32(3.4e38), -3.4e38, 1.0]
    got = _run_on_values(row[None, :], np.array([W]), 1, k, W)
    n_r = np.array([W])
    assert_topk_exact(got, row[None, :], n_r, k)


@pytest.mark.parametrize("W", [16384, 16385, 40000, 131072])
def test_long_rows(W):
    # Across the shared-memory cache limit and up to the sweep's longest rows.
    rng = np.random.default_rng(W)
    rows, next_n, k = 6, 2, 2048
    vals = rng.standard_normal((rows, W)).astype(np.float32)
    vals[1, ::3] = 0.5                          # many exact ties
    ctx = np.array([W, W - 7, 2000])
    got = _run_on_values(vals, ctx, next_n, k, W, stride=W + 5)
    n_r = np.clip(np.repeat(ctx, next_n) - next_n + np.tile(np.arange(next_n), 3) + 1, 0, W)
    assert_topk_exact(got, vals, n_r, k)


def _ties_order(v: np.ndarray, n: int, k: int) -> np.ndarray:
    """Expected entries of a row whose values near the k-th largest are exact
    ties: the columns above the k-th largest value ascending, then the lowest
    columns equal to it."""
    v = v[:n]
    if n <= k:
        return np.concatenate([np.arange(n), np.full(k - n, -1)])
    thr = np.sort(v)[::-1][k - 1]
    gt = np.flatnonzero(v > thr)
    eq = np.flatnonzero(v == thr)[:k - len(gt)]
    return np.concatenate([gt, eq])


@pytest.mark.parametrize("W", [20000, 65536, 131072])
def test_rows_split_over_a_cluster_match_one_cta_per_row(W):
    # Few rows wider than 16384 columns are split over a cluster of 2, 4 or 8
    # CTAs, 16384 columns each, while rows * cluster stays within four CTAs
    # per SM; more rows take one CTA each.  The selection and its order must
    # not depend on where the slices end: checked against the oracle's sets,
    # against the tie order on rows of exact ties, and entry for entry
    # against the same rows repeated until the launch takes one CTA per row.
    rng = np.random.default_rng(W + 1)
    k = 2048
    vals = np.full((5, W), -1.0, np.float32)
    vals[0, ::37] = 1.0
    vals[1, ::29] = 1.0
    vals[1, np.sort(rng.choice(W, 1000, replace=False))] = 2.0
    vals[2] = rng.standard_normal(W).astype(np.float32)
    vals[3] = rng.standard_normal(W).astype(np.float32)
    vals[4, ::5] = 3.0
    ctx = np.array([W, W, W, 1000, W - 16384 + 5])
    got = _run_on_values(vals, ctx, 1, k, W)
    assert_topk_exact(got, vals, ctx, k)
    for i in (0, 1, 3, 4):
        assert got[i].tolist() == _ties_order(vals[i], int(ctx[i]), k).tolist(), f"row {i}"
    cl = 2 if W <= 2 * 16384 else (4 if W <= 4 * 16384 else 8)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for rows in (4 * sms // cl - 4, 4 * sms // cl + 1):     # the largest clustered launch; one CTA per row
        reps = -(-rows // 5)
        again = _run_on_values(np.tile(vals, (reps, 1)), np.tile(ctx, reps), 1, k, W)
        assert (again == np.tile(got, (reps, 1))).all(), rows
