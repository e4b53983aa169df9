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


@pytest.mark.parametrize("batch,next_n,W", [(300, 3, 32768), (1100, 1, 20000), (400, 2, 100000),
                                            (153, 1, 20000), (1024, 1, 20000), (1025, 1, 20000),
                                            (77, 4, 40960)])
def test_many_rows_longest_first(batch, next_n, W):
    # More rows than one wave of CTAs, on both shared-memory kernels (one CTA
    # of 1024 threads per SM up to 40960 columns, ranking the batch once and
    # taking one row of every length tier; two of 512 beyond, each ranking
    # for its own row, where rows longer than 16384 columns are re-read from
    # L2 on each pass): one row past a wave (one CTA takes two rows), the
    # largest batch the ranking takes (1024 requests) and one more (one CTA
    # per row in row order), a request's rows kept together (next_n = 4).
    # The same sets as the oracle's top-k on the same values, and 0..n-1 then
    # -1 for the short rows.  Contexts span empty to the full width and repeat.
    rng = np.random.default_rng(batch + W)
    k = 2048
    ctx = np.exp(rng.uniform(0, np.log(W), size=batch)).astype(np.int64)
    ctx[rng.integers(0, batch, 8)] = 0
    ctx[rng.integers(0, batch, 8)] = W
    ctx[:20] = ctx[20:40]                                  # equal contexts in different places
    rows = batch * next_n
    vals = rng.standard_normal((rows, W)).astype(np.float32)
    got = _run_on_values(vals, ctx, next_n, k, W)
    n_r = np.clip(np.repeat(ctx, next_n) - next_n + np.tile(np.arange(next_n), batch) + 1, 0, W)
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


# ---- the large configurations: rows past byte 2^31, sweep points, KV past 2^31

def assert_topk_exact_on_device(view: torch.Tensor, idx: torch.Tensor, n_r: torch.Tensor, k: int,
                                what: str, chunk: int = 64):
    """The top-k property on the GPU's own fp32 logits, for every row, checked
    on the device (any size): entries [min(k, n_r), k) are -1; the others are
    distinct columns in [0, n_r); and no column of the row holds a value
    greater than the smallest selected one unless it is selected too (fewer
    than min(k, n_r) columns lie strictly above it).  Columns past n_r are
    -inf, so they never count."""
    rows = idx.shape[0]
    m = torch.clamp(n_r, max=k)
    col = torch.arange(k, device=idx.device)[None, :]
    live = col < m[:, None]
    assert bool((idx[~live] == -1).all()), f"{what}: padding not -1"
    assert bool(((idx >= 0) & (idx < n_r[:, None]))[live].all()), f"{what}: index outside [0, n_r)"
    srt, _ = torch.sort(torch.where(live, idx, torch.full_like(idx, -1)), dim=1)
    dup = (srt[:, 1:] == srt[:, :-1]) & (srt[:, 1:] >= 0)
    assert not bool(dup.any()), f"{what}: duplicate indices"
    for r0 in range(0, rows, chunk):
        r1 = min(rows, r0 + chunk)
        v = view[r0:r1]
        sel = torch.gather(v, 1, idx[r0:r1].clamp(min=0).long())
        sel = torch.where(live[r0:r1], sel, torch.full_like(sel, float("inf")))
        thr = sel.min(dim=1).values
        above = (v > thr[:, None]).sum(dim=1)
        full = m[r0:r1] > 0
        assert bool((above[full] < m[r0:r1][full]).all()), f"{what}: rows {r0}..{r1} miss a larger value"


WIDE_ROWS = [0, 1, 510, 511, 512, 513, 767, 1022, 1023]


@pytest.mark.slow
def test_wide_rows_past_2g():
    """The wide workload (logits [1024, 1<<20] fp32, 4 GiB; rows >= 512 start
    past byte 2^31 of the buffer, the rows an int32 byte offset loses: aiter
    PR 4244, "Root cause").  Logits, then top-k, on a sentinel-filled buffer:
    every row's top-k property on the device; sampled rows (always 510-513,
    767, 1022, 1023) against the fp64 oracle with the tie tolerance; then
    the oracle's own fp32 values written into those rows of the same 4 GiB
    buffer, so they still lie past 2^31 bytes, and the sets exactly equal to
    the oracle's top-k of those values."""
    w = synth.wide()
    logits = torch.full((w.rows, w.logits_stride), 12345.0, dtype=torch.float32, device="cuda")
    _, view, dev = run_logits(w, logits=logits)
    idx = run_topk(view, dev, w)
    torch.cuda.synchronize()
    n_r = row_ctx(w, cap_table=False)
    n_dev = torch.from_numpy(n_r).cuda()
    assert_topk_exact_on_device(view, idx, n_dev, w.topk, "wide")
    rng = np.random.default_rng(1)
    sample = sorted(set(WIDE_ROWS + rng.integers(0, w.rows, 8).tolist()))
    ref = oracle_logits(w, rows=sample, W=int(n_r[sample].max()) + 1)
    got = idx[sample].cpu().numpy()
    assert_topk_valid(got, ref, n_r[sample], w.topk, "wide top-k")
    # The oracle's fp32 values in the same rows of the 4 GiB buffer.
    ref32 = ref.astype(np.float32)
    for i, r in enumerate(sample):
        view[r, :ref32.shape[1]] = torch.from_numpy(ref32[i]).cuda()
    idx2 = run_topk(view, dev, w)
    torch.cuda.synchronize()
    assert_topk_exact(idx2[sample].cpu().numpy(), ref32, n_r[sample], w.topk)


@pytest.mark.slow
def test_wide_fused_rows_past_2g():
    """The fused logits + top-k launch on the wide workload: logits bit-equal
    to the logits launch's, indices entry for entry equal to the top-k
    launch's on them, the top-k property on every row, sampled rows (rows
    past byte 2^31 always among them) against the oracle."""
    w = synth.wide()
    dev = w.to_device()
    logits = torch.full((w.rows, w.logits_stride), 4321.0, dtype=torch.float32, device="cuda")
    idx = torch.full((w.rows, w.topk), -7, dtype=torch.int32, device="cuda")
    ws = torch.zeros(sai.logits_topk_workspace_bytes(w.batch) // 4, dtype=torch.int32, device="cuda")
    sai.paged_mqa_logits_topk(dev["q"], dev["kv"], w.page_size, dev["weights"], dev["context_lens"],
                              dev["block_table"], logits, w.max_model_len, w.topk, idx, ws,
                              num_pages=w.pool.num_pages)
    torch.cuda.synchronize()
    assert bool((ws == 0).all())
    n_r = row_ctx(w, cap_table=False)
    n_dev = torch.from_numpy(n_r).cuda()
    assert_topk_exact_on_device(logits, idx, n_dev, w.topk, "wide fused")
    rng = np.random.default_rng(2)
    sample = sorted(set(WIDE_ROWS + rng.integers(0, w.rows, 8).tolist()))
    ref = oracle_logits(w, rows=sample, W=int(n_r[sample].max()) + 1)
    assert_topk_valid(idx[sample].cpu().numpy(), ref, n_r[sample], w.topk, "wide fused top-k")
    # Against the two launches, on the same inputs: bit-equal logits, same indices.
    sep_idx = run_topk(logits, dev, w)
    torch.cuda.synchronize()
    assert torch.equal(sep_idx, idx), "fused indices differ from the top-k launch on the fused logits"
    sep = torch.empty_like(logits)
    run_logits(w, dev=dev, logits=sep)
    torch.cuda.synchronize()
    for r0 in range(0, w.rows, 128):
        assert torch.equal(sep[r0:r0 + 128], logits[r0:r0 + 128]), f"rows {r0}.. differ"


@pytest.mark.slow
def test_kv_pages_past_2g():
    """kv-2G: every page lies wholly past byte 2^31 of a 2.24 GB pool."""
    _both_checks(synth.kv2g())


SWEEP_SAMPLE = [(8, 1, 64, 1, 8192), (8, 4, 128, 16, 512), (16, 2, 64, 64, 512),
                (16, 4, 128, 1, 65536), (64, 1, 128, 16, 8192), (64, 4, 64, 256, 2),
                (256, 2, 128, 16, 8192), (256, 1, 64, 1, 131072), (256, 4, 128, 64, 512),
                (16, 1, 64, 16, 131072), (64, 2, 64, 256, 8192)]


@pytest.mark.parametrize("pt", SWEEP_SAMPLE, ids=lambda p: "P%d_n%d_H%d_B%d_ctx%d" % p)
def test_sweep_points(pt):
    """Sweep points: the top-k property on every row on the device; all rows
    against the oracle where the oracle is quick, else the first, middle and
    last rows."""
    w = synth.sweep_point(*pt)
    _, view, dev = run_logits(w)
    idx = run_topk(view, dev, w)
    torch.cuda.synchronize()
    n_r = row_ctx(w, cap_table=False)
    assert_topk_exact_on_device(view[:, :w.max_model_len], idx, torch.from_numpy(n_r).cuda(), w.topk,
                                "sweep")
    rows = list(range(w.rows)) if w.rows * w.max_model_len <= 4_000_000 else sorted({0, w.rows // 2, w.rows - 1})
    ref = oracle_logits(w, rows=rows)
    assert_topk_valid(idx[rows].cpu().numpy(), ref, n_r[rows], w.topk, "sweep top-k")
