"""GPU parity of `sai_paged_mqa_logits_topk`, the fused logits + top-k launch
(through the C ABI).

Per case: the fused launch's logits are bit-identical to those of
`sai_paged_mqa_logits` on the same inputs and within tolerance of the fp64
oracle; its indices are identical, entry for entry, to what
`sai_top_k_per_row_decode` selects from those logits, and valid against the
oracle's top-k with the tie tolerance; the workspace is zero again after the
call, and a second call gives the same outputs.
"""
import numpy as np
import pytest
import torch

import synth
import sparse_attention_indexer_03_gb300 as sai
from parity import (assert_logits_close, assert_topk_valid, oracle_logits, row_ctx, run_logits,
                    run_topk)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    sai.build()


def run_fused(w, dev, k=None, workspace=None, status=None):
    k = k or w.topk
    logits = torch.full((w.rows, w.logits_stride), 4321.0, dtype=torch.float32, device="cuda")
    idx = torch.full((w.rows, k + 2), -7, dtype=torch.int32, device="cuda")
    if workspace is None:
        workspace = torch.zeros(max(1, sai.logits_topk_workspace_bytes(w.batch) // 4), dtype=torch.int32,
                                device="cuda")
    sai.paged_mqa_logits_topk(dev["q"], dev["kv"], w.page_size, dev["weights"], dev["context_lens"],
                              dev["block_table"], logits, w.max_model_len, k, idx[:, :k], workspace,
                              num_pages=w.pool.num_pages, status=status)
    return logits, idx, workspace


def _check(w, k=None, oracle=True, repeat=True, sample=None):
    k = k or w.topk
    W = w.max_model_len
    dev = w.to_device()
    logits, idx, ws = run_fused(w, dev, k)
    # The separate launches on the same inputs.
    _, view, _ = run_logits(w, dev=dev, guard_rows=0)
    ref_idx = run_topk(view, dev, w, k=k)
    torch.cuda.synchronize()
    assert bool((ws == 0).all()), "workspace not restored to zero"
    if w.logits_stride > W:
        assert bool((logits[:, W:] == 4321.0).all()), "padding columns written"
    assert bool((idx[:, k:] == -7).all()), "entries past k written"
    assert torch.equal(logits[:, :W], view[:, :W]), "fused logits differ from the logits launch"
    assert torch.equal(idx[:, :k], ref_idx), "fused indices differ from the top-k launch"
    if oracle:
        ref = oracle_logits(w)
        assert_logits_close(logits[:, :W].cpu().numpy(), ref, "fused logits")
        assert_topk_valid(idx[:, :k].cpu().numpy(), ref, row_ctx(w), k, "fused top-k")
    if sample is not None:                            # the oracle on sampled rows only
        ref = oracle_logits(w, rows=sample)
        assert_logits_close(logits[sample, :W].cpu().numpy(), ref, "fused logits (sampled rows)")
        assert_topk_valid(idx[sample, :k].cpu().numpy(), ref, row_ctx(w)[sample], k, "fused top-k (sampled rows)")
    if repeat:
        logits2, idx2, _ = run_fused(w, dev, k, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(logits2[:, :W], logits[:, :W]) and torch.equal(idx2, idx), "second call differs"


def test_tiny():
    _check(synth.tiny())


def test_decode():
    _check(synth.decode())


def _mtp_sample(w, count=48):
    """Rows of the MTP batch for the oracle: the longest rows, the empty
    request's, rows just past and just below k, and random ones."""
    n_r = row_ctx(w)
    order = np.argsort(-n_r, kind="stable")
    near_k = np.argsort(np.abs(n_r - w.topk), kind="stable")[:8]
    empty = np.flatnonzero(n_r == 0)[:2]
    rng = np.random.default_rng(5)
    rows = set(order[:12].tolist()) | set(near_k.tolist()) | set(empty.tolist())
    rows |= set(rng.integers(0, w.rows, count).tolist())
    return sorted(rows)


@pytest.mark.slow
def test_mtp():
    w = synth.mtp()
    _check(w, oracle=False, sample=_mtp_sample(w))


@pytest.mark.parametrize("next_n,heads", [(1, 64), (2, 128), (3, 64), (3, 128), (4, 64), (4, 128)])
@pytest.mark.parametrize("page_size", [8, 64, 256])
def test_shapes(page_size, next_n, heads):
    w = synth.custom(batch=7, next_n=next_n, heads=heads, page_size=page_size,
                     context_lens=[0, 1, 129, 2500, 700, 3, 4096], max_model_len=4096,
                     seed=page_size * 10 + next_n)
    _check(w, k=256)


@pytest.mark.parametrize("k", [1, 5, 128, 2048])
def test_k_values_and_short_rows(k):
    w = synth.custom(batch=6, next_n=2, heads=64, page_size=16, context_lens=[2, 0, 300, 1500, 2049, 1],
                     max_model_len=2560, seed=100 + k)
    _check(w, k=k)


def test_many_small_requests():
    # More requests than CTAs, most with one tile: the per-request counters
    # see many CTAs complete several requests each.
    rng = np.random.default_rng(7)
    ctx = rng.integers(0, 400, size=700)
    ctx[::50] = 0
    w = synth.custom(batch=700, next_n=1, heads=64, page_size=16, context_lens=ctx, max_model_len=512,
                     seed=7)
    _check(w, k=64)


@pytest.mark.parametrize("next_n,heads", [(1, 64), (4, 64), (2, 128)])
def test_fill_heavy_launch(next_n, heads):
    # The -inf fill outweighs the tiles four times over: every CTA takes fill
    # units from the workspace's grid-wide counter, and the epilogue warps
    # select rows while the other warps fill.  Rows shorter than k (written
    # by the CTA that completes their request), rows longer than k (through
    # the ready queue), an empty request, and a width that is not a multiple
    # of the 4096-column fill unit, with a padded row stride.
    ctx = [0, 1, 127, 128, 129, 2047, 2048, 2049, 2050, 3000, 4500, 130, 2100, 3, 2600, 3777]
    w = synth.custom(batch=16, next_n=next_n, heads=heads, page_size=16, context_lens=ctx,
                     max_model_len=400000, logits_stride=400128, topk=2048, seed=40 + next_n + heads)
    _check(w, k=2048)


@pytest.mark.parametrize("batch", [1, 31, 32, 33, 95, 511, 512, 513])
def test_partition_batch_edges(batch):
    # The work partition reads a batch of up to 512 requests R = ceil(B / 32)
    # per lane (the last lanes partly or wholly past the batch) and walks
    # larger batches 32 requests at a time: batch sizes at those edges, with
    # empty requests and requests of one tile, through both launches.
    rng = np.random.default_rng(batch)
    ctx = rng.integers(0, 600, size=batch)
    ctx[::7] = 0
    ctx[1::11] = 128
    w = synth.custom(batch=batch, next_n=2, heads=64, page_size=16, context_lens=ctx, max_model_len=640,
                     seed=500 + batch)
    _check(w, k=64)


def test_all_contexts_empty():
    w = synth.custom(batch=5, next_n=2, heads=64, page_size=16, context_lens=[0, 0, 0, 0, 0],
                     max_model_len=256, seed=3)
    _check(w, k=16)


def test_context_clamped_to_table():
    # ctx beyond the table's capacity: rows are clamped to the capacity for
    # both the logits and the selection.
    w = synth.custom(batch=3, next_n=2, heads=64, page_size=16, context_lens=[100, 900, 40],
                     max_model_len=1024, table_stride=32, seed=11)
    dev = w.to_device()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    logits, idx, ws = run_fused(w, dev, k=64, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & sai.STATUS_CTX_CLAMPED
    assert bool((ws == 0).all())
    ref = oracle_logits(w)
    assert_logits_close(logits[:, :w.max_model_len].cpu().numpy(), ref)
    assert_topk_valid(idx[:, :64].cpu().numpy(), ref, row_ctx(w, cap_table=True), 64)
    logits2, idx2, _ = run_fused(w, dev, k=64, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(idx2, idx) and torch.equal(logits2, logits)


def test_workspace_too_small_is_rejected():
    w = synth.tiny()
    dev = w.to_device()
    ws = torch.zeros(12, dtype=torch.int32, device="cuda")       # batch 2 needs 13 words
    with pytest.raises(sai.SaiError) as e:
        run_fused(w, dev, workspace=ws)
    assert e.value.code == sai.ERR_WORKSPACE
