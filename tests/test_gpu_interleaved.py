"""GPU parity of `sai_paged_mqa_logits` on interleaved K-caches (each token's
128 value bytes followed by its 4 scale bytes, the cache the aiter PR 4244
reproducer builds), through the C ABI.

The interleaved launch stages each tile's pages as stored and rewrites them
into the layout the page-split launch loads directly, then runs the same MMA
and epilogue: on the same cache contents the two must give bit-identical
logits.  Checked against the oracle on ragged cases of every supported
(next_n, heads) and several page sizes, and against the page-split launch at
the decode and MTP workload sizes, where every CTA reuses each slot of its
ring of stages many times.
"""
import numpy as np
import pytest
import torch

import synth
import sparse_attention_indexer_03_gb300 as sai
from parity import assert_logits_close, assert_untouched, oracle_logits, run_logits

pytestmark = pytest.mark.gpu

CONFIGS = [(1, 64), (2, 64), (3, 64), (4, 64), (1, 128), (2, 128), (3, 128), (4, 128)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    sai.library()


def _launch(w, guard_rows=1):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    buf, view, _ = run_logits(w, guard_rows=guard_rows, status=status)
    torch.cuda.synchronize()
    assert_untouched(buf, view, w.max_model_len, guard_rows)
    return view, int(status.item())


@pytest.mark.parametrize("page_size", [8, 64, 256])
@pytest.mark.parametrize("next_n,heads", CONFIGS)
def test_ragged_cases_match_the_oracle(next_n, heads, page_size):
    # An empty request, one shorter than next_n, lengths off the page and tile
    # grids, W not a multiple of 128, stride > W.
    ctx = [0, 1, 2 * page_size + 3, 700, 389, next_n - 1, 1500]
    w = synth.custom(batch=len(ctx), next_n=next_n, heads=heads, page_size=page_size, context_lens=ctx,
                     max_model_len=1533, logits_stride=1541, table_stride=-(-1533 // page_size) + 1,
                     seed=page_size * 10 + next_n + heads, layout="interleaved")
    view, st = _launch(w, guard_rows=2)
    assert st == 0
    assert_logits_close(view[:, :w.max_model_len].cpu().numpy(), oracle_logits(w))


@pytest.mark.parametrize("next_n,heads", CONFIGS)
def test_many_tiles_per_cta_match_the_page_split_launch(next_n, heads):
    # About 1,900 tiles of 8-token pages: a dozen per CTA, so each slot of the
    # stage ring (2 to 6 deep) is refilled several times by alternating warps.
    rng = np.random.default_rng(next_n * 1000 + heads)
    ctx = rng.integers(3000, 9000, 40)
    kw = dict(batch=40, next_n=next_n, heads=heads, page_size=8, context_lens=ctx, max_model_len=9000,
              seed=next_n + heads)
    ws, wi = synth.custom(**kw), synth.custom(layout="interleaved", **kw)
    vs, st_s = _launch(ws)
    vi, st_i = _launch(wi)
    assert st_s == 0 and st_i == 0
    assert torch.equal(vs, vi)
    rows = np.array([0, 1, wi.rows // 2, wi.rows - 1])
    assert_logits_close(vi[rows, :wi.max_model_len].cpu().numpy(), oracle_logits(wi, rows=rows))


@pytest.mark.parametrize("name", ["decode", "mtp"])
def test_workloads_match_the_page_split_launch(name):
    ws, wi = getattr(synth, name)(), getattr(synth, name)(layout="interleaved")
    vs, st_s = _launch(ws, guard_rows=0)
    vi, st_i = _launch(wi, guard_rows=0)
    assert st_s == 0 and st_i == 0
    assert torch.equal(vs, vi)


def test_out_of_pool_pages_give_nan_and_status():
    w = synth.custom(batch=2, next_n=2, heads=64, page_size=16, context_lens=[100, 64], max_model_len=128,
                     seed=7, layout="interleaved")
    w.block_table[0, 2] = w.pool.num_pages        # tokens 32..47 of request 0
    w.block_table[1, 0] = -5                      # tokens 0..15 of request 1
    view, st = _launch(w)
    assert st & sai.STATUS_BAD_PAGE
    assert_logits_close(view[:, :w.max_model_len].cpu().numpy(), oracle_logits(w))
