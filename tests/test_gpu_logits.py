"""GPU parity of `sai_paged_mqa_logits` against the fp64 oracle (through the C ABI).

Full tensors for the small and medium workloads, sampled rows plus
any-size properties for the large ones, and the edge cases of the method
(empty and short MTP contexts, ragged widths and strides, out-of-pool page
ids, contexts longer than the output or the table, outputs and KV pages past
2^31 bytes).
"""
import numpy as np
import pytest
import torch

import synth
import sparse_attention_indexer_03_gb300 as sai
from conftest import golden_rows
from parity import (SENTINEL, alloc_logits, assert_logits_close, assert_untouched, oracle_logits,
                    row_ctx, run_logits)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    sai.library()


def _full_check(w, guard_rows=1, stride=None, layout=None):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    buf, view, dev = run_logits(w, stride=stride, guard_rows=guard_rows, status=status, kv_layout=layout)
    torch.cuda.synchronize()
    assert_untouched(buf, view, w.max_model_len, guard_rows)
    ref = oracle_logits(w)
    assert_logits_close(view[:, :w.max_model_len].cpu().numpy(), ref)
    return buf, view, dev, int(status.item())


def test_tiny():
    _, _, _, st = _full_check(synth.tiny())
    assert st == 0


def test_decode():
    _, _, _, st = _full_check(synth.decode())
    assert st == 0


@pytest.mark.slow
def test_mtp():
    w = synth.mtp()
    assert (w.context_lens == 0).sum() == 1
    _, _, _, st = _full_check(w, guard_rows=0)
    assert st == 0


@pytest.mark.parametrize("page_size", [8, 16, 32, 64, 128, 256])
@pytest.mark.parametrize("next_n,heads", [(1, 64), (2, 128), (3, 64), (3, 128), (4, 64), (4, 128)])
def test_page_sizes_and_mtp_rows(page_size, next_n, heads):
    # Ragged everything: contexts not multiples of the page or of 128, an empty
    # request, one shorter than next_n, W not a multiple of 128, stride > W.
    ctx = [0, 1, 2 * page_size + 3, 700, 389, next_n - 1]
    w = synth.custom(batch=len(ctx), next_n=next_n, heads=heads, page_size=page_size,
                     context_lens=ctx, max_model_len=733, logits_stride=741,
                     table_stride=-(-733 // page_size) + 1, seed=page_size * 10 + next_n)
    _, _, _, st = _full_check(w, guard_rows=2)
    assert st == 0


@pytest.mark.parametrize("layout", ["split", "interleaved"])
def test_kv_layouts(layout):
    w = synth.custom(batch=3, next_n=2, heads=64, page_size=16, context_lens=[333, 5, 1000],
                     max_model_len=1024, seed=3, layout=layout)
    _, _, _, st = _full_check(w)
    assert st == 0


def test_padded_table_entries_are_never_read():
    # Table entries past ceil(ctx / P) hold poison (INT32_MAX, -1); none may be
    # read, so no status bit may be raised.
    w = synth.custom(batch=3, next_n=1, heads=64, page_size=16, context_lens=[40, 17, 0],
                     max_model_len=256, table_stride=16, seed=5)
    for b, n in enumerate([40, 17, 0]):
        used = -(-n // 16)
        w.block_table[b, used:] = np.where(np.arange(16 - used) % 2 == 0, 2**31 - 1, -1)
    _, _, _, st = _full_check(w)
    assert st == 0


def test_out_of_pool_page_gives_nan_and_status():
    w = synth.custom(batch=2, next_n=2, heads=64, page_size=16, context_lens=[100, 64],
                     max_model_len=128, seed=7)
    w.block_table[0, 2] = w.pool.num_pages        # tokens 32..47 of request 0
    w.block_table[1, 0] = -5                      # tokens 0..15 of request 1
    _, _, _, st = _full_check(w)
    assert st & sai.STATUS_BAD_PAGE


def test_context_clamped_to_width_and_table():
    w = synth.custom(batch=2, next_n=2, heads=64, page_size=16, context_lens=[5000, 100],
                     max_model_len=300, table_stride=10, seed=9)
    _, _, _, st = _full_check(w)          # oracle clamps to min(W, 160)
    assert st & sai.STATUS_CTX_CLAMPED
    w2 = synth.custom(batch=1, next_n=1, heads=64, page_size=16, context_lens=[-3],
                      max_model_len=64, seed=9)
    _, _, _, st = _full_check(w2)
    assert st & sai.STATUS_CTX_CLAMPED


def test_batch_split_matches_one_launch():
    # One launch over the batch vs two launches over its halves (the
    # reproducer's chunk0 / chunk1 runs, aiter PR 4244).
    w = synth.custom(batch=6, next_n=2, heads=64, page_size=32, context_lens=[500, 3, 260, 0, 129, 77],
                     max_model_len=512, seed=11)
    _, full, dev = run_logits(w)
    halves = []
    for lo, hi in [(0, 3), (3, 6)]:
        part = torch.full((2 * (hi - lo), 512), SENTINEL, device="cuda")
        sai.paged_mqa_logits(dev["q"][lo:hi], dev["kv"], 32, dev["weights"][2 * lo:2 * hi],
                             dev["context_lens"][lo:hi], dev["block_table"][lo:hi], part, 512,
                             num_pages=w.pool.num_pages)
        halves.append(part)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(halves), full)


def test_first_untouched_rows_of_the_32bit_overflow_are_written():
    """aiter PR 4244 "Root cause": with 1024 rows of stride 1<<20 (resp. 600000)
    fp32 logits, a 32-bit byte offset first overflows at row 512 (resp. 895),
    and the unfixed kernel left every later row untouched.  Here every row is
    written and the rows on both sides of the boundary agree with a compact
    launch and with the oracle."""
    for rows, stride, first in [tuple(map(int, r)) for r in golden_rows("output_offset_overflow_rows.txt")]:
        assert rows * 0 + (2**31 + 4 * stride - 1) // (4 * stride) == first
        w = synth.custom(batch=rows // 4, next_n=4, heads=64, page_size=64,
                         context_lens=np.full(rows // 4, 300), max_model_len=300,
                         logits_stride=stride, table_stride=5, seed=13)
        buf = torch.full((rows, stride), SENTINEL, dtype=torch.float32, device="cuda")
        dev = w.to_device()
        sai.paged_mqa_logits(dev["q"], dev["kv"], 64, dev["weights"], dev["context_lens"],
                             dev["block_table"], buf, stride, num_pages=w.pool.num_pages)
        compact = torch.full((rows, 300), SENTINEL, dtype=torch.float32, device="cuda")
        sai.paged_mqa_logits(dev["q"], dev["kv"], 64, dev["weights"], dev["context_lens"],
                             dev["block_table"], compact, 300, num_pages=w.pool.num_pages)
        torch.cuda.synchronize()
        touched = (buf != SENTINEL).any(dim=1)
        assert bool(touched.all()), f"first untouched row {int((~touched).nonzero()[0])}"
        assert torch.equal(buf[:, :300], compact)
        sample = [0, first - 1, first, first + 1, rows - 1]
        ref = oracle_logits(w, rows=sample, W=300)
        assert_logits_close(buf[sample, :300].cpu().numpy(), ref)
        # Columns [300, stride) of the wide launch are -inf (W = stride there).
        assert bool((buf[:, 300:] == -np.inf).all())
        del buf


@pytest.mark.slow
def test_wide_rows_past_2g():
    """The wide workload: logits [1024, 1<<20] fp32 (4 GiB, rows >= 512 past
    2^31 bytes), page ids above 233,016.  Sampled rows vs the oracle, every
    row's -inf / finite split by its context."""
    w = synth.wide()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    logits = torch.full((w.rows, w.logits_stride), SENTINEL, dtype=torch.float32, device="cuda")
    _, view, dev = run_logits(w, status=status, logits=logits)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    n_r = torch.from_numpy(row_ctx(w)).cuda()
    assert torch.equal(torch.isfinite(view).sum(dim=1), n_r)
    assert torch.equal((view == -np.inf).sum(dim=1), w.max_model_len - n_r)
    # Sampled rows against the oracle over every finite column and 256 -inf
    # ones past the longest: the rows around the 2^31-byte boundary, both
    # ends, one row in every block of 32 (a row of each of the 32 row blocks
    # the CTAs' work splits into, roughly), and random ones.
    rng = np.random.default_rng(0)
    sample = set([0, 1, 510, 511, 512, 513, 767, 1022, 1023] + rng.integers(0, 1024, 24).tolist())
    sample |= set((np.arange(32) * 32 + rng.integers(0, 32, 32)).tolist())
    sample = sorted(sample)
    wmax = int(row_ctx(w)[sample].max()) + 256
    ref = oracle_logits(w, rows=sample, W=wmax)
    assert_logits_close(view[sample, :wmax].cpu().numpy(), ref)


@pytest.mark.slow
def test_kv_pages_past_2g():
    """Every page of the kv2g workload starts past byte 2^31 of the pool."""
    w = synth.kv2g()
    assert int(w.block_table.min()) * 16 * 132 >= 2**31
    _, _, _, st = _full_check(w)
    assert st == 0


SWEEP_SAMPLE = [(8, 1, 64, 1, 8192), (8, 4, 128, 16, 512), (16, 2, 64, 64, 512),
                (16, 4, 128, 1, 65536), (64, 1, 128, 16, 8192), (64, 4, 64, 256, 2),
                (256, 2, 128, 16, 8192), (256, 1, 64, 1, 131072), (256, 4, 128, 64, 512)]


@pytest.mark.parametrize("pt", SWEEP_SAMPLE, ids=lambda p: "P%d_n%d_H%d_B%d_ctx%d" % p)
def test_sweep_points(pt):
    w = synth.sweep_point(*pt)
    rows = w.rows
    if rows * w.max_model_len <= 8_000_000:
        _, _, _, st = _full_check(w)
        assert st == 0
        return
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    buf, view, dev = run_logits(w, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_untouched(buf, view, w.max_model_len, 1)
    sample = sorted(set([0, rows - 1, rows // 2]))
    ref = oracle_logits(w, rows=sample)
    assert_logits_close(view[sample, :w.max_model_len].cpu().numpy(), ref)
