"""GPU parity of `sai_gather_selected_kv` (through the C ABI): the int64 row
ids equal the oracle's and the gathered bytes equal the oracle's gather,
with -1 padding, bad table entries, page sizes from 1 to 64, several row
sizes, and rows whose byte offsets pass 2^31 in a 2.3 GB pool."""
import numpy as np
import pytest
import torch

import sparse_attention_indexer_03_gb300 as sai
from oracle import gather

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    sai.build()


def _case(rng, B, next_n, k, P, num_pages, max_ctx):
    ctx = rng.integers(1, max_ctx + 1, B)
    stride = -(-max_ctx // P)
    table = np.stack([rng.permutation(num_pages)[:stride] for _ in range(B)]).astype(np.int32)
    idx = np.full((B * next_n, k + 3), -7, np.int32)
    for r in range(B * next_n):
        n = int(ctx[r // next_n])
        m = min(k, n)
        idx[r, :k] = -1
        idx[r, :m] = np.sort(rng.choice(n, m, replace=False))
    return table, idx


@pytest.mark.parametrize("P,row_bytes", [(1, 576), (16, 576), (64, 16), (8, 656)])
def test_rows_and_ids_match_the_oracle(P, row_bytes):
    rng = np.random.default_rng(P * 1000 + row_bytes)
    B, next_n, k = 5, 2, 40
    num_pages = 4096 // P + 7
    table, idx = _case(rng, B, next_n, k, P, num_pages, max_ctx=300)
    table[1, 2] = -3                                     # a bad entry: status bit, zero rows
    pool = rng.integers(0, 256, num_pages * P * row_bytes, dtype=np.uint8)
    d_idx = torch.from_numpy(idx).cuda()
    d_tab = torch.from_numpy(table).cuda()
    d_pool = torch.from_numpy(pool).cuda()
    rows = idx.shape[0]
    ids = torch.full((rows, k), 123, dtype=torch.int64, device="cuda")
    out = torch.full((rows, k, row_bytes), 77, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sai.gather_selected_kv(d_idx[:, :k], next_n, d_tab, P, d_pool, row_bytes, row_ids=ids, out=out,
                           status=status)
    torch.cuda.synchronize()
    ref_ids = gather.kv_row_ids(idx[:, :k], table, next_n, P, num_pages)
    assert (ids.cpu().numpy() == ref_ids).all()
    ref_rows = gather.gather_kv_rows(pool, ref_ids, row_bytes)
    assert (out.cpu().numpy() == ref_rows).all()
    bad_used = any(((idx[r, :k] >= 0) & (idx[r, :k] // P == 2)).any() for r in (2, 3))
    assert bool(int(status.item()) & sai.STATUS_BAD_PAGE) == bad_used


def test_ids_only_and_rows_only():
    rng = np.random.default_rng(5)
    P, row_bytes, num_pages = 16, 64, 100
    table, idx = _case(rng, 3, 1, 20, P, num_pages, max_ctx=200)
    pool = rng.integers(0, 256, num_pages * P * row_bytes, dtype=np.uint8)
    d_idx, d_tab, d_pool = (torch.from_numpy(a).cuda() for a in (idx[:, :20], table, pool))
    ids = torch.empty((3, 20), dtype=torch.int64, device="cuda")
    sai.gather_selected_kv(d_idx, 1, d_tab, P, d_pool, row_bytes, row_ids=ids)
    out = torch.empty((3, 20, row_bytes), dtype=torch.uint8, device="cuda")
    sai.gather_selected_kv(d_idx, 1, d_tab, P, d_pool, row_bytes, out=out)
    torch.cuda.synchronize()
    ref_ids = gather.kv_row_ids(idx[:, :20], table, 1, P, num_pages)
    assert (ids.cpu().numpy() == ref_ids).all()
    assert (out.cpu().numpy() == gather.gather_kv_rows(pool, ref_ids, row_bytes)).all()


@pytest.mark.slow
def test_rows_past_2g_bytes():
    # A pool of 4,200,000 MLA rows (576 B, 2.42 GB) in pages of 16: rows past
    # 2^31 / 576 = 3,728,270 sit past 2^31 bytes.  Each row's bytes spell its
    # row id, so the expected bytes follow from the oracle's row ids.
    P, row_bytes, num_pages = 16, 576, 262_500
    n_rows = num_pages * P
    pool = torch.arange(n_rows, dtype=torch.int64, device="cuda")[:, None].expand(n_rows, row_bytes // 8)
    pool = pool.contiguous().view(torch.uint8).reshape(-1)
    rng = np.random.default_rng(3)
    B, k = 8, 512
    hi_pages = np.arange(233_000, num_pages)
    table = np.stack([rng.permutation(hi_pages)[:600] for _ in range(B)]).astype(np.int32)
    table[:, :4] = rng.integers(0, 1000, (B, 4))           # some low pages too
    idx = np.stack([np.sort(rng.choice(600 * P, k, replace=False)) for _ in range(B)]).astype(np.int32)
    ids = torch.empty((B, k), dtype=torch.int64, device="cuda")
    out = torch.empty((B, k, row_bytes), dtype=torch.uint8, device="cuda")
    sai.gather_selected_kv(torch.from_numpy(idx).cuda(), 1, torch.from_numpy(table).cuda(), P, pool, row_bytes,
                           row_ids=ids, out=out)
    torch.cuda.synchronize()
    ref_ids = gather.kv_row_ids(idx, table, 1, P, num_pages)
    assert (ref_ids > 3_728_270).sum() > 1000
    assert (ids.cpu().numpy() == ref_ids).all()
    spelled = out.cpu().numpy().view("<i8").reshape(B, k, row_bytes // 8)
    assert (spelled == ref_ids[:, :, None]).all()
