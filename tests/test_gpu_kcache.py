"""GPU parity of `sai_indexer_k_quant_insert` (through the C ABI): the cache
bytes after the write equal the oracle's byte for byte (codes, scales, and
every untouched byte), in both cache layouts, with padding and out-of-range
slots, and with slots whose byte offsets pass 2^31."""
import numpy as np
import pytest
import torch

import sparse_attention_indexer_03_gb300 as sai
from oracle import kcache

pytestmark = pytest.mark.gpu
D = 128


@pytest.fixture(scope="module", autouse=True)
def _lib():
    sai.build()


def _k_rows(rng, T):
    """bf16 rows with a spread of magnitudes, some all-zero, some with one huge value."""
    x = rng.standard_normal((T, D)).astype(np.float32) * np.exp(rng.uniform(-8, 8, (T, 1))).astype(np.float32)
    x[::17] = 0.0
    x[5::23, 3] = 3.0e4
    t = torch.from_numpy(x).to(torch.bfloat16)
    return t, t.view(torch.int16).numpy().view(np.uint16)


def _run(k, slots, cache, P, layout, status=None):
    kd, sd, cd = k.cuda(), torch.from_numpy(slots).cuda(), torch.from_numpy(cache).cuda()
    sai.indexer_k_quant_insert(kd, sd, cd, P, kv_layout=layout, status=status)
    torch.cuda.synchronize()
    return cd.cpu().numpy()


@pytest.mark.parametrize("layout", ["split", "interleaved"])
@pytest.mark.parametrize("P", [8, 64, 256])
def test_cache_bytes_match_the_oracle(P, layout):
    rng = np.random.default_rng(P + (layout == "split"))
    num_pages = 40
    T = 1000 if P >= 64 else 300
    slots = rng.permutation(num_pages * P)[:T].astype(np.int64)
    slots[::11] = -1                                         # padding tokens
    k, bits = _k_rows(rng, T)
    cache = rng.integers(0, 256, num_pages * P * (D + 4), dtype=np.uint8)   # old contents survive
    got = _run(k, slots, cache, P, layout)
    codes, scales = kcache.quantize_k_rows(bits)
    ref = kcache.insert_k_rows(cache, slots, codes, scales, num_pages, P, layout)
    bad = np.flatnonzero(got != ref)
    assert bad.size == 0, f"{bad.size} bytes differ, first at {bad[:5]}"


def test_out_of_range_slot_raises_status_and_writes_nothing():
    rng = np.random.default_rng(9)
    P, num_pages = 16, 4
    slots = np.array([3, num_pages * P, 70, -2], np.int64)
    k, bits = _k_rows(rng, 4)
    cache = np.zeros(num_pages * P * (D + 4), np.uint8)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _run(k, slots, cache, P, "split", status)
    assert int(status.item()) & sai.STATUS_BAD_PAGE
    codes, scales = kcache.quantize_k_rows(bits)
    ref = kcache.insert_k_rows(cache, slots, codes, scales, num_pages, P, "split")
    assert (got == ref).all()


def test_empty_batch_is_a_no_op():
    cache = torch.zeros(16 * 132, dtype=torch.uint8, device="cuda")
    sai.indexer_k_quant_insert(torch.zeros((0, D), dtype=torch.bfloat16, device="cuda"),
                               torch.zeros(0, dtype=torch.int64, device="cuda"), cache, 16)
    torch.cuda.synchronize()
    assert not bool(cache.any())


@pytest.mark.slow
def test_slots_past_2g_bytes():
    # A 2.4 GB pool of 16-token pages: token bytes past 2^31 start at page
    # 2^31 / 2112 = 1,016,800.  Tokens go to the pool's last pages and to a
    # few low pages; the written bytes are read back through int64 offsets.
    P, num_pages = 16, 1_150_000
    rng = np.random.default_rng(11)
    T = 4096
    hi = rng.choice(np.arange(1_016_000 * P, num_pages * P), T - 64, replace=False)
    lo = rng.choice(np.arange(0, 1000 * P), 64, replace=False)
    slots = np.concatenate([hi, lo]).astype(np.int64)
    k, bits = _k_rows(rng, T)
    cache = torch.zeros(num_pages * P * (D + 4), dtype=torch.uint8, device="cuda")
    sai.indexer_k_quant_insert(k.cuda(), torch.from_numpy(slots).cuda(), cache, P)
    torch.cuda.synchronize()
    codes, scales = kcache.quantize_k_rows(bits)
    s = torch.from_numpy(slots).cuda()
    page, pos = s // P, s % P
    base = page * (P * (D + 4))
    vidx = (base + pos * D)[:, None] + torch.arange(D, device="cuda")[None, :]
    sidx = (base + P * D + pos * 4)[:, None] + torch.arange(4, device="cuda")[None, :]
    assert (cache[vidx].cpu().numpy() == codes).all()
    got_sc = cache[sidx].cpu().numpy().copy().view("<f4").reshape(-1)
    assert (got_sc == scales).all()
    assert int(cache.sum(dtype=torch.int64).item()) == int(codes.astype(np.int64).sum() +
                                                           scales.view(np.uint8).astype(np.int64).sum())
