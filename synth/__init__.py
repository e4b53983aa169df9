"""Seeded synthetic inputs for the FP8 paged MQA indexer (logits, then top-k).

This module is shared by the CPU oracle's tests, the GPU parity tests, the
benchmark and the smoke run.  It draws random numbers, casts them to the
stored formats (OCP e4m3fn bytes, fp32) and lays them out in the paged
K-cache format.  It holds none of the scoring arithmetic: nothing here
dequantises, multiplies or selects.

Value distributions (the same for every workload):
  * q and K values: N(0, 1) draws cast to e4m3fn with round-to-nearest-even
    (torch's float8_e4m3fn conversion);
  * per-token K scale: U(0.5, 2) fp32;
  * head weights: N(0, 1) / sqrt(H) fp32.

Paged K-cache layout ("page-split", the reading adopted for the
`[num_blocks, block_size, 1, D + 4]` byte tensor of the reproducer in aiter
PR 4244, "fix silent tail-row drop in deepgemm_fp8_paged_mqa_logits at large
output stride", and for the separate per-page value and scale loads of aiter
PR 6626, "paged MQA logits: 8-token pages ...", section 1): page p occupies
`P * (D + 4)` bytes starting at byte `p * P * (D + 4)`; its first `P * D`
bytes are the P tokens' FP8 values, token-major; the next `4 * P` bytes are
the P tokens' fp32 scales, little-endian.  The "interleaved" variant stores
each token as D value bytes followed by its 4 scale bytes.

Only pages that some request reads are drawn; every other page of the pool
is zero.  A pool is therefore carried sparsely as (sorted page ids, page
bytes) and materialised on the device with one scatter.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

HEAD_DIM = 128
SCALE_BYTES = 4

LAYOUT_SPLIT = "split"
LAYOUT_INTERLEAVED = "interleaved"


def page_bytes(page_size: int, head_dim: int = HEAD_DIM) -> int:
    return page_size * (head_dim + SCALE_BYTES)


def to_e4m3_bytes(x: np.ndarray) -> np.ndarray:
    """Cast float32 values to OCP e4m3fn bytes (round to nearest even)."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


@dataclasses.dataclass
class KVPool:
    """A paged FP8 K-cache held sparsely: unlisted pages are all-zero."""

    num_pages: int
    page_size: int
    layout: str
    ids: np.ndarray      # int64 [n], sorted, unique page ids that hold data
    data: np.ndarray     # uint8 [n, page_bytes]

    @property
    def page_bytes(self) -> int:
        return page_bytes(self.page_size)

    @property
    def nbytes(self) -> int:
        return self.num_pages * self.page_bytes

    def dense(self) -> np.ndarray:
        """The whole pool as uint8 [num_pages, page_bytes] (small pools only)."""
        out = np.zeros((self.num_pages, self.page_bytes), np.uint8)
        out[self.ids] = self.data
        return out

    def to_device(self, device="cuda"):
        """One device buffer of num_pages * page_bytes bytes, data scattered in."""
        import torch

        buf = torch.zeros(self.num_pages * self.page_bytes, dtype=torch.uint8, device=device)
        if len(self.ids):
            view = buf.view(self.num_pages, self.page_bytes)
            ids = torch.from_numpy(self.ids).to(device)
            view.index_copy_(0, ids, torch.from_numpy(self.data).to(device))
        return buf


def pack_pages(values: np.ndarray, scales: np.ndarray, layout: str) -> np.ndarray:
    """Lay out pages from per-token values uint8 [n, P, D] and scales f32 [n, P]."""
    n, p, d = values.shape
    sc = np.ascontiguousarray(scales, dtype="<f4").view(np.uint8).reshape(n, p, SCALE_BYTES)
    if layout == LAYOUT_SPLIT:
        return np.concatenate([values.reshape(n, p * d), sc.reshape(n, p * SCALE_BYTES)], axis=1)
    if layout == LAYOUT_INTERLEAVED:
        return np.concatenate([values, sc], axis=2).reshape(n, p * (d + SCALE_BYTES))
    raise ValueError(f"unknown layout {layout!r}")


@dataclasses.dataclass
class Workload:
    """One batch of indexer inputs (host arrays) plus its shape parameters."""

    name: str
    batch: int
    next_n: int
    heads: int
    page_size: int
    max_model_len: int          # W: logical logits width
    logits_stride: int          # elements between logits rows (>= W)
    topk: int
    q: np.ndarray               # uint8 [B, next_n, H, D]   e4m3fn bytes
    weights: np.ndarray         # float32 [B * next_n, H]
    context_lens: np.ndarray    # int32 [B]
    block_table: np.ndarray     # int32 [B, block_table_stride]
    pool: KVPool
    seed: int
    head_dim: int = HEAD_DIM

    @property
    def rows(self) -> int:
        return self.batch * self.next_n

    @property
    def layout(self) -> str:
        return self.pool.layout

    def to_device(self, device="cuda") -> dict:
        """The inputs as device tensors: q, kv (flat pool bytes), weights,
        context_lens, block_table."""
        import torch

        return dict(q=torch.from_numpy(self.q).to(device),
                    kv=self.pool.to_device(device),
                    weights=torch.from_numpy(self.weights).to(device),
                    context_lens=torch.from_numpy(self.context_lens).to(device),
                    block_table=torch.from_numpy(self.block_table).to(device))


def _draw_pool(rng: np.random.Generator, num_pages: int, page_size: int,
               used_ids: np.ndarray, layout: str) -> KVPool:
    ids = np.unique(np.asarray(used_ids, dtype=np.int64))
    ids = ids[(ids >= 0) & (ids < num_pages)]
    n = len(ids)
    vals = to_e4m3_bytes(rng.standard_normal((n, page_size, HEAD_DIM), dtype=np.float32))
    scales = rng.uniform(0.5, 2.0, size=(n, page_size)).astype(np.float32)
    return KVPool(num_pages, page_size, layout, ids, pack_pages(vals, scales, layout))


def _used_page_ids(block_table: np.ndarray, context_lens: np.ndarray, page_size: int) -> np.ndarray:
    used = []
    for b in range(block_table.shape[0]):
        npg = -(-max(int(context_lens[b]), 0) // page_size)
        used.append(block_table[b, :min(npg, block_table.shape[1])])
    return np.concatenate(used) if used else np.zeros(0, np.int64)


def make_workload(name: str, *, batch: int, next_n: int, heads: int, page_size: int,
                  max_model_len: int, logits_stride: Optional[int], topk: int,
                  context_lens: np.ndarray, block_table: np.ndarray, num_pages: int,
                  rng: np.random.Generator, seed: int,
                  layout: str = LAYOUT_SPLIT) -> Workload:
    """Draw q, weights and the referenced pages for given shapes, lengths and table."""
    q = to_e4m3_bytes(rng.standard_normal((batch, next_n, heads, HEAD_DIM), dtype=np.float32))
    w = (rng.standard_normal((batch * next_n, heads), dtype=np.float32)
         / np.float32(math.sqrt(heads))).astype(np.float32)
    context_lens = np.asarray(context_lens, dtype=np.int32)
    block_table = np.ascontiguousarray(block_table, dtype=np.int32)
    pool = _draw_pool(rng, num_pages, page_size,
                      _used_page_ids(block_table, context_lens, page_size), layout)
    return Workload(name, batch, next_n, heads, page_size, max_model_len,
                    logits_stride if logits_stride is not None else max_model_len,
                    topk, q, w, context_lens, block_table, pool, seed)


# ---------------------------------------------------------------------------
# The named workloads.  Shapes and distributions follow the indexer decode
# workloads described for the op (B, next_n, H, page size, context mix,
# logits width, k); the seeds are fixed here.
# ---------------------------------------------------------------------------

SEEDS = {"tiny": 0, "decode": 1, "mtp": 2, "wide": 3, "kv2g": 4}


def tiny(layout: str = LAYOUT_SPLIT) -> Workload:
    """B=2, next_n=1, H=64, P=16, ctx {300, 17}, W=512, k=64; 20-page pool.

    Each request's table row is an independent random permutation of all 20
    pool pages (ctx 300 needs 19 pages), so the two requests share pages.
    """
    rng = np.random.Generator(np.random.PCG64(SEEDS["tiny"]))
    table = np.stack([rng.permutation(20) for _ in range(2)])
    return make_workload("tiny", batch=2, next_n=1, heads=64, page_size=16,
                         max_model_len=512, logits_stride=512, topk=64,
                         context_lens=np.array([300, 17]), block_table=table,
                         num_pages=20, rng=rng, seed=SEEDS["tiny"], layout=layout)


def decode(layout: str = LAYOUT_SPLIT) -> Workload:
    """B=64, next_n=1, H=64, P=64, ctx U[1024, 8192], W=8192, k=2048.

    Pool of 8192 pages; one random permutation of it, reshaped [64, 128], is
    the block table.
    """
    rng = np.random.Generator(np.random.PCG64(SEEDS["decode"]))
    ctx = rng.integers(1024, 8192, size=64, endpoint=True)
    table = rng.permutation(8192).reshape(64, 128)
    return make_workload("decode", batch=64, next_n=1, heads=64, page_size=64,
                         max_model_len=8192, logits_stride=8192, topk=2048,
                         context_lens=ctx, block_table=table, num_pages=8192,
                         rng=rng, seed=SEEDS["decode"], layout=layout)


def mtp(layout: str = LAYOUT_SPLIT) -> Workload:
    """B=256, next_n=4, H=128, P=8, ctx log-uniform in [2, 32768] with one empty
    context, W=32768, k=2048.

    Pool of 2^20 pages of 8 tokens; one random permutation of it, reshaped
    [256, 4096], is the block table.
    """
    rng = np.random.Generator(np.random.PCG64(SEEDS["mtp"]))
    ctx = np.rint(np.exp(rng.uniform(math.log(2), math.log(32768), size=256))).astype(np.int64)
    ctx[rng.integers(256)] = 0
    table = rng.permutation(1 << 20).reshape(256, 4096)
    return make_workload("mtp", batch=256, next_n=4, heads=128, page_size=8,
                         max_model_len=32768, logits_stride=32768, topk=2048,
                         context_lens=ctx, block_table=table, num_pages=1 << 20,
                         rng=rng, seed=SEEDS["mtp"], layout=layout)


WIDE_FIRST_PAGE = 233_017   # first block of 16 above the int32 row limit of 576-byte rows


def wide(layout: str = LAYOUT_SPLIT, batch: int = 256) -> Workload:
    """B=256, next_n=4, H=64, P=16, ctx U[4096, 16384], W = stride = 2^20, k=2048.

    Pool of 4,000,000 tokens (250,000 pages of 16).  Every request's table row
    is its own random permutation of the pool's top pages [233017, 250000),
    cut to 1024 entries, so rows >= 512 of the logits lie past 2^31 bytes.
    `batch` < 256 gives the same per-request shape with fewer requests (named
    wide_b<batch>; a case small enough for a profiler capture).
    """
    rng = np.random.Generator(np.random.PCG64(SEEDS["wide"]))
    ctx = rng.integers(4096, 16384, size=batch, endpoint=True)
    top = np.arange(WIDE_FIRST_PAGE, 250_000)
    table = np.stack([rng.permutation(top)[:1024] for _ in range(batch)])
    return make_workload("wide" if batch == 256 else f"wide_b{batch}", batch=batch, next_n=4, heads=64,
                         page_size=16,
                         max_model_len=1 << 20, logits_stride=1 << 20, topk=2048,
                         context_lens=ctx, block_table=table, num_pages=250_000,
                         rng=rng, seed=SEEDS["wide"], layout=layout)


KV2G_NUM_PAGES = 1_062_500          # 17,000,000 tokens of 16 per page: 2.24 GB
KV2G_FIRST_PAGE = 1_016_801         # first page of 16 x 132 B wholly past 2^31 bytes


def kv2g(layout: str = LAYOUT_SPLIT) -> Workload:
    """B=4, next_n=2, H=64, P=16, ctx 8192; every page id lies past byte 2^31."""
    rng = np.random.Generator(np.random.PCG64(SEEDS["kv2g"]))
    ids = np.arange(KV2G_FIRST_PAGE, KV2G_NUM_PAGES)
    table = np.stack([rng.choice(ids, size=512, replace=False) for _ in range(4)])
    return make_workload("kv2g", batch=4, next_n=2, heads=64, page_size=16,
                         max_model_len=8192, logits_stride=8192, topk=2048,
                         context_lens=np.full(4, 8192), block_table=table,
                         num_pages=KV2G_NUM_PAGES, rng=rng, seed=SEEDS["kv2g"], layout=layout)


SWEEP_PAGES = (8, 16, 64, 256)
SWEEP_NEXT_N = (1, 2, 4)
SWEEP_HEADS = (64, 128)
SWEEP_BATCH = (1, 16, 64, 256, 512)
SWEEP_CTX = (2, 512, 8192, 65536, 131072)


def sweep_points():
    """All 600 throughput-sweep points as (index, P, next_n, H, B, ctx)."""
    i = 0
    for p in SWEEP_PAGES:
        for n in SWEEP_NEXT_N:
            for h in SWEEP_HEADS:
                for b in SWEEP_BATCH:
                    for c in SWEEP_CTX:
                        yield i, p, n, h, b, c
                        i += 1


def sweep_point(page_size: int, next_n: int, heads: int, batch: int, ctx: int,
                layout: str = LAYOUT_SPLIT) -> Workload:
    """One sweep point: uniform context, W = ctx, row stride ceil(ctx/4)*4,
    pool = exactly the pages needed, randomly permuted into the table."""
    index = [i for i, p, n, h, b, c in sweep_points()
             if (p, n, h, b, c) == (page_size, next_n, heads, batch, ctx)]
    seed = 1000 + (index[0] if index else 999)
    rng = np.random.Generator(np.random.PCG64(seed))
    npg = -(-ctx // page_size)
    table = rng.permutation(batch * npg).reshape(batch, npg)
    return make_workload(f"sweep_P{page_size}_n{next_n}_H{heads}_B{batch}_ctx{ctx}",
                         batch=batch, next_n=next_n, heads=heads, page_size=page_size,
                         max_model_len=ctx, logits_stride=-(-ctx // 4) * 4, topk=2048,
                         context_lens=np.full(batch, ctx), block_table=table,
                         num_pages=batch * npg, rng=rng, seed=seed, layout=layout)


def custom(*, batch: int, next_n: int, heads: int, page_size: int, context_lens,
           max_model_len: int, logits_stride: Optional[int] = None, topk: int = 64,
           table_stride: Optional[int] = None, num_pages: Optional[int] = None,
           seed: int = 7, layout: str = LAYOUT_SPLIT, name: str = "custom") -> Workload:
    """Small ad-hoc workload: a random permutation of a pool just large enough."""
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx = np.asarray(context_lens, dtype=np.int64)
    need = int(max(1, -(-max(int(ctx.max(initial=0)), 1) // page_size)))
    stride = table_stride if table_stride is not None else need
    npages = num_pages if num_pages is not None else batch * stride
    table = np.stack([rng.permutation(npages)[:stride] for _ in range(batch)])
    return make_workload(name, batch=batch, next_n=next_n, heads=heads, page_size=page_size,
                         max_model_len=max_model_len, logits_stride=logits_stride, topk=topk,
                         context_lens=ctx, block_table=table, num_pages=npages, rng=rng,
                         seed=seed, layout=layout)


NAMED = {"tiny": tiny, "decode": decode, "mtp": mtp, "wide": wide, "kv2g": kv2g}


# ---------------------------------------------------------------- K-cache write
def kcache_batch(num_tokens: int, page_size: int, num_pages: int, seed: int = 5):
    """New K rows for the K-cache write: bf16 bits [T, 128] of N(0, 1) draws
    times a per-row factor exp(U(-2, 2)) (rows of different magnitudes), and
    T distinct slots drawn from the pool's num_pages * page_size (int64)."""
    import torch

    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((num_tokens, HEAD_DIM)).astype(np.float32)
    x *= np.exp(rng.uniform(-2, 2, (num_tokens, 1))).astype(np.float32)
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    slots = rng.choice(num_pages * page_size, size=num_tokens, replace=False).astype(np.int64)
    return bits, slots


# ---------------------------------------------------------------- consumer gather
def gather_batch(batch: int = 64, next_n: int = 1, k: int = 2048, page_size: int = 64,
                 num_pages: int = 8192, max_ctx: int = 8192, seed: int = 6):
    """Selected token positions as the top-k leaves them, for the decode
    shapes: context lengths U[1024, max_ctx], a block table that is one
    permutation of the pool reshaped [batch, num_pages / batch], and for each
    row a sorted random subset of min(k, ctx_r) positions, padded with -1.
    Returns (indices int32 [batch * next_n, k], block_table int32, context_lens)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx = rng.integers(1024, max_ctx, size=batch, endpoint=True)
    table = rng.permutation(num_pages).reshape(batch, num_pages // batch).astype(np.int32)
    idx = np.full((batch * next_n, k), -1, np.int32)
    for r in range(batch * next_n):
        n = max(0, int(ctx[r // next_n]) - next_n + r % next_n + 1)
        m = min(k, n)
        idx[r, :m] = np.sort(rng.choice(n, m, replace=False))
    return idx, table, ctx


# ---------------------------------------------------------------- sweep on the device
@dataclasses.dataclass
class DeviceWorkload:
    """A sweep point drawn directly on the device (pools of several GB are
    too slow to draw on the host).  Same value distributions as the host
    workloads, from torch's device generator: q and K values N(0, 1) cast to
    e4m3fn, scales U(0.5, 2), weights N(0, 1) / sqrt(H).  Uniform contexts,
    W = ctx, row stride ceil(ctx / 4) * 4, pool = exactly the pages the batch
    needs, randomly permuted into the block table.  For timing only: the
    parity tests use the host workloads, which the oracle can read."""

    name: str
    batch: int
    next_n: int
    heads: int
    page_size: int
    max_model_len: int
    logits_stride: int
    topk: int
    context_lens: np.ndarray    # host copy, int32 [B]
    block_table: object         # device int32 [B, npg]
    num_pages: int
    seed: int
    dev: dict                   # q, kv, weights, context_lens, block_table on the device
    head_dim: int = HEAD_DIM
    layout: str = LAYOUT_SPLIT

    @property
    def rows(self) -> int:
        return self.batch * self.next_n


def sweep_point_device(page_size: int, next_n: int, heads: int, batch: int, ctx: int, device,
                       seed: int = 0) -> DeviceWorkload:
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    npg = -(-ctx // page_size)
    num_pages = batch * npg
    P = page_size
    chunk_pages = max(1, (1 << 26) // (P * HEAD_DIM))      # 64 M values (256 MB of fp32) per draw
    kv = torch.empty(num_pages * P * (HEAD_DIM + SCALE_BYTES), dtype=torch.uint8, device=device)
    pages = kv.view(num_pages, P * (HEAD_DIM + SCALE_BYTES))
    for p0 in range(0, num_pages, chunk_pages):
        p1 = min(num_pages, p0 + chunk_pages)
        vals = torch.randn((p1 - p0, P * HEAD_DIM), generator=g, device=device)
        pages[p0:p1, :P * HEAD_DIM] = vals.to(torch.float8_e4m3fn).view(torch.uint8)
        sc = torch.rand((p1 - p0, P), generator=g, device=device) * 1.5 + 0.5
        pages[p0:p1, P * HEAD_DIM:] = sc.contiguous().view(torch.uint8)
        del vals, sc
    q = torch.randn((batch, next_n, heads, HEAD_DIM), generator=g, device=device)
    q = q.to(torch.float8_e4m3fn).view(torch.uint8)
    w = torch.randn((batch * next_n, heads), generator=g, device=device) / math.sqrt(heads)
    table = torch.randperm(num_pages, generator=g, device=device).to(torch.int32).view(batch, npg)
    ctx_h = np.full(batch, ctx, np.int32)
    dev = dict(q=q, kv=kv, weights=w.contiguous(), context_lens=torch.from_numpy(ctx_h).to(device),
               block_table=table.contiguous())
    return DeviceWorkload(f"sweep_P{page_size}_n{next_n}_H{heads}_B{batch}_ctx{ctx}", batch, next_n, heads,
                          page_size, ctx, -(-ctx // 4) * 4, 2048, ctx_h, table, num_pages, int(seed), dev)
