"""Plain definition of the consumer gather: the KV rows of the tokens that
the top-k selected, addressed through the block table with int64 row ids.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources.  The selected token positions are the top-k indices of each query
row (`top_k_per_row_decode`, aiter PR 4244, opening paragraph: the indices
fill the persistent sparse-KV index buffer that the sparse attention reads).
The addressing rule is ATOM PR 2533, "[MLA] Address Triton decode KV rows
with int64 ids", sections "Problem" and "Fix": a token-level KV row id
(page id * page size + position) is multiplied by the row stride (576 for
MLA) to form a byte offset, and that product must be taken in 64 bits; an
int32 product wraps for row ids >= 2^31 / 576 = 3,728,270, i.e. past block
233,016 of 16 tokens.

Readings taken where the pages are silent (each is listed in the design
notes):
  * the KV pool is token-major: row id j occupies bytes
    [j * row_bytes, (j + 1) * row_bytes);
  * row r = b * next_n + j of the indices belongs to request b; index t
    (a token position) lives in page block_table[b, t // P] at position t % P;
  * a -1 index (top-k padding) gives row id -1 and an all-zero output row;
    so does an index whose table entry lies past the table row or whose page
    id lies outside [0, num_pages) (the library also raises a status bit).
"""
from __future__ import annotations

import numpy as np


def kv_row_ids(indices: np.ndarray, block_table: np.ndarray, next_n: int, page_size: int,
               num_pages: int) -> np.ndarray:
    """int64 row ids `[rows, k]` of the selected tokens (-1 where none)."""
    indices = np.asarray(indices, dtype=np.int64)
    rows, k = indices.shape
    table = np.asarray(block_table, dtype=np.int64)
    out = np.full((rows, k), -1, dtype=np.int64)
    for r in range(rows):
        b = r // next_n
        for i in range(k):
            t = int(indices[r, i])
            if t < 0 or t // page_size >= table.shape[1]:
                continue
            page = int(table[b, t // page_size])
            if page < 0 or page >= num_pages:
                continue
            out[r, i] = page * page_size + t % page_size
    return out


def gather_kv_rows(pool: np.ndarray, row_ids: np.ndarray, row_bytes: int) -> np.ndarray:
    """Bytes `[rows, k, row_bytes]`: pool row j for each row id j >= 0, zeros
    for -1.  `pool` is the flat byte array of the token-major KV pool."""
    pool = np.asarray(pool, dtype=np.uint8).reshape(-1)
    rows, k = row_ids.shape
    out = np.zeros((rows, k, row_bytes), dtype=np.uint8)
    for r in range(rows):
        for i in range(k):
            j = int(row_ids[r, i])
            if j >= 0:
                off = j * row_bytes                      # Python integer: no wrap
                out[r, i] = pool[off:off + row_bytes]
    return out
