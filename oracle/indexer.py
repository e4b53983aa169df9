"""Plain fp64 definition of FP8 paged MQA logits and per-row top-k.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources.  The op, its arguments and the K-cache byte tensor are those of
`deepgemm_fp8_paged_mqa_logits` as called by the reproducer in aiter PR 4244,
"fix silent tail-row drop in deepgemm_fp8_paged_mqa_logits at large output
stride" (section "small reproducer": q `[B, next_n, H, D]` FP8, K-cache
`[num_blocks, block_size, 1, D + 4]` bytes whose last four bytes per token
are one fp32 scale, weights `[B * next_n, H]` fp32, context_lens `[B]`,
block table `[B, max_blocks]` int32, logits `[B * next_n, max_model_len]`
fp32).  The scoring rule is the DeepSeek-style indexer definition that the op
implements:

    logits[r, t] = sum_h w[r, h] * ReLU(q[r, h] . k[t]) * scale[t]

for t inside row r's causal context and -inf beyond it, where MTP row j of
a request with context length ctx sees ctx - next_n + j + 1 tokens.  The
per-row top-k that consumes the logits is `top_k_per_row_decode` (aiter PR
4244, opening paragraph: one logits launch, then top-k into the persistent
sparse-KV index buffer).

Readings taken where the pages are silent (each is listed in the design
notes):
  * page-split K-cache layout: a page's P * D value bytes come first, then
    its P fp32 scales (the interleaved per-token reading is available via
    `layout="interleaved"`);
  * FP8 is OCP e4m3fn;
  * a row's context is clamped to [0, min(W, table_stride * P)];
  * a page id outside [0, num_pages) yields NaN logits for that page's tokens;
  * top-k ties at the k-th value go to the lower index; short rows pad with -1.
"""
from __future__ import annotations

import numpy as np

D = 128
SCALE_BYTES = 4
E4M3FN_NAN_CODES = (0x7F, 0xFF)


# ---------------------------------------------------------------------------
# FP8 E4M3 ("fn") decoding, written out from the OCP 8-bit floating point
# definition: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
# exponent field 0 encodes subnormals m/8 * 2^-6; S.1111.111 is NaN; there is
# no infinity, so the largest finite magnitude is 1.75 * 2^8 = 448.
# ---------------------------------------------------------------------------
def e4m3fn_value(code: int) -> float:
    """The exact real value of one e4m3fn byte (NaN for the two NaN codes)."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    exp_field = (code >> 3) & 0xF
    mant = code & 0x7
    if exp_field == 0xF and mant == 0x7:
        return float("nan")
    if exp_field == 0:
        return sign * (mant / 8.0) * 2.0 ** (1 - 7)
    return sign * (1.0 + mant / 8.0) * 2.0 ** (exp_field - 7)


def e4m3fn_table() -> np.ndarray:
    """fp64 value of each of the 256 codes."""
    return np.array([e4m3fn_value(c) for c in range(256)], dtype=np.float64)


_TABLE = e4m3fn_table()


# ---------------------------------------------------------------------------
# Causal row context (MTP).
# ---------------------------------------------------------------------------
def row_context_lengths(context_lens, next_n: int, max_model_len: int,
                        table_stride: int, page_size: int) -> np.ndarray:
    """Tokens seen by each row r = b * next_n + j: ctx_b - next_n + j + 1,
    clamped to [0, min(W, table_stride * P)]."""
    cap = min(int(max_model_len), int(table_stride) * int(page_size))
    out = np.zeros(len(context_lens) * next_n, dtype=np.int64)
    for b, ctx in enumerate(np.asarray(context_lens, dtype=np.int64)):
        for j in range(next_n):
            out[b * next_n + j] = min(max(int(ctx) - next_n + j + 1, 0), cap)
    return out


# ---------------------------------------------------------------------------
# Reading K through the block table.
# ---------------------------------------------------------------------------
def _page_rows(pool_ids: np.ndarray, pool_data: np.ndarray, num_pages: int,
               page_ids: np.ndarray):
    """Bytes of each requested page (zero for pages the pool does not list) and
    a validity mask (False for ids outside [0, num_pages))."""
    page_ids = np.asarray(page_ids, dtype=np.int64)
    valid = (page_ids >= 0) & (page_ids < num_pages)
    pos = np.searchsorted(pool_ids, page_ids)
    pos_c = np.minimum(pos, max(len(pool_ids) - 1, 0))
    listed = valid & (len(pool_ids) > 0)
    if len(pool_ids):
        listed &= pool_ids[pos_c] == page_ids
    rows = np.zeros((len(page_ids), pool_data.shape[1]), np.uint8)
    if listed.any():
        rows[listed] = pool_data[pos_c[listed]]
    return rows, valid


def gather_request_tokens(pool_ids, pool_data, num_pages: int, page_size: int,
                          table_row: np.ndarray, n_tokens: int, layout: str = "split"):
    """K of one request's first n_tokens tokens: (values fp64 [n, D],
    scales fp64 [n], token_valid bool [n]).

    Token t lives in page table_row[t // P] at slot t % P.  In the page-split
    layout the slot's D value bytes start at byte slot * D of the page and its
    scale at byte P * D + 4 * slot; in the interleaved layout the slot occupies
    bytes [slot * (D + 4), (slot + 1) * (D + 4)), scale last.
    """
    t = np.arange(n_tokens, dtype=np.int64)
    page_of_t = np.asarray(table_row, dtype=np.int64)[t // page_size]
    slot = t % page_size
    pages, valid = _page_rows(pool_ids, pool_data, num_pages, page_of_t)
    if layout == "split":
        val_off = slot[:, None] * D + np.arange(D)[None, :]
        sc_off = page_size * D + SCALE_BYTES * slot[:, None] + np.arange(SCALE_BYTES)[None, :]
    elif layout == "interleaved":
        val_off = slot[:, None] * (D + SCALE_BYTES) + np.arange(D)[None, :]
        sc_off = slot[:, None] * (D + SCALE_BYTES) + D + np.arange(SCALE_BYTES)[None, :]
    else:
        raise ValueError(layout)
    rows = np.arange(n_tokens)[:, None]
    values = _TABLE[pages[rows, val_off]]
    scale_bytes = np.ascontiguousarray(pages[rows, sc_off])
    scales = scale_bytes.view("<f4").reshape(n_tokens).astype(np.float64)
    return values, scales, valid


# ---------------------------------------------------------------------------
# Logits.
# ---------------------------------------------------------------------------
def paged_mqa_logits(q, pool_ids, pool_data, num_pages: int, page_size: int,
                     weights, context_lens, block_table, next_n: int,
                     max_model_len: int, layout: str = "split", rows=None) -> np.ndarray:
    """fp64 logits [len(rows), W] (all rows when rows is None).

    For row r = b * next_n + j and t < ctx_r:
        s_h       = sum_d q[b, j, h, d] * k[t, d]            (exact in fp64)
        logit     = scale[t] * sum_h w[r, h] * max(s_h, 0)
    and -inf for ctx_r <= t < W.  Tokens of a page whose id is outside
    [0, num_pages) give NaN.

    Exactness: every e4m3fn value is a multiple of 2^-9 below 2^9 in
    magnitude, so a product is a multiple of 2^-18 below 2^18 and a 128-term
    sum needs fewer than 53 bits: s_h is exact whatever the summation order,
    so a library matmul may form it.
    """
    q = np.asarray(q)
    B, nn, H, dd = q.shape
    assert nn == next_n and dd == D
    weights = np.asarray(weights, dtype=np.float64).reshape(B * next_n, H)
    block_table = np.asarray(block_table)
    W = int(max_model_len)
    ctx_r = row_context_lengths(context_lens, next_n, W, block_table.shape[1], page_size)
    if rows is None:
        rows = np.arange(B * next_n)
    rows = np.asarray(rows, dtype=np.int64)
    out = np.full((len(rows), W), -np.inf, dtype=np.float64)
    by_request = {}
    for i, r in enumerate(rows):
        by_request.setdefault(int(r) // next_n, []).append((i, int(r)))
    qv = _TABLE[q]                                     # [B, next_n, H, D] fp64
    for b, items in by_request.items():
        n_tok = max(int(ctx_r[r]) for _, r in items)
        if n_tok == 0:
            continue
        kv, scale, valid = gather_request_tokens(pool_ids, pool_data, num_pages, page_size,
                                                 block_table[b], n_tok, layout)
        for i, r in items:
            j = r - b * next_n
            n = int(ctx_r[r])
            if n == 0:
                continue
            s = kv[:n] @ qv[b, j].T                    # [n, H], exact
            acc = np.maximum(s, 0.0) @ weights[r]      # sum_h w[r, h] * ReLU(s_h)
            logit = scale[:n] * acc
            logit[~valid[:n]] = np.nan
            out[i, :n] = logit
    return out


# ---------------------------------------------------------------------------
# Top-k.
# ---------------------------------------------------------------------------
def top_k_per_row(logits: np.ndarray, row_ctx: np.ndarray, k: int) -> np.ndarray:
    """int32 [rows, k]: for each row, the column indices of its min(k, ctx_r)
    largest values among columns [0, ctx_r), largest first, equal values in
    increasing column order; the remaining entries are -1."""
    logits = np.asarray(logits)
    out = np.full((logits.shape[0], k), -1, dtype=np.int32)
    for i in range(logits.shape[0]):
        n = int(row_ctx[i])
        if n <= 0:
            continue
        order = np.argsort(-logits[i, :n], kind="stable")
        take = order[:min(k, n)]
        out[i, :len(take)] = take
    return out
