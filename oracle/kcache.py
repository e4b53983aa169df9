"""Plain definition of the indexer K-cache write: per-token FP8 quantisation
of new K rows and their insertion into the paged cache through int64 slots.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources.  The cache token format is the one the logits op reads: D = 128
e4m3fn value bytes and one fp32 scale per token (the `[num_blocks,
block_size, 1, D + 4]` byte tensor of the reproducer in aiter PR 4244, "fix
silent tail-row drop in deepgemm_fp8_paged_mqa_logits at large output
stride", section "small reproducer"), in the page-split layout adopted for
the logits (values of a page's P tokens first, then their P scales) or the
interleaved per-token layout.  The write addresses the cache through slots
computed in int64, the rule ATOM PR 2533 ("[MLA] Address Triton decode KV
rows with int64 ids", section "Problem") states for the cache kernels: a
slot is page * P + position, and byte offsets are formed from it in 64 bits.

Readings taken where the pages are silent (each is listed in the design
notes):
  * input K rows are bf16 `[T, 128]`, one row per new token;
  * the token's scale is amax / 448 in fp32, 448 being the largest e4m3fn
    magnitude, and 1 when the row is all zero;
  * each value's code is e4m3fn(k / scale): the fp32 quotient (correctly
    rounded division) rounded to the nearest e4m3fn value, ties to the even
    code, magnitudes past 448 saturating to 448, the sign kept (a negative
    value that rounds to zero gives the code of -0);
  * a negative slot means "no token" and writes nothing; a slot at or past
    num_pages * P writes nothing either (the library raises a status bit).
"""
from __future__ import annotations

import numpy as np

from .indexer import D, SCALE_BYTES, e4m3fn_value

E4M3FN_MAX = 448.0

# Non-negative finite e4m3fn values in code order 0x00 .. 0x7E (ascending).
_POS_VALUES = np.array([e4m3fn_value(c) for c in range(0x7F)], dtype=np.float64)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) to their exact fp32 values."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def e4m3fn_encode(x: np.ndarray) -> np.ndarray:
    """Codes of fp32 values: nearest e4m3fn value, ties to the even code,
    saturating at +-448, sign kept.  No NaN or infinity is expected."""
    x = np.asarray(x, dtype=np.float32)
    mag = np.abs(x.astype(np.float64)).ravel()
    hi = np.searchsorted(_POS_VALUES, mag, side="left")        # first value >= mag
    hi_c = np.minimum(hi, len(_POS_VALUES) - 1)
    lo_c = np.maximum(hi - 1, 0)
    d_hi = _POS_VALUES[hi_c] - mag
    d_lo = mag - _POS_VALUES[lo_c]
    exact = _POS_VALUES[hi_c] == mag
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi_c % 2 == 0))
    code = np.where(exact, hi_c, np.where(take_hi, hi_c, lo_c))
    code = np.where(mag >= E4M3FN_MAX, 0x7E, code)                # saturate
    sign = np.signbit(x.ravel())
    return (code | np.where(sign, 0x80, 0)).astype(np.uint8).reshape(x.shape)


def quantize_k_rows(k_bf16: np.ndarray):
    """Per-token quantisation of K rows given as bf16 bits `[T, D]`.

    Returns (codes uint8 `[T, D]`, scales float32 `[T]`)."""
    k = bf16_to_f32(k_bf16).reshape(-1, D)
    amax = np.max(np.abs(k), axis=1)
    scales = np.where(amax > 0, amax / np.float32(E4M3FN_MAX), np.float32(1.0)).astype(np.float32)
    q = (k / scales[:, None]).astype(np.float32)
    return e4m3fn_encode(q), scales


def insert_k_rows(cache: np.ndarray, slot_mapping, codes: np.ndarray, scales: np.ndarray,
                  num_pages: int, page_size: int, layout: str = "split") -> np.ndarray:
    """Write each token t with slot_mapping[t] >= 0 into a copy of the paged
    cache bytes `cache` (num_pages * P * (D + 4) bytes) and return it."""
    out = np.array(cache, dtype=np.uint8, copy=True).reshape(-1)
    page_bytes = page_size * (D + SCALE_BYTES)
    scale_bytes = np.ascontiguousarray(scales, dtype="<f4").view(np.uint8).reshape(-1, SCALE_BYTES)
    for t, s in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        s = int(s)
        if s < 0 or s >= num_pages * page_size:
            continue
        page, pos = divmod(s, page_size)
        base = page * page_bytes
        if layout == "split":
            v0 = base + pos * D
            s0 = base + page_size * D + pos * SCALE_BYTES
        elif layout == "interleaved":
            v0 = base + pos * (D + SCALE_BYTES)
            s0 = v0 + D
        else:
            raise ValueError(layout)
        out[v0:v0 + D] = codes[t]
        out[s0:s0 + SCALE_BYTES] = scale_bytes[t]
    return out
