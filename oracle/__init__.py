"""CPU oracle for the FP8 paged MQA indexer decode path (logits, then top-k).

TEST INFRASTRUCTURE ONLY.  This package is the plain, slow, obviously
correct definition that the CUDA path is checked against.  Only the tests,
the smoke run's check and the benchmark's CPU-baseline leg may import it;
the product library never does, and nothing here shares code with it.

What it computes (fp64 throughout, fp32 only when a caller rounds the
result for comparison):

* `e4m3fn_value`: the OCP FP8 E4M3 ("fn": finite, no infinities) decoding
  rule, written out.
* `paged_mqa_logits`: for every query row r = b * next_n + j and every
  token t of the row's causal context,
      logits[r, t] = scale[t] * sum_h w[r, h] * max(q[b, j, h, :] . k[t, :], 0)
  and -inf for the rest of the row's W columns.  K is read from the paged
  FP8 cache through the block table.
* `top_k_per_row`: the indices of the k largest logits of each row's valid
  columns, ties broken towards the lower index, padded with -1.
* `kcache.quantize_k_rows` / `kcache.insert_k_rows`: the K-cache write that
  precedes the path: per-token FP8 quantisation (scale = amax / 448) and
  insertion into the paged cache through int64 slots.
* `gather.kv_row_ids` / `gather.gather_kv_rows`: the consumer's gather of
  the selected tokens' KV rows through int64 row ids.

Parity status: every function here is pinned by `tests/test_oracle_*.py`
against facts fixed outside this code (a library FP8 conversion, exact
rational brute force, closed forms, invariants, a library sort, the byte
values printed for the reproducer).  No function is "parity unpinned".
"""
from . import gather, kcache  # noqa: F401
from .indexer import (  # noqa: F401
    E4M3FN_NAN_CODES,
    e4m3fn_table,
    e4m3fn_value,
    row_context_lengths,
    gather_request_tokens,
    paged_mqa_logits,
    top_k_per_row,
)
