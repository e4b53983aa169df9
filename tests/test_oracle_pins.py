"""Pins of the CPU oracle to facts fixed outside its own code.

Each test ties one part of `oracle.indexer` to something it cannot agree with
by construction: a library FP8 conversion, exact rational arithmetic, a
closed form, an invariant the definition implies, a library sort, or bytes
printed by the source pages.  A plausible slip in the oracle (a dropped
scale, an inverted ReLU, an off-by-one MTP offset, a transposed operand, a
mis-read page slot) fails at least one of them.
"""
from fractions import Fraction
import struct

import numpy as np
import pytest
import torch

import oracle
import synth
from conftest import golden_rows

D = 128


def _lib_fp8_to_f64(codes: np.ndarray) -> np.ndarray:
    """Library decoding of e4m3fn bytes (torch), independent of the oracle's."""
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _call(w: synth.Workload, rows=None, W=None, table=None, pool=None, ctx=None):
    pool = pool if pool is not None else w.pool
    return oracle.paged_mqa_logits(
        w.q, pool.ids, pool.data, pool.num_pages, w.page_size, w.weights,
        w.context_lens if ctx is None else ctx,
        w.block_table if table is None else table, w.next_n,
        w.max_model_len if W is None else W, layout=pool.layout, rows=rows)


# --------------------------------------------------------------------- FP8
def test_e4m3fn_matches_library_conversion_on_all_codes():
    ours = oracle.e4m3fn_table()
    lib = _lib_fp8_to_f64(np.arange(256, dtype=np.uint8))
    nan = np.isnan(lib)
    assert set(np.nonzero(nan)[0].tolist()) == set(oracle.E4M3FN_NAN_CODES)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], lib[~nan])


def test_e4m3fn_range_facts():
    # OCP E4M3 ("fn"): largest finite 448, smallest subnormal 2^-9, no infinity.
    t = oracle.e4m3fn_table()
    assert np.nanmax(t) == 448.0 and np.nanmin(t) == -448.0
    assert t[0x7E] == 448.0 and t[0x01] == 2.0 ** -9 and t[0x38] == 1.0
    assert not np.isinf(t).any()


# ------------------------------------------------------------- page layout
def test_reproducer_scale_bytes_decode_to_one():
    (b0, b1, b2, b3, val), = golden_rows("reproducer_scale_bytes.txt")
    sbytes = [int(b0), int(b1), int(b2), int(b3)]
    # Two-token page laid out by hand (page-split: values of both tokens, then
    # both scales), so that slot and layout arithmetic are exercised too.
    P = 2
    page = np.zeros(P * (D + 4), np.uint8)
    page[0:D] = 0x38                        # token 0: all 1.0
    page[D:2 * D] = 0x40                    # token 1: all 2.0
    page[2 * D:2 * D + 4] = [0, 0, 0, 64]   # token 0 scale 2.0
    page[2 * D + 4:2 * D + 8] = sbytes      # token 1 scale from the fixture
    vals, scales, valid = oracle.gather_request_tokens(
        np.array([0]), page[None, :], 1, P, np.array([0]), 2, layout="split")
    assert scales[1] == float(val) == 1.0 and scales[0] == 2.0
    assert (vals[0] == 1.0).all() and (vals[1] == 2.0).all() and valid.all()
    # The same token in the interleaved layout: D values then 4 scale bytes.
    page2 = np.zeros(P * (D + 4), np.uint8)
    page2[D + 4:2 * D + 4] = 0x40
    page2[2 * D + 4:] = sbytes
    vals, scales, _ = oracle.gather_request_tokens(
        np.array([0]), page2[None, :], 1, P, np.array([0]), 2, layout="interleaved")
    assert scales[1] == 1.0 and (vals[1] == 2.0).all()


@pytest.mark.parametrize("layout", ["split", "interleaved"])
@pytest.mark.parametrize("P", [1, 4, 8, 16])
def test_pages_read_back_the_dense_cache(layout, P):
    """Pages written by the generator from a dense K give the dense K back."""
    rng = np.random.default_rng(11)
    n_pages, ntok = 6, 6 * P - 3
    vals = rng.integers(0, 256, size=(n_pages, P, D), dtype=np.uint8)
    vals[vals == 0x7F] = 0x01
    vals[vals == 0xFF] = 0x81
    scales = rng.uniform(0.5, 2, size=(n_pages, P)).astype(np.float32)
    data = synth.pack_pages(vals, scales, layout)
    ids = np.arange(n_pages)
    table = rng.permutation(n_pages)
    got_v, got_s, valid = oracle.gather_request_tokens(ids, data, n_pages, P, table, ntok, layout)
    dense_v = _lib_fp8_to_f64(vals[table].reshape(-1, D)[:ntok])
    dense_s = scales[table].reshape(-1)[:ntok].astype(np.float64)
    assert np.array_equal(got_v, dense_v) and np.array_equal(got_s, dense_s) and valid.all()


# ---------------------------------------------------------- brute force
def _fraction_logits(w: synth.Workload):
    """Exact rational logits by a per-(row, token, head, d) loop.

    Decoding goes through torch's FP8 conversion and struct's float32 unpack;
    page addressing follows the page-split layout: token t is slot t % P of
    page table[b, t // P]; values at slot * D, scale at P * D + 4 * slot.
    """
    P, W, nn = w.page_size, w.max_model_len, w.next_n
    dense = w.pool.dense()
    cap = min(W, w.block_table.shape[1] * P)
    qf = _lib_fp8_to_f64(w.q)
    out = {}
    for b in range(w.batch):
        for j in range(nn):
            r = b * nn + j
            n = min(max(int(w.context_lens[b]) - nn + j + 1, 0), cap)
            for t in range(W):
                if t >= n:
                    out[(r, t)] = None
                    continue
                page = dense[int(w.block_table[b, t // P])]
                slot = t % P
                k = _lib_fp8_to_f64(page[slot * D:(slot + 1) * D])
                scale = Fraction(struct.unpack("<f", bytes(page[P * D + 4 * slot:P * D + 4 * slot + 4]))[0])
                acc = Fraction(0)
                bound = Fraction(0)
                for h in range(w.heads):
                    s = sum(Fraction(qf[b, j, h, d]) * Fraction(k[d]) for d in range(D))
                    term = Fraction(float(w.weights[r, h])) * max(s, Fraction(0))
                    acc += term
                    bound += abs(term)
                out[(r, t)] = (scale * acc, abs(scale) * bound)
    return out


def test_logits_equal_exact_rational_brute_force():
    w = synth.custom(batch=2, next_n=2, heads=3, page_size=4, context_lens=[7, 2],
                     max_model_len=9, table_stride=3, num_pages=7, seed=5)
    got = _call(w)
    exact = _fraction_logits(w)
    for (r, t), v in exact.items():
        if v is None:
            assert got[r, t] == -np.inf
        else:
            val, bound = v
            assert abs(got[r, t] - float(val)) <= 1e-14 * float(bound) + 1e-300, (r, t)


# ----------------------------------------------------------- closed forms
def test_constant_q_and_k_closed_form():
    # q = a, k = c everywhere => logit = scale * 128 * a * c * sum_h w_h when a*c > 0.
    w = synth.custom(batch=2, next_n=1, heads=8, page_size=8, context_lens=[20, 11],
                     max_model_len=24, seed=9)
    a_code, c_code = 0x3C, 0x44           # 1.5 and 3.0
    w.q[:] = a_code
    data = w.pool.data.copy()
    data[:, :8 * D] = c_code
    pool = synth.KVPool(w.pool.num_pages, 8, "split", w.pool.ids, data)
    got = _call(w, pool=pool)
    a, c = 1.5, 3.0
    for b, n in enumerate([20, 11]):
        v, sc, _ = oracle.gather_request_tokens(pool.ids, pool.data, pool.num_pages, 8,
                                                w.block_table[b], n)
        want = sc * (D * a * c * w.weights[b].astype(np.float64).sum())
        assert np.allclose(got[b, :n], want, rtol=1e-15, atol=0)
        assert np.isneginf(got[b, n:]).all()
    # a * c < 0: every ReLU is zero.
    w.q[:] = 0xBC                          # -1.5
    got = _call(w, pool=pool)
    assert (got[0, :20] == 0).all() and (got[1, :11] == 0).all()


def test_one_hot_weights_select_one_relu_head():
    w = synth.custom(batch=1, next_n=2, heads=6, page_size=16, context_lens=[40],
                     max_model_len=40, seed=13)
    for r, h0 in [(0, 2), (1, 5)]:
        w.weights[r] = 0
        w.weights[r, h0] = 1
    got = _call(w)
    dense = w.pool.dense()
    kv = np.concatenate([dense[p][:16 * D].reshape(16, D) for p in w.block_table[0]])[:40]
    sc = np.concatenate([dense[p][16 * D:].view("<f4") for p in w.block_table[0]])[:40]
    kf = _lib_fp8_to_f64(kv)
    qf = _lib_fp8_to_f64(w.q)
    for j, h0 in [(0, 2), (1, 5)]:
        n = 40 - 2 + j + 1
        dots = kf[:n] @ qf[0, j, h0]
        assert (dots < 0).any() and (dots > 0).any()      # both signs occur
        want = np.where(dots > 0, dots, 0.0) * sc[:n]
        assert np.array_equal(got[j, :n], want)


def test_single_head_unit_weight_unit_scale_is_relu_of_gemv():
    w = synth.custom(batch=1, next_n=1, heads=1, page_size=8, context_lens=[33],
                     max_model_len=33, seed=17)
    w.weights[:] = 1
    data = w.pool.data.copy()
    data[:, 8 * D:] = np.frombuffer(struct.pack("<f", 1.0), np.uint8).tolist() * 8
    pool = synth.KVPool(w.pool.num_pages, 8, "split", w.pool.ids, data)
    got = _call(w, pool=pool)
    dense = pool.dense()
    kv = np.concatenate([dense[p][:8 * D].reshape(8, D) for p in w.block_table[0]])[:33]
    gemv = _lib_fp8_to_f64(kv) @ _lib_fp8_to_f64(w.q[0, 0, 0])
    assert np.array_equal(got[0], np.maximum(gemv, 0))


def test_reproducer_inputs_make_relu_inactive():
    """The reproducer's inputs (aiter PR 4244, "small reproducer"): q and K bytes
    in [1, 63] (positive e4m3 values), scale bytes of float32 1.0, unit
    weights.  Every dot product is positive, so the ReLU is the identity and
    logit[t] = sum_h q_h . k_t, a plain matrix product."""
    rng = np.random.default_rng(21)
    B, nn, H, P, ctx = 2, 2, 4, 16, 37
    (b0, b1, b2, b3, _), = golden_rows("reproducer_scale_bytes.txt")
    npg = -(-ctx // P)
    vals = rng.integers(1, 64, size=(npg, P, D), dtype=np.uint8)
    page_scale = np.tile(np.array([int(b0), int(b1), int(b2), int(b3)], np.uint8), P)
    data = np.concatenate([vals.reshape(npg, -1), np.tile(page_scale, (npg, 1))], axis=1)
    q = rng.integers(1, 64, size=(B, nn, H, D), dtype=np.uint8)
    table = np.tile(np.arange(npg), (B, 1))          # identity table, repeated
    got = oracle.paged_mqa_logits(q, np.arange(npg), data, npg, P, np.ones((B * nn, H)),
                                  np.array([ctx, ctx]), table, nn, ctx)
    kf = _lib_fp8_to_f64(vals.reshape(-1, D))[:ctx]
    qf = _lib_fp8_to_f64(q)
    for b in range(B):
        for j in range(nn):
            n = ctx - nn + j + 1
            want = kf[:n] @ qf[b, j].sum(axis=0)
            assert np.array_equal(got[b * nn + j, :n], want)


# -------------------------------------------------------------- invariants
def test_permuting_pool_pages_leaves_logits_unchanged():
    w = synth.custom(batch=3, next_n=2, heads=8, page_size=8, context_lens=[50, 0, 23],
                     max_model_len=64, seed=23)
    base = _call(w)
    rng = np.random.default_rng(1)
    perm = rng.permutation(w.pool.num_pages)          # page p moves to perm[p]
    dense = w.pool.dense()
    moved = np.zeros_like(dense)
    moved[perm] = dense
    pool2 = synth.KVPool(w.pool.num_pages, 8, "split", np.arange(w.pool.num_pages), moved)
    got = _call(w, pool=pool2, table=perm[w.block_table])
    assert np.array_equal(np.isneginf(got), np.isneginf(base))
    assert np.array_equal(got, base)


def test_row_context_masks_match_hand_count():
    # next_n = 3; ctx {5, 1, 0, 9} => rows see [3,4,5], [0,0,1], [0,0,0], [7,8,9].
    w = synth.custom(batch=4, next_n=3, heads=4, page_size=4, context_lens=[5, 1, 0, 9],
                     max_model_len=12, seed=29)
    got = _call(w)
    want = [3, 4, 5, 0, 0, 1, 0, 0, 0, 7, 8, 9]
    assert np.isfinite(got).sum(axis=1).tolist() == want
    for r, n in enumerate(want):
        assert np.isfinite(got[r, :n]).all() and np.isneginf(got[r, n:]).all()
    assert oracle.row_context_lengths([5, 1, 0, 9], 3, 12, 3, 4).tolist() == want


def test_mtp_row_equals_single_row_call():
    w = synth.custom(batch=2, next_n=4, heads=8, page_size=16, context_lens=[45, 3],
                     max_model_len=48, seed=31)
    full = _call(w)
    for b in range(2):
        for j in range(4):
            r = b * 4 + j
            n = max(int(w.context_lens[b]) - 4 + j + 1, 0)
            one = oracle.paged_mqa_logits(
                w.q[b:b + 1, j:j + 1], w.pool.ids, w.pool.data, w.pool.num_pages, 16,
                w.weights[r:r + 1], np.array([n]), w.block_table[b:b + 1], 1, 48)
            assert np.array_equal(one[0], full[r])


def test_compact_and_wide_width_agree_on_valid_columns():
    # Compact width (W = longest context) vs a wide one: identical on the valid
    # columns, -inf on the rest (aiter PR 4244, reproducer's compact reference).
    w = synth.custom(batch=2, next_n=2, heads=8, page_size=8, context_lens=[30, 17],
                     max_model_len=30, table_stride=8, seed=37)
    compact = _call(w)
    wide = _call(w, W=200)
    assert np.array_equal(wide[:, :30], compact)
    assert np.isneginf(wide[:, 30:]).all()


def test_batch_split_into_two_calls_is_identical():
    # One call over the batch vs two calls over its halves (aiter PR 4244,
    # reproducer's chunk0 / chunk1 runs).
    w = synth.custom(batch=4, next_n=2, heads=8, page_size=8, context_lens=[30, 17, 1, 24],
                     max_model_len=32, seed=41)
    full = _call(w)
    for lo, hi in [(0, 2), (2, 4)]:
        part = oracle.paged_mqa_logits(
            w.q[lo:hi], w.pool.ids, w.pool.data, w.pool.num_pages, 8,
            w.weights[lo * 2:hi * 2], w.context_lens[lo:hi], w.block_table[lo:hi], 2, 32)
        assert np.array_equal(part, full[lo * 2:hi * 2])


def test_context_is_clamped_to_width_and_table():
    w = synth.custom(batch=1, next_n=1, heads=4, page_size=4, context_lens=[12],
                     max_model_len=12, table_stride=3, seed=43)
    base = _call(w)
    big = _call(w, ctx=np.array([1000]))           # longer than W and than the table
    assert np.array_equal(big, base) and np.isfinite(base).all()
    narrow = _call(w, W=8)
    assert np.array_equal(narrow, base[:, :8])


def test_page_id_outside_pool_gives_nan_for_that_page_only():
    w = synth.custom(batch=1, next_n=1, heads=4, page_size=4, context_lens=[12],
                     max_model_len=12, seed=47)
    base = _call(w)
    for bad in (-1, w.pool.num_pages, 2 ** 31 - 1):
        table = w.block_table.copy()
        table[0, 1] = bad
        got = _call(w, table=table)
        assert np.isnan(got[0, 4:8]).all()
        assert np.array_equal(got[0, :4], base[0, :4]) and np.array_equal(got[0, 8:], base[0, 8:])


# ------------------------------------------------------------------ top-k
def test_top_k_matches_library_topk_on_distinct_values():
    rng = np.random.default_rng(3)
    vals = rng.permutation(5000).astype(np.float32).reshape(5, 1000) / 7
    ctx = np.array([1000, 999, 513, 64, 1])
    got = oracle.top_k_per_row(vals, ctx, 64)
    for i, n in enumerate(ctx):
        m = min(64, int(n))
        lib = torch.topk(torch.from_numpy(vals[i, :n]), m).indices.numpy()
        assert np.array_equal(got[i, :m], lib)        # distinct values: unique order
        assert (got[i, m:] == -1).all()


def test_top_k_ties_and_short_rows():
    row = np.array([[1.0, 3.0, 3.0, 2.0, 3.0, 3.0, 0.5, -np.inf]], np.float32)
    assert oracle.top_k_per_row(row, [7], 3).tolist() == [[1, 2, 4]]
    assert oracle.top_k_per_row(row, [3], 5).tolist() == [[1, 2, 0, -1, -1]]
    assert oracle.top_k_per_row(row, [0], 2).tolist() == [[-1, -1]]
    # Only columns below the row's context count, whatever lies past it.
    row2 = np.array([[0.0, 1.0, 9.0, 9.0]], np.float32)
    assert oracle.top_k_per_row(row2, [2], 1).tolist() == [[1]]


def test_top_k_of_full_sort_prefix():
    # Sorting the whole row with a library sort and cutting it gives the same set.
    rng = np.random.default_rng(5)
    vals = rng.standard_normal((8, 3000)).astype(np.float32)
    ctx = rng.integers(0, 3000, 8)
    got = oracle.top_k_per_row(vals, ctx, 2048)
    for i, n in enumerate(ctx):
        lib = np.sort(vals[i, :n])[::-1][:min(2048, n)]
        assert np.array_equal(np.sort(vals[i, got[i][got[i] >= 0]])[::-1], lib)
