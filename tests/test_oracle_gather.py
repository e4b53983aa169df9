"""Pins of the consumer-gather oracle (`oracle/gather.py`): rows whose bytes
spell their own row id, the row-id rule written as a closed form, the int64
offsets past the int32 limit that ATOM PR 2533 reports, and the padding and
out-of-pool cases."""
import numpy as np

from oracle import gather

MLA_ROW = 576


def _id_pool(n_rows: int, row_bytes: int) -> np.ndarray:
    """Pool whose row j holds j as little-endian int64, repeated."""
    reps = row_bytes // 8
    ids = np.repeat(np.arange(n_rows, dtype="<i8"), reps).reshape(n_rows, reps)
    return ids.view(np.uint8).reshape(-1)


def test_gathered_rows_spell_their_row_ids():
    rng = np.random.default_rng(0)
    P, num_pages, next_n = 4, 30, 2
    table = np.stack([rng.permutation(num_pages)[:6] for _ in range(3)])     # 3 requests, 24 tokens each
    idx = rng.integers(0, 24, (6, 5))
    idx[0, 4] = -1
    ids = gather.kv_row_ids(idx, table, next_n, P, num_pages)
    rows = gather.gather_kv_rows(_id_pool(num_pages * P, 64), ids, 64)
    got = rows.reshape(6, 5, 8, 8).view("<i8")[..., 0]
    for r in range(6):
        for i in range(5):
            t = idx[r, i]
            want = -1 if t < 0 else table[r // next_n, t // P] * P + t % P
            assert ids[r, i] == want
            assert (got[r, i] == (0 if want < 0 else want)).all()


def test_offsets_past_the_int32_limit_are_exact():
    # 2^31 / 576 = 3,728,270.2: row 3,728,270 (block 233,016, position 14)
    # is the last whose MLA offset fits in int32; row 3,728,271 (position 15)
    # is the first past it.
    P = 16
    table = np.array([[233016, 240000]])
    ids = gather.kv_row_ids(np.array([[14, 15, 24]]), table, 1, P, 250000)
    assert ids.tolist() == [[3728270, 3728271, 240000 * 16 + 8]]
    offs = [int(j) * MLA_ROW for j in ids[0]]
    assert offs[0] < 2 ** 31 < offs[1]
    wrapped = [(o + 2 ** 31) % 2 ** 32 - 2 ** 31 for o in offs]             # what an int32 product gives
    assert wrapped[0] == offs[0] and wrapped[1] < 0 and wrapped[2] < 0


def test_padding_and_bad_entries_give_zero_rows():
    P, num_pages = 8, 4
    table = np.array([[2, -1, 9, 1]])
    idx = np.array([[-1, 3, 9, 17, 40, 25]])            # pad, ok, page -1, page 9 (past pool), past table, ok
    ids = gather.kv_row_ids(idx, table, 1, P, num_pages)
    assert ids.tolist() == [[-1, 2 * 8 + 3, -1, -1, -1, 1 * 8 + 1]]
    pool = np.arange(num_pages * P * 16, dtype=np.int64).astype(np.uint8)
    rows = gather.gather_kv_rows(pool, ids, 16)
    assert not rows[0, [0, 2, 3, 4]].any()
    assert (rows[0, 1] == pool[19 * 16:20 * 16]).all()
