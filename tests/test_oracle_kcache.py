"""Pins of the K-cache write oracle (`oracle/kcache.py`) against facts fixed
outside it: a library FP8 conversion, the e4m3fn value table's own order,
closed forms of the scale, the FP8 rounding error bound, power-of-two
invariance, and the logits oracle's independent read path."""
import numpy as np
import pytest

import oracle
from oracle import kcache

D = 128


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    """bf16 bits of float32 values that are exactly representable in bf16."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    assert ((b & 0xFFFF) == 0).all()
    return (b >> 16).astype(np.uint16)


def _bf16_round(x: np.ndarray) -> np.ndarray:
    """Truncate float32 values to bf16-representable ones (any rounding will do
    for building inputs)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) & np.uint32(0xFFFF0000)
    return b.view(np.float32)


def test_encode_matches_torch_fp8_cast_in_range():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.uniform(-448, 448, 20000), rng.standard_normal(20000) * 3,
                        rng.standard_normal(20000) * 1e-3]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = kcache.e4m3fn_encode(x)
    assert (got == ref).all()


def test_encode_round_trips_every_finite_code():
    codes = np.array([c for c in range(256) if c not in oracle.E4M3FN_NAN_CODES], dtype=np.uint8)
    vals = np.array([oracle.e4m3fn_value(c) for c in codes], dtype=np.float32)
    got = kcache.e4m3fn_encode(vals)
    assert (got == codes).all()


def test_encode_ties_go_to_the_even_code_and_saturate():
    # 1.0625 lies halfway between 1.0 (0x38) and 1.125 (0x39); 1.1875 between
    # 1.125 (0x39) and 1.25 (0x3A).
    assert kcache.e4m3fn_encode(np.float32([1.0625, 1.1875, -1.0625]))[:].tolist() == [0x38, 0x3A, 0xB8]
    # Halfway between the two smallest subnormals 2^-9 (0x01) and 2^-8 (0x02).
    assert int(kcache.e4m3fn_encode(np.float32([1.5 * 2.0 ** -9]))[0]) == 0x02
    assert kcache.e4m3fn_encode(np.float32([448.0, 460.0, 1000.0, -1e6])).tolist() == [0x7E, 0x7E, 0x7E, 0xFE]
    assert kcache.e4m3fn_encode(np.float32([0.0, -0.0, -1e-9])).tolist() == [0x00, 0x80, 0x80]


def test_scale_is_amax_over_448_and_the_max_element_is_448():
    rng = np.random.default_rng(1)
    x = _bf16_round(rng.standard_normal((64, D)).astype(np.float32) * rng.uniform(0.01, 50, (64, 1)))
    codes, scales = kcache.quantize_k_rows(_bf16_bits(x))
    amax = np.abs(x).max(axis=1)
    assert (scales == (amax / np.float32(448.0)).astype(np.float32)).all()
    arg = np.abs(x).argmax(axis=1)
    top = codes[np.arange(64), arg]
    assert ((top & 0x7F) == 0x7E).all()
    assert ((top >> 7) == (x[np.arange(64), arg] < 0)).all()


def test_zero_row_has_scale_one_and_zero_codes():
    codes, scales = kcache.quantize_k_rows(np.zeros((2, D), np.uint16))
    assert scales.tolist() == [1.0, 1.0] and not codes.any()


def test_dequantised_values_within_the_fp8_rounding_bound():
    rng = np.random.default_rng(2)
    x = _bf16_round(rng.standard_normal((256, D)).astype(np.float32))
    codes, scales = kcache.quantize_k_rows(_bf16_bits(x))
    deq = oracle.e4m3fn_table()[codes] * scales[:, None].astype(np.float64)
    # Half an e4m3 ulp: 2^-4 relative for normals, 2^-10 absolute (times the
    # scale) for subnormals; the fp32 quotient adds 2^-24 relative.
    bound = np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * scales[:, None]) * (1 + 2.0 ** -20)
    assert (np.abs(deq - x) <= bound).all()


def test_power_of_two_scaling_moves_only_the_scale():
    rng = np.random.default_rng(3)
    x = _bf16_round(rng.standard_normal((32, D)).astype(np.float32))
    c0, s0 = kcache.quantize_k_rows(_bf16_bits(x))
    for m in (-7, 5):
        c1, s1 = kcache.quantize_k_rows(_bf16_bits(x * np.float32(2.0 ** m)))
        assert (c1 == c0).all()
        assert (s1 == s0 * np.float32(2.0 ** m)).all()


@pytest.mark.parametrize("layout", ["split", "interleaved"])
@pytest.mark.parametrize("page_size", [8, 64])
def test_inserted_tokens_read_back_through_the_logits_oracle(layout, page_size):
    # Write 3 * P tokens to pages chosen by a table, then read them back with
    # the logits oracle's independent gather of a request's tokens.
    rng = np.random.default_rng(page_size)
    num_pages = 7
    table = np.array([5, 0, 3])
    n = 3 * page_size
    x = _bf16_round(rng.standard_normal((n, D)).astype(np.float32))
    t = np.arange(n)
    slots = table[t // page_size] * page_size + t % page_size
    codes, scales = kcache.quantize_k_rows(_bf16_bits(x))
    cache = np.zeros(num_pages * page_size * (D + 4), np.uint8)
    cache = kcache.insert_k_rows(cache, slots, codes, scales, num_pages, page_size, layout)
    pool = cache.reshape(num_pages, -1)
    values, sc, valid = oracle.gather_request_tokens(np.arange(num_pages), pool, num_pages, page_size,
                                                     table, n, layout=layout)
    assert valid.all()
    assert (values == oracle.e4m3fn_table()[codes]).all()
    assert (sc == scales.astype(np.float64)).all()
    # Pages the table does not name stay zero.
    for p in (1, 2, 4, 6):
        assert not pool[p].any()


def test_negative_and_out_of_range_slots_write_nothing():
    codes = np.full((3, D), 0x11, np.uint8)
    scales = np.float32([2.0, 3.0, 4.0])
    cache = np.zeros(2 * 8 * (D + 4), np.uint8)
    out = kcache.insert_k_rows(cache, [-1, 16, 99], codes, scales, 2, 8)
    assert not out.any()
    out = kcache.insert_k_rows(cache, [-1, 15, -5], codes, scales, 2, 8)
    page1 = out.reshape(2, -1)[1]
    assert (page1[7 * D:8 * D] == 0x11).all()
    assert page1[8 * D + 7 * 4:8 * D + 8 * 4].view("<f4")[0] == 3.0
    assert out.reshape(2, -1)[0].sum() == 0
