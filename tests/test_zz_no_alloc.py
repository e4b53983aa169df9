"""`sai_paged_mqa_logits_topk_static`, the fused launch with the library's
static request counters instead of a caller workspace (through the C ABI).

Collected last so that it also runs after every other test in one process.
Two calls in a row must each match `sai_paged_mqa_logits_topk` with a zeroed
workspace: logits within the parity tolerance, indices entry for entry.
"""
import ctypes

import numpy as np
import pytest

import synth
import sparse_attention_indexer_03_gb300 as sai
from parity import ATOL, RTOL

STATIC_MAX_BATCH = 16384


def _call_static(lib, w, dev, logits, idx, k, stream):
    return lib.sai_paged_mqa_logits_topk_static(
        dev["q"].data_ptr(), dev["kv"].data_ptr(), w.pool.num_pages, w.page_size,
        dev["weights"].data_ptr(), dev["context_lens"].data_ptr(), dev["block_table"].data_ptr(),
        dev["block_table"].stride(0), w.batch, w.next_n, w.heads, w.head_dim,
        logits.data_ptr(), logits.stride(0), w.max_model_len, k, idx.data_ptr(), idx.stride(0),
        None, stream)


def _call_workspace(lib, w, dev, logits, idx, k, ws, stream):
    return lib.sai_paged_mqa_logits_topk(
        dev["q"].data_ptr(), dev["kv"].data_ptr(), w.pool.num_pages, w.page_size,
        dev["weights"].data_ptr(), dev["context_lens"].data_ptr(), dev["block_table"].data_ptr(),
        dev["block_table"].stride(0), w.batch, w.next_n, w.heads, w.head_dim,
        logits.data_ptr(), logits.stride(0), w.max_model_len, k, idx.data_ptr(), idx.stride(0),
        ws.data_ptr(), ws.numel() * ws.element_size(), None, stream)


def test_batch_beyond_the_static_counters_is_rejected():
    # Rejected before any CUDA call: the fake pointers are never used.
    sai.build()
    lib = sai.library()
    A16, A4 = 0x10000, 0x20000
    rc = lib.sai_paged_mqa_logits_topk_static(A16, A16, 20, 16, A16, A4, A4, 20, STATIC_MAX_BATCH + 1, 1, 64,
                                              128, A4, 512, 512, 64, A4, 64, None, None)
    assert rc == sai.ERR_WORKSPACE
    rc = lib.sai_paged_mqa_logits_topk_static(A16, A16, 20, 16, A16, A4, A4, 20, 2, 1, 64, 128, A4, 512,
                                              512, 64, None, 64, None, None)
    assert rc == sai.ERR_INVALID_ARGUMENT


def _fill_heavy():
    # -inf fill four times the tiles: the grid-wide fill counter (the static
    # array's word after the queue's head, tail and done count) is used.
    return synth.custom(batch=16, next_n=2, heads=64, page_size=16,
                        context_lens=[0, 1, 127, 2049, 3000, 130, 4100, 3, 2600, 3777, 4500, 128, 2047, 1, 300, 64],
                        max_model_len=400000, logits_stride=400128, topk=2048, seed=77)


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["tiny", "decode", "mtp", "fill_heavy"])
def test_two_calls_match_the_workspace_entry_point(name):
    import torch

    sai.build()
    lib = sai.library()
    w = {"tiny": synth.tiny, "decode": synth.decode, "mtp": synth.mtp, "fill_heavy": _fill_heavy}[name]()
    dev = w.to_device()
    k = w.topk
    stream = torch.cuda.current_stream().cuda_stream
    ref_logits = torch.empty((w.rows, w.logits_stride), dtype=torch.float32, device="cuda")
    ref_idx = torch.full((w.rows, k), -7, dtype=torch.int32, device="cuda")
    ws = torch.zeros(sai.logits_topk_workspace_bytes(w.batch) // 4, dtype=torch.int32, device="cuda")
    assert _call_workspace(lib, w, dev, ref_logits, ref_idx, k, ws, stream) == sai.OK
    torch.cuda.synchronize()
    W = w.max_model_len
    ref = ref_logits[:, :W].cpu().numpy().astype(np.float64)
    for _ in range(2):
        logits = torch.full((w.rows, w.logits_stride), 99.0, dtype=torch.float32, device="cuda")
        idx = torch.full((w.rows, k), -7, dtype=torch.int32, device="cuda")
        assert _call_static(lib, w, dev, logits, idx, k, stream) == sai.OK
        torch.cuda.synchronize()
        got = logits[:, :W].cpu().numpy().astype(np.float64)
        assert (np.isneginf(got) == np.isneginf(ref)).all()
        fin = np.isfinite(ref)
        assert (np.abs(got[fin] - ref[fin]) <= ATOL + RTOL * np.abs(ref[fin])).all()
        assert torch.equal(idx, ref_idx)


@pytest.mark.gpu
def test_reset_between_calls_keeps_the_static_entry_point_exact():
    # sai_paged_mqa_logits_topk_static_reset zeroes the static workspace on the
    # caller's stream (the remedy after a call that raised STATUS_TIMEOUT):
    # static calls before and after resets on the same stream still match the
    # workspace entry point entry for entry.
    import torch

    sai.build()
    lib = sai.library()
    w = synth.decode()
    dev = w.to_device()
    k = w.topk
    stream = torch.cuda.current_stream().cuda_stream
    ref_logits = torch.empty((w.rows, w.logits_stride), dtype=torch.float32, device="cuda")
    ref_idx = torch.full((w.rows, k), -7, dtype=torch.int32, device="cuda")
    ws = torch.zeros(sai.logits_topk_workspace_bytes(w.batch) // 4, dtype=torch.int32, device="cuda")
    assert _call_workspace(lib, w, dev, ref_logits, ref_idx, k, ws, stream) == sai.OK
    for _ in range(2):
        sai.paged_mqa_logits_topk_static_reset()
        logits = torch.full((w.rows, w.logits_stride), 99.0, dtype=torch.float32, device="cuda")
        idx = torch.full((w.rows, k), -7, dtype=torch.int32, device="cuda")
        assert _call_static(lib, w, dev, logits, idx, k, stream) == sai.OK
        torch.cuda.synchronize()
        assert torch.equal(idx, ref_idx)
        assert torch.equal(logits[:, :w.max_model_len], ref_logits[:, :w.max_model_len])
