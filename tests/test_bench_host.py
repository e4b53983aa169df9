"""Host-side logic of the benchmark, on CPU: the metric's row-token count, the
algorithmic byte and flop counts, and the cross-rank aggregation run as two
`gloo` ranks (the multi-GPU path has independent ranks and no data-path
collective; only the timing reduction crosses ranks)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import oracle
import synth


def test_row_tokens_matches_oracle_row_lengths():
    for w in (synth.tiny(), synth.custom(batch=4, next_n=3, heads=64, page_size=8,
                                         context_lens=[0, 2, 50, 17], max_model_len=40, seed=1)):
        n = oracle.row_context_lengths(w.context_lens, w.next_n, w.max_model_len,
                                       w.block_table.shape[1], w.page_size)
        assert bench.row_tokens(w) == int(n.sum())


def test_algorithmic_counts_tiny():
    w = synth.tiny()
    # K: (300 + 17) tokens x 132 B; table: 19 + 2 entries; q and w: 2 x 64 x 132;
    # output 2 x 512 x 4; context lengths 2 x 4.
    assert bench.logits_bytes(w) == 317 * 132 + 21 * 4 + 2 * 64 * 132 + 2 * 512 * 4 + 8
    assert bench.logits_flops(w) == 317 * 2 * 64 * 128
    assert bench.topk_bytes(w) == 317 * 4 + 2 * 64 * 4
    assert bench.epilogue_fp32_ops(w) == 317 * 64 * 2


def test_algorithmic_counts_mtp_rows_read_k_once_per_request():
    # next_n = 3, contexts 0, 2, 50, 17 clamped to W = 40: K is read once per
    # request (0 + 2 + 40 + 17 tokens), while the rows see 0, 1+2, 3 x 40,
    # 15+16+17 tokens.
    w = synth.custom(batch=4, next_n=3, heads=64, page_size=8, context_lens=[0, 2, 50, 17],
                     max_model_len=40, seed=1)
    assert w.block_table.shape[1] * w.page_size >= 40
    assert bench.row_tokens(w) == 0 + 3 + 120 + 48
    assert bench.logits_bytes(w) == (59 * 132 + (0 + 1 + 5 + 3) * 4 + 4 * 3 * 64 * 132
                                     + 12 * 40 * 4 + 4 * 4)
    assert bench.logits_flops(w) == 171 * 2 * 64 * 128
    assert bench.epilogue_fp32_ops(w) == 171 * 64 * 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = bench.rank_workload("tiny", rank)
        tok = bench.row_tokens(w)
        ms, total = bench.aggregate(1.0 + rank, tok, world, "cpu")
        out[rank] = (ms, total, tok)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_max_time_and_total_tokens():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0][0] == res[1][0] == 2.0                # slowest rank's time
    assert res[0][1] == res[1][1] == res[0][2] + res[1][2]


def test_single_rank_aggregate_is_identity():
    assert bench.aggregate(3.5, 17, 1) == (3.5, 17)
