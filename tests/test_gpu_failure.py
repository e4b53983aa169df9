"""The bounded pipeline wait on the GPU, made to run out without breaking a
pipeline (`sai_selftest_bounded_wait`: a shared-memory barrier nothing
arrives on): the wait ends within its budget or when another warp raises the
abort flag, SAI_STATUS_TIMEOUT reaches the host, and the context stays usable
(a logits launch afterwards still matches the oracle)."""
import time

import pytest
import torch

import synth
import sparse_attention_indexer_03_gb300 as sai
from parity import assert_logits_close, oracle_logits, run_logits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    sai.library()


def _timed_selftest(mode, cycles):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    sai.selftest_bounded_wait(mode, cycles, status)
    torch.cuda.synchronize()
    return int(status.item()), time.perf_counter() - t0


@pytest.mark.parametrize("mode", [0, 1])
def test_a_wait_that_never_completes_ends_and_reports_timeout(mode):
    # About 1 ms of SM clock either way: the budget itself (mode 0), or the
    # delay before the abort flag under the kernels' 2^31-cycle budget (mode 1).
    st, secs = _timed_selftest(mode, 2_000_000)
    assert st == sai.STATUS_TIMEOUT
    assert secs < 0.5, secs                     # far below the 2^31-cycle budget (about 1 s)


def test_the_context_stays_usable_after_a_timeout():
    st, _ = _timed_selftest(0, 100_000)
    assert st == sai.STATUS_TIMEOUT
    w = synth.tiny()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _, view, _ = run_logits(w, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_logits_close(view[:, :w.max_model_len].cpu().numpy(), oracle_logits(w))
