"""The C ABI without a GPU: the library loads, exports every function that
`include/sai.h` declares, and rejects bad arguments with the documented code
before any CUDA call (fake, never-dereferenced pointers are passed)."""
import ctypes
import os
import re

import pytest

import sparse_attention_indexer_03_gb300 as sai

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    sai.build()
    return sai.library()


def _declared():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            names |= set(re.findall(r"SAI_API\s+[\w\s\*]*?\b(sai_\w+)\s*\(", text))
    return names


def test_header_declares_the_entry_points():
    names = _declared()
    assert {"sai_paged_mqa_logits", "sai_top_k_per_row_decode", "sai_top_k_workspace_bytes",
            "sai_paged_mqa_logits_topk", "sai_paged_mqa_logits_topk_workspace_bytes",
            "sai_error_string", "sai_version"} <= names


def test_every_declared_symbol_is_exported(lib):
    for name in sorted(_declared()):
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_no_driver_library_needed_at_load():
    # The driver library is reached at run time through the CUDA runtime's
    # entry-point query, so libsai loads on a host without a GPU driver.
    import shutil
    import subprocess

    if shutil.which("readelf") is None:
        pytest.skip("readelf not available")
    out = subprocess.run(["readelf", "-d", sai.library_path()], capture_output=True, text=True).stdout
    needed = re.findall(r"\(NEEDED\).*\[(.+?)\]", out)
    assert needed and not any(n.startswith("libcuda.so") or n.startswith("libcudart") for n in needed), needed


def test_error_strings(lib):
    for code in (0, -1, -2, -3, -4, -5):
        assert lib.sai_error_string(code)
    assert lib.sai_version() >= 100


A16, A4 = 0x10000, 0x20000          # fake device addresses, 16- and 4-byte aligned


def _logits(lib, **kw):
    args = dict(q=A16, kv=A16, num_pages=20, page_size=16, weights=A16, ctx=A4, bt=A4, bt_stride=20,
                batch=2, next_n=1, heads=64, head_dim=128, logits=A4, stride=512, W=512, layout=0,
                status=None)
    args.update(kw)
    return lib.sai_paged_mqa_logits(args["q"], args["kv"], args["num_pages"], args["page_size"],
                                    args["weights"], args["ctx"], args["bt"], args["bt_stride"],
                                    args["batch"], args["next_n"], args["heads"], args["head_dim"],
                                    args["logits"], args["stride"], args["W"], args["layout"],
                                    args["status"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(batch=-1), sai.ERR_INVALID_ARGUMENT),
    (dict(q=None), sai.ERR_INVALID_ARGUMENT),
    (dict(kv=None), sai.ERR_INVALID_ARGUMENT),
    (dict(weights=None), sai.ERR_INVALID_ARGUMENT),
    (dict(ctx=None), sai.ERR_INVALID_ARGUMENT),
    (dict(bt=None), sai.ERR_INVALID_ARGUMENT),
    (dict(logits=None), sai.ERR_INVALID_ARGUMENT),
    (dict(stride=511), sai.ERR_INVALID_ARGUMENT),
    (dict(W=0), sai.ERR_INVALID_ARGUMENT),
    (dict(num_pages=0), sai.ERR_INVALID_ARGUMENT),
    (dict(bt_stride=0), sai.ERR_INVALID_ARGUMENT),
    (dict(next_n=0), sai.ERR_INVALID_ARGUMENT),
    (dict(layout=7), sai.ERR_INVALID_ARGUMENT),
    (dict(num_pages=2**62), sai.ERR_INVALID_ARGUMENT),
    (dict(head_dim=64), sai.ERR_UNSUPPORTED),
    (dict(page_size=4), sai.ERR_UNSUPPORTED),
    (dict(page_size=512), sai.ERR_UNSUPPORTED),
    (dict(next_n=5), sai.ERR_UNSUPPORTED),
    (dict(heads=96), sai.ERR_UNSUPPORTED),
    (dict(q=A16 + 8), sai.ERR_MISALIGNED),
    (dict(kv=A16 + 4), sai.ERR_MISALIGNED),
    (dict(weights=A16 + 4), sai.ERR_MISALIGNED),
    (dict(logits=A4 + 2), sai.ERR_MISALIGNED),
    (dict(bt=A4 + 1), sai.ERR_MISALIGNED),
    (dict(status=A4 + 2), sai.ERR_MISALIGNED),
    (dict(batch=0), sai.OK),                   # nothing to do: no launch
])
def test_logits_argument_validation(lib, kw, code):
    assert _logits(lib, **kw) == code


def _topk(lib, **kw):
    args = dict(logits=A4, stride=512, ctx=A4, batch=2, next_n=1, W=512, k=64, idx=A4, idx_stride=64,
                ws=None, ws_bytes=0)
    args.update(kw)
    return lib.sai_top_k_per_row_decode(args["logits"], args["stride"], args["ctx"], args["batch"],
                                        args["next_n"], args["W"], args["k"], args["idx"],
                                        args["idx_stride"], args["ws"], args["ws_bytes"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(batch=-1), sai.ERR_INVALID_ARGUMENT),
    (dict(logits=None), sai.ERR_INVALID_ARGUMENT),
    (dict(ctx=None), sai.ERR_INVALID_ARGUMENT),
    (dict(idx=None), sai.ERR_INVALID_ARGUMENT),
    (dict(k=0), sai.ERR_INVALID_ARGUMENT),
    (dict(idx_stride=63), sai.ERR_INVALID_ARGUMENT),
    (dict(stride=100), sai.ERR_INVALID_ARGUMENT),
    (dict(next_n=0), sai.ERR_INVALID_ARGUMENT),
    (dict(k=70000, idx_stride=70000), sai.ERR_UNSUPPORTED),
    (dict(W=2**31, stride=2**31), sai.ERR_UNSUPPORTED),
    (dict(logits=A4 + 1), sai.ERR_MISALIGNED),
    (dict(idx=A4 + 2), sai.ERR_MISALIGNED),
    (dict(batch=0), sai.OK),
])
def test_topk_argument_validation(lib, kw, code):
    assert _topk(lib, **kw) == code


def _fused(lib, **kw):
    args = dict(q=A16, kv=A16, num_pages=20, page_size=16, weights=A16, ctx=A4, bt=A4, bt_stride=20,
                batch=2, next_n=1, heads=64, head_dim=128, logits=A4, stride=512, W=512, k=64, idx=A4,
                idx_stride=64, ws=A4, ws_bytes=4 * (5 * 2 + 4), status=None)
    args.update(kw)
    return lib.sai_paged_mqa_logits_topk(
        args["q"], args["kv"], args["num_pages"], args["page_size"], args["weights"], args["ctx"],
        args["bt"], args["bt_stride"], args["batch"], args["next_n"], args["heads"], args["head_dim"],
        args["logits"], args["stride"], args["W"], args["k"], args["idx"], args["idx_stride"],
        args["ws"], args["ws_bytes"], args["status"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(batch=-1), sai.ERR_INVALID_ARGUMENT),
    (dict(q=None), sai.ERR_INVALID_ARGUMENT),
    (dict(logits=None), sai.ERR_INVALID_ARGUMENT),
    (dict(idx=None), sai.ERR_INVALID_ARGUMENT),
    (dict(k=0), sai.ERR_INVALID_ARGUMENT),
    (dict(idx_stride=63), sai.ERR_INVALID_ARGUMENT),
    (dict(stride=511), sai.ERR_INVALID_ARGUMENT),
    (dict(k=70000, idx_stride=70000), sai.ERR_UNSUPPORTED),
    (dict(heads=96), sai.ERR_UNSUPPORTED),
    (dict(q=A16 + 8), sai.ERR_MISALIGNED),
    (dict(idx=A4 + 2), sai.ERR_MISALIGNED),
    (dict(ws=A4 + 1), sai.ERR_MISALIGNED),
    (dict(ws=None), sai.ERR_WORKSPACE),
    (dict(ws_bytes=4 * (5 * 2 + 4) - 1), sai.ERR_WORKSPACE),
    (dict(batch=0, ws=None, ws_bytes=0), sai.OK),
])
def test_fused_argument_validation(lib, kw, code):
    assert _fused(lib, **kw) == code


def _quant(lib, **kw):
    args = dict(k=A16, T=10, D=128, slots=A16, cache=A16, num_pages=4, P=16, layout=0, status=None)
    args.update(kw)
    return lib.sai_indexer_k_quant_insert(args["k"], args["T"], args["D"], args["slots"], args["cache"],
                                          args["num_pages"], args["P"], args["layout"], args["status"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(T=-1), sai.ERR_INVALID_ARGUMENT),
    (dict(k=None), sai.ERR_INVALID_ARGUMENT),
    (dict(slots=None), sai.ERR_INVALID_ARGUMENT),
    (dict(cache=None), sai.ERR_INVALID_ARGUMENT),
    (dict(num_pages=0), sai.ERR_INVALID_ARGUMENT),
    (dict(layout=3), sai.ERR_INVALID_ARGUMENT),
    (dict(D=64), sai.ERR_UNSUPPORTED),
    (dict(P=12), sai.ERR_UNSUPPORTED),
    (dict(k=A16 + 8), sai.ERR_MISALIGNED),
    (dict(slots=A16 + 4), sai.ERR_MISALIGNED),
    (dict(cache=A16 + 4), sai.ERR_MISALIGNED),
    (dict(T=0), sai.OK),
])
def test_kcache_argument_validation(lib, kw, code):
    assert _quant(lib, **kw) == code


def _gather(lib, **kw):
    args = dict(idx=A4, idx_stride=64, rows=2, k=64, next_n=1, bt=A4, bt_stride=8, P=16, pool=A16,
                num_pages=10, row_bytes=576, ids=A16, out=A16, status=None)
    args.update(kw)
    return lib.sai_gather_selected_kv(args["idx"], args["idx_stride"], args["rows"], args["k"], args["next_n"],
                                      args["bt"], args["bt_stride"], args["P"], args["pool"], args["num_pages"],
                                      args["row_bytes"], args["ids"], args["out"], args["status"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(rows=-1), sai.ERR_INVALID_ARGUMENT),
    (dict(k=0), sai.ERR_INVALID_ARGUMENT),
    (dict(idx_stride=63), sai.ERR_INVALID_ARGUMENT),
    (dict(idx=None), sai.ERR_INVALID_ARGUMENT),
    (dict(bt=None), sai.ERR_INVALID_ARGUMENT),
    (dict(ids=None, out=None), sai.ERR_INVALID_ARGUMENT),
    (dict(pool=None), sai.ERR_INVALID_ARGUMENT),
    (dict(row_bytes=100), sai.ERR_UNSUPPORTED),
    (dict(row_bytes=8192), sai.ERR_UNSUPPORTED),
    (dict(pool=A16 + 8), sai.ERR_MISALIGNED),
    (dict(out=A16 + 8), sai.ERR_MISALIGNED),
    (dict(ids=A16 + 4), sai.ERR_MISALIGNED),
    (dict(idx=A4 + 2), sai.ERR_MISALIGNED),
    (dict(rows=0), sai.OK),
])
def test_gather_argument_validation(lib, kw, code):
    assert _gather(lib, **kw) == code


def test_workspace_query(lib):
    n = lib.sai_top_k_workspace_bytes(1024, 32768, 2048)
    assert n >= 0
    assert lib.sai_top_k_workspace_bytes(-1, 10, 10) == 0
    # a tile counter per request, a queue of four rows per request, head, tail, done
    assert lib.sai_paged_mqa_logits_topk_workspace_bytes(1000) == 4 * (5 * 1000 + 4)
    assert lib.sai_paged_mqa_logits_topk_workspace_bytes(0) == 0
    assert lib.sai_paged_mqa_logits_topk_workspace_bytes(-1) == 0


def test_binding_refuses_cpu_tensors():
    import torch

    t = torch.zeros(4)
    with pytest.raises((ValueError, TypeError)):
        sai.top_k_per_row_decode(t.view(2, 2), torch.zeros(2, dtype=torch.int32), 1, 2, 1,
                                 torch.zeros(2, 1, dtype=torch.int32))


@pytest.mark.parametrize("mode,cycles,status,code", [
    (2, 1000, 0x1000, sai.ERR_INVALID_ARGUMENT),      # no such mode
    (-1, 1000, 0x1000, sai.ERR_INVALID_ARGUMENT),
    (0, 0, 0x1000, sai.ERR_INVALID_ARGUMENT),         # cycles out of 1 .. 2^31
    (1, (1 << 31) + 1, 0x1000, sai.ERR_INVALID_ARGUMENT),
    (0, 1000, None, sai.ERR_INVALID_ARGUMENT),        # status is required
    (0, 1000, 0x1002, sai.ERR_MISALIGNED),
])
def test_bounded_wait_selftest_argument_validation(lib, mode, cycles, status, code):
    assert lib.sai_selftest_bounded_wait(mode, cycles, status, None) == code
