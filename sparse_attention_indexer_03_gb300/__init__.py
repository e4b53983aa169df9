"""Python binding of libsai, the GB300 sparse-attention indexer decode path.

Thin ctypes marshalling over the C ABI declared in `include/sai.h`: each
function checks tensor devices and dtypes, then passes raw device pointers,
sizes and the current CUDA stream to the library.  Every step of the
computation runs in the library's CUDA kernels; there is no fallback.  If
`libsai.so` has not been built, calls raise `LibraryNotBuilt`.

    paged_mqa_logits(q, kv_cache, page_size, weights, context_lens, block_table,
                     logits, max_model_len, ...)
    top_k_per_row_decode(logits, context_lens, next_n, max_model_len, k, indices, ...)
    paged_mqa_logits_topk(q, kv_cache, page_size, weights, context_lens, block_table,
                          logits, max_model_len, k, indices, workspace, ...)
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

from . import _build

__all__ = [
    "LibraryNotBuilt", "SaiError", "build", "library", "library_path",
    "paged_mqa_logits", "top_k_workspace_bytes", "top_k_per_row_decode",
    "logits_topk_workspace_bytes", "paged_mqa_logits_topk", "paged_mqa_logits_topk_static",
    "paged_mqa_logits_topk_static_reset",
    "indexer_k_quant_insert", "gather_selected_kv",
    "STATUS_BAD_PAGE", "STATUS_CTX_CLAMPED", "STATUS_TIMEOUT",
    "KV_PAGE_SPLIT", "KV_INTERLEAVED",
]

OK = 0
ERR_INVALID_ARGUMENT = -1
ERR_UNSUPPORTED = -2
ERR_MISALIGNED = -3
ERR_WORKSPACE = -4
ERR_CUDA = -5

STATUS_BAD_PAGE = 0x1
STATUS_CTX_CLAMPED = 0x2
STATUS_TIMEOUT = 0x4

KV_PAGE_SPLIT = 0
KV_INTERLEAVED = 1
_LAYOUTS = {"split": KV_PAGE_SPLIT, "interleaved": KV_INTERLEAVED,
            KV_PAGE_SPLIT: KV_PAGE_SPLIT, KV_INTERLEAVED: KV_INTERLEAVED}


class LibraryNotBuilt(RuntimeError):
    pass


class SaiError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {error_string(code)} ({code})")


_lib = None

_c = ctypes
_P = _c.c_void_p
_SIGS = {
    "sai_paged_mqa_logits": (_c.c_int, [_P, _P, _c.c_int64, _c.c_int32, _P, _P, _P, _c.c_int64,
                                        _c.c_int32, _c.c_int32, _c.c_int32, _c.c_int32,
                                        _P, _c.c_int64, _c.c_int64, _c.c_int32, _P, _P]),
    "sai_top_k_workspace_bytes": (_c.c_size_t, [_c.c_int32, _c.c_int64, _c.c_int32]),
    "sai_top_k_per_row_decode": (_c.c_int, [_P, _c.c_int64, _P, _c.c_int32, _c.c_int32, _c.c_int64,
                                            _c.c_int32, _P, _c.c_int64, _P, _c.c_size_t, _P]),
    "sai_paged_mqa_logits_topk_workspace_bytes": (_c.c_size_t, [_c.c_int32]),
    "sai_paged_mqa_logits_topk": (_c.c_int, [_P, _P, _c.c_int64, _c.c_int32, _P, _P, _P, _c.c_int64,
                                             _c.c_int32, _c.c_int32, _c.c_int32, _c.c_int32,
                                             _P, _c.c_int64, _c.c_int64, _c.c_int32, _P, _c.c_int64,
                                             _P, _c.c_size_t, _P, _P]),
    "sai_paged_mqa_logits_topk_static": (_c.c_int, [_P, _P, _c.c_int64, _c.c_int32, _P, _P, _P, _c.c_int64,
                                                    _c.c_int32, _c.c_int32, _c.c_int32, _c.c_int32,
                                                    _P, _c.c_int64, _c.c_int64, _c.c_int32, _P, _c.c_int64,
                                                    _P, _P]),
    "sai_paged_mqa_logits_topk_static_reset": (_c.c_int, [_P]),
    "sai_indexer_k_quant_insert": (_c.c_int, [_P, _c.c_int64, _c.c_int32, _P, _P, _c.c_int64, _c.c_int32,
                                              _c.c_int32, _P, _P]),
    "sai_gather_selected_kv": (_c.c_int, [_P, _c.c_int64, _c.c_int32, _c.c_int32, _c.c_int32, _P, _c.c_int64,
                                          _c.c_int32, _P, _c.c_int64, _c.c_int32, _P, _P, _P, _P]),
    "sai_selftest_bounded_wait": (_c.c_int, [_c.c_int32, _c.c_int64, _P, _P]),
    "sai_error_string": (_c.c_char_p, [_c.c_int]),
    "sai_version": (_c.c_int, []),
}


def library_path() -> str:
    return _build.LIB


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libsai.so for sm_103a (in-tree) and load it."""
    global _lib
    path = _build.build(force=force, verbose=verbose)
    _lib = None
    library()
    return path


def library() -> ctypes.CDLL:
    """The loaded libsai (raises LibraryNotBuilt if it is missing)."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise LibraryNotBuilt(f"{path} is missing: build it with "
                                  "sparse_attention_indexer_03_gb300.build()")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def error_string(code: int) -> str:
    try:
        return library().sai_error_string(code).decode()
    except LibraryNotBuilt:
        return f"code {code}"


def _stream_handle(stream) -> Optional[int]:
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t, dtype, name):
    import torch

    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name}: dtype {t.dtype} not accepted")
    return t.data_ptr()


def _logits_args(q, kv_cache, page_size, weights, context_lens, block_table, logits, max_model_len,
                 num_pages):
    """Marshalled arguments shared by the logits entry points, up to max_model_len."""
    import torch

    u8 = (torch.uint8, torch.float8_e4m3fn)
    if q.dim() != 4 or not q.is_contiguous():
        raise ValueError("q must be a contiguous [B, next_n, H, D] tensor")
    B, next_n, H, D = q.shape
    if not kv_cache.is_contiguous() or not weights.is_contiguous():
        raise ValueError("kv_cache and weights must be contiguous")
    if block_table.dim() != 2 or block_table.stride(1) != 1:
        raise ValueError("block_table must be [B, stride] with unit inner stride")
    if logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be [rows, stride] with unit inner stride")
    page_bytes = page_size * (D + 4)
    if num_pages is None:
        num_pages = kv_cache.numel() * kv_cache.element_size() // page_bytes
    return (_ptr(q, u8, "q"), _ptr(kv_cache, u8, "kv_cache"), int(num_pages), int(page_size),
            _ptr(weights, torch.float32, "weights"), _ptr(context_lens, torch.int32, "context_lens"),
            _ptr(block_table, torch.int32, "block_table"), int(block_table.stride(0)),
            int(B), int(next_n), int(H), int(D),
            _ptr(logits, torch.float32, "logits"), int(logits.stride(0)), int(max_model_len))


def paged_mqa_logits(q, kv_cache, page_size: int, weights, context_lens, block_table,
                     logits, max_model_len: int, *, num_pages: Optional[int] = None,
                     status=None, kv_layout="split", stream=None) -> None:
    """FP8 paged MQA logits into `logits` (see `sai_paged_mqa_logits`).

    q            uint8 or float8_e4m3fn [B, next_n, H, 128], contiguous
    kv_cache     uint8 / float8 bytes of num_pages * page_size * 132 (any shape, contiguous)
    weights      float32 [B * next_n, H], contiguous
    context_lens int32 [B]
    block_table  int32 [B, stride] (row stride from the tensor; inner stride 1)
    logits       float32 [B * next_n, >= max_model_len] (row stride from the tensor)
    status       optional int32/uint32-sized CUDA tensor of one element
    """
    import torch

    args = _logits_args(q, kv_cache, page_size, weights, context_lens, block_table, logits,
                        max_model_len, num_pages)
    code = library().sai_paged_mqa_logits(
        *args, int(_LAYOUTS[kv_layout]), _ptr(status, (torch.int32, torch.uint32), "status"),
        _stream_handle(stream))
    if code != OK:
        raise SaiError(code, "sai_paged_mqa_logits")


def logits_topk_workspace_bytes(batch: int) -> int:
    return int(library().sai_paged_mqa_logits_topk_workspace_bytes(int(batch)))


def paged_mqa_logits_topk(q, kv_cache, page_size: int, weights, context_lens, block_table,
                          logits, max_model_len: int, k: int, indices, workspace, *,
                          num_pages: Optional[int] = None, status=None, stream=None) -> None:
    """Logits and per-row top-k in one launch (see `sai_paged_mqa_logits_topk`).

    Arguments as `paged_mqa_logits` (page-split caches only) plus
    indices    int32 [B * next_n, >= k] (row stride from the tensor)
    workspace  CUDA tensor of >= logits_topk_workspace_bytes(B) bytes (4 * (5 B + 4)),
               zero before the first call; every call leaves it zero again.
    """
    import torch

    if indices.dim() != 2 or indices.stride(1) != 1:
        raise ValueError("indices must be [rows, stride] with unit inner stride")
    args = _logits_args(q, kv_cache, page_size, weights, context_lens, block_table, logits,
                        max_model_len, num_pages)
    ws_bytes = workspace.numel() * workspace.element_size()
    code = library().sai_paged_mqa_logits_topk(
        *args, int(k), _ptr(indices, torch.int32, "indices"), int(indices.stride(0)),
        _ptr(workspace, None, "workspace"), int(ws_bytes),
        _ptr(status, (torch.int32, torch.uint32), "status"), _stream_handle(stream))
    if code != OK:
        raise SaiError(code, "sai_paged_mqa_logits_topk")


def paged_mqa_logits_topk_static(q, kv_cache, page_size: int, weights, context_lens, block_table,
                                 logits, max_model_len: int, k: int, indices, *,
                                 num_pages: Optional[int] = None, status=None, stream=None) -> None:
    """`paged_mqa_logits_topk` with the library's static counters instead of a
    workspace (see `sai_paged_mqa_logits_topk_static`: batch <= 16384, calls
    on one device must not overlap)."""
    import torch

    if indices.dim() != 2 or indices.stride(1) != 1:
        raise ValueError("indices must be [rows, stride] with unit inner stride")
    args = _logits_args(q, kv_cache, page_size, weights, context_lens, block_table, logits,
                        max_model_len, num_pages)
    code = library().sai_paged_mqa_logits_topk_static(
        *args, int(k), _ptr(indices, torch.int32, "indices"), int(indices.stride(0)),
        _ptr(status, (torch.int32, torch.uint32), "status"), _stream_handle(stream))
    if code != OK:
        raise SaiError(code, "sai_paged_mqa_logits_topk_static")


def paged_mqa_logits_topk_static_reset(stream=None) -> None:
    """Zero the static workspace of `paged_mqa_logits_topk_static` on the
    current device (after a call that raised STATUS_TIMEOUT)."""
    code = library().sai_paged_mqa_logits_topk_static_reset(_stream_handle(stream))
    if code != OK:
        raise SaiError(code, "sai_paged_mqa_logits_topk_static_reset")


def indexer_k_quant_insert(k, slot_mapping, kv_cache, page_size: int, *, num_pages: Optional[int] = None,
                           kv_layout="split", status=None, stream=None) -> None:
    """Quantise K rows to FP8 and write them into the paged cache (see
    `sai_indexer_k_quant_insert`).

    k             bfloat16 [T, 128], contiguous
    slot_mapping  int64 [T]: page * page_size + position; negative = skip
    kv_cache      uint8 / float8 bytes of num_pages * page_size * 132 (contiguous)
    """
    import torch

    if k.dim() != 2 or not k.is_contiguous() or k.dtype != torch.bfloat16:
        raise ValueError("k must be a contiguous bfloat16 [T, head_dim] tensor")
    if slot_mapping.dim() != 1 or slot_mapping.numel() != k.shape[0]:
        raise ValueError("slot_mapping must be [T]")
    if not kv_cache.is_contiguous():
        raise ValueError("kv_cache must be contiguous")
    T, D = k.shape
    if num_pages is None:
        num_pages = kv_cache.numel() * kv_cache.element_size() // (page_size * (D + 4))
    code = library().sai_indexer_k_quant_insert(
        _ptr(k, torch.bfloat16, "k"), int(T), int(D), _ptr(slot_mapping, torch.int64, "slot_mapping"),
        _ptr(kv_cache, (torch.uint8, torch.float8_e4m3fn), "kv_cache"), int(num_pages), int(page_size),
        int(_LAYOUTS[kv_layout]), _ptr(status, (torch.int32, torch.uint32), "status"), _stream_handle(stream))
    if code != OK:
        raise SaiError(code, "sai_indexer_k_quant_insert")


def gather_selected_kv(indices, next_n: int, block_table, page_size: int, kv_pool, row_bytes: int, *,
                       row_ids=None, out=None, num_pages: Optional[int] = None, status=None,
                       stream=None) -> None:
    """Gather the selected tokens' KV rows and/or their int64 row ids (see
    `sai_gather_selected_kv`).

    indices      int32 [rows, >= k] (row stride from the tensor); k = indices.shape[1]
    block_table  int32 [rows / next_n, stride] (inner stride 1)
    kv_pool      uint8 bytes of num_pages * page_size * row_bytes (contiguous)
    row_ids      optional int64 [rows, k], contiguous
    out          optional uint8 [rows, k, row_bytes], contiguous
    """
    import torch

    if indices.dim() != 2 or indices.stride(1) != 1:
        raise ValueError("indices must be [rows, k] with unit inner stride")
    if block_table.dim() != 2 or block_table.stride(1) != 1:
        raise ValueError("block_table must be [B, stride] with unit inner stride")
    rows, k = indices.shape
    if out is not None and (not out.is_contiguous() or out.numel() * out.element_size() < rows * k * row_bytes):
        raise ValueError("out must be a contiguous [rows, k, row_bytes] byte tensor")
    if row_ids is not None and (not row_ids.is_contiguous() or row_ids.numel() < rows * k):
        raise ValueError("row_ids must be a contiguous [rows, k] int64 tensor")
    if num_pages is None:
        num_pages = kv_pool.numel() * kv_pool.element_size() // (page_size * row_bytes)
    code = library().sai_gather_selected_kv(
        _ptr(indices, torch.int32, "indices"), int(indices.stride(0)), int(rows), int(k), int(next_n),
        _ptr(block_table, torch.int32, "block_table"), int(block_table.stride(0)), int(page_size),
        _ptr(kv_pool, None, "kv_pool"), int(num_pages), int(row_bytes),
        _ptr(row_ids, torch.int64, "row_ids"), _ptr(out, None, "out"),
        _ptr(status, (torch.int32, torch.uint32), "status"), _stream_handle(stream))
    if code != OK:
        raise SaiError(code, "sai_gather_selected_kv")


def selftest_bounded_wait(mode: int, cycles: int, status, *, stream=None) -> None:
    """Run the bounded-wait self-test (see `sai_selftest_bounded_wait`):
    mode 0 lets the budget of `cycles` run out, mode 1 raises the abort flag
    after `cycles`; either way SAI_STATUS_TIMEOUT is OR-ed into `status`."""
    import torch

    code = library().sai_selftest_bounded_wait(int(mode), int(cycles), _ptr(status, torch.int32, "status"),
                                               _stream_handle(stream))
    if code != OK:
        raise SaiError(code, "sai_selftest_bounded_wait")


def top_k_workspace_bytes(rows: int, max_len: int, k: int) -> int:
    return int(library().sai_top_k_workspace_bytes(int(rows), int(max_len), int(k)))


def top_k_per_row_decode(logits, context_lens, next_n: int, max_model_len: int, k: int,
                         indices, *, workspace=None, stream=None) -> None:
    """Per-row top-k column indices into `indices` (see `sai_top_k_per_row_decode`).

    logits   float32 [B * next_n, >= max_model_len] (row stride from the tensor)
    indices  int32 [B * next_n, >= k] (row stride from the tensor)
    """
    import torch

    if logits.stride(1) != 1 or indices.stride(1) != 1:
        raise ValueError("logits and indices need unit inner stride")
    B = context_lens.numel()
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size()
    code = library().sai_top_k_per_row_decode(
        _ptr(logits, torch.float32, "logits"), int(logits.stride(0)),
        _ptr(context_lens, torch.int32, "context_lens"), int(B), int(next_n), int(max_model_len), int(k),
        _ptr(indices, torch.int32, "indices"), int(indices.stride(0)), ws_ptr, int(ws_bytes),
        _stream_handle(stream))
    if code != OK:
        raise SaiError(code, "sai_top_k_per_row_decode")
