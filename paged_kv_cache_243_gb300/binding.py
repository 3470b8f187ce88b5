"""ctypes binding of libpkv (include/pkv.h): argument marshalling only.

Every function here has the name of the C entry point without its `pkv_`
prefix, takes plain integers for pointers (device addresses) and raises
PkvError on a non-OK status. No computation happens in Python: a missing or
unloadable library raises, there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_float, c_int, c_int32, c_int64, c_size_t, c_void_p
from typing import Optional

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libpkv.so")

# pkv_dtype / pkv_quant / status values of include/pkv.h
F16, BF16, F32, I8, U4 = 0, 1, 2, 3, 4
QUANT_NONE, QUANT_PER_TOKEN, QUANT_PER_GROUP64 = 0, 1, 2
SELECT_PER_HEAD, SELECT_GROUP_SUM, SELECT_GROUP_MAX = 0, 1, 2
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_OUT_OF_PAGES, ERR_CUDA, ERR_WORKSPACE = range(6)
DEV_BAD_PAGE, DEV_BAD_SELECTED, DEV_BAD_POSITION, DEV_TIMEOUT, DEV_BAD_CONFIG = 1, 2, 4, 8, 16

EXPORTED = [
    "pkv_status_string", "pkv_abi_version", "pkv_tuning_reload", "pkv_kv_append", "pkv_page_score_topk",
    "pkv_attention_workspace_bytes", "pkv_paged_decode_attention", "pkv_append_decode_attention",
    "pkv_paged_decode_attention_noalloc",
    "pkv_alloc_create", "pkv_alloc_destroy", "pkv_alloc_reserve", "pkv_alloc_free",
    "pkv_alloc_num_free", "pkv_alloc_seq_pages", "pkv_alloc_check",
]


class PkvError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = status_string(status) if _lib is not None else str(status)
        super().__init__(f"{where}: {msg} (status {status})")


class PkvCache(ctypes.Structure):
    """Mirror of the C struct pkv_cache."""
    _fields_ = [
        ("num_pages", c_int32), ("page_size", c_int32), ("num_kv_heads", c_int32),
        ("head_dim", c_int32), ("kv_dtype", c_int), ("quant", c_int),
        ("k_pages", c_void_p), ("v_pages", c_void_p), ("kv_sz", c_void_p),
        ("tail", c_void_p), ("tail_rows", c_int32), ("page_meta", c_void_p),
    ]


_lib: Optional[ctypes.CDLL] = None


def library_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """Load libpkv.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"libpkv.so not built at {_LIB_PATH}; run __graft_entry__.build()")
    L = ctypes.CDLL(_LIB_PATH)
    P = POINTER(PkvCache)
    vp, i32, i64 = c_void_p, c_int32, c_int64
    sig = {
        "pkv_status_string": (ctypes.c_char_p, [c_int]),
        "pkv_abi_version": (i32, []),
        "pkv_tuning_reload": (None, []),
        "pkv_kv_append": (c_int, [P, i32, i32, vp, vp, c_int, vp, i32, vp, vp, vp, vp]),
        "pkv_page_score_topk": (c_int, [P, i32, i32, vp, c_int, vp, i32, vp, i32, i32, i32, vp, vp, vp, vp, vp]),
        "pkv_attention_workspace_bytes": (c_size_t, [P, i32, i32, i32, i32]),
        "pkv_paged_decode_attention": (c_int, [P, i32, i32, vp, c_int, c_float, vp, i32, vp, vp, vp,
                                               i32, i32, vp, c_int, i32, i32, vp, c_size_t, vp, vp]),
        "pkv_append_decode_attention": (c_int, [P, i32, i32, vp, vp, c_int, vp, c_int, c_float, vp, i32, vp,
                                                vp, c_int, i32, i32, vp, c_size_t, vp, vp]),
        "pkv_paged_decode_attention_noalloc": (c_int, [P, i32, i32, vp, c_int, c_float, vp, i32, vp, vp,
                                                       vp, i32, i32, vp, c_int, i32, vp, vp]),
        "pkv_alloc_create": (c_int, [i32, POINTER(c_void_p)]),
        "pkv_alloc_destroy": (None, [vp]),
        "pkv_alloc_reserve": (c_int, [vp, i64, i32, i32, vp, i32]),
        "pkv_alloc_free": (c_int, [vp, i64]),
        "pkv_alloc_num_free": (i32, [vp]),
        "pkv_alloc_seq_pages": (i32, [vp, i64]),
        "pkv_alloc_check": (i32, [vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def _check(status: int, where: str) -> None:
    if status != OK:
        raise PkvError(status, where)


def status_string(status: int) -> str:
    return lib().pkv_status_string(status).decode()


def abi_version() -> int:
    return lib().pkv_abi_version()


def tuning_reload() -> None:
    """Re-read the PKV_ATTN_* tuning variables from the environment."""
    lib().pkv_tuning_reload()


def kv_append(cache: PkvCache, batch: int, t_new: int, k_new: int, v_new: int, src_dtype: int,
              block_table: int, max_pages: int, positions: int, new_lens: int, dev_status: int,
              stream: int) -> None:
    _check(lib().pkv_kv_append(ctypes.byref(cache), batch, t_new, k_new, v_new, src_dtype,
                               block_table, max_pages, positions, new_lens or None,
                               dev_status or None, stream or None), "kv_append")


def page_score_topk(cache: PkvCache, batch: int, num_q_heads: int, q: int, q_dtype: int,
                    block_table: int, max_pages: int, seq_lens: int, top_k: int, sel_pages: int,
                    sel_count: int, scores_out: int, dev_status: int, stream: int,
                    group_mode: int = SELECT_PER_HEAD, early_start: int = 0) -> None:
    """group_mode and early_start come last here (keywords) and go after top_k in
    the C call."""
    _check(lib().pkv_page_score_topk(ctypes.byref(cache), batch, num_q_heads, q, q_dtype,
                                     block_table, max_pages, seq_lens, top_k, group_mode, early_start,
                                     sel_pages, sel_count, scores_out or None, dev_status or None,
                                     stream or None),
           "page_score_topk")


def attention_workspace_bytes(cache: PkvCache, batch: int, num_q_heads: int, sparse: int,
                              num_splits: int) -> int:
    """sparse: 0 dense, 1 page lists per query head, 2 lists shared by each group."""
    n = lib().pkv_attention_workspace_bytes(ctypes.byref(cache), batch, num_q_heads, int(sparse),
                                            num_splits)
    if n == 0:
        raise PkvError(ERR_INVALID_ARG, "attention_workspace_bytes")
    return n


def paged_decode_attention(cache: PkvCache, batch: int, num_q_heads: int, q: int, q_dtype: int,
                           sm_scale: float, block_table: int, max_pages: int, seq_lens: int,
                           sel_pages: int, sel_count: int, sel_stride: int, out: int,
                           out_dtype: int, num_splits: int, workspace: int, workspace_bytes: int,
                           dev_status: int, stream: int, fresh_rows: int = -1,
                           sel_shared: int = 0) -> None:
    """fresh_rows and sel_shared come last here (keywords; defaults: no early
    start, page lists per query head) and go to their places in the C call."""
    _check(lib().pkv_paged_decode_attention(ctypes.byref(cache), batch, num_q_heads, q, q_dtype,
                                            sm_scale, block_table, max_pages, seq_lens,
                                            sel_pages or None, sel_count or None, sel_stride,
                                            sel_shared, out, out_dtype, num_splits, fresh_rows, workspace,
                                            workspace_bytes, dev_status or None, stream or None),
           "paged_decode_attention")


def append_decode_attention(cache: PkvCache, batch: int, num_q_heads: int, k_new: int, v_new: int,
                            src_dtype: int, q: int, q_dtype: int, sm_scale: float, block_table: int,
                            max_pages: int, seq_lens: int, out: int, out_dtype: int, num_splits: int,
                            fresh_rows: int, workspace: int, workspace_bytes: int, dev_status: int,
                            stream: int) -> None:
    _check(lib().pkv_append_decode_attention(ctypes.byref(cache), batch, num_q_heads, k_new, v_new,
                                             src_dtype, q, q_dtype, sm_scale, block_table, max_pages,
                                             seq_lens, out, out_dtype, num_splits, fresh_rows, workspace,
                                             workspace_bytes, dev_status or None, stream or None),
           "append_decode_attention")


def paged_decode_attention_noalloc(cache: PkvCache, batch: int, num_q_heads: int, q: int,
                                   q_dtype: int, sm_scale: float, block_table: int, max_pages: int,
                                   seq_lens: int, sel_pages: int, sel_count: int, sel_stride: int,
                                   out: int, out_dtype: int, num_splits: int, dev_status: int,
                                   stream: int, sel_shared: int = 0) -> None:
    """paged_decode_attention with the library's fixed device scratch instead of a
    caller workspace (for callers that cannot allocate device memory)."""
    _check(lib().pkv_paged_decode_attention_noalloc(
        ctypes.byref(cache), batch, num_q_heads, q, q_dtype, sm_scale, block_table, max_pages,
        seq_lens, sel_pages or None, sel_count or None, sel_stride, sel_shared, out, out_dtype,
        num_splits, dev_status or None, stream or None), "paged_decode_attention_noalloc")


def alloc_create(num_pages: int) -> int:
    h = c_void_p()
    _check(lib().pkv_alloc_create(num_pages, ctypes.byref(h)), "alloc_create")
    return h.value


def alloc_destroy(h: int) -> None:
    lib().pkv_alloc_destroy(h)


def alloc_reserve(h: int, seq_id: int, total_tokens: int, page_size: int, row_ptr: int,
                  max_pages: int) -> None:
    _check(lib().pkv_alloc_reserve(h, seq_id, total_tokens, page_size, row_ptr, max_pages),
           "alloc_reserve")


def alloc_free(h: int, seq_id: int) -> None:
    _check(lib().pkv_alloc_free(h, seq_id), "alloc_free")


def alloc_num_free(h: int) -> int:
    return lib().pkv_alloc_num_free(h)


def alloc_seq_pages(h: int, seq_id: int) -> int:
    return lib().pkv_alloc_seq_pages(h, seq_id)


def alloc_check(h: int) -> int:
    return lib().pkv_alloc_check(h)
