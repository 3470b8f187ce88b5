"""Torch-facing helpers over the C ABI: a paged KV cache that owns its device
tensors, and the host page allocator.

PyTorch only allocates device memory and supplies the stream; every step of
append, scoring, selection and attention runs in libpkv's kernels.
"""
from __future__ import annotations

import ctypes
from typing import Dict, Optional, Tuple

import numpy as np
import torch

from . import binding as B

_TORCH_TO_PKV = {torch.float16: B.F16, torch.bfloat16: B.BF16, torch.float32: B.F32}
_NAME_TO_PKV = {"f16": B.F16, "bf16": B.BF16, "int8": B.I8, "u4": B.U4}
_PKV_TO_TORCH = {B.F16: torch.float16, B.BF16: torch.bfloat16, B.F32: torch.float32, B.I8: torch.uint8,
                 B.U4: torch.uint8}   # I8 pools hold the bytes u = code + 128
_QUANT = {"none": B.QUANT_NONE, "per_token": B.QUANT_PER_TOKEN, "per_group64": B.QUANT_PER_GROUP64}


def pkv_dtype(t: torch.Tensor) -> int:
    try:
        return _TORCH_TO_PKV[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}") from None


def _ptr(t: Optional[torch.Tensor]) -> int:
    return 0 if t is None else t.data_ptr()


def _stream(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _need(t: torch.Tensor, name: str, dtype=None, device=None) -> None:
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device}")


class PagedKVCache:
    """One layer's paged K/V pools (see pkv_cache in include/pkv.h for layouts)."""

    def __init__(self, num_pages: int, page_size: int, num_kv_heads: int, head_dim: int,
                 kv_dtype: str = "bf16", quant: str = "none", with_meta: bool = False,
                 tail_rows: int = 0, device: str = "cuda", poison: bool = False):
        self.num_pages, self.page_size = num_pages, page_size
        self.num_kv_heads, self.head_dim = num_kv_heads, head_dim
        self.kv_dtype, self.quant = _NAME_TO_PKV[kv_dtype], _QUANT[quant]
        self.device = torch.device(device)
        tdt = _PKV_TO_TORCH[self.kv_dtype]
        # 4-bit codes: two per byte
        shape = (num_pages, num_kv_heads, page_size, head_dim // 2 if self.kv_dtype == B.U4 else head_dim)
        self.k_pages = torch.empty(shape, dtype=tdt, device=self.device)
        self.v_pages = torch.empty(shape, dtype=tdt, device=self.device)
        self.device = self.k_pages.device      # concrete index (cuda:N)
        self.kv_sz = None
        self.tail = None
        if self.kv_dtype in (B.I8, B.U4):
            gran = 1 if self.quant == B.QUANT_PER_TOKEN else 64
            self.kv_sz = torch.empty((num_pages, num_kv_heads, page_size // gran, 4),
                                     dtype=torch.float32, device=self.device)
            if self.quant == B.QUANT_PER_GROUP64:
                rows = max(1, tail_rows)
                self.tail = torch.zeros((rows, num_kv_heads, 2, 2, 64, head_dim),
                                        dtype=torch.float32, device=self.device)
        self.page_meta = (torch.empty((num_pages, num_kv_heads, 2, head_dim), dtype=torch.float32,
                                      device=self.device) if with_meta else None)
        if poison:
            # unwritten slots read as NaN (float) / NaN scales (INT8): a stray read shows
            if self.kv_dtype in (B.I8, B.U4):
                self.k_pages.fill_(0)
                self.v_pages.fill_(0)
                self.kv_sz.fill_(float("nan"))
            else:
                self.k_pages.fill_(float("nan"))
                self.v_pages.fill_(float("nan"))
            if self.page_meta is not None:
                self.page_meta.fill_(float("nan"))
        self._desc = B.PkvCache(
            num_pages, page_size, num_kv_heads, head_dim, self.kv_dtype, self.quant,
            self.k_pages.data_ptr(), self.v_pages.data_ptr(), _ptr(self.kv_sz), _ptr(self.tail),
            0 if self.tail is None else self.tail.shape[0], _ptr(self.page_meta))
        self._ws: Dict[Tuple, torch.Tensor] = {}

    def descriptor(self) -> B.PkvCache:
        return self._desc

    # ------------------------------------------------------------------ append
    def append(self, k_new: torch.Tensor, v_new: torch.Tensor, block_table: torch.Tensor,
               positions: torch.Tensor, new_lens: Optional[torch.Tensor] = None,
               dev_status: Optional[torch.Tensor] = None,
               stream: Optional[torch.cuda.Stream] = None) -> None:
        """Write tokens k_new/v_new [B][T][Hkv][d] at positions[b] .. (+new_lens[b])."""
        for t, n in ((k_new, "k_new"), (v_new, "v_new")):
            _need(t, n, device=self.device)
        _need(block_table, "block_table", torch.int32, self.device)
        _need(positions, "positions", torch.int32, self.device)
        if new_lens is not None:
            _need(new_lens, "new_lens", torch.int32, self.device)
        Bsz, T = k_new.shape[0], k_new.shape[1]
        B.kv_append(self._desc, Bsz, T, k_new.data_ptr(), v_new.data_ptr(), pkv_dtype(k_new),
                    block_table.data_ptr(), block_table.shape[1], positions.data_ptr(),
                    _ptr(new_lens), _ptr(dev_status), _stream(stream))

    # ----------------------------------------------------------- score / top-K
    def score_topk(self, q: torch.Tensor, block_table: torch.Tensor, seq_lens: torch.Tensor,
                   top_k: int, want_scores: bool = False, dev_status: Optional[torch.Tensor] = None,
                   sel: Optional[torch.Tensor] = None, count: Optional[torch.Tensor] = None,
                   scores: Optional[torch.Tensor] = None,
                   stream: Optional[torch.cuda.Stream] = None, group_mode: int = 0,
                   early_start: bool = False):
        """Top-K pages per row: per (sequence, query head), or with group_mode 1 / 2
        (sum / max of the group's scores) per (sequence, kv head). Returns
        (sel [B][R][K], count [B][R], scores [B][R][max_pages] or None).

        early_start: the kernel launched just before on the stream writes nothing
        this call reads (q, tables, lengths, boxes), so the scoring starts under it."""
        _need(q, "q", device=self.device)
        Bsz, Hq = q.shape[0], q.shape[1]
        R = Hq if group_mode == 0 else self.num_kv_heads
        mp = block_table.shape[1]
        if sel is None:
            sel = torch.empty((Bsz, R, top_k), dtype=torch.int32, device=self.device)
        if count is None:
            count = torch.empty((Bsz, R), dtype=torch.int32, device=self.device)
        if want_scores and scores is None:
            scores = torch.empty((Bsz, R, mp), dtype=torch.float32, device=self.device)
        B.page_score_topk(self._desc, Bsz, Hq, q.data_ptr(), pkv_dtype(q), block_table.data_ptr(),
                          mp, seq_lens.data_ptr(), top_k, sel.data_ptr(), count.data_ptr(),
                          _ptr(scores), _ptr(dev_status), _stream(stream), group_mode=group_mode,
                          early_start=1 if early_start else 0)
        return sel, count, scores

    # --------------------------------------------------------------- attention
    def workspace(self, batch: int, num_q_heads: int, sparse: int, num_splits: int) -> torch.Tensor:
        """Zero-filled workspace of at least the size the library asks for (kept and reused).
        sparse: 0 dense, 1 page lists per query head, 2 lists shared by each group."""
        key = (batch, num_q_heads, int(sparse), num_splits)
        n = B.attention_workspace_bytes(self._desc, batch, num_q_heads, sparse, num_splits)
        ws = self._ws.get(key)
        if ws is None or ws.numel() < n:
            ws = torch.zeros(n, dtype=torch.uint8, device=self.device)
            self._ws[key] = ws
        return ws

    def attention(self, q: torch.Tensor, block_table: torch.Tensor, seq_lens: torch.Tensor,
                  sm_scale: Optional[float] = None, sel: Optional[torch.Tensor] = None,
                  sel_count: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                  out_dtype: torch.dtype = torch.float32, num_splits: int = 0,
                  dev_status: Optional[torch.Tensor] = None,
                  stream: Optional[torch.cuda.Stream] = None, fresh_rows: int = -1,
                  sel_shared: bool = False) -> torch.Tensor:
        """Decode attention for q [B][Hq][d]; dense, or over sel[b][h][:sel_count[b][h]] pages.

        fresh_rows >= 0 lets the call start while the kernel launched just before
        it on the stream still runs, on the promise that, of this call's inputs,
        that kernel writes only the K/V rows of the last fresh_rows tokens of each
        sequence (e.g. the kv_append of this step, fresh_rows = its token count;
        0 after another attention call)."""
        _need(q, "q", device=self.device)
        _need(block_table, "block_table", torch.int32, self.device)
        _need(seq_lens, "seq_lens", torch.int32, self.device)
        Bsz, Hq, d = q.shape
        if sm_scale is None:
            sm_scale = 1.0 / float(np.sqrt(d))
        if out is None:
            out = torch.empty((Bsz, Hq, d), dtype=out_dtype, device=self.device)
        sparse = sel is not None
        mode = 0 if not sparse else (2 if sel_shared else 1)
        ws = self.workspace(Bsz, Hq, mode, num_splits)
        B.paged_decode_attention(
            self._desc, Bsz, Hq, q.data_ptr(), pkv_dtype(q), float(sm_scale),
            block_table.data_ptr(), block_table.shape[1], seq_lens.data_ptr(), _ptr(sel),
            _ptr(sel_count), sel.shape[2] if sparse else 0, out.data_ptr(), pkv_dtype(out),
            num_splits, ws.data_ptr(), ws.numel(), _ptr(dev_status), _stream(stream),
            fresh_rows=fresh_rows, sel_shared=1 if (sparse and sel_shared) else 0)
        return out

    def append_attention(self, k_new: torch.Tensor, v_new: torch.Tensor, q: torch.Tensor,
                         block_table: torch.Tensor, seq_lens: torch.Tensor, sm_scale: Optional[float] = None,
                         out: Optional[torch.Tensor] = None, out_dtype: torch.dtype = torch.float32,
                         num_splits: int = 0, dev_status: Optional[torch.Tensor] = None,
                         stream: Optional[torch.cuda.Stream] = None, fresh_rows: int = -1) -> torch.Tensor:
        """One decode step: write k_new / v_new [B][Hkv][d] (each sequence's token at
        position seq_lens[b] - 1) and attend over [0, seq_lens[b]), in one call."""
        _need(q, "q", device=self.device)
        _need(k_new, "k_new", device=self.device)
        _need(v_new, "v_new", device=self.device)
        _need(block_table, "block_table", torch.int32, self.device)
        _need(seq_lens, "seq_lens", torch.int32, self.device)
        Bsz, Hq, d = q.shape
        if sm_scale is None:
            sm_scale = 1.0 / float(np.sqrt(d))
        if out is None:
            out = torch.empty((Bsz, Hq, d), dtype=out_dtype, device=self.device)
        ws = self.workspace(Bsz, Hq, 0, num_splits)
        src = B.BF16 if k_new.dtype == torch.bfloat16 else B.F16
        B.append_decode_attention(
            self._desc, Bsz, Hq, k_new.data_ptr(), v_new.data_ptr(), src, q.data_ptr(), pkv_dtype(q),
            float(sm_scale), block_table.data_ptr(), block_table.shape[1], seq_lens.data_ptr(),
            out.data_ptr(), pkv_dtype(out), num_splits, fresh_rows, ws.data_ptr(), ws.numel(),
            _ptr(dev_status), _stream(stream))
        return out


class PageAllocator:
    """Host free-list page allocator of libpkv (pkv_alloc_*)."""

    def __init__(self, num_pages: int):
        self._h = B.alloc_create(num_pages)
        self.num_pages = num_pages

    def reserve(self, seq_id: int, total_tokens: int, page_size: int, max_pages: int) -> np.ndarray:
        row = np.full(max_pages, -1, dtype=np.int32)
        B.alloc_reserve(self._h, seq_id, total_tokens, page_size,
                        row.ctypes.data_as(ctypes.c_void_p).value, max_pages)
        return row

    def free(self, seq_id: int) -> None:
        B.alloc_free(self._h, seq_id)

    @property
    def num_free(self) -> int:
        return B.alloc_num_free(self._h)

    def seq_pages(self, seq_id: int) -> int:
        return B.alloc_seq_pages(self._h, seq_id)

    def check(self) -> int:
        return B.alloc_check(self._h)

    def close(self) -> None:
        if self._h:
            B.alloc_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
