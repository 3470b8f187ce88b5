"""GB300 (sm_103a) paged KV-cache decode attention.

The compute lives in libpkv.so (include/pkv.h): kv_append, page_score_topk and
paged_decode_attention as hand-written CUDA kernels. `binding` marshals
arguments to the C ABI; `cache` wraps device tensors for PyTorch users.
"""
from . import binding  # noqa: F401

__all__ = ["binding", "build", "PagedKVCache", "PageAllocator"]


def build(verbose: bool = False, force: bool = False) -> str:
    from ._build import build as _b
    return _b(verbose=verbose, force=force)


def __getattr__(name):
    if name in ("PagedKVCache", "PageAllocator"):
        from . import cache
        return getattr(cache, name)
    raise AttributeError(name)
