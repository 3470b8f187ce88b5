"""The C-ABI library without a GPU: it builds, loads, exports every declared
symbol, rejects bad arguments before touching CUDA, and its host page
allocator follows the pages' rules."""
import json
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def B():
    from paged_kv_cache_243_gb300 import _build, binding
    _build.build()
    binding.lib()
    return binding


def declared_functions():
    src = open(os.path.join(ROOT, "include", "pkv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(B):
    names = declared_functions()
    assert len(names) >= 13
    L = B.lib()
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(B.EXPORTED)


def test_status_strings_and_version(B):
    src = open(os.path.join(ROOT, "include", "pkv.h")).read()
    assert B.abi_version() == int(re.search(r"#define PKV_ABI_VERSION (\d+)", src).group(1))
    assert B.status_string(B.OK) == "ok"
    assert B.status_string(B.ERR_OUT_OF_PAGES) == "out of pages"


def _desc(B, **kw):
    d = dict(num_pages=8, page_size=16, num_kv_heads=2, head_dim=64, kv_dtype=B.F16,
             quant=B.QUANT_NONE, k_pages=0x1000, v_pages=0x2000, kv_sz=0, tail=0, tail_rows=0, page_meta=0)
    d.update(kw)
    return B.PkvCache(**d)


def test_argument_checks_before_cuda(B):
    # every case below must fail in the host checks (no CUDA call is reached)
    cases = [
        (_desc(B, head_dim=96), B.ERR_UNSUPPORTED),
        (_desc(B, page_size=24), B.ERR_UNSUPPORTED),
        (_desc(B, kv_dtype=B.I8, quant=B.QUANT_PER_GROUP64, kv_sz=0x3000, page_size=32), B.ERR_UNSUPPORTED),
        (_desc(B, kv_dtype=B.I8, quant=B.QUANT_PER_TOKEN, kv_sz=0), B.ERR_INVALID_ARG),
        (_desc(B, kv_dtype=B.F16, quant=B.QUANT_PER_TOKEN), B.ERR_INVALID_ARG),
        (_desc(B, kv_dtype=B.U4, quant=B.QUANT_PER_TOKEN, kv_sz=0), B.ERR_INVALID_ARG),
        (_desc(B, kv_dtype=B.U4, quant=B.QUANT_PER_GROUP64, kv_sz=0x3000, page_size=64), B.ERR_UNSUPPORTED),
        (_desc(B, kv_dtype=B.U4, quant=B.QUANT_NONE, kv_sz=0x3000), B.ERR_INVALID_ARG),
        (_desc(B, k_pages=0x1001), B.ERR_INVALID_ARG),
        (_desc(B, num_pages=0), B.ERR_INVALID_ARG),
    ]
    for desc, want in cases:
        with pytest.raises(B.PkvError) as e:
            B.paged_decode_attention(desc, 1, 2, 0x4000, B.F16, 0.125, 0x5000, 4, 0x6000, 0, 0, 0,
                                     0x7000, B.F32, 0, 0x8000, 1 << 20, 0, 0)
        assert e.value.status == want
    good = _desc(B)
    with pytest.raises(B.PkvError) as e:   # null q
        B.paged_decode_attention(good, 1, 2, 0, B.F16, 0.125, 0x5000, 4, 0x6000, 0, 0, 0,
                                 0x7000, B.F32, 0, 0x8000, 1 << 20, 0, 0)
    assert e.value.status == B.ERR_INVALID_ARG
    with pytest.raises(B.PkvError) as e:   # misaligned out
        B.paged_decode_attention(good, 1, 2, 0x4000, B.F16, 0.125, 0x5000, 4, 0x6000, 0, 0, 0,
                                 0x7004, B.F32, 0, 0x8000, 1 << 20, 0, 0)
    assert e.value.status == B.ERR_INVALID_ARG
    with pytest.raises(B.PkvError) as e:   # fresh_rows below -1
        B.paged_decode_attention(good, 1, 2, 0x4000, B.F16, 0.125, 0x5000, 4, 0x6000, 0, 0, 0,
                                 0x7000, B.F32, 0, 0x8000, 1 << 20, 0, 0, fresh_rows=-2)
    assert e.value.status == B.ERR_INVALID_ARG
    with pytest.raises(B.PkvError) as e:   # sparse without counts
        B.paged_decode_attention(good, 1, 2, 0x4000, B.F16, 0.125, 0x5000, 4, 0x6000, 0x9000, 0, 4,
                                 0x7000, B.F32, 0, 0x8000, 1 << 20, 0, 0)
    assert e.value.status == B.ERR_INVALID_ARG
    with pytest.raises(B.PkvError) as e:   # scoring needs page metadata
        B.page_score_topk(good, 1, 2, 0x4000, B.F16, 0x5000, 4, 0x6000, 2, 0x9000, 0xA000, 0, 0, 0)
    assert e.value.status == B.ERR_INVALID_ARG
    with_meta = _desc(B, page_meta=0xB000)
    with pytest.raises(B.PkvError) as e:   # unknown selection mode
        B.page_score_topk(with_meta, 1, 2, 0x4000, B.F16, 0x5000, 4, 0x6000, 2, 0x9000, 0xA000, 0, 0, 0,
                          group_mode=3)
    assert e.value.status == B.ERR_INVALID_ARG
    with pytest.raises(B.PkvError) as e:   # early_start must be 0 or 1
        B.page_score_topk(with_meta, 1, 2, 0x4000, B.F16, 0x5000, 4, 0x6000, 2, 0x9000, 0xA000, 0, 0, 0,
                          early_start=2)
    assert e.value.status == B.ERR_INVALID_ARG
    for desc, src, want in ((_desc(B, kv_dtype=B.I8, quant=B.QUANT_PER_GROUP64, kv_sz=0x3000,
                                   page_size=64), B.F16, B.ERR_INVALID_ARG),   # per-group without a tail
                            (_desc(B, page_meta=0xB000), B.I8, B.ERR_INVALID_ARG),   # boxes, bad source
                            (good, B.BF16, B.ERR_UNSUPPORTED),     # fp16 cache, bf16 source
                            (good, B.I8, B.ERR_INVALID_ARG)):
        with pytest.raises(B.PkvError) as e:   # one-call decode step: what it refuses
            B.append_decode_attention(desc, 1, 2, 0xC000, 0xD000, src, 0x4000, B.F16, 0.125, 0x5000, 4,
                                      0x6000, 0x7000, B.F32, 0, -1, 0x8000, 1 << 20, 0, 0)
        assert e.value.status == want
    with pytest.raises(B.PkvError) as e:   # sel_shared must be 0 or 1
        B.paged_decode_attention(good, 1, 2, 0x4000, B.F16, 0.125, 0x5000, 4, 0x6000, 0x9000, 0xA000, 4,
                                 0x7000, B.F32, 0, 0x8000, 1 << 20, 0, 0, sel_shared=2)
    assert e.value.status == B.ERR_INVALID_ARG
    with pytest.raises(B.PkvError) as e:   # per-group append without a tail
        B.kv_append(_desc(B, kv_dtype=B.I8, quant=B.QUANT_PER_GROUP64, kv_sz=0x3000, page_size=64),
                    1, 1, 0x4000, 0x5000, B.F16, 0x6000, 4, 0x7000, 0, 0, 0)
    assert e.value.status == B.ERR_INVALID_ARG
    with pytest.raises(B.PkvError) as e:   # bad source dtype
        B.kv_append(good, 1, 1, 0x4000, 0x5000, B.I8, 0x6000, 4, 0x7000, 0, 0, 0)
    assert e.value.status == B.ERR_INVALID_ARG
    # empty batches are no-ops
    B.kv_append(good, 0, 1, 0x4000, 0x5000, B.F16, 0x6000, 4, 0x7000, 0, 0, 0)
    B.paged_decode_attention(good, 0, 2, 0x4000, B.F16, 0.125, 0x5000, 4, 0x6000, 0, 0, 0,
                             0x7000, B.F32, 0, 0x8000, 1 << 20, 0, 0)


def test_allocator_rules(B):
    from paged_kv_cache_243_gb300.cache import PageAllocator
    a = PageAllocator(10)
    # ceil(33 / 16) = 3 pages, taken from the front of the free list
    assert a.reserve(7, 33, 16, 4).tolist() == [0, 1, 2, -1]
    assert a.num_free == 7 and a.seq_pages(7) == 3
    # growing only takes the missing pages
    assert a.reserve(7, 64, 16, 4).tolist() == [0, 1, 2, 3]
    assert a.reserve(8, 80, 16, 8).tolist() == [4, 5, 6, 7, 8, -1, -1, -1]
    # a request the free list cannot meet fails and changes nothing
    with pytest.raises(B.PkvError) as e:
        a.reserve(9, 33, 16, 4)
    assert e.value.status == B.ERR_OUT_OF_PAGES
    assert a.num_free == 1 and a.seq_pages(9) == 0 and a.check() == 0
    # more pages than the block-table row holds is an argument error
    with pytest.raises(B.PkvError) as e:
        a.reserve(10, 100, 16, 4)
    assert e.value.status == B.ERR_INVALID_ARG
    a.free(7)
    assert a.num_free == 5 and a.check() == 0
    assert a.reserve(9, 33, 16, 4).tolist() == [9, 0, 1, -1]
    with pytest.raises(B.PkvError):
        a.free(12345)
    a.free(8)
    a.free(9)
    assert a.num_free == 10 and a.check() == 0
    a.close()


def test_allocator_matches_alignment_table(B):
    # the pages' table: 127 and 511 tokens occupy 2048 KB and 8192 KB at 16 KB/token
    from paged_kv_cache_243_gb300.cache import PageAllocator
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "alignment_table.json")))
    for row in g["rows"]:
        a = PageAllocator(64)
        r = a.reserve(1, row["tokens"], 16, 64)
        pages = int((r >= 0).sum())
        assert pages * 16 * 16 == row["aligned_kb"]
        a.close()
