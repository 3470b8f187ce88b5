"""Plain, slow fp64 CPU oracle for paged decode attention.

TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check of the entry module
and the benchmark's CPU-baseline / reference legs may import, call or run
anything here. The product package never imports it, and this package never
imports the product package: the two share no code. Inputs come from the
seeded generators in `synth`, which hold none of the method's arithmetic.

Sources, cited by short name and section:
  [Gemini page]      "GPU显存占用直降63%！Gemini KV Cache优化实战：FlashAttention-3适配全链路拆解"
                     (uyd888.cn/news/1049062)
  [KV-practice page] "LLM推理中的KV Cache优化与显存管理实践"
                     (intelliparadigm.com/article/weixin_31062533/2042388)
  [HBM-layout page]  "Transformer 推理的内存布局优化：从 HBM 带宽利用率的视角重新设计 KV Cache"
                     (pzsr.cn/news/13006)
  [TinyServe page]   "LLM推理中的KV缓存优化技术与TinyServe实践" (lpnh.cn/news/810111)

Every function is pinned by a `-m "not gpu"` test against something other
than itself (closed forms, brute force, invariants the pages state, worked
figures printed on the pages); see tests/test_oracle_*.py.
"""
from .quant import (  # noqa: F401
    quantize_block, quantize_rows, dequantize, dequant_f32_two_step,
    quantize_per_token, quantize_per_group, GroupAppendModel,
)
from .attention import (  # noqa: F401
    decode_attention, decode_attention_tokens, sparse_decode_attention,
    split_partials, combine_partials,
)
from .sparse import (  # noqa: F401
    page_bounding_boxes, page_scores, group_page_scores, select_top_k, top_k_count,
)
from .quant4 import (  # noqa: F401
    quantize_block_u4, quantize_rows_u4, quantize_per_token_u4, pack_u4, unpack_u4, dequantize_u4,
    per_token_u4_dequant, per_token_u4_bbox_values,
)
from .sizes import kv_cache_bytes, blocks_needed  # noqa: F401
