"""Plain, slow, obviously-correct CPU oracle for the paged KV cache hot path.

THIS PACKAGE IS TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline / reference legs of ``bench.py`` may import it.  The product
path (the CUDA library and its Python binding) never imports, links or calls it,
and it never imports the product path: the two share no code, headers, tables or
helpers.  The only thing both sides consume is the seeded input generator in
``workloads/``, which holds none of the method's arithmetic.

Everything is computed in float64 with numpy; stored cache elements are decoded
from their raw bits exactly (fp32 / fp16 / bf16 widen exactly, FP8 e4m3 is
decoded from its bit fields, NVFP4 from its E2M1 codes and E4M3 block scales).

Sources cited by key in the docstrings of this package:

[AGENTIC]  "宣稱省下 106 倍成本：vLLM 怎麼把 Serving 系統校準給 Agentic Workload"
           (datasciocean.com, ai-concept/vllm-agentic-serving).
[NOTES]    "大模型推理优化学习笔记" (fishingrodd.cn, 2026/10/30).
[LINEAGE]  "从静态批处理到状态化推理集群" (wineandchord.com,
           llm/landscape/lineages/inference-serving).
[DSV41]    vLLM x DeepSeek-V4.1-Flash agentic throughput write-up (yaoyouai.cn,
           news/405/vllm-deepseek-v41-flash-agentic-throughput-5x).
[ARCH]     summary of a vLLM V1 architecture deep-dive
           (ai.youdonthavefriends.com, llm/ai/deep-analysis/2026/08/08/vllm-architecture).

Parity status: every public function here is pinned by a ``-m "not gpu"`` test
in ``tests/test_oracle_pins.py`` against values the pages print, closed forms,
invariants, an independent library routine or brute force.  No function is
"parity unpinned".
"""

from .paged_attention import (  # noqa: F401
    DTYPE_BYTES,
    E2M1_MAX,
    E4M3_MAX,
    E5M2_MAX,
    attend,
    blocks_needed,
    bytes_per_block,
    copy_blocks,
    decode_bits,
    e2m1_encode,
    e2m1_table,
    e2m1_value,
    e4m3_encode,
    e4m3_value,
    e4m3_table,
    e5m2_encode,
    e5m2_table,
    e5m2_value,
    finalize_partial,
    gather_kv,
    kv_cache_bytes,
    merge_partials,
    NVFP4_GROUP,
    nvfp4_pack,
    nvfp4_quantize_row,
    nvfp4_rows,
    nvfp4_tile_bytes,
    paged_decode,
    paged_varlen,
    quantize_e4m3,
    quantize_e5m2,
    reshape_and_cache,
    softmax_partial,
    softmax_weights,
    query_positions,
)
