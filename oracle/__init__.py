"""CPU oracle for paged decode attention and its cache bookkeeping.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports, calls or links
this package: only the tests, the smoke check and the benchmark's CPU-baseline
and reference legs use it. It shares no code with the CUDA library (no common
helpers, tables or constants); the two meet only at the seeded inputs drawn by
the `synthetic` package.

It is deliberately plain and slow: fp64 arithmetic, whole-sequence gathers in
logical token order, and the textbook softmax with the maximum subtracted.

Sources (web pages on PagedAttention):
  * "Phase 7 · Document 04 — PagedAttention" (ai-engineer-zt0), §2 Core
    Concept (fixed-size blocks, shared physical pool, per-sequence block table,
    the C-style layout sketch, copy-on-write block sharing), §3 Mental Model
    (sharing picture), §11 Engineering Decision Framework and §13 question 4
    (capacity arithmetic).
  * The one-pool layout of `interleaved.py` (one record per physical block,
    K then V) is the layout sketch of Document 04 §2 taken literally.
  * The fp8 (E4M3) KV cache of `fp8.py` follows Document 04 §11/§12 (KV
    quantization as a way to fit more sequences); its format readings are in
    that module's docstring.
  * lux-666 notes "PagedAttention", sections 最小模型 (minimal model: logical
    blocks -> block table -> physical blocks, worked mapping 0->7, 1->2, 2->9),
    它为什么有效 (internal waste bounded by the last block; prefix sharing with
    copy-on-write), and "block size 是容量与 kernel 的共同参数" (ceil(seq_len /
    block_size) blocks per request).

Where the pages are silent the reading taken is stated in the function's
docstring. Every function here is pinned by tests that do not call the same
formula twice (brute force, closed forms, invariances, printed figures).
"""

from .attention import (  # noqa: F401
    gather_sequence,
    decode_attention,
    decode_attention_one,
    split_partials,
    merge_partials,
    split_context_attention,
)
from .cache_ops import append_kv, copy_blocks, swap_blocks  # noqa: F401
from .fp8 import (  # noqa: F401
    e4m3_decode,
    e4m3_encode,
    quantize_rows,
    append_kv_fp8,
    dequantize_pool,
    decode_attention_fp8,
)
from .interleaved import (  # noqa: F401
    kv_block_dtype,
    make_kv_pool,
    split_kv_pool,
    append_kv_interleaved,
    copy_blocks_interleaved,
    decode_attention_interleaved,
    decode_attention_interleaved_fp8,
)
from .allocator import BlockAllocator, OutOfBlocks, shared_prefix_blocks  # noqa: F401
from .accounting import (  # noqa: F401
    blocks_needed,
    paged_internal_waste,
    naive_slab_waste,
    concurrent_sequences,
)
from .step import (  # noqa: F401
    place_batch,
    decode_step,
    DecodeStepResult,
)
