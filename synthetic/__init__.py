"""Seeded synthetic inputs for paged decode attention.

This module only draws random numbers and lays them out. It holds none of the
method's arithmetic: no block tables, no slot computation, no attention. Both
the CUDA path's tests/benchmark and the CPU oracle take their inputs from here,
so the two sides see identical bytes while sharing no code of the method.

Every workload is a `DecodeBatch`: the lengths already in the cache before the
step (`prefill_lens`), the order in which the pool's physical block ids start
out on the free list (`free_order`), and the fp16 tensors. Where a config
needs allocator traffic before placement (alloc/free churn) or several decode
steps (the shared-prefix config), the draws for that traffic are generated
here too and passed in as plain data.

Draw order per config (one `numpy.random.default_rng(seed)` PCG64 stream):
lengths, free order, [churn ops], q, k_pool, v_pool, k_new, v_new. Integer
uniforms are inclusive on both ends.

An fp8 (E4M3) cache for a batch (`fp8_cache`) comes from a stream of its own:
its bytes are composed from random sign, exponent and mantissa fields, so no
quantization is computed here either.
"""

from .configs import (  # noqa: F401
    DecodeBatch,
    ChurnOp,
    SharedPrefixWorkload,
    make_batch,
    config1_tiny,
    config2_gqa_batch,
    config3_mha_lognormal,
    config4_shared_prefix,
    config5_long_context,
    CONFIG_NAMES,
    Fp8Cache,
    fp8_codes,
    fp8_codes_every_finite,
    fp8_finite_codes,
    fp8_cache,
)
