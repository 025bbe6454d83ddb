"""The seeded workload generators: deterministic, shaped as the configs say."""

import numpy as np

import synthetic


def test_tiny_config_shapes_and_determinism():
    a = synthetic.config1_tiny()
    b = synthetic.config1_tiny()
    assert a.prefill_lens.tolist() == [5, 16, 17, 40]
    assert a.q.shape == (4, 4, 64) and a.k_pool.shape == (32, 16, 4, 64)
    assert a.q.dtype == np.float16 and abs(float(a.k_pool.astype(np.float32).max())) <= 1.0
    assert sorted(a.free_order.tolist()) == list(range(32))
    assert a.q.tobytes() == b.q.tobytes() and a.v_new.tobytes() == b.v_new.tobytes()
    assert a.scale == np.float32(0.125)


def test_gqa_batch_small_variant():
    b = synthetic.config2_gqa_batch(num_seqs=5, lo=10, hi=40, head_dim=64)
    assert b.q.shape == (5, 32, 64) and b.k_pool.shape[2] == 8
    assert ((b.prefill_lens >= 10) & (b.prefill_lens <= 40)).all()
    need = sum(-(-int(L) // 16) for L in b.attended_lens)
    assert b.num_blocks == int(np.ceil(1.25 * need))


def test_churn_ops_are_balanced():
    b = synthetic.config3_mha_lognormal(num_seqs=8, num_heads=2, head_dim=16, churn_ops=500)
    live = set()
    for op in b.churn:
        if op.kind == "alloc":
            live.add(op.owner)
        else:
            live.remove(op.owner)
    assert not live and len(b.churn) > 100
    assert ((b.prefill_lens >= 16) & (b.prefill_lens <= 8192)).all()


def test_shared_prefix_step_inputs_keyed_by_step():
    w = synthetic.config4_shared_prefix(num_seqs=4, prefix_len=40, max_steps=5, head_dim=16)
    q1, k1, _ = w.step_inputs(0, 4)
    q2, _, _ = w.step_inputs(0, 4)
    q3, _, _ = w.step_inputs(1, 4)
    assert q1.tobytes() == q2.tobytes() and q1.tobytes() != q3.tobytes()
    assert k1.shape == (4, 8, 16)


def test_fp8_cache_is_seeded_and_finite():
    import synthetic
    b = synthetic.config1_tiny()
    a1 = synthetic.fp8_cache(b, seed=5)
    a2 = synthetic.fp8_cache(b, seed=5)
    assert (a1.k_pool == a2.k_pool).all() and (a1.v_scale == a2.v_scale).all()
    assert a1.k_pool.shape == b.k_pool.shape and a1.k_pool.dtype == np.uint8
    for pool in (a1.k_pool, a1.v_pool):
        assert not ((pool & 0x7F) == 0x7F).any()          # no NaN codes
        e = (pool >> 3) & 0xF
        assert e.min() >= 8 and e.max() <= 14
    assert (a1.k_scale > 0).all() and (a1.v_scale > 0).all()


def test_every_finite_code_generator():
    codes = synthetic.fp8_finite_codes()
    assert codes.size == 254 and codes.dtype == np.uint8
    assert 0x7F not in codes and 0xFF not in codes
    for c in (0x00, 0x80, 0x01, 0x07, 0x08, 0x7E, 0xFE, 0x3F):   # zeros, subnormals, 448
        assert c in codes
    rng = np.random.default_rng(3)
    a = synthetic.fp8_codes_every_finite(rng, (5, 16, 2, 128))     # 20480 = 80 tiles + 160
    counts = np.bincount(a.reshape(-1), minlength=256)
    assert counts[0x7F] == 0 and counts[0xFF] == 0
    fin = counts[codes]
    assert fin.min() >= 80 and fin.max() <= 81 and fin.sum() == a.size
    b = synthetic.fp8_codes_every_finite(np.random.default_rng(3), (5, 16, 2, 128))
    assert (a == b).all()
    c = synthetic.fp8_cache(synthetic.config1_tiny(), seed=5, every_code=True)
    assert set(np.unique(c.k_pool).tolist()) == set(codes.tolist())
