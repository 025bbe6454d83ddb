"""Append and block copy: exact bytes where written, untouched elsewhere."""

import numpy as np

import oracle


def _pools(nb=6, bs=4, h=2, d=8, seed=0):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((nb, bs, h, d)).astype(np.float16)
    v = rng.standard_normal((nb, bs, h, d)).astype(np.float16)
    return k, v


def test_append_writes_only_targeted_rows():
    k, v = _pools()
    rng = np.random.default_rng(1)
    kn = rng.standard_normal((3, 2, 8)).astype(np.float16)
    vn = rng.standard_normal((3, 2, 8)).astype(np.float16)
    slots = np.array([5, -1, 22], np.int32)       # block 1 row 1; skipped; block 5 row 2
    k2, v2 = oracle.append_kv(k, v, kn, vn, slots)
    assert k2[1, 1].tobytes() == kn[0].tobytes() and v2[5, 2].tobytes() == vn[2].tobytes()
    mask = np.ones(k.shape[:2], bool)
    mask[1, 1] = mask[5, 2] = False
    assert k2[mask].tobytes() == k[mask].tobytes() and v2[mask].tobytes() == v[mask].tobytes()
    assert k[1, 1].tobytes() != k2[1, 1].tobytes()       # inputs not modified in place


def test_copy_blocks_exact_and_reads_sources_before_writes():
    k, v = _pools()
    k2, v2 = oracle.copy_blocks(k, v, np.array([[0, 3], [2, 4]], np.int32))
    assert k2[3].tobytes() == k[0].tobytes() and v2[4].tobytes() == v[2].tobytes()
    for b in (0, 1, 2, 5):
        assert k2[b].tobytes() == k[b].tobytes() and v2[b].tobytes() == v[b].tobytes()


def test_nan_payload_is_copied_bit_for_bit():
    k, v = _pools()
    bits = np.array([0x7e01, 0xfc00, 0x8000], np.uint16).view(np.float16)
    k[0, 0, 0, :3] = bits
    k2, _ = oracle.copy_blocks(k, v, [[0, 1]])
    assert k2[1, 0, 0, :3].view(np.uint16).tolist() == [0x7e01, 0xfc00, 0x8000]
