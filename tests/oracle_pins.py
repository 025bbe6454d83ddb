"""Checks that pin the attention oracle to facts outside itself.

Each check takes the decode-attention function under test (normally
`oracle.decode_attention`) and raises AssertionError when it disagrees with:

  * brute force on tiny inputs (explicit per-token, per-dimension loops),
  * the textbook attention of a library (torch scaled_dot_product_attention,
    fp64, CPU) on a contiguous cache,
  * closed forms (one token, equal keys, constant values, a dominant key,
    empty sequence),
  * the paging invariances the pages state: a block table is only an
    indirection, so permuting physical blocks (the worked mapping 0->7, 1->2,
    2->9 of lux-666 notes "PagedAttention", 最小模型) or sharing a prefix block
    (A->[3,7,1], B->[3,9] of "Phase 7 · Document 04 — PagedAttention", §3
    Mental Model) leaves every output unchanged.

The mutation tests feed deliberately broken variants through the same checks
and require that at least one fails.
"""

from __future__ import annotations

import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name: str) -> dict:
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rand_case(seed, S, Hq, Hkv, D, BS, lens, nb=None):
    rng = np.random.default_rng(seed)
    mb = max(1, max(-(-L // BS) for L in lens))
    need = sum(-(-L // BS) for L in lens)
    nb = nb or need + 3
    perm = rng.permutation(nb)
    table = -np.ones((S, mb), dtype=np.int32)
    pos = 0
    for i, L in enumerate(lens):
        n = -(-L // BS)
        table[i, :n] = perm[pos:pos + n]
        pos += n
    q = rng.standard_normal((S, Hq, D)).astype(np.float16)
    kp = rng.standard_normal((nb, BS, Hkv, D)).astype(np.float16)
    vp = rng.standard_normal((nb, BS, Hkv, D)).astype(np.float16)
    return q, kp, vp, table, np.array(lens, dtype=np.int32)


def brute_force(q, kp, vp, table, lens, scale):
    """Per-token, per-dimension loops in plain Python floats."""
    S, Hq, D = q.shape
    BS, Hkv = kp.shape[1], kp.shape[2]
    G = Hq // Hkv
    sc = float(np.float32(scale))
    out = np.zeros((S, Hq, D))
    for i in range(S):
        L = int(lens[i])
        for h in range(Hq):
            kv = h // G
            scores = []
            for t in range(L):
                blk, off = int(table[i][t // BS]), t % BS
                dot = 0.0
                for d in range(D):
                    dot += float(q[i, h, d]) * float(kp[blk, off, kv, d])
                scores.append(sc * dot)
            if L == 0:
                continue
            mx = max(scores)
            w = [math.exp(s - mx) for s in scores]
            z = sum(w)
            for d in range(D):
                acc = 0.0
                for t in range(L):
                    blk, off = int(table[i][t // BS]), t % BS
                    acc += w[t] * float(vp[blk, off, kv, d])
                out[i, h, d] = acc / z
    return out


def check_brute_force(decode):
    # GQA 2, ragged lengths spanning several blocks, an empty sequence
    for seed, (S, Hq, Hkv, D, BS, lens) in enumerate([
        (3, 4, 2, 8, 4, [1, 7, 13]),
        (2, 6, 3, 16, 8, [17, 0]),
        (2, 2, 2, 4, 2, [5, 3]),
    ]):
        q, kp, vp, table, L = _rand_case(100 + seed, S, Hq, Hkv, D, BS, lens)
        scale = np.float32(1.0 / math.sqrt(D))
        ref = brute_force(q, kp, vp, table, L, scale)
        got = decode(q, kp, vp, table, L, scale)
        assert np.allclose(got, ref, rtol=1e-12, atol=1e-12), "brute force"


def check_library_sdpa(decode):
    import torch
    import torch.nn.functional as F
    rng = np.random.default_rng(7)
    Hq, Hkv, D, BS, L = 8, 2, 32, 16, 45
    G = Hq // Hkv
    nb = -(-L // BS)
    kp = rng.standard_normal((nb, BS, Hkv, D)).astype(np.float16)
    vp = rng.standard_normal((nb, BS, Hkv, D)).astype(np.float16)
    q = rng.standard_normal((1, Hq, D)).astype(np.float16)
    table = np.arange(nb, dtype=np.int32)[None, :]      # identity: contiguous
    scale = np.float32(1.0 / math.sqrt(D))
    K = torch.from_numpy(kp.reshape(nb * BS, Hkv, D)[:L].astype(np.float64))
    V = torch.from_numpy(vp.reshape(nb * BS, Hkv, D)[:L].astype(np.float64))
    K = K.permute(1, 0, 2).repeat_interleave(G, dim=0)[None]   # [1,Hq,L,D]
    V = V.permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
    Q = torch.from_numpy(q.astype(np.float64))[:, :, None, :]  # [1,Hq,1,D]
    ref = F.scaled_dot_product_attention(Q, K, V, scale=float(scale))[0, :, 0, :]
    got = decode(q, kp, vp, table, np.array([L], np.int32), scale)
    assert np.allclose(got[0], ref.numpy(), rtol=1e-11, atol=1e-12), "sdpa"


def check_closed_forms(decode):
    rng = np.random.default_rng(11)
    Hq = Hkv = 2
    D, BS = 8, 4
    scale = np.float32(0.5)
    # (1) one token: out == v_0 exactly
    kp = rng.standard_normal((3, BS, Hkv, D)).astype(np.float16)
    vp = rng.standard_normal((3, BS, Hkv, D)).astype(np.float16)
    q = rng.standard_normal((1, Hq, D)).astype(np.float16)
    got = decode(q, kp, vp, np.array([[2]], np.int32), np.array([1], np.int32), scale)
    assert np.array_equal(got[0], vp[2, 0].astype(np.float64)), "one token"
    # (2) equal keys: uniform weights, out == mean of V rows
    L = 10
    kp2 = np.repeat(kp[:1, :1], 3 * BS, axis=1).reshape(3, BS, Hkv, D)
    table = np.array([[1, 0, 2]], np.int32)
    got = decode(q, kp2, vp, table, np.array([L], np.int32), scale)
    rows = np.concatenate([vp[1], vp[0], vp[2]])[:L].astype(np.float64)
    assert np.allclose(got[0], rows.mean(0), rtol=1e-12, atol=1e-13), "equal keys"
    # (3) constant values: out == c whatever the keys
    vp3 = np.full_like(vp, np.float16(0.375))
    got = decode(q, kp, vp3, table, np.array([L], np.int32), scale)
    assert np.allclose(got, 0.375, rtol=0, atol=1e-14), "constant values"
    # (4) a dominant key: score gap of ~1e4 selects that row (no overflow)
    qd = np.zeros((1, Hq, D), np.float16)
    qd[0, :, 0] = 100.0
    kd = np.zeros((3, BS, Hkv, D), np.float16)
    kd[0, 2, :, 0] = 100.0          # logical token 4+2 = 6 (table [1,0,2])
    got = decode(qd, kd, vp, table, np.array([L], np.int32), np.float32(1.0))
    assert np.allclose(got[0], vp[0, 2].astype(np.float64), atol=1e-12), "dominant"
    # (5) empty sequence: zeros
    got = decode(q, kp, vp, table, np.array([0], np.int32), scale)
    assert np.array_equal(got, np.zeros_like(got)), "empty"


def check_worked_permutation(decode):
    """P2's worked table: blocks of request A at physical 7, 2, 9 of a
    ten-block pool give the same result as the contiguous layout 0, 1, 2."""
    g = golden("worked_block_table.json")
    phys = g["logical_to_physical"]
    nb = g["physical_blocks_pictured"]
    rng = np.random.default_rng(12)
    Hq, Hkv, D, BS = 4, 2, 16, 16
    L = 2 * BS + 5                         # three logical blocks, last partial
    contig_k = rng.standard_normal((3, BS, Hkv, D)).astype(np.float16)
    contig_v = rng.standard_normal((3, BS, Hkv, D)).astype(np.float16)
    q = rng.standard_normal((1, Hq, D)).astype(np.float16)
    kp = rng.standard_normal((nb, BS, Hkv, D)).astype(np.float16)   # noise
    vp = rng.standard_normal((nb, BS, Hkv, D)).astype(np.float16)
    for logical, p in enumerate(phys):
        kp[p] = contig_k[logical]
        vp[p] = contig_v[logical]
    scale = np.float32(0.25)
    a = decode(q, contig_k, contig_v, np.array([[0, 1, 2]], np.int32),
               np.array([L], np.int32), scale)
    b = decode(q, kp, vp, np.array([phys], np.int32), np.array([L], np.int32), scale)
    assert np.array_equal(a, b), "worked permutation"
    # a table that moves the partial tail block must change the result
    # (softmax attention ignores token order, so only the token set counts)
    c = decode(q, kp, vp, np.array([[phys[2], phys[1], phys[0]]], np.int32),
               np.array([L], np.int32), scale)
    assert not np.allclose(a, c), "table order ignored"


def check_sharing_picture(decode):
    """P3's picture: A -> [3,7,1], B -> [3,9]; B's output equals the output
    over a private copy of its blocks, and A is unaffected by B."""
    g = golden("sharing_picture.json")
    rng = np.random.default_rng(13)
    Hq, Hkv, D, BS = 2, 1, 16, 4
    nb = 10
    kp = rng.standard_normal((nb, BS, Hkv, D)).astype(np.float16)
    vp = rng.standard_normal((nb, BS, Hkv, D)).astype(np.float16)
    q = rng.standard_normal((2, Hq, D)).astype(np.float16)
    LA, LB = 3 * BS, 2 * BS - 1
    table = np.array([g["seq_A"], g["seq_B"] + [-1]], np.int32)
    both = decode(q, kp, vp, table, np.array([LA, LB], np.int32), np.float32(0.3))
    # private copies: B's blocks moved to fresh ids 0 and 4
    kp2, vp2 = kp.copy(), vp.copy()
    kp2[0], vp2[0] = kp[g["seq_B"][0]], vp[g["seq_B"][0]]
    kp2[4], vp2[4] = kp[g["seq_B"][1]], vp[g["seq_B"][1]]
    alone_b = decode(q[1:], kp2, vp2, np.array([[0, 4]], np.int32),
                     np.array([LB], np.int32), np.float32(0.3))
    alone_a = decode(q[:1], kp, vp, np.array([g["seq_A"]], np.int32),
                     np.array([LA], np.int32), np.float32(0.3))
    assert np.array_equal(both[1], alone_b[0]), "shared prefix B"
    assert np.array_equal(both[0], alone_a[0]), "shared prefix A"


ALL_DECODE_CHECKS = (check_brute_force, check_library_sdpa, check_closed_forms,
                     check_worked_permutation, check_sharing_picture)


def check_split_merge(split_fn, one_fn):
    """Any chunking of the context gives the unsplit result (fp64, 1e-12)."""
    rng = np.random.default_rng(21)
    for L in (1, 2, 15, 16, 17, 100):
        K = rng.standard_normal((L, 32))
        V = rng.standard_normal((L, 32))
        qv = rng.standard_normal(32) * 3
        ref = one_fn(qv, K, V, 0.2)
        for chunk in (1, 3, 16, 64, L):
            got = split_fn(qv, K, V, 0.2, chunk)
            assert np.allclose(got, ref, rtol=1e-12, atol=1e-12), (L, chunk)
    # reference itself against an explicit loop
    L = 9
    K = rng.standard_normal((L, 4))
    V = rng.standard_normal((L, 4))
    qv = rng.standard_normal(4)
    s = [0.2 * sum(qv[d] * K[t, d] for d in range(4)) for t in range(L)]
    w = [math.exp(x) for x in s]
    exp = [sum(w[t] * V[t, d] for t in range(L)) / sum(w) for d in range(4)]
    assert np.allclose(one_fn(qv, K, V, 0.2), exp, rtol=1e-12), "one"
