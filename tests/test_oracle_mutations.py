"""Plant plausible mistakes in copies of the oracle and require that the pins
catch each one. Every mutant runs on the CPU; nothing here touches a GPU."""

import numpy as np
import pytest

import oracle
from oracle import attention as att
from tests import oracle_pins as pins


def _fails_some_pin(decode):
    failed = []
    for check in pins.ALL_DECODE_CHECKS:
        try:
            check(decode)
        except (AssertionError, FloatingPointError, ValueError, IndexError):
            failed.append(check.__name__)
    return failed


def _decode_with(one=None, gather=None, kv_of=None):
    """A copy of the oracle's decode loop with one piece swapped out."""
    one = one or att.decode_attention_one
    gather = gather or att.gather_sequence

    def decode(q, kp, vp, table, lens, scale, seqs=None, heads=None):
        S, Hq, D = q.shape
        BS, Hkv = kp.shape[1], kp.shape[2]
        G = Hq // Hkv
        out = np.zeros((S, Hq, D))
        for i in range(S):
            L = int(lens[i])
            if L == 0:
                continue
            K = gather(kp, table[i], L, BS)
            V = gather(vp, table[i], L, BS)
            for h in range(Hq):
                kv = kv_of(h, G, Hkv) if kv_of else h // G
                out[i, h] = one(q[i, h], K[:, kv], V[:, kv], float(np.float32(scale)))
        return out
    return decode


def _gather_reversed_offsets(pool, row, L, BS):
    out = np.empty((L,) + pool.shape[2:])
    for t in range(L):
        out[t] = pool[int(row[t // BS]), BS - 1 - t % BS]
    return out


def _gather_ignoring_table(pool, row, L, BS):
    return pool.reshape((-1,) + pool.shape[2:])[:L].astype(np.float64)


def _one_no_scale(q, K, V, scale):
    return att.decode_attention_one(q, K, V, 1.0)


def _one_swapped_kv(q, K, V, scale):
    return att.decode_attention_one(q, V, K, scale)


def _one_no_max(q, K, V, scale):
    with np.errstate(over="ignore", invalid="ignore"):
        s = scale * (K @ q.astype(np.float64))
        e = np.exp(s)
        return (e / e.sum()) @ V


def _one_drop_last_token(q, K, V, scale):
    return att.decode_attention_one(q, K[:-1], V[:-1], scale) if len(K) > 1 else \
        att.decode_attention_one(q, K, V, scale)


def _one_unnormalised(q, K, V, scale):
    s = scale * (K @ q.astype(np.float64))
    return np.exp(s - s.max()) @ V


MUTANTS = {
    "dropped_scale": _decode_with(one=_one_no_scale),
    "k_v_swapped": _decode_with(one=_one_swapped_kv),
    "no_max_subtraction": _decode_with(one=_one_no_max),
    "last_token_dropped": _decode_with(one=_one_drop_last_token),
    "not_normalised": _decode_with(one=_one_unnormalised),
    "offset_reversed": _decode_with(gather=_gather_reversed_offsets),
    "table_ignored": _decode_with(gather=_gather_ignoring_table),
    "gqa_modulo_mapping": _decode_with(kv_of=lambda h, G, Hkv: h % Hkv),
}


def test_unmutated_copy_passes():
    assert _fails_some_pin(_decode_with()) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    assert _fails_some_pin(MUTANTS[name]), f"mutant {name} passed every pin"


def test_split_merge_mutant_caught():
    def bad_merge(ms, ls, accs):          # forgets to rescale by exp(m_j - M)
        return np.asarray(accs).sum(0) / np.asarray(ls).sum()

    def split_bad(qv, K, V, scale, chunk):
        L = K.shape[0]
        s = scale * (K @ qv)
        bounds = [(a, min(L, a + chunk)) for a in range(0, L, chunk)]
        return bad_merge(*att.split_partials(s, V, bounds))

    with pytest.raises(AssertionError):
        pins.check_split_merge(split_bad, oracle.decode_attention_one)


def _prefix_ignoring_whole_blocks(tables, lens, bs):
    k = min(len(t) for t in tables) if tables else 0
    first = list(tables[0]) if tables else []
    for t in tables[1:]:
        j = 0
        while j < k and t[j] == first[j]:
            j += 1
        k = j
    return first[:k]


def _prefix_ignoring_other_tables(tables, lens, bs):
    if not tables:
        return []
    k = min(min(len(t), int(L) // bs) for t, L in zip(tables, lens))
    return list(tables[0])[:k]


_shared_prefix_blocks = oracle.shared_prefix_blocks


def _prefix_one_block_short(tables, lens, bs):
    return _shared_prefix_blocks(tables, lens, bs)[:-1]


@pytest.mark.parametrize("mutant", [_prefix_ignoring_whole_blocks, _prefix_ignoring_other_tables,
                                    _prefix_one_block_short])
def test_shared_prefix_pins_catch_planted_mistakes(monkeypatch, mutant):
    """Each planted mistake in the shared-prefix definition fails one of its
    pins (the sharing picture, the special cases, the random-fork invariants)."""
    from oracle import allocator as alloc
    from tests import test_oracle_allocator as t
    monkeypatch.setattr(alloc, "shared_prefix_blocks", mutant)
    monkeypatch.setattr(oracle, "shared_prefix_blocks", mutant)
    failed = 0
    for check in (t.test_shared_prefix_of_the_sharing_picture, t.test_shared_prefix_special_cases,
                  t.test_shared_prefix_invariants_under_random_forks):
        try:
            check()
        except AssertionError:
            failed += 1
    assert failed > 0
