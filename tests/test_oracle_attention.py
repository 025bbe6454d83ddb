"""The attention oracle against brute force, a library routine, closed forms
and the paging invariances printed on the pages (see tests/oracle_pins.py)."""

import math

import numpy as np
import pytest

import oracle
from tests import oracle_pins as pins


@pytest.mark.parametrize("check", pins.ALL_DECODE_CHECKS, ids=lambda f: f.__name__)
def test_decode_attention_pins(check):
    check(oracle.decode_attention)


def test_split_merge_identity():
    pins.check_split_merge(oracle.split_context_attention, oracle.decode_attention_one)


def test_merge_handles_empty_chunks():
    ms, ls, accs = oracle.split_partials(np.array([0.5, 1.0]), np.eye(2), [(0, 0), (0, 2), (2, 2)])
    assert ms[0] == -np.inf and ls[0] == 0.0
    ref = oracle.decode_attention_one(np.array([1.0]), np.array([[0.5], [1.0]]), np.eye(2), 1.0)
    assert np.allclose(oracle.merge_partials(ms, ls, accs), ref, rtol=1e-15)


def test_gather_reads_rows_in_logical_order():
    BS, H, D = 4, 1, 1
    pool = np.arange(3 * BS, dtype=np.float16).reshape(3, BS, H, D)
    rows = oracle.gather_sequence(pool, [2, 0, 1], 10, BS)[:, 0, 0]
    assert rows.tolist() == [8, 9, 10, 11, 0, 1, 2, 3, 4, 5]


def test_sampled_rows_match_full():
    q, kp, vp, table, L = pins._rand_case(3, 4, 6, 2, 8, 4, [9, 0, 5, 12])
    full = oracle.decode_attention(q, kp, vp, table, L, np.float32(0.3))
    part = oracle.decode_attention(q, kp, vp, table, L, np.float32(0.3), seqs=[2], heads=[1, 5])
    assert np.array_equal(part[2, [1, 5]], full[2, [1, 5]])
    assert not part[0].any() and not part[2, 0].any()


def test_scale_is_fp32_widened():
    # 1/sqrt(128) is not exactly representable; the oracle uses the fp32 value
    q = np.zeros((1, 1, 2), np.float16); q[0, 0, 0] = 1
    kp = np.zeros((1, 2, 1, 2), np.float16); kp[0, 0, 0, 0] = 1
    vp = np.zeros((1, 2, 1, 2), np.float16); vp[0, 0, 0, 1] = 1
    out = oracle.decode_attention(q, kp, vp, np.array([[0]], np.int32), np.array([2]), 1 / math.sqrt(128))
    s = float(np.float32(1 / math.sqrt(128)))
    assert out[0, 0, 1] == pytest.approx(math.exp(s) / (math.exp(s) + 1), rel=1e-15)
