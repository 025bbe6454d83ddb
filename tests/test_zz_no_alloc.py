"""pa_decode_attention_fixed_scratch: the decode entry point that allocates
nothing, for callers that cannot give libpa a workspace (all their device
memory already belongs to their own KV pool and allocator, or they cannot
afford cudaMalloc's device synchronisation on the decode path). It runs the
same kernel with the same grid and chunking as pa_decode_attention, so its
result must be bit-equal to that call's, and within the attention tolerance
of the oracle, call after call, although every call reuses the same fixed
scratch array: calls of different batch sizes follow one another, so a call
finds the previous call's partial results where its own counters now sit.

This file is collected last so that a run stopping at the first failure has
already run every other test."""

import math

import numpy as np
import pytest

import oracle
from tests.gpu_helpers import assert_close_attention, poison_unread_rows

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _case(seed, lens, hq=32, hkv=8, d=128, bs=16):
    """(host arrays, device tensors) of a poisoned decode batch."""
    rng = np.random.default_rng(seed)
    mb = max(1, max(-(-L // bs) for L in lens))
    nb = sum(-(-L // bs) for L in lens) + 5
    perm = rng.permutation(nb)
    table = -np.ones((len(lens), mb), np.int32)
    pos = 0
    for i, L in enumerate(lens):
        n = -(-L // bs)
        table[i, :n] = perm[pos:pos + n]
        pos += n
    q = rng.standard_normal((len(lens), hq, d)).astype(np.float16)
    kp = rng.standard_normal((nb, bs, hkv, d)).astype(np.float16)
    vp = rng.standard_normal((nb, bs, hkv, d)).astype(np.float16)
    kp, vp = poison_unread_rows(kp, vp, table, lens, bs)
    lens = np.asarray(lens, np.int32)
    host = (q, kp, vp, table, lens)
    return host, [_dev(x) for x in host]


def test_fixed_scratch_matches_workspace_entry_and_oracle(libpa):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pa = libpa
    scale = np.float32(1.0 / math.sqrt(128))
    a = _case(1, [3000, 17, 1, 2049, 640, 0, 96])             # 7 sequences, long ones split
    b = _case(2, list(np.random.default_rng(3).integers(1, 2048, 40)))   # 40 sequences
    c = _case(5, [5000, 4000, 3000, 1])                        # 4 sequences, many chunks each
    # calls of different batch sizes in a row on the shared array, both ways
    for (host, dev) in (a, b, a, c, b):
        q, kp, vp, table, lens = dev
        ref = pa.pa_decode_attention(q, kp, vp, table, lens, scale)
        got = pa.pa_decode_attention_fixed_scratch(q, kp, vp, table, lens, scale)
        torch.cuda.synchronize()
        assert torch.equal(got, ref), "fixed scratch differs from the workspace entry"
        exp = oracle.decode_attention(*host[:4], host[4], scale)
        assert_close_attention(got.cpu().numpy(), exp, "fixed scratch vs oracle")
    assert pa.pa_device_error() == 0


def test_fixed_scratch_refuses_oversized_shapes(libpa):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _, (q, kp, vp, table, lens) = _case(4, [4000] * 8)
    with pytest.raises(libpa.PaError) as e:
        # one block per chunk: thousands of partial records, far above the fixed array
        libpa.pa_decode_attention_fixed_scratch(q, kp, vp, table, lens, 0.1, partition_tokens=16)
    assert e.value.status_name == "PA_ERR_UNSUPPORTED"
