"""pa_decode_attention_fixed_scratch: the decode entry point that allocates
nothing, for callers that cannot give libpa a workspace (all their device
memory already belongs to their own KV pool and allocator, or they cannot
afford cudaMalloc's device synchronisation on the decode path). It must give
the same result as pa_decode_attention with a caller workspace, call after
call, although every call reuses the same fixed scratch array.

This file is collected last so that a run stopping at the first failure has
already run every other test."""

import math

import numpy as np
import pytest

import synthetic
from tests.gpu_helpers import assert_close_attention, poison_unread_rows

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _case(seed, lens, hq=32, hkv=8, d=128, bs=16):
    rng = np.random.default_rng(seed)
    mb = max(-(-L // bs) for L in lens)
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
    return [_dev(x) for x in (q, kp, vp, table, np.asarray(lens, np.int32))]


def test_fixed_scratch_matches_workspace_entry_two_calls(libpa):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pa = libpa
    scale = 1.0 / math.sqrt(128)
    cases = [
        _case(1, [3000, 17, 1, 2049, 640, 0, 96]),              # long ones are split
        _case(2, list(np.random.default_rng(3).integers(1, 2048, 40))),
    ]
    for q, kp, vp, table, lens in cases:      # two calls in a row on the shared array
        ref = pa.pa_decode_attention(q, kp, vp, table, lens, scale)
        got = pa.pa_decode_attention_fixed_scratch(q, kp, vp, table, lens, scale)
        torch.cuda.synchronize()
        assert_close_attention(got.cpu().numpy(), ref.cpu().numpy().astype(np.float64),
                               "fixed scratch vs workspace")
    assert pa.pa_device_error() == 0


def test_fixed_scratch_refuses_oversized_shapes(libpa):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    q, kp, vp, table, lens = _case(4, [4000] * 8)
    with pytest.raises(libpa.PaError) as e:
        # one block per chunk: thousands of partial records, far above the fixed array
        libpa.pa_decode_attention_fixed_scratch(q, kp, vp, table, lens, 0.1, partition_tokens=16)
    assert e.value.status_name == "PA_ERR_UNSUPPORTED"
