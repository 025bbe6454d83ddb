"""Swapping on the GPU: pa_swap_blocks between the device pools and a pinned
host pool, driven by the native block manager, against the oracle's block
moves (bit for bit) and attention (before == after a round trip)."""

import numpy as np
import pytest

import oracle
from tests.gpu_helpers import assert_close_attention

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def pa(libpa):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return libpa


def _pairs(pairs, where):
    t = torch.tensor(np.asarray(pairs, np.int32).reshape(-1, 2))
    return t.pin_memory() if where == "host" else t.cuda()


@pytest.mark.parametrize("pairs_on", ["device", "host"])
def test_round_trip_through_pinned_host_pool(pa, pairs_on):
    rng = np.random.default_rng(5)
    nb, nh, bs, H, D = 64, 40, 16, 8, 128
    a = pa.BlockAllocator(nb, bs, rng.permutation(nb).tolist())
    ref = oracle.BlockAllocator(nb, bs, a.export_state()[0])
    a.add_host_pool(nh)
    ref.add_host_pool(nh)
    kp = rng.standard_normal((nb, bs, H, D)).astype(np.float16)
    vp = rng.standard_normal((nb, bs, H, D)).astype(np.float16)
    dk, dv = torch.from_numpy(kp).cuda(), torch.from_numpy(vp).cuda()
    hk = torch.zeros((nh, bs, H, D), dtype=torch.float16).pin_memory()
    hv = torch.zeros((nh, bs, H, D), dtype=torch.float16).pin_memory()
    for m in (a, ref):
        m.add_seq(1, 150)     # 10 blocks
        m.add_seq(2, 70)
    q = rng.standard_normal((1, 32, D)).astype(np.float16)
    t1 = np.array([a.table(1)], np.int32)
    before = pa.pa_decode_attention(torch.from_numpy(q).cuda(), dk, dv, torch.from_numpy(t1).cuda(),
                                    torch.tensor([150], dtype=torch.int32).cuda(), 0.09)
    out_pairs = a.swap_out(1)
    assert out_pairs == ref.swap_out(1)
    pa.pa_swap_blocks(dk, dv, hk, hv, _pairs(out_pairs, pairs_on))
    # the released device blocks are reused and overwritten
    a.add_seq(3, 160)
    ref.add_seq(3, 160)
    for b in a.table(3):
        dk[b] = float("nan")
        dv[b] = float("nan")
    in_pairs = a.swap_in(1)
    assert in_pairs == ref.swap_in(1)
    pa.pa_swap_blocks(hk, hv, dk, dv, _pairs(in_pairs, pairs_on))
    torch.cuda.synchronize()
    # bytes: host pool and the restored device blocks as the oracle moves them
    ehk, ehv = oracle.swap_blocks(kp, vp, np.zeros_like(hk.numpy()), np.zeros_like(hv.numpy()),
                                  out_pairs)
    assert np.array_equal(hk.numpy().view(np.uint16), ehk.view(np.uint16))
    for (h, d) in in_pairs:
        assert np.array_equal(dk[d].cpu().numpy().view(np.uint16), ehk[h].view(np.uint16))
        assert np.array_equal(dv[d].cpu().numpy().view(np.uint16), ehv[h].view(np.uint16))
    t1b = np.array([a.table(1)], np.int32)
    after = pa.pa_decode_attention(torch.from_numpy(q).cuda(), dk, dv, torch.from_numpy(t1b).cuda(),
                                   torch.tensor([150], dtype=torch.int32).cuda(), 0.09)
    torch.cuda.synchronize()
    assert torch.equal(before, after)
    exp = oracle.decode_attention(q, kp, vp, t1, [150], np.float32(0.09))
    assert_close_attention(after.cpu().numpy(), exp, "after swap round trip")
    assert a.export_state() == ref.export_state()
    assert a.export_host_state() == ref.export_host_state()
    assert pa.pa_device_error() == 0


def test_swap_fp8_pools(pa):
    rng = np.random.default_rng(6)
    kp = rng.integers(0, 256, (12, 16, 4, 128), dtype=np.uint8)
    vp = rng.integers(0, 256, (12, 16, 4, 128), dtype=np.uint8)
    hk = torch.zeros((5, 16, 4, 128), dtype=torch.uint8).pin_memory()
    hv = torch.zeros((5, 16, 4, 128), dtype=torch.uint8).pin_memory()
    pairs = [(7, 0), (2, 4), (11, 1)]
    pa.pa_swap_blocks(torch.from_numpy(kp).cuda(), torch.from_numpy(vp).cuda(), hk, hv,
                      _pairs(pairs, "host"))
    torch.cuda.synchronize()
    ek, ev = oracle.swap_blocks(kp, vp, np.zeros((5, 16, 4, 128), np.uint8),
                                np.zeros((5, 16, 4, 128), np.uint8), pairs)
    assert np.array_equal(hk.numpy(), ek) and np.array_equal(hv.numpy(), ev)


def test_pageable_host_memory_is_refused(pa):
    dk = torch.zeros((4, 16, 2, 128), dtype=torch.float16).cuda()
    hk = torch.zeros((4, 16, 2, 128), dtype=torch.float16)          # not pinned
    with pytest.raises(ValueError):
        pa.pa_swap_blocks(dk, dk, hk, hk, _pairs([(0, 1)], "device"))
