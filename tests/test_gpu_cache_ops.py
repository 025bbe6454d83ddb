"""Append and copy-on-write block copy on the GPU: bit-exact against the
oracle, only the targeted rows/blocks change, and out-of-range ids are
skipped and reported."""

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def pa(libpa):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return libpa


def _pools(nb, bs, h, d, seed):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((nb, bs, h, d)).astype(np.float16)
    v = rng.standard_normal((nb, bs, h, d)).astype(np.float16)
    k[0, 0, 0, :4] = np.array([0x7e01, 0xfc00, 0x8000, 0x0001], np.uint16).view(np.float16)
    return k, v


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("shape", [(40, 16, 8, 128), (33, 8, 4, 64), (20, 32, 32, 128)])
def test_append_bit_exact(pa, shape):
    nb, bs, h, d = shape
    k, v = _pools(nb, bs, h, d, 1)
    rng = np.random.default_rng(2)
    T = 25
    slots = rng.choice(nb * bs, T, replace=False).astype(np.int32)
    slots[3] = -1
    kn = rng.standard_normal((T, h, d)).astype(np.float16)
    vn = rng.standard_normal((T, h, d)).astype(np.float16)
    kn[0, 0, :2] = np.array([0x7c01, 0xffff], np.uint16).view(np.float16)   # NaN payloads
    ek, ev = oracle.append_kv(k, v, kn, vn, slots)
    dk, dv = dev(k), dev(v)
    pa.pa_append_kv(dev(kn), dev(vn), dk, dv, dev(slots))
    torch.cuda.synchronize()
    assert np.array_equal(dk.cpu().numpy().view(np.uint16), ek.view(np.uint16))
    assert np.array_equal(dv.cpu().numpy().view(np.uint16), ev.view(np.uint16))
    assert pa.pa_device_error() == 0


def test_append_out_of_range_slot(pa):
    k, v = _pools(10, 16, 2, 64, 3)
    kn = np.ones((2, 2, 64), np.float16)
    slots = np.array([5, 10 * 16], np.int32)        # second is one past the pool
    dk, dv = dev(k), dev(v)
    pa.pa_append_kv(dev(kn), dev(kn), dk, dv, dev(slots))
    ek, ev = oracle.append_kv(k, v, kn, kn, np.array([5, -1], np.int32))
    with pytest.raises(pa.PaError) as e:
        pa.pa_device_error()
    assert e.value.flags & pa.PA_DEVERR_BAD_SLOT
    assert np.array_equal(dk.cpu().numpy().view(np.uint16), ek.view(np.uint16))


@pytest.mark.parametrize("shape", [(300, 16, 8, 128), (50, 8, 32, 128), (64, 32, 4, 64)])
def test_copy_blocks_bit_exact(pa, shape):
    nb, bs, h, d = shape
    k, v = _pools(nb, bs, h, d, 4)
    rng = np.random.default_rng(5)
    ids = rng.permutation(nb)
    n = nb // 3
    pairs = np.stack([ids[:n], ids[n:2 * n]], 1).astype(np.int32)
    ek, ev = oracle.copy_blocks(k, v, pairs)
    dk, dv = dev(k), dev(v)
    pa.pa_copy_blocks(dk, dv, dev(pairs))
    torch.cuda.synchronize()
    assert np.array_equal(dk.cpu().numpy().view(np.uint16), ek.view(np.uint16))
    assert np.array_equal(dv.cpu().numpy().view(np.uint16), ev.view(np.uint16))
    assert pa.pa_device_error() == 0


def test_copy_blocks_bad_id(pa):
    k, v = _pools(8, 16, 2, 64, 6)
    pairs = np.array([[1, 2], [3, 99], [-1, 4], [5, 6]], np.int32)
    dk, dv = dev(k), dev(v)
    pa.pa_copy_blocks(dk, dv, dev(pairs))
    ek, ev = oracle.copy_blocks(k, v, np.array([[1, 2], [5, 6]], np.int32))
    with pytest.raises(pa.PaError) as e:
        pa.pa_device_error()
    assert e.value.flags & pa.PA_DEVERR_BAD_BLOCK
    assert np.array_equal(dk.cpu().numpy().view(np.uint16), ek.view(np.uint16))
    assert np.array_equal(dv.cpu().numpy().view(np.uint16), ev.view(np.uint16))
