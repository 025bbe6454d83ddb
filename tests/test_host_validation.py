"""Host-side argument checks: refused before any device work (no GPU needed)."""

import ctypes

import pytest

NULL = None


def _decode(lib, **kw):
    a = dict(q=NULL, k=NULL, v=NULL, table=NULL, lens=NULL, S=4, Hq=32, Hkv=8, D=128, BS=16,
             MB=8, NB=64, stride=0, scale=0.1, out=NULL, ws=NULL, wsb=0, pt=0, stream=NULL)
    a.update(kw)
    return lib.pa_decode_attention(a["q"], a["k"], a["v"], a["table"], a["lens"], a["S"], a["Hq"],
                                   a["Hkv"], a["D"], a["BS"], a["MB"], a["NB"], a["stride"],
                                   ctypes.c_float(a["scale"]), a["out"], a["ws"], a["wsb"],
                                   a["pt"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(Hq=30), 1),                 # not a multiple of kv heads
    (dict(Hq=48, Hkv=3), 4),          # ratio 16 unsupported
    (dict(D=96), 4),
    (dict(BS=64), 4),
    (dict(S=20000), 4),
    (dict(MB=0), 1),
    (dict(pt=24), 1),                 # not a multiple of the block size
    (dict(pt=-16), 1),
    (dict(NB=0), 1),
    (dict(scale=float("inf")), 1),
    (dict(), 1),                      # NULL pointers
    # the largest batch's block stream must keep 32-bit positions:
    # 16384 sequences x 1 head group x 131072 blocks = 2^31
    (dict(S=16384, Hq=8, Hkv=8, MB=131072), 4),
    # one-block chunks of a 2^20-block sequence overflow a counter word's arrivals
    (dict(S=1, Hq=8, Hkv=8, MB=1 << 20, pt=16), 4),
])
def test_decode_rejects(libpa, kw, status):
    lib = libpa.lib()
    assert _decode(lib, **kw) == status
    assert lib.pa_last_error() != b""


def test_decode_zero_sequences_is_a_no_op(libpa):
    assert _decode(libpa.lib(), S=0) == 0


def test_workspace_bytes(libpa):
    lib = libpa.lib()
    # an 8-byte arrival counter per (sequence, KV head), then two partial
    # records per chunk (at most 1024 chunks) and per KV head a CTA streams (8
    # here), each G x (head_dim + 2) floats
    n = lib.pa_decode_workspace_bytes(64, 32, 8, 128, 16, 129, 0)
    assert n >= 64 * 8 * 8 + 2 * 1024 * 8 * (4 * 130) * 4
    assert n % 256 == 0
    assert lib.pa_decode_workspace_bytes(64, 32, 8, 96, 16, 129, 0) == 0
    # a per-chunk cap of one block can need one chunk per block of the stream
    capped = lib.pa_decode_workspace_bytes(64, 32, 8, 128, 16, 129, 16)
    assert capped >= 64 * 8 * 8 + 2 * (64 * 129) * 8 * (4 * 130) * 4
    # records are padded to 16-byte multiples: G=1, head_dim 64 -> 68 floats
    assert lib.pa_decode_workspace_bytes(4, 1, 1, 64, 16, 4, 0) >= 4 * 8 + 2 * 1024 * 68 * 4
    assert lib.pa_decode_workspace_bytes(64, 32, 8, 128, 16, 129, 513) == 0


def test_cache_ops_reject(libpa):
    lib = libpa.lib()
    assert lib.pa_append_kv(NULL, NULL, NULL, NULL, NULL, 4, 8, 100, 16, 64, 0, NULL) == 4
    assert lib.pa_append_kv(NULL, NULL, NULL, NULL, NULL, -1, 8, 128, 16, 64, 0, NULL) == 1
    assert lib.pa_append_kv(NULL, NULL, NULL, NULL, NULL, 0, 8, 128, 16, 64, 0, NULL) == 0
    assert lib.pa_append_kv(NULL, NULL, NULL, NULL, NULL, 4, 8, 128, 16, 64, 0, NULL) == 1
    assert lib.pa_copy_blocks(NULL, NULL, NULL, 3, 0, 128, 16, 64, 0, NULL) == 1
    assert lib.pa_copy_blocks(NULL, NULL, NULL, 0, 8, 128, 16, 64, 0, NULL) == 0
    assert lib.pa_copy_blocks(NULL, NULL, NULL, 2, 8, 128, 16, 64, 0, NULL) == 1


# Stand-in addresses: every call below is refused by a host check that runs
# before any device work, so they are never dereferenced.
_K = 0x10000000
_E = 16 * 8 * 128          # values in one block of the shape used below


@pytest.mark.parametrize("v_off,stride,msg", [
    (64 * _E * 2, _E - 8, b"pool_block_stride"),     # shorter than a block
    (64 * _E * 2, _E + 4, b"pool_block_stride"),     # not a multiple of 16 bytes
    (64 * _E * 2 - 16, 0, b"overlap"),               # dense pools that overlap by 16 bytes
    (16, 2 * _E, b"overlap"),                        # records with V one vector into K
    (4 * _E - 16, 2 * _E, b"overlap"),               # V's end runs into the next record
])
def test_pool_layout_rejects(libpa, v_off, stride, msg):
    """Strided and record pools: strides shorter than a block or not a
    multiple of 16 bytes, and K blocks that overlap V blocks (v_off in bytes),
    are refused."""
    lib = libpa.lib()
    k = ctypes.c_void_p(_K)
    v = ctypes.c_void_p(_K + v_off)
    src = ctypes.c_void_p(0x20000000)
    slots = ctypes.c_void_p(0x30000000)
    assert lib.pa_append_kv(src, src, k, v, slots, 4, 8, 128, 16, 64, stride, NULL) == 1
    assert msg in lib.pa_last_error()
    assert lib.pa_copy_blocks(k, v, slots, 2, 8, 128, 16, 64, stride, NULL) == 1
    assert msg in lib.pa_last_error()


def test_record_pool_stride_is_accepted_up_to_the_device(libpa):
    """The record layout (v = k + one block, stride two blocks) passes every
    host check; without a GPU the call then stops at the device query."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("would launch on stand-in addresses")
    lib = libpa.lib()
    k = ctypes.c_void_p(_K)
    v = ctypes.c_void_p(_K + _E * 2)
    slots = ctypes.c_void_p(0x30000000)
    st = lib.pa_copy_blocks(k, v, slots, 2, 8, 128, 16, 64, 2 * _E, NULL)
    assert st == 5 and b"overlap" not in lib.pa_last_error()


def test_decode_rejects_bad_strides(libpa):
    lib = libpa.lib()
    assert _decode(lib, stride=_E - 8) == 1
    assert b"pool_block_stride" in lib.pa_last_error()
    assert _decode(lib, stride=_E + 4) == 1
    assert b"pool_block_stride" in lib.pa_last_error()
    assert _decode_fp8(lib, stride=_E + 8) == 1          # fp8: 8 bytes is not 16
    assert b"pool_block_stride" in lib.pa_last_error()


def _decode_fp8(lib, **kw):
    a = dict(q=NULL, k=NULL, v=NULL, ks=NULL, vs=NULL, table=NULL, lens=NULL, S=4, Hq=32, Hkv=8,
             D=128, BS=16, MB=8, NB=64, stride=0, scale=0.1, out=NULL, ws=NULL, wsb=0, pt=0,
             stream=NULL)
    a.update(kw)
    return lib.pa_decode_attention_fp8(a["q"], a["k"], a["v"], a["ks"], a["vs"], a["table"],
                                       a["lens"], a["S"], a["Hq"], a["Hkv"], a["D"], a["BS"],
                                       a["MB"], a["NB"], a["stride"], ctypes.c_float(a["scale"]),
                                       a["out"], a["ws"], a["wsb"], a["pt"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(Hq=30), 1),
    (dict(D=96), 4),
    (dict(BS=64), 4),
    (dict(), 1),                      # NULL pointers
])
def test_decode_fp8_rejects(libpa, kw, status):
    lib = libpa.lib()
    assert _decode_fp8(lib, **kw) == status
    assert lib.pa_last_error() != b""


def test_decode_fp8_zero_sequences_is_a_no_op(libpa):
    assert _decode_fp8(libpa.lib(), S=0) == 0


def test_cache_ops_fp8_reject(libpa):
    lib = libpa.lib()
    # NULL scales / pools with work to do
    assert lib.pa_append_kv_fp8(NULL, NULL, NULL, NULL, NULL, NULL, NULL, 4, 8, 128, 16, 64,
                                0, NULL) == 1
    assert lib.pa_append_kv_fp8(NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, 8, 128, 16, 64,
                                0, NULL) == 0
    assert lib.pa_copy_blocks_fp8(NULL, NULL, NULL, 0, 8, 128, 16, 64, 0, NULL) == 0
    assert lib.pa_copy_blocks_fp8(NULL, NULL, NULL, 2, 8, 120, 16, 64, 0, NULL) == 4  # 120 % 16
    assert lib.pa_copy_blocks_fp8(NULL, NULL, NULL, 2, 8, 128, 16, 64, 0, NULL) == 1


# pa_decode_append_attention: the attention call's checks, then its own
# arguments (the new rows and their slots) and the pools' disjointness, all
# before any device query. Fake aligned addresses stand for the arrays.
_FAKE = dict(q=0x10000, k=0x20000000, v=0x40000000, table=0x60000, lens=0x70000, out=0x80000)


def _append_attn(lib, **kw):
    a = dict(q=NULL, kn=NULL, vn=NULL, slots=NULL, k=NULL, v=NULL, table=NULL, lens=NULL, S=4,
             Hq=32, Hkv=8, D=128, BS=16, MB=8, NB=64, stride=0, scale=0.1, out=NULL, ws=NULL,
             wsb=0, pt=0, stream=NULL)
    a.update(kw)
    return lib.pa_decode_append_attention(
        a["q"], a["kn"], a["vn"], a["slots"], a["k"], a["v"], a["table"], a["lens"], a["S"],
        a["Hq"], a["Hkv"], a["D"], a["BS"], a["MB"], a["NB"], a["stride"],
        ctypes.c_float(a["scale"]), a["out"], a["ws"], a["wsb"], a["pt"], a["stream"])


@pytest.mark.parametrize("kw,status,msg", [
    (dict(), 1, b"NULL pointer"),                                   # the attention's arrays
    (dict(_FAKE, D=96), 4, b""),                                    # an unsupported shape
    (dict(_FAKE, scale=float("nan")), 1, b"scale"),
    (dict(_FAKE), 1, b"NULL k_new"),                                # the new rows and slots
    (dict(_FAKE, kn=0x90000, vn=0xA0000), 1, b"NULL k_new"),
    (dict(_FAKE, kn=0x90008, vn=0xA0000, slots=0xB0000), 1, b"misaligned k_new"),
    (dict(_FAKE, kn=0x90000, vn=0xA0000, slots=0xB0002), 1, b"misaligned k_new"),
    # V one block past K: every block of the two pools overlaps the other's
    (dict(_FAKE, v=0x20000000 + 32 * 1024, kn=0x90000, vn=0xA0000, slots=0xB0000), 1,
     b"overlap"),
])
def test_append_attention_rejects(libpa, kw, status, msg):
    lib = libpa.lib()
    assert _append_attn(lib, **kw) == status
    assert msg in lib.pa_last_error()


def test_append_attention_zero_sequences_is_a_no_op(libpa):
    assert _append_attn(libpa.lib(), S=0) == 0


def _step(lib, handle, ids, mb, nb, ncow, **kw):
    a = dict(slots=NULL, pairs=NULL, table=NULL, lens=NULL, q=NULL, kn=NULL, vn=NULL, k=NULL,
             v=NULL, Hq=32, Hkv=8, D=128, stride=0, scale=0.1, out=NULL, ws=NULL, wsb=0, pt=0,
             stream=NULL)
    a.update(kw)
    return lib.pa_decode_step(handle, ids.ctypes.data if ids is not None else NULL,
                              0 if ids is None else len(ids), mb, a["slots"], a["pairs"],
                              a["table"], a["lens"], ctypes.byref(ncow), a["q"], a["kn"], a["vn"],
                              a["k"], a["v"], a["Hq"], a["Hkv"], a["D"], nb, a["stride"],
                              ctypes.c_float(a["scale"]), a["out"], a["ws"], a["wsb"], a["pt"],
                              a["stream"])


def test_decode_step_refuses_before_planning(libpa):
    """pa_decode_step checks its handle and that the pool is the block
    manager's before it plans anything, and a plan that cannot be made
    (a table narrower than a sequence's blocks) changes nothing."""
    import numpy as np
    lib = libpa.lib()
    ncow = ctypes.c_int(7)
    assert _step(lib, NULL, None, 4, 64, ncow) == 1
    a = libpa.BlockAllocator(64, 16)
    a.add_seq(0, 40)                   # three blocks of 16 tokens
    a.add_seq(1, 16)                   # a full block: the next token opens a second
    ids = np.array([0, 1], np.int64)
    before = a.export_state()
    slots = np.zeros(2, np.int32)
    pairs = np.zeros((2, 2), np.int32)
    lens = np.zeros(2, np.int32)
    table = np.zeros((2, 4), np.int32)
    bufs = dict(slots=slots.ctypes.data, pairs=pairs.ctypes.data, table=table.ctypes.data,
                lens=lens.ctypes.data)
    # the pool is not the block manager's
    assert _step(lib, a._h, ids, 4, 32, ncow, **bufs) == 1
    assert b"block manager" in lib.pa_last_error()
    assert ncow.value == 0
    # sequence 0 needs three table columns: two are refused, all or nothing
    narrow = np.zeros((2, 2), np.int32)
    bufs_n = dict(bufs, table=narrow.ctypes.data)
    assert _step(lib, a._h, ids, 2, 64, ncow, **bufs_n) == 1
    assert b"needs more than 2 blocks" in lib.pa_last_error()
    assert a.export_state() == before
