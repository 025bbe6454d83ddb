"""The attention kernel's bounded waits, made to run out on purpose: with a
short limit (pa_set_wait_limit_ns) a pipeline wait gives up, the launch
records PA_DEVERR_TIMEOUT, lets the copies it already issued land and exits,
and the context stays usable. A normal call on the same workspace afterwards
matches the oracle.

The pages' rule for a system at its limit is to fail explicitly rather than
thrash ("Phase 7 · Document 04 — PagedAttention", §11 Engineering Decision
Framework); this checks that the kernel's failure path does exactly that,
without a fault or a hang: nothing here waits on a flag that is never set,
every wait simply gets a limit shorter than the work takes."""

import numpy as np
import pytest

import oracle
import synthetic
from tests.gpu_helpers import assert_close_attention, poison_unread_rows

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def pa(libpa):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return libpa


def d(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.fixture(scope="module")
def batch():
    """The 64-sequence GQA batch (U[128, 2048] tokens, 32q/8kv, D=128):
    long enough that sequences are split over CTAs and the merge warps wait
    for the consumers' messages."""
    b = synthetic.config2_gqa_batch()
    ref = oracle.decode_step(b, compute_attention=False)
    kp, vp = poison_unread_rows(ref.k_pool, ref.v_pool, ref.block_table, ref.seq_lens,
                                b.block_size)
    return b, kp, vp, ref.block_table, ref.seq_lens


def _expect_timeout_or_clean(pa, must_time_out):
    try:
        flags = pa.pa_device_error()
    except pa.PaError as e:
        assert e.flags == pa.PA_DEVERR_TIMEOUT, hex(e.flags)
        return True
    assert not must_time_out, "the wait limit did not run out"
    assert flags == 0
    return False


@pytest.mark.parametrize("entry", ["workspace", "fixed_scratch", "fp8"])
def test_short_wait_limit_times_out_then_recovers(pa, batch, entry):
    b, kp, vp, table, lens = batch
    dq, dt, dl = d(b.q), d(table), d(lens)
    sl = [0, 9, 31, 63]
    if entry == "fp8":
        c = synthetic.fp8_cache(b)
        dk, dv, ks, vs = d(c.k_pool), d(c.v_pool), d(c.k_scale), d(c.v_scale)
        ws = pa.alloc_workspace(b.num_seqs, b.num_q_heads, b.num_kv_heads, b.head_dim,
                                b.block_size, table.shape[1])
        call = lambda: pa.pa_decode_attention_fp8(dq, dk, dv, ks, vs, dt, dl, b.scale,
                                                  workspace=ws)
        exp = oracle.decode_attention_fp8(b.q, c.k_pool, c.v_pool, c.k_scale, c.v_scale,
                                          table, lens, b.scale, seqs=sl)
    else:
        dk, dv = d(kp), d(vp)
        if entry == "workspace":
            ws = pa.alloc_workspace(b.num_seqs, b.num_q_heads, b.num_kv_heads, b.head_dim,
                                    b.block_size, table.shape[1])
            call = lambda: pa.pa_decode_attention(dq, dk, dv, dt, dl, b.scale, workspace=ws)
        else:
            call = lambda: pa.pa_decode_attention_fixed_scratch(dq, dk, dv, dt, dl, b.scale)
        exp = oracle.decode_attention(b.q, kp, vp, table, lens, b.scale, seqs=sl)
    assert pa.pa_device_error() == 0
    try:
        # 1 ns: the first wait that is not already complete gives up
        pa.pa_set_wait_limit_ns(1)
        call()
        torch.cuda.synchronize()
        assert _expect_timeout_or_clean(pa, must_time_out=True)
        # limits that run out somewhere in the middle of the stream, with
        # copies in flight, or not at all: either way no other error
        for limit in (500, 3000, 15000):
            pa.pa_set_wait_limit_ns(limit)
            call()
            torch.cuda.synchronize()
            _expect_timeout_or_clean(pa, must_time_out=False)
    finally:
        pa.pa_set_wait_limit_ns(0)
    for _ in range(2):
        out = call()
        torch.cuda.synchronize()
        assert pa.pa_device_error() == 0
        assert_close_attention(out.cpu().numpy()[sl], exp[sl], f"after timeouts ({entry})")
