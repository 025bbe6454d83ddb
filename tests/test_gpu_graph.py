"""A decode step captured once in a CUDA graph and replayed: the replays reuse
the kernels' parameters (including the call tag of the arrival counters) and
must give, replay after replay with new queries, the same output bit for bit
as an eager call on the same inputs. Covers the plain step (copy, append,
attention), the shared-prefix step (two attention kernels with a
programmatic edge) and the allocation-free entry point."""

import numpy as np
import pytest

import synthetic

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def pa(libpa):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return libpa


def _capture(run):
    run.run_step()                      # eager first: one-time setup stays outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        run.run_step(stream=s)
    torch.cuda.synchronize()
    return g


def test_plain_step_replays(pa):
    from paged_kv_cache_40_gb300.engine import DecodeBatchRunner
    b = synthetic.config2_gqa_batch(num_seqs=9, lo=1, hi=700)
    run = DecodeBatchRunner(b)
    run.plan_step()
    g = _capture(run)
    gen = torch.Generator(device="cuda").manual_seed(5)
    for _ in range(4):
        run.q.copy_(torch.randn(run.q.shape, generator=gen, device="cuda").half())
        g.replay()
        torch.cuda.synchronize()
        eager = pa.pa_decode_attention(run.q, run.k_pool, run.v_pool, run.d_table, run.d_lens,
                                       float(b.scale))
        torch.cuda.synchronize()
        assert torch.equal(run.out, eager)
    assert pa.pa_device_error() == 0


def test_shared_prefix_step_replays(pa):
    from paged_kv_cache_40_gb300.engine import SharedPrefixRunner
    w = synthetic.config4_shared_prefix()
    run = SharedPrefixRunner(w)
    run.plan_step()
    g = _capture(run)
    gen = torch.Generator(device="cuda").manual_seed(6)
    for _ in range(3):
        run.q.copy_(torch.randn(run.q.shape, generator=gen, device="cuda").half())
        g.replay()
        torch.cuda.synchronize()
        eager = pa.pa_decode_attention_shared_prefix(run.q, run.k_pool, run.v_pool, run.d_prefix,
                                                     run.d_table, run.d_lens, float(w.scale))
        torch.cuda.synchronize()
        assert torch.equal(run.out, eager)
    assert pa.pa_device_error() == 0


def test_fixed_scratch_call_replays(pa):
    b = synthetic.config2_gqa_batch(num_seqs=6, lo=1, hi=1500)
    from paged_kv_cache_40_gb300.engine import DecodeBatchRunner
    run = DecodeBatchRunner(b)
    run.plan_step()
    run.run_step()
    out = torch.empty_like(run.q)
    pa.pa_decode_attention_fixed_scratch(run.q, run.k_pool, run.v_pool, run.d_table, run.d_lens,
                                         float(b.scale), out=out)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        pa.pa_decode_attention_fixed_scratch(run.q, run.k_pool, run.v_pool, run.d_table,
                                             run.d_lens, float(b.scale), out=out, stream=s)
    gen = torch.Generator(device="cuda").manual_seed(7)
    for _ in range(3):
        run.q.copy_(torch.randn(run.q.shape, generator=gen, device="cuda").half())
        g.replay()
        torch.cuda.synchronize()
        eager = pa.pa_decode_attention(run.q, run.k_pool, run.v_pool, run.d_table, run.d_lens,
                                       float(b.scale))
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
