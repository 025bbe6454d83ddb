"""One decode step of a batch through libpa: the host block manager assigns
slots (and copy-on-write pairs), then the device copies shared blocks, writes
the new K/V rows and runs paged decode attention.

Step order (the plain reading of "one decode step plus one append per
sequence"): reserve slots -> copy-on-write copies -> append -> attend over
every cached token including the appended one.

The batch object is any container with the fields of a decode batch:
num_blocks, block_size, num_q_heads, num_kv_heads, head_dim, prefill_lens,
free_order, churn (ops with kind/owner/nblocks), q, k_pool, v_pool, k_new,
v_new (numpy fp16) and scale.

With kv_dtype "fp8" the cache is E4M3 bytes with one fp32 scale per KV head
for K and V (given as k_pool, v_pool, k_scale, v_scale); the new tokens are
quantized by the append.

With layout "records" the cache is one pool of per-block records, each a
block's K rows then its V rows (the layout sketch of "Phase 7 · Document 04 —
PagedAttention", §2), held in `kv_pool`; `k_pool` / `v_pool` are its member
views and every call takes them as it takes two separate pools.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional, Tuple

import numpy as np

from . import (BlockAllocator, alloc_workspace, kv_block_pool, kv_views, pa_append_kv,
               pa_decode_append_attention,
               pa_append_kv_fp8, pa_copy_blocks, pa_copy_blocks_fp8, pa_decode_attention,
               pa_decode_attention_fp8, pa_decode_attention_shared_prefix,
               pa_decode_shared_prefix_workspace_bytes, pa_kernel_launches)


def _to_dev(arr, device, dtype=None):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(arr))
    if dtype is not None:
        t = t.to(dtype)
    return t.to(device)


def _device_pools(k, v, layout, device):
    """(kv_pool or None, k_pool, v_pool) on the device from host or device
    pools [NB][BS][Hkv][D]: two dense pools, or one record pool and its
    member views."""
    import torch
    dev = lambda p: p if isinstance(p, torch.Tensor) else _to_dev(p, device)
    if layout == "separate":
        return None, dev(k), dev(v)
    if layout != "records":
        raise ValueError("layout must be 'separate' or 'records'")
    kt, vt = dev(k), dev(v)
    nb, bs, h, d = (int(x) for x in kt.shape)
    kv = kv_block_pool(nb, bs, h, d, kt.dtype, device)
    kp, vp = kv_views(kv)
    kp.copy_(kt)
    vp.copy_(vt)
    return kv, kp, vp


@dataclass
class StepPlan:
    slots: np.ndarray          # int32 [S]
    cow_pairs: np.ndarray      # int32 [n][2]
    block_table: np.ndarray    # int32 [S][MB]
    seq_lens: np.ndarray       # int32 [S]


class DecodeBatchRunner:
    """Holds a batch's pools on the device and runs its decode step."""

    def __init__(self, batch, device="cuda", max_blocks: Optional[int] = None,
                 partition_tokens: int = 0, table_fill: int = -1, k_pool=None, v_pool=None,
                 kv_dtype: str = "fp16", k_scale=None, v_scale=None, layout: str = "separate"):
        import torch
        if kv_dtype not in ("fp16", "fp8"):
            raise ValueError("kv_dtype must be 'fp16' or 'fp8'")
        if kv_dtype == "fp8" and (k_pool is None or v_pool is None or k_scale is None
                                  or v_scale is None):
            raise ValueError("an fp8 cache needs k_pool, v_pool, k_scale and v_scale")
        self.kv_dtype = kv_dtype
        self.batch = batch
        self.device = torch.device(device)
        self.partition_tokens = partition_tokens
        a = BlockAllocator(batch.num_blocks, batch.block_size, batch.free_order)
        for op in getattr(batch, "churn", []):
            if op.kind == "alloc":
                a.add_seq(op.owner, op.nblocks * batch.block_size)
            else:
                a.free_seq(op.owner)
        S = int(batch.prefill_lens.shape[0])
        for i in range(S):
            a.add_seq(i, int(batch.prefill_lens[i]))
        self.alloc = a
        self.num_seqs = S
        bs = batch.block_size
        need = max(1, max(-(-(int(L) + 1) // bs) for L in batch.prefill_lens)) if S else 1
        self.max_blocks = int(max_blocks or need)
        self.table_fill = table_fill
        self.layout = layout
        self.kv_pool, self.k_pool, self.v_pool = _device_pools(
            batch.k_pool if k_pool is None else k_pool,
            batch.v_pool if v_pool is None else v_pool, layout, self.device)
        self.k_scale = _to_dev(k_scale, self.device, torch.float32) if k_scale is not None else None
        self.v_scale = _to_dev(v_scale, self.device, torch.float32) if v_scale is not None else None
        self.q = _to_dev(batch.q, self.device)
        self.k_new = _to_dev(batch.k_new, self.device)
        self.v_new = _to_dev(batch.v_new, self.device)
        self.out = torch.empty_like(self.q)
        self.workspace = alloc_workspace(S, batch.num_q_heads, batch.num_kv_heads,
                                         batch.head_dim, bs, self.max_blocks,
                                         partition_tokens, self.device)
        self.plan: Optional[StepPlan] = None

    # -- host: slot assignment ---------------------------------------------
    def plan_step(self) -> StepPlan:
        """Reserve one slot per sequence (host block manager) and upload the
        slot mapping, copy-on-write pairs and block tables."""
        import torch
        slots, pairs, table, lens = self.alloc.plan_step(np.arange(self.num_seqs, dtype=np.int64),
                                                         self.max_blocks, self.table_fill)
        plan = StepPlan(slots.copy(), pairs.copy(), table.copy(), lens.copy())
        self.plan = plan
        self.d_slots = _to_dev(plan.slots, self.device)
        self.d_pairs = _to_dev(plan.cow_pairs, self.device) if len(plan.cow_pairs) else None
        self.d_table = _to_dev(plan.block_table, self.device)
        self.d_lens = _to_dev(plan.seq_lens, self.device)
        return plan

    # -- device: the hot path ----------------------------------------------
    def copy_and_append(self, stream=None) -> None:
        fp8 = self.kv_dtype == "fp8"
        if self.d_pairs is not None:
            (pa_copy_blocks_fp8 if fp8 else pa_copy_blocks)(self.k_pool, self.v_pool, self.d_pairs,
                                                            stream=stream)
        if fp8:
            pa_append_kv_fp8(self.k_new, self.v_new, self.k_pool, self.v_pool, self.d_slots,
                             self.k_scale, self.v_scale, stream=stream)
        else:
            pa_append_kv(self.k_new, self.v_new, self.k_pool, self.v_pool, self.d_slots,
                         stream=stream)

    def step(self, stream=None):
        """The step's copy-on-write copies (if any), then the append and the
        attention: one pa_decode_append_attention kernel for an fp16 cache,
        pa_append_kv_fp8 and pa_decode_attention_fp8 for an E4M3 one."""
        if self.kv_dtype == "fp8":
            self.copy_and_append(stream)
            return self.attend(stream)
        if self.d_pairs is not None:
            pa_copy_blocks(self.k_pool, self.v_pool, self.d_pairs, stream=stream)
        pa_decode_append_attention(self.q, self.k_new, self.v_new, self.d_slots, self.k_pool,
                                   self.v_pool, self.d_table, self.d_lens,
                                   float(self.batch.scale), out=self.out,
                                   workspace=self.workspace,
                                   partition_tokens=self.partition_tokens, stream=stream)
        return self.out

    def attend(self, stream=None):
        if self.kv_dtype == "fp8":
            pa_decode_attention_fp8(self.q, self.k_pool, self.v_pool, self.k_scale, self.v_scale,
                                    self.d_table, self.d_lens, float(self.batch.scale),
                                    out=self.out, workspace=self.workspace,
                                    partition_tokens=self.partition_tokens, stream=stream)
        else:
            pa_decode_attention(self.q, self.k_pool, self.v_pool, self.d_table, self.d_lens,
                                float(self.batch.scale), out=self.out, workspace=self.workspace,
                                partition_tokens=self.partition_tokens, stream=stream)
        return self.out

    # -- host <-> device: one copy of the step's inputs ----------------------
    def pack_inputs(self) -> None:
        """Re-home the step's inputs (q, the new K/V rows, slots, copy pairs,
        tables, lengths; call after plan_step) in one device buffer with a
        pinned host mirror of the same layout (`packed_host`, views by
        name), so that
        upload_inputs() moves a step's inputs with a single host-to-device
        copy."""
        import torch
        names = ["q", "k_new", "v_new", "d_slots", "d_table", "d_lens"]
        if self.d_pairs is not None:
            names.append("d_pairs")
        offs, pos = [], 0
        for n in names:
            t = getattr(self, n)
            offs.append(pos)
            pos += (t.numel() * t.element_size() + 255) // 256 * 256
        dev_arena = torch.empty(pos, dtype=torch.uint8, device=self.device)
        host_arena = torch.empty(pos, dtype=torch.uint8).pin_memory()
        self.packed_host = {}
        for n, off in zip(names, offs):
            t = getattr(self, n)
            nb = t.numel() * t.element_size()
            dv = dev_arena[off:off + nb].view(t.dtype).view(t.shape)
            dv.copy_(t)
            hv = host_arena[off:off + nb].view(t.dtype).view(t.shape)
            hv.copy_(t.cpu())
            setattr(self, n, dv)
            self.packed_host[n] = hv
        self.input_arena, self.host_arena = dev_arena, host_arena

    def host_inputs(self) -> int:
        """Keep the step's inputs (q, the new K/V rows, slots, copy pairs,
        tables, lengths, the shared prefix's block list; call after
        plan_step) in pinned host memory, where the kernels read them
        through its device mapping over the CPU-GPU link: a step then needs
        no host-to-device copy call. Returns their bytes."""
        names = ["q", "k_new", "v_new", "d_slots", "d_table", "d_lens"]
        if self.d_pairs is not None:
            names.append("d_pairs")
        if getattr(self, "d_prefix", None) is not None:
            names.append("d_prefix")
        total = 0
        for n in names:
            h = getattr(self, n).cpu().pin_memory()
            setattr(self, n, h)
            total += h.numel() * h.element_size()
        return total

    def host_planned(self, sets: int = 2) -> int:
        """Plan every step straight into pinned host memory: `sets` rotating
        sets of buffers for the slot mapping, copy pairs, tables and lengths,
        which plan_step_host() fills with one block-manager call
        (pa_alloc_plan_step) and the kernels read in place through their
        device mapping; q and the new K/V rows stay in pinned host memory
        too. With two sets, step k+1 can be planned while the kernels of step
        k still read theirs; a set is written again only once the kernels that
        read it last have completed (see _take_plan_set). Returns the input
        bytes of one step."""
        import torch
        S, mb = self.num_seqs, self.max_blocks
        pin = lambda shape: torch.empty(shape, dtype=torch.int32).pin_memory()
        self._plan_sets = [(pin((S,)), pin((S, 2)), pin((S, mb)), pin((S,))) for _ in range(sets)]
        self._plan_views = [tuple(t.numpy() for t in st) for st in self._plan_sets]
        self._plan_ids = np.arange(S, dtype=np.int64)
        self._plan_next = 0
        self._plan_marks = [torch.cuda.Event() for _ in range(sets)]
        self._plan_marked = [False] * sets
        self._plan_stream = None
        total = 0
        for n in ("q", "k_new", "v_new"):
            h = getattr(self, n).cpu().pin_memory()
            setattr(self, n, h)
            total += h.numel() * h.element_size()
        return total + S * 4 * (1 + 2 + mb + 1)

    def prepare_native_steps(self, stream=None) -> None:
        """After host_planned(): one PreparedDecodeStep per set of plan
        buffers, so that run_native_step() plans and enqueues a whole step
        (copies, append, attention) in one library call."""
        from . import PreparedDecodeStep
        fp8 = self.kv_dtype == "fp8"
        self._native = [PreparedDecodeStep(self.alloc, self._plan_ids, self.max_blocks, st,
                                           self.q, self.k_new, self.v_new, self.k_pool,
                                           self.v_pool, float(self.batch.scale), self.out,
                                           self.workspace, self.partition_tokens, stream,
                                           k_scale=self.k_scale if fp8 else None,
                                           v_scale=self.v_scale if fp8 else None)
                        for st in self._plan_sets]
        import torch
        # the stream the prepared steps launch on (resolved as they resolved it)
        self._plan_stream = stream if stream is not None else torch.cuda.current_stream()

    def _take_plan_set(self) -> int:
        """Index of the next set of plan buffers, once the kernels that read it
        last have completed: each call first marks, with an event on the
        stream, the work enqueued so far (which includes the kernels that read
        the set planned last), then waits for the mark left on the set it is
        about to write. Host memory the kernels read in place is never
        rewritten under them, however far the host runs ahead."""
        import torch
        n = len(self._plan_sets)
        k = self._plan_next % n
        stream = self._plan_stream or torch.cuda.current_stream()
        if self._plan_next > 0:
            prev = (self._plan_next - 1) % n
            self._plan_marks[prev].record(stream)
            self._plan_marked[prev] = True
        if self._plan_marked[k]:
            self._plan_marks[k].synchronize()
        self._plan_next += 1
        return k

    def run_native_step(self) -> StepPlan:
        """One decode step through pa_decode_step (see prepare_native_steps);
        returns the plan it wrote (views of that set's pinned buffers)."""
        k = self._take_plan_set()
        ncow = self._native[k]()
        v = self._plan_views[k]
        S = self.num_seqs
        self.plan = StepPlan(v[0][:S], v[1][:ncow], v[2][:S], v[3][:S])
        return self.plan

    def plan_step_host(self) -> StepPlan:
        """One decode step planned by the block manager in a single call into
        the next set of pinned buffers (see host_planned); the step's kernels
        then read that set."""
        k = self._take_plan_set()
        slots, pairs, table, lens = self.alloc.plan_step(self._plan_ids, self.max_blocks,
                                                         self.table_fill, out=self._plan_views[k])
        st = self._plan_sets[k]
        self.d_slots, self.d_table, self.d_lens = st[0][:self.num_seqs], st[2][:self.num_seqs], \
            st[3][:self.num_seqs]
        self.d_pairs = st[1][:len(pairs)] if len(pairs) else None
        self.plan = StepPlan(slots, pairs, table, lens)
        return self.plan

    def upload_inputs(self, stream=None) -> int:
        """One host-to-device copy of the packed inputs; returns its bytes."""
        import torch
        if stream is None:
            self.input_arena.copy_(self.host_arena, non_blocking=True)
        else:
            with torch.cuda.stream(stream):
                self.input_arena.copy_(self.host_arena, non_blocking=True)
        return int(self.host_arena.numel())

    def run_step(self, stream=None):
        """copy-on-write copies (if any), append, attend (see step()).
        Returns how many kernels the library launched for it."""
        n0 = pa_kernel_launches()
        self.step(stream)
        return pa_kernel_launches() - n0

    def kv_bytes(self) -> int:
        """Algorithmic K+V bytes one attention launch reads."""
        b = self.batch
        esize = 1 if self.kv_dtype == "fp8" else 2
        return int(self.plan.seq_lens.astype(np.int64).sum()) * b.num_kv_heads * b.head_dim * esize * 2

    def io_bytes(self) -> int:
        """Algorithmic bytes of one attention launch: K/V rows attended, q,
        out, the table entries used and the lengths."""
        b = self.batch
        lens = self.plan.seq_lens.astype(np.int64)
        table_entries = int(sum(-(-int(L) // b.block_size) for L in lens))
        return (self.kv_bytes() + 2 * self.q.numel() * 2 + table_entries * 4 + lens.size * 4)


class SharedPrefixRunner(DecodeBatchRunner):
    """The first decode step of sequences that share one prompt prefix.

    Sequence 0 holds the prefix; sequences 1..S-1 are forks of it, so every
    prefix block is referenced by all S block tables ("Phase 7 · Document 04
    — PagedAttention", §2 block sharing and §3 Mental Model). The step appends
    one token per sequence: the prefix's partial last block is copied for
    every holder but the last, which writes in place (copy-on-write), then all
    sequences attend over prefix + new token. Repeating the step repeats the
    same copies and writes, so it can be timed in a loop.

    The workload object provides num_blocks, block_size, num_q_heads,
    num_kv_heads, head_dim, prefix_len, num_seqs, free_order, k_pool, v_pool,
    scale and step_inputs(step, num_active) -> (q, k_new, v_new).
    """

    def __init__(self, workload, device="cuda", partition_tokens: int = 0,
                 prefix_aware: bool = True, layout: str = "separate"):
        import torch
        w = workload
        self.prefix_aware = prefix_aware
        self.kv_dtype = "fp16"
        self.batch = w
        self.device = torch.device(device)
        self.partition_tokens = partition_tokens
        self.num_seqs = int(w.num_seqs)
        a = BlockAllocator(w.num_blocks, w.block_size, w.free_order)
        a.add_seq(0, int(w.prefix_len))
        for c in range(1, self.num_seqs):
            a.fork(0, c)
        self.alloc = a
        self.max_blocks = -(-(int(w.prefix_len) + 1) // w.block_size)
        self.table_fill = -1
        self.layout = layout
        self.kv_pool, self.k_pool, self.v_pool = _device_pools(w.k_pool, w.v_pool, layout,
                                                               self.device)
        self.k_scale = self.v_scale = None
        q, kn, vn = w.step_inputs(0, self.num_seqs)
        self.q = _to_dev(q, self.device)
        self.k_new = _to_dev(kn, self.device)
        self.v_new = _to_dev(vn, self.device)
        self.out = torch.empty_like(self.q)
        self.workspace = alloc_workspace(self.num_seqs, w.num_q_heads, w.num_kv_heads,
                                         w.head_dim, w.block_size, self.max_blocks,
                                         partition_tokens, self.device)
        # the full blocks of the prefix, shared by every table
        self.num_prefix_blocks = int(w.prefix_len) // w.block_size
        if prefix_aware:
            n = pa_decode_shared_prefix_workspace_bytes(self.num_seqs, w.num_q_heads,
                                                        w.num_kv_heads, w.head_dim, w.block_size,
                                                        self.max_blocks, self.num_prefix_blocks)
            self.workspace = torch.zeros(max(n, 16), dtype=torch.uint8, device=self.device)
        self.plan = None

    def plan_step(self):
        plan = super().plan_step()
        self.d_prefix = _to_dev(plan.block_table[0, :self.num_prefix_blocks].astype(np.int32),
                                self.device)
        return plan

    def step(self, stream=None):
        """The copies, the append, then the prefix-aware attention (or the
        generic one)."""
        self.copy_and_append(stream)
        return self.attend(stream)

    def attend(self, stream=None):
        if not self.prefix_aware:
            return super().attend(stream)
        pa_decode_attention_shared_prefix(self.q, self.k_pool, self.v_pool, self.d_prefix,
                                          self.d_table, self.d_lens, float(self.batch.scale),
                                          out=self.out, workspace=self.workspace, stream=stream)
        return self.out

    def prefix_flops(self) -> int:
        """Tensor-core flops of the shared prefix's contraction in one call:
        S = Q K^T and O = P V over every (sequence, query head) row and
        every prefix token, 2 flops per multiply-add."""
        w = self.batch
        tokens = self.num_prefix_blocks * w.block_size
        return 2 * 2 * self.num_seqs * w.num_q_heads * tokens * w.head_dim

    def unique_kv_bytes(self) -> int:
        """K+V bytes of the distinct rows the step attends (the shared prefix
        once, plus each sequence's private copy of the last block)."""
        w = self.batch
        rows = int(w.prefix_len) + self.num_seqs * (int(w.prefix_len) % w.block_size + 1)
        return rows * w.num_kv_heads * w.head_dim * 2 * 2
