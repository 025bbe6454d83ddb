"""Reference block manager: free list, reference counts, block tables.

Test infrastructure only (see the package docstring).

What the pages fix:
  * Blocks come from a pool of same-size physical blocks; a sequence's table
    maps logical block -> physical id ("Phase 7 · Document 04 —
    PagedAttention", §2 Core Concept; lux-666 notes "PagedAttention", 最小模型).
  * Allocation is on demand: a growing sequence takes one more block; a
    finished one frees its blocks at once (same passages).
  * A request of len tokens needs ceil(len / block_size) blocks (lux-666 notes,
    "block size 是容量与 kernel 的共同参数").
  * Prefix sharing points several tables at the same blocks, kept alive by
    reference counts; a write into a shared block copies that block first
    (Document 04, §2 "block sharing (copy-on-write)" and §3 Mental Model;
    lux-666 notes, prefix sharing section).

Readings taken where the pages are silent:
  * The free list is FIFO: allocation pops the front, a block whose count
    drops to zero is pushed to the back. A sequence's blocks are released in
    logical order. The initial order is given (default ascending).
  * A new block is taken exactly when the sequence's length is a multiple of
    the block size before the append.
  * Copy-on-write happens iff the block to be written has reference count > 1
    at write time; the writer gets a fresh block, the pair (old, new) is
    recorded and the old block's count drops by one. The last holder therefore
    writes in place.
  * Every operation is all-or-nothing: when the free list is too short the
    state is left unchanged and OutOfBlocks is raised.

Swapping (Document 04, §9/§10: under memory pressure a scheduler may preempt
a sequence by swapping its blocks out; the pages give no mechanism). Readings:
  * The manager also owns a pool of host blocks with its own FIFO free list.
  * swap_out(seq) takes one host block per logical block (in logical order),
    returns the (device, host) pairs to copy, then drops the sequence's device
    references in logical order: a block other tables still reference stays
    on the device for them. The sequence keeps its length; it cannot append,
    fork or appear in a table until it is swapped back in.
  * swap_in(seq) takes fresh device blocks (private: sharing is not restored),
    returns the (host, device) pairs to copy, then returns the host blocks to
    the host free list in logical order.
  * Freeing a swapped-out sequence returns its host blocks.
"""

from __future__ import annotations

from collections import deque
from typing import Dict, List, Optional, Tuple


class OutOfBlocks(RuntimeError):
    pass


class BlockAllocator:
    def __init__(self, num_blocks: int, block_size: int,
                 initial_free_order=None):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        order = list(range(num_blocks)) if initial_free_order is None else \
            [int(b) for b in initial_free_order]
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("initial free order must be a permutation of the pool")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.free: deque = deque(order)
        self.ref: List[int] = [0] * num_blocks
        self.tables: Dict[int, List[int]] = {}
        self.lens: Dict[int, int] = {}
        self.cow_copies = 0
        self.alloc_failures = 0
        self.host_free: deque = deque()
        self.num_host_blocks = 0
        self.host_tables: Dict[int, List[int]] = {}
        self.swap_outs = 0
        self.swap_ins = 0

    # -- helpers ------------------------------------------------------------
    def _take(self) -> int:
        b = self.free.popleft()
        self.ref[b] = 1
        return b

    def _release(self, b: int) -> None:
        self.ref[b] -= 1
        if self.ref[b] == 0:
            self.free.append(b)

    def _blocks_for(self, length: int) -> int:
        return -(-length // self.block_size)

    # -- operations ---------------------------------------------------------
    def add_seq(self, seq: int, length: int) -> None:
        """Register a sequence already holding `length` tokens."""
        if seq in self.lens or length < 0:
            raise ValueError("sequence exists or negative length")
        n = self._blocks_for(length)
        if n > len(self.free):
            self.alloc_failures += 1
            raise OutOfBlocks(f"need {n} blocks, {len(self.free)} free")
        self.tables[seq] = [self._take() for _ in range(n)]
        self.lens[seq] = length

    def fork(self, parent: int, child: int) -> None:
        """The child shares every block of the parent (counts + 1)."""
        if parent not in self.tables or child in self.lens:
            raise ValueError("bad fork")
        tab = list(self.tables[parent])
        for b in tab:
            self.ref[b] += 1
        self.tables[child] = tab
        self.lens[child] = self.lens[parent]

    def append_slot(self, seq: int) -> Tuple[int, int, int]:
        """Reserve the slot of the sequence's next token.

        Returns (slot, cow_src, cow_dst); cow_src = cow_dst = -1 when no copy
        is needed.
        """
        if seq not in self.tables:
            raise ValueError("unknown or swapped-out sequence")
        L = self.lens[seq]
        tab = self.tables[seq]
        BS = self.block_size
        cow_src = cow_dst = -1
        if L % BS == 0:
            if not self.free:
                self.alloc_failures += 1
                raise OutOfBlocks("no free block for growth")
            tab.append(self._take())
        else:
            last = tab[L // BS]
            if self.ref[last] > 1:
                if not self.free:
                    self.alloc_failures += 1
                    raise OutOfBlocks("no free block for copy-on-write")
                new = self._take()
                self.ref[last] -= 1
                tab[L // BS] = new
                cow_src, cow_dst = last, new
                self.cow_copies += 1
        slot = tab[L // BS] * BS + L % BS
        self.lens[seq] = L + 1
        return slot, cow_src, cow_dst

    def free_seq(self, seq: int) -> None:
        """Release every block of the sequence, in logical order (host
        blocks if it is swapped out)."""
        if seq in self.host_tables:
            for h in self.host_tables.pop(seq):
                self.host_free.append(h)
            self.lens.pop(seq)
            return
        tab = self.tables.pop(seq)
        self.lens.pop(seq)
        for b in tab:
            self._release(b)

    # -- swapping -------------------------------------------------------------
    def add_host_pool(self, num_host_blocks: int, initial_free_order=None) -> None:
        if self.num_host_blocks or num_host_blocks <= 0:
            raise ValueError("host pool exists or bad size")
        order = list(range(num_host_blocks)) if initial_free_order is None else \
            [int(b) for b in initial_free_order]
        if sorted(order) != list(range(num_host_blocks)):
            raise ValueError("host free order must be a permutation of the host pool")
        self.num_host_blocks = num_host_blocks
        self.host_free = deque(order)

    def swap_out(self, seq: int) -> List[Tuple[int, int]]:
        """(device, host) block pairs to copy, in logical order; the sequence
        then holds host blocks only."""
        if seq not in self.tables:
            raise ValueError("unknown or swapped-out sequence")
        tab = self.tables[seq]
        if len(tab) > len(self.host_free):
            self.alloc_failures += 1
            raise OutOfBlocks(f"need {len(tab)} host blocks, {len(self.host_free)} free")
        hosts = [self.host_free.popleft() for _ in tab]
        pairs = list(zip(tab, hosts))
        for b in tab:
            self._release(b)
        del self.tables[seq]
        self.host_tables[seq] = hosts
        self.swap_outs += 1
        return pairs

    def swap_in(self, seq: int) -> List[Tuple[int, int]]:
        """(host, device) block pairs to copy, in logical order; the sequence
        then holds fresh device blocks."""
        if seq not in self.host_tables:
            raise ValueError("sequence is not swapped out")
        hosts = self.host_tables[seq]
        if len(hosts) > len(self.free):
            self.alloc_failures += 1
            raise OutOfBlocks(f"need {len(hosts)} blocks, {len(self.free)} free")
        devs = [self._take() for _ in hosts]
        for h in hosts:
            self.host_free.append(h)
        del self.host_tables[seq]
        self.tables[seq] = devs
        self.swap_ins += 1
        return list(zip(hosts, devs))

    def export_host_state(self) -> Tuple[List[int], int, int, int]:
        """(host free list front to back, swapped-out sequences, swap-outs,
        swap-ins)."""
        return list(self.host_free), len(self.host_tables), self.swap_outs, self.swap_ins

    # -- inspection ---------------------------------------------------------
    def table(self, seq: int) -> List[int]:
        return list(self.tables[seq])

    def seq_len(self, seq: int) -> int:
        return self.lens[seq]

    def stats(self) -> dict:
        used = sum(1 for r in self.ref if r > 0)
        return {
            "num_blocks": self.num_blocks,
            "free": len(self.free),
            "used": used,
            "shared": sum(1 for r in self.ref if r > 1),
            "cow_copies": self.cow_copies,
            "alloc_failures": self.alloc_failures,
            "total_refs": sum(self.ref),
            "num_seqs": len(self.lens),
        }

    def export_state(self) -> Tuple[List[int], List[int]]:
        """(free list front to back, reference count per block)."""
        return list(self.free), list(self.ref)

    def shared_prefix(self, seqs) -> List[int]:
        """The whole blocks every sequence of `seqs` begins with; see
        shared_prefix_blocks. Swapped-out or unknown sequences raise."""
        return shared_prefix_blocks([self.tables[s] for s in seqs],
                                    [self.lens[s] for s in seqs], self.block_size)

    def dense_table(self, seqs, max_blocks: int, fill: int = -1):
        """int32-style nested list [len(seqs)][max_blocks], padded with `fill`."""
        rows = []
        for s in seqs:
            t = self.tables[s]
            if len(t) > max_blocks:
                raise ValueError("table longer than max_blocks")
            rows.append(t + [fill] * (max_blocks - len(t)))
        return rows


def shared_prefix_blocks(tables, lens, block_size: int) -> List[int]:
    """The physical blocks that every given sequence begins with, whole.

    Sequences forked from one prompt point their tables at the same physical
    blocks ("Phase 7 · Document 04 — PagedAttention", §2 block sharing and §3
    Mental Model, where A -> [b3, b7, b1] and B -> [b3, b9] share b3; lux-666
    notes "PagedAttention", prefix sharing). Reading: the shared prefix of a
    batch is the longest run of leading table entries that is the same in
    every table and whose blocks every sequence attends in full (k blocks
    with k * block_size <= its length), so that each sequence's attention
    splits into those k * block_size tokens and the rest of its own table.
    An empty batch has none; a single sequence's whole blocks are its own.
    """
    if not tables:
        return []
    k = min(min(len(t), int(L) // block_size) for t, L in zip(tables, lens))
    first = list(tables[0])
    for t in tables[1:]:
        j = 0
        while j < k and t[j] == first[j]:
            j += 1
        k = j
    return first[:k]
