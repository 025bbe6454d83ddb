// Host block manager: FIFO free list, reference counts, per-sequence tables.
//
// Follows "Phase 7 · Document 04 — PagedAttention", §2 Core Concept (a pool of
// same-size physical blocks handed out on demand and returned as soon as a
// sequence finishes; one table per sequence from logical block to physical
// id; prefix sharing by pointing several tables at one block and copying the
// block on the first divergent write) and lux-666 notes "PagedAttention"
// (最小模型: any free physical block can back a logical block; the block-size
// section: ceil(len / block_size) blocks per request; the prefix-sharing
// section: reference counts, copy-on-write at the fork boundary).
//
// The free list is a ring buffer over the pool ids (a FIFO): every id is in
// the ring at most once, so a ring of num_blocks entries never overflows.
// All state changes are all-or-nothing; a refused request leaves the state
// as it was.
//
// Swapping (Document 04, §9/§10: under memory pressure a scheduler may
// preempt a sequence by swapping its blocks): an optional host pool with its
// own FIFO ring. Swap-out takes one host block per logical block, reports
// the (device, host) pairs to copy and drops the sequence's device
// references (blocks other tables share stay for them); swap-in takes fresh
// private device blocks, reports the (host, device) pairs and returns the
// host blocks. A swapped-out sequence keeps its length but cannot append,
// fork or be tabled until it is swapped back in.
#include <algorithm>
#include <unordered_map>
#include <vector>

#include "pa_internal.h"

struct pa_allocator {
  int num_blocks = 0;
  int block_size = 0;
  // FIFO free list as a ring
  std::vector<int32_t> ring;
  int64_t head = 0;   // index of the front element
  int64_t count = 0;  // elements in the ring
  std::vector<int32_t> ref;
  struct Seq {
    std::vector<int32_t> table;  // device blocks (empty while swapped out)
    std::vector<int32_t> host;   // host blocks while swapped out
    int64_t len = 0;
    bool swapped = false;
    uint64_t plan_mark = 0;      // last step plan that listed this sequence
  };
  // step planning (pa_alloc_plan_step): the plans made so far, the batch's
  // sequences, and per block the batch's writes into it (zero between calls)
  uint64_t plans = 0;
  std::vector<Seq*> plan_seqs;
  std::vector<int32_t> plan_writes;
  std::vector<int32_t> plan_blocks;
  // host pool: FIFO ring as above
  int num_host = 0;
  std::vector<int32_t> hring;
  int64_t hhead = 0, hcount = 0;
  int64_t swapped_seqs = 0, swap_outs = 0, swap_ins = 0;
  int32_t host_take() {
    int32_t h = hring[hhead];
    hhead = (hhead + 1) % num_host;
    --hcount;
    return h;
  }
  void host_push(int32_t h) {
    hring[(hhead + hcount) % num_host] = h;
    ++hcount;
  }
  std::unordered_map<int64_t, Seq> seqs;
  int64_t cow_copies = 0;
  int64_t alloc_failures = 0;
  int64_t shared = 0;  // blocks with ref > 1
  int64_t used = 0;    // blocks with ref > 0
  int64_t total_refs = 0;

  int32_t take() {
    int32_t b = ring[head];
    head = (head + 1) % num_blocks;
    --count;
    ref[b] = 1;
    ++used;
    ++total_refs;
    return b;
  }
  void push_back(int32_t b) {
    ring[(head + count) % num_blocks] = b;
    ++count;
  }
  void inc(int32_t b) {
    if (ref[b] == 1) ++shared;
    ++ref[b];
    ++total_refs;
  }
  void dec(int32_t b) {
    --ref[b];
    --total_refs;
    if (ref[b] == 1) --shared;
    if (ref[b] == 0) {
      --used;
      push_back(b);
    }
  }
  int64_t blocks_for(int64_t len) const { return (len + block_size - 1) / block_size; }
};

namespace {
pa_status check_handle(const pa_allocator* a) {
  if (!a) return pa::fail(PA_ERR_INVALID_ARG, "allocator handle is NULL");
  return PA_OK;
}

pa_status append_to(pa_allocator* a, pa_allocator::Seq& s, int64_t seq_id, int32_t* slot,
                    int32_t* cs, int32_t* cd);

pa_status append_one(pa_allocator* a, int64_t seq_id, int32_t* slot, int32_t* cs,
                     int32_t* cd) {
  auto it = a->seqs.find(seq_id);
  if (it == a->seqs.end())
    return pa::fail(PA_ERR_INVALID_ARG, "append_slot: unknown sequence %lld",
                    (long long)seq_id);
  auto& s = it->second;
  if (s.swapped)
    return pa::fail(PA_ERR_INVALID_ARG, "append_slot: sequence %lld is swapped out",
                    (long long)seq_id);
  return append_to(a, s, seq_id, slot, cs, cd);
}

// The next token of sequence s (not swapped out): grow its table when its
// length is a multiple of the block size, copy-on-write when the block it
// writes is shared, then the slot of that token.
pa_status append_to(pa_allocator* a, pa_allocator::Seq& s, int64_t seq_id, int32_t* slot,
                    int32_t* cs, int32_t* cd) {
  const int64_t L = s.len;
  const int BS = a->block_size;
  int32_t src = -1, dst = -1;
  if (L % BS == 0) {
    if (a->count == 0) {
      ++a->alloc_failures;
      return pa::fail(PA_ERR_OUT_OF_BLOCKS, "append_slot: no free block to grow sequence %lld",
                      (long long)seq_id);
    }
    s.table.push_back(a->take());
  } else {
    const int32_t last = s.table[L / BS];
    if (a->ref[last] > 1) {
      if (a->count == 0) {
        ++a->alloc_failures;
        return pa::fail(PA_ERR_OUT_OF_BLOCKS,
                        "append_slot: no free block for copy-on-write of sequence %lld",
                        (long long)seq_id);
      }
      const int32_t fresh = a->take();
      a->dec(last);  // count stays >= 1: never returns to the free list here
      s.table[L / BS] = fresh;
      src = last;
      dst = fresh;
      ++a->cow_copies;
    }
  }
  *slot = s.table[L / BS] * BS + static_cast<int32_t>(L % BS);
  *cs = src;
  *cd = dst;
  s.len = L + 1;
  return PA_OK;
}
}  // namespace

namespace pa {
int alloc_block_size(const pa_allocator* a) { return a->block_size; }
int alloc_num_blocks(const pa_allocator* a) { return a->num_blocks; }
}  // namespace pa

extern "C" {

pa_status pa_alloc_create(int num_blocks, int block_size, const int32_t* order,
                          pa_allocator** out) {
  if (!out) return pa::fail(PA_ERR_INVALID_ARG, "pa_alloc_create: out is NULL");
  *out = nullptr;
  if (num_blocks <= 0 || block_size <= 0)
    return pa::fail(PA_ERR_INVALID_ARG, "pa_alloc_create: num_blocks=%d block_size=%d",
                    num_blocks, block_size);
  if (static_cast<int64_t>(num_blocks) * block_size > INT32_MAX)
    return pa::fail(PA_ERR_INVALID_ARG, "pa_alloc_create: slots exceed int32");
  pa_allocator* a = new pa_allocator();
  a->num_blocks = num_blocks;
  a->block_size = block_size;
  a->ring.resize(num_blocks);
  a->ref.assign(num_blocks, 0);
  std::vector<char> seen(num_blocks, 0);
  for (int i = 0; i < num_blocks; ++i) {
    const int32_t b = order ? order[i] : i;
    if (b < 0 || b >= num_blocks || seen[b]) {
      delete a;
      return pa::fail(PA_ERR_INVALID_ARG,
                      "pa_alloc_create: initial order is not a permutation (entry %d = %d)", i, b);
    }
    seen[b] = 1;
    a->ring[i] = b;
  }
  a->count = num_blocks;
  *out = a;
  return pa::ok();
}

void pa_alloc_destroy(pa_allocator* a) { delete a; }

pa_status pa_alloc_add_seq(pa_allocator* a, int64_t seq_id, int64_t len) {
  if (pa_status s = check_handle(a)) return s;
  if (len < 0) return pa::fail(PA_ERR_INVALID_ARG, "add_seq: negative length");
  if (a->seqs.count(seq_id))
    return pa::fail(PA_ERR_INVALID_ARG, "add_seq: sequence %lld exists", (long long)seq_id);
  const int64_t n = a->blocks_for(len);
  if (n > a->count) {
    ++a->alloc_failures;
    return pa::fail(PA_ERR_OUT_OF_BLOCKS, "add_seq: need %lld blocks, %lld free",
                    (long long)n, (long long)a->count);
  }
  pa_allocator::Seq s;
  s.len = len;
  s.table.reserve(static_cast<size_t>(n));
  for (int64_t i = 0; i < n; ++i) s.table.push_back(a->take());
  a->seqs.emplace(seq_id, std::move(s));
  return pa::ok();
}

pa_status pa_alloc_fork(pa_allocator* a, int64_t parent, int64_t child) {
  if (pa_status s = check_handle(a)) return s;
  auto it = a->seqs.find(parent);
  if (it == a->seqs.end() || it->second.swapped || a->seqs.count(child))
    return pa::fail(PA_ERR_INVALID_ARG,
                    "fork: parent %lld missing or swapped out, or child %lld exists",
                    (long long)parent, (long long)child);
  pa_allocator::Seq s = it->second;
  for (int32_t b : s.table) a->inc(b);
  a->seqs.emplace(child, std::move(s));
  return pa::ok();
}

pa_status pa_alloc_append_slot(pa_allocator* a, int64_t seq_id, int32_t* slot,
                               int32_t* cow_src, int32_t* cow_dst) {
  if (pa_status s = check_handle(a)) return s;
  if (!slot || !cow_src || !cow_dst)
    return pa::fail(PA_ERR_INVALID_ARG, "append_slot: NULL output");
  pa_status s = append_one(a, seq_id, slot, cow_src, cow_dst);
  return s == PA_OK ? pa::ok() : s;
}

pa_status pa_alloc_append_slots(pa_allocator* a, const int64_t* seq_ids, int n,
                                int32_t* slots, int32_t* cow_pairs, int* num_cow,
                                int* num_done) {
  if (pa_status s = check_handle(a)) return s;
  if (n < 0 || (n > 0 && (!seq_ids || !slots || !cow_pairs)) || !num_cow || !num_done)
    return pa::fail(PA_ERR_INVALID_ARG, "append_slots: bad arguments");
  *num_cow = 0;
  *num_done = 0;
  for (int i = 0; i < n; ++i) {
    int32_t cs, cd;
    pa_status s = append_one(a, seq_ids[i], &slots[i], &cs, &cd);
    if (s != PA_OK) return s;
    if (cs >= 0) {
      cow_pairs[2 * *num_cow] = cs;
      cow_pairs[2 * *num_cow + 1] = cd;
      ++*num_cow;
    }
    *num_done = i + 1;
  }
  return pa::ok();
}

pa_status pa_alloc_plan_step(pa_allocator* a, const int64_t* seq_ids, int n, int max_blocks,
                             int32_t fill, int32_t* slots, int32_t* cow_pairs, int* num_cow,
                             int32_t* table, int32_t* seq_lens) {
  if (pa_status s = check_handle(a)) return s;
  if (n < 0 || max_blocks <= 0 || !num_cow ||
      (n > 0 && (!seq_ids || !slots || !cow_pairs || !table || !seq_lens)))
    return pa::fail(PA_ERR_INVALID_ARG, "plan_step: bad arguments");
  *num_cow = 0;
  const int BS = a->block_size;
  const uint64_t mark = ++a->plans;
  a->plan_seqs.resize(static_cast<size_t>(n));
  // 1. every sequence known, present once, tabled after its append within
  //    max_blocks; the blocks the appends will take: one per sequence that
  //    grows, plus the copies. A block with r holders written by k sequences
  //    of the batch is copied min(k, r - 1) times: each writer copies while
  //    another holder is left, and the last holder writes in place.
  int64_t need = 0;
  for (int i = 0; i < n; ++i) {
    auto it = a->seqs.find(seq_ids[i]);
    if (it == a->seqs.end() || it->second.swapped)
      return pa::fail(PA_ERR_INVALID_ARG, "plan_step: sequence %lld unknown or swapped out",
                      (long long)seq_ids[i]);
    pa_allocator::Seq& sq = it->second;
    if (sq.plan_mark == mark)
      return pa::fail(PA_ERR_INVALID_ARG, "plan_step: sequence %lld listed twice",
                      (long long)seq_ids[i]);
    sq.plan_mark = mark;
    const bool grows = sq.len % BS == 0;
    if (static_cast<int64_t>(sq.table.size()) + (grows ? 1 : 0) > max_blocks)
      return pa::fail(PA_ERR_INVALID_ARG, "plan_step: sequence %lld needs more than %d blocks",
                      (long long)seq_ids[i], max_blocks);
    if (sq.len + 1 > INT32_MAX)
      return pa::fail(PA_ERR_INVALID_ARG, "plan_step: length exceeds int32");
    a->plan_seqs[i] = &sq;
  }
  if (a->plan_writes.size() != static_cast<size_t>(a->num_blocks))
    a->plan_writes.assign(static_cast<size_t>(a->num_blocks), 0);
  a->plan_blocks.clear();
  for (int i = 0; i < n; ++i) {
    const pa_allocator::Seq& sq = *a->plan_seqs[i];
    if (sq.len % BS == 0) {
      ++need;
    } else {
      const int32_t b = sq.table[sq.len / BS];
      if (a->ref[b] > 1 && a->plan_writes[b]++ == 0) a->plan_blocks.push_back(b);
    }
  }
  for (int32_t b : a->plan_blocks) {
    need += std::min<int64_t>(a->plan_writes[b], a->ref[b] - 1);
    a->plan_writes[b] = 0;
  }
  if (need > a->count) {
    ++a->alloc_failures;
    return pa::fail(PA_ERR_OUT_OF_BLOCKS, "plan_step: %lld blocks needed, %lld free",
                    (long long)need, (long long)a->count);
  }
  // 2. the appends (none can fail now), then the batch's tables and lengths
  for (int i = 0; i < n; ++i) {
    int32_t cs, cd;
    append_to(a, *a->plan_seqs[i], seq_ids[i], &slots[i], &cs, &cd);
    if (cs >= 0) {
      cow_pairs[2 * *num_cow] = cs;
      cow_pairs[2 * *num_cow + 1] = cd;
      ++*num_cow;
    }
  }
  for (int i = 0; i < n; ++i) {
    const pa_allocator::Seq& sq = *a->plan_seqs[i];
    int32_t* row = table + static_cast<size_t>(i) * max_blocks;
    std::copy(sq.table.begin(), sq.table.end(), row);
    std::fill(row + sq.table.size(), row + max_blocks, fill);
    seq_lens[i] = static_cast<int32_t>(sq.len);
  }
  return pa::ok();
}

pa_status pa_alloc_free_seq(pa_allocator* a, int64_t seq_id) {
  if (pa_status s = check_handle(a)) return s;
  auto it = a->seqs.find(seq_id);
  if (it == a->seqs.end())
    return pa::fail(PA_ERR_INVALID_ARG, "free_seq: unknown sequence %lld", (long long)seq_id);
  if (it->second.swapped) {
    for (int32_t h : it->second.host) a->host_push(h);
    --a->swapped_seqs;
  }
  for (int32_t b : it->second.table) a->dec(b);
  a->seqs.erase(it);
  return pa::ok();
}

pa_status pa_alloc_add_host_pool(pa_allocator* a, int num_host_blocks, const int32_t* order) {
  if (pa_status s = check_handle(a)) return s;
  if (a->num_host > 0 || num_host_blocks <= 0)
    return pa::fail(PA_ERR_INVALID_ARG, "add_host_pool: pool exists or size %d", num_host_blocks);
  std::vector<int32_t> ring(num_host_blocks);
  std::vector<char> seen(num_host_blocks, 0);
  for (int i = 0; i < num_host_blocks; ++i) {
    const int32_t h = order ? order[i] : i;
    if (h < 0 || h >= num_host_blocks || seen[h])
      return pa::fail(PA_ERR_INVALID_ARG,
                      "add_host_pool: order is not a permutation (entry %d = %d)", i, h);
    seen[h] = 1;
    ring[i] = h;
  }
  a->num_host = num_host_blocks;
  a->hring = std::move(ring);
  a->hhead = 0;
  a->hcount = num_host_blocks;
  return pa::ok();
}

pa_status pa_alloc_swap_out(pa_allocator* a, int64_t seq_id, int32_t* pairs, int cap, int* n) {
  if (pa_status s = check_handle(a)) return s;
  if (!n) return pa::fail(PA_ERR_INVALID_ARG, "swap_out: n is NULL");
  *n = 0;
  auto it = a->seqs.find(seq_id);
  if (it == a->seqs.end() || it->second.swapped)
    return pa::fail(PA_ERR_INVALID_ARG, "swap_out: sequence %lld unknown or swapped out",
                    (long long)seq_id);
  auto& sq = it->second;
  const int nb = static_cast<int>(sq.table.size());
  if (cap < nb || (nb > 0 && !pairs))
    return pa::fail(PA_ERR_INVALID_ARG, "swap_out: capacity %d < %d pairs", cap, nb);
  if (nb > a->hcount) {
    ++a->alloc_failures;
    return pa::fail(PA_ERR_OUT_OF_BLOCKS, "swap_out: need %d host blocks, %lld free", nb,
                    (long long)a->hcount);
  }
  sq.host.clear();
  for (int j = 0; j < nb; ++j) {
    const int32_t h = a->host_take();
    sq.host.push_back(h);
    pairs[2 * j] = sq.table[j];
    pairs[2 * j + 1] = h;
  }
  for (int32_t b : sq.table) a->dec(b);
  sq.table.clear();
  sq.swapped = true;
  ++a->swapped_seqs;
  ++a->swap_outs;
  *n = nb;
  return pa::ok();
}

pa_status pa_alloc_swap_in(pa_allocator* a, int64_t seq_id, int32_t* pairs, int cap, int* n) {
  if (pa_status s = check_handle(a)) return s;
  if (!n) return pa::fail(PA_ERR_INVALID_ARG, "swap_in: n is NULL");
  *n = 0;
  auto it = a->seqs.find(seq_id);
  if (it == a->seqs.end() || !it->second.swapped)
    return pa::fail(PA_ERR_INVALID_ARG, "swap_in: sequence %lld is not swapped out",
                    (long long)seq_id);
  auto& sq = it->second;
  const int nb = static_cast<int>(sq.host.size());
  if (cap < nb || (nb > 0 && !pairs))
    return pa::fail(PA_ERR_INVALID_ARG, "swap_in: capacity %d < %d pairs", cap, nb);
  if (nb > a->count) {
    ++a->alloc_failures;
    return pa::fail(PA_ERR_OUT_OF_BLOCKS, "swap_in: need %d blocks, %lld free", nb,
                    (long long)a->count);
  }
  sq.table.clear();
  for (int j = 0; j < nb; ++j) {
    const int32_t b = a->take();
    sq.table.push_back(b);
    pairs[2 * j] = sq.host[j];
    pairs[2 * j + 1] = b;
  }
  for (int32_t h : sq.host) a->host_push(h);
  sq.host.clear();
  sq.swapped = false;
  --a->swapped_seqs;
  ++a->swap_ins;
  *n = nb;
  return pa::ok();
}

pa_status pa_alloc_export_host_state(const pa_allocator* a, int32_t* free_order, int* num_free,
                                     int64_t* counts) {
  if (pa_status s = check_handle(a)) return s;
  if (!num_free || !counts || (a->num_host > 0 && !free_order))
    return pa::fail(PA_ERR_INVALID_ARG, "export_host_state: NULL output");
  for (int64_t i = 0; i < a->num_host; ++i)
    free_order[i] = i < a->hcount ? a->hring[(a->hhead + i) % a->num_host] : -1;
  *num_free = static_cast<int>(a->hcount);
  counts[0] = a->num_host;
  counts[1] = a->swapped_seqs;
  counts[2] = a->swap_outs;
  counts[3] = a->swap_ins;
  return pa::ok();
}

pa_status pa_alloc_get_table(const pa_allocator* a, int64_t seq_id, int32_t* out, int cap,
                             int* n) {
  if (pa_status s = check_handle(a)) return s;
  if (!n) return pa::fail(PA_ERR_INVALID_ARG, "get_table: n is NULL");
  auto it = a->seqs.find(seq_id);
  if (it == a->seqs.end() || it->second.swapped)
    return pa::fail(PA_ERR_INVALID_ARG, "get_table: sequence %lld unknown or swapped out",
                    (long long)seq_id);
  const auto& t = it->second.table;
  *n = static_cast<int>(t.size());
  if (cap < *n || (*n > 0 && !out))
    return pa::fail(PA_ERR_INVALID_ARG, "get_table: capacity %d < %d", cap, *n);
  std::copy(t.begin(), t.end(), out);
  return pa::ok();
}

pa_status pa_alloc_seq_len(const pa_allocator* a, int64_t seq_id, int64_t* len) {
  if (pa_status s = check_handle(a)) return s;
  auto it = a->seqs.find(seq_id);
  if (it == a->seqs.end() || !len)
    return pa::fail(PA_ERR_INVALID_ARG, "seq_len: unknown sequence %lld", (long long)seq_id);
  *len = it->second.len;
  return pa::ok();
}

pa_status pa_alloc_build_tables(const pa_allocator* a, const int64_t* seq_ids, int n,
                                int max_blocks, int32_t fill, int32_t* table,
                                int32_t* seq_lens) {
  if (pa_status s = check_handle(a)) return s;
  if (n < 0 || max_blocks <= 0 || (n > 0 && (!seq_ids || !table || !seq_lens)))
    return pa::fail(PA_ERR_INVALID_ARG, "build_tables: bad arguments");
  for (int i = 0; i < n; ++i) {
    auto it = a->seqs.find(seq_ids[i]);
    if (it == a->seqs.end() || it->second.swapped)
      return pa::fail(PA_ERR_INVALID_ARG, "build_tables: sequence %lld unknown or swapped out",
                      (long long)seq_ids[i]);
    const auto& t = it->second.table;
    if (static_cast<int64_t>(t.size()) > max_blocks)
      return pa::fail(PA_ERR_INVALID_ARG, "build_tables: sequence %lld holds %zu > %d blocks",
                      (long long)seq_ids[i], t.size(), max_blocks);
    if (it->second.len > INT32_MAX)
      return pa::fail(PA_ERR_INVALID_ARG, "build_tables: length exceeds int32");
    int32_t* row = table + static_cast<size_t>(i) * max_blocks;
    std::copy(t.begin(), t.end(), row);
    std::fill(row + t.size(), row + max_blocks, fill);
    seq_lens[i] = static_cast<int32_t>(it->second.len);
  }
  return pa::ok();
}

pa_status pa_alloc_shared_prefix(const pa_allocator* a, const int64_t* seq_ids, int n,
                                 int32_t* blocks, int cap, int* num_blocks) {
  if (pa_status s = check_handle(a)) return s;
  if (n < 0 || cap < 0 || !num_blocks || (n > 0 && !seq_ids))
    return pa::fail(PA_ERR_INVALID_ARG, "shared_prefix: bad arguments");
  *num_blocks = 0;
  const std::vector<int32_t>* first = nullptr;
  int64_t k = 0;  // length of the run common to the sequences seen so far
  for (int i = 0; i < n; ++i) {
    auto it = a->seqs.find(seq_ids[i]);
    if (it == a->seqs.end() || it->second.swapped)
      return pa::fail(PA_ERR_INVALID_ARG, "shared_prefix: sequence %lld unknown or swapped out",
                      (long long)seq_ids[i]);
    const auto& t = it->second.table;
    // blocks this sequence attends in full
    const int64_t whole = std::min<int64_t>(static_cast<int64_t>(t.size()),
                                            it->second.len / a->block_size);
    if (!first) {
      first = &t;
      k = whole;
      continue;
    }
    int64_t j = 0;
    const int64_t lim = std::min(k, whole);
    while (j < lim && t[j] == (*first)[j]) ++j;
    k = j;
  }
  *num_blocks = static_cast<int>(k);
  if (cap < k || (k > 0 && !blocks))
    return pa::fail(PA_ERR_INVALID_ARG, "shared_prefix: capacity %d < %lld", cap, (long long)k);
  if (k > 0) std::copy(first->begin(), first->begin() + k, blocks);
  return pa::ok();
}

pa_status pa_alloc_stats(const pa_allocator* a, pa_alloc_stats_t* out) {
  if (pa_status s = check_handle(a)) return s;
  if (!out) return pa::fail(PA_ERR_INVALID_ARG, "stats: out is NULL");
  out->num_blocks = a->num_blocks;
  out->free_blocks = a->count;
  out->used_blocks = a->used;
  out->shared_blocks = a->shared;
  out->cow_copies = a->cow_copies;
  out->alloc_failures = a->alloc_failures;
  out->total_refs = a->total_refs;
  out->num_seqs = static_cast<int64_t>(a->seqs.size());
  return pa::ok();
}

pa_status pa_alloc_export_state(const pa_allocator* a, int32_t* free_order, int* num_free,
                                int32_t* refcounts) {
  if (pa_status s = check_handle(a)) return s;
  if (!free_order || !num_free || !refcounts)
    return pa::fail(PA_ERR_INVALID_ARG, "export_state: NULL output");
  for (int64_t i = 0; i < a->num_blocks; ++i)
    free_order[i] = i < a->count ? a->ring[(a->head + i) % a->num_blocks] : -1;
  *num_free = static_cast<int>(a->count);
  std::copy(a->ref.begin(), a->ref.end(), refcounts);
  return pa::ok();
}

}  // extern "C"
