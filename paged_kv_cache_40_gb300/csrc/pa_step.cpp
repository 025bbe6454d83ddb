// One decode step in one call: the block manager plans it, then its kernels
// are enqueued ("Phase 7 · Document 04 — PagedAttention", §2: on-demand
// allocation and copy-on-write decide where each new token goes, and the
// attention kernel follows the tables the manager keeps; lux-666 notes
// "PagedAttention", 最小模型). A serving loop calls this once per step instead
// of planning, copying, appending and attending through separate calls.
#include "pa_internal.h"

extern "C" {

pa_status pa_decode_step(pa_allocator* a, const int64_t* seq_ids, int num_seqs, int max_blocks,
                         int32_t* slot_mapping, int32_t* cow_pairs, int32_t* block_table,
                         int32_t* seq_lens, int* num_cow, const pa_half* q, const pa_half* k_new,
                         const pa_half* v_new, pa_half* k_pool, pa_half* v_pool,
                         int num_q_heads, int num_kv_heads, int head_dim, int num_blocks,
                         int64_t pool_block_stride, float scale, pa_half* out, void* workspace,
                         size_t workspace_bytes, int partition_tokens, pa_stream_t stream) {
  if (!a || !num_cow) return pa::fail(PA_ERR_INVALID_ARG, "pa_decode_step: NULL handle or num_cow");
  *num_cow = 0;
  const int BS = pa::alloc_block_size(a);
  if (num_blocks != pa::alloc_num_blocks(a))
    return pa::fail(PA_ERR_INVALID_ARG,
                    "pa_decode_step: the pool has %d blocks, the block manager %d", num_blocks,
                    pa::alloc_num_blocks(a));
  // the whole plan is checked before anything changes (all or nothing)
  if (pa_status s = pa_alloc_plan_step(a, seq_ids, num_seqs, max_blocks, -1, slot_mapping,
                                       cow_pairs, num_cow, block_table, seq_lens))
    return s;
  if (num_seqs == 0) return pa::ok();
  if (*num_cow > 0) {
    if (pa_status s = pa_copy_blocks(k_pool, v_pool, cow_pairs, *num_cow, num_kv_heads, head_dim,
                                     BS, num_blocks, pool_block_stride, stream))
      return s;
  }
  return pa_decode_append_attention(q, k_new, v_new, slot_mapping, k_pool, v_pool, block_table,
                                    seq_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, BS,
                                    max_blocks, num_blocks, pool_block_stride, scale, out,
                                    workspace, workspace_bytes, partition_tokens, stream);
}

pa_status pa_decode_step_fp8(pa_allocator* a, const int64_t* seq_ids, int num_seqs,
                             int max_blocks, int32_t* slot_mapping, int32_t* cow_pairs,
                             int32_t* block_table, int32_t* seq_lens, int* num_cow,
                             const pa_half* q, const pa_half* k_new, const pa_half* v_new,
                             uint8_t* k_pool, uint8_t* v_pool, const float* k_scale,
                             const float* v_scale, int num_q_heads, int num_kv_heads,
                             int head_dim, int num_blocks, int64_t pool_block_stride, float scale,
                             pa_half* out, void* workspace, size_t workspace_bytes,
                             int partition_tokens, pa_stream_t stream) {
  if (!a || !num_cow)
    return pa::fail(PA_ERR_INVALID_ARG, "pa_decode_step_fp8: NULL handle or num_cow");
  *num_cow = 0;
  const int BS = pa::alloc_block_size(a);
  if (num_blocks != pa::alloc_num_blocks(a))
    return pa::fail(PA_ERR_INVALID_ARG,
                    "pa_decode_step_fp8: the pool has %d blocks, the block manager %d",
                    num_blocks, pa::alloc_num_blocks(a));
  if (pa_status s = pa_alloc_plan_step(a, seq_ids, num_seqs, max_blocks, -1, slot_mapping,
                                       cow_pairs, num_cow, block_table, seq_lens))
    return s;
  if (num_seqs == 0) return pa::ok();
  if (*num_cow > 0) {
    if (pa_status s = pa_copy_blocks_fp8(k_pool, v_pool, cow_pairs, *num_cow, num_kv_heads,
                                         head_dim, BS, num_blocks, pool_block_stride, stream))
      return s;
  }
  if (pa_status s = pa_append_kv_fp8(k_new, v_new, k_pool, v_pool, slot_mapping, k_scale,
                                     v_scale, num_seqs, num_kv_heads, head_dim, BS, num_blocks,
                                     pool_block_stride, stream))
    return s;
  return pa_decode_attention_fp8(q, k_pool, v_pool, k_scale, v_scale, block_table, seq_lens,
                                 num_seqs, num_q_heads, num_kv_heads, head_dim, BS, max_blocks,
                                 num_blocks, pool_block_stride, scale, out, workspace,
                                 workspace_bytes, partition_tokens, stream);
}

}  // extern "C"
