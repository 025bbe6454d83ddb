// Host-side pieces the kernels' launchers share: the cached TMA descriptors
// of the pools and the shared-prefix launch that the shared-prefix entry
// point calls before (when needed) the attention kernel's prefix mode.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "pa_internal.h"

namespace pa {

// A 4-D tensor map over a pool seen as (dim, token, KV head, block) with box
// {128-byte line, ts tokens, hg heads, 1} and the 128-byte swizzle.
struct MapKey {
  int device;
  const void* ptr;
  int D, BS, Hkv, NB, hg, ts;
  int esz;             // bytes per value: 2 (fp16) or 1 (E4M3)
  long long stride;    // bytes from one block to the next
  bool operator==(const MapKey& o) const {
    return device == o.device && ptr == o.ptr && D == o.D && BS == o.BS && Hkv == o.Hkv &&
           NB == o.NB && hg == o.hg && ts == o.ts && esz == o.esz && stride == o.stride;
  }
};
// The map of `key` (the last few are cached); PA_ERR_CUDA with a message if
// the driver refuses it.
pa_status pool_tensor_map(const MapKey& key, CUtensorMap* out);

// The prefix part of pa_decode_attention_shared_prefix (device pointers,
// already checked and mapped).
struct SharedPrefixCall {
  const void* q;                 // [S][Hq][D] fp16
  const int32_t* prefix_blocks;  // [P]
  float* records;                // the prefix chunks' partial records (unfused mode)
  int32_t* err;
  int num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks, num_blocks;
  int prefix_blocks_n;           // P
  float qscale;                  // scale * log2(e)
  const int32_t* block_table;    // [S][max_blocks], the whole table
  const int32_t* seq_lens;
  const void* k_pool;
  const void* v_pool;
  long long block_stride_bytes;
  void* out;                     // [S][Hq][D] fp16
};
// Launches the shared prefix's kernel on `stream`: the single launch that
// also attends each sequence's short suffix and writes the output
// (*suffix_pass = false), or the prefix kernel writing *chunks partial
// records per (sequence, KV head) for the attention kernel's prefix mode to
// fold in (*suffix_pass = true).
pa_status launch_shared_prefix(const SharedPrefixCall& call, const DeviceInfo& dev,
                               cudaStream_t stream, bool* suffix_pass, int* chunks);
// The most prefix chunks (records per (sequence, KV head)) it ever writes.
int max_prefix_chunks();

}  // namespace pa
