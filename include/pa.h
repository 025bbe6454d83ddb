/*
 * pa.h — C ABI of libpa: paged decode attention and its KV-cache bookkeeping,
 * hand-written CUDA for GB300 (sm_103a).
 *
 * The operations follow the PagedAttention pages:
 *   - "Phase 7 · Document 04 — PagedAttention" (ai-engineer-zt0), §2 Core
 *     Concept: the KV cache is cut into fixed-size blocks held in a shared pool
 *     of physical blocks; each sequence's block table maps logical token
 *     positions to scattered physical blocks; the attention kernel follows that
 *     indirection to gather K/V during the dot product; blocks are allocated on
 *     demand and freed at once; shared prefixes are copy-on-write (§2 "block
 *     sharing", §3 Mental Model).
 *   - lux-666 notes "PagedAttention", 最小模型 (minimal model): logical blocks
 *     -> block table -> physical blocks; the kernel reads the table and visits
 *     the physical blocks in logical token order; a growing request needs one
 *     more block, a finished one frees its own blocks.
 *
 * Conventions shared by every call
 *   - fp16 tensors are IEEE-754 binary16, passed as `pa_half*` (the raw 16-bit
 *     patterns). Index tensors are int32.
 *   - Pools: k_pool and v_pool each hold num_blocks physical blocks of
 *     [block_size][num_kv_heads][head_dim] values, row-major and contiguous
 *     within a block. Block b of a pool starts pool_block_stride values after
 *     block b-1 (0 = block_size*num_kv_heads*head_dim: a dense
 *     [num_blocks][block_size][num_kv_heads][head_dim] array). Pool "slot" s
 *     (0 <= s < num_blocks*block_size) is row s % block_size of block
 *     s / block_size.
 *   - The one-pool layout of the layout sketch ("Phase 7 · Document 04 —
 *     PagedAttention", §2 Core Concept: an array of per-block records, each a
 *     K array followed by a V array) is served by the same calls: with E =
 *     block_size*num_kv_heads*head_dim and kv the record array, pass
 *     k_pool = kv, v_pool = kv + E and pool_block_stride = 2*E. A stride must
 *     be at least E values and a multiple of 16 bytes. Calls that write the
 *     pools refuse a K and a V pool whose blocks overlap.
 *   - Memory is owned by the caller (the library never allocates or frees
 *     device memory); array pointers must be 16-byte aligned (index arrays
 *     4-byte). Pools and workspaces must be device memory. The arrays a call
 *     reads or writes in place (q, new K/V rows, slot mappings, copy pairs,
 *     block tables, lengths, scales, prefix block lists, outputs) may instead
 *     be pinned (page-locked) host memory, which the kernels then access
 *     through its device mapping over the CPU-GPU link, with no copy call;
 *     pageable host memory is refused with PA_ERR_INVALID_ARG before any
 *     launch. Device calls are
 *     asynchronous on `stream` (a cudaStream_t; NULL = the legacy default
 *     stream): arguments are checked on the host before any launch, and a
 *     PA_OK return means "launched", not "finished".
 *   - Data-dependent checks (a block id or slot outside the pool, a length
 *     longer than the table) happen on the device: the offending access is
 *     skipped and a device error word is set. pa_device_error() reads and
 *     clears it (it synchronises the stream).
 *   - Every call returns a pa_status. On failure, pa_last_error() gives a
 *     message for the calling thread. There is no fallback path: an unsupported
 *     shape or device is an error, never a silent change of method.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t pa_half;   /* IEEE-754 binary16 bit pattern */
typedef void* pa_stream_t;  /* cudaStream_t */

typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,    /* a host-checked argument is out of range */
  PA_ERR_OUT_OF_BLOCKS = 2,  /* the allocator's free list is too short */
  PA_ERR_BAD_BLOCK_ID = 3,   /* device: a block id / slot / length out of range */
  PA_ERR_UNSUPPORTED = 4,    /* shape or device this build does not serve */
  PA_ERR_CUDA = 5,           /* a CUDA runtime call failed */
  PA_ERR_TIMEOUT = 6         /* device: a bounded wait gave up */
} pa_status;

/* Message of the calling thread's last failed call ("" if none). */
PA_API const char* pa_last_error(void);
/* Static name of a status code. */
PA_API const char* pa_status_string(pa_status s);
/* Library version, major*10000 + minor*100 + patch. */
PA_API int pa_version(void);

/* ------------------------------------------------------------------------
 * Device error word.
 * Reads and clears the word the kernels set on data-dependent faults they
 * skipped (bad block id, bad slot, length beyond the table, bounded wait that
 * gave up). Synchronises `stream` first. *flags receives the raw bit set
 * (PA_DEVERR_*), and the return value is PA_ERR_BAD_BLOCK_ID or
 * PA_ERR_TIMEOUT when a bit was set, else PA_OK.
 * ---------------------------------------------------------------------- */
#define PA_DEVERR_BAD_BLOCK 1   /* block-table entry outside [0, num_blocks) */
#define PA_DEVERR_BAD_SLOT 2    /* slot outside [0, num_blocks*block_size) */
#define PA_DEVERR_BAD_LEN 4     /* seq_len < 0 or > max_blocks*block_size */
#define PA_DEVERR_TIMEOUT 8     /* a pipeline wait hit its time limit */
PA_API pa_status pa_device_error(pa_stream_t stream, int32_t* flags);

/* Time limit of the attention kernels' pipeline waits (the stage, q-slot and
 * merge handoffs inside pa_decode_attention, pa_decode_attention_fp8,
 * pa_decode_attention_fixed_scratch and the streaming pass of
 * pa_decode_attention_shared_prefix), taken by every later call of those
 * entry points from this process. The default, about one second, is far
 * above any wait of a healthy launch. A wait that runs out records
 * PA_DEVERR_TIMEOUT and the kernel stops streaming, lets the copies it
 * already issued land (always on the one-second limit) and exits; its
 * outputs are then undefined. A short limit makes that path run on demand,
 * so that a test can check it without a fault or a hang; 0 restores the
 * default. The pages have no counterpart: it belongs to the failure
 * handling of the pages' explicit-failure rule ("Phase 7 · Document 04 —
 * PagedAttention", §11: reject rather than thrash at the limit).
 * Errors: none (PA_OK). */
PA_API pa_status pa_set_wait_limit_ns(uint64_t limit_ns);

/* Number of kernels this library has enqueued in this process, on any
 * device or stream (every call counts the launches it made; a call that
 * launches nothing, such as pa_copy_blocks with no pairs, counts none).
 * Read it before and after a region of calls to know how many of the
 * library's kernels that region ran: pa_decode_attention_shared_prefix, for
 * one, launches one kernel or two depending on the suffix lengths. A
 * monotonic counter: no reset, no error. */
PA_API uint64_t pa_kernel_launches(void);

/* ------------------------------------------------------------------------
 * pa_append_kv — write each sequence's new K/V token into its cache slot.
 *
 * Source: the KV cache grows one token per decode step ("Phase 7 · Document
 * 04 — PagedAttention", §2 primer; lux-666 notes, 问题从哪里来); the block
 * manager decides where the token goes (same pages, on-demand allocation).
 *
 * k_new, v_new   device [num_tokens][num_kv_heads][head_dim] fp16 (read)
 * k_pool, v_pool device pools (written at the mapped rows only)
 * slot_mapping   device int32 [num_tokens]; token i goes to slot
 *                slot_mapping[i]; a negative slot skips the token; a slot
 *                >= num_blocks*block_size is skipped and sets
 *                PA_DEVERR_BAD_SLOT.
 * The copy is bit-exact. Two tokens mapped to the same slot race (one wins).
 * Errors: PA_ERR_INVALID_ARG (bad sizes or stride, NULL or misaligned
 *         pointers, overlapping K and V blocks), PA_ERR_UNSUPPORTED (head_dim
 *         not a multiple of 8), PA_ERR_CUDA.
 * ---------------------------------------------------------------------- */
PA_API pa_status pa_append_kv(const pa_half* k_new, const pa_half* v_new,
                       pa_half* k_pool, pa_half* v_pool,
                       const int32_t* slot_mapping, int num_tokens,
                       int num_kv_heads, int head_dim, int block_size,
                       int num_blocks, int64_t pool_block_stride,
                       pa_stream_t stream);

/* ------------------------------------------------------------------------
 * pa_copy_blocks — copy-on-write duplication of whole blocks.
 *
 * Source: "Phase 7 · Document 04 — PagedAttention", §2 "block sharing
 * (copy-on-write)": sequences that share a prefix point at the same physical
 * blocks and only the block that diverges is copied; §3 Mental Model; lux-666
 * notes, prefix sharing splits at the copy-on-write boundary.
 *
 * pairs      device int32 [num_pairs][2] = (src, dst) physical block ids.
 *            Block dst of both pools becomes a bit-exact copy of block src
 *            (all block_size rows, every KV head). Destinations must be
 *            distinct and must not appear as sources (the allocator's pairs
 *            satisfy this); otherwise the result is unspecified (no fault).
 *            An id outside [0, num_blocks) skips that pair and sets
 *            PA_DEVERR_BAD_BLOCK.
 * Errors: as pa_append_kv.
 * ---------------------------------------------------------------------- */
PA_API pa_status pa_copy_blocks(pa_half* k_pool, pa_half* v_pool,
                         const int32_t* pairs, int num_pairs,
                         int num_kv_heads, int head_dim, int block_size,
                         int num_blocks, int64_t pool_block_stride,
                         pa_stream_t stream);

/* ------------------------------------------------------------------------
 * pa_decode_attention — single-query attention over the paged cache.
 *
 * Source: "Phase 7 · Document 04 — PagedAttention", §2 Core Concept (the
 * layout sketch: per block K[BLOCK][HEADS][HEAD_DIM] and V likewise, one int32
 * table row per sequence, and attention reading K/V one block at a time
 * through that table); lux-666 notes, 最小模型 (the kernel reads the block
 * table and visits physical blocks in logical token order).
 *
 * For each sequence i and query head h (KV head kv = h / (num_q_heads /
 * num_kv_heads), consecutive groups):
 *   K[t], V[t] = pool[block_table[i][t / block_size]][t % block_size][kv]
 *   out[i][h] = sum_t softmax_t(scale * q[i][h] . K[t]) V[t],  t < seq_lens[i]
 * computed in fp32 (max-subtracted online softmax), rounded once to fp16.
 * A sequence of length 0 gets an all-zero output. The block stream of the
 * batch is cut into equal chunks, one per CTA, so a sequence may be split
 * across CTAs; the partial results of a split sequence are merged on the
 * device (log-sum-exp) by the last CTA to finish one of its chunks; the
 * caller sees one result.
 *
 * q            device [num_seqs][num_q_heads][head_dim] fp16
 * k_pool, v_pool  device pools (read only), pool_block_stride as above
 * block_table  device int32 [num_seqs][max_blocks_per_seq]; only the first
 *              ceil(seq_lens[i]/block_size) entries of row i are read.
 * seq_lens     device int32 [num_seqs], tokens attended (the appended one
 *              included); a value < 0 or > max_blocks_per_seq*block_size sets
 *              PA_DEVERR_BAD_LEN and is clamped into range.
 * scale        softmax scale (typically 1/sqrt(head_dim))
 * out          [num_seqs][num_q_heads][head_dim] fp16 (written): device
 *              memory, or pinned (page-locked) host memory, which the kernel
 *              writes through its device mapping (no separate copy back;
 *              visible to the host once the stream has been synchronised).
 *              Pageable host memory is refused (PA_ERR_INVALID_ARG). The
 *              same holds for `out` of every attention call below.
 * workspace    device scratch of >= pa_decode_workspace_bytes(...) bytes,
 *              16-byte aligned, owned by the caller. It holds an arrival
 *              counter per (sequence, KV head) and the fp32 partial results
 *              of split sequences. It needs no initialisation: each counter
 *              word carries a tag unique to the call that wrote it, and words
 *              with another tag count as empty. Calls sharing one workspace
 *              must not overlap on the device.
 * partition_tokens  0 = chunks as equal as the grid allows (the default);
 *              otherwise a positive multiple of block_size capping the
 *              tokens of one chunk (more, shorter chunks: a CTA then streams
 *              several).
 * The call enqueues one kernel on `stream`, launched as a programmatic
 * dependent: its CTAs may start while the previous kernel on the stream is
 * finishing, but they read no input (not even seq_lens) before that kernel
 * has completed, so any input may be written by the kernel just before.
 * After a PA_DEVERR_TIMEOUT report (pa_device_error), the counters of the
 * workspace that call used may hold arrivals under its tag: clear them with
 * pa_decode_workspace_init before a captured graph that uses the workspace
 * is replayed (eager calls take a new tag and need nothing).
 * Supported shapes: head_dim in {64, 128}; block_size in {8, 16, 32};
 * num_q_heads / num_kv_heads in {1, 2, 4, 8}; num_seqs <= 16384.
 * Errors: PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED (shape outside the list, or
 *         a device other than sm_103), PA_ERR_CUDA.
 * ---------------------------------------------------------------------- */
/* Bytes of workspace pa_decode_attention needs for this shape (0 if the
 * shape is invalid or unsupported). pa_decode_workspace_init zero-fills the
 * counters at the start of a workspace (num_seqs*num_kv_heads*8 bytes); the
 * attention call does not require it and it is kept for callers that clear
 * workspaces explicitly. */
PA_API size_t pa_decode_workspace_bytes(int num_seqs, int num_q_heads,
                                 int num_kv_heads, int head_dim,
                                 int block_size, int max_blocks_per_seq,
                                 int partition_tokens);

PA_API pa_status pa_decode_workspace_init(void* workspace, size_t workspace_bytes,
                                   int num_seqs, int num_kv_heads,
                                   pa_stream_t stream);

PA_API pa_status pa_decode_attention(const pa_half* q, const pa_half* k_pool,
                              const pa_half* v_pool,
                              const int32_t* block_table,
                              const int32_t* seq_lens, int num_seqs,
                              int num_q_heads, int num_kv_heads, int head_dim,
                              int block_size, int max_blocks_per_seq,
                              int num_blocks, int64_t pool_block_stride,
                              float scale, pa_half* out,
                              void* workspace, size_t workspace_bytes,
                              int partition_tokens, pa_stream_t stream);

/* ------------------------------------------------------------------------
 * pa_decode_attention_fixed_scratch — pa_decode_attention without a
 * caller-provided workspace; it allocates nothing.
 *
 * The pages have no counterpart for this call: it exists for callers that
 * cannot give the library scratch memory, for instance a serving process that
 * hands all of its device memory to its own KV pool and allocator up front,
 * or one that must not call cudaMalloc on the decode path because that call
 * synchronises the device. The scratch it needs (arrival counters and the
 * partial results of split sequences) lives in a fixed 16 MiB device array
 * inside libpa, which every GPU that loads the library keeps until the
 * process exits.
 *
 * Arguments, layouts and results are those of pa_decode_attention (same
 * kernel); only workspace and workspace_bytes are gone.
 * - The first call on a device resolves the array's device address (once per
 *   device, with that device current); make that first call before any stream
 *   capture.
 * - Every call uses the same array, which keeps what the last call left;
 *   the call clears the array's arrival counters on `stream` before its
 *   kernel (a memset, not an allocation), so a call cut short by a timeout
 *   leaves nothing behind for the next. Calls that overlap on the GPU (other
 *   streams, other host threads) race on the array and must not be issued.
 * - Shapes whose scratch would exceed 16 MiB (8 bytes per (sequence, KV
 *   head), plus two partial results of G x (head_dim + 2) floats per CTA of
 *   the grid and per KV head a CTA streams, up to 8) are refused with
 *   PA_ERR_UNSUPPORTED; use pa_decode_attention for them.
 * - No cudaMalloc, cudaFree or allocating library routine is called.
 * Errors: as pa_decode_attention, plus PA_ERR_UNSUPPORTED for the size limit.
 * ---------------------------------------------------------------------- */
PA_API pa_status pa_decode_attention_fixed_scratch(
    const pa_half* q, const pa_half* k_pool, const pa_half* v_pool,
    const int32_t* block_table, const int32_t* seq_lens, int num_seqs,
    int num_q_heads, int num_kv_heads, int head_dim, int block_size,
    int max_blocks_per_seq, int num_blocks, int64_t pool_block_stride,
    float scale, pa_half* out, int partition_tokens, pa_stream_t stream);

/* ------------------------------------------------------------------------
 * pa_decode_attention_shared_prefix — pa_decode_attention for a batch whose
 * sequences all begin with the same physical blocks (a shared prompt).
 *
 * Source: "Phase 7 · Document 04 — PagedAttention", §2 Core Concept (block
 * sharing: sequences reference the same physical blocks, copy-on-write on
 * divergence) and §3 Mental Model (A->[b3,b7,b1], B->[b3,b9]); lux-666 notes
 * "PagedAttention", prefix sharing. The pages share the blocks' memory; this
 * call also shares their reading: each prefix block of a KV head is streamed
 * once and contracted on tensor cores against the query rows of every
 * sequence, and each sequence's remaining blocks are streamed as in
 * pa_decode_attention, the two parts merged per (sequence, head).
 *
 * The result is that of pa_decode_attention with the same arguments
 * (prefix_blocks is a statement about block_table, not extra input):
 * precondition: block_table[i][j] == prefix_blocks[j] for j <
 * num_prefix_blocks and seq_lens[i] >= num_prefix_blocks * block_size for
 * every sequence i. A sequence shorter than the prefix sets
 * PA_DEVERR_BAD_LEN; a table that disagrees with prefix_blocks gives the
 * attention over prefix_blocks instead.
 *
 * prefix_blocks   device int32 [num_prefix_blocks], full blocks shared by
 *                 every sequence (num_prefix_blocks = 0 is plain
 *                 pa_decode_attention).
 * workspace       >= pa_decode_shared_prefix_workspace_bytes(...) bytes,
 *                 16-byte aligned, no initialisation needed.
 * Enqueues two kernels on `stream` (the second launched as a programmatic
 * dependent of the first). Supported: head_dim 128, block_size 16 or 32,
 * num_q_heads / num_kv_heads in {1, 2, 4, 8}.
 * Errors: as pa_decode_attention.
 * ---------------------------------------------------------------------- */
PA_API size_t pa_decode_shared_prefix_workspace_bytes(int num_seqs, int num_q_heads,
                                                      int num_kv_heads, int head_dim,
                                                      int block_size, int max_blocks_per_seq,
                                                      int num_prefix_blocks);

PA_API pa_status pa_decode_attention_shared_prefix(
    const pa_half* q, const pa_half* k_pool, const pa_half* v_pool,
    const int32_t* prefix_blocks, int num_prefix_blocks,
    const int32_t* block_table, const int32_t* seq_lens, int num_seqs,
    int num_q_heads, int num_kv_heads, int head_dim, int block_size,
    int max_blocks_per_seq, int num_blocks, int64_t pool_block_stride,
    float scale, pa_half* out, void* workspace, size_t workspace_bytes,
    pa_stream_t stream);

/* ------------------------------------------------------------------------
 * fp8 KV cache — the append, the block copy and decode attention over pools
 * of OCP E4M3 bytes with one fp32 scale per KV head for K and for V.
 *
 * Source: "Phase 7 · Document 04 — PagedAttention", §11 Engineering Decision
 * Framework (shrink per-sequence KV with `--kv-cache-dtype fp8`, KV
 * quantization) and §12 Hands-On Lab, step 3 (more sequences fit). The pages
 * fix no format; this library reads it as: a cached value is
 * e4m3(code) * scale[kv_head]; quantization is code = e4m3(fp32(x) /
 * scale[kv_head]) with the division in IEEE fp32 and round-to-nearest-even,
 * magnitudes above 448 saturating to 448.
 *
 * Pools: blocks of uint8 [block_size][num_kv_heads][head_dim], the same
 * order as the fp16 pools, one byte per value, pool_block_stride values
 * (bytes) apart (0 = dense). k_scale, v_scale: device fp32
 * [num_kv_heads], 4-byte aligned, read only. Ownership, streams, device error
 * word and status codes as for the fp16 calls.
 * ---------------------------------------------------------------------- */

/* pa_append_kv with quantization: row i of k_new/v_new (fp16, as in
 * pa_append_kv) is quantized per KV head and written at slot_mapping[i]. */
PA_API pa_status pa_append_kv_fp8(const pa_half* k_new, const pa_half* v_new,
                                  uint8_t* k_pool, uint8_t* v_pool,
                                  const int32_t* slot_mapping,
                                  const float* k_scale, const float* v_scale,
                                  int num_tokens, int num_kv_heads, int head_dim,
                                  int block_size, int num_blocks,
                                  int64_t pool_block_stride, pa_stream_t stream);

/* pa_copy_blocks over one-byte elements (head_dim a multiple of 16). */
PA_API pa_status pa_copy_blocks_fp8(uint8_t* k_pool, uint8_t* v_pool,
                                    const int32_t* pairs, int num_pairs,
                                    int num_kv_heads, int head_dim, int block_size,
                                    int num_blocks, int64_t pool_block_stride,
                                    pa_stream_t stream);

/* pa_append_kv then pa_decode_attention in one kernel, for one new token per
 * sequence (k_new/v_new row i belongs to sequence i): the step the pages'
 * decode loop takes ("Phase 7 · Document 04 — PagedAttention", §2: the
 * cache grows one token per step, then attention reads it through the
 * table). slot_mapping[i] must be the row of sequence i's last token
 * (position seq_lens[i] - 1 of its table), as the block manager assigns it;
 * the kernel writes the new K/V row there just before it copies that block,
 * so the attention includes it. A negative slot writes nothing (the row
 * already in the pool is attended); any other slot that is not that row is
 * not written and sets PA_DEVERR_BAD_SLOT. seq_lens count the new token.
 * Other arguments, layouts, the workspace and the errors are those of
 * pa_append_kv and pa_decode_attention (fp16 pools, K and V pools
 * disjoint). */
PA_API pa_status pa_decode_append_attention(const pa_half* q, const pa_half* k_new,
                                     const pa_half* v_new, const int32_t* slot_mapping,
                                     pa_half* k_pool, pa_half* v_pool,
                                     const int32_t* block_table, const int32_t* seq_lens,
                                     int num_seqs, int num_q_heads, int num_kv_heads,
                                     int head_dim, int block_size, int max_blocks_per_seq,
                                     int num_blocks, int64_t pool_block_stride, float scale,
                                     pa_half* out, void* workspace, size_t workspace_bytes,
                                     int partition_tokens, pa_stream_t stream);

/* pa_decode_attention over E4M3 pools: out[i][h] = sum_t softmax_t(scale *
 * q[i][h] . Kd[t]) Vd[t] with Kd, Vd the dequantized rows (code value times
 * the KV head's scale), computed in fp32 and rounded once to fp16. q, out,
 * block_table, seq_lens, workspace (sized by pa_decode_workspace_bytes with
 * the same shape) and partition_tokens as for pa_decode_attention.
 * Supported shapes: head_dim 128; block_size 16 or 32; num_q_heads /
 * num_kv_heads in {1, 2, 4, 8}; num_seqs <= 16384.
 * Errors: as pa_decode_attention. */
PA_API pa_status pa_decode_attention_fp8(const pa_half* q, const uint8_t* k_pool,
                                         const uint8_t* v_pool,
                                         const float* k_scale, const float* v_scale,
                                         const int32_t* block_table,
                                         const int32_t* seq_lens, int num_seqs,
                                         int num_q_heads, int num_kv_heads, int head_dim,
                                         int block_size, int max_blocks_per_seq,
                                         int num_blocks, int64_t pool_block_stride,
                                         float scale, pa_half* out,
                                         void* workspace, size_t workspace_bytes,
                                         int partition_tokens, pa_stream_t stream);

/* ------------------------------------------------------------------------
 * Host block allocator (block manager). Host memory only; no CUDA calls.
 *
 * Source: "Phase 7 · Document 04 — PagedAttention", §2 (a pool of physical
 * blocks allocated on demand and freed instantly; per-sequence block table;
 * copy-on-write sharing) and §3; lux-666 notes, 最小模型 (any free physical
 * block may back a logical block), the block-size section (a request of L
 * tokens holds ceil(L / block_size) blocks) and the prefix-sharing section
 * (reference counts, copy-on-write at the fork boundary).
 *
 * Rules fixed here where the pages leave them open:
 *   - the free list is FIFO: allocation takes the front; a block whose
 *     reference count drops to zero goes to the back; a sequence's blocks are
 *     released in logical order; the initial order is given or ascending;
 *   - a token appended at length L opens a new block iff L % block_size == 0;
 *   - writing into a block with reference count > 1 first moves the writer to
 *     a fresh block (copy-on-write pair (old, new) returned, old count - 1);
 *   - every call is all-or-nothing: on PA_ERR_OUT_OF_BLOCKS the state is
 *     unchanged (the batched append stops at the failing sequence).
 * Sequence ids are arbitrary int64 values. The handle is owned by the
 * library; it is not thread-safe (one thread at a time per handle).
 * ---------------------------------------------------------------------- */
typedef struct pa_allocator pa_allocator;

typedef struct pa_alloc_stats_t {
  int64_t num_blocks;
  int64_t free_blocks;
  int64_t used_blocks;    /* reference count > 0 */
  int64_t shared_blocks;  /* reference count > 1 */
  int64_t cow_copies;     /* copy-on-write pairs issued so far */
  int64_t alloc_failures; /* calls refused with PA_ERR_OUT_OF_BLOCKS */
  int64_t total_refs;     /* sum of reference counts = table entries */
  int64_t num_seqs;
} pa_alloc_stats_t;

/* initial_free_order: host int32 [num_blocks], a permutation of
 * 0..num_blocks-1, or NULL for ascending. */
PA_API pa_status pa_alloc_create(int num_blocks, int block_size,
                          const int32_t* initial_free_order,
                          pa_allocator** out);
PA_API void pa_alloc_destroy(pa_allocator* a);

/* Register sequence seq_id already holding `len` tokens: takes
 * ceil(len / block_size) blocks from the front of the free list. */
PA_API pa_status pa_alloc_add_seq(pa_allocator* a, int64_t seq_id, int64_t len);

/* child shares every block of parent (each reference count + 1). */
PA_API pa_status pa_alloc_fork(pa_allocator* a, int64_t parent, int64_t child);

/* Reserve the slot of the next token of seq_id (length grows by one).
 * *slot = physical_block * block_size + offset; *cow_src / *cow_dst = the
 * copy-on-write pair, or -1 / -1 when no copy is needed. */
PA_API pa_status pa_alloc_append_slot(pa_allocator* a, int64_t seq_id,
                               int32_t* slot, int32_t* cow_src,
                               int32_t* cow_dst);

/* Batched form for one decode step: sequences processed in array order.
 * slots: host int32 [n]; cow_pairs: host int32 [n][2], the first *num_cow
 * rows filled; *num_done = sequences processed before any failure. */
PA_API pa_status pa_alloc_append_slots(pa_allocator* a, const int64_t* seq_ids,
                                int n, int32_t* slots, int32_t* cow_pairs,
                                int* num_cow, int* num_done);

/* Release every block of seq_id (logical order) and forget the sequence. */
PA_API pa_status pa_alloc_free_seq(pa_allocator* a, int64_t seq_id);

/* Copy seq_id's table (physical ids, logical order) into out[0..cap);
 * *n = its full length (PA_ERR_INVALID_ARG if cap < *n). */
PA_API pa_status pa_alloc_get_table(const pa_allocator* a, int64_t seq_id,
                             int32_t* out, int cap, int* n);

PA_API pa_status pa_alloc_seq_len(const pa_allocator* a, int64_t seq_id,
                           int64_t* len);

/* One decode step of a batch planned in a single call: the next slot of
 * every sequence of seq_ids, in index order, exactly as
 * pa_alloc_append_slots gives them (growth, copy-on-write pairs), then the
 * batch's dense tables and lengths after those appends, exactly as
 * pa_alloc_build_tables gives them ("Phase 7 · Document 04 —
 * PagedAttention", §2 on-demand allocation and block sharing; lux-666 notes
 * "PagedAttention", 最小模型: the table the kernel reads is the block
 * manager's). Every output is written straight into the caller's buffers,
 * which may be the pinned host memory the step's kernels read in place.
 * seq_ids  host int64 [n], distinct
 * slots    int32 [n]; cow_pairs int32 [n][2] (src, dst) with *num_cow rows
 *          written; table int32 [n][max_blocks] (rows padded with fill);
 *          seq_lens int32 [n] (lengths after the append)
 * All or nothing: the whole batch is checked first (every sequence known,
 * not swapped out, listed once, its table after the append within
 * max_blocks) and the blocks its growth and copies take are counted against
 * the free list; a refused call changes nothing but the failure counter.
 * Errors: PA_ERR_INVALID_ARG, PA_ERR_OUT_OF_BLOCKS. */
PA_API pa_status pa_alloc_plan_step(pa_allocator* a, const int64_t* seq_ids, int n,
                             int max_blocks, int32_t fill, int32_t* slots,
                             int32_t* cow_pairs, int* num_cow, int32_t* table,
                             int32_t* seq_lens);

/* One decode step in one call: pa_alloc_plan_step for the batch seq_ids
 * (tables padded with -1), then, on `stream`, pa_copy_blocks of its
 * copy-on-write pairs (if any) and pa_decode_append_attention (every
 * sequence's new K/V row, then attention over the tables and lengths just
 * planned, in one kernel) ("Phase 7
 * · Document 04 — PagedAttention", §2 on-demand allocation and block
 * sharing; lux-666 notes "PagedAttention", 最小模型). The plan is written
 * into slot_mapping [n], cow_pairs [n][2] (*num_cow rows), block_table
 * [n][max_blocks] and seq_lens [n]: pinned host memory, which the kernels
 * read in place through its device mapping (the host writes them before the
 * launches; they must not be rewritten until this step's kernels have
 * completed). The block size is the block manager's; num_blocks must be its
 * pool size. q, k_new, v_new, the pools, out and the workspace are as in the
 * calls above (k_new/v_new row i and q row i belong to seq_ids[i]).
 * Errors: those of the four calls. A refused plan launches nothing and
 * changes nothing; an error after the plan leaves the block manager
 * advanced by the step. */
PA_API pa_status pa_decode_step(pa_allocator* a, const int64_t* seq_ids, int num_seqs,
                         int max_blocks, int32_t* slot_mapping, int32_t* cow_pairs,
                         int32_t* block_table, int32_t* seq_lens, int* num_cow,
                         const pa_half* q, const pa_half* k_new, const pa_half* v_new,
                         pa_half* k_pool, pa_half* v_pool, int num_q_heads,
                         int num_kv_heads, int head_dim, int num_blocks,
                         int64_t pool_block_stride, float scale, pa_half* out,
                         void* workspace, size_t workspace_bytes, int partition_tokens,
                         pa_stream_t stream);

/* pa_decode_step over an E4M3 cache: the same plan, then pa_copy_blocks_fp8,
 * pa_append_kv_fp8 (each new row quantized with the KV head's k_scale /
 * v_scale, device fp32 [num_kv_heads]) and pa_decode_attention_fp8 on
 * `stream`; arguments and plan buffers as for pa_decode_step, pools of
 * one-byte codes ("Phase 7 · Document 04 — PagedAttention", §11: the fp8
 * KV cache). Errors: those of the four calls, as for pa_decode_step. */
PA_API pa_status pa_decode_step_fp8(pa_allocator* a, const int64_t* seq_ids, int num_seqs,
                             int max_blocks, int32_t* slot_mapping, int32_t* cow_pairs,
                             int32_t* block_table, int32_t* seq_lens, int* num_cow,
                             const pa_half* q, const pa_half* k_new, const pa_half* v_new,
                             uint8_t* k_pool, uint8_t* v_pool, const float* k_scale,
                             const float* v_scale, int num_q_heads, int num_kv_heads,
                             int head_dim, int num_blocks, int64_t pool_block_stride,
                             float scale, pa_half* out, void* workspace,
                             size_t workspace_bytes, int partition_tokens, pa_stream_t stream);

/* Dense tables for a batch: table host int32 [n][max_blocks] (rows padded
 * with `fill`), seq_lens host int32 [n] = current lengths. */
PA_API pa_status pa_alloc_build_tables(const pa_allocator* a, const int64_t* seq_ids,
                                int n, int max_blocks, int32_t fill,
                                int32_t* table, int32_t* seq_lens);

/* The whole blocks that every sequence of a batch begins with ("Phase 7 ·
 * Document 04 — PagedAttention", §2 block sharing and §3 Mental Model;
 * lux-666 notes "PagedAttention", prefix sharing): the longest run of leading
 * table entries that is the same in every table and whose blocks every
 * sequence attends in full (run length k with k * block_size <= each length).
 * This is the prefix pa_decode_attention_shared_prefix takes.
 * seq_ids: host int64 [n]; blocks: host int32 [cap] receives the run's
 * physical ids in logical order; *num_blocks = the run's length. An empty
 * batch has none; one sequence's run is its whole blocks.
 * Sizing: when cap < the run's length (or blocks is NULL with a nonempty
 * run) the call returns PA_ERR_INVALID_ARG with *num_blocks set to the
 * length needed and `blocks` untouched, so a caller can ask with cap = 0.
 * Errors: PA_ERR_INVALID_ARG (bad arguments, a sequence unknown or swapped
 *         out; *num_blocks is then 0). The block manager's state is never
 *         modified. */
PA_API pa_status pa_alloc_shared_prefix(const pa_allocator* a, const int64_t* seq_ids,
                                 int n, int32_t* blocks, int cap, int* num_blocks);

PA_API pa_status pa_alloc_stats(const pa_allocator* a, pa_alloc_stats_t* out);

/* free_order: host int32 [num_blocks], front to back, *num_free entries
 * valid and the rest set to -1; refcounts: host int32 [num_blocks]. */
PA_API pa_status pa_alloc_export_state(const pa_allocator* a, int32_t* free_order,
                                int* num_free, int32_t* refcounts);

/* ------------------------------------------------------------------------
 * Swapping a sequence's blocks to a host pool and back (preemption).
 *
 * Source: "Phase 7 · Document 04 — PagedAttention", §9 (under memory
 * pressure the scheduler may evict/recompute or swap a sequence's blocks)
 * and §10 (preemption by evict/recompute/swap is a latency event). The pages
 * give no mechanism; this library's reading: the block manager owns an
 * optional host pool with its own FIFO free list (ids 0 .. num_host_blocks-1
 * of a caller-owned host pool with the device pool's block shape);
 * pa_alloc_swap_out takes one host block per logical block of the sequence
 * (all or nothing), writes the (device, host) pairs to copy in logical order
 * and drops the sequence's device references (blocks other tables share stay
 * for them); the sequence keeps its length but cannot append, fork or be
 * tabled until pa_alloc_swap_in takes fresh private device blocks (all or
 * nothing), writes the (host, device) pairs and returns the host blocks.
 * pa_alloc_free_seq of a swapped-out sequence returns its host blocks.
 * Issue the block copy (pa_swap_blocks) for swap-out pairs before any later
 * write can reuse the released device blocks (stream order suffices).
 * ---------------------------------------------------------------------- */

/* Host pool of num_host_blocks blocks; order = initial host free list
 * (a permutation, NULL = ascending). Once per handle. */
PA_API pa_status pa_alloc_add_host_pool(pa_allocator* a, int num_host_blocks,
                                        const int32_t* order);

/* pairs: host int32 [cap][2]; *n = blocks moved (pairs written). */
PA_API pa_status pa_alloc_swap_out(pa_allocator* a, int64_t seq_id, int32_t* pairs,
                                   int cap, int* n);
PA_API pa_status pa_alloc_swap_in(pa_allocator* a, int64_t seq_id, int32_t* pairs,
                                  int cap, int* n);

/* free_order: host int32 [num_host_blocks] (front to back, *num_free valid,
 * the rest -1); counts: host int64 [4] = host blocks, swapped-out sequences,
 * swap-outs, swap-ins. */
PA_API pa_status pa_alloc_export_host_state(const pa_allocator* a, int32_t* free_order,
                                            int* num_free, int64_t* counts);

/* Copy whole blocks between two pool pairs: block pairs[i][1] of dst_k/dst_v
 * := block pairs[i][0] of src_k/src_v, each block block_bytes bytes (a
 * multiple of 16; BS * Hkv * D * element size). Block b of a source pool
 * starts at b * src_block_stride bytes, of a destination pool at b *
 * dst_block_stride bytes (0 = block_bytes; otherwise at least block_bytes and
 * a multiple of 16). A one-pool record array moves as K and V members
 * (v = k + block_bytes, stride 2*block_bytes) or, with src_v == dst_v == NULL,
 * as whole records of block_bytes each. Each pool, and pairs (int32
 * [num_pairs][2]), may be device memory or pinned (page-locked) host memory,
 * which the kernel reads and writes through its device mapping. An id outside
 * [0, src_blocks) or [0, dst_blocks) skips that pair and sets
 * PA_DEVERR_BAD_BLOCK. Errors: PA_ERR_INVALID_ARG (pageable host memory,
 * NULL or misaligned pointers), PA_ERR_CUDA. */
PA_API pa_status pa_swap_blocks(const void* src_k, const void* src_v, int src_blocks,
                                int64_t src_block_stride, void* dst_k, void* dst_v,
                                int dst_blocks, int64_t dst_block_stride,
                                const int32_t* pairs, int num_pairs, int block_bytes,
                                pa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
