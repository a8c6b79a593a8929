/*
 * pkv.h — C ABI of the GB300 paged KV-cache library (libpkv.so).
 *
 * The library implements the data path of PagedAttention: a pool of equally
 * sized physical KV blocks handed out through per-sequence block tables, the
 * slot write of each step's new keys and values, the copy-on-write block copy,
 * and single-token decode attention that gathers K/V through the tables.
 *
 * Sources (web pages on PagedAttention):
 *   [A] "PagedAttention Memory Management" (apxml course page), sections
 *       "Calculating Physical Block Sizes" and "Complex Topologies and Memory
 *       Sharing".
 *   [B] "What problem does PagedAttention solve for the KV cache in vLLM?"
 *       (katajob Q&A), sections "What the KV cache is", "The paging idea" and
 *       "Sharing, the second dividend".
 *   [C] foundry page on paged block allocation for the KV cache, sections
 *       "In and out", "Concept", "The knobs", "Effect", "Evals" and
 *       "Failure modes".
 *   [D] "PagedAttention, clearly explained" (thread).
 *
 * Conventions
 *   - Every call that can fail returns a pkv_status; pkv_last_error() gives a
 *     message for the calling thread's last failure.
 *   - Host allocator calls are all-or-nothing: on error nothing changes.
 *   - Device buffers are owned by the caller (plain device pointers).  The
 *     library never allocates or frees device memory at run time; its only
 *     device memory is two fixed static arrays resident on each GPU that
 *     loads it: the device error word (pkv_device_status) and the scratch of
 *     pkv_attention_decode_noalloc.  Their addresses are looked up once per
 *     device and kept, so cudaDeviceReset while the library is in use is not
 *     supported.  A pool handle owns only host-side allocator state.
 *   - Device calls enqueue kernels on the given CUDA stream (a cudaStream_t
 *     passed as void*, NULL = legacy default stream) and return without
 *     synchronising; a launch failure returns PKV_ERR_CUDA.
 *   - A pool handle is not thread-safe; use one thread per handle.
 *
 * Memory layout of one layer's cache (the pages fix none; this is the
 * library's reading of "one large pre-allocated tensor per layer" [C]):
 *   k_cache, v_cache : [num_blocks][num_kv_heads][block_size][head_dim]
 *   elements of kv_dtype, row-major, 16-byte aligned base.  Physical slot s is
 *   block s / block_size, offset s % block_size.  A block id names the same
 *   slot range in every layer's tensors, so one block holds
 *   pkv_block_bytes(L, ...) bytes over all layers [A].
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1,   /* bad pointer, size, id or dtype combination */
  PKV_ERR_OUT_OF_BLOCKS = 2, /* the free-block stack cannot satisfy the call */
  PKV_ERR_UNKNOWN_SEQ = 3,   /* no live sequence with that id */
  PKV_ERR_UNSUPPORTED = 4,   /* valid but not compiled (head_dim, block_size, group) */
  PKV_ERR_CUDA = 5           /* a CUDA runtime call or kernel launch failed */
} pkv_status;

/* Element types.  PKV_E4M3 is the OCP 8-bit E4M3 ("FN": no infinities,
 * max 448) format with one scale per tensor (or per KV head, see
 * pkv_kv_desc.head_scales); the cache stores e4m3(round_fp32(x * inv_scale))
 * and reads back e4m3 * scale. */
typedef enum { PKV_F32 = 0, PKV_F16 = 1, PKV_BF16 = 2, PKV_E4M3 = 3 } pkv_dtype;

/* Shape of one layer's K/V cache tensors.
 * head_scales (E4M3 caches only; NULL otherwise): device float32
 * [4][num_kv_heads], 4-byte aligned, owned by the caller: row 0 the K scale
 * of each KV head, row 1 the V scale, row 2 the K inverse scale (what a slot
 * write multiplies by), row 3 the V inverse scale.  When set, KV head h is
 * stored and read with its own scales and the per-tensor scale arguments of
 * every call are ignored; NULL keeps the per-tensor arguments.  A cache's
 * bytes must be written and read with the same choice. */
typedef struct {
  int32_t num_blocks;   /* physical blocks in the pool */
  int32_t num_kv_heads; /* N_kv */
  int32_t head_dim;     /* D_head: 64 or 128 */
  int32_t block_size;   /* T_block tokens per block: 16 or 32 */
  int32_t kv_dtype;     /* pkv_dtype of the cache */
  const float* head_scales; /* per-KV-head E4M3 scales, or NULL */
} pkv_kv_desc;

typedef struct pkv_pool pkv_pool;

/* ------------------------------------------------------------ sizing [A] */

/* Bytes of one physical block, 2 * L * N_kv * D_head * T_block * P_bytes
 * ([A] "Calculating Physical Block Sizes").  Returns 0 if a factor is <= 0. */
PKV_API uint64_t pkv_block_bytes(int32_t num_layers, int32_t num_kv_heads, int32_t head_dim,
                         int32_t block_size, int32_t elem_bytes);

/* Whole blocks that fit budget_bytes (floor); 0 if block_bytes is 0. */
PKV_API uint64_t pkv_num_blocks_for_budget(uint64_t budget_bytes, uint64_t block_bytes);

/* Bytes per element of a pkv_dtype, 0 if unknown. */
PKV_API int32_t pkv_dtype_bytes(int32_t dtype);

/* ------------------------------------------------- host allocator [B][C][D]
 * A free-block stack, per-sequence block tables and per-block reference
 * counts.  Blocks are popped one per block_size tokens, only when the
 * previous block is full [D][C "Concept"]; fork copies the table and counts
 * each shared block once more [C "Concept"][A "Complex Topologies"]; a token
 * written into a partly filled block that other sequences still map first
 * moves this sequence onto a private copy (copy-on-write) [B "Sharing"];
 * finishing a sequence returns blocks whose count reaches zero [D].
 * Order rules (needed to reproduce tables exactly): the stack is LIFO; the
 * initial order is given top first (default: block 0 on top, then 1, 2, ...);
 * freeing pushes a sequence's blocks in logical order. */

/* Create an allocator over num_blocks blocks of block_size tokens.
 * initial_free_order: NULL or a host array of num_blocks distinct ids in
 * [0, num_blocks), top of the stack first.  *out receives the handle. */
PKV_API pkv_status pkv_pool_create(int32_t num_blocks, int32_t block_size,
                           const int32_t* initial_free_order, pkv_pool** out);
PKV_API void pkv_pool_destroy(pkv_pool* pool);

/* Register an empty sequence.  INVALID_ARG if the id is live. */
PKV_API pkv_status pkv_seq_create(pkv_pool* pool, int64_t seq_id);

/* Reserve slots for n_new tokens of one sequence.
 * slots_out   : host int64[n_new], slot of each new token
 *               (block * block_size + offset).
 * cow_out     : host int32[2 * cow_cap], receives (src, dst) block pairs that
 *               must be copied (pkv_copy_blocks) before the tokens are
 *               written; at most one pair per call.  May be NULL if cow_cap 0.
 * n_cow_out   : number of pairs written.
 * OUT_OF_BLOCKS if the stack cannot supply the blocks; INVALID_ARG if a copy
 * is needed and cow_cap is 0.  All-or-nothing. */
PKV_API pkv_status pkv_seq_append(pkv_pool* pool, int64_t seq_id, int32_t n_new, int64_t* slots_out,
                          int32_t* cow_out, int32_t cow_cap, int32_t* n_cow_out);

/* One decode step: append one token to each of n_seqs sequences, in order.
 * slots_out: host int64[n_seqs]; cow_out / cow_cap / n_cow_out as above (at
 * most n_seqs pairs).  A sequence named k times gets k tokens, in batch
 * order.  All-or-nothing over the whole batch: if any sequence cannot be
 * served, no sequence changes. */
PKV_API pkv_status pkv_batch_append(pkv_pool* pool, const int64_t* seq_ids, int32_t n_seqs,
                            int64_t* slots_out, int32_t* cow_out, int32_t cow_cap,
                            int32_t* n_cow_out);

/* The child (a new id) maps every block of the parent; counts + 1. */
PKV_API pkv_status pkv_seq_fork(pkv_pool* pool, int64_t parent_id, int64_t child_id);

/* Finish a sequence and return its unshared blocks to the stack (with prefix
 * caching, a published block whose count reaches 0 is kept for reuse
 * instead: see pkv_pool_enable_prefix_cache). */
PKV_API pkv_status pkv_seq_free(pkv_pool* pool, int64_t seq_id);

/* Copy one block table (logical order) into out[cap]; *n_blocks and
 * *context_len receive its length and the sequence's token count.  out may
 * be NULL when cap is 0 (query only); INVALID_ARG if cap is too small. */
PKV_API pkv_status pkv_seq_table(const pkv_pool* pool, int64_t seq_id, int32_t* out, int32_t cap,
                         int32_t* n_blocks, int64_t* context_len);

/* Tables of a batch as host int32[n_seqs][max_blocks], padded with -1, and
 * their context lengths int32[n_seqs].  INVALID_ARG if a table is longer
 * than max_blocks or a length exceeds INT32_MAX. */
PKV_API pkv_status pkv_block_tables(const pkv_pool* pool, const int64_t* seq_ids, int32_t n_seqs,
                            int32_t max_blocks, int32_t* tables_out, int32_t* context_lens_out);

/* pkv_block_tables for a buffer kept across decode steps: the same result
 * (row i = the table of seq_ids[i] padded with -1, context lengths), but a
 * row is only rewritten from its last entry on when it was last written by
 * this call for the same sequence and max_blocks, so a step costs O(n_seqs +
 * new entries) instead of O(n_seqs * max_blocks).  Between two calls a live
 * sequence's table only grows at its end, and a copy-on-write replaces only
 * the entry its next token lands in, which is never before the last entry
 * the row held (a table gains a block only when the previous one is full
 * [D][C "Concept"]; copy-on-write replaces the shared block being written
 * [A "Complex Topologies"]).
 *   tables_inout      host int32[n_seqs][max_blocks], caller-owned, kept
 *                     between calls (its first contents do not matter).
 *   rows_inout        host int64[n_seqs][2], caller-owned, opaque; all zero
 *                     the first time (or to force a full rewrite).  It
 *                     names the sequence incarnation a row holds (unique for
 *                     the pool's life: a sequence created again under the
 *                     same id, a fork child, a re-admitted sequence each get
 *                     a new one), so batches may reorder or replace rows.
 *   context_lens_out  host int32[n_seqs].
 * Errors as pkv_block_tables, checked before anything is written.  The
 * caller must not change a row between calls other than through this call
 * (or must zero its state). */
PKV_API pkv_status pkv_block_tables_update(const pkv_pool* pool, const int64_t* seq_ids,
                                           int32_t n_seqs, int32_t max_blocks,
                                           int32_t* tables_inout, int64_t* rows_inout,
                                           int32_t* context_lens_out);

/* Shared prefix of a batch: *n_blocks receives the number k of leading
 * block-table entries that every listed sequence maps to the same physical
 * blocks (one stored copy serves them all: [A "Complex Topologies"], [B
 * "Sharing, the second dividend"]), limited so that k * block_size <= len - 1
 * for every sequence (the block holding a sequence's last position, the one a
 * decode step writes, is never part of it).  Pass k to
 * pkv_attention_decode_shared_prefix.  UNKNOWN_SEQ / INVALID_ARG as
 * pkv_block_tables; 0 for an empty batch. */
PKV_API pkv_status pkv_shared_prefix_blocks(const pkv_pool* pool, const int64_t* seq_ids,
                                            int32_t n_seqs, int32_t* n_blocks);

/* Reference count of one block (0 = free). */
PKV_API pkv_status pkv_block_refcount(const pkv_pool* pool, int32_t block, int32_t* refcount);

/* Blocks an append can take: the free stack, plus (with prefix caching) the
 * published blocks nobody references. */
PKV_API int32_t pkv_num_free_blocks(const pkv_pool* pool);

/* The free stack, top first, into out[cap]; *n receives its size. */
PKV_API pkv_status pkv_free_stack(const pkv_pool* pool, int32_t* out, int32_t cap, int32_t* n);

/* Live sequences, the tokens they hold (a shared token once per sequence
 * holding it) and the blocks in use: referenced by a sequence (a shared
 * block counted once), or, with prefix caching, neither free nor reusable.
 * Without sharing, used_blocks * block_size - live_tokens is the
 * reserved-but-empty space the pages call waste ([C "Evals"]). */
PKV_API pkv_status pkv_pool_usage(const pkv_pool* pool, int64_t* live_seqs, int64_t* live_tokens,
                          int64_t* used_blocks);

/* ------------------------------------------------------ device kernels */

/* Slot write ("the number of new tokens about to be written" [C "In and
 * out"]): for token i with slot_mapping[i] = s >= 0,
 *   k_cache[s / T][h][s % T][:] = k[i][h][:]   (and v likewise)
 * for every KV head h.  Tokens with s < 0, or s >= num_blocks * T, are
 * skipped.
 *   k, v          : device [n_tokens][num_kv_heads][head_dim] of src_dtype
 *                   (F32, F16 or BF16), 16-byte aligned, contiguous.
 *   slot_mapping  : device int64[n_tokens].
 *   k_inv_scale, v_inv_scale : for an E4M3 cache the stored byte is
 *                   e4m3_satfinite(round_fp32(x * inv_scale)); ignored
 *                   otherwise.  A 16/32-bit cache requires src_dtype ==
 *                   kv_dtype and stores the input bits unchanged. */
PKV_API pkv_status pkv_write(void* k_cache, void* v_cache, const void* k, const void* v,
                     int32_t src_dtype, const int64_t* slot_mapping, int32_t n_tokens,
                     const pkv_kv_desc* desc, float k_inv_scale, float v_inv_scale,
                     void* stream);

/* Copy-on-write block copy ([B "Sharing"], [C "Concept"]): for each pair
 * (src, dst) and each layer l, block dst of k_caches[l] and v_caches[l]
 * becomes a byte copy of block src.
 *   k_caches, v_caches : host arrays of num_layers device pointers (<= 128).
 *   src_dst            : HOST int32[2 * n_pairs] (as returned by the
 *                        allocator); ids are checked against num_blocks.
 * Pairs must not overlap (no dst appears twice or as another pair's src); the
 * allocator never produces overlapping pairs. */
PKV_API pkv_status pkv_copy_blocks(void* const* k_caches, void* const* v_caches, int32_t num_layers,
                           const int32_t* src_dst, int32_t n_pairs, const pkv_kv_desc* desc,
                           void* stream);

/* Workspace bytes pkv_attention_decode needs for these sizes (split-K
 * partial results and merge counters).  0 if no split is needed. */
PKV_API size_t pkv_attention_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t max_blocks,
                                     const pkv_kv_desc* desc, int32_t partition_tokens);

/* Decode-attention kernel selection, process-wide (default AUTO).  AUTO uses
 * the tensor-core split kernel (TMA-staged tiles, MMA for q.K^T and p.V, one
 * CTA per (KV head, sequence, split), split-K merge fused) for 16-bit and
 * E4M3 caches with head_dim 128 (16-bit also 64), groups of up to 16 query
 * heads and partitions of at most 1024 blocks, and the CUDA-core kernel
 * otherwise.  SIMT forces the CUDA-core kernel; TENSOR_CORE makes
 * pkv_attention_decode return PKV_ERR_UNSUPPORTED for sizes it does not
 * cover, and keeps the positions past a shared prefix on the split kernel
 * (AUTO streams them through the tail queue where it applies: 16-bit caches,
 * head_dim 128, block size 16).  All kernels compute the same result within
 * rounding; the tail queue and the split kernel at the same partition give
 * the same bits. */
#define PKV_KERNEL_AUTO 0
#define PKV_KERNEL_SIMT 1
#define PKV_KERNEL_TENSOR_CORE 2
PKV_API pkv_status pkv_set_attention_kernel(int32_t kind);

/* Partition (tokens per split) pkv_attention_decode uses for these sizes.
 * A pair of context ctx gets ceil(ctx / partition) splits (the tensor-core
 * kernel shares its 64-token tiles evenly over them).  For partition_tokens 0
 * it is the smallest multiple of 64 (and of the block size) for which the
 * expected splits fit in one wave of resident CTAs on the current device; when
 * the (sequence, KV head) pairs alone fill two waves, half the longest context
 * (max_blocks * T / 2, rounded up), at least 4096 and at most 8192 tokens. */
PKV_API int32_t pkv_attention_partition(int32_t num_seqs, int32_t max_blocks, const pkv_kv_desc* desc,
                                int32_t partition_tokens);

/* Single-token decode attention through block tables ([D]: "the attention
 * kernel reads the block table and gathers keys and values"; [C "Concept"]):
 *   out[s][j][:] = softmax_p( q[s][j] . K_s[p] * softmax_scale ) V_s[p]
 * over logical positions p in [0, context_lens[s]), where
 *   K_s[p] = k_cache[block_tables[s][p / T]][j / G][p % T][:] * k_scale
 * (V likewise), G = num_q_heads / num_kv_heads (query head j reads KV head
 * j / G).  k_scale / v_scale multiply E4M3 caches and are ignored otherwise.
 *   out, q        : device [num_seqs][num_q_heads][head_dim] of q_dtype
 *                   (F32 with an F32 cache, F16 or BF16 with 16-bit and E4M3
 *                   caches); out has q's dtype.
 *   block_tables  : device int32[num_seqs][max_blocks]; entries past
 *                   ceil(ctx / T) are not read.
 *   context_lens  : device int32[num_seqs]; a length of 0 gives a zero output.
 *   partition_tokens : tokens per split-K partition, or 0 for an automatic
 *                   choice; a multiple of 64 and of block_size.  Split and
 *                   tile boundaries depend only on logical positions and
 *                   lengths, so results do not depend on which physical
 *                   blocks hold the tokens.
 *   workspace     : device buffer of at least
 *                   pkv_attention_workspace_bytes(...) bytes, 256-byte
 *                   aligned, ZERO-FILLED before its first use (every call
 *                   leaves it zeroed again); may be NULL if that size is 0.
 *                   Calls that share one workspace must not overlap in time.
 * The tensor-core kernels are launched with programmatic stream
 * serialization: they may be scheduled while the previous kernel in the stream
 * drains, and read no input before that kernel has completed.
 * Inputs the kernel finds invalid (a table entry outside [0, num_blocks) or a
 * context length outside [0, max_blocks * T]) make the affected heads' output
 * NaN; nothing outside the given buffers is read or written. */
PKV_API pkv_status pkv_attention_decode(void* out, const void* q, int32_t q_dtype, const void* k_cache,
                                const void* v_cache, const int32_t* block_tables,
                                int32_t max_blocks, const int32_t* context_lens,
                                int32_t num_seqs, int32_t num_q_heads, const pkv_kv_desc* desc,
                                float softmax_scale, float k_scale, float v_scale,
                                int32_t partition_tokens, void* workspace,
                                size_t workspace_bytes, void* stream);

/* One decode step: the step's new K/V of each sequence written at its logical
 * position ctx_s - 1 (the slot its block table gives: [C "In and out"], the
 * new tokens written into reserved slots; the context length counts the
 * step's token), then pkv_attention_decode over positions 0 .. ctx_s - 1.
 * The same as pkv_write (slots of positions ctx_s - 1) followed by
 * pkv_attention_decode, in one launch where the tensor-core split kernel
 * applies: the CTA that holds position ctx_s - 1 stores the token before it
 * reads that tile (else a small write kernel runs first).
 *   k_new, v_new : device [num_seqs][num_kv_heads][head_dim] in q_dtype
 *                  (E4M3 caches: rounded as x * k_inv_scale / x *
 *                  v_inv_scale, as pkv_write does).
 * A sequence with context 0 (or an invalid length or table entry) writes
 * nothing.  Block copies (copy-on-write) must run before this call.  Other
 * arguments as pkv_attention_decode. */
PKV_API pkv_status pkv_decode_step(void* out, const void* q, int32_t q_dtype, void* k_cache,
                                   void* v_cache, const void* k_new, const void* v_new,
                                   const int32_t* block_tables, int32_t max_blocks,
                                   const int32_t* context_lens, int32_t num_seqs,
                                   int32_t num_q_heads, const pkv_kv_desc* desc,
                                   float softmax_scale, float k_scale, float v_scale,
                                   float k_inv_scale, float v_inv_scale, int32_t partition_tokens,
                                   void* workspace, size_t workspace_bytes, void* stream);

/* Decode attention over a shared prefix ([A "Complex Topologies and Memory
 * Sharing"]: several sequences map the same prompt blocks; [B "Sharing, the
 * second dividend"]).  The same result as pkv_attention_decode (within
 * rounding), for a batch whose first prefix_blocks table entries are the
 * same physical blocks in every row (pkv_shared_prefix_blocks).  The call
 * reads those blocks once for all sequences instead of once per sequence:
 *   - a shared-prefix pass on the 5th-generation tensor cores (tcgen05)
 *     attends the queries of all sequences and heads of a KV head (M rows =
 *     num_seqs * group) to positions [0, P), P = prefix_blocks * block_size,
 *     read through row 0 of block_tables, and leaves per-row partial results
 *     (max, sum, unnormalised output) in the workspace;
 *   - the decode kernel attends positions [P, ctx) of each sequence and
 *     leaves its partials in the workspace too (16-bit caches at head_dim 128
 *     and block size 16: one-warp CTAs on every resident slot take (sequence,
 *     split, KV head) units from a queue in the workspace, longest first,
 *     keeping their copies streaming from one unit into the next);
 *   - a merge kernel combines every row's partials into out.
 * Because the reduction is split differently, results can differ from
 * pkv_attention_decode in the low-order bits ([C "Effect"]: reusing shared
 * blocks changes how the attention reduction is tiled).
 * partition_tokens (positions per split past the prefix): 0 picks 512 for
 * 16-bit caches at head_dim 128 and block size 16, else as
 * pkv_attention_partition with the longest context less P.
 * Requirements: every row's first prefix_blocks entries equal row 0's and
 * every context length is > P (a row that breaks either gets NaN outputs and
 * sets PKV_DEVICE_BAD_SHARED_PREFIX or PKV_DEVICE_BAD_LENGTH);
 * 0 <= prefix_blocks <= max_blocks.  The shared-prefix pass covers head_dim
 * 128 with 16-bit or E4M3 caches and softmax_scale > 0 under the tensor-core
 * decode kernel; for other shapes, for prefix_blocks 0, or with
 * PKV_KERNEL_SIMT the call is pkv_attention_decode.
 *   workspace : pkv_shared_prefix_workspace_bytes(...) bytes, 256-byte
 *               aligned, zero-filled before first use (left zeroed).
 * The prefix pass is launched first (on about a quarter of the SMs), then the
 * decode kernel as its programmatic dependent, which starts on the SMs the
 * pass leaves free (neither waits for the other; the decode grid completes
 * only after the pass: its last CTA waits for the pass's grid), then the
 * merge kernel. */
PKV_API size_t pkv_shared_prefix_workspace_bytes(int32_t num_seqs, int32_t num_q_heads,
                                                 int32_t max_blocks, const pkv_kv_desc* desc,
                                                 int32_t prefix_blocks, int32_t partition_tokens);
PKV_API pkv_status pkv_attention_decode_shared_prefix(
    void* out, const void* q, int32_t q_dtype, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int32_t max_blocks, const int32_t* context_lens,
    int32_t num_seqs, int32_t num_q_heads, const pkv_kv_desc* desc, int32_t prefix_blocks,
    float softmax_scale, float k_scale, float v_scale, int32_t partition_tokens, void* workspace,
    size_t workspace_bytes, void* stream);

/* pkv_decode_step over a shared prefix: the step's K/V written at position
 * ctx_s - 1 (which is past the prefix), then
 * pkv_attention_decode_shared_prefix; arguments as those two calls. */
PKV_API pkv_status pkv_decode_step_shared_prefix(
    void* out, const void* q, int32_t q_dtype, void* k_cache, void* v_cache, const void* k_new,
    const void* v_new, const int32_t* block_tables, int32_t max_blocks,
    const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads, const pkv_kv_desc* desc,
    int32_t prefix_blocks, float softmax_scale, float k_scale, float v_scale, float k_inv_scale,
    float v_inv_scale, int32_t partition_tokens, void* workspace, size_t workspace_bytes,
    void* stream);

/* ------------------------------------------------------ device errors
 * Invalid inputs that only the GPU sees (a table entry outside [0,
 * num_blocks), a context length outside its range, a broken shared-prefix
 * declaration) and bounded waits that gave up turn the affected outputs into
 * NaN and set bits in one error word per device, which every attention
 * kernel of the library ORs into (sticky until cleared). */
#define PKV_DEVICE_BAD_LENGTH 1          /* a context / chunk length outside its range */
#define PKV_DEVICE_BAD_TABLE 2           /* a block-table entry outside [0, num_blocks) */
#define PKV_DEVICE_WAIT_TIMEOUT 4        /* a bounded wait for a copy or an MMA gave up */
#define PKV_DEVICE_BAD_SHARED_PREFIX 8   /* a row does not map the declared shared prefix */

/* Synchronise `stream` (NULL = legacy default stream), then *flags receives
 * the current device's error word; clear != 0 then resets it to 0 (on that
 * stream).  The first call on a device looks up the word's address; make it
 * before any stream capture.  PKV_ERR_CUDA if a CUDA call fails. */
PKV_API pkv_status pkv_device_status(int32_t* flags, int32_t clear, void* stream);

/* Give-up limit, in nanoseconds, of the decode kernels' waits for a K/V stage
 * (default 50,000,000 = 50 ms), process-wide; 0 makes every stage wait give
 * up at once (used to exercise the failure path: the CTA still waits, with
 * its own 10 ms limit per copy, for the copies it has in flight, then writes
 * NaN and sets PKV_DEVICE_WAIT_TIMEOUT). */
PKV_API pkv_status pkv_set_stage_wait_limit(uint64_t nanoseconds);

/* Bytes of the fixed scratch array behind pkv_attention_decode_noalloc. */
#define PKV_NOALLOC_SCRATCH_BYTES (16u << 20)

/* Decode attention that allocates nothing.  The pages have no counterpart;
 * this is a library convenience for callers that cannot allocate device
 * memory: a plug-in whose host runtime owns all device memory and hands it
 * only input and output buffers, or a serving loop that must not call
 * cudaMalloc (which can synchronise the device) while it runs.
 * Arguments and result are those of pkv_attention_decode without the
 * workspace: the split-K scratch is a fixed array of
 * PKV_NOALLOC_SCRATCH_BYTES (16 MiB) in device memory that the library
 * declares and every GPU that loads the library holds until the process
 * exits.  Sizes whose scratch (pkv_attention_workspace_bytes) exceeds it are
 * rejected with PKV_ERR_INVALID_ARG before anything runs.
 * The first call on a device, with that device current, looks up the array's
 * device address (cudaGetSymbolAddress) and caches it; make that first call
 * before any stream capture.  All calls on a device share the array: calls
 * that overlap on the GPU race.  A completed call leaves the array's split-K
 * counters at zero; each call also clears them on its stream before the
 * kernel runs, so a call that never completed leaves nothing behind.
 * Nothing else needs clearing between calls. */
PKV_API pkv_status pkv_attention_decode_noalloc(void* out, const void* q, int32_t q_dtype,
                                                const void* k_cache, const void* v_cache,
                                                const int32_t* block_tables, int32_t max_blocks,
                                                const int32_t* context_lens, int32_t num_seqs,
                                                int32_t num_q_heads, const pkv_kv_desc* desc,
                                                float softmax_scale, float k_scale, float v_scale,
                                                int32_t partition_tokens, void* stream);

/* Prefill (multi-query, causal) attention through block tables: the chunk
 * of sequence s is its last n_s = query_start[s+1] - query_start[s] logical
 * positions ctx_s - n_s .. ctx_s - 1, whose K/V are already in the pool
 * (written by pkv_write, like a decode step's token); the query at position
 * p attends to positions 0 .. p ([B "What the KV cache is"]: every earlier
 * token's key and value serve the next token's attention; [B "The paging
 * idea"]: a sequence starts with the blocks of its prompt; [D]: later tokens
 * attend over the cached prompt):
 *   out[r][j][:] = softmax_{p' <= p}( q[r][j] . K_s[p'] * softmax_scale ) V_s[p']
 * for row r = query_start[s] + i at position p = ctx_s - n_s + i, K_s, V_s
 * gathered through block_tables as in pkv_attention_decode (query head j
 * reads KV head j / G).  A one-token chunk is decode attention.
 *   out, q        : device [total_q][num_q_heads][head_dim], chunks packed in
 *                   sequence order; q dtype = the cache dtype (F16 or BF16),
 *                   or F16 / BF16 with an E4M3 cache (K, V read as
 *                   e4m3 * k_scale / v_scale).
 *   query_start   : device int32[num_seqs + 1], non-decreasing, [0] = 0,
 *                   [num_seqs] = total_q.
 *   max_query_len : >= every n_s (sets the grid).
 *   context_lens  : device int32[num_seqs], chunk included (n_s <= ctx_s).
 *   k_scale, v_scale : E4M3 scales (ignored for 16-bit caches).
 * Supports 16-bit caches with head_dim 64 or 128 and E4M3 caches with
 * head_dim 128, block size 16 or 32 (others: PKV_ERR_UNSUPPORTED).  A sequence whose lengths are invalid
 * (ctx outside [0, max_blocks * T], n_s > ctx_s or n_s > max_query_len) or
 * whose table holds an entry outside [0, num_blocks) gets NaN rows; rows
 * outside [0, total_q) are never written.  Launched like the tensor-core
 * decode kernel (programmatic stream serialization); asynchronous on
 * `stream`. */
PKV_API pkv_status pkv_attention_prefill(void* out, const void* q, int32_t q_dtype,
                                         const void* k_cache, const void* v_cache,
                                         const int32_t* block_tables, int32_t max_blocks,
                                         const int32_t* context_lens, const int32_t* query_start,
                                         int32_t num_seqs, int32_t total_q, int32_t max_query_len,
                                         int32_t num_q_heads, const pkv_kv_desc* desc,
                                         float softmax_scale, float k_scale, float v_scale,
                                         void* stream);

/* Prefill kernel choice, process-wide: PKV_PREFILL_AUTO (tcgen05 UMMA with
 * TMEM accumulators for head_dim 128 and softmax_scale > 0 — 16-bit caches
 * directly, E4M3 caches widened exactly to f16 in shared memory — the
 * mma.sync kernel otherwise), PKV_PREFILL_MMA_SYNC (always the mma.sync
 * kernel) or PKV_PREFILL_TCGEN05 (the tcgen05 kernel; other shapes then
 * return PKV_ERR_UNSUPPORTED).  Both compute the same attention; their results
 * differ by rounding only.  PKV_ERR_INVALID_ARG for another value. */
#define PKV_PREFILL_AUTO 0
#define PKV_PREFILL_MMA_SYNC 1
#define PKV_PREFILL_TCGEN05 2
PKV_API pkv_status pkv_set_prefill_kernel(int32_t kind);

/* ---------------------------------------------------------- prefix caching
 * [C "The knobs"]: enable_prefix_caching hashes each filled block so that
 * unrelated requests share physical blocks; [C "Failure modes"]: sharing is
 * block-granular (block size 32: a shared 1,000-token prefix reuses at most
 * 992 tokens; a divergence inside a block loses the whole block); [B "Sharing,
 * the second dividend"]: when the tokens match, the blocks holding their KV
 * state are reused and that part of prefill is skipped.
 *
 * A full block whose token ids are known is published under the exact key
 * (entry of the previous block, its block_size token ids); a block whose
 * content is already published keeps the existing entry.  A published block
 * whose count reaches 0 is kept, least recently freed first (a sequence's
 * last block before its first), and taken again by a matching lookup or, once
 * the free stack is empty, evicted by an append (its entry dropped).  A
 * rolled-back append unpublishes the blocks it filled. */

/* Turn prefix caching on; only while the pool has no sequence. */
PKV_API pkv_status pkv_pool_enable_prefix_cache(pkv_pool* pool);

/* Create a sequence from a prompt of n_tokens token ids (host): it takes the
 * longest chain of published blocks matching the prompt's first full blocks,
 * at most (n_tokens - 1) / block_size of them (at least one prompt token is
 * left to compute), counts + 1.  *n_cached receives the tokens it holds (a
 * multiple of block_size); the caller appends the rest with
 * pkv_seq_append_tokens and writes only their K/V. */
PKV_API pkv_status pkv_seq_create_cached(pkv_pool* pool, int64_t seq_id, const int32_t* token_ids,
                                 int32_t n_tokens, int32_t* n_cached);

/* pkv_seq_append with the token ids of the new positions (host
 * int32[n_new]); blocks it fills are published.  Ids are kept only while
 * every earlier position's id is known (a plain pkv_seq_append stops them). */
PKV_API pkv_status pkv_seq_append_tokens(pkv_pool* pool, int64_t seq_id, const int32_t* token_ids,
                                 int32_t n_new, int64_t* slots_out, int32_t* cow_out,
                                 int32_t cow_cap, int32_t* n_cow_out);

/* Published blocks, published blocks at count 0, prompt tokens served from
 * the cache so far, and evictions. */
PKV_API pkv_status pkv_prefix_cache_stats(const pkv_pool* pool, int64_t* published_blocks,
                                  int64_t* reusable_blocks, int64_t* hit_tokens,
                                  int64_t* evictions);

/* The reusable (published, count 0) blocks in eviction order, first to go
 * first, into out[cap]; *n receives their number. */
PKV_API pkv_status pkv_reusable_blocks(const pkv_pool* pool, int32_t* out, int32_t cap, int32_t* n);

/* -------------------------------------------------------------- preemption
 * [C "The knobs"]: when the pool cannot satisfy a running sequence the engine
 * preempts it, drops its blocks and re-prefills it later (recompute);
 * [C "Effect"]: the scheduler preempts running sequences rather than failing
 * them, and a request can be preempted and restarted several times; [C
 * "Failure modes"]: the free-block watermark. */

/* One decode step with preemption: append one token to each sequence in
 * batch order, which is priority order.  When sequence i cannot get a block,
 * the lowest-priority sequence still running (the last one in the batch not
 * yet preempted, possibly i itself) is preempted (its blocks are freed as by
 * pkv_seq_free and it no longer exists) until i fits or is itself preempted.
 * slots_out[i] = -1 for preempted sequences (pkv_write skips negative slots);
 * preempted_out (host int64[n_seqs]) receives the preempted ids in order,
 * *n_preempted_out their number; cow_out must hold n_seqs pairs.  Never
 * fails for lack of blocks; UNKNOWN_SEQ / INVALID_ARG (a duplicate id) change
 * nothing.  A preempted sequence is re-admitted later with all its tokens
 * (recompute), e.g. by pkv_seq_admit or pkv_seq_create_cached. */
PKV_API pkv_status pkv_batch_append_preempt(pkv_pool* pool, const int64_t* seq_ids, int32_t n_seqs,
                                    int64_t* slots_out, int32_t* cow_out, int32_t cow_cap,
                                    int32_t* n_cow_out, int64_t* preempted_out,
                                    int32_t* n_preempted_out);

/* Admit a new sequence of n_tokens tokens (create + append) only if at least
 * watermark_blocks blocks stay free afterwards; else OUT_OF_BLOCKS and no
 * change.  slots_out: host int64[n_tokens]. */
PKV_API pkv_status pkv_seq_admit(pkv_pool* pool, int64_t seq_id, int32_t n_tokens,
                         int32_t watermark_blocks, int64_t* slots_out);

/* Message of the calling thread's last failure ("" if none). */
PKV_API const char* pkv_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
