// Internal interface between the decode-attention front end (attention.cu) and
// the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

// Everything a decode-attention kernel needs; passed by value as the kernel
// parameter.
struct DecodeArgs {
  void* out;                 // [B][Hq][D] q dtype
  const void* q;             // [B][Hq][D] q dtype
  const void* k_cache;       // [num_blocks][N_kv][T][D]
  const void* v_cache;
  const int32_t* tables;     // [B][max_blocks]
  const int32_t* ctx_lens;   // [B]
  float* ws_m;               // split-K partial maxima   [B][Hq][S] (log2 domain)
  float* ws_l;               // split-K partial sums      [B][Hq][S]
  float* ws_acc;             // split-K partial outputs   [B][Hq][S][D]
  int* counters;             // split-K arrival counters  [B][N_kv], zero between calls
  // fused slot write (tensor-core split kernel): when k_new is set, the CTA
  // holding position ctx - 1 of (sequence, KV head) first stores that
  // token's K/V ([B][N_kv][D], q dtype), E4M3-rounded with k_inv / v_inv
  const void* k_new;
  const void* v_new;
  float k_inv, v_inv;
  int32_t max_blocks, num_seqs, num_q_heads, num_kv_heads, group, num_blocks, block_size;
  int32_t partition;         // tokens per split (multiple of 64 and of T)
  int32_t max_splits;        // S
  float qk_scale;            // softmax_scale * k_scale * log2(e)
  float v_scale;             // 1, or the E4M3 V scale
  // E4M3 per-KV-head scales [4][N_kv] (K, V, K inverse, V inverse), or
  // NULL; when set they replace qk_scale's k_scale, v_scale, k_inv, v_inv
  const float* head_scales;
  float softmax_scale;
  // shared prefix (0: none): positions [0, prefix_tokens) of every sequence
  // are attended by the shared-prefix pass, the kernel launched just before
  // this one, whose prefix_splits partials sit in the last prefix_splits of
  // the max_splits slots; this kernel covers [prefix_tokens, ctx) and writes
  // partials, and the merge kernel after it combines them all
  int32_t prefix_tokens, prefix_splits;
  int* status;               // device error word (PKV_DEVICE_* bits, atomicOr)
  uint64_t wait_ns;          // give-up limit of a stage wait; 0 = give up at once
  int* done;                 // behind a shared-prefix pass: CTAs of this grid that have finished,
                             // then the tail queue's claim counter
  int32_t tail_queue;        // behind a shared-prefix pass: the tail queue form may run
};

// Prefill / shared-prefix pass arguments (attention_prefill.cu,
// attention_prefill_umma.cuh).
struct PrefillArgs {
  void* out;                  // [total_q][Hq][D]
  const void* q;              // [total_q][Hq][D]
  const int32_t* tables;      // [B][max_blocks]
  const int32_t* ctx_lens;    // [B], chunk included
  const int32_t* query_start; // [B + 1] row offsets of the chunks in q / out
  int32_t max_blocks, num_seqs, total_q, max_q_tiles, num_q_heads, num_kv_heads, group,
      num_blocks;
  float qk_scale;             // softmax_scale * log2(e) (* k_scale for E4M3)
  float v_scale;              // 1, or the E4M3 V scale
  const float* head_scales;   // E4M3 per-KV-head scales [4][N_kv], or NULL (replace the two above)
  float softmax_scale;
  int32_t ranked;             // tcgen05 kernel: grid (head, unit rank), units ranked longest first
  int* status;                // device error word
  // shared-prefix pass (grid (sequence group, key split, KV head)): the
  // query rows of a KV head are its (sequence, head) pairs; CTA x holds
  // sequences [x * sp_seqs, (x + 1) * sp_seqs), row s * group + j of its 256;
  // the keys are positions [k * sp_split, min(sp_tokens, (k + 1) * sp_split))
  // of table row 0; row (s, j)'s partial (max, sum, unnormalised output)
  // goes to split slot sp_slot0 + k of the decode workspace (ws_*, max_splits
  // slots), which the merge kernel after the decode kernel combines.
  int32_t sp_rows, sp_tokens, sp_split, sp_slot0, max_splits, sp_seqs;
  float* ws_m;
  float* ws_l;
  float* ws_acc;
};

// Device error word of the current device (looked up once per device);
// nullptr with *st set when a CUDA call fails.  Defined in status.cu.
int* device_status_word(pkv_status* st);

// Give-up limit of the decode kernels' stage waits (pkv_set_stage_wait_limit).
uint64_t stage_wait_limit_ns();

// Launch the shared-prefix pass (tcgen05, head_dim 128) for one (cache, q)
// dtype pair; grid (row pairs, key splits, KV heads).  Defined in
// attention_shared_prefix.cu.
template <typename KV, typename Q>
pkv_status launch_shared_prefix_pass(const PrefillArgs& a, int block_size, int key_splits,
                                     const CUtensorMap& kmap, const CUtensorMap& vmap,
                                     cudaStream_t st);

// The merge kernel after the decode kernel on the shared-prefix path
// (head_dim 128): every (sequence, query head)'s partials into out.  Defined
// in attention_shared_prefix.cu.
template <typename Q>
pkv_status launch_prefix_merge(const DecodeArgs& a, cudaStream_t st);

// Bytes at the start of a decode workspace that hold the split-K arrival
// counters (they must be zero when a call starts; every call leaves them
// zero).  0 when the sizes need no split.
size_t attention_counter_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t max_blocks,
                               const pkv_kv_desc* desc, int32_t partition_tokens);

// TMA tensor map of one pool tensor viewed as bytes [num_blocks * N_kv * T
// rows][D * P_kv], read with the 128-byte swizzle in boxes of T rows: whole
// rows (a 3-D (128 bytes, slab, row) view for 256-byte rows; the decode
// kernels) or one 128-byte slab per box (whole_rows false; prefill).
// Defined in attention.cu.
pkv_status pool_map(CUtensorMap* map, const void* base, const pkv_kv_desc* d, bool whole_rows = true);

// Write the step's K/V row of each sequence at logical position ctx - 1
// through its block table (a small kernel; defined in write_copy.cu).
pkv_status launch_write_last(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                             int32_t src_dtype, float k_inv_scale, float v_inv_scale,
                             const int32_t* tables, int32_t max_blocks, const int32_t* ctx_lens,
                             int32_t num_seqs, const pkv_kv_desc* desc, cudaStream_t st);

// Launch the CUDA-core decode kernel for one (cache dtype, q dtype) pair;
// returns PKV_ERR_UNSUPPORTED for a shape it was not compiled for.
template <typename KV, typename Q>
pkv_status launch_decode_simt(const DecodeArgs& a, int head_dim, int group_padded,
                              cudaStream_t stream);

}  // namespace pkv
