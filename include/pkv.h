/*
 * pkv.h — C ABI of libpkv.so: paged KV-cache decode path on one GPU.
 *
 * Three operations, each a hand-written CUDA kernel for sm_103a:
 *   pkv_kv_write                write new keys / values into cache slots
 *   pkv_paged_decode_attention  one-query-token attention over paged K/V
 *   pkv_copy_blocks             whole-block copies for copy-on-write
 *
 * Storage.  The key cache and the value cache are two separate pools of
 * fixed-size physical blocks, each laid out row-major as
 *     [num_blocks][num_kv_heads][block_size][head_dim]
 * so one (block, KV head) tile of block_size x head_dim scalars is contiguous
 * (at block size 16 and head size 128 that is 2048 elements per head per
 * block).  Scalars are IEEE binary16 or bfloat16.  A sequence reaches its
 * tokens through a block table: logical token t of sequence s lives in
 * physical block block_tables[s][t / block_size], slot t % block_size.
 * (vLLM PagedAttention & continuous batching, "PagedAttention: fixed blocks,
 * non-contiguous physical memory" and "The kernel page".)
 *
 * Conventions common to every call.
 *  - Every pointer argument except those documented as host values is a
 *    DEVICE pointer.  The caller owns every buffer; the library allocates
 *    nothing and keeps no state between calls.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  All work is enqueued asynchronously on it.
 *  - Arguments are validated on the host before anything is enqueued; on a
 *    validation failure the call returns PKV_ERR_INVALID_ARG or
 *    PKV_ERR_UNSUPPORTED and enqueues nothing.  A failed launch returns
 *    PKV_ERR_CUDA.
 *  - Errors that depend on device data (a block id outside the pool, a slot
 *    outside the pool, a sequence longer than its block table, a bad block
 *    pair) never trap: the kernel skips the offending access and ORs one of
 *    the PKV_DEVERR_* bits into *err_flag when err_flag is not NULL.  The
 *    caller reads the flag after synchronising the stream.
 *  - Calls on the same stream execute in order; calls that touch the same
 *    cache from different streams must be ordered by the caller.
 *  - pkv_kv_write, pkv_kv_write_layers, pkv_paged_decode_attention (and its
 *    fixed-scratch form) and pkv_paged_prefill_attention work on 16-bit
 *    pools: c.dtype PKV_FP8_E4M3 returns PKV_ERR_INVALID_ARG there (the
 *    *_fp8 calls serve 8-bit pools).
 */
#ifndef PKV_H_
#define PKV_H_

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
    PKV_ERR_INVALID_ARG = 1,          /* null pointer, negative size, inconsistent shapes */
    PKV_ERR_UNSUPPORTED = 2,          /* a valid shape this build does not implement */
    PKV_ERR_WORKSPACE_TOO_SMALL = 3,  /* workspace smaller than pkv_decode_workspace_bytes */
    PKV_ERR_CUDA = 4                  /* a CUDA launch or driver call failed */
} pkv_status;

/* Scalar types.  PKV_FP8_E4M3 is a storage type of pools only (see
 * "8-bit pools" below); queries, new keys / values and outputs are
 * PKV_FP16 or PKV_BF16. */
typedef enum { PKV_FP16 = 0, PKV_BF16 = 1, PKV_FP8_E4M3 = 2 } pkv_dtype;

/* Bits ORed into *err_flag by the kernels (device-side data errors). */
#define PKV_DEVERR_BAD_SLOT     1  /* slot_mapping[t] >= num_blocks * block_size */
#define PKV_DEVERR_BAD_BLOCK_ID 2  /* a block-table entry outside [0, num_blocks) */
#define PKV_DEVERR_BAD_SEQ_LEN  4  /* seq_len < 0, > max_seq_len or > table capacity */
#define PKV_DEVERR_BAD_PAIR     8  /* a copy pair with src or dst outside [0, num_blocks) */
#define PKV_DEVERR_TIMEOUT      16 /* a bounded on-chip wait gave up (never expected) */

/* Geometry of both caches (host value). */
typedef struct {
    int32_t num_blocks;    /* physical blocks in each pool, > 0 */
    int32_t num_kv_heads;  /* KV heads, > 0 */
    int32_t block_size;    /* token slots per block */
    int32_t head_dim;      /* scalars per head */
    pkv_dtype dtype;       /* storage type of the pools; for the 16-bit calls also the
                              type of q, k, v and out (PKV_FP16 or PKV_BF16 there) */
} pkv_cache_desc;

/*
 * Write the keys and values of new tokens into their cache slots.
 *
 * Decode writes the next token of a sequence into the spare slot of its last
 * block (vLLM PagedAttention & continuous batching, "PagedAttention", the
 * seven-token example); prefill writes every prompt token the same way.
 * The slot of token t is slot_mapping[t] = physical_block * block_size +
 * offset, so for every KV head h:
 *     k_cache[slot / B][h][slot % B][:] = k[t][h][:]   (and v likewise).
 *
 *   k, v          [num_tokens][num_kv_heads][head_dim], dtype of c, contiguous.
 *   slot_mapping  [num_tokens] int64.  A negative slot marks a padding token
 *                 and is skipped silently; a slot >= num_blocks * block_size
 *                 is skipped and sets PKV_DEVERR_BAD_SLOT.
 *   k_cache, v_cache  the pools, updated in place.
 *   Slots must be distinct among non-negative entries (two tokens written to
 *   one slot race).  head_dim must be a multiple of 8 and every row 16-byte
 *   aligned.  num_tokens == 0 is a no-op.
 */
PKV_API pkv_status pkv_kv_write(const void* k, const void* v, const int64_t* slot_mapping,
                        int32_t num_tokens, void* k_cache, void* v_cache, pkv_cache_desc c,
                        int32_t* err_flag, void* stream);

/*
 * Partition size (tokens) that pkv_paged_decode_attention uses for the
 * given request: `partition_size` itself when positive (it must then be a
 * multiple of block_size), else the automatic choice (512 tokens when
 * max_seq_len > 512, otherwise a single partition).  Returns a value
 * >= max_seq_len when every sequence is handled in one pass, or -1 when the
 * arguments are invalid.
 */
PKV_API int32_t pkv_decode_partition_size(int32_t max_seq_len, int32_t block_size,
                                  int32_t partition_size);

/*
 * Workspace bytes pkv_paged_decode_attention needs for these sizes (0 when
 * every sequence fits one partition).  The workspace holds per-partition
 * fp32 statistics: an accumulator row of head_dim floats plus a running
 * maximum and a running sum for each (sequence, query head, partition).
 */
PKV_API size_t pkv_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                                  int32_t max_seq_len, int32_t block_size,
                                  int32_t partition_size);

/*
 * Exact attention of one query token per sequence over its paged K/V.
 *
 * For sequence s, query head i and its KV head h = i / (num_q_heads /
 * num_kv_heads) (contiguous grouped-query groups; MHA when the ratio is 1,
 * MQA when num_kv_heads is 1):
 *     out[s][i] = sum_t softmax_t(scale * q[s][i] . K_t) V_t,  t < seq_lens[s],
 * with K_t, V_t read through block_tables[s].  PagedAttention leaves this
 * formula unchanged and only changes where K and V live (vLLM PagedAttention
 * & continuous batching, "PagedAttention" and "The kernel page").  The
 * softmax is computed block by block with the running maximum / running sum
 * of Eq. (4) of "Serving Language Models Within a Memory Budget"; sequences
 * longer than one partition are split into partitions whose (max, sum,
 * weighted-sum) statistics are merged by the same rule.  Products of
 * fp16/bf16 inputs accumulate in fp32; the output is rounded to the storage
 * dtype (round to nearest even).  An empty sequence (seq_len 0) yields zeros.
 *
 *   q             [num_seqs][num_q_heads][head_dim], contiguous.
 *   k_cache, v_cache  pools (see top); 16-byte aligned.
 *   block_tables  [num_seqs][max_blocks_per_seq] int32; only the first
 *                 ceil(seq_len / block_size) entries of a row are read.
 *   seq_lens      [num_seqs] int32 attended lengths.
 *   max_seq_len   HOST value, an upper bound of every seq_lens[s]; it sizes
 *                 the launch without a device-to-host read.  Must be
 *                 <= max_blocks_per_seq * block_size.
 *   scale         softmax scale, typically 1/sqrt(head_dim).
 *   partition_size  0 = automatic; > 0 tokens per partition (a multiple of
 *                 block_size); >= max_seq_len = single pass.
 *   workspace     device scratch of workspace_bytes >=
 *                 pkv_decode_workspace_bytes(...) (may be NULL when that is 0).
 *                 It holds partial softmax statistics; its contents need no
 *                 initialisation and are overwritten.  Calls that share a
 *                 workspace must not run concurrently.
 *   out           [num_seqs][num_q_heads][head_dim], dtype of c.
 * Supported: head_dim 128; num_q_heads / num_kv_heads <= 64; num_seqs <=
 * 65535; block_size 8, 16, 32, 64 or 128 in automatic mode when the group
 * is at most 16 query heads and num_seqs <= 4096 (the streaming kernel),
 * otherwise block_size 16 or 32 (the partition kernel).  Other valid shapes
 * return PKV_ERR_UNSUPPORTED.
 */
PKV_API pkv_status pkv_paged_decode_attention(const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                                      const int32_t* seq_lens, int32_t max_seq_len,
                                      int32_t num_seqs, int32_t num_q_heads, pkv_cache_desc c,
                                      float scale, int32_t partition_size, void* workspace,
                                      size_t workspace_bytes, void* out, int32_t* err_flag,
                                      void* stream);

/*
 * Paged prefill attention: many query tokens per sequence, causal.
 *
 * The prompt phase runs the known prompt as matrix-matrix work over the
 * cache (vLLM PagedAttention & continuous batching, "Prompt phase, decode
 * phase"); the prompt's keys and values are first written with
 * pkv_kv_write.  Sequence s holds n = seq_lens[s] tokens in its blocks; its
 * last q_len_s = cu_seqlens_q[s+1] - cu_seqlens_q[s] tokens are the queries
 * of this call, query i sitting at position n - q_len_s + i (the positions
 * before it are an earlier chunk of the prompt or a shared prefix already
 * cached).  Query i of query head h attends to positions 0 .. n - q_len_s + i
 * of KV head h / (num_q_heads / num_kv_heads):
 *     out[cu_q[s] + i][h] = softmax_t(scale * q . K_t) V_t.
 * Products of fp16/bf16 inputs accumulate in fp32; the output is rounded to
 * the storage dtype.
 *
 *   q             [total query tokens][num_q_heads][head_dim], contiguous,
 *                 16-byte aligned (rows move as 16-byte vectors); sequence
 *                 s's queries are rows cu_seqlens_q[s] .. cu_seqlens_q[s+1] - 1.
 *   cu_seqlens_q  DEVICE [num_seqs + 1] int32, non-decreasing, from 0.
 *   max_q_len     HOST value >= every q_len_s (sizes the launch).
 *   k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens,
 *   max_seq_len, scale: as pkv_paged_decode_attention.
 *   out           [total query tokens][num_q_heads][head_dim], 16-byte aligned.
 * A q or out that is not 16-byte aligned returns PKV_ERR_INVALID_ARG.
 * A sequence whose q_len is negative, above max_q_len or above its
 * seq_len, or whose seq_len exceeds max_seq_len, is skipped and sets
 * PKV_DEVERR_BAD_SEQ_LEN.  Supported: head_dim 128, block_size 8, 16, 32,
 * 64 or 128, num_q_heads / num_kv_heads <= 64, num_seqs <= 65535.
 */
PKV_API pkv_status pkv_paged_prefill_attention(const void* q, const int32_t* cu_seqlens_q,
                                               int32_t max_q_len, const void* k_cache,
                                               const void* v_cache, const int32_t* block_tables,
                                               int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                               int32_t max_seq_len, int32_t num_seqs,
                                               int32_t num_q_heads, pkv_cache_desc c, float scale,
                                               void* out, int32_t* err_flag, void* stream);

/* Size of the fixed device scratch of pkv_paged_decode_attention_fixed_scratch. */
#define PKV_FIXED_SCRATCH_BYTES ((size_t)16 << 20)

/*
 * pkv_paged_decode_attention for callers that cannot allocate device memory.
 * The paper has no counterpart to this entry point; it exists for callers
 * whose host application owns every GPU allocation (a server that hands its
 * plugins only pre-registered buffers, or a runtime with its own pool and a
 * fixed budget), where a cudaMalloc of their own could fail, fragment the
 * host's pool or synchronise the device at the wrong time.
 *
 * Same arguments, results and errors as pkv_paged_decode_attention, minus
 * the workspace: split-mode scratch comes from a fixed array of
 * PKV_FIXED_SCRATCH_BYTES compiled into the library, present on every GPU
 * that loads the library until the process exits.  The call allocates
 * nothing.  A request whose scratch need (pkv_decode_workspace_bytes)
 * exceeds PKV_FIXED_SCRATCH_BYTES returns PKV_ERR_WORKSPACE_TOO_SMALL and
 * enqueues nothing.  The array's device address is looked up once per
 * device, on that device's first call needing scratch, with the caller's
 * current device (which must own `stream` and the buffers); make that first
 * call before any stream capture.  All calls share the one array: calls whose
 * kernels can overlap on the GPU (other streams, other host threads) race on
 * it, so order them on one stream.  Its contents carry over between calls
 * and need no clearing.
 */
PKV_API pkv_status pkv_paged_decode_attention_fixed_scratch(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t max_seq_len, int32_t num_seqs,
    int32_t num_q_heads, pkv_cache_desc c, float scale, int32_t partition_size, void* out,
    int32_t* err_flag, void* stream);

/*
 * Copy whole physical blocks, for copy-on-write of a shared block.
 *
 * When a sequence must write into a block whose reference count is above
 * one, the block manager allocates a fresh block and the old block's
 * contents are copied into it (vLLM PagedAttention & continuous batching,
 * "Sharing with reference counts and copy-on-write"; the last partial block
 * of a shared prefix is copy-on-write).  For each pair p:
 *     k_cache[dst_p] = k_cache[src_p],  v_cache[dst_p] = v_cache[src_p]
 * over every KV head and every slot, filled or not, bit for bit.
 *
 *   c              any storage dtype, PKV_FP8_E4M3 included (blocks are
 *                  copied as bytes).
 *   src_dst_pairs  DEVICE [num_pairs][2] int64 (src, dst).  Destinations
 *                  must be distinct and no destination may be the source of
 *                  another pair (pairs run concurrently).  A pair with an
 *                  index outside [0, num_blocks) is skipped and sets
 *                  PKV_DEVERR_BAD_PAIR.  num_pairs == 0 is a no-op.
 */
PKV_API pkv_status pkv_copy_blocks(void* k_cache, void* v_cache, pkv_cache_desc c,
                           const int64_t* src_dst_pairs, int32_t num_pairs, int32_t* err_flag,
                           void* stream);

/*
 * Copy whole blocks from one pair of pools to another: the swap path of
 * preemption.  When physical blocks run out, all blocks of a preempted
 * sequence are copied to CPU memory managed by a second block allocator and
 * copied back when it resumes (vLLM PagedAttention & continuous batching,
 * "Preemption when blocks run out", Swap).  For each pair p:
 *     dst_k[dst_p] = src_k[src_p],  dst_v[dst_p] = src_v[src_p]
 * over every KV head and slot, bit for bit.
 *
 *   src_k, src_v  source pools of src_num_blocks blocks; dst_k, dst_v
 *                 destination pools of dst_num_blocks blocks.  Each pool is
 *                 device memory or page-locked host memory (cudaHostAlloc,
 *                 cudaHostRegister, torch pin_memory): the kernel reads and
 *                 writes host pools directly over the CPU-GPU link, one launch
 *                 for all pairs.  Pageable host memory is rejected with
 *                 PKV_ERR_INVALID_ARG.  The two pairs of pools must not overlap.
 *   c             shared geometry (num_kv_heads, block_size, head_dim, dtype,
 *                 PKV_FP8_E4M3 included); its num_blocks is not used.
 *   src_dst_pairs DEVICE [num_pairs][2] int64 (src block, dst block).
 *                 Destinations must be distinct.  A pair outside either pool
 *                 is skipped and sets PKV_DEVERR_BAD_PAIR.
 */
PKV_API pkv_status pkv_swap_blocks(const void* src_k, const void* src_v, int32_t src_num_blocks,
                                   void* dst_k, void* dst_v, int32_t dst_num_blocks,
                                   pkv_cache_desc c, const int64_t* src_dst_pairs,
                                   int32_t num_pairs, int32_t* err_flag, void* stream);

/* Most layers the *_layers calls take in one launch. */
#define PKV_MAX_LAYERS 128

/*
 * pkv_kv_write for num_layers layers in one launch: layer l writes k[l],
 * v[l] ([num_tokens][num_kv_heads][head_dim] each) into k_caches[l],
 * v_caches[l] at the same slot mapping (every layer of a model shares the
 * block tables).  k, v, k_caches, v_caches are HOST arrays of num_layers
 * device pointers, read during the call.  1 <= num_layers <= PKV_MAX_LAYERS.
 * Errors and conventions as pkv_kv_write.
 */
PKV_API pkv_status pkv_kv_write_layers(const void* const* k, const void* const* v,
                                       const int64_t* slot_mapping, int32_t num_tokens,
                                       void* const* k_caches, void* const* v_caches,
                                       int32_t num_layers, pkv_cache_desc c, int32_t* err_flag,
                                       void* stream);

/*
 * pkv_copy_blocks for num_layers layers in one launch: the same (src, dst)
 * pairs are applied to every layer's k_caches[l], v_caches[l] (HOST arrays
 * of num_layers device pointers).  1 <= num_layers <= PKV_MAX_LAYERS.
 * Errors and conventions as pkv_copy_blocks (any storage dtype).
 */
PKV_API pkv_status pkv_copy_blocks_layers(void* const* k_caches, void* const* v_caches,
                                          int32_t num_layers, pkv_cache_desc c,
                                          const int64_t* src_dst_pairs, int32_t num_pairs,
                                          int32_t* err_flag, void* stream);

/*
 * 8-bit pools (c.dtype == PKV_FP8_E4M3).
 *
 * The pages note that the key-value cache need not share the model's
 * precision and that changing it changes the numerics ("Serving Language
 * Models Within a Memory Budget", section 4, "Allocation efficiency is not
 * the entire memory budget").  This library's 8-bit format: each stored
 * scalar is one byte in the OCP FP8 E4M3 encoding (1 sign bit, 4 exponent
 * bits with bias 7, 3 mantissa bits, no infinities, S.1111.111 = NaN,
 * largest finite magnitude 448), and each pool has one scale factor, k_scale
 * for the key pool and v_scale for the value pool.  A scalar x is stored as
 * E4M3(x / scale), the quotient taken in binary32 and rounded to the nearest
 * code (ties to even), magnitudes above 448 saturating to 448; the code is
 * read back as code * scale.  Layout as the 16-bit pools with one-byte
 * scalars: [num_blocks][num_kv_heads][block_size][head_dim] bytes.  The
 * block copies (pkv_copy_blocks, pkv_swap_blocks, pkv_copy_blocks_layers)
 * take such pools as they are.
 */

/*
 * pkv_kv_write into 8-bit pools: the key row of token t, KV head h is stored
 * at slot slot_mapping[t] as E4M3(k[t][h][:] / k_scale), and values with
 * v_scale.
 *
 *   k, v          [num_tokens][num_kv_heads][head_dim] of kv_dtype (PKV_FP16
 *                 or PKV_BF16), contiguous, 16-byte aligned.
 *   k_cache, v_cache  pools of E4M3 codes; c.dtype must be PKV_FP8_E4M3.
 *   k_scale, v_scale  finite and > 0.
 * Slots, padding, errors and head_dim rules as pkv_kv_write (head_dim a
 * multiple of 16 here).  Non-finite inputs: infinities saturate to +-448,
 * NaN is stored as 0x7f.
 */
PKV_API pkv_status pkv_kv_write_fp8(const void* k, const void* v, pkv_dtype kv_dtype,
                                    const int64_t* slot_mapping, int32_t num_tokens,
                                    void* k_cache, void* v_cache, pkv_cache_desc c, float k_scale,
                                    float v_scale, int32_t* err_flag, void* stream);

/*
 * pkv_paged_decode_attention over 8-bit pools:
 *     out[s][i] = sum_t softmax_t(scale * q[s][i] . (k_scale * Kc_t)) (v_scale * Vc_t)
 * where Kc_t, Vc_t are the decoded E4M3 codes of token t.  The codes are
 * widened exactly to binary16 and multiplied with binary16 queries; a
 * bfloat16 query row is first multiplied by a power of two that brings its
 * largest magnitude into [2^14, 2^15) and rounded to binary16, the power of
 * two being divided out of its scores.  Products accumulate in fp32; the
 * output is rounded to q_dtype.
 *
 *   q, out        [num_seqs][num_q_heads][head_dim] of q_dtype (PKV_FP16 or
 *                 PKV_BF16).
 *   k_cache, v_cache  E4M3 pools (c.dtype == PKV_FP8_E4M3), 16-byte aligned.
 *   k_scale, v_scale  the pools' scales, finite and > 0.
 *   workspace     >= pkv_decode_workspace_bytes(num_seqs, num_q_heads,
 *                 head_dim, max_seq_len, block_size, 0) bytes.
 * Other arguments, errors and the empty-sequence rule as
 * pkv_paged_decode_attention in automatic mode.  Supported: head_dim 128,
 * block_size 8, 16, 32, 64 or 128, num_q_heads / num_kv_heads <= 16,
 * num_seqs <= 4096 (the streaming kernel); other valid shapes return
 * PKV_ERR_UNSUPPORTED.
 */
PKV_API pkv_status pkv_paged_decode_attention_fp8(
    const void* q, pkv_dtype q_dtype, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
    int32_t max_seq_len, int32_t num_seqs, int32_t num_q_heads, pkv_cache_desc c, float scale,
    float k_scale, float v_scale, void* workspace, size_t workspace_bytes, void* out,
    int32_t* err_flag, void* stream);

/* Static, NUL-terminated name of a status code. */
PKV_API const char* pkv_status_string(pkv_status status);

/* ABI version of this header (major * 100 + minor). */
PKV_API int32_t pkv_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
