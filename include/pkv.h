/*
 * pkv.h -- C ABI of libpkv: paged-KV decode attention for one GB300 (sm_103a).
 *
 * What the library computes
 * -------------------------
 * A paged KV cache keeps every sequence's keys and values in a pool of
 * fixed-size physical blocks; a per-sequence block table maps logical block i
 * (tokens [16i, 16i+16)) to a physical block, and the attention kernel gathers
 * K/V from those non-contiguous blocks itself, with no compaction copy
 * (Continuous-Batching-LLM-Inference-Engine README, feature list "Paged
 * KV-cache" and "PagedAttention kernel"). The model's forward writes new K/V
 * into the cache through slot mappings and reads them back in the paged decode
 * attention kernel (mini-inference-engine, Connections "Llama forward -> Paged
 * KV cache: writes and reads"; low-latency-distributed-llm-serving-
 * infrastructure, Connections "Paged attention -> KV cache manager: maps cache
 * slots"). The cache may be stored as INT8 (paged-inference-engine overview,
 * "paged INT8 KV storage").
 *
 * Layouts (all row-major, contiguous):
 *   k_cache, v_cache  [num_blocks, num_kv_heads, block_size, head_dim]
 *                     one (block, kv_head) tile is one contiguous run of
 *                     block_size*head_dim elements
 *   k_scales, v_scales [num_blocks, num_kv_heads] fp32 (INT8 caches only)
 *   block_tables      int32 [batch, max_blocks_per_seq]; entries past a
 *                     sequence's ceil(len/16) blocks are not read
 *   context_lens      int32 [batch], including the token appended this step
 *   q, out            [batch, num_q_heads, head_dim], q's dtype
 *   k_new, v_new      [num_tokens, num_kv_heads, head_dim]
 *   slot_mapping      int64 [num_tokens], slot = block*block_size + row,
 *                     negative = skip
 * Query head h reads KV head h / (num_q_heads / num_kv_heads).
 *
 * Ownership and synchronisation: every pointer argument is caller-owned
 * DEVICE memory, except the pkv_cache_desc pointer (host). The library
 * allocates nothing. Between calls it keeps only lookups, each made once:
 * two driver entry points (the tensor-map encoder of pkv_multiquery_attn and
 * the current-context query of pkv_decode_attn_noalloc) and, per CUDA
 * context, the address of pkv_decode_attn_noalloc's built-in scratch array. Every call only
 * enqueues kernels on `stream` and returns; inputs must stay valid until the
 * stream has executed them.
 *
 * Errors: arguments are checked on the host before anything is launched; a
 * bad argument returns PKV_ERR_* and launches nothing. Conditions only the GPU
 * can see (a block-table entry or slot outside the pool, a context length
 * outside the table, a bounded in-kernel wait that ran out) are OR-ed as
 * PKV_DEV_* bits into *dev_status when dev_status is non-NULL; the kernel
 * then skips the offending work instead of touching memory outside the
 * buffers. The library never clears *dev_status.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as the CUDA runtime's cudaStream_t; NULL = legacy default stream. */
typedef struct CUstream_st *cudaStream_t;

typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,   /* NULL / misaligned pointer, bad size or shape */
    PKV_ERR_UNSUPPORTED = 2,   /* valid but not built: head_dim, group, dtype  */
    PKV_ERR_WORKSPACE = 3,     /* workspace NULL or smaller than required      */
    PKV_ERR_CUDA = 4           /* a CUDA runtime call or launch failed         */
} pkv_status;

/* Bits OR-ed into *dev_status by the kernels. */
#define PKV_DEV_BAD_BLOCK  1u  /* block-table entry outside [0, num_blocks)    */
#define PKV_DEV_BAD_LENGTH 2u  /* context_len < 0 or > max_blocks_per_seq*16   */
#define PKV_DEV_BAD_SLOT   4u  /* slot >= num_blocks*block_size                */
#define PKV_DEV_TIMEOUT    8u  /* a bounded wait on an in-kernel copy ran out  */
#define PKV_DEV_BAD_INDEX 16u  /* pkv_merge_states: a row's range of states
                                  lies outside [0, num_states]              */

typedef enum { PKV_F16 = 0, PKV_BF16 = 1, PKV_I8 = 2 } pkv_dtype;

/* The physical KV block pool. block_size must be 16, head_dim 64 or 128. */
typedef struct {
    int32_t num_blocks;
    int32_t block_size;
    int32_t num_kv_heads;
    int32_t head_dim;
    pkv_dtype kv_dtype;       /* PKV_F16, PKV_BF16 or PKV_I8 */
} pkv_cache_desc;

/* Human-readable name of a status code (static string, never NULL). */
const char *pkv_status_string(pkv_status s);

/* ------------------------------------------------------------------------
 * KV append (cache write)
 *
 * Writes k_new[n], v_new[n] to slot slot_mapping[n] of k_cache / v_cache for
 * every n with slot >= 0 (the cache write that the forward pass performs each
 * step; see the file comment). Duplicate non-negative slots in one call are a
 * caller error.
 *
 * fp16 / bf16 caches: src_dtype must equal kv_dtype; the rows are stored bit
 * for bit. k_scales, v_scales, workspace may be NULL.
 *
 * INT8 caches (PKV_I8): src_dtype is PKV_F16 or PKV_BF16. Codes are symmetric
 * in [-127, 127] with one fp32 scale per (block, kv_head), K and V separately,
 * scale = absmax/127 and round-to-nearest-even. Per (block, kv_head) tile
 * touched by the call: a = max|x| over the call's new values in the tile,
 * s_c = a/127 (fp32, IEEE division); with s_o the stored scale (0 = never
 * written): s = s_c if s_o == 0; s = s_o if s_c <= s_o; otherwise s = s_c and
 * every stored code q of the tile becomes rne((float)q * s_o / s) (fp32, left
 * to right). New codes are clamp(rne(x / s), -127, 127), or 0 when s == 0.
 * k_scales / v_scales must start at 0 for never-written blocks. The call needs
 * a workspace of pkv_append_workspace_size(cache) bytes (80 bytes per
 * (block, kv_head) tile; 16-byte aligned), zero-filled before its first use:
 * each call leaves it zero-filled again, so one workspace serves every later
 * call on the same cache (calls that overlap on the GPU must not share it).
 * Inputs must be finite.
 *
 * Alignment: k_new, v_new, k_cache, v_cache 16-byte aligned.
 * ------------------------------------------------------------------------ */
size_t pkv_append_workspace_size(const pkv_cache_desc *cache);

pkv_status pkv_append(const void *k_new, const void *v_new, pkv_dtype src_dtype,
                      int32_t num_tokens, const int64_t *slot_mapping,
                      void *k_cache, void *v_cache, float *k_scales, float *v_scales,
                      const pkv_cache_desc *cache, void *workspace, size_t workspace_bytes,
                      uint32_t *dev_status, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Decode attention (one query token per sequence)
 *
 * out[b, h] = sum_p softmax_p(softmax_scale * <q[b,h], k_p>) * v_p over the
 * context_lens[b] tokens of sequence b, token p read from physical block
 * block_tables[b, p/16], row p%16 (the paged decode attention kernel of the
 * pages; see the file comment). INT8 values dequantise as code*scale[block,
 * kv_head]. context_lens[b] == 0 gives a zero row. Accumulation is fp32; out
 * is rounded to q's dtype (nearest-even).
 *
 * Work split: the (sequence, kv_head, block) units of the whole batch are cut
 * into num_parts equal contiguous ranges, one per worker warp (0 = the
 * device default of pkv_decode_default_parts). A sequence whose blocks fall in one
 * range is finished by that worker; the others leave fp32 partial states in
 * the workspace that the combine step merges:
 *   out = sum_i exp(m_i - M) o_i / sum_i exp(m_i - M) l_i,  M = max_i m_i.
 * num_parts, batch, num_q_heads and the cache must be the same in
 * pkv_decode_workspace_size, pkv_decode_split and pkv_decode_combine.
 *
 * Supported: block_size 16, head_dim 64 or 128, num_q_heads/num_kv_heads in
 * {1, 2, 4, 8}, 1 <= batch <= 8192; q_dtype == kv_dtype for fp16/bf16 caches,
 * q_dtype PKV_F16 or PKV_BF16 for INT8 caches. q, out, caches 16-byte aligned;
 * workspace 256-byte aligned.
 * ------------------------------------------------------------------------ */

/* The default num_parts on `device`: the split kernel's resident worker
 * warps, capped at 2 CTAs (8 warps) per SM for fp16/bf16 caches at head_dim
 * 128, where fewer, longer workers read the cache faster; INT8 caches run
 * CTAs of 6 warps, two per SM at batch 256 (fewer CTAs fit for much larger
 * batches). 0 if the configuration is unsupported. */
int32_t pkv_decode_default_parts(int32_t device, int32_t batch, int32_t num_q_heads,
                                 const pkv_cache_desc *cache);

/* Workspace bytes for these sizes (num_parts 0 = the current device's
 * default). Returns 0 for an unsupported configuration. */
size_t pkv_decode_workspace_size(int32_t batch, int32_t num_q_heads,
                                 const pkv_cache_desc *cache, int32_t num_parts);

/* Split phase and combine phase back to back on `stream`. */
pkv_status pkv_decode_attn(const void *q, pkv_dtype q_dtype,
                           const void *k_cache, const void *v_cache,
                           const float *k_scales, const float *v_scales,
                           const pkv_cache_desc *cache,
                           const int32_t *block_tables, int32_t max_blocks_per_seq,
                           const int32_t *context_lens, int32_t batch, int32_t num_q_heads,
                           float softmax_scale, void *out,
                           void *workspace, size_t workspace_bytes, int32_t num_parts,
                           uint32_t *dev_status, cudaStream_t stream);

/* Split phase only: each worker streams its range of KV blocks (online
 * softmax in fp32), writes finished sequences to out and partial states
 * (m, l, unnormalised o) to the workspace. Same arguments as pkv_decode_attn. */
pkv_status pkv_decode_split(const void *q, pkv_dtype q_dtype,
                            const void *k_cache, const void *v_cache,
                            const float *k_scales, const float *v_scales,
                            const pkv_cache_desc *cache,
                            const int32_t *block_tables, int32_t max_blocks_per_seq,
                            const int32_t *context_lens, int32_t batch, int32_t num_q_heads,
                            float softmax_scale, void *out,
                            void *workspace, size_t workspace_bytes, int32_t num_parts,
                            uint32_t *dev_status, cudaStream_t stream);

/* The decode step's cache write and attention in one call: writes k_new[b],
 * v_new[b] ([batch, num_kv_heads, head_dim]; the cache dtype for fp16 / bf16
 * caches, q_dtype for INT8 caches) at position context_lens[b] - 1 of each
 * sequence, i.e. physical block block_tables[b, (L-1)/16], row (L-1)%16
 * (nothing for L == 0), then computes pkv_decode_attn over the caches
 * including that token. The same result, bit for bit in the cache (codes
 * and scales for INT8) and in out, as pkv_append with those slots followed
 * by pkv_decode_attn, in fewer launches: for fp16 / bf16 caches the split
 * kernel copies each new row into shared memory in place of the tile's row
 * (from k_new / v_new, beside the cache rows before it) and stores it into
 * the cache from there (split [+ combine]); for INT8 caches one append
 * kernel settles each touched tile's scales, requantises it if a scale
 * grows and encodes the row, one warp per (sequence, kv head), without
 * pkv_append's gather pass (append + split [+ combine]; k_scales, v_scales
 * as for pkv_append, NULL for 16-bit caches). The block receiving a
 * sequence's new token must not be shared with another sequence
 * (copy-on-write). Same workspace as pkv_decode_attn; k_new, v_new 16-byte
 * aligned. run_combine = 0 runs only the split phase (as pkv_decode_split;
 * pkv_decode_combine must follow), 1 both. */
pkv_status pkv_decode_step(const void *q, pkv_dtype q_dtype, const void *k_new,
                           const void *v_new, void *k_cache, void *v_cache,
                           float *k_scales, float *v_scales,
                           const pkv_cache_desc *cache, const int32_t *block_tables,
                           int32_t max_blocks_per_seq, const int32_t *context_lens,
                           int32_t batch, int32_t num_q_heads, float softmax_scale, void *out,
                           void *workspace, size_t workspace_bytes, int32_t num_parts,
                           int32_t run_combine, uint32_t *dev_status, cudaStream_t stream);

/* Combine phase (the split-K reduce): merges the partial states a preceding
 * pkv_decode_split left in `workspace` into out, and writes zero rows for
 * empty sequences. Must follow that split call on the same stream with the
 * same batch, num_q_heads, cache, num_parts and workspace. */
pkv_status pkv_decode_combine(const pkv_cache_desc *cache, int32_t batch,
                              int32_t num_q_heads, pkv_dtype out_dtype, void *out,
                              const void *workspace, size_t workspace_bytes,
                              int32_t num_parts, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Merge of partial attention states (the split-K reduce on its own)
 *
 * Attention over a set of tokens may be computed piece by piece: piece i
 * leaves the state (m_i, l_i, o_i), m_i its largest score, l_i = sum_t
 * exp(s_t - m_i) and o_i = sum_t exp(s_t - m_i) v_t (unnormalised, natural
 * exponent). The attention over the union of the pieces is
 *   out = sum_i exp(m_i - M) o_i / sum_i exp(m_i - M) l_i,   M = max_i m_i,
 * whatever the partition: the flash-decoding reduce that pkv_decode_combine
 * applies to the split kernel's own pieces. This call merges states the
 * caller brings, e.g. the pieces of one sequence computed on several GPUs and
 * gathered (the decode kernel's work split is described under "Decode
 * attention"; the pages name no reduce, so its form is the split identity
 * above).
 *
 * part_m, part_l  fp32 [num_states, num_heads]
 * part_o          fp32 [num_states, num_heads, head_dim], 16-byte aligned
 * row_ptr         int32 [num_rows + 1], non-decreasing: row r merges states
 *                 row_ptr[r] .. row_ptr[r+1] - 1 (a range outside
 *                 [0, num_states] is flagged PKV_DEV_BAD_INDEX, row zeroed)
 * out             [num_rows, num_heads, head_dim] in out_dtype (PKV_F16 or
 *                 PKV_BF16), fp32 arithmetic, rounded to nearest even;
 *                 8-byte aligned
 * out_m, out_l    optional fp32 [num_rows, num_heads]: the merged M and
 *                 sum_i exp(m_i - M) l_i, so that (out_m, out_l, out * out_l)
 *                 is itself a state of the union
 * A state with m = -inf (or NaN) or l <= 0 contributes nothing; a row with no
 * other state gets zeros (out_m = -inf, out_l = 0). head_dim: a multiple of
 * 4, at most 512. All arrays are device memory.
 * ------------------------------------------------------------------------ */
pkv_status pkv_merge_states(const float *part_m, const float *part_l, const float *part_o,
                            int64_t num_states, const int32_t *row_ptr, int32_t num_rows,
                            int32_t num_heads, int32_t head_dim, pkv_dtype out_dtype,
                            void *out, float *out_m, float *out_l, uint32_t *dev_status,
                            cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Multi-query attention: speculative verification and prefill chunks
 *
 * n_b = cu_q[b+1] - cu_q[b] new query tokens per sequence (already appended
 * to the cache), causal among themselves: query i of sequence b sits at
 * position L_b - n_b + i (L_b = context_lens[b]) and attends to positions
 * 0 .. L_b - n_b + i. This is the target model scoring a draft's K tokens
 * plus one in one batched pass (Continuous-Batching-LLM-Inference-Engine
 * README, feature list "Speculative decoding") and a prefill chunk mixed into
 * a continuous batch (mini-inference-engine overview). n_b = 1 everywhere is
 * decode attention.
 *
 * q, out: [cu_q[batch], num_q_heads, head_dim]. fp16 / bf16 caches: q in
 * the cache's dtype; INT8 caches: q PKV_F16 or PKV_BF16 (16-byte aligned),
 * k_scales / v_scales as for pkv_decode_attn (NULL for 16-bit caches), values
 * dequantised as code * scale. cu_q: device int32 [batch+1], non-decreasing.
 * max_q_len bounds every n_b; a sequence with n_b > max_q_len, n_b > L_b or
 * L_b beyond its table is flagged PKV_DEV_BAD_LENGTH and its rows are not
 * written. The g = num_q_heads / num_kv_heads query heads of each KV head
 * and the n_b queries form the rows of a tensor-core tile. Supported:
 * head_dim 64 or 128, g in {1, 2, 4, 8}, batch <= 4096. Workspace:
 * pkv_multiquery_workspace_size with the same batch, num_q_heads, max_q_len,
 * cache and num_parts (0 = one range per resident worker); 256-byte aligned.
 * Caches 16-byte aligned.
 * Three kernels serve the call, by rows = max_q_len * g:
 *  - fp16 / bf16 caches, rows >= 128 (a prefill chunk), q and out 16-byte
 *    aligned: a tcgen05 / tensor-memory kernel with one CTA per (sequence,
 *    kv head, 128-row tile) and no split (num_parts and the workspace are
 *    then not used, but are still checked);
 *  - rows <= 24 (speculative verification) over fp16 / bf16 caches, or over
 *    INT8 caches at head_dim 128: an mma.sync kernel with the rows on the
 *    MMA's N side, one warp per worker (num_parts counts warps);
 *  - otherwise: an mma.sync kernel with 16 rows per warp, one CTA per
 *    worker.
 * The split kernels cut their stream of units into num_parts ranges and a
 * combine kernel merges the pieces through the workspace. All compute the
 * same causal attention within the same tolerance (INT8: within 2e-2 of
 * attention over the dequantised cache).
 * ------------------------------------------------------------------------ */
size_t pkv_multiquery_workspace_size(int32_t batch, int32_t num_q_heads, int32_t max_q_len,
                                     const pkv_cache_desc *cache, int32_t num_parts);

pkv_status pkv_multiquery_attn(const void *q, pkv_dtype q_dtype, const int32_t *cu_q,
                               int32_t max_q_len, const void *k_cache, const void *v_cache,
                               const float *k_scales, const float *v_scales,
                               const pkv_cache_desc *cache, const int32_t *block_tables,
                               int32_t max_blocks_per_seq, const int32_t *context_lens,
                               int32_t batch, int32_t num_q_heads, float softmax_scale,
                               void *out, void *workspace, size_t workspace_bytes,
                               int32_t num_parts, uint32_t *dev_status, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Copy-on-write block copy (fork / rollback)
 *
 * Copies whole physical blocks src_blocks[i] -> dst_blocks[i] (all kv heads,
 * K and V, and for INT8 caches the K and V scales), i < num_pairs: the
 * private copy a copy-on-write block gets before a sequence writes into it,
 * and the rollback of a rejected speculative draft onto such copies
 * (Continuous-Batching-LLM-Inference-Engine README, feature list "Paged
 * KV-cache": copy-on-write reference counting; "Speculative decoding":
 * KV-cache rollback uses copy-on-write).
 *
 * src_blocks, dst_blocks: device int32 [num_pairs]. A pair with an id outside
 * [0, num_blocks) is skipped and flagged PKV_DEV_BAD_BLOCK; src == dst is a
 * no-op. A block that is a destination and also a source in the same call
 * gives an unspecified result (pairs run in parallel). k_scales, v_scales may
 * be NULL except for INT8 caches. Caches 16-byte aligned.
 * ------------------------------------------------------------------------ */
pkv_status pkv_copy_blocks(void *k_cache, void *v_cache, float *k_scales, float *v_scales,
                           const pkv_cache_desc *cache, const int32_t *src_blocks,
                           const int32_t *dst_blocks, int32_t num_pairs, uint32_t *dev_status,
                           cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Decode attention without any allocation by anyone
 *
 * No counterpart on the source pages: this variant exists for callers that
 * cannot call cudaMalloc. Some runtimes plan all device memory ahead of time
 * and own the allocator, so a library may not take memory of its own; on a
 * latency-critical serving loop an allocation (and the device-wide
 * synchronisation a cudaFree brings) is not acceptable either; and such a
 * caller cannot size and keep a workspace for pkv_decode_attn.
 *
 * Same computation and arguments as pkv_decode_attn, without workspace and
 * workspace_bytes: the scratch is a fixed array of PKV_NOALLOC_SCRATCH_BYTES
 * compiled into the library, which every GPU that loads the library keeps
 * until the process exits. The function itself allocates nothing.
 *
 * - Calls that need more scratch than that (pkv_decode_workspace_size for
 *   the same batch, num_q_heads, cache and num_parts) return
 *   PKV_ERR_WORKSPACE and launch nothing.
 * - The array's device address belongs to a CUDA context: the first call in
 *   each context (e.g. the device's primary context, which the CUDA runtime
 *   uses) looks it up once, with that device current; later calls in the same
 *   context reuse it. Make that first call before any stream capture. Up to
 *   64 (device, context) pairs per process; more return PKV_ERR_UNSUPPORTED.
 * - All calls share the one array and it keeps the last call's contents;
 *   nothing in it needs to start at zero, since each call rewrites every part
 *   it later reads. Calls whose work overlaps on the GPU (other streams, other
 *   host threads) race on it: order them, e.g. on one stream.
 * ------------------------------------------------------------------------ */
#define PKV_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

pkv_status pkv_decode_attn_noalloc(const void *q, pkv_dtype q_dtype,
                                   const void *k_cache, const void *v_cache,
                                   const float *k_scales, const float *v_scales,
                                   const pkv_cache_desc *cache,
                                   const int32_t *block_tables, int32_t max_blocks_per_seq,
                                   const int32_t *context_lens, int32_t batch,
                                   int32_t num_q_heads, float softmax_scale, void *out,
                                   int32_t num_parts, uint32_t *dev_status,
                                   cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
