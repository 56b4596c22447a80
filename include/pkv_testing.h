/*
 * pkv_testing.h -- test hooks of libpkv. Not part of the serving API.
 *
 * The paged decode kernels bound every wait on an in-kernel copy: a wait that
 * runs out sets PKV_DEV_TIMEOUT in *dev_status, the warp stops, waits (again
 * bounded) for the copies it did issue and returns, so the CUDA context stays
 * usable. Nothing on the normal path makes a wait run out, so this hook makes
 * one run out on purpose, without any GPU fault: it arms one unit's stage for
 * 16 bytes more than its copies deliver. The source pages have no counterpart;
 * it exists so that the timeout path is exercised by a test. The hook acts
 * only on the stages a worker fills before its loop starts, so the kernels'
 * steady-state loop carries no test code.
 */
#ifndef PKV_TESTING_H
#define PKV_TESTING_H

#include "pkv.h"

#ifdef __cplusplus
extern "C" {
#endif

/* pkv_decode_attn (same arguments and checks) with two changes:
 *   wait_limit_ns  limit of each bounded wait, at most the built-in 4 s
 *   stall_worker   -1: none; otherwise the worker warp with this index (of
 *                  num_parts, or of the default count) never completes the
 *                  wait for its first unit (a worker without units: no stall)
 * After a stalled call *dev_status holds PKV_DEV_TIMEOUT and the rows of the
 * sequences whose pieces the stalled worker held are undefined; every other
 * row is correct. The call itself returns PKV_OK (the stall is seen on the
 * device). PKV_ERR_INVALID_ARG for a larger limit or stall_worker < -1. */
pkv_status pkv_testing_decode_attn_stall(const void *q, pkv_dtype q_dtype,
                                         const void *k_cache, const void *v_cache,
                                         const float *k_scales, const float *v_scales,
                                         const pkv_cache_desc *cache,
                                         const int32_t *block_tables,
                                         int32_t max_blocks_per_seq,
                                         const int32_t *context_lens, int32_t batch,
                                         int32_t num_q_heads, float softmax_scale, void *out,
                                         void *workspace, size_t workspace_bytes,
                                         int32_t num_parts, uint64_t wait_limit_ns,
                                         int32_t stall_worker, uint32_t *dev_status,
                                         cudaStream_t stream);

/* pkv_multiquery_attn (same arguments and checks) with the same two
 * changes, stall_cta naming a worker of the kernel that serves the call: for
 * query runs served by a split kernel, that worker's first unit (a CTA of the
 * 16-rows-per-warp kernel, a warp of the short-run kernel); for runs served
 * by the tcgen05 kernel, that CTA's first chunk never completes (the tcgen05
 * kernel bounds its waits at 2 s whatever the limit given). After a stalled
 * call *dev_status holds PKV_DEV_TIMEOUT plus a diagnostic bit naming the
 * waiting role (0x100 / 0x200: consumer / producer of a split kernel;
 * 0x400 / 0x800 / 0x1000: producer / MMA issuer / softmax of the tcgen05
 * kernel); rows the stalled work covered are undefined. */
pkv_status pkv_testing_multiquery_attn_stall(const void *q, pkv_dtype q_dtype,
                                             const int32_t *cu_q, int32_t max_q_len,
                                             const void *k_cache, const void *v_cache,
                                             const float *k_scales, const float *v_scales,
                                             const pkv_cache_desc *cache,
                                             const int32_t *block_tables,
                                             int32_t max_blocks_per_seq,
                                             const int32_t *context_lens, int32_t batch,
                                             int32_t num_q_heads, float softmax_scale,
                                             void *out, void *workspace, size_t workspace_bytes,
                                             int32_t num_parts, uint64_t wait_limit_ns,
                                             int32_t stall_cta, uint32_t *dev_status,
                                             cudaStream_t stream);

/* Which kernel pkv_multiquery_attn runs for these sizes (q and out taken as
 * 16-byte aligned), and its row-tile height: PKV_TESTING_MQ_TCGEN05
 * (128-row tiles, no split), PKV_TESTING_MQ_SHORT / PKV_TESTING_MQ_SHORT_I8
 * (query rows on the MMA's N side, one warp per worker; fp16 / bf16 and
 * INT8 caches), PKV_TESTING_MQ_ROWS16 (16 rows per warp, one CTA per
 * worker). num_parts must be positive (no device query). Returns the size
 * and argument checks of pkv_multiquery_workspace_size. */
#define PKV_TESTING_MQ_TCGEN05 0
#define PKV_TESTING_MQ_SHORT 1
#define PKV_TESTING_MQ_SHORT_I8 2
#define PKV_TESTING_MQ_ROWS16 3
pkv_status pkv_testing_multiquery_kernel(int32_t batch, int32_t num_q_heads, int32_t max_q_len,
                                         const pkv_cache_desc *cache, pkv_dtype q_dtype,
                                         int32_t num_parts, int32_t *kernel,
                                         int32_t *rows_per_tile);

#ifdef __cplusplus
}
#endif

#endif /* PKV_TESTING_H */
