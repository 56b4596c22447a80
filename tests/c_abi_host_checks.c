/*
 * libpkv's C ABI used from plain C: this file includes only pkv.h and the C
 * library, with no CUDA, C++ or Python, and links against libpkv.so.
 *
 * Every call below either is a size query with an explicit worker count or is
 * rejected by the library's host-side argument checks before anything touches
 * the CUDA runtime, so the program runs on a machine without a GPU. The fake
 * device pointers are never dereferenced. Prints "ok" and exits 0 when every
 * check holds; otherwise names each failed check on stderr and exits 1.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "pkv.h"

static int failures = 0;

#define CHECK(cond)                                                     \
    do {                                                                \
        if (!(cond)) {                                                  \
            fprintf(stderr, "check failed (line %d): %s\n", __LINE__, #cond); \
            ++failures;                                                 \
        }                                                               \
    } while (0)

static size_t align256(size_t x) { return (x + 255) / 256 * 256; }

/* Decode workspace: block prefix int32 [batch + 1], partial (m, l) fp32
 * [slots, g, 2] and partial o fp32 [slots, g, head_dim], each 256-byte
 * aligned, slots = batch * num_kv_heads + workers. */
static size_t decode_ws(int batch, int hkv, int g, int d, int workers) {
    const size_t slots = (size_t)batch * hkv + workers;
    return align256(4 * (size_t)(batch + 1)) + align256(slots * g * 2 * 4) +
           align256(slots * g * d * 4);
}

int main(void) {
    void *fake = (void *)(uintptr_t)0x100000;      /* 256-byte aligned, never read */
    void *fake8 = (void *)(uintptr_t)0x100008;     /* 8-byte aligned only */
    const pkv_cache_desc bf16 = {64, 16, 8, 128, PKV_BF16};
    const pkv_cache_desc i8 = {64, 16, 8, 128, PKV_I8};
    const pkv_cache_desc d96 = {64, 16, 8, 96, PKV_BF16};
    const pkv_cache_desc bs32 = {64, 32, 8, 128, PKV_BF16};

    /* status names */
    CHECK(strcmp(pkv_status_string(PKV_OK), "PKV_OK") == 0);
    CHECK(strncmp(pkv_status_string(PKV_ERR_WORKSPACE), "PKV_ERR_WORKSPACE", 17) == 0);
    CHECK(strcmp(pkv_status_string((pkv_status)99), "PKV_ERR_UNKNOWN") == 0);

    /* append: scratch sizes, nothing to do, rejected arguments */
    CHECK(pkv_append_workspace_size(&bf16) == 0);
    CHECK(pkv_append_workspace_size(&i8) == 80u * 64u * 8u);   /* 80 bytes per tile */
    CHECK(pkv_append_workspace_size(&d96) == 0);
    CHECK(pkv_append(NULL, NULL, PKV_BF16, 0, NULL, NULL, NULL, NULL, NULL, &bf16, NULL, 0,
                     NULL, NULL) == PKV_OK);
    CHECK(pkv_append(fake, fake, PKV_BF16, 4, fake, fake, fake, NULL, NULL, NULL, NULL, 0, NULL,
                     NULL) == PKV_ERR_INVALID_ARG);
    CHECK(pkv_append(fake8, fake, PKV_BF16, 4, fake, fake, fake, NULL, NULL, &bf16, NULL, 0,
                     NULL, NULL) == PKV_ERR_INVALID_ARG);
    CHECK(pkv_append(fake, fake, PKV_F16, 4, fake, fake, fake, NULL, NULL, &bf16, NULL, 0, NULL,
                     NULL) == PKV_ERR_INVALID_ARG);
    CHECK(pkv_append(fake, fake, PKV_BF16, 4, fake, fake, fake, NULL, NULL, &i8, fake, 1 << 20,
                     NULL, NULL) == PKV_ERR_INVALID_ARG);   /* INT8 without scales */
    CHECK(pkv_append(fake, fake, PKV_BF16, 4, fake, fake, fake, fake, fake, &i8, fake, 16, NULL,
                     NULL) == PKV_ERR_WORKSPACE);
    CHECK(pkv_append(fake, fake, PKV_BF16, 4, fake, fake, fake, NULL, NULL, &bs32, NULL, 0, NULL,
                     NULL) == PKV_ERR_UNSUPPORTED);

    /* decode workspace sizes with explicit worker counts (no device query) */
    CHECK(pkv_decode_workspace_size(256, 32, &bf16, 1216) == decode_ws(256, 8, 4, 128, 1216));
    CHECK(pkv_decode_workspace_size(256, 64, &bf16, 1216) == decode_ws(256, 8, 8, 128, 1216));
    CHECK(pkv_decode_workspace_size(7, 8, &bf16, 3) == decode_ws(7, 8, 1, 128, 3));
    CHECK(pkv_decode_workspace_size(256, 128, &bf16, 64) == 0);   /* group 16 */
    CHECK(pkv_decode_workspace_size(256, 12, &bf16, 64) == 0);    /* 12 % 8 != 0 */
    CHECK(pkv_decode_workspace_size(256, 32, &d96, 64) == 0);

    /* decode attention: rejected before any launch */
    CHECK(pkv_decode_attn(fake, PKV_BF16, fake, fake, NULL, NULL, &bf16, fake, 4, fake, 4, 128,
                          0.125f, fake, fake, 1u << 30, 64, NULL, NULL) == PKV_ERR_UNSUPPORTED);
    CHECK(pkv_decode_attn(fake, PKV_BF16, fake, fake, NULL, NULL, &bf16, fake, 4, fake, 0, 32,
                          0.125f, fake, fake, 1u << 30, 64, NULL, NULL) == PKV_OK);  /* empty */
    CHECK(pkv_decode_attn(fake8, PKV_BF16, fake, fake, NULL, NULL, &bf16, fake, 4, fake, 4, 32,
                          0.125f, fake, fake, 1u << 30, 64, NULL, NULL) == PKV_ERR_INVALID_ARG);
    CHECK(pkv_decode_attn(fake, PKV_BF16, fake, fake, NULL, NULL, &i8, fake, 4, fake, 4, 32,
                          0.125f, fake, fake, 1u << 30, 64, NULL, NULL) == PKV_ERR_INVALID_ARG);
    CHECK(pkv_decode_attn(fake, PKV_BF16, fake, fake, NULL, NULL, &bf16, fake, 4, fake, 4, 32,
                          0.125f, fake, fake, 64, 64, NULL, NULL) == PKV_ERR_WORKSPACE);
    CHECK(pkv_decode_split(fake, PKV_F16, fake, fake, NULL, NULL, &bf16, fake, 4, fake, 4, 32,
                           0.125f, fake, fake, 1u << 30, 64, NULL, NULL) == PKV_ERR_INVALID_ARG);
    CHECK(pkv_decode_combine(&bf16, 4, 32, PKV_BF16, fake, fake, 16, 64, NULL) ==
          PKV_ERR_WORKSPACE);
    CHECK(pkv_decode_step(fake, PKV_BF16, fake, fake, fake, fake, NULL, NULL, &i8, fake, 4, fake,
                          4, 32, 0.125f, fake, fake, 1u << 30, 64, 1, NULL, NULL) ==
          PKV_ERR_INVALID_ARG);   /* INT8 caches need their scales */
    CHECK(pkv_decode_step(fake, PKV_BF16, fake8, fake, fake, fake, NULL, NULL, &bf16, fake, 4, fake,
                          4, 32, 0.125f, fake, fake, 1u << 30, 64, 1, NULL, NULL) ==
          PKV_ERR_INVALID_ARG);
    CHECK(pkv_decode_attn_noalloc(fake, PKV_BF16, fake, fake, NULL, NULL, &d96, fake, 4, fake, 4,
                                  32, 0.125f, fake, 64, NULL, NULL) == PKV_ERR_UNSUPPORTED);
    CHECK(pkv_decode_attn_noalloc(fake, PKV_BF16, fake, fake, NULL, NULL, &bf16, fake, 4, fake,
                                  0, 32, 0.125f, fake, 64, NULL, NULL) == PKV_OK);   /* empty */

    /* multi-query attention and block copy */
    CHECK(pkv_multiquery_attn(fake, PKV_BF16, fake, 5, fake, fake, NULL, NULL, &bf16, fake, 4,
                              fake, 4, 128, 0.125f, fake, fake, 1u << 30, 16, NULL, NULL) ==
          PKV_ERR_UNSUPPORTED);                                     /* group 16 */
    CHECK(pkv_multiquery_attn(fake, PKV_BF16, fake, 0, fake, fake, NULL, NULL, &bf16, fake, 4,
                              fake, 4, 32, 0.125f, fake, fake, 1u << 30, 16, NULL, NULL) ==
          PKV_ERR_INVALID_ARG);                                     /* max_q_len 0 */
    CHECK(pkv_multiquery_attn(fake, PKV_BF16, fake, 5, fake, fake, NULL, NULL, &i8, fake, 4,
                              fake, 4, 32, 0.125f, fake, fake, 1u << 30, 16, NULL, NULL) ==
          PKV_ERR_INVALID_ARG);                                     /* INT8 needs scales */
    CHECK(pkv_copy_blocks(fake, fake, NULL, NULL, &bf16, fake, fake, 0, NULL, NULL) == PKV_OK);
    CHECK(pkv_copy_blocks(fake, fake, NULL, NULL, &bf16, fake, fake, -1, NULL, NULL) ==
          PKV_ERR_INVALID_ARG);
    CHECK(pkv_copy_blocks(fake, fake, NULL, NULL, &i8, fake, fake, 3, NULL, NULL) ==
          PKV_ERR_INVALID_ARG);                                     /* INT8 needs scales */

    /* merge of partial states */
    {
        const float *ff = (const float *)fake;
        CHECK(pkv_merge_states(ff, ff, ff, 8, fake, 0, 4, 128, PKV_BF16, fake, NULL, NULL, NULL,
                               NULL) == PKV_OK);                    /* no rows */
        CHECK(pkv_merge_states(ff, ff, ff, 8, fake, 2, 4, 126, PKV_BF16, fake, NULL, NULL, NULL,
                               NULL) == PKV_ERR_INVALID_ARG);       /* head_dim % 4 */
        CHECK(pkv_merge_states(ff, ff, ff, 8, fake, 2, 4, 1024, PKV_BF16, fake, NULL, NULL, NULL,
                               NULL) == PKV_ERR_UNSUPPORTED);       /* head_dim > 512 */
        CHECK(pkv_merge_states(ff, ff, ff, 8, fake, 2, 4, 128, PKV_I8, fake, NULL, NULL, NULL,
                               NULL) == PKV_ERR_INVALID_ARG);       /* out dtype */
        CHECK(pkv_merge_states(ff, ff, (const float *)fake8, 8, fake, 2, 4, 128, PKV_BF16, fake,
                               NULL, NULL, NULL, NULL) == PKV_ERR_INVALID_ARG);   /* o misaligned */
        CHECK(pkv_merge_states(NULL, ff, ff, 8, fake, 2, 4, 128, PKV_BF16, fake, NULL, NULL, NULL,
                               NULL) == PKV_ERR_INVALID_ARG);       /* m missing */
    }

    if (failures) {
        printf("%d check(s) failed\n", failures);
        return 1;
    }
    printf("ok\n");
    return 0;
}
