/*
 * A plain C11 client of include/fp8w8a8.h. It compiles with no C++ or CUDA
 * header, links the library, and runs argument checks that return before any
 * device work, so it is safe with or without a GPU: every call below is
 * refused on the host, or is a zero-size no-op. Exit status 0 means every
 * check passed; otherwise it is the number of the first failed check.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "fp8w8a8.h"

/* Non-null addresses that the refused calls never dereference. */
#define FAKE ((void *)(uintptr_t)0x10000) /* 16-byte aligned */
#define FAKE_F ((float *)(uintptr_t)0x10000)
#define ODD8 ((void *)(uintptr_t)0x10008) /* 8-byte aligned only */
#define ODD2_F ((float *)(uintptr_t)0x10002)
#define ODD2_I ((const int32_t *)(uintptr_t)0x10002)

static int n_checks;

#define EXPECT(call, want)                                                                          \
    do {                                                                                            \
        int st_ = (call);                                                                           \
        ++n_checks;                                                                                 \
        if (st_ != (want)) {                                                                        \
            fprintf(stderr, "check %d: %s returned %d, expected %d\n", n_checks, #call, st_, (want)); \
            return n_checks;                                                                        \
        }                                                                                           \
    } while (0)

int main(void)
{
    int s;

    /* activation groups */
    EXPECT(fp8_quant_act_group(FAKE, FAKE, FAKE_F, -1, 256, FP8_GROUP, NULL), FP8_ERR_SHAPE);
    EXPECT(fp8_quant_act_group(FAKE, FAKE, FAKE_F, 4, 256, 64, NULL), FP8_ERR_UNSUPPORTED);
    EXPECT(fp8_quant_act_group(FAKE, FAKE, FAKE_F, 4, 200, FP8_GROUP, NULL), FP8_ERR_SHAPE);
    EXPECT(fp8_quant_act_group(NULL, NULL, NULL, 0, 256, FP8_GROUP, NULL), FP8_OK);
    EXPECT(fp8_quant_act_group(FAKE, NULL, FAKE_F, 4, 256, FP8_GROUP, NULL), FP8_ERR_NULL);
    EXPECT(fp8_quant_act_group(ODD8, FAKE, FAKE_F, 4, 256, FP8_GROUP, NULL), FP8_ERR_ALIGN);
    EXPECT(fp8_quant_act_group(FAKE, FAKE, ODD2_F, 4, 256, FP8_GROUP, NULL), FP8_ERR_ALIGN);

    /* weight blocks */
    EXPECT(fp8_quant_weight_block(FAKE, FAKE, FAKE_F, 256, 256, 64, FP8_GROUP, NULL), FP8_ERR_UNSUPPORTED);
    EXPECT(fp8_quant_weight_block(FAKE, FAKE, FAKE_F, 256, 0, FP8_GROUP, FP8_GROUP, NULL), FP8_ERR_SHAPE);
    EXPECT(fp8_quant_weight_block(NULL, NULL, NULL, 0, 256, FP8_GROUP, FP8_GROUP, NULL), FP8_OK);

    /* per tensor */
    EXPECT(fp8_quant_per_tensor(FAKE, FAKE, FAKE_F, 4, 24, 0, NULL), FP8_ERR_SHAPE);
    EXPECT(fp8_quant_per_tensor(FAKE, FAKE, NULL, 4, 32, 0, NULL), FP8_ERR_NULL);
    EXPECT(fp8_quant_per_tensor(NULL, NULL, FAKE_F, 0, 32, 1, NULL), FP8_OK);

    /* block-scaled and grouped GEMM */
    EXPECT(fp8_block_gemm(FAKE, FAKE_F, FAKE, FAKE_F, FAKE, 4, 256, 256, FP8_GROUP, FP8_GROUP, FP8_GROUP, 0,
                          NULL, NULL),
           FP8_ERR_ARG);
    EXPECT(fp8_block_gemm(FAKE, FAKE_F, FAKE, FAKE_F, FAKE, 4, 256, 256, FP8_GROUP, FP8_GROUP, FP8_GROUP, 2,
                          NULL, NULL),
           FP8_ERR_ARG);
    EXPECT(fp8_block_gemm(FAKE, FAKE_F, FAKE, FAKE_F, FAKE, 4, 256, 256, FP8_GROUP, FP8_GROUP, FP8_GROUP,
                          FP8_MAX_GROUPS + 1, (const int32_t *)FAKE, NULL),
           FP8_ERR_UNSUPPORTED);
    EXPECT(fp8_block_gemm(FAKE, FAKE_F, FAKE, FAKE_F, FAKE, 4, 250, 256, FP8_GROUP, FP8_GROUP, FP8_GROUP, 1,
                          NULL, NULL),
           FP8_ERR_SHAPE);
    EXPECT(fp8_block_gemm(FAKE, FAKE_F, FAKE, FAKE_F, FAKE, 64, 256, 256, FP8_GROUP, FP8_GROUP, FP8_GROUP, 2,
                          ODD2_I, NULL),
           FP8_ERR_ALIGN);
    EXPECT(fp8_block_gemm(NULL, NULL, NULL, NULL, NULL, 0, 256, 256, FP8_GROUP, FP8_GROUP, FP8_GROUP, 1, NULL,
                          NULL),
           FP8_OK);

    /* per-tensor GEMM */
    EXPECT(fp8_tensor_gemm(FAKE, FAKE_F, FAKE, FAKE_F, FAKE, 4, 256, 8, NULL), FP8_ERR_SHAPE);
    EXPECT(fp8_tensor_gemm(FAKE, NULL, FAKE, FAKE_F, FAKE, 4, 256, 256, NULL), FP8_ERR_NULL);
    EXPECT(fp8_tensor_gemm(NULL, NULL, NULL, NULL, NULL, 0, 256, 256, NULL), FP8_OK);

    /* the whole linear layer */
    EXPECT(fp8_block_linear(FAKE, FAKE, FAKE_F, FAKE, FAKE_F, FAKE, 4, 256, 200, NULL), FP8_ERR_SHAPE);
    EXPECT(fp8_block_linear(FAKE, FAKE, FAKE_F, FAKE, FAKE_F, NULL, 4, 256, 256, NULL), FP8_ERR_NULL);

    /* dimensions past the documented limits */
    EXPECT(fp8_quant_act_group(FAKE, FAKE, FAKE_F, (int64_t)1 << 31, 256, FP8_GROUP, NULL), FP8_ERR_SHAPE);
    EXPECT(fp8_quant_weight_block(FAKE, FAKE, FAKE_F, (int64_t)1 << 31, 256, FP8_GROUP, FP8_GROUP, NULL),
           FP8_ERR_SHAPE);
    EXPECT(fp8_quant_per_tensor(FAKE, FAKE, FAKE_F, (int64_t)1 << 62, 16, 0, NULL), FP8_ERR_SHAPE);
    EXPECT(fp8_block_gemm(FAKE, FAKE_F, FAKE, FAKE_F, FAKE, 64, (int64_t)1 << 24, 256, FP8_GROUP, FP8_GROUP,
                          FP8_GROUP, FP8_MAX_GROUPS, (const int32_t *)FAKE, NULL),
           FP8_ERR_SHAPE); /* N * num_groups = 2^32 */
    EXPECT(fp8_tensor_gemm(FAKE, FAKE_F, FAKE, FAKE_F, FAKE, 4, 256, ((int64_t)1 << 31) + 16, NULL), FP8_ERR_SHAPE);
    EXPECT(fp8_block_linear(FAKE, FAKE, FAKE_F, FAKE, FAKE_F, FAKE, 4, (int64_t)1 << 31, 256, NULL), FP8_ERR_SHAPE);

    /* the grid limits of the group and block quantizers, exactly at and past the bound */
    EXPECT(fp8_quant_act_group(FAKE, FAKE, FAKE_F, 4, FP8_ACT_GROUP_MAX_K + FP8_GROUP, FP8_GROUP, NULL),
           FP8_ERR_SHAPE);
    EXPECT(fp8_quant_act_group(FAKE, FAKE, FAKE_F, 0, FP8_ACT_GROUP_MAX_K, FP8_GROUP, NULL), FP8_OK);
    EXPECT(fp8_quant_weight_block(FAKE, FAKE, FAKE_F, FP8_WEIGHT_BLOCK_MAX_N + 1, 256, FP8_GROUP, FP8_GROUP, NULL),
           FP8_ERR_SHAPE);

    /* row-wise quantization and GEMM */
    EXPECT(fp8_quant_rowwise(FAKE, FAKE, FAKE_F, 4, 24, NULL), FP8_ERR_SHAPE);
    EXPECT(fp8_quant_rowwise(FAKE, NULL, FAKE_F, 4, 32, NULL), FP8_ERR_NULL);
    EXPECT(fp8_quant_rowwise(ODD8, FAKE, FAKE_F, 4, 32, NULL), FP8_ERR_ALIGN);
    EXPECT(fp8_quant_rowwise(NULL, NULL, NULL, 0, 32, NULL), FP8_OK);
    EXPECT(fp8_rowwise_gemm(FAKE, FAKE_F, FAKE, FAKE_F, FAKE, 4, 24, 256, NULL), FP8_ERR_SHAPE);
    EXPECT(fp8_rowwise_gemm(FAKE, FAKE_F, FAKE, ODD2_F + 1, FAKE, 4, 256, 256, NULL), FP8_ERR_ALIGN); /* sw 16 B */
    EXPECT(fp8_rowwise_gemm(FAKE, FAKE_F, FAKE, NULL, FAKE, 4, 256, 256, NULL), FP8_ERR_NULL);

    /* FP8 KV cache */
    EXPECT(fp8_kv_cache_store(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE_F, FAKE_F, 4, 24, 8, NULL), FP8_ERR_SHAPE);
    EXPECT(fp8_kv_cache_store(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE_F, NULL, 4, 128, 8, NULL), FP8_ERR_NULL);
    EXPECT(fp8_kv_cache_load(FAKE, FAKE, FAKE, FAKE, (const int64_t *)ODD2_I, FAKE_F, FAKE_F, 4, 128, 8, NULL),
           FP8_ERR_ALIGN);
    EXPECT(fp8_kv_cache_load(NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, 128, 8, NULL), FP8_OK);

    /* the conversion self-test: n a multiple of 8, no pattern past 0xFFFFFFFF */
    EXPECT(fp8_selftest_encode_f32(0, 12, FAKE, NULL), FP8_ERR_SHAPE);
    EXPECT(fp8_selftest_encode_f32(0, -8, FAKE, NULL), FP8_ERR_SHAPE);
    EXPECT(fp8_selftest_encode_f32(0xFFFFFFF8u, 16, FAKE, NULL), FP8_ERR_SHAPE);
    EXPECT(fp8_selftest_encode_f32(0, 8, NULL, NULL), FP8_ERR_NULL);
    EXPECT(fp8_selftest_encode_f32(0, 8, ODD8, NULL), FP8_ERR_ALIGN);
    EXPECT(fp8_selftest_encode_f32(0xFFFFFFF8u, 0, NULL, NULL), FP8_OK);

    /* the error word needs somewhere to go */
    EXPECT(fp8_device_error(NULL, NULL, NULL), FP8_ERR_NULL);

    /* status text: one non-empty string per status, and one for unknown values */
    for (s = FP8_OK; s <= FP8_ERR_TIMEOUT + 1; ++s) {
        const char *text = fp8_status_string(s);
        ++n_checks;
        if (text == NULL || strlen(text) == 0) {
            fprintf(stderr, "check %d: no status text for %d\n", n_checks, s);
            return n_checks;
        }
    }

    printf("%d checks passed\n", n_checks);
    return 0;
}
