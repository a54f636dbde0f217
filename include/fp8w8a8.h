/*
 * fp8w8a8.h — C ABI of the GB300 (sm_103a) FP8 W8A8 linear-layer library.
 *
 * What the library computes (readings of the pages are marked as such):
 *
 *  - E4M3: 4 exponent bits, 3 mantissa bits, no infinity, range +-448
 *    ("[vLLM] FP8: 8비트 부동소수점 양자화", section "논문 핵심 내용" and its
 *    format table). Reading: bias 7, S.1111.111 is NaN, encoding rounds to
 *    nearest even and saturates to +-448, the sign of zero is kept.
 *  - Symmetric scales, dynamic per-token 128-groups for activations and
 *    static 128x128 blocks for weights; per-tensor scales, static or dynamic
 *    (same page, sections "스케일링 전략 체계" and "블록 양자화"; the online
 *    per-tensor mode of "서빙을 위한 양자화 가이드 FP8, AWQ, GPTQ", section
 *    "연산까지 빨라지는 W8A8, FP8").
 *    Reading: scale = fl32(max(amax, 1e-10) / 448) in IEEE FP32, code =
 *    e4m3(fl32(x / scale)) with a correctly rounded FP32 division.
 *  - GEMM on FP8 operands with high-precision accumulation, not a dequantize
 *    to BF16 followed by a BF16 GEMM ("FP8 and FP4: Throughput Needs Scaling",
 *    section "Kernel caveat가 마지막 관문이다"). Reading: FP32 accumulation
 *    on the tensor cores within each 128-wide K block, the block's activation
 *    and weight scales applied once per block in FP32, BF16 output.
 *  - Matrix dimensions multiples of 16 for the FP8 tensor-core path ("FP8
 *    serving slower than BF16", section "하드웨어 세대가 전제를 바꾼다").
 *
 * Conventions for every entry point:
 *  - All matrices are dense and row-major. Every data pointer is caller-owned
 *    DEVICE memory on the current CUDA device (BF16 as 2-byte values, E4M3 as
 *    1-byte codes, scales as FP32); data pointers must be 16-byte aligned,
 *    scale pointers 4-byte aligned. The library never allocates, frees or
 *    synchronises inside a call.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream). Work is enqueued asynchronously on it; outputs are valid once
 *    the stream reaches that point.
 *  - The return value is a status (FP8_OK = 0). Argument errors are detected
 *    on the host before anything is enqueued. A zero M (or rows) is a valid
 *    no-op.
 *  - The GEMMs, fp8_block_linear and fp8_quant_rowwise take each of M, N, K
 *    (and N * num_groups when grouped) up to INT_MAX; larger values give
 *    FP8_ERR_SHAPE. fp8_quant_act_group takes K up to FP8_ACT_GROUP_MAX_K and
 *    fp8_quant_weight_block N up to FP8_WEIGHT_BLOCK_MAX_N (the other size up
 *    to INT_MAX). fp8_quant_per_tensor takes any rows * cols that fits in half
 *    of the int64_t range.
 *  - Device-side waits in the kernels are bounded (about one second); if one
 *    expires the kernel stops early and records FP8_ERR_TIMEOUT, which
 *    fp8_device_error() reports. Kernels never trap.
 *  - A few arguments can only be checked on the device (a static scale, the
 *    grouped offsets, routed-row indices, KV cache slots and scales): a bad
 *    one is recorded as FP8_ERR_ARG in the same error word with the site that
 *    found it, the access it would have made is clamped or skipped so that no
 *    buffer is left, the call still completes, and its outputs are
 *    unspecified.
 *
 * Programmatic dependent launch (PDL). Some kernels are launched as
 * programmatic dependents of the work before them on the stream, and some
 * let the next kernel launch before they complete (griddepcontrol.
 * launch_dependents). A dependent always waits for its predecessor to
 * complete before it reads that predecessor's outputs - with one exception:
 * the decode GEMM (fp8_block_gemm dense, fp8_tensor_gemm, fp8_rowwise_gemm
 * and fp8_block_linear, each with M <= 16) starts loading qw before that wait.
 * So qw must not be written by a kernel that lets its dependents launch
 * early. Per entry point:
 *    fp8_quant_act_group     lets its dependent launch early (its q and s are
 *    (and _gather)           written after that): never use its codes as the
 *                            qw of a decode GEMM enqueued directly after it;
 *    fp8_quant_weight_block  does not (qw from it is safe);
 *    fp8_quant_per_tensor    does not, static or dynamic: its last kernel
 *                            triggers only by completing (qw from it is safe);
 *    fp8_quant_rowwise       does not (qw from it is safe);
 *    decode GEMM             lets its dependent launch early; it writes y
 *                            after its own wait, and reads only qw early;
 *    prefill GEMM            does not;
 *    fp8_block_linear        its quantizer lets its own GEMM launch early (the
 *                            GEMM reads qa and sa after its wait); its GEMM is
 *                            the decode or prefill GEMM above.
 * Work that is not this library's (torch kernels, copies) never triggers
 * early, so a plain stream order with it is always safe.
 */
#ifndef FP8W8A8_H
#define FP8W8A8_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum fp8_status {
    FP8_OK = 0,
    FP8_ERR_NULL = 1,        /* a required pointer is NULL */
    FP8_ERR_SHAPE = 2,       /* negative size, K == 0, or a size that breaks a multiple-of rule */
    FP8_ERR_ALIGN = 3,       /* data pointer not 16-byte aligned, scale pointer not 4-byte aligned */
    FP8_ERR_UNSUPPORTED = 4, /* group/block size other than 128, or too many groups */
    FP8_ERR_ARG = 5,         /* other invalid argument (num_groups, group_offsets) */
    FP8_ERR_DEVICE = 6,      /* current device is not compute capability 10.3 (sm_103a) */
    FP8_ERR_CUDA = 7,        /* a CUDA runtime call or kernel launch failed */
    FP8_ERR_TIMEOUT = 8      /* a bounded device-side wait expired (reported by fp8_device_error) */
};

/* Width of an activation group along K and the side of a weight block. */
#define FP8_GROUP 128
/* Largest num_groups accepted by fp8_block_gemm. */
#define FP8_MAX_GROUPS 256
/* Largest K of fp8_quant_act_group (65535 CTAs of 8 groups along K). */
#define FP8_ACT_GROUP_MAX_K ((int64_t)65535 * 8 * FP8_GROUP)
/* Largest N of fp8_quant_weight_block (65535 block rows). */
#define FP8_WEIGHT_BLOCK_MAX_N ((int64_t)65535 * FP8_GROUP)

/*
 * Dynamic activation quantization, one scale per token per 128-wide K group
 * (the "128 block dynamic symmetric" strategy, kFp8Dynamic128Sym, of the vLLM
 * page's section "스케일링 전략 체계"; reading: 1 x 128 groups along K).
 *
 *   x_bf16  [M][K] BF16, input.
 *   q_e4m3  [M][K] E4M3 codes, output.
 *   scales  [K/128][M] FP32, output: scales[g*M + m] belongs to row m, columns
 *           128g .. 128g+127 (M contiguous, so a GEMM tile reads a run of rows).
 *   group_k must be 128. K must be a positive multiple of 128; M >= 0 is any.
 * Errors: NULL, SHAPE, ALIGN, UNSUPPORTED, DEVICE, CUDA.
 */
int fp8_quant_act_group(const void *x_bf16, void *q_e4m3, float *scales,
                        int64_t M, int64_t K, int group_k, void *stream);

/*
 * Activation quantization of routed rows (mixture of experts): row m of the
 * output is row row_index[m] of x quantized as fp8_quant_act_group does, so the
 * expert-sorted codes that the grouped fp8_block_gemm reads are written
 * straight from the token-order activations, with no permuted copy of x
 * (Fp8MoEMethod of "[vLLM] FP8", section "Fp8Config: 온라인 vs 오프라인"; the
 * routing itself is the caller's). Quantization is per row, so the codes and
 * scales equal fp8_quant_act_group's on the permuted rows, bit for bit.
 *
 *   x_bf16     [M_src][K] BF16, input, token order.
 *   row_index  DEVICE int32 [M]: the source row of each routed row. A value
 *              outside [0, M_src) is recorded as FP8_ERR_ARG (site 303) in
 *              the device error word and reads row 0.
 *   q_e4m3     [M][K] E4M3, scales [K/128][M] FP32: outputs, routed order.
 *   group_k must be 128; K a positive multiple of 128 up to
 *   FP8_ACT_GROUP_MAX_K; M >= 0; M_src >= 1 when M > 0.
 * PDL: as fp8_quant_act_group.
 * Errors: NULL, SHAPE, ALIGN, UNSUPPORTED, DEVICE, CUDA.
 */
int fp8_quant_act_group_gather(const void *x_bf16, const int32_t *row_index, void *q_e4m3, float *scales,
                               int64_t M, int64_t M_src, int64_t K, int group_k, void *stream);

/*
 * Weight block quantization (offline, at load time), one scale per 128 x 128
 * block (weight_block_size of section "블록 양자화"; kFp8Static128BlockSym).
 *
 *   w_bf16  [N][K] BF16, input.
 *   q_e4m3  [N][K] E4M3 codes, output.
 *   scales  [ceil(N/128)][K/128] FP32, output (row-major). The last block row
 *           may be short when N is not a multiple of 128.
 *   block_n and block_k must be 128; K a positive multiple of 128; N >= 0.
 * Errors: NULL, SHAPE, ALIGN, UNSUPPORTED, DEVICE, CUDA.
 */
int fp8_quant_weight_block(const void *w_bf16, void *q_e4m3, float *scales,
                           int64_t N, int64_t K, int block_n, int block_k, void *stream);

/*
 * Per-tensor quantization (kFp8StaticTensorSym / kFp8DynamicTensorSym; the
 * online "--quantization fp8" mode that keeps one scale per tensor and
 * recomputes the activation scale every step).
 *
 *   x_bf16  [rows][cols] BF16, input.
 *   q_e4m3  [rows][cols] E4M3 codes, output.
 *   scale   ONE FP32 in device memory. is_static != 0: input, must hold a
 *           finite positive scale (checked on the device: otherwise
 *           FP8_ERR_ARG, site 301 or 302, is recorded in the error word).
 *           is_static == 0: output, receives fl32(max(amax, 1e-10) / 448) of
 *           the whole tensor.
 *   cols must be a positive multiple of 16; rows >= 0.
 * A dynamic call enqueues up to four launches (zero the slot, amax, quantize,
 * write the scale); the scale slot holds the amax bit pattern in between, so
 * it must not be read by other work until the call's work is done. The last
 * kernel of either mode lets nothing launch before it completes, so its codes
 * may be the weights of a decode GEMM enqueued directly after it.
 * Errors: NULL, SHAPE, ALIGN, DEVICE, CUDA.
 */
int fp8_quant_per_tensor(const void *x_bf16, void *q_e4m3, float *scale,
                         int64_t rows, int64_t cols, int is_static, void *stream);

/*
 * Block-scaled FP8 GEMM, Y = A * W^T with 1x128 activation groups and 128x128
 * weight blocks:
 *   Y[m,n] = bf16( sum_g Sa[g][m] * Sw[n/128][g] * sum_{k in g} dec(Qa[m,k]) dec(Qw[n,k]) )
 * The inner sums run on the tensor cores in FP32; each 128-wide K block is
 * scaled and added to an FP32 accumulator once.
 *
 *   qa   [M][K] E4M3, sa [K/128][M] FP32 (as written by fp8_quant_act_group).
 *   qw   [N][K] E4M3, sw [ceil(N/128)][K/128] FP32 (as written by
 *        fp8_quant_weight_block). Grouped: qw [num_groups][N][K] and
 *        sw [num_groups][ceil(N/128)][K/128], expert e at offset e*N*K / e*ceil(N/128)*(K/128).
 *   y    [M][N] BF16, output.
 *   block_n, block_k, group_k must be 128. K a positive multiple of 128,
 *   N a positive multiple of 16, M >= 0.
 *   num_groups == 1 and group_offsets == NULL: dense GEMM.
 *   Otherwise grouped (mixture-of-experts): group_offsets is DEVICE int32
 *   [num_groups+1], non-decreasing, with 0 <= offsets[0] and
 *   offsets[num_groups] <= M; rows [offsets[e], offsets[e+1]) of qa/y use
 *   expert e's weights. Rows outside [offsets[0], offsets[num_groups]) are not
 *   written. Offsets are read on the device and are trusted.
 *   num_groups in [1, FP8_MAX_GROUPS].
 * M <= 16 (dense) uses the weight-streaming decode kernel, otherwise the
 * tile-persistent prefill kernel. The decode kernel is a programmatic
 * dependent of the work before it on `stream` and starts reading qw before
 * that work has completed: qw must not be written by a kernel that allows
 * its dependents to launch early (see "Programmatic dependent launch" above;
 * fp8_quant_weight_block and fp8_quant_per_tensor never do, so a plain stream
 * order after them suffices).
 * Offsets that are not non-decreasing within [0, M] are recorded as
 * FP8_ERR_ARG (site 106) in the device error word; they are clamped into
 * [0, M], so nothing is accessed outside the buffers.
 * Errors: NULL, SHAPE, ALIGN, UNSUPPORTED, ARG, DEVICE, CUDA.
 */
int fp8_block_gemm(const void *qa, const float *sa, const void *qw, const float *sw,
                   void *y_bf16, int64_t M, int64_t N, int64_t K,
                   int block_n, int block_k, int group_k,
                   int num_groups, const int32_t *group_offsets, void *stream);

/*
 * Per-tensor FP8 GEMM: Y[m,n] = bf16( sa * sw * sum_k dec(Qa[m,k]) dec(Qw[n,k]) ),
 * FP32 accumulation over all of K, one scale product applied at the end.
 *
 *   qa [M][K] E4M3, qw [N][K] E4M3, y [M][N] BF16.
 *   sa, sw: ONE FP32 each, in DEVICE memory (as written by fp8_quant_per_tensor).
 *   K and N positive multiples of 16, M >= 0.
 * M <= 16 uses the decode kernel, with the same condition on qw as
 * fp8_block_gemm (fp8_quant_per_tensor, static or dynamic, satisfies it).
 * Errors: NULL, SHAPE, ALIGN, DEVICE, CUDA.
 */
int fp8_tensor_gemm(const void *qa, const float *sa, const void *qw, const float *sw,
                    void *y_bf16, int64_t M, int64_t N, int64_t K, void *stream);

/*
 * Row-wise quantization: one scale per row of a BF16 matrix. For activations
 * the rows are tokens (the dynamic per-token strategy, kFp8DynamicTokenSym,
 * of "[vLLM] FP8", section "스케일링 전략 체계"); for weights the rows are
 * output channels (the channel-wise weight scales of "서빙을 위한 양자화 가이드
 * FP8, AWQ, GPTQ", section "연산까지 빨라지는 W8A8, FP8").
 *
 *   x_bf16  [rows][cols] BF16, input.
 *   q_e4m3  [rows][cols] E4M3 codes, output.
 *   scales  [rows] FP32, output: fl32(max(amax of the row, 1e-10) / 448).
 *   cols a positive multiple of 16; rows >= 0.
 * The kernel lets nothing launch before it completes, so its codes may be the
 * weights of a decode GEMM enqueued directly after it.
 * Errors: NULL, SHAPE, ALIGN, DEVICE, CUDA.
 */
int fp8_quant_rowwise(const void *x_bf16, void *q_e4m3, float *scales, int64_t rows, int64_t cols,
                      void *stream);

/*
 * FP8 GEMM with per-token activation and per-channel weight scales:
 *   Y[m,n] = bf16( sa[m] * sw[n] * sum_k dec(Qa[m,k]) dec(Qw[n,k]) ),
 * FP32 accumulation over all of K, the scale product applied once at the end.
 *
 *   qa [M][K] E4M3 and sa [M] FP32 (as written by fp8_quant_rowwise on X).
 *   qw [N][K] E4M3 and sw [N] FP32 (as written by fp8_quant_rowwise on W);
 *   sw must be 16-byte aligned.
 *   y  [M][N] BF16, output.
 *   K and N positive multiples of 16, M >= 0.
 * M <= 16 uses the decode kernel, with the same condition on qw as
 * fp8_block_gemm (fp8_quant_rowwise satisfies it).
 * Errors: NULL, SHAPE, ALIGN, DEVICE, CUDA.
 */
int fp8_rowwise_gemm(const void *qa, const float *sa, const void *qw, const float *sw,
                     void *y_bf16, int64_t M, int64_t N, int64_t K, void *stream);

/*
 * FP8 KV cache, store: quantizes one step's keys and values into an E4M3
 * cache with one FP32 scale per tensor for keys and one for values (the FP8
 * KV cache of "[vLLM] FP8", section "KV 캐시 양자화", Fp8KVCacheMethod; the
 * scales are 1.0 when no calibrated scale is given).
 *
 *   key_bf16, value_bf16   [num_tokens][token_elems] BF16, inputs
 *                          (token_elems = KV heads * head dim).
 *   key_cache, value_cache [num_slots][token_elems] E4M3, written at the slots
 *                          below: cache[slot][e] = e4m3(fl32(x[t][e] / scale)).
 *                          A paged cache addresses slot = block * block_size
 *                          + offset (reading: slot-major layout).
 *   slot_mapping           DEVICE int64 [num_tokens]: the slot of token t; a
 *                          negative slot is padding and is skipped. A slot at
 *                          or beyond num_slots is skipped and recorded as
 *                          FP8_ERR_ARG (site 401) in the device error word.
 *   k_scale, v_scale       ONE FP32 each in DEVICE memory, positive and finite
 *                          (checked on the device: FP8_ERR_ARG, site 402).
 *   token_elems a positive multiple of 16; num_tokens, num_slots >= 0.
 * Distinct tokens must map to distinct slots (else the last writer is
 * unspecified). Launched as a programmatic dependent; lets nothing launch
 * before it completes.
 * Errors: NULL, SHAPE, ALIGN (data 16 bytes, slot_mapping 8, scales 4),
 * DEVICE, CUDA.
 */
int fp8_kv_cache_store(const void *key_bf16, const void *value_bf16, void *key_cache, void *value_cache,
                       const int64_t *slot_mapping, const float *k_scale, const float *v_scale,
                       int64_t num_tokens, int64_t token_elems, int64_t num_slots, void *stream);

/*
 * FP8 KV cache, load: gathers the cache slots of slot_mapping and
 * dequantizes them to BF16 for attention: x[t][e] = bf16(fl32(dec(cache[slot][e])
 * * scale)). Same arguments and rules as fp8_kv_cache_store, with the caches
 * as inputs and key_bf16 / value_bf16 as outputs; rows of skipped tokens are
 * not written.
 * Errors: NULL, SHAPE, ALIGN, DEVICE, CUDA.
 */
int fp8_kv_cache_load(const void *key_cache, const void *value_cache, void *key_bf16, void *value_bf16,
                      const int64_t *slot_mapping, const float *k_scale, const float *v_scale,
                      int64_t num_tokens, int64_t token_elems, int64_t num_slots, void *stream);

/*
 * W8A8 linear layer, Y = X * W^T, from BF16 activations: dynamic 1x128
 * activation quantization (as fp8_quant_act_group) followed by the
 * block-scaled GEMM (as fp8_block_gemm), dense.
 *
 *   x_bf16  [M][K] BF16, input.
 *   qa      [M][K] E4M3 and sa [K/128][M] FP32: outputs, the activation codes
 *           and scales (caller-owned; bit-identical to fp8_quant_act_group).
 *   qw, sw  as fp8_block_gemm (block_n = block_k = group_k = 128).
 *   y       [M][N] BF16, output.
 *   K a positive multiple of 128 up to FP8_ACT_GROUP_MAX_K, N a positive
 *   multiple of 16, M >= 0.
 * Two launches on `stream`: the quantization kernel, then the decode
 * (M <= 16) or prefill GEMM. The quantization kernel is a programmatic
 * dependent of the work before it, and the GEMM of the quantization kernel:
 * each starts its prologue (and the decode GEMM loads its first weights)
 * while its predecessor finishes, and waits for it before reading its output.
 * Errors: NULL, SHAPE, ALIGN, DEVICE, CUDA.
 */
int fp8_block_linear(const void *x_bf16, void *qa, float *sa, const void *qw, const float *sw,
                     void *y_bf16, int64_t M, int64_t N, int64_t K, void *stream);

/* Static, NUL-terminated description of a status code. Never NULL. */
const char *fp8_status_string(int status);

/*
 * Synchronises `stream`, then reads and clears the current device's error
 * word, which kernels set when a bounded wait expires or a device-checked
 * argument is bad (the first such event since the last read is kept).
 * *out_code receives FP8_OK, FP8_ERR_TIMEOUT or FP8_ERR_ARG; *out_site (may
 * be NULL) a number naming the wait or the check. Returns FP8_OK; FP8_ERR_NULL if out_code is NULL (checked
 * first, on the host); FP8_ERR_DEVICE if the current device is not sm_103;
 * FP8_ERR_CUDA if the synchronisation or the read failed (e.g. an earlier
 * kernel faulted).
 */
int fp8_device_error(void *stream, int *out_code, int *out_site);

/*
 * Self-test of the bounded device waits (a test hook, not part of the
 * computation). Launches on `stream` one CTA of the same wait machinery the
 * GEMM kernels use, with waits that can never complete:
 *  - one thread waits on an mbarrier that nobody arrives at; after the wait
 *    limit (about one second) it records FP8_ERR_TIMEOUT with site 901 in
 *    the device error word and raises the CTA's abort flag;
 *  - a second thread starts its own such wait half a limit later and returns
 *    as soon as it sees the flag, without recording (site 902 would show a
 *    failure to stop).
 * Nothing faults or hangs: the kernel ends about one second after it starts,
 * and the context stays usable. A following fp8_device_error reports
 * FP8_ERR_TIMEOUT and site 901 (and clears them).
 * Errors: DEVICE, CUDA.
 */
int fp8_selftest_bounded_wait(void *stream);

/*
 * Self-test of the E4M3 conversion (a test hook, not part of the computation).
 * Writes to out_e4m3[i], for 0 <= i < n, the code of the FP32 value whose bit
 * pattern is first_bits + i, by the same hardware conversion the quantizers
 * apply to their quotients (round to nearest even, saturating to +-448).
 * Sweeping all 2^32 patterns compares that conversion with an independent
 * encoder on every FP32 value.
 *
 *   out_e4m3  [n] bytes of DEVICE memory, output, 16-byte aligned.
 *   n         a multiple of 8, with first_bits + n <= 2^32.
 * Errors: NULL, SHAPE, ALIGN, DEVICE, CUDA.
 */
int fp8_selftest_encode_f32(uint32_t first_bits, int64_t n, void *out_e4m3, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8W8A8_H */
