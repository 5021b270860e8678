/*
 * A plain C11 client of include/fp8bs.h, linked against libfp8bs.so.
 *
 * Compiling it checks that the header is valid C and that every prototype
 * resolves to an exported symbol at link time (-Wl,--no-undefined on a
 * program that takes the address of every entry point); running it checks
 * each entry point's argument validation through the real C calling
 * convention.  Every call here is refused before the library touches CUDA,
 * so no GPU is needed.  Prints "checks <n> failures <f>" and exits non-zero
 * on any failure.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "fp8bs.h"

static int checks, failures;

static void expect(int got, int want, const char *what, int line)
{
    ++checks;
    if (got != want) {
        ++failures;
        printf("FAIL line %d: %s returned %d, expected %d\n", line, what, got, want);
    }
}
#define EXPECT(call, want) expect((call), (want), #call, __LINE__)

/* fake, never dereferenced device addresses */
#define A(v) ((void *)(uintptr_t)(v))

int main(void)
{
    /* every entry point, by address: a missing export fails the link */
    void (*const entry_points[])(void) = {
        (void (*)(void))fp8bs_quantize,        (void (*)(void))fp8bs_gemv,
        (void (*)(void))fp8bs_gemv_ex,         (void (*)(void))fp8bs_gemv_batch,
        (void (*)(void))fp8bs_gemv_ws,         (void (*)(void))fp8bs_gemv_ws_bytes,
        (void (*)(void))fp8bs_gemv_batch_ex,   (void (*)(void))mxfp8_quantize,
        (void (*)(void))mxfp8_gemv,            (void (*)(void))mxfp8_gemv_ex,
        (void (*)(void))mxfp8_gemv_batch,      (void (*)(void))mxfp8_gemv_batch_ex,
        (void (*)(void))fp8row_quantize,       (void (*)(void))fp8tensor_quantize,
        (void (*)(void))fp8row_gemv,           (void (*)(void))fp8row_gemv_ex,
        (void (*)(void))fp8tensor_gemv,        (void (*)(void))fp8tensor_gemv_ex,
        (void (*)(void))fp8bs_moe_gemv,        (void (*)(void))fp8kv_append,
        (void (*)(void))fp8kv_decode_attention, (void (*)(void))fp8act_quantize,
        (void (*)(void))w8a8_gemm,             (void (*)(void))w8a8_gemm_ex,
        (void (*)(void))fp8bs_select_path,     (void (*)(void))fp8bs_strerror,
        (void (*)(void))fp8bs_check_device_error, (void (*)(void))fp8bs_debug_wait_expiry,
        (void (*)(void))fp8bs_debug_encode_f32, (void (*)(void))fp8bs_version,
    };
    for (size_t i = 0; i < sizeof entry_points / sizeof entry_points[0]; ++i) {
        ++checks;
        if (!entry_points[i]) {
            ++failures;
            printf("FAIL: entry point %zu has no address\n", i);
        }
    }

    EXPECT(fp8bs_version(), 106);
    for (int st = FP8BS_ERR_PATH; st <= FP8BS_OK; ++st) {
        const char *s = fp8bs_strerror(st);
        ++checks;
        if (!s || !strcmp(s, "unknown status")) {
            ++failures;
            printf("FAIL: no text for status %d\n", st);
        }
    }

    const void *w = A(0x10000), *x = A(0x10000);
    uint8_t *c = (uint8_t *)A(0x20000);
    float *s = (float *)A(0x30000);
    void *y = A(0x40000);

    /* quantizers */
    EXPECT(fp8bs_quantize(w, 0, 10, 128, c, s, NULL), FP8BS_ERR_SHAPE);
    EXPECT(fp8bs_quantize(w, 10, 10, 64, c, s, NULL), FP8BS_ERR_BLOCK);
    EXPECT(fp8bs_quantize(NULL, 10, 10, 128, c, s, NULL), FP8BS_ERR_NULL);
    EXPECT(fp8bs_quantize(A(0x10001), 10, 10, 128, c, s, NULL), FP8BS_ERR_ALIGN);
    EXPECT(mxfp8_quantize(w, 10, 0, c, c, NULL), FP8BS_ERR_SHAPE);
    EXPECT(mxfp8_quantize(w, 10, 10, c, NULL, NULL), FP8BS_ERR_NULL);
    EXPECT(fp8row_quantize(w, 10, 10, c, A(0x30002), NULL), FP8BS_ERR_ALIGN);
    EXPECT(fp8tensor_quantize(w, -1, 10, c, s, NULL), FP8BS_ERR_SHAPE);
    EXPECT(fp8act_quantize(NULL, 1, 10, c, s, NULL), FP8BS_ERR_NULL);

    /* GEMVs: m == 0 is a no-op, shapes, pointers, alignment, paths */
    EXPECT(fp8bs_gemv(NULL, 0, NULL, NULL, 10, 10, NULL, NULL), FP8BS_OK);
    EXPECT(fp8bs_gemv(x, -1, c, s, 10, 10, y, NULL), FP8BS_ERR_SHAPE);
    EXPECT(fp8bs_gemv(x, 1, c, s, (int64_t)1 << 31, 10, y, NULL), FP8BS_ERR_SHAPE);
    EXPECT(fp8bs_gemv(x, 1, c, NULL, 10, 10, y, NULL), FP8BS_ERR_NULL);
    EXPECT(fp8bs_gemv(x, 1, c, A(0x30002), 10, 10, y, NULL), FP8BS_ERR_ALIGN);
    EXPECT(fp8bs_gemv_ex(x, 1, c, s, 10, 10, y, 9, NULL), FP8BS_ERR_PATH);
    EXPECT(fp8bs_gemv_ex(x, 1, c, s, 10, 10, y, FP8BS_PATH_DECODE, NULL), FP8BS_ERR_PATH);
    EXPECT(mxfp8_gemv(x, 1, c, NULL, 10, 32, y, NULL), FP8BS_ERR_NULL);
    EXPECT(mxfp8_gemv_ex(x, 40, c, c, 10, 24, y, FP8BS_PATH_PREFILL, NULL), FP8BS_ERR_PATH);
    EXPECT(fp8row_gemv(x, 1, c, s, 0, 10, y, NULL), FP8BS_ERR_SHAPE);
    EXPECT(fp8row_gemv_ex(x, 40, c, s, 10, 24, y, FP8BS_PATH_PREFILL, NULL), FP8BS_ERR_PATH);
    EXPECT(fp8tensor_gemv(x, 1, NULL, s, 10, 10, y, NULL), FP8BS_ERR_NULL);
    EXPECT(fp8tensor_gemv_ex(x, 1, c, s, 10, 10, y, -1, NULL), FP8BS_ERR_PATH);

    /* caller-provided workspace (decode path) */
    const int64_t need = fp8bs_gemv_ws_bytes(16, 4096);
    EXPECT(need == 2 * 16 * 4096 + 128 * 32, 1);
    EXPECT((int)fp8bs_gemv_ws_bytes(-1, 4096), FP8BS_ERR_SHAPE);
    EXPECT(fp8bs_gemv_ws(x, 16, c, s, 256, 4096, y, NULL, need, NULL), FP8BS_ERR_NULL);
    EXPECT(fp8bs_gemv_ws(x, 16, c, s, 256, 4096, y, A(0x50008), need, NULL), FP8BS_ERR_ALIGN);
    EXPECT(fp8bs_gemv_ws(x, 16, c, s, 256, 4096, y, A(0x50000), need - 1, NULL), FP8BS_ERR_SHAPE);

    /* batches: validated op by op before anything is launched */
    fp8bs_gemv_op ops[2] = {
        {x, c, s, y, 128, 256},
        {x, c, s, y, 128, 256},
    };
    EXPECT(fp8bs_gemv_batch(NULL, 0, 1, NULL), FP8BS_OK);
    EXPECT(fp8bs_gemv_batch(NULL, 2, 1, NULL), FP8BS_ERR_NULL);
    EXPECT(fp8bs_gemv_batch(ops, -1, 1, NULL), FP8BS_ERR_SHAPE);
    ops[1].k = 0;
    EXPECT(fp8bs_gemv_batch(ops, 2, 1, NULL), FP8BS_ERR_SHAPE);
    EXPECT(mxfp8_gemv_batch(ops, 2, 0, NULL), FP8BS_ERR_SHAPE);  /* shapes are checked even at m == 0 */
    ops[1].k = 200;
    EXPECT(fp8bs_gemv_batch_ex(ops, 2, 1, FP8BS_PATH_DECODE, NULL), FP8BS_ERR_PATH);
    ops[1].k = 256;
    ops[1].scales = A(0x30002);
    EXPECT(fp8bs_gemv_batch(ops, 2, 1, NULL), FP8BS_ERR_ALIGN);
    ops[1].k = 200;
    EXPECT(mxfp8_gemv_batch_ex(ops, 2, 40, FP8BS_PATH_PREFILL, NULL), FP8BS_ERR_PATH);

    /* W8A8, MoE, KV cache */
    EXPECT(w8a8_gemm(c, 1, s, c, NULL, 10, 10, y, NULL), FP8BS_ERR_NULL);
    EXPECT(w8a8_gemm_ex(c, 1, s, c, s, 10, 24, y, FP8BS_PATH_DECODE, NULL), FP8BS_ERR_PATH);
    EXPECT(fp8bs_moe_gemv(x, 1, (const int32_t *)A(0x50000), 0, c, s, 8, 128, 128, y, NULL), FP8BS_ERR_SHAPE);
    EXPECT(fp8bs_moe_gemv(x, 1, NULL, 2, c, s, 8, 128, 128, y, NULL), FP8BS_ERR_NULL);
    EXPECT(fp8bs_moe_gemv(x, 1, (const int32_t *)A(0x50000), 2, c, s, 8, 128, 120, y, NULL), FP8BS_ERR_PATH);
    EXPECT(fp8kv_append(x, 4, 8, 64, (const int32_t *)A(0x50000), s, c, 1024, NULL), FP8BS_ERR_SHAPE);
    EXPECT(fp8kv_append(A(0x10008), 4, 8, 128, (const int32_t *)A(0x50000), s, c, 1024, NULL), FP8BS_ERR_ALIGN);
    EXPECT(fp8kv_decode_attention(x, c, c, s, s, (const int32_t *)A(0x50000), 4, (const int32_t *)A(0x60000), 2,
                                  32, 8, 64, 16, 64, 64, 0.088f, y, NULL),
           FP8BS_ERR_SHAPE);
    EXPECT(fp8kv_decode_attention(NULL, c, c, s, s, (const int32_t *)A(0x50000), 4, (const int32_t *)A(0x60000), 2,
                                  32, 8, 128, 16, 64, 64, 0.088f, y, NULL),
           FP8BS_ERR_NULL);

    /* host-only helpers */
    EXPECT(fp8bs_select_path(1, 100, 4096, A(0x10000), A(0x20000), 0), FP8BS_PATH_DECODE);
    EXPECT(fp8bs_select_path(33, 100, 4096, A(0x10000), A(0x20000), 0), FP8BS_PATH_PREFILL);
    EXPECT(fp8bs_select_path(1, 100, 4100, A(0x10000), A(0x20000), 0), FP8BS_PATH_GENERIC);
    EXPECT(fp8bs_select_path(0, 100, 4096, A(0x10000), A(0x20000), 0), FP8BS_ERR_SHAPE);
    EXPECT(fp8bs_debug_encode_f32(0, 6, c, NULL), FP8BS_ERR_SHAPE);
    EXPECT(fp8bs_debug_encode_f32(0, 16, NULL, NULL), FP8BS_ERR_NULL);

    printf("checks %d failures %d\n", checks, failures);
    return failures != 0;
}
