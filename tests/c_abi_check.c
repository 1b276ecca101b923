/* c_abi_check.c -- a plain C99 caller of libmoe4.so (built and run by tests/test_abi.py).
 *
 * It shows that include/moe4.h is a C header (no C++ needed to call the library) and exercises
 * the calls that need no GPU: the library queries and the host-side argument checks, which
 * return before anything is enqueued.  Prints "ok" and exits 0 when every check holds. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "moe4.h"

#define CHECK(cond)                                                  \
    do {                                                             \
        if (!(cond)) {                                               \
            fprintf(stderr, "failed: %s (line %d)\n", #cond, __LINE__); \
            return 1;                                                \
        }                                                            \
    } while (0)

int main(void) {
    /* an address that is 16-byte aligned and never dereferenced: every call below fails its
       host-side checks first */
    void *fake = (void *)(uintptr_t)(1u << 20);
    CHECK(moe4_version() >= 100);
    CHECK(strcmp(moe4_status_string(MOE4_OK), "ok") == 0);
    CHECK(moe4_status_string(12345) != NULL);
    CHECK(moe4_workspace_size(MOE4_OP_NVFP4_QUANTIZE, 384, 0, 0) == 384 * sizeof(unsigned int));
    /* cols % 16 != 0 */
    CHECK(nvfp4_quantize((const uint16_t *)fake, 1, 16, 15, 16, (uint8_t *)fake, (uint8_t *)fake,
                         (float *)fake, NULL, MOE4_FOUR_OVER_SIX, fake, 64, NULL) == MOE4_ERR_ARG);
    /* no workspace for the amax pass */
    CHECK(nvfp4_quantize((const uint16_t *)fake, 1, 16, 16, 16, (uint8_t *)fake, (uint8_t *)fake,
                         (float *)fake, NULL, MOE4_FOUR_OVER_SIX, NULL, 0, NULL) == MOE4_ERR_WORKSPACE);
    /* rows % 32 != 0 */
    CHECK(mxfp8_requant_transpose_sr((const uint8_t *)fake, (const uint8_t *)fake, (const float *)fake, 1, 48,
                                     64, (uint8_t *)fake, (uint8_t *)fake, 0, 0, MOE4_SR, NULL) == MOE4_ERR_ARG);
    /* rows_total % 128 != 0 */
    CHECK(grouped_expert_gemm_nvfp4((const uint8_t *)fake, (const uint8_t *)fake, (const float *)fake,
                                    (const uint8_t *)fake, (const uint8_t *)fake, (const float *)fake,
                                    (const int32_t *)fake, 1, 100, 256, 256, fake, MOE4_OUT_BF16, NULL, 0,
                                    NULL) == MOE4_ERR_ARG);
    /* cols % 128 != 0 */
    CHECK(hadamard_quant((const uint16_t *)fake, 4, 64, (uint8_t *)fake, (uint8_t *)fake, (float *)fake,
                         MOE4_FOUR_OVER_SIX, fake, 4, NULL) == MOE4_ERR_ARG);
    printf("ok\n");
    return 0;
}
