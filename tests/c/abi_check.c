/* Plain C99 user of include/tcgemm.h: compiled and run by tests/test_abi_cpu.py
 * with gcc against libtcgemm.so, on a machine without a GPU.  It calls only
 * the entry points that validate arguments or size workspaces (no launch),
 * and exits non-zero on the first unexpected result. */
#include <stdio.h>
#include <stdint.h>
#include "tcgemm.h"

#define CHECK(cond)                                                    \
    do {                                                               \
        if (!(cond)) {                                                 \
            fprintf(stderr, "%s:%d: check failed: %s\n", __FILE__,     \
                    __LINE__, #cond);                                  \
            return 1;                                                  \
        }                                                              \
    } while (0)

int main(void) {
    /* fake, aligned device addresses: validation never dereferences them */
    const void* A = (const void*)(uintptr_t)0x10000;
    const void* B = (const void*)(uintptr_t)0x20000;
    const void* C = (const void*)(uintptr_t)0x30000;
    void* D = (void*)(uintptr_t)0x40000;
    tcg_epilogue epi = {NULL, TCG_BF16, TCG_ACT_GELU};

    CHECK(tcg_can_implement(300, 200, 128, TCG_BF16, A, 128, TCG_ROW, B, 128, TCG_COL, 1, C, 200, TCG_BF16,
                            D, 200, TCG_BF16, epi) == TCG_OK);
    CHECK(tcg_can_implement(-1, 200, 128, TCG_BF16, A, 128, TCG_ROW, B, 128, TCG_COL, 0, NULL, 0, TCG_BF16,
                            D, 200, TCG_BF16, epi) == TCG_ERR_INVALID_ARG);
    CHECK(tcg_can_implement(300, 200, 128, TCG_E4M3, A, 300, TCG_COL, B, 128, TCG_COL, 0, NULL, 0, TCG_BF16,
                            D, 200, TCG_BF16, epi) == TCG_ERR_UNSUPPORTED);
    CHECK(tcg_can_implement(300, 200, 128, TCG_BF16, (const char*)A + 1, 128, TCG_ROW, B, 128, TCG_COL, 0,
                            NULL, 0, TCG_BF16, D, 200, TCG_BF16, epi) == TCG_ERR_MISALIGNED);
    CHECK(tcg_workspace_size(8192, 8192, 8192, TCG_BF16) >= 256);
    CHECK(tcg_workspace_size(-1, 1, 1, TCG_BF16) == 0);
    CHECK(tcg_workspace_size_for(300, 200, 129, TCG_BF16, A, 129, TCG_ROW, B, 129, TCG_COL) >
          tcg_workspace_size(300, 200, 129, TCG_BF16));
    CHECK(tcg_grouped_workspace_size(16) > tcg_grouped_workspace_size(1));

    tcg_problem probs[2] = {
        {300, 200, 128, 1.0f, A, 128, B, 128, NULL, 0, D, 200, NULL},
        {0, 64, 64, 1.0f, A, 64, B, 64, NULL, 0, D, 64, NULL},
    };
    probs[1].lda = 63; /* empty problem: never checked against K */
    CHECK(tcg_gemm_grouped(2, probs, TCG_ROW, TCG_COL, 0.0f, TCG_BF16, TCG_BF16, epi, TCG_MXE4M3, NULL, 0,
                           NULL) == TCG_ERR_UNSUPPORTED);
    probs[0].lda = 100; /* lda < K */
    CHECK(tcg_gemm_grouped(2, probs, TCG_ROW, TCG_COL, 0.0f, TCG_BF16, TCG_BF16, epi, TCG_BF16, NULL, 0,
                           NULL) == TCG_ERR_INVALID_ARG);

    int rows[10 * 64];
    const int n = tcg_debug_schedule(4096, 4096, 4096, TCG_BF16, 152, 0, rows, 64);
    CHECK(n > 0);
    printf("abi_check ok: %d units in the 4096^3 schedule, %s\n", n, tcg_last_error());
    return 0;
}
