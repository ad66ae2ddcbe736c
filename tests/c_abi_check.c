/* A C11 program against include/dvl.h: the header is plain C and the
 * library's host entry points work without C++ or Python.  It calls only
 * functions that need no GPU (the ranks builder, the constants, the
 * argument checks, which fail before anything is enqueued, and the repair
 * step's selection where it selects nothing to copy) and prints
 * "c abi ok". */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "dvl.h"

#define CHECK(cond)                                                   \
    do {                                                              \
        if (!(cond)) {                                                \
            fprintf(stderr, "failed: %s (line %d)\n", #cond, __LINE__); \
            return 1;                                                 \
        }                                                             \
    } while (0)

int main(void)
{
    CHECK(dvl_version() > 0);
    CHECK(strcmp(dvl_status_string(DVL_OK), "") != 0);
    CHECK(dvl_workspace_bytes(1, 1) >= 512);
    CHECK(dvl_workspace_bytes(DVL_MAX_M + 1, 1) == 0);

    /* ranks builder: histogram, top-N after a forced set, union */
    const int32_t tokens[] = {3, 1, 3, 2, 3, 1, 7, 7, 7, 7};
    int64_t counts[8] = {0};
    CHECK(dvl_histogram(tokens, 10, 8, counts) == DVL_OK);
    CHECK(counts[7] == 4 && counts[3] == 3 && counts[1] == 2 && counts[2] == 1);
    const int32_t forced[] = {0};
    int32_t ranks[8];
    int32_t n = 0;
    CHECK(dvl_build_ranks(counts, 8, forced, 1, 4, 0, ranks, &n) == DVL_OK);
    CHECK(n == 4 && ranks[0] == 0 && ranks[1] == 7 && ranks[2] == 3 && ranks[3] == 1);
    const int32_t a[] = {1, 4, 6}, b[] = {2, 4, 9};
    int32_t u[6];
    CHECK(dvl_union_sorted(a, 3, b, 3, u, &n) == DVL_OK);
    CHECK(n == 5 && u[0] == 1 && u[1] == 2 && u[2] == 4 && u[3] == 6 && u[4] == 9);

    /* argument checks return before any launch */
    dvl_head head;
    memset(&head, 0, sizeof head);
    head.dtype = DVL_BF16;
    head.N = 100;
    head.K = 256;
    head.V = 100;
    head.w = (const void *)(uintptr_t)0x1000;
    int32_t ids[1];
    float logit[1];
    CHECK(dvl_draft_argmax(NULL, (const void *)(uintptr_t)0x3000, 1, ids, logit,
                           (void *)(uintptr_t)0x5000, 1 << 20, NULL) == DVL_ERR_INVALID_ARG);
    CHECK(dvl_draft_argmax(&head, (const void *)(uintptr_t)0x3000, 0, ids, logit,
                           (void *)(uintptr_t)0x5000, 1 << 20, NULL) == DVL_ERR_INVALID_ARG);
    head.dtype = 9;
    CHECK(dvl_score_ids(&head, (const void *)(uintptr_t)0x3000, 1,
                        (const int32_t *)(uintptr_t)0x2000, 4, logit, NULL) == DVL_ERR_INVALID_ARG);
    uint32_t bits = 0;
    CHECK(dvl_workspace_status(NULL, &bits, NULL) == DVL_ERR_INVALID_ARG);
    CHECK(dvl_noalloc_status(NULL, NULL) == DVL_ERR_INVALID_ARG);

    /* the repair step: ids already in the list, or no spare row left, copy
     * nothing (so nothing is enqueued and no GPU is needed) */
    head.dtype = DVL_BF16;
    int32_t row_of[100];
    for (int i = 0; i < 100; ++i)
        row_of[i] = -1;
    row_of[5] = 0;
    row_of[9] = 1;
    int32_t rows = 2, learned[4], nl = -1;
    const int32_t present[] = {9, 5, 9};
    void *wt = (void *)(uintptr_t)0x1000;
    int32_t *d2t = (int32_t *)(uintptr_t)0x2000;
    CHECK(dvl_learn_missing(&head, present, 3, row_of, &rows, 8, wt, NULL, d2t, learned, &nl,
                            NULL) == DVL_OK);
    CHECK(nl == 0 && rows == 2);
    const int32_t fresh[] = {7, 7, 3};
    CHECK(dvl_learn_missing(&head, fresh, 3, row_of, &rows, 2, wt, NULL, d2t, learned, &nl,
                            NULL) == DVL_OK);
    CHECK(nl == 0 && rows == 2 && row_of[7] == -1 && row_of[3] == -1);
    const int32_t outside[] = {7, 100};
    CHECK(dvl_learn_missing(&head, outside, 2, row_of, &rows, 8, wt, NULL, d2t, learned, &nl,
                            NULL) == DVL_ERR_OUT_OF_RANGE);
    CHECK(row_of[7] == -1 && rows == 2);
    CHECK(dvl_learn_missing(&head, fresh, 3, row_of, &rows, 1, wt, NULL, d2t, learned, &nl,
                            NULL) == DVL_ERR_INVALID_ARG); /* capacity below the rows in use */
    printf("c abi ok\n");
    return 0;
}
