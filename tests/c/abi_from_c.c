/* Uses the library through include/dflash2.h from plain C (C99): only calls that need no GPU.
 * Exit status 0 when every check holds; prints the first failing check otherwise. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "dflash2.h"

#define CHECK(cond)                                                  \
    do {                                                             \
        if (!(cond)) {                                               \
            fprintf(stderr, "check failed: %s (line %d)\n", #cond, __LINE__); \
            return 1;                                                \
        }                                                            \
    } while (0)

int main(void)
{
    df2_dims d = {1, 16, 4096, 151936, 8, 256};
    CHECK(dflash2_version() >= 300);
    CHECK(strcmp(dflash2_status_string(DF2_OK), "ok") == 0);
    CHECK(strlen(dflash2_status_string(DF2_ERR_TIMEOUT)) > 2);

    const size_t ws = dflash2_workspace_bytes(&d);
    CHECK(ws > 0 && ws % 256 == 0);
    CHECK(dflash2_select_host_workspace_bytes(&d) > ws);

    df2_dims bad = d;
    bad.k = 33;
    CHECK(dflash2_workspace_bytes(&bad) == 0);

    /* argument checks run before any CUDA call: these pointers are never dereferenced */
    void *p = (void *)(uintptr_t)0x200000;
    CHECK(dflash2_select(NULL, p, p, p, p, p, (const int32_t *)p, (float *)p, (int32_t *)p, NULL, NULL, NULL,
                         (void *)(uintptr_t)0x100000, ws, NULL) == DF2_ERR_INVALID_ARG);
    CHECK(dflash2_select(&bad, p, p, p, p, p, (const int32_t *)p, (float *)p, (int32_t *)p, NULL, NULL, NULL,
                         (void *)(uintptr_t)0x100000, ws, NULL) == DF2_ERR_UNSUPPORTED);
    CHECK(dflash2_select(&d, p, p, p, p, p, (const int32_t *)p, (float *)p, (int32_t *)p, NULL, NULL, NULL,
                         (void *)(uintptr_t)0x100000, ws - 256, NULL) == DF2_ERR_WORKSPACE);
    /* the walk options are checked before anything else of the call */
    df2_walk_opts w = {0.0f, 0.5f, NULL, NULL, NULL};
    CHECK(dflash2_select_walk(&d, &w, p, p, p, p, p, (const int32_t *)p, (float *)p, (int32_t *)p, NULL, NULL, NULL,
                              (void *)(uintptr_t)0x100000, ws, NULL) == DF2_ERR_INVALID_ARG);
    w.temperature = 1.0f;
    CHECK(dflash2_select_walk(&d, &w, p, p, p, p, p, (const int32_t *)p, (float *)p, (int32_t *)p, NULL, NULL, NULL,
                              (void *)(uintptr_t)0x100000, ws - 256, NULL) == DF2_ERR_WORKSPACE);
    CHECK(dflash2_selftest_wait_timeout(0, (void *)(uintptr_t)0x100000, ws, NULL) == DF2_ERR_INVALID_ARG);
    CHECK(dflash2_profile_events(p, NULL) == DF2_ERR_INVALID_ARG);
    printf("ok\n");
    return 0;
}
