/* A plain C99 caller of the library: include/dfl.h compiles as C with
 * -pedantic, and the host-only calls link and answer without a GPU. */
#include "dfl.h"

#include <stdio.h>
#include <string.h>

static int fails = 0;
#define CHECK(c)                                                   \
    do {                                                           \
        if (!(c)) {                                                \
            fprintf(stderr, "check failed: %s (line %d)\n", #c, __LINE__); \
            ++fails;                                               \
        }                                                          \
    } while (0)

int main(void) {
    dfl_shape s;
    size_t one, two;
    memset(&s, 0, sizeof s);
    s.N = 2; s.C = 64; s.B = 16; s.d = 256; s.Hq = 4; s.Hkv = 4; s.hd = 64;
    s.D = 1; s.L = 3; s.V = 1000; s.G = 15; s.row0 = 1; s.dtype = DFL_BF16;

    CHECK(strncmp(dfl_version(), "dfl", 3) == 0);
    CHECK(strcmp(dfl_status_string(DFL_OK), "ok") == 0);
    CHECK(strstr(dfl_status_string(DFL_ERR_WORKSPACE), "workspace") != NULL);

    one = dfl_workspace_size(DFL_OP_DRAFT_STEP, &s);
    s.D = 2;
    two = dfl_workspace_size(DFL_OP_DRAFT_STEP, &s);
    CHECK(one > 0 && two > one);   /* one more layer's mixed context features */

    /* argument checks answer on the host, before any device is touched */
    CHECK(dfl_greedy_accept(NULL, NULL, 1, 4, NULL, NULL, NULL) == DFL_ERR_INVALID_ARG);
    CHECK(dfl_draft_step(NULL, NULL, 0, NULL) == DFL_ERR_INVALID_ARG);
    CHECK(dfl_draft_step_host(NULL, NULL, 1, NULL, 0, NULL) == DFL_ERR_INVALID_ARG);
    CHECK(dfl_set_wait_limit_ns(0) == DFL_ERR_INVALID_ARG);

    if (fails == 0) printf("ok\n");
    return fails == 0 ? 0 : 1;
}
