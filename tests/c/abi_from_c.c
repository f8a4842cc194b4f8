/*
 * A plain C99 caller of the library's C ABI (include/tnd_attn.h): the header
 * must compile as C with every warning on, and the first-phase calls, the
 * status strings, the options and the plan must work from C without a GPU.
 * Prints "ok" and exits 0 when every check holds; otherwise names the check.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "tnd_attn.h"

#define CHECK(cond)                                                  \
    do {                                                             \
        if (!(cond)) {                                               \
            printf("failed: %s (line %d)\n", #cond, __LINE__);       \
            return 1;                                                \
        }                                                            \
    } while (0)

int main(void)
{
    /* two sequences of 300 and 190 rows, causal, 4 query heads on 2 kv heads */
    const int64_t cu[3] = {0, 300, 490};
    const int64_t inf = 2147483647;
    uint64_t ws = 0, ws_dv = 0;
    CHECK(tnd_attn_grad_workspace_size(TND_BF16, 2, cu, cu, NULL, 4, 2, 128, 128, 0.088, 1.0, inf, inf, 3, 0, 0,
                                       0, &ws) == TND_OK);
    CHECK(ws > 0);
    /* a value head dim below the query / key one runs on the CUDA-core kernels */
    CHECK(tnd_attn_grad_workspace_size(TND_BF16, 2, cu, cu, NULL, 4, 2, 128, 64, 0.088, 1.0, inf, inf, 3, 0, 0,
                                       0, &ws_dv) == TND_OK);
    CHECK(ws_dv > 0 && ws_dv < ws);
    CHECK(tnd_attn_fwd_workspace_size(TND_F32, 2, cu, cu, NULL, 4, 2, 64, 64, 0.125, 1.0, inf, inf, 0, 0, 0, 0,
                                      &ws) == TND_OK);
    /* argument errors come back before any device work */
    CHECK(tnd_attn_grad_workspace_size(TND_BF16, 2, cu, cu, NULL, 3, 2, 128, 128, 0.088, 1.0, inf, inf, 3, 0, 0,
                                       0, &ws) == TND_ERR_INVALID);
    CHECK(tnd_attn_grad_workspace_size(TND_BF16, 2, cu, cu, NULL, 4, 2, 128, 129, 0.088, 1.0, inf, inf, 3, 0, 0,
                                       0, &ws) == TND_ERR_INVALID);
    CHECK(tnd_attn_grad_workspace_size(TND_BF16, 2, NULL, cu, NULL, 4, 2, 128, 128, 0.088, 1.0, inf, inf, 3, 0,
                                       0, 0, &ws) == TND_ERR_NULLPTR);
    CHECK(tnd_attn_grad_workspace_size(TND_BF16, 2, cu, cu, NULL, 4, 2, 128, 128, 0.088, 1.0, inf, inf, 7, 0, 0,
                                       0, &ws) == TND_ERR_UNSUPPORTED);
    CHECK(tnd_attn_grad(NULL, NULL, NULL, NULL, NULL, 0, 1, NULL, NULL, NULL, NULL, NULL, NULL, TND_BF16, 2, cu, cu,
                        NULL, 4, 2, 128, 128, 0.088, 1.0, inf, inf, 3, NULL, NULL, NULL, NULL, NULL, 0, NULL) ==
          TND_ERR_NULLPTR);
    /* status strings and options */
    CHECK(strcmp(tnd_status_string((tnd_status)99), "unknown status") == 0);
    CHECK(tnd_status_string(TND_ERR_DEVICE_TIMEOUT)[0] != '\0');
    CHECK(tnd_attn_set_option(TND_OPT_DETERMINISTIC, 2) == TND_ERR_INVALID);
    CHECK(tnd_attn_set_option(TND_OPT_DETERMINISTIC, 1) == TND_OK);
    /* the gradient plan: every unit lies inside its sequence */
    int64_t units[4096 * 5];
    int64_t n_units = 0, kept = 0;
    CHECK(tnd_attn_grad_plan(2, cu, cu, NULL, 4, 2, inf, inf, 3, 0, units, 4096, &n_units, &kept) == TND_OK);
    CHECK(n_units > 0 && n_units <= 4096);
    for (int64_t u = 0; u < n_units; ++u) {
        const int64_t *e = units + 5 * u;
        const int64_t rows = cu[e[0] + 1] - cu[e[0]];
        CHECK(e[0] >= 0 && e[0] < 2 && e[1] >= 0 && e[1] < 2);
        CHECK(e[2] >= 0 && e[2] * 128 < rows);
        CHECK(e[3] >= 0 && e[3] <= e[4] && (e[4] - 1) * 128 < rows);
    }
    /* causal: 300*301/2 + 190*191/2 kept pairs per query head */
    CHECK(kept == 4 * (300 * 301 / 2 + 190 * 191 / 2));
    printf("ok\n");
    return 0;
}
