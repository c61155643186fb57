/* A plain C caller of the library's host-only entry points (no GPU needed): the tile layout
 * of a small 2D Laplacian, the panel SpMV's plan check, the reuse-interval choice of a
 * decision log, and an error path with its message. Prints one line per result; exits
 * non-zero on the first unexpected status. Built and run by tests/test_c_abi.py. */
#include <stdio.h>
#include <stdlib.h>

#include "evocg.h"

static int check(int st, int want, const char *what)
{
    if (st != want) {
        printf("FAIL %s: status %d (%s)\n", what, st, evocg_last_error());
        return 1;
    }
    return 0;
}

int main(void)
{
    /* 5-point Laplacian on a 20 x 20 grid, natural order */
    const int nx = 20, n = nx * nx;
    int64_t *rp = malloc(sizeof(int64_t) * (n + 1));
    int32_t *ci = malloc(sizeof(int32_t) * 5 * n);
    double *v = malloc(sizeof(double) * 5 * n);
    int64_t nnz = 0;
    rp[0] = 0;
    for (int i = 0; i < n; ++i) {
        const int x = i % nx, y = i / nx;
        if (y > 0) { ci[nnz] = i - nx; v[nnz++] = -1.0; }
        if (x > 0) { ci[nnz] = i - 1; v[nnz++] = -1.0; }
        ci[nnz] = i; v[nnz++] = 4.0;
        if (x < nx - 1) { ci[nnz] = i + 1; v[nnz++] = -1.0; }
        if (y < nx - 1) { ci[nnz] = i + nx; v[nnz++] = -1.0; }
        rp[i + 1] = nnz;
    }
    int64_t ntiles = 0, nslots = 0;
    if (check(evocg_tile_layout_host(n, rp, ci, v, 16, &ntiles, &nslots, NULL, NULL, NULL,
                                     NULL, NULL, NULL, NULL, NULL, NULL, NULL),
              EVOCG_OK, "layout sizes"))
        return 1;
    const int64_t nrb = (n + 15) / 16;
    int64_t *trp = malloc(sizeof(int64_t) * (nrb + 1));
    uint64_t *mask = malloc(sizeof(uint64_t) * ntiles);
    uint8_t *width = malloc((size_t)ntiles);
    if (check(evocg_tile_layout_host(n, rp, ci, v, 16, NULL, NULL, trp, NULL, NULL, mask,
                                     width, NULL, NULL, NULL, NULL, NULL),
              EVOCG_OK, "layout arrays"))
        return 1;
    int64_t rows_in_masks = 0, widest = 0;
    for (int64_t t = 0; t < ntiles; ++t) {
        for (int b = 0; b < 16; ++b) rows_in_masks += (mask[t] >> b) & 1u;
        if (width[t] > widest) widest = width[t];
    }
    printf("layout ntiles %lld nslots %lld nnz %lld tiles_in_last_rowblock %lld widest %lld\n",
           (long long)ntiles, (long long)nslots, (long long)nnz,
           (long long)(trp[nrb] - trp[nrb - 1]), (long long)widest);
    printf("rows_in_masks %lld\n", (long long)rows_in_masks);

    int64_t nb = 0;
    int ok = 0;
    if (check(evocg_panel_plan_host(n, rp, ci, v, 16, 8, 4096, &nb, &ok), EVOCG_OK, "plan"))
        return 1;
    printf("plan batches %lld valid %d\n", (long long)nb, ok);

    /* one block, 8 iterations: up at k = 3 (2 -> 1) and k = 5 (1 -> 0) */
    const uint8_t log[8] = {2, 2, 2, 1, 1, 0, 0, 0};
    int kstar = 0, ncand = 0;
    double frac[8];
    if (check(evocg_kstar_select(log, 8, 1, 0.1, &kstar, frac, 8, &ncand), EVOCG_OK, "kstar"))
        return 1;
    printf("kstar %d candidates %d frac %.3f %.3f %.3f %.3f\n", kstar, ncand, frac[0], frac[1],
           frac[2], frac[3]);

    /* tile size 24 is not supported: EINVAL with a message */
    if (check(evocg_tile_layout_host(n, rp, ci, v, 24, &ntiles, &nslots, NULL, NULL, NULL,
                                     NULL, NULL, NULL, NULL, NULL, NULL, NULL),
              EVOCG_EINVAL, "bad tile size"))
        return 1;
    printf("error %s\n", evocg_last_error());
    free(rp); free(ci); free(v); free(trp); free(mask); free(width);
    return 0;
}
