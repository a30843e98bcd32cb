/* A plain C99 consumer of include/gsa.h, linked against the in-tree
 * libgsa.so: host-side calls only (layout queries, workspace sizes, status
 * strings, argument errors), so it runs without a GPU.  Prints one line per
 * check and exits non-zero on the first failure. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "gsa.h"

static int fail(const char *what) {
    printf("FAIL %s\n", what);
    return 1;
}

int main(void) {
    const int64_t split[4] = {64, 128, 32, 96};
    gsa_layout_info info;
    int64_t doff[5], soff[5];
    /* MXFP8, width 256: 320 rows, 32-row blocks */
    if (gsa_layout(4, split, 256, GSA_MXFP8, &info, doff, soff) != GSA_OK) return fail("gsa_layout mxfp8");
    if (info.rows != 320 || info.row_data_bytes != 320 * 256 || info.row_scale_bytes != 320 * 256 / 32)
        return fail("mxfp8 rowwise sizes");
    if (doff[0] != 0 || doff[1] != 256 * 64 || doff[4] != info.col_data_bytes) return fail("mxfp8 column offsets");
    printf("ok gsa_layout mxfp8 rows=%lld col_data=%lld\n", (long long)info.rows, (long long)info.col_data_bytes);
    /* NVFP4: two codes per byte, E4M3 scales per 16, one amax per expert */
    if (gsa_layout(4, split, 256, GSA_NVFP4, &info, NULL, NULL) != GSA_OK) return fail("gsa_layout nvfp4");
    if (info.row_data_bytes != 320 * 128 || info.row_scale_bytes != 320 * 16 || info.amax_floats != 4)
        return fail("nvfp4 sizes");
    printf("ok gsa_layout nvfp4 amax_floats=%lld\n", (long long)info.amax_floats);
    /* workspace sizes are positive multiples of 256 bytes */
    {
        size_t ws = gsa_workspace_size(4, split, 256, GSA_ACT_SRELU, GSA_NVFP4);
        if (ws == 0 || ws % 256 != 0) return fail("gsa_workspace_size");
        printf("ok gsa_workspace_size %zu\n", ws);
    }
    /* argument errors come back as status codes, before any device work */
    {
        gsa_recipe r;
        gsa_act_params ap = {4.0f, 7.0f, 1.702f, 1.0f};
        gsa_qout q;
        gsa_status st;
        memset(&r, 0, sizeof r);
        memset(&q, 0, sizeof q);
        r.kind = GSA_NVFP4;
        st = grouped_scaled_act_fwd(NULL, NULL, split, 4, 256, GSA_ACT_SRELU, &ap, &r, &q, NULL, NULL, 0, NULL);
        if (st != GSA_ERR_INVALID_ARG) return fail("fwd without outputs");
        if (gsa_layout(0, split, 256, GSA_MXFP8, &info, NULL, NULL) != GSA_ERR_INVALID_ARG) return fail("E = 0");
        printf("ok errors: %s\n", gsa_status_string(st));
    }
    printf("all ok\n");
    return 0;
}
