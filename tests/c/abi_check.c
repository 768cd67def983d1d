/* Plain C11 user of include/pa.h: compiled with gcc -std=c11 -Wall -Werror
 * and linked against libpa.so by tests/test_abi.py.  It only makes calls
 * that need no GPU: sizes and layouts of a problem with num_sms given, and
 * argument checks that fail before anything is launched.  Prints one line
 * per check and exits non-zero on the first mismatch. */
#include <stdio.h>
#include <string.h>

#include "pa.h"

static int expect(const char *what, pa_status got, pa_status want) {
    printf("%s: %s\n", what, pa_status_string(got));
    if (got != want) {
        fprintf(stderr, "%s: got %s, want %s\n", what, pa_status_string(got), pa_status_string(want));
        return 1;
    }
    return 0;
}

int main(void) {
    pa_problem p;
    memset(&p, 0, sizeof p);
    p.batch = 4;
    p.next_n = 1;
    p.num_q_heads = 32;
    p.num_kv_heads = 8;
    p.head_dim_k = 128;
    p.head_dim_v = 128;
    p.block_size = 16;
    p.num_blocks = 1000;
    p.max_blocks_per_seq = 64;
    p.max_context_len = 1024;
    p.q_dtype = PA_BF16;
    p.kv_dtype = PA_BF16;
    p.out_dtype = PA_BF16;
    p.k_scale_mode = PA_SCALE_NONE;
    p.v_scale_mode = PA_SCALE_NONE;
    p.num_sms = 152;
    p.softmax_scale = 0.08838834764831845f;

    int bad = 0;
    size_t bytes = 0;
    pa_layout lo;
    printf("version %d\n", pa_version());
    bad |= expect("pa_workspace_size", pa_workspace_size(&p, &bytes), PA_OK);
    bad |= expect("pa_workspace_layout", pa_workspace_layout(&p, &lo), PA_OK);
    if (bytes != lo.total_bytes || bytes == 0) {
        fprintf(stderr, "workspace size %zu vs layout %zu\n", bytes, lo.total_bytes);
        bad = 1;
    }
    bad |= expect("pa_sparse_workspace_size", pa_sparse_workspace_size(&p, 64, &bytes), PA_OK);
    bad |= expect("pa_plan without a workspace", pa_plan(&p, NULL, NULL, NULL, 0, NULL), PA_ERR_WORKSPACE);
    bad |= expect("pa_run without a workspace",
                  pa_run(&p, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, NULL, NULL, NULL), PA_ERR_WORKSPACE);
    bad |= expect("pa_insert with a NULL pool",
                  pa_insert(&p, PA_BF16, (const void *)0x100000, (const void *)0x100000, (const int32_t *)0x100000,
                            (const int32_t *)0x100000, NULL, NULL, NULL, (void *)0x100000, NULL, NULL),
                  PA_ERR_INVALID_ARG);
    bad |= expect("pa_sparse_attention without a workspace",
                  pa_sparse_attention(&p, 64, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, NULL, NULL,
                                      NULL),
                  PA_ERR_WORKSPACE);
    p.head_dim_k = 100;
    bad |= expect("pa_workspace_size, D = 100", pa_workspace_size(&p, &bytes), PA_ERR_UNSUPPORTED);
    bad |= expect("pa_get_error without a word", pa_get_error(NULL, NULL, NULL), PA_ERR_INVALID_ARG);
    return bad;
}
