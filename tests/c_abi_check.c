/* Built by tests/test_abi.py as plain C11 against include/: the boundary must
 * be usable from C.  Takes the address of every entry point (so the link
 * resolves each one) and runs the host-only helpers, which need no GPU. */
#include <stdio.h>
#include <string.h>

#include "msm_g1.h"
#include "msm_g1_testing.h"

typedef void (*any_fn)(void);

int main(void) {
    const any_fn entry[] = {
        (any_fn)msm_g1_create,          (any_fn)msm_g1_create_batch,   (any_fn)msm_g1_run,
        (any_fn)msm_g1_run_batch,       (any_fn)msm_g1_run_host,       (any_fn)msm_g1_mul_generator,
        (any_fn)msm_g1_run_noalloc,     (any_fn)msm_g1_destroy,        (any_fn)msm_g1_set_param,
        (any_fn)msm_g1_get_param,       (any_fn)msm_g1_last_phase_ms,  (any_fn)msm_g1_last_stats,
        (any_fn)msm_g1_window_count,    (any_fn)msm_g1_auto_window,    (any_fn)msm_g1_scratch_bytes,
        (any_fn)msm_g1_strerror,        (any_fn)msm_g1_test_fq,        (any_fn)msm_g1_test_g1,
        (any_fn)msm_g1_test_batch_add,  (any_fn)msm_g1_test_digits,    (any_fn)msm_g1_test_glv_split,
        (any_fn)msm_g1_glv_constants,   (any_fn)msm_g1_debug_read,     (any_fn)msm_g1_test_rns,
    };
    for (size_t i = 0; i < sizeof(entry) / sizeof(entry[0]); i++)
        if (!entry[i]) return 2;
    if (msm_g1_window_count(16) != 16 || msm_g1_window_count(0) != MSM_G1_ERR_INVALID_ARG) return 3;
    if (msm_g1_scratch_bytes(1u << 10, 8) == 0 || msm_g1_scratch_bytes(0, 8) != 0) return 4;
    if (strcmp(msm_g1_strerror(MSM_G1_OK), "ok") != 0) return 5;
    msm_g1_ctx *ctx = NULL;
    if (msm_g1_create(NULL, 16, 8) != MSM_G1_ERR_INVALID_ARG) return 6;
    if (msm_g1_run(ctx, NULL, NULL, 0, 8, NULL, 0) != MSM_G1_ERR_INVALID_ARG) return 7;
    msm_g1_destroy(NULL);
    printf("c abi ok\n");
    return 0;
}
