/* A plain C99 caller of the library's C ABI (include/muon.h), built by
 * tests/test_c_abi.py with gcc -std=c99 -Wall -Wextra -Werror and linked against
 * libmuon_gb300.so.  It needs no GPU: it prints the struct layouts a C compiler
 * sees, the status strings, and what muon_plan_workspace_size reports for one
 * Qwen2.5-7B layer, one "key value" pair per line. */
#include <stddef.h>
#include <stdio.h>

#include "muon.h"

#define FIELD(type, f) printf("%s.%s %zu\n", #type, #f, offsetof(type, f))

int main(void) {
    printf("sizeof.muon_plan_opts %zu\n", sizeof(muon_plan_opts));
    FIELD(muon_plan_opts, keep_update);
    FIELD(muon_plan_opts, timing);
    FIELD(muon_plan_opts, single_sm_gemm);
    FIELD(muon_plan_opts, generic_small);
    FIELD(muon_plan_opts, chain_clusters);
    FIELD(muon_plan_opts, max_ns_steps);
    FIELD(muon_plan_opts, workspace_bytes);
    FIELD(muon_plan_opts, chunks);
    FIELD(muon_plan_opts, full_symmetric);
    FIELD(muon_plan_opts, small_fp32);
    FIELD(muon_plan_opts, check_finite);
    FIELD(muon_plan_opts, precision);
    FIELD(muon_plan_opts, split_max_r);
    FIELD(muon_plan_opts, full_rows);
    FIELD(muon_plan_opts, precision_of);
    printf("sizeof.muon_plan_info_t %zu\n", sizeof(muon_plan_info_t));
    FIELD(muon_plan_info_t, n_matrices);
    FIELD(muon_plan_info_t, n_buckets);
    FIELD(muon_plan_info_t, workspace_bytes);
    FIELD(muon_plan_info_t, launches_last_step);
    FIELD(muon_plan_info_t, sm_count);
    FIELD(muon_plan_info_t, n_chunks);
    FIELD(muon_plan_info_t, lower_chunks);
    FIELD(muon_plan_info_t, tuned_candidates);
    FIELD(muon_plan_info_t, chain_clusters);
    FIELD(muon_plan_info_t, split_buckets);
    FIELD(muon_plan_info_t, fp32_buckets);
    FIELD(muon_plan_info_t, colsq_len);
    printf("sizeof.muon_shape %zu\n", sizeof(muon_shape));

    for (int s = MUON_OK; s <= MUON_ERR_NONFINITE; ++s) printf("status.%d %s\n", s, muon_status_string((muon_status)s));

    const muon_shape layer[7] = {{3584, 3584}, {512, 3584},   {512, 3584},  {3584, 3584},
                                 {18944, 3584}, {18944, 3584}, {3584, 18944}};
    int64_t bytes = 0;
    int32_t buckets = 0, chunks = 0;
    muon_status st = muon_plan_workspace_size(layer, 7, MUON_BF16, NULL, &bytes, &buckets, &chunks);
    printf("layer.status %d\nlayer.bytes %lld\nlayer.buckets %d\nlayer.chunks %d\n", (int)st, (long long)bytes,
           (int)buckets, (int)chunks);

    muon_plan_opts opts = {0};
    opts.chunks = 4;
    st = muon_plan_workspace_size(layer, 7, MUON_BF16, &opts, &bytes, &buckets, &chunks);
    printf("chunked.status %d\nchunked.bytes %lld\nchunked.chunks %d\n", (int)st, (long long)bytes, (int)chunks);

    /* argument errors come back as codes, before any CUDA call */
    muon_plan plan = NULL;
    printf("bad.create %d\n", (int)muon_plan_create(layer, 0, MUON_BF16, NULL, &plan));
    printf("bad.step %d\n", (int)muon_step(NULL, NULL, NULL, NULL, 0.02f, 0.1f, 0.95f, 5, MUON_MODE_NS, NULL));
    muon_plan_destroy(NULL);
    return 0;
}
