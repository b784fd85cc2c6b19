/*
 * A plain C (C11) consumer of the KDA C ABI: it includes include/kda.h,
 * links against the CUDA library and calls the host-only parts of the API
 * (size queries, status names, argument checks that return before any
 * launch), so it runs without a GPU.  Prints one line per check and exits
 * non-zero on the first mismatch.
 */
#include <stdio.h>
#include <string.h>

#include "kda.h"

static int fails = 0;

static void expect(int ok, const char* what)
{
    printf("%s %s\n", ok ? "ok  " : "FAIL", what);
    if (!ok) ++fails;
}

int main(void)
{
    static float fake_param[4096] __attribute__((aligned(16)));
    kda_params p;
    memset(&p, 0, sizeof(p));
    p.num_heads = 32;
    p.head_dim_k = 128;
    p.head_dim_v = 128;
    p.conv_kernel = 4;
    p.gate_mode = KDA_GATE_SAFE;
    p.gate_lower_bound = -5.0f;
    p.l2_eps = 1e-6f;
    p.norm_eps = 1e-6f;
    p.scale = 1.0f;
    p.io_dtype = KDA_DTYPE_BF16;
    p.out_dtype = KDA_DTYPE_BF16;
    p.num_slots = 8;
    p.A_log = fake_param;
    p.dt_bias = fake_param;
    p.conv_weight = fake_param;
    p.norm_weight = NULL;

    expect(kda_abi_version() == 100, "abi version");
    expect(strcmp(kda_status_string(KDA_ERR_WORKSPACE), "KDA_ERR_WORKSPACE") == 0, "status string");
    /* the varlen prefill needs the longest-first schedule; few long chains take the split path's ring */
    expect(kda_prefill_workspace_bytes(&p, 8, 29273) > 0, "prefill workspace, 8 sequences");
    expect(kda_prefill_workspace_bytes(&p, 1, 32768) > kda_prefill_workspace_bytes(&p, 8, 29273),
           "prefill workspace, one long prompt (split path)");
    expect(kda_prefill_scan_workspace_bytes(&p, 1, 32768, 4) > (size_t)32768 * 32 * 128 * 8,
           "scan workspace holds raw outputs and corrections");
    expect(kda_verify_log_bytes(&p, 32, 8) > 0, "verify log bytes");
    expect(kda_prefill_static_workspace_capacity() == 256 * 1024, "static workspace capacity");
    /* errors returned before any launch */
    kda_params bad = p;
    bad.head_dim_k = 96;
    expect(kda_decode(&bad, 1, fake_param, fake_param, fake_param, fake_param, fake_param, NULL, NULL, fake_param,
                      fake_param, fake_param, NULL, (cudaStream_t)0) == KDA_ERR_UNSUPPORTED_GEOMETRY,
           "unsupported head width rejected");
    bad = p;
    bad.gate_lower_bound = 1.0f;
    expect(kda_decode(&bad, 1, fake_param, fake_param, fake_param, fake_param, fake_param, NULL, NULL, fake_param,
                      fake_param, fake_param, NULL, (cudaStream_t)0) == KDA_ERR_INVALID_BOUND,
           "positive safe-gate bound rejected");
    expect(kda_prefill_scan(&p, (const int32_t*)fake_param, 1, 64, fake_param, fake_param, fake_param, fake_param,
                            fake_param, NULL, NULL, fake_param, fake_param, fake_param, fake_param, 1 << 20, 0, NULL,
                            (cudaStream_t)0) == KDA_ERR_INVALID_ARGUMENT,
           "zero scan segments rejected");
    return fails ? 1 : 0;
}
