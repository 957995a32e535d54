/* A plain C client of the library: compiled by the CPU test suite with gcc
 * against include/crmsnorm.h and linked to libcrmsnorm.so.  It uses only the
 * calls that need no GPU (capability queries, status names, validation that
 * fails before any launch) and prints one line per check. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "crmsnorm.h"

static int fails = 0;

static void expect(const char *what, crmsn_status got, crmsn_status want)
{
    printf("%s: %s\n", what, crmsn_status_str(got));
    if (got != want) {
        printf("  expected %s\n", crmsn_status_str(want));
        ++fails;
    }
}

int main(void)
{
    void *fake = (void *)(uintptr_t)((uint64_t)1 << 40);   /* never dereferenced */
    expect("supports fwd H=4096", rmsnorm_supports(4096, CRMSN_BF16, CRMSN_OP_FWD), CRMSN_OK);
    expect("supports fwd H=4097", rmsnorm_supports(4097, CRMSN_BF16, CRMSN_OP_FWD),
           CRMSN_ERR_UNSUPPORTED_H);
    expect("supports block quant H=200", rmsnorm_supports(200, CRMSN_BF16, CRMSN_OP_BLOCK_QUANT),
           CRMSN_ERR_UNSUPPORTED_H);
    expect("supports layernorm bf16 weight", rmsnorm_supports(1024, CRMSN_BF16, CRMSN_OP_LAYERNORM),
           CRMSN_ERR_DTYPE);
    expect("fwd T=0", rmsnorm_fwd(NULL, 0, NULL, 0, NULL, CRMSN_BF16, 0.f, 1e-6f, 0, 4096,
                                  NULL, 0, NULL, NULL, 0, (cudaStream_t)0), CRMSN_OK);
    expect("fwd NULL x", rmsnorm_fwd(NULL, 4096, NULL, 0, fake, CRMSN_BF16, 0.f, 1e-6f, 4, 4096,
                                     fake, 4096, NULL, NULL, 0, (cudaStream_t)0), CRMSN_ERR_NULL);
    expect("fwd bad dtype", rmsnorm_fwd(fake, 4096, NULL, 0, fake, 7, 0.f, 1e-6f, 4, 4096,
                                        fake, 4096, NULL, NULL, 0, (cudaStream_t)0), CRMSN_ERR_DTYPE);
    expect("silu bad format", fused_rmsnorm_silu(fake, 256, 9, fake, 256, fake, CRMSN_BF16, 0.f,
                                                 NULL, 1e-6f, 4, 256, NULL, (cudaStream_t)0),
           CRMSN_ERR_DTYPE);
    expect("layernorm_quant bad kind", layernorm_quant(fake, 256, 5, fake, 256, fake, fake, fake,
                                                       1e-5f, 4, 256, NULL, NULL, (cudaStream_t)0),
           CRMSN_ERR_DTYPE);
    printf("%s\n", fails ? "FAILED" : "ALL OK");
    return fails != 0;
}
