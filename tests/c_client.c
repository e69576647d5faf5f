/* A plain C client of the library's ABI, built and run by tests/test_abi.py on the CPU: it calls
 * only what needs no GPU (version, the checkpoint size query, argument checks) and prints the
 * results for the test to compare. */
#include <stdio.h>

#include "mamba_scan.h"

int main(void) {
    mamba_scan_shape s = {4, 4096, 16, 2048, MAMBA_BF16};
    size_t bytes = 1;
    int rc;
    printf("version %d %d\n", mamba_scan_version(), MAMBA_SCAN_VERSION);
    rc = mamba_scan_fwd_train_ckpt_bytes(&s, &bytes);
    printf("ckpt_bytes %d %zu\n", rc, bytes);
    s.dstate = 65;
    rc = mamba_scan_fwd_train_ckpt_bytes(&s, &bytes);
    printf("bad_shape %d %s\n", rc, mamba_scan_last_error());
    rc = mamba_scan_fwd(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 1, NULL, NULL, NULL);
    printf("null_shape %d\n", rc);
    printf("launches %llu\n", (unsigned long long)mamba_scan_launch_count());
    return 0;
}
