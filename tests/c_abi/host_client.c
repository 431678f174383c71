/* A plain C client of the library's host-only entry points: it links
 * against libw8a8.so through the public header alone and prints what the
 * guard, the planner and the workspace calls report, so that a test can
 * compare them with the Python binding.  No GPU call is made. */
#include <stdio.h>

#include "w8a8.h"

int main(void)
{
    int reason = 0;
    const int ok = w8a8_shape_supported(6144, 4096, 4096, W8A8_BF16, W8A8_BF16, &reason);
    const int bad = w8a8_shape_supported(64, 12, 250, W8A8_BF16, W8A8_BF16, &reason);
    int64_t plan[5];
    const int planned = w8a8_gemm_plan(6144, 4096, 4096, 148, -1, plan);
    int breason = 0;
    const int bf16_ok = w8a8_bf16_linear_supported(64, 128, 1032, W8A8_BF16, &breason);
    printf("version %d\n", w8a8_version());
    printf("guard %d %d reason %d\n", ok, bad, reason);
    printf("plan %d %lld %lld %lld %lld %lld\n", planned, (long long)plan[0], (long long)plan[1],
           (long long)plan[2], (long long)plan[3], (long long)plan[4]);
    printf("workspace %zu %zu\n", w8a8_linear_workspace_min_bytes(6144, 4096),
           w8a8_linear_workspace_bytes(6144, 4096, 4096));
    printf("bf16 %d %d %zu\n", bf16_ok, breason, w8a8_bf16_linear_workspace_bytes(64, 128, 1032));
    printf("mlp %zu\n", w8a8_mlp_workspace_bytes(6144, 4096, 16384, 4096));
    printf("status %s\n", w8a8_status_str(W8A8_ERR_UNSUPPORTED_SHAPE));
    /* argument errors come back before any device work */
    printf("errors %d %d\n", (int)w8a8_linear(0, W8A8_BF16, 1, 64, 0, 0, 8, 0, W8A8_BF16, 0, 0, 0, 0),
           (int)w8a8_quantize_qk_blocks(0, W8A8_BF16, 1, 1, 8, 60, W8A8_LAYOUT_HND, 4, 0, 0, 0));
    return 0;
}
