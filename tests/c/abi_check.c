/* The library's header compiled as plain C99 and its host-only entry points called from
 * C: the boundary is usable without C++ or CUDA headers.  No call here reaches a GPU
 * (the validation case fails before any CUDA call). */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "mse.h"

int main(void) {
    int bad = 0;
    if (strcmp(mse_status_string(MSE_OK), "MSE_OK") != 0) bad |= 1;
    if (strcmp(mse_status_string(MSE_ERR_NOT_DIVISIBLE), "MSE_ERR_NOT_DIVISIBLE") != 0) bad |= 2;
    /* the sharding gate: opted in, sequence-parallel, eligible, tp 8, 7168 / 6144 */
    if (mse_shard_sequence_parallel_mlp(1, 1, 1, 8, 7168, 6144) != 1) bad |= 4;
    if (mse_shard_sequence_parallel_mlp(1, 1, 1, 5, 7168, 6144) != 0) bad |= 8;
    /* workspace sizes are non-decreasing in T */
    if (mlp_swiglu_workspace_bytes(64, 7168, 6144) > mlp_swiglu_workspace_bytes(300, 7168, 6144)) bad |= 16;
    /* 6144 % 5 != 0 is rejected before any device work */
    {
        uint16_t dummy[8];
        mse_status st = mlp_swiglu_shard_forward(dummy, 128, 7168, 6144, dummy, dummy, 5, 0, 5, dummy, MSE_BF16,
                                                 128 * 7168, dummy, (size_t)1 << 30, NULL);
        if (st != MSE_ERR_NOT_DIVISIBLE) bad |= 32;
    }
    /* launch plans are host arithmetic: the replicated decode layer's gate_up on 144 CTAs in two
     * parts per tile, the merged projection on 136 CTAs in eight */
    {
        int32_t plan[8];
        if (mse_mlp_launch_plan(64, 7168, 6144, 1, 1, 0, 152, plan) != MSE_OK || plan[0] != 1 || plan[1] != 144 ||
            plan[3] != 2)
            bad |= 64;
        if (mse_merged_launch_plan(128, 7168, 1536, 576, 16, 152, plan) != MSE_OK || plan[1] != 136 || plan[2] != 8)
            bad |= 128;
        if (mse_mlp_launch_plan(64, 7168, 6144, 8, 9, 0, 152, plan) != MSE_ERR_INVALID_ARG) bad |= 256;
    }
    printf("%s %d\n", mse_version(), bad);
    return bad;
}
