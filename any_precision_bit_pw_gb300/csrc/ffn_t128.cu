// Fused MoE layer kernel with 128-token tiles (prefill batches whose experts
// average 96 tokens or more): ffn_stream.cuh instantiated for this tile
// width.  Each dequantised weight tile feeds an N = 128 MMA, so the weights
// are dequantised half as often per token as with 64-token tiles.
#define PW_TILE_N 128
#define PW_KERNEL_NAME apl_ffn_t128_kernel
#define PW_LAUNCHER_NAME launch_ffn_t128
#include "ffn_stream.cuh"
