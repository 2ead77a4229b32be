// Fused MoE layer kernel with 16-token tiles (batches whose experts average
// fewer than 12 tokens): ffn_stream.cuh instantiated for this tile width.
#define PW_TILE_N 16
#define PW_KERNEL_NAME apl_ffn_t16_kernel
#define PW_LAUNCHER_NAME launch_ffn_t16
#include "ffn_stream.cuh"
