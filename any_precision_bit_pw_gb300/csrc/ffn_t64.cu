// Fused MoE layer kernel with 64-token tiles (batches whose experts average
// 12 tokens or more, prefill included): ffn_stream.cuh instantiated for this
// tile width.
#define PW_TILE_N 64
#define PW_KERNEL_NAME apl_ffn_t64_kernel
#define PW_LAUNCHER_NAME launch_ffn_t64
#include "ffn_stream.cuh"
