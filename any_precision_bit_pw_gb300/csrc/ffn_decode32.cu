// Fused MoE layer kernel with 32-token tiles (decode batches): ffn_stream.cuh
// instantiated for this tile width.
#define PW_TILE_N 32
#define PW_KERNEL_NAME apl_decode32_kernel
#define PW_LAUNCHER_NAME launch_decode32_kernel
#include "ffn_stream.cuh"
