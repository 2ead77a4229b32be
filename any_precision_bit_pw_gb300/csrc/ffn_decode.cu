// Fused MoE layer kernel with 16-token tiles (decode batches): ffn_stream.cuh
// instantiated for this tile width.
#define PW_TILE_N 16
#define PW_KERNEL_NAME apl_decode_kernel
#define PW_LAUNCHER_NAME launch_decode_kernel
#include "ffn_stream.cuh"
