// Fused MoE layer kernel with 64-token tiles (prefill batches): ffn_stream.cuh
// instantiated for this tile width.
#define PW_TILE_N 64
#define PW_KERNEL_NAME apl_prefill_kernel
#define PW_LAUNCHER_NAME launch_prefill_kernel
#include "ffn_stream.cuh"
