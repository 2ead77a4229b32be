// Fused MoE layer kernel for batches of one or two tokens per expert on the
// CUDA cores: ffn_stream.cuh instantiated with 2-token tiles, the dequant
// warps multiplying the dequantised weights with the token rows themselves
// (fp32 FMA of the exact fp16 products) instead of issuing tensor-core MMAs.
#define PW_TILE_N 2
#define PW_GEMV 1
#define PW_KERNEL_NAME apl_ffn_gemv_kernel
#define PW_LAUNCHER_NAME launch_ffn_gemv
#include "ffn_stream.cuh"
