// Internal declarations shared by the translation units of libpw.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "pw.h"

namespace pw {

// Device descriptor of one linear-block at its committed bitwidth (128 bytes).
// Written by pw_page_table_sync, read by the fused kernels.
struct alignas(16) BlockDesc {
  int32_t q;        // committed bitwidth (0 = not committed)
  int32_t rows;     // N
  int32_t cols;     // K
  int32_t parent;   // P
  int32_t seed;     // S
  int32_t layout;
  int32_t pad0, pad1;
  const uint32_t* planes[PW_MAX_BITS];  // planes 0..q-1 (MSB first); rest NULL
  const uint16_t* lut;                  // LUT_q, fp16 [rows][2^q]
  int64_t pad2[3];
};
static_assert(sizeof(BlockDesc) == 128, "descriptor must stay 128 bytes");

// Tiled plane layout: 128-row strips x 128-column tiles, 2048 bytes per tile
// per plane; see include/pw.h for the bit map.
constexpr int kTileRows = 128;
constexpr int kTileCols = 128;
constexpr int kTileBytes = 2048;

// Records a message for pw_last_error() and returns `code`.
int set_error(int code, const char* fmt, ...);
void clear_error();
int cuda_error(cudaError_t e, const char* what);

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Routing of L independent layers in one launch (route.cu): the arrays of
// layer l start at l*T*E (logits), l*T*(k+S) (ids, w, perm, inv_perm),
// l*(E+S) (offsets, mass); offsets, perm and inv_perm hold indices into the
// concatenated assignments of all layers.  Arguments are not checked.  With
// d_zero, the launch also zeroes zero_bytes there (16-byte aligned, a
// multiple of 16: the next fused launch's counters), and it lets the next
// kernel on the stream start early (programmatic dependent launch: that
// kernel waits for this grid's completion before it reads anything).
int route_layers(const float* d_logits, int L, int T, int E, int k, int S, int32_t* d_ids, float* d_w,
                 int32_t* d_offsets, int32_t* d_perm, int32_t* d_inv_perm, float* d_mass_accum, cudaStream_t s,
                 void* d_zero = nullptr, size_t zero_bytes = 0);

// Host-side descriptor of `block` of a page table, at its committed bitwidth
// (or at `bits_override` if > 0); fails unless the planes are attached.
int table_block(const pw_page_table* t, int block, BlockDesc* out, int bits_override);

}  // namespace pw

#define PW_CUDA_TRY(expr)                                  \
  do {                                                     \
    cudaError_t pw_e_ = (expr);                            \
    if (pw_e_ != cudaSuccess) return pw::cuda_error(pw_e_, #expr); \
  } while (0)
