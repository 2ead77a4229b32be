// Bit-plane packer and unpacker for the tiled layout.
//
// "PagedWeight" arXiv text, §1 and Figure 3: weights are stored in Any-Precision
// LLM's overlaid bit-plane format, where a subset of the planes gives a lower
// bitwidth.  Plane p (0 = most significant) holds bit P-1-p of each parent
// index, so the top b planes carry idx >> (P-b).
//
// Tiled layout (the library's own choice; the pages give none): a plane is a
// sequence of 512-byte tiles, strip-major, each covering 16 rows x 256 columns.
// Strip s holds rows 8s..8s+7 and rows N/2+8s..N/2+8s+7, so one warp sees the
// gate row m and the up row I+m of a gate_up block in the same lanes.  Lane l
// owns bytes 16l..16l+15 of a tile: four uint32 words w; bit 4*elem+step%4 of
// word step/4 is element `elem` of k-step `step` of the lane's m16n8k16
// A-fragment (elem 0..3: row g, columns 2c, 2c+1, 2c+8, 2c+9 of the step;
// elem 4..7: row g+8, same columns; g = l/4, c = l%4).
#include "pw_internal.h"

namespace {

struct PlanePtrs {
  uint32_t* p[PW_MAX_BITS];
};

// One thread per (strip, tile, lane): gathers the lane's 128 elements and
// writes 16 bytes to each plane.
__global__ void pack_kernel(const uint8_t* __restrict__ idx, int rows, int cols, int P, PlanePtrs planes) {
  const int tiles_per_strip = cols / pw::kTileCols;
  const long long n_threads = static_cast<long long>(rows / pw::kTileRows) * tiles_per_strip * 32;
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (tid >= n_threads) return;
  const int lane = static_cast<int>(tid & 31);
  const long long tile_id = tid >> 5;
  const int strip = static_cast<int>(tile_id / tiles_per_strip);
  const int tile = static_cast<int>(tile_id % tiles_per_strip);
  const int g = lane >> 2, c = lane & 3;
  const int half_rows = rows / 2;
  const uint8_t mask = static_cast<uint8_t>((1u << P) - 1u);
  uint32_t words[PW_MAX_BITS][4];
#pragma unroll
  for (int p = 0; p < PW_MAX_BITS; ++p)
#pragma unroll
    for (int w = 0; w < 4; ++w) words[p][w] = 0u;
  for (int step = 0; step < 16; ++step) {
    const int w = step >> 2, js = step & 3;
#pragma unroll
    for (int elem = 0; elem < 8; ++elem) {
      const int n = (elem >> 2) * half_rows + strip * 8 + g;
      const int j = tile * pw::kTileCols + step * 16 + 2 * c + (elem & 1) + 8 * ((elem >> 1) & 1);
      const uint32_t v = idx[static_cast<long long>(n) * cols + j] & mask;
      const int bit = 4 * elem + js;
#pragma unroll
      for (int p = 0; p < PW_MAX_BITS; ++p)
        if (p < P) words[p][w] |= ((v >> (P - 1 - p)) & 1u) << bit;
    }
  }
  const long long word_off = (static_cast<long long>(strip) * tiles_per_strip + tile) * (pw::kTileBytes / 4) + lane * 4;
#pragma unroll
  for (int p = 0; p < PW_MAX_BITS; ++p)
    if (p < P)
      *reinterpret_cast<uint4*>(planes.p[p] + word_off) = make_uint4(words[p][0], words[p][1], words[p][2], words[p][3]);
}

// One thread per element: reassembles the b-bit index from the top b planes.
__global__ void unpack_kernel(pw::BlockDesc d, int b, uint8_t* __restrict__ out) {
  const long long total = static_cast<long long>(d.rows) * d.cols;
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= total) return;
  const int n = static_cast<int>(i / d.cols), j = static_cast<int>(i % d.cols);
  const int half_rows = d.rows / 2;
  const int half = n / half_rows, r = n % half_rows;
  const int strip = r >> 3, g = r & 7;
  const int tile = j / pw::kTileCols, jj = j % pw::kTileCols;
  const int step = jj >> 4, t = jj & 15;
  const int c = (t & 7) >> 1, odd = t & 1, upper = t >> 3;
  const int lane = 4 * g + c, elem = 4 * half + 2 * upper + odd;
  const long long word = (static_cast<long long>(strip) * (d.cols / pw::kTileCols) + tile) * (pw::kTileBytes / 4) +
                         lane * 4 + (step >> 2);
  const int bit = 4 * elem + (step & 3);
  uint32_t v = 0;
  for (int p = 0; p < b; ++p) v = (v << 1) | ((__ldg(d.planes[p] + word) >> bit) & 1u);
  out[i] = static_cast<uint8_t>(v);
}

}  // namespace

extern "C" {

size_t pw_plane_bytes(int64_t rows, int64_t cols, int layout) {
  if (layout != PW_LAYOUT_TILED || rows <= 0 || cols <= 0 || rows % pw::kTileRows || cols % pw::kTileCols)
    return 0;
  return static_cast<size_t>(rows) * static_cast<size_t>(cols) / 8;
}

int pw_pack_bitplanes(const uint8_t* d_idx, int64_t rows, int64_t cols, int parent_bits,
                      uint32_t* const* h_planes, int layout, void* stream) {
  if (pw_plane_bytes(rows, cols, layout) == 0)
    return pw::set_error(PW_ERR_UNSUPPORTED, "pack: shape %lld x %lld needs rows %% 16 == 0 and cols %% 256 == 0",
                         static_cast<long long>(rows), static_cast<long long>(cols));
  if (rows > (1 << 30) || cols > (1 << 30))
    return pw::set_error(PW_ERR_UNSUPPORTED, "pack: shape too large");
  if (parent_bits < 1 || parent_bits > PW_MAX_BITS)
    return pw::set_error(PW_ERR_INVALID_ARG, "pack: parent_bits %d outside 1..8", parent_bits);
  if (!d_idx || !h_planes) return pw::set_error(PW_ERR_INVALID_ARG, "pack: NULL argument");
  PlanePtrs pp{};
  for (int p = 0; p < parent_bits; ++p) {
    if (!h_planes[p] || (reinterpret_cast<uintptr_t>(h_planes[p]) & 15))
      return pw::set_error(PW_ERR_INVALID_ARG, "pack: plane %d pointer NULL or not 16-byte aligned", p);
    pp.p[p] = h_planes[p];
  }
  const long long n_threads = rows / pw::kTileRows * (cols / pw::kTileCols) * 32;
  const int threads = 256;
  const long long blocks = (n_threads + threads - 1) / threads;
  pack_kernel<<<static_cast<unsigned>(blocks), threads, 0, pw::as_stream(stream)>>>(
      d_idx, static_cast<int>(rows), static_cast<int>(cols), parent_bits, pp);
  PW_CUDA_TRY(cudaGetLastError());
  return PW_OK;
}

int pw_unpack_indices(const pw_page_table* t, int block, int b, uint8_t* d_idx_out, void* stream) {
  if (b < 1 || b > PW_MAX_BITS) return pw::set_error(PW_ERR_INVALID_ARG, "unpack: b %d outside 1..8", b);
  if (!d_idx_out) return pw::set_error(PW_ERR_INVALID_ARG, "unpack: NULL output");
  pw::BlockDesc d;
  if (int e = pw::table_block(t, block, &d, b)) return e;
  const long long total = static_cast<long long>(d.rows) * d.cols;
  const int threads = 256;
  unpack_kernel<<<static_cast<unsigned>((total + threads - 1) / threads), threads, 0, pw::as_stream(stream)>>>(
      d, b, d_idx_out);
  PW_CUDA_TRY(cudaGetLastError());
  return PW_OK;
}

}  // extern "C"
