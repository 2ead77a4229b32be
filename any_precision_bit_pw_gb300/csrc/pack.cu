// Bit-plane packer and unpacker for the tiled layout.
//
// "PagedWeight" arXiv text, §1 and Figure 3: weights are stored in Any-Precision
// LLM's overlaid bit-plane format, where a subset of the planes gives a lower
// bitwidth.  Plane p (0 = most significant) holds bit P-1-p of each parent
// index, so the top b planes carry idx >> (P-b).
//
// Tiled layout (the library's own choice; the pages give none): a plane is a
// sequence of 2048-byte tiles, strip-major, each covering a 128-row strip and
// 128 columns.  Strip s holds rows 64s..64s+63 and N/2+64s..N/2+64s+63; row
// position pos = 32w + i within the strip is row 64s+16w+i (i < 16) or
// N/2+64s+16w+(i-16) (i >= 16), so in a gate_up block the gate row m and the up
// row m sit 16 lanes apart in the same warp.  Position pos owns 16 bytes of the
// tile (four little-endian words); column 32*word + 8*js + e of the tile is
// bit 4e + js of the word ("nibble" order: one shift and mask per plane gives
// the indices of 8 consecutive columns).
#include "pw_internal.h"

namespace {

struct PlanePtrs {
  uint32_t* p[PW_MAX_BITS];
};

__device__ __forceinline__ int strip_pos_row(int strip, int pos, int half_rows) {
  const int w = pos >> 5, i = pos & 31;
  return (i >> 4) * half_rows + strip * 64 + 16 * w + (i & 15);
}

// One thread per (strip, tile, pos): reads 128 indices of its row and writes
// 16 bytes to each plane.
__global__ void pack_kernel(const uint8_t* __restrict__ idx, int rows, int cols, int P, PlanePtrs planes) {
  const int tiles = cols / pw::kTileCols;
  const long long n_threads = static_cast<long long>(rows / pw::kTileRows) * tiles * pw::kTileRows;
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (tid >= n_threads) return;
  const int pos = static_cast<int>(tid % pw::kTileRows);
  const long long tile_id = tid / pw::kTileRows;
  const int strip = static_cast<int>(tile_id / tiles);
  const int tile = static_cast<int>(tile_id % tiles);
  const int n = strip_pos_row(strip, pos, rows / 2);
  const uint32_t mask = (1u << P) - 1u;
  uint32_t words[PW_MAX_BITS][4];
#pragma unroll
  for (int p = 0; p < PW_MAX_BITS; ++p)
#pragma unroll
    for (int w = 0; w < 4; ++w) words[p][w] = 0u;
  const uint4* src = reinterpret_cast<const uint4*>(idx + static_cast<long long>(n) * cols + tile * pw::kTileCols);
#pragma unroll
  for (int v = 0; v < 8; ++v) {   // 16 columns per uint4
    const uint4 q = src[v];
    const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int b = 0; b < 16; ++b) {
      const int jj = v * 16 + b;
      const uint32_t val = (qw[b >> 2] >> (8 * (b & 3))) & mask;
      const int w = jj >> 5, t = jj & 31;
      const int bit = 4 * (t & 7) + (t >> 3);
#pragma unroll
      for (int p = 0; p < PW_MAX_BITS; ++p)
        if (p < P) words[p][w] |= ((val >> (P - 1 - p)) & 1u) << bit;
    }
  }
  const long long word_off = (static_cast<long long>(strip) * tiles + tile) * (pw::kTileBytes / 4) + pos * 4;
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
  const int strip = r >> 6, rr = r & 63;
  const int pos = 32 * (rr >> 4) + (rr & 15) + 16 * half;
  const int tile = j / pw::kTileCols, jj = j % pw::kTileCols;
  const int word = jj >> 5, t = jj & 31;
  const int bit = 4 * (t & 7) + (t >> 3);
  const long long widx = (static_cast<long long>(strip) * (d.cols / pw::kTileCols) + tile) * (pw::kTileBytes / 4) +
                         pos * 4 + word;
  uint32_t v = 0;
  for (int p = 0; p < b; ++p) v = (v << 1) | ((__ldg(d.planes[p] + widx) >> bit) & 1u);
  out[i] = static_cast<uint8_t>(v);
}

// One thread per (row, entry) of a LUT: the entry's tiled byte offset is
// (strip*2^b + c)*256 + 4*((w%2)*32 + i) + 2*(w/2) for row position pos = 32w + i
// of its strip, so a strip's table is one contiguous run in the order of the
// kernels' shared LUT region (one bulk copy per unit).
__global__ void pack_lut_kernel(const uint16_t* __restrict__ lut, int rows, int bits, uint16_t* __restrict__ out) {
  const long long n = static_cast<long long>(rows) << bits;
  for (long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; t < n;
       t += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int row = static_cast<int>(t >> bits), c = static_cast<int>(t & ((1ll << bits) - 1));
    const int half_rows = rows / 2;
    const int half = row / half_rows, r = row % half_rows;
    const int strip = r / 64, rr = r % 64, w = rr / 16, i = rr % 16 + 16 * half;
    const long long byte = ((static_cast<long long>(strip) << bits) + c) * 256 + 4 * ((w % 2) * 32 + i) + 2 * (w / 2);
    out[byte / 2] = lut[t];
  }
}

}  // namespace

extern "C" {

int pw_pack_lut(const uint16_t* d_lut, int64_t rows, int bits, uint16_t* d_out, void* stream) {
  if (rows <= 0 || rows % pw::kTileRows || rows > (1 << 30))
    return pw::set_error(PW_ERR_UNSUPPORTED, "pack_lut: rows %lld must be a positive multiple of 128",
                         static_cast<long long>(rows));
  if (bits < 1 || bits > PW_MAX_BITS) return pw::set_error(PW_ERR_INVALID_ARG, "pack_lut: bits %d outside 1..8", bits);
  if (!d_lut || !d_out || d_lut == d_out || (reinterpret_cast<uintptr_t>(d_out) & 15))
    return pw::set_error(PW_ERR_INVALID_ARG, "pack_lut: NULL, aliased, or output not 16-byte aligned");
  const long long n = rows << bits;
  const int threads = 256;
  const long long blocks = (n + threads - 1) / threads;
  pack_lut_kernel<<<static_cast<unsigned>(blocks < 65535 ? blocks : 65535), threads, 0, pw::as_stream(stream)>>>(
      d_lut, static_cast<int>(rows), bits, d_out);
  PW_CUDA_TRY(cudaGetLastError());
  return PW_OK;
}

size_t pw_plane_bytes(int64_t rows, int64_t cols, int layout) {
  if (layout != PW_LAYOUT_TILED || rows <= 0 || cols <= 0 || rows % pw::kTileRows || cols % pw::kTileCols)
    return 0;
  return static_cast<size_t>(rows) * static_cast<size_t>(cols) / 8;
}

int pw_pack_bitplanes(const uint8_t* d_idx, int64_t rows, int64_t cols, int parent_bits,
                      uint32_t* const* h_planes, int layout, void* stream) {
  if (pw_plane_bytes(rows, cols, layout) == 0)
    return pw::set_error(PW_ERR_UNSUPPORTED, "pack: shape %lld x %lld needs rows and cols multiples of 128",
                         static_cast<long long>(rows), static_cast<long long>(cols));
  if (rows > (1 << 30) || cols > (1 << 30)) return pw::set_error(PW_ERR_UNSUPPORTED, "pack: shape too large");
  if (parent_bits < 1 || parent_bits > PW_MAX_BITS)
    return pw::set_error(PW_ERR_INVALID_ARG, "pack: parent_bits %d outside 1..8", parent_bits);
  if (!d_idx || !h_planes || (reinterpret_cast<uintptr_t>(d_idx) & 15))
    return pw::set_error(PW_ERR_INVALID_ARG, "pack: NULL argument or index buffer not 16-byte aligned");
  PlanePtrs pp{};
  for (int p = 0; p < parent_bits; ++p) {
    if (!h_planes[p] || (reinterpret_cast<uintptr_t>(h_planes[p]) & 15))
      return pw::set_error(PW_ERR_INVALID_ARG, "pack: plane %d pointer NULL or not 16-byte aligned", p);
    pp.p[p] = h_planes[p];
  }
  const long long n_threads = rows / pw::kTileRows * (cols / pw::kTileCols) * pw::kTileRows;
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
