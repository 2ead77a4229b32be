// Weight page table: per-block committed bitwidth q_i, desired bitwidth d_i,
// attached (GPU-resident) pages and the memory-size table M_i^b.
//
// "PagedWeight" arXiv text, §3 and §3.1: one row per linear-block (layer,
// expert, gate_up|down) holding B_i, q_i, d_i, the state of each bit-plane and
// M_i^b; one bit-plane with its LUT state is one weight page; lowering a block
// releases M_i^b - M_i^b' bytes (Eq. 3).  §3.1 / §3.3 ordering: an offload
// first lowers q_i and then retires the pages above it; a reload brings pages
// back first and raises q_i only once they are GPU-resident.
//
// The table borrows device pointers; it never allocates device memory.  A page
// is "attached" when the caller has handed its buffer to the table (the
// GPU-resident state); detaching it on a lowering hands ownership back.
#include <cstring>
#include <vector>

#include "pw_internal.h"

namespace {

struct BlockState {
  pw_block_info info{};
  int q = 0;
  int d = 0;
  const uint32_t* planes[PW_MAX_BITS] = {};
  const uint16_t* luts[PW_MAX_BITS + 1] = {};
};

bool bits_ok(const BlockState& b, int bits) {
  return bits >= b.info.seed_bits && bits <= b.info.parent_bits;
}

uint64_t resident_mask(const BlockState& b) {
  uint64_t m = 0;
  for (int p = 0; p < PW_MAX_BITS; ++p)
    if (b.planes[p]) m |= 1ull << p;
  for (int k = 0; k <= PW_MAX_BITS; ++k)
    if (b.luts[k]) m |= 1ull << (8 + k);
  return m;
}

int64_t block_bytes(const pw_block_info& in, int b) {
  // M_i^b: b planes plus the fp16 LUTs of bitwidths seed..b
  int64_t bytes = static_cast<int64_t>(b) * in.rows * in.cols / 8;
  for (int k = in.seed_bits; k <= b; ++k) bytes += in.rows * (int64_t{1} << k) * 2;
  return bytes;
}

}  // namespace

struct pw_page_table {
  std::vector<BlockState> blocks;
  std::vector<pw::BlockDesc> staging;
};

namespace {
int check_block(const pw_page_table* t, int block) {
  if (!t) return pw::set_error(PW_ERR_INVALID_ARG, "page table is NULL");
  if (block < 0 || block >= static_cast<int>(t->blocks.size()))
    return pw::set_error(PW_ERR_INVALID_ARG, "block %d out of range [0, %zu)", block, t->blocks.size());
  return PW_OK;
}
}  // namespace

extern "C" {

size_t pw_desc_bytes(int n_blocks) {
  return n_blocks > 0 ? static_cast<size_t>(n_blocks) * sizeof(pw::BlockDesc) : 0;
}

int pw_page_table_create(pw_page_table** out, int n_blocks, const pw_block_info* info) {
  if (!out || !info || n_blocks <= 0)
    return pw::set_error(PW_ERR_INVALID_ARG, "create: need out, info and n_blocks > 0");
  for (int i = 0; i < n_blocks; ++i) {
    const pw_block_info& in = info[i];
    if (in.layout != PW_LAYOUT_TILED)
      return pw::set_error(PW_ERR_UNSUPPORTED, "block %d: layout %d", i, in.layout);
    if (in.parent_bits < 1 || in.parent_bits > PW_MAX_BITS || in.seed_bits < 1 ||
        in.seed_bits > in.parent_bits)
      return pw::set_error(PW_ERR_INVALID_ARG, "block %d: need 1 <= seed <= parent <= 8", i);
    if (pw_plane_bytes(in.rows, in.cols, in.layout) == 0 || in.rows > (1 << 30) || in.cols > (1 << 30))
      return pw::set_error(PW_ERR_UNSUPPORTED, "block %d: shape %lld x %lld", i,
                           static_cast<long long>(in.rows), static_cast<long long>(in.cols));
  }
  auto* t = new (std::nothrow) pw_page_table;
  if (!t) return pw::set_error(PW_ERR_INVALID_ARG, "out of host memory");
  t->blocks.resize(n_blocks);
  for (int i = 0; i < n_blocks; ++i) t->blocks[i].info = info[i];
  *out = t;
  return PW_OK;
}

int pw_page_table_destroy(pw_page_table* t) {
  delete t;
  return PW_OK;
}

int pw_page_table_attach_plane(pw_page_table* t, int block, int plane, const uint32_t* d_plane) {
  if (int e = check_block(t, block)) return e;
  BlockState& b = t->blocks[block];
  if (plane < 0 || plane >= b.info.parent_bits)
    return pw::set_error(PW_ERR_INVALID_ARG, "plane %d outside [0, %d)", plane, b.info.parent_bits);
  if (!d_plane || (reinterpret_cast<uintptr_t>(d_plane) & 15))
    return pw::set_error(PW_ERR_INVALID_ARG, "plane pointer must be non-NULL and 16-byte aligned");
  b.planes[plane] = d_plane;
  return PW_OK;
}

int pw_page_table_attach_lut(pw_page_table* t, int block, int bits, const uint16_t* d_lut) {
  if (int e = check_block(t, block)) return e;
  BlockState& b = t->blocks[block];
  if (!bits_ok(b, bits))
    return pw::set_error(PW_ERR_INVALID_ARG, "LUT bitwidth %d outside [%d, %d]", bits, b.info.seed_bits,
                         b.info.parent_bits);
  if (!d_lut || (reinterpret_cast<uintptr_t>(d_lut) & 15))
    return pw::set_error(PW_ERR_INVALID_ARG, "LUT pointer must be non-NULL and 16-byte aligned");
  b.luts[bits] = d_lut;
  return PW_OK;
}

int pw_page_table_set_desired(pw_page_table* t, int block, int d) {
  if (int e = check_block(t, block)) return e;
  BlockState& b = t->blocks[block];
  if (!bits_ok(b, d)) return pw::set_error(PW_ERR_INVALID_ARG, "desired bitwidth %d not supported", d);
  b.d = d;
  return PW_OK;
}

int pw_page_table_set_bits(pw_page_table* t, int block, int q, uint64_t* released_mask) {
  if (released_mask) *released_mask = 0;
  if (int e = check_block(t, block)) return e;
  BlockState& b = t->blocks[block];
  if (!bits_ok(b, q))
    return pw::set_error(PW_ERR_INVALID_ARG, "bitwidth %d outside [%d, %d]", q, b.info.seed_bits,
                         b.info.parent_bits);
  if (q > b.q) {
    // reload order: every page of bitwidth <= q must already be resident
    for (int p = 0; p < q; ++p)
      if (!b.planes[p])
        return pw::set_error(PW_ERR_NOT_RESIDENT, "block %d: plane %d not resident, cannot raise to %d", block,
                             p, q);
    for (int k = b.info.seed_bits; k <= q; ++k)
      if (!b.luts[k])
        return pw::set_error(PW_ERR_NOT_RESIDENT, "block %d: LUT %d not resident, cannot raise to %d", block,
                             k, q);
    b.q = q;
    return PW_OK;
  }
  // lowering (or recommitting): commit first, then retire every page above q
  b.q = q;
  uint64_t mask = 0;
  for (int p = q; p < PW_MAX_BITS; ++p)
    if (b.planes[p]) {
      mask |= 1ull << p;
      b.planes[p] = nullptr;
    }
  for (int k = q + 1; k <= PW_MAX_BITS; ++k)
    if (b.luts[k]) {
      mask |= 1ull << (8 + k);
      b.luts[k] = nullptr;
    }
  if (released_mask) *released_mask = mask;
  return PW_OK;
}

int pw_page_table_get(const pw_page_table* t, int block, int* q, int* d, uint64_t* mask) {
  if (int e = check_block(t, block)) return e;
  const BlockState& b = t->blocks[block];
  if (q) *q = b.q;
  if (d) *d = b.d;
  if (mask) *mask = resident_mask(b);
  return PW_OK;
}

int64_t pw_page_table_bytes(const pw_page_table* t, int block, int b) {
  if (check_block(t, block)) return -1;
  const BlockState& s = t->blocks[block];
  if (!bits_ok(s, b)) return -1;
  return block_bytes(s.info, b);
}

int64_t pw_page_table_resident_bytes(const pw_page_table* t) {
  if (!t) return -1;
  int64_t total = 0;
  for (const BlockState& b : t->blocks)
    if (b.q > 0) total += block_bytes(b.info, b.q);
  return total;
}

int pw_page_table_sync(pw_page_table* t, void* d_desc, size_t desc_bytes, void* stream) {
  if (!t) return pw::set_error(PW_ERR_INVALID_ARG, "page table is NULL");
  const size_t need = pw_desc_bytes(static_cast<int>(t->blocks.size()));
  if (!d_desc || desc_bytes < need || (reinterpret_cast<uintptr_t>(d_desc) & 15))
    return pw::set_error(PW_ERR_INVALID_ARG, "descriptor buffer: need %zu bytes, 16-byte aligned", need);
  t->staging.assign(t->blocks.size(), pw::BlockDesc{});
  for (size_t i = 0; i < t->blocks.size(); ++i) {
    const BlockState& b = t->blocks[i];
    pw::BlockDesc& d = t->staging[i];
    d.q = b.q;
    d.rows = static_cast<int32_t>(b.info.rows);
    d.cols = static_cast<int32_t>(b.info.cols);
    d.parent = b.info.parent_bits;
    d.seed = b.info.seed_bits;
    d.layout = b.info.layout;
    for (int p = 0; p < b.q; ++p) d.planes[p] = b.planes[p];
    d.lut = b.q > 0 ? b.luts[b.q] : nullptr;
  }
  // The staging vector is pageable host memory: cudaMemcpyAsync copies it to
  // a driver staging buffer before returning, so it may be reused right away.
  PW_CUDA_TRY(cudaMemcpyAsync(d_desc, t->staging.data(), need, cudaMemcpyHostToDevice, pw::as_stream(stream)));
  return PW_OK;
}

}  // extern "C"

// Internal accessors for the test exports.
namespace pw {
int table_block(const pw_page_table* t, int block, BlockDesc* out, int bits_override) {
  if (int e = check_block(t, block)) return e;
  const BlockState& b = t->blocks[block];
  const int q = bits_override > 0 ? bits_override : b.q;
  if (q <= 0) return set_error(PW_ERR_NOT_RESIDENT, "block %d is not committed", block);
  *out = BlockDesc{};
  out->q = q;
  out->rows = static_cast<int32_t>(b.info.rows);
  out->cols = static_cast<int32_t>(b.info.cols);
  out->parent = b.info.parent_bits;
  out->seed = b.info.seed_bits;
  out->layout = b.info.layout;
  for (int p = 0; p < q && p < PW_MAX_BITS; ++p) {
    if (!b.planes[p]) return set_error(PW_ERR_NOT_RESIDENT, "block %d: plane %d not resident", block, p);
    out->planes[p] = b.planes[p];
  }
  out->lut = (q >= b.info.seed_bits && q <= b.info.parent_bits) ? b.luts[q] : nullptr;
  return PW_OK;
}
}  // namespace pw
