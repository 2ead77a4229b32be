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
//
// §3.3 asynchronous page movement: a page can also hold a host copy (CPU
// resident) and be in transfer.  Offload and reload are one cudaMemcpyAsync
// each on the caller's copy stream, tracked by an event the table owns; the
// table learns of completion only in pw_page_table_poll, so a reloaded page is
// attached (and q_i can be raised) only after its copy has finished, and a
// page above q_i whose offload copy is still in flight stays attached until
// the copy has finished.
#include <cstring>
#include <vector>

#include "pw_internal.h"

namespace {

constexpr int kPages = 2 * PW_MAX_BITS + 1;   // page ids: plane p = p, LUT of bitwidth b = 8 + b
enum : int { kXferNone = 0, kXferToCpu = 1, kXferToGpu = 2 };

struct PageXfer {
  void* host = nullptr;       // host copy (complete once `cpu`)
  bool cpu = false;
  int xfer = kXferNone;
  void* pending = nullptr;    // reload destination, attached when the copy completes
  cudaEvent_t ev = nullptr;
};

struct BlockState {
  pw_block_info info{};
  int q = 0;
  int d = 0;
  const uint32_t* planes[PW_MAX_BITS] = {};
  const uint16_t* luts[PW_MAX_BITS + 1] = {};
  PageXfer pages[kPages];
  uint64_t released_late = 0;   // pages above q detached by poll after their offload copy
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

int64_t page_bytes(const BlockState& b, int page) {
  if (page >= 0 && page < b.info.parent_bits) return b.info.rows * b.info.cols / 8;
  const int k = page - PW_MAX_BITS;
  if (page >= PW_MAX_BITS && page < kPages && bits_ok(b, k)) return b.info.rows * (int64_t{1} << k) * 2;
  return -1;
}

const void* attached(const BlockState& b, int page) {
  return page < PW_MAX_BITS ? static_cast<const void*>(b.planes[page])
                            : static_cast<const void*>(b.luts[page - PW_MAX_BITS]);
}

void set_attached(BlockState& b, int page, const void* d) {
  if (page < PW_MAX_BITS)
    b.planes[page] = static_cast<const uint32_t*>(d);
  else
    b.luts[page - PW_MAX_BITS] = static_cast<const uint16_t*>(d);
}

// Referenced by the committed bitwidth (planes 0..q-1, LUTs seed..q).
bool referenced(const BlockState& b, int page) {
  return page < PW_MAX_BITS ? page < b.q : (page - PW_MAX_BITS) <= b.q;
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
  if (!t) return PW_OK;
  // transfers still in flight finish before their events go away
  for (BlockState& b : t->blocks)
    for (PageXfer& x : b.pages)
      if (x.ev) {
        if (x.xfer != kXferNone) cudaEventSynchronize(x.ev);
        cudaEventDestroy(x.ev);
      }
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
  if (b.pages[plane].xfer != kXferNone)
    return pw::set_error(PW_ERR_BUSY, "block %d: plane %d has a transfer in flight", block, plane);
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
  if (b.pages[PW_MAX_BITS + bits].xfer != kXferNone)
    return pw::set_error(PW_ERR_BUSY, "block %d: LUT %d has a transfer in flight", block, bits);
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
  // (a page whose offload copy is still in flight is retired by the poll that
  // sees the copy finish)
  b.q = q;
  uint64_t mask = 0;
  for (int p = q; p < PW_MAX_BITS; ++p)
    if (b.planes[p] && b.pages[p].xfer != kXferToCpu) {
      mask |= 1ull << p;
      b.planes[p] = nullptr;
    }
  for (int k = q + 1; k <= PW_MAX_BITS; ++k)
    if (b.luts[k] && b.pages[PW_MAX_BITS + k].xfer != kXferToCpu) {
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

int64_t pw_page_bytes(const pw_page_table* t, int block, int page) {
  if (check_block(t, block)) return -1;
  return page_bytes(t->blocks[block], page);
}

int pw_page_offload(pw_page_table* t, int block, int page, void* h_dst, void* copy_stream) {
  if (int e = check_block(t, block)) return e;
  BlockState& b = t->blocks[block];
  const int64_t bytes = page_bytes(b, page);
  if (bytes < 0) return pw::set_error(PW_ERR_INVALID_ARG, "block %d: no page %d", block, page);
  if (!h_dst) return pw::set_error(PW_ERR_INVALID_ARG, "offload: NULL host buffer");
  PageXfer& x = b.pages[page];
  if (x.xfer != kXferNone) return pw::set_error(PW_ERR_BUSY, "block %d: page %d has a transfer in flight", block, page);
  const void* d = attached(b, page);
  if (!d) return pw::set_error(PW_ERR_NOT_RESIDENT, "block %d: page %d is not GPU-resident", block, page);
  if (!x.ev) PW_CUDA_TRY(cudaEventCreateWithFlags(&x.ev, cudaEventDisableTiming));
  cudaStream_t s = pw::as_stream(copy_stream);
  PW_CUDA_TRY(cudaMemcpyAsync(h_dst, d, static_cast<size_t>(bytes), cudaMemcpyDeviceToHost, s));
  PW_CUDA_TRY(cudaEventRecord(x.ev, s));
  x.host = h_dst;
  x.cpu = false;
  x.xfer = kXferToCpu;
  return PW_OK;
}

int pw_page_reload(pw_page_table* t, int block, int page, const void* h_src, void* d_dst, void* copy_stream) {
  if (int e = check_block(t, block)) return e;
  BlockState& b = t->blocks[block];
  const int64_t bytes = page_bytes(b, page);
  if (bytes < 0) return pw::set_error(PW_ERR_INVALID_ARG, "block %d: no page %d", block, page);
  if (!d_dst || (reinterpret_cast<uintptr_t>(d_dst) & 15))
    return pw::set_error(PW_ERR_INVALID_ARG, "reload: device buffer must be non-NULL and 16-byte aligned");
  PageXfer& x = b.pages[page];
  if (x.xfer != kXferNone) return pw::set_error(PW_ERR_BUSY, "block %d: page %d has a transfer in flight", block, page);
  if (attached(b, page)) return pw::set_error(PW_ERR_INVALID_ARG, "block %d: page %d is already GPU-resident", block, page);
  const void* src = h_src ? h_src : (x.cpu ? x.host : nullptr);
  if (!src) return pw::set_error(PW_ERR_NOT_RESIDENT, "block %d: page %d has no host copy", block, page);
  if (!x.ev) PW_CUDA_TRY(cudaEventCreateWithFlags(&x.ev, cudaEventDisableTiming));
  cudaStream_t s = pw::as_stream(copy_stream);
  PW_CUDA_TRY(cudaMemcpyAsync(d_dst, src, static_cast<size_t>(bytes), cudaMemcpyHostToDevice, s));
  PW_CUDA_TRY(cudaEventRecord(x.ev, s));
  x.pending = d_dst;
  x.xfer = kXferToGpu;
  return PW_OK;
}

int pw_page_table_poll(pw_page_table* t, int* in_flight) {
  if (in_flight) *in_flight = 0;
  if (!t) return pw::set_error(PW_ERR_INVALID_ARG, "page table is NULL");
  int pending = 0;
  for (size_t bi = 0; bi < t->blocks.size(); ++bi) {
    BlockState& b = t->blocks[bi];
    for (int page = 0; page < kPages; ++page) {
      PageXfer& x = b.pages[page];
      if (x.xfer == kXferNone) continue;
      const cudaError_t r = cudaEventQuery(x.ev);
      if (r == cudaErrorNotReady) {
        ++pending;
        continue;
      }
      if (r != cudaSuccess) return pw::cuda_error(r, "cudaEventQuery (page transfer)");
      if (x.xfer == kXferToCpu) {
        x.cpu = true;
        if (!referenced(b, page) && attached(b, page)) {
          set_attached(b, page, nullptr);
          b.released_late |= 1ull << page;
        }
      } else {
        set_attached(b, page, x.pending);
        x.pending = nullptr;
      }
      x.xfer = kXferNone;
    }
  }
  if (in_flight) *in_flight = pending;
  return PW_OK;
}

int pw_page_table_take_released(pw_page_table* t, int block, uint64_t* released_mask) {
  if (released_mask) *released_mask = 0;
  if (int e = check_block(t, block)) return e;
  BlockState& b = t->blocks[block];
  if (released_mask) *released_mask = b.released_late;
  b.released_late = 0;
  return PW_OK;
}

int pw_page_state(const pw_page_table* t, int block, int page, int* state, const void** d_ptr, void** h_ptr) {
  if (state) *state = 0;
  if (d_ptr) *d_ptr = nullptr;
  if (h_ptr) *h_ptr = nullptr;
  if (int e = check_block(t, block)) return e;
  const BlockState& b = t->blocks[block];
  if (page_bytes(b, page) < 0) return pw::set_error(PW_ERR_INVALID_ARG, "block %d: no page %d", block, page);
  const PageXfer& x = b.pages[page];
  int st = 0;
  if (attached(b, page)) st |= PW_PAGE_GPU;
  if (x.cpu) st |= PW_PAGE_CPU;
  if (x.xfer == kXferToCpu) st |= PW_PAGE_TO_CPU;
  if (x.xfer == kXferToGpu) st |= PW_PAGE_TO_GPU;
  if (state) *state = st;
  if (d_ptr) *d_ptr = attached(b, page);
  if (h_ptr) *h_ptr = x.host;
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
