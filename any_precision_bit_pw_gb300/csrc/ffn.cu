// Host entry points of the fused mixed-precision MoE expert layer and of the
// any-precision linear test export: argument checks, workspace layout, path
// choice, launch.  The kernel body is ffn_stream.cuh, instantiated for token
// tiles of 16 and 64; ffn_common.cuh describes the work units.
//
// "PagedWeight" arXiv text, §3.3 (Fused Mixed-Precision MoE Kernel).
#include <mutex>

#include "ffn_common.cuh"
#include "route_block.cuh"

namespace {

using pw::BlockDesc;
using pw_ffn::Params;
using pw_ffn::kDecodeSplitCols;
using pw_ffn::kMaxE;

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

struct WsLayout {
  size_t ctr, gather, h, part, xp, total;
  int nsplit, split_cols;
};

int choose_path(int T, int E, int k, int requested) {
  if (requested == PW_PATH_DECODE || requested == PW_PATH_PREFILL) return requested;
  // average tokens per expert: from a few dozen on, down units take all of I
  // (no K split) and routing runs as its own launch
  return (static_cast<long long>(T) * k >= 48ll * E) ? PW_PATH_PREFILL : PW_PATH_DECODE;
}

WsLayout ws_layout(int T, int H, int I, int E, int k, int path) {
  WsLayout L{};
  const long long A = static_cast<long long>(T) * k;
  L.split_cols = path == PW_PATH_PREFILL ? I : kDecodeSplitCols;
  L.nsplit = (I + L.split_cols - 1) / L.split_cols;
  const size_t ctr_words = 2 + static_cast<size_t>(E) * L.nsplit + static_cast<size_t>(H) / 128;
  L.ctr = 0;
  L.gather = ctr_words * 4;   // [0] x-gather shares done, [1] CTAs done (prefill combine), [2] routed
  L.h = align256(L.gather + 12);
  L.part = L.h + align256(static_cast<size_t>(A) * I * 2);
  L.xp = L.part + align256(static_cast<size_t>(L.nsplit) * A * H * 4);
  L.total = L.xp + align256(static_cast<size_t>(A) * H * 2);
  return L;
}

// Token-tile width: 16 while experts average fewer than 12 tokens, 64 below
// 96, else 128.  Measured on the 8x7B shape: at 8 tokens per expert and fewer
// the 64-token kernel is 25-45 % slower; at 16 and more it is 10-13 % faster
// (it needs fewer token groups, each of which reads and dequantises the
// weights again).  128-token tiles halve the dequantisation again for
// prefill batches.
int tile_width(int T, int E, int k) {
  const long long A = static_cast<long long>(T) * k;
  return A < 12ll * E ? 16 : (A < 96ll * E ? 64 : 128);
}

// Width 2: the CUDA-core instance.
int launch_width(int width, const Params& p, cudaStream_t s, bool after_route = false) {
  switch (width) {
    case 2: return pw_ffn::launch_ffn_gemv(p, s, after_route);
    case 16: return pw_ffn::launch_ffn_t16(p, s, after_route);
    case 64: return pw_ffn::launch_ffn_t64(p, s, after_route);
    default: return pw_ffn::launch_ffn_t128(p, s, after_route);
  }
}

// Workspace of the path pw_moe_apl_ffn picks by itself for this size.
WsLayout ws_layout(int T, int H, int I, int E, int k) {
  return ws_layout(T, H, I, E, k, choose_path(T, E, k, PW_PATH_AUTO));
}

int validate_shape(int T, int H, int I, int E, int k) {
  if (T < 0 || H <= 0 || I <= 0 || E < 1 || E > kMaxE || k < 1 || k > 16 || k > E)
    return pw::set_error(PW_ERR_INVALID_ARG, "ffn: bad sizes T=%d H=%d I=%d E=%d k=%d", T, H, I, E, k);
  if (H % 128 || I % 128)
    return pw::set_error(PW_ERR_UNSUPPORTED, "ffn: H and I must be multiples of 128 (H=%d I=%d)", H, I);
  if (static_cast<long long>(T) * k > (1 << 24) || static_cast<long long>(T) * k * I > (1ll << 31) ||
      static_cast<long long>(T) * H > (1ll << 31))
    return pw::set_error(PW_ERR_UNSUPPORTED, "ffn: problem too large");
  return PW_OK;
}

// The linear test export's ticket counter (zeroed before each launch).
static __device__ uint32_t g_linear_ctr[2];

}  // namespace

extern "C" {

size_t pw_moe_apl_ffn_workspace(int T, int H, int I, int E, int k) {
  if (validate_shape(T, H, I, E, k) != PW_OK) return 0;
  const size_t a = ws_layout(T, H, I, E, k, PW_PATH_DECODE).total;
  const size_t b = ws_layout(T, H, I, E, k, PW_PATH_PREFILL).total;
  return a > b ? a : b;
}

}  // extern "C"

namespace {

// Shared by the fused entry points: checks, workspace layout, path choice and
// launch.  `routed`: the routing arrays are outputs, computed from d_logits in
// the same launch on the decode path and by a routing launch just before on
// the prefill path.  `L` > 1 (routed only): L consecutive independent layers
// starting at `layer`, each with T tokens and E routed experts, run as one
// layer of L*T tokens and L*(E+S) experts whose routing never crosses layers.
int ffn_launch(bool routed, const void* d_desc, int layer, int L, const uint16_t* d_x, const float* d_logits, int T,
               int H, int I, int E, int k, int32_t* d_ids, const float* d_w, const int32_t* d_offsets,
               const int32_t* d_perm, const int32_t* d_inv_perm, float* d_mass_accum, void* d_ws, size_t ws_bytes,
               uint16_t* d_y, int32_t* d_status, const pw_ffn_options* opts, void* stream) {
  // routed call: E and k count routed experts; the options add S shared
  // experts (ids E .. E+S-1, one slot per token each, weight 1), so the layer
  // runs over E + S experts and k + S slots per token
  const int S = (routed && opts) ? opts->shared_experts : 0;
  if (S < 0) return pw::set_error(PW_ERR_INVALID_ARG, "ffn: shared_experts %d", S);
  if (L < 1 || L > kMaxE || (L > 1 && !routed)) return pw::set_error(PW_ERR_INVALID_ARG, "ffn: layers %d", L);
  const int ER = E, kR = k;
  E += S;
  k += S;
  if (int e = validate_shape(T, H, I, E, k)) return e;
  if (static_cast<long long>(L) * E > kMaxE)
    return pw::set_error(PW_ERR_UNSUPPORTED, "ffn: %d layers x %d experts exceed %d", L, E, kMaxE);
  if (int e = validate_shape(L * T, H, I, L * E, k)) return e;
  if (layer < 0) return pw::set_error(PW_ERR_INVALID_ARG, "ffn: layer %d", layer);
  if (routed && T > 0 && !d_logits) return pw::set_error(PW_ERR_INVALID_ARG, "routed ffn: NULL logits");
  if (routed && (!d_ids || !d_offsets))
    return pw::set_error(PW_ERR_INVALID_ARG, "ffn: routed call needs ids and offsets");
  if (T == 0)
    return routed ? pw::route_layers(d_logits, L, 0, ER, kR, S, d_ids, const_cast<float*>(d_w),
                                     const_cast<int32_t*>(d_offsets), const_cast<int32_t*>(d_perm),
                                     const_cast<int32_t*>(d_inv_perm), d_mass_accum, pw::as_stream(stream))
                  : PW_OK;
  // the L layers as one: every count below is the total over the layers
  const int E1 = E, T1 = T;
  E *= L;
  T *= L;
  if (!d_desc || !d_x || !d_w || !d_offsets || !d_perm || !d_inv_perm || !d_y || !d_status || !d_ws)
    return pw::set_error(PW_ERR_INVALID_ARG, "ffn: NULL argument");
  if ((reinterpret_cast<uintptr_t>(d_desc) & 15) || (reinterpret_cast<uintptr_t>(d_x) & 15) ||
      (reinterpret_cast<uintptr_t>(d_y) & 7))
    return pw::set_error(PW_ERR_INVALID_ARG, "ffn: descriptor/x must be 16-byte aligned, y 8-byte aligned");
  pw_ffn_options o{};
  if (opts) o = *opts;
  if (o.kernel != PW_KERNEL_AUTO && o.kernel != PW_KERNEL_TENSOR && o.kernel != PW_KERNEL_CUDA_CORES)
    return pw::set_error(PW_ERR_INVALID_ARG, "ffn: kernel %d", o.kernel);
  const int path = choose_path(T, E, k, o.path);
  const WsLayout W = ws_layout(T, H, I, E, k, path);
  if (ws_bytes < W.total || (reinterpret_cast<uintptr_t>(d_ws) & 255))
    return pw::set_error(PW_ERR_WORKSPACE, "ffn: workspace needs %zu bytes, 256-byte aligned (got %zu)", W.total,
                         ws_bytes);
  cudaStream_t s = pw::as_stream(stream);
  char* ws = static_cast<char*>(d_ws);
  Params p{};
  p.desc = static_cast<const BlockDesc*>(d_desc) + static_cast<long long>(layer) * E1 * 2;
  p.x = d_x;
  p.y = d_y;
  p.w = d_w;
  p.offsets = d_offsets;
  p.perm = d_perm;
  p.inv_perm = d_inv_perm;
  p.T = T;
  p.H = H;
  p.I = I;
  p.E = E;
  p.k = k;
  p.A = T * k;
  p.nsplit = W.nsplit;
  p.split_cols = W.split_cols;
  p.ctr = reinterpret_cast<uint32_t*>(ws + W.ctr);
  p.h = reinterpret_cast<uint16_t*>(ws + W.h);
  p.part = reinterpret_cast<float*>(ws + W.part);
  p.xp = reinterpret_cast<uint16_t*>(ws + W.xp);
  p.gather_ctr = reinterpret_cast<uint32_t*>(ws + W.gather);
  // the whole grid combines after the last unit (measured faster than each
  // strip's last down unit combining it, by up to 8 % at 128 tokens)
  p.grid_combine = (o.flags & PW_FFN_FLAG_STRIP_COMBINE) ? 0 : 1;
  p.status = d_status;
  p.wait_ns = (o.wait_timeout_us ? o.wait_timeout_us : 2000000u) * 1000ull;
  p.flags = o.flags;
  p.linear = 0;
  const int width = o.kernel == PW_KERNEL_CUDA_CORES ? 2 : tile_width(T, E, k);
  if (routed && (path == PW_PATH_PREFILL || !pw_route::warp_routes(T1, E1, k))) {
    // batches that one warp does not route (more than 32 tokens or 8 experts
    // per layer): a routing launch comes first, so that the fused kernel
    // holds no CTA-wide routing code and its grid does not wait on one CTA;
    // it also zeroes the fused launch's counters, and the fused kernel starts
    // while it finishes
    if (int e = pw::route_layers(d_logits, L, T1, ER, kR, S, d_ids, const_cast<float*>(d_w),
                                 const_cast<int32_t*>(d_offsets), const_cast<int32_t*>(d_perm),
                                 const_cast<int32_t*>(d_inv_perm), d_mass_accum, s, p.ctr, W.h - W.ctr))
      return e;
    return launch_width(width, p, s, true);
  } else if (routed) {
    p.logits = d_logits;
    p.route_shared = S;
    p.route_layers = L;
    p.ids_out = d_ids;
    p.mass_accum = d_mass_accum;
  }
  PW_CUDA_TRY(cudaMemsetAsync(p.ctr, 0, W.h - W.ctr, s));
  return launch_width(width, p, s);
}

}  // namespace

extern "C" {

int pw_moe_apl_ffn_ex(const void* d_desc, int layer, const uint16_t* d_x, int T, int H, int I, int E, int k,
                      const int32_t* d_ids, const float* d_w, const int32_t* d_offsets, const int32_t* d_perm,
                      const int32_t* d_inv_perm, void* d_ws, size_t ws_bytes, uint16_t* d_y, int32_t* d_status,
                      const pw_ffn_options* opts, void* stream) {
  (void)d_ids;
  return ffn_launch(false, d_desc, layer, 1, d_x, nullptr, T, H, I, E, k, nullptr, d_w, d_offsets, d_perm,
                    d_inv_perm, nullptr, d_ws, ws_bytes, d_y, d_status, opts, stream);
}

int pw_moe_route_apl_ffn_ex(const void* d_desc, int layer, const uint16_t* d_x, const float* d_logits, int T, int H,
                            int I, int E, int k, int32_t* d_ids, float* d_w, int32_t* d_offsets, int32_t* d_perm,
                            int32_t* d_inv_perm, float* d_mass_accum, void* d_ws, size_t ws_bytes, uint16_t* d_y,
                            int32_t* d_status, const pw_ffn_options* opts, void* stream) {
  return ffn_launch(true, d_desc, layer, 1, d_x, d_logits, T, H, I, E, k, d_ids, d_w, d_offsets, d_perm, d_inv_perm,
                    d_mass_accum, d_ws, ws_bytes, d_y, d_status, opts, stream);
}

int pw_moe_route_apl_ffn_layers(const void* d_desc, int layer0, int L, const uint16_t* d_x, const float* d_logits,
                                int T, int H, int I, int E, int k, int32_t* d_ids, float* d_w, int32_t* d_offsets,
                                int32_t* d_perm, int32_t* d_inv_perm, float* d_mass_accum, void* d_ws,
                                size_t ws_bytes, uint16_t* d_y, int32_t* d_status, const pw_ffn_options* opts,
                                void* stream) {
  return ffn_launch(true, d_desc, layer0, L, d_x, d_logits, T, H, I, E, k, d_ids, d_w, d_offsets, d_perm, d_inv_perm,
                    d_mass_accum, d_ws, ws_bytes, d_y, d_status, opts, stream);
}

int pw_moe_route_apl_ffn(const void* d_desc, int layer, const uint16_t* d_x, const float* d_logits, int T, int H,
                         int I, int E, int k, int32_t* d_ids, float* d_w, int32_t* d_offsets, int32_t* d_perm,
                         int32_t* d_inv_perm, float* d_mass_accum, void* d_ws, size_t ws_bytes, uint16_t* d_y,
                         int32_t* d_status, void* stream) {
  return pw_moe_route_apl_ffn_ex(d_desc, layer, d_x, d_logits, T, H, I, E, k, d_ids, d_w, d_offsets, d_perm,
                                 d_inv_perm, d_mass_accum, d_ws, ws_bytes, d_y, d_status, nullptr, stream);
}

int pw_moe_apl_ffn(const void* d_desc, int layer, const uint16_t* d_x, int T, int H, int I, int E, int k,
                   const int32_t* d_ids, const float* d_w, const int32_t* d_offsets, const int32_t* d_perm,
                   const int32_t* d_inv_perm, void* d_ws, size_t ws_bytes, uint16_t* d_y, int32_t* d_status,
                   void* stream) {
  return pw_moe_apl_ffn_ex(d_desc, layer, d_x, T, H, I, E, k, d_ids, d_w, d_offsets, d_perm, d_inv_perm, d_ws,
                           ws_bytes, d_y, d_status, nullptr, stream);
}

int pw_apl_linear(const pw_page_table* t, int block, const uint16_t* d_x, int M, float* d_out, void* stream) {
  if (M < 0) return pw::set_error(PW_ERR_INVALID_ARG, "linear: M < 0");
  BlockDesc d;
  if (int e = pw::table_block(t, block, &d, 0)) return e;
  if (d.q < 2 || d.q > PW_MAX_BITS) return pw::set_error(PW_ERR_UNSUPPORTED, "linear: bitwidth %d", d.q);
  if (!d.lut) return pw::set_error(PW_ERR_NOT_RESIDENT, "linear: LUT %d not attached", d.q);
  if (M == 0) return PW_OK;
  if (!d_x || !d_out || (reinterpret_cast<uintptr_t>(d_x) & 15))
    return pw::set_error(PW_ERR_INVALID_ARG, "linear: NULL or misaligned argument");
  if (static_cast<long long>(M) * d.cols > (1ll << 31))
    return pw::set_error(PW_ERR_UNSUPPORTED, "linear: problem too large");
  cudaStream_t s = pw::as_stream(stream);
  void* ctr = nullptr;
  PW_CUDA_TRY(cudaGetSymbolAddress(&ctr, g_linear_ctr));
  PW_CUDA_TRY(cudaMemsetAsync(ctr, 0, sizeof(uint32_t) * 2, s));
  Params p{};
  p.lin = d;
  p.x = d_x;
  p.out = d_out;
  p.M = M;
  p.ctr = static_cast<uint32_t*>(ctr);
  p.status = nullptr;
  p.wait_ns = 2000000000ull;
  p.linear = 1;
  p.nsplit = 1;
  p.split_cols = d.cols;
  return launch_width(M <= 2 ? 2 : (M <= 16 ? 16 : (M <= 64 ? 64 : 128)), p, s);
}

}  // extern "C"

// Entry point for callers that cannot allocate device memory.  Its scratch is
// this fixed array; host code must not hand the array's name to a kernel (on
// the host it is only a stand-in symbol), so the device address is looked up
// once per device with cudaGetSymbolAddress and cached for the life of the
// process (a cudaDeviceReset makes the cached address stale; the header says
// so).
// ---------------------------------------------------------------------------
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[PW_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {};

int noalloc_scratch(void** out) {
  int dev = 0;
  PW_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return pw::set_error(PW_ERR_UNSUPPORTED, "noalloc: device %d", dev);
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    PW_CUDA_TRY(cudaGetSymbolAddress(&p, g_noalloc_scratch));
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return PW_OK;
}

}  // namespace

extern "C" int pw_moe_apl_ffn_noalloc(const void* d_desc, int layer, const uint16_t* d_x, int T, int H, int I, int E,
                                      int k, const int32_t* d_ids, const float* d_w, const int32_t* d_offsets,
                                      const int32_t* d_perm, const int32_t* d_inv_perm, uint16_t* d_y,
                                      int32_t* d_status, void* stream) {
  if (int e = validate_shape(T, H, I, E, k)) return e;
  const size_t need = ws_layout(T, H, I, E, k).total;
  if (need > PW_NOALLOC_SCRATCH_BYTES)
    return pw::set_error(PW_ERR_WORKSPACE,
                         "noalloc: this call needs %zu bytes of scratch but the built-in array holds %u "
                         "(use pw_moe_apl_ffn with a caller workspace)",
                         need, PW_NOALLOC_SCRATCH_BYTES);
  void* scratch = nullptr;
  if (int e = noalloc_scratch(&scratch)) return e;
  // The regular path zeroes the counters it needs and writes every h and
  // partial value before reading it, so stale contents are harmless.
  return pw_moe_apl_ffn(d_desc, layer, d_x, T, H, I, E, k, d_ids, d_w, d_offsets, d_perm, d_inv_perm, scratch,
                        PW_NOALLOC_SCRATCH_BYTES, d_y, d_status, stream);
}
