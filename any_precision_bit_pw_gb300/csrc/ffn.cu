// Fused mixed-precision MoE expert layer (decode path) and the any-precision
// linear test export.
//
// "PagedWeight" arXiv text, §3.3 (Fused Mixed-Precision MoE Kernel): one
// kernel reads the weight pages directly, follows the committed bitwidth of
// every gate_up and down linear-block, and does the expert activation, the down
// projection and the output accumulation in one launch.
//
// Structure: a persistent launch (one wave of CTAs) whose warps take work
// units from an atomic ticket counter.  Tickets are issued in order: every
// gate_up unit of every active expert first, then every down unit.  A warp only
// takes a new ticket after finishing its previous unit, so when a down unit
// waits for the gate_up units it depends on, each of those is already held by
// a running warp and will finish: the waits always end (and are also bounded
// in time, after which the kernel reports PW_ERR_TIMEOUT and returns).
//
//  gate_up unit (expert e, strip s): rows 8s..8s+7 of the gate and of the up
//    projection over all H columns, for all of e's tokens; epilogue
//    h = silu(gate) * up rounded to fp16 into the workspace, in expert order.
//  down unit (expert e, split p, strip s): rows 8s..8s+7 and H/2+8s..+7 of down
//    over one K-split of I; fp32 partial sums into the workspace.
//  combine: the last down unit to finish a strip (over all experts and
//    splits) forms y[t][rows] = sum_j w[t][j] * sum_p partial[p][pos(t,j)][row]
//    in a fixed order (reproducible), rounds to fp16 and writes y.
#include <cuda_fp16.h>

#include <mutex>

#include "apl_core.cuh"

namespace {

using pw::BlockDesc;
using pw::kNtMax;

constexpr int kThreads = 384;
constexpr int kWarps = kThreads / 32;
constexpr int kSplitTiles = 8;  // down K-split: 2048 columns of I
constexpr int kMaxE = 256;
constexpr size_t kLutSmemPerWarp = pw::kLutRowsPerWarp * pw::kLutMaxEntries * sizeof(uint16_t);
constexpr size_t kSmemPerWarp = kLutSmemPerWarp + pw::kRingBytesPerWarp;
constexpr size_t kSmemBytes = kWarps * kSmemPerWarp;

struct FfnParams {
  const BlockDesc* desc;  // this layer's 2E descriptors
  const uint16_t* x;
  uint16_t* y;
  const float* w;
  const int32_t* offsets;
  const int32_t* perm;
  const int32_t* inv_perm;
  int T, H, I, E, k, A;
  int nsplit;
  uint16_t* h;      // [A][I] fp16, expert order
  float* part;      // [nsplit][A][H] fp32
  uint32_t* ctr;    // [0] ticket, [1] abort, [2, 2+E*nsplit) gate_up done, then [H/16] strip arrivals
  int32_t* status;
  uint64_t wait_ns;
  uint32_t flags;
};

__device__ __forceinline__ void report(int32_t* status, int code) { atomicCAS(status, 0, code); }

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

__device__ __forceinline__ bool desc_ok(const BlockDesc& d, int rows, int cols) {
  if (d.q < 2 || d.q > PW_MAX_BITS || d.rows != rows || d.cols != cols || d.lut == nullptr) return false;
  for (int p = 0; p < d.q; ++p)
    if (d.planes[p] == nullptr) return false;
  return true;
}

template <int Q>
__device__ void gate_up_q(const FfnParams& p, const BlockDesc& d, int off, int ne, int strip, uint16_t* lut_s,
                          uint32_t ring_s) {
  const int lane = static_cast<int>(pw::lane_id());
  const int g = lane >> 2, c = lane & 3;
  pw::load_strip_lut<Q>(d.lut, p.I, strip, lut_s);
  __syncwarp();
  for (int tb = 0; tb < ne; tb += 8 * kNtMax) {
    const int nt_count = min(kNtMax, (ne - tb + 7) / 8);
    int brow[kNtMax];
#pragma unroll
    for (int nt = 0; nt < kNtMax; ++nt) {
      const int tl = min(tb + nt * 8 + g, ne - 1);
      brow[nt] = (__ldg(p.perm + off + tl) / p.k) * p.H;
    }
    float acc[kNtMax][4];
#pragma unroll
    for (int nt = 0; nt < kNtMax; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[nt][i] = 0.f;
    pw::strip_mainloop<Q, false>(d, strip, 0, p.H / pw::kTileCols, lut_s, ring_s, p.x, brow, nt_count, acc);
    const int m = strip * 8 + g;
#pragma unroll
    for (int nt = 0; nt < kNtMax; ++nt) {
      if (nt < nt_count) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int tl = tb + nt * 8 + 2 * c + i;
          if (tl < ne) {
            const float hv = silu(acc[nt][i]) * acc[nt][2 + i];
            p.h[static_cast<long long>(off + tl) * p.I + m] = __half_as_ushort(__float2half_rn(hv));
          }
        }
      }
    }
  }
  __syncwarp();
}

template <int Q>
__device__ void down_q(const FfnParams& p, const BlockDesc& d, int off, int ne, int split, int strip,
                       uint16_t* lut_s, uint32_t ring_s) {
  const int lane = static_cast<int>(pw::lane_id());
  const int g = lane >> 2, c = lane & 3;
  pw::load_strip_lut<Q>(d.lut, p.H / 2, strip, lut_s);
  __syncwarp();
  const int t0 = split * kSplitTiles;
  const int t1 = min(t0 + kSplitTiles, p.I / pw::kTileCols);
  for (int tb = 0; tb < ne; tb += 8 * kNtMax) {
    const int nt_count = min(kNtMax, (ne - tb + 7) / 8);
    int brow[kNtMax];
#pragma unroll
    for (int nt = 0; nt < kNtMax; ++nt) {
      const int tl = min(tb + nt * 8 + g, ne - 1);
      brow[nt] = (off + tl) * p.I;
    }
    float acc[kNtMax][4];
#pragma unroll
    for (int nt = 0; nt < kNtMax; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[nt][i] = 0.f;
    pw::strip_mainloop<Q, true>(d, strip, t0, t1, lut_s, ring_s, p.h, brow, nt_count, acc);
    const int r0 = strip * 8 + g, r1 = p.H / 2 + strip * 8 + g;
#pragma unroll
    for (int nt = 0; nt < kNtMax; ++nt) {
      if (nt < nt_count) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int tl = tb + nt * 8 + 2 * c + i;
          if (tl < ne) {
            float* dst = p.part + (static_cast<long long>(split) * p.A + off + tl) * p.H;
            dst[r0] = acc[nt][i];
            dst[r1] = acc[nt][2 + i];
          }
        }
      }
    }
  }
  __syncwarp();
}

// y rows of one strip for every token, in a fixed summation order.
__device__ void combine_strip(const FfnParams& p, int strip) {
  const int lane = static_cast<int>(pw::lane_id());
  const int n_items = p.T * 16;
  for (int it = lane; it < n_items; it += 32) {
    const int t = it >> 4, ri = it & 15;
    const int row = ri < 8 ? strip * 8 + ri : p.H / 2 + strip * 8 + (ri - 8);
    float acc = 0.f;
    for (int j = 0; j < p.k; ++j) {
      const int slot = t * p.k + j;
      const int pos = __ldg(p.inv_perm + slot);
      const float wt = __ldg(p.w + slot);
      float s = 0.f;
      for (int sp = 0; sp < p.nsplit; ++sp) s += __ldcg(p.part + (static_cast<long long>(sp) * p.A + pos) * p.H + row);
      acc += wt * s;
    }
    p.y[static_cast<long long>(t) * p.H + row] = __half_as_ushort(__float2half_rn(acc));
  }
}

// Bounded wait of lane 0 until *ctr >= want; false if it ran out or the launch
// was aborted (then the unit is skipped and the status word says why).
__device__ bool wait_for(const FfnParams& p, const uint32_t* ctr, uint32_t want) {
  bool ok = true;
  if (pw::lane_id() == 0) {
    const uint64_t t0 = pw::global_ns();
    while (pw::ld_acquire_u32(ctr) < want) {
      if (*reinterpret_cast<volatile const uint32_t*>(p.ctr + 1) != 0u) {
        ok = false;
        break;
      }
      if (pw::global_ns() - t0 > p.wait_ns) {
        report(p.status, PW_ERR_TIMEOUT);
        atomicExch(p.ctr + 1, 1u);
        ok = false;
        break;
      }
      __nanosleep(256);
    }
  }
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

__global__ void __launch_bounds__(kThreads) ffn_decode_kernel(FfnParams p) {
  extern __shared__ __align__(16) uint16_t smem_lut[];
  __shared__ int s_act[kMaxE];
  __shared__ int s_nact;
  if (threadIdx.x == 0) {
    int n = 0;
    for (int e = 0; e < p.E; ++e)
      if (__ldg(p.offsets + e + 1) > __ldg(p.offsets + e)) s_act[n++] = e;
    s_nact = n;
  }
  __syncthreads();
  const int nact = s_nact;
  const int lane = static_cast<int>(pw::lane_id());
  const int warp = threadIdx.x >> 5;
  uint16_t* lut_s = smem_lut + warp * (kSmemPerWarp / sizeof(uint16_t));
  const uint32_t ring_s = static_cast<uint32_t>(__cvta_generic_to_shared(lut_s + kLutSmemPerWarp / sizeof(uint16_t)));
  const uint32_t gu_strips = static_cast<uint32_t>(p.I / 8);
  const uint32_t dn_strips = static_cast<uint32_t>(p.H / 16);
  const uint32_t n_gu = static_cast<uint32_t>(nact) * gu_strips;
  const uint32_t n_dn = static_cast<uint32_t>(nact) * dn_strips * static_cast<uint32_t>(p.nsplit);
  uint32_t* gu_done = p.ctr + 2;
  uint32_t* arrive = gu_done + p.E * p.nsplit;
  const int split_cols = kSplitTiles * pw::kTileCols;

  for (;;) {
    uint32_t u = 0;
    if (lane == 0) u = atomicAdd(p.ctr, 1u);
    u = __shfl_sync(0xffffffffu, u, 0);
    if (u >= n_gu + n_dn) break;
    if (u < n_gu) {
      const int e = s_act[u / gu_strips];
      const int strip = static_cast<int>(u % gu_strips);
      const BlockDesc d = p.desc[2 * e];
      const int off = __ldg(p.offsets + e), ne = __ldg(p.offsets + e + 1) - off;
      if (!desc_ok(d, 2 * p.I, p.H)) {
        if (lane == 0) report(p.status, d.q == 0 ? PW_ERR_NOT_RESIDENT : PW_ERR_UNSUPPORTED);
      } else {
        switch (d.q) {
          case 2: gate_up_q<2>(p, d, off, ne, strip, lut_s, ring_s); break;
          case 3: gate_up_q<3>(p, d, off, ne, strip, lut_s, ring_s); break;
          case 4: gate_up_q<4>(p, d, off, ne, strip, lut_s, ring_s); break;
          case 5: gate_up_q<5>(p, d, off, ne, strip, lut_s, ring_s); break;
          case 6: gate_up_q<6>(p, d, off, ne, strip, lut_s, ring_s); break;
          case 7: gate_up_q<7>(p, d, off, ne, strip, lut_s, ring_s); break;
          default: gate_up_q<8>(p, d, off, ne, strip, lut_s, ring_s); break;
        }
      }
      const bool drop = (p.flags & PW_FFN_FLAG_TEST_DROP_ONE_ARRIVAL) && u == 0;
      if (lane == 0 && !drop) {
        __threadfence();
        atomicAdd(gu_done + e * p.nsplit + (strip * 8) / split_cols, 1u);
      }
    } else {
      const uint32_t v = u - n_gu;
      const uint32_t per = dn_strips * static_cast<uint32_t>(p.nsplit);
      const int e = s_act[v / per];
      const uint32_t r = v % per;
      const int split = static_cast<int>(r / dn_strips);
      const int strip = static_cast<int>(r % dn_strips);
      const int c0 = split * split_cols;
      const uint32_t want = static_cast<uint32_t>((min(c0 + split_cols, p.I) - c0) / 8);
      if (!wait_for(p, gu_done + e * p.nsplit + split, want)) continue;
      const BlockDesc d = p.desc[2 * e + 1];
      const int off = __ldg(p.offsets + e), ne = __ldg(p.offsets + e + 1) - off;
      if (!desc_ok(d, p.H, p.I)) {
        if (lane == 0) report(p.status, d.q == 0 ? PW_ERR_NOT_RESIDENT : PW_ERR_UNSUPPORTED);
      } else {
        switch (d.q) {
          case 2: down_q<2>(p, d, off, ne, split, strip, lut_s, ring_s); break;
          case 3: down_q<3>(p, d, off, ne, split, strip, lut_s, ring_s); break;
          case 4: down_q<4>(p, d, off, ne, split, strip, lut_s, ring_s); break;
          case 5: down_q<5>(p, d, off, ne, split, strip, lut_s, ring_s); break;
          case 6: down_q<6>(p, d, off, ne, split, strip, lut_s, ring_s); break;
          case 7: down_q<7>(p, d, off, ne, split, strip, lut_s, ring_s); break;
          default: down_q<8>(p, d, off, ne, split, strip, lut_s, ring_s); break;
        }
      }
      uint32_t last = 0;
      if (lane == 0) {
        __threadfence();
        last = (atomicAdd(arrive + strip, 1u) == static_cast<uint32_t>(nact * p.nsplit) - 1u) ? 1u : 0u;
        if (last) __threadfence();
      }
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last) combine_strip(p, strip);
    }
  }
}

// ---------------------------------------------------------------------------
// Any-precision linear (test export): out[m][n] = sum_j W[n][j] x[m][j].
// ---------------------------------------------------------------------------
template <int Q>
__device__ void linear_q(const BlockDesc& d, const uint16_t* x, int M, float* out, int strip, int grp,
                         uint16_t* lut_s, uint32_t ring_s) {
  const int lane = static_cast<int>(pw::lane_id());
  const int g = lane >> 2, c = lane & 3;
  pw::load_strip_lut<Q>(d.lut, d.rows / 2, strip, lut_s);
  __syncwarp();
  const int tb = grp * 8 * kNtMax;
  const int nt_count = min(kNtMax, (M - tb + 7) / 8);
  int brow[kNtMax];
#pragma unroll
  for (int nt = 0; nt < kNtMax; ++nt) brow[nt] = min(tb + nt * 8 + g, M - 1) * d.cols;
  float acc[kNtMax][4];
#pragma unroll
  for (int nt = 0; nt < kNtMax; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[nt][i] = 0.f;
  pw::strip_mainloop<Q, false>(d, strip, 0, d.cols / pw::kTileCols, lut_s, ring_s, x, brow, nt_count, acc);
  const int r0 = strip * 8 + g, r1 = d.rows / 2 + strip * 8 + g;
#pragma unroll
  for (int nt = 0; nt < kNtMax; ++nt) {
    if (nt < nt_count) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int m = tb + nt * 8 + 2 * c + i;
        if (m < M) {
          out[static_cast<long long>(m) * d.rows + r0] = acc[nt][i];
          out[static_cast<long long>(m) * d.rows + r1] = acc[nt][2 + i];
        }
      }
    }
  }
}

__global__ void __launch_bounds__(kThreads) linear_kernel(BlockDesc d, const uint16_t* x, int M, float* out) {
  extern __shared__ __align__(16) uint16_t smem_lut[];
  const int warp = threadIdx.x >> 5;
  uint16_t* lut_s = smem_lut + warp * (kSmemPerWarp / sizeof(uint16_t));
  const uint32_t ring_s = static_cast<uint32_t>(__cvta_generic_to_shared(lut_s + kLutSmemPerWarp / sizeof(uint16_t)));
  const int strips = d.rows / 16;
  const int groups = (M + 8 * kNtMax - 1) / (8 * kNtMax);
  const long long unit = static_cast<long long>(blockIdx.x) * kWarps + warp;
  if (unit >= static_cast<long long>(strips) * groups) return;
  const int strip = static_cast<int>(unit % strips);
  const int grp = static_cast<int>(unit / strips);
  switch (d.q) {
    case 2: linear_q<2>(d, x, M, out, strip, grp, lut_s, ring_s); break;
    case 3: linear_q<3>(d, x, M, out, strip, grp, lut_s, ring_s); break;
    case 4: linear_q<4>(d, x, M, out, strip, grp, lut_s, ring_s); break;
    case 5: linear_q<5>(d, x, M, out, strip, grp, lut_s, ring_s); break;
    case 6: linear_q<6>(d, x, M, out, strip, grp, lut_s, ring_s); break;
    case 7: linear_q<7>(d, x, M, out, strip, grp, lut_s, ring_s); break;
    default: linear_q<8>(d, x, M, out, strip, grp, lut_s, ring_s); break;
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

struct WsLayout {
  size_t ctr, h, part, total;
  int nsplit;
};

WsLayout ws_layout(int T, int H, int I, int E, int k) {
  WsLayout L{};
  const long long A = static_cast<long long>(T) * k;
  const int split_cols = kSplitTiles * pw::kTileCols;
  L.nsplit = (I + split_cols - 1) / split_cols;
  const size_t ctr_words = 2 + static_cast<size_t>(E) * L.nsplit + static_cast<size_t>(H) / 16;
  L.ctr = 0;
  L.h = align256(ctr_words * 4);
  L.part = L.h + align256(static_cast<size_t>(A) * I * 2);
  L.total = L.part + align256(static_cast<size_t>(L.nsplit) * A * H * 4);
  return L;
}

int validate_shape(int T, int H, int I, int E, int k) {
  if (T < 0 || H <= 0 || I <= 0 || E < 1 || E > kMaxE || k < 1 || k > 8 || k > E)
    return pw::set_error(PW_ERR_INVALID_ARG, "ffn: bad sizes T=%d H=%d I=%d E=%d k=%d", T, H, I, E, k);
  if (H % pw::kTileCols || I % pw::kTileCols)
    return pw::set_error(PW_ERR_UNSUPPORTED, "ffn: H and I must be multiples of 256 (H=%d I=%d)", H, I);
  if (static_cast<long long>(T) * k > (1 << 24) || static_cast<long long>(H) * I > (1ll << 31))
    return pw::set_error(PW_ERR_UNSUPPORTED, "ffn: problem too large");
  return PW_OK;
}

int sm_count_cached() {
  static int count = 0;
  if (count == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  }
  return count;
}

int set_smem_attr(const void* fn, size_t bytes) {
  PW_CUDA_TRY(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes)));
  return PW_OK;
}

}  // namespace

extern "C" {

size_t pw_moe_apl_ffn_workspace(int T, int H, int I, int E, int k) {
  if (validate_shape(T, H, I, E, k) != PW_OK) return 0;
  return ws_layout(T, H, I, E, k).total;
}

int pw_moe_apl_ffn_ex(const void* d_desc, int layer, const uint16_t* d_x, int T, int H, int I, int E, int k,
                      const int32_t* d_ids, const float* d_w, const int32_t* d_offsets, const int32_t* d_perm,
                      const int32_t* d_inv_perm, void* d_ws, size_t ws_bytes, uint16_t* d_y, int32_t* d_status,
                      const pw_ffn_options* opts, void* stream) {
  (void)d_ids;
  if (int e = validate_shape(T, H, I, E, k)) return e;
  if (layer < 0) return pw::set_error(PW_ERR_INVALID_ARG, "ffn: layer %d", layer);
  if (T == 0) return PW_OK;
  if (!d_desc || !d_x || !d_w || !d_offsets || !d_perm || !d_inv_perm || !d_y || !d_status || !d_ws)
    return pw::set_error(PW_ERR_INVALID_ARG, "ffn: NULL argument");
  if ((reinterpret_cast<uintptr_t>(d_desc) & 15) || (reinterpret_cast<uintptr_t>(d_x) & 15) ||
      (reinterpret_cast<uintptr_t>(d_y) & 3))
    return pw::set_error(PW_ERR_INVALID_ARG, "ffn: descriptor/x must be 16-byte aligned, y 4-byte aligned");
  const WsLayout L = ws_layout(T, H, I, E, k);
  if (ws_bytes < L.total || (reinterpret_cast<uintptr_t>(d_ws) & 255))
    return pw::set_error(PW_ERR_WORKSPACE, "ffn: workspace needs %zu bytes, 256-byte aligned (got %zu)", L.total,
                         ws_bytes);
  pw_ffn_options o{};
  if (opts) o = *opts;
  if (o.path == PW_PATH_PREFILL) return pw::set_error(PW_ERR_UNSUPPORTED, "ffn: prefill path not built yet");
  cudaStream_t s = pw::as_stream(stream);
  char* ws = static_cast<char*>(d_ws);
  FfnParams p{};
  p.desc = static_cast<const BlockDesc*>(d_desc) + static_cast<long long>(layer) * E * 2;
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
  p.nsplit = L.nsplit;
  p.ctr = reinterpret_cast<uint32_t*>(ws + L.ctr);
  p.h = reinterpret_cast<uint16_t*>(ws + L.h);
  p.part = reinterpret_cast<float*>(ws + L.part);
  p.status = d_status;
  p.wait_ns = (o.wait_timeout_us ? o.wait_timeout_us : 2000000u) * 1000ull;
  p.flags = o.flags;

  static bool attr_done = false;
  if (!attr_done) {
    if (int e = set_smem_attr(reinterpret_cast<const void*>(ffn_decode_kernel), kSmemBytes)) return e;
    attr_done = true;
  }
  int per_sm = 0;
  PW_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ffn_decode_kernel, kThreads, kSmemBytes));
  const int sms = sm_count_cached();
  if (per_sm < 1 || sms < 1) return pw::set_error(PW_ERR_CUDA, "ffn: kernel cannot be resident (occupancy 0)");
  PW_CUDA_TRY(cudaMemsetAsync(p.ctr, 0, L.h - L.ctr, s));
  ffn_decode_kernel<<<sms * per_sm, kThreads, kSmemBytes, s>>>(p);
  PW_CUDA_TRY(cudaGetLastError());
  return PW_OK;
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
  if (!d_x || !d_out || (reinterpret_cast<uintptr_t>(d_x) & 3))
    return pw::set_error(PW_ERR_INVALID_ARG, "linear: NULL or misaligned argument");
  static bool attr_done = false;
  if (!attr_done) {
    if (int e = set_smem_attr(reinterpret_cast<const void*>(linear_kernel), kSmemBytes)) return e;
    attr_done = true;
  }
  const long long units = static_cast<long long>(d.rows / 16) * ((M + 8 * kNtMax - 1) / (8 * kNtMax));
  const long long blocks = (units + kWarps - 1) / kWarps;
  linear_kernel<<<static_cast<unsigned>(blocks), kThreads, kSmemBytes, pw::as_stream(stream)>>>(d, d_x, M, d_out);
  PW_CUDA_TRY(cudaGetLastError());
  return PW_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Entry point for callers that cannot allocate device memory.  Its scratch is
// this fixed array; host code must not hand the array's name to a kernel (on
// the host it is only a stand-in symbol), so the device address is looked up
// once per device with cudaGetSymbolAddress and cached.
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
