// Shared pieces of the fused MoE layer kernels: parameters, work units and
// their scheduling, and the combine step.
//
// "PagedWeight" arXiv text, §3.3 (Fused Mixed-Precision MoE Kernel): one
// kernel follows the committed bitwidth of every gate_up and down
// linear-block and runs the experts' gate_up with SiLU·mul, their down
// projection and the weighted sum of their outputs in one launch.
//
// Scheduling: a persistent launch (one CTA per SM) whose CTAs take work units
// from an atomic ticket counter.  Tickets are issued in order: every gate_up
// unit of every active expert first, then every down unit.  A CTA only takes a
// new ticket after finishing its previous unit, so when a down unit waits for
// the gate_up units it depends on, each of those is held by a running CTA and
// will finish; the wait is also bounded in time (PW_ERR_TIMEOUT).
//
// A unit is one 128-row strip of one block, one group of at most NMAX of the
// expert's tokens, and a K range:
//   gate_up (expert e, strip s, group g): all H columns; rows 64s..64s+63 of
//     the gate and of the up projection; epilogue h = silu(gate) * up,
//     rounded to fp16, into the workspace (expert-ordered positions).
//   down (expert e, split p, strip s, group g): one K-split of I; fp32
//     partial sums into the workspace.
//   combine: the last down unit of a strip (over experts, splits and groups)
//     forms y[t][rows] = sum_j w[t][j] * sum_p partial[p][pos(t,j)][row] in a
//     fixed order, rounds to fp16 and writes y.
#pragma once

#include <cuda_fp16.h>

#include "dequant.cuh"
#include "pw_internal.h"

namespace pw_ffn {

using pw::BlockDesc;

constexpr int kDeqWarps = 4;                // per group: one warp per TMEM lane quadrant
constexpr int kDeqThreads = 128;
constexpr int kAStages = 4;
constexpr int kACols = pw::kStageK / 2;     // 32 TMEM columns (fp16 pairs) per stage
constexpr int kDCol = kAStages * kACols;    // accumulator columns start here (per group)
constexpr int kRingBytes = 32768;           // per group: plane staging ring [slot][plane][pos][16 B]
constexpr int kDecodeSplitCols = 3072;      // down K-split of the decode path (24 tiles; measured best of 2048, 3072, 4096)
constexpr int kMaxE = 256;
constexpr int kBarsPerGroup = 16;

enum UnitKind : int { kNone = -1, kGateUp = 0, kDown = 1, kLinear = 2 };

struct Params {
  const BlockDesc* desc;   // this layer's 2E descriptors (fused mode)
  BlockDesc lin;           // the block (linear mode)
  const uint16_t* x;
  uint16_t* y;
  float* out;              // linear mode output [M][rows]
  const float* w;
  const int32_t* offsets;
  const int32_t* perm;
  const int32_t* inv_perm;
  int T, H, I, E, k, A, M;
  int nsplit, split_cols;
  uint16_t* h;
  float* part;
  uint16_t* xp;            // decode path: x rows in expert order [A][H]
  uint32_t* ctr;           // [0] ticket, [1] abort, [2, 2+E*nsplit) gate_up done, then strip arrivals
  uint32_t* gather_ctr;    // CTAs that finished their share of xp; [1]: CTAs done with all units;
                           // [2]: routing arrays written (routed call)
  int grid_combine;        // 1: every CTA combines after the last unit; 0: a strip's last down unit does
  // Routed call (routing in the same launch): CTA 0 computes ids, w, offsets,
  // perm and inv_perm from the logits and publishes them through
  // gather_ctr[2]; NULL logits: the routing arrays are inputs.  The kernels
  // read offsets, perm, inv_perm and w with ordinary (coherent) loads, not
  // the read-only path, because a routed call writes them in the same launch.
  const float* logits;
  int32_t* ids_out;
  float* mass_accum;
  int route_shared;        // shared experts: the last route_shared of each layer's experts, the last of k slots
  int route_layers;        // routed call over this many independent layers (T and E are the totals: each
                           // layer has T / route_layers tokens and E / route_layers experts)
  int32_t* status;
  uint64_t wait_ns;
  uint32_t flags;
  int linear;
};

struct Unit {
  int kind, e, strip, split, tg, off, nrows, npad, q, st0, nst, skip, combine;
  const BlockDesc* d;
};

struct Shared {            // small per-CTA state (static shared memory)
  Unit u;
  uint32_t tmem;
  int nact;
  int act[kMaxE];
  int ntg[kMaxE];
  int cum_gu[kMaxE + 1];
  int cum_dn[kMaxE + 1];
  int arrivals_per_strip;
  int abort;
};

// Shared-memory carve-up of one CTA (computed at kernel start).
struct Smem {
  uint8_t* b_ring;       // G x kBStages x kBStageBytes, 1024-aligned
  uint8_t* plane_ring;   // G x kRingBytes
  float* xch;            // group-1 partial sums [token][pos]
  uint32_t bar;          // G x kBarsPerGroup mbarriers (shared address)
  int* rows;             // G x NMAX B-row offsets
  uint32_t lut_region;   // 64 KB-aligned LUT region (shared address)
};

__device__ __forceinline__ void report(int32_t* status, int code) {
  if (status) atomicCAS(status, 0, code);
}
__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

__device__ __forceinline__ int strip_pos_row(int strip, int pos, int half_rows) {
  const int w = pos >> 5, i = pos & 31;
  return (i >> 4) * half_rows + strip * 64 + 16 * w + (i & 15);
}

__device__ __forceinline__ bool desc_ok(const BlockDesc& d, int rows, int cols) {
  if (d.q < 2 || d.q > PW_MAX_BITS || d.rows != rows || d.cols != cols || d.lut == nullptr) return false;
  for (int p = 0; p < d.q; ++p)
    if (d.planes[p] == nullptr) return false;
  return true;
}

// ---------------------------------------------------------------------------
// Unit scheduling (thread 0)
// ---------------------------------------------------------------------------
// `offs`: the expert offsets (E + 1 values), staged in shared memory.
template <int NMAX>
__device__ void setup_schedule(const Params& p, const int* offs, Shared& sh) {
  sh.cum_gu[0] = 0;
  sh.cum_dn[0] = 0;
  if (p.linear) {
    sh.nact = 0;
    sh.arrivals_per_strip = 0;
    return;
  }
  int n = 0, gu = 0, dn = 0, arr = 0;
  const int gu_strips = 2 * p.I / 128, dn_strips = p.H / 128;
  // the offsets must run from 0 to A without decreasing, or no unit is run
  // (a unit's rows are read and written at these offsets)
  bool offsets_ok = offs[0] == 0 && offs[p.E] == p.A;
  for (int e = 0; e < p.E && offsets_ok; ++e) offsets_ok = offs[e + 1] >= offs[e];
  if (!offsets_ok) {
    report(p.status, PW_ERR_INVALID_ARG);
    sh.nact = 0;
    sh.arrivals_per_strip = 0;
    return;
  }
  for (int e = 0; e < p.E; ++e) {
    const int ne = offs[e + 1] - offs[e];
    if (ne <= 0) continue;
    const int g = (ne + NMAX - 1) / NMAX;
    sh.act[n] = e;
    sh.ntg[n] = g;
    gu += gu_strips * g;
    dn += p.nsplit * dn_strips * g;
    arr += p.nsplit * g;
    ++n;
    sh.cum_gu[n] = gu;
    sh.cum_dn[n] = dn;
  }
  sh.nact = n;
  sh.arrivals_per_strip = arr;
}

// The active expert whose run of units holds unit v: the largest i < n with
// cum[i] <= v, for non-decreasing cum[0..n] with cum[0] = 0 <= v < cum[n]
// (binary search: up to 256 active experts).
__device__ __forceinline__ int last_at_most(const int* cum, int n, int v) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cum[mid] <= v) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Strip and token group of the r-th unit of a block of `strips` strips x
// `groups` token groups: tickets run through blocks of kStripRun strips, token
// group by token group, so a strip's planes and LUT are read again by its next
// token group about kStripRun units later, while they are still in L2 (32
// strips of 8-bit planes at K = 16384 are 64 MB), and not at the same time by
// neighbouring CTAs.
constexpr int kStripRun = 32;
__device__ __forceinline__ void strip_group(int r, int strips, int groups, int& strip, int& tg) {
  const int run = r / (kStripRun * groups);
  const int first = run * kStripRun;
  const int n = min(kStripRun, strips - first);
  const int w = r - first * groups;
  tg = w / n;
  strip = first + w % n;
}

// Fetch and decode the next unit into sh.u (thread 0 only).
template <int NMAX>
__device__ void next_unit(const Params& p, Shared& sh) {
  Unit u{};
  u.kind = kNone;
  u.combine = -1;
  if (sh.abort || *reinterpret_cast<volatile uint32_t*>(p.ctr + 1) != 0u) {
    sh.u = u;
    return;
  }
  const uint32_t t = atomicAdd(p.ctr, 1u);
  if (p.linear) {
    const BlockDesc& d = p.lin;
    const int strips = d.rows / 128, groups = (p.M + NMAX - 1) / NMAX;
    if (t < static_cast<uint32_t>(strips * groups)) {
      u.kind = kLinear;
      strip_group(static_cast<int>(t), strips, groups, u.strip, u.tg);
      u.off = 0;
      u.nrows = min(NMAX, p.M - u.tg * NMAX);
      u.npad = ((u.nrows + 15) / 16) * 16;
      u.q = d.q;
      u.st0 = 0;
      u.nst = d.cols / pw::kStageK;
      u.d = &p.lin;
    }
    sh.u = u;
    return;
  }
  const int n_gu = sh.cum_gu[sh.nact], n_dn = sh.cum_dn[sh.nact];
  const int gu_strips = 2 * p.I / 128, dn_strips = p.H / 128;
  int ai = 0;
  if (t < static_cast<uint32_t>(n_gu)) {
    ai = last_at_most(sh.cum_gu, sh.nact, static_cast<int>(t));
    const int rem = static_cast<int>(t) - sh.cum_gu[ai];
    u.kind = kGateUp;
    u.e = sh.act[ai];
    strip_group(rem, gu_strips, sh.ntg[ai], u.strip, u.tg);
    u.split = (u.strip * 64) / p.split_cols;
    u.d = p.desc + 2 * u.e;
    u.st0 = 0;
    u.nst = p.H / pw::kStageK;
  } else if (t < static_cast<uint32_t>(n_gu + n_dn)) {
    const int v = static_cast<int>(t) - n_gu;
    ai = last_at_most(sh.cum_dn, sh.nact, v);
    const int rem = v - sh.cum_dn[ai];
    u.kind = kDown;
    u.e = sh.act[ai];
    const int per_split = dn_strips * sh.ntg[ai];
    u.split = rem / per_split;
    const int r2 = rem % per_split;
    strip_group(r2, dn_strips, sh.ntg[ai], u.strip, u.tg);
    u.d = p.desc + 2 * u.e + 1;
    const int c0 = u.split * p.split_cols;
    u.st0 = c0 / pw::kStageK;
    u.nst = (min(c0 + p.split_cols, p.I) - c0) / pw::kStageK;
  } else {
    sh.u = u;
    return;
  }
  const int off0 = p.offsets[u.e], ne = p.offsets[u.e + 1] - off0;
  u.off = off0 + u.tg * NMAX;
  u.nrows = min(NMAX, ne - u.tg * NMAX);
  u.npad = ((u.nrows + 15) / 16) * 16;
  u.q = u.d->q;
  const bool ok = u.kind == kGateUp ? desc_ok(*u.d, 2 * p.I, p.H) : desc_ok(*u.d, p.H, p.I);
  if (!ok) {
    report(p.status, u.d->q == 0 ? PW_ERR_NOT_RESIDENT : PW_ERR_UNSUPPORTED);
    u.skip = 1;
  }
  if (u.kind == kDown && !u.skip) {
    // wait until every gate_up unit of this expert that produces h columns of
    // this split has finished (all token groups)
    const int c0 = u.split * p.split_cols;
    const int strips_in_split = (min(c0 + p.split_cols, p.I) - c0) / 64;
    const uint32_t want = static_cast<uint32_t>(strips_in_split * sh.ntg[ai]);
    const uint32_t* ctr = p.ctr + 2 + u.e * p.nsplit + u.split;
    const uint64_t t0 = pw::global_ns();
    uint32_t v;
    while (true) {
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
      if (v >= want) break;
      if (*reinterpret_cast<volatile uint32_t*>(p.ctr + 1) != 0u) {
        u.skip = 1;
        break;
      }
      if (pw::global_ns() - t0 > p.wait_ns) {
        report(p.status, PW_ERR_TIMEOUT);
        atomicExch(p.ctr + 1, 1u);
        u.skip = 1;
        break;
      }
      __nanosleep(200);
    }
  }
  sh.u = u;
}

__device__ __forceinline__ void dequant_bar_sync(int G) {
  if (G == 2) asm volatile("bar.sync 1, 256;" ::: "memory");
}

__device__ __forceinline__ void lds_v4(uint32_t addr, uint32_t (&v)[4]) {
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]) : "r"(addr));
}

// End-of-unit bookkeeping (thread 0, after every role of the CTA finished the
// unit): publish gate_up completion or a down arrival; returns the strip to
// combine when this down unit was the strip's last one, else -1.
__device__ __forceinline__ int finish_unit(const Params& p, const Shared& sh, const Unit& u, int u_skip) {
  int combine = -1;
  if (!u_skip && u.kind == kGateUp) {
    const bool drop = (p.flags & PW_FFN_FLAG_TEST_DROP_ONE_ARRIVAL) && u.e == sh.act[0] && u.strip == 0 && u.tg == 0;
    if (!drop) {
      __threadfence();
      atomicAdd(p.ctr + 2 + u.e * p.nsplit + u.split, 1u);
    }
  } else if (!u_skip && u.kind == kDown && !p.grid_combine) {
    __threadfence();
    const uint32_t prev = atomicAdd(p.ctr + 2 + p.E * p.nsplit + u.strip, 1u);
    if (prev + 1 == static_cast<uint32_t>(sh.arrivals_per_strip)) {
      __threadfence();
      combine = u.strip;
    }
  }
  return combine;
}

// The current device's SM count, looked up once per device (0 on failure).
inline int sm_count_cached() {
  constexpr int kDevs = 64;
  static int count[kDevs] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  int n = dev < kDevs ? count[dev] : 0;
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev < kDevs) count[dev] = n;
  }
  return n;
}

// ---------------------------------------------------------------------------
// Combine (whole CTA): y rows of one strip for every token, fixed order.
// An item is one token and four consecutive rows (float4 partial sums).  For
// each of the token's k slots, the partial sums of up to 8 K-splits are loaded
// together (independent loads), then added in split order.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void add4(float4& a, const float4 v) {
  a.x += v.x;
  a.y += v.y;
  a.z += v.z;
  a.w += v.w;
}

// y[t][row..row+3] (fp16) from the token's k partial-sum vectors.
__device__ __forceinline__ void combine_item(const Params& p, int t, int row) {
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < p.k; ++j) {
    const int slot = t * p.k + j;
    const int ps = p.inv_perm[slot];
    if (static_cast<unsigned>(ps) >= static_cast<unsigned>(p.A)) {   // not a permutation of the slots
      report(p.status, PW_ERR_INVALID_ARG);
      continue;
    }
    const float wt = p.w[slot];
    const float4* base = reinterpret_cast<const float4*>(p.part + static_cast<long long>(ps) * p.H + row);
    const long long sstride = static_cast<long long>(p.A) * p.H / 4;   // float4 per split
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int sp0 = 0; sp0 < p.nsplit; sp0 += 8) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        v[u] = sp0 + u < p.nsplit ? __ldcg(base + (sp0 + u) * sstride) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int u = 0; u < 8; ++u) add4(s, v[u]);
    }
    acc.x += wt * s.x;
    acc.y += wt * s.y;
    acc.z += wt * s.z;
    acc.w += wt * s.w;
  }
  const uint32_t lo = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(acc.x))) |
                      (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(acc.y))) << 16);
  const uint32_t hi = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(acc.z))) |
                      (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(acc.w))) << 16);
  *reinterpret_cast<uint2*>(p.y + static_cast<long long>(t) * p.H + row) = make_uint2(lo, hi);
}

// One strip (128 rows) for every token, by the threads of one CTA.
__device__ inline void combine_strip(const Params& p, int strip, int tid, int nthreads) {
  const int n_items = p.T * 32;
  for (int it = tid; it < n_items; it += nthreads) {
    const int t = it >> 5, r4 = (it & 31) * 4;
    combine_item(p, t, (r4 >> 6) * (p.H / 2) + strip * 64 + (r4 & 63));
  }
}

// Every row of every token, spread over all threads of the grid (after the
// last unit; the rows' partial sums are complete).
__device__ inline void combine_all(const Params& p, long long tid, long long nthreads) {
  const int q4 = p.H / 4;
  const long long n_items = static_cast<long long>(p.T) * q4;
  for (long long it = tid; it < n_items; it += nthreads)
    combine_item(p, static_cast<int>(it / q4), static_cast<int>(it % q4) * 4);
}

// Kernel launchers (one translation unit each, ffn_stream.cuh instantiated
// for 16-, 64- and 128-token tiles).
int launch_ffn_t16(const Params& p, cudaStream_t s, bool after_route = false);    // 16-token tiles
int launch_ffn_t64(const Params& p, cudaStream_t s, bool after_route = false);    // 64-token tiles
int launch_ffn_t128(const Params& p, cudaStream_t s, bool after_route = false);   // 128-token tiles
int launch_ffn_gemv(const Params& p, cudaStream_t s, bool after_route = false);   // 2-token tiles on the CUDA cores

}  // namespace pw_ffn
