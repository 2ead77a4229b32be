// Fused mixed-precision MoE expert layer on the 5th-generation tensor cores,
// and the any-precision linear test export.
//
// "PagedWeight" arXiv text, §3.3 (Fused Mixed-Precision MoE Kernel): one
// kernel reads the weight pages directly, follows the committed bitwidth of
// every gate_up and down linear-block, and does the expert activation, the down
// projection and the output accumulation in one launch.
//
// Structure: a persistent launch (one CTA per SM) whose CTAs take work units
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
//
// Inside a unit (warp roles), for each of G groups (G = 2 on the decode path,
// where the two groups split the unit's K range over the same strip):
//   4 dequant warps (128 threads, thread = one row = one TMEM lane): stream the
//     strip's committed bit-planes into a shared ring with cp.async (one
//     16-byte slice per row and plane per 128 columns, rows interleaved so
//     the reads are conflict-free), dequantise 64 columns per stage through
//     the row's LUT (dequant.cuh) and write the fp16 operand A straight into a
//     4-stage TMEM ring with tcgen05.st;
//   1 producer warp: gathers the B operand (the tokens' x rows, or h rows) for
//     each stage into a 128-byte-swizzled shared ring with cp.async, and its
//     lane 0 issues tcgen05.mma (A from TMEM, B from shared memory, fp32
//     accumulator in TMEM), releasing ring slots with tcgen05.commit;
//   epilogue: the dequant warps read the accumulator rows from TMEM (group 1
//     hands its partial sums to group 0 through shared memory).
#include <cuda_fp16.h>

#include <mutex>

#include "dequant.cuh"
#include "pw_internal.h"

namespace {

using pw::BlockDesc;

constexpr int kDeqWarps = 4;                // per group: one warp per TMEM lane quadrant
constexpr int kDeqThreads = 128;
constexpr int kAStages = 4;
constexpr int kACols = pw::kStageK / 2;     // 32 TMEM columns (fp16 pairs) per stage
constexpr int kDCol = kAStages * kACols;    // accumulator columns start here (per group)
constexpr int kRingBytes = 32768;           // per group: plane staging ring [slot][plane][pos][16 B]
constexpr int kDecodeSplitCols = 2048;      // down K-split of the decode path
constexpr int kMaxE = 256;
constexpr int kBarsPerGroup = 16;

enum UnitKind : int { kNone = -1, kGateUp = 0, kDown = 1, kLinear = 2 };

// NMAX: tokens per tile.  G: dequant groups per CTA; with G = 2 both groups
// work on the same strip (sharing its LUT) and split the unit's K range, and
// their accumulators are summed through shared memory in the epilogue.
//
// Dynamic shared memory: [pre][64 KB LUT region, 64 KB aligned][post].  The
// smaller of the two rings goes in front of the region (the gap up to the
// next 64 KB boundary), the larger one after it.
template <int NMAX, int G>
struct Cfg {
  static constexpr int kThreads = G * (kDeqThreads + 32);
  static constexpr int kBStages = NMAX <= 64 ? 4 : 3;
  static constexpr int kBLookahead = kBStages - 2;
  static constexpr int kBStageBytes = NMAX * 128;
  static constexpr int kGroupTmemCols = (kDCol + NMAX) <= 256 ? 256 : 512;
  static constexpr int kTmemCols = G * kGroupTmemCols;
  static constexpr int kBRingBytes = G * kBStages * kBStageBytes;
  static constexpr int kPlaneRingBytes = G * kRingBytes;
  static constexpr int kXBytes = G == 2 ? NMAX * kDeqThreads * 4 : 0;
  static constexpr int kBarBytes = G * kBarsPerGroup * 8;
  static constexpr int kRowsBytes = G * NMAX * 4;
  static constexpr bool kBInPre = kBRingBytes <= kPlaneRingBytes;
  static constexpr int kPreRing = kBInPre ? kBRingBytes : kPlaneRingBytes;
  static constexpr int kPostRing = kBInPre ? kPlaneRingBytes : kBRingBytes;
  static constexpr int kPreBytes = kPreRing + kXBytes + kBarBytes + kRowsBytes + 8192;  // + Shared
  static constexpr int kSmemBytes = 65536 + pw::kLutRegionBytes + kPostRing;
  static_assert(kBStageBytes % 1024 == 0, "B stages must keep 1024-byte alignment");
  static_assert(kTmemCols <= 512, "TMEM has 512 columns");
  static_assert(2 * kAStages + kBStages + 1 <= kBarsPerGroup, "barrier slots");
  static_assert(kPreBytes <= 65536 - 4096, "front part must fit below the first 64 KB boundary");
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

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
  uint32_t* ctr;           // [0] ticket, [1] abort, [2, 2+E*nsplit) gate_up done, then strip arrivals
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
template <int NMAX>
__device__ void setup_schedule(const Params& p, Shared& sh) {
  sh.cum_gu[0] = 0;
  sh.cum_dn[0] = 0;
  if (p.linear) {
    sh.nact = 0;
    sh.arrivals_per_strip = 0;
    return;
  }
  int n = 0, gu = 0, dn = 0, arr = 0;
  const int gu_strips = 2 * p.I / 128, dn_strips = p.H / 128;
  for (int e = 0; e < p.E; ++e) {
    const int ne = __ldg(p.offsets + e + 1) - __ldg(p.offsets + e);
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
      u.strip = static_cast<int>(t % strips);
      u.tg = static_cast<int>(t / strips);
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
    while (sh.cum_gu[ai + 1] <= static_cast<int>(t)) ++ai;
    const int rem = static_cast<int>(t) - sh.cum_gu[ai];
    u.kind = kGateUp;
    u.e = sh.act[ai];
    u.strip = rem % gu_strips;
    u.tg = rem / gu_strips;
    u.split = (u.strip * 64) / p.split_cols;
    u.d = p.desc + 2 * u.e;
    u.st0 = 0;
    u.nst = p.H / pw::kStageK;
  } else if (t < static_cast<uint32_t>(n_gu + n_dn)) {
    const int v = static_cast<int>(t) - n_gu;
    while (sh.cum_dn[ai + 1] <= v) ++ai;
    const int rem = v - sh.cum_dn[ai];
    u.kind = kDown;
    u.e = sh.act[ai];
    const int per_split = dn_strips * sh.ntg[ai];
    u.split = rem / per_split;
    const int r2 = rem % per_split;
    u.strip = r2 % dn_strips;
    u.tg = r2 / dn_strips;
    u.d = p.desc + 2 * u.e + 1;
    const int c0 = u.split * p.split_cols;
    u.st0 = c0 / pw::kStageK;
    u.nst = (min(c0 + p.split_cols, p.I) - c0) / pw::kStageK;
  } else {
    sh.u = u;
    return;
  }
  const int off0 = __ldg(p.offsets + u.e), ne = __ldg(p.offsets + u.e + 1) - off0;
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

// ---------------------------------------------------------------------------
// Dequant warps (group g: warps 4g..4g+3; pos = row position in the strip)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void dequant_bar_sync(int G) {
  if (G == 2) asm volatile("bar.sync 1, 256;" ::: "memory");
}

__device__ __forceinline__ void lds_v4(uint32_t addr, uint32_t (&v)[4]) {
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]) : "r"(addr));
}

template <int NMAX, int G, int Q>
__device__ __noinline__ void dequant_role(const Params& p, const Unit& u, const Smem& sm, uint32_t tmem,
                                          uint32_t& a_cnt, uint32_t unit_cnt, int& abort) {
  using C = Cfg<NMAX, G>;
  constexpr int kTileStrideW = pw::kTileBytes / 4;
  constexpr int kSlotBytes = Q * pw::kTileBytes;      // one tile of every plane, all 128 rows
  constexpr int D = (kRingBytes / kSlotBytes) > 4 ? 4 : (kRingBytes / kSlotBytes);
  static_assert(D >= 2, "ring too small");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = warp >> 2, wq = warp & 3;
  const int pos = wq * 32 + lane;
  const BlockDesc& d = *u.d;
  const int row = strip_pos_row(u.strip, pos, d.rows / 2);
  pw::RowDequant<Q> dq;
  if constexpr (Q <= 4) {
    dq.load(d.lut + static_cast<long long>(row) * (1 << Q), 0u, lane);
  } else {
    dq.set_row(sm.lut_region, wq, lane);
    if (g == 0) dq.load(d.lut + static_cast<long long>(row) * (1 << Q));
    if (G == 2)
      dequant_bar_sync(G);   // group 0 filled the table both groups read
    else
      __syncwarp();
  }

  // this group's share of the unit's tiles
  const int tiles = d.cols / pw::kTileCols;
  const int ntiles_all = u.nst / 2;
  const int half = (ntiles_all + 1) / 2;
  const int tb = (G == 2 && g == 1) ? half : 0;
  const int te = (G == 2 && g == 0) ? half : ntiles_all;
  const int ntiles = te - tb;
  const int tile0 = u.st0 / 2 + tb;
  const uint32_t* src[Q];
#pragma unroll
  for (int q = 0; q < Q; ++q)
    src[q] = d.planes[q] + (static_cast<long long>(u.strip) * tiles + tile0) * kTileStrideW + pos * 4;
  const uint32_t ring = pw::smem_u32(sm.plane_ring + g * kRingBytes) + pos * 16;
  auto issue = [&](int t) {
    if (t < ntiles) {
      const uint32_t slot = ring + (t % D) * kSlotBytes;
#pragma unroll
      for (int q = 0; q < Q; ++q)
        pw::cp_async_16(slot + q * pw::kTileBytes, src[q] + static_cast<long long>(t) * kTileStrideW);
    }
    pw::cp_async_commit();
  };
#pragma unroll
  for (int i = 0; i < D - 1; ++i) issue(i);

  const uint32_t bar = sm.bar + g * kBarsPerGroup * 8;
  const uint32_t tl = tmem + g * C::kGroupTmemCols + (static_cast<uint32_t>(32 * wq) << 16);
  for (int t = 0; t < ntiles; ++t) {
    issue(t + D - 1);
    pw::cp_async_wait<D - 1>();
    const uint32_t slot = ring + (t % D) * kSlotBytes;
    uint32_t w4[Q][4];
#pragma unroll
    for (int q = 0; q < Q; ++q) lds_v4(slot + q * pw::kTileBytes, w4[q]);
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const uint32_t as = a_cnt % kAStages, use = a_cnt / kAStages;
      if (use > 0 && !abort && !pw::mbar_wait(bar + 8 * (kAStages + as), (use - 1) & 1u, p.wait_ns)) abort = 1;
      pw::tc_fence_after();
#pragma unroll
      for (int wd = 0; wd < 2; ++wd) {
        uint32_t ww[Q];
#pragma unroll
        for (int q = 0; q < Q; ++q) ww[q] = w4[q][2 * hf + wd];
        uint32_t out[16];
        dq.word(ww, out);
        pw::tmem_st_x16(tl + as * kACols + 16 * wd, out);
      }
      pw::tmem_st_wait();
      pw::tc_fence_before();
      __syncwarp();
      if (lane == 0) pw::mbar_arrive(bar + 8 * as);
      ++a_cnt;
    }
  }
  pw::cp_async_wait<0>();

  // epilogue: accumulator row `pos` (TMEM lane), columns = tokens
  if (!abort && !pw::mbar_wait(bar + 8 * (2 * kAStages + C::kBStages), unit_cnt & 1u, p.wait_ns)) abort = 1;
  pw::tc_fence_after();
  float* xch = sm.xch;
  if (G == 2 && g == 1) {
    // hand this group's partial sums to group 0 ([token][pos] layout)
    for (int c = 0; c < u.npad / 16; ++c) {
      uint32_t v[16];
      if (ntiles > 0) {
        pw::tmem_ld_x16(tl + kDCol + 16 * c, v);
        pw::tmem_ld_wait();
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) xch[(16 * c + i) * kDeqThreads + pos] = ntiles > 0 ? __uint_as_float(v[i]) : 0.f;
    }
    pw::tc_fence_before();
    dequant_bar_sync(G);
    return;
  }
  if (G == 2) dequant_bar_sync(G);
  for (int c = 0; c < u.npad / 16; ++c) {
    uint32_t v[16];
    pw::tmem_ld_x16(tl + kDCol + 16 * c, v);
    pw::tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int n = 16 * c + i;
      float val = __uint_as_float(v[i]);
      if (G == 2) val += xch[n * kDeqThreads + pos];
      if (u.kind == kGateUp) {
        const float up = __shfl_down_sync(0xffffffffu, val, 16);
        if (lane < 16 && n < u.nrows) {
          const int m = u.strip * 64 + 16 * wq + lane;
          p.h[static_cast<long long>(u.off + n) * p.I + m] = __half_as_ushort(__float2half_rn(silu(val) * up));
        }
      } else if (u.kind == kDown) {
        if (n < u.nrows) p.part[(static_cast<long long>(u.split) * p.A + u.off + n) * p.H + row] = val;
      } else {
        if (n < u.nrows) p.out[static_cast<long long>(u.tg * NMAX + n) * d.rows + row] = val;
      }
    }
  }
  pw::tc_fence_before();
}

// ---------------------------------------------------------------------------
// Producer / MMA warp of group g (warp 4G + g)
// ---------------------------------------------------------------------------
template <int NMAX, int G>
__device__ void producer_role(const Params& p, const Unit& u, const Smem& sm, uint32_t tmem, uint32_t& a_cnt,
                              uint32_t& b_cnt, int& abort) {
  using C = Cfg<NMAX, G>;
  const int lane = threadIdx.x & 31;
  const int g = (threadIdx.x >> 5) - 4 * G;
  int* rows = sm.rows + g * NMAX;
  const uint16_t* bbase = u.kind == kDown ? p.h : p.x;
  for (int n = lane; n < u.npad; n += 32) {
    const int nn = min(n, u.nrows - 1);
    int r;
    if (u.kind == kGateUp)
      r = (__ldg(p.perm + u.off + nn) / p.k) * p.H;
    else if (u.kind == kDown)
      r = (u.off + nn) * p.I;
    else
      r = (u.tg * NMAX + nn) * u.d->cols;
    rows[n] = r;
  }
  __syncwarp();
  // this group's stages
  const int ntiles_all = u.nst / 2;
  const int half = (ntiles_all + 1) / 2;
  const int sb = 2 * ((G == 2 && g == 1) ? half : 0);
  const int se = 2 * ((G == 2 && g == 0) ? half : ntiles_all);
  const int nst = se - sb;
  const uint32_t bring = pw::smem_u32(sm.b_ring + g * C::kBStages * C::kBStageBytes);
  const uint32_t bar = sm.bar + g * kBarsPerGroup * 8;
  const uint32_t bar_b_empty = bar + 8 * (2 * kAStages);
  const uint32_t bar_done = bar + 8 * (2 * kAStages + C::kBStages);
  const uint32_t tg = tmem + g * C::kGroupTmemCols;
  const int chunks = u.npad * 8;
  auto issue = [&](int st) {
    const uint32_t slot = (b_cnt + st) % C::kBStages, use = (b_cnt + st) / C::kBStages;
    if (use > 0 && !abort && !pw::mbar_wait(bar_b_empty + 8 * slot, (use - 1) & 1u, p.wait_ns)) abort = 1;
    const uint32_t dst0 = bring + slot * C::kBStageBytes;
    const long long col = static_cast<long long>(u.st0 + sb + st) * pw::kStageK;
    for (int i = lane; i < chunks; i += 32) {
      const int n = i >> 3, c = i & 7;
      pw::cp_async_16(dst0 + n * 128 + ((c ^ (n & 7)) << 4), bbase + rows[n] + col + c * 8);
    }
  };
  constexpr int LA = C::kBLookahead;
#pragma unroll
  for (int i = 0; i < LA; ++i) {
    if (i < nst) issue(i);
    pw::cp_async_commit();
  }
  const uint32_t idesc = pw::idesc_f16_f32(128, u.npad);
  for (int st = 0; st < nst; ++st) {
    if (st + LA < nst) issue(st + LA);
    pw::cp_async_commit();
    pw::cp_async_wait<LA>();
    pw::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      const uint32_t as = a_cnt % kAStages;
      if (!abort && !pw::mbar_wait(bar + 8 * as, (a_cnt / kAStages) & 1u, p.wait_ns)) abort = 1;
      pw::tc_fence_after();
      const uint32_t bs = (b_cnt + st) % C::kBStages;
      const uint64_t bdesc = pw::sdesc_kmajor_sw128(bring + bs * C::kBStageBytes);
#pragma unroll
      for (int j = 0; j < pw::kStageK / 16; ++j)
        pw::tc_mma_ts(tg + kDCol, tg + as * kACols + 8 * j, bdesc + 2ull * j, idesc, (st > 0 || j > 0) ? 1u : 0u);
      pw::tc_commit(bar + 8 * (kAStages + as));
      pw::tc_commit(bar_b_empty + 8 * bs);
    }
    ++a_cnt;
    __syncwarp();
  }
  b_cnt += nst;
  pw::cp_async_wait<0>();
  if (lane == 0) {
    if (nst > 0)
      pw::tc_commit(bar_done);
    else
      pw::mbar_arrive(bar_done);
  }
  __syncwarp();
}

// ---------------------------------------------------------------------------
// Combine (whole CTA): y rows of one strip for every token, fixed order.
// ---------------------------------------------------------------------------
__device__ void combine_strip(const Params& p, int strip) {
  const int n_items = p.T * 128;
  for (int it = threadIdx.x; it < n_items; it += blockDim.x) {
    const int t = it >> 7, pos = it & 127;
    const int row = (pos >> 6) * (p.H / 2) + strip * 64 + (pos & 63);
    float acc = 0.f;
    for (int j = 0; j < p.k; ++j) {
      const int slot = t * p.k + j;
      const int ps = __ldg(p.inv_perm + slot);
      const float wt = __ldg(p.w + slot);
      float s = 0.f;
      for (int sp = 0; sp < p.nsplit; ++sp) s += __ldcg(p.part + (static_cast<long long>(sp) * p.A + ps) * p.H + row);
      acc += wt * s;
    }
    p.y[static_cast<long long>(t) * p.H + row] = __half_as_ushort(__float2half_rn(acc));
  }
}

template <int NMAX, int G>
__global__ void __launch_bounds__(Cfg<NMAX, G>::kThreads, 1) apl_tc_kernel(Params p) {
  using C = Cfg<NMAX, G>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // carve up dynamic shared memory around a 64 KB-aligned LUT region
  const uint32_t base = pw::smem_u32(smem_raw);
  const uint32_t pre = (base + 1023u) & ~1023u;
  const uint32_t region = (pre + static_cast<uint32_t>(C::kPreBytes) + 0xFFFFu) & ~0xFFFFu;
  const uint32_t post = region + static_cast<uint32_t>(pw::kLutRegionBytes);
  if (post + static_cast<uint32_t>(C::kPostRing) > base + static_cast<uint32_t>(C::kSmemBytes)) {
    if (threadIdx.x == 0) report(p.status, PW_ERR_UNSUPPORTED);   // unexpected shared-window base
    return;
  }
  auto at = [&](uint32_t addr) { return smem_raw + (addr - base); };
  Smem sm;
  uint32_t cur = pre;
  uint8_t* pre_ring = at(cur);
  cur += C::kPreRing;
  sm.xch = reinterpret_cast<float*>(at(cur));
  cur += C::kXBytes;
  sm.bar = cur;
  cur += C::kBarBytes;
  sm.rows = reinterpret_cast<int*>(at(cur));
  cur += C::kRowsBytes;
  Shared& sh = *reinterpret_cast<Shared*>(at((cur + 15u) & ~15u));
  sm.lut_region = region;
  if (C::kBInPre) {
    sm.b_ring = pre_ring;
    sm.plane_ring = at(post);
  } else {
    sm.plane_ring = pre_ring;
    sm.b_ring = at(post);
  }

  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int g = 0; g < G; ++g) {
      const uint32_t bar = sm.bar + g * kBarsPerGroup * 8;
      for (int i = 0; i < kAStages; ++i) {
        pw::mbar_init(bar + 8 * i, kDeqWarps);       // A full: one arrive per dequant warp
        pw::mbar_init(bar + 8 * (kAStages + i), 1);  // A empty: tcgen05.commit
      }
      for (int i = 0; i < C::kBStages; ++i) pw::mbar_init(bar + 8 * (2 * kAStages + i), 1);  // B empty
      pw::mbar_init(bar + 8 * (2 * kAStages + C::kBStages), 1);                            // unit MMAs done
    }
    pw::mbar_init_fence();
    sh.abort = 0;
    setup_schedule<NMAX>(p, sh);
  }
  if (warp == 0) {
    pw::tmem_alloc(pw::smem_u32(&sh.tmem), C::kTmemCols);
    pw::tmem_relinquish();
  }
  pw::tc_fence_before();
  __syncthreads();
  pw::tc_fence_after();
  const uint32_t tmem = sh.tmem;

  uint32_t a_cnt = 0, b_cnt = 0, unit_cnt = 0;
  int abort_local = 0;
  for (;;) {
    if (threadIdx.x == 0) next_unit<NMAX>(p, sh);
    pw::tc_fence_before();
    __syncthreads();
    pw::tc_fence_after();
    const Unit& u = sh.u;   // read from shared memory where used (keeps registers free)
    if (u.kind == kNone) break;
    const int u_skip = u.skip;
    if (!u_skip) {
      if (warp < kDeqWarps * G) {
        switch (u.q) {
          case 2: dequant_role<NMAX, G, 2>(p, u, sm, tmem, a_cnt, unit_cnt, abort_local); break;
          case 3: dequant_role<NMAX, G, 3>(p, u, sm, tmem, a_cnt, unit_cnt, abort_local); break;
          case 4: dequant_role<NMAX, G, 4>(p, u, sm, tmem, a_cnt, unit_cnt, abort_local); break;
          case 5: dequant_role<NMAX, G, 5>(p, u, sm, tmem, a_cnt, unit_cnt, abort_local); break;
          case 6: dequant_role<NMAX, G, 6>(p, u, sm, tmem, a_cnt, unit_cnt, abort_local); break;
          case 7: dequant_role<NMAX, G, 7>(p, u, sm, tmem, a_cnt, unit_cnt, abort_local); break;
          default: dequant_role<NMAX, G, 8>(p, u, sm, tmem, a_cnt, unit_cnt, abort_local); break;
        }
      } else {
        producer_role<NMAX, G>(p, u, sm, tmem, a_cnt, b_cnt, abort_local);
      }
      ++unit_cnt;
    }
    if (abort_local) {
      report(p.status, PW_ERR_TIMEOUT);
      sh.abort = 1;
    }
    pw::tc_fence_before();
    __syncthreads();
    pw::tc_fence_after();
    if (threadIdx.x == 0) {
      int combine = -1;
      if (!u_skip && u.kind == kGateUp) {
        const bool drop = (p.flags & PW_FFN_FLAG_TEST_DROP_ONE_ARRIVAL) && u.e == sh.act[0] && u.strip == 0 &&
                          u.tg == 0;
        if (!drop) {
          __threadfence();
          atomicAdd(p.ctr + 2 + u.e * p.nsplit + u.split, 1u);
        }
      } else if (!u_skip && u.kind == kDown) {
        __threadfence();
        const uint32_t prev = atomicAdd(p.ctr + 2 + p.E * p.nsplit + u.strip, 1u);
        if (prev + 1 == static_cast<uint32_t>(sh.arrivals_per_strip)) {
          __threadfence();
          combine = u.strip;
        }
      }
      sh.u.combine = combine;
    }
    __syncthreads();
    if (sh.u.combine >= 0) combine_strip(p, sh.u.combine);
  }
  pw::tc_fence_before();
  __syncthreads();
  pw::tc_fence_after();
  if (warp == 0) pw::tmem_dealloc(tmem, C::kTmemCols);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

struct WsLayout {
  size_t ctr, h, part, total;
  int nsplit, split_cols;
};

int choose_path(int T, int E, int k, int requested) {
  if (requested == PW_PATH_DECODE || requested == PW_PATH_PREFILL) return requested;
  // average tokens per expert: 256-token tiles pay off once experts see more
  // than a few dozen tokens
  return (static_cast<long long>(T) * k >= 48ll * E) ? PW_PATH_PREFILL : PW_PATH_DECODE;
}

WsLayout ws_layout(int T, int H, int I, int E, int k, int path) {
  WsLayout L{};
  const long long A = static_cast<long long>(T) * k;
  L.split_cols = path == PW_PATH_PREFILL ? I : kDecodeSplitCols;
  L.nsplit = (I + L.split_cols - 1) / L.split_cols;
  const size_t ctr_words = 2 + static_cast<size_t>(E) * L.nsplit + static_cast<size_t>(H) / 128;
  L.ctr = 0;
  L.h = align256(ctr_words * 4);
  L.part = L.h + align256(static_cast<size_t>(A) * I * 2);
  L.total = L.part + align256(static_cast<size_t>(L.nsplit) * A * H * 4);
  return L;
}

// Workspace of the path pw_moe_apl_ffn picks by itself for this size.
WsLayout ws_layout(int T, int H, int I, int E, int k) {
  return ws_layout(T, H, I, E, k, choose_path(T, E, k, PW_PATH_AUTO));
}

int validate_shape(int T, int H, int I, int E, int k) {
  if (T < 0 || H <= 0 || I <= 0 || E < 1 || E > kMaxE || k < 1 || k > 8 || k > E)
    return pw::set_error(PW_ERR_INVALID_ARG, "ffn: bad sizes T=%d H=%d I=%d E=%d k=%d", T, H, I, E, k);
  if (H % 128 || I % 128)
    return pw::set_error(PW_ERR_UNSUPPORTED, "ffn: H and I must be multiples of 128 (H=%d I=%d)", H, I);
  if (static_cast<long long>(T) * k > (1 << 24) || static_cast<long long>(T) * k * I > (1ll << 31) ||
      static_cast<long long>(T) * H > (1ll << 31))
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

template <int NMAX, int G>
int launch(const Params& p, cudaStream_t s) {
  using C = Cfg<NMAX, G>;
  static bool attr_done = false;
  if (!attr_done) {
    PW_CUDA_TRY(cudaFuncSetAttribute(apl_tc_kernel<NMAX, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     C::kSmemBytes));
    attr_done = true;
  }
  const int sms = sm_count_cached();
  if (sms < 1) return pw::set_error(PW_ERR_CUDA, "could not query the SM count");
  // one CTA per SM (the shared-memory footprint keeps it at one), each owning
  // C::kTmemCols of the SM's 512 TMEM columns
  apl_tc_kernel<NMAX, G><<<sms, C::kThreads, C::kSmemBytes, s>>>(p);
  PW_CUDA_TRY(cudaGetLastError());
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
  pw_ffn_options o{};
  if (opts) o = *opts;
  const int path = choose_path(T, E, k, o.path);
  const WsLayout L = ws_layout(T, H, I, E, k, path);
  if (ws_bytes < L.total || (reinterpret_cast<uintptr_t>(d_ws) & 255))
    return pw::set_error(PW_ERR_WORKSPACE, "ffn: workspace needs %zu bytes, 256-byte aligned (got %zu)", L.total,
                         ws_bytes);
  cudaStream_t s = pw::as_stream(stream);
  char* ws = static_cast<char*>(d_ws);
  Params p{};
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
  p.split_cols = L.split_cols;
  p.ctr = reinterpret_cast<uint32_t*>(ws + L.ctr);
  p.h = reinterpret_cast<uint16_t*>(ws + L.h);
  p.part = reinterpret_cast<float*>(ws + L.part);
  p.status = d_status;
  p.wait_ns = (o.wait_timeout_us ? o.wait_timeout_us : 2000000u) * 1000ull;
  p.flags = o.flags;
  p.linear = 0;
  PW_CUDA_TRY(cudaMemsetAsync(p.ctr, 0, L.h - L.ctr, s));
  return path == PW_PATH_PREFILL ? launch<256, 1>(p, s) : launch<32, 2>(p, s);
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
  return M > 32 ? launch<256, 1>(p, s) : launch<32, 2>(p, s);
}

}  // extern "C"

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
