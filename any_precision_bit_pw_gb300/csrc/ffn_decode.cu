// Fused MoE layer kernel for decode batches: token tiles of up to 16 and one
// 128-column tile per pipeline stage.  See ffn_common.cuh for the work units
// and their scheduling.
//
// Each CTA (one per SM) runs two groups on the same 128-row strip of a unit,
// splitting its K range; both share the strip's LUT.  Warp roles:
//   warps 0-7, two groups of 4 dequant warps (thread = one row = one TMEM
//     lane): per tile, each thread copies its 16-byte slice of every committed
//     plane plus its share of the B operand (the tokens' x or h columns of the
//     tile, two 16-byte chunks of a 128-byte-swizzled layout) into shared rings
//     with cp.async, several tiles ahead; dequantises the tile's 128 columns of
//     its row (dequant.cuh), stores them as operand A into a 3-slot TMEM ring
//     (tcgen05.st) and arrives on the tile's "full" barrier;
//   warps 8-9, one MMA warp per group (lane 0): per tile, waits for "full",
//     issues the tile's 8 tcgen05.mma (A from TMEM, B from shared memory, fp32
//     accumulator in TMEM) and one tcgen05.commit to the tile's "free" barrier,
//     which releases the tile's A slot and B slot together;
//   warp 10, the scheduler (lane 0): takes the next ticket, decodes it (for a
//     down unit: waits until its h columns exist) and publishes it in one of
//     two unit slots while the current unit runs.
// Consecutive units overlap: when the next unit is already published as the
// dequant warps finish a unit's tiles, they issue its first plane and B loads
// before running the current unit's epilogue.  They never block on the next
// unit there (that unit may be waiting for this one), so the unit order stays
// deadlock-free.
// The epilogue reads the accumulator rows from TMEM; group 1 hands its partial
// sums to group 0 through shared memory.  All mbarrier waits are bounded
// (PW_ERR_TIMEOUT); TMEM is released before the CTA exits.
#include "ffn_common.cuh"

namespace pw_ffn {
namespace {

constexpr int kN = 16;                          // tokens per tile
constexpr int kG = 2;                           // dequant groups (split K)
constexpr int kDeqAll = kG * kDeqThreads;       // 256 dequant threads
constexpr int kMmaWarp0 = kG * kDeqWarps;       // warps 8, 9
constexpr int kSchedWarp = kMmaWarp0 + kG;      // warp 10
constexpr int kThreads = (kSchedWarp + 1) * 32;
constexpr int kSA = 3;                          // TMEM A slots per group (tiles)
constexpr int kATileCols = 64;                  // TMEM columns per A tile (128 fp16 per row)
constexpr int kDColT = kSA * kATileCols;        // accumulator columns start here
constexpr int kGroupCols = 256;
constexpr int kTmemColsT = kG * kGroupCols;
constexpr int kF = 8;                           // completion barriers per group (tile index mod 8)
constexpr int kBSlots = 6;                      // B slots per group
constexpr int kBAtomBytes = kN * 128;           // 16 rows x 64 columns fp16, 128-byte swizzle
constexpr int kBSlotBytes = 2 * kBAtomBytes;    // 128 columns
constexpr int kPlaneRing = 32768;               // per group
constexpr int kBRingBytes = kG * kBSlots * kBSlotBytes;
constexpr int kXBytes = kN * kDeqThreads * 4;
constexpr int kBarBytes = 512;
constexpr int kRowsBytes = 2 * kN * 4;
constexpr int kStateBytes = 6144;
constexpr int kPreBytes = kBRingBytes + kBarBytes + kRowsBytes + kStateBytes;
constexpr int kPostBytes = kG * kPlaneRing + kXBytes;
constexpr int kSmemBytes = 65536 + pw::kLutRegionBytes + kPostBytes;
static_assert(kDColT + kN <= kGroupCols, "TMEM columns per group");
static_assert(kPreBytes <= 65536 - 4096, "front part must fit below the first 64 KB boundary");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

// barrier slots: per group g at 8*(20*g + i): full[kF], free[kF], done; then unit_ready[2], unit_free[2]
__device__ __forceinline__ uint32_t bar_full(uint32_t g0, int i) { return g0 + 8 * i; }
__device__ __forceinline__ uint32_t bar_free(uint32_t g0, int i) { return g0 + 8 * (kF + i); }
__device__ __forceinline__ uint32_t bar_done(uint32_t g0) { return g0 + 8 * (2 * kF); }
constexpr int kBarsPerGroupT = 20;
static_assert(2 * kF + 1 <= kBarsPerGroupT && (kG * kBarsPerGroupT + 4) * 8 <= kBarBytes, "barrier slots");

struct DecState {
  Shared sched;          // ticket decoding state (scheduler thread)
  Unit units[2];         // published units (double buffer)
  int combine;           // strip to combine after a unit, or -1
  int early;             // the next unit's first loads are already in flight
};
static_assert(sizeof(DecState) <= kStateBytes, "state size");

struct SmemT {
  uint8_t* b_ring;      // kG x kBSlots x kBSlotBytes
  uint8_t* plane_ring;  // kG x kPlaneRing
  float* xch;           // group-1 partial sums [token][pos]
  uint32_t bar;         // barriers (shared address)
  int* rows;            // [2][kN] B row offsets of the published units
  uint32_t lut_region;
  DecState* st;
};

__device__ __forceinline__ uint32_t group_bar(const SmemT& sm, int g) { return sm.bar + 8 * kBarsPerGroupT * g; }
__device__ __forceinline__ uint32_t unit_ready_bar(const SmemT& sm, int s) {
  return sm.bar + 8 * (kG * kBarsPerGroupT + s);
}
__device__ __forceinline__ uint32_t unit_free_bar(const SmemT& sm, int s) {
  return sm.bar + 8 * (kG * kBarsPerGroupT + 2 + s);
}

// Wait until the MMAs of this group's tile x have completed.
__device__ __forceinline__ void wait_tile_free(uint32_t g0, uint32_t x, const Params& p, int& abort) {
  if (!abort && !pw::mbar_wait(bar_free(g0, x % kF), (x / kF) & 1u, p.wait_ns)) abort = 1;
}

__device__ __forceinline__ void named_sync_dequant() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// This group's share [tb, te) of a unit's 128-column tiles (group 0 takes the
// larger half).
__device__ __forceinline__ void group_tiles(const Unit& u, int g, int& tb, int& te) {
  const int ntiles_all = u.nst / 2;
  const int half = (ntiles_all + 1) / 2;
  tb = g == 1 ? half : 0;
  te = g == 0 ? half : ntiles_all;
}

// Per-thread tile loader of one unit: its plane slices and its B chunks.
template <int Q>
struct TileLoader {
  static constexpr int kTileStrideW = pw::kTileBytes / 4;
  static constexpr int kSlotBytes = Q * pw::kTileBytes;
  static constexpr int D = (kPlaneRing / kSlotBytes) > 4 ? 4 : (kPlaneRing / kSlotBytes);
  static_assert(D >= 2 && D + 2 <= kBSlots, "ring depths");
  const uint32_t* src[Q];
  const uint16_t* bbase;
  const int* rows;
  uint32_t ring, bring, g0, tcnt;
  int ntiles, tile0, pos, nchunk;

  __device__ __forceinline__ void init(const Params& p, const Unit& u, const SmemT& sm, const int* urows, int g,
                                       int pos_, uint32_t tcnt_) {
    const BlockDesc& d = *u.d;
    int tb, te;
    group_tiles(u, g, tb, te);
    ntiles = te - tb;
    tile0 = u.st0 / 2 + tb;
    pos = pos_;
    tcnt = tcnt_;
    const int tiles = d.cols / pw::kTileCols;
#pragma unroll
    for (int q = 0; q < Q; ++q)
      src[q] = d.planes[q] + (static_cast<long long>(u.strip) * tiles + tile0) * kTileStrideW + pos * 4;
    ring = pw::smem_u32(sm.plane_ring + g * kPlaneRing) + pos * 16;
    bring = pw::smem_u32(sm.b_ring + g * kBSlots * kBSlotBytes);
    g0 = group_bar(sm, g);
    bbase = u.kind == kDown ? p.h : p.x;
    rows = urows;
    nchunk = u.npad / 8;   // i = pos + 128 m (m < npad / 8): row n = i / 16, chunk c = i % 16
  }

  // Copy tile t (this group's numbering) into ring slot t % D and B slot
  // (tcnt + t) % kBSlots; always commits one cp.async group.
  __device__ __forceinline__ void issue(int t, const Params& p, int& abort) const {
    if (t < ntiles) {
      const uint32_t x = tcnt + t;
      if (x >= kBSlots) wait_tile_free(g0, x - kBSlots, p, abort);
      const uint32_t slot = ring + (t % D) * kSlotBytes;
#pragma unroll
      for (int q = 0; q < Q; ++q)
        pw::cp_async_16(slot + q * pw::kTileBytes, src[q] + static_cast<long long>(t) * kTileStrideW);
      const uint32_t bslot = bring + (x % kBSlots) * kBSlotBytes;
      const long long col = static_cast<long long>(tile0 + t) * pw::kTileCols;
      for (int m = 0; m < nchunk; ++m) {
        const int i = pos + 128 * m;
        const int n = i >> 4, c = i & 15;
        pw::cp_async_16(bslot + (c >> 3) * kBAtomBytes + n * 128 + (((c & 7) ^ (n & 7)) << 4),
                        bbase + rows[n] + col + c * 8);
      }
    }
    pw::cp_async_commit();
  }

  __device__ __forceinline__ void prologue(const Params& p, int& abort) const {
#pragma unroll
    for (int i = 0; i < D - 1; ++i) issue(i, p, abort);
  }
};

template <int Q>
__device__ __noinline__ void issue_prologue(const Params& p, const Unit& u, const SmemT& sm, const int* urows,
                                            int g, int pos, uint32_t tcnt, int& abort) {
  TileLoader<Q> ld;
  ld.init(p, u, sm, urows, g, pos, tcnt);
  ld.prologue(p, abort);
  // warm L2 with this row's LUT for the unit's start
  const int row = strip_pos_row(u.strip, pos, u.d->rows / 2);
  const char* lut = reinterpret_cast<const char*>(u.d->lut + static_cast<long long>(row) * (1 << Q));
  for (int off = 0; off < (2 << Q); off += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(lut + off));
}

// One unit for a dequant thread: LUT, tiles, early start of the next unit,
// epilogue.  Returns whether the next unit's first loads were issued.
template <int Q>
__device__ __noinline__ bool dequant_unit(const Params& p, const Unit& u, const SmemT& sm, const int* urows,
                                          uint32_t tmem, uint32_t& tcnt, uint32_t unit_cnt, int slot, bool early,
                                          int& abort) {
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
    dq.template load<kG>(d.lut + static_cast<long long>(row) * (1 << Q), g);
    named_sync_dequant();   // both halves of every row's table are in place
  }
  TileLoader<Q> ld;
  ld.init(p, u, sm, urows, g, pos, tcnt);
  constexpr int D = TileLoader<Q>::D;
  if (!early) ld.prologue(p, abort);

  const uint32_t g0 = ld.g0;
  const uint32_t tl = tmem + g * kGroupCols + (static_cast<uint32_t>(32 * wq) << 16);
  for (int t = 0; t < ld.ntiles; ++t) {
    ld.issue(t + D - 1, p, abort);
    pw::cp_async_wait<D - 1>();
    pw::fence_proxy_async_smem();   // this thread's B chunks of tile t, for the tensor core
    const uint32_t rs = ld.ring + (t % D) * TileLoader<Q>::kSlotBytes;
    uint32_t w4[Q][4];
#pragma unroll
    for (int q = 0; q < Q; ++q) lds_v4(rs + q * pw::kTileBytes, w4[q]);
    const uint32_t x = tcnt + t;
    if (x >= kSA) wait_tile_free(g0, x - kSA, p, abort);
    pw::tc_fence_after();
    const uint32_t acol = tl + (x % kSA) * kATileCols;
#pragma unroll
    for (int wd = 0; wd < 4; ++wd) {
      uint32_t ww[Q];
#pragma unroll
      for (int q = 0; q < Q; ++q) ww[q] = w4[q][wd];
      uint32_t out[16];
      dq.word(ww, out);
      pw::tmem_st_x16(acol + 16 * wd, out);
    }
    pw::tmem_st_wait();
    pw::tc_fence_before();
    __syncwarp();
    if (lane == 0) pw::mbar_arrive(bar_full(g0, x % kF));
  }
  const int ntiles = ld.ntiles;
  tcnt += ntiles;
  pw::cp_async_wait<0>();

  // start the next unit's loads now if it is already published
  const int ns = slot ^ 1;
  if (threadIdx.x == 0) {
    const Unit& nu = sm.st->units[ns];
    sm.st->early = mbar_test(unit_ready_bar(sm, ns), ((unit_cnt + 1) >> 1) & 1u) && nu.kind != kNone;
  }
  named_sync_dequant();   // also: both groups are done with this unit's LUT region
  const bool next_early = sm.st->early != 0;
  if (next_early) {
    const Unit& nu = sm.st->units[ns];
    const int* nrows = sm.rows + ns * kN;
    switch (nu.q) {
      case 2: issue_prologue<2>(p, nu, sm, nrows, g, pos, tcnt, abort); break;
      case 3: issue_prologue<3>(p, nu, sm, nrows, g, pos, tcnt, abort); break;
      case 4: issue_prologue<4>(p, nu, sm, nrows, g, pos, tcnt, abort); break;
      case 5: issue_prologue<5>(p, nu, sm, nrows, g, pos, tcnt, abort); break;
      case 6: issue_prologue<6>(p, nu, sm, nrows, g, pos, tcnt, abort); break;
      case 7: issue_prologue<7>(p, nu, sm, nrows, g, pos, tcnt, abort); break;
      default: issue_prologue<8>(p, nu, sm, nrows, g, pos, tcnt, abort); break;
    }
  }

  // epilogue: accumulator row `pos` (TMEM lane), columns = tokens
  if (!abort && !pw::mbar_wait(bar_done(g0), unit_cnt & 1u, p.wait_ns)) abort = 1;
  pw::tc_fence_after();
  float* xch = sm.xch;
  uint32_t v[16];
  if (ntiles > 0) {
    pw::tmem_ld_x16(tl + kDColT, v);
    pw::tmem_ld_wait();
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = 0u;
  }
  pw::tc_fence_before();
  if (g == 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) xch[i * kDeqThreads + pos] = __uint_as_float(v[i]);
  }
  named_sync_dequant();
  if (g == 0) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float val = __uint_as_float(v[i]) + xch[i * kDeqThreads + pos];
      if (u.kind == kGateUp) {
        const float up = __shfl_down_sync(0xffffffffu, val, 16);
        if (lane < 16 && i < u.nrows) {
          const int m = u.strip * 64 + 16 * wq + lane;
          p.h[static_cast<long long>(u.off + i) * p.I + m] = __half_as_ushort(__float2half_rn(silu(val) * up));
        }
      } else if (u.kind == kDown) {
        if (i < u.nrows) p.part[(static_cast<long long>(u.split) * p.A + u.off + i) * p.H + row] = val;
      } else {
        if (i < u.nrows) p.out[static_cast<long long>(u.tg * kN + i) * d.rows + row] = val;
      }
    }
  }
  return next_early;
}

__device__ void mma_unit(const Unit& u, const SmemT& sm, uint32_t tmem, uint32_t& tcnt, const Params& p,
                         int& abort) {
  const int g = (threadIdx.x >> 5) - kMmaWarp0;
  int tb, te;
  group_tiles(u, g, tb, te);
  const int ntiles = te - tb;
  const uint32_t g0 = group_bar(sm, g);
  if ((threadIdx.x & 31) == 0) {
    const uint32_t bring = pw::smem_u32(sm.b_ring + g * kBSlots * kBSlotBytes);
    const uint32_t tg = tmem + g * kGroupCols;
    const uint32_t idesc = pw::idesc_f16_f32(128, u.npad);
    for (int t = 0; t < ntiles; ++t) {
      const uint32_t x = tcnt + t;
      if (!abort && !pw::mbar_wait(bar_full(g0, x % kF), (x / kF) & 1u, p.wait_ns)) abort = 1;
      pw::tc_fence_after();
      const uint32_t a = tg + (x % kSA) * kATileCols;
      const uint32_t b = bring + (x % kBSlots) * kBSlotBytes;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint64_t bdesc = pw::sdesc_kmajor_sw128(b + (j >> 2) * kBAtomBytes) + 2ull * (j & 3);
        pw::tc_mma_ts(tg + kDColT, a + 8 * j, bdesc, idesc, (t > 0 || j > 0) ? 1u : 0u);
      }
      pw::tc_commit(bar_free(g0, x % kF));
    }
    if (ntiles > 0)
      pw::tc_commit(bar_done(g0));
    else
      pw::mbar_arrive(bar_done(g0));
  }
  tcnt += ntiles;
  __syncwarp();
}

// Scheduler (one thread): publish units into the two slots, one ahead.
__device__ void scheduler(const Params& p, const SmemT& sm) {
  DecState& st = *sm.st;
  for (uint32_t i = 0;; ++i) {
    const int s = static_cast<int>(i & 1u);
    if (i >= 2 && !pw::mbar_wait(unit_free_bar(sm, s), ((i - 2) >> 1) & 1u, p.wait_ns)) {
      report(p.status, PW_ERR_TIMEOUT);
      st.sched.abort = 1;
    }
    Unit u;
    do {
      next_unit<kN>(p, st.sched);
      u = st.sched.u;
    } while (u.kind != kNone && u.skip);
    st.units[s] = u;
    if (u.kind != kNone) {
      int* rows = sm.rows + s * kN;
      for (int n = 0; n < kN; ++n) {
        const int nn = min(n, u.nrows - 1);
        int r;
        if (u.kind == kGateUp)
          r = (__ldg(p.perm + u.off + nn) / p.k) * p.H;
        else if (u.kind == kDown)
          r = (u.off + nn) * p.I;
        else
          r = (u.tg * kN + nn) * u.d->cols;
        rows[n] = r;
      }
    }
    pw::mbar_arrive(unit_ready_bar(sm, s));
    if (u.kind == kNone) return;
  }
}

// Wait (lane 0, then the whole warp) for unit i to be published.
__device__ __forceinline__ void wait_unit(const SmemT& sm, uint32_t i, const Params& p, int& abort) {
  if ((threadIdx.x & 31) == 0) {
    if (!pw::mbar_wait(unit_ready_bar(sm, static_cast<int>(i & 1u)), (i >> 1) & 1u, 4 * p.wait_ns)) {
      // the scheduler is stuck; stop after this unit
      abort = 1;
    }
  }
  __syncwarp();
}

__global__ void __launch_bounds__(kThreads, 1) apl_decode_kernel(Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t base = pw::smem_u32(smem_raw);
  const uint32_t pre = (base + 1023u) & ~1023u;
  const uint32_t region = (pre + static_cast<uint32_t>(kPreBytes) + 0xFFFFu) & ~0xFFFFu;
  const uint32_t post = region + static_cast<uint32_t>(pw::kLutRegionBytes);
  if (post + static_cast<uint32_t>(kPostBytes) > base + static_cast<uint32_t>(kSmemBytes)) {
    if (threadIdx.x == 0) report(p.status, PW_ERR_UNSUPPORTED);   // unexpected shared-window base
    return;
  }
  auto at = [&](uint32_t addr) { return smem_raw + (addr - base); };
  SmemT sm;
  uint32_t cur = pre;
  sm.b_ring = at(cur);
  cur += kBRingBytes;
  sm.bar = cur;
  cur += kBarBytes;
  sm.rows = reinterpret_cast<int*>(at(cur));
  cur += kRowsBytes;
  sm.st = reinterpret_cast<DecState*>(at((cur + 15u) & ~15u));
  sm.lut_region = region;
  sm.plane_ring = at(post);
  sm.xch = reinterpret_cast<float*>(at(post + kG * kPlaneRing));

  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int g = 0; g < kG; ++g) {
      const uint32_t g0 = group_bar(sm, g);
      for (int i = 0; i < kF; ++i) {
        pw::mbar_init(bar_full(g0, i), kDeqWarps);
        pw::mbar_init(bar_free(g0, i), 1);
      }
      pw::mbar_init(bar_done(g0), 1);
    }
    for (int s = 0; s < 2; ++s) {
      pw::mbar_init(unit_ready_bar(sm, s), 1);
      pw::mbar_init(unit_free_bar(sm, s), kG * kDeqWarps + kG);
    }
    pw::mbar_init_fence();
    sm.st->sched.abort = 0;
    setup_schedule<kN>(p, sm.st->sched);
  }
  if (warp == 0) {
    pw::tmem_alloc(pw::smem_u32(&sm.st->sched.tmem), kTmemColsT);
    pw::tmem_relinquish();
  }
  pw::tc_fence_before();
  __syncthreads();
  pw::tc_fence_after();
  const uint32_t tmem = sm.st->sched.tmem;

  int abort_local = 0;
  if (warp == kSchedWarp) {
    if ((threadIdx.x & 31) == 0) scheduler(p, sm);
  } else if (warp >= kMmaWarp0) {
    uint32_t tcnt = 0;
    for (uint32_t i = 0;; ++i) {
      wait_unit(sm, i, p, abort_local);
      const Unit& u = sm.st->units[i & 1u];
      if (u.kind == kNone || abort_local) break;
      mma_unit(u, sm, tmem, tcnt, p, abort_local);
      if ((threadIdx.x & 31) == 0) pw::mbar_arrive(unit_free_bar(sm, static_cast<int>(i & 1u)));
    }
  } else {
    uint32_t tcnt = 0;
    bool early = false;
    for (uint32_t i = 0;; ++i) {
      wait_unit(sm, i, p, abort_local);
      const int s = static_cast<int>(i & 1u);
      const Unit& u = sm.st->units[s];
      if (u.kind == kNone || abort_local) break;
      const int* urows = sm.rows + s * kN;
      switch (u.q) {
        case 2: early = dequant_unit<2>(p, u, sm, urows, tmem, tcnt, i, s, early, abort_local); break;
        case 3: early = dequant_unit<3>(p, u, sm, urows, tmem, tcnt, i, s, early, abort_local); break;
        case 4: early = dequant_unit<4>(p, u, sm, urows, tmem, tcnt, i, s, early, abort_local); break;
        case 5: early = dequant_unit<5>(p, u, sm, urows, tmem, tcnt, i, s, early, abort_local); break;
        case 6: early = dequant_unit<6>(p, u, sm, urows, tmem, tcnt, i, s, early, abort_local); break;
        case 7: early = dequant_unit<7>(p, u, sm, urows, tmem, tcnt, i, s, early, abort_local); break;
        default: early = dequant_unit<8>(p, u, sm, urows, tmem, tcnt, i, s, early, abort_local); break;
      }
      // every epilogue store of both groups is issued: publish the unit
      named_sync_dequant();
      if (threadIdx.x == 0) sm.st->combine = finish_unit(p, sm.st->sched, u, 0);
      named_sync_dequant();
      if (sm.st->combine >= 0) combine_strip(p, sm.st->combine, threadIdx.x, kDeqAll);
      if (abort_local) {
        report(p.status, PW_ERR_TIMEOUT);
        sm.st->sched.abort = 1;
      }
      if ((threadIdx.x & 31) == 0) pw::mbar_arrive(unit_free_bar(sm, s));
    }
  }
  pw::tc_fence_before();
  __syncthreads();
  pw::tc_fence_after();
  if (warp == 0) pw::tmem_dealloc(tmem, kTmemColsT);
}

}  // namespace

int launch_decode_kernel(const Params& p, cudaStream_t s) {
  static bool attr_done = false;
  if (!attr_done) {
    PW_CUDA_TRY(cudaFuncSetAttribute(apl_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes));
    attr_done = true;
  }
  const int sms = sm_count_cached();
  if (sms < 1) return pw::set_error(PW_ERR_CUDA, "could not query the SM count");
  // one CTA per SM: it owns all 512 TMEM columns
  apl_decode_kernel<<<sms, kThreads, kSmemBytes, s>>>(p);
  PW_CUDA_TRY(cudaGetLastError());
  return PW_OK;
}

}  // namespace pw_ffn
