// Fused MoE layer kernel body, instantiated per token-tile width: a
// translation unit defines PW_TILE_N (16, 32, 64 or 128 tokens per tile),
// PW_KERNEL_NAME and PW_LAUNCHER_NAME, then includes this file.  See
// ffn_common.cuh for the work units and their scheduling.
//
// One CTA per SM (persistent), in seven roles:
//   warps 0-15, dequant: four sets of four warps (one warp per TMEM lane
//     quadrant, one thread per row of the strip); tile x of the CTA's tile
//     stream goes to set x % 4.  A thread reads its row's 16 bytes of every
//     committed plane of its tile from a shared chunk, turns the row's 128
//     columns into fp16 through its LUT (dequant.cuh) and stores them as
//     operand A in one of the TMEM A slots (tcgen05.st);
//   MMA issuers (one thread per warp; 4 for N <= 32, 2 for N = 64, 1 for
//     N = 128, whose two accumulator buffers take half of TMEM): issuer k
//     takes the tiles x with x % issuers == k and issues each tile's eight
//     tcgen05.mma (A from TMEM, B from shared memory, fp32 accumulator in its
//     own double-buffered TMEM columns), committed to the tile's "free"
//     barrier, which releases its TMEM slot and its B slot.  Several issuing
//     warps are needed: one thread issues an N <= 128 MMA only every ~45 ns;
//   4 epilogue warps: copy each unit's LUT into a shared region one or two
//     units ahead (two halves used alternately), sum the issuers'
//     accumulators of a unit and write h = silu(gate)*up, down-projection
//     partial sums or the linear output; then publish the unit.  After the
//     last unit the whole grid runs the deterministic top-k combine (with
//     PW_FFN_FLAG_STRIP_COMBINE, a strip's last down unit combines it
//     instead);
//   plane loader warp: per chunk of a unit's consecutive tiles, one bulk copy
//     per plane (a run of tiles of one plane is contiguous) into a slot;
//   scheduler (one thread): takes tickets and publishes units into four slots
//     ahead of the other roles;
//   B loader (one thread): each tile's B operand (the N tokens' x or h
//     columns: one 3-D tensor-map box, both 64-column atoms, in the
//     128-byte-swizzled layout the tensor core reads) into a ring.
// Gate_up B rows are the routed tokens' x rows in expert order; every CTA
// gathers a share of them into the workspace at the start and the B loader
// waits for all shares before the first gate_up copy.
// All waits are bounded (PW_ERR_TIMEOUT); no role waits without a time limit
// on a barrier that a failed role could leave unfinished, every copy lands
// before its CTA exits, and TMEM is released before the CTA exits.
#include <cuda.h>

#include "ffn_common.cuh"
#include "route_block.cuh"

namespace pw_ffn {
namespace {

#ifndef PW_TILE_N
#error "define PW_TILE_N (16, 32, 64 or 128) before including ffn_stream.cuh"
#endif
#ifndef PW_GEMV
#define PW_GEMV 0
#endif
constexpr int kN = PW_TILE_N;                     // tokens per tile
// CUDA-core instance: the dequant warps multiply the dequantised weights with
// the tile's (at most kN = 2) token rows themselves (fp32 FMA) instead of
// handing them to the tensor core; no MMA issuers, no TMEM A slots
constexpr bool kGemv = PW_GEMV != 0;
static_assert(kGemv ? kN == 2 : (kN == 16 || kN == 32 || kN == 64 || kN == 128), "tile widths");
constexpr int kSets = 4;                          // dequant warp sets
constexpr int kIssuers = kGemv ? 0 : (kN <= 32 ? 4 : (kN == 64 ? 2 : 1));   // MMA issuing warps
constexpr int kAccSlots = kGemv ? kSets : kIssuers;   // partial accumulators summed by the epilogue
constexpr int kAccCols = kN < 16 ? 16 : kN;           // TMEM columns per partial accumulator
constexpr int kIssuersOr1 = kIssuers > 0 ? kIssuers : 1;
constexpr int kDeqWarpsAll = kSets * 4;           // warps 0-15
constexpr int kMmaWarp0 = kDeqWarpsAll;           // MMA issuers
constexpr int kEpiWarp0 = kMmaWarp0 + kIssuers;   // 4 epilogue warps
constexpr int kEpiThreads = 128;
constexpr int kLoadWarp = kEpiWarp0 + 4;          // plane chunks
constexpr int kSchedWarp = kLoadWarp + 1;
constexpr int kBLoadWarp = kSchedWarp + 1;        // B operands
constexpr int kThreads = (kBLoadWarp + 1) * 32;
constexpr int kSA = kGemv ? 0 : (kN <= 16 ? 6 : 4);   // TMEM A slots
constexpr int kSAOr1 = kSA > 0 ? kSA : 1;
constexpr int kATileCols = 64;                    // TMEM columns per A tile (128 fp16 per row)
constexpr int kDCol0 = kSA * kATileCols;          // accumulators: [buffer][issuer] x kN columns from here
constexpr int kTmemCols = 512;
constexpr int kF = 16;                            // tile barrier slots (tile index mod 16)
constexpr int kUS = 4;                            // unit slots
constexpr int kBS = kGemv ? 8 : (kN <= 32 ? 6 : (kN == 64 ? 3 : 2));   // B ring slots
constexpr int kBAtom = kN * 128;                  // kN rows x 64 fp16 (128-byte swizzle; unswizzled for kGemv)
constexpr int kBBytes = 2 * kBAtom;               // B of one tile
constexpr int kPS = kN <= 16 ? 4 : (kN == 64 ? 3 : 2);        // plane chunk slots
constexpr int kPSlotBytes = 32768;                // one chunk: up to 4 tiles x 4 planes or 2 tiles x 8 planes
constexpr int kSmemBytes = 232448;
constexpr uint32_t kHintNs = 20000;
// Unroll of the two half-rows of a tile: the 16- and 32-token kernels run
// faster with the smaller loop body (fewer instruction-fetch stalls), the
// 64-token kernel with both halves unrolled (measured).
constexpr int kHalfUnroll = kN <= 32 ? 1 : 2;
static_assert(kDCol0 + 2 * kAccSlots * kAccCols <= kTmemCols, "TMEM columns");
static_assert(kSA <= kF && 2 * kBS <= kF, "barrier reuse distances");
static_assert(4 * 4 * 2048 <= kPSlotBytes && 2 * 8 * 2048 <= kPSlotBytes, "chunk sizes");
static_assert(kGemv || kSets % kIssuersOr1 == 0, "issuers share sets evenly");
static_assert(pw_route::scratch_bytes(pw_route::kMaxE, kThreads / 32) <= pw::kLutRegionBytes,
              "routing scratch fits the LUT region");

enum : int {
  kBarAFull = 0,                  // [kF]  A slot written (4 warps of a set)
  kBarTFree = kF,                 // [kF]  tile's MMAs done (tcgen05.commit)
  kBarBFull = 2 * kF,             // [kBS] B slot loaded (transaction bytes)
  kBarPFull = 2 * kF + kBS,       // [kPS] plane chunk loaded (transaction bytes)
  kBarPFree = kBarPFull + kPS,    // [kPS] plane chunk consumed (16 dequant warps)
  kBarDone = kBarPFree + kPS,     // [2]   unit's accumulators complete (one arrival per issuer)
  kBarDFree = kBarDone + 2,       // [2]   accumulator read (4 epilogue warps)
  kBarRegReady = kBarDFree + 2,   // [2]   the unit's LUT landed in its region half (bulk copy bytes)
  kBarEpiDone = kBarRegReady + 2,
  kBarEpiGo = kBarEpiDone + 1,
  kBarUReady = kBarEpiGo + 1,     // [kUS]
  kBarUFree = kBarUReady + kUS,   // [kUS]
  kNumBars = kBarUFree + kUS
};
constexpr int kBarBytes = 512;
static_assert(kNumBars * 8 <= kBarBytes, "barrier area");
constexpr uint32_t kUnitFreeCount = kDeqWarpsAll + kIssuers + 4 + 2;

struct DecState {
  Shared sched;                              // ticket decoding state (scheduler thread)
  Unit units[kUS];                           // published units
  const uint32_t* planes[kUS][PW_MAX_BITS];  // each published unit's first tile, per plane
  uint32_t deq_done;                         // units finished, summed over the 16 dequant warps
  uint32_t bring;                            // B ring (shared address)
  uint32_t pslot[kPS];                       // plane chunk slots (shared addresses)
  int combine;
  int abort;                                 // CTA-wide: give up waiting
};

struct Sm {
  uint32_t bar;              // first barrier (shared address)
  uint32_t region;           // 64 KB-aligned LUT region (q >= 5)
  DecState* st;              // also holds the B ring and plane slot addresses
};

__device__ __forceinline__ uint32_t bar(const Sm sm, int i) { return sm.bar + 8u * static_cast<uint32_t>(i); }

__device__ __forceinline__ void fail(const Params& p, DecState& st) {
  st.abort = 1;
  report(p.status, PW_ERR_TIMEOUT);
  atomicExch(p.ctr + 1, 1u);
}

// Bounded wait for phase `parity`; gives up early once the CTA aborts.
__device__ __forceinline__ bool wait_bar(const Sm sm, int i, uint32_t parity, const Params& p) {
  const uint32_t b = bar(sm, i);
  if (pw::mbar_try_wait_hint(b, parity, kHintNs)) return true;
  const uint64_t t0 = pw::global_ns();
  volatile int* abort = &sm.st->abort;
  while (true) {
    if (pw::mbar_try_wait_hint(b, parity, kHintNs)) return true;
    if (*abort) return false;
    if (pw::global_ns() - t0 > p.wait_ns) {
      fail(p, *sm.st);
      return false;
    }
  }
}

// Bounded wait that ignores the abort flag (copies and MMAs already issued
// must land before the CTA exits).  Giving up (after 100 ms) is reported as
// PW_ERR_TIMEOUT.
__device__ __forceinline__ void drain_bar(const Sm sm, int i, uint32_t parity, int32_t* status) {
  const uint64_t t0 = pw::global_ns();
  while (!pw::mbar_try_wait_hint(bar(sm, i), parity, kHintNs))
    if (pw::global_ns() - t0 > 100000000ull) {
      report(status, PW_ERR_TIMEOUT);
      return;
    }
}

// Bounded wait until a shared counter reaches `target`.
__device__ __forceinline__ bool wait_count(const Sm sm, const uint32_t* ctr, uint32_t target, const Params& p) {
  const volatile uint32_t* c = ctr;
  if (*c >= target) {
    __threadfence_block();
    return true;
  }
  const uint64_t t0 = pw::global_ns();
  volatile int* abort = &sm.st->abort;
  while (*c < target) {
    if (*abort) return false;
    if (pw::global_ns() - t0 > p.wait_ns) {
      fail(p, *sm.st);
      return false;
    }
    __nanosleep(64);
  }
  __threadfence_block();
  return true;
}

// Lane 0 waits for unit i to be published; the warp then reads it.
__device__ __forceinline__ bool wait_unit(const Sm sm, uint32_t i, const Params& p) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = wait_bar(sm, kBarUReady + static_cast<int>(i % kUS), (i / kUS) & 1u, p);
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// TMEM column of partial accumulator k (an MMA issuer's, or a set's on the
// CUDA-core instance) in buffer db.
__device__ __forceinline__ uint32_t acc_col(uint32_t db, int k) {
  return kDCol0 + (db * kAccSlots + static_cast<uint32_t>(k)) * kAccCols;
}

// ---------------------------------------------------------------------------
// dequant warps
// ---------------------------------------------------------------------------
// Plane chunks: the loader copies a unit's tiles in chunks of consecutive
// tiles (4 for q <= 4, 3 for q = 5 in the 16-token kernel, else 2; at most 32
// KB and at most one tile per dequant set), one bulk copy per plane, into kPS
// fixed slots.  Slot layout: [plane][tile of the chunk][row pos][16 B], plane
// stride chunk_tiles * 2 KB.  Every dequant warp waits for each chunk and
// signals it consumed, whether or not its set has a tile in it.  (Three-tile
// chunks at q = 5 keep 30 instead of 20 KB of a slot in flight: 4 % faster at
// b = 5 with four slots; with the 64-token kernel's three slots they measured
// 2 % slower.)
__host__ __device__ constexpr int chunk_tiles(int q) { return q <= 4 ? 4 : (q == 5 && kN <= 16 ? 3 : 2); }
static_assert(3 * 5 * 2048 <= kPSlotBytes, "chunk sizes");

// Returns false when a wait gave up (the CTA aborts); a chunk the warp did
// not see land is then never released, so no copy can be issued over one
// still in flight.
template <int Q>
__device__ __forceinline__ bool dequant_unit(const Params& p, const Unit& u, const Sm sm, uint32_t tmem, uint32_t x0,
                                             uint32_t c0, uint32_t ui) {
  constexpr int kCt = chunk_tiles(Q);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int set = warp >> 2, qd = warp & 3;
  const int pos = qd * 32 + lane;
  bool ok = true;
  // q <= 3: LUT in registers; q >= 4: LUT in the shared region (for four
  // planes the transpose and shared lookups cost fewer logic ops than the
  // two-level register lookup)
  pw::RowDequant<Q, (Q <= 3)> dq;
  // the unit's LUT has landed in region half ui & 1 (one bulk copy of the
  // strip's table, issued one unit ahead; a q = 8 table fills the region)
  ok = wait_bar(sm, kBarRegReady + static_cast<int>(ui & 1u), (ui >> 1) & 1u, p);
  if constexpr (Q <= 3) {
    const uint32_t rowoff = static_cast<uint32_t>((qd & 1) * 32 + lane) * 4u + static_cast<uint32_t>(qd >> 1) * 2u;
    if (ok) dq.load_region(sm.region + (ui & 1u) * 32768u + rowoff);
  } else {
    dq.set_row(sm.region, qd, lane, static_cast<int>(ui & 1u));
  }
  const int nt = u.nst / 2;
  const int nch = (nt + kCt - 1) / kCt;
  const uint32_t tl = tmem + (static_cast<uint32_t>(32 * qd) << 16);
  float gacc[kGemv ? kN : 1];   // CUDA-core instance: this row's partial sums, one per token
#pragma unroll
  for (int r = 0; r < (kGemv ? kN : 1); ++r) gacc[r] = 0.f;
  for (int k = 0; k < nch; ++k) {
    const uint32_t c = c0 + static_cast<uint32_t>(k);
    const int ps = static_cast<int>(c % kPS);
    const int n_in = min(kCt, nt - k * kCt);
    const uint32_t xs = x0 + static_cast<uint32_t>(k * kCt);
    const int j = static_cast<int>((static_cast<uint32_t>(set) - xs) & 3u);   // this set's tile in the chunk
    const bool has = ok && j < n_in;
    if (ok) ok = wait_bar(sm, kBarPFull + ps, (c / kPS) & 1u, p);
    if (!ok) return false;
    if constexpr (kGemv) if (has) {
      // the tile's token rows (B slot x % kBS, row-major: atom of 64
      // columns, 128 bytes per row); the slot's previous tile (x - kBS,
      // another set's) must be consumed before its parity names tile x
      const uint32_t x = xs + static_cast<uint32_t>(j);
      if (x >= kBS && !wait_bar(sm, kBarTFree + static_cast<int>((x - kBS) % kF), ((x - kBS) / kF) & 1u, p))
        ok = false;
      if (ok && !wait_bar(sm, kBarBFull + static_cast<int>(x % kBS), (x / kBS) & 1u, p)) ok = false;
      if (ok) {
        const uint32_t src = sm.st->pslot[ps] + static_cast<uint32_t>(j) * pw::kTileBytes + pos * 16;
        const uint32_t bsm = sm.st->bring + (x % kBS) * kBBytes;
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t w2[Q][2];
#pragma unroll
          for (int q = 0; q < Q; ++q) pw::lds_v2(src + q * (kCt * pw::kTileBytes) + hh * 8, w2[q][0], w2[q][1]);
#pragma unroll
          for (int wd = 0; wd < 2; ++wd) {
            uint32_t ww[Q];
#pragma unroll
            for (int q = 0; q < Q; ++q) ww[q] = w2[q][wd];
            uint32_t out[16];
            dq.word(ww, out);
            // columns 32 * (2 hh + wd) .. + 31 of the tile: atom hh, 64 bytes
            // from byte 64 wd of each token row
            const uint32_t xrow = bsm + hh * kBAtom + wd * 64;
#pragma unroll
            for (int r = 0; r < kN; ++r) {
              if (r < u.nrows) {
                uint32_t xv[16];
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                  uint32_t v4[4];
                  pw::lds_v4u(xrow + r * 128 + c4 * 16, v4);
#pragma unroll
                  for (int m = 0; m < 4; ++m) xv[4 * c4 + m] = v4[m];
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  const float2 wf = __half22float2(*reinterpret_cast<const __half2*>(&out[i]));
                  const float2 xf = __half22float2(*reinterpret_cast<const __half2*>(&xv[i]));
                  gacc[r] = fmaf(wf.x, xf.x, gacc[r]);
                  gacc[r] = fmaf(wf.y, xf.y, gacc[r]);
                }
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) pw::mbar_arrive(bar(sm, kBarTFree + static_cast<int>(x % kF)));   // B slot consumed
      }
    }
    if constexpr (!kGemv) if (has) {
      const uint32_t x = xs + static_cast<uint32_t>(j);
      if (x >= kSA && !wait_bar(sm, kBarTFree + static_cast<int>((x - kSA) % kF), ((x - kSA) / kF) & 1u, p))
        ok = false;
      if (ok) {
        pw::tc_fence_after();
        const uint32_t acol = tl + (x % kSAOr1) * kATileCols;
        const uint32_t src = sm.st->pslot[ps] + static_cast<uint32_t>(j) * pw::kTileBytes + pos * 16;
#pragma unroll kHalfUnroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t w2[Q][2];
#pragma unroll
          for (int q = 0; q < Q; ++q) pw::lds_v2(src + q * (kCt * pw::kTileBytes) + hh * 8, w2[q][0], w2[q][1]);
#pragma unroll
          for (int wd = 0; wd < 2; ++wd) {
            uint32_t ww[Q];
#pragma unroll
            for (int q = 0; q < Q; ++q) ww[q] = w2[q][wd];
            uint32_t out[16];
            dq.word(ww, out);
            pw::tmem_st_x16(acol + 16 * (2 * hh + wd), out);
          }
        }
        pw::tmem_st_wait();
        pw::tc_fence_before();
        __syncwarp();
        if (lane == 0) pw::mbar_arrive(bar(sm, kBarAFull + static_cast<int>(x % kF)));
      }
    }
    __syncwarp();
    if (lane == 0) pw::mbar_arrive(bar(sm, kBarPFree + ps));   // this warp is done with the chunk
  }
  if constexpr (kGemv) {
    // the set's partial sums (its tiles x = set mod 4) into its accumulator
    // columns, once the epilogue has read unit ui - 2 from that buffer
    if (!ok) return false;
    const uint32_t db = ui & 1u;
    if (ui >= 2 && !wait_bar(sm, kBarDFree + static_cast<int>(db), ((ui - 2) >> 1) & 1u, p)) return false;
    const uint32_t v[2] = {__float_as_uint(gacc[0]), __float_as_uint(gacc[(kGemv && kN > 1) ? 1 : 0])};
    pw::tc_fence_after();
    pw::tmem_st_x2(tl + acc_col(db, set), v);
    pw::tmem_st_wait();
    pw::tc_fence_before();
    __syncwarp();
    if (lane == 0) pw::mbar_arrive(bar(sm, kBarDone + static_cast<int>(db)));
  }
  return ok;
}

__device__ __forceinline__ void dequant_role(const Params& p, const Sm sm, uint32_t tmem) {
  uint32_t x = 0, c = 0;
  for (uint32_t i = 0;; ++i) {
    if (!wait_unit(sm, i, p)) break;
    const Unit& u = sm.st->units[i % kUS];
    if (u.kind == kNone) break;
    bool ok;
    switch (u.q) {
      case 2: ok = dequant_unit<2>(p, u, sm, tmem, x, c, i); break;
      case 3: ok = dequant_unit<3>(p, u, sm, tmem, x, c, i); break;
      case 4: ok = dequant_unit<4>(p, u, sm, tmem, x, c, i); break;
      case 5: ok = dequant_unit<5>(p, u, sm, tmem, x, c, i); break;
      case 6: ok = dequant_unit<6>(p, u, sm, tmem, x, c, i); break;
      case 7: ok = dequant_unit<7>(p, u, sm, tmem, x, c, i); break;
      default: ok = dequant_unit<8>(p, u, sm, tmem, x, c, i); break;
    }
    // after an abort the warp stops: an unfinished unit is not counted, so
    // no LUT copy is issued into a region half whose copy may still be
    // in flight
    if (!ok) break;
    const int nt = u.nst / 2, ct = chunk_tiles(u.q);
    x += static_cast<uint32_t>(nt);
    c += static_cast<uint32_t>((nt + ct - 1) / ct);
    __syncwarp();
    if ((threadIdx.x & 31) == 0) {
      // a monotonic count, not a barrier phase: the LUT writers may look at it
      // several units later
      __threadfence_block();
      atomicAdd(&sm.st->deq_done, 1u);
      pw::mbar_arrive(bar(sm, kBarUFree + static_cast<int>(i % kUS)));
    }
  }
}

// ---------------------------------------------------------------------------
// plane loader warp: plane chunks and LUT prefetch (lane 0 waits and signals;
// lanes issue one bulk copy per plane)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void plane_loader_role(const Params& p, const Sm sm) {
  const int lane = threadIdx.x & 31;
  DecState& st = *sm.st;
  uint32_t c = 0;
  bool ok = true;
  for (uint32_t u = 0; ok; ++u) {
    if (!wait_unit(sm, u, p)) break;
    const int us = static_cast<int>(u % kUS);
    const Unit& un = st.units[us];
    if (un.kind == kNone) break;
    const BlockDesc& d = *un.d;
    const int Q = un.q, ct = chunk_tiles(Q), nt = un.nst / 2;
    if (lane == 0) {
      // the unit's LUT (its strip's table, one contiguous run) into L2 ahead
      // of the bulk copy into the region
      const uint32_t bytes = 256u << Q;
      pw::prefetch_l2(reinterpret_cast<const char*>(d.lut) + static_cast<long long>(un.strip) * bytes, bytes);
    }
    const uint32_t* plane = lane < Q ? st.planes[us][lane] : nullptr;
    for (int t0 = 0; t0 < nt; t0 += ct, ++c) {
      const int n_in = min(ct, nt - t0);
      const int ps = static_cast<int>(c % kPS);
      const uint32_t fb = bar(sm, kBarPFull + ps);
      int r = 1;
      if (lane == 0) {
        // the slot's previous chunk must be consumed by every dequant warp
        if (c >= kPS) r = wait_bar(sm, kBarPFree + ps, ((c - kPS) / kPS) & 1u, p);
        if (r) pw::mbar_arrive_expect_tx(fb, static_cast<uint32_t>(Q * n_in) * pw::kTileBytes);
      }
      if (!__shfl_sync(0xffffffffu, r, 0)) {
        ok = false;
        break;
      }
      if (lane < Q)
        pw::bulk_g2s(st.pslot[ps] + static_cast<uint32_t>(lane * ct) * pw::kTileBytes,
                     plane + static_cast<long long>(t0) * (pw::kTileBytes / 4),
                     static_cast<uint32_t>(n_in) * pw::kTileBytes, fb);
    }
    if (!ok) break;
    __syncwarp();
    if (lane == 0) pw::mbar_arrive(bar(sm, kBarUFree + static_cast<int>(u % kUS)));
  }
  // the last copies land before the CTA exits
  if (lane == 0)
    for (uint32_t y = c > static_cast<uint32_t>(kPS) ? c - kPS : 0u; y < c; ++y)
      drain_bar(sm, kBarPFull + static_cast<int>(y % kPS), (y / kPS) & 1u, p.status);
  __syncwarp();
}

// ---------------------------------------------------------------------------
// B loader (one thread): each tile's N token rows, one tensor-map box
// ---------------------------------------------------------------------------
__device__ __forceinline__ void b_loader_role(const Params& p, const Sm sm, const void* map_gu, const void* map_dn) {
  DecState& st = *sm.st;
  bool gathered = p.linear != 0;
  uint32_t x = 0;
  bool ok = true;
  for (uint32_t u = 0; ok; ++u) {
    if (!wait_bar(sm, kBarUReady + static_cast<int>(u % kUS), (u / kUS) & 1u, p)) break;
    const Unit& un = st.units[u % kUS];
    if (un.kind == kNone) break;
    if (un.kind == kGateUp && !gathered) {
      const uint64_t t0 = pw::global_ns();
      while (pw::ld_acquire_gpu(p.gather_ctr) < gridDim.x) {
        if (st.abort || pw::global_ns() - t0 > p.wait_ns) {
          if (!st.abort) fail(p, st);
          ok = false;
          break;
        }
        __nanosleep(100);
      }
      if (!ok) break;
      gathered = true;
    }
    if (un.kind != kLinear) pw::fence_proxy_async_global();   // x / h rows written by this kernel
    const void* map = un.kind == kDown ? map_dn : map_gu;
    const int brow = un.kind == kLinear ? un.tg * kN : un.off;
    const int tile0 = un.st0 / 2, nt = un.nst / 2;
    for (int t = 0; t < nt; ++t, ++x) {
      const int b = static_cast<int>(x % kBS);
      const uint32_t bb = bar(sm, kBarBFull + b);
      // the slot's previous tile (x - kBS) must be consumed by its MMAs
      if (x >= kBS && !wait_bar(sm, kBarTFree + static_cast<int>((x - kBS) % kF), ((x - kBS) / kF) & 1u, p)) {
        ok = false;
        break;
      }
      pw::mbar_arrive_expect_tx(bb, kBBytes);
      const uint32_t dst = st.bring + static_cast<uint32_t>(b) * kBBytes;
      const int col = (tile0 + t) * pw::kTileCols;
      pw::tma_load_3d(dst, map, 0, brow, col / 64, bb);
    }
    if (!ok) break;
    pw::mbar_arrive(bar(sm, kBarUFree + static_cast<int>(u % kUS)));
  }
  for (uint32_t y = x > static_cast<uint32_t>(kBS) ? x - kBS : 0u; y < x; ++y)
    drain_bar(sm, kBarBFull + static_cast<int>(y % kBS), (y / kBS) & 1u, p.status);
}

// ---------------------------------------------------------------------------
// MMA issuers: issuer k takes the tiles x with x % kIssuers == k and owns its
// own accumulators
// ---------------------------------------------------------------------------

__device__ __forceinline__ void mma_role(const Params& p, const Sm sm, uint32_t tmem, int k) {
  DecState& st = *sm.st;
  const uint32_t idesc = pw::idesc_f16_f32(128, kN);
  uint32_t x0 = 0;
  uint32_t last = 0;
  bool issued = false;
  for (uint32_t mu = 0;; ++mu) {
    if (!wait_bar(sm, kBarUReady + static_cast<int>(mu % kUS), (mu / kUS) & 1u, p)) break;
    const Unit& um = st.units[mu % kUS];
    if (um.kind == kNone) break;
    const uint32_t nt = static_cast<uint32_t>(um.nst / 2);
    const uint32_t db = mu & 1u;
    // this issuer's accumulator in buffer db is free once unit mu - 2's epilogue read it
    if (mu >= 2 && !wait_bar(sm, kBarDFree + static_cast<int>(db), ((mu - 2) >> 1) & 1u, p)) break;
    const uint32_t dcol = tmem + acc_col(db, k);
    bool ok = true, any = false;
    for (uint32_t x = x0 + ((static_cast<uint32_t>(k) - x0) % kIssuersOr1); x < x0 + nt; x += kIssuersOr1) {
      const int fs = static_cast<int>(x % kF), b = static_cast<int>(x % kBS);
      // B slot b last held tile x - kBS, which another issuer owns (kIssuers
      // does not divide kBS).  A parity wait only tells the two latest phases
      // apart, so that tile's phase must be complete before BFull's parity
      // names tile x: its MMAs being done implies it (they waited for it), and
      // the B loader waits for the same event before it refills the slot.
      if (x >= kBS && !wait_bar(sm, kBarTFree + static_cast<int>((x - kBS) % kF), ((x - kBS) / kF) & 1u, p)) {
        ok = false;
        break;
      }
      if (!wait_bar(sm, kBarBFull + b, (x / kBS) & 1u, p) || !wait_bar(sm, kBarAFull + fs, (x / kF) & 1u, p)) {
        ok = false;
        break;
      }
      pw::tc_fence_after();
      const uint32_t a = tmem + (x % kSAOr1) * kATileCols;
      const uint32_t bsm = sm.st->bring + static_cast<uint32_t>(b) * kBBytes;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint64_t bdesc = pw::sdesc_kmajor_sw128(bsm + (j >> 2) * kBAtom) + 2ull * (j & 3);
        pw::tc_mma_ts(dcol, a + 8 * j, bdesc, idesc, (any || j > 0) ? 1u : 0u);
      }
      pw::tc_commit(bar(sm, kBarTFree + fs));
      any = issued = true;
      last = x;
    }
    if (!ok) break;
    // one arrival per issuer on the unit's "done" barrier, after its MMAs
    if (any)
      pw::tc_commit(bar(sm, kBarDone + static_cast<int>(db)));
    else
      pw::mbar_arrive(bar(sm, kBarDone + static_cast<int>(db)));
    x0 += nt;
    pw::mbar_arrive(bar(sm, kBarUFree + static_cast<int>(mu % kUS)));
  }
  // the last MMAs complete before the CTA exits
  if (issued) drain_bar(sm, kBarTFree + static_cast<int>(last % kF), (last / kF) & 1u, p.status);
}

// ---------------------------------------------------------------------------
// epilogue warps: LUT region one unit ahead, then the unit's epilogue
// ---------------------------------------------------------------------------
// Copies of the units' LUTs into the shared region go out in unit order, from
// thread 0 of the epilogue warps; `next` is the first unit not copied yet and
// `last` the last one copied (drained at exit).
struct LutCopies {
  uint32_t next = 0;
  int last = -1;
  int last_h[2] = {-1, -1};   // the last copy into each region half
};

// One bulk copy of unit i's table (its strip's run of 2^q lines) into region
// half i & 1 (q = 8: the whole region), completing the half's barrier by its
// bytes.  The caller has seen every earlier user of those lines finish.
__device__ __forceinline__ void copy_lut(const Sm sm, uint32_t i, const Unit& u) {
  const int h = static_cast<int>(i & 1u);
  const uint32_t b = bar(sm, kBarRegReady + h);
  const uint32_t bytes = 256u << u.q;
  const char* src = reinterpret_cast<const char*>(u.d->lut) + static_cast<long long>(u.strip) * bytes;
  pw::fence_proxy_async_smem();   // the lines' earlier generic accesses before the async write
  pw::mbar_arrive_expect_tx(b, bytes);
  pw::bulk_g2s(sm.region + (u.q == 8 ? 0u : static_cast<uint32_t>(h) * 32768u), src, bytes, b);
}

// Copy unit i's LUT unless it went out early (lut_early), once every earlier
// user of its lines is finished: units up to i - 2 (the half's previous
// user), or up to i - 1 when unit i or i - 1 takes the whole region.  Returns
// 1 when done, 0 when unit i is the end marker, and -1 without waiting when
// `block` is false and unit i is not published yet.
__device__ __forceinline__ int lut_fill(const Params& p, const Sm sm, uint32_t i, bool& prev_q8, bool block,
                                        LutCopies& lc) {
  const int lane = threadIdx.x & 31;
  const int etid = threadIdx.x - kEpiWarp0 * 32;
  if (!block) {
    int pub = 0;
    if (lane == 0) pub = pw::mbar_test(bar(sm, kBarUReady + static_cast<int>(i % kUS)), (i / kUS) & 1u);
    if (!__shfl_sync(0xffffffffu, pub, 0)) return -1;
  }
  if (!wait_unit(sm, i, p)) return 0;
  const Unit& u = sm.st->units[i % kUS];
  if (u.kind == kNone) return 0;
  if (etid == 0) {
    if (lc.next <= i) {
      const uint32_t need = static_cast<uint32_t>(kDeqWarpsAll) * ((u.q == 8 || prev_q8) ? i : (i >= 1 ? i - 1 : 0u));
      // giving up (abort) issues nothing: a region half's phases complete
      // only by copies, which the exit drain relies on
      if (wait_count(sm, &sm.st->deq_done, need, p) && !*reinterpret_cast<volatile int*>(&sm.st->abort)) {
        copy_lut(sm, i, u);
        lc.last = lc.last_h[i & 1u] = static_cast<int>(i);
      }
      lc.next = i + 1;
    }
    prev_q8 = u.q == 8;
  }
  return 1;
}

// Thread 0 of the epilogue warps, once unit j - 2's MMAs are done: copy unit
// j's table now if it is next in order, published, neither j nor j - 1 takes
// the whole region, and every dequant warp has finished unit j - 2 (the
// half's previous user).  Otherwise lut_fill copies it later.  Never waits.
__device__ __forceinline__ void lut_early(const Sm sm, uint32_t j, LutCopies& lc) {
  if (lc.next != j || j < 2) return;
  if (!pw::mbar_test(bar(sm, kBarUReady + static_cast<int>(j % kUS)), (j / kUS) & 1u)) return;
  const Unit& u = sm.st->units[j % kUS];
  const Unit& prev = sm.st->units[(j - 1) % kUS];
  if (u.kind == kNone || u.q == 8 || prev.q == 8) return;
  if (*reinterpret_cast<volatile uint32_t*>(&sm.st->deq_done) < static_cast<uint32_t>(kDeqWarpsAll) * (j - 1)) return;
  __threadfence_block();
  copy_lut(sm, j, u);
  lc.last = lc.last_h[j & 1u] = static_cast<int>(j);
  lc.next = j + 1;
}

__device__ __forceinline__ void epilogue_unit(const Params& p, const Sm sm, uint32_t tmem, uint32_t i, uint32_t x0,
                                              LutCopies& lc) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qd = warp & 3;
  const int pos = qd * 32 + lane;
  const int etid = threadIdx.x - kEpiWarp0 * 32;
  DecState& st = *sm.st;
  const Unit& u = st.units[i % kUS];
  const uint32_t db = i & 1u;
  const bool ok = wait_bar(sm, kBarDone + static_cast<int>(db), (i >> 1) & 1u, p);
  if (etid == 0 && ok) lut_early(sm, i + 2, lc);   // unit i's region half is free again
  const uint32_t nt = static_cast<uint32_t>(u.nst / 2);
  const BlockDesc& d = *u.d;
  const int row = strip_pos_row(u.strip, pos, d.rows / 2);
  // 16 token columns at a time: the sum of the accumulators of the issuers
  // that hold a tile of the unit (issuer k holds x0 <= x < x0 + nt with
  // x % kIssuers == k, i.e. the unit's tiles t with t = k - x0 mod kIssuers).
  // The partial sums are added in the order of that residue, not of the
  // issuer, so the result does not depend on which CTA took the unit.
  // only the column chunks that hold the unit's tokens (a 64-token tile with
  // a small token group reads one chunk, not four)
  const int nc16 = min(kAccCols / 16, (u.nrows + 15) / 16);
#pragma unroll 1
  for (int c16 = 0; c16 < nc16; ++c16) {
    float acc[16];
#pragma unroll
    for (int n = 0; n < 16; ++n) acc[n] = 0.f;
    if (ok) {
      pw::tc_fence_after();
      for (int r = 0; r < kAccSlots; ++r) {
        if (static_cast<uint32_t>(r) >= nt) continue;
        const int k2 = static_cast<int>((static_cast<uint32_t>(r) + x0) % kAccSlots);
        uint32_t v[16];
        pw::tmem_ld_x16(tmem + acc_col(db, k2) + 16u * c16 + (static_cast<uint32_t>(32 * qd) << 16), v);
        pw::tmem_ld_wait();
#pragma unroll
        for (int n = 0; n < 16; ++n) acc[n] += __uint_as_float(v[n]);
      }
    }
    if (c16 == nc16 - 1) {
      pw::tc_fence_before();
      __syncwarp();
      if (lane == 0) pw::mbar_arrive(bar(sm, kBarDFree + static_cast<int>(db)));   // all columns read
    }
    if (ok) {
#pragma unroll
      for (int n0 = 0; n0 < 16; ++n0) {
        const int n = 16 * c16 + n0;
        const float val = acc[n0];
        if (u.kind == kGateUp) {
          const float up = __shfl_down_sync(0xffffffffu, val, 16);
          if (lane < 16 && n < u.nrows) {
            const int m = u.strip * 64 + 16 * qd + lane;
            p.h[static_cast<long long>(u.off + n) * p.I + m] = __half_as_ushort(__float2half_rn(silu(val) * up));
          }
        } else if (u.kind == kDown) {
          if (n < u.nrows) p.part[(static_cast<long long>(u.split) * p.A + u.off + n) * p.H + row] = val;
        } else {
          if (n < u.nrows) p.out[static_cast<long long>(u.tg * kN + n) * d.rows + row] = val;
        }
      }
    }
  }
  if (ok && u.kind == kGateUp) pw::fence_proxy_async_global();   // h is read back through TMA
  __syncwarp();
  if (lane == 0) pw::mbar_arrive(bar(sm, kBarEpiDone));
  if (etid == 0) {
    int c = -1;
    if (wait_bar(sm, kBarEpiDone, i & 1u, p) && ok) c = finish_unit(p, st.sched, u, 0);
    st.combine = c;
    pw::mbar_arrive(bar(sm, kBarEpiGo));
  }
  const bool go = wait_bar(sm, kBarEpiGo, i & 1u, p);
  const int c = *reinterpret_cast<volatile int*>(&st.combine);
  if (go && c >= 0) combine_strip(p, c, etid, kEpiThreads);
  __syncwarp();
  if (lane == 0) pw::mbar_arrive(bar(sm, kBarUFree + static_cast<int>(i % kUS)));
}

// The next unit's LUT goes first when that unit is already published; the
// role never waits for a publication before finishing the current unit's
// epilogue (the scheduler may be waiting, for a down unit, on exactly that
// epilogue's gate_up completion).
__device__ __forceinline__ void epilogue_role(const Params& p, const Sm sm, uint32_t tmem) {
  bool prev_q8 = false;
  LutCopies lc;
  int more = lut_fill(p, sm, 0, prev_q8, true, lc);
  uint32_t x0 = 0;
  for (uint32_t i = 0; more == 1; ++i) {
    // fill the next unit's table as soon as it is published, but do not wait
    // for its publication past the moment this unit's accumulators are ready
    int next = lut_fill(p, sm, i + 1, prev_q8, false, lc);
    while (next < 0) {
      int done = 0;
      if ((threadIdx.x & 31) == 0) done = pw::mbar_test(bar(sm, kBarDone + static_cast<int>(i & 1u)), (i >> 1) & 1u);
      if (__shfl_sync(0xffffffffu, done, 0) || sm.st->abort) break;
      __nanosleep(128);
      next = lut_fill(p, sm, i + 1, prev_q8, false, lc);
    }
    const uint32_t nt = static_cast<uint32_t>(sm.st->units[i % kUS].nst / 2);
    epilogue_unit(p, sm, tmem, i, x0, lc);
    x0 += nt;
    if (next < 0) next = lut_fill(p, sm, i + 1, prev_q8, true, lc);
    more = next;
  }
  // Every LUT copy lands before the CTA exits.  On the normal path the
  // dequant warps waited for each copy before reading the unit's table, so
  // only the last one can still be in flight here.  After an abort they stop
  // consuming units: the last copy into either half may be pending.
  if (sm.st->abort) {
    for (int h = 0; h < 2; ++h)
      if (lc.last_h[h] >= 0)
        drain_bar(sm, kBarRegReady + h, (static_cast<uint32_t>(lc.last_h[h]) >> 1) & 1u, p.status);
  } else if (lc.last >= 0) {
    drain_bar(sm, kBarRegReady + (lc.last & 1), (static_cast<uint32_t>(lc.last) >> 1) & 1u, p.status);
  }
}

// ---------------------------------------------------------------------------
// scheduler (one thread)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void scheduler_role(const Params& p, const Sm sm) {
  DecState& st = *sm.st;
  for (uint32_t i = 0;; ++i) {
    const int s = static_cast<int>(i % kUS);
    if (i >= kUS && !wait_bar(sm, kBarUFree + s, ((i - kUS) / kUS) & 1u, p)) st.sched.abort = 1;
    if (st.abort) st.sched.abort = 1;
    Unit u;
    do {
      next_unit<kN>(p, st.sched);
      u = st.sched.u;
    } while (u.kind != kNone && u.skip);
    st.units[s] = u;
    if (u.kind != kNone) {
      const BlockDesc& d = *u.d;
      const long long first = (static_cast<long long>(u.strip) * (d.cols / pw::kTileCols) + u.st0 / 2) *
                              (pw::kTileBytes / 4);
      for (int q = 0; q < u.q; ++q) st.planes[s][q] = d.planes[q] + first;
    }
    pw::mbar_arrive(bar(sm, kBarUReady + s));
    if (u.kind == kNone) return;
  }
}

// Carve the dynamic shared memory: barriers and state, then the B ring and
// the plane rings in the space around the 64 KB-aligned LUT region.
__device__ __forceinline__ bool carve(Sm& sm, uint8_t* smem_raw) {
  const uint32_t base = pw::smem_u32(smem_raw);
  const uint32_t end = base + static_cast<uint32_t>(kSmemBytes);
  const uint32_t small = (base + 1023u) & ~1023u;
  sm.bar = small;
  const uint32_t st_addr = small + kBarBytes;
  sm.st = reinterpret_cast<DecState*>(smem_raw + (st_addr - base));
  const uint32_t small_end = st_addr + static_cast<uint32_t>(sizeof(DecState));
  sm.region = (small_end + 0xFFFFu) & ~0xFFFFu;
  uint32_t a = (small_end + 1023u) & ~1023u, b = sm.region + static_cast<uint32_t>(pw::kLutRegionBytes);
  auto take = [&](uint32_t size, uint32_t& out) {
    if (a + size <= sm.region) {
      out = a;
      a += size;
      return true;
    }
    if (b + size <= end) {
      out = b;
      b += size;
      return true;
    }
    return false;
  };
  uint32_t bring = 0, pslot[kPS] = {};
  bool ok = take(kBS * kBBytes, bring);
  for (int s = 0; s < kPS; ++s) ok = ok && take(kPSlotBytes, pslot[s]);
  if (threadIdx.x == 0) {
    sm.st->bring = bring;
    for (int s = 0; s < kPS; ++s) sm.st->pslot[s] = pslot[s];
  }
  return ok && sm.region + static_cast<uint32_t>(pw::kLutRegionBytes) <= end;
}

__global__ void __launch_bounds__(kThreads, 1)
    PW_KERNEL_NAME(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap map_gu,
                      const __grid_constant__ CUtensorMap map_dn) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // launched early after a routing launch: wait for it (and its writes)
  // before touching global memory; a no-op otherwise
  asm volatile("griddepcontrol.wait;" ::: "memory");
  Sm sm;
  if (!carve(sm, smem_raw)) {
    if (threadIdx.x == 0) report(p.status, PW_ERR_UNSUPPORTED);   // unexpected shared-window base
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  DecState& st = *sm.st;
  // routed call (batches one warp routes: at most 32 tokens and 8 experts
  // per layer; the host routes larger ones in a launch before this one):
  // warp 0 of CTA l routes layer l of the route_layers layers, writing the
  // routing arrays of all layers in one concatenated index space (the LUT
  // region is its scratch: the pipeline has not started), and counts the
  // layer as published; every CTA waits for all of them before it schedules
  // or gathers (all CTAs are resident: one per SM)
  if (p.logits) {
    const int L = p.route_layers, S = p.route_shared;
    const int Tl = p.T / L, ETl = p.E / L;
    const long long Al = static_cast<long long>(Tl) * p.k;
    float* scratch = reinterpret_cast<float*>(smem_raw + (sm.region - pw::smem_u32(smem_raw)));
    for (int l = blockIdx.x; l < L; l += gridDim.x) {
      if (warp == 0) {
        if (pw_route::warp_routes(Tl, ETl, p.k)) {
          pw_route::route_warp(p.logits + static_cast<long long>(l) * Tl * (ETl - S), Tl, ETl - S, p.k - S, S,
                               p.ids_out + l * Al, const_cast<float*>(p.w) + l * Al,
                               const_cast<int32_t*>(p.offsets) + static_cast<long long>(l) * ETl,
                               const_cast<int32_t*>(p.perm) + l * Al, const_cast<int32_t*>(p.inv_perm) + l * Al,
                               p.mass_accum ? p.mass_accum + static_cast<long long>(l) * ETl : nullptr, scratch,
                               static_cast<int>(l * Al));
        } else if (lane == 0) {
          report(p.status, PW_ERR_INVALID_ARG);   // the host routes such batches before the launch
        }
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(p.gather_ctr + 2, 1u);
      }
    }
    if (threadIdx.x == 0) {
      int ok = 1;
      const uint64_t t0 = pw::global_ns();
      while (pw::ld_acquire_gpu(p.gather_ctr + 2) < static_cast<uint32_t>(L)) {
        if (pw::global_ns() - t0 > p.wait_ns) {
          report(p.status, PW_ERR_TIMEOUT);
          ok = 0;
          break;
        }
        __nanosleep(64);
      }
      st.abort = ok ? 0 : 1;
    }
    __syncthreads();
    if (*reinterpret_cast<volatile int*>(&st.abort)) return;   // nothing allocated or issued yet
  }
  // the expert offsets into shared memory (the LUT region: the pipeline has
  // not started), all threads at once, so that thread 0's schedule set-up
  // does not wait a global-memory latency per expert
  int* s_offs = reinterpret_cast<int*>(smem_raw + (sm.region - pw::smem_u32(smem_raw)));
  if (!p.linear)
    for (int e = static_cast<int>(threadIdx.x); e <= p.E; e += kThreads) s_offs[e] = p.offsets[e];
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 0; i < kF; ++i) {
      pw::mbar_init(bar(sm, kBarAFull + i), 4);
      pw::mbar_init(bar(sm, kBarTFree + i), kGemv ? 4 : 1);   // a tile's MMAs' commit, or its set's 4 warps
    }
    for (int i = 0; i < kBS; ++i) pw::mbar_init(bar(sm, kBarBFull + i), 1);
    for (int i = 0; i < kPS; ++i) {
      pw::mbar_init(bar(sm, kBarPFull + i), 1);
      pw::mbar_init(bar(sm, kBarPFree + i), kDeqWarpsAll);
    }
    for (int i = 0; i < 2; ++i) {
      pw::mbar_init(bar(sm, kBarDone + i), kGemv ? kDeqWarpsAll : kIssuers);
      pw::mbar_init(bar(sm, kBarDFree + i), 4);
      pw::mbar_init(bar(sm, kBarRegReady + i), 1);
    }
    pw::mbar_init(bar(sm, kBarEpiDone), 4);
    pw::mbar_init(bar(sm, kBarEpiGo), 1);
    for (int s = 0; s < kUS; ++s) {
      pw::mbar_init(bar(sm, kBarUReady + s), 1);
      pw::mbar_init(bar(sm, kBarUFree + s), kUnitFreeCount);
    }
    pw::mbar_init_fence();
    st.abort = 0;
    st.deq_done = 0;
    st.sched.abort = 0;
    setup_schedule<kN>(p, s_offs, st.sched);
  }
  if (warp == 0) {
    pw::tmem_alloc(pw::smem_u32(&st.sched.tmem), kTmemCols);
    pw::tmem_relinquish();
  }
  if (warp == kBLoadWarp && lane == 0) {
    pw::prefetch_tmap(&map_gu);
    if (!p.linear) pw::prefetch_tmap(&map_dn);
  }
  // gate_up B rows: this CTA's share of x gathered into expert order
  if (!p.linear) {
    const int vrow = p.H / 8;
    const long long nvec = static_cast<long long>(p.A) * vrow;
    for (long long v = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; v < nvec;
         v += static_cast<long long>(gridDim.x) * kThreads) {
      const int a = static_cast<int>(v / vrow), c = static_cast<int>(v % vrow);
      const int slot = p.perm[a];
      if (static_cast<unsigned>(slot) >= static_cast<unsigned>(p.A)) {   // not a permutation of the slots
        report(p.status, PW_ERR_INVALID_ARG);
        continue;
      }
      const int tok = slot / p.k;
      const uint4 val = __ldg(reinterpret_cast<const uint4*>(p.x + static_cast<long long>(tok) * p.H) + c);
      reinterpret_cast<uint4*>(p.xp + static_cast<long long>(a) * p.H)[c] = val;
    }
    pw::fence_proxy_async_global();
  }
  pw::tc_fence_before();
  __syncthreads();
  pw::tc_fence_after();
  if (!p.linear && threadIdx.x == 0) {
    __threadfence();
    atomicAdd(p.gather_ctr, 1u);
  }
  const uint32_t tmem = st.sched.tmem;

  if (warp < kDeqWarpsAll) {
    dequant_role(p, sm, tmem);
  } else if (warp < kEpiWarp0) {
    if constexpr (!kGemv)
      if (lane == 0) mma_role(p, sm, tmem, warp - kMmaWarp0);
  } else if (warp < kLoadWarp) {
    epilogue_role(p, sm, tmem);
  } else if (warp == kLoadWarp) {
    plane_loader_role(p, sm);
  } else if (warp == kSchedWarp) {
    if (lane == 0) scheduler_role(p, sm);
  } else if (lane == 0) {
    b_loader_role(p, sm, &map_gu, &map_dn);
  }
  pw::tc_fence_before();
  __syncthreads();
  pw::tc_fence_after();
  if (warp == 0) pw::tmem_dealloc(tmem, kTmemCols);
  if (p.grid_combine) {
    // every CTA is done with its units: combine all rows with the whole grid
    if (threadIdx.x == 0) {
      __threadfence();
      atomicAdd(p.gather_ctr + 1, 1u);
      const uint64_t t0 = pw::global_ns();
      while (pw::ld_acquire_gpu(p.gather_ctr + 1) < gridDim.x) {
        if (pw::global_ns() - t0 > p.wait_ns) {
          report(p.status, PW_ERR_TIMEOUT);
          break;
        }
        __nanosleep(256);
      }
    }
    __syncthreads();
    combine_all(p, static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x,
                static_cast<long long>(gridDim.x) * kThreads);
  }
}

// Row-major fp16 [rows][cols] seen as a 2-D tensor with 64 x kN boxes in the
// 128-byte swizzle (one B atom per box).
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

int encode_rows(CUtensorMap* m, const void* base, long long cols, long long rows) {
  static EncodeTiled fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    PW_CUDA_TRY(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q));
    if (!f || q != cudaDriverEntryPointSuccess)
      return pw::set_error(PW_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    fn = reinterpret_cast<EncodeTiled>(f);
  }
  // (64 columns of an atom, row, atom): one box holds both atoms of a tile
  const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(cols / 64)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 2, 128};
  const cuuint32_t box[3] = {64, kN, 2};
  const cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, kGemv ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return pw::set_error(PW_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return PW_OK;
}

}  // namespace

int PW_LAUNCHER_NAME(const Params& p, cudaStream_t s, bool after_route) {
  // the shared-memory opt-in is a per-device attribute of the kernel
  constexpr int kDevs = 64;
  static bool attr_done[kDevs] = {};
  int dev = 0;
  PW_CUDA_TRY(cudaGetDevice(&dev));
  if (dev >= kDevs || !attr_done[dev]) {
    PW_CUDA_TRY(cudaFuncSetAttribute(PW_KERNEL_NAME, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes));
    if (dev < kDevs) attr_done[dev] = true;
  }
  const int sms = sm_count_cached();
  if (sms < 1) return pw::set_error(PW_ERR_CUDA, "could not query the SM count");
  CUtensorMap gu, dn;
  if (p.linear) {
    if (int e = encode_rows(&gu, p.x, p.lin.cols, p.M)) return e;
    dn = gu;
  } else {
    if (int e = encode_rows(&gu, p.xp, p.H, p.A)) return e;
    if (int e = encode_rows(&dn, p.h, p.I, p.A)) return e;
  }
  // one CTA per SM: it owns all 512 TMEM columns.  After a routing launch
  // the kernel may start while the routing grid finishes (programmatic
  // dependent launch; it waits for that grid before it reads anything).
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(sms));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = after_route ? 1 : 0;
  PW_CUDA_TRY(cudaLaunchKernelEx(&cfg, PW_KERNEL_NAME, p, gu, dn));
  return PW_OK;
}

}  // namespace pw_ffn
