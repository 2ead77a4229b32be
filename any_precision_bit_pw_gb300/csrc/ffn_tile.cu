// Fused MoE layer kernel with token tiles of up to 256 (prefill batches; also
// the any-precision linear export for M > 16).  G = 1 here.  See ffn_common.cuh for the
// work units and their scheduling.
//
// Inside a unit (warp roles), for each of G groups:
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
//   epilogue: the dequant warps read the accumulator rows from TMEM (with G = 2
//     group 1 hands its partial sums to group 0 through shared memory).
// Every mbarrier wait is bounded; a thread whose wait runs out reports
// PW_ERR_TIMEOUT, stops waiting for the rest of the unit (it still arrives
// where it must, so the other roles reach the end of the unit) and the CTA
// takes no further units.  TMEM is always released before the CTA exits.
#include "ffn_common.cuh"

namespace pw_ffn {
namespace {

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

// ---------------------------------------------------------------------------
// Dequant warps (group g: warps 4g..4g+3; pos = row position in the strip)
// ---------------------------------------------------------------------------
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

template <int NMAX, int G>
__global__ void __launch_bounds__(Cfg<NMAX, G>::kThreads, 1) apl_tc_kernel(const __grid_constant__ Params p) {
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
    if (threadIdx.x == 0) sh.u.combine = finish_unit(p, sh, u, u_skip);
    __syncthreads();
    if (sh.u.combine >= 0) combine_strip(p, sh.u.combine, threadIdx.x, blockDim.x);
  }
  pw::tc_fence_before();
  __syncthreads();
  pw::tc_fence_after();
  if (warp == 0) pw::tmem_dealloc(tmem, C::kTmemCols);
}

template <int NMAX, int G>
int launch_tile(const Params& p, cudaStream_t s) {
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

}  // namespace

int launch_tile_kernel(const Params& p, cudaStream_t s, int nmax) {
  (void)nmax;
  return launch_tile<256, 1>(p, s);
}

}  // namespace pw_ffn
