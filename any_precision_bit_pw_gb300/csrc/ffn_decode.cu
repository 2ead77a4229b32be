// Fused MoE layer kernel for decode batches: token tiles of up to 16 and one
// 128-column tile per pipeline stage.  See ffn_common.cuh for the work units
// and their scheduling.
//
// Each CTA (one per SM) runs two groups on the same 128-row strip of a unit,
// splitting its K range; both share the strip's LUT.  In a group:
//   4 dequant warps (thread = one row = one TMEM lane): per tile, each thread
//     copies its 16-byte slice of every committed plane plus its share of the
//     B operand (the tokens' x or h columns of the tile, two 16-byte chunks of
//     a 128-byte-swizzled layout) into shared rings with cp.async, several
//     tiles ahead; dequantises the tile's 128 columns of its row (dequant.cuh)
//     and stores them as operand A into a 3-slot TMEM ring (tcgen05.st); then
//     arrives on the tile's "full" barrier.
//   1 MMA warp (lane 0): per tile, waits for "full", issues the tile's 8
//     tcgen05.mma (A from TMEM, B from shared memory, fp32 accumulator in TMEM)
//     and one tcgen05.commit to the tile's "free" barrier, which releases the
//     tile's A slot and B slot together.
// The epilogue reads the accumulator rows from TMEM; group 1 hands its partial
// sums to group 0 through shared memory.  All mbarrier waits are bounded
// (PW_ERR_TIMEOUT); TMEM is released before the CTA exits.
#include "ffn_common.cuh"

namespace pw_ffn {
namespace {

constexpr int kN = 16;                          // tokens per tile
constexpr int kG = 2;                           // dequant groups (split K)
constexpr int kThreads = kG * (kDeqThreads + 32);
constexpr int kSA = 3;                          // TMEM A slots per group (tiles)
constexpr int kATileCols = 64;                  // TMEM columns per A tile (128 fp16 per row)
constexpr int kDColT = kSA * kATileCols;        // accumulator columns start here
constexpr int kGroupCols = 256;
constexpr int kTmemColsT = kG * kGroupCols;
constexpr int kF = 8;                           // completion barriers per group (tile index mod 8)
constexpr int kBSlots = 5;                      // B slots per group
constexpr int kBAtomBytes = kN * 128;           // 16 rows x 64 columns fp16, 128-byte swizzle
constexpr int kBSlotBytes = 2 * kBAtomBytes;    // 128 columns
constexpr int kPlaneRing = 32768;               // per group
constexpr int kBRingBytes = kG * kBSlots * kBSlotBytes;
constexpr int kXBytes = kN * kDeqThreads * 4;
constexpr int kBarBytes = kG * 32 * 8;
constexpr int kRowsBytes = kN * 4;
constexpr int kPreBytes = kBRingBytes + kXBytes + kBarBytes + kRowsBytes + 8192;
constexpr int kSmemBytes = 65536 + pw::kLutRegionBytes + kG * kPlaneRing;
static_assert(kDColT + kN <= kGroupCols, "TMEM columns per group");
static_assert(kPreBytes <= 65536 - 4096, "front part must fit below the first 64 KB boundary");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(2 * kF + 1 <= 32, "barrier slots");

struct SmemT {
  uint8_t* b_ring;      // kG x kBSlots x kBSlotBytes
  uint8_t* plane_ring;  // kG x kPlaneRing
  float* xch;           // group-1 partial sums [token][pos]
  uint32_t bar;         // per group: full[kF], free[kF], done
  int* rows;            // B row offsets of the unit's tokens
  uint32_t lut_region;
};

__device__ __forceinline__ uint32_t bar_full(uint32_t g0, int i) { return g0 + 8 * i; }
__device__ __forceinline__ uint32_t bar_free(uint32_t g0, int i) { return g0 + 8 * (kF + i); }
__device__ __forceinline__ uint32_t bar_done(uint32_t g0) { return g0 + 8 * (2 * kF); }

// Wait until the MMAs of this group's tile x have completed.
__device__ __forceinline__ void wait_tile_free(uint32_t g0, uint32_t x, const Params& p, int& abort) {
  if (!abort && !pw::mbar_wait(bar_free(g0, x % kF), (x / kF) & 1u, p.wait_ns)) abort = 1;
}

template <int Q>
__device__ __noinline__ void dequant_role(const Params& p, const Unit& u, const SmemT& sm, uint32_t tmem,
                                          uint32_t& tcnt, uint32_t unit_cnt, int& abort) {
  constexpr int kTileStrideW = pw::kTileBytes / 4;
  constexpr int kSlotBytes = Q * pw::kTileBytes;
  constexpr int D = (kPlaneRing / kSlotBytes) > 4 ? 4 : (kPlaneRing / kSlotBytes);
  static_assert(D >= 2 && D + 1 <= kBSlots, "ring depths");
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
    dequant_bar_sync(kG);   // both halves of every row's table are in place
  }

  // this group's share of the unit's 128-column tiles
  const int tiles = d.cols / pw::kTileCols;
  const int ntiles_all = u.nst / 2;
  const int half = (ntiles_all + 1) / 2;
  const int tb = g == 1 ? half : 0;
  const int te = g == 0 ? half : ntiles_all;
  const int ntiles = te - tb;
  const int tile0 = u.st0 / 2 + tb;
  const uint32_t* src[Q];
#pragma unroll
  for (int q = 0; q < Q; ++q)
    src[q] = d.planes[q] + (static_cast<long long>(u.strip) * tiles + tile0) * kTileStrideW + pos * 4;
  const uint32_t ring = pw::smem_u32(sm.plane_ring + g * kPlaneRing) + pos * 16;
  const uint32_t bring = pw::smem_u32(sm.b_ring + g * kBSlots * kBSlotBytes);
  const uint32_t g0 = sm.bar + g * 32 * 8;
  const uint16_t* bbase = u.kind == kDown ? p.h : p.x;
  // this thread's B chunks: i = pos + 128 m (m < npad / 8); row n = i / 16, chunk c = i % 16
  const int nchunk = u.npad / 8;
  auto issue = [&](int t) {
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
                        bbase + sm.rows[n] + col + c * 8);
      }
    }
    pw::cp_async_commit();
  };
#pragma unroll
  for (int i = 0; i < D - 1; ++i) issue(i);

  const uint32_t tl = tmem + g * kGroupCols + (static_cast<uint32_t>(32 * wq) << 16);
  for (int t = 0; t < ntiles; ++t) {
    issue(t + D - 1);
    pw::cp_async_wait<D - 1>();
    pw::fence_proxy_async_smem();   // this thread's B chunks of tile t, for the tensor core
    const uint32_t slot = ring + (t % D) * kSlotBytes;
    uint32_t w4[Q][4];
#pragma unroll
    for (int q = 0; q < Q; ++q) lds_v4(slot + q * pw::kTileBytes, w4[q]);
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
  tcnt += ntiles;
  pw::cp_async_wait<0>();

  // epilogue: accumulator row `pos` (TMEM lane), columns = tokens
  if (!abort && !pw::mbar_wait(bar_done(g0), unit_cnt & 1u, p.wait_ns)) abort = 1;
  pw::tc_fence_after();
  float* xch = sm.xch;
  if (g == 1) {
    uint32_t v[16];
    if (ntiles > 0) {
      pw::tmem_ld_x16(tl + kDColT, v);
      pw::tmem_ld_wait();
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) xch[i * kDeqThreads + pos] = ntiles > 0 ? __uint_as_float(v[i]) : 0.f;
    pw::tc_fence_before();
    dequant_bar_sync(kG);
    return;
  }
  uint32_t v[16];
  pw::tmem_ld_x16(tl + kDColT, v);
  pw::tmem_ld_wait();
  pw::tc_fence_before();
  dequant_bar_sync(kG);
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

__device__ void mma_role(const Unit& u, const SmemT& sm, uint32_t tmem, uint32_t& tcnt, const Params& p,
                         int& abort) {
  const int g = (threadIdx.x >> 5) - 4 * kG;
  const int ntiles_all = u.nst / 2;
  const int half = (ntiles_all + 1) / 2;
  const int ntiles = g == 0 ? half : ntiles_all - half;
  const uint32_t g0 = sm.bar + g * 32 * 8;
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

__global__ void __launch_bounds__(kThreads, 1) apl_decode_kernel(Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t base = pw::smem_u32(smem_raw);
  const uint32_t pre = (base + 1023u) & ~1023u;
  const uint32_t region = (pre + static_cast<uint32_t>(kPreBytes) + 0xFFFFu) & ~0xFFFFu;
  const uint32_t post = region + static_cast<uint32_t>(pw::kLutRegionBytes);
  if (post + static_cast<uint32_t>(kG * kPlaneRing) > base + static_cast<uint32_t>(kSmemBytes)) {
    if (threadIdx.x == 0) report(p.status, PW_ERR_UNSUPPORTED);   // unexpected shared-window base
    return;
  }
  auto at = [&](uint32_t addr) { return smem_raw + (addr - base); };
  SmemT sm;
  uint32_t cur = pre;
  sm.b_ring = at(cur);
  cur += kBRingBytes;
  sm.xch = reinterpret_cast<float*>(at(cur));
  cur += kXBytes;
  sm.bar = cur;
  cur += kBarBytes;
  sm.rows = reinterpret_cast<int*>(at(cur));
  cur += kRowsBytes;
  Shared& sh = *reinterpret_cast<Shared*>(at((cur + 15u) & ~15u));
  sm.lut_region = region;
  sm.plane_ring = at(post);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int g = 0; g < kG; ++g) {
      const uint32_t g0 = sm.bar + g * 32 * 8;
      for (int i = 0; i < kF; ++i) {
        pw::mbar_init(bar_full(g0, i), kDeqWarps);
        pw::mbar_init(bar_free(g0, i), 1);
      }
      pw::mbar_init(bar_done(g0), 1);
    }
    pw::mbar_init_fence();
    sh.abort = 0;
    setup_schedule<kN>(p, sh);
  }
  if (warp == 0) {
    pw::tmem_alloc(pw::smem_u32(&sh.tmem), kTmemColsT);
    pw::tmem_relinquish();
  }
  pw::tc_fence_before();
  __syncthreads();
  pw::tc_fence_after();
  const uint32_t tmem = sh.tmem;

  uint32_t tcnt = 0, unit_cnt = 0;
  int abort_local = 0;
  for (;;) {
    if (warp == 0) {
      if (lane == 0) next_unit<kN>(p, sh);
      __syncwarp();
      const Unit& nu = sh.u;
      if (lane < kN && nu.kind != kNone && !nu.skip) {
        const int nn = min(lane, nu.nrows - 1);
        int r;
        if (nu.kind == kGateUp)
          r = (__ldg(p.perm + nu.off + nn) / p.k) * p.H;
        else if (nu.kind == kDown)
          r = (nu.off + nn) * p.I;
        else
          r = (nu.tg * kN + nn) * nu.d->cols;
        sm.rows[lane] = r;
      }
    }
    pw::tc_fence_before();
    __syncthreads();
    pw::tc_fence_after();
    const Unit& u = sh.u;
    if (u.kind == kNone) break;
    const int u_skip = u.skip;
    if (!u_skip) {
      if (warp < kDeqWarps * kG) {
        switch (u.q) {
          case 2: dequant_role<2>(p, u, sm, tmem, tcnt, unit_cnt, abort_local); break;
          case 3: dequant_role<3>(p, u, sm, tmem, tcnt, unit_cnt, abort_local); break;
          case 4: dequant_role<4>(p, u, sm, tmem, tcnt, unit_cnt, abort_local); break;
          case 5: dequant_role<5>(p, u, sm, tmem, tcnt, unit_cnt, abort_local); break;
          case 6: dequant_role<6>(p, u, sm, tmem, tcnt, unit_cnt, abort_local); break;
          case 7: dequant_role<7>(p, u, sm, tmem, tcnt, unit_cnt, abort_local); break;
          default: dequant_role<8>(p, u, sm, tmem, tcnt, unit_cnt, abort_local); break;
        }
      } else {
        mma_role(u, sm, tmem, tcnt, p, abort_local);
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
    if (sh.u.combine >= 0) combine_strip(p, sh.u.combine);
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
