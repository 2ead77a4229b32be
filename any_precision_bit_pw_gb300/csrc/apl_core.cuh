// Device building blocks of the any-precision dequant + tensor-core path.
//
// "PagedWeight" arXiv text, §1 / Figure 3 caption: a b-bit weight is the LUT
// entry (bitwidth-specific centroid) selected by the index formed from the top
// b bit-planes.  Here one warp owns one 16-row strip of a block: each lane
// loads its 16 bytes of every committed plane of a 256-column tile, assembles
// the q-bit indices of exactly the elements of its m16n8k16 A-fragments,
// looks them up in the strip's LUT rows (shared memory), and feeds the fp16
// fragments straight into mma.sync with fp32 accumulation -- the weights are
// never written back to memory in fp16.
#pragma once

#include <cuda_fp16.h>

#include "pw_internal.h"

namespace pw {

constexpr int kNtMax = 8;          // n-tiles of 8 tokens per pass (64 tokens)
constexpr int kLutRowsPerWarp = 16;
constexpr int kLutMaxEntries = 1 << PW_MAX_BITS;

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint4 ld_stream_v4(const uint32_t* p) {
  uint4 v;
  asm volatile("ld.global.cs.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ld_nc_u32(const uint16_t* p) {
  return __ldg(reinterpret_cast<const unsigned int*>(p));
}

__device__ __forceinline__ uint32_t ld_cg_u32(const uint16_t* p) {
  return __ldcg(reinterpret_cast<const unsigned int*>(p));
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Copy LUT rows of one strip into shared memory: rows r0..r0+7 and
// r0+N/2..r0+N/2+7 of LUT_q (fp16 [N][2^q]) -> lut_s[16][2^q].
template <int Q>
__device__ __forceinline__ void load_strip_lut(const uint16_t* __restrict__ lut, int half_rows, int strip,
                                               uint16_t* __restrict__ lut_s) {
  constexpr int kEnt = 1 << Q;
  constexpr int kVecPerHalf = 8 * kEnt * 2 / 16;  // uint4 per 8 rows
  const uint4* src0 = reinterpret_cast<const uint4*>(lut + static_cast<long long>(strip) * 8 * kEnt);
  const uint4* src1 = reinterpret_cast<const uint4*>(lut + (static_cast<long long>(half_rows) + strip * 8) * kEnt);
  uint4* dst = reinterpret_cast<uint4*>(lut_s);
  for (int i = lane_id(); i < 2 * kVecPerHalf; i += 32)
    dst[i] = i < kVecPerHalf ? __ldg(src0 + i) : __ldg(src1 + (i - kVecPerHalf));
}

// q-bit indices of the 8 fragment elements of k-step s, packed as two nibble
// words (elements e at bits 4e..4e+3): lo = index bits 3..0, hi = bits 7..4.
template <int Q>
__device__ __forceinline__ void step_indices(const uint32_t (&words)[Q], int js, uint32_t& lo, uint32_t& hi) {
  lo = 0u;
  hi = 0u;
#pragma unroll
  for (int p = 0; p < Q; ++p) {
    const uint32_t xb = (words[p] >> js) & 0x11111111u;
    const int bitpos = Q - 1 - p;
    if (bitpos >= 4)
      hi |= xb << (bitpos - 4);
    else
      lo |= xb << bitpos;
  }
}

template <int Q>
__device__ __forceinline__ uint32_t elem_index(uint32_t lo, uint32_t hi, int e) {
  const uint32_t l = (lo >> (4 * e)) & 0xFu;
  if (Q <= 4) return l;
  return l | (((hi >> (4 * e)) & 0xFu) << 4);
}

// Dequantised A-fragment of k-step 4w+js from word w of each plane.
template <int Q>
__device__ __forceinline__ void step_fragment(const uint32_t (&words)[Q], int js, const uint16_t* __restrict__ lut_g,
                                              const uint16_t* __restrict__ lut_g8, uint32_t (&a)[4]) {
  uint32_t lo, hi;
  step_indices<Q>(words, js, lo, hi);
  const uint32_t v0 = lut_g[elem_index<Q>(lo, hi, 0)];
  const uint32_t v1 = lut_g[elem_index<Q>(lo, hi, 1)];
  const uint32_t v2 = lut_g[elem_index<Q>(lo, hi, 2)];
  const uint32_t v3 = lut_g[elem_index<Q>(lo, hi, 3)];
  const uint32_t v4 = lut_g8[elem_index<Q>(lo, hi, 4)];
  const uint32_t v5 = lut_g8[elem_index<Q>(lo, hi, 5)];
  const uint32_t v6 = lut_g8[elem_index<Q>(lo, hi, 6)];
  const uint32_t v7 = lut_g8[elem_index<Q>(lo, hi, 7)];
  a[0] = v0 | (v1 << 16);  // row g,   cols 2c, 2c+1
  a[1] = v4 | (v5 << 16);  // row g+8, cols 2c, 2c+1
  a[2] = v2 | (v3 << 16);  // row g,   cols 2c+8, 2c+9
  a[3] = v6 | (v7 << 16);  // row g+8, cols 2c+8, 2c+9
}

// Per-warp shared-memory budget of the plane-staging ring.
constexpr int kRingBytesPerWarp = 8192;

// Pipeline depth (tiles) for bitwidth Q: as many 512-byte-per-plane tiles as
// fit in the ring, at most 4.
template <int Q>
struct RingDepth {
  static constexpr int value = (kRingBytesPerWarp / (Q * kTileBytes)) > 4 ? 4 : (kRingBytesPerWarp / (Q * kTileBytes));
};

__device__ __forceinline__ void cp_async_16(uint32_t smem_addr, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint32_t lds_u32(uint32_t smem_addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(smem_addr));
  return v;
}

// Main loop of one warp unit: strip `strip` of a block (tiles [t0, t1)),
// B operand = nt_count n-tiles whose row g (this lane's token) starts at
// element offset brow[nt] of `bbase`.  Each lane streams its own 16 bytes of
// every plane of the next tiles into its private slots of the warp's ring
// (cp.async, L2 only) while it works on the current tile, so no cross-lane
// synchronisation is needed.  kFromH: the B rows were written earlier in the
// same launch -> L2-only loads.
template <int Q, bool kFromH>
__device__ __forceinline__ void strip_mainloop(const BlockDesc& d, int strip, int t0, int t1,
                                               const uint16_t* __restrict__ lut_s, uint32_t ring_s,
                                               const uint16_t* __restrict__ bbase, const int (&brow)[kNtMax],
                                               int nt_count, float (&acc)[kNtMax][4]) {
  constexpr int D = RingDepth<Q>::value;
  constexpr int kStageBytes = Q * kTileBytes;
  const int lane = static_cast<int>(lane_id());
  const int g = lane >> 2, c = lane & 3;
  const uint16_t* lut_g = lut_s + g * (1 << Q);
  const uint16_t* lut_g8 = lut_s + (g + 8) * (1 << Q);
  const int tiles_per_strip = d.cols / kTileCols;
  const long long strip_word0 = static_cast<long long>(strip) * tiles_per_strip * (kTileBytes / 4) + lane * 4;
  const uint32_t* planes[Q];
#pragma unroll
  for (int p = 0; p < Q; ++p) planes[p] = d.planes[p] + strip_word0;
  const uint32_t my_slot = ring_s + lane * 16;

  auto issue = [&](int t, int stage) {
    if (t < t1) {
#pragma unroll
      for (int p = 0; p < Q; ++p)
        cp_async_16(my_slot + stage * kStageBytes + p * kTileBytes, planes[p] + static_cast<long long>(t) * (kTileBytes / 4));
    }
    cp_async_commit();
  };
#pragma unroll
  for (int i = 0; i < D - 1; ++i) issue(t0 + i, i);

  int stage = 0;
  for (int t = t0; t < t1; ++t) {
    issue(t + D - 1, (stage + D - 1) % D);
    cp_async_wait<D - 1>();
    const uint32_t base = my_slot + stage * kStageBytes;
    const int col_tile = t * kTileCols + 2 * c;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      uint32_t words[Q];
#pragma unroll
      for (int p = 0; p < Q; ++p) words[p] = lds_u32(base + p * kTileBytes + 4 * w);
#pragma unroll
      for (int js = 0; js < 4; ++js) {
        uint32_t a[4];
        step_fragment<Q>(words, js, lut_g, lut_g8, a);
        const int col = col_tile + 16 * (4 * w + js);
#pragma unroll
        for (int nt = 0; nt < kNtMax; ++nt) {
          if (nt < nt_count) {
            const uint16_t* bp = bbase + brow[nt] + col;
            const uint32_t b0 = kFromH ? ld_cg_u32(bp) : ld_nc_u32(bp);
            const uint32_t b1 = kFromH ? ld_cg_u32(bp + 8) : ld_nc_u32(bp + 8);
            mma_16816(acc[nt], a, b0, b1);
          }
        }
      }
    }
    stage = (stage + 1 == D) ? 0 : stage + 1;
  }
  cp_async_wait<0>();
}

}  // namespace pw
