// Per-row any-precision dequantisation for the tcgen05 path.
//
// "PagedWeight" arXiv text, §1 / Figure 3 caption: a b-bit weight is the entry
// of its row's bitwidth-specific LUT selected by the index formed from the top
// b bit-planes.  Here each thread of the four dequant warps owns one output
// row (one TMEM lane) of a 128-row strip and turns 64 consecutive columns per
// pipeline stage into 32 fp16 pairs for tcgen05.st:
//
//  * plane words use the "nibble" bit order of the tiled layout: within a
//    32-column word, column 8*js + e sits at bit 4*e + js, so one shift and
//    mask per plane yields the indices of 8 consecutive columns as nibbles;
//  * q <= 4: the LUT lives in registers as a low-byte and a high-byte table
//    and one prmt looks up four 8-bit halves at once (q = 4 selects between
//    two 8-entry halves with a byte mask built from the index MSB);
//  * q >= 5: an 8x8 bit transpose of the plane words yields byte indices;
//    the LUT lives in a 64 KB-aligned shared region with one bank per lane,
//    so one prmt forms each lookup address and lookups never conflict.
#pragma once

#include "tc_ptx.cuh"

namespace pw {

constexpr int kStageK = 64;                      // columns per pipeline stage

// Two zero-extended 16-bit values into one 32-bit pair (lo | hi << 16) as an
// integer multiply-add, which issues on the multiply-add pipe rather than the
// logic pipe that carries the masks and byte permutes.
__device__ __forceinline__ uint32_t pack_mad(uint32_t lo, uint32_t hi) {
  uint32_t r;
  asm("mad.lo.u32 %0, %1, 65536, %2;" : "=r"(r) : "r"(hi), "r"(lo));
  return r;
}

// Shifts by a count known after unrolling (0 allowed).
__device__ __forceinline__ uint32_t shl_mul(uint32_t x, int s) {
  return x << s;
}
__device__ __forceinline__ uint32_t shr_mul(uint32_t x, int s) {
  return x >> s;
}
constexpr int kLutRegionBytes = 65536;           // shared LUT region of a strip (q >= 5), 64 KB aligned

// Nibble selector of 8 consecutive columns (sub-block js) from one word per
// plane, using planes [P0, P1) as index bits (P1-1-p) .. 0.
template <int P0, int P1>
__device__ __forceinline__ uint32_t nibble_sel(const uint32_t* w, int js) {
  uint32_t s = 0u;
#pragma unroll
  for (int p = P0; p < P1; ++p) {
    const int k = P1 - 1 - p, sh = js - k;   // bit js of each nibble -> bit k
    const uint32_t t = sh >= 0 ? shr_mul(w[p], sh) : shl_mul(w[p], -sh);
    s |= t & (0x11111111u << k);
  }
  return s;
}

template <int Q, bool kInRegs = (Q <= 4)>
struct RowDequant;

// ---------------------------------------------------------------- q <= 4
template <int Q>
struct RowDequant<Q, true> {
  static constexpr int kT = (Q == 4) ? 4 : 2;
  uint32_t lo[kT], hi[kT];

  __device__ __forceinline__ void load(const uint16_t* __restrict__ lut_row, uint32_t, int) {
    if (Q == 2) {
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(lut_row));
      lo[0] = lo[1] = prmt(v.x, v.y, 0x6420u);
      hi[0] = hi[1] = prmt(v.x, v.y, 0x7531u);
    } else if (Q == 3) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(lut_row));
      lo[0] = prmt(v.x, v.y, 0x6420u);
      lo[1] = prmt(v.z, v.w, 0x6420u);
      hi[0] = prmt(v.x, v.y, 0x7531u);
      hi[1] = prmt(v.z, v.w, 0x7531u);
    } else {
      const uint4 v0 = __ldg(reinterpret_cast<const uint4*>(lut_row));
      const uint4 v1 = __ldg(reinterpret_cast<const uint4*>(lut_row) + 1);
      lo[0] = prmt(v0.x, v0.y, 0x6420u);
      lo[1] = prmt(v0.z, v0.w, 0x6420u);
      hi[0] = prmt(v0.x, v0.y, 0x7531u);
      hi[1] = prmt(v0.z, v0.w, 0x7531u);
      if (kT == 4) {
        lo[kT - 2] = prmt(v1.x, v1.y, 0x6420u);
        lo[kT - 1] = prmt(v1.z, v1.w, 0x6420u);
        hi[kT - 2] = prmt(v1.x, v1.y, 0x7531u);
        hi[kT - 1] = prmt(v1.z, v1.w, 0x7531u);
      }
    }
  }

  // The same tables from this row's LUT in shared memory (2^Q fp16 at `saddr`).
  __device__ __forceinline__ void load_shared(uint32_t saddr) {
    if (Q == 2) {
      uint32_t a, b;
      lds_v2(saddr, a, b);
      lo[0] = lo[1] = prmt(a, b, 0x6420u);
      hi[0] = hi[1] = prmt(a, b, 0x7531u);
    } else {
      uint32_t v[4];
      lds_v4u(saddr, v);
      lo[0] = prmt(v[0], v[1], 0x6420u);
      lo[1] = prmt(v[2], v[3], 0x6420u);
      hi[0] = prmt(v[0], v[1], 0x7531u);
      hi[1] = prmt(v[2], v[3], 0x7531u);
      if (kT == 4) {
        lds_v4u(saddr + 16, v);
        lo[kT - 2] = prmt(v[0], v[1], 0x6420u);
        lo[kT - 1] = prmt(v[2], v[3], 0x6420u);
        hi[kT - 2] = prmt(v[0], v[1], 0x7531u);
        hi[kT - 1] = prmt(v[2], v[3], 0x7531u);
      }
    }
  }

  // Four columns whose indices are the nibbles of s[15:0] -> two fp16 pairs.
  __device__ __forceinline__ void quad(uint32_t s, uint32_t& p01, uint32_t& p23) const {
    uint32_t l, h;
    if (Q <= 3) {
      l = prmt(lo[0], lo[1], s);
      h = prmt(hi[0], hi[1], s);
    } else {
      // entries 0..7 from the first half, 8..15 from the second; byte k of m
      // is 0xFF when nibble k >= 8 (sign-replicated index MSB)
      const uint32_t sx = s ^ 0x8888u;
      const uint32_t m = prmt(s << 4, s, 0xD9C8u);
      const uint32_t l0 = prmt(lo[0], lo[1], s), l1 = prmt(lo[kT - 2], lo[kT - 1], sx);
      const uint32_t h0 = prmt(hi[0], hi[1], s), h1 = prmt(hi[kT - 2], hi[kT - 1], sx);
      l = (l1 & m) | (l0 & ~m);
      h = (h1 & m) | (h0 & ~m);
    }
    p01 = prmt(l, h, 0x5140u);
    p23 = prmt(l, h, 0x7362u);
  }

  // ww[p]: one 32-column word of plane p -> 16 fp16 pairs (columns in order).
  __device__ __forceinline__ void word(const uint32_t (&ww)[Q], uint32_t (&out)[16]) const {
#pragma unroll
    for (int js = 0; js < 4; ++js) {
      const uint32_t s = nibble_sel<0, Q>(ww, js);
      quad(s, out[4 * js], out[4 * js + 1]);
      quad(s >> 16, out[4 * js + 2], out[4 * js + 3]);
    }
  }
};

// ---------------------------------------------------------------- q >= 5
// 8x8 bit-matrix transpose of the bytes of eight words (three rounds of delta
// swaps, all four byte lanes at once): afterwards bit c of byte j of X[i]
// holds what was bit i of byte j of X[c].
__device__ __forceinline__ void transpose8x8(uint32_t (&X)[8]) {
  // each exchange: the low part of a keeps its own bits and takes b's low
  // part shifted up; b keeps its high part and takes a's high part shifted
  // down (one shift and one three-input logic op per result)
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t a = X[i], b = X[i + 4];
    X[i] = (a & 0x0F0F0F0Fu) | (shl_mul(b, 4) & 0xF0F0F0F0u);
    X[i + 4] = (shr_mul(a, 4) & 0x0F0F0F0Fu) | (b & 0xF0F0F0F0u);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (i & 2) continue;
    const uint32_t a = X[i], b = X[i + 2];
    X[i] = (a & 0x33333333u) | (shl_mul(b, 2) & 0xCCCCCCCCu);
    X[i + 2] = (shr_mul(a, 2) & 0x33333333u) | (b & 0xCCCCCCCCu);
  }
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    const uint32_t a = X[i], b = X[i + 1];
    X[i] = (a & 0x55555555u) | (shl_mul(b, 1) & 0xAAAAAAAAu);
    X[i + 1] = (shr_mul(a, 1) & 0x55555555u) | (b & 0xAAAAAAAAu);
  }
}

// The LUTs of a 128-row strip live in one shared region aligned to 64 KB:
// entry c of every row is the 256-byte line c of the region; within a line,
// rows of warps 0/1 of the group use the low half-words and rows of warps 2/3
// the high half-words of words (warp & 1) * 32 + lane.  Every lane of a warp
// owns its own bank, so lookups never conflict, and the shared address of a
// lookup is the region base with the index byte dropped into byte 1 -- one
// prmt per column.
template <int Q>
struct RowDequant<Q, false> {
  uint32_t tblw;      // region | this row's offset within a line
  uint32_t hi7 = 0u;  // index bit 7 forced to 1: the table in lines 128..255 (Q < 8)

  __device__ __forceinline__ void set_row(uint32_t region, int wq, int lane) {
    tblw = region | (static_cast<uint32_t>((wq & 1) * 32 + lane) * 4u + static_cast<uint32_t>(wq >> 1) * 2u);
  }
  // Same, for a table written to half `half` of the region (Q < 8: lines
  // 128*half + c; Q = 8 uses the whole region).
  __device__ __forceinline__ void set_row(uint32_t region, int wq, int lane, int half) {
    set_row(region, wq, lane);
    hi7 = (Q < 8 && half) ? 0xFFFFFFFFu : 0u;
  }

  // Write part `part` of `nparts` of this row's LUT (2^Q fp16) into its
  // column of the region; all loads of the part are issued before any store.
  template <int kParts = 1>
  __device__ __forceinline__ void load(const uint16_t* __restrict__ lut_row, int part = 0) const {
    constexpr int kVec = (1 << Q) / 8 / kParts;    // uint4 (8 entries) per part
    const uint4* src = reinterpret_cast<const uint4*>(lut_row) + part * kVec;
    uint4 a[kVec];
#pragma unroll
    for (int c8 = 0; c8 < kVec; ++c8) a[c8] = __ldg(src + c8);
#pragma unroll
    for (int c8 = 0; c8 < kVec; ++c8) {
      const uint32_t av[4] = {a[c8].x, a[c8].y, a[c8].z, a[c8].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t c = static_cast<uint32_t>((part * kVec + c8) * 8 + 2 * i);
        sts_u16(tblw + c * 256u, av[i] & 0xFFFFu);
        sts_u16(tblw + (c + 1u) * 256u, av[i] >> 16);
      }
    }
  }

  // Copy this row's LUT from a row-major copy in shared memory (2^Q fp16 at
  // `srow`) into its column of the region.  kSets threads share the row; the
  // thread of set `set` writes 8-entry chunks set, set + kSets, ...  rotated by
  // the lane so that the lanes of a warp read different bank groups.
  template <int kSets>
  __device__ __forceinline__ void fill(uint32_t srow, int set, int lane) const {
    constexpr int kCh = (1 << Q) / 8;
    static_assert(kCh % kSets == 0, "chunks per set");
    constexpr int kPer = kCh / kSets;
    uint32_t v[kPer][4];
    int ch[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      ch[j] = (set + kSets * j + lane) & (kCh - 1);
      lds_v4u(srow + ch[j] * 16, v[j]);
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t c = static_cast<uint32_t>(ch[j] * 8 + 2 * i);
        sts_u16(tblw + c * 256u, v[j][i] & 0xFFFFu);
        sts_u16(tblw + (c + 1u) * 256u, v[j][i] >> 16);
      }
    }
  }

  // ww[p]: one 32-column word of plane p -> 16 fp16 pairs (columns in order).
  __device__ __forceinline__ void word(const uint32_t (&ww)[Q], uint32_t (&out)[16]) const {
    // row i of the bit matrix = index bit i = plane Q-1-i; missing bits are 0
    uint32_t X[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) X[i] = i < Q ? ww[Q - 1 - i] : (i == 7 ? hi7 : 0u);
    transpose8x8(X);
    // column 8*js + e now has its full index in byte e/2 of X[4*(e%2) + js]
#pragma unroll
    for (int js = 0; js < 4; ++js) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t sel = 0x7604u | (static_cast<uint32_t>(j) << 4);
        const uint32_t v0 = lds_u16(prmt(X[js], tblw, sel));
        const uint32_t v1 = lds_u16(prmt(X[4 + js], tblw, sel));
        out[4 * js + j] = pack_mad(v0, v1);
      }
    }
  }
};

// Write one row's LUT (2^Q fp16 at `lut_row`, global) into its column of the
// region: entry c at line c + 128*half (Q < 8) or line c (Q = 8).  `tblw` is
// the row's set_row() address.  Loads go out in batches of up to 8 x 16 bytes.
template <int Q>
__device__ __forceinline__ void region_fill(uint32_t tblw, const uint16_t* __restrict__ lut_row, int half) {
  constexpr int kCh = (1 << Q) / 8;
  constexpr int kB = kCh < 8 ? kCh : 8;
  const uint32_t base = tblw + ((Q < 8 && half) ? 128u * 256u : 0u);
  const uint4* src = reinterpret_cast<const uint4*>(lut_row);
#pragma unroll
  for (int c0 = 0; c0 < kCh; c0 += kB) {
    uint4 a[kB];
#pragma unroll
    for (int j = 0; j < kB; ++j) a[j] = __ldg(src + c0 + j);
#pragma unroll
    for (int j = 0; j < kB; ++j) {
      const uint32_t av[4] = {a[j].x, a[j].y, a[j].z, a[j].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t c = static_cast<uint32_t>((c0 + j) * 8 + 2 * i);
        sts_u16(base + c * 256u, av[i] & 0xFFFFu);
        sts_u16(base + (c + 1u) * 256u, av[i] >> 16);
      }
    }
  }
}

}  // namespace pw
