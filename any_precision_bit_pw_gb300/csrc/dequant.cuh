// Per-row any-precision dequantisation for the tcgen05 path.
//
// "PagedWeight" arXiv text, §1 / Figure 3 caption: a b-bit weight is the entry
// of its row's LUT for bitwidth b at the index formed from the top b
// bit-planes.  Here each thread of the four dequant warps owns one output
// row (one TMEM lane) of a 128-row strip and turns 64 consecutive columns per
// pipeline stage into 32 fp16 pairs for tcgen05.st:
//
//  * plane words use the "nibble" bit order of the tiled layout: within a
//    32-column word, column 8*js + e sits at bit 4*e + js, so one shift and
//    mask per plane yields the indices of 8 consecutive columns as nibbles;
//  * every unit's LUT arrives in a 64 KB-aligned shared region by one bulk
//    copy of its strip's table (LUT pages are stored in that order, see
//    pw_pack_lut): entry c of a row is on the 256-byte line c, at the row's
//    own bank;
//  * q <= 3 (4 for the register form): the thread reads its row's entries
//    into registers as a low-byte and a high-byte table, and one prmt looks
//    up four 8-bit halves at once (q = 4 selects between two 8-entry halves
//    with a byte mask built from the index MSB);
//  * q >= 4 in the kernels: a bit transpose of the plane words yields byte
//    indices (an 8x8 transpose for q >= 6; for q <= 5 a 4x4 transpose inside
//    nibbles for the low four index bits, the rest merged per nibble, which
//    takes 28 logic ops per 32 columns at q = 4 instead of 44), one prmt forms
//    each lookup address in the region, and lookups never conflict.
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

// 4x4 bit-matrix transpose inside every nibble of four words (two rounds of
// delta swaps): afterwards bit c of nibble n of L[i] holds what was bit i of
// nibble n of L[c].
__device__ __forceinline__ void transpose4x4(uint32_t (&L)[4]) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint32_t a = L[i], b = L[i + 2];
    L[i] = (a & 0x33333333u) | (shl_mul(b, 2) & 0xCCCCCCCCu);
    L[i + 2] = (shr_mul(a, 2) & 0x33333333u) | (b & 0xCCCCCCCCu);
  }
#pragma unroll
  for (int i = 0; i < 4; i += 2) {
    const uint32_t a = L[i], b = L[i + 1];
    L[i] = (a & 0x55555555u) | (shl_mul(b, 1) & 0xAAAAAAAAu);
    L[i + 1] = (shr_mul(a, 1) & 0x55555555u) | (b & 0xAAAAAAAAu);
  }
}

template <int Q, bool kInRegs = (Q <= 4)>
struct RowDequant;

// ---------------------------------------------------------------- q <= 4
template <int Q>
struct RowDequant<Q, true> {
  static constexpr int kT = (Q == 4) ? 4 : 2;
  uint32_t lo[kT], hi[kT];

  // The same tables from this row's LUT in the shared LUT region (the tiled
  // LUT order: entry c at `base + c*256`, base = the region half plus this
  // row's byte within a line).
  __device__ __forceinline__ void load_region(uint32_t base) {
    constexpr int kE = 1 << Q;
    uint32_t v[kE / 2];
#pragma unroll
    for (int j = 0; j < kE / 2; ++j)
      v[j] = lds_u16_ordered(base + (2 * j) * 256u) | (lds_u16_ordered(base + (2 * j + 1) * 256u) << 16);
    if (Q == 2) {
      lo[0] = lo[1] = prmt(v[0], v[1], 0x6420u);
      hi[0] = hi[1] = prmt(v[0], v[1], 0x7531u);
    } else {
      lo[0] = prmt(v[0], v[1], 0x6420u);
      lo[1] = prmt(v[2], v[3], 0x6420u);
      hi[0] = prmt(v[0], v[1], 0x7531u);
      hi[1] = prmt(v[2], v[3], 0x7531u);
      if (kT == 4) {
        lo[kT - 2] = prmt(v[4 % (kE / 2)], v[5 % (kE / 2)], 0x6420u);
        lo[kT - 1] = prmt(v[6 % (kE / 2)], v[7 % (kE / 2)], 0x6420u);
        hi[kT - 2] = prmt(v[4 % (kE / 2)], v[5 % (kE / 2)], 0x7531u);
        hi[kT - 1] = prmt(v[6 % (kE / 2)], v[7 % (kE / 2)], 0x7531u);
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
    if constexpr (Q == 3) {
      // the selectors of all four sub-blocks at once: after a 4x4 transpose
      // inside nibbles, nibble e of L[js] is the index of column 8*js + e
      // (bit 3 zero: prmt's plain byte mode)
      uint32_t L[4] = {ww[2], ww[1], ww[0], 0u};
      transpose4x4(L);
#pragma unroll
      for (int js = 0; js < 4; ++js) {
        quad(L[js], out[4 * js], out[4 * js + 1]);
        quad(L[js] >> 16, out[4 * js + 2], out[4 * js + 3]);
      }
    } else {
#pragma unroll
      for (int js = 0; js < 4; ++js) {
        const uint32_t s = nibble_sel<0, Q>(ww, js);
        quad(s, out[4 * js], out[4 * js + 1]);
        quad(s >> 16, out[4 * js + 2], out[4 * js + 3]);
      }
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

  // ww[p]: one 32-column word of plane p -> 16 fp16 pairs (columns in order).
  __device__ __forceinline__ void word(const uint32_t (&ww)[Q], uint32_t (&out)[16]) const {
    uint32_t X[8];
    if constexpr (Q <= 5) {
      // index bits 0-3 (planes Q-1 .. Q-4): after a 4x4 transpose inside every
      // nibble, nibble e of L[js] holds them for column 8*js + e
      uint32_t L[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) L[c] = c < Q ? ww[Q - 1 - c] : 0u;
      transpose4x4(L);
      // index bits 4-7 as a nibble per column: plane 0 in bit 0 (Q = 5) and
      // the region half in bit 3; spread the two nibbles into index bytes
      const uint32_t h = hi7 & (Q <= 4 ? 0x80808080u : 0x88888888u);
#pragma unroll
      for (int js = 0; js < 4; ++js) {
        if constexpr (Q <= 4) {
          X[js] = (L[js] & 0x0F0F0F0Fu) | h;
          X[4 + js] = (shr_mul(L[js], 4) & 0x0F0F0F0Fu) | h;
        } else {
          const uint32_t H = (shr_mul(ww[0], js) & 0x11111111u) | h;
          X[js] = (L[js] & 0x0F0F0F0Fu) | (shl_mul(H, 4) & 0xF0F0F0F0u);
          X[4 + js] = (shr_mul(L[js], 4) & 0x0F0F0F0Fu) | (H & 0xF0F0F0F0u);
        }
      }
    } else {
      // row i of the bit matrix = index bit i = plane Q-1-i; missing bits are 0
#pragma unroll
      for (int i = 0; i < 8; ++i) X[i] = i < Q ? ww[Q - 1 - i] : (i == 7 ? hi7 : 0u);
      transpose8x8(X);
    }
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

}  // namespace pw
