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
//  * q >= 5: the LUT lives in shared memory, one 4-byte column per lane
//    ("bank per lane": entry c of lane l's row at word c*32 + l), so the 32
//    lanes of a warp never conflict; for q = 8 a word holds entries c and
//    c+128.
#pragma once

#include "tc_ptx.cuh"

namespace pw {

constexpr int kStageK = 64;                      // columns per pipeline stage
constexpr int kLutBytesPerWarp = 128 * 128;      // shared LUT table of one warp (q >= 5)

// Nibble selector of 8 consecutive columns (sub-block js) from one word per
// plane, using planes [P0, P1) as index bits (P1-1-p) .. 0.
template <int P0, int P1>
__device__ __forceinline__ uint32_t nibble_sel(const uint32_t* w, int js) {
  uint32_t s = 0u;
#pragma unroll
  for (int p = P0; p < P1; ++p) s |= ((w[p] >> js) & 0x11111111u) << (P1 - 1 - p);
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
template <int Q>
struct RowDequant<Q, false> {
  static constexpr int kWords = (Q == 8) ? 128 : (1 << Q);
  uint32_t tbl;  // shared address of this lane's column

  // Fill this lane's column of the warp's table from its LUT row.
  __device__ __forceinline__ void load(const uint16_t* __restrict__ lut_row, uint32_t warp_tbl, int lane) {
    tbl = warp_tbl + static_cast<uint32_t>(lane) * 4u;
    const uint4* src = reinterpret_cast<const uint4*>(lut_row);
#pragma unroll 4
    for (int c8 = 0; c8 < kWords / 8; ++c8) {
      const uint4 a = __ldg(src + c8);
      uint4 b = make_uint4(0u, 0u, 0u, 0u);
      if (Q == 8) b = __ldg(src + c8 + 16);   // entries c + 128
      const uint32_t av[4] = {a.x, a.y, a.z, a.w};
      const uint32_t bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int c = c8 * 8 + 2 * i;
        const uint32_t e0 = av[i] & 0xFFFFu, e1 = av[i] >> 16;
        const uint32_t f0 = bv[i] & 0xFFFFu, f1 = bv[i] >> 16;
        sts_u32(tbl + static_cast<uint32_t>(c) * 128u, e0 | (f0 << 16));
        sts_u32(tbl + static_cast<uint32_t>(c + 1) * 128u, e1 | (f1 << 16));
      }
    }
  }

  __device__ __forceinline__ uint32_t look(uint32_t idx) const {
    if (Q == 8) return lds_u16(tbl + ((idx & 127u) << 7) + ((idx >> 7) << 1));
    return lds_u16(tbl + (idx << 7));
  }

  __device__ __forceinline__ void word(const uint32_t (&ww)[Q], uint32_t (&out)[16]) const {
#pragma unroll
    for (int js = 0; js < 4; ++js) {
      const uint32_t hi = nibble_sel<0, Q - 4>(ww, js);
      const uint32_t lo = nibble_sel<Q - 4, Q>(ww, js);
      uint32_t v[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint32_t idx = ((lo >> (4 * e)) & 0xFu) | (((hi >> (4 * e)) & 0xFu) << 4);
        v[e] = look(idx);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) out[4 * js + i] = v[2 * i] | (v[2 * i + 1] << 16);
    }
  }
};

}  // namespace pw
