// Top-k routing of one batch: route_block (the threads of one CTA) is the
// device function behind the routing launch (route.cu: pw_moe_route_topk and
// the routed fused calls whose batches one warp does not route); route_warp
// (one warp, small batches) is also the routing phase inside the fused
// routed layer (ffn_stream.cuh).
//
// "PagedWeight" arXiv text, §2.1: the router gives weights to E experts and
// the top K are selected per token; Eq. 1 defines the routing mass of expert e
// as the routing weight it received over the total.  The permutation (slots
// ordered by expert, then token, then choice) is what lets the fused layer
// process each expert's tokens as one contiguous group.
#pragma once

#include "pw_internal.h"

namespace pw_route {

constexpr int kMaxE = 256;   // routed + shared experts
constexpr int kMaxK = 16;    // slots per token: routed top-k + shared experts

// Shared-memory scratch route_block needs at least: 3*E ints, nwarps*E ints
// and E + 1 offsets.  With 2*T*K more floats it also keeps the weights (by
// slot, then in position order) for the routing mass; else it reads them back
// from w.
__host__ __device__ constexpr size_t scratch_bytes(int E, int nwarps) {
  return (static_cast<size_t>(3 + nwarps) * static_cast<size_t>(E) + static_cast<size_t>(E) + 1u) * 4u;
}

// Every thread of the CTA calls this (it synchronises the CTA).  blockDim.x is
// a multiple of 32; `scratch` is `scratch_cap` bytes of shared memory, at least
// scratch_bytes(E + S, warps).
// logits are [T][E] (routed experts).  Each token gets K = k + S slots: its
// top-k routed experts, then the S shared experts E .. E+S-1 with weight 1
// (experts every token passes through, added to the routed output).  Writes
// ids [T][K], w [T][K], offsets [E+S+1], perm [T*K] and inv_perm [T*K]
// (global); adds the routing mass of the batch (per expert, shared experts
// included) to mass_accum when it is not NULL, summed in a fixed order so that
// every result is the same from run to run.  The arrays are read back by this
// CTA, so they must not alias the logits.
// `base` is added to every offset, permutation entry and inverse-permutation
// entry written (not to ids): a batch routed as one layer of several whose
// assignment arrays are concatenated, this layer's slots starting at `base`
// (the caller offsets the array pointers to this layer's part).
__device__ inline void route_block(const float* __restrict__ logits, int T, int E, int k, int S, int32_t* ids,
                                   float* w, int32_t* offsets, int32_t* perm, int32_t* inv_perm,
                                   float* mass_accum, uint8_t* scratch, size_t scratch_cap, int base = 0) {
  const int K = k + S, ET = E + S;
  const int nthreads = static_cast<int>(blockDim.x), nwarps = nthreads >> 5;
  const int tid = static_cast<int>(threadIdx.x), lane = tid & 31, warp = tid >> 5;
  int* s_cnt = reinterpret_cast<int*>(scratch);
  int* s_base = s_cnt + ET;
  int* s_chunk = s_base + ET;
  int* s_wcnt = s_chunk + ET;   // [nwarps][E + S]
  int* s_off = s_wcnt + nwarps * ET;   // [E + S + 1] the offsets, for step 4
  float* s_wslot = reinterpret_cast<float*>(s_off + ET + 1);   // [T * K] weights by slot
  float* s_wpos = s_wslot + static_cast<long long>(T) * K;     // [T * K] weights in position order
  const bool wpos_smem = scratch_bytes(ET, nwarps) + static_cast<size_t>(T) * K * 8u <= scratch_cap;
  for (int e = tid; e < ET; e += nthreads) s_cnt[e] = 0;
  __syncthreads();

  // 1) top-k per token: largest logit first, ties to the lower expert index;
  //    weights = softmax renormalised over the picks = exp(l_j - l_max) / sum.
  //    Up to 32 experts one thread takes a token and loads its row into
  //    registers first (independent loads, one memory latency per token
  //    instead of one per logit); above 32 experts one warp takes a token
  //    (step 1b).  Step 3 reads the picks back from ids.
  for (int t = tid; t < T && E <= 32; t += nthreads) {
    const float* row = logits + static_cast<long long>(t) * E;
    int sel[kMaxK];
    float lsel[kMaxK];
    float v[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) v[e] = e < E ? __ldg(row + e) : 0.f;
    uint32_t taken = 0u;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      if (j >= k) break;
      int best = -1;
      float lb = 0.f;
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        if (e < E && !((taken >> e) & 1u) && (best < 0 || v[e] > lb)) {
          best = e;
          lb = v[e];
        }
      }
      taken |= 1u << best;
      sel[j] = best;
      lsel[j] = lb;
    }
    float den = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j)
      if (j < k) den += expf(lsel[j] - lsel[0]);
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      if (j >= K) break;
      const bool routed = j < k;
      const int e = routed ? sel[j] : E + (j - k);
      const float wj = routed ? expf(lsel[j] - lsel[0]) / den : 1.0f;
      ids[static_cast<long long>(t) * K + j] = e;
      w[static_cast<long long>(t) * K + j] = wj;
      if (wpos_smem) s_wslot[static_cast<long long>(t) * K + j] = wj;
      atomicAdd(&s_cnt[e], 1);
    }
  }
  // 1b) more than 32 experts: one warp per token, lane l holding logits
  //     l, l + 32, ...; each pick is a warp arg-max under the order of the
  //     scan above (larger logit, then the lower expert index), taken from
  //     lane 0 so that every lane agrees.  Lane j keeps pick j and writes
  //     slot j; the denominator is summed in pick order, as above.
  for (int t = warp; t < T && E > 32; t += nwarps) {
    const float* row = logits + static_cast<long long>(t) * E;
    float v[kMaxE / 32];
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i) v[i] = lane + 32 * i < E ? __ldg(row + lane + 32 * i) : 0.f;
    uint32_t taken = 0u;   // bit i: expert lane + 32 i already picked
    int my_e = -1;
    float my_l = 0.f, l0 = 0.f, den = 0.f;
    for (int j = 0; j < k; ++j) {
      int best = -1;
      float lb = 0.f;
#pragma unroll
      for (int i = 0; i < kMaxE / 32; ++i) {
        if (lane + 32 * i < E && !((taken >> i) & 1u) && (best < 0 || v[i] > lb)) {
          best = lane + 32 * i;
          lb = v[i];
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const int ob = __shfl_xor_sync(0xffffffffu, best, o);
        const float ol = __shfl_xor_sync(0xffffffffu, lb, o);
        if (ob >= 0 && (best < 0 || ol > lb || (ol == lb && ob < best))) {
          best = ob;
          lb = ol;
        }
      }
      best = __shfl_sync(0xffffffffu, best, 0);
      lb = __shfl_sync(0xffffffffu, lb, 0);
      if ((best & 31) == lane) taken |= 1u << (best >> 5);
      if (j == 0) l0 = lb;
      den += expf(lb - l0);
      if (lane == j) {
        my_e = best;
        my_l = lb;
      }
    }
    if (lane < K) {
      const int j = lane;
      const bool routed = j < k;
      const int e = routed ? my_e : E + (j - k);
      const float wj = routed ? expf(my_l - l0) / den : 1.0f;
      ids[static_cast<long long>(t) * K + j] = e;
      w[static_cast<long long>(t) * K + j] = wj;
      if (wpos_smem) s_wslot[static_cast<long long>(t) * K + j] = wj;
      atomicAdd(&s_cnt[e], 1);
    }
  }
  __syncthreads();

  // 2) expert offsets (exclusive scan of the counts) by warp 0: lane l scans
  //    experts [l*n, l*n + n), then a shuffle scan over the lanes' sums
  if (warp == 0) {
    const int n = (ET + 31) >> 5, e0 = lane * n;
    int part = 0;
    for (int e = e0; e < min(e0 + n, ET); ++e) part += s_cnt[e];
    int incl = part;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - part;
    for (int e = e0; e < min(e0 + n, ET); ++e) {
      offsets[e] = base + run;
      s_base[e] = run;
      s_off[e] = run;
      run += s_cnt[e];
    }
    if (lane == 31) {
      offsets[ET] = base + incl;
      s_off[ET] = incl;
    }
  }
  __syncthreads();

  // 3) stable placement, one token per thread per chunk: the rank of token t
  //    inside expert e is the number of earlier tokens of its warp that also
  //    chose e (the lanes' bits in the warp's mask for e), plus the counts of
  //    the earlier warps.  Only the warps that hold tokens of the chunk take
  //    part; a token picks an expert at most once.
  for (int c0 = 0; c0 < T; c0 += nthreads) {
    const int t = c0 + tid;
    const bool valid = t < T;
    const int nwa = (min(T - c0, nthreads) + 31) >> 5;
    int my[kMaxK];
    int rank[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      my[j] = (valid && j < K) ? ids[static_cast<long long>(t) * K + j] : -1;
      rank[j] = 0;
    }
    const unsigned lt_mask = (1u << lane) - 1u;
    if (warp < nwa) {
      unsigned* wmask = reinterpret_cast<unsigned*>(s_wcnt + warp * ET);   // this warp's row: lane masks
      for (int e = lane; e < ET; e += 32) wmask[e] = 0u;
      __syncwarp();
#pragma unroll
      for (int j = 0; j < kMaxK; ++j)
        if (my[j] >= 0) atomicOr(&wmask[my[j]], 1u << lane);
      __syncwarp();
#pragma unroll
      for (int j = 0; j < kMaxK; ++j)
        if (my[j] >= 0) rank[j] = __popc(wmask[my[j]] & lt_mask);
      __syncwarp();
      for (int e = lane; e < ET; e += 32) s_wcnt[warp * ET + e] = __popc(wmask[e]);
    }
    __syncthreads();
    for (int e = tid; e < ET; e += nthreads) {
      int run = 0;
      for (int wi = 0; wi < nwa; ++wi) {
        const int v = s_wcnt[wi * ET + e];
        s_wcnt[wi * ET + e] = run;
        run += v;
      }
      s_chunk[e] = run;
    }
    __syncthreads();
    if (valid) {
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) {
        if (j >= K) break;
        const int e = my[j];
        const int pos = s_base[e] + s_wcnt[warp * ET + e] + rank[j];
        const int slot = t * K + j;
        perm[pos] = base + slot;
        inv_perm[slot] = base + pos;
        if (wpos_smem) s_wpos[pos] = s_wslot[slot];
      }
    }
    __syncthreads();
    for (int e = tid; e < ET; e += nthreads) s_base[e] += s_chunk[e];
    __syncthreads();
  }

  // 4) Eq. 1 numerator, accumulated across calls: warp e sums expert e's
  //    routing weights in expert order (lane-strided, then a fixed shuffle
  //    tree), one addition per expert per call
  if (mass_accum) {
    for (int e = warp; e < ET; e += nwarps) {
      float acc = 0.f;
      for (int pos = s_off[e] + lane; pos < s_off[e + 1]; pos += 32) acc += wpos_smem ? s_wpos[pos] : w[perm[pos] - base];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) atomicAdd(&mass_accum[e], acc);
    }
  }
}

// The same routing by one warp, for batches of at most 32 tokens over at most
// kWarpMaxE experts (routed + shared) with at most kWarpMaxK slots per token:
// lane t routes token t, counts come from warp ballots, no CTA barrier.
// Every result equals route_block's bit for bit: the top-k and weights are
// the same per-token code (route_block's one-thread-per-token path for up to
// 32 experts), a token's position is
// its expert's offset plus the number of earlier tokens that chose the
// expert, and the routing mass is summed in the same order (by position,
// lane-strided, then the same shuffle tree).  Called by all 32 lanes of one
// warp; `s_wpos` is T*K floats of shared memory.
constexpr int kWarpMaxE = 8;
constexpr int kWarpMaxK = 4;
__host__ __device__ constexpr bool warp_routes(int T, int ET, int K) {
  return T <= 32 && ET <= kWarpMaxE && K <= kWarpMaxK;
}
__device__ inline void route_warp(const float* __restrict__ logits, int T, int E, int k, int S, int32_t* ids,
                                  float* w, int32_t* offsets, int32_t* perm, int32_t* inv_perm, float* mass_accum,
                                  float* s_wpos, int base = 0) {
  const int K = k + S, ET = E + S;
  const int t = static_cast<int>(threadIdx.x & 31);
  const bool valid = t < T;
  int sel[kWarpMaxK];
  float wsel[kWarpMaxK];
#pragma unroll
  for (int j = 0; j < kWarpMaxK; ++j) {
    sel[j] = -1;
    wsel[j] = 0.f;
  }
  if (valid) {
    const float* row = logits + static_cast<long long>(t) * E;
    float v[kWarpMaxE];
#pragma unroll
    for (int e = 0; e < kWarpMaxE; ++e) v[e] = e < E ? __ldg(row + e) : 0.f;
    float lsel[kWarpMaxK];
    uint32_t taken = 0u;
#pragma unroll
    for (int j = 0; j < kWarpMaxK; ++j) {
      if (j >= k) break;
      int best = -1;
      float lb = 0.f;
#pragma unroll
      for (int e = 0; e < kWarpMaxE; ++e) {
        if (e < E && !((taken >> e) & 1u) && (best < 0 || v[e] > lb)) {
          best = e;
          lb = v[e];
        }
      }
      taken |= 1u << best;
      sel[j] = best;
      lsel[j] = lb;
    }
    float den = 0.f;
#pragma unroll
    for (int j = 0; j < kWarpMaxK; ++j)
      if (j < k) den += expf(lsel[j] - lsel[0]);
#pragma unroll
    for (int j = 0; j < kWarpMaxK; ++j) {
      if (j >= K) break;
      const bool routed = j < k;
      sel[j] = routed ? sel[j] : E + (j - k);
      wsel[j] = routed ? expf(lsel[j] - lsel[0]) / den : 1.0f;
      ids[static_cast<long long>(t) * K + j] = sel[j];
      w[static_cast<long long>(t) * K + j] = wsel[j];
    }
  }
  // offsets: an exclusive scan of the per-expert counts (lane e holds expert
  // e's count and, after the scan, its first position)
  const unsigned lt_mask = (1u << t) - 1u;
  int my_cnt = 0, my_off = 0, total = 0;
  for (int e = 0; e < ET; ++e) {
    bool mine = false;
#pragma unroll
    for (int j = 0; j < kWarpMaxK; ++j) mine |= sel[j] == e;
    const int c = __popc(__ballot_sync(0xffffffffu, mine));
    if (t == e) {
      my_cnt = c;
      my_off = total;
    }
    total += c;
  }
  if (t < ET) offsets[t] = base + my_off;
  if (t == 0) offsets[ET] = base + total;
  // placement: position = the expert's offset + the earlier tokens that chose
  // it in any of their slots (a token picks an expert at most once)
  for (int ee = 0; ee < ET; ++ee) {
    bool mine = false;
    int jm = 0;
    float wm = 0.f;
#pragma unroll
    for (int j = 0; j < kWarpMaxK; ++j) {
      if (j < K && sel[j] == ee) {
        mine = true;
        jm = j;
        wm = wsel[j];
      }
    }
    const unsigned ball = __ballot_sync(0xffffffffu, mine);
    const int off_e = __shfl_sync(0xffffffffu, my_off, ee);
    if (mine) {
      const int pos = off_e + __popc(ball & lt_mask);
      const int slot = t * K + jm;
      perm[pos] = base + slot;
      inv_perm[slot] = base + pos;
      s_wpos[pos] = wm;
    }
  }
  __syncwarp();
  // Eq. 1 numerator: per expert, the weights in position order, lane-strided,
  // then the shuffle tree (route_block's order)
  if (mass_accum) {
    for (int e = 0; e < ET; ++e) {
      const int o0 = __shfl_sync(0xffffffffu, my_off, e), n = __shfl_sync(0xffffffffu, my_cnt, e);
      float acc = 0.f;
      for (int pos = o0 + t; pos < o0 + n; pos += 32) acc += s_wpos[pos];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (t == 0) atomicAdd(&mass_accum[e], acc);
    }
  }
  (void)my_cnt;
}

}  // namespace pw_route
