// Top-k routing of one batch by the threads of one CTA: the device function
// behind pw_moe_route_topk (route.cu) and the routing phase of the fused
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

// Shared-memory scratch of route_block: 3*E ints plus nwarps*E ints.
__host__ __device__ constexpr size_t scratch_bytes(int E, int nwarps) {
  return static_cast<size_t>(3 + nwarps) * static_cast<size_t>(E) * 4u;
}

// Every thread of the CTA calls this (it synchronises the CTA).  blockDim.x is
// a multiple of 32; `scratch` is shared memory of scratch_bytes(E + S, warps).
// logits are [T][E] (routed experts).  Each token gets K = k + S slots: its
// top-k routed experts, then the S shared experts E .. E+S-1 with weight 1
// (experts every token passes through, added to the routed output).  Writes
// ids [T][K], w [T][K], offsets [E+S+1], perm [T*K] and inv_perm [T*K]
// (global); adds the routing mass of the batch (per expert, shared experts
// included) to mass_accum when it is not NULL, summed in a fixed order so that
// every result is the same from run to run.  The arrays are read back by this
// CTA, so they must not alias the logits.
__device__ inline void route_block(const float* __restrict__ logits, int T, int E, int k, int S, int32_t* ids,
                                   float* w, int32_t* offsets, int32_t* perm, int32_t* inv_perm,
                                   float* mass_accum, uint8_t* scratch) {
  const int K = k + S, ET = E + S;
  const int nthreads = static_cast<int>(blockDim.x), nwarps = nthreads >> 5;
  const int tid = static_cast<int>(threadIdx.x), lane = tid & 31, warp = tid >> 5;
  int* s_cnt = reinterpret_cast<int*>(scratch);
  int* s_base = s_cnt + ET;
  int* s_chunk = s_base + ET;
  int* s_wcnt = s_chunk + ET;   // [nwarps][E + S]
  for (int e = tid; e < ET; e += nthreads) s_cnt[e] = 0;
  __syncthreads();

  // 1) top-k per token: largest logit first, ties to the lower expert index;
  //    weights = softmax renormalised over the picks = exp(l_j - l_max) / sum.
  //    Up to 32 experts the row is loaded into registers first (independent
  //    loads, one memory latency per token instead of one per logit).  When
  //    the batch fits one pass, each thread keeps its picks for step 3.
  const bool one_pass = T <= nthreads;
  int keep[kMaxK];
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) keep[j] = -1;
  for (int t = tid; t < T; t += nthreads) {
    const float* row = logits + static_cast<long long>(t) * E;
    int sel[kMaxK];
    float lsel[kMaxK];
    if (E <= 32) {
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
    } else {
      uint32_t taken[kMaxE / 32];
#pragma unroll
      for (int i = 0; i < kMaxE / 32; ++i) taken[i] = 0u;
      for (int j = 0; j < k; ++j) {
        int best = -1;
        float lb = 0.f;
        for (int e = 0; e < E; ++e) {
          if ((taken[e >> 5] >> (e & 31)) & 1u) continue;
          const float v = __ldg(row + e);
          if (best < 0 || v > lb) {
            best = e;
            lb = v;
          }
        }
        taken[best >> 5] |= 1u << (best & 31);
        sel[j] = best;
        lsel[j] = lb;
      }
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
      atomicAdd(&s_cnt[e], 1);
      keep[j] = e;
    }
  }
  __syncthreads();

  // 2) expert offsets (exclusive scan of the counts)
  if (tid == 0) {
    int run = 0;
    for (int e = 0; e < ET; ++e) {
      offsets[e] = run;
      s_base[e] = run;
      run += s_cnt[e];
    }
    offsets[ET] = run;
  }
  __syncthreads();

  // 3) stable placement, one token per thread per chunk: the rank of token t
  //    inside expert e is the number of earlier tokens that also chose e.
  for (int c0 = 0; c0 < T; c0 += nthreads) {
    const int t = c0 + tid;
    const bool valid = t < T;
    int my[kMaxK];
    int rank[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      my[j] = (valid && j < K) ? (one_pass ? keep[j] : ids[static_cast<long long>(t) * K + j]) : -1;
      rank[j] = 0;
    }
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int e = 0; e < ET; ++e) {
      int jj = -1;
#pragma unroll
      for (int j = 0; j < kMaxK; ++j)
        if (my[j] == e) jj = j;
      const unsigned ball = __ballot_sync(0xffffffffu, jj >= 0);
      if (jj >= 0) rank[jj] = __popc(ball & lt_mask);
      if (lane == 0) s_wcnt[warp * ET + e] = __popc(ball);
    }
    __syncthreads();
    for (int e = tid; e < ET; e += nthreads) {
      int run = 0;
      for (int wi = 0; wi < nwarps; ++wi) {
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
        perm[pos] = slot;
        inv_perm[slot] = pos;
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
      for (int pos = offsets[e] + lane; pos < offsets[e + 1]; pos += 32) acc += w[perm[pos]];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) atomicAdd(&mass_accum[e], acc);
    }
  }
}

}  // namespace pw_route
