// Top-k routing, expert-ordered permutation and routing mass in one launch.
//
// "PagedWeight" arXiv text, §2.1: the router gives weights to E experts and
// the top K are selected per token; Eq. 1 defines the routing mass of expert e
// as the routing weight it received over the total.  The permutation (slots
// ordered by expert, then token, then choice) is what lets the fused layer
// process each expert's tokens as one contiguous group.
//
// One CTA: routing work is at most a few thousand assignments per layer call,
// far below one wave; a single CTA keeps the counting sort exact and stable
// without a second launch.
#include "pw_internal.h"

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxE = 256;
constexpr int kMaxK = 8;

__global__ void __launch_bounds__(kThreads) route_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                         int32_t* __restrict__ ids, float* __restrict__ w,
                                                         int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                                                         int32_t* __restrict__ inv_perm, float* __restrict__ mass_accum) {
  __shared__ int s_cnt[kMaxE];
  __shared__ int s_base[kMaxE];
  __shared__ int s_chunk[kMaxE];
  __shared__ float s_mass[kMaxE];
  __shared__ int s_wcnt[kWarps][kMaxE];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int e = tid; e < E; e += kThreads) {
    s_cnt[e] = 0;
    s_mass[e] = 0.f;
  }
  __syncthreads();

  // 1) top-k per token: largest logit first, ties to the lower expert index;
  //    weights = softmax renormalised over the picks = exp(l_j - l_max) / sum.
  for (int t = tid; t < T; t += kThreads) {
    const float* row = logits + static_cast<long long>(t) * E;
    uint32_t taken[kMaxE / 32];
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i) taken[i] = 0u;
    int sel[kMaxK];
    float lsel[kMaxK];
    for (int j = 0; j < k; ++j) {
      int best = -1;
      float lb = 0.f;
      for (int e = 0; e < E; ++e) {
        if ((taken[e >> 5] >> (e & 31)) & 1u) continue;
        const float v = row[e];
        if (best < 0 || v > lb) {
          best = e;
          lb = v;
        }
      }
      taken[best >> 5] |= 1u << (best & 31);
      sel[j] = best;
      lsel[j] = lb;
    }
    float den = 0.f;
    for (int j = 0; j < k; ++j) den += expf(lsel[j] - lsel[0]);
    for (int j = 0; j < k; ++j) {
      const float wj = expf(lsel[j] - lsel[0]) / den;
      ids[static_cast<long long>(t) * k + j] = sel[j];
      w[static_cast<long long>(t) * k + j] = wj;
      atomicAdd(&s_cnt[sel[j]], 1);
      atomicAdd(&s_mass[sel[j]], wj);
    }
  }
  __syncthreads();

  // 2) expert offsets (exclusive scan of the counts)
  if (tid == 0) {
    int run = 0;
    for (int e = 0; e < E; ++e) {
      offsets[e] = run;
      s_base[e] = run;
      run += s_cnt[e];
    }
    offsets[E] = run;
  }
  __syncthreads();

  // 3) stable placement, one token per thread per chunk: the rank of token t
  //    inside expert e is the number of earlier tokens that also chose e.
  for (int c0 = 0; c0 < T; c0 += kThreads) {
    const int t = c0 + tid;
    const bool valid = t < T;
    int my[kMaxK];
    int rank[kMaxK];
    for (int j = 0; j < k; ++j) {
      my[j] = valid ? ids[static_cast<long long>(t) * k + j] : -1;
      rank[j] = 0;
    }
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int e = 0; e < E; ++e) {
      int jj = -1;
      for (int j = 0; j < k; ++j)
        if (my[j] == e) jj = j;
      const unsigned ball = __ballot_sync(0xffffffffu, jj >= 0);
      if (jj >= 0) rank[jj] = __popc(ball & lt_mask);
      if (lane == 0) s_wcnt[warp][e] = __popc(ball);
    }
    __syncthreads();
    for (int e = tid; e < E; e += kThreads) {
      int run = 0;
      for (int wi = 0; wi < kWarps; ++wi) {
        const int v = s_wcnt[wi][e];
        s_wcnt[wi][e] = run;
        run += v;
      }
      s_chunk[e] = run;
    }
    __syncthreads();
    if (valid) {
      for (int j = 0; j < k; ++j) {
        const int e = my[j];
        const int pos = s_base[e] + s_wcnt[warp][e] + rank[j];
        const int slot = t * k + j;
        perm[pos] = slot;
        inv_perm[slot] = pos;
      }
    }
    __syncthreads();
    for (int e = tid; e < E; e += kThreads) s_base[e] += s_chunk[e];
    __syncthreads();
  }

  // 4) Eq. 1 numerator, accumulated across calls
  if (mass_accum)
    for (int e = tid; e < E; e += kThreads) atomicAdd(&mass_accum[e], s_mass[e]);
}

}  // namespace

extern "C" int pw_moe_route_topk(const float* d_logits, int T, int E, int k, int32_t* d_ids, float* d_w,
                                 int32_t* d_offsets, int32_t* d_perm, int32_t* d_inv_perm, float* d_mass_accum,
                                 void* stream) {
  if (E < 1 || E > kMaxE || k < 1 || k > kMaxK || k > E)
    return pw::set_error(PW_ERR_UNSUPPORTED, "route: need 1 <= k <= min(E, 8), E <= 256 (E=%d k=%d)", E, k);
  if (T < 0 || T > (1 << 20)) return pw::set_error(PW_ERR_UNSUPPORTED, "route: T=%d outside [0, 2^20]", T);
  if (!d_offsets || (T > 0 && (!d_logits || !d_ids || !d_w || !d_perm || !d_inv_perm)))
    return pw::set_error(PW_ERR_INVALID_ARG, "route: NULL argument");
  route_kernel<<<1, kThreads, 0, pw::as_stream(stream)>>>(d_logits, T, E, k, d_ids, d_w, d_offsets, d_perm,
                                                         d_inv_perm, d_mass_accum);
  PW_CUDA_TRY(cudaGetLastError());
  return PW_OK;
}
