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
// without a second launch.  The algorithm is route_block.cuh.
#include "route_block.cuh"

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
using pw_route::kMaxE;
using pw_route::kMaxK;
constexpr size_t kScratch = 47 * 1024;
static_assert(pw_route::scratch_bytes(kMaxE, kWarps) <= kScratch, "routing scratch");

__global__ void __launch_bounds__(kThreads) route_kernel(const float* __restrict__ logits, int T, int E, int k, int S,
                                                         int32_t* __restrict__ ids, float* __restrict__ w,
                                                         int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                                                         int32_t* __restrict__ inv_perm, float* __restrict__ mass_accum) {
  // the required part plus room for the weights of up to ~2900 assignments
  __shared__ __align__(16) uint8_t scratch[kScratch];
  pw_route::route_block(logits, T, E, k, S, ids, w, offsets, perm, inv_perm, mass_accum, scratch, kScratch);
}

}  // namespace

extern "C" int pw_moe_route_topk_shared(const float* d_logits, int T, int E, int k, int S, int32_t* d_ids,
                                        float* d_w, int32_t* d_offsets, int32_t* d_perm, int32_t* d_inv_perm,
                                        float* d_mass_accum, void* stream) {
  if (E < 1 || k < 1 || k > E || S < 0 || E + S > kMaxE || k + S > kMaxK)
    return pw::set_error(PW_ERR_UNSUPPORTED,
                         "route: need 1 <= k <= E, S >= 0, E + S <= %d, k + S <= %d (E=%d k=%d S=%d)", kMaxE, kMaxK,
                         E, k, S);
  if (T < 0 || T > (1 << 20)) return pw::set_error(PW_ERR_UNSUPPORTED, "route: T=%d outside [0, 2^20]", T);
  if (!d_offsets || (T > 0 && (!d_logits || !d_ids || !d_w || !d_perm || !d_inv_perm)))
    return pw::set_error(PW_ERR_INVALID_ARG, "route: NULL argument");
  route_kernel<<<1, kThreads, 0, pw::as_stream(stream)>>>(d_logits, T, E, k, S, d_ids, d_w, d_offsets, d_perm,
                                                         d_inv_perm, d_mass_accum);
  PW_CUDA_TRY(cudaGetLastError());
  return PW_OK;
}

extern "C" int pw_moe_route_topk(const float* d_logits, int T, int E, int k, int32_t* d_ids, float* d_w,
                                 int32_t* d_offsets, int32_t* d_perm, int32_t* d_inv_perm, float* d_mass_accum,
                                 void* stream) {
  return pw_moe_route_topk_shared(d_logits, T, E, k, 0, d_ids, d_w, d_offsets, d_perm, d_inv_perm, d_mass_accum,
                                  stream);
}
