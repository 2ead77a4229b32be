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

constexpr int kThreads = 512;   // 128 registers a thread: the routing code does not spill
constexpr int kWarps = kThreads / 32;
using pw_route::kMaxE;
using pw_route::kMaxK;
constexpr size_t kScratch = 47 * 1024;
static_assert(pw_route::scratch_bytes(kMaxE, kWarps) <= kScratch, "routing scratch");

// CTA l routes layer l of a batch of independent layers whose arrays are
// concatenated layer after layer (one layer: a grid of one CTA).
__global__ void __launch_bounds__(kThreads) route_kernel(const float* __restrict__ logits, int T, int E, int k, int S,
                                                         int32_t* __restrict__ ids, float* __restrict__ w,
                                                         int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                                                         int32_t* __restrict__ inv_perm, float* __restrict__ mass_accum,
                                                         uint4* __restrict__ zero, int zero_n16) {
  // the required part plus room for the weights of up to ~3400 assignments
  __shared__ __align__(16) uint8_t scratch[kScratch];
  // the next kernel may start launching (it waits for this grid to complete
  // before it reads anything this one writes)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (blockIdx.x == 0)
    for (int i = static_cast<int>(threadIdx.x); i < zero_n16; i += kThreads) zero[i] = make_uint4(0u, 0u, 0u, 0u);
  const long long l = blockIdx.x, A = static_cast<long long>(T) * (k + S);
  if (pw_route::warp_routes(T, E + S, k + S)) {   // small batch: one warp, no CTA barrier (same results)
    if (threadIdx.x < 32)
      pw_route::route_warp(logits + l * T * E, T, E, k, S, ids + l * A, w + l * A, offsets + l * (E + S),
                           perm + l * A, inv_perm + l * A, mass_accum ? mass_accum + l * (E + S) : nullptr,
                           reinterpret_cast<float*>(scratch), static_cast<int>(l * A));
    return;
  }
  pw_route::route_block(logits + l * T * E, T, E, k, S, ids + l * A, w + l * A, offsets + l * (E + S), perm + l * A,
                        inv_perm + l * A, mass_accum ? mass_accum + l * (E + S) : nullptr, scratch, kScratch,
                        static_cast<int>(l * A));
}

}  // namespace

namespace pw {

// Routing of L independent layers in one launch (CTA l: layer l), with the
// offsets, permutation and inverse permutation in the concatenated index
// space of the layers' assignments.
int route_layers(const float* d_logits, int L, int T, int E, int k, int S, int32_t* d_ids, float* d_w,
                 int32_t* d_offsets, int32_t* d_perm, int32_t* d_inv_perm, float* d_mass_accum, cudaStream_t s,
                 void* d_zero, size_t zero_bytes) {
  route_kernel<<<L, kThreads, 0, s>>>(d_logits, T, E, k, S, d_ids, d_w, d_offsets, d_perm, d_inv_perm, d_mass_accum,
                                      static_cast<uint4*>(d_zero), d_zero ? static_cast<int>(zero_bytes / 16) : 0);
  PW_CUDA_TRY(cudaGetLastError());
  return PW_OK;
}

}  // namespace pw

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
  return pw::route_layers(d_logits, 1, T, E, k, S, d_ids, d_w, d_offsets, d_perm, d_inv_perm, d_mass_accum,
                          pw::as_stream(stream));
}

extern "C" int pw_moe_route_topk(const float* d_logits, int T, int E, int k, int32_t* d_ids, float* d_w,
                                 int32_t* d_offsets, int32_t* d_perm, int32_t* d_inv_perm, float* d_mass_accum,
                                 void* stream) {
  return pw_moe_route_topk_shared(d_logits, T, E, k, 0, d_ids, d_w, d_offsets, d_perm, d_inv_perm, d_mass_accum,
                                  stream);
}
