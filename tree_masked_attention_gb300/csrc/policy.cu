// tree_policy_loss: the per-occurrence clipped policy objective and its gradient with
// respect to each occurrence's log-probability (the incoming gradient of
// tree_logprob_bwd).
//
// Trie packing (agillm.io), "The training-loop change is small": for PPO/GRPO each
// occurrence keeps its own advantage, old log-probability, clipping rule, mask and
// weight (advantages are not averaged before the clipped loss). Tree Training
// (arXiv 2511.00413) §3.1 eq. 1: at ratio 1 this is the policy-gradient objective
// -A log p. With r = exp(logp - old_logp):
//   loss_o = -w m min(r A, clip(r, 1 - eps_low, 1 + eps_high) A)
//   grad_o = -w m A r where the unclipped term is the minimum, else 0.
// Elementwise over occurrences (memory-bound, 20 B read and 8 B written per
// occurrence); the sum is a second one-block pass in a fixed order (deterministic).
#include <cmath>

#include "common.h"

namespace tree {

__global__ void policy_loss_kernel(const float* __restrict__ logp, const float* __restrict__ old_logp,
                                   const float* __restrict__ adv, const float* __restrict__ weight,
                                   const uint8_t* __restrict__ mask, int64_t n, float lo, float hi,
                                   float* __restrict__ loss, float* __restrict__ grad) {
  const int64_t o = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (o >= n) return;
  const float a = adv[o];
  const float r = expf(logp[o] - old_logp[o]);
  const float u = r * a, c = fminf(fmaxf(r, lo), hi) * a;
  const bool take_unclipped = u <= c;
  float wm = weight ? weight[o] : 1.f;
  if (mask && mask[o] == 0) wm = 0.f;
  if (loss) loss[o] = -wm * (take_unclipped ? u : c);
  grad[o] = take_unclipped ? -wm * a * r : 0.f;
}

// One block: thread t adds entries t, t + 1024, ... in double, then a fixed tree.
__global__ void __launch_bounds__(1024) policy_sum_kernel(const float* __restrict__ loss, int64_t n,
                                                          float* __restrict__ out) {
  __shared__ double part[1024];
  double acc = 0.0;
  for (int64_t o = threadIdx.x; o < n; o += blockDim.x) acc += loss[o];
  part[threadIdx.x] = acc;
  __syncthreads();
  for (int s = blockDim.x / 2; s > 0; s >>= 1) {
    if (static_cast<int>(threadIdx.x) < s) part[threadIdx.x] += part[threadIdx.x + s];
    __syncthreads();
  }
  if (threadIdx.x == 0) *out = static_cast<float>(part[0]);
}

}  // namespace tree

extern "C" int tree_policy_loss(const float* logp, const float* old_logp, const float* advantage,
                                const float* weight, const uint8_t* mask, int64_t n_occ, float eps_low,
                                float eps_high, float* loss, float* grad_logp, float* loss_sum,
                                tree_stream_t stream) {
  tree::clear_error();
  if (n_occ < 0) return tree::fail(TREE_ERR_SHAPE, "tree_policy_loss: n_occ = %lld", static_cast<long long>(n_occ));
  if (!(eps_low >= 0.f && eps_low < 1.f) || !(eps_high >= 0.f) || !std::isfinite(eps_high))
    return tree::fail(TREE_ERR_INVALID_ARG, "tree_policy_loss: need 0 <= eps_low < 1 and finite eps_high >= 0");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (n_occ == 0) {  // (empty arrays may come as null pointers)
    if (loss_sum) TREE_CUDA_TRY(cudaMemsetAsync(loss_sum, 0, sizeof(float), st));
    return TREE_OK;
  }
  if (loss_sum && !loss)
    return tree::fail(TREE_ERR_INVALID_ARG, "tree_policy_loss: loss_sum needs the per-occurrence loss array");
  if (!logp || !old_logp || !advantage || !grad_logp)
    return tree::fail(TREE_ERR_INVALID_ARG, "tree_policy_loss: null pointer");
  tree::policy_loss_kernel<<<static_cast<unsigned>((n_occ + 255) / 256), 256, 0, st>>>(
      logp, old_logp, advantage, weight, mask, n_occ, 1.f - eps_low, 1.f + eps_high, loss, grad_logp);
  TREE_LAUNCH_CHECK("policy_loss_kernel");
  if (loss_sum) {
    tree::policy_sum_kernel<<<1, 1024, 0, st>>>(loss, n_occ, loss_sum);
    TREE_LAUNCH_CHECK("policy_sum_kernel");
  }
  return TREE_OK;
}
