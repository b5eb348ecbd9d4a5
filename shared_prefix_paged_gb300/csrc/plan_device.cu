// plan_device.cu — the common-prefix planner as a kernel, for steps captured in a CUDA
// graph.
//
// "vLLM Cascade Attention：用法、场景与原理解析" §十一: cascade cannot run inside a full
// CUDA graph because the use-cascade decision is taken per batch on the host, the
// number of kernel calls changes with it, and the block table is sliced to the
// prefix; §七: FlashInfer's cascade splits a plan step from the run step so that the
// run can be captured.  Here the plan itself runs on the device: it reads the batch's
// block table, lengths and computed-token counts where they already are (device
// memory) and writes the prefix length for the attention call into device memory,
// where cascade_attn_device_plan reads it.  So a step is the same fixed sequence of
// launches whatever the batch, and a prefix length of 0 (cascade not taken) makes the
// attention call compute the standard path.
//
// The arithmetic is cascade_plan's (§八 Step 1-2, §三), in parallel: the longest run,
// from block 0, of block ids every row shares within its first cdiv(seq_len, bs)
// entries is the smallest column where some row differs from row 0 (or the shortest
// row's used entries); then blocks to tokens, the cap to min(num_computed_tokens) and
// the floor to block_size; then the mode's use-cascade rule.
#include <climits>

#include "csp.h"
#include "kernels.cuh"

namespace csp {
namespace {

constexpr int kPlanThreads = 512;

__global__ void __launch_bounds__(kPlanThreads)
    plan_device_kernel(const int32_t* __restrict__ bt, int64_t stride, int num_reqs,
                       const int32_t* __restrict__ seq_lens,
                       const int32_t* __restrict__ computed, int bs, int mode,
                       int32_t* __restrict__ plan) {
  __shared__ int s_bad;
  __shared__ unsigned long long s_short, s_flat;
  __shared__ int s_minc, s_first;
  if (num_reqs == 0) {  // an empty batch: no prefix, no cascade
    if (threadIdx.x == 0) plan[0] = plan[1] = plan[2] = plan[3] = 0;
    return;
  }
  if (threadIdx.x == 0) {
    s_bad = 0;
    s_short = ULLONG_MAX;
    s_flat = 0ull;
    s_minc = INT_MAX;
  }
  __syncthreads();
  for (int r = threadIdx.x; r < num_reqs; r += blockDim.x) {
    const int sl = seq_lens[r], nc = computed[r];
    if (sl < 0 || nc < 0 || nc > sl) {
      s_bad = 1;
      continue;
    }
    const long long used = (static_cast<long long>(sl) + bs - 1) / bs;
    if (used > stride) s_bad = 1;
    atomicMin(&s_short, static_cast<unsigned long long>(used));
    atomicMin(&s_minc, nc);
    atomicAdd(&s_flat, static_cast<unsigned long long>(sl));
  }
  __syncthreads();
  if (s_bad) {
    if (threadIdx.x == 0) {
      plan[0] = 0;
      plan[1] = 0;
      plan[2] = 0;
      plan[3] = CSP_ERR_INVALID_ARG;
    }
    return;
  }
  // the first column where a row differs from row 0, within the shortest row's entries
  const long long width = static_cast<long long>(s_short);
  if (threadIdx.x == 0) s_first = static_cast<int>(width);
  __syncthreads();
  const long long pairs = static_cast<long long>(num_reqs - 1) * width;
  for (long long i = threadIdx.x; i < pairs; i += blockDim.x) {
    const long long k = i % width;
    if (k >= s_first) continue;  // a difference further left is already known
    const long long r = 1 + i / width;
    if (bt[r * stride + k] != bt[k]) atomicMin(&s_first, static_cast<int>(k));
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  long long cpl = static_cast<long long>(s_first) * bs;
  cpl = cpl < s_minc ? cpl : s_minc;
  cpl = (cpl / bs) * bs;
  int use = 0;
  switch (mode) {
    case CSP_MODE_FORCE_CASCADE:
      use = cpl > 0;
      break;
    case CSP_MODE_FORCE_FLAT:
      use = 0;
      break;
    case CSP_MODE_PAGE_THRESHOLDS:
      use = cpl >= 256 && num_reqs >= 8;
      break;
    default: {
      // the GB300 rule of cascade_plan: cascade when the standard path would stream at
      // least 8192 KV tokens and cascade cuts them by at least 1.8x
      const long long flat = static_cast<long long>(s_flat);
      const long long casc = cpl + flat - static_cast<long long>(num_reqs) * cpl;
      use = cpl > 0 && casc > 0 && flat >= 8192 && 5 * flat >= 9 * casc;
      break;
    }
  }
  plan[0] = use ? static_cast<int32_t>(cpl) : 0;
  plan[1] = use;
  plan[2] = static_cast<int32_t>(cpl);
  plan[3] = CSP_OK;
}

}  // namespace

cudaError_t launch_plan_device(const int32_t* block_table, int64_t bt_row_stride, int num_reqs,
                               const int32_t* seq_lens, const int32_t* computed, int block_size,
                               int mode, int32_t* plan, cudaStream_t stream) {
  plan_device_kernel<<<1, kPlanThreads, 0, stream>>>(block_table, bt_row_stride, num_reqs,
                                                     seq_lens, computed, block_size, mode, plan);
  return cudaGetLastError();
}

}  // namespace csp
