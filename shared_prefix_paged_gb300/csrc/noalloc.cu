// noalloc.cu — cascade_attn for callers that must not allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) on the path that runs
// attention: an engine whose device memory is all handed out up front by its own
// pool, a plugin inside a host framework that owns every allocation, or a
// latency-critical loop where an allocation would synchronise the device.  They
// still own their inputs and outputs, but have nowhere to put the workspace that
// cascade_attn needs for its split partial results.  This entry point gives them
// one: a fixed array in the library's own device memory, reserved when the library's
// device code is loaded on a GPU and held until the process exits.
#include <mutex>

#include "csp.h"

// Largest workspace this entry point can serve (16 MiB).  The N=64, P=4096, S=128
// decode batch with 32 query heads needs about 9.5 MiB.
static constexpr size_t kScratchBytes = static_cast<size_t>(16) << 20;

// One array per device, shared by every call of cascade_attn_noalloc on that device.
static __device__ __align__(256) unsigned char csp_noalloc_scratch[kScratchBytes];

namespace {

std::mutex g_setup_mutex;
void* g_scratch_addr[64] = {};

// Device address of the array on the current device.  The symbol's name in host
// code only stands in for it; the real address comes from the runtime, once per
// device, with that device current.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CSP_ERR_CUDA;
  if (dev < 0 || dev >= 64) return CSP_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, csp_noalloc_scratch) != cudaSuccess || p == nullptr)
      return CSP_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return CSP_OK;
}

}  // namespace

extern "C" int cascade_attn_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                    int32_t num_blocks, const int32_t* block_table,
                                    int64_t bt_row_stride, const int32_t* cu_seqlens_q,
                                    const int32_t* seqused_k, int32_t num_reqs,
                                    int32_t total_q, int32_t max_seqlen_q,
                                    int32_t max_seqlen_k, int32_t common_prefix_len,
                                    int32_t block_size, int32_t num_q_heads,
                                    int32_t num_kv_heads, int32_t head_dim,
                                    float softmax_scale, void* out, float* lse, void* stream) {
  size_t need = 0;
  int st = csp_workspace_size(num_reqs, total_q, max_seqlen_q, max_seqlen_k, common_prefix_len,
                              num_q_heads, num_kv_heads, head_dim, &need);
  if (st != CSP_OK) return st;
  if (need > kScratchBytes) return CSP_ERR_WORKSPACE;  // batch too large for the array
  void* scratch = nullptr;
  if ((st = scratch_address(&scratch)) != CSP_OK) return st;
  // The array keeps whatever the previous call left in it.  Only its 256-byte header
  // (the status word and the counters of the single-kernel schedule) must read zero
  // when a call begins; every partial result the merge reads is written earlier in
  // the same call.
  if (total_q > 0 && num_reqs > 0 &&
      cudaMemsetAsync(scratch, 0, 256, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return CSP_ERR_CUDA;
  return cascade_attn(q, k_cache, v_cache, num_blocks, block_table, bt_row_stride,
                      cu_seqlens_q, seqused_k, num_reqs, total_q, max_seqlen_q, max_seqlen_k,
                      common_prefix_len, block_size, num_q_heads, num_kv_heads, head_dim,
                      softmax_scale, out, lse, scratch, kScratchBytes, stream);
}
