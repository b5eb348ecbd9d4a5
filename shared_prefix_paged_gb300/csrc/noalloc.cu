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
#include <cuda.h>

#include <mutex>

#include "csp.h"

// Largest workspace this entry point can serve (16 MiB).  The N=64, P=4096, S=128
// decode batch with 32 query heads needs about 9.5 MiB.
static constexpr size_t kScratchBytes = static_cast<size_t>(16) << 20;

// One array per device, shared by every call of cascade_attn_noalloc on that device.
static __device__ __align__(256) unsigned char csp_noalloc_scratch[kScratchBytes];

namespace {

std::mutex g_setup_mutex;

// The array's device address on one device, valid for the context it was looked up
// in: a context torn down and created again (cudaDeviceReset, for one) reloads the
// library's device code, and the array with it, at another address.
struct ScratchEntry {
  unsigned long long ctx_id;
  void* addr;
};
ScratchEntry g_scratch[64] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Identity of the calling thread's current context (0 if it cannot be read).
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static bool looked_up = false;
  if (!looked_up) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
    looked_up = true;
  }
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx != nullptr &&
      get_id(ctx, &id) == CUDA_SUCCESS)
    return id;
  return 0;
}

// Device address of the array on the current device.  The symbol's name in host
// code only stands in for it; the real address comes from the runtime, with that
// device current, once per device and context.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CSP_ERR_CUDA;
  if (dev < 0 || dev >= 64) return CSP_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  const unsigned long long ctx = current_context_id();
  ScratchEntry& e = g_scratch[dev];
  if (e.addr == nullptr || ctx == 0 || e.ctx_id != ctx) {
    // (this lookup also makes the device's primary context current if none is)
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, csp_noalloc_scratch) != cudaSuccess || p == nullptr)
      return CSP_ERR_CUDA;
    e.addr = p;
    e.ctx_id = ctx != 0 ? ctx : current_context_id();
  }
  *out = e.addr;
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

extern "C" int csp_noalloc_status(void* stream, int32_t* status_out) {
  if (!status_out) return CSP_ERR_INVALID_ARG;
  void* scratch = nullptr;
  int st = scratch_address(&scratch);
  if (st != CSP_OK) return st;
  // the status word is the array's first 4 bytes (the workspace header's)
  return csp_workspace_status(scratch, stream, status_out);
}
