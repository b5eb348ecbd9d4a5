// prefix_attn.cu — the standalone prefix-phase kernel of cascade attention
// ("vLLM Cascade Attention：用法、场景与原理解析" §八 Step 5 Phase 1): one CTA per
// (KV head, 256-row block, key range); the work of a CTA is prefix_range
// (prefix_body.cuh).  The paged kernel that follows it on the stream merges the
// slots it writes.
#include "prefix_body.cuh"

namespace csp {
namespace {

using prefix::Layout;
using prefix::kThreads;

// Dynamic shared memory: the data area, the barrier area, and slack to align the
// base to 1024 bytes (128-byte swizzled TMA tiles).
template <int D>
constexpr int kDynamic = Layout<D>::kData + prefix::kBarBytes + 1024;

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefix_attn_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const PrefixArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Layout<D>::kData);
  // the suffix kernel (launched as a programmatic dependent) may start now; it reads
  // this grid's partials only after waiting for the grid to complete
  grid_launch_dependents();
  const int split = blockIdx.x % a.n_splits;
  const int pair = (blockIdx.x / a.n_splits) % a.pairs;
  const int kvh = blockIdx.x / (a.n_splits * a.pairs);
  const int key_tiles = (a.cpl - a.key_lo + prefix::kKeysN - 1) / prefix::kKeysN;
  const int t_first = min(split * a.tiles_per_split, key_tiles);
  const int t_last = min(t_first + a.tiles_per_split, key_tiles);
  prefix::prefix_range<D>(&tm_q, &tm_k, &tm_v, a, prefix::prefix_geom(a, pair), kvh, split,
                          t_first, t_last, smem, bars);
}

template <int D>
cudaLaunchConfig_t prefix_config(const PrefixArgs& a, cudaStream_t stream,
                                 cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_splits * a.pairs * a.num_kv_heads);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kDynamic<D>;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 0;
  return cfg;
}

template <int D>
cudaError_t prepare() {
  static std::atomic<uint64_t> attr_done{0};
  return set_smem_once(prefix_attn_kernel<D>, kDynamic<D>, attr_done);
}

template <int D>
cudaError_t launch_prefix_d(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                            const CUtensorMap& tm_v, const PrefixArgs& a, cudaStream_t stream) {
  cudaError_t e = prepare<D>();
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = prefix_config<D>(a, stream, attr);
  return cudaLaunchKernelEx(&cfg, prefix_attn_kernel<D>, tm_q, tm_k, tm_v, a);
}

}  // namespace

cudaError_t launch_prefix(int head_dim, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                          const CUtensorMap& tm_v, const PrefixArgs& a, cudaStream_t stream) {
  if (head_dim == 64) return launch_prefix_d<64>(tm_q, tm_k, tm_v, a, stream);
  return launch_prefix_d<128>(tm_q, tm_k, tm_v, a, stream);
}

}  // namespace csp
