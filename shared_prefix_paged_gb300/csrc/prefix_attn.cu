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
template <int D, bool kF8 = false>
constexpr int kDynamic = Layout<D, kF8>::kData + prefix::kBarBytes + 1024;

// kF8: an E4M3 KV cache (tm_k and tm_v its byte maps, tm_q the f16 queries), with two
// more warps that widen each tile.
template <int D, bool kF8>
__global__ void __launch_bounds__(kF8 ? prefix::kThreadsF8 : kThreads, 1)
    prefix_attn_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const PrefixArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Layout<D, kF8>::kData);
  // the suffix kernel (launched as a programmatic dependent) may start now; it reads
  // this grid's partials only after waiting for the grid to complete
  grid_launch_dependents();
  const int split = blockIdx.x % a.n_splits;
  const int pair = (blockIdx.x / a.n_splits) % a.pairs;
  const int kvh = blockIdx.x / (a.n_splits * a.pairs);
  const int key_tiles = (a.cpl - a.key_lo + prefix::kKeysN - 1) / prefix::kKeysN;
  const int t_first = min(split * a.tiles_per_split, key_tiles);
  const int t_last = min(t_first + a.tiles_per_split, key_tiles);
  prefix::prefix_range<D, false, kF8>(&tm_q, &tm_k, &tm_v, a, prefix::prefix_geom(a, pair),
                                      kvh, split, t_first, t_last, smem, bars);
}

// Every segment of a multi-level cascade in one grid: a CTA finds its segment in the
// table (the last one whose first CTA is at or before it; uniform across the CTA, read
// from parameter space) and runs the same body over the segment's rows, keys and slots.
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefix_segments_kernel(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v, const PrefixArgs base,
                           const __grid_constant__ SegmentTable t) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Layout<D>::kData);
  grid_launch_dependents();
  const int cta = static_cast<int>(blockIdx.x);
  int i = 0;
  for (int j = 1; j < t.n; ++j)
    if (t.s[j].cta0 <= cta) i = j;
  const SegmentDesc sd = t.s[i];
  PrefixArgs a = base;
  a.block_table = base.block_table + static_cast<int64_t>(sd.bt_row) * t.bt_stride;
  a.total_q = sd.tokens;
  a.key_lo = sd.key_lo;
  a.cpl = sd.key_hi;
  a.tok0 = sd.tok0;
  a.slot_base = sd.slot_base;
  a.n_splits = sd.splits;
  a.tiles_per_split = sd.tiles_per_split;
  a.pairs = sd.pairs;
  const int local = cta - sd.cta0;
  const int split = local % sd.splits;
  const int pair = (local / sd.splits) % sd.pairs;
  const int kvh = local / (sd.splits * sd.pairs);
  const int key_tiles = (sd.key_hi - sd.key_lo + prefix::kKeysN - 1) / prefix::kKeysN;
  const int t_first = min(split * sd.tiles_per_split, key_tiles);
  const int t_last = min(t_first + sd.tiles_per_split, key_tiles);
  prefix::prefix_range<D>(&tm_q, &tm_k, &tm_v, a, prefix::prefix_geom(a, pair), kvh, split,
                          t_first, t_last, smem, bars);
}

template <int D, bool kF8>
cudaLaunchConfig_t prefix_config(const PrefixArgs& a, cudaStream_t stream,
                                 cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_splits * a.pairs * a.num_kv_heads);
  cfg.blockDim = dim3(kF8 ? prefix::kThreadsF8 : kThreads);
  cfg.dynamicSmemBytes = kDynamic<D, kF8>;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 0;
  return cfg;
}

template <int D, bool kF8>
cudaError_t prepare() {
  static std::atomic<uint64_t> attr_done{0};
  return set_smem_once(prefix_attn_kernel<D, kF8>, kDynamic<D, kF8>, attr_done);
}

template <int D, bool kF8>
cudaError_t launch_prefix_d(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                            const CUtensorMap& tm_v, const PrefixArgs& a, cudaStream_t stream) {
  cudaError_t e = prepare<D, kF8>();
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = prefix_config<D, kF8>(a, stream, attr);
  return cudaLaunchKernelEx(&cfg, prefix_attn_kernel<D, kF8>, tm_q, tm_k, tm_v, a);
}

template <int D>
cudaError_t launch_segments_d(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                              const CUtensorMap& tm_v, const PrefixArgs& base,
                              const SegmentTable& t, int grid, cudaStream_t stream) {
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = set_smem_once(prefix_segments_kernel<D>, kDynamic<D>, attr_done);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kDynamic<D>;
  cfg.stream = stream;
  cfg.numAttrs = 0;
  return cudaLaunchKernelEx(&cfg, prefix_segments_kernel<D>, tm_q, tm_k, tm_v, base, t);
}

}  // namespace

cudaError_t launch_prefix_segments(int head_dim, const CUtensorMap& tm_q,
                                   const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                   const PrefixArgs& base, const SegmentTable& t, int grid,
                                   cudaStream_t stream) {
  if (head_dim == 64) return launch_segments_d<64>(tm_q, tm_k, tm_v, base, t, grid, stream);
  return launch_segments_d<128>(tm_q, tm_k, tm_v, base, t, grid, stream);
}

cudaError_t launch_prefix(int head_dim, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                          const CUtensorMap& tm_v, const PrefixArgs& a, cudaStream_t stream) {
  if (head_dim == 64) return launch_prefix_d<64, false>(tm_q, tm_k, tm_v, a, stream);
  return launch_prefix_d<128, false>(tm_q, tm_k, tm_v, a, stream);
}

cudaError_t launch_prefix_f8(int head_dim, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                             const CUtensorMap& tm_v, const PrefixArgs& a, cudaStream_t stream) {
  if (head_dim == 64) return launch_prefix_d<64, true>(tm_q, tm_k, tm_v, a, stream);
  return launch_prefix_d<128, true>(tm_q, tm_k, tm_v, a, stream);
}

}  // namespace csp
