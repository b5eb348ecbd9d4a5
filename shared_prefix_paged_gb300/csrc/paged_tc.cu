// paged_tc.cu — causal attention of each request over a range of its own KV pages,
// on tcgen05 tensor cores, for requests with many query rows per KV head (prefill
// and chunked prefill): the suffix phase of cascade attention (keys [cpl, seq_len),
// "vLLM Cascade Attention：用法、场景与原理解析" §八 Step 5 Phase 2) and the standard
// path (keys [0, seq_len), §五).
//
// A CTA owns up to 256 packed rows (query, head-in-group) of one request and one KV
// head, and one key split.  Its main loop is the prefix phase's (prefix_body.cuh):
// pages by TMA into a 4-deep ring of 64-key tiles, S = Q K^T and
// O += P V on tcgen05 with TMEM accumulators, the online softmax one TMEM lane (row)
// per thread.  Here each row also stops at its causal limit: query i of a request
// with q_len queries and seq_len keys sees keys <= seq_len - q_len + i (bottom-right
// alignment; the KV includes the new tokens).  The output step:
//  * standard path with one split: bf16 out and the natural-log LSE directly;
//  * after a prefix phase, each split writes its partial slot and a third kernel
//    (merge_slots, combine.cu) merges every row once both phases are done, so the
//    suffix never waits for the prefix grid;
//  * standard path with several splits: each writes a partial slot and counts itself
//    in its row groups (token, KV head); the last split of a group merges every slot
//    of its rows (merge.cuh).
#include "merge.cuh"
#include "prefix_body.cuh"

namespace csp {
namespace {

using prefix::Layout;
using prefix::kRowsCta;
using prefix::kThreads;

// Dynamic shared memory: the data area, the barrier area, and slack to align the
// base to 1024 bytes (128-byte swizzled tiles).
template <int D, bool kF8 = false>
constexpr int kDynamic = Layout<D, kF8>::kData + prefix::kBarBytes + 1024;

// One CTA of the suffix (or standard-path) grid: request row tile bx (request
// bx / row_tiles), KV head g, key split `split`.
template <int D, bool kF8 = false>
__device__ __forceinline__ void tc_suffix_cta(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                              const CUtensorMap* tm_v, const PagedArgs& a,
                                              int bx, int g, int split, uint8_t* smem,
                                              uint64_t* bars) {
  using L = Layout<D, kF8>;
  constexpr int kNThreads = kF8 ? prefix::kThreadsF8 : kThreads;
  const int r = bx / a.row_tiles;
  const int rt = bx % a.row_tiles;
  const int q0 = __ldg(a.cu_seqlens_q + r);
  const int q_len = __ldg(a.cu_seqlens_q + r + 1) - q0;
  const int seq = __ldg(a.seq_lens + r);
  const int rows_total = q_len * a.group;
  const int prow0 = rt * kRowsCta;
  if (prow0 >= rows_total) return;  // the request has fewer row tiles
  const int rows_here = min(kRowsCta, rows_total - prow0);
  const int gshift = __ffs(a.group) - 1;  // group is a power of two

  // keys of this split, clipped by the causal limit of the CTA's last row
  const int last_query = (prow0 + rows_here - 1) >> gshift;
  const int kbeg =
      (a.key_start_of != nullptr ? __ldg(a.key_start_of + r) : a.key_start) + split * a.split_keys;
  int kend = min(kbeg + a.split_keys, seq);
  kend = min(kend, seq - q_len + last_query + 1);
  const int ntiles = kend > kbeg ? (kend - kbeg + prefix::kKeysN - 1) / prefix::kKeysN : 0;

  // what the main loop reads besides the geometry: sizes, scale, the status word
  PrefixArgs pa;
  pa.k = a.k;
  pa.v = a.v;
  pa.block_table = a.block_table;
  pa.total_q = a.total_q;
  pa.num_q_heads = a.num_q_heads;
  pa.num_kv_heads = a.num_kv_heads;
  pa.group = a.group;
  pa.cpl = 0;
  pa.pairs = 0;
  pa.n_splits = 0;
  pa.tiles_per_split = 0;
  pa.scale_log2 = a.scale_log2;
  pa.part_o = nullptr;
  pa.part_lse = nullptr;
  pa.lse_stride = 0;
  pa.status = a.status;
  pa.v_scale = a.v_scale;
  prefix::RangeGeom geo;
  geo.bt = a.block_table + static_cast<int64_t>(r) * a.bt_stride;
  geo.key0 = kbeg;
  geo.key_end = max(kend, kbeg);
  geo.tok0 = q0;
  geo.prow0 = prow0;
  geo.rows_total = rows_total;
  geo.causal_base = seq - q_len;
  prefix::prefix_range<D, true, kF8>(tm_q, tm_k, tm_v, pa, geo, g, split, 0, ntiles, smem, bars);

  // 256 normalised rows (bf16) and their log2-sum-exp are staged and visible
  const __nv_bfloat16* stage = reinterpret_cast<const __nv_bfloat16*>(smem);
  const float* s_lse = reinterpret_cast<const float*>(smem + L::kLse);
  constexpr int kChunks = D / 8;
  constexpr float kLn2 = 0.69314718055994531f;
  const bool partial = a.part_o != nullptr;
  auto out_row = [&](int rr) {
    const int rho = prow0 + rr;
    return static_cast<int64_t>(q0 + (rho >> gshift)) * a.num_q_heads + g * a.group +
           (rho & (a.group - 1));
  };
  // the final rows (standard path, one split) or this split's partial slot
  for (int it = threadIdx.x; it < rows_here * kChunks; it += kNThreads) {
    const int rr = it / kChunks, c = it % kChunks;
    const int64_t orow = out_row(rr);
    const uint4 v = *reinterpret_cast<const uint4*>(stage + rr * L::kStageRow + c * 8);
    if (partial) {
      const int64_t prow =
          static_cast<int64_t>(a.n_prefix + split) * a.total_q * a.num_q_heads + orow;
      *reinterpret_cast<uint4*>(a.part_o + prow * D + c * 8) = v;
      if (c == 0) a.part_lse[prow] = s_lse[rr];
    } else {
      *reinterpret_cast<uint4*>(a.out + orow * D + c * 8) = v;
      if (c == 0 && a.lse != nullptr) a.lse[orow] = s_lse[rr] * kLn2;
    }
  }
  if (!partial || a.counters == nullptr) return;  // no counters: merge_slots follows

  // count this split in the row groups (tokens) it covered; the last split of a group
  // merges every slot of its rows
  MergeArgs m;
  m.part_o = a.part_o;
  m.part_lse = a.part_lse;
  m.counters = a.counters;
  m.n_parts = a.n_prefix + a.n_splits;
  m.n_count = a.n_splits + a.prefix_contributors;
  m.rows = a.total_q * a.num_q_heads;
  m.num_q_heads = a.num_q_heads;
  m.num_kv_heads = a.num_kv_heads;
  m.group = a.group;
  m.out = a.out;
  m.lse = a.lse;
  // shared scratch past the staged rows: the last-contributor flags, then the weights
  int* s_last = reinterpret_cast<int*>(smem + kRowsCta * L::kStageRow * 2);
  float* s_w = reinterpret_cast<float*>(s_last + kRowsCta + 1);
  const int tok_first = prow0 >> gshift;
  const int n_tok = ((prow0 + rows_here - 1) >> gshift) - tok_first + 1;
  count_and_merge_block<D>(m, q0 + tok_first, n_tok, g, rows_here, out_row,
                           [&](int rr) { return ((prow0 + rr) >> gshift) - tok_first; }, s_last,
                           s_w);
}

template <int D, bool kF8>
__global__ void __launch_bounds__(kF8 ? prefix::kThreadsF8 : kThreads, 1)
    paged_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const PagedArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Layout<D, kF8>::kData);
  tc_suffix_cta<D, kF8>(&tm_q, &tm_k, &tm_v, a, blockIdx.x, blockIdx.y, blockIdx.z, smem,
                        bars);
}

// The whole cascade step in one launch (prefill-shaped batches): CTAs [0, n_pre) are
// the prefix phase's (KV head, 256-row block, key range) CTAs, the rest the suffix
// grid's (request row tile, KV head, key split) CTAs in the order the suffix kernel
// numbers them.  Every CTA writes its partial slot and counts itself in the row
// groups (token, KV head) it covered, prefix ranges and suffix splits in the same
// counters; a group's last contributor merges every slot of its rows (merge.cuh).
// So no phase waits for the other and no kernel follows: the prefix CTAs, numbered
// first, start first and the suffix fills the SMs they leave free.
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    cascade_fused_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const PrefixArgs pa,
                         const PagedArgs ga, int n_pre) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kData);
  const int b = static_cast<int>(blockIdx.x);
  if (b >= n_pre) {
    const int s = b - n_pre;
    const int nx = ga.num_reqs * ga.row_tiles;
    tc_suffix_cta<D>(&tm_q, &tm_k, &tm_v, ga, s % nx, (s / nx) % ga.num_kv_heads,
                     s / (nx * ga.num_kv_heads), smem, bars);
    return;
  }
  // a prefix range: its slot `split`, written by the body
  const int split = b % pa.n_splits;
  const int pair = (b / pa.n_splits) % pa.pairs;
  const int kvh = b / (pa.n_splits * pa.pairs);
  const int key_tiles = (pa.cpl + prefix::kKeysN - 1) / prefix::kKeysN;
  const int t_first = min(split * pa.tiles_per_split, key_tiles);
  const int t_last = min(t_first + pa.tiles_per_split, key_tiles);
  prefix::prefix_range<D>(&tm_q, &tm_k, &tm_v, pa, prefix::prefix_geom(pa, pair), kvh, split,
                          t_first, t_last, smem, bars);
  // count it in the row groups of its 256 rows; the last contributor merges
  const int gshift = __ffs(pa.group) - 1;
  const int prow0 = pair * kRowsCta;
  const int rows_here = min(kRowsCta, pa.total_q * pa.group - prow0);
  if (rows_here <= 0) return;
  MergeArgs m;
  m.part_o = ga.part_o;
  m.part_lse = ga.part_lse;
  m.counters = ga.counters;
  m.n_parts = ga.n_prefix + ga.n_splits;
  m.n_count = ga.n_splits + ga.prefix_contributors;
  m.rows = ga.total_q * ga.num_q_heads;
  m.num_q_heads = ga.num_q_heads;
  m.num_kv_heads = ga.num_kv_heads;
  m.group = ga.group;
  m.out = ga.out;
  m.lse = ga.lse;
  int* s_last = reinterpret_cast<int*>(smem + kRowsCta * L::kStageRow * 2);
  float* s_w = reinterpret_cast<float*>(s_last + kRowsCta + 1);
  const int tok_first = prow0 >> gshift;
  const int n_tok = ((prow0 + rows_here - 1) >> gshift) - tok_first + 1;
  auto out_row = [&](int rr) {
    const int rho = prow0 + rr;
    return static_cast<int64_t>(rho >> gshift) * pa.num_q_heads + kvh * pa.group +
           (rho & (pa.group - 1));
  };
  count_and_merge_block<D>(m, tok_first, n_tok, kvh, rows_here, out_row,
                           [&](int rr) { return ((prow0 + rr) >> gshift) - tok_first; }, s_last,
                           s_w);
}

template <int D>
cudaError_t launch_fused_t(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                           const CUtensorMap& tm_v, const PrefixArgs& pa, const PagedArgs& ga,
                           int n_pre, int n_suf, cudaStream_t stream) {
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = set_smem_once(cascade_fused_kernel<D>, kDynamic<D>, attr_done);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_pre + n_suf);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kDynamic<D>;
  cfg.stream = stream;
  cfg.numAttrs = 0;
  return cudaLaunchKernelEx(&cfg, cascade_fused_kernel<D>, tm_q, tm_k, tm_v, pa, ga, n_pre);
}

template <int D, bool kF8>
cudaError_t launch_tc_t(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                        const CUtensorMap& tm_v, const PagedArgs& a, bool after_prefix,
                        cudaStream_t stream) {
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = set_smem_once(paged_tc_kernel<D, kF8>, kDynamic<D, kF8>, attr_done);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.num_reqs * a.row_tiles, a.num_kv_heads, a.n_splits);
  cfg.blockDim = dim3(kF8 ? prefix::kThreadsF8 : kThreads);
  cfg.dynamicSmemBytes = kDynamic<D, kF8>;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  // behind this call's prefix kernel: start on the SMs it leaves free; the merge
  // waits for the prefix grid
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = after_prefix ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, paged_tc_kernel<D, kF8>, tm_q, tm_k, tm_v, a);
}

}  // namespace

cudaError_t launch_cascade_fused(int head_dim, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                 const CUtensorMap& tm_v, const PrefixArgs& pa,
                                 const PagedArgs& ga, cudaStream_t stream) {
  const int n_pre = pa.n_splits * pa.pairs * pa.num_kv_heads;
  const int n_suf = ga.num_reqs * ga.row_tiles * ga.num_kv_heads * ga.n_splits;
  if (head_dim == 64) return launch_fused_t<64>(tm_q, tm_k, tm_v, pa, ga, n_pre, n_suf, stream);
  return launch_fused_t<128>(tm_q, tm_k, tm_v, pa, ga, n_pre, n_suf, stream);
}

cudaError_t launch_paged_tc(int head_dim, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                            const CUtensorMap& tm_v, const PagedArgs& a, bool after_prefix,
                            cudaStream_t stream) {
  if (head_dim == 64) return launch_tc_t<64, false>(tm_q, tm_k, tm_v, a, after_prefix, stream);
  return launch_tc_t<128, false>(tm_q, tm_k, tm_v, a, after_prefix, stream);
}

cudaError_t launch_paged_tc_f8(int head_dim, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                               const CUtensorMap& tm_v, const PagedArgs& a, bool after_prefix,
                               cudaStream_t stream) {
  if (head_dim == 64) return launch_tc_t<64, true>(tm_q, tm_k, tm_v, a, after_prefix, stream);
  return launch_tc_t<128, true>(tm_q, tm_k, tm_v, a, after_prefix, stream);
}

}  // namespace csp
