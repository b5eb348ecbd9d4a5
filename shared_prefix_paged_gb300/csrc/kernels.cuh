// kernels.cuh — host-side launch interface between the C ABI (api.cu) and the
// kernels.  Plain structs of pointers and sizes; no torch types.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace csp {

// Prefix phase ("vLLM Cascade Attention：用法、场景与原理解析" §八 Step 5, Phase 1):
// every query row of the batch against KV positions [0, cpl) of block_table row 0,
// no causal mask.  Rows are (token, head-in-group) pairs of one KV head packed into
// 128-row tiles; each CTA takes one tile, one KV head and a range of 128-key tiles
// and writes a normalised fp32 partial and its log2-sum-exp.
struct PrefixArgs {
  const int32_t* block_table;  // row 0: the shared pages
  int total_q;
  int num_q_heads;
  int num_kv_heads;
  int group;             // num_q_heads / num_kv_heads
  int cpl;               // common prefix length, multiple of 16
  int m_tiles;           // ceil(total_q * group / 128)
  int n_splits;          // key splits per (tile, KV head)
  int tiles_per_split;   // 128-key tiles per split
  float scale_log2;      // softmax_scale * log2(e)
  float* part_o;         // [n_splits][total_q][num_q_heads][D]
  float* part_lse;       // [n_splits][total_q][num_q_heads], log2 domain
  int* status;           // workspace status word
};

// Paged attention over a key range of each request (the suffix phase with
// key_start = cpl, §八 Step 5 Phase 2; the standard path with key_start = 0, §五).
struct PagedArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const int32_t* block_table;
  int64_t bt_stride;
  const int32_t* cu_seqlens_q;
  const int32_t* seq_lens;
  int num_reqs;
  int total_q;
  int num_q_heads;
  int num_kv_heads;
  int group;
  int key_start;         // first key position of the range
  int split_keys;        // keys per split, multiple of 64
  int n_splits;
  int row_tiles;         // CTAs along the packed rows of one request
  float scale_log2;
  float* part_o;         // partial mode: [slots][total_q][Hq][D] (slot = part_slot0 + split)
  float* part_lse;       //               [slots][total_q][Hq], log2 domain
  int part_slot0;
  __nv_bfloat16* out;    // direct mode (part_o == nullptr): final output
  float* lse;            //               natural-log LSE or nullptr
};

// Combine n_parts partial results per row into the final bf16 output and LSE.
struct CombineArgs {
  const float* part_o;
  const float* part_lse;
  int n_parts;
  int rows;              // total_q * num_q_heads
  __nv_bfloat16* out;
  float* lse;            // natural log, or nullptr
};

cudaError_t launch_prefix(int head_dim, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                          const CUtensorMap& tm_v, const PrefixArgs& a, cudaStream_t stream);
size_t prefix_smem_bytes(int head_dim);

cudaError_t launch_paged(int head_dim, bool decode, const PagedArgs& a, cudaStream_t stream);

cudaError_t launch_combine(int head_dim, const CombineArgs& a, cudaStream_t stream);

cudaError_t launch_merge_states(__nv_bfloat16* out, float* out_lse, const void* o1,
                                const float* l1, const void* o2, const float* l2, int rows,
                                int head_dim, bool f32_partials, cudaStream_t stream);

}  // namespace csp
