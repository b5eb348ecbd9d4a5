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
// no causal mask.  Rows are (token, head-in-group) pairs of one KV head; a CTA owns
// 256 of them (two 128-row M tiles).  The prefix's 64-key tiles are cut into
// n_splits ranges, one CTA and one workspace slot each; the suffix kernel merges
// those slots with its own partials (merge.cuh).
struct PrefixArgs {
  const __nv_bfloat16* k;      // K cache [num_blocks][16][num_kv_heads][D]
  const __nv_bfloat16* v;      // V cache, same layout
  const int32_t* block_table;  // row 0: the shared pages
  int total_q;
  int num_q_heads;
  int num_kv_heads;
  int group;             // num_q_heads / num_kv_heads
  int cpl;               // common prefix length, multiple of 16
  int pairs;             // ceil(total_q * group / 256): 256-row units per KV head
  int n_splits;          // key ranges per (unit, KV head)
  int tiles_per_split;   // 64-key tiles per range
  float scale_log2;      // softmax_scale * log2(e)
  __nv_bfloat16* part_o; // [n_parts][total_q][num_q_heads][D], normalised; slots [0, n_splits)
  float* part_lse;       // [n_parts][lse_stride], log2 domain (row t * num_q_heads + h)
  int64_t lse_stride;    // floats per LSE slot, >= total_q * num_q_heads
  int* status;           // workspace status word
  // A segment of a multi-level cascade (cascade_attn_levels): the rows are the query
  // tokens [tok0, tok0 + total_q) of the batch (block_table then points at the row of
  // the segment's first request), the keys [key_lo, cpl), and range s writes slot
  // slot_base + s of slots that hold rows_all rows each.  The defaults are the prefix
  // phase of a two-level cascade.
  int key_lo = 0;
  int tok0 = 0;
  int slot_base = 0;
  int64_t rows_all = 0;  // 0: total_q * num_q_heads
  // An FP8 (E4M3) KV cache: the V scale, applied to the normalised rows (the K scale is
  // folded into scale_log2 by the host).
  float v_scale = 1.f;
};

// The segments of a multi-level cascade in one grid (prefix_attn.cu): segment i owns
// CTAs [cta0, cta0 + Hkv * pairs * splits) and runs the prefix body over its query
// rows [tok0, tok0 + tokens) and keys [key_lo, key_hi) of block-table row bt_row,
// writing slots slot_base .. slot_base + splits - 1.  Passed by value (kernel
// parameter space), at most kMaxSegmentsPerLaunch segments.
constexpr int kMaxSegmentsPerLaunch = 48;
struct SegmentDesc {
  int cta0;
  int bt_row;
  int key_lo, key_hi;
  int tok0, tokens;
  int slot_base;
  int splits, tiles_per_split, pairs;
};
struct SegmentTable {
  int n;
  int64_t bt_stride;
  SegmentDesc s[kMaxSegmentsPerLaunch];
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
  __nv_bfloat16* part_o; // partial mode: [n_prefix + n_splits][total_q][Hq][D] (own slot: n_prefix + split)
  float* part_lse;       //               [n_prefix + n_splits][total_q][Hq], log2 domain
  int n_prefix;          //               prefix slots before the suffix ones (0: none)
  int* counters;         //               row-group counters (merge.cuh); the tcgen05 variant
                         //               with none leaves every merge to merge_slots
  __nv_bfloat16* out;    // final output: direct mode (part_o == nullptr) or last contributor
  float* lse;            // natural-log LSE or nullptr
  int* status;           // workspace status word (bounded waits of the tcgen05 variant)
  const int32_t* key_start_of = nullptr;  // per request (device), in place of key_start
                                          // (the suffixes of a multi-level cascade)
  int prefix_contributors = 0;  // prefix ranges counted in the same row-group counters
                                // (the fused launch)
  // The warp-MMA kernel with 2..8 key splits: the splits of a row tile run as one
  // thread-block cluster and merge through distributed shared memory (no counters).
  bool cluster_splits = false;
  // write every split's partial slot and merge nothing (a merge kernel follows)
  bool partials_only = false;
  // An FP8 (E4M3) KV cache (the *_f8 launchers): q then points at an f16 copy of the
  // queries, k and v at the E4M3 caches, and the V scale multiplies the normalised
  // rows (the K scale is folded into scale_log2).
  float v_scale = 1.f;
};

// Single-kernel cascade step for decode-like batches (decode_cascade.cu): at most 16
// packed rows (query, head-in-group) per request and KV head.  CTAs [0, prefix_ctas)
// run one prefix range each (pre.n_splits ranges per (KV head, 256-row block), range
// s = 64-key tiles [s*key_tiles/n_splits, (s+1)*key_tiles/n_splits), slot s), then
// stream prefix_units suffix units; the other CTAs share the remaining suffix units
// (request, KV head).  Suffix partials go to slot n_splits.  After a grid-wide barrier
// every CTA merges an equal share of the rows from slots [0, n_splits].
// Most partial results per row (the prefix ranges + the suffix): one merge reads at
// most 16 slots.
constexpr int kDecodeMaxParts = 16;

struct DecodeArgs {
  PrefixArgs pre;            // prefix phase; part_o / part_lse hold n_splits + 1 slots
  const __nv_bfloat16* q;    // [total_q][num_q_heads][D]
  const __nv_bfloat16* k;    // [num_blocks][16][num_kv_heads][D]
  const __nv_bfloat16* v;
  const int32_t* block_table;
  int64_t bt_stride;
  const int32_t* cu_seqlens_q;
  const int32_t* seq_lens;
  int num_reqs;
  int prefix_ctas;           // num_kv_heads * pre.pairs * pre.n_splits (<= grid)
  int prefix_units;          // suffix units each prefix CTA streams after its range
  int merge_rows;            // rows per merge chunk (the merge tensor maps' box)
  int unit_groups;           // 2: every suffix unit is one item (<= 128 keys) and two groups
                             // of four warps take alternate units; 1: all eight warps
  int key_tiles;             // ceil(cpl / 64)
  unsigned long long* bar_count;  // grid-barrier arrivals: a multiple of the grid at launch
                                  // (zero at first); each call adds the grid size
  __nv_bfloat16* out;
  float* lse;                // natural-log LSE or nullptr
  const int32_t* cpl_dev;    // null, or the prefix length in device memory (the launch
                             // plan was made for pre.cpl, an upper bound of it)
  int max_seqlen_k;          // the longest request's KV length
};

// grid <= the number of co-resident CTAs (one per SM); launched cooperatively.
// tm_po / tm_pl: the workspace slots as bf16 [n_splits + 1][rows][D] and fp32
// [n_splits + 1][pre.lse_stride], boxes of merge_rows rows (and of
// (merge_rows + 6) & ~3 LSEs).
// tm_k / tm_v: the K / V cache as pages of one KV head with both feature halves
// (boxes {64, 16, D / 64, 1} of {64, tokens, D / 64, Hkv}); tm_kp: K as {D, Hkv,
// tokens} with boxes {64, 1, 16}, for the prefix ranges.
cudaError_t launch_decode(int head_dim, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                          const CUtensorMap& tm_v, const CUtensorMap& tm_kp,
                          const CUtensorMap& tm_po,
                          const CUtensorMap& tm_pl, const DecodeArgs& a, int grid,
                          cudaStream_t stream);

cudaError_t launch_prefix(int head_dim, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                          const CUtensorMap& tm_v, const PrefixArgs& a, cudaStream_t stream);

// base: the fields every segment shares (caches, block_table row 0, heads, scale,
// slots and their strides, status); grid = the table's CTAs in all.
cudaError_t launch_prefix_segments(int head_dim, const CUtensorMap& tm_q,
                                   const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                   const PrefixArgs& base, const SegmentTable& t, int grid,
                                   cudaStream_t stream);

// after_prefix: launched right behind this call's prefix kernel on the same stream
// (programmatic dependent launch, so it runs concurrently with it).
cudaError_t launch_paged(int head_dim, const PagedArgs& a, bool after_prefix,
                         cudaStream_t stream);

// The same computation on tcgen05 for units of many rows (paged_tc.cu): one CTA per
// (request, KV head, 256-row tile, key split); a.row_tiles counts 256-row tiles.
// tm_q: q as bf16 [total_q][num_q_heads][D], boxes of 64 features x group heads x
// 128 / group tokens; tm_k: K as {D, Hkv, tokens}, boxes {64, 1, 16}; tm_v: V as
// {64, tokens, D / 64, Hkv}, boxes {64, 16, D / 64, 1}.
cudaError_t launch_paged_tc(int head_dim, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                            const CUtensorMap& tm_v, const PagedArgs& a, bool after_prefix,
                            cudaStream_t stream);

// The fused cascade step (paged_tc.cu): the prefix grid of `pa` and the tcgen05
// suffix grid of `ga` in one launch, merged by each row group's last contributor
// (ga.counters zero at the start, ga.prefix_contributors = pa.n_splits, ga.n_prefix =
// the prefix slots).  Maps as for launch_paged_tc.
cudaError_t launch_cascade_fused(int head_dim, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                 const CUtensorMap& tm_v, const PrefixArgs& pa,
                                 const PagedArgs& ga, cudaStream_t stream);

// merge_attn_states over n_parts slots of every row (rows = total_q * num_q_heads):
// part_o [n_parts][rows][D] bf16 normalised, part_lse [n_parts][rows] log2 domain ->
// bf16 out and the natural-log LSE (lse may be null).
cudaError_t launch_merge_slots(int head_dim, const __nv_bfloat16* part_o, const float* part_lse,
                               int n_parts, int64_t rows, __nv_bfloat16* out, float* lse,
                               cudaStream_t stream);

cudaError_t launch_merge_states(__nv_bfloat16* out, float* out_lse, const void* o1,
                                const float* l1, const void* o2, const float* l2, int rows,
                                int head_dim, bool f32_partials, cudaStream_t stream);

// The device planner (plan_device.cu): plan[0..3] = the prefix length to use (0 when
// cascade is not taken), use_cascade, the common prefix length, status.
cudaError_t launch_plan_device(const int32_t* block_table, int64_t bt_row_stride, int num_reqs,
                               const int32_t* seq_lens, const int32_t* computed, int block_size,
                               int mode, int32_t* plan, cudaStream_t stream);

// n floats at p set to v.
cudaError_t launch_fill_f32(float* p, int64_t n, float v, cudaStream_t stream);

// n bf16 values (a multiple of 8, 16-byte aligned) -> f16.
cudaError_t launch_bf16_to_f16(const void* in, void* out, int64_t n, cudaStream_t stream);

// The FP8 (E4M3) KV cache variants: tm_k and tm_v map the byte caches as {D, Hkv,
// tokens} with boxes {D, 1, 16} (no swizzle); tm_q and the paged kernels' q the f16
// queries; PrefixArgs / PagedArgs v_scale the V scale (the K scale is in scale_log2).
cudaError_t launch_prefix_f8(int head_dim, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                             const CUtensorMap& tm_v, const PrefixArgs& a, cudaStream_t stream);
cudaError_t launch_paged_f8(int head_dim, const PagedArgs& a, bool after_prefix,
                            cudaStream_t stream);
cudaError_t launch_paged_tc_f8(int head_dim, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                               const CUtensorMap& tm_v, const PagedArgs& a, bool after_prefix,
                               cudaStream_t stream);

// Attention sinks applied to a finished result (rows = tokens x heads, natural-log
// lse updated in place); head_dim / 8 divides 32.
cudaError_t launch_apply_sinks(__nv_bfloat16* out, float* lse, const float* sinks, int rows,
                               int heads, int head_dim, cudaStream_t stream);

}  // namespace csp
