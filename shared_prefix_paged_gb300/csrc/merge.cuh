// merge.cuh — in-kernel LSE merge of the partial results of a row group.
//
// A row group is one query token and one KV head: the `group` query heads that read
// that KV head.  The prefix phase leaves one partial per key range in workspace
// slots [0, n_prefix); every key split of the suffix phase (or of the standard
// path) leaves one in the slots after them.  A partial is the normalised output in
// bf16 plus its log2-sum-exp in fp32.  The suffix kernel waits for the prefix grid
// (programmatic dependent launch) before it merges, and its splits count themselves
// in the group's counter: the last one merges every slot ("vLLM Cascade Attention：
// 用法、场景与原理解析" §一 and §八 Step 5, merge_attn_states: out = sum_p e^(l_p - m)
// o_p / sum_p e^(l_p - m), lse = m + ln sum_p e^(l_p - m)) and writes bf16 out and
// the natural-log LSE.  The host clears the counters before each call.
#pragma once

#include "common.cuh"

namespace csp {

// Most partial results one row group can have (one lane each in the merge).
constexpr int kMaxParts = 32;

struct MergeArgs {
  const __nv_bfloat16* part_o;  // [n_parts][rows][D], normalised
  const float* part_lse;        // [n_parts][rows], log2 domain; -inf: empty
  int* counters;                // [total_q * num_kv_heads], zero at the start of the call
  int n_parts;                  // slots merged per row (<= kMaxParts)
  int n_count;                  // contributors counted per row group (suffix splits)
  int rows;                     // total_q * num_q_heads
  int num_q_heads;
  int num_kv_heads;
  int group;
  __nv_bfloat16* out;           // [total_q][num_q_heads][D]
  float* lse;                   // [total_q][num_q_heads] natural log, or nullptr
};

// Add 1 with acquire-release semantics at GPU scope: the partial results this CTA
// wrote before (ordered by a CTA barrier) are published, and those the other
// contributors published become visible to this CTA.
__device__ __forceinline__ int atomic_add_acq_rel_gpu(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
               : "memory");
  return old;
}

__device__ __forceinline__ float4 load_bf16x4_cg(const __nv_bfloat16* p) {
  const uint2 u = __ldcg(reinterpret_cast<const uint2*>(p));
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

__device__ __forceinline__ void store_bf16x4(__nv_bfloat16* p, float4 v) {
  *reinterpret_cast<uint2*>(p) = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
}

// Merge one output row with one warp.  Slots [0, n_parts) come from the workspace;
// `own` / `own_lse` (when own_lse is not -inf or has_own is set) is one more partial
// held in registers, features [4 lane, 4 lane + 4).  Lane p holds slot p's weight,
// then lane c accumulates features [4c, 4c+4) over all partials.
template <int D>
__device__ __forceinline__ void merge_row_warp(const MergeArgs& m, int64_t row, int lane,
                                               bool has_own, float4 own, float own_lse) {
  const float lp = lane < m.n_parts
                       ? __ldcg(m.part_lse + static_cast<int64_t>(lane) * m.rows + row)
                       : -INFINITY;
  float mx = fmaxf(lp, has_own ? own_lse : -INFINITY);
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, s));
  const float w = (mx == -INFINITY || lp == -INFINITY) ? 0.f : fast_exp2(lp - mx);
  const float w_own =
      (!has_own || mx == -INFINITY || own_lse == -INFINITY) ? 0.f : fast_exp2(own_lse - mx);
  float wsum = w;
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, s);
  wsum += w_own;
  const float inv = !(wsum <= 0.f) ? 1.f / wsum : 0.f;  // a NaN sum propagates
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (w_own != 0.f) {
    const float wo = w_own * inv;
    acc = make_float4(wo * own.x, wo * own.y, wo * own.z, wo * own.w);
  }
  // eight slots at a time: their loads are independent and go out together; an
  // empty slot (weight 0) is skipped by a select, so whatever it holds never mixes in
  const __nv_bfloat16* base = m.part_o + row * D + lane * 4;
  const int64_t slot_stride = static_cast<int64_t>(m.rows) * D;
  for (int p0 = 0; p0 < m.n_parts; p0 += 8) {
    float4 o[8];
    float wp[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int p = p0 + j;
      wp[j] = __shfl_sync(0xffffffffu, w, p & 31) * inv;
      if (p >= m.n_parts) wp[j] = 0.f;
      o[j] = (p < m.n_parts && lane < D / 4) ? load_bf16x4_cg(base + p * slot_stride)
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (wp[j] != 0.f) {
        acc.x = fmaf(wp[j], o[j].x, acc.x);
        acc.y = fmaf(wp[j], o[j].y, acc.y);
        acc.z = fmaf(wp[j], o[j].z, acc.z);
        acc.w = fmaf(wp[j], o[j].w, acc.w);
      }
    }
  }
  if (lane < D / 4) store_bf16x4(m.out + row * D + lane * 4, acc);
  if (lane == 0 && m.lse != nullptr)
    m.lse[row] = !(wsum <= 0.f) ? (mx + log2f(wsum)) * 0.69314718055994531f : -INFINITY;
}

// Called by every thread of the CTA (it contains __syncthreads) after the CTA wrote
// its partial rows for tokens [t_first, t_first + n_tokens) of KV head g.
// s_last: shared scratch of at least n_tokens ints.
template <int D>
__device__ __forceinline__ void count_and_merge(const MergeArgs& m, int t_first, int n_tokens,
                                                int g, int* s_last) {
  const int tid = threadIdx.x;
  const int nthr = blockDim.x;
  __syncthreads();  // every partial row of this CTA is written
  for (int i = tid; i < n_tokens; i += nthr) {
    int* c = m.counters + static_cast<int64_t>(t_first + i) * m.num_kv_heads + g;
    s_last[i] = atomic_add_acq_rel_gpu(c, 1) == m.n_count - 1;
  }
  __syncthreads();
  const int warp = tid >> 5, lane = tid & 31, nwarps = nthr >> 5;
  for (int k = warp; k < n_tokens * m.group; k += nwarps) {
    const int i = k / m.group;
    if (!s_last[i]) continue;
    const int64_t row = static_cast<int64_t>(t_first + i) * m.num_q_heads + g * m.group +
                        k % m.group;
    merge_row_warp<D>(m, row, lane, false, make_float4(0.f, 0.f, 0.f, 0.f), -INFINITY);
  }
}

// Block-wide merge of `n_rows` output rows, for a CTA that holds many rows of one
// row space (paged_tc.cu).  Row i is output row row_of(i); skip(i) leaves it alone.
// Slots [0, m.n_parts) come from the workspace; with `own` (bf16 rows at
// own + i * own_stride, log2-sum-exp own_lse[i]) one more partial comes from shared
// memory.  Every thread takes part and every load of a step is issued before its
// results are used, so the step costs about one memory round trip rather than one per
// row.  s_w: shared scratch of n_rows * (m.n_parts + 1) floats.  Called by every
// thread of the CTA (contains __syncthreads).
template <int D, typename RowOf, typename Skip>
__device__ __forceinline__ void merge_rows_block(const MergeArgs& m, int n_rows, RowOf row_of,
                                                 Skip skip, const __nv_bfloat16* own,
                                                 int own_stride, const float* own_lse,
                                                 float* s_w) {
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int np = m.n_parts;
  const int W = np + 1;
  // weights of every partial of a row (normalised) and the row's final LSE
  for (int i = tid; i < n_rows; i += nthr) {
    if (skip(i)) continue;
    const int64_t row = row_of(i);
    float* w = s_w + i * W;
    float mx = own ? own_lse[i] : -INFINITY;
#pragma unroll 4
    for (int p = 0; p < np; ++p) {
      const float l = __ldcg(m.part_lse + static_cast<int64_t>(p) * m.rows + row);
      w[p] = l;
      mx = fmaxf(mx, l);
    }
    float wsum = 0.f;
    for (int p = 0; p < np; ++p) {
      const float e = (w[p] == -INFINITY || mx == -INFINITY) ? 0.f : fast_exp2(w[p] - mx);
      w[p] = e;
      wsum += e;
    }
    const float w_own =
        (own && mx != -INFINITY && own_lse[i] != -INFINITY) ? fast_exp2(own_lse[i] - mx) : 0.f;
    wsum += w_own;
    const float inv = !(wsum <= 0.f) ? 1.f / wsum : 0.f;  // a NaN sum propagates
    for (int p = 0; p < np; ++p) w[p] *= inv;
    w[np] = w_own * inv;
    if (m.lse != nullptr)
      m.lse[row] = !(wsum <= 0.f) ? (mx + log2f(wsum)) * 0.69314718055994531f : -INFINITY;
  }
  __syncthreads();
  // the rows, 16 bytes (8 features) per item, eight items per thread in flight
  constexpr int kC = D / 8;
  const int n_items = n_rows * kC;
  const int64_t slot_stride = static_cast<int64_t>(m.rows) * D;
  for (int base = tid; base < n_items; base += 8 * nthr) {
    float acc[8][8];
    int64_t off[8];
    int ri[8];
    bool ok[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int it = base + j * nthr;
      const int i = it / kC, c = it % kC;
      ok[j] = it < n_items && !skip(i);
      ri[j] = i;
      off[j] = ok[j] ? row_of(i) * D + c * 8 : 0;
      const float wo = ok[j] ? s_w[i * W + np] : 0.f;
      if (own && wo != 0.f) {
        const uint4 u = *reinterpret_cast<const uint4*>(own + i * own_stride + c * 8);
        const uint32_t uu[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&uu[e]));
          acc[j][2 * e] = wo * f.x;
          acc[j][2 * e + 1] = wo * f.y;
        }
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[j][e] = 0.f;
      }
    }
    for (int p = 0; p < np; ++p) {
      uint4 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        v[j] = ok[j] ? __ldcg(reinterpret_cast<const uint4*>(m.part_o + p * slot_stride + off[j]))
                     : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float wp = ok[j] ? s_w[ri[j] * W + p] : 0.f;
        if (wp != 0.f) {  // an empty slot is never read into the sum
          const uint32_t uu[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f =
                __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&uu[e]));
            acc[j][2 * e] = fmaf(wp, f.x, acc[j][2 * e]);
            acc[j][2 * e + 1] = fmaf(wp, f.y, acc[j][2 * e + 1]);
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (ok[j])
        *reinterpret_cast<uint4*>(m.out + off[j]) =
            make_uint4(pack_bf16x2(acc[j][0], acc[j][1]), pack_bf16x2(acc[j][2], acc[j][3]),
                       pack_bf16x2(acc[j][4], acc[j][5]), pack_bf16x2(acc[j][6], acc[j][7]));
  }
}

// After a CTA has written its partial rows: count it in the row groups (token
// t_first + i, KV head g) for i in [0, n_tok); the group's m.n_count-th contributor
// merges the group's rows of this CTA (row i of n_rows is output row row_of(i), of the
// CTA's token tok_local(i)).  s_last: shared scratch of n_tok ints; s_w as for
// merge_rows_block.  Called by every thread of the CTA.
template <int D, typename RowOf, typename TokOf>
__device__ __forceinline__ void count_and_merge_block(const MergeArgs& m, int t_first, int n_tok,
                                                      int g, int n_rows, RowOf row_of,
                                                      TokOf tok_local, int* s_last, float* s_w) {
  __syncthreads();  // every partial row of this CTA is written
  for (int i = threadIdx.x; i < n_tok; i += blockDim.x) {
    int* c = m.counters + static_cast<int64_t>(t_first + i) * m.num_kv_heads + g;
    s_last[i] = atomic_add_acq_rel_gpu(c, 1) == m.n_count - 1;
  }
  __syncthreads();
  merge_rows_block<D>(m, n_rows, row_of, [&](int i) { return s_last[tok_local(i)] == 0; },
                      nullptr, 0, nullptr, s_w);
}

}  // namespace csp
