// combine.cu — the merge_states entry point's kernel: LSE merge of two partials.
//
// "vLLM Cascade Attention：用法、场景与原理解析" §一 and §八 Step 5 (merge_attn_states):
// partial results over disjoint key sets combine by log-sum-exp rescaling,
//   m = max(l1, l2),  w_i = e^(l_i - m),  out = (w1 o1 + w2 o2) / (w1 + w2),
//   lse = m + ln(w1 + w2).
// Elementwise and HBM-bound: D/8 threads per output row, 16-byte vector loads and
// stores, fp32 math.  (Inside cascade_attn the same merge runs in the attention
// kernels themselves, see merge.cuh, or, after a tcgen05 suffix phase, in
// merge_slots_kernel below.)
#include <algorithm>

#include "common.cuh"
#include "kernels.cuh"
#include "merge.cuh"

namespace csp {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// Two partials with natural-log LSEs (the merge_states entry point).  Each thread
// handles 8 features of one row.
template <bool kF32>
__global__ void __launch_bounds__(256)
    merge_states_kernel(__nv_bfloat16* __restrict__ out, float* __restrict__ out_lse,
                        const void* __restrict__ o1, const float* __restrict__ l1,
                        const void* __restrict__ o2, const float* __restrict__ l2, int rows,
                        int head_dim) {
  const int chunks = head_dim / 8;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<int64_t>(rows) * chunks) return;
  const int row = static_cast<int>(idx / chunks);
  const int c = static_cast<int>(idx % chunks);
  const float a = __ldg(l1 + row), b = __ldg(l2 + row);
  const float m = fmaxf(a, b);
  float w1 = 0.f, w2 = 0.f;
  if (m != -INFINITY) {
    w1 = exp2f((a - m) * kLog2e);
    w2 = exp2f((b - m) * kLog2e);
  }
  const float ws = w1 + w2;
  const float inv = !(ws <= 0.f) ? 1.f / ws : 0.f;  // a NaN sum propagates
  float x1[8], x2[8];
  const int64_t off = static_cast<int64_t>(row) * head_dim + c * 8;
  if constexpr (kF32) {
    const float4* p1 = reinterpret_cast<const float4*>(static_cast<const float*>(o1) + off);
    const float4* p2 = reinterpret_cast<const float4*>(static_cast<const float*>(o2) + off);
    const float4 u0 = __ldg(p1), u1 = __ldg(p1 + 1), v0 = __ldg(p2), v1 = __ldg(p2 + 1);
    x1[0] = u0.x; x1[1] = u0.y; x1[2] = u0.z; x1[3] = u0.w;
    x1[4] = u1.x; x1[5] = u1.y; x1[6] = u1.z; x1[7] = u1.w;
    x2[0] = v0.x; x2[1] = v0.y; x2[2] = v0.z; x2[3] = v0.w;
    x2[4] = v1.x; x2[5] = v1.y; x2[6] = v1.z; x2[7] = v1.w;
  } else {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(o1) + off));
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(o2) + off));
    const __nv_bfloat162* pu = reinterpret_cast<const __nv_bfloat162*>(&u);
    const __nv_bfloat162* pv = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 fu = __bfloat1622float2(pu[e]);
      const float2 fv = __bfloat1622float2(pv[e]);
      x1[2 * e] = fu.x; x1[2 * e + 1] = fu.y;
      x2[2 * e] = fv.x; x2[2 * e + 1] = fv.y;
    }
  }
  uint32_t w[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    // an empty side (lse = -inf, weight 0) contributes nothing, whatever its values
    const float y0 = (w1 != 0.f ? w1 * x1[2 * e] : 0.f) + (w2 != 0.f ? w2 * x2[2 * e] : 0.f);
    const float y1 = (w1 != 0.f ? w1 * x1[2 * e + 1] : 0.f) + (w2 != 0.f ? w2 * x2[2 * e + 1] : 0.f);
    w[e] = pack_bf16x2(y0 * inv, y1 * inv);
  }
  *reinterpret_cast<uint4*>(out + off) = make_uint4(w[0], w[1], w[2], w[3]);
  if (c == 0 && out_lse != nullptr) out_lse[row] = !(ws <= 0.f) ? m + logf(ws) : -INFINITY;
}

// n slots per row (the cascade call's partials, log2 domain): one thread per 8
// features of a row.  It issues every slot's LSE and 16-byte piece at once (the slot
// loop unrolled to kS >= n; the row's other threads read the same LSEs: one L1 line),
// then weighs them and writes 16 bytes of out (the first thread of a row also the
// LSE).  An empty slot (lse -inf) gets weight 0 and a select keeps whatever it holds
// out of the sum.
constexpr int kMergeThreads = 256;

template <int D, int kS>
__global__ void __launch_bounds__(kMergeThreads)
    merge_slots_kernel(const MergeArgs m) {
  constexpr int kC = D / 8;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * kMergeThreads + threadIdx.x;
  if (idx >= static_cast<int64_t>(m.rows) * kC) return;
  const int64_t row = idx / kC;
  const int c = static_cast<int>(idx % kC);
  float l[kS];
  uint4 u[kS];
#pragma unroll
  for (int s = 0; s < kS; ++s) {
    const int64_t prow = static_cast<int64_t>(min(s, m.n_parts - 1)) * m.rows + row;
    l[s] = s < m.n_parts ? __ldcg(m.part_lse + prow) : -INFINITY;
    u[s] = __ldcg(reinterpret_cast<const uint4*>(m.part_o + prow * D + c * 8));
  }
  float mx = -INFINITY;
#pragma unroll
  for (int s = 0; s < kS; ++s) mx = fmaxf(mx, l[s]);
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float wsum = 0.f;
#pragma unroll
  for (int s = 0; s < kS; ++s) {
    const float w = (l[s] == -INFINITY || mx == -INFINITY) ? 0.f : fast_exp2(l[s] - mx);
    wsum += w;
    const uint32_t uu[4] = {u[s].x, u[s].y, u[s].z, u[s].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&uu[e]));
      acc[2 * e] = w != 0.f ? fmaf(w, f.x, acc[2 * e]) : acc[2 * e];
      acc[2 * e + 1] = w != 0.f ? fmaf(w, f.y, acc[2 * e + 1]) : acc[2 * e + 1];
    }
  }
  const float inv = !(wsum <= 0.f) ? 1.f / wsum : 0.f;  // a NaN sum propagates
  *reinterpret_cast<uint4*>(m.out + row * D + c * 8) =
      make_uint4(pack_bf16x2(acc[0] * inv, acc[1] * inv), pack_bf16x2(acc[2] * inv, acc[3] * inv),
                 pack_bf16x2(acc[4] * inv, acc[5] * inv), pack_bf16x2(acc[6] * inv, acc[7] * inv));
  if (c == 0 && m.lse != nullptr)
    m.lse[row] = !(wsum <= 0.f) ? (mx + log2f(wsum)) * 0.69314718055994531f : -INFINITY;
}

template <int D>
void launch_slots_d(const MergeArgs& m, unsigned grid, cudaStream_t stream) {
  if (m.n_parts <= 2)
    merge_slots_kernel<D, 2><<<grid, kMergeThreads, 0, stream>>>(m);
  else if (m.n_parts <= 4)
    merge_slots_kernel<D, 4><<<grid, kMergeThreads, 0, stream>>>(m);
  else if (m.n_parts <= 8)
    merge_slots_kernel<D, 8><<<grid, kMergeThreads, 0, stream>>>(m);
  else if (m.n_parts <= 16)
    merge_slots_kernel<D, 16><<<grid, kMergeThreads, 0, stream>>>(m);
  else
    merge_slots_kernel<D, kMaxParts><<<grid, kMergeThreads, 0, stream>>>(m);
}

// Attention sinks on a finished result: the LSE merge of row (t, h) with an empty
// partial whose LSE is sinks[h] (one more key of value zero in the row's softmax):
//   lse' = ln(e^lse + e^s),  out' = out e^(lse - lse').
// Each thread rescales 8 features of one row; a row's threads sit in one warp (D / 8
// divides 32), which reads every row's LSE before any of them is rewritten.
__global__ void __launch_bounds__(256)
    apply_sinks_kernel(__nv_bfloat16* __restrict__ out, float* __restrict__ lse,
                       const float* __restrict__ sinks, int rows, int heads, int head_dim) {
  const int chunks = head_dim / 8;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const bool valid = idx < static_cast<int64_t>(rows) * chunks;
  const int row = valid ? static_cast<int>(idx / chunks) : 0;
  const int c = valid ? static_cast<int>(idx % chunks) : 0;
  const float l = valid ? lse[row] : 0.f;
  __syncwarp();
  if (!valid) return;
  const float s = __ldg(sinks + row % heads);
  const float m = fmaxf(l, s);
  float lnew = -INFINITY, w = 0.f;
  if (m != -INFINITY) {
    const float a = expf(l - m), b = expf(s - m);
    lnew = m + logf(a + b);
    w = a / (a + b);
  }
  uint4* p = reinterpret_cast<uint4*>(out + static_cast<int64_t>(row) * head_dim + c * 8);
  uint4 u = *p;
  __nv_bfloat162* pu = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __bfloat1622float2(pu[e]);
    pu[e] = __floats2bfloat162_rn(f.x * w, f.y * w);
  }
  *p = u;
  if (c == 0) lse[row] = lnew;
}

}  // namespace

cudaError_t launch_merge_slots(int head_dim, const __nv_bfloat16* part_o, const float* part_lse,
                               int n_parts, int64_t rows, __nv_bfloat16* out, float* lse,
                               cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  MergeArgs m = {};
  m.part_o = part_o;
  m.part_lse = part_lse;
  m.n_parts = n_parts;
  m.rows = static_cast<int>(rows);
  m.out = out;
  m.lse = lse;
  const int64_t threads = rows * (head_dim / 8);
  const unsigned grid = static_cast<unsigned>((threads + kMergeThreads - 1) / kMergeThreads);
  if (head_dim == 64)
    launch_slots_d<64>(m, grid, stream);
  else
    launch_slots_d<128>(m, grid, stream);
  return cudaGetLastError();
}

cudaError_t launch_merge_states(__nv_bfloat16* out, float* out_lse, const void* o1,
                                const float* l1, const void* o2, const float* l2, int rows,
                                int head_dim, bool f32_partials, cudaStream_t stream) {
  const int64_t threads = static_cast<int64_t>(rows) * (head_dim / 8);
  if (threads == 0) return cudaSuccess;
  const int grid = static_cast<int>((threads + 255) / 256);
  if (f32_partials)
    merge_states_kernel<true><<<grid, 256, 0, stream>>>(out, out_lse, o1, l1, o2, l2, rows, head_dim);
  else
    merge_states_kernel<false><<<grid, 256, 0, stream>>>(out, out_lse, o1, l1, o2, l2, rows, head_dim);
  return cudaGetLastError();
}

}  // namespace csp

namespace csp {

cudaError_t launch_apply_sinks(__nv_bfloat16* out, float* lse, const float* sinks, int rows,
                               int heads, int head_dim, cudaStream_t stream) {
  const int64_t threads = static_cast<int64_t>(rows) * (head_dim / 8);
  const int64_t grid = (threads + 255) / 256;
  apply_sinks_kernel<<<static_cast<unsigned>(grid), 256, 0, stream>>>(out, lse, sinks, rows,
                                                                     heads, head_dim);
  return cudaGetLastError();
}

}  // namespace csp

namespace csp {
namespace {

// n floats at p set to v (the level slots' LSEs of a multi-level cascade start at -inf:
// a row that no segment of a level holds then has weight 0 in that level's slots).
__global__ void __launch_bounds__(256) fill_f32_kernel(float* __restrict__ p, int64_t n, float v) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    p[i] = v;
}

}  // namespace

// bf16 -> f16, 8 values per thread (the queries of an FP8-cache call; exact for every
// bf16 value in f16's normal range, rounded to nearest below it).
__global__ void __launch_bounds__(256) bf16_to_f16_kernel(const uint4* __restrict__ in,
                                                          uint4* __restrict__ out, int64_t n8) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * 256) {
    const uint4 u = __ldg(in + i);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
      o[e] = pack_f16x2(f.x, f.y);
    }
    out[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

cudaError_t launch_bf16_to_f16(const void* in, void* out, int64_t n, cudaStream_t stream) {
  const int64_t n8 = n / 8;  // n is a multiple of 8 (rows of D features)
  if (n8 <= 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((n8 + 255) / 256, 4096);
  bf16_to_f16_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      static_cast<const uint4*>(in), static_cast<uint4*>(out), n8);
  return cudaGetLastError();
}

cudaError_t launch_fill_f32(float* p, int64_t n, float v, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, 4096);
  fill_f32_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p, n, v);
  return cudaGetLastError();
}

}  // namespace csp
