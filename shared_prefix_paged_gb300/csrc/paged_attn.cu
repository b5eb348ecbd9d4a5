// paged_attn.cu — causal attention of each request over a range of its own KV
// pages: the suffix phase of cascade attention (keys [cpl, seq_len), "vLLM Cascade
// Attention：用法、场景与原理解析" §八 Step 5 Phase 2) and the standard path (keys
// [0, seq_len), §五 and §十).
//
// This work streams each request's private pages from HBM once and does little
// arithmetic per byte, so the design aims at bandwidth:
//  * for decode-shaped rows: at most 16 per request and KV head (query tokens x heads
//    in the group); more rows take the tcgen05 variant (paged_tc.cu);
//  * one CTA per (request, KV head, key split); its rows are the request's
//    (query, head-in-group) pairs of that KV head, so all GQA heads of a KV head
//    share each page load;
//  * pages are fetched with 16-byte cp.async (coalesced: 16 threads per 256-byte
//    page row) into an XOR-swizzled shared tile of 64 keys, two stages deep;
//    keys past the range are zero-filled and never read from the block table;
//  * QK^T and PV run on warp-level bf16 MMA (m16n8k16) fed by ldmatrix; the online
//    softmax keeps its row max / sum with warp shuffles inside each 4-lane row group;
//  * the four warps split the keys of every tile and merge (max, sum, O) through
//    shared memory at the end;
//  * split-KV (FlashDecoding, §九) over long ranges: each split writes a normalised
//    bf16 partial + log2-sum-exp and the last split of a row group merges them with
//    the prefix phase's partials (merge.cuh); a single split merges its own result
//    in registers; the standard path with one split writes bf16 output and the
//    natural-log LSE directly.
#include "common.cuh"
#include "kernels.cuh"
#include "merge.cuh"

namespace csp {
namespace {

constexpr int kTileKeys = 64;
constexpr int kPage = 16;
constexpr int kThreads = 128;

template <int D>
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  // byte offset of 16-byte chunk `chunk` of row `row` in a [rows][D] bf16 tile
  return static_cast<uint32_t>(row * (D * 2) + ((chunk ^ (row & 7)) << 4));
}

template <int D, bool kF8 = false>
struct PagedLayout {
  // two 64-key tiles in flight (68 KB for D=128), so three CTAs fit on an SM.  An E4M3
  // cache keeps four tiles in flight as bytes (the same bytes in flight per SM with two
  // CTAs) and widens the current one into a single f16 K/V buffer (100 KB).
  static constexpr int kStages = kF8 ? 4 : 2;
  static constexpr int kRows = 16;
  static constexpr int kQBytes = kRows * D * 2;
  static constexpr int kKVBytes = kTileKeys * D * 2;
  static constexpr int kBufs = kF8 ? 1 : kStages;          // 16-bit K (and V) tiles
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kQBytes;
  static constexpr int kV = kK + kBufs * kKVBytes;
  static constexpr int kF8Tile = kTileKeys * D;             // E4M3 K (or V) tile
  static constexpr int kF8Base = kV + kBufs * kKVBytes;     // [stage][K, V] E4M3 tiles
  static constexpr int kLast = kF8Base + (kF8 ? kStages * 2 * kF8Tile : 0);  // int [64] flags
  static constexpr int kEnd = kLast + 64 * 4;
  // decode merge scratch (reuses the K/V stages after the last tile): per warp 16
  // rows of D floats with a padded stride, then per-warp max and sum
  static constexpr int kORow = D + 8;
  static constexpr int kMergeBytes = 4 * 16 * kORow * 4 + 2 * 4 * 16 * 4;
  // the cluster merge's exchange area after it: each row's normalised O (fp32) and
  // log2-sum-exp, read by the other CTAs of the cluster
  static constexpr int kXO = kK + kMergeBytes;
  static constexpr int kXL = kXO + 16 * D * 4;
  static_assert(kXL + 16 * 4 <= kLast, "merge scratch and exchange area");
};

// kF8: an E4M3 KV cache (a.k, a.v its bytes, a.q the f16 queries): the tiles arrive
// as bytes, are widened to f16 in shared memory (exact) and run on f16 MMAs; the V
// scale multiplies the normalised rows.
template <int D, bool kF8>
__global__ void __launch_bounds__(kThreads)
    paged_attn_kernel(const PagedArgs a) {
  using L = PagedLayout<D, kF8>;
  constexpr int kStages = L::kStages;
  constexpr int kChunks = D / 8;               // 16-byte chunks per row
  constexpr int kWarpKeys = 16;                // keys of a tile each warp handles
  constexpr int kNT = kWarpKeys / 8;           // S n-tiles per warp
  constexpr int kDT = D / 8;                   // O n-tiles

  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int r = blockIdx.x / a.row_tiles;
  const int rt = blockIdx.x % a.row_tiles;
  const int g = blockIdx.y;
  const int split = blockIdx.z;
  const int q0 = __ldg(a.cu_seqlens_q + r);
  const int q_len = __ldg(a.cu_seqlens_q + r + 1) - q0;
  const int seq = __ldg(a.seq_lens + r);
  const int rows_total = q_len * a.group;
  const int row0 = rt * L::kRows;
  if (row0 >= rows_total) return;
  const int rows_here = min(L::kRows, rows_total - row0);

  // key range of this split, clipped by the causal limit of the tile's last row
  const int last_query = (row0 + rows_here - 1) / a.group;
  const int kbeg =
      (a.key_start_of != nullptr ? __ldg(a.key_start_of + r) : a.key_start) + split * a.split_keys;
  int kend = min(kbeg + a.split_keys, seq);
  kend = min(kend, seq - q_len + last_query + 1);
  const int n_tiles = kend > kbeg ? (kend - kbeg + kTileKeys - 1) / kTileKeys : 0;

  const int32_t* bt_row = a.block_table + static_cast<int64_t>(r) * a.bt_stride;
  const uint32_t sbase = smem_u32(smem);

  auto load_tile = [&](int ti, int stage) {
    const int kt0 = kbeg + ti * kTileKeys;
    if constexpr (kF8) {
      // 16-byte chunks of E4M3 bytes (16 features each), [key][D bytes] per tile
      constexpr int kC16 = D / 16;
      const uint8_t* k8 = reinterpret_cast<const uint8_t*>(a.k);
      const uint8_t* v8 = reinterpret_cast<const uint8_t*>(a.v);
      uint8_t* sk = smem + L::kF8Base + stage * 2 * L::kF8Tile;
      uint8_t* sv = sk + L::kF8Tile;
#pragma unroll
      for (int x = threadIdx.x; x < kTileKeys * kC16; x += kThreads) {
        const int key = x / kC16, c = x % kC16;
        const int kabs = kt0 + key;
        const bool ok = kabs < kend;
        int64_t off = 0;
        if (ok) {
          const int blk = __ldg(bt_row + kabs / kPage);
          off = ((static_cast<int64_t>(blk) * kPage + kabs % kPage) * a.num_kv_heads + g) * D +
                c * 16;
        }
        cp_async_16(sk + key * D + c * 16, k8 + off, ok ? 16u : 0u);
        cp_async_16(sv + key * D + c * 16, v8 + off, ok ? 16u : 0u);
      }
      return;
    }
    uint8_t* sk = smem + L::kK + stage * L::kKVBytes;
    uint8_t* sv = smem + L::kV + stage * L::kKVBytes;
#pragma unroll
    for (int x = threadIdx.x; x < kTileKeys * kChunks; x += kThreads) {
      const int key = x / kChunks, c = x % kChunks;
      const int kabs = kt0 + key;
      const bool ok = kabs < kend;
      int64_t off = 0;
      if (ok) {
        const int blk = __ldg(bt_row + kabs / kPage);
        off = ((static_cast<int64_t>(blk) * kPage + kabs % kPage) * a.num_kv_heads + g) * D +
              c * 8;
      }
      cp_async_16(sk + swz<D>(key, c), a.k + off, ok ? 16u : 0u);
      cp_async_16(sv + swz<D>(key, c), a.v + off, ok ? 16u : 0u);
    }
  };

  // Q rows of this tile: packed row rho = query * group + head-in-group
#pragma unroll
  for (int x = threadIdx.x; x < L::kRows * kChunks; x += kThreads) {
    const int row = x / kChunks, c = x % kChunks;
    const int rho = row0 + row;
    const bool ok = rho < rows_total;
    int64_t off = 0;
    if (ok) {
      const int qi = rho / a.group, j = rho % a.group;
      off = (static_cast<int64_t>(q0 + qi) * a.num_q_heads + g * a.group + j) * D + c * 8;
    }
    cp_async_16(smem + L::kQ + swz<D>(row, c), a.q + off, ok ? 16u : 0u);
  }
  // every stage in flight from the start; a stage is refilled right after its
  // tile has been consumed
#pragma unroll
  for (int st = 0; st < kStages; ++st) {
    if (st < n_tiles) load_tile(st, st);
    cp_async_commit();
  }

  // per-warp state: all 16 rows (thread rows lane/4 and lane/4 + 8)
  const int kw0 = warp * 16;
  float o[kDT][4];
#pragma unroll
  for (int i = 0; i < kDT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  int pos[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int rho = row0 + (lane >> 2) + 8 * h;
    pos[h] = rho < rows_total ? seq - q_len + rho / a.group : -1;  // -1: padding row
  }
  uint32_t qa[D / 16][4];

  for (int ti = 0; ti < n_tiles; ++ti) {
    cp_async_wait<kStages - 1>();  // groups 0..ti (tile ti, and Q with tile 0) landed
    __syncthreads();
    if (ti == 0) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int row = (lane & 7) + ((lane >> 3) & 1) * 8;
        const int c = kk * 2 + (lane >> 4);
        ldmatrix_x4(sbase + L::kQ + swz<D>(row, c), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
      }
    }
    if constexpr (kF8) {
      // widen tile ti into the f16 K/V buffer (every warp finished tile ti - 1): this
      // thread's column c (16 features) of keys key0 + kStep i; the swizzle term
      // key & 7 is the same for every i
      constexpr int kC16 = D / 16;
      constexpr int kStep = kThreads / kC16;
      const int c = threadIdx.x % kC16, key0 = threadIdx.x / kC16;
      const uint8_t* src = smem + L::kF8Base + (ti % kStages) * 2 * L::kF8Tile + key0 * D + c * 16;
      const uint32_t lo_off = swz<D>(key0, 2 * c), hi_off = swz<D>(key0, 2 * c + 1);
#pragma unroll
      for (int i = 0; i < kTileKeys / kStep; ++i) {
        uint4 lo, hi;
        e4m3x16_to_f16(*reinterpret_cast<const uint4*>(src + i * kStep * D), lo, hi);
        *reinterpret_cast<uint4*>(smem + L::kK + i * kStep * D * 2 + lo_off) = lo;
        *reinterpret_cast<uint4*>(smem + L::kK + i * kStep * D * 2 + hi_off) = hi;
        e4m3x16_to_f16(*reinterpret_cast<const uint4*>(src + L::kF8Tile + i * kStep * D), lo,
                       hi);
        *reinterpret_cast<uint4*>(smem + L::kV + i * kStep * D * 2 + lo_off) = lo;
        *reinterpret_cast<uint4*>(smem + L::kV + i * kStep * D * 2 + hi_off) = hi;
      }
      __syncthreads();
    }
    {
    const int stage = kF8 ? 0 : ti % kStages;
    const uint32_t sk = sbase + L::kK + stage * L::kKVBytes;
    const uint32_t sv = sbase + L::kV + stage * L::kKVBytes;
    const int kt0 = kbeg + ti * kTileKeys;

    // S = Q K^T for this warp's keys
    float sacc[kNT][4];
#pragma unroll
    for (int i = 0; i < kNT; ++i) sacc[i][0] = sacc[i][1] = sacc[i][2] = sacc[i][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
      for (int np = 0; np < kNT / 2; ++np) {
        const int key = kw0 + np * 16 + (lane & 7) + (lane >> 4) * 8;
        const int c = kk * 2 + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(sk + swz<D>(key, c), b0, b1, b2, b3);
        if constexpr (kF8) {
          mma_f16_16816(sacc[2 * np], qa[kk], b0, b1);
          mma_f16_16816(sacc[2 * np + 1], qa[kk], b2, b3);
        } else {
          mma_bf16_16816(sacc[2 * np], qa[kk], b0, b1);
          mma_bf16_16816(sacc[2 * np + 1], qa[kk], b2, b3);
        }
      }
    }
    // mask, online softmax (base 2)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float mx = -INFINITY;
      const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) {
        // the two scores of a pair scaled in one paired instruction, then masked
        const float2 s2 = mul_f32x2(make_float2(sacc[nt][2 * h], sacc[nt][2 * h + 1]), sc2);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int kabs = kt0 + kw0 + nt * 8 + (lane & 3) * 2 + e;
          float& sref = sacc[nt][2 * h + e];
          sref = (kabs < kend && kabs <= pos[h]) ? (e ? s2.y : s2.x) : -INFINITY;
          mx = fmaxf(mx, sref);
        }
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_run[h], mx);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = exp2f(m_run[h] - m_use);
      float2 sum2 = make_float2(0.f, 0.f);
      const float2 nm2 = make_float2(-m_use, -m_use);
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) {
        const float2 x = add_f32x2(make_float2(sacc[nt][2 * h], sacc[nt][2 * h + 1]), nm2);
        sacc[nt][2 * h] = exp2f(x.x);
        sacc[nt][2 * h + 1] = exp2f(x.y);
        sum2 = add_f32x2(sum2, make_float2(sacc[nt][2 * h], sacc[nt][2 * h + 1]));
      }
      l_run[h] = l_run[h] * alpha + (sum2.x + sum2.y);
      m_run[h] = m_new;
      const float2 al2 = make_float2(alpha, alpha);
#pragma unroll
      for (int dt = 0; dt < kDT; ++dt) {
        const float2 r = mul_f32x2(make_float2(o[dt][2 * h], o[dt][2 * h + 1]), al2);
        o[dt][2 * h] = r.x;
        o[dt][2 * h + 1] = r.y;
      }
    }
    // O += P V
#pragma unroll
    for (int kk = 0; kk < kWarpKeys / 16; ++kk) {
      uint32_t pa[4];
      auto pack = [](float x, float y) { return kF8 ? pack_f16x2(x, y) : pack_bf16x2(x, y); };
      pa[0] = pack(sacc[2 * kk][0], sacc[2 * kk][1]);
      pa[1] = pack(sacc[2 * kk][2], sacc[2 * kk][3]);
      pa[2] = pack(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1]);
      pa[3] = pack(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3]);
#pragma unroll
      for (int dp = 0; dp < kDT / 2; ++dp) {
        const int key = kw0 + kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int c = dp * 2 + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(sv + swz<D>(key, c), b0, b1, b2, b3);
        if constexpr (kF8) {
          mma_f16_16816(o[2 * dp], pa, b0, b1);
          mma_f16_16816(o[2 * dp + 1], pa, b2, b3);
        } else {
          mma_bf16_16816(o[2 * dp], pa, b0, b1);
          mma_bf16_16816(o[2 * dp + 1], pa, b2, b3);
        }
      }
    }
    }
    __syncthreads();  // every warp is done with this stage
    if (ti + kStages < n_tiles) load_tile(ti + kStages, ti % kStages);
    cp_async_commit();
  }
  cp_async_wait<0>();

  // row sums across the 4 lanes of each row group
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
  }
  const bool partial = a.part_o != nullptr;
  constexpr float kLn2 = 0.69314718055994531f;
  MergeArgs m;
  m.part_o = a.part_o;
  m.part_lse = a.part_lse;
  m.counters = a.counters;
  m.n_parts = a.n_prefix + a.n_splits;
  m.n_count = a.n_splits;
  m.rows = a.total_q * a.num_q_heads;
  m.num_q_heads = a.num_q_heads;
  m.num_kv_heads = a.num_kv_heads;
  m.group = a.group;
  m.out = a.out;
  m.lse = a.lse;
  // one suffix split: this CTA merges its rows itself, in registers, with the prefix
  // slots; several splits: write a partial and let the last split merge, or (a cluster
  // of the splits) leave it in shared memory for the cluster merge below
  const bool merge_in_place = partial && a.n_splits == 1 && !a.partials_only;
  const bool in_cluster = a.cluster_splits;

  {
    // merge the four warps' (m, l, O) of the same 16 rows through shared memory
    __syncthreads();
    float* s_o = reinterpret_cast<float*>(smem + L::kK);   // [4][16][kORow]
    float* s_m = s_o + 4 * 16 * L::kORow;                   // [4][16]
    float* s_l = s_m + 4 * 16;                              // [4][16]
    if ((lane & 3) == 0) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        s_m[warp * 16 + (lane >> 2) + 8 * h] = m_run[h];
        s_l[warp * 16 + (lane >> 2) + 8 * h] = l_run[h];
      }
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int rr = (lane >> 2) + 8 * h;
      float mg = -INFINITY;
#pragma unroll
      for (int w = 0; w < 4; ++w) mg = fmaxf(mg, s_m[w * 16 + rr]);
      const float sc = (m_run[h] == -INFINITY) ? 0.f : exp2f(m_run[h] - mg);
      float* dst = s_o + (warp * 16 + rr) * L::kORow;
#pragma unroll
      for (int dt = 0; dt < kDT; ++dt) {
        const int d = dt * 8 + (lane & 3) * 2;
        *reinterpret_cast<float2*>(dst + d) = make_float2(o[dt][2 * h] * sc, o[dt][2 * h + 1] * sc);
      }
    }
    __syncthreads();
    // the prefix grid's partials are read below: wait for it (a no-op when this
    // kernel was not launched behind it)
    if (merge_in_place) grid_dependency_wait();
    // warp w finalises rows w, w+4, w+8, w+12; lane c owns features [4c, 4c+4)
    for (int rr = warp; rr < 16; rr += 4) {
      const int rho = row0 + rr;
      if (rho >= rows_total) break;
      float mg = -INFINITY;
#pragma unroll
      for (int w = 0; w < 4; ++w) mg = fmaxf(mg, s_m[w * 16 + rr]);
      float lsum = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float mw = s_m[w * 16 + rr];
        lsum += (mw == -INFINITY) ? 0.f : s_l[w * 16 + rr] * exp2f(mw - mg);
      }
      float inv = !(lsum <= 0.f) ? 1.f / lsum : 0.f;  // a NaN sum propagates
      if constexpr (kF8) inv *= a.v_scale;
      const float lse2 = !(lsum <= 0.f) ? mg + log2f(lsum) : -INFINITY;
      const int qi = rho / a.group, j = rho % a.group;
      const int64_t orow = static_cast<int64_t>(q0 + qi) * a.num_q_heads + g * a.group + j;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      if (lane < D / 4) {
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float4 v = *reinterpret_cast<const float4*>(s_o + (w * 16 + rr) * L::kORow + lane * 4);
          acc.x += v.x;
          acc.y += v.y;
          acc.z += v.z;
          acc.w += v.w;
        }
        acc = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
      }
      if (in_cluster) {
        float* xo = reinterpret_cast<float*>(smem + L::kXO);
        if (lane < D / 4) *reinterpret_cast<float4*>(xo + rr * D + lane * 4) = acc;
        if (lane == 0) reinterpret_cast<float*>(smem + L::kXL)[rr] = lse2;
      } else if (merge_in_place) {
        merge_row_warp<D>(m, orow, lane, true, acc, lse2);
      } else if (partial) {
        const int64_t prow = static_cast<int64_t>(a.n_prefix + split) * a.total_q *
                                 a.num_q_heads + orow;
        if (lane < D / 4) store_bf16x4(a.part_o + prow * D + lane * 4, acc);
        if (lane == 0) a.part_lse[prow] = lse2;
      } else {
        if (lane < D / 4) store_bf16x4(a.out + orow * D + lane * 4, acc);
        if (lane == 0 && a.lse != nullptr) a.lse[orow] = lse2 * kLn2;
      }
    }
  }

  if (in_cluster) {
    // The cluster is this row tile's key splits (cluster rank = split).  After the
    // barrier every CTA's rows are in its exchange area; CTA `rank` merges rows rank,
    // rank + n_splits, ... : the prefix slots (global memory, after the prefix grid)
    // and every split's partial (distributed shared memory), one warp per row.
    cluster_barrier();
    const int ns = a.n_splits;
    const int rank = static_cast<int>(cluster_rank());
    const int np = a.n_prefix;
    if (np > 0) grid_dependency_wait();
    const uint32_t xo0 = smem_u32(smem + L::kXO), xl0 = smem_u32(smem + L::kXL);
    for (int rr = rank + ns * warp; rr < rows_here; rr += ns * 4) {
      const int rho = row0 + rr;
      const int qi = rho / a.group, j = rho % a.group;
      const int64_t orow = static_cast<int64_t>(q0 + qi) * a.num_q_heads + g * a.group + j;
      // lane p: the log2-sum-exp of partial p (prefix slots first, then the splits)
      float lp = -INFINITY;
      if (lane < np)
        lp = __ldcg(a.part_lse + static_cast<int64_t>(lane) * m.rows + orow);
      else if (lane < np + ns)
        lp = ld_cluster_f32(cluster_map(xl0 + rr * 4, lane - np));
      float mx = lp;
#pragma unroll
      for (int sft = 16; sft > 0; sft >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, sft));
      const float w = (mx == -INFINITY || lp == -INFINITY) ? 0.f : fast_exp2(lp - mx);
      float wsum = w;
#pragma unroll
      for (int sft = 16; sft > 0; sft >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, sft);
      const float inv = !(wsum <= 0.f) ? 1.f / wsum : 0.f;  // a NaN sum propagates
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int p = 0; p < np + ns; ++p) {
        const float wp = __shfl_sync(0xffffffffu, w, p) * inv;
        if (wp == 0.f || lane >= D / 4) continue;  // an empty partial is never read
        const float4 v =
            p < np ? load_bf16x4_cg(a.part_o + (static_cast<int64_t>(p) * m.rows + orow) * D +
                                    lane * 4)
                   : ld_cluster_f32x4(cluster_map(xo0 + (rr * D + lane * 4) * 4, p - np));
        acc.x = fmaf(wp, v.x, acc.x);
        acc.y = fmaf(wp, v.y, acc.y);
        acc.z = fmaf(wp, v.z, acc.z);
        acc.w = fmaf(wp, v.w, acc.w);
      }
      if (lane < D / 4) store_bf16x4(a.out + orow * D + lane * 4, acc);
      if (lane == 0 && a.lse != nullptr)
        a.lse[orow] = !(wsum <= 0.f) ? (mx + log2f(wsum)) * kLn2 : -INFINITY;
    }
    // no CTA leaves while another may still read its exchange area
    cluster_barrier();
    return;
  }

  if (partial && !merge_in_place && a.counters != nullptr) {
    // several splits: count in the row groups; the last split merges every slot
    const int tok_first = row0 / a.group;
    const int n_tok = (row0 + rows_here - 1) / a.group - tok_first + 1;
    grid_dependency_wait();  // prefix partials are complete and visible
    __syncthreads();         // merge scratch no longer needed below
    count_and_merge<D>(m, q0 + tok_first, n_tok, g, reinterpret_cast<int*>(smem + L::kLast));
  }
}

template <int D, bool kF8>
cudaError_t launch_paged_t(const PagedArgs& a, bool after_prefix, cudaStream_t stream) {
  using L = PagedLayout<D, kF8>;
  const int smem = L::kEnd;
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = set_smem_once(paged_attn_kernel<D, kF8>, smem, attr_done);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.num_reqs * a.row_tiles, a.num_kv_heads, a.n_splits);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  // Right after the prefix kernel of the same call: start while it runs; the merge
  // with the prefix slots waits for the prefix grid (griddepcontrol.wait).
  if (after_prefix) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (a.cluster_splits) {  // a row tile's splits: one cluster
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = 1;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = static_cast<unsigned>(a.n_splits);
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, paged_attn_kernel<D, kF8>, a);
}

}  // namespace

cudaError_t launch_paged(int head_dim, const PagedArgs& a, bool after_prefix,
                         cudaStream_t stream) {
  if (head_dim == 64) return launch_paged_t<64, false>(a, after_prefix, stream);
  return launch_paged_t<128, false>(a, after_prefix, stream);
}

cudaError_t launch_paged_f8(int head_dim, const PagedArgs& a, bool after_prefix,
                            cudaStream_t stream) {
  if (head_dim == 64) return launch_paged_t<64, true>(a, after_prefix, stream);
  return launch_paged_t<128, true>(a, after_prefix, stream);
}

}  // namespace csp
