// prefix_attn.cu — the prefix phase of cascade attention on tcgen05 tensor cores.
//
// "vLLM Cascade Attention：用法、场景与原理解析" §五 and §十: the prefix phase treats
// every query of the batch as one sequence (cu_seqlens_q = [0, total_q]) so that one
// load of a shared KV page serves a whole tile of queries; §八 Step 5 Phase 1:
// non-causal attention over KV [0, common_prefix_len) read through block_table[:1].
//
// GB300 design (not the FlashAttention tiling the page describes):
//  * a CTA owns 256 packed rows (token, head-in-group) of ONE KV head as two 128-row
//    M tiles, so every K/V byte staged into shared memory serves 256 query rows and
//    all the GQA heads of that KV head;
//  * K and V pages (16 tokens x 64 features per box, 128-byte swizzle) are staged by
//    TMA into a 4-deep ring of 64-key tiles;
//  * per M tile, S = Q K^T (M=128, N=64) goes into one of two TMEM buffers, so the
//    tensor core computes S(i+1) while the softmax works on S(i); P (bf16) is
//    written back into the S buffer and used from TMEM as the A operand of
//    O += P V (N = D).  The two M tiles use all 512 TMEM columns;
//  * two softmax warpgroups (one per M tile) own one TMEM lane (row) per thread:
//    online softmax in base 2 on the special-function unit, O rescaled in TMEM only
//    when the running max grows by more than 2^8; warp 8 issues the MMAs, warp 9
//    the TMA loads;
//  * the prefix is cut into n_splits key ranges, one CTA each; a CTA stages its
//    normalised rows (bf16) through shared memory and writes them, coalesced, into
//    workspace slot `split`; the suffix kernel, which waits for this grid before it
//    merges, combines them with its own partials (merge.cuh).
#include "common.cuh"
#include "kernels.cuh"
#include "merge.cuh"

namespace csp {
namespace {

constexpr int kRowsM = 128;    // rows per M tile
constexpr int kRowsCta = 256;  // two M tiles
constexpr int kKeysN = 64;     // keys per tile
constexpr int kPage = 16;      // tokens per KV page
constexpr int kPagesPerTile = kKeysN / kPage;
constexpr int kStages = 4;
constexpr int kThreads = 320;  // 2 softmax warpgroups, MMA warp, TMA warp
constexpr int kWarpMma = 8;
constexpr int kWarpTma = 9;

template <int D>
struct Layout {
  static constexpr int kHalves = D / 64;
  static constexpr int kQHalf = kRowsM * 128;           // 128 rows x 64 bf16
  static constexpr int kKVHalf = kKeysN * 128;          // 64 keys x 64 bf16
  static constexpr int kQTile = kHalves * kQHalf;       // one M tile of Q
  static constexpr int kKVBytes = kHalves * kKVHalf;    // one K (or V) tile
  static constexpr int kQ = 0;                          // [2 M tiles][halves]
  static constexpr int kK0 = kQ + 2 * kQTile;
  static constexpr int kV0 = kK0 + kStages * kKVBytes;
  static constexpr int kRing = kV0 + kStages * kKVBytes;
  // after the main loop, [0, kRing) stages the CTA's 256 normalised rows:
  // [row][D + 8] bf16 (the padding spreads the rows one warp writes over all banks)
  static constexpr int kStageRow = D + 8;
  static_assert(kRowsCta * kStageRow * 2 <= kRing, "staging buffer fits Q + ring");
  static constexpr int kLse = kRing;                    // float [256]
  static constexpr int kBar = kLse + kRowsCta * 4;      // mbarriers + slot + flag
  static constexpr int kEnd = kBar + 256;
  static constexpr int kDynamic = kEnd + 1024;          // slack to align the base to 1024
};

// Barrier over one softmax warpgroup (id 1 or 2, 128 threads) that ORs a predicate.
__device__ __forceinline__ bool wg_bar_any(int id, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %2, 0;\n\t"
      "bar.red.or.pred q, %1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(id), "r"(static_cast<uint32_t>(pred))
      : "memory");
  return r != 0;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefix_attn_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const PrefixArgs a) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* bar_q = bars + 0;
  uint64_t* kv_full = bars + 1;   // [kStages]
  uint64_t* kv_empty = bars + 1 + kStages;  // [kStages]
  uint64_t* s_full = bars + 1 + 2 * kStages;    // [2 tiles][2 buffers]
  uint64_t* p_full = bars + 5 + 2 * kStages;    // [2 tiles][2 buffers]
  uint64_t* o_done = bars + 9 + 2 * kStages;    // [2 tiles] every PV
  uint64_t* o_last = bars + 11 + 2 * kStages;   // [2 tiles] the last PV
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 13 + 2 * kStages);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 14 + 2 * kStages);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int split = blockIdx.x % a.n_splits;
  const int pair = (blockIdx.x / a.n_splits) % a.pairs;
  const int kvh = blockIdx.x / (a.n_splits * a.pairs);
  const int key_tiles = (a.cpl + kKeysN - 1) / kKeysN;
  const int t_first = min(split * a.tiles_per_split, key_tiles);
  const int t_last = min(t_first + a.tiles_per_split, key_tiles);
  const int ntiles = t_last - t_first;
  const int rows_total = a.total_q * a.group;                 // packed rows of this KV head
  const bool has_m1 = pair * kRowsCta + kRowsM < rows_total;  // second M tile has rows

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int b = 0; b < 4; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_full[b], 128);
    }
    for (int m = 0; m < 2; ++m) {
      mbar_init(&o_done[m], 1);
      mbar_init(&o_last[m], 1);
    }
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == kWarpMma) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the suffix kernel (launched as a programmatic dependent) may start now; it reads
  // this grid's partials only after waiting for the grid to complete
  grid_launch_dependents();

  if (warp == kWarpTma) {
    // ------------------------------------------------------------ TMA producer --
    if (lane == 0 && ntiles > 0) {  // an empty key range loads nothing at all
      prefetch_tensormap(&tm_q);
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_v);
      const int mts = has_m1 ? 2 : 1;
      mbar_arrive_expect_tx(bar_q, mts * L::kQTile);
      for (int m = 0; m < mts; ++m)
#pragma unroll
        for (int h = 0; h < L::kHalves; ++h)
          tma_load_3d(smem + L::kQ + m * L::kQTile + h * L::kQHalf, &tm_q, bar_q, h * 64,
                      kvh * a.group, (pair * kRowsCta + m * kRowsM) / a.group);
    }
    // block id of page `lane` of tile t; pages past the prefix re-read the tile's
    // first page (their keys are masked)
    auto page_id = [&](int t) {
      const int valid_pages = min(kPagesPerTile, (a.cpl - t * kKeysN) / kPage);
      return lane < kPagesPerTile
                 ? __ldg(a.block_table + t * kPagesPerTile + (lane < valid_pages ? lane : 0))
                 : 0;
    };
    int blk_next = ntiles > 0 ? page_id(t_first) : 0;
    for (int i = 0; i < ntiles; ++i) {
      const int st = i % kStages;
      const int blk = blk_next;
      if (i + 1 < ntiles) blk_next = page_id(t_first + i + 1);  // in flight meanwhile
      if (i >= kStages) {
        bool ok = true;  // lane 0 waits; the decision is the same for the whole warp
        if (lane == 0)
          ok = mbar_wait(&kv_empty[st], ((i / kStages) - 1) & 1, abort_flag, a.status);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      }
      if (lane == 0) mbar_arrive_expect_tx(&kv_full[st], 2 * L::kKVBytes);
      __syncwarp();
      if (lane < kPagesPerTile) {
        uint8_t* dk = smem + L::kK0 + st * L::kKVBytes + lane * (kPage * 128);
        uint8_t* dv = smem + L::kV0 + st * L::kKVBytes + lane * (kPage * 128);
#pragma unroll
        for (int h = 0; h < L::kHalves; ++h) {
          tma_load_3d(dk + h * L::kKVHalf, &tm_k, &kv_full[st], h * 64, kvh, blk * kPage);
          tma_load_3d(dv + h * L::kKVHalf, &tm_v, &kv_full[st], h * 64, kvh, blk * kPage);
        }
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------- MMA issuer --
    if (lane == 0 && ntiles > 0) {
      constexpr uint32_t kIdS = umma_idesc_bf16(128, kKeysN, 0, 0);
      constexpr uint32_t kIdO = umma_idesc_bf16(128, D, 0, 1);
      const int mts = has_m1 ? 2 : 1;
      auto issue_s = [&](int i) {
        const uint32_t k_addr = smem_u32(smem + L::kK0 + (i % kStages) * L::kKVBytes);
        for (int m = 0; m < mts; ++m) {
          const uint32_t q_addr = smem_u32(smem + L::kQ + m * L::kQTile);
          const uint32_t d = tmem + m * 256 + (i & 1) * kKeysN;
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t qo = (k >> 2) * L::kQHalf + (k & 3) * 32;
            const uint32_t ko = (k >> 2) * L::kKVHalf + (k & 3) * 32;
            umma_bf16(d, umma_desc_sw128(q_addr + qo, 16, 1024),
                      umma_desc_sw128(k_addr + ko, 16, 1024), kIdS, k > 0 ? 1u : 0u);
          }
          umma_commit(&s_full[m * 2 + (i & 1)]);
        }
      };
      bool ok = mbar_wait(bar_q, 0, abort_flag, a.status) &&
                mbar_wait(&kv_full[0], 0, abort_flag, a.status);
      if (ok) {
        tc_fence_after();
        issue_s(0);
      }
      for (int i = 0; ok && i < ntiles; ++i) {
        if (i + 1 < ntiles) {
          ok = mbar_wait(&kv_full[(i + 1) % kStages], ((i + 1) / kStages) & 1, abort_flag,
                         a.status);
          if (!ok) break;
          tc_fence_after();
          issue_s(i + 1);  // S buffers (i+1)&1 were last read by PV(i-1), issued earlier
        }
        const uint32_t v_addr = smem_u32(smem + L::kV0 + (i % kStages) * L::kKVBytes);
        for (int m = 0; ok && m < mts; ++m) {
          ok = mbar_wait(&p_full[m * 2 + (i & 1)], (i >> 1) & 1, abort_flag, a.status);
          if (!ok) break;
          tc_fence_after();
          const uint32_t p_tmem = tmem + m * 256 + (i & 1) * kKeysN;
#pragma unroll
          for (int kk = 0; kk < kKeysN / 16; ++kk)
            umma_bf16_tmem_a(tmem + m * 256 + 2 * kKeysN, p_tmem + kk * 8,
                             umma_desc_sw128(v_addr + kk * 16 * 128, L::kKVHalf, 1024), kIdO,
                             (i > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&o_done[m]);
          if (i == ntiles - 1) umma_commit(&o_last[m]);
        }
        if (ok) umma_commit(&kv_empty[i % kStages]);
      }
    }
    __syncwarp();
  }

  // --------------------------------------------------------------- softmax --
  const int wg = warp >> 2;            // softmax warpgroup = M tile (warps 0-7)
  const int row = threadIdx.x & 127;   // TMEM lane == row within the M tile
  const uint32_t t_lane = tmem + wg * 256 + (static_cast<uint32_t>((warp & 3) * 32) << 16);
  const uint32_t tO = t_lane + 2 * kKeysN;
  float m_run = -INFINITY;  // running max, log2 domain
  float l_run = 0.f;
  bool have = false;
  const bool softmax_warp = warp < 8 && (wg == 0 || has_m1);
  if (softmax_warp) {
    bool failed = false;
    for (int i = 0; i < ntiles; ++i) {
      const int tile = t_first + i;
      const bool ok = mbar_wait(&s_full[wg * 2 + (i & 1)], (i >> 1) & 1, abort_flag, a.status);
      if (wg_bar_any(1 + wg, !ok)) {
        failed = true;
        break;
      }
      tc_fence_after();
      float sv[kKeysN];
      tmem_ld64_sync(t_lane + (i & 1) * kKeysN, sv);
      const int valid = a.cpl - tile * kKeysN;
      if (valid < kKeysN) {  // only the prefix's last tile can be partial
#pragma unroll
        for (int j = 0; j < kKeysN; ++j)
          if (j >= valid) sv[j] = -INFINITY;
      }
      // row max of the raw scores as a tree (scale > 0 keeps the order)
      float mx8[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) mx8[j] = sv[j];
#pragma unroll
      for (int j = 8; j < kKeysN; ++j) mx8[j & 7] = fmaxf(mx8[j & 7], sv[j]);
      const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) *
                       a.scale_log2;
      // rescale only when the running max grows by more than 2^8 (always on the
      // first tile, where m_run is -inf); otherwise keep the stale max: P <= 256
      const float m_new = fmaxf(m_run, mx);
      const bool grow = (m_new - m_run) > 8.f;
      float alpha = 1.f;
      if (grow) {
        alpha = fast_exp2(m_run - m_new);
        l_run *= alpha;
        m_run = m_new;
      }
      if (i > 0 && __any_sync(0xffffffffu, grow)) {
        // O must hold PV(i-1) before it is rescaled (the phase is unambiguous: PV(i)
        // cannot complete before this thread has written P(i))
        mbar_wait(&o_done[wg], (i - 1) & 1, abort_flag, a.status);
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tmem_ld32_sync(tO + c * 32, o);
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] *= alpha;
          tmem_st32(tO + c * 32, o);
        }
      }
      // p = 2^(s * scale * log2(e) - m): one FFMA and one ex2 per score
      uint32_t pw[kKeysN / 2];
      float sum4[4] = {0.f, 0.f, 0.f, 0.f};
      const float neg_m = -m_run;
#pragma unroll
      for (int j = 0; j < kKeysN / 2; ++j) {
        const float p0 = fast_exp2(fmaf(sv[2 * j], a.scale_log2, neg_m));
        const float p1 = fast_exp2(fmaf(sv[2 * j + 1], a.scale_log2, neg_m));
        sum4[j & 3] += p0 + p1;
        pw[j] = pack_bf16x2(p0, p1);
      }
      l_run += (sum4[0] + sum4[1]) + (sum4[2] + sum4[3]);
      tmem_st32_u(t_lane + (i & 1) * kKeysN, pw);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full[wg * 2 + (i & 1)]);
    }
    if (!failed && ntiles > 0) {
      // o_done's parity alone cannot tell PV(ntiles-1) from PV(ntiles-2), which may
      // still be running: o_last completes once, after every PV of the range
      const bool ok = mbar_wait(&o_last[wg], 0, abort_flag, a.status);
      have = !wg_bar_any(1 + wg, !ok);
    }
    tc_fence_before();
  }

  // ----------------------------------------- this split's partial -> slot --
  // every MMA of the CTA is complete once both warpgroups saw their last o_done
  // (or have nothing to do): Q and the ring become the staging buffer
  __syncthreads();
  __nv_bfloat16* stage = reinterpret_cast<__nv_bfloat16*>(smem);
  if (softmax_warp) {
    tc_fence_after();
    const float inv_l = have ? 1.f / l_run : 0.f;
    __nv_bfloat16* dst = stage + (wg * kRowsM + row) * L::kStageRow;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      float o[32];
      tmem_ld32_sync(tO + c * 32, o);
#pragma unroll
      for (int j = 0; j < 32; j += 8)
        *reinterpret_cast<uint4*>(dst + c * 32 + j) =
            make_uint4(pack_bf16x2(o[j] * inv_l, o[j + 1] * inv_l),
                       pack_bf16x2(o[j + 2] * inv_l, o[j + 3] * inv_l),
                       pack_bf16x2(o[j + 4] * inv_l, o[j + 5] * inv_l),
                       pack_bf16x2(o[j + 6] * inv_l, o[j + 7] * inv_l));
    }
  }
  // a row with no key in this range (or no query) gets -inf: weight 0 in the merge
  float* s_lse = reinterpret_cast<float*>(smem + L::kLse);
  if (warp < 8) s_lse[wg * kRowsM + row] = (softmax_warp && have) ? m_run + log2f(l_run)
                                                                  : -INFINITY;
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  // coalesced copy-out: a warp writes whole rows (D/8 lanes x 16 bytes each)
  {
    constexpr int kChunks = D / 8;
    const int gshift = __ffs(a.group) - 1;  // group is a power of two
    for (int it = threadIdx.x; it < kRowsCta * kChunks; it += kThreads) {
      const int r = it / kChunks;
      const int c = it % kChunks;
      const int packed = pair * kRowsCta + r;
      const int t = packed >> gshift;
      if (t >= a.total_q) continue;
      const int64_t prow = (static_cast<int64_t>(split) * a.total_q + t) * a.num_q_heads +
                           kvh * a.group + (packed & (a.group - 1));
      *reinterpret_cast<uint4*>(a.part_o + prow * D + c * 8) =
          *reinterpret_cast<const uint4*>(stage + r * L::kStageRow + c * 8);
      if (c == 0) a.part_lse[prow] = s_lse[r];
    }
  }
}

template <int D>
cudaLaunchConfig_t prefix_config(const PrefixArgs& a, cudaStream_t stream,
                                 cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_splits * a.pairs * a.num_kv_heads);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Layout<D>::kDynamic;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 0;
  return cfg;
}

template <int D>
cudaError_t prepare() {
  static std::atomic<uint64_t> attr_done{0};
  return set_smem_once(prefix_attn_kernel<D>, Layout<D>::kDynamic, attr_done);
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
