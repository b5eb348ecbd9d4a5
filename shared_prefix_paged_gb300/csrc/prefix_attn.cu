// prefix_attn.cu — the prefix phase of cascade attention on tcgen05 tensor cores.
//
// "vLLM Cascade Attention：用法、场景与原理解析" §五 and §十: the prefix phase treats
// every query of the batch as one sequence (cu_seqlens_q = [0, total_q]) so that one
// load of a shared KV page serves a whole tile of queries, and §八 Step 5 Phase 1:
// non-causal attention over KV [0, common_prefix_len) read through block_table[:1].
//
// GB300 design (not the FlashAttention tiling the page describes):
//  * M tile = 128 packed rows (token, head-in-group) of ONE KV head, so the GQA
//    heads that share a KV head share every K/V tile;
//  * K and V pages (16 tokens x 64 features per box, 128-byte swizzle) are staged
//    into shared memory by TMA, 8 pages per 128-key tile, double buffered;
//  * S = Q K^T and O += P V run as tcgen05.mma (M=128, N=128 or D, K=16 steps) with
//    fp32 accumulators in TMEM (S: columns 0-127, O: columns 128-255);
//  * four softmax warps own one TMEM lane (row) per thread: they read S with
//    tcgen05.ld, apply the online softmax in base 2, rescale O in TMEM only when the
//    running max grows by more than 2^8, and write P (bf16) into shared memory in
//    the 128-byte-swizzled K-major layout the PV MMA reads;
//  * warp 4 is the TMA producer; thread 0 issues the MMAs.
//  * the prefix length is split across CTAs for occupancy; each CTA writes a
//    normalised fp32 partial and its log2-sum-exp, merged by the combine kernel.
#include "common.cuh"
#include "kernels.cuh"

namespace csp {
namespace {

constexpr int kRowsM = 128;     // packed rows per CTA
constexpr int kKeysN = 128;     // keys per tile
constexpr int kPage = 16;       // tokens per KV page
constexpr int kPagesPerTile = kKeysN / kPage;
constexpr int kHalfBytes = 128 * 128;   // 128 rows x 64 bf16 (one swizzle-128 column block)
constexpr int kThreads = 160;           // 4 softmax warps + 1 producer warp

template <int D>
struct Layout {
  static constexpr int kHalves = D / 64;
  static constexpr int kTileBytes = kHalves * kHalfBytes;   // Q tile, or one K / V tile
  static constexpr int kQ = 0;
  static constexpr int kK0 = kQ + kTileBytes;
  static constexpr int kV0 = kK0 + 2 * kTileBytes;
  static constexpr int kP = kV0 + 2 * kTileBytes;
  static constexpr int kBar = kP + 2 * kHalfBytes;
  static constexpr int kEnd = kBar + 128;
  static constexpr int kDynamic = kEnd + 1024;   // slack to align the base to 1024 bytes
};

__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Barrier over the 128 softmax threads that also ORs a predicate across them.
__device__ __forceinline__ bool softmax_bar_any(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred))
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
  uint8_t* sQ = smem + L::kQ;
  uint8_t* sP = smem + L::kP;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* bar_q = bars + 0;
  uint64_t* bar_kv = bars + 1;    // [2] tile loaded
  uint64_t* bar_free = bars + 3;  // [2] PV of the tile in this stage finished
  uint64_t* bar_s = bars + 5;     // S of the current tile ready in TMEM
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 6);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 7);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int mt = blockIdx.x % a.m_tiles;
  const int rest = blockIdx.x / a.m_tiles;
  const int split = rest % a.n_splits;
  const int kvh = rest / a.n_splits;
  const int key_tiles = (a.cpl + kKeysN - 1) / kKeysN;
  const int t_first = split * a.tiles_per_split;
  const int t_last = min(t_first + a.tiles_per_split, key_tiles);
  const int ntiles = t_last - t_first;

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    mbar_init(&bar_kv[0], 1);
    mbar_init(&bar_kv[1], 1);
    mbar_init(&bar_free[0], 1);
    mbar_init(&bar_free[1], 1);
    mbar_init(bar_s, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------------ producer --
    if (lane == 0) {
      prefetch_tensormap(&tm_q);
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_v);
      mbar_arrive_expect_tx(bar_q, L::kTileBytes);
#pragma unroll
      for (int h = 0; h < L::kHalves; ++h)
        tma_load_3d(sQ + h * kHalfBytes, &tm_q, bar_q, h * 64, kvh * a.group,
                    mt * (kRowsM / a.group));
    }
    for (int i = 0; i < ntiles; ++i) {
      const int s = i & 1;
      const int tile = t_first + i;
      const int valid_pages = min(kPagesPerTile, (a.cpl - tile * kKeysN) / kPage);
      int blk = 0;
      if (lane < kPagesPerTile) {
        // pages past the prefix re-read the tile's first page; their keys are masked
        const int page = tile * kPagesPerTile + (lane < valid_pages ? lane : 0);
        blk = __ldg(a.block_table + page);
      }
      if (i >= 2 && !mbar_wait(&bar_free[s], ((i >> 1) - 1) & 1, abort_flag, a.status)) break;
      if (lane == 0) mbar_arrive_expect_tx(&bar_kv[s], 2 * L::kTileBytes);
      __syncwarp();
      if (lane < kPagesPerTile) {
        uint8_t* dk = smem + L::kK0 + s * L::kTileBytes + lane * (kPage * 128);
        uint8_t* dv = smem + L::kV0 + s * L::kTileBytes + lane * (kPage * 128);
#pragma unroll
        for (int h = 0; h < L::kHalves; ++h) {
          tma_load_3d(dk + h * kHalfBytes, &tm_k, &bar_kv[s], h * 64, kvh, blk * kPage);
          tma_load_3d(dv + h * kHalfBytes, &tm_v, &bar_kv[s], h * 64, kvh, blk * kPage);
        }
      }
    }
  } else {
    // ------------------------------------------------- softmax + MMA issue --
    const int row = threadIdx.x;  // TMEM lane == packed row within the tile
    const uint32_t t_warp = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const uint32_t tS = t_warp;
    const uint32_t tO = t_warp + 128;
    constexpr uint32_t kIdS = umma_idesc_bf16(128, kKeysN, 0, 0);
    constexpr uint32_t kIdO = umma_idesc_bf16(128, D, 0, 1);
    const uint32_t q_addr = smem_u32(sQ);
    const uint32_t p_addr = smem_u32(sP);
    float m_run = -INFINITY;  // running max, log2 domain
    float l_run = 0.f;
    bool failed = false;

    for (int i = 0; i < ntiles; ++i) {
      const int s = i & 1;
      const int tile = t_first + i;
      if (threadIdx.x == 0) {
        bool ok = (i > 0) || mbar_wait(bar_q, 0, abort_flag, a.status);
        ok = ok && mbar_wait(&bar_kv[s], (i >> 1) & 1, abort_flag, a.status);
        if (ok) {
          tc_fence_after();
          const uint32_t k_addr = smem_u32(smem + L::kK0 + s * L::kTileBytes);
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = (k >> 2) * kHalfBytes + (k & 3) * 32;
            umma_bf16(tmem, umma_desc_sw128(q_addr + off, 16, 1024),
                      umma_desc_sw128(k_addr + off, 16, 1024), kIdS, k > 0 ? 1u : 0u);
          }
          umma_commit(bar_s);
        }
      }
      const bool ok = mbar_wait(bar_s, i & 1, abort_flag, a.status);
      if (softmax_bar_any(!ok)) {
        failed = true;
        break;
      }
      tc_fence_after();

      float sv[kKeysN];
      tmem_ld128_sync(tS, sv);

      const int valid = min(kKeysN, a.cpl - tile * kKeysN);
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < kKeysN; ++j) {
        sv[j] = (j < valid) ? sv[j] * a.scale_log2 : -INFINITY;
        mx = fmaxf(mx, sv[j]);
      }
      // Rescale only when the running max grows by more than 2^8 (always on the
      // first tile, where m_run is -inf); otherwise keep the stale max: P <= 256.
      const float m_new = fmaxf(m_run, mx);
      const bool grow = (m_new - m_run) > 8.f;
      float alpha = 1.f;
      if (grow) {
        alpha = exp2f(m_run - m_new);
        l_run *= alpha;
        m_run = m_new;
      }
      // tcgen05.ld / st are warp-collective: the whole warp rescales if any lane grew.
      // O of the earlier tiles is complete here (bar_s covers every earlier MMA).
      if (i > 0 && __any_sync(0xffffffffu, grow)) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tmem_ld32_sync(tO + c * 32, o);
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] *= alpha;
          tmem_st32(tO + c * 32, o);
        }
        tmem_wait_st();
      }

      // P = exp2(s - m), bf16, into the swizzled K-major P tile (two 64-key halves)
      float sum = 0.f;
#pragma unroll
      for (int c = 0; c < kKeysN / 8; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p0 = exp2f(sv[c * 8 + 2 * e] - m_run);
          const float p1 = exp2f(sv[c * 8 + 2 * e + 1] - m_run);
          sum += p0 + p1;
          w[e] = pack_bf16x2(p0, p1);
        }
        const int half = c >> 3, chunk = c & 7;
        uint8_t* dst = sP + half * kHalfBytes + row * 128 + ((chunk ^ (row & 7)) << 4);
        *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
      }
      l_run += sum;
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar_sync(1, 128);
      if (threadIdx.x == 0) {
        tc_fence_after();
        const uint32_t v_addr = smem_u32(smem + L::kV0 + s * L::kTileBytes);
#pragma unroll
        for (int k = 0; k < kKeysN / 16; ++k) {
          const uint32_t aoff = (k >> 2) * kHalfBytes + (k & 3) * 32;
          umma_bf16(tmem + 128, umma_desc_sw128(p_addr + aoff, 16, 1024),
                    umma_desc_sw128(v_addr + k * 16 * 128, kHalfBytes, 1024), kIdO,
                    (i > 0 || k > 0) ? 1u : 0u);
        }
        umma_commit(&bar_free[s]);
      }
    }

    if (!failed && ntiles > 0) {
      const int last = ntiles - 1;
      const bool ok = mbar_wait(&bar_free[last & 1], (last >> 1) & 1, abort_flag, a.status);
      failed = softmax_bar_any(!ok);
    }
    if (!failed && ntiles > 0) {
      tc_fence_after();
      const int packed = mt * kRowsM + row;
      const int t = packed / a.group;
      const int h = kvh * a.group + packed % a.group;
      const bool live = t < a.total_q;
      const float inv_l = 1.f / l_run;
      const size_t prow = (static_cast<size_t>(split) * a.total_q + t) * a.num_q_heads + h;
      float* dst = a.part_o + prow * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float o[32];
        tmem_ld32_sync(tO + c * 32, o);
        if (live) {
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4*>(dst + c * 32 + j) =
                make_float4(o[j] * inv_l, o[j + 1] * inv_l, o[j + 2] * inv_l, o[j + 3] * inv_l);
        }
      }
      if (live) a.part_lse[prow] = m_run + log2f(l_run);
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

}  // namespace

size_t prefix_smem_bytes(int head_dim) {
  return head_dim == 64 ? Layout<64>::kDynamic : Layout<128>::kDynamic;
}

template <int D>
static cudaError_t launch_prefix_d(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                   const CUtensorMap& tm_v, const PrefixArgs& a,
                                   cudaStream_t stream) {
  const int smem = Layout<D>::kDynamic;
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = set_smem_once(prefix_attn_kernel<D>, smem, attr_done);
  if (e != cudaSuccess) return e;
  const int grid = a.m_tiles * a.n_splits * a.num_kv_heads;
  prefix_attn_kernel<D><<<grid, kThreads, smem, stream>>>(tm_q, tm_k, tm_v, a);
  return cudaGetLastError();
}

cudaError_t launch_prefix(int head_dim, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                          const CUtensorMap& tm_v, const PrefixArgs& a, cudaStream_t stream) {
  if (head_dim == 64) return launch_prefix_d<64>(tm_q, tm_k, tm_v, a, stream);
  return launch_prefix_d<128>(tm_q, tm_k, tm_v, a, stream);
}

}  // namespace csp
