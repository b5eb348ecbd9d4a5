// decode_cascade.cu — cascade attention for decode-like batches in one kernel.
//
// "vLLM Cascade Attention：用法、场景与原理解析" §八 Step 5: a prefix phase (every query
// of the batch, non-causal, over KV [0, cpl) of block_table row 0), a suffix phase
// (each request, causal, over its own KV [cpl, seq_len)) and merge_attn_states; §五 /
// §十: the prefix is read once for all queries instead of once per request.
//
// A decode batch moves far more suffix bytes than prefix bytes, while the prefix is
// the only dense contraction.  So the SMs take roles inside one grid of one CTA per
// SM (a cooperative launch, so every CTA is resident):
//  * CTAs [0, prefix_ctas) each run one range of the prefix on tcgen05 tensor cores
//    (prefix_range, prefix_body.cuh) and write a partial into slot `split`;
//  * the other CTAs stream the suffix units — one per (request, KV head), all its
//    rows (at most 16 packed (query, head-in-group) rows) in one warp-level MMA tile —
//    split evenly between them, so the prefix's compute and the suffix's HBM streaming
//    overlap on different SMs (the host picks the number of prefix ranges so that the
//    two roles end together);
//  * a grid-wide barrier, then every CTA merges a share of the rows: prefix slots
//    plus the suffix slot, by LSE rescaling, into bf16 out and the natural-log LSE.
//
// Suffix streaming within a CTA: two groups of four warps (warps 0-3 and 4-7), each
// an independent multistage pipeline over its own units.  Lane g of warp 8 walks the
// units of group g, resolves their request metadata and first block ids ahead of
// use, and queues them in shared memory.  A group loads its stages itself with
// 16-byte cp.async (128 threads issuing: on GB300 this path keeps more bytes in flight
// per SM than TMA page boxes do) into 128-byte-swizzled 64-key stages, two stages
// ahead of the one it computes; the first stage of a unit also carries its Q rows.
// Warp w of the group takes keys [16 w, 16 w + 16) of each stage: S = Q K^T and
// O += P V on mma.sync m16n8k16 (bf16 in, fp32 accumulate) fed by ldmatrix, masked
// by the request's causal limit (bottom-right alignment, §四), online softmax in
// base 2; at the unit's end the four warps merge through shared memory and write the
// normalised bf16 rows and their log2-sum-exp.
#include <type_traits>

#include "merge.cuh"
#include "prefix_body.cuh"

namespace csp {
namespace {

constexpr int kThreads = prefix::kThreads;  // 320: ten warps
constexpr int kKeys = 64;                   // keys per suffix stage
constexpr int kPage = 16;
constexpr int kTilePages = kKeys / kPage;
constexpr int kRows = 16;                   // packed rows of a suffix unit (one M tile)
constexpr int kGroups = 2;                  // streaming groups of four warps
constexpr int kWarpScheduler = 8;           // lane g schedules for group g
constexpr int kQueue = 4;                   // units resolved ahead, per group
constexpr int kDescPages = 8;               // block ids resolved ahead: two 64-key tiles

static_assert(kThreads == 320, "ten warps: 8 softmax/streaming, MMA/scheduler, TMA");

// A suffix unit resolved by the scheduler: its request's metadata and the physical
// blocks of its first two tiles.  ntiles < 0: no more units.
struct UnitDesc {
  int r, kvh, q0, q_len, seq_len, ntiles;
  int pages[kDescPages];
  int pad[2];
};

template <int D>
struct SLayout {
  static constexpr int kHalves = D / 64;
  static constexpr int kKVHalf = kKeys * 128;    // 64 keys x 64 features (128 B rows)
  static constexpr int kKV = kHalves * kKVHalf;  // one K (or V) stage
  static constexpr int kQHalf = kRows * 128;
  static constexpr int kQ = kHalves * kQHalf;
  static constexpr int kStage = 2 * kKV + kQ;    // K, V, then Q
  static constexpr int kRing = 221184;           // bytes of stages (216 KB)
  static constexpr int kGroupStages = kRing / kStage / kGroups > 4 ? 4 : kRing / kStage / kGroups;
  static constexpr int kGroupBytes = kGroupStages * kStage;
  // the data area serves both roles: the prefix's Q + ring + staging, or the stages
  static constexpr int kPrefixData = prefix::Layout<D>::kData;
  static constexpr int kData =
      kGroups * kGroupBytes > kPrefixData ? kGroups * kGroupBytes : kPrefixData;
  static constexpr int kPrefixBars = kData;                        // prefix::kBarBytes
  static constexpr int kSuffixBars = kPrefixBars + prefix::kBarBytes;
  static constexpr int kSuffixBarBytes = 1024;
  static constexpr int kDynamic = kSuffixBars + kSuffixBarBytes + 1024;  // + align slack
  static_assert(kGroupStages >= 3, "two stages in flight ahead of the computed one");
  static_assert(kStage % 1024 == 0 && (2 * kKV) % 1024 == 0, "swizzled stage alignment");
  static_assert(2 * kGroups * kQueue * 8 + kGroups * kGroupStages * 8 +
                        kGroups * kQueue * static_cast<int>(sizeof(UnitDesc)) + 32 <=
                    kSuffixBarBytes,
                "suffix barrier area");
  static_assert(kDynamic <= 227 * 1024, "one CTA per SM");
};

// Byte offset of 16-byte chunk c (of D/8) of row `row` in a [halves][rows][128 B]
// tile with the 128-byte swizzle (chunk index XOR row mod 8): conflict-free ldmatrix.
template <int kTileRows>
__device__ __forceinline__ uint32_t sw128(int row, int c) {
  return static_cast<uint32_t>((c >> 3) * (kTileRows * 128) + row * 128 +
                               (((c & 7) ^ (row & 7)) << 4));
}

__device__ __forceinline__ unsigned ld_acquire_gpu_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_gpu_u32(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void group_sync(int g) {
  asm volatile("bar.sync %0, 128;" ::"r"(1 + g) : "memory");
}

// ----------------------------------------------------------------- scheduler --
// Lane g of warp 8 for streaming group g (the two lanes run independently).  The
// suffix units are split evenly over the CTAs that run no prefix range: CTA c of those
// takes units [c*U/n, (c+1)*U/n), its group g every other one of them starting at g.
// As soon as one of the group's queue slots is free (a slot stays taken until the
// group has finished that unit), the lane reads the next unit's request query range
// and length and the block ids of its first two tiles, and posts it.  The block ids
// are read before the request's length is known: entries past the request's pages (up
// to the row stride) are read but never used.  Units without query rows are skipped.
// Ends with an end marker.
__device__ __forceinline__ void schedule_lane(const DecodeArgs& a, int g, uint64_t* q_full,
                                              uint64_t* q_empty, UnitDesc* queue,
                                              volatile int* abort_flag) {
  const PrefixArgs& p = a.pre;
  const int n_units = a.num_reqs * p.num_kv_heads;
  const int page0 = p.cpl / kPage;
  const int n_ctas = static_cast<int>(gridDim.x) - a.prefix_ctas;
  const int c = static_cast<int>(blockIdx.x) - a.prefix_ctas;
  const int u_end = c >= 0 ? static_cast<int>((static_cast<int64_t>(c) + 1) * n_units / n_ctas) : 0;
  int u = c >= 0 ? static_cast<int>(static_cast<int64_t>(c) * n_units / n_ctas) + g : u_end;
  for (int n = 0;; u += kGroups) {
    const int slot = n % kQueue;
    if (n >= kQueue && !mbar_wait(&q_empty[slot], ((n / kQueue) - 1) & 1, abort_flag, p.status))
      return;
    UnitDesc& d = queue[slot];
    if (u >= u_end) {
      d.ntiles = -1;
      mbar_arrive(&q_full[slot]);
      return;
    }
    const int r = u / p.num_kv_heads;
    const int q0 = __ldg(a.cu_seqlens_q + r);
    const int q_len = __ldg(a.cu_seqlens_q + r + 1) - q0;
    const int seq_len = __ldg(a.seq_lens + r);
    const int32_t* bt = a.block_table + static_cast<int64_t>(r) * a.bt_stride;
    int pg[kDescPages];
#pragma unroll
    for (int j = 0; j < kDescPages; ++j)
      pg[j] = __ldg(bt + min(static_cast<int64_t>(page0 + j), a.bt_stride - 1));
    if (q_len <= 0) continue;  // no query rows: nothing to compute or write
    const int nkeys = seq_len - p.cpl;
    d.r = r;
    d.kvh = u - r * p.num_kv_heads;
    d.q0 = q0;
    d.q_len = q_len;
    d.seq_len = seq_len;
    d.ntiles = nkeys > 0 ? (nkeys + kKeys - 1) / kKeys : 0;
#pragma unroll
    for (int j = 0; j < kDescPages; ++j) d.pages[j] = pg[j];
    mbar_arrive(&q_full[slot]);
    ++n;
  }
}

// ------------------------------------------------------------------ streaming --
// Streaming group g (warps 4g .. 4g+3, 128 threads) over the units its scheduler lane
// posts.  A cp.async pipeline of kGroupStages stages: the group issues the tile
// kGroupStages - 1 ahead of the one it computes (one commit group per tile), then
// waits for the computed tile's group and syncs.  Thread t loads the 16-byte chunks
// t, t + 128, ... of the tile's K and V (and, with a unit's first tile, of its Q
// rows); keys past the request and padding rows are zero-filled without a read.
// Returns after the end marker (or an abort).
template <int D>
__device__ __forceinline__ void stream_group(const DecodeArgs& a, int g, uint8_t* gsmem,
                                             uint64_t* q_full, uint64_t* q_empty,
                                             const UnitDesc* queue, uint64_t* st_full,
                                             volatile int* ready_flag,
                                             volatile int* abort_flag) {
  using L = SLayout<D>;
  constexpr int kS = L::kGroupStages;
  constexpr int kChunks = D / 8;          // 16-byte chunks per row
  constexpr int kPer = kKeys * kChunks / 128;   // K (and V) chunks per thread per tile
  constexpr int kQPer = kRows * kChunks / 128;  // Q chunks per thread
  constexpr int kDT = D / 8;              // O n-tiles (8 features each)
  constexpr int kORow = D + 4;            // merge scratch row stride (floats)
  static_assert(4 * kRows * kORow * 4 + 2 * 4 * kRows * 4 <= L::kStage, "merge scratch");
  const PrefixArgs& p = a.pre;
  const int tid = threadIdx.x & 127;
  const int lane = threadIdx.x & 31;
  const int wi = tid >> 5;
  const uint32_t gbase = smem_u32(gsmem);
  const int page0 = p.cpl / kPage;
  const int hkv = p.num_kv_heads;
  bool ok = true;

  // ---- load side: next tile (unit lu, tile lt); block ids of tiles lt, lt+1, lt+2
  int lu = 0, lt = 0, l_nt = 0;
  bool l_end = false;
  int issued = 0;
  int ids0[kTilePages], ids1[kTilePages], ids2[kTilePages];
  const int32_t* l_bt = a.block_table;
  auto far_ids = [&](int tile, int npages, int (&dst)[kTilePages]) {
#pragma unroll
    for (int q = 0; q < kTilePages; ++q) {
      const int pp = page0 + tile * kTilePages + q;
      dst[q] = pp < npages ? __ldg(l_bt + pp) : 0;
    }
  };
  // Issue the next tile if its unit's descriptor is there: `must` waits for it (the
  // group has nothing else to do), otherwise `ready` says whether it was posted.  The
  // tile's loads arrive on the stage's barrier once they have landed.
  auto issue = [&](bool must, bool ready) -> bool {
    if (l_end || !ok) return false;
    if (lt == 0) {
      // start of unit lu: its descriptor (posted by the scheduler lane)
      if (must) {
        ok = warp_mbar_wait(&q_full[lu % kQueue], (lu / kQueue) & 1, abort_flag, p.status);
      } else if (!ready) {
        return false;
      }
      if (ok) {
        const UnitDesc& d = queue[lu % kQueue];
        if (d.ntiles < 0) {
          l_end = true;
        } else {
          l_nt = max(d.ntiles, 1);  // no suffix key: one all-masked (zero-filled) tile
          l_bt = a.block_table + static_cast<int64_t>(d.r) * a.bt_stride;
#pragma unroll
          for (int q = 0; q < kTilePages; ++q) {
            ids0[q] = d.pages[q];
            ids1[q] = d.pages[kTilePages + q];
          }
          if (l_nt > 2) far_ids(2, (d.seq_len + kPage - 1) / kPage, ids2);
        }
      }
    }
    if (!l_end && ok) {
      const UnitDesc& d = queue[lu % kQueue];
      const int seq_len = d.seq_len, kvh = d.kvh;
      const int npages = (seq_len + kPage - 1) / kPage;
      const uint32_t sb = gbase + (issued % kS) * L::kStage;
      const int key0 = p.cpl + lt * kKeys;
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int x = tid + 128 * j;
        const int key = x / kChunks, c = x % kChunks;
        const int pq = key >> 4;
        // pages past the request re-read the tile's first page (its keys are masked)
        const int blk = page0 + lt * kTilePages + pq < npages ? ids0[pq] : ids0[0];
        const bool in = key0 + key < seq_len;
        const int64_t off =
            ((static_cast<int64_t>(blk) * kPage + (key & 15)) * hkv + kvh) * D + c * 8;
        cp_async_16_u32(sb + sw128<kKeys>(key, c), in ? a.k + off : a.k, in ? 16u : 0u);
        cp_async_16_u32(sb + L::kKV + sw128<kKeys>(key, c), in ? a.v + off : a.v,
                        in ? 16u : 0u);
      }
      if (lt == 0) {
        const int rows = d.q_len * p.group;
#pragma unroll
        for (int j = 0; j < kQPer; ++j) {
          const int x = tid + 128 * j;
          const int row = x / kChunks, c = x % kChunks;
          const bool in = row < rows;
          const int qi = row / p.group, hj = row - qi * p.group;
          const int64_t off =
              (static_cast<int64_t>(d.q0 + qi) * p.num_q_heads + kvh * p.group + hj) * D +
              c * 8;
          cp_async_16_u32(sb + 2 * L::kKV + sw128<kRows>(row, c), in ? a.q + off : a.q,
                          in ? 16u : 0u);
        }
      }
      cp_async_mbar_arrive(&st_full[issued % kS]);
      ++issued;
      if (++lt == l_nt) {
        ++lu;
        lt = 0;
      } else {
#pragma unroll
        for (int q = 0; q < kTilePages; ++q) {
          ids0[q] = ids1[q];
          ids1[q] = ids2[q];
        }
        if (lt + 2 < l_nt) far_ids(lt + 2, npages, ids2);
      }
      return true;
    }
    return false;
  };

  // ---- compute side: tile ct of unit cu; per-unit state in registers
  int cu = 0, ct = 0, c_nt = 0;
  int c_seq = 0, c_qlen = 0, c_q0 = 0, c_kvh = 0, rows_valid = 0;
  int pos[2] = {-1, -1};
  float o[kDT][4];
  float m_run[2], l_run[2];
  uint32_t qa[D / 16][4];
  const int kw0 = wi * 16;  // this warp's keys within a stage

  // Thread 0 of the group looks (without waiting) whether the next unit is posted; the
  // group sync publishes its answer, so every thread takes the same branch.
  // (two flags, alternating by tile, so the next answer never overwrites one a slow
  // warp has yet to read)
  auto probe_next = [&](int item) {
    if (tid == 0)
      ready_flag[item & 1] = (l_end || lt != 0) ? 1
                                       : (mbar_test_wait(&q_full[lu % kQueue], (lu / kQueue) & 1)
                                              ? 1 : 0);
  };
  issue(true, false);
  for (int s = 1; s < kS - 1; ++s) issue(false, false);
  for (int item = 0; ok; ++item) {
    if (item == issued) {
      // nothing loaded is left to compute: wait for the next unit (or the end)
      issue(true, false);
      if (!ok || item == issued) break;
    }
    probe_next(item);
    group_sync(g);  // the stage of tile item - 1 is no longer read by anyone: refill it
    issue(false, ready_flag[item & 1] != 0);
    // this tile's chunks from every thread have landed
    if (!(ok = warp_mbar_wait(&st_full[item % kS], (item / kS) & 1, abort_flag, p.status))) break;
    const uint32_t kb = gbase + (item % kS) * L::kStage;
    const uint32_t vb = kb + L::kKV;
    if (ct == 0) {
      const UnitDesc& d = queue[cu % kQueue];
      c_nt = max(d.ntiles, 1);
      c_seq = d.seq_len;
      c_qlen = d.q_len;
      c_q0 = d.q0;
      c_kvh = d.kvh;
      rows_valid = c_qlen * p.group;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int rho = (lane >> 2) + 8 * h;
        pos[h] = rho < rows_valid ? c_seq - c_qlen + rho / p.group : -1;
        m_run[h] = -INFINITY;
        l_run[h] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < kDT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
      const uint32_t qb = kb + 2 * L::kKV;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int row = (lane & 7) + ((lane >> 3) & 1) * 8;
        const int c = kk * 2 + (lane >> 4);
        ldmatrix_x4(qb + sw128<kRows>(row, c), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
      }
    }
    // S = Q K^T over this warp's 16 keys (two n-tiles of 8)
    float sacc[2][4];
#pragma unroll
    for (int i = 0; i < 2; ++i) sacc[i][0] = sacc[i][1] = sacc[i][2] = sacc[i][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int key = kw0 + (lane & 7) + (lane >> 4) * 8;
      const int c = kk * 2 + ((lane >> 3) & 1);
      uint32_t b0, b1, b2, b3;
      ldmatrix_x4(kb + sw128<kKeys>(key, c), b0, b1, b2, b3);
      mma_bf16_16816(sacc[0], qa[kk], b0, b1);
      mma_bf16_16816(sacc[1], qa[kk], b2, b3);
    }
    // mask (keys past the request, and the causal limit), online softmax in base 2
    const int key0 = p.cpl + ct * kKeys + kw0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float mx = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int kabs = key0 + nt * 8 + (lane & 3) * 2 + e;
          float& sref = sacc[nt][2 * h + e];
          sref = (kabs < c_seq && kabs <= pos[h]) ? sref * p.scale_log2 : -INFINITY;
          mx = fmaxf(mx, sref);
        }
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_run[h], mx);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = fast_exp2(m_run[h] - m_use);
      float sum = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float& sref = sacc[nt][2 * h + e];
          sref = fast_exp2(sref - m_use);
          sum += sref;
        }
      }
      l_run[h] = l_run[h] * alpha + sum;
      m_run[h] = m_new;
#pragma unroll
      for (int dt = 0; dt < kDT; ++dt) {
        o[dt][2 * h] *= alpha;
        o[dt][2 * h + 1] *= alpha;
      }
    }
    // O += P V over the same 16 keys
    uint32_t pa[4];
    pa[0] = pack_bf16x2(sacc[0][0], sacc[0][1]);
    pa[1] = pack_bf16x2(sacc[0][2], sacc[0][3]);
    pa[2] = pack_bf16x2(sacc[1][0], sacc[1][1]);
    pa[3] = pack_bf16x2(sacc[1][2], sacc[1][3]);
#pragma unroll
    for (int dp = 0; dp < kDT / 2; ++dp) {
      const int key = kw0 + (lane & 7) + ((lane >> 3) & 1) * 8;
      const int c = dp * 2 + (lane >> 4);
      uint32_t b0, b1, b2, b3;
      ldmatrix_x4_trans(vb + sw128<kKeys>(key, c), b0, b1, b2, b3);
      mma_bf16_16816(o[2 * dp], pa, b0, b1);
      mma_bf16_16816(o[2 * dp + 1], pa, b2, b3);
    }
    if (++ct < c_nt) continue;

    // ---- the unit's last tile: the four warps' (max, sum, O) -> one normalised
    // partial per row, through this stage's memory (nobody reads its K/V any more
    // once the group has synced; the next write to it comes after the next sync)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
    }
    group_sync(g);
    float* s_o = reinterpret_cast<float*>(gsmem + (item % kS) * L::kStage);  // [4][16][kORow]
    float* s_m = s_o + 4 * kRows * kORow;                                    // [4][16]
    float* s_l = s_m + 4 * kRows;                                            // [4][16]
    if ((lane & 3) == 0) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        s_m[wi * kRows + (lane >> 2) + 8 * h] = m_run[h];
        s_l[wi * kRows + (lane >> 2) + 8 * h] = l_run[h];
      }
    }
    group_sync(g);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int rr = (lane >> 2) + 8 * h;
      if (rr >= rows_valid) continue;
      float mg = -INFINITY;
#pragma unroll
      for (int w = 0; w < 4; ++w) mg = fmaxf(mg, s_m[w * kRows + rr]);
      const float sc = (m_run[h] == -INFINITY) ? 0.f : fast_exp2(m_run[h] - mg);
      float* dst = s_o + (wi * kRows + rr) * kORow;
#pragma unroll
      for (int dt = 0; dt < kDT; ++dt) {
        const int d = dt * 8 + (lane & 3) * 2;
        *reinterpret_cast<float2*>(dst + d) = make_float2(o[dt][2 * h] * sc, o[dt][2 * h + 1] * sc);
      }
    }
    group_sync(g);
    const int64_t slot_rows = static_cast<int64_t>(p.n_splits) * p.total_q * p.num_q_heads;
    // warp wi finalises rows wi, wi + 4, ...; lane c owns features [4c, 4c + 4)
    for (int rr = wi; rr < rows_valid; rr += 4) {
      float mg = -INFINITY;
#pragma unroll
      for (int w = 0; w < 4; ++w) mg = fmaxf(mg, s_m[w * kRows + rr]);
      float lsum = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float mw = s_m[w * kRows + rr];
        lsum += (mw == -INFINITY) ? 0.f : s_l[w * kRows + rr] * fast_exp2(mw - mg);
      }
      const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
      const int qi = rr / p.group, j = rr - qi * p.group;
      const int64_t prow =
          slot_rows + static_cast<int64_t>(c_q0 + qi) * p.num_q_heads + c_kvh * p.group + j;
      if (lane < D / 4) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float4 v =
              *reinterpret_cast<const float4*>(s_o + (w * kRows + rr) * kORow + lane * 4);
          acc.x += v.x;
          acc.y += v.y;
          acc.z += v.z;
          acc.w += v.w;
        }
        store_bf16x4(p.part_o + prow * D + lane * 4,
                     make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
      }
      if (lane == 0) p.part_lse[prow] = lsum > 0.f ? mg + log2f(lsum) : -INFINITY;
    }
    // the unit is done: its queue slot goes back to the scheduler lane
    if (tid == 0) mbar_arrive(&q_empty[cu % kQueue]);
    ++cu;
    ct = 0;
  }
  cp_async_wait<0>();
}

// -------------------------------------------------------------------- merge --
// merge_attn_states for one output row with 16 lanes (a half warp): slots [0, n) of
// the workspace, n <= kDecodeMaxParts.  Lane i holds the weight of slot i and
// features [i*D/16, (i+1)*D/16).  Every slot's loads are issued before any is used,
// so a row costs one round trip to L2.  An empty slot (lse -inf) gets weight 0 and
// whatever it holds never mixes in.
template <int D>
__device__ __forceinline__ void merge_row_half(const DecodeArgs& a, int64_t row, int n,
                                               int hl) {
  constexpr int kF = D / 16;  // features per lane: 8 (16 bytes) or 4 (8 bytes)
  using Vec = typename std::conditional<kF == 8, uint4, uint2>::type;
  static_assert(kDecodeMaxParts <= 16, "one slot weight per lane of a half warp");
  const PrefixArgs& p = a.pre;
  const int64_t rows = static_cast<int64_t>(p.total_q) * p.num_q_heads;
  const float lw = hl < n ? __ldcg(p.part_lse + hl * rows + row) : -INFINITY;
  Vec v[kDecodeMaxParts];
  const __nv_bfloat16* base = p.part_o + row * D + hl * kF;
#pragma unroll
  for (int s = 0; s < kDecodeMaxParts; ++s)
    if (s < n) v[s] = __ldcg(reinterpret_cast<const Vec*>(base + s * rows * D));
  const unsigned mask = 0xffffu << (threadIdx.x & 16);
  float mx = lw;
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(mask, mx, o, 16));
  const float w = (mx == -INFINITY || lw == -INFINITY) ? 0.f : fast_exp2(lw - mx);
  float wsum = w;
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) wsum += __shfl_xor_sync(mask, wsum, o, 16);
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  float acc[kF];
#pragma unroll
  for (int f = 0; f < kF; ++f) acc[f] = 0.f;
#pragma unroll
  for (int s = 0; s < kDecodeMaxParts; ++s) {
    const float ws = __shfl_sync(mask, w, s, 16) * inv;
    if (s < n && ws != 0.f) {
      const uint32_t* u = reinterpret_cast<const uint32_t*>(&v[s]);
#pragma unroll
      for (int f = 0; f < kF / 2; ++f) {
        const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[f]));
        acc[2 * f] = fmaf(ws, x.x, acc[2 * f]);
        acc[2 * f + 1] = fmaf(ws, x.y, acc[2 * f + 1]);
      }
    }
  }
  Vec o;
  uint32_t* ou = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
  for (int f = 0; f < kF / 2; ++f) ou[f] = pack_bf16x2(acc[2 * f], acc[2 * f + 1]);
  *reinterpret_cast<Vec*>(a.out + row * D + hl * kF) = o;
  if (hl == 0 && a.lse != nullptr)
    a.lse[row] = wsum > 0.f ? (mx + log2f(wsum)) * 0.69314718055994531f : -INFINITY;
}


// ------------------------------------------------------------------ the kernel --
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    decode_cascade_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const DecodeArgs a) {
  using L = SLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const PrefixArgs& p = a.pre;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // generation of the grid barrier at the end (read now, off the critical path)
  const unsigned g0 = threadIdx.x == 0 ? ld_acquire_gpu_u32(a.bar_gen) : 0u;

  // ---- role 1: one range of the prefix phase (tcgen05)
  if (static_cast<int>(blockIdx.x) < a.prefix_ctas) {
    const int b = blockIdx.x;
    const int split = b % p.n_splits;
    const int pair = (b / p.n_splits) % p.pairs;
    const int kvh = b / (p.n_splits * p.pairs);
    const int t_first = split * a.key_tiles / p.n_splits;
    const int t_last = (split + 1) * a.key_tiles / p.n_splits;
    prefix::prefix_range<D>(&tm_q, &tm_k, &tm_v, p, kvh, pair, split, t_first, t_last, smem,
                            reinterpret_cast<uint64_t*>(smem + L::kPrefixBars));
    // the staging buffer was read through the generic proxy and TMA wrote the stages;
    // the suffix role below rewrites the same memory
    fence_proxy_async_smem();
    __syncthreads();
  }

  // ---- role 2: suffix units from the shared counter, two streaming groups
  {
    constexpr int kS = L::kGroupStages;
    uint64_t* q_full = reinterpret_cast<uint64_t*>(smem + L::kSuffixBars);  // [2][kQueue]
    uint64_t* q_empty = q_full + kGroups * kQueue;                           // [2][kQueue]
    uint64_t* st_full = q_empty + kGroups * kQueue;                          // [2][kS]
    UnitDesc* queue = reinterpret_cast<UnitDesc*>(st_full + kGroups * kS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(queue + kGroups * kQueue);
    volatile int* ready_flag = abort_flag + 1;                               // [2][2]
    if (threadIdx.x == 0) {
      for (int i = 0; i < kGroups * kQueue; ++i) {
        mbar_init(&q_full[i], 1);
        mbar_init(&q_empty[i], 1);
      }
      for (int i = 0; i < kGroups * kS; ++i) mbar_init(&st_full[i], 128);  // group threads
      *abort_flag = 0;
      fence_mbarrier_init();
    }
    __syncthreads();
    if (warp == kWarpScheduler) {
      if (lane < kGroups)
        schedule_lane(a, lane, q_full + lane * kQueue, q_empty + lane * kQueue,
                      queue + lane * kQueue, abort_flag);
    } else if (warp < 4 * kGroups) {
      const int g = warp >> 2;
      stream_group<D>(a, g, smem + g * L::kGroupBytes, q_full + g * kQueue,
                      q_empty + g * kQueue, queue + g * kQueue, st_full + g * kS,
                      ready_flag + 2 * g, abort_flag);
    }
  }

  // ---- grid-wide barrier: every partial of the call is written.  The arrival is one
  // acquire-release add (the CTA barrier before it makes every thread's partial
  // stores part of what it releases); the last CTA advances the generation, which the
  // others read at their start (no CTA can advance it before every CTA has arrived).
  __syncthreads();
  if (threadIdx.x == 0) {
    const int old = atomic_add_acq_rel_gpu(a.bar_count, 1);
    if (old == static_cast<int>(gridDim.x) - 1) {
      st_release_gpu_u32(a.bar_gen, g0 + 1u);
      // nothing reads these again in this call: zero for the next one
      *a.bar_count = 0;
      *a.work_counter = 0;
    } else {
      const unsigned long long t0 = global_timer_ns();
      while (ld_acquire_gpu_u32(a.bar_gen) == g0) {
        if (global_timer_ns() - t0 > kWaitLimitNs) {
          atomicCAS(p.status, 0, kErrTimeout);
          break;
        }
        __nanosleep(64);
      }
    }
  }
  __syncthreads();

  // ---- merge_attn_states: prefix slots [0, n_splits) and the suffix slot n_splits
  {
    const int rows = p.total_q * p.num_q_heads;
    const int halves = kThreads / 16;
    for (int row = blockIdx.x * halves + (threadIdx.x >> 4); row < rows;
         row += gridDim.x * halves)
      merge_row_half<D>(a, row, p.n_splits + 1, threadIdx.x & 15);
  }
}

template <int D>
cudaError_t launch_decode_d(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                            const CUtensorMap& tm_v, const DecodeArgs& a, int grid,
                            cudaStream_t stream) {
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = set_smem_once(decode_cascade_kernel<D>, SLayout<D>::kDynamic, attr_done);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = SLayout<D>::kDynamic;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  // every CTA must be resident: the grid-wide barrier waits for all of them
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_cascade_kernel<D>, tm_q, tm_k, tm_v, a);
}

}  // namespace

cudaError_t launch_decode(int head_dim, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                          const CUtensorMap& tm_v, const DecodeArgs& a, int grid,
                          cudaStream_t stream) {
  if (head_dim == 64) return launch_decode_d<64>(tm_q, tm_k, tm_v, a, grid, stream);
  return launch_decode_d<128>(tm_q, tm_k, tm_v, a, grid, stream);
}

}  // namespace csp
