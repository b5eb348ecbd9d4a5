// decode_cascade.cu — cascade attention for decode-like batches in one kernel.
//
// "vLLM Cascade Attention：用法、场景与原理解析" §八 Step 5: a prefix phase (every query
// of the batch, non-causal, over KV [0, cpl) of block_table row 0), a suffix phase
// (each request, causal, over its own KV [cpl, seq_len)) and merge_attn_states; §五 /
// §十: the prefix is read once for all queries instead of once per request.
//
// A decode batch moves far more suffix bytes than prefix bytes, while the prefix is
// the only dense contraction.  On GB300 a single SM pulls only ~30-40 GB/s from HBM or
// L2 through cp.async or page-sized TMA boxes, so the whole GPU's bandwidth is there
// only while every SM streams.  So the SMs share the work inside one grid of one CTA
// per SM (a cooperative launch, so every CTA is resident):
//  * CTAs [0, prefix_ctas) each first run one range of the prefix on tcgen05 tensor
//    cores (prefix_range, prefix_body.cuh) and write a partial into slot `split`;
//    then, like every other CTA, they stream suffix units;
//  * a suffix unit is one (request, KV head): all its rows (at most 16 packed
//    (query, head-in-group) rows) in one warp-level MMA tile.  Each prefix CTA takes
//    prefix_units of them, the other CTAs share the rest evenly; the host picks the
//    number of prefix ranges and prefix_units so that every CTA ends together;
//  * a grid-wide barrier, then every CTA merges an equal share of the rows (prefix
//    slots plus the suffix slot, by LSE rescaling) into bf16 out and the natural-log
//    LSE: one round trip to L2 per row, spread over every SM.
//
// Suffix streaming within a CTA: warp 8 produces ring items (two 64-key tiles of a
// unit, loaded by TMA) and warps 0-7 compute them on mma.sync (see produce_items and
// consume_items).
#include <type_traits>

#include "merge.cuh"
#include "prefix_body.cuh"

namespace csp {
namespace {

constexpr int kThreads = prefix::kThreads;  // 352: eleven warps
constexpr int kKeys = 64;                   // keys per suffix stage
constexpr int kPage = 16;
constexpr int kTilePages = kKeys / kPage;
constexpr int kRows = 16;                   // packed rows of a suffix unit (one M tile)
constexpr int kStreamWarps = 8;             // warps 0-7 stream the suffix
constexpr int kWarpScheduler = 8;           // produces the suffix items
constexpr int kMergeBarOff = 512;           // merge barrier within the suffix barrier area

static_assert(kThreads == 352, "eleven warps: 8 softmax/streaming, 2 MMA (one the scheduler), loader");

template <int D>
struct SLayout {
  static constexpr int kHalves = D / 64;
  static constexpr int kKV = kKeys * D * 2;  // one K (or V) stage: [page][half][16 keys][128 B]
  static constexpr int kQHalf = kRows * 128;
  static constexpr int kQ = kHalves * kQHalf;
  static constexpr int kStage = 2 * kKV + kQ;    // K, V, then Q
  static constexpr int kItem = 2 * kStage;       // two tiles of one unit
  static constexpr int kRing = 221184;           // bytes of items (216 KB)
  static constexpr int kSlots = kRing / kItem > 6 ? 6 : kRing / kItem;
  // the data area serves both roles: the prefix's Q + ring + staging, or the items
  static constexpr int kPrefixData = prefix::Layout<D>::kData;
  static constexpr int kData = kSlots * kItem > kPrefixData ? kSlots * kItem : kPrefixData;
  static constexpr int kPrefixBars = kData;                        // prefix::kBarBytes
  static constexpr int kSuffixBars = kPrefixBars + prefix::kBarBytes;
  static constexpr int kSuffixBarBytes = 1024;
  static constexpr int kDynamic = kSuffixBars + kSuffixBarBytes + 1024;  // + align slack
  static_assert(kSlots >= 3, "two items in flight ahead of the computed one");
  static_assert(kStage % 1024 == 0 && (2 * kKV) % 1024 == 0, "swizzled stage alignment");
  static_assert(2 * kSlots * 8 + kSlots * 32 + 16 <= kSuffixBarBytes, "suffix barrier area");
  static_assert(kDynamic <= 227 * 1024, "one CTA per SM");
};

// Byte offset of 16-byte chunk c (of D/8) of row `row` in a [halves][rows][128 B]
// tile with the 128-byte swizzle (chunk index XOR row mod 8): conflict-free ldmatrix.
template <int kTileRows>
__device__ __forceinline__ uint32_t sw128(int row, int c) {
  return static_cast<uint32_t>((c >> 3) * (kTileRows * 128) + row * 128 +
                               (((c & 7) ^ (row & 7)) << 4));
}

// The same for a K or V stage as the page boxes leave it: [page][half][16 keys][128 B]
// (one box per page brings both feature halves), swizzled by the row's index.
template <int D>
__device__ __forceinline__ uint32_t kv_off(int key, int c) {
  const int r = (key >> 4) * (16 * (D / 64)) + (c >> 3) * 16 + (key & 15);
  return static_cast<uint32_t>(r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ unsigned ld_acquire_gpu_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_gpu_u32(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// the streaming warps of one unit group: named barrier 1 + group, kWPU warps
template <int kWPU>
__device__ __forceinline__ void group_sync(int group) {
  asm volatile("bar.sync %0, %1;" ::"r"(1 + group), "r"(kWPU * 32) : "memory");
}

// ------------------------------------------------------------------ streaming --
// The CTA's suffix units, two 64-key tiles of a unit at a time.  An "item" is a pair
// of stages holding tiles t and t + 1 of one unit (the second left empty when the
// unit has a single tile left); a unit's first item also carries its Q rows.  Items
// go through a ring of kSlots in shared memory:
//  * warp 8 produces them.  It walks the CTA's units (see unit_range), reads each
//    request's query range, length and block ids (lane j the id of the item's page j,
//    one item ahead), and fills a free slot: lane j < 16 issues one TMA box of the
//    item's K or V (one page of one KV head, both feature halves), and the lanes copy
//    the Q rows with 16-byte cp.async (rows past the unit's are zero-filled without a
//    read).  A page past the request re-reads the item's first page (its keys are
//    masked); the item's descriptor tells the consumers which unit and tiles it holds.
//  * warps 0-7 consume them: warps 0-3 compute the item's first tile and warps 4-7 its
//    second, warp w taking keys [16 (w % 4), 16 (w % 4) + 16): S = Q K^T and O += P V
//    on mma.sync m16n8k16 (bf16 in, fp32 accumulate) fed by ldmatrix, masked by the
//    request's causal limit (bottom-right alignment, §四), online softmax in base 2.
//    V rows past the request are zeroed first (a TMA page holds whatever the cache
//    has there).  At the unit's end the eight warps merge through the item's memory
//    and write the normalised bf16 rows and their log2-sum-exp into the suffix slot.
// Loads never hold up the computing warps: the producer alone waits for free slots.
struct ItemDesc {
  int q0, q_len, seq_len, kvh, ntiles, t0, pad0, pad1;  // ntiles < 0: no more items
};

// The CTA's units: a CTA that ran a prefix range takes the next prefix_units units in
// CTA order after it; the remaining units are split evenly over the other CTAs (CTA c
// of those n takes units [c*R/n, (c+1)*R/n) of the R left).
__device__ __forceinline__ void unit_range(const DecodeArgs& a, int& u_begin, int& u_end) {
  const int n_units = a.num_reqs * a.pre.num_kv_heads;
  const int b = static_cast<int>(blockIdx.x);
  const int64_t pre_units =
      min(static_cast<int64_t>(a.prefix_ctas) * a.prefix_units, static_cast<int64_t>(n_units));
  if (b < a.prefix_ctas) {
    u_begin = static_cast<int>(min(static_cast<int64_t>(b) * a.prefix_units, pre_units));
    u_end = static_cast<int>(min(static_cast<int64_t>(b + 1) * a.prefix_units, pre_units));
  } else {
    const int64_t rest = n_units - pre_units;
    const int n_ctas = static_cast<int>(gridDim.x) - a.prefix_ctas;
    const int c = b - a.prefix_ctas;
    u_begin = static_cast<int>(pre_units + c * rest / n_ctas);
    u_end = static_cast<int>(pre_units + (c + 1) * rest / n_ctas);
  }
}

template <int D>
__device__ __forceinline__ void produce_items(const DecodeArgs& a, const CUtensorMap* tm_k,
                                              const CUtensorMap* tm_v, uint8_t* ring,
                                              uint64_t* st_full, uint64_t* st_empty,
                                              ItemDesc* idesc, volatile int* abort_flag) {
  using L = SLayout<D>;
  constexpr int kS = L::kSlots;
  constexpr int kChunks = D / 8;
  constexpr int kBoxesPerTile = kTilePages * 2;  // pages x {K, V}, both feature halves each
  static_assert(2 * kBoxesPerTile <= 32, "one box per lane");
  const PrefixArgs& p = a.pre;
  const int lane = threadIdx.x & 31;
  const int page0 = p.cpl / kPage;
  const int hkv = p.num_kv_heads;
  int u, u_end;
  unit_range(a, u, u_end);
  // the unit being produced and the next one's metadata (read one unit ahead)
  int item = 0;
  // next unit's raw metadata: lanes 0-2 hold cu_seqlens_q[r], cu_seqlens_q[r+1],
  // seq_lens[r]; lanes 0-7 also the block ids of its first eight pages
  auto fetch = [&](int uu, int& meta, int& id) {
    meta = 0;
    id = 0;
    if (uu >= u_end) return;
    const int r = uu / hkv;
    const int32_t* bt = a.block_table + static_cast<int64_t>(r) * a.bt_stride;
    if (lane == 0) meta = __ldg(a.cu_seqlens_q + r);
    if (lane == 1) meta = __ldg(a.cu_seqlens_q + r + 1);
    if (lane == 2) meta = __ldg(a.seq_lens + r);
    // read before the request's length is known: entries past its pages (up to the
    // row stride) are read but never used
    if (lane < 2 * kTilePages) id = __ldg(bt + min(static_cast<int64_t>(page0 + lane), a.bt_stride - 1));
  };
  int n_meta, n_id;
  fetch(u, n_meta, n_id);
  bool ok = true;
  for (; ok; ++u) {
    // ---- unit u (or the end): its metadata, and the next unit's on its way
    int q0 = 0, q_len = 0, seq_len = 0, ids = 0;
    const bool end = u >= u_end;
    if (!end) {
      q0 = __shfl_sync(0xffffffffu, n_meta, 0);
      q_len = __shfl_sync(0xffffffffu, n_meta, 1) - q0;
      seq_len = __shfl_sync(0xffffffffu, n_meta, 2);
      ids = n_id;
      fetch(u + 1, n_meta, n_id);
      if (q_len <= 0) continue;  // no query rows: nothing to compute or write
    }
    const int kvh = u - (u / hkv) * hkv;
    const int nkeys = seq_len - p.cpl;
    const int nt = end ? -1 : max(1, (nkeys + kKeys - 1) / kKeys);  // >= 1 all-masked tile
    const int npages = (seq_len + kPage - 1) / kPage;
    const int32_t* bt = a.block_table + static_cast<int64_t>(end ? 0 : u / hkv) * a.bt_stride;
    // the end: one marker per consumer group (each group reads every unit_groups-th item)
    for (int t0 = 0; end ? t0 < 2 * a.unit_groups : t0 < nt; t0 += 2) {
      const int slot = item % kS;
      if (item >= kS &&
          !(ok = warp_mbar_wait(&st_empty[slot], ((item / kS) - 1) & 1, abort_flag, p.status)))
        break;
      const int tiles = end ? 0 : min(2, nt - t0);
      if (lane == 0) {
        ItemDesc& d = idesc[slot];
        d.q0 = q0;
        d.q_len = q_len;
        d.seq_len = seq_len;
        d.kvh = kvh;
        d.ntiles = nt;
        d.t0 = t0;
        mbar_arrive_expect_tx(&st_full[slot], static_cast<uint32_t>(tiles * 2 * L::kKV));
      }
      __syncwarp();
      // block ids of the item's pages: lane j holds page page0 + 4 t0 + j; the next
      // item's are read now, one item ahead
      int nxt = 0;
      if (t0 + 2 < nt && lane < 2 * kTilePages) {
        const int pp = page0 + (t0 + 2) * kTilePages + lane;
        nxt = pp < npages ? __ldg(bt + pp) : 0;
      }
      {
        const int h = lane / kBoxesPerTile, rem = lane % kBoxesPerTile;
        const int q = rem >> 1, kv = rem & 1;
        const int pq = (h * kTilePages + q) & (2 * kTilePages - 1);
        const int id_q = __shfl_sync(0xffffffffu, ids, pq);
        const int id_0 = __shfl_sync(0xffffffffu, ids, 0);
        const int page = page0 + t0 * kTilePages + pq;
        const int blk = page < npages ? id_q : id_0;
        if (lane < tiles * kBoxesPerTile) {
          uint8_t* dst = ring + slot * L::kItem + h * L::kStage + kv * L::kKV + q * (kPage * D * 2);
          tma_load_4d(dst, kv ? tm_v : tm_k, &st_full[slot], 0, blk * kPage, 0, kvh);
        }
      }
      if (t0 == 0 && !end) {
        const uint32_t qb = smem_u32(ring + slot * L::kItem + 2 * L::kKV);
        const int rows = q_len * p.group;
        for (int x = lane; x < kRows * kChunks; x += 32) {
          const int row = x / kChunks, c = x % kChunks;
          const bool in = row < rows;
          const int qi = row / p.group, hj = row - qi * p.group;
          const int64_t off =
              (static_cast<int64_t>(q0 + qi) * p.num_q_heads + kvh * p.group + hj) * D + c * 8;
          cp_async_16_u32(qb + sw128<kRows>(row, c), in ? a.q + off : a.q, in ? 16u : 0u);
        }
      }
      cp_async_mbar_arrive(&st_full[slot]);
      ++item;
      ids = nxt;
    }
    if (end) break;
  }
  cp_async_wait<0>();
}

// kG groups of 8 / kG streaming warps: group g takes items g, g + kG, g + 2 kG, ...
// (kG = 2 only when every unit is a single item, so a unit never spans two groups).
// Within a group, warp w' takes keys [w' * 16 kG, (w' + 1) * 16 kG) of the item's 128
// (kG blocks of 16 keys in one of its two tiles).
template <int D, int kG>
__device__ __forceinline__ void consume_items(const DecodeArgs& a, uint8_t* ring,
                                              uint64_t* st_full, uint64_t* st_empty,
                                              const ItemDesc* idesc, volatile int* abort_flag) {
  using L = SLayout<D>;
  constexpr int kS = L::kSlots;
  constexpr int kChunks = D / 8;          // 16-byte chunks per row
  constexpr int kDT = D / 8;              // O n-tiles (8 features each)
  constexpr int kORow = D + 4;            // merge scratch row (floats)
  constexpr int kWPU = kStreamWarps / kG; // warps per unit
  constexpr int kB = kG;                  // 16-key blocks per warp
  static_assert(kWPU * kRows * kORow * 4 + 2 * kWPU * kRows * 4 <= L::kItem,
                "merge scratch fits one item");
  const PrefixArgs& p = a.pre;
  const int tid = threadIdx.x;  // 0 .. 255
  const int lane = tid & 31;
  const int wi = tid >> 5;      // 0 .. 7
  const int grp = wi / kWPU;    // this warp's group
  const int wg = wi % kWPU;     // its index within the group
  const int half = (wg * 16 * kB) >> 6;      // which tile of the item this warp computes
  const int kw0 = (wg * 16 * kB) & 63;       // its first key within that tile
  const uint32_t rbase = smem_u32(ring);

  int c_nt = 0, c_seq = 0, c_qlen = 0, c_q0 = 0, c_kvh = 0, rows_valid = 0;
  int pos[2] = {-1, -1};
  float o[kDT][4];
  float m_run[2], l_run[2];
  uint32_t qa[D / 16][4];
  for (int item = grp;; item += kG) {
    const int slot = item % kS;
    const uint32_t par = (item / kS) & 1;
    if (!warp_mbar_wait(&st_full[slot], par, abort_flag, p.status)) break;
    // every lane observes the completed phase (the TMA bytes are visible to it)
    mbar_test_wait(&st_full[slot], par);
    const ItemDesc d = idesc[slot];
    if (d.ntiles < 0) break;
    const uint32_t ib = rbase + slot * L::kItem;
    const int t0 = d.t0;
    if (t0 == 0) {
      c_nt = d.ntiles;
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
      const uint32_t qb = ib + 2 * L::kKV;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int row = (lane & 7) + ((lane >> 3) & 1) * 8;
        const int c = kk * 2 + (lane >> 4);
        ldmatrix_x4(qb + sw128<kRows>(row, c), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
      }
    }
    if (t0 + half < c_nt) {
      const uint32_t kb = ib + half * L::kStage;
      const uint32_t vb = kb + L::kKV;
      const int key0 = p.cpl + (t0 + half) * kKeys + kw0;
      if (key0 + 16 * kB > c_seq) {
        // this warp's keys past the request: zero their V rows (P is 0 there, but the
        // page may hold anything)
        for (int x = lane; x < 16 * kB * kChunks; x += 32) {
          const int k = x / kChunks, c = x % kChunks;
          if (key0 + k >= c_seq)
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(
                             vb + kv_off<D>(kw0 + k, c)), "r"(0u)
                         : "memory");
        }
        __syncwarp();
      }
      // S = Q K^T over this warp's keys (two n-tiles of 8 per 16-key block)
      float sacc[2 * kB][4];
#pragma unroll
      for (int i = 0; i < 2 * kB; ++i) sacc[i][0] = sacc[i][1] = sacc[i][2] = sacc[i][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
        for (int b = 0; b < kB; ++b) {
          const int key = kw0 + 16 * b + (lane & 7) + (lane >> 4) * 8;
          const int c = kk * 2 + ((lane >> 3) & 1);
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4(kb + kv_off<D>(key, c), b0, b1, b2, b3);
          mma_bf16_16816(sacc[2 * b], qa[kk], b0, b1);
          mma_bf16_16816(sacc[2 * b + 1], qa[kk], b2, b3);
        }
      }
      // mask (keys past the request, and the causal limit), online softmax in base 2
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float mx = -INFINITY;
        const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
#pragma unroll
        for (int nt = 0; nt < 2 * kB; ++nt) {
          // the two scores of a pair scaled in one paired instruction, then masked
          const float2 s2 = mul_f32x2(make_float2(sacc[nt][2 * h], sacc[nt][2 * h + 1]), sc2);
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int kabs = key0 + nt * 8 + (lane & 3) * 2 + e;
            float& sref = sacc[nt][2 * h + e];
            sref = (kabs < c_seq && kabs <= pos[h]) ? (e ? s2.y : s2.x) : -INFINITY;
            mx = fmaxf(mx, sref);
          }
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        // keep the running max unless it grows by more than 2^8 (always on the row's
        // first unmasked keys, where it is -inf): then p = 2^(s - m) <= 256 and O and
        // l need rescaling only now and then
        if (mx > m_run[h] + 8.f) {
          const float alpha = fast_exp2(m_run[h] - mx);
          l_run[h] *= alpha;
#pragma unroll
          for (int dt = 0; dt < kDT; ++dt) {
            o[dt][2 * h] *= alpha;
            o[dt][2 * h + 1] *= alpha;
          }
          m_run[h] = mx;
        }
        const float m_use = (m_run[h] == -INFINITY) ? 0.f : m_run[h];
        float2 sum2 = make_float2(0.f, 0.f);
        const float2 nm2 = make_float2(-m_use, -m_use);
#pragma unroll
        for (int nt = 0; nt < 2 * kB; ++nt) {
          const float2 x = add_f32x2(make_float2(sacc[nt][2 * h], sacc[nt][2 * h + 1]), nm2);
          sacc[nt][2 * h] = fast_exp2(x.x);
          sacc[nt][2 * h + 1] = fast_exp2(x.y);
          sum2 = add_f32x2(sum2, make_float2(sacc[nt][2 * h], sacc[nt][2 * h + 1]));
        }
        l_run[h] += sum2.x + sum2.y;
      }
      // O += P V over the same keys
#pragma unroll
      for (int b = 0; b < kB; ++b) {
        uint32_t pa[4];
        pa[0] = pack_bf16x2(sacc[2 * b][0], sacc[2 * b][1]);
        pa[1] = pack_bf16x2(sacc[2 * b][2], sacc[2 * b][3]);
        pa[2] = pack_bf16x2(sacc[2 * b + 1][0], sacc[2 * b + 1][1]);
        pa[3] = pack_bf16x2(sacc[2 * b + 1][2], sacc[2 * b + 1][3]);
#pragma unroll
        for (int dp = 0; dp < kDT / 2; ++dp) {
          const int key = kw0 + 16 * b + (lane & 7) + ((lane >> 3) & 1) * 8;
          const int c = dp * 2 + (lane >> 4);
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4_trans(vb + kv_off<D>(key, c), b0, b1, b2, b3);
          mma_bf16_16816(o[2 * dp], pa, b0, b1);
          mma_bf16_16816(o[2 * dp + 1], pa, b2, b3);
        }
      }
    }
    if (t0 + 2 >= c_nt) {
      // ---- the unit's last item: the group's warps' (max, sum, O) -> one normalised
      // partial per row, through this item's memory (only this group reads the item)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
        l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
      }
      group_sync<kWPU>(grp);  // every warp of the group is done reading this item's K/V
      float* s_o = reinterpret_cast<float*>(ring + slot * L::kItem);  // [kWPU][16][kORow]
      float* s_m = s_o + kWPU * kRows * kORow;                        // [kWPU][16]
      float* s_l = s_m + kWPU * kRows;                                // [kWPU][16]
      // every warp's raw (max, sum, O) of its keys; the weights come in the final pass
      if ((lane & 3) == 0) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          s_m[wg * kRows + (lane >> 2) + 8 * h] = m_run[h];
          s_l[wg * kRows + (lane >> 2) + 8 * h] = l_run[h];
        }
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int rr = (lane >> 2) + 8 * h;
        if (rr >= rows_valid) continue;
        float* dst = s_o + (wg * kRows + rr) * kORow;
#pragma unroll
        for (int dt = 0; dt < kDT; ++dt) {
          const int dd = dt * 8 + (lane & 3) * 2;
          *reinterpret_cast<float2*>(dst + dd) = make_float2(o[dt][2 * h], o[dt][2 * h + 1]);
        }
      }
      group_sync<kWPU>(grp);
      const int64_t slot_rows = static_cast<int64_t>(p.n_splits) * p.total_q * p.num_q_heads;
      // warp w' finalises rows w', w' + kWPU, ...; lane c owns features [4c, 4c + 4)
      for (int rr = wg; rr < rows_valid; rr += kWPU) {
        float mw[kWPU];
        float mg = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWPU; ++w) {
          mw[w] = s_m[w * kRows + rr];
          mg = fmaxf(mg, mw[w]);
        }
        float lsum = 0.f;
#pragma unroll
        for (int w = 0; w < kWPU; ++w) {
          mw[w] = (mw[w] == -INFINITY) ? 0.f : fast_exp2(mw[w] - mg);  // warp w's weight
          lsum += s_l[w * kRows + rr] * mw[w];
        }
        const float inv = !(lsum <= 0.f) ? 1.f / lsum : 0.f;  // a NaN sum propagates
        const int qi = rr / p.group, j = rr - qi * p.group;
        const int64_t row = static_cast<int64_t>(c_q0 + qi) * p.num_q_heads + c_kvh * p.group + j;
        const int64_t prow = slot_rows + row;
        if (lane < D / 4) {
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int w = 0; w < kWPU; ++w) {
            const float4 v =
                *reinterpret_cast<const float4*>(s_o + (w * kRows + rr) * kORow + lane * 4);
            acc.x = fmaf(mw[w], v.x, acc.x);
            acc.y = fmaf(mw[w], v.y, acc.y);
            acc.z = fmaf(mw[w], v.z, acc.z);
            acc.w = fmaf(mw[w], v.w, acc.w);
          }
          store_bf16x4(p.part_o + prow * D + lane * 4,
                       make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
        }
        if (lane == 0)
          p.part_lse[p.n_splits * p.lse_stride + row] = !(lsum <= 0.f) ? mg + log2f(lsum) : -INFINITY;
      }
    }
    // the item goes back to the producer (its TMA will overwrite what this warp
    // wrote through the generic proxy)
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&st_empty[slot]);
  }
}

// ------------------------------------------------------------ staged merge --
// merge_attn_states for rows [b R / G, (b + 1) R / G) of CTA b, in chunks of
// a.merge_rows rows.  Thread 0 brings a chunk of every slot with two TMA tensor
// copies completing on `bar`: the bf16 rows ([slot][row][D], tm_po) and the LSEs
// ([slot][row], tm_pl, the run starting at the 16-byte boundary at or before the
// chunk); rows past the workspace's arrive zero-filled and are not merged.  Then half
// a warp merges each row: every lane computes the slots' weights from their LSEs and
// sums features [i*D/16, (i+1)*D/16) of every slot, its loop unrolled to kSlots >= the
// slot count.  An empty slot (lse -inf) gets weight 0.
template <int D, int kSlots>
__device__ __forceinline__ void merge_rows_staged(const DecodeArgs& a, const CUtensorMap* tm_po,
                                                  const CUtensorMap* tm_pl, uint8_t* smem,
                                                  uint64_t* bar, volatile int* abort_flag) {
  constexpr int kF = D / 16;
  using Vec = typename std::conditional<kF == 8, uint4, uint2>::type;
  const PrefixArgs& p = a.pre;
  const int n = p.n_splits + 1;  // slots
  const int chunk = a.merge_rows;
  const int lbox = (chunk + 6) & ~3;  // LSEs per slot in a chunk's copy
  const int64_t rows = static_cast<int64_t>(p.total_q) * p.num_q_heads;
  // (32-bit products while they fit: a 64-bit division costs hundreds of cycles)
  const bool small = rows * gridDim.x < (int64_t{1} << 31);
  const int64_t r0 = small ? static_cast<int64_t>(static_cast<uint32_t>(blockIdx.x * rows) / gridDim.x)
                           : static_cast<int64_t>(blockIdx.x) * rows / gridDim.x;
  const int64_t r1 = small ? static_cast<int64_t>(static_cast<uint32_t>((blockIdx.x + 1) * rows) /
                                                  gridDim.x)
                           : static_cast<int64_t>(blockIdx.x + 1) * rows / gridDim.x;
  const int hw = threadIdx.x >> 4, hl = threadIdx.x & 15;
  __nv_bfloat16* s_o = reinterpret_cast<__nv_bfloat16*>(smem);  // [n][chunk][D]
  float* s_l = reinterpret_cast<float*>(smem + static_cast<size_t>(n) * chunk * D * 2);  // [n][lbox]
  uint32_t phase = 0;
  for (int64_t c0 = r0; c0 < r1; c0 += chunk, phase ^= 1u) {
    const int m = static_cast<int>(min(static_cast<int64_t>(chunk), r1 - c0));
    const int l0 = static_cast<int>(c0 & ~int64_t{3});  // the LSE run's first row
    if (threadIdx.x == 0) {
      mbar_arrive_expect_tx(bar, static_cast<uint32_t>(n * chunk * D * 2 + n * lbox * 4));
      // the partials were written by other CTAs through the generic proxy; the copies
      // read them through the async proxy
      asm volatile("fence.proxy.async.global;" ::: "memory");
      tma_load_3d(s_o, tm_po, bar, 0, static_cast<int>(c0), 0);
      tma_load_2d(s_l, tm_pl, bar, l0, 0);
    }
    const bool ok = mbar_wait(bar, phase, abort_flag, p.status);
    const int lo = static_cast<int>(c0) - l0;
    // half-warp h takes rows h, h + kThreads / 16, ...
    for (int base = 2 * (hw >> 1); base < m; base += kThreads / 16) {
      const int i = base + (hw & 1);
      const bool in = ok && i < m;
      // every load first (slots past n read slot n - 1 and get weight 0; a partial is
      // always finite), then the weights, then the sums: no load waits on another
      float l[kSlots];
      Vec v[kSlots];
#pragma unroll
      for (int s = 0; s < kSlots; ++s) {
        const int sc = min(s, n - 1);
        l[s] = s_l[sc * lbox + lo + i];
        v[s] = *reinterpret_cast<const Vec*>(s_o + (static_cast<size_t>(sc) * chunk + i) * D +
                                             hl * kF);
      }
      float mx = -INFINITY;
#pragma unroll
      for (int s = 0; s < kSlots; ++s) {
        if (s >= n) l[s] = -INFINITY;
        mx = fmaxf(mx, l[s]);
      }
      if (!in) mx = -INFINITY;
      float wsum = 0.f;
#pragma unroll
      for (int s = 0; s < kSlots; ++s) {
        l[s] = (mx == -INFINITY || l[s] == -INFINITY) ? 0.f : fast_exp2(l[s] - mx);
        wsum += l[s];
      }
      float acc[kF];
#pragma unroll
      for (int f = 0; f < kF; ++f) acc[f] = 0.f;
#pragma unroll
      for (int s = 0; s < kSlots; ++s) {
        const uint32_t* u = reinterpret_cast<const uint32_t*>(&v[s]);
#pragma unroll
        for (int f = 0; f < kF / 2; ++f) {
          const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[f]));
          acc[2 * f] = fmaf(l[s], x.x, acc[2 * f]);
          acc[2 * f + 1] = fmaf(l[s], x.y, acc[2 * f + 1]);
        }
      }
      const float inv = !(wsum <= 0.f) ? 1.f / wsum : 0.f;
#pragma unroll
      for (int f = 0; f < kF; ++f) acc[f] *= inv;
      if (in) {
        const int64_t row = c0 + i;
        Vec o;
        uint32_t* ou = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
        for (int f = 0; f < kF / 2; ++f) ou[f] = pack_bf16x2(acc[2 * f], acc[2 * f + 1]);
        *reinterpret_cast<Vec*>(a.out + row * D + hl * kF) = o;
        if (hl == 0 && a.lse != nullptr)
          a.lse[row] = !(wsum <= 0.f) ? (mx + log2f(wsum)) * 0.69314718055994531f : -INFINITY;
      }
    }
    // the next chunk's copies overwrite what was read here
    __syncthreads();
  }
}

// ------------------------------------------------------------------ the kernel --
template <int D>
__device__ __forceinline__ void decode_body(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                            const CUtensorMap& tm_v, const CUtensorMap& tm_kp,
                                            const CUtensorMap& tm_po, const CUtensorMap& tm_pl,
                                            const DecodeArgs& a) {
  using L = SLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const PrefixArgs& p = a.pre;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // generation of the grid barrier at the end, read now with a relaxed load: nothing
  // waits on it until the barrier (an acquire here would hold thread 0, and through the
  // first CTA barrier every warp, for a round trip to memory).  The previous call
  // advanced it before that kernel ended, and this CTA's arrival below (a release)
  // orders the read before any CTA of this call can advance it.
  unsigned g0 = 0u;
  if (threadIdx.x == 0)
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(g0) : "l"(a.bar_gen) : "memory");
  // the first TMA through each map would otherwise wait for its descriptor
  if (threadIdx.x == 32 * kWarpScheduler) {
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_kp);
    prefetch_tensormap(&tm_po);
    prefetch_tensormap(&tm_pl);
  }

  // ---- role 1: one range of the prefix phase (tcgen05)
  if (static_cast<int>(blockIdx.x) < a.prefix_ctas) {
    const int b = blockIdx.x;
    const int split = b % p.n_splits;
    const int pair = (b / p.n_splits) % p.pairs;
    const int kvh = b / (p.n_splits * p.pairs);
    const int t_first = split * a.key_tiles / p.n_splits;
    const int t_last = (split + 1) * a.key_tiles / p.n_splits;
    prefix::prefix_range<D>(&tm_q, &tm_kp, &tm_v, p, prefix::prefix_geom(p, pair), kvh, split,
                            t_first, t_last, smem,
                            reinterpret_cast<uint64_t*>(smem + L::kPrefixBars));
    // the staging buffer was read through the generic proxy and TMA wrote the stages;
    // the suffix role below rewrites the same memory
    fence_proxy_async_smem();
    __syncthreads();
  }

  // ---- role 2: the suffix units, produced by warp 8 and computed by warps 0-7
  constexpr int kS = L::kSlots;
  uint64_t* st_full = reinterpret_cast<uint64_t*>(smem + L::kSuffixBars);  // [kS]
  uint64_t* st_empty = st_full + kS;                                        // [kS]
  ItemDesc* idesc = reinterpret_cast<ItemDesc*>(st_empty + kS);              // [kS]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(idesc + kS);
  uint64_t* merge_bar = reinterpret_cast<uint64_t*>(smem + L::kSuffixBars + kMergeBarOff);
  int u_begin, u_end;
  unit_range(a, u_begin, u_end);
  if (threadIdx.x == 0) {
    for (int i = 0; i < kS; ++i) {
      mbar_init(&st_full[i], 1 + 32);  // the producer's expect_tx + its lanes' copies
      mbar_init(&st_empty[i], kStreamWarps / a.unit_groups);  // the warps of one unit
    }
    mbar_init(merge_bar, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  if (u_begin < u_end) {  // (a prefix CTA may have none)
    if (warp == kWarpScheduler) {
      produce_items<D>(a, &tm_k, &tm_v, smem, st_full, st_empty, idesc, abort_flag);
    } else if (warp < kStreamWarps) {
      if (a.unit_groups == 2)
        consume_items<D, 2>(a, smem, st_full, st_empty, idesc, abort_flag);
      else
        consume_items<D, 1>(a, smem, st_full, st_empty, idesc, abort_flag);
    }
  }
  // the bulk copies of the merge below overwrite what was written here through the
  // generic proxy
  fence_proxy_async_smem();

  // ---- grid-wide barrier: every partial of the call is written.  The arrival is one
  // acquire-release add (the CTA barrier before it makes every thread's partial
  // stores part of what it releases); the last CTA zeroes the count and advances the
  // generation, which the others read at their start (no CTA can advance it before
  // every CTA has arrived).
  __syncthreads();
  if (threadIdx.x == 0) {
    const int old = atomic_add_acq_rel_gpu(a.bar_count, 1);
    if (old == static_cast<int>(gridDim.x) - 1) {
      *a.bar_count = 0;
      st_release_gpu_u32(a.bar_gen, g0 + 1u);
    } else {
      const long long c0 = clock64();
      unsigned spins = 0;
      while (ld_acquire_gpu_u32(a.bar_gen) == g0) {
        if ((++spins & 255u) == 0 && clock64() - c0 > kWaitLimitCycles) {
          if (p.status) atomicCAS(p.status, 0, kErrTimeout);
          break;
        }
      }
    }
  }
  __syncthreads();

  // ---- merge_attn_states: CTA b takes rows [b R / G, (b + 1) R / G) of the R rows,
  // which are contiguous in every slot: one bulk copy per slot brings a chunk of them
  // (and their LSEs) into shared memory, then half a warp merges each row
  // (the slot loop is unrolled to a bound: 8 when it suffices)
  if (p.n_splits + 1 <= 8)
    merge_rows_staged<D, 8>(a, &tm_po, &tm_pl, smem, merge_bar, abort_flag);
  else
    merge_rows_staged<D, kDecodeMaxParts>(a, &tm_po, &tm_pl, smem, merge_bar, abort_flag);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    decode_cascade_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v,
                          const __grid_constant__ CUtensorMap tm_kp,
                          const __grid_constant__ CUtensorMap tm_po,
                          const __grid_constant__ CUtensorMap tm_pl, const DecodeArgs a) {
  decode_body<D>(tm_q, tm_k, tm_v, tm_kp, tm_po, tm_pl, a);
}

// The same step with the prefix length read from device memory (*a.cpl_dev, written
// by the device planner before this launch): the launch plan was made for an upper
// bound of it, and everything that follows from the prefix length (the prefix's key
// tiles, where the suffix starts, whether a request's suffix fits one item) is set
// here from the value read.  A prefix length of 0 leaves the prefix ranges empty and
// gives every request all its keys in the suffix phase: the standard path.
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    decode_cascade_dev_kernel(const __grid_constant__ CUtensorMap tm_q,
                              const __grid_constant__ CUtensorMap tm_k,
                              const __grid_constant__ CUtensorMap tm_v,
                              const __grid_constant__ CUtensorMap tm_kp,
                              const __grid_constant__ CUtensorMap tm_po,
                              const __grid_constant__ CUtensorMap tm_pl, const DecodeArgs a_in) {
  __shared__ int s_cpl;
  if (threadIdx.x == 0) s_cpl = *a_in.cpl_dev;
  __syncthreads();
  DecodeArgs a = a_in;
  const int cpl = min(max(s_cpl, 0), a_in.pre.cpl);  // (never past the bound planned for)
  a.pre.cpl = cpl;
  a.key_tiles = (cpl + 63) / 64;
  a.unit_groups = a_in.max_seqlen_k - cpl <= 2 * 64 ? 2 : 1;
  decode_body<D>(tm_q, tm_k, tm_v, tm_kp, tm_po, tm_pl, a);
}

template <int D>
cudaError_t launch_decode_d(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                            const CUtensorMap& tm_v, const CUtensorMap& tm_kp,
                            const CUtensorMap& tm_po,
                            const CUtensorMap& tm_pl, const DecodeArgs& a, int grid,
                            cudaStream_t stream) {
  static std::atomic<uint64_t> attr_done{0}, attr_done_dev{0};
  auto kernel = a.cpl_dev ? decode_cascade_dev_kernel<D> : decode_cascade_kernel<D>;
  cudaError_t e = set_smem_once(kernel, SLayout<D>::kDynamic,
                                a.cpl_dev ? attr_done_dev : attr_done);
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
  return cudaLaunchKernelEx(&cfg, kernel, tm_q, tm_k, tm_v, tm_kp, tm_po, tm_pl, a);
}

}  // namespace

cudaError_t launch_decode(int head_dim, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                          const CUtensorMap& tm_v, const CUtensorMap& tm_kp,
                          const CUtensorMap& tm_po, const CUtensorMap& tm_pl,
                          const DecodeArgs& a, int grid, cudaStream_t stream) {
  if (head_dim == 64)
    return launch_decode_d<64>(tm_q, tm_k, tm_v, tm_kp, tm_po, tm_pl, a, grid, stream);
  return launch_decode_d<128>(tm_q, tm_k, tm_v, tm_kp, tm_po, tm_pl, a, grid, stream);
}

}  // namespace csp
