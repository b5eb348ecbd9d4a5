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
  static constexpr int kSuffixBarBytes = 2048;  // barriers, descriptors; then the exchange
  static constexpr int kXchOff = 1024;           // consumers' row maxima and sums (1 KB)
  static constexpr int kDynamic = kSuffixBars + kSuffixBarBytes + 1024;  // + align slack
  static_assert(kSlots >= 3, "two items in flight ahead of the computed one");
  static_assert(kStage % 1024 == 0 && (2 * kKV) % 1024 == 0, "swizzled stage alignment");
  static_assert(4 * kSlots * 8 + kSlots * 32 + 16 <= kMergeBarOff, "suffix barrier area");
  static_assert(kMergeBarOff + 8 <= kXchOff && kXchOff + 2 * 8 * 16 * 4 <= kSuffixBarBytes,
                "exchange area: [groups][2][warps per group][16] floats");
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

__device__ __forceinline__ unsigned long long ld_acquire_gpu_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned long long atom_add_acq_rel_gpu_u64(unsigned long long* p,
                                                                        unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.add.acq_rel.gpu.global.u64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v)
               : "memory");
  return old;
}

// the streaming warps of one unit group: named barrier 1 + group, kWPU warps
template <int kWPU>
__device__ __forceinline__ void group_sync(int group) {
  asm volatile("bar.sync %0, %1;" ::"r"(1 + group), "r"(kWPU * 32) : "memory");
}

// Items and their slot barriers.  Item i sits in ring slot i % kS and is computed by
// group i % groups; each (group, slot) pair has its own full and empty barrier, so that
// the items one barrier sees are exactly every L-th item (L = lcm(groups, kS)) and a
// waiter never skips one of its phases (with shared barriers a group that skips the
// other group's phase of a slot could take that phase's completion for its own).
template <int kG, int kS>
__device__ __forceinline__ int item_barrier(int i) {
  const unsigned u = static_cast<unsigned>(i);
  return static_cast<int>((u % kG) * kS + u % kS);
}
template <int kG, int kS>
__device__ __forceinline__ uint32_t item_parity(int i) {
  constexpr unsigned kPeriod = (kG == 2 && (kS & 1)) ? 2 * kS : kS;  // lcm(kG, kS)
  return (static_cast<unsigned>(i) / kPeriod) & 1u;
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
//    the unit's Q rows with 16-byte cp.async.  A page past the request re-reads the
//    item's first page (its keys are masked); the item's descriptor tells the consumers
//    which unit and tiles it holds.
//  * warps 0-7 consume them, in groups (see consume_items): S = Q K^T and O += P V on
//    mma.sync m16n8k16 (bf16 in, fp32 accumulate) fed by ldmatrix, masked by the
//    request's causal limit (bottom-right alignment, §四), online softmax in base 2.
//    Each warp of a group scores its own block of the item's keys, and accumulates
//    O for its own slice of the features over all of them: the group exchanges its
//    rows' maxima and P through shared memory, so the item goes back to the producer
//    as soon as P V is done and no O is merged across warps.  V rows past the request
//    are zeroed first (a TMA page holds whatever the cache has there).  At the unit's
//    end the group sums its rows' l and every warp writes its normalised slice of
//    the bf16 rows (and warp 0 their log2-sum-exp) into the suffix slot.
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

template <int D, int kG>
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
    for (int t0 = 0; end ? t0 < 2 * kG : t0 < nt; t0 += 2) {
      const int slot = item % kS;
      const int fb = item_barrier<kG, kS>(item);
      // the slot's previous item must have been given back
      if (item >= kS &&
          !(ok = warp_mbar_wait(&st_empty[item_barrier<kG, kS>(item - kS)],
                                item_parity<kG, kS>(item - kS), abort_flag,
                                p.status)))
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
        mbar_arrive_expect_tx(&st_full[fb], static_cast<uint32_t>(tiles * 2 * L::kKV));
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
          tma_load_4d(dst, kv ? tm_v : tm_k, &st_full[fb], 0, blk * kPage, 0, kvh);
        }
      }
      if (t0 == 0 && !end) {
        // only the unit's rows: the consumers mask every score of the rows past them
        // (by selection, so whatever those rows hold never reaches a result)
        const uint32_t qb = smem_u32(ring + slot * L::kItem + 2 * L::kKV);
        const int rows = q_len * p.group;
        for (int x = lane; x < rows * kChunks; x += 32) {
          const int row = x / kChunks, c = x % kChunks;
          const int qi = row / p.group, hj = row - qi * p.group;
          const int64_t off =
              (static_cast<int64_t>(q0 + qi) * p.num_q_heads + kvh * p.group + hj) * D + c * 8;
          cp_async_16_u32(qb + sw128<kRows>(row, c), a.q + off, 16u);
        }
      }
      cp_async_mbar_arrive(&st_full[fb]);
      ++item;
      ids = nxt;
    }
    if (end) break;
  }
  cp_async_wait<0>();
}

// kG groups of kWPU = 8 / kG streaming warps: group g takes items g, g + kG, g + 2 kG,
// ... (kG = 2 only when every unit is a single item, so a unit never spans two groups).
// Warp w' of a group:
//  * scores keys [16 kB w', 16 kB (w' + 1)) of the item's 128 (kB = kG blocks of 16
//    keys, in tile 16 kB w' / 64), masks and scales them, and posts its rows' maxima;
//  * after a group barrier, takes the group's maxima (so the running max, and every
//    rescaling of O and l, is the same in all the group's warps), forms P = 2^(S - m)
//    and stores it as bf16 over the K rows it alone read (16-key block b of the item
//    lands on the first 512 bytes of that block's K page, [16 rows][2 x 16 B] with the
//    chunk index XOR bit 2 of the row: conflict-free stores and ldmatrix);
//  * after a second group barrier, accumulates O for features [w' D / kWPU,
//    (w' + 1) D / kWPU) over all the item's keys, P fed by ldmatrix from those blocks
//    and V by ldmatrix.trans, and gives the item back;
//  * at the unit's end, sums its rows' l with the group's (a third barrier) and
//    writes its normalised features of the unit's rows.
template <int D, int kG>
__device__ __forceinline__ void consume_items(const DecodeArgs& a, uint8_t* ring,
                                              uint64_t* st_full, uint64_t* st_empty,
                                              const ItemDesc* idesc, float* xch,
                                              volatile int* abort_flag) {
  using L = SLayout<D>;
  constexpr int kS = L::kSlots;
  constexpr int kChunks = D / 8;           // 16-byte chunks per row
  constexpr int kWPU = kStreamWarps / kG;  // warps per unit
  constexpr int kB = kG;                   // 16-key blocks per warp
  constexpr int kNT = D / kWPU / 8;        // n-tiles (8 features each) of a warp's O slice
  constexpr int kPageBytes = kPage * D * 2;
  static_assert(kNT >= 1 && kNT <= 4 && (kNT == 1 || kNT % 2 == 0), "O slice of 8, 16 or 32");
  static_assert(kPageBytes >= kB * 512, "a P block fits its K page");
  const PrefixArgs& p = a.pre;
  const int tid = threadIdx.x;  // 0 .. 255
  const int lane = tid & 31;
  const int wi = tid >> 5;      // 0 .. 7
  const int grp = wi / kWPU;    // this warp's group
  const int wg = wi % kWPU;     // its index within the group
  const int half = (wg * 16 * kB) >> 6;      // which tile of the item this warp scores
  const int kw0 = (wg * 16 * kB) & 63;       // its first key within that tile
  const int g = lane >> 2;                   // rows g and g + 8 of the fragments
  const uint32_t rbase = smem_u32(ring);
  float* xm = xch + grp * (2 * kWPU * kRows);  // [kWPU][16] row maxima
  float* xl = xm + kWPU * kRows;               // [kWPU][16] row sums
  // P block `ks` (16 keys) of an item: the first 512 bytes of its K page
  auto p_block = [&](uint32_t ib, int ks) -> uint32_t {
    return ib + (ks >> 2) * L::kStage + (ks & 3) * kPageBytes;
  };

  int c_nt = 0, c_seq = 0, c_qlen = 0, c_q0 = 0, c_kvh = 0, rows_valid = 0;
  int pos[2] = {-1, -1};
  float o[kNT][4];
  float m_run[2], l_run[2];  // the group's running max; this lane's share of the sum
  uint32_t qa[D / 16][4];
  for (int item = grp;; item += kG) {
    const int slot = item % kS;
    const int fb = item_barrier<kG, kS>(item);
    const uint32_t par = item_parity<kG, kS>(item);
    if (!warp_mbar_wait(&st_full[fb], par, abort_flag, p.status)) break;
    // every lane observes the completed phase (the TMA bytes are visible to it)
    mbar_test_wait(&st_full[fb], par);
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
        const int rho = g + 8 * h;
        pos[h] = rho < rows_valid ? c_seq - c_qlen + rho / p.group : -1;
        m_run[h] = -INFINITY;
        l_run[h] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < kNT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
      const uint32_t qb = ib + 2 * L::kKV;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int row = (lane & 7) + ((lane >> 3) & 1) * 8;
        const int c = kk * 2 + (lane >> 4);
        ldmatrix_x4(qb + sw128<kRows>(row, c), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
      }
    }
    const int tiles = min(2, c_nt - t0);  // tiles this item holds
    const bool mine = half < tiles;       // this warp has keys in it
    // ---- S = Q K^T over this warp's keys (two n-tiles of 8 per 16-key block), masked
    // (keys past the request, and the causal limit) and scaled to base 2
    float sacc[2 * kB][4];
    float mx[2] = {-INFINITY, -INFINITY};
    if (mine) {
      const uint32_t kb = ib + half * L::kStage;
      const uint32_t vb = kb + L::kKV;
      const int key0 = p.cpl + (t0 + half) * kKeys + kw0;
      if (key0 + 16 * kB > c_seq) {
        // this warp's keys past the request: zero their V rows (P is 0 there, but the
        // page may hold anything); every warp of the group reads them after the
        // barriers below
        for (int x = lane; x < 16 * kB * kChunks; x += 32) {
          const int k = x / kChunks, c = x % kChunks;
          if (key0 + k >= c_seq)
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(
                             vb + kv_off<D>(kw0 + k, c)), "r"(0u)
                         : "memory");
        }
      }
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
      const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int nt = 0; nt < 2 * kB; ++nt) {
          // the two scores of a pair scaled in one paired instruction, then masked
          const float2 s2 = mul_f32x2(make_float2(sacc[nt][2 * h], sacc[nt][2 * h + 1]), sc2);
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int kabs = key0 + nt * 8 + (lane & 3) * 2 + e;
            float& sref = sacc[nt][2 * h + e];
            sref = (kabs < c_seq && kabs <= pos[h]) ? (e ? s2.y : s2.x) : -INFINITY;
            mx[h] = fmaxf(mx[h], sref);
          }
        }
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
      }
    }
    if ((lane & 3) == 0) {
      xm[wg * kRows + g] = mx[0];
      xm[wg * kRows + g + 8] = mx[1];
    }
    group_sync<kWPU>(grp);
    // ---- the group's maxima; keep the running max unless it grows by more than 2^8
    // (always on the row's first unmasked keys, where it is -inf): then p = 2^(s - m)
    // <= 256 and O and l need rescaling only now and then
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float mg = -INFINITY;
#pragma unroll
      for (int w = 0; w < kWPU; ++w) mg = fmaxf(mg, xm[w * kRows + g + 8 * h]);
      if (mg > m_run[h] + 8.f) {
        const float alpha = fast_exp2(m_run[h] - mg);
        l_run[h] *= alpha;
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
          o[nt][2 * h] *= alpha;
          o[nt][2 * h + 1] *= alpha;
        }
        m_run[h] = mg;
      }
    }
    if (mine) {
      // ---- P = 2^(S - m) as bf16 over this warp's K rows (read by it alone)
      float2 sum2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float m_use = (m_run[h] == -INFINITY) ? 0.f : m_run[h];
        const float2 nm2 = make_float2(-m_use, -m_use);
#pragma unroll
        for (int nt = 0; nt < 2 * kB; ++nt) {
          const float2 x = add_f32x2(make_float2(sacc[nt][2 * h], sacc[nt][2 * h + 1]), nm2);
          sacc[nt][2 * h] = fast_exp2(x.x);
          sacc[nt][2 * h + 1] = fast_exp2(x.y);
          sum2[h] = add_f32x2(sum2[h], make_float2(sacc[nt][2 * h], sacc[nt][2 * h + 1]));
        }
        l_run[h] += sum2[h].x + sum2[h].y;
      }
#pragma unroll
      for (int b = 0; b < kB; ++b) {
        const uint32_t pb = p_block(ib, wg * kB + b);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int row = g + 8 * h;
            const uint32_t addr =
                pb + row * 32 + ((j ^ ((row >> 2) & 1)) << 4) + (lane & 3) * 4;
            asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr),
                         "r"(pack_bf16x2(sacc[2 * b + j][2 * h], sacc[2 * b + j][2 * h + 1]))
                         : "memory");
          }
        }
      }
    }
    group_sync<kWPU>(grp);
    // ---- O (this warp's features) += P V over the item's keys
    {
      const int prow = (lane & 7) + ((lane >> 3) & 1) * 8;
      const uint32_t p_off = prow * 32 + (((lane >> 4) ^ ((prow >> 2) & 1)) << 4);
      const int vkey = (lane & 7) + ((lane >> 3) & 1) * 8;
      for (int ks = 0; ks < 4 * tiles; ++ks) {
        uint32_t pa[4];
        ldmatrix_x4(p_block(ib, ks) + p_off, pa[0], pa[1], pa[2], pa[3]);
        const uint32_t vb = ib + (ks >> 2) * L::kStage + L::kKV;
        const int key = (ks & 3) * 16 + vkey;
        if constexpr (kNT == 1) {
          uint32_t b0, b1;
          asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
                       : "=r"(b0), "=r"(b1)
                       : "r"(vb + kv_off<D>(key, wg)));
          mma_bf16_16816(o[0], pa, b0, b1);
        } else {
#pragma unroll
          for (int dp = 0; dp < kNT / 2; ++dp) {
            const int c = wg * kNT + dp * 2 + (lane >> 4);
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4_trans(vb + kv_off<D>(key, c), b0, b1, b2, b3);
            mma_bf16_16816(o[2 * dp], pa, b0, b1);
            mma_bf16_16816(o[2 * dp + 1], pa, b2, b3);
          }
        }
      }
    }
    // the item goes back to the producer (its TMA will overwrite what this warp wrote
    // there through the generic proxy: P, zeroed V rows)
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&st_empty[fb]);
    if (t0 + 2 >= c_nt) {
      // ---- the unit's end: the group's row sums, then this warp's normalised features
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
        l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
      }
      if ((lane & 3) == 0) {
        xl[wg * kRows + g] = l_run[0];
        xl[wg * kRows + g + 8] = l_run[1];
      }
      group_sync<kWPU>(grp);
      const int64_t slot_rows = static_cast<int64_t>(p.n_splits) * p.total_q * p.num_q_heads;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int rr = g + 8 * h;
        if (rr >= rows_valid) continue;
        float lsum = 0.f;
#pragma unroll
        for (int w = 0; w < kWPU; ++w) lsum += xl[w * kRows + rr];
        const float inv = !(lsum <= 0.f) ? 1.f / lsum : 0.f;  // a NaN sum propagates
        const int qi = rr / p.group, j = rr - qi * p.group;
        const int64_t row = static_cast<int64_t>(c_q0 + qi) * p.num_q_heads + c_kvh * p.group + j;
        __nv_bfloat16* dst = p.part_o + (slot_rows + row) * D + wg * kNT * 8 + (lane & 3) * 2;
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
          *reinterpret_cast<uint32_t*>(dst + nt * 8) =
              pack_bf16x2(o[nt][2 * h] * inv, o[nt][2 * h + 1] * inv);
        if (wg == 0 && (lane & 3) == 0)
          p.part_lse[p.n_splits * p.lse_stride + row] =
              !(lsum <= 0.f) ? m_run[h] + log2f(lsum) : -INFINITY;
      }
    }
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
  uint64_t* st_full = reinterpret_cast<uint64_t*>(smem + L::kSuffixBars);  // [2][kS]
  uint64_t* st_empty = st_full + 2 * kS;                                    // [2][kS]
  ItemDesc* idesc = reinterpret_cast<ItemDesc*>(st_empty + 2 * kS);          // [kS]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(idesc + kS);
  uint64_t* merge_bar = reinterpret_cast<uint64_t*>(smem + L::kSuffixBars + kMergeBarOff);
  float* xch = reinterpret_cast<float*>(smem + L::kSuffixBars + L::kXchOff);
  int u_begin, u_end;
  unit_range(a, u_begin, u_end);
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2 * kS; ++i) {  // per (group, slot)
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
      if (a.unit_groups == 2)
        produce_items<D, 2>(a, &tm_k, &tm_v, smem, st_full, st_empty, idesc, abort_flag);
      else
        produce_items<D, 1>(a, &tm_k, &tm_v, smem, st_full, st_empty, idesc, abort_flag);
    } else if (warp < kStreamWarps) {
      if (a.unit_groups == 2)
        consume_items<D, 2>(a, smem, st_full, st_empty, idesc, xch, abort_flag);
      else
        consume_items<D, 1>(a, smem, st_full, st_empty, idesc, xch, abort_flag);
    }
  }
  // the bulk copies of the merge below overwrite what was written here through the
  // generic proxy
  fence_proxy_async_smem();

  // ---- grid-wide barrier: every partial of the call is written.  Arrivals go to one
  // 64-bit count that is never reset: every call adds its grid size G (the SM count,
  // the same on every call), so call n moves it from n G to (n + 1) G and a CTA whose
  // arrival returned c waits for the next multiple of G above c.  The arrival is an
  // acquire-release add (the CTA barrier before it makes every thread's partial stores
  // part of what it releases); the last CTA's add itself completes the count, so no
  // store follows it on the critical path.
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned long long g = gridDim.x;
    const unsigned long long old = atom_add_acq_rel_gpu_u64(a.bar_count, 1ull);
    const unsigned long long target = old - old % g + g;
    if (old + 1ull != target) {
      const long long c0 = clock64();
      unsigned spins = 0;
      while (ld_acquire_gpu_u64(a.bar_count) < target) {
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
  // (the slot loop is unrolled to a bound: 8, 12 or 16 slots; every slot past the
  // call's costs each row a load and its FMAs)
  if (p.n_splits + 1 <= 8)
    merge_rows_staged<D, 8>(a, &tm_po, &tm_pl, smem, merge_bar, abort_flag);
  else if (p.n_splits + 1 <= 12)
    merge_rows_staged<D, 12>(a, &tm_po, &tm_pl, smem, merge_bar, abort_flag);
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
