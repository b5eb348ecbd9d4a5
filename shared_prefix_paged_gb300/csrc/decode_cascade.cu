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
// Suffix streaming within a CTA: warp 8 produces ring items (whole pages of every KV
// head, loaded by TMA) and warp h (< Hkv) computes KV head h of every item on
// mma.sync (see produce_suffix and consume_suffix).
#include <type_traits>

#include "merge.cuh"
#include "prefix_body.cuh"

namespace csp {
namespace {

constexpr int kThreads = prefix::kThreads;  // 352: eleven warps
constexpr int kPage = 16;
constexpr int kWarpProducer = 8;            // produces the suffix items
constexpr int kMergeBarOff = 512;           // merge barrier within the suffix barrier area

static_assert(kThreads == 352, "eleven warps: 8 softmax/consumers, 2 MMA (one the producer), loader");

template <int D>
struct SLayout {
  static constexpr int kRing = 221184;  // bytes for the suffix ring (216 KB)
  // the data area serves both roles: the prefix's Q + ring + staging, or the ring
  static constexpr int kPrefixData = prefix::Layout<D>::kData;
  static constexpr int kData = kRing > kPrefixData ? kRing : kPrefixData;
  static constexpr int kPrefixBars = kData;                        // prefix::kBarBytes
  static constexpr int kSuffixBars = kPrefixBars + prefix::kBarBytes;
  static constexpr int kSuffixBarBytes = 1024;
  static constexpr int kDynamic = kSuffixBars + kSuffixBarBytes + 1024;  // + align slack
  static_assert(kDynamic <= 227 * 1024, "one CTA per SM");
};

// Byte offset of 16-byte chunk c (of D/8) of key `key` (< 16) in one KV head's page
// as the page boxes leave it: [feature half][16 keys][128 B], 128-byte swizzle (the
// chunk index XOR the row's index mod 8): conflict-free ldmatrix.
template <int D>
__device__ __forceinline__ uint32_t kv_off(int key, int c) {
  const int r = (c >> 3) * 16 + key;
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

__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ uint4 lds_u128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ void sts_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// The transpose of an 8x8 matrix of 16-bit elements held as mma fragments: lane i
// holds row i / 4, columns 2 (i % 4) and 2 (i % 4) + 1, before and after.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// ------------------------------------------------------------------ streaming --
// The suffix phase of a CTA is its range of suffix units: unit u is the run of
// unit_pages suffix pages [j * unit_pages, (j + 1) * unit_pages) of request
// r = u / units_per_req (j = u % units_per_req), over every KV head.  Consecutive
// units of one request form a run: the CTA's piece of that request.  A run's pages go
// through a ring of ring_slots items in shared memory, item_pages pages each:
//  * warp 8 produces them.  It reads a run's query range and length (lanes 0-2) and the
//    block ids of an item's pages (one per lane), one run / one item ahead, and fills a
//    free slot: lane 2k (2k + 1) issues one TMA box with K (V) of the item's page k for
//    every KV head (16 tokens x Hkv x D, [head][feature half][16 tokens][128 B]); the
//    run's first item also brings its query rows ([token][Hq][D], one bulk copy).
//  * warp h computes KV head h of every item: S^T = K Q^T and O^T += V^T P^T on
//    mma.sync m16n8k16 (bf16 in, fp32 accumulate) with the page's 16 keys as M and the
//    head's packed rows (query, head-in-group) as N, fed by ldmatrix; the causal limit
//    (bottom-right alignment, §四) and an online softmax in base 2 with the row
//    reductions over the 8 lanes holding a row; P moves from the S^T fragments to the
//    B operand of O^T by a register transpose (movmatrix).  At the run's end the warp
//    writes its rows' normalised partial and log2-sum-exp into the piece's slot.
// Loads never hold up the computing warps: the producer alone waits for free slots.
struct ItemDesc {
  int r;        // request; < 0: no more items
  int q0, q_len, seq_len;
  int page0;    // the item's first suffix page (index within the request's suffix)
  int npages;   // pages in the item (0 for a run with no key left in this CTA's units)
  int flags;    // kFirst | kLast | kFill
  int piece;    // the run's suffix slot, counted from slot n_splits
};
constexpr int kFirst = 1;  // the run's first item (its Q rows come with it)
constexpr int kLast = 2;   // the run's last item: the piece's partial is written after it
constexpr int kFill = 4;   // ... and the run holds the request's last unit: the request's
                           // suffix slots that no CTA writes get lse = -inf

// Units [u_begin, u_end) of CTA b: a CTA that runs a prefix range takes the next
// prefix_units units in CTA order after it; the remaining R units go to the other n
// CTAs in order, evenly when R >= n (CTA c: [c R / n, (c + 1) R / n)), else one each
// to the first R.  So the CTAs holding one request's units are consecutive and each
// holds at least one of them.
__device__ __forceinline__ void unit_range_of(const DecodeArgs& a, int b, int& u_begin,
                                              int& u_end) {
  const int64_t n_units = static_cast<int64_t>(a.num_reqs) * a.units_per_req;
  const int64_t pre_units =
      min(static_cast<int64_t>(a.prefix_ctas) * a.prefix_units, n_units);
  if (b < a.prefix_ctas) {
    u_begin = static_cast<int>(min(static_cast<int64_t>(b) * a.prefix_units, pre_units));
    u_end = static_cast<int>(min(static_cast<int64_t>(b + 1) * a.prefix_units, pre_units));
    return;
  }
  const int64_t rest = n_units - pre_units;
  const int64_t n = static_cast<int64_t>(gridDim.x) - a.prefix_ctas;
  const int64_t c = b - a.prefix_ctas;
  if (rest >= n) {
    u_begin = static_cast<int>(pre_units + c * rest / n);
    u_end = static_cast<int>(pre_units + (c + 1) * rest / n);
  } else {
    u_begin = static_cast<int>(pre_units + min(c, rest));
    u_end = static_cast<int>(pre_units + min(c + 1, rest));
  }
}

// The CTA whose range holds unit u (the inverse of unit_range_of).
__device__ __forceinline__ int cta_of_unit(const DecodeArgs& a, int64_t u) {
  const int64_t n_units = static_cast<int64_t>(a.num_reqs) * a.units_per_req;
  const int64_t pre_units =
      min(static_cast<int64_t>(a.prefix_ctas) * a.prefix_units, n_units);
  if (u < pre_units) return static_cast<int>(u / a.prefix_units);
  const int64_t rest = n_units - pre_units;
  const int64_t n = static_cast<int64_t>(gridDim.x) - a.prefix_ctas;
  const int64_t up = u - pre_units;
  if (rest < n) return a.prefix_ctas + static_cast<int>(up);
  return a.prefix_ctas + static_cast<int>(((up + 1) * n - 1) / rest);
}

template <int D>
__device__ __forceinline__ void produce_suffix(const DecodeArgs& a, const CUtensorMap* tm_ks,
                                               const CUtensorMap* tm_vs, uint8_t* ring,
                                               uint64_t* st_full, uint64_t* st_empty,
                                               ItemDesc* idesc, volatile int* abort_flag) {
  const PrefixArgs& p = a.pre;
  const int lane = threadIdx.x & 31;
  const int K = a.units_per_req, PU = a.unit_pages, PI = a.item_pages, S = a.ring_slots;
  const int64_t col0 = p.cpl / kPage;  // block-table column of suffix page 0
  int u, u_end;
  unit_range_of(a, blockIdx.x, u, u_end);
  // lanes 0-2: cu_seqlens_q[r], cu_seqlens_q[r + 1], seq_lens[r]
  auto fetch_meta = [&](int r) -> int {
    int m = 0;
    if (lane == 0) m = __ldg(a.cu_seqlens_q + r);
    else if (lane == 1) m = __ldg(a.cu_seqlens_q + r + 1);
    else if (lane == 2) m = __ldg(a.seq_lens + r);
    return m;
  };
  // lane k < item_pages: the block id of suffix page pg + k of request r, read before
  // the request's length is known (an entry past its pages, within the row's stride,
  // is read but never used)
  auto fetch_ids = [&](int r, int pg) -> int {
    if (lane >= PI) return 0;
    const int64_t col = min(col0 + pg + lane, a.bt_stride - 1);
    return __ldg(a.block_table + static_cast<int64_t>(r) * a.bt_stride + col);
  };
  int item = 0;
  bool ok = true;
  int meta = 0, ids = 0;
  if (u < u_end) {
    const int r = u / K;
    meta = fetch_meta(r);
    ids = fetch_ids(r, (u - r * K) * PU);
  }
  while (ok && u < u_end) {
    const int r = u / K;
    const int ja = u - r * K;
    const int jb = min(K - 1, u_end - 1 - r * K);  // the run's last unit
    const int q0 = __shfl_sync(0xffffffffu, meta, 0);
    // (at most max_rows packed rows per KV head: the size of the slot's Q area)
    const int q_len = min(__shfl_sync(0xffffffffu, meta, 1) - q0, a.max_rows / p.group);
    const int seq_len = __shfl_sync(0xffffffffu, meta, 2);
    int it_ids = ids;
    // the next run's metadata and first block ids, one run ahead
    const int u_next = r * K + jb + 1;
    if (u_next < u_end) {
      const int rn = u_next / K;
      meta = fetch_meta(rn);
      ids = fetch_ids(rn, (u_next - rn * K) * PU);
    }
    if (q_len > 0) {  // a request without query rows this step has nothing to compute
      const int n_r = max(0, (seq_len - p.cpl + kPage - 1) / kPage);
      const int p_lo = ja * PU;
      const int npg = max(0, min((jb + 1) * PU, n_r) - p_lo);
      const int n_items = max(1, (npg + PI - 1) / PI);
      const int piece = static_cast<int>(blockIdx.x) - cta_of_unit(a, static_cast<int64_t>(r) * K);
      const bool holds_last = jb == K - 1;
      const uint32_t qbytes = static_cast<uint32_t>(q_len) * p.num_q_heads * D * 2;
      for (int it = 0; it < n_items; ++it) {
        const int slot = item % S;
        if (item >= S &&
            !(ok = warp_mbar_wait(&st_empty[slot], ((item / S) - 1) & 1, abort_flag, p.status)))
          break;
        const int pg0 = p_lo + it * PI;
        const int pages = max(0, min(PI, npg - it * PI));
        // the block ids of the run's next item, one item ahead
        const int nxt = it + 1 < n_items ? fetch_ids(r, pg0 + PI) : 0;
        const uint32_t qb = it == 0 ? qbytes : 0u;
        if (lane == 0) {
          ItemDesc& d = idesc[slot];
          d.r = r;
          d.q0 = q0;
          d.q_len = q_len;
          d.seq_len = seq_len;
          d.page0 = pg0;
          d.npages = pages;
          d.flags = (it == 0 ? kFirst : 0) | (it == n_items - 1 ? kLast : 0) |
                    (it == n_items - 1 && holds_last ? kFill : 0);
          d.piece = piece;
          mbar_arrive_expect_tx(&st_full[slot],
                                static_cast<uint32_t>(pages) * 2u * a.page_bytes + qb);
        }
        __syncwarp();
        uint8_t* base = ring + static_cast<size_t>(slot) * a.item_bytes;
        const int blk = __shfl_sync(0xffffffffu, it_ids, (lane >> 1) & 31);
        if (lane < 2 * pages) {
          const int k = lane >> 1, kv = lane & 1;
          tma_load_4d(base + (2 * k + kv) * a.page_bytes, kv ? tm_vs : tm_ks, &st_full[slot], 0,
                      blk * kPage, 0, 0);
        }
        if (qb > 0 && lane == 31)
          bulk_load(base + a.q_off, a.q + static_cast<int64_t>(q0) * p.num_q_heads * D, qb,
                    &st_full[slot]);
        ++item;
        it_ids = nxt;
      }
    }
    u = u_next;
  }
  // the end: one marker item that every consumer reads
  if (ok) {
    const int slot = item % S;
    if (item < S ||
        warp_mbar_wait(&st_empty[slot], ((item / S) - 1) & 1, abort_flag, p.status)) {
      if (lane == 0) {
        idesc[slot].r = -1;
        mbar_arrive_expect_tx(&st_full[slot], 0u);
      }
    }
  }
  __syncwarp();
}

// One page (16 keys) of KV head h for the warp's kNT x 8 packed rows.
template <int D, int kNT>
__device__ __forceinline__ void page_step(uint32_t kb, uint32_t vb, int key0,
                                          const uint32_t (&qf)[kNT][D / 16][2],
                                          float (&o)[D / 16][kNT][4], float (&m_run)[kNT][2],
                                          float (&l_part)[kNT][2], const int (&lim)[kNT][2],
                                          float scale_log2, int lane) {
  constexpr int kMT = D / 16;
  const int g = lane >> 2;
  // S^T = K Q^T: two accumulators per n-tile (even / odd k-steps) halve the chain
  float s[kNT][2][4];
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
    for (int x = 0; x < 2; ++x) s[nt][x][0] = s[nt][x][1] = s[nt][x][2] = s[nt][x][3] = 0.f;
  {
    const int key = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
    for (int kk = 0; kk < kMT; ++kk) {
      uint32_t ka[4];
      ldmatrix_x4(kb + kv_off<D>(key, kk * 2 + (lane >> 4)), ka[0], ka[1], ka[2], ka[3]);
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) mma_bf16_16816(s[nt][kk & 1], ka, qf[nt][kk][0], qf[nt][kk][1]);
    }
  }
  // masked scores (keys past a row's causal limit, or past the request), online softmax
  // in base 2; the row's 16 keys sit on the 8 lanes of one column (xor 4, 8, 16)
  uint32_t pb[kNT][2];
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt) {
    float pv[4];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float v0 = key0 + g <= lim[nt][e] ? (s[nt][0][e] + s[nt][1][e]) * scale_log2 : -INFINITY;
      const float v1 =
          key0 + g + 8 <= lim[nt][e] ? (s[nt][0][2 + e] + s[nt][1][2 + e]) * scale_log2 : -INFINITY;
      float mx = fmaxf(v0, v1);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      // keep the running max unless it grows by more than 2^8 (always on the row's
      // first unmasked keys, where it is -inf): p = 2^(s - m) <= 256, and O and l need
      // rescaling only now and then
      if (mx > m_run[nt][e] + 8.f) {
        const float alpha = fast_exp2(m_run[nt][e] - mx);
        l_part[nt][e] *= alpha;
#pragma unroll
        for (int mt = 0; mt < kMT; ++mt) {
          o[mt][nt][e] *= alpha;
          o[mt][nt][2 + e] *= alpha;
        }
        m_run[nt][e] = mx;
      }
      const float mu = m_run[nt][e] == -INFINITY ? 0.f : m_run[nt][e];
      pv[e] = fast_exp2(v0 - mu);
      pv[2 + e] = fast_exp2(v1 - mu);
      l_part[nt][e] += pv[e] + pv[2 + e];
    }
    // P^T (keys x rows) as two 8x8 blocks -> the B fragments of O^T += V^T P^T
    pb[nt][0] = movmatrix_trans(pack_bf16x2(pv[0], pv[1]));
    pb[nt][1] = movmatrix_trans(pack_bf16x2(pv[2], pv[3]));
  }
  // O^T += V^T P^T: m-tile mt holds features [16 mt, 16 mt + 16)
  {
    const int key = (lane & 7) + ((lane >> 4) & 1) * 8;
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt) {
      uint32_t va[4];
      ldmatrix_x4_trans(vb + kv_off<D>(key, mt * 2 + ((lane >> 3) & 1)), va[0], va[1], va[2],
                        va[3]);
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) mma_bf16_16816(o[mt][nt], va, pb[nt][0], pb[nt][1]);
    }
  }
}

// Warp h (< Hkv) computes KV head h of every item of the CTA's suffix stream, its
// packed rows in kNT n-tiles of 8.
template <int D, int kNT>
__device__ __forceinline__ void consume_suffix(const DecodeArgs& a, uint8_t* ring,
                                               uint64_t* st_full, uint64_t* st_empty,
                                               const ItemDesc* idesc, volatile int* abort_flag) {
  const PrefixArgs& p = a.pre;
  constexpr int kMT = D / 16;
  constexpr int kHB = kPage * D * 2;  // one KV head's page inside a page box
  const int lane = threadIdx.x & 31;
  const int h = threadIdx.x >> 5;     // the KV head
  const int g = lane >> 2, t = lane & 3;
  const int S = a.ring_slots;
  const uint32_t rbase = smem_u32(ring);
  uint32_t qf[kNT][kMT][2];
  float o[kMT][kNT][4];
  float m_run[kNT][2], l_part[kNT][2];
  int lim[kNT][2];  // the last key position a row sees (-1: a padding row)
  int rows_valid = 0, q0 = 0;
  for (int item = 0;; ++item) {
    const int slot = item % S;
    const uint32_t par = (item / S) & 1;
    if (!warp_mbar_wait(&st_full[slot], par, abort_flag, p.status)) break;
    // every lane observes the completed phase (the copied bytes are visible to it)
    mbar_test_wait(&st_full[slot], par);
    const ItemDesc d = idesc[slot];
    if (d.r < 0) break;
    const uint32_t ib = rbase + slot * a.item_bytes;
    if (d.flags & kFirst) {
      q0 = d.q0;
      rows_valid = d.q_len * p.group;
      // B fragments of Q^T: lane (g, t) holds row nt*8 + g, features kk*16 + 2t (+1)
      // and kk*16 + 8 + 2t (+1), from the item's Q rows ([token][Hq][D])
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) {
        const int n = nt * 8 + g;
        const bool in = n < rows_valid;
        const int qi = in ? n / p.group : 0, j = in ? n - qi * p.group : 0;
        const uint32_t qrow =
            ib + a.q_off + static_cast<uint32_t>((qi * p.num_q_heads + h * p.group + j) * D * 2);
#pragma unroll
        for (int kk = 0; kk < kMT; ++kk) {
          qf[nt][kk][0] = in ? lds_u32(qrow + (kk * 16 + 2 * t) * 2) : 0u;
          qf[nt][kk][1] = in ? lds_u32(qrow + (kk * 16 + 8 + 2 * t) * 2) : 0u;
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int n2 = nt * 8 + 2 * t + e;
          lim[nt][e] = n2 < rows_valid ? d.seq_len - d.q_len + n2 / p.group : -1;
          m_run[nt][e] = -INFINITY;
          l_part[nt][e] = 0.f;
        }
      }
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.f;
    }
    for (int k = 0; k < d.npages; ++k) {
      const uint32_t kb = ib + (2 * k) * a.page_bytes + h * kHB;
      const uint32_t vb = kb + a.page_bytes;
      const int key0 = p.cpl + (d.page0 + k) * kPage;
      if (key0 + kPage > d.seq_len) {
        // keys past the request: zero their V rows (P is 0 there, but the page may
        // hold anything, and 0 x NaN is NaN)
        const int nv = max(0, d.seq_len - key0);
        for (int x = lane; x < kPage * (D / 8); x += 32) {
          const int key = x / (D / 8), c = x % (D / 8);
          if (key >= nv)
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(vb + kv_off<D>(key, c)),
                         "r"(0u)
                         : "memory");
        }
        __syncwarp();
      }
      page_step<D, kNT>(kb, vb, key0, qf, o, m_run, l_part, lim, p.scale_log2, lane);
    }
    if (d.flags & kLast) {
      // ---- the piece's partial: normalised rows (bf16) and their log2-sum-exp
      float inv[kNT][2], lse2[kNT][2];
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float l = l_part[nt][e];
          l += __shfl_xor_sync(0xffffffffu, l, 4);
          l += __shfl_xor_sync(0xffffffffu, l, 8);
          l += __shfl_xor_sync(0xffffffffu, l, 16);
          inv[nt][e] = l > 0.f ? 1.f / l : 0.f;
          lse2[nt][e] = l > 0.f ? m_run[nt][e] + log2f(l) : -INFINITY;
        }
      // stage the rows [row][D] in this head's K page of the item (read already)
      const uint32_t stg = ib + h * kHB;
      __syncwarp();
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int n = nt * 8 + 2 * t + e;
            const uint32_t at = stg + static_cast<uint32_t>((n * D + mt * 16 + g) * 2);
            __nv_bfloat16 lo = __float2bfloat16_rn(o[mt][nt][e] * inv[nt][e]);
            __nv_bfloat16 hi = __float2bfloat16_rn(o[mt][nt][2 + e] * inv[nt][e]);
            sts_u16(at, *reinterpret_cast<uint16_t*>(&lo));
            sts_u16(at + 16, *reinterpret_cast<uint16_t*>(&hi));
          }
      __syncwarp();
      const int64_t rows_all = static_cast<int64_t>(p.total_q) * p.num_q_heads;
      const int slot_idx = p.n_splits + d.piece;
      auto grow = [&](int n) {
        const int qi = n / p.group;
        return static_cast<int64_t>(q0 + qi) * p.num_q_heads + h * p.group + (n - qi * p.group);
      };
      for (int x = lane; x < rows_valid * (D / 8); x += 32) {
        const int n = x / (D / 8), c = x % (D / 8);
        const uint4 v = lds_u128(stg + static_cast<uint32_t>((n * D + c * 8) * 2));
        *reinterpret_cast<uint4*>(p.part_o + (slot_idx * rows_all + grow(n)) * D + c * 8) = v;
      }
      if (g == 0) {
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int n = nt * 8 + 2 * t + e;
            if (n < rows_valid) p.part_lse[slot_idx * p.lse_stride + grow(n)] = lse2[nt][e];
          }
      }
      if (d.flags & kFill) {
        // this CTA holds the request's last unit: the request's suffix slots of CTAs
        // that hold none of its units (past the CTAs that do) read lse = -inf
        const int first = cta_of_unit(a, static_cast<int64_t>(d.r) * a.units_per_req);
        for (int sidx = 0; sidx < a.suffix_slots; ++sidx) {
          bool filled = false;
          if (first + sidx <= static_cast<int>(blockIdx.x)) {
            int ub, ue;
            unit_range_of(a, first + sidx, ub, ue);
            filled = ub < ue;
          }
          if (filled) continue;
          for (int n = lane; n < rows_valid; n += 32)
            p.part_lse[(p.n_splits + sidx) * p.lse_stride + grow(n)] = -INFINITY;
        }
      }
      __syncwarp();
    }
    // the item goes back to the producer (its copies will overwrite what this warp
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
// slot count.  An empty slot (lse -inf) gets weight 0 and its rows are not read into
// the sum (a suffix slot that no piece wrote holds whatever an earlier call left).
template <int D, int kSlots>
__device__ __forceinline__ void merge_rows_staged(const DecodeArgs& a, const CUtensorMap* tm_po,
                                                  const CUtensorMap* tm_pl, uint8_t* smem,
                                                  uint64_t* bar, volatile int* abort_flag) {
  constexpr int kF = D / 16;
  using Vec = typename std::conditional<kF == 8, uint4, uint2>::type;
  const PrefixArgs& p = a.pre;
  const int n = p.n_splits + a.suffix_slots;  // slots
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
        if (l[s] == 0.f) continue;
        const uint32_t* u = reinterpret_cast<const uint32_t*>(&v[s]);
#pragma unroll
        for (int f = 0; f < kF / 2; ++f) {
          const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[f]));
          acc[2 * f] = fmaf(l[s], x.x, acc[2 * f]);
          acc[2 * f + 1] = fmaf(l[s], x.y, acc[2 * f + 1]);
        }
      }
      const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
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
          a.lse[row] = wsum > 0.f ? (mx + log2f(wsum)) * 0.69314718055994531f : -INFINITY;
      }
    }
    // the next chunk's copies overwrite what was read here
    __syncthreads();
  }
}

// ------------------------------------------------------------------ the kernel --
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    decode_cascade_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_v,
                          const __grid_constant__ CUtensorMap tm_kp,
                          const __grid_constant__ CUtensorMap tm_ks,
                          const __grid_constant__ CUtensorMap tm_vs,
                          const __grid_constant__ CUtensorMap tm_po,
                          const __grid_constant__ CUtensorMap tm_pl, const DecodeArgs a) {
  using L = SLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const PrefixArgs& p = a.pre;
  const int warp = threadIdx.x >> 5;
  // generation of the grid barrier at the end (read now, off the critical path)
  const unsigned g0 = threadIdx.x == 0 ? ld_acquire_gpu_u32(a.bar_gen) : 0u;
  // the first TMA through each map would otherwise wait for its descriptor
  if (threadIdx.x == 32 * kWarpProducer) {
    prefetch_tensormap(&tm_ks);
    prefetch_tensormap(&tm_vs);
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

  // ---- role 2: the suffix units, produced by warp 8 and computed by warps [0, Hkv)
  const int S = a.ring_slots;
  uint64_t* st_full = reinterpret_cast<uint64_t*>(smem + L::kSuffixBars);  // [S]
  uint64_t* st_empty = st_full + kDecodeMaxRing;                           // [S]
  ItemDesc* idesc = reinterpret_cast<ItemDesc*>(st_empty + kDecodeMaxRing); // [S]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(idesc + kDecodeMaxRing);
  uint64_t* merge_bar = reinterpret_cast<uint64_t*>(smem + L::kSuffixBars + kMergeBarOff);
  int u_begin, u_end;
  unit_range_of(a, blockIdx.x, u_begin, u_end);
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&st_full[i], 1);                 // the producer's expect_tx arrival
      mbar_init(&st_empty[i], p.num_kv_heads);  // one arrival per consumer warp
    }
    mbar_init(merge_bar, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  if (u_begin < u_end) {  // (a prefix CTA may have none)
    if (warp == kWarpProducer) {
      produce_suffix<D>(a, &tm_ks, &tm_vs, smem, st_full, st_empty, idesc, abort_flag);
    } else if (warp < p.num_kv_heads) {
      if (a.max_rows <= 8)
        consume_suffix<D, 1>(a, smem, st_full, st_empty, idesc, abort_flag);
      else
        consume_suffix<D, 2>(a, smem, st_full, st_empty, idesc, abort_flag);
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
  if (p.n_splits + a.suffix_slots <= 8)
    merge_rows_staged<D, 8>(a, &tm_po, &tm_pl, smem, merge_bar, abort_flag);
  else
    merge_rows_staged<D, kDecodeMaxParts>(a, &tm_po, &tm_pl, smem, merge_bar, abort_flag);
}

template <int D>
cudaError_t launch_decode_d(const CUtensorMap& tm_q, const CUtensorMap& tm_v,
                            const CUtensorMap& tm_kp, const CUtensorMap& tm_ks,
                            const CUtensorMap& tm_vs, const CUtensorMap& tm_po,
                            const CUtensorMap& tm_pl, const DecodeArgs& a, int grid,
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
  return cudaLaunchKernelEx(&cfg, decode_cascade_kernel<D>, tm_q, tm_v, tm_kp, tm_ks, tm_vs,
                            tm_po, tm_pl, a);
}

}  // namespace

int decode_ring_bytes() { return SLayout<128>::kRing; }

cudaError_t launch_decode(int head_dim, const CUtensorMap& tm_q, const CUtensorMap& tm_v,
                          const CUtensorMap& tm_kp, const CUtensorMap& tm_ks,
                          const CUtensorMap& tm_vs, const CUtensorMap& tm_po,
                          const CUtensorMap& tm_pl, const DecodeArgs& a, int grid,
                          cudaStream_t stream) {
  if (head_dim == 64)
    return launch_decode_d<64>(tm_q, tm_v, tm_kp, tm_ks, tm_vs, tm_po, tm_pl, a, grid, stream);
  return launch_decode_d<128>(tm_q, tm_v, tm_kp, tm_ks, tm_vs, tm_po, tm_pl, a, grid, stream);
}

}  // namespace csp
