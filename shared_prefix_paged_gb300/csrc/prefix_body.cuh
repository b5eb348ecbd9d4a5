// prefix_body.cuh — one CTA's share of the prefix phase of cascade attention, on
// tcgen05 tensor cores.  Used by the standalone prefix kernel (prefix_attn.cu) and
// by the single-kernel decode schedule (decode_cascade.cu).
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
//  * warp 10 stages K and V by TMA into a 4-deep ring of 64-key tiles (128-byte
//    swizzle): K as [feature half][64 keys][128 B] (one box per page and half), V as
//    [page][feature half][16 keys][128 B] (one box per page); it alone waits for free
//    stages, so the softmax warps never issue copies;
//  * per M tile, S = Q K^T (M=128, N=64) goes into one of two TMEM buffers, so the
//    tensor core computes S(i+1) while the softmax works on S(i); P (bf16) is
//    written back into the S buffer and used from TMEM as the A operand of
//    O += P V (N = D).  The two M tiles use all 512 TMEM columns;
//  * two softmax warpgroups (one per M tile) own one TMEM lane (row) per thread:
//    online softmax in base 2 on the special-function unit, O rescaled in TMEM only
//    when the running max grows by more than 2^8; warps 8 and 9 issue the MMAs (one
//    per M tile), warp 9 also the Q load;
//  * a CTA covers one range of the prefix's key tiles and stages its normalised rows
//    (bf16) through shared memory, then writes them, coalesced, into workspace slot
//    `split`, with the log2-sum-exp of each row beside them; a later merge
//    (merge.cuh) combines the slots with the suffix phase's partials.
#pragma once

#include "common.cuh"
#include "kernels.cuh"

namespace csp {
namespace prefix {

constexpr int kRowsM = 128;    // rows per M tile
constexpr int kRowsCta = 256;  // two M tiles
constexpr int kKeysN = 64;     // keys per tile
constexpr int kPage = 16;      // tokens per KV page
constexpr int kPagesPerTile = kKeysN / kPage;
constexpr int kStages = 4;
constexpr int kThreads = 352;  // 2 softmax warpgroups, two MMA issuers, the K/V loader
// An FP8 (E4M3) KV cache: the loader warp and one more warp widen each tile to f16
// (exact: E4M3 is a subset of f16) for MMAs with f16 operands.
constexpr int kThreadsF8 = 384;
constexpr int kWarpConv = 11;
constexpr int kF8Stages = 6;   // E4M3 tiles in flight (the f16 ring is then 2 deep)
constexpr int kWarpMma = 8;
constexpr int kWarpTma = 9;    // Q by TMA, then the MMA issuer of M tile 1
constexpr int kWarpLoad = 10;  // K and V by TMA
template <int D, bool kF8 = false>
struct Layout {
  static constexpr int kStagesL = kF8 ? 2 : kStages;    // 16-bit K/V tiles in the ring
  static constexpr int kHalves = D / 64;
  static constexpr int kQHalf = kRowsM * 128;           // 128 rows x 64 bf16
  static constexpr int kKVHalf = kKeysN * 128;          // 64 keys x 64 bf16
  static constexpr int kQTile = kHalves * kQHalf;       // one M tile of Q
  static constexpr int kKVBytes = kHalves * kKVHalf;    // one K (or V) tile
  static constexpr int kVPage = kPage * D * 2;          // one page of V: both halves
  static constexpr int kQ = 0;                          // [2 M tiles][halves]
  static constexpr int kK0 = kQ + 2 * kQTile;
  static constexpr int kV0 = kK0 + kStagesL * kKVBytes;
  // E4M3 tiles as loaded: K [64 keys][D bytes], then V the same, per stage
  static constexpr int kF8Tile = kKeysN * D;
  static constexpr int kF8Stage = 2 * kF8Tile;
  static constexpr int kF8Ring = kV0 + kStagesL * kKVBytes;
  static constexpr int kRing = kF8Ring + (kF8 ? kF8Stages * kF8Stage : 0);
  // after the main loop, [0, kRing) stages the CTA's 256 normalised rows:
  // [row][D + 8] bf16 (the padding spreads the rows one warp writes over all banks)
  static constexpr int kStageRow = D + 8;
  static_assert(kRowsCta * kStageRow * 2 <= kRing, "staging buffer fits Q + ring");
  static constexpr int kLse = kRing;                    // float [256]
  static constexpr int kData = kLse + kRowsCta * 4;     // end of the data area
};

// Bytes of the caller's barrier area: up to 25 mbarriers, the TMEM slot and the abort
// flag.
constexpr int kBarBytes = 256;

// Where one CTA's rows and keys come from.  The prefix phase: the rows are every
// query row of the batch, the keys [0, cpl) through block-table row 0, unmasked.  A
// request's own range (paged_tc.cu): the rows are that request's, the keys
// [key0, key_end) through its block-table row, and packed row rho sees keys up to
// causal_base + rho / group (bottom-right causal alignment).
struct RangeGeom {
  const int32_t* bt;  // block-table row holding the range's pages
  int key0;           // key position of tile 0, a multiple of the page size
  int key_end;        // keys at or past it are neither loaded nor seen
  int tok0;           // Q token of packed row 0
  int prow0;          // the CTA's first packed row
  int rows_total;     // packed rows that exist; rows past them are padding
  int causal_base;    // kCausal: packed row rho sees keys <= causal_base + rho / group
};

__device__ __forceinline__ RangeGeom prefix_geom(const PrefixArgs& a, int pair) {
  RangeGeom g;
  g.bt = a.block_table;
  g.key0 = a.key_lo;
  g.key_end = a.cpl;
  g.tok0 = a.tok0;
  g.prow0 = pair * 256;
  g.rows_total = a.total_q * a.group;
  g.causal_base = 0;
  return g;
}

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

// One CTA's share of the prefix phase: packed rows [256 pair, 256 pair + 256) of KV
// head kvh against the prefix's 64-key tiles [t_first, t_last); the normalised
// partial goes to workspace slot `split`.  Called by every thread of a 320-thread CTA.
// smem: 1024-byte aligned, Layout<D>::kRing + 1 KB bytes (Q, the K/V ring, then the
// staging buffer and the row LSEs); bars: kBarBytes for the mbarriers, the TMEM slot
// and the abort flag.  Allocates and frees all 512 TMEM columns.  Ends with every
// global store of the partial issued; the caller syncs before reusing smem.
// With kCausal, rows and keys come from `geo` (a request's own range, causal mask)
// and the CTA stops once its 256 normalised rows (bf16, [row][Layout::kStageRow] at
// smem) and their log2-sum-exp (float [256] at smem + Layout::kLse; -inf for a row
// that saw no key) are staged and visible to every thread: the caller writes them.
// tm_k: the K cache as {D, Hkv, tokens} with boxes {64, 1, 16} (one page, one half);
// tm_v: the V cache as {64, tokens, D / 64, Hkv} with boxes {64, 16, D / 64, 1} (one
// page, both halves); both with the 128-byte swizzle.
template <int D, bool kCausal = false, bool kF8 = false>
__device__ __forceinline__ void prefix_range(const CUtensorMap* tm_q_p,
                                             const CUtensorMap* tm_k_p,
                                             const CUtensorMap* tm_v_p, const PrefixArgs& a,
                                             const RangeGeom& geo, int kvh, int split,
                                             int t_first, int t_last, uint8_t* smem,
                                             uint64_t* bars) {
  using L = Layout<D, kF8>;
  constexpr int kS = L::kStagesL;
  constexpr int kNThreads = kF8 ? kThreadsF8 : kThreads;
  const CUtensorMap& tm_q = *tm_q_p;
  const CUtensorMap& tm_k = *tm_k_p;
  const CUtensorMap& tm_v = *tm_v_p;
  uint64_t* bar_q = bars + 0;
  uint64_t* kv_full = bars + 1;   // [kS]
  uint64_t* kv_empty = bars + 1 + kS;  // [kS]
  uint64_t* s_full = bars + 1 + 2 * kS;    // [2 tiles][2 buffers]
  uint64_t* p_full = bars + 5 + 2 * kS;    // [2 tiles][2 buffers]
  uint64_t* o_last = bars + 11 + 2 * kS;   // [2 tiles] the last PV (9, 10 unused)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 13 + 2 * kS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 14 + 2 * kS);
  uint64_t* f8_full = bars + 15 + 2 * kS;               // [kF8Stages] E4M3 tiles landed
  uint64_t* f8_empty = bars + 15 + 2 * kS + kF8Stages;  // [kF8Stages] E4M3 tiles widened
  uint64_t* tail_in = bars + 15 + 2 * kS;   // bf16: the last tile landed (see the loader)
  // A range that ends inside a page (a request's last page) leaves slots past its end
  // in that page: whatever the cache holds there (NaN included) would reach O through
  // P = 0 times V in the MMA, so those V rows are zeroed before the PV reads them.
  const bool ragged_end = kCausal && (geo.key_end % kPage) != 0;
  static_assert((kF8 ? 15 + 2 * kS + 2 * kF8Stages : 16 + 2 * kS) * 8 <= kBarBytes,
                "barrier area");
  static_assert(!kF8 || kWarpConv * 32 + 32 == kThreadsF8, "the converter warp is the last");

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int ntiles = t_last - t_first;
  // The CTAs of the other KV heads read the same pages (other rows of them): each
  // head starts at its own point of the range, so at any time the CTAs of one range
  // read different pages rather than all hitting the same ones together.
  const int rot = (!kCausal && ntiles > 0) ? (kvh * ntiles) / a.num_kv_heads : 0;
  auto tile_of = [&](int i) {
    const int r = i + rot;
    return t_first + (r >= ntiles ? r - ntiles : r);
  };
  const int rows_total = geo.rows_total;             // packed rows of this KV head
  const bool has_m1 = geo.prow0 + kRowsM < rows_total;  // second M tile has rows

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < kS; ++s) {
      // bf16: the loader's expect_tx, the TMA bytes complete it; E4M3: every thread
      // of the two converter warps
      mbar_init(&kv_full[s], kF8 ? 64 : 1);
      mbar_init(&kv_empty[s], has_m1 ? 2 : 1);  // one commit per M tile's issuer
    }
    if constexpr (kF8) {
      for (int s = 0; s < kF8Stages; ++s) {
        mbar_init(&f8_full[s], 1);    // the loader's expect_tx
        mbar_init(&f8_empty[s], 64);  // every converter thread
      }
    } else {
      mbar_init(tail_in, 1);
    }
    for (int b = 0; b < 4; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_full[b], 128);
    }
    for (int m = 0; m < 2; ++m) mbar_init(&o_last[m], 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == kWarpMma) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kWarpTma) {
    // ------------------------------------------------------- Q by TMA (once) --
    if (lane == 0 && ntiles > 0) {  // an empty key range loads nothing at all
      prefetch_tensormap(&tm_q);
      const int mts = has_m1 ? 2 : 1;
      mbar_arrive_expect_tx(bar_q, mts * L::kQTile);
      for (int m = 0; m < mts; ++m)
#pragma unroll
        for (int h = 0; h < L::kHalves; ++h)
          tma_load_3d(smem + L::kQ + m * L::kQTile + h * L::kQHalf, &tm_q, bar_q, h * 64,
                      kvh * a.group, geo.tok0 + (geo.prow0 + m * kRowsM) / a.group);
    }
  }
  // ------------------------------------------------- MMA issuers, one per M tile --
  // Warp 8 issues for M tile 0, warp 9 (once Q is on its way) for M tile 1.  An MMA
  // issue is held until the tensor pipe takes it, so a single issuer stuck behind one
  // M tile's S could not issue the other tile's ready PV; with one issuer each, each
  // warpgroup's S -> softmax -> PV chain advances on its own.
  // Event loop: S(j) as soon as its K tile is in (and PV(j-2), the last reader of its
  // TMEM buffer, has been issued); PV(j) as soon as this warpgroup's P(j) is.  Stage j
  // goes back to the loaders once every M tile's PV(j) is done (kv_empty counts one
  // commit per issuer).
  if ((warp == kWarpMma || (warp == kWarpTma && has_m1)) && lane == 0 && ntiles > 0) {
    const int m = warp == kWarpMma ? 0 : 1;
    constexpr uint32_t kIdS =
        kF8 ? umma_idesc_f16(128, kKeysN, 0, 0) : umma_idesc_bf16(128, kKeysN, 0, 0);
    constexpr uint32_t kIdO = kF8 ? umma_idesc_f16(128, D, 0, 1) : umma_idesc_bf16(128, D, 0, 1);
    const uint32_t q_addr = smem_u32(smem + L::kQ + m * L::kQTile);
    const uint32_t tm = tmem + m * 256;
    auto issue_s = [&](int i) {
      const uint32_t k_addr = smem_u32(smem + L::kK0 + (i % kS) * L::kKVBytes);
      const uint32_t d = tm + (i & 1) * kKeysN;
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t qo = (k >> 2) * L::kQHalf + (k & 3) * 32;
        const uint32_t ko = (k >> 2) * L::kKVHalf + (k & 3) * 32;
        umma_bf16(d, umma_desc_sw128(q_addr + qo, 16, 1024),
                  umma_desc_sw128(k_addr + ko, 16, 1024), kIdS, k > 0 ? 1u : 0u);
      }
      umma_commit(&s_full[m * 2 + (i & 1)]);
    };
    bool ok = mbar_wait(bar_q, 0, abort_flag, a.status);
    int next_s = 0, next_pv = 0;
    unsigned idle = 0;
    long long c0 = 0;
    while (ok && next_pv < ntiles) {
      bool progressed = false;
      if (next_s < ntiles && next_s <= next_pv + 1 &&
          mbar_test_wait(&kv_full[next_s % kS], (next_s / kS) & 1)) {
        tc_fence_after();
        issue_s(next_s);
        ++next_s;
        progressed = true;
      }
      if (next_pv < next_s &&
          mbar_test_wait(&p_full[m * 2 + (next_pv & 1)], (next_pv >> 1) & 1)) {
        tc_fence_after();
        const int i = next_pv;
        const uint32_t v_addr = smem_u32(smem + L::kV0 + (i % kS) * L::kKVBytes);
        const uint32_t p_tmem = tm + (i & 1) * kKeysN;
#pragma unroll
        for (int kk = 0; kk < kKeysN / 16; ++kk)  // 16 keys = one page of V
          umma_bf16_tmem_a(tm + 2 * kKeysN, p_tmem + kk * 8,
                           umma_desc_sw128(v_addr + kk * L::kVPage, kPage * 128, 1024), kIdO,
                           (i > 0 || kk > 0) ? 1u : 0u);
        if (i == ntiles - 1) umma_commit(&o_last[m]);
        umma_commit(&kv_empty[i % kS]);
        ++next_pv;
        progressed = true;
      }
      if (progressed) {
        idle = 0;
      } else if ((++idle & 63u) == 0) {
        // bounded: nothing became ready for kWaitLimitCycles
        if (*abort_flag) {
          ok = false;
        } else if (idle == 64) {
          c0 = clock64();
        } else if (clock64() - c0 > kWaitLimitCycles) {
          *abort_flag = 1;
          if (a.status) atomicCAS(a.status, 0, kErrTimeout);
          ok = false;
        }
      }
    }
  }
  // ------------------------------------------------------- K/V loader (TMA) --
  // Tile j goes into stage j % kStages once PV(j - kStages) of every M tile is done.
  // Lane l holds the block id of page l % 4 of tile l / 4 of a window of eight tiles,
  // read a window ahead.  A page wholly past the range is loaded from an out-of-range
  // token coordinate: TMA fills it with zeros (no NaN from a page the cache never
  // wrote can reach O).
  if (!kF8 && warp == kWarpLoad && ntiles > 0) {
    constexpr int kIdTiles = 32 / kPagesPerTile;
    constexpr int kKBoxes = kPagesPerTile * L::kHalves;
    const int npages = (geo.key_end - geo.key0 + kPage - 1) / kPage;
    const int32_t* bt_pages = geo.bt + geo.key0 / kPage;
    auto load_ids = [&](int i_base) {
      const int i = i_base + lane / kPagesPerTile;
      const int page = tile_of(i) * kPagesPerTile + (lane & (kPagesPerTile - 1));
      return i < ntiles && page < npages ? __ldg(bt_pages + page) : -1;
    };
    int ids_cur = load_ids(0);
    int ids_nxt = ntiles > kIdTiles ? load_ids(kIdTiles) : -1;
    int issued = 0;
    for (int j = 0; j < ntiles; ++j) {
      const int st = j % kS;
      if (j >= kS && !warp_mbar_wait(&kv_empty[st], ((j / kS) - 1) & 1, abort_flag, a.status))
        break;
      if (j > 0 && j % kIdTiles == 0) {
        ids_cur = ids_nxt;
        ids_nxt = j + kIdTiles < ntiles ? load_ids(j + kIdTiles) : -1;
      }
      // a ragged last tile lands on tail_in; the warp zeroes its slots past the range
      // and then releases the stage (below)
      const bool fix = ragged_end && j == ntiles - 1;
      uint64_t* land = fix ? tail_in : &kv_full[st];
      if (lane == 0) mbar_arrive_expect_tx(land, 2 * L::kKVBytes);
      __syncwarp();
      // lanes [0, kKBoxes): K page lane / halves, half lane % halves; then one lane per
      // page of V
      const bool is_k = lane < kKBoxes;
      const int q = is_k ? lane / L::kHalves : lane - kKBoxes;
      const int blk = __shfl_sync(0xffffffffu, ids_cur, ((j % kIdTiles) * kPagesPerTile + q) & 31);
      const int tok = blk >= 0 ? blk * kPage : -kPage;  // -16: a box of zeros
      if (is_k) {
        const int h = lane % L::kHalves;
        tma_load_3d(smem + L::kK0 + st * L::kKVBytes + h * L::kKVHalf + q * (kPage * 128),
                    &tm_k, land, h * 64, kvh, tok);
      } else if (lane < kKBoxes + kPagesPerTile) {
        tma_load_4d(smem + L::kV0 + st * L::kKVBytes + q * L::kVPage, &tm_v, land, 0, tok, 0,
                    kvh);
      }
      if (fix) {
        // V rows of keys [key_end, the end of its page) of this tile: zero, made
        // visible to the tensor core's proxy, then the stage is released
        if (!warp_mbar_wait(tail_in, 0, abort_flag, a.status)) {
          if (lane == 0) {
            const long long c0 = clock64();
            while (!mbar_try_wait(tail_in, 0) && clock64() - c0 < kWaitLimitCycles) {
            }
          }
          __syncwarp();
          break;
        }
        const int kt = geo.key_end - (geo.key0 + tile_of(j) * kKeysN);  // first key to clear
        const int page = kt / kPage, r0 = kt % kPage;
        const int n16 = (kPage - r0) * L::kHalves * 8;                  // 16-byte pieces
        for (int x = lane; x < n16; x += 32) {
          const int r = r0 + x / (L::kHalves * 8);
          const int h = (x / 8) % L::kHalves;
          *reinterpret_cast<uint4*>(smem + L::kV0 + st * L::kKVBytes + page * L::kVPage +
                                    h * (kPage * 128) + r * 128 + (x % 8) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&kv_full[st]);
        // its phase of kv_full is complete: the wait below must count it, or it would
        // wait on the stage's previous (already passed) phase
        issued = j + 1;
        break;
      }
      issued = j + 1;
    }
    // after a failure the last tiles' copies may still be landing: they must land
    // before this CTA's shared memory is reused or released (a bounded wait each)
    if (lane == 0) {
      for (int j = issued > kS ? issued - kS : 0; j < issued; ++j) {
        const long long c0 = clock64();
        while (!mbar_try_wait(&kv_full[j % kS], (j / kS) & 1) &&
               clock64() - c0 < kWaitLimitCycles) {
        }
      }
    }
    __syncwarp();
  }
  // ------------------------------------------ E4M3 loader (TMA) and widening --
  // The loader brings tile j's E4M3 pages (K [16 keys][D bytes] per page, then V) into
  // stage j % kF8Stages once the converters are done with tile j - kF8Stages; the two
  // converter warps widen tile j into f16 ring stage j % 2 (the 128-byte swizzled
  // layout TMA writes for 16-bit tiles) once PV(j - 2) of every M tile is done, make
  // the writes visible to the tensor core's proxy and arrive on kv_full.
  if constexpr (kF8) {
    // widen this warp's half (part 0: the loader, 1: warp kWarpConv) of tile j
    auto widen = [&](int j, int part) -> bool {
      const int f = j % kF8Stages, st = j % kS;
      if (!warp_mbar_wait(&f8_full[f], (j / kF8Stages) & 1, abort_flag, a.status)) return false;
      if (j >= kS && !warp_mbar_wait(&kv_empty[st], ((j / kS) - 1) & 1, abort_flag, a.status))
        return false;
      // This thread's chunks: column c16 (16 features) of keys key0 + (64 / kC16) i
      // (the 64 threads of the two warps cover 64 / kC16 keys per step); within a
      // 128-byte row the swizzle term is key & 7, the same for every i.
      constexpr int kC16 = D / 16;           // 16-byte E4M3 chunks per key
      constexpr int kStep = 64 / kC16;       // keys per step
      const int t64 = part * 32 + lane;
      const int c16 = t64 % kC16, key0 = t64 / kC16;
      const int h = c16 >> 2, c8 = (c16 & 3) * 2;
      const int sw = key0 & 7;
      const int lo_off = (c8 ^ sw) << 4, hi_off = ((c8 + 1) ^ sw) << 4;
      const uint8_t* src = smem + L::kF8Ring + f * L::kF8Stage + key0 * D + c16 * 16;
      uint8_t* dk = smem + L::kK0 + st * L::kKVBytes + h * L::kKVHalf + key0 * 128;
      uint8_t* dv = smem + L::kV0 + st * L::kKVBytes + h * (kPage * 128) + key0 * 128;
#pragma unroll
      for (int i = 0; i < kKeysN / kStep; ++i) {
        uint4 lo, hi;
        e4m3x16_to_f16(*reinterpret_cast<const uint4*>(src + i * kStep * D), lo, hi);
        *reinterpret_cast<uint4*>(dk + i * kStep * 128 + lo_off) = lo;
        *reinterpret_cast<uint4*>(dk + i * kStep * 128 + hi_off) = hi;
      }
#pragma unroll
      for (int i = 0; i < kKeysN / kStep; ++i) {
        const int key = key0 + i * kStep;  // V rows: [page][half][16 keys][128 B]
        uint4 lo, hi;
        e4m3x16_to_f16(*reinterpret_cast<const uint4*>(src + L::kF8Tile + i * kStep * D), lo,
                       hi);
        uint8_t* row = dv + (key / kPage) * L::kVPage + (key % kPage - key0) * 128;
        *reinterpret_cast<uint4*>(row + lo_off) = lo;
        *reinterpret_cast<uint4*>(row + hi_off) = hi;
      }
      if (kCausal && j == ntiles - 1 && ragged_end) {
        // slots past the range in its last page: zero, not the cache's bytes (after this
        // thread's own writes above; the same thread wrote these rows)
#pragma unroll
        for (int i = 0; i < kKeysN / kStep; ++i) {
          const int key = key0 + i * kStep;
          if (geo.key0 + tile_of(j) * kKeysN + key >= geo.key_end) {
            uint8_t* row = dv + (key / kPage) * L::kVPage + (key % kPage - key0) * 128;
            *reinterpret_cast<uint4*>(row + lo_off) = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(row + hi_off) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&kv_full[st]);
      mbar_arrive(&f8_empty[f]);
      return true;
    };
    if (warp == kWarpLoad && ntiles > 0) {
      // step t: load tile t, then widen tile t - (kF8Stages - 1); the load of tile t
      // waits for the widening of tile t - kF8Stages, which this warp did a step
      // earlier and warp kWarpConv does on its own
      constexpr int kLag = kF8Stages - 1;
      constexpr int kIdTiles = 32 / kPagesPerTile;
      const int npages = (geo.key_end - geo.key0 + kPage - 1) / kPage;
      const int32_t* bt_pages = geo.bt + geo.key0 / kPage;
      auto load_ids = [&](int i_base) {
        const int i = i_base + lane / kPagesPerTile;
        const int page = tile_of(i) * kPagesPerTile + (lane & (kPagesPerTile - 1));
        return i < ntiles && page < npages ? __ldg(bt_pages + page) : -1;
      };
      int ids_cur = load_ids(0);
      int ids_nxt = ntiles > kIdTiles ? load_ids(kIdTiles) : -1;
      int issued = 0;
      bool ok = true;
      for (int t = 0; ok && t < ntiles + kLag; ++t) {
        if (t < ntiles) {
          const int f = t % kF8Stages;
          if (t >= kF8Stages &&
              !warp_mbar_wait(&f8_empty[f], ((t / kF8Stages) - 1) & 1, abort_flag, a.status))
            break;
          if (t > 0 && t % kIdTiles == 0) {
            ids_cur = ids_nxt;
            ids_nxt = t + kIdTiles < ntiles ? load_ids(t + kIdTiles) : -1;
          }
          if (lane == 0) mbar_arrive_expect_tx(&f8_full[f], L::kF8Stage);
          __syncwarp();
          // lanes [0, 4): K pages, [4, 8): V pages; one box of 16 keys x D bytes each
          const int q = lane & (kPagesPerTile - 1);
          const int blk =
              __shfl_sync(0xffffffffu, ids_cur, ((t % kIdTiles) * kPagesPerTile + q) & 31);
          const int tok = blk >= 0 ? blk * kPage : -kPage;  // -16: a box of zeros
          if (lane < 2 * kPagesPerTile) {
            const bool is_v = lane >= kPagesPerTile;
            tma_load_3d(smem + L::kF8Ring + f * L::kF8Stage + (is_v ? L::kF8Tile : 0) +
                            q * (kPage * D),
                        is_v ? &tm_v : &tm_k, &f8_full[f], 0, kvh, tok);
          }
          issued = t + 1;
        }
        if (t >= kLag) ok = widen(t - kLag, 0);
      }
      // after a failure the last tiles' copies may still be landing (a bounded wait each)
      if (lane == 0) {
        for (int j = issued > kF8Stages ? issued - kF8Stages : 0; j < issued; ++j) {
          const long long c0 = clock64();
          while (!mbar_try_wait(&f8_full[j % kF8Stages], (j / kF8Stages) & 1) &&
                 clock64() - c0 < kWaitLimitCycles) {
          }
        }
      }
      __syncwarp();
    }
    if (warp == kWarpConv && ntiles > 0) {
      for (int j = 0; j < ntiles; ++j)
        if (!widen(j, 1)) break;
    }
  }
  if (warp >= 8) __syncwarp();

  // --------------------------------------------------------------- softmax --
  const int wg = warp >> 2;            // softmax warpgroup = M tile (warps 0-7)
  const int row = threadIdx.x & 127;   // TMEM lane == row within the M tile
  const uint32_t t_lane = tmem + wg * 256 + (static_cast<uint32_t>((warp & 3) * 32) << 16);
  const uint32_t tO = t_lane + 2 * kKeysN;
  float m_run = -INFINITY;  // running max, log2 domain
  float l_run = 0.f;
  bool have = false;
  const bool softmax_warp = warp < 8 && (wg == 0 || has_m1);
  if (warp < 8) {
    // the first key past this thread's row: the range's end, or its causal limit
    int key_lim = geo.key_end;
    if (kCausal) {
      const int rho = geo.prow0 + wg * kRowsM + row;
      key_lim = min(key_lim, geo.causal_base + rho / a.group + 1);
    }

    // one tile of the online softmax: S(i) from TMEM -> P(i) back into TMEM (bf16)
    auto softmax_tile = [&](int i) -> bool {
      const int tile = tile_of(i);

      const bool ok =
          warp_mbar_wait(&s_full[wg * 2 + (i & 1)], (i >> 1) & 1, abort_flag, a.status);
      if (wg_bar_any(1 + wg, !ok)) return false;
      tc_fence_after();
      float sv[kKeysN];
      tmem_ld64_sync(t_lane + (i & 1) * kKeysN, sv);
      const int valid = key_lim - (geo.key0 + tile * kKeysN);
      if (valid < kKeysN) {  // the range's last tile, or past a causal limit
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
        // O must hold PV(i-1) before it is rescaled.  Stage (i-1) % kStages is freed
        // once every M tile's PV(i-1) is done; its phase is unambiguous: the stage's
        // previous tile (i-1-kStages) was freed before tile i-1 was loaded into it,
        // and its next tile's PV cannot complete before this thread writes P(i).
        warp_mbar_wait(&kv_empty[(i - 1) % kS], ((i - 1) / kS) & 1, abort_flag, a.status);
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
      // p = 2^(s * scale * log2(e) - m): one ex2 per score, the scaling and the row sum
      // as paired fp32 instructions (two scores each)
      uint32_t pw[kKeysN / 2];
      float2 sum2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      // a row whose keys so far are all masked keeps m_run = -inf: its p are 0
      const float neg_m = (kCausal && m_run == -INFINITY) ? 0.f : -m_run;
      const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
      const float2 nm2 = make_float2(neg_m, neg_m);
#pragma unroll
      for (int j = 0; j < kKeysN / 2; ++j) {
        const float2 x = fma_f32x2(make_float2(sv[2 * j], sv[2 * j + 1]), sc2, nm2);
        const float2 pp = make_float2(fast_exp2(x.x), fast_exp2(x.y));
        sum2[j & 1] = add_f32x2(sum2[j & 1], pp);
        pw[j] = kF8 ? pack_f16x2(pp.x, pp.y) : pack_bf16x2(pp.x, pp.y);
      }
      l_run += (sum2[0].x + sum2[1].x) + (sum2[0].y + sum2[1].y);
      tmem_st32_u(t_lane + (i & 1) * kKeysN, pw);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full[wg * 2 + (i & 1)]);
      return true;
    };

    bool failed = false;
    for (int i = 0; i < ntiles; ++i) {
      if (softmax_warp) {
        if (!softmax_tile(i)) {
          failed = true;
          break;
        }
      }
    }
    if (softmax_warp && !failed && ntiles > 0) {
      // o_last completes once, after every PV of the range
      const bool ok = warp_mbar_wait(&o_last[wg], 0, abort_flag, a.status);
      have = !wg_bar_any(1 + wg, !ok);
    }
    tc_fence_before();
  }

  // ----------------------------------------- this split's partial -> slot --
  // every MMA of the CTA is complete once both warpgroups saw their o_last
  // (or have nothing to do): Q and the ring become the staging buffer
  __syncthreads();
  __nv_bfloat16* stage = reinterpret_cast<__nv_bfloat16*>(smem);
  if (softmax_warp) {
    tc_fence_after();
    // a row that saw no key (l = 0) stages zeros; an E4M3 cache's V scale is applied
    // here, to the normalised rows
    float inv_l = (have && !(l_run <= 0.f)) ? 1.f / l_run : 0.f;  // NaN propagates
    if constexpr (kF8) inv_l *= a.v_scale;
    __nv_bfloat16* dst = stage + (wg * kRowsM + row) * L::kStageRow;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      float o[32];
      tmem_ld32_sync(tO + c * 32, o);
      if (inv_l == 0.f) {
#pragma unroll
        for (int j = 0; j < 32; ++j) o[j] = 0.f;
      }
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
  if (warp < 8)
    s_lse[wg * kRowsM + row] =
        (softmax_warp && have && !(l_run <= 0.f)) ? m_run + log2f(l_run) : -INFINITY;
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if constexpr (kCausal) return;  // the caller writes the staged rows
  // coalesced copy-out: a warp writes whole rows (D/8 lanes x 16 bytes each)
  {
    constexpr int kChunks = D / 8;
    const int gshift = __ffs(a.group) - 1;  // group is a power of two
    for (int it = threadIdx.x; it < kRowsCta * kChunks; it += kNThreads) {
      const int r = it / kChunks;
      const int c = it % kChunks;
      const int packed = geo.prow0 + r;
      if ((packed >> gshift) >= a.total_q) continue;
      const int t = a.tok0 + (packed >> gshift);
      const int64_t row = static_cast<int64_t>(t) * a.num_q_heads + kvh * a.group +
                          (packed & (a.group - 1));
      const int64_t rows_all =
          a.rows_all > 0 ? a.rows_all : static_cast<int64_t>(a.total_q) * a.num_q_heads;
      const int64_t slot = a.slot_base + split;
      const int64_t prow = slot * rows_all + row;
      *reinterpret_cast<uint4*>(a.part_o + prow * D + c * 8) =
          *reinterpret_cast<const uint4*>(stage + r * L::kStageRow + c * 8);
      if (c == 0) a.part_lse[slot * a.lse_stride + row] = s_lse[r];
    }
  }
}


}  // namespace prefix
}  // namespace csp
