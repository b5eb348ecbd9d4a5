// api.cu — the C ABI declared in include/csp.h: argument checks, the common-prefix
// planner, the launch plan (tiles, key splits, workspace partition), TMA tensor-map
// encoding and the launch sequence.  Everything here runs on the host.
#include <climits>
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "csp.h"
#include "kernels.cuh"
#include "merge.cuh"

namespace {

thread_local int g_last_cuda_error = 0;

int cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return CSP_ERR_CUDA;
}

constexpr int kPage = 16;
// Workspace header: [0] status word; [64] the 64-bit arrival count of the single-kernel
// decode schedule's grid barrier (each call adds its grid, the SM count, so the count
// stays a multiple of it between calls).
constexpr size_t kHeaderBytes = 256;
// Batches with a tcgen05 suffix (more than 16 rows per request and KV head) take the
// fused schedule unless the caller asks for another.
constexpr bool kFusedByDefault = false;
constexpr size_t kOffBarCount = 64;
// Shared memory the decode schedule's merge stages its bf16 rows in.
constexpr size_t kMergeSmemBytes = 192 * 1024;
// LSE box of a merge chunk: the chunk's rows, rounded out to 16-byte boundaries.
int merge_lse_box(int rows) { return (rows + 3 + 3) & ~3; }
// Most packed rows (query, head-in-group) per request and KV head that the decode
// schedule takes: one warp-level MMA tile.
constexpr int kDecodeRows = 16;
// CSP_MODE_AUTO takes cascade only when the standard path streams this many KV tokens
constexpr int64_t kAutoMinFlatTokens = 8192;
constexpr int kMaxSplits = 32;  // suffix splits; with the prefix's slots at most 32 partials per row

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }
int cdiv(int a, int b) { return (a + b - 1) / b; }

int device_sm_count(int* sms) {
  static std::atomic<int> cache[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev >= 0 && dev < 64) {
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) {
      *sms = v;
      return CSP_OK;
    }
  }
  int n = 0;
  e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  *sms = n;
  return CSP_OK;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// 3-D bf16 tensor map with a 128-byte swizzle: dims innermost first, strides of dims
// 1 and 2 in bytes, box in elements.
int make_map_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cuda_fail(cudaErrorNotSupported);
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {s1, s2};
  const cuuint32_t box[3] = {b0, b1, b2};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
  return CSP_OK;
}

// An E4M3 K or V cache [blocks][16][Hkv][D] (bytes) as {D, Hkv, tokens}, boxes {D, 1, 16}
// (one page of one KV head), no swizzle.
int make_map_bytes_3d(CUtensorMap* map, const void* base, int D, int Hkv, uint64_t ntok) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cuda_fail(cudaErrorNotSupported);
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hkv), ntok};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D),
                                 static_cast<cuuint64_t>(Hkv) * static_cast<cuuint64_t>(D)};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(D), 1, kPage};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
  return CSP_OK;
}

// A K or V cache [blocks][16][Hkv][D] seen as 4-D {64 features, tokens, D / 64
// feature halves, Hkv} (the halves and heads listed after the tokens), 128-byte
// swizzle, boxes {64, 16, D / 64, 1}: one page of one KV head lands in shared memory
// as [half][16 tokens][128 B], so 16 consecutive keys are consecutive swizzled rows.
int make_map_kv_pages(CUtensorMap* map, const void* base, int D, int Hkv, uint64_t ntok) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cuda_fail(cudaErrorNotSupported);
  const cuuint64_t dims[4] = {64, ntok, static_cast<cuuint64_t>(D / 64),
                              static_cast<cuuint64_t>(Hkv)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(Hkv) * D * 2, 128,
                                 static_cast<cuuint64_t>(D) * 2};
  const cuuint32_t box[4] = {64, kPage, static_cast<cuuint32_t>(D / 64), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
  return CSP_OK;
}

// Plain (unswizzled) tiled map of `rank` dims: the decode schedule's merge reads its
// workspace slots through these.
int make_map_plain(CUtensorMap* map, CUtensorMapDataType type, uint32_t rank, const void* base,
                   const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cuda_fail(cudaErrorNotSupported);
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, type, rank, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
  return CSP_OK;
}

bool supported_group(int g) { return g == 1 || g == 2 || g == 4 || g == 8 || g == 16; }

int check_shape(int num_reqs, int total_q, int max_q, int max_k, int Hq, int Hkv, int D, int bs) {
  if (num_reqs < 0 || total_q < 0 || max_q < 0 || max_k < 0 || Hq <= 0 || Hkv <= 0)
    return CSP_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return CSP_ERR_INVALID_ARG;
  if (!supported_group(Hq / Hkv)) return CSP_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return CSP_ERR_UNSUPPORTED;
  if (bs != kPage) return CSP_ERR_UNSUPPORTED;
  return CSP_OK;
}

// How one attention call is cut into CTAs and where its partials live.
struct LaunchPlan {
  int group = 1;
  // prefix phase (tcgen05): 256-row units x key ranges, one slot per range
  int p_pairs = 0, p_splits = 0, p_tiles_per_split = 0, p_slots = 0;
  // paged phase (suffix or standard path)
  bool decode = true;
  bool tc = false;      // many rows per (request, KV head): the tcgen05 kernel (paged_tc.cu)
  int s_row_tiles = 1, s_splits = 1, s_split_keys = 64;
  bool direct = false;  // paged kernel writes the final output itself
  int n_parts = 0;      // partial results per row group
  size_t off_counters = 0, off_part_o = 0, off_part_lse = 0, bytes = 0;
  // the fused schedule: prefix ranges and tcgen05 suffix units in one grid
  // (paged_tc.cu), merged by each row group's last contributor
  bool fused = false;
  // the two-kernel schedule with the warp-MMA suffix writing its partials and a merge
  // kernel after both phases (as after a tcgen05 suffix)
  bool split_merge = false;
  // the cost models' estimates (us): the single kernel at its best number of ranges,
  // the two-kernel schedule's split-merge at its best number of ranges
  double est_single_us = 0.0, est_split_us = 0.0;
  // single-kernel decode schedule (decode_cascade.cu)
  bool single = false;
  int d_splits = 0, d_prefix_ctas = 0, d_prefix_units = 0, d_grid = 0, d_merge_rows = 0;
  int64_t d_lse_stride = 0;
  size_t d_off_o = 0, d_off_lse = 0;
};

// sched_override: -1 (the cost model decides), CSP_SCHEDULE_TWO_KERNELS or
// CSP_SCHEDULE_SINGLE (taken where the single kernel can run); ranges_override > 0
// fixes the single kernel's number of prefix ranges.
void make_plan(int num_reqs, int total_q, int max_q, int max_k, int cpl, int Hq, int Hkv, int D,
               int sms, LaunchPlan* P, int sched_override = -1, int ranges_override = 0) {
  LaunchPlan p;
  p.group = Hq / Hkv;
  p.decode = static_cast<int64_t>(max_q) * p.group <= 16;
  // the fused schedule runs every suffix unit on the tcgen05 body
  p.tc = !p.decode || (cpl > 0 && sched_override == CSP_SCHEDULE_FUSED);
  const int max_len = std::max(0, max_k - cpl);
  if (cpl > 0) {
    const int rows = total_q * p.group;
    p.p_pairs = cdiv(rows, 256);
    const int key_tiles = cdiv(cpl, 64);
    const int base = p.p_pairs * Hkv;
    // Key ranges per (256-row block, KV head).  The suffix kernel runs on the SMs the
    // prefix leaves free, so the call takes about max(the prefix's waves x a CTA's
    // time, (prefix + suffix SM time) / SMs).  A prefix CTA costs its tiles plus ~3
    // tiles of fixed cost (set-up, the partial write-out) at ~1.22 us each; the suffix
    // streams half its longest range on average at ~32 GB/s per SM, plus ~5 us per CTA
    // of the tcgen05 variant.  More ranges also mean more slots for the suffix to merge.
    const double tile_us = 1.22;
    const double suf_bytes = static_cast<double>(num_reqs) * Hkv * (0.5 * max_len + 64.0) * 4.0 * D;
    const double suf_sm_us =
        suf_bytes / 32e3 + (p.tc ? 5.0 * num_reqs * Hkv * cdiv(max_q * p.group, 256) : 0.0);
    double best_cost = -1.0;
    for (int s = 1; s <= 16; s *= 2) {
      if (s > 1 && s > key_tiles) break;
      const int64_t ctas = static_cast<int64_t>(base) * s;
      const double cta_us = (cdiv(key_tiles, s) + 3) * tile_us;
      const double cost = std::max(cdiv64(ctas, sms) * cta_us, (ctas * cta_us + suf_sm_us) / sms);
      if (best_cost < 0.0 || cost < best_cost) {
        best_cost = cost;
        p.p_splits = s;
      }
    }
    p.p_tiles_per_split = cdiv(key_tiles, p.p_splits);
    p.p_slots = p.p_splits;
  }
  const int rows_per_cta = p.decode ? 16 : 256;
  p.s_row_tiles = std::max(1, cdiv(max_q * p.group, rows_per_cta));
  const int key_tiles = std::max(1, cdiv(max_len, 64));
  const int64_t units = static_cast<int64_t>(num_reqs) * p.s_row_tiles * Hkv;
  const int max_s = std::min(kMaxSplits, 32 - p.p_slots);
  int s = units > 0 ? static_cast<int>(std::min<int64_t>(cdiv64(2LL * sms, units), max_s)) : 1;
  // the warp-MMA kernel merges up to 8 splits of a row tile inside a thread-block cluster
  // (no counters, no global partials): take at most 8
  if (!p.tc) s = std::min(s, 8);
  if (p.tc) {
    // one CTA per SM: waves x (a split's tiles + ~5 tiles of fixed cost: the first
    // tile's latency, the output and the merge)
    int64_t best_cost = -1;
    for (int c = 1; c <= std::min(max_s, key_tiles); ++c) {
      const int64_t cost = cdiv64(units * c, sms) * (cdiv(key_tiles, c) + 5);
      if (best_cost < 0 || cost < best_cost) {
        best_cost = cost;
        s = c;
      }
    }
  }
  s = std::max(1, std::min(s, key_tiles));
  p.s_split_keys = cdiv(key_tiles, s) * 64;
  p.s_splits = std::max(1, cdiv(std::max(max_len, 1), p.s_split_keys));
  p.direct = (cpl == 0 && p.s_splits == 1);
  p.n_parts = p.direct ? 0 : p.p_slots + p.s_splits;
  const size_t rows_total = static_cast<size_t>(total_q) * Hq;
  p.off_counters = kHeaderBytes;
  p.off_part_o = p.off_counters + align256(static_cast<size_t>(total_q) * Hkv * 4);
  p.off_part_lse = p.off_part_o + align256(static_cast<size_t>(p.n_parts) * rows_total * D * 2);
  p.bytes = p.off_part_lse + align256(static_cast<size_t>(p.n_parts) * rows_total * 4);

  // Decode-like batches (a request's rows of one KV head fit one 16-row MMA tile):
  // one cooperative kernel.  d_base * s CTAs each run a prefix range and then stream
  // k suffix units; the other CTAs stream the rest of the suffix units from the
  // start.  s and k come from a cost model fitted to a sweep on one GB300 of N in
  // {16..256} x P in {1024..16384} (S = 128, Hq 32, Hkv 8, D 128) over 2-12 ranges
  // (99 points; rms error 2%, worst 6%), per CTA in us: a prefix range costs ~8.3 of
  // fixed work (its first tiles landing, writing its partial) plus its 64-key tiles,
  // each at its bytes' time at ~45 GB/s or ~0.87 per 256 rows (tensor core and
  // softmax), whichever is longer; a suffix unit takes its bytes' time at ~40 GB/s
  // (the copies and the computing warps pace it together), the first landing at ~5.9
  // (~1.8 after a range on a prefix CTA).  Both kinds of CTA should finish together.
  // The grid barrier and the merge after them cost ~0.9 plus ~0.08 per KB of slots a
  // CTA merges; on a tie the fewer prefix ranges win.  On that grid the pick was
  // within 2% of the best measured range count at every point.  The single kernel is
  // taken only if it is not expected to be slower than the two-kernel schedule (a
  // long prefix over many 256-row blocks leaves it too few SMs for one of the
  // phases).
  // The two-kernel schedule for decode-shaped rows: the prefix kernel on some SMs, the
  // warp-MMA suffix kernel writing its partials on the rest (neither waits for the
  // other), then the slot merge kernel.  Its number of prefix key ranges and its time
  // come from a cost model fitted to a sweep of N in {16..256} x P in {1024..16384}
  // (S = 128, Hq 32, Hkv 8, D 128, 1-12 ranges) and the long-prefix batch (N = 256,
  // P = 16384, S up to 1024, Hq 64) on one GB300: ~6 us of fixed cost; a prefix CTA
  // ~3 us plus its 64-key tiles at the longer of the copy time (~40 GB/s per SM) and
  // ~0.9 us per 256 rows; a suffix unit (request, KV head) ~1 us plus its bytes at
  // ~40 GB/s per SM, on the SMs the prefix leaves free and then on all; the merge
  // ~0.1 ns per row and slot.  On those 16 shapes its pick was the best measured range
  // count at 14 and within 5% at the other two.  Against an in-place merge (the suffix
  // waiting for the whole prefix grid) this schedule was 20-27% faster at N >= 128.
  int split_r = 1;
  if (cpl > 0 && !p.tc) {
    const int key_tiles = cdiv(cpl, 64);
    const int r_max = std::min(16, key_tiles);
    const int base = p.p_pairs * Hkv;
    const double rows_all = static_cast<double>(total_q) * Hq;
    const double t_tile =
        std::max(64.0 * 4.0 * D / 1024.0 / 40.0,
                 0.9 * std::min(256.0, static_cast<double>(total_q) * p.group) / 256.0);
    const double suf_sm_us = static_cast<double>(num_reqs) * Hkv *
                             (1.0 + (0.5 * max_len + 64.0) * 4.0 * D / 1024.0 / 40.0);
    double best = -1.0;
    for (int r = 1; r <= r_max; ++r) {
      const int64_t ctas = static_cast<int64_t>(base) * r;
      const double t_pre = 3.0 + cdiv(key_tiles, r) * t_tile;
      const double t = 6.0 +
                       std::max(cdiv64(ctas, sms) * t_pre, (ctas * t_pre + suf_sm_us) / sms) +
                       0.1e-3 * rows_all * (r + 1) * D / 128.0;
      if (best < 0.0 || t < best) {
        best = t;
        split_r = r;
      }
    }
    p.est_split_us = best;
  }
  const int d_base = p.p_pairs * Hkv;
  if (cpl > 0 && static_cast<int64_t>(max_q) * p.group <= kDecodeRows && d_base <= sms) {
    const int pre_tiles = cdiv(cpl, 64);
    const double kRate = 44.8e3, kUnitRate = 39.9e3;  // bytes per us per SM
    const double pair_rows = std::min(256.0, static_cast<double>(total_q) * p.group);
    const double tile_us = std::max(64.0 * 4.0 * D / kRate, 0.87 * pair_rows / 256.0);
    const double unit_us =
        (std::max(1, cdiv(max_len, 64)) * 64.0 * 4.0 * D + max_q * p.group * D * 2.0) /
        kUnitRate;
    const int64_t units = static_cast<int64_t>(num_reqs) * Hkv;
    const int s_max = std::max(1, std::min({pre_tiles, csp::kDecodeMaxParts - 1, sms / d_base}));
    // best number of prefix units for c ranges (and the model's time for it)
    auto best_k = [&](int c, double* t_out) {
      const int64_t pc = static_cast<int64_t>(d_base) * c;  // prefix CTAs
      const int64_t nc = sms - pc;                            // suffix-only CTAs
      const double pre_us = 8.3 + cdiv(pre_tiles, c) * tile_us;
      // the grid barrier and the merge: KB of slots per CTA
      const double merge_us =
          0.9 + 0.082e-3 * static_cast<double>(total_q) * Hq * (c + 1) * D * 2.0 / sms;
      const int64_t k_lo = nc > 0 ? 0 : cdiv64(units, pc);
      double best_t = -1.0;
      int kb = 0;
      for (int64_t kk = k_lo; kk <= cdiv64(units, pc); ++kk) {
        const int64_t rest = std::max<int64_t>(0, units - pc * kk);
        const int64_t per = nc > 0 ? cdiv64(rest, nc) : 0;
        // a prefix CTA's first suffix item lands ~1.8 after its range is written
        const double t =
            std::max(pre_us + (kk > 0 ? 1.8 : 0.0) + kk * unit_us, 5.9 + per * unit_us) +
            merge_us;
        if (best_t < 0.0 || t < best_t) {
          best_t = t;
          kb = static_cast<int>(kk);
        }
        if (per == 0) break;
      }
      *t_out = best_t;
      return kb;
    };
    int s = 1;
    double best = -1.0;
    for (int c = 1; c <= s_max; ++c) {
      double t;
      best_k(c, &t);
      if (best < 0.0 || t < best) {
        best = t;
        s = c;
      }
    }
    // the two-kernel schedule: its prefix kernel (p_splits ranges per block, in waves
    // over the SMs), while the SMs it leaves free start the suffix, which every SM
    // then streams (its own rates: a prefix tile at ~31 GB/s or ~1.22 us per 256
    // rows, a suffix unit at ~28.5 GB/s per SM)
    const double tile2_us = std::max(64.0 * 4.0 * D / 31e3, 1.22 * pair_rows / 256.0);
    const double unit2_us = unit_us * kUnitRate / 28.5e3;
    const double pre2_us = cdiv64(static_cast<int64_t>(d_base) * p.p_splits, sms) *
                           (3.5 + p.p_tiles_per_split * tile2_us + 3.4);
    const int64_t free_sms = std::max<int64_t>(0, sms - static_cast<int64_t>(d_base) * p.p_splits);
    const double two_us =
        pre2_us + 5.0 +
        std::max(0.0, static_cast<double>(units) * unit2_us - free_sms * pre2_us) / sms;
    p.est_single_us = best;
    // the single kernel when the model expects it to beat both two-kernel variants
    // (the one with an in-place merge, and, within the split-merge model's fitting
    // range of at least 64 query rows per KV head, the split-merge one)
    const bool split_fitted = static_cast<int64_t>(total_q) * p.group >= 64;
    p.single = sched_override == CSP_SCHEDULE_SINGLE ||
               (sched_override < 0 && best <= two_us &&
                (!split_fitted || best <= p.est_split_us));
    if (ranges_override > 0) s = std::min(ranges_override, s_max);
    double t_s;
    const int k = best_k(s, &t_s);
    p.d_splits = s;
    p.d_prefix_ctas = d_base * s;
    p.d_prefix_units = k;
    p.d_grid = sms;
    // slots: [0, s) the prefix ranges, s the suffix; an LSE slot is padded to a
    // multiple of four rows (the merge's tensor map wants 16-byte strides)
    p.d_lse_stride = (static_cast<int64_t>(rows_total) + 3) & ~int64_t{3};
    // rows per merge chunk: a CTA's share, within the box limit and the shared memory
    // the merge stages them in
    p.d_merge_rows = static_cast<int>(std::min<int64_t>(
        {cdiv64(static_cast<int64_t>(rows_total), sms), 252,
         static_cast<int64_t>(kMergeSmemBytes / (static_cast<size_t>(s + 1) * D * 2))}));
    p.d_merge_rows = std::max(p.d_merge_rows, 1);
    p.d_off_o = kHeaderBytes;
    p.d_off_lse = p.d_off_o + align256(static_cast<size_t>(s + 1) * rows_total * D * 2);
    // the workspace fits this schedule at any number of ranges (the most slots)
    const size_t lse_max = static_cast<size_t>(s_max + 1) * p.d_lse_stride * 4;
    p.bytes = std::max(p.bytes, kHeaderBytes +
                                    align256(static_cast<size_t>(s_max + 1) * rows_total * D * 2) +
                                    align256(lse_max));
  }
  // The two-kernel schedule for decode-shaped rows: the prefix kernel on some SMs, the
  // warp-MMA suffix kernel writing its partials on the rest (neither waits for the
  // other), then the slot merge kernel.  The number of prefix key ranges comes from a
  // cost model fitted to a sweep of N in {16..256} x P in {1024..16384} (S = 128, Hq
  // 32, Hkv 8, D 128, 1-12 ranges) on one GB300: a prefix CTA costs ~4 us plus its
  // 64-key tiles at the longer of the copy time (~40 GB/s per SM) and ~1 us per 256
  // rows; the suffix streams at ~20 GB/s per SM on the SMs the prefix leaves free and
  // then on all; the merge costs ~0.05 ns per row and slot.  On that grid its pick was
  // the best measured range count at 13 of 15 points and within 5% at the others.
  // Against an in-place merge (the suffix waiting for the whole prefix grid) this
  // schedule was 20-27% faster at N >= 128.  The workspace fits up to 16 ranges.
  if (cpl > 0 && !p.tc) {
    const int key_tiles = cdiv(cpl, 64);
    const int r_max = std::min(16, key_tiles);
    // the workspace fits this schedule at any number of ranges up to 16 (a caller's
    // override), whichever schedule the cost model picks
    const size_t rows_total = static_cast<size_t>(total_q) * Hq;
    const size_t fit = static_cast<size_t>(r_max + p.s_splits);
    const size_t off_o = p.off_counters + align256(static_cast<size_t>(total_q) * Hkv * 4);
    const size_t off_lse = off_o + align256(fit * rows_total * D * 2);
    p.bytes = std::max(p.bytes, off_lse + align256(fit * rows_total * 4));
    if (!p.single && sched_override != CSP_SCHEDULE_FUSED) {
      p.split_merge = true;
      p.p_splits = split_r;
      if (ranges_override > 0) p.p_splits = std::min(ranges_override, r_max);
      p.p_tiles_per_split = cdiv(key_tiles, p.p_splits);
      p.p_slots = p.p_splits;
      p.n_parts = p.p_slots + p.s_splits;
      p.off_part_o = off_o;
      p.off_part_lse = off_lse;
    }
  }
  p.fused = cpl > 0 && !p.single &&
            (sched_override == CSP_SCHEDULE_FUSED || (sched_override < 0 && p.tc && kFusedByDefault));
  *P = p;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// ------------------------------------------------------------------ multi-level --
// A multi-level cascade (§七: FlashInfer runs any number of levels): segments of
// consecutive requests that share keys [k_lo, k_hi), each computed by the prefix body
// over its requests' query rows into the slots of its level, then every request's
// suffix from its own start, then the LSE merge of every slot.
constexpr int kMaxLevels = 8;
constexpr int kSegInts = 7;  // level, r_lo, r_hi, k_lo, k_hi, tok_lo, tok_hi

struct LevelPlan {
  int n_levels = 0;
  int level_splits[kMaxLevels] = {};
  int level_base[kMaxLevels] = {};
  int n_prefix = 0;
  std::vector<int> seg_splits;  // key ranges of each segment
  LaunchPlan suf;               // the suffix (paged) part
  int n_parts = 0;
  size_t off_counters = 0, off_part_o = 0, off_part_lse = 0, bytes = 0;
};

// Host checks of a segment list: fields in range, and two segments that hold a request
// in common of different levels, the shallower one holding all of the deeper one's
// requests and ending where (or before) its keys start; so no key of a request is
// counted twice.
int check_segments(int num_reqs, int total_q, int max_k, const int32_t* segs, int n_seg) {
  if (n_seg < 0 || (n_seg > 0 && !segs)) return CSP_ERR_INVALID_ARG;
  for (int i = 0; i < n_seg; ++i) {
    const int32_t* s = segs + static_cast<int64_t>(i) * kSegInts;
    if (s[0] < 0 || s[0] >= kMaxLevels || s[1] < 0 || s[1] >= s[2] || s[2] > num_reqs ||
        s[3] < 0 || s[3] % kPage != 0 || s[4] % kPage != 0 || s[4] <= s[3] || s[4] > max_k ||
        s[5] < 0 || s[5] > s[6] || s[6] > total_q)
      return CSP_ERR_INVALID_ARG;
  }
  for (int i = 0; i < n_seg; ++i) {
    const int32_t* a = segs + static_cast<int64_t>(i) * kSegInts;
    for (int j = i + 1; j < n_seg; ++j) {
      const int32_t* b = segs + static_cast<int64_t>(j) * kSegInts;
      if (a[2] <= b[1] || b[2] <= a[1]) continue;
      const int32_t* up = a[0] < b[0] ? a : b;
      const int32_t* dn = a[0] < b[0] ? b : a;
      if (a[0] == b[0] || dn[1] < up[1] || dn[2] > up[2] || dn[3] < up[4])
        return CSP_ERR_INVALID_ARG;
    }
  }
  return CSP_OK;
}

int make_level_plan(int num_reqs, int total_q, int max_q, int max_k, const int32_t* segs,
                    int n_seg, int max_suffix_len, int Hq, int Hkv, int D, int sms,
                    LevelPlan* out) {
  LevelPlan L;
  int st = check_segments(num_reqs, total_q, max_k, segs, n_seg);
  if (st != CSP_OK) return st;
  if (max_suffix_len < 0 || max_suffix_len > max_k) return CSP_ERR_INVALID_ARG;
  // the suffix: as the two-kernel schedule's suffix kernel for suffixes of at most
  // max_suffix_len keys (its split count is settled below, once the prefix slots are)
  make_plan(num_reqs, total_q, max_q, max_k, max_k - max_suffix_len, Hq, Hkv, D, sms, &L.suf,
            CSP_SCHEDULE_TWO_KERNELS);
  // Key ranges per segment.  All segments run in one grid (one CTA per SM), next to the
  // suffix kernel on the SMs they leave free, so the call takes about max(the longest
  // CTA, (prefix + suffix SM time) / SMs); a CTA costs its tiles plus ~3 tiles of fixed
  // cost at ~1.22 us each (the prefix kernel's cost model), the suffix its bytes at
  // ~32 GB/s per SM.  Every segment aims at the same number of tiles per range (at
  // most 8 ranges); the levels' largest range counts add up to at most 24 slots; on a
  // tie the fewer ranges win.
  const int group = Hq / Hkv;
  const double tile_us = 1.22;
  const double suf_sm_us =
      static_cast<double>(num_reqs) * Hkv * (0.5 * max_suffix_len + 64.0) * 4.0 * D / 32e3;
  L.seg_splits.assign(n_seg, 1);
  double best = -1.0;
  for (int tp = 1 << 20; tp >= 2; tp = tp > 256 ? 256 : tp / 2) {
    std::vector<int> sp(n_seg, 1);
    int lvl[kMaxLevels] = {};
    double work = suf_sm_us, longest = 0.0;
    for (int i = 0; i < n_seg; ++i) {
      const int32_t* s = segs + static_cast<int64_t>(i) * kSegInts;
      const int tiles = cdiv(s[4] - s[3], 64);
      sp[i] = std::max(1, std::min(8, cdiv(tiles, tp)));
      lvl[s[0]] = std::max(lvl[s[0]], sp[i]);
      const int ctas = Hkv * cdiv((s[6] - s[5]) * group, 256) * sp[i];
      const double cta_us = (cdiv(tiles, sp[i]) + 3) * tile_us;
      work += ctas * cta_us;
      if (ctas > 0) longest = std::max(longest, cta_us);
    }
    int slots = 0;
    for (int d = 0; d < kMaxLevels; ++d) slots += lvl[d];
    if (slots > 24) continue;
    const double cost = std::max(longest, work / sms);
    if (best < 0.0 || cost < best) {
      best = cost;
      L.seg_splits = sp;
    }
  }
  for (int i = 0; i < n_seg; ++i) {
    const int32_t* s = segs + static_cast<int64_t>(i) * kSegInts;
    L.level_splits[s[0]] = std::max(L.level_splits[s[0]], L.seg_splits[i]);
    L.n_levels = std::max(L.n_levels, s[0] + 1);
  }
  for (int d = 0; d < L.n_levels; ++d) {
    L.level_base[d] = L.n_prefix;
    L.n_prefix += L.level_splits[d];
  }
  if (L.n_prefix > 24) return CSP_ERR_UNSUPPORTED;
  // at most 32 partials per row in all
  const int max_len = std::max(1, max_suffix_len);
  int split_keys = L.suf.s_split_keys;
  if (cdiv(max_len, split_keys) > 32 - L.n_prefix)
    split_keys = cdiv(cdiv(max_len, 32 - L.n_prefix), 64) * 64;
  L.suf.s_split_keys = split_keys;
  L.suf.s_splits = std::max(1, cdiv(max_len, split_keys));
  L.n_parts = L.n_prefix + L.suf.s_splits;
  const size_t rows = static_cast<size_t>(total_q) * Hq;
  L.off_counters = kHeaderBytes;
  L.off_part_o = L.off_counters + align256(static_cast<size_t>(total_q) * Hkv * 4);
  L.off_part_lse = L.off_part_o + align256(static_cast<size_t>(L.n_parts) * rows * D * 2);
  L.bytes = L.off_part_lse + align256(static_cast<size_t>(L.n_parts) * rows * 4);
  *out = L;
  return CSP_OK;
}

// The planner's walk (the same steps as oracle.planner.plan_levels, in C++).
struct LevelWalk {
  const int32_t* bt;
  int64_t stride;
  const int32_t* seq_lens;
  const int32_t* computed;
  const int64_t* used;
  const int32_t* tok;  // query token of request r: tok[r] .. tok[r + 1]
  int bs, max_levels, max_segments;
  int32_t* segs;
  int n = 0;
  int32_t* start;
  bool overflow = false;

  int64_t shared_run(int r_lo, int r_hi, int64_t col) const {
    int64_t k = col;
    for (;; ++k) {
      for (int r = r_lo; r < r_hi; ++r)
        if (k >= used[r]) return k - col;
      const int32_t first = bt[static_cast<int64_t>(r_lo) * stride + k];
      for (int r = r_lo + 1; r < r_hi; ++r)
        if (bt[static_cast<int64_t>(r) * stride + k] != first) return k - col;
    }
  }

  void walk(int r_lo, int r_hi, int64_t k_lo, int level) {
    if (level >= max_levels || overflow) return;
    int64_t k_next = k_lo;
    if (r_hi - r_lo >= 2) {
      const int64_t nb = shared_run(r_lo, r_hi, k_lo / bs);
      int64_t k_hi = (k_lo / bs + nb) * bs;
      int32_t min_c = INT32_MAX;
      for (int r = r_lo; r < r_hi; ++r) min_c = std::min(min_c, computed[r]);
      k_hi = std::min<int64_t>(k_hi, min_c);
      k_hi = (k_hi / bs) * bs;
      if (k_hi > k_lo) {
        if (n >= max_segments) {
          overflow = true;
          return;
        }
        int32_t* s = segs + static_cast<int64_t>(n) * kSegInts;
        s[0] = level;
        s[1] = r_lo;
        s[2] = r_hi;
        s[3] = static_cast<int32_t>(k_lo);
        s[4] = static_cast<int32_t>(k_hi);
        s[5] = tok[r_lo];
        s[6] = tok[r_hi];
        ++n;
        for (int r = r_lo; r < r_hi; ++r) start[r] = static_cast<int32_t>(k_hi);
        k_next = k_hi;
      }
    }
    // the runs of consecutive requests that share the block at k_next
    const int64_t col = k_next / bs;
    for (int r = r_lo; r < r_hi;) {
      int e = r + 1;
      if (col < used[r]) {
        while (e < r_hi && col < used[e] &&
               bt[static_cast<int64_t>(e) * stride + col] ==
                   bt[static_cast<int64_t>(r) * stride + col])
          ++e;
      }
      if (e - r >= 2 && !(r == r_lo && e == r_hi && k_next == k_lo)) walk(r, e, k_next, level + 1);
      r = e;
    }
  }
};


// Shared body of cascade_attn (cpl > 0) and paged_attn (cpl == 0).
int attention_call(const void* q, const void* k_cache, const void* v_cache, int32_t num_blocks,
                   const int32_t* block_table, int64_t bt_row_stride,
                   const int32_t* cu_seqlens_q, const int32_t* seqused_k, int32_t num_reqs,
                   int32_t total_q, int32_t max_seqlen_q, int32_t max_seqlen_k, int32_t cpl,
                   int32_t block_size, int32_t Hq, int32_t Hkv, int32_t D, float scale,
                   void* out, float* lse, void* workspace, size_t workspace_bytes,
                   void* stream_ptr, void* const* events = nullptr, int sched_override = -1,
                   int ranges_override = 0, const int32_t* cpl_dev = nullptr, bool kv_fp8 = false,
                   float k_scale = 1.f, float v_scale = 1.f) {
  int st = check_shape(num_reqs, total_q, max_seqlen_q, max_seqlen_k, Hq, Hkv, D, block_size);
  if (st != CSP_OK) return st;
  if (cpl < 0 || cpl % block_size != 0 || cpl > max_seqlen_k) return CSP_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return CSP_ERR_INVALID_ARG;
  if (num_blocks <= 0 || static_cast<int64_t>(num_blocks) * block_size > INT32_MAX)
    return CSP_ERR_INVALID_ARG;
  if (total_q == 0 || num_reqs == 0) return CSP_OK;
  if (!q || !k_cache || !v_cache || !block_table || !cu_seqlens_q || !seqused_k || !out)
    return CSP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return CSP_ERR_INVALID_ARG;
  if (bt_row_stride < cdiv(max_seqlen_k, block_size)) return CSP_ERR_INVALID_ARG;
  if (kv_fp8) {
    // an E4M3 cache runs on the two-kernel schedule (its kernels widen the tiles)
    if (!(k_scale > 0.f) || !std::isfinite(k_scale) || !(v_scale > 0.f) ||
        !std::isfinite(v_scale))
      return CSP_ERR_INVALID_ARG;
    if (cpl_dev != nullptr || (sched_override >= 0 && sched_override != CSP_SCHEDULE_TWO_KERNELS))
      return CSP_ERR_UNSUPPORTED;
    sched_override = CSP_SCHEDULE_TWO_KERNELS;
  }
  int sms = 0;
  if ((st = device_sm_count(&sms)) != CSP_OK) return st;
  LaunchPlan P;
  make_plan(num_reqs, total_q, max_seqlen_q, max_seqlen_k, cpl, Hq, Hkv, D, sms, &P,
            sched_override, ranges_override);
  // an E4M3 cache: the f16 copy of the queries after the plan's partition
  const size_t q16_off = align256(P.bytes);
  const size_t need =
      kv_fp8 ? q16_off + align256(static_cast<size_t>(total_q) * Hq * D * 2) : P.bytes;
  if (sched_override == CSP_SCHEDULE_SINGLE && !P.single) return CSP_ERR_UNSUPPORTED;
  // a prefix length in device memory: only the single-kernel schedule reads it there
  if (cpl_dev != nullptr && (!P.single || cpl == 0)) return CSP_ERR_UNSUPPORTED;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255) != 0 ||
      workspace_bytes < need)
    return CSP_ERR_WORKSPACE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* status = reinterpret_cast<int*>(ws);
  const void* q_in = q;  // the queries the kernels read
  int* counters = reinterpret_cast<int*>(ws + P.off_counters);
  __nv_bfloat16* part_o = reinterpret_cast<__nv_bfloat16*>(ws + P.off_part_o);
  float* part_lse = reinterpret_cast<float*>(ws + P.off_part_lse);
  const float scale_log2 = scale * 1.4426950408889634f * (kv_fp8 ? k_scale : 1.f);
  cudaError_t e;
  if (kv_fp8) {
    q_in = ws + q16_off;
    if ((e = csp::launch_bf16_to_f16(q, ws + q16_off, static_cast<int64_t>(total_q) * Hq * D,
                                     stream)) != cudaSuccess)
      return cuda_fail(e);
  }
  // the K/V maps of the tcgen05 kernels: 16-bit pages, or E4M3 pages
  auto kv_maps = [&](CUtensorMap* tk, CUtensorMap* tv) -> int {
    const uint64_t ntok = static_cast<uint64_t>(num_blocks) * block_size;
    const uint64_t row_b = static_cast<uint64_t>(D) * 2;
    int r;
    if (kv_fp8) {
      if ((r = make_map_bytes_3d(tk, k_cache, D, Hkv, ntok)) != CSP_OK) return r;
      return make_map_bytes_3d(tv, v_cache, D, Hkv, ntok);
    }
    if ((r = make_map_3d(tk, k_cache, D, Hkv, ntok, row_b, row_b * Hkv, 64, 1, kPage)) != CSP_OK)
      return r;
    return make_map_kv_pages(tv, v_cache, D, Hkv, ntok);
  };
  auto mark = [&](int i) -> cudaError_t {
    return events ? cudaEventRecord(static_cast<cudaEvent_t>(events[i]), stream) : cudaSuccess;
  };
  if (P.single) {
    CUtensorMap tm_q, tm_k, tm_v, tm_kp;
    const uint64_t row_b = static_cast<uint64_t>(D) * 2;
    const uint64_t ntok = static_cast<uint64_t>(num_blocks) * block_size;
    if ((st = make_map_3d(&tm_q, q, D, Hq, total_q, row_b, row_b * Hq, 64, P.group,
                          128 / P.group)) != CSP_OK ||
        (st = make_map_kv_pages(&tm_k, k_cache, D, Hkv, ntok)) != CSP_OK ||
        (st = make_map_kv_pages(&tm_v, v_cache, D, Hkv, ntok)) != CSP_OK ||
        (st = make_map_3d(&tm_kp, k_cache, D, Hkv, ntok, row_b, row_b * Hkv, 64, 1, kPage)) !=
            CSP_OK)
      return st;
    csp::DecodeArgs da;
    csp::PrefixArgs& pa = da.pre;
    pa.k = static_cast<const __nv_bfloat16*>(k_cache);
    pa.v = static_cast<const __nv_bfloat16*>(v_cache);
    pa.block_table = block_table;
    pa.total_q = total_q;
    pa.num_q_heads = Hq;
    pa.num_kv_heads = Hkv;
    pa.group = P.group;
    pa.cpl = cpl;
    pa.pairs = P.p_pairs;
    pa.n_splits = P.d_splits;
    pa.tiles_per_split = 0;  // ranges come from key_tiles and n_splits
    pa.scale_log2 = scale_log2;
    pa.part_o = reinterpret_cast<__nv_bfloat16*>(ws + P.d_off_o);
    pa.part_lse = reinterpret_cast<float*>(ws + P.d_off_lse);
    pa.lse_stride = P.d_lse_stride;
    pa.status = status;
    // the merge's views of the slots: bf16 rows [slot][row][D] and LSEs [slot][row]
    CUtensorMap tm_po, tm_pl;
    {
      const uint64_t n_slots = static_cast<uint64_t>(P.d_splits) + 1;
      const uint64_t rows = static_cast<uint64_t>(total_q) * Hq;
      const cuuint64_t od[3] = {static_cast<cuuint64_t>(D), rows, n_slots};
      const cuuint64_t os[2] = {row_b, rows * row_b};
      const cuuint32_t ob[3] = {static_cast<cuuint32_t>(D), static_cast<cuuint32_t>(P.d_merge_rows),
                                static_cast<cuuint32_t>(n_slots)};
      const cuuint64_t ld[2] = {static_cast<cuuint64_t>(P.d_lse_stride), n_slots};
      const cuuint64_t ls[1] = {static_cast<cuuint64_t>(P.d_lse_stride) * 4};
      const cuuint32_t lb[2] = {static_cast<cuuint32_t>(merge_lse_box(P.d_merge_rows)),
                                static_cast<cuuint32_t>(n_slots)};
      if ((st = make_map_plain(&tm_po, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, pa.part_o, od, os,
                               ob)) != CSP_OK ||
          (st = make_map_plain(&tm_pl, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, pa.part_lse, ld, ls,
                               lb)) != CSP_OK)
        return st;
    }
    da.q = static_cast<const __nv_bfloat16*>(q);
    da.k = static_cast<const __nv_bfloat16*>(k_cache);
    da.v = static_cast<const __nv_bfloat16*>(v_cache);
    da.block_table = block_table;
    da.bt_stride = bt_row_stride;
    da.cu_seqlens_q = cu_seqlens_q;
    da.seq_lens = seqused_k;
    da.num_reqs = num_reqs;
    da.prefix_ctas = P.d_prefix_ctas;
    da.prefix_units = P.d_prefix_units;
    da.merge_rows = P.d_merge_rows;
    // every request's suffix within one item (two 64-key tiles): two groups of four
    // warps take alternate units
    da.unit_groups = max_seqlen_k - cpl <= 2 * 64 ? 2 : 1;
    da.key_tiles = cdiv(cpl, 64);
    da.bar_count = reinterpret_cast<unsigned long long*>(ws + kOffBarCount);
    da.out = static_cast<__nv_bfloat16*>(out);
    da.lse = lse;
    da.cpl_dev = cpl_dev;
    da.max_seqlen_k = max_seqlen_k;
    // phase events: [0] before the kernel, [1..3] after it
    if ((e = mark(0)) != cudaSuccess) return cuda_fail(e);
    if ((e = csp::launch_decode(D, tm_q, tm_k, tm_v, tm_kp, tm_po, tm_pl, da, P.d_grid,
                                stream)) !=
        cudaSuccess)
      return cuda_fail(e);
    for (int i = 1; i < 4; ++i)
      if ((e = mark(i)) != cudaSuccess) return cuda_fail(e);
    return CSP_OK;
  }
  if ((e = mark(0)) != cudaSuccess) return cuda_fail(e);
  // After a prefix phase the tcgen05 suffix kernel writes its partials and a third
  // kernel merges every row (the two phases never wait for each other); otherwise the
  // suffix kernel merges, and several suffix splits count themselves in row-group
  // counters that start at zero in every call, whatever the workspace held.
  // The fused schedule counts prefix ranges and suffix splits in the same counters.
  const bool merge_after = (P.tc || P.split_merge) && cpl > 0 && !P.fused;
  // the warp-MMA kernel with 2..8 key splits merges them inside a thread-block cluster
  // (distributed shared memory): no counters
  const bool cluster =
      !P.tc && !P.fused && !P.split_merge && P.s_splits >= 2 && P.s_splits <= 8;
  if (P.n_parts > 0 && (P.s_splits > 1 || P.fused) && !merge_after && !cluster &&
      (e = cudaMemsetAsync(counters, 0, static_cast<size_t>(total_q) * Hkv * sizeof(int32_t),
                           stream)) != cudaSuccess)
    return cuda_fail(e);

  CUtensorMap tm_q, tm_k, tm_v;
  csp::PrefixArgs pa;
  if (cpl > 0) {
    const uint64_t row_b = static_cast<uint64_t>(D) * 2;
    if ((st = make_map_3d(&tm_q, q_in, D, Hq, total_q, row_b, row_b * Hq, 64, P.group,
                          128 / P.group)) != CSP_OK)
      return st;
    if ((st = kv_maps(&tm_k, &tm_v)) != CSP_OK) return st;
    pa.k = static_cast<const __nv_bfloat16*>(k_cache);
    pa.v = static_cast<const __nv_bfloat16*>(v_cache);
    pa.block_table = block_table;
    pa.total_q = total_q;
    pa.num_q_heads = Hq;
    pa.num_kv_heads = Hkv;
    pa.group = P.group;
    pa.cpl = cpl;
    pa.pairs = P.p_pairs;
    pa.n_splits = P.p_splits;
    pa.tiles_per_split = P.p_tiles_per_split;
    pa.scale_log2 = scale_log2;
    pa.part_o = part_o;
    pa.part_lse = part_lse;
    pa.lse_stride = static_cast<int64_t>(total_q) * Hq;
    pa.status = status;
    pa.v_scale = kv_fp8 ? v_scale : 1.f;
    if (!P.fused &&
        (e = kv_fp8 ? csp::launch_prefix_f8(D, tm_q, tm_k, tm_v, pa, stream)
                    : csp::launch_prefix(D, tm_q, tm_k, tm_v, pa, stream)) != cudaSuccess)
      return cuda_fail(e);
  }
  if ((e = mark(1)) != cudaSuccess) return cuda_fail(e);

  csp::PagedArgs ga;
  ga.q = static_cast<const __nv_bfloat16*>(q_in);
  ga.k = static_cast<const __nv_bfloat16*>(k_cache);
  ga.v = static_cast<const __nv_bfloat16*>(v_cache);
  ga.v_scale = kv_fp8 ? v_scale : 1.f;
  ga.block_table = block_table;
  ga.bt_stride = bt_row_stride;
  ga.cu_seqlens_q = cu_seqlens_q;
  ga.seq_lens = seqused_k;
  ga.num_reqs = num_reqs;
  ga.total_q = total_q;
  ga.num_q_heads = Hq;
  ga.num_kv_heads = Hkv;
  ga.group = P.group;
  ga.key_start = cpl;
  ga.split_keys = P.s_split_keys;
  ga.n_splits = P.s_splits;
  ga.row_tiles = P.s_row_tiles;
  ga.scale_log2 = scale_log2;
  ga.part_o = P.direct ? nullptr : part_o;
  ga.part_lse = P.direct ? nullptr : part_lse;
  ga.n_prefix = P.p_slots;
  ga.counters = counters;
  ga.out = static_cast<__nv_bfloat16*>(out);
  ga.lse = lse;
  ga.status = status;
  ga.cluster_splits = cluster;
  ga.partials_only = merge_after;
  if (merge_after || cluster) ga.counters = nullptr;
  // concurrent with the prefix kernel (programmatic dependent launch) unless phase
  // events sit between the two
  const bool overlap = cpl > 0 && events == nullptr;
  if (P.fused) {
    ga.prefix_contributors = P.p_splits;
    e = csp::launch_cascade_fused(D, tm_q, tm_k, tm_v, pa, ga, stream);
  } else if (P.tc) {
    CUtensorMap tm_q, tm_k, tm_v;
    const uint64_t row_b = static_cast<uint64_t>(D) * 2;
    if ((st = make_map_3d(&tm_q, q_in, D, Hq, total_q, row_b, row_b * Hq, 64, P.group,
                          128 / P.group)) != CSP_OK ||
        (st = kv_maps(&tm_k, &tm_v)) != CSP_OK)
      return st;
    e = kv_fp8 ? csp::launch_paged_tc_f8(D, tm_q, tm_k, tm_v, ga, overlap, stream)
               : csp::launch_paged_tc(D, tm_q, tm_k, tm_v, ga, overlap, stream);
  } else {
    e = kv_fp8 ? csp::launch_paged_f8(D, ga, overlap, stream)
               : csp::launch_paged(D, ga, overlap, stream);
  }
  if (e != cudaSuccess) return cuda_fail(e);
  if ((e = mark(2)) != cudaSuccess) return cuda_fail(e);
  // in stream order (no programmatic launch): both phases' slots are complete
  if (merge_after &&
      (e = csp::launch_merge_slots(D, part_o, part_lse, P.n_parts,
                                   static_cast<int64_t>(total_q) * Hq,
                                   static_cast<__nv_bfloat16*>(out), lse, stream)) != cudaSuccess)
    return cuda_fail(e);
  if ((e = mark(3)) != cudaSuccess) return cuda_fail(e);
  return CSP_OK;
}

}  // namespace

extern "C" {

int cascade_plan(const int32_t* block_table, int64_t bt_row_stride, int32_t num_reqs,
                 const int32_t* seq_lens, const int32_t* num_computed_tokens,
                 int32_t block_size, int32_t num_q_heads, int32_t num_kv_heads,
                 int32_t head_dim, int32_t num_sms, int32_t mode,
                 int32_t* common_prefix_len_out, int32_t* use_cascade_out) {
  if (!common_prefix_len_out || !use_cascade_out || num_reqs < 0 || block_size <= 0)
    return CSP_ERR_INVALID_ARG;
  if (mode < CSP_MODE_AUTO || mode > CSP_MODE_PAGE_THRESHOLDS) return CSP_ERR_INVALID_ARG;
  *common_prefix_len_out = 0;
  *use_cascade_out = 0;
  if (num_reqs == 0) return CSP_OK;
  if (!block_table || !seq_lens || !num_computed_tokens) return CSP_ERR_INVALID_ARG;
  // §八 Step 1: rows take part with their first cdiv(seq_len, bs) entries only
  int64_t shortest = INT64_MAX;
  int32_t min_computed = INT32_MAX;
  for (int r = 0; r < num_reqs; ++r) {
    if (seq_lens[r] < 0 || num_computed_tokens[r] < 0 || num_computed_tokens[r] > seq_lens[r])
      return CSP_ERR_INVALID_ARG;
    const int64_t used = cdiv64(seq_lens[r], block_size);
    if (used > bt_row_stride) return CSP_ERR_INVALID_ARG;
    shortest = std::min(shortest, used);
    min_computed = std::min(min_computed, num_computed_tokens[r]);
  }
  // the longest run shared by every row = the shortest of each row's run in common with
  // row 0, each bounded by what is left; rows are scanned in memory order
  int64_t ncpb = shortest;
  for (int r = 1; r < num_reqs && ncpb > 0; ++r) {
    const int32_t* row = block_table + static_cast<int64_t>(r) * bt_row_stride;
    // the common case: the whole run so far is shared (one memcmp); otherwise find the
    // first difference, 64-byte blocks first
    if (std::memcmp(row, block_table, static_cast<size_t>(ncpb) * sizeof(int32_t)) == 0)
      continue;
    int64_t k = 0;
    while (k + 16 <= ncpb && std::memcmp(row + k, block_table + k, 16 * sizeof(int32_t)) == 0)
      k += 16;
    while (k < ncpb && row[k] == block_table[k]) ++k;
    ncpb = k;
  }
  // §八 Step 2: blocks to tokens, cap to min(num_computed_tokens), floor to block_size
  int64_t cpl = ncpb * block_size;
  cpl = std::min<int64_t>(cpl, min_computed);
  cpl = (cpl / block_size) * block_size;
  *common_prefix_len_out = static_cast<int32_t>(cpl);

  // §三: never for a prefix under 256 tokens or a batch under 8 requests
  const bool thresholds = cpl >= 256 && num_reqs >= 8;
  int use = 0;
  switch (mode) {
    case CSP_MODE_FORCE_CASCADE:
      use = cpl > 0;
      break;
    case CSP_MODE_FORCE_FLAT:
      use = 0;
      break;
    case CSP_MODE_PAGE_THRESHOLDS:
      use = thresholds;
      break;
    default: {
      // GB300 rule, fitted to a cascade-vs-flat sweep of N in {4..256} x P in
      // {128..16384} (S = 128, Hkv 8, D 128) on one GB300: cascade when the standard
      // path would stream at least 8192 KV tokens (below that both calls are latency-
      // bound and the flat one, a single launch, is the faster) and cascade cuts those
      // tokens by at least 1.8x (the prefix read once instead of N times).  On that
      // grid it picked the faster path at every point; the pages' thresholds (prefix
      // >= 256, batch >= 8) lost up to 2.1x at N = 4.
      int64_t flat_tokens = 0, casc_tokens = cpl;
      for (int r = 0; r < num_reqs; ++r) {
        flat_tokens += seq_lens[r];
        casc_tokens += seq_lens[r] - cpl;
      }
      (void)num_q_heads;
      (void)num_kv_heads;
      (void)head_dim;
      (void)num_sms;
      use = cpl > 0 && casc_tokens > 0 && flat_tokens >= kAutoMinFlatTokens &&
            5 * flat_tokens >= 9 * casc_tokens;
      break;
    }
  }
  *use_cascade_out = use;
  return CSP_OK;
}

int csp_validate_batch(const int32_t* block_table, int64_t bt_row_stride, int32_t num_reqs,
                       const int32_t* seq_lens, const int32_t* cu_seqlens_q,
                       int32_t block_size, int32_t num_blocks, int32_t common_prefix_len,
                       int64_t* bad_index_out) {
  if (bad_index_out) *bad_index_out = -1;
  if (num_reqs < 0 || block_size <= 0 || num_blocks <= 0 || bt_row_stride < 0)
    return CSP_ERR_INVALID_ARG;
  if (num_reqs > 0 && (!block_table || !seq_lens)) return CSP_ERR_INVALID_ARG;
  int32_t min_len = num_reqs > 0 ? INT32_MAX : 0;
  for (int32_t r = 0; r < num_reqs; ++r) {
    const int32_t len = seq_lens[r];
    if (len < 0) return CSP_ERR_INVALID_ARG;
    min_len = len < min_len ? len : min_len;
    const int64_t pages = (static_cast<int64_t>(len) + block_size - 1) / block_size;
    if (pages > bt_row_stride) return CSP_ERR_INVALID_ARG;
    const int32_t* row = block_table + static_cast<int64_t>(r) * bt_row_stride;
    for (int64_t j = 0; j < pages; ++j) {
      if (row[j] < 0 || row[j] >= num_blocks) {
        if (bad_index_out) *bad_index_out = static_cast<int64_t>(r) * bt_row_stride + j;
        return CSP_ERR_INVALID_ARG;
      }
    }
    if (cu_seqlens_q) {
      if (r == 0 && cu_seqlens_q[0] != 0) return CSP_ERR_INVALID_ARG;
      const int64_t ql = static_cast<int64_t>(cu_seqlens_q[r + 1]) - cu_seqlens_q[r];
      if (ql < 0 || ql > len) return CSP_ERR_INVALID_ARG;
    }
  }
  if (common_prefix_len < 0 || common_prefix_len % block_size != 0 ||
      common_prefix_len > min_len)
    return CSP_ERR_INVALID_ARG;
  return CSP_OK;
}

int csp_workspace_size(int32_t num_reqs, int32_t total_q, int32_t max_seqlen_q,
                       int32_t max_seqlen_k, int32_t common_prefix_len, int32_t num_q_heads,
                       int32_t num_kv_heads, int32_t head_dim, size_t* bytes_out) {
  if (!bytes_out) return CSP_ERR_INVALID_ARG;
  int st = check_shape(num_reqs, total_q, max_seqlen_q, max_seqlen_k, num_q_heads, num_kv_heads,
                       head_dim, kPage);
  if (st != CSP_OK) return st;
  if (common_prefix_len < 0 || common_prefix_len % kPage != 0) return CSP_ERR_INVALID_ARG;
  int sms = 0;
  if ((st = device_sm_count(&sms)) != CSP_OK) return st;
  LaunchPlan P;
  make_plan(num_reqs, total_q, max_seqlen_q, max_seqlen_k, common_prefix_len, num_q_heads,
            num_kv_heads, head_dim, sms, &P);
  *bytes_out = P.bytes;
  return CSP_OK;
}

int cascade_attn(const void* q, const void* k_cache, const void* v_cache, int32_t num_blocks,
                 const int32_t* block_table, int64_t bt_row_stride, const int32_t* cu_seqlens_q,
                 const int32_t* seqused_k, int32_t num_reqs, int32_t total_q,
                 int32_t max_seqlen_q, int32_t max_seqlen_k, int32_t common_prefix_len,
                 int32_t block_size, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                 float softmax_scale, void* out, float* lse, void* workspace,
                 size_t workspace_bytes, void* stream) {
  return attention_call(q, k_cache, v_cache, num_blocks, block_table, bt_row_stride, cu_seqlens_q,
                        seqused_k, num_reqs, total_q, max_seqlen_q, max_seqlen_k,
                        common_prefix_len, block_size, num_q_heads, num_kv_heads, head_dim,
                        softmax_scale, out, lse, workspace, workspace_bytes, stream);
}

int cascade_attn_scheduled(const void* q, const void* k_cache, const void* v_cache,
                           int32_t num_blocks, const int32_t* block_table, int64_t bt_row_stride,
                           const int32_t* cu_seqlens_q, const int32_t* seqused_k,
                           int32_t num_reqs, int32_t total_q, int32_t max_seqlen_q,
                           int32_t max_seqlen_k, int32_t common_prefix_len, int32_t block_size,
                           int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                           float softmax_scale, void* out, float* lse, void* workspace,
                           size_t workspace_bytes, void* stream, int32_t schedule,
                           int32_t prefix_ranges) {
  if (schedule != CSP_SCHEDULE_TWO_KERNELS && schedule != CSP_SCHEDULE_SINGLE &&
      schedule != CSP_SCHEDULE_FUSED)
    return CSP_ERR_INVALID_ARG;
  if (prefix_ranges < 0 || common_prefix_len <= 0) return CSP_ERR_INVALID_ARG;
  return attention_call(q, k_cache, v_cache, num_blocks, block_table, bt_row_stride, cu_seqlens_q,
                        seqused_k, num_reqs, total_q, max_seqlen_q, max_seqlen_k,
                        common_prefix_len, block_size, num_q_heads, num_kv_heads, head_dim,
                        softmax_scale, out, lse, workspace, workspace_bytes, stream, nullptr,
                        schedule, prefix_ranges);
}

int cascade_attn_timed(const void* q, const void* k_cache, const void* v_cache,
                       int32_t num_blocks, const int32_t* block_table, int64_t bt_row_stride,
                       const int32_t* cu_seqlens_q, const int32_t* seqused_k, int32_t num_reqs,
                       int32_t total_q, int32_t max_seqlen_q, int32_t max_seqlen_k,
                       int32_t common_prefix_len, int32_t block_size, int32_t num_q_heads,
                       int32_t num_kv_heads, int32_t head_dim, float softmax_scale, void* out,
                       float* lse, void* workspace, size_t workspace_bytes, void* stream,
                       void* const* phase_events) {
  if (!phase_events) return CSP_ERR_INVALID_ARG;
  for (int i = 0; i < 4; ++i)
    if (!phase_events[i]) return CSP_ERR_INVALID_ARG;
  return attention_call(q, k_cache, v_cache, num_blocks, block_table, bt_row_stride, cu_seqlens_q,
                        seqused_k, num_reqs, total_q, max_seqlen_q, max_seqlen_k,
                        common_prefix_len, block_size, num_q_heads, num_kv_heads, head_dim,
                        softmax_scale, out, lse, workspace, workspace_bytes, stream,
                        phase_events);
}

int csp_workspace_size_fp8kv(int32_t num_reqs, int32_t total_q, int32_t max_seqlen_q,
                             int32_t max_seqlen_k, int32_t common_prefix_len, int32_t num_q_heads,
                             int32_t num_kv_heads, int32_t head_dim, size_t* bytes_out) {
  if (!bytes_out) return CSP_ERR_INVALID_ARG;
  int st = check_shape(num_reqs, total_q, max_seqlen_q, max_seqlen_k, num_q_heads, num_kv_heads,
                       head_dim, kPage);
  if (st != CSP_OK) return st;
  if (common_prefix_len < 0 || common_prefix_len % kPage != 0) return CSP_ERR_INVALID_ARG;
  int sms = 0;
  if ((st = device_sm_count(&sms)) != CSP_OK) return st;
  LaunchPlan P;
  make_plan(num_reqs, total_q, max_seqlen_q, max_seqlen_k, common_prefix_len, num_q_heads,
            num_kv_heads, head_dim, sms, &P, CSP_SCHEDULE_TWO_KERNELS);
  *bytes_out = align256(P.bytes) + align256(static_cast<size_t>(total_q) * num_q_heads * head_dim * 2);
  return CSP_OK;
}

int cascade_attn_fp8kv(const void* q, const void* k_cache, const void* v_cache,
                       int32_t num_blocks, const int32_t* block_table, int64_t bt_row_stride,
                       const int32_t* cu_seqlens_q, const int32_t* seqused_k, int32_t num_reqs,
                       int32_t total_q, int32_t max_seqlen_q, int32_t max_seqlen_k,
                       int32_t common_prefix_len, int32_t block_size, int32_t num_q_heads,
                       int32_t num_kv_heads, int32_t head_dim, float softmax_scale,
                       float k_scale, float v_scale, void* out, float* lse, void* workspace,
                       size_t workspace_bytes, void* stream) {
  return attention_call(q, k_cache, v_cache, num_blocks, block_table, bt_row_stride, cu_seqlens_q,
                        seqused_k, num_reqs, total_q, max_seqlen_q, max_seqlen_k,
                        common_prefix_len, block_size, num_q_heads, num_kv_heads, head_dim,
                        softmax_scale, out, lse, workspace, workspace_bytes, stream, nullptr, -1,
                        0, nullptr, true, k_scale, v_scale);
}

int paged_attn_fp8kv(const void* q, const void* k_cache, const void* v_cache, int32_t num_blocks,
                     const int32_t* block_table, int64_t bt_row_stride,
                     const int32_t* cu_seqlens_q, const int32_t* seqused_k, int32_t num_reqs,
                     int32_t total_q, int32_t max_seqlen_q, int32_t max_seqlen_k,
                     int32_t block_size, int32_t num_q_heads, int32_t num_kv_heads,
                     int32_t head_dim, float softmax_scale, float k_scale, float v_scale,
                     void* out, float* lse, void* workspace, size_t workspace_bytes,
                     void* stream) {
  return attention_call(q, k_cache, v_cache, num_blocks, block_table, bt_row_stride, cu_seqlens_q,
                        seqused_k, num_reqs, total_q, max_seqlen_q, max_seqlen_k, 0, block_size,
                        num_q_heads, num_kv_heads, head_dim, softmax_scale, out, lse, workspace,
                        workspace_bytes, stream, nullptr, -1, 0, nullptr, true, k_scale, v_scale);
}

int paged_attn(const void* q, const void* k_cache, const void* v_cache, int32_t num_blocks,
               const int32_t* block_table, int64_t bt_row_stride, const int32_t* cu_seqlens_q,
               const int32_t* seqused_k, int32_t num_reqs, int32_t total_q, int32_t max_seqlen_q,
               int32_t max_seqlen_k, int32_t block_size, int32_t num_q_heads,
               int32_t num_kv_heads, int32_t head_dim, float softmax_scale, void* out,
               float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  return attention_call(q, k_cache, v_cache, num_blocks, block_table, bt_row_stride, cu_seqlens_q,
                        seqused_k, num_reqs, total_q, max_seqlen_q, max_seqlen_k, 0, block_size,
                        num_q_heads, num_kv_heads, head_dim, softmax_scale, out, lse, workspace,
                        workspace_bytes, stream);
}

int merge_states(void* out, float* out_lse, const void* prefix_out, const float* prefix_lse,
                 const void* suffix_out, const float* suffix_lse, int32_t num_tokens,
                 int32_t num_heads, int32_t head_dim, int32_t partial_dtype, void* stream) {
  if (num_tokens < 0 || num_heads <= 0 || head_dim <= 0 || head_dim % 8 != 0 || head_dim > 512)
    return CSP_ERR_INVALID_ARG;
  if (partial_dtype != CSP_DTYPE_BF16 && partial_dtype != CSP_DTYPE_F32)
    return CSP_ERR_INVALID_ARG;
  if (num_tokens == 0) return CSP_OK;
  if (!out || !prefix_out || !prefix_lse || !suffix_out || !suffix_lse)
    return CSP_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(prefix_out) || !aligned16(suffix_out))
    return CSP_ERR_INVALID_ARG;
  cudaError_t e = csp::launch_merge_states(
      static_cast<__nv_bfloat16*>(out), out_lse, prefix_out, prefix_lse, suffix_out, suffix_lse,
      num_tokens * num_heads, head_dim, partial_dtype == CSP_DTYPE_F32,
      static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CSP_OK : cuda_fail(e);
}

int cascade_plan_device(const int32_t* block_table, int64_t bt_row_stride, int32_t num_reqs,
                        const int32_t* seq_lens, const int32_t* num_computed_tokens,
                        int32_t block_size, int32_t mode, int32_t* plan_out, void* stream) {
  if (!plan_out || num_reqs < 0 || block_size <= 0 || bt_row_stride < 0)
    return CSP_ERR_INVALID_ARG;
  if (mode < CSP_MODE_AUTO || mode > CSP_MODE_PAGE_THRESHOLDS) return CSP_ERR_INVALID_ARG;
  if (num_reqs > 0 && (!block_table || !seq_lens || !num_computed_tokens))
    return CSP_ERR_INVALID_ARG;
  cudaError_t e = csp::launch_plan_device(block_table, bt_row_stride, num_reqs, seq_lens,
                                          num_computed_tokens, block_size, mode, plan_out,
                                          static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CSP_OK : cuda_fail(e);
}

int cascade_attn_device_plan(const void* q, const void* k_cache, const void* v_cache,
                             int32_t num_blocks, const int32_t* block_table,
                             int64_t bt_row_stride, const int32_t* cu_seqlens_q,
                             const int32_t* seqused_k, int32_t num_reqs, int32_t total_q,
                             int32_t max_seqlen_q, int32_t max_seqlen_k, const int32_t* plan,
                             int32_t common_prefix_len_bound, int32_t block_size,
                             int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                             float softmax_scale, void* out, float* lse, void* workspace,
                             size_t workspace_bytes, void* stream) {
  if (!plan) return CSP_ERR_INVALID_ARG;
  return attention_call(q, k_cache, v_cache, num_blocks, block_table, bt_row_stride,
                        cu_seqlens_q, seqused_k, num_reqs, total_q, max_seqlen_q, max_seqlen_k,
                        common_prefix_len_bound, block_size, num_q_heads, num_kv_heads,
                        head_dim, softmax_scale, out, lse, workspace, workspace_bytes, stream,
                        nullptr, CSP_SCHEDULE_SINGLE, 0, plan);
}

int cascade_plan_levels(const int32_t* block_table, int64_t bt_row_stride, int32_t num_reqs,
                        const int32_t* seq_lens, const int32_t* num_computed_tokens,
                        int32_t block_size, int32_t max_levels, int32_t max_segments,
                        int32_t* segments_out, int32_t* num_segments_out,
                        int32_t* suffix_start_out) {
  if (!num_segments_out || num_reqs < 0 || block_size <= 0 || max_levels < 1 ||
      max_levels > kMaxLevels || max_segments < 0 || (max_segments > 0 && !segments_out))
    return CSP_ERR_INVALID_ARG;
  *num_segments_out = 0;
  if (num_reqs == 0) return CSP_OK;
  if (!block_table || !seq_lens || !num_computed_tokens || !suffix_start_out)
    return CSP_ERR_INVALID_ARG;
  std::vector<int64_t> used(num_reqs);
  std::vector<int32_t> tok(num_reqs + 1, 0);
  for (int r = 0; r < num_reqs; ++r) {
    if (seq_lens[r] < 0 || num_computed_tokens[r] < 0 || num_computed_tokens[r] > seq_lens[r])
      return CSP_ERR_INVALID_ARG;
    used[r] = cdiv64(seq_lens[r], block_size);
    if (used[r] > bt_row_stride) return CSP_ERR_INVALID_ARG;
    tok[r + 1] = tok[r] + (seq_lens[r] - num_computed_tokens[r]);
    suffix_start_out[r] = 0;
  }
  LevelWalk w{block_table, bt_row_stride, seq_lens, num_computed_tokens, used.data(), tok.data(),
              block_size, max_levels, max_segments, segments_out, 0, suffix_start_out};
  w.walk(0, num_reqs, 0, 0);
  if (w.overflow) return CSP_ERR_UNSUPPORTED;
  *num_segments_out = w.n;
  return CSP_OK;
}

int csp_workspace_size_levels(int32_t num_reqs, int32_t total_q, int32_t max_seqlen_q,
                              int32_t max_seqlen_k, const int32_t* segments,
                              int32_t num_segments, int32_t max_suffix_len, int32_t num_q_heads,
                              int32_t num_kv_heads, int32_t head_dim, size_t* bytes_out) {
  if (!bytes_out) return CSP_ERR_INVALID_ARG;
  int st = check_shape(num_reqs, total_q, max_seqlen_q, max_seqlen_k, num_q_heads, num_kv_heads,
                       head_dim, kPage);
  if (st != CSP_OK) return st;
  if ((st = check_segments(num_reqs, total_q, max_seqlen_k, segments, num_segments)) != CSP_OK)
    return st;
  if (max_suffix_len < 0 || max_suffix_len > max_seqlen_k) return CSP_ERR_INVALID_ARG;
  int sms = 0;
  if ((st = device_sm_count(&sms)) != CSP_OK) return st;
  LevelPlan L;
  if ((st = make_level_plan(num_reqs, total_q, max_seqlen_q, max_seqlen_k, segments,
                            num_segments, max_suffix_len, num_q_heads, num_kv_heads, head_dim,
                            sms, &L)) != CSP_OK)
    return st;
  *bytes_out = L.bytes;
  return CSP_OK;
}

int cascade_attn_levels(const void* q, const void* k_cache, const void* v_cache, int32_t num_blocks,
                        const int32_t* block_table, int64_t bt_row_stride,
                        const int32_t* cu_seqlens_q, const int32_t* seqused_k, int32_t num_reqs,
                        int32_t total_q, int32_t max_seqlen_q, int32_t max_seqlen_k,
                        const int32_t* segments, int32_t num_segments,
                        const int32_t* suffix_start, int32_t max_suffix_len, int32_t block_size,
                        int32_t Hq, int32_t Hkv, int32_t D, float softmax_scale, void* out,
                        float* lse, void* workspace, size_t workspace_bytes, void* stream_ptr) {
  int st = check_shape(num_reqs, total_q, max_seqlen_q, max_seqlen_k, Hq, Hkv, D, block_size);
  if (st != CSP_OK) return st;
  if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale)) return CSP_ERR_INVALID_ARG;
  if (num_blocks <= 0 || static_cast<int64_t>(num_blocks) * block_size > INT32_MAX)
    return CSP_ERR_INVALID_ARG;
  if (total_q == 0 || num_reqs == 0) return CSP_OK;
  if (!q || !k_cache || !v_cache || !block_table || !cu_seqlens_q || !seqused_k || !out ||
      !suffix_start)
    return CSP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return CSP_ERR_INVALID_ARG;
  if (bt_row_stride < cdiv(max_seqlen_k, block_size)) return CSP_ERR_INVALID_ARG;
  int sms = 0;
  if ((st = device_sm_count(&sms)) != CSP_OK) return st;
  LevelPlan L;
  if ((st = make_level_plan(num_reqs, total_q, max_seqlen_q, max_seqlen_k, segments, num_segments,
                            max_suffix_len, Hq, Hkv, D, sms, &L)) != CSP_OK)
    return st;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255) != 0 ||
      workspace_bytes < L.bytes)
    return CSP_ERR_WORKSPACE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* status = reinterpret_cast<int*>(ws);
  int* counters = reinterpret_cast<int*>(ws + L.off_counters);
  __nv_bfloat16* part_o = reinterpret_cast<__nv_bfloat16*>(ws + L.off_part_o);
  float* part_lse = reinterpret_cast<float*>(ws + L.off_part_lse);
  const int64_t rows = static_cast<int64_t>(total_q) * Hq;
  const int group = Hq / Hkv;
  const float scale_log2 = softmax_scale * 1.4426950408889634f;
  const LaunchPlan& P = L.suf;
  // as in the two-kernel schedule: the suffix writes its partials beside the segment
  // grid (neither waits for the other) and the slot merge follows
  const bool merge_after = true;
  const bool cluster = false;
  cudaError_t e;
  // a row no segment of a level holds reads lse = -inf (weight 0) in that level's slots
  if ((e = csp::launch_fill_f32(part_lse, L.n_prefix * rows, -INFINITY, stream)) != cudaSuccess)
    return cuda_fail(e);
  if (P.s_splits > 1 && !merge_after && !cluster &&
      (e = cudaMemsetAsync(counters, 0, static_cast<size_t>(total_q) * Hkv * sizeof(int32_t),
                           stream)) != cudaSuccess)
    return cuda_fail(e);
  CUtensorMap tm_q, tm_k, tm_v;
  const uint64_t row_b = static_cast<uint64_t>(D) * 2;
  const uint64_t ntok = static_cast<uint64_t>(num_blocks) * block_size;
  if ((st = make_map_3d(&tm_q, q, D, Hq, total_q, row_b, row_b * Hq, 64, group, 128 / group)) !=
          CSP_OK ||
      (st = make_map_3d(&tm_k, k_cache, D, Hkv, ntok, row_b, row_b * Hkv, 64, 1, kPage)) !=
          CSP_OK ||
      (st = make_map_kv_pages(&tm_v, v_cache, D, Hkv, ntok)) != CSP_OK)
    return st;
  // every segment with query rows in one grid (a table of at most
  // kMaxSegmentsPerLaunch segments per launch)
  csp::PrefixArgs pa;
  pa.k = static_cast<const __nv_bfloat16*>(k_cache);
  pa.v = static_cast<const __nv_bfloat16*>(v_cache);
  pa.block_table = block_table;
  pa.num_q_heads = Hq;
  pa.num_kv_heads = Hkv;
  pa.group = group;
  pa.scale_log2 = scale_log2;
  pa.part_o = part_o;
  pa.part_lse = part_lse;
  pa.lse_stride = rows;
  pa.rows_all = rows;
  pa.status = status;
  csp::SegmentTable table;
  table.n = 0;
  table.bt_stride = bt_row_stride;
  int grid = 0;
  bool launched = false;
  for (int i = 0; i <= num_segments; ++i) {
    if ((i == num_segments || table.n == csp::kMaxSegmentsPerLaunch) && table.n > 0) {
      if ((e = csp::launch_prefix_segments(D, tm_q, tm_k, tm_v, pa, table, grid, stream)) !=
          cudaSuccess)
        return cuda_fail(e);
      launched = true;
      table.n = 0;
      grid = 0;
    }
    if (i == num_segments) break;
    const int32_t* s = segments + static_cast<int64_t>(i) * kSegInts;
    const int tokens = s[6] - s[5];
    if (tokens == 0) continue;  // its requests have no query rows this step
    csp::SegmentDesc& sd = table.s[table.n++];
    sd.cta0 = grid;
    sd.bt_row = s[1];
    sd.key_lo = s[3];
    sd.key_hi = s[4];
    sd.tok0 = s[5];
    sd.tokens = tokens;
    sd.slot_base = L.level_base[s[0]];
    sd.splits = L.seg_splits[i];
    sd.tiles_per_split = cdiv(cdiv(s[4] - s[3], 64), sd.splits);
    sd.pairs = cdiv(tokens * group, 256);
    grid += Hkv * sd.pairs * sd.splits;
  }
  csp::PagedArgs ga;
  ga.q = static_cast<const __nv_bfloat16*>(q);
  ga.k = static_cast<const __nv_bfloat16*>(k_cache);
  ga.v = static_cast<const __nv_bfloat16*>(v_cache);
  ga.block_table = block_table;
  ga.bt_stride = bt_row_stride;
  ga.cu_seqlens_q = cu_seqlens_q;
  ga.seq_lens = seqused_k;
  ga.num_reqs = num_reqs;
  ga.total_q = total_q;
  ga.num_q_heads = Hq;
  ga.num_kv_heads = Hkv;
  ga.group = group;
  ga.key_start = 0;
  ga.key_start_of = suffix_start;
  ga.split_keys = P.s_split_keys;
  ga.n_splits = P.s_splits;
  ga.row_tiles = P.s_row_tiles;
  ga.scale_log2 = scale_log2;
  ga.part_o = part_o;
  ga.part_lse = part_lse;
  ga.n_prefix = L.n_prefix;
  ga.counters = (merge_after || cluster) ? nullptr : counters;
  ga.cluster_splits = cluster;
  ga.partials_only = merge_after;
  ga.out = static_cast<__nv_bfloat16*>(out);
  ga.lse = lse;
  ga.status = status;
  // concurrent with the last prefix grid (programmatic dependent launch: the suffix
  // waits for it before it reads the prefix slots; earlier prefix grids, launched
  // plainly, finished before it started)
  if (P.tc) {
    e = csp::launch_paged_tc(D, tm_q, tm_k, tm_v, ga, launched, stream);
  } else {
    e = csp::launch_paged(D, ga, launched, stream);
  }
  if (e != cudaSuccess) return cuda_fail(e);
  // in stream order (no programmatic launch): every slot is complete
  if (merge_after &&
      (e = csp::launch_merge_slots(D, part_o, part_lse, L.n_parts, rows,
                                   static_cast<__nv_bfloat16*>(out), lse, stream)) != cudaSuccess)
    return cuda_fail(e);
  return CSP_OK;
}

// ---------------------------------------------------------------- host step --
// One step from host buffers: the layout of the device scratch (256-byte aligned
// pieces): the attention call's workspace first (its header — the status word and the
// single kernel's barrier — stays at the scratch's start whatever the batch), then q,
// block table, cu_seqlens_q, seq_lens, out and lse.  Fills the sizes and maxima for the
// batch; returns CSP_OK or an argument error.
struct StepLayout {
  int32_t max_q = 0, max_k = 0;
  size_t off_q = 0, off_bt = 0, off_cu = 0, off_sl = 0, off_out = 0, off_lse = 0, off_ws = 0;
  size_t q_bytes = 0, bt_bytes = 0, out_bytes = 0, lse_bytes = 0, ws_bytes = 0, total = 0;
};

int step_layout(int32_t num_reqs, int32_t total_q, const int32_t* cu_seqlens_q,
                const int32_t* seq_lens, int64_t bt_row_stride, int32_t cpl, int32_t Hq,
                int32_t Hkv, int32_t D, StepLayout* L) {
  if (num_reqs < 0 || total_q < 0 || bt_row_stride < 0) return CSP_ERR_INVALID_ARG;
  if (num_reqs > 0 && (!cu_seqlens_q || !seq_lens)) return CSP_ERR_INVALID_ARG;
  StepLayout l;
  if (num_reqs > 0 && (cu_seqlens_q[0] != 0 || cu_seqlens_q[num_reqs] != total_q))
    return CSP_ERR_INVALID_ARG;
  for (int r = 0; r < num_reqs; ++r) {
    const int32_t ql = cu_seqlens_q[r + 1] - cu_seqlens_q[r];
    if (ql < 0 || seq_lens[r] < ql) return CSP_ERR_INVALID_ARG;
    l.max_q = std::max(l.max_q, ql);
    l.max_k = std::max(l.max_k, seq_lens[r]);
  }
  int st = csp_workspace_size(num_reqs, total_q, l.max_q, l.max_k, cpl, Hq, Hkv, D, &l.ws_bytes);
  if (st != CSP_OK) return st;
  l.q_bytes = static_cast<size_t>(total_q) * Hq * D * 2;
  l.bt_bytes = static_cast<size_t>(num_reqs) * bt_row_stride * 4;
  l.out_bytes = l.q_bytes;
  l.lse_bytes = static_cast<size_t>(total_q) * Hq * 4;
  l.off_ws = 0;
  l.off_q = align256(l.ws_bytes);
  l.off_bt = l.off_q + align256(l.q_bytes);
  l.off_cu = l.off_bt + align256(l.bt_bytes);
  l.off_sl = l.off_cu + align256(static_cast<size_t>(num_reqs + 1) * 4);
  l.off_out = l.off_sl + align256(static_cast<size_t>(num_reqs) * 4);
  l.off_lse = l.off_out + align256(l.out_bytes);
  l.total = l.off_lse + align256(l.lse_bytes);
  *L = l;
  return CSP_OK;
}

int csp_step_scratch_size(int32_t num_reqs, int32_t total_q, const int32_t* cu_seqlens_q,
                          const int32_t* seq_lens, int64_t bt_row_stride,
                          int32_t common_prefix_len, int32_t num_q_heads, int32_t num_kv_heads,
                          int32_t head_dim, size_t* bytes_out) {
  if (!bytes_out) return CSP_ERR_INVALID_ARG;
  StepLayout L;
  const int st = step_layout(num_reqs, total_q, cu_seqlens_q, seq_lens, bt_row_stride,
                             common_prefix_len, num_q_heads, num_kv_heads, head_dim, &L);
  if (st != CSP_OK) return st;
  *bytes_out = L.total;
  return CSP_OK;
}

int cascade_step_host(const void* q, const int32_t* block_table, int64_t bt_row_stride,
                      const int32_t* cu_seqlens_q, const int32_t* seq_lens,
                      const int32_t* num_computed_tokens, int32_t num_reqs, int32_t total_q,
                      const void* k_cache, const void* v_cache, int32_t num_blocks,
                      int32_t block_size, int32_t num_q_heads, int32_t num_kv_heads,
                      int32_t head_dim, float softmax_scale, int32_t mode, void* out, float* lse,
                      void* device_scratch, size_t scratch_bytes, void* stream_ptr,
                      int32_t* common_prefix_len_out) {
  if (total_q == 0 || num_reqs == 0) {
    if (common_prefix_len_out) *common_prefix_len_out = 0;
    return CSP_OK;
  }
  if (!q || !block_table || !cu_seqlens_q || !seq_lens || !num_computed_tokens || !out ||
      !lse)
    return CSP_ERR_INVALID_ARG;
  int32_t cpl = 0, use = 0;
  int st = cascade_plan(block_table, bt_row_stride, num_reqs, seq_lens, num_computed_tokens,
                        block_size, num_q_heads, num_kv_heads, head_dim, 0, mode, &cpl, &use);
  if (st != CSP_OK) return st;
  if (!use) cpl = 0;
  StepLayout L;
  if ((st = step_layout(num_reqs, total_q, cu_seqlens_q, seq_lens, bt_row_stride, cpl,
                        num_q_heads, num_kv_heads, head_dim, &L)) != CSP_OK)
    return st;
  if (!device_scratch || (reinterpret_cast<uintptr_t>(device_scratch) & 255) != 0 ||
      scratch_bytes < L.total)
    return CSP_ERR_WORKSPACE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  uint8_t* d = static_cast<uint8_t*>(device_scratch);
  cudaError_t e;
  // the step's inputs in: four copies (from pinned host memory they run asynchronously)
  if ((e = cudaMemcpyAsync(d + L.off_q, q, L.q_bytes, cudaMemcpyHostToDevice, stream)) !=
          cudaSuccess ||
      (e = cudaMemcpyAsync(d + L.off_bt, block_table, L.bt_bytes, cudaMemcpyHostToDevice,
                           stream)) != cudaSuccess ||
      (e = cudaMemcpyAsync(d + L.off_cu, cu_seqlens_q, static_cast<size_t>(num_reqs + 1) * 4,
                           cudaMemcpyHostToDevice, stream)) != cudaSuccess ||
      (e = cudaMemcpyAsync(d + L.off_sl, seq_lens, static_cast<size_t>(num_reqs) * 4,
                           cudaMemcpyHostToDevice, stream)) != cudaSuccess)
    return cuda_fail(e);
  st = attention_call(d + L.off_q, k_cache, v_cache, num_blocks,
                      reinterpret_cast<const int32_t*>(d + L.off_bt), bt_row_stride,
                      reinterpret_cast<const int32_t*>(d + L.off_cu),
                      reinterpret_cast<const int32_t*>(d + L.off_sl), num_reqs, total_q, L.max_q,
                      L.max_k, cpl, block_size, num_q_heads, num_kv_heads, head_dim,
                      softmax_scale, d + L.off_out, reinterpret_cast<float*>(d + L.off_lse),
                      d + L.off_ws, L.ws_bytes, stream);
  if (st != CSP_OK) return st;
  // the result out, and the host waits for it
  if ((e = cudaMemcpyAsync(out, d + L.off_out, L.out_bytes, cudaMemcpyDeviceToHost, stream)) !=
          cudaSuccess ||
      (e = cudaMemcpyAsync(lse, d + L.off_lse, L.lse_bytes, cudaMemcpyDeviceToHost, stream)) !=
          cudaSuccess ||
      (e = cudaStreamSynchronize(stream)) != cudaSuccess)
    return cuda_fail(e);
  if (common_prefix_len_out) *common_prefix_len_out = cpl;
  return CSP_OK;
}

int csp_apply_sinks(void* out, float* lse, const float* sinks, int32_t num_tokens,
                    int32_t num_heads, int32_t head_dim, void* stream) {
  if (num_tokens < 0 || num_heads <= 0 || head_dim <= 0 || head_dim % 8 != 0 ||
      32 % (head_dim / 8) != 0)
    return CSP_ERR_INVALID_ARG;
  if (num_tokens == 0) return CSP_OK;
  if (!out || !lse || !sinks || !aligned16(out)) return CSP_ERR_INVALID_ARG;
  if (static_cast<int64_t>(num_tokens) * num_heads > INT32_MAX) return CSP_ERR_INVALID_ARG;
  cudaError_t e = csp::launch_apply_sinks(static_cast<__nv_bfloat16*>(out), lse, sinks,
                                          num_tokens * num_heads, num_heads, head_dim,
                                          static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CSP_OK : cuda_fail(e);
}

int csp_workspace_status(const void* workspace, void* stream, int32_t* status_out) {
  if (!workspace || !status_out) return CSP_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(status_out, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return e == cudaSuccess ? CSP_OK : cuda_fail(e);
}

const char* csp_status_string(int status) {
  switch (status) {
    case CSP_OK: return "CSP_OK";
    case CSP_ERR_INVALID_ARG: return "CSP_ERR_INVALID_ARG";
    case CSP_ERR_UNSUPPORTED: return "CSP_ERR_UNSUPPORTED";
    case CSP_ERR_WORKSPACE: return "CSP_ERR_WORKSPACE";
    case CSP_ERR_CUDA: return "CSP_ERR_CUDA";
    case CSP_ERR_TIMEOUT: return "CSP_ERR_TIMEOUT";
    default: return "CSP_ERR_UNKNOWN";
  }
}

int csp_last_cuda_error(void) { return g_last_cuda_error; }

int csp_version(void) { return (1 << 16) | 1; }

int csp_cascade_schedule(int32_t num_reqs, int32_t total_q, int32_t max_seqlen_q,
                         int32_t max_seqlen_k, int32_t common_prefix_len, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_dim, int32_t* schedule_out,
                         int32_t* prefix_splits_out) {
  if (!schedule_out) return CSP_ERR_INVALID_ARG;
  int st = check_shape(num_reqs, total_q, max_seqlen_q, max_seqlen_k, num_q_heads, num_kv_heads,
                       head_dim, kPage);
  if (st != CSP_OK) return st;
  if (common_prefix_len <= 0 || common_prefix_len % kPage != 0 ||
      common_prefix_len > max_seqlen_k)
    return CSP_ERR_INVALID_ARG;
  int sms = 0;
  if ((st = device_sm_count(&sms)) != CSP_OK) return st;
  LaunchPlan P;
  make_plan(num_reqs, total_q, max_seqlen_q, max_seqlen_k, common_prefix_len, num_q_heads,
            num_kv_heads, head_dim, sms, &P);
  *schedule_out = P.single ? CSP_SCHEDULE_SINGLE
                           : (P.fused ? CSP_SCHEDULE_FUSED : CSP_SCHEDULE_TWO_KERNELS);
  if (prefix_splits_out) *prefix_splits_out = P.single ? P.d_splits : P.p_splits;
  return CSP_OK;
}

}  // extern "C"
