// dora_api.cu -- the C ABI (include/dora.h): argument checks, workspace plan,
// TMA descriptors and the launch sequence of the factored norm and compose.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "dora.h"
#include "common.cuh"
#include "finalize.cuh"

namespace dora {

static std::atomic<uint64_t> g_launches{0};
void note_launches(int n) { g_launches.fetch_add(static_cast<uint64_t>(n), std::memory_order_relaxed); }

namespace {

constexpr int kMaxMainSplits = 16;
#ifndef DORA_GRAM_CLUSTER
#define DORA_GRAM_CLUSTER 8
#endif
constexpr int kGramCluster = DORA_GRAM_CLUSTER;   // CTAs (K splits) per Gram block
constexpr int kGramClusterGrouped = 2;            // the same for a grouped launch
constexpr int kGramStages = 6;
static_assert(kMaxMainSplits <= kMaxFinalParts, "the fused finalize sums at most kMaxFinalParts splits");
static_assert(kMaxFinalParts <= kTf32MaxGramSplits, "the 3xTF32 segment table holds every split");
constexpr int kMaxDevices = 64;
constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;   // 2 s per pipeline wait

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ---------------------------------------------------------------- device info
struct DeviceInfo {
  int sms = 0;
  int ok = 0;   // 1: sm_10x device usable by this library, -1: not usable
};
std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

int current_device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DORA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (d.ok == 0) {
    int major = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return DORA_ERR_CUDA;
    d.sms = sms;
    d.ok = (major == 10) ? 1 : -1;
  }
  if (d.ok < 0) return DORA_ERR_NO_DEVICE;
  *out = d;
  return DORA_OK;
}

// ---------------------------------------------------------------- TMA descriptors
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Row-major [outer x inner] bf16 matrix, box [box_outer x 64], 128-byte swizzle,
// out-of-bounds elements read as zero.
bool make_map_bf16(CUtensorMap* map, const void* ptr, uint64_t inner, uint64_t outer,
                   uint32_t box_outer) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kTcBlockK), box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row-major [outer x inner] fp32 matrix, box [box_outer x 32], 128-byte
// swizzle, out-of-bounds elements read as zero.
bool make_map_f32(CUtensorMap* map, const void* ptr, uint64_t inner, uint64_t outer,
                  uint32_t box_outer) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 4};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kTf32BlockK), box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Gram blocks: the upper triangle of the nb x nb grid of 128-row blocks of
// G [rp x rp], each block bw columns wide.
int gram_nb(int rp) { return static_cast<int>((rp + 127) / 128); }
int gram_bw(int rp) { return rp > 128 ? 128 : rp; }

// Control block at the start of the workspace, zeroed by every call (int
// words): [0] device status, [32] work counter of the main pass,
// [64, 64 + 2 * pair tiles) K segments finished per 128-row group.
constexpr int kCtlWork = 32, kCtlTileDone = 64;

// ---------------------------------------------------------------- workspace plan
struct Plan {
  bool bf16 = true;
  int rp = 0;               // r rounded up to 16 (the MMA N extent)
  size_t off_status = 0, zero_bytes = 0, off_G = 0, off_Ghi = 0, off_Glo = 0;
  size_t off_Gpart = 0;     // fp32: K-segment partials of G
  size_t off_pbase = 0, off_pcross = 0, total = 0;
  int cap_base = 0, cap_cross = 0;
};

Plan make_plan(int64_t d_out, int64_t d_in, int64_t r, int dtype) {
  Plan p;
  p.bf16 = dtype == DORA_BF16;
  p.rp = static_cast<int>(ceil_div(r, 16) * 16);
  p.cap_base = kMaxMainSplits;
  p.cap_cross = kMaxMainSplits;
  size_t off = 0;
  p.off_status = off;
  const int64_t pair_tiles = ceil_div(d_out, 2 * kTcBlockM);
  off = align_up((kCtlTileDone + 2 * static_cast<size_t>(pair_tiles)) * 4, 256);
  p.zero_bytes = off;
  const size_t rp2 = static_cast<size_t>(p.rp) * p.rp;
  if (p.bf16) {
    p.off_Ghi = off;
    off = align_up(off + rp2 * 2, 256);
    p.off_Glo = off;
    off = align_up(off + rp2 * 2, 256);
  } else {
    p.off_G = off;
    off = align_up(off + rp2 * 4, 256);
    p.off_Gpart = off;
    off = align_up(off + static_cast<size_t>(kTf32MaxGramSplits) * r * r * 4, 256);
  }
  p.off_pbase = off;
  off = align_up(off + static_cast<size_t>(p.cap_base) * d_out * 4, 256);
  p.off_pcross = off;
  off = align_up(off + static_cast<size_t>(p.cap_cross) * d_out * 4, 256);
  p.total = off;
  (void)d_in;
  return p;
}

bool shape_ok(int64_t d_out, int64_t d_in, int64_t r, int dtype) {
  return d_out >= 0 && d_in >= 0 && r >= 0 && r <= DORA_MAX_RANK &&
         (dtype == DORA_BF16 || dtype == DORA_F32) && d_out < (int64_t(1) << 31) &&
         d_in < (int64_t(1) << 31);
}

int gcd_int(int a, int b) {
  while (b) {
    const int t = a % b;
    a = b;
    b = t;
  }
  return a;
}

// K splits of the pair main pass: minimise (items per cluster) x (K tiles per
// item + about three tiles of epilogue), items = pair_tiles x splits.
int pick_pair_splits(int64_t pair_tiles, int64_t k_tiles, int clusters, int max_splits) {
  int best = 1;
  double best_cost = 1e300;
  const int lim = static_cast<int>(k_tiles < max_splits ? k_tiles : max_splits);
  for (int s = 1; s <= (lim > 0 ? lim : 1); ++s) {
    const int64_t rounds = ceil_div(pair_tiles * s, clusters);
    const double cost = static_cast<double>(rounds) * (ceil_div(k_tiles, s) + 3.0);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

// K segments of each pair tile: long work first, short work to even out the
// finish; every extra item costs an accumulator drain.  With fewer pair tiles
// than pairs, each pair runs one or two items and the long first items set
// the finish: relative lengths 7 : 4 : 2 (on one GB300 at 8192 x 8192,
// r = 384 -- 140 K tiles, 32 pair tiles, 76 pairs of which the 24 that share
// SMs with the Gram kernel start late -- 7:4:2 and 9:5:3 took 49.3 us per
// norm, 3:2:1 51.0, 4:2:1 51.4, 7:3:2 52.8; four or more segments were
// slower).  With more pair tiles than pairs, 3 : 2 : 1 (28672 x 8192, 112
// pair tiles: 140.0 us against 142.3 with 7:4:2).  With few tiles, equal
// segments, as many as keep the pairs busy.
void plan_pair_segments(PairParams& pp, int clusters) {
  const int ktot = pp.kt_w + 2 * pp.kt_b;
  int nseg;
  if (3 * static_cast<int64_t>(pp.pair_tiles) >= clusters && ktot >= 6) {
    static const int w_few[3] = {7, 4, 2};
    static const int w_many[3] = {3, 2, 1};
    const int* w = pp.pair_tiles < clusters ? w_few : w_many;
    const int wsum = w[0] + w[1] + w[2];
    nseg = 3;
    int acc = 0;
    pp.seg_k[0] = 0;
    for (int i = 0; i < 3; ++i) {
      acc += w[i];
      pp.seg_k[i + 1] = static_cast<int>((static_cast<int64_t>(ktot) * acc + wsum / 2) / wsum);
    }
  } else {
    nseg = pick_pair_splits(pp.pair_tiles, ktot, clusters, kMaxMainSplits);
    for (int i = 0; i <= nseg; ++i)
      pp.seg_k[i] = static_cast<int>((static_cast<int64_t>(ktot) * i) / nseg);
  }
  pp.splits = nseg;
}

// Static ranges of the single-module main pass: pair slot i (its place in
// the start order) owns a contiguous range of the (pair tile, K tile)
// iterations and drains its accumulator only where the range crosses a tile
// boundary, so every pair finishes at about the same time.  The pairs that
// start after the Gram kernel (one per two of its CTAs; they take the last
// slots) get `lag` fewer K tiles: about 1 us + 0.7 us per Gram K tile of
// one CTA, against 0.47 us per main-pass K tile at r = 384 (tensor-bound;
// bound by W's HBM stream below r ~ 288).  Used with at least as many pair
// tiles as pairs, every range at least kMinRange K tiles long and no pair
// tile meeting more than kMaxMainSplits ranges; otherwise the K segments.
// Measured per call on one GB300 (static ranges against K segments):
// 28672 x 8192, r = 384: 131.7 against 140.9 us; with fewer tiles than
// pairs the segments won at 8192 x 8192, r = 384 (49.3 against 54.8-57.3 us
// over lags of 19 to 60 K tiles) and static ranges were within 5 % either
// way at 8192 x 8192, r = 128 and 11008 x 4096, r = 64.
#ifndef DORA_STATIC_RANGES
#define DORA_STATIC_RANGES 1
#endif
#ifndef DORA_RANGE_LATE_US0
#define DORA_RANGE_LATE_US0 1.0
#endif
#ifndef DORA_RANGE_LATE_US_PER_KT
#define DORA_RANGE_LATE_US_PER_KT 0.7
#endif
constexpr int64_t kMinRange = 8;

// K tiles a pair behind the Gram kernel starts after the others: about
// 1 us + 0.7 us per Gram K tile of one CTA, against 0.47 us per main-pass K
// tile at r = 384 (tensor-bound; bound by W's HBM stream below r ~ 288)
int64_t gram_lag_tiles(const PairParams& pp, int gram_kt) {
  const int rp = pp.n0 + pp.n1;
  const double tau_us = 0.47 * (rp > 288 ? rp : 288) / 384.0;
  return std::llround((DORA_RANGE_LATE_US0 + DORA_RANGE_LATE_US_PER_KT * gram_kt) / tau_us);
}

bool plan_pair_ranges(PairParams& pp, int clusters, int gram_ctas, int gram_kt) {
  pp.ranges = 0;
  if (!DORA_STATIC_RANGES || clusters <= 0 || pp.pair_tiles < clusters) return false;
  const int64_t ktot = pp.kt_w + 2 * static_cast<int64_t>(pp.kt_b);
  const int64_t iters = static_cast<int64_t>(pp.pair_tiles) * ktot;
  if (ktot <= 0 || iters >= (int64_t(1) << 30)) return false;
  const int64_t n = clusters;
  int64_t late = gram_ctas > 0 ? (gram_ctas + 1) / 2 : 0;
  if (late >= n) late = 0;
  const int64_t lag = late > 0 ? gram_lag_tiles(pp, gram_kt) : 0;
  const int64_t le = ceil_div(iters + late * lag, n);
  const int64_t ll = late > 0 ? (le - lag > 1 ? le - lag : 1) : le;
  const int64_t lmin = ll < le ? ll : le;
  if (lmin < kMinRange) return false;
  // a tile of ktot iterations meets at most ktot / lmin whole ranges, two
  // partial ones and the shortened last range
  if (ktot / lmin + 3 > kMaxMainSplits) return false;
  if ((n - late) * le + late * ll < iters) return false;     // the ranges cover every iteration
  pp.ranges = static_cast<int>(n);
  pp.ktot = static_cast<int>(ktot);
  pp.iters = static_cast<int>(iters);
  pp.n_early = static_cast<int>(n - late);
  pp.len_early = static_cast<int>(le);
  pp.len_late = static_cast<int>(ll);
  return true;
}

// Piece table of the single-module main pass with fewer pair tiles than
// pairs: every pair runs exactly one piece (a K range of one pair tile), so
// no pair pays for a second accumulator drain (about 2.4 us at r = 384),
// and the pieces are sized for when their pairs start.  The `late` pairs
// that share SMs with the Gram kernel start about `lag` K tiles after the
// others and claim last, so they get pieces `lag` tiles shorter.  A tile is
// cut into e pieces for early pairs and l for late ones; with F the longest
// early piece, e F + l (F - lag) >= ktot must hold.  The smallest F for which
// the tiles can be cut with at most n - late early and late late pieces is
// found by a small dynamic program over the tiles (they are all alike, so
// it only counts pieces).  Inside a tile the early pieces come first in K
// and the late ones (which start after the Gram kernel has finished) hold
// the (B, G') tiles at the end; the table lists the early pieces longest
// first, then the late ones.  Returns false (K segments are used) when the
// cut needs more than kMaxMainSplits pieces in a tile or kPairTabMax pieces.
// Measured on one GB300 at 8192 x 8192, r = 384: see plan_main_pass.
#ifndef DORA_PIECE_TABLE
#define DORA_PIECE_TABLE 1
#endif
// The cut depends only on (pair tiles, K tiles, pairs, late, lag); it is
// planned once per such key (a dynamic program of up to a few hundred
// thousand steps) and kept in a small cache, so a call costs a table copy.
struct PieceKey {
  int64_t T, K, clusters, late, lag;
  bool operator==(const PieceKey& o) const {
    return T == o.T && K == o.K && clusters == o.clusters && late == o.late && lag == o.lag;
  }
};
struct PieceEntry {
  PieceKey key;
  bool ok;
  int n_tab, n_tab_early;
  uint32_t tab[kPairTabMax][3];
};
std::mutex g_piece_mu;
PieceEntry g_piece_cache[16];
int g_piece_used = 0, g_piece_next = 0;

bool plan_pair_pieces_uncached(PairParams& pp, int clusters, int64_t late, int64_t lag, int64_t T);

// T tiles (the pass's own, or the ones left after whole tiles), numbered
// from tile_offset in the table.
bool plan_pair_pieces(PairParams& pp, int clusters, int64_t late, int64_t lag, int64_t T,
                      int64_t tile_offset) {
  pp.n_tab = 0;
  const int64_t K = pp.kt_w + 2 * static_cast<int64_t>(pp.kt_b);
  if (!DORA_PIECE_TABLE || T <= 0 || K <= 0 || T >= clusters || clusters > kPairTabMax ||
      tile_offset + T > 0xFFFF)
    return false;
  auto shift = [&]() {
    for (int i = 0; i < pp.n_tab; ++i) pp.tab[i][0] += static_cast<uint32_t>(tile_offset);
  };
  if (late >= clusters || lag <= 0) late = 0;
  if (late == 0) lag = 0;
  const PieceKey key{T, K, clusters, late, lag};
  std::lock_guard<std::mutex> lk(g_piece_mu);
  for (int i = 0; i < g_piece_used; ++i) {
    const PieceEntry& e = g_piece_cache[i];
    if (e.key == key) {
      if (!e.ok) return false;
      pp.n_tab = e.n_tab;
      pp.n_tab_early = e.n_tab_early;
      std::memcpy(pp.tab, e.tab, sizeof(uint32_t) * 3 * static_cast<size_t>(e.n_tab));
      shift();
      return true;
    }
  }
  const bool ok = plan_pair_pieces_uncached(pp, clusters, late, lag, T);
  PieceEntry& e = g_piece_cache[g_piece_next];
  g_piece_next = (g_piece_next + 1) % 16;
  if (g_piece_used < 16) ++g_piece_used;
  e.key = key;
  e.ok = ok;
  e.n_tab = ok ? pp.n_tab : 0;
  e.n_tab_early = ok ? pp.n_tab_early : 0;
  if (ok) std::memcpy(e.tab, pp.tab, sizeof(uint32_t) * 3 * static_cast<size_t>(pp.n_tab));
  if (ok) shift();
  return ok;
}

bool plan_pair_pieces_uncached(PairParams& pp, int clusters, int64_t late, int64_t lag,
                               int64_t T) {
  pp.n_tab = 0;
  const int64_t K = pp.kt_w + 2 * static_cast<int64_t>(pp.kt_b);
  const int64_t ne = clusters - late;
  constexpr int64_t kNone = int64_t(1) << 40;
  int64_t best_F = -1;
  std::vector<int64_t> lmin(kMaxMainSplits + 1);
  // dp[i][e]: fewest late pieces that cut i tiles with e early pieces
  std::vector<std::vector<int64_t>> dp;
  std::vector<std::vector<int>> pick;
  // no cut has a longest early piece below the mean piece over all pairs
  const int64_t f0 = (T * K + clusters - 1) / clusters;
  for (int64_t F = f0 > 1 ? f0 : 1; F <= K && best_F < 0; ++F) {
    const int64_t Fl = late > 0 ? F - lag : 0;
    for (int e = 0; e <= kMaxMainSplits; ++e) {
      const int64_t rest = K - e * F;
      if (rest <= 0) lmin[e] = e >= 1 ? 0 : kNone;
      else lmin[e] = Fl >= 1 ? (rest + Fl - 1) / Fl : kNone;
      if (lmin[e] != kNone && e + lmin[e] > kMaxMainSplits) lmin[e] = kNone;
    }
    dp.assign(static_cast<size_t>(T + 1), std::vector<int64_t>(static_cast<size_t>(ne + 1), kNone));
    pick.assign(static_cast<size_t>(T + 1), std::vector<int>(static_cast<size_t>(ne + 1), -1));
    dp[0][0] = 0;
    for (int64_t i = 0; i < T; ++i)
      for (int64_t u = 0; u <= ne; ++u) {
        if (dp[i][u] == kNone) continue;
        for (int e = 0; e <= kMaxMainSplits && u + e <= ne; ++e) {
          if (lmin[e] == kNone) continue;
          const int64_t v = dp[i][u] + lmin[e];
          if (v < dp[i + 1][u + e]) {
            dp[i + 1][u + e] = v;
            pick[i + 1][u + e] = e;
          }
        }
      }
    for (int64_t u = 0; u <= ne; ++u)
      if (dp[T][u] <= late) {
        best_F = F;
        break;
      }
  }
  if (best_F < 0) return false;
  const int64_t F = best_F;
  // among the cuts with that F, the one with the fewest pieces (each piece
  // costs an accumulator drain and a set of partials), then the fewest late ones
  int64_t u = -1;
  for (int64_t v = ne; v >= 0; --v)
    if (dp[T][v] <= late && (u < 0 || v + dp[T][v] < u + dp[T][u])) u = v;
  std::vector<int> e_of(static_cast<size_t>(T));
  for (int64_t i = T; i > 0; --i) {
    const int e = pick[i][u];
    e_of[static_cast<size_t>(i - 1)] = e;
    u -= e;
  }
  struct Piece { int tile, split, nsplit, kb, ke; bool early; };
  std::vector<Piece> early, latep;
  for (int64_t t = 0; t < T; ++t) {
    const int e = e_of[static_cast<size_t>(t)];
    const int64_t rest = K - e * F;
    const int l = rest <= 0 ? 0 : static_cast<int>(lmin[e]);
    const int n = e + l;
    // lengths: early x, late x - lag, summing to K (x <= F by the cut rule)
    std::vector<int64_t> len(static_cast<size_t>(n));
    const int64_t tot = K + static_cast<int64_t>(l) * (late > 0 ? lag : 0);
    for (int i = 0; i < n; ++i) {
      const int64_t x = tot / n + (i < tot % n ? 1 : 0);
      len[static_cast<size_t>(i)] = i < e ? x : x - lag;
    }
    // the last late piece absorbs rounding; every piece at least one K tile
    int64_t sum = 0;
    for (int i = 0; i < n; ++i) {
      if (len[static_cast<size_t>(i)] < 1) len[static_cast<size_t>(i)] = 1;
      sum += len[static_cast<size_t>(i)];
    }
    len[static_cast<size_t>(n - 1)] += K - sum;
    if (len[static_cast<size_t>(n - 1)] < 1) return false;
    int64_t at = 0;
    for (int i = 0; i < n; ++i) {
      const int64_t ke = at + len[static_cast<size_t>(i)];
      const Piece pc{static_cast<int>(t), i, n, static_cast<int>(at), static_cast<int>(ke), i < e};
      (i < e ? early : latep).push_back(pc);
      at = ke;
    }
    if (at != K) return false;
  }
  if (early.size() + latep.size() > static_cast<size_t>(kPairTabMax)) return false;
  auto longer = [](const Piece& a, const Piece& b) {
    return a.ke - a.kb != b.ke - b.kb ? a.ke - a.kb > b.ke - b.kb : a.tile < b.tile;
  };
  std::stable_sort(early.begin(), early.end(), longer);
  std::stable_sort(latep.begin(), latep.end(), longer);
  pp.n_tab_early = static_cast<int>(early.size());
  early.insert(early.end(), latep.begin(), latep.end());
  for (size_t i = 0; i < early.size(); ++i) {
    const Piece& q = early[i];
    pp.tab[i][0] = static_cast<uint32_t>(q.tile) | static_cast<uint32_t>(q.split) << 16 |
                   static_cast<uint32_t>(q.nsplit) << 24;
    pp.tab[i][1] = static_cast<uint32_t>(q.kb);
    pp.tab[i][2] = static_cast<uint32_t>(q.ke);
  }
  pp.n_tab = static_cast<int>(early.size());
  return true;
}

// Whole tiles and a piece table, with at least as many pair tiles as pairs:
// every pair runs w = T / pairs whole pair tiles (one item each, no partial
// sums), then one piece of the R = T - w pairs tiles left over, cut by the
// piece table's dynamic program (the late pairs' pieces shorter by the lag).
// Against static ranges (one contiguous run per pair, up to three pieces
// with a drain between each), a pair changes items once.  Used when the
// remainder is at least a quarter of the pairs (a few tiles left over would
// be cut into pieces shorter than the drain they cost) and the longest pair
// is at most kWholeSlack K tiles longer than a static range.
#ifndef DORA_WHOLE_PIECES
#define DORA_WHOLE_PIECES 1
#endif
constexpr int64_t kWholeSlack = 12;

bool plan_whole_pieces(PairParams& pp, int clusters, int64_t late, int64_t lag) {
  pp.n_whole = 0;
  pp.n_tab = 0;
  const int64_t T = pp.pair_tiles;
  const int64_t K = pp.kt_w + 2 * static_cast<int64_t>(pp.kt_b);
  const int64_t n = clusters;
  if (!DORA_WHOLE_PIECES || n <= 0 || T < n || T > 0xFFFF || K <= 0) return false;
  const int64_t w = T / n, R = T - w * n;
  if (4 * R < n) return false;
  if (late >= n || lag <= 0) late = 0;
  if (late == 0) lag = 0;
  if (!plan_pair_pieces(pp, clusters, late, lag, R, w * n)) return false;
  int64_t longest = 0;
  for (int i = 0; i < pp.n_tab; ++i) {
    const int64_t len = static_cast<int64_t>(pp.tab[i][2]) - pp.tab[i][1];
    longest = len > longest ? len : longest;
  }
  const int64_t range_len = (T * K + late * lag + n - 1) / n;
  const int n_early = pp.n_tab_early, n_late = pp.n_tab - pp.n_tab_early;
  if (w * K + longest > range_len + kWholeSlack || n_early > n - n_late) {
    pp.n_tab = 0;
    return false;
  }
  // one entry per pair: the early pieces for the first pairs, the late ones
  // for the last (the pairs that start behind the Gram kernel), none between
  uint32_t tab[kPairTabMax][3];
  std::memcpy(tab, pp.tab, sizeof(tab));
  for (int c = 0; c < n; ++c) {
    const int from = c < n_early ? c : (c >= n - n_late ? n_early + (c - (static_cast<int>(n) - n_late)) : -1);
    for (int k = 0; k < 3; ++k) pp.tab[c][k] = from >= 0 ? tab[from][k] : (k == 0 ? kNoPiece : 0u);
  }
  pp.n_tab = static_cast<int>(n);
  pp.n_whole = static_cast<int>(w);
  return true;
}

// Tensor-memory layout of the main pass's accumulators (tmem_cols: the
// padded rank rounded up to a power of two, at least 32): two buffers when
// two fit in the 512 columns, so a work item's MMAs run while the previous
// item's accumulator is drained.  With one N chunk of at most 128 columns
// each buffer holds two accumulators, one for the even and one for the odd
// K steps of every tile: MMAs into the same accumulator wait for each other
// (about 110 cycles each at N <= 128, more than their math), and two chains
// halve that wait.  On one GB300, 8192 x 8192 norms back to back, timing
// only: r = 128 38.6 -> 33.5 us, r = 64 38.0 -> 32.8 us; the 196-module
// stack at r = 128 2.67 -> 2.47 ms.
void set_accumulators(PairParams& pp, uint32_t tmem_cols) {
  if (pp.n1 == 0 && tmem_cols <= 128) {
    pp.par_off = tmem_cols;
    pp.acc_stride = 2 * tmem_cols;
    pp.acc_bufs = 2;
  } else {
    pp.par_off = 0;
    pp.acc_stride = tmem_cols;
    pp.acc_bufs = 2 * tmem_cols <= 512 ? 2 : 1;
  }
  pp.tmem_cols = pp.acc_stride * static_cast<uint32_t>(pp.acc_bufs);
}

// CTAs (K splits) of the single-module Gram kernel per 128 x 128 block: a
// power of two (the 128 block rows split evenly), at most one K tile per CTA
int gram_cluster_for(int k_tiles) {
  int c = kGramCluster;
  while (c > 1 && c > k_tiles) c >>= 1;
  return c;
}

// What one main-pass launch covers: the whole norm (W tiles, then the (B, G')
// tiles, fused finalize), the partials of a d_in slice (W tiles only, the
// sums written out), or the finalize from summed partials ((B, G') tiles only).
enum PassMode { kPassFull = 0, kPassSlice = 1, kPassFinal = 2 };

// The work decomposition of a single-module bf16 main pass: N split, K tiles,
// pair tiles, K segments or static ranges.  Returns the CTA pairs to launch.
// The norm and the schedule self-test both plan through here.
int plan_main_pass(PairParams& pp, int64_t d_out, int64_t d_in, int64_t r, int clusters_max,
                   int mode = kPassFull) {
  const int rp = static_cast<int>(ceil_div(r, 16) * 16);
  pp.n0 = rp <= 256 ? rp : static_cast<int>(ceil_div(rp / 2, 16) * 16);
  pp.n1 = rp - pp.n0;
  pp.kt_w = mode == kPassFinal ? 0 : static_cast<int>(ceil_div(d_in, kTcBlockK));
  pp.kt_b = mode == kPassSlice ? 0 : static_cast<int>(ceil_div(r, kTcBlockK));
  pp.pair_tiles = static_cast<int>(ceil_div(d_out, 2 * kTcBlockM));
  if (mode == kPassFinal && pp.pair_tiles < clusters_max) {
    // only the short (B, G') range: one item per pair tile, no K split
    pp.splits = 1;
    pp.seg_k[0] = 0;
    pp.seg_k[1] = 2 * pp.kt_b;
    pp.ranges = 0;
    return pp.pair_tiles;
  }
  plan_pair_segments(pp, clusters_max);
  // the Gram kernel shares the SMs with the first pairs unless the pass
  // starts from a finished G
  const int gnb = gram_nb(rp), gcl = gram_cluster_for(pp.kt_w);
  const int gram_ctas = mode == kPassFinal ? 0 : gnb * (gnb + 1) / 2 * gcl;
  const int gram_kt = static_cast<int>(ceil_div(pp.kt_w, gcl));
  const int64_t late = gram_ctas > 0 ? (gram_ctas + 1) / 2 : 0;
  const int64_t lag = gram_ctas > 0 ? gram_lag_tiles(pp, gram_kt) : 0;
  if (plan_whole_pieces(pp, clusters_max, late, lag)) return clusters_max;
  if (plan_pair_ranges(pp, clusters_max, gram_ctas, gram_kt)) return pp.ranges;
  if (plan_pair_pieces(pp, clusters_max, late, lag, pp.pair_tiles, 0)) return pp.n_tab;
  const int items = pp.pair_tiles * pp.splits;
  return items < clusters_max ? items : clusters_max;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? DORA_OK : DORA_ERR_CUDA; }

#define DORA_TRY(expr)                       \
  do {                                       \
    const cudaError_t e_ = (expr);           \
    if (e_ != cudaSuccess) return DORA_ERR_CUDA; \
  } while (0)

// The bf16 tensor-core path of the norm in one of three modes (PassMode).
//   kPassFull: G = A A^T with G' = (s/2) G split into two bf16 terms (one
//     cluster of CTAs per upper-triangular 128 x 128 block, K split across
//     the cluster), then the CTA-pair main pass with the BA-norm tiles folded
//     into its K loop, which also finalizes every 128-row group as its last K
//     segment lands.
//   kPassSlice: the partials of a d_in slice -- G = A A^T in fp32 into
//     part_out + 2 d_out, and the main pass over the W tiles only, its fused
//     finalize writing the sums of base and cross to part_out, part_out + d_out.
//   kPassFinal: G' from the summed G of part_in + 2 d_out (split kernel), the
//     main pass over the (B, G') tiles only, its finalize adding the summed
//     base and cross of part_in ahead of its own partials.
// zero_words: the pass also zeroes the workspace's control words -- in the
// Gram kernel that heads the chain when the main pass runs a piece table
// (it touches them only after waiting for that grid), else with the
// zeroing kernel first.
int run_bf16_pass(const void* W, const void* A, const void* B, int64_t d_out, int64_t d_in,
                  int64_t r, float s, const void* m, float eps, float* wnorm, float* g,
                  const Plan& plan, uint8_t* ws, int mode, float* part_out,
                  const float* part_in, cudaStream_t stream, void* ev_begin, void* ev_end,
                  bool zero_words = false) {
  int* status = reinterpret_cast<int*>(ws + plan.off_status);
  uint16_t* Ghi = reinterpret_cast<uint16_t*>(ws + plan.off_Ghi);
  uint16_t* Glo = reinterpret_cast<uint16_t*>(ws + plan.off_Glo);
  const int rp = plan.rp;
  const int gnb = gram_nb(rp), gbw = gram_bw(rp);
  const int k_tiles = static_cast<int>(ceil_div(d_in, kTcBlockK));
  const uint32_t tmem_cols = [&] {
    uint32_t c = 32;
    while (c < static_cast<uint32_t>(rp)) c <<= 1;
    return c;
  }();
  // N split of the pair MMAs: each CTA of the pair holds half of every chunk
  const int n0 = rp <= 256 ? rp : static_cast<int>(ceil_div(rp / 2, 16) * 16);
  const int n1 = rp - n0;
  const int y_box2 = n1 > 0 ? gcd_int(n0 / 2, n1 / 2) : n0 / 2;
  CUtensorMap mW, mA_x, mA_yg, mA_y2, mB_x, mGhi, mGlo;
  // (a slice of a module without rows only has its Gram partial)
  if (d_out > 0 && !make_map_bf16(&mB_x, B, r, d_out, kTcBlockM)) return DORA_ERR_CUDA;
  if (mode != kPassFinal) {
    if ((d_out > 0 && !make_map_bf16(&mW, W, d_in, d_out, kTcBlockM)) ||
        !make_map_bf16(&mA_x, A, d_in, r, kTcBlockM) ||
        !make_map_bf16(&mA_yg, A, d_in, r, gbw) || !make_map_bf16(&mA_y2, A, d_in, r, y_box2))
      return DORA_ERR_CUDA;
  } else {
    // no W and A tiles: the kernel only prefetches these descriptors
    mW = mB_x;
  }
  if (mode != kPassSlice) {
    if (!make_map_bf16(&mGhi, Ghi, rp, rp, y_box2) || !make_map_bf16(&mGlo, Glo, rp, rp, y_box2))
      return DORA_ERR_CUDA;
  } else {
    mGhi = mA_y2;
    mGlo = mA_y2;
  }
  if (mode == kPassFinal) mA_y2 = mGhi;

  // the main pass's work decomposition (host only), planned first: with a
  // piece table it never claims from the work counter, so the Gram kernel can
  // zero the control words in place of a kernel of its own
  PairParams pp{};
  int clusters = 0;
  if (d_out > 0) {
    pp.rows = static_cast<int>(d_out);
    pp.y_box_rows = y_box2;
    pp.stages = pair_pick_stages(rp, false);
    const int clusters_max = pair_max_clusters(pair_smem_bytes(rp, pp.stages, false));
    if (clusters_max <= 0) return DORA_ERR_CUDA;
    clusters = plan_main_pass(pp, d_out, d_in, r, clusters_max, mode);
    if (pp.n0 != n0 || pp.n1 != n1) return DORA_ERR_UNSUPPORTED;
  }
  const bool gram_zeroes = zero_words && mode != kPassFinal && d_out > 0 && table_mode(pp);
  if (zero_words && !gram_zeroes)
    DORA_TRY(launch_zero_words(status, static_cast<int>(plan.zero_bytes / 4), stream));

  if (mode == kPassFinal) {
    DORA_TRY(launch_gram_split(part_in + 2 * d_out, static_cast<int>(r), rp, 0.5f * s, Ghi, Glo,
                               stream));
  } else {
    GramParams pg{};
    pg.nb = gnb;
    pg.bw = gbw;
    pg.rp = rp;
    pg.k_tiles = k_tiles;
    pg.stages = kGramStages;
    pg.cluster = gram_cluster_for(k_tiles);
    pg.tmem_cols = gbw <= 32 ? 32u : (gbw <= 64 ? 64u : 128u);
    pg.scale = mode == kPassSlice ? 1.f : 0.5f * s;
    pg.G_hi = Ghi;
    pg.G_lo = Glo;
    if (mode == kPassSlice) {
      pg.G_f32 = part_out + 2 * d_out;
      pg.r_out = static_cast<int>(r);
    }
    pg.status = status;
    pg.timeout_ns = kDefaultTimeoutNs;
    if (gram_zeroes) {
      pg.zero_p = status;
      pg.zero_n = static_cast<int>(plan.zero_bytes / 4);
    }
    DORA_TRY(launch_gram(mA_x, mA_yg, pg, stream));
  }
  if (d_out == 0) return DORA_OK;

  pp.r = static_cast<int>(r);
  set_accumulators(pp, tmem_cols);
  pp.B = static_cast<const uint16_t*>(B);
  pp.m = static_cast<const uint16_t*>(m);
  // the sum over splits of rowsum(B o D) is cross + (s/2) ba, so the
  // finalize's 2s * cross term carries the BA-norm term too
  pp.two_s = 2.f * s;
  pp.s_sq = s * s;
  pp.eps = eps;
  pp.out_sumsq = reinterpret_cast<float*>(ws + plan.off_pbase);
  pp.out_dot = reinterpret_cast<float*>(ws + plan.off_pcross);
  pp.tile_done = status + kCtlTileDone;
  pp.wnorm = wnorm;
  pp.g = g;
  if (mode == kPassSlice) {
    pp.sums_base = part_out;
    pp.sums_cross = part_out + d_out;
  } else if (mode == kPassFinal) {
    pp.ext_base = part_in;
    pp.ext_cross = part_in + d_out;
  }
  pp.work_ctr = status + kCtlWork;
  pp.status = status;
  pp.timeout_ns = kDefaultTimeoutNs;
  if (ev_begin) DORA_TRY(cudaEventRecord(static_cast<cudaEvent_t>(ev_begin), stream));
  DORA_TRY(launch_gemm_pair(mW, mA_y2, mB_x, mGhi, mGlo, pp, clusters, stream));
  if (ev_end) DORA_TRY(cudaEventRecord(static_cast<cudaEvent_t>(ev_end), stream));
  return DORA_OK;
}

// The fp32 (3xTF32) tensor-core path of the norm, in the modes of
// run_bf16_pass.  kPassFull: G = A A^T in K segments (the blocks on or above
// the block diagonal; the first CTA zeroes the control words when zero_words
// is set), their sum scaled to G' = (s/2) G, then the pair pass over (W, A)
// and (B, G') tiles in N passes of up to 256 columns; the finalize kernel
// adds the partials.  kPassSlice:
// the Gram's segments summed unscaled into part_out + 2 d_out, the pass over
// the W tiles only, the sums of its partials written to part_out.
// kPassFinal: G' = (s/2) G from part_in + 2 d_out, the pass over the (B, G')
// tiles only, and the finalize adding part_in's base and cross first.
int run_f32_pass(const void* W, const void* A, const void* B, int64_t d_out, int64_t d_in,
                 int64_t r, float s, const void* m, float eps, float* wnorm, float* g,
                 const Plan& plan, uint8_t* ws, int mode, float* part_out,
                 const float* part_in, cudaStream_t stream, void* ev_begin, void* ev_end,
                 bool zero_words = false) {
  int* status = reinterpret_cast<int*>(ws + plan.off_status);
  float* G = reinterpret_cast<float*>(ws + plan.off_G);
  float* pbase = reinterpret_cast<float*>(ws + plan.off_pbase);
  float* pcross = reinterpret_cast<float*>(ws + plan.off_pcross);
  float* Gpart = reinterpret_cast<float*>(ws + plan.off_Gpart);
  const int rp = plan.rp;
  const int passes = static_cast<int>(ceil_div(rp, 256));
  const int n_pass = static_cast<int>(ceil_div(ceil_div(rp, passes), 16) * 16);
  const int yr = n_pass / 2;
  const int clusters_max = tf32_max_clusters();
  if (clusters_max <= 0) return DORA_ERR_CUDA;
  uint32_t acc_stride = 32;
  while (acc_stride < static_cast<uint32_t>(n_pass)) acc_stride <<= 1;
  const int kt_x = mode == kPassFinal ? 0 : static_cast<int>(ceil_div(d_in, kTf32BlockK));
  CUtensorMap mW, mA_x, mA_y, mB_x, mG_y;
  // (a slice of a module without rows only has its Gram partial)
  if (d_out > 0 && !make_map_f32(&mB_x, B, r, d_out, kTcBlockM)) return DORA_ERR_CUDA;
  if (mode != kPassFinal) {
    if ((d_out > 0 && !make_map_f32(&mW, W, d_in, d_out, kTcBlockM)) ||
        !make_map_f32(&mA_x, A, d_in, r, kTcBlockM) || !make_map_f32(&mA_y, A, d_in, r, yr))
      return DORA_ERR_CUDA;
  }
  if (mode != kPassSlice) {
    if (!make_map_f32(&mG_y, G, rp, rp, yr)) return DORA_ERR_CUDA;
  } else {
    mG_y = mA_y;
  }
  if (mode == kPassFinal) {
    // no (W, A) tiles: the kernel only prefetches these descriptors
    mW = mB_x;
    mA_y = mG_y;
  }

  if (mode == kPassFinal) {
    // one "segment": G' = (s/2) G, zero padded to rp x rp
    DORA_TRY(launch_gram_tf32_reduce(part_in + 2 * d_out, 1, static_cast<int>(r), rp, 0.5f * s,
                                     G, stream));
  } else {
    Tf32Params pg{};
    pg.rows = static_cast<int>(r);
    pg.n_pass = n_pass;
    pg.passes = passes;
    pg.kt_x = kt_x;
    pg.kt_b = 0;
    pg.pair_tiles = static_cast<int>(ceil_div(r, 2 * kTcBlockM));
    {
      // G is symmetric: the blocks (256-row tile t, N pass q) whose columns
      // all lie left of the tile's first row are mirror images of computed
      // ones (8192 x 8192, r = 512: three of the four)
      int units = 0;
      for (int t = 0; t < pg.pair_tiles; ++t)
        for (int q = 0; q < passes; ++q)
          if ((q + 1) * n_pass > 2 * kTcBlockM * t) {
            pg.unit_tile[units] = t;
            pg.unit_pass[units] = q;
            ++units;
          }
      pg.n_units = units;
      // one item per CTA pair: as many K segments as fill the grid once
      int sp = clusters_max / units;
      if (sp > kTf32MaxGramSplits) sp = kTf32MaxGramSplits;
      if (sp > kt_x) sp = kt_x;
      if (sp < 1) sp = 1;
      pg.splits = sp;
      for (int i = 0; i <= sp; ++i) pg.seg_k[i] = static_cast<int>((static_cast<int64_t>(kt_x) * i) / sp);
    }
    pg.n_items = pg.n_units * pg.splits;
    pg.stages = tf32_pick_stages(n_pass);
    pg.acc_stride = acc_stride;
    pg.r = static_cast<int>(r);
    pg.out_g = Gpart;
    if (zero_words && mode == kPassFull) {
      pg.zero_p = status;
      pg.zero_n = static_cast<int>(plan.zero_bytes / 4);
    }
    pg.status = status;
    pg.timeout_ns = kDefaultTimeoutNs;
    DORA_TRY(launch_gemm_tf32(mA_x, mA_y, mA_x, mA_y, pg, true,
                              pg.n_items < clusters_max ? pg.n_items : clusters_max, stream));
    if (mode == kPassSlice) {
      // G of this slice, [r x r] unscaled and unpadded
      DORA_TRY(launch_gram_tf32_reduce(Gpart, pg.splits, static_cast<int>(r), static_cast<int>(r),
                                       1.f, part_out + 2 * d_out, stream, n_pass, 1));
    } else {
      DORA_TRY(launch_gram_tf32_reduce(Gpart, pg.splits, static_cast<int>(r), rp, 0.5f * s, G,
                                       stream, n_pass, 1));
    }
  }
  if (d_out == 0) return DORA_OK;

  Tf32Params pm{};
  pm.rows = static_cast<int>(d_out);
  pm.n_pass = n_pass;
  pm.passes = passes;
  pm.kt_x = kt_x;
  pm.kt_b = mode == kPassSlice ? 0 : static_cast<int>(ceil_div(rp, kTf32BlockK));
  pm.pair_tiles = static_cast<int>(ceil_div(d_out, 2 * kTcBlockM));
  {
    const int ktot = pm.kt_x + pm.kt_b;
    const int sp = pick_pair_splits(static_cast<int64_t>(pm.pair_tiles) * passes, ktot,
                                    clusters_max, kMaxFinalParts / passes);
    pm.splits = sp;
    for (int i = 0; i <= sp; ++i) pm.seg_k[i] = static_cast<int>((static_cast<int64_t>(ktot) * i) / sp);
  }
  pm.n_items = pm.pair_tiles * passes * pm.splits;
  pm.stages = tf32_pick_stages(n_pass);
  pm.acc_stride = acc_stride;
  pm.B = static_cast<const float*>(B);
  pm.r = static_cast<int>(r);
  pm.out_sumsq = pbase;
  pm.out_dot = pcross;
  pm.status = status;
  pm.timeout_ns = kDefaultTimeoutNs;
  if (ev_begin) DORA_TRY(cudaEventRecord(static_cast<cudaEvent_t>(ev_begin), stream));
  DORA_TRY(launch_gemm_tf32(mW, mA_y, mB_x, mG_y, pm, false,
                            pm.n_items < clusters_max ? pm.n_items : clusters_max, stream));
  if (ev_end) DORA_TRY(cudaEventRecord(static_cast<cudaEvent_t>(ev_end), stream));
  if (mode == kPassSlice)
    return cuda_status(launch_sum_partials(d_out, pbase, pm.splits, pcross, passes * pm.splits,
                                           part_out, part_out + d_out, stream));
  return cuda_status(launch_finalize(d_out, pbase, pm.splits, pcross, passes * pm.splits, nullptr,
                                     0, s, m, /*is_bf16=*/0, eps, wnorm, g, stream,
                                     mode == kPassFinal ? part_in : nullptr,
                                     mode == kPassFinal ? part_in + d_out : nullptr));
}

int factored_norm_impl(const void* W, const void* A, const void* B, int dtype, int64_t d_out,
                       int64_t d_in, int64_t r, float s, const void* m, float eps, float* wnorm,
                       float* g, void* workspace, size_t workspace_bytes, void* stream_v,
                       void* ev_begin, void* ev_end) {
  // ------------------------------------------------ host-side checks, nothing enqueued yet
  if (!shape_ok(d_out, d_in, r, dtype)) {
    if (r > DORA_MAX_RANK && d_out >= 0 && d_in >= 0) return DORA_ERR_UNSUPPORTED;
    return DORA_ERR_INVALID_ARG;
  }
  if (!std::isfinite(s) || !(eps > 0.f) || !std::isfinite(eps)) return DORA_ERR_INVALID_ARG;
  if (d_out == 0) return DORA_OK;
  const bool bf16 = dtype == DORA_BF16;
  const size_t eb = bf16 ? 2 : 4;
  const bool adapter = (r > 0) && (s != 0.f) && (d_in > 0);
  if (!m || !wnorm || !g) return DORA_ERR_INVALID_ARG;
  if (d_in > 0 && !W) return DORA_ERR_INVALID_ARG;
  if (adapter && (!A || !B)) return DORA_ERR_INVALID_ARG;
  const size_t vec_bytes = static_cast<size_t>(d_out) * 4;
  if (overlap(wnorm, vec_bytes, g, vec_bytes)) return DORA_ERR_INVALID_ARG;
  if (d_in > 0 && overlap(wnorm, vec_bytes, W, d_out * d_in * eb)) return DORA_ERR_INVALID_ARG;
  if (d_in > 0 && overlap(g, vec_bytes, W, d_out * d_in * eb)) return DORA_ERR_INVALID_ARG;
  if (overlap(wnorm, vec_bytes, m, d_out * eb) || overlap(g, vec_bytes, m, d_out * eb))
    return DORA_ERR_INVALID_ARG;
  if (d_in > 0 && ((d_in * eb) % 16 != 0 || !aligned16(W))) return DORA_ERR_UNSUPPORTED;
  if (adapter && ((r * eb) % 16 != 0 || !aligned16(A) || !aligned16(B)))
    return DORA_ERR_UNSUPPORTED;
  const Plan plan = make_plan(d_out, d_in, r, dtype);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < plan.total)
    return DORA_ERR_WORKSPACE;

  DeviceInfo dev;
  const int dst = current_device_info(&dev);
  if (dst != DORA_OK) return dst;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* status = reinterpret_cast<int*>(ws + plan.off_status);
  float* pbase = reinterpret_cast<float*>(ws + plan.off_pbase);
  float* pcross = reinterpret_cast<float*>(ws + plan.off_pcross);

  // the tensor-core passes zero the control words themselves (in their Gram
  // kernel when they can), every other path with the zeroing kernel here
  if (!(adapter && d_in > 0))
    DORA_TRY(launch_zero_words(status, static_cast<int>(plan.zero_bytes / 4), stream));

  int n_base = 0;
  if (d_in == 0) {
    // W has no columns: every term is zero.
  } else if (!adapter) {
    // s = 0 or r = 0: only the base term (Algorithm 1 notes: no U, no G).
    if (ev_begin) DORA_TRY(cudaEventRecord(static_cast<cudaEvent_t>(ev_begin), stream));
    DORA_TRY(launch_row_sumsq(W, bf16, d_out, d_in, pbase, stream));
    if (ev_end) DORA_TRY(cudaEventRecord(static_cast<cudaEvent_t>(ev_end), stream));
    n_base = 1;
  } else if (bf16) {
    return run_bf16_pass(W, A, B, d_out, d_in, r, s, m, eps, wnorm, g, plan, ws, kPassFull,
                         nullptr, nullptr, stream, ev_begin, ev_end, /*zero_words=*/true);
  } else {
    return run_f32_pass(W, A, B, d_out, d_in, r, s, m, eps, wnorm, g, plan, ws, kPassFull,
                        nullptr, nullptr, stream, ev_begin, ev_end, /*zero_words=*/true);
  }
  DORA_TRY(launch_finalize(d_out, pbase, n_base, pcross, 0, nullptr, 0, s, m, bf16, eps, wnorm,
                           g, stream));
  return DORA_OK;
}

// ---------------------------------------------------------------- d_in-sharded norm
// Floats of the partials of one d_in slice: base [d_out], cross [d_out], G [r x r].
size_t partials_floats(int64_t d_out, int64_t r) {
  return 2 * static_cast<size_t>(d_out) + static_cast<size_t>(r) * static_cast<size_t>(r);
}

int norm_partials_impl(const void* W, const void* A, const void* B, int dtype, int64_t d_out,
                       int64_t d_in, int64_t r, float* partials, void* workspace,
                       size_t workspace_bytes, void* stream_v) {
  if (!shape_ok(d_out, d_in, r, dtype)) {
    if (r > DORA_MAX_RANK && d_out >= 0 && d_in >= 0) return DORA_ERR_UNSUPPORTED;
    return DORA_ERR_INVALID_ARG;
  }
  const size_t nf = partials_floats(d_out, r);
  if (nf == 0) return DORA_OK;
  if (!partials || (reinterpret_cast<uintptr_t>(partials) & 3u) != 0) return DORA_ERR_INVALID_ARG;
  const bool bf16 = dtype == DORA_BF16;
  const size_t eb = bf16 ? 2 : 4;
  const bool has_w = d_out > 0 && d_in > 0;
  const bool has_a = r > 0 && d_in > 0;
  if (has_w && !W) return DORA_ERR_INVALID_ARG;
  if (has_a && !A) return DORA_ERR_INVALID_ARG;
  if (has_w && r > 0 && !B) return DORA_ERR_INVALID_ARG;
  const size_t pbytes = nf * 4;
  if (has_w && overlap(partials, pbytes, W, d_out * d_in * eb)) return DORA_ERR_INVALID_ARG;
  if (has_a && overlap(partials, pbytes, A, r * d_in * eb)) return DORA_ERR_INVALID_ARG;
  if (has_w && r > 0 && overlap(partials, pbytes, B, d_out * r * eb)) return DORA_ERR_INVALID_ARG;
  if (d_in > 0 && (d_in * eb) % 16 != 0) return DORA_ERR_UNSUPPORTED;
  if (has_w && !aligned16(W)) return DORA_ERR_UNSUPPORTED;
  if (has_a && ((r * eb) % 16 != 0 || !aligned16(A))) return DORA_ERR_UNSUPPORTED;
  if (has_w && r > 0 && ((r * eb) % 16 != 0 || !aligned16(B))) return DORA_ERR_UNSUPPORTED;
  const Plan plan = make_plan(d_out, d_in, r, dtype);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < plan.total)
    return DORA_ERR_WORKSPACE;

  DeviceInfo dev;
  const int dst = current_device_info(&dev);
  if (dst != DORA_OK) return dst;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  DORA_TRY(launch_zero_words(reinterpret_cast<int*>(ws + plan.off_status),
                             static_cast<int>(plan.zero_bytes / 4), stream));

  if (!has_w && !has_a) {
    // an empty slice: every partial is zero
    return cuda_status(cudaMemsetAsync(partials, 0, pbytes, stream));
  }
  if (has_a) {
    // the Gram kernel and (with rows) the main pass over the W tiles
    if (bf16)
      return run_bf16_pass(W, A, B, d_out, d_in, r, 0.f, nullptr, 1.f, nullptr, nullptr, plan, ws,
                           kPassSlice, partials, nullptr, stream, nullptr, nullptr);
    return run_f32_pass(W, A, B, d_out, d_in, r, 0.f, nullptr, 1.f, nullptr, nullptr, plan, ws,
                        kPassSlice, partials, nullptr, stream, nullptr, nullptr);
  }
  // r = 0: base only, cross = 0
  DORA_TRY(launch_row_sumsq(W, bf16, d_out, d_in, partials, stream));
  return cuda_status(cudaMemsetAsync(partials + d_out, 0, static_cast<size_t>(d_out) * 4, stream));
}

int norm_finalize_impl(const float* partials, const void* B, int dtype, int64_t d_out, int64_t r,
                       float s, const void* m, float eps, float* wnorm, float* g, void* workspace,
                       size_t workspace_bytes, void* stream_v) {
  if (!shape_ok(d_out, 0, r, dtype)) {
    if (r > DORA_MAX_RANK && d_out >= 0) return DORA_ERR_UNSUPPORTED;
    return DORA_ERR_INVALID_ARG;
  }
  if (!std::isfinite(s) || !(eps > 0.f) || !std::isfinite(eps)) return DORA_ERR_INVALID_ARG;
  if (d_out == 0) return DORA_OK;
  const bool bf16 = dtype == DORA_BF16;
  const size_t eb = bf16 ? 2 : 4;
  const bool adapter = r > 0 && s != 0.f;
  if (!partials || !m || !wnorm || !g) return DORA_ERR_INVALID_ARG;
  if (adapter && !B) return DORA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(partials) & 3u) != 0) return DORA_ERR_INVALID_ARG;
  const size_t vec_bytes = static_cast<size_t>(d_out) * 4;
  const size_t pbytes = partials_floats(d_out, r) * 4;
  if (overlap(wnorm, vec_bytes, g, vec_bytes) || overlap(wnorm, vec_bytes, partials, pbytes) ||
      overlap(g, vec_bytes, partials, pbytes) || overlap(wnorm, vec_bytes, m, d_out * eb) ||
      overlap(g, vec_bytes, m, d_out * eb))
    return DORA_ERR_INVALID_ARG;
  if (adapter && ((r * eb) % 16 != 0 || !aligned16(B))) return DORA_ERR_UNSUPPORTED;
  const Plan plan = make_plan(d_out, 0, r, dtype);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < plan.total)
    return DORA_ERR_WORKSPACE;

  DeviceInfo dev;
  const int dst = current_device_info(&dev);
  if (dst != DORA_OK) return dst;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  DORA_TRY(launch_zero_words(reinterpret_cast<int*>(ws + plan.off_status),
                             static_cast<int>(plan.zero_bytes / 4), stream));
  if (!adapter) {
    // s = 0 or r = 0: wnorm^2 = base + 2 s cross (cross is 0 for r = 0)
    return cuda_status(launch_finalize(d_out, partials, 1, partials + d_out, 1, nullptr, 0, s, m,
                                       bf16, eps, wnorm, g, stream));
  }
  if (bf16)
    return run_bf16_pass(nullptr, nullptr, B, d_out, 0, r, s, m, eps, wnorm, g, plan, ws,
                         kPassFinal, nullptr, partials, stream, nullptr, nullptr);
  return run_f32_pass(nullptr, nullptr, B, d_out, 0, r, s, m, eps, wnorm, g, plan, ws, kPassFinal,
                      nullptr, partials, stream, nullptr, nullptr);
}

// ---------------------------------------------------------------- grouped norm
// K segments of one module in a grouped launch: 3 : 2 : 1 when the K range
// allows it (the grid is filled by all modules together), else one.
void plan_module_segments(int ktot, int* seg_k, int* splits) {
  if (ktot >= 6) {
    static const int w[3] = {3, 2, 1};
    int acc = 0;
    seg_k[0] = 0;
    for (int i = 0; i < 3; ++i) {
      acc += w[i];
      seg_k[i + 1] = static_cast<int>((static_cast<int64_t>(ktot) * acc + 3) / 6);
    }
    *splits = 3;
  } else {
    seg_k[0] = 0;
    seg_k[1] = ktot;
    *splits = 1;
  }
}

struct GroupedPlan {
  bool fused = false;         // the one-launch tensor-core path
  size_t zero_bytes = 0, off_pmods = 0, off_gmods = 0, total = 0;
  std::vector<size_t> off_ghi, off_glo, off_pbase, off_pcross, off_single;
  std::vector<int> tile_done_word, splits, seg0;
};

bool grouped_fused(int dtype, int64_t r, float s) { return dtype == DORA_BF16 && r > 0 && s != 0.f; }

// Workspace of a grouped norm: the control words and the module tables of the
// one-launch path first, then either that path's per-module regions (G'
// halves, partial sums) or, for the per-module path, one dora_factored_norm
// workspace per module.  The tables come before both, so a prepared plan
// keeps them whichever path a run takes.
GroupedPlan make_grouped_plan(const dora_norm_module* mods, int n, int64_t r, int dtype,
                              bool fused) {
  GroupedPlan gp;
  gp.fused = fused;
  int words = kCtlTileDone;
  for (int i = 0; i < n; ++i) {
    gp.tile_done_word.push_back(words);
    words += 2 * static_cast<int>(ceil_div(mods[i].d_out, 2 * kTcBlockM));
  }
  size_t off = align_up(static_cast<size_t>(words) * 4, 256);
  gp.zero_bytes = off;
  gp.off_pmods = off;
  off = align_up(off + sizeof(PairModule) * n, 256);
  gp.off_gmods = off;
  off = align_up(off + sizeof(GramModule) * n, 256);
  if (!fused) {
    for (int i = 0; i < n; ++i) {
      gp.off_single.push_back(off);
      off = align_up(off + make_plan(mods[i].d_out, mods[i].d_in, r, dtype).total, 256);
    }
    gp.total = off;
    return gp;
  }
  const int rp = static_cast<int>(ceil_div(r, 16) * 16);
  const size_t rp2 = static_cast<size_t>(rp) * rp;
  for (int i = 0; i < n; ++i) {
    const int ktot = static_cast<int>(ceil_div(mods[i].d_in, kTcBlockK) + 2 * ceil_div(r, kTcBlockK));
    int seg[17], nseg = 1;
    plan_module_segments(ktot, seg, &nseg);
    gp.splits.push_back(nseg);
    gp.off_ghi.push_back(off);
    off = align_up(off + rp2 * 2, 256);
    gp.off_glo.push_back(off);
    off = align_up(off + rp2 * 2, 256);
    gp.off_pbase.push_back(off);
    off = align_up(off + static_cast<size_t>(nseg) * mods[i].d_out * 4, 256);
    gp.off_pcross.push_back(off);
    off = align_up(off + static_cast<size_t>(nseg) * mods[i].d_out * 4, 256);
  }
  gp.total = off;
  return gp;
}

// host checks of one module, as dora_factored_norm does them
int check_module(const dora_norm_module& md, int64_t r, int dtype, float s, float eps) {
  if (!shape_ok(md.d_out, md.d_in, r, dtype)) {
    if (r > DORA_MAX_RANK && md.d_out >= 0 && md.d_in >= 0) return DORA_ERR_UNSUPPORTED;
    return DORA_ERR_INVALID_ARG;
  }
  if (!std::isfinite(s) || !(eps > 0.f) || !std::isfinite(eps)) return DORA_ERR_INVALID_ARG;
  if (md.d_out == 0) return DORA_OK;
  const size_t eb = dtype == DORA_BF16 ? 2 : 4;
  const bool adapter = (r > 0) && (s != 0.f) && (md.d_in > 0);
  if (!md.m || !md.wnorm || !md.g) return DORA_ERR_INVALID_ARG;
  if (md.d_in > 0 && !md.W) return DORA_ERR_INVALID_ARG;
  if (adapter && (!md.A || !md.B)) return DORA_ERR_INVALID_ARG;
  const size_t vec_bytes = static_cast<size_t>(md.d_out) * 4;
  if (overlap(md.wnorm, vec_bytes, md.g, vec_bytes)) return DORA_ERR_INVALID_ARG;
  if (md.d_in > 0 && (overlap(md.wnorm, vec_bytes, md.W, md.d_out * md.d_in * eb) ||
                      overlap(md.g, vec_bytes, md.W, md.d_out * md.d_in * eb)))
    return DORA_ERR_INVALID_ARG;
  if (overlap(md.wnorm, vec_bytes, md.m, md.d_out * eb) || overlap(md.g, vec_bytes, md.m, md.d_out * eb))
    return DORA_ERR_INVALID_ARG;
  if (md.d_in > 0 && ((md.d_in * eb) % 16 != 0 || !aligned16(md.W))) return DORA_ERR_UNSUPPORTED;
  if (adapter && ((r * eb) % 16 != 0 || !aligned16(md.A) || !aligned16(md.B)))
    return DORA_ERR_UNSUPPORTED;
  return DORA_OK;
}

// A grouped norm prepared once: the module list, the two workspace layouts
// and, when every module can take the one-launch path, its tables written to
// the workspace.  A run then only zeroes the control words and launches.
struct NormGroupedPlan {
  std::vector<dora_norm_module> mods;
  int dtype = 0;
  int64_t r = 0;
  uint8_t* ws = nullptr;
  size_t ws_bytes = 0;
  int device = -1;
  bool tables = false;  // the one-launch tables are in the workspace
  GroupedPlan fused_gp, single_gp;
  int n_items = 0, min_kt = 0;
};

// Whether the modules can take the one-launch path for some s != 0.
bool modules_fusable(const dora_norm_module* mods, int n, int64_t r, int dtype) {
  if (!grouped_fused(dtype, r, 1.f)) return false;
  for (int i = 0; i < n; ++i) {
    const dora_norm_module& md = mods[i];
    if (md.d_out == 0 || md.d_in == 0 || !md.A || !md.B) return false;
    if (!aligned16(md.A) || !aligned16(md.B)) return false;
  }
  return true;
}

// Host checks, layouts and (with write_tables) the one-launch tables, encoded
// and copied to the workspace on `stream`.
// The work items of a grouped main pass, independent of buffers: modules in
// item order (longest K first, so that the last items the persistent grid
// takes are short ones), each with its K tiles, pair tiles, K segments and
// first item.  K segments only when the pair tiles of all modules are too
// few to fill the persistent grid a few times over; a stack of many modules
// fills it with whole-K items, each one accumulator drain.  Returns the
// number of items.
struct GroupedItems {
  int kt_w, pair_tiles, splits, item_begin;
  int seg_k[17];
};

int plan_grouped_items(int n, const int64_t* d_out, const int64_t* d_in, int64_t r,
                       int clusters_max, std::vector<int>& order, std::vector<GroupedItems>& out) {
  const int kt_b = static_cast<int>(ceil_div(r, kTcBlockK));
  int64_t total_pairs = 0;
  for (int i = 0; i < n; ++i) total_pairs += ceil_div(d_out[i], 2 * kTcBlockM);
  const bool split_k = total_pairs < 4 * static_cast<int64_t>(clusters_max);
  order.resize(static_cast<size_t>(n));
  for (int i = 0; i < n; ++i) order[static_cast<size_t>(i)] = i;
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return d_in[a] > d_in[b]; });
  out.assign(static_cast<size_t>(n), GroupedItems{});
  int item = 0;
  for (int j = 0; j < n; ++j) {
    const int i = order[static_cast<size_t>(j)];
    GroupedItems& g = out[static_cast<size_t>(j)];
    g.kt_w = static_cast<int>(ceil_div(d_in[i], kTcBlockK));
    g.pair_tiles = static_cast<int>(ceil_div(d_out[i], 2 * kTcBlockM));
    if (split_k) {
      plan_module_segments(g.kt_w + 2 * kt_b, g.seg_k, &g.splits);
    } else {
      g.seg_k[0] = 0;
      g.seg_k[1] = g.kt_w + 2 * kt_b;
      g.splits = 1;
    }
    g.item_begin = item;
    item += g.pair_tiles * g.splits;
  }
  return item;
}

int grouped_prepare(const dora_norm_module* mods, int n, int dtype, int64_t r, void* workspace,
                    size_t workspace_bytes, bool write_tables, cudaStream_t stream,
                    NormGroupedPlan* P) {
  if (n < 0 || (n > 0 && !mods)) return DORA_ERR_INVALID_ARG;
  P->mods.assign(mods, mods + n);
  P->dtype = dtype;
  P->r = r;
  P->ws = static_cast<uint8_t*>(workspace);
  P->ws_bytes = workspace_bytes;
  P->tables = false;
  if (n == 0) return DORA_OK;
  const bool fusable = modules_fusable(mods, n, r, dtype);
  P->single_gp = make_grouped_plan(mods, n, r, dtype, false);
  size_t need = P->single_gp.total;
  if (fusable) {
    P->fused_gp = make_grouped_plan(mods, n, r, dtype, true);
    if (P->fused_gp.total > need) need = P->fused_gp.total;
  }
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < need)
    return DORA_ERR_WORKSPACE;
  DORA_TRY(cudaGetDevice(&P->device));
  if (!fusable || !write_tables) return DORA_OK;

  const GroupedPlan& gp = P->fused_gp;
  uint8_t* ws = P->ws;
  int* status = reinterpret_cast<int*>(ws);
  const int rp = static_cast<int>(ceil_div(r, 16) * 16);
  const int gbw = gram_bw(rp);
  const int n0 = rp <= 256 ? rp : static_cast<int>(ceil_div(rp / 2, 16) * 16);
  const int n1 = rp - n0;
  const int y_box2 = n1 > 0 ? gcd_int(n0 / 2, n1 / 2) : n0 / 2;

  const int clusters_max =
      pair_max_clusters(pair_smem_bytes(rp, pair_pick_stages(rp, true), true));
  if (clusters_max <= 0) return DORA_ERR_CUDA;
  std::vector<int64_t> d_out(static_cast<size_t>(n)), d_in(static_cast<size_t>(n));
  for (int i = 0; i < n; ++i) {
    d_out[static_cast<size_t>(i)] = mods[i].d_out;
    d_in[static_cast<size_t>(i)] = mods[i].d_in;
  }
  std::vector<int> order;
  std::vector<GroupedItems> items;
  const int n_items = plan_grouped_items(n, d_out.data(), d_in.data(), r, clusters_max, order, items);

  std::vector<PairModule> pm(n);
  std::vector<GramModule> gm(n);
  int min_kt = 1 << 30;
  for (int j = 0; j < n; ++j) {
    const int i = order[j];
    const dora_norm_module& md = mods[i];
    uint16_t* Ghi = reinterpret_cast<uint16_t*>(ws + gp.off_ghi[i]);
    uint16_t* Glo = reinterpret_cast<uint16_t*>(ws + gp.off_glo[i]);
    PairModule& p = pm[j];
    std::memset(&p, 0, sizeof(p));
    if (!make_map_bf16(&p.tW, md.W, md.d_in, md.d_out, kTcBlockM) ||
        !make_map_bf16(&p.tA, md.A, md.d_in, r, y_box2) ||
        !make_map_bf16(&p.tB, md.B, r, md.d_out, kTcBlockM) ||
        !make_map_bf16(&p.tGhi, Ghi, rp, rp, y_box2) || !make_map_bf16(&p.tGlo, Glo, rp, rp, y_box2))
      return DORA_ERR_CUDA;
    p.B = static_cast<const uint16_t*>(md.B);
    p.m = static_cast<const uint16_t*>(md.m);
    p.wnorm = md.wnorm;
    p.g = md.g;
    p.out_sumsq = reinterpret_cast<float*>(ws + gp.off_pbase[i]);
    p.out_dot = reinterpret_cast<float*>(ws + gp.off_pcross[i]);
    p.tile_done = status + gp.tile_done_word[i];
    const GroupedItems& it = items[static_cast<size_t>(j)];
    p.rows = static_cast<int>(md.d_out);
    p.kt_w = it.kt_w;
    p.pair_tiles = it.pair_tiles;
    p.splits = it.splits;
    std::memcpy(p.seg_k, it.seg_k, sizeof(p.seg_k));
    p.item_begin = it.item_begin;
    GramModule& q = gm[i];
    std::memset(&q, 0, sizeof(q));
    if (!make_map_bf16(&q.tAx, md.A, md.d_in, r, kTcBlockM) ||
        !make_map_bf16(&q.tAy, md.A, md.d_in, r, gbw))
      return DORA_ERR_CUDA;
    q.G_hi = Ghi;
    q.G_lo = Glo;
    q.k_tiles = p.kt_w;
    if (p.kt_w < min_kt) min_kt = p.kt_w;
  }
  // pageable sources: the copies have read them when the calls return
  DORA_TRY(cudaMemcpyAsync(ws + gp.off_pmods, pm.data(), sizeof(PairModule) * n,
                           cudaMemcpyHostToDevice, stream));
  DORA_TRY(cudaMemcpyAsync(ws + gp.off_gmods, gm.data(), sizeof(GramModule) * n,
                           cudaMemcpyHostToDevice, stream));
  P->tables = true;
  P->n_items = n_items;
  P->min_kt = min_kt;
  return DORA_OK;
}

// One pass of a prepared grouped norm with these s and eps.
int grouped_run(const NormGroupedPlan& P, float s, float eps, cudaStream_t stream) {
  const int n = static_cast<int>(P.mods.size());
  const int64_t r = P.r;
  const int dtype = P.dtype;
  for (int i = 0; i < n; ++i) {
    const int st = check_module(P.mods[i], r, dtype, s, eps);
    if (st != DORA_OK) return st;
  }
  if (n == 0) return DORA_OK;
  int cur = -1;
  DORA_TRY(cudaGetDevice(&cur));
  if (cur != P.device) return DORA_ERR_INVALID_ARG;
  if (!(P.tables && grouped_fused(dtype, r, s))) {
    const GroupedPlan& gp = P.single_gp;
    for (int i = 0; i < n; ++i) {
      const dora_norm_module& md = P.mods[i];
      const int st = factored_norm_impl(md.W, md.A, md.B, dtype, md.d_out, md.d_in, r, s, md.m,
                                        eps, md.wnorm, md.g, P.ws + gp.off_single[i],
                                        P.ws_bytes - gp.off_single[i], stream, nullptr, nullptr);
      if (st != DORA_OK) return st;
    }
    return DORA_OK;
  }
  DeviceInfo dev;
  const int dst = current_device_info(&dev);
  if (dst != DORA_OK) return dst;
  const GroupedPlan& gp = P.fused_gp;
  int* status = reinterpret_cast<int*>(P.ws);
  const int rp = static_cast<int>(ceil_div(r, 16) * 16);
  const int gnb = gram_nb(rp), gbw = gram_bw(rp);
  const uint32_t tmem_cols = [&] {
    uint32_t c = 32;
    while (c < static_cast<uint32_t>(rp)) c <<= 1;
    return c;
  }();
  const int n0 = rp <= 256 ? rp : static_cast<int>(ceil_div(rp / 2, 16) * 16);
  const int n1 = rp - n0;
  const int y_box2 = n1 > 0 ? gcd_int(n0 / 2, n1 / 2) : n0 / 2;
  const int kt_b = static_cast<int>(ceil_div(r, kTcBlockK));
  const PairModule* pm_dev = reinterpret_cast<const PairModule*>(P.ws + gp.off_pmods);
  const GramModule* gm_dev = reinterpret_cast<const GramModule*>(P.ws + gp.off_gmods);
  DORA_TRY(launch_zero_words(status, static_cast<int>(gp.zero_bytes / 4), stream));

  GramParams pg{};
  pg.nb = gnb;
  pg.bw = gbw;
  pg.rp = rp;
  pg.k_tiles = P.min_kt;
  pg.stages = kGramStages;
  // Many modules fill the grid with blocks of their own: a short K split
  // (2 CTAs per block) beats the single-module choice of 8, whose per-CTA
  // setup and cluster-wide reduction then dominate (196-module stack at
  // r = 128 on one GB300: 2.87 ms per grouped norm with 1 or 2, 2.89 with 4,
  // 2.96 with 8).
  pg.cluster = kGramClusterGrouped;
  while (pg.cluster > 1 && pg.cluster > P.min_kt) pg.cluster >>= 1;
  pg.tmem_cols = gbw <= 32 ? 32u : (gbw <= 64 ? 64u : 128u);
  pg.scale = 0.5f * s;
  pg.status = status;
  pg.timeout_ns = kDefaultTimeoutNs;
  DORA_TRY(launch_gram_grouped(gm_dev, n, pg, stream));

  PairParams pp{};
  pp.n0 = n0;
  pp.n1 = n1;
  pp.y_box_rows = y_box2;
  pp.kt_b = kt_b;
  pp.stages = pair_pick_stages(rp, true);
  const int clusters_max = pair_max_clusters(pair_smem_bytes(rp, pp.stages, true));
  if (clusters_max <= 0) return DORA_ERR_CUDA;
  pp.r = static_cast<int>(r);
  set_accumulators(pp, tmem_cols);
  pp.two_s = 2.f * s;
  pp.s_sq = s * s;
  pp.eps = eps;
  pp.work_ctr = status + kCtlWork;
  pp.status = status;
  pp.timeout_ns = kDefaultTimeoutNs;
  pp.mods = pm_dev;
  pp.n_mods = n;
  pp.n_items = P.n_items;
  const int clusters = P.n_items < clusters_max ? P.n_items : clusters_max;
  DORA_TRY(launch_gemm_pair_grouped(pp, clusters, stream));
  return DORA_OK;
}

int factored_norm_grouped_impl(const dora_norm_module* mods, int n, int dtype, int64_t r, float s,
                               float eps, void* workspace, size_t workspace_bytes, void* stream_v) {
  if (n < 0 || (n > 0 && !mods)) return DORA_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) {
    const int st = check_module(mods[i], r, dtype, s, eps);
    if (st != DORA_OK) return st;
  }
  if (n == 0) return DORA_OK;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  NormGroupedPlan P;
  const int st = grouped_prepare(mods, n, dtype, r, workspace, workspace_bytes,
                                 grouped_fused(dtype, r, s), stream, &P);
  if (st != DORA_OK) return st;
  return grouped_run(P, s, eps, stream);
}

// ---------------------------------------------------------------- allocation-free variant
// Scratch of dora_factored_norm_noalloc: a file-scope device array, so callers
// that cannot allocate device memory still get a workspace.  Every device
// that loads this library holds it until the process exits.  In host code the
// name is only a stand-in for the symbol; its device address comes from
// cudaGetSymbolAddress with the caller's device current.  The address is
// looked up on every call (a host-side table lookup once the module is
// loaded), so a context torn down and created again (cudaDeviceReset) never
// leaves a stale address behind.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

int noalloc_scratch(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return DORA_ERR_CUDA;
  *out = p;
  return DORA_OK;
}

}  // namespace
}  // namespace dora

using namespace dora;

extern "C" {

size_t dora_norm_workspace_size(int64_t d_out, int64_t d_in, int64_t r, int dtype) {
  if (!shape_ok(d_out, d_in, r, dtype)) return 0;
  return make_plan(d_out, d_in, r, dtype).total;
}

int dora_factored_norm(const void* W, const void* A, const void* B, int dtype, int64_t d_out,
                       int64_t d_in, int64_t r, float s, const void* m, float eps, float* wnorm,
                       float* g, void* workspace, size_t workspace_bytes, void* stream) {
  return factored_norm_impl(W, A, B, dtype, d_out, d_in, r, s, m, eps, wnorm, g, workspace,
                            workspace_bytes, stream, nullptr, nullptr);
}

int dora_factored_norm_timed(const void* W, const void* A, const void* B, int dtype,
                             int64_t d_out, int64_t d_in, int64_t r, float s, const void* m,
                             float eps, float* wnorm, float* g, void* workspace,
                             size_t workspace_bytes, void* stream, void* ev_main_begin,
                             void* ev_main_end) {
  return factored_norm_impl(W, A, B, dtype, d_out, d_in, r, s, m, eps, wnorm, g, workspace,
                            workspace_bytes, stream, ev_main_begin, ev_main_end);
}

int dora_factored_norm_noalloc(const void* W, const void* A, const void* B, int dtype,
                               int64_t d_out, int64_t d_in, int64_t r, float s, const void* m,
                               float eps, float* wnorm, float* g, void* stream) {
  // Refuse shapes whose workspace does not fit the built-in scratch before
  // touching the device.
  if (!shape_ok(d_out, d_in, r, dtype))
    return (r > DORA_MAX_RANK && d_out >= 0 && d_in >= 0) ? DORA_ERR_UNSUPPORTED
                                                          : DORA_ERR_INVALID_ARG;
  if (make_plan(d_out, d_in, r, dtype).total > kNoAllocScratchBytes) return DORA_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int st = noalloc_scratch(&scratch);
  if (st != DORA_OK) return st;
  return factored_norm_impl(W, A, B, dtype, d_out, d_in, r, s, m, eps, wnorm, g, scratch,
                            kNoAllocScratchBytes, stream, nullptr, nullptr);
}

size_t dora_norm_partials_floats(int64_t d_out, int64_t r) {
  if (d_out < 0 || r < 0 || r > DORA_MAX_RANK || d_out >= (int64_t(1) << 31)) return 0;
  return partials_floats(d_out, r);
}

int dora_norm_partials(const void* W, const void* A, const void* B, int dtype, int64_t d_out,
                       int64_t d_in, int64_t r, float* partials, void* workspace,
                       size_t workspace_bytes, void* stream) {
  return norm_partials_impl(W, A, B, dtype, d_out, d_in, r, partials, workspace, workspace_bytes,
                            stream);
}

size_t dora_norm_finalize_workspace_size(int64_t d_out, int64_t r, int dtype) {
  if (!shape_ok(d_out, 0, r, dtype)) return 0;
  return make_plan(d_out, 0, r, dtype).total;
}

int dora_norm_finalize_partials(const float* partials, const void* B, int dtype, int64_t d_out,
                                int64_t r, float s, const void* m, float eps, float* wnorm,
                                float* g, void* workspace, size_t workspace_bytes, void* stream) {
  return norm_finalize_impl(partials, B, dtype, d_out, r, s, m, eps, wnorm, g, workspace,
                            workspace_bytes, stream);
}

int dora_compose(const void* base, const void* lora, const float* g, float s, int dtype,
                 int64_t T, int64_t d_out, void* out, void* stream) {
  if (T < 0 || d_out < 0 || (dtype != DORA_BF16 && dtype != DORA_F32) || !std::isfinite(s))
    return DORA_ERR_INVALID_ARG;
  if (T == 0 || d_out == 0) return DORA_OK;
  if (!base || !lora || !g || !out) return DORA_ERR_INVALID_ARG;
  const size_t eb = dtype == DORA_BF16 ? 2 : 4;
  const size_t nbytes = static_cast<size_t>(T) * d_out * eb;
  // in place is fine (each element is read before it is written by the same
  // thread); a partial overlap is not
  if ((out != base && overlap(out, nbytes, base, nbytes)) ||
      (out != lora && overlap(out, nbytes, lora, nbytes)))
    return DORA_ERR_INVALID_ARG;
  if (overlap(g, static_cast<size_t>(d_out) * 4, out, nbytes)) return DORA_ERR_INVALID_ARG;
  DeviceInfo dev;
  const int dst = current_device_info(&dev);
  if (dst != DORA_OK) return dst;
  return cuda_status(launch_compose(base, lora, g, s, dtype == DORA_BF16, T, d_out, out, dev.sms,
                                    static_cast<cudaStream_t>(stream)));
}

size_t dora_norm_grouped_workspace_size(const dora_norm_module* modules, int n_modules,
                                        int64_t r, int dtype) {
  if (n_modules < 0 || (n_modules > 0 && !modules)) return 0;
  bool fused = grouped_fused(dtype, r, 1.f);
  for (int i = 0; i < n_modules; ++i) {
    if (!shape_ok(modules[i].d_out, modules[i].d_in, r, dtype)) return 0;
    if (modules[i].d_out == 0 || modules[i].d_in == 0) fused = false;
  }
  // room for both layouts: s (which decides the path) is not an argument here
  const size_t a = make_grouped_plan(modules, n_modules, r, dtype, fused).total;
  const size_t b = make_grouped_plan(modules, n_modules, r, dtype, false).total;
  return a > b ? a : b;
}

int dora_factored_norm_grouped(const dora_norm_module* modules, int n_modules, int dtype,
                               int64_t r, float s, float eps, void* workspace,
                               size_t workspace_bytes, void* stream) {
  return factored_norm_grouped_impl(modules, n_modules, dtype, r, s, eps, workspace,
                                    workspace_bytes, stream);
}

struct dora_norm_grouped_plan_s {
  NormGroupedPlan plan;
};

int dora_norm_grouped_plan_create(const dora_norm_module* modules, int n_modules, int dtype,
                                  int64_t r, void* workspace, size_t workspace_bytes,
                                  void* stream, dora_norm_grouped_plan* plan) {
  if (!plan) return DORA_ERR_INVALID_ARG;
  *plan = nullptr;
  if (n_modules < 0 || (n_modules > 0 && !modules)) return DORA_ERR_INVALID_ARG;
  // the checks of a run that do not depend on s and eps (a module without
  // adapter pointers is still accepted: it runs with s = 0)
  for (int i = 0; i < n_modules; ++i) {
    const int st = check_module(modules[i], r, dtype, 0.f, 1.f);
    if (st != DORA_OK) return st;
  }
  dora_norm_grouped_plan_s* h = new (std::nothrow) dora_norm_grouped_plan_s;
  if (!h) return DORA_ERR_INVALID_ARG;
  cudaStream_t st_ = static_cast<cudaStream_t>(stream);
  int st = grouped_prepare(modules, n_modules, dtype, r, workspace, workspace_bytes, true, st_,
                           &h->plan);
  if (st == DORA_OK && n_modules > 0 && cudaStreamSynchronize(st_) != cudaSuccess) st = DORA_ERR_CUDA;
  if (st != DORA_OK) {
    delete h;
    return st;
  }
  *plan = h;
  return DORA_OK;
}

int dora_norm_grouped_plan_run(dora_norm_grouped_plan plan, float s, float eps, void* stream) {
  if (!plan) return DORA_ERR_INVALID_ARG;
  return grouped_run(plan->plan, s, eps, static_cast<cudaStream_t>(stream));
}

void dora_norm_grouped_plan_destroy(dora_norm_grouped_plan plan) { delete plan; }

size_t dora_compose_grouped_workspace_size(int n_modules) {
  if (n_modules < 0) return 0;
  return align_up(sizeof(ComposeModule) * static_cast<size_t>(n_modules), 256);
}

int dora_compose_grouped(const dora_compose_module* modules, int n_modules, float s, int dtype,
                         void* workspace, size_t workspace_bytes, void* stream) {
  if (n_modules < 0 || (n_modules > 0 && !modules) || (dtype != DORA_BF16 && dtype != DORA_F32) ||
      !std::isfinite(s))
    return DORA_ERR_INVALID_ARG;
  const size_t eb = dtype == DORA_BF16 ? 2 : 4;
  bool vec = true;
  for (int i = 0; i < n_modules; ++i) {
    const dora_compose_module& md = modules[i];
    if (md.T < 0 || md.d_out < 0) return DORA_ERR_INVALID_ARG;
    if (md.T == 0 || md.d_out == 0) continue;
    if (!md.base || !md.lora || !md.g || !md.out) return DORA_ERR_INVALID_ARG;
    const size_t nbytes = static_cast<size_t>(md.T) * md.d_out * eb;
    if ((md.out != md.base && overlap(md.out, nbytes, md.base, nbytes)) ||
        (md.out != md.lora && overlap(md.out, nbytes, md.lora, nbytes)) ||
        overlap(md.g, static_cast<size_t>(md.d_out) * 4, md.out, nbytes))
      return DORA_ERR_INVALID_ARG;
    if ((md.d_out * eb) % 16 != 0 || !aligned16(md.base) || !aligned16(md.lora) ||
        !aligned16(md.out) || !aligned16(md.g))
      vec = false;
  }
  if (n_modules == 0) return DORA_OK;
  if (!vec) {
    for (int i = 0; i < n_modules; ++i) {
      const dora_compose_module& md = modules[i];
      const int st = dora_compose(md.base, md.lora, md.g, s, dtype, md.T, md.d_out, md.out, stream);
      if (st != DORA_OK) return st;
    }
    return DORA_OK;
  }
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < dora_compose_grouped_workspace_size(n_modules))
    return DORA_ERR_WORKSPACE;
  DeviceInfo dev;
  const int dst = current_device_info(&dev);
  if (dst != DORA_OK) return dst;
  std::vector<ComposeModule> cm(n_modules);
  int64_t units = 0;
  for (int i = 0; i < n_modules; ++i) {
    const dora_compose_module& md = modules[i];
    cm[i] = ComposeModule{md.base, md.lora, md.g, md.out, md.T, md.d_out, units};
    if (md.T > 0 && md.d_out > 0) units += compose_grouped_units(md.T, md.d_out, dtype == DORA_BF16);
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  DORA_TRY(cudaMemcpyAsync(workspace, cm.data(), sizeof(ComposeModule) * n_modules,
                           cudaMemcpyHostToDevice, st));
  return cuda_status(launch_compose_grouped(static_cast<const ComposeModule*>(workspace),
                                            n_modules, units, s, dtype == DORA_BF16, dev.sms, st));
}

int dora_compose_train(const void* base, const void* lora, const float* g, float s, int dtype,
                       int64_t T, int64_t d_out, void* out, void* inner, void* stream) {
  if (T < 0 || d_out < 0 || (dtype != DORA_BF16 && dtype != DORA_F32) || !std::isfinite(s))
    return DORA_ERR_INVALID_ARG;
  if (T == 0 || d_out == 0) return DORA_OK;
  if (!base || !lora || !g || !out || !inner) return DORA_ERR_INVALID_ARG;
  const size_t eb = dtype == DORA_BF16 ? 2 : 4;
  const size_t nbytes = static_cast<size_t>(T) * d_out * eb;
  const size_t gbytes = static_cast<size_t>(d_out) * 4;
  for (const void* o : {out, inner}) {
    if (overlap(o, nbytes, base, nbytes) || overlap(o, nbytes, lora, nbytes) ||
        overlap(o, nbytes, g, gbytes))
      return DORA_ERR_INVALID_ARG;
  }
  if (overlap(out, nbytes, inner, nbytes)) return DORA_ERR_INVALID_ARG;
  DeviceInfo dev;
  const int dst = current_device_info(&dev);
  if (dst != DORA_OK) return dst;
  return cuda_status(launch_compose_train(base, lora, g, s, dtype == DORA_BF16, T, d_out, out,
                                          inner, dev.sms, static_cast<cudaStream_t>(stream)));
}

size_t dora_compose_backward_workspace_size(int64_t T, int64_t d_out) {
  if (T < 0 || d_out < 0) return 0;
  return static_cast<size_t>(compose_backward_parts(T)) * static_cast<size_t>(d_out) * 4;
}

int dora_compose_backward(const void* d_out_grad, const void* inner, const float* g,
                          const float* wnorm, float eps, float s, int dtype, int64_t T,
                          int64_t d_out, void* d_base, void* d_lora, float* dmag,
                          void* workspace, size_t workspace_bytes, void* stream) {
  if (T < 0 || d_out < 0 || (dtype != DORA_BF16 && dtype != DORA_F32) || !std::isfinite(s))
    return DORA_ERR_INVALID_ARG;
  if (T == 0 || d_out == 0) return DORA_OK;
  if (!d_out_grad || !g || !d_base || !d_lora) return DORA_ERR_INVALID_ARG;
  const size_t eb = dtype == DORA_BF16 ? 2 : 4;
  const size_t nbytes = static_cast<size_t>(T) * d_out * eb;
  const size_t vbytes = static_cast<size_t>(d_out) * 4;
  if (dmag) {
    if (!inner || !wnorm || !(eps > 0.f) || !std::isfinite(eps)) return DORA_ERR_INVALID_ARG;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 15u) != 0 ||
        workspace_bytes < dora_compose_backward_workspace_size(T, d_out))
      return DORA_ERR_WORKSPACE;
  }
  // outputs overlap nothing they are computed from, nor each other
  const void* ins[4] = {d_out_grad, g, dmag ? inner : nullptr, dmag ? wnorm : nullptr};
  const size_t in_bytes[4] = {nbytes, vbytes, nbytes, vbytes};
  const void* outs[3] = {d_base, d_lora, dmag};
  const size_t out_bytes[3] = {nbytes, nbytes, vbytes};
  for (int o = 0; o < 3; ++o) {
    if (!outs[o]) continue;
    for (int i = 0; i < 4; ++i)
      if (ins[i] && overlap(outs[o], out_bytes[o], ins[i], in_bytes[i])) return DORA_ERR_INVALID_ARG;
    for (int o2 = o + 1; o2 < 3; ++o2)
      if (outs[o2] && overlap(outs[o], out_bytes[o], outs[o2], out_bytes[o2]))
        return DORA_ERR_INVALID_ARG;
    if (dmag && overlap(outs[o], out_bytes[o], workspace, workspace_bytes))
      return DORA_ERR_INVALID_ARG;
  }
  DeviceInfo dev;
  const int dst = current_device_info(&dev);
  if (dst != DORA_OK) return dst;
  return cuda_status(launch_compose_backward(d_out_grad, inner, g, wnorm, eps, s,
                                             dtype == DORA_BF16, T, d_out, d_base, d_lora, dmag,
                                             static_cast<float*>(workspace), dev.sms,
                                             static_cast<cudaStream_t>(stream)));
}

int dora_selftest_timeout(void* workspace, size_t workspace_bytes, unsigned timeout_us,
                          void* stream) {
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < 256)
    return DORA_ERR_WORKSPACE;
  if (timeout_us == 0 || timeout_us > 1000000u) return DORA_ERR_INVALID_ARG;
  DeviceInfo dev;
  const int dst = current_device_info(&dev);
  if (dst != DORA_OK) return dst;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* status = static_cast<int*>(workspace);
  DORA_TRY(cudaMemsetAsync(status, 0, sizeof(int), st));
  return cuda_status(launch_selftest_timeout(status, 1000ull * timeout_us, st));
}

int dora_selftest_schedule(int64_t d_out, int64_t d_in, int64_t r, int clusters,
                           int* schedule, int* max_pieces, int64_t* defects) {
  if (d_out < 1 || d_in < 1 || r < 1 || r > DORA_MAX_RANK || clusters < 1 || clusters > 65535 ||
      d_out >= (int64_t(1) << 31) || d_in >= (int64_t(1) << 31) || !schedule || !max_pieces ||
      !defects)
    return DORA_ERR_INVALID_ARG;
  PairParams pp{};
  const int launch = plan_main_pass(pp, d_out, d_in, r, clusters);
  const int ktot = pp.kt_w + 2 * pp.kt_b;
  // every piece the launched pairs would run, as (kb, ke, split, nsplit) per tile
  struct Piece { int kb, ke, split, nsplit; };
  std::vector<std::vector<Piece>> tiles(static_cast<size_t>(pp.pair_tiles));
  int64_t bad = 0;
  auto add = [&](int tile, int split, int kb, int ke, int nsplit) {
    if (tile < 0 || tile >= pp.pair_tiles) { ++bad; return; }
    tiles[static_cast<size_t>(tile)].push_back(Piece{kb, ke, split, nsplit});
  };
  int tile, split, kb, ke, nsplit;
  if (pp.ranges > 0) {
    if (launch != pp.ranges) ++bad;
    for (int slot = 0; slot < pp.ranges; ++slot) {
      const int64_t lo = range_start(pp, slot);
      int64_t cur = range_start(pp, slot + 1);
      for (int64_t x; (x = range_next(pp, lo, cur)) >= 0;) {
        range_piece(pp, x, tile, split, kb, ke, nsplit);
        add(tile, split, kb, ke, nsplit);
      }
    }
  } else if (table_mode(pp)) {
    if (pp.n_tab > kPairTabMax || launch > clusters) ++bad;
    if (pp.n_whole == 0 && launch != pp.n_tab) ++bad;
    if (pp.n_whole > 0 && launch != clusters) ++bad;
    for (int c = 0; c < launch; ++c)
      for (int n = 0;; ++n) {
        const int item = table_item(pp, c, n);
        if (item < 0) break;
        table_piece(pp, item, tile, split, kb, ke, nsplit);
        add(tile, split, kb, ke, nsplit);
      }
  } else {
    if (launch < 1 || launch > clusters) ++bad;
    for (int item = 0; item < pp.pair_tiles * pp.splits; ++item) {
      segment_piece(pp.seg_k, pp.splits, pp.pair_tiles, item, tile, split, kb, ke, nsplit);
      add(tile, split, kb, ke, nsplit);
    }
  }
  // each tile: pieces that tile [0, ktot) in K order, numbered 0 .. nsplit - 1,
  // at most as many as the workspace has partial planes, every piece non-empty
  int most = 0;
  for (auto& ps : tiles) {
    std::sort(ps.begin(), ps.end(), [](const Piece& a, const Piece& b) { return a.kb < b.kb; });
    const int n = static_cast<int>(ps.size());
    most = n > most ? n : most;
    if (n == 0 || n > kMaxMainSplits) { ++bad; continue; }
    int at = 0;
    for (int i = 0; i < n; ++i) {
      const Piece& q = ps[static_cast<size_t>(i)];
      if (q.kb != at || q.ke <= q.kb || q.split != i || q.nsplit != n) ++bad;
      at = q.ke;
    }
    if (at != ktot) ++bad;
  }
  *schedule = pp.ranges > 0 ? 1 : (pp.n_whole > 0 ? 3 : (pp.n_tab > 0 ? 2 : 0));
  *max_pieces = most;
  *defects = bad;
  return DORA_OK;
}

int dora_selftest_grouped_schedule(const int64_t* d_out, const int64_t* d_in, int n_modules,
                                   int64_t r, int clusters, int* max_pieces, int64_t* defects) {
  if (!d_out || !d_in || n_modules < 1 || n_modules > (1 << 20) || r < 1 || r > DORA_MAX_RANK ||
      clusters < 1 || clusters > 65535 || !max_pieces || !defects)
    return DORA_ERR_INVALID_ARG;
  int64_t total_tiles = 0;
  for (int i = 0; i < n_modules; ++i) {
    if (d_out[i] < 1 || d_in[i] < 1 || d_out[i] >= (int64_t(1) << 31) ||
        d_in[i] >= (int64_t(1) << 31))
      return DORA_ERR_INVALID_ARG;
    total_tiles += ceil_div(d_out[i], 2 * kTcBlockM);
  }
  if (total_tiles > (int64_t(1) << 22)) return DORA_ERR_INVALID_ARG;
  std::vector<int> order;
  std::vector<GroupedItems> items;
  const int n_items = plan_grouped_items(n_modules, d_out, d_in, r, clusters, order, items);
  const int kt_b = static_cast<int>(ceil_div(r, kTcBlockK));
  int64_t bad = 0;
  // the item order: a permutation of the modules, longest K first
  std::vector<int> seen(static_cast<size_t>(n_modules), 0);
  for (int j = 0; j < n_modules; ++j) {
    const int i = order[static_cast<size_t>(j)];
    if (i < 0 || i >= n_modules || seen[static_cast<size_t>(i)]++) ++bad;
    if (j > 0 && items[static_cast<size_t>(j)].kt_w > items[static_cast<size_t>(j - 1)].kt_w) ++bad;
  }
  // every item through the kernel's own module search and segment decode
  struct Piece { int kb, ke, split, nsplit; };
  std::vector<int64_t> tile_base(static_cast<size_t>(n_modules) + 1, 0);
  for (int j = 0; j < n_modules; ++j)
    tile_base[static_cast<size_t>(j) + 1] = tile_base[static_cast<size_t>(j)] + items[static_cast<size_t>(j)].pair_tiles;
  std::vector<std::vector<Piece>> tiles(static_cast<size_t>(tile_base.back()));
  for (int item = 0; item < n_items; ++item) {
    const int j = find_module([&](int m) { return items[static_cast<size_t>(m)].item_begin; },
                              n_modules, item);
    const GroupedItems& g = items[static_cast<size_t>(j)];
    int tile, split, kb, ke, nsplit;
    segment_piece(g.seg_k, g.splits, g.pair_tiles, item - g.item_begin, tile, split, kb, ke, nsplit);
    if (tile < 0 || tile >= g.pair_tiles) { ++bad; continue; }
    tiles[static_cast<size_t>(tile_base[static_cast<size_t>(j)] + tile)].push_back(Piece{kb, ke, split, nsplit});
  }
  int most = 0;
  for (int j = 0; j < n_modules; ++j) {
    const int ktot = items[static_cast<size_t>(j)].kt_w + 2 * kt_b;
    for (int64_t t = tile_base[static_cast<size_t>(j)]; t < tile_base[static_cast<size_t>(j) + 1]; ++t) {
      auto& ps = tiles[static_cast<size_t>(t)];
      std::sort(ps.begin(), ps.end(), [](const Piece& a, const Piece& b) { return a.kb < b.kb; });
      const int np = static_cast<int>(ps.size());
      most = np > most ? np : most;
      if (np == 0 || np > kMaxMainSplits) { ++bad; continue; }
      int at = 0;
      for (int k = 0; k < np; ++k) {
        const Piece& q = ps[static_cast<size_t>(k)];
        if (q.kb != at || q.ke <= q.kb || q.split != k || q.nsplit != np) ++bad;
        at = q.ke;
      }
      if (at != ktot) ++bad;
    }
  }
  *max_pieces = most;
  *defects = bad;
  return DORA_OK;
}

int dora_check_status(const void* workspace, void* stream) {
  if (!workspace) return DORA_ERR_INVALID_ARG;
  int h = -1;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&h, workspace, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return DORA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return DORA_ERR_CUDA;
  return h;
}

const char* dora_status_string(int status) {
  switch (status) {
    case DORA_OK: return "DORA_OK";
    case DORA_ERR_INVALID_ARG: return "DORA_ERR_INVALID_ARG: invalid argument";
    case DORA_ERR_UNSUPPORTED: return "DORA_ERR_UNSUPPORTED: shape, stride or alignment not supported";
    case DORA_ERR_WORKSPACE: return "DORA_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case DORA_ERR_CUDA: return "DORA_ERR_CUDA: a CUDA call failed";
    case DORA_ERR_TIMEOUT: return "DORA_ERR_TIMEOUT: a device pipeline wait ran out of time";
    case DORA_ERR_NO_DEVICE: return "DORA_ERR_NO_DEVICE: no sm_100-family GPU is current";
    default: return "unknown dora_status";
  }
}

int dora_version(void) { return (1 << 16) | 2; }

uint64_t dora_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
