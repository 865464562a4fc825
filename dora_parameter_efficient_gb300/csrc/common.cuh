// common.cuh -- shared declarations of the kernels behind the dora C ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace dora {

// device status word values (same numbers as dora_status)
constexpr int kStatusOk = 0;
constexpr int kStatusTimeout = 5;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}
// float -> bf16 bits, round to nearest even (finite inputs; NaN stays NaN)
__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return static_cast<uint16_t>((u >> 16) | 0x40u);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

// Compensated accumulation (Kahan): sum += x with the lost low part kept in c.
__device__ __forceinline__ void kahan_add(float& sum, float& c, float x) {
  const float y = __fsub_rn(x, c);
  const float t = __fadd_rn(sum, y);
  c = __fsub_rn(__fsub_rn(t, sum), y);
  sum = t;
}

// every kernel launch of the library is counted here (dora_launch_count)
void note_launches(int n);

// ------------------------------------------------------------------ Gram G = A A^T
constexpr int kTcBlockM = 128;
constexpr int kTcBlockK = 64;                 // bf16 elements per 128-byte smem row
constexpr uint32_t kTcXTileBytes = kTcBlockM * 128;
constexpr int kTcMaxStages = 8;
constexpr int kPairTabMax = 128;              // pieces of a piece-table main pass

struct GramParams {
  int nb;                // 128-row blocks per side of G (upper triangle computed)
  int bw;                // block width: 128, or the padded rank when nb == 1
  int rp;                // r padded to 16: G, G_hi, G_lo are [rp x rp]
  int k_tiles;           // 64-column tiles of d_in
  int stages;
  int cluster;           // CTAs per block (K split), one cluster per block
  uint32_t tmem_cols;
  float scale;           // G' = scale * G, split into G_hi + G_lo
  uint16_t* G_hi;
  uint16_t* G_lo;
  // partials mode: G itself (times scale) in fp32, [r_out x r_out] row-major,
  // written instead of the split (G_hi / G_lo unused)
  float* G_f32;
  int r_out;
  int* status;
  unsigned long long timeout_ns;
  // single-module launch heading the norm's chain: the first CTA zeroes these
  // control words of the workspace (status, work counter, completion
  // counters) before the main pass may launch (zero_n = 0: none)
  int* zero_p;
  int zero_n;
};

// one module of a grouped Gram launch (same rank, so the same block grid)
struct GramModule {
  CUtensorMap tAx, tAy;
  uint16_t* G_hi;
  uint16_t* G_lo;
  int k_tiles;
};

size_t gram_smem_bytes(int bw, int stages);
cudaError_t launch_gram(const CUtensorMap& tAx, const CUtensorMap& tAy, const GramParams& p,
                        cudaStream_t stream);
// grouped: p.k_tiles, p.G_hi, p.G_lo are taken from mods[]; p.cluster divides every
// module's K tiles evenly enough (<= the smallest k_tiles)
cudaError_t launch_gram_grouped(const GramModule* mods, int n_mods, const GramParams& p,
                                cudaStream_t stream);

// ------------------------------------------------------------------ CTA-pair main pass
// D [256-row pair tile x n0+n1] = X * Y^T over the K tiles of one work item,
// M = 256 per CTA pair (tcgen05 cta_group::2), persistent over items; the
// last K segment of each 128-row group to finish assembles wnorm and g for
// its rows.

// One module of a grouped launch (every module of the group has the same
// rank): its tensor maps, pointers, shape and K segments, in device memory.
struct PairModule {
  CUtensorMap tW, tA, tB, tGhi, tGlo;
  const uint16_t* B;
  const uint16_t* m;
  float* wnorm;
  float* g;
  float* out_sumsq;      // [splits][rows]
  float* out_dot;        // [splits][rows]
  int* tile_done;        // [pair_tiles][2] (zero at launch)
  int rows, kt_w, pair_tiles, splits;
  int item_begin;        // first work item of this module in the grid's item sequence
  int seg_k[17];
};

struct PairParams {
  int rows;              // d_out
  int n0, n1;            // N of the first / second MMA (n1 = 0 when r <= 256)
  int y_box_rows;        // rows per Y TMA box (divides n0/2 and n1/2)
  int kt_w;              // K tiles of (W, A)
  int kt_b;              // K tiles of (B, G'_hi), and again of (B, G'_lo)
  int splits;            // K segments per pair tile (<= 16)
  int seg_k[17];         // segment s covers K tiles [seg_k[s], seg_k[s + 1]); non-increasing lengths
  int pair_tiles;        // ceil(d_out / 256)
  int stages;
  int r;
  uint32_t tmem_cols;    // acc_bufs * acc_stride
  int acc_bufs;          // accumulator buffers (2 when two fit in the 512 TMEM columns)
  uint32_t acc_stride;   // TMEM columns per accumulator buffer
  uint32_t par_off;      // r <= 128: the odd K steps' accumulator, this many columns into
                         // the buffer (0: one accumulator per buffer)
  // epilogue and the fused finalize
  const uint16_t* B;     // [rows x r] bf16
  const uint16_t* m;     // [rows] bf16
  float two_s, s_sq, eps;
  float* out_sumsq;      // [splits][rows]
  float* out_dot;        // [splits][rows]
  int* tile_done;        // [pair_tiles][2] segments finished per 128-row group (zero at launch)
  float* wnorm;          // [rows]
  float* g;              // [rows]
  // single-module launch only (null otherwise):
  //   sums_base / sums_cross: the fused finalize writes the sums of the split
  //   partials (base = sum W^2, cross = rowsum(B o D)) here, rounded to fp32,
  //   instead of wnorm and g (the partials of a d_in slice);
  //   ext_base / ext_cross: summed partials of the whole d_in range, added
  //   ahead of the split partials before wnorm and g are assembled
  float* sums_base;
  float* sums_cross;
  const float* ext_base;
  const float* ext_cross;
  int* work_ctr;         // next unclaimed work item (or range slot); zero at launch
  int* status;
  unsigned long long timeout_ns;
  // static ranges (single-module launch, ranges != 0): the i-th CTA pair to
  // start owns iterations [S(i), S(i + 1)) of the (pair tile, K tile) space,
  // iteration = tile * ktot + K tile, S(i) = min(iters, i * len_early) for
  // i <= n_early and len_late per slot after that; a piece is the part of a
  // range inside one pair tile, and splits/seg_k are unused
  int ranges;            // CTA pairs launched (0: K segments handed out one by one)
  int ktot;              // K tiles per pair tile: kt_w + 2 * kt_b
  int iters;             // pair_tiles * ktot
  int n_early, len_early, len_late;
  // piece table (single-module launch, n_tab != 0 or n_whole != 0): pair c
  // runs n_whole whole pair tiles (c * n_whole ..), then the piece tab[c] =
  // {tile | split << 16 | nsplit << 24, kb, ke} if c < n_tab; the pieces cut
  // the tiles after the whole ones, one per pair, the long pieces first
  int n_tab;
  int n_whole;
  int n_tab_early;       // host: the table's first n_tab_early pieces are the early ones
  uint32_t tab[kPairTabMax][3];
  // grouped launch: the per-module fields above are unused, these are
  const PairModule* mods;
  int n_mods;
  int n_items;
};

// ---- work decomposition of a single-module main pass, shared by the kernel
// and the host-side schedule self-test.  One piece of work is a pair tile's
// K tiles [kb, ke); `split` numbers it among the pieces of its tile in K
// order (the plane its partial sums go to) and nsplit counts those pieces.

// Static ranges: first iteration of range slot i, and the slot whose range
// holds iteration x < iters.
__host__ __device__ inline int64_t range_start(const PairParams& p, int i) {
  const int64_t e = p.n_early;
  const int64_t v = i <= e ? i * static_cast<int64_t>(p.len_early)
                           : e * p.len_early + (i - e) * static_cast<int64_t>(p.len_late);
  return v < p.iters ? v : p.iters;
}

__host__ __device__ inline int range_of(const PairParams& p, int64_t x) {
  const int64_t head = static_cast<int64_t>(p.n_early) * p.len_early;
  return x < head ? static_cast<int>(x / p.len_early)
                  : p.n_early + static_cast<int>((x - head) / p.len_late);
}

// Static ranges: the piece that starts at iteration x.
__host__ __device__ inline void range_piece(const PairParams& p, int64_t x, int& tile, int& split,
                                            int& kb, int& ke, int& nsplit) {
  tile = static_cast<int>(x / p.ktot);
  const int64_t t0 = static_cast<int64_t>(tile) * p.ktot;
  const int c = range_of(p, x);
  const int64_t end = range_start(p, c + 1);
  const int c0 = range_of(p, t0);
  kb = static_cast<int>(x - t0);
  ke = end < t0 + p.ktot ? static_cast<int>(end - t0) : p.ktot;
  split = c - c0;
  nsplit = range_of(p, t0 + p.ktot - 1) - c0 + 1;
}

// Static ranges: the first iteration of the next piece a pair issues from
// its range [lo, cur), the last piece first (cur moves down to it), or -1.
__host__ __device__ inline int64_t range_next(const PairParams& p, int64_t lo, int64_t& cur) {
  if (cur <= lo) return -1;
  const int64_t t0 = (cur - 1) / p.ktot * p.ktot;
  cur = t0 > lo ? t0 : lo;
  return cur;
}

// Piece table: the n-th work item of pair c (its whole tiles first, then its
// piece), or -1.  A whole tile is an item with kWholeItem set.
constexpr int kWholeItem = 1 << 30;
__host__ __device__ inline bool table_mode(const PairParams& p) { return p.n_tab > 0 || p.n_whole > 0; }
constexpr uint32_t kNoPiece = 0xFFFFFFFFu;     // a table entry of a pair without a piece
__host__ __device__ inline int table_item(const PairParams& p, int c, int n) {
  if (n < p.n_whole) return kWholeItem | (c * p.n_whole + n);
  if (n == p.n_whole && c < p.n_tab && p.tab[c][0] != kNoPiece) return c;
  return -1;
}

// Piece table: work item -> its piece.
__host__ __device__ inline void table_piece(const PairParams& p, int item, int& tile, int& split,
                                            int& kb, int& ke, int& nsplit) {
  if (item & kWholeItem) {
    tile = item & (kWholeItem - 1);
    split = 0;
    nsplit = 1;
    kb = 0;
    ke = p.kt_w + 2 * p.kt_b;
    return;
  }
  const uint32_t w = p.tab[item][0];
  tile = static_cast<int>(w & 0xFFFFu);
  split = static_cast<int>((w >> 16) & 0xFFu);
  nsplit = static_cast<int>(w >> 24);
  kb = static_cast<int>(p.tab[item][1]);
  ke = static_cast<int>(p.tab[item][2]);
}

// K segments: work item -> its piece (items segment-major: every tile's
// first segment, then every tile's second, ...).
__host__ __device__ inline void segment_piece(const int* seg_k, int splits, int pair_tiles,
                                              int item, int& tile, int& split, int& kb, int& ke,
                                              int& nsplit) {
  split = item / pair_tiles;
  tile = item - split * pair_tiles;
  kb = seg_k[split];
  ke = seg_k[split + 1];
  nsplit = splits;
}

// Grouped launch: the module whose items hold `item`, by binary search over
// the modules' first items (begin(i), non-decreasing, begin(0) = 0).
template <class Begin>
__host__ __device__ inline int find_module(Begin begin, int n, int item) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (begin(mid) <= item) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// modules of a grouped launch whose first item is kept in shared memory
constexpr int kPairModCache = 2048;
size_t pair_smem_bytes(int n_pad, int stages, bool grouped);
int pair_pick_stages(int n_pad, bool grouped);
int pair_max_clusters(size_t smem_bytes);
cudaError_t launch_gemm_pair(const CUtensorMap& tW, const CUtensorMap& tA, const CUtensorMap& tB,
                             const CUtensorMap& tGhi, const CUtensorMap& tGlo, const PairParams& p,
                             int clusters, cudaStream_t stream);
cudaError_t launch_gemm_pair_grouped(const PairParams& p, int clusters, cudaStream_t stream);

// ------------------------------------------------------------------ fp32 inputs: 3xTF32 pair pass
// D [256-row pair tile x one N pass] = X * Y^T over the K tiles (32 fp32 each)
// of one work item, every product as x_hi y_hi + x_lo y_hi + x_hi y_lo.
// Work items (pair tile, N pass, K segment) are striped over the grid.
constexpr int kTf32BlockK = 32;               // fp32 elements per 128-byte smem row
constexpr int kTf32MaxGramSplits = 24;        // K segments of the fp32 Gram (workspace)

struct Tf32Params {
  int rows;              // rows of X: d_out (norm) or r (Gram)
  int n_pass;            // N of one pass (multiple of 16, <= 256)
  int passes;            // N passes: cover the padded rank
  int kt_x;              // K tiles of (X, Y)
  int kt_b;              // K tiles of (B, G') that follow them (norm); 0 for the Gram
  int splits;            // K segments
  int seg_k[kTf32MaxGramSplits + 1];   // segment s covers K tiles [seg_k[s], seg_k[s + 1]), none empty
  int pair_tiles;        // ceil(rows / 256)
  int n_items;           // pair_tiles * passes * splits
  int stages;
  uint32_t acc_stride;   // TMEM columns per accumulator buffer (two buffers)
  // norm
  const float* B;        // [rows x r]
  int r;
  float* out_sumsq;      // [splits][rows], written by pass-0 items
  float* out_dot;        // [passes * splits][rows], part pass * splits + split
  // Gram
  float* out_g;          // [splits][rows][r] partial G
  // blocks (pair tile, N pass) computed, n_units of them (0: all); G is
  // symmetric, so those strictly below the block diagonal are left out
  int n_units;
  int unit_tile[4], unit_pass[4];
  int* zero_p;           // control words this launch zeroes first (heading a norm), or null
  int zero_n;
  int* status;
  unsigned long long timeout_ns;
};

size_t tf32_smem_bytes(int n_pass, int stages);
int tf32_pick_stages(int n_pass);
int tf32_max_clusters();
// store = false: the norm pass (X = W then B, Y = A then G'); true: the Gram (X = Y = A)
cudaError_t launch_gemm_tf32(const CUtensorMap& tX, const CUtensorMap& tY, const CUtensorMap& tXb,
                             const CUtensorMap& tYb, const Tf32Params& p, bool store,
                             int clusters, cudaStream_t stream);
// G' [rp x rp] = scale * (sum over the splits of the partials, in split order); zero
// outside [r x r].  sym: the partials hold only the blocks (256-row tile, n_pass-column
// pass) on or above the block diagonal; the others are written as mirror images.
cudaError_t launch_gram_tf32_reduce(const float* parts, int splits, int r, int rp, float scale,
                                    float* Gp, cudaStream_t stream, int n_pass = 0,
                                    int sym = 0);

// ------------------------------------------------------------------ small kernels
// zeroes n ints at p (a norm workspace's control block); the next kernel may
// be launched as its programmatic dependent
cudaError_t launch_zero_words(int* p, int n, cudaStream_t stream);
cudaError_t launch_selftest_timeout(int* status, unsigned long long timeout_ns,
                                    cudaStream_t stream);
cudaError_t launch_row_sumsq(const void* X, int is_bf16, int64_t rows, int64_t cols,
                             float* out, cudaStream_t stream);
cudaError_t launch_finalize(int64_t d_out, const float* pbase, int n_base, const float* pcross,
                            int n_cross, const float* pba, int n_ba, float s, const void* m,
                            int is_bf16, float eps, float* wnorm, float* g,
                            cudaStream_t stream, const float* ext_base = nullptr,
                            const float* ext_cross = nullptr);
// the sums of the split partials (base and cross, in split order) rounded to
// fp32, written to sum_base / sum_cross: the partials of a d_in slice
cudaError_t launch_sum_partials(int64_t d_out, const float* pbase, int n_base,
                                const float* pcross, int n_cross, float* sum_base,
                                float* sum_cross, cudaStream_t stream);
// G' = scale * G [r x r] fp32 split into bf16 G'_hi + G'_lo [rp x rp], zero padded
cudaError_t launch_gram_split(const float* G, int r, int rp, float scale, uint16_t* G_hi,
                              uint16_t* G_lo, cudaStream_t stream);
cudaError_t launch_compose(const void* base, const void* lora, const float* g, float s,
                           int is_bf16, int64_t T, int64_t d_out, void* out, int num_sms,
                           cudaStream_t stream);

// one module of a grouped compose (device memory)
struct ComposeModule {
  const void* base;
  const void* lora;
  const float* g;
  void* out;
  int64_t T, d_out;
  int64_t unit_begin;    // first work unit of this module
};
int64_t compose_grouped_units(int64_t T, int64_t d_out, int is_bf16);
cudaError_t launch_compose_grouped(const ComposeModule* mods, int n_mods, int64_t n_units,
                                   float s, int is_bf16, int num_sms, cudaStream_t stream);

// ------------------------------------------------------------------ training path of the compose
constexpr int64_t kMaxDmParts = 256;   // row blocks of the magnitude-gradient column sums
int64_t compose_backward_parts(int64_t T);
cudaError_t launch_compose_train(const void* base, const void* lora, const float* g, float s,
                                 int is_bf16, int64_t T, int64_t d_out, void* out, void* inner,
                                 int num_sms, cudaStream_t stream);
cudaError_t launch_compose_backward(const void* dout, const void* inner, const float* g,
                                    const float* wnorm, float eps, float s, int is_bf16,
                                    int64_t T, int64_t d_out, void* d_base, void* d_lora,
                                    float* dmag, float* partials, int num_sms,
                                    cudaStream_t stream);

}  // namespace dora
