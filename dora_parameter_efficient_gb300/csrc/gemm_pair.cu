// gemm_pair.cu -- the main pass of the factored norm on CTA pairs (bf16 inputs).
//
// What it computes ("Scaling DoRA", Chinese write-up section 1.2.1 and
// Algorithm 1 of section 5.1; English summary "Factored Norm"), for every
// output row j and every split of the K range:
//
//   sumsq_j  = sum_k W_jk^2                       over the split's W columns
//   dot_j    = rowsum(B_j o D_j),  D = W A^T + (s/2) B G
//
// The BA-norm GEMM B G is folded into the same K loop: after the d_in/64 tiles
// of (W, A) come the r/64 tiles of (B, G'_hi) and of (B, G'_lo), where
// G'_hi + G'_lo = (s/2) G (two bf16 terms, computed beforehand).  Because the
// epilogue is linear in D, summing dot over the splits gives
// cross + (s/2) ba, and 2s (cross + (s/2) ba) = 2s cross + s^2 ba is exactly
// what the norm needs.  The last split of each 128-row group to finish sums
// the partials of every split in split order and assembles wnorm and g for
// those rows (the finalize of finalize.cuh): no separate kernel.
//
// Tiling for sm_103a:
//   * a cluster of 2 CTAs on 2 SMs forms one tcgen05 "CTA pair": the even CTA
//     issues tcgen05.mma.cta_group::2 with M = 256 (128 rows of W in each
//     CTA's shared memory), N = r padded to 16 (each CTA holds half of the
//     N rows of the A / G' tile), so each SM stages 16 KB of W and only half
//     of the [r x 64] A tile per K step;
//   * the accumulator D [128 x r] of each CTA lives in its own tensor memory;
//     for r <= 256 there are two of them, used by alternate work items, so
//     the MMAs of an item run while the epilogue drains the previous one;
//   * warp 0 of each CTA issues the TMA loads of its half; all loads of a
//     stage complete on the even CTA's `full` barrier; the even CTA's MMA
//     thread waits on it and, once the stage's MMAs are done, commits
//     `consumed` to both CTAs;
//   * warps 2-9 of each CTA then take the sum of squares of the stage's W
//     tile from shared memory (the bytes the MMAs just read: W leaves HBM
//     once) and release the stage to the producer (`empty`); spread over
//     the item's first tiles, each thread also fetches one 16-byte piece of
//     its B row per tile into registers, so no burst of global loads
//     competes with the TMA and MMA instructions;
//   * at the end of an item two warps per TMEM lane quadrant read the halves
//     of the D rows (tcgen05.ld, 16 columns at a time, the next load in
//     flight while the current columns are multiplied), dot them with B and
//     add the halves in a fixed order;
//   * the grid is persistent and the work is handed out dynamically: the
//     even CTA's TMA producer claims the next work item -- a (256-row tile,
//     K split) pair -- from a global counter when it has issued the loads of
//     the current one and publishes it to every role of both CTAs through a
//     small ring in shared memory.  A pair that starts late (its SMs still
//     busy with the Gram kernel, which this kernel may overlap) simply takes
//     fewer items.  Items are ordered segment-major with the K segments
//     shrinking along K, so long items go first, short ones fill in at the
//     end, and the last segment -- the one with the G' tiles -- goes last;
//   * with more pair tiles than pairs, a single-module launch uses static
//     ranges instead: the (pair tile, K tile) iterations are cut into one
//     contiguous range per pair (shorter ones for the pairs that start after
//     the Gram kernel), a pair's one atomic claim is its place in the start
//     order, and it drains its accumulator only where its range crosses a
//     tile boundary.  The ranges, so every partial sum, do not depend on
//     which pair runs which; a tile's partials are numbered in K order;
//   * the TMA producer runs ahead into the next item while the epilogue
//     drains the accumulator;
//   * W tiles are not prefetched into L2 ahead of their loads: with every
//     SM streaming W, extra prefetch requests only added traffic.
// Every wait is bounded by %globaltimer; on expiry the kernel records a
// timeout in the status word, stops issuing, drains what it issued and exits.
#include <cstring>

#include "common.cuh"
#include "finalize.cuh"
#include "ptx.cuh"

namespace dora {

namespace {

// acc + a^2 + b^2 for the two bf16 halves (a: low, b: high) of w, each step
// one mixed-precision FMA (bf16 operands, fp32 addend and result, rounded
// once): the bf16 product is exact in fp32, so each step equals
// fmaf(float(a), float(a), acc) without the two unpacking instructions
__device__ __forceinline__ float fma_sq_bf16x2(uint32_t w, float acc) {
  float r;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\t"
      "fma.rn.f32.bf16 %0, lo, lo, %2;\n\t"
      "fma.rn.f32.bf16 %0, hi, hi, %0;\n\t}"
      : "=f"(r)
      : "r"(w), "f"(acc));
  return r;
}

// Sum of squares of 8 bf16 values.
__device__ __forceinline__ float sumsq8(const uint4 v) {
  float acc = fma_sq_bf16x2(v.x, 0.f);
  acc = fma_sq_bf16x2(v.y, acc);
  acc = fma_sq_bf16x2(v.z, acc);
  return fma_sq_bf16x2(v.w, acc);
}

// Columns [c0, c0 + 8 * N) of one row of B (bf16); columns past r read as 0.
template <int N>
__device__ __forceinline__ void load_b_cols(const uint16_t* brow, int c0, int r, bool valid,
                                            uint4 (&dst)[N]) {
#pragma unroll
  for (int v = 0; v < N; ++v) {
    if (valid && c0 + v * 8 < r)
      dst[v] = __ldg(reinterpret_cast<const uint4*>(brow + c0) + v);
    else
      dst[v] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// acc += sum over 8 * N columns of B (bf16 pairs in `b`) times D (`v`)
template <int N>
__device__ __forceinline__ float dot_b(const uint4 (&b)[N], const float* v, float acc) {
#pragma unroll
  for (int q = 0; q < N; ++q) {
    const uint32_t w[4] = {b[q].x, b[q].y, b[q].z, b[q].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc = fmaf(bf16_lo(w[e]), v[q * 8 + 2 * e], acc);
      acc = fmaf(bf16_hi(w[e]), v[q * 8 + 2 * e + 1], acc);
    }
  }
  return acc;
}

// 16 bytes through the read-only path; volatile so the compiler keeps each
// load where it is written (spread over the K loop, not bunched)
__device__ __forceinline__ uint4 ldg_keep_order(const uint16_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// What a work item needs to know about its module: the kernel parameters for
// a single-module launch, one entry of the module table for a grouped one.
struct ModView {
  const CUtensorMap* tW;
  const CUtensorMap* tA;
  const CUtensorMap* tB;
  const CUtensorMap* tGhi;
  const CUtensorMap* tGlo;
  const uint16_t* B;
  const uint16_t* m;
  float* wnorm;
  float* g;
  float* out_sumsq;
  float* out_dot;
  int* tile_done;
  int rows, kt_w, pair_tiles, splits, item_begin;
  const int* seg_k;
};

__device__ __forceinline__ ModView single_view(const PairParams& p, const CUtensorMap* tW,
                                               const CUtensorMap* tA, const CUtensorMap* tB,
                                               const CUtensorMap* tGhi, const CUtensorMap* tGlo) {
  return ModView{tW, tA, tB, tGhi, tGlo, p.B, p.m, p.wnorm, p.g, p.out_sumsq, p.out_dot,
                 p.tile_done, p.rows, p.kt_w, p.pair_tiles, p.splits, 0, p.seg_k};
}

// the module of a work item in a grouped launch (modules in item order): a
// binary search over the modules' first items, read from the copy in shared
// memory (`begins`, the first kPairModCache modules) -- in global memory the
// search is a chain of dependent L2 reads that held up every item's first
// load and first MMA by a few microseconds
__device__ __forceinline__ ModView module_view(const PairParams& p, const int* begins, int item) {
  const bool cached = p.n_mods <= kPairModCache;
  const int lo = find_module(
      [&](int i) { return cached ? begins[i] : p.mods[i].item_begin; }, p.n_mods, item);
  const PairModule& md = p.mods[lo];
  return ModView{&md.tW, &md.tA, &md.tB, &md.tGhi, &md.tGlo, md.B, md.m, md.wnorm, md.g,
                 md.out_sumsq, md.out_dot, md.tile_done, md.rows, md.kt_w, md.pair_tiles,
                 md.splits, md.item_begin, md.seg_k};
}

template <bool kGrouped>
__device__ __forceinline__ ModView view_of(const PairParams& p, const ModView& single,
                                           const int* begins, int item) {
  if constexpr (kGrouped) return module_view(p, begins, item);
  else return single;
}

// Work item -> (pair tile, its K split, the split's K tile range, the number
// of splits of that tile) inside its module.
//   K segments: items are handed out segment by segment and the segments
//   shrink along K, so the long pieces of work go first and the short ones
//   fill in at the end (fewer idle pairs at the finish); the last segment
//   also holds the G' tiles.
//   Static ranges: the item is the first iteration of a piece; the pieces of
//   a tile are the ranges that meet it, numbered in K order.
//   Piece table: the item indexes a table of pieces planned on the host.
template <bool kGrouped>
__device__ __forceinline__ void item_range(const PairParams& p, const ModView& mv, int item,
                                           int& tile, int& split, int& kb, int& ke, int& nsplit) {
  if (!kGrouped && p.ranges > 0) {
    range_piece(p, item, tile, split, kb, ke, nsplit);
    return;
  }
  if (!kGrouped && table_mode(p)) {
    table_piece(p, item, tile, split, kb, ke, nsplit);
    return;
  }
  segment_piece(mv.seg_k, mv.splits, mv.pair_tiles, item - mv.item_begin, tile, split, kb, ke,
                nsplit);
}

// The completion counter of a 128-row group, incremented with acquire-release
// semantics at GPU scope by one thread after a barrier of the epilogue warps:
// the release publishes every epilogue thread's partial stores (they precede
// the barrier), the acquire orders the last segment's reads of the other
// segments' partials (after the next barrier) behind the other segments'
// releases.  No thread needs a fence of its own.
__device__ __forceinline__ int atom_add_acq_rel_gpu(int* p, int v) {
  int old;
  asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// global fp32 load that bypasses L1 (data written by other CTAs of this grid)
__device__ __forceinline__ float ld_cg_f(const float* p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
  return v;
}

// warp 0 TMA, warp 1 MMA, warps 2-9 epilogue (two per tensor-memory lane quadrant)
constexpr int kPairThreads = 320;
constexpr int kPairEpiThreads = 256;
constexpr int kPairEpiWarps = kPairEpiThreads / 32;
// work-item ring: claimed by the even CTA's producer, read by the even CTA's
// MMA thread, the odd CTA's producer and the epilogue warps of both CTAs
constexpr uint32_t kItemRing = 4;
constexpr uint32_t kItemReaders = 2 + 2 * kPairEpiWarps;

// The workspace's control words may be zeroed by the Gram kernel this grid
// depends on: a timeout is recorded in the status word only after that grid
// has finished (its own waits are bounded, so this wait ends too).
__device__ __forceinline__ void record_timeout(int* status) {
  griddep_wait();
  atomicExch(status, kStatusTimeout);
}

// The n-th work item of this CTA pair (-1: no more work), as published in the
// ring; the reader releases the slot on the even CTA's `item_empty`.
__device__ __forceinline__ int read_item(uint32_t n, uint64_t* item_full, const volatile int* item_slot,
                                         uint32_t item_empty0, uint64_t deadline, int* status,
                                         const PairParams* table) {
  // piece table: every role of both CTAs knows the pair's items (from its
  // cluster index) without the ring, so no role waits for a publication
  // across the pair
  if (table) return table_item(*table, static_cast<int>(blockIdx.x >> 1), static_cast<int>(n));
  const uint32_t slot = n % kItemRing;
  if (!mbar_wait_cluster(&item_full[slot], (n / kItemRing) & 1u, deadline)) {
    record_timeout(status);
    return -1;
  }
  const int item = item_slot[slot];
  mbar_arrive_cluster(item_empty0 + slot * 8u);
  return item;
}

// kPar (r <= 128, one N chunk): the K steps of a tile alternate between two
// accumulators -- even K steps into the buffer's first, odd ones into its
// second, p.par_off columns on -- and the epilogue adds the two.  MMAs that
// accumulate into the same tensor memory wait for each other (about 110
// cycles each at N <= 128, more than their math), so one chain of four per K
// tile set the tile rate at small ranks; two chains halve that wait.
template <bool kGrouped, bool kPar>
__global__ void __launch_bounds__(kPairThreads, 1)
    k_gemm_pair(const __grid_constant__ CUtensorMap tW, const __grid_constant__ CUtensorMap tA,
                const __grid_constant__ CUtensorMap tB, const __grid_constant__ CUtensorMap tGhi,
                const __grid_constant__ CUtensorMap tGlo, const __grid_constant__ PairParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t half_rows = static_cast<uint32_t>(p.n0 + p.n1) / 2u;
  const uint32_t stage_bytes = kTcXTileBytes + half_rows * 128u;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.stages * stage_bytes);
  uint64_t* empty = full + p.stages;
  uint64_t* consumed = empty + p.stages;
  uint64_t* accum_full = consumed + p.stages;   // [2]: one per accumulator buffer
  uint64_t* accum_empty = accum_full + 2;       // [2]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(accum_empty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  float* dot_half = reinterpret_cast<float*>(tmem_holder + 4);   // [2][128] second-half dots
  uint64_t* item_full = reinterpret_cast<uint64_t*>(dot_half + 256);
  uint64_t* item_empty = item_full + kItemRing;
  volatile int* item_slot = reinterpret_cast<volatile int*>(item_empty + kItemRing);
  volatile int* last_flag = item_slot + kItemRing;   // this CTA finished the last segment of its rows
  // grouped launch: the first item of each module (up to kPairModCache)
  int* mod_begin = reinterpret_cast<int*>(
      (reinterpret_cast<uintptr_t>(last_flag + 1) + 15) & ~static_cast<uintptr_t>(15));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();          // 0: issues the MMAs, 1: its peer
  const int n_items = kGrouped ? p.n_items : p.pair_tiles * p.splits;
  const ModView single = single_view(p, &tW, &tA, &tB, &tGhi, &tGlo);
  const uint32_t item_empty0 = map_to_rank(smem_u32(item_empty), 0);
  const uint64_t deadline = global_timer_ns() + p.timeout_ns;
  // piece table: pair c runs its n_whole whole tiles, then piece c (the table
  // lists the long pieces first, and clusters start in index order, so the
  // pairs behind the Gram kernel get the short ones): no claim on the
  // counter, and no item ring -- every role derives its items from the
  // cluster index
  const bool by_index = !kGrouped && table_mode(p);
  const PairParams* const table = by_index ? &p : nullptr;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kPairEpiWarps);   // every epilogue warp has read the W tile
      mbar_init(&consumed[s], 1);            // the stage's MMAs are done
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accum_full[b], 1);
      mbar_init(&accum_empty[b], 16);     // 8 epilogue warps in each CTA of the pair
    }
    for (uint32_t i = 0; i < kItemRing; ++i) {
      mbar_init(&item_full[i], 1);
      mbar_init(&item_empty[i], kItemReaders);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (!kGrouped && warp == 0 && lane == 0) {
    tma_prefetch_desc(&tW);
    tma_prefetch_desc(&tA);
    tma_prefetch_desc(&tB);
    tma_prefetch_desc(&tGhi);
    tma_prefetch_desc(&tGlo);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_holder, p.tmem_cols);
    tmem_relinquish_pair();
  }
  if (kGrouped && p.n_mods <= kPairModCache) {
    for (int i = threadIdx.x; i < p.n_mods; i += kPairThreads) mod_begin[i] = p.mods[i].item_begin;
  }
  tc_fence_before_sync();
  cluster_sync();          // barriers of both CTAs initialised, TMEM allocated in both
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    // -------------------------------------------------------------- TMA producer
    if (lane == 0) {
      const uint64_t pol_stream = l2_policy_evict_first();
      const uint64_t pol_keep = l2_policy_evict_last();
      const uint32_t full0 = map_to_rank(smem_u32(full), 0);
      const int h0 = p.n0 / 2, h1 = p.n1 / 2;
      const uint32_t stages = static_cast<uint32_t>(p.stages);
      // stage index and the parity of its current use, kept incrementally (a
      // runtime division per tile sits on the issuing thread's critical path)
      uint32_t s = 0, phase = 0, it = 0;
      bool stop = false;
      bool g_ready = false;      // G'_hi / G'_lo written by the preceding kernel
      const uint32_t slot1 = map_to_rank(smem_u32(const_cast<int*>(item_slot)), 1);
      const uint32_t full1 = map_to_rank(smem_u32(item_full), 1);
      int claimed = rank != 0 ? 0 : by_index ? static_cast<int>(blockIdx.x >> 1) : atomicAdd(p.work_ctr, 1);
      // static ranges: this pair's slot is its place in the start order; its
      // pieces are issued from the last to the first, so a pair's first piece
      // begins with W tiles and no pair meets a G' tile early
      int64_t range_lo = 0, range_cur = 0;
      if (!kGrouped && p.ranges > 0 && rank == 0 && claimed < p.ranges) {
        range_lo = range_start(p, claimed);
        range_cur = range_start(p, claimed + 1);
      }
      for (uint32_t n = 0; !stop; ++n) {
        int item;
        if (by_index) {
          item = read_item(n, item_full, item_slot, item_empty0, deadline, p.status, table);
        } else if (rank == 0) {
          // publish the claimed item (or the end) to both CTAs
          const uint32_t slot = n % kItemRing;
          if (n >= kItemRing &&
              !mbar_wait_cluster(&item_empty[slot], (n / kItemRing - 1) & 1u, deadline)) {
            record_timeout(p.status);
            *abort_flag = 1;
            break;
          }
          if (!kGrouped && p.ranges > 0) {
            item = static_cast<int>(range_next(p, range_lo, range_cur));
          } else {
            item = claimed < n_items ? claimed : -1;
          }
          item_slot[slot] = item;
          st_cluster_u32(slot1 + slot * 4u, static_cast<uint32_t>(item));
          mbar_arrive(&item_full[slot]);
          mbar_arrive_cluster(full1 + slot * 8u);
        } else {
          item = read_item(n, item_full, item_slot, item_empty0, deadline, p.status, table);
        }
        if (item < 0) break;
        const ModView mv = view_of<kGrouped>(p, single, mod_begin, item);
        if (kGrouped) {
          tma_prefetch_desc(mv.tW);
          tma_prefetch_desc(mv.tA);
        }
        int tile, split, kb, ke, nsplit;
        item_range<kGrouped>(p, mv, item, tile, split, kb, ke, nsplit);
        const int row0 = tile * 256 + static_cast<int>(rank) * 128;
        for (int kt = kb; kt < ke; ++kt, ++it) {
          // the slot's previous use (parity phase ^ 1) must have been consumed
          // by the MMAs and read by the epilogue warps
          if (it >= stages && !mbar_wait(&empty[s], phase ^ 1u, deadline)) {
            record_timeout(p.status);
            *abort_flag = 1;
            stop = true;
            break;
          }
          const CUtensorMap* xm;
          const CUtensorMap* ym;
          int kx;
          if (kt < mv.kt_w) {
            xm = mv.tW; ym = mv.tA; kx = kt * kTcBlockK;
          } else {
            // a G' tile (an item may start in either half of the G' range)
            if (!g_ready) {
              griddep_wait();
              g_ready = true;
            }
            xm = mv.tB;
            if (kt < mv.kt_w + p.kt_b) {
              ym = mv.tGhi; kx = (kt - mv.kt_w) * kTcBlockK;
            } else {
              ym = mv.tGlo; kx = (kt - mv.kt_w - p.kt_b) * kTcBlockK;
            }
          }
          uint8_t* xs = smem + s * stage_bytes;
          uint8_t* ys = xs + kTcXTileBytes;
          const uint32_t bar0 = full0 + s * 8u;
          if (rank == 0) mbar_arrive_expect_tx(&full[s], 2u * stage_bytes);
          tma_load_2d_pair(xs, xm, bar0, kx, row0, kt < mv.kt_w ? pol_stream : pol_keep);
          // this CTA's half of each N chunk of the Y tile
          for (int c = 0; c < h0; c += p.y_box_rows)
            tma_load_2d_pair(ys + c * 128, ym, bar0, kx, static_cast<int>(rank) * h0 + c, pol_keep);
          for (int c = 0; c < h1; c += p.y_box_rows)
            tma_load_2d_pair(ys + (h0 + c) * 128, ym, bar0, kx,
                             p.n0 + static_cast<int>(rank) * h1 + c, pol_keep);
          if (++s == stages) {
            s = 0;
            phase ^= 1u;
          }
        }
        if (rank == 0 && (kGrouped || p.ranges == 0))
          claimed = by_index ? n_items : atomicAdd(p.work_ctr, 1);
      }
      // A CTA that loaded no G' tile (every CTA for the partials of a d_in
      // slice) never waited for the Gram kernel this launch may overlap:
      // wait before exiting, so that this grid's completion covers the Gram's.
      if (!g_ready) griddep_wait();
      // The even CTA's `full` barriers count the loads of both CTAs: once the
      // last use of every stage has completed, no copy is still in flight.
      if (rank == 0) {
        const uint64_t drain_deadline = global_timer_ns() + p.timeout_ns;
        const uint32_t first = it > stages ? it - stages : 0;
        for (uint32_t i = first; i < it; ++i)
          if (!mbar_wait(&full[i % stages], (i / stages) & 1u, drain_deadline))
            record_timeout(p.status);
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer (even CTA)
    if (lane == 0 && rank == 0) {
      // Everything the issue loop needs is in registers: descriptors of stage 0
      // plus per-stage and per-K-step offsets (in the descriptors' 16-byte units).
      const uint32_t idesc0 = idesc_bf16_f32(256, p.n0);
      const uint32_t idesc1 = idesc_bf16_f32(256, p.n1 > 0 ? p.n1 : 16);
      const bool two = p.n1 > 0;
      const uint32_t nbuf = static_cast<uint32_t>(p.acc_bufs);
      const uint64_t dx0 = smem_desc_sw128(smem_u32(smem));
      const uint64_t dy0 = smem_desc_sw128(smem_u32(smem) + kTcXTileBytes);
      const uint64_t dy1_off = static_cast<uint64_t>(p.n0 / 2) * 128u >> 4;
      const uint64_t stage_step = stage_bytes >> 4;
      const uint32_t stages = static_cast<uint32_t>(p.stages);
      uint32_t s = 0, phase = 0;
      int icount = 0;
      bool stop = false;
      for (uint32_t n = 0; !stop; ++n, ++icount) {
        const int item = read_item(n, item_full, item_slot, item_empty0, deadline, p.status, table);
        if (item < 0) break;
        int tile, split, kb, ke, nsplit;
        item_range<kGrouped>(p, view_of<kGrouped>(p, single, mod_begin, item), item, tile, split, kb, ke,
                   nsplit);
        // accumulator buffer of this item, and how often it was used before
        const uint32_t buf = static_cast<uint32_t>(icount) % nbuf;
        const uint32_t use = static_cast<uint32_t>(icount) / nbuf;
        const uint32_t acc0 = tmem_base + buf * p.acc_stride;
        const uint32_t acc1 = acc0 + static_cast<uint32_t>(p.n0);
        if (use > 0 && !mbar_wait(&accum_empty[buf], (use - 1) & 1u, deadline)) {
          // the accumulator was never drained: issue nothing more
          record_timeout(p.status);
          *abort_flag = 1;
          break;
        }
        tc_fence_after_sync();
        for (int kt = kb; kt < ke; ++kt) {
          if (!mbar_wait(&full[s], phase, deadline)) {
            record_timeout(p.status);
            *abort_flag = 1;
            stop = true;
            break;
          }
          const uint64_t dx = dx0 + s * stage_step;
          const uint64_t dy = dy0 + s * stage_step;
          const uint32_t first = kt == kb ? 0u : 1u;
#pragma unroll
          for (int ks = 0; ks < kTcBlockK / 16; ++ks) {
            if constexpr (kPar) {
              // the first two K steps of an item start the two chains
              const uint32_t acc = (kt == kb && ks < 2) ? 0u : 1u;
              umma_bf16_pair(acc0 + ((ks & 1) ? p.par_off : 0u), dx + 2 * ks, dy + 2 * ks, idesc0,
                             acc);
            } else {
              const uint32_t acc = ks > 0 ? 1u : first;
              umma_bf16_pair(acc0, dx + 2 * ks, dy + 2 * ks, idesc0, acc);
              if (two) umma_bf16_pair(acc1, dx + 2 * ks, dy + dy1_off + 2 * ks, idesc1, acc);
            }
          }
          umma_commit_pair(&consumed[s], 0x3);
          if (++s == stages) {
            s = 0;
            phase ^= 1u;
          }
        }
        // both CTAs learn that this item's accumulator is complete
        umma_commit_pair(&accum_full[buf], 0x3);
      }
      // do not leave tensor-core work in flight behind the final barrier
      if (icount > 0) {
        const uint32_t last = static_cast<uint32_t>(icount - 1);
        if (!mbar_wait(&accum_full[last % nbuf], (last / nbuf) & 1u, global_timer_ns() + p.timeout_ns))
          record_timeout(p.status);
      }
    }
  } else if (warp < 2 + kPairEpiWarps) {
    // -------------------------------------------------------------- epilogue (both CTAs)
    // Warps 2-9: quadrant q = warp % 4 (the TMEM lanes = tile rows this warp
    // may read), half h = (warp - 2) / 4.  Half h owns accumulator columns
    // [h * cols0, ...) of all 32 rows of its quadrant, and the sums of
    // squares of rows 16h .. 16h + 15 of the quadrant.
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    const int trow = q * 32 + lane;
    const uint32_t tmem_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    const uint32_t accum_empty0 = map_to_rank(smem_u32(accum_empty), 0);
    const uint32_t nbuf = static_cast<uint32_t>(p.acc_bufs);
    const int nchunk = (p.r + 31) / 32;              // 32-column chunks of the accumulator
    const int c_lo = h == 0 ? 0 : (nchunk + 1) / 2;
    const int c_hi = h == 0 ? (nchunk + 1) / 2 : nchunk;
    // sum-of-squares mapping inside a stage's W tile (128 rows x 128 bytes,
    // 16-byte chunks permuted within each row by the 128-byte swizzle, which
    // a row sum does not see): one warp instruction reads 4 whole rows; lane
    // 8 * sub + chunk reads chunk `chunk` of row 32q + 16h + 4 * r4 + sub.
    // Columns and rows past the matrix were zero-filled by the TMA.
    const int sub = lane >> 3;
    const int chunk = lane & 7;
    const uint32_t x_off = static_cast<uint32_t>((q * 32 + 16 * h + sub) * 128 + chunk * 16);
    const uint32_t smem0 = smem_u32(smem);
    const uint32_t stages = static_cast<uint32_t>(p.stages);
    uint32_t s = 0, phase = 0;          // stage ring position (the producer's sequence)
    bool alive = true;                  // false once a wait has timed out
    int icount = 0;
    for (uint32_t n = 0;; ++n, ++icount) {
      int item = -1;
      if (alive && lane == 0) item = read_item(n, item_full, item_slot, item_empty0, deadline, p.status, table);
      item = __shfl_sync(0xFFFFFFFFu, item, 0);
      {
        // the 8 warps read the same item sequence; decide together anyway, as
        // they meet at named barriers (a timed-out read ends all of them)
        uint32_t all_ok;
        asm volatile(
            "{\n\t.reg .pred p, q;\n\t"
            "setp.ge.s32 p, %1, 0;\n\t"
            "bar.red.and.pred q, 1, %2, p;\n\t"
            "selp.u32 %0, 1, 0, q;\n\t}"
            : "=r"(all_ok)
            : "r"(item), "n"(kPairEpiThreads)
            : "memory");
        if (!all_ok) break;
      }
      const ModView mv = view_of<kGrouped>(p, single, mod_begin, item);
      int tile, split, kb, ke, nsplit;
      item_range<kGrouped>(p, mv, item, tile, split, kb, ke, nsplit);
      const int rowbase = tile * 256 + static_cast<int>(rank) * 128 + q * 32;
      const int grow = rowbase + lane;      // the row whose dot this lane computes
      const bool valid = grow < mv.rows;
      const uint16_t* brow = mv.B + static_cast<size_t>(valid ? grow : 0) * p.r;

      float sacc[4], scmp[4];
#pragma unroll
      for (int r4 = 0; r4 < 4; ++r4) sacc[r4] = scmp[r4] = 0.f;
      // one tile of the item: wait for its MMAs, sum squares of the W tile, release it
      auto epi_tile = [&](int kt) {
        if (alive && !mbar_wait(&consumed[s], phase, deadline)) {
          record_timeout(p.status);
          *abort_flag = 1;
          alive = false;
        }
        if (alive && kt < mv.kt_w) {
          const uint32_t xa = smem0 + s * stage_bytes + x_off;
#pragma unroll
          for (int r4 = 0; r4 < 4; ++r4) {
            uint4 v;
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                         : "r"(xa + r4 * 512u));
            kahan_add(sacc[r4], scmp[r4], sumsq8(v));
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (++s == stages) {
          s = 0;
          phase ^= 1u;
        }
      };
      // up to 192 columns of this lane's B half-row (64 with two accumulators,
      // r <= 128), two 16-byte pieces per tile
      constexpr int kBV = kPar ? 8 : 24;
      uint4 bb[kBV];
      int kt = kb;
#pragma unroll
      for (int v = 0; v < kBV; v += 2) {
        if (kt < ke) epi_tile(kt++);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int col = c_lo * 32 + (v + u) * 8;
          bb[v + u] = (valid && col < c_hi * 32 && col < p.r) ? ldg_keep_order(brow + col)
                                                              : make_uint4(0u, 0u, 0u, 0u);
        }
      }
#pragma unroll 1
      for (; kt < ke; ++kt) epi_tile(kt);

      // fold the 8 chunk lanes of each row; lane L < 16 then takes row 16h + L
      float ss = 0.f;
#pragma unroll
      for (int r4 = 0; r4 < 4; ++r4) {
        float t = __fsub_rn(sacc[r4], scmp[r4]);
        t += __shfl_xor_sync(0xFFFFFFFFu, t, 1);
        t += __shfl_xor_sync(0xFFFFFFFFu, t, 2);
        t += __shfl_xor_sync(0xFFFFFFFFu, t, 4);
        const float mine = __shfl_sync(0xFFFFFFFFu, t, (lane & 3) * 8);
        if ((lane >> 2) == r4) ss = mine;
      }
      {
        const int srow = rowbase + 16 * h + lane;
        if (lane < 16 && srow < mv.rows) mv.out_sumsq[static_cast<size_t>(split) * mv.rows + srow] = ss;
      }

      const uint32_t buf = static_cast<uint32_t>(icount) % nbuf;
      const uint32_t acc_row = tmem_row + buf * p.acc_stride;   // this item's accumulator
      bool ok = alive && mbar_wait(&accum_full[buf], (static_cast<uint32_t>(icount) / nbuf) & 1u, deadline);
      if (alive && !ok) {
        record_timeout(p.status);
        *abort_flag = 1;
      }
      tc_fence_after_sync();
      {
        // one decision for all 8 epilogue warps (they meet at named barriers below)
        uint32_t all_ok;
        asm volatile(
            "{\n\t.reg .pred p, q;\n\t"
            "setp.ne.u32 p, %1, 0;\n\t"
            "bar.red.and.pred q, 1, %2, p;\n\t"
            "selp.u32 %0, 1, 0, q;\n\t}"
            : "=r"(all_ok)
            : "r"(ok ? 1u : 0u), "n"(kPairEpiThreads)
            : "memory");
        ok = all_ok != 0;
      }
      float acc = 0.f;
      if (ok) {
        // chunks c_lo .. c_lo + 5, B held in bb; pieces at or past the padded
        // rank were never written by an MMA
        const int rp = p.n0 + p.n1;
        // 16-column pieces of this warp's half, the next one loading while
        // the current one is multiplied (columns in the same order as one
        // piece at a time, so the same sums)
        const int hc0 = 2 * c_lo;
        int nh = 2 * c_hi - hc0;
        if (nh > rp / 16 - hc0) nh = rp / 16 - hc0;
        if (nh > 12) nh = 12;
        if constexpr (kPar) {
          // two accumulators: each column is the sum of its even-K and odd-K
          // chains, added once in fp32 before the dot with B
#pragma unroll
          for (int k = 0; k < kBV / 2; ++k) {
            if (k < nh) {
              uint32_t ra[16], rb[16];
              tmem_load_16cols_async(acc_row + static_cast<uint32_t>((hc0 + k) * 16), ra);
              tmem_load_16cols_async(acc_row + p.par_off + static_cast<uint32_t>((hc0 + k) * 16), rb);
              tmem_wait_ld(ra);
              tmem_wait_ld(rb);
              float v[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) v[i] = __fadd_rn(__uint_as_float(ra[i]), __uint_as_float(rb[i]));
              const uint4 part[2] = {bb[2 * k], bb[2 * k + 1]};
              acc = dot_b<2>(part, v, acc);
            }
          }
        } else {
          uint32_t ra[16], rb[16];
          if (nh > 0) {
            tmem_load_16cols_async(acc_row + static_cast<uint32_t>(hc0 * 16), ra);
            tmem_wait_ld(ra);
          }
#pragma unroll
          for (int k = 0; k < 12; k += 2) {
            if (k < nh) {
              if (k + 1 < nh)
                tmem_load_16cols_async(acc_row + static_cast<uint32_t>((hc0 + k + 1) * 16), rb);
              float v[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(ra[i]);
              const uint4 part[2] = {bb[2 * k], bb[2 * k + 1]};
              acc = dot_b<2>(part, v, acc);
              if (k + 1 < nh) tmem_wait_ld(rb);
            }
            if (k + 1 < nh) {
              if (k + 2 < nh)
                tmem_load_16cols_async(acc_row + static_cast<uint32_t>((hc0 + k + 2) * 16), ra);
              float v[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(rb[i]);
              const uint4 part[2] = {bb[2 * k + 2], bb[2 * k + 3]};
              acc = dot_b<2>(part, v, acc);
              if (k + 2 < nh) tmem_wait_ld(ra);
            }
          }
          // ranks above 384: the rest of the half, B loaded now
          const int col_end = c_hi * 32 < rp ? c_hi * 32 : rp;
          for (int col = (c_lo + 6) * 32; col < col_end; col += 16) {
            uint4 part[2];
            load_b_cols<2>(brow, col, p.r, valid, part);
            uint32_t rv[16];
            tmem_load_16cols_async(acc_row + static_cast<uint32_t>(col), rv);
            tmem_wait_ld(rv);
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(rv[i]);
            acc = dot_b<2>(part, v, acc);
          }
        }
      }
      // accumulator drained: let the even CTA start the next item's MMAs
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(accum_empty0 + buf * 8u);
      if (!ok) break;
      // first half + second half, in that order, for each row (the halves
      // alternate between two buffers, so one barrier per item suffices)
      float* dh = dot_half + (icount & 1) * 128;
      if (h == 1) dh[trow] = acc;
      asm volatile("bar.sync 1, %0;" ::"n"(kPairEpiThreads) : "memory");
      if (h == 0 && valid) mv.out_dot[static_cast<size_t>(split) * mv.rows + grow] = acc + dh[trow];
      // the last segment of this 128-row group to finish assembles wnorm and
      // g for its rows from the partials of every segment, in segment order
      asm volatile("bar.sync 1, %0;" ::"n"(kPairEpiThreads) : "memory");
      if (warp == 2 && lane == 0) {
        // the completion counters may have been zeroed by the Gram kernel
        // this grid depends on (immediate once that grid has finished)
        griddep_wait();
        const int prev = atom_add_acq_rel_gpu(mv.tile_done + tile * 2 + static_cast<int>(rank), 1);
        *last_flag = prev == nsplit - 1 ? 1 : 0;
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kPairEpiThreads) : "memory");
      if (*last_flag && h == 0 && valid) {
        // segment partials added in segment order, carried as double-floats,
        // after the caller's summed partials of the whole d_in range (if any);
        // the first four segments' partials are loaded together (one L2
        // round trip on this item's critical tail instead of one per segment)
        df base{0.f, 0.f}, cross{0.f, 0.f};
        if (!kGrouped && p.ext_base) {
          base.hi = p.ext_base[grow];
          cross.hi = p.ext_cross[grow];
        }
        constexpr int kBatch = 4;
        float vb[kBatch], vc[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
          vb[i] = i < nsplit ? __ldcg(mv.out_sumsq + static_cast<size_t>(i) * mv.rows + grow) : 0.f;
          vc[i] = i < nsplit ? __ldcg(mv.out_dot + static_cast<size_t>(i) * mv.rows + grow) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
          if (i < nsplit) {
            float e;
            two_sum(base.hi, vb[i], base.hi, e);
            base.lo = __fadd_rn(base.lo, e);
            two_sum(cross.hi, vc[i], cross.hi, e);
            cross.lo = __fadd_rn(cross.lo, e);
          }
        }
#pragma unroll 1
        for (int i = kBatch; i < nsplit; ++i) {
          float e;
          two_sum(base.hi, ld_cg_f(mv.out_sumsq + static_cast<size_t>(i) * mv.rows + grow), base.hi, e);
          base.lo = __fadd_rn(base.lo, e);
          two_sum(cross.hi, ld_cg_f(mv.out_dot + static_cast<size_t>(i) * mv.rows + grow), cross.hi, e);
          cross.lo = __fadd_rn(cross.lo, e);
        }
        if (!kGrouped && p.sums_base) {
          // the partials of this d_in slice, rounded once to fp32
          p.sums_base[grow] = __fadd_rn(base.hi, base.lo);
          p.sums_cross[grow] = __fadd_rn(cross.hi, cross.lo);
        } else {
          float wn, gv;
          finalize_row(base, cross, nullptr, p.two_s, p.s_sq, bf16_to_f32(mv.m[grow]), p.eps, wn,
                       gv);
          mv.wnorm[grow] = wn;
          mv.g[grow] = gv;
        }
      }
    }
  }

  __syncwarp();              // whole warps at the aligned barriers below (roles ran on single lanes)
  tc_fence_before_sync();
  __syncthreads();
  // (No early trigger for the next kernel here: on one GB300 a compose
  // launched as this grid's dependent from this point ran the norm + compose
  // step 6 us slower than one launched when this grid completes.)
  cluster_sync();            // the peer may still read this CTA's shared memory until here
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, p.tmem_cols);
  }
}

}  // namespace

size_t pair_smem_bytes(int n_pad, int stages, bool grouped) {
  const size_t stage = kTcXTileBytes + static_cast<size_t>(n_pad / 2) * 128u;
  return 1024 + stage * stages + (3 * stages + 4) * 8 + 16 + 2 * 128 * 4 +
         2 * kItemRing * 8 + kItemRing * 4 + 4 + (grouped ? 16 + 4 * kPairModCache : 0);
}

int pair_pick_stages(int n_pad, bool grouped) {
  const size_t budget = 227 * 1024;
  int st = kTcMaxStages;
  while (st > 2 && pair_smem_bytes(n_pad, st, grouped) > budget) --st;
  return st;
}

// Co-resident CTA pairs.  Every shape of this kernel needs more than half of
// an SM's shared memory, so one CTA per SM and the count does not depend on
// the shape; the attribute is raised to the largest size once per device.
int pair_max_clusters(size_t smem_bytes) {
  (void)smem_bytes;
  constexpr int kMaxSmem = 227 * 1024;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  static int cached[64] = {0};
  if (dev < 64 && cached[dev]) return cached[dev];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kPairThreads, 1, 1);
  cfg.dynamicSmemBytes = kMaxSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaFuncSetAttribute(k_gemm_pair<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kMaxSmem) != cudaSuccess ||
      cudaFuncSetAttribute(k_gemm_pair<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kMaxSmem) != cudaSuccess ||
      cudaFuncSetAttribute(k_gemm_pair<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kMaxSmem) != cudaSuccess ||
      cudaFuncSetAttribute(k_gemm_pair<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kMaxSmem) != cudaSuccess ||
      cudaOccupancyMaxActiveClusters(&n, k_gemm_pair<false, false>, &cfg) != cudaSuccess)
    return 0;
  if (dev < 64) cached[dev] = n;
  return n;
}

cudaError_t launch_gemm_pair(const CUtensorMap& tW, const CUtensorMap& tA, const CUtensorMap& tB,
                             const CUtensorMap& tGhi, const CUtensorMap& tGlo, const PairParams& p,
                             int clusters, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  cfg.blockDim = dim3(kPairThreads, 1, 1);
  cfg.dynamicSmemBytes = pair_smem_bytes(p.n0 + p.n1, p.stages, false);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // may start while the Gram kernel still runs: only the TMA producer's
  // G' loads depend on it, and they wait for it (griddep_wait)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = p.par_off != 0
                      ? cudaLaunchKernelEx(&cfg, k_gemm_pair<false, true>, tW, tA, tB, tGhi, tGlo, p)
                      : cudaLaunchKernelEx(&cfg, k_gemm_pair<false, false>, tW, tA, tB, tGhi, tGlo, p);
  note_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Grouped launch: the tensor maps live in the module table (device memory);
// the kernel's map parameters are placeholders it never reads.
cudaError_t launch_gemm_pair_grouped(const PairParams& p, int clusters, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  cfg.blockDim = dim3(kPairThreads, 1, 1);
  cfg.dynamicSmemBytes = pair_smem_bytes(p.n0 + p.n1, p.stages, true);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  CUtensorMap none;
  std::memset(&none, 0, sizeof(none));
  cudaError_t e = p.par_off != 0
                      ? cudaLaunchKernelEx(&cfg, k_gemm_pair<true, true>, none, none, none, none, none, p)
                      : cudaLaunchKernelEx(&cfg, k_gemm_pair<true, false>, none, none, none, none, none, p);
  note_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dora
