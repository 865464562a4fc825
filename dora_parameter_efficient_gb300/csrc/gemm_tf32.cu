// gemm_tf32.cu -- the factored norm's GEMMs for fp32 inputs on the tensor
// cores ("Scaling DoRA", Chinese write-up sections 1.2.1 and 1.2.2 and
// Algorithm 1 of section 5.1: U = W A^T, G = A A^T and rowsum(B o (B G)),
// fp32 inputs accumulated in fp32).
//
// Precision.  The tensor cores multiply TF32 values: from an fp32 container
// they take the sign, the exponent and the top 10 fraction bits and ignore
// the low 13.  So the fp32 tile as loaded serves as hi = trunc_tf32(v), and
// the split warps write lo = v - hi (exact in fp32, |lo| < 2^-10 |v|) to a
// second tile; every product is taken as x_hi y_hi + x_lo y_hi + x_hi y_lo
// on kind::tf32 MMAs with fp32 accumulation -- the usual "3xTF32" scheme.
// The tensor core reads lo in turn to TF32 (an error below 2^-10 |lo|), and
// the dropped x_lo y_lo is below 2^-20 of the product, so each product is
// good to a few units of 2^-20.  Small integers split into hi = v, lo = 0,
// so integer-valued inputs still give exact results.  The sum of squares of
// W is taken on the CUDA cores from the raw fp32 tile, compensated across
// tiles.
//
// Two modes (template argument kStore):
//   * norm: for each row j of W and each work item (pair tile, N pass, K
//     segment), dot_j = rowsum(B_j o D_j) over the pass's columns, with
//     D = W A^T followed in K by B G', G' = (s/2) G, so the sum over the
//     items is cross + (s/2) ba, exactly as in the bf16 pass; items of N pass
//     0 also write the segment's sum of squares.  A separate finalize adds
//     the partials in a fixed order;
//   * Gram: D = A A^T over the item's K range, stored as an fp32 partial; a
//     reduce kernel adds the segments in order and scales by s/2.  G is
//     symmetric: only the (256-row tile, N pass) blocks on or above the block
//     diagonal are computed, and the reduce writes the others as mirror images.
//
// Tiling for sm_103a: CTA pairs (clusters of 2, tcgen05 cta_group::2), M = 256
// rows of X per pair (128 in each CTA), N = one pass of at most 256 columns
// (each CTA holds half of the pass's Y rows), K = 32 fp32 -- one 128-byte
// swizzled row -- per pipeline stage.  Two rings of shared-memory slots: raw
// slots receive the TMA loads, split slots hold the four TF32 operand tiles
// the MMAs read.  Per stage and CTA:
//   * warp 0 loads its X tile and its half of the Y tile (TMA) into a raw
//     slot and counts the bytes on its own `raw_full` barrier;
//   * warps 2-17 read the raw slot, write x_lo and y_lo into a split slot,
//     take the sum of squares of X when it is a W tile and fence their
//     writes for the async proxy; they hand the stage to warp 22 through a
//     named barrier (bar.arrive, no wait) and warp 22 makes the one arrive
//     on the even CTA's `sp_ready` barrier (a cluster-scope release, about
//     0.7 us, which paced the MMAs when every split warp made its own);
//   * warp 1 of the even CTA issues the 12 MMAs of the stage (4 K steps x 3
//     terms, reading hi from the raw slot and lo from the split slot) and
//     commits `raw_empty` and `sp_empty` to both CTAs, which frees both;
//   * warps 18-21 (one per TMEM lane quadrant) drain the accumulator of each
//     item -- two TMEM buffers, used by alternate items, so the MMAs of the
//     next item run meanwhile.
// The split slots are busy only from the split to the MMAs: three of them
// give the split of the next stages slack against the MMAs and leave the
// rest of shared memory to raw slots, so the loads run several stages ahead
// (8192 x 8192, r = 512 on one GB300: 269 us per norm with 3 split + 4 raw
// slots, 302 with 2 + 5, 297 with 4 + 3, measured with all sixteen split
// warps meeting at a barrier each stage before the signal warp existed).
// The grid is persistent and the items are striped over it (cluster c takes
// items c, c + clusters, ...): they are of equal size, and every role walks
// the same sequence with no hand-off.  Every mbarrier wait is bounded by
// %globaltimer; on expiry the kernel records a timeout in the status word and
// stops.  The named barriers between the split warps and the signal warp
// complete as long as every one of them walks its stages, which they do
// whether their bounded waits succeed or not (a split warp whose wait ran out
// syncs instead of arriving, so it cannot run ahead of the signal warp).
#include <cstring>

#include "common.cuh"
#include "finalize.cuh"
#include "ptx.cuh"

namespace dora {

namespace {

constexpr int kTfThreads = 736;        // warp 0 TMA, 1 MMA, 2-17 split, 18-21 drain, 22 signal
constexpr int kTfSplitWarps = 16;
constexpr int kTfSplitRows = 128 / kTfSplitWarps;   // tile rows per split warp
constexpr int kTfSplitIters = kTfSplitRows / 4;     // one warp instruction covers 4 rows
constexpr int kTfDrainWarps = 4;
constexpr uint32_t kTfXBytes = 128u * 128u;   // [128 rows x 32 fp32], 128-byte swizzle
constexpr uint32_t kTfSplitSlots = 3;

__device__ __forceinline__ float4 lds4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ void sts4(uint32_t addr, float4 v) {
  asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w)
               : "memory");
}

// x^2 + y^2 + z^2 + w^2 of one 16-byte chunk, in that order (one rounding
// per step, as the row sums of squares elsewhere)
__device__ __forceinline__ float sumsq4(const float4 v) {
  float sq4 = __fmul_rn(v.x, v.x);
  sq4 = fmaf(v.y, v.y, sq4);
  sq4 = fmaf(v.z, v.z, sq4);
  return fmaf(v.w, v.w, sq4);
}

// lo = v - trunc_tf32(v), the part of v the tensor core does not read; the
// subtraction is exact (both are within a factor of two, Sterbenz)
__device__ __forceinline__ float4 tf32_lo4(const float4 v) {
  return make_float4(__fsub_rn(v.x, tf32_trunc(v.x)), __fsub_rn(v.y, tf32_trunc(v.y)),
                     __fsub_rn(v.z, tf32_trunc(v.z)), __fsub_rn(v.w, tf32_trunc(v.w)));
}

struct TfItem {
  int tile, pass, split, kb, ke;
};

// work item -> (pair tile, N pass, K segment): segment-major
__device__ __forceinline__ TfItem tf_item(const Tf32Params& p, int item) {
  TfItem t;
  if (p.n_units > 0) {
    // the Gram's blocks on or above the block diagonal
    t.split = item / p.n_units;
    const int u = item - t.split * p.n_units;
    t.tile = p.unit_tile[u];
    t.pass = p.unit_pass[u];
  } else {
    const int per_split = p.pair_tiles * p.passes;
    t.split = item / per_split;
    const int rem = item - t.split * per_split;
    t.pass = rem / p.pair_tiles;
    t.tile = rem - t.pass * p.pair_tiles;
  }
  t.kb = p.seg_k[t.split];
  t.ke = p.seg_k[t.split + 1];
  return t;
}

// acc += sum over 32 columns of B (fp32, from global) times D (v); columns at
// or past r contribute nothing (r is a multiple of 4)
__device__ __forceinline__ float dot_b32(const float* brow, int col0, int r, bool valid,
                                         const float (&v)[32], int n, float acc) {
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    if (4 * g < n && valid && col0 + 4 * g < r) {
      const float4 b = __ldg(reinterpret_cast<const float4*>(brow + col0 + 4 * g));
      acc = fmaf(b.x, v[4 * g], acc);
      acc = fmaf(b.y, v[4 * g + 1], acc);
      acc = fmaf(b.z, v[4 * g + 2], acc);
      acc = fmaf(b.w, v[4 * g + 3], acc);
    }
  }
  return acc;
}

template <bool kStore>
__global__ void __launch_bounds__(kTfThreads, 1)
    k_gemm_tf32(const __grid_constant__ CUtensorMap tX, const __grid_constant__ CUtensorMap tY,
                const __grid_constant__ CUtensorMap tXb, const __grid_constant__ CUtensorMap tYb,
                const __grid_constant__ Tf32Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t yr = static_cast<uint32_t>(p.n_pass) / 2u;   // Y rows per CTA
  const uint32_t ybytes = yr * 128u;
  const uint32_t raw_bytes = kTfXBytes + ybytes;                // X, Y (the hi parts)
  const uint32_t sp_bytes = kTfXBytes + ybytes;                 // X lo, Y lo
  const uint32_t nraw = static_cast<uint32_t>(p.stages);
  uint8_t* sp_base = smem + nraw * raw_bytes;
  uint64_t* raw_full = reinterpret_cast<uint64_t*>(sp_base + kTfSplitSlots * sp_bytes);
  uint64_t* raw_empty = raw_full + nraw;
  uint64_t* sp_ready = raw_empty + nraw;                 // [kTfSplitSlots]
  uint64_t* sp_empty = sp_ready + kTfSplitSlots;         // [kTfSplitSlots]
  uint64_t* accum_full = sp_empty + kTfSplitSlots;       // [2]
  uint64_t* accum_empty = accum_full + 2;                // [2]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(accum_empty + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cid = static_cast<int>(cluster_id_x());
  const int ncl = static_cast<int>(num_clusters_x());
  const uint64_t deadline = global_timer_ns() + p.timeout_ns;

  // Heading a norm (a normal launch, so the stream's previous work -- which
  // may use these words -- has finished): the first CTA zeroes the control
  // words; the kernels behind this one touch them only after waiting for it.
  if (kStore && p.zero_n > 0 && blockIdx.x == 0)
    for (int i = static_cast<int>(threadIdx.x); i < p.zero_n; i += kTfThreads) p.zero_p[i] = 0;

  if (threadIdx.x == 0) {
    for (uint32_t s = 0; s < nraw; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], 1);               // the MMAs that read it are done
    }
    for (uint32_t s = 0; s < kTfSplitSlots; ++s) {
      mbar_init(&sp_ready[s], 2);   // the signal warps of both CTAs
      mbar_init(&sp_empty[s], 1);                   // the MMAs that read it are done
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accum_full[b], 1);
      mbar_init(&accum_empty[b], 2 * kTfDrainWarps);
    }
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tX);
    tma_prefetch_desc(&tY);
    if (!kStore) {
      tma_prefetch_desc(&tXb);
      tma_prefetch_desc(&tYb);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_holder, 2u * p.acc_stride);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  cluster_sync();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_holder;
  const uint32_t smem0 = smem_u32(smem);

  if (warp == 0) {
    // -------------------------------------------------------------- TMA producer (both CTAs)
    if (lane == 0) {
      const uint64_t pol_stream = l2_policy_evict_first();
      const uint64_t pol_keep = l2_policy_evict_last();
      uint32_t s = 0, phase = 0, it = 0;
      bool stop = false, g_ready = false;
      for (int item = cid; item < p.n_items && !stop; item += ncl) {
        const TfItem t = tf_item(p, item);
        const int row0 = t.tile * 256 + static_cast<int>(rank) * 128;
        const int yrow0 = t.pass * p.n_pass + static_cast<int>(rank * yr);
        for (int kt = t.kb; kt < t.ke; ++kt, ++it) {
          // the slot's previous contents must have been read by the MMAs (the
          // loaded tile is their hi operand; the split warps read it earlier)
          if (it >= nraw && !mbar_wait(&raw_empty[s], phase ^ 1u, deadline)) {
            atomicExch(p.status, kStatusTimeout);
            stop = true;
            break;
          }
          uint8_t* xs = smem + s * raw_bytes;
          uint8_t* ys = xs + kTfXBytes;
          mbar_arrive_expect_tx(&raw_full[s], raw_bytes);
          if (kt < p.kt_x) {
            tma_load_2d(xs, &tX, &raw_full[s], kt * kTf32BlockK, row0, kStore ? pol_keep : pol_stream);
            tma_load_2d(ys, &tY, &raw_full[s], kt * kTf32BlockK, yrow0, pol_keep);
          } else {
            // (B, G') tiles: G' comes from the preceding kernels
            if (!g_ready) {
              griddep_wait();
              g_ready = true;
            }
            const int kk = (kt - p.kt_x) * kTf32BlockK;
            tma_load_2d(xs, &tXb, &raw_full[s], kk, row0, pol_keep);
            tma_load_2d(ys, &tYb, &raw_full[s], kk, yrow0, pol_keep);
          }
          if (++s == nraw) {
            s = 0;
            phase ^= 1u;
          }
        }
      }
      // A CTA that loaded no G' tile never waited for the kernels this one
      // may overlap: wait before exiting, so that this grid's completion
      // covers theirs (for the Gram itself, a plain launch, a no-op).
      if (!g_ready) griddep_wait();
      // no copy may still be in flight when the CTA exits
      const uint64_t drain_deadline = global_timer_ns() + p.timeout_ns;
      const uint32_t first = it > nraw ? it - nraw : 0;
      for (uint32_t i = first; i < it; ++i)
        if (!mbar_wait(&raw_full[i % nraw], (i / nraw) & 1u, drain_deadline))
          atomicExch(p.status, kStatusTimeout);
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer (even CTA)
    if (lane == 0 && rank == 0) {
      const uint32_t idesc = idesc_tf32_f32(256, static_cast<uint32_t>(p.n_pass));
      const uint32_t sp0 = smem_u32(sp_base);
      const uint64_t dX0 = smem_desc_sw128(smem0);
      const uint64_t dY0 = smem_desc_sw128(smem0 + kTfXBytes);
      const uint64_t dXL0 = smem_desc_sw128(sp0);
      const uint64_t dYL0 = smem_desc_sw128(sp0 + kTfXBytes);
      const uint64_t raw_step = raw_bytes >> 4;
      const uint64_t sp_step = sp_bytes >> 4;
      uint32_t s = 0, phase = 0;          // split ring
      uint32_t rs = 0;                    // raw ring
      int icount = 0;
      bool stop = false;
      for (int item = cid; item < p.n_items && !stop; item += ncl, ++icount) {
        const TfItem t = tf_item(p, item);
        const uint32_t buf = static_cast<uint32_t>(icount) & 1u;
        const uint32_t use = static_cast<uint32_t>(icount) >> 1;
        if (use > 0 && !mbar_wait(&accum_empty[buf], (use - 1) & 1u, deadline)) {
          atomicExch(p.status, kStatusTimeout);
          break;
        }
        tc_fence_after_sync();
        const uint32_t acc = tmem_base + buf * p.acc_stride;
        for (int kt = t.kb; kt < t.ke; ++kt) {
          if (!mbar_wait_cluster(&sp_ready[s], phase, deadline)) {
            atomicExch(p.status, kStatusTimeout);
            stop = true;
            break;
          }
          tc_fence_after_sync();
          const uint64_t ro = static_cast<uint64_t>(rs) * raw_step;
          const uint64_t so = static_cast<uint64_t>(s) * sp_step;
#pragma unroll
          for (int ks = 0; ks < kTf32BlockK / 8; ++ks) {
            const uint64_t k = 2u * static_cast<uint64_t>(ks);   // 32 bytes per K step
            const uint32_t first = (kt == t.kb && ks == 0) ? 0u : 1u;
            umma_tf32_pair(acc, dX0 + ro + k, dY0 + ro + k, idesc, first);
            umma_tf32_pair(acc, dXL0 + so + k, dY0 + ro + k, idesc, 1u);
            umma_tf32_pair(acc, dX0 + ro + k, dYL0 + so + k, idesc, 1u);
          }
          umma_commit_pair(&raw_empty[rs], 0x3);
          umma_commit_pair(&sp_empty[s], 0x3);
          if (++rs == nraw) rs = 0;
          if (++s == kTfSplitSlots) {
            s = 0;
            phase ^= 1u;
          }
        }
        // also after a timeout: the wait below then covers every MMA issued
        umma_commit_pair(&accum_full[buf], 0x3);
      }
      if (icount > 0) {
        const uint32_t last = static_cast<uint32_t>(icount - 1);
        if (!mbar_wait(&accum_full[last & 1u], (last >> 1) & 1u, global_timer_ns() + p.timeout_ns))
          atomicExch(p.status, kStatusTimeout);
      }
    }
  } else if (warp < 2 + kTfSplitWarps) {
    // -------------------------------------------------------------- split (both CTAs)
    // Warp w handles rows 8w .. 8w + 7 of the X tile and of the Y half: one
    // instruction covers 4 whole rows (lane 8 * sub + chunk reads 16-byte
    // chunk `chunk` of row 8w + 4i + sub).  The 128-byte swizzle permutes
    // chunks within a row, which neither the split nor a row sum sees.
    const int w = warp - 2;
    const int sub = lane >> 3;
    const int chunk = lane & 7;
    const uint32_t sp0 = smem_u32(sp_base);
    uint32_t s = 0, phase = 0;          // raw ring
    uint32_t q = 0, qphase = 0, it = 0; // split ring
    bool alive = true;
    for (int item = cid; item < p.n_items; item += ncl) {
      const TfItem t = tf_item(p, item);
      const bool do_sq = !kStore && t.pass == 0;
      float sacc[kTfSplitIters], scmp[kTfSplitIters];
#pragma unroll
      for (int i = 0; i < kTfSplitIters; ++i) sacc[i] = scmp[i] = 0.f;
      for (int kt = t.kb; kt < t.ke; ++kt) {
        if (alive && !mbar_wait(&raw_full[s], phase, deadline)) {
          atomicExch(p.status, kStatusTimeout);
          alive = false;
        }
        // the split slot's previous use must have been read by the MMAs
        if (alive && it >= kTfSplitSlots && !mbar_wait(&sp_empty[q], qphase ^ 1u, deadline)) {
          atomicExch(p.status, kStatusTimeout);
          alive = false;
        }
        if (alive) {
          const uint32_t xa = smem0 + s * raw_bytes;
          const uint32_t xd = sp0 + q * sp_bytes;
          const bool sq = do_sq && kt < p.kt_x;
          const uint32_t ya = xa + kTfXBytes;
          const uint32_t yd = xd + kTfXBytes;
          // every load of the stage first, then the stores: the loads are
          // independent, so the warp waits out one shared-memory round trip
          // (slow while the tensor core streams its operands) instead of one
          // per load
          float4 vx[kTfSplitIters], vy[kTfSplitIters];
#pragma unroll
          for (int i = 0; i < kTfSplitIters; ++i)
            vx[i] = lds4(xa + static_cast<uint32_t>((kTfSplitRows * w + 4 * i + sub) * 128 + chunk * 16));
#pragma unroll
          for (int i = 0; i < kTfSplitIters; ++i) {
            const uint32_t row = static_cast<uint32_t>(kTfSplitRows * w + 4 * i + sub);
            if (row < yr) vy[i] = lds4(ya + row * 128u + static_cast<uint32_t>(chunk * 16));
          }
#pragma unroll
          for (int i = 0; i < kTfSplitIters; ++i) {
            const uint32_t off =
                static_cast<uint32_t>((kTfSplitRows * w + 4 * i + sub) * 128 + chunk * 16);
            if (sq) kahan_add(sacc[i], scmp[i], sumsq4(vx[i]));
            sts4(xd + off, tf32_lo4(vx[i]));
          }
#pragma unroll
          for (int i = 0; i < kTfSplitIters; ++i) {
            const uint32_t row = static_cast<uint32_t>(kTfSplitRows * w + 4 * i + sub);
            if (row < yr) sts4(yd + row * 128u + static_cast<uint32_t>(chunk * 16), tf32_lo4(vy[i]));
          }
          fence_async_smem_writes();
        }
        __syncwarp();
        // this warp's part is written and fenced: hand the stage to the
        // signal warp (a split warp runs at most three stages ahead of it:
        // the split slots; three barriers, one per slot, keep the phases
        // apart)
        if (alive)
          asm volatile("bar.arrive %0, %1;" ::"r"(1u + q), "n"(kTfSplitWarps * 32 + 32) : "memory");
        else   // a warp whose waits ran out must not run ahead of the signal warp
          asm volatile("bar.sync %0, %1;" ::"r"(1u + q), "n"(kTfSplitWarps * 32 + 32) : "memory");
        if (++s == nraw) {
          s = 0;
          phase ^= 1u;
        }
        ++it;
        if (++q == kTfSplitSlots) {
          q = 0;
          qphase ^= 1u;
        }
      }
      if (do_sq) {
#pragma unroll
        for (int i = 0; i < kTfSplitIters; ++i) {
          float v = __fsub_rn(sacc[i], scmp[i]);
          v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, 1));
          v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, 2));
          v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, 4));
          const int grow =
              t.tile * 256 + static_cast<int>(rank) * 128 + kTfSplitRows * w + 4 * i + sub;
          if (alive && chunk == 0 && grow < p.rows)
            p.out_sumsq[static_cast<size_t>(t.split) * p.rows + grow] = v;
        }
      }
    }
  } else if (warp == 2 + kTfSplitWarps + kTfDrainWarps) {
    // -------------------------------------------------------------- signal (both CTAs)
    // once all sixteen split warps of this CTA have handed in a stage, one
    // cluster-scope arrive on the even CTA's `sp_ready` barrier
    const uint32_t ready0 = map_to_rank(smem_u32(sp_ready), 0);
    uint32_t q = 0;
    for (int item = cid; item < p.n_items; item += ncl) {
      const TfItem t = tf_item(p, item);
      for (int kt = t.kb; kt < t.ke; ++kt) {
        asm volatile("bar.sync %0, %1;" ::"r"(1u + q), "n"(kTfSplitWarps * 32 + 32) : "memory");
        if (lane == 0) mbar_arrive_cluster(ready0 + q * 8u);
        if (++q == kTfSplitSlots) q = 0;
      }
    }
  } else {
    // -------------------------------------------------------------- drain (both CTAs)
    const int q = warp & 3;                       // TMEM lane quadrant this warp may read
    const uint32_t accum_empty0 = map_to_rank(smem_u32(accum_empty), 0);
    int icount = 0;
    for (int item = cid; item < p.n_items; item += ncl, ++icount) {
      const TfItem t = tf_item(p, item);
      const uint32_t buf = static_cast<uint32_t>(icount) & 1u;
      if (!mbar_wait(&accum_full[buf], (static_cast<uint32_t>(icount) >> 1) & 1u, deadline)) {
        atomicExch(p.status, kStatusTimeout);
        break;
      }
      tc_fence_after_sync();
      const int row = t.tile * 256 + static_cast<int>(rank) * 128 + q * 32 + lane;
      const bool valid = row < p.rows;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * p.acc_stride;
      const int col_base = t.pass * p.n_pass;
      float acc = 0.f;
      for (int c = 0; c < p.n_pass; c += 32) {
        const int n = p.n_pass - c >= 32 ? 32 : 16;   // n_pass is a multiple of 16
        float v[32];
        if (n == 32) {
          tmem_load_32cols(taddr + static_cast<uint32_t>(c), v);
        } else {
          uint32_t rv[16];
          tmem_load_16cols_async(taddr + static_cast<uint32_t>(c), rv);
          tmem_wait_ld(rv);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            v[i] = __uint_as_float(rv[i]);
            v[16 + i] = 0.f;
          }
        }
        if constexpr (!kStore) {
          const float* brow = p.B + static_cast<size_t>(valid ? row : 0) * p.r;
          acc = dot_b32(brow, col_base + c, p.r, valid, v, n, acc);
        } else {
          float* grow = p.out_g + (static_cast<size_t>(t.split) * p.rows + (valid ? row : 0)) * p.r;
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            const int col = col_base + c + 4 * g;
            if (4 * g < n && valid && col < p.r)
              *reinterpret_cast<float4*>(grow + col) =
                  make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(accum_empty0 + buf * 8u);
      if (!kStore && valid)
        p.out_dot[(static_cast<size_t>(t.pass) * p.splits + t.split) * p.rows + row] = acc;
    }
  }

  __syncwarp();              // whole warps at the aligned barriers below (roles ran on single lanes)
  tc_fence_before_sync();
  __syncthreads();
  // this CTA's work is done: the next kernel of the stream (a programmatic
  // dependent that waits for this grid before it reads) may start
  griddep_launch_dependents();
  cluster_sync();            // the peer may still read this CTA's shared memory until here
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, 2u * p.acc_stride);
  }
}

// G' = scale * (sum of the K-segment partials in segment order), zero padded.
// kVec: four neighbouring columns per thread with 16-byte loads and stores
// (r and rp multiples of 4, both arrays 16-byte aligned); the same sums.
template <bool kVec>
__global__ void k_gram_tf32_reduce(const float* __restrict__ parts, int splits, int r, int rp,
                                   float scale, float* __restrict__ Gp, int n_pass, int sym) {
  // a programmatic dependent of the Gram pass: the norm pass behind it may
  // launch now (it waits for this grid before its first G' tile); the sums
  // start once the Gram's partials are complete
  griddep_launch_dependents();
  griddep_wait();
  constexpr int kW = kVec ? 4 : 1;
  const int64_t idx = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * kW;
  if (idx >= static_cast<int64_t>(rp) * rp) return;
  const int i = static_cast<int>(idx / rp);
  const int j = static_cast<int>(idx - static_cast<int64_t>(i) * rp);
  // symmetric partials: the block of (row, col) -- 256-row tile, n_pass-column
  // pass -- lies strictly below the block diagonal when the whole pass is
  // left of the tile's first row; such an element is the mirror image of one
  // in a computed block (n_pass is a multiple of 16 and the kW columns are
  // aligned, so the test is the same for all of them)
  const bool inside = i < r && j < r;
  auto below = [&](int row, int col) {
    return sym != 0 && (col / n_pass + 1) * n_pass <= (row / 256) * 256;
  };
  if (inside && below(i, j)) return;     // written by the thread of its mirror image
  float out[kW];
#pragma unroll
  for (int c = 0; c < kW; ++c) out[c] = 0.f;
  if (inside) {
    // all loads first (they are independent), then the sums in segment order
    float v[kTf32MaxGramSplits][kW];
    const size_t plane = static_cast<size_t>(r) * r;
    const float* src = parts + static_cast<size_t>(i) * r + j;
#pragma unroll
    for (int sp = 0; sp < kTf32MaxGramSplits; ++sp) {
      if constexpr (kVec) {
        const float4 t = sp < splits ? __ldg(reinterpret_cast<const float4*>(src + sp * plane))
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
        v[sp][0] = t.x;
        v[sp][1] = t.y;
        v[sp][2] = t.z;
        v[sp][3] = t.w;
      } else {
        v[sp][0] = sp < splits ? __ldg(src + sp * plane) : 0.f;
      }
    }
#pragma unroll
    for (int c = 0; c < kW; ++c) {
      df acc{0.f, 0.f};
#pragma unroll
      for (int sp = 0; sp < kTf32MaxGramSplits; ++sp) {
        float e;
        two_sum(acc.hi, v[sp][c], acc.hi, e);
        acc.lo = __fadd_rn(acc.lo, e);
      }
      out[c] = __fmul_rn(scale, __fadd_rn(acc.hi, acc.lo));
    }
  }
  if constexpr (kVec) {
    *reinterpret_cast<float4*>(Gp + idx) = make_float4(out[0], out[1], out[2], out[3]);
  } else {
    Gp[idx] = out[0];
  }
  if (inside && below(j, i)) {
#pragma unroll
    for (int c = 0; c < kW; ++c) Gp[static_cast<int64_t>(j + c) * rp + i] = out[c];
  }
}

}  // namespace

// `stages` raw slots plus the split slots and the barriers
size_t tf32_smem_bytes(int n_pass, int stages) {
  const size_t ybytes = static_cast<size_t>(n_pass / 2) * 128u;
  const size_t raw = kTfXBytes + ybytes;
  const size_t sp = kTfXBytes + ybytes;
  return 1024 + raw * static_cast<size_t>(stages) + sp * kTfSplitSlots +
         (2 * static_cast<size_t>(stages) + 2 * kTfSplitSlots + 4) * 8 + 16;
}

int tf32_pick_stages(int n_pass) {
  const size_t budget = 227 * 1024;
  int st = kTcMaxStages;
  while (st > 2 && tf32_smem_bytes(n_pass, st) > budget) --st;
  return st;
}

// Co-resident CTA pairs (one CTA per SM: every shape needs most of an SM's
// shared memory); the attribute is raised to the largest size once per device.
int tf32_max_clusters() {
  constexpr int kMaxSmem = 227 * 1024;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  static int cached[64] = {0};
  if (dev < 64 && cached[dev]) return cached[dev];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kTfThreads, 1, 1);
  cfg.dynamicSmemBytes = kMaxSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaFuncSetAttribute(k_gemm_tf32<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kMaxSmem) != cudaSuccess ||
      cudaFuncSetAttribute(k_gemm_tf32<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kMaxSmem) != cudaSuccess ||
      cudaOccupancyMaxActiveClusters(&n, k_gemm_tf32<false>, &cfg) != cudaSuccess)
    return 0;
  if (dev < 64) cached[dev] = n;
  return n;
}

cudaError_t launch_gemm_tf32(const CUtensorMap& tX, const CUtensorMap& tY, const CUtensorMap& tXb,
                             const CUtensorMap& tYb, const Tf32Params& p, bool store,
                             int clusters, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  cfg.blockDim = dim3(kTfThreads, 1, 1);
  cfg.dynamicSmemBytes = tf32_smem_bytes(p.n_pass, p.stages);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // the norm pass may start while the G' reduce still runs: only its (B, G')
  // loads depend on it, and they wait for it (griddep_wait)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = store ? 1 : 2;
  cudaError_t e = store ? cudaLaunchKernelEx(&cfg, k_gemm_tf32<true>, tX, tY, tXb, tYb, p)
                        : cudaLaunchKernelEx(&cfg, k_gemm_tf32<false>, tX, tY, tXb, tYb, p);
  note_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_gram_tf32_reduce(const float* parts, int splits, int r, int rp, float scale,
                                    float* Gp, cudaStream_t stream, int n_pass, int sym) {
  if (sym && (n_pass <= 0 || n_pass % 16 != 0)) return cudaErrorInvalidValue;
  const bool vec = r % 4 == 0 && rp % 4 == 0 && (reinterpret_cast<uintptr_t>(parts) & 15u) == 0 &&
                   (reinterpret_cast<uintptr_t>(Gp) & 15u) == 0;
  const int64_t n = static_cast<int64_t>(rp) * rp / (vec ? 4 : 1);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((n + 255) / 256), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e =
      vec ? cudaLaunchKernelEx(&cfg, k_gram_tf32_reduce<true>, parts, splits, r, rp, scale, Gp,
                               n_pass, sym)
          : cudaLaunchKernelEx(&cfg, k_gram_tf32_reduce<false>, parts, splits, r, rp, scale, Gp,
                               n_pass, sym);
  note_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dora
