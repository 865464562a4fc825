// gram.cu -- G = A A^T for the factored norm (bf16 inputs), and its scaled
// two-term split G'_hi + G'_lo = (s/2) G that the main pass folds into its K
// loop ("Scaling DoRA", Chinese write-up section 1.2.1 and Algorithm 1 of
// section 5.1: the r x r Gram matrix that replaces the dense B A).  Only the
// split reaches the tensor core, so G itself is not stored.
//
// G is symmetric, so only the upper triangle of its grid of 128 x 128 blocks
// is computed; each block (bi, bj) is written to both places.  One cluster of
// C CTAs owns one block and splits its K range (d_in) C ways:
//   * warp 0 of each CTA streams [128 x 64] tiles of A rows bi*128.. and
//     bj*128.. through a shared-memory ring (TMA), warp 1 issues the
//     tcgen05.mma (M = 128, N = the block width as two halves, fp32
//     accumulator in tensor memory), warps 2-5 then move the CTA's partial
//     block from tensor memory into its shared memory;
//   * CTA q owns rows [q*128/C, (q+1)*128/C) of the block: every CTA sends
//     each owner its slice of the partial block with one bulk copy into the
//     owner's shared memory (distributed shared memory, completion counted
//     on the owner's mbarrier); the owner sums the C slices in rank order --
//     a fixed order, so the result is the same on every call -- and stores
//     G'_hi and G'_lo for its rows and their mirror image.
// The partial blocks never leave the cluster: no split-K buffer in global
// memory and no second kernel.  G'_hi = bf16(G'), G'_lo = bf16(G' - G'_hi),
// G' = (s/2) G rounded once to fp32: the two bf16 terms carry about 16
// significant bits of G' into the tensor core.  In partials mode (G_f32 set)
// the kernel stores scale * G itself in fp32, [r x r] row-major, instead of
// the split: the Gram partial of one d_in slice, which a caller adds across
// slices.
#include <cstring>

#include "common.cuh"
#include "ptx.cuh"

namespace dora {

namespace {

constexpr int kGramThreads = 192;    // warp 0 TMA, warp 1 MMA, warps 2-5 TMEM -> shared memory
constexpr int kGramTileBytes = 128 * 128;   // [128 rows x 64 bf16] with the 128-byte swizzle

// bulk copy of `bytes` from this CTA's shared memory into a cluster peer's,
// completion (bytes) counted on the peer's mbarrier
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst_cluster, uint32_t src_cta,
                                                  uint32_t bytes, uint32_t mbar_cluster) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst_cluster), "r"(src_cta), "r"(bytes), "r"(mbar_cluster)
      : "memory");
}

// generic-proxy writes to shared memory before async-proxy (bulk copy) reads
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// block index -> (bi, bj) of the upper triangle, row-major
__device__ __forceinline__ void gram_block(int b, int nb, int& bi, int& bj) {
  int i = 0;
  while (b >= nb - i) {
    b -= nb - i;
    ++i;
  }
  bi = i;
  bj = i + b;
}

template <bool kGrouped>
__global__ void __launch_bounds__(kGramThreads, 1)
    k_gram(const __grid_constant__ CUtensorMap tAx_param, const __grid_constant__ CUtensorMap tAy_param,
           const GramParams p_in, const GramModule* mods) {
  // the module of this cluster (grouped) or the kernel parameters
  GramParams p = p_in;
  const CUtensorMap* tAxp = &tAx_param;
  const CUtensorMap* tAyp = &tAy_param;
  int block_base = 0;
  if constexpr (kGrouped) {
    const int per_module = p_in.nb * (p_in.nb + 1) / 2 * static_cast<int>(p_in.cluster);
    const int mi = static_cast<int>(blockIdx.x) / per_module;
    block_base = mi * per_module;
    tAxp = &mods[mi].tAx;
    tAyp = &mods[mi].tAy;
    p.G_hi = mods[mi].G_hi;
    p.G_lo = mods[mi].G_lo;
    p.k_tiles = mods[mi].k_tiles;
  }
  const CUtensorMap& tAx = *tAxp;
  const CUtensorMap& tAy = *tAyp;
  // launched as a programmatic dependent of whatever precedes it in the
  // stream (the previous norm on this workspace, or the kernel that zeroes
  // the workspace's control words): nothing is read or written before that
  // grid has finished.  When this kernel heads the norm's chain its first CTA
  // zeroes the control words here; the main pass reads or writes them only
  // after waiting for this grid (griddepcontrol.wait), and another CTA of
  // this grid records a timeout only after its bounded wait (seconds) has
  // run out.  Then the main pass queued behind this kernel may start
  // launching; it waits for this grid to finish before it reads G'.
  griddep_wait();
  if (!kGrouped && p_in.zero_n > 0 && blockIdx.x == 0)
    for (int i = static_cast<int>(threadIdx.x); i < p_in.zero_n; i += kGramThreads) p_in.zero_p[i] = 0;
  griddep_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t y_bytes = static_cast<uint32_t>(p.bw) * 128u;
  const uint32_t stage_bytes = kGramTileBytes + y_bytes;
  // the stage ring, later reused for the CTA's partial block [128][bw + 4] fp32
  const uint32_t ring = p.stages * stage_bytes;
  // partial block + receive area + staged G' rows (hi, lo)
  const uint32_t part_bytes =
      2u * 128u * static_cast<uint32_t>(p.bw + 4) * 4u + 2u * 128u * static_cast<uint32_t>(p.bw) * 2u;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (ring > part_bytes ? ring : part_bytes));
  uint64_t* empty = full + p.stages;
  uint64_t* accum_full = empty + p.stages;
  uint64_t* recv_full = accum_full + 1;      // every slice sent to this CTA has landed
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(recv_full + 1);
  // partial block [128][ld] fp32 at the start of the ring, then the receive
  // area: C slices of this CTA's rows, [C][rows_per][ld]
  float* part = reinterpret_cast<float*>(smem);
  const int ld = p.bw + 4;
  const int rows_per = 128 / static_cast<int>(p.cluster);
  const uint32_t slice_bytes = static_cast<uint32_t>(rows_per * ld * 4);
  float* recv = part + 128 * ld;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t q = cluster_ctarank();
  const uint32_t C = p.cluster;
  int bi, bj;
  gram_block(static_cast<int>((blockIdx.x - block_base) / C), p.nb, bi, bj);
  const int kt_begin = static_cast<int>((static_cast<long long>(p.k_tiles) * q) / C);
  const int kt_end = static_cast<int>((static_cast<long long>(p.k_tiles) * (q + 1)) / C);
  const int n_iter = kt_end - kt_begin;
  const bool diag = bi == bj;
  const uint64_t deadline = global_timer_ns() + p.timeout_ns;
  bool ok = true;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accum_full, 1);
    mbar_init(recv_full, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tAx);
    tma_prefetch_desc(&tAy);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_last();   // A is re-read by every block row
      const uint32_t stages = static_cast<uint32_t>(p.stages);
      uint32_t s = 0, phase = 0;
      int issued = 0;
      for (int i = 0; i < n_iter; ++i) {
        if (i >= p.stages && !mbar_wait(&empty[s], phase ^ 1u, deadline)) {
          atomicExch(p.status, kStatusTimeout);
          break;
        }
        const int kx = (kt_begin + i) * 64;
        uint8_t* xs = smem + s * stage_bytes;
        if (diag) {
          // a diagonal block multiplies the tile by itself: X serves as Y
          mbar_arrive_expect_tx(&full[s], kGramTileBytes);
          tma_load_2d(xs, &tAx, &full[s], kx, bi * 128, pol);
        } else {
          mbar_arrive_expect_tx(&full[s], stage_bytes);
          tma_load_2d(xs, &tAx, &full[s], kx, bi * 128, pol);
          tma_load_2d(xs + kGramTileBytes, &tAy, &full[s], kx, bj * 128, pol);
        }
        issued = i + 1;
        if (++s == stages) {
          s = 0;
          phase ^= 1u;
        }
      }
      // no copy may still be landing when the stage ring is reused below
      const uint64_t drain_deadline = global_timer_ns() + p.timeout_ns;
      for (int i = issued > p.stages ? issued - p.stages : 0; i < issued; ++i)
        if (!mbar_wait(&full[i % p.stages], static_cast<uint32_t>(i / p.stages) & 1u,
                       drain_deadline))
          atomicExch(p.status, kStatusTimeout);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // the block width as two halves (two independent accumulators per K
      // step) when each half is a valid MMA width (a multiple of 16)
      const bool halves = p.bw % 32 == 0;
      const int nh = halves ? p.bw / 2 : p.bw;
      const uint32_t idesc = idesc_bf16_f32(128, nh);
      const uint64_t dx0 = smem_desc_sw128(smem_u32(smem));
      const uint64_t dy0 = smem_desc_sw128(smem_u32(smem) + (diag ? 0u : kGramTileBytes));
      const uint64_t dy1 = static_cast<uint64_t>(nh) * 128u >> 4;
      const uint64_t step = stage_bytes >> 4;
      const uint32_t stages = static_cast<uint32_t>(p.stages);
      uint32_t s = 0, phase = 0;
      for (int i = 0; i < n_iter; ++i) {
        if (!mbar_wait(&full[s], phase, deadline)) {
          atomicExch(p.status, kStatusTimeout);
          break;
        }
        const uint64_t dx = dx0 + s * step, dy = dy0 + s * step;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint32_t acc = (i > 0 || ks > 0) ? 1u : 0u;
          umma_bf16(tmem_base, dx + 2 * ks, dy + 2 * ks, idesc, acc);
          if (halves)
            umma_bf16(tmem_base + static_cast<uint32_t>(nh), dx + 2 * ks, dy + dy1 + 2 * ks,
                      idesc, acc);
        }
        umma_commit(&empty[s]);
        if (++s == stages) {
          s = 0;
          phase ^= 1u;
        }
      }
      // arrives once every MMA issued above has completed (at once if none)
      umma_commit(accum_full);
    }
  } else {
    // ------------------------------------------------------------ TMEM -> shared memory
    const int qd = warp & 3;                 // TMEM lane quadrant = rows 32 qd ..
    const int row = qd * 32 + lane;
    if (!mbar_wait(accum_full, 0, deadline)) {
      atomicExch(p.status, kStatusTimeout);
      ok = false;
    }
    tc_fence_after_sync();
    ok = __all_sync(0xFFFFFFFFu, ok);
    float* dst = part + row * ld;
    for (int c0 = 0; c0 < p.bw; c0 += 16) {
      uint32_t v[16];
      if (ok && n_iter > 0) {
        tmem_load_16cols_async(tmem_base + (static_cast<uint32_t>(qd * 32) << 16) +
                                   static_cast<uint32_t>(c0), v);
        tmem_wait_ld(v);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = 0u;      // an empty K slice adds nothing
      }
#pragma unroll
      for (int i = 0; i < 16; i += 4)
        *reinterpret_cast<float4*>(dst + c0 + i) =
            make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                        __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
    }
  }

  // this CTA's partial block is in shared memory; the bulk copies read it
  fence_proxy_async_smem();
  if (threadIdx.x == 0) mbar_arrive_expect_tx(recv_full, slice_bytes * C);
  __syncwarp();            // whole warps at the aligned barriers below
  tc_fence_before_sync();
  cluster_sync();          // every partial written, every receive area free and armed

  // ------------------------------------------------------------ cross-CTA sum
  if (threadIdx.x == 0) {
    // slice d (rows of owner d) goes to owner d's receive slot q
    const uint32_t part_local = smem_u32(part);
    const uint32_t recv_local = smem_u32(recv);
    for (uint32_t d = 0; d < C; ++d)
      bulk_copy_to_peer(map_to_rank(recv_local + q * slice_bytes, d),
                        part_local + d * slice_bytes, slice_bytes,
                        map_to_rank(smem_u32(recv_full), d));
  }
  __syncwarp();
  // one decision for the whole CTA (named barriers follow)
  const bool got = __syncthreads_and(mbar_wait(recv_full, 0, deadline) ? 1 : 0) != 0;
  // every slice sent to this CTA has landed (or its wait gave up): once every
  // CTA of the cluster has arrived here, no bulk copy between them is in
  // flight and each may leave without waiting for the others' stores below
  cluster_arrive();
  if (!got) {
    if (threadIdx.x == 0) atomicExch(p.status, kStatusTimeout);
  } else {
    // G' = scale * (sum of the C slices in rank order, a fixed order), split
    // into hi + lo; staged in shared memory past the receive area (the
    // partial block may still be read by this CTA's outgoing copies) so that
    // both the block and its mirror image are written with contiguous stores
    const int c4 = p.bw / 4;                 // float4 columns of a block row
    const int n = rows_per * c4;
    uint16_t* hi_s = reinterpret_cast<uint16_t*>(recv + 128 * ld);   // [rows_per][bw]
    uint16_t* lo_s = hi_s + rows_per * p.bw;                    // [rows_per][bw]
    for (int e = threadIdx.x; e < n; e += kGramThreads) {
      const int li = e / c4;                 // row inside this CTA's slice
      const int j = (e % c4) * 4;            // first of four columns
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (uint32_t src = 0; src < C; ++src) {
        const float4 v =
            *reinterpret_cast<const float4*>(recv + (src * rows_per + li) * ld + j);
        acc.x = __fadd_rn(acc.x, v.x);
        acc.y = __fadd_rn(acc.y, v.y);
        acc.z = __fadd_rn(acc.z, v.z);
        acc.w = __fadd_rn(acc.w, v.w);
      }
      const float a[4] = {acc.x, acc.y, acc.z, acc.w};
      const int gi = bi * 128 + static_cast<int>(q) * rows_per + li;
      const int gj = bj * 128 + j;
      if (p.G_f32) {
        // fp32 G (scaled), staged for the mirror image in the hi/lo area
        float* f_s = reinterpret_cast<float*>(hi_s);          // [rows_per][bw]
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float sc = __fmul_rn(p.scale, a[u]);
          f_s[li * p.bw + j + u] = sc;
          if (gi < p.r_out && gj + u < p.r_out)
            p.G_f32[static_cast<size_t>(gi) * p.r_out + gj + u] = sc;
        }
        continue;
      }
      uint16_t h4[4], l4[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float sc = __fmul_rn(p.scale, a[u]);
        h4[u] = f32_to_bf16_rn(sc);
        l4[u] = f32_to_bf16_rn(__fsub_rn(sc, bf16_to_f32(h4[u])));
      }
      const uint2 hv = make_uint2(h4[0] | (static_cast<uint32_t>(h4[1]) << 16),
                                  h4[2] | (static_cast<uint32_t>(h4[3]) << 16));
      const uint2 lv = make_uint2(l4[0] | (static_cast<uint32_t>(l4[1]) << 16),
                                  l4[2] | (static_cast<uint32_t>(l4[3]) << 16));
      *reinterpret_cast<uint2*>(hi_s + li * p.bw + j) = hv;
      *reinterpret_cast<uint2*>(lo_s + li * p.bw + j) = lv;
      // the block itself: four consecutive columns per thread (rp is a
      // multiple of 16, so a group of four is either inside or outside)
      if (gi < p.rp && gj < p.rp) {
        const size_t o = static_cast<size_t>(gi) * p.rp + gj;
        *reinterpret_cast<uint2*>(p.G_hi + o) = hv;
        *reinterpret_cast<uint2*>(p.G_lo + o) = lv;
      }
    }
    if (bi != bj) {
      // the mirrored block of the lower triangle: row gj, columns gi .. of
      // this slice; consecutive threads take consecutive columns
      asm volatile("bar.sync 2, %0;" ::"n"(kGramThreads) : "memory");
      const int n2 = p.bw * rows_per;
      for (int e = threadIdx.x; e < n2; e += kGramThreads) {
        const int j = e / rows_per;          // column inside the block -> mirror row
        const int li = e % rows_per;
        const int gi = bi * 128 + static_cast<int>(q) * rows_per + li;
        const int gj = bj * 128 + j;
        if (p.G_f32) {
          if (gi < p.r_out && gj < p.r_out)
            p.G_f32[static_cast<size_t>(gj) * p.r_out + gi] =
                reinterpret_cast<const float*>(hi_s)[li * p.bw + j];
        } else if (gi < p.rp && gj < p.rp) {
          const size_t t = static_cast<size_t>(gj) * p.rp + gi;
          p.G_hi[t] = hi_s[li * p.bw + j];
          p.G_lo[t] = lo_s[li * p.bw + j];
        }
      }
    }
  }

  __syncwarp();
  cluster_wait();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

}  // namespace

size_t gram_smem_bytes(int bw, int stages) {
  const size_t stage = kGramTileBytes + static_cast<size_t>(bw) * 128u;
  const size_t ring = stage * stages;
  // partial block + receive area + staged G' rows (hi, lo)
  const size_t part = static_cast<size_t>(2) * 128 * (bw + 4) * 4 + static_cast<size_t>(2) * 128 * bw * 2;
  return 1024 + (ring > part ? ring : part) + (2 * stages + 2) * 8 + 16;
}

namespace {

cudaError_t gram_configure() {
  static int configured_for[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !configured_for[dev]) {
    for (auto fn : {k_gram<false>, k_gram<true>}) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
    }
    configured_for[dev] = 1;
  }
  return cudaSuccess;
}

template <bool kGrouped>
cudaError_t gram_launch(const CUtensorMap& tAx, const CUtensorMap& tAy, const GramParams& p,
                        const GramModule* mods, int n_mods, cudaStream_t stream) {
  cudaError_t e = gram_configure();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.nb * (p.nb + 1) / 2 * p.cluster * n_mods), 1, 1);
  cfg.blockDim = dim3(kGramThreads, 1, 1);
  cfg.dynamicSmemBytes = gram_smem_bytes(p.bw, p.stages);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(p.cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, k_gram<kGrouped>, tAx, tAy, p, mods);
  note_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gram(const CUtensorMap& tAx, const CUtensorMap& tAy, const GramParams& p,
                        cudaStream_t stream) {
  return gram_launch<false>(tAx, tAy, p, nullptr, 1, stream);
}

cudaError_t launch_gram_grouped(const GramModule* mods, int n_mods, const GramParams& p,
                                cudaStream_t stream) {
  CUtensorMap none;
  std::memset(&none, 0, sizeof(none));
  return gram_launch<true>(none, none, p, mods, n_mods, stream);
}

}  // namespace dora
