// gemm_tc.cu -- the tensor-core pass of the factored norm (bf16 inputs).
//
// One CTA owns a 128-row tile of X and a contiguous range of K tiles (split-K
// over gridDim.y).  Warp roles:
//   warp 0     TMA producer: X tile [128 x 64] and Y tile [n_pad x 64] per stage
//   warp 1     allocates tensor memory; one thread issues tcgen05.mma into a
//              [128 x n_pad] fp32 accumulator
//   warps 2-5  epilogue: while the K loop runs they read every X tile from
//              shared memory and accumulate the row sums of squares; after the
//              last tile they read the accumulator rows from tensor memory
//              (warp w owns TMEM lanes 32*(w%4) .. +31, i.e. tile rows)
//
// Uses in the factored norm ("Scaling DoRA", Chinese write-up section 1.2.1,
// Algorithm 1 of section 5.1):
//   main pass  X = W, Y = A          : base = sum_k W^2 (SumSq), cross = rowsum(B o U) (DotB)
//   Gram       X = A, Y = A          : G partials (Store)
//   BA norm    X = B, Y = G_hi|G_lo  : ba = rowsum((B G) o B) (DotB), G split in two bf16 terms
// Every sum here is linear in the K range, so split-K partials add exactly
// like the chunks of Algorithm 1; they are summed in a fixed order later.
#include "common.cuh"
#include "ptx.cuh"

namespace dora {

namespace {

__device__ __forceinline__ void record_timeout(int* status) {
  atomicExch(status, kStatusTimeout);
}

__device__ __forceinline__ float sumsq_row128(const uint8_t* row, int rot) {
  // 128 bytes = 64 bf16 of one tile row; the 128-byte swizzle only permutes the
  // 16-byte chunks inside the row, which a sum does not see.  Starting at chunk
  // (row mod 8) keeps the 8 threads of a shared-memory phase on different banks.
  const uint4* p = reinterpret_cast<const uint4*>(row);
  float acc = 0.f;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 v = p[c ^ rot];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float a = bf16_lo(w[i]), b = bf16_hi(w[i]);
      acc = fmaf(a, a, acc);
      acc = fmaf(b, b, acc);
    }
  }
  return acc;
}

__global__ void __launch_bounds__(kTcThreads, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tx, const __grid_constant__ CUtensorMap ty0,
              const __grid_constant__ CUtensorMap ty1, const TcParams p) {
  // the kernel queued behind this one may start launching; it waits for this
  // grid to finish before it reads any of its results
  griddep_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t y_bytes = static_cast<uint32_t>(p.n_pad) * 128u;
  const uint32_t stage_bytes = kTcXTileBytes + y_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.stages * stage_bytes);
  uint64_t* empty = full + p.stages;
  uint64_t* accum_full = empty + p.stages;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(accum_full + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int split = blockIdx.y;
  const int splits = gridDim.y;
  // Gram mode: CTA x handles the upper-triangular 128x128 block (bi, bj) of
  // G = A A^T, i.e. X rows bi*128.. and Y rows bj*128..
  int row0 = blockIdx.x * kTcBlockM;
  int y_row0 = 0;
  if (p.gram_nb > 0) {
    int b = blockIdx.x, bi = 0;
    while (b >= p.gram_nb - bi) {
      b -= p.gram_nb - bi;
      ++bi;
    }
    row0 = bi * kTcBlockM;
    y_row0 = (bi + b) * kTcBlockM;
  }
  const int kt_begin = static_cast<int>((static_cast<long long>(p.k_tiles) * split) / splits);
  const int kt_end = static_cast<int>((static_cast<long long>(p.k_tiles) * (split + 1)) / splits);
  const int n_iter = kt_end - kt_begin;
  const bool do_sumsq = (p.mode & kTcSumSq) != 0;
  const uint64_t deadline = global_timer_ns() + p.timeout_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1 + (do_sumsq ? 4 : 0));
    }
    mbar_init(accum_full, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tx);
    tma_prefetch_desc(&ty0);
    tma_prefetch_desc(&ty1);
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
    // ---------------------------------------------------------------- producer
    if (lane == 0 && !p.inject_fault) {
      const uint64_t pol_x = l2_policy_evict_first();
      const uint64_t pol_y = l2_policy_evict_last();
      int issued = 0;
      const int stages = p.stages;
      int s = 0;
      uint32_t phase = 0;
      for (int i = 0; i < n_iter; ++i) {
        if (i >= stages && !mbar_wait(&empty[s], phase ^ 1u, deadline)) {
          record_timeout(p.status);
          *abort_flag = 1;
          break;
        }
        if (*abort_flag) break;
        const int kt = kt_begin + i;
        const bool second = kt >= p.k_tiles_pass;
        const int kx = (second ? kt - p.k_tiles_pass : kt) * kTcBlockK;
        const CUtensorMap* ym = second ? &ty1 : &ty0;
        uint8_t* xs = smem + s * stage_bytes;
        uint8_t* ys = xs + kTcXTileBytes;
        mbar_arrive_expect_tx(&full[s], stage_bytes);
        tma_load_2d(xs, &tx, &full[s], kx, row0, pol_x);
        for (int c = 0; c < p.n_pad; c += p.y_box_rows)
          tma_load_2d(ys + c * 128, ym, &full[s], kx, y_row0 + c, pol_y);
        issued = i + 1;
        if (++s == stages) {
          s = 0;
          phase ^= 1u;
        }
      }
      // Never leave a copy landing in shared memory after this CTA is gone:
      // wait (bounded, with a fresh limit) for the last load of every stage.
      const uint64_t drain_deadline = global_timer_ns() + p.timeout_ns;
      for (int i = issued > p.stages ? issued - p.stages : 0; i < issued; ++i) {
        if (!mbar_wait(&full[i % p.stages], static_cast<uint32_t>(i / p.stages) & 1u,
                       drain_deadline))
          record_timeout(p.status);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      // descriptors of stage 0 and register offsets; no parameter reloads in the loop
      const int n0 = p.n_pad < 256 ? p.n_pad : 256;
      const int n1 = p.n_pad - n0;
      const bool two = n1 > 0;
      const uint32_t idesc0 = idesc_bf16_f32(kTcBlockM, n0);
      const uint32_t idesc1 = idesc_bf16_f32(kTcBlockM, two ? n1 : 16);
      const uint32_t tmem1 = tmem_base + static_cast<uint32_t>(n0);
      const uint64_t dx0 = smem_desc_sw128(smem_u32(smem));
      const uint64_t dy0 = smem_desc_sw128(smem_u32(smem) + kTcXTileBytes);
      const uint64_t dy1_off = static_cast<uint64_t>(n0) * 128u >> 4;
      const uint64_t stage_step = stage_bytes >> 4;
      const int stages = p.stages;
      int s = 0;
      uint32_t phase = 0;
      for (int i = 0; i < n_iter; ++i) {
        if (!mbar_wait(&full[s], phase, deadline)) {
          record_timeout(p.status);
          *abort_flag = 1;
          break;
        }
        if (*abort_flag) break;
        const uint64_t dx = dx0 + s * stage_step;
        const uint64_t dy = dy0 + s * stage_step;
        const uint32_t first = i > 0 ? 1u : 0u;
#pragma unroll
        for (int ks = 0; ks < kTcBlockK / 16; ++ks) {
          const uint32_t acc = ks > 0 ? 1u : first;
          umma_bf16(tmem_base, dx + 2 * ks, dy + 2 * ks, idesc0, acc);
          if (two) umma_bf16(tmem1, dx + 2 * ks, dy + dy1_off + 2 * ks, idesc1, acc);
        }
        umma_commit(&empty[s]);
        if (++s == stages) {
          s = 0;
          phase ^= 1u;
        }
      }
      // arrives once every MMA issued above has completed
      umma_commit(accum_full);
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;                 // TMEM lane quadrant of this warp
    const int trow = q * 32 + lane;         // row inside the tile
    const int grow = row0 + trow;           // row of X
    const bool valid = grow < p.rows;
    const uint32_t tmem_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    float ss = 0.f, ss_c = 0.f;
    bool ok = true;
    if (do_sumsq) {
      const int stages = p.stages;
      int s = 0;
      uint32_t phase = 0;
      for (int i = 0; i < n_iter; ++i) {
        if (!mbar_wait(&full[s], phase, deadline)) {
          record_timeout(p.status);
          *abort_flag = 1;
          ok = false;
          break;
        }
        const float part = sumsq_row128(smem + s * stage_bytes + trow * 128, trow & 7);
        kahan_add(ss, ss_c, part);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (++s == stages) {
          s = 0;
          phase ^= 1u;
        }
      }
    }
    if (!mbar_wait(accum_full, 0, deadline)) {
      record_timeout(p.status);
      ok = false;
    }
    tc_fence_after_sync();
    ok = ok && !*abort_flag;
    ok = __all_sync(0xFFFFFFFFu, ok);
    if (ok) {
      if (p.mode & kTcDotB) {
        float acc = 0.f;
        const uint16_t* brow = p.B + static_cast<size_t>(valid ? grow : 0) * p.r;
        for (int c0 = 0; c0 < p.r; c0 += 32) {
          float v[32];
          tmem_load_32cols(tmem_row + static_cast<uint32_t>(c0), v);
          if (valid) {
            if (c0 + 32 <= p.r) {
              const uint4* bp = reinterpret_cast<const uint4*>(brow + c0);
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                const uint4 bv = __ldg(bp + c);
                const uint32_t w[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  acc = fmaf(bf16_lo(w[e]), v[c * 8 + 2 * e], acc);
                  acc = fmaf(bf16_hi(w[e]), v[c * 8 + 2 * e + 1], acc);
                }
              }
            } else {
#pragma unroll
              for (int c = 0; c < 32; ++c)
                if (c < p.r - c0) acc = fmaf(bf16_to_f32(brow[c0 + c]), v[c], acc);
            }
          }
        }
        if (valid) p.out_dot[static_cast<size_t>(split) * p.rows + grow] = acc;
      }
      if (p.mode & kTcStore) {
        // this CTA's [128 x n_pad] partial, row-major, slot (split, blockIdx.x)
        float* dst = p.out_store +
                     (static_cast<size_t>(split) * gridDim.x + blockIdx.x) * kTcBlockM * p.n_pad +
                     static_cast<size_t>(trow) * p.n_pad;
        for (int c0 = 0; c0 < p.n_pad; c0 += 32) {
          float v[32];
          tmem_load_32cols(tmem_row + static_cast<uint32_t>(c0), v);
#pragma unroll
          for (int c = 0; c < 32; c += 4)
            if (c0 + c < p.n_pad)
              *reinterpret_cast<float4*>(dst + c0 + c) = make_float4(v[c], v[c + 1], v[c + 2], v[c + 3]);
        }
      }
      if (do_sumsq && valid) p.out_sumsq[static_cast<size_t>(split) * p.rows + grow] = ss;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

}  // namespace

size_t tc_smem_bytes(int n_pad, int stages) {
  const size_t stage = kTcXTileBytes + static_cast<size_t>(n_pad) * 128u;
  return 1024 + stage * stages + (2 * stages + 1) * 8 + 16;
}

int tc_pick_stages(int n_pad) {
  const size_t budget = 227 * 1024;
  int st = kTcMaxStages;
  while (st > 2 && tc_smem_bytes(n_pad, st) > budget) --st;
  return st;
}

cudaError_t launch_gemm_tc(const CUtensorMap& tx, const CUtensorMap& ty0, const CUtensorMap& ty1,
                           const TcParams& p, int row_tiles, int splits, cudaStream_t stream) {
  const size_t smem = tc_smem_bytes(p.n_pad, p.stages);
  static int configured_for[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !configured_for[dev]) {
    e = cudaFuncSetAttribute(k_gemm_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    configured_for[dev] = 1;
  }
  dim3 grid(row_tiles, splits);
  k_gemm_tc<<<grid, kTcThreads, smem, stream>>>(tx, ty0, ty1, p);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace dora
