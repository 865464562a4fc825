// norm_simt.cu -- fp32-input pieces of the factored norm on CUDA cores, plus
// the small kernels shared by both input types (row sum of squares for the
// s = 0 branch and the finalize).
//
// The fp32 path computes the same three terms as the bf16 tensor-core path
// ("Scaling DoRA", Chinese write-up section 1.2.1; Algorithm 1, section 5.1)
// with plain fp32 FMA: U = W A^T tile by tile with the base sum of squares
// and rowsum(B o U) fused into the tile epilogue, G = A A^T, and
// rowsum((B G) o B).  Products of fp32 inputs are rounded here (unlike bf16
// products), so the K loop keeps 64x64 output tiles with fp32 accumulators
// and the sum of squares is accumulated per 16-column chunk, then
// compensated.
#include "common.cuh"
#include "finalize.cuh"
#include "ptx.cuh"

namespace dora {

namespace {

constexpr int kT = kSimtTile;   // 64x64 output tile
constexpr int kK = 16;          // K chunk
constexpr int kPad = 4;

__global__ void __launch_bounds__(256)
    k_gemm_simt(const float* __restrict__ X, const float* __restrict__ Y, int rows, int ncols,
                int K, const float* __restrict__ B, int ldb, float* __restrict__ out_sumsq,
                float* __restrict__ out_dot, float* __restrict__ out_store, int mode) {
  __shared__ __align__(16) float Xs[kK][kT + kPad];
  __shared__ __align__(16) float Ys[kK][kT + kPad];
  const int t = threadIdx.x;
  const int tx = t & 15, ty = t >> 4;
  const int row0 = blockIdx.x * kT, col0 = blockIdx.y * kT;
  const bool do_sumsq = (mode & kSimtSumSq) && blockIdx.y == 0;

  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  float ss = 0.f, ss_c = 0.f;

  // loader mapping: 64 rows x 16 k = 256 float4 lanes? 64*16/4 = 256 -> one float4 per thread
  const int lr = t >> 2;          // 0..63 tile row
  const int lk = (t & 3) * 4;     // 0,4,8,12
  for (int k0 = 0; k0 < K; k0 += kK) {
    float4 xv = make_float4(0.f, 0.f, 0.f, 0.f), yv = xv;
    const int gk = k0 + lk;
    if (row0 + lr < rows) {
      const float* src = X + static_cast<size_t>(row0 + lr) * K + gk;
      if (gk + 3 < K) xv = *reinterpret_cast<const float4*>(src);
      else {
        float tmp[4] = {0.f, 0.f, 0.f, 0.f};
        for (int e = 0; e < 4; ++e) if (gk + e < K) tmp[e] = src[e];
        xv = make_float4(tmp[0], tmp[1], tmp[2], tmp[3]);
      }
    }
    if (col0 + lr < ncols) {
      const float* src = Y + static_cast<size_t>(col0 + lr) * K + gk;
      if (gk + 3 < K) yv = *reinterpret_cast<const float4*>(src);
      else {
        float tmp[4] = {0.f, 0.f, 0.f, 0.f};
        for (int e = 0; e < 4; ++e) if (gk + e < K) tmp[e] = src[e];
        yv = make_float4(tmp[0], tmp[1], tmp[2], tmp[3]);
      }
    }
    __syncthreads();
    Xs[lk + 0][lr] = xv.x; Xs[lk + 1][lr] = xv.y; Xs[lk + 2][lr] = xv.z; Xs[lk + 3][lr] = xv.w;
    Ys[lk + 0][lr] = yv.x; Ys[lk + 1][lr] = yv.y; Ys[lk + 2][lr] = yv.z; Ys[lk + 3][lr] = yv.w;
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kK; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&Xs[kk][ty * 4]);
      const float4 b = *reinterpret_cast<const float4*>(&Ys[kk][tx * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w};
      const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    if (do_sumsq && t < kT) {
      float part = 0.f;
#pragma unroll
      for (int kk = 0; kk < kK; ++kk) part = fmaf(Xs[kk][t], Xs[kk][t], part);
      kahan_add(ss, ss_c, part);
    }
  }

  if (do_sumsq && t < kT && row0 + t < rows) out_sumsq[row0 + t] = ss;

  if (mode & kSimtDotB) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = row0 + ty * 4 + i;
      float part = 0.f;
      if (row < rows) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int col = col0 + tx * 4 + j;
          if (col < ncols) part = fmaf(acc[i][j], B[static_cast<size_t>(row) * ldb + col], part);
        }
      }
      // the 16 threads sharing `ty` are 16 consecutive lanes of one warp
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) part += __shfl_xor_sync(0xFFFFFFFFu, part, off);
      if (tx == 0 && row < rows) out_dot[static_cast<size_t>(blockIdx.y) * rows + row] = part;
    }
  }
  if (mode & kSimtStore) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = row0 + ty * 4 + i;
      if (row >= rows) continue;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int col = col0 + tx * 4 + j;
        if (col < ncols) out_store[static_cast<size_t>(row) * ncols + col] = acc[i][j];
      }
    }
  }
}

// One warp per row: sum of squares of a [rows x cols] matrix.
template <bool BF16>
__global__ void __launch_bounds__(256)
    k_row_sumsq(const void* __restrict__ X, int64_t rows, int64_t cols, float* __restrict__ out) {
  const int64_t row = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float acc = 0.f, acc_c = 0.f;
  if (BF16) {
    const uint16_t* p = static_cast<const uint16_t*>(X) + row * cols;
    const int64_t nvec = cols / 8;   // 16-byte chunks (cols*2 is a multiple of 16)
    const uint4* pv = reinterpret_cast<const uint4*>(p);
    for (int64_t v = lane; v < nvec; v += 32) {
      const uint4 x = __ldcs(pv + v);
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
      float part = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        part = fmaf(bf16_lo(w[e]), bf16_lo(w[e]), part);
        part = fmaf(bf16_hi(w[e]), bf16_hi(w[e]), part);
      }
      kahan_add(acc, acc_c, part);
    }
    for (int64_t c = nvec * 8 + lane; c < cols; c += 32) {
      const float f = bf16_to_f32(p[c]);
      kahan_add(acc, acc_c, f * f);
    }
  } else {
    const float* p = static_cast<const float*>(X) + row * cols;
    const int64_t nvec = cols / 4;
    const float4* pv = reinterpret_cast<const float4*>(p);
    for (int64_t v = lane; v < nvec; v += 32) {
      const float4 x = __ldcs(pv + v);
      float part = x.x * x.x;
      part = fmaf(x.y, x.y, part);
      part = fmaf(x.z, x.z, part);
      part = fmaf(x.w, x.w, part);
      kahan_add(acc, acc_c, part);
    }
    for (int64_t c = nvec * 4 + lane; c < cols; c += 32) kahan_add(acc, acc_c, p[c] * p[c]);
  }
  acc = __fsub_rn(acc, acc_c);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
  if (lane == 0) out[row] = acc;
}

// sum of n fp32 partials in split order, as a double-float
__device__ __forceinline__ df sum_parts(const float* __restrict__ p, int n, int64_t stride,
                                        int64_t j) {
  float v[kMaxFinalParts];
#pragma unroll
  for (int i = 0; i < kMaxFinalParts; ++i) v[i] = i < n ? __ldg(p + i * stride + j) : 0.f;
  return df_sum_in_order(v);
}

// One thread per output row: the finalize step written out in finalize.cuh.
__global__ void __launch_bounds__(64)
    k_finalize(int64_t d_out, const float* __restrict__ pbase, int n_base,
               const float* __restrict__ pcross, int n_cross, const float* __restrict__ pba,
               int n_ba, float two_s, float s_sq, const void* __restrict__ m, int is_bf16,
               float eps, float* __restrict__ wnorm, float* __restrict__ g) {
  // launched as a programmatic dependent of the pass that wrote the partials
  griddep_wait();
  const int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (j >= d_out) return;
  const df base = sum_parts(pbase, n_base, d_out, j);
  const df cross = sum_parts(pcross, n_cross, d_out, j);
  const df ba = n_ba > 0 ? sum_parts(pba, n_ba, d_out, j) : df{0.f, 0.f};
  const float mj = is_bf16 ? bf16_to_f32(static_cast<const uint16_t*>(m)[j])
                           : static_cast<const float*>(m)[j];
  finalize_row(base, cross, n_ba > 0 ? &ba : nullptr, two_s, s_sq, mj, eps, wnorm[j], g[j]);
}

}  // namespace

cudaError_t launch_gemm_simt(const float* X, const float* Y, int rows, int ncols, int K,
                             const float* B, int ldb, float* out_sumsq, float* out_dot,
                             float* out_store, int mode, cudaStream_t stream) {
  dim3 grid((rows + kT - 1) / kT, (ncols + kT - 1) / kT);
  k_gemm_simt<<<grid, 256, 0, stream>>>(X, Y, rows, ncols, K, B, ldb, out_sumsq, out_dot,
                                        out_store, mode);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_row_sumsq(const void* X, int is_bf16, int64_t rows, int64_t cols, float* out,
                             cudaStream_t stream) {
  const int64_t threads = rows * 32;
  const unsigned blocks = static_cast<unsigned>((threads + 255) / 256);
  if (is_bf16) k_row_sumsq<true><<<blocks, 256, 0, stream>>>(X, rows, cols, out);
  else k_row_sumsq<false><<<blocks, 256, 0, stream>>>(X, rows, cols, out);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_finalize(int64_t d_out, const float* pbase, int n_base, const float* pcross,
                            int n_cross, const float* pba, int n_ba, float s, const void* m,
                            int is_bf16, float eps, float* wnorm, float* g,
                            cudaStream_t stream) {
  if (n_base > kMaxFinalParts || n_cross > kMaxFinalParts || n_ba > kMaxFinalParts)
    return cudaErrorInvalidValue;
  const unsigned blocks = static_cast<unsigned>((d_out + 63) / 64);
  // 2s and s^2 are exact in fp32 for the power-of-two scales; otherwise they
  // carry one rounding each, far below the fp32 result's own rounding
  // may start while the producing kernel still runs; griddep_wait in the
  // kernel holds every read until that kernel has finished
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks, 1, 1);
  cfg.blockDim = dim3(64, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, k_finalize, d_out, pbase, n_base, pcross,
                                           n_cross, pba, n_ba, 2.f * s, s * s, m, is_bf16, eps,
                                           wnorm, g);
  note_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dora
