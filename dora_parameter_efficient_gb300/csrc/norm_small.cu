// norm_small.cu -- the small kernels of the factored norm shared by both input
// types: the row sum of squares of W for the s = 0 branch (Algorithm 1 of
// the Chinese write-up, section 5.1, notes: no U and no G when s = 0) and
// the stand-alone finalize of finalize.cuh, which adds the K-segment
// partials of the fp32 pass in segment order and assembles wnorm and g.
// Also the self-test of the device-side failure detection.
#include "common.cuh"
#include "finalize.cuh"
#include "ptx.cuh"

namespace dora {

namespace {

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

// sum of n fp32 partials in split order, as a double-float, after `first`
// (0 when there is nothing ahead of the splits)
__device__ __forceinline__ df sum_parts(const float* __restrict__ p, int n, int64_t stride,
                                        int64_t j, float first = 0.f) {
  float v[kMaxFinalParts];
#pragma unroll
  for (int i = 0; i < kMaxFinalParts; ++i) v[i] = i < n ? __ldg(p + i * stride + j) : 0.f;
  df acc{first, 0.f};
#pragma unroll
  for (int i = 0; i < kMaxFinalParts; ++i) {
    float e;
    two_sum(acc.hi, v[i], acc.hi, e);
    acc.lo = __fadd_rn(acc.lo, e);
  }
  return acc;
}

// One thread per output row: the finalize step written out in finalize.cuh.
__global__ void __launch_bounds__(64)
    k_finalize(int64_t d_out, const float* __restrict__ pbase, int n_base,
               const float* __restrict__ pcross, int n_cross, const float* __restrict__ pba,
               int n_ba, float two_s, float s_sq, const void* __restrict__ m, int is_bf16,
               float eps, float* __restrict__ wnorm, float* __restrict__ g,
               const float* __restrict__ ext_base, const float* __restrict__ ext_cross) {
  // launched as a programmatic dependent of the pass that wrote the partials
  griddep_wait();
  const int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (j >= d_out) return;
  // partials of the whole d_in range summed by the caller come first
  const df base = sum_parts(pbase, n_base, d_out, j, ext_base ? ext_base[j] : 0.f);
  const df cross = sum_parts(pcross, n_cross, d_out, j, ext_cross ? ext_cross[j] : 0.f);
  const df ba = n_ba > 0 ? sum_parts(pba, n_ba, d_out, j) : df{0.f, 0.f};
  const float mj = is_bf16 ? bf16_to_f32(static_cast<const uint16_t*>(m)[j])
                           : static_cast<const float*>(m)[j];
  finalize_row(base, cross, n_ba > 0 ? &ba : nullptr, two_s, s_sq, mj, eps, wnorm[j], g[j]);
}

// One thread per row: the split partials of base and cross summed in split
// order (double-float) and rounded once to fp32 -- the partials of one d_in
// slice that a caller adds across slices.
__global__ void __launch_bounds__(64)
    k_sum_partials(int64_t d_out, const float* __restrict__ pbase, int n_base,
                   const float* __restrict__ pcross, int n_cross, float* __restrict__ sum_base,
                   float* __restrict__ sum_cross) {
  griddep_wait();
  const int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (j >= d_out) return;
  const df base = sum_parts(pbase, n_base, d_out, j);
  const df cross = sum_parts(pcross, n_cross, d_out, j);
  sum_base[j] = __fadd_rn(base.hi, base.lo);
  sum_cross[j] = __fadd_rn(cross.hi, cross.lo);
}

// G' = scale * G for a fp32 G [r x r], split into bf16 G'_hi = bf16(G'),
// G'_lo = bf16(G' - G'_hi), [rp x rp] with zeros outside [r x r] -- the two
// terms the bf16 main pass folds into its K loop.
__global__ void __launch_bounds__(256)
    k_gram_split(const float* __restrict__ G, int r, int rp, float scale,
                 uint16_t* __restrict__ G_hi, uint16_t* __restrict__ G_lo) {
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<int64_t>(rp) * rp) return;
  const int i = static_cast<int>(idx / rp);
  const int j = static_cast<int>(idx - static_cast<int64_t>(i) * rp);
  uint16_t h = 0, l = 0;
  if (i < r && j < r) {
    const float v = __fmul_rn(scale, G[static_cast<int64_t>(i) * r + j]);
    h = f32_to_bf16_rn(v);
    l = f32_to_bf16_rn(__fsub_rn(v, bf16_to_f32(h)));
  }
  G_hi[idx] = h;
  G_lo[idx] = l;
}

// Zeroes the control words at the head of a norm workspace (the status word,
// the main pass's work counter and its completion counters).  It lets the
// next kernel of the norm -- launched as its programmatic dependent -- start
// at once; that kernel waits for this one (griddep_wait) before anything that
// depends on the zeros.  A kernel, not cudaMemsetAsync: on one GB300 the
// memset took about 3 us more per norm inside a CUDA graph and broke the
// programmatic chain in a stream.
__global__ void __launch_bounds__(256) k_zero_words(int* __restrict__ p, int n) {
  // itself a programmatic dependent of the previous work in the stream, which
  // may still use this workspace (the previous norm on it): zero afterwards
  griddep_wait();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) p[i] = 0;
  // only now may the Gram kernel's CTAs (most of an SM's shared memory
  // each) become resident, so that they never hold SMs the previous kernel
  // still has blocks waiting for
  griddep_launch_dependents();
}

// One thread waits, with the pipelines' bounded wait, on an mbarrier that
// nothing arrives on; when the limit passes it records the timeout in the
// status word, as a pipeline role does, and the kernel returns.
__global__ void k_selftest_timeout(int* status, unsigned long long timeout_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait(&bar, 0u, global_timer_ns() + timeout_ns)) atomicExch(status, kStatusTimeout);
  }
}

}  // namespace

cudaError_t launch_zero_words(int* p, int n, cudaStream_t stream) {
  const int blocks = n <= 2048 ? 1 : (n + 2047) / 2048 < 64 ? (n + 2047) / 2048 : 64;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, k_zero_words, p, n);
  note_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_selftest_timeout(int* status, unsigned long long timeout_ns,
                                    cudaStream_t stream) {
  k_selftest_timeout<<<1, 32, 0, stream>>>(status, timeout_ns);
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
                            cudaStream_t stream, const float* ext_base,
                            const float* ext_cross) {
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
                                           wnorm, g, ext_base, ext_cross);
  note_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_sum_partials(int64_t d_out, const float* pbase, int n_base,
                                const float* pcross, int n_cross, float* sum_base,
                                float* sum_cross, cudaStream_t stream) {
  if (n_base > kMaxFinalParts || n_cross > kMaxFinalParts) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((d_out + 63) / 64), 1, 1);
  cfg.blockDim = dim3(64, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, k_sum_partials, d_out, pbase, n_base, pcross,
                                           n_cross, sum_base, sum_cross);
  note_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_gram_split(const float* G, int r, int rp, float scale, uint16_t* G_hi,
                              uint16_t* G_lo, cudaStream_t stream) {
  const int64_t n = static_cast<int64_t>(rp) * rp;
  k_gram_split<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(G, r, rp, scale, G_hi,
                                                                           G_lo);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace dora
