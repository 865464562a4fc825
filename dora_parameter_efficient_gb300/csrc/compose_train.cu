// compose_train.cu -- the training path of the stable compose: a forward
// that also keeps `inner`, and a dual-output backward with the magnitude
// gradient as a deterministic column reduction.
//
// "Scaling DoRA", Chinese write-up sections 2.2, 4.2 and 5.2 (the fused
// backward tier): the forward keeps one activation-sized tensor, inner, for
// the magnitude gradient; the backward writes two outputs, the gradients of
// the base and adapter branches; dmag is a separate column sum, not float
// atomics, so it is the same on every run; with the magnitude frozen, inner
// and dmag are skipped.  The norm is a detached constant (section 1.2.2), so
//
//   forward   out   = (g - 1) * base + g * (s * lora)     (as compose.cu)
//             inner = base + s * lora                      (d out / d g)
//   backward  d_base = (g - 1) * d_out,  d_lora = g * s * d_out
//             dmag_j = sum_t d_out_tj * inner_tj / max(wnorm_j, eps)
//
// All four are HBM streams.  Layout: [T x d_out] row-major, g per column.
// Rows of 16-byte vectors stream through the column kernels: a thread keeps
// one column vector (8 bf16 or 4 fp32 columns) and its g values in registers
// and walks rows y, y + gridDim.y, ...; the backward thread also keeps the
// fp32 partial column sums of d_out * inner for its rows and writes them,
// one row of partials per blockIdx.y, for a second kernel to add in blockIdx.y
// order (compensated) and divide.  The column kernels launch as programmatic
// dependents of the preceding work.  Anything else takes element-wise kernels
// with the same arithmetic.
#include "common.cuh"
#include "ptx.cuh"

namespace dora {

namespace {

constexpr int kTrainThreads = 256;     // column vectors per block
// rows per thread and round of the forward, with two blocks per SM (on one
// GB300 at 2048 x 8192 bf16, back to back: 24.1 us with four rows and four
// blocks per SM, 23.6 with eight and two)
constexpr int kRowsInFlight = 8;

// stable compose of one element ((g - 1) passed in), as in compose.cu
__device__ __forceinline__ float compose_el(float b, float l, float g, float gm1, float s) {
  const float sl = __fmul_rn(s, l);
  const float sl_err = fmaf(s, l, -sl);
  const float p = __fmul_rn(gm1, b);
  const float p_err = fmaf(gm1, b, -p);
  return __fadd_rn(fmaf(g, sl, p), fmaf(g, sl_err, p_err));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

template <bool BF16>
struct Vec;
template <>
struct Vec<true> {
  static constexpr int N = 8;
  __device__ static void unpack(const uint4& v, float (&x)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[2 * e] = bf16_lo(w[e]);
      x[2 * e + 1] = bf16_hi(w[e]);
    }
  }
  __device__ static uint4 pack(const float (&x)[8]) {
    return make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                      pack_bf16x2(x[6], x[7]));
  }
};
template <>
struct Vec<false> {
  static constexpr int N = 4;
  __device__ static void unpack(const uint4& v, float (&x)[4]) {
    x[0] = __uint_as_float(v.x);
    x[1] = __uint_as_float(v.y);
    x[2] = __uint_as_float(v.z);
    x[3] = __uint_as_float(v.w);
  }
  __device__ static uint4 pack(const float (&x)[4]) {
    return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                      __float_as_uint(x[3]));
  }
};

template <bool BF16>
__device__ __forceinline__ float load_el(const void* p, int64_t i) {
  if (BF16) return bf16_to_f32(static_cast<const uint16_t*>(p)[i]);
  return static_cast<const float*>(p)[i];
}
template <bool BF16>
__device__ __forceinline__ void store_el(void* p, int64_t i, float v) {
  if (BF16) static_cast<uint16_t*>(p)[i] = f32_to_bf16_rn(v);
  else static_cast<float*>(p)[i] = v;
}

// ------------------------------------------------------------------ forward
// Column kernel: thread (blockIdx.x, threadIdx.x) owns column vector c; rows
// blockIdx.y, blockIdx.y + gridDim.y, ...
template <bool BF16>
__global__ void __launch_bounds__(kTrainThreads, 2)
    k_train_fwd_cols(const uint4* __restrict__ base, const uint4* __restrict__ lora,
                     const float* __restrict__ g, float s, int64_t T, int64_t dv,
                     uint4* __restrict__ out, uint4* __restrict__ inner) {
  constexpr int N = Vec<BF16>::N;
  // launched as a programmatic dependent of whatever precedes it (the norm
  // that wrote g): resident early, but nothing is read or written before
  // that grid has finished
  griddep_wait();
  const int64_t c = static_cast<int64_t>(blockIdx.x) * kTrainThreads + threadIdx.x;
  if (c >= dv) return;
  float gv[N], gm[N];
#pragma unroll
  for (int e = 0; e < N; ++e) {
    gv[e] = __ldg(g + c * N + e);
    gm[e] = __fsub_rn(gv[e], 1.0f);
  }
  const int64_t rstep = gridDim.y;
  for (int64_t r0 = blockIdx.y; r0 < T; r0 += rstep * kRowsInFlight) {
    uint4 bv[kRowsInFlight], lv[kRowsInFlight];
#pragma unroll
    for (int u = 0; u < kRowsInFlight; ++u) {
      const int64_t r = r0 + u * rstep;
      if (r < T) {
        bv[u] = __ldcs(base + r * dv + c);
        lv[u] = __ldcs(lora + r * dv + c);
      }
    }
#pragma unroll
    for (int u = 0; u < kRowsInFlight; ++u) {
      const int64_t r = r0 + u * rstep;
      if (r >= T) continue;
      float b[N], l[N], o[N], in[N];
      Vec<BF16>::unpack(bv[u], b);
      Vec<BF16>::unpack(lv[u], l);
#pragma unroll
      for (int e = 0; e < N; ++e) {
        o[e] = compose_el(b[e], l[e], gv[e], gm[e], s);
        in[e] = fmaf(s, l[e], b[e]);          // base + s * lora, one rounding
      }
      __stcs(out + r * dv + c, Vec<BF16>::pack(o));
      __stcs(inner + r * dv + c, Vec<BF16>::pack(in));
    }
  }
  // the next kernel of the stream (the backward) may launch; it waits for
  // this grid before it reads
  griddep_launch_dependents();
}

template <bool BF16>
__global__ void __launch_bounds__(256)
    k_train_fwd_any(const void* __restrict__ base, const void* __restrict__ lora,
                    const float* __restrict__ g, float s, int64_t T, int64_t d_out,
                    void* __restrict__ out, void* __restrict__ inner) {
  const int64_t n = T * d_out;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += stride) {
    const float gj = g[i % d_out];
    const float b = load_el<BF16>(base, i), l = load_el<BF16>(lora, i);
    store_el<BF16>(out, i, compose_el(b, l, gj, __fsub_rn(gj, 1.0f), s));
    store_el<BF16>(inner, i, fmaf(s, l, b));
  }
}

// ------------------------------------------------------------------ backward
// d_base = (g - 1) * d_out, d_lora = g * (s * d_out), each one rounding of an
// fp32 product chain; with DM, the partial column sums of d_out * inner
// (bf16 products are exact in fp32) over this thread's rows go to
// partials[blockIdx.y][column].
template <bool BF16, bool DM>
__global__ void __launch_bounds__(kTrainThreads, 2)
    k_train_bwd_cols(const uint4* __restrict__ dout, const uint4* __restrict__ inner,
                     const float* __restrict__ g, float s, int64_t T, int64_t dv,
                     uint4* __restrict__ d_base, uint4* __restrict__ d_lora,
                     float* __restrict__ partials) {
  constexpr int N = Vec<BF16>::N;
  // the finish kernel may be scheduled as blocks of this grid exit; it
  // waits for the whole grid (griddep_wait) before reading the partials
  if (DM) griddep_launch_dependents();
  // itself a programmatic dependent of the preceding work (the forward that
  // wrote inner): nothing is read or written before that grid has finished
  griddep_wait();
  const int64_t c = static_cast<int64_t>(blockIdx.x) * kTrainThreads + threadIdx.x;
  if (c >= dv) return;
  float gv[N], gm[N], acc[N];
#pragma unroll
  for (int e = 0; e < N; ++e) {
    gv[e] = __ldg(g + c * N + e);
    gm[e] = __fsub_rn(gv[e], 1.0f);
    acc[e] = 0.f;
  }
  const int64_t rstep = gridDim.y;
  // eight rows in flight with two blocks per SM: the same bytes in flight as
  // the forward's four with four blocks, and half the rows of partials for
  // the finish kernel (2048 x 8192 on one GB300: 31.5 -> 29.3 us)
  constexpr int kRowsInFlightB = 8;
  for (int64_t r0 = blockIdx.y; r0 < T; r0 += rstep * kRowsInFlightB) {
    uint4 dv_[kRowsInFlightB], iv[kRowsInFlightB];
#pragma unroll
    for (int u = 0; u < kRowsInFlightB; ++u) {
      const int64_t r = r0 + u * rstep;
      if (r < T) {
        dv_[u] = __ldcs(dout + r * dv + c);
        if (DM) iv[u] = __ldcs(inner + r * dv + c);
      }
    }
#pragma unroll
    for (int u = 0; u < kRowsInFlightB; ++u) {
      const int64_t r = r0 + u * rstep;
      if (r >= T) continue;
      float d[N], db[N], dl[N];
      Vec<BF16>::unpack(dv_[u], d);
#pragma unroll
      for (int e = 0; e < N; ++e) {
        db[e] = __fmul_rn(gm[e], d[e]);
        dl[e] = __fmul_rn(gv[e], __fmul_rn(s, d[e]));
      }
      __stcs(d_base + r * dv + c, Vec<BF16>::pack(db));
      __stcs(d_lora + r * dv + c, Vec<BF16>::pack(dl));
      if (DM) {
        float in[N];
        Vec<BF16>::unpack(iv[u], in);
#pragma unroll
        for (int e = 0; e < N; ++e) acc[e] = fmaf(d[e], in[e], acc[e]);
      }
    }
  }
  if (DM) {
    float* prow = partials + static_cast<int64_t>(blockIdx.y) * dv * N + c * N;
#pragma unroll
    for (int e = 0; e < N; ++e) prow[e] = acc[e];
  }
}

// Element-wise backward; with DM, block (x, y) covers rows y, y + gridDim.y,
// ... of the columns x * 256 + threadIdx.x, so the partials keep the same
// [gridDim.y][d_out] layout.
template <bool BF16, bool DM>
__global__ void __launch_bounds__(256)
    k_train_bwd_any(const void* __restrict__ dout, const void* __restrict__ inner,
                    const float* __restrict__ g, float s, int64_t T, int64_t d_out,
                    void* __restrict__ d_base, void* __restrict__ d_lora,
                    float* __restrict__ partials) {
  if (DM) griddep_launch_dependents();
  const int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (j >= d_out) return;
  const float gj = g[j], gm = __fsub_rn(gj, 1.0f);
  float acc = 0.f;
  for (int64_t r = blockIdx.y; r < T; r += gridDim.y) {
    const int64_t i = r * d_out + j;
    const float d = load_el<BF16>(dout, i);
    store_el<BF16>(d_base, i, __fmul_rn(gm, d));
    store_el<BF16>(d_lora, i, __fmul_rn(gj, __fmul_rn(s, d)));
    if (DM) acc = fmaf(d, load_el<BF16>(inner, i), acc);
  }
  if (DM) partials[static_cast<int64_t>(blockIdx.y) * d_out + j] = acc;
}

// dmag_j = (sum over p of partials[p][j]) / max(wnorm_j, eps).  A block of
// 1024 threads takes 32 columns: warp w sums parts [w n / 32, (w + 1) n / 32)
// for column lane (compensated; the at most 8 loads of a warp's range are
// all issued before the first add), then warp 0 adds the 32 warp sums in
// warp order.  The order depends only on n: the same result on every call.
// The pass runs after the backward's last block, so its time is the latency
// of those few loads: 32 warps per block (about 2.4 parts each at 76 row
// blocks) against 8 took the backward with dmag from 29.2 to 27.9 us at
// 2048 x 8192 on one GB300.  Launched as a programmatic dependent of the
// backward kernel.
constexpr int kFinishCols = 32;
constexpr int kFinishWarps = 32;
constexpr int kFinishPartsPerWarp = (kMaxDmParts + kFinishWarps - 1) / kFinishWarps;

__global__ void __launch_bounds__(kFinishCols * kFinishWarps)
    k_train_dm_finish(const float* __restrict__ partials, int nparts, int64_t d_out,
                      const float* __restrict__ wnorm, float eps, float* __restrict__ dmag) {
  __shared__ float ws_sum[kFinishWarps][kFinishCols], ws_cmp[kFinishWarps][kFinishCols];
  griddep_wait();            // the partials of the backward kernel
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t j = static_cast<int64_t>(blockIdx.x) * kFinishCols + lane;
  const bool ok = j < d_out;
  const int p0 = (nparts * w) / kFinishWarps, p1 = (nparts * (w + 1)) / kFinishWarps;
  float v[kFinishPartsPerWarp];
#pragma unroll
  for (int u = 0; u < kFinishPartsPerWarp; ++u)
    v[u] = (ok && p0 + u < p1) ? partials[static_cast<int64_t>(p0 + u) * d_out + j] : 0.f;
  float sum = 0.f, comp = 0.f;
#pragma unroll
  for (int u = 0; u < kFinishPartsPerWarp; ++u)
    if (p0 + u < p1) kahan_add(sum, comp, v[u]);
  ws_sum[w][lane] = sum;
  ws_cmp[w][lane] = comp;
  __syncthreads();
  if (w == 0 && ok) {
    float s2 = 0.f, c2 = 0.f;
#pragma unroll
    for (int q = 0; q < kFinishWarps; ++q) {
      kahan_add(s2, c2, ws_sum[q][lane]);
      kahan_add(s2, c2, -ws_cmp[q][lane]);
    }
    const float wv = wnorm[j];
    dmag[j] = __fdiv_rn(__fsub_rn(s2, c2), (wv > eps) ? wv : eps);
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// rows of blocks for a column grid of `xblocks`: about kBlocksPerSm blocks per
// SM in one wave, at most max_parts and at most T
int64_t row_blocks(int64_t xblocks, int64_t T, int num_sms, int64_t max_parts) {
  constexpr int kBlocksPerSm = 4;
  const int64_t target = static_cast<int64_t>(num_sms > 0 ? num_sms : 148) * kBlocksPerSm;
  int64_t y = (target + xblocks - 1) / xblocks;
  if (y > max_parts) y = max_parts;
  if (y > T) y = T;
  if (y > 65535) y = 65535;
  return y < 1 ? 1 : y;
}

}  // namespace

cudaError_t launch_compose_train(const void* base, const void* lora, const float* g, float s,
                                 int is_bf16, int64_t T, int64_t d_out, void* out, void* inner,
                                 int num_sms, cudaStream_t stream) {
  if (T == 0 || d_out == 0) return cudaSuccess;
  const int epv = is_bf16 ? 8 : 4;
  const bool vec = d_out % epv == 0 && aligned16(base) && aligned16(lora) && aligned16(out) &&
                   aligned16(inner);
  if (vec) {
    const int64_t dv = d_out / epv;
    const int64_t xb = (dv + kTrainThreads - 1) / kTrainThreads;
    const dim3 grid(static_cast<unsigned>(xb),
                    static_cast<unsigned>(row_blocks(xb, T, num_sms / 2, 65535)));  // 2 per SM
    // a programmatic dependent of the preceding work: on one GB300 the
    // forward back to back took 26.0 -> 24.1 us and the backward with dmag
    // 24.9 -> 22.7 us at 2048 x 8192 bf16 (its launch and ramp overlap the
    // previous kernel's tail)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kTrainThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const uint4* bp = static_cast<const uint4*>(base);
    const uint4* lp = static_cast<const uint4*>(lora);
    uint4* op = static_cast<uint4*>(out);
    uint4* ip = static_cast<uint4*>(inner);
    const cudaError_t le = is_bf16 ? cudaLaunchKernelEx(&cfg, k_train_fwd_cols<true>, bp, lp, g, s, T, dv, op, ip)
                                   : cudaLaunchKernelEx(&cfg, k_train_fwd_cols<false>, bp, lp, g, s, T, dv, op, ip);
    if (le != cudaSuccess) return le;
  } else {
    const int64_t n = T * d_out;
    int64_t blocks = (n + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms > 0 ? num_sms : 148) * 8;
    if (blocks > cap) blocks = cap;
    if (is_bf16)
      k_train_fwd_any<true><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
          base, lora, g, s, T, d_out, out, inner);
    else
      k_train_fwd_any<false><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
          base, lora, g, s, T, d_out, out, inner);
  }
  note_launches(1);
  return cudaGetLastError();
}

int64_t compose_backward_parts(int64_t T) {
  return T < kMaxDmParts ? (T > 0 ? T : 1) : kMaxDmParts;
}

cudaError_t launch_compose_backward(const void* dout, const void* inner, const float* g,
                                    const float* wnorm, float eps, float s, int is_bf16,
                                    int64_t T, int64_t d_out, void* d_base, void* d_lora,
                                    float* dmag, float* partials, int num_sms,
                                    cudaStream_t stream) {
  if (T == 0 || d_out == 0) return cudaSuccess;
  const bool dm = dmag != nullptr;
  const int epv = is_bf16 ? 8 : 4;
  const bool vec = d_out % epv == 0 && aligned16(dout) && aligned16(d_base) &&
                   aligned16(d_lora) && (!dm || aligned16(inner));
  const int64_t max_parts = compose_backward_parts(T);
  int64_t nparts;
  if (vec) {
    const int64_t dv = d_out / epv;
    const int64_t xb = (dv + kTrainThreads - 1) / kTrainThreads;
    nparts = row_blocks(xb, T, num_sms / 2, max_parts);   // two blocks per SM
    const dim3 grid(static_cast<unsigned>(xb), static_cast<unsigned>(nparts));
    const uint4* dp = static_cast<const uint4*>(dout);
    const uint4* ip = static_cast<const uint4*>(inner);
    uint4* bp = static_cast<uint4*>(d_base);
    uint4* lp = static_cast<uint4*>(d_lora);
    cudaLaunchConfig_t bcfg = {};
    bcfg.gridDim = grid;
    bcfg.blockDim = dim3(kTrainThreads, 1, 1);
    bcfg.stream = stream;
    cudaLaunchAttribute battr[1];
    battr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    battr[0].val.programmaticStreamSerializationAllowed = 1;
    bcfg.attrs = battr;
    bcfg.numAttrs = 1;
    cudaError_t le;
    if (is_bf16) le = dm ? cudaLaunchKernelEx(&bcfg, k_train_bwd_cols<true, true>, dp, ip, g, s, T, dv, bp, lp, partials)
                         : cudaLaunchKernelEx(&bcfg, k_train_bwd_cols<true, false>, dp, ip, g, s, T, dv, bp, lp, partials);
    else le = dm ? cudaLaunchKernelEx(&bcfg, k_train_bwd_cols<false, true>, dp, ip, g, s, T, dv, bp, lp, partials)
                 : cudaLaunchKernelEx(&bcfg, k_train_bwd_cols<false, false>, dp, ip, g, s, T, dv, bp, lp, partials);
    if (le != cudaSuccess) return le;
  } else {
    const int64_t xb = (d_out + 255) / 256;
    nparts = row_blocks(xb, T, num_sms, max_parts);
    const dim3 grid(static_cast<unsigned>(xb), static_cast<unsigned>(nparts));
    if (is_bf16) {
      if (dm) k_train_bwd_any<true, true><<<grid, 256, 0, stream>>>(dout, inner, g, s, T, d_out, d_base, d_lora, partials);
      else k_train_bwd_any<true, false><<<grid, 256, 0, stream>>>(dout, inner, g, s, T, d_out, d_base, d_lora, partials);
    } else {
      if (dm) k_train_bwd_any<false, true><<<grid, 256, 0, stream>>>(dout, inner, g, s, T, d_out, d_base, d_lora, partials);
      else k_train_bwd_any<false, false><<<grid, 256, 0, stream>>>(dout, inner, g, s, T, d_out, d_base, d_lora, partials);
    }
  }
  note_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || !dm) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((d_out + kFinishCols - 1) / kFinishCols), 1, 1);
  cfg.blockDim = dim3(kFinishCols * kFinishWarps, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, k_train_dm_finish, static_cast<const float*>(partials),
                         static_cast<int>(nparts), d_out, wnorm, eps, dmag);
  note_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dora
