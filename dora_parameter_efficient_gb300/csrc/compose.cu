// compose.cu -- the stable fused DoRA compose, a pure HBM stream.
//
//   out = (g - 1) * base + g * (s * lora)       ("Scaling DoRA", Chinese
//   write-up sections 2.1 / 2.1.1; English summary "Fused Kernels")
//
// One read of base, one of lora, one write of out; g (one fp32 per output
// feature, broadcast over tokens) stays in L1/L2.  The evaluation follows the
// write-up's order -- s * lora first, then g * (.) -- and keeps the small
// correction (g - 1) explicit, in fp32 registers.  Both products carry their
// exact rounding error (an error-free product via FMA, Dekker's TwoProduct),
// so the fp32 result is within about one fp32 ulp of the exact value before
// the single rounding to the output type, even where the two terms cancel.
//
// Layout: base/lora/out are [T x d_out] row-major.  Rows whose byte length is
// a multiple of 16 with 16-byte aligned pointers stream as 16-byte vectors
// (8 bf16 or 4 fp32 per load).  When a row holds a multiple of 256 vectors,
// each thread keeps one column vector for all its rows: its g values (and
// g - 1) stay in registers and no index arithmetic is left per element, so
// the kernel is bound by HBM, not by instruction issue.  Other vector shapes
// take a grid-stride loop, and anything unaligned the element-wise loop.
// Grids are sized to a multiple of the SM count.
#include "common.cuh"
#include "ptx.cuh"

namespace dora {

namespace {

// (g - 1) is passed in: exact for g in [0.5, 2] (Sterbenz), one rounding otherwise
__device__ __forceinline__ float compose1m(float b, float l, float g, float gm1, float s) {
  const float sl = __fmul_rn(s, l);
  const float sl_err = fmaf(s, l, -sl);          // s*l = sl + sl_err exactly
  const float p = __fmul_rn(gm1, b);
  const float p_err = fmaf(gm1, b, -p);          // (g-1)*b = p + p_err exactly
  return __fadd_rn(fmaf(g, sl, p), fmaf(g, sl_err, p_err));
}

__device__ __forceinline__ float compose1(float b, float l, float g, float s) {
  const float gm1 = __fsub_rn(g, 1.0f);          // exact for g in [0.5, 2] (Sterbenz)
  const float sl = __fmul_rn(s, l);
  const float sl_err = fmaf(s, l, -sl);          // s*l = sl + sl_err exactly
  const float p = __fmul_rn(gm1, b);
  const float p_err = fmaf(gm1, b, -p);          // (g-1)*b = p + p_err exactly
  return __fadd_rn(fmaf(g, sl, p), fmaf(g, sl_err, p_err));
}

constexpr int kUnroll = 4;
constexpr int kColThreads = 256;     // column vectors per block of the fixed-column kernel
constexpr int kRowUnroll = 4;

// two floats -> packed bf16x2 (lo in the low half), each rounded to nearest even
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// Fixed-column stream: block (x, y) owns column vectors [x * 256, x * 256 + 256)
// and rows y, y + gridDim.y, ...; requires d_out / EPV to be a multiple of 256.
template <bool BF16>
__global__ void __launch_bounds__(kColThreads, 4)
    k_compose_cols(const uint4* __restrict__ base, const uint4* __restrict__ lora,
                   const float* __restrict__ g, float s, int64_t T, int64_t dv,
                   uint4* __restrict__ out) {
  // launched as a programmatic dependent of whatever precedes it: the blocks
  // may be resident before that grid ends, but read nothing until it has
  griddep_wait();
  constexpr int EPV = BF16 ? 8 : 4;
  const int64_t c = static_cast<int64_t>(blockIdx.x) * kColThreads + threadIdx.x;
  float gv[EPV], gm[EPV];
#pragma unroll
  for (int q = 0; q < EPV / 4; ++q) {
    const float4 t = __ldg(reinterpret_cast<const float4*>(g + c * EPV) + q);
    gv[4 * q] = t.x;
    gv[4 * q + 1] = t.y;
    gv[4 * q + 2] = t.z;
    gv[4 * q + 3] = t.w;
  }
#pragma unroll
  for (int e = 0; e < EPV; ++e) gm[e] = __fsub_rn(gv[e], 1.0f);
  const int64_t rstep = gridDim.y;
  for (int64_t r0 = blockIdx.y; r0 < T; r0 += rstep * kRowUnroll) {
    uint4 bv[kRowUnroll], lv[kRowUnroll];
#pragma unroll
    for (int u = 0; u < kRowUnroll; ++u) {
      const int64_t r = r0 + u * rstep;
      if (r < T) {
        bv[u] = __ldcs(base + r * dv + c);
        lv[u] = __ldcs(lora + r * dv + c);
      }
    }
#pragma unroll
    for (int u = 0; u < kRowUnroll; ++u) {
      const int64_t r = r0 + u * rstep;
      if (r >= T) continue;
      uint4 o;
      if (BF16) {
        const uint32_t bw[4] = {bv[u].x, bv[u].y, bv[u].z, bv[u].w};
        const uint32_t lw[4] = {lv[u].x, lv[u].y, lv[u].z, lv[u].w};
        uint32_t ow[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float lo = compose1m(bf16_lo(bw[e]), bf16_lo(lw[e]), gv[2 * e], gm[2 * e], s);
          const float hi =
              compose1m(bf16_hi(bw[e]), bf16_hi(lw[e]), gv[2 * e + 1], gm[2 * e + 1], s);
          ow[e] = pack_bf16x2_rn(lo, hi);
        }
        o = make_uint4(ow[0], ow[1], ow[2], ow[3]);
      } else {
        o.x = __float_as_uint(compose1m(__uint_as_float(bv[u].x), __uint_as_float(lv[u].x), gv[0], gm[0], s));
        o.y = __float_as_uint(compose1m(__uint_as_float(bv[u].y), __uint_as_float(lv[u].y), gv[1], gm[1], s));
        o.z = __float_as_uint(compose1m(__uint_as_float(bv[u].z), __uint_as_float(lv[u].z), gv[2], gm[2], s));
        o.w = __float_as_uint(compose1m(__uint_as_float(bv[u].w), __uint_as_float(lv[u].w), gv[3], gm[3], s));
      }
      __stcs(out + r * dv + c, o);
    }
  }
  // the next kernel of the stream may launch (it waits for this grid)
  griddep_launch_dependents();
}

template <bool BF16>
__global__ void __launch_bounds__(256)
    k_compose(const void* __restrict__ base, const void* __restrict__ lora,
              const float* __restrict__ g, float s, int64_t T, int64_t d_out,
              void* __restrict__ out, int vec_ok) {
  griddep_wait();
  const int64_t n = T * d_out;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  constexpr int EPV = BF16 ? 8 : 4;   // elements per 16-byte vector
  if (vec_ok) {
    const int64_t nv = n / EPV;
    const int64_t dv = d_out / EPV;    // vectors per row
    const uint4* bp = static_cast<const uint4*>(base);
    const uint4* lp = static_cast<const uint4*>(lora);
    uint4* op = static_cast<uint4*>(out);
    for (int64_t v0 = tid; v0 < nv; v0 += nthreads * kUnroll) {
      uint4 bv[kUnroll], lv[kUnroll];
      int64_t vi[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        vi[u] = v0 + u * nthreads;
        if (vi[u] < nv) {
          bv[u] = __ldcs(bp + vi[u]);
          lv[u] = __ldcs(lp + vi[u]);
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        if (vi[u] >= nv) continue;
        const int64_t col = (vi[u] % dv) * EPV;
        if (BF16) {
          const float4 g0 = __ldg(reinterpret_cast<const float4*>(g + col));
          const float4 g1 = __ldg(reinterpret_cast<const float4*>(g + col) + 1);
          const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
          const uint32_t bw[4] = {bv[u].x, bv[u].y, bv[u].z, bv[u].w};
          const uint32_t lw[4] = {lv[u].x, lv[u].y, lv[u].z, lv[u].w};
          uint32_t ow[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float lo = compose1(bf16_lo(bw[e]), bf16_lo(lw[e]), gv[2 * e], s);
            const float hi = compose1(bf16_hi(bw[e]), bf16_hi(lw[e]), gv[2 * e + 1], s);
            ow[e] = static_cast<uint32_t>(f32_to_bf16_rn(lo)) |
                    (static_cast<uint32_t>(f32_to_bf16_rn(hi)) << 16);
          }
          __stcs(op + vi[u], make_uint4(ow[0], ow[1], ow[2], ow[3]));
        } else {
          const float4 gv = __ldg(reinterpret_cast<const float4*>(g + col));
          float4 o;
          o.x = compose1(__uint_as_float(bv[u].x), __uint_as_float(lv[u].x), gv.x, s);
          o.y = compose1(__uint_as_float(bv[u].y), __uint_as_float(lv[u].y), gv.y, s);
          o.z = compose1(__uint_as_float(bv[u].z), __uint_as_float(lv[u].z), gv.z, s);
          o.w = compose1(__uint_as_float(bv[u].w), __uint_as_float(lv[u].w), gv.w, s);
          __stcs(reinterpret_cast<float4*>(op) + vi[u], o);
        }
      }
    }
  } else {
    for (int64_t i = tid; i < n; i += nthreads) {
      const int64_t col = i % d_out;
      if (BF16) {
        const uint16_t b = static_cast<const uint16_t*>(base)[i];
        const uint16_t l = static_cast<const uint16_t*>(lora)[i];
        static_cast<uint16_t*>(out)[i] =
            f32_to_bf16_rn(compose1(bf16_to_f32(b), bf16_to_f32(l), g[col], s));
      } else {
        const float b = static_cast<const float*>(base)[i];
        const float l = static_cast<const float*>(lora)[i];
        static_cast<float*>(out)[i] = compose1(b, l, g[col], s);
      }
    }
  }
  griddep_launch_dependents();
}

// Grouped compose over a module table: unit u = (module, 16-row block,
// 256-vector column block), numbered module by module; block b takes units
// b, b + gridDim.x, ...  A thread keeps one column vector and its g values
// for the unit's rows.  Requires 16-byte rows (d_out a multiple of 8 bf16 /
// 4 fp32) and 16-byte aligned pointers in every module.
constexpr int kGroupRows = 16;

template <bool BF16>
__global__ void __launch_bounds__(kColThreads)
    k_compose_grouped(const ComposeModule* __restrict__ mods, int n_mods, int64_t n_units,
                      float s) {
  constexpr int EPV = BF16 ? 8 : 4;
  for (int64_t u = blockIdx.x; u < n_units; u += gridDim.x) {
    int lo = 0, hi = n_mods - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (mods[mid].unit_begin <= u) lo = mid;
      else hi = mid - 1;
    }
    const ComposeModule& md = mods[lo];
    const int64_t dv = md.d_out / EPV;
    const int64_t xblocks = (dv + kColThreads - 1) / kColThreads;
    const int64_t local = u - md.unit_begin;
    const int64_t rb = local / xblocks;
    const int64_t c = (local - rb * xblocks) * kColThreads + threadIdx.x;
    if (c >= dv) continue;
    const uint4* base = static_cast<const uint4*>(md.base);
    const uint4* lora = static_cast<const uint4*>(md.lora);
    uint4* out = static_cast<uint4*>(md.out);
    float gv[EPV], gm[EPV];
#pragma unroll
    for (int e = 0; e < EPV; ++e) {
      gv[e] = __ldg(md.g + c * EPV + e);
      gm[e] = __fsub_rn(gv[e], 1.0f);
    }
    const int64_t r0 = rb * kGroupRows;
    const int64_t r1 = r0 + kGroupRows < md.T ? r0 + kGroupRows : md.T;
    for (int64_t rr = r0; rr < r1; rr += kRowUnroll) {
      uint4 bv[kRowUnroll], lv[kRowUnroll];
#pragma unroll
      for (int k = 0; k < kRowUnroll; ++k) {
        if (rr + k < r1) {
          bv[k] = __ldcs(base + (rr + k) * dv + c);
          lv[k] = __ldcs(lora + (rr + k) * dv + c);
        }
      }
#pragma unroll
      for (int k = 0; k < kRowUnroll; ++k) {
        if (rr + k >= r1) continue;
        uint4 o;
        if (BF16) {
          const uint32_t bw[4] = {bv[k].x, bv[k].y, bv[k].z, bv[k].w};
          const uint32_t lw[4] = {lv[k].x, lv[k].y, lv[k].z, lv[k].w};
          uint32_t ow[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            ow[e] = pack_bf16x2_rn(compose1m(bf16_lo(bw[e]), bf16_lo(lw[e]), gv[2 * e], gm[2 * e], s),
                                   compose1m(bf16_hi(bw[e]), bf16_hi(lw[e]), gv[2 * e + 1], gm[2 * e + 1], s));
          o = make_uint4(ow[0], ow[1], ow[2], ow[3]);
        } else {
          o.x = __float_as_uint(compose1m(__uint_as_float(bv[k].x), __uint_as_float(lv[k].x), gv[0], gm[0], s));
          o.y = __float_as_uint(compose1m(__uint_as_float(bv[k].y), __uint_as_float(lv[k].y), gv[1], gm[1], s));
          o.z = __float_as_uint(compose1m(__uint_as_float(bv[k].z), __uint_as_float(lv[k].z), gv[2], gm[2], s));
          o.w = __float_as_uint(compose1m(__uint_as_float(bv[k].w), __uint_as_float(lv[k].w), gv[3], gm[3], s));
        }
        __stcs(out + (rr + k) * dv + c, o);
      }
    }
  }
}

}  // namespace

int64_t compose_grouped_units(int64_t T, int64_t d_out, int is_bf16) {
  const int64_t dv = d_out / (is_bf16 ? 8 : 4);
  return ((T + kGroupRows - 1) / kGroupRows) * ((dv + kColThreads - 1) / kColThreads);
}

cudaError_t launch_compose_grouped(const ComposeModule* mods, int n_mods, int64_t n_units,
                                   float s, int is_bf16, int num_sms, cudaStream_t stream) {
  if (n_units == 0) return cudaSuccess;
  int64_t blocks = static_cast<int64_t>(num_sms > 0 ? num_sms : 148) * 4;
  if (blocks > n_units) blocks = n_units;
  if (is_bf16)
    k_compose_grouped<true><<<static_cast<unsigned>(blocks), kColThreads, 0, stream>>>(mods, n_mods, n_units, s);
  else
    k_compose_grouped<false><<<static_cast<unsigned>(blocks), kColThreads, 0, stream>>>(mods, n_mods, n_units, s);
  note_launches(1);
  return cudaGetLastError();
}

namespace {

// Launch as a programmatic dependent of the previous work in the stream: the
// grid is set up while that work finishes; the kernels wait (griddep_wait)
// before their first read.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), dim3 grid, dim3 block,
                             cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
  note_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_compose(const void* base, const void* lora, const float* g, float s,
                           int is_bf16, int64_t T, int64_t d_out, void* out, int num_sms,
                           cudaStream_t stream) {
  const int64_t n = T * d_out;
  if (n == 0) return cudaSuccess;
  const int epv = is_bf16 ? 8 : 4;
  const auto aligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  const int vec_ok = (d_out % epv == 0) && aligned(base) && aligned(lora) && aligned(out) &&
                     aligned(g);
  const int64_t dv = d_out / epv;
  if (vec_ok && dv % kColThreads == 0) {
    // fixed-column kernel: one wave of 4 blocks of 256 threads per SM
    const int64_t xblocks = dv / kColThreads;
    const int64_t target = static_cast<int64_t>(num_sms > 0 ? num_sms : 148) * 4;
    int64_t yblocks = (target + xblocks - 1) / xblocks;
    if (yblocks > T) yblocks = T;
    if (yblocks > 65535) yblocks = 65535;
    if (yblocks < 1) yblocks = 1;
    const dim3 grid(static_cast<unsigned>(xblocks), static_cast<unsigned>(yblocks));
    const uint4* b4 = static_cast<const uint4*>(base);
    const uint4* l4 = static_cast<const uint4*>(lora);
    uint4* o4 = static_cast<uint4*>(out);
    return is_bf16 ? launch_dependent(k_compose_cols<true>, grid, dim3(kColThreads), stream, b4,
                                      l4, g, s, T, dv, o4)
                   : launch_dependent(k_compose_cols<false>, grid, dim3(kColThreads), stream, b4,
                                      l4, g, s, T, dv, o4);
  }
  const int64_t work = vec_ok ? (n / epv + kUnroll - 1) / kUnroll : n;
  int64_t blocks = (work + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms > 0 ? num_sms : 148) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const dim3 grid(static_cast<unsigned>(blocks));
  return is_bf16 ? launch_dependent(k_compose<true>, grid, dim3(256), stream, base, lora, g, s, T,
                                    d_out, out, static_cast<int>(vec_ok))
                 : launch_dependent(k_compose<false>, grid, dim3(256), stream, base, lora, g, s,
                                    T, d_out, out, static_cast<int>(vec_ok));
}

}  // namespace dora
