// Output side of one consistency step on the GPU (page "带分数正则的一致性蒸馏",
// section 一致性模型 (consistency model), its 蒸馏代码 listing):
//   - trigflow_output_jvp: F = (cos t x - x0) / sin t with x0 = c_skip x + c_out n
//     and its tangent (the JVP of the page's _process_output);
//   - scm_tangent_loss: the tangent target g with its warm-up, df/dt, the
//     per-sample NaN masks, the normalisation g / (||g||_2 + 0.1) and the loss
//     sum (F_theta - F_sg - g_n)^2.
// Tensors are [B, C, T, HW] fp32 with the time t given per (b, frame) as FP64
// [B, T].  The work is HBM-bound.  It is cut into rows of HW elements (one
// (b, c, frame) each), so every element of a row shares one set of per-frame
// coefficients, formed once per block in FP64 and rounded to fp32; the
// elementwise arithmetic is fp32 (the page's tensors are fp32) with 16-byte
// accesses when the rows allow them.  The norms and the loss are accumulated to
// near FP64 accuracy (the page converts g to double before normalising): exact
// products summed in fp32 pairs per thread, FP64 per block, then per sample in
// a fixed order, so results are reproducible.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace attnjvp {
namespace {

constexpr int kThreads = 256;
constexpr int kVecPerThread = 4;                            // float4 groups per thread per block
constexpr int64_t kChunkScalar = kThreads * 8;              // elements per block (scalar path)
// The target pass keeps fewer groups per thread (more blocks in flight per SM).
constexpr int kTgtVecPerThread = 4;

// Row segments: a work item is (row, chunk) with row = (b * C + c) * T + f.
struct Rows {
  int64_t HW, chunks, chunk_elems;  // chunk_elems: elements per item (vector: 4 * kChunkVec)
  int T, CT;
  bool vec;
};

Rows make_rows(int64_t C, int64_t T, int64_t HW, bool vec, int vec_per_thread = kVecPerThread) {
  Rows r;
  r.HW = HW;
  r.T = static_cast<int>(T);
  r.CT = static_cast<int>(C * T);
  r.vec = vec;
  r.chunk_elems = vec ? 4 * int64_t(kThreads) * vec_per_thread : kChunkScalar;
  r.chunks = (HW + r.chunk_elems - 1) / r.chunk_elems;
  return r;
}

// ---------------------------------------------------------------------------
// trigflow_output_jvp
// ---------------------------------------------------------------------------
struct OutCoef {
  float c_skip, c_out, t_c_skip, t_c_out, cos_t, sin_t, inv_sin, v;
};

__device__ __forceinline__ void out_one(const OutCoef& c, float xe, float ne, float txe, float tne, float& Fe,
                                        float& tFe) {
  const float x0 = c.c_skip * xe + c.c_out * ne;
  const float tx0 = c.t_c_skip * xe + c.c_skip * txe + c.t_c_out * ne + c.c_out * tne;
  const float num = c.cos_t * xe - x0;
  Fe = num * c.inv_sin;
  // d/dt of num / sin t along the tangents: (d num - F cos t v) / sin t
  tFe = ((-c.sin_t * c.v * xe + c.cos_t * txe - tx0) - Fe * c.cos_t * c.v) * c.inv_sin;
}

__global__ void __launch_bounds__(kThreads) output_jvp_kernel(const float* __restrict__ x, const float* __restrict__ n,
                                                              const float* __restrict__ tx,
                                                              const float* __restrict__ tn,
                                                              const double* __restrict__ t,
                                                              const double* __restrict__ tt, float* __restrict__ F,
                                                              float* __restrict__ tF, Rows rows) {
  __shared__ OutCoef coef;
  const int64_t item = blockIdx.x;
  const int64_t row = item / rows.chunks;
  const int64_t chunk = item - row * rows.chunks;
  if (threadIdx.x == 0) {
    const int b = static_cast<int>(row / rows.CT), f = static_cast<int>(row % rows.T);
    const double tm = t[static_cast<int64_t>(b) * rows.T + f], v = tt[static_cast<int64_t>(b) * rows.T + f];
    double s, c;
    sincos(tm, &s, &c);
    const double den = c + s, den2 = den * den;
    coef.c_skip = static_cast<float>(1.0 / den);
    coef.c_out = static_cast<float>(-s / den);
    coef.t_c_skip = static_cast<float>(v * (-(c - s) / den2));
    coef.t_c_out = static_cast<float>(v * (-1.0 / den2));
    coef.cos_t = static_cast<float>(c);
    coef.sin_t = static_cast<float>(s);
    coef.inv_sin = static_cast<float>(1.0 / s);
    coef.v = static_cast<float>(v);
  }
  __syncthreads();
  const OutCoef c = coef;
  const int64_t base = row * rows.HW;
  const int64_t lo = chunk * rows.chunk_elems;
  const int64_t hi = min(lo + rows.chunk_elems, rows.HW);
  if (rows.vec) {
#pragma unroll
    for (int k = 0; k < kVecPerThread; ++k) {
      const int64_t i = lo + 4 * (k * kThreads + threadIdx.x);
      if (i >= hi) break;
      const int64_t e = base + i;
      const float4 xv = *reinterpret_cast<const float4*>(x + e), nv = *reinterpret_cast<const float4*>(n + e);
      const float4 txv = *reinterpret_cast<const float4*>(tx + e), tnv = *reinterpret_cast<const float4*>(tn + e);
      float4 Fv, tFv;
      out_one(c, xv.x, nv.x, txv.x, tnv.x, Fv.x, tFv.x);
      out_one(c, xv.y, nv.y, txv.y, tnv.y, Fv.y, tFv.y);
      out_one(c, xv.z, nv.z, txv.z, tnv.z, Fv.z, tFv.z);
      out_one(c, xv.w, nv.w, txv.w, tnv.w, Fv.w, tFv.w);
      *reinterpret_cast<float4*>(F + e) = Fv;
      *reinterpret_cast<float4*>(tF + e) = tFv;
    }
  } else {
    for (int64_t i = lo + threadIdx.x; i < hi; i += kThreads) {
      const int64_t e = base + i;
      out_one(c, x[e], n[e], tx[e], tn[e], F[e], tF[e]);
    }
  }
}

// ---------------------------------------------------------------------------
// scm_tangent_loss
// ---------------------------------------------------------------------------
struct TgtCoef {
  float cos_t, sin_t, gap, xcoef;  // gap = cos t sqrt(1 - r^2 sin^2 t), xcoef = r cos t sin t
};

// A sum of products kept as an unevaluated pair hi + lo of fp32 values: each
// product a b enters exactly (p = a b and its error fma(a, b, -p)) and is
// added with Knuth's error-free two-sum, so the pair carries about 48
// significant bits, near the FP64 sum the page forms, without FP64 arithmetic
// per element (GB300's FP64 rate is far below its HBM rate).
struct PairSum {
  float hi = 0.f, lo = 0.f;
  __device__ __forceinline__ void add_product(float a, float b) {
    const float p = a * b;
    const float pe = fmaf(a, b, -p);
    const float s = hi + p;
    const float bb = s - hi;
    const float e = (hi - (s - bb)) + (p - bb);
    hi = s;
    lo += e + pe;
  }
  __device__ __forceinline__ double value() const { return static_cast<double>(hi) + static_cast<double>(lo); }
};

// Per-thread sums of g^2, a^2 and a g (a = F_theta - F_sg) and NaN flags.
struct Acc {
  PairSum gg, aa, ag;
  bool bad_g = false, bad_F = false;
};

__device__ __forceinline__ float tgt_one(const TgtCoef& c, float Ft, float Fs, float Fc, float xe, float te,
                                         float& dfdt, Acc& acc) {
  const float dF = Fs - Fc;
  const float g = -c.gap * dF - (c.xcoef * xe + te);
  dfdt = -c.cos_t * dF - (c.sin_t * xe + te);
  const float a = Ft - Fs;
  acc.gg.add_product(g, g);
  acc.aa.add_product(a, a);
  acc.ag.add_product(a, g);
  acc.bad_g |= isnan(g);
  acc.bad_F |= isnan(Ft);
  return g;
}

__device__ __forceinline__ double block_sum(double v, double* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  double s = 0.0;
  if (threadIdx.x == 0)
    for (int i = 0; i < kThreads / 32; ++i) s += red[i];
  return s;  // valid in thread 0
}

// Pass 1: g (unnormalised, into g_out) and df/dt; per-item sums of g^2, a^2
// and a g (pairs per thread, FP64 across the block); the samples' NaN flags.
__global__ void __launch_bounds__(kThreads) target_kernel(const float* __restrict__ F_theta,
                                                          const float* __restrict__ F_sg,
                                                          const float* __restrict__ F_tc,
                                                          const float* __restrict__ x,
                                                          const float* __restrict__ tF,
                                                          const double* __restrict__ t, double r,
                                                          float* __restrict__ g_out, float* __restrict__ dfdt,
                                                          double* __restrict__ part, int* __restrict__ nan_g,
                                                          int* __restrict__ nan_F, Rows rows) {
  __shared__ TgtCoef coef;
  __shared__ double red[kThreads / 32];
  const int64_t item = blockIdx.x;
  const int64_t row = item / rows.chunks;
  const int64_t chunk = item - row * rows.chunks;
  const int b = static_cast<int>(row / rows.CT);
  if (threadIdx.x == 0) {
    const int f = static_cast<int>(row % rows.T);
    double s, c;
    sincos(t[static_cast<int64_t>(b) * rows.T + f], &s, &c);
    coef.cos_t = static_cast<float>(c);
    coef.sin_t = static_cast<float>(s);
    coef.gap = static_cast<float>(c * sqrt(1.0 - r * r * s * s));
    coef.xcoef = static_cast<float>(r * c * s);
  }
  __syncthreads();
  const TgtCoef c = coef;
  const int64_t base = row * rows.HW;
  const int64_t lo = chunk * rows.chunk_elems;
  const int64_t hi = min(lo + rows.chunk_elems, rows.HW);
  Acc acc;
  if (rows.vec) {
#pragma unroll
    for (int k = 0; k < kTgtVecPerThread; ++k) {
      const int64_t i = lo + 4 * (k * kThreads + threadIdx.x);
      if (i >= hi) break;
      const int64_t e = base + i;
      const float4 Ft = *reinterpret_cast<const float4*>(F_theta + e);
      const float4 Fs = *reinterpret_cast<const float4*>(F_sg + e);
      const float4 Fc = *reinterpret_cast<const float4*>(F_tc + e);
      const float4 xv = *reinterpret_cast<const float4*>(x + e);
      const float4 te = *reinterpret_cast<const float4*>(tF + e);
      float4 g, d;
      g.x = tgt_one(c, Ft.x, Fs.x, Fc.x, xv.x, te.x, d.x, acc);
      g.y = tgt_one(c, Ft.y, Fs.y, Fc.y, xv.y, te.y, d.y, acc);
      g.z = tgt_one(c, Ft.z, Fs.z, Fc.z, xv.z, te.z, d.z, acc);
      g.w = tgt_one(c, Ft.w, Fs.w, Fc.w, xv.w, te.w, d.w, acc);
      *reinterpret_cast<float4*>(g_out + e) = g;
      *reinterpret_cast<float4*>(dfdt + e) = d;
    }
  } else {
    for (int64_t i = lo + threadIdx.x; i < hi; i += kThreads) {
      const int64_t e = base + i;
      g_out[e] = tgt_one(c, F_theta[e], F_sg[e], F_tc[e], x[e], tF[e], dfdt[e], acc);
    }
  }
  if (__any_sync(0xffffffffu, acc.bad_g) && (threadIdx.x & 31) == 0) atomicOr(&nan_g[b], 1);
  if (__any_sync(0xffffffffu, acc.bad_F) && (threadIdx.x & 31) == 0) atomicOr(&nan_F[b], 1);
  const double gg = block_sum(acc.gg.value(), red);
  const double aa = block_sum(acc.aa.value(), red);
  const double ag = block_sum(acc.ag.value(), red);
  if (threadIdx.x == 0) {
    part[3 * item + 0] = gg;
    part[3 * item + 1] = aa;
    part[3 * item + 2] = ag;
  }
}

// Per sample, from the item sums in a fixed order: s = 1 / (||g|| + 0.1) and
// loss = sum (a - s g)^2 = sum a^2 - 2 s sum a g + s^2 sum g^2 (exact algebra);
// a masked sample gets s = 0 and loss = 0 (g, F_theta and F_sg taken as 0).
__global__ void __launch_bounds__(kThreads) finish_kernel(const double* __restrict__ part, int64_t items_per_sample,
                                                          const int* __restrict__ nan_g,
                                                          const int* __restrict__ nan_F, double* __restrict__ scale,
                                                          double* __restrict__ loss) {
  __shared__ double red[kThreads / 32];
  const int b = blockIdx.x;
  double gg = 0.0, aa = 0.0, ag = 0.0;
  const double* p = part + 3 * static_cast<int64_t>(b) * items_per_sample;
  for (int64_t i = threadIdx.x; i < items_per_sample; i += kThreads) {
    gg += p[3 * i + 0];
    aa += p[3 * i + 1];
    ag += p[3 * i + 2];
  }
  gg = block_sum(gg, red);
  aa = block_sum(aa, red);
  ag = block_sum(ag, red);
  if (threadIdx.x == 0) {
    if (nan_g[b] | nan_F[b]) {
      scale[b] = 0.0;
      loss[b] = 0.0;
    } else {
      const double s = 1.0 / (sqrt(gg) + 0.1);
      scale[b] = s;
      loss[b] = aa - 2.0 * s * ag + s * s * gg;
    }
  }
}

// Pass 2: g_n = g s (exactly 0 for a masked sample, whatever g held).
__global__ void __launch_bounds__(kThreads) normalize_kernel(float* __restrict__ g, const double* __restrict__ scale,
                                                             const int* __restrict__ nan_g,
                                                             const int* __restrict__ nan_F, Rows rows) {
  const int64_t item = blockIdx.x;
  const int64_t row = item / rows.chunks;
  const int64_t chunk = item - row * rows.chunks;
  const int b = static_cast<int>(row / rows.CT);
  const bool masked = (nan_g[b] | nan_F[b]) != 0;
  const float s = static_cast<float>(scale[b]);
  const int64_t base = row * rows.HW;
  const int64_t lo = chunk * rows.chunk_elems;
  const int64_t hi = min(lo + rows.chunk_elems, rows.HW);
  if (rows.vec) {
#pragma unroll
    for (int k = 0; k < kVecPerThread; ++k) {
      const int64_t i = lo + 4 * (k * kThreads + threadIdx.x);
      if (i >= hi) break;
      float4* p = reinterpret_cast<float4*>(g + base + i);
      float4 v = *p;
      if (masked) {
        v = make_float4(0.f, 0.f, 0.f, 0.f);
      } else {
        v.x *= s;
        v.y *= s;
        v.z *= s;
        v.w *= s;
      }
      *p = v;
    }
  } else {
    for (int64_t i = lo + threadIdx.x; i < hi; i += kThreads) {
      const int64_t e = base + i;
      g[e] = masked ? 0.f : g[e] * s;
    }
  }
}

bool vec_ok(int64_t HW, std::initializer_list<const void*> ptrs) {
  if (HW % 4 != 0) return false;
  for (const void* p : ptrs)
    if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return false;
  return true;
}

}  // namespace

int64_t epilogue_items(int64_t B, int64_t C, int64_t T, int64_t HW) {
  return B * C * T * make_rows(C, T, HW, HW % 4 == 0).chunks;
}

int64_t scm_workspace_doubles(int64_t B, int64_t C, int64_t T, int64_t HW) {
  // the larger (scalar-path) item count, 3 sums per item, then the per-sample scale
  const int64_t items = B * C * T * make_rows(C, T, HW, false).chunks;
  return 3 * items + B;
}

cudaError_t launch_output_jvp(const float* x, const float* n, const float* tx, const float* tn, const double* t,
                              const double* tt, float* F, float* tF, int64_t B, int64_t C, int64_t T, int64_t HW,
                              cudaStream_t stream) {
  const Rows rows = make_rows(C, T, HW, vec_ok(HW, {x, n, tx, tn, F, tF}));
  const int64_t items = B * C * T * rows.chunks;
  output_jvp_kernel<<<static_cast<unsigned>(items), kThreads, 0, stream>>>(x, n, tx, tn, t, tt, F, tF, rows);
  return cudaGetLastError();
}

cudaError_t launch_scm_tangent_loss(const float* F_theta, const float* F_sg, const float* F_tc, const float* x,
                                    const float* tF, const double* t, double r, float* g_n, float* dfdt,
                                    double* loss, int* nan_g, int* nan_F, int64_t B, int64_t C, int64_t T, int64_t HW,
                                    double* ws, cudaStream_t stream) {
  const bool vec = vec_ok(HW, {F_theta, F_sg, F_tc, x, tF, g_n, dfdt});
  const Rows rows = make_rows(C, T, HW, vec, kTgtVecPerThread);
  const Rows nrows = make_rows(C, T, HW, vec);
  const int64_t items_per_sample = C * T * rows.chunks;
  const int64_t items = B * items_per_sample;
  double* part = ws;
  double* scale = ws + 3 * items;
  cudaError_t e = cudaMemsetAsync(nan_g, 0, B * sizeof(int), stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(nan_F, 0, B * sizeof(int), stream);
  if (e != cudaSuccess) return e;
  target_kernel<<<static_cast<unsigned>(items), kThreads, 0, stream>>>(F_theta, F_sg, F_tc, x, tF, t, r, g_n, dfdt,
                                                                      part, nan_g, nan_F, rows);
  finish_kernel<<<static_cast<unsigned>(B), kThreads, 0, stream>>>(part, items_per_sample, nan_g, nan_F, scale, loss);
  normalize_kernel<<<static_cast<unsigned>(B * C * T * nrows.chunks), kThreads, 0, stream>>>(g_n, scale, nan_g,
                                                                                             nan_F, nrows);
  return cudaGetLastError();
}

}  // namespace attnjvp
