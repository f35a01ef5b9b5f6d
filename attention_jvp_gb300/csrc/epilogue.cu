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
// coefficients, formed in FP64 (once per block for trigflow_output_jvp, once
// per frame by a prologue for scm_tangent_loss) and rounded to fp32; the
// elementwise arithmetic is fp32 (the page's tensors are fp32) with 16-byte
// accesses when the rows allow them.  The norms and the loss are accumulated to
// near FP64 accuracy (the page converts g to double before normalising): exact
// products summed as fp32 pairs per thread and across the block, FP64 per item
// and per sample, in a fixed order, so results are reproducible.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace attnjvp {
namespace {

constexpr int kThreads = 256;
constexpr int kVecPerThread = 4;                            // float4 groups per thread per block
constexpr int64_t kChunkScalar = kThreads * 8;              // elements per block (scalar path)
// The fused sCM pass: one item per row of a video latent (6240 pixels).
constexpr int kTgtVecPerThread = 8;

// Row segments: a work item is (row, chunk) with row = (b * C + c) * T + f.
struct Rows {
  int64_t HW, chunks, chunk_elems;  // chunk_elems: elements per item (vector: 4 * threads * groups per thread)
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
  // Adds another pair: the high parts by two-sum (exact), the rest in fp32.
  __device__ __forceinline__ void add_pair(float h2, float l2) {
    const float s = hi + h2;
    const float bb = s - hi;
    const float e = (hi - (s - bb)) + (h2 - bb);
    hi = s;
    lo += l2 + e;
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

// Block-wide sums of the three pairs, all in fp32 pair arithmetic (a
// shuffle tree per warp, then the warps in order); FP64 only for the block's
// result.  GB300's FP64 pipe is narrow enough that an FP64 tree per block
// would cost as much as the block's memory traffic.  Valid in thread 0.
__device__ __forceinline__ void block_sum_pairs(Acc& acc, float* red, double& gg, double& aa, double& ag) {
  PairSum* v[3] = {&acc.gg, &acc.aa, &acc.ag};
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      const float h2 = __shfl_down_sync(0xffffffffu, v[k]->hi, o);
      const float l2 = __shfl_down_sync(0xffffffffu, v[k]->lo, o);
      v[k]->add_pair(h2, l2);
    }
  }
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();  // red is free (a previous item may still be reading it)
  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      red[6 * w + 2 * k] = v[k]->hi;
      red[6 * w + 2 * k + 1] = v[k]->lo;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    PairSum t[3];
    for (int i = 0; i < kThreads / 32; ++i)
#pragma unroll
      for (int k = 0; k < 3; ++k) t[k].add_pair(red[6 * i + 2 * k], red[6 * i + 2 * k + 1]);
    gg = t[0].value();
    aa = t[1].value();
    ag = t[2].value();
  }
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

// Per-frame coefficients of the target (FP64, rounded once to fp32) and the
// per-call state: NaN flags, per-sample completion counters and ready flags,
// and the ticket counter of the fused pass, all zeroed here.
__global__ void __launch_bounds__(kThreads) scm_prologue_kernel(const double* __restrict__ t, double r, int64_t BT,
                                                                int64_t B, float* __restrict__ coef,
                                                                int* __restrict__ nan_g, int* __restrict__ nan_F,
                                                                unsigned long long* __restrict__ done,
                                                                unsigned long long* __restrict__ ready,
                                                                unsigned long long* __restrict__ ticket) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  if (i < BT) {
    double s, c;
    sincos(t[i], &s, &c);
    coef[4 * i + 0] = static_cast<float>(c);
    coef[4 * i + 1] = static_cast<float>(s);
    coef[4 * i + 2] = static_cast<float>(c * sqrt(1.0 - r * r * s * s));
    coef[4 * i + 3] = static_cast<float>(r * c * s);
  }
  if (i < B) {
    nan_g[i] = 0;
    nan_F[i] = 0;
    done[i] = 0;
    ready[i] = 0;
  }
  if (i == 0) *ticket = 0;
}

struct ScmArgs {
  const float *F_theta, *F_sg, *F_tc, *x, *tF;
  const float* coef;  // [B * T][4]
  float *g, *dfdt;
  double *part, *scale, *loss;
  int *nan_g, *nan_F, *status;
  unsigned long long *done, *ready, *ticket;
  int64_t n;  // items per sample
  int B;
  Rows rows;
};

// Ticket order of the fused pass, with a lag of L = min(8, B) samples: the
// target items of samples 0 .. L-1; then, for s = L .. B-1, the target items
// of sample s followed by the normalisation items of sample s-L; last the
// normalisation items of samples B-L .. B-1.  A normalisation item waits for
// its sample's scale, which the last of that sample's target items publishes;
// all of those hold earlier tickets, and a ticket is only ever taken by a
// running block, so every wait ends.  The lag exceeds the items a full grid
// holds at once (about a sample and a half of rows), so the waits are rare.
// It also means g is re-read from HBM: the traffic of the items in flight
// alone exceeds L2, so no order that waits for a whole sample could keep g
// there.
struct Unit {
  bool normalise;
  int b;
  int64_t item;  // item index over the whole call: b * n + (index within the sample)
};

__device__ __forceinline__ Unit unit_of(unsigned long long j, int64_t n, int B) {
  const int64_t q = static_cast<int64_t>(j / static_cast<unsigned long long>(n));
  const int64_t r = static_cast<int64_t>(j) - q * n;
  const int64_t L = B < 8 ? B : 8;
  int b;
  bool norm;
  if (q < L) {
    b = static_cast<int>(q), norm = false;
  } else if (q < 2 * int64_t(B) - L) {
    const int64_t k = q - L;
    if (k & 1) b = static_cast<int>(k / 2), norm = true;
    else b = static_cast<int>(L + k / 2), norm = false;
  } else {
    b = static_cast<int>(q - B), norm = true;
  }
  return {norm, b, b * n + r};
}

__device__ __forceinline__ unsigned long long ld_acquire(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// One target item: g (unnormalised, into g) and df/dt; the item's sums of
// g^2, a^2 and a g (fp32 pairs per thread, FP64 across the block) into
// part; the sample's NaN flags.  The block that completes its sample's last
// item reduces the sample's sums in item order and publishes scale and loss.
__device__ __forceinline__ void target_item(const ScmArgs& A, int b, int64_t item, float* pred, double* red,
                                            int* s_last) {
  const Rows& rows = A.rows;
  const int64_t row = item / rows.chunks;
  const int64_t chunk = item - row * rows.chunks;
  const int f = static_cast<int>(row % rows.T);
  const float* cp = A.coef + 4 * (static_cast<int64_t>(b) * rows.T + f);
  const TgtCoef c{__ldg(cp + 0), __ldg(cp + 1), __ldg(cp + 2), __ldg(cp + 3)};
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
      const float4 Ft = *reinterpret_cast<const float4*>(A.F_theta + e);
      const float4 Fs = *reinterpret_cast<const float4*>(A.F_sg + e);
      const float4 Fc = *reinterpret_cast<const float4*>(A.F_tc + e);
      const float4 xv = *reinterpret_cast<const float4*>(A.x + e);
      const float4 te = *reinterpret_cast<const float4*>(A.tF + e);
      float4 g, d;
      g.x = tgt_one(c, Ft.x, Fs.x, Fc.x, xv.x, te.x, d.x, acc);
      g.y = tgt_one(c, Ft.y, Fs.y, Fc.y, xv.y, te.y, d.y, acc);
      g.z = tgt_one(c, Ft.z, Fs.z, Fc.z, xv.z, te.z, d.z, acc);
      g.w = tgt_one(c, Ft.w, Fs.w, Fc.w, xv.w, te.w, d.w, acc);
      *reinterpret_cast<float4*>(A.g + e) = g;
      *reinterpret_cast<float4*>(A.dfdt + e) = d;
    }
  } else {
    for (int64_t i = lo + threadIdx.x; i < hi; i += kThreads) {
      const int64_t e = base + i;
      A.g[e] = tgt_one(c, A.F_theta[e], A.F_sg[e], A.F_tc[e], A.x[e], A.tF[e], A.dfdt[e], acc);
    }
  }
  if (__any_sync(0xffffffffu, acc.bad_g) && (threadIdx.x & 31) == 0) atomicOr(&A.nan_g[b], 1);
  if (__any_sync(0xffffffffu, acc.bad_F) && (threadIdx.x & 31) == 0) atomicOr(&A.nan_F[b], 1);
  double gg = 0.0, aa = 0.0, ag = 0.0;
  block_sum_pairs(acc, pred, gg, aa, ag);
  if (threadIdx.x == 0) {
    A.part[3 * item + 0] = gg;
    A.part[3 * item + 1] = aa;
    A.part[3 * item + 2] = ag;
    __threadfence();  // the sums and the NaN flags before the count
    const unsigned long long prev = atomicAdd(&A.done[b], 1ull);
    *s_last = prev + 1 == static_cast<unsigned long long>(A.n);
  }
  __syncthreads();
  if (!*s_last) return;
  // This block finished the sample: reduce its item sums in item order.
  __threadfence();
  double sgg = 0.0, saa = 0.0, sag = 0.0;
  const double* p = A.part + 3 * static_cast<int64_t>(b) * A.n;
  for (int64_t i = threadIdx.x; i < A.n; i += kThreads) {
    sgg += __ldcg(p + 3 * i + 0);
    saa += __ldcg(p + 3 * i + 1);
    sag += __ldcg(p + 3 * i + 2);
  }
  sgg = block_sum(sgg, red);
  saa = block_sum(saa, red);
  sag = block_sum(sag, red);
  if (threadIdx.x == 0) {
    const bool masked = (__ldcg(A.nan_g + b) | __ldcg(A.nan_F + b)) != 0;
    if (masked) {
      A.scale[b] = 0.0;
      A.loss[b] = 0.0;
    } else {
      const double s = 1.0 / (sqrt(sgg) + 0.1);
      A.scale[b] = s;
      A.loss[b] = saa - 2.0 * s * sag + s * s * sgg;
    }
    st_release(&A.ready[b], masked ? 2ull : 1ull);
  }
}

// One normalisation item: g_n = g s (exactly 0 for a masked sample, whatever
// g held), once the sample's scale is published.  g is read past L1: a cache
// line may straddle two rows, one of them written after this SM last saw it.
// Returns false when the wait ran out.
__device__ __forceinline__ bool normalise_item(const ScmArgs& A, int b, int64_t item, float* s_scale,
                                               int* s_state) {
  if (threadIdx.x == 0) {
    const uint64_t t0 = ptx::globaltimer_ns();
    unsigned long long st = ld_acquire(&A.ready[b]);
    while (st == 0) {
      __nanosleep(256);
      if (ptx::globaltimer_ns() - t0 > ptx::kWaitLimitNs) break;
      st = ld_acquire(&A.ready[b]);
    }
    if (st == 0) atomicOr(A.status, kStatusTimeout);
    *s_state = static_cast<int>(st);
    *s_scale = st == 1 ? static_cast<float>(__ldcg(A.scale + b)) : 0.f;
  }
  __syncthreads();
  const int state = *s_state;
  if (state == 0) return false;
  const bool masked = state == 2;
  const float s = *s_scale;
  const Rows& rows = A.rows;
  const int64_t row = item / rows.chunks;
  const int64_t chunk = item - row * rows.chunks;
  const int64_t base = row * rows.HW;
  const int64_t lo = chunk * rows.chunk_elems;
  const int64_t hi = min(lo + rows.chunk_elems, rows.HW);
  if (rows.vec) {
#pragma unroll
    for (int k = 0; k < kTgtVecPerThread; ++k) {
      const int64_t i = lo + 4 * (k * kThreads + threadIdx.x);
      if (i >= hi) break;
      float4* p = reinterpret_cast<float4*>(A.g + base + i);
      float4 v = __ldcg(p);
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
      float* p = A.g + base + i;
      *p = masked ? 0.f : __ldcg(p) * s;
    }
  }
  return true;
}

// The fused target / reduce / normalise pass: a persistent grid that takes
// items by ticket (see unit_of).  Capped at 40 registers a thread for six
// blocks an SM: more loads in flight.
__global__ void __launch_bounds__(kThreads, 6) scm_fused_kernel(ScmArgs A) {
  __shared__ double red[kThreads / 32];
  __shared__ float pred[6 * (kThreads / 32)];
  __shared__ unsigned long long s_ticket;
  __shared__ int s_last, s_state;
  __shared__ float s_scale;
  const unsigned long long total = 2ull * static_cast<unsigned long long>(A.B) * static_cast<unsigned long long>(A.n);
  for (;;) {
    if (threadIdx.x == 0) s_ticket = atomicAdd(A.ticket, 1ull);
    __syncthreads();
    const unsigned long long j = s_ticket;
    __syncthreads();  // every thread has read the ticket before it is replaced
    if (j >= total) return;
    const Unit u = unit_of(j, A.n, A.B);
    if (u.normalise) {
      if (!normalise_item(A, u.b, u.item, &s_scale, &s_state)) return;
    } else {
      target_item(A, u.b, u.item, pred, red, &s_last);
    }
  }
}

bool vec_ok(int64_t HW, std::initializer_list<const void*> ptrs) {
  if (HW % 4 != 0) return false;
  for (const void* p : ptrs)
    if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return false;
  return true;
}

// Workspace words (8 bytes each) of scm_tangent_loss, in this order.
struct ScmLayout {
  int64_t part, scale, coef, done, ready, ticket, words;
};

ScmLayout scm_layout(int64_t B, int64_t C, int64_t T, int64_t HW) {
  // the larger (scalar-path) item count, 3 sums per item
  const int64_t items = B * C * T * make_rows(C, T, HW, false).chunks;
  ScmLayout l;
  l.part = 0;
  l.scale = l.part + 3 * items;
  l.coef = l.scale + B;  // [B * T][4] fp32
  l.done = l.coef + 2 * B * T;
  l.ready = l.done + B;
  l.ticket = l.ready + B;
  l.words = l.ticket + 1;
  return l;
}

}  // namespace

int64_t epilogue_items(int64_t B, int64_t C, int64_t T, int64_t HW) {
  return B * C * T * make_rows(C, T, HW, HW % 4 == 0).chunks;
}

int64_t scm_workspace_doubles(int64_t B, int64_t C, int64_t T, int64_t HW) { return scm_layout(B, C, T, HW).words; }

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
                                    double* ws, int* status, cudaStream_t stream) {
  const bool vec = vec_ok(HW, {F_theta, F_sg, F_tc, x, tF, g_n, dfdt});
  const ScmLayout lay = scm_layout(B, C, T, HW);
  ScmArgs A;
  A.F_theta = F_theta, A.F_sg = F_sg, A.F_tc = F_tc, A.x = x, A.tF = tF;
  A.coef = reinterpret_cast<const float*>(ws + lay.coef);
  A.g = g_n, A.dfdt = dfdt;
  A.part = ws + lay.part, A.scale = ws + lay.scale, A.loss = loss;
  A.nan_g = nan_g, A.nan_F = nan_F, A.status = status;
  A.done = reinterpret_cast<unsigned long long*>(ws + lay.done);
  A.ready = reinterpret_cast<unsigned long long*>(ws + lay.ready);
  A.ticket = reinterpret_cast<unsigned long long*>(ws + lay.ticket);
  A.rows = make_rows(C, T, HW, vec, kTgtVecPerThread);
  A.n = C * T * A.rows.chunks;
  A.B = static_cast<int>(B);
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, scm_fused_kernel, kThreads, 0);
  if (e != cudaSuccess) return e;
  const int64_t BT = B * T;
  const int64_t pro_threads = BT > B ? BT : B;
  scm_prologue_kernel<<<static_cast<unsigned>((pro_threads + kThreads - 1) / kThreads), kThreads, 0, stream>>>(
      t, r, BT, B, const_cast<float*>(A.coef), nan_g, nan_F, A.done, A.ready, A.ticket);
  const int64_t units = 2 * B * A.n;
  int64_t grid = static_cast<int64_t>(sms) * (per_sm > 0 ? per_sm : 1);
  if (grid > units) grid = units;
  scm_fused_kernel<<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(A);
  return cudaGetLastError();
}

}  // namespace attnjvp
