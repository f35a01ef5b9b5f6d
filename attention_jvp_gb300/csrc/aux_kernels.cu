// Bandwidth-bound kernels around the fused attention JVP:
//   * exact merge of key-chunk partials (O_c, Ot_c, LSE_c, mu_c),
//   * fp32 -> bf16 rounding of inputs (contiguous, or gathered from strides),
//   * the TrigFlow tangent dx_t/dt = -sin t x0 + cos t eps.
// Each thread moves 16-byte vectors; grids are sized in whole waves of the
// GPU's SMs by the launchers below.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace attnjvp {
namespace {

// ---------------------------------------------------------------------------
// Key-chunk merge.  For row i and chunks c = 0..C-1 (all exact algebra on the
// streaming definitions; the page has no key split):
//   LSE = ln sum_c e^{LSE_c},  w_c = e^{LSE_c - LSE}
//   O   = sum_c w_c O_c
//   mu  = sum_c w_c mu_c
//   Ot  = sum_c w_c (Ot_c + mu_c O_c) - mu O
// One thread handles 4 consecutive columns of one row; d/4 threads per row.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) merge_kernel(const float* __restrict__ o_c, const float* __restrict__ ot_c,
                                                    const float* __restrict__ lse_c, const float* __restrict__ mu_c,
                                                    int n_chunks, float* __restrict__ out, float* __restrict__ out_t,
                                                    float* __restrict__ lse, float* __restrict__ mu, int64_t rows,
                                                    int d) {
  const int tpr = d >> 2;  // threads per row
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t row = gtid / tpr;
  const int col = static_cast<int>(gtid % tpr) * 4;
  if (row >= rows) return;

  float mx = -INFINITY;
  for (int c = 0; c < n_chunks; ++c) mx = fmaxf(mx, lse_c[c * rows + row]);
  float sum = 0.f;
  for (int c = 0; c < n_chunks; ++c) sum += expf(lse_c[c * rows + row] - mx);
  const float L = mx + logf(sum);

  float mu_row = 0.f;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f), t = o;
  for (int c = 0; c < n_chunks; ++c) {
    const float w = expf(lse_c[c * rows + row] - L);
    const float mc = mu_c[c * rows + row];
    mu_row += w * mc;
    const int64_t off = (static_cast<int64_t>(c) * rows + row) * d + col;
    const float4 oc = *reinterpret_cast<const float4*>(o_c + off);
    const float4 tc = *reinterpret_cast<const float4*>(ot_c + off);
    o.x += w * oc.x;
    o.y += w * oc.y;
    o.z += w * oc.z;
    o.w += w * oc.w;
    t.x += w * (tc.x + mc * oc.x);
    t.y += w * (tc.y + mc * oc.y);
    t.z += w * (tc.z + mc * oc.z);
    t.w += w * (tc.w + mc * oc.w);
  }
  t.x -= mu_row * o.x;
  t.y -= mu_row * o.y;
  t.z -= mu_row * o.z;
  t.w -= mu_row * o.w;
  const int64_t off = row * d + col;
  *reinterpret_cast<float4*>(out + off) = o;
  *reinterpret_cast<float4*>(out_t + off) = t;
  if (col == 0) {
    if (lse) lse[row] = L;
    if (mu) mu[row] = mu_row;
  }
}

// ---------------------------------------------------------------------------
// fp32 -> bf16, round to nearest even; 4 elements per thread, grid-stride.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) cast_f32_bf16_kernel(const float* __restrict__ in,
                                                            __nv_bfloat16* __restrict__ out, int64_t n) {
  const int64_t n4 = n >> 2;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
    const float4 v = reinterpret_cast<const float4*>(in)[i];
    const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
    const __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
    uint2 pk;
    pk.x = *reinterpret_cast<const uint32_t*>(&a);
    pk.y = *reinterpret_cast<const uint32_t*>(&b);
    reinterpret_cast<uint2*>(out)[i] = pk;
  }
  for (int64_t i = (n4 << 2) + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    out[i] = __float2bfloat16_rn(in[i]);
}

// ---------------------------------------------------------------------------
// Strided fp32 [b, s, h, c] (element strides sb, ss, sh; unit column stride)
// -> contiguous bf16 [B, H, S, d], round to nearest even.  One thread moves
// 4 columns (a float4 in, 8 bytes out), in the output's order so the stores
// coalesce; grid-stride.  d is a multiple of 4 and every stride a multiple of
// 4 elements, so each float4 load is 16-byte aligned.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) cast_strided_f32_bf16_kernel(const float* __restrict__ in,
                                                                    __nv_bfloat16* __restrict__ out, int64_t H,
                                                                    int64_t S, int q4, int64_t sb, int64_t ss,
                                                                    int64_t sh, int64_t n4) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
    const int64_t r = i / q4;  // output row (b, h, s)
    const int c4 = static_cast<int>(i - r * q4);
    const int64_t s = r % S, bh = r / S;
    const int64_t h = bh % H, b = bh / H;
    const float4 v = *reinterpret_cast<const float4*>(in + b * sb + s * ss + h * sh + 4 * c4);
    const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 pk;
    pk.x = *reinterpret_cast<const uint32_t*>(&lo);
    pk.y = *reinterpret_cast<const uint32_t*>(&hi);
    reinterpret_cast<uint2*>(out)[i] = pk;
  }
}

// ---------------------------------------------------------------------------
// TrigFlow tangent: out[b, i] = -sin(t_b) x0[b, i] + cos(t_b) eps[b, i].
// Block row y = sample b; sin/cos are taken in FP64 once per block, the
// element-wise combination in fp32 (the output precision).
// ---------------------------------------------------------------------------
// ``out`` may alias ``x0`` or ``eps`` (each element is read, then written, by one thread).
__global__ void __launch_bounds__(256) trigflow_tangent_kernel(const float* x0, const float* eps,
                                                               const double* __restrict__ t, float* out,
                                                               int64_t per_sample) {
  const int64_t b = blockIdx.y;
  double sd, cd;
  sincos(t[b], &sd, &cd);
  const float s = static_cast<float>(sd), c = static_cast<float>(cd);
  const float* xb = x0 + b * per_sample;
  const float* eb = eps + b * per_sample;
  float* ob = out + b * per_sample;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t tid0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  // Vector body only when the sample's base is 16-byte aligned.
  const bool vec = ((reinterpret_cast<uintptr_t>(xb) | reinterpret_cast<uintptr_t>(eb) |
                     reinterpret_cast<uintptr_t>(ob)) & 15u) == 0;
  const int64_t n4 = vec ? (per_sample >> 2) : 0;
  for (int64_t i = tid0; i < n4; i += stride) {
    const float4 xv = reinterpret_cast<const float4*>(xb)[i];
    const float4 ev = reinterpret_cast<const float4*>(eb)[i];
    float4 r;
    r.x = fmaf(c, ev.x, -s * xv.x);
    r.y = fmaf(c, ev.y, -s * xv.y);
    r.z = fmaf(c, ev.z, -s * xv.z);
    r.w = fmaf(c, ev.w, -s * xv.w);
    reinterpret_cast<float4*>(ob)[i] = r;
  }
  for (int64_t i = (n4 << 2) + tid0; i < per_sample; i += stride) ob[i] = fmaf(c, eb[i], -s * xb[i]);
}

// ---------------------------------------------------------------------------
// Failure-path self-test: one thread waits, with the kernels' own bounded-wait
// routine, on an mbarrier that nothing will ever complete.  The wait must give
// up after ``limit_ns`` and record the timeout in the status word; the kernel
// then returns normally, leaving the context usable.
// ---------------------------------------------------------------------------
__global__ void wait_selftest_kernel(int* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);  // expects one arrival that never comes
    abort_flag = 0;
    ptx::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) ptx::mbar_wait(&bar, 0, &abort_flag, status, kStatusTimeout, limit_ns);
}

int sm_count() {
  const int n = device_sm_count();
  return n > 0 ? n : 148;
}

}  // namespace

cudaError_t launch_merge(const float* o_c, const float* ot_c, const float* lse_c, const float* mu_c,
                         int64_t n_chunks, float* out, float* out_t, float* lse, float* mu, int64_t rows,
                         int64_t d, cudaStream_t stream) {
  const int64_t threads = rows * (d / 4);
  const int64_t blocks = (threads + 255) / 256;
  if (blocks == 0) return cudaSuccess;
  merge_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(o_c, ot_c, lse_c, mu_c, static_cast<int>(n_chunks),
                                                                  out, out_t, lse, mu, rows, static_cast<int>(d));
  return cudaGetLastError();
}

cudaError_t launch_cast_f32_bf16(const float* in, void* out, int64_t n, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  const int64_t want = (n / 4 + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  const int64_t blocks = want < 1 ? 1 : (want < cap ? want : cap);
  cast_f32_bf16_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(in, static_cast<__nv_bfloat16*>(out), n);
  return cudaGetLastError();
}

cudaError_t launch_cast_strided_f32_bf16(const float* in, void* out, int64_t B, int64_t H, int64_t S, int64_t d,
                                         const int64_t stride[3], cudaStream_t stream) {
  const int64_t n4 = B * H * S * (d / 4);
  if (n4 == 0) return cudaSuccess;
  const int64_t want = (n4 + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  const int64_t blocks = want < cap ? want : cap;
  cast_strided_f32_bf16_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      in, static_cast<__nv_bfloat16*>(out), H, S, static_cast<int>(d / 4), stride[0], stride[1], stride[2], n4);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(int* status, uint64_t limit_ns, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_trigflow_tangent(const float* x0, const float* eps, const double* t, float* out, int64_t B,
                                    int64_t per_sample, cudaStream_t stream) {
  const int64_t want = (per_sample / 4 + 255) / 256;
  int64_t per_b = (static_cast<int64_t>(sm_count()) * 8 + B - 1) / B;  // about 8 blocks per SM in total
  if (per_b < 1) per_b = 1;
  const int64_t gx = want < 1 ? 1 : (want < per_b ? want : per_b);
  dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(B));
  trigflow_tangent_kernel<<<grid, 256, 0, stream>>>(x0, eps, t, out, per_sample);
  return cudaGetLastError();
}

}  // namespace attnjvp
