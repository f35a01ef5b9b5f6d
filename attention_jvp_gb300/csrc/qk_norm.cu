// QK normalisation and its tangent: the input-side step of the attention JVP
// for a student that keeps RMS-normalised queries and keys (page "带分数正则的
// 一致性蒸馏", section 一致性模型 (consistency model): QK正则化 is kept).  The
// norm is the per-head RMSNorm of the page "Обслуживание Ideogram v4 менее чем
// за секунду" (dev48.org), section on fusing RMSNorm:
//     y = x rsqrt(mean(x^2) + eps) w
// over each row of d channels (one token of one head), and along a tangent xt
//     yt = w (xt rho - x rho^3 mean(x xt)),   rho = rsqrt(mean(x^2) + eps).
//
// HBM-bound: 8 algorithmic bytes per element (read x and xt, write y and yt,
// all bf16); the per-channel weight is read once per row from L1.  One launch
// covers the Q rows and then the K rows.  A group of d/8 threads (2 at d = 16)
// owns a row: each thread moves 16 bytes of x and of xt, the two row sums are
// reduced with xor shuffles inside the group, and the sums, rho and the
// outputs are formed in fp32 before rounding to bf16 (nearest even).  The grid
// is a whole number of waves of 256-thread blocks striding over the rows.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "internal.h"

namespace attnjvp {
namespace {

__device__ __forceinline__ void unpack8(const uint4& u, float f[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&p);
}

// G: threads per row (d / 8, at least 2); each thread holds 8 channels.
template <int G>
__global__ void __launch_bounds__(256) qk_rmsnorm_jvp_kernel(QkNormArgs a) {
  constexpr int kRowsPerBlock = 256 / G;
  const int sub = threadIdx.x % G;               // which 8 channels of the row
  const int slot = threadIdx.x / G;              // row slot within the block
  const int d = a.d;
  const float inv_d = 1.f / static_cast<float>(d);
  const int c0 = sub * 8;
  const int64_t total = a.rows_q + a.rows_k;
  // ``base`` is the same for every thread of the block, so the whole warp reaches
  // the shuffles; a slot past the last row adds zeros and stores nothing.
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * kRowsPerBlock; base < total;
       base += static_cast<int64_t>(gridDim.x) * kRowsPerBlock) {
    const int64_t r = base + slot;
    const bool valid = r < total;
    const bool is_q = r < a.rows_q;
    const int64_t row = is_q ? r : r - a.rows_q;
    const __nv_bfloat16* x = is_q ? a.q : a.k;
    const __nv_bfloat16* xt = is_q ? a.q_t : a.k_t;
    const float* w = is_q ? a.w_q : a.w_k;
    __nv_bfloat16* y = is_q ? a.qn : a.kn;
    __nv_bfloat16* yt = is_q ? a.qn_t : a.kn_t;
    const int64_t off = row * d + c0;
    float xv[8], tv[8];
    float ss = 0.f, sx = 0.f;
    if (valid) {
      unpack8(*reinterpret_cast<const uint4*>(x + off), xv);
      unpack8(*reinterpret_cast<const uint4*>(xt + off), tv);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        ss = fmaf(xv[i], xv[i], ss);
        sx = fmaf(xv[i], tv[i], sx);
      }
    }
    // Row sums over the G threads of the group (aligned runs of G lanes).
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) {
      ss += __shfl_xor_sync(0xffffffffu, ss, o, G);
      sx += __shfl_xor_sync(0xffffffffu, sx, o, G);
    }
    if (!valid) continue;
    const float rho = rsqrtf(ss * inv_d + a.eps);
    const float c = rho * rho * rho * (sx * inv_d);  // rho^3 mean(x xt)
    const float4 w0 = *reinterpret_cast<const float4*>(w + c0);
    const float4 w1 = *reinterpret_cast<const float4*>(w + c0 + 4);
    const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    float yo[8], to[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      yo[i] = xv[i] * rho * wv[i];
      to[i] = wv[i] * fmaf(tv[i], rho, -xv[i] * c);
    }
    uint4 py, pt;
    py.x = pack2(yo[0], yo[1]);
    py.y = pack2(yo[2], yo[3]);
    py.z = pack2(yo[4], yo[5]);
    py.w = pack2(yo[6], yo[7]);
    pt.x = pack2(to[0], to[1]);
    pt.y = pack2(to[2], to[3]);
    pt.z = pack2(to[4], to[5]);
    pt.w = pack2(to[6], to[7]);
    *reinterpret_cast<uint4*>(y + off) = py;
    *reinterpret_cast<uint4*>(yt + off) = pt;
  }
}

int sm_count_cached() {
  const int n = device_sm_count();
  return n > 0 ? n : 148;
}

template <int G>
cudaError_t launch_g(const QkNormArgs& a, cudaStream_t stream) {
  constexpr int kRowsPerBlock = 256 / G;
  const int64_t total = a.rows_q + a.rows_k;
  const int64_t want = (total + kRowsPerBlock - 1) / kRowsPerBlock;
  const int64_t cap = static_cast<int64_t>(sm_count_cached()) * 8;  // 8 blocks (2048 threads) per SM
  const int64_t blocks = want < cap ? want : cap;
  qk_rmsnorm_jvp_kernel<G><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_qk_rmsnorm_jvp(const QkNormArgs& a, cudaStream_t stream) {
  if (a.rows_q + a.rows_k == 0) return cudaSuccess;
  switch (a.d) {
    case 16: return launch_g<2>(a, stream);
    case 32: return launch_g<4>(a, stream);
    case 64: return launch_g<8>(a, stream);
    case 128: return launch_g<16>(a, stream);
    case 256: return launch_g<32>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace attnjvp
