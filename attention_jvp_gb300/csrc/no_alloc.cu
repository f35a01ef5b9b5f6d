// Split-KV attention JVP for callers that must not allocate device memory.
//
// The split path needs scratch space for the per-chunk partial results
// (O_c, Ot_c, LSE_c, mu_c) between the chunk launches and the merge.  The
// ordinary route (attn_jvp_fwd_chunk + attn_jvp_merge) leaves that buffer to
// the caller.  Some callers cannot provide it: code running inside a host
// framework that owns all device memory and hands out only the tensors of an
// operation, or latency-critical loops where a cudaMalloc/cudaFree (which can
// synchronise the device) is forbidden.  attn_jvp_fwd_split_noalloc keeps the
// partials in a fixed array compiled into this library instead, so it calls
// no allocator at all.
//
// The first call on a device looks up the array's device address once (with
// that device current) and caches it; make that first call before any stream
// capture.  The cache is keyed by device ordinal, so the library does not
// survive cudaDeviceReset (or any other teardown of the primary context)
// while it is loaded: the cached address would then point at released memory.
//
// Cost and limits: every GPU that loads the library reserves
// kNoAllocScratchBytes for the array until the process exits; a request whose
// partials (and, for fp32 inputs, bf16 copies of the inputs) do not fit is
// rejected with ATTNJVP_EINVAL before anything is launched.  All calls share the
// one array per device, so calls that can overlap on the GPU (different
// streams without ordering, or several host threads) race on it.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <mutex>

#include "../../include/attnjvp.h"
#include "internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB per device

// The scratch array.  Host code must not use this name as a pointer: on the
// host it is only a stand-in, and its device address comes from
// cudaGetSymbolAddress (see scratch_address below).
static __device__ __align__(256) unsigned char g_split_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned char* g_scratch_ptr[kMaxDevices] = {};

// Device address of the current device's scratch array, looked up once per
// device (with that device current) and cached.  Returns nullptr on failure.
unsigned char* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_split_scratch) != cudaSuccess || p == nullptr) return nullptr;
    g_scratch_ptr[dev] = static_cast<unsigned char*>(p);
  }
  return g_scratch_ptr[dev];
}

int reject(int code, const char* msg) {
  attnjvp::set_last_error(msg);
  return code;
}

}  // namespace

extern "C" int attn_jvp_fwd_split_noalloc(const void* q, const void* k, const void* v, const void* q_t,
                                          const void* k_t, const void* v_t, float* out, float* out_t, float* lse,
                                          float* mu, int64_t B, int64_t H, int64_t N, int64_t d, float scale,
                                          int dtype, int64_t n_chunks, void* stream) {
  // Every argument the chunk launches and the merge would check is checked first
  // (this also bounds B*H and N below 2^31, so the sizes below cannot overflow).
  int rc = attnjvp::check_attn_args(q, k, v, q_t, k_t, v_t, out, out_t, lse, mu, B, H, N, d, scale, dtype);
  if (rc != ATTNJVP_OK) return rc;
  if (n_chunks < 1 || n_chunks > N) return reject(ATTNJVP_EINVAL, "n_chunks must be in [1, N]");
  // Layout of the array: for fp32 inputs, first their six bf16 copies
  // [B, H, N, d] (each padded to 256 bytes); then the partials O_c and Ot_c
  // [C, rows, d] fp32, then LSE_c and mu_c [C, rows] fp32.
  const int64_t rows = B * H * N;
  const double copy_bytes = dtype == ATTNJVP_FP32 ? 6.0 * (double(rows * d) * 2.0 + 255.0) : 0.0;
  const double need = copy_bytes + double(n_chunks) * double(rows) * double(2 * d + 2) * 4.0;
  if (need > double(kNoAllocScratchBytes)) {
    char msg[400];
    snprintf(msg, sizeof(msg),
             "split partials%s need %.0f bytes but the built-in scratch holds %zu bytes "
             "(n_chunks * B * H * N * (2d + 2) * 4%s must not exceed it); use attn_jvp_fwd_chunk + "
             "attn_jvp_merge with a caller-provided buffer",
             dtype == ATTNJVP_FP32 ? " and bf16 input copies" : "", need, kNoAllocScratchBytes,
             dtype == ATTNJVP_FP32 ? " + 6 * B * H * N * d * 2" : "");
    return reject(ATTNJVP_EINVAL, msg);
  }
  unsigned char* base = scratch_address();
  if (!base) return reject(ATTNJVP_ECUDA, "could not look up the device address of the built-in scratch array");
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const void* in[6] = {q, k, v, q_t, k_t, v_t};
  if (dtype == ATTNJVP_FP32) {
    // Round each input to bf16 into the array; the kernels read the copies.
    const size_t each = (size_t(rows * d) * 2 + 255) / 256 * 256;
    for (int i = 0; i < 6; ++i) {
      void* dst = base + i * each;
      const cudaError_t e = attnjvp::launch_cast_f32_bf16(static_cast<const float*>(in[i]), dst, rows * d, cs);
      if (e != cudaSuccess) return reject(ATTNJVP_ECUDA, "fp32 -> bf16 cast launch failed");
      in[i] = dst;
    }
    base += 6 * each;
  }
  float* o_c = reinterpret_cast<float*>(base);
  float* ot_c = o_c + n_chunks * rows * d;
  float* lse_c = ot_c + n_chunks * rows * d;
  float* mu_c = lse_c + n_chunks * rows;
  // Every partial element is written by its chunk launch before the merge
  // reads it, so nothing left over from an earlier call is ever used.
  for (int64_t c = 0; c < n_chunks; ++c) {
    const int64_t a = (N * c) / n_chunks, b = (N * (c + 1)) / n_chunks;
    rc = attn_jvp_fwd_chunk(in[0], in[1], in[2], in[3], in[4], in[5], o_c + c * rows * d, ot_c + c * rows * d,
                            lse_c + c * rows, mu_c + c * rows, B, H, N, d, scale, ATTNJVP_BF16, a, b - a, stream);
    if (rc != ATTNJVP_OK) return rc;  // attn_jvp_last_error() already holds the reason
  }
  // The merge sets attn_jvp_last_error() itself (empty on success).
  return attn_jvp_merge(o_c, ot_c, lse_c, mu_c, n_chunks, out, out_t, lse, mu, B, H, N, d, stream);
}
