// C-ABI entry points: argument validation, per-device status word, error
// strings, tensor-map encoder lookup, and the host-side TrigFlow coefficients.
// Every check that needs no GPU runs before the first CUDA call, so invalid
// arguments are reported identically on machines without a device.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <utility>
#include <vector>

#include "../../include/attnjvp.h"
#include "internal.h"

namespace attnjvp {

// Per-device status word (kStatusTimeout bit set by a kernel whose bounded wait ran out).
__device__ int g_status_word;

namespace {

thread_local char g_last_error[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return code;
}

int ok() {
  g_last_error[0] = '\0';
  return ATTNJVP_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_status_ptr[kMaxDevices] = {};

// Device address of the current device's status word (nullptr on failure).
int* status_word(const char** why) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    *why = cudaGetErrorString(e);
    return nullptr;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    *why = "device ordinal out of range";
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_status_word);
    if (e != cudaSuccess) {
      *why = cudaGetErrorString(e);
      return nullptr;
    }
    g_status_ptr[dev] = static_cast<int*>(p);
  }
  return g_status_ptr[dev];
}

int g_sm_count[kMaxDevices] = {};
std::vector<std::pair<const void*, int>> g_smem_set;  // (kernel, device) pairs done

}  // namespace

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_sm_count[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 0;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

cudaError_t ensure_smem_limit(const void* func, int bytes, bool* first) {
  *first = false;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_mu);
  for (const auto& fd : g_smem_set)
    if (fd.first == func && fd.second == dev) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  g_smem_set.emplace_back(func, dev);
  *first = true;
  return cudaSuccess;
}

namespace {

// Head dims: the page's set, 16, 32, 64, 128 and 256, in the forward and the
// backward (at 256 two CTAs share each row tile, each accumulating half of the
// output columns).
int check_head_dim(int64_t d, bool) {
  if (d == 16 || d == 32 || d == 64 || d == 128 || d == 256) return ATTNJVP_OK;
  return fail(ATTNJVP_EUNSUPPORTED, "head dim %lld not supported (16, 32, 64, 128 or 256)", (long long)d);
}

}  // namespace

int check_attn_args(const void* q, const void* k, const void* v, const void* q_t, const void* k_t, const void* v_t,
                    const float* out, const float* out_t, const float* lse, const float* mu, int64_t B, int64_t H,
                    int64_t N, int64_t d, float scale, int dtype) {
  if (dtype != ATTNJVP_BF16 && dtype != ATTNJVP_FP32)
    return fail(ATTNJVP_EINVAL, "dtype code %d is neither ATTNJVP_BF16 (%d) nor ATTNJVP_FP32 (%d)", dtype,
                ATTNJVP_BF16, ATTNJVP_FP32);
  const void* in[6] = {q, k, v, q_t, k_t, v_t};
  const char* names[6] = {"q", "k", "v", "q_t", "k_t", "v_t"};
  for (int i = 0; i < 6; ++i) {
    if (!in[i]) return fail(ATTNJVP_EINVAL, "%s is NULL", names[i]);
    if (!aligned(in[i], 16))
      return fail(ATTNJVP_EINVAL, "%s is not 16-byte aligned (%s)", names[i],
                  dtype == ATTNJVP_BF16 ? "TMA base address" : "16-byte loads of the fp32 cast");
  }
  if (!out || !out_t) return fail(ATTNJVP_EINVAL, "out/out_t is NULL");
  if (!aligned(out, 16) || !aligned(out_t, 16)) return fail(ATTNJVP_EINVAL, "out/out_t is not 16-byte aligned");
  if ((lse && !aligned(lse, 4)) || (mu && !aligned(mu, 4))) return fail(ATTNJVP_EINVAL, "lse/mu misaligned");
  if (B < 1 || H < 1 || N < 1) return fail(ATTNJVP_EINVAL, "B, H, N must be >= 1 (got %lld, %lld, %lld)",
                                           (long long)B, (long long)H, (long long)N);
  if (B >= (int64_t(1) << 31) || H >= (int64_t(1) << 31) || B * H >= (int64_t(1) << 31) ||
      N >= (int64_t(1) << 31))
    return fail(ATTNJVP_EINVAL, "B*H and N must be < 2^31");
  if (!std::isfinite(scale) || !(scale > 0.f)) return fail(ATTNJVP_EINVAL, "scale must be finite and > 0");
  int rc = check_head_dim(d, true);
  if (rc != ATTNJVP_OK) return rc;
  const int64_t n_qtiles = (N + 127) / 128;
  // at a value head dim of 256 two CTAs share each query tile
  if (n_qtiles * B * H * 2 >= (int64_t(1) << 31)) return fail(ATTNJVP_EINVAL, "too many query tiles");
  return ATTNJVP_OK;
}

namespace {

// Element strides (batch, sequence, head) of a contiguous [B, H, N, d] tensor.
void contiguous_strides(int64_t H, int64_t N, int64_t d, int64_t st[3]) {
  st[0] = H * N * d;
  st[1] = d;
  st[2] = N * d;
}

// Launches the fused kernel on bf16 inputs.  ``st``: 12 element strides (batch,
// seq, head) of Q, K, V and O.
int launch_fwd(const void* q, const void* k, const void* v, const void* q_t, const void* k_t, const void* v_t,
               float* out, float* out_t, float* lse, float* mu, int64_t B, int64_t H, int64_t Nq, int64_t Nkv,
               int64_t d, int64_t d_v, const int64_t st[12], float scale, int64_t kv_start, int64_t kv_len,
               bool balance, int* status, cudaStream_t stream) {
  FwdArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.q_t = q_t;
  a.k_t = k_t;
  a.v_t = v_t;
  a.out = out;
  a.out_t = out_t;
  a.lse = lse;
  a.mu = mu;
  a.B = B;
  a.H = H;
  a.Nq = Nq;
  a.Nkv = Nkv;
  a.d = d;
  a.d_v = d_v;
  for (int i = 0; i < 3; ++i) {
    a.q_stride[i] = st[i];
    a.k_stride[i] = st[3 + i];
    a.v_stride[i] = st[6 + i];
    a.o_stride[i] = st[9 + i];
  }
  a.scale = scale;
  a.kv_start = kv_start;
  a.kv_len = kv_len;
  a.status = status;
  a.stream = stream;
  a.balance_tail = balance;
  const char* msg = "";
  cudaError_t e = launch_attn_jvp_fwd(a, &msg);
  if (e != cudaSuccess) return fail(ATTNJVP_ECUDA, "%s: %s", msg, cudaGetErrorString(e));
  return ok();
}

size_t round256(size_t n) { return (n + 255) / 256 * 256; }

// ``strides``: 12 element strides (batch, seq, head) of Q, K, V and O, or NULL
// for contiguous [B, H, N, d] tensors.  ``balance``: the kernel may cut the units
// of a short last wave into pieces over the keys (see FwdArgs::balance_tail).  fp32 inputs (``dtype`` ATTNJVP_FP32) are
// first rounded to bf16 into contiguous [B, H, S, d] copies in stream-ordered
// device memory (cudaMallocAsync on ``stream``), which is released on the same
// stream once the kernel has been enqueued after the copies.
int run_fwd(const void* q, const void* k, const void* v, const void* q_t, const void* k_t, const void* v_t,
            float* out, float* out_t, float* lse, float* mu, int64_t B, int64_t H, int64_t Nq, int64_t Nkv,
            int64_t d, int64_t d_v, const int64_t* strides, float scale, int dtype, int64_t kv_start,
            int64_t kv_len, bool balance, void* stream) {
  const char* why = "";
  int* status = status_word(&why);
  if (!status) return fail(ATTNJVP_ECUDA, "no CUDA device / status word: %s", why);
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  int64_t st[12];
  if (strides) {
    for (int i = 0; i < 12; ++i) st[i] = strides[i];
  } else {
    contiguous_strides(H, Nq, d, st);
    contiguous_strides(H, Nkv, d, st + 3);
    contiguous_strides(H, Nkv, d_v, st + 6);
    contiguous_strides(H, Nq, d_v, st + 9);
  }
  if (dtype == ATTNJVP_BF16)
    return launch_fwd(q, k, v, q_t, k_t, v_t, out, out_t, lse, mu, B, H, Nq, Nkv, d, d_v, st, scale, kv_start,
                      kv_len, balance, status, cs);
  // fp32: six bf16 copies, Q and Qt [B, H, Nq, d], K and Kt [B, H, Nkv, d], V and Vt [B, H, Nkv, d_v].
  const size_t bytes[3] = {round256(size_t(B * H * Nq * d) * 2), round256(size_t(B * H * Nkv * d) * 2),
                           round256(size_t(B * H * Nkv * d_v) * 2)};
  void* buf = nullptr;
  cudaError_t e = cudaMallocAsync(&buf, 2 * (bytes[0] + bytes[1] + bytes[2]), cs);
  if (e != cudaSuccess)
    return fail(ATTNJVP_ECUDA, "stream-ordered allocation of the bf16 copies failed: %s", cudaGetErrorString(e));
  const void* src[6] = {q, q_t, k, k_t, v, v_t};
  void* dst[6];
  unsigned char* p = static_cast<unsigned char*>(buf);
  for (int i = 0; i < 6; ++i) {
    dst[i] = p;
    p += bytes[i / 2];
  }
  const int64_t rows[3] = {Nq, Nkv, Nkv}, cols[3] = {d, d, d_v};
  for (int i = 0; i < 6 && e == cudaSuccess; ++i)
    e = launch_cast_strided_f32_bf16(static_cast<const float*>(src[i]), dst[i], B, H, rows[i / 2], cols[i / 2],
                                     st + 3 * (i / 2), cs);
  int rc;
  if (e != cudaSuccess) {
    rc = fail(ATTNJVP_ECUDA, "fp32 -> bf16 cast launch failed: %s", cudaGetErrorString(e));
  } else {
    int64_t bst[12];
    contiguous_strides(H, Nq, d, bst);
    contiguous_strides(H, Nkv, d, bst + 3);
    contiguous_strides(H, Nkv, d_v, bst + 6);
    for (int i = 9; i < 12; ++i) bst[i] = st[i];
    rc = launch_fwd(dst[0], dst[2], dst[4], dst[1], dst[3], dst[5], out, out_t, lse, mu, B, H, Nq, Nkv, d, d_v, bst,
                    scale, kv_start, kv_len, balance, status, cs);
  }
  e = cudaFreeAsync(buf, cs);
  if (rc == ATTNJVP_OK && e != cudaSuccess)
    rc = fail(ATTNJVP_ECUDA, "stream-ordered release of the bf16 copies failed: %s", cudaGetErrorString(e));
  return rc;
}

}  // namespace

void set_last_error(const char* msg) { snprintf(g_last_error, sizeof(g_last_error), "%s", msg ? msg : ""); }

TensorMapEncodeFn tensor_map_encoder() {
  static TensorMapEncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<TensorMapEncodeFn>(p);
  });
  return fn;
}

}  // namespace attnjvp

using namespace attnjvp;

extern "C" {

int attn_jvp_fwd(const void* q, const void* k, const void* v, const void* q_t, const void* k_t, const void* v_t,
                 float* out, float* out_t, float* lse, float* mu, int64_t B, int64_t H, int64_t N, int64_t d,
                 float scale, int dtype, void* stream) {
  int rc = check_attn_args(q, k, v, q_t, k_t, v_t, out, out_t, lse, mu, B, H, N, d, scale, dtype);
  if (rc != ATTNJVP_OK) return rc;
  return run_fwd(q, k, v, q_t, k_t, v_t, out, out_t, lse, mu, B, H, N, N, d, d, nullptr, scale, dtype, 0, N,
                 true, stream);
}

int attn_jvp_fwd_chunk(const void* q, const void* k, const void* v, const void* q_t, const void* k_t,
                       const void* v_t, float* out, float* out_t, float* lse, float* mu, int64_t B, int64_t H,
                       int64_t N, int64_t d, float scale, int dtype, int64_t kv_start, int64_t kv_len, void* stream) {
  int rc = check_attn_args(q, k, v, q_t, k_t, v_t, out, out_t, lse, mu, B, H, N, d, scale, dtype);
  if (rc != ATTNJVP_OK) return rc;
  if (!lse || !mu) return fail(ATTNJVP_EINVAL, "chunk mode needs lse and mu (the merge consumes them)");
  if (kv_start < 0 || kv_len < 1 || kv_start + kv_len > N)
    return fail(ATTNJVP_EINVAL, "key range [%lld, %lld) outside [0, %lld) or empty", (long long)kv_start,
                (long long)(kv_start + kv_len), (long long)N);
  return run_fwd(q, k, v, q_t, k_t, v_t, out, out_t, lse, mu, B, H, N, N, d, d, nullptr, scale, dtype, kv_start,
                 kv_len, false, stream);
}

int attn_jvp_fwd_ex(const void* q, const void* k, const void* v, const void* q_t, const void* k_t, const void* v_t,
                    float* out, float* out_t, float* lse, float* mu, int64_t B, int64_t H, int64_t Nq, int64_t Nkv,
                    int64_t d, int64_t d_v, const int64_t* strides, float scale, int dtype, int64_t kv_start,
                    int64_t kv_len, void* stream) {
  int rc = check_attn_args(q, k, v, q_t, k_t, v_t, out, out_t, lse, mu, B, H, Nq, d, scale, dtype);
  if (rc != ATTNJVP_OK) return rc;
  rc = check_head_dim(d_v, true);
  if (rc != ATTNJVP_OK) return rc;
  if (Nkv < 1 || Nkv >= (int64_t(1) << 31)) return fail(ATTNJVP_EINVAL, "N_kv must be in [1, 2^31)");
  if (kv_start < 0 || kv_len < 1 || kv_start + kv_len > Nkv)
    return fail(ATTNJVP_EINVAL, "key range [%lld, %lld) outside [0, %lld) or empty", (long long)kv_start,
                (long long)(kv_start + kv_len), (long long)Nkv);
  if (strides) {
    const char* what[4] = {"q", "k", "v", "out"};
    for (int g = 0; g < 4; ++g) {
      // bf16 inputs: TMA strides are multiples of 16 bytes; fp32 inputs: 16-byte loads of
      // the cast; fp32 outputs: float4 stores.
      const int64_t unit = (g < 3 && dtype == ATTNJVP_BF16) ? 8 : 4;
      for (int i = 0; i < 3; ++i) {
        const int64_t x = strides[3 * g + i];
        if (x < 0 || x % unit != 0 || x >= (int64_t(1) << 38))
          return fail(ATTNJVP_EINVAL, "%s stride %d is %lld: must be a non-negative multiple of %lld elements",
                      what[g], i, (long long)x, (long long)unit);
      }
    }
  }
  return run_fwd(q, k, v, q_t, k_t, v_t, out, out_t, lse, mu, B, H, Nq, Nkv, d, d_v, strides, scale, dtype,
                 kv_start, kv_len, kv_start == 0 && kv_len == Nkv, stream);
}

int attn_jvp_fwd_strided(const void* q, const void* k, const void* v, const void* q_t, const void* k_t,
                         const void* v_t, float* out, float* out_t, float* lse, float* mu, int64_t B, int64_t H,
                         int64_t Nq, int64_t Nkv, int64_t d, const int64_t* strides, float scale, int dtype,
                         int64_t kv_start, int64_t kv_len, void* stream) {
  // K and V share one stride set here (equal head dims)
  int64_t st[12];
  if (strides) {
    for (int i = 0; i < 3; ++i) {
      st[i] = strides[i];
      st[3 + i] = strides[3 + i];
      st[6 + i] = strides[3 + i];
      st[9 + i] = strides[6 + i];
    }
  }
  return attn_jvp_fwd_ex(q, k, v, q_t, k_t, v_t, out, out_t, lse, mu, B, H, Nq, Nkv, d, d, strides ? st : nullptr,
                         scale, dtype, kv_start, kv_len, stream);
}

int attn_jvp_fwd_last_wave_split(int64_t B, int64_t H, int64_t N_q, int64_t N_kv, int64_t d_v, int64_t* split) {
  if (!split) return fail(ATTNJVP_EINVAL, "split is NULL");
  if (B < 1 || H < 1 || N_q < 1 || N_kv < 1 || B * H >= (int64_t(1) << 31) || N_q >= (int64_t(1) << 31) ||
      N_kv >= (int64_t(1) << 31))
    return fail(ATTNJVP_EINVAL, "B, H, N_q, N_kv must be >= 1 (B*H, N_q and N_kv below 2^31)");
  const int rc = check_head_dim(d_v, true);
  if (rc != ATTNJVP_OK) return rc;
  const int n_sm = device_sm_count();
  if (n_sm <= 0) return fail(ATTNJVP_ECUDA, "no CUDA device to size the grid for");
  const int64_t grid = (N_q + 127) / 128 * B * H * (d_v > 128 ? 2 : 1);
  *split = last_wave_split(grid, N_kv, n_sm);
  return ok();
}

int attn_jvp_merge(const float* o_c, const float* ot_c, const float* lse_c, const float* mu_c, int64_t n_chunks,
                   float* out, float* out_t, float* lse, float* mu, int64_t B, int64_t H, int64_t N, int64_t d,
                   void* stream) {
  if (!o_c || !ot_c || !lse_c || !mu_c || !out || !out_t) return fail(ATTNJVP_EINVAL, "NULL tensor");
  if (!aligned(o_c, 16) || !aligned(ot_c, 16) || !aligned(out, 16) || !aligned(out_t, 16))
    return fail(ATTNJVP_EINVAL, "o_c/ot_c/out/out_t must be 16-byte aligned");
  if (!aligned(lse_c, 4) || !aligned(mu_c, 4) || (lse && !aligned(lse, 4)) || (mu && !aligned(mu, 4)))
    return fail(ATTNJVP_EINVAL, "per-row tensor misaligned");
  if (n_chunks < 1 || n_chunks > (1 << 20)) return fail(ATTNJVP_EINVAL, "n_chunks must be in [1, 2^20]");
  if (B < 1 || H < 1 || N < 1) return fail(ATTNJVP_EINVAL, "B, H, N must be >= 1");
  if (d < 4 || d > 256 || (d % 4) != 0) return fail(ATTNJVP_EINVAL, "d must be a multiple of 4 in [4, 256]");
  const int64_t rows = B * H * N;
  if (rows * (d / 4) / 256 >= (int64_t(1) << 31)) return fail(ATTNJVP_EINVAL, "too many rows");
  int dev;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(ATTNJVP_ECUDA, "no CUDA device: %s", cudaGetErrorString(e));
  e = launch_merge(o_c, ot_c, lse_c, mu_c, n_chunks, out, out_t, lse, mu, rows, d, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(ATTNJVP_ECUDA, "merge launch failed: %s", cudaGetErrorString(e));
  return ok();
}

int attn_jvp_cast_f32_bf16(const float* in, void* out, int64_t n, void* stream) {
  if (n < 0) return fail(ATTNJVP_EINVAL, "n must be >= 0");
  if (n == 0) return ok();
  if (!in || !out) return fail(ATTNJVP_EINVAL, "NULL tensor");
  if (!aligned(in, 16) || !aligned(out, 16)) return fail(ATTNJVP_EINVAL, "in/out must be 16-byte aligned");
  int dev;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(ATTNJVP_ECUDA, "no CUDA device: %s", cudaGetErrorString(e));
  e = launch_cast_f32_bf16(in, out, n, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(ATTNJVP_ECUDA, "cast launch failed: %s", cudaGetErrorString(e));
  return ok();
}

int qk_rmsnorm_jvp(const void* q, const void* q_t, const void* k, const void* k_t, const float* w_q,
                   const float* w_k, void* qn, void* qn_t, void* kn, void* kn_t, int64_t rows_q, int64_t rows_k,
                   int64_t d, float eps, void* stream) {
  if (rows_q < 0 || rows_k < 0) return fail(ATTNJVP_EINVAL, "rows_q and rows_k must be >= 0");
  if (d != 16 && d != 32 && d != 64 && d != 128 && d != 256)
    return fail(ATTNJVP_EUNSUPPORTED, "head dim %lld not supported (16, 32, 64, 128 or 256)", (long long)d);
  if (!std::isfinite(eps) || eps < 0.f) return fail(ATTNJVP_EINVAL, "eps must be finite and >= 0");
  if (rows_q > (int64_t(1) << 40) / d || rows_k > (int64_t(1) << 40) / d)
    return fail(ATTNJVP_EINVAL, "too many rows");
  struct {
    const void* p;
    const char* name;
    bool needed;
  } ptrs[10] = {{q, "q", rows_q > 0},     {q_t, "q_t", rows_q > 0},   {qn, "qn", rows_q > 0},
                {qn_t, "qn_t", rows_q > 0}, {w_q, "w_q", rows_q > 0}, {k, "k", rows_k > 0},
                {k_t, "k_t", rows_k > 0},   {kn, "kn", rows_k > 0},   {kn_t, "kn_t", rows_k > 0},
                {w_k, "w_k", rows_k > 0}};
  for (const auto& e : ptrs) {
    if (!e.needed) continue;
    if (!e.p) return fail(ATTNJVP_EINVAL, "%s is NULL", e.name);
    if (!aligned(e.p, 16)) return fail(ATTNJVP_EINVAL, "%s is not 16-byte aligned", e.name);
  }
  if (rows_q + rows_k == 0) return ok();
  int dev;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(ATTNJVP_ECUDA, "no CUDA device: %s", cudaGetErrorString(e));
  QkNormArgs a;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.q_t = static_cast<const __nv_bfloat16*>(q_t);
  a.k = static_cast<const __nv_bfloat16*>(k);
  a.k_t = static_cast<const __nv_bfloat16*>(k_t);
  a.w_q = w_q;
  a.w_k = w_k;
  a.qn = static_cast<__nv_bfloat16*>(qn);
  a.qn_t = static_cast<__nv_bfloat16*>(qn_t);
  a.kn = static_cast<__nv_bfloat16*>(kn);
  a.kn_t = static_cast<__nv_bfloat16*>(kn_t);
  a.rows_q = rows_q;
  a.rows_k = rows_k;
  a.d = static_cast<int>(d);
  a.eps = eps;
  e = launch_qk_rmsnorm_jvp(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(ATTNJVP_ECUDA, "QK-norm launch failed: %s", cudaGetErrorString(e));
  return ok();
}

int trigflow_coeffs(double t, double tau, double* c) {
  if (!c) return fail(ATTNJVP_EINVAL, "c is NULL");
  if (!std::isfinite(t) || !std::isfinite(tau)) return fail(ATTNJVP_EINVAL, "t and tau must be finite");
  const double s = std::sin(t), co = std::cos(t);
  const double den = co + s;
  if (!(den > 0.0)) return fail(ATTNJVP_EINVAL, "cos t + sin t <= 0: t outside (-pi/4, 3pi/4)");
  const double inv = 1.0 / den;
  c[0] = inv;
  c[1] = -s * inv;
  c[2] = inv;
  c[3] = tau * s * inv;
  return ok();
}

int trigflow_tangent(const float* x0, const float* eps, const double* t, float* out, int64_t B, int64_t per_sample,
                     void* stream) {
  if (!x0 || !eps || !t || !out) return fail(ATTNJVP_EINVAL, "NULL tensor");
  if (!aligned(x0, 16) || !aligned(eps, 16) || !aligned(out, 16) || !aligned(t, 8))
    return fail(ATTNJVP_EINVAL, "x0/eps/out must be 16-byte aligned and t 8-byte aligned");
  if (B < 1 || B > 65535) return fail(ATTNJVP_EINVAL, "B must be in [1, 65535]");
  if (per_sample < 1) return fail(ATTNJVP_EINVAL, "per_sample must be >= 1");
  int dev;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(ATTNJVP_ECUDA, "no CUDA device: %s", cudaGetErrorString(e));
  e = launch_trigflow_tangent(x0, eps, t, out, B, per_sample, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(ATTNJVP_ECUDA, "trigflow_tangent launch failed: %s", cudaGetErrorString(e));
  return ok();
}

int64_t attn_bwd_workspace_bytes(int64_t B, int64_t H, int64_t N_q) {
  if (B < 1 || H < 1 || N_q < 1) return fail(ATTNJVP_EINVAL, "B, H, N_q must be >= 1");
  if (B * H >= (int64_t(1) << 31) || N_q >= (int64_t(1) << 31)) return fail(ATTNJVP_EINVAL, "too large");
  ok();
  return attn_bwd_workspace_floats(B, H, N_q) * 4;
}

int attn_bwd(const void* q, const void* k, const void* v, const void* dout, const float* out, const float* lse,
             float* dq, float* dk, float* dv, int64_t B, int64_t H, int64_t N_q, int64_t N_kv, int64_t d, float scale,
             void* workspace, int64_t workspace_bytes, void* stream) {
  const void* in16[4] = {q, k, v, dout};
  const char* names[4] = {"q", "k", "v", "dout"};
  for (int i = 0; i < 4; ++i) {
    if (!in16[i]) return fail(ATTNJVP_EINVAL, "%s is NULL", names[i]);
    if (!aligned(in16[i], 16)) return fail(ATTNJVP_EINVAL, "%s is not 16-byte aligned (TMA base address)", names[i]);
  }
  if (!out || !lse || !aligned(out, 4) || !aligned(lse, 4)) return fail(ATTNJVP_EINVAL, "out/lse NULL or misaligned");
  if (!dq || !dk || !dv || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16))
    return fail(ATTNJVP_EINVAL, "dq/dk/dv NULL or not 16-byte aligned");
  if (!workspace || !aligned(workspace, 256)) return fail(ATTNJVP_EINVAL, "workspace NULL or not 256-byte aligned");
  if (B < 1 || H < 1 || N_q < 1 || N_kv < 1) return fail(ATTNJVP_EINVAL, "B, H, N_q, N_kv must be >= 1");
  if (B * H >= (int64_t(1) << 31) || N_q >= (int64_t(1) << 31) || N_kv >= (int64_t(1) << 31))
    return fail(ATTNJVP_EINVAL, "B*H, N_q and N_kv must be < 2^31");
  if (!std::isfinite(scale) || !(scale > 0.f)) return fail(ATTNJVP_EINVAL, "scale must be finite and > 0");
  int rc = check_head_dim(d, false);
  if (rc != ATTNJVP_OK) return rc;
  if (((N_q + 127) / 128) * B * H * 2 >= (int64_t(1) << 31) ||
      ((N_kv + 127) / 128) * B * H * 2 >= (int64_t(1) << 31))
    return fail(ATTNJVP_EINVAL, "too many row tiles");
  const int64_t need = attn_bwd_workspace_floats(B, H, N_q) * 4;
  if (workspace_bytes < need)
    return fail(ATTNJVP_EINVAL, "workspace holds %lld bytes, needs %lld", (long long)workspace_bytes, (long long)need);
  const char* why = "";
  int* st = status_word(&why);
  if (!st) return fail(ATTNJVP_ECUDA, "no CUDA device / status word: %s", why);
  BwdArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.dout = dout;
  a.out = out;
  a.lse = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.B = B;
  a.H = H;
  a.Nq = N_q;
  a.Nkv = N_kv;
  a.d = d;
  a.scale = scale;
  a.ws = static_cast<float*>(workspace);
  a.status = st;
  a.stream = static_cast<cudaStream_t>(stream);
  const char* msg = "";
  cudaError_t e = launch_attn_bwd(a, &msg);
  if (e != cudaSuccess) return fail(ATTNJVP_ECUDA, "%s: %s", msg, cudaGetErrorString(e));
  return ok();
}

int trigflow_coeffs_jvp(double t, double v, double tau, double* out) {
  if (!out) return fail(ATTNJVP_EINVAL, "out is NULL");
  if (!std::isfinite(t) || !std::isfinite(v) || !std::isfinite(tau))
    return fail(ATTNJVP_EINVAL, "t, v and tau must be finite");
  const double c = std::cos(t), s = std::sin(t), den = c + s;
  if (!(den > 0.0)) return fail(ATTNJVP_EINVAL, "cos t + sin t must be > 0 (t in (-pi/4, 3pi/4))");
  const double den2 = den * den;
  out[0] = 1.0 / den;
  out[1] = -s / den;
  out[2] = 1.0 / den;
  out[3] = tau * s / den;
  out[4] = v * (-(c - s) / den2);
  out[5] = v * (-1.0 / den2);
  out[6] = v * (-(c - s) / den2);
  out[7] = v * (tau / den2);
  return ok();
}

namespace {
int check_epilogue_shape(int64_t B, int64_t C, int64_t T, int64_t HW) {
  if (B < 1 || C < 1 || T < 1 || HW < 1) return fail(ATTNJVP_EINVAL, "B, C, T, HW must be >= 1");
  const int64_t lim = int64_t(1) << 31;
  if (B >= lim || C >= lim || T >= lim || HW >= (int64_t(1) << 40) || B * C >= lim || B * C * T >= lim)
    return fail(ATTNJVP_EINVAL, "B * C * T must be < 2^31 and HW < 2^40");
  if ((B * C * T) > (int64_t(1) << 46) / HW) return fail(ATTNJVP_EINVAL, "tensor too large");
  if (epilogue_items(B, C, T, 1) * ((HW + 2047) / 2048) >= lim) return fail(ATTNJVP_EINVAL, "tensor too large");
  return ATTNJVP_OK;
}
}  // namespace

int trigflow_output_jvp(const float* x, const float* n, const float* x_t, const float* n_t, const double* t,
                        const double* t_t, float* F, float* F_t, int64_t B, int64_t C, int64_t T, int64_t HW,
                        void* stream) {
  const void* ptrs[8] = {x, n, x_t, n_t, t, t_t, F, F_t};
  for (const void* p : ptrs)
    if (!p) return fail(ATTNJVP_EINVAL, "NULL tensor");
  for (int i = 0; i < 8; ++i)
    if (!aligned(ptrs[i], (i == 4 || i == 5) ? 8 : 4)) return fail(ATTNJVP_EINVAL, "misaligned tensor");
  int rc = check_epilogue_shape(B, C, T, HW);
  if (rc != ATTNJVP_OK) return rc;
  int dev;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(ATTNJVP_ECUDA, "no CUDA device: %s", cudaGetErrorString(e));
  e = launch_output_jvp(x, n, x_t, n_t, t, t_t, F, F_t, B, C, T, HW, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(ATTNJVP_ECUDA, "output-JVP launch failed: %s", cudaGetErrorString(e));
  return ok();
}

int64_t scm_tangent_loss_workspace_bytes(int64_t B, int64_t C, int64_t T, int64_t HW) {
  int rc = check_epilogue_shape(B, C, T, HW);
  if (rc != ATTNJVP_OK) return rc;
  ok();
  return scm_workspace_doubles(B, C, T, HW) * 8;
}

int scm_tangent_loss(const float* F_theta, const float* F_sg, const float* F_teacher, const float* x,
                     const float* F_t, const double* t, double r, float* g_n, float* df_dt, double* loss,
                     int32_t* nan_g, int32_t* nan_F, int64_t B, int64_t C, int64_t T, int64_t HW, void* workspace,
                     int64_t workspace_bytes, void* stream) {
  const void* ptrs[12] = {F_theta, F_sg, F_teacher, x, F_t, t, g_n, df_dt, loss, nan_g, nan_F, workspace};
  for (const void* p : ptrs)
    if (!p) return fail(ATTNJVP_EINVAL, "NULL tensor or workspace");
  for (int i = 0; i < 12; ++i)
    if (!aligned(ptrs[i], (i == 5 || i == 8 || i == 11) ? 8 : 4)) return fail(ATTNJVP_EINVAL, "misaligned tensor");
  if (!std::isfinite(r) || r < 0.0 || r > 1.0) return fail(ATTNJVP_EINVAL, "warm-up ratio r must be in [0, 1]");
  int rc = check_epilogue_shape(B, C, T, HW);
  if (rc != ATTNJVP_OK) return rc;
  const int64_t need = scm_workspace_doubles(B, C, T, HW) * 8;
  if (workspace_bytes < need)
    return fail(ATTNJVP_EINVAL, "workspace holds %lld bytes, needs %lld", (long long)workspace_bytes,
                (long long)need);
  const char* why = "";
  int* st = status_word(&why);
  if (!st) return fail(ATTNJVP_ECUDA, "no CUDA device / status word: %s", why);
  cudaError_t e = launch_scm_tangent_loss(F_theta, F_sg, F_teacher, x, F_t, t, r, g_n, df_dt, loss, nan_g, nan_F, B,
                                          C, T, HW, static_cast<double*>(workspace), st,
                                          static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(ATTNJVP_ECUDA, "sCM tangent/loss launch failed: %s", cudaGetErrorString(e));
  return ok();
}

int attn_jvp_selftest_wait(int64_t limit_ns, void* stream) {
  if (limit_ns < 1000 || limit_ns > 2000000000) return fail(ATTNJVP_EINVAL, "limit_ns must be in [1e3, 2e9]");
  const char* why = "";
  int* st = status_word(&why);
  if (!st) return fail(ATTNJVP_ECUDA, "no CUDA device / status word: %s", why);
  cudaError_t e = launch_wait_selftest(st, static_cast<uint64_t>(limit_ns), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(ATTNJVP_ECUDA, "self-test launch failed: %s", cudaGetErrorString(e));
  return ok();
}

int attn_jvp_status(int clear) {
  const char* why = "";
  int* st = status_word(&why);
  if (!st) return fail(ATTNJVP_ECUDA, "no CUDA device / status word: %s", why);
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail(ATTNJVP_ECUDA, "synchronize failed: %s", cudaGetErrorString(e));
  int word = 0;
  e = cudaMemcpy(&word, st, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(ATTNJVP_ECUDA, "status read failed: %s", cudaGetErrorString(e));
  if (clear) {
    const int zero = 0;
    e = cudaMemcpy(st, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return fail(ATTNJVP_ECUDA, "status clear failed: %s", cudaGetErrorString(e));
  }
  if (word & kStatusTimeout) return fail(ATTNJVP_ETIMEOUT, "a kernel's bounded wait ran out (status 0x%x)", word);
  return ok();
}

const char* attn_jvp_last_error(void) { return g_last_error; }

const char* attn_jvp_version(void) { return "0.1.0"; }

}  // extern "C"
