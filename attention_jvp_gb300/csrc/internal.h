// Internal launch interface between the C-ABI layer (capi.cu) and the kernel
// translation units.  Not installed; not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace attnjvp {

// Status bits a kernel ORs into the per-device status word.
constexpr int kStatusTimeout = 1;

struct FwdArgs {
  const void *q, *k, *v, *q_t, *k_t, *v_t;  // bf16; element (b, s, h, c) at b*st[0] + s*st[1] + h*st[2] + c
  float *out, *out_t, *lse, *mu;            // fp32 O, Ot at the output strides; lse/mu [B, H, Nq] or null
  int64_t B, H, Nq, Nkv;
  int64_t d, d_v;                           // head dims of Q/K and of V/O (each 16, 32, 64, 128 or 256)
  // element strides (batch, seq, head) of Q (and Qt), K (and Kt), V (and Vt), O (and Ot); head-dim stride 1
  int64_t q_stride[3], k_stride[3], v_stride[3], o_stride[3];
  float scale;
  int64_t kv_start, kv_len;
  int* status;                               // device status word
  cudaStream_t stream;
  // Cut the units of a short last wave into pieces over the keys (stream-ordered
  // allocation of their partial outputs and one merge launch).  Off for callers
  // that must not allocate and for key chunks, which are merged by their callers.
  bool balance_tail = false;
};

// Returns cudaSuccess or the failing CUDA error; ``*msg`` gets a static message.
cudaError_t launch_attn_jvp_fwd(const FwdArgs& a, const char** msg);

// Pieces per unit into which a balanced launch cuts the last wave of a grid of
// ``grid`` units over kv_len keys on n_sm SMs (1: no cut); the current device's
// SM count (0 if unknown).
int64_t last_wave_split(int64_t grid, int64_t kv_len, int n_sm);

// The current device's SM count, looked up once per device (0 if unknown).
int device_sm_count();
// Raises ``func``'s dynamic shared-memory limit to ``bytes`` on the current
// device, once per (kernel, device); ``*first`` tells whether this call did it.
// Thread-safe.
cudaError_t ensure_smem_limit(const void* func, int bytes, bool* first);
// Stream-ordered allocation of the last wave's partial outputs on ``stream``: from
// a per-device pool that keeps its memory mapped between calls (and lives as
// long as the process), or, while the stream is being captured into a CUDA
// graph, from the default pool as a graph memory node.  Freed with cudaFreeAsync.
cudaError_t piece_alloc(void** ptr, size_t bytes, cudaStream_t stream);

cudaError_t launch_merge(const float* o_c, const float* ot_c, const float* lse_c, const float* mu_c,
                         int64_t n_chunks, float* out, float* out_t, float* lse, float* mu, int64_t rows,
                         int64_t d, cudaStream_t stream);

cudaError_t launch_cast_f32_bf16(const float* in, void* out, int64_t n, cudaStream_t stream);

// fp32 element (b, s, h, c) at b*stride[0] + s*stride[1] + h*stride[2] + c -> contiguous
// bf16 [B, H, S, d]; d and the strides are multiples of 4, ``in`` 16-byte aligned.
cudaError_t launch_cast_strided_f32_bf16(const float* in, void* out, int64_t B, int64_t H, int64_t S, int64_t d,
                                         const int64_t stride[3], cudaStream_t stream);

cudaError_t launch_trigflow_tangent(const float* x0, const float* eps, const double* t, float* out, int64_t B,
                                    int64_t per_sample, cudaStream_t stream);

cudaError_t launch_wait_selftest(int* status, uint64_t limit_ns, cudaStream_t stream);

// Primal attention backward (attn_bwd.cu); contiguous [B, H, N, d] tensors.
struct BwdArgs {
  const void *q, *k, *v, *dout;  // bf16
  const float *out, *lse;        // forward's O (fp32) and natural-log LSE
  float *dq, *dk, *dv;           // fp32
  int64_t B, H, Nq, Nkv, d;
  float scale;
  float* ws;                     // attn_bwd_workspace_floats() floats
  int* status;
  cudaStream_t stream;
};
int64_t attn_bwd_workspace_floats(int64_t B, int64_t H, int64_t Nq);
cudaError_t launch_attn_bwd(const BwdArgs& a, const char** msg);

// QK normalisation and its tangent (qk_norm.cu); rows of d contiguous bf16 values.
struct QkNormArgs {
  const __nv_bfloat16 *q, *q_t, *k, *k_t;  // inputs; 16-byte aligned
  const float *w_q, *w_k;                  // per-channel weights [d]; 16-byte aligned
  __nv_bfloat16 *qn, *qn_t, *kn, *kn_t;    // outputs (may alias their own input)
  int64_t rows_q, rows_k;
  int d;                                   // 16, 32, 64, 128 or 256
  float eps;
};
cudaError_t launch_qk_rmsnorm_jvp(const QkNormArgs& a, cudaStream_t stream);

// Output side of a consistency step (epilogue.cu).
int64_t epilogue_items(int64_t B, int64_t C, int64_t T, int64_t HW);  // launch blocks
int64_t scm_workspace_doubles(int64_t B, int64_t C, int64_t T, int64_t HW);
cudaError_t launch_output_jvp(const float* x, const float* n, const float* tx, const float* tn, const double* t,
                              const double* tt, float* F, float* tF, int64_t B, int64_t C, int64_t T, int64_t HW,
                              cudaStream_t stream);
cudaError_t launch_scm_tangent_loss(const float* F_theta, const float* F_sg, const float* F_tc, const float* x,
                                    const float* tF, const double* t, double r, float* g_n, float* dfdt,
                                    double* loss, int* nan_g, int* nan_F, int64_t B, int64_t C, int64_t T, int64_t HW,
                                    double* ws, int* status, cudaStream_t stream);

// Argument checks shared by the forward entry points (capi.cu): pointers, alignment,
// sizes, scale, head dim and the dtype code.  Returns 0 or an ATTNJVP_E* code with
// attn_jvp_last_error() set; needs no GPU.
int check_attn_args(const void* q, const void* k, const void* v, const void* q_t, const void* k_t, const void* v_t,
                    const float* out, const float* out_t, const float* lse, const float* mu, int64_t B, int64_t H,
                    int64_t N, int64_t d, float scale, int dtype);

// Sets the calling thread's message returned by attn_jvp_last_error().
void set_last_error(const char* msg);

// cuTensorMapEncodeTiled obtained through the runtime (no link-time libcuda dependency).
typedef CUresult (*TensorMapEncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                      const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                      CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
TensorMapEncodeFn tensor_map_encoder();

}  // namespace attnjvp
