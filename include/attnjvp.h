/*
 * attnjvp.h — C ABI of the GB300 (sm_103a) forward-mode attention-JVP library.
 *
 * Operation (page "带分数正则的一致性蒸馏", gitcode.csdn.net, section 注意力
 * (attention) and section 前向 (forward)): for every batch b, head h and query
 * row i, with s the softmax scale,
 *     S_ij  = s q_i . k_j                      P_i = softmax_j(S_ij)
 *     St_ij = s (qt_i . k_j + q_i . kt_j)      (tangent of the scores, t_s)
 *     O_i   = sum_j P_ij v_j                   LSE_i = ln sum_j exp(S_ij)
 *     mu_i  = sum_j P_ij St_ij
 *     Ot_i  = sum_j P_ij vt_j + sum_j P_ij (St_ij - mu_i) v_j
 * i.e. the JVP t_o = P t_v + t_p V with t_p = P (.) t_s - (P t_s^T) P.  The
 * output tangent is a stop-gradient value: nothing here builds a graph.
 * Attention is non-causal and unmasked; attn_jvp_fwd_strided allows a different
 * number of keys than queries.
 *
 * Conventions for every entry point:
 *   - Tensors are DEVICE pointers (unless stated otherwise), row-major and
 *     contiguous.  Attention tensors are [B, H, N, d]; per-row outputs are
 *     [B, H, N].  The caller allocates and owns every buffer; the library keeps
 *     no pointer after a call returns.
 *   - ``stream`` is a cudaStream_t (NULL = legacy default stream).  Work is
 *     enqueued asynchronously on it; a return value of 0 means "validated and
 *     launched", not "finished".
 *   - Return value: 0 on success or a negative ATTNJVP_E* code; the matching
 *     human-readable message is available from attn_jvp_last_error() on the
 *     same host thread.  No entry point aborts, throws or falls back to the CPU.
 *   - Kernels wait on on-chip barriers with a bounded budget (one second per
 *     wait).  A wait that runs out records ATTNJVP_ETIMEOUT in a per-device
 *     status word, the kernel releases what it holds and returns early; read
 *     the word with attn_jvp_status() after synchronising the stream.
 *   - The library looks up the device addresses of its own device arrays (the
 *     status word, the no-alloc scratch) once per device and keeps them, so it
 *     does not survive cudaDeviceReset, or any other teardown of a device's
 *     primary context, while it is loaded.  For the same lifetime it keeps, per
 *     device, one stream-ordered memory pool for the partial outputs of a cut
 *     last wave (see attn_jvp_fwd), which it does not give back to the system.
 *   - Calls may be captured into a CUDA graph once the same entry point has run
 *     on the device outside capture (the first call looks up the device state
 *     above, which capture does not allow).  Under capture, the stream-ordered
 *     allocations of the fp32 path and of a cut last wave become graph memory
 *     nodes from the device's default pool.
 */
#ifndef ATTNJVP_H
#define ATTNJVP_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ATTNJVP_OK 0
#define ATTNJVP_EINVAL (-1)       /* bad argument: null / misaligned pointer, bad size, bad scale */
#define ATTNJVP_EUNSUPPORTED (-2) /* valid request this build does not implement (e.g. head dim) */
#define ATTNJVP_ECUDA (-3)        /* a CUDA runtime or driver call failed */
#define ATTNJVP_ETIMEOUT (-4)     /* a kernel's bounded wait ran out (see attn_jvp_status) */

/* Input dtype codes of the forward entry points (the ``dtype`` argument). */
#define ATTNJVP_BF16 0 /* bfloat16: read in place by the kernels (the timed path) */
#define ATTNJVP_FP32 1 /* float32: rounded to bf16 (nearest even) on the device first */

/*
 * Fused attention forward + JVP (the operation above) over all N keys.
 *   q, k, v, q_t, k_t, v_t : [B, H, N, d] of the type ``dtype`` names; each base
 *                            16-byte aligned.  Tangents have exactly the primals'
 *                            shape, layout and type (the page's host wrapper asserts
 *                            equal shape and stride, and its forward takes q in its
 *                            own dtype).
 *   out, out_t             : fp32 [B, H, N, d] — O and Ot; 16-byte aligned.
 *   lse, mu                : fp32 [B, H, N] — natural-log LSE and mu; either may be
 *                            NULL when not wanted.
 *   B, H, N                : >= 1 each; B*H < 2^31 and N < 2^31.
 *   d                      : head dimension: 16, 32, 64, 128 or 256 (the page's set;
 *                            others: ATTNJVP_EUNSUPPORTED).  At 256 two CTAs share a
 *                            128-row query tile, each accumulating half of the value
 *                            columns, so the scores are computed twice.
 *   scale                  : softmax scale s, finite and > 0 (the page's default is d^-1/2).
 *   dtype                  : ATTNJVP_BF16 or ATTNJVP_FP32 (any other code:
 *                            ATTNJVP_EINVAL).  The tensor cores take bf16 operands,
 *                            so fp32 inputs are rounded to bf16 (nearest even) on
 *                            the device before the same kernel runs.  The six bf16
 *                            copies (6 * B * H * N * d * 2 bytes) live in memory
 *                            the library takes with cudaMallocAsync on ``stream``
 *                            and gives back with cudaFreeAsync on ``stream`` after
 *                            the kernel (stream-ordered; no device synchronisation);
 *                            ATTNJVP_ECUDA if that allocation fails.  The outputs
 *                            are fp32 either way.
 * Last wave: the kernel runs one CTA per SM, so its units (a 128-row query tile,
 * or a value half of one at d = 256) run in waves of the SM count.  When the
 * last wave would be at most half full, each of its units is cut into 2 to 16
 * pieces over consecutive key ranges (at least four 64-key tiles each), which
 * spread over the whole GPU, and one more kernel merges them exactly (the
 * key-chunk merge).  The pieces' partial outputs, at most SMs x 128 rows x
 * (2 min(d, 128) + 2) floats, come from the library's stream-ordered pool on
 * ``stream``.  A cut row rounds P~ against its piece's own maximum, so it can
 * differ from an uncut computation in the last bits (within the tolerances
 * above); every other row is computed exactly as without the cut.
 */
int attn_jvp_fwd(const void* q, const void* k, const void* v,
                 const void* q_t, const void* k_t, const void* v_t,
                 float* out, float* out_t, float* lse, float* mu,
                 int64_t B, int64_t H, int64_t N, int64_t d,
                 float scale, int dtype, void* stream);

/*
 * Pieces per unit into which attn_jvp_fwd (and attn_jvp_fwd_ex / _strided over
 * the whole key range) cuts the last wave of this shape on the current device
 * (see "Last wave" above): 1 when it does not cut.  When it cuts, such a call
 * makes two kernel launches (the fused kernel, then the merge of the pieces)
 * instead of one.
 *   B, H, N_q, N_kv : >= 1 (B*H, N_q and N_kv below 2^31).
 *   d_v             : the value head dim (16, 32, 64, 128 or 256).
 *   split           : HOST; receives the count.
 * Returns ATTNJVP_ECUDA without a CUDA device.  Launches nothing.
 */
int attn_jvp_fwd_last_wave_split(int64_t B, int64_t H, int64_t N_q, int64_t N_kv,
                                 int64_t d_v, int64_t* split);

/*
 * Same operation restricted to the key range [kv_start, kv_start + kv_len):
 * every query row attends only to those keys.  The outputs are the chunk's
 * own normalised partials (O_c, Ot_c, LSE_c, mu_c); attn_jvp_merge combines
 * chunks exactly.  Arguments as attn_jvp_fwd, plus:
 *   lse, mu   : required (not NULL) — the merge needs them.
 *   kv_start  : >= 0;  kv_len >= 1;  kv_start + kv_len <= N.
 * A chunk is never cut into pieces (its caller merges chunks), so this call
 * takes no memory of its own for bf16 inputs.
 * (The page has no key split; chunking is exact algebra on the definitions above.)
 */
int attn_jvp_fwd_chunk(const void* q, const void* k, const void* v,
                       const void* q_t, const void* k_t, const void* v_t,
                       float* out, float* out_t, float* lse, float* mu,
                       int64_t B, int64_t H, int64_t N, int64_t d,
                       float scale, int dtype, int64_t kv_start, int64_t kv_len, void* stream);

/*
 * General form: strided layouts, as many or as few keys as queries, and an
 * optional key range.  Element (b, s, h, c) of a tensor is at
 *     b * stride_batch + s * stride_seq + h * stride_head + c
 * elements from its base (the head-dimension stride is 1), so [B, H, S, d],
 * the page's [B, S, H, d], and views such as q/k/v slices of a packed
 * [B, S, 3, H, d] tensor are all accepted without copies.
 *   q, q_t              : N_q query rows; share the query strides.
 *   k, k_t, v, v_t      : N_kv key rows; share the key strides (the page's
 *                         wrapper requires tangents to have the primals' strides).
 *                         All six of the type ``dtype`` names (as attn_jvp_fwd;
 *                         fp32 inputs are gathered into contiguous bf16 copies).
 *   out, out_t          : fp32 O and Ot at the output strides; 16-byte aligned.
 *   lse, mu             : fp32 [B, H, N_q] contiguous, or NULL.
 *   B, H, N_q, N_kv     : >= 1 each (cross-attention when N_q != N_kv).
 *   d                   : 16, 32, 64, 128 or 256.
 *   strides             : HOST array of 9 element strides — query (batch, seq,
 *                         head), key (batch, seq, head), output (batch, seq,
 *                         head) — or NULL for contiguous [B, H, N, d] everywhere.
 *                         Input strides must be non-negative multiples of 8
 *                         elements for bf16 (16 bytes, a TMA rule) and of 4 for
 *                         fp32 (16-byte loads), output strides multiples of 4; a
 *                         stride is ignored when its extent is 1.
 *                         Layouts in which output elements overlap give
 *                         unspecified results.
 *   kv_start, kv_len    : key range [kv_start, kv_start + kv_len) within [0, N_kv);
 *                         the whole range gives the full result (with the cut of
 *                         a short last wave of attn_jvp_fwd), a sub-range the
 *                         chunk partials of attn_jvp_fwd_chunk (never cut).
 * (The page's host wrapper hands [B, S, H, D] tensors to its kernel as
 * transposed views together with their strides; its section 前向 (forward)
 * allows seqlen_q != seqlen_kv and head dims {16, 32, 64, 128, 256}.)
 */
int attn_jvp_fwd_strided(const void* q, const void* k, const void* v,
                         const void* q_t, const void* k_t, const void* v_t,
                         float* out, float* out_t, float* lse, float* mu,
                         int64_t B, int64_t H, int64_t N_q, int64_t N_kv, int64_t d,
                         const int64_t* strides, float scale, int dtype,
                         int64_t kv_start, int64_t kv_len, void* stream);

/*
 * Most general form: attn_jvp_fwd_strided with a value head dim of its own.
 * V, Vt, O and Ot have d_v columns per head, Q, Qt, K and Kt have d.  (The
 * page's section 前向 (forward) documents v, tv as [B, H, S_kv, d_v] and o, to
 * as [B, H, S_q, d_v], with d_v free in the forward; its backward needs
 * d_v = d_qk.)  The default softmax scale there is d^-1/2 of the Q/K dim.
 *   d, d_v              : 16, 32, 64, 128 or 256 each.
 *   strides             : HOST array of 12 element strides — query, key, value
 *                         and output, each (batch, seq, head) — or NULL for
 *                         contiguous [B, H, N, d] (q, k) and [B, H, N, d_v]
 *                         (v, out) tensors.  Same rules as attn_jvp_fwd_strided.
 * Other arguments, ownership and errors as attn_jvp_fwd_strided, which is this
 * call with d_v = d and the key strides used for the values too.
 */
int attn_jvp_fwd_ex(const void* q, const void* k, const void* v,
                    const void* q_t, const void* k_t, const void* v_t,
                    float* out, float* out_t, float* lse, float* mu,
                    int64_t B, int64_t H, int64_t N_q, int64_t N_kv, int64_t d, int64_t d_v,
                    const int64_t* strides, float scale, int dtype,
                    int64_t kv_start, int64_t kv_len, void* stream);

/*
 * Exact merge of C key-chunk partials into the full-row result:
 *   LSE = ln sum_c e^{LSE_c},  w_c = e^{LSE_c - LSE},
 *   O = sum_c w_c O_c,  mu = sum_c w_c mu_c,  Ot = sum_c w_c (Ot_c + mu_c O_c) - mu O.
 *   o_c, ot_c   : fp32 [C, B, H, N, d] (chunk-major), 16-byte aligned.
 *   lse_c, mu_c : fp32 [C, B, H, N].
 *   out, out_t  : fp32 [B, H, N, d], 16-byte aligned;  lse, mu : fp32 [B, H, N] or NULL.
 *   n_chunks    : C >= 1.  d: a multiple of 4, 4 <= d <= 256.
 * Outputs must not alias inputs.
 */
int attn_jvp_merge(const float* o_c, const float* ot_c, const float* lse_c, const float* mu_c,
                   int64_t n_chunks, float* out, float* out_t, float* lse, float* mu,
                   int64_t B, int64_t H, int64_t N, int64_t d, void* stream);

/*
 * Split-KV attention JVP (the same result as attn_jvp_fwd_chunk over
 * n_chunks near-equal key ranges followed by attn_jvp_merge) for callers that
 * may not allocate device memory: for example code that runs inside a host
 * framework which owns all device memory and passes in only an operation's
 * tensors, or a loop where the implicit device synchronisation of
 * cudaMalloc/cudaFree is not allowed.  The pages have no counterpart; this is
 * an interface convenience around the split path above.
 *   Arguments as attn_jvp_fwd (dtype included), plus n_chunks in [1, N]; lse
 *   and mu may be NULL.  Every argument is checked before anything is launched.
 *   The chunk partials live in a 16 MiB array built into the library (one per
 *   device that loads it, held until the process exits), so
 *   n_chunks * B * H * N * (2d + 2) * 4 bytes must not exceed 16 MiB; for fp32
 *   inputs their bf16 copies, 6 * B * H * N * d * 2 bytes, go there too and
 *   count against the same limit.  Larger requests return ATTNJVP_EINVAL with
 *   the sizes in the message.  No allocator is called.  The first call on a
 *   device looks up the array's device address (cudaGetSymbolAddress); make that
 *   first call before any stream capture.  Every call on a device uses the same
 *   array: calls that can overlap on the GPU (unordered streams, concurrent host
 *   threads) race and must be serialised by the caller.  Each call writes every
 *   partial before reading it, so nothing from an earlier call leaks into a
 *   result.
 */
int attn_jvp_fwd_split_noalloc(const void* q, const void* k, const void* v,
                               const void* q_t, const void* k_t, const void* v_t,
                               float* out, float* out_t, float* lse, float* mu,
                               int64_t B, int64_t H, int64_t N, int64_t d,
                               float scale, int dtype, int64_t n_chunks, void* stream);

/*
 * QK normalisation and its tangent, the input side of the attention JVP for a
 * student that keeps RMS-normalised queries and keys (page "带分数正则的
 * 一致性蒸馏", section 一致性模型 (consistency model): QK正则化).  The norm is
 * the per-head RMSNorm of the page "Обслуживание Ideogram v4 менее чем за
 * секунду" (dev48.org), section on fusing RMSNorm.  For every row of d values
 * (one token of one head):
 *   rho = 1 / sqrt(mean(x^2) + eps),   y = x rho w,
 *   yt  = w (xt rho - x rho^3 mean(x xt))       (the JVP of y along xt).
 * One call normalises the Q rows with w_q and the K rows with w_k; the outputs
 * feed attn_jvp_fwd as its q, q_t, k, k_t.
 *   q, q_t, k, k_t     : bf16 [rows_q, d] and [rows_k, d]: any layout in which each
 *                        head's d values are contiguous ([B, H, N, d] and the page's
 *                        [B, N, H, d] are both B*H*N rows); 16-byte aligned.
 *   w_q, w_k           : fp32 [d], the norms' per-channel weights; 16-byte aligned.
 *   qn, qn_t, kn, kn_t : bf16 outputs shaped like their inputs (rounded to nearest
 *                        even from fp32 arithmetic); each may alias its own input.
 *   rows_q, rows_k     : >= 0; a zero count leaves that tensor's pointers unused.
 *   d                  : 16, 32, 64, 128 or 256 (others: ATTNJVP_EUNSUPPORTED).
 *   eps                : finite and >= 0.
 */
int qk_rmsnorm_jvp(const void* q, const void* q_t, const void* k, const void* k_t,
                   const float* w_q, const float* w_k, void* qn, void* qn_t, void* kn, void* kn_t,
                   int64_t rows_q, int64_t rows_k, int64_t d, float eps, void* stream);

/*
 * Round fp32 to bf16 (nearest-even) element-wise on the device, so fp32 inputs
 * can be fed to the bf16 kernels.  in: fp32 [n]; out: bf16 [n]; n >= 0.
 * Both 16-byte aligned.
 */
int attn_jvp_cast_f32_bf16(const float* in, void* out, int64_t n, void* stream);

/*
 * TrigFlow-to-rectified-flow preconditioning coefficients in FP64 (page
 * "带分数正则的一致性蒸馏", section 时间步转换 (timestep conversion),
 * RectifiedFlow_TrigFlowWrapper with sigma_data = 1):
 *   c[0] = c_skip  = 1 / (cos t + sin t)
 *   c[1] = c_out   = -sin t / (cos t + sin t)
 *   c[2] = c_in    = 1 / (cos t + sin t)
 *   c[3] = c_noise = tau * sin t / (cos t + sin t)      (the page's config uses tau = 1000)
 * Host function; c is a HOST array of 4 doubles.  Returns ATTNJVP_EINVAL when
 * c is NULL, t or tau is not finite, or cos t + sin t <= 0 (t outside
 * (-pi/4, 3pi/4); the documented domain is [0, pi/2]).
 */
int trigflow_coeffs(double t, double tau, double* c);

/*
 * Time derivative of the TrigFlow forward process x_t = cos t x0 + sin t eps
 * (same page and section; also the velocity F of the section's wrapper):
 *   out[b, i] = -sin(t[b]) x0[b, i] + cos(t[b]) eps[b, i]
 *   x0, eps, out : fp32 [B, per_sample] (device), 16-byte aligned.
 *   t            : FP64 [B] (device); sin/cos are taken in FP64 once per sample.
 *   B >= 1, per_sample >= 1.  out may alias x0 or eps.
 */
int trigflow_tangent(const float* x0, const float* eps, const double* t, float* out,
                     int64_t B, int64_t per_sample, void* stream);

/*
 * Attention JVP on HOST-resident tensors: the same operation and result as
 * attn_jvp_fwd (n_chunks == 1) or the split path (n_chunks > 1), with the
 * host<->device transfers done by the library and overlapped with compute.
 * The pages have no counterpart; it serves callers whose tensors live in host
 * memory and who would otherwise pay copy-in + compute + copy-out in series.
 *   q .. v_t            : HOST bf16 [B, H, N, d] (pinned memory for overlap;
 *                         pageable memory works but serialises the copies).
 *   out, out_t          : HOST fp32 [B, H, N, d];  lse, mu: HOST fp32 [B, H, N]
 *                         or NULL.
 *   B, H, N, d, scale   : as attn_jvp_fwd.
 *   n_chunks            : 1, or the number of key chunks of the split path (<= N).
 *   group_heads         : heads per pipelined item (>= 1), or 0 for automatic
 *                         (about 608 CTAs per item: four waves on a 152-SM GB300).
 *   workspace           : DEVICE buffer, 256-byte aligned, of at least
 *                         attn_jvp_fwd_host_workspace_bytes(B, H, N, d, n_chunks,
 *                         group_heads) bytes (three slots of group_heads heads);
 *                         owned by the caller.
 * Items of at most group_heads heads of one batch entry rotate through three
 * workspace slots, each computed on its own library-owned stream; item i+1 is
 * copied in and item i-1 copied out on two more library-owned streams while
 * item i computes, and consecutive items' kernels may overlap on the GPU.  The
 * first and last items are cut to a quarter group to shorten the exposed
 * first copy-in and last copy-out.
 * On return the work is enqueued; once ``stream`` has been synchronised every
 * output is in host memory.  Inputs must stay unchanged, and outputs unread,
 * until then.  Calls that share a workspace must be ordered on one stream.
 * Each item runs the device entry points on a [group, N, d] slice, so its
 * results equal a device-resident call on that slice bit for bit, and a call
 * on the whole tensor wherever neither call cuts a short last wave (see
 * attn_jvp_fwd).
 */
int attn_jvp_fwd_host(const void* q, const void* k, const void* v,
                      const void* q_t, const void* k_t, const void* v_t,
                      float* out, float* out_t, float* lse, float* mu,
                      int64_t B, int64_t H, int64_t N, int64_t d, float scale,
                      int64_t n_chunks, int64_t group_heads,
                      void* workspace, int64_t workspace_bytes, void* stream);

/*
 * Device workspace, in bytes, that attn_jvp_fwd_host needs for these sizes,
 * or a negative ATTNJVP_E* code for arguments attn_jvp_fwd_host would reject.
 * Needs no GPU.
 */
int64_t attn_jvp_fwd_host_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t d,
                                          int64_t n_chunks, int64_t group_heads);

/*
 * Primal attention backward (page section 反向 (backward)): for the upstream
 * gradient dO of O = softmax(s Q K^T) V,
 *   dV = P^T dO,  dP = dO V^T,  dS = P (.) (dP - rowsum(dP (.) P)),
 *   dQ = s dS K,  dK = s dS^T Q.
 *   q, dout        : bf16 [B, H, N_q, d];  k, v: bf16 [B, H, N_kv, d]; 16-byte aligned.
 *   out, lse       : the forward's O (fp32 [B, H, N_q, d]) and natural-log LSE
 *                    (fp32 [B, H, N_q]), as attn_jvp_fwd / attn_jvp_fwd_strided
 *                    write them.  P is rebuilt from lse; rowsum(dP (.) P) is
 *                    taken as rowsum(dO (.) O), equal since O = P V.
 *   dq, dk, dv     : fp32, shaped like q, k, v; 16-byte aligned.
 *   d              : 16, 32, 64, 128 or 256 (at 256 two CTAs share each row tile, each
 *                    accumulating half of the gradient columns, as dK and dV of 128
 *                    keys would fill tensor memory);  scale: the forward's scale.
 *   workspace      : DEVICE, 256-byte aligned, attn_bwd_workspace_bytes(B, H, N_q).
 * Two passes (keys resident for dK/dV, queries resident for dQ) recompute the
 * scores instead of accumulating dQ with atomics, so results are reproducible.
 * Each pass cuts a short last wave as attn_jvp_fwd does, over its streamed rows
 * (queries for dK/dV, keys for dQ), and adds the pieces' partial sums in a
 * second kernel; the partial sums come from the library's stream-ordered pool on
 * ``stream``.  The pieces fix the order of those additions, so results stay
 * reproducible for a given shape and GPU.
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* dout,
             const float* out, const float* lse, float* dq, float* dk, float* dv,
             int64_t B, int64_t H, int64_t N_q, int64_t N_kv, int64_t d, float scale,
             void* workspace, int64_t workspace_bytes, void* stream);

/* Workspace bytes attn_bwd needs, or a negative ATTNJVP_E* code.  Needs no GPU. */
int64_t attn_bwd_workspace_bytes(int64_t B, int64_t H, int64_t N_q);

/*
 * ---- Output side of one consistency step (page "带分数正则的一致性蒸馏",
 * section 一致性模型 (consistency model), its 蒸馏代码 listing). ----
 * Latent tensors are fp32 [B, C, T, HW] (the page's B_C_T_H_W with H and W
 * merged), contiguous, 4-byte aligned; the time t is FP64 [B, T] (one value
 * per batch entry and frame, broadcast over channels and pixels).
 */

/*
 * The wrapper coefficients at time t and their tangents (the page's
 * torch.func.jvp of its scaling function along v): out[0..3] = c_skip, c_out,
 * c_in, c_noise (as trigflow_coeffs); out[4..7] = v * d/dt of each.  Host
 * function, FP64.  EINVAL unless cos t + sin t > 0 and t, v, tau are finite.
 */
int trigflow_coeffs_jvp(double t, double v, double tau, double* out);

/*
 * The student prediction F from the network output and its tangent (the JVP
 * of the page's _process_output):
 *   x0 = c_skip(t) x + c_out(t) n,   F = (cos t x - x0) / sin t,
 *   F_t = d F along (x_t, n_t, t_t), the coefficients differentiated through t.
 *   x, n, x_t, n_t : DEVICE fp32 [B, C, T, HW]  (x = x_t of the process, n = the
 *                    network output, and their tangents).
 *   t, t_t         : DEVICE FP64 [B, T]; sin t must be non-zero.
 *   F, F_t         : DEVICE fp32 [B, C, T, HW].
 *   B * C * T < 2^31.  Coefficients are formed per frame in FP64, the
 *   elementwise arithmetic is fp32.
 */
int trigflow_output_jvp(const float* x, const float* n, const float* x_t, const float* n_t,
                        const double* t, const double* t_t, float* F, float* F_t,
                        int64_t B, int64_t C, int64_t T, int64_t HW, void* stream);

/*
 * Tangent target and sCM loss:
 *   g     = -cos t sqrt(1 - r^2 sin^2 t) (F_sg - F_teacher) - (r cos t sin t x + F_t)
 *   df_dt = -cos t (F_sg - F_teacher) - (sin t x + F_t)          (never masked)
 *   nan_g[b] / nan_F[b] = 1 when any element of sample b of g / F_theta is NaN;
 *   a flagged sample has g, F_theta and F_sg taken as 0;
 *   g_n   = g / (||g[b]||_2 + 0.1)                                (norm in FP64)
 *   loss[b] = sum over sample b of (F_theta - F_sg - g_n)^2       (FP64)
 *   F_theta, F_sg, F_teacher, x, F_t : DEVICE fp32 [B, C, T, HW] (student output,
 *                    its stop-gradient copy, teacher output, x_t, student tangent).
 *   t              : DEVICE FP64 [B, T].   r: warm-up ratio in [0, 1].
 *   g_n, df_dt     : DEVICE fp32 [B, C, T, HW] outputs (g_n rounded from FP64).
 *   loss           : DEVICE FP64 [B];  nan_g, nan_F: DEVICE int32 [B].
 *   workspace      : DEVICE, 8-byte aligned, scm_tangent_loss_workspace_bytes()
 *                    bytes.  It holds the call's per-item sums and its
 *                    scheduling counters, which the call resets itself (no
 *                    zeroing needed); calls that may run at the same time
 *                    (other streams) need workspaces of their own.  The sums
 *                    are reduced per sample in a fixed order, so
 *                    results are reproducible run to run.  The loss is formed
 *                    as sum a^2 - 2 s sum a g + s^2 sum g^2 (a = F_theta - F_sg,
 *                    s = 1 / (||g|| + 0.1)), exact algebra on the sum above.
 */
int scm_tangent_loss(const float* F_theta, const float* F_sg, const float* F_teacher,
                     const float* x, const float* F_t, const double* t, double r,
                     float* g_n, float* df_dt, double* loss, int32_t* nan_g, int32_t* nan_F,
                     int64_t B, int64_t C, int64_t T, int64_t HW,
                     void* workspace, int64_t workspace_bytes, void* stream);

/* Workspace bytes scm_tangent_loss needs, or a negative ATTNJVP_E* code.  Needs no GPU. */
int64_t scm_tangent_loss_workspace_bytes(int64_t B, int64_t C, int64_t T, int64_t HW);

/*
 * Failure-path self-test.  Launches one tiny kernel on ``stream`` that waits,
 * with the same bounded-wait routine the attention kernels use, on an
 * on-chip barrier nothing ever completes; the wait gives up after
 * ``limit_ns`` nanoseconds (1e3 .. 2e9) and records ATTNJVP_ETIMEOUT in the
 * device's status word, exactly as a stuck attention kernel would, without
 * faulting or hanging the GPU.  Afterwards attn_jvp_status() reports
 * ATTNJVP_ETIMEOUT (and clears the word when asked).  While the word is set,
 * attention kernels skip their work, so clear it before further launches.
 */
int attn_jvp_selftest_wait(int64_t limit_ns, void* stream);

/*
 * Reads (and, if ``clear`` is non-zero, resets) the status word of the current
 * device after a device-wide synchronisation.  Returns 0 when no kernel has
 * reported a problem since the last clear, ATTNJVP_ETIMEOUT when a bounded
 * wait ran out, ATTNJVP_ECUDA when the word cannot be read.
 */
int attn_jvp_status(int clear);

/* Message for the last non-zero return on the calling host thread ("" if none). */
const char* attn_jvp_last_error(void);

/* Library version, e.g. "0.1.0". */
const char* attn_jvp_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTNJVP_H */
