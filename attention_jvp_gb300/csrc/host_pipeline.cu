// Attention JVP on host-resident tensors with transfers overlapped with compute.
//
// The work is cut into items of at most ``group_heads`` heads of one batch
// entry.  Three device workspace slots rotate between items, each with its own
// compute stream.  While item i computes, item i+1's six inputs are copied in
// on a copy stream and item i-1's outputs are copied out on another, so for
// long sequences the transfers hide behind the tensor-core work.  Because
// consecutive items compute on different streams, the next item's CTAs fill
// the SMs that the previous item's last wave leaves idle.  The first and the
// last item are cut to a quarter of a group, which shortens the only
// transfers left exposed: the first copy-in and the last copy-out.
//
// Each item runs the same device entry points as a device-resident call
// (attn_jvp_fwd, or attn_jvp_fwd_chunk + attn_jvp_merge when n_chunks > 1)
// on a [group, N, d] slice, so its results are bit-identical to a single
// device call on the whole tensors.
//
// Ordering rules:
// - The copy and compute streams are created once per device and shared by
//   all calls.
// - Every dependency is an event made for the call; nothing relies on stream
//   order between the copy streams and the caller's stream.
// - All work starts after an event recorded on the caller's stream at entry,
//   so an earlier call on the same stream that used the same workspace has
//   finished with it.
// - At exit the caller's stream waits for the last copy-out: synchronising
//   that stream means every output has landed in host memory.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <mutex>
#include <vector>

#include "../../include/attnjvp.h"
#include "internal.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kSlots = 3;
constexpr int64_t kAutoGroupCtas = 608;  // about four waves of one CTA per SM on a 152-SM GB300
constexpr int64_t kAlign = 256;

std::mutex g_mu;
struct DeviceStreams {
  cudaStream_t h2d = nullptr, d2h = nullptr, compute[kSlots] = {};
};
DeviceStreams g_streams[kMaxDevices];

int reject(int code, const char* msg) {
  attnjvp::set_last_error(msg);
  return code;
}

int cuda_fail(const char* what, cudaError_t e) {
  char msg[256];
  snprintf(msg, sizeof(msg), "%s: %s", what, cudaGetErrorString(e));
  attnjvp::set_last_error(msg);
  return ATTNJVP_ECUDA;
}

int64_t round_up(int64_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

int64_t resolve_group(int64_t H, int64_t N, int64_t group_heads) {
  if (group_heads > 0) return group_heads < H ? group_heads : H;
  const int64_t qtiles = (N + 127) / 128;
  int64_t g = (kAutoGroupCtas + qtiles - 1) / qtiles;
  if (g < 1) g = 1;
  return g < H ? g : H;
}

// Byte layout of one workspace slot for ``g`` heads.
struct Slot {
  int64_t in[6];                 // bf16 [g, N, d] each
  int64_t out, out_t, lse, mu;   // fp32 [g, N, d], [g, N, d], [g, N], [g, N]
  int64_t o_c, ot_c, lse_c, mu_c;  // chunk partials (n_chunks > 1): [C, g, N, d] x2, [C, g, N] x2
  int64_t bytes;
};

Slot slot_layout(int64_t g, int64_t N, int64_t d, int64_t n_chunks) {
  Slot s{};
  int64_t off = 0;
  const int64_t elems = g * N * d;
  for (int i = 0; i < 6; ++i) {
    s.in[i] = off;
    off += round_up(elems * 2);
  }
  s.out = off;
  off += round_up(elems * 4);
  s.out_t = off;
  off += round_up(elems * 4);
  s.lse = off;
  off += round_up(g * N * 4);
  s.mu = off;
  off += round_up(g * N * 4);
  if (n_chunks > 1) {
    s.o_c = off;
    off += round_up(n_chunks * elems * 4);
    s.ot_c = off;
    off += round_up(n_chunks * elems * 4);
    s.lse_c = off;
    off += round_up(n_chunks * g * N * 4);
    s.mu_c = off;
    off += round_up(n_chunks * g * N * 4);
  }
  s.bytes = off;
  return s;
}

int check_shape(int64_t B, int64_t H, int64_t N, int64_t d, int64_t n_chunks, int64_t group_heads) {
  if (B < 1 || H < 1 || N < 1) return reject(ATTNJVP_EINVAL, "B, H, N must be >= 1");
  if (d != 16 && d != 32 && d != 64 && d != 128 && d != 256)
    return reject(ATTNJVP_EUNSUPPORTED, "head dim not supported (16, 32, 64, 128, 256)");
  if (n_chunks < 1 || n_chunks > N) return reject(ATTNJVP_EINVAL, "n_chunks must be in [1, N]");
  if (group_heads < 0) return reject(ATTNJVP_EINVAL, "group_heads must be >= 0 (0 = automatic)");
  if (N >= (int64_t(1) << 31) || B * H >= (int64_t(1) << 31)) return reject(ATTNJVP_EINVAL, "B*H and N must be < 2^31");
  return ATTNJVP_OK;
}

// The library's streams of the current device, created on first use.
int device_streams(DeviceStreams* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail("no CUDA device", e);
  if (dev < 0 || dev >= kMaxDevices) return reject(ATTNJVP_ECUDA, "device ordinal out of range");
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceStreams& ds = g_streams[dev];
  if (!ds.h2d) {
    DeviceStreams made;
    cudaStream_t* all[2 + kSlots] = {&made.h2d, &made.d2h, &made.compute[0], &made.compute[1], &made.compute[2]};
    for (cudaStream_t* st : all) {
      e = cudaStreamCreateWithFlags(st, cudaStreamNonBlocking);
      if (e != cudaSuccess) {
        for (cudaStream_t* done : all)
          if (*done) cudaStreamDestroy(*done);
        return cuda_fail("creating the library's streams", e);
      }
    }
    ds = made;
  }
  *out = ds;
  return ATTNJVP_OK;
}

// Events of one call: entry, and per slot inputs-ready / compute-done / outputs-copied.
struct Events {
  cudaEvent_t entry = nullptr, in_ready[kSlots] = {}, computed[kSlots] = {}, copied[kSlots] = {};
  cudaError_t create() {
    cudaError_t e = cudaEventCreateWithFlags(&entry, cudaEventDisableTiming);
    for (int s = 0; s < kSlots && e == cudaSuccess; ++s) {
      e = cudaEventCreateWithFlags(&in_ready[s], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&computed[s], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&copied[s], cudaEventDisableTiming);
    }
    return e;
  }
  // Destroying an event with work pending is allowed: its resources are
  // released once that work completes.
  ~Events() {
    if (entry) cudaEventDestroy(entry);
    for (int s = 0; s < kSlots; ++s) {
      if (in_ready[s]) cudaEventDestroy(in_ready[s]);
      if (computed[s]) cudaEventDestroy(computed[s]);
      if (copied[s]) cudaEventDestroy(copied[s]);
    }
  }
};

struct Item {
  int64_t b, h0, heads;
};

// Items of at most g heads, none spanning two batch entries; the first and
// the last item are cut to ceil(g / 4) heads when the call has more than one item.
std::vector<Item> make_items(int64_t B, int64_t H, int64_t g) {
  std::vector<Item> items;
  for (int64_t b = 0; b < B; ++b)
    for (int64_t h0 = 0; h0 < H; h0 += g) items.push_back({b, h0, (H - h0) < g ? (H - h0) : g});
  const int64_t r = (g + 3) / 4;
  if (items.size() > 1 && items.front().heads > r) {
    Item& f = items.front();
    const Item rest{f.b, f.h0 + r, f.heads - r};
    f.heads = r;
    items.insert(items.begin() + 1, rest);
  }
  if (items.size() > 1 && items.back().heads > r) {
    Item& l = items.back();
    const Item tail{l.b, l.h0 + l.heads - r, r};
    l.heads -= r;
    items.push_back(tail);
  }
  return items;
}

}  // namespace

extern "C" int64_t attn_jvp_fwd_host_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t d, int64_t n_chunks,
                                                     int64_t group_heads) {
  int rc = check_shape(B, H, N, d, n_chunks, group_heads);
  if (rc != ATTNJVP_OK) return rc;
  const int64_t g = resolve_group(H, N, group_heads);
  attnjvp::set_last_error("");
  return kSlots * slot_layout(g, N, d, n_chunks).bytes;
}

extern "C" int attn_jvp_fwd_host(const void* q, const void* k, const void* v, const void* q_t, const void* k_t,
                                 const void* v_t, float* out, float* out_t, float* lse, float* mu, int64_t B,
                                 int64_t H, int64_t N, int64_t d, float scale, int64_t n_chunks, int64_t group_heads,
                                 void* workspace, int64_t workspace_bytes, void* stream) {
  const void* in[6] = {q, k, v, q_t, k_t, v_t};
  for (int i = 0; i < 6; ++i)
    if (!in[i]) return reject(ATTNJVP_EINVAL, "a host input is NULL");
  if (!out || !out_t) return reject(ATTNJVP_EINVAL, "out/out_t is NULL");
  int rc = check_shape(B, H, N, d, n_chunks, group_heads);
  if (rc != ATTNJVP_OK) return rc;
  if (!workspace) return reject(ATTNJVP_EINVAL, "workspace is NULL");
  if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0)
    return reject(ATTNJVP_EINVAL, "workspace must be 256-byte aligned");
  const int64_t g = resolve_group(H, N, group_heads);
  const Slot lay = slot_layout(g, N, d, n_chunks);
  if (workspace_bytes < kSlots * lay.bytes) {
    char msg[200];
    snprintf(msg, sizeof(msg), "workspace holds %lld bytes, this call needs %lld (attn_jvp_fwd_host_workspace_bytes)",
             (long long)workspace_bytes, (long long)(kSlots * lay.bytes));
    return reject(ATTNJVP_EINVAL, msg);
  }
  DeviceStreams ds;
  rc = device_streams(&ds);
  if (rc != ATTNJVP_OK) return rc;
  const cudaStream_t caller = static_cast<cudaStream_t>(stream);
  const cudaStream_t h2d = ds.h2d, d2h = ds.d2h;
  Events ev;
  cudaError_t e = ev.create();
  if (e != cudaSuccess) return cuda_fail("creating events", e);
  if ((e = cudaEventRecord(ev.entry, caller)) != cudaSuccess) return cuda_fail("recording the entry event", e);

  unsigned char* ws = static_cast<unsigned char*>(workspace);
  const int64_t row_elems = N * d;
  const std::vector<Item> items = make_items(B, H, g);
  const int64_t n_items = static_cast<int64_t>(items.size());
  for (int64_t item = 0; item < n_items; ++item) {
    {
      const int64_t gh = items[item].heads;
      const int s = static_cast<int>(item % kSlots);
      const cudaStream_t cs = ds.compute[s];
      void* const cs_arg = static_cast<void*>(cs);
      unsigned char* base = ws + s * lay.bytes;
      const int64_t head0 = items[item].b * H + items[item].h0;  // first (b, h) row block in the host tensors
      const bool reuse = item >= kSlots;  // the slot held item - kSlots before
      // Copy in, once the slot's previous inputs are no longer read.
      if ((e = cudaStreamWaitEvent(h2d, reuse ? ev.computed[s] : ev.entry, 0)) != cudaSuccess)
        return cuda_fail("ordering the copy-in", e);
      for (int i = 0; i < 6; ++i) {
        e = cudaMemcpyAsync(base + lay.in[i], static_cast<const unsigned char*>(in[i]) + head0 * row_elems * 2,
                            gh * row_elems * 2, cudaMemcpyHostToDevice, h2d);
        if (e != cudaSuccess) return cuda_fail("copying an input to the device", e);
      }
      if ((e = cudaEventRecord(ev.in_ready[s], h2d)) != cudaSuccess) return cuda_fail("recording copy-in", e);
      // Compute, once the inputs are in and the slot's previous outputs are out.
      if ((e = cudaStreamWaitEvent(cs, ev.in_ready[s], 0)) != cudaSuccess) return cuda_fail("ordering compute", e);
      if (reuse && (e = cudaStreamWaitEvent(cs, ev.copied[s], 0)) != cudaSuccess)
        return cuda_fail("ordering compute", e);
      const void* dq = base + lay.in[0];
      const void* dk = base + lay.in[1];
      const void* dv = base + lay.in[2];
      const void* dqt = base + lay.in[3];
      const void* dkt = base + lay.in[4];
      const void* dvt = base + lay.in[5];
      float* dout = reinterpret_cast<float*>(base + lay.out);
      float* dout_t = reinterpret_cast<float*>(base + lay.out_t);
      float* dlse = reinterpret_cast<float*>(base + lay.lse);
      float* dmu = reinterpret_cast<float*>(base + lay.mu);
      if (n_chunks == 1) {
        rc = attn_jvp_fwd(dq, dk, dv, dqt, dkt, dvt, dout, dout_t, dlse, dmu, 1, gh, N, d, scale, ATTNJVP_BF16,
                          cs_arg);
        if (rc != ATTNJVP_OK) return rc;
      } else {
        float* o_c = reinterpret_cast<float*>(base + lay.o_c);
        float* ot_c = reinterpret_cast<float*>(base + lay.ot_c);
        float* lse_c = reinterpret_cast<float*>(base + lay.lse_c);
        float* mu_c = reinterpret_cast<float*>(base + lay.mu_c);
        const int64_t rows = gh * N;
        for (int64_t c = 0; c < n_chunks; ++c) {
          const int64_t a = (N * c) / n_chunks, z = (N * (c + 1)) / n_chunks;
          rc = attn_jvp_fwd_chunk(dq, dk, dv, dqt, dkt, dvt, o_c + c * rows * d, ot_c + c * rows * d,
                                  lse_c + c * rows, mu_c + c * rows, 1, gh, N, d, scale, ATTNJVP_BF16, a, z - a,
                                  cs_arg);
          if (rc != ATTNJVP_OK) return rc;
        }
        rc = attn_jvp_merge(o_c, ot_c, lse_c, mu_c, n_chunks, dout, dout_t, dlse, dmu, 1, gh, N, d, cs_arg);
        if (rc != ATTNJVP_OK) return rc;
      }
      if ((e = cudaEventRecord(ev.computed[s], cs)) != cudaSuccess) return cuda_fail("recording compute", e);
      // Copy out.
      if ((e = cudaStreamWaitEvent(d2h, ev.computed[s], 0)) != cudaSuccess) return cuda_fail("ordering copy-out", e);
      struct {
        void* dst;
        const void* src;
        int64_t bytes;
      } outs[4] = {
          {out + head0 * row_elems, dout, gh * row_elems * 4},
          {out_t + head0 * row_elems, dout_t, gh * row_elems * 4},
          {lse ? lse + head0 * N : nullptr, dlse, gh * N * 4},
          {mu ? mu + head0 * N : nullptr, dmu, gh * N * 4},
      };
      for (auto& o : outs) {
        if (!o.dst) continue;
        e = cudaMemcpyAsync(o.dst, o.src, o.bytes, cudaMemcpyDeviceToHost, d2h);
        if (e != cudaSuccess) return cuda_fail("copying an output to the host", e);
      }
      if ((e = cudaEventRecord(ev.copied[s], d2h)) != cudaSuccess) return cuda_fail("recording copy-out", e);
    }
  }
  // The caller's stream completes only after every output has reached the host.
  for (int s = 0; s < kSlots && s < n_items; ++s)
    if ((e = cudaStreamWaitEvent(caller, ev.copied[s], 0)) != cudaSuccess) return cuda_fail("joining copy-out", e);
  attnjvp::set_last_error("");
  return ATTNJVP_OK;
}
