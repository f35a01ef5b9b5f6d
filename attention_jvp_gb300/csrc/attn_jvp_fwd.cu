// Fused attention forward + forward-mode JVP for sm_103a (tcgen05 / TMEM / TMA).
//
// What it computes (page "带分数正则的一致性蒸馏", gitcode.csdn.net, section
// 注意力 (attention), the streaming JVP paragraph, and section 前向 (forward)):
// per query row, stream the keys in tiles while carrying a running max m, the
// exponential sum l, r = rowsum(P~ (.) St) and two accumulators
//     O~ = sum P~ V              T~ = sum P~ Vt + sum (P~ (.) St) V
// (the page's A + B in one accumulator, since only their sum is used), where
// P~ = exp(S - m) is the unnormalised softmax and every accumulator is
// rescaled by exp(m_old - m_new) when the running max grows.  At the end
//     O = O~ / l,  mu = r / l,  Ot = T~ / l - mu O,  LSE = m + ln l.
//
// GB300 mapping (one CTA = 128 query rows of one (batch, head)):
//   warp 0      TMA producer for Q, Qt (once) and the K/Kt ring
//   warp 1      TMEM allocator and the tcgen05.mma issuer of the value MMAs
//   warp 2      TMA producer for the V/Vt ring
//   warp 3      tcgen05.mma issuer of the score-tangent MMAs (St)
//   warps 4-7   softmax + JVP weights + lazy rescale + epilogue; thread t of
//               warp 4+w owns query row 32w+t, which is TMEM lane 32w+t, so
//               every row reduction is thread-local (no shuffles).
//   warp 8      tcgen05.mma issuer of the score MMAs (S)
// Three issuing threads keep the tensor pipe fed while any one of them waits
// on a barrier, and the short S chain (which gates the softmax of the next
// tile) never queues behind the long St chain of the same thread.
// Per 64-key tile j (tensor-core work, fp32 accumulation in TMEM):
//   S_b  = Q K_j^T                         (d-deep, N = 64)
//   St_c = [Qt Q] [K_j Kt_j]^T             (one 2d-deep chain, N = 64)
//   softmax warps: P~ = 2^(S*s*log2e - m), H~ = P~ (.) St * s, row sums in fp32,
//                  P~ and H~ rounded to bf16 and written back into St_c's columns
//   O += P~ V_j,  T += P~ Vt_j,  T += H~ V_j   (A operand read from TMEM)
// S buffers and St buffers are two separate TMEM rings.  An St buffer stays
// busy until the value MMAs have read the P~/H~ written into it, an S buffer
// only until the softmax has loaded it.  The long 2d-deep St chain therefore
// gets the deeper ring and is issued first, as soon as the value MMAs of tile
// j - NSt are done; the short S chain waits only for the softmax to have
// loaded tile j - NS.  Only MMAs of identical shape chain into one
// accumulator, the ordering tcgen05 guarantees without extra waits.
//
// Lazy rescale: a row keeps its reference max until a tile's max exceeds it by
// more than 8 (log2 units); only then are O, T, l, r rescaled.  All four share
// the same reference, so the final normalisation is exact.
//
// Head dims (the page's set, 16-256, for Q/K and for V independently): the
// kernel is a template over both, each rounded up to 64, 128 or 256.  The Q/K
// dim sets the score MMAs' depth and, through the resident Q and Qt, how many
// key tiles the rings hold.  The V dim sets the value MMAs and the TMEM layout.
// At a V dim of 256, O and T of 128 rows would fill TMEM, so two neighbouring
// CTAs share each query tile and each accumulates 128 of the value columns.
//
// Waves: each CTA holds all of an SM's TMEM, so the grid runs in waves of the
// SM count.  A last wave at most half full would leave most SMs idle for a
// whole CTA's time, so its units are cut into pieces over the keys, written as
// partials and merged by merge_pieces_kernel (see FwdGeom).
#include <cuda_runtime.h>
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace attnjvp {
namespace {

using namespace ptx;

// D: Q/K head dim rounded up to a multiple of 64 (16 and 32 run as 64, their
// missing columns zero-filled by TMA); DVF: the same for V/O.
template <int D, int DVF>
struct FwdCfg {
  static constexpr int kBM = 128;                  // query rows per CTA (= TMEM lanes)
  static constexpr int kBN = 64;                   // keys per tile
  static constexpr int kDC = D / 64;               // 64-element (128-byte) d-chunks of Q and K
  // Value columns per CTA.  O and T take 2 kDV TMEM columns; at a value head dim
  // of 256 the two whole would fill TMEM, so two CTAs share a query tile, each
  // accumulating half of the value columns (and each computing the full scores).
  static constexpr int kDV = DVF > 128 ? 128 : DVF;
  static constexpr int kVC = kDV / 64;             // 64-element chunks of a value tile
  static constexpr int kVSplit = DVF / kDV;        // CTAs per query tile
  static constexpr bool kSmallV = DVF == 64;       // value heads of 16, 32 or 64 columns
  // TMEM ring depths.  At 64 value columns the softmax chain bounds a tile, so the
  // S ring (which only waits for the softmax to load a tile) stays at one buffer and
  // the St ring, whose buffers wait for the value MMAs, takes the rest: measured
  // 1 % faster than three and three, and 4 % faster than two and four.
  static constexpr int kNS = 1;                     // S TMEM buffers
  static constexpr int kNSt = (kDV == 64) ? 5 : 3;  // St (then P~/H~) TMEM buffers
  static constexpr int kChunkQ = kBM * 128;        // one d-chunk of a Q tile (bytes)
  static constexpr int kChunkK = kBN * 128;        // one d-chunk of a key tile (bytes)
  static constexpr int kQBytes = kDC * kChunkQ;    // Q (or Qt) tile
  static constexpr int kKStage = 2 * kDC * kChunkK;  // K chunks, then Kt chunks
  static constexpr int kVStage = 2 * kVC * kChunkK;  // V chunks, then Vt chunks (this CTA's columns)
  // K/Kt and V/Vt ring stages: as many as shared memory holds, up to three each
  // (Q and Qt stay resident: 128 KB at d = 256, which leaves room for one).
  static constexpr int kRoom = 227 * 1024 - 1536 - 2 * kQBytes;
  static constexpr int kKS = kRoom >= 3 * (kKStage + kVStage) ? 3 : (kRoom >= 2 * (kKStage + kVStage) ? 2 : 1);
  static constexpr int kVS = kKS;
  // K/Kt ring units.  Normally a unit is a whole key tile and the ring holds kKS
  // of them.  With room for only one tile (Q/K head dim 256) the tile is split
  // into two units of half its d-chunks, so that the next tile's first half
  // loads while this tile's second half is in the score MMAs.
  static constexpr int kUPT = (kKS == 1 && kDC % 2 == 0) ? 2 : 1;  // units per key tile
  static constexpr int kUC = kDC / kUPT;                           // d-chunks of K (and of Kt) per unit
  static constexpr int kKU = kKS * kUPT;                           // units in the ring
  static constexpr int kKUnit = 2 * kUC * kChunkK;                 // K chunks, then Kt chunks
  static constexpr int kOffQ = 0;
  static constexpr int kOffQt = kQBytes;
  static constexpr int kOffK = 2 * kQBytes;
  static constexpr int kOffV = kOffK + kKU * kKUnit;
  static_assert(kKU * kKUnit >= 4 * 8192, "the key ring also holds the four 8 KB epilogue stages");
  static constexpr int kOffBar = kOffV + kVS * kVStage;
  static constexpr int kSmemBytes = kOffBar + 512 + 1024;  // + barriers + alignment slack
  // TMEM columns (fp32 each): O [0,DV), T [DV,2DV), S buffer b [2DV+64b, +64),
  // St buffer c [2DV+64NS+64c, +64)
  static constexpr uint32_t kColO = 0;
  static constexpr uint32_t kColT = kDV;
  static constexpr uint32_t kColS = 2 * kDV;
  static constexpr uint32_t kColSt = 2 * kDV + 64 * kNS;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kColSt + 64 * kNSt <= kTmemCols, "TMEM budget");
  static_assert(kNS <= 5 && kNSt <= 5 && kKU <= 3 && kVS <= 3, "barrier arrays");
  static_assert(kKU * kKUnit == kKS * kKStage, "K ring size");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

constexpr int kThreads = 288;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale once P~ could exceed 2^8

struct FwdMaps {
  CUtensorMap q, qt, k, kt, v, vt;
};

// The tensor maps are 4-D over (head-dimension column, sequence row, head,
// batch), each dimension with the tensor's own stride, so any strided layout
// with a unit head-dimension stride ([B, H, S, D], [B, S, H, D], slices of a
// packed QKV tensor, ...) is read in place.
struct FwdGeom {
  int H, Nq, n_qtiles, kv_start, kv_len;
  int d_v;                  // real value head dimension: the output columns written
  float scale;
  int64_t o_stride[3];      // output element strides: batch, sequence, head
  // Balance of a short last wave: the grid's units (query tile, value half) from
  // n_main on are each cut into ``split`` pieces over consecutive key ranges, one
  // CTA per piece; piece c takes key tiles [piece_t[c], piece_t[c + 1]) of the
  // launch's range.  A piece writes its normalised O, Ot (kDV columns per row,
  // 128 rows) and its LSE and mu to the ``part_*`` arrays, slot
  // (unit - n_main) * split + c, and merge_pieces_kernel combines them.
  // split == 1: no pieces, n_main is the grid.
  static constexpr int kMaxSplit = 16;
  int n_main, split;
  int piece_t[kMaxSplit + 1];
  float *part_o, *part_ot, *part_lse, *part_mu;
};

struct Barriers {
  uint64_t q_full;
  uint64_t k_full[3], k_empty[3];
  uint64_t v_full[3], v_empty[3];
  uint64_t s_full[5], st_full[5], s_free[5], p_full[5], pv_done[5];
  uint64_t drain, drain_s, drain_st;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Barriers) <= 512, "barrier block (512 bytes reserved in FwdCfg::kSmemBytes)");

// Online-softmax state of one query row (log2 units of the scaled scores).
struct RowState {
  float m = -INFINITY;  // reference max
  float l = 0.f;        // sum of P~
  float r = 0.f;        // sum of P~ (.) St s
};

// Softmax + JVP weights of one 64-key tile for the calling thread's query row.
// ``cS`` / ``cSt`` are the row's TMEM addresses of the tile's raw S and raw St
// (64 columns each).  ``on_loaded()`` runs once both are in registers (the S
// buffer is then free for a later tile's score MMAs).  On return P~ and H~ (bf16
// pairs) sit in columns 0-31 and 32-63 of the St buffer, their stores have
// completed and the tcgen05 fence that
// precedes the hand-off to the MMA thread has been executed.  When the row max
// grows by more than the threshold the accumulators O and T (columns 0-2D) are
// rescaled after ``wait_prev_pv()`` confirms the previous tile's value MMAs are
// done.  Returns false (warp-uniformly) when a wait gave up.
template <class C, class OnLoaded, class WaitPrevPv>
__device__ __forceinline__ bool softmax_tile(uint32_t lane_addr, uint32_t cS, uint32_t cSt, int valid, bool first,
                                             float c2,
                                             float scale, RowState& st, OnLoaded on_loaded,
                                             WaitPrevPv wait_prev_pv) {
  // The row's 64 raw scores and 64 raw score tangents; from then on the S
  // buffer may be overwritten (``on_loaded``).
  uint32_t raw[128];
  tmem_ld64x2_wait(cS, cSt, raw);
  tc_fence_before_sync();
  on_loaded();
  if (valid < 64) {
    // Tail tile: keys past the range get score -inf (weight 0) and tangent 0.
#pragma unroll
    for (int i = 0; i < 64; ++i)
      if (i >= valid) {
        raw[i] = __float_as_uint(-INFINITY);
        raw[64 + i] = 0u;
      }
  }
  // Row max of the raw scores (the scale is positive, so it keeps the order);
  // eight independent chains of three-input maxima keep the dependency depth short.
  auto f = [&](int i) { return __uint_as_float(raw[i]); };
  float mx8[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) mx8[k] = fmax3(f(k), f(8 + k), f(16 + k));
#pragma unroll
  for (int i = 24; i < 56; i += 16)
#pragma unroll
    for (int k = 0; k < 8; ++k) mx8[k] = fmax3(mx8[k], f(i + k), f(i + 8 + k));
#pragma unroll
  for (int k = 0; k < 8; ++k) mx8[k] = fmaxf(mx8[k], f(56 + k));
  const float mx = fmaxf(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(fmax3(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7])) * c2;
  float alpha = 1.f;
  bool rescale = false;
  if (first) {
    st.m = mx;
  } else if (mx > st.m + kRescaleThreshold) {
    alpha = ex2_approx(st.m - mx);
    st.m = mx;
    rescale = true;
  }
  // P~ = 2^(S s log2e - m): one paired FFMA per two scores, one MUFU ex2 per score.
  // Row sums run in four paired chains (eight fp32 lanes).
  const uint64_t c2x2 = f2_pack(c2, c2);
  const uint64_t negm2 = f2_pack(-st.m, -st.m);
  float p[64];
  uint64_t l4[4];
#pragma unroll
  for (int i = 0; i < 64; i += 2) {
    float x0, x1;
    f2_unpack(f2_fma(f2_pack(f(i), f(i + 1)), c2x2, negm2), x0, x1);
    p[i] = ex2_approx(x0);
    p[i + 1] = ex2_approx(x1);
    const uint64_t pp = f2_pack(p[i], p[i + 1]);
    const int k = (i >> 1) & 3;
    l4[k] = (i < 8) ? pp : f2_add(l4[k], pp);
  }
  float la, lb;
  f2_unpack(f2_add(f2_add(l4[0], l4[1]), f2_add(l4[2], l4[3])), la, lb);
  st.l = st.l * alpha + (la + lb);
  uint32_t pk[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) pk[i] = pack_bf16x2(p[2 * i], p[2 * i + 1]);
  // H~ = P~ (.) St s; its row sum is taken in fp32 before rounding to bf16.
  const uint64_t s2 = f2_pack(scale, scale);
  uint32_t hk[32];
  uint64_t r4[4];
#pragma unroll
  for (int i = 0; i < 64; i += 2) {
    const uint64_t hh = f2_mul(f2_pack(p[i], p[i + 1]), f2_mul(f2_pack(f(64 + i), f(65 + i)), s2));
    float h0, h1;
    f2_unpack(hh, h0, h1);
    hk[i >> 1] = pack_bf16x2(h0, h1);
    const int k = (i >> 1) & 3;
    r4[k] = (i < 8) ? hh : f2_add(r4[k], hh);
  }
  float ra, rb;
  f2_unpack(f2_add(f2_add(r4[0], r4[1]), f2_add(r4[2], r4[3])), ra, rb);
  st.r = st.r * alpha + (ra + rb);
  if (__any_sync(0xffffffffu, rescale)) {
    // O and T may only be touched once the previous tile's value MMAs are done.
    const bool ok = __all_sync(0xffffffffu, wait_prev_pv());
    if (!ok) return false;
    tc_fence_after_sync();
#pragma unroll 1
    for (int c0 = 0; c0 < 2 * C::kDV; c0 += 32) {
      uint32_t acc[32];
      tmem_ld32_wait(lane_addr + c0, acc);
#pragma unroll
      for (int i = 0; i < 32; ++i) acc[i] = __float_as_uint(__uint_as_float(acc[i]) * alpha);
      tmem_st32(lane_addr + c0, acc);
    }
  }
  tmem_st32(cSt, pk);
  tmem_st32(cSt + 32, hk);
  tmem_wait_st();
  tc_fence_before_sync();
  return true;
}

// Epilogue of one softmax warp's 32 rows: O = O~/l, mu = r/l, Ot = T~/l - mu O
// and LSE = (m + log2 l) ln 2, read from TMEM (O~ in columns 0-DV, T~ in DV-2DV).
// Each thread forms its own row 32 columns at a time, but stores from one thread
// per row would touch 32 rows (32 cache lines) per warp instruction, and the
// store path, not the bandwidth, bounds that.  So the warp passes each 32-column
// chunk through ``stage`` (its own 8 KB of shared memory: O, then Ot, 32 x 32
// floats each, 16-byte unit u of row r at unit u ^ (r mod 8), which spreads both
// the row-wise writes and the read-back over all banks) and writes it back four
// rows per instruction, eight lanes per 128-byte row segment.
// ``obase0``: element offset of the warp's first row in out / out_t (this CTA's
// value columns); ``ostride``: elements between rows; ``valid_rows``: rows of the
// warp that exist (the last query tile may be partial).  The CTA's value columns
// (the first d of them for d < 64) are written; LSE and mu where non-null.
template <class C>
__device__ __forceinline__ void write_rows(uint32_t lane_addr, const RowState& st, int64_t ridx, int64_t obase0,
                                           int64_t ostride, int valid_rows, int d, float* stage,
                                           float* __restrict__ out, float* __restrict__ out_t,
                                           float* __restrict__ lse_out, float* __restrict__ mu_out) {
  const int lane = threadIdx.x & 31;
  const float inv_l = 1.f / st.l;
  const float mu = st.r * inv_l;
  // The CTA's kDV value columns, except for the 16/32-wide value heads run as 64.
  constexpr int kDV = C::kDV;
  const int ncols = C::kSmallV ? d : kDV;
  float4* so = reinterpret_cast<float4*>(stage);        // [32 rows][8 units]
  float4* stt = reinterpret_cast<float4*>(stage + 1024);
  const int ru = lane & 7;   // read-back: unit of the row segment
  const int rr = lane >> 3;  // read-back: first row (then every fourth)
#pragma unroll 1
  for (int c0 = 0; c0 < ncols; c0 += 32) {
    uint32_t ov[32], tv[32];
    tmem_ld32_wait(lane_addr + c0, ov);
    tmem_ld32_wait(lane_addr + kDV + c0, tv);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float4 o, t;
      o.x = __uint_as_float(ov[4 * i + 0]) * inv_l;
      o.y = __uint_as_float(ov[4 * i + 1]) * inv_l;
      o.z = __uint_as_float(ov[4 * i + 2]) * inv_l;
      o.w = __uint_as_float(ov[4 * i + 3]) * inv_l;
      t.x = __uint_as_float(tv[4 * i + 0]) * inv_l - mu * o.x;
      t.y = __uint_as_float(tv[4 * i + 1]) * inv_l - mu * o.y;
      t.z = __uint_as_float(tv[4 * i + 2]) * inv_l - mu * o.z;
      t.w = __uint_as_float(tv[4 * i + 3]) * inv_l - mu * o.w;
      so[lane * 8 + (i ^ (lane & 7))] = o;
      stt[lane * 8 + (i ^ (lane & 7))] = t;
    }
    __syncwarp();
    const bool col_ok = !C::kSmallV || c0 + 4 * ru < ncols;
#pragma unroll 1
    for (int i = 0; i < 8; ++i) {
      const int r = rr + 4 * i;
      if (col_ok && r < valid_rows) {
        const int64_t off = obase0 + static_cast<int64_t>(r) * ostride + c0 + 4 * ru;
        // streaming stores: the outputs are not read again, so they should not
        // push the key and value tiles out of L2
        __stcs(reinterpret_cast<float4*>(out + off), so[r * 8 + (ru ^ (r & 7))]);
        __stcs(reinterpret_cast<float4*>(out_t + off), stt[r * 8 + (ru ^ (r & 7))]);
      }
    }
    __syncwarp();  // the next chunk overwrites the stage
  }
  if (lane < valid_rows) {
    if (lse_out) lse_out[ridx] = (st.m + __log2f(st.l)) * kLn2;
    if (mu_out) mu_out[ridx] = mu;
  }
}

template <int D, int DVF>
__global__ void __launch_bounds__(kThreads, 1)
    attn_jvp_fwd_kernel(const __grid_constant__ FwdMaps maps, const __grid_constant__ FwdGeom geom,
                        float* __restrict__ out, float* __restrict__ out_t, float* __restrict__ lse_out,
                        float* __restrict__ mu_out, int* status) {
  using C = FwdCfg<D, DVF>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Barriers* bars = reinterpret_cast<Barriers*>(smem + C::kOffBar);
  volatile int* abort_flag = &bars->abort_flag;

  // Another CTA already hit a wait timeout: the whole CTA does nothing (read once, decided uniformly).
  if (threadIdx.x == 0) bars->abort_flag = (*reinterpret_cast<volatile int*>(status) & kStatusTimeout) ? 1 : 0;
  __syncthreads();
  if (bars->abort_flag) return;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_qtiles = geom.n_qtiles;
  int kv_start = geom.kv_start, kv_len = geom.kv_len;
  const float scale = geom.scale;
  // A CTA past n_main is one piece of a unit of the last wave: that unit's key
  // tiles [t0, t1) of the launch's range.
  unsigned unit = blockIdx.x;
  int piece = -1;  // this CTA's partial-output slot, or -1 (outputs in place)
  if (unit >= static_cast<unsigned>(geom.n_main)) {
    piece = static_cast<int>(unit - geom.n_main);
    const unsigned u = static_cast<unsigned>(piece) / static_cast<unsigned>(geom.split);
    const int c = piece - static_cast<int>(u) * geom.split;
    unit = geom.n_main + u;
    const int k0 = geom.piece_t[c] * C::kBN;
    kv_len = min(geom.piece_t[c + 1] * C::kBN, kv_len) - k0;
    kv_start += k0;
  }
  // Both value halves of a query tile (d = 256) are neighbours in the grid, so
  // they stream the same key tiles through L2 at about the same time.
  const int vh = unit % C::kVSplit;  // which kDV value columns this CTA accumulates
  const unsigned qb = unit / C::kVSplit;  // unsigned: the divisions below stay unsigned
  const int bh = qb / n_qtiles;
  const int hh = bh % geom.H, bb = bh / geom.H;
  const int q0 = (qb % n_qtiles) * C::kBM;
  const int n_tiles = (kv_len + C::kBN - 1) / C::kBN;


  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < 5; ++s) {
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->st_full[s], 1);
      mbar_init(&bars->p_full[s], 4);  // one arrival per softmax warp
      mbar_init(&bars->pv_done[s], 1);
      mbar_init(&bars->s_free[s], 4);
    }
    for (int s = 0; s < 3; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 2);  // one commit from each score issuer
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    mbar_init(&bars->drain, 1);
    mbar_init(&bars->drain_s, 1);
    mbar_init(&bars->drain_st, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    // ---------------- TMA producer: Q, Qt and the K/Kt ring ----------------
    if (lane == 0) {
      prefetch_tensormap(&maps.q);
      prefetch_tensormap(&maps.qt);
      prefetch_tensormap(&maps.k);
      prefetch_tensormap(&maps.kt);
      mbar_arrive_expect_tx(&bars->q_full, 2 * C::kQBytes);
      for (int c = 0; c < C::kDC; ++c) {
        tma_load_4d(smem + C::kOffQ + c * C::kChunkQ, &maps.q, &bars->q_full, c * 64, q0, hh, bb);
        tma_load_4d(smem + C::kOffQt + c * C::kChunkQ, &maps.qt, &bars->q_full, c * 64, q0, hh, bb);
      }
      int issued = 0;  // ring units
      bool ok = true;
      for (int n = 0; n < n_tiles * C::kUPT && ok; ++n) {
        const int t = n / C::kUPT, u = n % C::kUPT;  // key tile, unit within it
        const int s = n % C::kKU;
        ok = mbar_wait(&bars->k_empty[s], ((n / C::kKU) & 1) ^ 1, abort_flag, status, kStatusTimeout);
        if (!ok) break;
        uint8_t* st = smem + C::kOffK + s * C::kKUnit;
        const int key0 = kv_start + t * C::kBN;
        mbar_arrive_expect_tx(&bars->k_full[s], C::kKUnit);
        for (int c = 0; c < C::kUC; ++c) {
          const int col = (u * C::kUC + c) * 64;
          tma_load_4d(st + c * C::kChunkK, &maps.k, &bars->k_full[s], col, key0, hh, bb);
          tma_load_4d(st + (C::kUC + c) * C::kChunkK, &maps.kt, &bars->k_full[s], col, key0, hh, bb);
        }
        issued = n + 1;
      }
      // Let copies still in flight land before the CTA's shared memory goes away.  This
      // runs on the normal path too: another role may give up right after the last copy
      // was issued, and then nothing else waits for it.
      volatile int no_abort = 0;
      mbar_wait(&bars->q_full, 0, &no_abort, nullptr, 0);
      for (int n = issued - C::kKU; n < issued; ++n)
        if (n >= 0) mbar_wait(&bars->k_full[n % C::kKU], (n / C::kKU) & 1, &no_abort, nullptr, 0);
    }
  } else if (warp == 2) {
    // ---------------- TMA producer: the V/Vt ring ----------------
    if (lane == 0) {
      prefetch_tensormap(&maps.v);
      prefetch_tensormap(&maps.vt);
      int issued = 0;
      bool ok = true;
      for (int t = 0; t < n_tiles && ok; ++t) {
        const int s = t % C::kVS;
        ok = mbar_wait(&bars->v_empty[s], ((t / C::kVS) & 1) ^ 1, abort_flag, status, kStatusTimeout);
        if (!ok) break;
        uint8_t* st = smem + C::kOffV + s * C::kVStage;
        const int key0 = kv_start + t * C::kBN;
        mbar_arrive_expect_tx(&bars->v_full[s], C::kVStage);
        for (int c = 0; c < C::kVC; ++c) {
          const int col = vh * C::kDV + c * 64;
          tma_load_4d(st + c * C::kChunkK, &maps.v, &bars->v_full[s], col, key0, hh, bb);
          tma_load_4d(st + (C::kVC + c) * C::kChunkK, &maps.vt, &bars->v_full[s], col, key0, hh, bb);
        }
        issued = t + 1;
      }
      volatile int no_abort = 0;  // drain, as the K/Kt producer does
      for (int t = issued - C::kVS; t < issued; ++t)
        if (t >= 0) mbar_wait(&bars->v_full[t % C::kVS], (t / C::kVS) & 1, &no_abort, nullptr, 0);
    }
  } else if (warp == 1 || warp == 3 || warp == 8) {
    // ---------------- tcgen05.mma issuers: warp 8 S, warp 3 St, warp 1 the value MMAs ----------------
    // Independent issuing threads; they meet only through the mbarriers below.
    if (lane == 0) {
      constexpr uint32_t kIdS = make_idesc_bf16_f32(128, C::kBN, false, false);  // Q K^T, both K-major
      constexpr uint32_t kIdPV = make_idesc_bf16_f32(128, C::kDV, false, true);  // P~ V, V is N-major
      // Descriptors are built once; an operand step adds its byte offset / 16 to the
      // start-address field (every offset here stays inside one CTA's shared memory).
      const uint64_t dQ = make_smem_desc_sw128(smem_u32(smem + C::kOffQ), 16, 1024);
      const uint64_t dQt = make_smem_desc_sw128(smem_u32(smem + C::kOffQt), 16, 1024);
      const uint64_t dK0 = make_smem_desc_sw128(smem_u32(smem + C::kOffK), 16, 1024);
      const uint64_t dV0 = make_smem_desc_sw128(smem_u32(smem + C::kOffV), C::kChunkK, 1024);
      auto off = [](uint64_t desc, uint32_t bytes) { return desc + static_cast<uint64_t>(bytes >> 4); };
      volatile int no_abort = 0;
      if (warp == 8) {
        bool ok = mbar_wait(&bars->q_full, 0, abort_flag, status, kStatusTimeout);
        for (int t = 0; ok && t < n_tiles; ++t) {
          const int b = t % C::kNS;
          const uint32_t dS = tmem + C::kColS + 64u * b;
#pragma unroll 1
          for (int u = 0; u < C::kUPT; ++u) {
            const int n = t * C::kUPT + u;
            const int s = n % C::kKU;
            ok = mbar_wait(&bars->k_full[s], (n / C::kKU) & 1, abort_flag, status, kStatusTimeout);
            // The S buffer is free once the softmax has loaded tile t - NS.
            if (ok && u == 0 && t >= C::kNS)
              ok = mbar_wait(&bars->s_free[b], ((t - C::kNS) / C::kNS) & 1, abort_flag, status, kStatusTimeout);
            if (!ok) break;
            tc_fence_after_sync();
            const uint64_t dK = off(dK0, s * C::kKUnit);
            // S_t = Q K_t^T over this unit's d-chunks
#pragma unroll
            for (int c = 0; c < C::kUC; ++c)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_ss(dS, off(dQ, (u * C::kUC + c) * C::kChunkQ + kk * 32), off(dK, c * C::kChunkK + kk * 32),
                       kIdS, (u | c | kk) != 0);
            mma_commit(&bars->k_empty[s]);
          }
          if (!ok) break;
          mma_commit(&bars->s_full[b]);
        }
        // Nothing may still be reading shared memory or TMEM when the CTA tears down.
        mma_commit(&bars->drain_s);
        mbar_wait(&bars->drain_s, 0, &no_abort, nullptr, 0);
      } else if (warp == 3) {
        bool ok = mbar_wait(&bars->q_full, 0, abort_flag, status, kStatusTimeout);
        for (int t = 0; ok && t < n_tiles; ++t) {
          const int bt = t % C::kNSt;
          const uint32_t dSt = tmem + C::kColSt + 64u * bt;
#pragma unroll 1
          for (int u = 0; u < C::kUPT; ++u) {
            const int n = t * C::kUPT + u;
            const int s = n % C::kKU;
            ok = mbar_wait(&bars->k_full[s], (n / C::kKU) & 1, abort_flag, status, kStatusTimeout);
            // The St buffer holds P~/H~ of tile t - NSt until that tile's value MMAs are done.
            if (ok && u == 0 && t >= C::kNSt)
              ok = mbar_wait(&bars->pv_done[bt], ((t - C::kNSt) / C::kNSt) & 1, abort_flag, status,
                             kStatusTimeout);
            if (!ok) break;
            tc_fence_after_sync();
            const uint64_t dK = off(dK0, s * C::kKUnit);
            // St_t = [Qt Q] [K_t Kt_t]^T : one accumulator, 2d deep (this unit's d-chunks)
#pragma unroll
            for (int c = 0; c < C::kUC; ++c)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_ss(dSt, off(dQt, (u * C::kUC + c) * C::kChunkQ + kk * 32), off(dK, c * C::kChunkK + kk * 32),
                       kIdS, (u | c | kk) != 0);
#pragma unroll
            for (int c = 0; c < C::kUC; ++c)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_ss(dSt, off(dQ, (u * C::kUC + c) * C::kChunkQ + kk * 32),
                       off(dK, (C::kUC + c) * C::kChunkK + kk * 32), kIdS, 1);
            mma_commit(&bars->k_empty[s]);
          }
          if (!ok) break;
          mma_commit(&bars->st_full[bt]);
        }
        mma_commit(&bars->drain_st);
        mbar_wait(&bars->drain_st, 0, &no_abort, nullptr, 0);
      } else {
        bool ok = true;
        for (int j = 0; ok && j < n_tiles; ++j) {
          const int bt = j % C::kNSt;
          const int s = j % C::kVS;
          ok = mbar_wait(&bars->p_full[bt], (j / C::kNSt) & 1, abort_flag, status, kStatusTimeout) &&
               mbar_wait(&bars->v_full[s], (j / C::kVS) & 1, abort_flag, status, kStatusTimeout);
          if (!ok) break;
          tc_fence_after_sync();
          const uint64_t dV = off(dV0, s * C::kVStage);
          const uint32_t aP = tmem + C::kColSt + 64u * bt;  // P~ packed bf16: 32 columns
          const uint32_t aH = aP + 32u;                       // H~ packed bf16: 32 columns
#pragma unroll
          for (int kk = 0; kk < C::kBN / 16; ++kk) {
            const uint64_t bV = off(dV, kk * 2048);
            const uint64_t bVt = off(dV, C::kVC * C::kChunkK + kk * 2048);
            const uint32_t acc = (j > 0 || kk > 0) ? 1u : 0u;
            mma_ts(tmem + C::kColO, aP + kk * 8, bV, kIdPV, acc);   // O += P~ V
            mma_ts(tmem + C::kColT, aP + kk * 8, bVt, kIdPV, acc);  // T += P~ Vt
            mma_ts(tmem + C::kColT, aH + kk * 8, bV, kIdPV, 1u);    // T += H~ V
          }
          mma_commit(&bars->v_empty[s]);
          mma_commit(&bars->pv_done[bt]);
        }
        mma_commit(&bars->drain);
        mbar_wait(&bars->drain, 0, &no_abort, nullptr, 0);
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ---------------- softmax / JVP / epilogue: one query row per thread ----------------
    const int quarter = warp - 4;
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float c2 = scale * kLog2e;
    RowState st;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      const int b = j % C::kNS;
      const int bt = j % C::kNSt;
      ok = mbar_wait(&bars->s_full[b], (j / C::kNS) & 1, abort_flag, status, kStatusTimeout) &&
           mbar_wait(&bars->st_full[bt], (j / C::kNSt) & 1, abort_flag, status, kStatusTimeout);
      ok = __all_sync(0xffffffffu, ok);  // keep the warp converged for the .sync.aligned TMEM ops
      if (!ok) break;
      tc_fence_after_sync();
      const uint32_t cS = lane_addr + C::kColS + 64u * b;
      const uint32_t cSt = lane_addr + C::kColSt + 64u * bt;
      const int valid = min(C::kBN, kv_len - j * C::kBN);
      // Hand-offs arrive once per warp: every lane has fenced its own TMEM
      // accesses, __syncwarp orders them before lane 0's arrival.
      ok = softmax_tile<C>(
          lane_addr, cS, cSt, valid, j == 0, c2, scale, st,
          [&]() {
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->s_free[b]);
          },
          [&]() {
            return mbar_wait(&bars->pv_done[(j - 1) % C::kNSt], ((j - 1) / C::kNSt) & 1, abort_flag, status,
                             kStatusTimeout);
          });
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full[bt]);
    }
    // ---------------- epilogue ----------------
    if (ok) ok = mbar_wait(&bars->pv_done[(n_tiles - 1) % C::kNSt], ((n_tiles - 1) / C::kNSt) & 1, abort_flag, status,
                           kStatusTimeout);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      tc_fence_after_sync();
      // Every MMA and copy of the CTA is done: the key ring's shared memory is free
      // and holds each softmax warp's 8 KB epilogue stage.
      fence_proxy_async_smem();
      const int qrow = q0 + row;
      const int wrow0 = q0 + quarter * 32;  // the warp's first query row
      float* stage = reinterpret_cast<float*>(smem + C::kOffK + quarter * 8192);
      // In place; or a piece's partial slot of 128 rows of kDV columns.  Every value
      // half computes the same LSE and mu; in place, the first one writes them.
      const bool part = piece >= 0;
      const int64_t slot = static_cast<int64_t>(piece) * C::kBM;
      const int64_t obase0 = part ? (slot + quarter * 32) * C::kDV
                                  : static_cast<int64_t>(bb) * geom.o_stride[0] +
                                        static_cast<int64_t>(wrow0) * geom.o_stride[1] +
                                        static_cast<int64_t>(hh) * geom.o_stride[2] + vh * C::kDV;
      write_rows<C>(lane_addr, st, part ? slot + row : static_cast<int64_t>(bh) * geom.Nq + qrow, obase0,
                    part ? C::kDV : geom.o_stride[1], min(32, geom.Nq - wrow0), geom.d_v, stage,
                    part ? geom.part_o : out, part ? geom.part_ot : out_t,
                    part ? geom.part_lse : (vh == 0 ? lse_out : nullptr),
                    part ? geom.part_mu : (vh == 0 ? mu_out : nullptr));
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// 4-D map over (column, sequence row, head, batch) with the tensor's strides
// (elements; the column stride is 1).  A dimension of extent 1 is never
// stepped, so its stride is replaced by the tensor's span to keep it a valid
// TMA stride whatever the caller passed.  Columns past ``d`` (d < 64) and rows
// past ``rows`` read as zero.
cudaError_t make_map(CUtensorMap* map, const void* ptr, int64_t d, int64_t rows, int64_t H, int64_t B,
                     const int64_t stride[3], int box_rows) {
  TensorMapEncodeFn enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  const int64_t extent[3] = {rows, H, B};
  int64_t st[3] = {stride[1], stride[2], stride[0]};  // sequence, head, batch
  int64_t span = d;
  for (int i = 0; i < 3; ++i)
    if (extent[i] > 1 && extent[i] * st[i] > span) span = extent[i] * st[i];
  for (int i = 0; i < 3; ++i)
    if (extent[i] == 1) st[i] = (span + 7) / 8 * 8;
  cuuint64_t gdim[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t gstr[3] = {static_cast<cuuint64_t>(st[0]) * 2, static_cast<cuuint64_t>(st[1]) * 2,
                        static_cast<cuuint64_t>(st[2]) * 2};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(box_rows), 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), gdim, gstr, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Combines the pieces of each split unit (see FwdGeom) into its outputs, by the
// exact merge of key ranges: LSE = ln sum_c e^{LSE_c}, w_c = e^{LSE_c - LSE},
// O = sum_c w_c O_c, mu = sum_c w_c mu_c, Ot = sum_c w_c (Ot_c + mu_c O_c) - mu O.
// One thread per 4 columns of one row of one unit.
template <class C>
__global__ void __launch_bounds__(256) merge_pieces_kernel(const __grid_constant__ FwdGeom geom, int n_units,
                                                           int ncols, float* __restrict__ out,
                                                           float* __restrict__ out_t, float* __restrict__ lse,
                                                           float* __restrict__ mu) {
  const int tpr = ncols >> 2;
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t rowid = gtid / tpr;  // unit * 128 + row
  if (rowid >= static_cast<int64_t>(n_units) * C::kBM) return;
  const int col = static_cast<int>(gtid % tpr) * 4;
  const int u = static_cast<int>(rowid / C::kBM), r = static_cast<int>(rowid % C::kBM);
  const unsigned unit = geom.n_main + u;
  const int vh = unit % C::kVSplit;
  const unsigned qb = unit / C::kVSplit;
  const int bh = qb / geom.n_qtiles;
  const int hh = bh % geom.H, bb = bh / geom.H;
  const int qrow = (qb % geom.n_qtiles) * C::kBM + r;
  if (qrow >= geom.Nq) return;
  const int split = geom.split;
  const int64_t s0 = static_cast<int64_t>(u) * split * C::kBM + r;  // slot row of piece 0
  float mx = -INFINITY;
  for (int c = 0; c < split; ++c) mx = fmaxf(mx, geom.part_lse[s0 + c * C::kBM]);
  float sum = 0.f;
  for (int c = 0; c < split; ++c) sum += expf(geom.part_lse[s0 + c * C::kBM] - mx);
  const float L = mx + logf(sum);
  float mu_row = 0.f;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f), t = o;
  for (int c = 0; c < split; ++c) {
    const int64_t sr = s0 + c * C::kBM;
    const float w = expf(geom.part_lse[sr] - L);
    const float mc = geom.part_mu[sr];
    mu_row += w * mc;
    const float4 oc = *reinterpret_cast<const float4*>(geom.part_o + sr * C::kDV + col);
    const float4 tc = *reinterpret_cast<const float4*>(geom.part_ot + sr * C::kDV + col);
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
  const int64_t off = static_cast<int64_t>(bb) * geom.o_stride[0] + static_cast<int64_t>(qrow) * geom.o_stride[1] +
                      static_cast<int64_t>(hh) * geom.o_stride[2] + vh * C::kDV + col;
  __stcs(reinterpret_cast<float4*>(out + off), o);
  __stcs(reinterpret_cast<float4*>(out_t + off), t);
  if (col == 0 && vh == 0) {
    const int64_t ridx = static_cast<int64_t>(bh) * geom.Nq + qrow;
    if (lse) lse[ridx] = L;
    if (mu) mu[ridx] = mu_row;
  }
}

}  // namespace

// A stream-ordered memory pool per device for the last wave's partial outputs.
// Its release threshold keeps the memory mapped between calls: a pool that gives
// its memory back at every synchronisation maps it again on the next call, which
// costs more than the cut saves.  It holds at most the largest set of partials a
// call has needed (SMs x 128 rows x (2 x 128 + 2) floats, about 20 MB on 152 SMs)
// and lives as long as the process.
static cudaError_t piece_pool(cudaMemPool_t* pool) {
  constexpr int kMaxDev = 64;
  static std::mutex mu;
  static cudaMemPool_t pools[kMaxDev] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!pools[dev]) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t p = nullptr;
    e = cudaMemPoolCreate(&p, &props);
    if (e != cudaSuccess) return e;
    uint64_t keep = ~uint64_t(0);
    e = cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &keep);
    if (e != cudaSuccess) {
      cudaMemPoolDestroy(p);
      return e;
    }
    pools[dev] = p;
  }
  *pool = pools[dev];
  return cudaSuccess;
}

cudaError_t piece_alloc(void** ptr, size_t bytes, cudaStream_t stream) {
  // A stream being captured into a CUDA graph takes the allocation as a graph
  // memory node from the device's default pool; otherwise the library's pool.
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(stream, &cap);
  if (e != cudaSuccess) return e;
  if (cap != cudaStreamCaptureStatusNone) return cudaMallocAsync(ptr, bytes, stream);
  cudaMemPool_t pool = nullptr;
  e = piece_pool(&pool);
  if (e != cudaSuccess) return e;
  return cudaMallocFromPoolAsync(ptr, bytes, pool, stream);
}

// Pieces per unit of the last wave (1: no cut) for a grid of ``grid`` units over
// kv_len keys on n_sm SMs: only a last wave at most half full is cut, into as
// many pieces as spread it over all SMs, at least four 64-key tiles each and at
// most FwdGeom::kMaxSplit.
int64_t last_wave_split(int64_t grid, int64_t kv_len, int n_sm) {
  if (n_sm <= 0 || grid < n_sm) return 1;
  const int64_t tail = grid % n_sm;
  if (tail == 0 || 2 * tail > n_sm) return 1;
  int64_t split = n_sm / tail;
  const int64_t nt = (kv_len + 63) / 64;
  if (split > nt / 4) split = nt / 4;
  if (split > FwdGeom::kMaxSplit) split = FwdGeom::kMaxSplit;
  return split >= 2 ? split : 1;
}


namespace {

template <int D, int DVF>
cudaError_t launch_d(const FwdArgs& a, const char** msg) {
  using C = FwdCfg<D, DVF>;
  FwdMaps maps;
  FwdGeom geom;
  cudaError_t e = cudaSuccess;
  const void* ptrs[6] = {a.q, a.q_t, a.k, a.k_t, a.v, a.v_t};
  CUtensorMap* dst[6] = {&maps.q, &maps.qt, &maps.k, &maps.kt, &maps.v, &maps.vt};
  for (int i = 0; i < 6 && e == cudaSuccess; ++i) {
    const int g = i / 2;  // Q and Qt, K and Kt, V and Vt
    const int64_t* st = g == 0 ? a.q_stride : (g == 1 ? a.k_stride : a.v_stride);
    e = make_map(dst[i], ptrs[i], g == 2 ? a.d_v : a.d, g == 0 ? a.Nq : a.Nkv, a.H, a.B, st,
                 g == 0 ? C::kBM : C::kBN);
  }
  if (e != cudaSuccess) {
    *msg = "cuTensorMapEncodeTiled rejected a tensor (alignment, stride or size)";
    return e;
  }
  auto kern = attn_jvp_fwd_kernel<D, DVF>;
  bool first = false;
  e = ensure_smem_limit(reinterpret_cast<const void*>(kern), C::kSmemBytes, &first);
  if (e != cudaSuccess) {
    *msg = "cudaFuncSetAttribute(max dynamic shared memory) failed";
    return e;
  }
  const int n_qtiles = static_cast<int>((a.Nq + C::kBM - 1) / C::kBM);
  geom.H = static_cast<int>(a.H);
  geom.Nq = static_cast<int>(a.Nq);
  geom.n_qtiles = n_qtiles;
  geom.kv_start = static_cast<int>(a.kv_start);
  geom.kv_len = static_cast<int>(a.kv_len);
  geom.d_v = static_cast<int>(a.d_v);
  geom.scale = a.scale;
  for (int i = 0; i < 3; ++i) geom.o_stride[i] = a.o_stride[i];
  const int64_t grid = static_cast<int64_t>(n_qtiles) * a.B * a.H * C::kVSplit;
  // One CTA per SM (the kernel takes all of TMEM), so the grid runs in waves of
  // the SM count.  When the last wave is at most half full, its units are cut
  // into pieces over the keys that spread over the whole GPU (at least four key
  // tiles each), merged afterwards.
  geom.n_main = static_cast<int>(grid);
  geom.split = 1;
  geom.part_o = geom.part_ot = geom.part_lse = geom.part_mu = nullptr;
  const int n_sm = device_sm_count();
  const int64_t tail = n_sm > 0 ? grid % n_sm : 0;
  const int64_t nt = (a.kv_len + C::kBN - 1) / C::kBN;
  const int64_t split = a.balance_tail ? last_wave_split(grid, a.kv_len, n_sm) : 1;
  void* ws = nullptr;
  if (split > 1) {
    const int64_t slots = tail * split * C::kBM;
    e = piece_alloc(&ws, static_cast<size_t>(slots) * (2 * C::kDV + 2) * sizeof(float), a.stream);
    if (e != cudaSuccess) {
      *msg = "stream-ordered allocation of the last wave's partial outputs failed";
      return e;
    }
    geom.n_main = static_cast<int>(grid - tail);
    geom.split = static_cast<int>(split);
    for (int c = 0; c <= split; ++c) geom.piece_t[c] = static_cast<int>(c * nt / split);
    geom.part_o = static_cast<float*>(ws);
    geom.part_ot = geom.part_o + slots * C::kDV;
    geom.part_lse = geom.part_ot + slots * C::kDV;
    geom.part_mu = geom.part_lse + slots;
  }
  const int64_t launched = geom.n_main + (grid - geom.n_main) * geom.split;
  kern<<<static_cast<unsigned>(launched), kThreads, C::kSmemBytes, a.stream>>>(maps, geom, a.out, a.out_t, a.lse,
                                                                               a.mu, a.status);
  e = cudaGetLastError();
  if (e != cudaSuccess) *msg = "attention-JVP kernel launch failed";
  if (ws) {
    if (e == cudaSuccess) {
      const int ncols = C::kSmallV ? static_cast<int>(a.d_v) : C::kDV;
      const int64_t threads = tail * C::kBM * (ncols / 4);
      merge_pieces_kernel<C><<<static_cast<unsigned>((threads + 255) / 256), 256, 0, a.stream>>>(
          geom, static_cast<int>(tail), ncols, a.out, a.out_t, a.lse, a.mu);
      e = cudaGetLastError();
      if (e != cudaSuccess) *msg = "merge of the last wave's pieces failed to launch";
    }
    const cudaError_t f = cudaFreeAsync(ws, a.stream);
    if (e == cudaSuccess && f != cudaSuccess) {
      *msg = "stream-ordered release of the last wave's partial outputs failed";
      e = f;
    }
  }
  return e;
}

}  // namespace

namespace {

// Head dim rounded up to the instantiation that runs it (0: none).
int padded_dim(int64_t d) {
  if (d == 16 || d == 32 || d == 64) return 64;
  if (d == 128 || d == 256) return static_cast<int>(d);
  return 0;
}

template <int D>
cudaError_t launch_dv(const FwdArgs& a, const char** msg) {
  switch (padded_dim(a.d_v)) {
    case 64: return launch_d<D, 64>(a, msg);
    case 128: return launch_d<D, 128>(a, msg);
    case 256: return launch_d<D, 256>(a, msg);
    default: *msg = "unsupported value head dimension"; return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_attn_jvp_fwd(const FwdArgs& a, const char** msg) {
  switch (padded_dim(a.d)) {
    case 64: return launch_dv<64>(a, msg);
    case 128: return launch_dv<128>(a, msg);
    case 256: return launch_dv<256>(a, msg);
    default: *msg = "unsupported head dimension"; return cudaErrorInvalidValue;
  }
}

}  // namespace attnjvp
