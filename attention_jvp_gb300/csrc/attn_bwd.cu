// Primal attention backward for sm_103a (tcgen05 / TMEM / TMA).
//
// What it computes (page "带分数正则的一致性蒸馏", section 反向 (backward)): with
// the upstream gradient dO of O = P V, P = softmax(S), S = s Q K^T,
//     dV = P^T dO,  dP = dO V^T,  dS = P (.) (dP - rowsum(dP (.) P)),
//     dQ = s dS K,  dK = s dS^T Q.
// P is rebuilt exactly from the forward's LSE (P = exp(s q.k - LSE)), and
// rowsum(dP (.) P) is taken as rowsum(dO (.) O), the same number by
// O = P V, computed once per query row by bwd_prep_kernel together with
// -LSE log2 e.
//
// Two passes, each one CTA per 128 resident rows of one (batch, head), each
// streaming 64-row tiles of the other side, with hand-offs like the forward
// kernel's:
//   dQ pass   (resident Q, dO; streamed K, V):  S1 = Q K^T, S2 = dO V^T,
//             dS = P (.) (S2 - D) per query row, dQ += dS K.
//   dK/dV pass (resident K, V; streamed Q, dO and the per-query -LSE log2 e
//             and -D):  S1 = K Q^T, S2 = V dO^T (both transposed: TMEM lane =
//             key), P^T and dS^T per key row, dV += P^T dO, dK += dS^T Q.
// At head dim 256 two CTAs share each resident tile, each accumulating half of
// the gradient columns (the fp32 dK and dV of 128 keys would fill TMEM); both
// form the full 256-deep scores.
// Warps: 0 TMA (resident tiles, then the ring of streamed tiles, which up to
// head dim 128 feeds both the score and the value MMAs, the value ring of its
// own at 256 and, in the dK/dV pass, the per-query vector ring, each refilled
// as soon as it frees),
// 1 TMEM + value MMAs, 2 S2 MMAs, 3 S1 MMAs, and two groups of
// elementwise warps (thread = resident row = TMEM lane): 4-7 take the even
// tiles, 8-11 the odd ones.  One group's per-tile chain (barrier waits, TMEM
// load, exp2 and packing, TMEM store, arrival) is about as long as the tile's
// MMAs, so a single group left the tensor pipe idle half the time; with two,
// one group's waits overlap the other's arithmetic.  The groups split the
// epilogue by 32-column chunks.  In the dQ pass the score MMAs take Q and dO
// from TMEM copies.  The two passes recompute S and dP (14 d flops
// per (query, key) pair instead of 10) but need no atomics, so results are
// deterministic.  A last wave at most half full is cut into pieces over the
// streamed rows, as in the forward, and a second kernel adds their partial sums.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace attnjvp {
namespace {

using namespace ptx;

constexpr int kModeDQ = 0;
constexpr int kModeDKDV = 1;

template <int D, int kMode>
struct BwdCfg {
  static constexpr bool kDKDV = kMode == kModeDKDV;
  static constexpr int kBM = 128;                  // resident rows per CTA (= TMEM lanes)
  static constexpr int kBN = 64;                   // streamed rows per tile
  static constexpr int kDC = D / 64;               // 64-element (128-byte) d-chunks
  // Gradient columns per CTA.  At head dim 256 the fp32 accumulators of one
  // resident tile (dK and dV: 512 columns) would fill TMEM, so two CTAs share
  // each resident tile, each accumulating half of the gradient columns (and
  // each forming the full 256-deep scores), as the forward does with O and T.
  static constexpr int kDV = D > 128 ? 128 : D;
  static constexpr int kVC = kDV / 64;             // 64-element chunks of a value tile
  static constexpr int kVSplit = D / kDV;          // CTAs per resident tile
  // dQ pass: the resident Q and dO also live in TMEM (bf16, D/2 columns each) as
  // the A operands of the score MMAs, which then read only the streamed tiles
  // from shared memory (with both operands there, a 64-wide score MMA wants
  // about 1.5x the shared-memory bandwidth).  Not at 256, where they do not fit.
  static constexpr bool kRTmem = !kDKDV && D <= 128;
  static constexpr int kNSt = 3;                   // S2 (then packed operands) TMEM buffers
  // S1 TMEM buffers: as many (up to 3) as the columns left beside the
  // accumulators, the resident copies and the S2 buffers hold.
  static constexpr int kFreeCols = 512 - (kDKDV ? 2 : 1) * kDV - (kRTmem ? D : 0) - 64 * kNSt;
  static constexpr int kNS = kFreeCols >= 192 ? 3 : 1;
  // Barrier slots of the S1 ring.  Tiles alternate between the two elementwise
  // groups; with a single buffer, consecutive tiles on one barrier would belong
  // to different groups, and a group could test a phase parity before the
  // previous phase completed.  Two slots (by tile parity) give each group its
  // own barrier.  With three buffers, the group reaching tile j + 3 has
  // finished tile j + 1, so tile j's phase (issued earlier by the same thread)
  // is complete.
  static constexpr int kSBar = kNS == 1 ? 2 : kNS;
  // Up to head dim 128 one ring serves both MMA kinds: the value MMAs take their
  // B operands (dK/dV pass: dO and Q; dQ pass: K) from the same stage as the
  // score MMAs, which then stays until the value MMAs of its tile are done.  A
  // second ring would load every streamed tile twice, and shared memory is what
  // bounds the 64-wide score MMAs (their operands, the value MMAs' B operands
  // and the TMA writes all go through it).
  // At 256 the resident tiles take 128 KB of shared memory, which leaves one
  // score stage and a value ring of its own with one (dK/dV) or two (dQ) stages
  // of this CTA's gradient columns only.
  static constexpr bool kShared = D <= 128;
  static constexpr int kKS = D == 256 ? 1 : (D == 128 ? 4 : 6);  // score-tile ring stages
  static constexpr int kVS = kShared ? 1 : (kDKDV ? 1 : 2);        // own value ring (head dim 256)
  static constexpr int kChunkR = kBM * 128;        // one d-chunk of a resident tile (bytes)
  static constexpr int kChunkX = kBN * 128;        // one d-chunk of a streamed tile (bytes)
  static constexpr int kRBytes = kDC * kChunkR;
  static constexpr int kKStage = 2 * kDC * kChunkX;              // X1 chunks, X2 chunks
  // Score ring units: normally a whole streamed tile; with room for one tile only
  // (head dim 256) two units of half its d-chunks each, so that the next tile's
  // first half loads while this tile's second half is in the score MMAs.
  static constexpr int kUPT = (kKS == 1 && kDC % 2 == 0) ? 2 : 1;  // units per tile
  static constexpr int kUC = kDC / kUPT;                           // d-chunks of X1 (and X2) per unit
  static constexpr int kKU = kKS * kUPT;                           // units in the ring
  static constexpr int kKUnit = 2 * kUC * kChunkX;                 // X1 chunks, then X2 chunks
  static constexpr int kVTensors = kDKDV ? 2 : 1;
  static constexpr int kVStage = kVTensors * kVC * kChunkX;      // dK/dV: dO, Q;  dQ: K (this CTA's columns)
  // dK/dV: the streamed queries' -LSE log2e and -D (64 + 64 floats) in a ring of
  // their own, released by the elementwise warps once read (the value ring is
  // released only by the value MMAs, two tiles later than they need it)
  static constexpr int kVecS = D == 256 ? 2 : 4;
  static constexpr int kVecSlot = 512;
  static constexpr int kVecRing = kDKDV ? kVecS * kVecSlot : 0;
  static constexpr int kOffR1 = 0;
  static constexpr int kOffR2 = kRBytes;
  static constexpr int kOffK = 2 * kRBytes;
  static constexpr int kOffV = kOffK + kKU * kKUnit;
  static constexpr int kOffVec = kOffV + (kShared ? 0 : kVS * kVStage);
  static constexpr int kOffBar = kOffVec + kVecRing;
  static constexpr int kBarBytes = 512;  // the Barriers block below
  static constexpr int kSmemBytes = kOffBar + kBarBytes + 1024;  // + alignment slack
  // TMEM: ACC1 [0, DV) (dQ or dV), ACC2 [DV, 2DV) (dK), the dQ pass's resident
  // copies, S1 buffers, S2 buffers (64 columns each)
  static constexpr uint32_t kColAcc1 = 0;
  static constexpr uint32_t kColAcc2 = kDV;
  static constexpr uint32_t kColR1 = (kDKDV ? 2 : 1) * kDV;  // dQ pass: Q, then dO (bf16 pairs)
  static constexpr uint32_t kColR2 = kColR1 + D / 2;
  static constexpr uint32_t kColS = kColR1 + (kRTmem ? D : 0);
  static constexpr uint32_t kColSt = kColS + 64 * kNS;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kColSt + 64 * kNSt <= kTmemCols, "TMEM budget");
  static_assert(kSBar <= 3 && kNSt <= 3 && kKU <= 6 && kVS <= 3 && kVecS <= 4, "barrier arrays");
  static_assert(!kShared || (kUPT == 1 && kVC == kDC), "a shared stage holds whole tiles of every column");
  static_assert(kKU * kKUnit == kKS * kKStage, "score ring size");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static_assert(kKU * kKUnit >= 8 * 4096, "the streamed-tile ring also holds the eight 4 KB epilogue stages");
  static_assert(kKStage % 1024 == 0 && kVStage % 1024 == 0, "stage alignment (128-byte swizzle atoms)");
};

constexpr int kThreads = 384;  // 12 warps
// Registers per thread after the split at the start of the kernel: the TMA and
// MMA warpgroup gives up what the elementwise warpgroups take.  The block's pool
// is its threads x the registers per thread it was launched with (the launch
// bounds allow 168), and ``setmaxnreg.inc`` waits until the pool has room, so
// the launch checks that the compiled count leaves enough.
constexpr int kRegsIssue = 88;
constexpr int kRegsElem = 208;
constexpr int kRegPoolNeeded = 128 * kRegsIssue + 256 * kRegsElem;
static_assert(kRegPoolNeeded <= kThreads * 168, "register split above the launch pool");
constexpr float kLog2e = 1.4426950408889634f;

struct BwdMaps {
  CUtensorMap r1, r2, x1, x2;  // resident and streamed bf16 tiles
  CUtensorMap nl2, nd;         // dK/dV pass: per-query -LSE log2e and -D, fp32 [B*H, Nq]
};

struct BwdGeom {
  int H, n_rtiles, n_res, n_str;  // resident / streamed row counts
  int nq_pad;                     // row length of the per-query vectors (N_q rounded up to 4)
  int d;
  float scale;
  const float* row_nl2;           // dQ pass: per resident row (query) -LSE log2e and -D
  const float* row_nd;
  float* out1;                    // dQ pass: dQ;  dK/dV pass: dV
  float* out2;                    // dK/dV pass: dK
  // Balance of a short last wave, as in the forward: the units (resident tile,
  // column half) from n_main on are cut into ``split`` pieces over the streamed
  // rows, piece c taking streamed tiles [piece_t[c], piece_t[c + 1]).  A piece
  // writes its partial sums (already scaled) to part1 / part2, slot
  // (unit - n_main) * split + c of 128 rows x kDV columns, and
  // bwd_merge_pieces_kernel adds the pieces of each unit.  split == 1: no pieces.
  static constexpr int kMaxSplit = 16;
  int n_main, split;
  int piece_t[kMaxSplit + 1];
  float *part1, *part2;
};

struct Barriers {
  uint64_t r_full;
  uint64_t k_full[6], k_empty[6];
  uint64_t v_full[3], v_empty[3];
  uint64_t vec_full[4], vec_empty[4];
  uint64_t s_full[3], st_full[3], s_free[3], p_full[3], pv_done[3];
  uint64_t drain, drain_s, drain_st;
  uint64_t acc_done;  // all value MMAs done (single use)
  uint64_t r_tmem;    // dQ pass: Q and dO copied into TMEM (one arrival per warp of group 0)
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Barriers) <= BwdCfg<128, kModeDQ>::kBarBytes, "barrier block");

// 64 TMEM columns of the calling thread's lane into r[kOff .. kOff + 63].
#define BWD_R8(o) "=r"(r[o + 0]), "=r"(r[o + 1]), "=r"(r[o + 2]), "=r"(r[o + 3]), \
                  "=r"(r[o + 4]), "=r"(r[o + 5]), "=r"(r[o + 6]), "=r"(r[o + 7])
template <int kOff>
__device__ __forceinline__ void tmem_ld64_wait(uint32_t taddr, uint32_t (&r)[128]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,"
      "%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,"
      "%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : BWD_R8(kOff + 0), BWD_R8(kOff + 8), BWD_R8(kOff + 16), BWD_R8(kOff + 24), BWD_R8(kOff + 32),
        BWD_R8(kOff + 40), BWD_R8(kOff + 48), BWD_R8(kOff + 56)
      : "r"(taddr)
      : "memory");
}
#undef BWD_R8

// Elementwise step of one 64-column tile for the calling thread's resident
// row, from raw S1 (raw[0..63]) and S2 (raw[64..127]) already loaded from
// TMEM.  cSt: the row's TMEM address of the S2 buffer, which receives the
// bf16 operands: dQ pass dS in columns 0-31 (bf16 pairs); dK/dV pass P^T in
// 0-31 and dS^T in 32-63.
// ``nl2`` / ``nd``: -LSE log2e and -D, per row (dQ pass, in registers) or per
// column (dK/dV pass, 64 values each in shared memory).  kMasked: only the
// first ``valid`` columns are real.
template <int kMode, bool kMasked>
__device__ __forceinline__ void bwd_tile(uint32_t (&raw)[128], uint32_t cSt, int valid, float c2, float row_nl2,
                                         float row_nd, const float* col_nl2, const float* col_nd) {
  if (kMasked) {
#pragma unroll
    for (int i = 0; i < 64; ++i)
      if (i >= valid) raw[i] = __float_as_uint(-INFINITY);  // weight 0
  }
  auto f = [&](int i) { return __uint_as_float(raw[i]); };
  const uint64_t c2x2 = f2_pack(c2, c2);
  auto step = [&](int i, uint64_t nl, uint64_t nd, uint32_t& pw, uint32_t& dw) {
    float x0, x1;
    f2_unpack(f2_fma(f2_pack(f(i), f(i + 1)), c2x2, nl), x0, x1);
    const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
    float d0, d1;
    f2_unpack(f2_mul(f2_pack(p0, p1), f2_add(f2_pack(f(64 + i), f(65 + i)), nd)), d0, d1);
    if (kMode == kModeDKDV) pw = pack_bf16x2(p0, p1);
    dw = pack_bf16x2(d0, d1);
  };
  if (kMode == kModeDQ) {
    uint32_t pk[32], dk[32];
    const uint64_t nl = f2_pack(row_nl2, row_nl2), nd = f2_pack(row_nd, row_nd);
#pragma unroll
    for (int i = 0; i < 64; i += 2) step(i, nl, nd, pk[i >> 1], dk[i >> 1]);
    tmem_st32(cSt, dk);
  } else {
    // Two halves of 32 columns, each stored as soon as it is packed, so that the
    // packed words of the first half are not live across the second.
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t pk[16], dk[16];
#pragma unroll
      for (int i = 32 * h; i < 32 * h + 32; i += 4) {
        // 16-byte broadcast reads (the vector slots are 512-byte aligned)
        const float4 a = *reinterpret_cast<const float4*>(col_nl2 + i);
        const float4 b = *reinterpret_cast<const float4*>(col_nd + i);
        const int w = (i - 32 * h) >> 1;
        step(i, f2_pack(a.x, a.y), f2_pack(b.x, b.y), pk[w], dk[w]);
        step(i + 2, f2_pack(a.z, a.w), f2_pack(b.z, b.w), pk[w + 1], dk[w + 1]);
      }
      tmem_st16(cSt + 16 * h, pk);
      tmem_st16(cSt + 32 + 16 * h, dk);
    }
  }
  tmem_wait_st();
  tc_fence_before_sync();
}

// kCut: the grid's last wave is cut into pieces (see BwdGeom).  A separate
// instantiation, so that grids without a cut run the plain code.
template <int D, int kMode, bool kCut>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_kernel(const __grid_constant__ BwdMaps maps, const __grid_constant__ BwdGeom geom, int* status) {
  using C = BwdCfg<D, kMode>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Barriers* bars = reinterpret_cast<Barriers*>(smem + C::kOffBar);
  volatile int* abort_flag = &bars->abort_flag;

  if (threadIdx.x == 0) bars->abort_flag = (*reinterpret_cast<volatile int*>(status) & kStatusTimeout) ? 1 : 0;
  __syncthreads();
  if (bars->abort_flag) return;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Both column halves of a resident tile (head dim 256) are neighbours in the
  // grid, so they stream the same tiles through L2 at about the same time.
  // A CTA past n_main is one piece of a unit of the last wave: that unit's
  // streamed tiles [piece_t[c], piece_t[c + 1]).
  unsigned unit = blockIdx.x;
  int piece = -1;  // this CTA's partial-output slot, or -1 (outputs in place)
  int t_first = 0, n_tiles = (geom.n_str + C::kBN - 1) / C::kBN;
  if (kCut && unit >= static_cast<unsigned>(geom.n_main)) {
    piece = static_cast<int>(unit - geom.n_main);
    const unsigned u = static_cast<unsigned>(piece) / static_cast<unsigned>(geom.split);
    const int c = piece - static_cast<int>(u) * geom.split;
    unit = geom.n_main + u;
    t_first = geom.piece_t[c];
    n_tiles = geom.piece_t[c + 1] - t_first;
  }
  const int str0 = t_first * C::kBN;  // first streamed row of this CTA
  const int vh = unit % C::kVSplit;       // which kDV gradient columns this CTA accumulates
  const unsigned rb = unit / C::kVSplit;  // unsigned: the divisions below stay unsigned
  const int bh = rb / geom.n_rtiles;
  const int hh = bh % geom.H, bb = bh / geom.H;
  const int r0 = (rb % geom.n_rtiles) * C::kBM;

  if (threadIdx.x == 0) {
    mbar_init(&bars->r_full, 1);
    for (int s = 0; s < 6; ++s) {
      mbar_init(&bars->k_full[s], 1);
      // one commit from each score issuer, and one from the value issuer when
      // its B operands come from the same stage
      mbar_init(&bars->k_empty[s], C::kShared ? 3 : 2);
    }
    for (int s = 0; s < 3; ++s) {
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->st_full[s], 1);
      mbar_init(&bars->p_full[s], 4);  // one arrival per elementwise warp
      mbar_init(&bars->pv_done[s], 1);
      mbar_init(&bars->s_free[s], 4);
    }
    mbar_init(&bars->drain, 1);
    mbar_init(&bars->drain_s, 1);
    mbar_init(&bars->drain_st, 1);
    mbar_init(&bars->acc_done, 1);
    mbar_init(&bars->r_tmem, 4);
    for (int s = 0; s < 4; ++s) {
      mbar_init(&bars->vec_full[s], 1);
      mbar_init(&bars->vec_empty[s], 4);  // one arrival per warp of the group that used the slot
    }
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

  // Registers: the TMA and MMA warps need few, the elementwise warps hold a
  // whole tile of scores per thread.  Each setmaxnreg is the first instruction of
  // the region it governs (all warps of a warpgroup execute the same one), so the
  // compiler allocates each region within its own count.
  if (warp >= 4) {
    setmaxnreg_inc<kRegsElem>();
    // ---------------- elementwise + epilogue: one resident row per thread; group 0
    // (warps 4-7) takes the even tiles, group 1 (warps 8-11) the odd ones ----------------
    const int group = (warp - 4) >> 2;
    const int quarter = warp & 3;  // TMEM lane quarter a warp may access
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float c2 = geom.scale * kLog2e;
    float row_nl2 = 0.f, row_nd = 0.f;
    if (!C::kDKDV && r0 + row < geom.n_res) {
      const int64_t ridx = static_cast<int64_t>(bh) * geom.nq_pad + r0 + row;
      row_nl2 = geom.row_nl2[ridx];
      row_nd = geom.row_nd[ridx];
    }
    bool ok = true;
    if (C::kRTmem && group == 0) {
      // Rows of Q and dO (128-byte-swizzled d-chunks: 16-byte unit u of row r at
      // unit u ^ (r mod 8)) into this thread's TMEM lane.
      ok = __all_sync(0xffffffffu, mbar_wait<1>(&bars->r_full, 0, abort_flag, status, kStatusTimeout));
      if (ok) {
#pragma unroll 1
        for (int m = 0; m < 2 * C::kDC; ++m) {
          const int c = m % C::kDC;
          const uint8_t* src = smem + (m < C::kDC ? C::kOffR1 : C::kOffR2) + c * C::kChunkR + row * 128;
          uint32_t w[32];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint4 x = *reinterpret_cast<const uint4*>(src + ((u ^ (row & 7)) << 4));
            w[4 * u] = x.x, w[4 * u + 1] = x.y, w[4 * u + 2] = x.z, w[4 * u + 3] = x.w;
          }
          tmem_st32(lane_addr + (m < C::kDC ? C::kColR1 : C::kColR2) + 32 * c, w);
        }
        tmem_wait_st();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->r_tmem);
      }
    }
    for (int j = group; ok && j < n_tiles; j += 2) {
      const int b = j % C::kNS;
      const int bs = j % C::kSBar;
      const int bt = j % C::kNSt;
      // S1 first, and its buffer released at once: the S1 ring is the short one,
      // and the next tile's S1 MMAs wait for it.
      ok = mbar_wait<1>(&bars->s_full[bs], (j / C::kSBar) & 1, abort_flag, status, kStatusTimeout);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after_sync();
      uint32_t raw[128];
      tmem_ld64_wait<0>(lane_addr + C::kColS + 64u * b, raw);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->s_free[bs]);
      ok = mbar_wait<1>(&bars->st_full[bt], (j / C::kNSt) & 1, abort_flag, status, kStatusTimeout);
      // dK/dV pass: the streamed queries' vectors
      const int sq = j % C::kVecS;
      if (C::kDKDV && ok)
        ok = mbar_wait<1>(&bars->vec_full[sq], (j / C::kVecS) & 1, abort_flag, status, kStatusTimeout);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after_sync();
      const uint32_t cSt = lane_addr + C::kColSt + 64u * bt;
      tmem_ld64_wait<64>(cSt, raw);
      const int valid = min(C::kBN, geom.n_str - str0 - j * C::kBN);
      const float* vec = reinterpret_cast<const float*>(smem + C::kOffVec + sq * C::kVecSlot);
      if (valid == C::kBN)
        bwd_tile<kMode, false>(raw, cSt, valid, c2, row_nl2, row_nd, vec, vec + 64);
      else
        bwd_tile<kMode, true>(raw, cSt, valid, c2, row_nl2, row_nd, vec, vec + 64);
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars->p_full[bt]);
        if (C::kDKDV) mbar_arrive(&bars->vec_empty[sq]);
      }
    }
    // ---------------- epilogue ----------------
    if (ok) ok = mbar_wait<1>(&bars->acc_done, 0, abort_flag, status, kStatusTimeout);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      tc_fence_after_sync();
      // Every MMA and copy of the CTA is done: the streamed-tile ring's shared
      // memory is free and holds each elementwise warp's 4 KB epilogue stage.
      // Stores from one thread per row would touch 32 rows per warp instruction,
      // so a warp passes each 32-column chunk through its stage (16-byte unit u of
      // row r at unit u ^ (r mod 8), conflict-free both ways) and writes it back
      // four rows per instruction, eight lanes per 128-byte row segment.
      fence_proxy_async_smem();
      float4* stage = reinterpret_cast<float4*>(smem + C::kOffK + (group * 4 + quarter) * 4096);
      const int ru = lane & 7, rr = lane >> 3;
      // in place, or a piece's slot of 128 rows of kDV columns
      const bool part = kCut && piece >= 0;
      const int64_t rstride = part ? C::kDV : geom.d;
      const int64_t obase0 = part ? (static_cast<int64_t>(piece) * C::kBM + quarter * 32) * C::kDV
                                  : (static_cast<int64_t>(bh) * geom.n_res + r0 + quarter * 32) * geom.d +
                                        vh * C::kDV;
      const int valid_rows = min(32, geom.n_res - (r0 + quarter * 32));
      // dQ pass: ACC1 = dS K, times s.  dK/dV pass: ACC1 = dV, ACC2 = dS^T Q, times s.
      // The groups take alternate 32-column chunks.
      int chunk = 0;
#pragma unroll 1
      for (int acc = 0; acc < (C::kDKDV ? 2 : 1); ++acc) {
        float* out = (C::kDKDV && acc == 1) ? (part ? geom.part2 : geom.out2) : (part ? geom.part1 : geom.out1);
        const float mul = (C::kDKDV && acc == 0) ? 1.f : geom.scale;
        const uint32_t col = acc == 0 ? C::kColAcc1 : C::kColAcc2;
        // this CTA's kDV columns, except for the 16/32-wide heads run as 64
        const int ncols = C::kDV == 128 ? C::kDV : geom.d;
#pragma unroll 1
        for (int c0 = 0; c0 < ncols; c0 += 32) {
          if ((chunk++ & 1) != group) continue;
          uint32_t v[32];
          tmem_ld32_wait(lane_addr + col + c0, v);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            stage[lane * 8 + (i ^ (lane & 7))] =
                make_float4(__uint_as_float(v[4 * i]) * mul, __uint_as_float(v[4 * i + 1]) * mul,
                            __uint_as_float(v[4 * i + 2]) * mul, __uint_as_float(v[4 * i + 3]) * mul);
          __syncwarp();
          if (c0 + 4 * ru < ncols) {
#pragma unroll 1
            for (int i = 0; i < 8; ++i) {
              const int r = rr + 4 * i;
              if (r < valid_rows)  // streaming stores: the gradients are not read again here
                __stcs(reinterpret_cast<float4*>(out + obase0 + r * rstride + c0 + 4 * ru), stage[r * 8 + (ru ^ (r & 7))]);
            }
          }
          __syncwarp();  // the next chunk overwrites the stage
        }
      }
    }
  } else {
    setmaxnreg_dec<kRegsIssue>();
    if (warp == 0) {
      // ---------------- TMA producer: resident tiles, then the score-tile ring (X1, X2) and
      // the value-tile ring, each refilled as soon as its own stage is free (the thread polls
      // both; the value ring frees much later than the score ring) ----------------
      if (lane == 0) {
        prefetch_tensormap(&maps.r1);
        prefetch_tensormap(&maps.r2);
        prefetch_tensormap(&maps.x1);
        prefetch_tensormap(&maps.x2);
        mbar_arrive_expect_tx(&bars->r_full, 2 * C::kRBytes);
        for (int c = 0; c < C::kDC; ++c) {
          tma_load_4d(smem + C::kOffR1 + c * C::kChunkR, &maps.r1, &bars->r_full, c * 64, r0, hh, bb);
          tma_load_4d(smem + C::kOffR2 + c * C::kChunkR, &maps.r2, &bars->r_full, c * 64, r0, hh, bb);
        }
        int tk = 0, tv = 0, tq = 0;  // next tile of each ring (tq: the vector ring)
        const int nq = C::kDKDV ? n_tiles : 0;
        const int nv = C::kShared ? 0 : n_tiles;  // tiles of the value ring of its own
        bool ok = true;
        uint64_t t0 = globaltimer_ns();
        uint32_t idle = 0;
        while (tk < n_tiles * C::kUPT || tv < nv || tq < nq) {
          bool progressed = false;
          if (tq < nq && mbar_test_wait(&bars->vec_empty[tq % C::kVecS], ((tq / C::kVecS) & 1) ^ 1)) {
            const int sq = tq % C::kVecS;
            float* vec = reinterpret_cast<float*>(smem + C::kOffVec + sq * C::kVecSlot);
            mbar_arrive_expect_tx(&bars->vec_full[sq], C::kVecSlot);
            tma_load_2d(vec, &maps.nl2, &bars->vec_full[sq], str0 + tq * C::kBN, bh);
            tma_load_2d(vec + 64, &maps.nd, &bars->vec_full[sq], str0 + tq * C::kBN, bh);
            ++tq;
            progressed = true;
          }
          // tk counts score-ring units: unit u of streamed tile tk / kUPT
          if (tk < n_tiles * C::kUPT && mbar_test_wait(&bars->k_empty[tk % C::kKU], ((tk / C::kKU) & 1) ^ 1)) {
            const int s = tk % C::kKU;
            const int row0 = str0 + (tk / C::kUPT) * C::kBN, u = tk % C::kUPT;
            uint8_t* st = smem + C::kOffK + s * C::kKUnit;
            mbar_arrive_expect_tx(&bars->k_full[s], C::kKUnit);
            for (int c = 0; c < C::kUC; ++c) {
              const int col = (u * C::kUC + c) * 64;
              tma_load_4d(st + c * C::kChunkX, &maps.x1, &bars->k_full[s], col, row0, hh, bb);
              tma_load_4d(st + (C::kUC + c) * C::kChunkX, &maps.x2, &bars->k_full[s], col, row0, hh, bb);
            }
            ++tk;
            progressed = true;
          }
          if (tv < nv && mbar_test_wait(&bars->v_empty[tv % C::kVS], ((tv / C::kVS) & 1) ^ 1)) {
            const int sv = tv % C::kVS;
            const int row0 = str0 + tv * C::kBN;
            uint8_t* vt = smem + C::kOffV + sv * C::kVStage;
            mbar_arrive_expect_tx(&bars->v_full[sv], C::kVStage);
            for (int c = 0; c < C::kVC; ++c) {  // this CTA's gradient columns
              const int col = vh * C::kDV + c * 64;
              if (C::kDKDV) {  // dO (for dV), then Q (for dK)
                tma_load_4d(vt + c * C::kChunkX, &maps.x2, &bars->v_full[sv], col, row0, hh, bb);
                tma_load_4d(vt + (C::kVC + c) * C::kChunkX, &maps.x1, &bars->v_full[sv], col, row0, hh, bb);
              } else {  // K (for dQ)
                tma_load_4d(vt + c * C::kChunkX, &maps.x1, &bars->v_full[sv], col, row0, hh, bb);
              }
            }
            ++tv;
            progressed = true;
          }
          if (progressed) {
            t0 = globaltimer_ns();
            idle = 0;
            continue;
          }
          __nanosleep(64);
          // Bounded: a second without either ring moving means a broken protocol.
          if ((++idle & 15u) == 0u) {
            if (*abort_flag) {
              ok = false;
            } else if (globaltimer_ns() - t0 > kWaitLimitNs) {
              *abort_flag = 1;
              atomicOr(status, kStatusTimeout);
              ok = false;
            }
            if (!ok) break;
          }
        }
        // Let copies still in flight land before the CTA's shared memory goes away, on the
        // normal path too (another role may give up right after the last copy was issued).
        volatile int no_abort = 0;
        mbar_wait(&bars->r_full, 0, &no_abort, nullptr, 0);
        for (int n = tk - C::kKU; n < tk; ++n)
          if (n >= 0) mbar_wait(&bars->k_full[n % C::kKU], (n / C::kKU) & 1, &no_abort, nullptr, 0);
        for (int t = tv - C::kVS; t < tv; ++t)
          if (t >= 0) mbar_wait(&bars->v_full[t % C::kVS], (t / C::kVS) & 1, &no_abort, nullptr, 0);
        for (int t = tq - C::kVecS; t < tq; ++t)
          if (t >= 0) mbar_wait(&bars->vec_full[t % C::kVecS], (t / C::kVecS) & 1, &no_abort, nullptr, 0);
      }
    } else {
      // ---------------- tcgen05.mma issuers: warp 3 S1, warp 2 S2, warp 1 the value MMAs ----------------
      if (lane == 0) {
        constexpr uint32_t kIdS = make_idesc_bf16_f32(128, C::kBN, false, false);  // both K-major
        constexpr uint32_t kIdPV = make_idesc_bf16_f32(128, C::kDV, false, true);  // B N-major
        const uint64_t dR1 = make_smem_desc_sw128(smem_u32(smem + C::kOffR1), 16, 1024);
        const uint64_t dR2 = make_smem_desc_sw128(smem_u32(smem + C::kOffR2), 16, 1024);
        const uint64_t dK0 = make_smem_desc_sw128(smem_u32(smem + C::kOffK), 16, 1024);
        // B operands of the value MMAs: a stage of the shared ring (X1 chunks, then X2
        // chunks) or of the value ring of its own
        const uint64_t dV0 =
            make_smem_desc_sw128(smem_u32(smem + (C::kShared ? C::kOffK : C::kOffV)), C::kChunkX, 1024);
        auto off = [](uint64_t desc, uint32_t bytes) { return desc + static_cast<uint64_t>(bytes >> 4); };
        volatile int no_abort = 0;
        if (warp == 3 || warp == 2) {
          // S1 = R1 X1^T (warp 3) or S2 = R2 X2^T (warp 2), d-deep, N = 64.
          const bool first = warp == 3;
          const uint64_t dA = first ? dR1 : dR2;
          const uint32_t aT = tmem + (first ? C::kColR1 : C::kColR2);  // dQ pass: A in TMEM
          const uint32_t xoff = first ? 0u : static_cast<uint32_t>(C::kUC * C::kChunkX);
          bool ok = C::kRTmem ? mbar_wait(&bars->r_tmem, 0, abort_flag, status, kStatusTimeout)
                              : mbar_wait(&bars->r_full, 0, abort_flag, status, kStatusTimeout);
          for (int t = 0; ok && t < n_tiles; ++t) {
            const int b = first ? t % C::kNS : t % C::kNSt;
            const int bs = first ? t % C::kSBar : b;  // barrier slot
            const uint32_t dst = tmem + (first ? C::kColS : C::kColSt) + 64u * b;
  #pragma unroll 1
            for (int u = 0; u < C::kUPT; ++u) {
              const int n = t * C::kUPT + u;
              const int s = n % C::kKU;
              ok = mbar_wait(&bars->k_full[s], (n / C::kKU) & 1, abort_flag, status, kStatusTimeout);
              // S1 buffers are free once the elementwise warps loaded tile t - NS; S2 buffers
              // hold the packed operands of tile t - NSt until its value MMAs are done.
              if (ok && u == 0 && first && t >= C::kNS)
                ok = mbar_wait(&bars->s_free[(t - C::kNS) % C::kSBar], ((t - C::kNS) / C::kSBar) & 1, abort_flag,
                               status, kStatusTimeout);
              if (ok && u == 0 && !first && t >= C::kNSt)
                ok = mbar_wait(&bars->pv_done[b], ((t - C::kNSt) / C::kNSt) & 1, abort_flag, status,
                               kStatusTimeout);
              if (!ok) break;
              tc_fence_after_sync();
              const uint64_t dX = off(dK0, s * C::kKUnit + xoff);
  #pragma unroll
              for (int c = 0; c < C::kUC; ++c)
  #pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                  const int cg = u * C::kUC + c;  // d-chunk of the resident operand
                  if constexpr (C::kRTmem)
                    mma_ts(dst, aT + (cg * 4 + kk) * 8, off(dX, c * C::kChunkX + kk * 32), kIdS, (u | c | kk) != 0);
                  else
                    mma_ss(dst, off(dA, cg * C::kChunkR + kk * 32), off(dX, c * C::kChunkX + kk * 32), kIdS,
                           (u | c | kk) != 0);
                }
              mma_commit(&bars->k_empty[s]);
            }
            if (!ok) break;
            mma_commit(first ? &bars->s_full[bs] : &bars->st_full[b]);
          }
          uint64_t* drain = first ? &bars->drain_s : &bars->drain_st;
          mma_commit(drain);
          mbar_wait(drain, 0, &no_abort, nullptr, 0);
        } else {
          bool ok = true;
          for (int j = 0; ok && j < n_tiles; ++j) {
            const int bt = j % C::kNSt;
            const int s = j % (C::kShared ? C::kKS : C::kVS);
            const uint32_t sphase = (j / (C::kShared ? C::kKS : C::kVS)) & 1;
            ok = mbar_wait(&bars->p_full[bt], (j / C::kNSt) & 1, abort_flag, status, kStatusTimeout) &&
                 mbar_wait(C::kShared ? &bars->k_full[s] : &bars->v_full[s], sphase, abort_flag, status,
                           kStatusTimeout);
            if (!ok) break;
            tc_fence_after_sync();
            // dK/dV pass: dO, then Q (shared stage: X2 = dO after X1 = Q).  dQ pass: K (X1).
            const uint64_t dV = off(dV0, C::kShared ? s * C::kKUnit : s * C::kVStage);
            const uint32_t dO_off = C::kShared ? C::kUC * C::kChunkX : 0;
            const uint32_t q_off = C::kShared ? 0 : C::kVC * C::kChunkX;
            const uint32_t a0 = tmem + C::kColSt + 64u * bt;  // dQ: dS;  dK/dV: P^T (then dS^T at +32)
  #pragma unroll
            for (int kk = 0; kk < C::kBN / 16; ++kk) {
              const uint32_t acc = (j > 0 || kk > 0) ? 1u : 0u;
              if (C::kDKDV) {
                mma_ts(tmem + C::kColAcc1, a0 + kk * 8, off(dV, dO_off + kk * 2048), kIdPV, acc);  // dV += P^T dO
                mma_ts(tmem + C::kColAcc2, a0 + 32 + kk * 8, off(dV, q_off + kk * 2048), kIdPV,
                       acc);  // dK += dS^T Q
              } else {
                mma_ts(tmem + C::kColAcc1, a0 + kk * 8, off(dV, kk * 2048), kIdPV, acc);  // dQ += dS K
              }
            }
            mma_commit(C::kShared ? &bars->k_empty[s] : &bars->v_empty[s]);
            mma_commit(&bars->pv_done[bt]);
          }
          if (ok) mma_commit(&bars->acc_done);
          mma_commit(&bars->drain);
          mbar_wait(&bars->drain, 0, &no_abort, nullptr, 0);
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// -LSE log2e and -D = -rowsum(dO (.) O) per query row, one warp per row,
// stored in rows of nq_pad floats per (b, h) (16-byte TMA strides).
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __nv_bfloat16* __restrict__ dO,
                                                       const float* __restrict__ O, const float* __restrict__ lse,
                                                       float* __restrict__ nl2, float* __restrict__ nd, int64_t rows,
                                                       int64_t nq, int64_t nq_pad, int d) {
  const int64_t r = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  float s = 0.f;
  for (int c = lane; c < d; c += 32) s = fmaf(__bfloat162float(dO[r * d + c]), O[r * d + c], s);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_down_sync(0xffffffffu, s, o);
  if (lane == 0) {
    const int64_t w = (r / nq) * nq_pad + r % nq;
    nl2[w] = -lse[r] * kLog2e;
    nd[w] = -s;
  }
}

// Adds the pieces of each cut unit (see BwdGeom) into its outputs: one thread per
// 4 columns of one row of one unit, both accumulators in the dK/dV pass.
template <class C>
__global__ void __launch_bounds__(256) bwd_merge_pieces_kernel(const __grid_constant__ BwdGeom geom, int n_units,
                                                               int ncols) {
  const int tpr = ncols >> 2;
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t rowid = gtid / tpr;  // unit * 128 + row
  if (rowid >= static_cast<int64_t>(n_units) * C::kBM) return;
  const int col = static_cast<int>(gtid % tpr) * 4;
  const int u = static_cast<int>(rowid / C::kBM), r = static_cast<int>(rowid % C::kBM);
  const unsigned unit = geom.n_main + u;
  const int vh = unit % C::kVSplit;
  const unsigned rb = unit / C::kVSplit;
  const int bh = rb / geom.n_rtiles;
  const int rrow = (rb % geom.n_rtiles) * C::kBM + r;
  if (rrow >= geom.n_res) return;
  const int64_t off = (static_cast<int64_t>(bh) * geom.n_res + rrow) * geom.d + vh * C::kDV + col;
#pragma unroll 1
  for (int acc = 0; acc < (C::kDKDV ? 2 : 1); ++acc) {
    const float* part = acc == 0 ? geom.part1 : geom.part2;
    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c = 0; c < geom.split; ++c) {
      const float4 x = *reinterpret_cast<const float4*>(
          part + ((static_cast<int64_t>(u) * geom.split + c) * C::kBM + r) * C::kDV + col);
      sum.x += x.x;
      sum.y += x.y;
      sum.z += x.z;
      sum.w += x.w;
    }
    *reinterpret_cast<float4*>((acc == 0 ? geom.out1 : geom.out2) + off) = sum;
  }
}

cudaError_t make_map4(CUtensorMap* map, const void* ptr, int64_t d, int64_t rows, int64_t H, int64_t B,
                      int box_rows) {
  TensorMapEncodeFn enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  cuuint64_t gdim[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t gstr[3] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(rows * d) * 2,
                        static_cast<cuuint64_t>(H * rows * d) * 2};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(box_rows), 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), gdim, gstr, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// fp32 [BH, rows] vector map (row stride ``pitch`` floats, a multiple of 4),
// 64-element boxes; rows past the end read as zero.
cudaError_t make_vec_map(CUtensorMap* map, const float* ptr, int64_t rows, int64_t pitch, int64_t BH) {
  TensorMapEncodeFn enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  cuuint64_t gdim[2] = {static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(BH)};
  cuuint64_t gstr[1] = {static_cast<cuuint64_t>(pitch) * 4};
  cuuint32_t box[2] = {64, 1};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(ptr), gdim, gstr, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Registers per thread the kernel was compiled with (-1 if unknown); looked up once.
template <int D, int kMode, bool kCut>
int compiled_regs() {
  static const int regs = [] {
    cudaFuncAttributes fa;
    return cudaFuncGetAttributes(&fa, attn_bwd_kernel<D, kMode, kCut>) == cudaSuccess ? fa.numRegs : -1;
  }();
  return regs;
}

template <int D, int kMode>
cudaError_t launch_pass(const BwdArgs& a, const float* nl2, const float* nd, const char** msg) {
  using C = BwdCfg<D, kMode>;
  const bool dkdv = kMode == kModeDKDV;
  BwdMaps maps;
  BwdGeom geom;
  const int64_t n_res = dkdv ? a.Nkv : a.Nq, n_str = dkdv ? a.Nq : a.Nkv;
  // Resident: dQ pass Q, dO; dK/dV pass K, V.  Streamed: dQ pass K, V; dK/dV pass Q, dO.
  const void* r1 = dkdv ? a.k : a.q;
  const void* r2 = dkdv ? a.v : a.dout;
  const void* x1 = dkdv ? a.q : a.k;
  const void* x2 = dkdv ? a.dout : a.v;
  cudaError_t e = make_map4(&maps.r1, r1, a.d, n_res, a.H, a.B, C::kBM);
  if (e == cudaSuccess) e = make_map4(&maps.r2, r2, a.d, n_res, a.H, a.B, C::kBM);
  if (e == cudaSuccess) e = make_map4(&maps.x1, x1, a.d, n_str, a.H, a.B, C::kBN);
  if (e == cudaSuccess) e = make_map4(&maps.x2, x2, a.d, n_str, a.H, a.B, C::kBN);
  const int64_t nq_pad = (a.Nq + 3) / 4 * 4;
  if (e == cudaSuccess && dkdv) e = make_vec_map(&maps.nl2, nl2, a.Nq, nq_pad, a.B * a.H);
  if (e == cudaSuccess && dkdv) e = make_vec_map(&maps.nd, nd, a.Nq, nq_pad, a.B * a.H);
  if (e != cudaSuccess) {
    *msg = "cuTensorMapEncodeTiled rejected a tensor (alignment or size)";
    return e;
  }
  if (!dkdv) {
    maps.nl2 = maps.r1;  // unused by the dQ pass
    maps.nd = maps.r1;
  }
  // A short last wave is cut into pieces over the streamed rows (the forward's
  // rule), whose partial sums a second kernel adds.
  const int n_rtiles = static_cast<int>((n_res + C::kBM - 1) / C::kBM);
  const int64_t grid = static_cast<int64_t>(n_rtiles) * a.B * a.H * C::kVSplit;
  const int n_sm = device_sm_count();
  const int64_t split = last_wave_split(grid, n_str, n_sm);
  auto kern = split > 1 ? attn_bwd_kernel<D, kMode, true> : attn_bwd_kernel<D, kMode, false>;
  // The warpgroups' register split must fit the pool the block launches with
  // (see kRegsIssue); a smaller compiled count would leave setmaxnreg.inc waiting.
  const int regs = split > 1 ? compiled_regs<D, kMode, true>() : compiled_regs<D, kMode, false>();
  if (regs * kThreads < kRegPoolNeeded) {
    *msg = "backward kernel compiled with fewer registers than its warpgroup split needs";
    return cudaErrorInvalidConfiguration;
  }
  bool first = false;
  e = ensure_smem_limit(reinterpret_cast<const void*>(kern), C::kSmemBytes, &first);
  if (e != cudaSuccess) {
    *msg = "cudaFuncSetAttribute(max dynamic shared memory) failed";
    return e;
  }
  geom.H = static_cast<int>(a.H);
  geom.n_rtiles = n_rtiles;
  geom.n_res = static_cast<int>(n_res);
  geom.n_str = static_cast<int>(n_str);
  geom.nq_pad = static_cast<int>(nq_pad);
  geom.d = static_cast<int>(a.d);
  geom.scale = a.scale;
  geom.row_nl2 = nl2;
  geom.row_nd = nd;
  geom.out1 = dkdv ? a.dv : a.dq;
  geom.out2 = dkdv ? a.dk : nullptr;
  const int64_t tail = split > 1 ? grid % n_sm : 0;
  geom.n_main = static_cast<int>(grid - tail);
  geom.split = static_cast<int>(split);
  geom.part1 = geom.part2 = nullptr;
  void* ws = nullptr;
  if (split > 1) {
    const int64_t nt = (n_str + C::kBN - 1) / C::kBN;
    for (int c = 0; c <= split; ++c) geom.piece_t[c] = static_cast<int>(c * nt / split);
    const int64_t slot_floats = tail * split * C::kBM * C::kDV;
    e = piece_alloc(&ws, static_cast<size_t>(slot_floats) * (dkdv ? 2 : 1) * sizeof(float), a.stream);
    if (e != cudaSuccess) {
      *msg = "stream-ordered allocation of the last wave's partial sums failed";
      return e;
    }
    geom.part1 = static_cast<float*>(ws);
    geom.part2 = dkdv ? geom.part1 + slot_floats : nullptr;
  }
  const int64_t launched = geom.n_main + tail * split;
  kern<<<static_cast<unsigned>(launched), kThreads, C::kSmemBytes, a.stream>>>(maps, geom, a.status);
  e = cudaGetLastError();
  if (e != cudaSuccess) *msg = "attention-backward kernel launch failed";
  if (ws) {
    if (e == cudaSuccess) {
      const int ncols = C::kDV == 128 ? C::kDV : static_cast<int>(a.d);
      const int64_t threads = tail * C::kBM * (ncols / 4);
      bwd_merge_pieces_kernel<C><<<static_cast<unsigned>((threads + 255) / 256), 256, 0, a.stream>>>(
          geom, static_cast<int>(tail), ncols);
      e = cudaGetLastError();
      if (e != cudaSuccess) *msg = "merge of the backward's last-wave pieces failed to launch";
    }
    const cudaError_t f = cudaFreeAsync(ws, a.stream);
    if (e == cudaSuccess && f != cudaSuccess) {
      *msg = "stream-ordered release of the last wave's partial sums failed";
      e = f;
    }
  }
  return e;
}

int64_t vec_floats(int64_t B, int64_t H, int64_t Nq) { return ((B * H * ((Nq + 3) / 4 * 4)) + 63) / 64 * 64; }

template <int D>
cudaError_t launch_bwd_d(const BwdArgs& a, const char** msg) {
  const int64_t rows = a.B * a.H * a.Nq;
  float* nl2 = a.ws;
  float* nd = a.ws + vec_floats(a.B, a.H, a.Nq);
  bwd_prep_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, a.stream>>>(
      static_cast<const __nv_bfloat16*>(a.dout), a.out, a.lse, nl2, nd, rows, a.Nq, (a.Nq + 3) / 4 * 4,
      static_cast<int>(a.d));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    *msg = "backward preprocessing launch failed";
    return e;
  }
  e = launch_pass<D, kModeDKDV>(a, nl2, nd, msg);
  if (e == cudaSuccess) e = launch_pass<D, kModeDQ>(a, nl2, nd, msg);
  return e;
}

}  // namespace

int64_t attn_bwd_workspace_floats(int64_t B, int64_t H, int64_t Nq) { return 2 * vec_floats(B, H, Nq); }

cudaError_t launch_attn_bwd(const BwdArgs& a, const char** msg) {
  if (a.d == 256) return launch_bwd_d<256>(a, msg);
  if (a.d == 128) return launch_bwd_d<128>(a, msg);
  if (a.d == 16 || a.d == 32 || a.d == 64) return launch_bwd_d<64>(a, msg);
  *msg = "unsupported head dimension";
  return cudaErrorInvalidValue;
}

}  // namespace attnjvp
