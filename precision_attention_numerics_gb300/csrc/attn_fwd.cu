// Causal FP8 (E4M3) attention forward on tcgen05 tensor cores.
//
// Method ("attention-numerics" project page, method and kernel settings;
// "Technische Samenvatting: P-Cast Precisie in FP8 Attention", sec. 1):
// per query row, KV tiles of width T are visited forward (0 -> diagonal) or
// reverse (diagonal -> 0); per tile
//   t_j = (q8 . k8_j) * c,  m' = max(m, max_j t_j),  alpha = 2^(m - m'),
//   P_j = 2^(t_j - m'),  l = alpha*l + sum_j P_j,  p8_j = E4M3(P_j * S),
//   O_acc = alpha*O_acc + sum_j p8_j v8_j;   O = O_acc * dv / (S * l).
// The running maximum is exact; O is rescaled whenever alpha != 1 (a
// skipped rescale with alpha == 1 is exact).
// Arithmetic per score (two at a time with the packed f32x2 instructions):
// the row maximum is taken on the raw q8.k8 sums (scaling by c > 0 commutes
// with rounding and max) - on tiles without a masked key it comes with the S
// load itself (tcgen05.ld.red, sm_103a) - then P*S = 2^(fma(s, c, log2 S - m'))
// comes out of one ex2, and the row sum accumulates P*S (= S*l, divided out
// at the end).
//
// Work unit: one 128-row query tile of two query heads that share a KV head
// (GQA); both use the same K/V tiles and the same KV range.  A persistent
// grid walks the units longest-first (query tiles nearest the end of the
// sequence have the most KV tiles), one unit per CTA per round, in rounds of
// alternating direction so that every CTA gets the same number of KV tiles.
//
// CTA = 384 threads:
//   warps 0-3  softmax warpgroup 0 (query head h0), TMEM lanes 0..127 = rows
//   warps 4-7  softmax warpgroup 1 (query head h0 + 1)
//   warps 8-11 control warpgroup (warp 11 only waits at the end)
//   warp 8     TMA producer: Q tiles once per unit (two buffers, so the next
//              unit's Q loads during this one, where shared memory allows),
//              K and V^T tiles through an NS-stage ring
//   warp 9     TMEM allocator; issues warpgroup 0's MMAs
//   warp 10    issues warpgroup 1's MMAs (each warpgroup's MMAs are in
//              order; the two streams do not wait for each other).  The MMA
//              warps run converged and let one elected lane issue: a lone
//              lane takes about twice as long per MMA.
// TMEM columns: S_w at [w*T, w*T+T), O_w at [2T + w*D, 2T + w*D + D).
// Shared memory: Q[QBUF buffers][2 warpgroups], P[2 warpgroups][2 buffers] (the
// E4M3 probabilities, written by the softmax threads in the 128-byte (or
// 64-byte) swizzled K-major layout the MMA reads; tile n of a warpgroup uses
// buffer n % 2, whose previous reader, P.V of tile n-2, is known complete),
// the K and V^T rings.
//
// Pipeline per warpgroup w and tile k:
//   MMA   S_w(k) = Q_w K(k)^T  (kind::f8f6f4, M=128, N=T, K=32 per instruction;
//         kind::f16 with K=16 for INT8 codes held in bf16)
//   SM    load S_w(k) from TMEM, then signal "S read"      -> MMA issues S_w(k+1)
//   SM    row max, alpha, P*S, E4M3 codes, row sum
//   SM    write P_w(k) to shared memory; only if some row's alpha != 1, wait
//         for O_w += P_w(k-1) V(k-1) and rescale O_w; signal "P ready"
//                                                          -> MMA issues O_w += P_w(k) V(k)
// P.V completions alternate between two barriers per warpgroup (product n
// on barrier n % 2), so the softmax waits only for the products it needs:
// product n-2 before reusing its P buffer, n-1 before a rescale.  "P ready"
// alternates the same way, because a warpgroup's warps drift apart by up to
// one tile.  S_w(k+1) and the P.V products thus run on the tensor core while
// the softmax warps compute.
//
// Every mbarrier wait is bounded; on a timeout the CTA records
// DEV_TIMEOUT, every role leaves its loop, outstanding TMA loads and MMAs are
// drained (again with a bound) and TMEM is freed before the CTA exits.
#include <cuda_bf16.h>

#include <cfloat>
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace attnq {
namespace {

constexpr int kRows = 128;
static_assert(kRows == kScaleTile, "a query tile is one scale tile");
constexpr int kThreads = 384;          // three warpgroups
constexpr int kProducerWarp = 8, kMmaWarp = 9;  // warps 9 and 10 issue the MMAs of warpgroups 0 and 1
// Register split: launched at 168 per thread (384 x 168 = 64,512); the two
// softmax warpgroups rise to 208, warpgroup 2 (producer, the two MMA warps,
// one idle warp) drops to 88: 2 x 128 x 208 + 128 x 88 = 64,512.
constexpr uint32_t kSoftmaxRegs = 208, kControlRegs = 88;
static_assert(2 * 128 * kSoftmaxRegs + 128 * kControlRegs <= kThreads * 168, "register split");
// Bound for draining in-flight copies and MMAs after an abort (independent of
// the wait limit, so an abort never leaves copies in flight).
constexpr uint64_t kDrainNs = 1000000000ull;

struct Params {
  int B, Hq, Hkv, N, G, pairs, n_qt, n_units;
  int paired;  // 1: the mirrored-pair schedule (unit_at), 0: alternating rounds of single units
  int causal, reverse;
  float S, log2S;
  const float* q_ds;
  const float* k_ds;
  const float* v_ds;
  int tiles;   // 1: q_ds and k_ds hold one descale per 128-token tile (n_st per slice)
  int n_st;    // scale tiles per slice
  double inv_sqrt_d, rot, log2e;
  void* O;
  int out_bf16;
  unsigned long long* uf;
  int k_sink;
  uint32_t* status;
  uint64_t wait_ns;
};

// I8: Q and K hold INT8 codes as bf16 (2 bytes an element) and S = Q K^T runs
// as kind::f16; P and V^T stay E4M3.
template <int D, int T, bool I8 = false>
struct Cfg {
  static constexpr int QE = I8 ? 2 : 1;      // bytes of a Q/K element
  static constexpr int QB = kRows * D * QE;  // bytes of one Q tile
  static constexpr int PB = kRows * T;       // bytes of one P tile
  static constexpr int KB = T * D * QE;      // bytes of one K stage
  static constexpr int VB = D * T;           // bytes of one V^T stage
  // Q buffers (units whose Q tiles are resident): two, so the next unit's Q
  // loads during this one, unless that leaves fewer than two K/V stages
  static constexpr int QBUF = (230400 - 4 * QB - 4 * PB) / (KB + VB) >= 2 ? 2 : 1;
  static constexpr int NS0 = (230400 - 2 * QBUF * QB - 4 * PB) / (KB + VB);
  static constexpr int NS = NS0 > 6 ? 6 : NS0;
  static constexpr int COLS_USED = 2 * T + 2 * D;
  static constexpr uint32_t TMEM_COLS = COLS_USED <= 256 ? 256u : 512u;
  // Q/K rows are D * QE bytes: 128-byte swizzle atoms side by side along K
  // (column blocks of rows x 128 bytes), or one 64-byte swizzled block for
  // 64-byte rows
  static constexpr uint32_t LAYOUT_QK = D * QE >= 128 ? 2u : 4u;  // 128B / 64B swizzle
  static constexpr uint32_t SBO_QK = D * QE >= 128 ? 1024u : 512u;
  static constexpr int QK_BLOCKS = D * QE >= 128 ? D * QE / 128 : 1;  // column blocks of a Q/K tile
  static constexpr int QK_BOX = D * QE >= 128 ? 128 : D * QE;         // bytes of a TMA box row
  static constexpr uint32_t LAYOUT_V = T == 128 ? 2u : 4u;    // V^T and P rows are T bytes
  static constexpr uint32_t SBO_V = 8u * T;
  static constexpr int NBARS = 4 + 4 * NS + 14 + 2;
  static constexpr size_t SMEM =
      1024 + 2 * QBUF * size_t(QB) + 4 * size_t(PB) + size_t(NS) * (KB + VB) + 8 * NBARS + 16;
  static_assert(COLS_USED <= 512, "TMEM budget");
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(NS >= 2, "pipeline depth");
};

struct Unit {
  int t, b, g, h0, nact, nt;
};

// Unit index (in decode_unit's numbering) of this CTA's k-th unit; p.n_units
// once the CTA has none left.  Two schedules, both handing the same KV-tile
// total to every CTA:
// * alternating rounds: units ordered longest first, one per CTA per round,
//   rounds of alternating direction (CTA i takes the i-th unit of an even
//   round and the i-th from the end of an odd one; a fixed stride would give
//   the CTAs with low indices the longer unit of every round);
// * mirrored pairs (causal, an even number of query tiles, many rounds): an
//   item is query tile n_qt-1-s followed by its mirror s of the same heads,
//   n_qt + 1 key tiles of 128 keys together, and items go one per CTA per
//   round in (batch, KV group)-major order.  The CTAs of a round then share
//   the K/V tiles of one or two KV groups, which stay in L2, where the
//   longest-first order keeps every group's K and V in use at once and reads
//   them from DRAM several times over.
__device__ __forceinline__ int unit_at(const Params& p, int k) {
  const int g = int(gridDim.x), i = int(blockIdx.x);
  if (!p.paired) return k * g + ((k & 1) ? g - 1 - i : i);
  const int half = p.n_qt / 2, per_grp = half * p.pairs;
  const int j = (k >> 1) * g + i;  // item
  if (j >= p.B * p.Hkv * per_grp) return p.n_units;
  const int grp = j / per_grp, rem = j % per_grp;  // grp = b * Hkv + kv group
  const int s = rem / p.pairs, pr = rem % p.pairs;
  const int t = (k & 1) ? s : p.n_qt - 1 - s;
  return (p.n_qt - 1 - t) * (p.B * p.Hkv * p.pairs) + grp * p.pairs + pr;
}

template <int T>
__device__ __forceinline__ Unit decode_unit(const Params& p, int u) {
  const int per_t = p.B * p.Hkv * p.pairs;
  Unit un;
  un.t = p.n_qt - 1 - u / per_t;
  int r = u % per_t;
  un.b = r / (p.Hkv * p.pairs);
  r %= p.Hkv * p.pairs;
  un.g = r / p.pairs;
  const int pr = r % p.pairs;
  un.h0 = un.g * p.G + 2 * pr;
  un.nact = (2 * pr + 1 < p.G) ? 2 : 1;
  const int last = min(un.t * kRows + kRows - 1, p.N - 1);
  un.nt = p.causal ? last / T + 1 : (p.N - 1) / T + 1;
  return un;
}

struct Bars {
  uint64_t* q_full;   // [2] (Q buffer)
  uint64_t* q_empty;  // [2]
  uint64_t* k_full;
  uint64_t* k_empty;
  uint64_t* v_full;
  uint64_t* v_empty;
  uint64_t* s_full;  // [2] S_w in TMEM (MMA commit)
  uint64_t* s_free;  // [2] S_w read by its warpgroup (128 arrivals)
  uint64_t* p_full;  // [2][2] P_w tile n written and O_w rescaled, on [w][n % 2] (128 arrivals)
  uint64_t* o_done;  // [2][2] O_w += P_w V of product n complete, on [w][n % 2] (MMA commit)
  uint64_t* o_free;  // [2] O_w read by the epilogue (128 arrivals)
  uint64_t* drain;
};

// Bounded wait that also gives up when another role has aborted.
// The thread sleeps inside try_wait (up to 20 us per try) instead of
// spinning, so waiting warps take few issue slots from the softmax warps.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, uint64_t limit_ns,
                                              volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  // suspend in try_wait for at most 20 us, and never longer than the limit
  const uint32_t hint = limit_ns < 20000ull ? uint32_t(limit_ns) : 20000u;
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, hint)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ void raise_abort(const Params& p, volatile int* abort_flag) {
  if (!*abort_flag) {
    *abort_flag = 1;
    atomicOr(p.status, DEV_TIMEOUT);
  }
}

// Warp-uniform wait.  Fast path: every lane tests the barrier and the warp
// votes (no divergence, no broadcast); otherwise lane 0 waits with the bound
// and the result is broadcast.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const Params& p,
                                          volatile int* abort_flag) {
  if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
  uint32_t ok = 0;
  if ((threadIdx.x & 31) == 0) ok = wait_or_abort(bar, parity, p.wait_ns, abort_flag) ? 1u : 0u;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  return ok != 0;
}

template <int D, int T, bool I8>
__device__ __forceinline__ void producer(const Params& p, const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                         uint8_t* sQ, uint8_t* sK, uint8_t* sV, const Bars& br, volatile int* abort_flag) {
  using C = Cfg<D, T, I8>;
  uint32_t it = 0, kc = 0, vc = 0;  // tiles walked, K and V loads issued
  // L2 priorities: K/V tiles are read again by the units of the other query
  // tiles of their head; a Q tile is read by its unit only
  const uint64_t keep = l2_evict_last_policy(), once = l2_evict_first_policy();
  int uc = 0;
  bool ok = true;
  bool q_issued = false;
  int q_last = 0;
  for (int k_r = 0, u = unit_at(p, 0); u < p.n_units && ok; u = unit_at(p, ++k_r), ++uc) {
    const Unit un = decode_unit<T>(p, u);
    const int qb = uc % C::QBUF;
    if (!wait_or_abort(br.q_empty + qb, ((uc / C::QBUF) & 1) ^ 1, p.wait_ns, abort_flag)) { ok = false; break; }
    uint8_t* q_dst = sQ + size_t(qb) * 2 * C::QB;
    mbar_arrive_expect_tx(br.q_full + qb, un.nact * C::QB);
#pragma unroll
    for (int cb = 0; cb < C::QK_BLOCKS; ++cb) {
      tma_load_3d_hint(q_dst + cb * (kRows * C::QK_BOX), tq, br.q_full + qb, cb * C::QK_BOX, un.t * kRows,
                       un.b * p.Hq + un.h0, once);
      if (un.nact == 2)
        tma_load_3d_hint(q_dst + C::QB + cb * (kRows * C::QK_BOX), tq, br.q_full + qb, cb * C::QK_BOX,
                         un.t * kRows, un.b * p.Hq + un.h0 + 1, once);
    }
    q_issued = true;
    q_last = uc;
    const int zkv = un.b * p.Hkv + un.g;
    for (int k = 0; k < un.nt; ++k, ++it) {
      const int jt = p.reverse ? un.nt - 1 - k : k;
      const int s = int(it % C::NS);
      const uint32_t ph = (it / C::NS) & 1u;
      if (!wait_or_abort(br.k_empty + s, ph ^ 1u, p.wait_ns, abort_flag)) { ok = false; break; }
      mbar_arrive_expect_tx(br.k_full + s, C::KB);
#pragma unroll
      for (int cb = 0; cb < C::QK_BLOCKS; ++cb)
        tma_load_3d_hint(sK + size_t(s) * C::KB + cb * (T * C::QK_BOX), tk, br.k_full + s, cb * C::QK_BOX, jt * T,
                         zkv, keep);
      ++kc;
      if (!wait_or_abort(br.v_empty + s, ph ^ 1u, p.wait_ns, abort_flag)) { ok = false; break; }
      mbar_arrive_expect_tx(br.v_full + s, C::VB);
      tma_load_3d_hint(sV + size_t(s) * C::VB, tv, br.v_full + s, jt * T, 0, zkv, keep);
      ++vc;
    }
  }
  if (!ok) {
    raise_abort(p, abort_flag);
    // Drain: wait for every load still in flight (its barrier phase completes
    // when the bytes land), bounded by the same limit.
    const uint64_t limit = kDrainNs;
    volatile int no_abort = 0;
    if (q_issued) {
      // the last QBUF Q loads may still be in flight
      for (int x = q_last; x >= 0 && x > q_last - C::QBUF; --x)
        wait_or_abort(br.q_full + (x % C::QBUF), (x / C::QBUF) & 1, limit, &no_abort);
    }
    for (uint32_t x = 0; x < uint32_t(C::NS); ++x) {
      if (x < kc) {
        const uint32_t last = kc - 1 - x;
        wait_or_abort(br.k_full + last % C::NS, (last / C::NS) & 1u, limit, &no_abort);
      }
      if (x < vc) {
        const uint32_t last = vc - 1 - x;
        wait_or_abort(br.v_full + last % C::NS, (last / C::NS) & 1u, limit, &no_abort);
      }
    }
  }
}

// Wait for a converged warp: every lane waits (they sleep in try_wait) and
// the result is voted, so the warp leaves converged.
__device__ __forceinline__ bool vote_wait(uint64_t* bar, uint32_t parity, const Params& p, volatile int* abort_flag) {
  const bool ok = wait_or_abort(bar, parity, p.wait_ns, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// Position in the K/V stage ring: stage s, and the parity of its current use.
struct Ring {
  uint32_t s, ph;
  __device__ __forceinline__ void next(uint32_t ns) {
    if (++s == ns) {
      s = 0;
      ph ^= 1u;
    }
  }
};

// Issues the MMAs of warpgroup w.  Run by a whole, converged warp: waits are
// voted, the elected lane issues each MMA and commit, and the shared
// memory descriptors are built from a low word stepped by (byte offset >> 4)
// in its start address field (every address stays below 256 KB, so the field
// never carries) and a constant high word.
// K/V stage and Q buffer barriers take one arrival from each of the two
// issuing warps (a commit when the warp's warpgroup used them, a plain arrive
// when it sat the unit out).
template <int D, int T, bool I8>
__device__ __forceinline__ void mma_issuer(const Params& p, int w, uint32_t tmem, uint8_t* sQ, uint8_t* sP,
                                           uint8_t* sK, uint8_t* sV, const Bars& br, volatile int* abort_flag) {
  using C = Cfg<D, T, I8>;
  constexpr uint32_t idS = I8 ? idesc_bf16_f32(kRows, T) : idesc_e4m3_f32(kRows, T);
  constexpr uint32_t idO = idesc_e4m3_f32(kRows, D);
  // descriptor = {start address field (low word), constant high word}
  const uint32_t hQK = uint32_t(smem_desc(0, 16, C::SBO_QK, C::LAYOUT_QK) >> 32);
  const uint32_t hV = uint32_t(smem_desc(0, 16, C::SBO_V, C::LAYOUT_V) >> 32);
  const uint32_t lQ0 = uint32_t(smem_desc(smem_u32(sQ) + uint32_t(w * C::QB), 16, C::SBO_QK, C::LAYOUT_QK));
  const uint32_t lK0 = uint32_t(smem_desc(smem_u32(sK), 16, C::SBO_QK, C::LAYOUT_QK));
  const uint32_t lP0 = uint32_t(smem_desc(smem_u32(sP) + uint32_t(2 * w * C::PB), 16, C::SBO_V, C::LAYOUT_V));
  const uint32_t lV0 = uint32_t(smem_desc(smem_u32(sV), 16, C::SBO_V, C::LAYOUT_V));
  const uint32_t tS = tmem + uint32_t(w * T), tO = tmem + uint32_t(2 * T + w * D);
  Ring rk{0u, 0u}, rv{0u, 0u};  // next K stage for an S product, next V stage for a P.V product
  int uc = 0;
  uint32_t n_s = 0;  // S products issued (whole kernel)
  uint32_t pc = 0;   // P.V products issued (whole kernel)
  uint32_t act = 0;  // units this warpgroup took part in (one o_free phase each)
  bool ok = true;
  bool issued_any = false;

  // S_w = Q_w K^T from K stage rk.s; the previous S_w must have been read by
  // the warpgroup.  Releases the K stage when the product completes.
  auto issue_S = [&](uint32_t lq) -> bool {
    if (!vote_wait(br.k_full + rk.s, rk.ph, p, abort_flag)) return false;
    if (n_s > 0 && !vote_wait(br.s_free + w, (n_s - 1) & 1u, p, abort_flag)) return false;
    ++n_s;
    tc_fence_after();
    const uint32_t lk = lK0 + rk.s * uint32_t(C::KB >> 4);
    if constexpr (I8) {
      // K steps of 16 bf16 (32 bytes): four per 128-byte column block, then
      // the next block (rows x 128 bytes further on)
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t cb = uint32_t(kk >> 2), sub = uint32_t(2 * (kk & 3));
        mma_f16_ss_elect(tS, pack_desc(lq + cb * uint32_t(kRows * 8) + sub, hQK),
                         pack_desc(lk + cb * uint32_t(T * 8) + sub, hQK), idS, kk > 0 ? 1u : 0u);
      }
    } else {
#pragma unroll
      for (int kk = 0; kk < D / 32; ++kk)
        mma_f8_ss_elect(tS, pack_desc(lq + 2 * kk, hQK), pack_desc(lk + 2 * kk, hQK), idS, kk > 0 ? 1u : 0u);
    }
    mma_commit_elect(br.s_full + w);
    mma_commit_elect(br.k_empty + rk.s);
    rk.next(C::NS);
    issued_any = true;
    return true;
  };

  for (int k_r = 0, u = unit_at(p, 0); u < p.n_units && ok; u = unit_at(p, ++k_r), ++uc) {
    const Unit un = decode_unit<T>(p, u);
    const int qb = uc % C::QBUF;
    if (!vote_wait(br.q_full + qb, (uc / C::QBUF) & 1, p, abort_flag)) { ok = false; break; }
    tc_fence_after();
    if (w >= un.nact) {
      // this warpgroup sits the unit out: release each stage and the Q buffer
      for (int k = 0; k < un.nt && ok; ++k) {
        if (!vote_wait(br.k_full + rk.s, rk.ph, p, abort_flag)) { ok = false; break; }
        mbar_arrive_elect(br.k_empty + rk.s);
        rk.next(C::NS);
        if (!vote_wait(br.v_full + rv.s, rv.ph, p, abort_flag)) { ok = false; break; }
        mbar_arrive_elect(br.v_empty + rv.s);
        rv.next(C::NS);
      }
      mbar_arrive_elect(br.q_empty + qb);
      continue;
    }
    const uint32_t lq = lQ0 + uint32_t(qb * (2 * C::QB >> 4));
    if (!issue_S(lq)) { ok = false; break; }
    if (un.nt == 1) mma_commit_elect(br.q_empty + qb);
    for (int k = 0; k < un.nt && ok; ++k) {
      if (k + 1 < un.nt) {
        if (!issue_S(lq)) { ok = false; break; }
        if (k + 1 == un.nt - 1) mma_commit_elect(br.q_empty + qb);
      }
      if (!vote_wait(br.v_full + rv.s, rv.ph, p, abort_flag)) { ok = false; break; }
      // O_w is overwritten by the unit's first product: the epilogue of the
      // warpgroup's previous unit must have read it
      if (k == 0 && !vote_wait(br.o_free + w, (act & 1u) ^ 1u, p, abort_flag)) { ok = false; break; }
      if (!vote_wait(br.p_full + 2 * w + (pc & 1u), (pc >> 1) & 1u, p, abort_flag)) { ok = false; break; }
      tc_fence_after();
      const uint32_t lp = lP0 + (pc & 1u) * uint32_t(C::PB >> 4);
      const uint32_t lv = lV0 + rv.s * uint32_t(C::VB >> 4);
#pragma unroll
      for (int kk = 0; kk < T / 32; ++kk)
        mma_f8_ss_elect(tO, pack_desc(lp + 2 * kk, hV), pack_desc(lv + 2 * kk, hV), idO, (k > 0 || kk > 0) ? 1u : 0u);
      mma_commit_elect(br.o_done + 2 * w + (pc & 1u));
      ++pc;
      mma_commit_elect(br.v_empty + rv.s);
      rv.next(C::NS);
    }
    ++act;
  }
  if (!ok) {
    if ((threadIdx.x & 31) == 0) raise_abort(p, abort_flag);
    if (issued_any) {
      volatile int no_abort = 0;
      mma_commit_elect(br.drain + w);
      if ((threadIdx.x & 31) == 0) wait_or_abort(br.drain + w, 0, kDrainNs, &no_abort);
      __syncwarp();
    }
  }
}

// Byte offset of 16-byte chunk c of row r in a K-major tile whose rows are T
// bytes, in the swizzled layout TMA writes and the MMA reads (128-byte
// swizzle for T = 128: 8-row groups of 1024 bytes, chunk c ^ (r % 8); 64-byte
// swizzle for T = 64: 8-row groups of 512 bytes, chunk c ^ ((r % 8) / 2)).
template <int T>
__device__ __forceinline__ uint32_t p_tile_offset(int r, int c) {
  if constexpr (T == 128) {
    return uint32_t((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
  } else {
    return uint32_t((r >> 3) * 512 + (r & 7) * 64 + ((c ^ ((r & 7) >> 1)) << 4));
  }
}

template <int D, int T, bool COUNT, bool TILES>
__device__ __forceinline__ void softmax_wg(const Params& p, int w, uint32_t tmem, uint8_t* sP, const Bars& br,
                                           volatile int* abort_flag) {
  const int r = threadIdx.x & 127;           // row in the query tile = TMEM lane
  const int wq = (threadIdx.x >> 5) & 3;     // warp within the warpgroup
  const uint32_t lane_off = uint32_t(wq * 32) << 16;
  const uint32_t tS = tmem + lane_off + uint32_t(w * T);
  const uint32_t tO = tmem + lane_off + uint32_t(2 * T + w * D);
  uint8_t* my_p = sP + size_t(2 * w) * kRows * T;
  uint32_t sc = 0, np = 0;  // S tiles read, P tiles written (= P.V products requested)
  // wait for P.V product n of this warpgroup (barrier n % 2, its (n / 2)-th phase)
  auto wait_pv = [&](uint32_t n) -> bool {
    return warp_wait(br.o_done + 2 * w + (n & 1u), (n >> 1) & 1u, p, abort_flag);
  };
  bool ok = true;
  for (int k_r = 0, u = unit_at(p, 0); u < p.n_units && ok; u = unit_at(p, ++k_r)) {
    const Unit un = decode_unit<T>(p, u);
    if (w >= un.nact) continue;  // sits the unit out: no arrival on o_free (its warps would not be in step)
    const int h = un.h0 + w;
    const int bh = un.b * p.Hq + h, bg = un.b * p.Hkv + un.g;
    // logit factor c = fl32(cq * dk), cq = fl32(dq * (1/sqrt d) * rot * log2 e)
    // in double once per unit; with per-tile scales dq is the query tile's and
    // dk the key tile's (one fp32 multiply per key tile, its descale loaded a
    // tile ahead)
    const double dq = double(TILES ? p.q_ds[int64_t(bh) * p.n_st + un.t] : p.q_ds[bh]);
    const float cq = __double2float_rn(__dmul_rn(__dmul_rn(__dmul_rn(dq, p.inv_sqrt_d), p.rot), p.log2e));
    const float* kd = TILES ? p.k_ds + int64_t(bg) * p.n_st : p.k_ds + bg;
    auto key_scale_tile = [&](int k) { return ((p.reverse ? un.nt - 1 - k : k) * T) / kScaleTile; };
    // A factor below the smallest normal float (Q and K descales near 1e-20
    // or less) makes every logit smaller than 2^-100 (|s| < 2^25), so every P is 1 in fp32
    // either way; raising c to FLT_MIN there changes no P and keeps the
    // masked keys' -inf * c at -inf (0 * -inf would be NaN).
    float c = fmaxf(__fmul_rn(cq, kd[TILES ? key_scale_tile(0) : 0]), FLT_MIN);
    float dk_next = 0.0f;
    if constexpr (TILES) {
      if (un.nt > 1) dk_next = kd[key_scale_tile(1)];
    }
    uint64_t c2 = pack2(c, c);
    const int i = un.t * kRows + r;
    float m = -INFINITY, l = 0.0f;
    uint32_t uf0 = 0, uf1 = 0;
    for (int k = 0; k < un.nt; ++k) {
      const int jt = p.reverse ? un.nt - 1 - k : k;
      const int j0 = jt * T;
      if (!warp_wait(br.s_full + w, sc & 1u, p, abort_flag)) { ok = false; break; }
      ++sc;
      tc_fence_after();
      if constexpr (TILES) {
        if (k > 0) {
          c = fmaxf(__fmul_rn(cq, dk_next), FLT_MIN);
          c2 = pack2(c, c);
          if (k + 1 < un.nt) dk_next = kd[key_scale_tile(k + 1)];
        }
      }
      const bool need_mask = (p.causal && j0 + T - 1 > un.t * kRows) || (j0 + T > p.N);
      // keys j0 + j are visible for j < lim (causal: j0 + j <= i; always j0 + j < N)
      const int lim = need_mask ? min(p.N - j0, p.causal ? i - j0 + 1 : T) : T;
      constexpr int H = T / 2;
      float sv[T];
      float smax;
      if (!need_mask) {
        // No key of the tile is masked: tcgen05.ld.red returns the maximum of
        // each 32-column load with the values, so the row max is the maximum
        // of T/32 numbers (the same value the software chains give).
        float hm[T / 32];
#pragma unroll
        for (int q = 0; q < T / 32; ++q)
          tmem_ld32f_max(tS + uint32_t(32 * q), *reinterpret_cast<float(*)[32]>(&sv[32 * q]), hm[q]);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < T / 32; ++q) reg_fence32(*reinterpret_cast<float(*)[32]>(&sv[32 * q]));
        // S_w is in registers: the MMA warp may overwrite it with the next tile
        tc_fence_before();
        mbar_arrive(br.s_free + w);
        smax = hm[0];
#pragma unroll
        for (int q = 1; q < T / 32; ++q) smax = fmaxf(smax, hm[q]);
      } else {
        // Diagonal or ragged tile: masked keys must not enter the maximum, so
        // S comes in two halves and the row max of the masked first half runs
        // while the second half is still on its way out of TMEM.
#pragma unroll
        for (int q = 0; q < H / 32; ++q) tmem_ld32f(tS + uint32_t(32 * q), *reinterpret_cast<float(*)[32]>(&sv[32 * q]));
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < H / 32; ++q) reg_fence32(*reinterpret_cast<float(*)[32]>(&sv[32 * q]));
#pragma unroll
        for (int q = H / 32; q < T / 32; ++q) tmem_ld32f(tS + uint32_t(32 * q), *reinterpret_cast<float(*)[32]>(&sv[32 * q]));
#pragma unroll
        for (int j = 0; j < H; ++j) sv[j] = (j < lim) ? sv[j] : -INFINITY;
        // row max of the raw sums (fl32(s * c) is monotone in s for c > 0):
        // eight independent two-input chains (the three-input form measured slower)
        float mx[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mx[e] = sv[e];
#pragma unroll
        for (int j = 8; j < H; j += 8) {
#pragma unroll
          for (int e = 0; e < 8; ++e) mx[e] = fmaxf(mx[e], sv[j + e]);
        }
        tmem_wait_ld();
#pragma unroll
        for (int q = H / 32; q < T / 32; ++q) reg_fence32(*reinterpret_cast<float(*)[32]>(&sv[32 * q]));
        tc_fence_before();
        mbar_arrive(br.s_free + w);
#pragma unroll
        for (int j = H; j < T; ++j) sv[j] = (j < lim) ? sv[j] : -INFINITY;
#pragma unroll
        for (int j = H; j < T; j += 8) {
#pragma unroll
          for (int e = 0; e < 8; ++e) mx[e] = fmaxf(mx[e], sv[j + e]);
        }
        smax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      }
      const float mt = (smax == -INFINITY) ? -INFINITY : __fmul_rn(smax, c);
      const float mnew = fmaxf(m, mt);
      const float muse = (mnew == -INFINITY) ? 0.0f : mnew;
      const float alpha = (mnew == -INFINITY) ? 1.0f : ex2(__fsub_rn(m, mnew));
      // P*S = 2^(s*c + (log2 S - m'))
      const float off = __fsub_rn(p.log2S, muse);
      const uint64_t off2 = pack2(off, off);
      uint64_t ls2[2] = {pack2(0.0f, 0.0f), pack2(0.0f, 0.0f)};
      // Codes go straight to P buffer np % 2, whose last reader was product
      // np - 2.  No wait is needed: the MMA warp issued P.V np - 2 before
      // S np, and the commit that signalled "S np complete" covers every
      // earlier tcgen05 operation of that warp.
      uint8_t* pbuf = my_p + size_t(np & 1u) * kRows * T;
#pragma unroll
      for (int cch = 0; cch < T / 16; ++cch) {
        uint32_t pw[4];
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          const int q = 4 * cch + qq;
          float PS[4];
          unpack2(ffma2(pack2(sv[4 * q], sv[4 * q + 1]), c2, off2), PS[0], PS[1]);
          unpack2(ffma2(pack2(sv[4 * q + 2], sv[4 * q + 3]), c2, off2), PS[2], PS[3]);
          // Without counters the flush-to-zero form is exact for the output: a
          // P*S below 2^-126 casts to the E4M3 code 0 either way, and its share
          // of the row sum is below fp32 resolution.  The counting build keeps
          // subnormal P*S, whose cast to 0 it must count.
#pragma unroll
          for (int e = 0; e < 4; ++e) PS[e] = COUNT ? ex2(PS[e]) : ex2_ftz(PS[e]);
          ls2[0] = fadd2(ls2[0], pack2(PS[0], PS[1]));
          ls2[1] = fadd2(ls2[1], pack2(PS[2], PS[3]));
          pw[qq] = pack_b16x2(cvt_e4m3x2(PS[0], PS[1]), cvt_e4m3x2(PS[2], PS[3]));
          if constexpr (COUNT) {
            if (i < p.N) {
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int jj = j0 + 4 * q + e;
                const uint32_t code = (pw[qq] >> (8 * e)) & 0xFFu;
                // P itself, 2^(fl(fl(s c) - m')) in fp32, is 0 once its exponent is
                // at most -150 (2^-150 rounds to 0); P*S formed in one step can
                // still be positive there, but P*S of a zero P is no underflow
                const bool p_pos = __fsub_rn(__fmul_rn(sv[4 * q + e], c), muse) > -150.0f;
                if (PS[e] > 0.0f && p_pos && code == 0u && jj >= p.k_sink) {
                  if (jt == 0) ++uf0;
                  else ++uf1;
                }
              }
            }
          }
        }
        *reinterpret_cast<uint4*>(pbuf + p_tile_offset<T>(r, cch)) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
      }
      ++np;
      float la, lb, lc, ld;
      unpack2(ls2[0], la, lb);
      unpack2(ls2[1], lc, ld);
      l = __fadd_rn(__fmul_rn(alpha, l), __fadd_rn(__fadd_rn(la, lb), __fadd_rn(lc, ld)));
      if (k > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
        // O_w += P_w(k-1) V(k-1) (product np - 2 now) must be complete before
        // O_w is rescaled; rows with alpha == 1 are multiplied by 1 (exact).
        if (!wait_pv(np - 2)) { ok = false; break; }
        tc_fence_after();
        const uint64_t a2 = pack2(alpha, alpha);
        // all D columns of the row in one round trip (the scores are dead here)
        uint32_t o[D];
#pragma unroll
        for (int q = 0; q < D / 32; ++q) tmem_ld32(tO + uint32_t(32 * q), *reinterpret_cast<uint32_t(*)[32]>(&o[32 * q]));
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < D / 32; ++q) reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&o[32 * q]));
#pragma unroll
        for (int e = 0; e < D; e += 2) {
          float x0, x1;
          unpack2(fmul2(pack2(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), a2), x0, x1);
          o[e] = __float_as_uint(x0);
          o[e + 1] = __float_as_uint(x1);
        }
#pragma unroll
        for (int q = 0; q < D / 32; ++q) tmem_st32(tO + uint32_t(32 * q), *reinterpret_cast<uint32_t(*)[32]>(&o[32 * q]));
        tmem_wait_st();
      }
      // The warps of a warpgroup are not in step: a warp may write P(n+1) and
      // arrive while another is still on P(n).  Alternating barriers keep
      // those arrivals apart (none can reach P(n+2) before P.V(n) is done).
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(br.p_full + 2 * w + ((np - 1) & 1u));
      m = mnew;
    }
    if (!ok) break;
    // epilogue: O = acc * dv / (S * l); the running sum already holds S * l
    if (!wait_pv(np - 1)) { ok = false; break; }
    tc_fence_after();
    const float scale = __fdiv_rn(p.v_ds[bg], l);
#pragma unroll 1
    for (int q = 0; q < D / 32; ++q) {
      uint32_t o[32];
      tmem_ld32(tO + uint32_t(32 * q), o);
      tmem_wait_ld();
      reg_fence32(o);
      if (i < p.N) {
        const int64_t off = (int64_t(bh) * p.N + i) * D + 32 * q;
        // O is written once: streaming stores (evict first)
        if (p.out_bf16) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.O) + off);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t wv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __nv_bfloat162 b2 = __floats2bfloat162_rn(__fmul_rn(__uint_as_float(o[8 * v + 2 * e]), scale),
                                                              __fmul_rn(__uint_as_float(o[8 * v + 2 * e + 1]), scale));
              wv[e] = *reinterpret_cast<const uint32_t*>(&b2);
            }
            __stcs(dst + v, make_uint4(wv[0], wv[1], wv[2], wv[3]));
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.O) + off);
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            __stcs(dst + v, make_float4(__fmul_rn(__uint_as_float(o[4 * v]), scale),
                                        __fmul_rn(__uint_as_float(o[4 * v + 1]), scale),
                                        __fmul_rn(__uint_as_float(o[4 * v + 2]), scale),
                                        __fmul_rn(__uint_as_float(o[4 * v + 3]), scale)));
          }
        }
      }
    }
    tc_fence_before();
    mbar_arrive(br.o_free + w);
    if constexpr (COUNT) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        uf0 += __shfl_xor_sync(0xffffffffu, uf0, o);
        uf1 += __shfl_xor_sync(0xffffffffu, uf1, o);
      }
      if ((threadIdx.x & 31) == 0) {
        if (uf0) atomicAdd(p.uf + 2 * bh, (unsigned long long)uf0);
        if (uf1) atomicAdd(p.uf + 2 * bh + 1, (unsigned long long)uf1);
      }
    }
  }
  if (!ok) raise_abort(p, abort_flag);
}

template <int D, int T, bool COUNT, bool TILES, bool I8>
__global__ void __launch_bounds__(kThreads, 1)
    k_attn_fwd(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
               const __grid_constant__ CUtensorMap tv, const Params p) {
  using C = Cfg<D, T, I8>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base by pointer arithmetic on the shared array (an
  // integer round trip would hide the address space and make every access
  // through it a generic one)
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sQ = sm;                          // [Q buffer][warpgroup]
  uint8_t* sP = sQ + 2 * C::QBUF * C::QB;    // [warpgroup][P buffer]
  uint8_t* sK = sP + 4 * C::PB;
  uint8_t* sV = sK + size_t(C::NS) * C::KB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + size_t(C::NS) * C::VB);
  Bars br;
  br.q_full = bars;
  br.q_empty = bars + 2;
  br.k_full = bars + 4;
  br.k_empty = br.k_full + C::NS;
  br.v_full = br.k_empty + C::NS;
  br.v_empty = br.v_full + C::NS;
  br.s_full = br.v_empty + C::NS;
  br.s_free = br.s_full + 2;
  br.p_full = br.s_free + 2;
  br.o_done = br.p_full + 4;
  br.o_free = br.o_done + 4;
  br.drain = br.o_free + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(br.drain + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(br.q_full + b, 1);
      mbar_init(br.q_empty + b, 2);
    }
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(br.k_full + s, 1);
      mbar_init(br.k_empty + s, 2);
      mbar_init(br.v_full + s, 1);
      mbar_init(br.v_empty + s, 2);
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(br.s_full + w, 1);
      mbar_init(br.s_free + w, 128);
      mbar_init(br.p_full + 2 * w, 128);
      mbar_init(br.p_full + 2 * w + 1, 128);
      mbar_init(br.o_done + 2 * w, 1);
      mbar_init(br.o_done + 2 * w + 1, 1);
      mbar_init(br.o_free + w, 128);
      mbar_init(br.drain + w, 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_holder, C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp >= 8) {
    regs_decrease<kControlRegs>();
    if (warp == kProducerWarp) {
      if (lane == 0) producer<D, T, I8>(p, &tq, &tk, &tv, sQ, sK, sV, br, abort_flag);
    } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
      mma_issuer<D, T, I8>(p, warp - kMmaWarp, tmem, sQ, sP, sK, sV, br, abort_flag);
    }
  } else {
    regs_increase<kSoftmaxRegs>();
    softmax_wg<D, T, COUNT, TILES>(p, warp >> 2, tmem, sP, br, abort_flag);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, int T, bool COUNT, bool TILES, bool I8>
cudaError_t run(const FwdArgs& a, cudaStream_t st) {
  using C = Cfg<D, T, I8>;
  CUtensorMap tq, tk, tv;
  const CUtensorMapSwizzle swqk = C::LAYOUT_QK == 2u ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  const CUtensorMapSwizzle swv = T == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  const uint64_t rq = uint64_t(D) * C::QE;  // bytes of a Q/K row
  if (encode_tiled_3d(&tq, a.q8, rq, a.N, uint64_t(a.B) * a.Hq, rq, uint64_t(a.N) * rq, C::QK_BOX, kRows, swqk) !=
      CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  if (encode_tiled_3d(&tk, a.k8, rq, a.N, uint64_t(a.B) * a.Hkv, rq, uint64_t(a.N) * rq, C::QK_BOX, T, swqk) !=
      CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  if (encode_tiled_3d(&tv, a.v8t, uint64_t(a.ldv), D, uint64_t(a.B) * a.Hkv, uint64_t(a.ldv), uint64_t(a.ldv) * D, T,
                      D, swv) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  Params p;
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.N = a.N;
  p.G = a.Hq / a.Hkv;
  p.pairs = (p.G + 1) / 2;
  p.n_qt = (a.N + kRows - 1) / kRows;
  p.n_units = p.n_qt * a.B * a.Hkv * p.pairs;
  p.causal = a.causal;
  p.reverse = a.reverse;
  p.S = a.S;
  p.log2S = float(std::log2(double(a.S)));
  p.q_ds = a.q_ds;
  p.k_ds = a.k_ds;
  p.v_ds = a.v_ds;
  p.tiles = a.tiles;
  p.n_st = (a.N + kScaleTile - 1) / kScaleTile;
  p.inv_sqrt_d = 1.0 / std::sqrt(double(D));
  p.rot = a.rotate ? 1.0 / double(D) : 1.0;
  p.log2e = 1.4426950408889634073599246810018921;
  p.O = a.O;
  p.out_bf16 = a.out_bf16;
  p.uf = a.underflow;
  p.k_sink = a.k_sink;
  p.status = a.status;
  p.wait_ns = a.wait_ns;
  auto kern = k_attn_fwd<D, T, COUNT, TILES, I8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(C::SMEM));
  if (e != cudaSuccess) return e;
  const int grid = p.n_units < a.num_sms ? p.n_units : a.num_sms;
  // mirrored pairs where every CTA gets the same number of items to within
  // 1 % (the last round nearly full) over at least four rounds
  {
    const int64_t items = int64_t(p.n_units) / 2, rounds = (items + grid - 1) / grid;
    p.paired = (a.causal && p.n_qt % 2 == 0 && items >= 4 * int64_t(grid) && 100 * rounds * grid <= 101 * items) ? 1 : 0;
  }
  kern<<<grid, kThreads, C::SMEM, st>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

template <int D, int T, bool I8>
cudaError_t run_count(const FwdArgs& a, cudaStream_t st) {
  if (a.tiles) return a.underflow ? run<D, T, true, true, I8>(a, st) : run<D, T, false, true, I8>(a, st);
  return a.underflow ? run<D, T, true, false, I8>(a, st) : run<D, T, false, false, I8>(a, st);
}

template <int D, int T>
cudaError_t run_format(const FwdArgs& a, cudaStream_t st) {
  return a.i8 ? run_count<D, T, true>(a, st) : run_count<D, T, false>(a, st);
}

}  // namespace

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t s) {
  if (a.d == 128) return a.T == 128 ? run_format<128, 128>(a, s) : run_format<128, 64>(a, s);
  return a.T == 128 ? run_format<64, 128>(a, s) : run_format<64, 64>(a, s);
}

}  // namespace attnq
