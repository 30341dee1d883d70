// Operand preparation ("attention-numerics" project page, method and kernel
// settings; "A rounding problem, not a rotation problem", 01 / Synthetic
// illustration):
//   mean key (K, optional) -> sign flip + unnormalised FWHT (Q, K, optional)
//   -> per-(batch, head) amax -> qs = 448/amax -> E4M3 RNE-satfinite cast.
//
// Bit-exactness: every float operation is a single IEEE add, subtract,
// multiply or divide in a fixed order (subtractions are fma(b, -1, a), which
// rounds a - b once), the FWHT uses the fixed butterfly schedule h = 1, 2, ...,
// d/2, the max is order-free, and the mean follows the fixed chunk order
// (128-token chunk sums in token order, then the chunk sums in order).
//
// One persistent kernel does every pass.  The work is a list of entries, one
// per (pass, slice), where a slice is one (batch, head) of Q, K or V and the
// passes are M (mean-key chunk sums, K with centring), A (amax) and C (cast).
// An entry's slice is cut into items of a few 128-row tiles; CTAs claim items
// in list order with an atomic ticket.  The list puts each slice's A entry a
// few steps after its M entry and its C entry a few steps after its A entry,
// so a slice's second and third reads mostly come from L2, and a pass waits
// only on entries claimed before it (C tiles wait until every A tile of their
// slice has added its amax and count, then compute the scale themselves;
// centred K tiles wait for the mean, published by the warp that completes the
// slice's M tiles): the earliest unfinished item never waits, so the kernel
// cannot deadlock, and
// it needs no co-residency.
//
// Causal-prefix statistics (the "attention-numerics" page, limitations: full-
// sequence means and scales see future tokens): with P < N the M and A passes
// cover only the first P tokens of a slice (their later items are empty and
// skipped), the mean divides by P, and the C pass casts all N tokens with the
// prefix's scale, checking the later tokens for non-finite values itself.
// That form is its own instance, so the full-sequence kernel carries none of it.
//
// CTA: warp 8 claims items and streams their tiles into a ring of shared
// memory stages with TMA (128-byte swizzle, rows beyond N read as zero;
// warps 9-11 only complete its warpgroup for the register split);
// warps 0-3 and 4-7 are two consumer groups that take alternate tiles, one
// row per thread.  The consumer warps run independently (each waits on the
// stage, counts its own rows and stores them), so no barrier ties the warps
// of a group together.  A row of d values is held as d/2 packed pairs
// (x_j, x_{j+d/2}), so stages h = 1 .. d/4 of the FWHT are packed f32x2
// adds and subtracts and stage d/2 adds the two halves of each pair (the
// amax pass skips it: max(|a + b|, |a - b|) rounds to fl(|a| + |b|)).  Codes
// leave through a per-warp staging buffer by TMA store: 32 rows in the
// natural layout, or 32 tokens x d channels of V transposed.
#include <cuda_bf16.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace attnq {
namespace {

constexpr int kTR = 128;           // rows per tile = tokens per mean-key chunk
constexpr int kTilesPerItem = 16;  // tiles per claimed item
// The last kTailEntries entries of the list (cast entries: the list ends with
// the casts of the slices whose amax came last) are claimed in items of
// kTilesPerItem / kTailSplit tiles, so the CTAs run out of work within a few
// tiles of one another instead of within one 16-tile item.
constexpr uint32_t kTailEntries = 7, kTailSplit = 4;
constexpr int kGroups = 2;         // consumer groups (4 warps, one row per thread)
constexpr int kConsumerWarps = 4 * kGroups;
constexpr int kFlowThreads = 128 * (kGroups + 1);  // consumer warpgroups + a warpgroup whose first warp is the producer
// Register split: launched at the even share of the register file (168 per
// thread for 384 threads); the consumer warpgroups rise to hold a row of 128
// fp32 values and the FWHT's working set without spilling, the producer's
// warpgroup drops: 2 x 128 x 232 + 128 x 40 = 64,512.
constexpr uint32_t kLaunchRegs = (65536u / kFlowThreads) & ~7u;
constexpr uint32_t kConsumerRegs = kGroups == 2 ? 232 : 160, kProducerRegs = kGroups == 2 ? 40 : 32;
static_assert(kGroups * 128 * kConsumerRegs + 128 * kProducerRegs <= kFlowThreads * kLaunchRegs, "register split");
static_assert(kTR == kScaleTile, "a ring tile is one scale tile");
constexpr int kLagA = 4, kLagC = 7;  // least list steps from a K slice's M entry to its A entry; A to C
constexpr uint32_t KIND_M = 0u, KIND_A = 1u, KIND_C = 2u, KIND_DONE = 3u;
constexpr uint32_t CTL_TICKET = 0, CTL_ABORT = 1, CTL_ENTRIES = 2;

// I8: Q and K leave as INT8 codes held in bf16 (2 bytes a code), so a warp's
// staging buffer is twice as large and each warp keeps one of them.
template <int D, bool BF16, bool I8 = false>
struct FlowCfg {
  static constexpr int ES = BF16 ? 2 : 4;
  static constexpr int ROW_BYTES = D * ES;
  static constexpr int NB = ROW_BYTES / 128;      // 128-byte boxes per input row
  static constexpr int SB = kTR * ROW_BYTES;      // input stage
  static constexpr int WB = (I8 ? 64 : 32) * D;   // a consumer warp's staging buffer (32 rows of codes)
  static constexpr int NBUF = I8 ? 1 : 2;         // staging buffers per consumer warp
  static constexpr int NOB = I8 ? (2 * D) / 128 : 1;  // 128-byte boxes per row of bf16 codes
  static constexpr int NST0 = (225280 - NBUF * kConsumerWarps * WB - 8192) / SB;
  // A multiple of kGroups: tile n goes to stage n % NST and to group
  // n % kGroups, so every stage serves one group only and its phases are
  // consumed in order.  A stage shared by two groups would let a group whose
  // tile is k phases ahead mistake an older phase of the same parity for it.
  static constexpr int NST1 = NST0 > 6 ? 6 : NST0;
  static constexpr int NST = NST1 - NST1 % kGroups;
  static constexpr int WORDS = BF16 ? D / 2 : D;  // 32-bit input words per row
  static constexpr size_t SMEM = 1024 + size_t(NST) * SB + size_t(NBUF * kConsumerWarps) * WB + 16 * NST +
                                 16 * NST + 8 * WORDS + 8 * (D / 2) + kConsumerWarps * 8 * (D / 2) +
                                 4 * 4 * 2 * kGroups + 8 * 2 * kGroups;
  static_assert(NST >= kGroups && NST % kGroups == 0, "pipeline depth: whole stages per group");
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct TileMeta {
  uint32_t kind, slice, row0;
  uint32_t last;  // 1 on the last tile of its item that the consuming group gets
};

struct SliceRef {
  int tensor;  // 0 Q, 1 K, 2 V
  int local;   // (b*H + h) within its tensor
};

__device__ __forceinline__ SliceRef slice_ref(const PrepareArgs& a, int s) {
  const int nq = a.B * a.Hq, nk = a.B * a.Hkv;
  SliceRef r;
  if (s < nq) {
    r.tensor = 0; r.local = s;
  } else if (s < nq + nk) {
    r.tensor = 1; r.local = s - nq;
  } else {
    r.tensor = 2; r.local = s - nq - nk;
  }
  return r;
}

__device__ __forceinline__ float max_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

// ---- per-call initialisation: counters, flags, the work list -----------------
__global__ void k_flow_init(PrepareArgs a) {
  const int nq = a.B * a.Hq, nk = a.B * a.Hkv, ns = nq + 2 * nk;
  for (int i = threadIdx.x; i < ns; i += blockDim.x) {
    a.amax_bits[i] = 0u;
    a.a_done[i] = 0u;
  }
  for (int i = threadIdx.x; i < nk; i += blockDim.x) {
    a.m_done[i] = 0u;
    a.mu_ready[i] = 0u;
  }
  if (!a.center && a.k_mean)
    for (int i = threadIdx.x; i < nk * a.d; i += blockDim.x) a.k_mean[i] = 0.0f;
  // Order of the slices' A entries.  Without centring: K, V, Q.  With
  // centring the M entry of K slice j sits at step j, and the A order is the
  // first L = min(kLagA, nk) V slices, then K and V alternating, then the
  // last L K slices, then Q: K slice j's A entry comes at least L steps after
  // its M entry, and the steps in between carry V work.
  const int L = a.center ? (kLagA < nk ? kLagA : nk) : 0;
  const int k0 = nq, v0 = nq + nk;
  auto aorder = [&](int i) -> int {
    if (!a.center) return i < nk ? k0 + i : (i < 2 * nk ? v0 + (i - nk) : i - 2 * nk);
    if (i < L) return v0 + i;
    i -= L;
    if (i < 2 * (nk - L)) return (i & 1) ? v0 + L + (i >> 1) : k0 + (i >> 1);
    i -= 2 * (nk - L);
    if (i < L) return k0 + (nk - L) + i;
    return i - L;
  };
  // A list step holds up to five entries, in a fixed order of kinds; each kind
  // occupies an interval [lo, hi) of steps, so the entries before step t are
  // counted in closed form and every thread writes its steps' entries in place.
  //   full-sequence scales: C of the slice whose A entry was kLagC steps
  //     earlier, A (aorder), M of K slice t;
  //   per-tile scales (Q and K need no A pass): C of V slice t - kLagC, C of K
  //     slice t - Lk (Lk = kLagA with centring, after its M entry), A of V
  //     slice t, M of K slice t, C of Q slice t.
  const int Lk = a.center ? kLagA : 0;
  int lo[5], hi[5];
  uint32_t kinds[5];
  int nk_kinds;
  if (!a.tiles) {
    nk_kinds = 3;
    lo[0] = kLagC; hi[0] = ns + kLagC; kinds[0] = KIND_C;
    lo[1] = 0; hi[1] = ns; kinds[1] = KIND_A;
    lo[2] = 0; hi[2] = a.center ? nk : 0; kinds[2] = KIND_M;
  } else {
    nk_kinds = 5;
    lo[0] = kLagC; hi[0] = nk + kLagC; kinds[0] = KIND_C;
    lo[1] = Lk; hi[1] = nk + Lk; kinds[1] = KIND_C;
    lo[2] = 0; hi[2] = nk; kinds[2] = KIND_A;
    lo[3] = 0; hi[3] = a.center ? nk : 0; kinds[3] = KIND_M;
    lo[4] = 0; hi[4] = nq; kinds[4] = KIND_C;
  }
  auto slice_of = [&](int kind_idx, int t) -> int {
    if (!a.tiles) return kind_idx == 0 ? aorder(t - kLagC) : kind_idx == 1 ? aorder(t) : k0 + t;
    switch (kind_idx) {
      case 0: return v0 + (t - kLagC);
      case 1: return k0 + (t - Lk);
      case 2: return v0 + t;
      case 3: return k0 + t;
      default: return t;
    }
  };
  int nsteps = 0;
  for (int x = 0; x < nk_kinds; ++x) nsteps = max(nsteps, hi[x]);
  auto first = [&](int t) -> uint32_t {
    uint32_t e = 0;
    for (int x = 0; x < nk_kinds; ++x)
      if (hi[x] > lo[x]) e += uint32_t(min(max(t, lo[x]), hi[x]) - lo[x]);
    return e;
  };
  for (int t = threadIdx.x; t < nsteps; t += blockDim.x) {
    uint32_t e = first(t);
    for (int x = 0; x < nk_kinds; ++x)
      if (t >= lo[x] && t < hi[x]) a.entries[e++] = (kinds[x] << 30) | uint32_t(slice_of(x, t));
  }
  if (threadIdx.x == 0) {
    a.ctl[CTL_TICKET] = 0u;
    a.ctl[CTL_ABORT] = 0u;
    a.ctl[CTL_ENTRIES] = first(nsteps);
  }
}

struct Flow {
  PrepareArgs a;
  int tiles_per_slice, items_per_slice;
  int tiles_stat;  // tiles holding the first P tokens (the M and A passes)
};

__device__ __forceinline__ void raise_abort(const PrepareArgs& a) {
  if (atomicExch(a.ctl + CTL_ABORT, 1u) == 0u) atomicOr(a.status, DEV_TIMEOUT);
}

__device__ __forceinline__ bool aborted(const PrepareArgs& a) {
  return *reinterpret_cast<volatile uint32_t*>(a.ctl + CTL_ABORT) != 0u;
}

// Bounded wait on an mbarrier phase (one thread).  A suspended try_wait can
// return long before its hint, so the abort flag (a global load) and the
// clock are checked only every 64 polls: a waiting thread then costs its
// sub-partition few issue slots.
__device__ __forceinline__ bool bar_wait(const PrepareArgs& a, uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  const uint32_t hint = a.wait_ns < 20000ull ? uint32_t(a.wait_ns) : 20000u;  // never sleep past the limit
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_sleep(bar, parity, hint)) return true;
    if ((it & 63u) == 0u && (aborted(a) || globaltimer_ns() - t0 > a.wait_ns)) return false;
  }
}

// Bound for draining in-flight loads after an abort: independent of the wait
// limit (which may be tiny) and of the abort flag, so no CTA leaves with a
// copy still writing its shared memory.
constexpr uint64_t kDrainNs = 1000000000ull;

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait_sleep(bar, parity, 20000u))
    if (globaltimer_ns() - t0 > kDrainNs) return;
}

// Bounded wait for a flag in global memory set by another CTA (one thread);
// acquire ordering for the data published before it.
__device__ __forceinline__ bool flag_wait(const PrepareArgs& a, const uint32_t* flag) {
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
    if (v) return true;
    if (aborted(a) || globaltimer_ns() - t0 > a.wait_ns) return false;
    __nanosleep(200);
  }
}

__device__ __forceinline__ void flag_set(uint32_t* flag) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(flag), "r"(1u) : "memory");
}

// qs = top/amax, descale = amax/top (IEEE division; top = 448 for E4M3 codes,
// 127 for INT8 codes); amax = 0 -> 1, 1; a NaN or an infinity in the slice
// gives qs = 0 and a NaN descale.
__device__ __forceinline__ void scale_from_amax(uint32_t bits, float top, float& qs, float& ds) {
  if (bits >= 0x7F800000u) {
    qs = 0.0f;
    ds = __uint_as_float(0x7FC00000u);
  } else if (bits == 0u) {
    qs = 1.0f;
    ds = 1.0f;
  } else {
    const float amax = __uint_as_float(bits);
    qs = __fdiv_rn(top, amax);
    ds = __fdiv_rn(amax, top);
  }
}

__device__ __forceinline__ void red_max_relaxed(uint32_t* p, uint32_t v) {
  asm volatile("red.relaxed.gpu.global.max.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Count of finished tiles, with release ordering for this thread's earlier
// writes (its red.max above all): a reader that acquires the final count sees
// every contribution to the slice's amax.
__device__ __forceinline__ void red_add_release(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ---- producer -------------------------------------------------------------
// PREFIX: statistics over the first P < N tokens (the M and A entries stop there).
template <int D, bool BF16, bool PREFIX, bool I8>
__device__ void producer(const Flow& f, const CUtensorMap* const* in_maps, uint8_t* stages, TileMeta* meta,
                         uint64_t* full, uint64_t* empty) {
  using C = FlowCfg<D, BF16, I8>;
  const PrepareArgs& a = f.a;
  const uint32_t ips = uint32_t(f.items_per_slice), n_ent = a.ctl[CTL_ENTRIES];
  const uint32_t tail_ent = n_ent < kTailEntries ? n_ent : kTailEntries;
  const uint32_t t_small = (n_ent - tail_ent) * ips;  // tickets before the small items
  const uint32_t total = t_small + tail_ent * ips * kTailSplit;
  // A slice's data is read again by a later pass (A after M, C after A):
  // keep it in L2 until the C pass reads it for the last time.
  const uint64_t keep = l2_evict_last_policy(), last_use = l2_evict_first_policy();
  uint32_t n = 0;  // tiles pushed
  bool ok = true;
  // The next ticket is claimed while the current item's last two tiles are
  // pushed, so the claim's round trip stays off the ring.  Items are still
  // finished in ticket order by this CTA, so the earliest unfinished item is
  // always some CTA's current one and never waits.
  uint32_t t = atomicAdd(a.ctl + CTL_TICKET, 1u);
  for (;;) {
    if (aborted(a)) { ok = false; break; }
    if (t >= total) break;
    uint32_t t_next = 0;
    const bool small = t >= t_small;
    const uint32_t ent = a.entries[small ? n_ent - tail_ent + (t - t_small) / (ips * kTailSplit) : t / ips];
    const uint32_t item = small ? (t - t_small) % (ips * kTailSplit) : t % ips;
    const int tpi = small ? kTilesPerItem / int(kTailSplit) : kTilesPerItem;
    const uint32_t kind = ent >> 30, s = ent & 0x3FFFFFFFu;
    const SliceRef r = slice_ref(a, int(s));
    const CUtensorMap* map = in_maps[r.tensor];
    const int row_begin = int(item) * kTR * tpi;
    // the M and A passes read only the first P tokens: their later items are
    // empty; so are the small items past a slice's last tile
    const int lim = (PREFIX && kind != KIND_C) ? a.P : a.N;
    const int nt = min(tpi, (lim - row_begin + kTR - 1) / kTR);
    if (nt <= 0) {
      t = atomicAdd(a.ctl + CTL_TICKET, 1u);
      continue;
    }
    for (int tl = 0; tl < nt && ok; ++tl, ++n) {
      if (tl == (nt > 2 ? nt - 2 : 0)) t_next = atomicAdd(a.ctl + CTL_TICKET, 1u);
      const int row0 = row_begin + tl * kTR;
      const uint32_t st = n % C::NST, ph = (n / C::NST) & 1u;
      if (!bar_wait(a, empty + st, ph ^ 1u)) { ok = false; break; }
      // tiles go round the groups: tl + kGroups is this group's next tile
      meta[st] = TileMeta{kind, s, uint32_t(row0), tl + kGroups >= nt ? 1u : 0u};
      mbar_arrive_expect_tx(full + st, C::SB);
#pragma unroll
      for (int b = 0; b < C::NB; ++b)
        tma_load_3d_hint(stages + size_t(st) * C::SB + b * (kTR * 128), map, full + st, b * 128, row0, r.local,
                         kind == KIND_C ? last_use : keep);
    }
    if (!ok) break;
    t = t_next;
  }
  if (ok) {
    // one end marker per consumer group (tiles go round the groups)
    for (int g = 0; g < kGroups; ++g, ++n) {
      const uint32_t st = n % C::NST, ph = (n / C::NST) & 1u;
      if (!bar_wait(a, empty + st, ph ^ 1u)) { ok = false; break; }
      meta[st] = TileMeta{KIND_DONE, 0u, 0u, 0u};
      mbar_arrive(full + st);
    }
  }
  if (!ok) {
    raise_abort(a);
    // drain: the loads of the last NST tiles may still be in flight
    for (uint32_t x = 0; x < uint32_t(C::NST) && x < n; ++x) {
      const uint32_t m = n - 1 - x;
      drain_wait(full + m % C::NST, (m / C::NST) & 1u);
    }
  }
}

// ---- consumer helpers -----------------------------------------------------
// Byte offset of 16-byte chunk c of row r in a swizzled tile of 128-byte rows.
__device__ __forceinline__ uint32_t sw128(int r, int c) { return uint32_t(r * 128 + ((c ^ (r & 7)) << 4)); }

// Byte offset of 16-byte chunk c of row r in a warp's staging buffer of D-byte
// rows, in the swizzle its tensor map uses (128-byte rows: chunk ^ r % 8;
// 64-byte rows: chunk ^ (r / 2) % 4): a warp writing one row per lane hits
// every bank group once per eight lanes.
template <int D>
__device__ __forceinline__ uint32_t stage_off(int r, int c) {
  if constexpr (D == 128) {
    return uint32_t(r * 128 + ((c ^ (r & 7)) << 4));
  } else {
    return uint32_t(r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
  }
}

// Bounded wait of a whole warp on an mbarrier phase: lane 0 sleeps on it, then
// every lane tests the phase itself (each lane's own acquire).  The phase
// cannot move on before this warp releases the stage, so the second test holds.
__device__ __forceinline__ bool warp_bar_wait(const PrepareArgs& a, uint64_t* bar, uint32_t parity) {
  if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
  uint32_t v = 0;
  if ((threadIdx.x & 31) == 0) v = bar_wait(a, bar, parity) ? 1u : 0u;
  if (__shfl_sync(0xffffffffu, v, 0) == 0u) return false;
  return __all_sync(0xffffffffu, mbar_try_wait(bar, parity));
}

// Bounded wait of a whole warp for a flag set by another CTA; once lane 0 has
// seen it, every lane reads it with acquire ordering before its own loads.
__device__ __forceinline__ bool warp_flag_wait(const PrepareArgs& a, const uint32_t* flag) {
  uint32_t v = 0;
  if ((threadIdx.x & 31) == 0) v = flag_wait(a, flag) ? 1u : 0u;
  if (__shfl_sync(0xffffffffu, v, 0) == 0u) return false;
  uint32_t seen;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(seen) : "l"(flag) : "memory");
  return __all_sync(0xffffffffu, seen != 0u);
}

// Bounded wait of a whole warp until a counter reaches `target` (another
// CTA's release adds); every lane then reads it with acquire ordering.
__device__ __forceinline__ bool warp_count_wait(const PrepareArgs& a, const uint32_t* ctr, uint32_t target) {
  uint32_t v = 0;
  if ((threadIdx.x & 31) == 0) {
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
      uint32_t c;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(c) : "l"(ctr) : "memory");
      if (c >= target) { v = 1u; break; }
      if (aborted(a) || globaltimer_ns() - t0 > a.wait_ns) break;
      __nanosleep(200);
    }
  }
  if (__shfl_sync(0xffffffffu, v, 0) == 0u) return false;
  uint32_t seen;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(seen) : "l"(ctr) : "memory");
  return __all_sync(0xffffffffu, seen >= target);
}

// Row r of an input stage as packed pairs P[j] = (x_j, x_{j+D/2}); with
// `flip`, the sign flip is applied as a sign-bit XOR on the raw values (exact,
// signed zeros included) - only for rows that are not centred, since the
// flip must follow the centring.
template <int D, bool BF16, bool FLIP>
__device__ __forceinline__ void load_row(const uint8_t* stage, int r, const uint32_t* smask, uint64_t (&P)[D / 2]) {
  using C = FlowCfg<D, BF16>;
  constexpr int PER = BF16 ? 8 : 4, CH = C::ROW_BYTES / 16;  // elements per chunk, chunks per row
  // The per-chunk offsets are recomputed for every tile (an opaque copy of
  // r % 8): hoisted out of the tile loop they would hold a register each.
  int r7 = r & 7;
  asm volatile("" : "+r"(r7));
  const uint8_t* rowp = stage + r * 128;
  auto chunk = [&](int q) -> uint4 {
    const int box = q / 8, cq = q % 8;
    uint4 u = *reinterpret_cast<const uint4*>(rowp + box * (kTR * 128) + ((cq ^ r7) << 4));
    if constexpr (FLIP && !BF16) {
      const uint4 m = *reinterpret_cast<const uint4*>(smask + 4 * q);
      u.x ^= m.x; u.y ^= m.y; u.z ^= m.z; u.w ^= m.w;
    }
    return u;
  };
  // bf16 with the flip: the high element is (w ^ m) & 0xFFFF0000, one
  // three-input logic op; the low one is (w << 16) + (m << 16), where adding
  // 0 or 2^31 modulo 2^32 is the XOR of bit 31 (one shift-and-add).
  auto mask = [&](int q, int lo) -> uint4 {
    return *reinterpret_cast<const uint4*>(smask + (lo ? C::WORDS : 0) + 4 * q);
  };
  // chunk q holds elements PER*q ..; it pairs with chunk q + CH/2 (elements + D/2)
#pragma unroll
  for (int q = 0; q < CH / 2; ++q) {
    const uint4 ua = chunk(q), ub = chunk(q + CH / 2);
    const uint32_t wa[4] = {ua.x, ua.y, ua.z, ua.w}, wb[4] = {ub.x, ub.y, ub.z, ub.w};
    uint32_t ha[4] = {0u, 0u, 0u, 0u}, hb[4] = {0u, 0u, 0u, 0u}, la[4] = {0u, 0u, 0u, 0u}, lb[4] = {0u, 0u, 0u, 0u};
    if constexpr (FLIP && BF16) {
      const uint4 mha = mask(q, 0), mhb = mask(q + CH / 2, 0), mla = mask(q, 1), mlb = mask(q + CH / 2, 1);
      ha[0] = mha.x; ha[1] = mha.y; ha[2] = mha.z; ha[3] = mha.w;
      hb[0] = mhb.x; hb[1] = mhb.y; hb[2] = mhb.z; hb[3] = mhb.w;
      la[0] = mla.x; la[1] = mla.y; la[2] = mla.z; la[3] = mla.w;
      lb[0] = mlb.x; lb[1] = mlb.y; lb[2] = mlb.z; lb[3] = mlb.w;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if constexpr (BF16) {
        P[PER * q + 2 * i] = pack2(__uint_as_float((wa[i] << 16) + la[i]), __uint_as_float((wb[i] << 16) + lb[i]));
        P[PER * q + 2 * i + 1] =
            pack2(__uint_as_float((wa[i] ^ ha[i]) & 0xFFFF0000u), __uint_as_float((wb[i] ^ hb[i]) & 0xFFFF0000u));
      } else {
        P[PER * q + i] = pack2(__uint_as_float(wa[i]), __uint_as_float(wb[i]));
      }
    }
  }
}

// Centre (x + (-mu), one rounding), then for centred rows the sign flip
// (a sign-bit XOR on the packed pair), then FWHT stages h = 1 .. D/4, which
// act within each half of the row (packed adds and subtracts).  The order is
// the method's: s * (x - mu) keeps the sign of a zero difference that
// s*x - s*mu would lose.  The last stage (h = D/2) is left to the caller.
template <int D, bool CENTER, bool ROTATE>
__device__ __forceinline__ void transform_stages(uint64_t (&P)[D / 2], const uint64_t* nmu, const uint64_t* pmask) {
  if constexpr (CENTER) {
#pragma unroll
    for (int j = 0; j < D / 2; ++j) P[j] = fadd2(P[j], nmu[j]);
    if constexpr (ROTATE) {
#pragma unroll
      for (int j = 0; j < D / 2; j += 2) {
        const uint4 m = *reinterpret_cast<const uint4*>(pmask + j);
        P[j] ^= (uint64_t(m.y) << 32) | m.x;
        P[j + 1] ^= (uint64_t(m.w) << 32) | m.z;
      }
    }
  }
  if constexpr (ROTATE) {
    const uint64_t neg1 = pack2(-1.0f, -1.0f);
#pragma unroll
    for (int h = 1; h < D / 2; h <<= 1) {
#pragma unroll
      for (int j = 0; j < D / 2; ++j) {
        if ((j & h) == 0) {
          const uint64_t u = P[j], v = P[j + h];
          P[j] = fadd2(u, v);
          P[j + h] = ffma2(v, neg1, u);  // u - v, one rounding
        }
      }
    }
  }
}

// Last FWHT stage: (a_j, b_j) -> (a_j + b_j, a_j - b_j), i.e. elements j and j + D/2.
template <int D>
__device__ __forceinline__ void final_stage(uint64_t (&P)[D / 2]) {
#pragma unroll
  for (int j = 0; j < D / 2; ++j) {
    float lo, hi;
    unpack2(P[j], lo, hi);
    P[j] = pack2(__fadd_rn(lo, hi), __fsub_rn(lo, hi));
  }
}

__device__ __forceinline__ float max3_nan(float a, float b, float c) {
  float d;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// amax of a row held as values: max over |x| (NaN wins).
template <int D>
__device__ __forceinline__ uint32_t plain_amax_bits(const uint64_t (&P)[D / 2]) {
  float m[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int j = 0; j < D / 2; ++j) {
    float lo, hi;
    unpack2(P[j], lo, hi);
    m[j & 3] = max3_nan(m[j & 3], fabsf(lo), fabsf(hi));
  }
  return __float_as_uint(max_nan(max_nan(m[0], m[1]), max_nan(m[2], m[3])));
}

// amax of a rotated row held before its last stage as pairs (a_j, b_j).  The
// last stage gives fl(a + b) and fl(a - b); the larger of |a + b| and |a - b|
// is |a| + |b|, and round-to-nearest-even is odd-symmetric and monotone, so
// max(|fl(a + b)|, |fl(a - b)|) = fl(|a| + |b|) exactly (a NaN or an infinity
// in either gives a NaN or an infinity, which the scale reports as non-finite).
template <int D>
__device__ __forceinline__ uint32_t rotated_amax_bits(const uint64_t (&P)[D / 2]) {
  float m[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int j = 0; j < D / 2; j += 2) {
    float a0, b0, a1, b1;
    unpack2(P[j], a0, b0);
    unpack2(P[j + 1], a1, b1);
    m[(j >> 1) & 3] = max3_nan(m[(j >> 1) & 3], __fadd_rn(fabsf(a0), fabsf(b0)), __fadd_rn(fabsf(a1), fabsf(b1)));
  }
  return __float_as_uint(max_nan(max_nan(m[0], m[1]), max_nan(m[2], m[3])));
}

// E4M3 codes of row values x_e * qs, e = 0..D-1, as D/4 words (byte e%4 of word e/4).
template <int D>
__device__ __forceinline__ void row_codes(const uint64_t (&P)[D / 2], float qs, uint32_t (&cw)[D / 4]) {
  const uint64_t q2 = pack2(qs, qs);
#pragma unroll
  for (int k = 0; k < D / 8; ++k) {
    float lo[4], hi[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) unpack2(fmul2(P[4 * k + i], q2), lo[i], hi[i]);
    cw[k] = pack_b16x2(cvt_e4m3x2(lo[0], lo[1]), cvt_e4m3x2(lo[2], lo[3]));              // elements 4k ..
    cw[k + D / 8] = pack_b16x2(cvt_e4m3x2(hi[0], hi[1]), cvt_e4m3x2(hi[2], hi[3]));      // elements D/2 + 4k ..
  }
}

// INT8 codes of a row held as pairs (x_j, x_{j+D/2}): the nearest integer of
// fl32(x * qs), ties to even, saturated to +-127, as bf16 values (exact), into
// the warp's staging buffer: boxes of 32 rows x 128 bytes (64 codes) in the
// 128-byte swizzle, row = lane.  The product is rounded to an integer by one
// round-to-integer instruction on the stored fp32 product.  (Adding and
// subtracting 1.5 * 2^23 instead gave codes one too small where fl32(x * qs)
// is an exact tie but the unrounded product lies just below it: the multiply
// and the add were not rounded separately.)
template <int D>
__device__ __forceinline__ void row_int8_codes(const uint64_t (&P)[D / 2], float qs, uint8_t* ob, int lane) {
  const uint64_t q2 = pack2(qs, qs);
  const uint32_t lim_lo = 0xC2FEC2FEu, lim_hi = 0x42FE42FEu;  // -127, 127 in bf16
#pragma unroll
  for (int c8 = 0; c8 < D / 16; ++c8) {
    // pairs 8 c8 .. 8 c8 + 7: codes 8 c8 .. (chunk c8) and D/2 + 8 c8 .. (chunk D/16 + c8)
    uint32_t wl[4], wh[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float a0, b0, a1, b1;
      unpack2(fmul2(P[8 * c8 + 2 * i], q2), a0, b0);
      unpack2(fmul2(P[8 * c8 + 2 * i + 1], q2), a1, b1);
      wl[i] = bf16x2_clamp(rintf(a0), rintf(a1), lim_lo, lim_hi);
      wh[i] = bf16x2_clamp(rintf(b0), rintf(b1), lim_lo, lim_hi);
    }
    const int ch = D / 16 + c8;
    *reinterpret_cast<uint4*>(ob + (c8 >> 3) * 4096 + lane * 128 + (((c8 & 7) ^ (lane & 7)) << 4)) =
        make_uint4(wl[0], wl[1], wl[2], wl[3]);
    *reinterpret_cast<uint4*>(ob + (ch >> 3) * 4096 + lane * 128 + (((ch & 7) ^ (lane & 7)) << 4)) =
        make_uint4(wh[0], wh[1], wh[2], wh[3]);
  }
}

// Mean key of K slice `sl` from the chunk sums of its first P tokens: per
// channel, the `chunks` sums added in chunk order, then one division by P.
// Lane l owns channels l, l + 32, ...; the loads run eight chunks ahead of the
// ordered adds.
template <int D>
__device__ __forceinline__ void finish_mean(const PrepareArgs& a, int tiles_per_slice, int chunks, int sl, int lane) {
  constexpr int CPL = D / 32;
  const float* base = a.mean_part + int64_t(sl) * tiles_per_slice * D + lane;
  float tot[CPL];
#pragma unroll
  for (int i = 0; i < CPL; ++i) tot[i] = 0.0f;
  int k = 0;
  for (; k + 8 <= chunks; k += 8) {
    float v[8][CPL];
#pragma unroll
    for (int u = 0; u < 8; ++u)
#pragma unroll
      for (int i = 0; i < CPL; ++i) v[u][i] = __ldcg(base + int64_t(k + u) * D + 32 * i);
#pragma unroll
    for (int u = 0; u < 8; ++u)
#pragma unroll
      for (int i = 0; i < CPL; ++i) tot[i] = __fadd_rn(tot[i], v[u][i]);
  }
  for (; k < chunks; ++k)
#pragma unroll
    for (int i = 0; i < CPL; ++i) tot[i] = __fadd_rn(tot[i], __ldcg(base + int64_t(k) * D + 32 * i));
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    const float mu = __fdiv_rn(tot[i], float(a.P));
    a.mu[sl * D + lane + 32 * i] = mu;
    if (a.k_mean) a.k_mean[sl * D + lane + 32 * i] = mu;
  }
}

// ---- the persistent kernel ----------------------------------------------------
// PREFIX is the causal-prefix form (P < N); without it the kernel is the
// full-sequence one and carries no prefix code.  I8: Q and K get INT8 codes
// (scale 127/amax) stored as bf16 values; V keeps E4M3.
template <int D, bool BF16, bool PREFIX, bool I8>
__global__ void __launch_bounds__(kFlowThreads, 1)
    k_prepare(const __grid_constant__ CUtensorMap in_q, const __grid_constant__ CUtensorMap in_k,
              const __grid_constant__ CUtensorMap in_v, const __grid_constant__ CUtensorMap out_q,
              const __grid_constant__ CUtensorMap out_k, const __grid_constant__ CUtensorMap out_v,
              const Flow f) {
  using C = FlowCfg<D, BF16, I8>;
  const PrepareArgs& a = f.a;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base by pointer arithmetic on the shared array (an
  // integer round trip would hide the address space and make every access
  // through it a generic one)
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* stages = sm;
  uint8_t* outb = stages + size_t(C::NST) * C::SB;               // [consumer warp][2] staging buffers
  TileMeta* meta = reinterpret_cast<TileMeta*>(outb + size_t(C::NBUF * kConsumerWarps) * C::WB);
  uint64_t* full = reinterpret_cast<uint64_t*>(meta + C::NST);
  uint64_t* empty = full + C::NST;
  // sign-bit mask per input word, then (bf16) the low element's sign moved to bit 31
  uint32_t* smask = reinterpret_cast<uint32_t*>(empty + C::NST);
  uint64_t* pmask = reinterpret_cast<uint64_t*>(smask + 2 * C::WORDS);  // sign-bit masks of the pairs (x_j, x_{j+D/2})
  uint64_t* nmu_all = pmask + D / 2;                               // per consumer warp: -mu as pairs [D/2]
  // per-tile scales: each group's four warp maxima of a tile, two slots by
  // tile parity, and the barriers (four arrivals) that publish them
  uint32_t* tmax = reinterpret_cast<uint32_t*>(nmu_all + kConsumerWarps * (D / 2));  // [group][2][4]
  uint64_t* xbar = reinterpret_cast<uint64_t*>(tmax + 4 * 2 * kGroups);              // [group][2]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 4);  // one arrival per consumer warp of the stage's group
    }
    for (int x = 0; x < 2 * kGroups; ++x) mbar_init(xbar + x, 4);
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < C::WORDS; i += blockDim.x) {
    uint32_t m = 0;
    if (a.rotate) {
      if constexpr (BF16) {
        m = (a.signs[2 * i] < 0 ? 0x8000u : 0u) | (a.signs[2 * i + 1] < 0 ? 0x80000000u : 0u);
      } else {
        m = a.signs[i] < 0 ? 0x80000000u : 0u;
      }
    }
    smask[i] = m;
    smask[C::WORDS + i] = m << 16;
  }
  for (int j = threadIdx.x; j < D / 2; j += blockDim.x) {
    const uint64_t lo = (a.rotate && a.signs[j] < 0) ? 0x80000000ull : 0ull;
    const uint64_t hi = (a.rotate && a.signs[j + D / 2] < 0) ? 0x80000000ull : 0ull;
    pmask[j] = lo | (hi << 32);
  }
  __syncthreads();

  if (warp >= kConsumerWarps) {
    regs_decrease<kProducerRegs>();
    if (warp == kConsumerWarps && lane == 0) {
      tma_prefetch_desc(&in_q);
      tma_prefetch_desc(&in_k);
      tma_prefetch_desc(&in_v);
      const CUtensorMap* maps[3] = {&in_q, &in_k, &in_v};
      producer<D, BF16, PREFIX, I8>(f, maps, stages, meta, full, empty);
    }
    return;
  }

  // Consumer warp: group g takes tiles g, g + kGroups, ... of the ring, and
  // warp w4 of the group rows 32*w4 .. 32*w4 + 31 of each.  Warps run
  // independently: each waits on the stage itself, keeps its own counts and
  // stores its own rows, so no barrier couples the warps of a group.
  regs_increase<kConsumerRegs>();
  const int g = warp >> 2, w4 = warp & 3, r = threadIdx.x & 127;
  uint64_t* nmu = nmu_all + warp * (D / 2);
  uint8_t* obuf = outb + size_t(C::NBUF * warp) * C::WB;
  const uint32_t tiles = uint32_t(f.tiles_per_slice);
  const uint32_t stat_tiles = uint32_t(f.tiles_stat);  // M and A tiles of a slice
  const int plen = PREFIX ? a.P : a.N;                 // tokens the M and A passes cover
  int mu_slice = -1;   // K slice whose -mu is in nmu
  int qs_slice = -1;   // slice whose scale is in qs
  float qs = 0.0f;
  uint32_t qs_bits = 0;  // the slice's amax bits
  uint32_t cbuf = 0;   // staging buffer parity
  bool stored = false;
  bool ok = true;
  uint32_t run_max = 0;    // amax bits of this lane's rows in the current item
  uint32_t run_tiles = 0;  // tiles of the current item this warp has finished
  uint32_t xc = 0;         // per-tile scale exchanges of this warp's group
  for (uint32_t j = 0;; ++j) {
    const uint32_t n = uint32_t(kGroups) * j + uint32_t(g);
    const uint32_t st = n % C::NST, ph = (n / C::NST) & 1u;
    if (!warp_bar_wait(a, full + st, ph)) { ok = false; break; }
    const TileMeta tm = meta[st];
    if (tm.kind == KIND_DONE) break;
    const uint8_t* stage = stages + size_t(st) * C::SB;
    const int s = int(tm.slice);
    const SliceRef sr = slice_ref(a, s);
    const int row0 = int(tm.row0);
    // rows the pass covers: every token for the cast, the first P for M and A
    const bool valid = row0 + r < (PREFIX && tm.kind != KIND_C ? plen : a.N);
    const bool qk = sr.tensor < 2;
    const float top = (I8 && qk) ? 127.0f : 448.0f;  // largest code of the slice's format
    const bool rotate = a.rotate && qk, center = a.center && sr.tensor == 1;

    if (tm.kind == KIND_M) {
      // chunk sum of each channel over the tile's tokens, in token order:
      // thread r owns channel r (warps past the last channel only release)
      const bool has = 32 * w4 < D;
      if (has) {
        const int rows = min(kTR, plen - row0);
        const int byte = r * C::ES, box = byte / 128, cq = (byte % 128) / 16, off = byte % 16;
        // loads in batches of 16 (independent), then the adds in token order
        float part = 0.0f;
        for (int t0 = 0; t0 < rows; t0 += 16) {
          float v[16];
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            const uint8_t* src = stage + box * (kTR * 128) + sw128(t0 + u, cq) + off;
            v[u] = BF16 ? __uint_as_float(uint32_t(*reinterpret_cast<const uint16_t*>(src)) << 16)
                        : *reinterpret_cast<const float*>(src);
          }
#pragma unroll
          for (int u = 0; u < 16; ++u)
            if (t0 + u < rows) part = __fadd_rn(part, v[u]);
        }
        a.mean_part[(int64_t(sr.local) * f.tiles_per_slice + row0 / kTR) * D + r] = part;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + st);
      if (!has) continue;
      ++run_tiles;
      if (!tm.last) continue;
      // this warp's chunks of the item are written: count them (one atomic per
      // warp and item); the warp that completes the slice computes its mean
      __threadfence();
      __syncwarp();
      uint32_t fin = 0;
      if (lane == 0)
        fin = atomicAdd(a.m_done + sr.local, run_tiles) + run_tiles == stat_tiles * uint32_t(D / 32) ? 1u : 0u;
      run_tiles = 0;
      if (__shfl_sync(0xffffffffu, fin, 0) != 0u) {
        __threadfence();
        finish_mean<D>(a, f.tiles_per_slice, f.tiles_stat, sr.local, lane);
        __threadfence();
        __syncwarp();
        if (lane == 0) flag_set(a.mu_ready + sr.local);
      }
      continue;
    }

    // centred K needs the slice's mean key
    if (center && mu_slice != sr.local) {
      if (!warp_flag_wait(a, a.mu_ready + sr.local)) { ok = false; break; }
      for (int jj = lane; jj < D / 2; jj += 32)
        nmu[jj] = pack2(-__ldcg(a.mu + sr.local * D + jj), -__ldcg(a.mu + sr.local * D + jj + D / 2));
      __syncwarp();
      mu_slice = sr.local;
    }

    // load and transform, each form compiled on its own (no per-chunk tests)
    uint64_t P[D / 2];
    if (rotate && !center) {
      load_row<D, BF16, true>(stage, r, smask, P);
    } else {
      load_row<D, BF16, false>(stage, r, smask, P);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty + st);  // the warp's rows are in registers
    if (center) {
      if (rotate) {
        transform_stages<D, true, true>(P, nmu, pmask);
      } else {
        transform_stages<D, true, false>(P, nmu, pmask);
      }
    } else if (rotate) {
      transform_stages<D, false, true>(P, nmu, pmask);
    }

    if (tm.kind == KIND_A) {
      if (valid) run_max = max(run_max, rotate ? rotated_amax_bits<D>(P) : plain_amax_bits<D>(P));
      ++run_tiles;
      if (!tm.last) continue;
      // end of the warp's share of the item: one max and one count
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) run_max = max(run_max, __shfl_xor_sync(0xffffffffu, run_max, o));
      if (lane == 0) {
        if (run_max) red_max_relaxed(a.amax_bits + s, run_max);
        red_add_release(a.a_done + s, run_tiles);
      }
      run_max = 0;
      run_tiles = 0;
      continue;
    }

    // KIND_C: the scale (the slice's, or with per-tile scales the tile's), the
    // last stage, codes staged for a TMA store
    if (a.tiles && qk) {
      // the tile's amax from its four warps, exchanged through shared memory
      uint32_t mx = valid ? (rotate ? rotated_amax_bits<D>(P) : plain_amax_bits<D>(P)) : 0u;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const uint32_t xb = 2u * uint32_t(g) + (xc & 1u);
      if (lane == 0) {
        tmax[4 * xb + w4] = mx;
        mbar_arrive(xbar + xb);
      }
      if (!warp_bar_wait(a, xbar + xb, (xc >> 1) & 1u)) { ok = false; break; }
      ++xc;
      const uint32_t bits = max(max(tmax[4 * xb], tmax[4 * xb + 1]), max(tmax[4 * xb + 2], tmax[4 * xb + 3]));
      float ds;
      scale_from_amax(bits, top, qs, ds);
      qs_slice = -1;  // qs is this tile's
      if (w4 == 0 && lane == 0) {
        (sr.tensor == 0 ? a.q_ds : a.k_ds)[int64_t(sr.local) * tiles + uint32_t(row0 / kScaleTile)] = ds;
        if (bits >= 0x7F800000u) atomicOr(a.status, DEV_NONFINITE);
      }
    } else {
      if (qs_slice != s) {
        // every A tile of the slice has added its amax (acquire on the count)
        if (!warp_count_wait(a, a.a_done + s, stat_tiles * 4u)) { ok = false; break; }
        qs_bits = __ldcg(a.amax_bits + s);
        float ds;
        scale_from_amax(qs_bits, top, qs, ds);
        qs_slice = s;
      }
      if (row0 == 0 && w4 == 0 && lane == 0) {
        // the warp with the slice's first rows publishes its descale
        float q2, ds;
        scale_from_amax(qs_bits, top, q2, ds);
        (sr.tensor == 0 ? a.q_ds : sr.tensor == 1 ? a.k_ds : a.v_ds)[sr.local] = ds;
        if (qs_bits >= 0x7F800000u) atomicOr(a.status, DEV_NONFINITE);
      }
      // tokens after the prefix took no part in the amax: check them here
      if (PREFIX && row0 + kTR > plen) {
        const bool bad = valid && row0 + r >= plen &&
                         (rotate ? rotated_amax_bits<D>(P) : plain_amax_bits<D>(P)) >= 0x7F800000u;
        if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(a.status, DEV_NONFINITE);
      }
    }
    if (rotate) final_stage<D>(P);
    const bool vt = sr.tensor == 2 && a.vt;
    const bool i8row = I8 && qk;  // INT8 codes in bf16, two bytes a code
    const int x0 = row0 + 32 * w4;  // the warp's first row (token)
    if (int64_t(x0) >= (vt ? a.ldv : int64_t(a.N))) continue;  // all of the warp's rows are past the end
    // the store that last read this buffer (two casts ago; the last one with
    // a single buffer) must be done with it
    if (stored && lane == 0) bulk_wait_read<C::NBUF - 1>();
    __syncwarp();
    uint8_t* ob = obuf + size_t(C::NBUF > 1 ? cbuf : 0u) * C::WB;
    if (i8row) {
      row_int8_codes<D>(P, qs, ob, lane);
    } else {
      uint32_t cw[D / 4];
      row_codes<D>(P, qs, cw);
      if (vt) {
        // channel-major [D][32 tokens]: a 4 x 4 byte transpose within each quad
        // of lanes turns word k of lane 4q + i (channels 4k .. 4k + 3 of token
        // 4q + i) into channel 4k + i of tokens 4q .. 4q + 3, one 32-bit store
        const int i4 = lane & 3;
#pragma unroll
        for (int k = 0; k < D / 4; ++k) {
          const uint32_t w = cw[k];
          // 16-bit halves with lane ^ 2, then bytes with lane ^ 1
          const uint32_t o1 = __shfl_xor_sync(0xffffffffu, w, 2);
          const uint32_t w1 = (i4 & 2) ? __byte_perm(w, o1, 0x3276) : __byte_perm(w, o1, 0x5410);
          const uint32_t o2 = __shfl_xor_sync(0xffffffffu, w1, 1);
          const uint32_t w2 = (i4 & 1) ? __byte_perm(w1, o2, 0x3715) : __byte_perm(w1, o2, 0x6240);
          *reinterpret_cast<uint32_t*>(ob + (4 * k + i4) * 32 + (lane & ~3)) = w2;
        }
      } else {
#pragma unroll
        for (int c = 0; c < D / 16; ++c)
          *reinterpret_cast<uint4*>(ob + stage_off<D>(lane, c)) =
              make_uint4(cw[4 * c], cw[4 * c + 1], cw[4 * c + 2], cw[4 * c + 3]);
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      const uint64_t once = l2_evict_first_policy();  // codes are written once and read by a later kernel
      if (i8row) {
        // one 128-byte box of 64 codes per store
#pragma unroll
        for (int b = 0; b < C::NOB; ++b)
          tma_store_3d_hint(sr.tensor == 0 ? &out_q : &out_k, ob + b * 4096, b * 128, x0, sr.local, once);
      } else if (vt) {
        tma_store_3d_hint(&out_v, ob, x0, 0, sr.local, once);
      } else {
        tma_store_3d_hint(sr.tensor == 0 ? &out_q : sr.tensor == 1 ? &out_k : &out_v, ob, 0, x0, sr.local, once);
      }
      bulk_commit();
    }
    stored = true;
    cbuf ^= 1u;
  }
  if (!ok) raise_abort(a);
  if (lane == 0 && stored) bulk_wait_all();
}

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

template <int D, bool BF16>
cudaError_t run(const PrepareArgs& a, cudaStream_t st) {
  using C = FlowCfg<D, BF16>;
  const int nq = a.B * a.Hq, nk = a.B * a.Hkv;
  const uint64_t rb = uint64_t(D) * C::ES, N = uint64_t(a.N);
  const CUtensorMapSwizzle swo = D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUtensorMap in_q, in_k, in_v, out_q, out_k, out_v;
  if (encode_tiled_3d(&in_q, a.Q, rb, N, nq, rb, rb * N, 128, kTR, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
      encode_tiled_3d(&in_k, a.K, rb, N, nk, rb, rb * N, 128, kTR, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
      encode_tiled_3d(&in_v, a.V, rb, N, nk, rb, rb * N, 128, kTR, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  // outputs: 32-row boxes, one per consumer warp; INT8 Q/K codes are bf16
  // rows of 2D bytes, stored as 128-byte boxes
  if (a.i8) {
    const uint64_t ob = 2 * uint64_t(D);
    if (encode_tiled_3d(&out_q, a.q8, ob, N, nq, ob, ob * N, 128, 32, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
        encode_tiled_3d(&out_k, a.k8, ob, N, nk, ob, ob * N, 128, 32, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  } else if (encode_tiled_3d(&out_q, a.q8, D, N, nq, D, D * N, D, 32, swo) != CUDA_SUCCESS ||
             encode_tiled_3d(&out_k, a.k8, D, N, nk, D, D * N, D, 32, swo) != CUDA_SUCCESS) {
    return cudaErrorInvalidValue;
  }
  if (a.vt) {
    if (encode_tiled_3d(&out_v, a.v8, uint64_t(a.ldv), D, nk, uint64_t(a.ldv), uint64_t(a.ldv) * D, 32, D,
                        CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  } else {
    if (encode_tiled_3d(&out_v, a.v8, D, N, nk, D, D * N, D, 32, swo) != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  Flow f;
  f.a = a;
  f.tiles_per_slice = (a.N + kTR - 1) / kTR;
  f.items_per_slice = (f.tiles_per_slice + kTilesPerItem - 1) / kTilesPerItem;
  f.tiles_stat = (a.P + kTR - 1) / kTR;
  k_flow_init<<<1, 256, 0, st>>>(a);
  const bool prefix = a.P < a.N;
  auto kern = a.i8 ? (prefix ? k_prepare<D, BF16, true, true> : k_prepare<D, BF16, false, true>)
                   : (prefix ? k_prepare<D, BF16, true, false> : k_prepare<D, BF16, false, false>);
  const size_t smem = a.i8 ? FlowCfg<D, BF16, true>::SMEM : C::SMEM;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  const int grid = a.num_sms > 0 ? a.num_sms : 1;
  kern<<<grid, kFlowThreads, smem, st>>>(in_q, in_k, in_v, out_q, out_k, out_v, f);
  return cudaGetLastError();
}

}  // namespace

size_t prepare_workspace_bytes(int B, int Hq, int Hkv, int N, int d, int center) {
  const size_t ns = size_t(B) * Hq + 2 * size_t(B) * Hkv, nk = size_t(B) * Hkv;
  size_t bytes = 2 * align256(ns * 4) + 2 * align256(nk * 4) + align256(16) + align256(3 * ns * 4 + 64);
  if (center) {
    const size_t nchunks = (size_t(N) + kTR - 1) / kTR;
    bytes += align256(nk * nchunks * d * 4) + align256(nk * d * 4);
  }
  return bytes;
}

void carve_prepare_workspace(PrepareArgs& a, void* ws) {
  const size_t ns = size_t(a.B) * a.Hq + 2 * size_t(a.B) * a.Hkv, nk = size_t(a.B) * a.Hkv;
  char* p = static_cast<char*>(ws);
  auto take = [&](size_t bytes) {
    char* q = p;
    p += align256(bytes);
    return q;
  };
  a.amax_bits = reinterpret_cast<uint32_t*>(take(ns * 4));
  a.a_done = reinterpret_cast<uint32_t*>(take(ns * 4));
  a.m_done = reinterpret_cast<uint32_t*>(take(nk * 4));
  a.mu_ready = reinterpret_cast<uint32_t*>(take(nk * 4));
  a.ctl = reinterpret_cast<uint32_t*>(take(16));
  a.entries = reinterpret_cast<uint32_t*>(take(3 * ns * 4 + 64));
  if (a.center) {
    const size_t nchunks = (size_t(a.N) + kTR - 1) / kTR;
    a.mean_part = reinterpret_cast<float*>(take(nk * nchunks * a.d * 4));
    a.mu = reinterpret_cast<float*>(take(nk * a.d * 4));
  } else {
    a.mean_part = nullptr;
    a.mu = nullptr;
  }
}

// ---- fixed scratch for callers that cannot allocate -------------------------
// attnq_prepare_static uses this file-scope array instead of a caller
// workspace.  Every GPU that loads the library keeps it until the process
// exits; all calls share it.  Its device address is looked up once per device
// (host code must not pass the symbol itself to a kernel: on the host it is
// only a stand-in).
static __device__ __align__(256) unsigned char g_prepare_scratch[kStaticScratchBytes];

cudaError_t static_scratch_address(void** out) {
  static std::mutex mu;
  static void* addr[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_prepare_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *out = addr[dev];
  return cudaSuccess;
}

cudaError_t launch_prepare(const PrepareArgs& a, cudaStream_t s) {
  if (a.d == 128) return a.bf16 ? run<128, true>(a, s) : run<128, false>(a, s);
  return a.bf16 ? run<64, true>(a, s) : run<64, false>(a, s);
}

}  // namespace attnq
