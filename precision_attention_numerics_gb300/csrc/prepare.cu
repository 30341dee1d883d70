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
// An entry's slice is cut into items of four 128-row tiles; CTAs claim items
// in list order with an atomic ticket.  The list puts each slice's A entry a
// few steps after its M entry and its C entry a few steps after its A entry,
// so a slice's second and third reads come from L2, and a pass waits only on
// entries claimed before it (the finisher of a slice's last A tile publishes
// its scale; the finisher of a K slice's last M tile publishes its mean): the
// earliest unfinished item never waits, so the kernel cannot deadlock, and
// it needs no co-residency.
//
// CTA: warp 8 claims items and streams their tiles into a ring of shared
// memory stages with TMA (128-byte swizzle, rows beyond N read as zero;
// warps 9-11 only complete its warpgroup for the register split);
// warps 0-3 and 4-7 are two consumer groups that take alternate tiles, one
// row per thread.  A row of d values is held as d/2 packed pairs
// (x_j, x_{j+d/2}), so stages h = 1 .. d/4 of the FWHT are packed f32x2
// adds and subtracts and stage d/2 adds the two halves of each pair.  Casts
// in the natural layout leave from registers (each thread stores its row);
// V in the transposed layout goes channel-major through shared memory and
// leaves by TMA store.
#include <cuda_bf16.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace attnq {
namespace {

constexpr int kTR = 128;           // rows per tile = tokens per mean-key chunk
constexpr int kTilesPerItem = 16;  // tiles per claimed item
constexpr int kGroups = 2;         // consumer groups (128 threads, one row each)
constexpr int kFlowThreads = 384;  // two consumer warpgroups + a warpgroup whose warp 8 is the producer
// Register split: launched at 168 per thread (384 x 168 = 64,512); the consumer
// warpgroups rise to 232 (a row of 128 fp32 values and the FWHT's working set
// fit without spilling), the producer's warpgroup drops to 40:
// 2 x 128 x 232 + 128 x 40 = 64,512.
constexpr uint32_t kConsumerRegs = 232, kProducerRegs = 40;
static_assert(2 * 128 * kConsumerRegs + 128 * kProducerRegs <= kFlowThreads * 168, "register split");
constexpr int kLagA = 4, kLagC = 3;  // list steps from a slice's M entry to its A entry, and A to C
constexpr uint32_t KIND_M = 0u, KIND_A = 1u, KIND_C = 2u, KIND_DONE = 3u;
constexpr uint32_t CTL_TICKET = 0, CTL_ABORT = 1, CTL_ENTRIES = 2;

template <int D, bool BF16>
struct FlowCfg {
  static constexpr int ES = BF16 ? 2 : 4;
  static constexpr int ROW_BYTES = D * ES;
  static constexpr int NB = ROW_BYTES / 128;      // 128-byte boxes per input row
  static constexpr int SB = kTR * ROW_BYTES;      // input stage
  static constexpr int OB = kTR * D;              // output buffer (codes)
  static constexpr int NST0 = (225280 - 2 * kGroups * OB - 4096) / SB;
  // A multiple of kGroups: tile n goes to stage n % NST and to group
  // n % kGroups, so every stage serves one group only and its phases are
  // consumed in order.  A stage shared by two groups would let a group whose
  // tile is k phases ahead mistake an older phase of the same parity for it.
  static constexpr int NST1 = NST0 > 6 ? 6 : NST0;
  static constexpr int NST = NST1 - NST1 % kGroups;
  static constexpr int WORDS = BF16 ? D / 2 : D;  // 32-bit input words per row
  static constexpr size_t SMEM = 1024 + size_t(NST) * SB + size_t(2 * kGroups) * OB + 16 * NST + 16 * NST +
                                 4 * WORDS + 8 * (D / 2) + kGroups * (8 * (D / 2) + 64);
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
    a.s_ready[i] = 0u;
  }
  for (int i = threadIdx.x; i < nk; i += blockDim.x) {
    a.m_done[i] = 0u;
    a.mu_ready[i] = 0u;
  }
  if (!a.center && a.k_mean)
    for (int i = threadIdx.x; i < nk * a.d; i += blockDim.x) a.k_mean[i] = 0.0f;
  if (threadIdx.x == 0) {
    // slice order: K first (their M entries lead), then V, then Q
    auto order = [&](int t) { return t < nk ? nq + t : (t < 2 * nk ? nq + t : t - 2 * nk); };
    uint32_t e = 0;
    for (int t = 0; t < ns + kLagA + kLagC; ++t) {
      const int tc = t - kLagA - kLagC, ta = t - kLagA;
      if (tc >= 0 && tc < ns) a.entries[e++] = (KIND_C << 30) | uint32_t(order(tc));
      if (ta >= 0 && ta < ns) a.entries[e++] = (KIND_A << 30) | uint32_t(order(ta));
      if (a.center && t < nk) a.entries[e++] = (KIND_M << 30) | uint32_t(order(t));
    }
    a.ctl[CTL_TICKET] = 0u;
    a.ctl[CTL_ABORT] = 0u;
    a.ctl[CTL_ENTRIES] = e;
  }
}

struct Flow {
  PrepareArgs a;
  int tiles_per_slice, items_per_slice;
};

__device__ __forceinline__ void raise_abort(const PrepareArgs& a) {
  if (atomicExch(a.ctl + CTL_ABORT, 1u) == 0u) atomicOr(a.status, DEV_TIMEOUT);
}

__device__ __forceinline__ bool aborted(const PrepareArgs& a) {
  return *reinterpret_cast<volatile uint32_t*>(a.ctl + CTL_ABORT) != 0u;
}

// Bounded wait on an mbarrier phase (one thread).
__device__ __forceinline__ bool bar_wait(const PrepareArgs& a, uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  const uint32_t hint = a.wait_ns < 20000ull ? uint32_t(a.wait_ns) : 20000u;  // never sleep past the limit
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, hint)) return true;
    if (aborted(a) || globaltimer_ns() - t0 > a.wait_ns) return false;
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

// qs = 448/amax, descale = amax/448 (IEEE division); amax = 0 -> 1, 1.
__device__ void publish_scale(const PrepareArgs& a, int s) {
  const uint32_t bits = atomicOr(a.amax_bits + s, 0u);
  float qs, ds;
  if (bits >= 0x7F800000u) {  // a NaN or an infinity reached the slice
    atomicOr(a.status, DEV_NONFINITE);
    qs = 0.0f;
    ds = __uint_as_float(0x7FC00000u);
  } else if (bits == 0u) {
    qs = 1.0f;
    ds = 1.0f;
  } else {
    const float amax = __uint_as_float(bits);
    qs = __fdiv_rn(448.0f, amax);
    ds = __fdiv_rn(amax, 448.0f);
  }
  a.qs[s] = qs;
  const SliceRef r = slice_ref(a, s);
  (r.tensor == 0 ? a.q_ds : r.tensor == 1 ? a.k_ds : a.v_ds)[r.local] = ds;
  __threadfence();
  flag_set(a.s_ready + s);
}

// ---- producer -------------------------------------------------------------
template <int D, bool BF16>
__device__ void producer(const Flow& f, const CUtensorMap* const* in_maps, uint8_t* stages, TileMeta* meta,
                         uint64_t* full, uint64_t* empty) {
  using C = FlowCfg<D, BF16>;
  const PrepareArgs& a = f.a;
  const uint32_t total = a.ctl[CTL_ENTRIES] * uint32_t(f.items_per_slice);
  uint32_t n = 0;  // tiles pushed
  bool ok = true;
  for (;;) {
    if (aborted(a)) { ok = false; break; }
    const uint32_t t = atomicAdd(a.ctl + CTL_TICKET, 1u);
    if (t >= total) break;
    const uint32_t ent = a.entries[t / uint32_t(f.items_per_slice)];
    const uint32_t item = t % uint32_t(f.items_per_slice);
    const uint32_t kind = ent >> 30, s = ent & 0x3FFFFFFFu;
    const SliceRef r = slice_ref(a, int(s));
    const CUtensorMap* map = in_maps[r.tensor];
    const int row_begin = int(item) * kTR * kTilesPerItem;
    const int nt = min(kTilesPerItem, (a.N - row_begin + kTR - 1) / kTR);
    for (int tl = 0; tl < nt && ok; ++tl, ++n) {
      const int row0 = row_begin + tl * kTR;
      const uint32_t st = n % C::NST, ph = (n / C::NST) & 1u;
      if (!bar_wait(a, empty + st, ph ^ 1u)) { ok = false; break; }
      // tiles alternate between the groups: tl + 2 is this group's next tile
      meta[st] = TileMeta{kind, s, uint32_t(row0), tl + 2 >= nt ? 1u : 0u};
      mbar_arrive_expect_tx(full + st, C::SB);
#pragma unroll
      for (int b = 0; b < C::NB; ++b)
        tma_load_3d(stages + size_t(st) * C::SB + b * (kTR * 128), map, full + st, b * 128, row0, r.local);
    }
    if (!ok) break;
  }
  if (ok) {
    // one end marker per consumer group (tiles alternate between the groups)
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

// Row r of an input stage as packed pairs P[j] = (x_j, x_{j+D/2}); with
// `flip`, the sign flip is applied as a sign-bit XOR on the raw values (exact,
// signed zeros included) - only for rows that are not centred, since the
// flip must follow the centring.
template <int D, bool BF16>
__device__ __forceinline__ void load_row(const uint8_t* stage, int r, const uint32_t* smask, bool flip,
                                         uint64_t (&P)[D / 2]) {
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
    if (flip) {
      const uint4 m = *reinterpret_cast<const uint4*>(smask + 4 * q);
      u.x ^= m.x; u.y ^= m.y; u.z ^= m.z; u.w ^= m.w;
    }
    return u;
  };
  // chunk q holds elements PER*q ..; it pairs with chunk q + CH/2 (elements + D/2)
#pragma unroll
  for (int q = 0; q < CH / 2; ++q) {
    const uint4 ua = chunk(q), ub = chunk(q + CH / 2);
    const uint32_t wa[4] = {ua.x, ua.y, ua.z, ua.w}, wb[4] = {ub.x, ub.y, ub.z, ub.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if constexpr (BF16) {
        P[PER * q + 2 * i] = pack2(__uint_as_float(wa[i] << 16), __uint_as_float(wb[i] << 16));
        P[PER * q + 2 * i + 1] = pack2(__uint_as_float(wa[i] & 0xFFFF0000u), __uint_as_float(wb[i] & 0xFFFF0000u));
      } else {
        P[PER * q + i] = pack2(__uint_as_float(wa[i]), __uint_as_float(wb[i]));
      }
    }
  }
}

// Centre (x + (-mu), one rounding), then for centred rows the sign flip
// (a sign-bit XOR on the packed pair), then the unnormalised FWHT.  The
// order is the method's: s * (x - mu) keeps the sign of a zero difference
// that s*x - s*mu would lose.
template <int D>
__device__ __forceinline__ void transform(uint64_t (&P)[D / 2], bool center, const uint64_t* nmu,
                                          const uint64_t* pmask, bool rotate) {
  if (center) {
#pragma unroll
    for (int j = 0; j < D / 2; ++j) P[j] = fadd2(P[j], nmu[j]);
    if (rotate) {
#pragma unroll
      for (int j = 0; j < D / 2; j += 2) {
        const uint4 m = *reinterpret_cast<const uint4*>(pmask + j);
        P[j] ^= (uint64_t(m.y) << 32) | m.x;
        P[j + 1] ^= (uint64_t(m.w) << 32) | m.z;
      }
    }
  }
  if (rotate) {
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
#pragma unroll
    for (int j = 0; j < D / 2; ++j) {
      float lo, hi;
      unpack2(P[j], lo, hi);
      P[j] = pack2(__fadd_rn(lo, hi), __fsub_rn(lo, hi));
    }
  }
}

template <int D>
__device__ __forceinline__ uint32_t row_amax_bits(const uint64_t (&P)[D / 2]) {
  float m[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int j = 0; j < D / 2; ++j) {
    float lo, hi;
    unpack2(P[j], lo, hi);
    m[(2 * j) & 3] = max_nan(m[(2 * j) & 3], fabsf(lo));
    m[(2 * j + 1) & 3] = max_nan(m[(2 * j + 1) & 3], fabsf(hi));
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

// ---- the persistent kernel ----------------------------------------------------
template <int D, bool BF16>
__global__ void __launch_bounds__(kFlowThreads, 1)
    k_prepare(const __grid_constant__ CUtensorMap in_q, const __grid_constant__ CUtensorMap in_k,
              const __grid_constant__ CUtensorMap in_v, const __grid_constant__ CUtensorMap out_vt, const Flow f) {
  using C = FlowCfg<D, BF16>;
  const PrepareArgs& a = f.a;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = sm;
  uint8_t* outb = stages + size_t(C::NST) * C::SB;               // [group][2]
  TileMeta* meta = reinterpret_cast<TileMeta*>(outb + size_t(2 * kGroups) * C::OB);
  uint64_t* full = reinterpret_cast<uint64_t*>(meta + C::NST);
  uint64_t* empty = full + C::NST;
  uint32_t* smask = reinterpret_cast<uint32_t*>(empty + C::NST);  // sign-bit mask per input word
  uint64_t* pmask = reinterpret_cast<uint64_t*>(smask + C::WORDS);  // sign-bit masks of the pairs (x_j, x_{j+D/2})
  uint8_t* gbase = reinterpret_cast<uint8_t*>(pmask + D / 2);      // per group: nmu[D/2] (8 B), 64 B scratch

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 4);  // one arrival per consumer warp
    }
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
  }
  for (int j = threadIdx.x; j < D / 2; j += blockDim.x) {
    const uint64_t lo = (a.rotate && a.signs[j] < 0) ? 0x80000000ull : 0ull;
    const uint64_t hi = (a.rotate && a.signs[j + D / 2] < 0) ? 0x80000000ull : 0ull;
    pmask[j] = lo | (hi << 32);
  }
  __syncthreads();

  if (warp >= 4 * kGroups) {
    regs_decrease<kProducerRegs>();
    if (warp == 4 * kGroups && lane == 0) {
      tma_prefetch_desc(&in_q);
      tma_prefetch_desc(&in_k);
      tma_prefetch_desc(&in_v);
      const CUtensorMap* maps[3] = {&in_q, &in_k, &in_v};
      producer<D, BF16>(f, maps, stages, meta, full, empty);
    }
    return;
  }

  // consumer group g: tiles g, g + 2, g + 4, ... of the ring sequence
  regs_increase<kConsumerRegs>();
  const int g = warp >> 2, r = threadIdx.x & 127;
  uint64_t* nmu = reinterpret_cast<uint64_t*>(gbase + g * (8 * (D / 2) + 64));
  uint32_t* gscr = reinterpret_cast<uint32_t*>(nmu + D / 2);  // [0..3] warp maxima, [4] verdict
  const uint32_t gbar = 1u + uint32_t(g);
  int mu_bg = -1;      // K slice whose -(s*mu) is in nmu
  int qs_slice = -1;   // slice whose scale is in qs
  float qs = 0.0f;
  uint32_t cbuf = 0;   // output buffer parity
  bool stored = false;
  bool ok = true;
  uint32_t run_max = 0;   // this warp's amax over the group's tiles of the current item
  uint32_t run_tiles = 0; // tiles of the current item this group has finished
  // group-uniform verdict of thread 0's wait
  auto group_verdict = [&](bool mine) -> bool {
    if (r == 0) gscr[4] = mine ? 1u : 0u;
    named_bar_sync(gbar, 128);
    const bool v = gscr[4] != 0u;
    named_bar_sync(gbar, 128);
    return v;
  };
  for (uint32_t j = 0;; ++j) {
    const uint32_t n = 2u * j + uint32_t(g);
    const uint32_t st = n % C::NST, ph = (n / C::NST) & 1u;
    bool got = true;
    if (!__all_sync(0xffffffffu, mbar_try_wait(full + st, ph))) {
      uint32_t v = 0;
      if (lane == 0) v = bar_wait(a, full + st, ph) ? 1u : 0u;
      got = __shfl_sync(0xffffffffu, v, 0) != 0u;
    }
    // the store that last read the output buffer a cast tile would use (two
    // casts ago) must be done with it before the group's next barrier
    if (got && r == 0 && stored && meta[st].kind == KIND_C && a.vt &&
        slice_ref(a, int(meta[st].slice)).tensor == 2)
      bulk_wait_read<1>();
    if (!group_verdict(got)) { ok = false; break; }
    const TileMeta tm = meta[st];
    if (tm.kind == KIND_DONE) break;
    const uint8_t* stage = stages + size_t(st) * C::SB;
    const int s = int(tm.slice);
    const SliceRef sr = slice_ref(a, s);
    const int row0 = int(tm.row0);
    const bool valid = row0 + r < a.N;
    const bool qk = sr.tensor < 2;
    const bool rotate = a.rotate && qk, center = a.center && sr.tensor == 1;

    if (tm.kind == KIND_M) {
      // chunk sum of each channel over the tile's tokens, in token order
      const int rows = min(kTR, a.N - row0);
      if (r < D) {
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
      ++run_tiles;
      if (!tm.last) continue;
      // the group's chunks of this item are written: count them (one atomic
      // per item), and the group that completes the slice computes its mean
      if (r < D) __threadfence();
      named_bar_sync(gbar, 128);
      if (r == 0)
        gscr[4] = (atomicAdd(a.m_done + sr.local, run_tiles) + run_tiles == uint32_t(f.tiles_per_slice)) ? 1u : 0u;
      run_tiles = 0;
      named_bar_sync(gbar, 128);
      if (gscr[4]) {
        // last chunks of this K slice: mean = (chunk sums in order) / N
        __threadfence();
        if (r < D) {
          float total = 0.0f;
          for (int k = 0; k < f.tiles_per_slice; ++k)
            total = __fadd_rn(total, __ldcg(a.mean_part + (int64_t(sr.local) * f.tiles_per_slice + k) * D + r));
          const float mu = __fdiv_rn(total, float(a.N));
          a.mu[sr.local * D + r] = mu;
          if (a.k_mean) a.k_mean[sr.local * D + r] = mu;
        }
        __threadfence();
        named_bar_sync(gbar, 128);
        if (r == 0) flag_set(a.mu_ready + sr.local);
      }
      named_bar_sync(gbar, 128);
      continue;
    }

    // centred K needs the slice's mean key
    if (center && mu_bg != sr.local) {
      bool have = true;
      if (r == 0) have = flag_wait(a, a.mu_ready + sr.local);
      if (!group_verdict(have)) { ok = false; break; }
      if (r < D / 2) nmu[r] = pack2(-__ldcg(a.mu + sr.local * D + r), -__ldcg(a.mu + sr.local * D + r + D / 2));
      named_bar_sync(gbar, 128);
      mu_bg = sr.local;
    }

    uint64_t P[D / 2];
    load_row<D, BF16>(stage, r, smask, rotate && !center, P);
    __syncwarp();
    if (lane == 0) mbar_arrive(empty + st);  // the row is in registers
    transform<D>(P, center, nmu, pmask, rotate);

    if (tm.kind == KIND_A) {
      uint32_t m = valid ? row_amax_bits<D>(P) : 0u;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
      run_max = max(run_max, m);
      ++run_tiles;
      if (!tm.last) continue;
      // end of the group's share of the item: one max and one count per item
      if (lane == 0) gscr[warp & 3] = run_max;
      named_bar_sync(gbar, 128);
      if (r == 0) {
        const uint32_t mm = max(max(gscr[0], gscr[1]), max(gscr[2], gscr[3]));
        if (mm) atomicMax(a.amax_bits + s, mm);
        __threadfence();
        if (atomicAdd(a.a_done + s, run_tiles) + run_tiles == uint32_t(f.tiles_per_slice)) {
          __threadfence();
          publish_scale(a, s);
        }
      }
      run_max = 0;
      run_tiles = 0;
      continue;
    }

    // KIND_C: the slice's scale, then codes through shared memory to TMA
    if (qs_slice != s) {
      bool have = true;
      if (r == 0) have = flag_wait(a, a.s_ready + s);
      if (!group_verdict(have)) { ok = false; break; }
      qs = __ldcg(a.qs + s);
      qs_slice = s;
    }
    uint32_t cw[D / 4];
    row_codes<D>(P, qs, cw);
    if (!(sr.tensor == 2 && a.vt)) {
      // natural layout: each thread writes its own row's codes (16-byte stores)
      if (valid) {
        uint4* dst = reinterpret_cast<uint4*>((sr.tensor == 0 ? a.q8 : sr.tensor == 1 ? a.k8 : a.v8) +
                                              (int64_t(sr.local) * a.N + row0 + r) * D);
#pragma unroll
        for (int c = 0; c < D / 16; ++c) dst[c] = make_uint4(cw[4 * c], cw[4 * c + 1], cw[4 * c + 2], cw[4 * c + 3]);
      }
      continue;
    }
    // V^T: channel-major tile through shared memory (byte (channel c, token r)
    // of a [D][128] tile, 128-byte swizzle), then one TMA store
    uint8_t* ob = outb + size_t(2 * g + cbuf) * C::OB;
#pragma unroll
    for (int c = 0; c < D; ++c) ob[sw128(c, r >> 4) + (r & 15)] = uint8_t((cw[c >> 2] >> (8 * (c & 3))) & 0xFFu);
    fence_proxy_async_smem();
    named_bar_sync(gbar, 128);
    if (r == 0) {
      tma_store_3d(&out_vt, ob, row0, 0, sr.local);
      bulk_commit();
    }
    stored = true;
    cbuf ^= 1u;
  }
  if (!ok) raise_abort(a);
  if (r == 0 && stored) bulk_wait_all();
}

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

template <int D, bool BF16>
cudaError_t run(const PrepareArgs& a, cudaStream_t st) {
  using C = FlowCfg<D, BF16>;
  const int nq = a.B * a.Hq, nk = a.B * a.Hkv;
  const uint64_t rb = uint64_t(D) * C::ES;
  CUtensorMap in_q, in_k, in_v, out_vt;
  if (encode_tiled_3d(&in_q, a.Q, rb, a.N, nq, rb, rb * a.N, 128, kTR, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
      encode_tiled_3d(&in_k, a.K, rb, a.N, nk, rb, rb * a.N, 128, kTR, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
      encode_tiled_3d(&in_v, a.V, rb, a.N, nk, rb, rb * a.N, 128, kTR, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  if (a.vt) {
    if (encode_tiled_3d(&out_vt, a.v8, uint64_t(a.ldv), D, nk, uint64_t(a.ldv), uint64_t(a.ldv) * D, kTR, D,
                        CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  } else {
    out_vt = in_v;  // not used: casts write the natural layout from registers
  }
  Flow f;
  f.a = a;
  f.tiles_per_slice = (a.N + kTR - 1) / kTR;
  f.items_per_slice = (f.tiles_per_slice + kTilesPerItem - 1) / kTilesPerItem;
  k_flow_init<<<1, 256, 0, st>>>(a);
  auto kern = k_prepare<D, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(C::SMEM));
  if (e != cudaSuccess) return e;
  const int grid = a.num_sms > 0 ? a.num_sms : 1;
  kern<<<grid, kFlowThreads, C::SMEM, st>>>(in_q, in_k, in_v, out_vt, f);
  return cudaGetLastError();
}

}  // namespace

size_t prepare_workspace_bytes(int B, int Hq, int Hkv, int N, int d, int center) {
  const size_t ns = size_t(B) * Hq + 2 * size_t(B) * Hkv, nk = size_t(B) * Hkv;
  size_t bytes = 4 * align256(ns * 4) + 2 * align256(nk * 4) + align256(16) + align256(3 * ns * 4 + 64);
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
  a.qs = reinterpret_cast<float*>(take(ns * 4));
  a.a_done = reinterpret_cast<uint32_t*>(take(ns * 4));
  a.s_ready = reinterpret_cast<uint32_t*>(take(ns * 4));
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
