// CPU oracle for causal FP8 (E4M3) attention with the numerics options of the
// attention-numerics pages.  TEST INFRASTRUCTURE ONLY: the tests, the smoke
// check and the benchmark's CPU-baseline leg call it; the product path never
// does.  It shares no code, header, table or constant with the CUDA library.
//
// Plain, slow, obviously correct: one loop per definition, double or float
// exactly where the method fixes it.  Compile without fast-math and with
// -ffp-contract=off so every float operation rounds once, in program order.
//
// Sources (page titles and sections):
//  [AN]  "attention-numerics" project page - method and kernel settings: per
//        (batch, head) full-sequence Q/K/V scales; rotation of Q and K (never
//        V); mean-key subtraction preserves exact attention.
//  [RR]  "A rounding problem, not a rotation problem" - 01 / Synthetic
//        illustration: one maximum-based FP8 scale per tensor, fixed
//        random-sign Hadamard, E4M3FN round-to-nearest-even saturating at
//        +-448, mean subtraction before rotation; 02 / Measured heads:
//        log(1 + relative Frobenius error) per head.
//  [PC]  "Technische Samenvatting: P-Cast Precisie in FP8 Attention" - sec. 1
//        (online softmax over KV blocks forward or reverse; P multiplied by a
//        static S before the E4M3 cast and divided out in the epilogue),
//        sec. 2 (round-to-zero threshold 2^-10), sec. 3-4 (kernel-faithful
//        simulation with Q, K, V in FP32 and only P cast).
//
// Readings where the pages are silent are stated at each function.
//
// Parity pins for every function live in tests/test_oracle_*.py.

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

// ---------------------------------------------------------------------------
// E4M3FN, written from the format definition [RR]: 1 sign bit, 4 exponent
// bits (bias 7), 3 mantissa bits; exponent field 0 holds subnormals m * 2^-9;
// S.1111.111 is NaN; there are no infinities; the largest finite value is
// S.1111.110 = 448.
// ---------------------------------------------------------------------------

double e4m3_value(unsigned code) {
  const unsigned s = (code >> 7) & 1u, e = (code >> 3) & 15u, m = code & 7u;
  if (e == 15u && m == 7u) return std::numeric_limits<double>::quiet_NaN();
  double mag = (e == 0u) ? std::ldexp(double(m), -9) : std::ldexp(1.0 + double(m) / 8.0, int(e) - 7);
  return s ? -mag : mag;
}

struct E4M3Table {
  double pos[127];   // values of codes 0x00 .. 0x7E, ascending
  double dec[256];
  E4M3Table() {
    for (unsigned c = 0; c < 256; ++c) dec[c] = e4m3_value(c);
    for (unsigned c = 0; c < 127; ++c) pos[c] = dec[c];
  }
};
const E4M3Table& tab() { static E4M3Table t; return t; }

// Round-to-nearest-even of the exact real value x onto the E4M3 grid,
// saturating: |x| > 448 (including infinity) gives +-448 [RR]; NaN gives 0x7F.
// The sign survives a round to zero (-tiny -> 0x80).
uint8_t e4m3_encode(float x) {
  if (std::isnan(x)) return 0x7F;
  const unsigned sign = std::signbit(x) ? 0x80u : 0u;
  const double a = std::fabs(double(x));
  const double* v = tab().pos;
  if (a >= v[126]) return uint8_t(sign | 126u);
  // largest k with v[k] <= a
  int lo = 0, hi = 126;
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (v[mid] <= a) lo = mid; else hi = mid;
  }
  unsigned k = unsigned(lo);
  if (v[k] == a) return uint8_t(sign | k);
  // compare 2a with v[k] + v[k+1]: both sides exact in double
  const double twice = 2.0 * a, mid2 = v[k] + v[k + 1];
  unsigned r;
  if (twice < mid2) r = k;
  else if (twice > mid2) r = k + 1;
  else r = (k % 2u == 0u) ? k : k + 1;
  return uint8_t(sign | r);
}

inline double dec(uint8_t c) { return tab().dec[c]; }

// ---------------------------------------------------------------------------
// Symmetric INT8 code of a float (the Q.K format of the INT8-QK / FP8-PV
// kernel that the "attention-numerics" page, method and kernel settings,
// runs): the nearest integer, ties to even, saturated to [-127, 127].  The
// page names only the format; -128 is left unused so the code range is
// symmetric like the max-based scale that feeds it.  NaN gives 0 (non-finite
// inputs are rejected before any cast).
// ---------------------------------------------------------------------------
int8_t int8_encode(float y) {
  if (std::isnan(y)) return 0;
  const double a = double(y);
  if (a >= 127.0) return 127;
  if (a <= -127.0) return -127;
  const double f = std::floor(a);
  const double frac = a - f;  // exact: a and f are within 2^8 of each other
  long k = long(f);
  if (frac > 0.5 || (frac == 0.5 && k % 2 != 0)) k += 1;
  return int8_t(k);
}

// bf16 bit pattern -> float (exact)
inline float bf16_to_float(uint16_t u) {
  uint32_t b = uint32_t(u) << 16;
  float f;
  std::memcpy(&f, &b, 4);
  return f;
}

// double -> bf16 bit pattern, round to nearest even, one rounding.
uint16_t double_to_bf16(double x) {
  if (std::isnan(x)) return 0x7FC0;
  const uint16_t sign = std::signbit(x) ? 0x8000 : 0;
  double a = std::fabs(x);
  if (a == 0.0) return sign;
  // bf16: 8 significant bits, exponents -126..127, subnormals step 2^-133
  int e;
  std::frexp(a, &e);          // a = f * 2^e, f in [0.5, 1)
  int exp_unbiased = e - 1;   // a in [2^(e-1), 2^e)
  int q = std::max(exp_unbiased, -126) - 7;  // quantum
  double scaled = std::ldexp(a, -q);
  double r = std::nearbyint(scaled);  // default rounding mode: nearest even
  double y = std::ldexp(r, q);
  if (y >= std::ldexp(1.0, 128)) return uint16_t(sign | 0x7F80);  // overflow -> inf
  float f = float(y);  // exact: y has <= 8 significant bits
  uint32_t b;
  std::memcpy(&b, &f, 4);
  return uint16_t(sign | ((b >> 16) & 0x7FFF));
}

inline bool finite_f(float x) { return std::isfinite(x); }

// Unnormalised fast Walsh-Hadamard transform in float, stages h = 1, 2, ...,
// d/2, pairs (j, j+h) -> (a+b, a-b).  [AN] and [RR] name the transform but not
// its normalisation; the unnormalised form is exact up to float rounding and
// its factor d (a power of two) is folded into the logit scale.
void fwht(float* x, int d) {
  for (int h = 1; h < d; h <<= 1)
    for (int i = 0; i < d; i += 2 * h)
      for (int j = i; j < i + h; ++j) {
        float a = x[j], b = x[j + h];
        x[j] = a + b;
        x[j + h] = a - b;
      }
}

template <class F>
void parallel_for(int64_t n, int threads, F&& f) {
  if (threads <= 1 || n <= 1) {
    for (int64_t i = 0; i < n; ++i) f(i);
    return;
  }
  std::atomic<int64_t> next(0);
  std::vector<std::thread> pool;
  int t = int(std::min<int64_t>(threads, n));
  for (int w = 0; w < t; ++w)
    pool.emplace_back([&]() {
      for (;;) {
        int64_t i = next.fetch_add(1);
        if (i >= n) break;
        f(i);
      }
    });
  for (auto& th : pool) th.join();
}

int g_threads = 0;
int nthreads() {
  if (g_threads > 0) return g_threads;
  unsigned h = std::thread::hardware_concurrency();
  return h ? int(h) : 1;
}

constexpr double LOG2E = 1.4426950408889634073599246810018921;  // 1/ln 2

}  // namespace

extern "C" {

enum { ORC_OK = 0, ORC_EINVAL = 1, ORC_ENONFINITE = 4 };
enum { ORC_ROTATE = 1u, ORC_CENTER_K = 2u, ORC_TILE_SCALES = 8u, ORC_I8QK = 16u };
// Scale tile of the per-tile variant: 128 consecutive tokens of one (batch,
// head), aligned at token 0.
constexpr int ORC_SCALE_TILE = 128;
enum { ORC_F32 = 0, ORC_BF16 = 1 };

void orc_set_threads(int t) { g_threads = t; }
int orc_get_threads(void) { return nthreads(); }

double orc_e4m3_decode(uint8_t c) { return dec(c); }
uint8_t orc_e4m3_encode(float x) { return e4m3_encode(x); }
void orc_int8_encode_array(const float* x, int8_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = int8_encode(x[i]);
}

void orc_e4m3_encode_array(const float* x, uint8_t* out, int64_t n) {
  const int64_t blk = 1 << 20;
  parallel_for((n + blk - 1) / blk, nthreads(), [&](int64_t b) {
    int64_t lo = b * blk, hi = std::min(n, lo + blk);
    for (int64_t i = lo; i < hi; ++i) out[i] = e4m3_encode(x[i]);
  });
}

// Encode every float32 bit pattern in [start, start + count).
void orc_e4m3_encode_bits_range(uint64_t start, int64_t count, uint8_t* out) {
  const int64_t blk = 1 << 20;
  parallel_for((count + blk - 1) / blk, nthreads(), [&](int64_t b) {
    int64_t lo = b * blk, hi = std::min(count, lo + blk);
    for (int64_t i = lo; i < hi; ++i) {
      uint32_t bits = uint32_t(start + uint64_t(i));
      float f;
      std::memcpy(&f, &bits, 4);
      out[i] = e4m3_encode(f);
    }
  });
}

void orc_double_to_bf16_array(const double* x, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = double_to_bf16(x[i]);
}

void orc_fwht(float* x, int d) { fwht(x, d); }

// ---------------------------------------------------------------------------
// Operand preparation [AN], [RR]:
//   1. upcast to float (bf16 -> float is exact);
//   2. K only, if CENTER_K: subtract the full-sequence mean key of its
//      (batch, KV head), computed before rotation [RR];
//   3. if ROTATE: multiply by the fixed sign vector and apply the FWHT, Q and
//      K only, never V [AN];
//   4. one scale per (batch, head) and tensor over the whole sequence [AN]:
//      amax = max |x|, qs = 448/amax, descale = amax/448 (float, IEEE
//      division); amax == 0 gives qs = descale = 1;
//   5. x8 = E4M3(fl32(x * qs)).
// Causal-prefix statistics (the "attention-numerics" page, limitations, notes
// that full-sequence means and scales see future tokens; it defines no
// generation-safe form, so the plainest one is taken): with stat_len = P,
// 0 < P <= N, the mean key and the per-(batch, head) amax are taken over the
// first P tokens of the slice only, and all N tokens are centred and cast with
// them; a later value above the prefix amax saturates at +-448 by the cast's
// rule.  P = N (or 0) is the full-sequence preparation.  Per-tile scales are
// local to their tile and do not change.  The non-finite check still covers
// every token.
// Reading of the mean (pages silent on its arithmetic): float sums in a fixed
// order - per channel, each 128-token chunk summed in token order starting
// from 0, then the chunk sums added in chunk order - and one IEEE division by
// N.  Any vector subtracted from every key leaves exact attention unchanged,
// so the mean needs no more precision than float; the fixed order makes it
// reproducible bit for bit.
// Outputs are in the natural [B, H, N, d] layout.
// ---------------------------------------------------------------------------

static float load_in(const void* p, int dtype, int64_t i) {
  return dtype == ORC_BF16 ? bf16_to_float(static_cast<const uint16_t*>(p)[i])
                           : static_cast<const float*>(p)[i];
}

int orc_mean_key(int N, int d, int dtype, const void* K_head, float* mu) {
  for (int c = 0; c < d; ++c) {
    float total = 0.0f;
    for (int j0 = 0; j0 < N; j0 += 128) {
      float part = 0.0f;
      for (int j = j0; j < std::min(N, j0 + 128); ++j) part = part + load_in(K_head, dtype, int64_t(j) * d + c);
      total = total + part;
    }
    mu[c] = total / float(N);
  }
  return ORC_OK;
}

// qs = top/amax and descale = amax/top (IEEE division), top = 448 for E4M3
// and 127 for INT8 codes; amax = 0 gives 1, 1.
static void scale_of(float amax, float top, float* qs, float* ds) {
  *qs = 1.0f;
  *ds = 1.0f;
  if (amax > 0.0f) {
    *qs = top / amax;
    *ds = amax / top;
  }
}

// One tensor slice [N, d] of one (batch, head): transform, scale, cast.  With
// `per_tile`, every ORC_SCALE_TILE-row tile gets its own maximum-based scale
// (the emulator's per-tile scales that the "attention-numerics" page, method
// and kernel settings, contrasts with the full-sequence API scales) and
// descale[t] is tile t's; otherwise one scale for the slice.
// Without `per_tile` the slice's amax is taken over its first P tokens.  With
// `int8` the codes are symmetric INT8 (scale top 127, int8_encode) stored as
// two's-complement bytes, otherwise E4M3 (top 448).
static int prepare_slice(int N, int P, int d, int dtype, const void* X, bool rotate, const int8_t* signs,
                         const float* mu /* or null */, uint8_t* x8, float* descale, float* transformed_out,
                         bool per_tile = false, bool int8 = false) {
  std::vector<float> t(size_t(N) * d);
  bool finite = true;
  for (int j = 0; j < N; ++j) {
    float* r = &t[size_t(j) * d];
    for (int c = 0; c < d; ++c) {
      float x = load_in(X, dtype, int64_t(j) * d + c);
      if (!finite_f(x)) finite = false;
      if (mu) x = x - mu[c];
      if (rotate) x = signs[c] < 0 ? -x : x;
      r[c] = x;
    }
    if (rotate) fwht(r, d);
  }
  if (!finite) return ORC_ENONFINITE;
  for (float x : t)
    if (!finite_f(x)) return ORC_ENONFINITE;
  const int rows_per_scale = per_tile ? ORC_SCALE_TILE : N;
  for (int j0 = 0, tile = 0; j0 < N; j0 += rows_per_scale, ++tile) {
    const size_t i0 = size_t(j0) * d, i1 = size_t(std::min(N, j0 + rows_per_scale)) * d;
    const size_t a1 = per_tile ? i1 : size_t(P) * d;  // rows the amax is taken over
    float amax = 0.0f;
    for (size_t i = i0; i < a1; ++i) amax = std::max(amax, std::fabs(t[i]));
    float qs, ds;
    scale_of(amax, int8 ? 127.0f : 448.0f, &qs, &ds);
    descale[tile] = ds;
    for (size_t i = i0; i < i1; ++i) {
      const float y = t[i] * qs;
      x8[i] = int8 ? uint8_t(int8_encode(y)) : e4m3_encode(y);
    }
  }
  if (transformed_out) std::memcpy(transformed_out, t.data(), t.size() * sizeof(float));
  return ORC_OK;
}

int orc_prepare(int B, int Hq, int Hkv, int N, int d, int dtype, unsigned flags, int stat_len, const int8_t* signs,
                const void* Q, const void* K, const void* V, uint8_t* q8, uint8_t* k8, uint8_t* v8,
                float* q_descale, float* k_descale, float* v_descale, float* k_mean) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || N <= 0 || d <= 0 || (d & (d - 1)) || Hq % Hkv) return ORC_EINVAL;
  if (stat_len < 0 || stat_len > N) return ORC_EINVAL;
  const int P = stat_len == 0 ? N : stat_len;  // tokens the mean and the slice scales see
  const bool rotate = flags & ORC_ROTATE, center = flags & ORC_CENTER_K, tiles = flags & ORC_TILE_SCALES;
  const bool i8 = flags & ORC_I8QK;  // Q and K as INT8 codes, V stays E4M3
  if (rotate && !signs) return ORC_EINVAL;
  const size_t es = dtype == ORC_BF16 ? 2 : 4;
  const int64_t slice = int64_t(N) * d;
  // descales per slice, or per scale tile of Q and K slices
  const int64_t per = tiles ? (N + ORC_SCALE_TILE - 1) / ORC_SCALE_TILE : 1;
  std::atomic<int> status(ORC_OK);
  std::vector<float> mus(size_t(B) * Hkv * d, 0.0f);
  const int64_t nq = int64_t(B) * Hq, nk = int64_t(B) * Hkv;
  parallel_for(nq + 2 * nk, nthreads(), [&](int64_t u) {
    int rc;
    if (u < nq) {
      rc = prepare_slice(N, P, d, dtype, static_cast<const char*>(Q) + es * slice * u, rotate, signs, nullptr,
                         q8 + slice * u, q_descale + per * u, nullptr, tiles, i8);
    } else if (u < nq + nk) {
      int64_t g = u - nq;
      const void* Kh = static_cast<const char*>(K) + es * slice * g;
      float* mu = nullptr;
      if (center) {
        mu = &mus[size_t(g) * d];
        orc_mean_key(P, d, dtype, Kh, mu);  // the mean of the first P tokens
      }
      rc = prepare_slice(N, P, d, dtype, Kh, rotate, signs, mu, k8 + slice * g, k_descale + per * g, nullptr, tiles,
                         i8);
    } else {
      int64_t g = u - nq - nk;
      rc = prepare_slice(N, P, d, dtype, static_cast<const char*>(V) + es * slice * g, false, nullptr, nullptr,
                         v8 + slice * g, v_descale + g, nullptr);
    }
    if (rc != ORC_OK) status.store(rc);
  });
  if (k_mean) std::memcpy(k_mean, mus.data(), mus.size() * sizeof(float));
  return status.load();
}

// ---------------------------------------------------------------------------
// Exact causal attention in double ("ideal causal FP64 attention" [AN]):
// O[i] = sum_{j<=i} softmax_j(q_i.k_j / sqrt(d)) v_j on the original inputs,
// two-pass max-subtracted softmax with std::exp.  Query head h reads KV head
// h / (Hq / Hkv).  Computes the (bh, row) pairs listed (all when lists are
// null); output is compact [n_bh, n_rows, d].
// ---------------------------------------------------------------------------
int orc_attn_exact(int B, int Hq, int Hkv, int N, int d, int dtype, const void* Q, const void* K, const void* V,
                   int causal, const int32_t* bh_list, int n_bh, const int32_t* rows, int n_rows, double* O) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || N <= 0 || d <= 0 || Hq % Hkv) return ORC_EINVAL;
  if (!bh_list) n_bh = B * Hq;
  if (!rows) n_rows = N;
  const int group = Hq / Hkv;
  const int64_t slice = int64_t(N) * d;
  const double inv_sqrt_d = 1.0 / std::sqrt(double(d));
  const int RB = 16;
  const int64_t nblk = (n_rows + RB - 1) / RB;
  parallel_for(int64_t(n_bh) * nblk, nthreads(), [&](int64_t task) {
    int ib = int(task / nblk), rb = int(task % nblk);
    int bh = bh_list ? bh_list[ib] : ib;
    int b = bh / Hq, h = bh % Hq, g = h / group;
    int64_t qoff = (int64_t(b) * Hq + h) * slice, kvoff = (int64_t(b) * Hkv + g) * slice;
    std::vector<double> q(d), logit(N), acc(d);
    for (int r = rb * RB; r < std::min(n_rows, rb * RB + RB); ++r) {
      int i = rows ? rows[r] : r;
      int jmax = causal ? i : N - 1;
      for (int c = 0; c < d; ++c) q[c] = load_in(Q, dtype, qoff + int64_t(i) * d + c);
      double m = -std::numeric_limits<double>::infinity();
      for (int j = 0; j <= jmax; ++j) {
        double s = 0.0;
        for (int c = 0; c < d; ++c) s += q[c] * double(load_in(K, dtype, kvoff + int64_t(j) * d + c));
        logit[j] = s * inv_sqrt_d;
        m = std::max(m, logit[j]);
      }
      double z = 0.0;
      std::fill(acc.begin(), acc.end(), 0.0);
      for (int j = 0; j <= jmax; ++j) {
        double w = std::exp(logit[j] - m);
        z += w;
        for (int c = 0; c < d; ++c) acc[c] += w * double(load_in(V, dtype, kvoff + int64_t(j) * d + c));
      }
      double* o = O + (int64_t(ib) * n_rows + r) * d;
      for (int c = 0; c < d; ++c) o[c] = acc[c] / z;
    }
  });
  return ORC_OK;
}

// ---------------------------------------------------------------------------
// Kernel-faithful emulation of the quantised forward pass [PC sec. 1-4]:
// per query row, visit the KV tiles of width T (aligned at token 0) that hold
// at least one unmasked key, forward (0 -> diagonal) or reverse (diagonal -> 0).
// For each tile:
//   s_j  = fl32(sum_c q_c k_jc)          (exact in double for E4M3 operands)
//   t_j  = fl32(s_j * c)                 c = logit factor in log2 units
//   m'   = max(m, max_j t_j)             exact running maximum
//   a    = exp2(m - m'), 0 while m = -inf
//   P_j  = fl32(exp2(fl32(t_j - m')))
//   l    = fl32(a * l), then + P_j in ascending j (float)
//   p8_j = E4M3(fl32(P_j * S))           the P cast; S divided out at the end
//   acc  = fl32(fl32(a * acc) + fl32(sum_j dec(p8_j) v_j))
// epilogue: O = acc * dv / (S * l) in double.
// Readings: the row sum l uses P before the cast (only S is divided out in
// the epilogue, and the lost mass is what the pages call the MSE source);
// the running max is exact (no lazy rescaling); tiles with no unmasked key
// are not visited (a kernel that visits them must leave m, l, acc unchanged).
//
// Underflow counters per (b, h): in-mask keys j >= k_sink with P_j * S > 0
// whose cast gives 0, split into [0] KV tile 0 and [1] all later tiles.
//
// mode bit 0 (ORC_NO_PCAST): skip the P cast (p8 replaced by fl32(P * S)) -
// for pinning the online softmax against exact attention.
// ---------------------------------------------------------------------------
enum { ORC_NO_PCAST = 1 };

}  // extern "C"

namespace {

struct RowCtx {
  int N, d, T, causal, order, k_sink, mode;
  float c, S;
  const float* c_tile;  // with per-tile scales: logit factor per key scale tile (c unused)
};

// Shared tile loop.  qrow: d doubles; key(j,c), val(j,c) return doubles.
template <class KeyF, class ValF>
void emulate_row(const RowCtx& x, int i, const double* qrow, KeyF key, ValF val, float* acc_out, float* l_out,
                        uint64_t* uf) {
  const int jmax = x.causal ? i : x.N - 1;
  const int ntiles = jmax / x.T + 1;
  std::vector<float> t(x.T), P(x.T), acc(x.d, 0.0f);
  std::vector<double> pv(x.d);
  float m = -std::numeric_limits<float>::infinity(), l = 0.0f;
  for (int step = 0; step < ntiles; ++step) {
    const int tile = x.order == 0 ? step : ntiles - 1 - step;
    const int j0 = tile * x.T, j1 = std::min(jmax, j0 + x.T - 1);
    const int n = j1 - j0 + 1;
    float mt = -std::numeric_limits<float>::infinity();
    for (int jj = 0; jj < n; ++jj) {
      double s = 0.0;
      for (int c = 0; c < x.d; ++c) s += qrow[c] * key(j0 + jj, c);
      float sf = float(s);
      t[jj] = sf * (x.c_tile ? x.c_tile[(j0 + jj) / ORC_SCALE_TILE] : x.c);
      mt = std::max(mt, t[jj]);
    }
    const float mnew = std::max(m, mt);
    const float alpha = (m == -std::numeric_limits<float>::infinity()) ? 0.0f : float(std::exp2(double(m - mnew)));
    for (int jj = 0; jj < n; ++jj) P[jj] = float(std::exp2(double(t[jj] - mnew)));
    l = alpha * l;
    for (int jj = 0; jj < n; ++jj) l = l + P[jj];
    std::fill(pv.begin(), pv.end(), 0.0);
    for (int jj = 0; jj < n; ++jj) {
      const float ps = P[jj] * x.S;
      double p;
      if (x.mode & ORC_NO_PCAST) {
        p = double(ps);
      } else {
        const uint8_t code = e4m3_encode(ps);
        p = dec(code);
        const int j = j0 + jj;
        if (uf && j >= x.k_sink && ps > 0.0f && code == 0) uf[tile == 0 ? 0 : 1] += 1;
      }
      if (p != 0.0)
        for (int c = 0; c < x.d; ++c) pv[c] += p * val(j0 + jj, c);
    }
    for (int c = 0; c < x.d; ++c) acc[c] = (alpha * acc[c]) + float(pv[c]);
    m = mnew;
  }
  for (int c = 0; c < x.d; ++c) acc_out[c] = acc[c];
  *l_out = l;
}

}  // namespace

extern "C" {

// Quantised forward on E4M3 operands in the natural [B, H, N, d] layout (with
// ORC_I8QK, q8 and k8 hold INT8 codes: q.k is then an exact integer sum, and
// the descales are amax/127).
// c = fl32(cq * dk) with cq = fl32(dq * (1/sqrt d) * (ROTATE ? 1/d : 1) * log2 e)
// evaluated in double: the unnormalised FWHT on Q and K multiplies q.k by
// exactly d.  Softmax scale reading: the pages do not state it; the standard
// 1/sqrt(d).  The pages fix no evaluation order for c; this one needs a
// single fp32 multiply per key scale.  With ORC_TILE_SCALES, q_ds and k_ds hold
// one descale per scale tile, cq is the query row's tile's and dk the key's
// tile's (the key tiles T divide the scale tile, so c is constant within a
// key tile).
int orc_attn_quant(int B, int Hq, int Hkv, int N, int d, unsigned flags, const uint8_t* q8, const uint8_t* k8,
                   const uint8_t* v8, const float* q_ds, const float* k_ds, const float* v_ds, float S, int kv_order,
                   int causal, int T, int k_sink, int mode, const int32_t* bh_list, int n_bh, const int32_t* rows,
                   int n_rows, double* O, uint64_t* underflow /* [n_bh, 2] or null */) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || N <= 0 || d <= 0 || T <= 0 || Hq % Hkv || !(S > 0.0f)) return ORC_EINVAL;
  const bool tiles = flags & ORC_TILE_SCALES;
  if (tiles && ORC_SCALE_TILE % T) return ORC_EINVAL;
  if (!bh_list) n_bh = B * Hq;
  if (!rows) n_rows = N;
  const int group = Hq / Hkv;
  const int64_t slice = int64_t(N) * d;
  const bool rotate = flags & ORC_ROTATE;
  const bool i8 = flags & ORC_I8QK;
  const int nst = tiles ? (N + ORC_SCALE_TILE - 1) / ORC_SCALE_TILE : 1;  // descales per Q/K slice
  const int RB = 16;
  const int64_t nblk = (n_rows + RB - 1) / RB;
  std::vector<uint64_t> uf_part(size_t(n_bh) * nblk * 2, 0);
  parallel_for(int64_t(n_bh) * nblk, nthreads(), [&](int64_t task) {
    int ib = int(task / nblk), rb = int(task % nblk);
    int bh = bh_list ? bh_list[ib] : ib;
    int b = bh / Hq, h = bh % Hq, g = h / group;
    const uint8_t* qh = q8 + (int64_t(b) * Hq + h) * slice;
    const uint8_t* kh = k8 + (int64_t(b) * Hkv + g) * slice;
    const uint8_t* vh = v8 + (int64_t(b) * Hkv + g) * slice;
    auto logit_factor = [&](float dq, float dk) {
      const float cq = float(double(dq) * (1.0 / std::sqrt(double(d))) * (rotate ? 1.0 / double(d) : 1.0) * LOG2E);
      return cq * dk;
    };
    const float* qd = q_ds + (int64_t(b) * Hq + h) * nst;
    const float* kd = k_ds + (int64_t(b) * Hkv + g) * nst;
    RowCtx x{N, d, T, causal, kv_order, k_sink, mode, logit_factor(qd[0], kd[0]), S, nullptr};
    std::vector<float> c_tile(nst);
    const double dv = double(v_ds[b * Hkv + g]);
    std::vector<double> q(d);
    std::vector<float> acc(d);
    for (int r = rb * RB; r < std::min(n_rows, rb * RB + RB); ++r) {
      int i = rows ? rows[r] : r;
      if (tiles) {
        for (int t = 0; t < nst; ++t) c_tile[t] = logit_factor(qd[i / ORC_SCALE_TILE], kd[t]);
        x.c_tile = c_tile.data();
      }
      for (int c = 0; c < d; ++c) q[c] = i8 ? double(int8_t(qh[int64_t(i) * d + c])) : dec(qh[int64_t(i) * d + c]);
      float l;
      emulate_row(
          x, i, q.data(),
          [&](int j, int c) { return i8 ? double(int8_t(kh[int64_t(j) * d + c])) : dec(kh[int64_t(j) * d + c]); },
          [&](int j, int c) { return dec(vh[int64_t(j) * d + c]); }, acc.data(), &l,
          underflow ? &uf_part[(size_t(ib) * nblk + rb) * 2] : nullptr);
      double* o = O + (int64_t(ib) * n_rows + r) * d;
      for (int c = 0; c < d; ++c) o[c] = double(acc[c]) * dv / (double(S) * double(l));
    }
  });
  if (underflow)
    for (int ib = 0; ib < n_bh; ++ib) {
      underflow[2 * ib] = underflow[2 * ib + 1] = 0;
      for (int64_t rb = 0; rb < nblk; ++rb) {
        underflow[2 * ib] += uf_part[(size_t(ib) * nblk + rb) * 2];
        underflow[2 * ib + 1] += uf_part[(size_t(ib) * nblk + rb) * 2 + 1];
      }
    }
  return ORC_OK;
}

// P-only ("kernel-faithful") mode [PC sec. 3-4]: Q, K, V stay float; only P
// is cast.  s_j = fl32(sum_c q_c k_jc in double), c = fl32(log2 e / sqrt d),
// epilogue O = acc / (S * l).  Same tile loop as above.
int orc_attn_ponly(int B, int Hq, int Hkv, int N, int d, const float* Q, const float* K, const float* V, float S,
                   int kv_order, int causal, int T, int k_sink, int mode, const int32_t* bh_list, int n_bh,
                   const int32_t* rows, int n_rows, double* O, uint64_t* underflow) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || N <= 0 || d <= 0 || T <= 0 || Hq % Hkv || !(S > 0.0f)) return ORC_EINVAL;
  if (!bh_list) n_bh = B * Hq;
  if (!rows) n_rows = N;
  const int group = Hq / Hkv;
  const int64_t slice = int64_t(N) * d;
  const float cfac = float(LOG2E / std::sqrt(double(d)));
  const int RB = 16;
  const int64_t nblk = (n_rows + RB - 1) / RB;
  std::vector<uint64_t> uf_part(size_t(n_bh) * nblk * 2, 0);
  parallel_for(int64_t(n_bh) * nblk, nthreads(), [&](int64_t task) {
    int ib = int(task / nblk), rb = int(task % nblk);
    int bh = bh_list ? bh_list[ib] : ib;
    int b = bh / Hq, h = bh % Hq, g = h / group;
    const float* qh = Q + (int64_t(b) * Hq + h) * slice;
    const float* kh = K + (int64_t(b) * Hkv + g) * slice;
    const float* vh = V + (int64_t(b) * Hkv + g) * slice;
    RowCtx x{N, d, T, causal, kv_order, k_sink, mode, cfac, S, nullptr};
    std::vector<double> q(d);
    std::vector<float> acc(d);
    for (int r = rb * RB; r < std::min(n_rows, rb * RB + RB); ++r) {
      int i = rows ? rows[r] : r;
      for (int c = 0; c < d; ++c) q[c] = qh[int64_t(i) * d + c];
      float l;
      emulate_row(
          x, i, q.data(), [&](int j, int c) { return double(kh[int64_t(j) * d + c]); },
          [&](int j, int c) { return double(vh[int64_t(j) * d + c]); }, acc.data(), &l,
          underflow ? &uf_part[(size_t(ib) * nblk + rb) * 2] : nullptr);
      double* o = O + (int64_t(ib) * n_rows + r) * d;
      for (int c = 0; c < d; ++c) o[c] = double(acc[c]) / (double(S) * double(l));
    }
  });
  if (underflow)
    for (int ib = 0; ib < n_bh; ++ib) {
      underflow[2 * ib] = underflow[2 * ib + 1] = 0;
      for (int64_t rb = 0; rb < nblk; ++rb) {
        underflow[2 * ib] += uf_part[(size_t(ib) * nblk + rb) * 2];
        underflow[2 * ib + 1] += uf_part[(size_t(ib) * nblk + rb) * 2 + 1];
      }
    }
  return ORC_OK;
}

// Per-head error [RR, 02 / Measured heads]: e = log1p(||O - Oref||_F / ||Oref||_F)
// with both sums in double over one head's n elements.
int orc_err(int64_t n_heads, int64_t n, const double* O, const double* Oref, double* err) {
  for (int64_t h = 0; h < n_heads; ++h) {
    double num = 0.0, den = 0.0;
    for (int64_t i = 0; i < n; ++i) {
      double dlt = O[h * n + i] - Oref[h * n + i];
      num += dlt * dlt;
      den += Oref[h * n + i] * Oref[h * n + i];
    }
    err[h] = (den > 0.0) ? std::log1p(std::sqrt(num / den))
                         : (num == 0.0 ? 0.0 : std::numeric_limits<double>::infinity());
  }
  return ORC_OK;
}

}  // extern "C"
