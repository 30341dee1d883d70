// Operand preparation kernels ("attention-numerics" project page, method and
// kernel settings; "A rounding problem, not a rotation problem", 01 /
// Synthetic illustration):
//   mean key (K, optional) -> sign flip + unnormalised FWHT (Q, K, optional)
//   -> per-(batch, head) amax -> qs = 448/amax -> E4M3 RNE-satfinite cast.
//
// Bit-exactness: every float operation here is a single IEEE add, subtract,
// multiply or divide in a fixed order (no contraction is possible: no
// multiply feeds an add), the FWHT uses a fixed butterfly schedule, the max
// is order-free, and the mean follows the fixed chunk order.  The HBM passes
// read the inputs with 16-byte loads and write 8-byte E4M3 groups; a warp
// covers two (d = 128) or four (d = 64) rows.
#include <cuda_bf16.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace attnq {
namespace {

constexpr int kMeanChunk = 128;   // tokens per partial sum of the mean key
constexpr int kThreads = 256;

template <bool BF16>
__device__ __forceinline__ void load8(const void* base, int64_t off, float (&x)[8]) {
  if constexpr (BF16) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + off));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + off);
    const float4 a = __ldg(p), b = __ldg(p + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
}

template <bool BF16>
__device__ __forceinline__ float load1(const void* base, int64_t off) {
  if constexpr (BF16) {
    return __uint_as_float(uint32_t(__ldg(static_cast<const uint16_t*>(base) + off)) << 16);
  } else {
    return __ldg(static_cast<const float*>(base) + off);
  }
}

// x holds elements 8*sub .. 8*sub+7 of one row; the row's D/8 lanes are
// consecutive and aligned in the warp.  All 32 lanes must call this.
template <int D>
__device__ __forceinline__ void transform(float (&x)[8], int sub, bool center, const float (&mu)[8], bool rotate,
                                          const int8_t (&sg)[8]) {
  if (center) {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = __fsub_rn(x[e], mu[e]);
  }
  if (rotate) {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = sg[e] < 0 ? -x[e] : x[e];
    // butterfly stages h = 1, 2, 4 inside the lane
#pragma unroll
    for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
      for (int i = 0; i < 8; i += 2 * h) {
#pragma unroll
        for (int j = i; j < i + h; ++j) {
          const float a = x[j], b = x[j + h];
          x[j] = __fadd_rn(a, b);
          x[j + h] = __fsub_rn(a, b);
        }
      }
    }
    // stages h = 8, 16, ..., D/2 across lanes: partner lane sub ^ (h/8)
#pragma unroll
    for (int m = 1; m < D / 8; m <<= 1) {
      const bool upper = (sub & m) != 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float o = __shfl_xor_sync(0xffffffffu, x[e], m);
        x[e] = upper ? __fsub_rn(o, x[e]) : __fadd_rn(x[e], o);
      }
    }
  }
}

struct SliceInfo {
  const void* src;
  int tensor;   // 0 Q, 1 K, 2 V
  int local;    // (b*H + h) within its tensor
};

__device__ __forceinline__ SliceInfo slice_info(const PrepareArgs& a, int s, size_t esize) {
  const int nq = a.B * a.Hq, nk = a.B * a.Hkv;
  const int64_t slice = int64_t(a.N) * a.d;
  SliceInfo r;
  if (s < nq) {
    r.tensor = 0; r.local = s; r.src = static_cast<const char*>(a.Q) + esize * slice * s;
  } else if (s < nq + nk) {
    r.tensor = 1; r.local = s - nq; r.src = static_cast<const char*>(a.K) + esize * slice * (s - nq);
  } else {
    r.tensor = 2; r.local = s - nq - nk; r.src = static_cast<const char*>(a.V) + esize * slice * (s - nq - nk);
  }
  return r;
}

// ---- mean key: fixed order (128-token chunks in token order, then chunks in order)
template <bool BF16>
__global__ void k_mean_partial(PrepareArgs a, int nchunks) {
  const int chunk = blockIdx.x, bg = blockIdx.y, c = threadIdx.x;
  const size_t es = BF16 ? 2 : 4;
  const void* base = static_cast<const char*>(a.K) + es * int64_t(bg) * a.N * a.d;
  const int j0 = chunk * kMeanChunk, j1 = min(a.N, j0 + kMeanChunk);
  float part = 0.0f;
  for (int j = j0; j < j1; ++j) part = __fadd_rn(part, load1<BF16>(base, int64_t(j) * a.d + c));
  a.mean_part[(int64_t(bg) * nchunks + chunk) * a.d + c] = part;
}

__global__ void k_mean_final(PrepareArgs a, int nchunks) {
  const int bg = blockIdx.x, c = threadIdx.x;
  float total = 0.0f;
  for (int k = 0; k < nchunks; ++k) total = __fadd_rn(total, a.mean_part[(int64_t(bg) * nchunks + k) * a.d + c]);
  const float mu = __fdiv_rn(total, float(a.N));
  a.mu[bg * a.d + c] = mu;
  if (a.k_mean) a.k_mean[bg * a.d + c] = mu;
}

__global__ void k_zero_f32(float* p, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) p[i] = 0.0f;
}

// ---- pass 1: amax of the transformed slice
template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads) k_amax(PrepareArgs a) {
  constexpr int L = D / 8, RPB = kThreads / L;
  const int s = blockIdx.y;
  const SliceInfo si = slice_info(a, s, BF16 ? 2 : 4);
  const bool rotate = a.rotate && si.tensor < 2, center = a.center && si.tensor == 1;
  const int sub = threadIdx.x % L, rloc = threadIdx.x / L;
  float mu[8];
  int8_t sg[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    mu[e] = center ? a.mu[si.local * D + 8 * sub + e] : 0.0f;
    sg[e] = rotate ? a.signs[8 * sub + e] : int8_t(1);
  }
  uint32_t mx = 0;
  for (int base = blockIdx.x * RPB; base < a.N; base += gridDim.x * RPB) {
    const int row = base + rloc;
    const bool valid = row < a.N;
    float x[8];
    if (valid) {
      load8<BF16>(si.src, int64_t(row) * D + 8 * sub, x);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = 0.0f;
    }
    transform<D>(x, sub, center, mu, rotate, sg);
    if (valid) {
#pragma unroll
      for (int e = 0; e < 8; ++e) mx = max(mx, __float_as_uint(x[e]) & 0x7FFFFFFFu);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  __shared__ uint32_t red[kThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t m = 0;
    for (int w = 0; w < kThreads / 32; ++w) m = max(m, red[w]);
    atomicMax(&a.amax_bits[s], m);
  }
}

// ---- scales: qs = 448/amax, descale = amax/448 (IEEE division)
__global__ void k_scales(PrepareArgs a, int nslices) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= nslices) return;
  const uint32_t bits = a.amax_bits[s];
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
  const int nq = a.B * a.Hq, nk = a.B * a.Hkv;
  if (s < nq) a.q_ds[s] = ds;
  else if (s < nq + nk) a.k_ds[s - nq] = ds;
  else a.v_ds[s - nq - nk] = ds;
}

__device__ __forceinline__ uint2 cast8(const float (&x)[8], float qs) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    w[i] = cvt_e4m3x2(__fmul_rn(x[2 * i], qs), __fmul_rn(x[2 * i + 1], qs));
  }
  return make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
}

// ---- pass 2: transform again, scale, cast (natural [.., N, d] layout)
template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads) k_cast(PrepareArgs a, int skip_v) {
  constexpr int L = D / 8, RPB = kThreads / L;
  const int s = blockIdx.y;
  const SliceInfo si = slice_info(a, s, BF16 ? 2 : 4);
  if (skip_v && si.tensor == 2) return;
  const bool rotate = a.rotate && si.tensor < 2, center = a.center && si.tensor == 1;
  const int sub = threadIdx.x % L, rloc = threadIdx.x / L;
  float mu[8];
  int8_t sg[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    mu[e] = center ? a.mu[si.local * D + 8 * sub + e] : 0.0f;
    sg[e] = rotate ? a.signs[8 * sub + e] : int8_t(1);
  }
  const float qs = a.qs[s];
  uint8_t* dst = (si.tensor == 0 ? a.q8 : si.tensor == 1 ? a.k8 : a.v8) + int64_t(si.local) * a.N * D;
  for (int base = blockIdx.x * RPB; base < a.N; base += gridDim.x * RPB) {
    const int row = base + rloc;
    const bool valid = row < a.N;
    float x[8];
    if (valid) {
      load8<BF16>(si.src, int64_t(row) * D + 8 * sub, x);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = 0.0f;
    }
    transform<D>(x, sub, center, mu, rotate, sg);
    if (valid) *reinterpret_cast<uint2*>(dst + int64_t(row) * D + 8 * sub) = cast8(x, qs);
  }
}

// ---- V cast into the transposed layout [B, Hkv, d, ldv]; tokens N..ldv-1 get 0
template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads) k_cast_vt(PrepareArgs a) {
  constexpr int L = D / 8, RPB = kThreads / L, TOK = 64;
  __shared__ __align__(16) uint8_t tile[D][TOK];
  const int bg = blockIdx.y, j0 = blockIdx.x * TOK;
  const int sub = threadIdx.x % L, rloc = threadIdx.x / L;
  const int s = a.B * a.Hq + a.B * a.Hkv + bg;
  const float qs = a.qs[s];
  const size_t es = BF16 ? 2 : 4;
  const void* src = static_cast<const char*>(a.V) + es * int64_t(bg) * a.N * D;
#pragma unroll
  for (int p = 0; p < TOK / RPB; ++p) {
    const int jl = p * RPB + rloc, j = j0 + jl;
    float x[8];
    if (j < a.N) {
      load8<BF16>(src, int64_t(j) * D + 8 * sub, x);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = 0.0f;
    }
    const uint2 c = cast8(x, qs);
#pragma unroll
    for (int e = 0; e < 8; ++e) tile[8 * sub + e][jl] = uint8_t(((e < 4 ? c.x : c.y) >> (8 * (e & 3))) & 0xFFu);
  }
  __syncthreads();
  uint8_t* dst = a.v8 + int64_t(bg) * D * a.ldv;
  for (int q = threadIdx.x; q < D * (TOK / 16); q += kThreads) {
    const int c = q / (TOK / 16), part = q % (TOK / 16);
    const int64_t j = int64_t(j0) + 16 * part;
    if (j < a.ldv) *reinterpret_cast<uint4*>(dst + int64_t(c) * a.ldv + j) = *reinterpret_cast<const uint4*>(&tile[c][16 * part]);
  }
}

template <int D, bool BF16>
cudaError_t run(const PrepareArgs& a, cudaStream_t st) {
  const int nslices = a.B * a.Hq + 2 * a.B * a.Hkv;
  cudaError_t e = cudaMemsetAsync(a.amax_bits, 0, sizeof(uint32_t) * nslices, st);
  if (e != cudaSuccess) return e;
  if (a.center) {
    const int nchunks = (a.N + kMeanChunk - 1) / kMeanChunk;
    k_mean_partial<BF16><<<dim3(nchunks, a.B * a.Hkv), D, 0, st>>>(a, nchunks);
    k_mean_final<<<a.B * a.Hkv, D, 0, st>>>(a, nchunks);
  } else if (a.k_mean) {
    const int n = a.B * a.Hkv * D;
    k_zero_f32<<<(n + 255) / 256, 256, 0, st>>>(a.k_mean, n);
  }
  constexpr int RPB = kThreads / (D / 8);
  const int rb = (a.N + RPB - 1) / RPB;
  const int gx = rb < 64 ? rb : 64;
  k_amax<D, BF16><<<dim3(gx, nslices), kThreads, 0, st>>>(a);
  k_scales<<<(nslices + 127) / 128, 128, 0, st>>>(a, nslices);
  k_cast<D, BF16><<<dim3(gx, nslices), kThreads, 0, st>>>(a, a.vt);
  if (a.vt) {
    const int tiles = int((a.ldv + 63) / 64);
    k_cast_vt<D, BF16><<<dim3(tiles, a.B * a.Hkv), kThreads, 0, st>>>(a);
  }
  return cudaGetLastError();
}

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

size_t prepare_workspace_bytes(int B, int Hq, int Hkv, int N, int d, int center) {
  const size_t nslices = size_t(B) * Hq + 2 * size_t(B) * Hkv;
  size_t bytes = align256(nslices * 4) + align256(nslices * 4);
  if (center) {
    const size_t nchunks = (size_t(N) + kMeanChunk - 1) / kMeanChunk;
    bytes += align256(size_t(B) * Hkv * nchunks * d * 4) + align256(size_t(B) * Hkv * d * 4);
  }
  return bytes;
}

void carve_prepare_workspace(PrepareArgs& a, void* ws) {
  const size_t nslices = size_t(a.B) * a.Hq + 2 * size_t(a.B) * a.Hkv;
  char* p = static_cast<char*>(ws);
  a.amax_bits = reinterpret_cast<uint32_t*>(p);
  p += align256(nslices * 4);
  a.qs = reinterpret_cast<float*>(p);
  p += align256(nslices * 4);
  if (a.center) {
    const size_t nchunks = (size_t(a.N) + kMeanChunk - 1) / kMeanChunk;
    a.mean_part = reinterpret_cast<float*>(p);
    p += align256(size_t(a.B) * a.Hkv * nchunks * a.d * 4);
    a.mu = reinterpret_cast<float*>(p);
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
