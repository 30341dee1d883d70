// FP64 reference attention ("A rounding problem, not a rotation problem",
// 02 / Measured heads: the error of each head is measured against the ideal
// causal attention in FP64):
//   O_ref[b,h,i] = sum_{j<=i} softmax_j(q_i . k_j / sqrt(d)) v_j,
// on the original (unquantised, unrotated, uncentred) inputs upcast exactly
// to double; query head h reads KV head h / (Hq / Hkv).
//
// Online softmax in double over key tiles of 32: a warp owns 4 query rows,
// lane l scores key l of the tile for each row (the query rows broadcast from
// shared memory), the row max and sum go through warp shuffles, and lane l
// accumulates output columns l, l + 32, ...  The order of the sums differs
// from a two-pass softmax only by double rounding (~1e-16 relative).
// GB300's FP64 rate bounds it: it is a checking tool, not part of the timed
// path.
#include <cmath>

#include "internal.h"

namespace attnq {
namespace {

constexpr int kWarps = 8, kRowsPerWarp = 4, kRows = kWarps * kRowsPerWarp, kKeys = 32;

template <bool BF16>
__device__ __forceinline__ double load_in(const void* p, int64_t i) {
  if constexpr (BF16) {
    return double(__uint_as_float(uint32_t(static_cast<const uint16_t*>(p)[i]) << 16));
  } else {
    return double(static_cast<const float*>(p)[i]);
  }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kWarps * 32) k_ref_attn(RefArgs a) {
  extern __shared__ double sm[];
  double* qs = sm;                          // [kRows][D]
  double* ks = qs + kRows * D;              // [kKeys][D + 1]
  double* vs = ks + kKeys * (D + 1);        // [kKeys][D]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.y, b = bh / a.Hq, h = bh % a.Hq, g = h / (a.Hq / a.Hkv);
  const int i0 = blockIdx.x * kRows;
  const int64_t qoff = int64_t(bh) * a.N * D, kvoff = (int64_t(b) * a.Hkv + g) * a.N * D;
  for (int x = threadIdx.x; x < kRows * D; x += blockDim.x) {
    const int r = x / D, c = x % D, i = i0 + r;
    qs[x] = i < a.N ? load_in<BF16>(a.Q, qoff + int64_t(i) * D + c) : 0.0;
  }
  const double scale = 1.0 / sqrt(double(D));
  constexpr int CPL = D / 32;  // output columns per lane
  double m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][CPL];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.0;
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[r][c] = 0.0;
  }
  const int last_row = min(i0 + kRows, a.N) - 1;
  const int jend = a.causal ? last_row + 1 : a.N;  // keys [0, jend) can be visible
  for (int j0 = 0; j0 < jend; j0 += kKeys) {
    __syncthreads();
    for (int x = threadIdx.x; x < kKeys * D; x += blockDim.x) {
      const int kk = x / D, c = x % D, j = j0 + kk;
      const bool in = j < a.N;
      ks[kk * (D + 1) + c] = in ? load_in<BF16>(a.K, kvoff + int64_t(j) * D + c) : 0.0;
      vs[kk * D + c] = in ? load_in<BF16>(a.V, kvoff + int64_t(j) * D + c) : 0.0;
    }
    __syncthreads();
    const int j = j0 + lane;
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const int rr = warp * kRowsPerWarp + r, i = i0 + rr;
      const double* q = qs + rr * D;
      const double* k = ks + lane * (D + 1);
      double s = 0.0;
#pragma unroll 8
      for (int c = 0; c < D; ++c) s = fma(q[c], k[c], s);
      s *= scale;
      const bool vis = j < a.N && i < a.N && (!a.causal || j <= i);
      if (!vis) s = -INFINITY;
      double tmax = s;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) tmax = fmax(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
      const double mnew = fmax(m[r], tmax);
      if (mnew == -INFINITY) continue;  // nothing visible yet for this row
      const double alpha = exp(m[r] - mnew);
      const double p = vis ? exp(s - mnew) : 0.0;
      double psum = p;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
      l[r] = fma(alpha, l[r], psum);
      m[r] = mnew;
#pragma unroll
      for (int c = 0; c < CPL; ++c) acc[r][c] *= alpha;
      for (int kk = 0; kk < kKeys; ++kk) {
        const double pk = __shfl_sync(0xffffffffu, p, kk);
        if (pk == 0.0) continue;  // warp-uniform: pk is the same in every lane
#pragma unroll
        for (int c = 0; c < CPL; ++c) acc[r][c] = fma(pk, vs[kk * D + lane + 32 * c], acc[r][c]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int i = i0 + warp * kRowsPerWarp + r;
    if (i >= a.N) continue;
    double* o = a.O_ref + qoff + int64_t(i) * D;
#pragma unroll
    for (int c = 0; c < CPL; ++c) o[lane + 32 * c] = acc[r][c] / l[r];
  }
}

template <int D, bool BF16>
cudaError_t run(const RefArgs& a, cudaStream_t st) {
  const size_t smem = sizeof(double) * (size_t(kRows) * D + size_t(kKeys) * (D + 1) + size_t(kKeys) * D);
  auto kern = k_ref_attn<D, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  const dim3 grid((a.N + kRows - 1) / kRows, a.B * a.Hq);
  kern<<<grid, kWarps * 32, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ref_attn(const RefArgs& a, cudaStream_t s) {
  if (a.d == 128) return a.bf16 ? run<128, true>(a, s) : run<128, false>(a, s);
  return a.bf16 ? run<64, true>(a, s) : run<64, false>(a, s);
}

}  // namespace attnq
