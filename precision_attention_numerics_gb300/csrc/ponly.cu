// P-only forward ("Technische Samenvatting: P-Cast Precisie in FP8
// Attention", sec. 3-4: kernel-faithful simulation with Q, K, V in FP32 and
// only P cast to E4M3).  Same tile loop as the FP8 kernel:
//   t_j = fl32(q.k_j) * c, m' = max(m, max_j t_j), alpha = 2^(m - m'),
//   P_j = 2^(t_j - m'), l = alpha*l + sum P_j, p8_j = E4M3(P_j * S),
//   acc = alpha*acc + sum_j dec(p8_j) v_j,  O = acc / (S*l).
// A CTA owns 32 query rows of one head (4 per warp); K and V tiles are
// staged in shared memory (K rows padded by one word against bank conflicts).
// A warp handles one row at a time: lane L scores keys L, L+32, ...; output
// channels L, L+32, ... accumulate in registers.
#include <cuda_fp16.h>

#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace attnq {
namespace {

constexpr int kRows = 32, kWarps = 8, kRowsPerWarp = kRows / kWarps;

template <int D>
__global__ void __launch_bounds__(kWarps * 32) k_ponly(PonlyArgs a, float c) {
  extern __shared__ float smem[];
  float* sQ = smem;                      // [kRows][D]
  float* sK = sQ + kRows * D;            // [T][D+1]
  float* sV = sK + a.T * (D + 1);        // [T][D]
  constexpr int CPL = D / 32;            // output channels per lane
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int bh = blockIdx.y, b = bh / a.Hq, h = bh % a.Hq, g = h / (a.Hq / a.Hkv);
  const int r0 = blockIdx.x * kRows;
  const int64_t qoff = int64_t(bh) * a.N * D, kvoff = (int64_t(b) * a.Hkv + g) * a.N * D;

  for (int x = threadIdx.x; x < kRows * D; x += blockDim.x) {
    const int r = x / D, cc = x % D;
    sQ[x] = (r0 + r < a.N) ? a.Q[qoff + int64_t(r0 + r) * D + cc] : 0.0f;
  }

  const int last_row = min(a.N - 1, r0 + kRows - 1);
  const int nt = a.causal ? last_row / a.T + 1 : (a.N - 1) / a.T + 1;

  float m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][CPL];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.0f;
#pragma unroll
    for (int k = 0; k < CPL; ++k) acc[r][k] = 0.0f;
  }
  uint32_t uf0 = 0, uf1 = 0;

  for (int step = 0; step < nt; ++step) {
    const int tile = a.reverse ? nt - 1 - step : step;
    const int j0 = tile * a.T;
    __syncthreads();
    for (int x = threadIdx.x; x < a.T * D; x += blockDim.x) {
      const int jl = x / D, cc = x % D, j = j0 + jl;
      const bool in = j < a.N;
      sK[jl * (D + 1) + cc] = in ? a.K[kvoff + int64_t(j) * D + cc] : 0.0f;
      sV[jl * D + cc] = in ? a.V[kvoff + int64_t(j) * D + cc] : 0.0f;
    }
    __syncthreads();
#pragma unroll 1
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const int rl = warp * kRowsPerWarp + r, i = r0 + rl;
      if (i >= a.N) continue;  // warp-uniform
      const int jmax = a.causal ? i : a.N - 1;
      // scores for keys j0 + lane + 32*kk, kk < 4 (keys past T or the row are masked)
      float t[4];
      float mt = -INFINITY;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        t[kk] = -INFINITY;
        const int jl = lane + 32 * kk, j = j0 + jl;
        if (jl < a.T && j <= jmax) {
          float s = 0.0f;
          const float* qr = sQ + rl * D;
          const float* kr = sK + jl * (D + 1);
#pragma unroll 8
          for (int cc = 0; cc < D; ++cc) s = fmaf(qr[cc], kr[cc], s);
          t[kk] = s * c;
        }
        mt = fmaxf(mt, t[kk]);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
      const float mnew = fmaxf(m[r], mt);
      if (mnew == -INFINITY) continue;  // no unmasked key yet: nothing changes
      const float alpha = ex2(m[r] - mnew);  // m = -inf -> 0
      float psum = 0.0f, p[4];
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const float P = ex2(t[kk] - mnew);   // masked -> 0
        psum += P;
        const float ps = P * a.S;
        const uint16_t code2 = cvt_e4m3x2(ps, ps);   // same code in both bytes
        p[kk] = e4m3x2_to_f2(code2).x;
        if (a.underflow && ps > 0.0f && (code2 & 0xFFu) == 0u) {
          const int j = j0 + lane + 32 * kk;
          if (j >= a.k_sink) {
            if (tile == 0) ++uf0;
            else ++uf1;
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
      l[r] = alpha * l[r] + psum;
      float pv[CPL];
#pragma unroll
      for (int k = 0; k < CPL; ++k) pv[k] = 0.0f;
      const int jend = min(a.T, jmax - j0 + 1);
      for (int jl = 0; jl < jend; ++jl) {
        const float pj = __shfl_sync(0xffffffffu, p[(jl >> 5) & 3], jl & 31);
        if (pj != 0.0f) {
#pragma unroll
          for (int k = 0; k < CPL; ++k) pv[k] = fmaf(pj, sV[jl * D + lane + 32 * k], pv[k]);
        }
      }
#pragma unroll
      for (int k = 0; k < CPL; ++k) acc[r][k] = alpha * acc[r][k] + pv[k];
      m[r] = mnew;
    }
  }
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int i = r0 + warp * kRowsPerWarp + r;
    if (i >= a.N) continue;
    const float inv = 1.0f / (a.S * l[r]);
#pragma unroll
    for (int k = 0; k < CPL; ++k) a.O[qoff + int64_t(i) * D + lane + 32 * k] = acc[r][k] * inv;
  }
  if (a.underflow) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      uf0 += __shfl_xor_sync(0xffffffffu, uf0, o);
      uf1 += __shfl_xor_sync(0xffffffffu, uf1, o);
    }
    if (lane == 0) {
      if (uf0) atomicAdd(a.underflow + 2 * bh, (unsigned long long)uf0);
      if (uf1) atomicAdd(a.underflow + 2 * bh + 1, (unsigned long long)uf1);
    }
  }
}

template <int D>
cudaError_t run(const PonlyArgs& a, cudaStream_t st) {
  const size_t smem = sizeof(float) * (size_t(kRows) * D + size_t(a.T) * (D + 1) + size_t(a.T) * D);
  cudaError_t e = cudaFuncSetAttribute(k_ponly<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  const float c = float(1.4426950408889634 / std::sqrt(double(D)));
  dim3 grid((a.N + kRows - 1) / kRows, a.B * a.Hq);
  k_ponly<D><<<grid, kWarps * 32, smem, st>>>(a, c);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ponly(const PonlyArgs& a, cudaStream_t s) {
  return a.d == 128 ? run<128>(a, s) : run<64>(a, s);
}

}  // namespace attnq
