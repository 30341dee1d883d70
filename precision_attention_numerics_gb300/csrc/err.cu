// Per-head error ("A rounding problem, not a rotation problem", 02 / Measured
// heads): err = log1p(||O - O_ref||_F / ||O_ref||_F), both squared norms in
// fp64.  A cluster of kCluster CTAs owns one head; each CTA reduces a fixed
// strided share in a fixed tree order and CTA rank 0 adds the partials in
// rank order through distributed shared memory, so the result is
// deterministic and no scratch memory is needed.
#include <cooperative_groups.h>

#include <cmath>

#include "internal.h"

namespace cg = cooperative_groups;

namespace attnq {
namespace {

constexpr int kCluster = 8, kThreads = 512;

template <bool BF16>
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads) k_err(ErrArgs a) {
  __shared__ double s_num[kThreads / 32], s_den[kThreads / 32];
  __shared__ double part[2];
  cg::cluster_group cl = cg::this_cluster();
  const int rank = int(cl.block_rank());
  const int head = blockIdx.x / kCluster;
  const int64_t n = a.per_head;
  const double* ref = a.O_ref + int64_t(head) * n;
  double num = 0.0, den = 0.0;
  const int64_t stride = int64_t(kCluster) * kThreads;
  for (int64_t i = int64_t(rank) * kThreads + threadIdx.x; i < n; i += stride) {
    double o;
    if constexpr (BF16) {
      o = double(__uint_as_float(uint32_t(static_cast<const uint16_t*>(a.O)[int64_t(head) * n + i]) << 16));
    } else {
      o = double(static_cast<const float*>(a.O)[int64_t(head) * n + i]);
    }
    const double r = ref[i];
    const double dlt = o - r;
    num = fma(dlt, dlt, num);
    den = fma(r, r, den);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    num += __shfl_down_sync(0xffffffffu, num, off);
    den += __shfl_down_sync(0xffffffffu, den, off);
  }
  if ((threadIdx.x & 31) == 0) {
    s_num[threadIdx.x >> 5] = num;
    s_den[threadIdx.x >> 5] = den;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double tn = 0.0, td = 0.0;
    for (int w = 0; w < kThreads / 32; ++w) {
      tn += s_num[w];
      td += s_den[w];
    }
    part[0] = tn;
    part[1] = td;
  }
  cl.sync();
  if (rank == 0 && threadIdx.x == 0) {
    double tn = 0.0, td = 0.0;
    for (int r = 0; r < kCluster; ++r) {
      const double* p = cl.map_shared_rank(part, r);
      tn += p[0];
      td += p[1];
    }
    double e;
    if (td > 0.0) e = log1p(sqrt(tn / td));
    else e = (tn == 0.0) ? 0.0 : __longlong_as_double(0x7FF0000000000000LL);
    a.err[head] = e;
  }
  cl.sync();
}

}  // namespace

cudaError_t launch_err(const ErrArgs& a, cudaStream_t s) {
  dim3 grid(a.n_heads * kCluster);
  if (a.o_bf16) k_err<true><<<grid, kThreads, 0, s>>>(a);
  else k_err<false><<<grid, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace attnq
