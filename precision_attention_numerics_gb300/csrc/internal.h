// Launchers shared between the kernel translation units and the C-ABI layer.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace attnq {

// ---- prepare -------------------------------------------------------------
// Tokens per scale tile of the per-tile Q/K scales (tiles aligned at token 0).
constexpr int kScaleTile = 128;

struct PrepareArgs {
  int B, Hq, Hkv, N, d;
  int P;              // tokens the mean key and the slice scales are taken over (1..N)
  int bf16;           // input element type: 1 bf16, 0 fp32
  int rotate, center, vt;
  int tiles;          // per-tile Q/K scales
  int i8;             // Q and K as INT8 codes held in bf16 (V stays E4M3)
  const int8_t* signs;
  const void* Q;
  const void* K;
  const void* V;
  uint8_t* q8;
  uint8_t* k8;
  uint8_t* v8;
  float* q_ds;
  float* k_ds;
  float* v_ds;
  float* k_mean;      // optional
  int64_t ldv;        // row length of transposed V
  // workspace carve-up
  uint32_t* amax_bits;  // [nslices]
  uint32_t* a_done;     // [nslices] warp-tiles whose amax is in amax_bits
  uint32_t* m_done;     // [B*Hkv] mean-key chunks summed
  uint32_t* mu_ready;   // [B*Hkv] mean key published
  uint32_t* ctl;        // [4] ticket, abort, number of entries
  uint32_t* entries;    // [3*nslices] work list: kind << 30 | slice
  float* mean_part;     // [B*Hkv*nchunks*d]
  float* mu;            // [B*Hkv*d]
  uint32_t* status;
  int num_sms;
  uint64_t wait_ns;
};

size_t prepare_workspace_bytes(int B, int Hq, int Hkv, int N, int d, int center);
// Size of the fixed scratch array behind attnq_prepare_static (ATTNQ_STATIC_SCRATCH_BYTES).
constexpr size_t kStaticScratchBytes = size_t(4) << 20;
// Device address of that array on the current device (looked up once per device).
cudaError_t static_scratch_address(void** out);
void carve_prepare_workspace(PrepareArgs& a, void* ws);
cudaError_t launch_prepare(const PrepareArgs& a, cudaStream_t s);

// ---- attention forward (tcgen05) -----------------------------------------
struct FwdArgs {
  int B, Hq, Hkv, N, d, T;
  int causal, reverse;
  int rotate;
  int tiles;          // per-tile Q/K scales
  int i8;             // q8, k8: INT8 codes held in bf16 (S = Q K^T as kind::f16)
  float S;
  const uint8_t* q8;
  const uint8_t* k8;
  const uint8_t* v8t;
  int64_t ldv;
  const float* q_ds;
  const float* k_ds;
  const float* v_ds;
  void* O;
  int out_bf16;
  unsigned long long* underflow;
  int k_sink;
  uint32_t* status;
  uint64_t wait_ns;
  int num_sms;
};
cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t s);

// ---- P-only forward (SIMT fp32) -------------------------------------------
struct PonlyArgs {
  int B, Hq, Hkv, N, d, T;
  int causal, reverse;
  float S;
  const float* Q;
  const float* K;
  const float* V;
  float* O;
  unsigned long long* underflow;
  int k_sink;
};
cudaError_t launch_ponly(const PonlyArgs& a, cudaStream_t s);

// ---- per-head error ----------------------------------------------------------
struct ErrArgs {
  int n_heads;
  int64_t per_head;
  const void* O;
  int o_bf16;
  const double* O_ref;
  double* err;
};
cudaError_t launch_err(const ErrArgs& a, cudaStream_t s);

// ---- FP64 reference attention ----------------------------------------------
struct RefArgs {
  int B, Hq, Hkv, N, d;
  int bf16, causal;
  const void* Q;
  const void* K;
  const void* V;
  double* O_ref;
};
cudaError_t launch_ref_attn(const RefArgs& a, cudaStream_t s);

// ---- driver entry point for tensor maps ------------------------------------
CUresult encode_tiled_3d(CUtensorMap* map, const void* base, uint64_t dim0, uint64_t dim1, uint64_t dim2,
                         uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box1,
                         CUtensorMapSwizzle swizzle);

}  // namespace attnq
