// C ABI of libattnq: argument validation, workspace carve-up, tensor maps,
// launches and the device status word.  Declarations and their contracts are
// in include/attnq.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <atomic>
#include <cstring>
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "attnq.h"
#include "internal.h"
#include "ptx.cuh"

namespace attnq {

__device__ uint32_t g_status;  // DEV_* bits, one word per device

namespace {

constexpr int kMaxDevices = 64;
uint32_t* g_status_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};
bool g_sm103[kMaxDevices] = {};
std::mutex g_mu;

// Per-device set-up: the status word's device address, SM count and
// architecture check.  Done once per device with that device current.
attnq_status device_setup(int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTNQ_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return ATTNQ_EUNSUPPORTED;
  *dev_out = dev;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_status_ptr[dev]) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return ATTNQ_ECUDA;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return ATTNQ_ECUDA;
    g_sm103[dev] = (major == 10 && minor == 3);
    g_num_sms[dev] = sms;
    g_status_ptr[dev] = static_cast<uint32_t*>(p);
  }
  return g_sm103[dev] ? ATTNQ_OK : ATTNQ_EUNSUPPORTED;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Value of x > 0 rounded to the nearest E4M3 value, ties to even, saturating
// at 448: normal binades 2^e (e >= -6) hold 8 values 2^(e-3) apart, below
// 2^-6 the step is 2^-9.
double e4m3_round_host(double x) {
  if (x >= 448.0) return 448.0;
  const int e = int(std::floor(std::log2(x)));
  const double q = std::ldexp(1.0, e < -6 ? -9 : e - 3);
  return std::nearbyint(x / q) * q;  // default rounding mode: half to even
}

// A P-cast scale is usable by attnq_fwd unless it lies within a relative 2^-20
// of a point where the E4M3 rounding of P * S changes: the kernel forms P * S
// in one exp2 of fma(s, c, log2 S - m'), so the row maximum's P * S, exactly S
// in the two-step form, comes out S (1 +- a few 2^-24) and would round to
// either neighbour of such a point (S = 100, halfway between 96 and 104, is
// one).
bool pcast_scale_ok(float S) {
  if (!(std::isfinite(S) && S > 0.0f && S <= 448.0f)) return false;
  const double s = double(S), r = std::ldexp(1.0, -20);
  return e4m3_round_host(s * (1.0 - r)) == e4m3_round_host(s * (1.0 + r));
}

attnq_status check_desc(const attnq_desc* d) {
  if (!d) return ATTNQ_EINVAL;
  if (d->B <= 0 || d->Hq <= 0 || d->Hkv <= 0 || d->N <= 0 || d->d <= 0) return ATTNQ_EINVAL;
  if (d->Hq % d->Hkv != 0) return ATTNQ_EINVAL;
  if ((d->flags & ~uint32_t(ATTNQ_ROTATE | ATTNQ_CENTER_K | ATTNQ_VT_LAYOUT | ATTNQ_TILE_SCALES | ATTNQ_I8QK)) != 0)
    return ATTNQ_EINVAL;
  if (d->stat_len < 0 || d->stat_len > d->N) return ATTNQ_EINVAL;
  if (d->d != 64 && d->d != 128) return ATTNQ_EUNSUPPORTED;
  // grid.y of the prepare passes and int32 indices of rows
  const int64_t nslices = int64_t(d->B) * d->Hq + 2 * int64_t(d->B) * d->Hkv;
  if (nslices > 65535) return ATTNQ_EUNSUPPORTED;
  if (int64_t(d->N) * d->d > (int64_t(1) << 31)) return ATTNQ_EUNSUPPORTED;
  return ATTNQ_OK;
}

attnq_status from_cuda(cudaError_t e) { return e == cudaSuccess ? ATTNQ_OK : ATTNQ_ECUDA; }

// Host-side NVTX range around each call's launches (visible to profilers that
// attach an NVTX tool; a no-op otherwise).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

std::atomic<uint64_t> g_wait_ns{2000000000ull};  // limit of every wait inside the kernels (2 s)
// Carve-up of the harm-report workspace (every piece 256-byte aligned).
struct HarmLayout {
  size_t o_ref, o, q8, k8, v8, q_ds, k_ds, v_ds, k_mean, prep, total;
};

size_t a256(size_t x) { return (x + 255) & ~size_t(255); }

HarmLayout harm_layout(const attnq_desc* d) {
  const size_t nq = size_t(d->B) * d->Hq, nk = size_t(d->B) * d->Hkv, rows = size_t(d->N) * d->d;
  attnq_desc full = *d;
  full.flags = ATTNQ_ROTATE | ATTNQ_CENTER_K | ATTNQ_VT_LAYOUT;
  HarmLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += a256(bytes);
    return at;
  };
  L.o_ref = take(8 * nq * rows);
  L.o = take(4 * nq * rows);
  L.q8 = take(nq * rows);
  L.k8 = take(nk * rows);
  L.v8 = take(nk * size_t(d->d) * size_t(attnq_vt_ld(d->N)));
  L.q_ds = take(4 * nq);
  L.k_ds = take(4 * nk);
  L.v_ds = take(4 * nk);
  L.k_mean = take(4 * nk * d->d);
  L.prep = take(attnq_prepare_workspace(&full));
  L.total = off;
  return L;
}

// Carve-up of the host-pipeline workspace: two input sets, the prepared
// operands and their scales, the prepare workspace, two outputs.
struct PipeLayout {
  size_t in[2][3], q8, k8, v8, q_ds, k_ds, v_ds, k_mean, prep, out[2], total;
  size_t in_bytes[3], out_bytes;
};

PipeLayout pipe_layout(const attnq_desc* d, int32_t out_dtype) {
  const size_t nq = size_t(d->B) * d->Hq, nk = size_t(d->B) * d->Hkv, rows = size_t(d->N) * d->d;
  const size_t es = d->in_dtype == ATTNQ_BF16 ? 2 : 4, eo = out_dtype == ATTNQ_BF16 ? 2 : 4;
  PipeLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += a256(bytes);
    return at;
  };
  L.in_bytes[0] = es * nq * rows;
  L.in_bytes[1] = es * nk * rows;
  L.in_bytes[2] = es * nk * rows;
  for (int b = 0; b < 2; ++b)
    for (int t = 0; t < 3; ++t) L.in[b][t] = take(L.in_bytes[t]);
  const size_t nst = (d->flags & ATTNQ_TILE_SCALES) ? size_t(attnq_scale_tiles(d->N)) : 1;
  const size_t qe = (d->flags & ATTNQ_I8QK) ? 2 : 1;  // bytes of a Q/K code
  L.q8 = take(qe * nq * rows);
  L.k8 = take(qe * nk * rows);
  L.v8 = take(nk * size_t(d->d) * size_t(attnq_vt_ld(d->N)));
  L.q_ds = take(4 * nq * nst);
  L.k_ds = take(4 * nk * nst);
  L.v_ds = take(4 * nk);
  L.k_mean = take(4 * nk * d->d);
  L.prep = take(attnq_prepare_workspace(d));
  L.out_bytes = eo * nq * rows;
  for (int b = 0; b < 2; ++b) L.out[b] = take(L.out_bytes);
  L.total = off;
  return L;
}

// Events of one pipelined call, destroyed with it (an event still pending at
// destruction is released by the runtime once it completes).
struct PipeEvents {
  cudaEvent_t ev[9] = {};
  int made = 0;
  cudaError_t create() {
    for (; made < 9; ++made) {
      const cudaError_t e = cudaEventCreateWithFlags(&ev[made], cudaEventDisableTiming);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  ~PipeEvents() {
    for (int i = 0; i < made; ++i) cudaEventDestroy(ev[i]);
  }
};

}  // namespace

namespace {
// cuTensorMapEncodeTiled is looked up through the runtime, so the library
// does not link the driver library directly (and loads on hosts without one).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}
}  // namespace

CUresult encode_tiled_3d(CUtensorMap* map, const void* base, uint64_t dim0, uint64_t dim1, uint64_t dim2,
                         uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box1,
                         CUtensorMapSwizzle swizzle) {
  const EncodeTiledFn fn = encode_fn();
  if (!fn) return CUDA_ERROR_NOT_FOUND;
  const cuuint64_t dims[3] = {dim0, dim1, dim2};
  const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  const cuuint32_t box[3] = {box0, box1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

namespace {

// Kernel arguments of one preparation (the workspace is carved by the caller).
PrepareArgs prepare_args(const attnq_desc* desc, const void* Q, const void* K, const void* V, uint8_t* q8,
                         uint8_t* k8, uint8_t* v8, const attnq_scales* out, int dev) {
  PrepareArgs a{};
  a.B = desc->B; a.Hq = desc->Hq; a.Hkv = desc->Hkv; a.N = desc->N; a.d = desc->d;
  a.P = desc->stat_len > 0 ? desc->stat_len : desc->N;
  a.bf16 = desc->in_dtype == ATTNQ_BF16;
  a.rotate = (desc->flags & ATTNQ_ROTATE) != 0;
  a.center = (desc->flags & ATTNQ_CENTER_K) != 0;
  a.vt = (desc->flags & ATTNQ_VT_LAYOUT) != 0;
  a.tiles = (desc->flags & ATTNQ_TILE_SCALES) != 0;
  a.i8 = (desc->flags & ATTNQ_I8QK) != 0;
  a.signs = desc->signs;
  a.Q = Q; a.K = K; a.V = V; a.q8 = q8; a.k8 = k8; a.v8 = v8;
  a.q_ds = out->q_descale; a.k_ds = out->k_descale; a.v_ds = out->v_descale; a.k_mean = out->k_mean;
  a.ldv = attnq_vt_ld(desc->N);
  a.status = g_status_ptr[dev];
  a.num_sms = g_num_sms[dev];
  a.wait_ns = g_wait_ns.load();
  return a;
}

}  // namespace

}  // namespace attnq

using namespace attnq;

extern "C" {

int32_t attnq_version(void) { return 200; }

const char* attnq_status_string(attnq_status s) {
  switch (s) {
    case ATTNQ_OK: return "ATTNQ_OK";
    case ATTNQ_EINVAL: return "ATTNQ_EINVAL: invalid argument";
    case ATTNQ_EUNSUPPORTED: return "ATTNQ_EUNSUPPORTED: unsupported size, option or device";
    case ATTNQ_ECUDA: return "ATTNQ_ECUDA: CUDA call failed";
    case ATTNQ_ENONFINITE: return "ATTNQ_ENONFINITE: non-finite input";
    case ATTNQ_ETIMEOUT: return "ATTNQ_ETIMEOUT: device wait timed out";
  }
  return "unknown attnq status";
}

int32_t attnq_scale_tiles(int32_t N) { return N <= 0 ? 0 : (N + ATTNQ_SCALE_TILE - 1) / ATTNQ_SCALE_TILE; }

int64_t attnq_vt_ld(int32_t N) { return N <= 0 ? 0 : (int64_t(N) + 15) / 16 * 16; }

attnq_status attnq_hadamard_signs(uint64_t seed, int32_t d, int8_t* host_out) {
  if (!host_out || d <= 0) return ATTNQ_EINVAL;
  for (int32_t c = 0; c < d; ++c) {
    uint64_t z = seed + uint64_t(c + 1) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    z = z ^ (z >> 31);
    host_out[c] = (z >> 63) ? int8_t(-1) : int8_t(1);
  }
  return ATTNQ_OK;
}

size_t attnq_prepare_workspace(const attnq_desc* desc) {
  if (check_desc(desc) != ATTNQ_OK) return 0;
  return prepare_workspace_bytes(desc->B, desc->Hq, desc->Hkv, desc->N, desc->d,
                                 (desc->flags & ATTNQ_CENTER_K) ? 1 : 0);
}

attnq_status attnq_prepare(const attnq_desc* desc, const void* Q, const void* K, const void* V, uint8_t* q8,
                           uint8_t* k8, uint8_t* v8, const attnq_scales* out, void* workspace, size_t ws_bytes,
                           cudaStream_t stream) {
  attnq_status st = check_desc(desc);
  if (st != ATTNQ_OK) return st;
  if (desc->in_dtype != ATTNQ_F32 && desc->in_dtype != ATTNQ_BF16) return ATTNQ_EINVAL;
  if (!Q || !K || !V || !q8 || !k8 || !v8 || !out || !out->q_descale || !out->k_descale || !out->v_descale)
    return ATTNQ_EINVAL;
  if ((desc->flags & ATTNQ_ROTATE) && !desc->signs) return ATTNQ_EINVAL;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(q8) || !aligned16(k8) || !aligned16(v8))
    return ATTNQ_EINVAL;
  const size_t need = attnq_prepare_workspace(desc);
  if (!workspace || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return ATTNQ_EINVAL;
  int dev;
  st = device_setup(&dev);
  if (st != ATTNQ_OK) return st;
  PrepareArgs a = prepare_args(desc, Q, K, V, q8, k8, v8, out, dev);
  carve_prepare_workspace(a, workspace);
  const NvtxRange range("attnq_prepare");
  return from_cuda(launch_prepare(a, stream));
}

attnq_status attnq_prepare_static(const attnq_desc* desc, const void* Q, const void* K, const void* V, uint8_t* q8,
                                  uint8_t* k8, uint8_t* v8, const attnq_scales* out, cudaStream_t stream) {
  static_assert(kStaticScratchBytes == ATTNQ_STATIC_SCRATCH_BYTES, "header and library disagree");
  attnq_status st = check_desc(desc);
  if (st != ATTNQ_OK) return st;
  if (desc->in_dtype != ATTNQ_F32 && desc->in_dtype != ATTNQ_BF16) return ATTNQ_EINVAL;
  if (!Q || !K || !V || !q8 || !k8 || !v8 || !out || !out->q_descale || !out->k_descale || !out->v_descale)
    return ATTNQ_EINVAL;
  if ((desc->flags & ATTNQ_ROTATE) && !desc->signs) return ATTNQ_EINVAL;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(q8) || !aligned16(k8) || !aligned16(v8))
    return ATTNQ_EINVAL;
  // larger problems need more scratch than the fixed array holds
  if (attnq_prepare_workspace(desc) > kStaticScratchBytes) return ATTNQ_EUNSUPPORTED;
  int dev;
  st = device_setup(&dev);
  if (st != ATTNQ_OK) return st;
  void* scratch = nullptr;
  if (static_scratch_address(&scratch) != cudaSuccess) return ATTNQ_ECUDA;
  PrepareArgs a = prepare_args(desc, Q, K, V, q8, k8, v8, out, dev);
  carve_prepare_workspace(a, scratch);   // the launch itself clears the counters it uses
  const NvtxRange range("attnq_prepare");
  return from_cuda(launch_prepare(a, stream));
}

attnq_status attnq_fwd(const attnq_desc* desc, const uint8_t* q8, const uint8_t* k8, const uint8_t* v8,
                       const attnq_scales* scales, float S, int32_t kv_order, int32_t causal, int32_t kv_tile,
                       void* O, int32_t out_dtype, uint64_t* underflow_opt, int32_t k_sink, cudaStream_t stream) {
  attnq_status st = check_desc(desc);
  if (st != ATTNQ_OK) return st;
  if (!q8 || !k8 || !v8 || !scales || !scales->q_descale || !scales->k_descale || !scales->v_descale || !O)
    return ATTNQ_EINVAL;
  if (!aligned16(q8) || !aligned16(k8) || !aligned16(v8) || !aligned16(O)) return ATTNQ_EINVAL;
  if (!pcast_scale_ok(S)) return ATTNQ_EINVAL;
  if (kv_order != ATTNQ_KV_FORWARD && kv_order != ATTNQ_KV_REVERSE) return ATTNQ_EINVAL;
  if (causal != 0 && causal != 1) return ATTNQ_EINVAL;
  if (out_dtype != ATTNQ_F32 && out_dtype != ATTNQ_BF16) return ATTNQ_EINVAL;
  if (k_sink < 0) return ATTNQ_EINVAL;
  if (kv_tile != 64 && kv_tile != 128) return ATTNQ_EUNSUPPORTED;
  if (!(desc->flags & ATTNQ_VT_LAYOUT)) return ATTNQ_EUNSUPPORTED;
  int dev;
  st = device_setup(&dev);
  if (st != ATTNQ_OK) return st;
  FwdArgs a{};
  a.B = desc->B; a.Hq = desc->Hq; a.Hkv = desc->Hkv; a.N = desc->N; a.d = desc->d; a.T = kv_tile;
  a.causal = causal; a.reverse = kv_order == ATTNQ_KV_REVERSE;
  a.rotate = (desc->flags & ATTNQ_ROTATE) != 0;
  a.tiles = (desc->flags & ATTNQ_TILE_SCALES) != 0;
  a.i8 = (desc->flags & ATTNQ_I8QK) != 0;
  a.S = S;
  a.q8 = q8; a.k8 = k8; a.v8t = v8; a.ldv = attnq_vt_ld(desc->N);
  a.q_ds = scales->q_descale; a.k_ds = scales->k_descale; a.v_ds = scales->v_descale;
  a.O = O; a.out_bf16 = out_dtype == ATTNQ_BF16;
  a.underflow = reinterpret_cast<unsigned long long*>(underflow_opt);
  a.k_sink = k_sink;
  a.status = g_status_ptr[dev];
  a.wait_ns = g_wait_ns.load();
  a.num_sms = g_num_sms[dev];
  const NvtxRange range("attnq_fwd");
  return from_cuda(launch_fwd(a, stream));
}

attnq_status attnq_fwd_ponly(const attnq_desc* desc, const float* Q, const float* K, const float* V, float S,
                             int32_t kv_order, int32_t causal, int32_t kv_tile, float* O, uint64_t* underflow_opt,
                             int32_t k_sink, cudaStream_t stream) {
  attnq_status st = check_desc(desc);
  if (st != ATTNQ_OK) return st;
  if (!Q || !K || !V || !O) return ATTNQ_EINVAL;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return ATTNQ_EINVAL;
  if (!(std::isfinite(S) && S > 0.0f && S <= 448.0f)) return ATTNQ_EINVAL;
  if (kv_order != ATTNQ_KV_FORWARD && kv_order != ATTNQ_KV_REVERSE) return ATTNQ_EINVAL;
  if (causal != 0 && causal != 1) return ATTNQ_EINVAL;
  if (k_sink < 0) return ATTNQ_EINVAL;
  if (kv_tile < 16 || kv_tile > 128 || kv_tile % 16) return ATTNQ_EUNSUPPORTED;
  int dev;
  st = device_setup(&dev);
  if (st != ATTNQ_OK) return st;
  PonlyArgs a{};
  a.B = desc->B; a.Hq = desc->Hq; a.Hkv = desc->Hkv; a.N = desc->N; a.d = desc->d; a.T = kv_tile;
  a.causal = causal; a.reverse = kv_order == ATTNQ_KV_REVERSE;
  a.S = S;
  a.Q = Q; a.K = K; a.V = V; a.O = O;
  a.underflow = reinterpret_cast<unsigned long long*>(underflow_opt);
  a.k_sink = k_sink;
  const NvtxRange range("attnq_fwd_ponly");
  return from_cuda(launch_ponly(a, stream));
}

attnq_status attnq_err(const attnq_desc* desc, const void* O, int32_t o_dtype, const double* O_ref,
                       double* err_out, cudaStream_t stream) {
  attnq_status st = check_desc(desc);
  if (st != ATTNQ_OK) return st;
  if (!O || !O_ref || !err_out) return ATTNQ_EINVAL;
  if (o_dtype != ATTNQ_F32 && o_dtype != ATTNQ_BF16) return ATTNQ_EINVAL;
  int dev;
  st = device_setup(&dev);
  if (st != ATTNQ_OK) return st;
  ErrArgs a{};
  a.n_heads = desc->B * desc->Hq;
  a.per_head = int64_t(desc->N) * desc->d;
  a.O = O;
  a.o_bf16 = o_dtype == ATTNQ_BF16;
  a.O_ref = O_ref;
  a.err = err_out;
  const NvtxRange range("attnq_err");
  return from_cuda(launch_err(a, stream));
}

attnq_status attnq_ref_attention(const attnq_desc* desc, const void* Q, const void* K, const void* V,
                                 int32_t causal, double* O_ref, cudaStream_t stream) {
  attnq_status st = check_desc(desc);
  if (st != ATTNQ_OK) return st;
  if (desc->in_dtype != ATTNQ_F32 && desc->in_dtype != ATTNQ_BF16) return ATTNQ_EINVAL;
  if (!Q || !K || !V || !O_ref || (causal != 0 && causal != 1)) return ATTNQ_EINVAL;
  int dev;
  st = device_setup(&dev);
  if (st != ATTNQ_OK) return st;
  RefArgs a{};
  a.B = desc->B; a.Hq = desc->Hq; a.Hkv = desc->Hkv; a.N = desc->N; a.d = desc->d;
  a.bf16 = desc->in_dtype == ATTNQ_BF16;
  a.causal = causal;
  a.Q = Q; a.K = K; a.V = V; a.O_ref = O_ref;
  const NvtxRange range("attnq_ref_attention");
  return from_cuda(launch_ref_attn(a, stream));
}


size_t attnq_harm_workspace(const attnq_desc* desc) {
  if (check_desc(desc) != ATTNQ_OK) return 0;
  return harm_layout(desc).total;
}

attnq_status attnq_harm_report(const attnq_desc* desc, const void* Q, const void* K, const void* V, float S,
                               int32_t kv_order, int32_t kv_tile, void* workspace, size_t ws_bytes,
                               double* err_out, cudaStream_t stream) {
  attnq_status st = check_desc(desc);
  if (st != ATTNQ_OK) return st;
  if (!desc->signs || !err_out || !workspace) return ATTNQ_EINVAL;
  if (!pcast_scale_ok(S)) return ATTNQ_EINVAL;
  const HarmLayout L = harm_layout(desc);
  if (ws_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return ATTNQ_EINVAL;
  char* w = static_cast<char*>(workspace);
  double* O_ref = reinterpret_cast<double*>(w + L.o_ref);
  st = attnq_ref_attention(desc, Q, K, V, 1, O_ref, stream);
  if (st != ATTNQ_OK) return st;
  attnq_scales sc{reinterpret_cast<float*>(w + L.q_ds), reinterpret_cast<float*>(w + L.k_ds),
                  reinterpret_cast<float*>(w + L.v_ds), reinterpret_cast<float*>(w + L.k_mean)};
  const uint32_t conds[4] = {0u, ATTNQ_ROTATE, ATTNQ_CENTER_K, ATTNQ_ROTATE | ATTNQ_CENTER_K};
  const size_t nbh = size_t(desc->B) * desc->Hq;
  for (int c = 0; c < 4; ++c) {
    attnq_desc dc = *desc;
    dc.flags = conds[c] | ATTNQ_VT_LAYOUT;
    uint8_t* q8 = reinterpret_cast<uint8_t*>(w + L.q8);
    uint8_t* k8 = reinterpret_cast<uint8_t*>(w + L.k8);
    uint8_t* v8 = reinterpret_cast<uint8_t*>(w + L.v8);
    st = attnq_prepare(&dc, Q, K, V, q8, k8, v8, &sc, w + L.prep, L.total - L.prep, stream);
    if (st != ATTNQ_OK) return st;
    float* O = reinterpret_cast<float*>(w + L.o);
    st = attnq_fwd(&dc, q8, k8, v8, &sc, S, kv_order, 1, kv_tile, O, ATTNQ_F32, nullptr, 0, stream);
    if (st != ATTNQ_OK) return st;
    st = attnq_err(&dc, O, ATTNQ_F32, O_ref, err_out + c * nbh, stream);
    if (st != ATTNQ_OK) return st;
  }
  return ATTNQ_OK;
}

size_t attnq_host_pipeline_workspace(const attnq_desc* desc, int32_t out_dtype) {
  if (check_desc(desc) != ATTNQ_OK) return 0;
  if (desc->in_dtype != ATTNQ_F32 && desc->in_dtype != ATTNQ_BF16) return 0;
  if (out_dtype != ATTNQ_F32 && out_dtype != ATTNQ_BF16) return 0;
  return pipe_layout(desc, out_dtype).total;
}

attnq_status attnq_attention_host(const attnq_desc* desc, int32_t n_steps, const void* const* Q_host,
                                  const void* const* K_host, const void* const* V_host, float S,
                                  int32_t kv_order, int32_t causal, int32_t kv_tile, void* const* O_host,
                                  int32_t out_dtype, void* workspace, size_t ws_bytes, cudaStream_t compute,
                                  cudaStream_t copy_in, cudaStream_t copy_out) {
  attnq_status st = check_desc(desc);
  if (st != ATTNQ_OK) return st;
  if (desc->in_dtype != ATTNQ_F32 && desc->in_dtype != ATTNQ_BF16) return ATTNQ_EINVAL;
  if (out_dtype != ATTNQ_F32 && out_dtype != ATTNQ_BF16) return ATTNQ_EINVAL;
  if (n_steps < 0 || (n_steps > 0 && (!Q_host || !K_host || !V_host || !O_host))) return ATTNQ_EINVAL;
  for (int32_t i = 0; i < n_steps; ++i)
    if (!Q_host[i] || !K_host[i] || !V_host[i] || !O_host[i]) return ATTNQ_EINVAL;
  if (compute == copy_in || compute == copy_out || copy_in == copy_out) return ATTNQ_EINVAL;
  // what attnq_prepare and attnq_fwd would refuse, refused before any work
  if (!(desc->flags & ATTNQ_VT_LAYOUT)) return ATTNQ_EUNSUPPORTED;
  if ((desc->flags & ATTNQ_ROTATE) && !desc->signs) return ATTNQ_EINVAL;
  if (!pcast_scale_ok(S)) return ATTNQ_EINVAL;
  if (kv_order != ATTNQ_KV_FORWARD && kv_order != ATTNQ_KV_REVERSE) return ATTNQ_EINVAL;
  if (causal != 0 && causal != 1) return ATTNQ_EINVAL;
  if (kv_tile != 64 && kv_tile != 128) return ATTNQ_EUNSUPPORTED;
  const PipeLayout L = pipe_layout(desc, out_dtype);
  if (!workspace || ws_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return ATTNQ_EINVAL;
  int dev;
  st = device_setup(&dev);
  if (st != ATTNQ_OK) return st;
  if (n_steps == 0) return ATTNQ_OK;
  const NvtxRange range("attnq_attention_host");
  PipeEvents E;
  if (E.create() != cudaSuccess) return ATTNQ_ECUDA;
  // ev[0 + b]: inputs of buffer b copied in; ev[2 + b]: buffer b read by its prepare;
  // ev[4 + b]: output buffer b written; ev[6 + b]: output buffer b copied out;
  // ev[8]: start (the work enqueued on `compute` so far)
  cudaEvent_t* in_ready = E.ev, *in_free = E.ev + 2, *out_ready = E.ev + 4, *out_free = E.ev + 6, start = E.ev[8];
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  if (!ok(cudaEventRecord(start, compute)) || !ok(cudaStreamWaitEvent(copy_in, start, 0)) ||
      !ok(cudaStreamWaitEvent(copy_out, start, 0)))
    return ATTNQ_ECUDA;
  char* w = static_cast<char*>(workspace);
  uint8_t* q8 = reinterpret_cast<uint8_t*>(w + L.q8);
  uint8_t* k8 = reinterpret_cast<uint8_t*>(w + L.k8);
  uint8_t* v8 = reinterpret_cast<uint8_t*>(w + L.v8);
  attnq_scales sc{reinterpret_cast<float*>(w + L.q_ds), reinterpret_cast<float*>(w + L.k_ds),
                  reinterpret_cast<float*>(w + L.v_ds), reinterpret_cast<float*>(w + L.k_mean)};
  const void* const* host_in[3] = {Q_host, K_host, V_host};
  for (int32_t i = 0; i < n_steps; ++i) {
    const int b = i & 1;
    // inputs of step i into buffer b, once step i-2's prepare has read it
    if (!ok(cudaStreamWaitEvent(copy_in, in_free[b], 0))) return ATTNQ_ECUDA;
    for (int t = 0; t < 3; ++t)
      if (!ok(cudaMemcpyAsync(w + L.in[b][t], host_in[t][i], L.in_bytes[t], cudaMemcpyHostToDevice, copy_in)))
        return ATTNQ_ECUDA;
    if (!ok(cudaEventRecord(in_ready[b], copy_in)) || !ok(cudaStreamWaitEvent(compute, in_ready[b], 0)))
      return ATTNQ_ECUDA;
    st = attnq_prepare(desc, w + L.in[b][0], w + L.in[b][1], w + L.in[b][2], q8, k8, v8, &sc, w + L.prep,
                       L.total - L.prep, compute);
    if (st != ATTNQ_OK) return st;
    if (!ok(cudaEventRecord(in_free[b], compute))) return ATTNQ_ECUDA;
    // output buffer b, once step i-2's output has been copied out
    if (!ok(cudaStreamWaitEvent(compute, out_free[b], 0))) return ATTNQ_ECUDA;
    st = attnq_fwd(desc, q8, k8, v8, &sc, S, kv_order, causal, kv_tile, w + L.out[b], out_dtype, nullptr, 0,
                   compute);
    if (st != ATTNQ_OK) return st;
    if (!ok(cudaEventRecord(out_ready[b], compute)) || !ok(cudaStreamWaitEvent(copy_out, out_ready[b], 0)) ||
        !ok(cudaMemcpyAsync(O_host[i], w + L.out[b], L.out_bytes, cudaMemcpyDeviceToHost, copy_out)) ||
        !ok(cudaEventRecord(out_free[b], copy_out)))
      return ATTNQ_ECUDA;
  }
  // `compute` waits for the last output copy
  if (!ok(cudaStreamWaitEvent(compute, out_free[(n_steps - 1) & 1], 0))) return ATTNQ_ECUDA;
  return ATTNQ_OK;
}

uint64_t attnq_set_wait_limit_ns(uint64_t ns) {
  return g_wait_ns.exchange(ns);
}

attnq_status attnq_device_status(cudaStream_t stream) {
  int dev;
  attnq_status st = device_setup(&dev);
  if (st != ATTNQ_OK) return st;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return ATTNQ_ECUDA;
  uint32_t bits = 0;
  if (cudaMemcpy(&bits, g_status_ptr[dev], sizeof(bits), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTNQ_ECUDA;
  if (bits) {
    const uint32_t zero = 0;
    if (cudaMemcpy(g_status_ptr[dev], &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return ATTNQ_ECUDA;
  }
  if (bits & DEV_NONFINITE) return ATTNQ_ENONFINITE;
  if (bits & DEV_TIMEOUT) return ATTNQ_ETIMEOUT;
  return ATTNQ_OK;
}

}  // extern "C"
