/*
 * attnq - causal FP8 (E4M3) attention forward with the numerics options of
 * the attention-numerics pages, for GB300 (sm_103a).
 *
 * Sources (page titles and sections):
 *  [AN] "attention-numerics" project page, method and kernel settings:
 *       per-(batch, head) Q/K/V scales over the full sequence; the same
 *       Hadamard transform on Q and K, never V; mean-key subtraction keeps
 *       exact attention; ideal causal FP64 attention as the reference.
 *  [RR] "A rounding problem, not a rotation problem", 01 / Synthetic
 *       illustration (one maximum-based FP8 scale, fixed random-sign
 *       Hadamard, E4M3FN round-to-nearest-even saturating at +-448, mean
 *       subtraction before rotation) and 02 / Measured heads
 *       (log(1 + relative Frobenius error) per head).
 *  [PC] "Technische Samenvatting: P-Cast Precisie in FP8 Attention", sec. 1
 *       (online softmax over KV blocks forward 0->N or reverse N->0; static
 *       scale S multiplied into P before the E4M3 cast and divided out in the
 *       epilogue) and sec. 3-4 (kernel-faithful simulation: Q, K, V in FP32,
 *       only P cast).
 *
 * Conventions for every call:
 *  - Tensor arguments are DEVICE pointers owned by the caller, contiguous,
 *    16-byte aligned, in the layouts stated below.  The library keeps no
 *    allocation between calls and allocates none during a call; scratch
 *    memory comes from the caller's workspace.
 *  - Calls are asynchronous on `stream`.  The return value reports argument
 *    and launch errors found before or at launch.  Errors found on the device
 *    (non-finite input, a wait that timed out) are recorded in a per-device
 *    status word and reported by attnq_device_status().
 *  - The library caches, per device, the device addresses of its status word
 *    and of the attnq_prepare_static scratch array.  cudaDeviceReset destroys
 *    the context they belong to: after it the library must not be used again
 *    in that process.
 *  - No C++ exception crosses this interface.  Functions are thread-safe for
 *    distinct streams except where stated.
 *  - Requires an sm_103 device; other devices give ATTNQ_EUNSUPPORTED.
 */
#ifndef ATTNQ_H_
#define ATTNQ_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTNQ_OK = 0,
  ATTNQ_EINVAL = 1,        /* bad argument: null pointer, bad size, misaligned, workspace too small */
  ATTNQ_EUNSUPPORTED = 2,  /* valid but not supported here: d, kv_tile, device */
  ATTNQ_ECUDA = 3,         /* a CUDA runtime/driver call failed */
  ATTNQ_ENONFINITE = 4,    /* a NaN or infinity in an input (or produced by the transform) */
  ATTNQ_ETIMEOUT = 5       /* a device-side wait gave up (the kernel returned early) */
} attnq_status;

/* desc.flags */
enum { ATTNQ_ROTATE = 1u, ATTNQ_CENTER_K = 2u, ATTNQ_VT_LAYOUT = 4u, ATTNQ_TILE_SCALES = 8u, ATTNQ_I8QK = 16u };
/* tokens per scale tile of ATTNQ_TILE_SCALES */
enum { ATTNQ_SCALE_TILE = 128 };
/* element types of Q/K/V inputs and of O */
enum { ATTNQ_F32 = 0, ATTNQ_BF16 = 1 };
/* KV-tile visiting order of the online softmax [PC sec. 1] */
enum { ATTNQ_KV_FORWARD = 0, ATTNQ_KV_REVERSE = 1 };

/*
 * Problem description.  Q is [B, Hq, N, d]; K and V are [B, Hkv, N, d];
 * query head h reads KV head h / (Hq / Hkv) (Hq must be a multiple of Hkv).
 * d is 64 or 128.  in_dtype is ATTNQ_F32 or ATTNQ_BF16 (inputs of
 * attnq_prepare).  flags:
 *   ATTNQ_ROTATE    multiply Q and K rows by `signs` and apply the
 *                   unnormalised fast Walsh-Hadamard transform [AN], [RR];
 *   ATTNQ_CENTER_K  subtract from K the mean key of its (batch, KV head) over
 *                   all N tokens, before rotation [AN], [RR];
 *   ATTNQ_VT_LAYOUT v8 is stored transposed, [B, Hkv, d, ldv] with
 *                   ldv = attnq_vt_ld(N) (tokens N .. ldv-1 are zero);
 *   ATTNQ_TILE_SCALES  Q and K get one max-based scale per 128-token tile of
 *                   each (batch, head), tiles aligned at token 0, instead of
 *                   one per (batch, head) (the emulator's per-tile scales that
 *                   the "attention-numerics" page, method and kernel settings,
 *                   contrasts with the API's full-sequence scales); V keeps
 *                   one scale per (batch, head).
 *   ATTNQ_I8QK      INT8-QK / FP8-PV (the INT8-QK / FP8-PV kernel the
 *                   "attention-numerics" page, method and kernel settings,
 *                   runs; the page names only the formats): Q and K get
 *                   symmetric INT8 codes, the nearest integer (ties to even)
 *                   of fl32(x * qs) with qs = 127/amax, saturated to +-127,
 *                   stored as bf16 values (2 bytes per code: the integers are
 *                   exact in bf16, and GB300 multiplies them exactly on its
 *                   bf16 tensor path, its INT8 path being far slower); q.k is
 *                   then an exact integer sum (|q.k| <= 128 * 127^2 < 2^24, so
 *                   fp32 accumulation keeps it exactly).  V and P stay E4M3.
 * signs: DEVICE pointer to d int8 values, each +1 or -1; required when
 * ATTNQ_ROTATE is set, ignored otherwise.
 * stat_len: 0 (full sequence), or P in 1..N: causal-prefix statistics.  The
 *   mean key and the one-per-(batch, head) amax of attnq_prepare are taken
 *   over the first P tokens of each slice only, and all N tokens are centred
 *   and cast with them; a later value above the prefix amax saturates at
 *   +-448 by the cast's rule.  The "attention-numerics" page (limitations)
 *   notes that full-sequence means and scales see future tokens; this is the
 *   generation-safe form when the first P tokens are a prompt known before
 *   the rest.  Per-tile Q/K scales (ATTNQ_TILE_SCALES) are local to their
 *   tile and ignore it; V's scale and the mean key still use it.
 *   A zero-initialised descriptor has stat_len = 0.
 */
typedef struct {
  int32_t B, Hq, Hkv, N, d;
  int32_t in_dtype;
  uint32_t flags;
  const int8_t* signs;
  int32_t stat_len;
} attnq_desc;

/*
 * Per-(batch, head) descales (amax / 448, fp32) written by attnq_prepare and
 * read by attnq_fwd: q_descale [B*Hq], k_descale and v_descale [B*Hkv].
 * With ATTNQ_TILE_SCALES: q_descale [B*Hq*nt] and k_descale [B*Hkv*nt],
 * nt = attnq_scale_tiles(N), tile t of slice s at s*nt + t; v_descale as above.
 * k_mean: optional [B*Hkv*d] fp32 output of the mean key (may be NULL).
 */
typedef struct {
  float* q_descale;
  float* k_descale;
  float* v_descale;
  float* k_mean;
} attnq_scales;

/* Scale tiles per (batch, head) slice: ceil(N / ATTNQ_SCALE_TILE); 0 if N <= 0. */
int32_t attnq_scale_tiles(int32_t N);

/* Library version: major*10000 + minor*100 + patch. */
int32_t attnq_version(void);

/* Human-readable name of a status code (static storage). */
const char* attnq_status_string(attnq_status s);

/*
 * Row length in bytes of the transposed V layout: N rounded up to 16
 * (TMA needs 16-byte row strides).  Returns 0 for N <= 0.
 */
int64_t attnq_vt_ld(int32_t N);

/*
 * Fixed random signs for the Hadamard rotation [RR: "fixed random-sign
 * Hadamard"]: sign c is -1 when bit 63 of SplitMix64 output c+1 of stream
 * `seed` is set, else +1.  Writes d values to HOST memory host_out.
 */
attnq_status attnq_hadamard_signs(uint64_t seed, int32_t d, int8_t* host_out);

/* Bytes of device workspace attnq_prepare needs for `desc` (0 on a bad desc). */
size_t attnq_prepare_workspace(const attnq_desc* desc);

/*
 * Operand preparation [AN], [RR]: for every (batch, head) slice of Q, K, V
 *   1. upcast to fp32;
 *   2. K only, with ATTNQ_CENTER_K: subtract the mean key mu (fp32; per
 *      channel, 128-token chunks of the first P tokens summed in token
 *      order, chunk sums added in chunk order, one IEEE division by P;
 *      P = desc->stat_len, or N when it is 0);
 *   3. Q and K only, with ATTNQ_ROTATE: x <- FWHT(signs * x), unnormalised,
 *      butterfly stages h = 1, 2, ..., d/2;
 *   4. amax = max |x| over the first P tokens of the slice (over each
 *      128-token tile for Q and K with ATTNQ_TILE_SCALES); descale =
 *      amax/top and qs = top/amax (IEEE fp32 division; 1 and 1 when
 *      amax == 0), top = 448, or 127 for Q and K with ATTNQ_I8QK;
 *   5. x8 = E4M3 code of fl32(x * qs), round-to-nearest-even, saturating
 *      (Q and K with ATTNQ_I8QK: the INT8 code of fl32(x * qs) as a bf16).
 * Q, K, V: DEVICE, in_dtype elements, [B,H,N,d].  q8 [B,Hq,N,d], k8
 * [B,Hkv,N,d]: DEVICE uint8 E4M3 codes (with ATTNQ_I8QK: bf16, 2 bytes
 * each).  v8: [B,Hkv,N,d], or [B,Hkv,d,attnq_vt_ld(N)] with
 * ATTNQ_VT_LAYOUT.  out: descales (and the
 * optional mean key) as DEVICE pointers.  workspace: DEVICE, at least
 * attnq_prepare_workspace(desc) bytes, 256-byte aligned; its contents need no
 * initialisation and are garbage afterwards.  A non-finite value in an input
 * slice (or produced by its transform), inside the prefix or after it, sets
 * ATTNQ_ENONFINITE in the device status; outputs are then unspecified.
 * Returns ATTNQ_EINVAL for stat_len < 0 or > N.
 */
attnq_status attnq_prepare(const attnq_desc* desc, const void* Q, const void* K, const void* V, uint8_t* q8,
                           uint8_t* k8, uint8_t* v8, const attnq_scales* out, void* workspace, size_t ws_bytes,
                           cudaStream_t stream);

/*
 * attnq_prepare without a caller workspace.  The pages have no counterpart:
 * this is a calling convention, not part of the method.  It is for callers
 * that cannot allocate device memory when they call (for example a plugin
 * hook of an inference runtime that must not allocate, or a process whose
 * device memory is owned by another allocator).  The scratch lives in a fixed
 * ATTNQ_STATIC_SCRATCH_BYTES array inside the library, which every GPU that
 * loads the library holds until the process exits.  Arguments and results as
 * attnq_prepare.  Returns ATTNQ_EUNSUPPORTED, before launching anything, when
 * attnq_prepare_workspace(desc) exceeds ATTNQ_STATIC_SCRATCH_BYTES.  The
 * first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  The call allocates nothing.  All calls share the one array and
 * it keeps the last call's contents (each call clears what must start at
 * zero): calls whose kernels overlap on the GPU - other streams, other host
 * threads - race on it and must be serialised by the caller.
 */
#define ATTNQ_STATIC_SCRATCH_BYTES (4u << 20)
attnq_status attnq_prepare_static(const attnq_desc* desc, const void* Q, const void* K, const void* V, uint8_t* q8,
                                  uint8_t* k8, uint8_t* v8, const attnq_scales* out, cudaStream_t stream);

/*
 * Causal FP8 attention forward [AN], [PC sec. 1]: for each query row i and
 * the KV tiles of width kv_tile (aligned at token 0) holding a key j <= i
 * (every key when causal == 0), visited forward (0 -> diagonal) or reverse
 * (diagonal -> 0):
 *   s_j = q8_i . k8_j (exact products, fp32 accumulation; with ATTNQ_I8QK
 *         an exact integer sum of INT8 codes held in bf16);
 *   t_j = s_j * c,  c = fl32(cq * dk), cq = fl32(dq / sqrt(d) * (ROTATE ? 1/d : 1) * log2 e)
 *   (cq in double);
 *   m' = max(m, max_j t_j);  alpha = 2^(m - m');  P_j = 2^(t_j - m');
 *   l = alpha * l + sum_j P_j;  p8_j = E4M3(P_j * S);
 *   acc = alpha * acc + sum_j p8_j * v8_j;
 * and finally O = acc * dv / (S * l).  The running maximum is exact (no
 * lazy rescaling).  The kernel evaluates P_j * S in one step, as
 * 2^(fma(s_j, c, log2 S - m')) with ex2.approx (exact 2^x for S a power of
 * two; for other S, log2 S rounded to fp32), and its row sum accumulates
 * P_j * S, which equals S * l up to rounding; the cast and the division by
 * S * l are as stated.  E4M3 codes, and so the underflow counts, can
 * therefore differ from the literal two-step P then P * S where P * S lies
 * within a few ulp of a rounding boundary.  The fma takes the exact product
 * s_j * c where the two-step form rounds t_j to fp32 first: each P differs
 * from it by a relative |t_j| * 2^-25 at most (t in log2 units), under 1e-4
 * for |t_j| < 2^12.  A factor c below the smallest
 * normal float (FLT_MIN) is raised to FLT_MIN: every logit is then below
 * 2^-100 in magnitude either way (|s_j| < 2^25) and every P is 1 in fp32, so no result
 * changes, and masked keys keep P * S = 0.  A factor above the largest
 * float (descale products near 1e39 and beyond: logits past the fp32 range)
 * makes c infinite, as in the plain two-step evaluation: masked keys still
 * give P * S = 0, and an unmasked score of exactly 0 gives NaN.  With ATTNQ_TILE_SCALES, dq is row i's query tile's and dk
 * key j's tile's descale (kv_tile divides the scale tile, so c is constant
 * within a KV tile).  desc: shape and flags of the attnq_prepare call that made
 * the operands (ATTNQ_VT_LAYOUT is required; in_dtype is ignored).
 * q8, k8, v8, scales: DEVICE, as written by attnq_prepare.  S: finite, in
 * (0, 448], and not within a relative 2^-20 of a point where E4M3 rounding
 * changes (S = 100, halfway between the codes 96 and 104, is refused with
 * ATTNQ_EINVAL): the row maximum's P * S, exactly S in the two-step form,
 * comes out of the single exp2 within a few 2^-24 of S and must round as S
 * does.  The pages' 1, 256 and 448 are E4M3 values, as is every power of two
 * in range.  kv_order: ATTNQ_KV_FORWARD or ATTNQ_KV_REVERSE.  kv_tile: 64 or
 * 128.  O: DEVICE [B,Hq,N,d] of out_dtype (ATTNQ_F32 or ATTNQ_BF16, RNE).
 * underflow_opt: NULL, or DEVICE uint64 [B*Hq*2] that the call ADDS to:
 * [2*bh] counts in-mask keys j >= k_sink of KV tile 0 whose P*S > 0 was cast
 * to 0, [2*bh+1] the same over all later tiles [PC sec. 1-2].
 */
attnq_status attnq_fwd(const attnq_desc* desc, const uint8_t* q8, const uint8_t* k8, const uint8_t* v8,
                       const attnq_scales* scales, float S, int32_t kv_order, int32_t causal, int32_t kv_tile,
                       void* O, int32_t out_dtype, uint64_t* underflow_opt, int32_t k_sink, cudaStream_t stream);

/*
 * P-only ("kernel-faithful simulation") forward [PC sec. 3-4]: the loop of
 * attnq_fwd on fp32 Q [B,Hq,N,d], K, V [B,Hkv,N,d] (DEVICE) with fp32 dot
 * products, c = fl32(log2 e / sqrt(d)), only P cast to E4M3, O = acc/(S*l)
 * (DEVICE fp32 [B,Hq,N,d]).  desc.flags and desc.in_dtype are ignored.
 * Other arguments as attnq_fwd.  d is 64 or 128; kv_tile 16..128, a
 * multiple of 16.
 */
attnq_status attnq_fwd_ponly(const attnq_desc* desc, const float* Q, const float* K, const float* V, float S,
                             int32_t kv_order, int32_t causal, int32_t kv_tile, float* O, uint64_t* underflow_opt,
                             int32_t k_sink, cudaStream_t stream);

/*
 * Per-head error [RR, 02 / Measured heads]: err[bh] = log1p(||O - O_ref||_F
 * / ||O_ref||_F) over the N*d outputs of head bh, with both squared norms
 * accumulated in fp64.  O: DEVICE [B,Hq,N,d] of o_dtype; O_ref: DEVICE fp64
 * [B,Hq,N,d]; err_out: DEVICE fp64 [B*Hq] (overwritten).  A head with
 * ||O_ref|| = 0 gives 0 when O equals O_ref there, else +infinity.
 */
attnq_status attnq_err(const attnq_desc* desc, const void* O, int32_t o_dtype, const double* O_ref,
                       double* err_out, cudaStream_t stream);

/*
 * FP64 reference attention ("A rounding problem, not a rotation problem",
 * 02 / Measured heads: errors are measured against the ideal causal attention
 * in FP64): O_ref[b,h,i] = sum_j softmax_j(q_i . k_j / sqrt(d)) v_j over
 * j <= i (causal = 1) or all j (causal = 0), on the original inputs upcast
 * exactly to double.  desc: B, Hq, Hkv, N, d and in_dtype are used, flags and
 * signs are ignored.  Q, K, V: DEVICE [B,H,N,d] of in_dtype; O_ref: DEVICE fp64
 * [B,Hq,N,d] (overwritten).  Online softmax in double; differs from a two-pass
 * evaluation only by double rounding.  Bounded by the GPU's FP64 rate: a
 * checking tool, not a fast path.
 */
attnq_status attnq_ref_attention(const attnq_desc* desc, const void* Q, const void* K, const void* V,
                                 int32_t causal, double* O_ref, cudaStream_t stream);

/*
 * Batched four-condition report [RR, 02 / Measured heads; 03 / harm score]:
 * for each condition c = 0 unrotated, 1 rotated, 2 centred, 3 centred and
 * rotated, runs attnq_prepare (flags = the condition | ATTNQ_VT_LAYOUT) and
 * attnq_fwd (causal, fp32 output) on Q, K, V and writes the per-head error
 * against attnq_ref_attention to err_out[c * B*Hq + bh] (DEVICE fp64 [4][B*Hq]).
 * A head's rotation harm score is err[1] - err[0] (the pages average it over
 * the batch, their "texts").  desc->signs (DEVICE, d entries of +-1) is
 * required; desc->flags is ignored (the conditions use E4M3 codes and one
 * scale per (batch, head)); desc->stat_len applies.  workspace: DEVICE, 256-byte aligned, at
 * least attnq_harm_workspace(desc) bytes (it holds the fp64 reference, the
 * fp32 output, the E4M3 operands and the prepare workspace).  S: as for
 * attnq_fwd (checked before any launch).  Errors of any other step are
 * returned as that step returns them.
 */
size_t attnq_harm_workspace(const attnq_desc* desc);
attnq_status attnq_harm_report(const attnq_desc* desc, const void* Q, const void* K, const void* V, float S,
                               int32_t kv_order, int32_t kv_tile, void* workspace, size_t ws_bytes,
                               double* err_out, cudaStream_t stream);

/*
 * Host-buffer pipeline over the whole path (no counterpart on the pages: the
 * pages' prepare -> causal FP8 attention forward, "attention-numerics" method
 * and kernel settings, run on inputs that live in host memory).  For each step
 * i < n_steps, with the same desc, S, kv_order, causal and kv_tile:
 *   Q_host[i], K_host[i], V_host[i] --copy--> device, attnq_prepare,
 *   attnq_fwd --> device O --copy--> O_host[i].
 * desc->flags must include ATTNQ_VT_LAYOUT.  Q/K/V_host[i]: HOST [B,H,N,d] of
 * desc->in_dtype; O_host[i]: HOST [B,Hq,N,d] of out_dtype (ATTNQ_F32 or
 * ATTNQ_BF16).  The arrays of pointers are read during the call only.  Host
 * buffers should be page-locked (cudaHostAlloc / cudaHostRegister); pageable
 * memory still gives the right result, but its copies do not overlap.
 * Streams: the kernels run on `compute`, input copies on `copy_in`, output
 * copies on `copy_out` (three distinct streams of the current device).  The
 * workspace holds two input and two output buffers, so step i+1's inputs are
 * copied in and step i-1's output out while step i's kernels run.  All work of
 * the call starts after the work enqueued on `compute` before it, and the call
 * makes `compute` wait for its last output copy: once `compute` is
 * synchronised every O_host[i] is written.  The call returns after enqueueing.
 * workspace: DEVICE, 256-byte aligned, at least
 * attnq_host_pipeline_workspace(desc, out_dtype) bytes; the caller keeps it
 * (and the host buffers) alive until `compute` has synchronised.  Argument
 * errors (and a desc that attnq_prepare or attnq_fwd would refuse) are
 * returned before anything is enqueued; ATTNQ_ECUDA if a copy or an event
 * operation fails, after which part of the work may be enqueued.  Device-side
 * conditions are reported by attnq_device_status as for the two calls.
 */
size_t attnq_host_pipeline_workspace(const attnq_desc* desc, int32_t out_dtype);
attnq_status attnq_attention_host(const attnq_desc* desc, int32_t n_steps, const void* const* Q_host,
                                  const void* const* K_host, const void* const* V_host, float S,
                                  int32_t kv_order, int32_t causal, int32_t kv_tile, void* const* O_host,
                                  int32_t out_dtype, void* workspace, size_t ws_bytes, cudaStream_t compute,
                                  cudaStream_t copy_in, cudaStream_t copy_out);

/*
 * Synchronises `stream`, then returns and clears the device status word of
 * the current device: ATTNQ_OK, ATTNQ_ENONFINITE or ATTNQ_ETIMEOUT (the
 * first error recorded since the last call), or ATTNQ_ECUDA when the
 * synchronisation itself failed.  Not thread-safe against kernels of this
 * library running on other streams of the same device.
 */
attnq_status attnq_device_status(cudaStream_t stream);

/*
 * Failure-detection knob (no counterpart on the pages): every wait inside the
 * library's kernels (on an mbarrier, or on a flag another CTA publishes) gives
 * up after `ns` nanoseconds, records ATTNQ_ETIMEOUT in the device status word
 * and lets the kernel finish: in-flight copies and tensor-core operations are
 * drained with a separate one-second bound, tensor memory is freed.  With
 * ns = 0 any wait that is not already satisfied gives up at once, which drives
 * the timeout path without a hang.  Applies to launches made after the call
 * (process-wide); returns the previous value.  Default 2,000,000,000 (2 s).
 */
uint64_t attnq_set_wait_limit_ns(uint64_t ns);

#ifdef __cplusplus
}
#endif

#endif /* ATTNQ_H_ */
