/*
 * pfa.h -- C ABI of libpfa: stabilised BF16 flash attention (forward and
 * backward) for one GB300 GPU (sm_103a).
 *
 * The method is the one analysed in Qiu & Yao, "Why Low-Precision Transformer
 * Training Fails: An Analysis on Flash Attention" (ICLR 2026). Citations name the
 * page that describes each operation:
 *   [PK] priors.kr post "BF16 플래시 어텐션은 왜 수천 스텝 뒤에 무너질까"
 *   [BN] bud-325 note "Why Low-Precision Transformer Training Fails: An Analysis
 *        on Flash Attention"
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensors are dense, contiguous, row-major [B, H, N, d] with d innermost
 *    ("BHND"). Q, O, dO, dQ have H = H_q heads; K, V, dK, dV have H = H_kv heads;
 *    query head h reads key/value head h / (H_q / H_kv). lse and delta are
 *    [B, H_q, N] FP32.
 *  - BF16 tensors are passed as pointers to raw bfloat16 bit patterns
 *    (pfa_bf16). FP32 tensors are float pointers.
 *  - Every data pointer is DEVICE memory on the current CUDA device, owned by the
 *    caller, 16-byte aligned. The library allocates nothing and never
 *    synchronises: all work is enqueued on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream) and results are ready when that stream reaches them.
 *  - Supported sizes: B, H_q, H_kv >= 1 with H_q % H_kv == 0; N >= 1 (any length,
 *    ragged tails are masked); d in {64, 128}; B * H * N * d < 2^31 elements per
 *    tensor. `scale` is alpha in S = alpha Q K^T and must be finite and > 0
 *    (1/sqrt(d) is the usual choice). causal != 0 lets query i see keys j <= i.
 *  - Return value: PFA_OK (0) or a negative PFA_ERR_* code. Arguments are checked
 *    before anything is enqueued; on an argument error nothing is launched. No
 *    C++ exception crosses this interface.
 *  - Kernels never trap. A kernel whose internal pipeline wait exceeds about one
 *    second gives up, sets a bit in the library's device error word and returns;
 *    pfa_device_error() reads that word.
 *  - Every kernel is launched as a programmatic dependent of the work before it
 *    on `stream`: it may start its setup while the previous kernel finishes, but
 *    touches no global memory until that kernel has completed, so stream order
 *    is kept. It also lets the next kernel on the stream start early; a caller's
 *    kernel launched the same way must wait (griddepcontrol.wait) before reading
 *    this library's outputs.
 */
#ifndef PFA_H_
#define PFA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* pfa_stream_t; /* == cudaStream_t */
typedef uint16_t pfa_bf16;                /* raw bfloat16 bit pattern */

enum {
  PFA_OK = 0,
  PFA_ERR_INVALID_ARG = -1, /* null pointer, bad size, bad mode/beta/eps/scale */
  PFA_ERR_MISALIGNED = -2,  /* a pointer is not 16-byte aligned */
  PFA_ERR_UNSUPPORTED = -3, /* no sm_103 device current, or driver lacks TMA map encoding */
  PFA_ERR_LAUNCH = -4,      /* a CUDA launch or runtime call failed */
  PFA_ERR_DEVICE = -5,      /* pfa_device_error(): a kernel reported a failure */
  PFA_ERR_TOO_LARGE = -6    /* pfa_attn_bwd_noalloc: problem exceeds its fixed buffer */
};

/* Device error word bits, as returned by pfa_device_error(). */
#define PFA_DEVERR_TIMEOUT 1    /* a bounded pipeline wait gave up */
#define PFA_DEVERR_SMEM_ALIGN 2 /* dynamic shared memory was not 1024-byte aligned */

/* Diagnostic counters, int64 each, in DEVICE memory owned by the caller. Calls
 * ADD to them (the caller zeroes them). Definitions, per row of the forward pass:
 *   repeated_rows  rows whose maximum score r_m is reached again within eps
 *                  ([PK] the fix, paper §4; the quantity of paper Fig. 13);
 *   ones           entries whose BF16 Pbar = exp(S - m) equals 1.0 under the
 *                  row's final shift m ([PK] core idea: the exact-1 entries that
 *                  bias the BF16 sum);
 *   nonfinite_rows rows whose normaliser l is 0 or not finite (the underflow of
 *                  [PK] caveats / paper App. C). */
typedef struct pfa_counters {
  int64_t repeated_rows;
  int64_t ones;
  int64_t nonfinite_rows;
} pfa_counters;

/* Forward pass ([PK] equations and the fix of paper §4; [BN] Method, Algorithm 1).
 * Per row i: S = alpha q_i K^T over the visible keys, r_m = max S, the row is
 * "repeated" when a second score lies within `eps` of r_m, and the shift m is
 *   fix_mode 0: m = r_m (plain safe softmax);
 *   fix_mode 1: repeated rows m = beta*r_m if r_m > 0, 0 if r_m < 0, 2^-5 if
 *               r_m == 0; other rows m = r_m;
 *   fix_mode 2: repeated rows m = r_m + 2^-5; other rows m = r_m.
 * Pbar = exp(S - m) in FP32, l = its row sum (FP32), O = (BF16(Pbar) V) / l
 * rounded to BF16 (the product accumulates in FP32), lse = m + ln(l) in FP32.
 *   q [B,H_q,N,d], k, v [B,H_kv,N,d] (in); o [B,H_q,N,d], lse [B,H_q,N] (out).
 *   beta > 1 (mode 1; [PK] recommends 2..8; ignored otherwise).
 *   eps >= 0 finite: the tie tolerance ([PK] suggests 1e-3). It selects the rows
 *   the fix shifts in modes 1 and 2, and the rows counted in repeated_rows (every
 *   mode); it is ignored in mode 0 without counters.
 *   counters: optional (NULL skips the counting work).
 * With the beta shift, rows with a large repeated maximum can underflow (l = 0):
 * O is then NaN, lse is -inf and the row is counted in nonfinite_rows, as the
 * pages describe the failure; no guard is applied. */
int pfa_attn_fwd(const pfa_bf16* q, const pfa_bf16* k, const pfa_bf16* v, pfa_bf16* o, float* lse,
                 int B, int H_q, int H_kv, int N, int d, int causal, float scale, int fix_mode,
                 float beta, float eps, pfa_counters* counters, pfa_stream_t stream);

/* Training-time monitor of the forward pass (no counterpart in the paper; the
 * quantity of paper Fig. 13 -- the rows whose maximum repeats, counted by
 * pfa_counters -- and the two views of it that a tiled kernel can report), in
 * DEVICE memory owned by the caller. Calls ADD to it (the caller zeroes it).
 *   operational_ones  BF16 Pbar entries equal to 1.0 that the kernel handed to the
 *                     Pbar V product, over every 128-key tile of every row, each
 *                     under the shift in use for that tile (the running maximum and
 *                     the repetition flag of the keys up to that tile). Before a
 *                     row's final maximum is seen, its earlier tiles can carry ones
 *                     that pfa_counters.ones (final shift only) does not count.
 *   tie_hist[b]       rows whose maximum r_m has multiplicity b + 1 (entries within
 *                     eps of r_m), b = 0..6, and b = 7 for multiplicity >= 8. The
 *                     kernel counts the entries within eps of its running maximum,
 *                     restarting when the maximum rises by more than eps: exact
 *                     whenever distinct scores near a row's maximum lie more than
 *                     eps apart (always when scores are exact multiples of a grid
 *                     coarser than eps), an upper bound otherwise. */
#define PFA_TIE_BINS 8
typedef struct pfa_monitor {
  int64_t operational_ones;
  int64_t tie_hist[PFA_TIE_BINS];
} pfa_monitor;

/* Options of pfa_attn_fwd_ex (no counterpart in the paper), OR-ed into `flags`. */
#define PFA_FWD_UNFUSED_BF16_PV 1u /* study profile, d = 64 only: each 128-key tile's
                                      product Pbar V is rounded to BF16 and accumulated
                                      across tiles in BF16 (Obar = bf16(bf16(Obar x corr)
                                      + bf16(Pbar V))), and l sums the BF16 Pbar; the way an
                                      implementation that stores the unnormalised product
                                      in BF16 computes O ([PK] caveats: the analysed code
                                      keeps P V in BF16). Not a fast path. */

#define PFA_FWD_PBAR_E4M3 2u         /* study, d = 64: Pbar is rounded to FP8 E4M3 (nearest,
                                        ties to even, saturating) before the Pbar V product */
#define PFA_FWD_PBAR_MXFP4 4u        /* study, d = 64: Pbar is rounded to MXFP4: E2M1 values
                                        with one power-of-two scale 2^(floor(log2 amax) - 2)
                                        per 32 consecutive keys. With either narrow format l
                                        sums the rounded values (the weights the product
                                        uses); the rounded values are exact in BF16, so the
                                        BF16 product with FP32 accumulation computes what a
                                        product in that format does. The pages leave open how
                                        the bias behaves with fewer mantissa bits ([PK] open
                                        questions). Combine with PFA_FWD_UNFUSED_BF16_PV for the
                                        paper's profile; not with each other. */
#define PFA_FWD_PAIR_CTA 8u          /* d = 128, the fused path (no monitor, no study flag):
                                        the two CTAs of a thread-block cluster share every
                                        tensor-core product (tcgen05 cta_group::2, M = 256),
                                        each holding half of each K and V tile, so that a
                                        CTA's K / V loads and shared-memory operand reads
                                        halve. Same outputs and counters as without it, up to
                                        the FP32 summation order of the products. */

/* pfa_attn_fwd with the monitor and options (no counterpart in the paper).
 * counters and monitor are optional (NULL); flags 0 and monitor NULL is
 * pfa_attn_fwd exactly. The study flags with d != 64, and PFA_FWD_PAIR_CTA with
 * d != 128, a monitor or a study flag, return PFA_ERR_UNSUPPORTED; unknown flag
 * bits, or both narrow formats, PFA_ERR_INVALID_ARG. eps must be finite and >= 0
 * when a monitor is given. */
int pfa_attn_fwd_ex(const pfa_bf16* q, const pfa_bf16* k, const pfa_bf16* v, pfa_bf16* o, float* lse,
                    int B, int H_q, int H_kv, int N, int d, int causal, float scale, int fix_mode,
                    float beta, float eps, pfa_counters* counters, pfa_monitor* monitor,
                    unsigned flags, pfa_stream_t stream);

/* delta = rowsum(dO o O) in FP32 from the BF16 forward output ([PK] three-line
 * summary and method, paper §3.2; [BN] Key claims).
 *   o, dO [B,H_q,N,d] (in); delta [B,H_q,N] (out). */
int pfa_attn_delta(const pfa_bf16* o, const pfa_bf16* dO, float* delta, int B, int H_q, int N,
                   int d, pfa_stream_t stream);

/* pfa_attn_delta, and in the same pass the dQ workspace of pfa_attn_bwd zeroed (no
 * counterpart in the paper): the workspace's row (b, h, i) of d FP32 values is
 * cleared by the threads that read row i of O and dO, so the backward call can skip
 * its own zeroing pass (pfa_attn_bwd_ex with PFA_BWD_WORKSPACE_ZEROED), one pass over
 * memory fewer per step. Useful at d = 64, where pfa_attn_bwd uses the workspace.
 *   o, dO [B,H_q,N,d] (in); delta [B,H_q,N] (out);
 *   dq_accum: the workspace, at least B*H_q*N*d FP32 values, 16-byte aligned (out: zero).
 * Same checks and errors as pfa_attn_delta; dq_accum NULL is PFA_ERR_INVALID_ARG. */
int pfa_attn_delta_zero(const pfa_bf16* o, const pfa_bf16* dO, float* delta, float* dq_accum, int B,
                        int H_q, int N, int d, pfa_stream_t stream);

/* delta = rowsum(dP o P) with P = exp(alpha Q K^T - lse) and dP = dO V^T
 * recomputed: the mathematically equal alternative of [PK] method, paper §3.2.
 *   q, dO [B,H_q,N,d], k, v [B,H_kv,N,d], lse [B,H_q,N] (in); delta (out). */
int pfa_attn_delta_alt(const pfa_bf16* q, const pfa_bf16* k, const pfa_bf16* v, const pfa_bf16* dO,
                       const float* lse, float* delta, int B, int H_q, int H_kv, int N, int d,
                       int causal, float scale, pfa_stream_t stream);

/* Backward pass ([PK] equations: dS = alpha P o (dP - delta), dQ = dS K; with
 * dK = dS^T Q and dV = P^T dO summed over the query heads of a key/value head).
 * P is recomputed from lse; the fix does not change the backward pass ([PK] the
 * fix paragraph; [BN] Results).
 *   q, dO [B,H_q,N,d], k, v [B,H_kv,N,d], lse, delta [B,H_q,N] (in);
 *   dq [B,H_q,N,d], dk, dv [B,H_kv,N,d] (out, BF16);
 *   dq_accum: FP32 workspace of pfa_bwd_workspace_bytes() bytes, caller-owned
 *   device memory; its contents on entry are ignored (it is zeroed on `stream`).
 * At d = 64 the key-outer kernel reduce-adds each key tile's dQ into the
 * workspace, which is then converted to BF16. At d = 128 dQ comes from the
 * query-outer pass of pfa_attn_bwd_ex (PFA_BWD_DQ_DETERMINISTIC), which is faster
 * there; the workspace is then not touched. */
int pfa_attn_bwd(const pfa_bf16* q, const pfa_bf16* k, const pfa_bf16* v, const pfa_bf16* dO,
                 const float* lse, const float* delta, pfa_bf16* dq, pfa_bf16* dk, pfa_bf16* dv,
                 float* dq_accum, int B, int H_q, int H_kv, int N, int d, int causal, float scale,
                 pfa_stream_t stream);

/* The backward kernel alone, accumulating dQ in FP32 (no counterpart in the
 * paper): dq_accum += dS K (dS = alpha P o (dP - delta) as above, so alpha
 * enters once), and dK, dV (BF16) are written, with the same
 * arguments, equations and checks as pfa_attn_bwd. dq_accum is [B, H_q, N, d]
 * FP32, caller-owned device memory, 16-byte aligned; it is neither zeroed nor
 * converted. For gradient accumulation across calls (micro-batches or chunks of
 * keys), or to keep dQ in FP32. pfa_attn_bwd is: zero the workspace, this
 * call, convert the workspace to BF16. */
int pfa_attn_bwd_accum(const pfa_bf16* q, const pfa_bf16* k, const pfa_bf16* v, const pfa_bf16* dO,
                       const float* lse, const float* delta, float* dq_accum, pfa_bf16* dk,
                       pfa_bf16* dv, int B, int H_q, int H_kv, int N, int d, int causal, float scale,
                       pfa_stream_t stream);

/* Options of pfa_attn_bwd_ex (no counterpart in the paper), OR-ed into `flags`. */
#define PFA_BWD_DQ_DETERMINISTIC 1u /* dQ by a separate query-outer pass: one CTA sums each
                                       dQ row over the key tiles in a fixed order into FP32,
                                       so repeated calls give identical bits */
#define PFA_BWD_DQ_SPLIT 2u         /* (implies the query-outer pass) dS enters the dQ product
                                       as two BF16 terms, hi = bf16(dS) and lo = bf16(dS - hi):
                                       about 16 significant bits instead of 8. For inputs where
                                       keys that share a large feature get nearly cancelling dS
                                       (a sink key copied into other positions), where the single
                                       BF16 cast of dS dominates the error of dQ. */
#define PFA_BWD_WORKSPACE_ZEROED 4u /* (the reduce-add dQ of pfa_attn_bwd) the caller vouches that
                                       dq_accum holds zeros, as pfa_attn_delta_zero on the same
                                       stream leaves it; the zeroing pass is skipped. Ignored
                                       by the query-outer pass, which uses no workspace. */

/* The backward pass of pfa_attn_bwd with options (no counterpart in the paper).
 * flags == 0 is pfa_attn_bwd exactly; PFA_BWD_WORKSPACE_ZEROED alone is pfa_attn_bwd
 * without its zeroing pass. With PFA_BWD_DQ_DETERMINISTIC or
 * PFA_BWD_DQ_SPLIT the key-outer kernel computes dK and dV only, and a
 * query-outer pass recomputes S, P, dP and dS per query tile to form
 * dQ = dS K (the equation of pfa_attn_bwd, [PK] equations; alpha is in dS): it costs two
 * more products per tile pair (S and dP again) and, with the split, a second dQ
 * product. dq_accum is then not used and may be NULL. Other unknown flag bits
 * return PFA_ERR_INVALID_ARG. Same arguments, layouts and checks as
 * pfa_attn_bwd otherwise. */
int pfa_attn_bwd_ex(const pfa_bf16* q, const pfa_bf16* k, const pfa_bf16* v, const pfa_bf16* dO,
                    const float* lse, const float* delta, pfa_bf16* dq, pfa_bf16* dk, pfa_bf16* dv,
                    float* dq_accum, int B, int H_q, int H_kv, int N, int d, int causal, float scale,
                    unsigned flags, pfa_stream_t stream);

/* The same backward pass for callers that cannot allocate device memory (no
 * counterpart in the paper; this is a deployment convenience). Some callers are
 * not allowed to call cudaMalloc at all: runtimes that reserve all device memory
 * up front in their own pool, real-time loops that cannot take cudaMalloc's
 * implicit device synchronisation, or plugins that are handed only their input
 * and output buffers. This entry point takes exactly the arguments of
 * pfa_attn_bwd except dq_accum: the FP32 dQ accumulation buffer is a fixed
 * library-owned array of 8,388,608 floats (32 MiB) that every GPU loading the
 * library holds until the process exits. It allocates nothing.
 *   - Limit: B * H_q * N * d must not exceed 8,388,608; larger problems return
 *     PFA_ERR_TOO_LARGE before anything is launched (use pfa_attn_bwd instead).
 *   - The first call on a device looks up the array's device address with that
 *     device current; make that first call before any stream capture.
 *   - All calls share the one array per device and it keeps the last call's
 *     contents; each call zeroes it on `stream` first. Calls whose work overlaps
 *     on the GPU (different streams without ordering between them) race on it:
 *     order them on one stream or with events. */
int pfa_attn_bwd_noalloc(const pfa_bf16* q, const pfa_bf16* k, const pfa_bf16* v,
                         const pfa_bf16* dO, const float* lse, const float* delta, pfa_bf16* dq,
                         pfa_bf16* dk, pfa_bf16* dv, int B, int H_q, int H_kv, int N, int d,
                         int causal, float scale, pfa_stream_t stream);

/* Bytes of the dq_accum workspace pfa_attn_bwd needs: B*H_q*N*d*4 (0 on bad sizes). */
size_t pfa_bwd_workspace_bytes(int B, int H_q, int N, int d);

/* Human-readable name of a PFA_* status code (static string, never NULL). */
const char* pfa_status_string(int status);

/* Description of the most recent CUDA runtime error behind a PFA_ERR_LAUNCH
 * returned to the calling thread ("no CUDA error" if there was none). */
const char* pfa_last_error(void);

/* Reads (and, if clear != 0, resets) the device error word of the current device.
 * Returns the PFA_DEVERR_* bits (>= 0) or a negative PFA_ERR_* code. This call
 * synchronises the current device. */
int pfa_device_error(int clear);

/* Where the first bounded wait that gave up (PFA_DEVERR_TIMEOUT) since the last
 * pfa_device_error(1) was: 0 if none, else kernel id in bits 56-59 (1 forward,
 * 2 backward, 3 delta via dP o P, 4 pfa_wait_probe, 5 the query-outer dQ pass), bit 55
 * set for a teardown
 * (drain) wait,
 * bit 54 the awaited phase parity, bits 32-53 the barrier's byte offset in the
 * kernel's shared memory, bits 0-31 blockIdx.x. Negative: a PFA_ERR_* code.
 * Synchronises the current device. */
long long pfa_device_error_site(void);

/* Self-test of the failure path (no counterpart in the paper). Enqueues on
 * `stream` one warp that waits on a shared-memory mbarrier nothing completes; the
 * wait is bounded like every pipeline wait of the library, so after about a
 * second the warp gives up, records its site (kernel id 4, offset 0, parity 0)
 * and sets PFA_DEVERR_TIMEOUT in the device error word. No fault or trap is
 * raised and the device stays usable. Read the result with pfa_device_error and
 * pfa_device_error_site, and clear it with pfa_device_error(1). Returns PFA_OK,
 * PFA_ERR_UNSUPPORTED or PFA_ERR_LAUNCH. */
int pfa_wait_probe(pfa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PFA_H_ */
