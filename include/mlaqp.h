/*
 * mlaqp.h -- C ABI of the GB300 (sm_103a) fused MLA decode query projection.
 *
 * The operation (SparkInfer PR #75 "Add BF16 MLA query projection and
 * assembly", sections What and Contract; vLLM PR #174 "Fuse MXFP8 and BF16
 * MLA query assembly", section What): for every token m < M and head h < H
 *
 *   acc[m,h,n] = sum_{k<128} q_nope[m,h,k] * W_UK_T[h,k,n]   (FP32 accumulate)
 *   out[m,h,n]       = bf16_rne(acc)                        n < 512, BF16 out
 *                    = e4m3_satfinite(bf16_rne(acc)/q_scale)         E4M3 out
 *   out[m,h,512+j]   = q_pe[m,h,j]                          j < 64,  BF16 out
 *                    = e4m3_satfinite(q_pe[m,h,j]/q_scale)           E4M3 out
 *
 * in ONE kernel launch: the 64-wide RoPE part is appended by the projection's
 * epilogue, with no separate concat kernel (vLLM PR #174, section What).
 * The projection is rounded to BF16 before the optional E4M3 conversion, the
 * staged operation boundary (SparkInfer PR #75, section Contract).
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The
 *     library never allocates, frees or synchronises on the run path.
 *   - Supported domain (vLLM PR #174, section What: "capability-gated"
 *     H = 8/11/16 and M = 1..32): num_heads H in {8, 11, 16}, tokens
 *     1 <= M <= 256, nope dim 128 (192, the GLM dim of SparkInfer PR #75,
 *     section What, through mlaqp_run_strided), latent dim 512, rope dim 64,
 *     on an sm_103 (GB300) device.  M <= 32 is the decode domain of the
 *     pages; 33..256 extends it to the multi-token-prediction and
 *     prefill-sized steps that the pages leave to the staged BMM (vLLM PR
 *     #174, sections Safety scope and E2E topology matrix): the decode
 *     (mma.sync) kernel runs in 32-token chunks up to M = 64, and beyond
 *     while its 8*H*ceil(M/32) CTAs fit the device at four per SM (nope dim
 *     128; three for 192): H = 8 to M = 256, H = 11 to 192, H = 16 to 128 on
 *     152 SMs; otherwise a tcgen05
 *     (TMEM-accumulator) kernel takes its place.
 *   - Status codes are the mlaqp_status values; on any non-OK status a
 *     message is available from mlaqp_last_error() on the same thread.
 *
 * Layouts (row-major, element strides in elements, no padding unless said):
 *   q_nope        BF16 [M, H, 128]
 *   q_pe          BF16 [M, H, 64]
 *   weight        BF16 [H, 128, 512]  (MLAQP_WEIGHT_BF16), latent (N) fastest
 *                 E4M3 [H, 128, 512]  (MLAQP_WEIGHT_MXFP8), OCP E4M3FN codes
 *   weight_scale  E8M0 [H, 128, 16]   (MXFP8 only): byte x scales the 32
 *                 latent elements n in [32*j, 32*j+32) of row (h,k) by
 *                 2^(x-127) (pages: sf_axis="n", b_major="n"; block size 32
 *                 along N and the [H,K,N/32] order are this library's
 *                 reading, the pages give no layout)
 *   q_scale       one FP32 value in device memory (E4M3 output only), read
 *                 by the kernel at run time so CUDA-graph replays see
 *                 updates made between replays
 *   out           BF16 or E4M3; element (m,h,j), j < 576, is at
 *                 out[m*out_row_stride + h*576 + j].  Rows >= M and the
 *                 padding between 576*H and out_row_stride are never written.
 */
#ifndef MLAQP_H_
#define MLAQP_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream; NULL is the legacy default stream. */
typedef struct CUstream_st* mlaqp_stream_t;

typedef enum {
  MLAQP_WEIGHT_BF16 = 0,  /* BF16 W_UK_T                                   */
  MLAQP_WEIGHT_MXFP8 = 1  /* E4M3 W_UK_T + one E8M0 scale per 32 latent elts */
} mlaqp_weight_format;

typedef enum {
  MLAQP_OUT_BF16 = 0,     /* BF16 output; q_scale must be NULL             */
  MLAQP_OUT_E4M3 = 1      /* E4M3 output scaled by 1/q_scale; q_scale needed */
} mlaqp_out_dtype;

typedef enum {
  MLAQP_OK = 0,
  MLAQP_ERR_UNSUPPORTED = 1,  /* shape, format or device outside the domain */
  MLAQP_ERR_INVALID_ARG = 2,  /* NULL/misaligned/overlapping pointer, bad
                                 stride, scale given where it must be absent */
  MLAQP_ERR_CUDA = 3          /* a CUDA runtime call failed (message kept)  */
} mlaqp_status;

#define MLAQP_NOPE_DIM 128
#define MLAQP_LATENT_DIM 512
#define MLAQP_ROPE_DIM 64
#define MLAQP_OUT_DIM 576
#define MLAQP_MAX_M 256        /* tokens per call                      */
#define MLAQP_MAX_M_DECODE 32   /* largest M of one decode-kernel chunk */

/*
 * Capability check (SparkInfer PR #75, review of api.py `can_implement`:
 * num_heads, max_m, nope_dim, latent_dim, output dtype, weight format,
 * device).  Returns 1 when a call with these sizes, formats and device is
 * covered, else 0 (and a reason via mlaqp_last_error()).  Launches nothing.
 * device < 0 means the calling thread's current CUDA device.
 */
int mlaqp_can_implement(int num_heads, int max_m, int nope_dim, int latent_dim,
                        int rope_dim, int weight_format, int out_dtype, int device);

/*
 * Prewarm (SparkInfer PR #75, walkthrough: the API prewarms weight and M
 * regimes before the first run; vLLM PR #174, section Layout and topology:
 * prewarm limited to graph-visible M).  Loads the kernel images of every
 * specialisation that a run with M <= max_m would use on `device` (< 0:
 * current), so that later runs -- including runs captured into a CUDA graph
 * -- trigger no module loading.  Idempotent and thread-safe.  Returns
 * MLAQP_OK, MLAQP_ERR_UNSUPPORTED or MLAQP_ERR_CUDA.
 */
int mlaqp_prewarm(int num_heads, int max_m, int weight_format, int out_dtype, int device);

/*
 * Run one layer call (SparkInfer PR #75, walkthrough "project q_nope and
 * append q_pe", "write output tensor").  One kernel launch on `stream`,
 * asynchronous, no host synchronisation, no allocation: capturable into a
 * CUDA graph.  Pointer arguments as in the layout table above.
 *
 *   weight_scale   required for MLAQP_WEIGHT_MXFP8, must be NULL for BF16
 *   q_scale        required for MLAQP_OUT_E4M3, must be NULL for BF16 output
 *                  (vLLM PR #174, section What: "BF16 output omits the unused
 *                  scale argument"; SparkInfer PR #75, section Contract:
 *                  "E4M3 output requires one")
 *   out_row_stride elements between token rows of `out`, >= 576*H, and
 *                  out_row_stride * element size a multiple of 16 bytes
 *   M              0 returns MLAQP_OK without launching; 1..256 supported
 *
 * q_nope, weight, weight_scale and out must be 16-byte aligned, q_pe and
 * q_scale 4-byte aligned; the bytes written to `out` may not overlap any
 * input.  Errors are reported before anything is launched.
 */
int mlaqp_run(const void* q_nope, const void* q_pe, const void* weight,
              const void* weight_scale, void* out, int64_t out_row_stride,
              const float* q_scale, int M, int H, int weight_format, int out_dtype,
              mlaqp_stream_t stream);

/*
 * As mlaqp_run, but launched with programmatic dependent launch: the kernel
 * may start while earlier kernels on `stream` are still running, streams
 * its weights and scales, reads q_scale, prefetches the q_nope / q_pe lines
 * into L2, and only then waits for the previous kernel to finish before it
 * reads q_nope and q_pe or writes `out`.  It also lets the next kernel on
 * the stream start early -- for M <= 32 right at its entry -- so in a chain
 * of such launches more than one earlier kernel can still be running when a
 * kernel starts.  Use it only when `weight`, `weight_scale` and `q_scale`
 * are not written by any kernel that may still be running: not by the
 * preceding programmatic-dependent launches on `stream` back to the last
 * ordinary launch (model weights and per-tensor scales written at load
 * time, or by host copies between graph replays, satisfy this).
 */
int mlaqp_run_pdl(const void* q_nope, const void* q_pe, const void* weight,
                  const void* weight_scale, void* out, int64_t out_row_stride,
                  const float* q_scale, int M, int H, int weight_format, int out_dtype,
                  mlaqp_stream_t stream);

/*
 * General form of mlaqp_run (pdl = 0) / mlaqp_run_pdl (pdl = 1): the same operation
 * with nope dim `nope_dim` (128 or 192) and strided inputs, so that q_nope
 * and q_pe can be views into the upstream per-head [.., nope_dim + 64]
 * projection output, or head-major [H, M, nope_dim] (the layout of the
 * SparkInfer PR #75 BMM, section What), without a copy:
 *   q_nope element (m,h,k) at q_nope[m*q_nope_token_stride + h*q_nope_head_stride + k]
 *   q_pe   element (m,h,j) at q_pe[m*q_pe_token_stride + h*q_pe_head_stride + j]
 * Strides are in elements, >= 0; q_nope strides must be multiples of 8
 * (16-byte rows), q_pe strides multiples of 2.  weight is [H, nope_dim, 512]
 * (BF16 or E4M3) and weight_scale [H, nope_dim, 16]; everything else is as
 * for mlaqp_run.
 *
 * pdl = 2 (opt-in, no counterpart on the pages): as pdl = 1, and where the
 * call runs the tcgen05 kernel it lets the next kernel on the stream launch at
 * its entry rather than after it has allocated tensor memory (about 0.5 us
 * less per layer call in a chain).  The caller promises the tensor-memory
 * contract this needs: no kernel launched after this call on `stream`, while
 * it may still be running, allocates tensor memory (tcgen05.alloc) before
 * its own dependency wait -- otherwise such a kernel could hold the columns
 * this call is waiting for while it waits for this call, and neither would
 * finish.  Every kernel of this library allocates tensor memory only after
 * its dependency wait, so chains of its calls meet the contract.  For the
 * mma.sync kernels, pdl = 2 is pdl = 1.  Other values return MLAQP_ERR_INVALID_ARG.
 */
int mlaqp_run_strided(const void* q_nope, int64_t q_nope_token_stride, int64_t q_nope_head_stride,
                      const void* q_pe, int64_t q_pe_token_stride, int64_t q_pe_head_stride,
                      const void* weight, const void* weight_scale, void* out,
                      int64_t out_row_stride, const float* q_scale, int M, int H, int nope_dim,
                      int weight_format, int out_dtype, int pdl, mlaqp_stream_t stream);

/*
 * Optional L2 warm-up of one layer's weights (vLLM PR #174, section
 * Performance evidence: the per-layer query time inside a decode step,
 * where the kernel before this op produces q_nope / q_pe and usually does
 * not let dependent kernels start early).  Launches one small kernel on
 * `stream` that asks the GPU to fetch `weight` ([H, nope_dim, 512], BF16 or
 * E4M3) and `weight_scale` ([H, nope_dim, 16] E8M0 for MXFP8, else NULL)
 * into L2 and returns without waiting for the data; a following mlaqp_run
 * of the same layer then finds its weights in L2.  Place it before the
 * kernels that produce q_nope / q_pe, ideally on a parallel branch (a forked
 * stream or graph branch), and not so early that other traffic evicts the
 * ~1-2 MB again.  pdl != 0 launches it with programmatic dependent launch:
 * it issues its fetches without waiting for the previous kernel and lets the
 * next one launch at once; it exits only after the previous kernel has
 * finished, so a following kernel's dependency wait still covers everything
 * launched before it.  Same pointer rules as mlaqp_run; no allocation,
 * graph-capturable.
 * Returns MLAQP_OK, MLAQP_ERR_UNSUPPORTED, MLAQP_ERR_INVALID_ARG or
 * MLAQP_ERR_CUDA.
 */
int mlaqp_prefetch_weights(const void* weight, const void* weight_scale, int num_heads, int nope_dim,
                           int weight_format, int pdl, mlaqp_stream_t stream);

/*
 * Launch geometry a run with these arguments (nope dim 128) uses on the
 * current device, for reporting: grid size in CTAs and threads per CTA.
 * Where the choice depends on the device's SM count (9 <= M <= 32, M > 64)
 * it queries the device.  Returns MLAQP_OK, MLAQP_ERR_UNSUPPORTED, or the
 * device query's status (MLAQP_ERR_CUDA without a usable device).
 */
int mlaqp_launch_shape(int M, int H, int weight_format, int out_dtype, int* grid_ctas,
                       int* threads_per_cta);

/*
 * Test hook (no counterpart on the pages): the launch a query call would
 * make on a device with `sm_count` SMs, computed on the host alone (no
 * device access), by the same code the run path uses: arm as in
 * mlaqp_debug_run_arm (MLAQP_ARM_AUTO: the library's choice; the chosen
 * MLAQP_ARM_* value is returned in *arm_out), the token chunk of a CTA-tile
 * launch (*chunk_tokens, 0: one launch over all tokens), where a CTA lets the
 * next kernel launch (*trig: 0 at entry, 1 after the dependency wait -- for
 * the tcgen05 kernel, after its tensor-memory allocation --, 2 once its
 * weight tile is ready), the CTAs-per-SM cap the shared-memory padding
 * imposes (*cta_cap, 0: none; only with pdl != 0), and the grid and block
 * size.  Any output pointer may be NULL.  Returns MLAQP_OK,
 * MLAQP_ERR_INVALID_ARG (bad enum, pdl, arm or sm_count) or
 * MLAQP_ERR_UNSUPPORTED (domain, or a forced arm that does not cover the
 * call).
 */
int mlaqp_debug_plan(int M, int H, int nope_dim, int weight_format, int out_dtype, int pdl, int arm,
                     int sm_count, int* arm_out, int* chunk_tokens, int* trig, int* cta_cap,
                     int* grid_ctas, int* threads_per_cta);

/*
 * Test hook (no counterpart on the pages): as mlaqp_debug_plan, for a V
 * call with contiguous x: *form 0 = the column-tile kernel reading x with
 * plain loads, 1 = the x-multicast kernel, 2 = the tcgen05 cluster kernel;
 * *chunk_tokens = tokens per grid.z chunk; *cluster = CTAs per cluster (1:
 * none).  Returns MLAQP_OK, MLAQP_ERR_INVALID_ARG or MLAQP_ERR_UNSUPPORTED.
 */
int mlaqp_debug_v_plan(int M, int H, int weight_format, int pdl, int sm_count, int* form,
                       int* chunk_tokens, int* trig, int* cta_cap, int* grid_ctas,
                       int* threads_per_cta, int* cluster);

/*
 * Device status word (diagnostic, not for the hot path): every in-kernel
 * wait on a copy-completion barrier is bounded in time; a CTA that gives up
 * sets MLAQP_DEVSTATUS_WAIT_TIMEOUT here and returns without writing its
 * part of `out`.  Reads the OR of all bits set on the current device since
 * the last reset into *status (synchronising with the device); reset != 0
 * clears it.  Returns MLAQP_OK, MLAQP_ERR_INVALID_ARG or MLAQP_ERR_CUDA.
 */
#define MLAQP_DEVSTATUS_WAIT_TIMEOUT 1u
int mlaqp_device_status(unsigned int* status, int reset);

/*
 * Test hook for the bounded waits (no counterpart on the pages): as
 * mlaqp_run, with the wait bound set to wait_limit_ns and the copy barrier
 * told to expect extra_tx_bytes (<= 2^19) more than the copies deliver, so
 * that extra_tx_bytes > 0 makes every CTA's wait run out: the kernel then
 * records MLAQP_DEVSTATUS_WAIT_TIMEOUT, writes nothing and returns.  The
 * copies themselves complete normally.  Not for production use.
 */
int mlaqp_debug_run_bounded_wait(const void* q_nope, const void* q_pe, const void* weight,
                                 const void* weight_scale, void* out, int64_t out_row_stride,
                                 const float* q_scale, int M, int H, int weight_format,
                                 int out_dtype, unsigned long long wait_limit_ns,
                                 unsigned int extra_tx_bytes, mlaqp_stream_t stream);

/*
 * Measurement hook (no counterpart on the pages): as mlaqp_run_strided, but
 * the kernel form is forced instead of chosen by the library, so that the
 * forms can be timed against each other on the same call:
 *   MLAQP_ARM_AUTO      the library's choice (what mlaqp_run uses)
 *   MLAQP_ARM_WARP_MMA  warp-tile kernel, mma.sync tensor-core contraction
 *                       (M <= 32)
 *   MLAQP_ARM_WARP_FMA  warp-tile kernel, FP32 FMA contraction on the CUDA
 *                       cores with a warp-shuffle reduction (M <= 8,
 *                       nope_dim 128)
 *   MLAQP_ARM_CTA_MMA   the CTA-tile mma.sync kernel (64 latent columns per
 *                       CTA, q_nope staged in shared memory; any M, in
 *                       32-token chunks above 32)
 *   MLAQP_ARM_TCGEN05   the tcgen05 kernel (TMEM accumulator; any M)
 * A form that does not cover the call returns MLAQP_ERR_UNSUPPORTED; every
 * form computes the same result within the projection tolerance, with
 * identical q_pe columns and E4M3 codes.  Not for production use.
 */
#define MLAQP_ARM_AUTO 0
#define MLAQP_ARM_WARP_MMA 1
#define MLAQP_ARM_WARP_FMA 2
#define MLAQP_ARM_CTA_MMA 3
#define MLAQP_ARM_TCGEN05 4
int mlaqp_debug_run_arm(const void* q_nope, int64_t q_nope_token_stride, int64_t q_nope_head_stride,
                        const void* q_pe, int64_t q_pe_token_stride, int64_t q_pe_head_stride,
                        const void* weight, const void* weight_scale, void* out,
                        int64_t out_row_stride, const float* q_scale, int M, int H, int nope_dim,
                        int weight_format, int out_dtype, int pdl, int arm, mlaqp_stream_t stream);

/*
 * Measurement hook (no counterpart on the pages): overrides, process-wide,
 * the launch policy of the mma.sync kernels: trig = 0 lets the
 * next kernel on the stream launch at kernel entry, 1 after the dependency
 * wait; cta_cap = 1..8 pads shared memory so that at most that many CTAs
 * share an SM (0: no padding).  trig = -1 restores the library's policy.
 * Affects launches made after the call (and graphs captured after it).  Not
 * for production use.  Returns MLAQP_OK or MLAQP_ERR_INVALID_ARG.
 */
int mlaqp_debug_set_policy(int trig, int cta_cap);

/*
 * Diagnostic (no counterpart on the pages): launches a kernel of `ctas` x
 * `threads` that does nothing but the programmatic-launch protocol (trigger
 * the next kernel, wait for the previous one), with (pdl != 0) or without
 * programmatic dependent launch.  A CUDA graph of such launches measures the
 * per-launch floor of a dependent chain, the bound on any one-launch-per-
 * layer operation.  Returns MLAQP_OK, MLAQP_ERR_INVALID_ARG or
 * MLAQP_ERR_CUDA.
 */
int mlaqp_debug_launch_null(int ctas, int threads, int pdl, mlaqp_stream_t stream);

/*
 * V up-projection, the step after attention over the latent cache (the
 * pages name it only as the downstream V up-projection, vLLM PR #174,
 * section Safety scope; the weight formats follow the query side, section
 * What).  For every token m < M and head h < H:
 *
 *   out[m,h,d] = bf16_rne( sum_{c<512} x[m,h,c] * W_UV[h,c,d] )   d < 128, FP32 accumulation
 *
 * in one kernel launch on `stream`, asynchronous, no allocation, no host
 * synchronisation.
 *   x              BF16 attention output in the latent space; element (m,h,c)
 *                  at x[m*x_token_stride + h*x_head_stride + c], c < 512;
 *                  strides in elements, >= 0, multiples of 8; 16-byte aligned
 *   weight         W_UV [H, 512, 128], output (d) axis fastest: BF16
 *                  (MLAQP_WEIGHT_BF16) or OCP E4M3FN codes (MLAQP_WEIGHT_MXFP8);
 *                  16-byte aligned
 *   weight_scale   E8M0 [H, 512, 4] for MXFP8 (byte j of row (h,c) scales
 *                  d in [32j, 32j+32) by 2^(x-127)), NULL for BF16
 *   out            BF16; element (m,h,d) at out[m*out_row_stride + h*128 + d];
 *                  out_row_stride >= 128*H and a multiple of 8 elements;
 *                  16-byte aligned; rows >= M and the padding are not written;
 *                  may not overlap an input
 *   M              0 returns MLAQP_OK without launching; 1..256 supported
 *                  (an mma.sync kernel over 32-token chunks up to M = 64,
 *                  and beyond while its 8*H*ceil(M/32) CTAs stay within 2.6
 *                  per SM (H = 8 to M = 192, H = 11 to 128, H = 16 to 96 on
 *                  152 SMs; at H = 8 and 9 <= M <= 32 two chunks of 8 or, for
 *                  MXFP8, 16 tokens); from M = 9 (BF16) or 12 (MXFP8)
 *                  launched in clusters of the 8 CTAs of a (head, chunk),
 *                  which share x through one TMA multicast per CTA where
 *                  the strides form a tensor map.  Otherwise a tcgen05
 *                  kernel launched in clusters of 4 CTAs, whose tensor
 *                  memory is taken after the dependency wait and freed
 *                  before it returns)
 *   H              8, 11 or 16
 *   pdl            1: programmatic dependent launch, as mlaqp_run_pdl (the
 *                  weights and scales must not be written by any kernel that
 *                  may still be running, see mlaqp_run_pdl); 2: the same,
 *                  and where the call runs the tcgen05 kernel the next kernel
 *                  may launch at this one's entry, under the tensor-memory
 *                  contract of
 *                  mlaqp_run_strided's pdl = 2; 0: ordinary launch; other
 *                  values return MLAQP_ERR_INVALID_ARG
 * Status codes as for mlaqp_run.
 */
#define MLAQP_V_HEAD_DIM 128
int mlaqp_v_up_run(const void* x, int64_t x_token_stride, int64_t x_head_stride, const void* weight,
                   const void* weight_scale, void* out, int64_t out_row_stride, int M, int H,
                   int weight_format, int pdl, mlaqp_stream_t stream);

/* 1 if mlaqp_v_up_run covers (num_heads, max_m, weight_format) on `device`
 * (< 0: current), else 0 with a reason in mlaqp_last_error().  Launches
 * nothing. */
int mlaqp_v_up_can_implement(int num_heads, int max_m, int weight_format, int device);

/* Loads every V up-projection kernel a call with M <= max_m can use, as
 * mlaqp_prewarm does for the query projection.  Call before graph capture. */
int mlaqp_v_up_prewarm(int num_heads, int max_m, int weight_format, int device);

/* Test hook for the V up-projection's bounded waits, as
 * mlaqp_debug_run_bounded_wait (no counterpart on the pages). */
int mlaqp_debug_v_up_bounded_wait(const void* x, int64_t x_token_stride, int64_t x_head_stride,
                                  const void* weight, const void* weight_scale, void* out,
                                  int64_t out_row_stride, int M, int H, int weight_format,
                                  unsigned long long wait_limit_ns, unsigned int extra_tx_bytes,
                                  mlaqp_stream_t stream);

/* Message of the last non-OK status returned on this thread ("" if none). */
const char* mlaqp_last_error(void);

/* Library version: major*10000 + minor*100 + patch. */
int mlaqp_version(void);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* MLAQP_H_ */
