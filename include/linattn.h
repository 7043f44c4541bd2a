/*
 * linattn.h -- C ABI of the GB300 (sm_103a) causal Taylor linear-attention
 * library (liblinattn.so).
 *
 * The operation (BASED reading notes, "Simple linear attention language
 * models balance the recall-throughput tradeoff", sec. 2.2 Eqs. (1)-(3)):
 *
 *   s_i = s_{i-1} + phi(k_i) v_i^T      z_i = z_{i-1} + phi(k_i)
 *   y_i = phi(q_i)^T s_i / (phi(q_i)^T z_i + eps)
 *
 * with the second-order Taylor feature map of sec. 2.3 (d' = 16, D = 273):
 *
 *   phi(x) = [1, xbar, vec(xbar xbar^T) / sqrt(2)],   xbar = x / d'^(1/4) = x / 2
 *   phi(q)^T phi(k) = 1 + q.k/4 + (q.k)^2/32
 *
 * Feature order in every state buffer: f = 0 constant, f = 1 + a linear,
 * f = 17 + 16 a + b quadratic (a, b in 0..15).
 *
 * Common conventions for every entry point:
 *  - Every data pointer is a DEVICE pointer to a dense row-major array
 *    (la_prefill_host: activations and states in host memory, see there);
 *    the caller owns and allocates every buffer.  The library allocates no
 *    memory and keeps no state between calls (apart from the device status
 *    word read by la_check_device_status).
 *  - Activations q, k, v, k_e, v_e and the output y have dtype `dtype`
 *    (LA_DTYPE_BF16 or LA_DTYPE_F32).  States s, z are always fp32.
 *    Layouts: q, k [B][H][N][d_feat]; v, y [B][H][N][64]; k_e [B][H][M][16];
 *    v_e [B][H][M][64]; s [B][H][D][64]; z [B][H][D] (D = 273 at d_feat = 16).
 *  - d_v = 64.  d_feat = 16 everywhere; la_prefill and la_decode_step also take
 *    d_feat = 8, 24, 32 (D = 1 + d_feat + d_feat^2 rows in every state buffer,
 *    general CUDA-core path).  Anything else is LA_ERR_UNSUPPORTED.
 *  - Every pointer must be 16-byte aligned (LA_ERR_MISALIGNED else).
 *  - s0 / z0 may be NULL, meaning a zero initial state (both or neither).
 *    s_out / z_out may be NULL, meaning "do not write the final state".
 *  - Input and output buffers must not overlap, except that la_decode_step
 *    accepts s_out == s_in and z_out == z_in exactly (update in place).
 *  - Work is enqueued on `stream` (NULL = legacy default stream) and runs
 *    asynchronously.  Argument errors are detected on the host and returned
 *    before anything is launched; a launch failure returns LA_ERR_CUDA.
 *  - No exception, abort or process exit ever crosses this boundary.
 *  - eps is added to the denominator; the pages say an epsilon is added
 *    without giving its value, and 0 is the default used by every test.
 */
#ifndef LINATTN_H_
#define LINATTN_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define LA_API __attribute__((visibility("default")))
#else
#define LA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as the CUDA runtime's cudaStream_t (a pointer to an opaque
 * struct), declared here so this header needs no CUDA include. */
typedef struct CUstream_st *la_stream_t;

typedef enum {
    LA_OK = 0,
    LA_ERR_INVALID_ARG = 1,   /* bad shape, NULL required pointer, M > N, overlap */
    LA_ERR_UNSUPPORTED = 2,   /* d_feat != 16, d_v != 64, unknown dtype, no sm_103 device */
    LA_ERR_MISALIGNED = 3,    /* a pointer is not 16-byte aligned */
    LA_ERR_CUDA = 4,          /* a CUDA runtime call or kernel launch failed */
    LA_ERR_TIMEOUT = 5,       /* a bounded device-side wait gave up (see la_check_device_status) */
    LA_ERR_SCRATCH_TOO_SMALL = 6  /* la_prefix_prefill_noalloc: the problem needs more scratch than
                                     the library's fixed buffer holds (use la_prefix_prefill) */
} la_status;

typedef enum {
    LA_DTYPE_F32 = 0,   /* fp32 activations: CUDA-core fp32 kernels */
    LA_DTYPE_BF16 = 1   /* bf16 activations: tensor-core kernels, fp32 accumulate */
} la_dtype;

#define LA_D_FEAT 16
#define LA_D_V 64
#define LA_D_PHI 273   /* 1 + 16 + 16*16 */

/*
 * la_prefill -- causal prefill from an optional initial state.
 *
 * Computes y_i for i = 1..N of every (b, h) with the recurrence above,
 * starting from s0/z0 (state passing: "Understanding and Improving Length
 * Generalization in Recurrent Models" reading notes, sec. 2.5 Eq. (4) with
 * the identity transition, so the initial state just adds to the sums), and
 * writes the final state s_N = s0 + sum_i phi(k_i) v_i^T, z_N likewise.
 *
 *   q, k   in   [B][H][N][16] dtype
 *   v      in   [B][H][N][64] dtype
 *   s0     in   [B][H][273][64] fp32 or NULL;  z0 in [B][H][273] fp32 or NULL
 *   y      out  [B][H][N][64] dtype (bf16: rounded to nearest even)
 *   s_out  out  [B][H][273][64] fp32 or NULL;  z_out out [B][H][273] fp32 or NULL
 *
 * B, H >= 1, N >= 0 (N = 0 only copies s0/z0, or zeros, to s_out/z_out).
 */
LA_API la_status la_prefill(const void *q, const void *k, const void *v,
                     const float *s0, const float *z0,
                     void *y, float *s_out, float *z_out,
                     int64_t B, int64_t H, int64_t N, int d_feat, int d_v,
                     la_dtype dtype, float eps, la_stream_t stream);

/*
 * la_prefill_ws -- la_prefill with a caller workspace that lets the bf16
 * tensor-core path balance its last wave of heads.
 *
 * The kernel runs one CTA per (b, h) on each SM, so B*H heads take
 * ceil(B*H / SMs) waves and the last wave leaves SMs idle.  With a workspace,
 * the heads of the last wave are each split into two pieces along the
 * sequence: the first piece runs on an otherwise idle SM early and hands its
 * state to the second through the workspace (the blockwise state carry of the
 * BASED reading notes, sec. 2.5, across two CTAs).  The results are those of
 * la_prefill up to fp32 rounding order in the handed-over state; they are
 * reproducible on a given device (the split depends on its SM count).
 *
 * With bf16 activations and d_feat = 24 or 32, the workspace instead holds
 * the buffers of a chunked form whose contractions run on the tensor cores
 * (the same blockwise form, BASED notes sec. 2.5, with the symmetric compact
 * feature map of sec. 2.3 for that d': 325 or 561 features; the chunk states,
 * the read-out and the intra-chunk products are cuBLASLt batched GEMMs with
 * bf16 operands and fp32 accumulation).  Its results equal la_prefill's up to
 * bf16 rounding (the states before each chunk are rounded to bf16 for the
 * read-out); the final state's antisymmetric part is s0's, passed through.
 * That workspace is large: about 3.3 KB (d' = 24) or 5.1 KB (d' = 32) per
 * (b, h) token of ceil(N / 128) * 128 tokens, plus 32 MB.
 *
 *   workspace: DEVICE buffer of at least la_prefill_workspace_size(B, H, N,
 *   d_feat, dtype) bytes, 256-byte aligned, owned by the caller, not read
 *   before written.  It must not be used by two calls whose work overlaps on
 *   the GPU.  NULL, or too small, runs exactly la_prefill.
 * All other arguments, layouts and errors are those of la_prefill (padding and
 * decay have no workspace form at d_feat != 16).  la_prefill_workspace_size
 * returns 0 where the workspace has no use (fp32 activations; N = 0 at
 * d_feat 24, 32).
 */
LA_API size_t la_prefill_workspace_size(int64_t B, int64_t H, int64_t N, int d_feat, la_dtype dtype);
/* The split la_prefill_ws (and the prefix call) make on the current device for
 * these sizes: *split_heads heads (the last ones) run as the chunks [0,
 * *split_chunk) and [*split_chunk, ceil(N/128)); 0 and 0 when none. */
LA_API la_status la_prefill_split_info(int64_t B, int64_t H, int64_t N, int *split_heads,
                                       int *split_chunk);
LA_API la_status la_prefill_ws(const void *q, const void *k, const void *v,
                               const float *s0, const float *z0,
                               void *y, float *s_out, float *z_out,
                               void *workspace, size_t workspace_bytes,
                               int64_t B, int64_t H, int64_t N, int d_feat, int d_v,
                               la_dtype dtype, float eps, la_stream_t stream);

/*
 * la_prefill_host -- la_prefill for activations and states that live in host
 * memory: the same computation, with the host <-> device copies inside the
 * call and overlapped with the kernels.
 *
 * q, k, v, s0, z0, y, s_out, z_out have la_prefill's shapes, dtypes and
 * NULL rules, but may be any memory the CUDA runtime can address (copies use
 * cudaMemcpyDefault).  For the copies to overlap they must be page-locked
 * (cudaHostAlloc / cudaHostRegister); pageable memory gives correct results
 * without the overlap.  No alignment is required of them.
 *
 * workspace: DEVICE buffer of at least la_prefill_host_workspace_size(B, H,
 * N, d_feat, dtype) bytes, 256-byte aligned, owned by the caller; it holds the
 * device copies of the slices in flight.  The (b, h) rows are processed in up
 * to 8 slices, up to 3 at a time, each on a stream created for the call (with
 * events ordering it after the work already on `stream` and `stream` after
 * it); streams and events are released when their work completes.
 *
 * The call returns once the work is enqueued: the host outputs are valid
 * after `stream` has reached this point (cudaStreamSynchronize).  The inputs
 * must stay unchanged, and the outputs untouched, until then.  Not for use
 * while `stream` is being captured into a CUDA graph (the call creates and
 * destroys streams); la_prefill on device buffers is the capturable form.
 * d_feat 8/16/24/32 and both dtypes as la_prefill; no padding or decay.
 * Errors as la_prefill; a workspace that is too small is LA_ERR_INVALID_ARG.
 */
LA_API size_t la_prefill_host_workspace_size(int64_t B, int64_t H, int64_t N, int d_feat,
                                             la_dtype dtype);
LA_API la_status la_prefill_host(const void *q, const void *k, const void *v,
                          const float *s0, const float *z0,
                          void *y, float *s_out, float *z_out,
                          void *workspace, size_t workspace_bytes,
                          int64_t B, int64_t H, int64_t N, int d_feat, int d_v,
                          la_dtype dtype, float eps, la_stream_t stream);

/*
 * la_prefix_workspace_size -- bytes of device scratch la_prefix_prefill
 * needs for these sizes (0 when M == 0).  The result depends only on
 * (B, H, M).
 */
LA_API size_t la_prefix_workspace_size(int64_t B, int64_t H, int64_t M);

/*
 * la_prefix_prefill -- JRT-RNN prefix linear attention ("Just read twice"
 * reading notes, sec. 2.6, Eqs. (3)-(4)).
 *
 * A non-causal prefix state is built from a second K/V set over its M
 * positions,
 *   s_E = sum_{j<=M} phi(k_e_j) v_e_j^T,   z_E = sum_{j<=M} phi(k_e_j),
 * and every causal position reads it in addition to the causal state:
 *   y_i = phi(q_i)(s0 + s_E + s_{D,i}) / (phi(q_i)(z0 + z_E + z_{D,i}) + eps).
 * The final state is the merge s0 + s_E + s_{D,N} (Eq. (4)).
 *
 *   k_e in [B][H][M][16] dtype, v_e in [B][H][M][64] dtype (ignored if M == 0)
 *   0 <= M <= N, else LA_ERR_INVALID_ARG.
 *   workspace: device buffer of la_prefix_workspace_size(B, H, M) bytes,
 *   256-byte aligned, owned by the caller, not read before it is written; it
 *   may be reused once the call's work on `stream` is done.  That size
 *   includes a region through which the prefill hands state between the two
 *   pieces of a split head (see la_prefill_ws); a smaller workspace that
 *   still holds the prefix partial states (B*H*nseg * 70,980 bytes, rounded
 *   up; see la_prefix_prefill_noalloc) runs without split heads.
 * Other arguments as for la_prefill.
 */
LA_API la_status la_prefix_prefill(const void *q, const void *k, const void *v,
                            const void *k_e, const void *v_e, int64_t M,
                            const float *s0, const float *z0,
                            void *y, float *s_out, float *z_out,
                            void *workspace, size_t workspace_bytes,
                            int64_t B, int64_t H, int64_t N, int d_feat, int d_v,
                            la_dtype dtype, float eps, la_stream_t stream);

/*
 * la_prefill_padded, la_prefix_prefill_padded -- the same two calls for a
 * batch of left-padded sequences ("Just read twice" reading notes, sec. 2.7:
 * prompts shorter than M are left-padded to M and the padding is masked in
 * the prefix linear attention; sec. 4.7: padding must stay out of the
 * linear-attention state).
 *
 *   left_pad  in  [B] int32, DEVICE pointer, 4-byte aligned, required:
 *             row b's first p_b = left_pad[b] positions are padding,
 *             0 <= p_b <= N.
 *
 * For row b, prefix positions j < min(p_b, M) and causal positions i < p_b
 * contribute nothing to s_E, the causal sums or the final state, and
 * y_i = 0 for i < p_b.  Every other output equals that of the unpadded call
 * on the valid tokens alone (q, k, v from position p_b on, k_e, v_e from
 * min(p_b, M) on).  p_b = 0 for every row gives the unpadded result.
 *
 * The counts live in device memory and are checked there: a count outside
 * [0, N] is clamped to that range and recorded in the device status word, so
 * the next la_check_device_status returns LA_ERR_INVALID_ARG.  A NULL
 * left_pad is LA_ERR_INVALID_ARG; left_pad must not overlap an output.
 * All other arguments, layouts and errors are those of la_prefill /
 * la_prefix_prefill.
 */
LA_API la_status la_prefill_padded(const void *q, const void *k, const void *v,
                                   const float *s0, const float *z0, const int32_t *left_pad,
                                   void *y, float *s_out, float *z_out,
                                   int64_t B, int64_t H, int64_t N, int d_feat, int d_v,
                                   la_dtype dtype, float eps, la_stream_t stream);

LA_API la_status la_prefix_prefill_padded(const void *q, const void *k, const void *v,
                                          const void *k_e, const void *v_e, int64_t M,
                                          const float *s0, const float *z0, const int32_t *left_pad,
                                          void *y, float *s_out, float *z_out,
                                          void *workspace, size_t workspace_bytes,
                                          int64_t B, int64_t H, int64_t N, int d_feat, int d_v,
                                          la_dtype dtype, float eps, la_stream_t stream);

/*
 * la_prefill_decay, la_decode_step_decay -- the causal prefill and the decode
 * step with a fixed per-head decay gamma_h ("Understanding and Improving
 * Length Generalization in Recurrent Models" reading notes, sec. 2.1 Eq. (1)
 * with A_t = gamma_h I; the BASED reading notes, sec. 2.4, mention fixed
 * per-head decay rates in some runs):
 *
 *   s_i = gamma_h s_(i-1) + phi(k_i) v_i^T,   z_i = gamma_h z_(i-1) + phi(k_i),
 *   y_i = phi(q_i)^T s_i / (phi(q_i)^T z_i + eps),   s_(-1) = s0, z_(-1) = z0
 *
 * so the initial state reaches position i (0-based) as gamma^(i+1) s0 (sec.
 * 2.5, Eq. (4)).  gamma = 1 is the undecayed recurrence.
 *
 *   gamma  in  [H] fp32, DEVICE pointer, 4-byte aligned, required;
 *              0 <= gamma_h <= 1.
 *
 * A rate outside [0, 1] (or NaN) is clamped on the device (NaN to 0) and
 * recorded in the device status word: the next la_check_device_status
 * returns LA_ERR_INVALID_ARG.  gamma must not overlap an output.  All other
 * arguments, layouts and errors are those of la_prefill / la_decode_step.
 * There is no decayed prefix call: the pages do not say how the non-causal
 * prefix state would decay.
 */
LA_API la_status la_prefill_decay(const void *q, const void *k, const void *v,
                                  const float *s0, const float *z0, const float *gamma,
                                  void *y, float *s_out, float *z_out,
                                  int64_t B, int64_t H, int64_t N, int d_feat, int d_v,
                                  la_dtype dtype, float eps, la_stream_t stream);

/* la_prefill_decay with the workspace of la_prefill_ws (split heads of the last
 * wave; la_prefill_workspace_size gives its size).  NULL or too small a
 * workspace runs exactly la_prefill_decay. */
LA_API la_status la_prefill_decay_ws(const void *q, const void *k, const void *v,
                                     const float *s0, const float *z0, const float *gamma,
                                     void *y, float *s_out, float *z_out,
                                     void *workspace, size_t workspace_bytes,
                                     int64_t B, int64_t H, int64_t N, int d_feat, int d_v,
                                     la_dtype dtype, float eps, la_stream_t stream);

LA_API la_status la_decode_step_decay(const void *q, const void *k, const void *v,
                                      const float *gamma, const float *s_in, const float *z_in,
                                      float *s_out, float *z_out, void *y,
                                      int64_t B, int64_t H, int d_feat, int d_v,
                                      la_dtype dtype, float eps, la_stream_t stream);

/*
 * la_decode_step -- one recurrent decode step per (b, h) (BASED reading
 * notes, sec. 2.2 Eq. (2) for one token; sec. 2.5 notes that decoding still
 * reads and writes the whole persistent state).  The state is updated first
 * and then read, so y uses s + phi(k) v^T.
 *
 *   q, k   in   [B][H][16] dtype;  v in [B][H][64] dtype
 *   s_in   in   [B][H][273][64] fp32;  z_in in [B][H][273] fp32 (required)
 *   s_out  out  [B][H][273][64] fp32;  z_out out [B][H][273] fp32 (required;
 *               may be exactly s_in / z_in for an in-place update)
 *   y      out  [B][H][64] dtype
 */
LA_API la_status la_decode_step(const void *q, const void *k, const void *v,
                         const float *s_in, const float *z_in,
                         float *s_out, float *z_out, void *y,
                         int64_t B, int64_t H, int d_feat, int d_v,
                         la_dtype dtype, float eps, la_stream_t stream);

/*
 * Compact state layout (d_feat = 16 only).
 *
 * The BASED reading notes (sec. 2.3) observe that vec(xbar xbar^T) holds each
 * product xbar_a xbar_b (a != b) twice, so the same kernel
 *   phi(q)^T phi(k) = 1 + q.k/4 + (q.k)^2/32
 * is reached with 1 + d' + d'(d'+1)/2 = 153 features: the squares scaled by
 * 1/sqrt(2) and each cross term once, unscaled:
 *
 *   phi_c(x) = [1, xbar_a (a = 0..15), xbar_a^2 / sqrt(2) (a = b), xbar_a xbar_b (a < b)]
 *
 * Sec. 2.5 notes that decoding reads and writes the whole state every step;
 * the compact state is 153 rows instead of 273 (1.78x fewer bytes).
 *
 *   s_c [B][H][153][64] fp32,  z_c [B][H][153] fp32
 *   row 0: constant; row 1 + a: linear xbar_a;
 *   row 17 + c(a, b), a <= b: quadratic, c(a, b) = 16 a - a (a - 1) / 2 + (b - a)
 *   (row-major over the upper triangle: (0,0) is row 17, (0,15) row 32,
 *   (1,1) row 33, (15,15) row 152).
 *
 * Relation to the 273-row state s: s_c[0] = s[0], s_c[1 + a] = s[1 + a],
 *   s_c[17 + c(a, a)] = s[17 + 17 a],
 *   s_c[17 + c(a, b)] = (s[17 + 16 a + b] + s[17 + 16 b + a]) / sqrt(2)  (a < b),
 * and the same for z.  Only the symmetric part of the 273-row quadratic
 * block survives: the antisymmetric part (s[ab] - s[ba]) / 2 is DROPPED by
 * the conversion.  It is zero in every state the recurrence builds (phi(k)
 * is symmetric in (a, b)) and no output ever reads it (phi(q) is symmetric
 * too), so y and every later compact state are unaffected; only a 273-row
 * state that was set by hand with an antisymmetric part does not come back
 * from a round trip.  From compact to 273 rows, the cross term is split
 * evenly: s[ab] = s[ba] = s_c[17 + c(a, b)] / sqrt(2).
 *
 * All compact entry points take d_feat = 16 and d_v = 64 only
 * (LA_ERR_UNSUPPORTED else); pointers, alignment (16 bytes), overlap and
 * stream rules are the common ones above.
 */
#define LA_D_COMPACT 153   /* 1 + 16 + 16*17/2 */

/*
 * la_state_to_compact / la_state_from_compact -- convert B*H states between
 * the 273-row and the compact layout (formulas above).
 *   s  [B][H][273][64], z  [B][H][273] fp32 (DEVICE)
 *   s_c [B][H][153][64], z_c [B][H][153] fp32 (DEVICE)
 * Every pointer is required; input and output must not overlap.
 */
LA_API la_status la_state_to_compact(const float *s, const float *z, float *s_c, float *z_c,
                                     int64_t B, int64_t H, int d_feat, int d_v,
                                     la_stream_t stream);
LA_API la_status la_state_from_compact(const float *s_c, const float *z_c, float *s, float *z,
                                       int64_t B, int64_t H, int d_feat, int d_v,
                                       la_stream_t stream);

/*
 * la_prefill_compact -- la_prefill with the initial and final states in the
 * compact layout: s0_c / z0_c [B][H][153][64] / [B][H][153] fp32 or NULL (both
 * or neither; NULL = zero state), s_out_c / z_out_c likewise or NULL.  y is
 * the same as la_prefill's on the unfolded state (the dropped antisymmetric
 * part is invisible to it).  dtype LA_DTYPE_BF16 only (the tensor-core path,
 * whose internal state is already this 153-feature form); LA_DTYPE_F32 is
 * LA_ERR_UNSUPPORTED (use la_prefill and la_state_to_compact).  Other
 * arguments and errors as la_prefill.
 */
LA_API la_status la_prefill_compact(const void *q, const void *k, const void *v,
                                    const float *s0_c, const float *z0_c,
                                    void *y, float *s_out_c, float *z_out_c,
                                    int64_t B, int64_t H, int64_t N, int d_feat, int d_v,
                                    la_dtype dtype, float eps, la_stream_t stream);

/*
 * la_decode_step_compact -- la_decode_step on a compact state: with
 * phi_c as above, s_c += phi_c(k) v^T, z_c += phi_c(k), then
 * y = phi_c(q)^T s_c / (phi_c(q)^T z_c + eps).
 *   q, k [B][H][16], v [B][H][64] dtype (bf16 or fp32)
 *   s_in_c, z_in_c, s_out_c, z_out_c: compact layout, all required;
 *   s_out_c == s_in_c and z_out_c == z_in_c exactly is the in-place update.
 *   y [B][H][64] dtype.
 * Errors as la_decode_step.
 */
LA_API la_status la_decode_step_compact(const void *q, const void *k, const void *v,
                                        const float *s_in_c, const float *z_in_c,
                                        float *s_out_c, float *z_out_c, void *y,
                                        int64_t B, int64_t H, int d_feat, int d_v,
                                        la_dtype dtype, float eps, la_stream_t stream);

/*
 * la_prefix_prefill_noalloc -- the same computation as la_prefix_prefill, for
 * callers that cannot allocate device memory when they call (for example a
 * serving loop that must not trigger the device synchronisation an
 * allocation implies, or a plug-in whose host process owns all device memory
 * through its own allocator).  There is no counterpart on the pages; it
 * exists only for such callers.
 *
 * Instead of a caller-provided workspace it uses one scratch buffer of
 * la_noalloc_scratch_bytes() bytes (32 MiB) that the library reserves in
 * device memory on every device where it is loaded, until the process exits.
 *   - No memory is allocated by the call (no cudaMalloc, no allocating
 *     library routine).  The caller still passes all inputs and outputs.
 *   - The first call on a device looks up the buffer's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before capturing the stream into a CUDA graph.
 *   - Problems with la_prefix_workspace_size(B, H, M) larger than the buffer
 *     return LA_ERR_SCRATCH_TOO_SMALL before any work is queued.  The call
 *     needs B*H*nseg partial states of 70,980 bytes, with nseg =
 *     min(16, ceil(256 / (B*H)), ceil(M / 128)) prefix segments (fewer once
 *     their length is rounded up to 128 tokens), so B*H*nseg <= 472 fits.
 *     When the buffer also holds la_prefix_workspace_size(B, H, M) bytes, the
 *     prefill splits its last wave of heads as la_prefill_ws does.
 *   - Every call on a device shares the buffer, and the buffer keeps the last
 *     call's contents.  Nothing in it needs to start at zero (each call
 *     writes every part it reads).  Calls whose work overlaps on the GPU (two
 *     streams, or two threads) race on the buffer and give wrong results:
 *     serialise them.
 * All other arguments, layouts and errors are those of la_prefix_prefill.
 */
LA_API la_status la_prefix_prefill_noalloc(const void *q, const void *k, const void *v,
                                           const void *k_e, const void *v_e, int64_t M,
                                           const float *s0, const float *z0,
                                           void *y, float *s_out, float *z_out,
                                           int64_t B, int64_t H, int64_t N, int d_feat, int d_v,
                                           la_dtype dtype, float eps, la_stream_t stream);

/* Size in bytes of the fixed scratch buffer used by la_prefix_prefill_noalloc. */
LA_API size_t la_noalloc_scratch_bytes(void);

/* Static English description of a status code (never NULL). */
LA_API const char *la_status_string(la_status status);

/*
 * la_check_device_status -- synchronizes `stream`, then reads and clears the
 * library's device status word on the current device.  Returns LA_ERR_TIMEOUT
 * if any kernel since the last check gave up a bounded wait (its outputs are
 * then undefined), else LA_ERR_INVALID_ARG if a padded call met a padding
 * count outside [0, N] or a decayed call a rate outside [0, 1] (it was
 * clamped), LA_ERR_CUDA if the synchronization failed, LA_OK else.
 */
LA_API la_status la_check_device_status(la_stream_t stream);

/*
 * la_debug_timeout_probe -- test aid for the failure path: enqueues on
 * `stream` a one-thread kernel that waits, with the library's bounded wait,
 * on a barrier that nothing completes.  After about one second the wait gives
 * up, records a timeout in the device status word and the kernel returns (no
 * trap, no fault; the context stays usable).  The next la_check_device_status
 * returns LA_ERR_TIMEOUT.  Returns LA_ERR_CUDA if the launch failed.
 */
LA_API la_status la_debug_timeout_probe(la_stream_t stream);

/* Library version as major*10000 + minor*100 + patch. */
LA_API int la_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LINATTN_H_ */
