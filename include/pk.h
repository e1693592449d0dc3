/*
 * pk.h -- packed-sequence RoPE attention on one GB300 (sm_103a): the forward pass (pk_attend
 * and its typed forms, pk_attend_noalloc, pk_attend_mixed), its backward pass
 * (pk_attend_backward), the tile schedule (pk_schedule) and the standalone rotation (pk_rope).
 *
 * The operation (hanzo-kernel 0.2.42 packed.rs, module doc and fn attend / fn attend_ref):
 * attention over packed variable-length sequences straight from a packed QKV projection,
 * with the rotary embedding applied to q and k inside the kernel and each query reading
 * only its own sequence's keys, optionally within a symmetric window.
 *
 *   qkv  [T, 3*H*64]  row t holds token t's q (columns h*64 .. h*64+63 for head h), then
 *                     its k (columns H*64 + h*64 ..), then its v (columns 2*H*64 + h*64 ..).
 *   cos, sin [P, 32]  rotary tables indexed by position within a sequence, same element
 *                     type as qkv; P must be at least the longest sequence (not checked:
 *                     P is not an argument).
 *   cu   [S+1]        uint32 first token of each sequence: cu[0] = 0, non-decreasing,
 *                     cu[S] = T. Empty sequences are allowed.
 *   out  [T, H*64]    out[t, h*64 + d], same element type as qkv.
 *   lse  [H, T]       float32, natural-log log-sum-exp of each row's scaled scores.
 *
 * For token t = cu[s] + i of sequence s (length L = cu[s+1] - cu[s]) and head h:
 *   q' = rot(q_t, i) * scale,  k'_j = rot(k_{cu[s]+j}, j)  with the half-split rotation
 *        rot(x, p)[u] = x[u] cos[p,u] - x[u+32] sin[p,u],
 *        rot(x, p)[u+32] = x[u] sin[p,u] + x[u+32] cos[p,u]       (u < 32)
 *   score_j = q' . k'_j for keys j < L with window == 0 or |i - j| <= window
 *   lse = m + ln(sum_j exp(score_j - m)), out = sum_j exp(score_j - lse) v_{cu[s]+j}.
 * `window` = 0 lets every key of the sequence through (the pages' "0: every key").
 *
 * Kernels and precision (enum pk_kernel; pk_forward_kernel says which one a call runs):
 *   - 1 <= window <= 16, any element type: PK_KERNEL_BAND, CUDA cores, every product and sum
 *     in fp32 from the stored values (a row sees at most 33 keys: the work is moving qkv).
 *   - otherwise fp32 inputs: PK_KERNEL_F32, CUDA cores, fp32; or (PK_ATTN=split, or picked by
 *     pk_attend_tuned) PK_KERNEL_SPLIT: q and k rotated in fp32, then every value of q', k', v
 *     and of the probabilities taken as a pair of bf16 values hi + lo (16 significant bits)
 *     and each product as three bf16 tensor-core products with fp32 accumulation -- within
 *     the fp32 tolerance, on the tensor cores. It keeps a copy of qkv's size (T x 6 H x 64
 *     bf16 values) in the stream's workspace.
 *   - otherwise bf16 and fp16 inputs: a tensor-core kernel (tcgen05, fp32 accumulation) after
 *     rotation in fp32, the rotated q and k rounded to the input type; a positive scale
 *     multiplies the fp32 scores, any other scale the rotated q; the probabilities are
 *     rounded to the input type before the product with v. pk_attend and its typed forms
 *     run PK_KERNEL_TC (or the one PK_ATTN names); pk_attend_tuned picks by timing.
 *
 * Conventions for every entry point below:
 *   - All array pointers are DEVICE pointers of the current CUDA device; the caller owns
 *     them and the stream. Calls are asynchronous on `stream` (0 = the legacy stream).
 *   - qkv, cos, sin and out must be 16-byte aligned; cu and lse 4-byte aligned.
 *   - The library keeps, per (device, stream), a small workspace it allocates on first use
 *     and grows when a larger T arrives (tile records and a control word); pk_release()
 *     frees all of them. Calls on one stream are ordered; calls on different streams use
 *     different workspaces. A call may be captured in a CUDA graph once an earlier,
 *     uncaptured call on the same stream has allocated a workspace large enough for T;
 *     a captured call that would have to allocate returns PK_ERR_CAPTURE, nothing launched.
 *   - Return value: PK_OK, or an error code below. Errors found on the host (arguments,
 *     alignment, launch) are returned at once and nothing is launched. Errors found by
 *     the device (a malformed cu, a wait that ran out of time) are recorded in the
 *     stream's status word, read by pk_last_status(). The kernels never trap.
 *
 * Environment (read by the library, for tests and debugging):
 *   PK_TIMEOUT_MS          bound of every pipeline wait inside the kernels (default 2000);
 *                          read at the first call of the process.
 *   PK_DEBUG_SKIP_ARRIVE=1 test hook of the tensor-core kernels, read at every call: the
 *                          producer of each CTA withholds its first work-item hand-off, so
 *                          the call ends with PK_ERR_TIMEOUT after one wait bound and writes
 *                          no valid output; later calls without it are unaffected.
 *   PK_ATTN=q4|tc_single   pk_attend and its typed forms run PK_KERNEL_Q4 or
 *                          PK_KERNEL_TC_SINGLE instead of PK_KERNEL_TC for bf16 / fp16 inputs
 *                          outside the narrow windows (read at every call).
 *   PK_ATTN=split          the same for fp32 inputs with an fp32 output: PK_KERNEL_SPLIT
 *                          instead of PK_KERNEL_F32.
 */
#ifndef PK_H
#define PK_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t */

enum pk_status {
    PK_OK = 0,
    PK_ERR_ARG = 1,          /* null pointer with T > 0, S < 0, T < 0, H < 1, window < 0,
                                T or H beyond the limits, cu inconsistent with S and T */
    PK_ERR_ALIGN = 2,        /* a pointer is not aligned as required */
    PK_ERR_CUDA = 3,         /* a CUDA runtime or driver call failed */
    PK_ERR_UNSUPPORTED = 4,  /* the current device is not sm_103 (GB300) */
    PK_ERR_BAD_CU = 5,       /* device: cu[0] != 0, cu decreasing, or cu[S] != T */
    PK_ERR_TIMEOUT = 6,      /* device: a pipeline wait exceeded its bound; results invalid */
    PK_ERR_NOMEM = 7,        /* workspace allocation failed */
    PK_ERR_INTERNAL = 8,     /* device: schedule exceeded its capacity (a library bug) */
    PK_ERR_TOO_LARGE = 9,    /* pk_attend_noalloc: T above PK_NOALLOC_MAX_T */
    PK_ERR_CAPTURE = 10      /* the stream is being captured and its workspace would have to
                                be allocated or grown: make one uncaptured call first */
};

enum pk_dtype { PK_F32 = 0, PK_BF16 = 1, PK_F16 = 2 };

/* The forward kernels (pk_kernel_name gives each one's name). */
enum pk_kernel {
    PK_KERNEL_BAND = 0,       /* narrow windows: CUDA cores, fp32, no tile schedule */
    PK_KERNEL_F32 = 1,        /* fp32 inputs: CUDA cores, fp32, one tile record per CTA item */
    PK_KERNEL_TC = 2,         /* 16-bit: tcgen05, two query tiles of a record pair per SM,
                                 128-key stream tiles */
    PK_KERNEL_Q4 = 3,         /* 16-bit: tcgen05, two pipes of two query tiles per SM,
                                 64-key stream tiles */
    PK_KERNEL_TC_SINGLE = 4,  /* 16-bit: PK_KERNEL_TC with one tile record per work item */
    PK_KERNEL_SPLIT = 5       /* fp32: tcgen05 on bf16 hi / lo operand pairs, three products each
                                 (S = Qh Kh + Qh Kl + Ql Kh, O += Ph Vh + Ph Vl + Pl Vh), after a
                                 pre-pass that writes the rotated split copy; fp32 output only */
};

/* Limits: T <= PK_MAX_T, H <= PK_MAX_H. */
#define PK_MAX_T 2147483647LL
#define PK_MAX_H 1024

/*
 * Forward pass, bf16 qkv / cos / sin / out (the parameter list of the method's entry
 * point: pk_attend(qkv, cos, sin, cu, S, T, H, window, scale, out, lse, stream)).
 */
int pk_attend(const void *qkv, const void *cos, const void *sin, const uint32_t *cu, int S,
              int64_t T, int H, int window, float scale, void *out, float *lse,
              struct CUstream_st *stream);

/* The same for an explicit element type: bf16, fp16, fp32. */
int pk_attend_bf16(const void *qkv, const void *cos, const void *sin, const uint32_t *cu, int S,
                   int64_t T, int H, int window, float scale, void *out, float *lse,
                   struct CUstream_st *stream);
int pk_attend_f16(const void *qkv, const void *cos, const void *sin, const uint32_t *cu, int S,
                  int64_t T, int H, int window, float scale, void *out, float *lse,
                  struct CUstream_st *stream);
int pk_attend_f32(const void *qkv, const void *cos, const void *sin, const uint32_t *cu, int S,
                  int64_t T, int H, int window, float scale, void *out, float *lse,
                  struct CUstream_st *stream);

/* The same with the element type as an argument (enum pk_dtype). */
int pk_attend_dt(int dtype, const void *qkv, const void *cos, const void *sin,
                 const uint32_t *cu, int S, int64_t T, int H, int window, float scale, void *out,
                 float *lse, struct CUstream_st *stream);

/*
 * pk_attend_tuned -- the forward pass at the fastest usable kernel for the call's shape
 * (the pages' attend_tuned: each usable variant is timed once per key, the fastest is kept).
 *   - The arguments of pk_attend_dt, plus `longest`: the length of the longest sequence
 *     (host value; only the tuning key uses it).
 *   - Key: (current device, dtype, H, window + 1 (0 when window = 0), T rounded up to a power
 *     of two, longest rounded up to a power of two); pk_tune_key writes it as text.
 *   - Usable kernels: PK_KERNEL_BAND for 1 <= window <= 16 (its fp32 arithmetic keeps fp16
 *     inputs of large magnitude in tolerance), PK_KERNEL_F32 and PK_KERNEL_SPLIT for other
 *     fp32 calls, and PK_KERNEL_TC, PK_KERNEL_TC_SINGLE and PK_KERNEL_Q4 for other bf16 /
 *     fp16 calls.
 *   - A key met for the first time with more than one usable kernel is tuned on the call's
 *     own arguments: each kernel runs once untimed, then three rounds time two runs of each
 *     kernel in turn between two events on `stream` (the host waiting for the second); a
 *     kernel's time is its best round. The output is then that of one more run of the winner. Such a first call synchronizes the stream and cannot be captured in
 *     a CUDA graph (it returns PK_ERR_CAPTURE, nothing launched); later calls with the key
 *     are asynchronous. The cache lives until pk_tune_clear() or the end of the process.
 *   - Errors as pk_attend; longest < 0 gives PK_ERR_ARG.
 */
int pk_attend_tuned(int dtype, const void *qkv, const void *cos, const void *sin,
                    const uint32_t *cu, int S, int64_t T, int H, int window, float scale,
                    int64_t longest, void *out, float *lse, struct CUstream_st *stream);

/* The kernel pk_attend_tuned keeps for a key on the current device (enum pk_kernel), or -1
 * when the key has not been tuned. */
int pk_tune_pick(int dtype, int H, int window, int64_t T, int64_t longest);

/* The text of a tuning key, "dtype=bf16,heads=12,window=0,tokens=32768,longest=512", into
 * buf (n bytes, NUL-terminated). PK_ERR_ARG when it does not fit or an argument is invalid.
 * Needs no device. */
int pk_tune_key(int dtype, int H, int window, int64_t T, int64_t longest, char *buf, int n);

/* Forgets every tuned key. */
int pk_tune_clear(void);

/* The kernel pk_attend_dt runs for an element type and window (enum pk_kernel). Needs no
 * device. */
int pk_forward_kernel(int dtype, int window);

/* Name of a forward kernel (static storage; "" for an unknown id). */
const char *pk_kernel_name(int kernel);

/*
 * The tile schedule alone (for inspection and tests). Runs the device scheduler on `cu`
 * (device pointer) and copies its records to `tiles` (device pointer, room for `cap`
 * records of 8 uint32 each: q0, rows, k0, nk, seq, nseq, kind, ktiles -- query tokens
 * [q0, q0+rows), key tokens [k0, k0+nk), member sequences [seq, seq+nseq), kind 0 for a
 * 128-row piece of one sequence and 1 for a group of short sequences, ktiles =
 * ceil(nk/128)). Synchronizes `stream` and writes the record count to *nt (host pointer).
 * Returns PK_ERR_BAD_CU for a malformed cu (then *nt = 0), PK_ERR_ARG when cap is too small.
 * The rule (packed.rs fn layout for sequences longer than 64 tokens; short sequences packed
 * greedily into groups of at most 128 rows within 1024-token windows) is stated in full in
 * the oracle that checks it.
 */
int pk_schedule(const uint32_t *cu, int S, int64_t T, int window, uint32_t *tiles, int64_t cap,
                int64_t *nt, struct CUstream_st *stream);

/* Records pk_schedule can write for T tokens: enough room for `tiles`. */
int64_t pk_schedule_capacity(int64_t T);

/*
 * Synchronizes `stream`, returns the first device-detected error recorded for it since
 * the last call (PK_OK if none) and clears it.
 */
int pk_last_status(struct CUstream_st *stream);

/*
 * Kernel timing. pk_profile_start(n) makes the next n forward calls on the current device
 * record a CUDA event pair on their stream around each of their two kernels (the tile
 * scheduler, or for narrow windows the check of cu, and the attention kernel). pk_profile_stop() synchronizes those events, writes
 * the summed durations in milliseconds and the number of calls recorded, and stops the
 * recording. Returns PK_ERR_ARG for n < 1 or null outputs, PK_ERR_CUDA on event failures.
 */
int pk_profile_start(int n);
int pk_profile_stop(double *schedule_ms, double *attend_ms, int *calls);

/*
 * pk_attend_noalloc: the same forward pass for callers that cannot allocate device memory.
 * hanzo-kernel 0.2.42 packed.rs has no counterpart to this entry point.
 *
 * pk_attend allocates a small workspace with cudaMalloc on first use per stream. Callers
 * that plan every byte of device memory themselves (a serving process with a fixed budget,
 * a plugin whose enqueue step may not allocate, an application whose pool allocator owns
 * the device) or that cannot afford the synchronization a cudaMalloc brings use this call
 * instead: it allocates nothing, and runs the kernels pk_attend_dt runs for the same
 * arguments (pk_forward_kernel; PK_KERNEL_F32 where that is PK_KERNEL_SPLIT, whose copy of
 * qkv has no place in a fixed scratch area) on a scratch area compiled into
 * the library (a static __device__ array of about 4 MB, present on every GPU that loads
 * the library until the process exits).
 *   - dtype: enum pk_dtype; the other arguments as pk_attend.
 *   - T at most PK_NOALLOC_MAX_T tokens; larger T returns PK_ERR_TOO_LARGE, nothing launched.
 *   - status: optional device pointer (NULL: none). The call writes there, in stream order,
 *     the device-detected result of this call (PK_OK, PK_ERR_BAD_CU, PK_ERR_TIMEOUT).
 *     pk_last_status does not see this entry point's device errors.
 *   - The first call on a device does a one-time set-up with that device current (device
 *     check, kernel attributes, the scratch array's device address); make it before any
 *     stream capture.
 *   - All calls share the one scratch area, which keeps the last call's contents (each call
 *     clears its control block first): calls that overlap on the GPU race, so order them
 *     (one stream, or events between streams).
 */
#define PK_NOALLOC_MAX_T 1048576LL
int pk_attend_noalloc(int dtype, const void *qkv, const void *cos, const void *sin,
                      const uint32_t *cu, int S, int64_t T, int H, int window, float scale,
                      void *out, float *lse, int *status, struct CUstream_st *stream);

/*
 * pk_attend_backward -- the backward pass (the pages' attend_back): the gradient of
 * sum(dout * out) with respect to qkv, through the rotation, for a forward call with the
 * same arguments. Per query row i and visible key j: P_ij = exp(scale q'_i . k'_j - lse_i),
 * D_i = dout_i . out_i, dS_ij = P_ij (dout_i . v_j - D_i); dv_j = sum_i P_ij dout_i,
 * dq_i = rot^T(scale sum_j dS_ij k'_j), dk_j = rot^T(scale sum_i dS_ij q'_i).
 *   - dtype, qkv, cos, sin, cu, S, T, H, window, scale: as the forward call (pk_attend_dt).
 *   - out [T, H*64] (dtype) and lse [H, T] (fp32): the forward's outputs.
 *   - dout [T, H*64] (dtype): the gradient of the loss with respect to out.
 *   - dqkv [T, 3*H*64] (dtype): written with the gradients of q | k | v.
 *   - bf16 / fp16: tensor-core products (tcgen05, accumulators in tensor memory; with
 *     PK_BWD_MMA_SYNC=1 in the environment the warp-level mma.sync kernel instead) with q',
 *     k', P and dS rounded to dtype as operands and fp32 accumulation; fp32: fp32 arithmetic
 *     on the CUDA cores. One rounding of dqkv to dtype.
 *   - Allocates, on first use per (device, stream) and when a larger H*T arrives, an fp32
 *     scratch of about H*T*(1 + 3*64) floats (kept with the workspace, freed by pk_release).
 *     The capture rule of the workspace applies to it: a captured call that would have to
 *     allocate it returns PK_ERR_CAPTURE, nothing launched.
 *   - Alignment and errors as pk_attend (dout, dqkv 16-byte aligned); device errors (bad cu)
 *     in pk_last_status(stream).
 */
int pk_attend_backward(int dtype, const void *qkv, const void *cos, const void *sin,
                       const uint32_t *cu, int S, int64_t T, int H, int window, float scale,
                       const void *out, const float *lse, const void *dout, void *dqkv,
                       struct CUstream_st *stream);

/*
 * pk_attend_mixed -- fp32 inputs, fp32 arithmetic, a 16-bit output: kime's attention variant
 * with an FP32 qkv and a half output (the qkv stays FP32 because FP16 rounding of q and k
 * moves the softmax; the pages' plan.rs, fn types). Same operation as pk_attend_f32 (the
 * CUDA-core path), with out = O / l rounded once to out_dtype.
 *   - out_dtype: PK_F16 or PK_BF16 (PK_F32 gives pk_attend_f32); out [T, H*64] of that type.
 *   - qkv, cos, sin: fp32, as pk_attend_f32; the other arguments, alignment and errors as pk_attend.
 */
int pk_attend_mixed(int out_dtype, const float *qkv, const float *cos, const float *sin,
                    const uint32_t *cu, int S, int64_t T, int H, int window, float scale,
                    void *out, float *lse, struct CUstream_st *stream);

/*
 * pk_attend_mixed_ops -- fp32 storage with 16-bit tensor-core operands (the pages' generic
 * attend with storage type F = f32 and operand type M = f16 or bf16, as packed.rs's tests run
 * it): q and k are rotated in fp32 from the fp32 qkv and tables, q', k', v and the
 * probabilities are rounded to op_dtype as the operands of the products, which accumulate in
 * fp32, and out is written in fp32.
 *   - op_dtype: PK_F16 or PK_BF16 (otherwise PK_ERR_ARG).
 *   - qkv, cos, sin: fp32 as pk_attend_f32; out [T, H*64] fp32; lse [H, T] fp32; the other
 *     arguments, alignment, capture and errors as pk_attend.
 *   - For fp32 inputs whose values are representable in op_dtype the result equals the
 *     op_dtype path's (pk_attend_dt with op_dtype inputs and PK_KERNEL_TC), out before its
 *     rounding to op_dtype, bit for bit.
 *   - Allocates, on first use per (device, stream) and when a larger T*H arrives, the rotated
 *     16-bit copy of qkv (T*3*H*64 elements, kept with the workspace, freed by pk_release).
 *   - Kernels: the tile scheduler, the rotation into the copy, PK_KERNEL_TC (fp32 output).
 */
int pk_attend_mixed_ops(int op_dtype, const float *qkv, const float *cos, const float *sin,
                        const uint32_t *cu, int S, int64_t T, int H, int window, float scale,
                        float *out, float *lse, struct CUstream_st *stream);

/*
 * pk_rope -- the standalone rotary embedding of a packed qkv: the pages' rope op
 * (hanzo-kernel fast ops, FastOp::Rope and its graph fallback), applied as kime's rope step
 * applies it, to every q and k head vector of qkv.
 *   - For a head vector x (64 features) of a token at in-sequence position p (the token minus
 *     the start of its sequence in cu), with h = dims / 2, c_j = cos[p h + j], s_j = sin[p h + j]:
 *     pair j < h is (j, j + h) (traditional = 0: the two halves) or (2j, 2j + 1)
 *     (traditional != 0: interleaved pairs); forwards (inverse = 0)
 *         y_a = x_a c_j - x_b s_j,  y_b = x_a s_j + x_b c_j,
 *     inversely (inverse != 0, the transposed rotation: the gradient of the forward one)
 *         y_a = x_a c_j + x_b s_j,  y_b = x_b c_j - x_a s_j;
 *     features dims .. 63 are copied. Arithmetic in fp32, one rounding to the element type.
 *   - dtype: enum pk_dtype, for x, y, cos and sin alike.
 *   - x, y: device [T, 3 H 64] (q | k | v blocks, heads contiguous, as pk_attend's qkv). y may
 *     be x (in place: v is left as it is); otherwise v is copied, and x and y must not overlap.
 *     4-byte aligned (8-byte for PK_F32).
 *   - cos, sin: device [P, dims / 2] tables; P >= the longest sequence. Element-aligned.
 *   - cu, S, T: as pk_attend (device cu[S + 1], cu[0] = 0, non-decreasing, cu[S] = T).
 *   - H in [1, PK_MAX_H]; dims even in [2, 64].
 *   - status: optional device int (NULL: none), written in stream order: PK_OK, or
 *     PK_ERR_BAD_CU when cu is malformed or a position reaches P (such tokens are skipped).
 *   - Returns PK_OK or PK_ERR_ARG / PK_ERR_ALIGN / PK_ERR_UNSUPPORTED / PK_ERR_CUDA (nothing
 *     launched). Asynchronous on `stream`; allocates nothing.
 */
int pk_rope(int dtype, const void *x, void *y, const void *cos, const void *sin, int64_t P,
            const uint32_t *cu, int S, int64_t T, int H, int dims, int traditional, int inverse,
            int *status, struct CUstream_st *stream);

/* Text of a status code (static storage). */
const char *pk_status_string(int status);

/* Library version: major * 10000 + minor * 100 + patch. */
int pk_version(void);

/* Frees every workspace, after synchronizing each device that holds one (so it may be called
 * after the streams the workspaces were made for have been destroyed). */
int pk_release(void);

#ifdef __cplusplus
}
#endif

#endif /* PK_H */
