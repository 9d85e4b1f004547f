/*
 * la.h -- C ABI of the GB300 (sm_103a) causal linear-attention library.
 *
 * What is computed (feature map phi(x) = elu(x) + 1 = x + 1 for x >= 0 and
 * exp(x) for x < 0, applied elementwise to q and to k, never to v):
 *
 *   S_t = S_{t-1} + phi(k_t) v_t^T        state, dk x dv, rows = key components
 *   z_t = z_{t-1} + phi(k_t)              normaliser, dk
 *   o_t = phi(q_t)^T S_t / (phi(q_t)^T z_t + eps)
 *
 * with S_0 = 0, z_0 = 0 and the state inclusive of token t ("Linear
 * Attention: KV를 고정 크기 상태에 누적하기", section "상태 갱신과 읽기를 식으로
 * 정리하기": S_{t+1} = S_t + k_t v_t^T, z_{t+1} = z_t + k_t, y_t read from
 * S_{t+1}; feature map from the "Transformers are RNNs" review, feature-map
 * table). Non-causal attention reads the full-sequence state S_N for every
 * query ("Linear Attention: KV를 고정 크기 상태에 누적하기", fig. 2). No
 * 1/sqrt(d) scale is applied inside; scale the inputs if one is wanted.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Layout: q, k are [B, H, N, dk], v, out are [B, H, N, dv], contiguous,
 *    row-major (token-major within a head). States S are [B, H, dk, dv] and
 *    normalisers z are [B, H, dk], fp32, contiguous.
 *  - dtype: LA_BF16 means q, k, v, out (and gradients) are bfloat16;
 *    LA_F32 means float32. Arithmetic, states and normalisers are fp32 in
 *    both cases; bf16 results are rounded to nearest even.
 *  - Supported head sizes: dk, dv in {16, 32, 64, 128}.
 *  - Pointers: every data pointer is device memory owned by the caller and
 *    must be 16-byte aligned. The library allocates nothing: scratch space is
 *    passed in as `workspace` (sizes from the *_workspace_size queries).
 *  - Streams: `stream` is a cudaStream_t (NULL = legacy default stream).
 *    Calls validate their arguments synchronously and then only enqueue
 *    kernels; they return before the GPU work finishes.
 *  - Errors: a non-OK status means nothing was enqueued (LA_ERR_INVALID_ARG,
 *    LA_ERR_UNSUPPORTED) or a launch failed (LA_ERR_CUDA). la_last_error()
 *    gives a one-line reason, per calling thread. Empty problems (B, H or N
 *    equal to 0) are valid and enqueue nothing except zeroing S_final/z_final.
 *  - Device: kernels are built for sm_103a (GB300) only; on another device
 *    the launch fails with LA_ERR_CUDA.
 */
#ifndef LA_H_
#define LA_H_

#include <stddef.h>

#if defined(__GNUC__)
#define LA_API __attribute__((visibility("default")))
#else
#define LA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum la_status {
  LA_OK = 0,
  LA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, negative size, bad eps, short workspace */
  LA_ERR_UNSUPPORTED = 2, /* head size or dtype outside the supported set */
  LA_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed */
  LA_ERR_TIMEOUT = 4      /* reserved: a device-side bounded wait gave up */
} la_status;

typedef enum la_dtype { LA_F32 = 0, LA_BF16 = 1 } la_dtype;

/* An opaque cudaStream_t. */
typedef void* la_stream_t;

/* Human-readable name of a status code. Never NULL. */
LA_API const char* la_status_string(la_status status);

/* One-line reason for the last non-OK status returned on this thread
 * ("" if none). The pointer stays valid until the next call on this thread. */
LA_API const char* la_last_error(void);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
LA_API int la_version(void);

/*
 * Bytes of scratch memory la_forward needs for these sizes (0 if none).
 * Holds one fp32 (dk*dv + dk) state per (batch, head, sequence segment).
 * Negative sizes or unsupported head sizes return 0 (la_forward then reports
 * the error).
 */
LA_API size_t la_forward_workspace_size(int B, int H, int N, int dk, int dv,
                                 int causal, la_dtype dtype);

/*
 * Forward pass over whole sequences.
 *
 *   causal != 0 : o_t = phi(q_t)^T S_t / (phi(q_t)^T z_t + eps), S_t over j <= t
 *                 ("상태공간모델·선형 어텐션 — 어텐션의 O(N²) 대안", section 2,
 *                 masked form = recurrence)
 *   causal == 0 : every query reads S_N, z_N (association reorder,
 *                 "Linear Attention, 곱의 순서를 바꾸면 생기는 일", section
 *                 "곱의 순서를 바꾸면 기억이 요약이 된다")
 *
 * q, k      [B,H,N,dk]  in, dtype
 * v         [B,H,N,dv]  in, dtype
 * out       [B,H,N,dv]  out, dtype (must not alias the inputs)
 * eps       >= 0, finite, added to the denominator
 * S_final   [B,H,dk,dv] fp32 out or NULL: the full-sequence state S_N
 * z_final   [B,H,dk]    fp32 out or NULL: z_N (both or neither)
 * workspace device scratch of at least la_forward_workspace_size(...) bytes,
 *           NULL allowed when that size is 0. Contents on entry are ignored.
 *
 * The sequence is processed in chunks on the tensor cores; segments of one
 * sequence run on different SMs and are joined by a prefix scan of their
 * fp32 state sums kept in `workspace`.
 */
LA_API la_status la_forward(const void* q, const void* k, const void* v, void* out,
                     int B, int H, int N, int dk, int dv, int causal,
                     float eps, la_dtype dtype, float* S_final, float* z_final,
                     void* workspace, size_t workspace_bytes,
                     la_stream_t stream);

/*
 * la_forward on inputs and outputs in HOST memory: the call copies q, k, v to
 * the device, runs the forward and copies out back, overlapping the three.
 * The B*H sequences are split into `slices` groups of whole sequences
 * (contiguous in the [B,H,N,d] layout); slice i's host-to-device copies run on
 * an internal copy stream while slice i-1 is computed on `stream` and slice
 * i-2's output returns on a second internal copy stream, through two device
 * staging slots in `workspace`. The outputs equal la_forward's on the same
 * inputs (each slice is an independent la_forward call over its sequences).
 *
 * q, k      [B,H,N,dk] dtype, host memory, in
 * v         [B,H,N,dv] dtype, host memory, in
 * out       [B,H,N,dv] dtype, host memory, out (must not alias the inputs)
 * slices    >= 1; clamped to B*H. 1 runs copy, compute, copy in sequence.
 * workspace device scratch of at least la_forward_host_workspace_size(...)
 *           bytes (the two staging slots and one la_forward workspace),
 *           16-byte aligned.
 * stream    work is ordered after the work already on `stream`, and the
 *           call's last copy to `out` is complete when `stream` reaches the
 *           point after this call (the internal streams join it there).
 *
 * Page-locked (pinned) host memory gives the overlap; pageable memory works
 * but each copy then blocks the calling thread. No final state is returned
 * (use la_forward for S_final, z_final). Not for CUDA-graph capture. Errors
 * as la_forward; on an error after the first enqueue, work already enqueued
 * still completes and `stream` still joins the internal streams.
 */
LA_API size_t la_forward_host_workspace_size(int B, int H, int N, int dk, int dv,
                                              int causal, la_dtype dtype, int slices);
LA_API la_status la_forward_host(const void* q, const void* k, const void* v, void* out,
                                 int B, int H, int N, int dk, int dv, int causal,
                                 float eps, la_dtype dtype, int slices,
                                 void* workspace, size_t workspace_bytes,
                                 la_stream_t stream);

/*
 * One recurrent inference step per (batch, head), in place on the state:
 *
 *   S <- S + phi(k) v^T;  z <- z + phi(k);  out = phi(q)^T S / (phi(q)^T z + eps)
 *
 * ("Linear Attention: KV를 고정 크기 상태에 누적하기", section "상태 갱신과 읽기를
 * 식으로 정리하기"; constant work per token as in "Linear Attention, 곱의 순서를
 * 바꾸면 생기는 일", section "곱의 순서를 바꾸면 기억이 요약이 된다").
 *
 * S    [B,H,dk,dv] fp32 in/out      z [B,H,dk] fp32 in/out
 * q, k [B,H,dk] dtype in            v [B,H,dv] dtype in
 * out  [B,H,dv] dtype out
 * The read uses the state after the update (inclusive of this token), so a
 * prefill of t tokens followed by this step equals la_forward's output t.
 */
LA_API la_status la_decode_step(float* S, float* z, const void* q, const void* k,
                         const void* v, void* out, int B, int H, int dk,
                         int dv, float eps, la_dtype dtype,
                         la_stream_t stream);

/*
 * T consecutive decode steps per (batch, head) in one call: for t = 0 .. T-1,
 * the step of la_decode_step with token t (same formulas, same inclusive read).
 * The state is read and written once per call, not once per token, so its
 * traffic is shared by the T tokens (multi-token decode: a prompt appended to
 * a cached state, or several tokens verified at once; "Linear Attention: KV를
 * 고정 크기 상태에 누적하기", section "상태 갱신과 읽기를 식으로 정리하기").
 *
 * S    [B,H,dk,dv] fp32 in/out      z [B,H,dk] fp32 in/out
 * q, k [B,H,T,dk] dtype in          v [B,H,T,dv] dtype in
 * out  [B,H,T,dv] dtype out
 * T >= 0 (T = 0 leaves S and z unchanged). With T = 1 it equals
 * la_decode_step; from a prefill of t tokens its outputs equal la_forward's
 * outputs t .. t+T-1 on the appended tokens. Errors as la_decode_step.
 */
LA_API la_status la_decode_steps(float* S, float* z, const void* q, const void* k,
                          const void* v, void* out, int B, int H, int T, int dk,
                          int dv, float eps, la_dtype dtype, la_stream_t stream);

/*
 * Decay-gated decode: T steps per (batch, head) in one call, the whole summary
 * multiplied by a per-head factor alpha before each token is added ("Linear
 * Attention, 곱의 순서를 바꾸면 생기는 일", the paragraph on 감쇠 게이팅; the
 * recurrence h_t = a h_{t-1} + x_t of "상태공간모델·선형 어텐션", section 3):
 *
 *   S <- alpha S + phi(k) v^T;  z <- alpha z + phi(k);
 *   out = phi(q)^T S / (phi(q)^T z + eps)
 *
 * alpha [H] fp32 device memory, one factor per head (alpha = 1 gives
 * la_decode_steps; values above 1 make the state grow without bound and are
 * not checked). Other arguments and errors as la_decode_steps. Where
 * la_decode_path(dk, dv, dtype, T) is 1 the call runs on the tensor cores
 * (the decay weights as bf16 hi + lo rows of the update, the state within
 * 1e-5 of its largest entry against the fp32 recurrence).
 */
LA_API la_status la_decode_steps_decay(float* S, float* z, const void* q, const void* k,
                                const void* v, void* out, int B, int H, int T, int dk,
                                int dv, const float* alpha, float eps, la_dtype dtype,
                                la_stream_t stream);

/*
 * Decay-gated causal forward: the outputs of la_decode_steps_decay run over
 * the whole sequence from the zero state, computed chunk by chunk on the
 * tensor cores (the chunked form of the same recurrence: inside a chunk the
 * causal weights phi(q_t).phi(k_j) carry alpha^(t-j); across chunks the
 * carried state decays by alpha per token).
 *
 * q, k, v, out as la_forward (bf16, dk = dv = 64 only; LA_ERR_UNSUPPORTED
 * otherwise); alpha [H] fp32 device memory, each in [0.5, 1] (smaller factors
 * underflow the chunk's weights; not checked); S_final, z_final as la_forward
 * (the decayed state after the last token); workspace sized by
 * la_forward_workspace_size(B, H, N, 64, 64, 1, LA_BF16).
 */
LA_API la_status la_forward_decay(const void* q, const void* k, const void* v, void* out,
                           int B, int H, int N, int dk, int dv, const float* alpha, float eps,
                           la_dtype dtype, float* S_final, float* z_final,
                           void* workspace, size_t workspace_bytes, la_stream_t stream);

/*
 * Gradients of the decay-gated causal attention (la_decode_steps_decay run
 * over the whole sequence from the zero state; la_forward_decay's outputs):
 * dq, dk, dv of L = sum(dout * out) by the same forward and reverse
 * cumulative sums as la_backward, with the reverse sums decaying like the
 * state, R_j = phi(q_j) a_j^T + alpha R_{j+1}, r_j = b_j phi(q_j) + alpha
 * r_{j+1} (the chain rule through S_t = alpha S_{t-1} + phi(k_t) v_t^T).
 *
 * Arguments as la_backward with causal = 1, plus alpha [H] fp32 device
 * memory, one factor per head in (0, 1] (not checked). Runs on the CUDA-core
 * kernels (f32 or bf16, every supported head size), segments of each
 * sequence in parallel: the segment sums are decayed to their ends and
 * combined by a decaying scan. Workspace: la_backward_workspace_size(B, H,
 * N, dk, dv, 1, dtype) bytes. NULL alpha is LA_ERR_INVALID_ARG.
 */
LA_API la_status la_backward_decay(const void* q, const void* k, const void* v,
                                   const void* dout, void* dq, void* dk_, void* dv_,
                                   int B, int H, int N, int dk, int dv,
                                   const float* alpha, float eps, la_dtype dtype,
                                   void* workspace, size_t workspace_bytes,
                                   la_stream_t stream);

/*
 * Delta-rule decode: T steps per (batch, head) in one call; each step reads
 * the state with the key and adds only the difference to the value (the
 * paragraph on 델타 규칙 of the same page):
 *
 *   u = S^T k;  S <- S + k (v - u)^T;  out = S^T q
 *
 * q and k are used as given (no feature map) and the read is not normalised,
 * as in the page's example; with unit-norm keys a write replaces what the key
 * held. S [B,H,dk,dv] fp32 in/out; q, k [B,H,T,dk], v [B,H,T,dv] in, out
 * [B,H,T,dv] out, dtype. Errors as la_decode_steps. Where
 * la_decode_path(dk, dv, dtype, T) is 1 the call runs on the tensor cores in
 * groups of 16 tokens: the increments of a group solve a unit lower-
 * triangular system (the chunked form of the same recurrence), the state is
 * read with its bf16 high and low parts, and the state stays within 1e-5 of
 * its largest entry against the fp32 token recurrence.
 */
LA_API la_status la_decode_steps_delta(float* S, const void* q, const void* k, const void* v,
                                void* out, int B, int H, int T, int dk, int dv,
                                la_dtype dtype, la_stream_t stream);

/*
 * How la_forward splits a call of these sizes (with a final state requested
 * or not: the split may differ), for tests and tuning. out[5] receives: the
 * segments per sequence P, the tokens per segment, the state-pass CTAs per
 * segment F, the number of balanced pieces (0 when the call runs by
 * segments) and the 128-token chunks per piece. With pieces, the heads'
 * chunks are laid end to end and cut into equal pieces, one CTA each, so
 * that every SM gets the same work even when B*H does not divide the SM
 * count (causal tensor-core forward at d = 128 without a final state).
 * On the tensor-core paths the split also weighs the state records each
 * segment or piece sums before its first chunk, so calls with few heads get
 * fewer, longer segments than the CUDA-core path.
 * LA_ERR_INVALID_ARG for sizes outside la_forward's range or a NULL out.
 */
LA_API la_status la_forward_plan(int B, int H, int N, int dk, int dv, int causal, la_dtype dtype,
                                 int final_state, int* out);

/*
 * Delta rule over whole sequences: the same recurrence as
 * la_decode_steps_delta, N tokens per (batch, head), computed chunk by chunk
 * (32 tokens). Within a chunk the increments u'_t = v_t - S_{t-1}^T k_t solve
 * a unit lower-triangular system (I + A) U' = V - K S_0, A the chunk's key
 * products k_t . k_j below the diagonal; then out = Q S_0 + (Q K^T, j <= t) U'
 * and S <- S_0 + K^T U'. Exact up to rounding against the token-by-token
 * update; the work per chunk is dense products instead of N dependent steps.
 *
 * S [B,H,dk,dv] fp32 in/out (the state before the first token; after the
 * call, the state after the last one); q, k [B,H,N,dk], v [B,H,N,dv] in,
 * out [B,H,N,dv] out, dtype; fp32 arithmetic. dk == dv in {16, 32, 64, 128}
 * (otherwise LA_ERR_UNSUPPORTED); N = 0 or B*H = 0 is a no-op. Pointers
 * 16-byte aligned device memory, not overlapping. Errors as la_decode_steps.
 * bf16 at d = 128 with B*H >= 64 runs the tensor-core kernel of
 * la_decode_steps_delta (groups of 16 tokens; the state read and the update
 * as MMAs with the fp32 state split into bf16 hi + lo, the triangular solve
 * per value index), which is faster there; otherwise 32-token chunks on the
 * CUDA cores, the state split into 32-column blocks.
 */
LA_API la_status la_forward_delta(float* S, const void* q, const void* k, const void* v,
                                  void* out, int B, int H, int N, int dk, int dv,
                                  la_dtype dtype, la_stream_t stream);

/*
 * State snapshot / restore: dst_S <- src_S ([B,H,dk,dv] fp32) and, if both
 * are given, dst_z <- src_z ([B,H,dk] fp32), on `stream`. The same call saves
 * a state (prefix caching) and puts it back; a later step from the restored
 * state repeats the original bit for bit. Pointers 16-byte aligned, device
 * memory, not overlapping; dst_z and src_z both NULL or both non-NULL.
 */
LA_API la_status la_state_copy(float* dst_S, float* dst_z, const float* src_S,
                        const float* src_z, int B, int H, int dk, int dv,
                        la_stream_t stream);

/*
 * Bytes of scratch memory la_backward needs (0 if none): one fp32 state and
 * one fp32 reverse accumulator (dk*dv + dk each) per (batch, head, segment)
 * plus two fp32 scalars per token (the denominator and the normaliser's
 * gradient coefficient), no per-token states. The tensor-core and CUDA-core
 * paths may split the sequences into different segments: the size covers
 * both.
 */
LA_API size_t la_backward_workspace_size(int B, int H, int N, int dk, int dv,
                                  int causal, la_dtype dtype);

/*
 * Gradients of L = sum(dout * out) with out = la_forward(q, k, v), by
 * forward and reverse cumulative sums, storing no per-token states ("Transformers
 * are RNNs" review, section "그래디언트 계산 — 선형 시간·상수 메모리"; the
 * formulas are re-derived since the page lost them):
 *
 *   D_t = phi(q_t).z_t + eps, o_t = S_t^T phi(q_t) / D_t,
 *   a_t = dout_t / D_t,  b_t = -(dout_t . o_t) / D_t,
 *   dphi(q_t) = S_t a_t + b_t z_t,
 *   R_j = sum_{t>=j} phi(q_t) a_t^T,  r_j = sum_{t>=j} b_t phi(q_t),
 *   dphi(k_j) = R_j v_j + r_j,  dv_j = R_j^T phi(k_j),
 *   dq = dphi(q) * phi'(q),  dk = dphi(k) * phi'(k)
 * (non-causal: S_t -> S_N, R_j -> R_0).
 *
 * q, k, v, dout as in la_forward (dout has out's shape); dq [B,H,N,dk],
 * dk_ [B,H,N,dk], dv_ [B,H,N,dv] out, dtype. workspace as in la_forward,
 * sized by la_backward_workspace_size.
 */
LA_API la_status la_backward(const void* q, const void* k, const void* v,
                      const void* dout, void* dq, void* dk_, void* dv_, int B,
                      int H, int N, int dk, int dv, int causal, float eps,
                      la_dtype dtype, void* workspace, size_t workspace_bytes,
                      la_stream_t stream);

/*
 * la_backward reusing the state records that the matching la_forward call
 * left in its workspace (save-for-backward): the backward's own pass over k
 * and v, which rebuilds the per-segment sums of S and z, is skipped.
 *
 * saved        the workspace given to la_forward (not la_forward_decay, whose
 *              records are decayed) with the same q, k, v, B, H, N, dk, dv,
 *              causal and dtype, unchanged since, and under the same
 *              la_set_path setting; saved_bytes at least
 *              la_forward_workspace_size(...) of those arguments. It is read,
 *              not written.
 * workspace    the backward's own scratch, la_backward_workspace_size(...)
 *              bytes, separate from `saved`.
 * Other arguments and the results as la_backward. The records are used by
 * the tensor-core path (bf16, dk = dv = 64); on the CUDA-core path the
 * backward recomputes them and `saved` is only checked for size. NULL `saved`
 * is LA_ERR_INVALID_ARG.
 */
LA_API la_status la_backward_saved(const void* q, const void* k, const void* v,
                                   const void* dout, void* dq, void* dk_, void* dv_,
                                   int B, int H, int N, int dk, int dv, int causal,
                                   float eps, la_dtype dtype, const void* saved,
                                   size_t saved_bytes, void* workspace,
                                   size_t workspace_bytes, la_stream_t stream);

/*
 * Kernel-path selection, for tests and measurements. LA_PATH_AUTO (the
 * default) takes the tensor-core (tcgen05) kernels where they apply (bf16;
 * forward dk = dv in {64, 128}, backward dk = dv = 64, causal or not) and the
 * CUDA-core kernels elsewhere; LA_PATH_SIMT
 * forces the CUDA-core kernels everywhere. Process-wide; returns the
 * previous setting, or -1 for an unknown value (setting unchanged).
 */
enum { LA_PATH_AUTO = 0, LA_PATH_SIMT = 1 };
LA_API int la_set_path(int path);

/* Which path la_forward / la_backward take for these arguments under the
 * current setting: 0 = CUDA-core, 1 = tensor-core; -1 if unsupported. */
LA_API int la_forward_path(int dk, int dv, la_dtype dtype, int causal);
LA_API int la_backward_path(int dk, int dv, la_dtype dtype, int causal);
/* Which kernel la_decode_steps (and la_decode_steps_decay,
 * la_decode_steps_delta) takes for T tokens per call: 1 = tensor-core (bf16,
 * dk = dv = 128, T >= 2), 0 = CUDA-core; -1 if unsupported. */
LA_API int la_decode_path(int dk, int dv, la_dtype dtype, int T);

/*
 * Device-side status. The tensor-core kernels bound every wait on another
 * warp or on the copy engine; if one ever gives up, the kernel stops early
 * (its outputs are then incomplete), frees its tensor memory and records
 * LA_ERR_TIMEOUT in a per-device status word. la_device_status reads that
 * word for the current device (a synchronous copy: synchronise the streams
 * that ran the library's kernels first), returns LA_OK or LA_ERR_TIMEOUT and,
 * if `clear` is non-zero, resets it.
 */
LA_API la_status la_device_status(int clear);

/*
 * Test switch for the bounded waits above. The next causal tensor-core
 * la_forward launch (bf16, dk = dv in {64, 128}) has its MMA-issuing thread
 * wait on a barrier that nothing ever completes: the wait gives up after its
 * limit (2 s), the kernel winds down without issuing any MMA, and
 * la_device_status reports LA_ERR_TIMEOUT. That call's outputs are
 * unspecified; later calls run normally. One-shot, process-wide. For tests of
 * the failure path only; it faults nothing.
 */
LA_API void la_test_timeout_next_forward(void);

/*
 * Forward pass for callers that cannot allocate device memory.
 *
 * The pages describe no counterpart to this entry point: it exists for
 * integration. la_forward needs scratch memory, which callers normally
 * allocate once and pass in. Some callers cannot: plugin or custom-operator
 * hosts that own all device memory and hand an operator only its input and
 * output buffers, and latency-critical serving loops where cudaMalloc's
 * implicit device synchronisation is unacceptable.
 *
 * la_forward_noalloc computes exactly what la_forward computes, with the
 * same arguments except the workspace, which here is a file-scope device
 * array of LA_NOALLOC_SCRATCH_BYTES inside the library. Every GPU that loads
 * the library holds that array until the process exits.
 *
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current) and caches it for the
 *    life of the process.
 *    A cudaDeviceReset (or anything else that destroys the device's primary
 *    context) leaves the cached address stale: calling la_forward_noalloc on
 *    that device afterwards is not supported.
 *  - Problems whose scratch (la_forward_workspace_size) exceeds
 *    LA_NOALLOC_SCRATCH_BYTES are rejected with LA_ERR_INVALID_ARG before
 *    anything is launched.
 *  - It calls no cudaMalloc, cudaFree or other allocating routine.
 *  - All calls on a device share the one array, which keeps the last call's
 *    contents; nothing in it needs to start at zero (each call writes every
 *    record it reads). Calls whose GPU work overlaps (different streams
 *    without ordering) race on the array: order them on one stream.
 */
#define LA_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
LA_API la_status la_forward_noalloc(const void* q, const void* k, const void* v, void* out,
                                    int B, int H, int N, int dk, int dv, int causal,
                                    float eps, la_dtype dtype, float* S_final,
                                    float* z_final, la_stream_t stream);

/*
 * Measurement hooks (no effect on results).
 *
 * la_profile_enable(1) clears the record and starts timing: every later call
 * records a CUDA event pair on its stream around each kernel span listed
 * below. la_profile_enable(0) stops recording. la_profile_read waits for the
 * recorded events, writes up to `max` (label, milliseconds) pairs in call
 * order and returns how many spans were recorded (possibly more than `max`).
 * Events are created lazily with cudaEventCreate; no device memory is
 * allocated. la_launch_count returns the number of kernels this library has
 * launched in the process so far.
 */
enum {
  LA_SPAN_FWD_STATE = 0,   /* la_forward: per-segment state sums          */
  LA_SPAN_FWD_SCAN = 1,    /* la_forward: segment prefix scan             */
  LA_SPAN_FWD_OUTPUT = 2,  /* la_forward: chunked output kernel           */
  LA_SPAN_DECODE = 3,      /* la_decode_step                              */
  LA_SPAN_BWD_STATE = 4,   /* la_backward: per-segment state sums + scan  */
  LA_SPAN_BWD_SWEEP1 = 5,  /* la_backward: forward sweep (dq)             */
  LA_SPAN_BWD_SCAN = 6,    /* la_backward: reverse segment scan           */
  LA_SPAN_BWD_SWEEP2 = 7   /* la_backward: reverse sweep (dk, dv)         */
};
LA_API la_status la_profile_enable(int on);
LA_API int la_profile_read(int* labels, float* ms, int max);
LA_API long long la_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* LA_H_ */
