/*
 * qgemv.h -- C ABI of libqgemv: the batch-1 / few-token decode GEMV
 * y = W.x with Q4_0 weights and Q8_0-quantised activations, on one GB300.
 *
 * The operation (minfer README, "How it works": gemv_dp4a, a q4_0 GEMV with
 * int8 activations; "The optimization journey", M3.5 and M9):
 *   - W is an N x K matrix in Q4_0 blocks of 32 weights along K: an fp16
 *     scale d, then 16 bytes whose low nibble is element j and high nibble
 *     element j+16 (j < 16); weight = (n - 8) * d.  18 bytes per block.
 *   - x holds T token columns of K fp32 values.  Each block of 32 is
 *     quantised to Q8_0: d = amax/127 (fp32, stored as fp16), and
 *     q = round-half-away-from-zero(x * (1/d)) as int8, 1/d taken from the
 *     fp32 d (all zero when amax = 0).
 *   - For every output row i, token t and block b the exact integer sum
 *     isum = sum_j (n_j - 8) * q_j is formed (minfer M15/M16: "identical
 *     per-block integer sums"), scaled by d_w * d_x and accumulated in fp32.
 *
 * Summation order.  Every entry point, for every T and every launch shape,
 * accumulates one output in the same fixed order, which depends on K only:
 * K is cut into segments of 16 blocks; inside a segment the blocks with
 * b % 4 == j form four running sums (fp32 fused multiply-add, in increasing
 * b, starting from +0), combined as (s0 + s1) + (s2 + s3); the segment
 * results are then added in increasing segment order.  So a token's outputs
 * are bit-identical whether it runs alone or with up to 7 others (minfer
 * M16), and the argmax of every entry point agrees with the argmax of its
 * own y.
 *
 * Data layouts (all little-endian, all in device memory unless stated):
 *   W, QGEMV_W_GGML   : GGML row-major Q4_0, [N][K/32] blocks of 18 bytes.
 *   W, QGEMV_W_PACKED : the same bytes re-laid out by qgemv_pack_q4_0
 *                       (same byte count, 18*N*K/32).  Rows are grouped in
 *                       slabs of 16; a slab holds K/32 blocks for 16 rows in
 *                       "quads" of up to 4 blocks: first the 16 rows x 4
 *                       blocks of nibble bytes (row-major, 16 bytes each;
 *                       in a full quad, block jq of row r sits in chunk
 *                       (jq + r/2) mod 4 of its row), then their fp16 scales
 *                       ([row r8 < 8][block][r8, r8+8]).
 *                       The last N % 16 rows stay in GGML layout after the
 *                       slabs.
 *   xq (Q8_0, planar) : for R rows of K values, R*K int8 values ([r][k]),
 *                       then R*K/32 fp16 scales ([r][b]), then zero padding
 *                       to a multiple of 16 bytes: qgemv_xq_bytes(R, K).
 *   x                 : fp32 [T][K] (token-major).
 *   y                 : fp32 [T][N] (token-major).
 *
 * Ownership and errors.  The caller owns every buffer.  The library never
 * allocates, frees or synchronises in these calls: every call only validates
 * its arguments on the host and enqueues kernels on the given stream, so
 * results are ready in stream order.  Invalid arguments return an error
 * before anything is enqueued.  A launch failure returns QGEMV_ERR_CUDA.  A
 * kernel that waits too long on one of its own asynchronous copies gives up,
 * records QGEMV_ERR_TIMEOUT in a per-device status word (see
 * qgemv_device_status) and returns; its outputs are then undefined.  No C++
 * exception crosses the ABI.  Calls are thread-safe; two calls that share a
 * workspace must not overlap on the GPU.
 *
 * Launch order.  The GEMV calls launch with programmatic dependent launch:
 * a GEMV kernel may start, and read the weights W, while the preceding
 * kernel in the stream is still running, if that kernel allows it
 * (griddepcontrol.launch_dependents); activations, outputs, workspace and a
 * gather's expert ids (and so the weights a gather reads) are touched only
 * after the preceding kernel has completed.  So W must not be written by a preceding kernel that allows
 * early launch before its writes are done (the library's own kernels that
 * allow it never write weights).
 *
 * Workspace.  Calls that take (ws, ws_bytes) use it for split-K partial
 * sums, completion counters and argmax candidates.  The matching
 * *_workspace_bytes query gives the size (device-independent, at least 16
 * KB).  Its first 16 KB hold completion counters (and, in their last 64
 * bytes, the argmax's running maxima) and must be zero-filled once before
 * the first use
 * (e.g. cudaMemsetAsync); every call that completes without a device-status
 * error leaves them at zero again, so a workspace can be reused directly,
 * by calls of any kind and shape, as long as it is large enough.
 *
 * Alignment: W, xq and ws 16 bytes; x and y 4 bytes; strides accordingly.
 * Limits: K % 32 == 0; 1 <= T <= 8 for the GEMV calls; 1 <= N < 2^31.
 */
#ifndef QGEMV_H
#define QGEMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle (identical to cudaStream_t); NULL is the legacy
 * default stream. */
struct CUstream_st;
typedef struct CUstream_st *qgemv_stream_t;

typedef enum {
    QGEMV_OK = 0,
    QGEMV_ERR_INVALID_ARG = 1, /* null pointer, bad size, overlap, T out of range */
    QGEMV_ERR_MISALIGNED = 2,  /* a pointer or stride breaks the alignment rules */
    QGEMV_ERR_UNSUPPORTED = 3, /* a shape the kernels do not cover (T*K too large) */
    QGEMV_ERR_WORKSPACE = 4,   /* ws is NULL or smaller than the query says */
    QGEMV_ERR_CUDA = 5,        /* a CUDA runtime call failed (launch, attribute) */
    QGEMV_ERR_TIMEOUT = 6,     /* reported through qgemv_device_status only */
    QGEMV_ERR_BAD_ID = 7,      /* gather: an expert id outside [0, n_experts) */
    QGEMV_ERR_INTERNAL = 8
} qgemv_status;

typedef enum { QGEMV_W_GGML = 0, QGEMV_W_PACKED = 1 } qgemv_wlayout;

/* Human-readable name of a status code (static string). */
const char *qgemv_status_string(qgemv_status s);

/* Library version as 10000*major + 100*minor + patch. */
int qgemv_version(void);

/* Bytes of an N x K Q4_0 matrix in either layout: 18 * N * K / 32.
 * Returns 0 for an invalid shape. */
size_t qgemv_q4_0_bytes(int64_t N, int64_t K);

/* Bytes of a planar Q8_0 buffer for R rows of K: R*K + roundup16(2*R*K/32).
 * Returns 0 for an invalid shape. */
size_t qgemv_xq_bytes(int R, int64_t K);

/* Re-lay out an N x K GGML Q4_0 matrix into the packed device layout (a
 * byte permutation, so the result has the same size).  Done once at load
 * time; minfer README M15 repacks weights at load into row groups so that a
 * warp reads contiguous bytes.  w_ggml and w_packed are device buffers of
 * qgemv_q4_0_bytes(N, K) bytes that must not overlap; w_packed must be
 * 16-byte aligned. */
qgemv_status qgemv_pack_q4_0(const void *w_ggml, void *w_packed, int64_t N, int64_t K,
                             qgemv_stream_t stream);

/* Inverse of qgemv_pack_q4_0 (w_packed 16-byte aligned). */
qgemv_status qgemv_unpack_q4_0(const void *w_packed, void *w_ggml, int64_t N, int64_t K,
                               qgemv_stream_t stream);

/* Quantise fp32 activations to planar Q8_0 (block rule above; minfer README
 * "How it works": int8 activations; colibri qwen36 docs, dense int8 IDOT
 * GEMV: scale amax/127).  x is [batch][R][K] fp32; xq receives `batch`
 * consecutive planar buffers of qgemv_xq_bytes(R, K) bytes each.  R >= 1
 * rows (not limited to 8), batch >= 1.  xq must be 16-byte aligned. */
qgemv_status qgemv_quantize_q8_0(const float *x, void *xq, int R, int64_t K, int batch,
                                 qgemv_stream_t stream);

/* Workspace bytes for qgemv_q4_0, qgemv_q4_0_f32, qgemv_q4_0_argmax and
 * qgemv_q4_0_argmax_f32 on an N x K matrix with T tokens (0 for an invalid
 * shape). */
size_t qgemv_workspace_bytes(int64_t N, int64_t K, int T);

/* y[T][N] = W . x for T pre-quantised token columns (xq, planar Q8_0 of T
 * rows).  Weights are streamed once from HBM (minfer README, M15: decode is
 * bandwidth / bytes per token). */
qgemv_status qgemv_q4_0(const void *W, qgemv_wlayout layout, const void *xq, float *y,
                        int64_t N, int64_t K, int T, void *ws, size_t ws_bytes,
                        qgemv_stream_t stream);

/* Same as qgemv_q4_0 with fp32 input x[T][K] (4-byte aligned): the GEMV
 * kernel quantises the activations itself (Q8_0, the same bytes as
 * qgemv_quantize_q8_0) while it builds its shared-memory copy of them; one
 * launch, which streams weights before it reads x. */
qgemv_status qgemv_q4_0_f32(const void *W, qgemv_wlayout layout, const float *x, float *y,
                            int64_t N, int64_t K, int T, void *ws, size_t ws_bytes,
                            qgemv_stream_t stream);

/* lm_head GEMV with fused argmax (minfer README "How it works": device-side
 * argmax; M19: per-CTA candidates merged associatively).  idx[t] (int64,
 * device) receives, per token, the lowest row index whose output is maximal
 * (equality by IEEE ==, so -0 equals +0).  y_or_null, when not NULL,
 * receives the full y[T][N] exactly as qgemv_q4_0 would write it. */
qgemv_status qgemv_q4_0_argmax(const void *W, qgemv_wlayout layout, const void *xq,
                               float *y_or_null, int64_t *idx, int64_t N, int64_t K, int T,
                               void *ws, size_t ws_bytes, qgemv_stream_t stream);

/* qgemv_q4_0_argmax with fp32 input x[T][K] (4-byte aligned), quantised
 * inside the kernel as in qgemv_q4_0_f32: one launch for the lm_head of a
 * decode step.  Same workspace as qgemv_q4_0_argmax. */
qgemv_status qgemv_q4_0_argmax_f32(const void *W, qgemv_wlayout layout, const float *x, float *y_or_null,
                                   int64_t *idx, int64_t N, int64_t K, int T, void *ws, size_t ws_bytes,
                                   qgemv_stream_t stream);

/* lm_head GEMV with the two best rows per token (minfer README M19: the
 * step keeps each token's top-2 margin; top-2 merging is associative, so the
 * result does not depend on the merge order).  idx2 (int64 [T][2], device)
 * and val2 (fp32 [T][2], device) receive, per token t:
 *   idx2[t][0], val2[t][0]: the row qgemv_q4_0_argmax returns, and its output;
 *   idx2[t][1], val2[t][1]: the argmax of the other rows (lowest index among
 *     equal outputs, -0 == +0), and its output;
 * so val2[t][0] - val2[t][1] >= 0 is the token's margin.  Values are y's
 * exactly, except that -0 is returned as +0.  With N == 1 the second row is
 * -1 and its value -infinity.  y_or_null as in qgemv_q4_0_argmax.  idx2 and
 * val2 must not overlap each other, y or the workspace.  Workspace: as
 * qgemv_q4_0_argmax (qgemv_workspace_bytes). */
qgemv_status qgemv_q4_0_top2(const void *W, qgemv_wlayout layout, const void *xq,
                             float *y_or_null, int64_t *idx2, float *val2, int64_t N, int64_t K,
                             int T, void *ws, size_t ws_bytes, qgemv_stream_t stream);

/* qgemv_q4_0_top2 with fp32 input x[T][K] (4-byte aligned), quantised inside
 * the kernel: one launch for the lm_head of a verify step. */
qgemv_status qgemv_q4_0_top2_f32(const void *W, qgemv_wlayout layout, const float *x,
                                 float *y_or_null, int64_t *idx2, float *val2, int64_t N,
                                 int64_t K, int T, void *ws, size_t ws_bytes,
                                 qgemv_stream_t stream);

/* ---- Q8_0 weights: a second weight format on the same path (minfer README
 * "How it works": gemv_q8_dp4a, int8 weights with int8 activations; M14: the
 * lm_head held as Q8_0).  A weight block is 34 bytes, fp16 d then 32 int8 q,
 * and the weight is q * d.  GGML layout: row-major [N][K/32] blocks. */

/* One-time repack of a GGML Q8_0 matrix into the device layout (same byte
 * count, 34 * N * K/32): 16-row slabs of 8-block stages, each row's 16-byte
 * chunks of codes placed so that the GEMV's lanes read conflict-free, then the
 * stage's fp16 scales; the N % 16 tail rows stay in GGML layout after the
 * slabs.  w_packed 16-byte aligned, not overlapping w_ggml.  The inverse is
 * qgemv_unpack_q8_0. */
qgemv_status qgemv_pack_q8_0(const void *w_ggml, void *w_packed, int64_t N, int64_t K,
                             qgemv_stream_t stream);
qgemv_status qgemv_unpack_q8_0(const void *w_packed, void *w_ggml, int64_t N, int64_t K,
                               qgemv_stream_t stream);

/* ---- Requantisation to Q4_0 at load (minfer README M14: the lm_head
 * requantised from Q8_0 to q4_0, 248 MB to 131 MB; M18: Q8_0 heads
 * requantised to q4_0 when the model loads).  The pages give no encoder;
 * these use GGML's q4_0 encoder, per block of 32 values x:
 *   m = the first element of largest |x| (+0 for a block of zeros),
 *   d = m / -8 in fp32 (m is code 0), id = 1/d (0 when d = 0),
 *   code_j = min(15, floor(x_j * id + 8.5)), multiply and add each rounded
 *   to nearest even; d stored as fp16 (round to nearest even).
 * Output: GGML Q4_0 blocks [N][K/32][18] (pack with qgemv_pack_q4_0 for the
 * GEMV).  A block whose d is an fp32 subnormal (1/d overflows) gets codes
 * 0 for x < 0, 15 for x > 0 and 0 for x = 0.  Values must be finite: a
 * block holding an inf or NaN gets unspecified bytes.  Inputs are not modified; output must not overlap them.
 * Enqueued on `stream`, no synchronisation. */

/* fp32 w[N][K] (row-major, 4-byte aligned) -> Q4_0 (2-byte aligned). */
qgemv_status qgemv_requant_f32_q4_0(const float *w, void *w_q4, int64_t N, int64_t K,
                                    qgemv_stream_t stream);
/* GGML Q8_0 weight blocks [N][K/32][34] (2-byte aligned; values q * d,
 * exact in fp32) -> Q4_0 (2-byte aligned). */
qgemv_status qgemv_requant_q8_0_q4_0(const void *w_q8, void *w_q4, int64_t N, int64_t K,
                                     qgemv_stream_t stream);

/* Workspace bytes for qgemv_q8_0 (0 when the launch needs none; 0 also for
 * an invalid shape). */
size_t qgemv_q8_0_workspace_bytes(int64_t N, int64_t K, int T);

/* y[T][N] = W . x for packed Q8_0 weights W and planar Q8_0 activations xq
 * (T rows, as qgemv_quantize_q8_0 writes them).  Per block the int32 sum
 * sum w q is exact; (d_w d_x) isum is accumulated in fp32 in a fixed order that
 * depends on K only: per row, the blocks of each 8-block stage in two
 * interleaved halves (even, odd blocks) summed in increasing order from +0,
 * the halves added, then the stage sums added in order.  Outputs are
 * bit-identical for every T and launch shape.  W, xq 16-byte aligned; y
 * 4-byte aligned and not overlapping W, xq or ws.  Returns
 * QGEMV_ERR_UNSUPPORTED when T * K activation bytes (plus their scales and
 * one weight stage per warp) exceed shared memory (about T * K <= 150000),
 * QGEMV_ERR_WORKSPACE when ws is smaller than qgemv_q8_0_workspace_bytes.
 * The workspace must be zero-filled before its first use and is left zeroed. */
qgemv_status qgemv_q8_0(const void *W, const void *xq, float *y, int64_t N, int64_t K, int T,
                        void *ws, size_t ws_bytes, qgemv_stream_t stream);

/* ---- Grouped int4 weights with per-vector int8 activations (colibri
 * qwen36 docs: the gs64 container, one scale per group of 64 weights, its
 * nibbles repacked once into a planar layout where one AND gives a group's
 * first 32 elements in order and one shift the other 32; the dense int8 IDOT
 * GEMV: the activation quantised to int8 once per call with one scale
 * amax / 127, the integer sums exact and scaled afterwards).
 * Row planes (host or device, the container's form):
 *   wq     [N][K/64][32] bytes: byte j of a group holds element j (low
 *          nibble) and element j + 32 (high nibble); weight = (n - 8) * s;
 *   wscale [N][K/64] fp32: the groups' scales s.
 * Activations: q int8 [T][K] and one fp32 scale s_x per token row.
 * Output: y[t][i] = s_x[t] * sum_g s[i][g] * isum, isum the exact int32 sum
 * over the group, accumulated in fp32 in a fixed order that depends on K
 * only: per stage of 8 groups the even and the odd groups each summed in
 * increasing order from +0 (one fused multiply-add of s * (16 isum) per
 * group), the two added, the stage sums added in order, the total times
 * 1/16, then times s_x; bit-identical for every T and launch shape.
 * K % 64 == 0. */

/* Bytes of the packed layout: 36 * N * K / 64 (0 for an invalid shape). */
size_t qgemv_gs64_bytes(int64_t N, int64_t K);

/* One-time repack of the row planes (device buffers) into the device layout:
 * 16-row slabs of 8-group stages (4608 bytes), each row's 16-byte nibble
 * chunks placed so the GEMV's lanes read shared memory conflict-free, then
 * the stage's scales; the N % 16 tail rows follow, each as its nibbles then
 * its scales.  wscale 4-byte aligned, w_packed 16-byte aligned (not
 * overlapping the planes).  qgemv_unpack_gs64 is the inverse. */
qgemv_status qgemv_pack_gs64(const void *wq, const float *wscale, void *w_packed, int64_t N, int64_t K,
                             qgemv_stream_t stream);
qgemv_status qgemv_unpack_gs64(const void *w_packed, void *wq, float *wscale, int64_t N, int64_t K,
                               qgemv_stream_t stream);

/* Per-vector int8 quantisation of R rows x[R][K] (fp32, 4-byte aligned):
 * s[r] = amax / 127 over the whole row (fp32 IEEE division), 1/s from it
 * (0 when amax = 0), q[r][k] = round-half-away(x * (1/s)) as int8.  One
 * launch; q, s device buffers not overlapping x. */
qgemv_status qgemv_quantize_vec_i8(const float *x, int8_t *q, float *s, int R, int64_t K, qgemv_stream_t stream);

/* Workspace bytes for qgemv_gs64 (0 when the launch needs none; 0 also for
 * an invalid shape).  Zero-filled before its first use, left zeroed. */
size_t qgemv_gs64_workspace_bytes(int64_t N, int64_t K, int T);

/* y[T][N] = W . x for packed gs64 weights W (16-byte aligned), activation
 * codes q [T][K] (16-byte aligned) and scales s [T] (4-byte aligned); y
 * 4-byte aligned, not overlapping W, q, s or ws.  Returns
 * QGEMV_ERR_UNSUPPORTED when the T * K codes do not fit shared memory beside
 * one weight stage per warp (about T * K <= 200000), QGEMV_ERR_WORKSPACE when
 * ws is smaller than qgemv_gs64_workspace_bytes. */
qgemv_status qgemv_gs64(const void *W, const int8_t *q, const float *s, float *y, int64_t N, int64_t K, int T,
                        void *ws, size_t ws_bytes, qgemv_stream_t stream);

/* The same GEMV on fp32 activations x [T][K] (4-byte aligned), quantised
 * inside the launch with qgemv_quantize_vec_i8's steps (each CTA forms the
 * row maxima and the codes itself): y is bit-identical to
 * qgemv_quantize_vec_i8 followed by qgemv_gs64, in one launch.  Workspace,
 * limits and errors as qgemv_gs64; y must not overlap W, x or ws. */
qgemv_status qgemv_gs64_f32(const void *W, const float *x, float *y, int64_t N, int64_t K, int T, void *ws,
                            size_t ws_bytes, qgemv_stream_t stream);

/* ---- The FFN of a decode step (minfer README M15: the whole layer runs
 * around its GEMVs; colibri qwen36 docs: gate and up share one pass over the
 * activation):  y = W_down . Q8_0(SiLU(W_gate . x) * (W_up . x)).
 * On packed weights with T <= 4 (d_model % 16 == 0, d_ff % 32 == 0) one
 * cooperative launch runs all three steps (see qgemv_set_ffn_fused): it
 * streams gate and up, writes h's Q8_0 codes, waits (bounded) until every
 * CTA's share of h is written, and reduces the down projection, whose
 * weights it has streamed meanwhile; otherwise three launches on `stream`,
 * chained by programmatic dependent launch:
 *   1. gate and up, one sequence launch over the same fp32 x[T][d_model]
 *      (quantised inside the kernel; outputs g, u fp32 [T][d_ff] in ws);
 *   2. h = SiLU(g) * u with SiLU(g) = g / (1 + exp(-g)), exp by Cody and
 *      Waite's method (split ln 2, Taylor series to r^7/7!, exact 2^k), every
 *      step an fp32 operation rounded to nearest in a fixed order; h is
 *      quantised to planar Q8_0 exactly as qgemv_quantize_q8_0 would;
 *   3. the down projection (d_model x d_ff) on those codes into y[T][d_model].
 * W_gate, W_up: d_ff x d_model; W_down: d_model x d_ff; all in `layout`.
 * ws: qgemv_ffn_workspace_bytes(d_model, d_ff, T) bytes, 256-byte aligned,
 * zero-filled before its first use (left so).  y must not overlap x, W_down
 * or ws. */
size_t qgemv_ffn_workspace_bytes(int64_t d_model, int64_t d_ff, int T);
qgemv_status qgemv_q4_0_ffn(const void *W_gate, const void *W_up, const void *W_down, qgemv_wlayout layout,
                            const float *x, float *y, int64_t d_model, int64_t d_ff, int T,
                            void *ws, size_t ws_bytes, qgemv_stream_t stream);

/* The same chain with a residual added to the down projection's output
 * (the decode step's FFN block: y = residual + W_down . h; minfer README
 * M19).  The down launch is a one-item sequence with the residual epilogue:
 * y = (W_down . h) + residual[t][i], one fp32 add after the same GEMV bits.
 * residual [T][d_model] fp32, 4-byte aligned; it may be y itself, and must
 * otherwise not overlap y or the workspace.  The workspace is
 * qgemv_ffn_workspace_bytes, as for qgemv_q4_0_ffn. */
qgemv_status qgemv_q4_0_ffn_residual(const void *W_gate, const void *W_up, const void *W_down,
                                     qgemv_wlayout layout, const float *x, const float *residual, float *y,
                                     int64_t d_model, int64_t d_ff, int T, void *ws, size_t ws_bytes,
                                     qgemv_stream_t stream);

/* Test hook: step 2 of qgemv_q4_0_ffn alone.  g, u fp32 [T][F]; hq receives
 * T rows of F int8 codes then the [T][F/32] fp16 scales (16-byte aligned,
 * qgemv_xq_bytes(T, F) bytes). */
qgemv_status qgemv_debug_silu_mul_q8(const float *g, const float *u, void *hq, int T, int64_t F,
                                     qgemv_stream_t stream);

/* A whole verify step in one launch: qgemv_q4_0_top2_f32 (without logits)
 * followed by the verify rule on its first rows, applied by the kernel's
 * last CTA after the final merge: *n_commit receives what
 * qgemv_verify_commit(tokens, idx2, 2, T, n_commit) would write.  tokens
 * (int64 [T], device) as in qgemv_verify_commit; n_commit (int32, device)
 * must not overlap the other buffers. */
qgemv_status qgemv_q4_0_verify_f32(const void *W, qgemv_wlayout layout, const float *x,
                                   const int64_t *tokens, int64_t *idx2, float *val2,
                                   int32_t *n_commit, int64_t N, int64_t K, int T, void *ws,
                                   size_t ws_bytes, qgemv_stream_t stream);

/* The lossless verify rule of speculative greedy decoding (minfer README
 * M17: a verify step runs [current, draft_1..draft_K] and commits up to and
 * including the first prediction that disagrees with its draft).
 * tokens (int64 [T], device): tokens[0] is the step's current token,
 * tokens[1..T-1] its drafts; pred (int64, device): pred[t * pred_stride]
 * is the greedy prediction after tokens[0..t] (pred_stride 1 for idx from
 * qgemv_q4_0_argmax, 2 for the first rows of qgemv_q4_0_top2's idx2).  Writes to *n_commit (int32, device) the number of committed
 * predictions, 1 + the length of the leading run of t with
 * tokens[t + 1] == pred[t]; the committed tokens are pred[0..n-1].
 * 1 <= T <= 32.  One single-warp launch on `stream`; no workspace. */
qgemv_status qgemv_verify_commit(const int64_t *tokens, const int64_t *pred, int pred_stride,
                                 int T, int32_t *n_commit, qgemv_stream_t stream);

/* Allocation-free variant of qgemv_q4_0_argmax (the paper has no
 * counterpart; this is a convenience of this library).  For callers that
 * cannot allocate device memory where they run the lm_head -- a plugin that
 * only receives its input and output tensors, a runtime with a fixed memory
 * budget, or code inside a region where allocation is not allowed -- it
 * takes no workspace: its scratch is one 4 MiB array in the library's own
 * device memory, held by every GPU that loads the library until the process
 * exits.  Arguments and results are those of qgemv_q4_0_argmax.
 *   - Shapes with qgemv_workspace_bytes(N, K, T) > 4 MiB return
 *     QGEMV_ERR_UNSUPPORTED.
 *   - Every argument is checked before any CUDA call: a refused call
 *     enqueues nothing.
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current) and keeps it for the life of the
 *     process; make that first call before any stream capture, and do not
 *     use the call after a cudaDeviceReset of that device (the array then
 *     moves, and the kept address is stale).
 *   - Every call shares the array and clears its counters at the start (an
 *     asynchronous memset on `stream`); calls that overlap on the GPU, from
 *     any stream or thread, race and give undefined results.
 *   - It allocates and frees nothing. */
qgemv_status qgemv_q4_0_argmax_noalloc(const void *W, qgemv_wlayout layout, const void *xq,
                                       float *y_or_null, int64_t *idx, int64_t N, int64_t K, int T,
                                       qgemv_stream_t stream);

/* One GEMV of a sequence (layer set): weights, planar Q8_0 activations of
 * T rows, and output y[T][N]. */
typedef struct {
    const void *W;
    const void *xq;
    float *y;
    int64_t N;
    int64_t K;
} qgemv_seq_item;

/* Workspace bytes for qgemv_q4_0_seq on this list (0 if invalid).  From
 * T = 5 on (tensor-core path) this includes one region of segment sums per
 * CTA of this device, which lets all warps of a CTA share a matrix piece of
 * fewer slabs than warps; a workspace with fewer regions (down to the 16 KB
 * counter area that an unsplit list needs) gives the same bits, more slowly. */
size_t qgemv_seq_workspace_bytes(const qgemv_seq_item *items, int n, int T);

/* Run n GEMVs (host array `items`, read during the call only) in list order
 * in one persistent launch per 200 items (minfer README M15: one persistent
 * kernel streams every matrix of the token and keeps DRAM busy).  Every
 * item's inputs must be ready when the call is enqueued: no item may read
 * another item's y.  All items share T and the layout. */
qgemv_status qgemv_q4_0_seq(const qgemv_seq_item *items, int n, qgemv_wlayout layout, int T,
                            void *ws, size_t ws_bytes, qgemv_stream_t stream);

/* One GEMV of a sequence with fp32 input x[T][K]. */
typedef struct {
    const void *W;
    const float *x;
    float *y;
    int64_t N;
    int64_t K;
} qgemv_seq_f32_item;

/* ---- Sequences with an output epilogue (minfer README M19: the QKV bias
 * and the residual adds are the GEMVs' epilogues in the pages' decode step):
 *   y[t][i] = (W.x[t])[i] + bias[i] + residual[t][i]
 * with the GEMV value computed exactly as by qgemv_q4_0_seq (the same bits),
 * then the two fp32 adds, each rounded to nearest, in that order; either
 * term may be NULL.  x is planar Q8_0 (x_f32 = 0) or fp32 [T][K] quantised
 * inside the kernel (x_f32 = 1).  bias [N] and residual [T][N] are 4-byte
 * aligned inputs; residual may be y itself (y += W.x + bias in place) but
 * must not otherwise overlap any output. */
typedef struct {
    const void *W;
    const void *x;
    float *y;
    int64_t N;
    int64_t K;
    const float *bias;
    const float *residual;
} qgemv_seq_ep_item;

/* Workspace bytes for qgemv_q4_0_seq_ep on this list (0 if invalid). */
size_t qgemv_seq_ep_workspace_bytes(const qgemv_seq_ep_item *items, int n, int T, int x_f32);
qgemv_status qgemv_q4_0_seq_ep(const qgemv_seq_ep_item *items, int n, qgemv_wlayout layout, int T, int x_f32,
                               void *ws, size_t ws_bytes, qgemv_stream_t stream);

/* Workspace bytes for qgemv_q4_0_seq_f32 on this list (0 if invalid). */
size_t qgemv_seq_f32_workspace_bytes(const qgemv_seq_f32_item *items, int n, int T);

/* qgemv_q4_0_seq with fp32 inputs x[T][K] (4-byte aligned): the GEMV kernel
 * quantises each item's activations (Q8_0, the same bytes as
 * qgemv_quantize_q8_0) while it builds its shared-memory copy of them, so a
 * sequence is one launch per 200 items, streaming weights before it reads x
 * (minfer README M15: the activation is quantised once, then the weights
 * stream).  The workspace is the sequence's own (no activation area). */
qgemv_status qgemv_q4_0_seq_f32(const qgemv_seq_f32_item *items, int n, qgemv_wlayout layout, int T,
                                void *ws, size_t ws_bytes, qgemv_stream_t stream);

/* One matrix of a routed-expert (MoE) gather: expert e's copy of this
 * matrix starts at W + e * expert_stride (bytes); slot s reads activations
 * xq + s * xq_stride (bytes; 0 = shared by all slots) and writes
 * y + s * y_stride (floats). */
typedef struct {
    const void *W;
    int64_t expert_stride;
    const void *xq;
    int64_t xq_stride;
    float *y;
    int64_t y_stride;
    int64_t N;
    int64_t K;
} qgemv_gather_matrix;

/* Workspace bytes for qgemv_q4_0_gather (0 if invalid). */
size_t qgemv_gather_workspace_bytes(const qgemv_gather_matrix *mats, int n_mats, int n_ids, int T);

/* Routed-expert GEMV (colibri qwen36 docs: 256 experts, top-8 + 1 shared;
 * only the selected experts' bytes are streamed).  For every slot
 * s < n_ids and every matrix m: y_m[s] = W_m[ids[s]] . xq_m[s].  ids is a
 * device int32 array; an id outside [0, n_experts) is not read from: its
 * outputs are left untouched and the device status word records
 * QGEMV_ERR_BAD_ID.  One launch covers all matrices and slots (n_mats <= 4). */
qgemv_status qgemv_q4_0_gather(const qgemv_gather_matrix *mats, int n_mats, const int32_t *ids,
                               int n_ids, int n_experts, qgemv_wlayout layout, int T, void *ws,
                               size_t ws_bytes, qgemv_stream_t stream);

/* A gather matrix with fp32 activations: slot s reads x + s * x_stride
 * (bytes; 0 = shared by all slots), fp32 [T][K], 4-byte aligned. */
typedef struct {
    const void *W;
    int64_t expert_stride;
    const float *x;
    int64_t x_stride;
    float *y;
    int64_t y_stride;
    int64_t N;
    int64_t K;
} qgemv_gather_f32_matrix;

/* Workspace bytes for qgemv_q4_0_gather_f32 (0 if invalid). */
size_t qgemv_gather_f32_workspace_bytes(const qgemv_gather_f32_matrix *mats, int n_mats, int n_ids, int T);

/* qgemv_q4_0_gather with fp32 activations, quantised inside the kernel (the
 * same bytes as qgemv_quantize_q8_0): a routed-expert step is one launch. */
qgemv_status qgemv_q4_0_gather_f32(const qgemv_gather_f32_matrix *mats, int n_mats, const int32_t *ids,
                                   int n_ids, int n_experts, qgemv_wlayout layout, int T, void *ws,
                                   size_t ws_bytes, qgemv_stream_t stream);

/* Test hook: the exact per-block integer sums the GEMV kernels form,
 * isums[T][N][K/32] int32 (device), from the same unpack / int8-dot code. */
qgemv_status qgemv_debug_block_isums(const void *W, qgemv_wlayout layout, const void *xq,
                                     int32_t *isums, int64_t N, int64_t K, int T,
                                     qgemv_stream_t stream);

/* Test hook: the same sums as the tensor-core (MMA) path forms them (minfer
 * README M16: the batched path and the one-token path form identical
 * per-block integer sums).  Per 16 rows and block, the nibbles enter two
 * f16 MMAs as subnormal operands and the activations as q and q / 16,
 * converted as the GEMV kernel converts them: f16_image = 1 from the f16
 * operand words of small activation images, 0 from the int8 image's
 * biased bytes; the accumulator starts from the folded offset -8 sum(q) and
 * ends at isum * 2^-24, which the hook writes as int32.  Arguments and
 * output layout as qgemv_debug_block_isums. */
qgemv_status qgemv_debug_block_isums_tc(const void *W, qgemv_wlayout layout, const void *xq, int32_t *isums,
                                        int64_t N, int64_t K, int T, int f16_image, qgemv_stream_t stream);

/* Measurement hook: stream `bytes` of device memory from `src` once, with
 * no arithmetic, to measure the HBM read bandwidth an access pattern
 * reaches (minfer README M15: bench/roofline.cu).  method 0: one CTA per SM
 * of `warps` warps, each keeping `depth` 1-D bulk copies of `stage_bytes` in
 * flight into shared memory (the GEMV kernel's pattern); method 1: 128-bit
 * global loads, `warps` warps per CTA, two CTAs per SM, 4 (depth <= 4) or 8
 * loads in flight per thread.  `sink` (8 bytes, device) is written only in
 * a case that never occurs, so the loads stay live. */
qgemv_status qgemv_debug_stream_read(const void *src, size_t bytes, int method, int warps, int depth,
                                     int stage_bytes, unsigned long long *sink, qgemv_stream_t stream);

/* Tuning of the streaming kernel (0 restores the default for any of them;
 * results never depend on it -- the summation order is fixed by K):
 *   ctas_per_sm: CTAs resident per SM (1 = one CTA of up to 16 warps;
 *                2 = two CTAs of 8 warps), waves: CTAs per SM slot in one
 *                launch, mma_min_T: token count from which T > 1 runs on the
 *                f16 tensor-core path (mma.sync m16n8k16 over exact
 *                integer operands; default 5, 9 = never) instead of dp4a,
 *   ring_depth:  weight stages in flight per warp (1..6; default 3 for
 *                one-token sequences, else 2), used where the activations
 *                leave room.
 * Process-wide; affects launches enqueued afterwards. */
qgemv_status qgemv_set_tuning(int ctas_per_sm, int waves, int mma_min_T, int ring_depth);

/* qgemv_q4_0_ffn and qgemv_q4_0_ffn_residual as one fused launch (on = 1,
 * the default) where it applies -- packed weights, T <= 4, d_model % 16 ==
 * 0, d_ff % 32 == 0 -- or always as the three launches (on = 0).  Results
 * do not change (the same steps in the same order).  Process-wide. */
qgemv_status qgemv_set_ffn_fused(int on);

/* Token count from which packed sequences (qgemv_q4_0_seq, _seq_f32)
 * run on the tcgen05 tensor-core kernel (1..8; 9 = never, the default; 0
 * restores the default).  The kernel is off by default because the
 * mma.sync path measures faster on GB300 at every T.  It applies to launches without epilogues whose matrices all
 * have N % 16 == 0 and K % 256 == 0 and whose workspace is as large as
 * qgemv_seq_workspace_bytes (or _seq_f32_) returns while it is enabled;
 * other launches keep the other kernels.  Results do not change: every path
 * forms the same block sums and adds them in the same order.  fp32 inputs
 * are quantised first, in one launch, into the workspace.  Process-wide. */
qgemv_status qgemv_set_tc_min_tokens(int tc_min_T);

/* Read and clear the current device's status word: QGEMV_OK, or the first
 * asynchronous error a kernel recorded (QGEMV_ERR_TIMEOUT, QGEMV_ERR_BAD_ID)
 * into *code_out.  Synchronises with the device (a query, not part of the
 * hot path).  Returns QGEMV_ERR_CUDA if the device cannot be read. */
qgemv_status qgemv_device_status(int *code_out);

#ifdef __cplusplus
}
#endif

#endif /* QGEMV_H */
