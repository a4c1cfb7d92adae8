// qgemv_launch.h -- internal host-side interface between the C ABI and the
// kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "qgemv_internal.cuh"

namespace qg {

inline long long roundup16(long long v) { return (v + 15) & ~15ll; }

// Planar Q8_0 bytes for R rows of K (see include/qgemv.h).
inline long long xq_bytes_host(long long R, long long K) { return R * K + roundup16(2 * R * (K / QK)); }

cudaError_t launch_quantize(const float *x, void *xq, int R, long long K, int batch, cudaStream_t st);

cudaError_t launch_stream_bench(const void *src, long long bytes, int method, int warps, int depth, int stage_bytes,
                                unsigned long long *out, unsigned *status, int sms, cudaStream_t st);
cudaError_t launch_pack(const void *src, void *dst, long long N, long long K, bool to_packed, cudaStream_t st);
cudaError_t launch_isums(const void *W, bool packed, const void *xq, int32_t *isums, long long N, long long K, int T,
                         cudaStream_t st);
// The tensor-core path's block sums (isums_tc.cu): f16_image selects the
// operands of small activation images (built in f16) or of the int8 image.
cudaError_t launch_isums_tc(const void *W, bool packed, const void *xq, int32_t *isums, long long N, long long K,
                            int T, bool f16_image, cudaStream_t st);
cudaError_t launch_q8_pack(const void *src, void *dst, long long N, long long K, bool to_packed, cudaStream_t st);
// Q8_0-weight GEMV (q8_kernel.cu): plans, and launches when do_launch.
// *ws_need: workspace bytes; *unsupported: 1 the activations do not fit
// shared memory, 2 the workspace is missing or too small (nothing launched).
cudaError_t launch_q8(const void *W, const void *xq, float *y, long long N, long long K, int T, void *ws,
                      long long ws_bytes, bool do_launch, int sms, int smem_budget, unsigned *status,
                      cudaStream_t st, long long *ws_need, int *unsupported);
// gs64 grouped int4 weights with per-vector int8 activations (gs64_kernel.cu):
// the pack between the row planes and the device layout, the per-row
// quantiser, and the GEMV (plans, and launches when do_launch; as launch_q8).
cudaError_t launch_gs64_pack(void *wq, float *wsc, void *packed, long long N, long long K, bool to_packed,
                             cudaStream_t st);
cudaError_t launch_quantize_vec_i8(const float *x, int8_t *q, float *s, int R, long long K, cudaStream_t st);
cudaError_t launch_gs64(const void *W, const int8_t *q, const float *sx, const float *xf, float *y, long long N,
                        long long K, int T, void *ws, long long ws_bytes, bool do_launch, int sms, int smem_budget,
                        unsigned *status, cudaStream_t st, long long *ws_need, int *unsupported);
cudaError_t launch_silu_mul_q8(const float *g, const float *u, void *hq, int T, long long F, bool pdl, cudaStream_t st);
// Requantisation to GGML Q4_0 blocks (kernels_misc.cu): nblocks blocks of
// fp32 [32] (from_q8 false) or GGML Q8_0 (from_q8 true) into 18-byte blocks.
cudaError_t launch_requant_q4_0(const void *src, bool from_q8, void *dst, long long nblocks, cudaStream_t st);
cudaError_t launch_verify_commit(const long long *tokens, const long long *pred, int pred_stride, int T,
                                 int32_t *n_commit, cudaStream_t st);

// The few-token GEMV on tcgen05 tensor cores (gemv_tc.cu): a list of up to
// MAXG_SEQ packed GEMVs with N % 16 == 0 and K % 256 == 0.  Workspace: warp
// arrival counters in its first TC_CNT_BYTES (zero, and left zero), then the
// segment sums of tiles shared by warp groups.
struct TcSpec {
    const void *W;
    const void *xq;  // planar Q8_0 activations of T rows
    float *y;
    long long N, K;
};
constexpr long long TC_CNT_BYTES = 16384;
bool tc_eligible(const TcSpec *s, int n, int T);
long long tc_ws_bytes(const TcSpec *s, int n, int grid);
cudaError_t launch_tc(const TcSpec *s, int n, int T, uint8_t *ws, int grid, unsigned *status, cudaStream_t st);
// Q8_0 quantisation of n activation blocks x[i] (fp32 [T][K[i]]) into planar
// buffers xq[i] (kernels_misc.cu): one launch for a whole sequence, of at
// most max_ctas CTAs of 256 threads (few enough to be resident at once).
cudaError_t launch_quantize_list(const float *const *x, uint8_t *const *xq, const long long *K, int n, int T,
                                 int max_ctas, cudaStream_t st);

// The decode FFN step in one cooperative launch (ffn_fused.cu), T <= 4,
// packed weights, d_model % 16 == 0, d_ff % 32 == 0, one CTA per SM of a
// grid of `grid` CTAs.  cnt: two zeroed counters (left zero); hq: T * d_ff +
// 2 * T * d_ff / 32 bytes.
bool ffn_fused_eligible(long long d_model, long long d_ff, int T);
bool ffn_fused_fits(long long d_model, long long d_ff, int T, int grid, int smem_budget);
cudaError_t launch_ffn_fused(const void *Wg, const void *Wu, const void *Wd, const float *x, const float *res,
                             float *y, long long d_model, long long d_ff, int T, uint8_t *hq, unsigned *cnt, int grid,
                             int smem_budget, unsigned *status, cudaStream_t st);

// The streaming GEMV kernel, one instantiation per (T, parameter-block size,
// argmax, tensor-core path).  Defined in gemv_t<T>.cu.
// EPI: the sequence output epilogue (bias, residual) is compiled in.
template <int T, int MAXG, bool ARGMAX, bool MMA, bool EPI = false>
cudaError_t launch_stream(const Params<MAXG> &P, int grid, size_t smem, cudaStream_t st, bool pdl);

}  // namespace qg
