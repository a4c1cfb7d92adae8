// qgemv_internal.cuh -- shared definitions of libqgemv's kernels and host code.
//
// Arithmetic (minfer README, "The optimization journey", M9 and M15/M16):
//   isum(t,i,b) = sum_j (n_j - 8) q_j  (exact int32), formed with dp4a on the
//   unsigned nibbles and the folded offset -8 * sum_j q_j (M9: "folded -8
//   offset"); y += (d_w * d_x) * isum in fp32, in the fixed order described
//   in include/qgemv.h (it depends on K only, and is the same for every T).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace qg {

constexpr int QK = 32;                // weights per Q4_0 / Q8_0 block
constexpr int Q4_BYTES = 18;          // fp16 scale + 16 nibble bytes
constexpr int SLAB_ROWS = 16;         // rows per packed slab
constexpr int QUAD = 4;               // blocks per quad tile
constexpr int SEG_BLOCKS = 16;        // blocks per summation segment (= one pipeline stage)
constexpr int SLAB_COL_BYTES = SLAB_ROWS * Q4_BYTES;    // 288: one block column of a slab
constexpr int QUAD_BYTES = QUAD * SLAB_COL_BYTES;       // 1152
constexpr int SEG_BYTES = SEG_BLOCKS * SLAB_COL_BYTES;  // 4608
constexpr int NWARPS_MAX = 16;        // consumer warps per CTA (one CTA per SM); 8..16 at run time
constexpr int NTHREADS_MAX = NWARPS_MAX * 32;
constexpr int MAX_RING = 6;           // pipeline stages per warp, upper bound
constexpr int MAX_GRID = 1024;        // argmax candidate slots
constexpr int SPLIT_SLAB_THRESHOLD = 608;  // split K below four slabs per CTA of a 152-SM grid (measured)
constexpr int MAGIC_I = 0x4B400000;   // bits of 12582912.0f = 1.5 * 2^23
constexpr float MAGIC_F = 12582912.0f;

// Status codes written by kernels into the per-device status word.
constexpr unsigned ST_TIMEOUT = 6;
constexpr unsigned ST_BAD_ID = 7;

// One matrix family of a launch: a single GEMV (count = 1), or one matrix
// of a routed-expert gather (count = slots).
struct Group {
    const uint8_t *W;       // instance 0 weights (packed or GGML)
    // The instance strides mean something only in gathers (count > 1 or
    // expert ids); a launch with ParamHead::epilogue set is a sequence of
    // single instances and reads the same words as its epilogue pointers.
    union {
        long long w_stride;  // gathers: bytes between instances (experts)
        const float *bias;   // epilogue launches: bias[N] added to y (or nullptr)
    };
    const uint8_t *xq;      // planar Q8_0 of slot 0
    long long xq_stride;    // bytes between slots (0: shared)
    float *y;               // y[T][N] of slot 0
    union {
        long long y_stride;  // gathers: floats between slots
        const float *res;    // epilogue launches: residual[T][N] added after the bias (or nullptr; may be y)
    };
    int N, K, count, split;
    int nb, nseg, nslabs, tail_rows;  // nslabs: slab items (GGML: ceil(N/16)); tail: packed N%16
    int items_per_inst;               // nslabs * split + (tail_rows > 0)
    int xq_bytes;                     // planar Q8_0 bytes per slot (T rows)
    long long inst_bytes;             // 18 * N * nb
    long long slab_bytes;             // 288 * nb
    long long cost_begin;             // prefix of the launch's weighted bytes (the CTA partition)
    int item_begin;                   // prefix of the launch's items (a launch has < 2^31 items)
    int cost;                         // partition weight of one weight byte, in sixteenths
    unsigned *cnt;                    // split-K arrival counters [count][nslabs]
    float *part;                      // split-K partials [count][nslabs][nseg][T][16]
};

// Scalar launch parameters (copied to shared memory at kernel entry).
struct ParamHead {
    int ngroups;
    int ggml;               // weights in GGML layout (no TMA staging)
    int nwarps;             // warps per CTA (blockDim.x / 32)
    int ring_depth;         // stages per warp
    int kmax, nbmax;        // largest K / blocks per row over the groups
    int off_d, off_cd, off_bar, off_ring;  // dynamic shared-memory layout
    int off_runs, off_hbuf, off_hflag;     //   (balanced-mode tables)
    int off_gcache;                        //   (group descriptors of the CTA's range)
    int xq_area;            // bytes at offset 0 for activations
    int balanced_ok;        // every group unsplit: CTAs may balance by stages
    const int *ids;         // gather: slot -> expert id (nullptr: slot index)
    int n_experts;
    int xf32;               // the groups' activations are fp32 [T][K], quantised in the kernel
    long long total_cost, total_items;  // weighted bytes, items of the launch
    unsigned long long *am_cand;  // argmax: [gridDim][T] candidate keys
    unsigned long long *am_key;   // argmax alone: [T] running maxima (zero between launches)
    unsigned *am_cnt;             // argmax: CTA arrival counter
    long long *am_idx;            // argmax: result [T] (or nullptr)
    long long *am_idx2;           // top-2: rows [T][2] (or nullptr)
    float *am_val2;               // top-2: values [T][2] (with am_idx2)
    int epilogue;                 // groups carry bias / residual pointers (sequences only)
    int part_ovh_kb;              // host partition only: fixed cost of each group instance, in KB of weights
    float *sg_part;               // small groups: per-CTA segment sums (or nullptr)
    int sg_stride;                //   floats per CTA region
    int sg_ctas;                  //   CTAs 0..sg_ctas-1 have a region
    const long long *vc_tokens;   // verify: the step's tokens [T] (or nullptr)
    int *vc_n;                    // verify: committed predictions (with vc_tokens)
    unsigned *status;             // per-device status word
};

template <int MAXG>
struct Params : ParamHead {
    Group g[MAXG];
    unsigned char cta_g0[MAX_GRID + 1];  // group holding the first item of CTA c's range
    int cta_i0[MAX_GRID + 1];            // first item of CTA c's range (cta_i0[grid]: the launch's items)
};

constexpr int MAXG_SMALL = 4;
constexpr int GCACHE_GROUPS = 34;  // launch groups a CTA caches in shared memory (MAX_RUNS + 2)
constexpr int MAXG_SEQ = 200;  // keeps the parameter block under the 32 KB kernel-parameter limit
static_assert(MAXG_SEQ <= 256, "CTA start groups are stored as bytes");
static_assert(sizeof(Params<MAXG_SEQ>) <= 32764, "kernel parameters are limited to 32764 bytes");

// ------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, unsigned bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, unsigned parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// 1-D bulk asynchronous copy global -> own CTA's shared memory, completing
// on an mbarrier (transaction bytes).  dst, src 16-byte aligned; bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, unsigned bytes, uint64_t *bar,
                                         uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Hint: bring [src, src + bytes) into L2 (bytes % 16 == 0, src 16-byte
// aligned); completes on its own, no barrier.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, unsigned bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Programmatic dependent launch: wait for the preceding grid's completion
// and memory flush / allow the next grid to be scheduled early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

// 16 bytes from shared memory (16-byte aligned shared address).
__device__ __forceinline__ uint4 lds128(uint32_t a)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}

// sum of 4 (unsigned byte of a) * (signed byte of b) + c.
__device__ __forceinline__ int dp4a_us(unsigned a, int b, int c)
{
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// sum of 4 (signed byte of a) * (signed byte of b) + c.
__device__ __forceinline__ int dp4a_ss(int a, int b, int c)
{
    int d;
    asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;  // 2 s: far beyond any single copy
constexpr uint64_t DRAIN_LIMIT_NS = 100000000ull;  // 0.1 s per stage when draining after an abort

// Bounded wait on an mbarrier phase.  Gives up after `limit_ns`, raises the
// CTA's abort flag and records ST_TIMEOUT; returns false then (and at once
// when the CTA has already aborted).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, unsigned parity, volatile int *abort_flag,
                                                  unsigned *status, uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (*abort_flag) return false;
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) {
            *abort_flag = 1;
            atomicCAS(status, 0u, ST_TIMEOUT);
            return false;
        }
    }
}

// Wait used only while draining copies after an abort (ignores the flag).
__device__ __forceinline__ void mbar_drain(uint64_t *bar, unsigned parity)
{
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > DRAIN_LIMIT_NS) return;
}

// ------------------------------------------------------------- block arithmetic

__device__ __forceinline__ int roundup16_dev(int v) { return (v + 15) & ~15; }

// Position of block jq's 16 nibble bytes among the nbq chunks of row r in a
// quad tile.  Full quads rotate by r / 2, so that both the one-token lanes
// (16-byte loads of one block, rows r and r + 8) and the tensor-core lanes
// (word j of all four blocks) hit distinct shared-memory banks.
__host__ __device__ __forceinline__ int quad_chunk(int jq, int r, int nbq)
{
    return nbq == QUAD ? ((jq + (r >> 1)) & 3) : jq;
}

// Byte offsets, in the packed layout, of block b of row `row` (a row of a
// full slab): its 16 nibble bytes and its fp16 scale.
__host__ __device__ __forceinline__ void packed_offsets(long long row, int b, int nb, long long &nib_off,
                                                        long long &sc_off)
{
    const long long s = row / SLAB_ROWS;
    const int r = static_cast<int>(row - s * SLAB_ROWS);
    const int q = b / QUAD, jq = b - q * QUAD;
    const int nbq = nb - q * QUAD < QUAD ? nb - q * QUAD : QUAD;
    const long long base = s * static_cast<long long>(SLAB_COL_BYTES) * nb + static_cast<long long>(q) * QUAD_BYTES;
    nib_off = base + (r * nbq + quad_chunk(jq, r, nbq)) * 16;
    sc_off = base + 256 * nbq + ((r % 8) * nbq + jq) * 4 + (r / 8) * 2;
}

// Shared-memory image of one GEMV's activations: T rows of K int8 (rows
// padded on the tensor-core (MMA) path so that the eight token rows fall in
// distinct banks), the fp16 scales as copied, then per block and token the folded
// constant and d_x / 16 ({int, float} pairs, [block][T or 8]).
// Tensor-core path constants per 4 blocks: for each block and token pair p
// the accumulator start {C(2p), C(2p+1), C(2p), C(2p+1)} (4 x 4 x 16 bytes),
// then the fp16 d_x pairs {d_x(2p), d_x(2p+1)} ordered [pair][block] (64 bytes).
constexpr int CD_MMA_QUAD = 320;

// Tensor-core path activation images up to this size hold the B operand
// ready-made in f16 (64 bytes per token and block); larger ones hold the
// int8 activations, converted by each warp as it goes.
constexpr int MMA_F16_IMAGE_MAX = 40960;

struct XqLayout {
    int f16;      // tensor-core path: f16 operand image (else int8)
    int xstride;  // bytes between token rows
    int off_d;    // fp16 scales
    int off_cd;   // folded constants
    int cdw;      // tokens per block in the dp4a constants (T)
    int bytes;    // whole image, 128-byte multiple
};

__host__ __device__ inline XqLayout xq_layout(int T, int K, bool mma)
{
    const int nb = K / QK;
    XqLayout L;
    L.f16 = 0;
    if (mma) {
        // f16 operand rows of 64 bytes per block; a row stride of 16 (mod 128)
        // bytes puts the same block of eight token rows in distinct banks
        const int xs = 64 * nb + ((nb & 1) ? 80 : 16);
        if (static_cast<long long>(T) * xs <= MMA_F16_IMAGE_MAX) {
            L.f16 = 1;
            L.xstride = xs;
            L.off_d = T * xs;  // no fp16 scales: the image is built from global memory
            L.off_cd = L.off_d;
            L.cdw = 8;
            L.bytes = (L.off_cd + CD_MMA_QUAD * ((nb + QUAD - 1) / QUAD) + 127) & ~127;
            return L;
        }
    }
    L.xstride = K;
    if (mma) {
        const int kw = K / 4;                    // words per row
        L.xstride = K + 4 * ((36 - (kw & 31)) & 31);  // words per row = 4 (mod 32)
    }
    L.off_d = T * L.xstride;
    L.off_cd = (L.off_d + 2 * T * nb + 15) & ~15;
    L.cdw = mma ? 8 : T;
    // dp4a: 8 bytes per token and block; MMA: 320 bytes per 4 blocks
    const int cd_bytes = mma ? CD_MMA_QUAD * ((nb + QUAD - 1) / QUAD) : 8 * L.cdw * nb;
    L.bytes = (L.off_cd + cd_bytes + 127) & ~127;
    return L;
}

// Q8_0 steps shared by every quantiser: d = amax / 127 (IEEE division),
// 1/d from the fp32 d (0 when d = 0), q = roundf(x * (1/d)) -- halfway cases
// away from zero -- and d stored as fp16, round to nearest even.
__device__ __forceinline__ void q8_scale(float amax, float &d, float &id)
{
    d = __fdiv_rn(amax, 127.0f);
    id = (d != 0.0f) ? __fdiv_rn(1.0f, d) : 0.0f;
}
__device__ __forceinline__ int q8_code(float v, float id) { return static_cast<int>(roundf(__fmul_rn(v, id))); }
__device__ __forceinline__ unsigned short q8_half(float d) { return __half_as_ushort(__float2half_rn(d)); }

// One block of 32 fp32 activations quantised to Q8_0 by one thread, with the
// warp quantiser's steps (the maximum is exact in any order, so the bytes are
// the same): the codes as two uint4 (elements 0..15, 16..31) and the fp16
// scale.  vec: x is 16-byte aligned.
__device__ __forceinline__ void q8_block_thread(const float *x, bool vec, uint4 &qa, uint4 &qb, unsigned short &dh)
{
    float v[QK];
    if (vec) {
#pragma unroll
        for (int i = 0; i < QK / 4; ++i) {
            const float4 f = __ldcg(reinterpret_cast<const float4 *>(x) + i);
            v[4 * i] = f.x;
            v[4 * i + 1] = f.y;
            v[4 * i + 2] = f.z;
            v[4 * i + 3] = f.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < QK; ++i) v[i] = __ldcg(x + i);
    }
    float amax = fabsf(v[0]);
#pragma unroll
    for (int i = 1; i < QK; ++i) amax = fmaxf(amax, fabsf(v[i]));
    float d, id;
    q8_scale(amax, d, id);
    unsigned w[QK / 4];
#pragma unroll
    for (int k = 0; k < QK / 4; ++k)
        w[k] = (static_cast<unsigned>(q8_code(v[4 * k], id)) & 0xFFu) |
               ((static_cast<unsigned>(q8_code(v[4 * k + 1], id)) & 0xFFu) << 8) |
               ((static_cast<unsigned>(q8_code(v[4 * k + 2], id)) & 0xFFu) << 16) |
               ((static_cast<unsigned>(q8_code(v[4 * k + 3], id)) & 0xFFu) << 24);
    qa = make_uint4(w[0], w[1], w[2], w[3]);
    qb = make_uint4(w[4], w[5], w[6], w[7]);
    dh = q8_half(d);
}


// h = SiLU(g) * u, quantised to planar Q8_0 for the down projection (minfer
// README M15: the FFN between the GEMVs of a decode step).  exp by Cody and
// Waite's method (W. J. Cody, W. Waite, "Software Manual for the Elementary
// Functions", 1980): x = k ln2 + r, k = rint(x log2 e), ln 2 split into a
// head whose products with k are exact and a tail; exp(r) by its Taylor
// series to r^7/7! in Horner form; the exact scale 2^k.  x is clamped to
// [-87, 88].  Every operation is an explicitly rounded fp32 one, in the
// order written, so the values (and so the codes) are a fixed function of
// g and u.
__device__ __forceinline__ float ffn_exp(float x)
{
    x = fminf(fmaxf(x, -87.0f), 88.0f);
    const float k = rintf(__fmul_rn(x, 1.44269504088896340736f));
    float r = __fmaf_rn(-k, 0.693145751953125f, x);   // ln 2 head: 13 significant bits
    r = __fmaf_rn(-k, 1.42860682030941723212e-6f, r);  // ln 2 - head
    float p = 1.0f / 5040.0f;
    p = __fmaf_rn(p, r, 1.0f / 720.0f);
    p = __fmaf_rn(p, r, 1.0f / 120.0f);
    p = __fmaf_rn(p, r, 1.0f / 24.0f);
    p = __fmaf_rn(p, r, 1.0f / 6.0f);
    p = __fmaf_rn(p, r, 0.5f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    return __fmul_rn(p, __int_as_float((static_cast<int>(k) + 127) << 23));
}

__device__ __forceinline__ float ffn_silu(float g) { return __fdiv_rn(g, __fadd_rn(1.0f, ffn_exp(-g))); }

// p[0] + p[stride] + ... + p[(n - 1) stride], added in index order from
// p[0] (the fixed order of a split sum), loaded from L2 B at a time so that
// the loads' latencies overlap instead of adding up.
template <int B = 8>
__device__ __forceinline__ float ordered_sum_ldcg(const float *p, int n, long long stride)
{
    float v = __ldcg(p);
    for (int i = 1; i < n; i += B) {
        float x[B];
#pragma unroll
        for (int k = 0; k < B; ++k) x[k] = i + k < n ? __ldcg(p + (i + k) * stride) : 0.0f;
#pragma unroll
        for (int k = 0; k < B; ++k)
            if (i + k < n) v = __fadd_rn(v, x[k]);
    }
    return v;
}

// fp16 bits -> fp32 (exact).
__device__ __forceinline__ float h2f(unsigned bits16)
{
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16 & 0xFFFFu)));
}

// MAGIC_I + 16 * isum for one weight block and one activation block, where
// c16 = MAGIC_I - 128 * sum(q) (the folded -8 offset, times 16).  n = 4 words
// of nibble bytes (byte k: element k in the low nibble, element k+16 in the
// high nibble); qa = activation elements 0..15, qb = elements 16..31.  The
// low nibbles are masked in place; the high nibbles are masked without a
// shift, so each byte holds 16 * n and that chain sums 16x; the two dp4a
// chains meet in one shift-add.  |16 * isum| <= 520192 < 2^22.
__device__ __forceinline__ int block_dot16_magic(const uint4 &n, const uint4 &qa, const uint4 &qb, int c16)
{
    int lo = 0, hi = c16;
    lo = dp4a_us(n.x & 0x0F0F0F0Fu, (int)qa.x, lo);
    hi = dp4a_us(n.x & 0xF0F0F0F0u, (int)qb.x, hi);
    lo = dp4a_us(n.y & 0x0F0F0F0Fu, (int)qa.y, lo);
    hi = dp4a_us(n.y & 0xF0F0F0F0u, (int)qb.y, hi);
    lo = dp4a_us(n.z & 0x0F0F0F0Fu, (int)qa.z, lo);
    hi = dp4a_us(n.z & 0xF0F0F0F0u, (int)qb.z, hi);
    lo = dp4a_us(n.w & 0x0F0F0F0Fu, (int)qa.w, lo);
    hi = dp4a_us(n.w & 0xF0F0F0F0u, (int)qb.w, hi);
    return (lo << 4) + hi;
}

// The folded-offset constant of one activation block: MAGIC_I - 128 * sum(q).
__device__ __forceinline__ int block_fold16_const(const uint4 &qa, const uint4 &qb)
{
    const int ones = 0x01010101;
    int s = 0;
    s = dp4a_ss((int)qa.x, ones, s);
    s = dp4a_ss((int)qa.y, ones, s);
    s = dp4a_ss((int)qa.z, ones, s);
    s = dp4a_ss((int)qa.w, ones, s);
    s = dp4a_ss((int)qb.x, ones, s);
    s = dp4a_ss((int)qb.y, ones, s);
    s = dp4a_ss((int)qb.z, ones, s);
    s = dp4a_ss((int)qb.w, ones, s);
    return MAGIC_I - 128 * s;
}

// (MAGIC_I + v) read as a float is 12582912 + v exactly for |v| < 2^22;
// subtracting 12582912 gives (float)v exactly.
__device__ __forceinline__ float magic_to_float(int s) { return __fsub_rn(__int_as_float(s), MAGIC_F); }

// Order-preserving 64-bit key for argmax: larger value first, then lower
// row.  -0 is folded onto +0 so IEEE equality decides ties.
__device__ __forceinline__ unsigned long long argmax_key(float v, unsigned row)
{
    if (v == 0.0f) v = 0.0f;
    unsigned u = __float_as_uint(v);
    unsigned k = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return (static_cast<unsigned long long>(k) << 32) | static_cast<unsigned long long>(0xFFFFFFFFu - row);
}

// One 18-byte Q4_0 block in GGML layout (only 2-byte aligned) from global memory.
__device__ __forceinline__ void load_ggml_block(const uint8_t *p, uint4 &nib, unsigned &d)
{
    const unsigned short *h = reinterpret_cast<const unsigned short *>(p);
    d = __ldg(h);
    unsigned w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) w[k] = __ldg(h + 1 + k);
    nib.x = w[0] | (w[1] << 16);
    nib.y = w[2] | (w[3] << 16);
    nib.z = w[4] | (w[5] << 16);
    nib.w = w[6] | (w[7] << 16);
}

}  // namespace qg
