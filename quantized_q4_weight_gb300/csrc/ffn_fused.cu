// ffn_fused.cu -- the decode FFN step in one persistent launch (minfer README
// M15: one persistent kernel runs the layer and keeps DRAM busy; colibri
// qwen36 docs: gate and up share one pass over the activation):
//     y = W_down . Q8_0(SiLU(W_gate . x) * (W_up . x))  [+ residual]
//
// One CTA per SM, launched cooperatively (all CTAs resident: the down
// projection waits for every CTA's share of h).  Phase A: the h blocks (32
// rows of d_ff: two gate slabs and two up slabs) are dealt to CTAs in turn;
// four warps stream one block's four slabs, each CTA quantises x itself (the
// standalone quantiser's bytes), and one warp per block forms h = SiLU(g) * u
// and its Q8_0 codes (the steps of the three-launch chain's middle kernel) in
// global memory, then counts the block done.  Phase B: the down projection's
// (slab, segment) stages are dealt to CTAs in contiguous ranges, and inside
// a CTA to the warps that phase A leaves idle first; each warp's ring holds
// its stages from the start, so the down weights stream while phase A runs.
// After a bounded wait for all h blocks, each CTA copies h's codes into
// shared memory and every warp reduces its stages; the segment sums of a
// slab are added in segment order by the last warp to finish one (atomic
// counter), then the residual.  Every fp32 step is the one of the chain, in
// the same order, so y is bit-identical to qgemv_q4_0_ffn's three launches.
#include <algorithm>
#include <atomic>
#include <cstring>

#include "gemv_kernel.cuh"
#include "qgemv_launch.h"

namespace qg {

constexpr int FF_WARPS = 16;
constexpr int FF_THREADS = FF_WARPS * 32;
constexpr int FF_RING = 2;    // weight stages in flight per warp
constexpr int FF_HB = 4;      // h blocks a CTA works on at once (four warps each)
constexpr int FF_CNT_WORDS = 4096;  // counters in the workspace's first 16 KB

struct FfnParams {
    const uint8_t *Wg, *Wu, *Wd;  // packed weights
    const float *x;               // [T][d_model]
    const float *res;             // [T][d_model] or nullptr
    float *y;                     // [T][d_model]
    uint8_t *hq;                  // planar Q8_0 of h: [T][d_ff] codes, then [T][d_ff / 32] fp16 scales
    float *part;                  // down segment sums [nslab_dn][nseg_dn][T][16]
    unsigned *cnt;                // [0] h blocks done, [1] CTAs past the wait, [2 + s] down slab s arrivals
    unsigned *status;
    long long slab_up, slab_dn;   // bytes of one packed slab (288 nb)
    int d_model, d_ff;
    int nb_up, nb_dn, nseg_up, nseg_dn, nslab_dn;
    int nhb;                      // h blocks: d_ff / 32
    int ndn;                      // down stages: nslab_dn * nseg_dn
    int off_ring, off_bar, off_hbuf;  // shared memory: [activation area][hbuf][barriers][rings]
};

// The stages one warp consumes, in order: its phase-A slab items (round by
// round, all segments of K = d_model each), then its phase-B stages (one
// down (slab, segment) each).
struct FfWalk {
    int phase;          // 0: A, 1: B, 2: done
    int round, seg;     // A: round, segment of the current slab item
    int k;              // B: index among the CTA's down stages
    int nrounds, nhb_cta, dn0, dn1;

    __device__ __forceinline__ bool a_item(int warp, int rnd) const { return FF_HB * rnd + (warp >> 2) < nhb_cta; }

    __device__ __forceinline__ void settle(const FfnParams &P, int warp)
    {
        while (phase == 0 && (round >= nrounds || !a_item(warp, round))) {
            if (round >= nrounds) {
                phase = 1;
                k = FF_WARPS - 1 - warp;  // this warp's first stage: items k with k % 16 == 15 - warp
                break;
            }
            ++round;
        }
        if (phase == 1 && dn0 + k >= dn1) phase = 2;
    }

    __device__ __forceinline__ void init(const FfnParams &P, int warp)
    {
        const int G = gridDim.x, c = blockIdx.x;
        nhb_cta = c < P.nhb ? (P.nhb - c + G - 1) / G : 0;
        nrounds = (nhb_cta + FF_HB - 1) / FF_HB;
        dn0 = static_cast<int>(static_cast<long long>(P.ndn) * c / G);
        dn1 = static_cast<int>(static_cast<long long>(P.ndn) * (c + 1) / G);
        phase = 0;
        round = 0;
        seg = 0;
        k = 0;
        settle(P, warp);
    }

    __device__ __forceinline__ void advance(const FfnParams &P, int warp)
    {
        if (phase == 0) {
            if (++seg < P.nseg_up) return;
            seg = 0;
            ++round;
            settle(P, warp);
        } else if (phase == 1) {
            k += FF_WARPS;
            if (dn0 + k >= dn1) phase = 2;
        }
    }

    // The h block of this warp's phase-A item, and the item's slab and matrix.
    __device__ __forceinline__ int hb(int warp) const { return blockIdx.x + gridDim.x * (FF_HB * round + (warp >> 2)); }

    __device__ __forceinline__ const uint8_t *src(const FfnParams &P, int warp) const
    {
        if (phase == 0) {
            const int slab = 2 * hb(warp) + (warp & 1);
            const uint8_t *W = (warp & 2) ? P.Wu : P.Wg;
            return W + static_cast<long long>(slab) * P.slab_up + static_cast<long long>(seg) * SEG_BYTES;
        }
        const int i = dn0 + k, s = i / P.nseg_dn, sg = i - s * P.nseg_dn;
        return P.Wd + static_cast<long long>(s) * P.slab_dn + static_cast<long long>(sg) * SEG_BYTES;
    }

    __device__ __forceinline__ unsigned bytes(const FfnParams &P) const
    {
        if (phase == 0) return static_cast<unsigned>(SLAB_COL_BYTES * min(SEG_BLOCKS, P.nb_up - SEG_BLOCKS * seg));
        const int sg = (dn0 + k) % P.nseg_dn;
        return static_cast<unsigned>(SLAB_COL_BYTES * min(SEG_BLOCKS, P.nb_dn - SEG_BLOCKS * sg));
    }
};

template <int T>
__global__ void __launch_bounds__(FF_THREADS, 1) ffn_fused_kernel(const __grid_constant__ FfnParams P)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_abort;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r8 = lane >> 2, j = lane & 3;
    using LO = LaneOut<T, false>;
    constexpr int NO = LO::N;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + P.off_bar) + warp * FF_RING;
    uint8_t *ring = smem + P.off_ring + static_cast<size_t>(warp) * FF_RING * SEG_BYTES;
    float *hbuf = reinterpret_cast<float *>(smem + P.off_hbuf);  // [FF_HB][2 (gate, up)][32 rows][T]
    volatile int *abort_flag = &s_abort;

    if (tid == 0) s_abort = 0;
    if (lane == 0)
        for (int d = 0; d < FF_RING; ++d) mbar_init(&bar[d], 1);
    fence_mbar_init();
    __syncthreads();

    // weights first: phase A's slabs and the down stages depend on no kernel
    FfWalk fill, use;
    fill.init(P, warp);
    use = fill;
    const uint64_t pol = l2_policy_evict_first();
    int slot = 0, issued = 0, waited = 0;  // fills issued; fills seen complete
    unsigned phase_bit = 0;
    auto issue = [&](int into) {
        if (lane == 0) {
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&bar[into], fill.bytes(P));
            bulk_g2s(ring + into * SEG_BYTES, fill.src(P, warp), fill.bytes(P), &bar[into], pol);
        }
        ++issued;
        fill.advance(P, warp);
    };
    for (int d = 0; d < FF_RING && fill.phase < 2; ++d) issue(d);
    // the next stage in this warp's order, once its copy has landed
    bool ok = true;
    auto take = [&]() -> const uint8_t * {
        if (ok) {
            ok = mbar_wait_bounded(&bar[slot], phase_bit, abort_flag, P.status, WAIT_LIMIT_NS);
            waited += ok ? 1 : 0;
        }
        return ring + slot * SEG_BYTES;
    };
    auto release = [&]() {
        __syncwarp();
        if (fill.phase < 2 && ok) issue(slot);
        if (++slot == FF_RING) {
            slot = 0;
            phase_bit ^= 1u;
        }
    };

    // ---- phase A: x quantised in shared memory, then the h blocks
    pdl_wait();
    quantize_image<T, false>(smem, P.x, P.d_model, tid, FF_THREADS);
    __syncthreads();
    {
        const XqLayout L = xq_layout(T, P.d_model, false);
        const XqView xv{reinterpret_cast<const int8_t *>(smem), L.xstride,
                        reinterpret_cast<const int2 *>(smem + L.off_cd), L.cdw};
        for (int rnd = 0; rnd < use.nrounds; ++rnd) {
            if (use.phase == 0 && use.round == rnd) {
                // this warp's slab item: all segments in order
                float yv[NO];
                for (int sg = 0; sg < P.nseg_up; ++sg) {
                    float Pk[NO];
                    const uint8_t *stg = take();
                    if (ok)
                        segment_sum<T, false>(true, stg, nullptr, 0, sg, P.nb_up, r8, j, xv, Pk);
                    else
#pragma unroll
                        for (int k2 = 0; k2 < NO; ++k2) Pk[k2] = 0.0f;
                    release();
                    use.advance(P, warp);
#pragma unroll
                    for (int k2 = 0; k2 < NO; ++k2) yv[k2] = sg == 0 ? Pk[k2] : __fadd_rn(yv[k2], Pk[k2]);
                }
                // rows r8 and r8 + 8 of the slab, every token (lanes j == 0)
                float *hb = hbuf + ((warp >> 2) * 2 + ((warp >> 1) & 1)) * 32 * T;
#pragma unroll
                for (int k2 = 0; k2 < NO; ++k2)
                    if (LO::owner(k2, j)) hb[(16 * (warp & 1) + LO::row(k2, r8)) * T + LO::tok(k2, j)] = yv[k2];
            }
            __syncthreads();
            // one warp per h block of the round: h = SiLU(g) * u, then Q8_0
            const int hbl = warp;
            if (hbl < FF_HB && FF_HB * rnd + hbl < use.nhb_cta) {
                const int hbi = blockIdx.x + gridDim.x * (FF_HB * rnd + hbl);
                const float *gb = hbuf + (hbl * 2) * 32 * T, *ub = gb + 32 * T;
#pragma unroll
                for (int t = 0; t < T; ++t) {
                    const float h = __fmul_rn(ffn_silu(gb[lane * T + t]), ub[lane * T + t]);
                    float amax = fabsf(h);
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
                    float d, id;
                    q8_scale(amax, d, id);
                    P.hq[static_cast<long long>(t) * P.d_ff + hbi * QK + lane] =
                        static_cast<uint8_t>(static_cast<int8_t>(q8_code(h, id)));
                    if (lane == 0)
                        reinterpret_cast<unsigned short *>(P.hq + static_cast<long long>(T) * P.d_ff)[t * P.nhb + hbi] =
                            q8_half(d);
                }
                __threadfence();
                __syncwarp();
                if (lane == 0) atomicAdd(P.cnt, 1u);
            }
            __syncthreads();  // hbuf is reused by the next round
        }
    }

    // ---- every h block done (bounded wait by one thread per CTA)
    __shared__ int s_go;
    if (tid == 0) {
        const uint64_t t0 = global_timer_ns();
        unsigned v = 0;
        for (;;) {
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(P.cnt) : "memory");
            if (v >= static_cast<unsigned>(P.nhb) || *abort_flag) break;
            if (global_timer_ns() - t0 > WAIT_LIMIT_NS) {
                *abort_flag = 1;
                atomicCAS(P.status, 0u, ST_TIMEOUT);
                break;
            }
        }
        s_go = (v >= static_cast<unsigned>(P.nhb) && !*abort_flag) ? 1 : 0;
        // the last CTA past the wait leaves both counters at zero
        if (atomicAdd(P.cnt + 1, 1u) == gridDim.x - 1) {
            P.cnt[0] = 0u;
            P.cnt[1] = 0u;
        }
    }
    __syncthreads();
    pdl_launch_dependents();  // only now: every CTA of this grid is past its wait
    const bool go = s_go != 0;

    // ---- phase B: h's codes in shared memory, then the down stages
    if (go) {
        const XqLayout L = xq_layout(T, P.d_ff, false);
        const uint4 *src = reinterpret_cast<const uint4 *>(P.hq);
        uint4 *dst = reinterpret_cast<uint4 *>(smem);
        for (int i = tid; i < T * P.d_ff / 16; i += FF_THREADS) dst[i] = __ldcg(src + i);
        const unsigned short *hs = reinterpret_cast<const unsigned short *>(P.hq + static_cast<long long>(T) * P.d_ff);
        unsigned short *ds = reinterpret_cast<unsigned short *>(smem + L.off_d);
        for (int i = tid; i < T * P.nhb; i += FF_THREADS) ds[i] = __ldcg(hs + i);
        __syncthreads();
        build_fold_constants<T, false>(smem, P.d_ff, tid, FF_THREADS);
    }
    __syncthreads();
    {
        const XqLayout L = xq_layout(T, P.d_ff, false);
        const XqView xv{reinterpret_cast<const int8_t *>(smem), L.xstride,
                        reinterpret_cast<const int2 *>(smem + L.off_cd), L.cdw};
        while (use.phase == 1) {
            const int i = use.dn0 + use.k, s = i / P.nseg_dn, sg = i - s * P.nseg_dn;
            float Pk[NO];
            const uint8_t *stg = take();
            if (ok && go)
                segment_sum<T, false>(true, stg, nullptr, 0, sg, P.nb_dn, r8, j, xv, Pk);
            else
#pragma unroll
                for (int k2 = 0; k2 < NO; ++k2) Pk[k2] = 0.0f;
            release();
            use.advance(P, warp);
            if (!go) continue;
            float *pb = P.part + (static_cast<long long>(s) * P.nseg_dn + sg) * T * 16;
#pragma unroll
            for (int k2 = 0; k2 < NO; ++k2)
                if (LO::owner(k2, j)) pb[LO::tok(k2, j) * 16 + LO::row(k2, r8)] = Pk[k2];
            // the last warp to finish a segment of slab s adds all of them in order
            __threadfence();
            __syncwarp();
            unsigned old = 0;
            if (lane == 0) old = atomicAdd(P.cnt + 2 + s, 1u);
            old = __shfl_sync(0xFFFFFFFFu, old, 0);
            if (old == static_cast<unsigned>(P.nseg_dn - 1)) {
                __threadfence();
                if (lane < 16) {
                    const float *pr = P.part + static_cast<long long>(s) * P.nseg_dn * T * 16;
                    const int row = s * 16 + lane;
#pragma unroll
                    for (int t = 0; t < T; ++t) {
                        float v = ordered_sum_ldcg(pr + t * 16 + lane, P.nseg_dn, T * 16);
                        const long long yi = static_cast<long long>(t) * P.d_model + row;
                        if (P.res != nullptr) v = __fadd_rn(v, P.res[yi]);
                        P.y[yi] = v;
                    }
                }
                __syncwarp();
                if (lane == 0) P.cnt[2 + s] = 0u;
            }
        }
    }
    // copies still in flight (only after an abort): wait for them, bounded;
    // fill i went to slot i % FF_RING, completing that slot's phase i / FF_RING
    for (int i = waited; i < issued; ++i) mbar_drain(&bar[i % FF_RING], static_cast<unsigned>((i / FF_RING) & 1));
}

// ------------------------------------------------------------ host side

bool ffn_fused_eligible(long long d_model, long long d_ff, int T)
{
    return T >= 1 && T <= 4 && d_model % SLAB_ROWS == 0 && d_ff % QK == 0 && d_model >= SLAB_ROWS && d_ff >= QK &&
           2 + d_model / SLAB_ROWS <= FF_CNT_WORDS;
}

// Shared memory: the activation area (x's image in phase A, h's in phase
// B), the h buffer, barriers, rings.
static long long ffn_smem(long long d_model, long long d_ff, int T, int &off_hbuf, int &off_bar, int &off_ring)
{
    const long long xa = std::max(xq_layout(T, static_cast<int>(d_model), false).bytes,
                                  xq_layout(T, static_cast<int>(d_ff), false).bytes);
    off_hbuf = static_cast<int>((xa + 127) / 128 * 128);
    off_bar = off_hbuf + (FF_HB * 2 * 32 * T * 4 + 127) / 128 * 128;
    off_ring = off_bar + (FF_WARPS * FF_RING * 8 + 127) / 128 * 128;
    return off_ring + static_cast<long long>(FF_WARPS) * FF_RING * SEG_BYTES;
}

bool ffn_fused_fits(long long d_model, long long d_ff, int T, int smem_budget)
{
    int a, b, c;
    return ffn_fused_eligible(d_model, d_ff, T) && ffn_smem(d_model, d_ff, T, a, b, c) <= smem_budget;
}

template <int T>
static cudaError_t launch_ffn_t(const FfnParams &P, int grid, size_t smem, cudaStream_t st)
{
    auto kern = ffn_fused_kernel<T>;
    static std::atomic<unsigned long long> raised{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(raised.load(std::memory_order_acquire) & bit)) {
        int optin = 0;
        e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return e;
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, kern);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 optin - static_cast<int>(fa.sharedSizeBytes));
        if (e != cudaSuccess) return e;
        raised.fetch_or(bit, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(FF_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    // cooperative: every CTA resident at once (phase B waits for all of them)
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, kern, P);
    if (e != cudaSuccess) {  // without early launch, if the two cannot be combined
        (void)cudaGetLastError();
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kern, P);
    }
    return e;
}

cudaError_t launch_ffn_fused(const void *Wg, const void *Wu, const void *Wd, const float *x, const float *res,
                             float *y, long long d_model, long long d_ff, int T, uint8_t *hq, float *part,
                             unsigned *cnt, int grid, int smem_budget, unsigned *status, cudaStream_t st)
{
    if (!ffn_fused_eligible(d_model, d_ff, T)) return cudaErrorInvalidValue;
    FfnParams P;
    memset(&P, 0, sizeof(P));
    P.Wg = static_cast<const uint8_t *>(Wg);
    P.Wu = static_cast<const uint8_t *>(Wu);
    P.Wd = static_cast<const uint8_t *>(Wd);
    P.x = x;
    P.res = res;
    P.y = y;
    P.hq = hq;
    P.part = part;
    P.cnt = cnt;
    P.status = status;
    P.d_model = static_cast<int>(d_model);
    P.d_ff = static_cast<int>(d_ff);
    P.nb_up = P.d_model / QK;
    P.nb_dn = P.d_ff / QK;
    P.nseg_up = (P.nb_up + SEG_BLOCKS - 1) / SEG_BLOCKS;
    P.nseg_dn = (P.nb_dn + SEG_BLOCKS - 1) / SEG_BLOCKS;
    P.nslab_dn = P.d_model / SLAB_ROWS;
    P.slab_up = static_cast<long long>(SLAB_COL_BYTES) * P.nb_up;
    P.slab_dn = static_cast<long long>(SLAB_COL_BYTES) * P.nb_dn;
    P.nhb = P.d_ff / QK;
    P.ndn = P.nslab_dn * P.nseg_dn;
    const long long smem = ffn_smem(d_model, d_ff, T, P.off_hbuf, P.off_bar, P.off_ring);
    if (smem > smem_budget) return cudaErrorInvalidValue;
    switch (T) {
    case 1: return launch_ffn_t<1>(P, grid, static_cast<size_t>(smem), st);
    case 2: return launch_ffn_t<2>(P, grid, static_cast<size_t>(smem), st);
    case 3: return launch_ffn_t<3>(P, grid, static_cast<size_t>(smem), st);
    case 4: return launch_ffn_t<4>(P, grid, static_cast<size_t>(smem), st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qg
