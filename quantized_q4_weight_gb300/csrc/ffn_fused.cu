// ffn_fused.cu -- the decode FFN step in one persistent launch (minfer README
// M15: one persistent kernel runs the layer and keeps DRAM busy; colibri
// qwen36 docs: gate and up share one pass over the activation):
//     y = W_down . Q8_0(SiLU(W_gate . x) * (W_up . x))  [+ residual]
//
// One CTA per SM, launched cooperatively (all CTAs resident: the down
// projection waits for every CTA's share of h).  Work is dealt in weight
// stages (one 16-block segment of one 16-row slab, 4608 bytes): a CTA's
// stages are its phase-A stages, then its phase-B stages, and warp w of the
// CTA streams every sixteenth of them through its own ring.
//   Phase A: the h blocks (32 rows of d_ff: two gate slabs and two up
//   slabs) are dealt to CTAs in turn; a block's 4 x nseg_up stages go to
//   the warps, each writing its segment sums to shared memory.  Each CTA
//   quantises x itself (the standalone quantiser's bytes).  One warp per
//   block then adds every row's segment sums in segment order, forms
//   h = SiLU(g) * u and its Q8_0 codes (the steps of the three-launch
//   chain's middle kernel) in global memory, and counts the block done.
//   Phase B: the down projection's slabs are dealt to CTAs in turn, a
//   slab's nseg_dn stages to the warps; after a bounded wait for all h
//   blocks each CTA copies h's codes into shared memory, every warp reduces
//   its stages, and the slab's segment sums are added in segment order in
//   shared memory, then the residual.
// Every fp32 step is the one of the chain, in the same order, so y is
// bit-identical to qgemv_q4_0_ffn's three launches.  Before the dependency
// wait each warp asks L2 for its first stages, so the layer streams from
// HBM while the CTA waits for its input.
#include <algorithm>
#include <atomic>
#include <cstring>

#include "gemv_kernel.cuh"
#include "qgemv_launch.h"

namespace qg {

constexpr int FF_WARPS = 16;
constexpr int FF_THREADS = FF_WARPS * 32;
constexpr int FF_RING = 2;      // weight stages in flight per warp
constexpr int FF_HB = 4;        // h blocks a CTA works on at once
constexpr int FF_PREFETCH = 4;  // stages per warp requested into L2 beyond its ring at the start

struct FfnParams {
    const uint8_t *Wg, *Wu, *Wd;  // packed weights
    const float *x;               // [T][d_model]
    const float *res;             // [T][d_model] or nullptr
    float *y;                     // [T][d_model]
    uint8_t *hq;                  // planar Q8_0 of h: [T][d_ff] codes, then [T][d_ff / 32] fp16 scales
    unsigned *cnt;                // [0] h blocks done, [1] CTAs past the wait (both left at zero)
    unsigned *status;
    long long slab_up, slab_dn;   // bytes of one packed slab (288 nb)
    int d_model, d_ff;
    int nb_up, nb_dn, nseg_up, nseg_dn, nslab_dn;
    int nhb;                      // h blocks: d_ff / 32
    int off_part, off_bar, off_ring;  // shared memory: [activation area][segment sums][barriers][rings]
};

// The stages one warp consumes, in order: its phase-A stages round by round
// (a round is up to FF_HB of the CTA's h blocks, stage a of a round being
// (h block a / (4 nseg_up), slab (a / nseg_up) % 4, segment a % nseg_up)),
// then its phase-B stages (stage b: the CTA's down slab b / nseg_dn,
// segment b % nseg_dn); warp w takes the stages whose index is w modulo 16
// in phase A and 15 - w in phase B, so that the warps with fewer phase-A
// stages take the down stages first.
struct FfWalk {
    int phase;        // 0: A, 1: B, 2: done
    int round, a, na; // A: round, stage in it, stages in it
    int b;            // B: stage among the CTA's down stages
    int nrounds, nhb_cta, nb_cta;

    __device__ __forceinline__ void start_round(const FfnParams &P)
    {
        na = min(FF_HB, nhb_cta - FF_HB * round) * 4 * P.nseg_up;
    }

    __device__ __forceinline__ void settle(const FfnParams &P, int warp)
    {
        while (phase == 0 && a >= na) {
            if (++round >= nrounds) {
                phase = 1;
                b = FF_WARPS - 1 - warp;
                break;
            }
            a = warp;
            start_round(P);
        }
        if (phase == 1 && b >= nb_cta) phase = 2;
    }

    __device__ __forceinline__ void init(const FfnParams &P, int warp)
    {
        const int G = gridDim.x, c = blockIdx.x;
        nhb_cta = c < P.nhb ? (P.nhb - c + G - 1) / G : 0;
        nrounds = (nhb_cta + FF_HB - 1) / FF_HB;
        nb_cta = (c < P.nslab_dn ? (P.nslab_dn - c + G - 1) / G : 0) * P.nseg_dn;
        phase = 0;
        round = 0;
        a = warp;
        na = 0;
        b = 0;
        if (nrounds > 0) start_round(P);
        settle(P, warp);
    }

    __device__ __forceinline__ void advance(const FfnParams &P, int warp)
    {
        if (phase == 0) {
            a += FF_WARPS;
            settle(P, warp);
        } else if (phase == 1) {
            b += FF_WARPS;
            if (b >= nb_cta) phase = 2;
        }
    }

    // the segment of the current stage
    __device__ __forceinline__ int seg(const FfnParams &P) const
    {
        return phase == 0 ? a % P.nseg_up : b % P.nseg_dn;
    }

    __device__ __forceinline__ const uint8_t *src(const FfnParams &P) const
    {
        if (phase == 0) {
            const int hl = a / (4 * P.nseg_up), m = (a / P.nseg_up) & 3, sg = a % P.nseg_up;
            const int hb = blockIdx.x + gridDim.x * (FF_HB * round + hl);
            const uint8_t *W = (m & 2) ? P.Wu : P.Wg;
            return W + static_cast<long long>(2 * hb + (m & 1)) * P.slab_up + static_cast<long long>(sg) * SEG_BYTES;
        }
        const int si = b / P.nseg_dn, sg = b - si * P.nseg_dn;
        return P.Wd + static_cast<long long>(blockIdx.x + gridDim.x * si) * P.slab_dn +
               static_cast<long long>(sg) * SEG_BYTES;
    }

    __device__ __forceinline__ unsigned bytes(const FfnParams &P) const
    {
        const int sg = seg(P), nb = phase == 0 ? P.nb_up : P.nb_dn;
        return static_cast<unsigned>(SLAB_COL_BYTES * min(SEG_BLOCKS, nb - SEG_BLOCKS * sg));
    }
};

template <int T>
__global__ void __launch_bounds__(FF_THREADS, 1) ffn_fused_kernel(const __grid_constant__ FfnParams P)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_abort;
    __shared__ int s_go;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r8 = lane >> 2, j = lane & 3;
    using LO = LaneOut<T, false>;
    constexpr int NO = LO::N;
    constexpr int TS = T * 16;  // floats of one stage's segment sums: [T][16 rows]
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + P.off_bar) + warp * FF_RING;
    uint8_t *ring = smem + P.off_ring + static_cast<size_t>(warp) * FF_RING * SEG_BYTES;
    float *part = reinterpret_cast<float *>(smem + P.off_part);
    volatile int *abort_flag = &s_abort;

    if (tid == 0) s_abort = 0;
    if (lane == 0)
        for (int d = 0; d < FF_RING; ++d) mbar_init(&bar[d], 1);
    fence_mbar_init();
    __syncthreads();

    // the weights depend on no kernel: each warp's stages, in its order
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
            bulk_g2s(ring + into * SEG_BYTES, fill.src(P), fill.bytes(P), &bar[into], pol);
        }
        ++issued;
        fill.advance(P, warp);
    };
    // Before the dependency wait: x's lines, then every warp's first stages
    // (its whole share of the layer in the usual shapes) are requested into
    // L2, so HBM streams the layer while the CTA waits; the ring copies
    // themselves start only once x is quantised, so that x's load does not
    // queue behind a ring's worth of weight data returning to this SM.  (x
    // may still be being written by the kernel before this one: a prefetch
    // only moves lines into L2, which the writes update.  Only x's whole
    // 16-byte units are prefetched, so nothing outside x is read.)
    if (tid == 0) {
        const uintptr_t a = reinterpret_cast<uintptr_t>(P.x);
        const uintptr_t b = a + 4ull * T * P.d_model;
        const uintptr_t a16 = (a + 15) & ~static_cast<uintptr_t>(15), b16 = b & ~static_cast<uintptr_t>(15);
        if (b16 > a16) bulk_prefetch_l2(reinterpret_cast<const void *>(a16), static_cast<unsigned>(b16 - a16));
    }
    __syncwarp();
    if (lane == 0) {
        FfWalk pf = fill;
        for (int d = 0; d < FF_RING + FF_PREFETCH && pf.phase < 2; ++d) {
            bulk_prefetch_l2(pf.src(P), pf.bytes(P));
            pf.advance(P, warp);
        }
    }
    bool ok = true;
    // The warp's next stage: waits for its copy, reduces it against the
    // activation image xv into this lane's segment sums, frees the slot for
    // the next fill, and stores the sums as part[idx][t][row].
    auto stage = [&](const XqView &xv, int nb, bool live) {
        const int sg = use.seg(P), idx = use.phase == 0 ? use.a : use.b;
        if (ok) {
            ok = mbar_wait_bounded(&bar[slot], phase_bit, abort_flag, P.status, WAIT_LIMIT_NS);
            waited += ok ? 1 : 0;
        }
        float Pk[NO];
        if (ok && live)
            segment_sum<T, false>(true, ring + slot * SEG_BYTES, nullptr, 0, sg, nb, r8, j, xv, Pk);
        else
#pragma unroll
            for (int k2 = 0; k2 < NO; ++k2) Pk[k2] = 0.0f;
        __syncwarp();
        if (fill.phase < 2 && ok) issue(slot);
        if (++slot == FF_RING) {
            slot = 0;
            phase_bit ^= 1u;
        }
        use.advance(P, warp);
        float *pp = part + idx * TS;
#pragma unroll
        for (int k2 = 0; k2 < NO; ++k2)
            if (LO::owner(k2, j)) pp[LO::tok(k2, j) * 16 + LO::row(k2, r8)] = Pk[k2];
    };

    // ---- phase A: x quantised in shared memory, then the h blocks
    pdl_wait();
    quantize_image<T, false>(smem, P.x, P.d_model, tid, FF_THREADS);
    for (int d = 0; d < FF_RING && fill.phase < 2; ++d) issue(d);
    __syncthreads();
    {
        const XqLayout L = xq_layout(T, P.d_model, false);
        const XqView xv{reinterpret_cast<const int8_t *>(smem), L.xstride,
                        reinterpret_cast<const int2 *>(smem + L.off_cd), L.cdw};
        for (int rnd = 0; rnd < use.nrounds; ++rnd) {
            while (use.phase == 0 && use.round == rnd) stage(xv, P.nb_up, true);
            __syncthreads();
            // one warp per h block of the round: lane = row of the block
            // (gate and up slab 2 hb + lane / 16, row lane % 16); each
            // output's segment sums added in segment order, h = SiLU(g) * u,
            // then Q8_0
            const int hbl = warp;
            if (hbl < FF_HB && FF_HB * rnd + hbl < use.nhb_cta) {
                const int hbi = blockIdx.x + gridDim.x * (FF_HB * rnd + hbl);
                const float *pg = part + (hbl * 4 + (lane >> 4)) * P.nseg_up * TS + (lane & 15);
                const float *pu = pg + 2 * P.nseg_up * TS;
#pragma unroll
                for (int t = 0; t < T; ++t) {
                    float g = pg[t * 16], u = pu[t * 16];
                    for (int sg = 1; sg < P.nseg_up; ++sg) {
                        g = __fadd_rn(g, pg[sg * TS + t * 16]);
                        u = __fadd_rn(u, pu[sg * TS + t * 16]);
                    }
                    const float h = __fmul_rn(ffn_silu(g), u);
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
            }
            __syncthreads();  // (the segment sums are reused by the next round)
            // the round's h blocks are written: one fence makes the whole
            // CTA's writes visible before they are counted
            if (tid == 0) {
                const int nr = min(FF_HB, use.nhb_cta - FF_HB * rnd);
                __threadfence();
                atomicAdd(P.cnt, static_cast<unsigned>(nr));
            }
        }
    }

    // ---- every h block done (bounded wait by one thread per CTA)
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
        while (use.phase == 1) stage(xv, P.nb_dn, go);
    }
    __syncthreads();
    // each output of the CTA's slabs: its segment sums in segment order, then the residual
    if (go)
        for (int i = tid; i < use.nb_cta / P.nseg_dn * TS; i += FF_THREADS) {
            const int si = i / TS, rem = i - si * TS, t = rem >> 4, row = rem & 15;
            const float *pp = part + si * P.nseg_dn * TS + rem;
            float v = pp[0];
            for (int sg = 1; sg < P.nseg_dn; sg += 8) {
                float x8[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) x8[k] = sg + k < P.nseg_dn ? pp[(sg + k) * TS] : 0.0f;
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    if (sg + k < P.nseg_dn) v = __fadd_rn(v, x8[k]);
            }
            const long long yi = static_cast<long long>(t) * P.d_model + (blockIdx.x + gridDim.x * si) * SLAB_ROWS + row;
            if (P.res != nullptr) v = __fadd_rn(v, P.res[yi]);
            P.y[yi] = v;
        }
    // copies still in flight (only after an abort): wait for them, bounded;
    // fill i went to slot i % FF_RING, completing that slot's phase i / FF_RING
    for (int i = waited; i < issued; ++i) mbar_drain(&bar[i % FF_RING], static_cast<unsigned>((i / FF_RING) & 1));
}

// ------------------------------------------------------------ host side

bool ffn_fused_eligible(long long d_model, long long d_ff, int T)
{
    return T >= 1 && T <= 4 && d_model % SLAB_ROWS == 0 && d_ff % QK == 0 && d_model >= SLAB_ROWS && d_ff >= QK;
}

// Shared memory: the activation area (x's image in phase A, h's in phase
// B), the segment sums (a round's phase-A stages, or the CTA's down
// stages), barriers, rings.
static long long ffn_smem(long long d_model, long long d_ff, int T, int grid, int &off_part, int &off_bar,
                          int &off_ring)
{
    const long long xa = std::max(xq_layout(T, static_cast<int>(d_model), false).bytes,
                                  xq_layout(T, static_cast<int>(d_ff), false).bytes);
    const long long nb_up = d_model / QK, nb_dn = d_ff / QK;
    const long long nseg_up = (nb_up + SEG_BLOCKS - 1) / SEG_BLOCKS, nseg_dn = (nb_dn + SEG_BLOCKS - 1) / SEG_BLOCKS;
    const long long nhb = d_ff / QK, nslab = d_model / SLAB_ROWS;
    const long long hb_round = std::min<long long>(FF_HB, (nhb + grid - 1) / grid);
    const long long slabs_cta = (nslab + grid - 1) / grid;
    const long long sums = std::max(hb_round * 4 * nseg_up, slabs_cta * nseg_dn) * T * 16 * 4;
    off_part = static_cast<int>((xa + 127) / 128 * 128);
    off_bar = off_part + static_cast<int>((sums + 127) / 128 * 128);
    off_ring = off_bar + (FF_WARPS * FF_RING * 8 + 127) / 128 * 128;
    return off_ring + static_cast<long long>(FF_WARPS) * FF_RING * SEG_BYTES;
}

bool ffn_fused_fits(long long d_model, long long d_ff, int T, int grid, int smem_budget)
{
    if (!ffn_fused_eligible(d_model, d_ff, T) || grid < 1) return false;
    int a, b, c;
    return ffn_smem(d_model, d_ff, T, grid, a, b, c) <= smem_budget;
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
                             float *y, long long d_model, long long d_ff, int T, uint8_t *hq, unsigned *cnt, int grid,
                             int smem_budget, unsigned *status, cudaStream_t st)
{
    if (!ffn_fused_eligible(d_model, d_ff, T) || grid < 1) return cudaErrorInvalidValue;
    FfnParams P;
    memset(&P, 0, sizeof(P));
    P.Wg = static_cast<const uint8_t *>(Wg);
    P.Wu = static_cast<const uint8_t *>(Wu);
    P.Wd = static_cast<const uint8_t *>(Wd);
    P.x = x;
    P.res = res;
    P.y = y;
    P.hq = hq;
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
    const long long smem = ffn_smem(d_model, d_ff, T, grid, P.off_part, P.off_bar, P.off_ring);
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
