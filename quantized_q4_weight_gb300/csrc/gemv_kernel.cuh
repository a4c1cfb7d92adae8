// gemv_kernel.cuh -- the weight-streaming Q4_0 x Q8_0 GEMV kernel.
//
// One persistent CTA per SM, 8 warps.  A launch covers a list of GEMVs
// ("groups" x "instances"); their work is cut into items -- one 16-row slab
// over all of K, or (split-K) over one 16-block segment of K -- and the items
// are dealt to CTAs as contiguous ranges of equal weight bytes.  Inside a CTA
// the items of each (group, instance) run go round-robin to the warps.
//
// Weight bytes reach shared memory through 1-D bulk asynchronous copies
// (TMA, cp.async.bulk) into a per-warp ring of stages (one stage = one
// 16-block segment of a slab = 4608 bytes), each completing on its own
// mbarrier; the next stage is issued as soon as a slot is consumed, so every
// warp keeps ring_depth stages in flight.  The activations of the current
// run (planar Q8_0) are copied into shared memory once per CTA, together with
// each block's folded-offset constant and fp32 scale.
//
// Lane mapping (minfer README M15 repacks rows into groups so a warp reads
// contiguous bytes; here 16-row slabs): lane = 4 * r8 + j handles rows r8 and
// r8 + 8 of the slab and the blocks b with b % 4 == j.  Per block it unpacks
// the nibbles with two masks (M9: SIMD nibble masking), forms the exact
// integer block sum with dp4a and the folded -8 offset (M9), and accumulates
// (d_w * d_x) * isum with one fp32 fused multiply-add.  At the end of a
// segment the four phases are combined by a fixed two-level shuffle tree;
// segments are added in order.  The order depends only on K (include/qgemv.h).
//
// Every wait on an asynchronous copy is bounded (see mbar_wait_bounded); a
// CTA that gives up records a status word, stops issuing copies, drains the
// ones in flight (again bounded) and finishes without further waits.
#pragma once

#include "qgemv_internal.cuh"

namespace qg {

struct ItemInfo {
    int gi, e;             // group, instance (slot)
    int kind;              // 0: slab item, 1: packed tail (GGML rows after the slabs)
    int slab, seg0, seg1;  // slab index and the segments [seg0, seg1) it covers
    int rows;              // rows present (16, or fewer in a tail / last GGML slab)
    bool bad;              // gather slot with an expert id out of range
    const uint8_t *Wi;     // this instance's weights
};

template <int MAXG>
__device__ __forceinline__ int group_of_item(const Params<MAXG> &P, long long i, int gi)
{
    while (gi + 1 < P.ngroups && P.g[gi + 1].item_begin <= i) ++gi;
    return gi;
}

template <int MAXG>
__device__ __forceinline__ ItemInfo decode_item(const Params<MAXG> &P, long long i, int &gi_hint)
{
    ItemInfo it;
    const int gi = group_of_item(P, i, gi_hint);
    gi_hint = gi;
    const Group &g = P.g[gi];
    const int local = static_cast<int>(i - g.item_begin);  // a launch has < 2^31 items
    const int ipi = g.items_per_inst;
    const int e = local / ipi;
    const int r = local - e * ipi;
    int expert = e;
    it.bad = false;
    if (P.ids != nullptr) {
        expert = __ldg(P.ids + e);
        it.bad = expert < 0 || expert >= P.n_experts;
        if (it.bad) expert = 0;
    }
    it.gi = gi;
    it.e = e;
    it.Wi = g.W + static_cast<long long>(expert) * g.w_stride;
    const int split = g.split;
    if (r < g.nslabs * split) {
        it.kind = 0;
        it.slab = r / split;
        const int part = r - it.slab * split;
        const int spp = (g.nseg + split - 1) / split;
        it.seg0 = part * spp;
        it.seg1 = min(g.nseg, it.seg0 + spp);
        it.rows = min(SLAB_ROWS, g.N - it.slab * SLAB_ROWS);
    } else {
        it.kind = 1;
        it.slab = g.nslabs;
        it.seg0 = 0;
        it.seg1 = g.nseg;
        it.rows = g.tail_rows;
    }
    return it;
}

// First item whose (virtual) start byte is >= X.  Items are laid out in the
// byte space as: slab s, segment part p at s * slab_bytes + seg0 * SEG_BYTES;
// the tail after the slabs.
template <int MAXG>
__device__ long long first_item_at_or_after(const Params<MAXG> &P, long long X)
{
    if (X >= P.total_bytes) return P.total_items;
    int gi = 0;
    while (gi + 1 < P.ngroups && P.g[gi + 1].byte_begin <= X) ++gi;
    const Group &g = P.g[gi];
    const long long local = X - g.byte_begin;
    const long long e = local / g.inst_bytes;
    const long long rem = local - e * g.inst_bytes;
    const long long base = g.item_begin + e * g.items_per_inst;
    if (rem == 0) return base;
    const long long slabs_bytes = static_cast<long long>(g.nslabs) * g.slab_bytes;
    if (rem < slabs_bytes) {
        const long long s = rem / g.slab_bytes;
        const long long r2 = rem - s * g.slab_bytes;
        if (r2 == 0) return base + s * g.split;
        const int spp = (g.nseg + g.split - 1) / g.split;
        const long long pb = static_cast<long long>(spp) * SEG_BYTES;
        const long long p = (r2 + pb - 1) / pb;
        if (p >= g.split) return base + (s + 1) * g.split;
        return base + s * g.split + p;
    }
    if (rem == slabs_bytes) return base + static_cast<long long>(g.nslabs) * g.split;
    return base + g.items_per_inst;
}

// End of the run (same group and instance) that contains item i, clipped to i1.
template <int MAXG>
__device__ __forceinline__ long long run_end(const Params<MAXG> &P, long long i, long long i1, int &gi_hint)
{
    const int gi = group_of_item(P, i, gi_hint);
    gi_hint = gi;
    const Group &g = P.g[gi];
    const int e = static_cast<int>(i - g.item_begin) / g.items_per_inst;
    const long long end = g.item_begin + static_cast<long long>(e + 1) * g.items_per_inst;
    return end < i1 ? end : i1;
}

// Walks this warp's sequence of weight stages (copied by TMA), in the same
// order the compute loop consumes them.
template <int MAXG>
struct StageCursor {
    long long it, rend, i1;
    int st, gi;
    bool valid;
    ItemInfo info;

    __device__ __forceinline__ int nstages(const Params<MAXG> &P) const
    {
        return (P.ggml || info.kind != 0 || info.bad) ? 0 : info.seg1 - info.seg0;
    }

    // Move to this warp's next item (it + nwarps, or the first one of a later run).
    __device__ __forceinline__ bool next_item(const Params<MAXG> &P, int warp)
    {
        it += P.nwarps;
        while (it >= rend) {
            const long long ra = rend;
            if (ra >= i1) return false;
            rend = run_end(P, ra, i1, gi);
            it = ra + warp;
        }
        return true;
    }

    __device__ __forceinline__ void settle(const Params<MAXG> &P, int warp)
    {
        // skip items without copied stages
        while (valid) {
            info = decode_item(P, it, gi);
            if (nstages(P) > 0) return;
            valid = next_item(P, warp);
        }
    }

    __device__ __forceinline__ void init(const Params<MAXG> &P, long long i0, long long i1_, int warp)
    {
        i1 = i1_;
        gi = 0;
        st = 0;
        valid = false;
        if (P.ggml || i0 >= i1) return;
        rend = i0;       // empty run: next_item starts at the run beginning at i0
        it = i0;
        valid = next_item(P, warp);
        settle(P, warp);
    }

    __device__ __forceinline__ void advance(const Params<MAXG> &P, int warp)
    {
        if (++st < nstages(P)) return;
        st = 0;
        valid = next_item(P, warp);
        settle(P, warp);
    }

    __device__ __forceinline__ const uint8_t *src(const Params<MAXG> &P) const
    {
        return info.Wi + static_cast<long long>(info.slab) * P.g[info.gi].slab_bytes +
               static_cast<long long>(info.seg0 + st) * SEG_BYTES;
    }

    __device__ __forceinline__ unsigned bytes(const Params<MAXG> &P) const
    {
        const int nb = P.g[info.gi].nb;
        return static_cast<unsigned>(SLAB_COL_BYTES * min(SEG_BLOCKS, nb - SEG_BLOCKS * (info.seg0 + st)));
    }
};

// acc[h][t] += (d_w(h) * d_x(t)) * isum for one block b of rows h = 0, 1.
template <int T>
__device__ __forceinline__ void fma_block(const uint4 &n0, const uint4 &n1, float dw0, float dw1, int b, int K,
                                          int nb, const int8_t *xs_q, const int2 *xs_cd, float (&acc)[2][T])
{
#pragma unroll
    for (int t = 0; t < T; ++t) {
        const uint4 *xp = reinterpret_cast<const uint4 *>(xs_q + t * K + b * QK);
        const uint4 qa = xp[0], qb = xp[1];
        const int2 cd = xs_cd[t * nb + b];
        const int s0 = block_dot_magic(n0, qa, qb, cd.x);
        const int s1 = block_dot_magic(n1, qa, qb, cd.x);
        const float dx = __int_as_float(cd.y);
        acc[0][t] = __fmaf_rn(__fmul_rn(dw0, dx), magic_to_float(s0), acc[0][t]);
        acc[1][t] = __fmaf_rn(__fmul_rn(dw1, dx), magic_to_float(s1), acc[1][t]);
    }
}

// One segment from a shared-memory stage in the packed quad layout.
template <int T>
__device__ __forceinline__ void segment_from_stage(const uint8_t *stage, int s, int K, int nb, int r8, int j,
                                                   const int8_t *xs_q, const int2 *xs_cd, float (&acc)[2][T])
{
    const int nbs = min(SEG_BLOCKS, nb - SEG_BLOCKS * s);
#pragma unroll
    for (int qq = 0; qq < SEG_BLOCKS / QUAD; ++qq) {
        const int nbq = min(QUAD, nbs - QUAD * qq);
        if (j < nbq) {
            const uint8_t *q = stage + qq * QUAD_BYTES;
            const uint4 n0 = *reinterpret_cast<const uint4 *>(q + (r8 * nbq + j) * 16);
            const uint4 n1 = *reinterpret_cast<const uint4 *>(q + ((r8 + 8) * nbq + j) * 16);
            const unsigned sc = *reinterpret_cast<const unsigned *>(q + 256 * nbq + (r8 * nbq + j) * 4);
            fma_block<T>(n0, n1, h2f(sc), h2f(sc >> 16), SEG_BLOCKS * s + QUAD * qq + j, K, nb, xs_q, xs_cd, acc);
        }
    }
}

// A full segment (16 blocks = 4 full quads) from a shared-memory stage:
// branch-free, every load of the segment issued before the arithmetic.
template <int T>
__device__ __forceinline__ void segment_full_from_stage(const uint8_t *stage, int s, int K, int nb, int r8, int j,
                                                        const int8_t *xs_q, const int2 *xs_cd, float (&acc)[2][T])
{
    const int lo = (r8 * QUAD + j) * 16;
    uint4 n0[4], n1[4];
    unsigned sc[4];
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) {
        const uint8_t *q = stage + qq * QUAD_BYTES;
        n0[qq] = *reinterpret_cast<const uint4 *>(q + lo);
        n1[qq] = *reinterpret_cast<const uint4 *>(q + lo + 8 * QUAD * 16);
        sc[qq] = *reinterpret_cast<const unsigned *>(q + 256 * QUAD + (r8 * QUAD + j) * 4);
    }
#pragma unroll
    for (int qq = 0; qq < 4; ++qq)
        fma_block<T>(n0[qq], n1[qq], h2f(sc[qq]), h2f(sc[qq] >> 16), SEG_BLOCKS * s + QUAD * qq + j, K, nb, xs_q,
                     xs_cd, acc);
}

// One segment read directly from GGML-layout rows in global memory (rows of
// the packed tail, or every row when the weights are not packed).
template <int T>
__device__ __forceinline__ void segment_from_ggml(const uint8_t *rows_base, int rows, int s, int K, int nb, int r8,
                                                  int j, const int8_t *xs_q, const int2 *xs_cd, float (&acc)[2][T])
{
    const int nbs = min(SEG_BLOCKS, nb - SEG_BLOCKS * s);
    const long long row_bytes = static_cast<long long>(nb) * Q4_BYTES;
#pragma unroll
    for (int qq = 0; qq < SEG_BLOCKS / QUAD; ++qq) {
        const int nbq = min(QUAD, nbs - QUAD * qq);
        if (j < nbq) {
            const int b = SEG_BLOCKS * s + QUAD * qq + j;
            uint4 n0 = make_uint4(0, 0, 0, 0), n1 = make_uint4(0, 0, 0, 0);
            unsigned d0 = 0, d1 = 0;
            if (r8 < rows) load_ggml_block(rows_base + r8 * row_bytes + b * Q4_BYTES, n0, d0);
            if (r8 + 8 < rows) load_ggml_block(rows_base + (r8 + 8) * row_bytes + b * Q4_BYTES, n1, d1);
            fma_block<T>(n0, n1, h2f(d0), h2f(d1), b, K, nb, xs_q, xs_cd, acc);
        }
    }
}

// Combine the four phase sums of a segment: (s0 + s1) + (s2 + s3), the same
// bits on all four lanes of a row pair.
template <int T>
__device__ __forceinline__ void combine_phases(float (&acc)[2][T])
{
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int t = 0; t < T; ++t) {
            float v = acc[h][t];
            v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, 1));
            v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, 2));
            acc[h][t] = v;
        }
}

// Warps per CTA a T-token kernel may use: 16 for T <= 2, 8 above (the
// wider accumulators need more than 128 registers per thread).
__host__ __device__ constexpr int max_warps_for(int T) { return T <= 2 ? NWARPS_MAX : 8; }

template <int T, int MAXG, bool ARGMAX>
__global__ void __launch_bounds__(max_warps_for(T) * 32, 1) qgemv_stream_kernel(const __grid_constant__ Params<MAXG> P)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_abort;
    __shared__ int s_last;
    __shared__ unsigned long long s_best[NWARPS_MAX * T];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nw = P.nwarps, nthreads = nw * 32;
    const int r8 = lane >> 2, j = lane & 3;
    const int D = P.ring_depth;
    int8_t *xs_q = reinterpret_cast<int8_t *>(smem);
    const unsigned short *xs_d = reinterpret_cast<const unsigned short *>(smem + P.off_d);
    int2 *xs_cd = reinterpret_cast<int2 *>(smem + P.off_cd);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + P.off_bar);
    uint64_t *wbar = bars + warp * D;
    uint64_t *xbar = bars + nw * D;
    uint8_t *ring = smem + P.off_ring + static_cast<size_t>(warp) * D * SEG_BYTES;
    volatile int *abort_flag = &s_abort;

    if (tid == 0) {
        s_abort = 0;
        mbar_init(xbar, 1);
    }
    if (lane == 0)
        for (int d = 0; d < D; ++d) mbar_init(&wbar[d], 1);
    fence_mbar_init();
    __syncthreads();
    pdl_launch_dependents();

    const long long b0 = P.total_bytes * blockIdx.x / gridDim.x;
    const long long b1 = P.total_bytes * (blockIdx.x + 1) / gridDim.x;
    const long long i0 = first_item_at_or_after(P, b0);
    const long long i1 = first_item_at_or_after(P, b1);

    const uint64_t pol_w = l2_policy_evict_first();
    const uint64_t pol_x = l2_policy_evict_last();

    // Weights do not depend on the preceding kernel: start streaming them now.
    // Ring bookkeeping: `issued` stages were copied; the next one to consume
    // sits in slot `slot`, whose mbarrier is in phase `phase`.
    StageCursor<MAXG> cur;
    cur.init(P, i0, i1, warp);
    int issued = 0, consumed = 0, slot = 0;
    unsigned phase = 0;
    for (int d = 0; d < D && cur.valid; ++d) {
        if (lane == 0) {
            mbar_arrive_expect_tx(&wbar[d], cur.bytes(P));
            bulk_g2s(ring + d * SEG_BYTES, cur.src(P), cur.bytes(P), &wbar[d], pol_w);
        }
        cur.advance(P, warp);
        ++issued;
    }

    // Activations (and every output) depend on the preceding kernel.
    pdl_wait();

    unsigned long long best[T];
#pragma unroll
    for (int t = 0; t < T; ++t) best[t] = 0ull;

    int gi_hint = 0, gi_item = 0;
    unsigned xphase = 0;
    bool x_unconfirmed = false;  // thread 0: an activation copy was issued but not seen complete
    for (long long ra = i0; ra < i1;) {
        const long long rb = run_end(P, ra, i1, gi_hint);
        const Group &g = P.g[gi_hint];
        const int K = g.K, nb = g.nb, N = g.N;
        const int e_run = static_cast<int>(ra - g.item_begin) / g.items_per_inst;

        // ---- this run's activations into shared memory (whole CTA)
        __syncthreads();
        if (tid == 0 && !*abort_flag) {
            x_unconfirmed = true;
            fence_proxy_async_smem();
            const uint8_t *src = g.xq + static_cast<long long>(e_run) * g.xq_stride;
            const unsigned qbytes = static_cast<unsigned>(T * K);
            const unsigned dbytes = static_cast<unsigned>(g.xq_bytes) - qbytes;
            mbar_arrive_expect_tx(xbar, qbytes + dbytes);
            bulk_g2s(xs_q, src, qbytes, xbar, pol_x);
            bulk_g2s(smem + P.off_d, src + qbytes, dbytes, xbar, pol_x);
        }
        const bool xok = mbar_wait_bounded(xbar, xphase, abort_flag, P.status, WAIT_LIMIT_NS);
        if (xok) x_unconfirmed = false;
        xphase ^= 1u;
        if (xok)
            for (int i = tid; i < T * nb; i += nthreads) {
                const int t = i / nb, b = i - t * nb;
                const uint4 *qp = reinterpret_cast<const uint4 *>(xs_q + t * K + b * QK);
                const int c = block_fold_const(qp[0], qp[1]);
                xs_cd[i] = make_int2(c, __float_as_int(h2f(xs_d[i])));
            }
        __syncthreads();

        // ---- this warp's items of the run
        for (long long it = ra + warp; it < rb; it += nw) {
            const ItemInfo inf = decode_item(P, it, gi_item);
            if (inf.bad) {
                if (lane == 0) atomicCAS(P.status, 0u, ST_BAD_ID);
                continue;
            }
            const bool direct = P.ggml || inf.kind != 0;
            const bool split = g.split > 1 && inf.kind == 0;  // a packed tail is never split
            const uint8_t *rows_base =
                inf.kind != 0 ? inf.Wi + static_cast<long long>(g.nslabs) * g.slab_bytes
                              : inf.Wi + static_cast<long long>(inf.slab) * SLAB_ROWS * nb * Q4_BYTES;
            float yv[2][T];
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int t = 0; t < T; ++t) yv[h][t] = 0.0f;

            for (int s = inf.seg0; s < inf.seg1; ++s) {
                float acc[2][T];
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int t = 0; t < T; ++t) acc[h][t] = 0.0f;

                if (direct) {
                    if (xok) segment_from_ggml<T>(rows_base, inf.rows, s, K, nb, r8, j, xs_q, xs_cd, acc);
                } else {
                    const bool ok = mbar_wait_bounded(&wbar[slot], phase, abort_flag, P.status, WAIT_LIMIT_NS);
                    const uint8_t *stage = ring + slot * SEG_BYTES;
                    if (ok && xok) {
                        if (SEG_BLOCKS * (s + 1) <= nb)
                            segment_full_from_stage<T>(stage, s, K, nb, r8, j, xs_q, xs_cd, acc);
                        else
                            segment_from_stage<T>(stage, s, K, nb, r8, j, xs_q, xs_cd, acc);
                    }
                    __syncwarp();
                    const int aborted = __shfl_sync(0xFFFFFFFFu, *abort_flag, 0);
                    if (cur.valid && !aborted) {  // refill the slot just consumed
                        if (lane == 0) {
                            fence_proxy_async_smem();
                            const unsigned nbytes = cur.bytes(P);
                            mbar_arrive_expect_tx(&wbar[slot], nbytes);
                            bulk_g2s(ring + slot * SEG_BYTES, cur.src(P), nbytes, &wbar[slot], pol_w);
                        }
                        cur.advance(P, warp);
                        ++issued;
                    }
                    ++consumed;
                    if (++slot == D) {
                        slot = 0;
                        phase ^= 1u;
                    }
                }
                combine_phases<T>(acc);

                if (split) {
                    // split-K: publish this segment's partial sums
                    float *pb = g.part + ((static_cast<long long>(inf.e) * g.nslabs + inf.slab) * g.nseg + s) * T * 16;
                    if (j == 0) {
#pragma unroll
                        for (int t = 0; t < T; ++t) {
                            pb[t * 16 + r8] = acc[0][t];
                            pb[t * 16 + r8 + 8] = acc[1][t];
                        }
                    }
                } else {
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int t = 0; t < T; ++t) yv[h][t] = (s == 0) ? acc[h][t] : __fadd_rn(yv[h][t], acc[h][t]);
                }
            }

            float *ye = g.y + static_cast<long long>(inf.e) * g.y_stride;
            const int row0 = inf.slab * SLAB_ROWS;
            if (split) {
                __threadfence();
                __syncwarp();
                unsigned old = 0;
                unsigned *cnt = g.cnt + static_cast<long long>(inf.e) * g.nslabs + inf.slab;
                if (lane == 0) old = atomicAdd(cnt, 1u);
                old = __shfl_sync(0xFFFFFFFFu, old, 0);
                if (old == static_cast<unsigned>(g.split - 1)) {
                    __threadfence();
                    const float *pb = g.part + (static_cast<long long>(inf.e) * g.nslabs + inf.slab) * g.nseg * T * 16;
                    if (lane < inf.rows) {
                        const int row = row0 + lane;
#pragma unroll
                        for (int t = 0; t < T; ++t) {
                            float v = __ldcg(pb + t * 16 + lane);
                            for (int s2 = 1; s2 < g.nseg; ++s2) v = __fadd_rn(v, __ldcg(pb + (s2 * T + t) * 16 + lane));
                            if (ye != nullptr) ye[static_cast<long long>(t) * N + row] = v;
                            if (ARGMAX) best[t] = max(best[t], argmax_key(v, static_cast<unsigned>(row)));
                        }
                    }
                    __syncwarp();
                    if (lane == 0) *cnt = 0u;
                }
            } else if (j == 0) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int lr = r8 + 8 * h;
                    if (lr < inf.rows) {
                        const int row = row0 + lr;
#pragma unroll
                        for (int t = 0; t < T; ++t) {
                            if (ye != nullptr) ye[static_cast<long long>(t) * N + row] = yv[h][t];
                            if (ARGMAX) best[t] = max(best[t], argmax_key(yv[h][t], static_cast<unsigned>(row)));
                        }
                    }
                }
            }
        }
        ra = rb;
    }

    // Copies still in flight (only after an abort): wait for them, bounded.
    for (int n = consumed; n < issued; ++n) {
        mbar_drain(&wbar[slot], phase);
        if (++slot == D) {
            slot = 0;
            phase ^= 1u;
        }
    }
    if (x_unconfirmed) mbar_drain(xbar, xphase ^ 1u);

    if (ARGMAX) {
#pragma unroll
        for (int t = 0; t < T; ++t) {
            unsigned long long v = best[t];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const unsigned long long o = __shfl_xor_sync(0xFFFFFFFFu, v, off);
                v = o > v ? o : v;
            }
            if (lane == 0) s_best[warp * T + t] = v;
        }
        __syncthreads();
        if (tid < T) {
            unsigned long long m = 0ull;
            for (int w = 0; w < nw; ++w) m = max(m, s_best[w * T + tid]);
            P.am_cand[static_cast<long long>(blockIdx.x) * T + tid] = m;
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) s_last = (atomicAdd(P.am_cnt, 1u) == gridDim.x - 1) ? 1 : 0;
        __syncthreads();
        if (s_last) {
            __threadfence();
            if (tid < T) {
                unsigned long long m = 0ull;
                for (unsigned c = 0; c < gridDim.x; ++c) m = max(m, __ldcg(P.am_cand + static_cast<long long>(c) * T + tid));
                P.am_idx[tid] = static_cast<long long>(0xFFFFFFFFull - (m & 0xFFFFFFFFull));
            }
            if (tid == 0) *P.am_cnt = 0u;
        }
    }
}

}  // namespace qg
