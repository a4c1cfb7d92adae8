// gemv_kernel.cuh -- the weight-streaming Q4_0 x Q8_0 GEMV kernel.
//
// One persistent CTA per SM (16 warps, or 8 where registers or shared memory
// ask for it).  A launch covers a list of GEMVs ("groups" x "instances");
// their work is cut into items -- one 16-row slab over all of K, or
// (split-K) over one 16-block segment of K -- and the items are dealt to
// CTAs as contiguous ranges of equal weighted bytes (a byte of a group
// whose per-block work costs more counts more).  Inside a CTA the runs
// (items of one group instance) are cut into groups whose activations fit
// shared memory together, and each group's stages are split evenly over the
// warps (balanced mode); split-K launches process runs in turn instead.
//
// Weight bytes reach shared memory through 1-D bulk asynchronous copies
// (TMA, cp.async.bulk) into a per-warp ring of stages (one stage = one
// 16-block segment of a slab = 4608 bytes), each completing on its own
// mbarrier; the next stage is issued as soon as a slot is consumed, so every
// warp keeps ring_depth stages in flight.  The activations of a run are
// copied into shared memory once per CTA (or quantised there from fp32),
// together with each block's folded-offset constant and scale.
//
// One-token lanes (dp4a path; minfer README M15 repacks rows into groups so
// a warp reads contiguous bytes, here 16-row slabs): lane = 4 * r8 + j
// handles rows r8 and r8 + 8 of the slab and the blocks b with b % 4 == j.
// Per block it unpacks the nibbles with two masks (M9: SIMD nibble masking),
// forms the exact integer block sum with dp4a and the folded -8 offset (M9),
// and accumulates (d_w * d_x) * isum with one fp32 fused multiply-add.  At
// the end of a segment the four phases are combined by a fixed two-level
// shuffle tree; segments are added in order.  Several tokens on the tensor
// cores (see "MMA path") keep the same order.  The order depends only on K
// (include/qgemv.h).
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

// ------------------------------------------------------------------ lane outputs
//
// The (row, token) outputs a lane owns.  dp4a lanes (one token): rows r8 and
// r8 + 8 of the slab, every token; the four lanes of a row pair hold equal
// values after the phase combine and lane j == 0 writes.  MMA lanes (T > 1):
// rows g and g + 8, tokens 2j and 2j + 1 -- the accumulator layout of
// mma.m16n8k16 (element k: row g + 8 (k >> 1), token 2j + (k & 1)).
template <int T, bool MMA_>
struct LaneOut {
    static constexpr bool MMA = MMA_;
    static constexpr int N = MMA ? 4 : 2 * T;
    __device__ static __forceinline__ int row(int k, int r8) { return MMA ? r8 + 8 * (k >> 1) : r8 + 8 * (k / T); }
    __device__ static __forceinline__ int tok(int k, int j) { return MMA ? 2 * j + (k & 1) : k % T; }
    __device__ static __forceinline__ bool owner(int k, int j) { return MMA ? (2 * j + (k & 1)) < T : j == 0; }
};

struct XqView {
    const int8_t *q;   // token rows at q + t * xstride
    int xstride;
    const int2 *cd;    // dp4a: per block cdw {folded constant, d_x / 16}; MMA: CD_MMA_QUAD per 4 blocks
    int cdw;
    // tensor-core path: f16 operand image (else int8); this lane's ldmatrix
    // row offsets within a stage, and the shared-memory addresses of its
    // activation rows and constants at block 0
    int f16;
    uint32_t oa1, oa2, osc, xa0, ca0;
};

// The tensor-core lane offsets of an activation image (see mma_segment_full_ldsm).
template <int T>
__device__ __forceinline__ void mma_lane_offsets(XqView &xv, int g, int j)
{
    const int lane = threadIdx.x & 31;
    const int m = lane >> 3, rr = lane & 7;
    const int row = rr + 8 * (m & 1), rot = rr >> 1;
    xv.oa1 = (row * QUAD + (((m >> 1) + rot) & 3)) * 16;
    xv.oa2 = (row * QUAD + (((m >> 1) + 2 + rot) & 3)) * 16;
    xv.osc = 256 * QUAD + g * 16;
    const int tok = T == 8 ? rr : min(rr, T - 1);
    // int8 image: block l >> 4 (+ 2), bytes 16 ((l >> 3) & 1); f16 image:
    // 16-byte chunk l >> 3 of the block's 64 bytes
    xv.xa0 = smem_addr(xv.q + tok * xv.xstride + (xv.f16 ? m * 16 : (m >> 1) * QK + (m & 1) * 16));
    xv.ca0 = smem_addr(xv.cd) + 16 * j;
}

// ------------------------------------------------------------------ dp4a path (T == 1)

// acc[h][t] += (d_w(h) * d_x(t)) * isum for one block b of rows h = 0, 1,
// formed as (d_w * (d_x / 16)) * (16 isum): the same real product, so one
// fused multiply-add rounds it exactly as (d_w * d_x) * isum would.
template <int T>
__device__ __forceinline__ void fma_block(const uint4 &n0, const uint4 &n1, float dw0, float dw1, int b,
                                          const XqView &xv, float (&acc)[2][T])
{
#pragma unroll
    for (int t = 0; t < T; ++t) {
        const uint4 *xp = reinterpret_cast<const uint4 *>(xv.q + t * xv.xstride + b * QK);
        const uint4 qa = xp[0], qb = xp[1];
        const int2 cd = xv.cd[b * xv.cdw + t];
        const int s0 = block_dot16_magic(n0, qa, qb, cd.x);  // MAGIC + 16 isum
        const int s1 = block_dot16_magic(n1, qa, qb, cd.x);
        const float dx = __int_as_float(cd.y);               // d_x / 16 (exact)
        acc[0][t] = __fmaf_rn(__fmul_rn(dw0, dx), magic_to_float(s0), acc[0][t]);
        acc[1][t] = __fmaf_rn(__fmul_rn(dw1, dx), magic_to_float(s1), acc[1][t]);
    }
}

// One segment from a shared-memory stage in the packed quad layout.
template <int T>
__device__ __forceinline__ void segment_from_stage(const uint8_t *stage, int s, int nb, int r8, int j,
                                                   const XqView &xv, float (&acc)[2][T])
{
    const int nbs = min(SEG_BLOCKS, nb - SEG_BLOCKS * s);
#pragma unroll
    for (int qq = 0; qq < SEG_BLOCKS / QUAD; ++qq) {
        const int nbq = min(QUAD, nbs - QUAD * qq);
        if (j < nbq) {
            const uint8_t *q = stage + qq * QUAD_BYTES;
            const int c = quad_chunk(j, r8, nbq);  // rows r8 and r8 + 8 share the rotation
            const uint4 n0 = *reinterpret_cast<const uint4 *>(q + (r8 * nbq + c) * 16);
            const uint4 n1 = *reinterpret_cast<const uint4 *>(q + ((r8 + 8) * nbq + c) * 16);
            const unsigned sc = *reinterpret_cast<const unsigned *>(q + 256 * nbq + (r8 * nbq + j) * 4);
            fma_block<T>(n0, n1, h2f(sc), h2f(sc >> 16), SEG_BLOCKS * s + QUAD * qq + j, xv, acc);
        }
    }
}

// A full segment (16 blocks = 4 full quads): branch-free, every load of the
// segment issued before the arithmetic.
template <int T>
__device__ __forceinline__ void segment_full_from_stage(const uint8_t *stage, int s, int r8, int j,
                                                        const XqView &xv, float (&acc)[2][T])
{
    const int lo = (r8 * QUAD + quad_chunk(j, r8, QUAD)) * 16;
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
        fma_block<T>(n0[qq], n1[qq], h2f(sc[qq]), h2f(sc[qq] >> 16), SEG_BLOCKS * s + QUAD * qq + j, xv, acc);
}

// One segment read directly from GGML-layout rows in global memory (rows of
// the packed tail, or every row when the weights are not packed).
template <int T>
__device__ __forceinline__ void segment_from_ggml(const uint8_t *rows_base, int rows, int s, int nb, int r8, int j,
                                                  const XqView &xv, float (&acc)[2][T])
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
            fma_block<T>(n0, n1, h2f(d0), h2f(d1), b, xv, acc);
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

// ------------------------------------------------------------------ MMA path (T > 1)
//
// Two mma.sync.m16n8k16 (f16 x f16 -> f32) per block form the 16 x 8 block
// sums (16 rows of the slab, 8 token columns, zero past T), scaled by 2^-24.
// Every operand is exact in f16: the nibbles enter as f16 subnormals (the
// masked bits themselves, n 2^-24 or 16 n 2^-24), the activations as small
// integers or integers / 16.  Every product and partial sum is a multiple of
// 2^-24 below 2^-8, so the fp32 accumulator holds isum 2^-24 exactly.
//
// Lane (g, j) supplies word j of rows g and g + 8 (bytes 4j..4j+3: elements
// 4j..4j+3 in the low nibbles, 16+4j..16+4j+3 in the high nibbles) and
// activation words j and 4 + j of token g.  The k index of the first MMA
// runs over the low-nibble elements in the order 4j, 4j+2 (k = 2j, 2j+1) and
// 4j+1, 4j+3 (k = 2j+8, 2j+9); the second MMA the same over the high nibbles.
//   low nibbles:  A = n 2^-24    (one AND: w & 0x000F000F),   B = q
//   high nibbles: A = 16 n 2^-24 (one AND: w & 0x00F000F0),   B = q / 16
// so the MMAs add (sum n q) 2^-24; the first MMA's accumulator input is the
// folded offset C = -8 sum(q) 2^-24 (per token and block) and the second
// ends at isum 2^-24.  Activations, stored as q xor 0x80, become f16
// 1024 + (q xor 0x80) with one PRMT, and one f16x2 add (or fma by 1/16)
// recovers q (or q / 16) exactly.  The lane keeps one fp32 sum per block
// phase (b % 4) and output and adds (d_w * d_x) * (isum 2^-24) with one
// fused multiply-add: d_w * d_x is exact in fp32.  Every value of the
// accumulation is a multiple of 2^-72 (or zero), far above the fp32
// subnormal range, so each rounding is that of the unscaled sum scaled by
// 2^-24; the segment sum is scaled back by 2^24 (exact).  The result is the
// dp4a lanes' (d_w * (d_x / 16)) * (16 isum), rounded the same.

__device__ __forceinline__ void mma_f16(float (&d)[4], unsigned a0, unsigned a1, unsigned a2, unsigned a3,
                                        unsigned b0, unsigned b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ unsigned hadd2_u(unsigned a, unsigned b)
{
    unsigned d;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ unsigned hfma2_u(unsigned a, unsigned b, unsigned c)
{
    unsigned d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

constexpr float MMA_SCALE = 5.9604644775390625e-8f;  // 2^-24
constexpr float MMA_UNSCALE = 16777216.0f;           // 2^24
constexpr unsigned H2_Q_BIAS = 0x64806480u;    // f16x2 1152: 1024 + (q xor 0x80) = 1152 + q
constexpr unsigned H2_NEG_1152 = 0xE480E480u;  // f16x2 (-1152, -1152)
constexpr unsigned H2_SIXTEENTH = 0x2C002C00u; // f16x2 (1/16, 1/16)
constexpr unsigned H2_NEG_72 = 0xD480D480u;    // f16x2 (-72, -72): (1152 + q) / 16 - 72 = q / 16

// Activation bytes 0, 2 (even) or 1, 3 (odd) of a word of the biased image
// (bytes q xor 0x80) as f16x2 1024 + (q xor 0x80) = 1152 + q.
__device__ __forceinline__ unsigned act_even(unsigned w) { return __byte_perm(w, 0x64646464u, 0x4240); }
__device__ __forceinline__ unsigned act_odd(unsigned w) { return __byte_perm(w, 0x64646464u, 0x4341); }

// d0 += c0, d1 += c1: one add.rn.f32x2 (two IEEE additions).
__device__ __forceinline__ void fadd2(float &d0, float &d1, float c0, float c1)
{
    asm("{\n\t.reg .b64 ra, rc;\n\t"
        "mov.b64 ra, {%0, %1};\n\t"
        "mov.b64 rc, {%2, %3};\n\t"
        "add.rn.f32x2 ra, ra, rc;\n\t"
        "mov.b64 {%0, %1}, ra;\n\t}"
        : "+f"(d0), "+f"(d1)
        : "f"(c0), "f"(c1));
}

// 2^24: w >> 8 as the high word of w * 2^24, an integer multiply (FMA pipe)
// rather than a shift (ALU pipe, the busier one on the tensor-core path).
// A constant-bank value, so the compiler keeps the multiply.
__constant__ unsigned c_shr8_mul = 1u << 24;

// acc0 += s0 * d0, acc1 += s1 * d1: one fma.rn.f32x2 (two IEEE fused
// multiply-adds, rounded as two fma.rn.f32 would be).
__device__ __forceinline__ void ffma2(float &a0, float &a1, float s0, float s1, float d0, float d1)
{
    asm("{\n\t.reg .b64 ra, rs, rd;\n\t"
        "mov.b64 ra, {%0, %1};\n\t"
        "mov.b64 rs, {%2, %3};\n\t"
        "mov.b64 rd, {%4, %5};\n\t"
        "fma.rn.f32x2 ra, rs, rd, ra;\n\t"
        "mov.b64 {%0, %1}, ra;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(s0), "f"(s1), "f"(d0), "f"(d1));
}

// The four fp32 products of two fp16 pairs, w = {w0, w1}, x = {x0, x1}:
// w0 x0, w0 x1, w1 x0, w1 x1.  Each product of two fp16 values is exact in
// fp32; fma.rn.f32.f16 with a -0 addend returns it as fp32 multiplication
// of the widened values would.
__device__ __forceinline__ void h2_outer(unsigned w, unsigned x, float &p00, float &p01, float &p10, float &p11)
{
    asm("{\n\t.reg .b16 w0, w1, x0, x1;\n\t"
        "mov.b32 {w0, w1}, %4;\n\t"
        "mov.b32 {x0, x1}, %5;\n\t"
        "fma.rn.f32.f16 %0, w0, x0, %6;\n\t"
        "fma.rn.f32.f16 %1, w0, x1, %6;\n\t"
        "fma.rn.f32.f16 %2, w1, x0, %6;\n\t"
        "fma.rn.f32.f16 %3, w1, x1, %6;\n\t}"
        : "=f"(p00), "=f"(p01), "=f"(p10), "=f"(p11)
        : "r"(w), "r"(x), "f"(-0.0f));
}

// d = A B + C for one m16n8k16 tile with the accumulator start c.
__device__ __forceinline__ void mma_f16_c(float (&d)[4], unsigned a0, unsigned a1, unsigned a2, unsigned a3,
                                          unsigned b0, unsigned b1, const float4 &c)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c.x), "f"(c.y), "f"(c.z), "f"(c.w));
}

// Four 8 x 8 b16 matrices from shared memory; lane l gives the address of
// row l & 7 of matrix l >> 3 and receives word l & 3 of row l >> 2 of each.
__device__ __forceinline__ void ldsm_x4(unsigned &r0, unsigned &r1, unsigned &r2, unsigned &r3, uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ float4 lds_f4(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint4 lds_u4(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ unsigned lds_u32(uint32_t addr)
{
    unsigned v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

// One block for this lane's four outputs from its words: weight word j of
// rows g and g + 8 (wg, wg8), biased activation words j and 4 + j of token g
// (ql, qh), the rows' fp16 scales (sc), the accumulator start cq =
// {C(2j), C(2j+1), C(2j), C(2j+1)} and the fp16 pair {d_x(2j), d_x(2j+1)}.
// The same from the B registers of the two MMAs: (bl0, bl1) = {q} over the
// low-nibble k order, (bh0, bh1) = {q / 16} over the high-nibble k order.
// The block sums alone: d[k] = isum 2^-24 (exact) for row g + 8 (k >> 1),
// token 2j + (k & 1).  Two MMAs over the low and the high nibbles, the first
// starting from the folded offset cq.
__device__ __forceinline__ void mma_block_sums(unsigned wg, unsigned wg8, unsigned bl0, unsigned bl1, unsigned bh0,
                                               unsigned bh1, const float4 &cq, float (&d)[4])
{
    const unsigned g1 = __umulhi(wg, c_shr8_mul), g9 = __umulhi(wg8, c_shr8_mul);  // wg >> 8, wg8 >> 8
    mma_f16_c(d, wg & 0x000F000Fu, wg8 & 0x000F000Fu, g1 & 0x000F000Fu, g9 & 0x000F000Fu, bl0, bl1, cq);
    mma_f16(d, wg & 0x00F000F0u, wg8 & 0x00F000F0u, g1 & 0x00F000F0u, g9 & 0x00F000F0u, bh0, bh1);
}

__device__ __forceinline__ void mma_block_core(unsigned wg, unsigned wg8, unsigned bl0, unsigned bl1, unsigned bh0,
                                               unsigned bh1, unsigned sc, const float4 &cq, unsigned dx, float (&acc)[4])
{
    float d[4];
    mma_block_sums(wg, wg8, bl0, bl1, bh0, bh1, cq, d);
    float s00, s01, s10, s11;  // (d_w d_x) for rows g, g + 8 and tokens 2j, 2j + 1
    h2_outer(sc, dx, s00, s01, s10, s11);
    ffma2(acc[0], acc[1], s00, s01, d[0], d[1]);
    ffma2(acc[2], acc[3], s10, s11, d[2], d[3]);
}

// The B registers of the two MMAs from biased activation words (bytes
// q xor 0x80): ql holds elements 4j..4j+3, qh elements 16+4j..16+4j+3.
__device__ __forceinline__ void mma_b_from_biased(unsigned ql, unsigned qh, unsigned &bl0, unsigned &bl1,
                                                  unsigned &bh0, unsigned &bh1)
{
    bl0 = hadd2_u(act_even(ql), H2_NEG_1152);
    bl1 = hadd2_u(act_odd(ql), H2_NEG_1152);
    bh0 = hfma2_u(act_even(qh), H2_SIXTEENTH, H2_NEG_72);
    bh1 = hfma2_u(act_odd(qh), H2_SIXTEENTH, H2_NEG_72);
}

__device__ __forceinline__ void mma_block_words(unsigned wg, unsigned wg8, unsigned ql, unsigned qh, unsigned sc,
                                                const float4 &cq, unsigned dx, float (&acc)[4])
{
    unsigned bl0, bl1, bh0, bh1;
    mma_b_from_biased(ql, qh, bl0, bl1, bh0, bh1);
    mma_block_core(wg, wg8, bl0, bl1, bh0, bh1, sc, cq, dx, acc);
}

// Shared-memory addresses of block b's constants for lane j (token pair j).
__device__ __forceinline__ uint32_t mma_cq_addr(const XqView &xv, int b)
{
    return xv.ca0 + (b >> 2) * CD_MMA_QUAD + (b & 3) * 64;
}
__device__ __forceinline__ uint32_t mma_dx_addr(const XqView &xv, int b, int j)
{
    return xv.ca0 - 16 * j + (b >> 2) * CD_MMA_QUAD + 256 + (j * 4 + (b & 3)) * 4;
}

template <int T>
__device__ __forceinline__ void mma_block(unsigned wg, unsigned wg8, unsigned sc, int b, int g, int j,
                                          const XqView &xv, float (&acc)[4])
{
    // Token columns past T read token T - 1: a column of B only reaches its
    // own outputs, which no lane stores.
    const int tg = T == 8 ? g : min(g, T - 1);
    const float4 cq = lds_f4(mma_cq_addr(xv, b));
    const unsigned dx = lds_u32(mma_dx_addr(xv, b, j));
    if (xv.f16) {
        const unsigned *xr = reinterpret_cast<const unsigned *>(xv.q + tg * xv.xstride + b * 64);
        mma_block_core(wg, wg8, xr[j], xr[4 + j], xr[8 + j], xr[12 + j], sc, cq, dx, acc);
    } else {
        const unsigned *xr = reinterpret_cast<const unsigned *>(xv.q + tg * xv.xstride + b * QK);
        mma_block_words(wg, wg8, xr[j], xr[4 + j], sc, cq, dx, acc);
    }
}

// The operands of one quad of a full segment (see mma_segment_full_ldsm):
// the ldmatrix words (weights w, activations x) and the per-block constants.
struct MmaWords {
    unsigned w[8], x[8];
};
struct MmaConsts {
    uint4 sc, dx;
    float4 cq[4];
};

// Quad qq of the segment whose stage starts at shared address st and whose
// first block is b0 (a multiple of 16).
__device__ __forceinline__ void mma_quad_words(MmaWords &o, const XqView &xv, uint32_t st, int b0, int qq)
{
    const uint32_t q = st + qq * QUAD_BYTES;
    ldsm_x4(o.w[0], o.w[1], o.w[2], o.w[3], q + xv.oa1);
    ldsm_x4(o.w[4], o.w[5], o.w[6], o.w[7], q + xv.oa2);
    const uint32_t xa = xv.xa0 + (b0 + QUAD * qq) * QK;
    ldsm_x4(o.x[0], o.x[1], o.x[2], o.x[3], xa);
    ldsm_x4(o.x[4], o.x[5], o.x[6], o.x[7], xa + 2 * QK);
}

__device__ __forceinline__ void mma_quad_consts(MmaConsts &o, const XqView &xv, uint32_t st, int b0, int qq)
{
    o.sc = lds_u4(st + qq * QUAD_BYTES + xv.osc);
    const uint32_t cq = xv.ca0 + (b0 / QUAD + qq) * CD_MMA_QUAD;
#pragma unroll
    for (int jq = 0; jq < QUAD; ++jq) o.cq[jq] = lds_f4(cq + jq * 64);
    o.dx = lds_u4(cq + 256);  // ca0 includes 16 j: the pair's d_x for the quad's four blocks
}

// The weight words of quad qq only (f16 operand image).
__device__ __forceinline__ void mma_quad_weights(MmaWords &o, const XqView &xv, uint32_t st, int qq)
{
    const uint32_t q = st + qq * QUAD_BYTES;
    ldsm_x4(o.w[0], o.w[1], o.w[2], o.w[3], q + xv.oa1);
    ldsm_x4(o.w[4], o.w[5], o.w[6], o.w[7], q + xv.oa2);
}

// One quad on the f16 operand image: one ldmatrix.x4 per block gives the
// four B registers of its two MMAs (chunk c of the block's 64 bytes).
__device__ __forceinline__ void mma_quad_compute_f16(const MmaWords &o, const MmaConsts &c, const XqView &xv, int bq,
                                                     float (&acc)[4][4])
{
    const unsigned sc[4] = {c.sc.x, c.sc.y, c.sc.z, c.sc.w};
    const unsigned dx[4] = {c.dx.x, c.dx.y, c.dx.z, c.dx.w};
#pragma unroll
    for (int jq = 0; jq < QUAD; ++jq) {
        unsigned x0, x1, x2, x3;
        ldsm_x4(x0, x1, x2, x3, xv.xa0 + (bq + jq) * 64);
        mma_block_core(o.w[2 * jq], o.w[2 * jq + 1], x0, x1, x2, x3, sc[jq], c.cq[jq], dx[jq], acc[jq]);
    }
}

__device__ __forceinline__ void mma_quad_compute(const MmaWords &o, const MmaConsts &c, float (&acc)[4][4])
{
    mma_block_words(o.w[0], o.w[1], o.x[0], o.x[1], c.sc.x, c.cq[0], c.dx.x, acc[0]);
    mma_block_words(o.w[2], o.w[3], o.x[2], o.x[3], c.sc.y, c.cq[1], c.dx.y, acc[1]);
    mma_block_words(o.w[4], o.w[5], o.x[4], o.x[5], c.sc.z, c.cq[2], c.dx.z, acc[2]);
    mma_block_words(o.w[6], o.w[7], o.x[6], o.x[7], c.sc.w, c.cq[3], c.dx.w, acc[3]);
}

// A full segment from a stage in the packed layout, with ldmatrix: per quad
// one x4 load brings weight word j of rows g and g + 8 of two blocks, one
// more the other two blocks, and two more the activation words of the four
// blocks.  Lane l names, for the weights, row (l & 7) + 8 ((l >> 3) & 1) of
// block l >> 4 (+ 2 in the second load); for the activations, token
// min(l & 7, T - 1) of block l >> 4 (+ 2), bytes 16 ((l >> 3) & 1) onwards.
// The rotation keeps each group of eight 16-byte rows in distinct banks.
// On the f16 operand image one x4 load per block gives its B registers.
template <int T>
__device__ __forceinline__ void mma_segment_full_ldsm(const uint8_t *stage, int s, const XqView &xv,
                                                      float (&acc)[4][4])
{
    const uint32_t st = smem_addr(stage);
    const int b0 = SEG_BLOCKS * s;
    if (xv.f16) {
#pragma unroll 1
        for (int qq = 0; qq < SEG_BLOCKS / QUAD; ++qq) {
            MmaWords w;
            MmaConsts c;
            mma_quad_weights(w, xv, st, qq);
            mma_quad_consts(c, xv, st, b0, qq);
            mma_quad_compute_f16(w, c, xv, b0 + QUAD * qq, acc);
        }
        return;
    }
#pragma unroll 1
    for (int qq = 0; qq < SEG_BLOCKS / QUAD; ++qq) {
        MmaWords w;
        MmaConsts c;
        mma_quad_words(w, xv, st, b0, qq);
        mma_quad_consts(c, xv, st, b0, qq);
        mma_quad_compute(w, c, acc);
    }
}

// One segment from a stage; `full` segments (16 blocks) take the branch-free form.
template <int T>
__device__ __forceinline__ void mma_segment_from_stage(const uint8_t *stage, bool full, int s, int nb, int g, int j,
                                                       const XqView &xv, float (&acc)[4][4])
{
    if (full) {
        mma_segment_full_ldsm<T>(stage, s, xv, acc);
        return;
    }
    const int nbs = min(SEG_BLOCKS, nb - SEG_BLOCKS * s);
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) {
        const int nbq = min(QUAD, nbs - QUAD * qq);
        const uint8_t *q = stage + qq * QUAD_BYTES;
#pragma unroll
        for (int jq = 0; jq < 4; ++jq)
            if (jq < nbq) {  // warp-uniform
                const int c = quad_chunk(jq, g, nbq);
                const unsigned wg = *reinterpret_cast<const unsigned *>(q + (g * nbq + c) * 16 + 4 * j);
                const unsigned wg8 = *reinterpret_cast<const unsigned *>(q + ((g + 8) * nbq + c) * 16 + 4 * j);
                const unsigned sc = *reinterpret_cast<const unsigned *>(q + 256 * nbq + (g * nbq + jq) * 4);
                mma_block<T>(wg, wg8, sc, SEG_BLOCKS * s + QUAD * qq + jq, g, j, xv, acc[jq]);
            }
    }
}

__device__ __forceinline__ unsigned ldg_u32_a2(const uint8_t *p)  // 2-byte aligned 32-bit load
{
    const unsigned short *h = reinterpret_cast<const unsigned short *>(p);
    return static_cast<unsigned>(__ldg(h)) | (static_cast<unsigned>(__ldg(h + 1)) << 16);
}

template <int T>
__device__ __forceinline__ void mma_segment_from_ggml(const uint8_t *rows_base, int rows, int s, int nb, int g, int j,
                                                      const XqView &xv, float (&acc)[4][4])
{
    const int nbs = min(SEG_BLOCKS, nb - SEG_BLOCKS * s);
    const long long row_bytes = static_cast<long long>(nb) * Q4_BYTES;
#pragma unroll 1
    for (int qq = 0; qq < 4; ++qq) {
#pragma unroll
        for (int jq = 0; jq < 4; ++jq) {  // static phase index: accumulators stay in registers
            const int i = QUAD * qq + jq;
            if (i < nbs) {                // warp-uniform
                const int b = SEG_BLOCKS * s + i;
                unsigned wg = 0, wg8 = 0, d0 = 0, d1 = 0;
                if (g < rows) {
                    const uint8_t *p = rows_base + g * row_bytes + b * Q4_BYTES;
                    d0 = __ldg(reinterpret_cast<const unsigned short *>(p));
                    wg = ldg_u32_a2(p + 2 + 4 * j);
                }
                if (g + 8 < rows) {
                    const uint8_t *p = rows_base + (g + 8) * row_bytes + b * Q4_BYTES;
                    d1 = __ldg(reinterpret_cast<const unsigned short *>(p));
                    wg8 = ldg_u32_a2(p + 2 + 4 * j);
                }
                mma_block<T>(wg, wg8, d0 | (d1 << 16), b, g, j, xv, acc[jq]);
            }
        }
    }
}

// ------------------------------------------------------------------ either path

// The ordered sum of one segment for this lane's outputs.
template <int T, bool MMA>
__device__ __forceinline__ void segment_sum(bool from_stage, const uint8_t *stage, const uint8_t *rows_base, int rows,
                                            int s, int nb, int r8, int j, const XqView &xv,
                                            float (&P)[LaneOut<T, MMA>::N])
{
    const bool full = SEG_BLOCKS * (s + 1) <= nb;
    if constexpr (MMA) {
        float acc[4][4];
#pragma unroll
        for (int p = 0; p < 4; ++p)
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[p][k] = 0.0f;
        if (from_stage)
            mma_segment_from_stage<T>(stage, full, s, nb, r8, j, xv, acc);
        else
            mma_segment_from_ggml<T>(rows_base, rows, s, nb, r8, j, xv, acc);
#pragma unroll
        for (int k = 0; k < 4; k += 2) {  // (s0 + s1) + (s2 + s3), two outputs per add.rn.f32x2
            float u0 = acc[0][k], u1 = acc[0][k + 1], v0 = acc[2][k], v1 = acc[2][k + 1];
            fadd2(u0, u1, acc[1][k], acc[1][k + 1]);
            fadd2(v0, v1, acc[3][k], acc[3][k + 1]);
            fadd2(u0, u1, v0, v1);
            P[k] = __fmul_rn(u0, MMA_UNSCALE);  // exact: back from the 2^-24 scale
            P[k + 1] = __fmul_rn(u1, MMA_UNSCALE);
        }
    } else {
        float acc[2][T];
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int t = 0; t < T; ++t) acc[h][t] = 0.0f;
        if (from_stage) {
            if (full)
                segment_full_from_stage<T>(stage, s, r8, j, xv, acc);
            else
                segment_from_stage<T>(stage, s, nb, r8, j, xv, acc);
        } else {
            segment_from_ggml<T>(rows_base, rows, s, nb, r8, j, xv, acc);
        }
        combine_phases<T>(acc);
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int t = 0; t < T; ++t) P[h * T + t] = acc[h][t];
    }
}

// The tensor-core accumulator start of one token's block: the folded
// offset -8 sum(q), at the 2^-24 scale of the subnormal nibble operands.
__device__ __forceinline__ float mma_fold_const(int sum_q)
{
    return __fmul_rn(static_cast<float>(-8 * sum_q), MMA_SCALE);  // exact: |8 sum(q)| < 2^15
}

// Tensor-core constants of block b, token t: C into both slots of the
// pair's accumulator start, the raw fp16 d_x into the pair's d_x word.
__device__ __forceinline__ void mma_store_consts(uint8_t *cd, int b, int t, float C, unsigned short dx)
{
    uint8_t *q = cd + (b >> 2) * CD_MMA_QUAD;
    float *cq = reinterpret_cast<float *>(q + (b & 3) * 64 + (t >> 1) * 16);
    cq[t & 1] = C;
    cq[2 + (t & 1)] = C;
    reinterpret_cast<unsigned short *>(q + 256 + ((t >> 1) * 4 + (b & 3)) * 4)[t & 1] = dx;
}

// Builds one run's activation image in shared memory after its copy landed:
// per block and token the folded constant and the activation scale.  dp4a
// path: {MAGIC - 128 sum(q), d_x / 16} per token; MMA path: the activation
// bytes are rewritten as q xor 0x80, and each token's accumulator start
// C = -8 sum(q) 2^-24 (fp32, mma_fold_const) and fp16 d_x go to the
// CD_MMA_QUAD layout, with zeros for the token columns past T.
template <int T, bool MMA>
__device__ __forceinline__ void build_fold_constants(uint8_t *img, int K, int tid, int nthreads)
{
    const XqLayout L = xq_layout(T, K, MMA);
    const int nb = K / QK;
    const int8_t *xq = reinterpret_cast<const int8_t *>(img);
    int8_t *xq_w = reinterpret_cast<int8_t *>(img);
    const unsigned short *xd = reinterpret_cast<const unsigned short *>(img + L.off_d);
    int2 *cd = reinterpret_cast<int2 *>(img + L.off_cd);
    for (int i = tid; i < L.cdw * nb; i += nthreads) {
        const int b = i / L.cdw, t = i - b * L.cdw;
        if (t < T) {
            const uint4 *qp = reinterpret_cast<const uint4 *>(xq + t * L.xstride + b * QK);
            const float dx = h2f(xd[t * nb + b]);
            if constexpr (MMA) {
                const uint4 qa = qp[0], qb = qp[1];
                uint4 *qw = reinterpret_cast<uint4 *>(xq_w + t * L.xstride + b * QK);
                const unsigned flip = 0x80808080u;  // the MMA operands read q xor 0x80
                qw[0] = make_uint4(qa.x ^ flip, qa.y ^ flip, qa.z ^ flip, qa.w ^ flip);
                qw[1] = make_uint4(qb.x ^ flip, qb.y ^ flip, qb.z ^ flip, qb.w ^ flip);
                const int ones = 0x01010101;
                int slo = 0, shi = 0;
                slo = dp4a_ss((int)qa.x, ones, slo);
                slo = dp4a_ss((int)qa.y, ones, slo);
                slo = dp4a_ss((int)qa.z, ones, slo);
                slo = dp4a_ss((int)qa.w, ones, slo);
                shi = dp4a_ss((int)qb.x, ones, shi);
                shi = dp4a_ss((int)qb.y, ones, shi);
                shi = dp4a_ss((int)qb.z, ones, shi);
                shi = dp4a_ss((int)qb.w, ones, shi);
                mma_store_consts(img + L.off_cd, b, t, mma_fold_const(slo + shi), xd[t * nb + b]);
            } else {
                cd[i] = make_int2(block_fold16_const(qp[0], qp[1]), __float_as_int(__fmul_rn(dx, 0.0625f)));
            }
        } else if constexpr (MMA) {
            mma_store_consts(img + L.off_cd, b, t, 0.0f, 0);
        } else {
            cd[i] = make_int2(MAGIC_I, 0);
        }
    }
}

// One run's int8 activation image quantised in the kernel from fp32
// activations x[T][K] in global memory, with its per-block constants, in one
// pass, for images of at most nthreads / 8 blocks: the bytes a copy of the
// planar Q8_0 activations followed by build_fold_constants would leave (codes
// at row t * xstride -- rewritten as q xor 0x80 on the tensor-core path --
// fp16 scales at off_d, constants at off_cd).  Eight consecutive threads take
// one block, four values each; the block maximum and the code sum are
// combined with shuffles inside the eight-lane group (the maximum is exact in
// any order, so every byte equals the standalone quantiser's).  nthreads is a
// multiple of 32, so each group lies in one warp.
template <int T, bool MMA>
__device__ __forceinline__ void quantize_image_small(uint8_t *img, const float *x, int K, int tid, int nthreads)
{
    const XqLayout L = xq_layout(T, K, MMA);
    const int nb = K / QK;
    const bool act = tid < T * nb * 8;  // eight-lane groups are wholly in or out
    const int blk = (act ? tid : 0) >> 3, sub = tid & 7;
    const int t = blk / nb, b = blk - t * nb;
    const float *xp = x + static_cast<long long>(t) * K + b * QK + 4 * sub;
    float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (act) {
        if ((reinterpret_cast<uintptr_t>(x) & 15) == 0) {
            v = __ldcg(reinterpret_cast<const float4 *>(xp));
        } else {
            v.x = __ldcg(xp);
            v.y = __ldcg(xp + 1);
            v.z = __ldcg(xp + 2);
            v.w = __ldcg(xp + 3);
        }
    }
    float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 4));
    float d, id;
    q8_scale(amax, d, id);
    const int c0 = q8_code(v.x, id), c1 = q8_code(v.y, id), c2 = q8_code(v.z, id), c3 = q8_code(v.w, id);
    int sq = c0 + c1 + c2 + c3;
    sq += __shfl_xor_sync(0xFFFFFFFFu, sq, 1);
    sq += __shfl_xor_sync(0xFFFFFFFFu, sq, 2);
    sq += __shfl_xor_sync(0xFFFFFFFFu, sq, 4);
    if (act) {
        unsigned w = (static_cast<unsigned>(c0) & 0xFFu) | ((static_cast<unsigned>(c1) & 0xFFu) << 8) |
                     ((static_cast<unsigned>(c2) & 0xFFu) << 16) | ((static_cast<unsigned>(c3) & 0xFFu) << 24);
        if (MMA) w ^= 0x80808080u;  // the MMA operands read q xor 0x80
        *reinterpret_cast<unsigned *>(img + t * L.xstride + b * QK + 4 * sub) = w;
        if (sub == 0) {
            const unsigned short dh = q8_half(d);
            reinterpret_cast<unsigned short *>(img + L.off_d)[t * nb + b] = dh;
            if constexpr (MMA)
                mma_store_consts(img + L.off_cd, b, t, mma_fold_const(sq), dh);
            else
                reinterpret_cast<int2 *>(img + L.off_cd)[b * L.cdw + t] =
                    make_int2(MAGIC_I - 128 * sq, __float_as_int(__fmul_rn(h2f(dh), 0.0625f)));
        }
    }
    if constexpr (MMA && T < 8)  // token columns past T: zero constants
        for (int i = tid; i < (8 - T) * nb; i += nthreads) {
            const int bb = i / (8 - T), tt = T + (i - bb * (8 - T));
            mma_store_consts(img + L.off_cd, bb, tt, 0.0f, 0);
        }
}

// The codes and scales of one run's int8 activation image quantised in the
// kernel from fp32 activations x[T][K] in global memory, one block per
// thread: the bytes a copy of the planar Q8_0 activations would bring (codes
// at row t * xstride, fp16 scales at off_d); build_fold_constants follows.
template <int T, bool MMA>
__device__ __forceinline__ void quantize_image_codes(uint8_t *img, const float *x, int K, int tid, int nthreads)
{
    const XqLayout L = xq_layout(T, K, MMA);
    const int nb = K / QK;
    const bool vec = (reinterpret_cast<uintptr_t>(x) & 15) == 0;
    unsigned short *xd = reinterpret_cast<unsigned short *>(img + L.off_d);
    for (int i = tid; i < T * nb; i += nthreads) {
        const int t = i / nb, b = i - t * nb;
        uint4 qa, qb;
        unsigned short dh;
        q8_block_thread(x + static_cast<long long>(t) * K + b * QK, vec, qa, qb, dh);
        uint4 *dst = reinterpret_cast<uint4 *>(img + t * L.xstride + b * QK);
        dst[0] = qa;
        dst[1] = qb;
        xd[t * nb + b] = dh;
    }
}

// One run's int8 activation image (codes, scales and constants) quantised
// in the kernel from fp32 activations: small images in one pass of eight
// threads per block, larger ones one block per thread and then the
// constants.  The bytes are the same either way.
template <int T, bool MMA>
__device__ __forceinline__ void quantize_image(uint8_t *img, const float *x, int K, int tid, int nthreads)
{
    if (T * (K / QK) * 8 <= nthreads) {
        quantize_image_small<T, MMA>(img, x, K, tid, nthreads);
    } else {
        quantize_image_codes<T, MMA>(img, x, K, tid, nthreads);
        __syncthreads();
        build_fold_constants<T, MMA>(img, K, tid, nthreads);
    }
}

// One token's block of the f16 operand image: from its codes (qa: elements
// 0..15, qb: 16..31) the 16 words {q[e(k)] : k = 0..7}, {q[e(k)] : k =
// 8..15}, {q[16 + e(k)] / 16 : k = 0..7}, {q[16 + e(k)] / 16 : k = 8..15}
// (e as below), each value exact in f16.
__device__ __forceinline__ void f16_block_words(const uint4 &qa, const uint4 &qb, unsigned (&w)[16])
{
    const int8_t *qlo = reinterpret_cast<const int8_t *>(&qa);
    const int8_t *qhi = reinterpret_cast<const int8_t *>(&qb);
#pragma unroll
    for (int k = 0; k < 16; k += 2) {
        const int i0 = 4 * ((k & 7) >> 1) + (k >> 3);  // e(k); e(k + 1) = e(k) + 2
        const __half2 lo = __floats2half2_rn(static_cast<float>(qlo[i0]), static_cast<float>(qlo[i0 + 2]));
        const __half2 hi = __floats2half2_rn(static_cast<float>(qhi[i0]) * 0.0625f,
                                             static_cast<float>(qhi[i0 + 2]) * 0.0625f);
        w[k >> 1] = *reinterpret_cast<const unsigned *>(&lo);
        w[8 + (k >> 1)] = *reinterpret_cast<const unsigned *>(&hi);
    }
}

// Builds one run's f16 operand image (tensor-core path, small images)
// straight from the planar Q8_0 activations in global memory (F32: from fp32
// activations, quantised here by q8_block_thread): per token row
// and block 64 bytes, the chunks {q[e(k)] : k = 0..7}, {q[e(k)] : k = 8..15},
// {q[16 + e(k)] / 16 : k = 0..7}, {q[16 + e(k)] / 16 : k = 8..15} with
// e(2i) = 4i, e(2i+1) = 4i+2, e(2i+8) = 4i+1, e(2i+9) = 4i+3 (the MMA k
// order of the weight words), plus the constants of build_fold_constants.
// Every value is an integer, or one over 16, held exactly in f16.
template <int T, bool F32>
__device__ __forceinline__ void build_f16_image(uint8_t *img, const uint8_t *src, int K, int tid, int nthreads)
{
    const XqLayout L = xq_layout(T, K, true);
    const int nb = K / QK;
    const unsigned short *xd = reinterpret_cast<const unsigned short *>(src + T * K);
    const bool vec = (reinterpret_cast<uintptr_t>(src) & 15) == 0;
    for (int i = tid; i < 8 * nb; i += nthreads) {
        const int t = i / nb, b = i - t * nb;
        if (t < T) {
            uint4 qa, qb;
            unsigned short dh;
            if constexpr (F32) {
                q8_block_thread(reinterpret_cast<const float *>(src) + static_cast<long long>(t) * K + b * QK, vec, qa, qb,
                                dh);
            } else {
                const uint4 *qp = reinterpret_cast<const uint4 *>(src + static_cast<long long>(t) * K + b * QK);
                qa = __ldcg(qp);
                qb = __ldcg(qp + 1);
                dh = __ldcg(xd + static_cast<long long>(t) * nb + b);
            }
            unsigned w[16];
            f16_block_words(qa, qb, w);
            uint4 *dst = reinterpret_cast<uint4 *>(img + t * L.xstride + b * 64);
#pragma unroll
            for (int c = 0; c < 4; ++c) dst[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
            const int ones = 0x01010101;
            int slo = 0, shi = 0;
            slo = dp4a_ss((int)qa.x, ones, slo);
            slo = dp4a_ss((int)qa.y, ones, slo);
            slo = dp4a_ss((int)qa.z, ones, slo);
            slo = dp4a_ss((int)qa.w, ones, slo);
            shi = dp4a_ss((int)qb.x, ones, shi);
            shi = dp4a_ss((int)qb.y, ones, shi);
            shi = dp4a_ss((int)qb.z, ones, shi);
            shi = dp4a_ss((int)qb.w, ones, shi);
            mma_store_consts(img + L.off_cd, b, t, mma_fold_const(slo + shi), dh);
        } else {
            mma_store_consts(img + L.off_cd, b, t, 0.0f, 0);
        }
    }
}

// Copies one run's activations (planar Q8_0, T rows of K) into an image;
// one copy per token row on the MMA path (padded rows).  Returns the bytes.
template <int T, bool MMA>
__device__ __forceinline__ unsigned copy_activations(uint8_t *img, const uint8_t *src, int K, unsigned dbytes,
                                                     uint64_t *bar, uint64_t pol)
{
    const XqLayout L = xq_layout(T, K, MMA);
    if (L.xstride == K) {
        bulk_g2s(img, src, static_cast<unsigned>(T * K), bar, pol);
    } else {
#pragma unroll
        for (int t = 0; t < T; ++t) bulk_g2s(img + t * L.xstride, src + t * K, static_cast<unsigned>(K), bar, pol);
    }
    bulk_g2s(img + L.off_d, src + T * K, dbytes, bar, pol);
    return static_cast<unsigned>(T * K) + dbytes;
}


// Warps per CTA a T-token kernel may use: 16 (128 registers per thread),
// except the dp4a path above four tokens, whose per-token accumulators need
// more registers (8 warps).  Measured at three and four tokens: 16 warps at
// 128 registers, with a few spilled words, beat 8 warps without spills.
__host__ __device__ constexpr int max_warps_for(int T, bool mma) { return (mma || T <= 4) ? NWARPS_MAX : 8; }

// ------------------------------------------------------------------ balanced mode
//
// When a CTA's runs (consecutive items of one GEMV instance) all fit their
// activations in shared memory at once, the CTA loads them all up front and
// splits its stages (16-block segments) evenly over its warps: warp w takes
// the contiguous stages [S w / nw, S (w + 1) / nw).  A slab cut by such a
// boundary keeps the fixed summation order: the warp holding its first
// segments processes them first and leaves their ordered sum H in shared
// memory; the warp holding the rest processes them last, continuing the
// ordered sum from H.  Each warp therefore walks: its boundary head, its
// whole slabs, its boundary tail.

constexpr int MAX_RUNS = 32;
constexpr long long WARM_L2_BYTES = 262144;  // L2 warm-up per CTA (bytes)
constexpr int WARM_L2_PIECE = 16384;
static_assert(GCACHE_GROUPS >= MAX_RUNS, "a balanced CTA's groups must fit the descriptor cache");

struct RunInfo {
    const uint8_t *Wi;  // instance weights (expert resolved)
    float *y;           // instance output
    int stage0;         // CTA-local index of the run's first stage
    int nstages;        // stages of the run in this CTA (items * nseg)
    int first_local;    // index of the run's first item within its instance
    int gi, e;          // group, instance (slot)
    int nseg, nb, K, N, nslabs;
    int xq_off;         // shared-memory offset of the run's activations
    int bad;            // gather slot with an expert id out of range
};

// Walks CTA-local stages over up to three intervals, in order, keeping the
// position (run r, item ii of the run, segment s) and the current run's
// fields in registers; the run table is read only when the run changes.
struct Walker {
    int k, kend, iv;             // current stage, end of the current interval, interval index
    int b1, e1, b2, e2;          // intervals 1 and 2
    int r, ii, s, item_end, run_end_k;
    int nseg, nb, first_local, nslabs, bad;
    const uint8_t *Wi;
    bool valid;

    __device__ __forceinline__ void load_run(const RunInfo *runs)
    {
        const RunInfo &R = runs[r];
        run_end_k = R.stage0 + R.nstages;
        nseg = R.nseg;
        nb = R.nb;
        first_local = R.first_local;
        nslabs = R.nslabs;
        bad = R.bad;
        Wi = R.Wi;
    }

    __device__ __forceinline__ void locate(const RunInfo *runs)
    {
        while (k >= runs[r].stage0 + runs[r].nstages) ++r;
        while (k < runs[r].stage0) --r;
        load_run(runs);
        const int ks = k - runs[r].stage0;
        ii = ks / nseg;
        s = ks - ii * nseg;
        item_end = k - s + nseg;
    }

    __device__ __forceinline__ bool enter(const RunInfo *runs, int b, int e)
    {
        k = b;
        kend = e;
        if (b >= e) return false;
        locate(runs);
        return true;
    }

    __device__ __forceinline__ void next_interval(const RunInfo *runs)
    {
        valid = false;
        while (iv < 2) {
            ++iv;
            if (enter(runs, iv == 1 ? b1 : b2, iv == 1 ? e1 : e2)) {
                valid = true;
                return;
            }
        }
    }

    __device__ __forceinline__ void init(const RunInfo *runs, int b0, int e0, int b1_, int e1_, int b2_, int e2_)
    {
        b1 = b1_;
        e1 = e1_;
        b2 = b2_;
        e2 = e2_;
        iv = 0;
        r = 0;
        valid = enter(runs, b0, e0);
        if (!valid) next_interval(runs);
    }

    // Jump to the start of the next item (or the next interval).
    __device__ __forceinline__ void next_item(const RunInfo *runs)
    {
        if (item_end >= kend) {
            next_interval(runs);
            return;
        }
        k = item_end;
        s = 0;
        if (k >= run_end_k) {
            ++r;
            load_run(runs);
            ii = 0;
        } else {
            ++ii;
        }
        item_end = k + nseg;
    }

    // One stage forward.
    __device__ __forceinline__ void step(const RunInfo *runs)
    {
        if (k + 1 == item_end || k + 1 >= kend) {
            next_item(runs);
            return;
        }
        ++k;
        ++s;
    }

    __device__ __forceinline__ bool item_is_tma(bool ggml) const { return !ggml && !bad && first_local + ii < nslabs; }

    __device__ __forceinline__ void skip_untransferred(const RunInfo *runs, bool ggml)
    {
        while (valid && !item_is_tma(ggml)) next_item(runs);
    }

    __device__ __forceinline__ const uint8_t *src() const
    {
        return Wi + static_cast<long long>(first_local + ii) * SLAB_COL_BYTES * nb + static_cast<long long>(s) * SEG_BYTES;
    }

    __device__ __forceinline__ unsigned bytes() const
    {
        return static_cast<unsigned>(SLAB_COL_BYTES * min(SEG_BLOCKS, nb - SEG_BLOCKS * s));
    }
};

// Per-warp ring of TMA stages: slot / phase of the next stage to consume.
struct Ring {
    uint8_t *base;
    uint64_t *bar;
    int D, slot, issued, consumed;
    unsigned phase;

    __device__ __forceinline__ uint8_t *stage() const { return base + slot * SEG_BYTES; }

    __device__ __forceinline__ void issue(int lane, int into, const uint8_t *src, unsigned nbytes, uint64_t pol)
    {
        if (lane == 0) {
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&bar[into], nbytes);
            bulk_g2s(base + into * SEG_BYTES, src, nbytes, &bar[into], pol);
        }
        ++issued;
    }

    __device__ __forceinline__ void pop()
    {
        ++consumed;
        if (++slot == D) {
            slot = 0;
            phase ^= 1u;
        }
    }

    __device__ __forceinline__ void drain()
    {
        while (consumed < issued) {
            mbar_drain(&bar[slot], phase);
            pop();
        }
    }
};

// Top-2 of distinct 64-bit keys (0 = none): push one key, or merge another
// pair.  Merging is associative and exact, so every order of merges gives
// the same pair.
__device__ __forceinline__ void top2_push(unsigned long long &b1, unsigned long long &b2, unsigned long long key)
{
    const unsigned long long lo = b1 < key ? b1 : key;
    b1 = b1 < key ? key : b1;
    b2 = b2 < lo ? lo : b2;
}
__device__ __forceinline__ void top2_merge(unsigned long long &b1, unsigned long long &b2, unsigned long long c1,
                                           unsigned long long c2)
{
    top2_push(b1, b2, c1);
    b2 = b2 < c2 ? c2 : b2;
}
__device__ __forceinline__ void top2_warp(unsigned long long &b1, unsigned long long &b2)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const unsigned long long o1 = __shfl_xor_sync(0xFFFFFFFFu, b1, off);
        const unsigned long long o2 = __shfl_xor_sync(0xFFFFFFFFu, b2, off);
        top2_merge(b1, b2, o1, o2);
    }
}

// Row and value of a key (argmax_key's inverse; -0 came in as +0).
__device__ __forceinline__ long long key_row(unsigned long long k)
{
    return k ? static_cast<long long>(0xFFFFFFFFull - (k & 0xFFFFFFFFull)) : -1ll;
}
__device__ __forceinline__ float key_value(unsigned long long k)
{
    if (!k) return -__int_as_float(0x7F800000);
    const unsigned u = static_cast<unsigned>(k >> 32);
    return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}

// A lane's two best keys for the tokens it tracks.  Lane (r8, j) tracks the
// tokens t with jt(t) == j: on the tensor-core path the tokens it computes,
// 2j and 2j + 1; on the dp4a path, where the four lanes of a row pair hold
// the same outputs, t = j, j + 4.  Slot indices are compile-time constants.
template <int T, bool MMA>
struct Top2Lane {
    static constexpr int S = MMA ? 2 : (T + 3) / 4;
    __host__ __device__ static constexpr int jt(int t) { return MMA ? t >> 1 : t & 3; }
    __host__ __device__ static constexpr int slot(int t) { return MMA ? t & 1 : t >> 2; }
    __host__ __device__ static constexpr int token(int sl, int j) { return MMA ? 2 * j + sl : 4 * sl + j; }
    unsigned long long b1[S], b2[S];
};

// The output epilogue of a sequence launch (minfer README M19: the QKV bias
// and the residual adds run in the GEMV's epilogue): y = (v + bias[row]) +
// residual[t][row], each add an fp32 operation rounded to nearest; either
// term may be absent.  The residual is read with a plain load: it may be y
// itself, read and then written by this thread.
__device__ __forceinline__ float apply_epilogue(float v, const float *bias, const float *res, long long yi, int row)
{
    if (bias != nullptr) v = __fadd_rn(v, __ldg(bias + row));
    if (res != nullptr) v = __fadd_rn(v, res[yi]);
    return v;
}

// Write this lane's finished outputs (rows below `rows`) and fold them into
// the top-2 keys of their tokens.  bias / res: the sequence epilogue (or nullptr).
template <int T, bool MMA, bool ARGMAX>
__device__ __forceinline__ void store_outputs(float *ye, int N, int row0, int rows, int r8, int j,
                                              const float (&yv)[LaneOut<T, MMA>::N], Top2Lane<T, MMA> &st,
                                              const float *bias = nullptr, const float *res = nullptr)
{
    using LO = LaneOut<T, MMA>;
    using TL2 = Top2Lane<T, MMA>;
#pragma unroll
    for (int k = 0; k < LO::N; ++k) {
        const int lr = LO::row(k, r8), t = LO::tok(k, j);
        if (lr >= rows) continue;
        if (LO::owner(k, j) && ye != nullptr) {
            const long long yi = static_cast<long long>(t) * N + row0 + lr;
            ye[yi] = ARGMAX ? yv[k] : apply_epilogue(yv[k], bias, res, yi, row0 + lr);
        }
        // static slot: (k & 1) on the tensor-core path, (k % T) / 4 on dp4a
        const int sl = MMA ? (k & 1) : ((k % T) >> 2);
        if (ARGMAX && t < T && (MMA || TL2::jt(k % T) == j))
            top2_push(st.b1[sl], st.b2[sl], argmax_key(yv[k], static_cast<unsigned>(row0 + lr)));
    }
}

// The epilogue's terms of this lane's outputs, loaded when a visit starts so
// that their latency hides behind the visit's segments (a load at the store
// stalls the streaming warp once per slab).  Absent terms are not loaded.
template <int T, bool MMA>
__device__ __forceinline__ void load_epilogue(const float *bias, const float *res, int N, int row0, int rows, int r8,
                                              int j, bool stores, float (&eb)[LaneOut<T, MMA>::N],
                                              float (&er)[LaneOut<T, MMA>::N])
{
    using LO = LaneOut<T, MMA>;
#pragma unroll
    for (int k = 0; k < LO::N; ++k) {
        const int lr = LO::row(k, r8), t = LO::tok(k, j);
        const bool own = stores && LO::owner(k, j) && lr < rows;
        eb[k] = (own && bias != nullptr) ? __ldg(bias + row0 + lr) : 0.0f;
        er[k] = (own && res != nullptr) ? res[static_cast<long long>(t) * N + row0 + lr] : 0.0f;
    }
}

// store_outputs with the epilogue terms already loaded (non-argmax launches).
template <int T, bool MMA>
__device__ __forceinline__ void store_outputs_ep(float *ye, int N, int row0, int rows, int r8, int j,
                                                 const float (&yv)[LaneOut<T, MMA>::N],
                                                 const float (&eb)[LaneOut<T, MMA>::N],
                                                 const float (&er)[LaneOut<T, MMA>::N], bool has_b, bool has_r)
{
    using LO = LaneOut<T, MMA>;
#pragma unroll
    for (int k = 0; k < LO::N; ++k) {
        const int lr = LO::row(k, r8), t = LO::tok(k, j);
        if (lr >= rows || !LO::owner(k, j)) continue;
        float v = yv[k];
        if (has_b) v = __fadd_rn(v, eb[k]);
        if (has_r) v = __fadd_rn(v, er[k]);
        ye[static_cast<long long>(t) * N + row0 + lr] = v;
    }
}

// Bounded spin on a shared-memory flag written by another warp of the CTA.
__device__ __forceinline__ bool wait_flag(volatile int *flag, volatile int *abort_flag, unsigned *status)
{
    if (*flag) return true;
    const uint64_t t0 = global_timer_ns();
    while (!*flag) {
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > WAIT_LIMIT_NS) {
            *abort_flag = 1;
            atomicCAS(status, 0u, ST_TIMEOUT);
            return false;
        }
    }
    return true;
}

template <int T, int MAXG, bool ARGMAX, bool MMA, bool EPI>
__global__ void __launch_bounds__(max_warps_for(T, MMA) * 32, 1) qgemv_stream_kernel(const __grid_constant__ Params<MAXG> P)
{
    using LO = LaneOut<T, MMA>;
    constexpr int NO = LO::N;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_abort;
    __shared__ int s_last;
    __shared__ int s_nruns;   // > 0: balanced mode with this many runs
    __shared__ int s_ngroups; // groups of consecutive runs whose activations fit together
    __shared__ int s_grp[MAX_RUNS + 1];  // first run of each group, then the run count
    __shared__ long long s_i0, s_i1;     // the CTA's item range
    __shared__ unsigned long long s_best[ARGMAX ? max_warps_for(T, MMA) * T * 2 : 1];  // [warp][t][2]
    __shared__ long long s_pred[ARGMAX ? T : 1];  // verify: the step's predictions

    __shared__ ParamHead H;              // the scalar launch parameters
    // small groups spread over all warps: sequence launches on the
    // tensor-core path only (the int8 path's groups are rarely that small)
    constexpr bool SMALL_GROUPS = MMA && !ARGMAX && MAXG == MAXG_SEQ;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // One round of parallel parameter reads into shared memory: the scalar
    // header, this CTA's item range from the host's table, and the
    // descriptors of the launch groups from g0 (holding the range's first
    // item) to gn (holding the next range's first item; the range ends in gn
    // or before it).
    // (one-group launches skip the table: their descriptor loads then start
    // in the same round as the header's)
    const bool one = P.ngroups == 1;
    const int g0 = one ? 0 : P.cta_g0[blockIdx.x], gn = one ? 0 : P.cta_g0[blockIdx.x + 1];
    const int ngc = min(gn - g0 + 1, GCACHE_GROUPS);
    Group *gcache = reinterpret_cast<Group *>(smem + P.off_gcache);
    {
        static_assert(sizeof(ParamHead) % 8 == 0, "the header is copied in 8-byte words");
        static_assert(sizeof(Group) % 8 == 0, "group descriptors are copied in 8-byte words");
        constexpr int HW = static_cast<int>(sizeof(ParamHead) / 8);
        if (tid < HW)
            reinterpret_cast<unsigned long long *>(&H)[tid] =
                reinterpret_cast<const unsigned long long *>(static_cast<const ParamHead *>(&P))[tid];
        const unsigned long long *src = reinterpret_cast<const unsigned long long *>(&P.g[g0]);
        unsigned long long *dst = reinterpret_cast<unsigned long long *>(gcache);
        const int words = ngc * static_cast<int>(sizeof(Group) / 8);
        for (int wd = tid; wd < words; wd += blockDim.x) dst[wd] = src[wd];
        if (tid == blockDim.x - 1) {
            s_i0 = P.cta_i0[blockIdx.x];
            s_i1 = P.cta_i0[blockIdx.x + 1];
            s_abort = 0;
        }
    }
    __syncthreads();
    // Warm-up: the warps ask L2 for the first bytes of this CTA's weights (in
    // its first group, packed slabs only) in 16 KB pieces, one piece per
    // warp in turn (so that no warp, thread 0's least, waits on many
    // prefetch issues before the run table), so that HBM works while the
    // prologue and the activations are prepared and the first stage copies
    // find their bytes in L2.  Bounded by the group's slabs.
    if (lane == 0 && !H.ggml) {
        const Group &g = gcache[0];
        const long long li0 = s_i0 - g.item_begin;
        const long long li1 = gn == g0 ? s_i1 - g.item_begin : static_cast<long long>(g.items_per_inst) * g.count;
        if (g.split == 1 && g.count == 1 && li0 < g.nslabs && li1 > li0) {
            const long long lo = li0 * g.slab_bytes, hi = (li1 < g.nslabs ? li1 : g.nslabs) * g.slab_bytes;
            const long long end = hi - lo > WARM_L2_BYTES ? lo + WARM_L2_BYTES : hi;
            const int nwp = static_cast<int>(blockDim.x >> 5);
            for (long long c = lo + static_cast<long long>(nwp - 1 - warp) * WARM_L2_PIECE; c < end;
                 c += static_cast<long long>(nwp) * WARM_L2_PIECE)
                bulk_prefetch_l2(g.W + c, static_cast<unsigned>(min(static_cast<long long>(WARM_L2_PIECE), end - c)));
        }
    }
    const int nw = H.nwarps, nthreads = nw * 32;
    const int r8 = lane >> 2, j = lane & 3;
    const int D = H.ring_depth;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + H.off_bar);
    uint64_t *xbar = bars + nw * D;
    RunInfo *runs = reinterpret_cast<RunInfo *>(smem + H.off_runs);
    float *hbuf = reinterpret_cast<float *>(smem + H.off_hbuf);          // [nw][T][16]
    volatile int *hflag = reinterpret_cast<volatile int *>(smem + H.off_hflag);
    volatile int *abort_flag = &s_abort;
    const bool ggml = H.ggml != 0;
    const bool f32in = H.xf32 != 0;  // activations arrive as fp32 and are quantised here

    Ring ring;
    ring.base = smem + H.off_ring + static_cast<size_t>(warp) * D * SEG_BYTES;
    ring.bar = bars + warp * D;
    ring.D = D;
    ring.slot = 0;
    ring.phase = 0;
    ring.issued = 0;
    ring.consumed = 0;

    const long long i0 = s_i0, i1 = s_i1;

    if (tid == 0) {
        mbar_init(xbar, 1);
        // Run table for the balanced mode (thread 0 walks the CTA's runs),
        // cut into groups of consecutive runs whose activation images fit the
        // activation area together; each group's images start at offset 0.
        int nr = 0, stages = 0, xoff = 0, ng = 0;
        bool fits = H.balanced_ok != 0 && gn - g0 < ngc;  // a longer span has more runs than MAX_RUNS
        s_grp[0] = 0;
        int gh = g0;
        for (long long ra = i0; ra < i1 && fits;) {
            while (gh + 1 <= gn && gcache[gh + 1 - g0].item_begin <= ra) ++gh;
            const Group &g = gcache[gh - g0];
            const int ra_inst = static_cast<int>(ra - g.item_begin) / g.items_per_inst;
            const long long rb = min(i1, g.item_begin + static_cast<long long>(ra_inst + 1) * g.items_per_inst);
            if (nr == MAX_RUNS) {
                fits = false;
                break;
            }
            const int local = static_cast<int>(ra - g.item_begin);
            const int e = local / g.items_per_inst;
            // a gather's expert ids may still be written by the preceding
            // kernel: its runs take expert 0 here, and after the dependency
            // wait each run's weights and bad-id flag are patched (the
            // table's shape does not depend on the ids: every expert of a
            // matrix has the same shape)
            const int expert = H.ids != nullptr ? 0 : e, bad = 0;
            RunInfo &R = runs[nr];
            R.Wi = g.W + static_cast<long long>(expert) * g.w_stride;
            R.y = g.y + static_cast<long long>(e) * g.y_stride;
            R.stage0 = stages;
            R.nstages = static_cast<int>(rb - ra) * g.nseg;
            R.first_local = local - e * g.items_per_inst;
            R.gi = gh;
            R.e = e;
            R.nseg = g.nseg;
            R.nb = g.nb;
            R.K = g.K;
            R.N = g.N;
            R.nslabs = g.nslabs;
            R.bad = bad;
            const int xb = xq_layout(T, g.K, MMA).bytes;
            if (xb > H.xq_area) fits = false;
            if (nr > 0 && xoff + xb > H.xq_area) {  // close the group
                s_grp[++ng] = nr;
                xoff = 0;
            }
            R.xq_off = xoff;
            xoff += xb;
            stages += R.nstages;
            ++nr;
            ra = rb;
        }
        if (nr == 0) fits = false;
        s_grp[++ng] = nr;
        s_nruns = fits ? nr : 0;
        s_ngroups = ng;
    }
    if (lane == 0)
        for (int d = 0; d < D; ++d) mbar_init(&ring.bar[d], 1);
    if (tid < nw) hflag[tid] = 0;
    fence_mbar_init();
    __syncthreads();
    pdl_launch_dependents();

    const uint64_t pol_w = l2_policy_evict_first();
    const uint64_t pol_x = l2_policy_evict_last();
    const int nruns = s_nruns;
    // (the run-synced mode's stage walkers read a gather's ids themselves)
    if (H.ids != nullptr && nruns == 0) pdl_wait();

    Top2Lane<T, MMA> st;  // the lane's two best keys per token (argmax launches)
#pragma unroll
    for (int sl = 0; sl < Top2Lane<T, MMA>::S; ++sl) st.b1[sl] = st.b2[sl] = 0ull;
    bool x_unconfirmed = false;  // thread 0: an activation copy was issued but not seen complete
    unsigned xphase = 0;

    if (nruns > 0) {
        // ================================================= balanced mode
        // (the run's groups g0..gn are all in the descriptor cache)
        const int ngroups = s_ngroups;
        for (int gidx = 0; gidx < ngroups; ++gidx) {
            const int rg0 = s_grp[gidx], rg1 = s_grp[gidx + 1];
            const int S0 = runs[rg0].stage0, S1 = runs[rg1 - 1].stage0 + runs[rg1 - 1].nstages;
            const int S = S1 - S0;
            // warps taking part: each must get at least one whole slab, so
            // that a slab is shared by two warps at most (every run of the
            // group holds whole slabs, so one warp always qualifies)
            int nseg_max = 1;
            for (int r = rg0; r < rg1; ++r) nseg_max = max(nseg_max, runs[r].nseg);
            // a small group (one run of fewer whole slabs than warps, e.g. a
            // few slabs of a projection whose activations need shared memory
            // alone): every warp takes an equal range of its stages, writes
            // each segment sum to this CTA's workspace region, and after a
            // barrier the CTA adds them per output in segment order
            const bool small_grp = SMALL_GROUPS && !ggml && H.sg_part != nullptr && static_cast<int>(blockIdx.x) < H.sg_ctas &&
                                   rg1 - rg0 == 1 &&
                                   runs[rg0].nstages < nw * runs[rg0].nseg && !runs[rg0].bad &&
                                   runs[rg0].first_local + runs[rg0].nstages / runs[rg0].nseg <= runs[rg0].nslabs &&
                                   runs[rg0].nstages * T * 16 <= H.sg_stride;
            const int nwg = small_grp ? min(nw, S) : max(1, min(nw, S / nseg_max));
            const int a = warp < nwg ? S0 + static_cast<int>(static_cast<unsigned>(S) * warp / nwg) : S1;
            const int b = warp < nwg ? S0 + static_cast<int>(static_cast<unsigned>(S) * (warp + 1) / nwg) : S1;
            // boundary items: is stage p inside (not at the start of) an item?
            auto item_start = [&](int p) {
                int r = rg0;
                while (p >= runs[r].stage0 + runs[r].nstages) ++r;
                return p - (p - runs[r].stage0) % runs[r].nseg;
            };
            int head_b = b, tail_e = a;
            if (!small_grp && b < S1 && b > a) {
                const int st = item_start(b);
                if (st != b) head_b = st;  // [st, b) is the head of an item continued by warp + 1
            }
            if (!small_grp && a > S0 && a < b) {
                const int st = item_start(a);
                if (st != a) {
                    int r = rg0;
                    while (a >= runs[r].stage0 + runs[r].nstages) ++r;
                    tail_e = st + runs[r].nseg;  // [a, tail_e) finishes an item begun by warp - 1
                }
            }

            // weights first (they depend neither on the preceding kernel nor on
            // the previous group); the ring is empty here, and its next slots
            // in consumption order start at ring.slot
            Walker cur;
            cur.init(runs, head_b, b, tail_e, head_b, a, tail_e);
            if (gidx == 0 && H.ids != nullptr) {
                // a gather's expert ids, now that the preceding kernel is
                // done: each run's weights and bad-id flag
                pdl_wait();
                for (int r = tid; r < nruns; r += nthreads) {
                    RunInfo &R = runs[r];
                    const Group &g = gcache[R.gi - g0];
                    int expert = __ldg(H.ids + R.e);
                    const int bad = (expert < 0 || expert >= H.n_experts) ? 1 : 0;
                    if (bad) expert = 0;
                    R.Wi = g.W + static_cast<long long>(expert) * g.w_stride;
                    R.bad = bad;
                }
                __syncthreads();
                if (cur.valid) cur.load_run(runs);
            }
            cur.skip_untransferred(runs, ggml);
            for (int d = 0; d < D && cur.valid; ++d) {
                ring.issue(lane, (ring.slot + d) % D, cur.src(), cur.bytes(), pol_w);
                cur.step(runs);
                cur.skip_untransferred(runs, ggml);
            }
            if (gidx == 0) {
                if (H.ids == nullptr) pdl_wait();  // (a gather waited above, before reading its ids)
            } else {
                // every warp is done with the previous group's activations and
                // hand-off sums; the whole CTA stops together after an abort
                if (__syncthreads_or(*abort_flag)) break;
                if (tid < nw) hflag[tid] = 0;
            }
            // the group's activations, one transaction count on one barrier
            if (tid == 0 && !*abort_flag) {
                // f16 operand images and fp32 activations are read from global memory instead
                unsigned tx = 0;
                for (int r = rg0; r < rg1; ++r)
                    if (!f32in && !xq_layout(T, runs[r].K, MMA).f16)
                        tx += static_cast<unsigned>(gcache[runs[r].gi - g0].xq_bytes);
                x_unconfirmed = true;
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(xbar, tx);
                for (int r = rg0; r < rg1; ++r) {
                    const RunInfo &R = runs[r];
                    const Group &g = gcache[R.gi - g0];
                    if (f32in || xq_layout(T, R.K, MMA).f16) continue;
                    const unsigned dbytes = static_cast<unsigned>(g.xq_bytes - T * R.K);
                    copy_activations<T, MMA>(smem + R.xq_off, g.xq + static_cast<long long>(R.e) * g.xq_stride, R.K, dbytes,
                                        xbar, pol_x);
                }
            }
            const bool xok = mbar_wait_bounded(xbar, xphase, abort_flag, H.status, WAIT_LIMIT_NS);
            xphase ^= 1u;
            if (xok && tid == 0) x_unconfirmed = false;
            if (xok)
                for (int r = rg0; r < rg1; ++r) {
                    const RunInfo &R = runs[r];
                    const Group &g = gcache[R.gi - g0];
                    const uint8_t *src = g.xq + static_cast<long long>(R.e) * g.xq_stride;
                    if (MMA && xq_layout(T, R.K, MMA).f16) {
                        if (f32in)
                            build_f16_image<T, true>(smem + R.xq_off, src, R.K, tid, nthreads);
                        else
                            build_f16_image<T, false>(smem + R.xq_off, src, R.K, tid, nthreads);
                    } else if (f32in) {  // int8 image quantised here from the fp32 activations
                        quantize_image<T, MMA>(smem + R.xq_off, reinterpret_cast<const float *>(src), R.K, tid, nthreads);
                    } else {
                        build_fold_constants<T, MMA>(smem + R.xq_off, R.K, tid, nthreads);
                    }
                }
            __syncthreads();

            // compute, one visit (the segments of one slab inside one interval) at a time
            Walker w;
            w.init(runs, head_b, b, tail_e, head_b, a, tail_e);
            bool ok = xok;
            while (w.valid) {
                const RunInfo &R = runs[w.r];
                const int s_first = w.s;
                const int seg_end = min(w.nseg, s_first + (w.kend - w.k));
                const int li = w.first_local + w.ii;
                const bool tail_item = li >= w.nslabs;
                const bool direct = ggml || tail_item;
                const int nb = w.nb;
                const int rows = tail_item ? gcache[R.gi - g0].tail_rows : min(SLAB_ROWS, R.N - li * SLAB_ROWS);
                const uint8_t *rows_base = w.Wi + static_cast<long long>(li) * SLAB_ROWS * nb * Q4_BYTES;
                const XqLayout L = xq_layout(T, R.K, MMA);
                XqView xv{reinterpret_cast<const int8_t *>(smem + R.xq_off), L.xstride,
                          reinterpret_cast<const int2 *>(smem + R.xq_off + L.off_cd), L.cdw};
                if constexpr (MMA) {
                    xv.f16 = L.f16;
                    mma_lane_offsets<T>(xv, r8, j);
                }
                float yv[NO];
    #pragma unroll
                for (int k = 0; k < NO; ++k) yv[k] = 0.0f;
                float eb[EPI ? NO : 1], er[EPI ? NO : 1];
                const float *ep_bias = nullptr, *ep_res = nullptr;
                if constexpr (EPI) {
                    // this warp stores the slab's outputs: fetch the epilogue's terms now
                    const Group &gg = gcache[R.gi - g0];
                    ep_bias = gg.bias;
                    ep_res = gg.res;
                    load_epilogue<T, MMA>(ep_bias, ep_res, R.N, li * SLAB_ROWS, rows, r8, j,
                                          !small_grp && seg_end == w.nseg && !w.bad, eb, er);
                }
                if (s_first > 0 && !small_grp) {
                    // tail of a slab begun by warp - 1: continue from its ordered sum
                    if (lane == 0) wait_flag(&hflag[warp - 1], abort_flag, H.status);
                    __syncwarp();
                    __threadfence_block();
                    const float *H = hbuf + (warp - 1) * T * 16;
    #pragma unroll
                    for (int k = 0; k < NO; ++k) {
                        const int t = LO::tok(k, j);
                        yv[k] = t < T ? H[t * 16 + LO::row(k, r8)] : 0.0f;
                    }
                }
                for (int sg = s_first; sg < seg_end; ++sg) {
                    float Pk[NO];
                    bool have = false;
                    if (w.bad) {
                        // nothing is read for an out-of-range expert id
                    } else if (direct) {
                        if (ok) {
                            segment_sum<T, MMA>(false, nullptr, rows_base, rows, sg, nb, r8, j, xv, Pk);
                            have = true;
                        }
                    } else {
                        if (ok) ok = mbar_wait_bounded(&ring.bar[ring.slot], ring.phase, abort_flag, H.status, WAIT_LIMIT_NS);
                        if (ok) {
                            segment_sum<T, MMA>(true, ring.stage(), nullptr, 0, sg, nb, r8, j, xv, Pk);
                            have = true;
                        }
                        __syncwarp();
                        if (cur.valid && ok) {  // refill the slot just consumed
                            ring.issue(lane, ring.slot, cur.src(), cur.bytes(), pol_w);
                            cur.step(runs);
                            cur.skip_untransferred(runs, ggml);
                        }
                        ring.pop();
                    }
                    if (!have) {
    #pragma unroll
                        for (int k = 0; k < NO; ++k) Pk[k] = 0.0f;
                    }
                    if (small_grp) {  // the segment sum, for the CTA's ordered fold below
                        // (the region's base is re-read from shared memory: no register holds it)
                        float *pb = *reinterpret_cast<float *volatile *>(&H.sg_part) +
                                    static_cast<long long>(blockIdx.x) * H.sg_stride +
                                    ((li - w.first_local) * w.nseg + sg) * T * 16;
    #pragma unroll
                        for (int k = 0; k < NO; ++k)
                            if (LO::owner(k, j)) pb[LO::tok(k, j) * 16 + LO::row(k, r8)] = Pk[k];
                        continue;
                    }
    #pragma unroll
                    for (int k = 0; k < NO; ++k) yv[k] = (sg == 0) ? Pk[k] : __fadd_rn(yv[k], Pk[k]);
                }
                if (small_grp) {
                    // outputs come from the fold after the group
                } else if (seg_end < w.nseg) {
                    // head of a slab that warp + 1 finishes: leave the ordered sum
                    float *H = hbuf + warp * T * 16;
    #pragma unroll
                    for (int k = 0; k < NO; ++k)
                        if (LO::owner(k, j)) H[LO::tok(k, j) * 16 + LO::row(k, r8)] = yv[k];
                    __threadfence_block();
                    __syncwarp();
                    if (lane == 0) hflag[warp] = 1;
                } else if (!w.bad) {
                    if constexpr (EPI)
                        store_outputs_ep<T, MMA>(R.y, R.N, li * SLAB_ROWS, rows, r8, j, yv, eb, er, ep_bias != nullptr,
                                                 ep_res != nullptr);
                    else
                        store_outputs<T, MMA, ARGMAX>(R.y, R.N, li * SLAB_ROWS, rows, r8, j, yv, st);
                } else if (lane == 0) {
                    atomicCAS(H.status, 0u, ST_BAD_ID);
                }
                w.next_item(runs);
            }
            if (small_grp) {
                // every segment sum of the group is written: add them per
                // output (slab, token, row) in segment order
                __syncthreads();
                const RunInfo &R = runs[rg0];
                const int nsl = R.nstages / R.nseg;
                const float *pr = H.sg_part + static_cast<long long>(blockIdx.x) * H.sg_stride;
                for (int o = tid; o < nsl * T * 16; o += nthreads) {
                    const int sl = o / (T * 16), t = (o / 16) % T, row = o % 16;
                    const float *p = pr + static_cast<long long>(sl) * R.nseg * T * 16 + t * 16 + row;
                    float v = p[0];
                    for (int sg = 1; sg < R.nseg; ++sg) v = __fadd_rn(v, p[static_cast<long long>(sg) * T * 16]);
                    const int orow = (R.first_local + sl) * SLAB_ROWS + row;
                    const long long yi = static_cast<long long>(t) * R.N + orow;
                    if constexpr (EPI) {
                        const Group &gg = gcache[R.gi - g0];
                        v = apply_epilogue(v, gg.bias, gg.res, yi, orow);
                    }
                    R.y[yi] = v;
                }
            }
        }
    } else {
        // ================================================= run-synced mode
        // (small launches, split-K, or activations that do not all fit)
        StageCursor<MAXG> cur;
        cur.init(P, i0, i1, warp);
        for (int d = 0; d < D && cur.valid; ++d) {
            ring.issue(lane, d, cur.src(P), cur.bytes(P), pol_w);
            cur.advance(P, warp);
        }
        if (H.ids == nullptr) pdl_wait();  // (a gather waited before its stage walkers)

        int gi_hint = 0, gi_item = 0;
        for (long long ra = i0; ra < i1;) {
            const long long rb = run_end(P, ra, i1, gi_hint);
            const Group &g = P.g[gi_hint];
            const int K = g.K, nb = g.nb, N = g.N;
            const int e_run = static_cast<int>(ra - g.item_begin) / g.items_per_inst;
            const XqLayout L = xq_layout(T, K, MMA);
            XqView xv{reinterpret_cast<const int8_t *>(smem), L.xstride,
                      reinterpret_cast<const int2 *>(smem + L.off_cd), L.cdw};
            if constexpr (MMA) {
                xv.f16 = L.f16;
                mma_lane_offsets<T>(xv, r8, j);
            }

            __syncthreads();
            if (tid == 0 && !*abort_flag) {
                x_unconfirmed = true;
                fence_proxy_async_smem();
                const unsigned dbytes = static_cast<unsigned>(g.xq_bytes - T * K);
                if (L.f16 || f32in) {  // built from global memory below
                    mbar_arrive_expect_tx(xbar, 0);
                } else {
                    mbar_arrive_expect_tx(xbar, static_cast<unsigned>(T * K) + dbytes);
                    copy_activations<T, MMA>(smem, g.xq + static_cast<long long>(e_run) * g.xq_stride, K, dbytes, xbar,
                                             pol_x);
                }
            }
            const bool xok = mbar_wait_bounded(xbar, xphase, abort_flag, H.status, WAIT_LIMIT_NS);
            if (xok) x_unconfirmed = false;
            xphase ^= 1u;
            const uint8_t *xsrc = g.xq + static_cast<long long>(e_run) * g.xq_stride;
            if (xok) {
                if (MMA && L.f16) {
                    if (f32in)
                        build_f16_image<T, true>(smem, xsrc, K, tid, nthreads);
                    else
                        build_f16_image<T, false>(smem, xsrc, K, tid, nthreads);
                } else if (f32in) {  // int8 image quantised here from the fp32 activations
                    quantize_image<T, MMA>(smem, reinterpret_cast<const float *>(xsrc), K, tid, nthreads);
                } else {
                    build_fold_constants<T, MMA>(smem, K, tid, nthreads);
                }
            }
            __syncthreads();

            for (long long it = ra + warp; it < rb; it += nw) {
                const ItemInfo inf = decode_item(P, it, gi_item);
                if (inf.bad) {
                    if (lane == 0) atomicCAS(H.status, 0u, ST_BAD_ID);
                    continue;
                }
                const bool direct = ggml || inf.kind != 0;
                const bool split = g.split > 1 && inf.kind == 0;  // a packed tail is never split
                const uint8_t *rows_base =
                    inf.kind != 0 ? inf.Wi + static_cast<long long>(g.nslabs) * g.slab_bytes
                                  : inf.Wi + static_cast<long long>(inf.slab) * SLAB_ROWS * nb * Q4_BYTES;
                float yv[NO];
#pragma unroll
                for (int k = 0; k < NO; ++k) yv[k] = 0.0f;

                for (int sg = inf.seg0; sg < inf.seg1; ++sg) {
                    float Pk[NO];
                    bool have = false;
                    if (direct) {
                        if (xok) {
                            segment_sum<T, MMA>(false, nullptr, rows_base, inf.rows, sg, nb, r8, j, xv, Pk);
                            have = true;
                        }
                    } else {
                        const bool ok = mbar_wait_bounded(&ring.bar[ring.slot], ring.phase, abort_flag, H.status,
                                                          WAIT_LIMIT_NS);
                        if (ok && xok) {
                            segment_sum<T, MMA>(true, ring.stage(), nullptr, 0, sg, nb, r8, j, xv, Pk);
                            have = true;
                        }
                        __syncwarp();
                        const int aborted = __shfl_sync(0xFFFFFFFFu, *abort_flag, 0);
                        if (cur.valid && !aborted) {
                            ring.issue(lane, ring.slot, cur.src(P), cur.bytes(P), pol_w);
                            cur.advance(P, warp);
                        }
                        ring.pop();
                    }
                    if (!have) {
#pragma unroll
                        for (int k = 0; k < NO; ++k) Pk[k] = 0.0f;
                    }
                    if (split) {
                        float *pb =
                            g.part + ((static_cast<long long>(inf.e) * g.nslabs + inf.slab) * g.nseg + sg) * T * 16;
#pragma unroll
                        for (int k = 0; k < NO; ++k)
                            if (LO::owner(k, j)) pb[LO::tok(k, j) * 16 + LO::row(k, r8)] = Pk[k];
                    } else {
#pragma unroll
                        for (int k = 0; k < NO; ++k) yv[k] = (sg == 0) ? Pk[k] : __fadd_rn(yv[k], Pk[k]);
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
                        const float *pb =
                            g.part + (static_cast<long long>(inf.e) * g.nslabs + inf.slab) * g.nseg * T * 16;
                        unsigned long long kt[ARGMAX ? T : 1];  // this lane's row's key per token
#pragma unroll
                        for (int t = 0; t < (ARGMAX ? T : 1); ++t) kt[t] = 0ull;
                        if (lane < inf.rows) {
                            const int row = row0 + lane;
#pragma unroll
                            for (int t = 0; t < T; ++t) {
                                const float v = ordered_sum_ldcg(pb + t * 16 + lane, g.nseg, T * 16);
                                if (ye != nullptr) {
                                    const long long yi = static_cast<long long>(t) * N + row;
                                    ye[yi] = EPI ? apply_epilogue(v, g.bias, g.res, yi, row) : v;
                                }
                                if (ARGMAX) kt[ARGMAX ? t : 0] = argmax_key(v, static_cast<unsigned>(row));
                            }
                        }
                        if constexpr (ARGMAX) {
                            using TL2 = Top2Lane<T, MMA>;
#pragma unroll
                            for (int t = 0; t < T; ++t) {  // the warp's pair, into a lane that tracks t
                                unsigned long long a1 = kt[t], a2 = 0ull;
                                top2_warp(a1, a2);
                                if (lane == TL2::jt(t)) top2_merge(st.b1[TL2::slot(t)], st.b2[TL2::slot(t)], a1, a2);
                            }
                        }
                        __syncwarp();
                        if (lane == 0) *cnt = 0u;
                    }
                } else {
                    store_outputs<T, MMA, ARGMAX>(ye, N, row0, inf.rows, r8, j, yv, st, EPI ? g.bias : nullptr,
                                                  EPI ? g.res : nullptr);
                }
            }
            ra = rb;
        }
    }

    // Copies still in flight (only after an abort): wait for them, bounded.
    ring.drain();
    if (x_unconfirmed) mbar_drain(xbar, xphase ^ 1u);

    if (ARGMAX) {
        // top-2 per token: lanes with the same j (lane bits 2..4 are r8), then
        // warps, then this CTA's candidate pair
#pragma unroll
        for (int sl = 0; sl < Top2Lane<T, MMA>::S; ++sl) {
            unsigned long long v1 = st.b1[sl], v2 = st.b2[sl];
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                const unsigned long long o1 = __shfl_xor_sync(0xFFFFFFFFu, v1, off);
                const unsigned long long o2 = __shfl_xor_sync(0xFFFFFFFFu, v2, off);
                top2_merge(v1, v2, o1, o2);
            }
            const int t = Top2Lane<T, MMA>::token(sl, lane);
            if (lane < 4 && t < T) {
                s_best[(warp * T + t) * 2] = v1;
                s_best[(warp * T + t) * 2 + 1] = v2;
            }
        }
        __syncthreads();
        // the argmax alone (no top-2, no verify rule): each CTA folds its best
        // key into a running maximum per token (exact in any order); the last
        // CTA reads and clears it
        const bool alone = H.am_idx2 == nullptr && H.vc_tokens == nullptr;
        if (tid < T) {
            unsigned long long m1 = 0ull, m2 = 0ull;
            for (int w = 0; w < nw; ++w) top2_merge(m1, m2, s_best[(w * T + tid) * 2], s_best[(w * T + tid) * 2 + 1]);
            if (alone) {
                if (m1) atomicMax(H.am_key + tid, m1);
            } else {
                H.am_cand[(static_cast<long long>(blockIdx.x) * T + tid) * 2] = m1;
                H.am_cand[(static_cast<long long>(blockIdx.x) * T + tid) * 2 + 1] = m2;
            }
            __threadfence();  // the candidates are visible before the arrival below
        }
        __syncthreads();
        if (tid == 0) s_last = (atomicAdd(H.am_cnt, 1u) == gridDim.x - 1) ? 1 : 0;
        __syncthreads();
        if (s_last && alone) {
            __threadfence();
            if (tid < T) {
                const unsigned long long k = atomicExch(H.am_key + tid, 0ull);
                if (H.am_idx != nullptr) H.am_idx[tid] = key_row(k);
            }
            if (tid == 0) *H.am_cnt = 0u;
        } else if (s_last) {
            // the warps split the tokens: warp w merges token w % T over part
            // w / T of the CTAs' candidate pairs (one pair per lane in turn),
            // then one thread per token merges the parts
            __threadfence();
            const int parts = nw / T;  // nw >= 8 >= T
            if (warp < parts * T) {
                const int t = warp % T, p = warp / T;
                unsigned long long m1 = 0ull, m2 = 0ull;
#pragma unroll 4
                for (unsigned c = p * 32 + lane; c < gridDim.x; c += parts * 32)
                    top2_merge(m1, m2, __ldcg(H.am_cand + (static_cast<long long>(c) * T + t) * 2),
                               __ldcg(H.am_cand + (static_cast<long long>(c) * T + t) * 2 + 1));
                top2_warp(m1, m2);
                if (lane == 0) {
                    s_best[(p * T + t) * 2] = m1;
                    s_best[(p * T + t) * 2 + 1] = m2;
                }
            }
            __syncthreads();
            if (tid < T) {
                unsigned long long m1 = 0ull, m2 = 0ull;
                for (int w = 0; w < parts; ++w)
                    top2_merge(m1, m2, s_best[(w * T + tid) * 2], s_best[(w * T + tid) * 2 + 1]);
                if (H.am_idx != nullptr) H.am_idx[tid] = key_row(m1);
                if (H.am_idx2 != nullptr) {
                    H.am_idx2[2 * tid] = key_row(m1);
                    H.am_idx2[2 * tid + 1] = key_row(m2);
                    H.am_val2[2 * tid] = key_value(m1);
                    H.am_val2[2 * tid + 1] = key_value(m2);
                }
                if (H.vc_tokens != nullptr) s_pred[tid] = key_row(m1);
            }
            if (H.vc_tokens != nullptr) {
                // the verify rule on this step's predictions (minfer README M17): commit
                // pred[0] and each later one while every draft equalled the prediction before it
                __syncthreads();
                if (tid == 0) {
                    int n = 1;
                    while (n < T && H.vc_tokens[n] == s_pred[n - 1]) ++n;
                    *H.vc_n = n;
                }
            }
            if (tid == 0) *H.am_cnt = 0u;
        }
    }
}

}  // namespace qg
