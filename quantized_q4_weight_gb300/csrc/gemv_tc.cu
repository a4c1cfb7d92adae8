// gemv_tc.cu -- the few-token (verify) GEMV on the fifth-generation tensor
// cores: tcgen05.mma with the weight operand in tensor memory (minfer README
// M16: the multi-token path puts the tokens in the MMA's N dimension and
// forms the same per-block integer sums as the one-token path).
//
// Work.  A launch is a list of GEMVs (items), each cut into 128-row tiles (8
// packed slabs) and 16-block segments of K; a unit is one (tile, segment).
// Units are numbered in list order (item, tile, segment) and every warp group
// of the grid (two per CTA) takes a contiguous range of them.
//
// A warp group is four compute warps (thread R of the group owns row R of
// the tile, which is tensor-memory lane R) and one issuer thread:
//   - the issuer keeps TC_NQ quad stages in flight (TMA, one 1152-byte copy
//     per slab: 8 slabs x 4 blocks), copies each unit's activation codes and
//     scales (planar Q8_0, from L2) a unit ahead, and issues two MMAs per
//     block once the four warps have written its A operand;
//   - per unit the compute threads build the B operand in shared memory:
//     for 8 token columns (zeros past T) and each block, the activations q
//     (low-nibble half) and q / 16 (high-nibble half) in f16, in the
//     no-swizzle K-major core-matrix layout, 8 more zero columns for N = 16,
//     and per block and token the folded offset C = -8 sum(q) 2^-24 and d_x;
//   - per block each thread turns its row's 32 nibbles into the A operand
//     -- f16 subnormals n 2^-24 (one AND per two) and 16 n 2^-24 for the
//     high nibbles, exactly as the mma.sync path -- and writes them to
//     tensor memory with one tcgen05.st; the MMAs (M = 128, N = 16, K = 16,
//     f32 accumulate, exact here) leave sum(n q) 2^-24 in the D columns;
//   - one block later the thread reads its row's 8 sums back (tcgen05.ld),
//     adds C (exact) and accumulates (d_w d_x) (isum 2^-24) into the phase
//     sums of the fixed order: per segment four phases (b % 4) from +0,
//     combined (s0 + s1) + (s2 + s3), scaled back by 2^24, segments added in
//     order -- the same arithmetic as the dp4a and mma.sync paths, so y is
//     bit-identical to theirs.
// A tile cut between warp groups (or CTAs) writes its segment sums to the
// workspace; the last part to arrive (atomic counter) adds them in order.
//
// Every wait is bounded; a group that gives up records QGEMV_ERR_TIMEOUT,
// stops, waits (bounded) for its copies and MMAs in flight, and the CTA
// frees its tensor memory before it returns.
#include <atomic>
#include <cstring>
#include <memory>

#include "gemv_kernel.cuh"
#include "qgemv_launch.h"

namespace qg {

constexpr int TC_GROUPS = 2;                              // warp groups per CTA
constexpr int TC_THREADS = (TC_GROUPS * 4 + TC_GROUPS) * 32;  // 4 compute warps + 1 issuer warp per group
constexpr int TC_NS = 2;                                  // unit stages in flight per group
constexpr int TC_STAGE = 8 * SEG_BYTES;                   // one unit of 8 slabs: 36864 bytes
constexpr int TC_QCOLS = QUAD * 16;                       // tensor-memory columns of a quad's A (or D)
constexpr int TC_BSRC = 8 * 512;                          // a unit's activation codes, 8 tokens: 4096
constexpr int TC_BHALF = 256;                             // B half-block: tokens 0..7, 2 K-groups x 128 bytes
constexpr int TC_BTILE = SEG_BLOCKS * 2 * TC_BHALF;       // a unit's B operand: 8192
constexpr int TC_CONST = SEG_BLOCKS * 16 * 4;             // per block C[8], d_x[8]: 1024
constexpr int TC_OFF_BSRC = TC_NS * TC_STAGE;
constexpr int TC_OFF_BTILE = TC_OFF_BSRC + 2 * TC_BSRC;
constexpr int TC_OFF_CONST = TC_OFF_BTILE + 2 * TC_BTILE;
// Constants are read by every compute thread (not only by the MMAs), and a
// warp may run a quad ahead of the others: three slots, so that the slot a
// unit's constants are written to was last read two units before.
constexpr int TC_NCONST = 3;
constexpr int TC_OFF_ZERO = TC_OFF_CONST + TC_NCONST * TC_CONST;  // the zero token columns 8..15 of every B half-block
constexpr int TC_OFF_BAR = TC_OFF_ZERO + TC_BHALF;
constexpr int TC_NBAR = TC_NS + 2 + 2;                    // stage full, A written, D ready
constexpr int TC_GROUP_BYTES = (TC_OFF_BAR + 8 * TC_NBAR + 127) / 128 * 128;
constexpr int TC_SMEM = TC_GROUPS * TC_GROUP_BYTES;
constexpr int TC_TMEM_COLS = 512;                         // per group: A of two quads, then D of two quads
static_assert(TC_OFF_BTILE % 128 == 0 && TC_OFF_ZERO % 128 == 0, "B operands are addressed in 16-byte units");
static_assert(TC_SMEM <= 220 * 1024, "shared memory of the tensor-core kernel");

// One GEMV of a tensor-core launch.
struct TcItem {
    const uint8_t *W;         // packed weights (N % 16 == 0)
    const uint8_t *xq;        // planar Q8_0 activations of T rows
    float *y;                 // [T][N]
    long long slab_bytes;     // 288 * nb
    long long unit_begin;     // first unit of the item
    int N, K, nb, nseg, ntiles, pad;
};

struct TcParams {
    int nitems;
    int pad0;
    long long total_units;
    int groups;               // warp groups in the grid
    int slot_floats;          // workspace floats per split-tile slot: nseg_max * 8 * 128
    float *part;              // [groups][slot_floats] segment sums of split tiles
    unsigned *cnt;            // [groups][4] arrival counters of warp w's rows (left at zero)
    unsigned *status;
    TcItem it[MAXG_SEQ];
};
static_assert(sizeof(TcParams) <= 32764, "kernel parameters are limited to 32764 bytes");

// ------------------------------------------------------------ tcgen05 helpers

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// A row's 16 A-operand words into 16 columns of tensor memory.
__device__ __forceinline__ void tc_st16(uint32_t taddr, const unsigned (&a)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16};" ::"r"(taddr),
        "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(a[4]), "r"(a[5]), "r"(a[6]), "r"(a[7]), "r"(a[8]), "r"(a[9]),
        "r"(a[10]), "r"(a[11]), "r"(a[12]), "r"(a[13]), "r"(a[14]), "r"(a[15])
        : "memory");
}
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tc_ld8(uint32_t taddr, float (&d)[8])
{
    unsigned r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) d[i] = __uint_as_float(r[i]);
}

// D = A (tensor memory) x B (shared-memory descriptor) [+ D]; kind::f16.
__device__ __forceinline__ void tc_mma(uint32_t d_t, uint32_t a_t, uint64_t bdesc, uint32_t idesc, int accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_t),
        "r"(a_t), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// One arrival on `bar` once every MMA this thread issued before has completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

// The same two, issued by one elected lane of a converged warp (the whole
// warp runs the issuing loop, so its operands are warp-uniform).
__device__ __forceinline__ void tc_mma_elect(uint32_t d_t, uint32_t a_t, uint64_t bdesc, uint32_t idesc, int accumulate)
{
    asm volatile(
        "{\n\t.reg .pred e, p;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_t),
        "r"(a_t), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void tc_commit_elect(uint64_t *bar)
{
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Instruction descriptor: f16 A and B (K-major), f32 D, M = 128, N = 16.
constexpr uint32_t TC_IDESC = (1u << 4) | ((16u >> 3) << 17) | ((128u >> 4) << 24);

// Shared-memory descriptor of a B half-block: no swizzle, K-major core
// matrices of 8 rows x 16 bytes; K-direction stride 128 bytes (leading byte
// offset); the N-direction stride (stride byte offset) leads from tokens
// 0..7 at saddr to the shared zero block that stands for tokens 8..15.
__device__ __forceinline__ uint64_t tc_bdesc(uint32_t saddr, uint32_t zaddr)
{
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(128 >> 4) << 16) |
           (static_cast<uint64_t>(((zaddr - saddr) >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

// {a0, a1} * {b0, b1}, {a0, a1} + {b0, b1}: one f32x2 operation each (two
// IEEE operations, rounded to nearest).
__device__ __forceinline__ void fmul2(float &r0, float &r1, float a0, float a1, float b0, float b1)
{
    asm("{\n\t.reg .b64 ra, rb, rr;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rr, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rr;\n\t}"
        : "=f"(r0), "=f"(r1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// 16 bytes global -> shared by this thread (L2 only), completed by cp_async_wait.
__device__ __forceinline__ void cp_async16(void *dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// ------------------------------------------------------------ unit walk

struct TcUnit {
    int item, tile, seg, nblk, nsl;  // nsl: slabs in the tile (1..8)
    long long tile_u0;               // the tile's first unit
};

__device__ __forceinline__ void tc_decode(const TcParams &P, long long u, int &hint, TcUnit &U)
{
    while (hint + 1 < P.nitems && P.it[hint + 1].unit_begin <= u) ++hint;
    const TcItem &I = P.it[hint];
    const int local = static_cast<int>(u - I.unit_begin);  // an item has fewer than 2^31 units
    U.item = hint;
    U.tile = local / I.nseg;
    U.seg = local - U.tile * I.nseg;
    U.nblk = min(SEG_BLOCKS, I.nb - SEG_BLOCKS * U.seg);
    U.nsl = min(8, I.N / SLAB_ROWS - 8 * U.tile);
    U.tile_u0 = I.unit_begin + static_cast<long long>(U.tile) * I.nseg;
}

// First unit of warp group g (of G) over U units; the group covering unit v.
__device__ __forceinline__ long long tc_group_start(long long U, int G, long long g) { return U * g / G; }
__device__ __forceinline__ int tc_group_of(long long U, int G, long long v)
{
    long long g = v * G / U;
    while (g + 1 < G && tc_group_start(U, G, g + 1) <= v) ++g;
    while (g > 0 && tc_group_start(U, G, g) > v) --g;
    return static_cast<int>(g);
}

// Bounded wait by one thread; raises the CTA abort flag on timeout.
__device__ __forceinline__ bool tc_wait(uint64_t *bar, unsigned parity, volatile int *abort_flag, unsigned *status)
{
    return mbar_wait_bounded(bar, parity, abort_flag, status, WAIT_LIMIT_NS);
}

__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, unsigned parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// The same bound for waits expected to end within a block's time (the
// issuer's wait for the four warps, the warps' wait for MMAs issued seven
// blocks ago): a spin on the non-blocking test, so that no suspension of the
// waiting thread adds to the per-block time.
__device__ __forceinline__ bool tc_spin(uint64_t *bar, unsigned parity, volatile int *abort_flag, unsigned *status)
{
    if (mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (*abort_flag) return false;
        for (int i = 0; i < 64; ++i)
            if (mbar_test_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > WAIT_LIMIT_NS) {
            *abort_flag = 1;
            atomicCAS(status, 0u, ST_TIMEOUT);
            return false;
        }
    }
}

// ------------------------------------------------------------ kernel

template <int T>
__global__ void __launch_bounds__(TC_THREADS, 1) qgemv_tc_kernel(const __grid_constant__ TcParams P)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool issuer = warp >= 4 * TC_GROUPS;
    const int g = issuer ? warp - 4 * TC_GROUPS : warp >> 2;
    const int R = tid & 127;  // compute threads: row of the tile (tensor-memory lane)
    uint8_t *gs = smem + g * TC_GROUP_BYTES;
    uint8_t *ring = gs;
    uint8_t *bsrc = gs + TC_OFF_BSRC;
    uint8_t *btile = gs + TC_OFF_BTILE;
    uint8_t *cst = gs + TC_OFF_CONST;
    uint64_t *bars = reinterpret_cast<uint64_t *>(gs + TC_OFF_BAR);
    uint64_t *st_full = bars, *a_full = bars + TC_NS, *d_full = bars + TC_NS + 2;
    volatile int *abort_flag = &s_abort;

    if (tid == 0) s_abort = 0;
    if (issuer && lane == 0) {
        for (int i = 0; i < TC_NS; ++i) mbar_init(&st_full[i], 1);
        for (int i = 0; i < 2; ++i) mbar_init(&a_full[i], 4);  // one arrival per compute warp
        for (int i = 0; i < 2; ++i) mbar_init(&d_full[i], 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&s_tmem)),
                     "r"(TC_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (!issuer) {
        // B tiles, constants and the zero block start at zero: the token
        // columns past T are never written again
        uint4 *z = reinterpret_cast<uint4 *>(btile);
        for (int i = R; i < (TC_OFF_BAR - TC_OFF_BTILE) / 16; i += 128) z[i] = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_launch_dependents();

    // this group's tensor-memory columns: A of quad buffers 0 and 1 (4 blocks
    // x 16 columns each), then D of quad buffers 0 and 1
    const uint32_t tm = s_tmem + static_cast<uint32_t>(g * 4 * TC_QCOLS);
    const long long U = P.total_units;
    const long long gg = static_cast<long long>(blockIdx.x) * TC_GROUPS + g;
    const long long u0 = tc_group_start(U, P.groups, gg), u1 = tc_group_start(U, P.groups, gg + 1);

    if (issuer) {
        // The whole warp runs this loop (converged): lane 0 arms each
        // barrier, lanes issue the slab copies in parallel, one elected lane
        // issues the MMAs and commits.
        int hint = 0, fhint = 0;
        long long fu = u0, fi = 0;  // stage fills: the next unit, fills so far
        const uint64_t pol = l2_policy_evict_first();
        auto fill_stage = [&]() {
            TcUnit F;
            tc_decode(P, fu, fhint, F);
            const TcItem &I = P.it[F.item];
            const int slot = static_cast<int>(fi % TC_NS);
            uint64_t *bar = &st_full[slot];
            const unsigned bytes = static_cast<unsigned>(SLAB_COL_BYTES * F.nblk);  // one slab's segment
            if (lane == 0) {
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(bar, static_cast<unsigned>(F.nsl) * bytes);
            }
            __syncwarp();
            if (lane < F.nsl)
                bulk_g2s(ring + slot * TC_STAGE + lane * SEG_BYTES,
                         I.W + (static_cast<long long>(F.tile) * 8 + lane) * I.slab_bytes +
                             static_cast<long long>(F.seg) * SEG_BYTES,
                         bytes, bar, pol);
            ++fi;
            ++fu;
        };
        for (int n = 0; n < TC_NS && fu < u1; ++n) fill_stage();  // weights first: no dependency
        long long q = 0;  // quads issued
        bool ok = true;
        const uint32_t zaddr = smem_addr(gs + TC_OFF_ZERO);
        for (long long u = u0; u < u1 && ok; ++u) {
            TcUnit W;
            tc_decode(P, u, hint, W);
            const long long j = u - u0;
            const uint32_t bt = smem_addr(btile + (j & 1) * TC_BTILE);
            for (int qq = 0; qq < W.nblk / QUAD; ++qq, ++q) {
                const int b = static_cast<int>(q & 1);
                const bool w = tc_spin(&a_full[b], static_cast<unsigned>((q >> 1) & 1), abort_flag, P.status);
                ok = __all_sync(0xFFFFFFFFu, w) != 0;
                if (!ok) break;
                tc_fence_after();
                const uint32_t a_t = tm + static_cast<uint32_t>(b * TC_QCOLS);
                const uint32_t d_t = tm + static_cast<uint32_t>((2 + b) * TC_QCOLS);
#pragma unroll
                for (int jb = 0; jb < QUAD; ++jb) {
                    const uint32_t bb = bt + (qq * QUAD + jb) * 2 * TC_BHALF;
                    tc_mma_elect(d_t + jb * 16, a_t + jb * 16, tc_bdesc(bb, zaddr), TC_IDESC, 0);
                    tc_mma_elect(d_t + jb * 16, a_t + jb * 16 + 8, tc_bdesc(bb + TC_BHALF, zaddr), TC_IDESC, 1);
                }
                tc_commit_elect(&d_full[b]);
                __syncwarp();
            }
            // every warp has read this unit's stage: refill it
            if (ok && fu < u1) fill_stage();
        }
        // After an abort: wait (bounded) for the copies and MMAs still in
        // flight.  A slot is refilled (a D buffer recommitted) only after
        // the compute warps consumed its previous phase, so the last phase
        // of each barrier is the only one that can be pending: the last fill
        // f of slot i is the largest f < count with f % n == i.
        if (*abort_flag && lane == 0) {
            for (int i = 0; i < TC_NS; ++i) {
                const long long f = fi - 1 - ((fi - 1 - i) % TC_NS + TC_NS) % TC_NS;
                if (f >= 0) mbar_drain(&st_full[i], static_cast<unsigned>((f / TC_NS) & 1));
            }
            for (int i = 0; i < 2; ++i) {
                const long long c = q - 1 - ((q - 1 - i) % 2 + 2) % 2;
                if (c >= 0) mbar_drain(&d_full[i], static_cast<unsigned>((c >> 1) & 1));
            }
        }
        __syncwarp();
    } else {
        pdl_wait();
        const int wq = (tid >> 5) & 3;
        const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
        int hint = 0, nhint = 0, bhint = 0;
        float acc[4][T], yv[T];
#pragma unroll
        for (int p = 0; p < 4; ++p)
#pragma unroll
            for (int t = 0; t < T; ++t) acc[p][t] = 0.0f;
#pragma unroll
        for (int t = 0; t < T; ++t) yv[t] = 0.0f;
        // The pending quad: its sums are read back while the next quad is
        // converted (the MMAs of one quad overlap the next quad's work).
        float pdw[QUAD] = {0.0f, 0.0f, 0.0f, 0.0f};  // its rows' d_w
        uint32_t pca = 0;                             // its blocks' constants
        bool p_valid = false, p_end = false;          // pending; ends a segment
        TcUnit cu, pu = {0, 0, 0, 0, 0, 0};
        long long sp_tile = -1;  // the split tile whose slot and part count are cached
        int sp_gf = 0, sp_parts = 1;
        bool ok = true;
        long long qi = 0;  // quads of the range so far
        // This thread's share of a unit's activations: block R / 8, token R % 8.
        const int ablk = R >> 3, atok = R & 7;
        unsigned short dh_next = 0;  // its scale, loaded a unit ahead
        // The codes (cp.async, 32 bytes into source slot s) and the scale of
        // unit v, for this thread's (block, token).
        auto prefetch_src = [&](long long v, int slot) {
            TcUnit N;
            tc_decode(P, v, nhint, N);
            if (ablk < N.nblk && atok < T) {
                const TcItem &I = P.it[N.item];
                const uint8_t *src = I.xq + static_cast<long long>(atok) * I.K + (N.seg * SEG_BLOCKS + ablk) * QK;
                uint8_t *dst = bsrc + slot * TC_BSRC + atok * 512 + ablk * QK;
                cp_async16(dst, src);
                cp_async16(dst + 16, src + 16);
                dh_next = __ldg(reinterpret_cast<const unsigned short *>(
                    I.xq + static_cast<long long>(T) * I.K +
                    (static_cast<long long>(atok) * I.nb + N.seg * SEG_BLOCKS + ablk) * 2));
            }
            cp_async_commit();
        };

        // every wait's outcome is made warp-uniform: the tcgen05 loads and
        // stores below are warp-collective
        auto wait_all = [&](uint64_t *bar, long long n) {
            const bool w = ok && tc_wait(bar, static_cast<unsigned>(n & 1), abort_flag, P.status);
            return __all_sync(0xFFFFFFFFu, w) != 0;
        };
        auto spin_all = [&](uint64_t *bar, long long n) {
            const bool w = ok && tc_spin(bar, static_cast<unsigned>(n & 1), abort_flag, P.status);
            return __all_sync(0xFFFFFFFFu, w) != 0;
        };
        // The pending quad's sums: wait for its MMAs and start the loads.
        auto fetch = [&](long long qq_, float (&d)[QUAD][8]) {
            const int b = static_cast<int>(qq_ & 1);
            ok = spin_all(&d_full[b], qq_ >> 1);
            tc_fence_after();
#pragma unroll
            for (int jb = 0; jb < QUAD; ++jb) {
                unsigned rr[8];
                asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                             : "=r"(rr[0]), "=r"(rr[1]), "=r"(rr[2]), "=r"(rr[3]), "=r"(rr[4]), "=r"(rr[5]),
                               "=r"(rr[6]), "=r"(rr[7])
                             : "r"(tm + lane_base + static_cast<uint32_t>((2 + b) * TC_QCOLS + jb * 16))
                             : "memory");
#pragma unroll
                for (int i = 0; i < 8; ++i) d[jb][i] = __uint_as_float(rr[i]);
            }
        };
        // At a segment's end: fold the segment; at a tile's end store (or
        // hand the segment sums of a split tile to the workspace).
        auto seg_fold = [&]() {
            const TcItem &I = P.it[pu.item];
            const long long tu1 = pu.tile_u0 + I.nseg;
            const bool split = pu.tile_u0 < u0 || tu1 > u1;
            float Ps[T];
#pragma unroll
            for (int t = 0; t < T; ++t) {
                Ps[t] = __fmul_rn(__fadd_rn(__fadd_rn(acc[0][t], acc[1][t]), __fadd_rn(acc[2][t], acc[3][t])),
                                  MMA_UNSCALE);
#pragma unroll
                for (int p = 0; p < 4; ++p) acc[p][t] = 0.0f;
            }
            if (!split) {
                const int row = pu.tile * 128 + R;
                const bool live = R < pu.nsl * SLAB_ROWS;
#pragma unroll
                for (int t = 0; t < T; ++t) yv[t] = pu.seg == 0 ? Ps[t] : __fadd_rn(yv[t], Ps[t]);
                if (pu.seg == I.nseg - 1 && live && ok)
#pragma unroll
                    for (int t = 0; t < T; ++t) I.y[static_cast<long long>(t) * I.N + row] = yv[t];
                return;
            }
            // a tile shared with other groups: its slot belongs to the group
            // holding its first unit; the parts are the distinct owners of
            // its units (a group with an empty range owns none), counted once
            // per tile by walking the group starts inside it
            if (pu.tile_u0 != sp_tile) {
                sp_tile = pu.tile_u0;
                sp_gf = tc_group_of(U, P.groups, pu.tile_u0);
                sp_parts = 1;
                long long prev = tc_group_start(U, P.groups, sp_gf);
                for (long long g2 = sp_gf + 1; g2 < P.groups; ++g2) {
                    const long long st = tc_group_start(U, P.groups, g2);
                    if (st >= tu1) break;
                    sp_parts += st != prev;  // a non-empty group begins inside the tile
                    prev = st;
                }
            }
            const int gf = sp_gf, parts = sp_parts;
            float *slot = P.part + static_cast<long long>(gf + 1) * P.slot_floats;
#pragma unroll
            for (int t = 0; t < T; ++t) slot[(pu.seg * 8 + t) * 128 + R] = Ps[t];
            const bool part_end = pu.seg == I.nseg - 1 || pu.tile_u0 + pu.seg + 1 == u1;
            if (!part_end || !ok) return;
            // Warp w of every part arrives on the counter of rows 32w..32w+31;
            // the last of them adds those rows' segment sums in order, each
            // lane its own row, loading four segments ahead of the adds.
            __threadfence();
            __syncwarp();
            unsigned last = 0;
            unsigned *cw = P.cnt + (gf + 1) * 4 + wq;
            if (lane == 0) last = atomicAdd(cw, 1u) == static_cast<unsigned>(parts - 1) ? 1u : 0u;
            if (__shfl_sync(0xFFFFFFFFu, last, 0)) {
                __threadfence();
                float v[T];
#pragma unroll
                for (int t = 0; t < T; ++t) v[t] = __ldcg(slot + t * 128 + R);
                int s2 = 1;
                for (; s2 + 4 <= I.nseg; s2 += 4) {
                    float x[4][T];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int t = 0; t < T; ++t) x[i][t] = __ldcg(slot + ((s2 + i) * 8 + t) * 128 + R);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int t = 0; t < T; ++t) v[t] = __fadd_rn(v[t], x[i][t]);
                }
                for (; s2 < I.nseg; ++s2)
#pragma unroll
                    for (int t = 0; t < T; ++t) v[t] = __fadd_rn(v[t], __ldcg(slot + (s2 * 8 + t) * 128 + R));
                if (R < pu.nsl * SLAB_ROWS)
#pragma unroll
                    for (int t = 0; t < T; ++t) I.y[static_cast<long long>(t) * I.N + pu.tile * 128 + R] = v[t];
                __syncwarp();
                if (lane == 0) *cw = 0u;
            }
        };
        // The pending quad's four blocks into the phase sums (block jb of a
        // quad has phase jb), then its segment's fold if it ends one.
        auto accumulate = [&](const float (&d)[QUAD][8]) {
#pragma unroll
            for (int jb = 0; jb < QUAD; ++jb) {
                const uint32_t ca = pca + jb * 64;
                const float4 c0 = lds_f4(ca), c1 = lds_f4(ca + 16), x0 = lds_f4(ca + 32), x1 = lds_f4(ca + 48);
                const float C[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
                const float dx[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
                // (d_w d_x) is exact; D + C = isum 2^-24 exactly; two tokens per op
#pragma unroll
                for (int t = 0; t + 1 < T; t += 2) {
                    float s0, s1, v0 = d[jb][t], v1 = d[jb][t + 1];
                    fmul2(s0, s1, pdw[jb], pdw[jb], dx[t], dx[t + 1]);
                    fadd2(v0, v1, C[t], C[t + 1]);
                    ffma2(acc[jb][t], acc[jb][t + 1], s0, s1, v0, v1);
                }
                if (T & 1)
                    acc[jb][T - 1] =
                        __fmaf_rn(__fmul_rn(pdw[jb], dx[T - 1]), __fadd_rn(d[jb][T - 1], C[T - 1]), acc[jb][T - 1]);
            }
            if (p_end) seg_fold();
        };

        // B operand and constants of unit v (slot j & 1), from the codes this
        // thread copied and the scale it loaded a unit ahead
        auto build_b = [&](long long v, long long j) {
            TcUnit B;
            tc_decode(P, v, bhint, B);
            cp_async_wait();
            {
                const unsigned short dh = dh_next;
                if (ablk < B.nblk && atok < T) {
                    const uint8_t *src = bsrc + (j & 1) * TC_BSRC + atok * 512 + ablk * QK;
                    const uint4 qa = *reinterpret_cast<const uint4 *>(src);
                    const uint4 qb = *reinterpret_cast<const uint4 *>(src + 16);
                    const unsigned w[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
                    const int ones = 0x01010101;
                    int sq = 0;
#pragma unroll
                    for (int i = 0; i < 8; ++i) sq = dp4a_ss(static_cast<int>(w[i]), ones, sq);
                    unsigned lo[8], hi[8];  // k order: elements 4i + {0, 2, 1, 3}
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const unsigned bl = w[i] ^ 0x80808080u, bh = w[4 + i] ^ 0x80808080u;
                        lo[2 * i] = hadd2_u(act_even(bl), H2_NEG_1152);
                        lo[2 * i + 1] = hadd2_u(act_odd(bl), H2_NEG_1152);
                        hi[2 * i] = hfma2_u(act_even(bh), H2_SIXTEENTH, H2_NEG_72);
                        hi[2 * i + 1] = hfma2_u(act_odd(bh), H2_SIXTEENTH, H2_NEG_72);
                    }
                    uint8_t *bb = btile + (j & 1) * TC_BTILE + ablk * 2 * TC_BHALF + atok * 16;
                    *reinterpret_cast<uint4 *>(bb) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    *reinterpret_cast<uint4 *>(bb + 128) = make_uint4(lo[4], lo[5], lo[6], lo[7]);
                    *reinterpret_cast<uint4 *>(bb + TC_BHALF) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<uint4 *>(bb + TC_BHALF + 128) = make_uint4(hi[4], hi[5], hi[6], hi[7]);
                    float *cc = reinterpret_cast<float *>(cst + (j % TC_NCONST) * TC_CONST + ablk * 64);
                    cc[atok] = mma_fold_const(sq);
                    cc[8 + atok] = h2f(dh);
                }
                fence_proxy_async_smem();  // the B operand, for the tensor cores
            }
        };

        // Unit j + 1's B operand is built in the middle of unit j, once every
        // MMA of unit j - 1 (which read that slot) is known complete: after
        // the read-back of unit j's first quad.  Its activations were copied
        // a unit earlier.
        if (u0 < u1) {
            prefetch_src(u0, 0);
            build_b(u0, 0);
            if (u0 + 1 < u1) prefetch_src(u0 + 1, 1);
        }
        for (long long u = u0; u < u1 && ok; ++u) {
            const long long j = u - u0;
            tc_decode(P, u, hint, cu);
            // this unit's weights
            ok = wait_all(&st_full[j % TC_NS], j / TC_NS);
            if (!ok) break;
            const bool live = R < cu.nsl * SLAB_ROWS;
            const int sl = R >> 4, r = R & 15;
            const uint32_t st0 = smem_addr(ring + (j % TC_NS) * TC_STAGE) + sl * SEG_BYTES;
            for (int qq = 0; qq < cu.nblk / QUAD && ok; ++qq, ++qi) {
                const uint32_t st = st0 + qq * QUAD_BYTES;
                const uint4 sw = live ? lds_u4(st + 1024 + (r & 7) * 16) : make_uint4(0u, 0u, 0u, 0u);
                // this quad's A operand: four blocks, each row's 32 nibbles
                const uint32_t a_col = tm + lane_base + static_cast<uint32_t>((qi & 1) * TC_QCOLS);
#pragma unroll
                for (int jb = 0; jb < QUAD; ++jb) {
                    const uint4 n = live ? lds_u4(st + (r * QUAD + ((jb + (r >> 1)) & 3)) * 16)
                                         : make_uint4(0u, 0u, 0u, 0u);
                    const unsigned nw[4] = {n.x, n.y, n.z, n.w};
                    unsigned a[16];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const unsigned w8 = __umulhi(nw[i], c_shr8_mul);  // nw >> 8
                        a[2 * i] = nw[i] & 0x000F000Fu;
                        a[2 * i + 1] = w8 & 0x000F000Fu;
                        a[8 + 2 * i] = nw[i] & 0x00F000F0u;
                        a[8 + 2 * i + 1] = w8 & 0x00F000F0u;
                    }
                    tc_st16(a_col + jb * 16, a);
                }
                // then the pending quad's sums (its MMAs ran during the conversion)
                float d[QUAD][8];
                if (p_valid) fetch(qi - 1, d);
                if (p_valid) asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                tc_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&a_full[qi & 1]);
                if (p_valid) accumulate(d);
                // this quad becomes the pending one
                const unsigned swv[4] = {sw.x, sw.y, sw.z, sw.w};
#pragma unroll
                for (int jb = 0; jb < QUAD; ++jb) pdw[jb] = h2f((r >> 3) ? (swv[jb] >> 16) : swv[jb]);
                pca = smem_addr(cst + (j % TC_NCONST) * TC_CONST + qq * QUAD * 64);
                p_end = qq == cu.nblk / QUAD - 1;
                pu = cu;
                p_valid = true;
                if (qq == 0 && u + 1 < u1) {  // unit j - 1's last quad has been read back
                    build_b(u + 1, j + 1);
                    if (u + 2 < u1) prefetch_src(u + 2, static_cast<int>(j & 1));
                }
            }
        }
        // the last quad
        if (ok && p_valid) {
            float d[QUAD][8];
            fetch(qi - 1, d);
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            tc_fence_before();
            if (ok) accumulate(d);
        }
        cp_async_wait();  // no copy outlives the kernel
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(s_tmem), "r"(TC_TMEM_COLS)
                                : "memory");
}

}  // namespace qg

// ------------------------------------------------------------ host side

namespace qg {

bool tc_eligible(const TcSpec *s, int n, int T)
{
    if (n < 1 || n > MAXG_SEQ || T < 1 || T > 8) return false;
    for (int i = 0; i < n; ++i)
        if (s[i].N < SLAB_ROWS || s[i].N % SLAB_ROWS != 0 || s[i].K % 256 != 0 || s[i].N >= (1ll << 31))
            return false;
    return true;
}

static long long tc_units(const TcSpec *s, int n, int &nseg_max)
{
    long long u = 0;
    nseg_max = 1;
    for (int i = 0; i < n; ++i) {
        const long long nb = s[i].K / QK, nseg = (nb + SEG_BLOCKS - 1) / SEG_BLOCKS, ntiles = (s[i].N + 127) / 128;
        u += ntiles * nseg;
        if (nseg > nseg_max) nseg_max = static_cast<int>(nseg);
    }
    return u;
}

long long tc_ws_bytes(const TcSpec *s, int n, int grid)
{
    int nseg_max = 1;
    tc_units(s, n, nseg_max);
    const long long groups = static_cast<long long>(grid) * TC_GROUPS;
    return TC_CNT_BYTES + groups * nseg_max * 8 * 128 * 4;
}

template <int T>
static cudaError_t launch_tc_t(const TcParams &P, int grid, cudaStream_t st)
{
    auto kern = qgemv_tc_kernel<T>;
    static std::atomic<unsigned long long> raised{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(raised.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, TC_SMEM);
        if (e != cudaSuccess) return e;
        raised.fetch_or(bit, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(TC_THREADS);
    cfg.dynamicSmemBytes = TC_SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, P);
}

cudaError_t launch_tc(const TcSpec *s, int n, int T, uint8_t *ws, int grid, unsigned *status, cudaStream_t st)
{
    // four arrival counters per warp group must fit the counter area
    if (grid < 1 || static_cast<long long>(grid) * TC_GROUPS * 4 * 4 > TC_CNT_BYTES) return cudaErrorInvalidValue;
    std::unique_ptr<TcParams> P(new TcParams());
    memset(P.get(), 0, sizeof(TcParams));
    int nseg_max = 1;
    P->total_units = tc_units(s, n, nseg_max);
    P->nitems = n;
    P->groups = grid * TC_GROUPS;
    P->slot_floats = nseg_max * 8 * 128;
    P->cnt = reinterpret_cast<unsigned *>(ws);
    P->part = reinterpret_cast<float *>(ws + TC_CNT_BYTES);
    P->status = status;
    long long u = 0;
    for (int i = 0; i < n; ++i) {
        TcItem &I = P->it[i];
        I.W = static_cast<const uint8_t *>(s[i].W);
        I.xq = static_cast<const uint8_t *>(s[i].xq);
        I.y = s[i].y;
        I.N = static_cast<int>(s[i].N);
        I.K = static_cast<int>(s[i].K);
        I.nb = I.K / QK;
        I.nseg = (I.nb + SEG_BLOCKS - 1) / SEG_BLOCKS;
        I.ntiles = (I.N + 127) / 128;
        I.slab_bytes = static_cast<long long>(SLAB_COL_BYTES) * I.nb;
        I.unit_begin = u;
        u += static_cast<long long>(I.ntiles) * I.nseg;
    }
    switch (T) {
    case 1: return launch_tc_t<1>(*P, grid, st);
    case 2: return launch_tc_t<2>(*P, grid, st);
    case 3: return launch_tc_t<3>(*P, grid, st);
    case 4: return launch_tc_t<4>(*P, grid, st);
    case 5: return launch_tc_t<5>(*P, grid, st);
    case 6: return launch_tc_t<6>(*P, grid, st);
    case 7: return launch_tc_t<7>(*P, grid, st);
    case 8: return launch_tc_t<8>(*P, grid, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qg
