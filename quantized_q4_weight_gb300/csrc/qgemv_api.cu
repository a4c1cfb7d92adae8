// qgemv_api.cu -- the C ABI of libqgemv (include/qgemv.h): argument
// validation, launch planning and kernel launches.  Host code only, apart
// from the per-device status word.
#include <algorithm>
#include <atomic>
#include <cstring>
#include <memory>
#include <mutex>
#include <vector>

#include "../../include/qgemv.h"
#include "gemv_kernel.cuh"
#include "qgemv_launch.h"

using namespace qg;

// Per-device status word: kernels record the first asynchronous error here.
__device__ unsigned g_qgemv_status = 0;

namespace {

constexpr int kMaxDevices = 64;

struct DevInfo {
    bool ready = false;
    int sms = 0;
    int smem_optin = 0;   // per CTA
    int smem_per_sm = 0;
    unsigned *status = nullptr;
};

// Launch shape of the streaming kernel (0 = default): CTAs resident per SM
// (1: one CTA of up to 16 warps; 2: two CTAs of 8 warps), waves of CTAs per
// launch and weight stages per warp.  Results never depend on them.
std::atomic<int> g_ctas_per_sm{0}, g_waves{0}, g_ring_depth{0};
// Token count from which T > 1 runs on the f16 tensor-core path (0 = default).
std::atomic<int> g_mma_min_T{0};
constexpr int kDefaultMmaMinT = 5;
// Token count from which packed sequences run on the tcgen05 kernel (0 =
// default; 9 = never).  Off by default: on GB300 the mma.sync path is faster
// at every T (3B 36-layer set, T = 8: 0.37 ms against 0.73 ms).
std::atomic<int> g_tc_min_T{0};
constexpr int kDefaultTcMinT = 9;

// The decode FFN step as one fused launch where it applies (1) or always as
// three launches (0).
std::atomic<int> g_ffn_fused{1};

inline bool tc_for(int T)
{
    const int m = g_tc_min_T.load(std::memory_order_relaxed);
    return T >= (m >= 1 ? m : kDefaultTcMinT);
}

inline bool mma_for(int T)
{
    const int m = g_mma_min_T.load(std::memory_order_relaxed);
    return T >= 2 && T >= (m >= 2 ? m : kDefaultMmaMinT);
}

std::mutex g_dev_mu;
DevInfo g_dev[kMaxDevices];

qgemv_status device_info(DevInfo &out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QGEMV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DevInfo &d = g_dev[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return QGEMV_ERR_CUDA;
        if (cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return QGEMV_ERR_CUDA;
        if (cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess)
            return QGEMV_ERR_CUDA;
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_qgemv_status) != cudaSuccess) return QGEMV_ERR_CUDA;
        d.status = static_cast<unsigned *>(p);
        d.ready = true;
    }
    out = d;
    return QGEMV_OK;
}

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline long long align_up(long long v, long long a) { return (v + a - 1) / a * a; }

struct Range {
    uintptr_t lo, hi;
};
inline Range range(const void *p, long long bytes)
{
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return Range{a, a + static_cast<uintptr_t>(bytes)};
}
inline bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

bool shape_ok(long long N, long long K)
{
    return N >= 1 && N < (1ll << 31) && K >= QK && K % QK == 0 && K <= (1ll << 24) && N * (K / QK) < (1ll << 40);
}

// One matrix family of a launch, as the caller describes it.
struct GroupSpec {
    const void *W;
    long long w_stride;
    const void *xq;
    long long xq_stride;
    float *y;
    long long y_stride;
    long long N, K;
    int count;
    const float *bias = nullptr;  // sequence epilogue: bias[N] (count 1 only)
    const float *res = nullptr;   // sequence epilogue: residual[T][N] (count 1 only; may be y)
};

// Launch plan: the kernel parameter block (without device pointers into the
// workspace until `ws` is given), the workspace size and the shared memory.
template <int MAXG>
struct Plan {
    Params<MAXG> P;
    long long ws_bytes = 0;
    size_t smem = 0;
};

// Workspace layout, the same for every entry point: a counter area of
// CNT_AREA bytes (index 0: argmax arrival counter; then the split-K
// counters of each split group), then the data (argmax candidates, split-K
// partials).  Counters are only ever used as counters and every completed
// call leaves them at zero, so calls of any kind may share a workspace.
constexpr long long CNT_AREA = 16384;
constexpr long long AM_KEY_BYTES = 64;  // the last 64 bytes of the counter area: argmax running maxima [T]
static_assert(CNT_AREA / 4 > SPLIT_SLAB_THRESHOLD, "split-K counters must fit the counter area");

// Partition weight of one weight byte of a group, in sixteenths, so that
// CTAs get equal time rather than equal bytes where the per-block work
// differs: on the tensor-core path (compute-bound) a group whose activations
// take the int8 image, too large for the f16 operand image, converts them to
// f16 in every warp and block; measured at about 1.125 times the time per
// byte of an f16-image group.  The partition never changes a result.
constexpr int PART_OVH_KB_MMA = 256;   // tensor-core path (T >= 5 by default)
constexpr int PART_OVH_KB_DP4A = 176;  // dp4a path at three and four tokens
constexpr int PART_OVH_KB_FEW = 96;    // dp4a path at one and two tokens

inline int partition_cost(int T, int K, bool mma)
{
    return mma && !xq_layout(T, K, true).f16 ? 18 : 16;
}

// The fixed partition cost of each GEMV a CTA meets, in KB of weights.
inline int partition_overhead_kb(int T, bool mma)
{
    return mma ? PART_OVH_KB_MMA : (T >= 3 ? PART_OVH_KB_DP4A : PART_OVH_KB_FEW);
}

template <int MAXG>
qgemv_status make_plan(const GroupSpec *gs, int n, int T, bool ggml, bool argmax, uint8_t *ws, int smem_limit,
                       Plan<MAXG> &pl, int ctas_per_sm = 1, bool mma = false)
{
    if (n < 1 || n > MAXG) return QGEMV_ERR_INTERNAL;
    Params<MAXG> &P = pl.P;
    memset(&P, 0, sizeof(P));
    P.ngroups = n;
    P.ggml = ggml ? 1 : 0;
    long long total_slabs = 0;
    for (int i = 0; i < n; ++i) {
        const long long nb = gs[i].K / QK;
        const long long nslabs = ggml ? (gs[i].N + SLAB_ROWS - 1) / SLAB_ROWS : gs[i].N / SLAB_ROWS;
        total_slabs += nslabs * gs[i].count;
        (void)nb;
    }
    // The partition's fixed cost of each group instance (each GEMV a CTA
    // meets costs a group barrier and its activation image).  Per-CTA timing
    // probes fitted about 12 us per GEMV at T = 8, 5 us at T = 4 (36-layer
    // 3B set) and 2 us at T = 1 (28-layer 1.5B set) beyond the per-byte
    // costs; same-box sweeps of the charge were best at 256 KB (T = 8; 0,
    // 128, 448 and 704 KB slower), 176 KB (T = 4; 96 and 320 KB slower) and
    // 96 KB (T = 1, 2: the 1.5B set 0.7 % and the MoE gather 9 % faster than
    // none; 144, 192, 320 KB slower).  The int8-image groups stay at 18/16
    // per byte (20/16 measured worse).
    // (A launch of one matrix has nothing to balance: the charge would only
    // leave its first CTAs idle.)
    long long instances = 0;
    for (int i = 0; i < n; ++i) instances += gs[i].count;
    P.part_ovh_kb = instances > 1 ? partition_overhead_kb(T, mma) : 0;
    const long long ovh = static_cast<long long>(P.part_ovh_kb) * 1024 * 16;
    long long off = CNT_AREA;  // data
    long long cnt_off = 4;     // counters (argmax arrival counter at 0)
    if (argmax) {
        P.am_cnt = ws ? reinterpret_cast<unsigned *>(ws) : nullptr;
        P.am_key = ws ? reinterpret_cast<unsigned long long *>(ws + CNT_AREA - AM_KEY_BYTES) : nullptr;
        P.am_cand = ws ? reinterpret_cast<unsigned long long *>(ws + off) : nullptr;
        off = align_up(off + static_cast<long long>(MAX_GRID) * T * 16, 256);  // a key pair per CTA and token
    }
    long long cost = 0, items = 0;
    int kmax = 0, nbmax = 0;
    for (int i = 0; i < n; ++i) {
        Group &g = P.g[i];
        const GroupSpec &s = gs[i];
        g.W = static_cast<const uint8_t *>(s.W);
        g.w_stride = s.w_stride;
        g.xq = static_cast<const uint8_t *>(s.xq);
        g.xq_stride = s.xq_stride;
        g.y = s.y;
        g.y_stride = s.y_stride;
        if (s.bias != nullptr || s.res != nullptr) {
            // a sequence item (one instance): the stride words carry the epilogue
            if (s.count != 1 || s.w_stride != 0 || s.y_stride != 0) return QGEMV_ERR_INTERNAL;
            g.bias = s.bias;
            g.res = s.res;
            P.epilogue = 1;
        }
        g.N = static_cast<int>(s.N);
        g.K = static_cast<int>(s.K);
        g.count = s.count;
        g.nb = g.K / QK;
        g.nseg = (g.nb + SEG_BLOCKS - 1) / SEG_BLOCKS;
        if (ggml) {
            g.nslabs = (g.N + SLAB_ROWS - 1) / SLAB_ROWS;
            g.tail_rows = 0;
        } else {
            g.nslabs = g.N / SLAB_ROWS;
            g.tail_rows = g.N % SLAB_ROWS;
        }
        g.split = (g.nseg > 1 && g.nslabs > 0 && total_slabs < SPLIT_SLAB_THRESHOLD) ? g.nseg : 1;
        g.items_per_inst = g.nslabs * g.split + (g.tail_rows > 0 ? 1 : 0);
        g.xq_bytes = static_cast<int>(xq_bytes_host(T, g.K));
        g.slab_bytes = static_cast<long long>(SLAB_COL_BYTES) * g.nb;
        g.inst_bytes = g.nslabs * g.slab_bytes + static_cast<long long>(g.tail_rows) * g.nb * Q4_BYTES;
        g.cost = partition_cost(T, g.K, mma);
        g.cost_begin = cost;
        g.item_begin = static_cast<int>(items);
        cost += (ovh + g.inst_bytes * g.cost) * g.count;
        items += static_cast<long long>(g.items_per_inst) * g.count;
        if (g.split > 1) {
            const long long nc = static_cast<long long>(g.count) * g.nslabs;
            g.cnt = ws ? reinterpret_cast<unsigned *>(ws + cnt_off) : nullptr;
            cnt_off += nc * 4;
            if (cnt_off > CNT_AREA - AM_KEY_BYTES) return QGEMV_ERR_INTERNAL;  // the argmax maxima end the area
            g.part = ws ? reinterpret_cast<float *>(ws + off) : nullptr;
            off = align_up(off + nc * g.nseg * T * 16 * 4, 256);
        }
        if (g.K > kmax) kmax = g.K;
        if (g.nb > nbmax) nbmax = g.nb;
    }
    P.total_cost = cost;
    P.total_items = items;
    P.kmax = kmax;
    P.nbmax = nbmax;
    pl.ws_bytes = off;

    // Shared memory: [activation area][run table][boundary sums][flags][barriers][rings].
    // The activation area holds one run's activations in the run-synced mode
    // ([T][kmax] int8, fp16 scales, folded constants) and as many runs as fit
    // in the balanced mode.
    long long need_x = 0;  // the largest single-run activation image
    for (int i = 0; i < n; ++i) need_x = std::max<long long>(need_x, xq_layout(T, P.g[i].K, mma).bytes);
    P.off_d = 0;
    P.off_cd = 0;
    const long long tables = align_up(static_cast<long long>(MAX_RUNS) * sizeof(RunInfo), 128) +
                             align_up(static_cast<long long>(NWARPS_MAX) * T * 16 * 4, 128) + 128 +
                             align_up(static_cast<long long>(std::min(GCACHE_GROUPS, n)) * sizeof(Group), 128);
    P.balanced_ok = 1;
    for (int i = 0; i < n; ++i)
        if (P.g[i].split > 1) P.balanced_ok = 0;
    P.ring_depth = 0;
    // 2 stages per warp and the widest warp count that leaves room for the
    // largest activation image; then, on the tensor-core path (whose warps
    // are compute-bound), the widest count at one stage; then 8 warps.
    const int wide = ctas_per_sm > 1 ? 8 : max_warps_for(T, mma);
    const int rd = g_ring_depth.load(std::memory_order_relaxed);
    // measured defaults: three stages per warp pay off for long one-token
    // sequences only (layer sets); single matrices, lm_head and gathers run two
    const int D0 = rd > 0 ? rd : (!mma && T == 1 && MAXG == MAXG_SEQ ? 3 : 2);
    const int choices[5][2] = {{wide, D0}, {mma ? wide : 8, mma ? 1 : D0}, {8, D0}, {8, 2}, {8, 1}};
    for (const auto &c : choices) {
        const int nw = c[0], D = c[1];
        const long long bars = align_up(8ll * (nw * D + 1), 128);
        const long long rings = ggml ? 0 : static_cast<long long>(nw) * D * SEG_BYTES;
        long long xa = smem_limit > 0 ? smem_limit - tables - bars - rings : need_x;
        xa = xa / 128 * 128;
        if (xa >= need_x) {
            P.nwarps = nw;
            P.ring_depth = D;
            P.xq_area = static_cast<int>(xa);
            P.off_runs = static_cast<int>(xa);
            P.off_hbuf = static_cast<int>(xa + align_up(static_cast<long long>(MAX_RUNS) * sizeof(RunInfo), 128));
            P.off_hflag = static_cast<int>(P.off_hbuf + align_up(static_cast<long long>(NWARPS_MAX) * T * 16 * 4, 128));
            P.off_gcache = P.off_hflag + 128;
            P.off_bar = static_cast<int>(xa + tables);
            P.off_ring = static_cast<int>(xa + tables + bars);
            pl.smem = static_cast<size_t>(xa + tables + bars + rings);
            break;
        }
    }
    if (P.ring_depth == 0) return QGEMV_ERR_UNSUPPORTED;
    if (items >= (1ll << 31)) return QGEMV_ERR_UNSUPPORTED;
    return QGEMV_OK;
}

template <int MAXG, bool ARGMAX>
cudaError_t dispatch_T(const Params<MAXG> &P, int T, bool mma, int grid, size_t smem, cudaStream_t st, bool pdl)
{
#define QG_CASE(t)                                                                                         \
    case t:                                                                                                \
        return mma ? launch_stream<t, MAXG, ARGMAX, true>(P, grid, smem, st, pdl)                          \
                   : launch_stream<t, MAXG, ARGMAX, false>(P, grid, smem, st, pdl);
    switch (T) {
    case 1: return launch_stream<1, MAXG, ARGMAX, false>(P, grid, smem, st, pdl);
    QG_CASE(2)
    QG_CASE(3)
    QG_CASE(4)
    QG_CASE(5)
    QG_CASE(6)
    QG_CASE(7)
    QG_CASE(8)
    default: return cudaErrorInvalidValue;
    }
#undef QG_CASE
}

// Sequence launches with the output epilogue: compiled for each T's default
// path only (dp4a below five tokens, tensor cores from five); a launch on the
// other path (moved by qgemv_set_tuning) is refused with cudaErrorNotSupported.
cudaError_t dispatch_ep(const Params<MAXG_SEQ> &P, int T, bool mma, int grid, size_t smem, cudaStream_t st)
{
    if (mma != (T >= kDefaultMmaMinT)) return cudaErrorNotSupported;
    switch (T) {
    case 1: return launch_stream<1, MAXG_SEQ, false, false, true>(P, grid, smem, st, true);
    case 2: return launch_stream<2, MAXG_SEQ, false, false, true>(P, grid, smem, st, true);
    case 3: return launch_stream<3, MAXG_SEQ, false, false, true>(P, grid, smem, st, true);
    case 4: return launch_stream<4, MAXG_SEQ, false, false, true>(P, grid, smem, st, true);
    case 5: return launch_stream<5, MAXG_SEQ, false, true, true>(P, grid, smem, st, true);
    case 6: return launch_stream<6, MAXG_SEQ, false, true, true>(P, grid, smem, st, true);
    case 7: return launch_stream<7, MAXG_SEQ, false, true, true>(P, grid, smem, st, true);
    case 8: return launch_stream<8, MAXG_SEQ, false, true, true>(P, grid, smem, st, true);
    default: return cudaErrorInvalidValue;
    }
}

// CTAs per SM for a T-token launch, and the dynamic shared-memory budget of
// one CTA (the kernel's static arrays take at most 600 bytes).
inline int ctas_per_sm_for(int T, bool sequence)
{
    const int c = g_ctas_per_sm.load(std::memory_order_relaxed);
    if (!mma_for(T) && T > 4) return 1;  // 8 warps of wide accumulators fill the register file
    if (c >= 1 && c <= 2) return c;
    (void)sequence;  // measured: one CTA per SM with three stages per warp beats two CTAs of 8 warps
    return 1;
}
inline int smem_budget(const DevInfo &d, int ctas_per_sm)
{
    const int per = ctas_per_sm > 1 ? d.smem_per_sm / ctas_per_sm - 1024 : d.smem_optin;
    return per - 2048;
}
// Plan with the preferred CTAs per SM; if the activations do not fit two
// CTAs' shared memory, one CTA per SM.
template <int MAXG>
qgemv_status plan_launch(const GroupSpec *gs, int n, int T, bool ggml, bool argmax, uint8_t *ws, const DevInfo &d,
                         int &cps, Plan<MAXG> &pl)
{
    const bool mma = mma_for(T);
    // argmax kernels hold [warps][T][2] key pairs in static shared memory (up to 2 KB)
    const int extra = argmax ? 1024 : 0;
    qgemv_status s = make_plan<MAXG>(gs, n, T, ggml, argmax, ws, smem_budget(d, cps) - extra, pl, cps, mma);
    if (s == QGEMV_ERR_UNSUPPORTED && cps > 1) {
        cps = 1;
        s = make_plan<MAXG>(gs, n, T, ggml, argmax, ws, smem_budget(d, cps) - extra, pl, cps, mma);
    }
    return s;
}

// The first item whose weights start at or after position X of the launch's
// weighted byte space (each group's bytes times its cost), for the group g
// that holds X (g.cost_begin <= X <= the next group's cost_begin; X below the
// launch's total).  Within an instance, slab s and its segment part p start at
// (s * slab_bytes + p * spp * SEG_BYTES) * cost; the tail follows the slabs.
// Each instance is preceded by a fixed cost ovh (its activations' set-up):
// a position inside it maps to the instance's first item.
inline long long first_item_in_group(const Group &g, long long X, long long ovh)
{
    const long long local = X - g.cost_begin;
    const long long inst = ovh + g.inst_bytes * g.cost, slab = g.slab_bytes * g.cost;
    const long long e = local / inst;
    const long long rem = local - e * inst - ovh;
    const long long base = g.item_begin + e * g.items_per_inst;
    if (rem <= 0) return base;
    const long long slabs_bytes = static_cast<long long>(g.nslabs) * slab;
    if (rem < slabs_bytes) {
        const long long s = rem / slab;
        const long long r2 = rem - s * slab;
        if (r2 == 0) return base + s * g.split;
        const int spp = (g.nseg + g.split - 1) / g.split;
        const long long pb = static_cast<long long>(spp) * SEG_BYTES * g.cost;
        const long long p = (r2 + pb - 1) / pb;
        if (p >= g.split) return base + (s + 1) * g.split;
        return base + s * g.split + p;
    }
    if (rem == slabs_bytes) return base + static_cast<long long>(g.nslabs) * g.split;
    return base + g.items_per_inst;
}

// Each CTA's range of the launch's weighted bytes, [total c / grid,
// total (c + 1) / grid), as items: the first item of every range (and the
// launch's item count after the last one), and the group holding that item,
// so that the kernel's prologue reads its range and descriptors in one round.
template <int MAXG>
void set_cta_groups(Params<MAXG> &P, int grid)
{
    const long long ovh = static_cast<long long>(P.part_ovh_kb) * 1024 * 16;
    int gi = 0;
    for (int c = 0; c <= grid; ++c) {
        const long long x = P.total_cost * c / grid;
        const long long b = x >= P.total_cost ? P.total_cost - 1 : x;
        while (gi + 1 < P.ngroups && P.g[gi + 1].cost_begin <= b) ++gi;
        P.cta_g0[c] = static_cast<unsigned char>(gi);
        P.cta_i0[c] = static_cast<int>(x >= P.total_cost ? P.total_items : first_item_in_group(P.g[gi], x, ovh));
    }
}

inline int grid_for(const DevInfo &d, int ctas_per_sm)
{
    const int w = g_waves.load(std::memory_order_relaxed);
    const long long g = static_cast<long long>(d.sms) * ctas_per_sm * (w >= 1 ? w : 1);
    return static_cast<int>(g < MAX_GRID ? g : MAX_GRID);
}

// Shared argument checks of the single-matrix GEMV calls.
qgemv_status check_single(const void *W, qgemv_wlayout layout, const void *xin, long long xin_bytes,
                          const float *y, long long N, long long K, int T, const void *ws)
{
    if (!shape_ok(N, K) || T < 1 || T > 8) return QGEMV_ERR_INVALID_ARG;
    if (layout != QGEMV_W_GGML && layout != QGEMV_W_PACKED) return QGEMV_ERR_INVALID_ARG;
    if (!W || !xin) return QGEMV_ERR_INVALID_ARG;
    if (!aligned(W, layout == QGEMV_W_PACKED ? 16 : 2)) return QGEMV_ERR_MISALIGNED;
    if (ws && !aligned(ws, 256)) return QGEMV_ERR_MISALIGNED;
    if (y) {
        if (!aligned(y, 4)) return QGEMV_ERR_MISALIGNED;
        const Range ry = range(y, 4ll * T * N);
        if (overlap(ry, range(W, 18ll * N * (K / QK))) || overlap(ry, range(xin, xin_bytes)))
            return QGEMV_ERR_INVALID_ARG;
    }
    return QGEMV_OK;
}

long long single_ws_bytes(long long N, long long K, int T)
{
    GroupSpec gs{nullptr, 0, nullptr, 0, nullptr, 0, N, K, 1};
    Plan<MAXG_SMALL> pl;
    make_plan<MAXG_SMALL>(&gs, 1, T, false, true, nullptr, 0, pl);
    Plan<MAXG_SMALL> pg;  // the GGML layout splits its partial slab too
    make_plan<MAXG_SMALL>(&gs, 1, T, true, true, nullptr, 0, pg);
    return pl.ws_bytes > pg.ws_bytes ? pl.ws_bytes : pg.ws_bytes;
}

qgemv_status run_single(const void *W, qgemv_wlayout layout, const void *xq, float *y, long long *idx, long long N,
                        long long K, int T, void *ws, size_t ws_bytes, cudaStream_t st, bool argmax, bool pdl,
                        bool xf32 = false, long long *idx2 = nullptr, float *val2 = nullptr,
                        const long long *vc_tokens = nullptr, int *vc_n = nullptr)
{
    DevInfo dev;
    qgemv_status s = device_info(dev);
    if (s != QGEMV_OK) return s;
    GroupSpec gs{W, 0, xq, 0, y, 0, N, K, 1};
    Plan<MAXG_SMALL> pl;
    int cps = ctas_per_sm_for(T, false);
    s = plan_launch<MAXG_SMALL>(&gs, 1, T, layout == QGEMV_W_GGML, argmax, static_cast<uint8_t *>(ws), dev, cps, pl);
    if (s != QGEMV_OK) return s;
    if (static_cast<long long>(ws_bytes) < pl.ws_bytes) return QGEMV_ERR_WORKSPACE;
    pl.P.status = dev.status;
    pl.P.xf32 = xf32 ? 1 : 0;
    pl.P.am_idx = reinterpret_cast<long long *>(idx);
    pl.P.am_idx2 = idx2;
    pl.P.am_val2 = val2;
    pl.P.vc_tokens = vc_tokens;
    pl.P.vc_n = vc_n;
    const int grid = grid_for(dev, cps);
    set_cta_groups(pl.P, grid);
    const cudaError_t e = argmax ? dispatch_T<MAXG_SMALL, true>(pl.P, T, mma_for(T), grid, pl.smem, st, pdl)
                                 : dispatch_T<MAXG_SMALL, false>(pl.P, T, mma_for(T), grid, pl.smem, st, pdl);
    return e == cudaSuccess ? QGEMV_OK : QGEMV_ERR_CUDA;
}

}  // namespace

// =====================================================================
extern "C" {

const char *qgemv_status_string(qgemv_status s)
{
    switch (s) {
    case QGEMV_OK: return "QGEMV_OK";
    case QGEMV_ERR_INVALID_ARG: return "QGEMV_ERR_INVALID_ARG";
    case QGEMV_ERR_MISALIGNED: return "QGEMV_ERR_MISALIGNED";
    case QGEMV_ERR_UNSUPPORTED: return "QGEMV_ERR_UNSUPPORTED";
    case QGEMV_ERR_WORKSPACE: return "QGEMV_ERR_WORKSPACE";
    case QGEMV_ERR_CUDA: return "QGEMV_ERR_CUDA";
    case QGEMV_ERR_TIMEOUT: return "QGEMV_ERR_TIMEOUT";
    case QGEMV_ERR_BAD_ID: return "QGEMV_ERR_BAD_ID";
    case QGEMV_ERR_INTERNAL: return "QGEMV_ERR_INTERNAL";
    }
    return "QGEMV_UNKNOWN_STATUS";
}

int qgemv_version(void) { return 100; }

size_t qgemv_q4_0_bytes(int64_t N, int64_t K)
{
    if (!shape_ok(N, K)) return 0;
    return static_cast<size_t>(18ll * N * (K / QK));
}

size_t qgemv_xq_bytes(int R, int64_t K)
{
    if (R < 1 || K < QK || K % QK != 0 || K > (1ll << 24)) return 0;
    return static_cast<size_t>(xq_bytes_host(R, K));
}

qgemv_status qgemv_pack_q4_0(const void *w_ggml, void *w_packed, int64_t N, int64_t K, qgemv_stream_t stream)
{
    if (!shape_ok(N, K) || !w_ggml || !w_packed) return QGEMV_ERR_INVALID_ARG;
    if (!aligned(w_packed, 16) || !aligned(w_ggml, 2)) return QGEMV_ERR_MISALIGNED;
    const long long bytes = 18ll * N * (K / QK);
    if (overlap(range(w_ggml, bytes), range(w_packed, bytes))) return QGEMV_ERR_INVALID_ARG;
    return launch_pack(w_ggml, w_packed, N, K, true, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? QGEMV_OK
               : QGEMV_ERR_CUDA;
}

qgemv_status qgemv_unpack_q4_0(const void *w_packed, void *w_ggml, int64_t N, int64_t K, qgemv_stream_t stream)
{
    if (!shape_ok(N, K) || !w_ggml || !w_packed) return QGEMV_ERR_INVALID_ARG;
    if (!aligned(w_packed, 16) || !aligned(w_ggml, 2)) return QGEMV_ERR_MISALIGNED;
    const long long bytes = 18ll * N * (K / QK);
    if (overlap(range(w_ggml, bytes), range(w_packed, bytes))) return QGEMV_ERR_INVALID_ARG;
    return launch_pack(w_packed, w_ggml, N, K, false, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? QGEMV_OK
               : QGEMV_ERR_CUDA;
}

qgemv_status qgemv_quantize_q8_0(const float *x, void *xq, int R, int64_t K, int batch, qgemv_stream_t stream)
{
    if (!x || !xq || R < 1 || batch < 1 || K < QK || K % QK != 0 || K > (1ll << 24)) return QGEMV_ERR_INVALID_ARG;
    if (static_cast<long long>(R) * batch > (1ll << 31)) return QGEMV_ERR_INVALID_ARG;
    if (!aligned(xq, 16) || !aligned(x, 4)) return QGEMV_ERR_MISALIGNED;
    if (overlap(range(x, 4ll * batch * R * K), range(xq, xq_bytes_host(R, K) * batch))) return QGEMV_ERR_INVALID_ARG;
    return launch_quantize(x, xq, R, K, batch, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? QGEMV_OK
               : QGEMV_ERR_CUDA;
}

size_t qgemv_workspace_bytes(int64_t N, int64_t K, int T)
{
    if (!shape_ok(N, K) || T < 1 || T > 8) return 0;
    return static_cast<size_t>(single_ws_bytes(N, K, T));
}

qgemv_status qgemv_q4_0(const void *W, qgemv_wlayout layout, const void *xq, float *y, int64_t N, int64_t K, int T,
                        void *ws, size_t ws_bytes, qgemv_stream_t stream)
{
    qgemv_status s = check_single(W, layout, xq, shape_ok(N, K) ? xq_bytes_host(T, K) : 0, y, N, K, T, ws);
    if (s != QGEMV_OK) return s;
    if (!y) return QGEMV_ERR_INVALID_ARG;
    if (!aligned(xq, 16)) return QGEMV_ERR_MISALIGNED;
    if (!ws) return QGEMV_ERR_WORKSPACE;
    if (overlap(range(y, 4ll * T * N), range(ws, static_cast<long long>(ws_bytes)))) return QGEMV_ERR_INVALID_ARG;
    return run_single(W, layout, xq, y, nullptr, N, K, T, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream), false,
                      true);
}

qgemv_status qgemv_q4_0_f32(const void *W, qgemv_wlayout layout, const float *x, float *y, int64_t N, int64_t K,
                            int T, void *ws, size_t ws_bytes, qgemv_stream_t stream)
{
    qgemv_status s = check_single(W, layout, x, 4ll * T * K, y, N, K, T, ws);
    if (s != QGEMV_OK) return s;
    if (!y) return QGEMV_ERR_INVALID_ARG;
    if (!aligned(x, 4)) return QGEMV_ERR_MISALIGNED;
    if (!ws) return QGEMV_ERR_WORKSPACE;
    const long long need = single_ws_bytes(N, K, T);
    if (static_cast<long long>(ws_bytes) < need) return QGEMV_ERR_WORKSPACE;
    if (overlap(range(y, 4ll * T * N), range(ws, need)) || overlap(range(x, 4ll * T * K), range(ws, need)))
        return QGEMV_ERR_INVALID_ARG;
    // The kernel quantises x itself, after griddepcontrol.wait, so it may
    // start (and stream weights) while the kernel that produced x finishes.
    return run_single(W, layout, x, y, nullptr, N, K, T, ws, static_cast<size_t>(need),
                      reinterpret_cast<cudaStream_t>(stream), false, true, true);
}

// Argument checks of the argmax calls, host only (no CUDA call).  ws ==
// nullptr: the library's own scratch, which no caller buffer can overlap.
static qgemv_status argmax_check(const void *W, qgemv_wlayout layout, const void *xin, bool xf32,
                                 const float *y_or_null, const int64_t *idx, int64_t N, int64_t K, int T,
                                 const void *ws, size_t ws_bytes)
{
    const long long xin_bytes = !shape_ok(N, K) ? 0 : xf32 ? 4ll * T * K : xq_bytes_host(T, K);
    qgemv_status s = check_single(W, layout, xin, xin_bytes, y_or_null, N, K, T, ws);
    if (s != QGEMV_OK) return s;
    if (!idx) return QGEMV_ERR_INVALID_ARG;
    if (!aligned(xin, xf32 ? 4 : 16) || !aligned(idx, 8)) return QGEMV_ERR_MISALIGNED;
    if (y_or_null && overlap(range(idx, 8ll * T), range(y_or_null, 4ll * T * N))) return QGEMV_ERR_INVALID_ARG;
    if (xf32 && overlap(range(xin, xin_bytes), range(idx, 8ll * T))) return QGEMV_ERR_INVALID_ARG;
    if (!ws) return QGEMV_OK;
    const Range rw = range(ws, static_cast<long long>(ws_bytes));
    if (overlap(range(idx, 8ll * T), rw) || (y_or_null && overlap(range(y_or_null, 4ll * T * N), rw)))
        return QGEMV_ERR_INVALID_ARG;
    if (xf32 && overlap(range(xin, xin_bytes), rw)) return QGEMV_ERR_INVALID_ARG;
    return QGEMV_OK;
}

// The argmax calls: quantised (xq) or fp32 (x, xf32) activations.
static qgemv_status argmax_call(const void *W, qgemv_wlayout layout, const void *xin, bool xf32, float *y_or_null,
                                int64_t *idx, int64_t N, int64_t K, int T, void *ws, size_t ws_bytes,
                                qgemv_stream_t stream)
{
    const qgemv_status s = argmax_check(W, layout, xin, xf32, y_or_null, idx, N, K, T, ws, ws_bytes);
    if (s != QGEMV_OK) return s;
    if (!ws) return QGEMV_ERR_WORKSPACE;
    return run_single(W, layout, xin, y_or_null, reinterpret_cast<long long *>(idx), N, K, T, ws, ws_bytes,
                      reinterpret_cast<cudaStream_t>(stream), true, true, xf32);
}

qgemv_status qgemv_q4_0_argmax(const void *W, qgemv_wlayout layout, const void *xq, float *y_or_null, int64_t *idx,
                               int64_t N, int64_t K, int T, void *ws, size_t ws_bytes, qgemv_stream_t stream)
{
    return argmax_call(W, layout, xq, false, y_or_null, idx, N, K, T, ws, ws_bytes, stream);
}

qgemv_status qgemv_q4_0_argmax_f32(const void *W, qgemv_wlayout layout, const float *x, float *y_or_null,
                                   int64_t *idx, int64_t N, int64_t K, int T, void *ws, size_t ws_bytes,
                                   qgemv_stream_t stream)
{
    return argmax_call(W, layout, x, true, y_or_null, idx, N, K, T, ws, ws_bytes, stream);
}

// The top-2 calls: the argmax calls' checks, with the [T][2] row and value
// outputs in place of idx.
static qgemv_status top2_call(const void *W, qgemv_wlayout layout, const void *xin, bool xf32, float *y_or_null,
                              int64_t *idx2, float *val2, int64_t N, int64_t K, int T, void *ws, size_t ws_bytes,
                              qgemv_stream_t stream, const int64_t *tokens = nullptr, int32_t *n_commit = nullptr)
{
    const long long xin_bytes = !shape_ok(N, K) ? 0 : xf32 ? 4ll * T * K : xq_bytes_host(T, K);
    qgemv_status s = check_single(W, layout, xin, xin_bytes, y_or_null, N, K, T, ws);
    if (s != QGEMV_OK) return s;
    if (!idx2 || !val2) return QGEMV_ERR_INVALID_ARG;
    if (!aligned(xin, xf32 ? 4 : 16) || !aligned(idx2, 8) || !aligned(val2, 4)) return QGEMV_ERR_MISALIGNED;
    if (!ws) return QGEMV_ERR_WORKSPACE;
    const Range rw = range(ws, static_cast<long long>(ws_bytes));
    const Range ri = range(idx2, 16ll * T), rv = range(val2, 8ll * T);
    if (overlap(ri, rw) || overlap(rv, rw) || overlap(ri, rv)) return QGEMV_ERR_INVALID_ARG;
    if (y_or_null) {
        const Range ry = range(y_or_null, 4ll * T * N);
        if (overlap(ry, rw) || overlap(ry, ri) || overlap(ry, rv)) return QGEMV_ERR_INVALID_ARG;
    }
    if (xf32) {
        const Range rx = range(xin, xin_bytes);
        if (overlap(rx, rw) || overlap(rx, ri) || overlap(rx, rv)) return QGEMV_ERR_INVALID_ARG;
    }
    if (tokens || n_commit) {
        if (!tokens || !n_commit) return QGEMV_ERR_INVALID_ARG;
        if (!aligned(tokens, 8) || !aligned(n_commit, 4)) return QGEMV_ERR_MISALIGNED;
        const Range rn = range(n_commit, 4);
        if (overlap(rn, rw) || overlap(rn, ri) || overlap(rn, rv) || overlap(rn, range(tokens, 8ll * T)) ||
            (y_or_null && overlap(rn, range(y_or_null, 4ll * T * N))))
            return QGEMV_ERR_INVALID_ARG;
    }
    return run_single(W, layout, xin, y_or_null, nullptr, N, K, T, ws, ws_bytes,
                      reinterpret_cast<cudaStream_t>(stream), true, true, xf32, reinterpret_cast<long long *>(idx2),
                      val2, reinterpret_cast<const long long *>(tokens), n_commit);
}

qgemv_status qgemv_q4_0_top2(const void *W, qgemv_wlayout layout, const void *xq, float *y_or_null, int64_t *idx2,
                             float *val2, int64_t N, int64_t K, int T, void *ws, size_t ws_bytes,
                             qgemv_stream_t stream)
{
    return top2_call(W, layout, xq, false, y_or_null, idx2, val2, N, K, T, ws, ws_bytes, stream);
}

qgemv_status qgemv_q4_0_top2_f32(const void *W, qgemv_wlayout layout, const float *x, float *y_or_null,
                                 int64_t *idx2, float *val2, int64_t N, int64_t K, int T, void *ws, size_t ws_bytes,
                                 qgemv_stream_t stream)
{
    return top2_call(W, layout, x, true, y_or_null, idx2, val2, N, K, T, ws, ws_bytes, stream);
}

// ------------------------------------------------------------ Q8_0 weights

qgemv_status qgemv_pack_q8_0(const void *w_ggml, void *w_packed, int64_t N, int64_t K, qgemv_stream_t stream)
{
    if (!shape_ok(N, K) || !w_ggml || !w_packed) return QGEMV_ERR_INVALID_ARG;
    if (!aligned(w_packed, 16)) return QGEMV_ERR_MISALIGNED;
    if (overlap(range(w_ggml, 34ll * N * (K / QK)), range(w_packed, 34ll * N * (K / QK)))) return QGEMV_ERR_INVALID_ARG;
    return launch_q8_pack(w_ggml, w_packed, N, K, true, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? QGEMV_OK
               : QGEMV_ERR_CUDA;
}

qgemv_status qgemv_requant_f32_q4_0(const float *w, void *w_q4, int64_t N, int64_t K, qgemv_stream_t stream)
{
    if (!shape_ok(N, K) || !w || !w_q4) return QGEMV_ERR_INVALID_ARG;
    if (!aligned(w, 4) || !aligned(w_q4, 2)) return QGEMV_ERR_MISALIGNED;
    if (overlap(range(w, 4ll * N * K), range(w_q4, 18ll * N * (K / QK)))) return QGEMV_ERR_INVALID_ARG;
    return launch_requant_q4_0(w, false, w_q4, N * (K / QK), reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? QGEMV_OK
               : QGEMV_ERR_CUDA;
}

qgemv_status qgemv_requant_q8_0_q4_0(const void *w_q8, void *w_q4, int64_t N, int64_t K, qgemv_stream_t stream)
{
    if (!shape_ok(N, K) || !w_q8 || !w_q4) return QGEMV_ERR_INVALID_ARG;
    if (!aligned(w_q8, 2) || !aligned(w_q4, 2)) return QGEMV_ERR_MISALIGNED;
    if (overlap(range(w_q8, 34ll * N * (K / QK)), range(w_q4, 18ll * N * (K / QK)))) return QGEMV_ERR_INVALID_ARG;
    return launch_requant_q4_0(w_q8, true, w_q4, N * (K / QK), reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? QGEMV_OK
               : QGEMV_ERR_CUDA;
}

qgemv_status qgemv_unpack_q8_0(const void *w_packed, void *w_ggml, int64_t N, int64_t K, qgemv_stream_t stream)
{
    if (!shape_ok(N, K) || !w_ggml || !w_packed) return QGEMV_ERR_INVALID_ARG;
    if (!aligned(w_packed, 16)) return QGEMV_ERR_MISALIGNED;
    if (overlap(range(w_ggml, 34ll * N * (K / QK)), range(w_packed, 34ll * N * (K / QK)))) return QGEMV_ERR_INVALID_ARG;
    return launch_q8_pack(w_packed, w_ggml, N, K, false, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? QGEMV_OK
               : QGEMV_ERR_CUDA;
}

size_t qgemv_q8_0_workspace_bytes(int64_t N, int64_t K, int T)
{
    if (!shape_ok(N, K) || T < 1 || T > 8) return 0;
    DevInfo dev;
    int sms = 152, budget = 230400;
    if (device_info(dev) == QGEMV_OK) {
        sms = dev.sms;
        budget = dev.smem_optin - 2048;
    }
    long long need = 0;
    int uns = 0;
    launch_q8(nullptr, nullptr, nullptr, N, K, T, nullptr, 0, false, sms, budget, nullptr, nullptr, &need, &uns);
    return static_cast<size_t>(need);
}

qgemv_status qgemv_q8_0(const void *W, const void *xq, float *y, int64_t N, int64_t K, int T, void *ws,
                        size_t ws_bytes, qgemv_stream_t stream)
{
    if (!shape_ok(N, K) || T < 1 || T > 8 || !W || !xq || !y) return QGEMV_ERR_INVALID_ARG;
    if (!aligned(W, 16) || !aligned(xq, 16) || !aligned(y, 4) || (ws && !aligned(ws, 256))) return QGEMV_ERR_MISALIGNED;
    const Range ry = range(y, 4ll * T * N);
    if (overlap(ry, range(W, 34ll * N * (K / QK))) || overlap(ry, range(xq, xq_bytes_host(T, K))) ||
        (ws && overlap(ry, range(ws, static_cast<long long>(ws_bytes)))))
        return QGEMV_ERR_INVALID_ARG;
    DevInfo dev;
    qgemv_status s = device_info(dev);
    if (s != QGEMV_OK) return s;
    long long need = 0;
    int uns = 0;
    const cudaError_t e = launch_q8(W, xq, y, N, K, T, ws, static_cast<long long>(ws_bytes), true, dev.sms,
                                    dev.smem_optin - 2048, dev.status, reinterpret_cast<cudaStream_t>(stream), &need,
                                    &uns);
    if (uns) return uns == 1 ? QGEMV_ERR_UNSUPPORTED : QGEMV_ERR_WORKSPACE;
    return e == cudaSuccess ? QGEMV_OK : QGEMV_ERR_CUDA;
}

// ------------------------------------------------------------ gs64 int4 groups

static bool gs64_shape_ok(long long N, long long K) { return shape_ok(N, K) && K % 64 == 0; }

size_t qgemv_gs64_bytes(int64_t N, int64_t K)
{
    return gs64_shape_ok(N, K) ? static_cast<size_t>(36ll * N * (K / 64)) : 0;
}

qgemv_status qgemv_pack_gs64(const void *wq, const float *wscale, void *w_packed, int64_t N, int64_t K,
                             qgemv_stream_t stream)
{
    if (!gs64_shape_ok(N, K) || !wq || !wscale || !w_packed) return QGEMV_ERR_INVALID_ARG;
    if (!aligned(wscale, 4) || !aligned(w_packed, 16)) return QGEMV_ERR_MISALIGNED;
    const Range rp = range(w_packed, 36ll * N * (K / 64));
    if (overlap(rp, range(wq, 32ll * N * (K / 64))) || overlap(rp, range(wscale, 4ll * N * (K / 64))))
        return QGEMV_ERR_INVALID_ARG;
    return launch_gs64_pack(const_cast<void *>(wq), const_cast<float *>(wscale), w_packed, N, K, true,
                            reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? QGEMV_OK
               : QGEMV_ERR_CUDA;
}

qgemv_status qgemv_unpack_gs64(const void *w_packed, void *wq, float *wscale, int64_t N, int64_t K,
                               qgemv_stream_t stream)
{
    if (!gs64_shape_ok(N, K) || !wq || !wscale || !w_packed) return QGEMV_ERR_INVALID_ARG;
    if (!aligned(wscale, 4) || !aligned(w_packed, 16)) return QGEMV_ERR_MISALIGNED;
    const Range rp = range(w_packed, 36ll * N * (K / 64)), rq = range(wq, 32ll * N * (K / 64)),
                rs = range(wscale, 4ll * N * (K / 64));
    if (overlap(rp, rq) || overlap(rp, rs) || overlap(rq, rs)) return QGEMV_ERR_INVALID_ARG;
    return launch_gs64_pack(wq, wscale, const_cast<void *>(w_packed), N, K, false,
                            reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? QGEMV_OK
               : QGEMV_ERR_CUDA;
}

qgemv_status qgemv_quantize_vec_i8(const float *x, int8_t *q, float *s, int R, int64_t K, qgemv_stream_t stream)
{
    if (R < 1 || R > 65535 || K < 1 || K > (1ll << 24) || !x || !q || !s) return QGEMV_ERR_INVALID_ARG;
    if (!aligned(x, 4) || !aligned(s, 4)) return QGEMV_ERR_MISALIGNED;
    const Range rx = range(x, 4ll * R * K), rq = range(q, 1ll * R * K), rs = range(s, 4ll * R);
    if (overlap(rx, rq) || overlap(rx, rs) || overlap(rq, rs)) return QGEMV_ERR_INVALID_ARG;
    return launch_quantize_vec_i8(x, q, s, R, K, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? QGEMV_OK
               : QGEMV_ERR_CUDA;
}

size_t qgemv_gs64_workspace_bytes(int64_t N, int64_t K, int T)
{
    if (!gs64_shape_ok(N, K) || T < 1 || T > 8) return 0;
    DevInfo dev;
    int sms = 152, budget = 230400;
    if (device_info(dev) == QGEMV_OK) {
        sms = dev.sms;
        budget = dev.smem_optin - 2048;
    }
    long long need = 0;
    int uns = 0;
    launch_gs64(nullptr, nullptr, nullptr, nullptr, nullptr, N, K, T, nullptr, 0, false, sms, budget, nullptr, nullptr,
                &need, &uns);
    return static_cast<size_t>(need);
}

qgemv_status qgemv_gs64(const void *W, const int8_t *q, const float *s, float *y, int64_t N, int64_t K, int T,
                        void *ws, size_t ws_bytes, qgemv_stream_t stream)
{
    if (!gs64_shape_ok(N, K) || T < 1 || T > 8 || !W || !q || !s || !y) return QGEMV_ERR_INVALID_ARG;
    if (!aligned(W, 16) || !aligned(q, 16) || !aligned(s, 4) || !aligned(y, 4) || (ws && !aligned(ws, 256)))
        return QGEMV_ERR_MISALIGNED;
    const Range ry = range(y, 4ll * T * N);
    if (overlap(ry, range(W, 36ll * N * (K / 64))) || overlap(ry, range(q, 1ll * T * K)) ||
        overlap(ry, range(s, 4ll * T)) || (ws && overlap(ry, range(ws, static_cast<long long>(ws_bytes)))))
        return QGEMV_ERR_INVALID_ARG;
    DevInfo dev;
    qgemv_status st = device_info(dev);
    if (st != QGEMV_OK) return st;
    long long need = 0;
    int uns = 0;
    const cudaError_t e = launch_gs64(W, q, s, nullptr, y, N, K, T, ws, static_cast<long long>(ws_bytes), true,
                                      dev.sms, dev.smem_optin - 2048, dev.status,
                                      reinterpret_cast<cudaStream_t>(stream), &need, &uns);
    if (uns) return uns == 1 ? QGEMV_ERR_UNSUPPORTED : QGEMV_ERR_WORKSPACE;
    return e == cudaSuccess ? QGEMV_OK : QGEMV_ERR_CUDA;
}

qgemv_status qgemv_gs64_f32(const void *W, const float *x, float *y, int64_t N, int64_t K, int T, void *ws,
                            size_t ws_bytes, qgemv_stream_t stream)
{
    if (!gs64_shape_ok(N, K) || T < 1 || T > 8 || !W || !x || !y) return QGEMV_ERR_INVALID_ARG;
    if (!aligned(W, 16) || !aligned(x, 4) || !aligned(y, 4) || (ws && !aligned(ws, 256))) return QGEMV_ERR_MISALIGNED;
    const Range ry = range(y, 4ll * T * N);
    if (overlap(ry, range(W, 36ll * N * (K / 64))) || overlap(ry, range(x, 4ll * T * K)) ||
        (ws && overlap(ry, range(ws, static_cast<long long>(ws_bytes)))))
        return QGEMV_ERR_INVALID_ARG;
    DevInfo dev;
    qgemv_status st = device_info(dev);
    if (st != QGEMV_OK) return st;
    long long need = 0;
    int uns = 0;
    const cudaError_t e = launch_gs64(W, nullptr, nullptr, x, y, N, K, T, ws, static_cast<long long>(ws_bytes), true,
                                      dev.sms, dev.smem_optin - 2048, dev.status,
                                      reinterpret_cast<cudaStream_t>(stream), &need, &uns);
    if (uns) return uns == 1 ? QGEMV_ERR_UNSUPPORTED : QGEMV_ERR_WORKSPACE;
    return e == cudaSuccess ? QGEMV_OK : QGEMV_ERR_CUDA;
}

// ------------------------------------------------------------ FFN step

// Workspace of qgemv_q4_0_ffn: [gate/up sequence][g][u][h codes][down call],
// each part 256-byte aligned; off[0..4] the parts' offsets.  0: bad shape.
static long long ffn_parts(int64_t d_model, int64_t d_ff, int T, long long off[5])
{
    if (!shape_ok(d_ff, d_model) || !shape_ok(d_model, d_ff) || T < 1 || T > 8) return 0;
    const qgemv_seq_item it[2] = {{nullptr, nullptr, nullptr, d_ff, d_model}, {nullptr, nullptr, nullptr, d_ff, d_model}};
    off[0] = 0;
    off[1] = align_up(static_cast<long long>(qgemv_seq_workspace_bytes(it, 2, T)), 256);
    off[2] = off[1] + align_up(4ll * T * d_ff, 256);
    off[3] = off[2] + align_up(4ll * T * d_ff, 256);
    off[4] = off[3] + align_up(xq_bytes_host(T, d_ff), 256);
    // down: a single call, or a one-item sequence with the residual epilogue
    const qgemv_seq_item dn[1] = {{nullptr, nullptr, nullptr, d_model, d_ff}};
    const long long d1 = static_cast<long long>(qgemv_workspace_bytes(d_model, d_ff, T));
    const long long d2 = static_cast<long long>(qgemv_seq_workspace_bytes(dn, 1, T));
    return off[4] + align_up(d1 > d2 ? d1 : d2, 256);
}

size_t qgemv_ffn_workspace_bytes(int64_t d_model, int64_t d_ff, int T)
{
    long long off[5];
    return static_cast<size_t>(ffn_parts(d_model, d_ff, T, off));
}

qgemv_status qgemv_debug_silu_mul_q8(const float *g, const float *u, void *hq, int T, int64_t F, qgemv_stream_t stream)
{
    if (T < 1 || T > 8 || !shape_ok(1, F) || !g || !u || !hq) return QGEMV_ERR_INVALID_ARG;
    if (!aligned(g, 4) || !aligned(u, 4) || !aligned(hq, 16)) return QGEMV_ERR_MISALIGNED;
    const Range rh = range(hq, xq_bytes_host(T, F));
    if (overlap(rh, range(g, 4ll * T * F)) || overlap(rh, range(u, 4ll * T * F))) return QGEMV_ERR_INVALID_ARG;
    return launch_silu_mul_q8(g, u, hq, T, F, false, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? QGEMV_OK
               : QGEMV_ERR_CUDA;
}

static qgemv_status ffn_chain(const void *W_gate, const void *W_up, const void *W_down, qgemv_wlayout layout,
                              const float *x, const float *residual, float *y, int64_t d_model, int64_t d_ff, int T,
                              void *ws, size_t ws_bytes, qgemv_stream_t stream);
static qgemv_status launch_seq(const qgemv_seq_item *items, int n, qgemv_wlayout layout, int T, void *ws,
                               size_t ws_bytes, cudaStream_t st, bool xf32, const float *const *bias,
                               const float *const *res);

qgemv_status qgemv_q4_0_ffn(const void *W_gate, const void *W_up, const void *W_down, qgemv_wlayout layout,
                            const float *x, float *y, int64_t d_model, int64_t d_ff, int T, void *ws,
                            size_t ws_bytes, qgemv_stream_t stream)
{
    return ffn_chain(W_gate, W_up, W_down, layout, x, nullptr, y, d_model, d_ff, T, ws, ws_bytes, stream);
}

qgemv_status qgemv_q4_0_ffn_residual(const void *W_gate, const void *W_up, const void *W_down, qgemv_wlayout layout,
                                     const float *x, const float *residual, float *y, int64_t d_model, int64_t d_ff,
                                     int T, void *ws, size_t ws_bytes, qgemv_stream_t stream)
{
    if (!residual) return QGEMV_ERR_INVALID_ARG;
    return ffn_chain(W_gate, W_up, W_down, layout, x, residual, y, d_model, d_ff, T, ws, ws_bytes, stream);
}

static qgemv_status ffn_chain(const void *W_gate, const void *W_up, const void *W_down, qgemv_wlayout layout,
                              const float *x, const float *residual, float *y, int64_t d_model, int64_t d_ff, int T,
                              void *ws, size_t ws_bytes, qgemv_stream_t stream)
{
    long long off[5];
    const long long need = ffn_parts(d_model, d_ff, T, off);
    if (need == 0 || !W_gate || !W_up || !W_down || !x || !y) return QGEMV_ERR_INVALID_ARG;
    if (layout != QGEMV_W_GGML && layout != QGEMV_W_PACKED) return QGEMV_ERR_INVALID_ARG;
    if (!aligned(x, 4) || !aligned(y, 4)) return QGEMV_ERR_MISALIGNED;
    if (!ws) return QGEMV_ERR_WORKSPACE;
    if (!aligned(ws, 256)) return QGEMV_ERR_MISALIGNED;
    if (static_cast<long long>(ws_bytes) < need) return QGEMV_ERR_WORKSPACE;
    const Range ry = range(y, 4ll * T * d_model), rw = range(ws, need);
    if (overlap(ry, rw) || overlap(ry, range(x, 4ll * T * d_model)) || overlap(range(x, 4ll * T * d_model), rw) ||
        overlap(ry, range(W_down, 18ll * d_model * (d_ff / QK))))
        return QGEMV_ERR_INVALID_ARG;
    if (residual) {  // may be y itself; otherwise it overlaps nothing the chain writes
        if (!aligned(residual, 4)) return QGEMV_ERR_MISALIGNED;
        const Range rr = range(residual, 4ll * T * d_model);
        if (residual != y && (overlap(rr, ry) || overlap(rr, rw))) return QGEMV_ERR_INVALID_ARG;
    }
    uint8_t *w = static_cast<uint8_t *>(ws);
    // one fused launch: h's codes where the chain keeps them, counters in
    // the workspace's zeroed counter area
    if (layout == QGEMV_W_PACKED && g_ffn_fused.load(std::memory_order_relaxed)) {
        DevInfo dev;
        qgemv_status ds = device_info(dev);
        if (ds != QGEMV_OK) return ds;
        if (ffn_fused_fits(d_model, d_ff, T, dev.sms, dev.smem_optin - 2048)) {
            const cudaError_t e =
                launch_ffn_fused(W_gate, W_up, W_down, x, residual, y, d_model, d_ff, T, w + off[3],
                                 reinterpret_cast<unsigned *>(w), dev.sms, dev.smem_optin - 2048, dev.status,
                                 reinterpret_cast<cudaStream_t>(stream));
            return e == cudaSuccess ? QGEMV_OK : QGEMV_ERR_CUDA;
        }
    }
    float *g = reinterpret_cast<float *>(w + off[1]);
    float *u = reinterpret_cast<float *>(w + off[2]);
    void *hq = w + off[3];
    // gate and up: one sequence launch over the same fp32 x (quantised in the kernel)
    const qgemv_seq_f32_item gu[2] = {{W_gate, x, g, d_ff, d_model}, {W_up, x, u, d_ff, d_model}};
    qgemv_status s = qgemv_q4_0_seq_f32(gu, 2, layout, T, w + off[0], static_cast<size_t>(off[1]), stream);
    if (s != QGEMV_OK) return s;
    if (launch_silu_mul_q8(g, u, hq, T, d_ff, true, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return QGEMV_ERR_CUDA;
    if (!residual)
        return qgemv_q4_0(W_down, layout, hq, y, d_model, d_ff, T, w + off[4], static_cast<size_t>(need - off[4]),
                          stream);
    // down with the residual epilogue: a one-item sequence launch
    const qgemv_seq_item dn[1] = {{W_down, hq, y, d_model, d_ff}};
    const float *const bias[1] = {nullptr};
    const float *const res[1] = {residual};
    return launch_seq(dn, 1, layout, T, w + off[4], static_cast<size_t>(need - off[4]),
                      reinterpret_cast<cudaStream_t>(stream), false, bias, res);
}

qgemv_status qgemv_q4_0_verify_f32(const void *W, qgemv_wlayout layout, const float *x, const int64_t *tokens,
                                  int64_t *idx2, float *val2, int32_t *n_commit, int64_t N, int64_t K, int T,
                                  void *ws, size_t ws_bytes, qgemv_stream_t stream)
{
    return top2_call(W, layout, x, true, nullptr, idx2, val2, N, K, T, ws, ws_bytes, stream, tokens, n_commit);
}

qgemv_status qgemv_verify_commit(const int64_t *tokens, const int64_t *pred, int pred_stride, int T,
                                 int32_t *n_commit, qgemv_stream_t stream)
{
    if (T < 1 || T > 32 || pred_stride < 1 || !tokens || !pred || !n_commit) return QGEMV_ERR_INVALID_ARG;
    if (!aligned(tokens, 8) || !aligned(pred, 8) || !aligned(n_commit, 4)) return QGEMV_ERR_MISALIGNED;
    return launch_verify_commit(reinterpret_cast<const long long *>(tokens), reinterpret_cast<const long long *>(pred),
                                pred_stride, T, n_commit, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? QGEMV_OK
               : QGEMV_ERR_CUDA;
}

// Small groups of a tensor-core sequence launch (a CTA's share of one
// matrix, fewer whole slabs than warps, alone in shared memory) are spread
// over all warps when the workspace holds a region of segment sums for the
// CTA: up to
// NWARPS_MAX - 1 slabs of the launch's longest rows.  Without it they run one
// slab per warp; the results are the same bits either way.
inline long long sg_stride_floats(const GroupSpec *gs, int n, int T)
{
    long long nseg_max = 1;
    for (int i = 0; i < n; ++i) nseg_max = std::max(nseg_max, (gs[i].K / QK + SEG_BLOCKS - 1) / SEG_BLOCKS);
    return (NWARPS_MAX - 1) * nseg_max * T * 16;
}

// CTAs of a sequence launch given a small-group region by the workspace size
// below: the grid on this device, else one CTA on each of 152 SMs.
inline long long sg_ctas_hint(int T)
{
    DevInfo dev;
    if (device_info(dev) != QGEMV_OK) return 152;
    return grid_for(dev, ctas_per_sm_for(T, true));
}

// The tcgen05 path of one launch's items (c0, cn): eligible or not, and its
// workspace (with the quantised activations' area for fp32 inputs).
static bool tc_chunk(const qgemv_seq_item *items, int c0, int cn, int T, qgemv_wlayout layout, std::vector<TcSpec> &sp)
{
    if (layout != QGEMV_W_PACKED || !tc_for(T)) return false;
    sp.resize(cn);
    for (int i = 0; i < cn; ++i) {
        const qgemv_seq_item &it = items[c0 + i];
        sp[i] = TcSpec{it.W, it.xq, it.y, it.N, it.K};
    }
    return tc_eligible(sp.data(), cn, T);
}

static long long tc_grid()
{
    DevInfo dev;
    return device_info(dev) == QGEMV_OK ? dev.sms : 152;
}

static long long tc_chunk_ws(const std::vector<TcSpec> &sp, int T, bool xf32)
{
    long long b = align_up(tc_ws_bytes(sp.data(), static_cast<int>(sp.size()), static_cast<int>(tc_grid())), 256);
    if (xf32)
        for (const TcSpec &s : sp) b += align_up(xq_bytes_host(T, s.K), 256);
    return b;
}

static size_t seq_ws(const qgemv_seq_item *items, int n, int T, bool xf32);

size_t qgemv_seq_workspace_bytes(const qgemv_seq_item *items, int n, int T) { return seq_ws(items, n, T, false); }

static size_t seq_ws(const qgemv_seq_item *items, int n, int T, bool xf32)
{
    if (!items || n < 1 || T < 1 || T > 8) return 0;
    long long total = 0;
    for (int c0 = 0; c0 < n; c0 += MAXG_SEQ) {
        const int cn = (n - c0) < MAXG_SEQ ? (n - c0) : MAXG_SEQ;
        std::vector<GroupSpec> gs(cn);
        for (int i = 0; i < cn; ++i) {
            const qgemv_seq_item &it = items[c0 + i];
            if (!shape_ok(it.N, it.K)) return 0;
            gs[i] = GroupSpec{it.W, 0, it.xq, 0, it.y, 0, it.N, it.K, 1};
        }
        std::unique_ptr<Plan<MAXG_SEQ>> pa(new Plan<MAXG_SEQ>()), pb(new Plan<MAXG_SEQ>());
        make_plan<MAXG_SEQ>(gs.data(), cn, T, false, false, nullptr, 0, *pa);
        make_plan<MAXG_SEQ>(gs.data(), cn, T, true, false, nullptr, 0, *pb);
        long long b = pa->ws_bytes > pb->ws_bytes ? pa->ws_bytes : pb->ws_bytes;
        if (pa->P.balanced_ok && mma_for(T)) b = align_up(b, 256) + sg_ctas_hint(T) * sg_stride_floats(gs.data(), cn, T) * 4;
        std::vector<TcSpec> sp;
        if (tc_chunk(items, c0, cn, T, QGEMV_W_PACKED, sp)) b = std::max(b, tc_chunk_ws(sp, T, xf32));
        if (b > total) total = b;  // consecutive launches reuse the workspace
    }
    return static_cast<size_t>(total);
}

static qgemv_status check_seq(const qgemv_seq_item *items, int n, qgemv_wlayout layout, int T, void *ws,
                              size_t ws_bytes, bool xf32 = false, const float *const *bias = nullptr,
                              const float *const *res = nullptr)
{
    if (!items || n < 1 || T < 1 || T > 8) return QGEMV_ERR_INVALID_ARG;
    if (layout != QGEMV_W_GGML && layout != QGEMV_W_PACKED) return QGEMV_ERR_INVALID_ARG;
    if (!ws) return QGEMV_ERR_WORKSPACE;
    if (!aligned(ws, 256)) return QGEMV_ERR_MISALIGNED;
    // Every output range must overlap no other range (weights and activations
    // may be shared between items): sort all ranges, sweep once.
    struct Tagged {
        Range r;
        bool out;
    };
    std::vector<Tagged> v;
    v.reserve(3 * static_cast<size_t>(n) + 1);
    v.push_back(Tagged{range(ws, static_cast<long long>(ws_bytes)), false});
    for (int i = 0; i < n; ++i) {
        const qgemv_seq_item &a = items[i];
        if (!shape_ok(a.N, a.K) || !a.W || !a.xq || !a.y) return QGEMV_ERR_INVALID_ARG;
        if (!aligned(a.W, layout == QGEMV_W_PACKED ? 16 : 2) || !aligned(a.xq, xf32 ? 4 : 16) || !aligned(a.y, 4))
            return QGEMV_ERR_MISALIGNED;
        v.push_back(Tagged{range(a.W, 18ll * a.N * (a.K / QK)), false});
        v.push_back(Tagged{range(a.xq, xf32 ? 4ll * T * a.K : xq_bytes_host(T, a.K)), false});
        v.push_back(Tagged{range(a.y, 4ll * T * a.N), true});
        // epilogue inputs: a residual equal to y is read in place (same element, same thread)
        if (bias && bias[i]) {
            if (!aligned(bias[i], 4)) return QGEMV_ERR_MISALIGNED;
            v.push_back(Tagged{range(bias[i], 4ll * a.N), false});
        }
        if (res && res[i] && res[i] != a.y) {
            if (!aligned(res[i], 4)) return QGEMV_ERR_MISALIGNED;
            v.push_back(Tagged{range(res[i], 4ll * T * a.N), false});
        }
    }
    std::sort(v.begin(), v.end(), [](const Tagged &x, const Tagged &y) { return x.r.lo < y.r.lo; });
    uintptr_t hi_any = 0, hi_out = 0;
    for (const Tagged &t : v) {
        if (t.r.lo < (t.out ? hi_any : hi_out)) return QGEMV_ERR_INVALID_ARG;
        if (t.r.hi > hi_any) hi_any = t.r.hi;
        if (t.out && t.r.hi > hi_out) hi_out = t.r.hi;
    }
    return QGEMV_OK;
}

// The launches of a sequence (checked): one persistent GEMV launch per
// MAXG_SEQ items.  xf32: the items' activations are fp32 x[T][K], quantised
// inside the GEMV kernel.
static qgemv_status launch_seq(const qgemv_seq_item *items, int n, qgemv_wlayout layout, int T, void *ws,
                               size_t ws_bytes, cudaStream_t st, bool xf32, const float *const *bias = nullptr,
                               const float *const *res = nullptr)
{
    DevInfo dev;
    qgemv_status s = device_info(dev);
    if (s != QGEMV_OK) return s;
    std::vector<GroupSpec> gs(MAXG_SEQ);
    std::unique_ptr<Plan<MAXG_SEQ>> pl(new Plan<MAXG_SEQ>());
    for (int c0 = 0; c0 < n; c0 += MAXG_SEQ) {
        const int cn = (n - c0) < MAXG_SEQ ? (n - c0) : MAXG_SEQ;
        // the tcgen05 kernel (plain packed sequences whose workspace holds its
        // sums; fp32 inputs are quantised first, into the workspace, in one launch)
        std::vector<TcSpec> sp;
        if (!bias && !res && tc_chunk(items, c0, cn, T, layout, sp) &&
            static_cast<long long>(ws_bytes) >= tc_chunk_ws(sp, T, xf32)) {
            uint8_t *w = static_cast<uint8_t *>(ws);
            if (xf32) {
                long long off = align_up(tc_ws_bytes(sp.data(), cn, dev.sms), 256);
                std::vector<const float *> xs(cn);
                std::vector<uint8_t *> xqs(cn);
                std::vector<long long> ks(cn);
                for (int i = 0; i < cn; ++i) {
                    xs[i] = static_cast<const float *>(sp[i].xq);
                    xqs[i] = w + off;
                    ks[i] = sp[i].K;
                    sp[i].xq = w + off;
                    off += align_up(xq_bytes_host(T, sp[i].K), 256);
                }
                if (launch_quantize_list(xs.data(), xqs.data(), ks.data(), cn, T, 2 * dev.sms, st) != cudaSuccess)
                    return QGEMV_ERR_CUDA;
            }
            if (launch_tc(sp.data(), cn, T, w, dev.sms, dev.status, st) != cudaSuccess) return QGEMV_ERR_CUDA;
            continue;
        }
        for (int i = 0; i < cn; ++i) {
            const qgemv_seq_item &it = items[c0 + i];
            gs[i] = GroupSpec{it.W, 0, it.xq, 0, it.y, 0, it.N, it.K, 1};
            gs[i].bias = bias ? bias[c0 + i] : nullptr;
            gs[i].res = res ? res[c0 + i] : nullptr;
        }
        int cps = ctas_per_sm_for(T, true);
        s = plan_launch<MAXG_SEQ>(gs.data(), cn, T, layout == QGEMV_W_GGML, false, static_cast<uint8_t *>(ws), dev,
                                  cps, *pl);
        const int grid = grid_for(dev, cps);
        if (s != QGEMV_OK) return s;
        if (static_cast<long long>(ws_bytes) < pl->ws_bytes) return QGEMV_ERR_WORKSPACE;
        pl->P.status = dev.status;
        pl->P.xf32 = xf32 ? 1 : 0;
        if (pl->P.balanced_ok && layout != QGEMV_W_GGML && mma_for(T)) {
            const long long off = align_up(pl->ws_bytes, 256), stride = sg_stride_floats(gs.data(), cn, T);
            const long long room = static_cast<long long>(ws_bytes) - off;
            const long long nc = room > 0 ? std::min<long long>(grid, room / (stride * 4)) : 0;
            if (nc > 0 && stride <= INT32_MAX) {
                pl->P.sg_part = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + off);
                pl->P.sg_stride = static_cast<int>(stride);
                pl->P.sg_ctas = static_cast<int>(nc);
            }
        }
        set_cta_groups(pl->P, grid);
        if (pl->P.epilogue) {
            const cudaError_t e = dispatch_ep(pl->P, T, mma_for(T), grid, pl->smem, st);
            if (e == cudaErrorNotSupported) return QGEMV_ERR_UNSUPPORTED;
            if (e != cudaSuccess) return QGEMV_ERR_CUDA;
        } else if (dispatch_T<MAXG_SEQ, false>(pl->P, T, mma_for(T), grid, pl->smem, st, true) != cudaSuccess) {
            return QGEMV_ERR_CUDA;
        }
    }
    return QGEMV_OK;
}

qgemv_status qgemv_q4_0_seq(const qgemv_seq_item *items, int n, qgemv_wlayout layout, int T, void *ws,
                            size_t ws_bytes, qgemv_stream_t stream)
{
    const qgemv_status s = check_seq(items, n, layout, T, ws, ws_bytes);
    if (s != QGEMV_OK) return s;
    return launch_seq(items, n, layout, T, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream), false);
}

// The fp32-input sequence as a sequence whose activation pointers are the
// fp32 inputs (the kernel quantises them; no workspace for activations).
static bool seq_f32_items(const qgemv_seq_f32_item *items, int n, std::vector<qgemv_seq_item> &sq)
{
    sq.resize(n);
    for (int i = 0; i < n; ++i) {
        if (!shape_ok(items[i].N, items[i].K)) return false;
        sq[i] = qgemv_seq_item{items[i].W, items[i].x, items[i].y, items[i].N, items[i].K};
    }
    return true;
}

size_t qgemv_seq_f32_workspace_bytes(const qgemv_seq_f32_item *items, int n, int T)
{
    if (!items || n < 1 || T < 1 || T > 8) return 0;
    std::vector<qgemv_seq_item> sq;
    if (!seq_f32_items(items, n, sq)) return 0;
    return seq_ws(sq.data(), n, T, true);
}

qgemv_status qgemv_q4_0_seq_f32(const qgemv_seq_f32_item *items, int n, qgemv_wlayout layout, int T, void *ws,
                                size_t ws_bytes, qgemv_stream_t stream)
{
    if (!items || n < 1 || T < 1 || T > 8) return QGEMV_ERR_INVALID_ARG;
    std::vector<qgemv_seq_item> sq;
    if (!seq_f32_items(items, n, sq)) return QGEMV_ERR_INVALID_ARG;
    const qgemv_status s = check_seq(sq.data(), n, layout, T, ws, ws_bytes, true);
    if (s != QGEMV_OK) return s;
    return launch_seq(sq.data(), n, layout, T, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream), true);
}

static bool seq_ep_items(const qgemv_seq_ep_item *items, int n, std::vector<qgemv_seq_item> &sq,
                         std::vector<const float *> &bias, std::vector<const float *> &res)
{
    sq.resize(n);
    bias.resize(n);
    res.resize(n);
    for (int i = 0; i < n; ++i) {
        if (!shape_ok(items[i].N, items[i].K)) return false;
        sq[i] = qgemv_seq_item{items[i].W, items[i].x, items[i].y, items[i].N, items[i].K};
        bias[i] = items[i].bias;
        res[i] = items[i].residual;
    }
    return true;
}

size_t qgemv_seq_ep_workspace_bytes(const qgemv_seq_ep_item *items, int n, int T, int x_f32)
{
    (void)x_f32;  // the same plans either way
    if (!items || n < 1 || T < 1 || T > 8) return 0;
    std::vector<qgemv_seq_item> sq;
    std::vector<const float *> bias, res;
    if (!seq_ep_items(items, n, sq, bias, res)) return 0;
    return qgemv_seq_workspace_bytes(sq.data(), n, T);
}

qgemv_status qgemv_q4_0_seq_ep(const qgemv_seq_ep_item *items, int n, qgemv_wlayout layout, int T, int x_f32,
                               void *ws, size_t ws_bytes, qgemv_stream_t stream)
{
    if (!items || n < 1 || T < 1 || T > 8 || (x_f32 != 0 && x_f32 != 1)) return QGEMV_ERR_INVALID_ARG;
    std::vector<qgemv_seq_item> sq;
    std::vector<const float *> bias, res;
    if (!seq_ep_items(items, n, sq, bias, res)) return QGEMV_ERR_INVALID_ARG;
    const qgemv_status s = check_seq(sq.data(), n, layout, T, ws, ws_bytes, x_f32 != 0, bias.data(), res.data());
    if (s != QGEMV_OK) return s;
    return launch_seq(sq.data(), n, layout, T, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream), x_f32 != 0,
                      bias.data(), res.data());
}

extern "C++" {
// One gather matrix, quantised (xq) or fp32 (x) activations alike.
struct GatherIn {
    const void *W;
    long long expert_stride;
    const void *x;  // planar Q8_0, or fp32 [T][K] on the fp32 call
    long long x_stride;
    float *y;
    long long y_stride;
    long long N, K;
};

static GatherIn gather_in(const qgemv_gather_matrix &a)
{
    return GatherIn{a.W, a.expert_stride, a.xq, a.xq_stride, a.y, a.y_stride, a.N, a.K};
}
static GatherIn gather_in(const qgemv_gather_f32_matrix &a)
{
    return GatherIn{a.W, a.expert_stride, a.x, a.x_stride, a.y, a.y_stride, a.N, a.K};
}

static qgemv_status gather_specs(const GatherIn *mats, int n_mats, int n_ids, int T, GroupSpec *gs)
{
    if (!mats || n_mats < 1 || n_mats > MAXG_SMALL || n_ids < 1 || T < 1 || T > 8) return QGEMV_ERR_INVALID_ARG;
    for (int m = 0; m < n_mats; ++m) {
        const GatherIn &a = mats[m];
        if (!shape_ok(a.N, a.K)) return QGEMV_ERR_INVALID_ARG;
        if (n_ids > 1 && a.y_stride < static_cast<long long>(T) * a.N) return QGEMV_ERR_INVALID_ARG;
        if (a.expert_stride < 0 || a.x_stride < 0) return QGEMV_ERR_INVALID_ARG;
        gs[m] = GroupSpec{a.W, a.expert_stride, a.x, a.x_stride, a.y, a.y_stride, a.N, a.K, n_ids};
    }
    return QGEMV_OK;
}

template <class M>
static size_t gather_ws(const M *mats, int n_mats, int n_ids, int T)
{
    if (!mats || n_mats < 1 || n_mats > MAXG_SMALL) return 0;
    GatherIn in[MAXG_SMALL];
    for (int m = 0; m < n_mats; ++m) in[m] = gather_in(mats[m]);
    GroupSpec gs[MAXG_SMALL];
    if (gather_specs(in, n_mats, n_ids, T, gs) != QGEMV_OK) return 0;
    Plan<MAXG_SMALL> a, b;
    make_plan<MAXG_SMALL>(gs, n_mats, T, false, false, nullptr, 0, a);
    make_plan<MAXG_SMALL>(gs, n_mats, T, true, false, nullptr, 0, b);
    return static_cast<size_t>(a.ws_bytes > b.ws_bytes ? a.ws_bytes : b.ws_bytes);
}

}  // extern "C++"

size_t qgemv_gather_workspace_bytes(const qgemv_gather_matrix *mats, int n_mats, int n_ids, int T)
{
    return gather_ws(mats, n_mats, n_ids, T);
}

size_t qgemv_gather_f32_workspace_bytes(const qgemv_gather_f32_matrix *mats, int n_mats, int n_ids, int T)
{
    return gather_ws(mats, n_mats, n_ids, T);
}

// The gather calls (checked here).  xf32: activations are fp32 x[T][K],
// quantised inside the kernel.  Launched with programmatic dependent launch:
// the kernel reads the expert ids (which the preceding kernel may write)
// only after its dependency wait.
static qgemv_status gather_call(const GatherIn *mats, int n_mats, const int32_t *ids, int n_ids, int n_experts,
                                qgemv_wlayout layout, int T, void *ws, size_t ws_bytes, qgemv_stream_t stream,
                                bool xf32)
{
    GroupSpec gs[MAXG_SMALL];
    qgemv_status s = gather_specs(mats, n_mats, n_ids, T, gs);
    if (s != QGEMV_OK) return s;
    if (layout != QGEMV_W_GGML && layout != QGEMV_W_PACKED) return QGEMV_ERR_INVALID_ARG;
    if (!ids || n_experts < 1) return QGEMV_ERR_INVALID_ARG;
    if (!aligned(ids, 4)) return QGEMV_ERR_MISALIGNED;
    if (!ws) return QGEMV_ERR_WORKSPACE;
    if (!aligned(ws, 256)) return QGEMV_ERR_MISALIGNED;
    const Range rw = range(ws, static_cast<long long>(ws_bytes));
    const long long xa = xf32 ? 4 : 16;
    for (int m = 0; m < n_mats; ++m) {
        const GatherIn &a = mats[m];
        if (!a.W || !a.x || !a.y) return QGEMV_ERR_INVALID_ARG;
        const size_t wa = layout == QGEMV_W_PACKED ? 16 : 2;
        if (!aligned(a.W, wa) || a.expert_stride % static_cast<long long>(wa) != 0 || !aligned(a.x, xa) ||
            a.x_stride % xa != 0 || !aligned(a.y, 4))
            return QGEMV_ERR_MISALIGNED;
        const Range ry = range(a.y, 4ll * ((n_ids - 1) * a.y_stride + static_cast<long long>(T) * a.N));
        if (overlap(ry, rw)) return QGEMV_ERR_INVALID_ARG;
        for (int k = 0; k < n_mats; ++k) {
            const GatherIn &b = mats[k];
            const long long wb = (n_experts - 1) * b.expert_stride + 18ll * b.N * (b.K / QK);
            const long long xb = (n_ids - 1) * b.x_stride + (xf32 ? 4ll * T * b.K : xq_bytes_host(T, b.K));
            if (overlap(ry, range(b.W, wb)) || overlap(ry, range(b.x, xb))) return QGEMV_ERR_INVALID_ARG;
            if (k != m && overlap(ry, range(b.y, 4ll * ((n_ids - 1) * b.y_stride + static_cast<long long>(T) * b.N))))
                return QGEMV_ERR_INVALID_ARG;
        }
    }
    DevInfo dev;
    s = device_info(dev);
    if (s != QGEMV_OK) return s;
    Plan<MAXG_SMALL> pl;
    int cps = ctas_per_sm_for(T, false);
    s = plan_launch<MAXG_SMALL>(gs, n_mats, T, layout == QGEMV_W_GGML, false, static_cast<uint8_t *>(ws), dev, cps,
                                pl);
    if (s != QGEMV_OK) return s;
    if (static_cast<long long>(ws_bytes) < pl.ws_bytes) return QGEMV_ERR_WORKSPACE;
    pl.P.status = dev.status;
    pl.P.ids = ids;
    pl.P.n_experts = n_experts;
    pl.P.xf32 = xf32 ? 1 : 0;
    const int grid = grid_for(dev, cps);
    set_cta_groups(pl.P, grid);
    return dispatch_T<MAXG_SMALL, false>(pl.P, T, mma_for(T), grid, pl.smem, reinterpret_cast<cudaStream_t>(stream), true) ==
                   cudaSuccess
               ? QGEMV_OK
               : QGEMV_ERR_CUDA;
}

qgemv_status qgemv_q4_0_gather(const qgemv_gather_matrix *mats, int n_mats, const int32_t *ids, int n_ids,
                               int n_experts, qgemv_wlayout layout, int T, void *ws, size_t ws_bytes,
                               qgemv_stream_t stream)
{
    if (!mats || n_mats < 1 || n_mats > MAXG_SMALL) return QGEMV_ERR_INVALID_ARG;
    GatherIn in[MAXG_SMALL];
    for (int m = 0; m < n_mats; ++m) in[m] = gather_in(mats[m]);
    return gather_call(in, n_mats, ids, n_ids, n_experts, layout, T, ws, ws_bytes, stream, false);
}

qgemv_status qgemv_q4_0_gather_f32(const qgemv_gather_f32_matrix *mats, int n_mats, const int32_t *ids, int n_ids,
                                   int n_experts, qgemv_wlayout layout, int T, void *ws, size_t ws_bytes,
                                   qgemv_stream_t stream)
{
    if (!mats || n_mats < 1 || n_mats > MAXG_SMALL) return QGEMV_ERR_INVALID_ARG;
    GatherIn in[MAXG_SMALL];
    for (int m = 0; m < n_mats; ++m) in[m] = gather_in(mats[m]);
    return gather_call(in, n_mats, ids, n_ids, n_experts, layout, T, ws, ws_bytes, stream, true);
}

qgemv_status qgemv_debug_block_isums(const void *W, qgemv_wlayout layout, const void *xq, int32_t *isums, int64_t N,
                                     int64_t K, int T, qgemv_stream_t stream)
{
    if (!shape_ok(N, K) || T < 1 || T > 8 || !W || !xq || !isums) return QGEMV_ERR_INVALID_ARG;
    if (layout != QGEMV_W_GGML && layout != QGEMV_W_PACKED) return QGEMV_ERR_INVALID_ARG;
    if (!aligned(W, layout == QGEMV_W_PACKED ? 16 : 2) || !aligned(xq, 16) || !aligned(isums, 4))
        return QGEMV_ERR_MISALIGNED;
    return launch_isums(W, layout == QGEMV_W_PACKED, xq, isums, N, K, T, reinterpret_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? QGEMV_OK
               : QGEMV_ERR_CUDA;
}

qgemv_status qgemv_debug_block_isums_tc(const void *W, qgemv_wlayout layout, const void *xq, int32_t *isums,
                                        int64_t N, int64_t K, int T, int f16_image, qgemv_stream_t stream)
{
    if (!shape_ok(N, K) || T < 1 || T > 8 || !W || !xq || !isums) return QGEMV_ERR_INVALID_ARG;
    if (layout != QGEMV_W_GGML && layout != QGEMV_W_PACKED) return QGEMV_ERR_INVALID_ARG;
    if (f16_image != 0 && f16_image != 1) return QGEMV_ERR_INVALID_ARG;
    if (!aligned(W, layout == QGEMV_W_PACKED ? 16 : 2) || !aligned(xq, 16) || !aligned(isums, 4))
        return QGEMV_ERR_MISALIGNED;
    return launch_isums_tc(W, layout == QGEMV_W_PACKED, xq, isums, N, K, T, f16_image != 0,
                           reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? QGEMV_OK
               : QGEMV_ERR_CUDA;
}

qgemv_status qgemv_debug_stream_read(const void *src, size_t bytes, int method, int warps, int depth,
                                     int stage_bytes, unsigned long long *sink, qgemv_stream_t stream)
{
    if (!src || !sink || bytes < 16 || (method != 0 && method != 1) || warps < 1 || warps > 32 || depth < 1)
        return QGEMV_ERR_INVALID_ARG;
    if (method == 0 && (stage_bytes < 16 || stage_bytes % 16 != 0 || depth > 16 ||
                        static_cast<long long>(warps) * depth * stage_bytes > 200 * 1024))
        return QGEMV_ERR_INVALID_ARG;
    if (!aligned(src, 16) || !aligned(sink, 8)) return QGEMV_ERR_MISALIGNED;
    DevInfo dev;
    qgemv_status s = device_info(dev);
    if (s != QGEMV_OK) return s;
    return launch_stream_bench(src, static_cast<long long>(bytes), method, warps, depth, stage_bytes, sink, dev.status,
                               dev.sms, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? QGEMV_OK
               : QGEMV_ERR_CUDA;
}

qgemv_status qgemv_set_tuning(int ctas_per_sm, int waves, int mma_min_T, int ring_depth)
{
    if (ctas_per_sm < 0 || ctas_per_sm > 2 || waves < 0 || waves > 6 || mma_min_T < 0 || mma_min_T > 9 ||
        ring_depth < 0 || ring_depth > MAX_RING)
        return QGEMV_ERR_INVALID_ARG;
    g_ctas_per_sm.store(ctas_per_sm);
    g_waves.store(waves);
    g_mma_min_T.store(mma_min_T);
    g_ring_depth.store(ring_depth);
    return QGEMV_OK;
}

qgemv_status qgemv_set_ffn_fused(int on)
{
    if (on != 0 && on != 1) return QGEMV_ERR_INVALID_ARG;
    g_ffn_fused.store(on);
    return QGEMV_OK;
}

qgemv_status qgemv_set_tc_min_tokens(int tc_min_T)
{
    if (tc_min_T < 0 || tc_min_T > 9) return QGEMV_ERR_INVALID_ARG;
    g_tc_min_T.store(tc_min_T);
    return QGEMV_OK;
}

qgemv_status qgemv_device_status(int *code_out)
{
    if (!code_out) return QGEMV_ERR_INVALID_ARG;
    DevInfo dev;
    qgemv_status s = device_info(dev);
    if (s != QGEMV_OK) return s;
    if (cudaDeviceSynchronize() != cudaSuccess) return QGEMV_ERR_CUDA;
    unsigned v = 0, zero = 0;
    if (cudaMemcpy(&v, dev.status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return QGEMV_ERR_CUDA;
    if (cudaMemcpy(dev.status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return QGEMV_ERR_CUDA;
    *code_out = static_cast<int>(v);
    return QGEMV_OK;
}

}  // extern "C"

// =====================================================================
// Allocation-free lm_head argmax.
//
// Some callers cannot allocate device memory at the point where they run
// the lm_head: a plugin that a host framework hands only its input and
// output tensors, a runtime whose device memory is fixed up front, or code
// already inside a region where allocation is forbidden.  For them this
// entry point takes its scratch (completion counters, per-CTA argmax
// candidates, split-K partial sums) from one fixed array that lives in the
// library's own device memory, so the caller passes inputs and outputs only.

namespace {
constexpr long long kNoAllocScratchBytes = 4ll << 20;  // 4 MiB per device
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices] = {};
}  // namespace

// Held by every GPU that loads the library until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

extern "C" qgemv_status qgemv_q4_0_argmax_noalloc(const void *W, qgemv_wlayout layout, const void *xq,
                                                  float *y_or_null, int64_t *idx, int64_t N, int64_t K, int T,
                                                  qgemv_stream_t stream)
{
    if (!shape_ok(N, K) || T < 1 || T > 8) return QGEMV_ERR_INVALID_ARG;
    if (single_ws_bytes(N, K, T) > kNoAllocScratchBytes) return QGEMV_ERR_UNSUPPORTED;
    // Every argument check first, on the host: a refused call makes no CUDA
    // call and enqueues nothing (so it cannot clear the counters of a call
    // still running on another stream).
    const qgemv_status chk = argmax_check(W, layout, xq, false, y_or_null, idx, N, K, T, nullptr, 0);
    if (chk != QGEMV_OK) return chk;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QGEMV_ERR_CUDA;
    void *scratch = nullptr;
    {
        // Once per device, with that device current: the array's device
        // address (host code cannot use the symbol itself as a pointer).
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        if (g_noalloc_ptr[dev] == nullptr) {
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return QGEMV_ERR_CUDA;
            g_noalloc_ptr[dev] = p;
        }
        scratch = g_noalloc_ptr[dev];
    }
    // All calls share the array and it keeps the last call's contents: the
    // counters must start at zero, so clear them on the caller's stream.
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(scratch, 0, static_cast<size_t>(CNT_AREA), st) != cudaSuccess) return QGEMV_ERR_CUDA;
    return run_single(W, layout, xq, y_or_null, reinterpret_cast<long long *>(idx), N, K, T, scratch,
                      static_cast<size_t>(kNoAllocScratchBytes), st, true, true);
}
