// qgemm_api.cu -- the C ABI (include/qgemm.h): argument validation, path
// selection, TMA descriptor set-up, counters, options and device status.
// Host code only, apart from the device status word.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "qgemm.h"

namespace {

// ------------------------------------------------------------ errors
thread_local char g_err[256] = {0};

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}
void clear_err() { g_err[0] = 0; }
int cuda_fail(cudaError_t e, const char* what) {
    return fail(QGEMM_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// ------------------------------------------------------------ global state
std::atomic<uint64_t> g_cnt[13];
enum { C_QUANT, C_XPREP, C_Q4K_TC, C_Q6K_TC, C_Q4K_SMALL, C_Q6K_SMALL, C_PREPACK, C_SPLITK, C_ROUTED, C_PTQ1_TC,
       C_PTQ1_PREPACK, C_SMALL_FUSED, C_SIDE };
// SMALL_M_MAX defaults to the measured crossover: the streaming kernel wins up
// to 8 tokens at K = N = 5120 and at K = 4096, N = 14336.
// Q4K_SIDE_MIN_TILES defaults to the measured crossover (Q4_K fp32 entry,
// CUDA-graph steps on one GB300, side-data kernel against side words made in
// the GEMM): with one to three token tiles per weight tile the kernel adds
// more than it saves (K = N = 5120: M = 64 26.7 against 24.6 us, M = 256 39.9
// against 38.7, M = 384 41.4 against 39.4); at four the two are even (M = 512
// 57.8 and 57.8; K = 2048, N = 11008: 47.6 and 47.6); beyond, it saves (M =
// 2048: 135.5 against 140.6 us).
std::atomic<int64_t> g_opt[6] = {{qg::SMALL_M_LIMIT}, {0}, {0}, {0}, {0}, {4}};
// the wait limit and the test-only skip switch, as the kernels take them
qg::WaitCfg wait_cfg() {
    return qg::WaitCfg{static_cast<int>(g_opt[QGEMM_OPT_WAIT_LIMIT_US].load()),
                       static_cast<int>(g_opt[QGEMM_OPT_TEST_SKIP_ARRIVAL].load())};
}
std::atomic<cudaEvent_t> g_ev_before{nullptr}, g_ev_after{nullptr};

}  // namespace

// Device status: [0] = bits, [1] = 1 + site of the first timed-out wait.
__device__ __align__(8) uint32_t g_qgemm_status[qg::ST_WORDS];

namespace {

constexpr int MAX_DEV = 64;
struct DevState {
    bool init = false;
    cudaError_t init_err = cudaSuccess;
    uint32_t* status = nullptr;
    int sm_count = 0;
};
std::mutex g_mtx;
DevState g_dev[MAX_DEV];

int device_state(DevState** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= MAX_DEV) return fail(QGEMM_EUNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_mtx);
    DevState& st = g_dev[dev];
    if (!st.init) {
        st.init = true;
        e = cudaGetSymbolAddress(reinterpret_cast<void**>(&st.status), g_qgemm_status);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, dev);
        for (int wt : {4, 6, 1})
            for (int bm : {16, 32, 64, 128})
                if (e == cudaSuccess) e = qg::tc_prepare(wt, bm);
        st.init_err = e;
    }
    if (st.init_err != cudaSuccess) return cuda_fail(st.init_err, "device set-up");
    *out = &st;
    return QGEMM_OK;
}

// ------------------------------------------------------------ TMA descriptors
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// 2D tiled map: `inner` elements per row (contiguous), `outer` rows,
// `row_bytes` between rows, box {box_inner, box_outer}; out of range -> zeros.
int make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
             uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(QGEMM_ECUDA, "cuTensorMapEncodeTiled not available from the driver");
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(QGEMM_ECUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    return QGEMM_OK;
}

// A 3D map: dims {inner, mid, outer} elements, byte strides of mid and outer.
int make_map3(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t mid, uint64_t outer,
              uint64_t mid_bytes, uint64_t outer_bytes, uint32_t box_inner, uint32_t box_mid, uint32_t box_outer,
              CUtensorMapSwizzle swz) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(QGEMM_ECUDA, "cuTensorMapEncodeTiled not available from the driver");
    const cuuint64_t dims[3] = {inner, mid, outer};
    const cuuint64_t strides[2] = {mid_bytes, outer_bytes};
    const cuuint32_t box[3] = {box_inner, box_mid, box_outer};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(QGEMM_ECUDA, "cuTensorMapEncodeTiled (3D) failed (%d)", static_cast<int>(r));
    return QGEMM_OK;
}

// ------------------------------------------------------------ validation
int check_q8k(const int8_t* xqs, const float* xd, const int16_t* xbsums) {
    if (!xqs || !xd || !xbsums) return fail(QGEMM_EINVAL, "null Q8_K plane");
    if (!aligned(xqs, 16) || !aligned(xd, 16) || !aligned(xbsums, 16))
        return fail(QGEMM_EALIGN, "Q8_K planes must be 16-byte aligned");
    return QGEMM_OK;
}
int check_mk(int64_t M, int64_t K) {
    if (M < 0) return fail(QGEMM_EINVAL, "M must be >= 0 (got %lld)", static_cast<long long>(M));
    if (K < 256 || K % 256 != 0)
        return fail(QGEMM_EINVAL, "K must be a positive multiple of 256 (got %lld)", static_cast<long long>(K));
    if (M >= (int64_t(1) << 31) || K >= (int64_t(1) << 31))
        return fail(QGEMM_EUNSUPPORTED, "M and K must be below 2^31");
    return QGEMM_OK;
}

struct Plan {
    int bm;
    qg::TcWork work;   // without its pointers
};

// Tile width from M; the work list from the tile count and the SM count.
// With fewer tiles than SMs every tile is cut into K parts so that the parts
// fill the SMs (a part is still a whole 128-row x BM-token tile over a K
// range: the pages' BigTile lesson that a tile must be shared is kept).
// With more tiles than SMs, a last round that would leave at least half of
// the SMs idle is cut the same way and the earlier rounds stay whole
// (measured on GB300, M=512 K=5120 N=5120: 160 tiles, the last round's 8 cut
// into 8 parts, 73 -> 58 us; 344 tiles, 40 into 3 parts, 51.5 -> 50.7 us).
Plan plan_tc(int64_t M, int64_t N, int64_t K, int sm_count) {
    Plan p{};
    const int64_t fbm = g_opt[QGEMM_OPT_FORCE_BM].load();
    if (fbm == 16 || fbm == 32 || fbm == 64 || fbm == 128)
        p.bm = static_cast<int>(fbm);
    else
        p.bm = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128;
    const int64_t nb = K / 256;
    qg::TcWork& w = p.work;
    w.n_tiles = static_cast<int>((N + 127) / 128);
    w.m_tiles = static_cast<int>((M + p.bm - 1) / p.bm);
    // Work order.  Token tiles vary fastest, so the CTAs running at once share
    // a few weight tiles and sweep the activations.  Past 32 MiB of fp16
    // activations a sweep no longer stays in L2 beside the Y being written
    // (measured on GB300, M=8192 K=5120 N=5120: 1.52 GB of DRAM reads for
    // ~0.1 GB of operands).  The token tiles are then taken in groups of
    // about 32 MiB, each group swept by all weight tiles before the next:
    // every weight tile is read once per group, every activation once.
    // (Measured on GB300 at M=8192 K=N=5120, one build against another on
    // the same GPU: groups of 32 MiB 445 us, of 16 MiB 449 us, of 8 MiB
    // 445 us; an earlier build ran 1.5% slower with a single group.)
    {
        const int64_t tile_act = static_cast<int64_t>(p.bm) * K * 2;   // fp16 bytes of one token tile
        int64_t g = w.m_tiles;
        if (M * K * 2 > (int64_t(32) << 20)) g = (int64_t(32) << 20) / tile_act;
        if (g < 1) g = 1;
        w.m_group = static_cast<int>(g < w.m_tiles ? g : w.m_tiles);
    }
    {
        // (see TcWork; measured on GB300: the two 32-bit divisions this replaces
        // in every role's work decode cost 0.5% at M=8192 K=N=5120)
        auto magic = [](int64_t d, uint64_t& mul, int& shr) {
            if (d < 1) d = 1;   // (no tiles: never used)
            int l = 0;
            while ((int64_t(1) << l) < d) ++l;
            mul = ((uint64_t(1) << (32 + l)) + uint64_t(d) - 1) / uint64_t(d);
            shr = 32 + l;
        };
        const int64_t ng = (w.m_tiles + w.m_group - 1) / w.m_group;
        magic(int64_t(w.m_group) * w.n_tiles, w.dv_gsz_mul, w.dv_gsz_shr);
        magic(w.m_group, w.dv_mg_mul, w.dv_mg_shr);
        magic(w.m_tiles - (ng - 1) * w.m_group, w.dv_ml_mul, w.dv_ml_shr);
    }
    const int64_t T = static_cast<int64_t>(w.n_tiles) * w.m_tiles;
    const int64_t maxparts = nb / 2 > 1 ? (nb / 2 < 8 ? nb / 2 : 8) : 1;   // >= 2 superblocks per part
    int64_t parts = 1, full = T;
    const int64_t fs = g_opt[QGEMM_OPT_FORCE_SPLITS].load();
    if (fs > 0) {
        parts = fs < nb ? fs : nb;
        full = parts > 1 ? 0 : T;
    } else {
        const int64_t G = sm_count > 0 ? sm_count : 1;
        if (T < G) {
            parts = G / T;
            if (parts > maxparts) parts = maxparts;
            full = parts > 1 ? 0 : T;
        } else if (T % G != 0 && 2 * (T % G) <= G) {
            // a short last round: its tiles are cut so that every SM takes a part
            const int64_t tail = T % G;
            int64_t pp = G / tail;
            if (pp > maxparts) pp = maxparts;
            if (pp > 1) parts = pp, full = T - tail;
        }
    }
    if (T - full > qg::TC_MAX_CUT_TILES) parts = 1, full = T;   // counters are finite
    if (parts > 1 && nb * parts >= (int64_t(1) << 31)) parts = (int64_t(1) << 31) / nb - 1;   // 32-bit part bounds
    if (parts <= 1) parts = 1, full = T;
    w.full_items = static_cast<int>(full);
    w.parts = static_cast<int>(parts);
    w.items = static_cast<int>(full + (T - full) * parts);
    return p;
}

size_t plane_bytes(int64_t M, int64_t K) {
    const int64_t nb = K / 256, Mp = (M + 3) / 4 * 4;
    return align256(size_t(M) * K * 2) + align256(size_t(M) * (K / 16) * 2) + align256(size_t(nb) * Mp * 4);
}
constexpr size_t COUNTER_BYTES = qg::TC_COUNTERS * sizeof(int);

// The Q4_K side words (qg::launch_q4k_side) of an N x K weight matrix: two
// 32-byte slabs per row and superblock, then the fp32 scales e [nb][Np].
int64_t side_np(int64_t N) { return (N + 3) / 4 * 4; }
size_t side_slab_bytes(int64_t N, int64_t K) { return align256(size_t(K / 256) * 2 * size_t(N) * 32); }
size_t side_bytes(int64_t N, int64_t K) {
    return N > 0 ? side_slab_bytes(N, K) + align256(size_t(K / 256) * size_t(side_np(N)) * 4) : 0;
}

size_t partial_bytes(const Plan& p) {
    const int64_t cut = static_cast<int64_t>(p.work.n_tiles) * p.work.m_tiles - p.work.full_items;
    return cut > 0 ? size_t(cut) * p.work.parts * 128 * p.bm * sizeof(float) : 0;
}

// SM count for sizing the workspace: the current device's, else a bound.
int sizing_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) ==
                                                   cudaSuccess && n > 0)
        return n;
    cudaGetLastError();   // (no device: clear the sticky-free error state)
    return 160;
}

// The workspace of the tile GEMM: the operand planes, the cut-tile counters,
// the Q4_K side words (sized by N), then the partial tiles of the cut tiles.
struct WsPlanes {
    __half* xh;
    __half* xbs;
    float* dxT;
    int64_t Mp;
    int* counters;
    uint32_t* side;
    float* side_e;
    float* partials;
};
WsPlanes ws_planes(void* ws, int64_t M, int64_t K, int64_t N = 0) {
    uint8_t* base = static_cast<uint8_t*>(ws);
    WsPlanes p{};
    p.Mp = (M + 3) / 4 * 4;
    p.xh = reinterpret_cast<__half*>(base);
    p.xbs = reinterpret_cast<__half*>(base + align256(size_t(M) * K * 2));
    p.dxT = reinterpret_cast<float*>(base + align256(size_t(M) * K * 2) + align256(size_t(M) * (K / 16) * 2));
    p.counters = reinterpret_cast<int*>(base + plane_bytes(M, K));
    uint8_t* side = base + plane_bytes(M, K) + COUNTER_BYTES;
    p.side = reinterpret_cast<uint32_t*>(side);
    p.side_e = reinterpret_cast<float*>(side + side_slab_bytes(N, K));
    p.partials = reinterpret_cast<float*>(side + side_bytes(N, K));
    return p;
}

// Q4_K tile GEMM (not routed): the side words come precomputed (their own
// kernel, loaded by the GEMM) when a weight tile meets at least
// QGEMM_OPT_Q4K_SIDE_MIN_TILES token tiles, else the GEMM makes them itself.
bool q4k_side_precomputed(const Plan& pl) { return pl.work.m_tiles >= g_opt[QGEMM_OPT_Q4K_SIDE_MIN_TILES].load(); }

int run_tc(int wtype, const void* w, int64_t N, int64_t K, int64_t ldw, const int8_t* xqs, const float* xd,
           const int16_t* xbsums, int64_t M, void* y, int64_t ldy, void* ws, size_t ws_bytes,
           cudaStream_t stream, bool prepared, const qg::Epi& epi = qg::Epi{}, bool side_ready = false) {
    DevState* ds = nullptr;
    int rc = device_state(&ds);
    if (rc) return rc;
    const size_t need = qgemm_workspace_bytes(M, N, K);
    if (!ws || ws_bytes < need)
        return fail(QGEMM_EINVAL, "workspace of %zu bytes needed (got %zu)", need, ws ? ws_bytes : size_t(0));
    if (!aligned(ws, 256)) return fail(QGEMM_EALIGN, "workspace must be 256-byte aligned");

    const Plan pl = plan_tc(M, N, K, ds->sm_count);
    const int64_t nb = K / 256;
    const WsPlanes wp = ws_planes(ws, M, K, N);
    const int64_t Mp = wp.Mp;
    __half* xh = wp.xh;
    __half* xbs = wp.xbs;
    float* dxT = wp.dxT;

    cudaError_t e = cudaSuccess;
    // Q4_K: the side words come precomputed (see gemm_tc_kernel.cuh) for
    // enough token tiles, made here unless the caller made them already
    const bool pre = wtype == 4 && q4k_side_precomputed(pl);
    const bool side_now = pre && !side_ready;
    if (side_now) {
        e = qg::launch_q4k_side(w, N, nb, ldw, wp.side, wp.side_e, side_np(N), stream);
        if (e != cudaSuccess) return cuda_fail(e, "side-data launch");
        g_cnt[C_SIDE]++;
    }
    if (!prepared) {
        // (a prepared workspace already holds these planes: qgemm_quantize_q8k_prep;
        // after the side-data kernel this one runs beside it)
        e = qg::launch_xprep(xqs, xd, xbsums, M, K, xh, xbs, dxT, Mp, wp.counters, stream, side_now);
        if (e != cudaSuccess) return cuda_fail(e, "operand preparation launch");
        g_cnt[C_XPREP]++;
    }

    CUtensorMap tm_w, tm_xh, tm_xbs, tm_dx;
    const int blk = wtype == 4 ? qg::Q4K_BLOCK : wtype == 6 ? qg::Q6K_PACKED : 2 * qg::PTQ1_PACKED;
    if ((rc = make_map(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, uint64_t(nb) * blk, N, ldw, blk, 128,
                       CU_TENSOR_MAP_SWIZZLE_NONE)))
        return rc;
    if ((rc = make_map(&tm_xh, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, xh, K, M, uint64_t(K) * 2, 64, pl.bm,
                       CU_TENSOR_MAP_SWIZZLE_128B)))
        return rc;
    if ((rc = make_map(&tm_xbs, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, xbs, K / 16, M, uint64_t(K / 16) * 2, 16, pl.bm,
                       CU_TENSOR_MAP_SWIZZLE_32B)))
        return rc;
    if ((rc = make_map(&tm_dx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dxT, Mp, nb, uint64_t(Mp) * 4, pl.bm, 1,
                       CU_TENSOR_MAP_SWIZZLE_NONE)))
        return rc;
    CUtensorMap tm_side, tm_e;
    if (pre) {
        // slabs [2 nb][N][8 words]: a 128-row box of both slabs of superblock b lands as the
        // two 32-byte-swizzled correction operands the MMA reads
        if ((rc = make_map3(&tm_side, CU_TENSOR_MAP_DATA_TYPE_UINT32, wp.side, 8, N, uint64_t(2) * nb, 32,
                            uint64_t(N) * 32, 8, 128, 2, CU_TENSOR_MAP_SWIZZLE_32B)))
            return rc;
        if ((rc = make_map(&tm_e, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, wp.side_e, N, nb, uint64_t(side_np(N)) * 4, 128, 1,
                           CU_TENSOR_MAP_SWIZZLE_NONE)))
            return rc;
    }

    qg::TcLaunch a{};
    a.wtype = wtype;
    a.bm = pl.bm;
    a.M = M;
    a.N = N;
    a.K = K;
    a.work = pl.work;
    a.work.counters = wp.counters;
    a.work.partials = wp.partials;
    a.work.wait = wait_cfg();
    a.sm_count = ds->sm_count;
    a.y = y;
    a.ldy = ldy;
    a.epi = epi;
    a.status = ds->status;
    a.tm_w = &tm_w;
    a.tm_xh = &tm_xh;
    a.tm_xbs = wtype == 4 ? &tm_xbs : nullptr;
    a.tm_dx = &tm_dx;
    a.tm_side = pre ? &tm_side : nullptr;
    a.tm_e = pre ? &tm_e : nullptr;
    cudaEvent_t evb = g_ev_before.load(), eva = g_ev_after.load();
    if (evb) cudaEventRecord(evb, stream);
    e = qg::launch_gemm_tc(a, stream);
    if (eva) cudaEventRecord(eva, stream);
    if (e != cudaSuccess) return cuda_fail(e, "tile GEMM launch");
    g_cnt[wtype == 4 ? C_Q4K_TC : wtype == 6 ? C_Q6K_TC : C_PTQ1_TC]++;
    if (pl.work.parts > 1) g_cnt[C_SPLITK]++;
    return QGEMM_OK;
}

// Small-M path: the Q8_K planes are read directly; no workspace, one launch.
int run_small(int wtype, const void* w, int64_t N, int64_t K, int64_t ldw, const int8_t* xqs, const float* xd,
              const int16_t* xbsums, int64_t M, void* y, int64_t ldy, cudaStream_t stream,
              const qg::Epi& epi = qg::Epi{}) {
    DevState* ds = nullptr;
    int rc = device_state(&ds);
    if (rc) return rc;
    qg::SmallLaunch a{};
    a.wtype = wtype;
    a.M = M;
    a.N = N;
    a.K = K;
    a.w = w;
    a.ldw = ldw;
    a.act.xqs = xqs;
    a.act.xd = xd;
    a.act.xbs = xbsums;
    a.y = y;
    a.ldy = ldy;
    a.epi = epi;
    a.sm_count = ds->sm_count;
    a.status = ds->status;
    a.wait = wait_cfg();
    cudaEvent_t evb = g_ev_before.load(), eva = g_ev_after.load();
    if (evb) cudaEventRecord(evb, stream);
    cudaError_t e = qg::launch_small(a, stream);
    if (eva) cudaEventRecord(eva, stream);
    if (e != cudaSuccess) return cuda_fail(e, "small-M launch");
    g_cnt[wtype == 4 ? C_Q4K_SMALL : C_Q6K_SMALL]++;
    return QGEMM_OK;
}

// Path choice by token count (the pages' column-count routing): the
// streaming kernel up to QGEMM_OPT_SMALL_M_MAX tokens, the tile GEMM above.
bool use_small(int wtype, int64_t M, int64_t K) {
    return M <= g_opt[QGEMM_OPT_SMALL_M_MAX].load() && qg::small_supported(wtype, M, K);
}

// Small-M path with the quantizer fused in: the kernel quantizes fp32 X
// itself (and stores the Q8_K planes); one launch.
int run_small_fused(int wtype, const void* w, int64_t N, int64_t K, int64_t ldw, const float* x, int64_t ldx,
                    int8_t* qs, float* d, int16_t* bsums, int64_t M, float* y, int64_t ldy, cudaStream_t stream) {
    DevState* ds = nullptr;
    int rc = device_state(&ds);
    if (rc) return rc;
    qg::SmallLaunch a{};
    a.wtype = wtype;
    a.M = M;
    a.N = N;
    a.K = K;
    a.w = w;
    a.ldw = ldw;
    a.act.x = x;
    a.act.ldx = ldx;
    a.act.oqs = qs;
    a.act.od = d;
    a.act.obs = bsums;
    a.y = y;
    a.ldy = ldy;
    a.sm_count = ds->sm_count;
    a.status = ds->status;
    a.wait = wait_cfg();
    cudaEvent_t evb = g_ev_before.load(), eva = g_ev_after.load();
    if (evb) cudaEventRecord(evb, stream);
    cudaError_t e = qg::launch_small(a, stream);
    if (eva) cudaEventRecord(eva, stream);
    if (e != cudaSuccess) return cuda_fail(e, "small-M (fused quantizer) launch");
    g_cnt[wtype == 4 ? C_Q4K_SMALL : C_Q6K_SMALL]++;
    g_cnt[C_SMALL_FUSED]++;
    return QGEMM_OK;
}

// ---- routed GEMM (MUL_MAT_ID): workspace = routing arrays, then the operand
// planes of the P = M * top_k routed rows.
struct IdWs {
    int* row_off;    // [E + 1]
    int* row_end;    // [E]
    int* tile_off;   // [E + 1]
    int* perm;       // [R], R = routed_rows_max(P, E)
    __half* xh;      // [P][K]
    __half* xbs;     // [P][K/16]
    float* dxT;      // [nb][Pp]
    int64_t Pp;
};
// routed rows (pairs plus per-expert padding to a multiple of 4) and their planes
size_t id_route_bytes(int64_t P, int64_t E) {
    return 3 * align256(size_t(E + 1) * 4) + align256(size_t(qg::routed_rows_max(P, E)) * 4);
}
IdWs id_ws(void* ws, int64_t P, int64_t E, int64_t K) {
    const int64_t R = qg::routed_rows_max(P, E);
    uint8_t* b = static_cast<uint8_t*>(ws);
    const size_t a = align256(size_t(E + 1) * 4);
    IdWs w{};
    w.row_off = reinterpret_cast<int*>(b);
    w.row_end = reinterpret_cast<int*>(b + a);
    w.tile_off = reinterpret_cast<int*>(b + 2 * a);
    w.perm = reinterpret_cast<int*>(b + 3 * a);
    uint8_t* planes = b + id_route_bytes(P, E);
    w.Pp = (R + 3) / 4 * 4;
    w.xh = reinterpret_cast<__half*>(planes);
    w.xbs = reinterpret_cast<__half*>(planes + align256(size_t(R) * K * 2));
    w.dxT = reinterpret_cast<float*>(planes + align256(size_t(R) * K * 2) + align256(size_t(R) * (K / 16) * 2));
    return w;
}
// token-tile width from the mean number of routed rows per expert
int id_bm(int64_t P, int64_t E) {
    const int64_t fbm = g_opt[QGEMM_OPT_FORCE_BM].load();
    if (fbm == 16 || fbm == 32 || fbm == 64 || fbm == 128) return static_cast<int>(fbm);
    const int64_t avg = (P + E - 1) / E;
    return avg <= 16 ? 16 : avg <= 32 ? 32 : avg <= 64 ? 64 : 128;
}

int run_id(int wtype, const void* w, int64_t E, int64_t N, int64_t K, int64_t ldw, const int8_t* xqs,
           const float* xd, const int16_t* xbsums, int64_t M, const int32_t* ids, int64_t top_k, float* y,
           int64_t ldy, void* ws, size_t ws_bytes, cudaStream_t stream) {
    DevState* ds = nullptr;
    int rc = device_state(&ds);
    if (rc) return rc;
    const int64_t P = M * top_k;
    const size_t need = qgemm_id_workspace_bytes(M, top_k, E, K);
    if (!ws || ws_bytes < need)
        return fail(QGEMM_EINVAL, "workspace of %zu bytes needed (got %zu)", need, ws ? ws_bytes : size_t(0));
    if (!aligned(ws, 256)) return fail(QGEMM_EALIGN, "workspace must be 256-byte aligned");
    const IdWs iw = id_ws(ws, P, E, K);
    const int bm = id_bm(P, E);
    const int64_t nb = K / 256;

    const int64_t R = qg::routed_rows_max(P, E);
    cudaError_t e = qg::launch_route(ids, P, static_cast<int>(E), bm, iw.row_off, iw.row_end, iw.tile_off, iw.perm,
                                     ds->status, stream);
    if (e != cudaSuccess) return cuda_fail(e, "routing launch");
    e = qg::launch_xgather(xqs, xd, xbsums, K, static_cast<int>(top_k), iw.perm, iw.row_off + E, R, iw.xh, iw.xbs,
                           iw.dxT, iw.Pp, stream);
    if (e != cudaSuccess) return cuda_fail(e, "routed operand gather launch");

    CUtensorMap tm_w, tm_xh, tm_xbs, tm_dx;
    const int blk = wtype == 4 ? qg::Q4K_BLOCK : qg::Q6K_PACKED;
    // the experts' weight rows stacked: E * N rows of the same row stride
    if ((rc = make_map(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, uint64_t(nb) * blk, E * N, ldw, blk, 128,
                       CU_TENSOR_MAP_SWIZZLE_NONE)))
        return rc;
    if ((rc = make_map(&tm_xh, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, iw.xh, K, R, uint64_t(K) * 2, 64, bm,
                       CU_TENSOR_MAP_SWIZZLE_128B)))
        return rc;
    if ((rc = make_map(&tm_xbs, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, iw.xbs, K / 16, R, uint64_t(K / 16) * 2, 16, bm,
                       CU_TENSOR_MAP_SWIZZLE_32B)))
        return rc;
    if ((rc = make_map(&tm_dx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, iw.dxT, iw.Pp, nb, uint64_t(iw.Pp) * 4, bm, 1,
                       CU_TENSOR_MAP_SWIZZLE_NONE)))
        return rc;

    qg::TcLaunch a{};
    a.wtype = wtype;
    a.bm = bm;
    a.M = R;
    a.N = N;
    a.K = K;
    a.work.n_tiles = static_cast<int>((N + 127) / 128);
    a.work.m_tiles = 0;
    a.work.m_group = 1;   // (unused: the routed work list is read on the device)
    a.work.parts = 1;
    // the routed work list is read on the device; the grid is sized for its bound
    const int64_t bound = int64_t(a.work.n_tiles) * ((P + bm - 1) / bm + E);
    if (bound >= (int64_t(1) << 31)) return fail(QGEMM_EUNSUPPORTED, "routed work list too long");
    a.work.full_items = static_cast<int>(bound);
    a.work.items = static_cast<int>(bound);
    a.work.experts = static_cast<int>(E);
    a.work.tile_off = iw.tile_off;
    a.work.row_off = iw.row_off;
    a.work.row_end = iw.row_end;
    a.work.perm = iw.perm;
    a.work.wait = wait_cfg();
    a.sm_count = ds->sm_count;
    a.y = y;
    a.ldy = ldy;
    a.status = ds->status;
    a.tm_w = &tm_w;
    a.tm_xh = &tm_xh;
    a.tm_xbs = wtype == 4 ? &tm_xbs : nullptr;
    a.tm_dx = &tm_dx;
    cudaEvent_t evb = g_ev_before.load(), eva = g_ev_after.load();
    if (evb) cudaEventRecord(evb, stream);
    e = qg::launch_gemm_tc(a, stream);
    if (eva) cudaEventRecord(eva, stream);
    if (e != cudaSuccess) return cuda_fail(e, "routed tile GEMM launch");
    g_cnt[wtype == 4 ? C_Q4K_TC : C_Q6K_TC]++;
    g_cnt[C_ROUTED]++;
    return QGEMM_OK;
}


}  // namespace

namespace qg {
int set_last_error(int code, const char* msg) { return fail(code, "%s", msg); }
}  // namespace qg

extern "C" {

int qgemm_version(void) { return 100; }

const char* qgemm_last_error(void) { return g_err; }

int qgemm_quantize_q8k(const float* x, int64_t M, int64_t K, int64_t ldx, int8_t* qs, float* d, int16_t* bsums,
                       qgemm_stream_t stream) {
    clear_err();
    int rc = check_mk(M, K);
    if (rc) return rc;
    if (M == 0) return QGEMM_OK;
    if (!x) return fail(QGEMM_EINVAL, "x is null");
    if (ldx < K) return fail(QGEMM_EINVAL, "ldx (%lld) < K (%lld)", (long long)ldx, (long long)K);
    if (!aligned(x, 16) || ldx % 4 != 0) return fail(QGEMM_EALIGN, "x must be 16-byte aligned with ldx % 4 == 0");
    if ((rc = check_q8k(qs, d, bsums))) return rc;
    cudaError_t e = qg::launch_quantize_q8k(x, M, K, ldx, qs, d, bsums, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
    g_cnt[C_QUANT]++;
    return QGEMM_OK;
}

size_t qgemm_q8k_bytes(int64_t M, int64_t K) {
    if (M <= 0 || K <= 0 || K % 256) return 0;
    return align256(size_t(M) * K) + align256(size_t(M) * (K / 256) * 4) + align256(size_t(M) * (K / 16) * 2);
}

int qgemm_q8k_planes(void* base, int64_t M, int64_t K, int8_t** qs, float** d, int16_t** bsums) {
    clear_err();
    int rc = check_mk(M, K);
    if (rc) return rc;
    if (!base || !qs || !d || !bsums) return fail(QGEMM_EINVAL, "null pointer");
    if (!aligned(base, 256)) return fail(QGEMM_EALIGN, "the Q8_K buffer must be 256-byte aligned");
    uint8_t* b = static_cast<uint8_t*>(base);
    *qs = reinterpret_cast<int8_t*>(b);
    *d = reinterpret_cast<float*>(b + align256(size_t(M) * K));
    *bsums = reinterpret_cast<int16_t*>(b + align256(size_t(M) * K) + align256(size_t(M) * (K / 256) * 4));
    return QGEMM_OK;
}

size_t qgemm_q8k_aos_bytes(int64_t M, int64_t K) {
    if (M <= 0 || K <= 0 || K % 256) return 0;
    return size_t(M) * size_t(K / 256) * qg::Q8K_AOS_BLOCK;
}

static int aos_common(const void* aos, int64_t M, int64_t K, const int8_t* qs, const float* d,
                      const int16_t* bsums) {
    int rc = check_mk(M, K);
    if (rc || M == 0) return rc;
    if (!aos) return fail(QGEMM_EINVAL, "null 292-byte block buffer");
    if (!aligned(aos, 4)) return fail(QGEMM_EALIGN, "the 292-byte block buffer must be 4-byte aligned");
    return check_q8k(qs, d, bsums);
}

int qgemm_pack_q8k_aos(const int8_t* qs, const float* d, const int16_t* bsums, int64_t M, int64_t K, void* aos,
                       qgemm_stream_t stream) {
    clear_err();
    int rc = aos_common(aos, M, K, qs, d, bsums);
    if (rc || M == 0) return rc;
    cudaError_t e = qg::launch_q8k_aos(const_cast<int8_t*>(qs), const_cast<float*>(d), const_cast<int16_t*>(bsums),
                                       M, K, aos, true, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "Q8_K pack launch");
    return QGEMM_OK;
}

int qgemm_unpack_q8k_aos(const void* aos, int64_t M, int64_t K, int8_t* qs, float* d, int16_t* bsums,
                         qgemm_stream_t stream) {
    clear_err();
    int rc = aos_common(aos, M, K, qs, d, bsums);
    if (rc || M == 0) return rc;
    cudaError_t e = qg::launch_q8k_aos(qs, d, bsums, M, K, const_cast<void*>(aos), false,
                                       reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "Q8_K unpack launch");
    return QGEMM_OK;
}

size_t qgemm_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    if (M <= 0 || K <= 0 || K % 256) return 0;
    const size_t base = plane_bytes(M, K) + COUNTER_BYTES;
    if (N <= 0) return base;
    return base + side_bytes(N, K) + partial_bytes(plan_tc(M, N, K, sizing_sm_count()));
}

static int gemm_common_checks(const void* w, int64_t N, int64_t K, const int8_t* xqs, const float* xd,
                              const int16_t* xbsums, int64_t M, const void* y, int64_t ldy, int y_align = 4) {
    int rc = check_mk(M, K);
    if (rc) return rc;
    if (N < 1) return fail(QGEMM_EINVAL, "N must be >= 1 (got %lld)", (long long)N);
    if (N >= (int64_t(1) << 31)) return fail(QGEMM_EUNSUPPORTED, "N must be below 2^31");
    if (M == 0) return QGEMM_OK;
    if (!w) return fail(QGEMM_EINVAL, "weights pointer is null");
    if (!aligned(w, 16)) return fail(QGEMM_EALIGN, "weights must be 16-byte aligned");
    if ((rc = check_q8k(xqs, xd, xbsums))) return rc;
    if (!y) return fail(QGEMM_EINVAL, "y is null");
    if (ldy < N) return fail(QGEMM_EINVAL, "ldy (%lld) < N (%lld)", (long long)ldy, (long long)N);
    if (!aligned(y, y_align)) return fail(QGEMM_EALIGN, "y must be %d-byte aligned", y_align);
    return QGEMM_OK;
}

static int id_checks(const void* w, int64_t E, int64_t N, int64_t K, const int8_t* xqs, const float* xd,
              const int16_t* xbsums, int64_t M, const int32_t* ids, int64_t top_k, float* y, int64_t ldy) {
    int rc = gemm_common_checks(w, N, K, xqs, xd, xbsums, M, y, ldy);
    if (rc) return rc;
    if (E < 1 || E > qg::ROUTE_MAX_EXPERTS)
        return fail(QGEMM_EINVAL, "experts must be in 1..%d (got %lld)", qg::ROUTE_MAX_EXPERTS, (long long)E);
    if (top_k < 1) return fail(QGEMM_EINVAL, "top_k must be >= 1 (got %lld)", (long long)top_k);
    if (E * N >= (int64_t(1) << 31)) return fail(QGEMM_EUNSUPPORTED, "experts * N must be below 2^31");
    if (M * top_k >= (int64_t(1) << 31)) return fail(QGEMM_EUNSUPPORTED, "M * top_k must be below 2^31");
    if (M == 0) return QGEMM_OK;
    if (!ids) return fail(QGEMM_EINVAL, "ids is null");
    if (!aligned(ids, 4)) return fail(QGEMM_EALIGN, "ids must be 4-byte aligned");
    return QGEMM_OK;
}

int qgemm_q4k(const void* w, int64_t N, int64_t K, int64_t ldw, const int8_t* xqs, const float* xd,
              const int16_t* xbsums, int64_t M, float* y, int64_t ldy, void* workspace, size_t workspace_bytes,
              qgemm_stream_t stream) {
    clear_err();
    int rc = gemm_common_checks(w, N, K, xqs, xd, xbsums, M, y, ldy);
    if (rc || M == 0) return rc;
    if (ldw < (K / 256) * qg::Q4K_BLOCK) return fail(QGEMM_EINVAL, "ldw smaller than a row of Q4_K blocks");
    if (ldw % 16 != 0) return fail(QGEMM_EALIGN, "ldw must be a multiple of 16 bytes");
    if (use_small(4, M, K))
        return run_small(4, w, N, K, ldw, xqs, xd, xbsums, M, y, ldy, reinterpret_cast<cudaStream_t>(stream));
    return run_tc(4, w, N, K, ldw, xqs, xd, xbsums, M, y, ldy, workspace, workspace_bytes,
                  reinterpret_cast<cudaStream_t>(stream), false);
}

size_t qgemm_q6k_packed_bytes(int64_t N, int64_t K) {
    if (N <= 0 || K <= 0 || K % 256) return 0;
    return size_t(N) * size_t(K / 256) * qg::Q6K_PACKED;
}

int qgemm_q6k_prepack(const void* w_aos, int64_t N, int64_t K, int64_t ldw, void* w_packed, qgemm_stream_t stream) {
    clear_err();
    if (N < 1) return fail(QGEMM_EINVAL, "N must be >= 1");
    if (K < 256 || K % 256) return fail(QGEMM_EINVAL, "K must be a positive multiple of 256");
    if (!w_aos || !w_packed) return fail(QGEMM_EINVAL, "null pointer");
    if (ldw < (K / 256) * qg::Q6K_BLOCK) return fail(QGEMM_EINVAL, "ldw smaller than a row of Q6_K blocks");
    if (!aligned(w_packed, 16)) return fail(QGEMM_EALIGN, "w_packed must be 16-byte aligned");
    cudaError_t e = qg::launch_q6k_prepack(static_cast<const uint8_t*>(w_aos), N, K, ldw,
                                           static_cast<uint8_t*>(w_packed), reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "prepack launch");
    g_cnt[C_PREPACK]++;
    return QGEMM_OK;
}

int qgemm_q6k(const void* w_packed, int64_t N, int64_t K, const int8_t* xqs, const float* xd,
              const int16_t* xbsums, int64_t M, float* y, int64_t ldy, void* workspace, size_t workspace_bytes,
              qgemm_stream_t stream) {
    clear_err();
    int rc = gemm_common_checks(w_packed, N, K, xqs, xd, xbsums, M, y, ldy);
    if (rc || M == 0) return rc;
    const int64_t ldw = (K / 256) * qg::Q6K_PACKED;
    if (use_small(6, M, K))
        return run_small(6, w_packed, N, K, ldw, xqs, xd, xbsums, M, y, ldy, reinterpret_cast<cudaStream_t>(stream));
    return run_tc(6, w_packed, N, K, ldw, xqs, xd, xbsums, M, y, ldy, workspace, workspace_bytes,
                  reinterpret_cast<cudaStream_t>(stream), false);
}

static int quantize_prep_impl(const float* x, int64_t M, int64_t K, int64_t ldx, int8_t* qs, float* d, int16_t* bsums,
                              void* workspace, size_t workspace_bytes, qgemm_stream_t stream, bool dependent) {
    clear_err();
    int rc = check_mk(M, K);
    if (rc) return rc;
    if (M == 0) return QGEMM_OK;
    if (!x) return fail(QGEMM_EINVAL, "x is null");
    if (ldx < K) return fail(QGEMM_EINVAL, "ldx (%lld) < K (%lld)", (long long)ldx, (long long)K);
    if (!aligned(x, 16) || ldx % 4 != 0) return fail(QGEMM_EALIGN, "x must be 16-byte aligned with ldx % 4 == 0");
    if ((rc = check_q8k(qs, d, bsums))) return rc;
    const size_t need = plane_bytes(M, K) + COUNTER_BYTES;   // the planes and counters it writes
    if (!workspace || workspace_bytes < need)
        return fail(QGEMM_EINVAL, "workspace of %zu bytes needed (got %zu)", need,
                    workspace ? workspace_bytes : size_t(0));
    if (!aligned(workspace, 256)) return fail(QGEMM_EALIGN, "workspace must be 256-byte aligned");
    const WsPlanes wp = ws_planes(workspace, M, K);
    cudaError_t e = qg::launch_quantize_q8k(x, M, K, ldx, qs, d, bsums, reinterpret_cast<cudaStream_t>(stream), wp.xh,
                                            wp.xbs, wp.dxT, wp.Mp, wp.counters, dependent);
    if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
    g_cnt[C_QUANT]++;
    return QGEMM_OK;
}

int qgemm_quantize_q8k_prep(const float* x, int64_t M, int64_t K, int64_t ldx, int8_t* qs, float* d,
                            int16_t* bsums, void* workspace, size_t workspace_bytes, qgemm_stream_t stream) {
    return quantize_prep_impl(x, M, K, ldx, qs, d, bsums, workspace, workspace_bytes, stream, false);
}

// fp32 activations in, Y out: the fused small-M kernel for the fewest tokens,
// else the quantizer (writing the tile GEMM's operand planes for M above the
// small-M path) and the GEMM.
static int run_f32(int wtype, const void* w, int64_t N, int64_t K, int64_t ldw, const float* x, int64_t ldx,
                   int8_t* qs, float* d, int16_t* bsums, int64_t M, float* y, int64_t ldy, void* workspace,
                   size_t workspace_bytes, qgemm_stream_t stream) {
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (use_small(wtype, M, K)) {
        if (M <= qg::SMALL_FUSED_M_MAX) return run_small_fused(wtype, w, N, K, ldw, x, ldx, qs, d, bsums, M, y, ldy, st);
        const cudaError_t e = qg::launch_quantize_q8k(x, M, K, ldx, qs, d, bsums, st);
        if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
        g_cnt[C_QUANT]++;
        return run_small(wtype, w, N, K, ldw, qs, d, bsums, M, y, ldy, st);
    }
    // Q4_K: the side words first (they need only the weights), so that the GEMM
    // still starts under the quantizer
    bool side_ready = false;
    DevState* ds = nullptr;
    if (wtype == 4) {
        if (int rc = device_state(&ds)) return rc;
    }
    if (wtype == 4 && q4k_side_precomputed(plan_tc(M, N, K, ds->sm_count))) {
        const size_t need = qgemm_workspace_bytes(M, N, K);
        if (!workspace || workspace_bytes < need)
            return fail(QGEMM_EINVAL, "workspace of %zu bytes needed (got %zu)", need,
                        workspace ? workspace_bytes : size_t(0));
        if (!aligned(workspace, 256)) return fail(QGEMM_EALIGN, "workspace must be 256-byte aligned");
        const WsPlanes wp = ws_planes(workspace, M, K, N);
        const cudaError_t e = qg::launch_q4k_side(w, N, K / 256, ldw, wp.side, wp.side_e, side_np(N), st);
        if (e != cudaSuccess) return cuda_fail(e, "side-data launch");
        g_cnt[C_SIDE]++;
        side_ready = true;
    }
    int rc = quantize_prep_impl(x, M, K, ldx, qs, d, bsums, workspace, workspace_bytes, stream, side_ready);
    if (rc) return rc;
    return run_tc(wtype, w, N, K, ldw, qs, d, bsums, M, y, ldy, workspace, workspace_bytes, st, true, qg::Epi{},
                  side_ready);
}

static int f32_checks(const float* x, int64_t ldx, int64_t M, int64_t K) {
    if (M == 0) return QGEMM_OK;
    if (!x) return fail(QGEMM_EINVAL, "x is null");
    if (ldx < K) return fail(QGEMM_EINVAL, "ldx (%lld) < K (%lld)", (long long)ldx, (long long)K);
    if (!aligned(x, 16) || ldx % 4 != 0) return fail(QGEMM_EALIGN, "x must be 16-byte aligned with ldx % 4 == 0");
    return QGEMM_OK;
}

int qgemm_q4k_f32(const void* w, int64_t N, int64_t K, int64_t ldw, const float* x, int64_t ldx, int64_t M,
                  int8_t* qs, float* d, int16_t* bsums, float* y, int64_t ldy, void* workspace,
                  size_t workspace_bytes, qgemm_stream_t stream) {
    clear_err();
    int rc = gemm_common_checks(w, N, K, qs, d, bsums, M, y, ldy);
    if (rc || M == 0) return rc;
    if ((rc = f32_checks(x, ldx, M, K))) return rc;
    if (ldw < (K / 256) * qg::Q4K_BLOCK) return fail(QGEMM_EINVAL, "ldw smaller than a row of Q4_K blocks");
    if (ldw % 16 != 0) return fail(QGEMM_EALIGN, "ldw must be a multiple of 16 bytes");
    return run_f32(4, w, N, K, ldw, x, ldx, qs, d, bsums, M, y, ldy, workspace, workspace_bytes, stream);
}

int qgemm_q6k_f32(const void* w_packed, int64_t N, int64_t K, const float* x, int64_t ldx, int64_t M, int8_t* qs,
                  float* d, int16_t* bsums, float* y, int64_t ldy, void* workspace, size_t workspace_bytes,
                  qgemm_stream_t stream) {
    clear_err();
    int rc = gemm_common_checks(w_packed, N, K, qs, d, bsums, M, y, ldy);
    if (rc || M == 0) return rc;
    if ((rc = f32_checks(x, ldx, M, K))) return rc;
    const int64_t ldw = (K / 256) * qg::Q6K_PACKED;
    return run_f32(6, w_packed, N, K, ldw, x, ldx, qs, d, bsums, M, y, ldy, workspace, workspace_bytes, stream);
}

int qgemm_q4k_prepared(const void* w, int64_t N, int64_t K, int64_t ldw, const int8_t* xqs, const float* xd,
                       const int16_t* xbsums, int64_t M, float* y, int64_t ldy, const void* workspace,
                       size_t workspace_bytes, qgemm_stream_t stream) {
    clear_err();
    int rc = gemm_common_checks(w, N, K, xqs, xd, xbsums, M, y, ldy);
    if (rc || M == 0) return rc;
    if (ldw < (K / 256) * qg::Q4K_BLOCK) return fail(QGEMM_EINVAL, "ldw smaller than a row of Q4_K blocks");
    if (ldw % 16 != 0) return fail(QGEMM_EALIGN, "ldw must be a multiple of 16 bytes");
    if (use_small(4, M, K))
        return run_small(4, w, N, K, ldw, xqs, xd, xbsums, M, y, ldy, reinterpret_cast<cudaStream_t>(stream));
    return run_tc(4, w, N, K, ldw, xqs, xd, xbsums, M, y, ldy, const_cast<void*>(workspace), workspace_bytes,
                  reinterpret_cast<cudaStream_t>(stream), true);
}

int qgemm_q6k_prepared(const void* w_packed, int64_t N, int64_t K, const int8_t* xqs, const float* xd,
                       const int16_t* xbsums, int64_t M, float* y, int64_t ldy, const void* workspace,
                       size_t workspace_bytes, qgemm_stream_t stream) {
    clear_err();
    int rc = gemm_common_checks(w_packed, N, K, xqs, xd, xbsums, M, y, ldy);
    if (rc || M == 0) return rc;
    const int64_t ldw = (K / 256) * qg::Q6K_PACKED;
    if (use_small(6, M, K))
        return run_small(6, w_packed, N, K, ldw, xqs, xd, xbsums, M, y, ldy, reinterpret_cast<cudaStream_t>(stream));
    return run_tc(6, w_packed, N, K, ldw, xqs, xd, xbsums, M, y, ldy, const_cast<void*>(workspace), workspace_bytes,
                  reinterpret_cast<cudaStream_t>(stream), true);
}

// The output epilogue of the _ex calls: validated, then passed to the kernels.
static int epi_checks(const qgemm_epilogue* ep, qg::Epi* out, int* y_align) {
    *out = qg::Epi{};
    *y_align = 4;
    if (!ep) return QGEMM_OK;   // fp32, no bias, no activation
    if (ep->out_type < QGEMM_OUT_F32 || ep->out_type > QGEMM_OUT_BF16)
        return fail(QGEMM_EINVAL, "unknown out_type %d", ep->out_type);
    if (ep->activation < QGEMM_ACT_NONE || ep->activation > QGEMM_ACT_GELU)
        return fail(QGEMM_EINVAL, "unknown activation %d", ep->activation);
    if (ep->bias && !aligned(ep->bias, 4)) return fail(QGEMM_EALIGN, "bias must be 4-byte aligned");
    out->out = ep->out_type;
    out->act = ep->activation;
    out->bias = ep->bias;
    *y_align = ep->out_type == QGEMM_OUT_F32 ? 4 : 2;
    return QGEMM_OK;
}

int qgemm_q4k_ex(const void* w, int64_t N, int64_t K, int64_t ldw, const int8_t* xqs, const float* xd,
                 const int16_t* xbsums, int64_t M, void* y, int64_t ldy, const qgemm_epilogue* epilogue,
                 void* workspace, size_t workspace_bytes, qgemm_stream_t stream) {
    clear_err();
    qg::Epi epi;
    int y_align = 4;
    int rc = epi_checks(epilogue, &epi, &y_align);
    if (rc) return rc;
    rc = gemm_common_checks(w, N, K, xqs, xd, xbsums, M, y, ldy, y_align);
    if (rc || M == 0) return rc;
    if (ldw < (K / 256) * qg::Q4K_BLOCK) return fail(QGEMM_EINVAL, "ldw smaller than a row of Q4_K blocks");
    if (ldw % 16 != 0) return fail(QGEMM_EALIGN, "ldw must be a multiple of 16 bytes");
    if (use_small(4, M, K))
        return run_small(4, w, N, K, ldw, xqs, xd, xbsums, M, y, ldy, reinterpret_cast<cudaStream_t>(stream), epi);
    return run_tc(4, w, N, K, ldw, xqs, xd, xbsums, M, y, ldy, workspace, workspace_bytes,
                  reinterpret_cast<cudaStream_t>(stream), false, epi);
}

int qgemm_q6k_ex(const void* w_packed, int64_t N, int64_t K, const int8_t* xqs, const float* xd,
                 const int16_t* xbsums, int64_t M, void* y, int64_t ldy, const qgemm_epilogue* epilogue,
                 void* workspace, size_t workspace_bytes, qgemm_stream_t stream) {
    clear_err();
    qg::Epi epi;
    int y_align = 4;
    int rc = epi_checks(epilogue, &epi, &y_align);
    if (rc) return rc;
    rc = gemm_common_checks(w_packed, N, K, xqs, xd, xbsums, M, y, ldy, y_align);
    if (rc || M == 0) return rc;
    const int64_t ldw = (K / 256) * qg::Q6K_PACKED;
    if (use_small(6, M, K))
        return run_small(6, w_packed, N, K, ldw, xqs, xd, xbsums, M, y, ldy, reinterpret_cast<cudaStream_t>(stream),
                         epi);
    return run_tc(6, w_packed, N, K, ldw, xqs, xd, xbsums, M, y, ldy, workspace, workspace_bytes,
                  reinterpret_cast<cudaStream_t>(stream), false, epi);
}

int qgemm_get_counters(qgemm_counters* out) {
    if (!out) return fail(QGEMM_EINVAL, "null counters pointer");
    out->quantize = g_cnt[C_QUANT];
    out->xprep = g_cnt[C_XPREP];
    out->q4k_tc = g_cnt[C_Q4K_TC];
    out->q6k_tc = g_cnt[C_Q6K_TC];
    out->q4k_small = g_cnt[C_Q4K_SMALL];
    out->q6k_small = g_cnt[C_Q6K_SMALL];
    out->q6k_prepack = g_cnt[C_PREPACK];
    out->split_k = g_cnt[C_SPLITK];
    out->routed = g_cnt[C_ROUTED];
    out->ptq1_tc = g_cnt[C_PTQ1_TC];
    out->ptq1_prepack = g_cnt[C_PTQ1_PREPACK];
    out->small_fused = g_cnt[C_SMALL_FUSED];
    out->q4k_side = g_cnt[C_SIDE];
    return QGEMM_OK;
}

size_t qgemm_ptq1_packed_bytes(int64_t N, int64_t K) {
    if (N <= 0 || K <= 0 || K % 256) return 0;
    return size_t(N) * size_t(K / 128) * qg::PTQ1_PACKED;
}

int qgemm_ptq1_prepack(const void* w, int64_t N, int64_t K, int64_t ldw, void* w_packed, qgemm_stream_t stream) {
    clear_err();
    if (N < 1) return fail(QGEMM_EINVAL, "N must be >= 1");
    if (K < 256 || K % 256) return fail(QGEMM_EINVAL, "K must be a positive multiple of 256");
    if (!w || !w_packed) return fail(QGEMM_EINVAL, "null pointer");
    if (ldw < (K / 128) * qg::PTQ1_BLOCK) return fail(QGEMM_EINVAL, "ldw smaller than a row of PTQ1_0 blocks");
    if (!aligned(w_packed, 16)) return fail(QGEMM_EALIGN, "w_packed must be 16-byte aligned");
    cudaError_t e = qg::launch_ptq1_prepack(static_cast<const uint8_t*>(w), N, K, ldw,
                                            static_cast<uint8_t*>(w_packed), reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "prepack launch");
    g_cnt[C_PTQ1_PREPACK]++;
    return QGEMM_OK;
}

int qgemm_ptq1(const void* w_packed, int64_t N, int64_t K, const int8_t* xqs, const float* xd, const int16_t* xbsums,
               int64_t M, float* y, int64_t ldy, void* workspace, size_t workspace_bytes, qgemm_stream_t stream) {
    clear_err();
    int rc = gemm_common_checks(w_packed, N, K, xqs, xd, xbsums, M, y, ldy);
    if (rc || M == 0) return rc;
    const int64_t ldw = (K / 128) * qg::PTQ1_PACKED;
    // (every M on the tile GEMM: the small-M streaming kernel has no PTQ1_0 decode)
    return run_tc(1, w_packed, N, K, ldw, xqs, xd, xbsums, M, y, ldy, workspace, workspace_bytes,
                  reinterpret_cast<cudaStream_t>(stream), false);
}

int qgemm_ptq1_prepared(const void* w_packed, int64_t N, int64_t K, const int8_t* xqs, const float* xd,
                        const int16_t* xbsums, int64_t M, float* y, int64_t ldy, const void* workspace,
                        size_t workspace_bytes, qgemm_stream_t stream) {
    clear_err();
    int rc = gemm_common_checks(w_packed, N, K, xqs, xd, xbsums, M, y, ldy);
    if (rc || M == 0) return rc;
    const int64_t ldw = (K / 128) * qg::PTQ1_PACKED;
    return run_tc(1, w_packed, N, K, ldw, xqs, xd, xbsums, M, y, ldy, const_cast<void*>(workspace), workspace_bytes,
                  reinterpret_cast<cudaStream_t>(stream), true);
}

int qgemm_ptq1_f32(const void* w_packed, int64_t N, int64_t K, const float* x, int64_t ldx, int64_t M, int8_t* qs,
                   float* d, int16_t* bsums, float* y, int64_t ldy, void* workspace, size_t workspace_bytes,
                   qgemm_stream_t stream) {
    clear_err();
    int rc = gemm_common_checks(w_packed, N, K, qs, d, bsums, M, y, ldy);
    if (rc || M == 0) return rc;
    if ((rc = f32_checks(x, ldx, M, K))) return rc;
    const int64_t ldw = (K / 128) * qg::PTQ1_PACKED;
    // (every M on the tile GEMM: the small-M streaming kernel has no PTQ1_0 decode)
    rc = qgemm_quantize_q8k_prep(x, M, K, ldx, qs, d, bsums, workspace, workspace_bytes, stream);
    if (rc) return rc;
    return run_tc(1, w_packed, N, K, ldw, qs, d, bsums, M, y, ldy, workspace, workspace_bytes,
                  reinterpret_cast<cudaStream_t>(stream), true);
}

size_t qgemm_id_workspace_bytes(int64_t M, int64_t top_k, int64_t experts, int64_t K) {
    if (M <= 0 || top_k < 1 || experts < 1 || K <= 0 || K % 256) return 0;
    const int64_t P = M * top_k;
    return id_route_bytes(P, experts) + plane_bytes(qg::routed_rows_max(P, experts), K);
}

int qgemm_q4k_id(const void* w, int64_t experts, int64_t N, int64_t K, int64_t ldw, const int8_t* xqs,
                 const float* xd, const int16_t* xbsums, int64_t M, const int32_t* ids, int64_t top_k, float* y,
                 int64_t ldy, void* workspace, size_t workspace_bytes, qgemm_stream_t stream) {
    clear_err();
    int rc = id_checks(w, experts, N, K, xqs, xd, xbsums, M, ids, top_k, y, ldy);
    if (rc || M == 0) return rc;
    if (ldw < (K / 256) * qg::Q4K_BLOCK) return fail(QGEMM_EINVAL, "ldw smaller than a row of Q4_K blocks");
    if (ldw % 16 != 0) return fail(QGEMM_EALIGN, "ldw must be a multiple of 16 bytes");
    return run_id(4, w, experts, N, K, ldw, xqs, xd, xbsums, M, ids, top_k, y, ldy, workspace, workspace_bytes,
                  reinterpret_cast<cudaStream_t>(stream));
}

int qgemm_q6k_id(const void* w_packed, int64_t experts, int64_t N, int64_t K, const int8_t* xqs, const float* xd,
                 const int16_t* xbsums, int64_t M, const int32_t* ids, int64_t top_k, float* y, int64_t ldy,
                 void* workspace, size_t workspace_bytes, qgemm_stream_t stream) {
    clear_err();
    int rc = id_checks(w_packed, experts, N, K, xqs, xd, xbsums, M, ids, top_k, y, ldy);
    if (rc || M == 0) return rc;
    const int64_t ldw = (K / 256) * qg::Q6K_PACKED;
    return run_id(6, w_packed, experts, N, K, ldw, xqs, xd, xbsums, M, ids, top_k, y, ldy, workspace,
                  workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

int qgemm_reset_counters(void) {
    for (auto& c : g_cnt) c = 0;
    return QGEMM_OK;
}

int qgemm_get_device_status(uint32_t* bits, uint32_t* site) {
    clear_err();
    DevState* ds = nullptr;
    int rc = device_state(&ds);
    if (rc) return rc;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    uint32_t h[2] = {0, 0};
    e = cudaMemcpyFromSymbol(h, g_qgemm_status, sizeof(h));
    if (e != cudaSuccess) return cuda_fail(e, "reading device status");
    const uint32_t z[2] = {0, 0};
    e = cudaMemcpyToSymbol(g_qgemm_status, z, sizeof(z));
    if (e != cudaSuccess) return cuda_fail(e, "clearing device status");
    if (bits) *bits = h[0];
    if (site) *site = h[1];
    if (h[0] & QGEMM_DEV_TIMEOUT)
        return fail(QGEMM_ETIMEOUT, "a pipeline wait gave up (site %u); the kernel left Y unwritten", h[1]);
    if (h[0]) return fail(QGEMM_EDEVICE, "device-side value check failed (status bits %#x)", h[0]);
    return QGEMM_OK;
}

int qgemm_set_option(int option, int64_t value) {
    clear_err();
    if (option < 0 || option > QGEMM_OPT_Q4K_SIDE_MIN_TILES) return fail(QGEMM_EINVAL, "unknown option %d", option);
    if (value < 0) return fail(QGEMM_EINVAL, "option values are >= 0");
    if (option == QGEMM_OPT_FORCE_BM && value != 0 && value != 16 && value != 32 && value != 64 && value != 128)
        return fail(QGEMM_EINVAL, "FORCE_BM must be 0, 16, 32, 64 or 128");
    if (option == QGEMM_OPT_SMALL_M_MAX && value > qg::SMALL_M_LIMIT)
        return fail(QGEMM_EINVAL, "SMALL_M_MAX must be 0..%d", qg::SMALL_M_LIMIT);
    if (option == QGEMM_OPT_WAIT_LIMIT_US && value > 10000000)
        return fail(QGEMM_EINVAL, "WAIT_LIMIT_US must be 0..10000000 (10 s)");
    if (option == QGEMM_OPT_TEST_SKIP_ARRIVAL && value > 2) return fail(QGEMM_EINVAL, "TEST_SKIP_ARRIVAL must be 0..2");
    if (option == QGEMM_OPT_Q4K_SIDE_MIN_TILES && value > (int64_t(1) << 30))
        return fail(QGEMM_EINVAL, "Q4K_SIDE_MIN_TILES must be 0..2^30");
    g_opt[option] = value;
    return QGEMM_OK;
}

int64_t qgemm_get_option(int option) {
    if (option < 0 || option > QGEMM_OPT_Q4K_SIDE_MIN_TILES) return -1;
    return g_opt[option].load();
}

int qgemm_set_profile_events(qgemm_event_t before, qgemm_event_t after) {
    g_ev_before = reinterpret_cast<cudaEvent_t>(before);
    g_ev_after = reinterpret_cast<cudaEvent_t>(after);
    return QGEMM_OK;
}

}  // extern "C"
