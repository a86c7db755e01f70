// C ABI of the QSA indexer library: argument checks, workspace layout, tensor
// maps, path choice and the launch sequence.  Declarations: include/qsa.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "qsa.h"
#include "qsa_internal.h"

namespace {

using namespace qsa;

__device__ uint32_t g_device_status;   // one per device: error bits recorded by the kernels

constexpr int MAX_DEVICES = 64;
constexpr double OVERSAMPLE = 1.5;     // least expected candidates per row / k on the filter path
constexpr double SAMPLE_MARGIN = 4.5;  // standard deviations between the expected candidate count and k

struct DeviceInfo {
    bool probed = false;
    bool usable = false;
    int sms = 0;
    uint32_t *status = nullptr;
};

std::mutex g_mu;
DeviceInfo g_dev[MAX_DEVICES];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
// process-wide switches (qsa_set_config); atomics, so that a switch set on one
// host thread is read whole on another
std::atomic<int64_t> g_cfg_path{0};
std::atomic<bool> g_overlap{true};          // dependent launches inside a call (QSA_CFG_OVERLAP)
std::atomic<uint64_t> g_wait_ns{2000000000ull};
std::atomic<int> g_cluster{0};              // candidate selector CTAs per row (QSA_CFG_CLUSTER)
thread_local int32_t g_launches = 0;

// Optional per-launch CUDA-event timing (test / benchmark instrument).
enum Kind { K_PLAN = 0, K_SCORE_LOGITS, K_SCORE_SAMPLE, K_SCORE_FILTER, K_SCORE_BLOCKS,
            K_SEL_DENSE, K_SEL_THRESH, K_SEL_CAND, K_SEL_UNUSED, K_PAD, K_KINDS };
struct Pending { cudaEvent_t a, b; int kind; };
std::atomic<bool> g_timing{false};
std::vector<Pending> g_pending;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t take_event()
{
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

// Runs `launch` (returns cudaError_t as int), bracketed by events when timing.
template <typename F>
int timed(int kind, void *stream, F &&launch)
{
    if (!g_timing) return launch();
    std::lock_guard<std::mutex> lk(g_mu);
    Pending p{take_event(), take_event(), kind};
    cudaEventRecord(p.a, static_cast<cudaStream_t>(stream));
    int rc = launch();
    cudaEventRecord(p.b, static_cast<cudaStream_t>(stream));
    g_pending.push_back(p);
    return rc;
}

qsa_status from_status_bits(uint32_t bits)
{
    if (bits & ST_TIMEOUT) return QSA_ERR_TIMEOUT;
    if (bits & ST_BAD_PAGE) return QSA_ERR_BAD_PAGE;
    if (bits & ST_BAD_ROW) return QSA_ERR_INVALID_ARG;
    return QSA_OK;
}

qsa_status device_info(DeviceInfo **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
        cudaGetLastError();
        return QSA_ERR_NO_DEVICE;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo &d = g_dev[dev];
    if (!d.probed) {
        d.probed = true;
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        void *sym = nullptr;
        // the kernels are built for sm_103a only
        d.usable = (major == 10 && minor == 3) &&
                   cudaGetSymbolAddress(&sym, g_device_status) == cudaSuccess && d.sms > 0;
        d.status = static_cast<uint32_t *>(sym);
        if (d.usable && !g_encode) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q) == cudaSuccess &&
                q == cudaDriverEntryPointSuccess)
                g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        if (!g_encode) d.usable = false;
        cudaGetLastError();
    }
    if (!d.usable) return QSA_ERR_NO_DEVICE;
    *out = &d;
    return QSA_OK;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// log2 of a power of two (page sizes and the sample stride are powers of two)
int32_t log2_exact(int32_t x)
{
    int32_t l = 0;
    while ((1 << l) < x) ++l;
    return l;
}

int32_t pow2_floor(double x)
{
    int32_t p = 1;
    while (p * 2 <= x) p *= 2;
    return p;
}

// Sampled-threshold filter parameters for a top-k of k over rows of up to max_len.
//
// The threshold is the m-th largest of the scores in every stride-th key tile,
// so the number of a row's positions at or above it is about m * stride, with a
// spread of about stride * sqrt(m) (m gaps between consecutive sampled order
// statistics, each about stride positions wide).  The stride is kept at 16
// tiles or more (the sampling pass and the threshold then stay a small share
// of the step) and m is chosen so that the expected count lies SAMPLE_MARGIN
// spreads above k; the cap holds the count up to five spreads above its mean.
struct FilterShape {
    int32_t stride;     // sample every stride-th key tile
    int32_t cap;        // candidate slots per row
    int64_t sample_ld;  // columns of the sample matrix
    float oversample;   // expected candidates / k
};

FilterShape filter_shape(int64_t max_len, int32_t k)
{
    FilterShape f;
    f.stride = std::max(16, std::min(32, pow2_floor(OVERSAMPLE * k / 128.0)));
    // sampled scores at or above the threshold: the root of
    // m - k / stride = SAMPLE_MARGIN * sqrt(m)
    const double kt = static_cast<double>(k) / f.stride;
    const double x = 0.5 * (SAMPLE_MARGIN + std::sqrt(SAMPLE_MARGIN * SAMPLE_MARGIN + 4.0 * kt));
    const double m = std::max(OVERSAMPLE * kt, x * x);
    f.oversample = static_cast<float>(m / kt);
    // candidates the selector holds; a multiple of 4 so that the selector's
    // arrays after the cap-sized one stay 16-byte aligned (the selector adds 8
    // sampled scores to m)
    const int64_t k64 = k;
    const double spread = 5.0 * f.stride * std::sqrt(m + 8.0);
    const int64_t need = static_cast<int64_t>(std::ceil((m + 8.0) * f.stride + spread));
    f.cap = static_cast<int32_t>((std::max({2 * k64 + 256, k64 + 512, need}) + 3) / 4 * 4);
    const int64_t tiles = (max_len + TILE_M - 1) / TILE_M;
    f.sample_ld = std::max<int64_t>(TILE_M, (tiles + f.stride - 1) / f.stride * TILE_M);
    return f;
}

// Key tiles per row in the candidate arrays: a multiple of 8, so that every
// row's mask words fill whole 128-byte lines.
int64_t cand_tiles_ld(int64_t ld) { return ((ld + TILE_M - 1) / TILE_M + 7) / 8 * 8; }

bool use_filter(int32_t rows, int64_t max_len, int32_t k)
{
    (void)rows;
    if (g_cfg_path == 1) return false;
    if (g_cfg_path == 2) return true;
    // below k ~ 340 the dense selector is the faster one (measured)
    return OVERSAMPLE * k / 128.0 >= 4.0 && max_len >= 3LL * k;
}

struct Layout {
    size_t plan, row_vis, groups, item_prefix, sample_prefix, scores, sample, tau, flag, cand_mask;
    size_t total;
};

// Workspace regions (256-byte aligned).  `scores` holds either the dense
// logits [R, ld] (dense path) or the candidate slots [tiles_ld, R, 128] of the
// filter path (a call uses one of the two), sized for the larger; the
// score-only call needs none of it.
Layout layout(int32_t R, int64_t ld, int32_t k, bool with_scores = true)
{
    Layout L{};
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = up(o + bytes, 256); return at; };
    L.plan = take(sizeof(Plan));
    L.row_vis = take(sizeof(int32_t) * R);
    L.groups = take(sizeof(Group) * R);
    L.item_prefix = take(sizeof(int32_t) * (static_cast<size_t>(R) + 1));
    L.sample_prefix = take(sizeof(int32_t) * (static_cast<size_t>(R) + 1));
    const size_t tiles = static_cast<size_t>(cand_tiles_ld(ld));
    const size_t dense = sizeof(float) * static_cast<size_t>(R) * static_cast<size_t>(ld);
    const size_t slots = sizeof(float) * tiles * static_cast<size_t>(R) * TILE_M;
    L.scores = take(with_scores ? std::max(dense, slots) : 0);
    const FilterShape f = filter_shape(ld, std::max(k, 1));
    L.sample = take(sizeof(float) * static_cast<size_t>(R) * static_cast<size_t>(f.sample_ld));
    L.tau = take(sizeof(float) * R);
    L.flag = take(sizeof(int32_t) * R);
    L.cand_mask = take(sizeof(uint32_t) * static_cast<size_t>(R) * tiles * 4);
    L.total = o;
    return L;
}

qsa_status launch_rc(int rc)
{
    if (rc == 0) { ++g_launches; return QSA_OK; }
    return QSA_ERR_LAUNCH;
}

qsa_status make_tmap(CUtensorMap *tm, const void *base, uint64_t rows, uint32_t box_rows)
{
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(HEAD_DIM), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(HEAD_DIM * 2)};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? QSA_OK : QSA_ERR_INVALID_ARG;
}

// 3-D FP16 map with 128-byte swizzle: dims (innermost first) and byte strides
// of dims 1 and 2; boxes of {64, box1, box2}.
qsa_status make_tmap3(CUtensorMap *tm, const void *base, uint64_t d1, uint64_t d2, uint64_t s1, uint64_t s2,
                      uint32_t box1, uint32_t box2)
{
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(HEAD_DIM), static_cast<cuuint64_t>(d1), static_cast<cuuint64_t>(d2)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(s1), static_cast<cuuint64_t>(s2)};
    cuuint32_t box[3] = {64, box1, box2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? QSA_OK : QSA_ERR_INVALID_ARG;
}

bool supported_heads(int32_t H) { return H == 1 || H == 2 || H == 4 || H == 8; }

// Workspace of the block scorer: plan over the H * rows virtual rows, their
// request / token / block counts, and the block-score matrix [H * rows, max_blocks].
struct BlockLayout {
    size_t plan, vreq, vtok, vblk, row_vis, groups, item_prefix, sample_prefix, scores, total;
};

BlockLayout block_layout(int64_t RV, int64_t max_blocks)
{
    BlockLayout L{};
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = up(o + bytes, 256); return at; };
    L.plan = take(sizeof(Plan));
    L.vreq = take(sizeof(int32_t) * RV);
    L.vtok = take(sizeof(int32_t) * RV);
    L.vblk = take(sizeof(int32_t) * RV);
    L.row_vis = take(sizeof(int32_t) * RV);
    L.groups = take(sizeof(Group) * RV);
    L.item_prefix = take(sizeof(int32_t) * (RV + 1));
    L.sample_prefix = take(sizeof(int32_t) * (RV + 1));
    L.scores = take(sizeof(float) * RV * max_blocks);
    L.total = o;
    return L;
}

qsa_status check_keys(const qsa_paged_keys *keys)
{
    if (!keys || !keys->k_cache || !keys->block_table) return QSA_ERR_INVALID_ARG;
    if (keys->num_pages < 1 || keys->num_reqs < 1 || keys->max_pages_per_req < 1)
        return QSA_ERR_INVALID_ARG;
    if (keys->head_dim != HEAD_DIM) return QSA_ERR_UNSUPPORTED;
    const int32_t P = keys->page_positions;
    if (P < 8 || P > 256 || (P & (P - 1)) != 0) return QSA_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(keys->num_pages) * P >= INT32_MAX) return QSA_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(keys->max_pages_per_req) * P >= INT32_MAX) return QSA_ERR_UNSUPPORTED;
    if (!aligned(keys->k_cache, 16) || !aligned(keys->block_table, 4)) return QSA_ERR_INVALID_ARG;
    return QSA_OK;
}

// Shared prologue of the two scoring calls: plan + tensor maps.
struct ScoreSetup {
    Layout L;
    uint8_t *ws;
    CUtensorMap tq, tk, tk128;   // queries, key boxes of one page, key boxes of one tile
    ScoreParams sp;
};

// Every scorer launch follows the call's plan kernel or another kernel of
// the call, so it may overlap its predecessor.
int launch_scorer(const ScoreSetup &s, int grid, void *stream)
{
    return launch_score(s.sp, &s.tq, &s.tk, &s.tk128, grid, g_overlap, stream);
}

qsa_status setup_score(ScoreSetup &s, const void *q, const float *w, int32_t rows, int32_t H,
                       const qsa_paged_keys *keys, const int32_t *row_req, const int32_t *row_visible,
                       int64_t ld, int64_t max_len, int32_t k, int32_t sample_stride, void *ws,
                       size_t ws_bytes, DeviceInfo *d, void *stream, bool with_scores = true)
{
    s.L = layout(rows, ld, k, with_scores);
    if (!ws || ws_bytes < s.L.total) return QSA_ERR_WORKSPACE;
    if (!aligned(ws, 256)) return QSA_ERR_INVALID_ARG;
    s.ws = static_cast<uint8_t *>(ws);
    qsa_status st = make_tmap(&s.tq, q, static_cast<uint64_t>(rows) * H, N_MAX);
    if (st != QSA_OK) return st;
    st = make_tmap(&s.tk, keys->k_cache,
                   static_cast<uint64_t>(keys->num_pages) * keys->page_positions,
                   static_cast<uint32_t>(std::min(keys->page_positions, TILE_M)));
    if (st != QSA_OK) return st;
    // (with fewer than 128 cache rows no run of a whole tile exists; the map
    // is then never used and only has to be valid)
    const uint64_t cache_rows = static_cast<uint64_t>(keys->num_pages) * keys->page_positions;
    st = make_tmap(&s.tk128, keys->k_cache, cache_rows,
                   cache_rows >= TILE_M ? TILE_M : static_cast<uint32_t>(std::min(keys->page_positions, TILE_M)));
    if (st != QSA_OK) return st;
    auto at = [&](size_t off) { return s.ws + off; };
    const int32_t group_rows = N_MAX / H;
    st = launch_rc(timed(K_PLAN, stream, [&] {
        return launch_plan(row_req, row_visible, rows, group_rows, keys->num_reqs, max_len, sample_stride,
                           reinterpret_cast<int32_t *>(at(s.L.row_vis)),
                           reinterpret_cast<Group *>(at(s.L.groups)),
                           reinterpret_cast<int32_t *>(at(s.L.item_prefix)),
                           reinterpret_cast<int32_t *>(at(s.L.sample_prefix)),
                           reinterpret_cast<Plan *>(at(s.L.plan)), d->status, stream);
    }));
    if (st != QSA_OK) return st;
    ScoreParams &p = s.sp;
    std::memset(&p, 0, sizeof(p));
    p.w = w;
    p.row_vis = reinterpret_cast<const int32_t *>(at(s.L.row_vis));
    p.groups = reinterpret_cast<const Group *>(at(s.L.groups));
    p.item_prefix = reinterpret_cast<const int32_t *>(at(s.L.item_prefix));
    p.sample_prefix = reinterpret_cast<const int32_t *>(at(s.L.sample_prefix));
    p.plan = reinterpret_cast<const Plan *>(at(s.L.plan));
    p.block_table = keys->block_table;
    p.max_pages = keys->max_pages_per_req;
    p.num_pages = keys->num_pages;
    p.page_pos = keys->page_positions;
    p.page_box = std::min(keys->page_positions, TILE_M);
    p.page_pos_shift = log2_exact(keys->page_positions);
    p.page_box_shift = log2_exact(p.page_box);
    p.sample_shift = log2_exact(sample_stride);
    p.H = H;
    p.R = rows;
    p.sample_stride = sample_stride;
    p.status = d->status;
    p.wait_limit_ns = g_wait_ns;
    return QSA_OK;
}

qsa_status check_common(const void *q, const float *w, int32_t rows, int32_t H,
                        const qsa_paged_keys *keys, const int32_t *row_req,
                        const int32_t *row_visible)
{
    if (rows < 0) return QSA_ERR_INVALID_ARG;
    if (!q || !w || !row_req || !row_visible) return QSA_ERR_INVALID_ARG;
    if (!supported_heads(H)) return QSA_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(rows) * H >= INT32_MAX) return QSA_ERR_UNSUPPORTED;
    if (!aligned(q, 16)) return QSA_ERR_INVALID_ARG;
    // every int32 / float array is read element by element: 4-byte aligned
    if (!aligned(w, 4) || !aligned(row_req, 4) || !aligned(row_visible, 4)) return QSA_ERR_INVALID_ARG;
    return check_keys(keys);
}

}  // namespace

extern "C" {

size_t qsa_workspace_bytes(int32_t rows, int32_t row_capacity, int32_t k, int32_t flags)
{
    (void)flags;
    if (rows <= 0) return 256;
    const int64_t ld = std::max<int64_t>(8, (static_cast<int64_t>(std::max(row_capacity, 0)) + 7) / 8 * 8);
    return layout(rows, ld, std::max(k, 1), row_capacity > 1 || k > 1).total;
}

const char *qsa_status_string(qsa_status s)
{
    switch (s) {
    case QSA_OK: return "ok";
    case QSA_ERR_INVALID_ARG: return "invalid argument";
    case QSA_ERR_UNSUPPORTED: return "unsupported shape";
    case QSA_ERR_WORKSPACE: return "workspace missing or too small";
    case QSA_ERR_LAUNCH: return "kernel launch failed";
    case QSA_ERR_BAD_PAGE: return "block table holds a page id outside the key cache";
    case QSA_ERR_TIMEOUT: return "a device pipeline wait timed out";
    case QSA_ERR_CUDA: return "CUDA runtime error";
    case QSA_ERR_NO_DEVICE: return "no usable sm_103 device";
    case QSA_ERR_STATIC_LIMIT: return "call needs more scratch than the library's static buffer (QSA_STATIC_SCRATCH_BYTES)";
    }
    return "unknown status";
}

qsa_status qsa_set_config(int32_t key, int64_t value)
{
    if (key == QSA_CFG_PATH) {
        if (value < 0 || value > 2) return QSA_ERR_INVALID_ARG;
        g_cfg_path = value;
        return QSA_OK;
    }
    if (key == QSA_CFG_KERNEL_TIMING) {
        if (value < 0 || value > 1) return QSA_ERR_INVALID_ARG;
        g_timing = value != 0;
        return QSA_OK;
    }
    if (key == QSA_CFG_OVERLAP) {
        if (value < 0 || value > 1) return QSA_ERR_INVALID_ARG;
        g_overlap = value != 0;
        return QSA_OK;
    }
    if (key == QSA_CFG_CLUSTER) {
        if (!(value == 0 || value == 1 || value == 2 || value == 4 || value == 8)) return QSA_ERR_INVALID_ARG;
        g_cluster = static_cast<int>(value);
        return QSA_OK;
    }
    if (key == QSA_CFG_WAIT_LIMIT_NS) {
        if (value <= 0) return QSA_ERR_INVALID_ARG;
        g_wait_ns = static_cast<uint64_t>(value);
        return QSA_OK;
    }
    return QSA_ERR_INVALID_ARG;
}

int32_t qsa_last_launch_count(void) { return g_launches; }

int32_t qsa_last_cluster_size(void) { return qsa::last_cluster; }

qsa_status qsa_sparse_attention(const void *q, int32_t rows, int32_t hq, const void *k_cache, const void *v_cache,
                                int32_t num_pages, int32_t page_tokens, int32_t hkv, int32_t head_dim,
                                const int32_t *block_table, int32_t num_reqs, int32_t max_pages,
                                const int32_t *row_req, const int32_t *row_token, const int32_t *sel, int32_t k,
                                float scale, float *out, void *stream)
{
    g_launches = 0;
    if (rows < 0 || k < 0 || hq < 1 || hkv < 1 || num_pages < 1 || num_reqs < 1 || max_pages < 1)
        return QSA_ERR_INVALID_ARG;
    if (head_dim != 256 || hq % hkv != 0 || hq / hkv > 16 || hkv > 65535) return QSA_ERR_UNSUPPORTED;
    if (page_tokens < 8 || page_tokens > 256 || (page_tokens & (page_tokens - 1))) return QSA_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(max_pages) * page_tokens >= INT32_MAX ||
        static_cast<int64_t>(num_pages) * page_tokens * hkv * 256 >= (int64_t{1} << 62))
        return QSA_ERR_UNSUPPORTED;
    if (!(scale > 0.0f) || !std::isfinite(scale)) return QSA_ERR_INVALID_ARG;
    if (rows == 0) return QSA_OK;
    if (!q || !k_cache || !v_cache || !block_table || !row_req || !row_token || !out || (k > 0 && !sel))
        return QSA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16))
        return QSA_ERR_INVALID_ARG;
    if (!aligned(block_table, 4) || !aligned(row_req, 4) || !aligned(row_token, 4) || !aligned(sel, 4))
        return QSA_ERR_INVALID_ARG;
    DeviceInfo *d = nullptr;
    qsa_status st = device_info(&d);
    if (st != QSA_OK) return st;
    AttendParams p;
    std::memset(&p, 0, sizeof(p));
    p.q = q;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_table = block_table;
    p.row_req = row_req;
    p.row_token = row_token;
    p.sel = sel;
    p.out = out;
    p.rows = rows;
    p.hq = hq;
    p.hkv = hkv;
    p.k = k;
    p.num_pages = num_pages;
    p.page_tokens = page_tokens;
    p.page_shift = log2_exact(page_tokens);
    p.num_reqs = num_reqs;
    p.max_pages = max_pages;
    p.scale = scale;
    p.status = d->status;
    p.wait_limit_ns = g_wait_ns;
    return launch_rc(launch_attend(p, stream));
}

qsa_status qsa_rope_table(float *table, int32_t n_blocks, int32_t rope_dim, double theta, void *stream)
{
    g_launches = 0;
    if (n_blocks < 0 || rope_dim < 0 || rope_dim > HEAD_DIM || (rope_dim & 7)) return QSA_ERR_INVALID_ARG;
    if (!(theta > 0.0) || !std::isfinite(theta)) return QSA_ERR_INVALID_ARG;
    if (n_blocks == 0 || rope_dim == 0) return QSA_OK;
    if (!table || !aligned(table, 16)) return QSA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(n_blocks) * rope_dim >= INT32_MAX) return QSA_ERR_UNSUPPORTED;
    DeviceInfo *d = nullptr;
    qsa_status st = device_info(&d);
    if (st != QSA_OK) return st;
    return launch_rc(launch_rope_table(table, n_blocks, rope_dim, theta, stream));
}

qsa_status qsa_index_key_produce(const void *x, const float *pool_logit, int32_t n_reqs,
                                 const int32_t *seq_start, const int32_t *pos_start, int32_t max_tokens,
                                 const float *norm_weight, float eps, const float *rope_table,
                                 int32_t rope_blocks, int32_t rope_dim, int32_t window,
                                 const qsa_paged_keys *keys, void *stream)
{
    g_launches = 0;
    if (n_reqs < 0 || max_tokens < 0 || rope_blocks < 0) return QSA_ERR_INVALID_ARG;
    if (window != 4 && window != 8) return QSA_ERR_UNSUPPORTED;
    if (rope_dim < 0 || rope_dim > HEAD_DIM || (rope_dim & 7)) return QSA_ERR_INVALID_ARG;
    if (!(eps >= 0.0f) || !std::isfinite(eps)) return QSA_ERR_INVALID_ARG;
    qsa_status st = check_keys(keys);
    if (st != QSA_OK) return st;
    if (n_reqs == 0 || max_tokens == 0) return QSA_OK;
    if (n_reqs > keys->num_reqs || n_reqs > 65535) return QSA_ERR_UNSUPPORTED;
    if (!x || !seq_start || !pos_start || !norm_weight) return QSA_ERR_INVALID_ARG;
    if (!aligned(x, 8) || !aligned(norm_weight, 16)) return QSA_ERR_INVALID_ARG;
    if (!aligned(pool_logit, 4) || !aligned(seq_start, 4) || !aligned(pos_start, 4)) return QSA_ERR_INVALID_ARG;
    if (rope_dim > 0 && (!rope_table || !aligned(rope_table, 16))) return QSA_ERR_INVALID_ARG;
    DeviceInfo *d = nullptr;
    if ((st = device_info(&d)) != QSA_OK) return st;
    ProduceParams p;
    std::memset(&p, 0, sizeof(p));
    p.x = x;
    p.pool_logit = pool_logit;
    p.seq_start = seq_start;
    p.pos_start = pos_start;
    p.norm_weight = norm_weight;
    p.rope_table = rope_table;
    p.k_cache = const_cast<void *>(keys->k_cache);
    p.block_table = keys->block_table;
    p.n_reqs = n_reqs;
    p.num_pages = keys->num_pages;
    p.page_positions = keys->page_positions;
    p.page_shift = log2_exact(keys->page_positions);
    p.max_pages = keys->max_pages_per_req;
    p.rope_dim = rope_dim;
    p.rope_blocks = rope_dim > 0 ? rope_blocks : INT32_MAX;
    p.window = window;
    p.eps = eps;
    p.status = d->status;
    return launch_rc(launch_produce(p, max_tokens, stream));
}

qsa_status qsa_kernel_times(double *ms, int32_t *launches, int32_t n)
{
    std::lock_guard<std::mutex> lk(g_mu);
    qsa_status st = QSA_OK;
    for (const Pending &p : g_pending) {
        float t = 0.f;
        if (cudaEventSynchronize(p.b) != cudaSuccess || cudaEventElapsedTime(&t, p.a, p.b) != cudaSuccess) {
            cudaGetLastError();
            st = QSA_ERR_CUDA;
        } else if (p.kind < n) {
            if (ms) ms[p.kind] += t;
            if (launches) launches[p.kind] += 1;
        }
        g_event_pool.push_back(p.a);
        g_event_pool.push_back(p.b);
    }
    g_pending.clear();
    return st;
}

qsa_status qsa_get_device_status(void *stream)
{
    DeviceInfo *d = nullptr;
    qsa_status st = device_info(&d);
    if (st != QSA_OK) return st;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return QSA_ERR_CUDA;
    }
    uint32_t bits = 0;
    const uint32_t zero = 0;
    if (cudaMemcpy(&bits, d->status, sizeof(bits), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(d->status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaGetLastError();
        return QSA_ERR_CUDA;
    }
    return from_status_bits(bits);
}

qsa_status qsa_index_score(const void *q, const float *w, int32_t rows, int32_t H,
                           const qsa_paged_keys *keys, const int32_t *row_req,
                           const int32_t *row_visible, float *logits, int64_t ld_logits,
                           void *ws, size_t ws_bytes, void *stream)
{
    g_launches = 0;
    qsa_status st = check_common(q, w, rows, H, keys, row_req, row_visible);
    if (st != QSA_OK) return st;
    if (!logits || ld_logits < 1 || !aligned(logits, 4)) return QSA_ERR_INVALID_ARG;
    if (rows == 0) return QSA_OK;
    DeviceInfo *d = nullptr;
    if ((st = device_info(&d)) != QSA_OK) return st;
    const int64_t max_len = std::min<int64_t>(ld_logits,
        static_cast<int64_t>(keys->max_pages_per_req) * keys->page_positions);
    ScoreSetup s;
    // the score-only call needs no logits scratch: size the layout for one column
    st = setup_score(s, q, w, rows, H, keys, row_req, row_visible, 1, max_len, 1, 1, ws,
                     ws_bytes, d, stream, false);
    if (st != QSA_OK) return st;
    s.sp.mode = SCORE_LOGITS;
    s.sp.out = logits;
    s.sp.ld = ld_logits;
    s.sp.pad_inf = 1;
    st = launch_rc(timed(K_SCORE_LOGITS, stream, [&] { return launch_scorer(s, d->sms, stream); }));
    if (st != QSA_OK) return st;
    return launch_rc(timed(K_PAD, stream, [&] {
        return launch_pad(logits, ld_logits, rows,
                          reinterpret_cast<const int32_t *>(s.ws + s.L.row_vis), g_overlap, stream);
    }));
}

qsa_status qsa_topk_exact(const float *logits, int64_t ld_logits, int32_t rows,
                          const int32_t *row_visible, int32_t k, int32_t *out_idx,
                          float *out_val, void *ws, size_t ws_bytes, void *stream)
{
    (void)ws;
    (void)ws_bytes;
    g_launches = 0;
    if (rows < 0 || k < 0 || ld_logits < 1) return QSA_ERR_INVALID_ARG;
    if (k > QSA_MAX_K) return QSA_ERR_UNSUPPORTED;
    if (rows == 0 || k == 0) return QSA_OK;
    if (!logits || !row_visible || !out_idx) return QSA_ERR_INVALID_ARG;
    if (!aligned(logits, 4) || !aligned(row_visible, 4) || !aligned(out_idx, 4) || !aligned(out_val, 4))
        return QSA_ERR_INVALID_ARG;
    if (ld_logits > INT32_MAX) return QSA_ERR_UNSUPPORTED;
    DeviceInfo *d = nullptr;
    qsa_status st = device_info(&d);
    if (st != QSA_OK) return st;
    SelectParams p;
    std::memset(&p, 0, sizeof(p));
    p.mode = SEL_DENSE;
    p.R = rows;
    p.k = k;
    p.logits = logits;
    p.ld = ld_logits;
    p.max_len = ld_logits;
    p.row_vis = row_visible;
    p.out_idx = out_idx;
    p.out_val = out_val;
    p.smem_cap = std::max(8192, k);
    p.status = d->status;
    // the call's only kernel: ordered after the caller's work as usual
    return launch_rc(timed(K_SEL_DENSE, stream, [&] { return launch_select(p, rows, false, stream); }));
}

qsa_status qsa_select_paged_tokens(const void *q, const float *w, int32_t rows, int32_t H,
                                   const qsa_paged_keys *keys, const int32_t *row_req,
                                   const int32_t *row_visible, int32_t k, int32_t *out_idx,
                                   float *out_val, void *ws, size_t ws_bytes, void *stream)
{
    g_launches = 0;
    qsa_status st = check_common(q, w, rows, H, keys, row_req, row_visible);
    if (st != QSA_OK) return st;
    if (k < 0) return QSA_ERR_INVALID_ARG;
    if (k > QSA_MAX_K) return QSA_ERR_UNSUPPORTED;
    if (!out_idx) return QSA_ERR_INVALID_ARG;
    if (!aligned(out_idx, 4) || !aligned(out_val, 4)) return QSA_ERR_INVALID_ARG;
    if (rows == 0 || k == 0) return QSA_OK;
    DeviceInfo *d = nullptr;
    if ((st = device_info(&d)) != QSA_OK) return st;
    const int64_t ld = static_cast<int64_t>(keys->max_pages_per_req) * keys->page_positions;
    const bool filter = use_filter(rows, ld, k);
    const FilterShape f = filter_shape(ld, k);
    ScoreSetup s;
    st = setup_score(s, q, w, rows, H, keys, row_req, row_visible, ld, ld, k,
                     filter ? f.stride : 1, ws, ws_bytes, d, stream);
    if (st != QSA_OK) return st;
    auto at = [&](size_t off) { return s.ws + off; };
    float *logits = reinterpret_cast<float *>(at(s.L.scores));

    SelectParams sel;
    std::memset(&sel, 0, sizeof(sel));
    sel.R = rows;
    sel.k = k;
    sel.max_len = ld;
    sel.row_vis = reinterpret_cast<const int32_t *>(at(s.L.row_vis));
    sel.plan = reinterpret_cast<Plan *>(at(s.L.plan));
    sel.out_idx = out_idx;
    sel.out_val = out_val;
    sel.status = d->status;
    sel.row_flag = reinterpret_cast<int32_t *>(at(s.L.flag));

    if (!filter) {
        s.sp.mode = SCORE_LOGITS;
        s.sp.out = logits;
        s.sp.ld = ld;
        if ((st = launch_rc(timed(K_SCORE_LOGITS, stream, [&] { return launch_scorer(s, d->sms, stream); }))) != QSA_OK) return st;
        sel.mode = SEL_DENSE;
        sel.logits = logits;
        sel.ld = ld;
        sel.smem_cap = std::max(8192, k);
        return launch_rc(timed(K_SEL_DENSE, stream, [&] { return launch_select(sel, rows, g_overlap, stream); }));
    }

    float *sample = reinterpret_cast<float *>(at(s.L.sample));
    float *tau = reinterpret_cast<float *>(at(s.L.tau));
    uint32_t *cand_mask = reinterpret_cast<uint32_t *>(at(s.L.cand_mask));
    float *cand_score = logits;                     // the same region, laid out by (tile, row)
    const int32_t tiles_ld = static_cast<int32_t>(cand_tiles_ld(ld));

    // 1. scores of every stride-th key tile
    s.sp.mode = SCORE_SAMPLE;
    s.sp.out = sample;
    s.sp.ld = f.sample_ld;
    if ((st = launch_rc(timed(K_SCORE_SAMPLE, stream, [&] { return launch_scorer(s, d->sms, stream); }))) != QSA_OK) return st;
    // 2. per-row threshold tau_r: a sample quantile that keeps ~oversample * k positions
    SelectParams th = sel;
    th.mode = SEL_THRESH;
    th.logits = sample;
    th.ld = f.sample_ld;
    th.cap = f.cap;
    th.sample_stride = f.stride;
    th.tau = tau;
    th.oversample = f.oversample;
    th.smem_cap = static_cast<int32_t>(std::min<int64_t>(f.sample_ld, TH_STAGE));   // staged scores per row
    if ((st = launch_rc(timed(K_SEL_THRESH, stream, [&] { return launch_select(th, rows, g_overlap, stream); }))) != QSA_OK) return st;
    // 3. full scoring pass keeping only scores >= tau_r
    s.sp.mode = SCORE_FILTER;
    s.sp.tau = tau;
    s.sp.cand_score = cand_score;
    s.sp.cand_mask = cand_mask;
    s.sp.tiles_ld = tiles_ld;
    if ((st = launch_rc(timed(K_SCORE_FILTER, stream, [&] { return launch_scorer(s, d->sms, stream); }))) != QSA_OK) return st;
    // 4. exact top-k of each candidate list; a row whose list cannot be
    //    trusted (fewer than min(k, V) candidates, more than the selector
    //    holds, or a tie bucket at the cut too large to order there) is
    //    re-scored in plain FP32 by its CTA and selected densely
    SelectParams cs = sel;
    cs.mode = SEL_CAND;
    cs.cand_score = cand_score;
    cs.cand_mask = cand_mask;
    cs.tiles_ld = tiles_ld;
    cs.cap = f.cap;
    cs.logits = logits;
    cs.ld = ld;
    cs.q = static_cast<const uint16_t *>(q);
    cs.w = w;
    cs.k_cache = static_cast<const uint16_t *>(keys->k_cache);
    cs.block_table = keys->block_table;
    cs.row_req = row_req;
    cs.H = H;
    cs.max_pages = keys->max_pages_per_req;
    cs.num_pages = keys->num_pages;
    cs.page_pos = keys->page_positions;
    cs.fb_scores = cand_score;
    return launch_rc(timed(K_SEL_CAND, stream, [&] { return launch_select(cs, rows, g_overlap, stream, g_cluster); }));
}

size_t qsa_block_select_workspace_bytes(int32_t rows, int32_t H, int32_t max_blocks, int32_t k)
{
    (void)k;
    if (rows <= 0 || H <= 0) return 256;
    return block_layout(static_cast<int64_t>(rows) * H, std::max(max_blocks, 1)).total;
}

qsa_status qsa_block_select(const void *q, int32_t rows, int32_t H, const void *k_cache, int32_t num_pages,
                            const int32_t *block_table, int32_t num_reqs, int32_t max_blocks,
                            const int32_t *row_req, const int32_t *row_token, int32_t k, int32_t *out_idx,
                            float *out_val, void *ws, size_t ws_bytes, void *stream)
{
    g_launches = 0;
    if (rows < 0 || k < 0 || H < 1 || num_pages < 1 || num_reqs < 1 || max_blocks < 1) return QSA_ERR_INVALID_ARG;
    if (k > QSA_MAX_K || H > 16) return QSA_ERR_UNSUPPORTED;
    const int64_t RV = static_cast<int64_t>(rows) * H;
    if (RV >= INT32_MAX || static_cast<int64_t>(num_reqs) * H >= INT32_MAX ||
        static_cast<int64_t>(max_blocks) * TILE_M >= INT32_MAX || static_cast<int64_t>(num_pages) * TILE_M >= INT32_MAX)
        return QSA_ERR_UNSUPPORTED;
    if (rows == 0 || k == 0) return QSA_OK;
    if (!q || !k_cache || !block_table || !row_req || !row_token || !out_idx) return QSA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_cache, 16)) return QSA_ERR_INVALID_ARG;
    if (!aligned(block_table, 4) || !aligned(row_req, 4) || !aligned(row_token, 4) || !aligned(out_idx, 4) ||
        !aligned(out_val, 4))
        return QSA_ERR_INVALID_ARG;
    DeviceInfo *d = nullptr;
    qsa_status st = device_info(&d);
    if (st != QSA_OK) return st;
    const BlockLayout L = block_layout(RV, max_blocks);
    if (!ws || ws_bytes < L.total) return QSA_ERR_WORKSPACE;
    if (!aligned(ws, 256)) return QSA_ERR_INVALID_ARG;
    uint8_t *w8 = static_cast<uint8_t *>(ws);
    auto i32 = [&](size_t off) { return reinterpret_cast<int32_t *>(w8 + off); };
    // queries [rows][H][128], boxes of one head x BR_ROWS rows; keys [pages *
    // 128 tokens][H][128], boxes of one head x 128 tokens (strides increase
    // with the dimension in both maps)
    CUtensorMap tq, tk;
    if ((st = make_tmap3(&tq, q, static_cast<uint64_t>(H), static_cast<uint64_t>(rows), HEAD_DIM * 2,
                         static_cast<uint64_t>(H) * HEAD_DIM * 2, 1, BR_ROWS)) != QSA_OK)
        return st;
    if ((st = make_tmap3(&tk, k_cache, static_cast<uint64_t>(H), static_cast<uint64_t>(num_pages) * TILE_M,
                         HEAD_DIM * 2, static_cast<uint64_t>(H) * HEAD_DIM * 2, 1, TILE_M)) != QSA_OK)
        return st;
    const int32_t RVi = static_cast<int32_t>(RV);
    if ((st = launch_rc(launch_block_rows(row_req, row_token, rows, H, num_reqs, i32(L.vreq), i32(L.vtok),
                                          i32(L.vblk), d->status, stream))) != QSA_OK)
        return st;
    if ((st = launch_rc(timed(K_PLAN, stream, [&] {
             // groups of BR_ROWS virtual rows of one head, tiles of two 128-token blocks
             return launch_plan(i32(L.vreq), i32(L.vtok), RVi, BR_ROWS, num_reqs * H,
                                static_cast<int64_t>(max_blocks) * TILE_M, 1, i32(L.row_vis),
                                reinterpret_cast<Group *>(w8 + L.groups), i32(L.item_prefix), i32(L.sample_prefix),
                                reinterpret_cast<Plan *>(w8 + L.plan), d->status, stream, 8);
         }))) != QSA_OK)
        return st;
    ScoreParams sp;
    std::memset(&sp, 0, sizeof(sp));
    sp.row_vis = i32(L.row_vis);
    sp.groups = reinterpret_cast<const Group *>(w8 + L.groups);
    sp.item_prefix = i32(L.item_prefix);
    sp.sample_prefix = i32(L.sample_prefix);
    sp.plan = reinterpret_cast<const Plan *>(w8 + L.plan);
    sp.block_table = block_table;
    sp.max_pages = max_blocks;
    sp.num_pages = num_pages;
    sp.page_pos = TILE_M;
    sp.page_box = TILE_M;
    sp.page_pos_shift = log2_exact(TILE_M);
    sp.page_box_shift = sp.page_pos_shift;
    sp.H = 1;
    sp.R = RVi;
    sp.mode = SCORE_BLOCKMAX;
    sp.sample_stride = 1;
    sp.out = reinterpret_cast<float *>(w8 + L.scores);
    sp.ld = max_blocks;
    sp.status = d->status;
    sp.wait_limit_ns = g_wait_ns;
    sp.blk_heads = H;
    sp.blk_reqs = num_reqs;
    sp.blk_rows = rows;
    if ((st = launch_rc(timed(K_SCORE_BLOCKS, stream, [&] {
             return launch_score_blockrows(sp, &tq, &tk, d->sms, g_overlap, stream);
         }))) != QSA_OK)
        return st;
    SelectParams sel;
    std::memset(&sel, 0, sizeof(sel));
    sel.mode = SEL_DENSE;
    sel.R = RVi;
    sel.k = k;
    sel.logits = reinterpret_cast<const float *>(w8 + L.scores);
    sel.ld = max_blocks;
    sel.max_len = max_blocks;
    sel.row_vis = i32(L.vblk);
    sel.out_idx = out_idx;
    sel.out_val = out_val;
    sel.smem_cap = std::max(8192, k);
    sel.status = d->status;
    sel.out_heads = H;
    return launch_rc(timed(K_SEL_DENSE, stream, [&] { return launch_select(sel, RVi, g_overlap, stream); }));
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free variant: the workspace is a buffer inside the library.

namespace {

static __device__ __align__(256) uint8_t g_static_scratch[QSA_STATIC_SCRATCH_BYTES];

struct StaticScratch {
    bool ready = false;
    void *ptr = nullptr;
};
StaticScratch g_static[MAX_DEVICES];

}  // namespace

extern "C" qsa_status qsa_select_paged_tokens_noalloc(const void *q, const float *w, int32_t rows,
                                                      int32_t H, const qsa_paged_keys *keys,
                                                      const int32_t *row_req,
                                                      const int32_t *row_visible, int32_t k,
                                                      int32_t *out_idx, float *out_val, void *stream)
{
    g_launches = 0;
    if (!keys || keys->max_pages_per_req < 1 || keys->page_positions < 1 || rows < 0 || k < 0)
        return QSA_ERR_INVALID_ARG;
    if (k > QSA_MAX_K) return QSA_ERR_UNSUPPORTED;
    const int64_t ld = static_cast<int64_t>(keys->max_pages_per_req) * keys->page_positions;
    if (ld > INT32_MAX) return QSA_ERR_UNSUPPORTED;
    const size_t need = qsa_workspace_bytes(rows, static_cast<int32_t>(ld), k, 0);
    if (need > QSA_STATIC_SCRATCH_BYTES) return QSA_ERR_STATIC_LIMIT;
    // the same device check as every other entry point, before the symbol lookup
    DeviceInfo *info = nullptr;
    qsa_status dst = device_info(&info);
    if (dst != QSA_OK) return dst;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
        cudaGetLastError();
        return QSA_ERR_NO_DEVICE;
    }
    {
        std::lock_guard<std::mutex> lk(g_mu);
        StaticScratch &st = g_static[dev];
        if (!st.ready) {
            // In host code g_static_scratch names a host-side stand-in; the
            // kernels need this device's address of the buffer.
            void *ptr = nullptr;
            if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || !ptr) {
                cudaGetLastError();
                return QSA_ERR_CUDA;
            }
            st.ptr = ptr;
            st.ready = true;
        }
    }
    return qsa_select_paged_tokens(q, w, rows, H, keys, row_req, row_visible, k, out_idx, out_val,
                                   g_static[dev].ptr, QSA_STATIC_SCRATCH_BYTES, stream);
}
