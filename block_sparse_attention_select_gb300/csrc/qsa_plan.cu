// Plan kernel: sanitises the per-row metadata and splits the query rows into
// groups (consecutive rows of one request, at most 256 / H rows, so that one
// group is the N side of one tensor-core tile), then lays the (group, key tile)
// work items out for the persistent scorer.
#include <cuda_runtime.h>

#include <algorithm>

#include "qsa_device.cuh"
#include "qsa_internal.h"

namespace qsa {
namespace {

constexpr int PLAN_THREADS = 1024;
constexpr int PLAN_SMEM_ROWS = 4096;    // rows whose sanitised V stays in shared memory
constexpr int PLAN_SMEM_GROUPS = 1024;  // groups whose first row / length bound stay there

template <typename Op>
__device__ int32_t block_incl_scan(int32_t v, int32_t *wbuf, Op op, int32_t ident)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x = op(x, y);
    }
    if (lane == 31) wbuf[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int32_t t = wbuf[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int32_t y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t = op(t, y);
        }
        wbuf[lane] = t;
    }
    __syncthreads();
    int32_t r = wid > 0 ? op(wbuf[wid - 1], x) : x;
    __syncthreads();
    (void)ident;
    return r;
}

struct OpMax { __device__ int32_t operator()(int32_t a, int32_t b) const { return a > b ? a : b; } };
struct OpAdd { __device__ int32_t operator()(int32_t a, int32_t b) const { return a + b; } };

__global__ void __launch_bounds__(PLAN_THREADS)
plan_kernel(const int32_t *__restrict__ row_req, const int32_t *__restrict__ row_visible,
            int32_t R, int32_t G, int32_t num_reqs, int64_t max_len, int32_t sample_stride, int32_t tile_shift,
            int32_t *__restrict__ row_vis, Group *__restrict__ groups,
            int32_t *__restrict__ item_prefix, int32_t *__restrict__ sample_prefix,
            Plan *__restrict__ plan, uint32_t *status)
{
    __shared__ int32_t wbuf[32];
    __shared__ int32_t s_req[PLAN_THREADS];
    __shared__ int32_t s_vis[PLAN_SMEM_ROWS];     // row_vis of rows < PLAN_SMEM_ROWS
    __shared__ int32_t s_row0[PLAN_SMEM_GROUPS];  // first row of groups < PLAN_SMEM_GROUPS
    __shared__ int32_t s_vmax[PLAN_SMEM_GROUPS];
    __shared__ int32_t carry_req, carry_run, carry_gid, carry_items, carry_samples;
    const int tid = threadIdx.x;
    wait_prior_grid();
    allow_next_grid();
    if (tid == 0) { carry_req = -2; carry_run = 0; carry_gid = 0; }
    __syncthreads();

    // Phase 1: sanitise rows, find group starts.  A thread takes RPT
    // consecutive rows per round (a run of rows of one request starts where
    // the request changes, a group every G rows of a run); its rows of the
    // next round are loaded while this round is scanned.
    constexpr int RPT = 4;
    constexpr int32_t ROUND = PLAN_THREADS * RPT;
    int32_t nx_req[RPT], nx_vis[RPT];
#pragma unroll
    for (int q = 0; q < RPT; ++q) {
        const int32_t r = tid * RPT + q;
        nx_req[q] = r < R ? row_req[r] : 0;
        nx_vis[q] = r < R ? row_visible[r] : 0;
    }
    for (int32_t base = 0; base < R; base += ROUND) {
        const int32_t r0 = base + tid * RPT;       // this thread's first row
        int32_t req[RPT];
        int64_t vv[RPT];
#pragma unroll
        for (int q = 0; q < RPT; ++q) {
            req[q] = nx_req[q];
            vv[q] = nx_vis[q];
            const int32_t rn = r0 + ROUND + q;
            if (rn < R) { nx_req[q] = row_req[rn]; nx_vis[q] = row_visible[rn]; }
        }
#pragma unroll
        for (int q = 0; q < RPT; ++q) {
            const int32_t r = r0 + q;
            if (r < R) {
                int32_t b = req[q];
                int64_t v = vv[q];
                bool bad = false;
                if (b < 0 || b >= num_reqs) { b = -1; v = 0; bad = true; }
                if (v < 0) { v = 0; bad = true; }
                if (v > max_len) { v = max_len; bad = true; }
                if (bad) record_error(status, ST_BAD_ROW);
                row_vis[r] = static_cast<int32_t>(v);
                if (r < PLAN_SMEM_ROWS) s_vis[r] = static_cast<int32_t>(v);
                req[q] = b;
            } else {
                req[q] = -1;
            }
        }
        s_req[tid] = req[RPT - 1];
        __syncthreads();
        int32_t prev = tid > 0 ? s_req[tid - 1] : carry_req;
        uint32_t beg = 0;                          // bit q: row r0 + q starts a run
        int32_t run_last = -1;                     // this thread's latest run start
#pragma unroll
        for (int q = 0; q < RPT; ++q) {
            const int32_t r = r0 + q;
            if (r < R && (r == 0 || req[q] != prev)) {
                beg |= 1u << q;
                run_last = r;
            }
            prev = req[q];
        }
        // the run start in effect before this thread's rows: the latest one
        // of the threads before it, else the previous round's
        const int32_t run_incl = block_incl_scan(run_last, wbuf, OpMax(), -1);
        s_req[tid] = run_incl;                     // every read of s_req above is done (the scan's barriers)
        __syncthreads();
        int32_t rs = tid > 0 ? s_req[tid - 1] : -1;
        if (rs < 0) rs = carry_run;
        uint32_t gb = 0;                           // bit q: row r0 + q starts a group
        int32_t gcnt = 0, rq = rs;
#pragma unroll
        for (int q = 0; q < RPT; ++q) {
            const int32_t r = r0 + q;
            if (beg & (1u << q)) rq = r;
            if (r < R && (r - rq) % G == 0) {
                gb |= 1u << q;
                ++gcnt;
            }
        }
        const int32_t g_incl = block_incl_scan(gcnt, wbuf, OpAdd(), 0);
        int32_t gid = carry_gid + g_incl - gcnt;
#pragma unroll
        for (int q = 0; q < RPT; ++q) {
            if (gb & (1u << q)) {
                const int32_t r = r0 + q;
                groups[gid].row0 = r;
                groups[gid].req = req[q];
                if (gid < PLAN_SMEM_GROUPS) s_row0[gid] = r;
                ++gid;
            }
        }
        __syncthreads();
        // carries from the thread holding the round's last row
        const int32_t last = min(R, base + ROUND) - 1;
        if (tid == (last - base) / RPT) {
            const int ql = (last - base) % RPT;
            int32_t rl = rs, cr = req[0];
#pragma unroll
            for (int q = 0; q < RPT; ++q) {
                if (q <= ql && (beg & (1u << q))) rl = r0 + q;
                if (q == ql) cr = req[q];
            }
            carry_req = cr;
            carry_run = rl;
            carry_gid = gid;
        }
        __syncthreads();
    }
    const int32_t n_groups = carry_gid;

    // Phase 2: rows and longest / shortest visible length of each group, one
    // warp per group.
    {
        const int wid = tid >> 5, lane = tid & 31;
        for (int32_t g = wid; g < n_groups; g += PLAN_THREADS / 32) {
            const int32_t r0 = g < PLAN_SMEM_GROUPS ? s_row0[g] : groups[g].row0;
            const int32_t r1 = g + 1 < n_groups ? (g + 1 < PLAN_SMEM_GROUPS ? s_row0[g + 1] : groups[g + 1].row0) : R;
            int32_t vmax = 0, vmin = INT32_MAX;
            for (int32_t r = r0 + lane; r < r1; r += 32) {
                const int32_t v = r < PLAN_SMEM_ROWS ? s_vis[r] : row_vis[r];
                vmax = max(vmax, v);
                vmin = min(vmin, v);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                vmax = max(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
                vmin = min(vmin, __shfl_xor_sync(0xffffffffu, vmin, o));
            }
            if (lane == 0) {
                groups[g].nrows = r1 - r0;
                groups[g].vmax = vmax;
                groups[g].vmin = vmin;
                if (g < PLAN_SMEM_GROUPS) s_vmax[g] = vmax;
            }
        }
    }
    __syncthreads();

    // Phase 3: item offsets (all key tiles, and the sampled tiles only).
    if (tid == 0) { carry_items = 0; carry_samples = 0; }
    __syncthreads();
    for (int32_t base = 0; base < n_groups; base += PLAN_THREADS) {
        const int32_t g = base + tid;
        int32_t tiles = 0, stiles = 0;
        if (g < n_groups) {
            tiles = ((g < PLAN_SMEM_GROUPS ? s_vmax[g] : groups[g].vmax) + (1 << tile_shift) - 1) >> tile_shift;
            stiles = (tiles + sample_stride - 1) / sample_stride;
        }
        const int32_t it = block_incl_scan(tiles, wbuf, OpAdd(), 0);
        const int32_t st = block_incl_scan(stiles, wbuf, OpAdd(), 0);
        if (g < n_groups) {
            item_prefix[g] = carry_items + it - tiles;
            sample_prefix[g] = carry_samples + st - stiles;
        }
        __syncthreads();
        if (tid == PLAN_THREADS - 1) {
            carry_items += it;
            carry_samples += st;
        }
        __syncthreads();
    }
    if (tid == 0) {
        item_prefix[n_groups] = carry_items;
        sample_prefix[n_groups] = carry_samples;
        plan->n_groups = n_groups;
        plan->n_items = carry_items;
        plan->n_sample_items = carry_samples;
        plan->any_fallback = 0;
    }
}

}  // namespace

int launch_plan(const int32_t *row_req, const int32_t *row_visible, int32_t R, int32_t group_rows,
                int32_t num_reqs, int64_t max_len, int32_t sample_stride, int32_t *row_vis,
                Group *groups, int32_t *item_prefix, int32_t *sample_prefix, Plan *plan,
                uint32_t *status, void *stream, int32_t tile_shift)
{
    const int32_t G = group_rows;
    plan_kernel<<<1, PLAN_THREADS, 0, static_cast<cudaStream_t>(stream)>>>(
        row_req, row_visible, R, G, num_reqs, max_len, sample_stride, tile_shift, row_vis, groups,
        item_prefix, sample_prefix, plan, status);
    return static_cast<int>(cudaGetLastError());
}

}  // namespace qsa

namespace qsa {
namespace {

// -inf for every position from the end of a row's last scored tile to ld.
__global__ void pad_kernel(float *__restrict__ logits, int64_t ld, int32_t R,
                           const int32_t *__restrict__ row_vis)
{
    const int32_t r = blockIdx.x;
    wait_prior_grid();                      // last kernel of its call: nothing to allow
    if (r >= R) return;
    const int64_t from = (static_cast<int64_t>(row_vis[r]) + TILE_M - 1) / TILE_M * TILE_M;
    float *row = logits + static_cast<int64_t>(r) * ld;
    const float ninf = -__int_as_float(0x7f800000);
    for (int64_t j = from + threadIdx.x; j < ld; j += blockDim.x) row[j] = ninf;
}

}  // namespace

int launch_pad(float *logits, int64_t ld, int32_t R, const int32_t *row_vis, bool overlap, void *stream)
{
    void *args[] = {&logits, &ld, &R, const_cast<int32_t **>(&row_vis)};
    return launch_kernel(reinterpret_cast<const void *>(&pad_kernel), dim3(R), dim3(256), 0,
                         static_cast<cudaStream_t>(stream), overlap, args);
}

}  // namespace qsa

namespace qsa {
namespace {

// Virtual rows of the block scorer (one per query row and KV head).
__global__ void block_rows_kernel(const int32_t *__restrict__ row_req, const int32_t *__restrict__ row_token,
                                  int32_t R, int32_t H, int32_t num_reqs, int32_t *__restrict__ vreq,
                                  int32_t *__restrict__ vtok, int32_t *__restrict__ vblk, uint32_t *status)
{
    const int64_t n = static_cast<int64_t>(R) * H;
    for (int64_t v = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; v < n;
         v += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int32_t h = static_cast<int32_t>(v / R), r = static_cast<int32_t>(v % R);
        const int32_t b = row_req[r];
        const int32_t t = row_token[r];
        const bool ok = b >= 0 && b < num_reqs && t >= 0;
        if (!ok && h == 0) record_error(status, ST_BAD_ROW);
        vreq[v] = ok ? b + h * num_reqs : -1;
        const int32_t tok = ok ? t + 1 : 0;
        vtok[v] = tok;
        vblk[v] = (tok + TILE_M - 1) / TILE_M;
    }
}

}  // namespace

int launch_block_rows(const int32_t *row_req, const int32_t *row_token, int32_t R, int32_t H,
                      int32_t num_reqs, int32_t *vreq, int32_t *vtok, int32_t *vblk, uint32_t *status,
                      void *stream)
{
    const int64_t n = static_cast<int64_t>(R) * H;
    const int grid = static_cast<int>(std::min<int64_t>((n + 255) / 256, 1024));
    block_rows_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(row_req, row_token, R, H, num_reqs,
                                                                          vreq, vtok, vblk, status);
    return static_cast<int>(cudaGetLastError());
}

}  // namespace qsa
