// Index scorer: the per-head contraction q[r,h,:] . k_j on the 5th-generation
// tensor cores (tcgen05.mma kind::f16, FP16 in, FP32 accumulate in TMEM), fed
// by TMA gathers of key pages through the block table, with the head
// reduction logit = sum_h w[r,h] * max(dot, 0) and the causal mask fused into
// the TMEM read-out.
//
// Tile: M = 128 key positions (TMEM lanes) x N = (rows of a group) * H
// (TMEM columns, <= 256) x K = 128.  Keys are the A operand because they
// differ per tile, the group's queries are the B operand and stay resident in
// shared memory while the CTA walks the group's key tiles.  One persistent CTA
// per SM: warp 0 issues TMA, warp 1 issues MMAs, 16 epilogue warps drain TMEM
// (double-buffered accumulators, 2 x 256 columns; each warp owns one lane
// quarter x 64 columns) and write the results.
//
// The block scorer (per-head maximum over 128-token blocks) has its own
// kernel at the end of this file, with the virtual rows on the TMEM lanes.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "qsa_device.cuh"
#include "qsa_internal.h"

namespace qsa {
namespace {

constexpr uint32_t Q_HALF_BYTES = N_MAX * 128;          // 256 rows x 128 B
constexpr uint32_t Q_BYTES = 2 * Q_HALF_BYTES;            // 64 KiB
constexpr uint32_t K_HALF_BYTES = TILE_M * 128;           // 128 rows x 128 B
constexpr uint32_t K_STAGE_BYTES = 2 * K_HALF_BYTES;      // 32 KiB
constexpr uint32_t SMEM_TILES = Q_BYTES + KSTAGES * K_STAGE_BYTES;
constexpr uint32_t TMEM_COLS = 512;

struct __align__(8) Ctrl {
    uint64_t full[KSTAGES];
    uint64_t empty[KSTAGES];
    uint64_t q_full;
    uint64_t q_empty;
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int32_t abort;
};

// Group data of one epilogue warp: the rows of its 64 accumulator columns,
// private to the warp so that a group change needs no barrier across warps.
struct EpiRows {
    __align__(16) float w[64];   // weights by row pair: w[(r / 2) * 2H + 2h + r % 2], r = row - first row of the warp
    __align__(16) int32_t vis[64];   // V of each row
    __align__(16) float tau[64];     // FILTER threshold of each row
    __align__(16) uint32_t masks[32];   // FILTER: mask words of the chunk being drained
};

static_assert(sizeof(Ctrl) % 16 == 0, "EpiRows must stay 16-byte aligned");
constexpr uint32_t SMEM_BYTES = SMEM_TILES + sizeof(Ctrl) + EPI_WARPS * sizeof(EpiRows) + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// Walks the same (group, tile) sequence in every role of a CTA.  The current
// group's item range is kept in registers: with most of the SM's unified
// L1/shared memory taken by shared memory, a per-item reload of the prefix
// would be an L2 round trip on every role's critical path.
struct ItemCursor {
    const int32_t *prefix;
    int32_t g, it, it_end, stride;
    int32_t g_first, g_next;     // items of group g: [g_first, g_next)
    // Halving search for the group holding item it0: the last g with
    // prefix[g] <= it0 (prefix is non-decreasing, prefix[0] = 0).  Every
    // value it leaves in the cursor comes from loads at uniform addresses.
    // (With the warp-wide search below in the drain and MMA roles as well, the
    // bounds taken from lane shuffles, the filter pass ran ~10 % slower: the
    // drain loop is issue-bound and sensitive to how its tile numbers are
    // derived.)
    __device__ void init(const int32_t *pre, int32_t n_groups, int32_t it0, int32_t it1, int32_t s)
    {
        int32_t lo = 0, hi = n_groups - 1;
        while (lo < hi) {
            int32_t mid = (lo + hi + 1) >> 1;
            if (__ldg(pre + mid) <= it0) lo = mid; else hi = mid - 1;
        }
        set(pre, lo, it0, it1, s);
    }
    // The same search by all 32 lanes of a warp (same arguments): each round
    // the lanes read 32 entries spread over the remaining range and a ballot
    // keeps the last one <= it0, so up to 32 groups take one L2 round trip
    // instead of one per halving.  For the producer warp, whose first loads
    // wait for it.
    __device__ void init_warp(const int32_t *pre, int32_t n_groups, int32_t it0, int32_t it1, int32_t s, int lane)
    {
        int32_t lo = 0, span = n_groups;        // g in [lo, lo + span), prefix[lo] <= it0
        while (span > 1) {
            const int32_t step = (span + 31) >> 5;
            const int32_t i = lo + lane * step;
            const bool le = i < lo + span && __ldg(pre + i) <= it0;
            const uint32_t b = __ballot_sync(0xffffffffu, le);
            const int32_t j = 31 - __clz(b);    // lane 0 reads prefix[lo] <= it0, so b != 0
            lo += j * step;
            span = min(step, span - j * step);
        }
        set(pre, lo, it0, it1, s);
    }
    __device__ void set(const int32_t *pre, int32_t g0, int32_t it0, int32_t it1, int32_t s)
    {
        prefix = pre;
        it = it0;
        it_end = it1;
        stride = s;
        g = g0;
        g_first = __ldg(prefix + g);
        g_next = __ldg(prefix + g + 1);
    }
    __device__ bool valid() const { return it < it_end; }
    __device__ void settle()
    {
        while (it >= g_next) {
            ++g;
            g_first = g_next;
            g_next = __ldg(prefix + g + 1);
        }
    }
    __device__ int32_t tile() const { return (it - g_first) * stride; }
    __device__ void next() { ++it; }
};

// d = a * b + c on packed FP32 pairs (one instruction on sm_100-family SMs).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ float relu_f(uint32_t acc) { return fmaxf(__uint_as_float(acc), 0.0f); }

// Scores of two query rows (a, b) at one key position:
//   s = sum_h w[row, h] * max(acc[row, h], 0),  heads in order h = 0 .. H-1,
// each head one fused multiply-add onto an accumulator that starts at +0 (so
// no score is -0), the two rows side by side in one packed FMA per head.
// wp: the pair's weights interleaved by head, (w[a,h], w[b,h]) for h = 0 ...
// Every mode of the scorer (logits, sampled tiles, filter) uses this same
// arithmetic, so a score is the same bit pattern whichever pass computed it.
template <int H>
__device__ __forceinline__ float2 relu_pair_sum(const float *wp, const uint32_t *acc_a, const uint32_t *acc_b)
{
    float2 s = make_float2(0.0f, 0.0f);
    if constexpr (H == 1) {
        const float2 ww = *reinterpret_cast<const float2 *>(wp);
        s = ffma2(ww, make_float2(relu_f(acc_a[0]), relu_f(acc_b[0])), s);
    } else {
#pragma unroll
        for (int h = 0; h < H; h += 2) {
            const float4 ww = *reinterpret_cast<const float4 *>(wp + 2 * h);
            s = ffma2(make_float2(ww.x, ww.y), make_float2(relu_f(acc_a[h]), relu_f(acc_b[h])), s);
            s = ffma2(make_float2(ww.z, ww.w), make_float2(relu_f(acc_a[h + 1]), relu_f(acc_b[h + 1])), s);
        }
    }
    return s;
}

// Drains this warp's 64 accumulator columns (64 / H query rows) of one tile.
// Lane i holds key position tile * 128 + quarter * 32 + i.  FULL: every row
// of the group sees the whole tile, so no per-element visibility test.
template <int H, int MODE, bool FULL, bool ALLROWS>
__device__ __forceinline__ void epilogue_rows(const ScoreParams &p, EpiRows &e, const Group &gr,
                                              int32_t tile, uint32_t taddr, int cq, int quarter,
                                              int lane, uint32_t lt_mask, int32_t nmine)
{
    constexpr int RPC = 32 / H;          // rows per 32-column chunk
    constexpr int RPW = 64 / H;          // rows per warp
    constexpr int B = RPC < 8 ? RPC : 8; // rows scored together: independent chains, no branches
    static_assert(B % 4 == 0, "row pairs, thresholds read four rows at a time");
    const int32_t p_in_tile = quarter * 32 + lane;
    const int32_t j = tile * TILE_M + p_in_tile;
    const int64_t r0 = static_cast<int64_t>(gr.row0) + cq * RPW;     // first row of this warp
    float *slot0 = nullptr;
    uint32_t *mask0 = nullptr;
    float *out0 = nullptr;
    if constexpr (MODE == SCORE_FILTER) {
        // this quarter's slot column in the (tile, r0) region: a row further is
        // TILE_M floats further (an immediate offset), a slot row 4 floats
        slot0 = p.cand_score + (static_cast<int64_t>(tile) * p.R + r0) * TILE_M + quarter;
        mask0 = p.cand_mask + (r0 * p.tiles_ld + tile) * 4 + quarter;
    } else if constexpr (MODE == SCORE_SAMPLE) {
        out0 = p.out + r0 * p.ld + static_cast<int64_t>(tile >> p.sample_shift) * TILE_M + p_in_tile;
    } else {
        out0 = p.out + r0 * p.ld + j;
    }
    const uint32_t mask_row = static_cast<uint32_t>(p.tiles_ld) * 4u;   // mask words from one row to the next
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
        const int32_t c0 = ch * RPC;
        if (!ALLROWS && c0 >= nmine) break;                  // warp-uniform
        uint32_t v[32];
        tmem_ld_32x32b_x32(taddr + static_cast<uint32_t>(cq * 64 + ch * 32), v);
        tmem_ld_wait();
#pragma unroll
        for (int b0 = 0; b0 < RPC; b0 += B) {
            if (!ALLROWS && c0 + b0 >= nmine) break;         // warp-uniform
            float s[B];
#pragma unroll
            for (int i = 0; i < B; i += 2) {
                const float2 sp = relu_pair_sum<H>(e.w + (c0 + b0 + i) * H, v + (b0 + i) * H, v + (b0 + i + 1) * H);
                s[i] = sp.x;
                s[i + 1] = sp.y;
            }
            float tau[B];
            if constexpr (MODE == SCORE_FILTER) {
#pragma unroll
                for (int i = 0; i < B; i += 4) {
                    const float4 t4 = *reinterpret_cast<const float4 *>(e.tau + c0 + b0 + i);
                    tau[i] = t4.x; tau[i + 1] = t4.y; tau[i + 2] = t4.z; tau[i + 3] = t4.w;
                }
            }
            if constexpr (MODE == SCORE_FILTER) {
                // staged over the block's rows (compares, then ballots, then
                // ranks and stores), so that the rows' short dependent chains
                // interleave
                bool take[B];
                uint32_t m[B];
#pragma unroll
                for (int i = 0; i < B; ++i) {
                    const int32_t el = c0 + b0 + i;
                    const bool live = ALLROWS || el < nmine;  // warp-uniform
                    take[i] = live && (FULL || j < e.vis[el]) && s[i] >= tau[i];
                }
#pragma unroll
                for (int i = 0; i < B; ++i) m[i] = __ballot_sync(0xffffffffu, take[i]);
                if (lane == 0) {
#pragma unroll
                    for (int i = 0; i < B; i += 4)
                        *reinterpret_cast<uint4 *>(&e.masks[b0 + i]) = make_uint4(m[i], m[i + 1], m[i + 2], m[i + 3]);
                }
#pragma unroll
                for (int i = 0; i < B; ++i) {
                    // a passing lane's slot row: the passing lanes below it
                    const uint32_t rk = static_cast<uint32_t>(__popc(m[i] & lt_mask));
                    if (take[i]) (slot0 + rk * 4u)[(c0 + b0 + i) * TILE_M] = s[i];
                }
            } else {
#pragma unroll
                for (int i = 0; i < B; ++i) {
                    const int32_t el = c0 + b0 + i;
                    const bool live = ALLROWS || el < nmine;  // warp-uniform
                    const bool ok = live && (FULL || j < e.vis[el]);
                    if constexpr (MODE == SCORE_SAMPLE) {
                        if (ok) out0[el * p.ld] = s[i];
                    } else {
                        float *dst = out0 + el * p.ld;
                        if (ok) *dst = s[i];
                        else if (live && p.pad_inf && j < p.ld) *dst = -__int_as_float(0x7f800000);
                    }
                }
            }
        }
        if constexpr (MODE == SCORE_FILTER) {
            // one store for the chunk: lane i writes the mask word of row c0 + i
            // (gathered through the warp's shared-memory slots, not a select per row)
            __syncwarp();
            if (lane < RPC && (ALLROWS || c0 + lane < nmine))
                mask0[static_cast<uint32_t>(c0 + lane) * mask_row] = e.masks[lane];
            __syncwarp();
        }
    }
}

// Key-tile producer, warp 0 of both scorers.  The whole warp walks the CTA's
// items; lane i owns key box i of a tile.  On a group change lane 0 waits
// until the previous group's MMAs have released the query buffer and calls
// load_q (which arms q_full).  Block-table entries are loaded PREFETCH items
// ahead so that the page-id round trip never sits in front of a TMA issue.
// Before returning (also after an abort) the warp waits, bounded, for every
// copy it issued, so that none lands in shared memory after the CTA ends.
template <int KST, typename LoadQ>
__device__ __forceinline__ void produce_tiles(const ScoreParams &p, const CUtensorMap *tmap_k,
                                              const CUtensorMap *tmap_k128, uint8_t *k_s, uint64_t *full,
                                              uint64_t *empty, uint64_t *q_full, uint64_t *q_empty,
                                              const int32_t *prefix, int32_t n_groups, int32_t it0, int32_t it1,
                                              int32_t stride, int lane, volatile int *abort, uint64_t lim,
                                              LoadQ load_q)
{
    constexpr int PREFETCH = 8;
    ItemCursor cur, ahead;
    cur.init_warp(prefix, n_groups, it0, it1, stride, lane);
    // the first group's queries are requested before the page ids: their
    // load does not wait for the block-table round trip
    cur.settle();
    int32_t cur_g = cur.g, q_loads = 1, stage = 0;
    Group gr = p.groups[cur_g];
    if (lane == 0) load_q(gr);
    ahead = cur;
    Group ga = gr;
    int32_t ga_g = cur_g;                   // group held in ga (reloaded on a change only)
    auto page_id = [&](ItemCursor &a) -> int32_t {
        if (!a.valid()) return -1;
        a.settle();
        if (a.g != ga_g) {
            ga_g = a.g;
            ga = p.groups[a.g];
        }
        const int32_t pos0 = a.tile() * TILE_M;
        const int32_t nbox = (min(TILE_M, ga.vmax - pos0) + p.page_box - 1) >> p.page_box_shift;
        if (lane >= nbox || ga.req < 0) return -1;
        const int32_t pos = pos0 + lane * p.page_box;
        return __ldg(p.block_table + static_cast<int64_t>(ga.req) * p.max_pages + (pos >> p.page_pos_shift));
    };
    int32_t ring[PREFETCH];
#pragma unroll
    for (int d = 0; d < PREFETCH; ++d) {
        ring[d] = page_id(ahead);
        ahead.next();
    }
    uint32_t phase = 0;
    uint32_t loaded = 0;                    // bit s: stage s holds an issued copy (of parity bit KST + s)
    bool stop = false;
    // the ring slot read in an iteration is refilled in the same iteration
    // and read again PREFETCH iterations later (no move of a pending load)
    while (cur.valid() && !stop) {
#pragma unroll
        for (int u = 0; u < PREFETCH; ++u) {
            if (!cur.valid()) break;
            cur.settle();
            const int32_t pid = ring[u];
            ring[u] = page_id(ahead);
            ahead.next();
            if (cur.g != cur_g) {
                cur_g = cur.g;
                gr = p.groups[cur_g];
                bool ok = true;
                if (lane == 0) {
                    ok = mbar_wait(q_empty, (q_loads - 1) & 1, abort, lim);
                    if (ok) load_q(gr);
                }
                if (__any_sync(0xffffffffu, !ok)) { stop = true; break; }
                ++q_loads;
            }
            if (__any_sync(0xffffffffu, !mbar_wait(&empty[stage], phase ^ 1u, abort, lim))) {
                stop = true;
                break;
            }
            const int32_t pos0 = cur.tile() * TILE_M;
            const int32_t nbox = (min(TILE_M, gr.vmax - pos0) + p.page_box - 1) >> p.page_box_shift;
            if (lane == 0)
                mbar_arrive_expect_tx(&full[stage], static_cast<uint32_t>(nbox * p.page_box * 256));
            __syncwarp();
            loaded = (loaded & ~(1u << (KST + stage))) | (1u << stage) | (phase << (KST + stage));
            const int32_t pos = pos0 + lane * p.page_box;
            const bool good = pid >= 0 && pid < p.num_pages;
            int32_t y = good ? pid * p.page_pos + (pos & (p.page_pos - 1))
                             : p.num_pages * p.page_pos;   // past the end: TMA fills zeros
            if (lane < nbox && !good) record_error(p.status, ST_BAD_PAGE);
            // a full tile whose pages are physically consecutive is one box per K half
            const int32_t y0 = __shfl_sync(0xffffffffu, y, 0);
            const bool run = nbox * p.page_box == TILE_M &&
                             __all_sync(0xffffffffu, lane >= nbox || (good && y == y0 + lane * p.page_box));
            uint8_t *dst = k_s + stage * K_STAGE_BYTES;
            if (run) {
                if (lane == 0) {
                    tma_load_2d(dst, tmap_k128, &full[stage], 0, y0);
                    tma_load_2d(dst + K_HALF_BYTES, tmap_k128, &full[stage], 64, y0);
                }
            } else if (lane < nbox) {
                dst += lane * p.page_box * 128;
                tma_load_2d(dst, tmap_k, &full[stage], 0, y);
                tma_load_2d(dst + K_HALF_BYTES, tmap_k, &full[stage], 64, y);
            }
            if (++stage == KST) { stage = 0; phase ^= 1u; }
            cur.next();
        }
    }
    // copies still in flight (only after an abort: otherwise the MMA thread
    // has waited for all of them)
    if (lane == 0) {
        mbar_wait_bounded(q_full, (q_loads - 1) & 1, lim);
        for (int s = 0; s < KST; ++s)
            if (loaded & (1u << s)) mbar_wait_bounded(&full[s], (loaded >> (KST + s)) & 1u, lim);
    }
    __syncwarp();
}

template <int H, int MODE>
__device__ __forceinline__ void epilogue_tile(const ScoreParams &p, EpiRows &e, const Group &gr,
                                              int32_t tile, uint32_t taddr, int cq, int quarter,
                                              int lane, uint32_t lt_mask)
{
    constexpr int RPW = 64 / H;
    const int32_t nmine = min(RPW, gr.nrows - cq * RPW);
    if (nmine <= 0) return;
    const bool full = (tile + 1) * TILE_M <= gr.vmin;
    if (nmine == RPW) {
        if (full) epilogue_rows<H, MODE, true, true>(p, e, gr, tile, taddr, cq, quarter, lane, lt_mask, nmine);
        else epilogue_rows<H, MODE, false, true>(p, e, gr, tile, taddr, cq, quarter, lane, lt_mask, nmine);
    } else {
        if (full) epilogue_rows<H, MODE, true, false>(p, e, gr, tile, taddr, cq, quarter, lane, lt_mask, nmine);
        else epilogue_rows<H, MODE, false, false>(p, e, gr, tile, taddr, cq, quarter, lane, lt_mask, nmine);
    }
}

template <int H>
__global__ void __launch_bounds__(SCORE_THREADS, 1)
score_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
             const __grid_constant__ CUtensorMap tmap_k128, const ScoreParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint8_t *q_s = smem;
    uint8_t *k_s = smem + Q_BYTES;
    Ctrl &c = *reinterpret_cast<Ctrl *>(smem + SMEM_TILES);
    EpiRows *epi_rows = reinterpret_cast<EpiRows *>(smem + SMEM_TILES + sizeof(Ctrl));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // prologue: barriers, TMEM and descriptor prefetch touch no global
    // memory, so they run while the previous kernel of the stream finishes
    if (threadIdx.x == 0) {
        for (int s = 0; s < KSTAGES; ++s) {
            mbar_init(&c.full[s], 1);
            mbar_init(&c.empty[s], 1);
        }
        mbar_init(&c.q_full, 1);
        mbar_init(&c.q_empty, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&c.acc_full[b], 1);
            mbar_init(&c.acc_empty[b], EPI_WARPS);
        }
        mbar_init(&c.drain, 1);
        c.abort = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc(&c.tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmap_q);
        tma_prefetch_desc(&tmap_k);
        tma_prefetch_desc(&tmap_k128);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = c.tmem_base;
    volatile int *abort = &c.abort;
    const uint64_t lim = p.wait_limit_ns;
    wait_prior_grid();

    const bool sampled = p.mode == SCORE_SAMPLE;
    const int32_t n_items = sampled ? p.plan->n_sample_items : p.plan->n_items;
    const int32_t it0 = static_cast<int32_t>((static_cast<int64_t>(n_items) * blockIdx.x) / gridDim.x);
    const int32_t it1 = static_cast<int32_t>((static_cast<int64_t>(n_items) * (blockIdx.x + 1)) / gridDim.x);
    const int32_t n_groups = p.plan->n_groups;
    const int32_t *prefix = sampled ? p.sample_prefix : p.item_prefix;
    const int32_t stride = sampled ? p.sample_stride : 1;

    if (it0 >= it1) {
        // no item for this CTA: straight to the teardown
    } else if (warp == 0) {
        // ------------------------------------------------ TMA producer --
        // the group's queries: rows row0 .. of [rows * H, 128]
        auto load_q = [&](const Group &g) {
            mbar_arrive_expect_tx(&c.q_full, Q_BYTES);
            tma_load_2d(q_s, &tmap_q, &c.q_full, 0, g.row0 * H);
            tma_load_2d(q_s + Q_HALF_BYTES, &tmap_q, &c.q_full, 64, g.row0 * H);
        };
        produce_tiles<KSTAGES>(p, &tmap_k, &tmap_k128, k_s, c.full, c.empty, &c.q_full, &c.q_empty, prefix,
                               n_groups, it0, it1, stride, lane, abort, lim, load_q);
    } else if (warp == 1) {
        // ------------------------------------------------- MMA issuer --
        if (lane == 0) {
            ItemCursor cur;
            cur.init(prefix, n_groups, it0, it1, stride);
            const uint64_t q_desc0 = sw128_kmajor_desc(smem_u32(q_s));
            int32_t cur_g = -1, stage = 0, q_uses = 0;
            uint32_t phase = 0, acc_cnt = 0, idesc = 0, idle_arrivals = 0;
            bool have_q = false;
            for (; cur.valid(); cur.next()) {
                cur.settle();
                if (cur.g != cur_g) {
                    cur_g = cur.g;
                    const Group gr = p.groups[cur_g];
                    if (have_q) umma_commit(&c.q_empty);   // previous group's MMAs done -> q free
                    if (!mbar_wait(&c.q_full, q_uses & 1, abort, lim)) break;
                    ++q_uses;
                    have_q = true;
                    const int n = ((gr.nrows * H + 15) / 16) * 16;
                    idesc = umma_idesc_f16_f32(TILE_M, n);
                    // drain warps whose 64 columns hold no row of this group
                    // skip its tiles; their release of each accumulator is
                    // given here, after the previous use of that buffer ended
                    static_assert(EPI_WARPS == 16, "4 lane quarters x 4 column blocks of 64");
                    idle_arrivals = static_cast<uint32_t>(4 * (4 - min(4, (gr.nrows + 64 / H - 1) / (64 / H))));
                }
                if (!mbar_wait(&c.full[stage], phase, abort, lim)) break;
                const uint32_t b = acc_cnt & 1u;
                if (!mbar_wait(&c.acc_empty[b], ((acc_cnt >> 1) & 1u) ^ 1u, abort, lim)) break;
                tc_fence_after();
                // descriptor of base + off = descriptor of base + off / 16 (the
                // 14-bit start-address field cannot carry within shared memory)
                const uint64_t a0 = sw128_kmajor_desc(smem_u32(k_s + stage * K_STAGE_BYTES));
                const uint32_t d = tmem + b * 256u;
#pragma unroll
                for (int kk = 0; kk < HEAD_DIM / 16; ++kk) {
                    const uint32_t off = static_cast<uint32_t>((kk & 3) * 32);
                    umma_f16(d, a0 + (((kk >> 2) * K_HALF_BYTES + off) >> 4),
                             q_desc0 + (((kk >> 2) * Q_HALF_BYTES + off) >> 4), idesc, kk > 0 ? 1u : 0u);
                }
                umma_commit(&c.empty[stage]);
                umma_commit(&c.acc_full[b]);
                if (idle_arrivals) mbar_arrive_cnt(&c.acc_empty[b], idle_arrivals);
                if (++stage == KSTAGES) { stage = 0; phase ^= 1u; }
                ++acc_cnt;
            }
            // every MMA issued by this thread has finished before TMEM is freed
            umma_commit(&c.drain);
            mbar_wait(&c.drain, 0, abort, lim);
        }
    } else {
        // --------------------------------------------------- epilogue --
        const int ew = warp - 2;
        const int quarter = warp & 3;           // TMEM lanes this warp may read
        const int cq = ew >> 2;                 // accumulator columns [cq * 64, +64)
        uint32_t lt_mask;
        asm("mov.u32 %0, %%lanemask_lt;" : "=r"(lt_mask));
        EpiRows &er = epi_rows[ew];
        ItemCursor cur;
        cur.init(prefix, n_groups, it0, it1, stride);
        int32_t cur_g = -1;
        uint32_t acc_cnt = 0;
        Group gr{};
        for (; cur.valid(); cur.next()) {
            cur.settle();
            if (cur.g != cur_g) {
                cur_g = cur.g;
                gr = p.groups[cur_g];
                constexpr int32_t RPW = 64 / H;
                const int32_t first = cq * RPW;
                const int32_t nmine = max(0, min(RPW, gr.nrows - first));
                __syncwarp();
                for (int32_t i = lane; i < RPW * H; i += 32) {
                    const int32_t rr = i / H, h = i % H;          // rows past the group weigh 0
                    er.w[(rr >> 1) * 2 * H + 2 * h + (rr & 1)] =
                        rr < nmine ? __ldg(p.w + static_cast<int64_t>(gr.row0 + first + rr) * H + h) : 0.0f;
                }
                for (int32_t i = lane; i < nmine; i += 32) {
                    const int32_t r = gr.row0 + first + i;
                    er.vis[i] = __ldg(p.row_vis + r);
                    er.tau[i] = p.mode == SCORE_FILTER ? __ldg(p.tau + r) : 0.0f;
                }
                __syncwarp();
            }
            const uint32_t b = acc_cnt & 1u;
            if (cq * (64 / H) >= gr.nrows) {    // no row of this group here: the MMA thread releases for us
                ++acc_cnt;
                continue;
            }
            // (every lane gives up together: the TMEM loads are warp-wide)
            if (!__all_sync(0xffffffffu, mbar_wait(&c.acc_full[b], (acc_cnt >> 1) & 1u, abort, lim))) break;
            tc_fence_after();
            const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + b * 256u;
            const int32_t t = cur.tile();
            switch (p.mode) {
            case SCORE_FILTER: epilogue_tile<H, SCORE_FILTER>(p, er, gr, t, taddr, cq, quarter, lane, lt_mask); break;
            case SCORE_SAMPLE: epilogue_tile<H, SCORE_SAMPLE>(p, er, gr, t, taddr, cq, quarter, lane, lt_mask); break;
            default: epilogue_tile<H, SCORE_LOGITS>(p, er, gr, t, taddr, cq, quarter, lane, lt_mask); break;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&c.acc_empty[b]);
            ++acc_cnt;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    allow_next_grid();                      // this CTA's global writes are all issued
    if (c.abort && threadIdx.x == 0) record_error(p.status, ST_TIMEOUT);
    if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

template <int H>
int launch_h(const ScoreParams &p, const void *tq, const void *tk, const void *tk128, int grid, bool overlap,
             cudaStream_t s)
{
    // once per device (calls from several host threads may race here)
    static std::mutex mu;
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return static_cast<int>(cudaErrorInvalidDevice);
    {
        std::lock_guard<std::mutex> lk(mu);
        if (!attr_done[dev]) {
            cudaError_t e = cudaFuncSetAttribute(score_kernel<H>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(SMEM_BYTES));
            if (e != cudaSuccess) return static_cast<int>(e);
            attr_done[dev] = true;
        }
    }
    void *args[] = {const_cast<void *>(tq), const_cast<void *>(tk), const_cast<void *>(tk128),
                    const_cast<ScoreParams *>(&p)};
    return launch_kernel(reinterpret_cast<const void *>(&score_kernel<H>), dim3(grid), dim3(SCORE_THREADS),
                         SMEM_BYTES, s, overlap, args);
}

// ---------------------------------------------------------------------------
// Block scorer with the virtual rows on the TMEM lanes (BLOCKMAX).
//
// D[row, token] = Q_h K^T for a group of up to 256 virtual rows of one head
// (the queries, resident in shared memory) against a tile of N = 256 tokens of
// two 128-token pages (the keys), K = 128.  The group is split into two halves
// of 128 rows; each half is one M = 128 MMA into its own 256-column TMEM
// accumulator, so one key tile (64 KB) feeds 2 x 8.4 MFLOP, half the key bytes
// per FLOP of a 128-row group.  A block score is the maximum of a row's dot
// products over the block's tokens, so each drain thread owns one row and
// reduces its block's 128 accumulator columns in registers: no exchange
// between warps.  16 drain warps: half w / 8, lane quarter w % 4, block
// (w / 4) % 2 of the tile; half 1 drains while half 0's next MMA runs.
constexpr int BR_M = 128;                                 // rows per MMA: one half of a group
constexpr int BR_THREADS = 64 + 32 * 16;                  // TMA warp, MMA warp, 2 x 8 drain warps
constexpr int BR_KST = 2;                                 // key stages of 64 KiB
constexpr uint32_t BR_QHALF = BR_ROWS * 128;              // queries: one K half of 256 rows, 32 KiB
constexpr uint32_t BR_KHALF = 2 * TILE_M * 128;           // keys: one K half of 256 tokens, 32 KiB
constexpr uint32_t BR_STAGE = 2 * BR_KHALF;
constexpr uint32_t BR_TILES = 2 * BR_QHALF + BR_KST * BR_STAGE;
static_assert(BR_ROWS == 2 * BR_M, "a group is two MMA halves");

struct __align__(8) BrCtrl {
    uint64_t full[BR_KST];
    uint64_t empty[BR_KST];
    uint64_t q_full;
    uint64_t q_empty;
    uint64_t acc_full[2];       // per half
    uint64_t acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int32_t abort;
};
constexpr uint32_t BR_SMEM = BR_TILES + sizeof(BrCtrl) + 1024;
static_assert(BR_SMEM <= 232448, "shared memory budget");

// The producer warp of the block scorer: per tile, pages 2t and 2t + 1 of the
// group's (virtual) request, each as two boxes of [128 tokens][64 dims] (lane
// i issues page i).  Like produce_tiles, it waits (bounded) for its own
// copies before returning.
__device__ __forceinline__ void produce_block_tiles(const ScoreParams &p, const CUtensorMap *tmap_q,
                                                    const CUtensorMap *tmap_k, uint8_t *q_s, uint8_t *k_s,
                                                    BrCtrl &c, const int32_t *prefix, int32_t n_groups,
                                                    int32_t it0, int32_t it1, int lane, volatile int *abort,
                                                    uint64_t lim)
{
    ItemCursor cur;
    cur.init_warp(prefix, n_groups, it0, it1, 1, lane);
    cur.settle();
    int32_t cur_g = cur.g, q_loads = 1, stage = 0;
    Group gr = p.groups[cur_g];
    auto load_q = [&](const Group &g) {
        const int32_t h = g.row0 / p.blk_rows, r0 = g.row0 - h * p.blk_rows;
        mbar_arrive_expect_tx(&c.q_full, 2 * BR_QHALF);
        tma_load_3d(q_s, tmap_q, &c.q_full, 0, h, r0);
        tma_load_3d(q_s + BR_QHALF, tmap_q, &c.q_full, 64, h, r0);
    };
    if (lane == 0) load_q(gr);
    uint32_t phase = 0, loaded = 0;
    bool stop = false;
    for (; cur.valid() && !stop; cur.next()) {
        cur.settle();
        if (cur.g != cur_g) {
            cur_g = cur.g;
            gr = p.groups[cur_g];
            bool ok = true;
            if (lane == 0) {
                ok = mbar_wait(&c.q_empty, (q_loads - 1) & 1, abort, lim);
                if (ok) load_q(gr);
            }
            if (__any_sync(0xffffffffu, !ok)) break;
            ++q_loads;
        }
        const int32_t blk0 = cur.tile() * 2;
        const int32_t nblk = min(2, (gr.vmax + TILE_M - 1) / TILE_M - blk0);
        // page ids of the tile's blocks (before the stage wait: the round trip overlaps it)
        int32_t pid = -1;
        if (lane < nblk && gr.req >= 0)
            pid = __ldg(p.block_table + static_cast<int64_t>(gr.req % p.blk_reqs) * p.max_pages + blk0 + lane);
        if (__any_sync(0xffffffffu, !mbar_wait(&c.empty[stage], phase ^ 1u, abort, lim))) {
            stop = true;
            break;
        }
        if (lane == 0) mbar_arrive_expect_tx(&c.full[stage], static_cast<uint32_t>(nblk) * 2u * TILE_M * 128u);
        __syncwarp();
        loaded = (loaded & ~(1u << (BR_KST + stage))) | (1u << stage) | (phase << (BR_KST + stage));
        if (lane < nblk) {
            const bool good = pid >= 0 && pid < p.num_pages;
            if (!good) record_error(p.status, ST_BAD_PAGE);
            const int32_t y = (good ? pid : p.num_pages) * TILE_M;      // past the end: TMA fills zeros
            const int32_t h = gr.row0 / p.blk_rows;
            uint8_t *dst = k_s + stage * BR_STAGE + lane * (TILE_M * 128);
            tma_load_3d(dst, tmap_k, &c.full[stage], 0, h, y);
            tma_load_3d(dst + BR_KHALF, tmap_k, &c.full[stage], 64, h, y);
        }
        if (++stage == BR_KST) { stage = 0; phase ^= 1u; }
    }
    if (lane == 0) {
        mbar_wait_bounded(&c.q_full, (q_loads - 1) & 1, lim);
        for (int s = 0; s < BR_KST; ++s)
            if (loaded & (1u << s)) mbar_wait_bounded(&c.full[s], (loaded >> (BR_KST + s)) & 1u, lim);
    }
    __syncwarp();
}

__global__ void __launch_bounds__(BR_THREADS, 1)
score_blockrows_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                       const ScoreParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint8_t *q_s = smem;                        // [K half][256 rows][128 B]
    uint8_t *k_s = smem + 2 * BR_QHALF;         // stages of [K half][256 tokens][128 B]
    BrCtrl &c = *reinterpret_cast<BrCtrl *>(smem + BR_TILES);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < BR_KST; ++s) {
            mbar_init(&c.full[s], 1);
            mbar_init(&c.empty[s], 1);
        }
        mbar_init(&c.q_full, 1);
        mbar_init(&c.q_empty, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&c.acc_full[b], 1);
            mbar_init(&c.acc_empty[b], 8);
        }
        mbar_init(&c.drain, 1);
        c.abort = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc(&c.tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmap_q);
        tma_prefetch_desc(&tmap_k);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = c.tmem_base;
    volatile int *abort = &c.abort;
    const uint64_t lim = p.wait_limit_ns;
    wait_prior_grid();

    const int32_t n_items = p.plan->n_items;
    const int32_t it0 = static_cast<int32_t>((static_cast<int64_t>(n_items) * blockIdx.x) / gridDim.x);
    const int32_t it1 = static_cast<int32_t>((static_cast<int64_t>(n_items) * (blockIdx.x + 1)) / gridDim.x);
    const int32_t n_groups = p.plan->n_groups;
    const int32_t *prefix = p.item_prefix;

    if (it0 >= it1) {
        // no item for this CTA
    } else if (warp == 0) {
        produce_block_tiles(p, &tmap_q, &tmap_k, q_s, k_s, c, prefix, n_groups, it0, it1, lane, abort, lim);
    } else if (warp == 1) {
        // ------------------------------------------------- MMA issuer --
        if (lane == 0) {
            ItemCursor cur;
            cur.init(prefix, n_groups, it0, it1, 1);
            constexpr uint32_t idesc = umma_idesc_f16_f32(BR_M, 2 * TILE_M);
            const uint64_t q_desc0 = sw128_kmajor_desc(smem_u32(q_s));
            int32_t cur_g = -1, stage = 0, q_uses = 0, halves = 1;
            uint32_t phase = 0, uses[2] = {0, 0};
            bool have_q = false;
            for (; cur.valid(); cur.next()) {
                cur.settle();
                if (cur.g != cur_g) {
                    cur_g = cur.g;
                    halves = p.groups[cur_g].nrows > BR_M ? 2 : 1;
                    if (have_q) umma_commit(&c.q_empty);   // previous group's MMAs done -> queries free
                    if (!mbar_wait(&c.q_full, q_uses & 1, abort, lim)) break;
                    ++q_uses;
                    have_q = true;
                }
                if (!mbar_wait(&c.full[stage], phase, abort, lim)) break;
                // descriptor of base + off = descriptor of base + off / 16 (the
                // 14-bit start-address field cannot carry within shared memory)
                const uint64_t k_desc0 = sw128_kmajor_desc(smem_u32(k_s + stage * BR_STAGE));
                bool ok = true;
                for (int hf = 0; hf < halves; ++hf) {
                    if (!mbar_wait(&c.acc_empty[hf], (uses[hf] & 1u) ^ 1u, abort, lim)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < HEAD_DIM / 16; ++kk) {
                        const uint32_t off = static_cast<uint32_t>((kk & 3) * 32);
                        umma_f16(tmem + static_cast<uint32_t>(hf) * 256u,
                                 q_desc0 + (((kk >> 2) * BR_QHALF + static_cast<uint32_t>(hf) * BR_M * 128u + off) >> 4),
                                 k_desc0 + (((kk >> 2) * BR_KHALF + off) >> 4), idesc, kk > 0 ? 1u : 0u);
                    }
                    umma_commit(&c.acc_full[hf]);
                    ++uses[hf];
                }
                if (!ok) break;
                umma_commit(&c.empty[stage]);
                if (++stage == BR_KST) { stage = 0; phase ^= 1u; }
            }
            umma_commit(&c.drain);
            mbar_wait(&c.drain, 0, abort, lim);
        }
    } else {
        // --------------------------------------------------- epilogue --
        const int ew = warp - 2;
        const int hf = ew >> 3;                 // half of the group: accumulator columns [256 hf, +256)
        const int lq = warp & 3;                // TMEM lanes [32 lq, +32): virtual rows of the half
        const int bt = (ew >> 2) & 1;           // block bt of each tile: columns [128 bt, +128)
        const int32_t rig = hf * BR_M + lq * 32 + lane;
        const uint32_t taddr = tmem + (static_cast<uint32_t>(lq * 32) << 16) +
                               static_cast<uint32_t>(hf * 256 + bt * TILE_M);
        ItemCursor cur;
        cur.init(prefix, n_groups, it0, it1, 1);
        int32_t cur_g = -1;
        uint32_t uses = 0;
        bool active = false;                    // the group has rows in this half
        bool mine = false;
        int32_t vis = 0;                        // tokens the row sees
        float *orow = nullptr;
        for (; cur.valid(); cur.next()) {
            cur.settle();
            if (cur.g != cur_g) {
                cur_g = cur.g;
                const Group gr = p.groups[cur_g];
                active = gr.nrows > hf * BR_M;
                mine = rig < gr.nrows;
                const int64_t v = static_cast<int64_t>(gr.row0) + rig;
                // a lane past the group's rows takes the unmasked path: its
                // maximum is never stored, and a masked pass over all 128
                // columns would hold up the whole warp
                vis = mine ? __ldg(p.row_vis + v) : INT32_MAX;
                orow = p.out + v * p.ld;
            }
            if (!active) continue;              // no MMA for this half either
            if (!__all_sync(0xffffffffu, mbar_wait(&c.acc_full[hf], uses & 1u, abort, lim))) break;
            tc_fence_after();
            const int32_t blk = cur.tile() * 2 + bt;        // the block this warp reduces
            const int32_t tok0 = blk * TILE_M;
            // the block's 128 columns, 32 at a time, three-operand maxima;
            // tokens at or past the row's end are left out
            float mx = -__int_as_float(0x7f800000);
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t u[32];
                tmem_ld_32x32b_x32(taddr + static_cast<uint32_t>(ch * 32), u);
                tmem_ld_wait();
                const int32_t lim_c = vis - (tok0 + ch * 32);   // columns of this chunk the row sees
                if (lim_c >= 32) {
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        float m3;
                        asm("max.f32 %0, %1, %2, %3;" : "=f"(m3) : "f"(mx), "f"(__uint_as_float(u[i])),
                            "f"(__uint_as_float(u[i + 1])));
                        mx = m3;
                    }
                } else if (lim_c > 0) {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (i < lim_c) mx = fmaxf(mx, __uint_as_float(u[i]));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&c.acc_empty[hf]);
            if (mine && tok0 < vis) orow[blk] = mx;
            ++uses;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    allow_next_grid();
    if (c.abort && threadIdx.x == 0) record_error(p.status, ST_TIMEOUT);
    if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

int launch_score_blockrows(const ScoreParams &p, const void *tmap_q3, const void *tmap_k, int grid, bool overlap,
                           void *stream)
{
    static std::mutex mu;
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return static_cast<int>(cudaErrorInvalidDevice);
    {
        std::lock_guard<std::mutex> lk(mu);
        if (!attr_done[dev]) {
            cudaError_t e = cudaFuncSetAttribute(score_blockrows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(BR_SMEM));
            if (e != cudaSuccess) return static_cast<int>(e);
            attr_done[dev] = true;
        }
    }
    void *args[] = {const_cast<void *>(tmap_q3), const_cast<void *>(tmap_k), const_cast<ScoreParams *>(&p)};
    return launch_kernel(reinterpret_cast<const void *>(&score_blockrows_kernel), dim3(grid), dim3(BR_THREADS),
                         BR_SMEM, static_cast<cudaStream_t>(stream), overlap, args);
}

namespace {
}  // namespace

uint32_t score_smem_bytes() { return SMEM_BYTES; }

int launch_score(const ScoreParams &p, const void *tmap_q, const void *tmap_k, const void *tmap_k128,
                 int grid, bool overlap, void *stream)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (p.H) {
    case 1: return launch_h<1>(p, tmap_q, tmap_k, tmap_k128, grid, overlap, s);
    case 2: return launch_h<2>(p, tmap_q, tmap_k, tmap_k128, grid, overlap, s);
    case 4: return launch_h<4>(p, tmap_q, tmap_k, tmap_k128, grid, overlap, s);
    case 8: return launch_h<8>(p, tmap_q, tmap_k, tmap_k128, grid, overlap, s);
    default: return static_cast<int>(cudaErrorInvalidValue);
    }
}

}  // namespace qsa
