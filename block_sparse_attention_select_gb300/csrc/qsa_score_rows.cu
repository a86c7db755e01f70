// Index scorer for groups of up to 128 query rows of one request (prefill
// chunks): query rows on the TMEM lanes.
//
// Per group the H query heads sit in tensor memory as the A operand
// (128 lanes x H*64 columns, two FP16 values per column); key pages stream
// through shared memory by TMA (the block-table gather) and are the B operand
// in 32-position sub-tiles, so each tcgen05.mma is M=128 rows x N=32
// positions x K=16 and the only shared-memory operand traffic is the keys.
// The accumulators of one sub-tile are H x 32 FP32 columns, double-buffered.
//
// Each epilogue thread owns one query row (its TMEM lane) and 8 positions of
// every sub-tile: its head weights, threshold and visible length live in
// registers, it copies its accumulators out of TMEM, releases the buffer at
// once and then forms logit = sum_h w_h * max(dot_h, 0) per position.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "qsa_device.cuh"
#include "qsa_internal.h"

namespace qsa {
namespace {

constexpr int ROWS = 128;                 // query rows per group (TMEM lanes, MMA M)
constexpr int SUB = 32;                   // key positions per MMA (N)
constexpr int SUBS = TILE_M / SUB;        // sub-tiles per key tile
constexpr int RSTAGES = 6;                // key tiles in flight
constexpr uint32_t K_HALF = TILE_M * 128; // one K half (64 dims) of a key tile
constexpr uint32_t K_STAGE = 2 * K_HALF;  // 32 KiB
constexpr int R_EPI_WARPS = 16;           // 4 per lane quarter; part = 8 positions of a sub-tile
constexpr int R_THREADS = 64 + 32 * R_EPI_WARPS;

struct __align__(8) RCtrl {
    uint64_t full[RSTAGES];
    uint64_t empty[RSTAGES];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t q_ready;
    uint64_t drain;
    uint32_t tmem_base;
    int32_t abort;
};

constexpr uint32_t R_SMEM = RSTAGES * K_STAGE + sizeof(RCtrl) + 1024;
static_assert(R_SMEM <= 232448, "shared memory budget");

template <int H>
constexpr uint32_t tmem_cols()
{
    return H * 64 + 2 * H * SUB <= 128 ? 128 : (H * 64 + 2 * H * SUB <= 256 ? 256 : 512);
}

struct Cursor {
    const int32_t *prefix;
    int32_t g, it, it_end, stride;
    __device__ void init(const int32_t *pre, int32_t n_groups, int32_t it0, int32_t it1, int32_t s)
    {
        prefix = pre;
        it = it0;
        it_end = it1;
        stride = s;
        int32_t lo = 0, hi = n_groups - 1;
        while (lo < hi) {
            const int32_t mid = (lo + hi + 1) >> 1;
            if (__ldg(prefix + mid) <= it0) lo = mid; else hi = mid - 1;
        }
        g = lo;
    }
    __device__ bool valid() const { return it < it_end; }
    __device__ void settle() { while (it >= __ldg(prefix + g + 1)) ++g; }
    __device__ int32_t tile() const { return (it - __ldg(prefix + g)) * stride; }
    __device__ void next() { ++it; }
};

// D[tmem] (+)= A[tmem] * B[smem desc]^T, kind::f16, one CTA.
__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_x8(uint32_t taddr, uint32_t (&v)[8])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
                   "=r"(v[6]), "=r"(v[7])
                 : "r"(taddr)
                 : "memory");
}

// 32 lanes x 16 columns from registers (thread i -> lane base + i).
__device__ __forceinline__ void tmem_st_x16(uint32_t taddr, const uint32_t (&v)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

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

template <int H>
__device__ __forceinline__ float wrelu(const float (&w)[H], const uint32_t (&v)[H][8], int i)
{
    if constexpr (H == 1) {
        return fmaf(w[0], fmaxf(__uint_as_float(v[0][i]), 0.0f), 0.0f);
    } else {
        float2 s = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int h = 0; h < H; h += 2)
            s = ffma2(make_float2(w[h], w[h + 1]),
                      make_float2(fmaxf(__uint_as_float(v[h][i]), 0.0f),
                                  fmaxf(__uint_as_float(v[h + 1][i]), 0.0f)),
                      s);
        return s.x + s.y;
    }
}

template <int H>
__global__ void __launch_bounds__(R_THREADS, 1)
score_rows_kernel(const __grid_constant__ CUtensorMap tmap_k, const ScoreParams p,
                  const uint16_t *__restrict__ q)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint8_t *k_s = smem;
    RCtrl &c = *reinterpret_cast<RCtrl *>(smem + RSTAGES * K_STAGE);
    constexpr uint32_t TCOLS = tmem_cols<H>();
    constexpr uint32_t DCOL = H * 64;               // first accumulator column
    constexpr uint32_t DBUF = H * SUB;               // columns per accumulator buffer

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const bool sampled = p.mode == SCORE_SAMPLE;
    const int32_t n_items = sampled ? p.plan->n_sample_items : p.plan->n_items;
    const int32_t it0 = static_cast<int32_t>((static_cast<int64_t>(n_items) * blockIdx.x) / gridDim.x);
    const int32_t it1 = static_cast<int32_t>((static_cast<int64_t>(n_items) * (blockIdx.x + 1)) / gridDim.x);
    if (it0 >= it1) return;
    const int32_t n_groups = p.plan->n_groups;
    const int32_t *prefix = sampled ? p.sample_prefix : p.item_prefix;
    const int32_t stride = sampled ? p.sample_stride : 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < RSTAGES; ++s) {
            mbar_init(&c.full[s], 1);
            mbar_init(&c.empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&c.acc_full[b], 1);
            mbar_init(&c.acc_empty[b], R_EPI_WARPS);
        }
        mbar_init(&c.q_ready, R_EPI_WARPS);
        mbar_init(&c.drain, 1);
        c.abort = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc(&c.tmem_base, TCOLS);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) tma_prefetch_desc(&tmap_k);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = c.tmem_base;
    volatile int *abort = &c.abort;
    const uint64_t lim = p.wait_limit_ns;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer --
        // Lane i owns key box i of a tile; page ids are fetched PF items ahead
        // into a register ring that is only ever read PF iterations later.
        constexpr int PF = 4;
        Cursor cur, ahead;
        cur.init(prefix, n_groups, it0, it1, stride);
        ahead = cur;
        auto page_id = [&](Cursor &a) -> int32_t {
            if (!a.valid()) return -1;
            a.settle();
            const Group ga = p.groups[a.g];
            const int32_t pos0 = a.tile() * TILE_M;
            const int32_t nbox = (min(TILE_M, ga.vmax - pos0) + p.page_box - 1) / p.page_box;
            if (lane >= nbox || ga.req < 0) return -1;
            return __ldg(p.block_table + static_cast<int64_t>(ga.req) * p.max_pages +
                         (pos0 + lane * p.page_box) / p.page_pos);
        };
        int32_t ring[PF];
#pragma unroll
        for (int d = 0; d < PF; ++d) {
            ring[d] = page_id(ahead);
            ahead.next();
        }
        int32_t stage = 0;
        uint32_t phase = 0;
        bool stop = false;
        while (cur.valid() && !stop) {
#pragma unroll
            for (int u = 0; u < PF; ++u) {
                if (!cur.valid()) break;
                cur.settle();
                const int32_t pid = ring[u];
                ring[u] = page_id(ahead);
                ahead.next();
                const Group gr = p.groups[cur.g];
                if (__any_sync(0xffffffffu, !mbar_wait(&c.empty[stage], phase ^ 1u, abort, lim))) {
                    stop = true;
                    break;
                }
                const int32_t pos0 = cur.tile() * TILE_M;
                const int32_t nbox = (min(TILE_M, gr.vmax - pos0) + p.page_box - 1) / p.page_box;
                if (lane == 0)
                    mbar_arrive_expect_tx(&c.full[stage], static_cast<uint32_t>(nbox * p.page_box * 256));
                __syncwarp();
                if (lane < nbox) {
                    const int32_t pos = pos0 + lane * p.page_box;
                    int32_t y;
                    if (pid >= 0 && pid < p.num_pages) {
                        y = pid * p.page_pos + (pos % p.page_pos);
                    } else {
                        record_error(p.status, ST_BAD_PAGE);
                        y = p.num_pages * p.page_pos;      // past the end: TMA fills zeros
                    }
                    uint8_t *dst = k_s + stage * K_STAGE + lane * p.page_box * 128;
                    tma_load_2d(dst, &tmap_k, &c.full[stage], 0, y);
                    tma_load_2d(dst + K_HALF, &tmap_k, &c.full[stage], 64, y);
                }
                if (++stage == RSTAGES) { stage = 0; phase ^= 1u; }
                cur.next();
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------- MMA issuer --
        if (lane == 0) {
            Cursor cur;
            cur.init(prefix, n_groups, it0, it1, stride);
            int32_t cur_g = -1, stage = 0;
            uint32_t phase = 0, sub_cnt = 0, q_cnt = 0;
            const uint32_t idesc = umma_idesc_f16_f32(ROWS, SUB);
            for (; cur.valid(); cur.next()) {
                cur.settle();
                if (cur.g != cur_g) {
                    cur_g = cur.g;
                    if (!mbar_wait(&c.q_ready, q_cnt & 1u, abort, lim)) break;
                    ++q_cnt;
                    tc_fence_after();
                }
                const Group gr = p.groups[cur.g];
                if (!mbar_wait(&c.full[stage], phase, abort, lim)) break;
                tc_fence_after();
                const int32_t pos0 = cur.tile() * TILE_M;
                const int32_t nsub = (min(TILE_M, gr.vmax - pos0) + SUB - 1) / SUB;
                const uint32_t kbase = smem_u32(k_s + stage * K_STAGE);
                bool ok = true;
                for (int32_t sp = 0; sp < nsub; ++sp) {
                    const uint32_t b = sub_cnt & 1u;
                    if (!mbar_wait(&c.acc_empty[b], ((sub_cnt >> 1) & 1u) ^ 1u, abort, lim)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d0 = tmem + DCOL + b * DBUF;
#pragma unroll
                    for (int h = 0; h < H; ++h) {
#pragma unroll
                        for (int kk = 0; kk < HEAD_DIM / 16; ++kk) {
                            const uint64_t bd = sw128_kmajor_desc(kbase + (kk >> 2) * K_HALF +
                                                                  sp * SUB * 128 + (kk & 3) * 32);
                            umma_f16_ts(d0 + h * SUB, tmem + h * 64 + kk * 8, bd, idesc, kk > 0 ? 1u : 0u);
                        }
                    }
                    umma_commit(&c.acc_full[b]);
                    ++sub_cnt;
                }
                if (!ok) break;
                umma_commit(&c.empty[stage]);
                if (++stage == RSTAGES) { stage = 0; phase ^= 1u; }
            }
            umma_commit(&c.drain);
            mbar_wait(&c.drain, 0, abort, lim);
        }
    } else {
        // --------------------------------------------------- epilogue --
        const int ew = warp - 2;
        const int quarter = warp & 3;              // TMEM lanes = group rows quarter*32 ..
        const int part = ew >> 2;                  // positions part*8 .. of every sub-tile
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const int32_t rl = quarter * 32 + lane;    // this thread's row within the group
        Cursor cur;
        cur.init(prefix, n_groups, it0, it1, stride);
        int32_t cur_g = -1;
        uint32_t sub_cnt = 0;
        float wv[H];
        float tau = 0.0f;
        int32_t V = 0, r = 0;
        bool row_ok = false;
        Group gr{};
        for (; cur.valid(); cur.next()) {
            cur.settle();
            if (cur.g != cur_g) {
                // every MMA of the previous group has completed (its last
                // accumulators were consumed): A may be overwritten
                cur_g = cur.g;
                gr = p.groups[cur_g];
                r = gr.row0 + rl;
                row_ok = rl < gr.nrows;
#pragma unroll
                for (int h = 0; h < H; ++h) wv[h] = row_ok ? __ldg(p.w + static_cast<int64_t>(r) * H + h) : 0.0f;
                V = row_ok ? __ldg(p.row_vis + r) : 0;
                tau = (row_ok && p.mode == SCORE_FILTER) ? __ldg(p.tau + r) : 0.0f;
                // this warp writes head h = part (and part + 4, ...) of its 32 rows
                for (int h = part; h < H; h += 4) {
                    const uint4 *src = reinterpret_cast<const uint4 *>(q + (static_cast<int64_t>(r) * H + h) * HEAD_DIM);
#pragma unroll
                    for (int c16 = 0; c16 < 4; ++c16) {
                        uint32_t pk[16];
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const uint4 x = row_ok ? __ldg(src + c16 * 4 + t) : make_uint4(0, 0, 0, 0);
                            pk[4 * t] = x.x; pk[4 * t + 1] = x.y; pk[4 * t + 2] = x.z; pk[4 * t + 3] = x.w;
                        }
                        tmem_st_x16(tmem + lane_off + h * 64 + c16 * 16, pk);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&c.q_ready);
            }
            const int32_t tile = cur.tile();
            const int32_t pos0 = tile * TILE_M;
            const int32_t nsub = (min(TILE_M, gr.vmax - pos0) + SUB - 1) / SUB;
            uint32_t found = 0;
            uint2 *cand_row = nullptr;
            if (p.mode == SCORE_FILTER)
                cand_row = p.cand + ((static_cast<int64_t>(r) * p.tiles_ld + tile) * 4 + part) * CAND_SLOTS;
            bool ok = true;
            for (int32_t sp = 0; sp < nsub; ++sp) {
                const uint32_t b = sub_cnt & 1u;
                if (!mbar_wait(&c.acc_full[b], (sub_cnt >> 1) & 1u, abort, lim)) { ok = false; break; }
                tc_fence_after();
                uint32_t v[H][8];
#pragma unroll
                for (int h = 0; h < H; ++h)
                    tmem_ld_x8(tmem + lane_off + DCOL + b * DBUF + h * SUB + part * 8, v[h]);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&c.acc_empty[b]);
                ++sub_cnt;
                if (!row_ok) continue;
                const int32_t j0 = pos0 + sp * SUB + part * 8;
                const bool full = j0 + 8 <= V;
                if (p.mode == SCORE_FILTER) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float s = wrelu<H>(wv, v, i);
                        if ((full || j0 + i < V) && s >= tau) {
                            cand_row[found] = make_uint2(__float_as_uint(s), static_cast<uint32_t>(j0 + i));
                            ++found;
                        }
                    }
                } else {
                    float o[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) o[i] = wrelu<H>(wv, v, i);
                    float *dst;
                    if (sampled)
                        dst = p.out + static_cast<int64_t>(r) * p.ld +
                              static_cast<int64_t>(tile / p.sample_stride) * TILE_M + (j0 - pos0);
                    else
                        dst = p.out + static_cast<int64_t>(r) * p.ld + j0;
                    if (full && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
                        reinterpret_cast<float4 *>(dst)[0] = make_float4(o[0], o[1], o[2], o[3]);
                        reinterpret_cast<float4 *>(dst)[1] = make_float4(o[4], o[5], o[6], o[7]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            if (j0 + i < V) dst[i] = o[i];
                            else if (!sampled && p.pad_inf && j0 + i < p.ld) dst[i] = -__int_as_float(0x7f800000);
                        }
                    }
                }
            }
            if (!ok) break;
            if (p.mode == SCORE_FILTER && row_ok)
                p.cand_cnt[(static_cast<int64_t>(r) * p.tiles_ld + tile) * 4 + part] = static_cast<uint8_t>(found);
            if (!sampled && p.mode != SCORE_FILTER && p.pad_inf && row_ok) {
                // positions of skipped sub-tiles (past the group's longest row)
                for (int32_t sp = nsub; sp < SUBS; ++sp)
                    for (int i = 0; i < 8; ++i) {
                        const int32_t j = pos0 + sp * SUB + part * 8 + i;
                        if (j < p.ld) p.out[static_cast<int64_t>(r) * p.ld + j] = -__int_as_float(0x7f800000);
                    }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (c.abort && threadIdx.x == 0) record_error(p.status, ST_TIMEOUT);
    if (warp == 1) tmem_dealloc(tmem, TCOLS);
}

template <int H>
int launch_rows_h(const ScoreParams &p, const void *tk, const void *q, int grid, cudaStream_t s)
{
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return static_cast<int>(cudaErrorInvalidDevice);
    if (!attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(score_rows_kernel<H>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(R_SMEM));
        if (e != cudaSuccess) return static_cast<int>(e);
        attr_done[dev] = true;
    }
    score_rows_kernel<H><<<grid, R_THREADS, R_SMEM, s>>>(*static_cast<const CUtensorMap *>(tk), p,
                                                         static_cast<const uint16_t *>(q));
    return static_cast<int>(cudaGetLastError());
}

}  // namespace

int launch_score_rows(const ScoreParams &p, const void *tmap_k, const void *q, int grid, void *stream)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (p.H) {
    case 1: return launch_rows_h<1>(p, tmap_k, q, grid, s);
    case 2: return launch_rows_h<2>(p, tmap_k, q, grid, s);
    case 4: return launch_rows_h<4>(p, tmap_k, q, grid, s);
    default: return static_cast<int>(cudaErrorInvalidValue);
    }
}

}  // namespace qsa
