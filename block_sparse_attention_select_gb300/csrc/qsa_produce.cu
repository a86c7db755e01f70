// Index-key producer, the step before the indexer ("spec(MODEL-MM-QWEN4-EXP)
// ...", section "The component deep-dives": one stored index-key state per four
// tokens, emitted at the token with (position + 1) % 4 == 0, RMSNorm on the
// pooled key, RoPE at the block-start position; the DSv4 compress kernel pools
// with a learned softmax over an overlapping window of eight tokens).
//
// Two produced blocks i per warp (one with the 8-token window), lane l
// holding dimensions [4l, 4l + 4):
// the windows' token keys are loaded at once (one 256-byte line per token per
// warp), pooled with softmax weights of the pooling logits (the
// mean without them), RMS-normalised with a warp reduction, rotated with the
// cos / sin row of the block from a table built once (qsa_rope_table, FP64
// angles), and stored as FP16 into slot i % P of page block_table[b][i / P].
// HBM-bound: 4 (or 8) x 256 bytes read and 256 bytes written per block.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "qsa_device.cuh"
#include "qsa_internal.h"

namespace qsa {
namespace {

constexpr int PROD_WARPS = 8;      // warps per CTA
// keys per warp: two for window 4; window 8 already holds eight token lines
// per key (two keys per warp there cost spills and one CTA per SM, measured
// slower)
template <int W>
__host__ __device__ constexpr int keys_per_warp() { return W == 4 ? 2 : 1; }

// four FP16 values held as raw bits (two registers) until they are used
__device__ __forceinline__ float4 half4_to_float4(uint2 u)
{
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&u.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}

// W: the pooling window (4 or 8 tokens).  Each warp takes KPW keys, i_base
// and i_base + PROD_WARPS * k, and requests every load of all of them before
// it computes any: one memory round trip per warp.  (A persistent variant
// that kept three rounds of loads in flight per warp measured slower.)
template <int W>
__global__ void __launch_bounds__(PROD_WARPS * 32, 4)
produce_kernel(const ProduceParams p)
{
    constexpr int KPW = keys_per_warp<W>();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int32_t b = blockIdx.y;
    wait_prior_grid();
    if (b >= p.n_reqs) return;
    const int32_t t0 = p.seq_start[b];
    const int32_t n = p.seq_start[b + 1] - t0;
    const int32_t p0 = p.pos_start[b];
    if (n <= 0) return;
    if (p0 < 0 || static_cast<int64_t>(p0) + n > INT32_MAX - 8) {
        if (threadIdx.x == 0 && blockIdx.x == 0) record_error(p.status, ST_BAD_ROW);
        return;
    }
    // blocks [i_lo, i_hi): complete within the new tokens, and every existing
    // position of the window among them (window start max(0, 4i + 4 - W) >= p0)
    const int32_t i_hi = (p0 + n) >> 2;
    const int32_t i_lo = p0 == 0 ? 0 : (p0 + W - 1) >> 2;
    if (threadIdx.x == 0 && blockIdx.x == 0 && i_hi - i_lo > static_cast<int32_t>(gridDim.x) * PROD_WARPS * KPW)
        record_error(p.status, ST_BAD_ROW);            // more new tokens than max_tokens promised
    const int32_t i_base = i_lo + static_cast<int32_t>(blockIdx.x) * PROD_WARPS * KPW + warp;
    if (i_base >= i_hi) return;                         // warp-uniform

    const int32_t h = p.rope_dim >> 1;                  // a multiple of 4
    const int32_t d0 = 4 * lane;
    const bool lo_half = d0 < h, hi_half = !lo_half && d0 < p.rope_dim;
    const int32_t j0 = lo_half ? d0 : d0 - h;

    // ---- every load of every key of this warp, before any arithmetic: the
    //      window's token lines, pooling logits, RoPE row and page id
    uint2 xr[KPW][W];
    float lg[KPW][W];
    float4 cs[KPW], sn[KPW];
    int32_t page[KPW], nw[KPW];
#pragma unroll
    for (int k = 0; k < KPW; ++k) {
        const int32_t i = i_base + k * PROD_WARPS;
        cs[k] = make_float4(1.0f, 1.0f, 1.0f, 1.0f);
        sn[k] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        page[k] = -1;
        nw[k] = 0;
        if (i < i_hi) {                                 // warp-uniform
            const int32_t first = max(0, 4 * i + 4 - W);
            nw[k] = 4 * i + 4 - first;                  // W, or less at block 0 when W = 8
            const int64_t r0 = static_cast<int64_t>(t0) + first - p0;
            const __half *xw = static_cast<const __half *>(p.x) + r0 * HEAD_DIM + 4 * lane;
#pragma unroll
            for (int w = 0; w < W; ++w) {
                if (w < nw[k]) {
                    xr[k][w] = __ldg(reinterpret_cast<const uint2 *>(xw + w * HEAD_DIM));
                    lg[k][w] = p.pool_logit ? __ldg(p.pool_logit + r0 + w) : 0.0f;
                }
            }
            if ((lo_half || hi_half) && i < p.rope_blocks) {
                const float *row = p.rope_table + static_cast<int64_t>(i) * p.rope_dim;
                cs[k] = __ldg(reinterpret_cast<const float4 *>(row + j0));
                sn[k] = __ldg(reinterpret_cast<const float4 *>(row + h + j0));
            }
            const int32_t pi = i >> p.page_shift;
            if (pi < p.max_pages) page[k] = __ldg(p.block_table + static_cast<int64_t>(b) * p.max_pages + pi);
        }
    }
    const float4 g = __ldg(reinterpret_cast<const float4 *>(p.norm_weight) + lane);
    const int src = lo_half ? lane + (h >> 2) : (hi_half ? lane - (h >> 2) : lane);

#pragma unroll
    for (int k = 0; k < KPW; ++k) {
        const int32_t i = i_base + k * PROD_WARPS;
        if (i >= i_hi) break;                           // warp-uniform (keys in order)

        // ---- pool: softmax of the logits over the window (equal logits = mean)
        float m = lg[k][0];
#pragma unroll
        for (int w = 1; w < W; ++w)
            if (w < nw[k]) m = fmaxf(m, lg[k][w]);
        float e[W], sum = 0.0f;
#pragma unroll
        for (int w = 0; w < W; ++w) {
            e[w] = 0.0f;
            if (w < nw[k]) {
                e[w] = expf(lg[k][w] - m);
                sum += e[w];
            }
        }
        const float inv_sum = 1.0f / sum;
        float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int w = 0; w < W; ++w) {
            if (w < nw[k]) {
                const float a = e[w] * inv_sum;
                const float4 xv = half4_to_float4(xr[k][w]);
                v[0] = fmaf(a, xv.x, v[0]);
                v[1] = fmaf(a, xv.y, v[1]);
                v[2] = fmaf(a, xv.z, v[2]);
                v[3] = fmaf(a, xv.w, v[3]);
            }
        }

        // ---- RMSNorm over the 128 dimensions
        float ss = v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float r = rsqrtf(ss * (1.0f / HEAD_DIM) + p.eps);
        float y[4] = {v[0] * r * g.x, v[1] * r * g.y, v[2] * r * g.z, v[3] * r * g.w};

        // ---- RoPE at position 4i: pairs (j, j + h) of the first rope_dim dims
        float yp[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) yp[c] = __shfl_sync(0xffffffffu, y[c], src);
        if (lo_half || hi_half) {
            const float cc[4] = {cs[k].x, cs[k].y, cs[k].z, cs[k].w};
            const float sc[4] = {sn[k].x, sn[k].y, sn[k].z, sn[k].w};
#pragma unroll
            for (int c = 0; c < 4; ++c)
                y[c] = lo_half ? y[c] * cc[c] - yp[c] * sc[c] : yp[c] * sc[c] + y[c] * cc[c];
        }

        // ---- store into the block's page slot
        if (i >= p.rope_blocks || (i >> p.page_shift) >= p.max_pages) {
            if (lane == 0) record_error(p.status, ST_BAD_ROW);
            continue;
        }
        if (page[k] < 0 || page[k] >= p.num_pages) {
            if (lane == 0) record_error(p.status, ST_BAD_PAGE);
            continue;
        }
        const int64_t slot = static_cast<int64_t>(page[k]) * p.page_positions + (i & (p.page_positions - 1));
        __half2 o0 = __floats2half2_rn(y[0], y[1]), o1 = __floats2half2_rn(y[2], y[3]);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t *>(&o0);
        u.y = *reinterpret_cast<uint32_t *>(&o1);
        *reinterpret_cast<uint2 *>(static_cast<__half *>(p.k_cache) + slot * HEAD_DIM + 4 * lane) = u;
    }
}

// Row i: cos(4i * theta^(-2j / rope_dim)) for j < rope_dim / 2, then the sines;
// angles and their cos / sin in FP64, stored as FP32.
__global__ void rope_table_kernel(float *__restrict__ table, int32_t n_blocks, int32_t rope_dim, double theta)
{
    const int32_t h = rope_dim >> 1;
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= static_cast<int64_t>(n_blocks) * h) return;
    const int32_t i = static_cast<int32_t>(idx / h), j = static_cast<int32_t>(idx % h);
    const double a = 4.0 * static_cast<double>(i) * pow(theta, -2.0 * j / rope_dim);
    double s, c;
    sincos(a, &s, &c);
    table[static_cast<int64_t>(i) * rope_dim + j] = static_cast<float>(c);
    table[static_cast<int64_t>(i) * rope_dim + h + j] = static_cast<float>(s);
}

}  // namespace

int launch_produce(const ProduceParams &p, int32_t max_tokens, void *stream)
{
    const int32_t blocks_per_req = max_tokens / 4 + 2;
    const int kpw = p.window == 8 ? keys_per_warp<8>() : keys_per_warp<4>();
    const dim3 grid((blocks_per_req + PROD_WARPS * kpw - 1) / (PROD_WARPS * kpw), p.n_reqs);
    void *args[] = {const_cast<ProduceParams *>(&p)};
    const void *k = p.window == 8 ? reinterpret_cast<const void *>(&produce_kernel<8>)
                                  : reinterpret_cast<const void *>(&produce_kernel<4>);
    return launch_kernel(k, grid, dim3(PROD_WARPS * 32), 0, static_cast<cudaStream_t>(stream), false, args);
}

int launch_rope_table(float *table, int32_t n_blocks, int32_t rope_dim, double theta, void *stream)
{
    const int64_t n = static_cast<int64_t>(n_blocks) * (rope_dim >> 1);
    const int64_t grid = (n + 255) / 256;
    rope_table_kernel<<<static_cast<unsigned>(grid), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        table, n_blocks, rope_dim, theta);
    return static_cast<int>(cudaGetLastError());
}

}  // namespace qsa
