// Sparse-attention consumer, the step after the indexer ("spec(MODEL-MM-
// QWEN4-EXP) ...", section "The component deep-dives": QSA attends raw tokens
// selected at ratio-4 granularity; plain GQA, 24 query heads over 2 KV heads,
// head_dim 256).
//
// Row r (a query at token t of request b) attends the tokens 4j .. 4j + 3 of
// every selected index position j and the tokens 4V .. t of its unfinished
// block (V = (t + 1) / 4).  One CTA per (row, KV head): the GROUP query heads
// of that KV head share every gathered K / V line.  Tokens go in chunks of 32:
// the chunk's K and V rows are gathered through the block table into shared
// memory (K rows padded by one word so that lane-per-token reads hit distinct
// banks), lane c scores token c for the warp's heads, each head keeps an
// online softmax (running max and sum), and every thread accumulates two of
// the 256 output dimensions for all GROUP heads.  FP32 throughout, output FP32.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "qsa_device.cuh"
#include "qsa_internal.h"

namespace qsa {
namespace {

constexpr int AT_D = 256;               // head dimension
constexpr int AT_THREADS = 128;
constexpr int AT_WARPS = AT_THREADS / 32;
constexpr int AT_CHUNK = 32;            // tokens per chunk (one per lane)
constexpr int AT_MAXG = 16;             // query heads per KV head
constexpr int K_LD = AT_D + 2;          // halves per padded K row (129 words)

struct AttendShared {
    float q[AT_MAXG][AT_D];                 // pre-scaled queries
    __half k[AT_CHUNK][K_LD];
    __half v[AT_CHUNK][AT_D];
    float pw[AT_MAXG][AT_CHUNK];            // this chunk's softmax numerators
    float alpha[AT_MAXG];                   // rescale of the running output
    float m[AT_MAXG], l[AT_MAXG];           // running max and sum per head
    int32_t tok[AT_CHUNK];                  // token positions of the chunk (-1 = none)
};

__global__ void __launch_bounds__(AT_THREADS)
attend_kernel(const AttendParams p)
{
    extern __shared__ __align__(16) uint8_t smem_raw[];
    AttendShared &sh = *reinterpret_cast<AttendShared *>(smem_raw);
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int32_t r = blockIdx.x, g = blockIdx.y;
    wait_prior_grid();
    if (r >= p.rows || g >= p.hkv) return;
    const int group = p.hq / p.hkv;
    const int32_t b = p.row_req[r];
    const int32_t tok_r = p.row_token[r];
    if (b < 0 || b >= p.num_reqs || tok_r < 0 ||
        static_cast<int64_t>(tok_r) >= static_cast<int64_t>(p.max_pages) * p.page_tokens) {
        if (t == 0 && g == 0) record_error(p.status, ST_BAD_ROW);
        return;                                          // uniform: the row's output is left as it was
    }
    const int32_t vis = (tok_r + 1) >> 2;               // complete index positions
    const int32_t tail0 = 4 * vis;                       // first token of the unfinished block

    // queries of this KV head's group, scaled
    for (int i = t; i < group * AT_D; i += AT_THREADS) {
        const int h = i / AT_D, d = i % AT_D;
        sh.q[h][d] = __half2float(static_cast<const __half *>(p.q)[(static_cast<int64_t>(r) * p.hq + g * group + h) *
                                                                    AT_D + d]) * p.scale;
    }
    if (t < AT_MAXG) {
        sh.m[t] = -INFINITY;
        sh.l[t] = 0.0f;
    }
    float acc[AT_MAXG][2];
#pragma unroll
    for (int h = 0; h < AT_MAXG; ++h) acc[h][0] = acc[h][1] = 0.0f;

    const int32_t *selr = p.sel + static_cast<int64_t>(r) * p.k;
    // token stream: 4 tokens per selection slot (slots holding -1 or a bad
    // position contribute none), then the tail tokens tail0 .. tok_r
    const int32_t n_stream = 4 * p.k + (tok_r - tail0 + 1);
    const __half *kc = static_cast<const __half *>(p.k_cache);
    const __half *vc = static_cast<const __half *>(p.v_cache);
    const int32_t *bt = p.block_table + static_cast<int64_t>(b) * p.max_pages;
    __syncthreads();

    for (int32_t c0 = 0; c0 < n_stream; c0 += AT_CHUNK) {
        // ---- token positions of the chunk
        if (t < AT_CHUNK) {
            const int32_t s = c0 + t;
            int32_t pos = -1;
            if (s < 4 * p.k) {
                const int32_t j = selr[s >> 2];
                if (j >= 0 && j < vis) pos = 4 * j + (s & 3);
                else if (j >= vis && (s & 3) == 0) record_error(p.status, ST_BAD_ROW);
            } else if (s < n_stream) {
                pos = tail0 + (s - 4 * p.k);
            }
            sh.tok[t] = pos;
        }
        __syncthreads();
        // ---- gather K and V rows: warp w takes tokens w, w + 4, ...; lane l
        //      copies halves [8l, 8l + 8) of a row (16 bytes)
        for (int c = warp; c < AT_CHUNK; c += AT_WARPS) {
            const int32_t pos = sh.tok[c];
            uint4 kv4 = make_uint4(0u, 0u, 0u, 0u), vv4 = make_uint4(0u, 0u, 0u, 0u);
            if (pos >= 0) {
                const int32_t page = bt[pos >> p.page_shift];
                if (page >= 0 && page < p.num_pages) {
                    const int64_t line = ((static_cast<int64_t>(page) * p.page_tokens + (pos & (p.page_tokens - 1))) *
                                          p.hkv + g) * AT_D;
                    kv4 = __ldg(reinterpret_cast<const uint4 *>(kc + line) + lane);
                    vv4 = __ldg(reinterpret_cast<const uint4 *>(vc + line) + lane);
                } else if (lane == 0) {
                    record_error(p.status, ST_BAD_PAGE);
                }
            }
            // K rows are 129 words apart: store word by word
            const uint32_t kw[4] = {kv4.x, kv4.y, kv4.z, kv4.w};
            uint32_t *krow = reinterpret_cast<uint32_t *>(&sh.k[c][0]);
#pragma unroll
            for (int i = 0; i < 4; ++i) krow[4 * lane + i] = kw[i];
            reinterpret_cast<uint4 *>(&sh.v[c][0])[lane] = vv4;
        }
        __syncthreads();
        // ---- scores: warp w handles heads w, w + 4, ...; lane c token c
        const bool live = sh.tok[lane] >= 0;
        for (int h = warp; h < group; h += AT_WARPS) {
            float s = 0.0f;
            const __half2 *krow = reinterpret_cast<const __half2 *>(&sh.k[lane][0]);
            const float2 *qh = reinterpret_cast<const float2 *>(&sh.q[h][0]);
#pragma unroll 8
            for (int d2 = 0; d2 < AT_D / 2; ++d2) {
                const float2 kf = __half22float2(krow[d2]);
                const float2 qf = qh[d2];
                s = fmaf(qf.x, kf.x, s);
                s = fmaf(qf.y, kf.y, s);
            }
            s = live ? s : -INFINITY;
            float mx = s;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float m_old = sh.m[h];
            const float m_new = fmaxf(m_old, mx);
            // no live token yet: nothing to weigh (m stays -inf)
            const float e = (live && m_new > -INFINITY) ? __expf(s - m_new) : 0.0f;
            float se = e;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) se += __shfl_xor_sync(0xffffffffu, se, o);
            sh.pw[h][lane] = e;
            if (lane == 0) {
                const float a = m_old > -INFINITY ? __expf(m_old - m_new) : 0.0f;
                sh.alpha[h] = a;
                sh.l[h] = sh.l[h] * a + se;
                sh.m[h] = m_new;
            }
        }
        __syncthreads();
        // ---- PV: thread t owns dimensions 2t, 2t + 1 of every head
#pragma unroll
        for (int h = 0; h < AT_MAXG; ++h) {
            if (h < group) {                              // acc stays in registers: constant indices only
                const float a = sh.alpha[h];
                acc[h][0] *= a;
                acc[h][1] *= a;
            }
        }
#pragma unroll 4
        for (int c = 0; c < AT_CHUNK; ++c) {
            const float2 vf = __half22float2(reinterpret_cast<const __half2 *>(&sh.v[c][0])[t]);
#pragma unroll
            for (int h = 0; h < AT_MAXG; ++h) {
                if (h < group) {
                    const float w = sh.pw[h][c];
                    acc[h][0] = fmaf(w, vf.x, acc[h][0]);
                    acc[h][1] = fmaf(w, vf.y, acc[h][1]);
                }
            }
        }
        __syncthreads();                                  // tok / k / v / pw are rewritten next chunk
    }
    // ---- normalise and store
#pragma unroll
    for (int h = 0; h < AT_MAXG; ++h) {
        if (h < group) {
            const float l = sh.l[h];
            const float inv = l > 0.0f ? 1.0f / l : 0.0f;
            const float2 o = make_float2(acc[h][0] * inv, acc[h][1] * inv);
            reinterpret_cast<float2 *>(p.out + (static_cast<int64_t>(r) * p.hq + g * group + h) * AT_D)[t] = o;
        }
    }
}

}  // namespace

size_t attend_smem_bytes() { return sizeof(AttendShared); }

int launch_attend(const AttendParams &p, void *stream)
{
    static size_t done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return static_cast<int>(cudaErrorInvalidDevice);
    const size_t smem = sizeof(AttendShared);
    if (smem > done[dev]) {
        const cudaError_t e = cudaFuncSetAttribute(attend_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem));
        if (e != cudaSuccess) return static_cast<int>(e);
        done[dev] = smem;
    }
    void *args[] = {const_cast<AttendParams *>(&p)};
    return launch_kernel(reinterpret_cast<const void *>(&attend_kernel), dim3(p.rows, p.hkv), dim3(AT_THREADS),
                         smem, static_cast<cudaStream_t>(stream), false, args);
}

}  // namespace qsa
