// Sparse-attention consumer, the step after the indexer ("spec(MODEL-MM-
// QWEN4-EXP) ...", section "The component deep-dives": QSA attends raw tokens
// selected at ratio-4 granularity; plain GQA, 24 query heads over 2 KV heads,
// head_dim 256).
//
// Row r (a query at token t of request b) attends the tokens 4j .. 4j + 3 of
// every selected index position j and the tokens 4V .. t of its unfinished
// block (V = (t + 1) / 4).  One CTA of 256 threads per (row, KV head): the G
// query heads of that KV head (G <= 16) share every gathered K / V row.
// Tokens go in chunks of 128, both contractions on the 5th-generation tensor
// cores (kind::f16, FP16 operands, FP32 accumulators in TMEM):
//   S^T[token, head] = K_chunk . Q^T   M = 128 tokens, N = 16 heads, K = 256
//   O^T[dim, head]  += V^T . P^T       M = 2 x 128 dims, N = 32, K = 128 tokens
// Every operand is K-major in the 128-byte swizzle layout: K rows are gathered
// straight into that layout; V rows are gathered into a staging tile and
// transposed in shared memory (8 x 8 blocks: ldmatrix.trans then stmatrix).
// Warp w reads TMEM lane quarter w % 4 and owns heads 8 (w / 4) .. + 7: in
// the softmax, tokens 32 (w % 4) .. + 31 of the chunk (scores scaled in FP32;
// each head's running maximum comes from warp max-reductions combined
// through shared memory; the numerators p go to the PV product as an FP16
// pair, p_hi = fp16(p) and p_lo = fp16(p - p_hi) in columns 0..15 and 16..31
// of N, so their rounding stays near FP32); in the output, dimensions
// 32 (w % 4) + lane and that + 128, kept in registers and rescaled by
// exp(m_old - m_new) per chunk.  Each thread also
// keeps its share of its heads' softmax denominators, summed over the CTA at
// the end.
// The gather of chunk c + 1 (cp.async) is issued as soon as chunk c's score
// product is done and runs under chunk c's softmax, PV product and output
// update.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "qsa_device.cuh"
#include "qsa_internal.h"

namespace qsa {
namespace {

constexpr int AT_D = 256;                   // head dimension
// head sets (warps per TMEM lane quarter): 2 measured 5.01 ms at the 1,616-row
// bench, 4 (512 threads, 4 heads per warp) 5.24 ms
constexpr int AT_SETS = 2;
constexpr int AT_THREADS = 128 * AT_SETS;
constexpr int AT_WARPS = AT_THREADS / 32;
constexpr int AT_CHUNK = 128;               // tokens per chunk (MMA M of the score product)
constexpr int AT_MAXG = 16;                 // query heads per KV head (MMA N of the score product)
constexpr int AT_HPW = AT_MAXG / AT_SETS;   // heads per warp
constexpr int AT_TPW = 32 / AT_SETS;        // tokens each warp copies per chunk
constexpr uint32_t AT_TMEM_COLS = 128;      // S: columns 0..15; O: 32..63 (dims 0..127), 64..95 (128..255)

// shared memory, offsets from a 1024-byte aligned base
constexpr uint32_t SM_K = 0;                         // A of S: [4 K blocks][128 tokens][128 B]
constexpr uint32_t SM_VS = SM_K + 4 * 16384;          // V staging: [128 tokens][512 B], 16-B chunks swizzled
constexpr uint32_t SM_VT = SM_VS + 128 * 512;         // A of O: [2 dim halves][2 K blocks][128 dims][128 B]
constexpr uint32_t SM_Q = SM_VT + 4 * 16384;          // B of S: [4 K blocks][16 heads][128 B]
constexpr uint32_t SM_P = SM_Q + 4 * 2048;            // B of O: [2 K blocks][32 rows][128 B]
constexpr uint32_t SM_CTRL = SM_P + 2 * 4096;
struct AtCtrl {
    uint64_t bar_s;                         // score product done
    uint64_t bar_o;                         // PV product done
    uint32_t tmem_base;
    int32_t abort;
    uint32_t wmax[AT_SETS][4][AT_HPW];      // [head set][lane quarter][head]: maxima of the chunk (score keys)
    float lsum[AT_SETS][4][AT_HPW];         // the same for the denominators (end of the row)
};
constexpr uint32_t AT_SMEM = SM_CTRL + sizeof(AtCtrl) + 1024;
static_assert(AT_SMEM <= 232448, "shared memory budget");

// Byte offset of 16-byte chunk c (0..7) of row `row` in a K-major tile with
// the 128-byte swizzle (rows of 128 B, 8-row atoms of 1024 B).
__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t c)
{
    return (row >> 3) * 1024u + (row & 7u) * 128u + ((c ^ (row & 7u)) << 4);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool fill)
{
    // a 16-byte copy, or 16 zero bytes (source size 0: nothing is read)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(fill ? 16 : 0)
                 : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// N (4 or 8) consecutive 32-bit columns of this warp's 32 TMEM lanes.
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[N])
{
    static_assert(N == 4 || N == 8, "x4 or x8");
    uint32_t u[N];
    if constexpr (N == 4) {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3])
                     : "r"(taddr)
                     : "memory");
    } else {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7])
                     : "r"(taddr)
                     : "memory");
    }
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] = __uint_as_float(u[i]);
}

// Every thread waits for the phase; false on every thread when any gave up.
__device__ __forceinline__ bool wait_all_threads(uint64_t *bar, uint32_t parity, volatile int *abort, uint64_t lim)
{
    const bool ok = mbar_wait(bar, parity, abort, lim);
    return __syncthreads_and(ok) != 0;
}

__global__ void __launch_bounds__(AT_THREADS, 1)
attend_kernel(const AttendParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sb = smem_u32(smem);
    AtCtrl &c = *reinterpret_cast<AtCtrl *>(smem + SM_CTRL);
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int lq = warp & 3, hs = warp >> 2;      // TMEM lane quarter, head set
    const int32_t r = blockIdx.x, g = blockIdx.y;

    if (t == 0) {
        mbar_init(&c.bar_s, 1);
        mbar_init(&c.bar_o, 1);
        c.abort = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(&c.tmem_base, AT_TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = c.tmem_base;
    volatile int *abort = &c.abort;
    const uint64_t lim = p.wait_limit_ns;

    const int group = p.hq / p.hkv;
    const int32_t b = r < p.rows ? p.row_req[r] : -1;
    const int32_t tok_r = r < p.rows ? p.row_token[r] : -1;
    const bool row_ok = r < p.rows && g < p.hkv && b >= 0 && b < p.num_reqs && tok_r >= 0 &&
                        static_cast<int64_t>(tok_r) < static_cast<int64_t>(p.max_pages) * p.page_tokens;
    if (!row_ok) {
        if (t == 0 && g == 0 && r < p.rows) record_error(p.status, ST_BAD_ROW);
    } else {
        const int32_t vis = (tok_r + 1) >> 2;           // complete index positions
        const int32_t tail0 = 4 * vis;                   // first token of the unfinished block
        // token stream: 4 tokens per selection slot (slots holding -1 or a bad
        // position contribute none), then the tail tokens tail0 .. tok_r
        const int32_t n_stream = 4 * p.k + (tok_r - tail0 + 1);
        const int32_t n_chunks = (n_stream + AT_CHUNK - 1) / AT_CHUNK;
        const int32_t *selr = p.sel + static_cast<int64_t>(r) * p.k;
        const __half *kc = static_cast<const __half *>(p.k_cache);
        const __half *vc = static_cast<const __half *>(p.v_cache);
        const int32_t *bt = p.block_table + static_cast<int64_t>(b) * p.max_pages;

        // queries of this KV head's group as the B operand (heads past the
        // group are zero rows)
        const __half *qr = static_cast<const __half *>(p.q) + (static_cast<int64_t>(r) * p.hq + g * group) * AT_D;
        for (int i = t; i < AT_MAXG * 32; i += AT_THREADS) {
            const int h = i >> 5, l = i & 31;                // head, 16-byte chunk of its 512-byte row
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (h < group) v = __ldg(reinterpret_cast<const uint4 *>(qr + h * AT_D) + l);
            *reinterpret_cast<uint4 *>(smem + SM_Q + (l >> 3) * 2048 + sw128(h, l & 7)) = v;
        }

        // Token lookups of the thread's softmax token 32 lq + lane of each
        // chunk, run ahead of the copies: while chunk c is copied, the page of
        // chunk c + 1 and the selection slot of chunk c + 2 are loaded, so no
        // copy waits for a dependent global load.
        const int32_t t_soft = lq * 32 + lane;
        auto slot_of = [&](int32_t ch) -> int32_t {          // selection slot value (or 0 past the slots)
            const int32_t st = ch * AT_CHUNK + t_soft;
            return ch < n_chunks && st < 4 * p.k ? selr[st >> 2] : 0;
        };
        auto pos_of = [&](int32_t ch, int32_t j) -> int32_t {  // token position, -1 = none (with the checks)
            const int32_t st = ch * AT_CHUNK + t_soft;
            if (ch >= n_chunks) return -1;
            if (st < 4 * p.k) {
                if (j >= 0 && j < vis) return 4 * j + (st & 3);
                if (j >= vis && (st & 3) == 0) record_error(p.status, ST_BAD_ROW);
                return -1;
            }
            return st < n_stream ? tail0 + (st - 4 * p.k) : -1;
        };
        auto page_of = [&](int32_t pos) -> int32_t { return pos >= 0 ? bt[pos >> p.page_shift] : -1; };
        int32_t pos_c = pos_of(0, slot_of(0));
        int32_t page_c = page_of(pos_c);
        int32_t slot_n = slot_of(1);
        // copy destinations: the warp's tokens T0 + j (T0 a multiple of 8, so
        // T & 7 = j & 7) in the K tile (16-byte chunk lane % 8 of K block
        // lane / 8) and in the V staging tile (chunk lane, swizzled by T & 7);
        // warp w copies tokens 32 lq + AT_TPW hs + j, j < AT_TPW (one 512-byte
        // K row and V row each, lane l taking 16-byte chunk l)
        const uint32_t T0 = static_cast<uint32_t>(lq * 32 + hs * AT_TPW);
        const uint32_t k_dst0 = sb + SM_K + static_cast<uint32_t>(lane >> 3) * 16384u + (T0 >> 3) * 1024u;
        const uint32_t v_dst0 = sb + SM_VS + T0 * 512u;
        const __half *kc_l = kc + g * AT_D + lane * 8;     // this lane's 16 bytes of KV head g
        const __half *vc_l = vc + g * AT_D + lane * 8;
        const int64_t line_elems = static_cast<int64_t>(p.hkv) * AT_D;
        // gather of chunk ch (the chunks in order); returns whether the
        // thread's softmax token is live
        auto gather = [&](int32_t ch) -> bool {
            int32_t line_mine = -1;                        // page-token row of the cache, -1 = none
            if (pos_c >= 0) {
                if (page_c >= 0 && page_c < p.num_pages) line_mine = page_c * p.page_tokens + (pos_c & (p.page_tokens - 1));
                else record_error(p.status, ST_BAD_PAGE);
            }
#pragma unroll
            for (int j = 0; j < AT_TPW; ++j) {
                const int32_t line = __shfl_sync(0xffffffffu, line_mine, hs * AT_TPW + j);
                const int64_t off = static_cast<int64_t>(line < 0 ? 0 : line) * line_elems;
                const uint32_t jj = static_cast<uint32_t>(j & 7);
                cp_async16(k_dst0 + (j >> 3) * 1024u + jj * 128u + (((static_cast<uint32_t>(lane) & 7u) ^ jj) << 4),
                           kc_l + off, line >= 0);
                cp_async16(v_dst0 + static_cast<uint32_t>(j) * 512u + ((static_cast<uint32_t>(lane) ^ jj) << 4),
                           vc_l + off, line >= 0);
            }
            pos_c = pos_of(ch + 1, slot_n);
            page_c = page_of(pos_c);                       // in flight until the next call
            slot_n = slot_of(ch + 2);
            return line_mine >= 0;
        };

        // this thread's heads AT_HPW hs .. + AT_HPW - 1: output dims d0 = 32 lq + lane
        // and d0 + 128, the running maximum and rescale (the same in every
        // thread of the head set) and its share of the denominators
        float o_lo[AT_HPW], o_hi[AT_HPW], m_run[AT_HPW], alpha[AT_HPW], l_part[AT_HPW];
#pragma unroll
        for (int h = 0; h < AT_HPW; ++h) {
            o_lo[h] = o_hi[h] = 0.0f;
            m_run[h] = -INFINITY;
            alpha[h] = 0.0f;
            l_part[h] = 0.0f;
        }
        const uint32_t taddr = tmem + (static_cast<uint32_t>(lq * 32) << 16);
        constexpr uint32_t idesc_s = umma_idesc_f16_f32(AT_CHUNK, AT_MAXG);
        constexpr uint32_t idesc_o = umma_idesc_f16_f32(128, 2 * AT_MAXG);
        // output update with chunk c's PV product (alpha: that chunk's rescale)
        // (columns 32 + 32 half + head for p_hi, + 16 for p_lo)
        auto take_o = [&]() {
            float a[AT_HPW], bq[AT_HPW];
            const uint32_t hc = static_cast<uint32_t>(AT_HPW * hs);
            tmem_ld_cols(taddr + 32u + hc, a);
            tmem_ld_cols(taddr + 48u + hc, bq);
#pragma unroll
            for (int h = 0; h < AT_HPW; ++h) o_lo[h] = fmaf(o_lo[h], alpha[h], a[h] + bq[h]);
            tmem_ld_cols(taddr + 64u + hc, a);
            tmem_ld_cols(taddr + 80u + hc, bq);
#pragma unroll
            for (int h = 0; h < AT_HPW; ++h) o_hi[h] = fmaf(o_hi[h], alpha[h], a[h] + bq[h]);
        };

        bool live = n_chunks > 0 ? gather(0) : false;
        uint32_t ph = 0;
        bool ok = true;
        for (int32_t ch = 0; ch < n_chunks; ++ch) {
            // 1. the chunk's K and V rows (and, first time, Q) are in shared memory
            cp_async_wait_all();
            fence_proxy_async_smem();
            __syncthreads();
            // 2. S^T = K . Q^T
            if (t == 0) {
                tc_fence_after();
                const uint64_t a0 = sw128_kmajor_desc(sb + SM_K), b0 = sw128_kmajor_desc(sb + SM_Q);
#pragma unroll
                for (int kk = 0; kk < AT_D / 16; ++kk) {
                    const uint32_t off = static_cast<uint32_t>((kk & 3) * 32);
                    umma_f16(tmem, a0 + (((kk >> 2) * 16384u + off) >> 4), b0 + (((kk >> 2) * 2048u + off) >> 4),
                             idesc_s, kk > 0 ? 1u : 0u);
                }
                umma_commit(&c.bar_s);
            }
            // 3. the previous chunk's PV product into the output (V^T and P are free after it)
            if (ch > 0) {
                if (!wait_all_threads(&c.bar_o, (ph - 1) & 1u, abort, lim)) { ok = false; break; }
                tc_fence_after();
                take_o();
            }
            // 4. V^T: 8 x 8 blocks (8 tokens x 8 dims), four per instruction.
            //    Warp w moves dims 32 (w % 8) .. + 31 (16-byte chunks 4 (w % 8) + i
            //    of the staging rows, i = lane / 8) of the 8-token blocks
            //    tb = w / 8, w / 8 + AT_WARPS / 8, ...; lane l addresses row
            //    l % 8 of matrix l / 8.
            {
                const uint32_t tj = static_cast<uint32_t>(lane & 7);
                const uint32_t db = static_cast<uint32_t>((warp & 7) * 4 + (lane >> 3));   // source chunk (dims 8 db ..)
                const uint32_t src0 = sb + SM_VS + tj * 512u + ((db ^ tj) << 4);    // token 8 tb + tj: + tb * 4 KiB
                const uint32_t D = db * 8u + tj;                                     // destination row (dim)
                const uint32_t dst0 = sb + SM_VT + (D >> 7) * 32768u + ((D & 127u) >> 3) * 1024u + tj * 128u;
#pragma unroll
                for (int tb = warp >> 3; tb < AT_CHUNK / 8; tb += AT_WARPS / 8) {
                    uint32_t x0, x1, x2, x3;
                    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                                 : "=r"(x0), "=r"(x1), "=r"(x2), "=r"(x3)
                                 : "r"(src0 + static_cast<uint32_t>(tb) * 4096u));
                    const uint32_t dst = dst0 + static_cast<uint32_t>(tb >> 3) * 16384u +
                                         (((static_cast<uint32_t>(tb) & 7u) ^ tj) << 4);
                    asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(x0),
                                 "r"(x1), "r"(x2), "r"(x3)
                                 : "memory");
                }
            }
            // 5. softmax of the chunk (token t_soft, this warp's heads)
            if (!wait_all_threads(&c.bar_s, ph & 1u, abort, lim)) { ok = false; break; }
            tc_fence_after();
            float s[AT_HPW];
            tmem_ld_cols(taddr + static_cast<uint32_t>(AT_HPW * hs), s);
#pragma unroll
            for (int h = 0; h < AT_HPW; ++h) {
                s[h] = live ? s[h] * p.scale : -INFINITY;
                const uint32_t kmax = __reduce_max_sync(0xffffffffu, score_key(s[h]));
                if (lane == 0) c.wmax[hs][lq][h] = kmax;
            }
            __syncthreads();
            // the next chunk's rows: K and the V staging are free (S is done,
            // every warp has finished its part of V^T), so the copies run
            // under this chunk's softmax, PV product and output update
            const bool live_next = ch + 1 < n_chunks ? gather(ch + 1) : false;
#pragma unroll
            for (int h = 0; h < AT_HPW; ++h) {
                uint32_t km = c.wmax[hs][0][h];
#pragma unroll
                for (int q = 1; q < 4; ++q) km = max(km, c.wmax[hs][q][h]);
                const float m_new = fmaxf(m_run[h], key_score(km));
                alpha[h] = m_run[h] > -INFINITY ? __expf(m_run[h] - m_new) : 0.0f;
                m_run[h] = m_new;
            }
            // P rows h (hi) and 16 + h (lo), column t_soft: K block t_soft / 64, element t_soft % 64
            const uint32_t cb = static_cast<uint32_t>((t_soft & 63) >> 3), eo = static_cast<uint32_t>(t_soft & 7) * 2;
            uint8_t *pb = smem + SM_P + (t_soft >> 6) * 4096;
#pragma unroll
            for (int h8 = 0; h8 < AT_HPW; ++h8) {
                const int h = hs * AT_HPW + h8;
                const float m_new = m_run[h8];
                const float e = (live && m_new > -INFINITY) ? __expf(s[h8] - m_new) : 0.0f;
                l_part[h8] = fmaf(l_part[h8], alpha[h8], e);
                const __half e_hi = __float2half_rn(e);
                const __half e_lo = __float2half_rn(e - __half2float(e_hi));
                *reinterpret_cast<__half *>(pb + sw128(h, cb) + eo) = e_hi;
                *reinterpret_cast<__half *>(pb + sw128(16 + h, cb) + eo) = e_lo;
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncthreads();
            // 6. O^T (this chunk's share, fresh accumulators) = V^T . P^T
            if (t == 0) {
                tc_fence_after();
                const uint64_t b0 = sw128_kmajor_desc(sb + SM_P);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const uint64_t a0 = sw128_kmajor_desc(sb + SM_VT + half * 32768u);
#pragma unroll
                    for (int kk = 0; kk < AT_CHUNK / 16; ++kk) {
                        const uint32_t off = static_cast<uint32_t>((kk & 3) * 32);
                        umma_f16(tmem + 32u + 32u * half, a0 + (((kk >> 2) * 16384u + off) >> 4),
                                 b0 + (((kk >> 2) * 4096u + off) >> 4), idesc_o, kk > 0 ? 1u : 0u);
                    }
                }
                umma_commit(&c.bar_o);
            }
            ++ph;
            live = live_next;
        }
        if (ok && n_chunks > 0) {
            if (wait_all_threads(&c.bar_o, (ph - 1) & 1u, abort, lim)) {
                tc_fence_after();
                take_o();
            } else {
                ok = false;
            }
        }
        cp_async_wait_all();
        // 8. denominators over the CTA, then the output
#pragma unroll
        for (int h = 0; h < AT_HPW; ++h) {
            float v = l_part[h];
#pragma unroll
            for (int o2 = 16; o2 > 0; o2 >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o2);
            if (lane == 0) c.lsum[hs][lq][h] = v;
        }
        __syncthreads();
        if (ok) {
            const int32_t d0 = lq * 32 + lane;
#pragma unroll
            for (int h8 = 0; h8 < AT_HPW; ++h8) {
                const int h = hs * AT_HPW + h8;
                if (h < group) {
                    const float l = (c.lsum[hs][0][h8] + c.lsum[hs][1][h8]) + (c.lsum[hs][2][h8] + c.lsum[hs][3][h8]);
                    const float inv = l > 0.0f ? 1.0f / l : 0.0f;
                    float *out = p.out + (static_cast<int64_t>(r) * p.hq + g * group + h) * AT_D;
                    out[d0] = o_lo[h8] * inv;
                    out[d0 + 128] = o_hi[h8] * inv;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (c.abort && t == 0) record_error(p.status, ST_TIMEOUT);
    if (warp == 0) tmem_dealloc(tmem, AT_TMEM_COLS);
}

}  // namespace

size_t attend_smem_bytes() { return AT_SMEM; }

int launch_attend(const AttendParams &p, void *stream)
{
    static std::mutex mu;
    static bool done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return static_cast<int>(cudaErrorInvalidDevice);
    {
        std::lock_guard<std::mutex> lk(mu);
        if (!done[dev]) {
            const cudaError_t e = cudaFuncSetAttribute(attend_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       static_cast<int>(AT_SMEM));
            if (e != cudaSuccess) return static_cast<int>(e);
            done[dev] = true;
        }
    }
    void *args[] = {const_cast<AttendParams *>(&p)};
    return launch_kernel(reinterpret_cast<const void *>(&attend_kernel), dim3(p.rows, p.hkv), dim3(AT_THREADS),
                         AT_SMEM, static_cast<cudaStream_t>(stream), false, args);
}

}  // namespace qsa
