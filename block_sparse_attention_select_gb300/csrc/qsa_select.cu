// Exact top-k selector: one CTA per query row.
//
// A score becomes key32 = score_key(score) (larger score -> larger key) and an
// element's full key is (key32, ~position): larger full key = higher score,
// then lower position, the exact lexicographic order with its deterministic
// tie rule.  The row's candidates are brought into shared memory, the k-th
// largest key is found by radix select with 11-bit digits taken over the
// live key range (so the bins stay evenly filled whatever the score scale),
// ties at the cut are settled on ~position, and the winners are ordered by a
// counting sort on the top bits of (key32 - cut) followed by small in-bucket
// sorts.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "qsa_device.cuh"
#include "qsa_internal.h"

namespace qsa {
namespace {

constexpr int NT = 512;               // threads per row
constexpr int NBINS = 2048;           // 11-bit digits
constexpr int SMALL_BUCKET = 16;      // buckets up to this size: one thread sorts them

struct SelShared {
    uint32_t hist[NBINS];
    uint32_t bstart[NBINS];
    uint32_t wtot[32];
    uint32_t red_min[32], red_max[32];
    uint32_t cut_digit, cut_above, count, total, taken, nbig, flag, pad_;
    uint32_t big[NBINS / 4];          // buckets needing a warp sort (at most k / 17 <= 482)
};

// ---------------------------------------------------------------- helpers --

__device__ __forceinline__ void clear_hist(SelShared &sh)
{
    for (int i = threadIdx.x; i < NBINS; i += NT) sh.hist[i] = 0;
    __syncthreads();
}

// Digit d holding the k_rem-th largest element counted in sh.hist (bins in
// ascending digit order); sets sh.cut_digit and sh.cut_above (elements in
// higher digits).  Requires 1 <= k_rem <= total count.
__device__ __forceinline__ void find_cut(SelShared &sh, uint32_t k_rem)
{
    const int t = threadIdx.x;
    uint32_t c[4], sum = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        c[i] = sh.hist[NBINS - 1 - (4 * t + i)];
        sum += c[i];
    }
    uint32_t before = block_excl_scan<NT>(sum, sh.wtot, nullptr);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (before < k_rem && k_rem <= before + c[i]) {
            sh.cut_digit = static_cast<uint32_t>(NBINS - 1 - (4 * t + i));
            sh.cut_above = before;
        }
        before += c[i];
    }
    __syncthreads();
}

__device__ __forceinline__ int span_shift(uint32_t span)
{
    const int bits = span ? 32 - __clz(span) : 0;      // span < 2^bits
    return bits > 11 ? bits - 11 : 0;
}

__device__ void block_minmax(SelShared &sh, uint32_t lo, uint32_t hi, uint32_t &out_lo, uint32_t &out_hi)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if (lane == 0) { sh.red_min[wid] = lo; sh.red_max[wid] = hi; }
    __syncthreads();
    if (wid == 0) {
        lo = lane < NT / 32 ? sh.red_min[lane] : 0xffffffffu;
        hi = lane < NT / 32 ? sh.red_max[lane] : 0u;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
            hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
        }
        if (lane == 0) { sh.red_min[0] = lo; sh.red_max[0] = hi; }
    }
    __syncthreads();
    out_lo = sh.red_min[0];
    out_hi = sh.red_max[0];
    __syncthreads();
}

// k_rem-th largest of {val(i) : pred(i), i < n}, every such value lying in
// [lo, hi] (n_in_range of them).  Returns the value; k_rem_out = its rank
// among the elements equal to it (1-based), eq_out = how many equal it.
template <typename Val, typename Pred>
__device__ uint32_t kth_largest(SelShared &sh, int32_t n, uint32_t k_rem, uint32_t lo, uint32_t hi,
                                uint32_t n_in_range, Val val, Pred pred, uint32_t &k_rem_out,
                                uint32_t &eq_out)
{
    uint32_t eq = n_in_range;
    while (lo != hi) {
        const int shift = span_shift(hi - lo);
        clear_hist(sh);
        for (int32_t i = threadIdx.x; i < n; i += NT) {
            if (!pred(i)) continue;
            const uint32_t v = val(i);
            if (v >= lo && v <= hi) atomicAdd(&sh.hist[(v - lo) >> shift], 1u);
        }
        __syncthreads();
        find_cut(sh, k_rem);
        const uint32_t d = sh.cut_digit;
        k_rem -= sh.cut_above;
        eq = sh.hist[d];
        const uint32_t nlo = lo + (d << shift);
        const uint64_t nhi = static_cast<uint64_t>(nlo) + ((1ull << shift) - 1);
        hi = static_cast<uint32_t>(min(static_cast<uint64_t>(hi), nhi));
        lo = nlo;
        __syncthreads();
        if (shift == 0) break;
    }
    k_rem_out = k_rem;
    eq_out = eq;
    return lo;
}

// In-place descending sort of a[0, m) by one warp: bitonic network in the
// variant whose comparators all point the same way, so positions >= m act as
// -infinity padding and are never touched.
__device__ void warp_sort_desc(uint64_t *a, int32_t m)
{
    const int lane = threadIdx.x & 31;
    int32_t M = 1;
    while (M < m) M <<= 1;
    for (int32_t size = 2; size <= M; size <<= 1) {
        const int32_t half = size >> 1;
        for (int32_t i = lane; i < (M >> 1); i += 32) {
            const int32_t blk = i / half, off = i % half;
            const int32_t x = blk * size + off, y = blk * size + size - 1 - off;
            if (y < m) {
                const uint64_t u = a[x], v = a[y];
                if (u < v) { a[x] = v; a[y] = u; }
            }
        }
        __syncwarp();
        for (int32_t stride = half >> 1; stride > 0; stride >>= 1) {
            for (int32_t i = lane; i < (M >> 1); i += 32) {
                const int32_t x = 2 * stride * (i / stride) + (i % stride), y = x + stride;
                if (y < m) {
                    const uint64_t u = a[x], v = a[y];
                    if (u < v) { a[x] = v; a[y] = u; }
                }
            }
            __syncwarp();
        }
    }
}

// Selects the top kk of the n elements (keys, inv) in shared memory and
// writes them, ordered, into out64 (as (key32 << 32) | inv).
__device__ void select_and_sort(SelShared &sh, const uint32_t *keys, const uint32_t *inv, int32_t n,
                                int32_t kk, uint64_t *out64)
{
    if (kk <= 0) return;
    uint32_t kmin = 0xffffffffu, kmax = 0u;
    for (int32_t i = threadIdx.x; i < n; i += NT) {
        kmin = min(kmin, keys[i]);
        kmax = max(kmax, keys[i]);
    }
    block_minmax(sh, kmin, kmax, kmin, kmax);

    uint32_t T = kmin, U = 0;       // selected: key > T, or key == T and inv >= U
    if (kk < n) {
        uint32_t k_rem, eq;
        T = kth_largest(sh, n, static_cast<uint32_t>(kk), kmin, kmax, static_cast<uint32_t>(n),
                        [&](int32_t i) { return keys[i]; }, [&](int32_t) { return true; }, k_rem, eq);
        if (eq > k_rem) {
            // cut score tied: keep the k_rem lowest positions (largest ~position)
            uint32_t imin = 0xffffffffu, imax = 0u;
            for (int32_t i = threadIdx.x; i < n; i += NT)
                if (keys[i] == T) { imin = min(imin, inv[i]); imax = max(imax, inv[i]); }
            block_minmax(sh, imin, imax, imin, imax);
            uint32_t k2, eq2;
            U = kth_largest(sh, n, k_rem, imin, imax, eq, [&](int32_t i) { return inv[i]; },
                            [&](int32_t i) { return keys[i] == T; }, k2, eq2);
        }
    }
    auto selected = [&](int32_t i) { const uint32_t k = keys[i]; return k > T || (k == T && inv[i] >= U); };

    // counting sort on the top 11 bits of (key - T), descending
    const int shift = span_shift(kmax - T);
    clear_hist(sh);
    for (int32_t i = threadIdx.x; i < n; i += NT)
        if (selected(i)) atomicAdd(&sh.hist[NBINS - 1 - ((keys[i] - T) >> shift)], 1u);
    __syncthreads();
    {   // bstart[b] = elements in buckets before b (bucket 0 = largest keys)
        const int t = threadIdx.x;
        uint32_t c[4], sum = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) { c[i] = sh.hist[4 * t + i]; sum += c[i]; }
        uint32_t before = block_excl_scan<NT>(sum, sh.wtot, nullptr);
#pragma unroll
        for (int i = 0; i < 4; ++i) { sh.bstart[4 * t + i] = before; before += c[i]; }
        if (t == 0) sh.nbig = 0;
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 4; ++i) sh.hist[4 * t + i] = sh.bstart[4 * t + i];   // cursors
        __syncthreads();
    }
    for (int32_t i = threadIdx.x; i < n; i += NT) {
        if (!selected(i)) continue;
        const uint32_t b = NBINS - 1 - ((keys[i] - T) >> shift);
        const uint32_t pos = atomicAdd(&sh.hist[b], 1u);
        out64[pos] = (static_cast<uint64_t>(keys[i]) << 32) | inv[i];
    }
    __syncthreads();
    // in-bucket order: small buckets by one thread each, larger ones by a warp
    for (int b = threadIdx.x; b < NBINS; b += NT) {
        const uint32_t s0 = sh.bstart[b], m = sh.hist[b] - s0;
        if (m <= 1) continue;
        if (m > SMALL_BUCKET) {
            sh.big[atomicAdd(&sh.nbig, 1u)] = b;
            continue;
        }
        uint64_t *a = out64 + s0;
        for (uint32_t x = 1; x < m; ++x) {
            const uint64_t v = a[x];
            uint32_t y = x;
            while (y > 0 && a[y - 1] < v) { a[y] = a[y - 1]; --y; }
            a[y] = v;
        }
    }
    __syncthreads();
    for (uint32_t q = threadIdx.x >> 5; q < sh.nbig; q += NT / 32) {
        const uint32_t b = sh.big[q];
        warp_sort_desc(out64 + sh.bstart[b], static_cast<int32_t>(sh.hist[b] - sh.bstart[b]));
    }
    __syncthreads();
}

__device__ void write_row(const SelectParams &p, int32_t r, const uint64_t *buf, int32_t kk)
{
    int32_t *oi = p.out_idx + static_cast<int64_t>(r) * p.k;
    float *ov = p.out_val ? p.out_val + static_cast<int64_t>(r) * p.k : nullptr;
    for (int32_t i = threadIdx.x; i < p.k; i += NT) {
        if (i < kk) {
            const uint64_t e = buf[i];
            oi[i] = static_cast<int32_t>(~static_cast<uint32_t>(e));
            if (ov) ov[i] = key_score(static_cast<uint32_t>(e >> 32));
        } else {
            oi[i] = -1;
            if (ov) ov[i] = -__int_as_float(0x7f800000);
        }
    }
}

// Streaming narrowing over a long row in global memory (fixed 11/11/10-bit
// digits of key32): stops as soon as every element at or above the current
// cut digit fits in shared memory (gathers them and returns their count), or
// returns -1 with the exact cut key when ties keep it too large.
__device__ __forceinline__ int level_shift(int lv) { return lv == 0 ? 21 : (lv == 1 ? 10 : 0); }
__device__ __forceinline__ uint32_t level_mask(int lv) { return lv < 2 ? 0x7FFu : 0x3FFu; }

__device__ int32_t stream_narrow(SelShared &sh, const float *__restrict__ row, int32_t n, uint32_t k,
                                 int32_t cap, uint32_t *keys, uint32_t *inv, uint32_t &T_out,
                                 uint32_t &k_rem_out, bool gather)
{
    uint32_t prefix = 0, pmask = 0, k_rem = k, above = 0;
    for (int lv = 0; lv < 3; ++lv) {
        clear_hist(sh);
        for (int32_t i = threadIdx.x; i < n; i += NT) {
            const uint32_t key = score_key(__ldcg(row + i));
            if ((key & pmask) == prefix) atomicAdd(&sh.hist[(key >> level_shift(lv)) & level_mask(lv)], 1u);
        }
        __syncthreads();
        find_cut(sh, k_rem);
        const uint32_t d = sh.cut_digit;
        const uint32_t eq = sh.hist[d];
        k_rem -= sh.cut_above;
        above += sh.cut_above;
        prefix |= d << level_shift(lv);
        pmask |= level_mask(lv) << level_shift(lv);
        __syncthreads();
        if (gather && above + eq <= static_cast<uint32_t>(cap)) {
            if (threadIdx.x == 0) sh.count = 0;
            __syncthreads();
            for (int32_t i = threadIdx.x; i < n; i += NT) {
                const uint32_t key = score_key(__ldcg(row + i));
                if ((key & pmask) >= prefix) {
                    const uint32_t slot = atomicAdd(&sh.count, 1u);
                    keys[slot] = key;
                    inv[slot] = ~static_cast<uint32_t>(i);
                }
            }
            __syncthreads();
            return static_cast<int32_t>(sh.count);
        }
    }
    T_out = prefix;
    k_rem_out = k_rem;
    return -1;
}

// Everything above the exact cut key T, then the k_rem lowest positions that
// hold T, in position order.
__device__ int32_t gather_cut_in_order(SelShared &sh, const float *__restrict__ row, int32_t n,
                                       uint32_t T, uint32_t k_rem, uint32_t *keys, uint32_t *inv)
{
    if (threadIdx.x == 0) { sh.count = 0; sh.taken = 0; }
    __syncthreads();
    for (int32_t base = 0; base < n; base += NT) {
        const int32_t i = base + threadIdx.x;
        const uint32_t key = i < n ? score_key(__ldcg(row + i)) : 0u;
        if (i < n && key > T) {
            const uint32_t slot = atomicAdd(&sh.count, 1u);
            keys[slot] = key;
            inv[slot] = ~static_cast<uint32_t>(i);
        }
        const uint32_t tie = (i < n && key == T) ? 1u : 0u;
        const uint32_t taken = sh.taken;
        const uint32_t rank = block_excl_scan<NT>(tie, sh.wtot, &sh.total);
        if (tie && taken + rank < k_rem) {
            const uint32_t slot = atomicAdd(&sh.count, 1u);
            keys[slot] = key;
            inv[slot] = ~static_cast<uint32_t>(i);
        }
        __syncthreads();
        if (threadIdx.x == 0) sh.taken = taken + sh.total;
        __syncthreads();
        if (sh.taken >= k_rem) {
            for (int32_t j = base + NT + threadIdx.x; j < n; j += NT) {
                const uint32_t kj = score_key(__ldcg(row + j));
                if (kj > T) {
                    const uint32_t slot = atomicAdd(&sh.count, 1u);
                    keys[slot] = kj;
                    inv[slot] = ~static_cast<uint32_t>(j);
                }
            }
            break;
        }
    }
    __syncthreads();
    return static_cast<int32_t>(sh.count);
}

// Plain FP32 scores of row r, written to `row` (multiply then add, head by
// head, in the order of the definition).  Used only for rows whose candidate
// list the filter could not certify; qf is shared scratch for H * 128 floats.
__device__ void simt_score_row(const SelectParams &p, int32_t r, int32_t V, float *row, float *qf)
{
    const int32_t H = p.H;
    for (int32_t i = threadIdx.x; i < H * HEAD_DIM; i += NT)
        qf[i] = __half2float(__ushort_as_half(p.q[static_cast<int64_t>(r) * H * HEAD_DIM + i]));
    __syncthreads();
    const int32_t *bt = p.block_table + static_cast<int64_t>(p.row_req[r]) * p.max_pages;
    for (int32_t j = threadIdx.x; j < V; j += NT) {
        const int32_t pid = __ldg(bt + j / p.page_pos);
        float s = 0.0f;
        if (pid >= 0 && pid < p.num_pages) {
            const uint4 *kr = reinterpret_cast<const uint4 *>(
                p.k_cache + (static_cast<int64_t>(pid) * p.page_pos + j % p.page_pos) * HEAD_DIM);
            for (int32_t h = 0; h < H; ++h) {
                float dot = 0.0f;
#pragma unroll 1
                for (int t = 0; t < HEAD_DIM / 8; ++t) {
                    const uint4 kv = __ldg(kr + t);
                    const __half *kh = reinterpret_cast<const __half *>(&kv);
                    const float *qv = qf + h * HEAD_DIM + t * 8;
#pragma unroll
                    for (int d = 0; d < 8; ++d) dot = __fadd_rn(dot, __fmul_rn(qv[d], __half2float(kh[d])));
                }
                s = __fadd_rn(s, __fmul_rn(__ldg(p.w + static_cast<int64_t>(r) * H + h), dot > 0.0f ? dot : 0.0f));
            }
        } else {
            record_error(p.status, ST_BAD_PAGE);   // as on the tensor path: the page reads as zeros
        }
        row[j] = s + 0.0f;
    }
    __syncthreads();
}

__global__ void __launch_bounds__(NT, 2)
select_kernel(const SelectParams p)
{
    extern __shared__ __align__(16) uint8_t smem_raw[];
    SelShared &sh = *reinterpret_cast<SelShared *>(smem_raw);
    uint64_t *out64 = reinterpret_cast<uint64_t *>(smem_raw + sizeof(SelShared));
    uint32_t *keys = reinterpret_cast<uint32_t *>(out64 + (p.mode == SEL_THRESH ? 0 : p.k));
    uint32_t *inv = keys + p.smem_cap;

    const int32_t r = blockIdx.x;
    if (r >= p.R) return;
    int32_t V = p.row_vis[r];
    if (V < 0 || V > p.max_len) {
        if (threadIdx.x == 0) record_error(p.status, ST_BAD_ROW);
        V = static_cast<int32_t>(max(static_cast<int64_t>(0), min(static_cast<int64_t>(V), p.max_len)));
    }

    if (p.mode == SEL_THRESH) {
        // tau_r from the sampled scores of row r (columns [0, n_s) of its sample row)
        const int32_t tiles = (V + TILE_M - 1) / TILE_M;
        int32_t n_s = 0;
        if (tiles > 0) {
            const int32_t t_last = ((tiles - 1) / p.sample_stride) * p.sample_stride;
            n_s = (t_last / p.sample_stride) * TILE_M + min(TILE_M, V - t_last * TILE_M);
        }
        float tau = -__int_as_float(0x7f800000);
        if (V > p.cap && n_s > 0) {
            const double want = static_cast<double>(p.oversample) * p.k * n_s / V;
            int32_t m = static_cast<int32_t>(ceil(want)) + 8;
            m = max(1, min(m, n_s));
            const float *row = p.logits + static_cast<int64_t>(r) * p.ld;
            uint32_t T;
            if (n_s <= p.smem_cap) {
                uint32_t lo = 0xffffffffu, hi = 0u;
                for (int32_t i = threadIdx.x; i < n_s; i += NT) {
                    const uint32_t kv = score_key(__ldcg(row + i));
                    keys[i] = kv;
                    lo = min(lo, kv);
                    hi = max(hi, kv);
                }
                block_minmax(sh, lo, hi, lo, hi);
                uint32_t k2, eq2;
                T = kth_largest(sh, n_s, static_cast<uint32_t>(m), lo, hi, static_cast<uint32_t>(n_s),
                                [&](int32_t i) { return keys[i]; }, [&](int32_t) { return true; }, k2, eq2);
            } else {
                uint32_t k2;
                stream_narrow(sh, row, n_s, static_cast<uint32_t>(m), 0, nullptr, nullptr, T, k2, false);
            }
            tau = key_score(T);
        }
        if (threadIdx.x == 0) p.tau[r] = tau;
        return;
    }

    int32_t n = -1;
    const int32_t kk_target = min(p.k, V);
    const float *row = p.logits + static_cast<int64_t>(r) * p.ld;
    if (p.mode == SEL_CAND) {
        // gather the candidate slots of the row's key tiles, in position order
        const int32_t ne = ((V + TILE_M - 1) / TILE_M) * 4;
        const uint8_t *cnt = p.cand_cnt + static_cast<int64_t>(r) * p.tiles_ld * 4;
        const uint2 *slots = p.cand + static_cast<int64_t>(r) * p.tiles_ld * 4 * CAND_SLOTS;
        const int32_t per = (ne + NT - 1) / NT;
        const int32_t e0 = min(ne, static_cast<int32_t>(threadIdx.x) * per), e1 = min(ne, e0 + per);
        uint32_t sum = 0;
        bool over = false;
        for (int32_t e = e0; e < e1; ++e) {
            const uint32_t c = cnt[e];
            over |= c > CAND_SLOTS;
            sum += min(c, static_cast<uint32_t>(CAND_SLOTS));
        }
        uint32_t base = block_excl_scan<NT>(sum, sh.wtot, &sh.total);
        const bool any_over = __syncthreads_or(over) != 0;
        const uint32_t total = sh.total;
        if (any_over || total < static_cast<uint32_t>(kk_target) || total > static_cast<uint32_t>(p.smem_cap)) {
            // the sample misled the threshold for this row: score it in full here
            if (threadIdx.x == 0) {
                p.row_flag[r] = 1;
                atomicExch(&p.plan->any_fallback, 1);
            }
            float *fb = p.fb_logits + static_cast<int64_t>(r) * p.max_len;
            simt_score_row(p, r, V, fb, reinterpret_cast<float *>(keys));
            row = fb;
        } else {
            if (threadIdx.x == 0) p.row_flag[r] = 0;
            for (int32_t e = e0; e < e1; ++e) {
                const uint32_t c = cnt[e];
                for (uint32_t s = 0; s < c; ++s) {
                    const uint2 v = slots[static_cast<int64_t>(e) * CAND_SLOTS + s];
                    keys[base] = score_key(__uint_as_float(v.x));
                    inv[base] = ~v.y;
                    ++base;
                }
            }
            __syncthreads();
            n = static_cast<int32_t>(total);
        }
    }
    if (n < 0) {
        if (V <= p.smem_cap) {
            for (int32_t i = threadIdx.x; i < V; i += NT) {
                keys[i] = score_key(__ldcg(row + i));
                inv[i] = ~static_cast<uint32_t>(i);
            }
            __syncthreads();
            n = V;
        } else {
            uint32_t T, k_rem;
            n = stream_narrow(sh, row, V, static_cast<uint32_t>(kk_target), p.smem_cap, keys, inv, T,
                              k_rem, true);
            if (n < 0) n = gather_cut_in_order(sh, row, V, T, k_rem, keys, inv);
        }
    }
    const int32_t kk = min(p.k, n);
    select_and_sort(sh, keys, inv, n, kk, out64);
    write_row(p, r, out64, kk);
}

}  // namespace

size_t select_smem_bytes(int32_t smem_cap)
{
    return sizeof(SelShared) + static_cast<size_t>(smem_cap) * 8;
}

int launch_select(const SelectParams &p, void *stream)
{
    const size_t smem = sizeof(SelShared) + static_cast<size_t>(p.mode == SEL_THRESH ? 0 : p.k) * 8 +
                        static_cast<size_t>(p.smem_cap) * 8;
    static size_t attr_bytes[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return static_cast<int>(cudaErrorInvalidDevice);
    if (smem > attr_bytes[dev]) {
        cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return static_cast<int>(e);
        attr_bytes[dev] = smem;
    }
    select_kernel<<<p.R, NT, smem, static_cast<cudaStream_t>(stream)>>>(p);
    return static_cast<int>(cudaGetLastError());
}

}  // namespace qsa
