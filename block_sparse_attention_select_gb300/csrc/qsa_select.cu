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

#include <algorithm>
#include <mutex>

#include "qsa_device.cuh"
#include "qsa_internal.h"

namespace qsa {
namespace {

constexpr int NT = 256;               // threads per row
constexpr int NBINS = 2048;           // 11-bit digits
constexpr int BPT = NBINS / NT;       // bins per thread in scans
constexpr int SMALL_BUCKET = 16;      // buckets up to this size: one thread sorts them
constexpr int SLACK = 512;            // room past k for the bucket holding the k-th element
constexpr uint32_t RANK_MAX = 32;     // buckets up to this size are ordered by rank counting

struct SelShared {
    uint32_t hist[NBINS];
    uint32_t bstart[NBINS];
    uint32_t wtot[32];
    uint32_t red_min[32], red_max[32];
    uint32_t cut_digit, cut_above, count, total, taken, nbig, flag, pad_;
    uint32_t big[512];                // buckets needing a warp sort
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
    uint32_t c[BPT], sum = 0;
#pragma unroll
    for (int i = 0; i < BPT; ++i) {
        c[i] = sh.hist[NBINS - 1 - (BPT * t + i)];
        sum += c[i];
    }
    uint32_t before = block_excl_scan<NT>(sum, sh.wtot, nullptr);
#pragma unroll
    for (int i = 0; i < BPT; ++i) {
        if (before < k_rem && k_rem <= before + c[i]) {
            sh.cut_digit = static_cast<uint32_t>(NBINS - 1 - (BPT * t + i));
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

// In-place descending sort of a[0, m) by NTHR threads (thread index tid):
// bitonic network in the variant whose comparators all point the same way, so
// positions >= m act as -infinity padding and are never touched.  Every block
// and stride is a power of two, so comparator indices are shifts and masks.
// BLOCK: the whole CTA sorts (barriers between stages), else one warp.
template <int NTHR, bool BLOCK>
__device__ __forceinline__ void bitonic_sort_desc(uint64_t *a, int32_t m, int tid)
{
    int lm = 0;
    while ((1 << lm) < m) ++lm;
    const int32_t npairs = (1 << lm) >> 1;
    auto sync = [] {
        if constexpr (BLOCK) __syncthreads();
        else __syncwarp();
    };
    for (int ls = 1; ls <= lm; ++ls) {                    // merge blocks of 2^ls
        const int lh = ls - 1;
        for (int32_t i = tid; i < npairs; i += NTHR) {
            const int32_t blk = i >> lh, off = i & ((1 << lh) - 1);
            const int32_t x = (blk << ls) + off, y = (blk << ls) + (1 << ls) - 1 - off;
            if (y < m) {
                const uint64_t u = a[x], v = a[y];
                if (u < v) { a[x] = v; a[y] = u; }
            }
        }
        sync();
        for (int lst = lh - 1; lst >= 0; --lst) {          // stride 2^lst
            for (int32_t i = tid; i < npairs; i += NTHR) {
                const int32_t x = ((i >> lst) << (lst + 1)) + (i & ((1 << lst) - 1)), y = x + (1 << lst);
                if (y < m) {
                    const uint64_t u = a[x], v = a[y];
                    if (u < v) { a[x] = v; a[y] = u; }
                }
            }
            sync();
        }
    }
}

__device__ void warp_sort_desc(uint64_t *a, int32_t m) { bitonic_sort_desc<32, false>(a, m, threadIdx.x & 31); }

// bstart[b] = elements in buckets before b (bucket 0 holds the largest keys);
// hist[] becomes the scatter cursors.
__device__ __forceinline__ void bucket_starts(SelShared &sh)
{
    const int t = threadIdx.x;
    uint32_t c[BPT], sum = 0;
#pragma unroll
    for (int i = 0; i < BPT; ++i) { c[i] = sh.hist[BPT * t + i]; sum += c[i]; }
    uint32_t before = block_excl_scan<NT>(sum, sh.wtot, nullptr);
#pragma unroll
    for (int i = 0; i < BPT; ++i) { sh.bstart[BPT * t + i] = before; before += c[i]; }
    if (t == 0) sh.nbig = 0;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < BPT; ++i) sh.hist[BPT * t + i] = sh.bstart[BPT * t + i];   // cursors
    __syncthreads();
}

// Descending sort of a[0, m), m <= 32, by one warp in registers.
__device__ __forceinline__ void warp_sort32_desc(uint64_t *a, int32_t m)
{
    const int lane = threadIdx.x & 31;
    uint64_t x = lane < m ? a[lane] : 0ull;          // 0 sorts last (real keys are > 0)
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const uint64_t y = __shfl_xor_sync(0xffffffffu, x, stride);
            const bool keep_max = ((lane & stride) == 0) == ((lane & size) == 0 || size == 32);
            x = keep_max ? (x > y ? x : y) : (x < y ? x : y);
        }
    }
    if (lane < m) a[lane] = x;
}

// Descending sort of N 64-bit keys held in registers (bitonic network,
// fully unrolled: no memory traffic, no divergence inside the network).
template <int N>
__device__ __forceinline__ void reg_sort_desc(uint64_t (&x)[N])
{
#pragma unroll
    for (int size = 2; size <= N; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
#pragma unroll
            for (int i = 0; i < N; ++i) {
                const int j = i ^ stride;
                if (j > i) {
                    const bool desc = (i & size) == 0;
                    const uint64_t a = x[i], b = x[j];
                    const bool swap = desc ? a < b : a > b;
                    x[i] = swap ? b : a;
                    x[j] = swap ? a : b;
                }
            }
        }
    }
}

template <int N>
__device__ __forceinline__ void small_sort(uint64_t *a, uint32_t m)
{
    uint64_t x[N];
#pragma unroll
    for (int i = 0; i < N; ++i) x[i] = static_cast<uint32_t>(i) < m ? a[i] : 0ull;   // 0 sorts last
    reg_sort_desc<N>(x);
#pragma unroll
    for (int i = 0; i < N; ++i)
        if (static_cast<uint32_t>(i) < m) a[i] = x[i];
}

// Orders every bucket b < nb in place (buckets were filled by scatter;
// hist[b] is its end): buckets of up to 16 by one thread with a register
// sorting network, larger ones by a warp.
__device__ void sort_buckets(SelShared &sh, uint64_t *out64, int nb)
{
    for (int b = threadIdx.x; b < nb; b += NT) {
        const uint32_t s0 = sh.bstart[b], m = sh.hist[b] - s0;
        if (m <= 1) continue;
        if (m > SMALL_BUCKET) {
            sh.big[atomicAdd(&sh.nbig, 1u)] = b;
            continue;
        }
        if (m <= 4) small_sort<4>(out64 + s0, m);
        else if (m <= 8) small_sort<8>(out64 + s0, m);
        else small_sort<16>(out64 + s0, m);
    }
    __syncthreads();
    for (uint32_t q = threadIdx.x >> 5; q < sh.nbig; q += NT / 32) {
        const uint32_t b = sh.big[q];
        const int32_t m = static_cast<int32_t>(sh.hist[b] - sh.bstart[b]);
        if (m <= 32) warp_sort32_desc(out64 + sh.bstart[b], m);
        else warp_sort_desc(out64 + sh.bstart[b], m);
    }
    __syncthreads();
}

// Top kk of the n elements in one counting-sort pass: buckets are the top 11
// bits of (key32 - min key); only the buckets down to the one holding the
// kk-th element are written to out64 (capacity out_cap) and ordered.
// Returns false, touching nothing, when those buckets would not fit.
__device__ bool bucket_topk(SelShared &sh, const uint32_t *keys, const uint32_t *inv, int32_t n,
                            int32_t kk, uint64_t *out64, int32_t out_cap, uint64_t *ranked)
{
    uint32_t kmin = 0xffffffffu, kmax = 0u;
    for (int32_t i = threadIdx.x; i < n; i += NT) {
        kmin = min(kmin, keys[i]);
        kmax = max(kmax, keys[i]);
    }
    block_minmax(sh, kmin, kmax, kmin, kmax);
    // Buckets over [lo, kmax].  When the buckets down to the cut span a much
    // smaller key range than the whole row (a long tail of low scores, or the
    // spike of exact zeros, below the top kk), count once more over that range
    // only, so that the buckets to be ordered are small.
    uint32_t lo = kmin, total = static_cast<uint32_t>(n);
    int shift = span_shift(kmax - lo);
    int bb;
    uint32_t need;
    for (int level = 0;; ++level) {
        clear_hist(sh);
        for (int32_t i = threadIdx.x; i < n; i += NT)
            if (keys[i] >= lo) atomicAdd(&sh.hist[NBINS - 1 - ((keys[i] - lo) >> shift)], 1u);
        __syncthreads();
        bucket_starts(sh);
        // boundary bucket: the one whose range [bstart, end) contains position kk - 1
        if (threadIdx.x == 0) sh.cut_digit = NBINS;
        __syncthreads();
        for (int b = threadIdx.x; b < NBINS; b += NT) {
            const uint32_t s0 = sh.bstart[b];
            const uint32_t e = (b + 1 < NBINS) ? sh.bstart[b + 1] : total;
            if (s0 < static_cast<uint32_t>(kk) && static_cast<uint32_t>(kk) <= e) sh.cut_digit = b;
        }
        __syncthreads();
        bb = static_cast<int>(sh.cut_digit);
        if (bb >= NBINS) return false;                                      // uniform
        need = (bb + 1 < NBINS) ? sh.bstart[bb + 1] : total;
        const uint32_t lo2 = lo + (static_cast<uint32_t>(NBINS - 1 - bb) << shift);
        const int shift2 = span_shift(kmax - lo2);
        if (level > 0 || shift == 0 || shift2 + 3 > shift) break;          // uniform
        lo = lo2;                          // every key >= lo2 lies in buckets <= bb: need of them
        shift = shift2;
        total = need;
        __syncthreads();
    }
    if (need > static_cast<uint32_t>(out_cap)) return false;   // uniform
    for (int32_t i = threadIdx.x; i < n; i += NT) {
        if (keys[i] < lo) continue;
        const uint32_t b = NBINS - 1 - ((keys[i] - lo) >> shift);
        if (b > static_cast<uint32_t>(bb)) continue;
        const uint32_t pos = atomicAdd(&sh.hist[b], 1u);
        out64[pos] = (static_cast<uint64_t>(keys[i]) << 32) | inv[i];
    }
    if (threadIdx.x == 0) sh.nbig = 0;
    __syncthreads();
    // Order inside buckets by rank counting: the thread of position p counts
    // the larger keys of its bucket.  Positions are handed out in bucket
    // order, so neighbouring threads scan the same bucket (no divergence);
    // buckets above RANK_MAX go to a warp sort instead.  keys/inv are dead
    // now, and `ranked` reuses their space.
    for (uint32_t pos = threadIdx.x; pos < need; pos += NT) {
        const uint64_t x = out64[pos];
        const uint32_t b = NBINS - 1 - ((static_cast<uint32_t>(x >> 32) - lo) >> shift);
        const uint32_t s0 = sh.bstart[b], e = sh.hist[b];
        if (e - s0 > RANK_MAX) {
            if (pos == s0) sh.big[atomicAdd(&sh.nbig, 1u)] = b;
            continue;
        }
        uint32_t rk = 0;
        for (uint32_t q = s0; q < e; ++q) rk += out64[q] > x;
        ranked[s0 + rk] = x;
    }
    __syncthreads();
    for (uint32_t q = threadIdx.x >> 5; q < sh.nbig; q += NT / 32) {
        const uint32_t b = sh.big[q];
        const uint32_t s0 = sh.bstart[b], m = sh.hist[b] - s0;
        warp_sort_desc(out64 + s0, static_cast<int32_t>(m));
        for (uint32_t t = threadIdx.x & 31; t < m; t += 32) ranked[s0 + t] = out64[s0 + t];
    }
    __syncthreads();
    return true;
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
    bucket_starts(sh);
    for (int32_t i = threadIdx.x; i < n; i += NT) {
        if (!selected(i)) continue;
        const uint32_t b = NBINS - 1 - ((keys[i] - T) >> shift);
        const uint32_t pos = atomicAdd(&sh.hist[b], 1u);
        out64[pos] = (static_cast<uint64_t>(keys[i]) << 32) | inv[i];
    }
    __syncthreads();
    sort_buckets(sh, out64, NBINS);
}

__device__ void write_row(const SelectParams &p, int32_t r, const uint64_t *buf, int32_t kk)
{
    int64_t ro = r;
    if (p.out_heads > 1) {                  // virtual row r = h * n + row -> output row row * H + h
        const int32_t n = p.R / p.out_heads;
        ro = static_cast<int64_t>(r % n) * p.out_heads + r / n;
    }
    int32_t *oi = p.out_idx + ro * p.k;
    float *ov = p.out_val ? p.out_val + ro * p.k : nullptr;
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

// A row of scores in global memory: element i at base[(i >> 7) * tile_stride
// + (i & 127)].  Dense logits are one contiguous run (tile_stride = TILE_M); a
// row the candidate selector re-scores lives in its own 128-float regions of
// the candidate array, TILE_M * R floats apart.
struct RowView {
    float *base;
    int64_t tile_stride;
    __device__ __forceinline__ float *at(int32_t i) const { return base + (i >> 7) * tile_stride + (i & 127); }
    __device__ __forceinline__ float ld(int32_t i) const { return __ldcg(at(i)); }
};

// Calls f(i, key32 of element i) for i = threadIdx.x, ... over [0, n) of the
// row, in some order.  A row whose base and tile stride are 16-byte multiples
// is read four elements per load, four loads in flight per thread (a 128-float
// tile holds whole groups of four); other rows element by element.
template <typename F>
__device__ __forceinline__ void for_each_key(const RowView row, int32_t n, F f)
{
    int32_t done = 0;
    if ((reinterpret_cast<uintptr_t>(row.base) & 15u) == 0 && (row.tile_stride & 3) == 0) {
        const int32_t n4 = n >> 2;
#pragma unroll 4
        for (int32_t v = threadIdx.x; v < n4; v += NT) {
            const int32_t i = v << 2;
            const float4 x = __ldcg(reinterpret_cast<const float4 *>(row.at(i)));
            f(i, score_key(x.x));
            f(i + 1, score_key(x.y));
            f(i + 2, score_key(x.z));
            f(i + 3, score_key(x.w));
        }
        done = n4 << 2;
    }
    for (int32_t i = done + threadIdx.x; i < n; i += NT) f(i, score_key(row.ld(i)));
}

// Streaming narrowing over a long row in global memory (fixed 11/11/10-bit
// digits of key32): stops as soon as every element at or above the current
// cut digit fits in shared memory (gathers them and returns their count), or
// returns -1 with the exact cut key when ties keep it too large.
__device__ __forceinline__ int level_shift(int lv) { return lv == 0 ? 21 : (lv == 1 ? 10 : 0); }
__device__ __forceinline__ uint32_t level_mask(int lv) { return lv < 2 ? 0x7FFu : 0x3FFu; }

__device__ int32_t stream_narrow(SelShared &sh, const RowView row, int32_t n, uint32_t k,
                                 int32_t cap, uint32_t *keys, uint32_t *inv, uint32_t &T_out,
                                 uint32_t &k_rem_out, bool gather)
{
    uint32_t prefix = 0, pmask = 0, k_rem = k, above = 0;
    for (int lv = 0; lv < 3; ++lv) {
        clear_hist(sh);
        const int sft = level_shift(lv);
        const uint32_t msk = level_mask(lv);
        for_each_key(row, n, [&](int32_t, uint32_t key) {
            if ((key & pmask) == prefix) atomicAdd(&sh.hist[(key >> sft) & msk], 1u);
        });
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
            for_each_key(row, n, [&](int32_t i, uint32_t key) {
                if ((key & pmask) >= prefix) {
                    const uint32_t slot = atomicAdd(&sh.count, 1u);
                    keys[slot] = key;
                    inv[slot] = ~static_cast<uint32_t>(i);
                }
            });
            __syncthreads();
            return static_cast<int32_t>(sh.count);
        }
    }
    T_out = prefix;
    k_rem_out = k_rem;
    return -1;
}

// A long row's top kk through a sampled threshold: the keys of every
// SAMPLE_TILES-th 128-score tile are staged, T = the m-th largest of them
// (m = w + 4 sqrt(w) + 8 with w = 1.5 kk n_s / V, the expected share of the
// top kk in the sample plus a margin), and one pass over the row gathers every
// key >= T.  When at least kk keys reach T, the kk-th largest key of the row
// is >= T, so the gathered keys hold the row's top kk: the result is exact.
// Returns their count, or -1 (nothing usable in keys / inv) when fewer than
// kk or more than cap reach T, or the sample does not fit.
constexpr int32_t SAMPLE_TILES = 16;

__device__ int32_t sample_gather(SelShared &sh, const RowView row, int32_t V, int32_t kk, int32_t cap,
                                 uint32_t *keys, uint32_t *inv)
{
    const int32_t tiles = (V + TILE_M - 1) / TILE_M;
    const int32_t nst = (tiles + SAMPLE_TILES - 1) / SAMPLE_TILES;
    const int32_t last = (nst - 1) * SAMPLE_TILES;
    const int32_t n_s = (nst - 1) * TILE_M + min(TILE_M, V - last * TILE_M);
    if (kk <= 0 || n_s > cap) return -1;                      // uniform
    // sampled element i: tile (i / 128) * SAMPLE_TILES, slot i % 128
    auto src = [&](int32_t i) { return ((i >> 7) * SAMPLE_TILES << 7) + (i & 127); };
    uint32_t kmin = 0xffffffffu, kmax = 0u;
    if ((reinterpret_cast<uintptr_t>(row.base) & 15u) == 0 && (row.tile_stride & 3) == 0) {
        for (int32_t v = threadIdx.x; v < (n_s >> 2); v += NT) {
            const float4 x = __ldcg(reinterpret_cast<const float4 *>(row.at(src(v << 2))));
            const uint32_t k4[4] = {score_key(x.x), score_key(x.y), score_key(x.z), score_key(x.w)};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                keys[(v << 2) + j] = k4[j];
                kmin = min(kmin, k4[j]);
                kmax = max(kmax, k4[j]);
            }
        }
        for (int32_t i = ((n_s >> 2) << 2) + threadIdx.x; i < n_s; i += NT) {
            const uint32_t kv = score_key(row.ld(src(i)));
            keys[i] = kv;
            kmin = min(kmin, kv);
            kmax = max(kmax, kv);
        }
    } else {
        for (int32_t i = threadIdx.x; i < n_s; i += NT) {
            const uint32_t kv = score_key(row.ld(src(i)));
            keys[i] = kv;
            kmin = min(kmin, kv);
            kmax = max(kmax, kv);
        }
    }
    block_minmax(sh, kmin, kmax, kmin, kmax);                 // its barriers also publish keys[]
    const float w = 1.5f * static_cast<float>(kk) * static_cast<float>(n_s) / static_cast<float>(V);
    const uint32_t m = static_cast<uint32_t>(min(static_cast<float>(n_s), ceilf(w + 4.0f * sqrtf(w)) + 8.0f));
    uint32_t k_rem, eq;
    const uint32_t T = kth_largest(sh, n_s, m, kmin, kmax, static_cast<uint32_t>(n_s),
                                   [&](int32_t i) { return keys[i]; }, [&](int32_t) { return true; }, k_rem, eq);
    if (threadIdx.x == 0) sh.count = 0;
    __syncthreads();                                          // the sample is dead: keys[] is reused
    for_each_key(row, V, [&](int32_t i, uint32_t key) {
        if (key >= T) {
            const uint32_t slot = atomicAdd(&sh.count, 1u);
            if (slot < static_cast<uint32_t>(cap)) {
                keys[slot] = key;
                inv[slot] = ~static_cast<uint32_t>(i);
            }
        }
    });
    __syncthreads();
    const uint32_t cnt = sh.count;
    __syncthreads();                                          // sh.count is reused by the caller
    if (cnt < static_cast<uint32_t>(kk) || cnt > static_cast<uint32_t>(cap)) return -1;
    return static_cast<int32_t>(cnt);
}

// Everything above the exact cut key T, then the k_rem lowest positions that
// hold T, in position order.
__device__ int32_t gather_cut_in_order(SelShared &sh, const RowView row, int32_t n,
                                       uint32_t T, uint32_t k_rem, uint32_t *keys, uint32_t *inv)
{
    if (threadIdx.x == 0) { sh.count = 0; sh.taken = 0; }
    __syncthreads();
    for (int32_t base = 0; base < n; base += NT) {
        const int32_t i = base + threadIdx.x;
        const uint32_t key = i < n ? score_key(row.ld(i)) : 0u;
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
                const uint32_t kj = score_key(row.ld(j));
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
__device__ void simt_score_row(const SelectParams &p, int32_t r, int32_t V, const RowView row, float *qf)
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
        *row.at(j) = s + 0.0f;
    }
    __syncthreads();
}

// Entries of the ordered-output buffer: k plus room for the bucket holding
// the k-th element.
__host__ __device__ __forceinline__ int32_t out_capacity(const SelectParams &p) { return p.k + SLACK; }

// One row of the dense selection: logits[r, 0:V_r] from HBM or, with
// `rescore`, the row re-scored here first (plain FP32) into its own regions
// of the candidate array.
// Shared memory: sh, then out64[k + SLACK], keys[smem_cap], inv[smem_cap].
__device__ __forceinline__ void select_row(const SelectParams &p, int32_t r, bool rescore, SelShared &sh,
                           uint64_t *out64, uint32_t *keys, uint32_t *inv, int32_t smem_cap)
{
    int32_t V = p.row_vis[r];
    if (V < 0 || V > p.max_len) {
        if (threadIdx.x == 0) record_error(p.status, ST_BAD_ROW);
        V = static_cast<int32_t>(max(static_cast<int64_t>(0), min(static_cast<int64_t>(V), p.max_len)));
    }
    const int32_t kk_target = min(p.k, V);
    RowView row{const_cast<float *>(p.logits) + static_cast<int64_t>(r) * p.ld, TILE_M};
    if (rescore) {
        // the row's own candidate regions, dead once the selector gives up on them
        row = RowView{p.fb_scores + static_cast<int64_t>(r) * TILE_M, static_cast<int64_t>(p.R) * TILE_M};
        simt_score_row(p, r, V, row, reinterpret_cast<float *>(keys));
    }
    int32_t n;
    if (V <= smem_cap) {
        for_each_key(row, V, [&](int32_t i, uint32_t key) {
            keys[i] = key;
            inv[i] = ~static_cast<uint32_t>(i);
        });
        __syncthreads();
        n = V;
    } else {
        n = sample_gather(sh, row, V, kk_target, smem_cap, keys, inv);
        if (n < 0) {
            uint32_t T, k_rem;
            n = stream_narrow(sh, row, V, static_cast<uint32_t>(kk_target), smem_cap, keys, inv, T, k_rem, true);
            if (n < 0) n = gather_cut_in_order(sh, row, V, T, k_rem, keys, inv);
        }
    }
    const int32_t kk = min(p.k, n);
    const uint64_t *result = out64;
    if (kk > 0) {
        uint64_t *ranked = reinterpret_cast<uint64_t *>(keys);   // keys + inv: smem_cap 8-byte slots
        if (bucket_topk(sh, keys, inv, n, kk, out64, min(out_capacity(p), smem_cap), ranked))
            result = ranked;
        else
            select_and_sort(sh, keys, inv, n, kk, out64);
    }
    write_row(p, r, result, kk);
    __syncthreads();
}

// The same, kept out of line for the candidate selector, where it runs only
// for the rare rows whose candidate list cannot be trusted.
__device__ __noinline__ void select_row_cold(const SelectParams &p, int32_t r, SelShared &sh,
                                             uint64_t *out64, uint32_t *keys, uint32_t *inv,
                                             int32_t smem_cap)
{
    select_row(p, r, true, sh, out64, keys, inv, smem_cap);
}

// Dense rows (logits in HBM): rows r = blockIdx.x, blockIdx.x + gridDim.x, ...
// (shared memory allows two CTAs per SM at the usual capacity)
__global__ void __launch_bounds__(NT, 2)
select_kernel(const SelectParams p)
{
    extern __shared__ __align__(16) uint8_t smem_raw[];
    SelShared &sh = *reinterpret_cast<SelShared *>(smem_raw);
    uint64_t *out64 = reinterpret_cast<uint64_t *>(smem_raw + sizeof(SelShared));
    uint32_t *keys = reinterpret_cast<uint32_t *>(out64 + out_capacity(p));
    uint32_t *inv = keys + p.smem_cap;
    wait_prior_grid();                      // last kernel of its call: nothing to allow
    for (int32_t r = blockIdx.x; r < p.R; r += gridDim.x)
        select_row(p, r, false, sh, out64, keys, inv, p.smem_cap);
}

// ------------------------------------------------------------- small k --
//
// Dense rows with k <= WK (the block scorer's top-16 blocks): one warp per
// row.  Every element becomes its full key (key32 << 32 | ~index), all
// distinct, so the order is exact.  Pass 1: each lane's largest key; T = the
// K-th largest of the 32 lane maxima, so at least K elements reach T and the
// top K lie among those that do.  Pass 2 collects the elements >= T into the
// warp's buffer (ballot compaction) and a warp sort orders them.  When more
// than WT_CAP elements reach T (one lane holding many of the largest), the
// row falls back to per-lane sorted lists of the K largest keys (most
// elements only compare with the smallest) merged by min(k, V) rounds of a
// warp-wide maximum.
constexpr int WK = 16;
constexpr int WT_CAP = 128;             // elements >= T the warp buffer holds

__device__ __forceinline__ uint64_t full_key(float f, int32_t j)
{
    return (static_cast<uint64_t>(score_key(f)) << 32) | ~static_cast<uint32_t>(j);
}
__device__ __forceinline__ uint64_t dense_key(const float *row, int32_t j) { return full_key(__ldg(row + j), j); }

template <int K>
__global__ void __launch_bounds__(256)
warp_topk_kernel(const SelectParams p)
{
    __shared__ uint64_t wbuf[8][WT_CAP];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int32_t r = static_cast<int32_t>(blockIdx.x) * 8 + static_cast<int32_t>(wid);
    wait_prior_grid();                      // last kernel of its call: nothing to allow
    if (r >= p.R) return;
    int32_t V = p.row_vis[r];
    if (V < 0 || V > p.max_len) {
        if (lane == 0) record_error(p.status, ST_BAD_ROW);
        V = static_cast<int32_t>(max(static_cast<int64_t>(0), min(static_cast<int64_t>(V), p.max_len)));
    }
    const float *row = p.logits + static_cast<int64_t>(r) * p.ld;
    int64_t ro = r;
    if (p.out_heads > 1) {                  // virtual row r = h * n + row -> output row row * H + h
        const int32_t n = p.R / p.out_heads;
        ro = static_cast<int64_t>(r % n) * p.out_heads + r / n;
    }
    int32_t *oi = p.out_idx + ro * p.k;
    float *ov = p.out_val ? p.out_val + ro * p.k : nullptr;
    const int32_t kk = min(p.k, V);
    uint64_t *buf = wbuf[wid];

    // a 16-byte aligned row is read four elements per load (lane l takes
    // elements 4 (l + 32 i) .. + 3), the rest of it element by element
    const bool vec = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
    const int32_t V4 = vec ? V >> 2 : 0;
    const float4 *row4 = reinterpret_cast<const float4 *>(row);

    // pass 1: the lane's largest key (0, below every real key, for none)
    uint64_t mx = 0ull;
#pragma unroll 4
    for (int32_t v = lane; v < V4; v += 32) {
        const float4 x = __ldg(row4 + v);
        const int32_t j = v << 2;
        const uint64_t a = max(full_key(x.x, j), full_key(x.y, j + 1));
        const uint64_t b = max(full_key(x.z, j + 2), full_key(x.w, j + 3));
        mx = max(mx, max(a, b));
    }
    for (int32_t j = 4 * V4 + lane; j < V; j += 32) {
        const uint64_t key = dense_key(row, j);
        mx = key > mx ? key : mx;
    }
    buf[lane] = mx;
    __syncwarp();
    warp_sort32_desc(buf, 32);
    __syncwarp();
    const uint64_t T = buf[K - 1];
    __syncwarp();
    // pass 2: the elements >= T into the buffer (in any order: the keys are
    // distinct and sorted below)
    const uint32_t lt = (1u << lane) - 1u;
    uint32_t cnt = 0;
    for (int32_t v0 = 0; v0 < V4; v0 += 32) {
        const int32_t v = v0 + lane;
        uint64_t key[4] = {0ull, 0ull, 0ull, 0ull};
        if (v < V4) {
            const float4 x = __ldg(row4 + v);
            key[0] = full_key(x.x, v << 2);
            key[1] = full_key(x.y, (v << 2) + 1);
            key[2] = full_key(x.z, (v << 2) + 2);
            key[3] = full_key(x.w, (v << 2) + 3);
        }
        uint32_t at = cnt, tot = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const uint32_t bal = __ballot_sync(0xffffffffu, v < V4 && key[e] >= T);
            at += static_cast<uint32_t>(__popc(bal & lt));
            tot += static_cast<uint32_t>(__popc(bal));
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (v < V4 && key[e] >= T) {
                if (at < static_cast<uint32_t>(WT_CAP)) buf[at] = key[e];
                ++at;
            }
        }
        cnt += tot;
    }
    for (int32_t j0 = 4 * V4; j0 < V; j0 += 32) {
        const int32_t j = j0 + lane;
        const uint64_t key = j < V ? dense_key(row, j) : 0ull;
        const bool take = j < V && key >= T;
        const uint32_t bal = __ballot_sync(0xffffffffu, take);
        const uint32_t at = cnt + static_cast<uint32_t>(__popc(bal & lt));
        if (take && at < static_cast<uint32_t>(WT_CAP)) buf[at] = key;
        cnt += static_cast<uint32_t>(__popc(bal));
    }
    __syncwarp();
    if (cnt <= static_cast<uint32_t>(WT_CAP)) {               // uniform
        warp_sort_desc(buf, static_cast<int32_t>(cnt));
        __syncwarp();
        for (int32_t o = lane; o < kk; o += 32) {
            const uint64_t best = buf[o];
            oi[o] = static_cast<int32_t>(~static_cast<uint32_t>(best));
            if (ov) ov[o] = key_score(static_cast<uint32_t>(best >> 32));
        }
    } else {
        uint64_t x[K];
#pragma unroll
        for (int i = 0; i < K; ++i) x[i] = 0ull;
        for (int32_t j = lane; j < V; j += 32) {
            const uint64_t key = dense_key(row, j);
            if (key > x[K - 1]) {
                x[K - 1] = key;
#pragma unroll
                for (int i = K - 1; i > 0; --i) {
                    const uint64_t a = x[i - 1], b = x[i];
                    x[i - 1] = b > a ? b : a;
                    x[i] = b > a ? a : b;
                }
            }
        }
        for (int32_t o = 0; o < kk; ++o) {
            uint64_t best = x[0];
#pragma unroll
            for (int sft = 16; sft > 0; sft >>= 1) {
                const uint64_t other = __shfl_xor_sync(0xffffffffu, best, sft);
                best = other > best ? other : best;
            }
            if (x[0] == best) {             // exactly one lane: the keys are distinct
#pragma unroll
                for (int i = 0; i < K - 1; ++i) x[i] = x[i + 1];
                x[K - 1] = 0ull;
            }
            if (lane == 0) {
                oi[o] = static_cast<int32_t>(~static_cast<uint32_t>(best));
                if (ov) ov[o] = key_score(static_cast<uint32_t>(best >> 32));
            }
        }
    }
    for (int32_t o = kk + lane; o < p.k; o += 32) {
        oi[o] = -1;
        if (ov) ov[o] = -__int_as_float(0x7f800000);
    }
}

// ------------------------------------------------------------ candidates --
//
// One CTA per row.  The row's candidates (layout in qsa_internal.h) are read
// exactly: the mask words first (one coalesced load per thread and quarter),
// then, after one block scan for the offsets, one 4-byte cp.async per
// candidate from its slot straight into the compact score array, so only
// slots the filter pass wrote this call are touched (every read is an L2 hit
// of that pass's output).  The candidates become full keys (key32 << 32 |
// ~position); the top kk are then ordered by one counting pass on the top 11
// bits of (key32 - smallest key) plus rank counting inside the buckets, and
// each element's rank is its output index, so the result goes straight to
// HBM.  A row whose list cannot be trusted (fewer than min(k, V) candidates,
// more than cap, or a cut bucket too large to order here) is re-scored in
// plain FP32 and selected densely by the same CTA (row_flag records it).
constexpr int CT = 256;               // threads per row
static_assert(CT == NT, "the in-kernel fallback runs the dense selection with the same block");
constexpr int BIG_MAX = 320;          // > (QSA_MAX_K + SLACK) / (RANK_MAX + 1)
constexpr uint32_t BLOCK_SORT_MIN = 128;   // larger buckets are sorted by the whole CTA
constexpr int QPR = 8;                // quarters per thread whose mask words are loaded together

struct CandShared {
    uint32_t hist[NBINS];
    uint32_t wtot[2][CT / 32];
    uint32_t red_min[CT / 32], red_max[CT / 32];
    uint32_t cut, need, nbig, pad_;
    uint32_t big[BIG_MAX];
};

constexpr size_t CAND_HEAD = ((sizeof(CandShared) > sizeof(SelShared) ? sizeof(CandShared) : sizeof(SelShared)) + 15) / 16 * 16;
constexpr size_t CAND_HEAD_C = (sizeof(CandShared) + 15) / 16 * 16;   // cand_kernel: its own head only
constexpr size_t SEL_HEAD = (sizeof(SelShared) + 15) / 16 * 16;

// Positions of the candidates: 32-bit, stored inverted (~position), or, for
// rows of at most 65,536 positions, 16-bit, stored as is.  Either way an
// element's full key is (key32 << 32) | ~position.
__device__ __forceinline__ void put_pos(uint32_t *a, uint32_t i, uint32_t pos) { a[i] = ~pos; }
__device__ __forceinline__ void put_pos(uint16_t *a, uint32_t i, uint32_t pos) { a[i] = static_cast<uint16_t>(pos); }
__device__ __forceinline__ uint32_t inv_pos(const uint32_t *a, uint32_t i) { return a[i]; }
__device__ __forceinline__ uint32_t inv_pos(const uint16_t *a, uint32_t i) { return ~static_cast<uint32_t>(a[i]); }

// Exclusive prefix of v over the block with a single barrier; wt alternates
// between two buffers so that consecutive calls need no barrier in between.
__device__ __forceinline__ uint32_t cand_scan(uint32_t v, uint32_t *wt, uint32_t &total)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wt[wid] = x;
    __syncthreads();
    uint32_t before = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < CT / 32; ++w) {
        const uint32_t c = wt[w];
        before += w < wid ? c : 0u;
        tot += c;
    }
    total = tot;
    return before + x - v;
}

__device__ __forceinline__ void discard_l2_line(const void *p)
{
    asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}

// 4-byte asynchronous copy global -> shared (completed by cp_async_wait_all).
__device__ __forceinline__ void cp_async4(void *dst_smem, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst_smem)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Gathers the candidates of quarters [e_lo, e_hi) of row r (layout in
// qsa_internal.h).  Thread t takes quarters e_lo + t, e_lo + t + CT, ... in
// rounds of QPR: their mask words are loaded together, one block scan gives
// the thread's offset, and each candidate's score is copied asynchronously
// from its slot (slot row j of quarter q at float 4j + q of the (tile, row)
// region) to a_key[done + ...], its ~position to a_pos.  Stops with overflow
// set (the count past cap) instead of writing past cap.  The copies are
// complete after cp_async_wait_all() and a barrier.
template <typename PosT>
__device__ __forceinline__ void gather_quarters(const SelectParams &p, int32_t r, int32_t e_lo, int32_t e_hi,
                                                uint32_t *a_key, PosT *a_pos, CandShared &sh, int &sbuf,
                                                uint32_t &done, bool &overflow)
{
    const int t = threadIdx.x;
    const uint32_t *mrow = p.cand_mask + static_cast<int64_t>(r) * p.tiles_ld * 4;
    const float *srow = p.cand_score + static_cast<int64_t>(r) * TILE_M;    // tile t at + t * R * TILE_M
    for (int32_t e0 = e_lo; e0 < e_hi; e0 += QPR * CT) {
        uint32_t m[QPR], cnt = 0;
#pragma unroll
        for (int u = 0; u < QPR; ++u) {
            const int32_t e = e0 + t + u * CT;
            m[u] = e < e_hi ? __ldcg(mrow + e) : 0u;
        }
#pragma unroll
        for (int u = 0; u < QPR; ++u) cnt += __popc(m[u]);
        uint32_t ctot;
        const uint32_t before = cand_scan(cnt, sh.wtot[sbuf], ctot);
        sbuf ^= 1;
        if (done + ctot > static_cast<uint32_t>(p.cap)) { overflow = true; return; }   // uniform
        uint32_t o = done + before;
#pragma unroll
        for (int u = 0; u < QPR; ++u) {
            const int32_t e = e0 + t + u * CT;
            uint32_t mm = m[u];
            const int32_t tile = e >> 2, q = e & 3;
            const float *slot = srow + static_cast<int64_t>(tile) * p.R * TILE_M + q;
            const uint32_t pos0 = static_cast<uint32_t>(tile * TILE_M + q * 32);
            for (uint32_t j = 0; mm != 0u; ++j) {
                const uint32_t bit = static_cast<uint32_t>(__ffs(mm) - 1);
                mm &= mm - 1u;
                cp_async4(a_key + o, slot + 4 * j);
                put_pos(a_pos, o, pos0 + bit);
                ++o;
            }
        }
        done += ctot;
    }
}

// a_key[0, n): scores -> order-preserving keys; block-wide min and max (the
// barrier inside also publishes a_key to the block).
__device__ __forceinline__ void keys_and_range(uint32_t *a_key, uint32_t n, CandShared &sh, uint32_t &kmin,
                                               uint32_t &kmax)
{
    const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
    kmin = 0xffffffffu;
    kmax = 0u;
    for (uint32_t i = t; i < n; i += CT) {
        const uint32_t key = score_key(__uint_as_float(a_key[i]));
        a_key[i] = key;
        kmin = min(kmin, key);
        kmax = max(kmax, key);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
        kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
    }
    if (lane == 0) { sh.red_min[wid] = kmin; sh.red_max[wid] = kmax; }
    __syncthreads();
#pragma unroll
    for (int w = 0; w < CT / 32; ++w) { kmin = min(kmin, sh.red_min[w]); kmax = max(kmax, sh.red_max[w]); }
}

// One counting pass over the keys >= lo of a_key[0, n) into 11-bit buckets of
// width 2^shift (bucket 0 holds the largest keys), sh.hist zero on entry;
// leaves in sh.hist each bucket's start (the scatter cursors) and returns the
// bucket holding the kk-th largest key (bb) and the end of that bucket (need).
__device__ __forceinline__ void count_and_cut(const uint32_t *a_key, uint32_t n, uint32_t lo, int shift, uint32_t kk,
                                              CandShared &sh, int &sbuf, uint32_t &bb, uint32_t &need)
{
    const int t = threadIdx.x;
    for (uint32_t i = t; i < n; i += CT) {
        const uint32_t key = a_key[i];
        if (key >= lo) atomicAdd(&sh.hist[NBINS - 1 - ((key - lo) >> shift)], 1u);
    }
    __syncthreads();
    uint32_t c[BPT], sum = 0;
#pragma unroll
    for (int i = 0; i < BPT; ++i) { c[i] = sh.hist[BPT * t + i]; sum += c[i]; }
    uint32_t all;
    uint32_t start = cand_scan(sum, sh.wtot[sbuf], all);
    sbuf ^= 1;
#pragma unroll
    for (int i = 0; i < BPT; ++i) {
        if (start < kk && kk <= start + c[i]) { sh.cut = BPT * t + i; sh.need = start + c[i]; }
        sh.hist[BPT * t + i] = start;        // scatter cursor
        start += c[i];
    }
    __syncthreads();
    bb = sh.cut;
    need = sh.need;
}

// Shared memory of cand_kernel<PosT>: its own head, bq[k + SLACK], a_key[cap],
// a_pos[cap]; a row that falls back reuses the same bytes as SelShared,
// out64[k + SLACK] and fb_cap (p.smem_cap) staged keys and positions, so the
// fallback's larger head costs no resident CTAs.  With 16-bit positions a
// top-2,048 CTA takes 55 KB: four per SM.
template <typename PosT>
constexpr int cand_ctas_per_sm() { return sizeof(PosT) == 2 ? 4 : 3; }

template <typename PosT>
__global__ void __launch_bounds__(CT, cand_ctas_per_sm<PosT>())
cand_kernel(const SelectParams p)
{
    extern __shared__ __align__(16) uint8_t smem_raw[];
    CandShared &sh = *reinterpret_cast<CandShared *>(smem_raw);
    uint64_t *bq = reinterpret_cast<uint64_t *>(smem_raw + CAND_HEAD_C);        // k + SLACK entries
    uint32_t *a_key = reinterpret_cast<uint32_t *>(bq + p.k + SLACK);            // cap entries: scores, then keys
    PosT *a_pos = reinterpret_cast<PosT *>(a_key + p.cap);                       // cap entries: positions
    const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
    const int32_t r = blockIdx.x;
    for (int i = t; i < NBINS; i += CT) sh.hist[i] = 0;
    if (t == 0) sh.nbig = 0;
    wait_prior_grid();                      // last kernel of its call: nothing to allow
    if (r >= p.R) return;
    // a row whose list cannot be trusted is re-scored and selected densely
    // right here, in the same shared memory (SelShared over the head)
    auto fallback = [&]() {
        if (t == 0) {
            p.row_flag[r] = 1;
            atomicExch(&p.plan->any_fallback, 1);
        }
        __syncthreads();
        uint64_t *out64 = reinterpret_cast<uint64_t *>(smem_raw + SEL_HEAD);
        uint32_t *keys = reinterpret_cast<uint32_t *>(out64 + p.k + SLACK);
        select_row_cold(p, r, *reinterpret_cast<SelShared *>(smem_raw), out64, keys, keys + p.smem_cap, p.smem_cap);
    };
    int32_t V = p.row_vis[r];
    if (V < 0 || V > p.max_len) {
        if (t == 0) record_error(p.status, ST_BAD_ROW);
        V = static_cast<int32_t>(max(static_cast<int64_t>(0), min(static_cast<int64_t>(V), p.max_len)));
    }
    const int32_t kk_target = min(p.k, V);
    const int32_t ntile = (V + TILE_M - 1) / TILE_M;
    const int32_t nq = ntile * 4;
    const uint32_t *mrow = p.cand_mask + static_cast<int64_t>(r) * p.tiles_ld * 4;

    uint32_t done = 0;
    bool overflow = false;
    int sbuf = 0;
    gather_quarters(p, r, 0, nq, a_key, a_pos, sh, sbuf, done, overflow);
    cp_async_wait_all();
    __syncthreads();
    // every mask word of the row has been read: drop its lines from L2 unwritten
    for (int32_t l = t; l < (ntile * 16 + 127) / 128; l += CT) discard_l2_line(mrow + l * 32);
    const uint32_t n = done;
    if (overflow || n < static_cast<uint32_t>(kk_target)) {   // uniform
        fallback();
        return;
    }
    // ---- scores -> order-preserving keys, and their range
    uint32_t kmin, kmax;
    keys_and_range(a_key, n, sh, kmin, kmax);
    const uint32_t kk = min(static_cast<uint32_t>(p.k), n);
    int32_t *oi = p.out_idx + static_cast<int64_t>(r) * p.k;
    float *ov = p.out_val ? p.out_val + static_cast<int64_t>(r) * p.k : nullptr;
    if (kk > 0) {
        // ---- counting pass: bucket 0 holds the largest keys; when the
        //      buckets down to the cut span a much narrower key range than
        //      all candidates (every position a candidate: scores down to the
        //      spike of exact zeros), count once more over that range only, so
        //      that the buckets to be ordered stay small
        uint32_t lo = kmin;
        int shift = span_shift(kmax - kmin);
        uint32_t bb = 0, need = 0;
        for (int level = 0; level < 2; ++level) {
            count_and_cut(a_key, n, lo, shift, kk, sh, sbuf, bb, need);
            if (level == 1 || shift == 0) break;
            const uint32_t lo2 = lo + (static_cast<uint32_t>(NBINS - 1 - bb) << shift);
            const int shift2 = span_shift(kmax - lo2);
            if (shift2 + 3 > shift) break;                         // uniform
            lo = lo2;
            shift = shift2;
            for (int i = t; i < NBINS; i += CT) sh.hist[i] = 0;
            __syncthreads();
        }
        if (need > static_cast<uint32_t>(p.k + SLACK)) {           // uniform: huge tie bucket at the cut
            fallback();
            return;
        }
        const uint32_t kmin_sel = lo;                              // every ordered key is >= lo
        // ---- scatter the buckets down to the cut
        for (uint32_t i = t; i < n; i += CT) {
            const uint32_t key = a_key[i];
            if (key < lo) continue;
            const uint32_t b = NBINS - 1 - ((key - lo) >> shift);
            if (b <= bb) bq[atomicAdd(&sh.hist[b], 1u)] = (static_cast<uint64_t>(key) << 32) | inv_pos(a_pos, i);
        }
        __syncthreads();
        // ---- rank inside the bucket = place in the output (hist[b] is now
        //      the end of bucket b, hence the start of bucket b + 1)
        // four positions per iteration: four independent chains
        constexpr int NP = 4;
        for (uint32_t p0 = t; p0 < need; p0 += NP * CT) {
            uint64_t x[NP];
            uint32_t s0[NP], m[NP], rk[NP];
#pragma unroll
            for (int h = 0; h < NP; ++h) {
                const uint32_t pos = p0 + h * CT;
                m[h] = 0u;
                s0[h] = 0xffffffffu;                              // no output unless ranked below
                x[h] = 0ull;
                if (pos < need) {
                    x[h] = bq[pos];
                    const uint32_t b = NBINS - 1 - ((static_cast<uint32_t>(x[h] >> 32) - kmin_sel) >> shift);
                    s0[h] = b ? sh.hist[b - 1] : 0u;
                    const uint32_t e = sh.hist[b];
                    if (e - s0[h] > RANK_MAX) {
                        if (pos == s0[h]) sh.big[atomicAdd(&sh.nbig, 1u)] = b;
                        s0[h] = 0xffffffffu;                      // ordered by the warp sort below
                    } else {
                        m[h] = e - s0[h];
                    }
                }
                rk[h] = s0[h];
            }
            const uint32_t mx = max(max(m[0], m[1]), max(m[2], m[3]));
            for (uint32_t q = 0; q < mx; ++q) {
#pragma unroll
                for (int h = 0; h < NP; ++h)
                    if (q < m[h]) rk[h] += bq[s0[h] + q] > x[h];
            }
#pragma unroll
            for (int h = 0; h < NP; ++h) {
                if (rk[h] < kk) {
                    oi[rk[h]] = static_cast<int32_t>(~static_cast<uint32_t>(x[h]));
                    if (ov) ov[rk[h]] = key_score(static_cast<uint32_t>(x[h] >> 32));
                }
            }
        }
        __syncthreads();
        // buckets too large for rank counting: those above BLOCK_SORT_MIN (a
        // tie bucket at the cut, typically one) by the whole CTA in turn, the
        // others by one warp each
        const uint32_t nbig = sh.nbig;
        for (uint32_t q = 0; q < nbig; ++q) {                      // uniform
            const uint32_t b = sh.big[q];
            const uint32_t s0 = b ? sh.hist[b - 1] : 0u, m = sh.hist[b] - s0;
            if (m <= BLOCK_SORT_MIN) continue;
            bitonic_sort_desc<CT, true>(bq + s0, static_cast<int32_t>(m), t);
            for (uint32_t i = t; i < m && s0 + i < kk; i += CT) {
                const uint64_t x = bq[s0 + i];
                oi[s0 + i] = static_cast<int32_t>(~static_cast<uint32_t>(x));
                if (ov) ov[s0 + i] = key_score(static_cast<uint32_t>(x >> 32));
            }
        }
        for (uint32_t q = wid; q < nbig; q += CT / 32) {
            const uint32_t b = sh.big[q];
            const uint32_t s0 = b ? sh.hist[b - 1] : 0u, m = sh.hist[b] - s0;
            if (m > BLOCK_SORT_MIN) continue;
            warp_sort_desc(bq + s0, static_cast<int32_t>(m));
            for (uint32_t i = lane; i < m && s0 + i < kk; i += 32) {
                const uint64_t x = bq[s0 + i];
                oi[s0 + i] = static_cast<int32_t>(~static_cast<uint32_t>(x));
                if (ov) ov[s0 + i] = key_score(static_cast<uint32_t>(x >> 32));
            }
        }
    }
    for (int32_t i = static_cast<int32_t>(kk) + t; i < p.k; i += CT) {
        oi[i] = -1;
        if (ov) ov[i] = -__int_as_float(0x7f800000);
    }
    if (t == 0) p.row_flag[r] = 0;
}

// ---------------------------------------------------- cluster candidates --
//
// The same selection for batches with fewer rows than the GPU has SMs (decode
// batches): the C CTAs of a thread-block cluster share one row, and their
// shared memories are joined through distributed shared memory.
//  1. CTA c gathers quarters [c nq / C, (c + 1) nq / C) of the row, makes
//     keys and takes their range;
//  2. every CTA reads the C counts and ranges (the row's key range is then
//     known to all), counts its keys into the row's 11-bit buckets, and after
//     a cluster barrier sums the C histograms, which gives each bucket's place
//     in the output and this CTA's cursor inside it (the CTAs before it in the
//     cluster come first);
//  3. every CTA writes its keys of the buckets down to the cut into CTA 0's
//     ordered buffer (remote stores);
//  4. CTA c owns the buckets that start in its share [c need / C, (c + 1)
//     need / C) of the buffer, copies them into its own shared memory first,
//     ranks their elements and writes them out.
// Every CTA takes the same cluster barriers (the decisions between them are
// made from the same summed data); a row that cannot be certified is re-scored
// by CTA 0 alone after the last barrier.  The cluster size comes from the
// device's occupancy query at launch, never from the compute capability.
struct ClusterInfo {
    uint32_t n, kmin, kmax, overflow;
};

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t v;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(v));
    return v;
}
__device__ __forceinline__ uint32_t cluster_nctarank()
{
    uint32_t v;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(v));
    return v;
}
// All threads of all CTAs of the cluster; orders shared-memory writes before
// it with remote reads after it.
__device__ __forceinline__ void cluster_barrier()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of `local` (this CTA's shared memory) in CTA `cta` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(const void *local, uint32_t cta)
{
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(local)), "r"(cta));
    return a;
}
// Remote loads carry no memory clobber: the cluster barriers order them with
// the writes they read, and the compiler may issue several before the first
// result is used.
__device__ __forceinline__ uint4 peer_ld128(uint32_t a)
{
    uint4 v;
    asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ uint64_t peer_ld64(uint32_t a)
{
    uint64_t v;
    asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ void peer_st64(uint32_t a, uint64_t v)
{
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(a), "l"(v) : "memory");
}

__global__ void __launch_bounds__(CT, 2)
cand_cluster_kernel(const SelectParams p)
{
    extern __shared__ __align__(16) uint8_t smem_raw[];
    CandShared &sh = *reinterpret_cast<CandShared *>(smem_raw);                 // hist: summed counts
    uint64_t *bq = reinterpret_cast<uint64_t *>(smem_raw + CAND_HEAD);          // k + SLACK entries
    uint32_t *a_key = reinterpret_cast<uint32_t *>(bq + p.k + SLACK);            // cap: scores, then keys
    uint32_t *a_pos = a_key + p.cap;                                             // cap: ~position
    // NBINS: this CTA's counts, 16-byte aligned for the peers' vector loads
    uint32_t *own = reinterpret_cast<uint32_t *>((reinterpret_cast<uintptr_t>(a_pos + p.cap) + 15) & ~uintptr_t{15});
    uint32_t *bstart = own + NBINS;                                              // NBINS: bucket starts
    ClusterInfo &ci = *reinterpret_cast<ClusterInfo *>(bstart + NBINS);
    const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
    const uint32_t C = cluster_nctarank(), c = cluster_ctarank();
    const int32_t r = static_cast<int32_t>(blockIdx.x / C);
    for (int i = t; i < NBINS; i += CT) own[i] = 0;
    if (t == 0) sh.nbig = 0;
    wait_prior_grid();                      // last kernel of its call: nothing to allow
    int32_t V = p.row_vis[r];
    if (V < 0 || V > p.max_len) {
        if (t == 0 && c == 0) record_error(p.status, ST_BAD_ROW);
        V = static_cast<int32_t>(max(static_cast<int64_t>(0), min(static_cast<int64_t>(V), p.max_len)));
    }
    const int32_t kk_target = min(p.k, V);
    const int32_t nq = ((V + TILE_M - 1) / TILE_M) * 4;

    // ---- 1. this CTA's slice
    uint32_t done = 0;
    bool overflow = false;
    int sbuf = 0;
    gather_quarters(p, r, static_cast<int32_t>(static_cast<int64_t>(nq) * c / C),
                    static_cast<int32_t>(static_cast<int64_t>(nq) * (c + 1) / C), a_key, a_pos, sh, sbuf, done,
                    overflow);
    cp_async_wait_all();
    __syncthreads();
    uint32_t kmin = 0xffffffffu, kmax = 0u;
    if (!overflow) keys_and_range(a_key, done, sh, kmin, kmax);   // uniform in the CTA
    if (t == 0) ci = ClusterInfo{done, kmin, kmax, overflow ? 1u : 0u};
    cluster_barrier();                                                          // (1)
    // ---- 2. the row's count and key range
    uint32_t n = 0, any_over = 0;
    {
        uint4 info[8];                      // C <= 8: every load issued before the first is used
#pragma unroll
        for (uint32_t x = 0; x < 8; ++x)
            if (x < C) info[x] = peer_ld128(peer_addr(&ci, x));
#pragma unroll
        for (uint32_t x = 0; x < 8; ++x) {
            if (x >= C) break;
            n += info[x].x;
            kmin = min(kmin, info[x].y);
            kmax = max(kmax, info[x].z);
            any_over |= info[x].w;
        }
    }
    auto finish_fallback = [&]() {
        cluster_barrier();                  // nobody reads this CTA's shared memory any more
        if (c != 0) return;
        if (t == 0) {
            p.row_flag[r] = 1;
            atomicExch(&p.plan->any_fallback, 1);
        }
        __syncthreads();
        select_row_cold(p, r, *reinterpret_cast<SelShared *>(smem_raw), bq, a_key, a_pos, p.cap);
    };
    if (any_over || n > static_cast<uint32_t>(p.cap) || n < static_cast<uint32_t>(kk_target)) {   // cluster-uniform
        finish_fallback();
        return;
    }
    int32_t *oi = p.out_idx + static_cast<int64_t>(r) * p.k;
    float *ov = p.out_val ? p.out_val + static_cast<int64_t>(r) * p.k : nullptr;
    if (n == 0) {                           // cluster-uniform: nothing visible, all padding
        cluster_barrier();
        if (c == 0) {
            for (int32_t i = t; i < p.k; i += CT) {
                oi[i] = -1;
                if (ov) ov[i] = -__int_as_float(0x7f800000);
            }
            if (t == 0) p.row_flag[r] = 0;
        }
        return;
    }
    const uint32_t kk = min(static_cast<uint32_t>(p.k), n);   // >= 1
    // counting rounds over the keys >= lo (a second, narrower one when the
    // buckets down to the cut span a much smaller key range, as in the
    // one-CTA selector); each sums the C histograms between two barriers
    uint32_t lo = kmin;
    int shift = span_shift(kmax - kmin);
    uint32_t bb = 0, need = 0;
    for (int level = 0; level < 2; ++level) {
        for (uint32_t i = t; i < done; i += CT) {
            const uint32_t key = a_key[i];
            if (key >= lo) atomicAdd(&own[NBINS - 1 - ((key - lo) >> shift)], 1u);
        }
        __syncthreads();
        cluster_barrier();                                                      // (2) every count is in
        // summed counts of this thread's BPT buckets and this CTA's share before it
        uint32_t cnt[BPT], mine_before[BPT], sum = 0;
#pragma unroll
        for (int i = 0; i < BPT; ++i) { cnt[i] = 0; mine_before[i] = 0; }
        static_assert(BPT == 8, "two 16-byte loads per CTA and thread");
        {
            uint4 h[8][2];                  // C <= 8: all loads in flight before the sums
#pragma unroll
            for (uint32_t x = 0; x < 8; ++x) {
                if (x < C) {
                    const uint32_t a = peer_addr(own + BPT * t, x);
                    h[x][0] = peer_ld128(a);
                    h[x][1] = peer_ld128(a + 16);
                }
            }
#pragma unroll
            for (uint32_t x = 0; x < 8; ++x) {
                if (x >= C) break;
                const uint32_t v[8] = {h[x][0].x, h[x][0].y, h[x][0].z, h[x][0].w,
                                       h[x][1].x, h[x][1].y, h[x][1].z, h[x][1].w};
#pragma unroll
                for (int i = 0; i < BPT; ++i) {
                    if (x < c) mine_before[i] += v[i];
                    cnt[i] += v[i];
                }
            }
        }
#pragma unroll
        for (int i = 0; i < BPT; ++i) sum += cnt[i];
        uint32_t all;
        uint32_t start = cand_scan(sum, sh.wtot[sbuf], all);
        sbuf ^= 1;
#pragma unroll
        for (int i = 0; i < BPT; ++i) {
            const int b = BPT * t + i;
            if (start < kk && kk <= start + cnt[i]) { sh.cut = b; sh.need = start + cnt[i]; }
            bstart[b] = start;
            sh.hist[b] = start + mine_before[i];            // this CTA's scatter cursor in bucket b
            start += cnt[i];
        }
        __syncthreads();
        bb = sh.cut;
        need = sh.need;
        cluster_barrier();                                                      // (3) counts read everywhere
        if (level == 1 || shift == 0) break;
        const uint32_t lo2 = lo + (static_cast<uint32_t>(NBINS - 1 - bb) << shift);
        const int shift2 = span_shift(kmax - lo2);
        if (shift2 + 3 > shift) break;                                          // cluster-uniform
        lo = lo2;
        shift = shift2;
        for (int i = t; i < NBINS; i += CT) own[i] = 0;
        __syncthreads();
    }
    if (need > static_cast<uint32_t>(p.k + SLACK)) {         // cluster-uniform: huge tie bucket at the cut
        finish_fallback();
        return;
    }
    // ---- 3. this CTA's keys of the buckets down to the cut -> CTA 0's buffer
    const uint32_t bq0 = peer_addr(bq, 0);
    for (uint32_t i = t; i < done; i += CT) {
        const uint32_t key = a_key[i];
        if (key < lo) continue;
        const uint32_t b = NBINS - 1 - ((key - lo) >> shift);
        if (b <= bb) peer_st64(bq0 + 8u * atomicAdd(&sh.hist[b], 1u), (static_cast<uint64_t>(key) << 32) | a_pos[i]);
    }
    cluster_barrier();                                                          // (4) CTA 0's buffer complete
    // ---- 4. the buckets starting in this CTA's share of the buffer
    auto bucket_of = [&](uint32_t pos) {    // last bucket whose start is <= pos (bstart is non-decreasing)
        int lo = 0, hi = NBINS - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (bstart[mid] <= pos) lo = mid; else hi = mid - 1;
        }
        return lo;
    };
    auto first_start_at_or_after = [&](uint32_t pos) -> uint32_t {
        if (pos >= need) return need;
        const int b = bucket_of(pos);
        return bstart[b] == pos ? pos : (b + 1 < NBINS ? bstart[b + 1] : need);
    };
    const uint32_t s_lo = first_start_at_or_after(static_cast<uint32_t>(static_cast<uint64_t>(need) * c / C));
    const uint32_t s_hi = c + 1 == C ? need : first_start_at_or_after(static_cast<uint32_t>(static_cast<uint64_t>(need) * (c + 1) / C));
    // copy [s_lo, s_hi) of CTA 0's buffer to the front of this CTA's own one
    // (CTA 0 ranks its share in place)
    uint64_t *loc = bq;
    const int64_t shift_pos = c == 0 ? 0 : static_cast<int64_t>(s_lo);
    if (c != 0)
        for (uint32_t i = s_lo + t; i < s_hi; i += CT) loc[i - s_lo] = peer_ld64(bq0 + 8u * i);
    __syncthreads();
    for (uint32_t pos = s_lo + t; pos < s_hi; pos += CT) {
        const uint64_t x = loc[pos - shift_pos];
        const uint32_t b = NBINS - 1 - ((static_cast<uint32_t>(x >> 32) - lo) >> shift);
        const uint32_t s0 = bstart[b], e = b + 1 < NBINS ? bstart[b + 1] : need;
        if (e - s0 > RANK_MAX) {
            if (pos == s0) sh.big[atomicAdd(&sh.nbig, 1u)] = b;
            continue;
        }
        uint32_t rk = s0;
        for (uint32_t q = s0; q < e; ++q) rk += loc[q - shift_pos] > x;
        if (rk < kk) {
            oi[rk] = static_cast<int32_t>(~static_cast<uint32_t>(x));
            if (ov) ov[rk] = key_score(static_cast<uint32_t>(x >> 32));
        }
    }
    __syncthreads();
    for (uint32_t qb = wid; qb < sh.nbig; qb += CT / 32) {
        const uint32_t b = sh.big[qb];
        const uint32_t s0 = bstart[b], m = (b + 1 < NBINS ? bstart[b + 1] : need) - s0;
        warp_sort_desc(loc + (s0 - shift_pos), static_cast<int32_t>(m));
        for (uint32_t i = lane; i < m && s0 + i < kk; i += 32) {
            const uint64_t x = loc[s0 - shift_pos + i];
            oi[s0 + i] = static_cast<int32_t>(~static_cast<uint32_t>(x));
            if (ov) ov[s0 + i] = key_score(static_cast<uint32_t>(x >> 32));
        }
    }
    cluster_barrier();                                                          // (5) CTA 0's buffer no longer read
    if (c == 0) {
        for (int32_t i = static_cast<int32_t>(kk) + t; i < p.k; i += CT) {
            oi[i] = -1;
            if (ov) ov[i] = -__int_as_float(0x7f800000);
        }
        if (t == 0) p.row_flag[r] = 0;
    }
}

// ------------------------------------------------------------- threshold --
//
// tau_r for the filter pass: a value with about m sampled scores at or above
// it, m = oversample * k * n_s / V_r (+8), the expected share of the top k in
// the sample.  tau only has to be low enough; the candidate count it yields
// is checked by the candidate selector, so the search stops as soon as the
// bin holding the m-th sampled key is small.  One CTA of TH_THREADS per row:
// the row's keys are staged in shared memory (rows longer than the staging
// area are read from global memory in every pass instead).
constexpr int TH_BINS = 256;

template <int TH_THREADS>
struct ThShared {
    uint32_t hist[TH_BINS];
    uint32_t red[4][TH_THREADS / 32];
    uint32_t cut_d, cut_above, cut_eq, pad_;
};

// Block-wide min, max, min and sum of four per-thread values (one barrier).
template <int TH_THREADS>
__device__ __forceinline__ void th_reduce(ThShared<TH_THREADS> &sh, uint32_t &a_min, uint32_t &b_max, uint32_t &c_min,
                                          uint32_t &d_sum)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        a_min = min(a_min, __shfl_xor_sync(0xffffffffu, a_min, o));
        b_max = max(b_max, __shfl_xor_sync(0xffffffffu, b_max, o));
        c_min = min(c_min, __shfl_xor_sync(0xffffffffu, c_min, o));
        d_sum += __shfl_xor_sync(0xffffffffu, d_sum, o);
    }
    if (lane == 0) { sh.red[0][wid] = a_min; sh.red[1][wid] = b_max; sh.red[2][wid] = c_min; sh.red[3][wid] = d_sum; }
    __syncthreads();
    a_min = sh.red[0][0]; b_max = sh.red[1][0]; c_min = sh.red[2][0]; d_sum = sh.red[3][0];
#pragma unroll
    for (int w = 1; w < TH_THREADS / 32; ++w) {
        a_min = min(a_min, sh.red[0][w]);
        b_max = max(b_max, sh.red[1][w]);
        c_min = min(c_min, sh.red[2][w]);
        d_sum += sh.red[3][w];
    }
}

// The key that about m of the n_s keys key_at(i) reach, searched in [lo, hi]
// (every key counted lies there).
// STAGED: the keys are in stage[] (16-byte aligned); otherwise the scores are
// read from row[] in every pass.
template <int TH_THREADS, bool STAGED>
__device__ uint32_t thresh_search(ThShared<TH_THREADS> &sh, const uint32_t *stage, const float *row, int32_t n_s,
                                  uint32_t m, uint32_t lo, uint32_t hi)
{
    const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
    const uint32_t stop = max(8u, m / 16);
    uint32_t k_left = m;
    while (lo != hi) {
        const uint32_t span = hi - lo;
        const int bits = 32 - __clz(span);
        const int shift = bits > 8 ? bits - 8 : 0;            // (hi - lo) >> shift < TH_BINS
        for (int b = t; b < TH_BINS; b += TH_THREADS) sh.hist[b] = 0;
        __syncthreads();
        // one unsigned compare per key: kv in [lo, hi] <=> kv - lo <= span
        if constexpr (STAGED) {
            const uint4 *st4 = reinterpret_cast<const uint4 *>(stage);
            const int32_t nv = n_s >> 2;
            for (int32_t v = t; v < nv; v += TH_THREADS) {
                const uint4 kq = st4[v];
                const uint32_t d0 = kq.x - lo, d1 = kq.y - lo, d2 = kq.z - lo, d3 = kq.w - lo;
                if (d0 <= span) atomicAdd(&sh.hist[d0 >> shift], 1u);
                if (d1 <= span) atomicAdd(&sh.hist[d1 >> shift], 1u);
                if (d2 <= span) atomicAdd(&sh.hist[d2 >> shift], 1u);
                if (d3 <= span) atomicAdd(&sh.hist[d3 >> shift], 1u);
            }
            for (int32_t i = 4 * nv + t; i < n_s; i += TH_THREADS) {
                const uint32_t d = stage[i] - lo;
                if (d <= span) atomicAdd(&sh.hist[d >> shift], 1u);
            }
        } else {
            for (int32_t i = t; i < n_s; i += TH_THREADS) {
                const uint32_t d = score_key(__ldcg(row + i)) - lo;
                if (d <= span) atomicAdd(&sh.hist[d >> shift], 1u);
            }
        }
        __syncthreads();
        if (wid == 0) {
            // lane l holds bins 255-8l down to 248-8l: lanes in descending key order
            uint32_t c[8], s = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                c[j] = sh.hist[TH_BINS - 1 - 8 * lane - j];
                s += c[j];
            }
            uint32_t incl = s;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            uint32_t above = incl - s;
            if (above < k_left && k_left <= incl) {
                // exactly one lane: k_left lies in one of its bins
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (k_left <= above + c[j]) {
                        sh.cut_d = static_cast<uint32_t>(TH_BINS - 1 - 8 * lane - j);
                        sh.cut_above = above;
                        sh.cut_eq = c[j];
                        break;
                    }
                    above += c[j];
                }
            }
        }
        __syncthreads();
        const uint32_t d = sh.cut_d, eq = sh.cut_eq;
        k_left -= sh.cut_above;
        const uint32_t nlo = lo + (d << shift);
        const uint64_t nhi = static_cast<uint64_t>(nlo) + ((1ull << shift) - 1);
        hi = static_cast<uint32_t>(min(static_cast<uint64_t>(hi), nhi));
        lo = nlo;
        if (eq <= stop) break;                                // uniform
    }
    return lo;
}

template <int TH_THREADS>
__global__ void __launch_bounds__(TH_THREADS)
thresh_kernel(const SelectParams p)
{
    extern __shared__ __align__(16) uint8_t smem_raw[];
    ThShared<TH_THREADS> &sh = *reinterpret_cast<ThShared<TH_THREADS> *>(smem_raw);
    uint32_t *stage = reinterpret_cast<uint32_t *>(smem_raw + sizeof(ThShared<TH_THREADS>));
    const int t = threadIdx.x;
    const int32_t r = blockIdx.x;
    wait_prior_grid();
    if (r >= p.R) return;
    int32_t V = p.row_vis[r];
    if (V < 0 || V > p.max_len) {
        if (t == 0) record_error(p.status, ST_BAD_ROW);
        V = static_cast<int32_t>(max(static_cast<int64_t>(0), min(static_cast<int64_t>(V), p.max_len)));
    }
    // sampled tiles 0, s, 2s, ... of the row, the last one possibly partial
    const int32_t tiles = (V + TILE_M - 1) / TILE_M;
    int32_t n_s = 0;
    if (tiles > 0) {
        const int32_t t_last = ((tiles - 1) / p.sample_stride) * p.sample_stride;
        n_s = (t_last / p.sample_stride) * TILE_M + min(TILE_M, V - t_last * TILE_M);
    }
    float tau = -__int_as_float(0x7f800000);
    if (V > p.cap && n_s > 0) {                               // uniform
        // (single precision: this is a sizing heuristic, and FP64 is slow here)
        const float want = p.oversample * static_cast<float>(p.k) * static_cast<float>(n_s) / static_cast<float>(V);
        const uint32_t m = static_cast<uint32_t>(max(1, min(static_cast<int32_t>(ceilf(want)) + 8, n_s)));
        const float *row = p.logits + static_cast<int64_t>(r) * p.ld;
        const bool staged = n_s <= p.smem_cap;
        // one pass: keys, their range, and the range of the keys above zero;
        // when at least m are positive the spike of exact zeros (every head
        // clipped) lies below the cut and is left out of the range
        const uint32_t zk = score_key(0.0f);
        uint32_t lo = 0xffffffffu, hi = 0u, lo_pos = 0xffffffffu, npos = 0;
        auto take_key = [&](uint32_t kv) {
            lo = min(lo, kv);
            hi = max(hi, kv);
            if (kv > zk) { lo_pos = min(lo_pos, kv); ++npos; }
        };
        const int32_t nv = n_s >> 2;                          // row start is 16-byte aligned
        for (int32_t v = t; v < nv; v += TH_THREADS) {
            const float4 x = __ldcg(reinterpret_cast<const float4 *>(row) + v);
            const uint4 kq = make_uint4(score_key(x.x), score_key(x.y), score_key(x.z), score_key(x.w));
            take_key(kq.x); take_key(kq.y); take_key(kq.z); take_key(kq.w);
            if (staged) reinterpret_cast<uint4 *>(stage)[v] = kq;
        }
        for (int32_t i = 4 * nv + t; i < n_s; i += TH_THREADS) {
            const uint32_t kv = score_key(__ldcg(row + i));
            take_key(kv);
            if (staged) stage[i] = kv;
        }
        th_reduce(sh, lo, hi, lo_pos, npos);                  // its barrier also publishes stage[]
        if (npos >= m) lo = lo_pos;
        const uint32_t T = staged
            ? thresh_search<TH_THREADS, true>(sh, stage, row, n_s, m, lo, hi)
            : thresh_search<TH_THREADS, false>(sh, stage, row, n_s, m, lo, hi);
        tau = key_score(T);
    }
    if (t == 0) p.tau[r] = tau;
    allow_next_grid();
}

}  // namespace

size_t select_smem_bytes(int32_t smem_cap)
{
    return sizeof(SelShared) + static_cast<size_t>(smem_cap) * 8;
}

namespace {

// serialises the attribute updates of the kernels below (callers on several
// host threads)
std::mutex g_attr_mu;

template <typename K>
int set_smem(K kernel, size_t smem, size_t (&done)[64])
{
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return static_cast<int>(cudaErrorInvalidDevice);
    std::lock_guard<std::mutex> lk(g_attr_mu);
    if (smem > done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return static_cast<int>(e);
        // all of the unified L1 / shared memory as shared memory: these kernels
        // are latency-bound and live on the number of resident CTAs
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 static_cast<int>(cudaSharedmemCarveoutMaxShared));
        if (e != cudaSuccess) return static_cast<int>(e);
        done[dev] = smem;
    }
    return 0;
}

}  // namespace

size_t cand_smem_bytes(int32_t k, int32_t cap, bool pos16, int32_t *fb_cap)
{
    const size_t out = static_cast<size_t>(k + SLACK) * 8;
    const size_t plain = CAND_HEAD_C + out + static_cast<size_t>(cap) * (4 + (pos16 ? 2 : 4));
    // the fallback stages at least max(k, 1024) keys and positions
    const size_t fb_min = SEL_HEAD + out + static_cast<size_t>(std::max(k, 1024)) * 8;
    const size_t bytes = (std::max(plain, fb_min) + 15) / 16 * 16;
    if (fb_cap) *fb_cap = static_cast<int32_t>((bytes - SEL_HEAD - out) / 8);
    return bytes;
}

size_t cand_cluster_smem_bytes(int32_t k, int32_t cap)
{
    // the cluster kernel keeps the layout with the larger head and 32-bit positions
    const size_t base = CAND_HEAD + static_cast<size_t>(k + SLACK) * 8 + static_cast<size_t>(cap) * 8;
    return base + 16 + 2 * NBINS * 4 + sizeof(ClusterInfo);   // 16: alignment of the counts
}

namespace {

std::mutex g_cluster_mu;
int g_max_cluster[64][2] = {};       // per device: the queried maximum and the shared memory it was asked for

// CTAs per row of the candidate selector: pref 0 (automatic) and 1 = one CTA
// per row; 2, 4, 8 = that cluster size, capped by the largest cluster the
// device reports it can co-schedule for this kernel and shared-memory size.
// Automatic stays at one CTA per row: measured on the 64-row decode batch
// (k 2,048), clusters of 2 / 4 / 8 took the selector from 18.1 us to 18.6 /
// 24.4 / 58.6 us; the per-row phases are latency-bound and do not shrink by
// the split as fast as the merge's barriers and remote traffic cost.
int cand_cluster_size(const SelectParams &p, int pref)
{
    if (pref <= 1) return 1;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 1;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    (void)sms;
    const int want = pref;
    const int csmem = static_cast<int>(cand_cluster_smem_bytes(p.k, p.cap));
    std::lock_guard<std::mutex> lk(g_cluster_mu);
    if (g_max_cluster[dev][1] != csmem) {
        int maxc = 1;
        if (cudaFuncSetAttribute(cand_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, csmem) == cudaSuccess) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(8);
            cfg.blockDim = dim3(CT);
            cfg.dynamicSmemBytes = static_cast<size_t>(csmem);
            if (cudaOccupancyMaxPotentialClusterSize(&maxc, reinterpret_cast<const void *>(&cand_cluster_kernel), &cfg) !=
                cudaSuccess)
                maxc = 1;
        }
        cudaGetLastError();
        g_max_cluster[dev][0] = std::max(1, std::min(8, maxc));
        g_max_cluster[dev][1] = csmem;
    }
    int C = 1;
    while (C * 2 <= std::min(want, g_max_cluster[dev][0])) C *= 2;
    return C;
}

}  // namespace

int last_cluster = 1;

int launch_select(const SelectParams &p, int grid, bool overlap, void *stream, int cluster_pref)
{
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    void *args[] = {const_cast<SelectParams *>(&p)};
    if (grid <= 0) return static_cast<int>(cudaGetLastError());
    if (p.mode == SEL_THRESH) {
        // p.smem_cap: staged scores per row, a multiple of 4 and at most TH_STAGE
        if (p.smem_cap < 0 || p.smem_cap > TH_STAGE || (p.smem_cap & 3)) return static_cast<int>(cudaErrorInvalidValue);
        // a wider block for long samples (sparser sampling at small k)
        if (p.smem_cap <= 4096) {
            static size_t done[64] = {};
            const size_t smem = sizeof(ThShared<128>) + static_cast<size_t>(p.smem_cap) * 4;
            if (int rc = set_smem(thresh_kernel<128>, smem, done)) return rc;
            return launch_kernel(reinterpret_cast<const void *>(&thresh_kernel<128>), dim3(p.R), dim3(128), smem, st,
                                 overlap, args);
        } else {
            static size_t done[64] = {};
            const size_t smem = sizeof(ThShared<256>) + static_cast<size_t>(p.smem_cap) * 4;
            if (int rc = set_smem(thresh_kernel<256>, smem, done)) return rc;
            return launch_kernel(reinterpret_cast<const void *>(&thresh_kernel<256>), dim3(p.R), dim3(256), smem, st,
                                 overlap, args);
        }
    }
    if (p.mode == SEL_CAND) {
        // few rows: one thread-block cluster per row, its size from the
        // device's occupancy query; a refused launch retries at half the size
        // and ends at one CTA per row
        int C = cand_cluster_size(p, cluster_pref);
        while (C > 1) {
            static size_t cdone[64] = {};
            const size_t csmem = cand_cluster_smem_bytes(p.k, p.cap);
            if (int rc = set_smem(cand_cluster_kernel, csmem, cdone)) return rc;
            cudaLaunchAttribute attr[2];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = static_cast<unsigned>(C);
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[1].val.programmaticStreamSerializationAllowed = 1;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(static_cast<unsigned>(p.R) * static_cast<unsigned>(C));
            cfg.blockDim = dim3(CT);
            cfg.dynamicSmemBytes = csmem;
            cfg.stream = st;
            cfg.attrs = attr;
            cfg.numAttrs = overlap ? 2u : 1u;
            if (cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(&cand_cluster_kernel), args) == cudaSuccess &&
                cudaGetLastError() == cudaSuccess) {
                last_cluster = C;
                return 0;
            }
            cudaGetLastError();             // refused: a smaller cluster, or none
            C /= 2;
        }
        last_cluster = 1;
        // 16-bit positions when every row fits (four CTAs per SM at k = 2,048)
        const bool pos16 = p.max_len <= 65536;
        SelectParams q = p;
        const size_t smem = cand_smem_bytes(p.k, p.cap, pos16, &q.smem_cap);
        void *qargs[] = {&q};
        if (pos16) {
            static size_t done16[64] = {};
            if (int rc = set_smem(cand_kernel<uint16_t>, smem, done16)) return rc;
            return launch_kernel(reinterpret_cast<const void *>(&cand_kernel<uint16_t>), dim3(p.R), dim3(CT), smem,
                                 st, overlap, qargs);
        }
        static size_t done32[64] = {};
        if (int rc = set_smem(cand_kernel<uint32_t>, smem, done32)) return rc;
        return launch_kernel(reinterpret_cast<const void *>(&cand_kernel<uint32_t>), dim3(p.R), dim3(CT), smem, st,
                             overlap, qargs);
    }
    if (p.k <= WK)                          // small k: one warp per row
        return launch_kernel(reinterpret_cast<const void *>(&warp_topk_kernel<WK>), dim3((p.R + 7) / 8), dim3(256), 0,
                             st, overlap, args);
    static size_t done[64] = {};
    const size_t smem = sizeof(SelShared) + static_cast<size_t>(out_capacity(p)) * 8 +
                        static_cast<size_t>(p.smem_cap) * 8;
    if (int rc = set_smem(select_kernel, smem, done)) return rc;
    return launch_kernel(reinterpret_cast<const void *>(&select_kernel), dim3(grid), dim3(NT), smem, st, overlap, args);
}

}  // namespace qsa
