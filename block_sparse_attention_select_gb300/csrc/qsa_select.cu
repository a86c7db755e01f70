// Exact top-k selector: one CTA per query row, radix select on order-preserving
// keys.  A score becomes key32 = score_key(score) (larger score -> larger key)
// and an element's full key is (key32, ~position), so larger full key = higher
// score, then lower position: the exact lexicographic order with its
// deterministic tie rule.  Selection runs digit by digit (11, 11, 10 bits of
// key32, then of ~position only when the cutoff score is tied) with shared
// histograms; the k winners are gathered and sorted (bitonic, shared memory).
#include <cuda_runtime.h>

#include "qsa_device.cuh"
#include "qsa_internal.h"

namespace qsa {
namespace {

constexpr int NT = 512;               // threads per row
constexpr int NBINS = 2048;           // 11-bit digits
// digit levels of a 32-bit key: bits 31..21, 20..10, 9..0
__device__ __forceinline__ int level_shift(int lv) { return lv == 0 ? 21 : (lv == 1 ? 10 : 0); }
__device__ __forceinline__ uint32_t level_mask(int lv) { return lv < 2 ? 0x7FFu : 0x3FFu; }

struct SelShared {
    uint32_t hist[NBINS];
    uint32_t wtot[32];
    uint32_t cut_digit, cut_above, count, total, taken, pad_[3];
};

// Largest digit d with (# elements of digit > d) < k_rem, i.e. the digit that
// holds the k_rem-th largest element; returns it with the count above it.
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

__device__ __forceinline__ void clear_hist(SelShared &sh)
{
    for (int i = threadIdx.x; i < NBINS; i += NT) sh.hist[i] = 0;
    __syncthreads();
}

// Radix select over the n elements in (keys, inv) held in shared memory:
// gathers the top kk by (key32, inv) into sortbuf (unordered), kk <= n.
__device__ void smem_select_gather(SelShared &sh, const uint32_t *keys, const uint32_t *inv,
                                   int32_t n, int32_t kk, uint64_t *sortbuf)
{
    uint32_t T = 0, U = 0;
    if (kk < n) {
        uint32_t prefix = 0, pmask = 0, k_rem = static_cast<uint32_t>(kk), eq = 0;
        for (int lv = 0; lv < 3; ++lv) {
            clear_hist(sh);
            for (int32_t i = threadIdx.x; i < n; i += NT) {
                const uint32_t key = keys[i];
                if ((key & pmask) == prefix)
                    atomicAdd(&sh.hist[(key >> level_shift(lv)) & level_mask(lv)], 1u);
            }
            __syncthreads();
            find_cut(sh, k_rem);
            const uint32_t d = sh.cut_digit;
            k_rem -= sh.cut_above;
            eq = sh.hist[d];
            prefix |= d << level_shift(lv);
            pmask |= level_mask(lv) << level_shift(lv);
            __syncthreads();
        }
        T = prefix;
        if (eq > k_rem) {
            // cutoff score tied: keep the k_rem lowest positions (largest ~position)
            uint32_t p2 = 0, m2 = 0;
            for (int lv = 0; lv < 3; ++lv) {
                clear_hist(sh);
                for (int32_t i = threadIdx.x; i < n; i += NT) {
                    const uint32_t v = inv[i];
                    if (keys[i] == T && (v & m2) == p2)
                        atomicAdd(&sh.hist[(v >> level_shift(lv)) & level_mask(lv)], 1u);
                }
                __syncthreads();
                find_cut(sh, k_rem);
                const uint32_t d = sh.cut_digit;
                k_rem -= sh.cut_above;
                p2 |= d << level_shift(lv);
                m2 |= level_mask(lv) << level_shift(lv);
                __syncthreads();
            }
            U = p2;
        }
    }
    if (threadIdx.x == 0) sh.count = 0;
    __syncthreads();
    for (int32_t i = threadIdx.x; i < n; i += NT) {
        const uint32_t key = keys[i], v = inv[i];
        if (kk >= n || key > T || (key == T && v >= U)) {
            const uint32_t slot = atomicAdd(&sh.count, 1u);
            sortbuf[slot] = (static_cast<uint64_t>(key) << 32) | v;
        }
    }
    __syncthreads();
}

// Descending bitonic sort of sortbuf[0, npow2); entries past `valid` are zero.
__device__ void bitonic_desc(uint64_t *buf, int32_t valid, int32_t npow2)
{
    for (int32_t i = valid + threadIdx.x; i < npow2; i += NT) buf[i] = 0;
    __syncthreads();
    for (int32_t size = 2; size <= npow2; size <<= 1) {
        for (int32_t stride = size >> 1; stride > 0; stride >>= 1) {
            for (int32_t i = threadIdx.x; i < (npow2 >> 1); i += NT) {
                const int32_t a = 2 * stride * (i / stride) + (i % stride);
                const int32_t b = a + stride;
                const uint64_t x = buf[a], y = buf[b];
                const bool desc = (a & size) == 0;
                if ((x < y) == desc) {
                    buf[a] = y;
                    buf[b] = x;
                }
            }
            __syncthreads();
        }
    }
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

// Streaming radix passes over a row in global memory (scores, implicit
// positions).  Narrows the cut digit by digit until the elements at or above
// it fit in the shared buffers (then gathers them there) or the cut score is
// exact.  Returns the number of gathered elements, or -1 when the cut is
// exact and still does not fit (T_out, above_out then describe it).
__device__ int32_t stream_narrow(SelShared &sh, const float *__restrict__ row, int32_t n,
                                 uint32_t k, int32_t cap, uint32_t *keys, uint32_t *inv,
                                 uint32_t &T_out, uint32_t &above_out, uint32_t &k_rem_out,
                                 bool gather)
{
    uint32_t prefix = 0, pmask = 0, k_rem = k, above = 0;
    for (int lv = 0; lv < 3; ++lv) {
        clear_hist(sh);
        for (int32_t i = threadIdx.x; i < n; i += NT) {
            const uint32_t key = score_key(__ldg(row + i));
            if ((key & pmask) == prefix)
                atomicAdd(&sh.hist[(key >> level_shift(lv)) & level_mask(lv)], 1u);
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
                const uint32_t key = score_key(__ldg(row + i));
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
    above_out = above;
    k_rem_out = k_rem;
    return -1;
}

__global__ void __launch_bounds__(NT)
select_kernel(const SelectParams p)
{
    extern __shared__ __align__(16) uint8_t smem_raw[];
    SelShared &sh = *reinterpret_cast<SelShared *>(smem_raw);
    uint64_t *sortbuf = reinterpret_cast<uint64_t *>(smem_raw + sizeof(SelShared));
    uint32_t *keys = reinterpret_cast<uint32_t *>(sortbuf + p.sort_cap);
    uint32_t *inv = keys + p.smem_cap;

    const int32_t r = blockIdx.x;
    if (r >= p.R) return;
    int32_t V = p.row_vis[r];
    if (V < 0 || V > p.max_len) {
        if (threadIdx.x == 0) record_error(p.status, ST_BAD_ROW);
        V = static_cast<int32_t>(max(static_cast<int64_t>(0), min(static_cast<int64_t>(V), p.max_len)));
    }

    if (p.mode == SEL_THRESH) {
        // tau_r from the sampled scores of row r (columns [0, n_s) of the sample row)
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
            uint32_t T, above, k_rem;
            stream_narrow(sh, p.logits + static_cast<int64_t>(r) * p.ld, n_s,
                          static_cast<uint32_t>(m), 0, nullptr, nullptr, T, above, k_rem, false);
            tau = key_score(T);
        }
        if (threadIdx.x == 0) {
            p.tau[r] = tau;
            p.cand_count_w[r] = 0;
        }
        return;
    }

    if (p.mode == SEL_DENSE_FLAGGED && p.row_flag[r] == 0) return;

    int32_t n;
    const int32_t kk_target = min(p.k, V);
    if (p.mode == SEL_CAND) {
        const int32_t cnt = p.cand_count[r];
        if (cnt > p.cap || cnt < kk_target) {
            if (threadIdx.x == 0) {
                p.row_flag[r] = 1;
                atomicExch(&p.plan->any_fallback, 1);
            }
            return;
        }
        if (threadIdx.x == 0) p.row_flag[r] = 0;
        const uint2 *src = p.cand + static_cast<int64_t>(r) * p.cap;
        for (int32_t i = threadIdx.x; i < cnt; i += NT) {
            const uint2 e = src[i];
            keys[i] = score_key(__uint_as_float(e.x));
            inv[i] = ~e.y;
        }
        __syncthreads();
        n = cnt;
    } else {
        const float *row = p.logits + static_cast<int64_t>(r) * p.ld;
        if (V <= p.smem_cap) {
            for (int32_t i = threadIdx.x; i < V; i += NT) {
                keys[i] = score_key(__ldg(row + i));
                inv[i] = ~static_cast<uint32_t>(i);
            }
            __syncthreads();
            n = V;
        } else {
            uint32_t T, above, k_rem;
            n = stream_narrow(sh, row, V, static_cast<uint32_t>(kk_target), p.smem_cap, keys, inv,
                              T, above, k_rem, true);
            if (n < 0) {
                // exact cut score with too many ties: everything above it, then the
                // k_rem lowest positions holding the cut score, in position order
                if (threadIdx.x == 0) { sh.count = 0; sh.taken = 0; }
                __syncthreads();
                for (int32_t base = 0; base < V; base += NT) {
                    const int32_t i = base + threadIdx.x;
                    const uint32_t key = i < V ? score_key(__ldg(row + i)) : 0u;
                    if (i < V && key > T) {
                        const uint32_t slot = atomicAdd(&sh.count, 1u);
                        keys[slot] = key;
                        inv[slot] = ~static_cast<uint32_t>(i);
                    }
                    const uint32_t tie = (i < V && key == T) ? 1u : 0u;
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
                        // the rest of the row can only add scores above the cut
                        for (int32_t j = base + NT + threadIdx.x; j < V; j += NT) {
                            const uint32_t kj = score_key(__ldg(row + j));
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
                n = static_cast<int32_t>(sh.count);
            }
        }
    }
    const int32_t kk = min(p.k, n);
    smem_select_gather(sh, keys, inv, n, kk, sortbuf);
    int32_t npow2 = 1;
    while (npow2 < kk) npow2 <<= 1;
    bitonic_desc(sortbuf, kk, npow2);
    write_row(p, r, sortbuf, kk);
}

}  // namespace

size_t select_smem_bytes(int32_t smem_cap, int32_t sort_cap)
{
    return sizeof(SelShared) + static_cast<size_t>(sort_cap) * 8 + static_cast<size_t>(smem_cap) * 8;
}

int launch_select(const SelectParams &p, void *stream)
{
    const size_t smem = select_smem_bytes(p.smem_cap, p.sort_cap);
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
