// sa_topk.cu -- top-k selection of compressed positions for sm_103a.
//
// The index lists of the "DeepSeek-V4.1 > 40 layers" page come from an
// indexer (`_compress_topk_idxs`: `idxs = self.indexer(x, qr, latent,
// start_pos, offset)`, `index_topk` = 512 positions, int32, offset by the
// window length `kv.size(1)`, -1 where fewer positions exist).  Its scoring
// body is not on the pages; this is the selection over given scores:
//   per row, the k largest scores among those that are not -inf or NaN
//   (masked positions), ties to the smaller position; the chosen positions,
//   in ascending order, plus `offset`; -1 after them when fewer than k exist.
//
// One CTA per row.  Scores become order-preserving 32-bit keys; a four-pass
// radix select (8 bits per pass, most significant first) finds the k-th
// largest key: each pass histograms the keys that share the prefix chosen so
// far (the first pass, where a few bins take most keys, into one histogram
// per warp, summed afterwards) and a block-wide scan over the bins, largest
// first, picks the bin that holds the k-th key.  The first pass is folded
// into the pass that computes the keys.  The ordered pass gives each warp a
// contiguous range of positions: the warps count their keys above the
// threshold and equal to it, and then write, with ballots, every position
// above it and the first positions equal to it, so that the output is in
// ascending position order.  Rows of up to CACHE_KEYS scores keep their keys
// in shared memory; longer rows are read again from global memory (L2) on
// every pass.
#include "sa_internal.h"
#include "sa_ptx.cuh"

namespace sa {
namespace topk {

constexpr int THREADS = 256, WARPS = THREADS / 32;
constexpr int CACHE_KEYS = 16384;   // 64 KB of keys in shared memory
constexpr int BATCH = 16;           // scores a thread loads before it uses any of them

// Order-preserving key of an fp32 score (larger score -> larger key, equal
// scores -> equal keys, so -0 and +0 tie as they compare equal); 0 for scores
// that are never selected (-inf, NaN), which no selectable score maps to
// (every selectable key is at least 0x00800000).
__device__ __forceinline__ uint32_t key_of(float x)
{
    if (x != x || x == -INFINITY)
        return 0u;
    const uint32_t b = x == 0.0f ? 0u : __float_as_uint(x);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Inclusive block-wide sum of one int per thread; also returns the total.
__device__ __forceinline__ int block_scan(int v, int *warp_sums, int &total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o)
            x += y;
    }
    if (lane == 31)
        warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int s = lane < WARPS ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o)
                s += y;
        }
        if (lane < WARPS)
            warp_sums[lane] = s;
    }
    __syncthreads();
    total = warp_sums[WARPS - 1];
    const int before = warp > 0 ? warp_sums[warp - 1] : 0;
    __syncthreads();
    return before + x;
}

static_assert(THREADS == 256, "one thread per histogram bin");

// CACHED: the row's keys stay in shared memory (L <= CACHE_KEYS)
template <bool CACHED>
__global__ void __launch_bounds__(THREADS) topk_kernel(const float *__restrict__ scores, int64_t row_stride,
                                                       int L, int k, int offset, int32_t *__restrict__ out)
{
    extern __shared__ uint32_t cache[];   // keys of this row when L <= CACHE_KEYS
    __shared__ int hist[256];
    __shared__ int whist[WARPS][256];     // first pass: one histogram per warp
    __shared__ int warp_sums[WARPS];
    __shared__ int wcount[2][WARPS];
    __shared__ uint32_t sel_prefix;
    __shared__ int sel_remaining;
    const int64_t row = blockIdx.x;
    const float *src = scores + row * row_stride;
    int32_t *dst = out + row * (int64_t)k;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    auto key_at = [&](int j) -> uint32_t {
        if constexpr (CACHED)
            return cache[j];
        else
            return key_of(__ldg(src + j));
    };

    // keys (into shared memory when they fit), the number of selectable
    // positions and the histogram of their top byte (one per warp, summed)
#pragma unroll
    for (int w = 0; w < WARPS; ++w)
        whist[w][t] = 0;
    __syncthreads();
    int nv = 0;
    for (int base = 0; base < L; base += THREADS * BATCH) {
        float v[BATCH];
#pragma unroll
        for (int u = 0; u < BATCH; ++u) {
            const int j = base + THREADS * u + t;
            v[u] = j < L ? __ldg(src + j) : -INFINITY;
        }
#pragma unroll
        for (int u = 0; u < BATCH; ++u) {
            const int j = base + THREADS * u + t;
            const uint32_t kk = key_of(v[u]);   // 0 past the end
            if (CACHED && j < L)
                cache[j] = kk;
            nv += kk != 0u;
            if (kk != 0u)
                atomicAdd(&whist[warp][kk >> 24], 1);
        }
    }
    int valid = 0;
    block_scan(nv, warp_sums, valid);
    {
        int sum = 0;
#pragma unroll
        for (int w = 0; w < WARPS; ++w)
            sum += whist[w][t];
        hist[t] = sum;
    }
    __syncthreads();

    // threshold: the k-th largest key and how many keys equal to it are taken;
    // with no more than k selectable keys, all of them (threshold 1, below
    // every selectable key)
    uint32_t thr = 1u;
    int take_eq = 0;
    if (valid > k) {
        uint32_t prefix = 0u, mask = 0u;
        int need = k;
        for (int pass = 3; pass >= 0; --pass) {
            const int shift = 8 * pass;
            if (pass < 3) {
                hist[t] = 0;
                __syncthreads();
                for (int base = 0; base < L; base += THREADS * BATCH) {
                    uint32_t kb[BATCH];
#pragma unroll
                    for (int u = 0; u < BATCH; ++u) {
                        const int j = base + THREADS * u + t;
                        kb[u] = j < L ? key_at(j) : 0u;
                    }
                    // below the top byte the keys that share a prefix spread over
                    // the bins: plain atomics
#pragma unroll
                    for (int u = 0; u < BATCH; ++u)
                        if (kb[u] != 0u && (kb[u] & mask) == prefix)
                            atomicAdd(&hist[(kb[u] >> shift) & 255u], 1);
                }
                __syncthreads();
            }
            // thread i holds bin 255 - i: the running count from the top first
            // reaches `need` in the bin of the need-th largest key
            const int c = hist[255 - t];
            int tot = 0;
            const int cum = block_scan(c, warp_sums, tot);
            if (cum >= need && cum - c < need) {
                sel_prefix = prefix | ((uint32_t)(255 - t) << shift);
                sel_remaining = need - (cum - c);
            }
            __syncthreads();
            prefix = sel_prefix;
            need = sel_remaining;
            mask |= 0xFFu << shift;
            __syncthreads();
        }
        thr = prefix;
        take_eq = need;
    }

    // ordered pass: warp w takes positions [w0, w1), a multiple of 32 wide
    const int per = ((L + WARPS - 1) / WARPS + 31) & ~31;
    const int w0 = min(L, warp * per), w1 = min(L, w0 + per);
    int gt = 0, eq = 0;
    for (int base = w0; base < w1; base += 32) {
        const int j = base + lane;
        const uint32_t kk = j < w1 ? key_at(j) : 0u;
        gt += __popc(__ballot_sync(0xffffffffu, kk > thr));
        eq += __popc(__ballot_sync(0xffffffffu, kk == thr && kk != 0u));
    }
    if (lane == 0) {
        wcount[0][warp] = gt;
        wcount[1][warp] = eq;
    }
    __syncthreads();
    int gt_before = 0, eq_before = 0, gt_all = 0, eq_all = 0;
#pragma unroll
    for (int i = 0; i < WARPS; ++i) {
        gt_before += i < warp ? wcount[0][i] : 0;
        eq_before += i < warp ? wcount[1][i] : 0;
        gt_all += wcount[0][i];
        eq_all += wcount[1][i];
    }
    int pos = gt_before + min(eq_before, take_eq);
    int eq_seen = eq_before;
    const unsigned below = (1u << lane) - 1u;
    for (int base = w0; base < w1; base += 32) {
        const int j = base + lane;
        const uint32_t kk = j < w1 ? key_at(j) : 0u;
        const bool is_eq = kk == thr && kk != 0u;
        const unsigned eqm = __ballot_sync(0xffffffffu, is_eq);
        const bool take = kk > thr || (is_eq && eq_seen + __popc(eqm & below) < take_eq);
        const unsigned tm = __ballot_sync(0xffffffffu, take);
        if (take) {
            const int o = pos + __popc(tm & below);
            if (o < k)
                dst[o] = j + offset;
        }
        pos += __popc(tm);
        eq_seen += __popc(eqm);
    }
    const int taken = gt_all + min(eq_all, take_eq);
    for (int i = min(taken, k) + t; i < k; i += THREADS)
        dst[i] = -1;
}

}  // namespace topk

cudaError_t launch_topk(const float *scores, int64_t row_stride, int64_t rows, int L, int k, int offset,
                        int32_t *out, cudaStream_t st)
{
    if (rows == 0 || k == 0)
        return cudaSuccess;
    if (L <= topk::CACHE_KEYS) {
        cudaError_t e = cudaFuncSetAttribute(topk::topk_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)(topk::CACHE_KEYS * 4));
        if (e != cudaSuccess)
            return e;
        topk::topk_kernel<true><<<(unsigned)rows, topk::THREADS, (size_t)L * 4, st>>>(scores, row_stride, L, k,
                                                                                     offset, out);
    } else {
        topk::topk_kernel<false><<<(unsigned)rows, topk::THREADS, 0, st>>>(scores, row_stride, L, k, offset, out);
    }
    return cudaGetLastError();
}

}  // namespace sa
