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
// largest key; one ordered pass then writes every position above it and the
// first positions equal to it, with block-wide prefix counts so that the
// output is in ascending position order.  Rows of up to CACHE_KEYS scores
// keep their keys in shared memory; longer rows are read again from global
// memory (L2) on every pass.
#include "sa_internal.h"
#include "sa_ptx.cuh"

namespace sa {
namespace topk {

constexpr int THREADS = 256;
constexpr int CACHE_KEYS = 16384;   // 64 KB of keys in shared memory

// Order-preserving key of an fp32 score (larger score -> larger key, equal
// scores -> equal keys, so -0 and +0 tie as they compare equal); 0 for scores
// that are never selected (-inf, NaN), which no selectable score maps to.
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
        int s = lane < THREADS / 32 ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o)
                s += y;
        }
        if (lane < THREADS / 32)
            warp_sums[lane] = s;
    }
    __syncthreads();
    total = warp_sums[THREADS / 32 - 1];
    const int before = warp > 0 ? warp_sums[warp - 1] : 0;
    __syncthreads();
    return before + x;
}

__global__ void __launch_bounds__(THREADS) topk_kernel(const float *__restrict__ scores, int64_t row_stride,
                                                       int L, int k, int offset, int32_t *__restrict__ out)
{
    extern __shared__ uint32_t cache[];   // keys of this row when L <= CACHE_KEYS
    __shared__ int hist[256];
    __shared__ int warp_sums[THREADS / 32];
    __shared__ uint32_t sel_prefix, sel_mask;
    __shared__ int sel_remaining, n_valid;
    const int64_t row = blockIdx.x;
    const float *src = scores + row * row_stride;
    int32_t *dst = out + row * (int64_t)k;
    const bool cached = L <= CACHE_KEYS;
    const int t = threadIdx.x;
    auto key_at = [&](int j) -> uint32_t { return cached ? cache[j] : key_of(__ldg(src + j)); };

    // keys (into shared memory when they fit) and the number of selectable positions
    int nv = 0;
    for (int j = t; j < L; j += THREADS) {
        const uint32_t kk = key_of(__ldg(src + j));
        if (cached)
            cache[j] = kk;
        nv += kk != 0u;
    }
    int total = 0;
    block_scan(nv, warp_sums, total);
    if (t == 0) {
        n_valid = total;
        sel_prefix = 0u;
        sel_mask = 0u;
        sel_remaining = k;
    }
    __syncthreads();
    const int valid = n_valid;

    // threshold: the k-th largest key (or the smallest selectable one when
    // there are no more than k); sel_remaining = how many keys equal to it are taken
    if (valid > k) {
        for (int pass = 3; pass >= 0; --pass) {
            for (int i = t; i < 256; i += THREADS)
                hist[i] = 0;
            __syncthreads();
            const uint32_t prefix = sel_prefix, mask = sel_mask;
            const int shift = 8 * pass;
            for (int j = t; j < L; j += THREADS) {
                const uint32_t kk = key_at(j);
                if (kk != 0u && (kk & mask) == prefix)
                    atomicAdd(&hist[(kk >> shift) & 255u], 1);
            }
            __syncthreads();
            if (t == 0) {
                int need = sel_remaining, b = 255;
                for (; b > 0; --b) {
                    if (hist[b] >= need)
                        break;
                    need -= hist[b];
                }
                sel_prefix = prefix | ((uint32_t)b << shift);
                sel_mask = mask | (0xFFu << shift);
                sel_remaining = need;
            }
            __syncthreads();
        }
    }
    const uint32_t thr = valid > k ? sel_prefix : 1u;   // 1: every selectable key is taken
    const int take_eq = valid > k ? sel_remaining : L;

    // ordered pass: positions above the threshold, then the first take_eq equal to it
    int written = 0, eq_seen = 0;
    for (int base = 0; base < L; base += THREADS) {
        const int j = base + t;
        const uint32_t kk = j < L ? key_at(j) : 0u;
        const int is_gt = kk > thr ? 1 : 0;
        const int is_eq = (kk == thr && kk != 0u) ? 1 : 0;
        int eq_total = 0;
        const int eq_rank = block_scan(is_eq, warp_sums, eq_total) - is_eq + eq_seen;
        const int take = is_gt | (is_eq & (eq_rank < take_eq ? 1 : 0));
        int take_total = 0;
        const int pos = block_scan(take, warp_sums, take_total) - take + written;
        if (take && pos < k)
            dst[pos] = j + offset;
        written += take_total;
        eq_seen += eq_total;
    }
    const int n_out = written < k ? written : k;
    for (int i = n_out + t; i < k; i += THREADS)
        dst[i] = -1;
}

}  // namespace topk

cudaError_t launch_topk(const float *scores, int64_t row_stride, int64_t rows, int L, int k, int offset,
                        int32_t *out, cudaStream_t st)
{
    if (rows == 0 || k == 0)
        return cudaSuccess;
    const size_t smem = L <= topk::CACHE_KEYS ? (size_t)L * 4 : 0;
    cudaError_t e = cudaFuncSetAttribute(topk::topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(topk::CACHE_KEYS * 4));
    if (e != cudaSuccess)
        return e;
    topk::topk_kernel<<<(unsigned)rows, topk::THREADS, smem, st>>>(scores, row_stride, L, k, offset, out);
    return cudaGetLastError();
}

}  // namespace sa
