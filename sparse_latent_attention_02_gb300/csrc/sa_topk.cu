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
// One CTA of four warps per row (with 4096-score rows nine are resident per
// SM; four warps a row measured faster than two, three, six or eight).
// Scores become order-preserving
// 32-bit keys; a three-pass radix select (11, 11 and 10 bits, most significant
// first) finds the k-th largest key: each pass histograms the keys that share
// the prefix chosen so far into 2048 bins, and one warp scans the bins,
// largest first (64 a lane, then two a lane within the lane's range that holds
// the k-th key), to pick the bin that holds it; the search ends early once
// that bin is taken whole.  The first pass is folded into the pass that
// computes the keys, which also finds the last selectable position: the later
// passes stop there.  The ordered pass gives each warp a contiguous range of
// positions.  When every key above the threshold is taken and none equal to it
// (the usual case: only ties leave a share of equal keys), each warp collects
// its chosen positions in order, with one ballot over 32 positions at a time,
// in its own segment of the histogram's shared memory, and the segments are
// written out one after another.  Otherwise the warps first count their keys
// above the threshold and equal to it, and then write, with ballots, every
// position above it and the first positions equal to it; either way the output
// is in ascending position order.  Rows of up to CACHE_KEYS scores keep their
// keys in shared memory; longer rows are read again from global memory (L2) on
// every pass.
#include "sa_internal.h"
#include "sa_ptx.cuh"

namespace sa {
namespace topk {

constexpr int THREADS = 128, WARPS = THREADS / 32;
constexpr int CACHE_KEYS = 16384;   // 64 KB of keys in shared memory
constexpr int BATCH = 16;           // scores a thread loads before it uses any of them
constexpr int BINS = 2048;          // 11-bit digits
constexpr int SWEEP_VEC = 2;        // groups of four keys a thread loads before it uses any of them
constexpr int VBATCH = 4;           // groups of four scores a thread loads before it uses any of them

// Order-preserving key of an fp32 score (larger score -> larger key, equal
// scores -> equal keys, so -0 and +0 tie as they compare equal); 0 for scores
// that are never selected (-inf, NaN), which no selectable score maps to
// (every selectable key is at least 0x00800000).  Adding +0 turns -0 into +0
// and leaves every other value, subnormals included, as it is (the library
// is built without flush-to-zero).
__device__ __forceinline__ uint32_t key_of(float x)
{
    const uint32_t b = __float_as_uint(x + 0.0f);
    const uint32_t kk = b ^ ((uint32_t)((int32_t)b >> 31) | 0x80000000u);
    return x > -INFINITY ? kk : 0u;
}

static_assert(BINS == 32 * 64, "64 histogram bins per lane in the bin search");

// One warp: the bin of the need-th largest key, counting from the top bin
// down.  Lane l sums bins 2047 - 64l down to 1984 - 64l (its 16-byte loads
// rotated by l, so that eight lanes read eight different bank groups), a scan
// over the lanes finds the lane whose range holds the key, and the warp then
// scans that range two bins a lane.  Gives the bin, the keys still needed
// within it and whether they are all of its keys; returns false instead, with
// nothing found, when `all_if_few` is set and the histogram's total is at
// most `need` (every key is taken).
__device__ __forceinline__ bool find_bin(const int *hist, int need, bool all_if_few, int lane, int &bin,
                                         int &remaining, bool &whole)
{
    const int base = BINS - 64 * (lane + 1);
    int sum = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int4 v = *reinterpret_cast<const int4 *>(&hist[base + 4 * ((i + lane) & 15)]);
        sum += v.x + v.y + v.z + v.w;
    }
    int cum = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, cum, o);
        if (lane >= o)
            cum += y;
    }
    if (all_if_few && __shfl_sync(0xffffffffu, cum, 31) <= need)
        return false;
    const unsigned hit = __ballot_sync(0xffffffffu, cum >= need);
    const int L = hit != 0u ? __ffs(hit) - 1 : 31;
    const int before = __shfl_sync(0xffffffffu, cum - sum, L);
    const int need2 = need - before;
    // lane i: bins 63 - 2i (hi) and 62 - 2i (lo) of lane L's range
    const int b2 = BINS - 64 * (L + 1) + 62 - 2 * lane;
    const int2 pr = *reinterpret_cast<const int2 *>(&hist[b2]);
    const int pair = pr.x + pr.y;
    int cp = pair;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, cp, o);
        if (lane >= o)
            cp += y;
    }
    const unsigned hit2 = __ballot_sync(0xffffffffu, cp >= need2);
    const int I = hit2 != 0u ? __ffs(hit2) - 1 : 31;
    const int run = cp - pair;   // keys in the bins above this lane's pair
    const bool in_hi = run + pr.y >= need2;
    const int my_bin = in_hi ? b2 + 1 : b2;
    const int my_rem = in_hi ? need2 - run : need2 - run - pr.y;
    const bool my_whole = in_hi ? run + pr.y == need2 : run + pr.y + pr.x == need2;
    bin = __shfl_sync(0xffffffffu, my_bin, I);
    remaining = __shfl_sync(0xffffffffu, my_rem, I);
    whole = __shfl_sync(0xffffffffu, (int)my_whole, I) != 0;
    return true;
}
// positions a warp can stage in its segment of the histogram's memory (16 bits each)
constexpr int STAGE_PER_WARP = BINS * 2 / WARPS;   // 1024

// CACHED: the row's keys stay in shared memory (L <= CACHE_KEYS)
template <bool CACHED>
__global__ void __launch_bounds__(THREADS, CACHED ? 9 : 8) topk_kernel(const float *__restrict__ scores, int64_t row_stride,
                                                       int L, int k, int offset, int32_t *__restrict__ out)
{
    extern __shared__ __align__(16) uint32_t cache[];   // keys of this row when L <= CACHE_KEYS
    __shared__ __align__(16) int hist[BINS];
    __shared__ int wcount[2][WARPS];
    __shared__ uint32_t sel_prefix;
    __shared__ int sel_remaining;
    __shared__ bool sel_whole;
    __shared__ bool sel_all;
    __shared__ int last_valid;
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
    // keys j .. j+3 (j a multiple of 4), 0 from position lim on
    auto keys4 = [&](int j, int lim, uint32_t *kb) {
        if constexpr (CACHED) {
            if (j + 4 <= lim) {
                const uint4 v = *reinterpret_cast<const uint4 *>(cache + j);
                kb[0] = v.x;
                kb[1] = v.y;
                kb[2] = v.z;
                kb[3] = v.w;
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    kb[i] = j + i < lim ? cache[j + i] : 0u;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                kb[i] = j + i < lim ? key_of(__ldg(src + j + i)) : 0u;
        }
    };

    // keys (into shared memory when they fit), the histogram of their top 11
    // bits and the last selectable position: the later passes stop after it
    // (a causal row ends in masked positions).  A thread visits its
    // positions in increasing order, so the last one it saw is its largest.
    for (int i = t; i < BINS / 4; i += THREADS)
        reinterpret_cast<int4 *>(hist)[i] = make_int4(0, 0, 0, 0);
    if (t == 0)
        last_valid = -1;
    __syncthreads();
    int last = -1;
    if ((reinterpret_cast<uintptr_t>(src) & 15u) == 0u) {
        // 16-byte aligned row: four scores a load
        constexpr int VB = CACHED ? VBATCH : VBATCH / 2;   // the uncached kernel has fewer registers to spare
        for (int base = 0; base < L; base += 4 * THREADS * VB) {
            float4 v[VB];
#pragma unroll
            for (int u = 0; u < VB; ++u) {
                const int j = base + 4 * (THREADS * u + t);
                if (j + 4 <= L) {
                    v[u] = __ldg(reinterpret_cast<const float4 *>(src + j));
                } else {
                    v[u].x = j < L ? __ldg(src + j) : -INFINITY;
                    v[u].y = j + 1 < L ? __ldg(src + j + 1) : -INFINITY;
                    v[u].z = j + 2 < L ? __ldg(src + j + 2) : -INFINITY;
                    v[u].w = -INFINITY;   // j + 3 >= L here
                }
            }
#pragma unroll
            for (int u = 0; u < VB; ++u) {
                const int j = base + 4 * (THREADS * u + t);
                const uint32_t kk[4] = {key_of(v[u].x), key_of(v[u].y), key_of(v[u].z), key_of(v[u].w)};
                if (CACHED) {
                    if (j + 4 <= L) {
                        *reinterpret_cast<uint4 *>(cache + j) = make_uint4(kk[0], kk[1], kk[2], kk[3]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            if (j + i < L)
                                cache[j + i] = kk[i];
                    }
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (kk[i] != 0u)   // 0 past the end
                        atomicAdd(&hist[kk[i] >> 21], 1);
                // the last selectable position, to the end of its group of four
                if ((kk[0] | kk[1] | kk[2] | kk[3]) != 0u)
                    last = j + 3;
            }
        }
    } else {
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
                if (kk != 0u) {
                    atomicAdd(&hist[kk >> 21], 1);
                    last = j;
                }
            }
        }
    }
    last = __reduce_max_sync(0xffffffffu, last);
    if (lane == 0)
        atomicMax(&last_valid, last);
    __syncthreads();
    const int Lv = min(last_valid + 1, L);   // positions from Lv on are all masked

    // threshold: every key above thr is taken, and the first take_eq keys
    // equal to it.  With no more than k selectable keys (the histogram's
    // total), all of them: thr 1, below every selectable key.  A pass whose
    // chosen bin holds exactly the keys still needed ends the search: thr is
    // then the largest key below that bin.
    uint32_t thr = 1u;
    int take_eq = 0;
    {
        uint32_t prefix = 0u, mask = 0u;
        int need = k;
#pragma unroll 1
        for (int pass = 0; pass < 3; ++pass) {
            const int shift = pass == 0 ? 21 : pass == 1 ? 10 : 0;
            const uint32_t dmask = pass < 2 ? 2047u : 1023u;
            if (pass > 0) {
                for (int i = t; i < BINS / 4; i += THREADS)
                    reinterpret_cast<int4 *>(hist)[i] = make_int4(0, 0, 0, 0);
                __syncthreads();
                for (int base = 0; base < Lv; base += 4 * THREADS * SWEEP_VEC) {
                    uint32_t kb[4 * SWEEP_VEC];
#pragma unroll
                    for (int u = 0; u < SWEEP_VEC; ++u)
                        keys4(base + 4 * (THREADS * u + t), Lv, kb + 4 * u);
                    // below the top digit the keys that share a prefix spread over
                    // the bins: plain atomics (no key of 0 matches: every prefix
                    // chosen is nonzero)
#pragma unroll
                    for (int u = 0; u < 4 * SWEEP_VEC; ++u)
                        if ((kb[u] & mask) == prefix)
                            atomicAdd(&hist[(kb[u] >> shift) & dmask], 1);
                }
                __syncthreads();
            }
            // one warp finds the bin of the need-th largest key; with no more
            // than k selectable keys in the first pass (the histogram's total),
            // all of them are taken
            if (warp == 0) {
                int bin = 0, rem = 0;
                bool wh = false;
                const bool found = find_bin(hist, need, pass == 0, lane, bin, rem, wh);
                if (lane == 0) {
                    sel_all = !found;
                    sel_prefix = prefix | ((uint32_t)bin << shift);
                    sel_remaining = rem;
                    sel_whole = wh;
                }
            }
            __syncthreads();
            if (sel_all)   // the same in every thread
                break;
            prefix = sel_prefix;
            need = sel_remaining;
            mask |= dmask << shift;
            const bool whole = sel_whole;
            // (warp 0 writes the selection again only after the next pass's
            // two barriers, which every thread reaches after reading it)
            if (whole) {   // every key of the bin is taken
                thr = prefix - 1u;
                take_eq = 0;
                break;
            }
            if (pass == 2) {   // the bin is one key value
                thr = prefix;
                take_eq = need;
            }
        }
    }

    // ordered pass over the positions before Lv: warp w takes [w0, w1), a
    // multiple of 128 wide; its counts read four consecutive keys a lane
    const int per = ((Lv + WARPS - 1) / WARPS + 127) & ~127;
    const int w0 = min(Lv, warp * per), w1 = min(Lv, w0 + per);
    const unsigned below = (1u << lane) - 1u;
    if (CACHED && take_eq == 0 && k <= STAGE_PER_WARP) {
        // every key above thr is taken, no other (at most k of them): each warp
        // stages its positions (below CACHE_KEYS: 16 bits) in order in its own
        // segment of the histogram's memory, which the passes are done with
        uint16_t *seg = reinterpret_cast<uint16_t *>(hist) + warp * STAGE_PER_WARP;
        int n = 0;
        for (int base = w0; base < w1; base += 128) {
            uint32_t kb[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int j = base + 32 * i + lane;
                kb[i] = j < w1 ? key_at(j) : 0u;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const bool take = kb[i] > thr;
                const unsigned tm = __ballot_sync(0xffffffffu, take);
                const int o = n + __popc(tm & below);
                if (take && o < STAGE_PER_WARP)
                    seg[o] = (uint16_t)(base + 32 * i + lane);
                n += __popc(tm);
            }
        }
        if (lane == 0)
            wcount[0][warp] = n;
        __syncthreads();
        int before = 0, all = 0;
#pragma unroll
        for (int i = 0; i < WARPS; ++i) {
            before += i < warp ? wcount[0][i] : 0;
            all += wcount[0][i];
        }
        const int m = min(min(n, STAGE_PER_WARP), max(0, k - before));
        for (int i = lane; i < m; i += 32)
            dst[before + i] = (int)seg[i] + offset;
        for (int i = min(all, k) + t; i < k; i += THREADS)
            dst[i] = -1;
        return;
    }
    // (no key of 0 equals thr: thr is 1 or a selectable key)
    int gt = 0, eq = 0;
    for (int base = w0; base < w1; base += 128) {
        uint32_t kb[4];
        keys4(base + 4 * lane, w1, kb);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            gt += kb[i] > thr;
            eq += kb[i] == thr;
        }
    }
    gt = __reduce_add_sync(0xffffffffu, gt);
    eq = __reduce_add_sync(0xffffffffu, eq);
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
    // writes: lane l takes keys base + l, base + 32 + l, ... so that each
    // ballot covers 32 consecutive positions; pos counts the positions
    // written before them, eq_seen the keys equal to thr (the first take_eq
    // of all are taken)
    int pos = gt_before + min(eq_before, take_eq);
    int eq_seen = eq_before;
    for (int base = w0; base < w1; base += 128) {
        uint32_t kb[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int j = base + 32 * i + lane;
            kb[i] = j < w1 ? key_at(j) : 0u;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const bool is_eq = kb[i] == thr;
            const unsigned eqm = __ballot_sync(0xffffffffu, is_eq);
            bool take = kb[i] > thr;
            if (eqm != 0u)   // the same in every lane
                take = take || (is_eq && eq_seen + __popc(eqm & below) < take_eq);
            const unsigned tm = __ballot_sync(0xffffffffu, take);
            if (take) {
                const int o = pos + __popc(tm & below);
                if (o < k)
                    dst[o] = base + 32 * i + lane + offset;
            }
            pos += __popc(tm);
            eq_seen += __popc(eqm);
        }
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
