// sa_attn.cu -- sparse latent attention for sm_103a (tcgen05 + TMEM).
//
// The step is `sparse_attn(q, kv, attn_sink, topk_idxs, softmax_scale)` of the
// `Attention.forward` excerpt on the "DeepSeek-V4.1 > Output projection" page:
// for each query, all 64 heads attend over one list of latent rows gathered
// from kv[b] (keys == values, 512 features), with a per-head sink logit in the
// softmax denominator and -1 meaning "skip".
//
// Design (one CTA per SM, persistent over a static schedule of segments):
//   * A segment is one query's index list (or a contiguous piece of it when
//     there are fewer queries than SMs).  Its valid entries are compacted and
//     processed in chunks of 128 gathered rows.
//   * Transposed orientation, so that every MMA has M = 128:
//       S^T[128 rows x 64 heads]  = K_chunk[128 x 512] . Q^T        (TMEM cols   0..63)
//       O^T[512 feats x 64 heads] += V_chunk^T[512 x 128] . P^T     (TMEM cols 256..511)
//     The chunk sits in shared memory once, 128-byte swizzled; it is the
//     K-major A operand of the first product and the MN-major A operand of
//     the second.  Q (64 KB) stays resident for the whole segment.
//   * Warp roles: warps 0-3 softmax + epilogue (thread i owns TMEM lane i =
//     chunk row i during the softmax, output feature 128*tile + i in the
//     epilogue); warp 4 compacts the index list and gathers rows with 16-byte
//     cp.async into the swizzled layout; warp 5 allocates TMEM and issues the
//     MMAs (one elected lane).
//   * Online softmax in base 2 with the sink as the starting maximum and a
//     lazy rescale: the running maximum moves only when a score exceeds it by
//     more than 2^8, so O^T in TMEM is almost never rewritten.  Row sums are
//     kept per thread (per row) and reduced once per segment.
//   * Every wait is bounded (bounded_wait); a timeout raises a CTA abort flag,
//     all roles leave their loops, in-flight copies and MMAs are drained, TMEM
//     is released and the error word gets ERRBIT_TIMEOUT.
#include <cuda_bf16.h>

#include "sa_internal.h"
#include "sa_ptx.cuh"

namespace sa {
namespace attn {

constexpr int H = 64, D = 512, CH = 128;
constexpr int THREADS = 192;
constexpr int WARP_PRODUCER = 4, WARP_MMA = 5;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float RESCALE_THRESHOLD = 8.0f;   // log2 units

constexpr uint32_t QBLK_BYTES = H * 64 * 2;     // one 64-feature block of Q: 8 KB
constexpr uint32_t Q_BYTES = 8 * QBLK_BYTES;    // 64 KB
constexpr uint32_t SLICE_BYTES = CH * 64 * 2;   // one 64-feature slice of a chunk: 16 KB
constexpr uint32_t KV_BYTES = 8 * SLICE_BYTES;  // 128 KB
constexpr uint32_t P_BYTES = CH * H * 2;        // 16 KB

constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_KV = OFF_Q + Q_BYTES;
constexpr uint32_t OFF_P = OFF_KV + KV_BYTES;
constexpr uint32_t OFF_IDX = OFF_P + P_BYTES;
constexpr uint32_t OFF_RED = OFF_IDX + 4 * SA_MAX_K;   // float [4][64]
constexpr uint32_t OFF_M = OFF_RED + 4 * 64 * 4;       // float [64] running max (log2 units)
constexpr uint32_t OFF_AUX = OFF_M + 64 * 4;           // float [64] factors / 1/den
constexpr uint32_t OFF_BAR = OFF_AUX + 64 * 4;         // mbarriers
constexpr uint32_t OFF_MISC = OFF_BAR + 32 * 8;        // [0] TMEM base, [1] abort flag
constexpr uint32_t SMEM_USED = OFF_MISC + 64;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;      // slack for 1024-byte alignment
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

enum : uint32_t {
    B_QFULL = 0,
    B_QEMPTY,
    B_KVFULL0,
    B_KVFREE0 = B_KVFULL0 + 4,
    B_SFULL = B_KVFREE0 + 4,
    B_PFULL,
    B_PVDONE,
    B_OFREE,
    B_DONE,
    NUM_BARS
};
static_assert(NUM_BARS <= 32, "barrier area");

constexpr uint32_t TMEM_COLS = 512, TM_S = 0, TM_O = 256;
constexpr uint32_t IDESC_QK = idesc_bf16(128, 64, 0, 0);
constexpr uint32_t IDESC_PV = idesc_bf16(128, 64, 1, 1);

// ------------------------------------------------------------------ schedule

struct Seg {
    int64_t q;
    int j0, j1;
    bool full;
    int slot;
};

struct SegIter {
    int64_t lo, hi, cur, q;
};

__device__ __forceinline__ void seg_begin(const AttnParams &p, SegIter &it)
{
    if (p.split) {
        it.lo = (int64_t)blockIdx.x * p.per_cta;
        it.hi = min(it.lo + p.per_cta, p.BT * (int64_t)p.K);
        it.cur = it.lo;
    } else {
        it.q = blockIdx.x;
    }
}

__device__ __forceinline__ bool seg_next(const AttnParams &p, SegIter &it, Seg &s)
{
    if (!p.split) {
        if (it.q >= p.BT)
            return false;
        s.q = it.q;
        s.j0 = 0;
        s.j1 = p.K;
        s.full = true;
        s.slot = -1;
        it.q += gridDim.x;
        return true;
    }
    if (it.cur >= it.hi)
        return false;
    s.q = it.cur / p.K;
    const int64_t qs = s.q * p.K;
    const int64_t end = min(it.hi, qs + p.K);
    s.j0 = (int)(it.cur - qs);
    s.j1 = (int)(end - qs);
    s.full = (s.j0 == 0 && s.j1 == p.K);
    s.slot = (it.cur == it.lo) ? 2 * (int)blockIdx.x : 2 * (int)blockIdx.x + 1;
    it.cur = end;
    return true;
}

// Number of entries of idx[q, j0:j1] inside [0, N) (whole warp).
__device__ __forceinline__ int count_valid(const int32_t *il, int j0, int j1, int N, int lane)
{
    int n = 0;
    for (int j = j0; j < j1; j += 32) {
        const int jj = j + lane;
        const int v = jj < j1 ? __ldg(il + jj) : -1;
        n += __popc(__ballot_sync(0xffffffffu, v >= 0 && v < N));
    }
    return n;
}

// Warp-uniform bounded wait: lane 0 polls, the result is broadcast.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          uint64_t limit_ns, int lane)
{
    int ok = 0;
    if (lane == 0)
        ok = bounded_wait(bar, parity, abort_flag, limit_ns) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Drain wait that ignores the abort flag (the awaited operation is in flight
// and will complete); bounded by time only.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > limit_ns)
            break;
    }
}

// Reduce 64 per-thread values over the 32 lanes of a warp with 62 shuffles:
// each step halves the values a lane keeps.  On return v[0], v[1] hold the
// warp-wide result for heads head0 and head0 + 1.
template <bool MAX>
__device__ __forceinline__ void warp_reduce64(float (&v)[64], int lane, int &head0)
{
#define SA_RED_STEP(W, BIT)                                                      \
    {                                                                            \
        const bool up = (lane & (BIT)) != 0;                                     \
        _Pragma("unroll") for (int i = 0; i < (W); ++i)                          \
        {                                                                        \
            const float keep = up ? v[i + (W)] : v[i];                           \
            const float send = up ? v[i] : v[i + (W)];                           \
            const float got = __shfl_xor_sync(0xffffffffu, send, (BIT));         \
            v[i] = MAX ? fmaxf(keep, got) : keep + got;                          \
        }                                                                        \
    }
    SA_RED_STEP(32, 16)
    SA_RED_STEP(16, 8)
    SA_RED_STEP(8, 4)
    SA_RED_STEP(4, 2)
    SA_RED_STEP(2, 1)
#undef SA_RED_STEP
    head0 = ((lane & 16) ? 32 : 0) + ((lane & 8) ? 16 : 0) + ((lane & 4) ? 8 : 0) +
            ((lane & 2) ? 4 : 0) + ((lane & 1) ? 2 : 0);
}

// ------------------------------------------------------------------ roles

__device__ void producer_role(const AttnParams &p, uint8_t *smem, uint32_t sbase, int lane,
                              volatile int *abort_flag)
{
    int32_t *cidx = reinterpret_cast<int32_t *>(smem + OFF_IDX);
    const uint32_t bar0 = sbase + OFF_BAR;
    uint32_t ph_qempty = 0, ph_kvfree[4] = {0, 0, 0, 0};
    uint32_t q_loads = 0;
    bool ok = true;
    SegIter it;
    seg_begin(p, it);
    Seg s;
    while (ok && seg_next(p, it, s)) {
        const int32_t *il = p.idx + s.q * (int64_t)p.K;
        // compact the valid entries of this segment into shared memory
        int n = 0;
        bool bad = false;
        for (int j = s.j0; j < s.j1; j += 32) {
            const int jj = j + lane;
            const int v = jj < s.j1 ? __ldg(il + jj) : -1;
            const bool valid = v >= 0 && v < p.N;
            bad |= (jj < s.j1) && (v < -1 || v >= p.N);
            const uint32_t m = __ballot_sync(0xffffffffu, valid);
            if (valid)
                cidx[n + __popc(m & ((1u << lane) - 1u))] = v;
            n += __popc(m);
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0)
            atomicOr(p.err, ERRBIT_INDEX);
        __syncwarp();
        const int nc = (n + CH - 1) / CH;
        if (nc == 0)
            continue;

        // Q of this query: wait until the previous segment's QK products are done with it
        ok = warp_wait(bar0 + 8 * B_QEMPTY, ph_qempty ^ 1u, abort_flag, p.timeout_ns, lane);
        ph_qempty ^= 1u;
        if (!ok)
            break;
        if (lane == 0) {
            const uint32_t bq = bar0 + 8 * B_QFULL;
            mbar_arrive_expect_tx(bq, Q_BYTES);
            for (int kb = 0; kb < 8; ++kb)
                tma_load_2d(sbase + OFF_Q + kb * QBLK_BYTES, &p.tm_q, kb * 64, (int32_t)(s.q * H), bq);
        }
        ++q_loads;

        const uint16_t *kvb = p.kv + (size_t)(s.q / p.T) * (size_t)p.N * D;
        const int half = lane >> 4, within = lane & 15;
        for (int c = 0; c < nc && ok; ++c) {
            const int rows = min(CH, n - c * CH);
            const int32_t *crow = cidx + c * CH;
            for (int d = 0; d < 4; ++d) {
                ok = warp_wait(bar0 + 8 * (B_KVFREE0 + d), ph_kvfree[d] ^ 1u, abort_flag, p.timeout_ns,
                               lane);
                ph_kvfree[d] ^= 1u;
                if (!ok)
                    break;
                // slices 2d, 2d+1: 128 rows x 2 x 128 B = 2048 pieces of 16 B, 64 per lane
                const int sl = 2 * d + (within >> 3), pc = within & 7;
                const uint32_t dst0 = sbase + OFF_KV + sl * SLICE_BYTES;
                const uint16_t *src0 = kvb + sl * 64 + pc * 8;
#pragma unroll 8
                for (int i = 0; i < 64; ++i) {
                    const int r = 2 * i + half;
                    const bool v = r < rows;
                    const int row = v ? crow[r] : 0;
                    cp_async16(dst0 + r * 128 + ((pc ^ (r & 7)) << 4), src0 + (size_t)row * D,
                               v ? 16u : 0u);
                }
                cp_async_commit();
                if (d > 0) {
                    cp_async_wait<1>();
                    fence_proxy_async_smem();
                    mbar_arrive(bar0 + 8 * (B_KVFULL0 + d - 1));
                }
            }
            if (!ok)
                break;
            cp_async_wait<0>();
            fence_proxy_async_smem();
            mbar_arrive(bar0 + 8 * (B_KVFULL0 + 3));
        }
    }
    cp_async_wait_all();
    // a Q load still in flight must land before the CTA can exit
    if (q_loads > 0 && lane == 0)
        drain_wait(bar0 + 8 * B_QFULL, (q_loads - 1u) & 1u, p.timeout_ns);
    __syncwarp();
}

__device__ void mma_role(const AttnParams &p, uint32_t sbase, uint32_t tmem, int lane,
                         volatile int *abort_flag)
{
    const uint32_t bar0 = sbase + OFF_BAR;
    uint32_t ph_qfull = 0, ph_kvfull[4] = {0, 0, 0, 0}, ph_pfull = 0, ph_ofree = 0;
    bool ok = true;
    SegIter it;
    seg_begin(p, it);
    Seg s;
    while (ok && seg_next(p, it, s)) {
        const int n = count_valid(p.idx + s.q * (int64_t)p.K, s.j0, s.j1, p.N, lane);
        const int nc = (n + CH - 1) / CH;
        if (nc == 0)
            continue;
        ok = warp_wait(bar0 + 8 * B_QFULL, ph_qfull, abort_flag, p.timeout_ns, lane);
        ph_qfull ^= 1u;
        if (!ok)
            break;
        for (int c = 0; c < nc && ok; ++c) {
            // S^T = K_chunk . Q^T over 32 steps of 16 features
            for (int d = 0; d < 4; ++d) {
                ok = warp_wait(bar0 + 8 * (B_KVFULL0 + d), ph_kvfull[d], abort_flag, p.timeout_ns, lane);
                ph_kvfull[d] ^= 1u;
                if (!ok)
                    break;
                tc_fence_after();
                if (lane == 0) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int kk = 8 * d + k, sl = kk >> 2, sub = kk & 3;
                        const uint64_t a =
                            smem_desc_sw128(sbase + OFF_KV + sl * SLICE_BYTES + sub * 32, 16, 1024);
                        const uint64_t b =
                            smem_desc_sw128(sbase + OFF_Q + sl * QBLK_BYTES + sub * 32, 16, 1024);
                        mma_bf16_ss(tmem + TM_S, a, b, IDESC_QK, kk > 0 ? 1u : 0u);
                    }
                }
                __syncwarp();
            }
            if (!ok)
                break;
            if (lane == 0) {
                mma_commit(bar0 + 8 * B_SFULL);
                if (c == nc - 1)
                    mma_commit(bar0 + 8 * B_QEMPTY);
            }
            __syncwarp();
            ok = warp_wait(bar0 + 8 * B_PFULL, ph_pfull, abort_flag, p.timeout_ns, lane);
            ph_pfull ^= 1u;
            if (!ok)
                break;
            if (c == 0) {
                // the previous segment's epilogue must have read O^T out of TMEM
                ok = warp_wait(bar0 + 8 * B_OFREE, ph_ofree ^ 1u, abort_flag, p.timeout_ns, lane);
                ph_ofree ^= 1u;
                if (!ok)
                    break;
            }
            tc_fence_after();
            // O^T += V^T . P^T: four 128-feature tiles, 8 steps of 16 rows each
            if (lane == 0) {
#pragma unroll
                for (int d = 0; d < 4; ++d) {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t a = smem_desc_sw128(
                            sbase + OFF_KV + (2 * d) * SLICE_BYTES + kk * 2048, SLICE_BYTES, 1024);
                        const uint64_t b = smem_desc_sw128(sbase + OFF_P + kk * 2048, 8192, 1024);
                        mma_bf16_ss(tmem + TM_O + 64 * d, a, b, IDESC_PV,
                                    (c > 0 || kk > 0) ? 1u : 0u);
                    }
                    mma_commit(bar0 + 8 * (B_KVFREE0 + d));
                }
                mma_commit(bar0 + 8 * B_PVDONE);
            }
            __syncwarp();
        }
    }
    // every MMA issued must complete before TMEM is released
    if (lane == 0) {
        mma_commit(bar0 + 8 * B_DONE);
        drain_wait(bar0 + 8 * B_DONE, 0, p.timeout_ns);
    }
    __syncwarp();
}

__device__ void softmax_role(const AttnParams &p, uint8_t *smem, uint32_t sbase, uint32_t tmem,
                             int warp, int lane, volatile int *abort_flag)
{
    const int t = threadIdx.x;   // 0..127
    float *red = reinterpret_cast<float *>(smem + OFF_RED);
    float *m_s = reinterpret_cast<float *>(smem + OFF_M);
    float *aux = reinterpret_cast<float *>(smem + OFF_AUX);
    const uint32_t bar0 = sbase + OFF_BAR;
    const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);   // this warp's TMEM lane quarter
    uint32_t ph_sfull = 0, ph_pvdone = 0;
    SegIter it;
    seg_begin(p, it);
    Seg s;
    while (seg_next(p, it, s)) {
        const int n = count_valid(p.idx + s.q * (int64_t)p.K, s.j0, s.j1, p.N, lane);
        const int nc = (n + CH - 1) / CH;

        bar_sync(1, 128);   // the previous epilogue is done with m_s / aux
        if (t < 64)
            m_s[t] = __ldg(p.sink + t) * LOG2E;
        bar_sync(1, 128);

        float l[64];
#pragma unroll
        for (int h = 0; h < 64; ++h)
            l[h] = 0.f;

        bool aborted = false;
        for (int c = 0; c < nc; ++c) {
            const bool w1 = warp_wait(bar0 + 8 * B_SFULL, ph_sfull, abort_flag, p.timeout_ns, lane);
            ph_sfull ^= 1u;
            if (bar_red_or(1, 128, !w1 || *abort_flag)) {
                aborted = true;
                break;
            }
            tc_fence_after();
            uint32_t r[64];
            tmem_ld32(tl + TM_S, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
            tmem_ld32(tl + TM_S + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
            tmem_wait_ld();
            const bool vrow = c * CH + t < n;
            float x[64];
            bool need = false;
#pragma unroll
            for (int h = 0; h < 64; ++h) {
                x[h] = vrow ? __uint_as_float(r[h]) * p.scale_log2 : -INFINITY;
                need |= x[h] > m_s[h] + RESCALE_THRESHOLD;
            }
            // PV of the previous chunk must be complete before P is rewritten
            // or O^T rescaled.
            bool w2 = true;
            if (c > 0) {
                w2 = warp_wait(bar0 + 8 * B_PVDONE, ph_pvdone, abort_flag, p.timeout_ns, lane);
                ph_pvdone ^= 1u;
            }
            if (bar_red_or(1, 128, !w2 || *abort_flag)) {
                aborted = true;
                break;
            }
            if (bar_red_or(1, 128, need)) {
                // move the running maximum to this chunk's maximum (per head)
                int h0;
                warp_reduce64<true>(x, lane, h0);
                red[warp * 64 + h0] = x[0];
                red[warp * 64 + h0 + 1] = x[1];
                bar_sync(1, 128);
                if (t < 64) {
                    const float mx = fmaxf(fmaxf(red[t], red[64 + t]), fmaxf(red[128 + t], red[192 + t]));
                    const float mo = m_s[t];
                    const float mn = fmaxf(mo, mx);
                    aux[t] = ex2(mo - mn);
                    m_s[t] = mn;
                }
                bar_sync(1, 128);
#pragma unroll
                for (int h = 0; h < 64; ++h)
                    l[h] *= aux[h];
                if (c > 0) {
#pragma unroll 1
                    for (int d = 0; d < 4; ++d) {
#pragma unroll 1
                        for (int hh = 0; hh < 2; ++hh) {
                            uint32_t o[32];
                            const uint32_t ta = tl + TM_O + 64 * d + 32 * hh;
                            tmem_ld32(ta, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                o[i] = __float_as_uint(__uint_as_float(o[i]) * aux[32 * hh + i]);
                            tmem_st32(ta, o);
                        }
                    }
                    tmem_wait_st();
                }
                // x was consumed by the reduction: rebuild it from S^T
                tmem_ld32(tl + TM_S, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
                tmem_ld32(tl + TM_S + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
                tmem_wait_ld();
#pragma unroll
                for (int h = 0; h < 64; ++h)
                    x[h] = vrow ? __uint_as_float(r[h]) * p.scale_log2 : -INFINITY;
            }
            // probabilities in bf16 (the MMA operand) and their row sums
            uint32_t pk[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float p0 = ex2(x[2 * i] - m_s[2 * i]);
                const float p1 = ex2(x[2 * i + 1] - m_s[2 * i + 1]);
                pk[i] = pack_bf16x2(p0, p1);
                l[2 * i] += bf16lo_to_f32(pk[i]);
                l[2 * i + 1] += bf16hi_to_f32(pk[i]);
            }
            uint8_t *prow = smem + OFF_P + t * 128;
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8)
                *reinterpret_cast<uint4 *>(prow + ((c8 ^ (t & 7)) << 4)) =
                    make_uint4(pk[4 * c8], pk[4 * c8 + 1], pk[4 * c8 + 2], pk[4 * c8 + 3]);
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar0 + 8 * B_PFULL);
        }
        if (aborted)
            break;
        if (nc > 0) {
            const bool w = warp_wait(bar0 + 8 * B_PVDONE, ph_pvdone, abort_flag, p.timeout_ns, lane);
            ph_pvdone ^= 1u;
            if (bar_red_or(1, 128, !w || *abort_flag))
                break;
            tc_fence_after();
        }

        // row sums: reduce the per-row partials over the 128 threads
        {
            int h0;
            warp_reduce64<false>(l, lane, h0);
            red[warp * 64 + h0] = l[0];
            red[warp * 64 + h0 + 1] = l[1];
        }
        bar_sync(1, 128);
        if (t < 64) {
            const float lt = red[t] + red[64 + t] + red[128 + t] + red[192 + t];
            if (s.full) {
                const float den = lt + ex2(__ldg(p.sink + t) * LOG2E - m_s[t]);
                aux[t] = lt > 0.f ? 1.f / den : 0.f;
            } else {
                float *pm = p.part + (size_t)s.slot * PART_STRIDE + PART_O;
                pm[t] = m_s[t];
                pm[64 + t] = lt;
                aux[t] = 1.f;
            }
        }
        bar_sync(1, 128);

        // epilogue: thread t owns feature 128*d + t of every head
        const bool rope_here = s.full && p.rope_dim > 0;
#pragma unroll 1
        for (int d = 0; d < 4; ++d) {
            const int dim = 128 * d + t;
            float o[64];
            if (nc > 0) {
                uint32_t u[64];
                tmem_ld32(tl + TM_O + 64 * d, *reinterpret_cast<uint32_t(*)[32]>(&u[0]));
                tmem_ld32(tl + TM_O + 64 * d + 32, *reinterpret_cast<uint32_t(*)[32]>(&u[32]));
                tmem_wait_ld();
#pragma unroll
                for (int h = 0; h < 64; ++h)
                    o[h] = __uint_as_float(u[h]) * aux[h];
            } else {
#pragma unroll
                for (int h = 0; h < 64; ++h)
                    o[h] = 0.f;
            }
            if (rope_here && dim >= D - p.rope_dim) {   // warp-uniform
                const int i = (dim - (D - p.rope_dim)) >> 1;
                const float *cs = p.rope + ((size_t)(s.q % p.T) * (p.rope_dim >> 1) + i) * 2;
                const float cth = __ldg(cs), sth = __ldg(cs + 1);
                const bool odd = dim & 1;
#pragma unroll
                for (int h = 0; h < 64; ++h) {
                    const float other = __shfl_xor_sync(0xffffffffu, o[h], 1);
                    o[h] = odd ? (o[h] * cth - other * sth) : (o[h] * cth + other * sth);
                }
            }
            if (!s.full) {
                float *po = p.part + (size_t)s.slot * PART_STRIDE + dim;
#pragma unroll
                for (int h = 0; h < 64; ++h)
                    po[h * 512] = o[h];
            } else if (p.out_f32) {
                float *po = reinterpret_cast<float *>(p.out) + (size_t)s.q * (H * D) + dim;
#pragma unroll
                for (int h = 0; h < 64; ++h)
                    po[h * 512] = o[h];
            } else {
                __nv_bfloat16 *po = reinterpret_cast<__nv_bfloat16 *>(p.out) + (size_t)s.q * (H * D) + dim;
#pragma unroll
                for (int h = 0; h < 64; ++h)
                    po[h * 512] = __float2bfloat16_rn(o[h]);
            }
        }
        if (nc > 0) {
            tc_fence_before();
            mbar_arrive(bar0 + 8 * B_OFREE);
        }
    }
}

__global__ void __launch_bounds__(THREADS, 1) attn_kernel(const __grid_constant__ AttnParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_MISC + 4);
    const uint32_t bar0 = sbase + OFF_BAR;

    if (threadIdx.x == 0) {
        mbar_init(bar0 + 8 * B_QFULL, 1);
        mbar_init(bar0 + 8 * B_QEMPTY, 1);
        for (int d = 0; d < 4; ++d) {
            mbar_init(bar0 + 8 * (B_KVFULL0 + d), 32);
            mbar_init(bar0 + 8 * (B_KVFREE0 + d), 1);
        }
        mbar_init(bar0 + 8 * B_SFULL, 1);
        mbar_init(bar0 + 8 * B_PFULL, 128);
        mbar_init(bar0 + 8 * B_PVDONE, 1);
        mbar_init(bar0 + 8 * B_OFREE, 128);
        mbar_init(bar0 + 8 * B_DONE, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&p.tm_q);
    }
    if (warp == WARP_MMA) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == WARP_PRODUCER)
        producer_role(p, smem, sbase, lane, abort_flag);
    else if (warp == WARP_MMA)
        mma_role(p, sbase, tmem, lane, abort_flag);
    else
        softmax_role(p, smem, sbase, tmem, warp, lane, abort_flag);

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag)
        atomicOr(p.err, ERRBIT_TIMEOUT);
    if (warp == WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ split combine
//
// For a query whose index list was cut into pieces, merge the pieces' (m, l, O)
// (m in log2 units, O unnormalised):
//   M = max(sink*log2e, max_s m_s);  w_s = 2^(m_s - M)
//   o = sum_s w_s O_s / (sum_s w_s l_s + 2^(sink*log2e - M))
constexpr int MAX_PIECES = SA_MAX_K / 128 + 2;

__global__ void __launch_bounds__(256) combine_kernel(const __grid_constant__ AttnParams p)
{
    __shared__ float w_s[MAX_PIECES][64];
    __shared__ float inv_den[64];
    __shared__ int slots[MAX_PIECES];
    const int64_t q = blockIdx.x;
    const int64_t e0 = q * p.K, e1 = e0 + p.K;
    const int c0 = (int)(e0 / p.per_cta), c1 = (int)((e1 - 1) / p.per_cta);
    if (c0 == c1)
        return;   // one CTA held the whole list and wrote the output itself
    const int np = c1 - c0 + 1;
    const int t = threadIdx.x;
    if (t < np) {
        const int c = c0 + t;
        slots[t] = ((int64_t)c * p.per_cta >= e0) ? 2 * c : 2 * c + 1;
    }
    __syncthreads();
    if (t < 64) {
        const float sl = __ldg(p.sink + t) * LOG2E;
        float M = sl;
        for (int i = 0; i < np; ++i)
            M = fmaxf(M, p.part[(size_t)slots[i] * PART_STRIDE + PART_O + t]);
        float den = 0.f, lsum = 0.f;
        for (int i = 0; i < np; ++i) {
            const float *pm = p.part + (size_t)slots[i] * PART_STRIDE + PART_O;
            const float w = (M == -INFINITY) ? 0.f : ex2(pm[t] - M);
            w_s[i][t] = w;
            den += w * pm[64 + t];
            lsum += pm[64 + t];
        }
        den += (M == -INFINITY) ? 0.f : ex2(sl - M);
        inv_den[t] = (lsum > 0.f && den > 0.f) ? 1.f / den : 0.f;
    }
    __syncthreads();
    // 64 x 512 outputs, 4 consecutive features per thread per step
    for (int e = 4 * t; e < H * D; e += 4 * 256) {
        const int h = e >> 9, dim = e & 511;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int i = 0; i < np; ++i) {
            const float4 v = *reinterpret_cast<const float4 *>(p.part + (size_t)slots[i] * PART_STRIDE + e);
            const float w = w_s[i][h];
            acc.x += w * v.x;
            acc.y += w * v.y;
            acc.z += w * v.z;
            acc.w += w * v.w;
        }
        float o[4] = {acc.x * inv_den[h], acc.y * inv_den[h], acc.z * inv_den[h], acc.w * inv_den[h]};
        if (p.rope_dim > 0 && dim >= D - p.rope_dim) {
            const float *cs = p.rope + ((size_t)(q % p.T) * (p.rope_dim >> 1) + ((dim - (D - p.rope_dim)) >> 1)) * 2;
#pragma unroll
            for (int k = 0; k < 4; k += 2) {
                const float c = __ldg(cs + k), sn = __ldg(cs + k + 1);
                const float a = o[k], b = o[k + 1];
                o[k] = a * c + b * sn;
                o[k + 1] = -a * sn + b * c;
            }
        }
        if (p.out_f32) {
            *reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.out) + q * (H * D) + e) =
                make_float4(o[0], o[1], o[2], o[3]);
        } else {
            uint2 pk = make_uint2(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]));
            *reinterpret_cast<uint2 *>(reinterpret_cast<uint16_t *>(p.out) + q * (H * D) + e) = pk;
        }
    }
}

}  // namespace attn

// ------------------------------------------------------------------ host side

Schedule attn_schedule(int64_t BT, int K, int num_sms)
{
    Schedule s{};
    if (num_sms < 1)
        num_sms = 1;
    if (BT >= num_sms || K == 0) {
        s.split = 0;
        s.grid = (int)(BT < num_sms ? BT : num_sms);
        s.per_cta = 0;
        return s;
    }
    const int64_t total = BT * K;
    int64_t e = (total + num_sms - 1) / num_sms;
    if (e < 128)
        e = 128;
    e = (e + 31) / 32 * 32;
    s.split = 1;
    s.per_cta = e;
    s.grid = (int)((total + e - 1) / e);
    return s;
}

size_t attn_workspace_bytes(int64_t BT, int K, int num_sms)
{
    const Schedule s = attn_schedule(BT, K, num_sms);
    size_t bytes = WS_HEADER;
    if (s.split)
        bytes += (size_t)2 * s.grid * PART_STRIDE * sizeof(float);
    return (bytes + 255) / 256 * 256;
}

cudaError_t launch_attention(AttnParams &p, const Schedule &s, cudaStream_t st)
{
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(attn::attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)attn::SMEM_BYTES);
        if (e != cudaSuccess)
            return e;
        attr_done = true;
    }
    p.split = s.split;
    p.per_cta = s.per_cta;
    if (s.grid == 0)
        return cudaSuccess;
    attn::attn_kernel<<<s.grid, attn::THREADS, attn::SMEM_BYTES, st>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || !s.split)
        return e;
    attn::combine_kernel<<<(unsigned)p.BT, 256, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace sa
