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
//   * Warp roles (24 warps): warps 0-3 softmax + epilogue (thread i owns
//     TMEM lane i = chunk row i during the softmax, output feature
//     128*tile + i in the epilogue); warps 4-19 gather the rows with 16-byte
//     cp.async straight into the swizzled layout (an SM needs about sixteen
//     warps of outstanding copies to draw ~40 B/clk of scattered rows from
//     L2; a single TMA-issuing thread or warp reaches ~6 B/clk); warp 20
//     compacts each index list into a double-buffered shared list, loads Q
//     by TMA and, when kv is larger than L2, warms L2 with the next
//     segment's rows; warp 21 allocates TMEM and issues the MMAs (one
//     elected lane).  setmaxnreg gives the softmax warpgroup 240 registers
//     per thread and every other warp 48.
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
constexpr int NUM_GATHER_WARPS = 16;
constexpr int WARP_GATHER0 = 4;                 // warps 4 .. 19
constexpr int WARP_CONTROL = 20, WARP_MMA = 21; // warps 22, 23 only lend registers
constexpr int THREADS = 24 * 32;
constexpr int ROWS_PER_GATHER_WARP = CH / NUM_GATHER_WARPS;   // 8
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
constexpr uint32_t OFF_IDX = OFF_P + P_BYTES;          // int32 [2][SA_MAX_K] compacted lists
constexpr uint32_t OFF_RED = OFF_IDX + 2 * 4 * SA_MAX_K;   // float [4][64]
constexpr uint32_t OFF_M = OFF_RED + 4 * 64 * 4;       // float [64] running max (log2 units)
constexpr uint32_t OFF_AUX = OFF_M + 64 * 4;           // float [64] factors / 1/den
constexpr uint32_t OFF_SEGN = OFF_AUX + 64 * 4;        // int [2] list lengths
constexpr uint32_t OFF_BAR = OFF_SEGN + 16;            // mbarriers
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
    B_LFULL0,
    B_LEMPTY0 = B_LFULL0 + 2,
    B_DONE = B_LEMPTY0 + 2,
    NUM_BARS
};
constexpr uint32_t LEMPTY_ARRIVALS = NUM_GATHER_WARPS + 1 + 4;   // gather warps, MMA, softmax warps
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
    int64_t q;
    bool done;
};

__device__ __forceinline__ void seg_begin(const AttnParams &p, SegIter &it)
{
    (void)p;
    it.q = blockIdx.x;
    it.done = false;
}

// Whole mode: CTA i takes queries i, i + grid, ...  Split mode: CTA c takes
// piece c % pieces (entries [i*per_cta, min((i+1)*per_cta, K))) of query
// c / pieces and leaves its partial result in slot c.
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
    if (it.done)
        return false;
    it.done = true;
    const int piece = (int)(blockIdx.x % (unsigned)p.pieces);
    s.q = blockIdx.x / p.pieces;
    s.j0 = (int)(piece * p.per_cta);
    s.j1 = (int)min((int64_t)p.K, (piece + 1) * p.per_cta);
    s.full = false;
    s.slot = (int)blockIdx.x;
    return s.q < p.BT && s.j0 < s.j1;
}

// Keep the entries of idx[q, j0:j1] that are inside [0, N), in list order, in
// cidx; `bad` is set if an entry other than -1 falls outside [0, N).
__device__ __forceinline__ int compact_list(const int32_t *il, int j0, int j1, int N, int32_t *cidx,
                                            int lane, bool &bad)
{
    int n = 0;
    for (int j = j0; j < j1; j += 256) {
        int v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int jj = j + 32 * u + lane;
            v[u] = jj < j1 ? __ldg(il + jj) : -1;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const bool valid = v[u] >= 0 && v[u] < N;
            bad |= v[u] < -1 || v[u] >= N;
            const uint32_t m = __ballot_sync(0xffffffffu, valid);
            if (valid)
                cidx[n + __popc(m & ((1u << lane) - 1u))] = v[u];
            n += __popc(m);
        }
    }
    return n;
}

// Warm L2 with the latent rows a segment will gather (whole warp).
__device__ __forceinline__ void prefetch_segment_rows(const AttnParams &p, const Seg &s, int lane)
{
    const int32_t *il = p.idx + s.q * (int64_t)p.K;
    const uint16_t *kvb = p.kv + (size_t)(s.q / p.T) * (size_t)p.N * D;
    for (int j = s.j0; j < s.j1; j += 256) {
        int v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int jj = j + 32 * u + lane;
            v[u] = jj < s.j1 ? __ldg(il + jj) : -1;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (v[u] >= 0 && v[u] < p.N)
                prefetch_l2(kvb + (size_t)v[u] * D, D * 2);
    }
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

// Warp 20: compacts every segment's index list (double-buffered), publishes
// its length, and loads the segment's Q by TMA.
__device__ void control_role(const AttnParams &p, uint8_t *smem, uint32_t sbase, int lane,
                             volatile int *abort_flag)
{
    int *segn = reinterpret_cast<int *>(smem + OFF_SEGN);
    const uint32_t bar0 = sbase + OFF_BAR;
    uint32_t ph_qempty = 0, ph_lempty[2] = {0, 0};
    uint32_t q_loads = 0;
    bool ok = true;
    SegIter it;
    seg_begin(p, it);
    Seg s;
    bool have = seg_next(p, it, s);
    if (have && p.prefetch_rows)
        prefetch_segment_rows(p, s, lane);
    for (int k = 0; ok && have; ++k) {
        const int b = k & 1;
        // every consumer of this list buffer is done with the segment before
        ok = warp_wait(bar0 + 8 * (B_LEMPTY0 + b), ph_lempty[b] ^ 1u, abort_flag, p.timeout_ns, lane);
        ph_lempty[b] ^= 1u;
        if (!ok)
            break;
        int32_t *cidx = reinterpret_cast<int32_t *>(smem + OFF_IDX) + b * SA_MAX_K;
        bool bad = false;
        const int n = compact_list(p.idx + s.q * (int64_t)p.K, s.j0, s.j1, p.N, cidx, lane, bad);
        if (__any_sync(0xffffffffu, bad) && lane == 0)
            atomicOr(p.err, ERRBIT_INDEX);
        if (lane == 0)
            segn[b] = n;
        __syncwarp();
        // all 32 lanes arrive: each releases its entries.  The failure-detection
        // test withholds the first list so that every consumer's bounded wait
        // runs out.
        if (!(p.hold_lists && k == 0))
            mbar_arrive(bar0 + 8 * (B_LFULL0 + b));
        if (p.prefetch_rows) {
            SegIter la = it;
            Seg sn;
            if (seg_next(p, la, sn))
                prefetch_segment_rows(p, sn, lane);
        }
        if (n > 0) {
            // Q of this query, once the previous segment's QK products are done with it
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
        }
        have = seg_next(p, it, s);
    }
    // a Q load still in flight must land before the CTA can exit
    if (lane == 0 && q_loads > 0)
        drain_wait(bar0 + 8 * B_QFULL, (q_loads - 1u) & 1u, p.timeout_ns);
    __syncwarp();
}

// Warps 4-19: gather the compacted rows, chunk by chunk, tile by tile (two
// 64-feature slices of the 128 rows per tile).  Warp gi copies rows
// 8gi .. 8gi+7; rows past the end of the list are zero-filled.
__device__ void gather_role(const AttnParams &p, uint8_t *smem, uint32_t sbase, int gi, int lane,
                            volatile int *abort_flag)
{
    const int *segn = reinterpret_cast<const int *>(smem + OFF_SEGN);
    const uint32_t bar0 = sbase + OFF_BAR;
    uint32_t ph_lfull[2] = {0, 0}, ph_kvfree[4] = {0, 0, 0, 0};
    bool ok = true;
    SegIter it;
    seg_begin(p, it);
    Seg s;
    for (int k = 0; ok && seg_next(p, it, s); ++k) {
        const int b = k & 1;
        ok = warp_wait(bar0 + 8 * (B_LFULL0 + b), ph_lfull[b], abort_flag, p.timeout_ns, lane);
        ph_lfull[b] ^= 1u;
        if (!ok)
            break;
        const int n = segn[b];
        const int32_t *cidx = reinterpret_cast<const int32_t *>(smem + OFF_IDX) + b * SA_MAX_K;
        const int nc = (n + CH - 1) / CH;
        const uint16_t *kvb = p.kv + (size_t)(s.q / p.T) * (size_t)p.N * D;
        for (int c = 0; c < nc && ok; ++c) {
            const int rows = min(CH, n - c * CH);
            // this lane's four (row, 16-byte piece) jobs; the rows are the same for every tile
            int r[4], row[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                r[i] = ROWS_PER_GATHER_WARP * gi + ((i * 32 + lane) >> 4);
                row[i] = r[i] < rows ? cidx[c * CH + r[i]] : -1;
            }
            const int pc = lane & 15;   // piece: slice (2d + pc / 8), 16-byte chunk pc % 8
            for (int d = 0; d < 4; ++d) {
                ok = warp_wait(bar0 + 8 * (B_KVFREE0 + d), ph_kvfree[d] ^ 1u, abort_flag, p.timeout_ns,
                               lane);
                ph_kvfree[d] ^= 1u;
                if (!ok)
                    break;
                const int sl = 2 * d + (pc >> 3), ch = pc & 7;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t dst = sbase + OFF_KV + sl * SLICE_BYTES + r[i] * 128 + ((ch ^ (r[i] & 7)) << 4);
                    const uint16_t *src = kvb + (size_t)(row[i] < 0 ? 0 : row[i]) * D + sl * 64 + ch * 8;
                    cp_async16(dst, src, row[i] < 0 ? 0u : 16u);
                }
                cp_async_commit();
                if (d > 0) {
                    cp_async_wait<1>();
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(bar0 + 8 * (B_KVFULL0 + d - 1));
                }
            }
            if (!ok)
                break;
            cp_async_wait<0>();
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar0 + 8 * (B_KVFULL0 + 3));
        }
        if (!ok)
            break;
        __syncwarp();
        if (lane == 0)
            mbar_arrive(bar0 + 8 * (B_LEMPTY0 + b));
    }
    cp_async_wait_all();
    __syncwarp();
}

// Lane 0 of warp 21 runs this role alone: the tensor pipe reaches its rate
// only when MMAs are issued back to back, so the issuing thread avoids warp
// divergence and keeps its descriptor arithmetic to one add per MMA (the
// start-address field, address >> 4, is the low 14 bits of a descriptor).
__device__ void mma_role(const AttnParams &p, uint8_t *smem, uint32_t sbase, uint32_t tmem,
                         volatile int *abort_flag)
{
    const uint32_t bar0 = sbase + OFF_BAR;
    const int *segn = reinterpret_cast<const int *>(smem + OFF_SEGN);
    uint32_t ph_qfull = 0, ph_kvfull[4] = {0, 0, 0, 0}, ph_pfull = 0, ph_ofree = 0;
    uint32_t ph_lfull[2] = {0, 0};
    // S^T = K . Q^T: A = chunk (K-major), B = Q (K-major)
    const uint64_t d_qk_a = smem_desc_sw128(sbase + OFF_KV, 16, 1024);
    const uint64_t d_qk_b = smem_desc_sw128(sbase + OFF_Q, 16, 1024);
    // O^T += V^T . P^T: A = chunk (MN-major, 64-feature groups one slice apart), B = P^T (MN-major)
    const uint64_t d_pv_a = smem_desc_sw128(sbase + OFF_KV, SLICE_BYTES, 1024);
    const uint64_t d_pv_b = smem_desc_sw128(sbase + OFF_P, 8192, 1024);
    bool ok = true;
    SegIter it;
    seg_begin(p, it);
    Seg s;
    for (int k = 0; ok && seg_next(p, it, s); ++k) {
        const int b = k & 1;
        ok = bounded_wait(bar0 + 8 * (B_LFULL0 + b), ph_lfull[b], abort_flag, p.timeout_ns);
        ph_lfull[b] ^= 1u;
        if (!ok)
            break;
        const int n = segn[b];
        mbar_arrive(bar0 + 8 * (B_LEMPTY0 + b));
        const int nc = (n + CH - 1) / CH;
        if (nc == 0)
            continue;
        ok = bounded_wait(bar0 + 8 * B_QFULL, ph_qfull, abort_flag, p.timeout_ns);
        ph_qfull ^= 1u;
        if (!ok)
            break;
        for (int c = 0; c < nc && ok; ++c) {
            // S^T = K_chunk . Q^T over 32 steps of 16 features, tile by tile as they land
#pragma unroll
            for (int d = 0; d < 4; ++d) {
                ok = bounded_wait(bar0 + 8 * (B_KVFULL0 + d), ph_kvfull[d], abort_flag, p.timeout_ns);
                ph_kvfull[d] ^= 1u;
                if (!ok)
                    break;
                tc_fence_after();
#pragma unroll
                for (int k8 = 0; k8 < 8; ++k8) {
                    const int kk = 8 * d + k8;
                    const uint32_t oa = ((kk >> 2) * SLICE_BYTES + (kk & 3) * 32) >> 4;
                    const uint32_t ob = ((kk >> 2) * QBLK_BYTES + (kk & 3) * 32) >> 4;
                    mma_bf16_ss(tmem + TM_S, d_qk_a + oa, d_qk_b + ob, IDESC_QK, kk > 0 ? 1u : 0u);
                }
            }
            if (!ok)
                break;
            mma_commit(bar0 + 8 * B_SFULL);
            if (c == nc - 1)
                mma_commit(bar0 + 8 * B_QEMPTY);
            ok = bounded_wait(bar0 + 8 * B_PFULL, ph_pfull, abort_flag, p.timeout_ns);
            ph_pfull ^= 1u;
            if (!ok)
                break;
            if (c == 0) {
                // the previous segment's epilogue must have read O^T out of TMEM
                ok = bounded_wait(bar0 + 8 * B_OFREE, ph_ofree ^ 1u, abort_flag, p.timeout_ns);
                ph_ofree ^= 1u;
                if (!ok)
                    break;
            }
            tc_fence_after();
            // O^T += V^T . P^T: four 128-feature tiles, 8 steps of 16 rows each
            const uint32_t acc0 = c > 0 ? 1u : 0u;
#pragma unroll
            for (int d = 0; d < 4; ++d) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t oa = ((2 * d) * SLICE_BYTES + kk * 2048) >> 4;
                    const uint32_t ob = (kk * 2048) >> 4;
                    mma_bf16_ss(tmem + TM_O + 64 * d, d_pv_a + oa, d_pv_b + ob, IDESC_PV,
                                kk > 0 ? 1u : acc0);
                }
                mma_commit(bar0 + 8 * (B_KVFREE0 + d));
            }
            mma_commit(bar0 + 8 * B_PVDONE);
        }
    }
    // every MMA issued must complete before TMEM is released
    mma_commit(bar0 + 8 * B_DONE);
    drain_wait(bar0 + 8 * B_DONE, 0, p.timeout_ns);
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
    const int *segn = reinterpret_cast<const int *>(smem + OFF_SEGN);
    uint32_t ph_sfull = 0, ph_pvdone = 0, ph_lfull[2] = {0, 0};
    SegIter it;
    seg_begin(p, it);
    Seg s;
    for (int k = 0; seg_next(p, it, s); ++k) {
        const int b = k & 1;
        const bool w0 = warp_wait(bar0 + 8 * (B_LFULL0 + b), ph_lfull[b], abort_flag, p.timeout_ns, lane);
        ph_lfull[b] ^= 1u;
        // also: the previous epilogue is done with m_s / aux
        if (bar_red_or(1, 128, !w0 || *abort_flag))
            break;
        const int n = segn[b];
        __syncwarp();
        if (lane == 0)
            mbar_arrive(bar0 + 8 * (B_LEMPTY0 + b));
        const int nc = (n + CH - 1) / CH;

        if (t < 64)
            m_s[t] = __ldg(p.sink + t) * LOG2E;
        bar_sync(1, 128);

        float l[64];
#pragma unroll
        for (int h = 0; h < 64; ++h)
            l[h] = 0.f;

        bool aborted = false;
        for (int c = 0; c < nc; ++c) {
            // S^T of this chunk is ready; PV of the previous chunk (issued before
            // this chunk's QK) has then finished too, so P may be rewritten and
            // O^T rescaled
            bool wok = warp_wait(bar0 + 8 * B_SFULL, ph_sfull, abort_flag, p.timeout_ns, lane);
            ph_sfull ^= 1u;
            if (c > 0) {
                wok = warp_wait(bar0 + 8 * B_PVDONE, ph_pvdone, abort_flag, p.timeout_ns, lane) && wok;
                ph_pvdone ^= 1u;
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
            // one barrier in the common case: it carries the rescale vote and
            // any failed wait; a second one tells the two apart
            if (bar_red_or(1, 128, need || !wok || *abort_flag)) {
                if (bar_red_or(1, 128, !wok || *abort_flag)) {
                    aborted = true;
                    break;
                }
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

        // epilogue: thread t owns feature 128*d + t of every head; TMEM is read
        // in halves of 32 heads
        const bool rope_here = s.full && p.rope_dim > 0;
        uint16_t *stg = reinterpret_cast<uint16_t *>(smem + OFF_P);
#pragma unroll 1
        for (int e = 0; e < 8; ++e) {
            const int d = e >> 1, hh = e & 1;
            const int dim = 128 * d + t;
            uint32_t u[32];
            if (nc > 0) {
                tmem_ld32(tl + TM_O + 32 * e, u);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    u[i] = __float_as_uint(__uint_as_float(u[i]) * aux[32 * hh + i]);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    u[i] = 0u;
            }
            if (rope_here && dim >= D - p.rope_dim) {   // warp-uniform
                const int pi = (dim - (D - p.rope_dim)) >> 1;
                const float *cs = p.rope + ((size_t)(s.q % p.T) * (p.rope_dim >> 1) + pi) * 2;
                const float cth = __ldg(cs), sth = __ldg(cs + 1);
                const bool odd = dim & 1;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float o = __uint_as_float(u[i]);
                    const float other = __shfl_xor_sync(0xffffffffu, o, 1);
                    u[i] = __float_as_uint(odd ? (o * cth - other * sth) : (o * cth + other * sth));
                }
            }
            if (!s.full) {
                float *po = p.part + (size_t)s.slot * PART_STRIDE + (size_t)(32 * hh) * 512 + dim;
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    po[i * 512] = __uint_as_float(u[i]);
            } else if (p.out_f32) {
                float *po = reinterpret_cast<float *>(p.out) + (size_t)s.q * (H * D) + (size_t)(32 * hh) * 512 + dim;
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    po[i * 512] = __uint_as_float(u[i]);
            } else {
                // stage the tile as [64 heads][128 features] bf16 in the P buffer
                // (free once the last PV is done); after both halves, write whole
                // 256-byte head rows with 16-byte stores
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    stg[(32 * hh + i) * 128 + t] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(u[i])));
                if (hh == 1) {
                    bar_sync(1, 128);
                    uint8_t *gout = reinterpret_cast<uint8_t *>(p.out) + ((size_t)s.q * (H * D) + 128 * d) * 2;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int c = t + 128 * i;   // 16-byte piece c: head c / 16, part c % 16
                        const int h = c >> 4, part = c & 15;
                        const uint4 v = *reinterpret_cast<const uint4 *>(smem + OFF_P + h * 256 + part * 16);
                        *reinterpret_cast<uint4 *>(gout + (size_t)h * D * 2 + part * 16) = v;
                    }
                    bar_sync(1, 128);
                }
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
            mbar_init(bar0 + 8 * (B_KVFULL0 + d), NUM_GATHER_WARPS);
            mbar_init(bar0 + 8 * (B_KVFREE0 + d), 1);
        }
        mbar_init(bar0 + 8 * B_SFULL, 1);
        mbar_init(bar0 + 8 * B_PFULL, 128);
        mbar_init(bar0 + 8 * B_PVDONE, 1);
        mbar_init(bar0 + 8 * B_OFREE, 128);
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar0 + 8 * (B_LFULL0 + b), 32);
            mbar_init(bar0 + 8 * (B_LEMPTY0 + b), LEMPTY_ARRIVALS);
        }
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

    if (warp < 4) {
        // the softmax warpgroup keeps 64 scores and 64 row sums per thread
        asm volatile("setmaxnreg.inc.sync.aligned.u32 240;" ::: "memory");
        softmax_role(p, smem, sbase, tmem, warp, lane, abort_flag);
    } else {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 48;" ::: "memory");
        if (warp < WARP_GATHER0 + NUM_GATHER_WARPS)
            gather_role(p, smem, sbase, warp - WARP_GATHER0, lane, abort_flag);
        else if (warp == WARP_CONTROL)
            control_role(p, smem, sbase, lane, abort_flag);
        else if (warp == WARP_MMA && lane == 0)
            mma_role(p, smem, sbase, tmem, abort_flag);
    }

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
constexpr int MAX_PIECES = SA_MAX_K / 128;
constexpr int COMBINE_HEADS = 4;   // heads per block: grid (B*T, 64 / COMBINE_HEADS)

__global__ void __launch_bounds__(256) combine_kernel(const __grid_constant__ AttnParams p)
{
    __shared__ float w_s[MAX_PIECES][COMBINE_HEADS];
    __shared__ float inv_den[COMBINE_HEADS];
    __shared__ int slots[MAX_PIECES];
    const int64_t q = blockIdx.x;
    const int h0 = blockIdx.y * COMBINE_HEADS;
    const int np = p.pieces;   // the query's pieces sit in slots q*pieces .. q*pieces + pieces - 1
    const int t = threadIdx.x;
    if (t < np)
        slots[t] = (int)(q * p.pieces + t);
    __syncthreads();
    if (t < COMBINE_HEADS) {
        const int h = h0 + t;
        const float sl = __ldg(p.sink + h) * LOG2E;
        float M = sl;
        for (int i = 0; i < np; ++i)
            M = fmaxf(M, p.part[(size_t)slots[i] * PART_STRIDE + PART_O + h]);
        float den = 0.f, lsum = 0.f;
        for (int i = 0; i < np; ++i) {
            const float *pm = p.part + (size_t)slots[i] * PART_STRIDE + PART_O;
            const float w = (M == -INFINITY) ? 0.f : ex2(pm[h] - M);
            w_s[i][t] = w;
            den += w * pm[64 + h];
            lsum += pm[64 + h];
        }
        den += (M == -INFINITY) ? 0.f : ex2(sl - M);
        inv_den[t] = (lsum > 0.f && den > 0.f) ? 1.f / den : 0.f;
    }
    __syncthreads();
    // this block's 4 heads x 512 features: 8 consecutive features per thread
    const int hl = (8 * t) >> 9;
    const int dim = (8 * t) & 511;
    const int e = (h0 + hl) * D + dim;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (int i = 0; i < np; ++i) {
        const float4 *src = reinterpret_cast<const float4 *>(p.part + (size_t)slots[i] * PART_STRIDE + e);
        const float4 a = src[0], b = src[1];
        const float w = w_s[i][hl];
        acc[0] += w * a.x; acc[1] += w * a.y; acc[2] += w * a.z; acc[3] += w * a.w;
        acc[4] += w * b.x; acc[5] += w * b.y; acc[6] += w * b.z; acc[7] += w * b.w;
    }
    float o[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
        o[k] = acc[k] * inv_den[hl];
    if (p.rope_dim > 0 && dim >= D - p.rope_dim) {
        const float *cs = p.rope + ((size_t)(q % p.T) * (p.rope_dim >> 1) + ((dim - (D - p.rope_dim)) >> 1)) * 2;
#pragma unroll
        for (int k = 0; k < 8; k += 2) {
            const float c = __ldg(cs + k), sn = __ldg(cs + k + 1);
            const float a = o[k], b = o[k + 1];
            o[k] = a * c + b * sn;
            o[k + 1] = -a * sn + b * c;
        }
    }
    if (p.out_f32) {
        float4 *dst = reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.out) + q * (H * D) + e);
        dst[0] = make_float4(o[0], o[1], o[2], o[3]);
        dst[1] = make_float4(o[4], o[5], o[6], o[7]);
    } else {
        *reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(p.out) + q * (H * D) + e) =
            make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]), pack_bf16x2(o[4], o[5]),
                       pack_bf16x2(o[6], o[7]));
    }
}

}  // namespace attn

// ------------------------------------------------------------------ host side

Schedule attn_schedule(int64_t BT, int K, int num_sms)
{
    Schedule s{};
    if (num_sms < 1)
        num_sms = 1;
    // Fewer queries than SMs: cut each list into equal pieces (at least one
    // 128-row chunk each) so that about every SM holds one piece.
    int pieces = 1;
    if (BT > 0 && BT < num_sms && K > 0) {
        const int64_t by_sms = num_sms / BT;
        const int64_t by_len = (K + 127) / 128;
        pieces = (int)(by_sms < by_len ? by_sms : by_len);
        if (pieces < 1)
            pieces = 1;
    }
    if (pieces == 1) {
        s.split = 0;
        s.grid = (int)(BT < num_sms ? BT : num_sms);
        s.per_cta = 0;
        s.pieces = 1;
        return s;
    }
    s.split = 1;
    s.pieces = pieces;
    s.per_cta = ((K + pieces - 1) / pieces + 31) / 32 * 32;
    s.grid = (int)(BT * pieces);
    return s;
}

size_t attn_workspace_bytes(int64_t BT, int K, int num_sms)
{
    const Schedule s = attn_schedule(BT, K, num_sms);
    size_t bytes = WS_HEADER;
    if (s.split)
        bytes += (size_t)s.grid * PART_STRIDE * sizeof(float);
    return (bytes + 255) / 256 * 256;
}

cudaError_t launch_attention(AttnParams &p, const Schedule &s, cudaStream_t st)
{
    cudaError_t ea = cudaFuncSetAttribute(attn::attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)attn::SMEM_BYTES);
    if (ea != cudaSuccess)
        return ea;
    p.split = s.split;
    p.per_cta = s.per_cta;
    p.pieces = s.pieces;
    if (s.grid == 0)
        return cudaSuccess;
    attn::attn_kernel<<<s.grid, attn::THREADS, attn::SMEM_BYTES, st>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || !s.split)
        return e;
    attn::combine_kernel<<<dim3((unsigned)p.BT, attn::H / attn::COMBINE_HEADS), 256, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace sa
