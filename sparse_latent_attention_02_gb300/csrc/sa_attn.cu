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
//   * Warp roles (28 warps): warps 0-7 softmax + epilogue (two warps per
//     TMEM lane quarter, each with 32 of the 64 heads: a thread owns chunk
//     row 32*(w%4) + lane during the softmax and that output feature of
//     each 128-feature tile in the epilogue); warps 8-23 gather the rows
//     with 16-byte cp.async straight into the swizzled layout (an SM needs
//     about sixteen warps of outstanding copies to draw ~40 B/clk of
//     scattered rows from L2; a single TMA-issuing thread or warp reaches
//     ~6 B/clk); warp 24 loads Q by TMA, compacts each index list into a
//     double-buffered shared list and, when kv is larger than L2, warms L2
//     with the next segment's rows; warp 25 allocates TMEM and issues the
//     MMAs (one elected lane); warps 26-27 only complete the last
//     warpgroup.  setmaxnreg gives the softmax warps 112 registers per
//     thread, the gather warps 56 and the last warpgroup 56.
//   * Online softmax in base 2 with the sink as the starting maximum and a
//     lazy rescale: the running maximum moves only when a score exceeds it by
//     more than 2^8, so O^T in TMEM is almost never rewritten.  Row sums are
//     kept per thread (per row) and reduced once per segment.
//   * Every wait is bounded (bounded_wait); a timeout raises a CTA abort flag,
//     all roles leave their loops, in-flight copies and MMAs are drained, TMEM
//     is released and the error word gets ERRBIT_TIMEOUT.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sa_internal.h"
#include "sa_ptx.cuh"

namespace sa {
namespace attn {

constexpr int H = 64, D = 512, CH = 128;
constexpr int NUM_SOFTMAX_WARPS = 8;            // warps 0 .. 7: two per TMEM lane quarter
constexpr int SMX_THREADS = NUM_SOFTMAX_WARPS * 32;
constexpr int NUM_GATHER_WARPS = 16;
constexpr int WARP_GATHER0 = NUM_SOFTMAX_WARPS; // warps 8 .. 23
constexpr int WARP_CONTROL = WARP_GATHER0 + NUM_GATHER_WARPS, WARP_MMA = WARP_CONTROL + 1;
// setmaxnreg must be executed by every warp of a warpgroup: the block is whole
// warpgroups (warps 26, 27 have no role and only lend registers).
constexpr int THREADS = 28 * 32;                // 896
// Register split (setmaxnreg, per warpgroup): the launch gives every thread
// 72; the softmax warps take 112, the gather warps 56 and the last
// warpgroup (control, MMA) 56: 256*112 + 512*56 + 128*56 = 896*72.
constexpr int REGS_SOFTMAX = 112, REGS_GATHER = 56, REGS_LAST = 56, REGS_LAUNCH = 72;
constexpr int GATHER_THREADS = NUM_GATHER_WARPS * 32, LAST_THREADS = THREADS - SMX_THREADS - GATHER_THREADS;
static_assert(THREADS % 128 == 0 && NUM_SOFTMAX_WARPS % 4 == 0, "setmaxnreg acts on whole warpgroups");
static_assert(THREADS >= (WARP_MMA + 1) * 32, "every role has a warp");
static_assert(REGS_LAUNCH * THREADS <= 65536 && (65536 / THREADS) / 8 * 8 == REGS_LAUNCH,
              "launch register count");
static_assert(NUM_GATHER_WARPS % 4 == 0 && LAST_THREADS == 128, "one warpgroup after the gather warps");
static_assert(SMX_THREADS * REGS_SOFTMAX + GATHER_THREADS * REGS_GATHER + LAST_THREADS * REGS_LAST <=
                  THREADS * REGS_LAUNCH,
              "register split exceeds the launch allocation");
constexpr int MAX_CLUSTER = 8;                                // list pieces of one query
constexpr int GATHER_GROUP_WARPS = NUM_GATHER_WARPS / 2;          // each group owns two tiles
constexpr int ROWS_PER_GATHER_WARP = CH / GATHER_GROUP_WARPS;     // 16
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
constexpr uint32_t OFF_RAW = OFF_MISC + 64;           // int32 [SA_MAX_K] list as read from idx
constexpr uint32_t OFF_XSTAT = OFF_RAW + 4 * SA_MAX_K;   // float [pieces][2][64 / pieces] peers' (m, l)
constexpr uint32_t OFF_SINK = OFF_XSTAT + 2 * 64 * 4;    // float [64] sink * log2(e)
constexpr uint32_t SMEM_USED = OFF_SINK + 64 * 4;
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
    B_XRDY,      // split schedule: every peer's chunk buffer is free to receive
    B_XFULL,     // split schedule: every peer's partial for this CTA's heads has arrived
    NUM_BARS
};
constexpr uint32_t LEMPTY_ARRIVALS = NUM_GATHER_WARPS + 1 + NUM_SOFTMAX_WARPS;   // gather warps, MMA, softmax warps
static_assert(NUM_BARS <= 32, "barrier area");

constexpr uint32_t TMEM_COLS = 512, TM_S = 0, TM_O = 256;
constexpr uint32_t IDESC_QK = idesc_bf16(128, 64, 0, 0);
constexpr uint32_t IDESC_PV = idesc_bf16(128, 64, 1, 1);

// ------------------------------------------------------------------ schedule

struct Seg {
    int64_t q;
    int j0, j1;
    bool full;
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
// c / pieces; the pieces of a query are the CTAs of one cluster, rank = piece.
__device__ __forceinline__ bool seg_next(const AttnParams &p, SegIter &it, Seg &s)
{
    if (!p.split) {
        if (it.q >= p.BT)
            return false;
        s.q = it.q;
        s.j0 = 0;
        s.j1 = p.K;
        s.full = true;
        it.q += gridDim.x;
        return true;
    }
    if (it.done)
        return false;
    it.done = true;
    const int piece = (int)(blockIdx.x % (unsigned)p.pieces);
    s.q = blockIdx.x / p.pieces;
    // an empty piece still takes part in its cluster's merge (with no rows)
    s.j0 = (int)min((int64_t)p.K, piece * p.per_cta);
    s.j1 = (int)min((int64_t)p.K, (piece + 1) * p.per_cta);
    s.full = false;
    return s.q < p.BT;
}

// Latent row v (0 <= v < N) of batch element bidx.  One source: row v of kv.
// Two sources (the window ring and the compressed cache of the pages, read in
// place instead of concatenated): row v of source 0 when v < W, else row
// v - W of source 1.  The kernel is built for each case, so that the one-source
// gather keeps its single multiply-add per copy.
template <bool TWO>
__device__ __forceinline__ const uint16_t *kv_row(const AttnParams &p, int64_t bidx, int v)
{
    if (!TWO)
        return p.kv + ((size_t)bidx * (size_t)p.kv_bstride + (size_t)v) * D;
    return v < p.W ? p.kv + ((size_t)bidx * (size_t)p.kv_bstride + (size_t)v) * D
                   : p.kv2 + ((size_t)bidx * (size_t)p.kv2_bstride + (size_t)(v - p.W)) * D;
}

// Start copying idx[q, j0:j1] into the staging buffer (whole warp, one
// 4-byte cp.async per entry, all in flight at once: one memory round trip).
__device__ __forceinline__ void stage_list(const AttnParams &p, const Seg &s, uint32_t raw, int lane)
{
    const int32_t *il = p.idx + s.q * (int64_t)p.K;
    if (in_bounds(s.q < p.BT && s.j0 >= 0 && s.j1 <= p.K && s.j1 - s.j0 <= SA_MAX_K, p.err))
        for (int j = s.j0 + lane; j < s.j1; j += 32)
            cp_async4(raw + 4u * (uint32_t)(j - s.j0), il + j);
    cp_async_commit();
}

// Keep the staged entries that are inside [0, N), in list order, in cidx;
// `bad` is set if an entry other than -1 falls outside [0, N).
__device__ __forceinline__ int compact_staged(const int32_t *raw, int len, int N, int32_t *cidx, int lane,
                                              bool &bad)
{
    int n = 0;
    const uint32_t below = (1u << lane) - 1u;
    for (int j = 0; j < len; j += 128) {
        int v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int jj = j + 32 * u + lane;
            v[u] = jj < len ? raw[jj] : -1;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const bool valid = v[u] >= 0 && v[u] < N;
            bad |= v[u] < -1 || v[u] >= N;
            const uint32_t m = __ballot_sync(0xffffffffu, valid);
            if (valid)
                cidx[n + __popc(m & below)] = v[u];
            n += __popc(m);
        }
    }
    return n;
}

// Checked build: [ptr, ptr + bytes) lies inside the rows of the source that
// list index v reads (every batch element's rows of that source).
template <bool TWO>
__device__ __forceinline__ bool row_inside(const AttnParams &p, int v, const void *ptr, size_t bytes)
{
    const int64_t B = p.BT / p.T;
    if (TWO && v >= p.W)
        return inside(ptr, bytes, p.kv2, ((size_t)(B - 1) * (size_t)p.kv2_bstride + (size_t)(p.N - p.W)) * D * 2);
    return inside(ptr, bytes, p.kv, ((size_t)(B - 1) * (size_t)p.kv_bstride + (size_t)(TWO ? p.W : p.N)) * D * 2);
}

// Checked build: the same for the fp4 codes (D/2 bytes a row) and scales (D/16).
__device__ __forceinline__ bool fp4_inside(const AttnParams &p, const uint8_t *ptr, size_t bytes, bool scales)
{
    const int64_t B = p.BT / p.T;
    const size_t rows = (size_t)(B - 1) * (size_t)p.kv2_bstride + (size_t)(p.N - p.W);
    return scales ? inside(ptr, bytes, p.kv2_scales, rows * (D / 16)) : inside(ptr, bytes, p.kv2_codes, rows * (D / 2));
}

// Warm L2 with latent rows (whole warp, one line prefetch per 128 bytes):
// rows list[j0 .. j1) of batch element bidx, skipping entries outside [0, N).
template <bool TWO, bool FP4>
__device__ __forceinline__ void prefetch_rows(const AttnParams &p, int64_t bidx, const int32_t *list, int j0,
                                              int j1, int lane)
{
    // lane = 8 * (row within a group of 4) + line
    const int line = lane & 7;
    for (int j = j0 + (lane >> 3); j < j1; j += 4) {
        const int v = list[j];
        if (v < 0 || v >= p.N)
            continue;
        if (FP4 && v >= p.W) {   // fp4 row: 256 code bytes and 32 scale bytes
            const size_t cr = (size_t)bidx * (size_t)p.kv2_bstride + (size_t)(v - p.W);
            if (line < 2)
                prefetch_l2_line(p.kv2_codes + cr * (D / 2) + line * 128);
            else if (line == 2)
                prefetch_l2_line(p.kv2_scales + cr * (D / 16));
        } else {
            prefetch_l2_line(reinterpret_cast<const uint8_t *>(kv_row<TWO>(p, bidx, v)) + line * 128);
        }
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

// Reduce 32 per-thread values over the 32 lanes of a warp with 31 shuffles:
// each step halves the values a lane keeps.  Returns the warp-wide result for
// value index `lane`.
template <bool MAX>
__device__ __forceinline__ float warp_reduce32(float (&v)[32], int lane)
{
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) {
        const bool up = (lane & w) != 0;
#pragma unroll
        for (int i = 0; i < w; ++i) {
            const float keep = up ? v[i + w] : v[i];
            const float send = up ? v[i] : v[i + w];
            const float got = __shfl_xor_sync(0xffffffffu, send, w);
            v[i] = MAX ? fmaxf(keep, got) : keep + got;
        }
    }
    return v[0];
}

// ------------------------------------------------------------------ roles

// Wait until the previous segment's QK products are done with Q, then load
// this segment's Q (64 heads x 512 features) by TMA (whole warp, lane 0 issues).
__device__ __forceinline__ bool load_q(const AttnParams &p, uint32_t sbase, const Seg &s, uint32_t &ph_qempty,
                                       uint32_t &q_loads, volatile int *abort_flag, int lane)
{
    const uint32_t bar0 = sbase + OFF_BAR;
    const bool ok = warp_wait(bar0 + 8 * B_QEMPTY, ph_qempty ^ 1u, abort_flag, p.timeout_ns, lane);
    ph_qempty ^= 1u;
    if (!ok)
        return false;
    if (lane == 0) {
        const uint32_t bq = bar0 + 8 * B_QFULL;
        if (in_bounds(s.q < p.BT, p.err)) {
            mbar_arrive_expect_tx(bq, Q_BYTES);
            for (int kb = 0; kb < 8; ++kb)
                tma_load_2d(sbase + OFF_Q + kb * QBLK_BYTES, &p.tm_q, kb * 64, (int32_t)(s.q * H), bq);
        } else {
            mbar_arrive(bq);
        }
    }
    ++q_loads;
    return true;
}

// Warp 24: loads every segment's Q by TMA and its index list into the
// staging buffer, compacts the list into a double-buffered shared list and
// publishes its length.  When kv is larger than L2 it then warms L2 with the
// next segment's rows while the current segment is processed.
template <bool TWO, bool FP4>
__device__ void control_role(const AttnParams &p, uint8_t *smem, uint32_t sbase, int lane,
                             volatile int *abort_flag)
{
    int *segn = reinterpret_cast<int *>(smem + OFF_SEGN);
    const int32_t *raw = reinterpret_cast<const int32_t *>(smem + OFF_RAW);
    const uint32_t raw_u32 = sbase + OFF_RAW;
    const uint32_t bar0 = sbase + OFF_BAR;
    uint32_t ph_qempty = 0, ph_lempty[2] = {0, 0};
    uint32_t q_loads = 0;
    bool ok = true;
    SegIter it;
    seg_begin(p, it);
    Seg s, sn;
    bool have = seg_next(p, it, s);
    if (have) {
        // the kernel's prologue already started copying the first list;
        // the first segment's Q is requested before that list is read
        ok = load_q(p, sbase, s, ph_qempty, q_loads, abort_flag, lane);
    }
    for (int k = 0; ok && have; ++k) {
        const int b = k & 1;
        // every consumer of this list buffer is done with the segment before
        ok = warp_wait(bar0 + 8 * (B_LEMPTY0 + b), ph_lempty[b] ^ 1u, abort_flag, p.timeout_ns, lane);
        ph_lempty[b] ^= 1u;
        if (!ok)
            break;
        cp_async_wait_all();
        if (k == 0) {   // the sinks arrived with the first list: to log2 units
            float *sink_s = reinterpret_cast<float *>(smem + OFF_SINK);
            sink_s[lane] *= LOG2E;
            sink_s[lane + 32] *= LOG2E;
        }
        __syncwarp();
        int32_t *cidx = reinterpret_cast<int32_t *>(smem + OFF_IDX) + b * SA_MAX_K;
        bool bad = false;
        const int n = compact_staged(raw, s.j1 - s.j0, p.N, cidx, lane, bad);
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
        // Q of a later segment, once the previous segment's QK products are done with it
        if (k > 0) {
            ok = load_q(p, sbase, s, ph_qempty, q_loads, abort_flag, lane);
            if (!ok)
                break;
        }
        have = seg_next(p, it, sn);
        if (have) {
            stage_list(p, sn, raw_u32, lane);
            if (p.prefetch_rows) {
                cp_async_wait_all();
                __syncwarp();
                prefetch_rows<TWO, FP4>(p, sn.q / p.T, raw, 0, sn.j1 - sn.j0, lane);
            }
            s = sn;
        }
    }
    cp_async_wait_all();
    // a Q load still in flight must land before the CTA can exit
    if (lane == 0 && q_loads > 0)
        drain_wait(bar0 + 8 * B_QFULL, (q_loads - 1u) & 1u, p.timeout_ns);
    __syncwarp();
}

// Two E4M3 ("fn") scale bytes (low byte first) as two bf16 pairs, each
// holding its scale times 2^112 twice.  The hardware conversion to f16 is
// exact (E4M3 values are f16 normals), and so are the products and the bf16
// roundings (at most four significant bits, exponents within range); NaN
// stays NaN.
__device__ __forceinline__ void scales_x2112(uint32_t two_bytes, uint32_t &s0, uint32_t &s1)
{
    uint32_t h;
    asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h) : "r"(two_bytes));
    const float f0 = __half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu))) * 0x1p112f;
    const float f1 = __half2float(__ushort_as_half((unsigned short)(h >> 16))) * 0x1p112f;
    s0 = pack_bf16x2(f0, f0);
    s1 = pack_bf16x2(f1, f1);
}

// Eight e2m1 codes (byte i: feature 2i in the low nibble, 2i+1 in the high
// one) times their group's scale, as four packed bf16 pairs.  The hardware
// converts each code pair to f16 exactly; a code is zero or an f16 normal
// whose mantissa has only its top bit, so moving the exponent and mantissa
// right by three bits gives the bf16 bit pattern of the code times 2^-112,
// and one bf16 product with `scale2` (scale times 2^112, both halves) gives
// code times scale, exactly (at most five significant bits).
__device__ __forceinline__ uint4 dequant_e2m1x8(uint32_t codes, uint32_t scale2)
{
    uint32_t h[4];
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(codes));
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t b = ((h[i] >> 3) & 0x0FFF0FFFu) | (h[i] & 0x80008000u);
        asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(w[i]) : "r"(b), "r"(scale2));
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Warps 8-23: gather the compacted rows, chunk by chunk, in two groups of
// eight warps: group g fills tiles g and g + 2 (a tile is two 64-feature
// slices of the 128 rows), so all four tiles of a chunk can be in flight at
// once and each tile is refilled as soon as the PV product frees it.  Warp w
// of a group copies rows 16w .. 16w+15; rows past the end of the list are
// zero-filled.
template <bool TWO, bool FP4>
__device__ void gather_role(const AttnParams &p, uint8_t *smem, uint32_t sbase, int gi, int lane,
                            volatile int *abort_flag)
{
    const int *segn = reinterpret_cast<const int *>(smem + OFF_SEGN);
    const uint32_t bar0 = sbase + OFF_BAR;
    const int grp = gi / GATHER_GROUP_WARPS, wg = gi % GATHER_GROUP_WARPS;
    uint32_t ph_lfull[2] = {0, 0}, ph_kvfree[2] = {0, 0};
    bool ok = true;
    SegIter it;
    seg_begin(p, it);
    Seg s;
    const int pc = lane & 15;   // piece: slice (2d + pc / 8), 16-byte chunk pc % 8
    for (int k = 0; ok && seg_next(p, it, s); ++k) {
        const int b = k & 1;
        ok = warp_wait(bar0 + 8 * (B_LFULL0 + b), ph_lfull[b], abort_flag, p.timeout_ns, lane);
        ph_lfull[b] ^= 1u;
        if (!ok)
            break;
        const int n = segn[b];
        const int32_t *cidx = reinterpret_cast<const int32_t *>(smem + OFF_IDX) + b * SA_MAX_K;
        const int nc = (n + CH - 1) / CH;
        const int64_t bidx = s.q / p.T;
        // this batch element's rows in each source (the second only with two sources)
        const uint16_t *kvb = p.kv + (size_t)bidx * (size_t)p.kv_bstride * D;
        const uint16_t *kvb2 = TWO ? p.kv2 + ((size_t)bidx * (size_t)p.kv2_bstride - (size_t)p.W) * D : nullptr;
        auto row_ptr = [&](int v) -> const uint16_t * {
            return (TWO && v >= p.W) ? kvb2 + (size_t)v * D : kvb + (size_t)v * D;
        };
        for (int c = 0; c < nc && ok; ++c) {
            const int rows = min(CH, n - c * CH);
            // bf16 rows: this lane's eight (row, 16-byte piece) jobs, rows r0 + 2i;
            // the rows are the same for both tiles
            const int r0 = ROWS_PER_GATHER_WARP * wg + (lane >> 4);
            int row[8];
            // fp4 rows: this lane's two rows rf + 8j, 32 features (quarter qq of
            // the tile: 16 code bytes, 2 scales) of each; the loads of both tiles
            // are issued before the tiles are free
            const int qq = lane & 3, rf = ROWS_PER_GATHER_WARP * wg + (lane >> 2);
            int rv[2];
            uint4 code[2][2];
            uint32_t scl[2][2];
            if constexpr (!FP4) {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    row[i] = r0 + 2 * i < rows ? cidx[c * CH + r0 + 2 * i] : -1;
            } else {
#pragma unroll
                for (int j = 0; j < 2; ++j)
                    rv[j] = rf + 8 * j < rows ? cidx[c * CH + rf + 8 * j] : -1;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        code[e][j] = make_uint4(0u, 0u, 0u, 0u);
                        scl[e][j] = 0u;
                        if (rv[j] >= p.W) {
                            const size_t cr = (size_t)bidx * (size_t)p.kv2_bstride + (size_t)(rv[j] - p.W);
                            const int d = grp + 2 * e;
                            const uint8_t *cp = p.kv2_codes + cr * (D / 2) + 64 * d + 16 * qq;
                            const uint8_t *sp = p.kv2_scales + cr * (D / 16) + 8 * d + 2 * qq;
                            if (in_bounds(fp4_inside(p, cp, 16, false) && fp4_inside(p, sp, 2, true), p.err)) {
                                code[e][j] = __ldg(reinterpret_cast<const uint4 *>(cp));
                                scl[e][j] = (uint32_t)__ldg(sp) | ((uint32_t)__ldg(sp + 1) << 8);
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int d = grp + 2 * e;
                ok = warp_wait(bar0 + 8 * (B_KVFREE0 + d), ph_kvfree[e] ^ 1u, abort_flag, p.timeout_ns, lane);
                ph_kvfree[e] ^= 1u;
                if (!ok)
                    break;
                if constexpr (!FP4) {
                    const int sl = 2 * d + (pc >> 3), ch = pc & 7;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int r = r0 + 2 * i;
                        const uint32_t dst = sbase + OFF_KV + sl * SLICE_BYTES + r * 128 + ((ch ^ (r & 7)) << 4);
                        const uint16_t *src = row_ptr(row[i] < 0 ? 0 : row[i]) + sl * 64 + ch * 8;
                        // (a row that fails its source check is zero-filled from a
                        // valid address, like an empty slot)
                        const bool live = row[i] >= 0 && in_bounds(row_inside<TWO>(p, row[i], src, 16), p.err);
                        if (in_bounds(r < CH && sl < 8, p.err))
                            cp_async16(dst, live || row[i] < 0 ? src : row_ptr(0), live ? 16u : 0u);
                    }
                } else {
                    // quarter qq: slice 2d + qq / 2, 16-byte chunks 4 (qq % 2) .. +3
                    const int sl = 2 * d + (qq >> 1), ch0 = 4 * (qq & 1);
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int r = rf + 8 * j, v = rv[j];
                        const uint32_t roff = OFF_KV + sl * SLICE_BYTES + r * 128;
                        if (!in_bounds(r < CH && sl < 8, p.err))
                            continue;
                        if (v >= p.W) {
                            uint32_t s0, s1;
                            scales_x2112(scl[e][j], s0, s1);
                            const uint32_t cw[4] = {code[e][j].x, code[e][j].y, code[e][j].z, code[e][j].w};
#pragma unroll
                            for (int m = 0; m < 4; ++m)
                                *reinterpret_cast<uint4 *>(smem + roff + (((ch0 + m) ^ (r & 7)) << 4)) =
                                    dequant_e2m1x8(cw[m], m < 2 ? s0 : s1);
                        } else {
                            // window row, or an empty slot (copies nothing; its
                            // source is any valid address)
                            const uint16_t *src =
                                v >= 0 ? kvb + (size_t)v * D + 128 * d + 32 * qq
                                       : (p.W > 0 ? kvb : reinterpret_cast<const uint16_t *>(p.kv2_codes));
                            const bool live = v >= 0 && in_bounds(row_inside<true>(p, v, src, 64), p.err);
                            const uint16_t *dead = v >= 0 ? kvb : src;   // a valid address for no bytes
#pragma unroll
                            for (int m = 0; m < 4; ++m)
                                cp_async16(sbase + roff + (((ch0 + m) ^ (r & 7)) << 4), live ? src + 8 * m : dead,
                                           live ? 16u : 0u);
                        }
                    }
                }
                cp_async_commit();
            }
            if (!ok)
                break;
            cp_async_wait<1>();
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar0 + 8 * (B_KVFULL0 + grp));
            cp_async_wait<0>();
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar0 + 8 * (B_KVFULL0 + grp + 2));
            // kv larger than L2: this chunk has landed; start bringing this warp's
            // part of the next chunk (its rows, its two tiles' 128-byte lines) into
            // L2 while the chunk is used, so that the refill after the PV product
            // does not wait for HBM
            if (p.prefetch_rows && c + 1 < nc) {
                const int j = (c + 1) * CH + ROWS_PER_GATHER_WARP * wg + (lane >> 1);
                if (j < n && FP4 && cidx[j] >= p.W) {
                    // fp4 row: group g warms code line g; group 0 also the scales
                    const size_t cr = (size_t)bidx * (size_t)p.kv2_bstride + (size_t)(cidx[j] - p.W);
                    if ((lane & 1) == 0)
                        prefetch_l2_line(p.kv2_codes + cr * (D / 2) + 128 * grp);
                    else if (grp == 0)
                        prefetch_l2_line(p.kv2_scales + cr * (D / 16));
                } else if (j < n) {
                    const uint8_t *rp = reinterpret_cast<const uint8_t *>(row_ptr(cidx[j])) +
                                        (grp + 2 * (lane & 1)) * 256;
                    prefetch_l2_line(rp);
                    prefetch_l2_line(rp + 128);
                }
            }
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

// Lane 0 of warp 25 runs this role alone: the tensor pipe reaches its rate
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
        // Q is loaded for every segment
        ok = bounded_wait(bar0 + 8 * B_QFULL, ph_qfull, abort_flag, p.timeout_ns);
        ph_qfull ^= 1u;
        if (!ok)
            break;
        if (nc == 0) {
            mbar_arrive(bar0 + 8 * B_QEMPTY);
            continue;
        }
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

// Warp-uniform bounded wait for arrivals from other CTAs of the cluster.
__device__ __forceinline__ bool warp_wait_cluster(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                                  uint64_t limit_ns, int lane)
{
    int ok = 0;
    if (lane == 0)
        ok = bounded_wait_cluster(bar, parity, abort_flag, limit_ns) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Split schedule: the P pieces of one query's list run as one cluster, and
// CTA r of the cluster finishes heads [r*HP, (r+1)*HP), HP = 64 / P.  A CTA
// offers its chunk buffer (arrives on each peer's XRDY barrier) once its own
// last PV product is done.  Once all its peers have offered theirs, every CTA
// writes each peer its unnormalised O^T columns for that peer's heads, read
// from TMEM and rounded to bf16 pairs of adjacent heads, straight into the
// peer's chunk buffer (slot `me` of P slots, one 4-byte pair per feature and
// head pair), together with its (m, l) for those heads, by asynchronous
// stores (st.async) whose bytes complete on the peer's XFULL barrier; each
// CTA armed its own XFULL barrier with the bytes it expects.  The receiver
// merges the pieces:
//   M = max_r m_r (each m_r starts at the sink),  w_r = 2^(m_r - M),
//   o = sum_r w_r O_r / (sum_r w_r l_r + 2^(sink*log2e - M))
// then applies the inverse RoPE when asked and writes its heads.  bf16 keeps
// the partials' full range whatever the magnitude of kv (distributed shared
// memory moves only ~13 bytes per clock per SM, so the partials go at half
// the width of fp32); the CTA's own partial stays fp32.
// Softmax warps only: warp (quarter qd, half hf) handles features
// 128d + 32qd + lane of tiles d = 2hf, 2hf + 1.  False when a wait ran out.

// Write NV heads' values of one feature (this lane's `f`, one value per head
// in v) as bf16 into out[head][f] rows of D features, without staging: the two
// lanes of an adjacent-feature pair swap half of their values, so that the
// even lane writes features (f, f + 1) of the first NV/2 heads and the odd
// lane those of the last NV/2, as 4-byte words (a warp's store covers two
// contiguous 64-byte runs).
template <int NV>
__device__ __forceinline__ void store_bf16_pairs(uint16_t *out_h0, int f, const float (&v)[NV], int lane)
{
    const bool odd = lane & 1;
    const int f0 = f & ~1;
#pragma unroll
    for (int i = 0; i < NV / 2; ++i) {
        const float send = odd ? v[i] : v[NV / 2 + i];
        const float got = __shfl_xor_sync(0xffffffffu, send, 1);
        const int h = odd ? NV / 2 + i : i;
        const uint32_t w = odd ? pack_bf16x2(got, v[NV / 2 + i]) : pack_bf16x2(v[i], got);
        *reinterpret_cast<uint32_t *>(out_h0 + (size_t)h * D + f0) = w;
    }
}

template <int P>
__device__ bool cluster_merge(const AttnParams &p, uint8_t *smem, uint32_t sbase, uint32_t tl, const Seg &s,
                              int nc, int t, int qd, int hf, volatile int *abort_flag, int lane)
{
    constexpr int HP = H / P;
    // one piece's O for HP heads: bf16 [HP / 2][512] pairs of heads (2j, 2j + 1) per feature
    constexpr uint32_t SLOT_BYTES = HP * D * 2;
    static_assert(P * SLOT_BYTES <= KV_BYTES, "receive slots fit the chunk buffer");
    const uint32_t me = cluster_ctarank();
    const uint32_t bar0 = sbase + OFF_BAR;
    const float *m_s = reinterpret_cast<const float *>(smem + OFF_M);
    const float *lt = reinterpret_cast<const float *>(smem + OFF_AUX);   // this piece's row sums
    const float *xst = reinterpret_cast<const float *>(smem + OFF_XSTAT);   // [P][2][HP] peers' (m, l)
    float *wts = reinterpret_cast<float *>(smem + OFF_RED);   // [P][HP] weights w_r / den
    const uint32_t *recv = reinterpret_cast<const uint32_t *>(smem + OFF_KV);   // [P][HP / 2][512] bf16 pairs
    const int fl = 32 * qd + lane;   // feature within a 128-feature tile

    // every peer's partial and (m, l) land on this CTA's XFULL barrier as bytes
    if (t == 0)
        mbar_arrive_expect_tx(bar0 + 8 * B_XFULL, (uint32_t)(P - 1) * (SLOT_BYTES + 2 * HP * 4));
    // (this CTA offered its buffer on each peer's XRDY barrier as soon as its
    // last PV product was done)
    bool ok = warp_wait_cluster(bar0 + 8 * B_XRDY, 0, abort_flag, p.timeout_ns, lane);
    if (bar_red_or(1, SMX_THREADS, !ok || *abort_flag))
        return false;

    // send: peer g gets columns g*HP .. g*HP + HP-1 of every 128-feature tile
#pragma unroll 1
    for (int gi = 1; gi < P; ++gi) {
        const uint32_t g = (me + (uint32_t)gi) % (uint32_t)P;   // peers in a rotated order
        const uint32_t dst = mapa_shared(sbase + OFF_KV + me * SLOT_BYTES, g);
        const uint32_t rbar = mapa_shared(bar0 + 8 * B_XFULL, g);
        if (t < HP) {
            const uint32_t xs = mapa_shared(sbase + OFF_XSTAT + (me * 2 * HP + t) * 4, g);
            st_async_b32(xs, __float_as_uint(m_s[g * HP + t]), rbar);
            st_async_b32(xs + 4 * HP, __float_as_uint(lt[g * HP + t]), rbar);
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int d = 2 * hf + e;
            uint32_t v[HP];
            if (nc > 0) {
#pragma unroll
                for (int j = 0; j < HP / 8; ++j)
                    tmem_ld8(tl + TM_O + 64 * d + g * HP + 8 * j, *reinterpret_cast<uint32_t(*)[8]>(&v[8 * j]));
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int i = 0; i < HP; ++i)
                    v[i] = 0u;
            }
#pragma unroll
            for (int i = 0; i < HP; i += 2)
                st_async_b32(dst + (uint32_t)(((i / 2) * D + 128 * d + fl) * 4),
                             pack_bf16x2(__uint_as_float(v[i]), __uint_as_float(v[i + 1])), rbar);
        }
    }

    ok = warp_wait_cluster(bar0 + 8 * B_XFULL, 0, abort_flag, p.timeout_ns, lane);
    if (bar_red_or(1, SMX_THREADS, !ok || *abort_flag))
        return false;

    if (t < HP) {
        const int h = (int)me * HP + t;
        const float sl = reinterpret_cast<const float *>(smem + OFF_SINK)[h];
        float M = m_s[h];
#pragma unroll
        for (int r = 0; r < P; ++r)
            if (r != (int)me)
                M = fmaxf(M, xst[r * 2 * HP + t]);
        float w[P];
        float den = 0.f;
#pragma unroll
        for (int r = 0; r < P; ++r) {
            const float mr = r == (int)me ? m_s[h] : xst[r * 2 * HP + t];
            const float lr = r == (int)me ? lt[h] : xst[r * 2 * HP + HP + t];
            w[r] = M == -INFINITY ? 0.f : ex2(mr - M);
            den += w[r] * lr;
        }
        den += M == -INFINITY ? 0.f : ex2(sl - M);
        const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
        for (int r = 0; r < P; ++r)
            wts[r * HP + t] = w[r] * inv;
    }
    bar_sync(1, SMX_THREADS);

#pragma unroll 1
    for (int e = 0; e < 2; ++e) {
        const int d = 2 * hf + e;
        const int f = 128 * d + fl;
        uint32_t v[HP];
        if (nc > 0) {
#pragma unroll
            for (int j = 0; j < HP / 8; ++j)
                tmem_ld8(tl + TM_O + 64 * d + me * HP + 8 * j, *reinterpret_cast<uint32_t(*)[8]>(&v[8 * j]));
            tmem_wait_ld();
        } else {
#pragma unroll
            for (int i = 0; i < HP; ++i)
                v[i] = 0u;
        }
        // weights read four heads at a time (16-byte shared loads, the same
        // address in every lane)
        const float4 *w4 = reinterpret_cast<const float4 *>(wts);
        float o[HP];
#pragma unroll
        for (int i = 0; i < HP; i += 4) {
            const float4 a = w4[(me * HP + i) / 4];
            o[i] = a.x * __uint_as_float(v[i]);
            o[i + 1] = a.y * __uint_as_float(v[i + 1]);
            o[i + 2] = a.z * __uint_as_float(v[i + 2]);
            o[i + 3] = a.w * __uint_as_float(v[i + 3]);
        }
#pragma unroll
        for (int r = 0; r < P; ++r) {
            if (r == (int)me)
                continue;
#pragma unroll
            for (int i = 0; i < HP; i += 4) {
                const float4 a = w4[(r * HP + i) / 4];
                const uint32_t x0 = recv[(r * HP + i) / 2 * D + f];
                const uint32_t x1 = recv[((r * HP + i) / 2 + 1) * D + f];
                o[i] += a.x * bf16lo_to_f32(x0);
                o[i + 1] += a.y * bf16hi_to_f32(x0);
                o[i + 2] += a.z * bf16lo_to_f32(x1);
                o[i + 3] += a.w * bf16hi_to_f32(x1);
            }
        }
        if (p.rope_dim > 0 && f >= D - p.rope_dim) {   // warp-uniform
            const int pi = (f - (D - p.rope_dim)) >> 1;
            const float *cs = p.rope + ((size_t)(s.q % p.T) * (p.rope_dim >> 1) + pi) * 2;
            const float cth = __ldg(cs), sth = __ldg(cs + 1);
            const bool odd = f & 1;
#pragma unroll
            for (int i = 0; i < HP; ++i) {
                const float other = __shfl_xor_sync(0xffffffffu, o[i], 1);
                o[i] = odd ? (o[i] * cth - other * sth) : (o[i] * cth + other * sth);
            }
        }
        if (!in_bounds(s.q < p.BT && (int)(me + 1) * HP <= H && f < D, p.err)) {
        } else if (p.out_f32) {
            float *po = reinterpret_cast<float *>(p.out) + (size_t)s.q * (H * D) + (size_t)(me * HP) * D + f;
#pragma unroll
            for (int i = 0; i < HP; ++i)
                po[i * D] = o[i];
        } else {
            store_bf16_pairs<HP>(reinterpret_cast<uint16_t *>(p.out) + (size_t)s.q * (H * D) + (size_t)(me * HP) * D, f,
                                 o, lane);
        }
    }
    return true;
}

// Warps 0-7: softmax and epilogue.  Warp w reads TMEM lane quarter qd = w % 4
// (chunk rows 32qd .. 32qd + 31, one per thread) and owns heads
// 32hf .. 32hf + 31, hf = w / 4.
__device__ void softmax_role(const AttnParams &p, uint8_t *smem, uint32_t sbase, uint32_t tmem,
                             int warp, int lane, volatile int *abort_flag)
{
    const int t = threadIdx.x;   // 0..255
    const int qd = warp & 3, hf = warp >> 2;
    const int row = 32 * qd + lane;
    const int hb = 32 * hf;      // first head of this thread
    float *red = reinterpret_cast<float *>(smem + OFF_RED);   // [4 quarters][64 heads]
    float *m_s = reinterpret_cast<float *>(smem + OFF_M);
    float *aux = reinterpret_cast<float *>(smem + OFF_AUX);
    const uint32_t bar0 = sbase + OFF_BAR;
    const uint32_t tl = tmem + ((uint32_t)(qd * 32) << 16);   // this warp's TMEM lane quarter
    const int *segn = reinterpret_cast<const int *>(smem + OFF_SEGN);
    uint32_t ph_sfull = 0, ph_lfull[2] = {0, 0};
    uint32_t chunks = 0;   // chunks processed so far: PV(j) is the (j+1)-th PVDONE completion
    SegIter it;
    seg_begin(p, it);
    Seg s;
    for (int k = 0; seg_next(p, it, s); ++k) {
        const int b = k & 1;
        const bool w0 = warp_wait(bar0 + 8 * (B_LFULL0 + b), ph_lfull[b], abort_flag, p.timeout_ns, lane);
        ph_lfull[b] ^= 1u;
        // also: the previous epilogue is done with m_s / aux
        if (bar_red_or(1, SMX_THREADS, !w0 || *abort_flag))
            break;
        const int n = segn[b];
        __syncwarp();
        if (lane == 0)
            mbar_arrive(bar0 + 8 * (B_LEMPTY0 + b));
        const int nc = (n + CH - 1) / CH;

        if (t < 64)
            m_s[t] = reinterpret_cast<const float *>(smem + OFF_SINK)[t];
        bar_sync(1, SMX_THREADS);

        float l[32];
#pragma unroll
        for (int i = 0; i < 32; ++i)
            l[i] = 0.f;

        bool aborted = false;
        for (int c = 0; c < nc; ++c) {
            // S^T of this chunk is ready.  Its commit tracks every MMA issued
            // before it, including the previous chunk's PV (issued before this
            // chunk's QK): P may be rewritten and O^T rescaled without waiting
            // for PVDONE.
            const bool wok = warp_wait(bar0 + 8 * B_SFULL, ph_sfull, abort_flag, p.timeout_ns, lane);
            ph_sfull ^= 1u;
            ++chunks;
            tc_fence_after();
            uint32_t r[32];
            tmem_ld32(tl + TM_S + hb, r);
            tmem_wait_ld();
            const bool vrow = c * CH + row < n;
            float x[32];
            bool need = false;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                x[i] = vrow ? __uint_as_float(r[i]) * p.scale_log2 : -INFINITY;
                need |= x[i] > m_s[hb + i] + RESCALE_THRESHOLD;
            }
            // probabilities in bf16 (the MMA operand) against the current maxima,
            // computed before the vote so that the barrier absorbs the warps'
            // skew; they are recomputed in the rare chunk that moves a maximum
            uint32_t pk[16];
            auto probabilities = [&]() {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    pk[i] = pack_bf16x2(ex2(x[2 * i] - m_s[hb + 2 * i]), ex2(x[2 * i + 1] - m_s[hb + 2 * i + 1]));
            };
            probabilities();
            // one barrier in the common case: it carries the rescale vote and
            // any failed wait; a second one tells the two apart
            if (bar_red_or(1, SMX_THREADS, need || !wok || *abort_flag)) {
                if (bar_red_or(1, SMX_THREADS, !wok || *abort_flag)) {
                    aborted = true;
                    break;
                }
                // move the running maximum to this chunk's maximum (per head)
                red[qd * 64 + hb + lane] = warp_reduce32<true>(x, lane);
                bar_sync(1, SMX_THREADS);
                if (t < 64) {
                    const float mx = fmaxf(fmaxf(red[t], red[64 + t]), fmaxf(red[128 + t], red[192 + t]));
                    const float mo = m_s[t];
                    const float mn = fmaxf(mo, mx);
                    aux[t] = ex2(mo - mn);
                    m_s[t] = mn;
                }
                bar_sync(1, SMX_THREADS);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    l[i] *= aux[hb + i];
                if (c > 0) {
#pragma unroll 1
                    for (int d = 0; d < 4; ++d) {
                        uint32_t o[32];
                        const uint32_t ta = tl + TM_O + 64 * d + hb;
                        tmem_ld32(ta, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            o[i] = __float_as_uint(__uint_as_float(o[i]) * aux[hb + i]);
                        tmem_st32(ta, o);
                    }
                    tmem_wait_st();
                }
                // x was consumed by the reduction: rebuild it from S^T
                tmem_ld32(tl + TM_S + hb, r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    x[i] = vrow ? __uint_as_float(r[i]) * p.scale_log2 : -INFINITY;
                probabilities();
            }
            // row sums of the rounded probabilities
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                l[2 * i] += bf16lo_to_f32(pk[i]);
                l[2 * i + 1] += bf16hi_to_f32(pk[i]);
            }
            // P^T row `row`: 64 heads x bf16 = 128 bytes, 16-byte chunks swizzled
            uint8_t *prow = smem + OFF_P + row * 128;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int c8 = 4 * hf + j;
                *reinterpret_cast<uint4 *>(prow + ((c8 ^ (row & 7)) << 4)) =
                    make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar0 + 8 * B_PFULL);
        }
        if (aborted)
            break;
        if (nc > 0) {
            // the segment's last PV: completion number `chunks`; every earlier
            // one has completed (each chunk's S^T commit covered the PV before it)
            const bool w = warp_wait(bar0 + 8 * B_PVDONE, (chunks - 1u) & 1u, abort_flag, p.timeout_ns, lane);
            if (bar_red_or(1, SMX_THREADS, !w || *abort_flag))
                break;
            tc_fence_after();
        }
        // split schedule: the chunk buffer is free; offer it to the peers now,
        // ahead of the row sums (they write their partials into it)
        if (!s.full && t < p.pieces && t != (int)cluster_ctarank())
            mbar_arrive_remote(mapa_shared(bar0 + 8 * B_XRDY, (uint32_t)t));

        // row sums: reduce the per-row partials over the rows of each warp, then the quarters
        red[qd * 64 + hb + lane] = warp_reduce32<false>(l, lane);
        bar_sync(1, SMX_THREADS);
        if (t < 64) {
            const float lt = red[t] + red[64 + t] + red[128 + t] + red[192 + t];
            if (s.full) {
                const float den = lt + ex2(reinterpret_cast<const float *>(smem + OFF_SINK)[t] - m_s[t]);
                aux[t] = lt > 0.f ? 1.f / den : 0.f;
            } else {
                aux[t] = lt;
            }
        }
        bar_sync(1, SMX_THREADS);

        if (!s.full) {
            bool mok = false;
            switch (p.pieces) {
            case 2: mok = cluster_merge<2>(p, smem, sbase, tl, s, nc, t, qd, hf, abort_flag, lane); break;
            case 4: mok = cluster_merge<4>(p, smem, sbase, tl, s, nc, t, qd, hf, abort_flag, lane); break;
            case 8: mok = cluster_merge<8>(p, smem, sbase, tl, s, nc, t, qd, hf, abort_flag, lane); break;
            default: break;
            }
            if (!mok)
                break;
            if (nc > 0) {
                tc_fence_before();
                mbar_arrive(bar0 + 8 * B_OFREE);
            }
            continue;
        }

        // epilogue: thread (qd, lane, hf) owns feature 128d + 32qd + lane of heads hb .. hb + 31
        const bool rope_here = p.rope_dim > 0;
#pragma unroll 1
        for (int d = 0; d < 4; ++d) {
            const int dim = 128 * d + row;
            uint32_t u[32];
            if (nc > 0) {
                tmem_ld32(tl + TM_O + 64 * d + hb, u);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    u[i] = __float_as_uint(__uint_as_float(u[i]) * aux[hb + i]);
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
            if (!in_bounds(s.q < p.BT && hb + 32 <= H && dim < D, p.err)) {
            } else if (p.out_f32) {
                float *po = reinterpret_cast<float *>(p.out) + (size_t)s.q * (H * D) + (size_t)hb * D + dim;
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    po[i * D] = __uint_as_float(u[i]);
            } else {
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    v[i] = __uint_as_float(u[i]);
                store_bf16_pairs<32>(reinterpret_cast<uint16_t *>(p.out) + (size_t)s.q * (H * D) + (size_t)hb * D, dim,
                                     v, lane);
            }
        }
        if (nc > 0) {
            tc_fence_before();
            mbar_arrive(bar0 + 8 * B_OFREE);
        }
    }
}

template <bool TWO, bool FP4>
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
            mbar_init(bar0 + 8 * (B_KVFULL0 + d), GATHER_GROUP_WARPS);
            mbar_init(bar0 + 8 * (B_KVFREE0 + d), 1);
        }
        mbar_init(bar0 + 8 * B_SFULL, 1);
        mbar_init(bar0 + 8 * B_PFULL, SMX_THREADS);
        mbar_init(bar0 + 8 * B_PVDONE, 1);
        mbar_init(bar0 + 8 * B_OFREE, SMX_THREADS);
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar0 + 8 * (B_LFULL0 + b), 32);
            mbar_init(bar0 + 8 * (B_LEMPTY0 + b), LEMPTY_ARRIVALS);
        }
        mbar_init(bar0 + 8 * B_DONE, 1);
        mbar_init(bar0 + 8 * B_XRDY, p.split ? (uint32_t)(p.pieces - 1) : 1u);
        mbar_init(bar0 + 8 * B_XFULL, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&p.tm_q);
    }
    if (warp == WARP_MMA) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    // Programmatic dependent launch: everything above may overlap the previous
    // kernel in the stream; every global memory access below waits for it to
    // complete.  The next kernel may be scheduled as this grid's CTAs leave.
    griddep_wait();
    griddep_launch_dependents();
    // the control warp starts copying the sinks and the first index list now,
    // so that their latency overlaps the rest of the set-up; it waits for the
    // copies, scales the sinks and publishes both with the first list
    if (warp == WARP_CONTROL) {
        cp_async4(sbase + OFF_SINK + 4u * lane, p.sink + lane);
        cp_async4(sbase + OFF_SINK + 4u * (lane + 32), p.sink + lane + 32);
        SegIter it;
        seg_begin(p, it);
        Seg s;
        if (seg_next(p, it, s))
            stage_list(p, s, sbase + OFF_RAW, lane);
        else
            cp_async_commit();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // the peers' barriers are initialised before any CTA of the cluster arrives on them
    if (p.split) {
        __syncwarp();
        cluster_sync();
    }

    if (warp < NUM_SOFTMAX_WARPS) {
        // the softmax warps keep 32 scores and 32 row sums per thread
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(REGS_SOFTMAX) : "memory");
        softmax_role(p, smem, sbase, tmem, warp, lane, abort_flag);
    } else if (warp < WARP_GATHER0 + NUM_GATHER_WARPS) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REGS_GATHER) : "memory");
        gather_role<TWO, FP4>(p, smem, sbase, warp - WARP_GATHER0, lane, abort_flag);
    } else {
        // the last warpgroup: control warp, MMA warp and two warps without a role
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REGS_LAST) : "memory");
        if (warp == WARP_CONTROL)
            control_role<TWO, FP4>(p, smem, sbase, lane, abort_flag);
        else if (warp == WARP_MMA && lane == 0)
            mma_role(p, smem, sbase, tmem, abort_flag);
    }

    tc_fence_before();
    __syncthreads();
    // no CTA leaves while a peer may still write into its shared memory
    if (p.split) {
        __syncwarp();
        cluster_sync();
    }
    if (threadIdx.x == 0 && *abort_flag)
        atomicOr(p.err, ERRBIT_TIMEOUT);
    if (warp == WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
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
    // 128-row chunk each), a power of two up to the cluster limit, so that
    // about every SM holds one piece and the pieces' heads split evenly.
    int pieces = 1;
    if (BT > 0 && BT < num_sms && K > 0) {
        int64_t lim = num_sms / BT;
        const int64_t by_len = (K + 127) / 128;
        if (by_len < lim)
            lim = by_len;
        if (lim > attn::MAX_CLUSTER)
            lim = attn::MAX_CLUSTER;
        while (pieces * 2 <= lim)
            pieces *= 2;
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

size_t attn_workspace_bytes(int64_t BT, int K)
{
    (void)BT;
    (void)K;
    // the split pieces of a query merge on chip: only the error header
    return WS_HEADER;
}

cudaError_t launch_attention(AttnParams &p, const Schedule &s, cudaStream_t st)
{
    // the two-source builds only when a second source is in use
    const bool second = p.W < p.N;
    void (*kernel)(AttnParams) = second && p.kv2_codes ? attn::attn_kernel<true, true>
                                 : second && p.kv2  ? attn::attn_kernel<true, false>
                                                    : attn::attn_kernel<false, false>;
    cudaError_t ea = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)attn::SMEM_BYTES);
    if (ea != cudaSuccess)
        return ea;
    p.split = s.split;
    p.per_cta = s.per_cta;
    p.pieces = s.pieces;
    if (s.grid == 0)
        return cudaSuccess;
    // the pieces of one query form a cluster (they merge through distributed
    // shared memory); programmatic dependent launch lets the set-up overlap
    // the previous kernel in the stream
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)s.grid);
    cfg.blockDim = dim3(attn::THREADS);
    cfg.dynamicSmemBytes = attn::SMEM_BYTES;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (s.split) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = (unsigned)s.pieces;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

}  // namespace sa
