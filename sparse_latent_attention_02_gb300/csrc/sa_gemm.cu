// sa_gemm.cu -- the grouped low-rank output projection `wo_a` for sm_103a.
//
// "DeepSeek-V4.1 > Output projection" page, Attention.forward: the attention
// output viewed as [B, T, G, H*D/G] is multiplied group by group with
// `wo_a.weight.view(G, R, -1)` (`einsum("bsgd,grd->bsgr")`), a block-diagonal
// product -- G independent GEMMs that share one launch:
//   y[m, g*R + r] = sum_d o[m, g*Din + d] * W[g*R + r, d]
//
// bf16 weights (wo_a_pair_kernel): persistent over clusters of two CTAs,
// one per SM, each pair computing tiles of 256 tokens x 256 rank columns with
// tcgen05.mma.cta_group::2 (M = 256 split across the pair, N = 256, K = 16),
// K in blocks of 64 features through a 6-stage TMA ring (128-byte swizzle)
// in which each CTA holds its own 128 tokens and 128 rank rows; two TMEM
// accumulators per CTA so that the epilogue of one tile overlaps the main
// loop of the next.
//
// fp8 weights (the page notes that an fp8 grouped GEMM would halve the
// weight's memory): W is stored as E4M3 with one fp32 scale per 128 x 128
// block.  From 512 tokens on, the weight is decoded once into a bf16 copy
// (dequant_fp8_kernel) and multiplied by the bf16 kernel.  Below that,
// wo_a_fp8_kernel (one CTA per SM) decodes it on the fly: tiles of 256 tokens
// x 128 rank columns (two M=128 MMAs share each weight block, so every weight
// is decoded once per 256 tokens) in four 48 KB stages.  Warp 14 streams the
// 128 x 64 blocks of raw E4M3 bytes by TMA into a ring of their own, ahead of
// the stages; warps 6-13 write each into its stage's swizzled bf16 weight
// slot as bf16(fp32(value * scale)) -- the weight the page's bf16 conversion
// would give -- as soon as the MMAs have released the slot, while the
// activations' TMA for the same stage is in flight.  Only the weight's bytes
// change; the products are the bf16 GEMM's.
#include <atomic>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sa_internal.h"
#include "sa_ptx.cuh"

namespace sa {
namespace gemm {

constexpr int BK = 64;
constexpr int FP8_BLOCK = 128;                // weight rows / columns per fp32 scale
constexpr int CONV_WARP0 = 6, CONV_THREADS = 256;
constexpr int RAW_WARP = CONV_WARP0 + CONV_THREADS / 32;   // 14: TMA of the raw weights

// The fp8-weight kernel's configuration.
struct Cfg {
    static constexpr int BM = 256;                             // tokens per tile
    static constexpr int BN = 128;                             // rank columns per tile
    static constexpr int HALVES = BM / 128;                    // M=128 MMAs per K step
    static constexpr uint32_t A_BYTES = BM * BK * 2;           // 32 KB
    static constexpr uint32_t B_BYTES = BN * BK * 2;           // 16 KB (the decoded weights)
    static constexpr uint32_t RAW_BYTES = BN * BK;             // raw E4M3 weights of one K block
    static constexpr uint32_t ACC_COLS = HALVES * BN;          // TMEM columns of one accumulator
    static constexpr int STAGES = 4;
    static constexpr int THREADS = 192 + CONV_THREADS + 32;
    static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr uint32_t OFF_RAW = STAGES * STAGE_BYTES;  // raw ring, one slot per stage
    static constexpr uint32_t OFF_BAR = OFF_RAW + STAGES * RAW_BYTES;
    static constexpr uint32_t OFF_MISC = OFF_BAR + 32 * 8;
    static constexpr uint32_t SMEM_BYTES = OFF_MISC + 64 + 1024;
    static constexpr uint32_t IDESC = idesc_bf16(128, BN, 0, 0);
    // barriers: TMA full, stage empty, converted, raw full / free,
    // accumulators, done
    static constexpr uint32_t B_FULL0 = 0, B_EMPTY0 = STAGES, B_CONV0 = 2 * STAGES, B_RAWFULL0 = 3 * STAGES,
                              B_RAWFREE0 = 4 * STAGES, B_ACCFULL0 = 5 * STAGES, B_ACCEMPTY0 = B_ACCFULL0 + 2,
                              B_DONE = B_ACCEMPTY0 + 2, NUM_BARS = B_DONE + 1;
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
    static_assert(NUM_BARS <= 32, "barrier area");
    static_assert(2 * ACC_COLS <= 512, "two accumulators in TMEM");
    static_assert(BN % FP8_BLOCK == 0, "a weight tile spans whole scale blocks");
};

// Sixteen E4M3 weights times their block's scale, as sixteen bf16 (two
// 16-byte pieces): each byte pair is converted to f16 by the hardware
// (exact), widened to fp32 (exact), multiplied by the scale with one fp32
// rounding and rounded to bf16.
__device__ __forceinline__ void dequant_e4m3x16(const uint4 &w, float scale, uint4 &lo, uint4 &hi)
{
    const uint32_t in[4] = {w.x, w.y, w.z, w.w};
    uint32_t out[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t h0, h1;
        asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
            "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
            : "=r"(h0), "=r"(h1)
            : "r"(in[i]));
        const __half2 p0 = *reinterpret_cast<const __half2 *>(&h0), p1 = *reinterpret_cast<const __half2 *>(&h1);
        out[2 * i] = pack_bf16x2(__fmul_rn(__low2float(p0), scale), __fmul_rn(__high2float(p0), scale));
        out[2 * i + 1] = pack_bf16x2(__fmul_rn(__low2float(p1), scale), __fmul_rn(__high2float(p1), scale));
    }
    lo = make_uint4(out[0], out[1], out[2], out[3]);
    hi = make_uint4(out[4], out[5], out[6], out[7]);
}

// Warp-uniform bounded wait (lane 0 polls).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          uint64_t limit_ns, int lane)
{
    int ok = 0;
    if (lane == 0)
        ok = bounded_wait(bar, parity, abort_flag, limit_ns) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

struct TileMap {
    int num_m, num_n, total;
    __device__ void at(int id, int &g, int &mb, int &nb) const
    {
        nb = id % num_n;
        const int rest = id / num_n;
        mb = rest % num_m;
        g = rest / num_m;
    }
};

__global__ void __launch_bounds__(Cfg::THREADS, 1) wo_a_fp8_kernel(const __grid_constant__ GemmParams p)
{
    using C = Cfg;
    constexpr int STAGES = C::STAGES, BM = C::BM, BN = C::BN;
    constexpr uint32_t STAGE_BYTES = C::STAGE_BYTES, OFF_BAR = C::OFF_BAR, OFF_MISC = C::OFF_MISC;
    constexpr uint32_t A_BYTES = C::A_BYTES;
    constexpr uint32_t B_FULL0 = C::B_FULL0, B_EMPTY0 = C::B_EMPTY0, B_CONV0 = C::B_CONV0,
                       B_RAWFULL0 = C::B_RAWFULL0, B_RAWFREE0 = C::B_RAWFREE0, B_ACCFULL0 = C::B_ACCFULL0,
                       B_ACCEMPTY0 = C::B_ACCEMPTY0, B_DONE = C::B_DONE;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + OFF_BAR;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_MISC + 4);

    TileMap tm;
    tm.num_m = (p.M + BM - 1) / BM;
    tm.num_n = p.R / BN;
    tm.total = tm.num_m * tm.num_n * p.G;
    const int kblocks = p.Din / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar0 + 8 * (B_FULL0 + s), 1);
            mbar_init(bar0 + 8 * (B_EMPTY0 + s), 1);
            mbar_init(bar0 + 8 * (B_CONV0 + s), CONV_THREADS / 32);
            mbar_init(bar0 + 8 * (B_RAWFULL0 + s), 1);
            mbar_init(bar0 + 8 * (B_RAWFREE0 + s), CONV_THREADS / 32);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar0 + 8 * (B_ACCFULL0 + a), 1);
            mbar_init(bar0 + 8 * (B_ACCEMPTY0 + a), 128);
        }
        mbar_init(bar0 + 8 * B_DONE, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&p.tm_a);
        prefetch_tmap(&p.tm_b8);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------- TMA producer
        if (lane == 0) {
            uint32_t stage = 0, ph = 0;
            bool ok = true;
            uint32_t issued = 0;
            for (int id = blockIdx.x; id < tm.total && ok; id += gridDim.x) {
                int g, mb, nb;
                tm.at(id, g, mb, nb);
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!bounded_wait(bar0 + 8 * (B_EMPTY0 + stage), ph ^ 1u, abort_flag, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = bar0 + 8 * (B_FULL0 + stage);
                    const uint32_t sa_ = sbase + stage * STAGE_BYTES;
                    mbar_arrive_expect_tx(fb, A_BYTES);
                    // activations: 128-row boxes (rows past M read as zero)
#pragma unroll
                    for (int h = 0; h < C::HALVES; ++h)
                        tma_load_2d(sa_ + h * 128 * BK * 2, &p.tm_a, g * p.Din + kb * BK, mb * BM + 128 * h, fb);
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        ph ^= 1u;
                    }
                }
            }
            // the last load of every stage must land before the CTA may exit:
            // load n went to stage n % STAGES, phase (n / STAGES) & 1
            for (uint32_t k = 0; k < STAGES && k < issued; ++k) {
                const uint32_t n = issued - 1 - k;
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(bar0 + 8 * (B_FULL0 + n % STAGES), (n / STAGES) & 1u))
                    if (globaltimer_ns() - t0 > p.timeout_ns)
                        break;
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            uint32_t stage = 0, ph = 0;
            uint32_t acc_ph[2] = {0, 0};
            int local = 0;
            bool ok = true;
            for (int id = blockIdx.x; id < tm.total && ok; id += gridDim.x, ++local) {
                const int a = local & 1;
                if (!bounded_wait(bar0 + 8 * (B_ACCEMPTY0 + a), acc_ph[a] ^ 1u, abort_flag, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                acc_ph[a] ^= 1u;
                tc_fence_after();
                const uint32_t dt = tmem + (uint32_t)(a * C::ACC_COLS);
                for (int kb = 0; kb < kblocks; ++kb) {
                    // the stage's TMA has landed and the converters are done
                    if (!bounded_wait(bar0 + 8 * (B_FULL0 + stage), ph, abort_flag, p.timeout_ns) ||
                        !bounded_wait(bar0 + 8 * (B_CONV0 + stage), ph, abort_flag, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa_ = sbase + stage * STAGE_BYTES;
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        const uint64_t bd = smem_desc_sw128(sa_ + A_BYTES + k * 32, 16, 1024);
#pragma unroll
                        for (int h = 0; h < C::HALVES; ++h) {
                            const uint64_t ad = smem_desc_sw128(sa_ + h * 128 * BK * 2 + k * 32, 16, 1024);
                            mma_bf16_ss(dt + (uint32_t)(h * BN), ad, bd, C::IDESC, (kb > 0 || k > 0) ? 1u : 0u);
                        }
                    }
                    mma_commit(bar0 + 8 * (B_EMPTY0 + stage));
                    if (++stage == STAGES) {
                        stage = 0;
                        ph ^= 1u;
                    }
                }
                if (ok)
                    mma_commit(bar0 + 8 * (B_ACCFULL0 + a));
            }
            mma_commit(bar0 + 8 * B_DONE);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(bar0 + 8 * B_DONE, 0))
                if (globaltimer_ns() - t0 > p.timeout_ns)
                    break;
        }
        __syncwarp();
    } else if (warp == RAW_WARP) {
        // ---------------- TMA of the raw E4M3 weight blocks into their ring
        if (lane == 0) {
            uint32_t slot = 0, ph = 0, issued = 0;
            bool ok = true;
            for (int id = blockIdx.x; id < tm.total && ok; id += gridDim.x) {
                int g, mb, nb;
                tm.at(id, g, mb, nb);
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!bounded_wait(bar0 + 8 * (B_RAWFREE0 + slot), ph ^ 1u, abort_flag, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = bar0 + 8 * (B_RAWFULL0 + slot);
                    mbar_arrive_expect_tx(fb, C::RAW_BYTES);
                    tma_load_2d(sbase + C::OFF_RAW + slot * C::RAW_BYTES, &p.tm_b8, kb * BK, g * p.R + nb * BN, fb);
                    ++issued;
                    if (++slot == STAGES) {
                        slot = 0;
                        ph ^= 1u;
                    }
                }
            }
            for (uint32_t k = 0; k < STAGES && k < issued; ++k) {
                const uint32_t n = issued - 1 - k;
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(bar0 + 8 * (B_RAWFULL0 + n % STAGES), (n / STAGES) & 1u))
                    if (globaltimer_ns() - t0 > p.timeout_ns)
                        break;
            }
        }
        __syncwarp();
    } else if (warp >= CONV_WARP0) {
        // ---------------- fp8 weights -> swizzled bf16 operand (warps 6..13).
        // Thread ct converts 16-byte pieces i = ct + 256 it of the raw BN x 64
        // block (row i / 4, piece i % 4 = features 16 (i % 4) ..); the block lies
        // in one 128 x 128 scale block.  Raw slot and stage advance together.
        const int ct = threadIdx.x - CONV_WARP0 * 32;
        const int scale_cols = p.Din / FP8_BLOCK;
        constexpr int ITEMS = BN * BK / 16 / CONV_THREADS;
        static_assert(ITEMS * CONV_THREADS * 16 == BN * BK, "converter items");
        uint32_t stage = 0, ph = 0;
        bool ok = true;
        for (int id = blockIdx.x; id < tm.total && ok; id += gridDim.x) {
            int g, mb, nb;
            tm.at(id, g, mb, nb);
            const int n0 = g * p.R + nb * BN;
            for (int kb = 0; kb < kblocks; ++kb) {
                // the raw block has landed and the MMAs have released the stage
                ok = warp_wait(bar0 + 8 * (B_RAWFULL0 + stage), ph, abort_flag, p.timeout_ns, lane) &&
                     warp_wait(bar0 + 8 * (B_EMPTY0 + stage), ph ^ 1u, abort_flag, p.timeout_ns, lane);
                if (!ok)
                    break;
                const float s = __ldg(p.b_scales + (size_t)(n0 / FP8_BLOCK) * scale_cols + (kb * BK) / FP8_BLOCK);
                const uint8_t *raw = smem + C::OFF_RAW + stage * C::RAW_BYTES;
                uint8_t *dst = smem + stage * STAGE_BYTES + A_BYTES;
                uint4 w[ITEMS];
#pragma unroll
                for (int it = 0; it < ITEMS; ++it) {
                    const int i = ct + CONV_THREADS * it;
                    w[it] = *reinterpret_cast<const uint4 *>(raw + (i >> 2) * BK + 16 * (i & 3));
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar0 + 8 * (B_RAWFREE0 + stage));
#pragma unroll
                for (int it = 0; it < ITEMS; ++it) {
                    const int i = ct + CONV_THREADS * it, r = i >> 2, j = i & 3;
                    uint4 lo, hi;
                    dequant_e4m3x16(w[it], s, lo, hi);
                    *reinterpret_cast<uint4 *>(dst + r * 128 + (((2 * j) ^ (r & 7)) << 4)) = lo;
                    *reinterpret_cast<uint4 *>(dst + r * 128 + (((2 * j + 1) ^ (r & 7)) << 4)) = hi;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar0 + 8 * (B_CONV0 + stage));
                if (++stage == STAGES) {
                    stage = 0;
                    ph ^= 1u;
                }
            }
        }
    } else {
        // ---------------- epilogue: warps 2..5 -> TMEM lane quarters 2,3,0,1;
        // accumulator half h holds tile rows 128h .. 128h+127
        const int quarter = warp & 3;
        const int row_in_half = quarter * 32 + lane;
        uint32_t acc_ph[2] = {0, 0};
        int local = 0;
        for (int id = blockIdx.x; id < tm.total; id += gridDim.x, ++local) {
            const int a = local & 1;
            int ok = 0;
            if (lane == 0)
                ok = bounded_wait(bar0 + 8 * (B_ACCFULL0 + a), acc_ph[a], abort_flag, p.timeout_ns) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            acc_ph[a] ^= 1u;
            if (bar_red_or(1, 128, ok == 0))
                break;
            tc_fence_after();
            int g, mb, nb;
            tm.at(id, g, mb, nb);
#pragma unroll 1
            for (int h = 0; h < C::HALVES; ++h) {
                const int m = mb * BM + 128 * h + row_in_half;
                const uint32_t ta = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(a * C::ACC_COLS + h * BN);
                uint16_t *yrow = p.y + (size_t)m * (p.G * p.R) + g * p.R + nb * BN;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(ta + 32 * c, v);
                    tmem_wait_ld();
                    if (m < p.M && in_bounds(inside(yrow + 32 * c, 64, p.y, (size_t)p.M * p.G * p.R * 2), p.err)) {
                        uint4 *dst = reinterpret_cast<uint4 *>(yrow + 32 * c);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            dst[j] = make_uint4(
                                pack_bf16x2(__uint_as_float(v[8 * j + 0]), __uint_as_float(v[8 * j + 1])),
                                pack_bf16x2(__uint_as_float(v[8 * j + 2]), __uint_as_float(v[8 * j + 3])),
                                pack_bf16x2(__uint_as_float(v[8 * j + 4]), __uint_as_float(v[8 * j + 5])),
                                pack_bf16x2(__uint_as_float(v[8 * j + 6]), __uint_as_float(v[8 * j + 7])));
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(bar0 + 8 * (B_ACCEMPTY0 + a));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag)
        atomicOr(p.err, ERRBIT_TIMEOUT);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------- two-SM bf16 GEMM
//
// bf16 weights: a cluster of two CTAs (one per SM) computes tiles of 256
// tokens x 256 rank columns with tcgen05.mma.cta_group::2 (M = 256 across
// the pair, N = 256, K = 16), issued by the even CTA.  Per 64-wide K block
// each CTA's stage holds its 128 tokens of A and its 128 rank rows of B
// (32 KB), so each SM's shared memory takes 32 KB of TMA writes and serves
// 32 KB of operand reads per 512 MMA cycles -- about the 128 bytes per clock
// it can move -- where one SM alone with N = 256 needs 48 KB of each.
//   warp 0 (both CTAs): TMA producer; each stage's two loads complete their
//     bytes on the even CTA's full barrier (two arrivals: one per CTA)
//   warp 1: TMEM owner (both CTAs, collective pair allocation) and, in the
//     even CTA, the MMA issuer; its commits arrive on both CTAs' barriers
//   warps 2-5 (both CTAs): epilogue from their own TMEM (tile rows 128 r ..,
//     r = rank), releasing the accumulator on the even CTA's barrier
namespace pair {

constexpr int BM = 256, BN = 256, STAGES = 6, THREADS = 192;
constexpr uint32_t A_BYTES = 128 * BK * 2;        // this CTA's 128 tokens x 64 features
constexpr uint32_t B_BYTES = 128 * BK * 2;        // this CTA's 128 rank rows x 64 features
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t OFF_BAR = STAGES * STAGE_BYTES;
constexpr uint32_t OFF_MISC = OFF_BAR + 32 * 8;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 64 + 1024;
constexpr uint32_t ACC_COLS = BN;                  // one accumulator: 256 TMEM columns
constexpr uint32_t IDESC = idesc_bf16(256, BN, 0, 0);
// barriers: full (even CTA: both CTAs' loads), empty (each CTA), accumulator
// full (each CTA) / empty (even CTA: both CTAs' epilogues), done (even CTA)
constexpr uint32_t B_FULL0 = 0, B_EMPTY0 = STAGES, B_ACCFULL0 = 2 * STAGES, B_ACCEMPTY0 = B_ACCFULL0 + 2,
                   B_DONE = B_ACCEMPTY0 + 2, NUM_BARS = B_DONE + 1;
constexpr uint32_t EPI_WARPS = 4;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
static_assert(NUM_BARS <= 32, "barrier area");
static_assert(2 * ACC_COLS <= 512, "two accumulators in TMEM");

__global__ void __launch_bounds__(THREADS, 1) wo_a_pair_kernel(const __grid_constant__ GemmParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + OFF_BAR;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_MISC + 4);
    // the even CTA's barriers, as cluster addresses
    const uint32_t lead0 = mapa_shared(bar0, 0);

    TileMap tm;
    tm.num_m = (p.M + BM - 1) / BM;
    tm.num_n = p.R / BN;
    tm.total = tm.num_m * tm.num_n * p.G;
    const int kblocks = p.Din / BK;
    const int pair_id = (int)(blockIdx.x >> 1), num_pairs = (int)(gridDim.x >> 1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar0 + 8 * (B_FULL0 + s), 2);
            mbar_init(bar0 + 8 * (B_EMPTY0 + s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar0 + 8 * (B_ACCFULL0 + a), 1);
            mbar_init(bar0 + 8 * (B_ACCEMPTY0 + a), 2 * EPI_WARPS);
        }
        mbar_init(bar0 + 8 * B_DONE, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&p.tm_a);
        prefetch_tmap(&p.tm_b);
    }
    if (warp == 1)
        tmem_alloc_pair(smem_u32(tmem_slot), 512);
    tc_fence_before();
    __syncthreads();
    // both CTAs' barriers are initialised before either arrives on the other's
    __syncwarp();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------- TMA producer (both CTAs)
        if (lane == 0) {
            uint32_t stage = 0, ph = 0, issued = 0;
            bool ok = true;
            for (int id = pair_id; id < tm.total && ok; id += num_pairs) {
                int g, mb, nb;
                tm.at(id, g, mb, nb);
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!bounded_wait(bar0 + 8 * (B_EMPTY0 + stage), ph ^ 1u, abort_flag, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = lead0 + 8 * (B_FULL0 + stage);
                    const uint32_t sa_ = sbase + stage * STAGE_BYTES;
                    mbar_arrive_expect_tx_cluster(fb, STAGE_BYTES);
                    // this CTA's 128 tokens (rows past M read as zero) and 128 rank rows
                    tma_load_2d_pair(sa_, &p.tm_a, g * p.Din + kb * BK, mb * BM + 128 * (int)rank, fb);
                    tma_load_2d_pair(sa_ + A_BYTES, &p.tm_b, kb * BK, g * p.R + nb * BN + 128 * (int)rank, fb);
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        ph ^= 1u;
                    }
                }
            }
            // the even CTA sees every load land (its full barriers count both
            // CTAs' bytes) before the pair may leave: load n went to stage
            // n % STAGES, phase (n / STAGES) & 1
            if (rank == 0) {
                for (uint32_t k = 0; k < STAGES && k < issued; ++k) {
                    const uint32_t n = issued - 1 - k;
                    const uint64_t t0 = globaltimer_ns();
                    while (!mbar_try_wait(bar0 + 8 * (B_FULL0 + n % STAGES), (n / STAGES) & 1u))
                        if (globaltimer_ns() - t0 > p.timeout_ns)
                            break;
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer (even CTA)
        if (rank == 0 && lane == 0) {
            uint32_t stage = 0, ph = 0;
            uint32_t acc_ph[2] = {0, 0};
            int local = 0;
            bool ok = true;
            for (int id = pair_id; id < tm.total && ok; id += num_pairs, ++local) {
                const int a = local & 1;
                // both CTAs' epilogues have drained this accumulator
                if (!bounded_wait(bar0 + 8 * (B_ACCEMPTY0 + a), acc_ph[a] ^ 1u, abort_flag, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                acc_ph[a] ^= 1u;
                tc_fence_after();
                const uint32_t dt = tmem + (uint32_t)(a * ACC_COLS);
                for (int kb = 0; kb < kblocks; ++kb) {
                    // both CTAs' loads of the stage have landed
                    if (!bounded_wait(bar0 + 8 * (B_FULL0 + stage), ph, abort_flag, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa_ = sbase + stage * STAGE_BYTES;
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        const uint64_t ad = smem_desc_sw128(sa_ + k * 32, 16, 1024);
                        const uint64_t bd = smem_desc_sw128(sa_ + A_BYTES + k * 32, 16, 1024);
                        mma_bf16_ss_pair(dt, ad, bd, IDESC, (kb > 0 || k > 0) ? 1u : 0u);
                    }
                    // the stage is free in both CTAs once these products complete
                    mma_commit_pair(bar0 + 8 * (B_EMPTY0 + stage), 3);
                    if (++stage == STAGES) {
                        stage = 0;
                        ph ^= 1u;
                    }
                }
                if (ok)
                    mma_commit_pair(bar0 + 8 * (B_ACCFULL0 + a), 3);
            }
            mma_commit_pair(bar0 + 8 * B_DONE, 1);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(bar0 + 8 * B_DONE, 0))
                if (globaltimer_ns() - t0 > p.timeout_ns)
                    break;
        }
        __syncwarp();
    } else {
        // ---------------- epilogue: warps 2..5 -> TMEM lane quarters 2,3,0,1
        // (tile rows 128 rank + 32 quarter + lane)
        const int quarter = warp & 3;
        const int row = 128 * (int)rank + quarter * 32 + lane;
        uint32_t acc_ph[2] = {0, 0};
        int local = 0;
        for (int id = pair_id; id < tm.total; id += num_pairs, ++local) {
            const int a = local & 1;
            int ok = 0;
            if (lane == 0)
                ok = bounded_wait(bar0 + 8 * (B_ACCFULL0 + a), acc_ph[a], abort_flag, p.timeout_ns) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            acc_ph[a] ^= 1u;
            if (bar_red_or(1, 32 * EPI_WARPS, ok == 0))
                break;
            tc_fence_after();
            int g, mb, nb;
            tm.at(id, g, mb, nb);
            const int m = mb * BM + row;
            const uint32_t ta = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(a * ACC_COLS);
            uint16_t *yrow = p.y + (size_t)m * (p.G * p.R) + g * p.R + nb * BN;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(ta + 32 * c, v);
                tmem_wait_ld();
                if (m < p.M && in_bounds(inside(yrow + 32 * c, 64, p.y, (size_t)p.M * p.G * p.R * 2), p.err)) {
                    uint4 *dst = reinterpret_cast<uint4 *>(yrow + 32 * c);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        dst[j] = make_uint4(
                            pack_bf16x2(__uint_as_float(v[8 * j + 0]), __uint_as_float(v[8 * j + 1])),
                            pack_bf16x2(__uint_as_float(v[8 * j + 2]), __uint_as_float(v[8 * j + 3])),
                            pack_bf16x2(__uint_as_float(v[8 * j + 4]), __uint_as_float(v[8 * j + 5])),
                            pack_bf16x2(__uint_as_float(v[8 * j + 6]), __uint_as_float(v[8 * j + 7])));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive_remote(lead0 + 8 * (B_ACCEMPTY0 + a));
        }
    }

    tc_fence_before();
    __syncthreads();
    // neither CTA releases its tensor memory or leaves while the pair's
    // products, loads or arrivals may still touch it
    __syncwarp();
    cluster_sync();
    if (threadIdx.x == 0 && *abort_flag)
        atomicOr(p.err, ERRBIT_TIMEOUT);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, 512);
    }
}

}  // namespace pair

// E4M3 weight [rows, cols] with one fp32 scale per 128 x 128 block -> bf16
// [rows, cols], each value bf16(fp32(e4m3 * scale)) as in the fused decoders;
// a thread converts 16 bytes per step (grid-stride).  cols % 128 == 0.
__global__ void __launch_bounds__(256) dequant_fp8_kernel(const uint8_t *__restrict__ w8,
                                                          const float *__restrict__ scales,
                                                          uint16_t *__restrict__ w16, int rows, int cols)
{
    const int per_row = cols / 16;
    const int total = rows * per_row;
    const int scale_cols = cols / FP8_BLOCK;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
        const int r = i / per_row, c = (i - r * per_row) * 16;
        const size_t off = (size_t)r * cols + c;
        const uint4 w = __ldg(reinterpret_cast<const uint4 *>(w8 + off));
        const float sc = __ldg(scales + (size_t)(r / FP8_BLOCK) * scale_cols + c / FP8_BLOCK);
        uint4 lo, hi;
        dequant_e4m3x16(w, sc, lo, hi);
        uint4 *dst = reinterpret_cast<uint4 *>(w16 + off);
        dst[0] = lo;
        dst[1] = hi;
    }
}

}  // namespace gemm

cudaError_t launch_dequant_fp8(const uint8_t *w8, const float *scales, uint16_t *w16, int rows, int cols,
                               int num_sms, cudaStream_t st)
{
    const int64_t total = (int64_t)rows * (cols / 16);
    if (total <= 0)
        return cudaSuccess;
    int64_t blocks = (total + 255) / 256;
    if (blocks > (int64_t)num_sms * 8)
        blocks = (int64_t)num_sms * 8;
    gemm::dequant_fp8_kernel<<<(unsigned)blocks, 256, 0, st>>>(w8, scales, w16, rows, cols);
    return cudaGetLastError();
}

cudaError_t launch_wo_a(const GemmParams &p, int num_sms, cudaStream_t st)
{
    const bool fp8 = p.b_scales != nullptr;
    if (!fp8) {
        // bf16 weights: the two-SM kernel, persistent over as many clusters of
        // two CTAs as can be resident at once (a cluster needs both SMs in one
        // GPC, so that is fewer than half the SMs: a grid of half the SMs
        // would leave a second wave)
        cudaError_t e = cudaFuncSetAttribute(gemm::pair::wo_a_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)gemm::pair::SMEM_BYTES);
        if (e != cudaSuccess)
            return e;
        const int tiles = ((p.M + gemm::pair::BM - 1) / gemm::pair::BM) * (p.R / gemm::pair::BN) * p.G;
        cudaLaunchConfig_t cfg = {};
        cfg.blockDim = dim3(gemm::pair::THREADS);
        cfg.dynamicSmemBytes = gemm::pair::SMEM_BYTES;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        // resident clusters: asked once per device (a host query, nothing enqueued)
        static std::atomic<int> resident_of[64];
        int dev = 0;
        e = cudaGetDevice(&dev);
        if (e != cudaSuccess)
            return e;
        int resident = dev < 64 ? resident_of[dev].load() : 0;
        if (resident <= 0) {
            cfg.gridDim = dim3((unsigned)(num_sms / 2 * 2));
            e = cudaOccupancyMaxActiveClusters(&resident, gemm::pair::wo_a_pair_kernel, &cfg);
            if (e != cudaSuccess)
                return e;
            if (dev < 64)
                resident_of[dev].store(resident);
        }
        int pairs = tiles < resident ? tiles : resident;
        if (pairs <= 0)
            return tiles <= 0 ? cudaSuccess : cudaErrorLaunchOutOfResources;
        cfg.gridDim = dim3((unsigned)(2 * pairs));
        return cudaLaunchKernelEx(&cfg, gemm::pair::wo_a_pair_kernel, p);
    }
    // fp8 weights decoded inside the kernel (fewer than 512 tokens)
    using C = gemm::Cfg;
    cudaError_t e = cudaFuncSetAttribute(gemm::wo_a_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)C::SMEM_BYTES);
    if (e != cudaSuccess)
        return e;
    const int tiles = ((p.M + C::BM - 1) / C::BM) * (p.R / C::BN) * p.G;
    const int grid = tiles < num_sms ? tiles : num_sms;
    if (grid <= 0)
        return cudaSuccess;
    gemm::wo_a_fp8_kernel<<<grid, C::THREADS, C::SMEM_BYTES, st>>>(p);
    return cudaGetLastError();
}

}  // namespace sa
