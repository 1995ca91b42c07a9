// sa_gemm.cu -- the grouped low-rank output projection `wo_a` for sm_103a.
//
// "DeepSeek-V4.1 > Output projection" page, Attention.forward: the attention
// output viewed as [B, T, G, H*D/G] is multiplied group by group with
// `wo_a.weight.view(G, R, -1)` (`einsum("bsgd,grd->bsgr")`), a block-diagonal
// product -- G independent GEMMs that share one launch:
//   y[m, g*R + r] = sum_d o[m, g*Din + d] * W[g*R + r, d]
//
// Persistent kernel, one CTA per SM.  Tiles of 128 tokens x 256 rank columns,
// K in blocks of 64 features.  Warp 0 feeds a 4-stage shared-memory ring with
// TMA (128-byte swizzle), warp 1 issues tcgen05.mma (M=128, N=256, K=16) into
// one of two TMEM accumulators, warps 2-5 drain the other accumulator to bf16.
#include <cuda_bf16.h>

#include "sa_internal.h"
#include "sa_ptx.cuh"

namespace sa {
namespace gemm {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int THREADS = 192;
constexpr uint32_t A_BYTES = BM * BK * 2;     // 16 KB
constexpr uint32_t B_BYTES = BN * BK * 2;     // 32 KB
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t OFF_BAR = STAGES * STAGE_BYTES;
constexpr uint32_t OFF_MISC = OFF_BAR + 16 * 8;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 64 + 1024;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

enum : uint32_t { B_FULL0 = 0, B_EMPTY0 = STAGES, B_ACCFULL0 = 2 * STAGES, B_ACCEMPTY0 = 2 * STAGES + 2,
                  B_DONE = 2 * STAGES + 4, NUM_BARS };
static_assert(NUM_BARS <= 16, "barrier area");
constexpr uint32_t IDESC = idesc_bf16(BM, BN, 0, 0);

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

__global__ void __launch_bounds__(THREADS, 1) wo_a_kernel(const __grid_constant__ GemmParams p)
{
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
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar0 + 8 * (B_ACCFULL0 + a), 1);
            mbar_init(bar0 + 8 * (B_ACCEMPTY0 + a), 128);
        }
        mbar_init(bar0 + 8 * B_DONE, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&p.tm_a);
        prefetch_tmap(&p.tm_b);
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
                    mbar_arrive_expect_tx(fb, STAGE_BYTES);
                    tma_load_2d(sa_, &p.tm_a, g * p.Din + kb * BK, mb * BM, fb);
                    tma_load_2d(sa_ + A_BYTES, &p.tm_b, kb * BK, g * p.R + nb * BN, fb);
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
                const uint32_t dt = tmem + (uint32_t)(a * BN);
                for (int kb = 0; kb < kblocks; ++kb) {
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
                        mma_bf16_ss(dt, ad, bd, IDESC, (kb > 0 || k > 0) ? 1u : 0u);
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
    } else {
        // ---------------- epilogue: warps 2..5 -> TMEM lane quarters 2,3,0,1
        const int quarter = warp & 3;
        const int row_in_tile = quarter * 32 + lane;
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
            const int m = mb * BM + row_in_tile;
            const uint32_t ta = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(a * BN);
            uint16_t *yrow = p.y + (size_t)m * (p.G * p.R) + g * p.R + nb * BN;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(ta + 32 * c, v);
                tmem_wait_ld();
                if (m < p.M) {
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

}  // namespace gemm

cudaError_t launch_wo_a(const GemmParams &p, int num_sms, cudaStream_t st)
{
    cudaError_t e = cudaFuncSetAttribute(gemm::wo_a_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)gemm::SMEM_BYTES);
    if (e != cudaSuccess)
        return e;
    const int tiles = ((p.M + gemm::BM - 1) / gemm::BM) * (p.R / gemm::BN) * p.G;
    const int grid = tiles < num_sms ? tiles : num_sms;
    if (grid <= 0)
        return cudaSuccess;
    gemm::wo_a_kernel<<<grid, gemm::THREADS, gemm::SMEM_BYTES, st>>>(p);
    return cudaGetLastError();
}

}  // namespace sa
