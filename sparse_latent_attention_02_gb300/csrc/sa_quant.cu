// sa_quant.cu -- fp4 quantization of latent rows for the compressed cache (sm_103a).
//
// The "DeepSeek-V4.1 > 40 layers" page quantizes the compressor's latents with
// `fp4_act_quant(latent, 16, True, scale_dtype=torch.float8_e4m3fn)` before
// they are cached; the function's body is not on the pages.  This kernel
// writes the packed form that the attention kernel's fp4 gather reads:
//   - per group of 16 features an E4M3 scale: the group's largest magnitude
//     over 6 (the largest e2m1 value), divided in fp32 and rounded to the
//     nearest E4M3 value (ties to even, saturating at 448);
//   - per feature an e2m1 code of x / scale (fp32 division): the nearest of
//     0, .5, 1, 1.5, 2, 3, 4, 6 (ties to the even code, saturating at 6), sign
//     in bit 3, kept for results of zero; a scale of zero gives codes of zero
//     with x's sign;
//   - two codes a byte, the even feature in the low nibble.
// Inputs are finite or infinite (a NaN's codes are unspecified).
//
// One thread per group: two 16-byte loads of bf16, eight bytes of codes and
// one scale byte out, so that a warp covers 32 consecutive groups (1 KiB in,
// 288 bytes out for a 512-feature row).
//
// No division per feature: the code of x is the number of the seven halfway
// points t = .25, .75, 1.25, 1.75, 2.5, 3.5, 5 that x / scale passes, and
// "|x| / scale passes t" is decided as "|x| passes t * scale", which is exact
// in fp32 (t has at most three significant bits, the scale four).  The two
// agree for every bf16 x: |x| (eight significant bits) differs from t * scale
// either not at all or by at least 2^-8 of it, far more than the fp32
// rounding of |x| / scale could move.  A halfway value goes to the even code,
// so for t = .25, 1.25, 2.5 and 5 "passes" means strictly above, tested as
// "at least the next bf16 value" (the threshold's bit pattern plus one).
// t * scale is a bf16 value too (seven significant bits at most, inside bf16's
// range), so the tests run on pairs of features as packed bf16 compares, each
// adding 1.0 or 0.0 to a pair of bf16 accumulators that start at 128: there
// the low bits of the pattern are the count itself (128 + c for c <= 7).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sa_internal.h"

namespace sa {
namespace quant {

constexpr int THREADS = 256;

// e2m1 codes of a pair of bf16 features w (the even one in the low half):
// one byte, the even feature's code in the low nibble.  T[k]: threshold k in
// both halves.
__device__ __forceinline__ uint32_t e2m1_pair(uint32_t w, const __nv_bfloat162 (&T)[7])
{
    const uint32_t a = w & 0x7FFF7FFFu;
    const __nv_bfloat162 ab = *reinterpret_cast<const __nv_bfloat162 *>(&a);
    const uint32_t base = 0x43004300u;   // 128.0 in both halves
    __nv_bfloat162 acc = *reinterpret_cast<const __nv_bfloat162 *>(&base);
#pragma unroll
    for (int k = 0; k < 7; ++k)
        acc = __hadd2(acc, __hge2(ab, T[k]));
    const uint32_t cnt = *reinterpret_cast<const uint32_t *>(&acc) & 0x000F000Fu;
    const uint32_t code = cnt | ((w >> 12) & 0x00080008u);   // sign bits 15 and 31 -> 3 and 19
    return (code & 0xFu) | ((code >> 12) & 0xF0u);
}

// nearest E4M3 byte of q >= 0 (hardware conversion: round to nearest even,
// saturating to the largest finite value), and the value it stands for
__device__ __forceinline__ uint32_t e4m3_byte(float q, float &value)
{
    uint16_t pair;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(pair) : "f"(q));
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));
    value = __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
    return pair & 0xFFu;
}

// log2_groups: log2 of the groups a row when that is a power of two (then the
// row and group of a thread come from a shift and a mask), else -1
__global__ void __launch_bounds__(THREADS) fp4_quant_kernel(const uint16_t *__restrict__ latent, int64_t row_stride,
                                                            int64_t rows, int groups, int log2_groups,
                                                            uint8_t *__restrict__ codes, uint8_t *__restrict__ scales)
{
    const int64_t i = (int64_t)blockIdx.x * THREADS + threadIdx.x;   // group over all rows
    if (i >= rows * groups)
        return;
    const int64_t r = log2_groups >= 0 ? i >> log2_groups : i / groups;
    const int g = (int)(i - r * groups);
    const uint4 *src = reinterpret_cast<const uint4 *>(latent + r * row_stride + 16 * g);
    const uint4 w[2] = {__ldg(src), __ldg(src + 1)};
    const uint32_t u[8] = {w[0].x, w[0].y, w[0].z, w[0].w, w[1].x, w[1].y, w[1].z, w[1].w};
    // the group's largest magnitude: a packed maximum over the pairs'
    // magnitudes, then the larger half (non-negative floats order as their bit
    // patterns)
    const uint32_t a0 = u[0] & 0x7FFF7FFFu;
    __nv_bfloat162 m2 = *reinterpret_cast<const __nv_bfloat162 *>(&a0);
#pragma unroll
    for (int j = 1; j < 8; ++j) {
        const uint32_t aj = u[j] & 0x7FFF7FFFu;
        m2 = __hmax2(m2, *reinterpret_cast<const __nv_bfloat162 *>(&aj));
    }
    const uint32_t mm = *reinterpret_cast<const uint32_t *>(&m2);
    const uint32_t amax = max(mm << 16, mm & 0xFFFF0000u);
    float s;
    const uint32_t sb = e4m3_byte(__fdiv_rn(__uint_as_float(amax), 6.0f), s);
    // thresholds t * scale as bf16 in both halves (+1 where a value exactly
    // halfway rounds down)
    const float tv[7] = {0.25f, 0.75f, 1.25f, 1.75f, 2.5f, 3.5f, 5.0f};
    __nv_bfloat162 T[7];
#pragma unroll
    for (int k = 0; k < 7; ++k) {
        const uint32_t h = (__float_as_uint(tv[k] * s) >> 16) + ((k & 1) == 0 ? 1u : 0u);
        const uint32_t hh = h * 0x10001u;
        T[k] = *reinterpret_cast<const __nv_bfloat162 *>(&hh);
    }
    uint32_t c[2] = {0u, 0u};
#pragma unroll
    for (int j = 0; j < 8; ++j)
        c[j >> 2] |= e2m1_pair(u[j], T) << (8 * (j & 3));
    if (!(s > 0.f)) {   // a scale of zero: codes of zero with the features' signs
        c[0] &= 0x88888888u;
        c[1] &= 0x88888888u;
    }
    *reinterpret_cast<uint2 *>(codes + r * (int64_t)(8 * groups) + 8 * g) = make_uint2(c[0], c[1]);
    scales[r * groups + g] = (uint8_t)sb;
}

}  // namespace quant

cudaError_t launch_fp4_quantize(const uint16_t *latent, int64_t row_stride, int64_t rows, int D, uint8_t *codes,
                                uint8_t *scales, cudaStream_t st)
{
    const int groups = D / 16;
    const int64_t total = rows * groups;
    if (total == 0)
        return cudaSuccess;
    int log2_groups = -1;
    if ((groups & (groups - 1)) == 0)
        for (log2_groups = 0; (1 << log2_groups) < groups; ++log2_groups) {
        }
    const int64_t blocks = (total + quant::THREADS - 1) / quant::THREADS;
    quant::fp4_quant_kernel<<<(unsigned)blocks, quant::THREADS, 0, st>>>(latent, row_stride, rows, groups,
                                                                          log2_groups, codes, scales);
    return cudaGetLastError();
}

}  // namespace sa
