// sa_internal.h -- declarations shared by the library's translation units.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/sa.h"

namespace sa {

// Bits of the device error word (first 4 bytes of every workspace).
constexpr uint32_t ERRBIT_INDEX = 1u;
constexpr uint32_t ERRBIT_TIMEOUT = 2u;
constexpr uint32_t ERRBIT_BOUNDS = 4u;   // checked build: an address check failed

#ifdef __CUDACC__
// The checked build (compiled with SA_CHECKED) tests the addresses the
// kernels compute from run-time values before it uses them: a failed test
// sets ERRBIT_BOUNDS in the error word and the caller skips the access.  In
// the normal build the test compiles away.
__device__ __forceinline__ bool in_bounds(bool ok, uint32_t *err)
{
#ifdef SA_CHECKED
    if (!ok)
        atomicOr(err, ERRBIT_BOUNDS);
    return ok;
#else
    (void)ok;
    (void)err;
    return true;
#endif
}

// [p, p + bytes) lies inside [base, base + extent)
__device__ __forceinline__ bool inside(const void *p, size_t bytes, const void *base, size_t extent)
{
    const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(base);
    return a >= b && a - b <= extent && bytes <= extent - (a - b);
}
#endif

// Workspace layout of the attention call: [0, 256) header (error word).
constexpr size_t WS_HEADER = 256;

struct AttnParams {
    CUtensorMap tm_q;          // q as 2-D [B*T*H rows, D cols] bf16, box 64x64, 128B swizzle
    // latent rows, bf16 [.., D], device memory or page-locked host memory: list
    // index v < W is row v of source 0, index v >= W is row v - W of source 1
    // (one source: W = N); each source has its own batch stride, in rows
    const uint16_t *kv;
    const uint16_t *kv2;
    int64_t kv_bstride, kv2_bstride;
    int W;
    // source 1 in fp4 instead (kv2 unused): per row D/2 bytes of e2m1 codes
    // and D/16 E4M3 scales, same batch stride in rows
    const uint8_t *kv2_codes;
    const uint8_t *kv2_scales;
    const int32_t *idx;        // int32 [B*T, K]
    const float *sink;         // fp32 [H]
    void *out;                 // [B*T, H, D] bf16 or fp32
    uint32_t *err;             // error word (workspace)
    const float *rope;         // fp32 [T, rope_dim/2, 2] or null
    float scale_log2;          // softmax scale * log2(e)
    int64_t BT;                // B * T
    int T, N, K;
    int out_f32;
    int split;                 // 0: whole queries, CTA i takes i, i+grid, ...; 1: list pieces
    int64_t per_cta;           // split: list entries per piece (the last piece may be shorter)
    int pieces;                // split: pieces per query (2, 4 or 8), one cluster per query;
                               // CTA c takes piece c % pieces of query c / pieces
    int rope_dim;              // 0 = no rotary epilogue
    int prefetch_rows;         // 1: warm L2 with the next segment's rows (kv larger than L2)
    int hold_lists;            // failure-detection test hook: never publish the first index list
    uint64_t timeout_ns;       // bound on every device-side wait
};

struct Schedule {
    int grid;
    int split;
    int64_t per_cta;
    int pieces;
};

// Decide the grid and the split of the index lists for this shape and device.
Schedule attn_schedule(int64_t BT, int K, int num_sms);
// Workspace bytes of the attention call (a function of the shape only, so that
// a short workspace is refused before any CUDA call).
size_t attn_workspace_bytes(int64_t BT, int K);

// Enqueue the attention kernel (a cluster launch in the split schedule).
cudaError_t launch_attention(AttnParams &p, const Schedule &s, cudaStream_t st);

struct GemmParams {
    CUtensorMap tm_a;          // o as 2-D [M rows, G*Din cols] bf16, box 64x128
    CUtensorMap tm_b;          // W as 2-D [G*R rows, Din cols] bf16, box 64x128 (one CTA's half of a tile)
    CUtensorMap tm_b8;         // fp8 W: E4M3 bytes [G*R rows, Din cols], box 64x128, no swizzle
    const float *b_scales;     // fp8 W: fp32 [G*R/128, Din/128] block scales; null for bf16 W
    uint16_t *y;               // bf16 [M, G*R]
    uint32_t *err;
    int M, G, R, Din;
    uint64_t timeout_ns;
};

cudaError_t launch_wo_a(const GemmParams &p, int num_sms, cudaStream_t st);
// E4M3 weight [rows, cols] + fp32 128 x 128 block scales -> bf16 [rows, cols].
cudaError_t launch_dequant_fp8(const uint8_t *w8, const float *scales, uint16_t *w16, int rows, int cols,
                               int num_sms, cudaStream_t st);

// fp4 codes and E4M3 group scales of bf16 latent rows (see sa_fp4_quantize).
cudaError_t launch_fp4_quantize(const uint16_t *latent, int64_t row_stride, int64_t rows, int D, uint8_t *codes,
                                uint8_t *scales, cudaStream_t st);

// Top-k selection of positions per row of scores (see sa_topk_indices).
cudaError_t launch_topk(const float *scores, int64_t row_stride, int64_t rows, int L, int k, int offset,
                        int32_t *out, cudaStream_t st);

// The one-source attention call (sa_sparse_attn) with every host check done
// before anything is enqueued; with clear_error_word, the workspace's 4-byte
// error word is zeroed on the stream after the checks, right before the
// launch (for callers whose scratch keeps an earlier call's contents).
sa_status attn_call(const void *q, const void *kv, const float *sink, const int32_t *idx, float scale, int B,
                    int T, int H, int D, int N, int K, void *out, sa_dtype out_dtype, void *workspace,
                    size_t ws_bytes, cudaStream_t stream, bool clear_error_word);

// Host argument checks of the attention entry points (no CUDA call).
sa_status check_attn_args(const void *q, const void *kv, const float *sink, const int32_t *idx,
                          float scale, int B, int T, int H, int D, int N, int K, const void *out,
                          const void *ws);

// Encode a 2-D bf16 tensor map (row-major [rows, cols], 128B swizzle).
bool encode_tmap_2d(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                    uint32_t box_cols, uint32_t box_rows);
// Encode a 2-D byte tensor map (row-major [rows, cols], no swizzle).
bool encode_tmap_2d_u8(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                       uint32_t box_cols, uint32_t box_rows);

}  // namespace sa
