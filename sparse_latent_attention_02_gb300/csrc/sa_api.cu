// sa_api.cu -- the C ABI of include/sa.h: argument checks, workspace layout,
// tensor-map encoding and kernel launches.  No torch types cross this boundary.
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <cudaTypedefs.h>
#include <atomic>
#include <mutex>

#include "sa_internal.h"

namespace sa {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

// Bound on every device-side wait.  A stage normally waits microseconds; a
// second means the pipeline is stuck.  SA_WAIT_TIMEOUT_MS overrides it.
uint64_t wait_timeout_ns()
{
    static uint64_t ns = [] {
        const char *e = std::getenv("SA_WAIT_TIMEOUT_MS");
        long ms = e ? std::strtol(e, nullptr, 10) : 0;
        if (ms <= 0)
            ms = 1000;
        return (uint64_t)ms * 1000000ull;
    }();
    return ns;
}

// Test hook for failure detection, read once per process: SA_TEST_HOLD_LISTS=n
// makes the first n attention calls of the process withhold their first
// index list, so their bounded waits run out and they report SA_ERR_TIMEOUT
// without faulting or hanging the GPU; later calls run normally.
bool hold_lists()
{
    static const long holds = [] {
        const char *e = std::getenv("SA_TEST_HOLD_LISTS");
        const long n = e ? std::strtol(e, nullptr, 10) : 0;
        return n > 0 ? n : 0L;
    }();
    static std::atomic<long> calls{0};
    return holds > 0 && calls.fetch_add(1) < holds;
}

bool current_sms(int *sms)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return false;
    return cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && *sms > 0;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// kv may live in device (or managed) memory, or in page-locked host memory
// registered with CUDA: then its device address is used and the kernel
// gathers the rows it needs straight from host memory over the CPU-GPU link.
// Anything else (pageable host memory, unknown pointers) is refused here,
// before anything is enqueued.
sa_status resolve_kv(const void *kv, const void **dev_kv, bool *host)
{
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, kv) != cudaSuccess) {
        (void)cudaGetLastError();
        return SA_ERR_INVALID_ARG;
    }
    switch (a.type) {
    case cudaMemoryTypeDevice:
    case cudaMemoryTypeManaged:
        *dev_kv = kv;
        *host = false;
        return SA_OK;
    case cudaMemoryTypeHost:
        if (!a.devicePointer)
            return SA_ERR_INVALID_ARG;
        *dev_kv = a.devicePointer;
        *host = true;
        return SA_OK;
    default:
        return SA_ERR_INVALID_ARG;
    }
}

// The latent rows come from one or two sources (see AttnParams): list index
// v < W is row v of kv (batch stride kv_bstride rows), v >= W is row v - W of
// kv2 (batch stride kv2_bstride rows); N = W + rows of kv2.
struct KvSources {
    const void *kv;
    int64_t kv_bstride;
    int W;
    const void *kv2;
    int64_t kv2_bstride;
    const void *codes = nullptr;    // source 1 in fp4 instead of kv2: e2m1 codes and E4M3 scales
    const void *scales = nullptr;
};

sa_status fill_attn_params(AttnParams &p, const void *q, const KvSources &src, const float *sink,
                           const int32_t *idx, float scale, int B, int T, int N, int K, void *out,
                           bool out_f32, void *ws)
{
    std::memset(&p, 0, sizeof p);
    const uint64_t rows = (uint64_t)B * T * SA_HEADS;
    if (!encode_tmap_2d(&p.tm_q, q, rows, SA_HEAD_DIM, 64, 64))
        return SA_ERR_CUDA;
    const void *dev_kv = src.kv, *dev_kv2 = src.kv2;
    bool host_kv = false, host_kv2 = false;
    if ((int64_t)B * T > 0 && K > 0) {
        if (src.W > 0) {
            const sa_status st = resolve_kv(src.kv, &dev_kv, &host_kv);
            if (st != SA_OK)
                return st;
        }
        if (N > src.W && !src.codes) {
            const sa_status st = resolve_kv(src.kv2, &dev_kv2, &host_kv2);
            if (st != SA_OK)
                return st;
        }
        if (N > src.W && src.codes) {
            const void *c = nullptr, *sc = nullptr;
            bool hc = false, hs = false;
            sa_status st = resolve_kv(src.codes, &c, &hc);
            if (st == SA_OK)
                st = resolve_kv(src.scales, &sc, &hs);
            if (st != SA_OK)
                return st;
            p.kv2_codes = static_cast<const uint8_t *>(c);
            p.kv2_scales = static_cast<const uint8_t *>(sc);
            host_kv2 = hc || hs;
        }
    }
    // warm L2 with upcoming rows only when kv lives in device memory too large
    // to stay resident in L2
    p.prefetch_rows = !host_kv && !host_kv2 && (uint64_t)B * N * SA_HEAD_DIM * 2 > ((uint64_t)96 << 20) ? 1 : 0;
    p.kv = static_cast<const uint16_t *>(dev_kv);
    p.kv2 = static_cast<const uint16_t *>(dev_kv2);
    p.kv_bstride = src.kv_bstride;
    p.kv2_bstride = src.kv2_bstride;
    p.W = src.W;
    p.idx = idx;
    p.sink = sink;
    p.out = out;
    p.err = static_cast<uint32_t *>(ws);
    p.scale_log2 = scale * 1.4426950408889634f;
    p.BT = (int64_t)B * T;
    p.T = T;
    p.N = N;
    p.K = K;
    p.out_f32 = out_f32 ? 1 : 0;
    p.timeout_ns = wait_timeout_ns();
    p.hold_lists = hold_lists() ? 1 : 0;
    return SA_OK;
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// y[m, g*R + r] = sum_d a[m, g*Din + d] * w[g*R + r, d] for m < M (bf16 in and
// out, fp32 accumulation) on the persistent tcgen05 GEMM.  With w_scales, w
// is E4M3 bytes with one fp32 scale per 128 x 128 block, dequantized to bf16
// inside the kernel.
sa_status grouped_gemm(const void *a, const void *w, const float *w_scales, void *y, int64_t M, int G, int R,
                       int Din, void *ws, int sms, cudaStream_t s)
{
    GemmParams g;
    std::memset(&g, 0, sizeof g);
    if (!encode_tmap_2d(&g.tm_a, a, (uint64_t)M, (uint64_t)G * Din, 64, 128))
        return SA_ERR_CUDA;
    if (w_scales ? !encode_tmap_2d_u8(&g.tm_b8, w, (uint64_t)G * R, (uint64_t)Din, 64, 128)
                 : !encode_tmap_2d(&g.tm_b, w, (uint64_t)G * R, (uint64_t)Din, 64, 128))
        return SA_ERR_CUDA;
    g.b_scales = w_scales;
    g.y = static_cast<uint16_t *>(y);
    g.err = static_cast<uint32_t *>(ws);
    g.M = (int)M;
    g.G = G;
    g.R = R;
    g.Din = Din;
    g.timeout_ns = wait_timeout_ns();
    return launch_wo_a(g, sms, s) == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

}  // namespace

// Checks shared by the attention entry points; nothing is enqueued before them.
sa_status check_attn_args(const void *q, const void *kv, const float *sink, const int32_t *idx,
                          float scale, int B, int T, int H, int D, int N, int K, const void *out,
                          const void *ws)
{
    if (B < 0 || T < 0 || H < 0 || D < 0 || N < 0 || K < 0)
        return SA_ERR_INVALID_ARG;
    if (H != SA_HEADS || D != SA_HEAD_DIM || K > SA_MAX_K)
        return SA_ERR_UNSUPPORTED;
    if (!std::isfinite(scale))
        return SA_ERR_INVALID_ARG;
    if (!ws || !aligned(ws, 256))
        return SA_ERR_INVALID_ARG;
    if ((int64_t)B * T == 0)
        return SA_OK;
    if ((int64_t)B * T * H >= (int64_t)1 << 31 || (int64_t)B * N >= (int64_t)1 << 31)
        return SA_ERR_UNSUPPORTED;
    if (!out || !aligned(out, 16))
        return SA_ERR_INVALID_ARG;
    if (K > 0) {
        if (!q || !aligned(q, 16) || !sink || !idx || !aligned(idx, 4))
            return SA_ERR_INVALID_ARG;
        if (N > 0 && (!kv || !aligned(kv, 16)))
            return SA_ERR_INVALID_ARG;
    }
    return SA_OK;
}

sa_status attn_call(const void *q, const void *kv, const float *sink, const int32_t *idx, float scale, int B,
                    int T, int H, int D, int N, int K, void *out, sa_dtype out_dtype, void *workspace,
                    size_t ws_bytes, cudaStream_t s, bool clear_error_word)
{
    sa_status st = check_attn_args(q, kv, sink, idx, scale, B, T, H, D, N, K, out, workspace);
    if (st != SA_OK)
        return st;
    if (out_dtype != SA_BF16 && out_dtype != SA_F32)
        return SA_ERR_INVALID_ARG;
    const int64_t BT = (int64_t)B * T;
    if (BT == 0)
        return SA_OK;
    if (ws_bytes < attn_workspace_bytes(BT, K))
        return SA_ERR_WORKSPACE;
    int sms = 0;
    if (!current_sms(&sms))
        return SA_ERR_CUDA;
    const size_t esz = out_dtype == SA_F32 ? 4 : 2;
    AttnParams p;
    if (K > 0) {
        const KvSources src{kv, N, N, nullptr, 0};
        st = fill_attn_params(p, q, src, sink, idx, scale, B, T, N, K, out, out_dtype == SA_F32, workspace);
        if (st != SA_OK)
            return st;
    }
    // every host check has passed: from here on only enqueueing
    if (clear_error_word && cudaMemsetAsync(workspace, 0, sizeof(uint32_t), s) != cudaSuccess)
        return SA_ERR_CUDA;
    if (K == 0)
        return cudaMemsetAsync(out, 0, (size_t)BT * H * D * esz, s) == cudaSuccess ? SA_OK : SA_ERR_CUDA;
    const Schedule sch = attn_schedule(BT, K, sms);
    return launch_attention(p, sch, s) == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

namespace {

// The driver's cuTensorMapEncodeTiled, looked up once (null if unavailable).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult qr{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}

}  // namespace

bool encode_tmap_2d(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                    uint32_t box_cols, uint32_t box_rows)
{
    const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode)
        return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tmap_2d_u8(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                       uint32_t box_cols, uint32_t box_rows)
{
    const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode)
        return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace sa

using namespace sa;

extern "C" {

size_t sa_sparse_attn_workspace_size(int B, int T, int H, int D, int K)
{
    (void)H;
    (void)D;
    if (B < 0 || T < 0 || K < 0)
        return WS_HEADER;
    return attn_workspace_bytes((int64_t)B * T, K);
}

sa_status sa_sparse_attn(const void *q, const void *kv, const float *sink, const int32_t *idx,
                         float scale, int B, int T, int H, int D, int N, int K, void *out,
                         sa_dtype out_dtype, void *workspace, size_t ws_bytes, void *stream)
{
    return attn_call(q, kv, sink, idx, scale, B, T, H, D, N, K, out, out_dtype, workspace, ws_bytes,
                     static_cast<cudaStream_t>(stream), false);
}

// Shared by the two-source entry points: checks, then one launch.
static sa_status two_source_call(const void *q, const KvSources &src, int C, const float *sink, const int32_t *idx,
                          float scale, int B, int T, int H, int D, int K, void *out, sa_dtype out_dtype,
                          void *workspace, size_t ws_bytes, void *stream)
{
    const int W = src.W;
    if (W < 0 || C < 0 || (int64_t)W + C >= ((int64_t)1 << 31))
        return SA_ERR_INVALID_ARG;
    const int N = W + C;
    const void *any_src = W > 0 ? src.kv : (src.codes ? src.codes : src.kv2);
    sa_status st = check_attn_args(q, any_src, sink, idx, scale, B, T, H, D, N, K, out, workspace);
    if (st != SA_OK)
        return st;
    if (out_dtype != SA_BF16 && out_dtype != SA_F32)
        return SA_ERR_INVALID_ARG;
    const int64_t BT = (int64_t)B * T;
    if (BT == 0)
        return SA_OK;
    if (K > 0) {
        if (W > 0 && (!src.kv || !aligned(src.kv, 16) || src.kv_bstride < W))
            return SA_ERR_INVALID_ARG;
        if (C > 0) {
            if (src.kv2_bstride < C)
                return SA_ERR_INVALID_ARG;
            if (src.codes ? (!aligned(src.codes, 16) || !src.scales) : (!src.kv2 || !aligned(src.kv2, 16)))
                return SA_ERR_INVALID_ARG;
        }
        if ((int64_t)B * (W > 0 ? src.kv_bstride : 0) >= ((int64_t)1 << 40) ||
            (int64_t)B * (C > 0 ? src.kv2_bstride : 0) >= ((int64_t)1 << 40))
            return SA_ERR_UNSUPPORTED;
    }
    if (ws_bytes < attn_workspace_bytes(BT, K))
        return SA_ERR_WORKSPACE;
    int sms = 0;
    if (!current_sms(&sms))
        return SA_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t esz = out_dtype == SA_F32 ? 4 : 2;
    if (K == 0)
        return cudaMemsetAsync(out, 0, (size_t)BT * H * D * esz, s) == cudaSuccess ? SA_OK : SA_ERR_CUDA;
    AttnParams p;
    st = fill_attn_params(p, q, src, sink, idx, scale, B, T, N, K, out, out_dtype == SA_F32, workspace);
    if (st != SA_OK)
        return st;
    const Schedule sch = attn_schedule(BT, K, sms);
    return launch_attention(p, sch, s) == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

sa_status sa_sparse_attn_two_source(const void *q, const void *window_kv, int W, int64_t window_bstride,
                                    const void *compressed_kv, int C, int64_t compressed_bstride,
                                    const float *sink, const int32_t *idx, float scale, int B, int T, int H,
                                    int D, int K, void *out, sa_dtype out_dtype, void *workspace,
                                    size_t ws_bytes, void *stream)
{
    const KvSources src{window_kv, window_bstride, W, compressed_kv, compressed_bstride};
    return two_source_call(q, src, C, sink, idx, scale, B, T, H, D, K, out, out_dtype, workspace, ws_bytes,
                           stream);
}

sa_status sa_sparse_attn_two_source_fp4(const void *q, const void *window_kv, int W, int64_t window_bstride,
                                        const uint8_t *codes, const uint8_t *scales, int C,
                                        int64_t compressed_bstride, const float *sink, const int32_t *idx,
                                        float scale, int B, int T, int H, int D, int K, void *out,
                                        sa_dtype out_dtype, void *workspace, size_t ws_bytes, void *stream)
{
    if (C > 0 && (!codes || !scales))
        return SA_ERR_INVALID_ARG;
    KvSources src{window_kv, window_bstride, W, nullptr, compressed_bstride};
    src.codes = C > 0 ? codes : nullptr;
    src.scales = C > 0 ? scales : nullptr;
    return two_source_call(q, src, C, sink, idx, scale, B, T, H, D, K, out, out_dtype, workspace, ws_bytes,
                           stream);
}

size_t sa_sparse_attn_rope_wo_a_workspace_size(int B, int T, int H, int D, int K, int G, int R)
{
    (void)G;
    (void)R;
    const size_t attn = sa_sparse_attn_workspace_size(B, T, H, D, K);
    if (B < 0 || T < 0 || H < 0 || D < 0)
        return attn;
    return round256(attn) + round256((size_t)B * T * H * D * 2);
}

namespace {

// fp8 wo_a: with at least this many tokens the weight is decoded into a bf16
// workspace copy before a bf16 GEMM; below it the GEMM decodes the weight
// blocks in shared memory (measured on GB300: the GEMM-side decoding is
// faster at 64 and 256 tokens, the copy from 1024 tokens on).
constexpr int64_t FP8_DECODE_FIRST_TOKENS = 512;

// Host checks of the tail arguments.  rope_dim is a multiple of 32 so that
// every warp of the epilogue either rotates all of its 32 features or none.
// fp8 weights (fp8 true): whole 128 x 128 scale blocks and 4-byte aligned scales.
sa_status check_tail_args(int H, int D, const float *rope_cos_sin, int rope_dim, const void *wo_a, int G,
                          int R, bool fp8 = false, const float *wo_a_scales = nullptr)
{
    if (G <= 0 || R <= 0 || rope_dim < 0)
        return SA_ERR_INVALID_ARG;
    if ((H * D) % G != 0 || ((H * D) / G) % 64 != 0 || R % 256 != 0 || rope_dim % 32 != 0 || rope_dim > D)
        return SA_ERR_UNSUPPORTED;
    if (fp8 && ((H * D) / G) % 128 != 0)
        return SA_ERR_UNSUPPORTED;
    if (!wo_a || !aligned(wo_a, 16) || (rope_dim > 0 && !rope_cos_sin))
        return SA_ERR_INVALID_ARG;
    if (fp8 && (!wo_a_scales || !aligned(wo_a_scales, 4)))
        return SA_ERR_INVALID_ARG;
    return SA_OK;
}

// Attention with the inverse RoPE in its epilogue (bf16 o kept in the
// workspace after the attention's own part), then the grouped wo_a into y
// [B*T, G*R] bf16.  Arguments already checked.
sa_status attn_rope_wo_a(const void *q, const void *kv, const float *sink, const int32_t *idx, float scale,
                         int B, int T, int H, int D, int N, int K, const float *rope_cos_sin, int rope_dim,
                         const void *wo_a, const float *wo_a_scales, int G, int R, void *y, void *workspace,
                         size_t attn_ws, int sms, cudaStream_t s)
{
    const int64_t BT = (int64_t)B * T;
    void *o = static_cast<uint8_t *>(workspace) + attn_ws;
    // 1) sparse attention with the inverse rotary embedding fused into its
    //    epilogue, bf16 output kept in the workspace
    if (K == 0) {
        if (cudaMemsetAsync(o, 0, (size_t)BT * H * D * 2, s) != cudaSuccess)
            return SA_ERR_CUDA;
    } else {
        AttnParams p;
        const KvSources src{kv, N, N, nullptr, 0};
        const sa_status st = fill_attn_params(p, q, src, sink, idx, scale, B, T, N, K, o, false, workspace);
        if (st != SA_OK)
            return st;
        p.rope = rope_cos_sin;
        p.rope_dim = rope_dim;
        const Schedule sch = attn_schedule(BT, K, sms);
        if (launch_attention(p, sch, s) != cudaSuccess)
            return SA_ERR_CUDA;
    }
    // 2) grouped wo_a (bf16, or fp8 with block scales)
    return grouped_gemm(o, wo_a, wo_a_scales, y, BT, G, R, H * D / G, workspace, sms, s);
}

}  // namespace

sa_status sa_sparse_attn_rope_wo_a(const void *q, const void *kv, const float *sink,
                                   const int32_t *idx, float scale, int B, int T, int H, int D,
                                   int N, int K, const float *rope_cos_sin, int rope_dim,
                                   const void *wo_a, int G, int R, void *out, void *workspace,
                                   size_t ws_bytes, void *stream)
{
    sa_status st = check_attn_args(q, kv, sink, idx, scale, B, T, H, D, N, K, out, workspace);
    if (st != SA_OK)
        return st;
    const int64_t BT = (int64_t)B * T;
    if (BT == 0)
        return G <= 0 || R <= 0 || rope_dim < 0 ? SA_ERR_INVALID_ARG : SA_OK;
    st = check_tail_args(H, D, rope_cos_sin, rope_dim, wo_a, G, R);
    if (st != SA_OK)
        return st;
    if (BT >= ((int64_t)1 << 31) / 128)
        return SA_ERR_UNSUPPORTED;
    const size_t attn_ws = round256(attn_workspace_bytes(BT, K));
    const size_t o_bytes = round256((size_t)BT * H * D * 2);
    if (ws_bytes < attn_ws + o_bytes)
        return SA_ERR_WORKSPACE;
    int sms = 0;
    if (!current_sms(&sms))
        return SA_ERR_CUDA;
    return attn_rope_wo_a(q, kv, sink, idx, scale, B, T, H, D, N, K, rope_cos_sin, rope_dim, wo_a, nullptr, G, R,
                          out, workspace, attn_ws, sms, static_cast<cudaStream_t>(stream));
}

sa_status sa_sparse_attn_rope_wo_a_fp8(const void *q, const void *kv, const float *sink, const int32_t *idx,
                                       float scale, int B, int T, int H, int D, int N, int K,
                                       const float *rope_cos_sin, int rope_dim, const uint8_t *wo_a_e4m3,
                                       const float *wo_a_scales, int G, int R, void *out, void *workspace,
                                       size_t ws_bytes, void *stream)
{
    sa_status st = check_attn_args(q, kv, sink, idx, scale, B, T, H, D, N, K, out, workspace);
    if (st != SA_OK)
        return st;
    const int64_t BT = (int64_t)B * T;
    if (BT == 0)
        return G <= 0 || R <= 0 || rope_dim < 0 ? SA_ERR_INVALID_ARG : SA_OK;
    st = check_tail_args(H, D, rope_cos_sin, rope_dim, wo_a_e4m3, G, R, true, wo_a_scales);
    if (st != SA_OK)
        return st;
    if (BT >= ((int64_t)1 << 31) / 128)
        return SA_ERR_UNSUPPORTED;
    const size_t attn_ws = round256(attn_workspace_bytes(BT, K));
    const size_t o_bytes = round256((size_t)BT * H * D * 2);
    const bool decode_first = BT >= FP8_DECODE_FIRST_TOKENS;
    const size_t w_bytes = decode_first ? round256((size_t)R * H * D * 2) : 0;   // bf16 copy of wo_a
    if (ws_bytes < attn_ws + o_bytes + w_bytes)
        return SA_ERR_WORKSPACE;
    int sms = 0;
    if (!current_sms(&sms))
        return SA_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (!decode_first)   // few tokens: the GEMM decodes the weight blocks itself
        return attn_rope_wo_a(q, kv, sink, idx, scale, B, T, H, D, N, K, rope_cos_sin, rope_dim, wo_a_e4m3,
                              wo_a_scales, G, R, out, workspace, attn_ws, sms, s);
    // many tokens: the weight is decoded once into a bf16 copy in the workspace
    // (one bandwidth-bound pass) and the grouped GEMM runs on bf16 operands
    uint16_t *w16 = reinterpret_cast<uint16_t *>(static_cast<uint8_t *>(workspace) + attn_ws + o_bytes);
    if (launch_dequant_fp8(wo_a_e4m3, wo_a_scales, w16, G * R, H * D / G, sms, s) != cudaSuccess)
        return SA_ERR_CUDA;
    return attn_rope_wo_a(q, kv, sink, idx, scale, B, T, H, D, N, K, rope_cos_sin, rope_dim, w16, nullptr, G, R,
                          out, workspace, attn_ws, sms, s);
}

size_t sa_sparse_attn_rope_wo_a_fp8_workspace_size(int B, int T, int H, int D, int K, int G, int R)
{
    const size_t fused = sa_sparse_attn_rope_wo_a_workspace_size(B, T, H, D, K, G, R);
    if (B < 0 || T < 0 || H < 0 || D < 0 || R < 0 || (int64_t)B * T < FP8_DECODE_FIRST_TOKENS)
        return fused;
    return round256(fused) + round256((size_t)R * H * D * 2);
}

size_t sa_sparse_attn_block_tail_workspace_size(int B, int T, int H, int D, int K, int G, int R)
{
    const size_t fused = sa_sparse_attn_rope_wo_a_workspace_size(B, T, H, D, K, G, R);
    if (B < 0 || T < 0 || G < 0 || R < 0)
        return fused;
    return round256(fused) + round256((size_t)B * T * G * R * 2);
}

sa_status sa_sparse_attn_block_tail(const void *q, const void *kv, const float *sink, const int32_t *idx,
                                    float scale, int B, int T, int H, int D, int N, int K,
                                    const float *rope_cos_sin, int rope_dim, const void *wo_a, int G, int R,
                                    const void *wo_b, int dim, void *out, void *workspace, size_t ws_bytes,
                                    void *stream)
{
    sa_status st = check_attn_args(q, kv, sink, idx, scale, B, T, H, D, N, K, out, workspace);
    if (st != SA_OK)
        return st;
    const int64_t BT = (int64_t)B * T;
    if (BT == 0)
        return G <= 0 || R <= 0 || rope_dim < 0 || dim <= 0 ? SA_ERR_INVALID_ARG : SA_OK;
    st = check_tail_args(H, D, rope_cos_sin, rope_dim, wo_a, G, R);
    if (st != SA_OK)
        return st;
    if (dim <= 0)
        return SA_ERR_INVALID_ARG;
    if (dim % 256 != 0 || ((int64_t)G * R) % 64 != 0)
        return SA_ERR_UNSUPPORTED;
    if (!wo_b || !aligned(wo_b, 16))
        return SA_ERR_INVALID_ARG;
    if (BT >= ((int64_t)1 << 31) / 128)
        return SA_ERR_UNSUPPORTED;
    const size_t attn_ws = round256(attn_workspace_bytes(BT, K));
    const size_t o_bytes = round256((size_t)BT * H * D * 2);
    const size_t y_bytes = round256((size_t)BT * G * R * 2);
    if (ws_bytes < attn_ws + o_bytes + y_bytes)
        return SA_ERR_WORKSPACE;
    int sms = 0;
    if (!current_sms(&sms))
        return SA_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void *y = static_cast<uint8_t *>(workspace) + attn_ws + o_bytes;
    st = attn_rope_wo_a(q, kv, sink, idx, scale, B, T, H, D, N, K, rope_cos_sin, rope_dim, wo_a, nullptr, G, R,
                        y, workspace, attn_ws, sms, s);
    if (st != SA_OK)
        return st;
    // 3) wo_b: one dense [dim, G*R] projection of the flattened groups
    return grouped_gemm(y, wo_b, nullptr, out, BT, 1, dim, G * R, workspace, sms, s);
}

sa_status sa_topk_indices(const float *scores, int64_t row_stride, int64_t rows, int L, int k, int offset,
                          int32_t *out, void *stream)
{
    if (rows < 0 || L < 0 || k < 0 || row_stride < L || rows >= ((int64_t)1 << 31))
        return SA_ERR_INVALID_ARG;
    if ((int64_t)L + offset >= ((int64_t)1 << 31) || offset < 0)
        return SA_ERR_INVALID_ARG;
    if (rows == 0 || k == 0)
        return SA_OK;
    if (!out || !aligned(out, 4) || (L > 0 && (!scores || !aligned(scores, 4))))
        return SA_ERR_INVALID_ARG;
    return launch_topk(scores, row_stride, rows, L, k, offset, out, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? SA_OK
               : SA_ERR_CUDA;
}

sa_status sa_fp4_quantize(const void *latent, int64_t rows, int64_t row_stride, int D, uint8_t *codes,
                          uint8_t *scales, void *stream)
{
    if (rows < 0 || D <= 0 || D % 16 != 0 || row_stride < D || row_stride % 8 != 0)
        return SA_ERR_INVALID_ARG;
    if (rows > ((int64_t)1 << 31) * 256 / (D / 16) - 1)
        return SA_ERR_INVALID_ARG;
    if (rows == 0)
        return SA_OK;
    if (!latent || !codes || !scales || !aligned(latent, 16) || !aligned(codes, 8))
        return SA_ERR_INVALID_ARG;
    return launch_fp4_quantize(static_cast<const uint16_t *>(latent), row_stride, rows, D, codes, scales,
                               static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? SA_OK
               : SA_ERR_CUDA;
}

sa_status sa_rope_table(double theta, int start_pos, int T, int rope_dim, float *cos_sin_host)
{
    if (T < 0 || rope_dim <= 0 || rope_dim % 2 != 0 || !(theta > 0.0) || start_pos < 0)
        return SA_ERR_INVALID_ARG;
    if (T > 0 && !cos_sin_host)
        return SA_ERR_INVALID_ARG;
    const int half = rope_dim / 2;
    for (int t = 0; t < T; ++t) {
        const double pos = (double)start_pos + t;
        for (int i = 0; i < half; ++i) {
            const double ang = pos * std::pow(theta, -2.0 * i / rope_dim);
            cos_sin_host[((size_t)t * half + i) * 2] = (float)std::cos(ang);
            cos_sin_host[((size_t)t * half + i) * 2 + 1] = (float)std::sin(ang);
        }
    }
    return SA_OK;
}

sa_status sa_check_errors(void *workspace, void *stream)
{
    if (!workspace)
        return SA_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return SA_ERR_CUDA;
    uint32_t w = 0;
    if (cudaMemcpy(&w, workspace, sizeof w, cudaMemcpyDeviceToHost) != cudaSuccess)
        return SA_ERR_CUDA;
    if (w) {
        const uint32_t z = 0;
        if (cudaMemcpy(workspace, &z, sizeof z, cudaMemcpyHostToDevice) != cudaSuccess)
            return SA_ERR_CUDA;
    }
    if (w & ERRBIT_BOUNDS)
        return SA_ERR_BOUNDS;
    if (w & ERRBIT_TIMEOUT)
        return SA_ERR_TIMEOUT;
    if (w & ERRBIT_INDEX)
        return SA_ERR_INDEX;
    return SA_OK;
}

const char *sa_status_string(sa_status s)
{
    switch (s) {
    case SA_OK: return "ok";
    case SA_ERR_INVALID_ARG: return "invalid argument (null, negative or misaligned)";
    case SA_ERR_UNSUPPORTED: return "shape outside the supported fast path";
    case SA_ERR_WORKSPACE: return "workspace too small";
    case SA_ERR_INDEX: return "an index outside [-1, N) was seen and skipped";
    case SA_ERR_TIMEOUT: return "a bounded device wait ran out";
    case SA_ERR_CUDA: return "CUDA runtime or driver error";
    case SA_ERR_BOUNDS: return "an address check of the checked build failed; the access was skipped";
    }
    return "unknown status";
}

}  // extern "C"
