/*
 * sa.h -- C ABI of the GB300 (sm_103a) sparse latent attention library.
 *
 * The operation is the `sparse_attn(q, kv, attn_sink, topk_idxs,
 * softmax_scale)` step of DeepSeek-V4.1's attention, as called in the
 * `Attention.forward` excerpt of the "DeepSeek-V4.1 > Output projection" page,
 * together with the two steps that follow it there: the inverse rotary
 * embedding of the last rope_head_dim output features and the block-diagonal
 * grouped projection `einsum("bsgd,grd->bsgr", o, wo_a)`.
 *
 * For every query (b, t) and head h, with S the list entries idx[b,t,j] != -1:
 *   s_j    = scale * <q[b,t,h,:], kv[b, idx_j, :]>
 *   M      = max(sink[h], max_j s_j)
 *   o[h,:] = sum_j e^(s_j - M) kv[b, idx_j, :] / (e^(sink[h] - M) + sum_j e^(s_j - M))
 * All heads share the gathered latent rows, which serve as both keys and
 * values.  The sink is one extra logit per head with no value row and is not
 * multiplied by the scale.  An entry of -1 contributes nothing wherever it
 * sits in the list; any other listed entry contributes one term (a repeated
 * index counts twice).  An empty list gives o = 0.
 *
 * Conventions for every entry point:
 *   - Device pointers name memory on the current CUDA device; the caller owns
 *     all of it.  The library keeps no per-call state and allocates nothing.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  All work
 *     is enqueued asynchronously on it; host-detectable argument errors return
 *     before anything is enqueued.
 *   - Device-detected problems (an index outside [-1, N), a bounded internal
 *     wait that ran out) are OR-ed into an error word at the start of the
 *     workspace; `sa_check_errors` synchronises the stream, reads and clears
 *     it.  The kernels never trap: a bad index is skipped.
 *   - The workspace must be zero-filled before its first use (the error word
 *     and internal counters start at zero); the library leaves it reusable.
 *     Two calls that share a workspace must not run concurrently.
 *   - Fast path only: H == 64 heads, D == 512 features; other shapes return
 *     SA_ERR_UNSUPPORTED.  1 <= K <= SA_MAX_K, or K == 0 (all-zero output).
 *   - The library is also built with address checks in its kernels
 *     (libsa_checked.so, this same ABI): every address a kernel computes from
 *     run-time values is tested before use, and a failed test skips the
 *     access and sets the error word's bounds bit (SA_ERR_BOUNDS).
 */
#ifndef SA_H_
#define SA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SA_OK = 0,
    SA_ERR_INVALID_ARG = 1,   /* null pointer, negative size, misaligned pointer */
    SA_ERR_UNSUPPORTED = 2,   /* shape outside the fast path (H, D, K, rope_dim, G, R) */
    SA_ERR_WORKSPACE = 3,     /* workspace smaller than the *_workspace_size query */
    SA_ERR_INDEX = 4,         /* device saw an index outside [-1, N); it was skipped */
    SA_ERR_TIMEOUT = 5,       /* a bounded device wait ran out; outputs are invalid */
    SA_ERR_CUDA = 6,          /* a CUDA runtime/driver call failed (no device, launch error) */
    SA_ERR_BOUNDS = 7         /* checked build only: an address check failed and the access was
                                 skipped; outputs are invalid */
} sa_status;

typedef enum { SA_BF16 = 0, SA_F32 = 1 } sa_dtype;

#define SA_HEADS 64
#define SA_HEAD_DIM 512
#define SA_MAX_K 1024

/*
 * Bytes of workspace `sa_sparse_attn` needs for this shape on the current
 * device.  Always a multiple of 256 and at least 256 (the error word); the
 * size may depend on the shape and on the device's SM count, so query it
 * rather than assuming the minimum.
 */
size_t sa_sparse_attn_workspace_size(int B, int T, int H, int D, int K);

/*
 * sparse_attn ("DeepSeek-V4.1 > Output projection" page, Attention.forward).
 *   q      bf16 [B, T, H, D] contiguous, 16-byte aligned
 *   kv     bf16 [B, N, D] contiguous, 16-byte aligned: per batch row the
 *          window ring rows followed by the compressed rows.  Device memory,
 *          or page-locked host memory registered with CUDA (cudaHostAlloc,
 *          cudaHostRegister): then the kernel gathers only the rows the
 *          lists name straight from host memory over the CPU-GPU link, and
 *          the rest of kv never moves.  Any other pointer (pageable host
 *          memory, unknown) returns SA_ERR_INVALID_ARG before anything is
 *          enqueued.  Every other buffer is device memory.
 *   sink   fp32 [H]
 *   idx    int32 [B, T, K] contiguous; values in [0, N) or -1 (skip)
 *   scale  softmax scale applied to q.k (the pages use D ** -0.5)
 *   out    [B, T, H, D] contiguous, 16-byte aligned, bf16 or fp32 (out_dtype)
 *   workspace / ws_bytes: device scratch, 256-byte aligned, zeroed once
 * Returns SA_OK once the work is enqueued.
 */
sa_status sa_sparse_attn(const void *q, const void *kv, const float *sink,
                         const int32_t *idx, float scale, int B, int T, int H,
                         int D, int N, int K, void *out, sa_dtype out_dtype,
                         void *workspace, size_t ws_bytes, void *stream);

/*
 * sa_sparse_attn over the two latent sources of the "DeepSeek-V4.1 > Output
 * projection" page's Attention.forward without concatenating them: the
 * window ring (`window_kv_cache`, [max_batch, window, D]) and the compressed
 * cache (`compress_kv_cache`, [max_batch, max_len / ratio, D]) that the page
 * joins with torch.cat before calling sparse_attn.  The result is the same
 * as sa_sparse_attn on kv = cat(window[:, :W], compressed[:, :C]) with N = W + C.
 *   window_kv      bf16, row v < W of batch element b at
 *                  window_kv + (b * window_bstride + v) * D; rows 16-byte aligned
 *   W              rows of the window source per batch element (>= 0)
 *   window_bstride batch stride of the window source, in rows (>= W)
 *   compressed_kv  bf16, list index v >= W reads its row v - W of batch
 *                  element b at compressed_kv + (b * compressed_bstride + v - W) * D
 *   C, compressed_bstride  as for the window source
 *   idx            int32 [B, T, K]; values in [0, W + C) or -1 (skip)
 * Each source may be device memory or page-locked host memory (as kv of
 * sa_sparse_attn); an unused source (W or C zero) may be NULL.  Other
 * arguments, workspace and errors as for sa_sparse_attn.  Rows of a source
 * beyond W or C (padding of a cache) are never read.
 */
sa_status sa_sparse_attn_two_source(const void *q, const void *window_kv, int W,
                                    int64_t window_bstride, const void *compressed_kv,
                                    int C, int64_t compressed_bstride, const float *sink,
                                    const int32_t *idx, float scale, int B, int T, int H,
                                    int D, int K, void *out, sa_dtype out_dtype,
                                    void *workspace, size_t ws_bytes, void *stream);

/*
 * sa_sparse_attn_two_source with the compressed cache stored as fp4: the
 * "DeepSeek-V4.1 > 40 layers" page quantizes each compressed latent to fp4 in
 * groups of 16 with an E4M3 scale per group (`fp4_act_quant(latent, 16, True,
 * scale_dtype=torch.float8_e4m3fn)`) before caching it, so its values lie on
 * that grid and this packed form holds them exactly in 288 bytes per row
 * instead of 1024.  The kernel decodes each gathered row into bf16 in shared
 * memory; the result is the same as sa_sparse_attn_two_source on the decoded
 * cache.
 *   codes  uint8, row v - W of batch element b at codes + (b * compressed_bstride
 *          + v - W) * D/2: byte i holds feature 2i in its low nibble and 2i+1 in
 *          its high nibble, each an e2m1 code (bit 3 sign, bits 2..0 index the
 *          magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6); 16-byte aligned
 *   scales uint8, at scales + (b * compressed_bstride + v - W) * D/16 + g: the
 *          E4M3 scale (bias 7, no infinities, S.1111.111 = NaN) of features
 *          16g .. 16g+15
 *   compressed_bstride  batch stride of both, in rows (>= C)
 * Other arguments as for sa_sparse_attn_two_source; the window source stays bf16.
 */
sa_status sa_sparse_attn_two_source_fp4(const void *q, const void *window_kv, int W,
                                        int64_t window_bstride, const uint8_t *codes,
                                        const uint8_t *scales, int C,
                                        int64_t compressed_bstride, const float *sink,
                                        const int32_t *idx, float scale, int B, int T,
                                        int H, int D, int K, void *out, sa_dtype out_dtype,
                                        void *workspace, size_t ws_bytes, void *stream);

/*
 * Bytes of workspace `sa_sparse_attn_rope_wo_a` needs: the attention
 * workspace plus the bf16 attention output [B, T, H, D] it keeps between the
 * two steps.
 */
size_t sa_sparse_attn_rope_wo_a_workspace_size(int B, int T, int H, int D, int K,
                                               int G, int R);

/*
 * sparse_attn, then the inverse rotary embedding of the last rope_dim
 * features of every head (`apply_rotary_emb(o[..., -rd:], freqs_cis, True)`),
 * then the grouped projection (`o.view(B, T, G, -1)` einsum
 * `wo_a.weight.view(G, R, -1)`), all from the same page's Attention.forward.
 *   (q, kv, sink, idx, scale, B, T, H, D, N, K) as for sa_sparse_attn
 *   rope_cos_sin fp32 [T, rope_dim/2, 2]: row t holds (cos, sin) of
 *          pos_t * w_i for the frequency pairs i of query t (same for every
 *          batch row; see sa_rope_table).  Feature pair i is (D - rope_dim + 2i,
 *          D - rope_dim + 2i + 1), rotated as one complex number by -pos_t*w_i.
 *   rope_dim 64 (a multiple of 32, <= D)
 *   wo_a   bf16 [G, R, H*D/G] contiguous, 16-byte aligned ([out, in] per group)
 *   G, R   8 groups x 1024 rank on the fast path
 *   out    bf16 [B, T, G*R] contiguous, 16-byte aligned
 */
sa_status sa_sparse_attn_rope_wo_a(const void *q, const void *kv, const float *sink,
                                   const int32_t *idx, float scale, int B, int T,
                                   int H, int D, int N, int K,
                                   const float *rope_cos_sin, int rope_dim,
                                   const void *wo_a, int G, int R, void *out,
                                   void *workspace, size_t ws_bytes, void *stream);

/*
 * sa_sparse_attn_rope_wo_a with the grouped weight kept in fp8 (the same
 * page: the checkpoint's wo_a is fp8, its conversion dequantizes it to bf16,
 * and an fp8 grouped GEMM would halve the weight's memory).  The kernel reads
 * the E4M3 bytes and dequantizes them in shared memory to exactly the bf16
 * weight that conversion gives, so the result equals sa_sparse_attn_rope_wo_a
 * on that bf16 weight:
 *   W[n, d] = bf16(fp32(e4m3(wo_a_e4m3[n, d]) * wo_a_scales[n / 128, d / 128]))
 * (n = g*R + r; the product rounded to fp32, then to bf16, both to nearest
 * even).  The pages do not give the scale layout; one fp32 scale per
 * 128 x 128 block is taken.
 *   (q ... rope_dim, G, R, out) as for sa_sparse_attn_rope_wo_a
 *   wo_a_e4m3   E4M3 bytes [G, R, H*D/G] contiguous, 16-byte aligned
 *   wo_a_scales fp32 [G*R/128, H*D/G/128] contiguous, 4-byte aligned
 *   workspace   sa_sparse_attn_rope_wo_a_fp8_workspace_size bytes: the fused
 *          call's workspace, plus, with B*T >= 512 tokens, the bf16 copy of
 *          the weight (R*H*D*2 bytes) that the call decodes into before a
 *          bf16 grouped GEMM; with fewer tokens the GEMM decodes the weight
 *          blocks in shared memory (no copy).  The result is the same.
 * H*D/G must be a multiple of 128 (SA_ERR_UNSUPPORTED otherwise).
 */
size_t sa_sparse_attn_rope_wo_a_fp8_workspace_size(int B, int T, int H, int D, int K,
                                                   int G, int R);

sa_status sa_sparse_attn_rope_wo_a_fp8(const void *q, const void *kv, const float *sink,
                                       const int32_t *idx, float scale, int B, int T,
                                       int H, int D, int N, int K,
                                       const float *rope_cos_sin, int rope_dim,
                                       const uint8_t *wo_a_e4m3, const float *wo_a_scales,
                                       int G, int R, void *out, void *workspace,
                                       size_t ws_bytes, void *stream);

/*
 * Bytes of workspace `sa_sparse_attn_block_tail` needs: the fused call's
 * workspace plus the bf16 wo_a output [B, T, G*R] kept between the GEMMs.
 */
size_t sa_sparse_attn_block_tail_workspace_size(int B, int T, int H, int D, int K,
                                                int G, int R);

/*
 * The whole tail of the same page's Attention.forward: sa_sparse_attn_rope_wo_a,
 * then `x = self.wo_b(o.flatten(2))` -- the "Output projection" page's wo_b,
 * a linear map of the G*R = 8192 group features to the model width (5120)
 * without bias, weight stored [out, in] like every module of the page.  On one
 * GPU its row-parallel all-reduce is the identity.
 *   (q ... R) as for sa_sparse_attn_rope_wo_a
 *   wo_b   bf16 [dim, G*R] contiguous, 16-byte aligned
 *   dim    model width, a multiple of 256 (5120)
 *   out    bf16 [B, T, dim] contiguous, 16-byte aligned
 * The wo_a output is rounded to bf16 between the two products, as the page's
 * bf16 einsum does.
 */
sa_status sa_sparse_attn_block_tail(const void *q, const void *kv, const float *sink,
                                    const int32_t *idx, float scale, int B, int T, int H,
                                    int D, int N, int K, const float *rope_cos_sin,
                                    int rope_dim, const void *wo_a, int G, int R,
                                    const void *wo_b, int dim, void *out, void *workspace,
                                    size_t ws_bytes, void *stream);

/*
 * Top-k selection of compressed positions, the step that produces the
 * compressed part of the index lists (the "DeepSeek-V4.1 > 40 layers" page's
 * `_compress_topk_idxs`: the indexer returns int32 positions, `index_topk` =
 * 512 of them, offset by the window length `kv.size(1)`).  The indexer's
 * scoring is not on the pages; this is the selection over given scores:
 *   scores fp32, row r at scores + r * row_stride, L positions per row;
 *          a score of -inf or NaN marks a position that may not be chosen
 *   out    int32 [rows, k]: the positions of the k largest scores (ties to
 *          the smaller position), in ascending order, each plus `offset`;
 *          -1 after them when a row has fewer than k positions to choose
 * Device memory; asynchronous on `stream`.  SA_ERR_INVALID_ARG for negative
 * sizes, row_stride < L, offset < 0 or null / misaligned (4-byte) pointers.
 */
sa_status sa_topk_indices(const float *scores, int64_t row_stride, int64_t rows, int L,
                          int k, int offset, int32_t *out, void *stream);

/*
 * fp4 quantization of latent rows into the compressed-cache layout that
 * sa_sparse_attn_two_source_fp4 reads: the "DeepSeek-V4.1 > 40 layers" page,
 * `_compress_kv`, `fp4_act_quant(latent, 16, True,
 * scale_dtype=torch.float8_e4m3fn)` (its body is not on the pages; this is the
 * library's reading).  Per group of 16 features: scale = E4M3(amax / 6), amax
 * the group's largest magnitude, 6 the largest e2m1 value, the division in
 * fp32, rounded to the nearest E4M3 value (ties to even, saturating at 448);
 * each feature's code = e2m1(x / scale) (fp32 division), the nearest of
 * 0, .5, 1, 1.5, 2, 3, 4, 6 (ties to the even code, saturating at 6), sign in
 * bit 3 (kept for results of zero); a scale of zero gives codes of zero with
 * x's sign.  The decoded value code * scale is what the cache then holds.
 *
 *   latent      bf16 [rows, D] in device memory, row i at latent + i*row_stride
 *               elements; 16-byte aligned, row_stride a multiple of 8 and >= D;
 *               finite or infinite values (a NaN's codes are unspecified)
 *   D           features per row, a positive multiple of 16
 *   codes       uint8 [rows, D/2] contiguous, 8-byte aligned: byte j holds
 *               features 2j (low nibble) and 2j+1 (high nibble)
 *   scales      uint8 [rows, D/16] contiguous: the E4M3 scale of features
 *               16g .. 16g+15
 *
 * Device memory; asynchronous on `stream`.  SA_ERR_INVALID_ARG for bad sizes,
 * null or misaligned pointers (before anything is enqueued).  rows == 0 is a
 * no-op.
 */
sa_status sa_fp4_quantize(const void *latent, int64_t rows, int64_t row_stride, int D,
                          uint8_t *codes, uint8_t *scales, void *stream);

/*
 * Host helper: fill cos_sin_host fp32 [T, rope_dim/2, 2] with
 * (cos, sin)((start_pos + t) * theta ** (-2i / rope_dim)), computed in double.
 * This is the precomputed rotary table of Attention.__init__ (plain theta, no
 * long-context frequency correction).  Returns SA_ERR_INVALID_ARG on bad sizes.
 */
sa_status sa_rope_table(double theta, int start_pos, int T, int rope_dim,
                        float *cos_sin_host);

/*
 * sa_sparse_attn without a workspace argument, for callers that cannot
 * allocate device memory where they run attention (an allocator or memory-pool
 * callback, a plugin whose host framework owns every device allocation, a
 * real-time loop that must not enter the driver's allocator).  The pages have
 * no counterpart: this is a convenience of this library.
 *
 * The scratch is a 64 KiB array in the library's device image: every process
 * that loads the library holds it on every GPU it uses, until exit.  Shapes
 * whose scratch (sa_sparse_attn_workspace_size) exceeds 64 KiB return
 * SA_ERR_WORKSPACE before anything is enqueued; every shape sa_sparse_attn
 * accepts needs 256 bytes.  Nothing is allocated: no cudaMalloc, no
 * cudaFree, no allocating library routine.
 *
 * The first call on a device looks up the array's device address (with that
 * device current) and caches it for the life of the process; make that first
 * call before any stream capture.  The cached address does not survive
 * cudaDeviceReset on that device.  All calls share the one array and it keeps
 * the last call's contents: each call zeroes its error word (enqueued on
 * `stream` after every host check has passed, right before the kernel), so
 * calls whose work overlaps on the GPU race and must not be issued on
 * different streams at the same time.
 *
 * Arguments as for sa_sparse_attn, without workspace/ws_bytes.  If scratch_out
 * is not NULL it receives the array's device address; pass it to
 * sa_check_errors to read this call's device-side error report.
 */
sa_status sa_sparse_attn_noalloc(const void *q, const void *kv, const float *sink,
                                 const int32_t *idx, float scale, int B, int T, int H,
                                 int D, int N, int K, void *out, sa_dtype out_dtype,
                                 void **scratch_out, void *stream);

/*
 * Synchronise `stream`, read the workspace error word, clear it, and return
 * SA_ERR_BOUNDS, SA_ERR_TIMEOUT, SA_ERR_INDEX (in that order of precedence)
 * or SA_OK.
 */
sa_status sa_check_errors(void *workspace, void *stream);

/* Static description of a status code. */
const char *sa_status_string(sa_status s);

#ifdef __cplusplus
}
#endif

#endif /* SA_H_ */
