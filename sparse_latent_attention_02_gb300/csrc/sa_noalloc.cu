// sa_noalloc.cu -- sparse_attn for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run attention:
// code inside a custom allocator or memory-pool callback, plugins of a host
// framework that owns every device allocation, and real-time loops that must
// not hit the driver's allocator (it may synchronise the device).  For them
// this file provides one entry point that needs no workspace argument: its
// scratch lives in a file-scope device array that exists for as long as the
// library is loaded.
//
// Cost of the convenience: every process that loads this library holds
// SCRATCH_BYTES (64 KiB) of device memory on every GPU it uses, until exit.
#include <mutex>

#include "sa_internal.h"

namespace {

// The attention call's workspace is its 256-byte header (the error word):
// the pieces of a split list merge on chip.  64 KiB leaves room to spare.
constexpr size_t SCRATCH_BYTES = 64u << 10;
static __device__ __align__(256) unsigned char g_scratch[SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;
std::mutex g_mutex;
void *g_scratch_ptr[MAX_DEVICES] = {};

// Device address of g_scratch on the current device.  Looked up once per
// device (with that device current) and kept for the life of the process;
// the name g_scratch itself is only a host-side stand-in and must never be
// handed to a kernel.  The kept address does not survive cudaDeviceReset (or
// anything else that unloads the library's device code on that device).
sa_status scratch_address(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES)
        return SA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p)
            return SA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return SA_OK;
}

}  // namespace

extern "C" sa_status sa_sparse_attn_noalloc(const void *q, const void *kv, const float *sink,
                                            const int32_t *idx, float scale, int B, int T, int H,
                                            int D, int N, int K, void *out, sa_dtype out_dtype,
                                            void **scratch_out, void *stream)
{
    // the host checks that need no device first (a dummy, aligned workspace
    // address stands in for the scratch array here)
    sa_status st = sa::check_attn_args(q, kv, sink, idx, scale, B, T, H, D, N, K, out,
                                       reinterpret_cast<void *>(256));
    if (st != SA_OK)
        return st;
    if (out_dtype != SA_BF16 && out_dtype != SA_F32)
        return SA_ERR_INVALID_ARG;
    // Shapes whose scratch would not fit the static array are refused before
    // anything is enqueued.
    if ((int64_t)B * T > 0 && sa::attn_workspace_bytes((int64_t)B * T, K) > SCRATCH_BYTES)
        return SA_ERR_WORKSPACE;
    void *ws = nullptr;
    st = scratch_address(&ws);
    if (st != SA_OK)
        return st;
    if (scratch_out)
        *scratch_out = ws;
    // The array keeps the previous call's contents: the call clears the error
    // word on the stream, after all of its host checks, right before its launch.
    return sa::attn_call(q, kv, sink, idx, scale, B, T, H, D, N, K, out, out_dtype, ws, SCRATCH_BYTES,
                         static_cast<cudaStream_t>(stream), true);
}
