"""GB300-native sparse latent attention (DeepSeek-V4.1 ``sparse_attn`` step).

A thin ctypes binding over ``libsa.so`` (the C ABI of ``include/sa.h``); every
step of the computation runs in the library's sm_103a kernels.  PyTorch only
supplies device memory and the current stream.  When the library is missing
or no GPU is present, the calls raise -- there is no fallback.

    out = sparse_attn(q, kv, sink, idx, scale)            # bf16 [B,T,64,512]
    y   = sparse_attn_rope_wo_a(q, kv, sink, idx, scale, rope_cos_sin, wo_a)
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from ._build import LIB as _LIB_PATH, LIB_CHECKED as _LIB_CHECKED_PATH, build  # noqa: F401

__all__ = ["sparse_attn", "sparse_attn_two_source", "sparse_attn_two_source_fp4", "sparse_attn_rope_wo_a",
           "sparse_attn_block_tail",
           "topk_indices", "fp4_quantize", "rope_table", "workspace_size",
           "fused_workspace_size", "fused_fp8_workspace_size", "check_errors", "SAError", "library", "build"]

HEADS, HEAD_DIM, MAX_K = 64, 512, 1024
_STATUS = {0: "SA_OK", 1: "SA_ERR_INVALID_ARG", 2: "SA_ERR_UNSUPPORTED", 3: "SA_ERR_WORKSPACE",
           4: "SA_ERR_INDEX", 5: "SA_ERR_TIMEOUT", 6: "SA_ERR_CUDA", 7: "SA_ERR_BOUNDS"}
EXPORTS = ("sa_sparse_attn_workspace_size", "sa_sparse_attn", "sa_sparse_attn_two_source",
           "sa_sparse_attn_rope_wo_a_workspace_size", "sa_sparse_attn_rope_wo_a",
           "sa_rope_table", "sa_check_errors", "sa_status_string", "sa_sparse_attn_noalloc",
           "sa_sparse_attn_block_tail_workspace_size", "sa_sparse_attn_block_tail",
           "sa_topk_indices", "sa_sparse_attn_two_source_fp4", "sa_sparse_attn_rope_wo_a_fp8",
           "sa_sparse_attn_rope_wo_a_fp8_workspace_size", "sa_fp4_quantize")


class SAError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = int(code)
        msg = library().sa_status_string(int(code)).decode()
        super().__init__(f"{where}: {_STATUS.get(int(code), code)} ({msg})")


_lock = threading.Lock()
_lib = None


def library(path: str | None = None, checked: bool = False) -> ctypes.CDLL:
    """Load ``libsa.so`` (raises if it has not been built) and make it the
    library every call of this module uses.  ``checked`` loads the build whose
    kernels test their computed addresses (``libsa_checked.so``, same ABI; a
    failed test surfaces as SA_ERR_BOUNDS)."""
    global _lib
    with _lock:
        if _lib is None or path is not None or checked:
            p = path or (_LIB_CHECKED_PATH if checked else _LIB_PATH)
            if not os.path.exists(p):
                raise RuntimeError(f"{p} is missing: build the CUDA library first "
                                   "(sparse_latent_attention_02_gb300.build())")
            lib = ctypes.CDLL(p)
            V, I, F, D, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_double, ctypes.c_size_t
            lib.sa_sparse_attn_workspace_size.restype = Z
            lib.sa_sparse_attn_workspace_size.argtypes = [I, I, I, I, I]
            lib.sa_sparse_attn.restype = I
            lib.sa_sparse_attn.argtypes = [V, V, V, V, F, I, I, I, I, I, I, V, I, V, Z, V]
            L = ctypes.c_int64
            lib.sa_sparse_attn_two_source.restype = I
            lib.sa_sparse_attn_two_source.argtypes = [V, V, I, L, V, I, L, V, V, F, I, I, I, I, I, V, I,
                                                      V, Z, V]
            lib.sa_sparse_attn_rope_wo_a_workspace_size.restype = Z
            lib.sa_sparse_attn_rope_wo_a_workspace_size.argtypes = [I, I, I, I, I, I, I]
            lib.sa_sparse_attn_rope_wo_a.restype = I
            lib.sa_sparse_attn_rope_wo_a.argtypes = [V, V, V, V, F, I, I, I, I, I, I, V, I, V, I, I,
                                                     V, V, Z, V]
            lib.sa_sparse_attn_rope_wo_a_fp8_workspace_size.restype = Z
            lib.sa_sparse_attn_rope_wo_a_fp8_workspace_size.argtypes = [I, I, I, I, I, I, I]
            lib.sa_sparse_attn_rope_wo_a_fp8.restype = I
            lib.sa_sparse_attn_rope_wo_a_fp8.argtypes = [V, V, V, V, F, I, I, I, I, I, I, V, I, V, V, I,
                                                         I, V, V, Z, V]
            lib.sa_sparse_attn_block_tail_workspace_size.restype = Z
            lib.sa_sparse_attn_block_tail_workspace_size.argtypes = [I, I, I, I, I, I, I]
            lib.sa_sparse_attn_block_tail.restype = I
            lib.sa_sparse_attn_block_tail.argtypes = [V, V, V, V, F, I, I, I, I, I, I, V, I, V, I, I,
                                                      V, I, V, V, Z, V]
            lib.sa_sparse_attn_two_source_fp4.restype = I
            lib.sa_sparse_attn_two_source_fp4.argtypes = [V, V, I, L, V, V, I, L, V, V, F, I, I, I, I, I,
                                                          V, I, V, Z, V]
            lib.sa_fp4_quantize.restype = I
            lib.sa_fp4_quantize.argtypes = [V, ctypes.c_int64, ctypes.c_int64, I, V, V, V]
            lib.sa_topk_indices.restype = I
            lib.sa_topk_indices.argtypes = [V, ctypes.c_int64, ctypes.c_int64, I, I, I, V, V]
            lib.sa_rope_table.restype = I
            lib.sa_rope_table.argtypes = [D, I, I, I, V]
            lib.sa_check_errors.restype = I
            lib.sa_check_errors.argtypes = [V, V]
            lib.sa_status_string.restype = ctypes.c_char_p
            lib.sa_status_string.argtypes = [I]
            lib.sa_sparse_attn_noalloc.restype = I
            lib.sa_sparse_attn_noalloc.argtypes = [V, V, V, V, F, I, I, I, I, I, I, V, I,
                                                   ctypes.POINTER(ctypes.c_void_p), V]
            if path is None:
                _lib = lib
            else:
                return lib
    return _lib


def _check(code: int, where: str):
    if code != 0:
        raise SAError(code, where)


def _need(t: torch.Tensor, name: str, dtype, ndim: int, pinned_ok: bool = False):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    if not t.is_cuda and not (pinned_ok and t.is_pinned()):
        raise ValueError(f"{name} must live on a CUDA device"
                         + (" or in page-locked host memory" if pinned_ok else ""))
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _stream_ptr(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


_ws_cache: dict = {}


def _workspace(nbytes: int, device: torch.device, key: str, stream=None) -> torch.Tensor:
    """A zero-initialised scratch buffer per device, stream and kind of call,
    grown on demand.  Calls on different streams get different buffers: the
    fused calls keep the attention output there between their kernels, so a
    shared buffer would let concurrent calls overwrite each other's.  Each
    buffer is allocated on the stream that uses it, so the caching allocator
    reuses a replaced one only after that stream's pending work."""
    s = stream if stream is not None else torch.cuda.current_stream()
    k = (device.index, key, int(s.cuda_stream))
    ws = _ws_cache.get(k)
    if ws is None or ws.numel() < nbytes:
        with torch.cuda.stream(s):
            ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
        _ws_cache[k] = ws
    return ws


def workspace_size(B: int, T: int, K: int) -> int:
    return int(library().sa_sparse_attn_workspace_size(B, T, HEADS, HEAD_DIM, K))


def fused_workspace_size(B: int, T: int, K: int, G: int, R: int) -> int:
    return int(library().sa_sparse_attn_rope_wo_a_workspace_size(B, T, HEADS, HEAD_DIM, K, G, R))


def fused_fp8_workspace_size(B: int, T: int, K: int, G: int, R: int) -> int:
    return int(library().sa_sparse_attn_rope_wo_a_fp8_workspace_size(B, T, HEADS, HEAD_DIM, K, G, R))


def _attn_args(q, kv, sink, idx):
    _need(q, "q", torch.bfloat16, 4)
    # kv may stay in page-locked host memory: the kernel gathers its rows from there
    _need(kv, "kv", torch.bfloat16, 3, pinned_ok=True)
    _need(sink, "sink", torch.float32, 1)
    _need(idx, "idx", torch.int32, 3)
    B, T, H, D = q.shape
    if kv.shape[0] != B or kv.shape[2] != D:
        raise ValueError(f"kv {tuple(kv.shape)} does not match q {tuple(q.shape)}")
    if sink.shape[0] != H or idx.shape[:2] != (B, T):
        raise ValueError("sink / idx shapes do not match q")
    devs = {t.device for t in (q, sink, idx)} | ({kv.device} if kv.is_cuda else set())
    if len(devs) != 1:
        raise ValueError("all device inputs must be on one device")
    return B, T, H, D, kv.shape[1], idx.shape[2]


def sparse_attn(q: torch.Tensor, kv: torch.Tensor, sink: torch.Tensor, idx: torch.Tensor,
                scale: float, out: torch.Tensor | None = None,
                out_dtype: torch.dtype = torch.bfloat16, workspace: torch.Tensor | None = None,
                stream=None, check: bool = False) -> torch.Tensor:
    """``sparse_attn(q, kv, attn_sink, topk_idxs, softmax_scale)`` -> [B, T, H, D].

    q bf16 [B,T,64,512], kv bf16 [B,N,512], sink fp32 [64], idx int32 [B,T,K].
    ``check=True`` synchronises and raises on a device-side error (bad index).
    """
    B, T, H, D, N, K = _attn_args(q, kv, sink, idx)
    if out is None:
        out = torch.empty((B, T, H, D), dtype=out_dtype, device=q.device)
    else:
        _need(out, "out", out.dtype, 4)
    if out.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("out must be bf16 or fp32")
    lib = library()
    need = int(lib.sa_sparse_attn_workspace_size(B, T, H, D, K))
    if workspace is None:
        workspace = _workspace(need, q.device, "attn", stream)
    code = lib.sa_sparse_attn(q.data_ptr(), kv.data_ptr(), sink.data_ptr(), idx.data_ptr(),
                              float(scale), B, T, H, D, N, K, out.data_ptr(),
                              1 if out.dtype == torch.float32 else 0, workspace.data_ptr(),
                              workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    _check(code, "sa_sparse_attn")
    if check:
        check_errors(workspace, stream)
    return out


def _source(t: torch.Tensor | None, name: str, used: int | None, B: int, D: int):
    """(pointer, used rows, batch stride in rows) of one latent source [Bmax, rows, D]."""
    if t is None:
        if used:
            raise ValueError(f"{name} is missing")
        return 0, 0, 0
    _need_rows(t, name, D)
    if t.shape[0] < B:
        raise ValueError(f"{name} has {t.shape[0]} batch rows, q has {B}")
    rows = t.shape[1] if used is None else int(used)
    if not 0 <= rows <= t.shape[1]:
        raise ValueError(f"{name}: {rows} rows used of {t.shape[1]}")
    return t.data_ptr(), rows, t.stride(0) // D


def _need_rows(t: torch.Tensor, name: str, D: int):
    if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or t.dim() != 3 or t.shape[2] != D:
        raise TypeError(f"{name} must be a bf16 tensor [batch, rows, {D}]")
    if not t.is_cuda and not t.is_pinned():
        raise ValueError(f"{name} must live on a CUDA device or in page-locked host memory")
    if t.stride(2) != 1 or t.stride(1) != D or t.stride(0) % D:
        raise ValueError(f"{name} must have contiguous {D}-element rows")


def sparse_attn_two_source(q: torch.Tensor, window_kv: torch.Tensor | None,
                           compressed_kv: torch.Tensor | None, sink: torch.Tensor, idx: torch.Tensor,
                           scale: float, W: int | None = None, C: int | None = None,
                           out: torch.Tensor | None = None, out_dtype: torch.dtype = torch.bfloat16,
                           workspace: torch.Tensor | None = None, stream=None,
                           check: bool = False) -> torch.Tensor:
    """sparse_attn over the window ring and the compressed cache read in place:
    the same result as ``sparse_attn(q, cat(window_kv[:, :W], compressed_kv[:, :C], 1), ...)``.

    window_kv bf16 [Bmax, >= W, 512] and compressed_kv bf16 [Bmax, >= C, 512] may be
    views of larger caches (their batch strides are used); W and C default to
    their row counts; idx values lie in [0, W + C) or are -1.
    """
    _need(q, "q", torch.bfloat16, 4)
    _need(sink, "sink", torch.float32, 1)
    _need(idx, "idx", torch.int32, 3)
    B, T, H, D = q.shape
    if sink.shape[0] != H or idx.shape[:2] != (B, T):
        raise ValueError("sink / idx shapes do not match q")
    pw, W, sw = _source(window_kv, "window_kv", W, B, D)
    pc, C, sc = _source(compressed_kv, "compressed_kv", C, B, D)
    K = idx.shape[2]
    if out is None:
        out = torch.empty((B, T, H, D), dtype=out_dtype, device=q.device)
    else:
        _need(out, "out", out.dtype, 4)
    if out.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("out must be bf16 or fp32")
    lib = library()
    need = int(lib.sa_sparse_attn_workspace_size(B, T, H, D, K))
    if workspace is None:
        workspace = _workspace(need, q.device, "attn", stream)
    code = lib.sa_sparse_attn_two_source(q.data_ptr(), pw, W, sw, pc, C, sc, sink.data_ptr(),
                                         idx.data_ptr(), float(scale), B, T, H, D, K, out.data_ptr(),
                                         1 if out.dtype == torch.float32 else 0, workspace.data_ptr(),
                                         workspace.numel() * workspace.element_size(),
                                         _stream_ptr(stream))
    _check(code, "sa_sparse_attn_two_source")
    if check:
        check_errors(workspace, stream)
    return out


def sparse_attn_two_source_fp4(q: torch.Tensor, window_kv: torch.Tensor | None,
                               codes: torch.Tensor | None, scales: torch.Tensor | None,
                               sink: torch.Tensor, idx: torch.Tensor, scale: float,
                               W: int | None = None, C: int | None = None,
                               out: torch.Tensor | None = None,
                               out_dtype: torch.dtype = torch.bfloat16,
                               workspace: torch.Tensor | None = None, stream=None,
                               check: bool = False) -> torch.Tensor:
    """sparse_attn_two_source with the compressed cache as fp4: codes uint8
    [Bmax, >= C, 256] (two e2m1 codes per byte, low nibble first) and scales
    uint8 [Bmax, >= C, 32] (E4M3, one per 16 features); the window stays bf16."""
    _need(q, "q", torch.bfloat16, 4)
    _need(sink, "sink", torch.float32, 1)
    _need(idx, "idx", torch.int32, 3)
    B, T, H, D = q.shape
    if sink.shape[0] != H or idx.shape[:2] != (B, T):
        raise ValueError("sink / idx shapes do not match q")
    pw, W, sw = _source(window_kv, "window_kv", W, B, D)
    if codes is None or scales is None:
        if C:
            raise ValueError("codes and scales are needed when C > 0")
        pc = ps = 0
        C, sc = 0, 0
    else:
        for t, name, width in ((codes, "codes", D // 2), (scales, "scales", D // 16)):
            if not isinstance(t, torch.Tensor) or t.dtype != torch.uint8 or t.dim() != 3 or t.shape[2] != width:
                raise TypeError(f"{name} must be a uint8 tensor [batch, rows, {width}]")
            if not t.is_cuda and not t.is_pinned():
                raise ValueError(f"{name} must live on a CUDA device or in page-locked host memory")
            if t.stride(2) != 1 or t.stride(1) != width or t.shape[0] < B:
                raise ValueError(f"{name} must have contiguous rows and >= {B} batch rows")
        if codes.shape[:2] != scales.shape[:2] or codes.stride(0) // (D // 2) != scales.stride(0) // (D // 16):
            raise ValueError("codes and scales must have the same rows and batch stride")
        C = codes.shape[1] if C is None else int(C)
        if not 0 <= C <= codes.shape[1]:
            raise ValueError(f"{C} rows used of {codes.shape[1]}")
        pc, ps, sc = codes.data_ptr(), scales.data_ptr(), codes.stride(0) // (D // 2)
    K = idx.shape[2]
    if out is None:
        out = torch.empty((B, T, H, D), dtype=out_dtype, device=q.device)
    else:
        _need(out, "out", out.dtype, 4)
    if out.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("out must be bf16 or fp32")
    lib = library()
    need = int(lib.sa_sparse_attn_workspace_size(B, T, H, D, K))
    if workspace is None:
        workspace = _workspace(need, q.device, "attn", stream)
    code = lib.sa_sparse_attn_two_source_fp4(q.data_ptr(), pw, W, sw, pc, ps, C, sc, sink.data_ptr(),
                                             idx.data_ptr(), float(scale), B, T, H, D, K, out.data_ptr(),
                                             1 if out.dtype == torch.float32 else 0, workspace.data_ptr(),
                                             workspace.numel() * workspace.element_size(),
                                             _stream_ptr(stream))
    _check(code, "sa_sparse_attn_two_source_fp4")
    if check:
        check_errors(workspace, stream)
    return out


def sparse_attn_rope_wo_a(q: torch.Tensor, kv: torch.Tensor, sink: torch.Tensor,
                          idx: torch.Tensor, scale: float, rope_cos_sin: torch.Tensor,
                          wo_a: torch.Tensor, out: torch.Tensor | None = None,
                          workspace: torch.Tensor | None = None, stream=None,
                          check: bool = False) -> torch.Tensor:
    """sparse_attn, inverse RoPE on the last rope_dim features, grouped wo_a.

    rope_cos_sin fp32 [T, rope_dim/2, 2]; wo_a bf16 [G, R, H*D/G]; returns bf16 [B, T, G*R].
    """
    B, T, H, D, N, K = _attn_args(q, kv, sink, idx)
    _need(rope_cos_sin, "rope_cos_sin", torch.float32, 3)
    _need(wo_a, "wo_a", torch.bfloat16, 3)
    G, R, Din = wo_a.shape
    if rope_cos_sin.shape[0] != T or rope_cos_sin.shape[2] != 2:
        raise ValueError("rope_cos_sin must be [T, rope_dim/2, 2]")
    if G * Din != H * D:
        raise ValueError("wo_a must be [G, R, H*D/G]")
    rope_dim = 2 * rope_cos_sin.shape[1]
    if out is None:
        out = torch.empty((B, T, G * R), dtype=torch.bfloat16, device=q.device)
    else:
        _need(out, "out", torch.bfloat16, 3)
    lib = library()
    need = int(lib.sa_sparse_attn_rope_wo_a_workspace_size(B, T, H, D, K, G, R))
    if workspace is None:
        workspace = _workspace(need, q.device, "fused", stream)
    code = lib.sa_sparse_attn_rope_wo_a(q.data_ptr(), kv.data_ptr(), sink.data_ptr(),
                                        idx.data_ptr(), float(scale), B, T, H, D, N, K,
                                        rope_cos_sin.data_ptr(), rope_dim, wo_a.data_ptr(), G, R,
                                        out.data_ptr(), workspace.data_ptr(),
                                        workspace.numel() * workspace.element_size(),
                                        _stream_ptr(stream))
    _check(code, "sa_sparse_attn_rope_wo_a")
    if check:
        check_errors(workspace, stream)
    return out


def sparse_attn_rope_wo_a_fp8(q: torch.Tensor, kv: torch.Tensor, sink: torch.Tensor,
                              idx: torch.Tensor, scale: float, rope_cos_sin: torch.Tensor,
                              wo_a_e4m3: torch.Tensor, wo_a_scales: torch.Tensor,
                              out: torch.Tensor | None = None,
                              workspace: torch.Tensor | None = None, stream=None,
                              check: bool = False) -> torch.Tensor:
    """sparse_attn_rope_wo_a with wo_a in fp8: E4M3 bytes uint8 [G, R, H*D/G]
    and fp32 scales [G*R/128, H*D/G/128], one per 128 x 128 block, dequantized
    in the kernel to bf16(fp32(value * scale)).  Returns bf16 [B, T, G*R]."""
    B, T, H, D, N, K = _attn_args(q, kv, sink, idx)
    _need(rope_cos_sin, "rope_cos_sin", torch.float32, 3)
    _need(wo_a_e4m3, "wo_a_e4m3", torch.uint8, 3)
    _need(wo_a_scales, "wo_a_scales", torch.float32, 2)
    G, R, Din = wo_a_e4m3.shape
    if rope_cos_sin.shape[0] != T or rope_cos_sin.shape[2] != 2:
        raise ValueError("rope_cos_sin must be [T, rope_dim/2, 2]")
    if G * Din != H * D:
        raise ValueError("wo_a_e4m3 must be [G, R, H*D/G]")
    if tuple(wo_a_scales.shape) != ((G * R + 127) // 128, (Din + 127) // 128):
        raise ValueError("wo_a_scales must be [G*R/128, H*D/G/128]")
    rope_dim = 2 * rope_cos_sin.shape[1]
    if out is None:
        out = torch.empty((B, T, G * R), dtype=torch.bfloat16, device=q.device)
    else:
        _need(out, "out", torch.bfloat16, 3)
    lib = library()
    if workspace is None:
        need = int(lib.sa_sparse_attn_rope_wo_a_fp8_workspace_size(B, T, H, D, K, G, R))
        workspace = _workspace(need, q.device, "fused_fp8", stream)
    code = lib.sa_sparse_attn_rope_wo_a_fp8(q.data_ptr(), kv.data_ptr(), sink.data_ptr(),
                                            idx.data_ptr(), float(scale), B, T, H, D, N, K,
                                            rope_cos_sin.data_ptr(), rope_dim, wo_a_e4m3.data_ptr(),
                                            wo_a_scales.data_ptr(), G, R, out.data_ptr(),
                                            workspace.data_ptr(),
                                            workspace.numel() * workspace.element_size(),
                                            _stream_ptr(stream))
    _check(code, "sa_sparse_attn_rope_wo_a_fp8")
    if check:
        check_errors(workspace, stream)
    return out


def sparse_attn_block_tail(q: torch.Tensor, kv: torch.Tensor, sink: torch.Tensor,
                           idx: torch.Tensor, scale: float, rope_cos_sin: torch.Tensor,
                           wo_a: torch.Tensor, wo_b: torch.Tensor, out: torch.Tensor | None = None,
                           workspace: torch.Tensor | None = None, stream=None,
                           check: bool = False) -> torch.Tensor:
    """The attention block's tail: sparse_attn, inverse RoPE, grouped wo_a, then wo_b.

    rope_cos_sin fp32 [T, rope_dim/2, 2]; wo_a bf16 [G, R, H*D/G]; wo_b bf16 [dim, G*R]
    ([out, in]); returns bf16 [B, T, dim].
    """
    B, T, H, D, N, K = _attn_args(q, kv, sink, idx)
    _need(rope_cos_sin, "rope_cos_sin", torch.float32, 3)
    _need(wo_a, "wo_a", torch.bfloat16, 3)
    _need(wo_b, "wo_b", torch.bfloat16, 2)
    G, R, Din = wo_a.shape
    dim = wo_b.shape[0]
    if rope_cos_sin.shape[0] != T or rope_cos_sin.shape[2] != 2:
        raise ValueError("rope_cos_sin must be [T, rope_dim/2, 2]")
    if G * Din != H * D:
        raise ValueError("wo_a must be [G, R, H*D/G]")
    if wo_b.shape[1] != G * R:
        raise ValueError("wo_b must be [dim, G*R]")
    rope_dim = 2 * rope_cos_sin.shape[1]
    if out is None:
        out = torch.empty((B, T, dim), dtype=torch.bfloat16, device=q.device)
    else:
        _need(out, "out", torch.bfloat16, 3)
    lib = library()
    need = int(lib.sa_sparse_attn_block_tail_workspace_size(B, T, H, D, K, G, R))
    if workspace is None:
        workspace = _workspace(need, q.device, "tail", stream)
    code = lib.sa_sparse_attn_block_tail(q.data_ptr(), kv.data_ptr(), sink.data_ptr(), idx.data_ptr(),
                                         float(scale), B, T, H, D, N, K, rope_cos_sin.data_ptr(),
                                         rope_dim, wo_a.data_ptr(), G, R, wo_b.data_ptr(), dim,
                                         out.data_ptr(), workspace.data_ptr(),
                                         workspace.numel() * workspace.element_size(),
                                         _stream_ptr(stream))
    _check(code, "sa_sparse_attn_block_tail")
    if check:
        check_errors(workspace, stream)
    return out


def topk_indices(scores: torch.Tensor, k: int, offset: int = 0, out: torch.Tensor | None = None,
                 stream=None) -> torch.Tensor:
    """Positions of the k largest scores per row (-inf / NaN never chosen, ties
    to the smaller position), ascending, plus ``offset``; -1 padded.

    scores fp32 [..., L] on the GPU (rows of unit stride); returns int32 [..., k].
    """
    if not isinstance(scores, torch.Tensor) or scores.dtype != torch.float32 or scores.dim() < 1:
        raise TypeError("scores must be an fp32 tensor [..., L]")
    if not scores.is_cuda:
        raise ValueError("scores must live on a CUDA device")
    if scores.stride(-1) != 1:
        raise ValueError("scores rows must be contiguous")
    L = scores.shape[-1]
    lead = scores.shape[:-1]
    rows = 1
    for n in lead:
        rows *= int(n)
    flat = scores.reshape(rows, L)
    if out is None:
        out = torch.empty((*lead, k), dtype=torch.int32, device=scores.device)
    elif out.dtype != torch.int32 or out.shape != (*lead, k) or not out.is_contiguous():
        raise ValueError("out must be a contiguous int32 [..., k]")
    code = library().sa_topk_indices(flat.data_ptr() if L > 0 else None,
                                     flat.stride(0) if rows > 0 else L, rows, L, int(k), int(offset),
                                     out.data_ptr() if out.numel() else None, _stream_ptr(stream))
    _check(code, "sa_topk_indices")
    return out


def fp4_quantize(latent: torch.Tensor, codes: torch.Tensor | None = None, scales: torch.Tensor | None = None,
                 stream=None) -> tuple[torch.Tensor, torch.Tensor]:
    """Latent rows bf16 [..., D] -> the fp4 compressed-cache form read by
    :func:`sparse_attn_two_source_fp4`: (codes uint8 [..., D/2], scales uint8
    [..., D/16]), an E4M3 scale of amax / 6 per 16 features and e2m1 codes of
    x / scale (``fp4_act_quant(latent, 16, True, scale_dtype=float8_e4m3fn)``).

    Rows may be strided (stride a multiple of 8 elements); D % 16 == 0."""
    if not isinstance(latent, torch.Tensor) or latent.dtype != torch.bfloat16 or latent.dim() < 1:
        raise TypeError("latent must be a bf16 tensor [..., D]")
    if not latent.is_cuda:
        raise ValueError("latent must live on a CUDA device")
    if latent.stride(-1) != 1:
        raise ValueError("latent rows must be contiguous")
    D = latent.shape[-1]
    lead = latent.shape[:-1]
    rows = 1
    for n in lead:
        rows *= int(n)
    flat = latent.reshape(rows, D)
    if codes is None:
        codes = torch.empty((*lead, D // 2), dtype=torch.uint8, device=latent.device)
    if scales is None:
        scales = torch.empty((*lead, D // 16), dtype=torch.uint8, device=latent.device)
    if codes.dtype != torch.uint8 or codes.shape != (*lead, D // 2) or not codes.is_contiguous():
        raise ValueError("codes must be a contiguous uint8 [..., D/2]")
    if scales.dtype != torch.uint8 or scales.shape != (*lead, D // 16) or not scales.is_contiguous():
        raise ValueError("scales must be a contiguous uint8 [..., D/16]")
    if rows == 0:
        return codes, scales
    code = library().sa_fp4_quantize(flat.data_ptr(), rows, flat.stride(0), D, codes.data_ptr(),
                                     scales.data_ptr(), _stream_ptr(stream))
    _check(code, "sa_fp4_quantize")
    return codes, scales


def block_tail_workspace_size(B: int, T: int, K: int, G: int, R: int) -> int:
    return int(library().sa_sparse_attn_block_tail_workspace_size(B, T, HEADS, HEAD_DIM, K, G, R))


def rope_table(theta: float, start_pos: int, T: int, rope_dim: int = 64) -> torch.Tensor:
    """Host-built fp32 [T, rope_dim/2, 2] (cos, sin) table (double-precision angles)."""
    t = torch.empty((T, rope_dim // 2, 2), dtype=torch.float32)
    _check(library().sa_rope_table(float(theta), int(start_pos), int(T), int(rope_dim),
                                   t.data_ptr() if T > 0 else None), "sa_rope_table")
    return t


def check_errors(workspace: torch.Tensor, stream=None):
    """Synchronise, read and clear the workspace error word; raise SAError if set.

    A device-detected error (an index outside [-1, N), a wait that ran out)
    stays OR-ed into the workspace's error word across later calls on the same
    workspace until this function reads and clears it: a clean call does not
    clear an earlier call's error."""
    _check(library().sa_check_errors(workspace.data_ptr(), _stream_ptr(stream)), "device")
