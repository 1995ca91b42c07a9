"""fp64 CPU oracle for sparse latent attention -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never loads it and
shares no code with it.

The arithmetic lives in ``sa_oracle.c`` (plain C, fp64, OpenMP over queries);
this module compiles it with gcc on first use and exposes numpy-facing
wrappers:

* :func:`sparse_attn`   -- the ``sparse_attn(q, kv, attn_sink, topk_idxs,
  softmax_scale)`` step of the "DeepSeek-V4.1 > Output projection" page
  (``Attention.forward`` excerpt), with the sink as an extra softmax logit and
  -1 as "skip";
* :func:`inverse_rope`  -- ``apply_rotary_emb(o[..., -rd:], freqs_cis, True)``
  read as consecutive complex pairs rotated by ``-pos * theta**(-2i/rd)``;
* :func:`wo_a`          -- the block-diagonal ``einsum("bsgd,grd->bsgr")``;
* :func:`dequant_fp8_weight` -- the fp8 ``wo_a`` weight (E4M3, fp32 scale per
  128 x 128 block) dequantized to bf16, as the page's conversion does before
  the einsum.
* :func:`fp4_quantize`  -- ``fp4_act_quant(latent, 16, True,
  scale_dtype=torch.float8_e4m3fn)`` of the "DeepSeek-V4.1 > 40 layers" page,
  read as an E4M3 scale of amax / 6 per 16 features and e2m1 codes of x /
  scale, both rounded to nearest with ties to even (:func:`e4m3_encode`,
  :func:`e2m1_encode`), in the packed layout :func:`dequant_fp4` reads.

Every function is pinned by ``tests/test_oracle_pins.py`` against a dense
masked brute force, closed forms and invariants; nothing here is "parity
unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libsa_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``sa_oracle.c`` into ``libsa_oracle.so`` next to it."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.sa_oracle_sparse_attn.restype = i64
            lib.sa_oracle_sparse_attn.argtypes = [P, P, P, P, f64, i32, i32, i32,
                                                  i32, i32, i32, P, i64, P, i32]
            lib.sa_oracle_inverse_rope.restype = None
            lib.sa_oracle_inverse_rope.argtypes = [P, i64, P, i32, i32, i32, f64, i32]
            lib.sa_oracle_wo_a.restype = None
            lib.sa_oracle_wo_a.argtypes = [P, P, i64, i32, i32, i32, P, i32]
            lib.sa_oracle_threads.restype = i32
            lib.sa_oracle_threads.argtypes = [i32]
            _lib = lib
    return _lib


def threads(n: int = 0) -> int:
    """How many OpenMP threads a call with ``n_threads=n`` uses (0 = all)."""
    return int(_load().sa_oracle_threads(int(n)))


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _as_bf16_bits(x) -> np.ndarray:
    """Accept raw bf16 bits (uint16/int16 numpy) or a torch bf16 tensor."""
    if hasattr(x, "view") and hasattr(x, "dtype") and str(x.dtype) == "torch.bfloat16":
        import torch
        x = x.detach().cpu().contiguous().view(torch.int16).numpy()
    a = np.ascontiguousarray(x)
    if a.dtype not in (np.uint16, np.int16):
        raise TypeError("expected bf16 bit patterns (uint16) or a torch.bfloat16 tensor")
    return a.view(np.uint16)


def _np(x, dtype) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(x, dtype=dtype)


def sparse_attn(q, kv, sink, idx, scale: float, queries=None, n_threads: int = 0):
    """fp64 ``sparse_attn``.

    q bf16 [B,T,H,D]; kv bf16 [B,N,D]; sink fp32 [H]; idx int32 [B,T,K].
    ``queries``: optional 1-D list of flattened query numbers ``b*T+t``.
    Returns (out fp64 [n_queries,H,D] -- [B,T,H,D] when ``queries`` is None,
    number of queries that met an index outside [-1, N)).
    """
    qb, kvb = _as_bf16_bits(q), _as_bf16_bits(kv)
    B, T, H, D = qb.shape
    Bk, N, Dk = kvb.shape
    s = _np(sink, np.float32)
    ix = _np(idx, np.int32)
    if Bk != B or Dk != D or s.shape != (H,) or ix.shape[:2] != (B, T):
        raise ValueError("shape mismatch")
    K = ix.shape[2]
    if queries is None:
        ql, nq, qp = None, B * T, None
    else:
        ql = np.ascontiguousarray(queries, dtype=np.int64).reshape(-1)
        if ql.size and (ql.min() < 0 or ql.max() >= B * T):
            raise ValueError("query number out of range")
        nq, qp = ql.size, _ptr(ql)
    out = np.zeros((nq, H, D), dtype=np.float64)
    bad = _load().sa_oracle_sparse_attn(_ptr(qb), _ptr(kvb), _ptr(s), _ptr(ix),
                                        float(scale), B, T, H, D, N, K, qp, nq,
                                        _ptr(out), int(n_threads))
    if queries is None:
        out = out.reshape(B, T, H, D)
    return out, int(bad)


def sparse_attn_two_source(q, window_kv, W: int, compressed_kv, C: int, sink, idx, scale: float,
                           queries=None, n_threads: int = 0):
    """fp64 ``sparse_attn`` over the window ring and the compressed cache, as the
    "DeepSeek-V4.1 > Output projection" page's Attention.forward builds its kv:
    ``torch.cat([window_kv, compress_kv], dim=1)`` (first W window rows, then
    the first C compressed rows of each batch element), then ``sparse_attn``.
    window_kv / compressed_kv bf16 [>= B, >= W / >= C, D] (None when W / C is 0).
    """
    qb = _as_bf16_bits(q)
    B, _, _, D = qb.shape
    parts = []
    if W:
        parts.append(_as_bf16_bits(window_kv)[:B, :W])
    if C:
        parts.append(_as_bf16_bits(compressed_kv)[:B, :C])
    kv = np.concatenate(parts, axis=1) if parts else np.zeros((B, 0, D), dtype=np.uint16)
    return sparse_attn(qb, np.ascontiguousarray(kv), sink, idx, scale, queries=queries, n_threads=n_threads)


E2M1_MAGNITUDES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def e4m3_values(b) -> np.ndarray:
    """OCP FP8 E4M3 ("fn": bias 7, no infinities, S.1111.111 = NaN) bytes -> fp64."""
    b = np.asarray(b, dtype=np.int64)
    e, m = (b >> 3) & 15, b & 7
    v = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    v = np.where((e == 15) & (m == 7), np.nan, v)
    return np.where(b & 0x80, -v, v)


def dequant_fp4(codes, scales) -> np.ndarray:
    """fp4 compressed rows (the "DeepSeek-V4.1 > 40 layers" page's
    `fp4_act_quant(latent, 16, True, scale_dtype=torch.float8_e4m3fn)`: e2m1
    values in groups of 16 features with an E4M3 scale each) -> fp64 values.
    codes uint8 [..., D/2]: byte i = feature 2i (low nibble), 2i+1 (high);
    e2m1 code: bit 3 sign, bits 2..0 index the magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6.
    scales uint8 [..., D/16]: E4M3 scale of features 16g .. 16g+15."""
    c = np.asarray(codes, dtype=np.uint8)
    nib = np.stack([c & 15, c >> 4], axis=-1).reshape(*c.shape[:-1], 2 * c.shape[-1]).astype(np.int64)
    mag = np.asarray(E2M1_MAGNITUDES)[nib & 7]
    val = np.where(nib & 8, -mag, mag)
    sc = np.repeat(e4m3_values(scales), 16, axis=-1)
    return val * sc


def _nearest_even(x, grid, even) -> np.ndarray:
    """Index into `grid` (ascending, non-negative) of the value nearest to each
    |x|, halfway cases to the index whose `even` flag is set; |x| above the
    largest grid value takes the largest (saturation)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    g = np.asarray(grid, dtype=np.float64)
    hi = np.clip(np.searchsorted(g, a, side="left"), 0, len(g) - 1)   # first grid value >= a
    lo = np.clip(hi - 1, 0, len(g) - 1)
    dlo, dhi = a - g[lo], g[hi] - a
    pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(np.asarray(even)[lo], lo, hi)))
    return np.where(a >= g[-1], len(g) - 1, pick)


def e4m3_encode(x) -> np.ndarray:
    """Values -> OCP FP8 E4M3 ("fn") bytes: the nearest finite E4M3 value,
    halfway cases to the even mantissa, magnitudes past 448 to 448; the sign
    kept (also for results of zero)."""
    x = np.asarray(x, dtype=np.float64)
    mags = np.arange(0x7F, dtype=np.int64)                  # 0x00 .. 0x7E: every finite magnitude
    idx = _nearest_even(x, e4m3_values(mags), (mags & 1) == 0)
    return (idx | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)


def e2m1_encode(x) -> np.ndarray:
    """Values -> e2m1 codes (bit 3 sign, bits 2..0 index 0, .5, 1, 1.5, 2, 3,
    4, 6): the nearest magnitude, halfway cases to the even index, past 6 to
    6; the sign kept (also for results of zero)."""
    x = np.asarray(x, dtype=np.float64)
    idx = _nearest_even(x, E2M1_MAGNITUDES, np.arange(8) % 2 == 0)
    return (idx | np.where(np.signbit(x), 8, 0)).astype(np.uint8)


def fp4_quantize(latent_bf16) -> tuple[np.ndarray, np.ndarray]:
    """The "DeepSeek-V4.1 > 40 layers" page's `fp4_act_quant(latent, 16, True,
    scale_dtype=torch.float8_e4m3fn)` (its body is not on the pages; this is
    the reading the library implements): per group of 16 features, the scale
    is E4M3(amax / 6) (amax the group's largest magnitude, 6 the largest e2m1
    value, the division in fp32), each value's code is e2m1(x / scale) (fp32
    division; a zero scale gives codes of zero with x's sign).

    latent_bf16: bf16 bit patterns uint16 [..., D], D % 16 == 0, finite or
    infinite values.  Returns (codes uint8 [..., D/2], low nibble = even
    feature; scales uint8 [..., D/16]) in the layout of `dequant_fp4`."""
    u = np.asarray(latent_bf16, dtype=np.uint16)
    x = (u.astype(np.uint32) << 16).view(np.float32)
    g = x.reshape(*x.shape[:-1], x.shape[-1] // 16, 16)
    amax = np.max(np.abs(g), axis=-1)
    sb = e4m3_encode(amax / np.float32(6.0))                  # fp32 division
    s = e4m3_values(sb).astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        v = np.where(s > 0, g / np.where(s > 0, s, np.float32(1)), g * np.float32(0))   # fp32 division
    c = e2m1_encode(v).reshape(*x.shape[:-1], x.shape[-1])
    codes = (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)
    return codes, sb


def bf16_bits_exact(x) -> np.ndarray:
    """fp64 values that bf16 holds exactly -> bf16 bit patterns (uint16)."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    if not np.array_equal(f.astype(np.float64), np.asarray(x, dtype=np.float64), equal_nan=True):
        raise ValueError("value not representable in fp32")
    u = f.view(np.uint32)
    if np.any(u & 0xFFFF):
        raise ValueError("value not representable in bf16")
    return (u >> 16).astype(np.uint16)


def round_bf16(x) -> np.ndarray:
    """fp32 values -> bf16 bit patterns (uint16), rounded to nearest with ties
    to even (add 0x7FFF plus the kept part's lowest bit, truncate); NaN stays a
    quiet NaN."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    r = np.where(np.isnan(f), (u >> 16) | 0x40, r)
    return r.astype(np.uint16)


FP8_BLOCK = 128


def dequant_fp8_weight(w8, scales) -> np.ndarray:
    """fp8 grouped ``wo_a`` weight (the "DeepSeek-V4.1 > Output projection"
    page keeps ``wo_a`` in fp8 and dequantizes it to bf16 before the einsum):
    E4M3 bytes [rows, cols] with one fp32 scale per 128 x 128 block
    (scales [ceil(rows/128), ceil(cols/128)]) -> bf16 bit patterns [rows, cols]:
    the product value x scale rounded to fp32, then to bf16 (both to nearest
    even).  The fp64 product is exact (4 x 24 significant bits)."""
    w = np.asarray(w8, dtype=np.uint8)
    sc = np.asarray(scales, dtype=np.float32).astype(np.float64)
    rows, cols = w.shape
    nb_r, nb_c = -(-rows // FP8_BLOCK), -(-cols // FP8_BLOCK)
    if sc.shape != (nb_r, nb_c):
        raise ValueError("scales must be [ceil(rows/128), ceil(cols/128)]")
    s = np.repeat(np.repeat(sc, FP8_BLOCK, axis=0)[:rows], FP8_BLOCK, axis=1)[:, :cols]
    with np.errstate(invalid="ignore", over="ignore"):
        prod = (e4m3_values(w) * s).astype(np.float32)
    return round_bf16(prod)


def sparse_attn_two_source_fp4(q, window_kv, W: int, codes, scales, C: int, sink, idx, scale: float,
                               queries=None, n_threads: int = 0):
    """sparse_attn_two_source with the compressed rows given as fp4: they are
    decoded (exactly, into bf16) and the two sources concatenated."""
    qb = _as_bf16_bits(q)
    B = qb.shape[0]
    comp = None
    if C:
        comp = bf16_bits_exact(dequant_fp4(np.asarray(codes)[:B, :C], np.asarray(scales)[:B, :C]))
    return sparse_attn_two_source(qb, window_kv, W, comp, C, sink, idx, scale, queries=queries,
                                  n_threads=n_threads)


def topk_indices(scores, k: int, offset: int = 0) -> np.ndarray:
    """Top-k selection of compressed positions (the "DeepSeek-V4.1 > 40 layers"
    page's `_compress_topk_idxs`: int32 positions offset by the window length,
    -1 where fewer exist), over given scores: per row the positions of the k
    largest scores that are not -inf or NaN, ties to the smaller position,
    returned in ascending order plus ``offset``, then -1.
    scores float [..., L] -> int32 [..., k] (one stable sort per row)."""
    a = np.asarray(scores, dtype=np.float64)
    L = a.shape[-1]
    rows = a.reshape(int(np.prod(a.shape[:-1], dtype=np.int64)), L)
    out = np.full((rows.shape[0], k), -1, dtype=np.int64)
    for r, row in enumerate(rows):
        pos = np.nonzero(~(np.isnan(row) | (row == -np.inf)))[0]
        # descending score, then ascending position
        order = pos[np.lexsort((pos, -row[pos]))][:k]
        chosen = np.sort(order)
        out[r, :chosen.size] = chosen + offset
    return out.reshape(*a.shape[:-1], k).astype(np.int32)


def inverse_rope(o: np.ndarray, pos, rope_dim: int, theta: float, n_threads: int = 0):
    """In-place-free inverse rotary embedding of the last ``rope_dim`` features.

    o fp64 [..., H, D]; pos int [...] (one position per row of o).
    """
    x = np.array(o, dtype=np.float64, copy=True, order="C")
    H, D = x.shape[-2:]
    p = np.ascontiguousarray(np.broadcast_to(np.asarray(pos, dtype=np.int64),
                                             x.shape[:-2])).reshape(-1)
    n = p.size
    _load().sa_oracle_inverse_rope(_ptr(x), n, _ptr(p), H, D, int(rope_dim),
                                   float(theta), int(n_threads))
    return x


def wo_b(y: np.ndarray, W) -> np.ndarray:
    """``x = self.wo_b(o.flatten(2))`` of the "DeepSeek-V4.1 > Output projection"
    page: a bias-free linear map, weight bf16 [dim, G*R] ([out, in]);
    y fp64 [n, G*R] -> fp64 [n, dim] (one fp64 matrix product)."""
    w = _as_bf16_bits(W).astype(np.uint32) << 16
    w = w.view(np.float32).astype(np.float64)
    y = np.asarray(y, dtype=np.float64)
    if y.ndim != 2 or w.ndim != 2 or y.shape[1] != w.shape[1]:
        raise ValueError("shape mismatch")
    return y @ w.T


def wo_a(o: np.ndarray, W, n_threads: int = 0):
    """Grouped projection: o fp64 [n, G, Din], W bf16 [G, R, Din] -> fp64 [n, G, R]."""
    x = np.ascontiguousarray(o, dtype=np.float64)
    w = _as_bf16_bits(W)
    G, R, Din = w.shape
    lead = x.shape[:-2]
    if x.shape[-2:] != (G, Din):
        raise ValueError("o must end in [G, Din]")
    n = int(np.prod(lead)) if lead else 1
    y = np.zeros(lead + (G, R), dtype=np.float64)
    _load().sa_oracle_wo_a(_ptr(x), _ptr(w), n, G, R, Din, _ptr(y), int(n_threads))
    return y
