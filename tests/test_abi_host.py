"""The C-ABI library builds, loads and rejects bad arguments on the host
(CPU only: no call here reaches a kernel)."""
import ctypes
import math
import os
import re

import numpy as np
import pytest

import sparse_latent_attention_02_gb300 as sa

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "sa.h")
OK, INVALID, UNSUPPORTED = 0, 1, 2


@pytest.fixture(scope="module")
def lib():
    sa.build()
    return sa.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sa_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 7
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(sa.EXPORTS)


def test_checked_build_exports_the_same_symbols(lib):
    """The build with address checks in its kernels (libsa_checked.so) is
    built beside libsa.so and exports the same ABI."""
    checked = ctypes.CDLL(sa._LIB_CHECKED_PATH)
    for n in declared_functions():
        assert hasattr(checked, n), n
    checked.sa_status_string.restype = ctypes.c_char_p
    assert b"checked build" in checked.sa_status_string(7)


def _declarations():
    """name -> (return type, [parameter types]) of every function in sa.h."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    out = {}
    for ret, name, params in re.findall(r"(sa_status|size_t|const char \*)\s*(sa_[a-z0-9_]+)\s*\(([^)]*)\)\s*;",
                                         text):
        types = [re.sub(r"\s+[A-Za-z_][A-Za-z0-9_]*$", "", x.strip()) for x in params.split(",")]
        out[name] = (ret, [t for t in types if t and t != "void"])
    return out


def _kind(c_type):
    """The C type of a header parameter as the ctypes type the binding must use."""
    if "*" in c_type:
        return "pointer"
    return {"int": "int", "sa_dtype": "int", "sa_status": "int", "int64_t": "int64", "size_t": "size",
            "float": "float", "double": "double"}[c_type]


def _ctypes_kind(t):
    if t in (ctypes.c_void_p, ctypes.c_char_p) or (isinstance(t, type) and issubclass(t, ctypes._Pointer)):
        return "pointer"
    return {ctypes.c_int: "int", ctypes.c_int64: "int64", ctypes.c_size_t: "size", ctypes.c_float: "float",
            ctypes.c_double: "double"}[t]


def test_binding_signatures_match_the_header(lib):
    """Every function's ctypes argument list has the header's arity and, slot
    by slot, its kind (pointer, int, int64, size_t, float, double); return
    types too.  A slip here would pass garbage through the ABI unseen."""
    decl = _declarations()
    assert set(decl) == set(sa.EXPORTS)
    for name, (ret, params) in decl.items():
        fn = getattr(lib, name)
        got = [_ctypes_kind(t) for t in fn.argtypes]
        assert got == [_kind(p) for p in params], name
        want_ret = {"sa_status": ctypes.c_int, "size_t": ctypes.c_size_t, "const char *": ctypes.c_char_p}[ret]
        assert fn.restype == want_ret, name


def test_status_strings(lib):
    for code in range(8):
        s = lib.sa_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.sa_status_string(99).decode() == "unknown status"


def _attn(lib, **kw):
    a = dict(q=16, kv=16, sink=16, idx=16, scale=0.1, B=1, T=1, H=64, D=512, N=8, K=4,
             out=16, dt=0, ws=256, wsb=1 << 20, stream=None)
    a.update(kw)
    return lib.sa_sparse_attn(a["q"], a["kv"], a["sink"], a["idx"], a["scale"], a["B"], a["T"],
                              a["H"], a["D"], a["N"], a["K"], a["out"], a["dt"], a["ws"],
                              a["wsb"], a["stream"])


def test_host_argument_checks(lib):
    # these are rejected before any CUDA call (pointers are never dereferenced)
    assert _attn(lib, H=32) == UNSUPPORTED
    assert _attn(lib, D=256) == UNSUPPORTED
    assert _attn(lib, K=sa.MAX_K + 1) == UNSUPPORTED
    assert _attn(lib, B=-1) == INVALID
    assert _attn(lib, K=-3) == INVALID
    assert _attn(lib, ws=None) == INVALID
    assert _attn(lib, ws=128) == INVALID          # workspace must be 256-byte aligned
    assert _attn(lib, out=None) == INVALID
    assert _attn(lib, out=8) == INVALID           # output must be 16-byte aligned
    assert _attn(lib, q=None) == INVALID
    assert _attn(lib, kv=24) == INVALID
    assert _attn(lib, idx=2) == INVALID
    assert _attn(lib, sink=None) == INVALID
    assert _attn(lib, scale=float("nan")) == INVALID
    assert _attn(lib, dt=7) in (INVALID, 6)      # bad dtype (or no device to query)
    # empty problems are fine and touch nothing
    assert _attn(lib, B=0, q=None, out=None) == OK
    assert _attn(lib, T=0) == OK


def test_fused_argument_checks(lib):
    def call(**kw):
        a = dict(q=16, kv=16, sink=16, idx=16, scale=0.1, B=1, T=1, H=64, D=512, N=8, K=4,
                 rope=16, rope_dim=64, w=16, G=8, R=1024, out=16, ws=256, wsb=1 << 30,
                 stream=None)
        a.update(kw)
        return lib.sa_sparse_attn_rope_wo_a(a["q"], a["kv"], a["sink"], a["idx"], a["scale"],
                                            a["B"], a["T"], a["H"], a["D"], a["N"], a["K"],
                                            a["rope"], a["rope_dim"], a["w"], a["G"], a["R"],
                                            a["out"], a["ws"], a["wsb"], a["stream"])
    assert call(G=0) == INVALID
    assert call(G=3) == UNSUPPORTED               # 64*512 not divisible into 64-multiples
    assert call(R=1000) == UNSUPPORTED
    assert call(rope_dim=6) == UNSUPPORTED
    assert call(rope_dim=1024) == UNSUPPORTED
    assert call(w=None) == INVALID
    assert call(rope=None) == INVALID
    assert call(H=16) == UNSUPPORTED


def test_block_tail_argument_checks(lib):
    def call(**kw):
        a = dict(q=16, kv=16, sink=16, idx=16, scale=0.1, B=1, T=1, H=64, D=512, N=8, K=4,
                 rope=16, rope_dim=64, wa=16, G=8, R=1024, wb=16, dim=5120, out=16, ws=256,
                 wsb=1 << 31, stream=None)
        a.update(kw)
        return lib.sa_sparse_attn_block_tail(a["q"], a["kv"], a["sink"], a["idx"], a["scale"],
                                             a["B"], a["T"], a["H"], a["D"], a["N"], a["K"],
                                             a["rope"], a["rope_dim"], a["wa"], a["G"], a["R"],
                                             a["wb"], a["dim"], a["out"], a["ws"], a["wsb"],
                                             a["stream"])
    assert call(dim=0) == INVALID
    assert call(dim=5000) == UNSUPPORTED          # not a multiple of 256
    assert call(wb=None) == INVALID
    assert call(wb=8) == INVALID                  # 16-byte alignment
    assert call(rope_dim=16) == UNSUPPORTED       # rotated features must fill whole warps (32)
    assert call(G=3) == UNSUPPORTED
    n = lib.sa_sparse_attn_block_tail_workspace_size(2, 4096, 64, 512, 640, 8, 1024)
    f = lib.sa_sparse_attn_rope_wo_a_workspace_size(2, 4096, 64, 512, 640, 8, 1024)
    assert n >= f + 2 * 4096 * 8 * 1024 * 2 and n % 256 == 0


def test_topk_argument_checks(lib):
    def call(scores=16, stride=8, rows=2, L=8, k=4, offset=0, out=16):
        return lib.sa_topk_indices(scores, stride, rows, L, k, offset, out, None)
    assert call(stride=4) == INVALID              # rows overlap
    assert call(scores=None) == INVALID
    assert call(out=None) == INVALID
    assert call(out=2) == INVALID                 # 4-byte alignment
    assert call(offset=-1) == INVALID
    assert call(L=-1) == INVALID
    assert call(scores=2) == INVALID              # 4-byte alignment of the scores
    assert call(L=100, stride=100, offset=2**31 - 100) == INVALID   # last position + offset past int32
    assert call(rows=2**31) == INVALID            # more rows than a grid holds
    assert call(k=-1) == INVALID
    assert call(rows=0) == OK                     # nothing to do, nothing touched
    assert call(k=0) == OK
    assert call(rows=0, scores=None, out=None) == OK


def test_workspace_size_queries(lib):
    # without a device the size falls back to one SM; it is always >= 256, 256-aligned
    for B, T, K in [(1, 16, 192), (64, 1, 640), (1, 8192, 640), (0, 0, 0)]:
        n = lib.sa_sparse_attn_workspace_size(B, T, 64, 512, K)
        assert n >= 256 and n % 256 == 0
        f = lib.sa_sparse_attn_rope_wo_a_workspace_size(B, T, 64, 512, K, 8, 1024)
        assert f >= n + B * T * 64 * 512 * 2


def test_rope_table_host_helper(lib):
    t = sa.rope_table(160000.0, 3, 5, 64).numpy().astype(np.float64)
    assert t.shape == (5, 32, 2)
    for tt in range(5):
        for i in range(32):
            ang = (3 + tt) * 160000.0 ** (-2.0 * i / 64)
            assert abs(t[tt, i, 0] - math.cos(ang)) < 1e-7
            assert abs(t[tt, i, 1] - math.sin(ang)) < 1e-7
    assert lib.sa_rope_table(160000.0, 0, 4, 63, None) == INVALID
    assert lib.sa_rope_table(-1.0, 0, 4, 64, None) == INVALID


def test_check_errors_rejects_null(lib):
    assert lib.sa_check_errors(None, None) == INVALID


def test_binding_rejects_cpu_tensors():
    import torch
    q = torch.zeros(1, 1, 64, 512, dtype=torch.bfloat16)
    kv = torch.zeros(1, 4, 512, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        sa.sparse_attn(q, kv, torch.zeros(64), torch.zeros(1, 1, 4, dtype=torch.int32), 0.1)
    with pytest.raises(TypeError):
        sa.sparse_attn(q.float(), kv, torch.zeros(64), torch.zeros(1, 1, 4, dtype=torch.int32), 0.1)


def test_fused_fp8_argument_checks(lib):
    def call(**kw):
        a = dict(q=16, kv=16, sink=16, idx=16, scale=0.1, B=1, T=1, H=64, D=512, N=8, K=4,
                 rope=16, rope_dim=64, w8=16, sc=16, G=8, R=1024, out=16, ws=256, wsb=1 << 30,
                 stream=None)
        a.update(kw)
        return lib.sa_sparse_attn_rope_wo_a_fp8(a["q"], a["kv"], a["sink"], a["idx"], a["scale"],
                                                a["B"], a["T"], a["H"], a["D"], a["N"], a["K"],
                                                a["rope"], a["rope_dim"], a["w8"], a["sc"], a["G"],
                                                a["R"], a["out"], a["ws"], a["wsb"], a["stream"])
    assert call(sc=None) == INVALID               # fp8 weights need their scales
    assert call(sc=18) == INVALID                 # scales 4-byte aligned
    assert call(w8=None) == INVALID
    assert call(w8=8) == INVALID                  # weights 16-byte aligned
    assert call(G=512) == UNSUPPORTED             # 64 features per group: not whole 128-wide scale blocks
    assert call(R=1000) == UNSUPPORTED
    assert call(G=0) == INVALID
    assert call(B=0, q=None, out=None) == OK      # empty problems touch nothing


def test_fp8_tail_workspace_size(lib):
    """Below 512 tokens the fp8 tail needs the bf16 tail's workspace (the GEMM
    decodes the weight itself); from 512 tokens on, plus the bf16 copy of the
    weight (R * H * D * 2 bytes) that the call decodes into."""
    for B, T in [(1, 1), (64, 1), (2, 255), (1, 511)]:
        assert (lib.sa_sparse_attn_rope_wo_a_fp8_workspace_size(B, T, 64, 512, 640, 8, 1024)
                == lib.sa_sparse_attn_rope_wo_a_workspace_size(B, T, 64, 512, 640, 8, 1024))
    for B, T in [(1, 512), (2, 4096)]:
        base = lib.sa_sparse_attn_rope_wo_a_workspace_size(B, T, 64, 512, 640, 8, 1024)
        got = lib.sa_sparse_attn_rope_wo_a_fp8_workspace_size(B, T, 64, 512, 640, 8, 1024)
        assert got == base + 1024 * 64 * 512 * 2 and got % 256 == 0


class _Schedule(ctypes.Structure):
    _fields_ = [("grid", ctypes.c_int), ("split", ctypes.c_int), ("per_cta", ctypes.c_int64),
                ("pieces", ctypes.c_int)]


def _schedule_fn(lib):
    # sa::attn_schedule(int64_t BT, int K, int num_sms): host arithmetic only
    fn = getattr(lib, "_ZN2sa13attn_scheduleElii")
    fn.restype = _Schedule
    fn.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int]
    return fn


def test_attention_schedule_on_the_workload_shapes(lib):
    sched = _schedule_fn(lib)
    s = sched(64, 640, 152)          # decode: two pieces of 320 entries, one wave of 128 CTAs
    assert (s.split, s.pieces, s.per_cta, s.grid) == (1, 2, 320, 128)
    s = sched(128, 640, 152)         # long decode: whole queries, one CTA each
    assert (s.split, s.pieces, s.grid) == (0, 1, 128)
    s = sched(8192, 640, 152)        # prefill: a persistent grid of one CTA per SM
    assert (s.split, s.pieces, s.grid) == (0, 1, 152)
    s = sched(16, 192, 152)          # tiny: two pieces (the list holds two 128-row chunks at most)
    assert (s.split, s.pieces, s.per_cta, s.grid) == (1, 2, 96, 32)
    s = sched(1, 1024, 152)          # one query, the longest list: the cluster limit
    assert (s.pieces, s.per_cta, s.grid) == (8, 128, 8)


def test_attention_schedule_invariants(lib):
    """For any shape: one wave of CTAs; pieces a power of two within the
    cluster limit and no more than the list's 128-row chunks; pieces a
    multiple of 32 entries that cover the list, none of them empty."""
    sched = _schedule_fn(lib)
    rng = np.random.default_rng(8)
    for _ in range(3000):
        sms = int(rng.integers(1, 200))
        BT = int(rng.integers(1, 3 * sms))
        K = int(rng.integers(1, 1025))
        s = sched(BT, K, sms)
        if s.split == 0:
            assert s.pieces == 1 and s.grid == min(BT, sms)
            continue
        P = s.pieces
        assert P >= 2 and P & (P - 1) == 0 and P <= 8 and P <= -(-K // 128)
        assert s.grid == BT * P <= sms
        assert s.per_cta % 32 == 0 and P * s.per_cta >= K and (P - 1) * s.per_cta < K
    assert sched(0, 640, 152).grid == 0 and sched(5, 0, 152).split == 0


WORKSPACE = 3


def test_workspace_one_byte_short_is_refused(lib):
    """Every entry point that takes a workspace refuses one a byte smaller
    than its size query with SA_ERR_WORKSPACE, before any CUDA call (so the
    check holds without a device; the pointers are never dereferenced)."""
    L = lib
    for B, T, K in [(1, 16, 192), (64, 1, 640), (2, 4096, 640), (3, 5, 0)]:
        need = L.sa_sparse_attn_workspace_size(B, T, 64, 512, K)
        assert _attn(L, B=B, T=T, K=K, wsb=need - 1) == WORKSPACE
        assert _attn(L, B=B, T=T, K=K, wsb=need) != WORKSPACE
        two = lambda wsb: L.sa_sparse_attn_two_source(16, 16, 4, 4, 16, 4, 4, 16, 16, 0.1, B, T, 64, 512, K,
                                                      16, 0, 256, wsb, None)
        assert two(need - 1) == WORKSPACE and two(need) != WORKSPACE
        fp4 = lambda wsb: L.sa_sparse_attn_two_source_fp4(16, 16, 4, 4, 16, 16, 4, 4, 16, 16, 0.1, B, T, 64,
                                                          512, K, 16, 0, 256, wsb, None)
        assert fp4(need - 1) == WORKSPACE and fp4(need) != WORKSPACE
        fneed = L.sa_sparse_attn_rope_wo_a_workspace_size(B, T, 64, 512, K, 8, 1024)
        fused = lambda wsb: L.sa_sparse_attn_rope_wo_a(16, 16, 16, 16, 0.1, B, T, 64, 512, 8, K, 16, 64, 16,
                                                       8, 1024, 16, 256, wsb, None)
        assert fused(fneed - 1) == WORKSPACE and fused(fneed) != WORKSPACE
        eneed = L.sa_sparse_attn_rope_wo_a_fp8_workspace_size(B, T, 64, 512, K, 8, 1024)
        fp8 = lambda wsb: L.sa_sparse_attn_rope_wo_a_fp8(16, 16, 16, 16, 0.1, B, T, 64, 512, 8, K, 16, 64,
                                                         16, 16, 8, 1024, 16, 256, wsb, None)
        assert fp8(eneed - 1) == WORKSPACE and fp8(eneed) != WORKSPACE
        bneed = L.sa_sparse_attn_block_tail_workspace_size(B, T, 64, 512, K, 8, 1024)
        tail = lambda wsb: L.sa_sparse_attn_block_tail(16, 16, 16, 16, 0.1, B, T, 64, 512, 8, K, 16, 64, 16,
                                                       8, 1024, 16, 5120, 16, 256, wsb, None)
        assert tail(bneed - 1) == WORKSPACE and tail(bneed) != WORKSPACE


def test_fp4_quantize_host_checks(lib):
    """sa_fp4_quantize refuses bad sizes and misaligned pointers before any
    CUDA call (pointers are never dereferenced); zero rows is a no-op."""
    q = lib.sa_fp4_quantize
    assert q(256, -1, 512, 512, 256, 256, None) == INVALID
    assert q(256, 4, 512, 500, 256, 256, None) == INVALID      # D not a multiple of 16
    assert q(256, 4, 500, 512, 256, 256, None) == INVALID      # row stride below D
    assert q(256, 4, 516, 512, 256, 256, None) == INVALID      # row stride not a multiple of 8
    assert q(264, 4, 512, 512, 256, 256, None) == INVALID      # latent not 16-byte aligned
    assert q(256, 4, 512, 512, 260, 256, None) == INVALID      # codes not 8-byte aligned
    assert q(None, 4, 512, 512, 256, 256, None) == INVALID
    assert q(None, 0, 512, 512, None, None, None) == OK       # no rows: nothing to do
