"""The checked build (libsa_checked.so: the kernels test every address they
compute from run-time values before using it, and a failed test sets the
error word's bounds bit) gives bit for bit the normal build's results and
reports no failure, on every entry point and schedule: list pieces merged in
a cluster, whole queries per CTA, two sources, fp4 rows, the fused tails with
bf16 and fp8 weights (decoded in the GEMM and decoded first), the block tail,
the workspace-free call, top-k and the fp4 quantization."""
import ctypes

import pytest
import torch

import sparse_latent_attention_02_gb300 as sa
from sparse_latent_attention_02_gb300 import inputs as I

from parity_util import to_dev

pytestmark = pytest.mark.gpu

SCALE = 512 ** -0.5


@pytest.fixture(scope="module", autouse=True)
def _built():
    sa.build()
    yield
    sa.library(sa._LIB_PATH)


def both(fn):
    """fn() with the normal library, then with the checked one (the calls
    inside pass check=True, so a bounds failure raises SAError)."""
    sa.library(sa._LIB_PATH)
    a = fn()
    torch.cuda.synchronize()
    sa.library(checked=True)
    try:
        b = fn()
        torch.cuda.synchronize()
    finally:
        sa.library(sa._LIB_PATH)
    return a, b


def _attn_inputs(B, T, K, N, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, T, 64, 512, generator=g).to(torch.bfloat16)
    kv = I.rms_rows(torch.randn(B, N, 512, generator=g)).to(torch.bfloat16)
    sink = torch.randn(64, generator=g)
    idx = torch.randint(0, N, (B, T, K), generator=g, dtype=torch.int32)
    idx[torch.rand(B, T, K, generator=g) < 0.1] = -1
    return to_dev(dict(q=q, kv=kv, sink=sink, idx=idx))


@pytest.mark.parametrize("B,T,K,N,dt", [
    (4, 1, 640, 4224, torch.bfloat16),   # decode shape: list pieces, cluster merge
    (1, 200, 300, 600, torch.float32),   # whole queries per CTA, fp32 output
    (3, 5, 1000, 2000, torch.bfloat16),  # eight pieces a query
])
def test_checked_attention(B, T, K, N, dt):
    x = _attn_inputs(B, T, K, N, seed=B * 7 + K)
    a, b = both(lambda: sa.sparse_attn(x["q"], x["kv"], x["sink"], x["idx"], SCALE, out_dtype=dt, check=True))
    assert torch.equal(a, b)


def test_checked_two_sources_bf16_and_fp4():
    B, T, K, W, C = 3, 2, 256, 128, 900
    g = torch.Generator().manual_seed(11)
    D = 512
    win = I.rms_rows(torch.randn(B + 1, W + 8, D, generator=g)).to(torch.bfloat16).cuda()
    cmp_ = I.rms_rows(torch.randn(B + 1, C + 16, D, generator=g)).to(torch.bfloat16).cuda()
    codes = torch.randint(0, 256, (B + 1, C + 16, D // 2), generator=g, dtype=torch.int32).to(torch.uint8).cuda()
    scales = (0x20 + torch.randint(0, 8, (B + 1, C + 16, D // 16), generator=g)).to(torch.uint8).cuda()
    x = to_dev(dict(q=torch.randn(B, T, 64, D, generator=g).to(torch.bfloat16), sink=torch.randn(64, generator=g),
                    idx=torch.randint(-1, W + C, (B, T, K), generator=g, dtype=torch.int32)))
    a, b = both(lambda: sa.sparse_attn_two_source(x["q"], win, cmp_, x["sink"], x["idx"], SCALE, W=W, C=C,
                                                  check=True))
    assert torch.equal(a, b)
    a, b = both(lambda: sa.sparse_attn_two_source_fp4(x["q"], win, codes, scales, x["sink"], x["idx"], SCALE,
                                                      W=W, C=C, check=True))
    assert torch.equal(a, b)


@pytest.mark.parametrize("T", [300, 600])   # fp8 weight decoded in the GEMM / decoded first
def test_checked_tails(T):
    B, K, N, G, R = 1, 192, 400, 8, 512
    x = _attn_inputs(B, T, K, N, seed=T)
    g = torch.Generator().manual_seed(T + 1)
    w = 0.02 * torch.randn(G, R, 64 * 512 // G, generator=g)
    w16 = w.to(torch.bfloat16).cuda()
    w8, sc = I.fp8_weight(w)
    w8, sc = w8.cuda(), sc.cuda()
    wo_b = (0.02 * torch.randn(512, G * R, generator=g)).to(torch.bfloat16).cuda()
    rope = sa.rope_table(160000.0, 0, T, 64).cuda()
    a, b = both(lambda: sa.sparse_attn_rope_wo_a(x["q"], x["kv"], x["sink"], x["idx"], SCALE, rope, w16,
                                                 check=True))
    assert torch.equal(a, b)
    a, b = both(lambda: sa.sparse_attn_rope_wo_a_fp8(x["q"], x["kv"], x["sink"], x["idx"], SCALE, rope, w8, sc,
                                                     check=True))
    assert torch.equal(a, b)
    a, b = both(lambda: sa.sparse_attn_block_tail(x["q"], x["kv"], x["sink"], x["idx"], SCALE, rope, w16, wo_b,
                                                  check=True))
    assert torch.equal(a, b)


def _noalloc(x):
    """The workspace-free call through the C ABI; its error word must read clean."""
    lib = sa.library()
    B, T = x["q"].shape[:2]
    out = torch.empty(B, T, 64, 512, dtype=torch.bfloat16, device="cuda")
    scratch = ctypes.c_void_p()
    st = torch.cuda.current_stream().cuda_stream
    code = lib.sa_sparse_attn_noalloc(x["q"].data_ptr(), x["kv"].data_ptr(), x["sink"].data_ptr(),
                                      x["idx"].data_ptr(), SCALE, B, T, 64, 512, x["kv"].shape[1],
                                      x["idx"].shape[2], out.data_ptr(), 0, ctypes.byref(scratch), st)
    assert code == 0
    assert lib.sa_check_errors(scratch.value, st) == 0
    return out


def test_checked_noalloc_and_topk():
    x = _attn_inputs(2, 3, 640, 1000, seed=5)
    a, b = both(lambda: _noalloc(x))
    assert torch.equal(a, b)
    g = torch.Generator(device="cuda").manual_seed(3)
    for L, k in ((4096, 512), (40000, 700)):
        sc = torch.randn((64, L), generator=g, device="cuda")
        sc[:, L // 2:] = torch.where(sc[:, L // 2:] > 1.5, float("-inf"), sc[:, L // 2:])
        a, b = both(lambda: sa.topk_indices(sc, k, offset=128))
        assert torch.equal(a, b)
    lat = I.rms_rows(torch.randn(300, 512, generator=torch.Generator().manual_seed(4))).to(torch.bfloat16).cuda()
    (ca, sa_), (cb, sb) = both(lambda: sa.fp4_quantize(lat))
    assert torch.equal(ca, cb) and torch.equal(sa_, sb)
