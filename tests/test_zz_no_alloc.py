"""The workspace-free entry point (`sa_sparse_attn_noalloc`), for callers that
cannot allocate device memory where they run attention.

Its scratch is a static array inside the library, shared by every call and
never cleared between calls except for the error word.  The test calls it
twice in a row through the C ABI, on different inputs, and checks each output
against the ordinary `sa_sparse_attn` (own workspace) on the same inputs; the
second call must not see anything left over from the first.  It lives in a
file of its own, collected last, and passes alone in a fresh process too.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import sparse_latent_attention_02_gb300 as sa
from sparse_latent_attention_02_gb300 import inputs as I

from parity_util import compare

pytestmark = pytest.mark.gpu


def _inputs(seed, B, T, K, N, bad=False, kv_scale=1.0):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, T, 64, 512, generator=g).to(torch.bfloat16).cuda()
    kv = (I.rms_rows(torch.randn(B, N, 512, generator=g)) * kv_scale).to(torch.bfloat16).cuda()
    sink = torch.randn(64, generator=g).cuda()
    idx = torch.randint(0, N, (B, T, K), generator=g, dtype=torch.int32)
    idx[torch.rand(B, T, K, generator=g) < 0.1] = -1
    if bad:
        idx[0, 0, 3] = N + 5
    return q, kv, sink, idx.cuda()


def _noalloc(lib, q, kv, sink, idx, out):
    B, T, H, D = q.shape
    scratch = ctypes.c_void_p()
    code = lib.sa_sparse_attn_noalloc(q.data_ptr(), kv.data_ptr(), sink.data_ptr(),
                                      idx.data_ptr(), 512 ** -0.5, B, T, H, D, kv.shape[1],
                                      idx.shape[2], out.data_ptr(),
                                      1 if out.dtype == torch.float32 else 0,
                                      ctypes.byref(scratch),
                                      torch.cuda.current_stream().cuda_stream)
    return code, scratch.value


@pytest.mark.parametrize("B,T,K,N,dtype,kv_scale", [
    (8, 1, 640, 4224, torch.bfloat16, 1.0),     # few queries: split lists merged inside a cluster
    (8, 1, 640, 4224, torch.float32, 1e5),      # the same, kv far above fp16's range
    (2, 100, 300, 700, torch.float32, 1.0),     # enough queries for whole lists per CTA
])
def test_noalloc_matches_workspace_entry_two_calls(B, T, K, N, dtype, kv_scale):
    sa.build()
    lib = sa.library()
    for call, seed in enumerate((101, 202)):
        q, kv, sink, idx = _inputs(seed + B, B, T, K, N, kv_scale=kv_scale)
        out = torch.empty(B, T, 64, 512, dtype=dtype, device="cuda")
        code, scratch = _noalloc(lib, q, kv, sink, idx, out)
        assert code == 0, sa.SAError(code, "sa_sparse_attn_noalloc")
        assert scratch
        lib_code = lib.sa_check_errors(scratch, torch.cuda.current_stream().cuda_stream)
        assert lib_code == 0
        ref = sa.sparse_attn(q, kv, sink, idx, 512 ** -0.5, out_dtype=dtype, check=True)
        torch.cuda.synchronize()
        compare(out.double().cpu().numpy() / kv_scale, ref.double().cpu().numpy() / kv_scale,
                f"call {call}")
        if kv_scale != 1.0:
            # and against the oracle itself
            want, bad = oracle.sparse_attn(q.cpu(), kv.cpu(), sink.cpu(), idx.cpu(), 512 ** -0.5)
            assert bad == 0
            compare(out.double().cpu().numpy() / kv_scale, want / kv_scale, f"call {call} vs oracle")


def test_noalloc_reports_errors_per_call():
    sa.build()
    lib = sa.library()
    q, kv, sink, idx = _inputs(7, 4, 1, 640, 1000, bad=True)
    out = torch.empty(4, 1, 64, 512, dtype=torch.bfloat16, device="cuda")
    code, scratch = _noalloc(lib, q, kv, sink, idx, out)
    assert code == 0
    assert lib.sa_check_errors(scratch, torch.cuda.current_stream().cuda_stream) == 4
    # the next clean call starts from a cleared error word
    q, kv, sink, idx = _inputs(8, 4, 1, 640, 1000)
    code, scratch = _noalloc(lib, q, kv, sink, idx, out)
    assert code == 0
    assert lib.sa_check_errors(scratch, torch.cuda.current_stream().cuda_stream) == 0


def test_noalloc_rejects_bad_arguments_before_enqueueing():
    sa.build()
    lib = sa.library()
    scratch = ctypes.c_void_p()
    code = lib.sa_sparse_attn_noalloc(16, 16, 16, 16, 0.1, 1, 1, 32, 512, 8, 4, 16, 0,
                                      ctypes.byref(scratch), None)
    assert code == 2 and scratch.value is None
