"""Failure detection on the GPU without a GPU fault.

Every wait inside the kernels is bounded.  With SA_TEST_HOLD_LISTS=n the
first n attention calls of the process withhold their first index list (a
flag that nothing sets), so every role's wait in both CTAs of a pair runs out
after SA_WAIT_TIMEOUT_MS; the kernel must leave cleanly, report
SA_ERR_TIMEOUT through the workspace error word, and leave the CUDA context
usable: the calls after them must match the oracle.  The test runs in a
child process so that its short wait limit and the hold (read once per
process) do not reach the other tests.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

CHILD = r"""
import os, sys, time
sys.path.insert(0, os.environ["SA_REPO"])
sys.path.insert(0, os.path.join(os.environ["SA_REPO"], "tests"))
import torch
import oracle
import sparse_latent_attention_02_gb300 as sa
from sparse_latent_attention_02_gb300 import inputs as I
from parity_util import compare

g = torch.Generator().manual_seed(5)
cases = []
# one query per CTA pair, then pairs that walk several queries
for B, T, K, N in [(1, 4, 300, 500), (2, 90, 200, 400)]:
    q = torch.randn(B, T, 64, 512, generator=g).to(torch.bfloat16)
    kv = I.rms_rows(torch.randn(B, N, 512, generator=g)).to(torch.bfloat16)
    sink = torch.randn(64, generator=g)
    idx = torch.randint(0, N, (B, T, K), generator=g, dtype=torch.int32)
    dev = (q.cuda(), kv.cuda(), sink.cuda(), idx.cuda())
    ws = torch.zeros(sa.workspace_size(B, T, K), dtype=torch.uint8, device="cuda")
    cases.append(((B, T), (q, kv, sink, idx), dev, ws))
# the first two calls of this process are held (SA_TEST_HOLD_LISTS=2)
for (B, T), _, (dq, dkv, ds, di), ws in cases:
    t0 = time.time()
    sa.sparse_attn(dq, dkv, ds, di, 512 ** -0.5, workspace=ws)
    try:
        sa.check_errors(ws)
        raise SystemExit("no timeout reported")
    except sa.SAError as e:
        assert e.code == 5, e
    held = time.time() - t0
    assert held < 5.0, held
    print(f"B{B} T{T}: timeout reported after {held:.2f} s")
# the context survives: the next calls match the oracle
for (B, T), (q, kv, sink, idx), (dq, dkv, ds, di), ws in cases:
    out = sa.sparse_attn(dq, dkv, ds, di, 512 ** -0.5, workspace=ws, out_dtype=torch.float32)
    sa.check_errors(ws)
    ref, _ = oracle.sparse_attn(q, kv, sink, idx, 512 ** -0.5)
    compare(out.double().cpu().numpy(), ref, f"after timeout B{B} T{T}")
    print(f"B{B} T{T}: next call correct")
print("ok")
"""


def test_bounded_wait_runs_out_and_context_survives():
    import sparse_latent_attention_02_gb300 as sa
    sa.build()
    repo = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, SA_REPO=repo, SA_WAIT_TIMEOUT_MS="100", SA_TEST_HOLD_LISTS="2")
    r = subprocess.run([sys.executable, "-c", CHILD], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "ok" in r.stdout
