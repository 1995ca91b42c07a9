"""GPU parity: the sm_103a kernels against the fp64 oracle on the same seeded
inputs, through the C ABI.  Index handling is checked exactly (one-hot index
probe, skip handling, error reporting); values within max-abs 2e-2 and
relative Frobenius 5e-3."""
import numpy as np
import pytest
import torch

import oracle
import sparse_latent_attention_02_gb300 as sa
from sparse_latent_attention_02_gb300 import inputs as I

from parity_util import cached_workspace, compare, oracle_rows, sample_queries, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    sa.build()
    sa.library()
    oracle.build()


def run(x, scale, out_dtype=torch.bfloat16):
    g = to_dev(x)
    out = sa.sparse_attn(g["q"], g["kv"], g["sink"], g["idx"], scale, out_dtype=out_dtype)
    ws = cached_workspace("attn")
    sa.check_errors(ws)
    return out


def full_oracle(x, scale):
    ref, bad = oracle.sparse_attn(x["q"], x["kv"], x["sink"], x["idx"], scale)
    assert bad == 0
    return ref


# ---------------------------------------------------------------- the five workloads


def test_tiny_workload_fp32():
    wl = I.WORKLOADS["tiny"]
    x = I.make_inputs(wl, seed=0)
    got = run(x, wl.scale, torch.float32)
    compare(got.double().cpu().numpy(), full_oracle(x, wl.scale), "tiny")


def test_decode_workload_all_queries():
    wl = I.WORKLOADS["decode"]
    x = I.make_inputs(wl, seed=1, device="cuda")
    got = run(x, wl.scale)
    ref = oracle_rows(x, np.arange(wl.n_queries), wl.scale)
    compare(got.reshape(-1, 64, 512).double().cpu().numpy(), ref, "decode")


def test_long_decode_workload_all_queries():
    wl = I.WORKLOADS["long_decode"]
    x = I.make_inputs(wl, seed=2, device="cuda")
    got = run(x, wl.scale)
    ref = oracle_rows(x, np.arange(wl.n_queries), wl.scale)
    compare(got.reshape(-1, 64, 512).double().cpu().numpy(), ref, "long_decode")
    del x, got
    torch.cuda.empty_cache()


def test_prefill_workload_all_queries():
    """Every one of the 8192 queries against the oracle, block by block (each
    block of 1024 queries within the bound on its own)."""
    wl = I.WORKLOADS["prefill"]
    x = I.make_inputs(wl, seed=3, device="cuda")
    got = run(x, wl.scale).reshape(-1, 64, 512)
    for q0 in range(0, wl.n_queries, 1024):
        qs = np.arange(q0, min(q0 + 1024, wl.n_queries))
        ref = oracle_rows(x, qs, wl.scale)
        compare(got[q0:q0 + len(qs)].double().cpu().numpy(), ref, f"prefill queries {q0}..{qs[-1]}")


def test_fused_tail_workload_rows():
    """Attention, inverse RoPE and grouped wo_a on the fused-tail workload:
    544 rows against the fp64 oracle chain, among them both rows on either side
    of every 128-token tile boundary of the GEMM and both batch elements' ends."""
    wl = I.WORKLOADS["fused_tail"]
    x = I.make_inputs(wl, seed=4, device="cuda")
    rope = sa.rope_table(wl.theta, 0, wl.T, wl.rope_dim).cuda()
    y = sa.sparse_attn_rope_wo_a(x["q"], x["kv"], x["sink"], x["idx"], wl.scale, rope, x["wo_a"])
    sa.check_errors(cached_workspace("fused"))
    edges = [r for m in range(128, wl.n_queries, 128) for r in (m - 1, m)]
    qs = sample_queries(wl.n_queries, 544 - len(edges) - 4, seed=4,
                        include=[0, 4095, 4096, 8191] + edges)
    assert len(qs) >= 512
    o = oracle_rows(x, qs, wl.scale)
    o = oracle.inverse_rope(o, qs % wl.T, wl.rope_dim, wl.theta)
    yref = oracle.wo_a(o.reshape(len(qs), wl.G, -1), x["wo_a"].cpu())
    got = y.reshape(-1, wl.G * wl.R)[torch.as_tensor(qs, device="cuda")].double().cpu().numpy()
    compare(got, yref.reshape(len(qs), -1), "fused_tail")


# ---------------------------------------------------------------- schedules and shapes


@pytest.mark.parametrize("B,T,K,N", [
    (2, 80, 192, 300),     # 160 queries >= SM count: whole lists per CTA
    (3, 5, 640, 700),      # few queries: lists cut into pieces + combine
    (1, 1, 1000, 2000),    # one query spread over many CTAs
    (7, 3, 129, 150),      # ragged chunk tail (129 = 128 + 1)
    (1, 200, 1, 10),       # one entry per list
    (2, 2, 1024, 4096),    # longest list
])
def test_shapes_and_schedules(B, T, K, N):
    g = torch.Generator().manual_seed(B * 1000 + T * 10 + K)
    q = torch.randn(B, T, 64, 512, generator=g).to(torch.bfloat16)
    kv = I.rms_rows(torch.randn(B, N, 512, generator=g)).to(torch.bfloat16)
    sink = torch.randn(64, generator=g)
    idx = torch.randint(0, N, (B, T, K), generator=g, dtype=torch.int32)
    idx[torch.rand(B, T, K, generator=g) < 0.2] = -1
    x = dict(q=q, kv=kv, sink=sink, idx=idx)
    got = run(x, 512 ** -0.5)
    compare(got.double().cpu().numpy(), full_oracle(x, 512 ** -0.5), f"B{B} T{T} K{K}")


def test_empty_and_all_skip_lists():
    g = torch.Generator().manual_seed(7)
    B, T, K, N = 2, 9, 300, 64
    q = torch.randn(B, T, 64, 512, generator=g).to(torch.bfloat16)
    kv = I.rms_rows(torch.randn(B, N, 512, generator=g)).to(torch.bfloat16)
    sink = torch.randn(64, generator=g)
    idx = torch.randint(0, N, (B, T, K), generator=g, dtype=torch.int32)
    idx[0, 3] = -1
    idx[1, 8] = -1
    idx[1, 0, 150:] = -1
    x = dict(q=q, kv=kv, sink=sink, idx=idx)
    got = run(x, 512 ** -0.5, torch.float32)
    assert torch.count_nonzero(got[0, 3]) == 0 and torch.count_nonzero(got[1, 8]) == 0
    compare(got.double().cpu().numpy(), full_oracle(x, 512 ** -0.5), "all-skip rows")
    # K == 0: all-zero output
    z = run(dict(q=q, kv=kv, sink=sink, idx=torch.zeros(B, T, 0, dtype=torch.int32)), 0.1)
    assert torch.count_nonzero(z) == 0


def test_index_probe_exact():
    """q = 0, sink = -inf, row r of kv = e_r: o * (valid count) are the exact
    multiplicities of each row in the list (fp32 output, powers of two exact)."""
    N, K, T = 512, 256, 12
    kv = torch.eye(N, 512).unsqueeze(0).to(torch.bfloat16)
    q = torch.zeros(1, T, 64, 512, dtype=torch.bfloat16)
    sink = torch.full((64,), float("-inf"))
    g = torch.Generator().manual_seed(11)
    idx = torch.randint(0, N, (1, T, K), generator=g, dtype=torch.int32)
    # make the valid count a power of two in every list: 128 or 256 or 64 valid entries
    for t in range(T):
        keep = [256, 128, 64, 32][t % 4]
        idx[0, t, torch.randperm(K, generator=g)[:K - keep]] = -1
    got = run(dict(q=q, kv=kv, sink=sink, idx=idx), 1.0, torch.float32).cpu()
    for t in range(T):
        valid = idx[0, t][idx[0, t] >= 0].long()
        counts = torch.bincount(valid, minlength=N).float()
        want = counts / valid.numel()
        assert torch.equal(got[0, t], want.expand(64, N)), f"query {t}"


def test_bad_index_reported_and_skipped():
    g = torch.Generator().manual_seed(13)
    B, T, K, N = 1, 4, 200, 100
    q = torch.randn(B, T, 64, 512, generator=g).to(torch.bfloat16)
    kv = I.rms_rows(torch.randn(B, N, 512, generator=g)).to(torch.bfloat16)
    sink = torch.randn(64, generator=g)
    idx = torch.randint(0, N, (B, T, K), generator=g, dtype=torch.int32)
    clean = idx.clone()
    idx[0, 1, 7] = N          # out of range
    idx[0, 2, 50] = -5        # negative other than -1
    clean[0, 1, 7] = -1
    clean[0, 2, 50] = -1
    gd = to_dev(dict(q=q, kv=kv, sink=sink, idx=idx))
    out = sa.sparse_attn(gd["q"], gd["kv"], gd["sink"], gd["idx"], 512 ** -0.5,
                         out_dtype=torch.float32)
    with pytest.raises(sa.SAError) as e:
        sa.check_errors(cached_workspace("attn"))
    assert e.value.code == 4
    ref = full_oracle(dict(q=q, kv=kv, sink=sink, idx=clean), 512 ** -0.5)
    compare(out.double().cpu().numpy(), ref, "bad index skipped")
    # the error word was cleared by the read
    sa.check_errors(cached_workspace("attn"))


@pytest.mark.parametrize("mode", ["sink_minus_inf", "dominant_sink", "wide_logits"])
def test_sink_and_rescale_paths(mode):
    g = torch.Generator().manual_seed(17)
    B, T, K, N = 2, 3, 640, 700
    q = torch.randn(B, T, 64, 512, generator=g)
    kv = I.rms_rows(torch.randn(B, N, 512, generator=g))
    sink = torch.randn(64, generator=g)
    idx = torch.stack([torch.randperm(N, generator=g)[:K] for _ in range(B * T)]).reshape(B, T, K)
    idx = idx.to(torch.int32)
    if mode == "sink_minus_inf":
        sink = torch.full((64,), float("-inf"))
    elif mode == "dominant_sink":
        sink = torch.full((64,), 8.0)
        q = q * 4
    else:
        # scores grow along the list, so the running maximum moves chunk after chunk
        ramp = torch.linspace(0.0, 0.7, N).unsqueeze(-1)
        kv = kv * (1.0 + ramp)
        idx, _ = torch.sort(idx, dim=-1)
        q = q.abs() + 0.2
        kv = kv.abs()
    x = dict(q=q.to(torch.bfloat16), kv=kv.to(torch.bfloat16), sink=sink, idx=idx)
    got = run(x, 512 ** -0.5, torch.float32)
    compare(got.double().cpu().numpy(), full_oracle(x, 512 ** -0.5), mode)


@pytest.mark.parametrize("B,T,K,N", [
    (64, 1, 640, 1000),    # two list pieces per query
    (4, 1, 640, 1000),     # four pieces
    (1, 1, 1000, 2000),    # eight pieces
])
@pytest.mark.parametrize("case", ["kv_times_1e5", "kv_times_1e-5", "sink_20", "sink_100"])
def test_split_merge_extreme_magnitudes(B, T, K, N, case):
    """The pieces of a split list merge through distributed shared memory as
    fp16 after a per-head power-of-two scaling: kv far above fp16's range
    (|v| up to ~4e5), far below its normal range, a sink that leaves tiny row
    sums (20) and one that leaves none at all (100: every probability below
    float's normal range) all match the oracle, relative to their own scale."""
    g = torch.Generator().manual_seed(29 + B + K)
    q = torch.randn(B, T, 64, 512, generator=g)
    kv = I.rms_rows(torch.randn(B, N, 512, generator=g))
    sink = torch.randn(64, generator=g)
    idx = torch.randint(0, N, (B, T, K), generator=g, dtype=torch.int32)
    idx[torch.rand(B, T, K, generator=g) < 0.1] = -1
    scale = 1.0
    if case == "kv_times_1e5":
        kv, scale = kv * 1e5, 1e5
    elif case == "kv_times_1e-5":
        kv, scale = kv * 1e-5, 1e-5
    elif case == "sink_20":
        sink = torch.full((64,), 20.0)
    else:
        sink = torch.full((64,), 100.0)
    x = dict(q=q.to(torch.bfloat16), kv=kv.to(torch.bfloat16), sink=sink, idx=idx)
    got = run(x, 512 ** -0.5, torch.float32).double().cpu().numpy()
    ref = full_oracle(x, 512 ** -0.5)
    assert np.all(np.isfinite(got))
    if case == "sink_100":
        # the exact outputs are ~1e-41: zero within any absolute bound
        assert np.abs(got - ref).max() <= 1e-30
    elif case == "sink_20":
        # outputs ~1e-5: compared relative to their own magnitude
        s_ref = np.abs(ref).max()
        compare(got / s_ref, ref / s_ref, case)
    else:
        compare(got / scale, ref / scale, case)


def test_repeated_indices_count_twice():
    g = torch.Generator().manual_seed(19)
    q = torch.randn(1, 2, 64, 512, generator=g).to(torch.bfloat16)
    kv = I.rms_rows(torch.randn(1, 50, 512, generator=g)).to(torch.bfloat16)
    sink = torch.randn(64, generator=g)
    idx = torch.randint(0, 5, (1, 2, 300), generator=g, dtype=torch.int32)   # many repeats
    x = dict(q=q, kv=kv, sink=sink, idx=idx)
    got = run(x, 512 ** -0.5, torch.float32)
    compare(got.double().cpu().numpy(), full_oracle(x, 512 ** -0.5), "repeats")


def test_repeat_calls_are_deterministic():
    wl = I.scaled(I.WORKLOADS["decode"], B=8)
    x = to_dev(I.make_inputs(wl, seed=5))
    a = sa.sparse_attn(x["q"], x["kv"], x["sink"], x["idx"], wl.scale)
    b = sa.sparse_attn(x["q"], x["kv"], x["sink"], x["idx"], wl.scale)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_kv_in_pinned_host_memory():
    """kv left in page-locked host memory: the kernel gathers the listed rows
    straight from there; the result is bit-identical to kv in device memory.
    Pageable host memory is refused before anything is enqueued."""
    g = torch.Generator().manual_seed(23)
    for B, T, K, N in [(4, 1, 640, 1000), (1, 200, 300, 500)]:   # split and whole schedules
        q = torch.randn(B, T, 64, 512, generator=g).to(torch.bfloat16)
        kv = I.rms_rows(torch.randn(B, N, 512, generator=g)).to(torch.bfloat16)
        sink = torch.randn(64, generator=g)
        idx = torch.randint(0, N, (B, T, K), generator=g, dtype=torch.int32)
        idx[torch.rand(B, T, K, generator=g) < 0.1] = -1
        x = dict(q=q, kv=kv, sink=sink, idx=idx)
        on_device = run(x, 512 ** -0.5, torch.float32)
        gd = to_dev(x)
        on_host = sa.sparse_attn(gd["q"], kv.pin_memory(), gd["sink"], gd["idx"], 512 ** -0.5,
                                 out_dtype=torch.float32, check=True)
        assert torch.equal(on_host, on_device), f"B{B} T{T}"
        compare(on_host.double().cpu().numpy(), full_oracle(x, 512 ** -0.5), f"host kv B{B} T{T}")
    # pageable memory: refused by the binding, and by the C ABI itself
    pageable = kv.clone()
    with pytest.raises(ValueError):
        sa.sparse_attn(gd["q"], pageable, gd["sink"], gd["idx"], 0.1)
    lib = sa.library()
    out = torch.empty(1, T, 64, 512, dtype=torch.float32, device="cuda")
    ws = cached_workspace("attn")
    code = lib.sa_sparse_attn(gd["q"].data_ptr(), pageable.data_ptr(), gd["sink"].data_ptr(),
                              gd["idx"].data_ptr(), 0.1, 1, T, 64, 512, N, K, out.data_ptr(), 1,
                              ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
    assert code == 1   # SA_ERR_INVALID_ARG


@pytest.mark.parametrize("B,T,K,W,C,host_c", [
    (4, 1, 640, 128, 4096, False),    # decode shape, split schedule
    (1, 40, 300, 128, 600, False),    # whole queries per CTA
    (2, 3, 200, 0, 500, False),       # compressed rows only
    (2, 3, 100, 128, 0, False),       # window rows only
    (3, 2, 256, 128, 900, True),      # compressed cache in page-locked host memory
])
def test_two_source_matches_concatenation(B, T, K, W, C, host_c):
    """The window ring and the compressed cache read in place (caches larger
    than the rows in use, their padding NaN) give exactly the result of one
    kv made by concatenating the rows in use, and match the oracle."""
    g = torch.Generator().manual_seed(B * 100 + K)
    D = 512
    nan_bf16 = torch.tensor(float("nan"), dtype=torch.bfloat16)
    win = torch.full((B + 1, W + 8, D), nan_bf16.item(), dtype=torch.bfloat16)
    cmp_ = torch.full((B + 1, C + 16, D), nan_bf16.item(), dtype=torch.bfloat16)
    win[:B, :W] = I.rms_rows(torch.randn(B, W, D, generator=g)).to(torch.bfloat16)
    cmp_[:B, :C] = I.rms_rows(torch.randn(B, C, D, generator=g)).to(torch.bfloat16)
    q = torch.randn(B, T, 64, D, generator=g).to(torch.bfloat16)
    sink = torch.randn(64, generator=g)
    idx = torch.randint(0, W + C, (B, T, K), generator=g, dtype=torch.int32)
    idx[torch.rand(B, T, K, generator=g) < 0.1] = -1
    gd = to_dev(dict(q=q, sink=sink, idx=idx))
    win_d = win.cuda() if W else None
    cmp_d = (cmp_.pin_memory() if host_c else cmp_.cuda()) if C else None
    got = sa.sparse_attn_two_source(gd["q"], win_d, cmp_d, gd["sink"], gd["idx"], 512 ** -0.5,
                                    W=W, C=C, out_dtype=torch.float32, check=True)
    cat = torch.cat([win[:B, :W], cmp_[:B, :C]], dim=1).contiguous()
    one = sa.sparse_attn(gd["q"], cat.cuda(), gd["sink"], gd["idx"], 512 ** -0.5,
                         out_dtype=torch.float32, check=True)
    assert torch.equal(got, one)
    ref, bad = oracle.sparse_attn_two_source(q, win, W, cmp_, C, sink, idx, 512 ** -0.5)
    assert bad == 0
    compare(got.double().cpu().numpy(), ref, f"two sources B{B} W{W} C{C}")


def test_block_tail_workload_sampled():
    """sparse_attn -> inverse RoPE -> grouped wo_a -> wo_b on the block-tail
    workload, sampled rows against the fp64 chain of oracle steps."""
    wl = I.WORKLOADS["block_tail"]
    x = I.make_inputs(wl, seed=4, device="cuda")
    rope = sa.rope_table(wl.theta, 0, wl.T, wl.rope_dim).cuda()
    z = sa.sparse_attn_block_tail(x["q"], x["kv"], x["sink"], x["idx"], wl.scale, rope, x["wo_a"],
                                  x["wo_b"], check=True)
    edges = [r for m in range(512, wl.n_queries, 512) for r in (m - 1, m)]
    qs = sample_queries(wl.n_queries, 96, seed=5, include=[0, 4095, 4096, 8191] + edges)
    o = oracle_rows(x, qs, wl.scale)
    o = oracle.inverse_rope(o, qs % wl.T, wl.rope_dim, wl.theta)
    y = oracle.wo_a(o.reshape(len(qs), wl.G, -1), x["wo_a"].cpu())
    zref = oracle.wo_b(y.reshape(len(qs), -1), x["wo_b"].cpu())
    got = z.reshape(-1, wl.dim)[torch.as_tensor(qs, device="cuda")].double().cpu().numpy()
    # wo_b's outputs reach several units: each may also differ by 2^-7 of its magnitude
    # (its own bf16 rounding is 2^-9)
    compare(got, zref, "block_tail", per_value=True)


@pytest.mark.parametrize("rows,L,k,mode", [
    (256, 4096, 512, "causal"),   # prefill-like: the visible prefix grows row by row
    (64, 4096, 512, "full"),      # decode-like
    (8, 65536, 512, "full"),      # long context: keys re-read from L2 on every pass
    (32, 1000, 512, "ties"),      # many equal scores: ties go to the smaller position
    (16, 300, 512, "masked"),     # NaN and -inf, fewer than k positions to choose
    (4, 0, 16, "empty"),          # no positions at all
    (24, 1030, 64, "narrow"),     # scores a few ulps apart and signed zeros: the low digits decide
    (24, 1030, 64, "tiny"),       # subnormals, signed zeros and -inf: subnormals are not zero
    (4, 16383, 512, "full"),      # the longest row whose keys stay in shared memory
    (4, 16385, 512, "full"),      # the shortest row read again from L2 on every pass
    (16, 1024, 512, "cluster"),   # every key in one first-pass bin: the later digits decide
    (16, 1025, 512, "cluster"),   # the same with a ragged last group of four keys
    (16, 4096, 512, "cluster"),   # scores 1.1 + 1e-4 N(0,1): the low digits decide
    (16, 4096, 512, "flat"),      # all equal but 10% masked: ties decide every position
    (8, 20000, 512, "cluster"),   # the same with the keys read again from L2
])
def test_topk_matches_oracle(rows, L, k, mode):
    """The top-k selection is exact: the same int32 positions, in the same
    order, as the oracle's sort."""
    g = torch.Generator().manual_seed(rows * 7 + L)
    s = torch.randn(rows, L, generator=g)
    if mode == "causal":
        for r in range(rows):
            s[r, (r * L) // rows + 1:] = float("-inf")
    elif mode == "ties":
        s = torch.round(s * 4) / 4
    elif mode == "narrow":
        s = 1.0 + torch.randint(0, 3, (rows, L), generator=g).double() * 2.0 ** -23
        s = s.float()
        s[:, ::7] = -0.0
        s[:, 1::7] = 0.0
    elif mode == "tiny":
        vals = torch.tensor([-1e-40, -0.0, 0.0, 1e-45, 1e-40, 2e-40, float("-inf")])
        s = vals[torch.randint(0, len(vals), (rows, L), generator=g)]
    elif mode == "cluster":
        s = 1.1 + 1e-4 * s   # one top-digit bin: [1, 1.25)
    elif mode == "flat":
        s = torch.ones(rows, L)
        s[torch.rand(rows, L, generator=g) < 0.1] = float("-inf")
    elif mode == "masked":
        s[torch.rand(rows, L, generator=g) < 0.1] = float("nan")
        s[torch.rand(rows, L, generator=g) < 0.2] = float("-inf")
    got = sa.topk_indices(s.cuda(), k, offset=128)
    torch.cuda.synchronize()
    ref = oracle.topk_indices(s.numpy(), k, offset=128)
    assert np.array_equal(got.cpu().numpy(), ref)


def test_topk_unaligned_rows():
    """Rows cut from a wider tensor start on and off 16-byte boundaries, so
    both load paths of the first pass run in one launch; each row ends in a
    masked tail of its own length, one row is masked throughout."""
    g = torch.Generator().manual_seed(77)
    rows, L, k = 48, 2051, 300
    big = torch.randn(rows, L + 1, generator=g)
    for r in range(rows):
        big[r, 1 + (r * 97) % L:] = float("-inf")
    big[5, :] = float("-inf")
    s = big.cuda()[:, 1:]
    assert s.stride(0) == L + 1
    got = sa.topk_indices(s, k, offset=7)
    torch.cuda.synchronize()
    ref = oracle.topk_indices(big[:, 1:].contiguous().numpy(), k, offset=7)
    assert np.array_equal(got.cpu().numpy(), ref)


@pytest.mark.parametrize("B,T,K,W,C,host_c", [
    (4, 1, 640, 128, 4096, False),    # decode shape, split schedule
    (1, 40, 300, 128, 600, False),    # whole queries per CTA
    (2, 3, 200, 0, 500, False),       # fp4 rows only
    (3, 2, 256, 128, 900, True),      # fp4 cache in page-locked host memory
])
def test_two_source_fp4_matches_decoded_cache(B, T, K, W, C, host_c):
    """Compressed rows stored as fp4 (e2m1 codes, an E4M3 scale per 16
    features) give exactly the result of the bf16 call on the decoded cache,
    and match the oracle.  Scale padding is E4M3 NaN: reading any row past C,
    or a spare batch row, would show in the output."""
    g = torch.Generator().manual_seed(B * 31 + C)
    D = 512
    nan_bf16 = float("nan")
    win = torch.full((B + 1, W + 8, D), nan_bf16, dtype=torch.bfloat16)
    win[:B, :W] = I.rms_rows(torch.randn(B, W, D, generator=g)).to(torch.bfloat16)
    codes = torch.randint(0, 256, (B + 1, C + 16, D // 2), generator=g, dtype=torch.int32).to(torch.uint8)
    scales = torch.full((B + 1, C + 16, D // 16), 0x7F, dtype=torch.uint8)
    # positive scales in [0.25, 0.47): with codes drawn uniformly the decoded
    # rows have an RMS near 1, like the RMS-normalised latents they stand for
    scales[:B, :C] = (0x20 + torch.randint(0, 8, (B, C, D // 16), generator=g)).to(torch.uint8)
    q = torch.randn(B, T, 64, D, generator=g).to(torch.bfloat16)
    sink = torch.randn(64, generator=g)
    idx = torch.randint(0, W + C, (B, T, K), generator=g, dtype=torch.int32)
    idx[torch.rand(B, T, K, generator=g) < 0.1] = -1
    gd = to_dev(dict(q=q, sink=sink, idx=idx))
    win_d = win.cuda() if W else None
    place = (lambda t: t.pin_memory()) if host_c else (lambda t: t.cuda())
    got = sa.sparse_attn_two_source_fp4(gd["q"], win_d, place(codes), place(scales), gd["sink"], gd["idx"],
                                        512 ** -0.5, W=W, C=C, out_dtype=torch.float32, check=True)
    decoded = torch.from_numpy(oracle.bf16_bits_exact(
        oracle.dequant_fp4(codes[:B, :C].numpy(), scales[:B, :C].numpy())).view(np.int16)).view(torch.bfloat16)
    ref16 = sa.sparse_attn_two_source(gd["q"], win_d, decoded.cuda(), gd["sink"], gd["idx"], 512 ** -0.5,
                                      W=W, C=C, out_dtype=torch.float32, check=True)
    assert torch.equal(got, ref16)
    ref, bad = oracle.sparse_attn_two_source_fp4(q, win, W, codes.numpy(), scales.numpy(), C, sink, idx,
                                                 512 ** -0.5)
    assert bad == 0
    compare(got.double().cpu().numpy(), ref, f"fp4 two sources B{B} W{W} C{C}")


@pytest.mark.gpu
def test_fp4_every_scale_byte():
    """Every E4M3 scale byte but the two NaNs (zero, subnormals, up to 448)
    and every code byte go through the in-kernel decoding: the result equals
    the bf16 call on the decoded cache bit for bit."""
    g = torch.Generator().manual_seed(5)
    B, T, W, C, D = 2, 3, 8, 16, 512
    win = I.rms_rows(torch.randn(B, W, D, generator=g)).to(torch.bfloat16)
    codes = torch.randint(0, 256, (B, C, D // 2), generator=g, dtype=torch.int32).to(torch.uint8)
    codes[0, 0] = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    sb = torch.arange(B * C * (D // 16), dtype=torch.int32) % 256
    sb[(sb == 0x7F) | (sb == 0xFF)] = 0
    scales = sb.to(torch.uint8).view(B, C, D // 16)
    q = (0.01 * torch.randn(B, T, 64, D, generator=g)).to(torch.bfloat16)
    sink = torch.randn(64, generator=g)
    idx = torch.arange(W + C, dtype=torch.int32).repeat(B, T, 1)
    gd = to_dev(dict(q=q, sink=sink, idx=idx))
    got = sa.sparse_attn_two_source_fp4(gd["q"], win.cuda(), codes.cuda(), scales.cuda(), gd["sink"], gd["idx"],
                                        512 ** -0.5, W=W, C=C, out_dtype=torch.float32, check=True)
    decoded = torch.from_numpy(oracle.bf16_bits_exact(
        oracle.dequant_fp4(codes.numpy(), scales.numpy())).view(np.int16)).view(torch.bfloat16)
    ref16 = sa.sparse_attn_two_source(gd["q"], win.cuda(), decoded.cuda(), gd["sink"], gd["idx"], 512 ** -0.5,
                                      W=W, C=C, out_dtype=torch.float32, check=True)
    assert torch.isfinite(ref16).all()
    assert torch.equal(got, ref16)


@pytest.mark.parametrize("B,T,K,N,G,R", [
    (2, 300, 192, 400, 8, 512),     # 600 tokens: four full 128-token tiles and a ragged one
    (1, 130, 640, 1000, 4, 256),    # wider groups (8192 features per group)
    (3, 7, 64, 100, 16, 256),       # narrow groups (2048 features), one partial tile
])
def test_fused_tail_fp8_matches_dequantized_weight(B, T, K, N, G, R):
    """wo_a kept in fp8 (E4M3 + a scale per 128 x 128 block): the result equals
    the bf16 fused call on the weight the oracle dequantizes, bit for bit, and
    the oracle chain on sampled rows."""
    g = torch.Generator().manual_seed(B * 100 + G)
    q = torch.randn(B, T, 64, 512, generator=g).to(torch.bfloat16)
    kv = I.rms_rows(torch.randn(B, N, 512, generator=g)).to(torch.bfloat16)
    sink = torch.randn(64, generator=g)
    idx = torch.randint(0, N, (B, T, K), generator=g, dtype=torch.int32)
    idx[torch.rand(B, T, K, generator=g) < 0.1] = -1
    w = 0.02 * torch.randn(G, R, 64 * 512 // G, generator=g)
    w8, sc = I.fp8_weight(w)
    wdq = torch.from_numpy(oracle.dequant_fp8_weight(w8.reshape(G * R, -1).numpy(), sc.numpy())
                           .view(np.int16)).view(torch.bfloat16).reshape(G, R, -1)
    rope = sa.rope_table(160000.0, 0, T, 64).cuda()
    x = to_dev(dict(q=q, kv=kv, sink=sink, idx=idx))
    got = sa.sparse_attn_rope_wo_a_fp8(x["q"], x["kv"], x["sink"], x["idx"], 512 ** -0.5, rope, w8.cuda(),
                                       sc.cuda(), check=True)
    ref16 = sa.sparse_attn_rope_wo_a(x["q"], x["kv"], x["sink"], x["idx"], 512 ** -0.5, rope, wdq.cuda(),
                                     check=True)
    assert torch.equal(got, ref16)
    qs = sample_queries(B * T, 12, seed=G, include=(0, B * T - 1))
    o = oracle_rows(dict(q=q, kv=kv, sink=sink, idx=idx), qs, 512 ** -0.5)
    o = oracle.inverse_rope(o, qs % T, 64, 160000.0)
    yref = oracle.wo_a(o.reshape(len(qs), G, -1), wdq)
    compare(got.reshape(-1, G * R)[torch.as_tensor(qs, device="cuda")].double().cpu().numpy(),
            yref.reshape(len(qs), -1), f"fp8 tail G{G}")


@pytest.mark.parametrize("M", [1, 127, 128, 129, 255, 256, 257, 520])
def test_tails_at_pair_tile_edges(M):
    """The bf16 GEMMs run on CTA pairs, each pair a tile of 256 tokens (128
    per CTA): token counts on both sides of 128 and 256, and below 128 where
    the second CTA of the pair holds no token.  Every row of the fused tail
    (G = 8, R = 256) and of a block tail (then wo_b to 512 features) against
    the fp64 chain of oracle steps."""
    g = torch.Generator().manual_seed(7000 + M)
    B, T, K, N, G, R, dim = 1, M, 64, 100, 8, 256, 512
    q = torch.randn(B, T, 64, 512, generator=g).to(torch.bfloat16)
    kv = I.rms_rows(torch.randn(B, N, 512, generator=g)).to(torch.bfloat16)
    sink = torch.randn(64, generator=g)
    idx = torch.randint(0, N, (B, T, K), generator=g, dtype=torch.int32)
    idx[torch.rand(B, T, K, generator=g) < 0.1] = -1
    wa = (0.02 * torch.randn(G, R, 64 * 512 // G, generator=g)).to(torch.bfloat16)
    wb = (0.02 * torch.randn(dim, G * R, generator=g)).to(torch.bfloat16)
    rope = sa.rope_table(160000.0, 0, T, 64).cuda()
    x = to_dev(dict(q=q, kv=kv, sink=sink, idx=idx))
    y = sa.sparse_attn_rope_wo_a(x["q"], x["kv"], x["sink"], x["idx"], 512 ** -0.5, rope, wa.cuda(), check=True)
    z = sa.sparse_attn_block_tail(x["q"], x["kv"], x["sink"], x["idx"], 512 ** -0.5, rope, wa.cuda(), wb.cuda(),
                                  check=True)
    qs = np.arange(B * T)
    o = oracle_rows(dict(q=q, kv=kv, sink=sink, idx=idx), qs, 512 ** -0.5)
    o = oracle.inverse_rope(o, qs % T, 64, 160000.0)
    yref = oracle.wo_a(o.reshape(len(qs), G, -1), wa)
    compare(y.reshape(-1, G * R).double().cpu().numpy(), yref.reshape(len(qs), -1), f"fused tail M{M}")
    zref = oracle.wo_b(yref.reshape(len(qs), -1), wb)
    compare(z.reshape(-1, dim).double().cpu().numpy(), zref, f"block tail M{M}", per_value=True)


def test_fused_calls_on_two_streams_keep_their_own_workspace():
    """Fused calls in flight on two streams at once, each with the binding's
    default workspace (where the attention output waits for the GEMM), give
    exactly what each gives alone."""
    g = torch.Generator().manual_seed(5)
    B, T, K, N, G, R = 2, 300, 192, 400, 8, 512

    def make():
        q = torch.randn(B, T, 64, 512, generator=g).to(torch.bfloat16)
        kv = I.rms_rows(torch.randn(B, N, 512, generator=g)).to(torch.bfloat16)
        sink = torch.randn(64, generator=g)
        idx = torch.randint(0, N, (B, T, K), generator=g, dtype=torch.int32)
        return to_dev(dict(q=q, kv=kv, sink=sink, idx=idx))

    xs = [make(), make()]
    w = (0.02 * torch.randn(G, R, 64 * 512 // G, generator=g)).to(torch.bfloat16).cuda()
    rope = sa.rope_table(160000.0, 0, T, 64).cuda()
    call = lambda x, st=None: sa.sparse_attn_rope_wo_a(x["q"], x["kv"], x["sink"], x["idx"], 512 ** -0.5,
                                                       rope, w, stream=st)
    ref = [call(x) for x in xs]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    outs = []
    for _ in range(4):
        for x, st in zip(xs, streams):
            with torch.cuda.stream(st):
                outs.append(call(x, st))
    torch.cuda.synchronize()
    for i, y in enumerate(outs):
        assert torch.equal(y, ref[i % 2])


def test_fused_tail_fp8_workload_sampled():
    """The fused-tail workload (B=2, T=4096) with its wo_a as an fp8 checkpoint."""
    wl = I.WORKLOADS["fused_tail"]
    x = I.make_inputs(wl, seed=4, device="cuda")
    w8, sc = I.fp8_weight(x["wo_a"])
    rope = sa.rope_table(wl.theta, 0, wl.T, wl.rope_dim).cuda()
    y = sa.sparse_attn_rope_wo_a_fp8(x["q"], x["kv"], x["sink"], x["idx"], wl.scale, rope, w8, sc, check=True)
    wdq = torch.from_numpy(oracle.dequant_fp8_weight(w8.reshape(wl.G * wl.R, -1).cpu().numpy(),
                                                     sc.cpu().numpy()).view(np.int16)).view(torch.bfloat16)
    qs = sample_queries(wl.n_queries, 16, seed=6, include=(0, 4095, 4096, 8191))
    o = oracle_rows(x, qs, wl.scale)
    o = oracle.inverse_rope(o, qs % wl.T, wl.rope_dim, wl.theta)
    yref = oracle.wo_a(o.reshape(len(qs), wl.G, -1), wdq.reshape(wl.G, wl.R, -1))
    got = y.reshape(-1, wl.G * wl.R)[torch.as_tensor(qs, device="cuda")].double().cpu().numpy()
    compare(got, yref.reshape(len(qs), -1), "fused_tail fp8")


@pytest.mark.parametrize("T", [40, 600])   # weight decoded in the GEMM / into a bf16 copy first
def test_fused_tail_fp8_special_weights(T):
    """fp8 weights with NaN bytes, zero and subnormal-scale blocks, and large
    scales: the bf16 call on the oracle's dequantized weight gives the same
    outputs, NaN in the same places, on both decoding paths."""
    g = torch.Generator().manual_seed(77)
    B, K, N, G, R = 1, 64, 80, 8, 256
    din = 64 * 512 // G
    q = torch.randn(B, T, 64, 512, generator=g).to(torch.bfloat16)
    kv = I.rms_rows(torch.randn(B, N, 512, generator=g)).to(torch.bfloat16)
    sink = torch.randn(64, generator=g)
    idx = torch.randint(0, N, (B, T, K), generator=g, dtype=torch.int32)
    w8 = torch.randint(0, 256, (G, R, din), generator=g, dtype=torch.int32).to(torch.uint8)
    w8[(w8 & 0x7F) == 0x7F] = 0x33
    w8[1, 5, 17] = 0x7F                     # two NaN weights: rows 1*256+5 and 3*256+200 become NaN
    w8[3, 200, 1000] = 0xFF
    sc = (torch.rand(G * R // 128, din // 128, generator=g) * 1e-3 + 1e-5)
    sc[0, 0] = 300.0                        # conversion-unit path
    sc[2, 3] = 2.0 ** 20
    sc[4, 1] = 1e-40                        # subnormal scale
    sc[5, 2] = 0.0                          # zero block
    wdq = torch.from_numpy(oracle.dequant_fp8_weight(w8.reshape(G * R, -1).numpy(), sc.numpy())
                           .view(np.int16)).view(torch.bfloat16).reshape(G, R, -1)
    rope = sa.rope_table(160000.0, 0, T, 64).cuda()
    x = to_dev(dict(q=q, kv=kv, sink=sink, idx=idx))
    got = sa.sparse_attn_rope_wo_a_fp8(x["q"], x["kv"], x["sink"], x["idx"], 512 ** -0.5, rope, w8.cuda(),
                                       sc.cuda(), check=True).float()
    ref = sa.sparse_attn_rope_wo_a(x["q"], x["kv"], x["sink"], x["idx"], 512 ** -0.5, rope, wdq.cuda(),
                                   check=True).float()
    nan = torch.isnan(ref)
    assert torch.equal(torch.isnan(got), nan)
    assert nan[..., 1 * R + 5].all() and nan[..., 3 * R + 200].all() and nan.sum() == 2 * B * T
    assert torch.equal(got[~nan], ref[~nan])


@pytest.mark.parametrize("seed", range(8))
def test_random_shapes_against_oracle(seed):
    """Seeded random problems across the schedules (whole lists, two to eight
    list pieces per query, ragged chunks, -1 anywhere, repeated indices): the
    plain call, the two-source call and the two-source fp4 call against the
    oracle, and the two-source call against the plain call on the
    concatenated rows (bit for bit)."""
    rng = np.random.default_rng(1000 + seed)
    B = int(rng.integers(1, 5))
    T = int(rng.integers(1, 40))
    K = int(rng.integers(1, 1025))
    W = int(rng.integers(0, 200))
    C = int(rng.integers(1, 1500))
    N = W + C
    g = torch.Generator().manual_seed(2000 + seed)
    q = torch.randn(B, T, 64, 512, generator=g).to(torch.bfloat16)
    kv = I.rms_rows(torch.randn(B, N, 512, generator=g)).to(torch.bfloat16)
    sink = 2 * torch.randn(64, generator=g)
    idx = torch.randint(0, N, (B, T, K), generator=g, dtype=torch.int32)
    idx[torch.rand(B, T, K, generator=g) < float(rng.uniform(0, 0.5))] = -1
    x = dict(q=q, kv=kv, sink=sink, idx=idx)
    got = run(x, 512 ** -0.5)
    ref = full_oracle(x, 512 ** -0.5)
    compare(got.double().cpu().numpy(), ref, f"random {seed}: B{B} T{T} K{K} N{N}")
    gd = to_dev(x)
    two = sa.sparse_attn_two_source(gd["q"], gd["kv"][:, :W].contiguous() if W else None,
                                    gd["kv"][:, W:].contiguous(), gd["sink"], gd["idx"], 512 ** -0.5,
                                    W=W, C=C, check=True)
    assert torch.equal(two, got)
    # fp4 compressed rows: codes and scales drawn directly
    codes = torch.randint(0, 256, (B, C, 256), generator=g, dtype=torch.int32).to(torch.uint8)
    scales = (0x20 + torch.randint(0, 8, (B, C, 32), generator=g, dtype=torch.int32)).to(torch.uint8)
    win = kv[:, :W].contiguous()
    got4 = sa.sparse_attn_two_source_fp4(gd["q"], win.cuda() if W else None, codes.cuda(), scales.cuda(),
                                         gd["sink"], gd["idx"], 512 ** -0.5, W=W, C=C, out_dtype=torch.float32,
                                         check=True)
    ref4, bad = oracle.sparse_attn_two_source_fp4(q, win, W, codes.numpy(), scales.numpy(), C, sink, idx,
                                                  512 ** -0.5)
    assert bad == 0
    compare(got4.double().cpu().numpy(), ref4, f"random fp4 {seed}")


# ---------------------------------------------------------------- fp4 quantizer

def _special_groups(rng):
    """Groups of 16 features that exercise the rounding rules: all zero, signed
    zeros, a scale that underflows E4M3, the bf16 extremes and infinities
    (scale saturates at 448), values exactly halfway between e2m1 magnitudes
    (amax 6: scale 1), and a scale rounded down (codes saturate at 6)."""
    g = []
    g.append(np.zeros(16))
    g.append(np.array([-0.0, 0.0] * 8))
    g.append(np.full(16, 1e-30) * rng.choice([-1, 1], 16))
    g.append(np.array([3.3895e38, -3.3895e38] + [1.0] * 14))
    g.append(np.array([np.inf, -2.0, 1e30] + [0.5] * 13))
    g.append(np.array([6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5,
                       -5.0, 0.0]))
    g.append(np.array([6.25, -6.25, 3.0, 0.2] + [0.1] * 12))
    return np.concatenate(g)


def test_fp4_quantize_matches_oracle():
    """Codes and scales bit for bit against the oracle on RMS-normalised latent
    rows (the cache's inputs), rows of wide dynamic range, the special groups,
    and strided rows (each row cut from a wider one)."""
    rng = np.random.default_rng(31)
    rows, D = 3000, 512
    x = I.rms_rows(torch.from_numpy(rng.standard_normal((rows, D)).astype(np.float32)))
    x[100:200] *= torch.from_numpy(np.exp2(rng.integers(-60, 60, (100, 1))).astype(np.float32))
    spec = _special_groups(rng)
    x[7, :spec.size] = torch.from_numpy(spec.astype(np.float32))
    wide = torch.zeros(rows, D + 8, dtype=torch.bfloat16)
    wide[:, :D] = x.to(torch.bfloat16)
    lat = wide.cuda()[:, :D]                           # row stride D + 8
    codes, scales = sa.fp4_quantize(lat)
    torch.cuda.synchronize()
    bits = wide[:, :D].contiguous().view(torch.int16).numpy().view(np.uint16)
    rc, rs = oracle.fp4_quantize(bits)
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


def test_fp4_quantized_cache_through_the_attention_call():
    """The producer and the consumer agree: latents quantized by the library
    and read by the fp4 call give exactly the bf16 call on the cache the oracle
    decodes from those codes (and its own codes are the oracle's)."""
    g = torch.Generator().manual_seed(41)
    B, T, K, W, C, D = 2, 3, 400, 128, 700, 512
    win = I.rms_rows(torch.randn(B, W, D, generator=g)).to(torch.bfloat16).cuda()
    lat = I.rms_rows(torch.randn(B, C, D, generator=g)).to(torch.bfloat16).cuda()
    codes, scales = sa.fp4_quantize(lat)
    q = torch.randn(B, T, 64, D, generator=g).to(torch.bfloat16).cuda()
    sink = torch.randn(64, generator=g).cuda()
    idx = torch.randint(0, W + C, (B, T, K), generator=g, dtype=torch.int32).cuda()
    got = sa.sparse_attn_two_source_fp4(q, win, codes, scales, sink, idx, 512 ** -0.5, W=W, C=C,
                                        out_dtype=torch.float32, check=True)
    rc, rs = oracle.fp4_quantize(lat.cpu().view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(codes.cpu().numpy(), rc) and np.array_equal(scales.cpu().numpy(), rs)
    dec = torch.from_numpy(oracle.bf16_bits_exact(oracle.dequant_fp4(rc, rs)).view(np.int16)).view(torch.bfloat16)
    ref = sa.sparse_attn_two_source(q, win, dec.cuda(), sink, idx, 512 ** -0.5, W=W, C=C,
                                    out_dtype=torch.float32, check=True)
    assert torch.equal(got, ref)


@pytest.mark.parametrize("D", [16, 48, 1040])
def test_fp4_quantize_other_widths(D):
    """Row widths whose group count is not a power of two (and a single group),
    against the oracle bit for bit."""
    rng = np.random.default_rng(D)
    rows = 777
    x = torch.from_numpy((rng.standard_normal((rows, D)) * np.exp2(rng.integers(-20, 20, (rows, 1))))
                         .astype(np.float32)).to(torch.bfloat16)
    codes, scales = sa.fp4_quantize(x.cuda())
    rc, rs = oracle.fp4_quantize(x.view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)
