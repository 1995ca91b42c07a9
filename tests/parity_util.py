"""Helpers shared by the GPU parity tests: run the CUDA path, run the fp64
oracle on the same inputs (all queries, or a sample), compare."""
import numpy as np
import torch

import oracle
import sparse_latent_attention_02_gb300 as sa

# Bound stated for bf16 outputs (and used for fp32 outputs too).
MAX_ABS = 2e-2
REL_FRO = 5e-3


def to_dev(x, dev="cuda"):
    return {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in x.items()}


def compare(got, ref, what="", per_value=False):
    """Element-wise comparison: max-abs <= 2e-2 and relative Frobenius <= 5e-3.
    ``per_value``: each element may also differ by 2^-7 of its own magnitude
    (four times its bf16 rounding, half an ulp = 2^-9), for bf16 outputs whose
    values reach well above 1."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    if per_value:
        err = err - 2.0 ** -7 * np.abs(ref)
    max_abs = float(err.max()) if err.size else 0.0
    nref = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(got - ref) / nref) if nref > 0 else float(np.linalg.norm(got))
    assert max_abs <= MAX_ABS and rel <= REL_FRO, \
        f"{what}: max-abs {max_abs:.3e}{' beyond 2^-7|ref|' if per_value else ''} (<= {MAX_ABS}), " \
        f"rel-Frobenius {rel:.3e} (<= {REL_FRO})"
    return max_abs, rel


def sample_queries(BT, n, seed=0, include=()):
    rng = np.random.default_rng(seed)
    s = set(int(i) for i in include if 0 <= i < BT)
    s.update(int(i) for i in rng.choice(BT, size=min(n, BT), replace=False))
    return np.array(sorted(s), dtype=np.int64)


def oracle_rows(x, queries, scale):
    """fp64 oracle on the listed flattened queries of a [B, T] problem, copying only
    what those queries read from the device tensors."""
    q, kv, sink, idx = x["q"], x["kv"], x["sink"], x["idx"]
    B, T = q.shape[:2]
    queries = np.asarray(queries, dtype=np.int64)
    out = np.empty((queries.size, q.shape[2], q.shape[3]))
    for b in np.unique(queries // T):
        sel = queries[queries // T == b]
        t_sel = torch.as_tensor(sel % T)
        qb = q[b:b + 1, t_sel.to(q.device)].cpu()
        ib = idx[b:b + 1, t_sel.to(idx.device)].cpu()
        kvb = kv[b:b + 1].cpu()
        ref, bad = oracle.sparse_attn(qb, kvb, sink.cpu(), ib, scale)
        assert bad == 0
        out[np.searchsorted(queries, sel)] = ref[0]
    return out


def cached_workspace(kind: str):
    """The binding's default workspace of one kind of call ("attn", "fused", ...)
    on the current device and stream."""
    return sa._ws_cache[(torch.cuda.current_device(), kind, int(torch.cuda.current_stream().cuda_stream))]
