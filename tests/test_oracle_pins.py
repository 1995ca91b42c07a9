"""Pins for the fp64 oracle, checked against things other than itself.

* a dense masked-attention brute force in the pattern of the "GLM-5 > Sparse
  latent attention" page (``eager_attention_forward`` plus the index mask built
  with ``scatter`` and filled with -inf), with the sink appended as one more
  logit whose value row is zero;
* a pure-Python scalar brute force on a very small case;
* closed forms: one valid index, equal scores, sink -> -inf, a dominant sink;
* invariants: permutation of the index list, -1 anywhere, the all-skip row,
  K = 0, repeated indices counted as separate terms, a one-hot index probe;
* the rotary embedding's special angles, group law and complex-number form;
* the grouped projection against a dense block-diagonal matmul.
"""
import math

import numpy as np
import pytest
import torch

import oracle

RNG = np.random.default_rng(1234)


def bf16(x):
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


def f64(t):
    return t.to(torch.float32).numpy().astype(np.float64)


def rand_case(B, T, H, D, N, K, p_skip=0.3, seed=0, distinct=True):
    rng = np.random.default_rng(seed)
    q = bf16(rng.standard_normal((B, T, H, D)))
    kv = bf16(rng.standard_normal((B, N, D)))
    sink = rng.standard_normal(H).astype(np.float32)
    idx = np.empty((B, T, K), dtype=np.int32)
    for b in range(B):
        for t in range(T):
            if distinct:
                row = rng.permutation(N)[:K]
            else:
                row = rng.integers(0, N, size=K)
            row = np.where(rng.random(K) < p_skip, -1, row)
            idx[b, t] = row
    return q, kv, sink, idx


def dense_bruteforce(q, kv, sink, idx, scale):
    """Dense masked softmax attention: every latent row scored, the rows not in
    the list masked with -inf, the sink appended as an extra logit (zero value)."""
    qd, kvd = f64(q), f64(kv)
    B, T, H, D = qd.shape
    N = kvd.shape[1]
    out = np.zeros((B, T, H, D))
    for b in range(B):
        for t in range(T):
            keep = np.zeros(N, dtype=bool)
            sel = idx[b, t][idx[b, t] >= 0]
            keep[sel] = True
            logits = (qd[b, t] @ kvd[b].T) * scale                  # [H, N]
            logits = np.where(keep[None, :], logits, -np.inf)
            logits = np.concatenate([logits, sink.astype(np.float64)[:, None]], 1)
            m = logits.max(1, keepdims=True)
            e = np.exp(logits - m)
            p = e / e.sum(1, keepdims=True)
            vals = np.concatenate([kvd[b], np.zeros((1, D))], 0)    # sink row carries no value
            out[b, t] = p @ vals
    return out


@pytest.mark.parametrize("H,D,N,K", [(1, 8, 24, 10), (4, 16, 40, 17), (64, 512, 64, 48)])
def test_dense_bruteforce(H, D, N, K):
    q, kv, sink, idx = rand_case(2, 3, H, D, N, K, seed=H + D)
    scale = D ** -0.5
    ref = dense_bruteforce(q, kv, sink, idx, scale)
    got, bad = oracle.sparse_attn(q, kv, sink, idx, scale)
    assert bad == 0
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)


def test_scalar_python_bruteforce():
    q, kv, sink, idx = rand_case(1, 2, 2, 4, 7, 5, seed=7)
    qd, kvd = f64(q), f64(kv)
    scale = 0.37
    got, _ = oracle.sparse_attn(q, kv, sink, idx, scale)
    for t in range(2):
        for h in range(2):
            terms = []
            for j in idx[0, t]:
                if j < 0:
                    continue
                s = scale * sum(float(qd[0, t, h, d]) * float(kvd[0, j, d]) for d in range(4))
                terms.append((s, [float(kvd[0, j, d]) for d in range(4)]))
            logits = [s for s, _ in terms] + [float(sink[h])]
            m = max(logits)
            den = sum(math.exp(x - m) for x in logits)
            o = [sum(math.exp(s - m) * r[d] for s, r in terms) / den for d in range(4)]
            np.testing.assert_allclose(got[0, t, h], o, rtol=1e-13, atol=1e-15)


def test_single_valid_index_closed_form():
    q, kv, sink, idx = rand_case(1, 1, 8, 32, 12, 6, seed=3)
    idx[:] = -1
    idx[0, 0, 4] = 9
    scale = 32 ** -0.5
    got, _ = oracle.sparse_attn(q, kv, sink, idx, scale)
    row = f64(kv)[0, 9]
    s = scale * (f64(q)[0, 0] @ row)                        # [H]
    w = np.exp(s) / (np.exp(s) + np.exp(sink.astype(np.float64)))
    np.testing.assert_allclose(got[0, 0], w[:, None] * row[None, :], rtol=1e-13)


def test_dominant_sink():
    """sink = +8 with large logits: the sink share is visible, not ~0.1%."""
    q, kv, sink, idx = rand_case(1, 1, 4, 16, 8, 4, seed=5)
    q = bf16(4.0 * f64(q))
    sink = np.full(4, 8.0, dtype=np.float32)
    idx[:] = -1
    idx[0, 0, 0] = 3
    scale = 16 ** -0.5
    got, _ = oracle.sparse_attn(q, kv, sink, idx, scale)
    row = f64(kv)[0, 3]
    s = scale * (f64(q)[0, 0] @ row)
    w = 1.0 / (1.0 + np.exp(8.0 - s))
    np.testing.assert_allclose(got[0, 0], w[:, None] * row[None, :], rtol=1e-12)
    assert np.all(w < 0.99)


def test_sink_minus_inf_is_plain_softmax():
    q, kv, sink, idx = rand_case(2, 2, 4, 16, 20, 9, seed=11)
    sink = np.full(4, -np.inf, dtype=np.float32)
    scale = 0.25
    got, _ = oracle.sparse_attn(q, kv, sink, idx, scale)
    qd, kvd = f64(q), f64(kv)
    for b in range(2):
        for t in range(2):
            sel = idx[b, t][idx[b, t] >= 0]
            s = scale * qd[b, t] @ kvd[b, sel].T
            p = np.exp(s - s.max(1, keepdims=True))
            p /= p.sum(1, keepdims=True)
            np.testing.assert_allclose(got[b, t], p @ kvd[b, sel], rtol=1e-12, atol=1e-15)
    # a single index with sink -inf returns the row exactly
    idx[:] = -1
    idx[0, 0, 2] = 5
    got, _ = oracle.sparse_attn(q, kv, sink, idx, scale)
    assert np.array_equal(got[0, 0], np.broadcast_to(kvd[0, 5], (4, 16)))


def test_equal_scores_mean():
    """q = 0: every score is 0, o = mean(rows) * n / (n + e^sink)."""
    _, kv, sink, idx = rand_case(1, 1, 3, 8, 30, 12, seed=13)
    q = bf16(np.zeros((1, 1, 3, 8)))
    got, _ = oracle.sparse_attn(q, kv, sink, idx, 0.5)
    sel = idx[0, 0][idx[0, 0] >= 0]
    n = sel.size
    mean = f64(kv)[0, sel].mean(0)
    factor = n / (n + np.exp(sink.astype(np.float64)))
    np.testing.assert_allclose(got[0, 0], factor[:, None] * mean[None, :], rtol=1e-13)


def test_permutation_invariance_and_skip_anywhere():
    q, kv, sink, idx = rand_case(2, 4, 8, 64, 50, 30, p_skip=0.4, seed=17)
    scale = 64 ** -0.5
    ref, _ = oracle.sparse_attn(q, kv, sink, idx, scale)
    rng = np.random.default_rng(0)
    perm = idx.copy()
    for b in range(2):
        for t in range(4):
            perm[b, t] = perm[b, t][rng.permutation(30)]
    got, _ = oracle.sparse_attn(q, kv, sink, perm, scale)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-15)
    # padding the list with -1 (front or back) changes nothing
    pad = np.full((2, 4, 7), -1, dtype=np.int32)
    got2, _ = oracle.sparse_attn(q, kv, sink, np.concatenate([pad, idx, pad], 2), scale)
    np.testing.assert_allclose(got2, ref, rtol=1e-12, atol=1e-15)


def test_all_skip_and_empty_lists_give_zero():
    q, kv, sink, idx = rand_case(1, 3, 4, 16, 10, 5, seed=19)
    idx[:] = -1
    got, _ = oracle.sparse_attn(q, kv, sink, idx, 0.3)
    assert np.array_equal(got, np.zeros_like(got))
    got, _ = oracle.sparse_attn(q, kv, np.full(4, -np.inf, np.float32), idx, 0.3)
    assert np.array_equal(got, np.zeros_like(got))
    got, _ = oracle.sparse_attn(q, kv, sink, np.zeros((1, 3, 0), np.int32), 0.3)
    assert got.shape == (1, 3, 4, 16) and not got.any()


def test_repeated_index_counts_twice():
    _, kv, _, _ = rand_case(1, 1, 2, 8, 6, 3, seed=23)
    q = bf16(np.zeros((1, 1, 2, 8)))
    sink = np.full(2, -np.inf, dtype=np.float32)
    idx = np.array([[[4, 1, 4]]], dtype=np.int32)
    got, _ = oracle.sparse_attn(q, kv, sink, idx, 1.0)
    kvd = f64(kv)[0]
    np.testing.assert_allclose(got[0, 0], np.broadcast_to((2 * kvd[4] + kvd[1]) / 3, (2, 8)),
                               rtol=1e-15)


def test_index_probe_multiplicities():
    """q = 0, sink = -inf, row r of kv = e_r: o * V equals each row's multiplicity."""
    N, D, K = 40, 64, 50
    kv = bf16(np.eye(N, D)[None])
    q = bf16(np.zeros((1, 2, 3, D)))
    sink = np.full(3, -np.inf, dtype=np.float32)
    rng = np.random.default_rng(29)
    idx = rng.integers(-1, N, size=(1, 2, K)).astype(np.int32)
    got, _ = oracle.sparse_attn(q, kv, sink, idx, 1.0)
    for t in range(2):
        valid = idx[0, t][idx[0, t] >= 0]
        counts = np.bincount(valid, minlength=D)
        np.testing.assert_allclose(got[0, t] * valid.size, np.broadcast_to(counts, (3, D)),
                                   atol=1e-12)


def test_out_of_range_index_is_reported_and_skipped():
    q, kv, sink, idx = rand_case(1, 2, 2, 8, 10, 4, p_skip=0.0, seed=31)
    clean, bad0 = oracle.sparse_attn(q, kv, sink, idx, 0.5)
    assert bad0 == 0
    idx2 = np.concatenate([idx, np.array([[[10], [-2]]], dtype=np.int32)], 2)
    got, bad = oracle.sparse_attn(q, kv, sink, idx2, 0.5)
    assert bad == 2
    np.testing.assert_allclose(got, clean, rtol=1e-14)


def test_query_subset_matches_full():
    q, kv, sink, idx = rand_case(2, 5, 4, 16, 30, 12, seed=37)
    full, _ = oracle.sparse_attn(q, kv, sink, idx, 0.25)
    sub, _ = oracle.sparse_attn(q, kv, sink, idx, 0.25, queries=[7, 0, 4])
    flat = full.reshape(10, 4, 16)
    assert np.array_equal(sub, flat[[7, 0, 4]])


# ---------------------------------------------------------------- rotary


def test_rope_position_zero_is_identity_and_prefix_untouched():
    x = RNG.standard_normal((3, 4, 128))
    y = oracle.inverse_rope(x, np.zeros(3, np.int64), 64, 160000.0)
    assert np.array_equal(y, x)
    y = oracle.inverse_rope(x, np.array([5, 77, 4095]), 64, 160000.0)
    assert np.array_equal(y[..., :64], x[..., :64])


def test_rope_special_angles():
    x = np.zeros((1, 1, 64))
    x[0, 0, 0] = 1.0            # pair 0 = (1, 0); frequency theta**0 = 1
    x[0, 0, 33] = 1.0           # pair 16 = (0, 1); frequency 160000**-0.5 = 1/400
    y = oracle.inverse_rope(x, np.array([1]), 64, 160000.0)
    np.testing.assert_allclose(y[0, 0, :2], [math.cos(1.0), -math.sin(1.0)], rtol=1e-15)
    y = oracle.inverse_rope(x, np.array([400]), 64, 160000.0)
    np.testing.assert_allclose(y[0, 0, 32:34], [math.sin(1.0), math.cos(1.0)], rtol=1e-12)


def test_rope_norm_group_law_and_complex_form():
    x = RNG.standard_normal((5, 2, 96))
    p1 = np.array([3, 10, 100, 1000, 4095])
    p2 = np.array([7, 1, 50, 3, 1])
    y = oracle.inverse_rope(x, p1, 64, 160000.0)
    pairs = lambda a: a[..., 32:].reshape(5, 2, 32, 2)
    np.testing.assert_allclose(np.linalg.norm(pairs(y), axis=-1),
                               np.linalg.norm(pairs(x), axis=-1), rtol=1e-13)
    yy = oracle.inverse_rope(y, p2, 64, 160000.0)
    np.testing.assert_allclose(yy, oracle.inverse_rope(x, p1 + p2, 64, 160000.0),
                               rtol=1e-9, atol=1e-12)
    # the forward embedding as complex multiplication by exp(+i p w), then the inverse
    w = 160000.0 ** (-np.arange(32) * 2.0 / 64)
    z = pairs(x)[..., 0] + 1j * pairs(x)[..., 1]
    zf = z * np.exp(1j * p1[:, None, None] * w[None, None, :])
    xf = x.copy()
    xf[..., 32:] = np.stack([zf.real, zf.imag], -1).reshape(5, 2, 64)
    np.testing.assert_allclose(oracle.inverse_rope(xf, p1, 64, 160000.0), x,
                               rtol=1e-9, atol=1e-12)


# ---------------------------------------------------------------- wo_a


def test_wo_a_single_group_is_matmul():
    o = RNG.standard_normal((6, 1, 40))
    W = bf16(RNG.standard_normal((1, 24, 40)))
    y = oracle.wo_a(o, W)
    np.testing.assert_allclose(y[:, 0], o[:, 0] @ f64(W)[0].T, rtol=1e-12)


def test_wo_a_block_diagonal_dense():
    G, R, Din, n = 4, 12, 20, 9
    o = RNG.standard_normal((n, G, Din))
    W = bf16(RNG.standard_normal((G, R, Din)))
    Wd = f64(W)
    full = np.zeros((G * R, G * Din))
    for g in range(G):
        full[g * R:(g + 1) * R, g * Din:(g + 1) * Din] = Wd[g]
    y = oracle.wo_a(o, W)
    np.testing.assert_allclose(y.reshape(n, G * R), o.reshape(n, G * Din) @ full.T,
                               rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------------ two latent sources

def _two_sources(B, Bmax, W, Wmax, C, Cmax, D, seed):
    """Window and compressed caches larger than the rows in use, padding = NaN."""
    rng = np.random.default_rng(seed)
    nan = float("nan")
    win = np.full((Bmax, Wmax, D), nan, dtype=np.float32)
    cmp_ = np.full((Bmax, Cmax, D), nan, dtype=np.float32)
    win[:B, :W] = rng.standard_normal((B, W, D))
    cmp_[:B, :C] = rng.standard_normal((B, C, D))
    return bf16(win), bf16(cmp_)


def test_two_source_padding_is_never_read():
    """Rows of either cache beyond W / C (and spare batch rows) hold NaN and
    never reach the output; the result is sparse_attn on the rows in use."""
    B, T, H, D, W, C, K = 2, 3, 4, 8, 5, 9, 10
    win, cmp_ = _two_sources(B, 3, W, 7, C, 12, D, seed=3)
    rng = np.random.default_rng(4)
    q = bf16(rng.standard_normal((B, T, H, D)))
    sink = rng.standard_normal(H).astype(np.float32)
    idx = rng.integers(-1, W + C, size=(B, T, K)).astype(np.int32)
    out, bad = oracle.sparse_attn_two_source(q, win, W, cmp_, C, sink, idx, 0.3)
    assert bad == 0 and np.all(np.isfinite(out))
    used = torch.cat([win[:B, :W], cmp_[:B, :C]], dim=1)
    ref, _ = oracle.sparse_attn(q, used, sink, idx, 0.3)
    assert np.array_equal(out, ref)


@pytest.mark.parametrize("v", [0, 4, 5, 13])
def test_two_source_index_reaches_the_right_row(v):
    """q = 0 and sink = -inf make the output the mean of the listed rows: a
    list holding only index v returns window row v (v < W) or compressed row
    v - W (v >= W), exactly."""
    B, T, H, D, W, C = 1, 1, 2, 8, 5, 9
    win, cmp_ = _two_sources(B, 1, W, 6, C, 10, D, seed=5)
    q = bf16(np.zeros((B, T, H, D)))
    sink = np.full(H, -np.inf, dtype=np.float32)
    idx = np.array([[[v, -1, -1]]], dtype=np.int32)
    out, bad = oracle.sparse_attn_two_source(q, win, W, cmp_, C, sink, idx, 1.0)
    row = win[0, v] if v < W else cmp_[0, v - W]
    assert bad == 0
    assert np.array_equal(out[0, 0, 0], f64(row)) and np.array_equal(out[0, 0, 1], f64(row))


def test_two_source_one_source_empty():
    """W = 0 reads only the compressed cache; C = 0 only the window."""
    B, T, H, D = 1, 2, 2, 8
    win, cmp_ = _two_sources(B, 1, 6, 6, 7, 7, D, seed=6)
    rng = np.random.default_rng(7)
    q = bf16(rng.standard_normal((B, T, H, D)))
    sink = rng.standard_normal(H).astype(np.float32)
    idx = rng.integers(0, 6, size=(B, T, 4)).astype(np.int32)
    only_w, _ = oracle.sparse_attn_two_source(q, win, 6, None, 0, sink, idx, 0.5)
    only_c, _ = oracle.sparse_attn_two_source(q, None, 0, cmp_, 7, sink, idx, 0.5)
    assert np.array_equal(only_w, oracle.sparse_attn(q, win, sink, idx, 0.5)[0])
    assert np.array_equal(only_c, oracle.sparse_attn(q, cmp_[:, :7], sink, idx, 0.5)[0])


# ------------------------------------------------------------------ wo_b

def test_wo_b_equals_one_group_wo_a_and_a_hand_case():
    """wo_b (one fp64 matrix product) against the independent grouped loop of
    wo_a with a single group, and a 2 x 2 case worked by hand."""
    rng = np.random.default_rng(11)
    n, din, dim = 5, 64, 48
    y = rng.standard_normal((n, din))
    W = bf16(0.1 * rng.standard_normal((dim, din)))
    got = oracle.wo_b(y, W)
    ref = oracle.wo_a(y.reshape(n, 1, din), W.reshape(1, dim, din)).reshape(n, dim)
    assert np.allclose(got, ref, rtol=1e-13, atol=1e-13)
    # [[1, 2], [3, 4]] @ [[1, 0.5], [-2, 0.25]]^T = [[2, -1.5], [5, -5]]
    yh = np.array([[1.0, 2.0], [3.0, 4.0]])
    Wh = bf16([[1.0, 0.5], [-2.0, 0.25]])
    assert np.array_equal(oracle.wo_b(yh, Wh), np.array([[2.0, -1.5], [5.0, -5.0]]))


# ------------------------------------------------------------------ top-k selection

def _topk_brute(row, k, offset):
    """Pick the largest remaining score k times (smaller position on ties)."""
    left = [(j, x) for j, x in enumerate(row) if not (math.isnan(x) or x == -math.inf)]
    chosen = []
    for _ in range(min(k, len(left))):
        best = max(left, key=lambda jx: (jx[1], -jx[0]))
        chosen.append(best[0])
        left.remove(best)
    chosen.sort()
    return [j + offset for j in chosen] + [-1] * (k - len(chosen))


def test_topk_brute_force_with_ties_and_masks():
    rng = np.random.default_rng(21)
    for trial in range(40):
        L, k = int(rng.integers(0, 30)), int(rng.integers(1, 12))
        row = np.round(rng.standard_normal(L), 1)          # many ties
        row[rng.random(L) < 0.2] = -np.inf
        row[rng.random(L) < 0.05] = np.nan
        got = oracle.topk_indices(row[None, :], k, offset=7)[0].tolist()
        assert got == _topk_brute(row.tolist(), k, 7), (trial, row, k)


def test_topk_defining_property():
    """Every chosen score is at least every score left out; as many positions
    as can be chosen; ascending; offset applied; -1 after them."""
    rng = np.random.default_rng(22)
    scores = rng.standard_normal((6, 500)).astype(np.float32)
    for r in range(6):
        scores[r, 400 - 60 * r:] = -np.inf                 # causal-style masked tails
    k = 256
    got = oracle.topk_indices(scores, k, offset=128)
    for r in range(6):
        valid = np.nonzero(np.isfinite(scores[r]))[0]
        sel = got[r][got[r] >= 0] - 128
        assert sel.size == min(k, valid.size)
        assert np.all(np.diff(sel) > 0) and np.all(got[r][sel.size:] == -1)
        rest = np.setdiff1d(valid, sel)
        if rest.size and sel.size:
            assert scores[r, sel].min() >= scores[r, rest].max()


def test_topk_signed_zeros_tie():
    """-0.0 and +0.0 compare equal, so they tie and the smaller position wins."""
    row = np.array([1.0, -0.0, 0.0, -0.0, 2.0])
    assert oracle.topk_indices(row[None, :], 3)[0].tolist() == [0, 1, 4]


def test_topk_subnormals_are_not_zero():
    """fp32 subnormal scores keep their order: above +-0, below the smallest
    normal number, negative ones below -0 (brute force over random rows)."""
    vals = np.array([-1e-40, -0.0, 0.0, 1e-45, 1e-40, 2e-40, 1.2e-38, -np.inf, np.nan], np.float32)
    assert vals[3] > 0 and vals[4] < np.finfo(np.float32).tiny            # really subnormal
    row = np.array([0.0, 1e-45, -1e-40, 2e-40, -0.0], np.float32)
    assert oracle.topk_indices(row[None, :], 2)[0].tolist() == [1, 3]
    rng = np.random.default_rng(23)
    for trial in range(30):
        L, k = int(rng.integers(1, 40)), int(rng.integers(1, 15))
        row = vals[rng.integers(0, len(vals), L)]
        got = oracle.topk_indices(row[None, :], k, offset=3)[0].tolist()
        assert got == _topk_brute([float(x) for x in row], k, 3), (trial, row, k)


# ------------------------------------------------------------------ fp4 compressed rows

def test_e2m1_codes_and_nibble_order():
    """The 16 e2m1 codes decode to +-{0, .5, 1, 1.5, 2, 3, 4, 6} (OCP MX
    element values); byte i holds feature 2i in its low nibble."""
    codes = np.array([[0x10, 0x32, 0x54, 0x76, 0x98, 0xBA, 0xDC, 0xFE]], dtype=np.uint8)
    scales = np.array([[0x38]], dtype=np.uint8)            # 1.0
    got = oracle.dequant_fp4(codes, scales)[0]
    want = [0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6]
    assert np.array_equal(got, np.array(want))


@pytest.mark.parametrize("byte,value", [(0x38, 1.0), (0xB8, -1.0), (0x7E, 448.0), (0x08, 2.0 ** -6),
                                        (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x00, 0.0),
                                        (0x40, 2.0), (0x3C, 1.5)])
def test_e4m3_known_bytes(byte, value):
    assert oracle.e4m3_values(byte) == value


def test_e4m3_nan_and_scale_applies_per_group():
    assert np.isnan(oracle.e4m3_values(0x7F)) and np.isnan(oracle.e4m3_values(0xFF))
    codes = np.full((1, 16), 0x22, dtype=np.uint8)          # every feature code 2 = 1.0
    scales = np.array([[0x38, 0x40]], dtype=np.uint8)       # groups: 1.0, 2.0
    got = oracle.dequant_fp4(codes, scales)[0]
    assert np.array_equal(got, np.r_[np.ones(16), 2 * np.ones(16)])


def test_fp4_values_are_exact_in_bf16():
    """Every code times every finite E4M3 scale is a bf16 value (so the GPU's
    bf16 decode loses nothing)."""
    finite = [b for b in range(256) if (b & 0x7F) != 0x7F]
    codes = np.tile(np.arange(256, dtype=np.uint8), (len(finite), 1)).reshape(len(finite), 256)
    scales = np.repeat(np.array(finite, dtype=np.uint8)[:, None], 32, axis=1)
    vals = oracle.dequant_fp4(codes, scales)
    oracle.bf16_bits_exact(vals)                           # raises if any is not exact


def test_e4m3_matches_torch_float8_for_every_byte():
    """The oracle's E4M3 decoding against PyTorch's float8_e4m3fn dtype, all 256 bytes."""
    b = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_values(b)
    lib = torch.from_numpy(b).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(lib))
    ok = ~np.isnan(ours)
    assert np.array_equal(ours[ok], lib[ok])


def test_round_bf16_matches_torch_including_ties():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(200000) * np.exp2(rng.integers(-130, 120, 200000))).astype(np.float32)
    special = np.array([0x3F808000, 0x3F818000, 0x3F80FFFF, 0x7F7FFFFF, 0x00000001, 0x80008000,
                        0x00018000, 0x7F800000, 0xFF800000, 0x80000000], dtype=np.uint32).view(np.float32)
    x = np.concatenate([x, special])
    ours = oracle.round_bf16(x)
    lib = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, lib)
    # ties to even by hand: 1 + 2^-8 lies halfway between 1 and 1 + 2^-7 -> 1
    assert oracle.round_bf16(np.float32(1 + 2 ** -8)) == 0x3F80
    assert oracle.round_bf16(np.float32(1 + 3 * 2 ** -8)) == 0x3F82


def test_fp8_weight_power_of_two_scales_are_exact():
    """A power-of-two scale only moves the exponent: the dequantized weight is
    the E4M3 value times the scale, exactly."""
    rng = np.random.default_rng(3)
    w8 = rng.integers(0, 256, (256, 256), dtype=np.uint8)
    w8[(w8 & 0x7F) == 0x7F] = 0x11
    sc = np.exp2(rng.integers(-20, 10, (2, 2))).astype(np.float32)
    got = oracle.dequant_fp8_weight(w8, sc)
    want = oracle.bf16_bits_exact(oracle.e4m3_values(w8) * np.repeat(np.repeat(sc, 128, 0), 128, 1))
    assert np.array_equal(got, want)


def test_fp8_weight_matches_torch_dequantization_and_block_layout():
    """General scales: PyTorch's own float8 decoding, fp32 product and bf16
    rounding agree; each element takes the scale of its own 128 x 128 block
    (ragged last blocks included), checked element by element."""
    rng = np.random.default_rng(4)
    rows, cols = 300, 200
    w8 = rng.integers(0, 256, (rows, cols), dtype=np.uint8)
    w8[(w8 & 0x7F) == 0x7F] = 0x22
    sc = (rng.random((3, 2)) * 1e-2 + 1e-3).astype(np.float32)
    got = oracle.dequant_fp8_weight(w8, sc)
    lib_w = torch.from_numpy(w8).view(torch.float8_e4m3fn).float()
    for i in range(rows):
        s_row = torch.from_numpy(np.array([sc[i // 128, j // 128] for j in range(cols)], dtype=np.float32))
        lib = (lib_w[i] * s_row).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(got[i], lib), i
    with pytest.raises(ValueError):
        oracle.dequant_fp8_weight(w8, sc[:2])


# ---------------------------------------------------------------- fp4 quantizer

def test_e4m3_encode_matches_torch_float8_rounding():
    """The oracle's E4M3 encoding (nearest, ties to the even mantissa) against
    PyTorch's float8_e4m3fn conversion on in-range values, with every halfway
    point between neighbouring E4M3 values included."""
    rng = np.random.default_rng(21)
    x = (rng.uniform(-1, 1, 50000) * np.exp2(rng.integers(-12, 9, 50000))).astype(np.float32)
    mags = oracle.e4m3_values(np.arange(0x7F))
    mid = ((mags[:-1] + mags[1:]) / 2).astype(np.float32)            # exact in fp32
    x = np.concatenate([x, mid, -mid, mags.astype(np.float32)])
    x = x[np.abs(x) <= 448]
    ours = oracle.e4m3_encode(x)
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, lib)


def test_e4m3_encode_saturates_and_keeps_the_sign():
    assert list(oracle.e4m3_encode(np.array([448.0, 464.0, 1e30, np.inf, -1e30]))) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE]
    assert list(oracle.e4m3_encode(np.array([0.0, -0.0, 2.0 ** -11, -(2.0 ** -11)]))) == [0x00, 0x80, 0x00, 0x80]


def test_e2m1_encode_halfway_cases_by_hand():
    # halfway between two magnitudes -> the even index (0, 1.0, 2.0, 4.0)
    x = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 0.26, 2.6, 5.1, 7.0, np.inf, -0.0, -0.1, -3.0]
    want = [0, 2, 2, 4, 4, 6, 6, 1, 5, 7, 7, 7, 8, 8, 8 | 5]
    assert list(oracle.e2m1_encode(np.array(x))) == want


def test_fp4_quantize_worked_group():
    """One group worked by hand: amax 12 -> scale E4M3(2.0) = 0x40, then each
    value / 2 to the nearest e2m1 magnitude."""
    x = np.zeros(16, dtype=np.float32)
    x[:8] = [3.0, -1.5, 0.4, 12.0, -12.0, 5.0, 2.5, -0.0]
    codes, scales = oracle.fp4_quantize(oracle.round_bf16(x)[None])
    assert scales[0, 0] == 0x40
    # x / 2 = 1.5, -0.75, 0.2, 6, -6, 2.5, 1.25, -0: idx 3, 2 (tie), 0, 7, 7, 4 (tie), 2 (tie), 0
    nib = [3, 8 | 2, 0, 7, 8 | 7, 4, 2, 8] + [0] * 8
    want = [nib[2 * i] | (nib[2 * i + 1] << 4) for i in range(8)]
    assert list(codes[0]) == want


def test_fp4_quantize_round_trips_the_fp4_grid():
    """Values on the fp4 grid whose group holds a +-6 code: decoding, then
    quantizing again, gives the same codes and scales (amax / 6 is then the
    scale exactly)."""
    rng = np.random.default_rng(22)
    rows, D = 64, 512
    nib = rng.integers(0, 16, (rows, D))
    g = nib.reshape(rows, D // 16, 16)
    pos = rng.integers(0, 16, (rows, D // 16))
    np.put_along_axis(g, pos[..., None], 7 | (8 * rng.integers(0, 2, (rows, D // 16, 1))), axis=-1)
    codes = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    scales = rng.integers(0x08, 0x70, (rows, D // 16)).astype(np.uint8)    # normal scales, 6 x scale finite
    vals = oracle.dequant_fp4(codes, scales)
    c2, s2 = oracle.fp4_quantize(oracle.bf16_bits_exact(vals))
    assert np.array_equal(s2, scales)
    assert np.array_equal(c2, codes)


def test_fp4_quantize_zero_group_and_rounded_down_scale():
    x = np.zeros((2, 16), dtype=np.float32)
    x[0, 3] = -0.0
    x[1, 0] = 6.25          # amax / 6 = 1.0417 -> scale 1.0 (0x38): 6.25 saturates to code 6
    x[1, 1] = -6.25
    codes, scales = oracle.fp4_quantize(oracle.round_bf16(x))
    assert scales[0, 0] == 0x00 and scales[1, 0] == 0x38
    assert codes[0, 1] == 0x80 and np.all(np.delete(codes[0], 1) == 0)     # the -0 keeps its sign
    assert codes[1, 0] == (7 | ((8 | 7) << 4))
