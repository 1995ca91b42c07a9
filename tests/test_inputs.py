"""The synthetic workloads follow the shapes printed on the pages and the
index recipes stated for each workload (CPU only)."""
import json
import os

import numpy as np
import pytest
import torch

from sparse_latent_attention_02_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "deepseek_v41_attention_config.json")


def test_workloads_use_the_pages_shapes():
    cfg = json.load(open(GOLDEN))
    # o_groups * o_lora_rank * dim is the printed wo_b parameter count
    assert cfg["o_groups"] * cfg["o_lora_rank"] * cfg["dim"] == cfg["wo_b_parameters_per_instance"]
    for wl in I.WORKLOADS.values():
        assert wl.H == cfg["n_heads"] and wl.D == cfg["head_dim"]
        assert wl.W == cfg["window_size"]
        assert wl.ratio in cfg["compress_ratios_used"]
        assert wl.scale == cfg["head_dim"] ** -0.5
        if wl.kind != "all_causal":
            assert wl.topk == cfg["index_topk"] and wl.K == wl.W + wl.topk
        if wl.tail:
            assert (wl.G, wl.R, wl.rope_dim) == (cfg["o_groups"], cfg["o_lora_rank"],
                                                 cfg["rope_head_dim"])
            assert wl.theta == cfg["compress_rope_theta"]
            assert wl.H * wl.D // wl.G == 4096
    assert I.RMS_EPS == cfg["norm_eps"]


def _check_window(row, p, W):
    first = max(0, p - W + 1)
    want = [x % W for x in range(first, p + 1)]
    assert list(row[:len(want)]) == want
    return len(want)


def test_tiny_recipe():
    wl = I.WORKLOADS["tiny"]
    x = I.make_inputs(wl, seed=0)
    idx = x["idx"].numpy()[0]
    counts = (idx >= 0).sum(1)
    assert counts.min() == 170 and counts.max() == 192
    for t in range(wl.T):
        p = wl.pos0 + t
        nw = _check_window(idx[t], p, wl.W)
        comp = idx[t, nw:counts[t]]
        assert list(comp) == [wl.W + j for j in range(p // 2 + 1)]
        assert np.all(idx[t, counts[t]:] == -1)
    # kv rows are RMS-normalised before rounding
    kv = x["kv"].float()
    rms = kv.pow(2).mean(-1).sqrt()
    assert torch.allclose(rms, torch.ones_like(rms), atol=1e-2)


def test_decode_recipe():
    wl = I.WORKLOADS["decode"]
    g = torch.Generator().manual_seed(0)
    idx = I.make_indices(wl, g).numpy()[:, 0]
    assert idx.shape == (64, 640) and np.all(idx >= 0)
    for b in range(64):
        assert list(idx[b, :128]) == list(range(128))
        comp = idx[b, 128:]
        assert len(set(comp.tolist())) == 512 and comp.min() >= 128 and comp.max() < 128 + 4096


def test_long_decode_recipe_scatters_skips():
    wl = I.scaled(I.WORKLOADS["long_decode"], B=4)
    g = torch.Generator().manual_seed(0)
    idx = I.make_indices(wl, g).numpy()[:, 0]
    for b in range(4):
        comp = idx[b, 128:]
        assert (comp == -1).sum() == 51
        valid = comp[comp >= 0]
        assert len(set(valid.tolist())) == 461 and valid.max() < 128 + 65536
        # the -1 entries are not all at the end
        assert (comp[:461] == -1).any()


def test_prefill_recipe():
    wl = I.scaled(I.WORKLOADS["prefill"], T=1500)
    g = torch.Generator().manual_seed(3)
    idx = I.make_indices(wl, g).numpy()[0]
    for t in [0, 1, 2, 5, 126, 127, 128, 700, 1023, 1024, 1025, 1499]:
        row = idx[t]
        nw = _check_window(row, t, wl.W)
        nc = min(512, t // 2)
        comp = row[nw:nw + nc]
        assert len(set(comp.tolist())) == nc
        if nc:
            assert comp.min() >= wl.W and comp.max() <= wl.W + t // 2
        assert np.all(row[nw + nc:] == -1)
    # valid pairs of the full 8192-query prefill: sum of window + compressed counts
    t = np.arange(8192)
    assert int((np.minimum(t + 1, 128) + np.minimum(512, t // 2)).sum()) == 4972096


def test_fused_tail_recipe():
    """Two batch rows of the prefill recipe at T = 4096: 4,701,312 valid pairs
    (2 x (516,160 window + 1,834,496 compressed)), compressed rows <= t//2."""
    wl = I.WORKLOADS["fused_tail"]
    g = torch.Generator().manual_seed(4)
    idx = I.make_indices(wl, g).numpy()
    assert idx.shape == (2, 4096, 640)
    assert int((idx >= 0).sum()) == 4_701_312
    t = np.arange(4096)
    assert int(np.minimum(t + 1, 128).sum()) == 516_160 and int(np.minimum(512, t // 2).sum()) == 1_834_496
    for b in range(2):
        for t in [0, 3, 127, 128, 1023, 1024, 2047, 4095]:
            row = idx[b, t]
            nw = _check_window(row, t, wl.W)
            nc = min(512, t // 2)
            comp = row[nw:nw + nc]
            assert len(set(comp.tolist())) == nc
            if nc:
                assert comp.min() >= wl.W and comp.max() <= wl.W + t // 2
            assert np.all(row[nw + nc:] == -1)
    # the two batch rows draw their compressed rows independently
    assert not np.array_equal(idx[0, 4095], idx[1, 4095])


def test_block_tail_shares_the_fused_tail_lists():
    a, b = I.WORKLOADS["fused_tail"], I.WORKLOADS["block_tail"]
    assert (a.B, a.T, a.K, a.W, a.C) == (b.B, b.T, b.K, b.W, b.C)
    ia = I.make_indices(a, torch.Generator().manual_seed(9)).numpy()
    ib = I.make_indices(b, torch.Generator().manual_seed(9)).numpy()
    assert np.array_equal(ia, ib)
