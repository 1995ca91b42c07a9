"""Seeded synthetic inputs for sparse latent attention.

This module is shared by the tests, the benchmark and the fp64 oracle's
callers.  It holds only the input recipes -- random draws, the RMS
normalisation of the synthetic latent rows, and the layout of the index lists
-- and none of the attention arithmetic.

Layout of one batch row's latent rows ("DeepSeek-V4.1 > Output projection"
page, ``Attention.forward``: ``kv = torch.cat([window_kv, compress_kv], 1)``):
rows ``[0, W)`` are the sliding-window ring (slot = position mod W, the ring of
the "DeepSeek-V4.1 > 40 layers" page) and rows ``[W, W + C)`` the compressed
positions, so compressed position ``j`` appears as index ``W + j`` (the
``offset = kv.size(1)`` of ``_compress_kv``).  ``-1`` marks an empty slot.
"""
from __future__ import annotations

import dataclasses
import math

import torch

# eps of the pages' RMSNorm (config.json ``norm_eps``); used only to build the
# synthetic latent rows.
RMS_EPS = 1e-20


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int              # batch rows
    T: int              # queries per batch row
    H: int              # heads (n_heads)
    D: int              # head_dim (latent row width)
    W: int              # window ring slots (window_size)
    C: int              # compressed rows per batch row
    ratio: int          # compress ratio
    K: int              # index-list length per query
    pos0: int           # position of the first query of each batch row
    topk: int           # index_topk: compressed positions listed per query
    kind: str           # index recipe: "all_causal" | "decode" | "prefill"
    skip_frac: float = 0.0      # fraction of compressed entries set to -1 in place
    out_f32: bool = False
    # fused tail (inverse RoPE on the last rope_dim features + grouped wo_a)
    tail: bool = False
    G: int = 8          # o_groups
    R: int = 1024       # o_lora_rank
    rope_dim: int = 64  # rope_head_dim
    theta: float = 160000.0   # compress_rope_theta
    # block tail: the fused tail, then wo_b (G*R group features -> dim)
    wo_b: bool = False
    dim: int = 5120

    @property
    def N(self) -> int:
        return self.W + self.C

    @property
    def scale(self) -> float:
        return self.D ** -0.5

    @property
    def n_queries(self) -> int:
        return self.B * self.T


WORKLOADS = {
    # 16 prefill queries at positions 112..127 over 128 window + 64 compressed rows
    "tiny": Workload("tiny", B=1, T=16, H=64, D=512, W=128, C=64, ratio=2, K=192,
                     pos0=112, topk=64, kind="all_causal", out_f32=True),
    # one decode query per batch row at position 8191 (8192-token context, ratio 2)
    "decode": Workload("decode", B=64, T=1, H=64, D=512, W=128, C=4096, ratio=2, K=640,
                       pos0=8191, topk=512, kind="decode"),
    # 65536-token context, ratio 1; 10% of the 512 compressed entries are -1
    "long_decode": Workload("long_decode", B=128, T=1, H=64, D=512, W=128, C=65536,
                            ratio=1, K=640, pos0=65535, topk=512, kind="decode",
                            skip_frac=0.1),
    # 8192-token prefill, ratio 2
    "prefill": Workload("prefill", B=1, T=8192, H=64, D=512, W=128, C=4096, ratio=2,
                        K=640, pos0=0, topk=512, kind="prefill"),
    # two 4096-token prefills, then inverse RoPE and grouped wo_a
    "fused_tail": Workload("fused_tail", B=2, T=4096, H=64, D=512, W=128, C=4096,
                           ratio=2, K=640, pos0=0, topk=512, kind="prefill", tail=True),
    # the same, continued through wo_b to the model width
    "block_tail": Workload("block_tail", B=2, T=4096, H=64, D=512, W=128, C=4096,
                           ratio=2, K=640, pos0=0, topk=512, kind="prefill", tail=True, wo_b=True),
}


def scaled(wl: Workload, **changes) -> Workload:
    """A copy of a workload with some fields changed (smaller test cases)."""
    return dataclasses.replace(wl, **changes)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def rms_rows(x: torch.Tensor, eps: float = RMS_EPS) -> torch.Tensor:
    """Row RMS normalisation with unit weight, in fp32 (input recipe only)."""
    return x * torch.rsqrt(x.pow(2).mean(-1, keepdim=True) + eps)


def positions(wl: Workload, device="cpu") -> torch.Tensor:
    """int64 [B, T]: the position of every query."""
    t = torch.arange(wl.T, dtype=torch.int64, device=device) + wl.pos0
    return t.unsqueeze(0).expand(wl.B, wl.T).contiguous()


def _window_part(pos: torch.Tensor, W: int) -> torch.Tensor:
    """int32 [Q, W]: ring slots of positions max(0, p-W+1)..p, ascending, -1 padded
    at the end when fewer than W positions exist."""
    Q = pos.numel()
    j = torch.arange(W, device=pos.device, dtype=torch.int64)
    p = pos.reshape(Q, 1)
    first = torch.clamp(p - (W - 1), min=0)
    n = p - first + 1                             # how many window positions exist
    posj = first + j                              # ascending positions
    slot = torch.remainder(posj, W)
    return torch.where(j < n, slot, torch.full_like(slot, -1)).to(torch.int32), n


def _random_subset(limit: torch.Tensor, count: torch.Tensor, C: int, topk: int,
                   g: torch.Generator) -> torch.Tensor:
    """int64 [Q, topk]: for each row, ``count`` distinct uniform draws from
    [0, limit] (inclusive) in random order, then -1."""
    Q = limit.numel()
    dev = limit.device
    keys = torch.rand((Q, C), generator=g, device=dev)
    cand = torch.arange(C, device=dev).unsqueeze(0)
    keys = torch.where(cand <= limit.reshape(Q, 1), keys, torch.full_like(keys, 2.0))
    k = min(topk, C)
    sel = torch.topk(keys, k, dim=1, largest=False, sorted=True).indices
    r = torch.arange(k, device=dev).unsqueeze(0)
    sel = torch.where(r < count.reshape(Q, 1), sel, torch.full_like(sel, -1))
    if k < topk:
        sel = torch.cat([sel, torch.full((Q, topk - k), -1, device=dev, dtype=sel.dtype)], 1)
    return sel


def _pack_valid_first(parts: torch.Tensor) -> torch.Tensor:
    """Stable-move every -1 of each row to the end."""
    invalid = (parts < 0).to(torch.int8)
    order = torch.sort(invalid, dim=1, stable=True).indices
    return torch.gather(parts, 1, order)


def make_indices(wl: Workload, g: torch.Generator, device="cpu") -> torch.Tensor:
    """int32 [B, T, K] index lists following the workload's recipe."""
    pos = positions(wl, device).reshape(-1)
    Q = pos.numel()
    win, _ = _window_part(pos, wl.W)
    climit = torch.div(pos, wl.ratio, rounding_mode="floor")     # compressed rows <= pos // ratio
    climit = torch.clamp(climit, max=wl.C - 1)
    if wl.kind == "all_causal":
        j = torch.arange(wl.C, device=device).unsqueeze(0)
        comp = torch.where(j <= climit.reshape(Q, 1), j, torch.full_like(j, -1)).expand(Q, wl.C)
    elif wl.kind == "decode":
        comp = _random_subset(climit, torch.full_like(climit, wl.topk), wl.C, wl.topk, g)
    elif wl.kind == "prefill":
        count = torch.clamp(torch.div(pos, wl.ratio, rounding_mode="floor"), max=wl.topk)
        comp = _random_subset(climit, count, wl.C, wl.topk, g)
    else:
        raise ValueError(wl.kind)
    comp = torch.where(comp >= 0, comp + wl.W, comp)
    if wl.skip_frac > 0:
        n_skip = int(math.floor(wl.skip_frac * wl.topk))
        kill = torch.topk(torch.rand((Q, comp.shape[1]), generator=g, device=device),
                          n_skip, dim=1).indices
        comp = comp.scatter(1, kill, -1)
        parts = torch.cat([win.to(torch.int64), comp], 1)       # -1s stay in place
    else:
        parts = _pack_valid_first(torch.cat([win.to(torch.int64), comp], 1))
    K = parts.shape[1]
    if K < wl.K:
        parts = torch.cat([parts, torch.full((Q, wl.K - K), -1, device=device,
                                             dtype=parts.dtype)], 1)
    elif K > wl.K:
        if bool((parts[:, wl.K:] >= 0).any()):
            raise ValueError("index recipe does not fit K")
        parts = parts[:, :wl.K]
    return parts.to(torch.int32).reshape(wl.B, wl.T, wl.K).contiguous()


def make_inputs(wl: Workload, seed: int = 0, device="cpu") -> dict:
    """All inputs of one workload, drawn from one seeded generator on ``device``.

    q ~ N(0,1) bf16 [B,T,H,D]; kv rows N(0,1), RMS-normalised in fp32, bf16
    [B,N,D]; sink ~ N(0,1) fp32 [H]; idx int32 [B,T,K]; pos int64 [B,T].  With
    the fused tail also W ~ N(0, 0.02) bf16 [G, R, H*D/G] drawn from seed+1, and
    with the block tail wo_b ~ N(0, 0.02) bf16 [dim, G*R] drawn from seed+2.
    """
    device = torch.device(device)
    g = _gen(seed, device)
    q = torch.randn((wl.B, wl.T, wl.H, wl.D), generator=g, device=device,
                    dtype=torch.float32).to(torch.bfloat16)
    kv = torch.empty((wl.B, wl.N, wl.D), dtype=torch.bfloat16, device=device)
    for b in range(wl.B):       # one batch row at a time keeps fp32 scratch small
        x = torch.randn((wl.N, wl.D), generator=g, device=device, dtype=torch.float32)
        kv[b] = rms_rows(x).to(torch.bfloat16)
    sink = torch.randn((wl.H,), generator=g, device=device, dtype=torch.float32)
    idx = make_indices(wl, g, device)
    out = {"q": q, "kv": kv, "sink": sink, "idx": idx, "pos": positions(wl, device),
           "scale": wl.scale}
    if wl.tail:
        gw = _gen(seed + 1, device)
        din = wl.H * wl.D // wl.G
        out["wo_a"] = (0.02 * torch.randn((wl.G, wl.R, din), generator=gw, device=device,
                                          dtype=torch.float32)).to(torch.bfloat16)
    if wl.wo_b:
        gb = _gen(seed + 2, device)
        out["wo_b"] = (0.02 * torch.randn((wl.dim, wl.G * wl.R), generator=gb, device=device,
                                          dtype=torch.float32)).to(torch.bfloat16)
    return out


def fp8_weight(w: torch.Tensor, block: int = 128) -> tuple[torch.Tensor, torch.Tensor]:
    """A synthetic fp8 checkpoint of a weight [rows, cols] (or [G, R, cols],
    rows = G*R): one fp32 scale per block x block tile, the tile's largest
    magnitude over 448 (the largest E4M3 value), and the E4M3 bytes of
    weight / scale (PyTorch's float8_e4m3fn conversion).  Returns
    (uint8 bytes shaped like w, fp32 scales [ceil(rows/block), ceil(cols/block)])."""
    shape = w.shape
    w2 = w.reshape(-1, shape[-1]).float()
    rows, cols = w2.shape
    nb_r, nb_c = -(-rows // block), -(-cols // block)
    pad = torch.zeros(nb_r * block, nb_c * block, dtype=torch.float32, device=w.device)
    pad[:rows, :cols] = w2.abs()
    amax = pad.view(nb_r, block, nb_c, block).amax(dim=(1, 3))
    scales = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    s_full = scales.repeat_interleave(block, 0)[:rows].repeat_interleave(block, 1)[:, :cols]
    codes = (w2 / s_full).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes.reshape(shape).contiguous(), scales.contiguous()
