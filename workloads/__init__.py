"""Seeded synthetic inputs for the verification workloads.

This module is the one piece that both the CUDA path's tests and the float64
oracle consume.  It produces *inputs only*: target logits, draft proposal
distributions q (the stand-in for a draft model), draft tokens sampled from
q, uniforms, DSpark confidences, and the DDTree target rows.  It computes
none of the verification method itself (no p, no acceptance, no residual,
no tree, no verify length); the random numbers the method consumes are
drawn here and passed in as inputs.

Workload shapes follow the settings the source pages use: an EAGLE-3 draft
of 3 tokens on a Llama-3.1-8B vocabulary (128256), DFlash/DSpark blocks of
7-8 on a Qwen3-8B vocabulary (151936), a 16-position DDTree block.  No
public dataset is used; the seeded Gaussian logits stand in for model
outputs.

All tensors are generated with torch on the requested device from a seeded
``torch.Generator``; the same call on the same device and torch build yields
the same bits.  Tests hand the CUDA library and the oracle the very same
tensors (the oracle receives host copies), so both sides always see
identical inputs.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch

# name -> (index, description); the seed of a workload is 1000 + index
WORKLOADS = {
    "chain_small": (0, "chain verify B=4 K=4 V=1000, fp32 logits N(0,2^2), T=1, no top-k"),
    "eagle3": (1, "chain verify B=64 K=3 V=128256, bf16 logits N(0,3^2), T=0.8, no top-k"),
    "dflash": (2, "block-draft chain verify B=256 K=8 V=151936, fp32 logits N(0,3^2), T=1, top-k 50"),
    "ddtree": (3, "DDTree B=32 L=16 budget 64 V=151936, q fp32, target bf16"),
    "dspark": (4, "DSpark adaptive ragged verify B=512 Kmax=8 V=128256, bf16, T=1, top-k 50"),
    "dflash_vs": (5, "block-draft chain verify, DFlash shape, every row with its own logit scale "
                     "U[0.5, 6] and offset U[-20, 20], T=1, top-k 50"),
    "eagle2": (6, "EAGLE-2 dynamic tree B=32 V=151936: 6 expansion steps, 10 children per node, "
                  "frontier 10, budget 60; conditional draft rows softmax(N(0,3^2)) per path"),
}

DEFAULTS = {
    "chain_small": dict(B=4, K=4, V=1000, dtype="f32", sigma=2.0, T=1.0, top_k=0),
    "eagle3": dict(B=64, K=3, V=128256, dtype="bf16", sigma=3.0, T=0.8, top_k=0),
    "dflash": dict(B=256, K=8, V=151936, dtype="f32", sigma=3.0, T=1.0, top_k=50),
    "ddtree": dict(B=32, L=16, N=64, V=151936),
    "dspark": dict(B=512, K=8, V=128256, dtype="bf16", sigma=3.0, T=1.0, top_k=50,
                   a=1.0, b=0.15),
    "dflash_vs": dict(B=256, K=8, V=151936, dtype="f32", sigma=3.0, T=1.0, top_k=50),
    "eagle2": dict(B=32, V=151936, steps=6, K2=10, Fn=10, N=60, sigma=3.0),
}


def seed_of(name: str) -> int:
    return 1000 + WORKLOADS[name][0]


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _sample_rows(q2d: torch.Tensor, g: torch.Generator) -> torch.Tensor:
    """One token per row of the probability matrix q2d (the draft's sample)."""
    if q2d.shape[0] == 0:
        return torch.empty(0, dtype=torch.int32, device=q2d.device)
    out = []
    step = 4096
    for s in range(0, q2d.shape[0], step):
        out.append(torch.multinomial(q2d[s:s + step], 1, generator=g).squeeze(1))
    return torch.cat(out).to(torch.int32)


def _truncate_top(z: torch.Tensor, k: int) -> torch.Tensor:
    """Draft-side truncation of the noisy draft logits to their k largest
    entries (the draft model's own top-k); the rest become -inf."""
    if k <= 0 or k >= z.shape[-1]:
        return z
    kth = torch.topk(z, k, dim=-1).values[..., -1:]
    return torch.where(z >= kth, z, torch.full_like(z, float("-inf")))


@dataclass
class ChainInputs:
    """Inputs of one chain-verification call (dense layout)."""
    name: str
    logits: torch.Tensor          # [B, K+1, V] fp32 or bf16
    q: torch.Tensor               # [B, K, V] fp32 probabilities
    draft: torch.Tensor           # [B, K] int32
    uniforms: torch.Tensor        # [B, K+1] fp32 in [0, 1)
    temperature: float
    top_k: int
    draft_greedy: Optional[torch.Tensor] = None   # [B, K] argmax of the noisy draft logits
    conf: Optional[torch.Tensor] = None           # [B, K] DSpark confidences
    meta: dict = field(default_factory=dict)

    @property
    def B(self):
        return self.draft.shape[0]

    @property
    def K(self):
        return self.draft.shape[1]

    @property
    def V(self):
        return self.logits.shape[-1]


def make_chain(name: str, device="cpu", seed: Optional[int] = None, **over) -> ChainInputs:
    """Chain workloads: 'chain_small', 'eagle3', 'dflash', 'dspark' (dense
    rows for every position up to Kmax; the ragged call packs them).

    Keyword overrides (B, K, V, ...) shrink a workload for quick tests while
    keeping its value distributions.
    """
    cfg = dict(DEFAULTS[name])
    cfg.update(over)
    B, K, V = cfg["B"], cfg["K"], cfg["V"]
    seed = seed_of(name) if seed is None else seed
    g = _gen(device, seed)
    sigma = cfg["sigma"]
    logits32 = torch.randn((B, K + 1, V), generator=g, device=device) * sigma
    row_scale = None
    if name == "dflash_vs":
        # every row its own scale and offset: the top-k threshold of one row
        # says little about the next row's (or the next call's)
        row_scale = torch.rand((B, K + 1, 1), generator=g, device=device) * 5.5 + 0.5
        offset = torch.rand((B, K + 1, 1), generator=g, device=device) * 40.0 - 20.0
        logits32 = logits32 / sigma * row_scale + offset
    if cfg["dtype"] == "bf16":
        logits = logits32.to(torch.bfloat16)
        base = logits.float()
    else:
        logits = logits32
        base = logits32
    base = base[:, :K, :]
    draft_greedy = None
    if name == "chain_small":
        z = base + torch.randn((B, K, V), generator=g, device=device) * 0.5
    elif name == "eagle3":
        z = base * 0.9 + torch.randn((B, K, V), generator=g, device=device)
        draft_greedy = torch.argmax(z, dim=-1).to(torch.int32)
    elif name in ("dflash", "dflash_vs"):
        # noise std grows linearly from 0.5 to 2.0 across the block (relative
        # to the row's own scale for the varying-scale variant)
        stds = torch.linspace(0.5, 2.0, K, device=device) if K > 1 else torch.full((1,), 0.5, device=device)
        noise = torch.randn((B, K, V), generator=g, device=device) * stds.view(1, K, 1)
        if row_scale is not None:
            noise = noise * (row_scale[:, :K] / sigma)
        z = base + noise
        del noise
        z = _truncate_top(z, cfg["top_k"])       # "top-k applied to both p and q"
    elif name == "dspark":
        z = base + torch.randn((B, K, V), generator=g, device=device) * 1.0
    else:
        raise ValueError(name)
    q = torch.softmax(z, dim=-1).float().contiguous()
    del z
    draft = _sample_rows(q.view(B * K, V), g).view(B, K)
    uniforms = torch.rand((B, K + 1), generator=g, device=device)
    conf = None
    if name == "dspark":
        # conditional confidences c_i ~ Beta(8, 2), drawn from two Gammas
        ga = torch._standard_gamma(torch.full((B, K), 8.0, device=device), generator=g)
        gb = torch._standard_gamma(torch.full((B, K), 2.0, device=device), generator=g)
        conf = (ga / (ga + gb)).float()
    return ChainInputs(name=name, logits=logits.contiguous(), q=q, draft=draft.contiguous(),
                       uniforms=uniforms.contiguous(), temperature=cfg["T"], top_k=cfg["top_k"],
                       draft_greedy=draft_greedy, conf=conf,
                       meta=dict(cfg, seed=seed))


def pack_ragged(logits: torch.Tensor, q: torch.Tensor, k: torch.Tensor,
                l_row_off: torch.Tensor, q_row_off: torch.Tensor):
    """Gather the first k_b+1 logits rows and first k_b q rows of every
    request into packed row-major buffers at the given row offsets.

    This is layout only: the offsets come from the caller (the verify-length
    step of whichever side is under test)."""
    B, _, V = logits.shape
    kc = k.to(torch.int64).cpu()
    lo = l_row_off.to(torch.int64).cpu()
    qo = q_row_off.to(torch.int64).cpu()
    nl, nq = int(lo[B]), int(qo[B])
    pl = torch.empty((max(nl, 1), V), dtype=logits.dtype, device=logits.device)
    pq = torch.empty((max(nq, 1), V), dtype=q.dtype, device=q.device)
    for b in range(B):
        kb = int(kc[b])
        pl[int(lo[b]):int(lo[b]) + kb + 1] = logits[b, :kb + 1]
        if kb > 0:
            pq[int(qo[b]):int(qo[b]) + kb] = q[b, :kb]
    return pl, pq


@dataclass
class TreeInputs:
    name: str
    q_logits: torch.Tensor     # [B, L, V] fp32 draft logits of the block drafter
    q: torch.Tensor            # [B, L, V] fp32 per-position marginals
    budget: int
    meta: dict = field(default_factory=dict)


def make_tree(name: str = "ddtree", device="cpu", seed: Optional[int] = None, **over) -> TreeInputs:
    """DDTree block: per-position marginals q_i = softmax(N(0, 3^2)) of a
    block drafter (fp32), and the node budget."""
    cfg = dict(DEFAULTS[name])
    cfg.update(over)
    B, L, V = cfg["B"], cfg["L"], cfg["V"]
    seed = seed_of(name) if seed is None else seed
    g = _gen(device, seed)
    ql = torch.randn((B, L, V), generator=g, device=device) * 3.0
    q = torch.softmax(ql, dim=-1).float().contiguous()
    return TreeInputs(name=name, q_logits=ql, q=q, budget=cfg["N"], meta=dict(cfg, seed=seed))


def tree_target_logits(tree: TreeInputs, depth: torch.Tensor, seed: Optional[int] = None,
                       dtype=torch.bfloat16) -> torch.Tensor:
    """Target logits [B, N, V] for the nodes of a built tree: the row of a
    node at depth d is the drafter's logits of position d+1 plus N(0, 1)
    noise; a node at the last depth L gets fresh N(0, 3^2) logits.  Unused
    node slots (depth < 0) get fresh N(0, 3^2) logits too."""
    B, L, V = tree.q_logits.shape
    N = depth.shape[1]
    dev = tree.q_logits.device
    seed = (seed_of(tree.name) + 7919) if seed is None else seed
    g = _gen(dev, seed)
    d = depth.to(torch.int64).to(dev)
    out = torch.randn((B, N, V), generator=g, device=dev)            # N(0, 1)
    fresh = torch.randn((B, N, V), generator=g, device=dev) * 3.0    # N(0, 3^2)
    use_q = (d >= 0) & (d < L)
    idx = d.clamp(0, L - 1)
    base = torch.gather(tree.q_logits, 1, idx.unsqueeze(-1).expand(B, N, V))
    out = torch.where(use_q.unsqueeze(-1), base + out, fresh)
    return out.to(dtype).contiguous()


def tree_uniforms(tree: TreeInputs, max_depth: int, seed: Optional[int] = None) -> torch.Tensor:
    """Uniforms [B, max_depth+1] in [0, 1) for a stochastic tree walk (one
    per depth), seeded."""
    B = tree.q_logits.shape[0]
    dev = tree.q_logits.device
    g = _gen(dev, (seed_of(tree.name) + 4093) if seed is None else seed)
    return torch.rand((B, max_depth + 1), generator=g, device=dev).contiguous()


def path_key(path) -> int:
    """A stable 32-bit key of a token path (the draft's conditioning)."""
    import zlib
    import numpy as np
    return zlib.crc32(np.asarray(path, dtype=np.int32).tobytes())


def eagle2_rows(paths, V: int, seed: int, device="cpu", sigma: float = 3.0) -> torch.Tensor:
    """Conditional draft rows for an EAGLE-2 step: paths[b][f] is the token
    path of request b's frontier slot f (None: no row).  Row (b, f) is
    softmax(N(0, sigma^2)) drawn from a generator seeded by (seed, b, path),
    so the same node gets the same row whatever the step or the caller.
    Returns [B, F, V] fp32 (absent rows zero)."""
    B = len(paths)
    F = max((len(p) for p in paths), default=1) or 1
    out = torch.zeros((B, F, V), dtype=torch.float32, device=device)
    for b in range(B):
        for f, path in enumerate(paths[b]):
            if path is None:
                continue
            g = _gen(device, (int(seed) * 1000003 + b * 7919 + path_key(path)) % (1 << 62))
            z = torch.randn((V,), generator=g, device=device) * sigma
            out[b, f] = torch.softmax(z, dim=-1)
    return out


def rotate_copies(fn, name: str, n: int, **kw):
    """n independently seeded copies of a workload (seeds s, s+100, ...),
    used to keep successive benchmark steps from re-reading rows that the
    previous step left in L2."""
    return [fn(name, seed=seed_of(name) + 100 * i, **kw) for i in range(n)]
