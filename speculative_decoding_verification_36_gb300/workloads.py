"""Seeded synthetic workloads for the verify step (inputs only).

This module is the one piece of Python shared by the benchmark, the GPU parity
tests and the oracle tests.  It makes logits, drafted tokens and candidate
trees with torch's seeded generators and holds none of the verify step's own
arithmetic: drafted tokens are drawn with ``torch.multinomial`` /
``torch.argmax`` / ``torch.topk``, i.e. the way a drafter would produce them.

The five presets restate the synthetic workloads of the speculative-decoding
verify benchmark (no page measures the verify step on real model outputs, so
seeded logits with the stated shapes and value distributions stand in for
them):

  c1  chain, B=1,    K=4, V=32000,  fp32, tau=1.0: target N(0, 3^2);
      draft = target + N(0, 1^2); Philox seed 0.
  c2  chain, B=64,   K=5, V=128256, bf16, tau=1.0: target N(0, 4^2) plus +8 on
      one uniformly random id per row; draft = 0.8 * target + N(0, 1.5^2).
  c3  chain, B=256,  K=8, V=152064, bf16, tau=0.7: target N(0, 4^2) plus the
      Zipf(1.1)-shaped prior -1.1 * ln(v + 1); draft = target + N(0, 2^2).
  c4  greedy, B=1024, K=4, V=128256, bf16, tau=0: target N(0, 4^2); each
      drafted token is the target argmax with probability 0.7, else uniform.
  c5  tree greedy, B=32, N=30 (complete binary tree of depth 4 in BFS order),
      V=128256, bf16: target N(0, 4^2) for the root and every node; the two
      children of a node carry the top-2 ids of (that node's row + N(0, 1^2)).

The stochastic tree workload (spec_tree_verify_sampling) takes a tree preset's
shapes and a temperature: target N(0, 4^2) for the root and every node, draft
= target + N(0, 1.5^2) row by row, and the children of a node drawn i.i.d.
(with replacement) from softmax(that node's draft row / tau).

Logits are generated in fp32 and rounded to the preset's dtype before the
draft tokens are drawn, so tokens come from exactly the bits the verifier
reads.  Drafted chain tokens are drawn from softmax(draft / tau).
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class ChainPreset:
    name: str
    B: int
    K: int
    V: int
    dtype: torch.dtype
    temperature: float
    seed: int
    kind: str  # "c1" | "c2" | "c3" | "c4"


@dataclass(frozen=True)
class TreePreset:
    name: str
    B: int
    depth: int
    V: int
    dtype: torch.dtype
    seed: int

    @property
    def N(self) -> int:
        return 2 ** (self.depth + 1) - 2


PRESETS = {
    "c1": ChainPreset("c1", 1, 4, 32000, torch.float32, 1.0, 0, "c1"),
    "c2": ChainPreset("c2", 64, 5, 128256, torch.bfloat16, 1.0, 0, "c2"),
    "c3": ChainPreset("c3", 256, 8, 152064, torch.bfloat16, 0.7, 0, "c3"),
    "c4": ChainPreset("c4", 1024, 4, 128256, torch.bfloat16, 0.0, 0, "c4"),
    "c5": TreePreset("c5", 32, 4, 128256, torch.bfloat16, 0),
}

_PRESET_INDEX = {"c1": 1, "c2": 2, "c3": 3, "c4": 4, "c5": 5}


def preset(name: str, **overrides):
    """A preset with some fields replaced (e.g. a smaller B or V)."""
    return replace(PRESETS[name], **overrides)


def _gen(device, kind: str, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(12345 + 1000 * _PRESET_INDEX.get(kind, 0) + int(seed))
    return g


def _randn(shape, g, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def _sample_rows(logits_f32: torch.Tensor, temperature: float, g) -> torch.Tensor:
    """One token per row from softmax(logits / temperature) (torch.multinomial)."""
    flat = logits_f32.reshape(-1, logits_f32.shape[-1])
    probs = torch.softmax(flat / temperature, dim=-1)
    out = torch.empty(flat.shape[0], dtype=torch.int64, device=flat.device)
    step = 4096
    for i in range(0, flat.shape[0], step):
        out[i:i + step] = torch.multinomial(probs[i:i + step], 1, generator=g).squeeze(-1)
    return out.reshape(logits_f32.shape[:-1]).to(torch.int32)


def make_chain(p: ChainPreset, device="cpu", seed: int | None = None):
    """Inputs of a chain preset.

    Returns dict(target [B,K+1,V], draft [B,K,V] (None for the greedy preset),
    tokens [B,K] int32, temperature, seed).
    """
    seed = p.seed if seed is None else seed
    g = _gen(device, p.kind, seed)
    B, K, V = p.B, p.K, p.V
    if p.kind == "c1":
        t32 = 3.0 * _randn((B, K + 1, V), g, device)
        target = t32.to(p.dtype)
        d32 = target[:, :K].float() + 1.0 * _randn((B, K, V), g, device)
    elif p.kind == "c2":
        t32 = 4.0 * _randn((B, K + 1, V), g, device)
        spike = torch.randint(0, V, (B, K + 1, 1), generator=g, device=device)
        t32.scatter_add_(2, spike, torch.full((B, K + 1, 1), 8.0, device=device))
        target = t32.to(p.dtype)
        d32 = 0.8 * target[:, :K].float() + 1.5 * _randn((B, K, V), g, device)
    elif p.kind == "c3":
        prior = -1.1 * torch.log(torch.arange(V, device=device, dtype=torch.float32) + 1.0)
        t32 = 4.0 * _randn((B, K + 1, V), g, device) + prior
        target = t32.to(p.dtype)
        d32 = target[:, :K].float() + 2.0 * _randn((B, K, V), g, device)
    elif p.kind == "c4":
        t32 = 4.0 * _randn((B, K + 1, V), g, device)
        target = t32.to(p.dtype)
        amax = torch.argmax(target[:, :K].float(), dim=-1).to(torch.int32)
        rand = torch.randint(0, V, (B, K), generator=g, device=device, dtype=torch.int32)
        keep = torch.rand((B, K), generator=g, device=device) < 0.7
        tokens = torch.where(keep, amax, rand).contiguous()
        return dict(target=target.contiguous(), draft=None, tokens=tokens,
                    temperature=0.0, seed=seed)
    else:
        raise ValueError(p.kind)
    draft = d32.to(p.dtype).contiguous()
    tokens = _sample_rows(draft.float(), p.temperature, g)
    return dict(target=target.contiguous(), draft=draft, tokens=tokens.contiguous(),
                temperature=p.temperature, seed=seed)


def complete_binary_parents(depth: int) -> torch.Tensor:
    """parent_idx of a complete binary tree of the given depth in BFS order
    (the root itself is not a node; its two children are nodes 0 and 1)."""
    n = 2 ** (depth + 1) - 2
    return torch.tensor([i // 2 - 1 for i in range(n)], dtype=torch.int32)


def make_tree(p: TreePreset, device="cpu", seed: int | None = None, parents=None):
    """Inputs of a tree preset: dict(target [B,N+1,V], tokens [B,N], parents [B,N]).

    ``parents`` overrides the complete binary tree with any BFS-ordered parent
    list; every node's children then take the top ids of (its row + noise)."""
    seed = p.seed if seed is None else seed
    g = _gen(device, "c5", seed)
    par = complete_binary_parents(p.depth) if parents is None else torch.as_tensor(
        parents, dtype=torch.int32)
    N = int(par.numel())
    B, V = p.B, p.V
    target = (4.0 * _randn((B, N + 1, V), g, device)).to(p.dtype).contiguous()
    tokens = torch.empty((B, N), dtype=torch.int32, device=device)
    children = {}
    for i, pr in enumerate(par.tolist()):
        children.setdefault(pr, []).append(i)
    for pr, kids in children.items():
        row = target[:, pr + 1].float() + _randn((B, V), g, device)
        top = torch.topk(row, len(kids), dim=-1).indices.to(torch.int32)
        for j, node in enumerate(kids):
            tokens[:, node] = top[:, j]
    parents_b = par.to(device).unsqueeze(0).expand(B, N).contiguous()
    return dict(target=target, tokens=tokens.contiguous(), parents=parents_b)


def make_tree_sampling(p: TreePreset, temperature: float = 1.0, device="cpu", seed: int | None = None,
                       parents=None):
    """Inputs of the stochastic tree workload: dict(target, draft [B,N+1,V],
    tokens, parents [B,N], temperature).  ``parents`` overrides the complete
    binary tree with any BFS-ordered parent list."""
    seed = p.seed if seed is None else seed
    g = _gen(device, "c5s", seed)
    par = complete_binary_parents(p.depth) if parents is None else torch.as_tensor(
        parents, dtype=torch.int32)
    N = int(par.numel())
    B, V = p.B, p.V
    target = (4.0 * _randn((B, N + 1, V), g, device)).to(p.dtype).contiguous()
    draft = (target.float() + 1.5 * _randn((B, N + 1, V), g, device)).to(p.dtype).contiguous()
    tokens = torch.empty((B, N), dtype=torch.int32, device=device)
    children = {}
    for i, pr in enumerate(par.tolist()):
        children.setdefault(pr, []).append(i)
    for pr, kids in children.items():
        probs = torch.softmax(draft[:, pr + 1].float() / temperature, dim=-1)
        drawn = torch.multinomial(probs, len(kids), replacement=True, generator=g).to(torch.int32)
        for j, node in enumerate(kids):
            tokens[:, node] = drawn[:, j]
    parents_b = par.to(device).unsqueeze(0).expand(B, N).contiguous()
    return dict(target=target, draft=draft, tokens=tokens.contiguous(), parents=parents_b,
                temperature=float(temperature))


def make_ngram_histories(B: int, Lmax: int, V: int = 128256, seed: int = 0, copy_prob: float = 0.5,
                         device="cpu", alphabet: int | None = None):
    """Token histories for n-gram drafting: dict(tokens [B, Lmax] int32,
    lengths [B] int32).

    The pages place n-gram lookup on input-grounded, repetitive work
    (summaries and code edits that echo their input), so each history is
    built from segments: with probability copy_prob a segment copies a span
    of 8-64 tokens from earlier in the same history, otherwise it is 8-64
    fresh tokens drawn uniformly from [0, V) (or [0, alphabet) when given, for
    dense small-vocabulary cases).  Lengths are uniform in [Lmax / 2, Lmax];
    entries past a row's length are -7 (never read)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(12345 + 1000 * 7 + int(seed))
    hi = V if alphabet is None else alphabet
    tokens = torch.full((B, Lmax), -7, dtype=torch.int32)
    lengths = torch.randint(max(Lmax // 2, 0), Lmax + 1, (B,), generator=g, dtype=torch.int32)
    for b in range(B):
        L = int(lengths[b])
        row = []
        while len(row) < L:
            n = int(torch.randint(8, 65, (1,), generator=g))
            if row and float(torch.rand((1,), generator=g)) < copy_prob:
                start = int(torch.randint(0, len(row), (1,), generator=g))
                seg = row[start:start + n]
            else:
                seg = torch.randint(0, hi, (n,), generator=g, dtype=torch.int32).tolist()
            row.extend(seg)
        tokens[b, :L] = torch.tensor(row[:L], dtype=torch.int32)
    return dict(tokens=tokens.to(device), lengths=lengths.to(device))
