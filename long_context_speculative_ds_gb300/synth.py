"""Seeded synthetic inputs for the tree-verify step.

This module only draws inputs: random bf16 queries and paged K/V caches,
random draft trees, shuffled page tables, fp32 logits, draft tokens and
uniforms, with the shapes and distributions of the five workloads below.
It computes none of the verify step's results; the CUDA path and the float64
oracle both consume the tensors it returns.

Workloads follow the problem statement of DiffSpec-style long-context
speculation (vllm-diffspec README, "What DiffSpec Does" and "Key Results":
Llama-3.1-8B at 32K-128K context; adaptive-specdec README: Qwen3-8B target).

Distributions:
  * Q, K, V ~ N(0, 1), rounded to bf16.
  * target logits ~ N(0, 2) (variance 2); draft logits either i.i.d. N(0, 2)
    ("iid") or target + N(0, 1) ("noisy").
  * page table: a random permutation of one shared page pool, consecutive runs
    of that permutation per sequence (so sequences interleave physically).
  * tree: parent[j] uniform among earlier nodes that still satisfy the depth
    and branching caps; node 0 is the root (parent -1).
  * planted salient chunks: every key of a planted chunk is replaced by
    |k| * (0.5 u + sqrt(0.75) v_perp), u the unit mean of that KV head's group
    of tree queries and v_perp a random unit vector orthogonal to u (cosine 0.5).
  * draft tokens: for rejection workloads each child of node i is drawn from
    softmax(draft[i]) by the Gumbel-max trick; for greedy workloads the first
    child of i copies argmax(target[i]) with probability 0.6, every other
    token is uniform over the vocabulary.
  * uniforms ~ U[0, 1) fp32, two per node.

Seeds: the structure of workload number n uses seed 1000*n; layer l of that
workload uses seed 1000*n + 1 + l.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass
from typing import List, Optional, Sequence

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    number: int
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    layers: int
    page_size: int
    ctx_lens: Optional[Sequence[int]]      # None: drawn log-uniform in ctx_range
    tree_sizes: Optional[Sequence[int]]    # None: drawn uniform in tree_range
    max_depth: int
    max_branch: int
    chunk_size: int
    top_k: int
    window: int
    vocab: int
    accept: str                            # "greedy", "reject" or "both"
    planted: int                           # planted salient chunks per sequence
    draft: Optional[str]                   # None, "iid" or "noisy"
    ctx_range: Sequence[int] = (4096, 131072)
    tree_range: Sequence[int] = (16, 64)
    # RoPE base of the draft's compact cache (the model family's rotary theta:
    # 500000 for Llama 3.1, 1000000 for Qwen3, 10000 for the tiny case)
    rope_base: float = 10000.0

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 4, 2, 64, 1, 16, (512,), (8,), 4, 64,
                     32, 4, 64, 256, "both", 0, "iid"),
    "llama8b-32k": Workload("llama8b-32k", 2, 1, 32, 8, 128, 1, 16, (32768,),
                            (32,), 8, 3, 64, 64, 1024, 128256, "greedy", 16,
                            None, rope_base=500000.0),
    "llama8b-64k": Workload("llama8b-64k", 3, 1, 32, 8, 128, 1, 16, (65536,),
                            (64,), 10, 4, 64, 128, 2048, 128256, "reject", 32,
                            "noisy", rope_base=500000.0),
    "llama8b-128k-32l": Workload("llama8b-128k-32l", 4, 1, 32, 8, 128, 32, 16,
                                 (131072,), (64,), 10, 4, 64, 256, 2048,
                                 128256, "greedy", 32, None, rope_base=500000.0),
    "qwen3-8b-ragged-b8": Workload("qwen3-8b-ragged-b8", 5, 8, 32, 8, 128, 36,
                                   16, None, None, 10, 4, 64, 128, 1024,
                                   151936, "reject", 0, "noisy",
                                   rope_base=1000000.0),
}


@dataclass
class Structure:
    """Per-step structure shared by all layers (host tensors, int32)."""
    workload: Workload
    ctx_lens: List[int]
    tree_sizes: List[int]
    tree_offsets: List[int]
    parents: List[int]          # local parent index per node, -1 for roots
    page_table: torch.Tensor    # [batch, max_pages] int32, -1 where unused
    num_pages: int
    max_pages: int
    planted_chunks: List[List[int]]

    @property
    def n_nodes(self) -> int:
        return self.tree_offsets[-1]


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randint(g: torch.Generator, lo: int, hi: int) -> int:
    """Uniform integer in [lo, hi]."""
    return int(torch.randint(lo, hi + 1, (1,), generator=g).item())


def random_tree(n: int, max_depth: int, max_branch: int,
                g: torch.Generator) -> List[int]:
    """Topologically ordered parent array: parent[0] = -1, parent[j] < j."""
    if n <= 0:
        return []
    parents = [-1]
    depth = [0]
    nchild = [0]
    for j in range(1, n):
        eligible = [i for i in range(j)
                    if depth[i] < max_depth and nchild[i] < max_branch]
        if not eligible:
            raise ValueError("tree caps leave no eligible parent")
        p = eligible[_randint(g, 0, len(eligible) - 1)]
        parents.append(p)
        depth.append(depth[p] + 1)
        nchild.append(0)
        nchild[p] += 1
    return parents


def make_structure(wl: Workload, seed: Optional[int] = None,
                   ctx_lens: Optional[Sequence[int]] = None,
                   tree_sizes: Optional[Sequence[int]] = None,
                   parents: Optional[Sequence[int]] = None,
                   spare_pages: int = 0) -> Structure:
    g = _gen(1000 * wl.number if seed is None else seed)
    B = wl.batch
    if ctx_lens is None:
        ctx_lens = wl.ctx_lens
    if ctx_lens is None:
        lo, hi = wl.ctx_range
        u = torch.rand(B, generator=g, dtype=torch.float64)
        ctx_lens = [int(round(math.exp(math.log(lo) + float(x) *
                                       (math.log(hi) - math.log(lo)))))
                    for x in u]
    ctx_lens = [int(x) for x in ctx_lens]
    if tree_sizes is None:
        tree_sizes = wl.tree_sizes
    if tree_sizes is None:
        lo, hi = wl.tree_range
        tree_sizes = [_randint(g, lo, hi) for _ in range(B)]
    tree_sizes = [int(x) for x in tree_sizes]
    assert len(ctx_lens) == B and len(tree_sizes) == B
    offsets = [0]
    for t in tree_sizes:
        offsets.append(offsets[-1] + t)
    if parents is None:
        parents = []
        for t in tree_sizes:
            parents += random_tree(t, wl.max_depth, wl.max_branch, g)
    parents = [int(x) for x in parents]
    assert len(parents) == offsets[-1]

    P = wl.page_size
    need = [-(-(L + T) // P) for L, T in zip(ctx_lens, tree_sizes)]
    num_pages = sum(need) + spare_pages
    max_pages = max(1, max(need) if need else 1)
    perm = torch.randperm(max(num_pages, 1), generator=g)[:num_pages]
    table = torch.full((B, max_pages), -1, dtype=torch.int32)
    pos = 0
    for b in range(B):
        table[b, :need[b]] = perm[pos:pos + need[b]].to(torch.int32)
        pos += need[b]

    planted = []
    for b in range(B):
        ws = max(0, ctx_lens[b] - wl.window)
        n_cand = ws // wl.chunk_size
        n = min(wl.planted, n_cand)
        if n > 0:
            pick = torch.randperm(n_cand, generator=g)[:n]
            planted.append(sorted(int(c) for c in pick))
        else:
            planted.append([])
    return Structure(wl, ctx_lens, tree_sizes, offsets, parents, table,
                     num_pages, max_pages, planted)


def _slot_index(st: Structure, b: int, t: torch.Tensor):
    P = st.workload.page_size
    page = st.page_table[b].to(torch.int64)[t // P]
    return page, t % P


def make_layer(st: Structure, layer: int = 0, device="cpu",
               layout: str = "NHD", seed: Optional[int] = None,
               plant: bool = True):
    """Q [n_nodes, H_q, D] and paged K, V caches (bf16) for one layer.

    NHD layout: [num_pages, page_size, H_kv, D]; HND: [num_pages, H_kv,
    page_size, D].  The tree's own keys/values occupy slots
    ctx_len .. ctx_len + T - 1 of each sequence, in node order.
    """
    wl = st.workload
    s = (1000 * wl.number + 1 + layer) if seed is None else seed
    g = _gen(s, device)
    H, Hkv, D, P = wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.page_size
    npg = max(st.num_pages, 1)
    q = torch.randn(st.n_nodes, H, D, generator=g, device=device,
                    dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn(npg, P, Hkv, D, generator=g, device=device,
                    dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn(npg, P, Hkv, D, generator=g, device=device,
                    dtype=torch.float32).to(torch.bfloat16)
    if plant:
        G = H // Hkv
        C = wl.chunk_size
        for b in range(wl.batch):
            if not st.planted_chunks[b]:
                continue
            n0, n1 = st.tree_offsets[b], st.tree_offsets[b + 1]
            qb = q[n0:n1].float().view(n1 - n0, Hkv, G, D)
            u = qb.mean(dim=(0, 2))                                # [Hkv, D]
            u = u / u.norm(dim=-1, keepdim=True)
            toks = torch.cat([torch.arange(c * C, (c + 1) * C)
                              for c in st.planted_chunks[b]]).to(device)
            page, off = _slot_index(st, b, toks.cpu())
            page, off = page.to(device), off.to(device)
            kk = k[page, off].float()                              # [n, Hkv, D]
            r = torch.randn(kk.shape, generator=g, device=device)
            r = r - (r * u).sum(-1, keepdim=True) * u
            r = r / r.norm(dim=-1, keepdim=True)
            newk = kk.norm(dim=-1, keepdim=True) * (0.5 * u + math.sqrt(0.75) * r)
            k[page, off] = newk.to(torch.bfloat16)
    if layout == "HND":
        k = k.permute(0, 2, 1, 3).contiguous()
        v = v.permute(0, 2, 1, 3).contiguous()
    elif layout != "NHD":
        raise ValueError(layout)
    return q, k, v


def make_source_cache(st: Structure, device="cpu", layout: str = "NHD",
                      seed: Optional[int] = None):
    """The draft's canonical K/V cache that the compact gather copies from:
    one more single-layer paged cache sharing the target's page table."""
    wl = st.workload
    return make_layer(st, layer=-1, device=device, layout=layout,
                      seed=(1000 * wl.number + 999) if seed is None else seed,
                      plant=False)[1:]


@dataclass
class AcceptInputs:
    target_logits: torch.Tensor            # [n_nodes, V] fp32
    draft_logits: Optional[torch.Tensor]   # [n_nodes, V] fp32 or None
    draft_tokens: torch.Tensor             # [n_nodes] int32 (root ignored)
    uniforms: torch.Tensor                 # [n_nodes, 2] fp32


def make_accept_inputs(st: Structure, mode: str, device="cpu",
                       seed: Optional[int] = None,
                       draft: Optional[str] = None) -> AcceptInputs:
    wl = st.workload
    s = (1000 * wl.number + 500) if seed is None else seed
    g = _gen(s)                     # drawn on the host, then moved
    n, V = st.n_nodes, wl.vocab
    draft = draft if draft is not None else (wl.draft or "noisy")
    target = torch.randn(n, V, generator=g) * math.sqrt(2.0)
    dl = None
    if mode == "reject":
        if draft == "iid":
            dl = torch.randn(n, V, generator=g) * math.sqrt(2.0)
        else:
            dl = target + torch.randn(n, V, generator=g)
    tokens = torch.zeros(n, dtype=torch.int32)
    for b in range(wl.batch):
        n0 = st.tree_offsets[b]
        seen_child = set()
        for j in range(1, st.tree_sizes[b]):
            p = st.parents[n0 + j]
            if mode == "reject":
                # Gumbel-max: argmax(l + G) is a draw from softmax(l).
                u = torch.rand(V, generator=g, dtype=torch.float64)
                u = u.clamp_min(1e-300)
                gum = -torch.log(-torch.log(u))
                tokens[n0 + j] = int(torch.argmax(dl[n0 + p].double() + gum))
            else:
                first = p not in seen_child
                seen_child.add(p)
                coin = float(torch.rand(1, generator=g))
                rnd = _randint(g, 0, V - 1)
                if first and coin < 0.6:
                    tokens[n0 + j] = int(torch.argmax(target[n0 + p]))
                else:
                    tokens[n0 + j] = rnd
    uniforms = torch.rand(n, 2, generator=g, dtype=torch.float32)
    out = AcceptInputs(target.to(device), None if dl is None else dl.to(device),
                       tokens.to(device), uniforms.to(device))
    return out


def tiny_workload(**kw) -> Workload:
    """A small custom workload for edge-case tests."""
    base = WORKLOADS["tiny"]
    return base.replace(name="custom", number=kw.pop("number", 90), **kw)
