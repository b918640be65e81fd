"""Seeded synthetic workloads for the tree-verify step.

This module only draws inputs: draft trees, target/draft logits and draft
tokens.  It holds none of the verify arithmetic (no filtering, no acceptance
test, no residual), so both the CUDA path and the CPU oracle can consume what
it produces without sharing any of the method's code.

Draft tokens stand in for a draft model: at T > 0 every child of node u is an
independent draw from softmax(q_u / T) (siblings i.i.d., with replacement); at
T == 0 the children of u are the top-k_u tokens of q_u.  The pages' benchmark
suites and trained models are not available; the shapes below (vocabulary
sizes of LLaMA-2 / LLaMA-3 class models, 10- to 60-node trees) follow the
workloads the pages describe.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    N: int
    V: int
    dtype: str            # "f32" or "bf16"
    tree: str             # "chain", "eagle10", "random"
    depth: int
    temperature: float
    top_k: int
    top_p: float
    logits: str           # "gauss" or "zipf"
    sigma: float = 3.0    # std of the target logits ("gauss")
    draft_noise: float = 1.0
    max_branch: int = 4
    extra: dict = field(default_factory=dict)

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


# The five workloads.  B, N, V, dtype, tree shape and sampling parameters are fixed
# by the workload definitions; reduced variants for fast tests come from .with_().
WORKLOADS = {
    # chain draft gamma=3 (4 rows incl. root), V=32, 10,000 rounds as 10,000 batch rows
    "chain_g3_v32": Workload("chain_g3_v32", B=10000, N=4, V=32, dtype="f32", tree="chain",
                             depth=3, temperature=1.0, top_k=0, top_p=1.0, logits="gauss",
                             sigma=3.0, draft_noise=1.0),
    # EAGLE-1 style 10-draft static tree, depth 3, V=32000
    "eagle10_v32000": Workload("eagle10_v32000", B=1, N=11, V=32000, dtype="f32",
                               tree="eagle10", depth=3, temperature=1.0, top_k=0, top_p=1.0,
                               logits="gauss", sigma=3.0, draft_noise=1.0),
    # 60-node depth-6 random trees, B=64, V=128256 bf16, T=0.7, top-p 0.9
    "tree60_b64_v128256": Workload("tree60_b64_v128256", B=64, N=60, V=128256, dtype="bf16",
                                   tree="random", depth=6, temperature=0.7, top_k=0, top_p=0.9,
                                   logits="gauss", sigma=3.0, draft_noise=1.5),
    # 26-node depth-5 random trees, B=256, V=152064 bf16, Zipf-shaped bias, T=1, top-k 50, top-p .95
    "tree26_b256_v152064": Workload("tree26_b256_v152064", B=256, N=26, V=152064, dtype="bf16",
                                    tree="random", depth=5, temperature=1.0, top_k=50,
                                    top_p=0.95, logits="zipf", sigma=2.0),
    # fused LM head: B=32 x 60 nodes of d=4096 features, V=128256, T=0.8, top-p 0.9
    "lmhead_tree60_b32_v128256": Workload("lmhead_tree60_b32_v128256", B=32, N=60, V=128256,
                                          dtype="bf16", tree="random", depth=6,
                                          temperature=0.8, top_k=0, top_p=0.9, logits="lmhead",
                                          extra={"d": 4096, "w_std": 0.02}),
}

# EAGLE-1's static tree (root branching 4, then 3/2/1, three draft levels, 10 draft
# tokens), read as: node 1 has 3 children, node 2 has 1, node 5 has 2.
EAGLE10_PARENTS = [-1, 0, 0, 0, 0, 1, 1, 1, 2, 5, 5]


def chain_tree(n: int) -> np.ndarray:
    return np.array([-1] + list(range(n - 1)), dtype=np.int32)


def random_tree(n: int, depth: int, max_branch: int, rng: np.random.Generator) -> np.ndarray:
    """A tree with exactly n nodes, depth exactly `depth` and at most `max_branch`
    children per node: a root-to-depth spine, then children attached to uniformly
    chosen nodes that are shallower than `depth` and not yet full; finally the
    nodes are relabelled in breadth-first order (siblings keep creation order)."""
    if n < depth + 1:
        raise ValueError("need at least depth+1 nodes")
    parent = [-1] + list(range(depth))
    node_depth = list(range(depth + 1))
    nchild = [1] * depth + [0]
    while len(parent) < n:
        open_nodes = [i for i in range(len(parent)) if node_depth[i] < depth and nchild[i] < max_branch]
        u = open_nodes[int(rng.integers(len(open_nodes)))]
        parent.append(u)
        node_depth.append(node_depth[u] + 1)
        nchild.append(0)
        nchild[u] += 1
    children = [[] for _ in range(n)]
    for c in range(1, n):
        children[parent[c]].append(c)
    order = [0]
    for u in order:
        order.extend(children[u])
    new_id = {old: i for i, old in enumerate(order)}
    out = np.empty(n, dtype=np.int32)
    for old in order:
        out[new_id[old]] = -1 if parent[old] < 0 else new_id[parent[old]]
    return out


def make_parents(w: Workload, seed: int) -> np.ndarray:
    """[B, N] int32 parent indices for workload w (node 0 = root, parent < node)."""
    if w.tree == "chain":
        return np.tile(chain_tree(w.N), (w.B, 1))
    if w.tree == "eagle10":
        if w.N != len(EAGLE10_PARENTS):
            raise ValueError("eagle10 tree has 11 rows")
        return np.tile(np.array(EAGLE10_PARENTS, dtype=np.int32), (w.B, 1))
    rng = np.random.default_rng(seed)
    return np.stack([random_tree(w.N, w.depth, w.max_branch, rng) for _ in range(w.B)])


def tree_depth(parents: np.ndarray) -> int:
    parents = np.atleast_2d(parents)
    dmax = 0
    for row in parents:
        d = np.zeros(len(row), dtype=np.int64)
        for n in range(1, len(row)):
            d[n] = d[row[n]] + 1
        dmax = max(dmax, int(d.max()))
    return dmax


def _torch_dtype(w: Workload):
    return torch.float32 if w.dtype == "f32" else torch.bfloat16


def padded_pitch(V: int, elem_bytes: int) -> int:
    """Row pitch (elements) of a 16-byte aligned row of V elements."""
    per = 16 // elem_bytes
    return (V + per - 1) // per * per


def empty_rows(shape, dtype, device):
    """An uninitialised [..., V] tensor whose rows start on 16-byte boundaries (a view
    into a buffer padded to an aligned row pitch)."""
    V = shape[-1]
    Vp = padded_pitch(V, torch.tensor([], dtype=dtype).element_size())
    buf = torch.empty(tuple(shape[:-1]) + (Vp,), dtype=dtype, device=device)
    return buf[..., :V]


def make_logits(w: Workload, seed: int, device="cpu", chunk_rows: int = 512):
    """Target and draft logits, each [B, N, V] in the workload's dtype (rows on
    16-byte boundaries: a padded row pitch when V * elem_bytes is not a multiple of 16).

    gauss: target z ~ N(0, sigma^2) i.i.d.; draft = z + N(0, draft_noise^2).
    zipf:  bias(v) = -1.1 ln(rank(v)), rank from a per-row affine permutation
           v -> (a v + c) mod V with gcd(a, V) = 1; target = bias + e,
           draft = bias + 0.8 e + 0.6 e', with e, e' ~ N(0, sigma^2).
    """
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    B, N, V = w.B, w.N, w.V
    dt = _torch_dtype(w)
    p = empty_rows((B, N, V), dt, device)
    q = empty_rows((B, N, V), dt, device)
    pf = p.as_strided((B * N, V), (p.stride(1), 1))   # row view over all B*N rows
    qf = q.as_strided((B * N, V), (q.stride(1), 1))
    rows = B * N
    if w.logits == "zipf":
        rng = np.random.default_rng(seed + 7919)
        coprimes = np.array([a for a in range(1, min(V, 100003)) if math.gcd(a, V) == 1][:4096])
        a_row = torch.as_tensor(coprimes[rng.integers(len(coprimes), size=rows)], device=device)
        c_row = torch.as_tensor(rng.integers(V, size=rows), device=device)
    v = torch.arange(V, device=device, dtype=torch.int64)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        shape = (r1 - r0, V)
        if w.logits == "gauss":
            z = torch.randn(shape, generator=g, device=device) * w.sigma
            d = z + torch.randn(shape, generator=g, device=device) * w.draft_noise
        elif w.logits == "zipf":
            rank = (a_row[r0:r1, None] * v[None, :] + c_row[r0:r1, None]) % V + 1
            bias = -1.1 * torch.log(rank.to(torch.float32))
            e = torch.randn(shape, generator=g, device=device) * w.sigma
            e2 = torch.randn(shape, generator=g, device=device) * w.sigma
            z = bias + e
            d = bias + 0.8 * e + 0.6 * e2
        else:
            raise ValueError(f"logits kind {w.logits!r} is produced by make_lmhead_inputs")
        pf[r0:r1] = z.to(dt)
        qf[r0:r1] = d.to(dt)
    return p, q


def make_lmhead_inputs(w: Workload, seed: int, device="cpu"):
    """Features F [B*N, d] ~ N(0,1) and LM-head weight W [V, d] ~ N(0, w_std^2), bf16."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    d = w.extra["d"]
    feats = torch.randn((w.B * w.N, d), generator=g, device=device).to(torch.bfloat16)
    weight = (torch.randn((w.V, d), generator=g, device=device) * w.extra["w_std"]).to(torch.bfloat16)
    return feats, weight


def build_lmhead_inputs(w: Workload, seed: int, device="cpu"):
    """Inputs of the fused LM-head workload: features F [B*N, d], weight W [V, d], the
    draft logits q [B, N, V] (bf16 of the fp32 product F W^T plus N(0, 1) noise, made
    once here with torch.matmul), the tree and the draft tokens drawn from q."""
    feats, weight = make_lmhead_inputs(w, seed, device=device)
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) + 7919)
    rows = w.B * w.N
    Vp = padded_pitch(w.V, 2)
    buf = torch.empty((rows, Vp), dtype=torch.bfloat16, device=device)
    for r0 in range(0, rows, 256):
        r1 = min(rows, r0 + 256)
        ref = torch.matmul(feats[r0:r1].float(), weight.float().t())
        buf[r0:r1, :w.V] = (ref + torch.randn(ref.shape, generator=g, device=device)).to(
            torch.bfloat16)
    q = buf.view(w.B, w.N, Vp)[..., :w.V]
    parents = make_parents(w, seed)
    tokens = make_draft_tokens(w, q, parents, seed)
    return {"features": feats, "weight": weight, "q": q, "parents": parents, "tokens": tokens,
            "max_depth": tree_depth(parents), "workload": w}


def make_draft_tokens(w: Workload, q: torch.Tensor, parents: np.ndarray, seed: int) -> np.ndarray:
    """[B, N] int32 draft tokens; entry 0 (root) is 0 and is never read.

    T > 0: each child of u is an independent draw from softmax(q_u / T).
    T == 0: the children of u, in node order, are the top-k_u tokens of q_u.
    """
    B, N, V = q.shape
    parents = np.asarray(parents)
    nchild = np.zeros((B, N), dtype=np.int64)
    for b in range(B):
        for c in range(1, N):
            nchild[b, parents[b, c]] += 1
    kmax = int(nchild.max()) if N > 1 else 0
    tokens = np.zeros((B, N), dtype=np.int32)
    if kmax == 0:
        return tokens
    g = torch.Generator(device=q.device)
    g.manual_seed(int(seed) + 104729)
    draws = torch.empty((B, N, kmax), dtype=torch.int64, device=q.device)
    for b0 in range(0, B, 64):
        b1 = min(B, b0 + 64)
        rows = q[b0:b1].reshape(-1, V).float()
        if w.temperature > 0:
            probs = torch.softmax(rows / w.temperature, dim=-1)
            s = torch.multinomial(probs, kmax, replacement=True, generator=g)
        else:
            s = torch.topk(rows, kmax, dim=-1).indices
        draws[b0:b1] = s.view(b1 - b0, N, kmax)
    draws = draws.cpu().numpy()
    for b in range(B):
        slot = np.zeros(N, dtype=np.int64)
        for c in range(1, N):
            u = parents[b, c]
            tokens[b, c] = draws[b, u, slot[u]]
            slot[u] += 1
    return tokens


def build_inputs(w: Workload, seed: int, device="cpu"):
    """Everything one verify call needs, as a dict (logits on `device`, tree arrays on host)."""
    parents = make_parents(w, seed)
    p, q = make_logits(w, seed, device=device)
    tokens = make_draft_tokens(w, q, parents, seed)
    return {
        "p": p, "q": q, "parents": parents, "tokens": tokens,
        "max_depth": tree_depth(parents), "workload": w,
    }


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw uint16 bits of a bf16 tensor (for the oracle's exact bf16 input path)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def host_logits(t: torch.Tensor) -> np.ndarray:
    """Host copy in the oracle's input format: float32 as is, bf16 as raw bits."""
    if t.dtype == torch.bfloat16:
        return bf16_bits(t)
    return t.detach().cpu().contiguous().numpy()


# ---------------------------------------------------------------------------------------
# Draft candidates of an EAGLE-2 dynamic tree (EAGLE / EAGLE-2 paper translation,
# sections 2.3.1-2.3.2).  The sizes follow the method's usual setting: every expanded
# node gets `children` candidates, `expand_k` nodes of a layer are expanded, `layers`
# layers in all (10 / 10 / 6 gives 510 candidates; keeping m = 59 of them makes a
# 60-node draft).  Which nodes are expanded is drawn at random here, not ranked by value:
# the tree build reads whatever candidate list it is given.
# ---------------------------------------------------------------------------------------
@dataclass
class DraftCandidates:
    parent: np.ndarray   # [B, n] int32, -1 = child of the root, else an earlier candidate
    token: np.ndarray    # [B, n] int32
    prob: np.ndarray     # [B, n] float32 confidences in [0, 1]
    root: np.ndarray     # [B] int32


def make_draft_candidates(B: int, layers: int = 6, expand_k: int = 10, children: int = 10,
                          seed: int = 0, vocab: int = 128256, levels: int = 0) -> DraftCandidates:
    """Seeded candidate lists in creation order.  The confidences of one parent's children
    are a random split of at most 1 listed in descending order (the draft model's top
    children); levels > 0 rounds every confidence down to a multiple of 1/levels, which
    makes many values tie."""
    rng = np.random.default_rng(seed)
    n = children + (layers - 1) * expand_k * children
    par = np.empty((B, n), dtype=np.int32)
    prob = np.empty((B, n), dtype=np.float32)
    for b in range(B):
        groups = [-1]
        start = 0
        for layer in range(layers):
            pos = start
            for g in groups:
                w = rng.exponential(1.0, size=children + 1)
                share = np.sort(w[:children] / w.sum())[::-1]
                par[b, pos:pos + children] = g
                prob[b, pos:pos + children] = share.astype(np.float32)
                pos += children
            layer_nodes = np.arange(start, pos)
            start = pos
            if layer + 1 < layers:
                groups = sorted(rng.choice(layer_nodes, size=min(expand_k, len(layer_nodes)),
                                           replace=False).tolist())
    if levels > 0:
        prob = (np.floor(prob * levels) / levels).astype(np.float32)
    token = rng.integers(0, vocab, size=(B, n)).astype(np.int32)
    root = rng.integers(0, vocab, size=B).astype(np.int32)
    return DraftCandidates(par, token, prob, root)
