"""Seeded synthetic inputs for the tests, the oracle checks and the benchmark.

This module holds none of the packing, attention or log-prob arithmetic. It only
draws token sequences shaped like the agentic workloads that the pages describe
(shared prompts, chains of tool-step branches, random sparse trees), random
tensors, and rounds float32 values to bfloat16 so that both sides of a parity
check start from the same representable inputs. Every generator is a pure
function of its seed (numpy PCG64 via ``default_rng``), so it gives the same
result on x86 and Arm hosts.

A generated tree never merges two siblings by accident: when a new branch is
attached to a node, its first token is redrawn until it differs from the first
token of every existing child of that node, so the trie built from the returned
sequences has exactly the generated shape.
"""
from __future__ import annotations

import dataclasses
import numpy as np

__all__ = [
    "bf16_round", "normal", "SynthTree", "tiny_tree", "agentic_short", "agentic_long",
    "galton_watson", "lm_head_tree", "random_sequences", "attention_config",
    "lm_head_config", "conv1d_config", "CONFIGS",
]


def bf16_round(x: np.ndarray, chunk: int = 1 << 24) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns float32.

    Works in place-sized chunks so that a multi-GB weight matrix needs no
    multi-GB temporary.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty_like(x)
    src = x.reshape(-1).view(np.uint32)
    dst = out.reshape(-1).view(np.uint32)
    for s in range(0, src.size, chunk):
        b = src[s:s + chunk].astype(np.uint64)
        b = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
        dst[s:s + chunk] = b.astype(np.uint32)
    return out


def normal(seed: int, shape, std: float = 1.0, bf16: bool = False) -> np.ndarray:
    """float32 N(0, std^2) samples from ``default_rng(seed)``, optionally bf16-rounded."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return bf16_round(x) if bf16 else x


@dataclasses.dataclass
class SynthTree:
    """A generated segment tree and the input sequences drawn from it."""
    seqs: list            # list of np.int32 token arrays, in insertion order
    n_tokens: int         # unique tokens in the generated tree
    seed: int
    note: str = ""


class _TreeBuilder:
    """Segment tree under construction: node = (parent, tokens, children)."""

    def __init__(self, rng: np.random.Generator, vocab: int):
        self.rng = rng
        self.vocab = vocab
        self.parent: list[int] = []
        self.tokens: list[np.ndarray] = []
        self.children: list[list[int]] = []
        self.root_children: list[int] = []

    def _segment(self, n: int, avoid_first) -> np.ndarray:
        seg = self.rng.integers(0, self.vocab, size=n, dtype=np.int64).astype(np.int32)
        while n > 0 and int(seg[0]) in avoid_first:
            seg[0] = self.rng.integers(0, self.vocab)
        return seg

    def add(self, parent: int, n: int) -> int:
        sibs = self.root_children if parent < 0 else self.children[parent]
        avoid = {int(self.tokens[c][0]) for c in sibs}
        seg = self._segment(n, avoid)
        node = len(self.tokens)
        self.parent.append(parent)
        self.tokens.append(seg)
        self.children.append([])
        sibs.append(node)
        return node

    def depth(self, node: int) -> int:
        d = 0
        while self.parent[node] >= 0:
            node = self.parent[node]
            d += 1
        return d

    def path_tokens(self, node: int) -> np.ndarray:
        chain = []
        while node >= 0:
            chain.append(self.tokens[node])
            node = self.parent[node]
        return np.concatenate(chain[::-1]).astype(np.int32)

    def leaves_dfs(self) -> list[int]:
        out, stack = [], list(reversed(self.root_children))
        while stack:
            n = stack.pop()
            if not self.children[n]:
                out.append(n)
            stack.extend(reversed(self.children[n]))
        return out

    def n_tokens(self) -> int:
        return int(sum(len(t) for t in self.tokens))


def tiny_tree(seed: int = 0, vocab: int = 512) -> SynthTree:
    """Three 44-token sequences: a 24-token prefix, then child A (20 tokens, a leaf)
    and child B (8 tokens) that splits into two 12-token leaves; 76 unique tokens."""
    b = _TreeBuilder(np.random.default_rng(seed), vocab)
    p = b.add(-1, 24)
    a = b.add(p, 20)
    c = b.add(p, 8)
    l1 = b.add(c, 12)
    l2 = b.add(c, 12)
    seqs = [b.path_tokens(a), b.path_tokens(l1), b.path_tokens(l2)]
    return SynthTree(seqs, b.n_tokens(), seed, "prefix 24 -> {A 20, B 8 -> {12, 12}}")


def agentic_short(seed: int = 0, vocab: int = 32000, prompt: int = 256, n_traj: int = 4,
                  n_steps: int = 4, branch: int = 128) -> SynthTree:
    """Shared prompt, then ``n_traj`` trajectories that each append one new branch per
    step; every (trajectory, step) context is one input sequence, trajectory-major."""
    b = _TreeBuilder(np.random.default_rng(seed), vocab)
    root = b.add(-1, prompt)
    seqs = []
    for _ in range(n_traj):
        node = root
        for _ in range(n_steps):
            node = b.add(node, branch)
            seqs.append(b.path_tokens(node))
    return SynthTree(seqs, b.n_tokens(), seed,
                     f"prompt {prompt}, {n_traj} traj x {n_steps} steps x {branch}")


def agentic_long(seed: int = 0, vocab: int = 32000, prompt: int = 1024, n_traj: int = 8,
                 n_steps: int = 8, branch: int = 256, p_share: float = 0.3) -> SynthTree:
    """Shared prompt, ``n_traj`` trajectories of ``n_steps`` steps. At each step, when
    the current node already has children, the trajectory follows one of them
    (uniform choice) with probability ``p_share``; otherwise it appends a new branch.
    Every (trajectory, step) context is one input sequence, trajectory-major."""
    rng = np.random.default_rng(seed)
    b = _TreeBuilder(rng, vocab)
    root = b.add(-1, prompt)
    seqs = []
    for _ in range(n_traj):
        node = root
        for _ in range(n_steps):
            kids = b.children[node]
            if kids and rng.random() < p_share:
                node = kids[int(rng.integers(len(kids)))]
            else:
                node = b.add(node, branch)
            seqs.append(b.path_tokens(node))
    return SynthTree(seqs, b.n_tokens(), seed,
                     f"prompt {prompt}, {n_traj} traj x {n_steps} steps x {branch}, share {p_share}")


def galton_watson(seed: int = 0, budget: int = 16384, vocab: int = 32000, max_depth: int = 7,
                  fanout=(1, 3), seg=(64, 512)) -> SynthTree:
    """Galton-Watson tree grown breadth-first: every node at depth < ``max_depth``
    (root depth 0, so at most ``max_depth + 1`` levels) gets U{fanout} children with
    U[seg] tokens each, until ``budget`` tokens exist (the last segment is clipped).
    The input sequences are the root-to-leaf paths, leaves in depth-first order."""
    rng = np.random.default_rng(seed)
    b = _TreeBuilder(rng, vocab)
    first = int(min(rng.integers(seg[0], seg[1] + 1), budget))
    root = b.add(-1, first)
    total = first
    queue = [root]
    head = 0
    while head < len(queue) and total < budget:
        n = queue[head]
        head += 1
        if b.depth(n) >= max_depth:
            continue
        f = int(rng.integers(fanout[0], fanout[1] + 1))
        for _ in range(f):
            ln = int(min(rng.integers(seg[0], seg[1] + 1), budget - total))
            c = b.add(n, ln)
            total += ln
            queue.append(c)
            if total >= budget:
                break
    seqs = [b.path_tokens(n) for n in b.leaves_dfs()]
    return SynthTree(seqs, b.n_tokens(), seed,
                     f"Galton-Watson depth<={max_depth + 1} levels, fanout U{fanout}, seg U{seg}, budget {budget}")


def lm_head_tree(rows: int = 8192, occ_range=(17500, 18500), first_seed: int = 0) -> SynthTree:
    """Galton-Watson tree of ``rows`` tokens whose sequences yield a number of
    next-token occurrences (sum over sequences of length - 1) inside ``occ_range``;
    the first seed from ``first_seed`` upward that lands there is used."""
    s = first_seed
    while True:
        t = galton_watson(seed=s, budget=rows)
        n_occ = sum(len(q) - 1 for q in t.seqs)
        if t.n_tokens == rows and occ_range[0] <= n_occ <= occ_range[1]:
            t.note += f"; seed searched from {first_seed}: {s}, {n_occ} occurrences"
            return t
        s += 1


def random_sequences(rng: np.random.Generator, n_seqs: int, max_len: int, vocab: int,
                     min_len: int = 0) -> list:
    """Short random sequences over a small vocabulary, so that prefixes collide often."""
    out = []
    for _ in range(n_seqs):
        ln = int(rng.integers(min_len, max_len + 1))
        out.append(rng.integers(0, vocab, size=ln).astype(np.int32))
    return out


# Workload table: the shapes of the five measured workloads.
CONFIGS = {
    "tiny_fp32": dict(kind="attn", tree=tiny_tree, Hq=1, Hkv=1, d=64, dtype="f32",
                      vocab=512, lm_hidden=64, lm_std=0.02),
    "agentic_short": dict(kind="attn", tree=agentic_short, Hq=32, Hkv=8, d=128, dtype="bf16"),
    "agentic_long": dict(kind="attn", tree=agentic_long, Hq=32, Hkv=8, d=128, dtype="bf16"),
    "galton_watson": dict(kind="attn", tree=galton_watson, Hq=32, Hkv=8, d=128, dtype="bf16"),
    "lm_head": dict(kind="lm", tree=lm_head_tree, K_h=4096, V=128256, dtype="bf16", w_std=0.02),
}


def attention_config(name: str, T: int, seed: int = 0):
    """Q, K, V (float32, bf16-rounded when the workload is bf16) and a dO for a
    packed tree of ``T`` rows under workload ``name``; seeds 1..4 of ``seed*16``."""
    c = CONFIGS[name]
    bf = c["dtype"] == "bf16"
    base = 16 * seed
    q = normal(base + 1, (T, c["Hq"], c["d"]), bf16=bf)
    k = normal(base + 2, (T, c["Hkv"], c["d"]), bf16=bf)
    v = normal(base + 3, (T, c["Hkv"], c["d"]), bf16=bf)
    do = normal(base + 4, (T, c["Hq"], c["d"]), bf16=bf)
    return q, k, v, do


def lm_head_config(T: int, K_h: int, V: int, n_occ: int, bf16: bool, seed: int = 0,
                   w_std: float = 0.02, random_targets: bool = True):
    """Hidden [T, K_h] ~ N(0,1), W [K_h, V] ~ N(0, w_std^2), per-occurrence targets
    uniform over V and weights uniform on (0, 1]."""
    base = 16 * seed
    h = normal(base + 5, (T, K_h), bf16=bf16)
    w = normal(base + 6, (K_h, V), std=w_std, bf16=bf16)
    rng = np.random.default_rng(base + 7)
    tg = rng.integers(0, V, size=n_occ).astype(np.int32) if random_targets else None
    wt = (1.0 - rng.random(n_occ)).astype(np.float32)     # (0, 1]
    return h, w, tg, wt


def conv1d_config(T: int, C: int, K: int, bf16: bool, seed: int = 0):
    """Inputs of the depthwise conv1d: x [T, C] ~ N(0,1), taps w [C, K] ~ N(0, 0.5^2),
    bias [C] ~ N(0, 0.1^2), output gradient dy [T, C] ~ N(0,1) (float32, bf16-rounded
    when ``bf16``)."""
    return (normal(seed * 4 + 1, (T, C), bf16=bf16), normal(seed * 4 + 2, (C, K), 0.5, bf16=bf16),
            normal(seed * 4 + 3, (C,), 0.1, bf16=bf16), normal(seed * 4 + 4, (T, C), bf16=bf16))
