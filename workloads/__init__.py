"""Seeded synthetic inputs for tree verification.

This module is the only code shared by the CUDA path's tests/bench and by the
CPU oracle.  It draws random inputs and lays them out; it computes nothing the
verification step computes (no ancestor sets, no attention, no argmax, no
acceptance).

Shapes follow the workloads the JETFLOW summary evaluates (Qwen3-8B and
Qwen3-30B-A3B attention shapes, draft budgets 16 and 256: "4. Resultados
Experimentales") and the DFlash-TfM summary's best-first / top-w tree
construction ("2. Construcción de Árboles").  Public benchmark prompts are not
used: random tensors of the same shapes stand in for them.

Layouts (all C-contiguous numpy arrays):
  q            uint16 (bf16 bits) [nb*B][Hq][D]      token-major, node-major within a sequence
  k_cache      uint16 (bf16 bits) [num_blocks][Hkv][page][D]
  v_cache      same as k_cache
  block_table  int32 [nb][max_pages]                 padded with -1
  prefix_lens  int32 [nb]
  parent       int32 [nb][B]                         parent[b][0] = -1, 0 <= parent[b][i] < i
  logits       uint16 (bf16 bits) [nb*B][V]
  draft        int32 [nb][B]                         draft[b][0] is not used
Tree node t of sequence b has its K/V at logical position prefix_lens[b] + t.
"""
from __future__ import annotations

import heapq
from dataclasses import dataclass, field

import numpy as np
import torch

PAGE = 16

__all__ = [
    "PAGE", "Workload", "f32_to_bf16", "bf16_to_f32", "tree_window", "tree_best_first",
    "make_workload", "config", "CONFIG_NAMES", "logical_kv", "GdnWorkload", "make_gdn_workload", "gdn_config",
]


def f32_to_bf16(x) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (torch's CPU conversion)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def bf16_to_f32(u) -> np.ndarray:
    """bf16 bit patterns -> fp32 (exact)."""
    u = np.ascontiguousarray(u, dtype=np.uint16)
    return (u.astype(np.uint32) << 16).view(np.float32)


def _normal_bf16(rng: np.random.Generator, shape, sigma: float = 0.5, chunk: int = 1 << 24) -> np.ndarray:
    """N(0,1)*sigma rounded to bf16, drawn in chunks to bound host memory."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = f32_to_bf16(rng.standard_normal(e - s, dtype=np.float32) * np.float32(sigma))
    return out.reshape(shape)


# ----------------------------------------------------------------------------- trees

def tree_window(rng: np.random.Generator, B: int, window: int = 4) -> np.ndarray:
    """parent[i] uniform over the previous `window` nodes: U[max(0, i-window), i-1]."""
    p = np.empty(B, dtype=np.int32)
    p[0] = -1
    for i in range(1, B):
        p[i] = rng.integers(max(0, i - window), i)
    return p


def tree_best_first(rng: np.random.Generator, B: int, n_cand: int = 8, alpha: float = 0.3,
                    child_cap=4, max_depth: int = 16) -> np.ndarray:
    """Best-first draft-tree expansion with cumulative log-prob branch scores.

    Follows the JETFLOW summary, §2 "Estrategia de Entrenamiento" (tree
    construction: branch score = cumulative draft log-probability, best-first
    expansion up to a budget).  Draft probabilities are synthetic: each popped
    node draws Dirichlet(alpha) over `n_cand` candidates and pushes its top
    `child_cap` of them (an int, or a callable rng -> int) while its depth is
    below `max_depth`.  Node index = pop order, so the result is topological.
    Ties in the heap are broken by push order.
    """
    for attempt in range(64):
        parent = [-1]
        depth = [0]
        heap: list = []
        counter = 0

        def expand(node: int, score: float):
            nonlocal counter
            if depth[node] >= max_depth:
                return
            probs = rng.dirichlet(np.full(n_cand, alpha))
            cap = child_cap(rng) if callable(child_cap) else int(child_cap)
            top = np.argsort(-probs, kind="stable")[:cap]
            for c in top:
                s = score + float(np.log(max(float(probs[c]), 1e-300)))
                heapq.heappush(heap, (-s, counter, node))
                counter += 1

        expand(0, 0.0)
        while len(parent) < B and heap:
            negs, _, par = heapq.heappop(heap)
            node = len(parent)
            parent.append(par)
            depth.append(depth[par] + 1)
            expand(node, -negs)
        if len(parent) == B:
            return np.asarray(parent, dtype=np.int32)
    raise RuntimeError("best-first generator could not reach the budget")


# ----------------------------------------------------------------------------- workloads

@dataclass
class Workload:
    name: str
    nb: int
    B: int
    Hq: int
    Hkv: int
    D: int
    V: int
    prefix_lens: np.ndarray
    parent: np.ndarray
    block_table: np.ndarray
    num_blocks: int
    q: np.ndarray
    k_cache: np.ndarray
    v_cache: np.ndarray
    logits: np.ndarray
    draft: np.ndarray
    planted: np.ndarray          # per node: the token planted as the row's likely maximum
    meta: dict = field(default_factory=dict)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def max_pages(self) -> int:
        return self.block_table.shape[1]


def make_workload(name: str, nb: int, B: int, Hq: int, Hkv: int, D: int, V: int,
                  prefix_lens, trees, seed: int, shuffle_pages: bool = True,
                  sigma: float = 0.5, accept_p: float = 0.7, plant: float = 8.0,
                  extra_pages: int = 0, with_logits: bool = True) -> Workload:
    """Lay out one seeded verify-step input.

    trees: list of nb parent arrays (or a callable rng -> parent array).
    Logits are N(0,1) per entry with +`plant` added at one uniformly drawn
    token per node, so each row has a known likely maximum; the draft token of
    node i>=1 is the parent's planted token with probability `accept_p`, else
    uniform in [0, V).  Every cache slot (used or not) holds finite values.
    """
    ss = np.random.SeedSequence(seed)
    r_tree, r_pages, r_q, r_k, r_v, r_log, r_draft = [np.random.default_rng(s) for s in ss.spawn(7)]
    prefix_lens = np.asarray(prefix_lens, dtype=np.int32).reshape(nb)
    if callable(trees):
        parents = [np.asarray(trees(r_tree), dtype=np.int32) for _ in range(nb)]
    else:
        parents = [np.asarray(t, dtype=np.int32) for t in trees]
    parent = np.stack(parents).astype(np.int32).reshape(nb, B)

    pages_per_seq = [(int(p) + B + PAGE - 1) // PAGE for p in prefix_lens]
    num_blocks = int(sum(pages_per_seq)) + extra_pages
    max_pages = max(pages_per_seq)
    phys = np.arange(num_blocks, dtype=np.int32)
    if shuffle_pages:
        phys = r_pages.permutation(phys).astype(np.int32)
    block_table = np.full((nb, max_pages), -1, dtype=np.int32)
    o = 0
    for b in range(nb):
        n = pages_per_seq[b]
        block_table[b, :n] = phys[o:o + n]
        o += n

    q = _normal_bf16(r_q, (nb * B, Hq, D), sigma)
    k_cache = _normal_bf16(r_k, (num_blocks, Hkv, PAGE, D), sigma)
    v_cache = _normal_bf16(r_v, (num_blocks, Hkv, PAGE, D), sigma)

    planted = r_log.integers(0, V, size=(nb, B)).astype(np.int32)
    if with_logits:
        logits = np.empty((nb * B, V), dtype=np.uint16)
        for row in range(nb * B):
            x = r_log.standard_normal(V, dtype=np.float32)
            x[planted.reshape(-1)[row]] += np.float32(plant)
            logits[row] = f32_to_bf16(x)
    else:
        logits = np.zeros((0, V), dtype=np.uint16)

    draft = np.zeros((nb, B), dtype=np.int32)
    for b in range(nb):
        for i in range(1, B):
            if r_draft.random() < accept_p:
                draft[b, i] = planted[b, parent[b, i]]
            else:
                draft[b, i] = r_draft.integers(0, V)
    return Workload(name=name, nb=nb, B=B, Hq=Hq, Hkv=Hkv, D=D, V=V, prefix_lens=prefix_lens,
                    parent=parent, block_table=block_table, num_blocks=num_blocks, q=q,
                    k_cache=k_cache, v_cache=v_cache, logits=logits, draft=draft, planted=planted,
                    meta={"seed": seed, "shuffle_pages": shuffle_pages})


CONFIG_NAMES = {
    1: "qwen3-8b-attn nb=1 B=16 P=512 identity-pages V=4096",
    2: "qwen3-8b-attn nb=1 B=256 best-first P=4096 shuffled-pages V=151936",
    3: "qwen3-8b-attn nb=8 B=64 best-first P~U[2048,16384] shuffled-pages V=151936",
    4: "qwen3-30b-a3b-attn nb=32 B=16 P=8192 shuffled-pages V=151936",
    5: "qwen3-8b-attn nb=4 B=256 best-first P=32768 shuffled-pages V=151936",
}


def config(n: int, seed: int = 0, with_logits: bool = True) -> Workload:
    """The five verify-step workloads (Qwen3-8B: 32 q / 8 kv heads; Qwen3-30B-A3B: 32 / 4; head dim 128)."""
    name = CONFIG_NAMES[n]
    if n == 1:
        return make_workload(name, 1, 16, 32, 8, 128, 4096, [512], lambda r: tree_window(r, 16, 4),
                             seed, shuffle_pages=False, with_logits=with_logits)
    if n == 2:
        return make_workload(name, 1, 256, 32, 8, 128, 151936, [4096],
                             lambda r: tree_best_first(r, 256, child_cap=4, max_depth=16),
                             seed, with_logits=with_logits)
    if n == 3:
        pr = np.random.default_rng(np.random.SeedSequence([seed, 3]))
        pl = pr.integers(2048, 16384 + 1, size=8)
        return make_workload(name, 8, 64, 32, 8, 128, 151936, pl,
                             lambda r: tree_best_first(r, 64, child_cap=lambda rr: int(rr.integers(1, 4)),
                                                       max_depth=12),
                             seed, with_logits=with_logits)
    if n == 4:
        return make_workload(name, 32, 16, 32, 4, 128, 151936, [8192] * 32,
                             lambda r: tree_window(r, 16, 4), seed, with_logits=with_logits)
    if n == 5:
        return make_workload(name, 4, 256, 32, 8, 128, 151936, [32768] * 4,
                             lambda r: tree_best_first(r, 256, child_cap=4, max_depth=24),
                             seed, with_logits=with_logits)
    raise ValueError(n)


def logical_kv(w: Workload, b: int, which: str = "k") -> np.ndarray:
    """Gather sequence b's cache rows in logical order: [P_b + B][Hkv][D] bf16 bits.

    Plain fancy indexing through the block table; used by tests to build
    contiguous tensors for library pins.
    """
    cache = w.k_cache if which == "k" else w.v_cache
    n = int(w.prefix_lens[b]) + w.B
    pos = np.arange(n)
    pages = w.block_table[b, pos // PAGE]
    return cache[pages, :, pos % PAGE, :]


# --------------------------------------------------------------------- Gated DeltaNet

@dataclass
class GdnWorkload:
    """Inputs of one Gated DeltaNet tree-verification step (one layer).

    q, k, v  uint16 (bf16 bits) [nb*B][H][D]   q and k L2-normalised per head before rounding
    alpha    float32 [nb*B][H]                 gate in [0.85, 1)
    beta     float32 [nb*B][H]                 write strength in [0.1, 0.9)
    S0       float32 [nb][H][D][D]             committed state (rows: key dim, columns: value dim)
    parent   int32 [nb][B]                     topologically ordered tree, parent[b][0] = -1
    """
    name: str
    nb: int
    B: int
    H: int
    D: int
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    alpha: np.ndarray
    beta: np.ndarray
    S0: np.ndarray
    parent: np.ndarray


def _unit_bf16(rng, shape):
    x = rng.standard_normal(shape, dtype=np.float32)
    x /= np.linalg.norm(x, axis=-1, keepdims=True)
    return f32_to_bf16(x)


def make_gdn_workload(name: str, nb: int, B: int, H: int, D: int, trees, seed: int,
                      s0_sigma: float = 0.1) -> GdnWorkload:
    """Seeded GDN inputs: normalised q/k, N(0,1)*0.5 v, gates, write strengths, a random state."""
    ss = np.random.SeedSequence(seed)
    r_tree, r_q, r_k, r_v, r_a, r_s = [np.random.default_rng(x) for x in ss.spawn(6)]
    if callable(trees):
        parents = [np.asarray(trees(r_tree), dtype=np.int32) for _ in range(nb)]
    else:
        parents = [np.asarray(t, dtype=np.int32) for t in trees]
    parent = np.stack(parents).astype(np.int32).reshape(nb, B)
    q = _unit_bf16(r_q, (nb * B, H, D))
    k = _unit_bf16(r_k, (nb * B, H, D))
    v = _normal_bf16(r_v, (nb * B, H, D), 0.5)
    alpha = r_a.uniform(0.85, 1.0, size=(nb * B, H)).astype(np.float32)
    beta = r_a.uniform(0.1, 0.9, size=(nb * B, H)).astype(np.float32)
    S0 = (r_s.standard_normal((nb, H, D, D), dtype=np.float32) * np.float32(s0_sigma)).astype(np.float32)
    return GdnWorkload(name=name, nb=nb, B=B, H=H, D=D, q=q, k=k, v=v, alpha=alpha, beta=beta, S0=S0, parent=parent)


def gdn_config(seed: int = 0) -> GdnWorkload:
    """The GDN workload: one sequence, a 128-node best-first tree (the DFlash-TfM summary's
    tree size for its fused-kernel figure), 32 heads of dimension 128 (the head shape of the
    Qwen3.6-27B GDN layers the summary evaluates is not printed; 32 x 128 is this recipe's)."""
    return make_gdn_workload("gdn nb=1 B=128 H=32 D=128 best-first", 1, 128, 32, 128,
                             lambda r: tree_best_first(r, 128, child_cap=4, max_depth=16), seed)
