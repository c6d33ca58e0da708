"""Pins for the CPU oracle: each test ties it to something other than itself.

Sources of truth used here:
  * a hand-worked example (tests/golden/tree_example.json) derived from the
    tree-causal mask of the JETFLOW summary (§2 "Arquitectura Central");
  * library routines: networkx ancestry, torch scaled_dot_product_attention
    (fp64, CPU), scipy logsumexp, numpy argmax;
  * closed forms and special cases (zero query, chain tree = causal
    attention, single node = decode attention, star tree);
  * invariances the mask semantics imply (sibling relabelling, physical page
    placement) and brute-force path enumeration on every small tree.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tree_example.json")


def _bits(mask_row):
    return {w * 32 + b for w, word in enumerate(mask_row) for b in range(32) if (int(word) >> b) & 1}


def _random_trees(rng, B, n):
    out = []
    for k in range(n):
        if k % 3 == 0:
            out.append(wl.tree_window(rng, B, window=int(rng.integers(1, 6))))
        elif k % 3 == 1:
            out.append(wl.tree_best_first(rng, B, child_cap=int(rng.integers(1, 5)), max_depth=B))
        else:
            p = np.array([-1] + [int(rng.integers(0, i)) for i in range(1, B)], dtype=np.int32)
            out.append(p)
    return out


def _small_workload(seed, nb, B, Hq, Hkv, D, prefix, shuffle=True, trees=None):
    rng = np.random.default_rng(seed)
    if trees is None:
        trees = _random_trees(rng, B, nb)
    return wl.make_workload("pin", nb, B, Hq, Hkv, D, 64, prefix, trees, seed,
                            shuffle_pages=shuffle, extra_pages=3, with_logits=False)


def _f64(u16):
    return wl.bf16_to_f32(u16).astype(np.float64)


# ------------------------------------------------------------------------ mask

def test_mask_golden_example():
    fx = json.load(open(GOLDEN))["tree"]
    mask, depth = oracle.build_mask(np.array([fx["parent"]], dtype=np.int32))
    assert mask[0, :, 0].tolist() == fx["mask_words"]
    assert depth[0].tolist() == fx["depth"]


@pytest.mark.parametrize("B", [1, 2, 31, 32, 33, 64, 100, 255, 256])
def test_mask_matches_networkx_ancestry(B):
    nx = pytest.importorskip("networkx")
    rng = np.random.default_rng(B)
    trees = _random_trees(rng, B, 3)
    mask, depth = oracle.build_mask(np.stack(trees))
    for t, p in enumerate(trees):
        g = nx.DiGraph()
        g.add_nodes_from(range(B))
        g.add_edges_from((int(p[i]), i) for i in range(1, B))
        lengths = nx.single_source_shortest_path_length(g, 0)
        for i in range(B):
            assert _bits(mask[t, i]) == nx.ancestors(g, i) | {i}
            assert depth[t, i] == lengths[i]


def test_mask_invariants():
    rng = np.random.default_rng(7)
    trees = _random_trees(rng, 200, 6)
    mask, depth = oracle.build_mask(np.stack(trees))
    for t in range(len(trees)):
        sets = [_bits(mask[t, i]) for i in range(200)]
        for i, s in enumerate(sets):
            assert len(s) == depth[t, i] + 1
            assert 0 in s and i in s and max(s) == i
            for j in s:
                assert sets[j] <= s
        # unused high bits of the last word stay clear
        assert all(max(_bits(mask[t, i])) < 200 for i in range(200))


@pytest.mark.parametrize("bad", [[0, 0, 1], [-1, 1, 0], [-1, 0, -1], [-1, 0, 5], [-1, 0, 2]])
def test_mask_rejects_non_topological(bad):
    with pytest.raises(oracle.OracleError):
        oracle.build_mask(np.array([bad], dtype=np.int32))


# ------------------------------------------------------------------- attention

def test_attention_golden_example():
    fx = json.load(open(GOLDEN))["attention"]
    q = wl.f32_to_bf16(np.array(fx["q"], dtype=np.float32)).reshape(3, 1, 2)
    kc = np.zeros((1, 1, 16, 2), dtype=np.uint16)
    vc = np.zeros((1, 1, 16, 2), dtype=np.uint16)
    kc[0, 0, :4] = wl.f32_to_bf16(np.array(fx["k_logical"], dtype=np.float32))
    vc[0, 0, :4] = wl.f32_to_bf16(np.array(fx["v_logical"], dtype=np.float32))
    O, L = oracle.attn(q, kc, vc, np.array([[0]], np.int32), np.array([fx["prefix_len"]], np.int32),
                       np.array([fx["parent"]], np.int32), 1, 1, scale=fx["scale"])
    np.testing.assert_allclose(O[:, 0, :], np.array(fx["O"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(L[:, 0], np.array(fx["LSE"]), rtol=0, atol=1e-12)


def _sdpa_last_row(qv, K, Vv, scale):
    """Library pin: torch SDPA (fp64, CPU), one query attending to all given keys."""
    qt = torch.from_numpy(qv)[None, None, None, :]
    kt = torch.from_numpy(K)[None, None]
    vt = torch.from_numpy(Vv)[None, None]
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)[0, 0, 0].numpy()


@pytest.mark.parametrize("G,D,P", [(1, 8, 0), (2, 16, 17), (4, 16, 40), (4, 8, 33)])
def test_attention_each_node_equals_attention_over_its_root_path(G, D, P):
    """Per-branch factorisation: row i = last row of causal attention over prefix ++ path(i)."""
    nx = pytest.importorskip("networkx")
    from scipy.special import logsumexp
    Hkv = 2
    Hq = Hkv * G
    w = _small_workload(100 + G + D + P, nb=2, B=8, Hq=Hq, Hkv=Hkv, D=D, prefix=[P, P + 5])
    O, L = oracle.attn_workload(w)
    scale = 1.0 / math.sqrt(D)
    for b in range(w.nb):
        Kl = _f64(wl.logical_kv(w, b, "k"))
        Vl = _f64(wl.logical_kv(w, b, "v"))
        Pb = int(w.prefix_lens[b])
        g = nx.DiGraph()
        g.add_edges_from((int(w.parent[b, i]), i) for i in range(1, w.B))
        g.add_node(0)
        for i in range(w.B):
            path = nx.shortest_path(g, 0, i)
            keys = list(range(Pb)) + [Pb + t for t in path]
            for h in range(Hq):
                kvh = h // G
                qv = _f64(w.q[b * w.B + i, h])
                ref = _sdpa_last_row(qv, Kl[keys, kvh], Vl[keys, kvh], scale)
                np.testing.assert_allclose(O[b * w.B + i, h], ref, rtol=0, atol=1e-12)
                lse = logsumexp(scale * (Kl[keys, kvh] @ qv))
                assert abs(L[b * w.B + i, h] - lse) < 1e-12


def test_attention_chain_tree_equals_causal_attention():
    """A chain-shaped tree is ordinary causal attention over prefix ++ chain."""
    B, P, Hq, Hkv, D = 12, 37, 4, 2, 16
    chain = np.arange(-1, B - 1, dtype=np.int32)
    w = _small_workload(5, nb=1, B=B, Hq=Hq, Hkv=Hkv, D=D, prefix=[P], trees=[chain])
    O, _ = oracle.attn_workload(w)
    K = torch.from_numpy(_f64(wl.logical_kv(w, 0, "k"))).permute(1, 0, 2)   # [Hkv][P+B][D]
    Vv = torch.from_numpy(_f64(wl.logical_kv(w, 0, "v"))).permute(1, 0, 2)
    K = K.repeat_interleave(Hq // Hkv, dim=0)
    Vv = Vv.repeat_interleave(Hq // Hkv, dim=0)
    q = torch.from_numpy(_f64(w.q)).permute(1, 0, 2)                      # [Hq][B][D]
    allowed = torch.ones(B, P + B, dtype=torch.bool).tril(diagonal=P)     # row i sees keys <= P+i
    ref = torch.nn.functional.scaled_dot_product_attention(q, K, Vv, attn_mask=allowed)
    np.testing.assert_allclose(O, ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def test_attention_single_node_is_decode_attention():
    w = _small_workload(9, nb=3, B=1, Hq=8, Hkv=2, D=16, prefix=[0, 5, 48])
    O, _ = oracle.attn_workload(w)
    for b in range(3):
        K = _f64(wl.logical_kv(w, b, "k"))
        Vv = _f64(wl.logical_kv(w, b, "v"))
        for h in range(8):
            ref = _sdpa_last_row(_f64(w.q[b, h]), K[:, h // 4], Vv[:, h // 4], 0.25)
            np.testing.assert_allclose(O[b, h], ref, rtol=0, atol=1e-12)


def test_attention_zero_query_closed_form():
    """q = 0 makes every visible score 0: O = mean of the visible V rows, LSE = ln(#visible)."""
    rng = np.random.default_rng(3)
    B, P = 9, 21
    trees = _random_trees(rng, B, 2)
    w = _small_workload(11, nb=2, B=B, Hq=2, Hkv=1, D=8, prefix=[P, 0], trees=trees)
    w.q[:] = 0
    O, L = oracle.attn_workload(w)
    for b in range(2):
        Pb = int(w.prefix_lens[b])
        Vl = _f64(wl.logical_kv(w, b, "v"))
        for i in range(B):
            path = [i]
            while path[-1] != 0:
                path.append(int(w.parent[b, path[-1]]))
            rows = list(range(Pb)) + [Pb + t for t in path]
            np.testing.assert_allclose(O[b * B + i, :, :], np.broadcast_to(Vl[rows, 0].mean(0), (2, 8)),
                                       rtol=0, atol=1e-12)
            np.testing.assert_allclose(L[b * B + i], math.log(len(rows)), rtol=0, atol=1e-12)


def test_attention_star_tree_sees_prefix_root_and_self():
    B, P = 6, 19
    star = np.array([-1] + [0] * (B - 1), dtype=np.int32)
    w = _small_workload(12, nb=1, B=B, Hq=2, Hkv=2, D=8, prefix=[P], trees=[star])
    O, _ = oracle.attn_workload(w)
    K = _f64(wl.logical_kv(w, 0, "k"))
    Vv = _f64(wl.logical_kv(w, 0, "v"))
    for i in range(B):
        rows = list(range(P + 1)) + ([P + i] if i else [])
        for h in range(2):
            ref = _sdpa_last_row(_f64(w.q[i, h]), K[rows, h], Vv[rows, h], 1 / math.sqrt(8))
            np.testing.assert_allclose(O[i, h], ref, rtol=0, atol=1e-12)


def _random_topological_relabel(rng, parent):
    """A node relabelling that keeps every parent before its children (random sibling order)."""
    B = len(parent)
    children = [[] for _ in range(B)]
    for i in range(1, B):
        children[parent[i]].append(i)
    order, frontier = [], [0]
    while frontier:
        k = int(rng.integers(0, len(frontier)))
        n = frontier.pop(k)
        order.append(n)
        frontier.extend(children[n])
    new_of_old = np.empty(B, dtype=np.int64)
    new_of_old[np.array(order)] = np.arange(B)
    new_parent = np.full(B, -1, dtype=np.int32)
    for old in range(1, B):
        new_parent[new_of_old[old]] = new_of_old[parent[old]]
    return new_of_old, new_parent


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_attention_invariant_under_sibling_relabelling(seed):
    rng = np.random.default_rng(seed)
    B, P, Hq, Hkv, D = 10, 23, 4, 2, 8
    w = _small_workload(20 + seed, nb=1, B=B, Hq=Hq, Hkv=Hkv, D=D, prefix=[P])
    O, L = oracle.attn_workload(w)
    nmap, npar = _random_topological_relabel(rng, w.parent[0])
    assert (npar[1:] < np.arange(1, B)).all()
    w2 = _small_workload(20 + seed, nb=1, B=B, Hq=Hq, Hkv=Hkv, D=D, prefix=[P], trees=[npar])
    # same data, relabelled: q rows and the tree slots of the cache move with the nodes
    w2.q[nmap] = w.q
    w2.k_cache[:] = w.k_cache
    w2.v_cache[:] = w.v_cache
    w2.block_table[:] = w.block_table
    for old in range(B):
        for cache, cache2 in ((w.k_cache, w2.k_cache), (w.v_cache, w2.v_cache)):
            po, pn = P + old, P + int(nmap[old])
            cache2[w.block_table[0, pn // 16], :, pn % 16] = cache[w.block_table[0, po // 16], :, po % 16]
    O2, L2 = oracle.attn_workload(w2)
    np.testing.assert_allclose(O2[nmap], O, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L2[nmap], L, rtol=0, atol=1e-12)


def test_attention_independent_of_physical_page_placement():
    w1 = _small_workload(31, nb=3, B=7, Hq=4, Hkv=2, D=8, prefix=[40, 3, 70], shuffle=False)
    w2 = _small_workload(31, nb=3, B=7, Hq=4, Hkv=2, D=8, prefix=[40, 3, 70], shuffle=True)
    # place w1's logical rows into w2's (shuffled) pages
    for b in range(3):
        for which in ("k", "v"):
            src = wl.logical_kv(w1, b, which)
            cache = w2.k_cache if which == "k" else w2.v_cache
            pos = np.arange(src.shape[0])
            cache[w2.block_table[b, pos // 16], :, pos % 16, :] = src
    w2.q[:] = w1.q
    w2.parent[:] = w1.parent
    O1, L1 = oracle.attn_workload(w1)
    O2, L2 = oracle.attn_workload(w2)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


def test_attention_key_ranges_merge_to_the_whole():
    w = _small_workload(41, nb=2, B=9, Hq=4, Hkv=2, D=16, prefix=[50, 130])
    O, L = oracle.attn_workload(w)
    for cuts in ([0, 16, -1], [0, 7, 64, 128, -1], [0, 55, 56, 131, 135, -1]):
        parts = []
        for lo, hi in zip(cuts[:-1], cuts[1:]):
            parts.append(oracle.attn_workload(w, key_range=(lo, hi)))
        Om, Lm = oracle.lse_merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
        np.testing.assert_allclose(Om, O, rtol=0, atol=1e-12)
        np.testing.assert_allclose(Lm, L, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------- argmax

def test_argmax_matches_numpy_first_occurrence():
    rng = np.random.default_rng(5)
    for V in (1, 2, 7, 1000, 4099):
        vals = rng.integers(-3, 4, size=(20, V)).astype(np.float32) * np.float32(0.5)  # many ties
        u = wl.f32_to_bf16(vals)
        assert np.array_equal(oracle.argmax(u), np.argmax(wl.bf16_to_f32(u), axis=1))
        x = wl.f32_to_bf16(rng.standard_normal((5, V), dtype=np.float32))
        assert np.array_equal(oracle.argmax(x), np.argmax(wl.bf16_to_f32(x), axis=1))


def test_argmax_signed_zero_and_nan():
    rows = np.array([[0x8000, 0x0000, 0xBF80],        # -0, +0, -1  -> first zero (index 0)
                     [0x3F80, 0x7FC0, 0x7F80],        # 1, NaN, +inf -> NaN counts as the max
                     [0xFF80, 0xFF80, 0xFF80],        # all -inf -> 0
                     [0x3F80, 0x7F80, 0xFFC1]],       # 1, +inf, -NaN -> the NaN
                    dtype=np.uint16)
    ref = torch.argmax(torch.from_numpy(wl.bf16_to_f32(rows)), dim=1).numpy()
    assert oracle.argmax(rows).tolist() == ref.tolist() == [0, 1, 0, 2]


# ------------------------------------------------------------------ acceptance

def test_accept_golden_example():
    fx = json.load(open(GOLDEN))
    parent = np.array([fx["tree"]["parent"]], dtype=np.int32)
    a = fx["accept"]
    logits = wl.f32_to_bf16(np.array(a["logits"], dtype=np.float32))
    for case in a["cases"]:
        am, n_acc, path, bonus = oracle.accept(logits, np.array([case["draft"]], np.int32), parent)
        assert am.tolist() == a["argmax"]
        assert n_acc[0] == case["n_acc"] and bonus[0] == case["bonus"]
        assert path[0].tolist() == case["path"]


def _brute_accept(parent, draft, am):
    """Enumerate every root-to-node path by DFS over child lists; keep the deepest fully matching one."""
    B = len(parent)
    children = [[] for _ in range(B)]
    for i in range(1, B):
        children[parent[i]].append(i)
    best = (0, 0, [0])                       # (length, -index, path)
    stack = [[0]]
    while stack:
        path = stack.pop()
        v = path[-1]
        key = (len(path) - 1, -v)
        if key > best[:2]:
            best = (len(path) - 1, -v, path)
        for c in children[v]:
            if draft[c] == am[v]:
                stack.append(path + [c])
    return best[0], best[2]


def _all_trees(B):
    return itertools.product(*[range(i) for i in range(1, B)])


@pytest.mark.parametrize("B", [1, 2, 3, 4, 5, 6, 7])
def test_accept_matches_exhaustive_path_enumeration(B):
    rng = np.random.default_rng(B)
    V = 3
    trees = [np.array((-1,) + t, dtype=np.int32) for t in _all_trees(B)]
    for parent in trees:
        for _ in range(2):
            logits = wl.f32_to_bf16(rng.integers(0, 3, size=(B, V)).astype(np.float32))
            draft = rng.integers(0, V, size=B).astype(np.int32)
            am, n_acc, path, bonus = oracle.accept(logits, draft, parent)
            am_ref = np.argmax(wl.bf16_to_f32(logits), axis=1)
            assert np.array_equal(am, am_ref)
            depth, p = _brute_accept(parent, draft, am_ref)
            assert n_acc[0] == depth
            assert path[0, :depth + 1].tolist() == p and (path[0, depth + 1:] == -1).all()
            assert bonus[0] == am_ref[p[-1]]


def test_accept_closed_forms():
    B, V = 9, 11
    chain = np.arange(-1, B - 1, dtype=np.int32)
    rng = np.random.default_rng(0)
    logits = wl.f32_to_bf16(rng.standard_normal((B, V), dtype=np.float32))
    am = np.argmax(wl.bf16_to_f32(logits), axis=1)
    draft = np.zeros(B, np.int32)
    draft[1:] = am[:-1]                                  # every draft matches: all accepted
    _, n_acc, path, bonus = oracle.accept(logits, draft, chain)
    assert n_acc[0] == B - 1 and path[0].tolist() == list(range(B)) and bonus[0] == am[-1]
    draft[1:] = (am[:-1] + 1) % V                        # nothing matches: root only
    _, n_acc, path, bonus = oracle.accept(logits, draft, chain)
    assert n_acc[0] == 0 and path[0].tolist() == [0] + [-1] * (B - 1) and bonus[0] == am[0]


def test_accept_rejects_non_topological():
    with pytest.raises(oracle.OracleError):
        oracle.accept(np.zeros((3, 4), np.uint16), np.zeros(3, np.int32), np.array([-1, 2, 0], np.int32))


# ------------------------------------------------------------------ KV commit

def _root_path(parent, v):
    out = []
    while v != -1:
        out.append(int(v))
        v = int(parent[v])
    return out[::-1]


def _commit_inputs(rng, parent):
    """A random acceptance outcome: the root path of a random node, as tv_accept returns it."""
    nb, B = parent.shape
    n_acc = np.zeros(nb, np.int32)
    path = np.full((nb, B), -1, np.int32)
    for b in range(nb):
        p = _root_path(parent[b], int(rng.integers(0, B)))
        n_acc[b] = len(p) - 1
        path[b, :len(p)] = p
    return n_acc, path


@pytest.mark.parametrize("seed", range(6))
def test_kv_commit_keeps_what_each_accepted_node_attended_to(seed):
    """Before the commit, node path[k] attends to the prefix and its root path path[0..k]
    (JETFLOW §2 mask).  After it, those keys are exactly positions [0, P + k], so a chain
    tree over the committed cache queried with the path nodes' queries gives the same rows:
    the same keys in the same order, hence bit-identical fp64 results."""
    rng = np.random.default_rng(100 + seed)
    w = _small_workload(seed, nb=3, B=12, Hq=4, Hkv=2, D=16, prefix=[0, 5, 37])
    n_acc, path = _commit_inputs(rng, w.parent)
    O_tree, L_tree = oracle.attn_workload(w)
    k2, v2, new_pl = oracle.kv_commit(w.k_cache, w.v_cache, w.block_table, w.prefix_lens, n_acc, path)
    assert np.array_equal(new_pl, w.prefix_lens + n_acc + 1)
    chain = np.tile(np.arange(-1, w.B - 1, dtype=np.int32), (w.nb, 1))
    q_chain = np.zeros_like(w.q)
    for b in range(w.nb):
        for k in range(n_acc[b] + 1):
            q_chain[b * w.B + k] = w.q[b * w.B + path[b, k]]
    O_ch, L_ch = oracle.attn(q_chain, k2, v2, w.block_table, w.prefix_lens, chain, w.Hq, w.Hkv)
    for b in range(w.nb):
        for k in range(n_acc[b] + 1):
            assert np.array_equal(O_ch[b * w.B + k], O_tree[b * w.B + path[b, k]])
            assert np.array_equal(L_ch[b * w.B + k], L_tree[b * w.B + path[b, k]])


def test_kv_commit_moves_only_the_accepted_rows():
    rng = np.random.default_rng(7)
    w = _small_workload(7, nb=4, B=20, Hq=4, Hkv=2, D=8, prefix=[3, 0, 16, 50])
    n_acc, path = _commit_inputs(rng, w.parent)
    k2, v2, new_pl = oracle.kv_commit(w.k_cache, w.v_cache, w.block_table, w.prefix_lens, n_acc, path)
    w2 = wl.Workload(**{**w.__dict__, "k_cache": k2, "v_cache": v2})
    for b in range(w.nb):
        P, n = int(w.prefix_lens[b]), int(n_acc[b])
        for which in ("k", "v"):
            before, after = wl.logical_kv(w, b, which), wl.logical_kv(w2, b, which)
            assert np.array_equal(after[:P + 1], before[:P + 1])              # prefix and root
            assert np.array_equal(after[P + n + 1:], before[P + n + 1:])      # everything past the path
            for k in range(1, n + 1):
                assert np.array_equal(after[P + k], before[P + path[b, k]])
    # physical pages no block table points at are untouched
    used = set(int(x) for x in w.block_table.reshape(-1) if x >= 0)
    for blk in range(w.num_blocks):
        if blk not in used:
            assert np.array_equal(k2[blk], w.k_cache[blk]) and np.array_equal(v2[blk], w.v_cache[blk])


def test_kv_commit_closed_forms():
    w = _small_workload(8, nb=2, B=9, Hq=2, Hkv=1, D=8, prefix=[4, 30],
                        trees=[np.arange(-1, 8, dtype=np.int32)] * 2)
    # nothing accepted: only the root is committed, no row moves
    path = np.full((2, 9), -1, np.int32)
    path[:, 0] = 0
    k2, v2, pl = oracle.kv_commit(w.k_cache, w.v_cache, w.block_table, w.prefix_lens, np.zeros(2, np.int32), path)
    assert np.array_equal(k2, w.k_cache) and np.array_equal(v2, w.v_cache)
    assert pl.tolist() == [5, 31]
    # a chain accepted in full is already in place
    full = np.tile(np.arange(9, dtype=np.int32), (2, 1))
    k2, v2, pl = oracle.kv_commit(w.k_cache, w.v_cache, w.block_table, w.prefix_lens, np.full(2, 8, np.int32), full)
    assert np.array_equal(k2, w.k_cache) and np.array_equal(v2, w.v_cache)
    assert pl.tolist() == [13, 39]


@pytest.mark.parametrize("bad", [[0, 2, 2], [1, 2, 3], [0, 5, 3], [0, 1, 9]])
def test_kv_commit_rejects_a_path_that_is_not_a_root_path(bad):
    w = _small_workload(9, nb=1, B=9, Hq=2, Hkv=1, D=8, prefix=[4])
    path = np.full((1, 9), -1, np.int32)
    path[0, :3] = bad
    with pytest.raises(oracle.OracleError):
        oracle.kv_commit(w.k_cache, w.v_cache, w.block_table, w.prefix_lens, np.array([2], np.int32), path)


# --------------------------------------------------------------- tree building

def _tree_inputs(seed, nb, Dmax, K):
    """Distinct random log-probs, sorted best first per depth; token = 1000 * depth + rank."""
    rng = np.random.default_rng(seed)
    lp = np.log(rng.dirichlet([0.3] * K, size=(nb, Dmax)) + 1e-9).astype(np.float32)
    lp = -np.sort(-lp, axis=-1)
    tok = np.broadcast_to((1000 * np.arange(1, Dmax + 1)[:, None] + np.arange(K)[None, :]).astype(np.int32),
                          (nb, Dmax, K)).copy()
    return lp, tok


def _all_paths(lp, Dmax, K):
    """Every node of the full K-ary tree as (rank path, fp32 score accumulated root to leaf)."""
    out = [((), np.float32(0.0))]
    frontier = [((), np.float32(0.0))]
    for d in range(Dmax):
        nxt = []
        for path, s in frontier:
            for c in range(K):
                nxt.append((path + (c,), np.float32(s + lp[d, c])))
        out += nxt
        frontier = nxt
    return out


def _rank_paths(parent, token):
    """Rank path of every node, read off the tokens (token % 1000 = rank)."""
    paths = [()]
    for i in range(1, len(parent)):
        paths.append(paths[parent[i]] + (int(token[i]) % 1000,))
    return paths


@pytest.mark.parametrize("Dmax,K,B", [(3, 4, 20), (4, 3, 60), (2, 5, 31), (6, 2, 64)])
def test_build_tree_best_first_is_the_top_B_nodes_by_score(Dmax, K, B):
    """w = 1: the nodes are the B best-scoring nodes of the full tree (log-probs <= 0, so the
    set is closed under taking parents), created in decreasing score order (brute force)."""
    lp, tok = _tree_inputs(Dmax * 10 + K, 2, Dmax, K)
    parent, token, score = oracle.build_tree(lp, tok, B, 1)
    for b in range(2):
        every = sorted(_all_paths(lp[b], Dmax, K), key=lambda t: -t[1])
        want = [p for p, _ in every[:B]]
        assert _rank_paths(parent[b], token[b]) == want
        assert np.all(np.diff(score[b]) <= 0)
        for i in range(1, B):
            assert score[b, i] == np.float32(score[b, parent[b, i]] + lp[b, len(want[i]) - 1, want[i][-1]])


@pytest.mark.parametrize("w", [2, 3, 8, 64])
def test_build_tree_top_w_rounds(w):
    """Each round takes the w best candidates available when it starts (children of nodes made
    in earlier rounds), in order, recomputed here from the output tree alone."""
    Dmax, K, B = 5, 4, 100
    lp, tok = _tree_inputs(w, 1, Dmax, K)
    parent, token, score = oracle.build_tree(lp, tok, B, w)
    par, paths = parent[0], _rank_paths(parent[0], token[0])
    made = 1
    while made < B:
        have = set(paths[:made])
        avail = []
        for u in range(made):
            if len(paths[u]) < Dmax:
                for c in range(K):
                    if paths[u] + (c,) not in have:
                        avail.append((-np.float32(score[0, u] + lp[0, len(paths[u]), c]), u, c))
        avail.sort()
        take = min(w, B - made, len(avail))  # a round takes fewer when fewer are available
        for t in range(take):
            i = made + t
            assert (par[i], paths[i][-1]) == (avail[t][1], avail[t][2])
            assert score[0, i] == -avail[t][0]
        made += take


def test_build_tree_closed_forms():
    lp, tok = _tree_inputs(5, 1, 6, 3)
    # one candidate per depth: a chain whose scores are the running sums
    p1, t1, s1 = oracle.build_tree(lp[:, :, :1].copy(), tok[:, :, :1].copy(), 7, 3)
    assert p1[0].tolist() == [-1, 0, 1, 2, 3, 4, 5]
    assert np.array_equal(s1[0, 1:], np.cumsum(lp[0, :, 0], dtype=np.float32))
    # depth 1 only: a star of the best candidates in rank order
    p2, t2, s2 = oracle.build_tree(lp[:, :1].copy(), tok[:, :1].copy(), 4, 1)
    assert p2[0].tolist() == [-1, 0, 0, 0] and t2[0].tolist() == [-1, 1000, 1001, 1002]
    # a budget larger than the full tree is an argument error
    with pytest.raises(oracle.OracleError):
        oracle.build_tree(lp[:, :1].copy(), tok[:, :1].copy(), 5, 1)


# ------------------------------------------------------ Gated DeltaNet over a tree

def _gdn_path(parent, i):
    out = []
    while i != -1:
        out.append(i)
        i = int(parent[i])
    return out[::-1]


def _gdn_small(seed, nb=2, B=12, H=2, D=16, trees=None):
    rng = np.random.default_rng(seed)
    if trees is None:
        trees = _random_trees(rng, B, nb)
    return wl.make_gdn_workload("pin", nb, B, H, D, trees, seed)


def test_gdn_zero_write_strength_closed_form():
    """beta = 0: the state only decays, o_i = (prod of alpha on i's root path) S0^T q_i."""
    w = _gdn_small(1)
    beta = np.zeros_like(w.beta)
    O = oracle.gdn_tree(w.q, w.k, w.v, w.alpha, beta, w.S0, w.parent)
    for b in range(w.nb):
        for i in range(w.B):
            g = np.prod([np.float64(w.alpha[b * w.B + j]) for j in _gdn_path(w.parent[b], i)], axis=0)  # [H]
            for h in range(w.H):
                want = g[h] * (w.S0[b, h].astype(np.float64).T @ _f64(w.q[b * w.B + i, h]))
                assert np.allclose(O[b * w.B + i, h], want, rtol=1e-12, atol=1e-14)


def test_gdn_unit_keys_overwrite_rows():
    """alpha = beta = 1 and unit keys e_r: each step replaces row r of the state by v, so node i's
    state is S0 with the rows of its path's keys replaced (a key met twice keeps the later v)."""
    B, D = 10, 16
    rng = np.random.default_rng(3)
    w = _gdn_small(3, nb=1, B=B, H=1, D=D)
    rows = rng.integers(0, D, size=B)
    k = np.zeros((B, 1, D), np.float32)
    k[np.arange(B), 0, rows] = 1.0
    kb = wl.f32_to_bf16(k)
    ones = np.ones_like(w.alpha)
    O = oracle.gdn_tree(w.q, kb, w.v, ones, ones, w.S0, w.parent)
    for i in range(B):
        S = w.S0[0, 0].astype(np.float64).copy()
        for j in _gdn_path(w.parent[0], i):
            S[rows[j]] = _f64(w.v[j, 0])
        assert np.allclose(O[i, 0], S.T @ _f64(w.q[i, 0]), rtol=1e-12, atol=1e-14)


def test_gdn_matches_the_masked_triangular_solve():
    """The chunked form the pages sketch (DFlash-TfM §3): with gamma_i the product of alpha on
    i's root path, (I + X) U = beta (V - gamma K S0), X_ij = beta_i (gamma_i / gamma_j) k_i.k_j
    for j a strict ancestor of i, and O = gamma Q S0 + Y U, Y_ij = (gamma_i / gamma_j) q_i.k_j
    for j an ancestor of i or i itself.  Solved densely by numpy, it must equal the per-path
    recurrence."""
    w = _gdn_small(5, nb=2, B=14, H=3, D=16)
    O = oracle.gdn_tree(w.q, w.k, w.v, w.alpha, w.beta, w.S0, w.parent)
    for b in range(w.nb):
        anc = [set(_gdn_path(w.parent[b], i)) for i in range(w.B)]
        for h in range(w.H):
            r = slice(b * w.B, (b + 1) * w.B)
            Q, Kk, Vv = _f64(w.q[r, h]), _f64(w.k[r, h]), _f64(w.v[r, h])
            al, be = w.alpha[r, h].astype(np.float64), w.beta[r, h].astype(np.float64)
            S0 = w.S0[b, h].astype(np.float64)
            gam = np.array([np.prod([al[j] for j in anc[i]]) for i in range(w.B)])
            X = np.zeros((w.B, w.B))
            Y = np.zeros((w.B, w.B))
            for i in range(w.B):
                for j in anc[i]:
                    Y[i, j] = gam[i] / gam[j] * (Q[i] @ Kk[j])
                    if j != i:
                        X[i, j] = be[i] * gam[i] / gam[j] * (Kk[i] @ Kk[j])
            U = np.linalg.solve(np.eye(w.B) + X, be[:, None] * (Vv - gam[:, None] * (Kk @ S0)))
            want = gam[:, None] * (Q @ S0) + Y @ U
            assert np.allclose(O[r, h], want, rtol=1e-9, atol=1e-11)


def test_gdn_invariant_under_sibling_relabelling():
    rng = np.random.default_rng(8)
    w = _gdn_small(8, nb=1, B=12, H=2, D=16)
    parent = w.parent[0]
    new_of_old, new_parent = _random_topological_relabel(rng, parent)
    old_of_new = np.argsort(new_of_old)
    O = oracle.gdn_tree(w.q, w.k, w.v, w.alpha, w.beta, w.S0, w.parent)
    O2 = oracle.gdn_tree(w.q[old_of_new], w.k[old_of_new], w.v[old_of_new], w.alpha[old_of_new],
                         w.beta[old_of_new], w.S0, new_parent[None])
    assert np.allclose(O2[new_of_old], O, rtol=1e-12, atol=1e-14)


# ------------------------------------------- Gated DeltaNet: commit of the accepted branch

def _gdn_accepted(w, seed):
    """An accepted root path per sequence: a random node's root path (root first)."""
    rng = np.random.default_rng(seed)
    n_acc = np.zeros(w.nb, np.int32)
    path = np.full((w.nb, w.B), -1, np.int32)
    for b in range(w.nb):
        p = _gdn_path(w.parent[b], int(rng.integers(0, w.B)))
        n_acc[b] = len(p) - 1
        path[b, :len(p)] = p
    return n_acc, path


def test_gdn_commit_zero_write_strength_closed_form():
    """beta = 0: the state only decays, S_new = (prod of alpha on the accepted path) S0."""
    w = _gdn_small(21)
    n_acc, path = _gdn_accepted(w, 1)
    beta = np.zeros_like(w.beta)
    S = oracle.gdn_commit(w.k, w.v, w.alpha, beta, w.S0, n_acc, path)
    for b in range(w.nb):
        rows = [b * w.B + j for j in path[b, :n_acc[b] + 1]]
        g = np.prod(w.alpha[rows].astype(np.float64), axis=0)  # [H]
        for h in range(w.H):
            assert np.allclose(S[b, h], g[h] * w.S0[b, h].astype(np.float64), rtol=1e-12, atol=1e-14)


def test_gdn_commit_matches_the_chunked_form():
    """The chunked (WY) form along the accepted path p_0 .. p_n: with gamma_t the product of
    alpha over p_0 .. p_t and r_ts = gamma_t / gamma_s, (I + X) U = beta (V - gamma K S0) with
    X_ts = beta_t r_ts k_t.k_s (s < t), and S_new = gamma_n S0 + sum_s r_ns k_s u_s^T.  Solved
    densely by numpy, it must equal the step-by-step recurrence."""
    w = _gdn_small(22, nb=3, B=16, H=2, D=16)
    n_acc, path = _gdn_accepted(w, 2)
    S = oracle.gdn_commit(w.k, w.v, w.alpha, w.beta, w.S0, n_acc, path)
    for b in range(w.nb):
        rows = [b * w.B + j for j in path[b, :n_acc[b] + 1]]
        n = len(rows)
        for h in range(w.H):
            Kk, Vv = _f64(w.k[rows, h]), _f64(w.v[rows, h])
            al, be = w.alpha[rows, h].astype(np.float64), w.beta[rows, h].astype(np.float64)
            S0 = w.S0[b, h].astype(np.float64)
            gam = np.cumprod(al)
            X = np.zeros((n, n))
            for t in range(n):
                for s in range(t):
                    X[t, s] = be[t] * gam[t] / gam[s] * (Kk[t] @ Kk[s])
            U = np.linalg.solve(np.eye(n) + X, be[:, None] * (Vv - gam[:, None] * (Kk @ S0)))
            want = gam[-1] * S0 + (Kk * (gam[-1] / gam)[:, None]).T @ U
            assert np.allclose(S[b, h], want, rtol=1e-9, atol=1e-11)


def test_gdn_commit_agrees_with_the_tree_outputs():
    """The accepted node's tree output is its state's read-out, so S_new^T q_{p_n} equals it."""
    w = _gdn_small(23, nb=2, B=14, H=3, D=16)
    n_acc, path = _gdn_accepted(w, 3)
    S = oracle.gdn_commit(w.k, w.v, w.alpha, w.beta, w.S0, n_acc, path)
    O = oracle.gdn_tree(w.q, w.k, w.v, w.alpha, w.beta, w.S0, w.parent)
    for b in range(w.nb):
        last = b * w.B + int(path[b, n_acc[b]])
        for h in range(w.H):
            assert np.allclose(S[b, h].T @ _f64(w.q[last, h]), O[last, h], rtol=1e-10, atol=1e-12)


def test_gdn_commit_root_only_is_one_step():
    """n_acc = 0 commits the root alone: one step of the recurrence from S0."""
    w = _gdn_small(24, nb=1, B=6, H=2, D=8)
    path = np.full((1, 6), -1, np.int32)
    path[0, 0] = 0
    S = oracle.gdn_commit(w.k, w.v, w.alpha, w.beta, w.S0, np.zeros(1, np.int32), path)
    for h in range(w.H):
        kk, vv = _f64(w.k[0, h]), _f64(w.v[0, h])
        a, be = float(w.alpha[0, h]), float(w.beta[0, h])
        S0 = w.S0[0, h].astype(np.float64)
        want = a * (np.eye(w.D) - be * np.outer(kk, kk)) @ S0 + be * np.outer(kk, vv)
        assert np.allclose(S[0, h], want, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("bad", [[1, 2], [0, 3, 3], [0, 20]])
def test_gdn_commit_rejects_a_path_that_is_not_a_root_path(bad):
    w = _gdn_small(25, nb=1, B=12, H=1, D=8)
    path = np.full((1, 12), -1, np.int32)
    path[0, :len(bad)] = bad
    with pytest.raises(oracle.OracleError):
        oracle.gdn_commit(w.k, w.v, w.alpha, w.beta, w.S0, np.array([len(bad) - 1], np.int32), path)
