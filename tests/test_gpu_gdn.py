"""GPU parity of tv_gdn_tree (Gated DeltaNet tree verification) against the fp64 oracle.

Every output element is compared.  Tolerance: the device works in fp32 (bf16 q/k/v
read exactly).  Each output element is gamma_i (S0^T q_i)_c plus one term per node
on i's root path, and each of those is a length-128 fp32 dot product (or a product
of them) whose rounding error is at most 128 * 2^-24 times the sum of the absolute
products, which these inputs bound by 4 (unit q and k, |S0| entries under 0.6, |v|
and |u| under 3).  A node at depth d therefore stays within
tol(d) = (d + 2) * 128 * 2^-24 * 4 of the exact value (5.5e-4 at depth 16), which
the tests apply node by node.  A dropped ancestor term moves an output by about
beta |k_i.k_j| |u_j| ~ 0.02, a wrong gate power by ~0.1 |S0^T q| ~ 0.005.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
import tree_speculative_decoding_tv_gb300 as tv
import workloads as wl
from tests.helpers import bf16_dev, i32_dev

pytestmark = pytest.mark.gpu

TOL16 = 18 * 128 * 2.0 ** -24 * 4


def _tol(parent):
    """Per-node tolerance [nb*B][1][1] from each node's depth."""
    nb, B = parent.shape
    dep = np.zeros((nb, B))
    for b in range(nb):
        for i in range(1, B):
            dep[b, i] = dep[b, parent[b, i]] + 1
    return ((dep + 2) * 128 * 2.0 ** -24 * 4).reshape(nb * B, 1, 1)


def _assert_close(got, ref, parent):
    err = np.abs(got - ref) - _tol(parent)
    assert np.isfinite(got).all()
    assert err.max() <= 0, f"error over tolerance by {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}"


def _dev(w):
    f = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return dict(q=bf16_dev(w.q), k=bf16_dev(w.k), v=bf16_dev(w.v), alpha=f(w.alpha), beta=f(w.beta), S0=f(w.S0),
                parent=i32_dev(w.parent))


def _run(w, status=None):
    d = _dev(w)
    st = torch.zeros(1, dtype=torch.int32, device="cuda") if status is None else status
    O = tv.gdn_tree(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["S0"], d["parent"], status=st)
    torch.cuda.synchronize()
    return O, int(st.item())


def _chain(B):
    return np.arange(-1, B - 1, dtype=np.int32)


def _star(B):
    p = np.zeros(B, np.int32)
    p[0] = -1
    return p


def _random_tree(B):
    def gen(r):
        p = np.empty(B, np.int32)
        p[0] = -1
        for i in range(1, B):
            p[i] = r.integers(max(0, i - 8), i)  # a recent node: deep and bushy
        return p
    return gen


CASES = {
    "single node": (1, 1, 3, lambda r: np.array([-1], np.int32)),
    "chain of 33 (ragged row tile)": (2, 33, 2, lambda r: _chain(33)),
    "star of 64": (1, 64, 2, lambda r: _star(64)),
    "best-first 48, 3 sequences": (3, 48, 4, lambda r: wl.tree_best_first(r, 48, child_cap=4, max_depth=16)),
    "random 200": (1, 200, 2, _random_tree(200)),
    "best-first 256 (largest tree)": (1, 256, 2, lambda r: wl.tree_best_first(r, 256, child_cap=4, max_depth=16)),
    "chain of 256": (1, 256, 1, lambda r: _chain(256)),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_gdn_tree_matches_oracle(case):
    nb, B, H, trees = CASES[case]
    w = wl.make_gdn_workload(case, nb, B, H, 128, trees, seed=zlib.crc32(case.encode()))
    O, st = _run(w)
    assert st == 0
    ref = oracle.gdn_tree(w.q, w.k, w.v, w.alpha, w.beta, w.S0, w.parent)
    _assert_close(O.cpu().numpy().astype(np.float64), ref, w.parent)


def test_gdn_tree_full_size():
    """The benchmarked workload (1 sequence, 128-node best-first tree, 32 heads of 128), every element."""
    w = wl.gdn_config(seed=4321)
    O, st = _run(w)
    assert st == 0
    ref = oracle.gdn_tree(w.q, w.k, w.v, w.alpha, w.beta, w.S0, w.parent)
    _assert_close(O.cpu().numpy().astype(np.float64), ref, w.parent)


def test_gdn_tree_sibling_relabelling_permutes_outputs():
    """At any size: relabelling nodes by another topological order permutes the outputs
    (each node's output depends only on its own root path)."""
    w = wl.make_gdn_workload("relabel", 1, 96, 8, 128,
                             lambda r: wl.tree_best_first(r, 96, child_cap=4, max_depth=16), seed=77)
    rng = np.random.default_rng(5)
    par = w.parent[0]
    # a random topological order: repeatedly take a random node whose parent is already placed
    placed, order = {-1}, []
    avail = [0]
    children = {i: [j for j in range(w.B) if par[j] == i] for i in range(w.B)}
    while avail:
        x = avail.pop(int(rng.integers(len(avail))))
        order.append(x)
        placed.add(x)
        avail += children[x]
    old_of_new = np.array(order)
    new_of_old = np.argsort(old_of_new)
    new_parent = np.array([-1 if par[o] < 0 else new_of_old[par[o]] for o in old_of_new], np.int32)
    w2 = wl.GdnWorkload(name="relabelled", nb=1, B=w.B, H=w.H, D=w.D, q=w.q[old_of_new], k=w.k[old_of_new],
                        v=w.v[old_of_new], alpha=w.alpha[old_of_new], beta=w.beta[old_of_new], S0=w.S0,
                        parent=new_parent[None])
    O1, s1 = _run(w)
    O2, s2 = _run(w2)
    assert s1 == 0 and s2 == 0
    d = (O2.cpu() - O1.cpu()[torch.from_numpy(old_of_new)]).abs().max().item()
    assert d <= 2 * TOL16  # best-first trees here are at most 16 deep


def test_gdn_tree_rejects_non_topological_parent():
    w = wl.make_gdn_workload("bad", 2, 16, 2, 128, lambda r: _chain(16), seed=3)
    w.parent[1, 5] = 9  # a later node as parent
    O, st = _run(w)
    assert st == 2  # TV_ERR_NOT_TOPOLOGICAL


def test_gdn_tree_empty_batch_is_a_no_op():
    z = torch.empty((0, 4, 128), dtype=torch.bfloat16, device="cuda")
    a = torch.empty((0, 4), dtype=torch.float32, device="cuda")
    S0 = torch.empty((0, 4, 128, 128), dtype=torch.float32, device="cuda")
    parent = torch.empty((0, 8), dtype=torch.int32, device="cuda")
    O = tv.gdn_tree(z, z, z, a, a, S0, parent)
    torch.cuda.synchronize()
    assert O.shape == (0, 4, 128)


def test_gdn_tree_in_a_cuda_graph():
    """The two launches capture and replay in a CUDA graph; the replay matches the eager call."""
    w = wl.gdn_config(seed=11)
    d = _dev(w)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    O = torch.empty((w.nb * w.B, w.H, w.D), dtype=torch.float32, device="cuda")
    ws = torch.empty(tv.lib().tv_gdn_tree_workspace_size(w.nb, w.B, w.H, w.D), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        tv.gdn_tree(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["S0"], d["parent"], out=O, workspace=ws,
                    status=st, stream=s)
    torch.cuda.synchronize()
    eager = O.clone()
    O.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        tv.gdn_tree(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["S0"], d["parent"], out=O, workspace=ws,
                    status=st, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(O, eager)


# ------------------------------------------- commit of the accepted branch (tv_gdn_commit)

def _accepted_paths(w, seed, deepest=False):
    """Per sequence, a node's root path (root first): a random node, or the deepest one."""
    rng = np.random.default_rng(seed)
    n_acc = np.zeros(w.nb, np.int32)
    path = np.full((w.nb, w.B), -1, np.int32)
    for b in range(w.nb):
        par = w.parent[b]
        dep = np.zeros(w.B, int)
        for i in range(1, w.B):
            dep[i] = dep[par[i]] + 1
        i = int(np.argmax(dep)) if deepest else int(rng.integers(0, w.B))
        p = []
        while i != -1:
            p.append(i)
            i = int(par[i])
        p = p[::-1]
        n_acc[b] = len(p) - 1
        path[b, :len(p)] = p
    return n_acc, path


def _commit_tol(n_acc, ref):
    """fp32 bound per element: (L + 2) length-128 dot products, each within 128 * 2^-24 of the
    sum of its absolute products, <= sqrt(128) max|S| for unit keys, plus |v| <= 3 terms."""
    L = n_acc.astype(np.float64) + 1
    scale = 11.4 * np.abs(ref).max(axis=(1, 2, 3)) + 3.0
    return ((L + 2) * 128 * 2.0 ** -24 * scale).reshape(-1, 1, 1, 1)


def _commit_dev(w, n_acc, path, in_place=False):
    d = _dev(w)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    S0 = d["S0"].clone()
    out = tv.gdn_commit(d["k"], d["v"], d["alpha"], d["beta"], S0, torch.from_numpy(n_acc).cuda(),
                        torch.from_numpy(path).cuda(), out=S0 if in_place else None, status=st)
    torch.cuda.synchronize()
    return out, int(st.item())


COMMIT_CASES = {
    "random paths, 3 sequences": (3, 48, 4, lambda r: wl.tree_best_first(r, 48, child_cap=4, max_depth=16), False),
    "deepest path of a 256-node tree": (1, 256, 2, lambda r: wl.tree_best_first(r, 256, child_cap=4, max_depth=16),
                                        True),
    "chain of 64, accepted whole": (2, 64, 2, lambda r: _chain(64), True),
    "single node": (2, 1, 3, lambda r: np.array([-1], np.int32), False),
    "33 heads, 2 sequences": (2, 32, 33, lambda r: wl.tree_best_first(r, 32, child_cap=3, max_depth=12), True),
}


@pytest.mark.parametrize("in_place", [False, True])
@pytest.mark.parametrize("case", sorted(COMMIT_CASES))
def test_gdn_commit_matches_oracle(case, in_place):
    nb, B, H, trees, deepest = COMMIT_CASES[case]
    w = wl.make_gdn_workload(case, nb, B, H, 128, trees, seed=zlib.crc32(case.encode()) + 1)
    n_acc, path = _accepted_paths(w, 7, deepest)
    out, st = _commit_dev(w, n_acc, path, in_place)
    assert st == 0
    ref = oracle.gdn_commit(w.k, w.v, w.alpha, w.beta, w.S0, n_acc, path)
    err = np.abs(out.cpu().numpy().astype(np.float64) - ref) - _commit_tol(n_acc, ref)
    assert err.max() <= 0, f"over tolerance by {err.max():.3e}"


def test_gdn_commit_reads_out_the_accepted_nodes_tree_output():
    """On the device too: the committed state read through the last accepted node's query
    equals that node's tv_gdn_tree output."""
    w = wl.gdn_config(seed=31)
    n_acc, path = _accepted_paths(w, 8, deepest=True)
    S, st = _commit_dev(w, n_acc, path)
    O, st2 = _run(w)
    assert st == 0 and st2 == 0
    last = int(path[0, n_acc[0]])
    q = torch.from_numpy(wl.bf16_to_f32(w.q[last]).astype(np.float32)).cuda()  # [H][D]
    readout = torch.einsum("hrc,hr->hc", S[0], q)
    # both sides approximate S_last^T q_last: the tree output within its per-node bound, the
    # read-out within sqrt(128) (unit q) times the state's bound plus its own dot product
    ref = oracle.gdn_commit(w.k, w.v, w.alpha, w.beta, w.S0, n_acc, path)
    s_tol = float(_commit_tol(n_acc, ref).max())
    smax = float(np.abs(ref).max())
    tol = (n_acc[0] + 2) * 128 * 2.0 ** -24 * 4 + 128 ** 0.5 * s_tol + 128 * 2.0 ** -24 * 128 ** 0.5 * smax
    assert (readout - O[last]).abs().max().item() <= tol


def test_gdn_commit_rejects_a_bad_path():
    w = wl.make_gdn_workload("bad", 2, 16, 2, 128, lambda r: _chain(16), seed=4)
    n_acc = np.array([3, 2], np.int32)
    path = np.full((2, 16), -1, np.int32)
    path[0, :4] = [0, 1, 2, 3]
    path[1, :3] = [0, 5, 5]  # not strictly increasing
    out, st = _commit_dev(w, n_acc, path)
    assert st == 1  # TV_ERR_INVALID_ARG
    assert torch.equal(out[1].cpu(), torch.from_numpy(w.S0[1]))  # nothing committed there
